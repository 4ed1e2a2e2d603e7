// api.cu - the exported C ABI of libattn.so (see include/attn.h).
//
// Validates arguments on the host, derives the RoPE frequency table, builds
// TMA tensor maps and launches the kernels on the caller's stream.  Nothing is
// allocated: every buffer belongs to the caller.
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <atomic>
#include <mutex>

#include <cudaTypedefs.h>

#include "attn.h"
#include "kernels.h"

namespace attn {
namespace {

// Status word written by device-side bounded waits (bit 0: a wait expired).
__device__ unsigned int g_status;

std::atomic<unsigned long long> g_launches{0};
std::atomic<unsigned long long> g_wait_limit_ns{2000000000ull};

constexpr int kMaxDevices = 64;
struct DeviceInfo {
  bool ready;
  int sms;
  int l2_bytes;
  unsigned int* status;
};
DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

// Per-device facts, fetched once per device with that device current.
int device_info(DeviceInfo* out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_dev_mu);
  DeviceInfo& d = g_dev[dev];
  if (!d.ready) {
    if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return ATTN_ERR_CUDA;
    if (cudaDeviceGetAttribute(&d.l2_bytes, cudaDevAttrL2CacheSize, dev) != cudaSuccess) return ATTN_ERR_CUDA;
    if (cudaGetSymbolAddress(reinterpret_cast<void**>(&d.status), g_status) != cudaSuccess) return ATTN_ERR_CUDA;
    d.ready = true;
  }
  *out = d;
  return ATTN_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 4-D tensor map over a bf16 tensor indexed (d, head, position, batch) with
// the given byte strides of head / position / batch: boxes of 64 dims x 1 head x
// box_rows positions x 1 batch, 128-byte swizzle (the canonical K-major operand
// layout of the tensor cores), zero fill outside the tensor.
bool make_map4(CUtensorMap* map, const void* base, int D, int heads, int rows, int B, unsigned long long head_stride,
               unsigned long long row_stride, unsigned long long batch_stride, int box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(heads),
                              static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(B)};
  const cuuint64_t strides[3] = {head_stride, row_stride, batch_stride};
  const cuuint32_t box[4] = {64, 1, static_cast<cuuint32_t>(box_rows), 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D tensor map over a bf16 tensor indexed (d, row, batch): boxes of 64 dims x
// box_rows rows x 1 batch, 128-byte swizzle, zero fill outside.
bool make_map3(CUtensorMap* map, const void* base, int D, int rows, int B, unsigned long long row_stride,
               unsigned long long batch_stride, int box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(B)};
  const cuuint64_t strides[2] = {row_stride, batch_stride};
  const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(box_rows), 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// MLA shape served by the tensor-core decode kernel (one 576-dim latent head, V = its first 512 dims).
bool mla_shape(int B, int n_h, int n_kv, int D_qk, int D_v, bool bf16) {
  return bf16 && n_h == 128 && n_kv == 1 && D_qk == 576 && D_v == 512 && B <= 1024;
}

// Dense BSHD tensor [B, S, heads, D], boxes of 128 positions.
bool make_bshd_map(CUtensorMap* map, const void* base, int B, int S, int heads, int D) {
  const unsigned long long hs = static_cast<unsigned long long>(D) * 2;
  return make_map4(map, base, D, heads, S, B, hs, hs * heads, hs * heads * S, 128);
}

// The dtype argument: element type in the low byte, ATTN_ROPE_HALF optionally
// OR'd in.  False for anything else.
bool parse_dtype(attn_dtype_t dtype, bool* bf16, bool* half) {
  const unsigned d = static_cast<unsigned>(dtype);
  const unsigned elem = d & 0xffu, flags = d & ~0xffu;
  if (elem != ATTN_F32 && elem != ATTN_BF16) return false;
  if (flags & ~static_cast<unsigned>(ATTN_ROPE_HALF)) return false;
  *bf16 = elem == ATTN_BF16;
  *half = flags != 0;
  return true;
}

// theta_i = base^(-2i/dims) expressed in turns per position, split hi + lo.
RopeFreq make_rope(float base, int dims, bool half) {
  RopeFreq f;
  memset(&f, 0, sizeof(f));
  if (!(base > 0.f) || dims <= 0) return f;
  f.n_pairs = dims / 2;
  f.half = half ? 1 : 0;
  const double two_pi = 6.283185307179586476925286766559;
  for (int i = 0; i < f.n_pairs; ++i) {
    const double turns = pow(static_cast<double>(base), -2.0 * i / dims) / two_pi;
    f.hi[i] = static_cast<float>(turns);
    f.lo[i] = static_cast<float>(turns - static_cast<double>(f.hi[i]));
  }
  return f;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool overlap(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

int finish(cudaError_t e, int launches) {
  g_launches.fetch_add(static_cast<unsigned long long>(launches));
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

const float kLog2e = 1.4426950408889634f;

// One warp waits on a barrier that nothing arrives on; the bounded wait gives
// up after limit_ns and records STATUS_TIMEOUT.
__global__ void wait_timeout_check_kernel(unsigned int* status, unsigned long long limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncwarp();
  const WaitCtl w{&abort_flag, status, limit_ns};
  mbar_wait(&bar, 0, w);
}

}  // namespace
}  // namespace attn

using namespace attn;

extern "C" {

const char* attn_strerror(int code) {
  switch (code) {
    case ATTN_OK: return "ok";
    case ATTN_ERR_ARG: return "invalid argument";
    case ATTN_ERR_UNSUPPORTED: return "unsupported head size or dtype";
    case ATTN_ERR_ALIGN: return "pointer not 16-byte aligned";
    case ATTN_ERR_CUDA: return "CUDA runtime error";
    case ATTN_ERR_TIMEOUT: return "a device-side bounded wait expired";
    case ATTN_ERR_WORKSPACE: return "workspace too small";
    default: return "unknown error";
  }
}

}  // extern "C"

namespace attn {
namespace {
int rope_impl(void* x_out, const void* x_in, const int* positions, int B, int S, int n_heads, int D, int rope_offset,
              int rope_dims, float rope_base, int pos_offset, attn_dtype_t dtype, void* stream) {
  if (!x_out || !x_in || B <= 0 || S <= 0 || n_heads <= 0 || D <= 0) return ATTN_ERR_ARG;
  bool bf16 = false, half = false;
  if (!parse_dtype(dtype, &bf16, &half)) return ATTN_ERR_ARG;
  if (!(rope_base > 0.f) || rope_offset < 0 || rope_dims <= 0 || rope_offset + rope_dims > D || pos_offset < 0)
    return ATTN_ERR_ARG;
  const int unit = bf16 ? 8 : 2;  // a thread's chunk of dims; with half pairing each half is whole chunks
  if (D % unit || rope_offset % unit || rope_dims % (half ? 2 * unit : unit)) return ATTN_ERR_ARG;
  if (rope_dims / 2 > kMaxRopePairs) return ATTN_ERR_UNSUPPORTED;
  if (!aligned16(x_out) || !aligned16(x_in) || (reinterpret_cast<uintptr_t>(positions) & 3u)) return ATTN_ERR_ALIGN;
  const size_t bytes = static_cast<size_t>(B) * S * n_heads * D * (bf16 ? 2 : 4);
  if (x_out != x_in && overlap(x_out, bytes, x_in, bytes)) return ATTN_ERR_ARG;
  RopeArgs ra{x_out, x_in, B, S, n_heads, D, rope_offset, rope_dims, pos_offset, positions};
  int launches = 0;
  const cudaError_t e =
      launch_rope(ra, make_rope(rope_base, rope_dims, half), bf16, static_cast<cudaStream_t>(stream), &launches);
  return finish(e, launches);
}
}  // namespace
}  // namespace attn

extern "C" {

int attn_rope(void* x_out, const void* x_in, int B, int S, int n_heads, int D, int rope_offset, int rope_dims,
              float rope_base, int pos_offset, attn_dtype_t dtype, void* stream) {
  return rope_impl(x_out, x_in, nullptr, B, S, n_heads, D, rope_offset, rope_dims, rope_base, pos_offset, dtype,
                   stream);
}

int attn_rope_at(void* x_out, const void* x_in, const int* positions, int B, int S, int n_heads, int D,
                 int rope_offset, int rope_dims, float rope_base, attn_dtype_t dtype, void* stream) {
  if (!positions) return ATTN_ERR_ARG;
  return rope_impl(x_out, x_in, positions, B, S, n_heads, D, rope_offset, rope_dims, rope_base, 0, dtype, stream);
}

namespace attn {
namespace {
int prefill_impl(const void* q, const void* k, const void* v, void* out, void* k_rot, float* lse, int B, int S,
                 int n_h, int n_kv, int D_qk, int D_v, float rope_base, int rope_offset, int rope_dims, float scale,
                 int causal, int window, int n_sink, attn_dtype_t dtype, void* stream);
}  // namespace
}  // namespace attn

int attn_prefill(const void* q, const void* k, const void* v, void* out, void* k_rot, float* lse, int B, int S,
                 int n_h, int n_kv, int D_h, float rope_base, float scale, int causal, attn_dtype_t dtype,
                 void* stream) {
  return prefill_impl(q, k, v, out, k_rot, lse, B, S, n_h, n_kv, D_h, D_h, rope_base, 0, D_h, scale, causal, 0, 0,
                      dtype, stream);
}

int attn_prefill_window(const void* q, const void* k, const void* v, void* out, void* k_rot, float* lse, int B,
                        int S, int n_h, int n_kv, int D_h, float rope_base, float scale, int window, int n_sink,
                        attn_dtype_t dtype, void* stream) {
  if (window <= 0 || n_sink < 0) return ATTN_ERR_ARG;
  return prefill_impl(q, k, v, out, k_rot, lse, B, S, n_h, n_kv, D_h, D_h, rope_base, 0, D_h, scale, 1, window,
                      n_sink, dtype, stream);
}

int attn_prefill_mla(const void* q, const void* k, const void* v, void* out, void* k_rot, float* lse, int B, int S,
                     int n_h, int n_kv, int D_qk, int D_v, float rope_base, int rope_offset, int rope_dims,
                     float scale, int causal, attn_dtype_t dtype, void* stream) {
  return prefill_impl(q, k, v, out, k_rot, lse, B, S, n_h, n_kv, D_qk, D_v, rope_base, rope_offset, rope_dims, scale,
                      causal, 0, 0, dtype, stream);
}

}  // extern "C"

namespace attn {
namespace {
int prefill_impl(const void* q, const void* k, const void* v, void* out, void* k_rot, float* lse, int B, int S,
                 int n_h, int n_kv, int D_qk, int D_v, float rope_base, int rope_offset, int rope_dims, float scale,
                 int causal, int window, int n_sink, attn_dtype_t dtype, void* stream) {
  if (!q || !k || !v || !out) return ATTN_ERR_ARG;
  if (B <= 0 || S <= 0 || n_h <= 0 || n_kv <= 0 || D_qk <= 0 || D_v <= 0 || n_h % n_kv) return ATTN_ERR_ARG;
  bool bf16 = false, half = false;
  if (!parse_dtype(dtype, &bf16, &half)) return ATTN_ERR_ARG;
  if (causal != 0 && causal != 1) return ATTN_ERR_ARG;
  const bool rope = rope_base > 0.f;
  const int unit = bf16 ? 8 : 2;  // vector width of the kernels' loads, in elements
  if (rope && (rope_offset < 0 || rope_dims <= 0 || rope_offset + rope_dims > D_qk)) return ATTN_ERR_ARG;
  if (D_qk > 256 || D_v > 256 || D_qk % unit || D_v % unit) return ATTN_ERR_UNSUPPORTED;
  if (rope && (rope_offset % unit || rope_dims % (half ? 2 * unit : unit))) return ATTN_ERR_UNSUPPORTED;
  if (rope && rope_dims / 2 > kMaxRopePairs) return ATTN_ERR_UNSUPPORTED;
  if (rope && !k_rot) return ATTN_ERR_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || (rope && !aligned16(k_rot)) ||
      (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)))
    return ATTN_ERR_ALIGN;
  const size_t esz = bf16 ? 2 : 4;
  const size_t k_bytes = static_cast<size_t>(B) * S * n_kv * D_qk * esz;
  if (rope && overlap(k_rot, k_bytes, k, k_bytes)) return ATTN_ERR_ARG;

  DeviceInfo dev;
  if (int rc = device_info(&dev)) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const float sc = scale > 0.f ? scale : 1.0f / sqrtf(static_cast<float>(D_qk));
  int launches = 0;
  cudaError_t e = cudaSuccess;
  const RopeFreq rf = make_rope(rope_base, rope ? rope_dims : 0, half);
  if (rope) {
    // rotated keys, written once: the form a KV cache stores
    RopeArgs ra{k_rot, k, B, S, n_kv, D_qk, rope_offset, rope_dims, 0, nullptr};
    e = launch_rope(ra, rf, bf16, st, &launches);
    if (e != cudaSuccess) return finish(e, launches);
  }
  PrefillArgs pa{q, rope ? k_rot : k, v, out, lse, B, S, n_h, n_kv, D_qk, sc * kLog2e, causal, dev.status,
                 g_wait_limit_ns.load(), S, 0, S, window, n_sink, D_v, rope ? rope_offset : 0};
  // Folded dealing (prefill_tc.cu) keeps the CTAs running at one time on few K/V
  // heads, at the price of a coarser last wave (double items of equal weight).
  // It needs every tile pair p to have a partner n_pairs - 1 - p of complementary
  // weight (whole causal prompts, an even number of pairs), and it pays when the
  // K/V of all heads is well beyond L2 - heaviest-first waves touch every head -
  // and there are several waves of double items.  Measured on prefill_tc.cu: the
  // MLA prefill shape (K/V 2.7x L2) gained 4%, the Llama-3-8B shape (1.1x L2) lost
  // 3%.  The CTA-pair kernel of the MLA shape deals heaviest-first only (folded, it
  // measured 1% slower).
  {
    const long long n_pairs = (S + 255) / 256;
    const long long kv_bytes = static_cast<long long>(B) * n_kv * S * (D_qk + D_v) * static_cast<long long>(esz);
    const long long n_double = static_cast<long long>(B) * n_h * n_pairs / 2;
    pa.fold = (causal && window == 0 && n_pairs % 2 == 0 && kv_bytes > 2LL * dev.l2_bytes &&
               n_double >= 4LL * dev.sms) ? 1 : 0;
  }
  // GQA: a work item takes one Q tile of two heads that read the same K/V head (prefill_tc.cu)
  pa.head_pairs = (n_h / n_kv) % 2 == 0 ? 1 : 0;
  if (prefill_pair_supported(D_qk, D_v, bf16, window)) {
    // the MLA prefill shape on CTA pairs: each CTA loads 64-key halves of the K tiles
    CUtensorMap maps[3];
    const unsigned long long hs = static_cast<unsigned long long>(D_qk) * 2;
    if (!make_bshd_map(&maps[0], q, B, S, n_h, D_qk) ||
        !make_map4(&maps[1], pa.k, D_qk, n_kv, S, B, hs, hs * n_kv, hs * n_kv * S, 64) ||
        !make_bshd_map(&maps[2], v, B, S, n_kv, D_v))
      return finish(cudaErrorInvalidValue, launches);
    e = launch_prefill_pair(pa, rf, maps, st, &launches);
  } else if (prefill_tc_supported(D_qk, D_v, bf16)) {
    CUtensorMap maps[3];
    if (!make_bshd_map(&maps[0], q, B, S, n_h, D_qk) || !make_bshd_map(&maps[1], pa.k, B, S, n_kv, D_qk) ||
        !make_bshd_map(&maps[2], v, B, S, n_kv, D_v))
      return finish(cudaErrorInvalidValue, launches);
    e = launch_prefill_tc(pa, rf, maps, dev.sms, st, &launches);
  } else {
    e = launch_prefill_simt(pa, rf, bf16, st, &launches);
  }
  return finish(e, launches);
}

}  // namespace
}  // namespace attn

extern "C" {

int attn_prefill_chunk(const void* q, const void* kcache, const void* vcache, void* out, float* lse, int B, int S_q,
                       int q_offset, int max_len, int n_h, int n_kv, int D_h, float rope_base, float scale,
                       int causal, attn_dtype_t dtype, void* stream) {
  if (!q || !kcache || !vcache || !out) return ATTN_ERR_ARG;
  if (B <= 0 || S_q <= 0 || n_h <= 0 || n_kv <= 0 || D_h <= 0 || n_h % n_kv) return ATTN_ERR_ARG;
  if (q_offset < 0 || max_len <= 0 || static_cast<long long>(q_offset) + S_q > max_len) return ATTN_ERR_ARG;
  bool bf16 = false, half = false;
  if (!parse_dtype(dtype, &bf16, &half)) return ATTN_ERR_ARG;
  if (causal != 0 && causal != 1) return ATTN_ERR_ARG;
  if (D_h > 256 || D_h % ((bf16 ? 8 : 2) * (rope_base > 0.f && half ? 2 : 1))) return ATTN_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(kcache) || !aligned16(vcache) || !aligned16(out) ||
      (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)))
    return ATTN_ERR_ALIGN;
  DeviceInfo dev;
  if (int rc = device_info(&dev)) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const float sc = scale > 0.f ? scale : 1.0f / sqrtf(static_cast<float>(D_h));
  const int S_k = q_offset + S_q;
  PrefillArgs pa{q, kcache, vcache, out, lse, B, S_q, n_h, n_kv, D_h, sc * kLog2e, causal, dev.status,
                 g_wait_limit_ns.load(), S_k, q_offset, max_len, 0, 0, D_h, 0};
  pa.head_pairs = (n_h / n_kv) % 2 == 0 ? 1 : 0;  // GQA: one Q tile of two heads per work item
  const RopeFreq rf = make_rope(rope_base, D_h, half);
  int launches = 0;
  cudaError_t e;
  if (prefill_tc_supported(D_h, D_h, bf16)) {
    // K/V maps cover only the S_k visible rows of each sequence: rows past them read as zero
    CUtensorMap maps[3];
    const unsigned long long hs = static_cast<unsigned long long>(D_h) * 2;
    if (!make_bshd_map(&maps[0], q, B, S_q, n_h, D_h) ||
        !make_map4(&maps[1], kcache, D_h, n_kv, S_k, B, hs, hs * n_kv, hs * n_kv * max_len, 128) ||
        !make_map4(&maps[2], vcache, D_h, n_kv, S_k, B, hs, hs * n_kv, hs * n_kv * max_len, 128))
      return finish(cudaErrorInvalidValue, launches);
    e = launch_prefill_tc(pa, rf, maps, dev.sms, st, &launches);
  } else {
    e = launch_prefill_simt(pa, rf, bf16, st, &launches);
  }
  return finish(e, launches);
}

int attn_kv_append(const void* k_new, const void* v_new, void* kcache, void* vcache, int v_token_stride,
                   const int* start, int B, int C, int n_kv, int D_qk, int D_v, int max_len, float rope_base,
                   int rope_offset, int rope_dims, attn_dtype_t dtype, void* stream) {
  if (!k_new || !kcache || !start || (v_new && !vcache)) return ATTN_ERR_ARG;
  if (B <= 0 || C <= 0 || n_kv <= 0 || D_qk <= 0 || D_v <= 0 || max_len <= 0 || v_token_stride < 0)
    return ATTN_ERR_ARG;
  bool bf16 = false, half = false;
  if (!parse_dtype(dtype, &bf16, &half)) return ATTN_ERR_ARG;
  if (D_qk % 8 || D_v % 8) return ATTN_ERR_ARG;
  const bool rope = rope_base > 0.f;
  if (rope && (rope_offset < 0 || rope_dims <= 0 || rope_offset % 8 || rope_dims % (half ? 16 : 8) ||
               rope_offset + rope_dims > D_qk))
    return ATTN_ERR_ARG;
  if (rope && rope_dims / 2 > kMaxRopePairs) return ATTN_ERR_UNSUPPORTED;
  const long long ldv = v_token_stride ? v_token_stride : static_cast<long long>(n_kv) * D_v;
  if (!aligned16(k_new) || !aligned16(kcache) || (v_new && (!aligned16(v_new) || !aligned16(vcache))) ||
      (reinterpret_cast<uintptr_t>(start) & 3u))
    return ATTN_ERR_ALIGN;
  KvAppendArgs ka{k_new, v_new, kcache, vcache, ldv, start, B, C, n_kv, D_qk, D_v, max_len, rope ? rope_offset : 0};
  int launches = 0;
  const cudaError_t e = launch_kv_append(ka, make_rope(rope_base, rope ? rope_dims : 0, half), bf16,
                                         static_cast<cudaStream_t>(stream), &launches);
  return finish(e, launches);
}

size_t attn_decode_workspace_size(int B, int n_h, int n_kv, int D_qk, int D_v, int max_len, attn_dtype_t dtype) {
  if (B <= 0 || n_h <= 0 || n_kv <= 0 || n_h % n_kv || D_qk <= 0 || D_v <= 0 || max_len <= 0) return static_cast<size_t>(-1);
  bool bf16 = false, half = false;
  if (!parse_dtype(dtype, &bf16, &half)) return static_cast<size_t>(-1);
  int chunk = 0;
  const int ns = decode_plan_splits(B, n_h, n_kv, D_qk, D_v, max_len, &chunk);
  size_t slots = static_cast<size_t>(B) * n_h * ns;
  if (mla_shape(B, n_h, n_kv, D_qk, D_v, bf16)) {
    // one partial per (pair, sequence) piece: at most pairs + B - 1 of them
    const size_t mla_slots = static_cast<size_t>(kMlaMaxPairs + B) * n_h;
    if (mla_slots > slots) slots = mla_slots;
  }
  const size_t o_bytes = (slots * D_v * sizeof(float) + 255) & ~size_t(255);
  return o_bytes + ((slots * sizeof(float) + 255) & ~size_t(255)) + 256;  // + scheduler counters
}

namespace attn {
namespace {
int decode_impl(const void* q, const void* kcache, const void* vcache, int v_token_stride, const int* seqlens,
                void* out, float* lse, int B, int n_h, int n_kv, int D_qk, int D_v, int max_len, float rope_base,
                int rope_offset, int rope_dims, float scale, int window, int n_sink, attn_dtype_t dtype,
                void* workspace, size_t workspace_bytes, void* stream);
}  // namespace
}  // namespace attn

int attn_decode(const void* q, const void* kcache, const void* vcache, int v_token_stride, const int* seqlens,
                void* out, float* lse, int B, int n_h, int n_kv, int D_qk, int D_v, int max_len, float rope_base,
                int rope_offset, int rope_dims, float scale, attn_dtype_t dtype, void* workspace,
                size_t workspace_bytes, void* stream) {
  return decode_impl(q, kcache, vcache, v_token_stride, seqlens, out, lse, B, n_h, n_kv, D_qk, D_v, max_len,
                     rope_base, rope_offset, rope_dims, scale, 0, 0, dtype, workspace, workspace_bytes, stream);
}

int attn_decode_window(const void* q, const void* kcache, const void* vcache, int v_token_stride, const int* seqlens,
                       void* out, float* lse, int B, int n_h, int n_kv, int D_qk, int D_v, int max_len,
                       float rope_base, int rope_offset, int rope_dims, float scale, int window, int n_sink,
                       attn_dtype_t dtype, void* workspace, size_t workspace_bytes, void* stream) {
  if (window <= 0 || n_sink < 0) return ATTN_ERR_ARG;
  return decode_impl(q, kcache, vcache, v_token_stride, seqlens, out, lse, B, n_h, n_kv, D_qk, D_v, max_len,
                     rope_base, rope_offset, rope_dims, scale, window, n_sink, dtype, workspace, workspace_bytes,
                     stream);
}

}  // extern "C"

namespace attn {
namespace {
int decode_impl(const void* q, const void* kcache, const void* vcache, int v_token_stride, const int* seqlens,
                void* out, float* lse, int B, int n_h, int n_kv, int D_qk, int D_v, int max_len, float rope_base,
                int rope_offset, int rope_dims, float scale, int window, int n_sink, attn_dtype_t dtype,
                void* workspace, size_t workspace_bytes, void* stream) {
  if (!q || !kcache || !vcache || !seqlens || !out || !workspace) return ATTN_ERR_ARG;
  if (B <= 0 || n_h <= 0 || n_kv <= 0 || n_h % n_kv || D_qk <= 0 || D_v <= 0 || max_len <= 0) return ATTN_ERR_ARG;
  bool bf16 = false, half = false;
  if (!parse_dtype(dtype, &bf16, &half)) return ATTN_ERR_ARG;
  if (v_token_stride < 0) return ATTN_ERR_ARG;
  const long long ldv = v_token_stride ? v_token_stride : static_cast<long long>(n_kv) * D_v;
  if (ldv < static_cast<long long>(n_kv) * D_v && vcache != kcache) return ATTN_ERR_ARG;
  if (D_qk % 8 || D_v % 8 || ldv % 8) return ATTN_ERR_UNSUPPORTED;
  if (D_qk > 640 || D_v > 512) return ATTN_ERR_UNSUPPORTED;
  const bool rope = rope_base > 0.f;
  if (rope && (rope_offset < 0 || rope_dims <= 0 || rope_dims % 2 || rope_offset % 2 ||
               rope_offset + rope_dims > D_qk))
    return ATTN_ERR_ARG;
  if (rope && rope_dims / 2 > kMaxRopePairs) return ATTN_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(kcache) || !aligned16(vcache) || !aligned16(out) || !aligned16(workspace) ||
      (reinterpret_cast<uintptr_t>(seqlens) & 3u) || (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)))
    return ATTN_ERR_ALIGN;
  const size_t need = attn_decode_workspace_size(B, n_h, n_kv, D_qk, D_v, max_len, dtype);
  if (workspace_bytes < need) return ATTN_ERR_WORKSPACE;

  DeviceInfo dev;
  if (int rc = device_info(&dev)) return rc;
  int chunk = 0;
  int ns = decode_plan_splits(B, n_h, n_kv, D_qk, D_v, max_len, &chunk);
  size_t slots = static_cast<size_t>(B) * n_h * ns;
  if (mla_shape(B, n_h, n_kv, D_qk, D_v, bf16)) {
    const size_t mla_slots = static_cast<size_t>(kMlaMaxPairs + B) * n_h;
    if (mla_slots > slots) slots = mla_slots;
  }
  float* ws_o = static_cast<float*>(workspace);
  float* ws_lse = reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                           ((slots * D_v * sizeof(float) + 255) & ~size_t(255)));
  unsigned int* ws_ctr = reinterpret_cast<unsigned int*>(reinterpret_cast<char*>(ws_lse) +
                                                         ((slots * sizeof(float) + 255) & ~size_t(255)));
  // the tensor-core and streaming kernels rotate whole 8-dim chunks of the query
  const bool chunked_rope = !rope || (rope_offset % 8 == 0 && rope_dims % (half ? 16 : 8) == 0);
  const bool use_mla = window == 0 && mla_shape(B, n_h, n_kv, D_qk, D_v, bf16) &&
                       decode_mla_supported(B, n_h, n_kv, D_qk, D_v, ldv, vcache == kcache, bf16) &&
                       chunked_rope && (!rope || decode_mla_rope_ok(rope_offset, rope_dims, half));
  if (use_mla) {
    ns = decode_mla_pairs(dev.sms);  // the kernel runs 2 CTAs per pair
    chunk = 0;
  }
  const float sc = scale > 0.f ? scale : 1.0f / sqrtf(static_cast<float>(D_qk));
  DecodeArgs da{q, kcache, vcache, ldv, seqlens, out, lse, B, n_h, n_kv, D_qk, D_v, max_len,
                rope ? rope_offset : 0, sc * kLog2e, ws_o, ws_lse, ns, chunk, dev.status, g_wait_limit_ns.load(),
                window, n_sink, ws_ctr};
  int launches = 0;
  const RopeFreq rf = make_rope(rope_base, rope ? rope_dims : 0, half);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (use_mla) {
    CUtensorMap maps[2];
    const unsigned long long row = static_cast<unsigned long long>(D_qk) * 2;
    if (!make_map3(&maps[0], q, D_qk, n_h, B, row, row * n_h, 64) ||
        !make_map3(&maps[1], kcache, D_qk, max_len, B, row, row * max_len, kMlaTileKeys))
      return finish(cudaErrorInvalidValue, launches);
    e = launch_decode_mla(da, rf, maps, st, &launches);
  } else if (decode_tc_supported(n_h, n_kv, D_qk, D_v, bf16, rope_offset, rope_dims, rope)) {
    // K and V tiles of 128 keys on the tensor cores (keys on M, the head group on N)
    CUtensorMap maps[2];
    const unsigned long long ks = static_cast<unsigned long long>(D_qk) * 2;
    const unsigned long long vs = static_cast<unsigned long long>(ldv) * 2;
    if (!make_map4(&maps[0], kcache, D_qk, n_kv, max_len, B, ks, ks * n_kv, ks * n_kv * max_len, kStreamTileKeys) ||
        !make_map4(&maps[1], vcache, D_v, n_kv, max_len, B, static_cast<unsigned long long>(D_v) * 2, vs,
                   vs * max_len, kStreamTileKeys))
      return finish(cudaErrorInvalidValue, launches);
    // fewer, longer chunks than the generic plan: each chunk pays a query load, a
    // pipeline fill and an epilogue (never more splits than the workspace holds)
    DecodeArgs dt = da;
    while (dt.chunk < kDecodeTcMinChunk && dt.chunk < max_len) dt.chunk *= 2;
    dt.n_split = (max_len + dt.chunk - 1) / dt.chunk;
    e = launch_decode_tc(dt, rf, maps, dev.sms, st, &launches);
  } else if (window == 0 && chunked_rope && decode_stream_supported(n_h, n_kv, D_qk, D_v, bf16)) {
    // K and V stream through shared memory in 64-key tiles
    CUtensorMap maps[2];
    const unsigned long long ks = static_cast<unsigned long long>(D_qk) * 2;
    const unsigned long long vs = static_cast<unsigned long long>(ldv) * 2;
    if (!make_map4(&maps[0], kcache, D_qk, n_kv, max_len, B, ks, ks * n_kv, ks * n_kv * max_len, kStreamTileKeys) ||
        !make_map4(&maps[1], vcache, D_v, n_kv, max_len, B, static_cast<unsigned long long>(D_v) * 2, vs,
                   vs * max_len, kStreamTileKeys))
      return finish(cudaErrorInvalidValue, launches);
    e = launch_decode_stream(da, rf, maps, dev.sms, st, &launches);
  } else {
    e = launch_decode(da, rf, bf16, st, &launches);
  }
  return finish(e, launches);
}

}  // namespace
}  // namespace attn

extern "C" {

// ---------------------------------------------------------------------------
// Decode with library-owned scratch, for callers that cannot allocate.
// ---------------------------------------------------------------------------
}  // extern "C"

namespace attn {
namespace {

// File-scope scratch of attn_decode_static: one per device that loads the
// library, shared by every call on that device.  In host code the name is only
// a stand-in; the device address comes from cudaGetSymbolAddress below.
__device__ __align__(256) unsigned char g_decode_scratch[ATTN_DECODE_STATIC_SCRATCH_BYTES];

void* g_scratch_addr[kMaxDevices];
std::mutex g_scratch_mu;

// Device address of g_decode_scratch on the current device, looked up once per
// device with that device current.
int static_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || p == nullptr) return ATTN_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return ATTN_OK;
}

}  // namespace
}  // namespace attn

extern "C" {

int attn_decode_static(const void* q, const void* kcache, const void* vcache, int v_token_stride, const int* seqlens,
                       void* out, float* lse, int B, int n_h, int n_kv, int D_qk, int D_v, int max_len,
                       float rope_base, int rope_offset, int rope_dims, float scale, attn_dtype_t dtype,
                       void* stream) {
  const size_t need = attn_decode_workspace_size(B, n_h, n_kv, D_qk, D_v, max_len, dtype);
  if (need == static_cast<size_t>(-1)) return ATTN_ERR_ARG;
  if (need > ATTN_DECODE_STATIC_SCRATCH_BYTES) return ATTN_ERR_WORKSPACE;
  void* scratch = nullptr;
  if (int rc = static_scratch(&scratch)) return rc;
  return attn_decode(q, kcache, vcache, v_token_stride, seqlens, out, lse, B, n_h, n_kv, D_qk, D_v, max_len,
                     rope_base, rope_offset, rope_dims, scale, dtype, scratch, ATTN_DECODE_STATIC_SCRATCH_BYTES,
                     stream);
}

int attn_device_status(void* stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return ATTN_ERR_CUDA;
  DeviceInfo dev;
  if (int rc = device_info(&dev)) return rc;
  unsigned int s = 0;
  if (cudaMemcpy(&s, dev.status, sizeof(s), cudaMemcpyDeviceToHost) != cudaSuccess) return ATTN_ERR_CUDA;
  if (s == 0) return ATTN_OK;
  const unsigned int zero = 0;
  if (cudaMemcpy(dev.status, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) return ATTN_ERR_CUDA;
  return (s & STATUS_TIMEOUT) ? ATTN_ERR_TIMEOUT : ATTN_ERR_CUDA;
}

int attn_check_wait_timeout(void* stream) {
  DeviceInfo dev;
  if (int rc = device_info(&dev)) return rc;
  wait_timeout_check_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(dev.status, g_wait_limit_ns.load());
  return finish(cudaGetLastError(), 1);
}

unsigned long long attn_launch_count(void) { return g_launches.load(); }

void attn_set_wait_limit_ns(unsigned long long ns) { g_wait_limit_ns.store(ns ? ns : 1ull); }

}  // extern "C"

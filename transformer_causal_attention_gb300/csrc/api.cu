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

// 4-D tensor map over a BSHD bf16 tensor [B, S, heads, D]: boxes of
// 64 head-dims x 1 head x 128 positions x 1 batch, 128-byte swizzle (the
// canonical K-major layout of the tensor-core operands), zero fill outside.
bool make_bshd_map(CUtensorMap* map, const void* base, int B, int S, int heads, int D) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(heads),
                              static_cast<cuuint64_t>(S), static_cast<cuuint64_t>(B)};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(heads) * D * 2,
                                 static_cast<cuuint64_t>(S) * heads * D * 2};
  const cuuint32_t box[4] = {64, 1, 128, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// theta_i = base^(-2i/dims) expressed in turns per position, split hi + lo.
RopeFreq make_rope(float base, int dims) {
  RopeFreq f;
  memset(&f, 0, sizeof(f));
  if (!(base > 0.f) || dims <= 0) return f;
  f.n_pairs = dims / 2;
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

int attn_rope(void* x_out, const void* x_in, int B, int S, int n_heads, int D, int rope_offset, int rope_dims,
              float rope_base, int pos_offset, attn_dtype_t dtype, void* stream) {
  if (!x_out || !x_in || B <= 0 || S <= 0 || n_heads <= 0 || D <= 0) return ATTN_ERR_ARG;
  if (dtype != ATTN_F32 && dtype != ATTN_BF16) return ATTN_ERR_ARG;
  if (!(rope_base > 0.f) || rope_offset < 0 || rope_dims <= 0 || rope_offset + rope_dims > D || pos_offset < 0)
    return ATTN_ERR_ARG;
  const int unit = dtype == ATTN_BF16 ? 8 : 2;
  if (D % unit || rope_offset % unit || rope_dims % unit) return ATTN_ERR_ARG;
  if (rope_dims / 2 > kMaxRopePairs) return ATTN_ERR_UNSUPPORTED;
  if (!aligned16(x_out) || !aligned16(x_in)) return ATTN_ERR_ALIGN;
  const size_t bytes = static_cast<size_t>(B) * S * n_heads * D * (dtype == ATTN_BF16 ? 2 : 4);
  if (x_out != x_in && overlap(x_out, bytes, x_in, bytes)) return ATTN_ERR_ARG;
  RopeArgs ra{x_out, x_in, B, S, n_heads, D, rope_offset, rope_dims, pos_offset};
  int launches = 0;
  const cudaError_t e =
      launch_rope(ra, make_rope(rope_base, rope_dims), dtype == ATTN_BF16, static_cast<cudaStream_t>(stream), &launches);
  return finish(e, launches);
}

int attn_prefill(const void* q, const void* k, const void* v, void* out, void* k_rot, float* lse, int B, int S,
                 int n_h, int n_kv, int D_h, float rope_base, float scale, int causal, attn_dtype_t dtype,
                 void* stream) {
  if (!q || !k || !v || !out) return ATTN_ERR_ARG;
  if (B <= 0 || S <= 0 || n_h <= 0 || n_kv <= 0 || D_h <= 0 || n_h % n_kv) return ATTN_ERR_ARG;
  if (dtype != ATTN_F32 && dtype != ATTN_BF16) return ATTN_ERR_ARG;
  if (causal != 0 && causal != 1) return ATTN_ERR_ARG;
  const bool bf16 = dtype == ATTN_BF16;
  if (D_h > 256 || D_h % (bf16 ? 8 : 2)) return ATTN_ERR_UNSUPPORTED;
  const bool rope = rope_base > 0.f;
  if (rope && !k_rot) return ATTN_ERR_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || (rope && !aligned16(k_rot)) ||
      (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)))
    return ATTN_ERR_ALIGN;
  const size_t esz = bf16 ? 2 : 4;
  const size_t kv_bytes = static_cast<size_t>(B) * S * n_kv * D_h * esz;
  if (rope && overlap(k_rot, kv_bytes, k, kv_bytes)) return ATTN_ERR_ARG;

  DeviceInfo dev;
  if (int rc = device_info(&dev)) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const float sc = scale > 0.f ? scale : 1.0f / sqrtf(static_cast<float>(D_h));
  int launches = 0;
  cudaError_t e = cudaSuccess;
  const RopeFreq rf = make_rope(rope_base, D_h);
  if (rope) {
    RopeArgs ra{k_rot, k, B, S, n_kv, D_h, 0, D_h, 0};
    e = launch_rope(ra, rf, bf16, st, &launches);
    if (e != cudaSuccess) return finish(e, launches);
  }
  PrefillArgs pa{q, rope ? k_rot : k, v, out, lse, B, S, n_h, n_kv, D_h, sc * kLog2e, causal, dev.status,
                 g_wait_limit_ns.load()};
  if (prefill_tc_supported(D_h, bf16)) {
    CUtensorMap maps[3];
    if (!make_bshd_map(&maps[0], q, B, S, n_h, D_h) || !make_bshd_map(&maps[1], pa.k, B, S, n_kv, D_h) ||
        !make_bshd_map(&maps[2], v, B, S, n_kv, D_h))
      return finish(cudaErrorInvalidValue, launches);
    e = launch_prefill_tc(pa, rf, maps, dev.sms, st, &launches);
  } else {
    e = launch_prefill_simt(pa, rf, bf16, st, &launches);
  }
  return finish(e, launches);
}

size_t attn_decode_workspace_size(int B, int n_h, int n_kv, int D_qk, int D_v, int max_len, attn_dtype_t dtype) {
  if (B <= 0 || n_h <= 0 || n_kv <= 0 || n_h % n_kv || D_qk <= 0 || D_v <= 0 || max_len <= 0) return static_cast<size_t>(-1);
  if (dtype != ATTN_F32 && dtype != ATTN_BF16) return static_cast<size_t>(-1);
  int chunk = 0;
  const int ns = decode_plan_splits(B, n_h, n_kv, D_qk, D_v, max_len, &chunk);
  const size_t slots = static_cast<size_t>(B) * n_h * ns;
  const size_t o_bytes = (slots * D_v * sizeof(float) + 255) & ~size_t(255);
  return o_bytes + ((slots * sizeof(float) + 255) & ~size_t(255));
}

int attn_decode(const void* q, const void* kcache, const void* vcache, int v_token_stride, const int* seqlens,
                void* out, float* lse, int B, int n_h, int n_kv, int D_qk, int D_v, int max_len, float rope_base,
                int rope_offset, int rope_dims, float scale, attn_dtype_t dtype, void* workspace,
                size_t workspace_bytes, void* stream) {
  if (!q || !kcache || !vcache || !seqlens || !out || !workspace) return ATTN_ERR_ARG;
  if (B <= 0 || n_h <= 0 || n_kv <= 0 || n_h % n_kv || D_qk <= 0 || D_v <= 0 || max_len <= 0) return ATTN_ERR_ARG;
  if (dtype != ATTN_F32 && dtype != ATTN_BF16) return ATTN_ERR_ARG;
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
  const int ns = decode_plan_splits(B, n_h, n_kv, D_qk, D_v, max_len, &chunk);
  const size_t slots = static_cast<size_t>(B) * n_h * ns;
  float* ws_o = static_cast<float*>(workspace);
  float* ws_lse = reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                           ((slots * D_v * sizeof(float) + 255) & ~size_t(255)));
  const float sc = scale > 0.f ? scale : 1.0f / sqrtf(static_cast<float>(D_qk));
  DecodeArgs da{q, kcache, vcache, ldv, seqlens, out, lse, B, n_h, n_kv, D_qk, D_v, max_len,
                rope ? rope_offset : 0, sc * kLog2e, ws_o, ws_lse, ns, chunk, dev.status, g_wait_limit_ns.load()};
  int launches = 0;
  const cudaError_t e = launch_decode(da, make_rope(rope_base, rope ? rope_dims : 0), dtype == ATTN_BF16,
                                      static_cast<cudaStream_t>(stream), &launches);
  return finish(e, launches);
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

unsigned long long attn_launch_count(void) { return g_launches.load(); }

void attn_set_wait_limit_ns(unsigned long long ns) { g_wait_limit_ns.store(ns ? ns : 1ull); }

}  // extern "C"

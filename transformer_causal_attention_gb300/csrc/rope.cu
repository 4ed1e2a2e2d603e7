// rope.cu - standalone rotary position embedding of [B, S, n_heads, D] rows.
//
// Rotates the pairs of the span [rope_offset, rope_offset + rope_dims) by
// pos * theta_i ("Transformer架构从Attention到DecoderBlock" §8.3): pairs
// (2i, 2i+1), or (j, j + rope_dims/2) in the split-halves layout.  This is the
// pass that writes rotated keys (the KV-cache form, "Transformer架构完全深度解析"
// §7) before the prefill kernel reads them.
//
// A row sits at position pos_offset + s (s = its index in the sequence), or at
// positions[b * S + s] when the caller gives a position per row (tokens whose
// absolute slots are not consecutive, e.g. a batch of requests at different
// depths, "Transformer架构完全深度解析" §7: each cached key carries its own
// absolute position).
//
// One thread owns a chunk of CH consecutive dims of one token for ALL heads, so
// the sin/cos of its pairs are computed once and reused n_heads times.  In the
// split-halves layout the thread owning a chunk of the first half also owns the
// chunk rope_dims/2 later, which holds the other member of each of its pairs.
// The kernel is bound by HBM bandwidth (read + write once).
#include "kernels.h"

namespace attn {
namespace {

template <typename T, int CH>
__device__ __forceinline__ void load_chunk(const T* p, float* x) {
  if constexpr (sizeof(T) == 2 && CH == 8) {
    bf16x8_to_f32(*reinterpret_cast<const uint4*>(p), x);
  } else {
#pragma unroll
    for (int e = 0; e < CH; ++e) x[e] = to_f32(p[e]);
  }
}

template <typename T, int CH>
__device__ __forceinline__ void store_chunk(T* p, const float* x) {
  if constexpr (sizeof(T) == 2 && CH == 8) {
    *reinterpret_cast<uint4*>(p) = f32_to_bf16x8(x);
  } else {
#pragma unroll
    for (int e = 0; e < CH; ++e) p[e] = from_f32<T>(x[e]);
  }
}

// Rotate n_rows rows (stride `stride` elements) of the chunk at span-relative
// dim `rel` from src to dst at position pos.  The caller skips chunks of the
// second half in the split-halves layout (their owner is rel - n_pairs).
// The frequencies of the rotation (hi and lo words, n_pairs each) sit in shared memory: every
// thread reads those of its own chunk, and lanes with different chunks read different words,
// which a kernel-parameter array would serve one address at a time.
struct SmemFreq {
  const float* hi;
  const float* lo;
  int n_pairs;
  bool half;
};
__device__ __forceinline__ SmemFreq stage_freq(const RopeFreq& f, float* buf) {
  for (int i = threadIdx.x; i < f.n_pairs; i += blockDim.x) {
    buf[i] = f.hi[i];
    buf[kMaxRopePairs + i] = f.lo[i];
  }
  __syncthreads();
  return SmemFreq{buf, buf + kMaxRopePairs, f.n_pairs, f.half != 0};
}

template <typename T, int CH>
__device__ __forceinline__ void rotate_chunk_rows(const T* src, T* dst, long long stride, int n_rows, int rel, int pos,
                                                  const SmemFreq& f) {
  if (f.half) {
    float sn[CH], cs[CH];
#pragma unroll
    for (int e = 0; e < CH; ++e) rope_sincos(pos, f.hi[rel + e], f.lo[rel + e], &sn[e], &cs[e]);
    for (int h = 0; h < n_rows; ++h) {
      float x0[CH], x1[CH];
      load_chunk<T, CH>(src + h * stride, x0);
      load_chunk<T, CH>(src + h * stride + f.n_pairs, x1);
#pragma unroll
      for (int e = 0; e < CH; ++e) rotate_pair(x0[e], x1[e], sn[e], cs[e]);
      store_chunk<T, CH>(dst + h * stride, x0);
      store_chunk<T, CH>(dst + h * stride + f.n_pairs, x1);
    }
  } else {
    float sn[CH / 2], cs[CH / 2];
#pragma unroll
    for (int p = 0; p < CH / 2; ++p) rope_sincos(pos, f.hi[rel / 2 + p], f.lo[rel / 2 + p], &sn[p], &cs[p]);
    for (int h = 0; h < n_rows; ++h) {
      float x[CH];
      load_chunk<T, CH>(src + h * stride, x);
#pragma unroll
      for (int p = 0; p < CH / 2; ++p) rotate_pair(x[2 * p], x[2 * p + 1], sn[p], cs[p]);
      store_chunk<T, CH>(dst + h * stride, x);
    }
  }
}

// Rows whose chunks one thread loads before it stores any of them, so that its loads are in
// flight together (a chunk is 16 bytes of bf16; kept as loaded until its row is rotated).
constexpr int kRowBatch = 8;

// bf16, adjacent pairs: the 8-dim chunk at src of n_rows rows stride elements apart, rotated by
// the angles of pairs rel / 2 .. rel / 2 + 3 at position pos, to dst.  In place (dst == src) is
// fine: each row is stored after its own load.
__device__ __forceinline__ void rotate_rows_bf16(const __nv_bfloat16* src, __nv_bfloat16* dst, long long stride,
                                                 int n_rows, int rel, int pos, const SmemFreq& f) {
  float sn[4], cs[4];
#pragma unroll
  for (int p = 0; p < 4; ++p) rope_sincos(pos, f.hi[rel / 2 + p], f.lo[rel / 2 + p], &sn[p], &cs[p]);
  for (int hb = 0; hb < n_rows; hb += kRowBatch) {
    uint4 raw[kRowBatch];
#pragma unroll
    for (int e = 0; e < kRowBatch; ++e)
      if (hb + e < n_rows) raw[e] = *reinterpret_cast<const uint4*>(src + (hb + e) * stride);
#pragma unroll
    for (int e = 0; e < kRowBatch; ++e)
      if (hb + e < n_rows) {
        float x[8];
        bf16x8_to_f32(raw[e], x);
#pragma unroll
        for (int p = 0; p < 4; ++p) rotate_pair(x[2 * p], x[2 * p + 1], sn[p], cs[p]);
        *reinterpret_cast<uint4*>(dst + (hb + e) * stride) = f32_to_bf16x8(x);
      }
  }
}

// bf16: the 8-dim chunk at src of n_rows rows copied to dst as it is, loads batched as above.
__device__ __forceinline__ void copy_rows_bf16(const __nv_bfloat16* src, __nv_bfloat16* dst, long long stride,
                                               int n_rows) {
  for (int hb = 0; hb < n_rows; hb += kRowBatch) {
    uint4 raw[kRowBatch];
#pragma unroll
    for (int e = 0; e < kRowBatch; ++e)
      if (hb + e < n_rows) raw[e] = *reinterpret_cast<const uint4*>(src + (hb + e) * stride);
#pragma unroll
    for (int e = 0; e < kRowBatch; ++e)
      if (hb + e < n_rows) *reinterpret_cast<uint4*>(dst + (hb + e) * stride) = raw[e];
  }
}

template <typename T, int CH>
__global__ void __launch_bounds__(256) rope_kernel(RopeArgs a, RopeFreq rf) {
  __shared__ float freq[2 * kMaxRopePairs];
  const SmemFreq f = stage_freq(rf, freq);
  const int chunks = a.D / CH;
  const long long total = static_cast<long long>(a.B) * a.S * chunks;
  const T* in = static_cast<const T*>(a.in);
  T* out = static_cast<T*>(a.out);
  for (long long idx = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; idx < total;
       idx += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int c = static_cast<int>(idx % chunks);
    const long long tok = idx / chunks;  // b * S + s
    const int s = static_cast<int>(tok % a.S);
    const int d0 = c * CH;
    const int rel = d0 - a.rope_offset;
    const long long off = tok * a.n_heads * a.D + d0;
    if (rel >= 0 && rel < a.rope_dims) {
      if (f.half && rel >= f.n_pairs) continue;  // rotated by the owner of its partner chunk
      const int pos = a.positions ? a.positions[tok] : a.pos_offset + s;
      if constexpr (sizeof(T) == 2 && CH == 8) {
        if (!f.half) {
          rotate_rows_bf16(in + off, out + off, a.D, a.n_heads, rel, pos, f);
          continue;
        }
      }
      rotate_chunk_rows<T, CH>(in + off, out + off, a.D, a.n_heads, rel, pos, f);
    } else if (in != out) {
      if constexpr (sizeof(T) == 2 && CH == 8) {
        copy_rows_bf16(in + off, out + off, a.D, a.n_heads);
      } else {
        for (int h = 0; h < a.n_heads; ++h) {
          float x[CH];
          load_chunk<T, CH>(in + off + h * a.D, x);
          store_chunk<T, CH>(out + off + h * a.D, x);
        }
      }
    }
  }
}

// One thread per (sequence b, new token c, 8-dim chunk): the new key row is
// rotated at its absolute position start[b] + c and written to that cache
// slot for every KV head, the value row is copied next to it (bf16: the heads'
// chunks in batches of kRowBatch loads before their stores).
//
// A decode step appends one token per sequence: too few (token, chunk) items to keep
// the GPU's loads in flight when each thread walks all heads one after another, so the
// launcher then gives every head its own thread (head_groups = n_kv; each thread computes
// its own sin/cos), and otherwise one thread per (token, chunk) for all heads.
template <typename T>
__global__ void __launch_bounds__(256) kv_append_kernel(KvAppendArgs a, RopeFreq rf) {
  __shared__ float freq[2 * kMaxRopePairs];
  const SmemFreq f = stage_freq(rf, freq);
  const int kch = a.D_qk / 8, vch = a.v_new ? a.D_v / 8 : 0;
  const int per_tok = kch + vch;
  const int hg = a.head_groups, hpt = a.n_kv / hg;  // heads per thread
  const long long total = static_cast<long long>(a.B) * a.C * per_tok * hg;
  for (long long idx = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; idx < total;
       idx += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int ch = static_cast<int>(idx % per_tok);
    const long long r = idx / per_tok;
    const int h0 = static_cast<int>(r % hg) * hpt;
    const long long bc = r / hg;
    const int c = static_cast<int>(bc % a.C);
    const int b = static_cast<int>(bc / a.C);
    const int pos = a.start[b] + c;
    if (pos < 0 || pos >= a.max_len) continue;  // slots outside the cache are never written
    const long long slot = static_cast<long long>(b) * a.max_len + pos;
    if (ch < kch) {
      const int d0 = ch * 8;
      const int rel = d0 - a.rope_offset;
      const T* src = static_cast<const T*>(a.k_new) + (bc * a.n_kv + h0) * a.D_qk + d0;
      T* dst = static_cast<T*>(a.kcache) + (slot * a.n_kv + h0) * a.D_qk + d0;
      if (rel >= 0 && rel < 2 * f.n_pairs) {
        if (f.half && rel >= f.n_pairs) continue;  // written with its partner chunk
        if constexpr (sizeof(T) == 2) {
          if (!f.half) {
            rotate_rows_bf16(src, dst, a.D_qk, hpt, rel, pos, f);
            continue;
          }
        }
        rotate_chunk_rows<T, 8>(src, dst, a.D_qk, hpt, rel, pos, f);
      } else {
        for (int h = 0; h < hpt; ++h) {
          float x[8];
          load_chunk<T, 8>(src + h * a.D_qk, x);
          store_chunk<T, 8>(dst + h * a.D_qk, x);
        }
      }
    } else {
      const int d0 = (ch - kch) * 8;
      const T* src = static_cast<const T*>(a.v_new) + (bc * a.n_kv + h0) * a.D_v + d0;
      T* dst = static_cast<T*>(a.vcache) + slot * a.v_token_stride + h0 * a.D_v + d0;
      if (a.v_token_stride % 8 == 0) {  // every value chunk starts on a 16-byte boundary: copy whole chunks
        if constexpr (sizeof(T) == 2) {  // 16-byte chunks as they are
          copy_rows_bf16(src, dst, a.D_v, hpt);
        } else {
          for (int h = 0; h < hpt; ++h) {
            float x[8];
            load_chunk<T, 8>(src + h * a.D_v, x);
            store_chunk<T, 8>(dst + h * a.D_v, x);
          }
        }
      } else {
        for (int h = 0; h < hpt; ++h)
#pragma unroll
          for (int e = 0; e < 8; ++e) dst[h * a.D_v + e] = src[h * a.D_v + e];
      }
    }
  }
}

}  // namespace

cudaError_t launch_kv_append(const KvAppendArgs& args, const RopeFreq& rope, bool bf16, cudaStream_t st,
                             int* launches) {
  KvAppendArgs a = args;
  const int per_tok = a.D_qk / 8 + (a.v_new ? a.D_v / 8 : 0);
  const long long items = static_cast<long long>(a.B) * a.C * per_tok;
  // fewer (token, chunk) items than two waves of resident threads (152 SMs x 2048):
  // one thread per head as well
  a.head_groups = items < 2LL * 152 * 2048 ? a.n_kv : 1;
  const long long total = items * a.head_groups;
  long long blocks = (total + 255) / 256;
  if (blocks > 152LL * 16) blocks = 152LL * 16;
  if (blocks < 1) blocks = 1;
  if (bf16)
    kv_append_kernel<__nv_bfloat16><<<static_cast<unsigned>(blocks), 256, 0, st>>>(a, rope);
  else
    kv_append_kernel<float><<<static_cast<unsigned>(blocks), 256, 0, st>>>(a, rope);
  *launches += 1;
  return cudaGetLastError();
}

cudaError_t launch_rope(const RopeArgs& a, const RopeFreq& rope, bool bf16, cudaStream_t st, int* launches) {
  const int CH = bf16 ? 8 : 2;
  const long long total = static_cast<long long>(a.B) * a.S * (a.D / CH);
  long long blocks = (total + 255) / 256;
  if (blocks > 152LL * 16) blocks = 152LL * 16;
  if (blocks < 1) blocks = 1;
  if (bf16)
    rope_kernel<__nv_bfloat16, 8><<<static_cast<unsigned>(blocks), 256, 0, st>>>(a, rope);
  else
    rope_kernel<float, 2><<<static_cast<unsigned>(blocks), 256, 0, st>>>(a, rope);
  *launches += 1;
  return cudaGetLastError();
}

}  // namespace attn

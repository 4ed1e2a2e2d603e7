// rope.cu - standalone rotary position embedding of [B, S, n_heads, D] rows.
//
// Rotates the pairs (2i, 2i+1) of the span [rope_offset, rope_offset + rope_dims)
// by pos * theta_i ("Transformer架构从Attention到DecoderBlock" §8.3).  This is the
// pass that writes rotated keys (the KV-cache form, "Transformer架构完全深度解析"
// §7) before the prefill kernel reads them.
//
// One thread owns a chunk of CH consecutive dims of one token for ALL heads, so
// the sin/cos of its pairs are computed once and reused n_heads times.  The
// kernel is bound by HBM bandwidth (read + write once).
#include "kernels.h"

namespace attn {
namespace {

template <typename T, int CH>
__global__ void __launch_bounds__(256) rope_kernel(RopeArgs a, RopeFreq f) {
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
    const bool rotated = d0 >= a.rope_offset && d0 < a.rope_offset + a.rope_dims;
    if (!rotated && in == out) continue;
    float sn[CH / 2], cs[CH / 2];
    if (rotated) {
      const int pair0 = (d0 - a.rope_offset) / 2;
#pragma unroll
      for (int p = 0; p < CH / 2; ++p) rope_sincos(a.pos_offset + s, f.hi[pair0 + p], f.lo[pair0 + p], &sn[p], &cs[p]);
    }
    const long long row0 = tok * a.n_heads;
    for (int h = 0; h < a.n_heads; ++h) {
      const long long off = (row0 + h) * a.D + d0;
      if constexpr (sizeof(T) == 2 && CH == 8) {
        uint4 u = *reinterpret_cast<const uint4*>(in + off);
        if (rotated) {
          float x[8];
          bf16x8_to_f32(u, x);
#pragma unroll
          for (int p = 0; p < 4; ++p) rotate_pair(x[2 * p], x[2 * p + 1], sn[p], cs[p]);
          u = f32_to_bf16x8(x);
        }
        *reinterpret_cast<uint4*>(out + off) = u;
      } else {
        float x[CH];
#pragma unroll
        for (int e = 0; e < CH; ++e) x[e] = to_f32(in[off + e]);
        if (rotated) {
#pragma unroll
          for (int p = 0; p < CH / 2; ++p) rotate_pair(x[2 * p], x[2 * p + 1], sn[p], cs[p]);
        }
#pragma unroll
        for (int e = 0; e < CH; ++e) out[off + e] = from_f32<T>(x[e]);
      }
    }
  }
}

// One thread per (sequence b, new token c, 8-dim chunk): the new key row is
// rotated at its absolute position start[b] + c and written to that cache
// slot for every KV head, the value row is copied next to it.
template <typename T>
__global__ void __launch_bounds__(256) kv_append_kernel(KvAppendArgs a, RopeFreq f) {
  const int kch = a.D_qk / 8, vch = a.v_new ? a.D_v / 8 : 0;
  const int per_tok = kch + vch;
  const long long total = static_cast<long long>(a.B) * a.C * per_tok;
  for (long long idx = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; idx < total;
       idx += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int ch = static_cast<int>(idx % per_tok);
    const long long bc = idx / per_tok;
    const int c = static_cast<int>(bc % a.C);
    const int b = static_cast<int>(bc / a.C);
    const int pos = a.start[b] + c;
    if (pos < 0 || pos >= a.max_len) continue;  // slots outside the cache are never written
    const long long slot = static_cast<long long>(b) * a.max_len + pos;
    if (ch < kch) {
      const int d0 = ch * 8;
      const bool rot = d0 >= a.rope_offset && d0 < a.rope_offset + 2 * f.n_pairs;
      float sn[4], cs[4];
      if (rot) {
        const int p0 = (d0 - a.rope_offset) / 2;
#pragma unroll
        for (int p = 0; p < 4; ++p) rope_sincos(pos, f.hi[p0 + p], f.lo[p0 + p], &sn[p], &cs[p]);
      }
      const T* src = static_cast<const T*>(a.k_new) + (bc * a.n_kv) * a.D_qk + d0;
      T* dst = static_cast<T*>(a.kcache) + slot * a.n_kv * a.D_qk + d0;
      for (int h = 0; h < a.n_kv; ++h) {
        float x[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) x[e] = to_f32(src[h * a.D_qk + e]);
        if (rot) {
#pragma unroll
          for (int p = 0; p < 4; ++p) rotate_pair(x[2 * p], x[2 * p + 1], sn[p], cs[p]);
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) dst[h * a.D_qk + e] = from_f32<T>(x[e]);
      }
    } else {
      const int d0 = (ch - kch) * 8;
      const T* src = static_cast<const T*>(a.v_new) + (bc * a.n_kv) * a.D_v + d0;
      T* dst = static_cast<T*>(a.vcache) + slot * a.v_token_stride + d0;
      for (int h = 0; h < a.n_kv; ++h)
#pragma unroll
        for (int e = 0; e < 8; ++e) dst[h * a.D_v + e] = src[h * a.D_v + e];
    }
  }
}

}  // namespace

cudaError_t launch_kv_append(const KvAppendArgs& a, const RopeFreq& rope, bool bf16, cudaStream_t st, int* launches) {
  const int per_tok = a.D_qk / 8 + (a.v_new ? a.D_v / 8 : 0);
  const long long total = static_cast<long long>(a.B) * a.C * per_tok;
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

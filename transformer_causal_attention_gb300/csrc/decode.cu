// decode.cu - single-token decode over a KV cache: split-KV partials on CUDA
// cores, then a log-sum-exp combine.
//
// Decode reads every cached key and value once and does ~2 FLOPs per byte
// (GQA, G = 4), so it is bound by HBM bandwidth ("Transformer架构完全深度解析" §9:
// decode is memory-bound; "Transformer 与 LLM" slide 10).  The kernel therefore
// aims at bytes in flight, not at tensor cores:
//   * one CTA per (sequence b, KV head g, group of HG query heads, key chunk);
//     the HG heads share every K/V row it loads (GQA: K/V are not replicated,
//     "Transformer架构从Attention到DecoderBlock" §6.3);
//   * a half-warp covers one key row with 16-byte loads (8 bf16 per lane), NB
//     rows per step, so each warp keeps 2*NB*(row bytes) of loads in flight;
//   * scores are reduced across the half-warp by xor-shuffles and folded into
//     a running max / running sum per head (online softmax,
//     "Transformer架构完全深度解析" §13);
//   * the 16 half-warps of the CTA merge their (m, l, O) in shared memory and the
//     CTA writes one normalised partial (O_j, lse_j) per head;
//   * the combine kernel merges the chunks of a sequence:
//     lse = log2 sum_j 2^lse_j,  O = sum_j 2^(lse_j - lse) O_j.
// The query is rotated at position seqlens[b] - 1 (the new token's slot: the
// cache already holds its rotated key, "Transformer架构完全深度解析" §9).
#include <math.h>

#include "kernels.h"

namespace attn {
namespace {

constexpr int kThreads = 256;
constexpr int kHalfWarps = kThreads / 16;

// 8 consecutive elements as stored, and their fp32 values.
template <typename T> struct Raw8;
template <> struct Raw8<__nv_bfloat16> {
  uint4 u;
  __device__ __forceinline__ void load(const __nv_bfloat16* p) { u = __ldg(reinterpret_cast<const uint4*>(p)); }
  __device__ __forceinline__ void zero() { u = make_uint4(0, 0, 0, 0); }
  __device__ __forceinline__ void unpack(float* f) const { bf16x8_to_f32(u, f); }
};
template <> struct Raw8<float> {
  float4 a, b;
  __device__ __forceinline__ void load(const float* p) {
    a = __ldg(reinterpret_cast<const float4*>(p));
    b = __ldg(reinterpret_cast<const float4*>(p) + 1);
  }
  __device__ __forceinline__ void zero() { a = b = make_float4(0.f, 0.f, 0.f, 0.f); }
  __device__ __forceinline__ void unpack(float* f) const {
    f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
    f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
  }
};

template <typename T, int NQC, int NVC, int HG, int NB>
__global__ void __launch_bounds__(kThreads) decode_split_kernel(DecodeArgs a, RopeFreq f) {
  extern __shared__ float smem[];
  float* q_s = smem;                                  // [HG][NQC*128]
  float* red_o = q_s + HG * NQC * 128;                // [16][HG][NVC*128]
  float* red_m = red_o + kHalfWarps * HG * NVC * 128;  // [16][HG]
  float* red_l = red_m + kHalfWarps * HG;              // [16][HG]

  const int split = blockIdx.x;
  const int G = a.n_h / a.n_kv;
  const int n_hg = G / HG;
  const int g = blockIdx.y / n_hg;
  const int h0 = g * G + (blockIdx.y % n_hg) * HG;
  const int b = blockIdx.z;
  const int L = min(max(a.seqlens[b], 1), a.max_len);
  const int c_lo = split * a.chunk, c_hi = min(L, c_lo + a.chunk);
  int vlo[2], vhi[2];
  const int nr = decode_visible(L, a.window, a.n_sink, vlo, vhi);
  bool any = false;
  for (int r = 0; r < nr; ++r) any |= max(c_lo, vlo[r]) < min(c_hi, vhi[r]);
  if (!any) return;  // the combine pass never reads this chunk
  const int pos = L - 1;

  // rotated, pre-scaled queries of the HG heads
  const T* qb = static_cast<const T*>(a.q) + (static_cast<long long>(b) * a.n_h + h0) * a.D_qk;
  for (int idx = threadIdx.x; idx < HG * (NQC * 64); idx += kThreads) {
    // pair slot p covers dims (2p, 2p + 1), except inside the rotated span
    // (rope_offset is even) where it is rotation pair j = p - rope_offset / 2
    const int i = idx / (NQC * 64), p = idx % (NQC * 64);
    const int j = p - a.rope_offset / 2;
    const bool rot = j >= 0 && j < f.n_pairs;
    int2 d = make_int2(2 * p, 2 * p + 1);
    if (rot) {
      d = rope_pair_dims(f, j);
      d.x += a.rope_offset;
      d.y += a.rope_offset;
    }
    float x0 = 0.f, x1 = 0.f;
    if (2 * p < a.D_qk) {
      x0 = to_f32(qb[i * a.D_qk + d.x]);
      x1 = to_f32(qb[i * a.D_qk + d.y]);
      if (rot) {
        float s, c;
        rope_sincos(pos, f.hi[j], f.lo[j], &s, &c);
        rotate_pair(x0, x1, s, c);
      }
    }
    q_s[i * NQC * 128 + d.x] = x0 * a.scale_log2;
    q_s[i * NQC * 128 + d.y] = x1 * a.scale_log2;
  }
  __syncthreads();

  const int hw = threadIdx.x >> 4, hl = threadIdx.x & 15;
  float qr[HG][NQC][8];
#pragma unroll
  for (int i = 0; i < HG; ++i)
#pragma unroll
    for (int c = 0; c < NQC; ++c)
#pragma unroll
      for (int e = 0; e < 8; ++e) qr[i][c][e] = q_s[i * NQC * 128 + c * 128 + hl * 8 + e];

  float o[HG][NVC][8];
  float m_run[HG], l_run[HG];
#pragma unroll
  for (int i = 0; i < HG; ++i) {
    m_run[i] = -INFINITY;
    l_run[i] = 0.f;
#pragma unroll
    for (int c = 0; c < NVC; ++c)
#pragma unroll
      for (int e = 0; e < 8; ++e) o[i][c][e] = 0.f;
  }

  const long long k_tok = static_cast<long long>(a.n_kv) * a.D_qk;
  const T* kb = static_cast<const T*>(a.kcache) + static_cast<long long>(b) * a.max_len * k_tok +
                static_cast<long long>(g) * a.D_qk;
  const T* vb = static_cast<const T*>(a.vcache) + static_cast<long long>(b) * a.max_len * a.v_token_stride +
                static_cast<long long>(g) * a.D_v;

  // A warp takes 2*NB consecutive keys per step (NB per half-warp); the trip
  // count is uniform across the warp so the full-mask shuffles are legal.
  // The chunk's keys are walked as (at most two) visible ranges.
  const int warp = threadIdx.x >> 5;
  for (int r = 0; r < nr; ++r) {
  const int start = max(c_lo, vlo[r]), end = min(c_hi, vhi[r]);
  for (int base = start + warp * 2 * NB; base < end; base += (kThreads / 32) * 2 * NB) {
    const int key0 = base + (hw & 1) * NB;
    Raw8<T> kr[NB][NQC], vr[NB][NVC];
#pragma unroll
    for (int j = 0; j < NB; ++j) {
      const bool ok = key0 + j < end;
#pragma unroll
      for (int c = 0; c < NQC; ++c) {
        const int d = c * 128 + hl * 8;
        if (ok && d < a.D_qk) kr[j][c].load(kb + (key0 + j) * k_tok + d);
        else kr[j][c].zero();
      }
#pragma unroll
      for (int c = 0; c < NVC; ++c) {
        const int d = c * 128 + hl * 8;
        if (ok && d < a.D_v) vr[j][c].load(vb + (key0 + j) * a.v_token_stride + d);
        else vr[j][c].zero();
      }
    }
    float s[NB][HG];
#pragma unroll
    for (int j = 0; j < NB; ++j) {
#pragma unroll
      for (int i = 0; i < HG; ++i) s[j][i] = 0.f;
#pragma unroll
      for (int c = 0; c < NQC; ++c) {
        float kf[8];
        kr[j][c].unpack(kf);
#pragma unroll
        for (int i = 0; i < HG; ++i)
#pragma unroll
          for (int e = 0; e < 8; ++e) s[j][i] = fmaf(qr[i][c][e], kf[e], s[j][i]);
      }
#pragma unroll
      for (int i = 0; i < HG; ++i) {
#pragma unroll
        for (int off = 8; off > 0; off >>= 1) s[j][i] += __shfl_xor_sync(0xffffffffu, s[j][i], off);
        if (key0 + j >= end) s[j][i] = -INFINITY;
      }
    }
#pragma unroll
    for (int i = 0; i < HG; ++i) {
      float mx = s[0][i];
#pragma unroll
      for (int j = 1; j < NB; ++j) mx = fmaxf(mx, s[j][i]);
      const float m_new = fmaxf(m_run[i], mx);
      // -inf only while this half-warp has seen no valid key: weights stay 0
      const float m_ref = (m_new == -INFINITY) ? 0.f : m_new;
      const float alpha = fast_exp2(m_run[i] - m_ref);
      float psum = 0.f;
#pragma unroll
      for (int j = 0; j < NB; ++j) {
        s[j][i] = fast_exp2(s[j][i] - m_ref);
        psum += s[j][i];
      }
      l_run[i] = l_run[i] * alpha + psum;
      m_run[i] = m_new;
#pragma unroll
      for (int c = 0; c < NVC; ++c)
#pragma unroll
        for (int e = 0; e < 8; ++e) o[i][c][e] *= alpha;
    }
#pragma unroll
    for (int j = 0; j < NB; ++j) {
#pragma unroll
      for (int c = 0; c < NVC; ++c) {
        float vf[8];
        vr[j][c].unpack(vf);
#pragma unroll
        for (int i = 0; i < HG; ++i)
#pragma unroll
          for (int e = 0; e < 8; ++e) o[i][c][e] = fmaf(s[j][i], vf[e], o[i][c][e]);
      }
    }
  }

  }  // visible ranges

  // merge the 16 half-warps
#pragma unroll
  for (int i = 0; i < HG; ++i) {
    if (hl == 0) {
      red_m[hw * HG + i] = m_run[i];
      red_l[hw * HG + i] = l_run[i];
    }
#pragma unroll
    for (int c = 0; c < NVC; ++c)
#pragma unroll
      for (int e = 0; e < 8; ++e) red_o[(hw * HG + i) * NVC * 128 + c * 128 + hl * 8 + e] = o[i][c][e];
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < HG * a.D_v; idx += kThreads) {
    const int i = idx / a.D_v, d = idx % a.D_v;
    float M = -INFINITY;
    for (int w = 0; w < kHalfWarps; ++w) M = fmaxf(M, red_m[w * HG + i]);
    float num = 0.f, den = 0.f;
    for (int w = 0; w < kHalfWarps; ++w) {
      const float mw = red_m[w * HG + i];
      if (mw == -INFINITY) continue;  // this half-warp saw no key
      const float sc = fast_exp2(mw - M);
      num = fmaf(red_o[(w * HG + i) * NVC * 128 + d], sc, num);
      den = fmaf(red_l[w * HG + i], sc, den);
    }
    const long long slot = (static_cast<long long>(b) * a.n_h + h0 + i) * a.n_split + split;
    a.ws_o[slot * a.D_v + d] = num / den;
    if (d == 0) a.ws_lse[slot] = M + log2f(den);
  }
}

// Four consecutive fp32 values stored as T.
template <typename T>
__device__ __forceinline__ void store4(T* p, float4 v);
template <>
__device__ __forceinline__ void store4<float>(float* p, float4 v) {
  *reinterpret_cast<float4*>(p) = v;
}
template <>
__device__ __forceinline__ void store4<__nv_bfloat16>(__nv_bfloat16* p, float4 v) {
  const __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y), hi = __floats2bfloat162_rn(v.z, v.w);
  uint2 u;
  u.x = *reinterpret_cast<const uint32_t*>(&lo);
  u.y = *reinterpret_cast<const uint32_t*>(&hi);
  *reinterpret_cast<uint2*>(p) = u;
}

// One warp per (sequence b, head h): the chunk partials' maximum and weight sum by
// shuffles, then D_v output dims as 16-byte loads of the partials (4 dims per lane per
// step).  No block-wide step, so the warps of a block never wait for one another.
constexpr int kCombineWarps = 8;

template <typename T>
__global__ void __launch_bounds__(kCombineWarps * 32) decode_combine_kernel(DecodeArgs a) {
  const int lane = threadIdx.x & 31;
  const int bh = blockIdx.x * kCombineWarps + (threadIdx.x >> 5);
  if (bh >= a.B * a.n_h) return;  // whole warps only
  const int b = bh / a.n_h;
  const int L = min(max(a.seqlens[b], 1), a.max_len);
  const int ns = (L + a.chunk - 1) / a.chunk;
  const float* lse = a.ws_lse + static_cast<long long>(bh) * a.n_split;
  int lo0, hi0, lo1 = 0, hi1 = 0;
  {
    int vlo[2], vhi[2];
    const int nr = decode_visible(L, a.window, a.n_sink, vlo, vhi);
    lo0 = vlo[0];
    hi0 = vhi[0];
    if (nr == 2) {
      lo1 = vlo[1];
      hi1 = vhi[1];
    }
  }
  auto written = [&](int j) {  // chunk j holds a visible key, so its partial was written
    const int c0 = j * a.chunk, c1 = min(L, (j + 1) * a.chunk);
    return max(c0, lo0) < min(c1, hi0) || max(c0, lo1) < min(c1, hi1);
  };
  float M = -INFINITY;
  for (int j = lane; j < ns; j += 32)
    if (written(j)) M = fmaxf(M, lse[j]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  const float* po = a.ws_o + static_cast<long long>(bh) * a.n_split * a.D_v;
  T* out = static_cast<T*>(a.out) + static_cast<long long>(bh) * a.D_v;
  float den = 0.f;
  // dims d0 = 4 lane + 128 c; D_v <= 512, a multiple of 8
  float4 acc[4];
#pragma unroll
  for (int c = 0; c < 4; ++c) acc[c] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int j0 = 0; j0 < ns; j0 += 32) {
    const float wl = (j0 + lane < ns && written(j0 + lane)) ? exp2f(lse[j0 + lane] - M) : 0.f;
    den += wl;
    const int nj = min(32, ns - j0);
    for (int jj = 0; jj < nj; ++jj) {
      const float w = __shfl_sync(0xffffffffu, wl, jj);
      if (w == 0.f) continue;  // uniform across the warp
      const float* pj = po + static_cast<long long>(j0 + jj) * a.D_v;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int d0 = 4 * lane + 128 * c;
        if (d0 < a.D_v) {
          const float4 v = *reinterpret_cast<const float4*>(pj + d0);
          acc[c].x = fmaf(w, v.x, acc[c].x);
          acc[c].y = fmaf(w, v.y, acc[c].y);
          acc[c].z = fmaf(w, v.z, acc[c].z);
          acc[c].w = fmaf(w, v.w, acc[c].w);
        }
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
  const float inv = 1.f / den;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const int d0 = 4 * lane + 128 * c;
    if (d0 < a.D_v)
      store4<T>(out + d0, make_float4(acc[c].x * inv, acc[c].y * inv, acc[c].z * inv, acc[c].w * inv));
  }
  if (a.lse != nullptr && lane == 0) a.lse[bh] = (M + log2f(den)) * 0.69314718055994530942f;
}

// Query heads per CTA: more heads share each loaded K/V row, but every head
// costs registers for its query slice and output slice.
int pick_hg(int G, int D_qk, int D_v) {
  if (D_qk > 256 || D_v > 256) return 1;
  if (D_qk <= 128 && D_v <= 128 && G % 4 == 0) return 4;
  if (G % 2 == 0) return 2;
  return 1;
}

template <typename T, int NQC, int NVC, int HG>
cudaError_t launch_split(const DecodeArgs& a, const RopeFreq& f, cudaStream_t st) {
  constexpr int NB = (NQC + NVC > 4) ? 2 : 4;
  const size_t smem = sizeof(float) * (HG * NQC * 128 + kHalfWarps * HG * NVC * 128 + 2 * kHalfWarps * HG);
  auto kern = decode_split_kernel<T, NQC, NVC, HG, NB>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  dim3 grid(a.n_split, a.n_kv * ((a.n_h / a.n_kv) / HG), a.B);
  kern<<<grid, kThreads, smem, st>>>(a, f);
  return cudaGetLastError();
}

template <typename T, int NQC, int NVC>
cudaError_t launch_hg(const DecodeArgs& a, const RopeFreq& f, cudaStream_t st) {
  const int hg = pick_hg(a.n_h / a.n_kv, a.D_qk, a.D_v);
  if constexpr (NQC + NVC <= 2) {
    if (hg == 4) return launch_split<T, NQC, NVC, 4>(a, f, st);
  }
  if constexpr (NQC + NVC <= 4) {
    if (hg >= 2) return launch_split<T, NQC, NVC, 2>(a, f, st);
  }
  return launch_split<T, NQC, NVC, 1>(a, f, st);
}

template <typename T>
cudaError_t launch_t(const DecodeArgs& a, const RopeFreq& f, cudaStream_t st) {
  const int nq = (a.D_qk + 127) / 128, nv = (a.D_v + 127) / 128;
  if (nq == 1 && nv == 1) return launch_hg<T, 1, 1>(a, f, st);
  if (nq <= 2 && nv <= 2) return launch_hg<T, 2, 2>(a, f, st);
  return launch_hg<T, 5, 4>(a, f, st);
}

}  // namespace

// Number of key chunks per sequence and the chunk length: the smallest power
// of two >= 256 keys that keeps the grid near 8192 CTAs (several waves over 152
// SMs) while bounding the partial-result workspace.
int decode_plan_splits(int B, int n_h, int n_kv, int D_qk, int D_v, int max_len, int* chunk) {
  const int G = n_h / n_kv;
  const long long units = static_cast<long long>(B) * n_kv * (G / pick_hg(G, D_qk, D_v));
  int c = 256;
  while (c < max_len && units * ((max_len + c - 1) / c) > 8192) c *= 2;
  int ns = (max_len + c - 1) / c;
  while (ns > 1024) {  // the combine kernel keeps one weight per chunk in shared memory
    c *= 2;
    ns = (max_len + c - 1) / c;
  }
  *chunk = c;
  return ns;
}

cudaError_t launch_decode_combine(const DecodeArgs& a, bool bf16, cudaStream_t st, int* launches) {
  const unsigned grid = static_cast<unsigned>((a.B * a.n_h + kCombineWarps - 1) / kCombineWarps);
  if (bf16)
    decode_combine_kernel<__nv_bfloat16><<<grid, kCombineWarps * 32, 0, st>>>(a);
  else
    decode_combine_kernel<float><<<grid, kCombineWarps * 32, 0, st>>>(a);
  *launches += 1;
  return cudaGetLastError();
}

cudaError_t launch_decode(const DecodeArgs& a, const RopeFreq& rope, bool bf16, cudaStream_t st, int* launches) {
  *launches += 1;
  const cudaError_t e = bf16 ? launch_t<__nv_bfloat16>(a, rope, st) : launch_t<float>(a, rope, st);
  if (e != cudaSuccess) return e;
  return launch_decode_combine(a, bf16, st, launches);
}

}  // namespace attn

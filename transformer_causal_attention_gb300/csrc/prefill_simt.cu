// prefill_simt.cu - CUDA-core prefill for head sizes / dtypes without a
// tensor-core kernel (fp32 inputs, unusual D_h).
//
// One warp owns one query row (b, h, m).  Its lanes score 32 keys at a time
// (full dot products against the rotated, pre-scaled query held in shared
// memory), then fold the 32 scores into the running maximum m and running sum
// l of the online softmax ("Transformer架构完全深度解析" §13:
// m_new = max(m_old, x), l_new = e^(m_old - m_new) l_old + e^(x - m_new)) and
// accumulate the weighted values, each lane owning D_h/32 output dims.  Keys
// after the query are never visited (causal skip, "2.7 Transformer Decoder
// Block完整解析" §3.3).  Scores live in the log2 domain (scale * log2 e folded
// into the query), so exp is exp2.
#include <math.h>

#include "kernels.h"

namespace attn {
namespace {

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

template <typename T, int DMAX>
__global__ void __launch_bounds__(128) prefill_simt_kernel(PrefillArgs a, RopeFreq f) {
  __shared__ float q_s[4][DMAX];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long total = static_cast<long long>(a.B) * a.n_h * a.S;
  const long long row = static_cast<long long>(blockIdx.x) * 4 + warp;
  if (row >= total) return;  // whole warp leaves together; only __syncwarp is used below
  const int D = a.D;
  const int m = static_cast<int>(row % a.S);
  const long long bh = row / a.S;
  const int h = static_cast<int>(bh % a.n_h);
  const int b = static_cast<int>(bh / a.n_h);
  const int g = h / (a.n_h / a.n_kv);

  const T* qrow = static_cast<const T*>(a.q) + ((static_cast<long long>(b) * a.S + m) * a.n_h + h) * D;
  for (int p = lane; p < D / 2; p += 32) {
    // pair slot p covers dims (2p, 2p + 1), except inside the rotated span
    // (rope_offset is even) where it is rotation pair j = p - rope_offset / 2
    const int j = p - a.rope_offset / 2;
    const bool rot = j >= 0 && j < f.n_pairs;
    int2 d = make_int2(2 * p, 2 * p + 1);
    if (rot) {
      d = rope_pair_dims(f, j);
      d.x += a.rope_offset;
      d.y += a.rope_offset;
    }
    float x0 = to_f32(qrow[d.x]), x1 = to_f32(qrow[d.y]);
    if (rot) {
      float s, c;
      rope_sincos(a.q_offset + m, f.hi[j], f.lo[j], &s, &c);
      rotate_pair(x0, x1, s, c);
    }
    q_s[warp][d.x] = x0 * a.scale_log2;
    q_s[warp][d.y] = x1 * a.scale_log2;
  }
  __syncwarp();

  const int Dv = a.D_v;
  const long long row_stride = static_cast<long long>(a.n_kv) * D;     // between consecutive keys
  const long long vrow_stride = static_cast<long long>(a.n_kv) * Dv;   // between consecutive values
  const T* kbase = static_cast<const T*>(a.k) + (static_cast<long long>(b) * a.kv_rows * a.n_kv + g) * D;
  const T* vbase = static_cast<const T*>(a.v) + (static_cast<long long>(b) * a.kv_rows * a.n_kv + g) * Dv;
  constexpr int NT = DMAX / 32;
  float acc[NT];
#pragma unroll
  for (int t = 0; t < NT; ++t) acc[t] = 0.f;
  float m_run = -INFINITY, l = 0.f;
  const int pos = a.q_offset + m;
  const int n_end = a.causal ? pos + 1 : a.S_k;
  // visible keys: [0, n_end), or with a window the sinks [0, n_sink) and [pos - window + 1, n_end)
  int win_lo = 0;
  if (a.window > 0) win_lo = max(0, pos - a.window + 1);
  const int sink_end = (a.window > 0 && a.n_sink < win_lo) ? a.n_sink : 0;
  if (a.window > 0 && a.n_sink >= win_lo) win_lo = 0;  // sinks and window overlap: one range

  for (int range = 0; range < 2; ++range) {
    const int r_lo = range == 0 ? 0 : win_lo, r_hi = range == 0 ? sink_end : n_end;
    for (int n0 = r_lo; n0 < r_hi; n0 += 32) {
      const int n = n0 + lane;
      float s = -INFINITY;
      if (n < r_hi) {
        const T* kr = kbase + n * row_stride;
        float dot = 0.f;
        for (int d = 0; d < D; ++d) dot = fmaf(q_s[warp][d], to_f32(kr[d]), dot);
        s = dot;
      }
      const float m_new = fmaxf(m_run, warp_max(s));  // finite: lane 0 always holds a visible key
      const float alpha = exp2f(m_run - m_new);
      const float p = (n < r_hi) ? exp2f(s - m_new) : 0.f;
      l = l * alpha + warp_sum(p);
#pragma unroll
      for (int t = 0; t < NT; ++t) acc[t] *= alpha;
      const int cnt = min(32, r_hi - n0);
      for (int j = 0; j < cnt; ++j) {
        const float pj = __shfl_sync(0xffffffffu, p, j);
        const T* vr = vbase + (n0 + j) * vrow_stride;
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          const int d = lane + 32 * t;
          if (d < Dv) acc[t] = fmaf(pj, to_f32(vr[d]), acc[t]);
        }
      }
      m_run = m_new;
    }
  }

  T* orow = static_cast<T*>(a.out) + ((static_cast<long long>(b) * a.S + m) * a.n_h + h) * Dv;
  const float inv_l = 1.f / l;
#pragma unroll
  for (int t = 0; t < NT; ++t) {
    const int d = lane + 32 * t;
    if (d < Dv) orow[d] = from_f32<T>(acc[t] * inv_l);
  }
  if (a.lse != nullptr && lane == 0)
    a.lse[(static_cast<long long>(b) * a.n_h + h) * a.S + m] = (m_run + log2f(l)) * 0.69314718055994530942f;
}

template <typename T>
cudaError_t launch_t(const PrefillArgs& a, const RopeFreq& f, cudaStream_t st) {
  const long long rows = static_cast<long long>(a.B) * a.n_h * a.S;
  const unsigned blocks = static_cast<unsigned>((rows + 3) / 4);
  const int dmax = a.D > a.D_v ? a.D : a.D_v;  // the query row and the output row share DMAX
  if (dmax <= 32)
    prefill_simt_kernel<T, 32><<<blocks, 128, 0, st>>>(a, f);
  else if (dmax <= 64)
    prefill_simt_kernel<T, 64><<<blocks, 128, 0, st>>>(a, f);
  else if (dmax <= 128)
    prefill_simt_kernel<T, 128><<<blocks, 128, 0, st>>>(a, f);
  else
    prefill_simt_kernel<T, 256><<<blocks, 128, 0, st>>>(a, f);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill_simt(const PrefillArgs& a, const RopeFreq& rope, bool bf16, cudaStream_t st,
                                int* launches) {
  *launches += 1;
  return bf16 ? launch_t<__nv_bfloat16>(a, rope, st) : launch_t<float>(a, rope, st);
}

}  // namespace attn

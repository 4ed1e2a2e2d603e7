// decode_stream.cu - split-KV GQA decode with K/V streamed through shared
// memory by TMA (bf16, D_qk = D_v = 128, G a multiple of 4).
//
// Decode reads each cached key/value row once and is bound by HBM bandwidth
// ("Transformer架构完全深度解析" §9).  To keep enough bytes in flight the kernel
// is persistent (one CTA per SM) and splits roles:
//   warp 0      TMA producer: for every work unit (sequence b, chunk of keys,
//               group of 4 query heads, KV head g) it first asks for the whole
//               unit to be pulled into L2 (many DRAM reads in flight, each line
//               used shortly after), then streams 64-key K and V tiles into a
//               5-stage ring (32 KB per stage, 128-byte swizzle);
//   warps 1-8   consumers: each half-warp scores 4 keys of a tile against the 4
//               query heads (lane = 8 dims, packed fp32x2 FMAs), reduces the 16
//               partial dot products with a reduce-scatter butterfly (15
//               shuffles, one finished score per lane), folds them into the
//               running max / running sum per head (online softmax,
//               "Transformer架构完全深度解析" §13) and accumulates P V.
// At the end of a unit the 16 half-warps merge in shared memory and write one
// normalised partial (O_j, log2-sum) per head; the combine kernel of decode.cu
// merges the chunks of each sequence.  Rows past seqlens[b] that a tile
// carries are masked (score -inf) and never touch the accumulators.
#include <math.h>

#include "kernels.h"

namespace attn {
namespace {

constexpr int D = 128;
constexpr int HG = 4;                 // query heads per unit
constexpr int BK = kStreamTileKeys;   // keys per tile
static_assert(BK == 64, "16 half-warps x 4 keys");
constexpr int NB = 4;                 // keys per half-warp per tile (16 half-warps x 4 = BK)
constexpr int kStages = 5;
constexpr int kConsumerWarps = 8;
constexpr int kThreads = 32 * (1 + kConsumerWarps);
constexpr int kTileBytes = BK * D * 2;     // one K or V tile
constexpr int kBlockBytes = BK * 128;      // one 64-dim column block of a tile
constexpr int kStageBytes = 2 * kTileBytes;
constexpr int kRedOff = kStages * kStageBytes;
constexpr int kRedBytes = 16 * HG * D * 4 + 2 * 16 * HG * 4;
constexpr int kBarOff = kRedOff + kRedBytes;
constexpr int kSmemBytes = kBarOff + 256 + 1024;

struct Bars {
  uint64_t full[kStages], empty[kStages];
  uint64_t merge;  // consumer-only barrier (every consumer thread arrives)
  int abort_flag;
};

struct Unit {
  int b, g, h0, start, end, L;
};

// Units enumerate (b, chunk, head group, g) with the KV head fastest: CTAs that
// run side by side read the other heads of the same cached tokens, so every
// 2 KB token row (all heads) is fetched from DRAM at about the same time.
// Chunks past the sequence are empty.
__device__ __forceinline__ bool unit_at(int u, const DecodeArgs& a, Unit& w) {
  const int n_hg = (a.n_h / a.n_kv) / HG;
  w.g = u % a.n_kv;
  int r = u / a.n_kv;
  const int hg = r % n_hg;
  r /= n_hg;
  const int split = r % a.n_split;
  w.b = r / a.n_split;
  w.h0 = w.g * (a.n_h / a.n_kv) + hg * HG;
  w.L = min(max(a.seqlens[w.b], 1), a.max_len);
  w.start = split * a.chunk;
  w.end = min(w.L, w.start + a.chunk);
  return w.start < w.L;
}

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, const WaitCtl& w) {
  const bool ok = mbar_wait(bar, parity, w);
  return __all_sync(0xffffffffu, ok);
}

// Barrier over the consumer warps built on an mbarrier, so that it is bounded:
// a CTA that gives up releases every waiter instead of hanging on bar.sync.
__device__ __forceinline__ bool consumer_sync(uint64_t* bar, uint32_t& phase, const WaitCtl& w) {
  mbar_arrive(bar);
  const bool ok = warp_wait(bar, phase, w);
  phase ^= 1;
  return ok;
}

__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity, unsigned long long limit_ns) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > limit_ns) return;
  }
}

// 8 bf16 of a swizzled tile row: chunk c (16 bytes) of row r sits at chunk c ^ (r & 7).
__device__ __forceinline__ uint4 tile_chunk(const uint8_t* tile, int r, int c) {
  return *reinterpret_cast<const uint4*>(tile + (c >> 3) * kBlockBytes + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

__global__ void __launch_bounds__(kThreads, 1)
    decode_stream_kernel(const __grid_constant__ DecodeArgs a, const __grid_constant__ RopeFreq f,
                         const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v) {
  extern __shared__ uint8_t smem_raw[];
  // aligned by pointer arithmetic on the shared array, so that the compiler keeps shared-memory addressing
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  Bars* bars = reinterpret_cast<Bars*>(smem + kBarOff);
  float* red_o = reinterpret_cast<float*>(smem + kRedOff);  // [16][HG][D]
  float* red_m = red_o + 16 * HG * D;                        // [16][HG]
  float* red_l = red_m + 16 * HG;                            // [16][HG]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_units = a.B * a.n_kv * ((a.n_h / a.n_kv) / HG) * a.n_split;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bars->full[s], 1);
      mbar_init(&bars->empty[s], kConsumerWarps);
    }
    mbar_init(&bars->merge, 32 * kConsumerWarps);
    bars->abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  const WaitCtl wc{&bars->abort_flag, a.status, a.wait_limit_ns};

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      uint32_t st = 0, ph = 0, issued = 0, last_ph = 0;
      for (int u = blockIdx.x; u < n_units; u += gridDim.x) {
        Unit w;
        if (!unit_at(u, a, w)) continue;
        for (int k0 = w.start; k0 < w.end; k0 += BK)
          for (int db = 0; db < D / 64; ++db) {
            tma_prefetch_l2_4d(&tm_k, db * 64, w.g, k0, w.b);
            tma_prefetch_l2_4d(&tm_v, db * 64, w.g, k0, w.b);
          }
        for (int k0 = w.start; k0 < w.end; k0 += BK) {
          if (!mbar_wait(&bars->empty[st], ph ^ 1, wc)) goto producer_done;
          mbar_arrive_expect_tx(&bars->full[st], kStageBytes);
          uint8_t* kdst = smem + st * kStageBytes;
          for (int db = 0; db < D / 64; ++db) {
            tma_load_4d(kdst + db * kBlockBytes, &tm_k, &bars->full[st], db * 64, w.g, k0, w.b);
            tma_load_4d(kdst + kTileBytes + db * kBlockBytes, &tm_v, &bars->full[st], db * 64, w.g, k0, w.b);
          }
          issued |= 1u << st;
          last_ph = (last_ph & ~(1u << st)) | (ph << st);
          if (++st == kStages) { st = 0; ph ^= 1; }
        }
      }
    producer_done:
      if (bars->abort_flag)
        for (int s = 0; s < kStages; ++s)
          if (issued & (1u << s)) drain_wait(&bars->full[s], (last_ph >> s) & 1, a.wait_limit_ns);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ consumers
    const int cw = warp - 1;                 // consumer warp 0..7
    const int hw = cw * 2 + (lane >> 4);     // half-warp 0..15
    const int hl = lane & 15;                // lane within the half-warp: dims [8 hl, 8 hl + 8)
    const int my_key = hl >> 2, my_head = hl & 3;  // (key, head) this lane finishes after the butterfly
    uint32_t st = 0, ph = 0, mph = 0;
    for (int u = blockIdx.x; u < n_units; u += gridDim.x) {
      Unit w;
      if (!unit_at(u, a, w)) continue;
      const int pos = w.L - 1;  // the new token's position
      // this lane's 8 query dims of each head, rotated at the new token's position and pre-scaled
      float2 q2[HG][4];
      const __nv_bfloat16* qb =
          static_cast<const __nv_bfloat16*>(a.q) + (static_cast<long long>(w.b) * a.n_h + w.h0) * D + hl * 8;
      const int rel = hl * 8 - a.rope_offset;  // this lane's chunk within the rotated span (offset % 8 == 0)
      const bool in_span = rel >= 0 && rel < 2 * f.n_pairs;
      if (!f.half) {
        float sn[4], cs[4];
#pragma unroll
        for (int p = 0; p < 4; ++p)
          if (in_span) rope_sincos(pos, f.hi[rel / 2 + p], f.lo[rel / 2 + p], &sn[p], &cs[p]);
#pragma unroll
        for (int h = 0; h < HG; ++h) {
          float x[8];
          bf16x8_to_f32(*reinterpret_cast<const uint4*>(qb + h * D), x);
#pragma unroll
          for (int p = 0; p < 4; ++p) {
            if (in_span) rotate_pair(x[2 * p], x[2 * p + 1], sn[p], cs[p]);
            q2[h][p] = make_float2(x[2 * p] * a.scale_log2, x[2 * p + 1] * a.scale_log2);
          }
        }
      } else {
        // split halves: dim rel + e pairs with rel + e +- n_pairs, held by the lane
        // n_pairs / 8 chunks away (n_pairs % 8 == 0); every lane joins the shuffles
        const bool first = rel < f.n_pairs;
        const int jb = first ? rel : rel - f.n_pairs;  // pair index of element 0
        const int partner = (lane & 16) | (in_span ? (first ? hl + f.n_pairs / 8 : hl - f.n_pairs / 8) : hl);
        float sn[8], cs[8];
#pragma unroll
        for (int e = 0; e < 8; ++e)
          if (in_span) rope_sincos(pos, f.hi[jb + e], f.lo[jb + e], &sn[e], &cs[e]);
#pragma unroll
        for (int h = 0; h < HG; ++h) {
          float x[8];
          bf16x8_to_f32(*reinterpret_cast<const uint4*>(qb + h * D), x);
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const float y = __shfl_sync(0xffffffffu, x[e], partner);
            if (in_span) {
              float lo = first ? x[e] : y, hi = first ? y : x[e];
              rotate_pair(lo, hi, sn[e], cs[e]);
              x[e] = first ? lo : hi;
            }
          }
#pragma unroll
          for (int p = 0; p < 4; ++p) q2[h][p] = make_float2(x[2 * p] * a.scale_log2, x[2 * p + 1] * a.scale_log2);
        }
      }
      float2 o2[HG][4];
      float m_run[HG];
#pragma unroll
      for (int h = 0; h < HG; ++h) {
        m_run[h] = -INFINITY;
#pragma unroll
        for (int p = 0; p < 4; ++p) o2[h][p] = make_float2(0.f, 0.f);
      }
      float l_own = 0.f;  // running sum of head my_head
      bool ok = true;
      for (int k0 = w.start; k0 < w.end; k0 += BK) {
        if (!warp_wait(&bars->full[st], ph, wc)) { ok = false; break; }
        const uint8_t* kt = smem + st * kStageBytes;
        const uint8_t* vt = kt + kTileBytes;
        const int r0 = hw * NB;  // first tile row of this half-warp
        // partial dot products over this lane's 8 dims: part[j][h]
        float part[NB][HG];
#pragma unroll
        for (int j = 0; j < NB; ++j) {
          float x[8];
          bf16x8_to_f32(tile_chunk(kt, r0 + j, hl), x);
#pragma unroll
          for (int h = 0; h < HG; ++h) {
            float2 acc = __fmul2_rn(q2[h][0], make_float2(x[0], x[1]));
            acc = __ffma2_rn(q2[h][1], make_float2(x[2], x[3]), acc);
            acc = __ffma2_rn(q2[h][2], make_float2(x[4], x[5]), acc);
            acc = __ffma2_rn(q2[h][3], make_float2(x[6], x[7]), acc);
            part[j][h] = acc.x + acc.y;
          }
        }
        // reduce-scatter over the 16 lanes: value index v = j*HG + h ends in lane v
        float v8[8], v4[4], v2[2], s;
#pragma unroll
        for (int i = 0; i < 8; ++i) {  // exchange with lane ^ 8: keep the half selected by bit 3
          const float mine = (hl & 8) ? part[(i + 8) / HG][(i + 8) % HG] : part[i / HG][i % HG];
          const float other = (hl & 8) ? part[i / HG][i % HG] : part[(i + 8) / HG][(i + 8) % HG];
          v8[i] = mine + __shfl_xor_sync(0xffffffffu, other, 8);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float mine = (hl & 4) ? v8[i + 4] : v8[i];
          const float other = (hl & 4) ? v8[i] : v8[i + 4];
          v4[i] = mine + __shfl_xor_sync(0xffffffffu, other, 4);
        }
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const float mine = (hl & 2) ? v4[i + 2] : v4[i];
          const float other = (hl & 2) ? v4[i] : v4[i + 2];
          v2[i] = mine + __shfl_xor_sync(0xffffffffu, other, 2);
        }
        {
          const float mine = (hl & 1) ? v2[1] : v2[0];
          const float other = (hl & 1) ? v2[0] : v2[1];
          s = mine + __shfl_xor_sync(0xffffffffu, other, 1);
        }
        // s is the score of (key r0 + my_key, head my_head); mask rows past the sequence
        const bool valid = k0 + r0 + my_key < w.end;
        if (!valid) s = -INFINITY;
        // per-head maximum over the 4 keys (lanes my_head, +4, +8, +12)
        float mx = fmaxf(s, __shfl_xor_sync(0xffffffffu, s, 4));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
        float alpha[HG];
        float m_ref_own = 0.f;
#pragma unroll
        for (int h = 0; h < HG; ++h) {
          const float mh = __shfl_sync(0xffffffffu, mx, h, 16);
          const float m_new = fmaxf(m_run[h], mh);
          const float m_ref = (m_new == -INFINITY) ? 0.f : m_new;  // no valid key yet: weights stay 0
          alpha[h] = fast_exp2(m_run[h] - m_ref);
          m_run[h] = m_new;
          if (h == my_head) m_ref_own = m_ref;
        }
        const float p = fast_exp2(s - m_ref_own);
        float psum = p + __shfl_xor_sync(0xffffffffu, p, 4);
        psum += __shfl_xor_sync(0xffffffffu, psum, 8);
        float alpha_own = alpha[0];
#pragma unroll
        for (int h = 1; h < HG; ++h)
          if (h == my_head) alpha_own = alpha[h];
        l_own = l_own * alpha_own + psum;
#pragma unroll
        for (int h = 0; h < HG; ++h) {
          const float2 a2 = make_float2(alpha[h], alpha[h]);
#pragma unroll
          for (int q = 0; q < 4; ++q) o2[h][q] = __fmul2_rn(o2[h][q], a2);
        }
        // O += P V over this half-warp's keys.  Rows past the sequence may hold
        // anything (even NaN): they are read as zero, and their weight is 0.
#pragma unroll
        for (int j = 0; j < NB; ++j) {
          float x[8];
          if (k0 + r0 + j < w.end) {
            bf16x8_to_f32(tile_chunk(vt, r0 + j, hl), x);
          } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) x[e] = 0.f;
          }
#pragma unroll
          for (int h = 0; h < HG; ++h) {
            const float pj = __shfl_sync(0xffffffffu, p, j * HG + h, 16);
            const float2 p2 = make_float2(pj, pj);
#pragma unroll
            for (int q = 0; q < 4; ++q) o2[h][q] = __ffma2_rn(p2, make_float2(x[2 * q], x[2 * q + 1]), o2[h][q]);
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->empty[st]);
        if (++st == kStages) { st = 0; ph ^= 1; }
      }
      if (!__all_sync(0xffffffffu, ok)) break;

      // merge the 16 half-warps of the CTA and write this unit's partial per head
      if (!consumer_sync(&bars->merge, mph, wc)) break;  // previous unit's merge has finished reading
#pragma unroll
      for (int h = 0; h < HG; ++h) {
        float* dst = red_o + (hw * HG + h) * D + hl * 8;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          dst[2 * q] = o2[h][q].x;
          dst[2 * q + 1] = o2[h][q].y;
        }
        if (hl == 0) red_m[hw * HG + h] = m_run[h];
      }
      if (hl < HG) red_l[hw * HG + hl] = l_own;  // lane hl < 4 owns head hl (my_head == hl, my_key == 0)
      if (!consumer_sync(&bars->merge, mph, wc)) break;
      const int t = threadIdx.x - 32;
      for (int idx = t; idx < HG * D; idx += 32 * kConsumerWarps) {
        const int h = idx / D, d = idx % D;
        float M = -INFINITY;
#pragma unroll
        for (int x = 0; x < 16; ++x) M = fmaxf(M, red_m[x * HG + h]);
        float num = 0.f, den = 0.f;
#pragma unroll
        for (int x = 0; x < 16; ++x) {
          const float mx2 = red_m[x * HG + h];
          if (mx2 == -INFINITY) continue;
          const float sc = fast_exp2(mx2 - M);
          num = fmaf(red_o[(x * HG + h) * D + d], sc, num);
          den = fmaf(red_l[x * HG + h], sc, den);
        }
        const long long slot = (static_cast<long long>(w.b) * a.n_h + w.h0 + h) * a.n_split + w.start / a.chunk;
        a.ws_o[slot * D + d] = num / den;
        if (d == 0) a.ws_lse[slot] = M + log2f(den);
      }
    }
  }
  __syncthreads();
}

}  // namespace

bool decode_stream_supported(int n_h, int n_kv, int D_qk, int D_v, bool bf16) {
  return bf16 && D_qk == D && D_v == D && ((n_h / n_kv) % HG) == 0;
}

cudaError_t launch_decode_stream(const DecodeArgs& a, const RopeFreq& rope, const CUtensorMap* maps, int num_sms,
                                 cudaStream_t st, int* launches) {
  cudaError_t e = cudaFuncSetAttribute(decode_stream_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  const long long units = static_cast<long long>(a.B) * a.n_kv * ((a.n_h / a.n_kv) / HG) * a.n_split;
  const int grid = static_cast<int>(units < num_sms ? units : num_sms);
  decode_stream_kernel<<<grid, kThreads, kSmemBytes, st>>>(a, rope, maps[0], maps[1]);
  *launches += 1;
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_decode_combine(a, true, st, launches);
}

}  // namespace attn

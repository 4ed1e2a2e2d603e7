// prefill_tc.cu - causal prefill on the 5th-generation tensor cores (sm_103a).
//
// FlashAttention-style tiling ("Transformer架构完全深度解析" §13): Q is cut into
// 128-row tiles, K/V into 128-key tiles; for every (Q tile, KV tile) pair the
// score tile S = Q K^T is formed on chip, folded into the running maximum m and
// running sum l of the online softmax, and P V is added to the output
// accumulator, so S never reaches HBM.  Key tiles that lie wholly after a query
// tile are skipped by index ("2.7 Transformer Decoder Block完整解析" §3.3); only
// the diagonal tile applies the -inf mask.
//
// GB300 mapping (one persistent CTA per SM, 384 threads):
//   warp 0      TMA producer: Q tiles once per work item, K/V tiles through a
//               ring of shared-memory stages (128-byte swizzle).
//   warp 1      allocates 512 TMEM columns; lane 0 issues every tcgen05.mma:
//               S_t = Q_t K_j^T (A, B from shared memory) and O_t += P_t V_j
//               (P read from TMEM, V from shared memory as an MN-major operand).
//   warps 4-7   softmax warpgroup of Q tile 0, warps 8-11 of Q tile 1: each thread
//               owns one query row (TMEM lane), so row max / row sum need no
//               shuffles.  P is written back over S in TMEM as bf16.  The output
//               is rescaled only when the row maximum grows by more than 2^8
//               (exact: l and O always share the same reference maximum).
//   A work item is two adjacent Q tiles of one (batch, head); while one
//   warpgroup computes its softmax, the tensor core runs the other tile's MMAs.
//   Items are taken heaviest-first (latest Q tiles see the most keys).
// RoPE: the query tile is rotated in shared memory right after its TMA load
// (once per item); keys arrive already rotated (written once by the rope pass).
// TMEM columns: [0,128) S/P of tile 0, [128,256) S/P of tile 1,
//               [256, 256+D) O of tile 0, [256+D, 256+2D) O of tile 1.
#include <math.h>

#include "kernels.h"

namespace attn {
namespace {

constexpr int BM = 128;  // query rows per Q tile
constexpr int BN = 128;  // keys per KV tile
constexpr int kThreads = 384;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

template <int D>
struct Cfg {
  static constexpr int kDBlocks = D / 64;         // 64-element (128-byte) column blocks
  static constexpr int kTileBytes = BM * D * 2;   // one bf16 Q, K or V tile
  static constexpr int kBlockBytes = BM * 128;    // one column block of a tile
  static constexpr int kStages = (D == 64) ? 3 : 2;
  static constexpr int kQOff = 0;
  static constexpr int kKOff = kQOff + 2 * kTileBytes;
  static constexpr int kVOff = kKOff + kStages * kTileBytes;
  static constexpr int kBarOff = kVOff + kStages * kTileBytes;
  static constexpr int kSmemBytes = kBarOff + 512 + 1024;  // barriers + alignment slack
  static constexpr uint32_t kOCol0 = 256;
  static constexpr uint32_t kIdescQK = idesc_bf16_f32(BM, BN, false);
  static constexpr uint32_t kIdescPV = idesc_bf16_f32(BM, D, true);
};

struct Bars {
  uint64_t q_full[2], q_ready[2], q_empty[2];
  uint64_t s_full[2], p_full[2], o_done[2], o_empty[2];
  uint64_t k_full[3], k_empty[3], v_full[3], v_empty[3];
  uint64_t fin;
  uint32_t tmem_base;
  int abort_flag;
};

// Key tiles of one Q tile: [0, ns) (attention-sink tiles kept outside the
// window) followed by [jl, jh] (the window up to the diagonal).  Without a
// window ns = 0, jl = 0 and jh is the last tile at or before the diagonal.
struct TileRange {
  int ns, jl, jh;
  __device__ __forceinline__ int count() const { return ns + jh - jl + 1; }
  __device__ __forceinline__ bool has(int j) const { return j < ns || (j >= jl && j <= jh); }
  __device__ __forceinline__ int at(int i) const { return i < ns ? i : jl + i - ns; }  // i-th tile
};

struct Item {
  int b, h, g, qt0;
  TileRange r0, r1;  // the two Q tiles
  int ns_u, n_load;  // loaded tiles: [0, ns_u) then [r0.jl, r1.jh]
  __device__ __forceinline__ int load_at(int v) const { return v < ns_u ? v : r0.jl + v - ns_u; }
};

__device__ __forceinline__ TileRange tile_range(int qt, const PrefillArgs& a, int n_kt) {
  TileRange r;
  if (!a.causal) {
    r.ns = 0;
    r.jl = 0;
    r.jh = n_kt - 1;
    return r;
  }
  const int first_pos = a.q_offset + qt * BM;
  const int last_pos = a.q_offset + min(qt * BM + BM - 1, a.S - 1);
  r.jh = last_pos / BN;
  if (a.window > 0) {
    r.jl = max(0, first_pos - a.window + 1) / BN;
    r.ns = min((a.n_sink + BN - 1) / BN, r.jl);
  } else {
    r.jl = 0;
    r.ns = 0;
  }
  return r;
}

__device__ __forceinline__ Item decode_item(int idx, const PrefillArgs& a, int n_pairs_q, int n_kt) {
  Item it;
  const int bh_count = a.B * a.n_h;
  const int p = n_pairs_q - 1 - idx / bh_count;  // heaviest (latest) tile pairs first
  const int bh = idx % bh_count;
  it.b = bh / a.n_h;
  it.h = bh % a.n_h;
  it.g = it.h / (a.n_h / a.n_kv);
  it.qt0 = 2 * p;
  it.r0 = tile_range(it.qt0, a, n_kt);
  it.r1 = tile_range(it.qt0 + 1, a, n_kt);
  // tile 1's window starts no earlier and ends no earlier than tile 0's, and its
  // sink tiles beyond tile 0's lie inside tile 0's window, so the union is:
  it.ns_u = it.r0.ns;
  it.n_load = it.ns_u + it.r1.jh - it.r0.jl + 1;
  return it;
}

// Wait that ignores the CTA abort flag but still gives up after limit_ns; used
// only to drain copies / MMAs in flight before the CTA exits.
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity, unsigned long long limit_ns) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > limit_ns) return;
  }
}

// Every lane waits, then the warp agrees: a give-up on any lane is a give-up
// for the whole warp, so warp-collective tcgen05 instructions after the wait
// are always executed by all 32 lanes or by none.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, const WaitCtl& w) {
  const bool ok = mbar_wait(bar, parity, w);
  return __all_sync(0xffffffffu, ok);
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_tc_kernel(const __grid_constant__ PrefillArgs a, const __grid_constant__ RopeFreq f,
                      const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v) {
  using C = Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Bars* bars = reinterpret_cast<Bars*>(smem + C::kBarOff);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const int n_qt = (a.S + BM - 1) / BM;
  const int n_kt = (a.S_k + BN - 1) / BN;
  const int n_pairs_q = (n_qt + 1) / 2;
  const int n_items = a.B * a.n_h * n_pairs_q;

  if (threadIdx.x == 0) {
    for (int t = 0; t < 2; ++t) {
      mbar_init(&bars->q_full[t], 1);
      mbar_init(&bars->q_ready[t], 128);
      mbar_init(&bars->q_empty[t], 128);
      mbar_init(&bars->s_full[t], 1);
      mbar_init(&bars->p_full[t], 128);
      mbar_init(&bars->o_done[t], 1);
      mbar_init(&bars->o_empty[t], 128);
    }
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&bars->k_full[s], 1);
      mbar_init(&bars->k_empty[s], 1);
      mbar_init(&bars->v_full[s], 1);
      mbar_init(&bars->v_empty[s], 1);
    }
    mbar_init(&bars->fin, 1);
    bars->abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&bars->tmem_base, 512);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  const WaitCtl wc{&bars->abort_flag, a.status, a.wait_limit_ns};

  // Q tile t lives at smem + kQOff + t * kTileBytes (arithmetic, not an array:
  // runtime-indexed local arrays would live in local memory)
  auto q_smem = [&](int t) { return smem + C::kQOff + t * C::kTileBytes; };

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      uint32_t kst = 0, kph = 0, vst = 0, vph = 0;
      uint32_t k_issued = 0, v_issued = 0;  // bit s: stage s has had a load issued
      uint32_t k_last_ph = 0, v_last_ph = 0;  // bit s: phase parity of that load
      uint32_t q_issued = 0;
      uint32_t it = 0;
      for (int idx = blockIdx.x; idx < n_items; idx += gridDim.x, ++it) {
        const Item itm = decode_item(idx, a, n_pairs_q, n_kt);
        for (int t = 0; t < 2; ++t) {
          if (!mbar_wait(&bars->q_empty[t], (it & 1) ^ 1, wc)) goto producer_done;
          mbar_arrive_expect_tx(&bars->q_full[t], C::kTileBytes);
          for (int db = 0; db < C::kDBlocks; ++db)
            tma_load_4d(q_smem(t) + db * C::kBlockBytes, &tm_q, &bars->q_full[t], db * 64, itm.h,
                        (itm.qt0 + t) * BM, itm.b);
          q_issued = it + 1;
        }
        for (int v = 0; v < itm.n_load; ++v) {
          const int j = itm.load_at(v);
          if (!mbar_wait(&bars->k_empty[kst], kph ^ 1, wc)) goto producer_done;
          mbar_arrive_expect_tx(&bars->k_full[kst], C::kTileBytes);
          uint8_t* kdst = smem + C::kKOff + kst * C::kTileBytes;
          for (int db = 0; db < C::kDBlocks; ++db)
            tma_load_4d(kdst + db * C::kBlockBytes, &tm_k, &bars->k_full[kst], db * 64, itm.g, j * BN, itm.b);
          k_issued |= 1u << kst;
          k_last_ph = (k_last_ph & ~(1u << kst)) | (kph << kst);
          if (++kst == C::kStages) { kst = 0; kph ^= 1; }

          if (!mbar_wait(&bars->v_empty[vst], vph ^ 1, wc)) goto producer_done;
          mbar_arrive_expect_tx(&bars->v_full[vst], C::kTileBytes);
          uint8_t* vdst = smem + C::kVOff + vst * C::kTileBytes;
          for (int db = 0; db < C::kDBlocks; ++db)
            tma_load_4d(vdst + db * C::kBlockBytes, &tm_v, &bars->v_full[vst], db * 64, itm.g, j * BN, itm.b);
          v_issued |= 1u << vst;
          v_last_ph = (v_last_ph & ~(1u << vst)) | (vph << vst);
          if (++vst == C::kStages) { vst = 0; vph ^= 1; }
        }
      }
    producer_done:
      if (bars->abort_flag) {  // let every copy in flight land before shared memory goes away
        for (int s = 0; s < C::kStages; ++s) {
          if (k_issued & (1u << s)) drain_wait(&bars->k_full[s], (k_last_ph >> s) & 1, a.wait_limit_ns);
          if (v_issued & (1u << s)) drain_wait(&bars->v_full[s], (v_last_ph >> s) & 1, a.wait_limit_ns);
        }
        if (q_issued)
          for (int t = 0; t < 2; ++t) drain_wait(&bars->q_full[t], (q_issued - 1) & 1, a.wait_limit_ns);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t q_addr0 = smem_u32(q_smem(0));
      uint32_t kst = 0, kph = 0, vst = 0, vph = 0;
      uint32_t pph0 = 0u, pph1 = 0u;
      uint32_t it = 0;
      auto issue_qk = [&](int t, uint32_t stage) {
        const uint32_t kbase = smem_u32(smem + C::kKOff + stage * C::kTileBytes);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * C::kBlockBytes + (kk & 3) * 32;
          mma_ss(tmem + t * 128u, sdesc_sw128(q_addr0 + t * C::kTileBytes + off, 16, 1024),
                 sdesc_sw128(kbase + off, 16, 1024), C::kIdescQK, kk > 0 ? 1u : 0u);
        }
      };
      auto issue_pv = [&](int t, uint32_t stage, bool accumulate) {
        const uint32_t vbase = smem_u32(smem + C::kVOff + stage * C::kTileBytes);
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk) {
          mma_ts(tmem + C::kOCol0 + t * D, tmem + t * 128u + kk * 8,
                 sdesc_sw128(vbase + kk * 16 * 128, C::kBlockBytes, 1024), C::kIdescPV,
                 (accumulate || kk > 0) ? 1u : 0u);
        }
      };
      for (int idx = blockIdx.x; idx < n_items; idx += gridDim.x, ++it) {
        const Item itm = decode_item(idx, a, n_pairs_q, n_kt);
        // Loaded tile v feeds Q tile t when t's range has it.  Per loaded tile:
        // P V of every member tile, then QK of the next loaded tile for its
        // members (so S_t is reused only after P_t was consumed; MMAs run in order).
        bool q_seen0 = false, q_seen1 = false, pv_seen0 = false, pv_seen1 = false;
        if (!mbar_wait(&bars->k_full[kst], kph, wc)) goto mma_done;
        {
          const int j0 = itm.load_at(0);
          for (int t = 0; t < 2; ++t) {
            if (!(t ? itm.r1 : itm.r0).has(j0)) continue;
            if (!mbar_wait(&bars->q_ready[t], it & 1, wc)) goto mma_done;
            (t ? q_seen1 : q_seen0) = true;
            tc_fence_after();
            issue_qk(t, kst);
            mma_commit(&bars->s_full[t]);
          }
        }
        mma_commit(&bars->k_empty[kst]);
        if (++kst == C::kStages) { kst = 0; kph ^= 1; }
        for (int v = 0; v < itm.n_load; ++v) {
          const int j = itm.load_at(v);
          const bool next = v + 1 < itm.n_load;
          const int jn = next ? itm.load_at(v + 1) : -1;
          if (!mbar_wait(&bars->v_full[vst], vph, wc)) goto mma_done;
          bool k_ready = false;
          for (int t = 0; t < 2; ++t) {
            const TileRange& r = t ? itm.r1 : itm.r0;
            if (r.has(j)) {
              if (!mbar_wait(&bars->p_full[t], t ? pph1 : pph0, wc)) goto mma_done;
              if (t) pph1 ^= 1; else pph0 ^= 1;
              const bool seen = t ? pv_seen1 : pv_seen0;
              if (!seen && !mbar_wait(&bars->o_empty[t], (it & 1) ^ 1, wc)) goto mma_done;
              tc_fence_after();
              issue_pv(t, vst, seen);
              if (t) pv_seen1 = true; else pv_seen0 = true;
              if (j == r.jh) mma_commit(&bars->o_done[t]);
            }
            if (t == 1) {
              mma_commit(&bars->v_empty[vst]);
              if (++vst == C::kStages) { vst = 0; vph ^= 1; }
            }
            if (next && r.has(jn)) {
              if (!k_ready) {
                if (!mbar_wait(&bars->k_full[kst], kph, wc)) goto mma_done;
                k_ready = true;
              }
              const bool qs = t ? q_seen1 : q_seen0;
              if (!qs && !mbar_wait(&bars->q_ready[t], it & 1, wc)) goto mma_done;
              if (t) q_seen1 = true; else q_seen0 = true;
              tc_fence_after();
              issue_qk(t, kst);
              mma_commit(&bars->s_full[t]);
            }
          }
          if (next) {
            mma_commit(&bars->k_empty[kst]);
            if (++kst == C::kStages) { kst = 0; kph ^= 1; }
          }
        }
      }
    mma_done:
      // every MMA issued so far completes before TMEM is released
      mma_commit(&bars->fin);
      drain_wait(&bars->fin, 0, a.wait_limit_ns);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax warpgroups
    const int t = (warp - 4) >> 2;     // Q tile of this warpgroup
    const int quad = warp & 3;         // TMEM lane quadrant
    const int r = quad * 32 + lane;    // query row within the tile
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t s_addr = tmem + lane_off + (t ? 128u : 0u);
    const uint32_t o_addr = tmem + lane_off + C::kOCol0 + (t ? D : 0);
    uint32_t sph = 0;
    uint32_t it = 0;
    for (int idx = blockIdx.x; idx < n_items; idx += gridDim.x, ++it) {
      const Item itm = decode_item(idx, a, n_pairs_q, n_kt);
      const int qt = itm.qt0 + t;
      const TileRange rng = t ? itm.r1 : itm.r0;
      const int n_t = rng.count();
      const int m = qt * BM + r;  // query row
      const int pos = a.q_offset + m;  // its absolute position
      if (!warp_wait(&bars->q_full[t], it & 1, wc)) break;
      if (f.n_pairs) {
        // rotate this thread's query row in place (swizzled layout: the 16-byte
        // chunk c of row r sits at chunk c ^ (r & 7) of the row's 128-byte line)
        uint8_t* row = q_smem(t) + r * 128;
#pragma unroll 1
        for (int c = 0; c < D / 8; ++c) {
          uint4* p = reinterpret_cast<uint4*>(row + (c >> 3) * C::kBlockBytes + (((c & 7) ^ (r & 7)) << 4));
          float x[8];
          bf16x8_to_f32(*p, x);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            float sn, cs;
            rope_sincos(pos, f.hi[c * 4 + e], f.lo[c * 4 + e], &sn, &cs);
            rotate_pair(x[2 * e], x[2 * e + 1], sn, cs);
          }
          *p = f32_to_bf16x8(x);
        }
        fence_proxy_async_smem();
      }
      mbar_arrive(&bars->q_ready[t]);

      float m_run = -INFINITY, l_run = 0.f;
      bool ok = true;
      for (int i = 0; i < n_t; ++i) {
        const int j = rng.at(i);  // key tile
        if (!warp_wait(&bars->s_full[t], sph, wc)) { ok = false; break; }
        sph ^= 1;
        tc_fence_after();
        uint32_t sr[BN];
#pragma unroll
        for (int c = 0; c < BN / 32; ++c) tmem_ld32(s_addr + c * 32, sr + c * 32);
        tmem_wait_ld();
        float s[BN];
#pragma unroll
        for (int c = 0; c < BN; ++c) s[c] = __uint_as_float(sr[c]);
        const int key0 = j * BN;
        const int tile_pos0 = a.q_offset + qt * BM;  // position of the Q tile's first row
        if (a.window > 0 && tile_pos0 + BM - 1 - key0 >= a.window && key0 + BN > a.n_sink) {
          // some key of this tile is outside some row's window (and not a sink)
#pragma unroll
          for (int c = 0; c < BN; ++c) {
            const int key = key0 + c;
            if (key > pos || (pos - key >= a.window && key >= a.n_sink)) s[c] = -INFINITY;
          }
        } else if (a.causal && key0 + BN - 1 > tile_pos0) {
          // some key of this tile lies after some query of the Q tile: mask key > position
#pragma unroll
          for (int c = 0; c < BN; ++c)
            if (key0 + c > pos) s[c] = -INFINITY;
        } else if (!a.causal && key0 + BN > a.S_k) {
#pragma unroll
          for (int c = 0; c < BN; ++c)
            if (key0 + c >= a.S_k) s[c] = -INFINITY;
        }
        // row maximum: 8 independent chains, then a tree (a single chain of 127
        // dependent max operations would dominate the warp's latency)
        float m8[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) m8[i] = s[i];
#pragma unroll
        for (int c = 8; c < BN; ++c) m8[c & 7] = fmaxf(m8[c & 7], s[c]);
#pragma unroll
        for (int w2 = 4; w2 > 0; w2 >>= 1)
#pragma unroll
          for (int i = 0; i < w2; ++i) m8[i] = fmaxf(m8[i], m8[i + w2]);
        const float mx = m8[0] * a.scale_log2;
        // Move to a new reference maximum only when the row maximum grew by more
        // than the threshold; O and l are then scaled by alpha = 2^(m_old - m_new).
        const bool need = mx > m_run + kRescaleThreshold;
        float alpha = 1.f;
        if (need) {
          if (i > 0) alpha = fast_exp2(m_run - mx);
          l_run *= alpha;
          m_run = mx;
        }
        // p = 2^(s * scale*log2e - m), two columns per packed fp32x2 FMA; the row
        // sum runs in 4 independent packed accumulators
        uint32_t pr[BN / 2];
        const float2 sl2 = make_float2(a.scale_log2, a.scale_log2);
        // a row whose tiles so far held no visible key keeps m = -inf: its
        // weights are 0 (reference 0 avoids -inf - -inf)
        const float m_ref = (m_run == -INFINITY) ? 0.f : m_run;
        const float2 nm2 = make_float2(-m_ref, -m_ref);
        float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
        for (int c = 0; c < BN / 2; ++c) {
          const float2 x = __ffma2_rn(make_float2(s[2 * c], s[2 * c + 1]), sl2, nm2);
          const float2 pp = make_float2(fast_exp2(x.x), fast_exp2(x.y));
          acc[c & 3] = __fadd2_rn(acc[c & 3], pp);
          pr[c] = pack_bf16x2(pp.x, pp.y);
        }
        acc[0] = __fadd2_rn(__fadd2_rn(acc[0], acc[1]), __fadd2_rn(acc[2], acc[3]));
        l_run += acc[0].x + acc[0].y;
        tmem_st32(s_addr, pr);
        tmem_st32(s_addr + 32, pr + 32);
        // O rescale, once the scores are dead (fewer live registers).  P V(j-1)
        // has completed (s_full of tile j was committed after it), P V(j) waits
        // for p_full below.  TMEM loads/stores are warp-collective: the whole
        // warp rescales when any of its rows needs it (alpha is 1 for the others).
        if (__any_sync(0xffffffffu, need && i > 0)) {
#pragma unroll 1
          for (int c = 0; c < D / 32; ++c) {
            uint32_t orow[32];
            tmem_ld32(o_addr + c * 32, orow);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) orow[e] = __float_as_uint(__uint_as_float(orow[e]) * alpha);
            tmem_st32(o_addr + c * 32, orow);
          }
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&bars->p_full[t]);
      }
      if (!ok) break;

      // epilogue: O / l -> out (rows past S are computed but not stored)
      if (!warp_wait(&bars->o_done[t], it & 1, wc)) break;
      tc_fence_after();
      mbar_arrive(&bars->q_empty[t]);  // every MMA reading Q_t has completed
      const float inv_l = 1.f / l_run;
      const bool store = m < a.S;
      __nv_bfloat16* orow_g = static_cast<__nv_bfloat16*>(a.out) +
                              ((static_cast<long long>(itm.b) * a.S + m) * a.n_h + itm.h) * D;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t orow[32];
        tmem_ld32(o_addr + c * 32, orow);
        tmem_wait_ld();
        if (store) {
          uint32_t packed[16];
#pragma unroll
          for (int e = 0; e < 16; ++e)
            packed[e] = pack_bf16x2(__uint_as_float(orow[2 * e]) * inv_l, __uint_as_float(orow[2 * e + 1]) * inv_l);
          uint4* dst = reinterpret_cast<uint4*>(orow_g + c * 32);
#pragma unroll
          for (int e = 0; e < 4; ++e)
            dst[e] = make_uint4(packed[4 * e], packed[4 * e + 1], packed[4 * e + 2], packed[4 * e + 3]);
        }
      }
      tc_fence_before();
      mbar_arrive(&bars->o_empty[t]);
      if (store && a.lse != nullptr)
        a.lse[(static_cast<long long>(itm.b) * a.n_h + itm.h) * a.S + m] =
            (m_run + log2f(l_run)) * 0.69314718055994530942f;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

bool prefill_tc_supported(int D, bool bf16) { return bf16 && (D == 64 || D == 128); }

cudaError_t launch_prefill_tc(const PrefillArgs& a, const RopeFreq& rope, const CUtensorMap* maps, int num_sms,
                              cudaStream_t st, int* launches) {
  const int n_qt = (a.S + BM - 1) / BM;
  const long long n_items = static_cast<long long>(a.B) * a.n_h * ((n_qt + 1) / 2);
  const int grid = static_cast<int>(n_items < num_sms ? n_items : num_sms);
  cudaError_t e;
  if (a.D == 64) {
    auto k = prefill_tc_kernel<64>;
    e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<64>::kSmemBytes);
    if (e != cudaSuccess) return e;
    k<<<grid, kThreads, Cfg<64>::kSmemBytes, st>>>(a, rope, maps[0], maps[1], maps[2]);
  } else {
    auto k = prefill_tc_kernel<128>;
    e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<128>::kSmemBytes);
    if (e != cudaSuccess) return e;
    k<<<grid, kThreads, Cfg<128>::kSmemBytes, st>>>(a, rope, maps[0], maps[1], maps[2]);
  }
  *launches += 1;
  return cudaGetLastError();
}

}  // namespace attn

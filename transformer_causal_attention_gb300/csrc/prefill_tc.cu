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

struct Item {
  int b, h, g, qt0, n0, n1;
};

// Key tiles a causal Q tile needs: up to the tile holding its last query's position.
__device__ __forceinline__ int causal_tiles(int qt, const PrefillArgs& a) {
  const int last_row = min(qt * BM + BM - 1, a.S - 1);
  return (a.q_offset + last_row) / BN + 1;
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
  if (a.causal) {
    it.n0 = causal_tiles(it.qt0, a);
    it.n1 = causal_tiles(it.qt0 + 1, a);
  } else {
    it.n0 = it.n1 = n_kt;
  }
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

  uint8_t* q_smem[2] = {smem + C::kQOff, smem + C::kQOff + C::kTileBytes};

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
            tma_load_4d(q_smem[t] + db * C::kBlockBytes, &tm_q, &bars->q_full[t], db * 64, itm.h,
                        (itm.qt0 + t) * BM, itm.b);
          q_issued = it + 1;
        }
        for (int j = 0; j < itm.n1; ++j) {
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
      const uint32_t s_col[2] = {0u, 128u};
      const uint32_t o_col[2] = {C::kOCol0, C::kOCol0 + D};
      uint32_t q_addr[2] = {smem_u32(q_smem[0]), smem_u32(q_smem[1])};
      uint32_t kst = 0, kph = 0, vst = 0, vph = 0;
      uint32_t pph[2] = {0u, 0u};
      uint32_t it = 0;
      auto issue_qk = [&](int t, uint32_t stage) {
        const uint32_t kbase = smem_u32(smem + C::kKOff + stage * C::kTileBytes);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * C::kBlockBytes + (kk & 3) * 32;
          mma_ss(tmem + s_col[t], sdesc_sw128(q_addr[t] + off, 16, 1024), sdesc_sw128(kbase + off, 16, 1024),
                 C::kIdescQK, kk > 0 ? 1u : 0u);
        }
      };
      auto issue_pv = [&](int t, uint32_t stage, bool accumulate) {
        const uint32_t vbase = smem_u32(smem + C::kVOff + stage * C::kTileBytes);
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk) {
          mma_ts(tmem + o_col[t], tmem + s_col[t] + kk * 8, sdesc_sw128(vbase + kk * 16 * 128, C::kBlockBytes, 1024),
                 C::kIdescPV, (accumulate || kk > 0) ? 1u : 0u);
        }
      };
      for (int idx = blockIdx.x; idx < n_items; idx += gridDim.x, ++it) {
        const Item itm = decode_item(idx, a, n_pairs_q, n_kt);
        // first key tile: S_0 and S_1
        if (!mbar_wait(&bars->k_full[kst], kph, wc)) goto mma_done;
        for (int t = 0; t < 2; ++t) {
          if (!mbar_wait(&bars->q_ready[t], it & 1, wc)) goto mma_done;
          tc_fence_after();
          issue_qk(t, kst);
          mma_commit(&bars->s_full[t]);
        }
        mma_commit(&bars->k_empty[kst]);
        if (++kst == C::kStages) { kst = 0; kph ^= 1; }
        for (int j = 0; j < itm.n1; ++j) {
          if (!mbar_wait(&bars->v_full[vst], vph, wc)) goto mma_done;
          if (j < itm.n0) {
            if (!mbar_wait(&bars->p_full[0], pph[0], wc)) goto mma_done;
            pph[0] ^= 1;
            if (j == 0 && !mbar_wait(&bars->o_empty[0], (it & 1) ^ 1, wc)) goto mma_done;
            tc_fence_after();
            issue_pv(0, vst, j > 0);
            if (j == itm.n0 - 1) mma_commit(&bars->o_done[0]);
          }
          const bool next = j + 1 < itm.n1;
          if (next) {
            if (!mbar_wait(&bars->k_full[kst], kph, wc)) goto mma_done;
            tc_fence_after();
            if (j + 1 < itm.n0) {
              issue_qk(0, kst);
              mma_commit(&bars->s_full[0]);
            }
          }
          if (!mbar_wait(&bars->p_full[1], pph[1], wc)) goto mma_done;
          pph[1] ^= 1;
          if (j == 0 && !mbar_wait(&bars->o_empty[1], (it & 1) ^ 1, wc)) goto mma_done;
          tc_fence_after();
          issue_pv(1, vst, j > 0);
          mma_commit(&bars->v_empty[vst]);
          if (++vst == C::kStages) { vst = 0; vph ^= 1; }
          if (j == itm.n1 - 1) mma_commit(&bars->o_done[1]);
          if (next) {
            issue_qk(1, kst);
            mma_commit(&bars->s_full[1]);
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
      const int n_t = t ? itm.n1 : itm.n0;
      const int m = qt * BM + r;  // query row
      const int pos = a.q_offset + m;  // its absolute position
      if (!warp_wait(&bars->q_full[t], it & 1, wc)) break;
      if (f.n_pairs) {
        // rotate this thread's query row in place (swizzled layout: the 16-byte
        // chunk c of row r sits at chunk c ^ (r & 7) of the row's 128-byte line)
        uint8_t* row = q_smem[t] + r * 128;
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
      for (int j = 0; j < n_t; ++j) {
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
        if (a.causal && key0 + BN - 1 > a.q_offset + qt * BM) {
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
          if (j > 0) alpha = fast_exp2(m_run - mx);
          l_run *= alpha;
          m_run = mx;
        }
        // TMEM loads/stores are warp-collective: the whole warp rescales when any
        // of its rows needs it (alpha is 1 for the others).
        if (__any_sync(0xffffffffu, need && j > 0)) {
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
        // p = 2^(s * scale*log2e - m), two columns per packed fp32x2 FMA; the row
        // sum runs in 4 independent packed accumulators
        uint32_t pr[BN / 2];
        const float2 sl2 = make_float2(a.scale_log2, a.scale_log2);
        const float2 nm2 = make_float2(-m_run, -m_run);
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

// prefill_pair.cu - the MLA prefill (non-absorbed path: q/k head dim 192, v head dim 128) on
// the tensor cores of a CTA pair (sm_103a).
//
// "Transformer 与 LLM" slide 06: the prefill takes the non-absorbed path, per head scores
// q . [k^C ; k^R] over 128 content and 64 rotary dims, and 128-dim values.  The tiling is the
// FlashAttention-style one of prefill_tc.cu ("Transformer架构完全深度解析" §13), with the two
// CTAs of a cluster acting as one tensor-core unit (tcgen05.mma.cta_group::2, issued by the
// even CTA).  A work item is four consecutive 128-row Q tiles of one (batch, head), taken as
// two pair tiles of 256 rows: pair tile A = Q tiles 4p (CTA 0) and 4p + 1 (CTA 1), pair tile
// B = 4p + 2 and 4p + 3.  Per key tile j:
//   S_t = Q_t K_j^T  with M = 256 (each CTA supplies its 128 query rows from its own shared
//                    memory) and N = 128 keys split over the pair: CTA r loads only keys
//                    [64 r, 64 r + 64) of the tile;
//   O_t += P_t V_j   with P from each CTA's own TMEM and N = 128 value dims split over the
//                    pair: CTA r loads only dims [64 r, 64 r + 64) of the tile.
// So each CTA holds half of every K and V tile: with 192-dim keys the shared memory then
// takes three K and V stages next to two Q tiles, where prefill_tc.cu's <192, 128> layout
// has room for one V stage.  The softmax is that of prefill_tc.cu, one thread per query row
// of the CTA's own tile, P handed to the issuer once per key tile; a pair tile's key
// range is the one of its later (CTA 1) tile, so CTA 0 also computes the one key tile after
// its own diagonal, entirely masked.
// Hand-offs to the issuer from the odd CTA's warps are arrivals on the even CTA's barriers
// with a CTA-scope release (pair.cuh): with a cluster-scope release each arrival reached the
// issuer ~0.5 us later and the Llama-shaped instantiation of this kernel took 2.33 ms against
// 1.59 ms.  At head dim 128 (Llama-3-8B shape) the kernel measured 1.59 ms against
// prefill_tc.cu's 1.567 ms, so those heads run there: per key tile the issuer issues 32 pair
// MMAs at ~76 cycles each without waiting for P, the same per-SM tensor time and issue
// overhead as the single-CTA kernel.  On the MLA shape it measured 0.670 ms against 0.683 ms.
// Roles (384 threads, one CTA per SM): warp 0 K producer, warp 1 TMEM owner and (in CTA 0)
// MMA issuer, warp 2 Q and V producer, warp 3 idle, warps 4-7 / 8-11 the softmax warpgroups of
// pair tiles A / B.  Barriers that the issuer waits on live in CTA 0 and count one arrival
// per softmax warp of both CTAs; the commits that free a stage or announce S or O reach both.
// TMEM (512 columns, allocated for the pair): S/P of A and B at 0 and 128, O of A and B at 256
// and 384.
#include <math.h>

#include <atomic>

#include "kernels.h"
#include "pair.cuh"

namespace attn {
namespace {

constexpr int BM = 128;  // query rows per CTA per pair tile
constexpr int BN = 128;  // keys per key tile
constexpr int DQK = 192;  // query / key head dim: 128 content + 64 rotary dims
constexpr int DV = 128;   // value head dim
constexpr int kThreads = 384;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

constexpr int kLaunchRegs = 168;
constexpr int kRegsCtl = 152, kRegsSoftmax = 176;
constexpr int kRegsNeeded = 4 * 32 * kRegsCtl + 8 * 32 * kRegsSoftmax;
static_assert(kRegsNeeded <= kThreads * kLaunchRegs, "register split exceeds the launch's pool");

// Shared memory: every tile in 64-dim (128-byte) column blocks with the 128-byte swizzle.
// Two Q slots (the next item's tile of a slot loads once the slot's last Q K has run) and
// three stages of this CTA's K and V halves: 216 KB.
constexpr int kQBlockBytes = BM * 128;           // one 64-dim block of a Q tile (16 KB)
constexpr int kQTileBytes = BM * DQK * 2;        // 48 KB: 128 rows x 192 dims
constexpr int kKHalfBlock = (BN / 2) * 128;      // 8 KB: 64 keys x 64 dims
constexpr int kKHalfBytes = (DQK / 64) * kKHalfBlock;  // this CTA's half of a K tile: 64 keys x 192 dims
constexpr int kVHalfBytes = BN * 128;            // this CTA's half of a V tile: 128 keys x 64 dims
constexpr int kQSlots = 2, kKStages = 3, kVStages = 3;
constexpr int kQOff = 0;
constexpr int kKOff = kQOff + kQSlots * kQTileBytes;
constexpr int kVOff = kKOff + kKStages * kKHalfBytes;
constexpr int kBarOff = kVOff + kVStages * kVHalfBytes;
constexpr int kFreqOff = kBarOff + 512;
constexpr int kSmemBytes = kFreqOff + 2 * kMaxRopePairs * 4 + 1024;  // + alignment slack
static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");
static_assert(kKOff % 1024 == 0 && kVOff % 1024 == 0, "operand alignment");

constexpr uint32_t kOCol0 = 256;
constexpr uint32_t kIdescQK = idesc_bf16_f32(2 * BM, BN, false);
constexpr uint32_t kIdescPV = idesc_bf16_f32(2 * BM, DV, true);
constexpr uint32_t kWarpArrivals = 8;  // softmax warps of a pair tile in both CTAs

struct Bars {
  uint64_t q_full[kQSlots], q_ready[kQSlots], q_empty[kQSlots];
  uint64_t s_full[2], p_full[2], o_done[2], o_empty[2];
  uint64_t k_full[kKStages], k_empty[kKStages], v_full[kVStages], v_empty[kVStages];
  uint64_t fin;
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(Bars) <= 512, "barrier block");

struct TileRange {
  int jh;  // key tiles [0, jh]
  __device__ __forceinline__ int count() const { return jh + 1; }
  __device__ __forceinline__ bool has(int j) const { return j <= jh; }
};

struct Item {
  int b, h, g, qt0;   // Q tiles qt0 .. qt0 + 3
  TileRange r0, r1;   // pair tiles A and B
  int n_load;         // key tiles [0, n_load)
};

// Key tiles of the 256 query rows starting at Q tile qt.
__device__ __forceinline__ TileRange pair_range(int qt, const PrefillArgs& a, int n_kt) {
  TileRange r;
  if (!a.causal) {
    r.jh = n_kt - 1;
    return r;
  }
  r.jh = (a.q_offset + min(qt * BM + 2 * BM - 1, a.S - 1)) / BN;
  return r;
}

// This pair's k-th item: heaviest-first waves over the pairs, every other wave in reverse order.
__device__ __forceinline__ int item_at(uint32_t k) {
  const int g = static_cast<int>(gridDim.x >> 1), c = static_cast<int>(blockIdx.x >> 1);
  return static_cast<int>(k) * g + ((k & 1u) ? g - 1 - c : c);
}

__device__ __forceinline__ Item decode_item(int idx, const PrefillArgs& a, int n_quads, int n_kt) {
  Item it;
  const int bh_count = a.B * a.n_h;
  const int p = n_quads - 1 - idx / bh_count;  // heaviest (latest) quads first
  const int bh = idx % bh_count;
  it.b = bh / a.n_h;
  it.h = bh % a.n_h;
  it.g = it.h / (a.n_h / a.n_kv);
  it.qt0 = 4 * p;
  it.r0 = pair_range(it.qt0, a, n_kt);
  it.r1 = pair_range(it.qt0 + 2, a, n_kt);
  it.n_load = it.r1.jh + 1;
  return it;
}

// Rotate the span [rope_offset, rope_offset + 2 n_pairs) of query row r (position pos) of a Q
// tile in shared memory (the layout and pairing of prefill_tc.cu's rotation), frequencies from
// shared memory.
__device__ __noinline__ void rotate_row(uint8_t* row, int r, int pos, int rope_offset, int n_pairs, bool half,
                                        const float* f_hi, const float* f_lo) {
  auto chunk = [&](int c) -> uint8_t* { return row + (c >> 3) * kQBlockBytes + (((c & 7) ^ (r & 7)) << 4); };
  const int c0 = rope_offset / 8;
  if (half) {
    const int hc = n_pairs / 8;
#pragma unroll 1
    for (int i = 0; i < hc; ++i) {
      uint4* p0 = reinterpret_cast<uint4*>(chunk(c0 + i));
      uint4* p1 = reinterpret_cast<uint4*>(chunk(c0 + i + hc));
      float x0[8], x1[8];
      bf16x8_to_f32(*p0, x0);
      bf16x8_to_f32(*p1, x1);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        float sn, cs;
        rope_sincos_fast(pos, f_hi[i * 8 + e], f_lo[i * 8 + e], &sn, &cs);
        rotate_pair(x0[e], x1[e], sn, cs);
      }
      *p0 = f32_to_bf16x8(x0);
      *p1 = f32_to_bf16x8(x1);
    }
  } else {
#pragma unroll 1
    for (int i = 0; i < n_pairs / 4; ++i) {
      uint4* p = reinterpret_cast<uint4*>(chunk(c0 + i));
      float x[8];
      bf16x8_to_f32(*p, x);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float sn, cs;
        rope_sincos_fast(pos, f_hi[i * 4 + e], f_lo[i * 4 + e], &sn, &cs);
        rotate_pair(x[2 * e], x[2 * e + 1], sn, cs);
      }
      *p = f32_to_bf16x8(x);
    }
  }
}

__global__ void __launch_bounds__(kThreads, 1)
    prefill_pair_kernel(const __grid_constant__ PrefillArgs a, const __grid_constant__ RopeFreq f,
                        const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k64,
                        const __grid_constant__ CUtensorMap tm_v) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  Bars* bars = reinterpret_cast<Bars*>(smem + kBarOff);
  float* const f_hi = reinterpret_cast<float*>(smem + kFreqOff);
  float* const f_lo = f_hi + kMaxRopePairs;
  for (int i = threadIdx.x; i < f.n_pairs; i += kThreads) {  // made visible by the cluster sync below
    f_hi[i] = f.hi[i];
    f_lo[i] = f.lo[i];
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint32_t r;  // this CTA's rank in the pair
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));

  const int n_qt = (a.S + BM - 1) / BM;
  const int n_kt = (a.S_k + BN - 1) / BN;
  const int n_quads = (n_qt + 3) / 4;
  const int n_items = a.B * a.n_h * n_quads;

  if (threadIdx.x == 0) {
    for (int q = 0; q < kQSlots; ++q) {
      mbar_init(&bars->q_full[q], 1);
      mbar_init(&bars->q_ready[q], kWarpArrivals);
      mbar_init(&bars->q_empty[q], 128);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&bars->s_full[t], 1);
      mbar_init(&bars->p_full[t], kWarpArrivals);
      mbar_init(&bars->o_done[t], 1);
      mbar_init(&bars->o_empty[t], kWarpArrivals);
    }
    for (int s = 0; s < kKStages; ++s) {
      mbar_init(&bars->k_full[s], 1);
      mbar_init(&bars->k_empty[s], 1);
    }
    for (int s = 0; s < kVStages; ++s) {
      mbar_init(&bars->v_full[s], 1);
      mbar_init(&bars->v_empty[s], 1);
    }
    mbar_init(&bars->fin, 1);
    bars->abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(
                     smem_u32(&bars->tmem_base))
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k64);
    tma_prefetch_desc(&tm_v);
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers exist before either signals the other
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  const WaitCtl wc{&bars->abort_flag, a.status, a.wait_limit_ns};

  // Q tile t of this CTA's k-th item lives in slot (2k + t) mod kQSlots (its u-th use, parity u & 1)
  auto q_smem = [&](uint32_t slot) { return smem + kQOff + slot * kQTileBytes; };
  auto q_advance = [](uint32_t& slot, uint32_t& par, uint32_t by) {
    slot += by;
    if (slot >= static_cast<uint32_t>(kQSlots)) {
      slot -= kQSlots;
      par ^= 1u;
    }
  };

  if (warp < 4) {
    setmaxnreg_dec<kRegsCtl>();
    if (warp == 0 || warp == 2) {
      // ------------------------------------------------------------ producers (both CTAs)
      // warp 0: this CTA's half of every K tile (keys [64 r, +64)); warp 2: the CTA's two Q tiles
      // of each item, then its half of every V tile (dims [64 r, +64)).  K and V halves complete
      // on the even CTA's barriers, so the issuer sees a whole tile with one wait.
      if (lane == 0) {
        const bool is_v = warp == 2;
        uint64_t* const full = is_v ? bars->v_full : bars->k_full;
        uint64_t* const empty = is_v ? bars->v_empty : bars->k_empty;
        const int n_stages = is_v ? kVStages : kKStages;
        uint32_t st = 0, ph = 0, issued = 0, last_ph = 0;
        uint32_t q_armed = 0, q_last = 0, it = 0, qs = 0, qp = 0;
        for (int idx = item_at(it); idx < n_items; idx = item_at(++it)) {
          const Item itm = decode_item(idx, a, n_quads, n_kt);
          if (is_v) {
            for (int t = 0; t < 2; ++t, q_advance(qs, qp, 1)) {
              if (!mbar_wait(&bars->q_empty[qs], qp ^ 1, wc)) goto load_done;
              mbar_arrive_expect_tx(&bars->q_full[qs], kQTileBytes);
              for (int db = 0; db < DQK / 64; ++db)
                tma_load_4d(q_smem(qs) + db * kQBlockBytes, &tm_q, &bars->q_full[qs], db * 64, itm.h,
                            (itm.qt0 + 2 * t + static_cast<int>(r)) * BM, itm.b);
              q_armed |= 1u << qs;
              q_last = (q_last & ~(1u << qs)) | (qp << qs);
            }
          }
          for (int v = 0; v < itm.n_load; ++v) {
            if (!wait_cl(&empty[st], ph ^ 1, wc)) goto load_done;
            if (r == 0) mbar_arrive_expect_tx(&full[st], 2 * (is_v ? kVHalfBytes : kKHalfBytes));
            const uint32_t bar0 = cluster_addr(&full[st], 0);
            if (is_v) {
              tma_load_4d_pair(smem + kVOff + st * kVHalfBytes, &tm_v, bar0, 64 * static_cast<int>(r), itm.g, v * BN,
                               itm.b);
            } else {
              for (int db = 0; db < DQK / 64; ++db)
                tma_load_4d_pair(smem + kKOff + st * kKHalfBytes + db * kKHalfBlock, &tm_k64, bar0, db * 64, itm.g,
                                 v * BN + (BN / 2) * static_cast<int>(r), itm.b);
            }
            issued |= 1u << st;
            last_ph = (last_ph & ~(1u << st)) | (ph << st);
            if (++st == static_cast<uint32_t>(n_stages)) { st = 0; ph ^= 1; }
          }
        }
      load_done:
        if (bars->abort_flag) {
          // copies in flight may still land: give them time before the CTA can leave (the K and V
          // barriers may sit in the other CTA, so waiting on them is not always possible here)
          for (int q = 0; q < kQSlots; ++q)
            if (q_armed & (1u << q)) drain_wait_cl(&bars->q_full[q], (q_last >> q) & 1, a.wait_limit_ns);
          if (issued) {
            const uint64_t t0 = globaltimer_ns();
            while (globaltimer_ns() - t0 < 200000ull) {
            }
          }
        }
      }
      __syncwarp();
    } else if (warp == 1) {
      // ------------------------------------------------------------ MMA issuer (CTA 0)
      // Per loaded key tile j, for each pair tile t that needs it: P_t V(j) then Q_t K(j + 1), with
      // the decision-free steady loop, as in prefill_tc.cu.
      if (lane == 0 && r == 0) {
        const uint64_t q_desc0 = sdesc_sw128(smem_u32(q_smem(0)), 16, 1024);
        const uint64_t k_desc0 = sdesc_sw128(smem_u32(smem + kKOff), 16, 1024);
        const uint64_t v_desc0 = sdesc_sw128(smem_u32(smem + kVOff), kQBlockBytes, 1024);
        uint32_t kst = 0, kph = 0, vst = 0, vph = 0, pph0 = 0, pph1 = 0;
        uint32_t it = 0;
        uint32_t qs0 = 0, qp0 = 0;  // slot and parity of the Q tiles of pair tile A of the current item
        // Q_t K over the dims [64 half, 64 half + 64), or all dims (half < 0)
        auto issue_qk_part = [&](int t, uint32_t qslot, uint32_t stage, int half) {
          const uint64_t a0 = q_desc0 + ((qslot * kQTileBytes) >> 4);
          const uint64_t b0 = k_desc0 + ((stage * kKHalfBytes) >> 4);
          const int k_lo = half > 0 ? DQK / 32 : 0, k_hi = half == 0 ? DQK / 32 : DQK / 16;
#pragma unroll
          for (int kk = k_lo; kk < k_hi; ++kk)
            mma_pair(tmem + t * 128u, a0 + (((kk >> 2) * kQBlockBytes + (kk & 3) * 32) >> 4),
                     b0 + (((kk >> 2) * kKHalfBlock + (kk & 3) * 32) >> 4), kIdescQK, kk > 0 ? 1u : 0u);
        };
        auto issue_qk = [&](int t, uint32_t qslot, uint32_t stage) { issue_qk_part(t, qslot, stage, -1); };
        // P_t V over the tile's 128 keys (P of keys [16 kk, 16 kk + 16) in TMEM columns [8 kk, 8 kk + 8)
        // of the tile's S columns)
        auto issue_pv = [&](int t, uint32_t stage, bool accumulate) {
          const uint64_t b0 = v_desc0 + ((stage * kVHalfBytes) >> 4);
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk)
            mma_pair_ts(tmem + kOCol0 + t * DV, tmem + t * 128u + kk * 8, b0 + ((kk * 16 * 128) >> 4), kIdescPV,
                        (accumulate || kk > 0) ? 1u : 0u);
        };
        for (int idx = item_at(it); idx < n_items; idx = item_at(++it)) {
          const Item itm = decode_item(idx, a, n_quads, n_kt);
          bool pv_seen0 = false, pv_seen1 = false;
          uint32_t qs1 = qs0, qp1 = qp0;
          q_advance(qs1, qp1, 1);
          if (!wait_cl(&bars->k_full[kst], kph, wc)) goto mma_done;
          for (int t = 0; t < 2; ++t) {  // key tile 0 is in both pair tiles' ranges
            if (!wait_cl(&bars->q_ready[t ? qs1 : qs0], t ? qp1 : qp0, wc)) goto mma_done;
            tc_fence_after();
            issue_qk(t, t ? qs1 : qs0, kst);
            commit_both(&bars->s_full[t]);
          }
          commit_both(&bars->k_empty[kst]);
          if (++kst == kKStages) { kst = 0; kph ^= 1; }
          // key tiles [vs, ve): both pair tiles take P V(j) and Q K(j + 1), neither at its first
          const int vs = 1, ve = itm.r0.jh;
          for (int v = 0; v < itm.n_load; ++v) {
            if (v == vs && vs < ve) {
              if (!wait_cl(&bars->v_full[vst], vph, wc)) goto mma_done;
              if (!wait_cl(&bars->k_full[kst], kph, wc)) goto mma_done;
              for (; v < ve; ++v) {
                if (!wait_cl(&bars->p_full[0], pph0, wc)) goto mma_done;
                pph0 ^= 1;
                tc_fence_after();
                issue_pv(0, vst, true);
                issue_qk(0, qs0, kst);
                commit_both(&bars->s_full[0]);
                if (!wait_cl(&bars->p_full[1], pph1, wc)) goto mma_done;
                pph1 ^= 1;
                tc_fence_after();
                issue_pv(1, vst, true);
                commit_both(&bars->v_empty[vst]);
                if (++vst == kVStages) { vst = 0; vph ^= 1; }
                issue_qk_part(1, qs1, kst, 0);
                uint32_t kst_n = kst + 1, kph_n = kph;
                if (kst_n == static_cast<uint32_t>(kKStages)) { kst_n = 0; kph_n ^= 1; }
                if (v + 1 < ve) {
                  if (!wait_cl(&bars->v_full[vst], vph, wc)) goto mma_done;
                  if (!wait_cl(&bars->k_full[kst_n], kph_n, wc)) goto mma_done;
                }
                issue_qk_part(1, qs1, kst, 1);
                commit_both(&bars->s_full[1]);
                commit_both(&bars->k_empty[kst]);
                kst = kst_n;
                kph = kph_n;
              }
            }
            const int j = v;
            const bool next = v + 1 < itm.n_load;
            const int jn = v + 1;
            if (!wait_cl(&bars->v_full[vst], vph, wc)) goto mma_done;
            bool k_ready = false;
            for (int t = 0; t < 2; ++t) {
              const TileRange& rg = t ? itm.r1 : itm.r0;
              const bool pv = rg.has(j), qk = next && rg.has(jn);
              if (pv) {
                if (!wait_cl(&bars->p_full[t], t ? pph1 : pph0, wc)) goto mma_done;
                if (t) pph1 ^= 1; else pph0 ^= 1;
                if (!(t ? pv_seen1 : pv_seen0) && !wait_cl(&bars->o_empty[t], (it & 1) ^ 1, wc)) goto mma_done;
              }
              if (qk && !k_ready) {
                if (!wait_cl(&bars->k_full[kst], kph, wc)) goto mma_done;
                k_ready = true;
              }
              tc_fence_after();
              if (pv) {
                issue_pv(t, vst, t ? pv_seen1 : pv_seen0);
                if (t) pv_seen1 = true; else pv_seen0 = true;
                if (j == rg.jh) commit_both(&bars->o_done[t]);
              }
              if (t == 1) {
                commit_both(&bars->v_empty[vst]);
                if (++vst == kVStages) { vst = 0; vph ^= 1; }
              }
              if (qk) {
                issue_qk(t, t ? qs1 : qs0, kst);
                commit_both(&bars->s_full[t]);
              }
            }
            if (next) {
              commit_both(&bars->k_empty[kst]);
              if (++kst == kKStages) { kst = 0; kph ^= 1; }
            }
          }
          q_advance(qs0, qp0, 2);
        }
      mma_done:
        // every MMA issued so far completes before TMEM is released
        commit_local(&bars->fin);
        drain_wait_cl(&bars->fin, 0, a.wait_limit_ns);
      }
      __syncwarp();
    }
  } else {
    setmaxnreg_inc<kRegsSoftmax>();
    // ------------------------------------------------------------ softmax warpgroups (both CTAs)
    const int t = (warp - 4) >> 2;     // pair tile of this warpgroup
    const int quad = warp & 3;         // TMEM lane quadrant
    const int row = quad * 32 + lane;  // query row within this CTA's tile
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t s_addr = tmem + lane_off + (t ? 128u : 0u);
    const uint32_t o_addr = tmem + lane_off + kOCol0 + (t ? DV : 0);
    // the barriers the issuer waits on (in CTA 0): one arrival per warp
    const uint32_t q_ready0 = cluster_addr(&bars->q_ready[0], 0);
    const uint32_t p_full0 = cluster_addr(&bars->p_full[t], 0);
    const uint32_t o_empty0 = cluster_addr(&bars->o_empty[t], 0);
    auto warp_arrive = [&](uint32_t bar_cluster) {
      __syncwarp();
      if (lane == 0) arrive_cluster_cta(bar_cluster);
    };
    uint32_t sph = 0;
    uint32_t it = 0;
    uint32_t cur_qs = static_cast<uint32_t>(t), cur_qp = 0;  // this tile's Q slot and parity in the current item
    // wait for the tile's load, rotate this thread's row, hand the tile to the issuer
    auto prepare_q = [&](uint32_t qs, uint32_t qp, int item_idx) -> bool {
      if (!warp_wait_cl(&bars->q_full[qs], qp, wc)) return false;
      if (f.n_pairs) {
        const Item nx = decode_item(item_idx, a, n_quads, n_kt);
        const int qt = nx.qt0 + 2 * t + static_cast<int>(r);
        rotate_row(q_smem(qs) + row * 128, row, a.q_offset + qt * BM + row, a.rope_offset, f.n_pairs, f.half != 0,
                   f_hi, f_lo);
        fence_proxy_async_smem();
      }
      warp_arrive(q_ready0 + qs * 8);
      return true;
    };
    int idx = item_at(0);
    if (idx < n_items && !prepare_q(cur_qs, cur_qp, idx)) idx = n_items;
    while (idx < n_items) {
      const Item itm = decode_item(idx, a, n_quads, n_kt);
      const int qt = itm.qt0 + 2 * t + static_cast<int>(r);
      const TileRange rng = t ? itm.r1 : itm.r0;
      const int n_t = rng.count();
      const int m = qt * BM + row;     // query row
      const int pos = a.q_offset + m;  // its absolute position
      const int tile_pos0 = a.q_offset + qt * BM;

      float m_run = -INFINITY, l_run = 0.f;
      bool ok = true;
      for (int i = 0; i < n_t; ++i) {
        const int j = i;  // key tile
        if (!warp_wait_cl(&bars->s_full[t], sph, wc)) { ok = false; break; }
        sph ^= 1;
        tc_fence_after();
        // the last Q K of this pair tile has completed: the producer may load the next item's Q
        if (i == n_t - 1) mbar_arrive(&bars->q_empty[cur_qs]);
        uint32_t sr[BN];
#pragma unroll
        for (int c = 0; c < BN / 32; ++c) tmem_ld32(s_addr + c * 32, sr + c * 32);
        tmem_wait_ld();
        float s[BN];
#pragma unroll
        for (int c = 0; c < BN; ++c) s[c] = __uint_as_float(sr[c]);
        const int key0 = j * BN;
        if (a.causal && key0 + BN - 1 > tile_pos0) {
          // some key of this tile lies after some query of this CTA's rows: mask key > position
#pragma unroll
          for (int c = 0; c < BN; ++c)
            if (key0 + c > pos) s[c] = -INFINITY;
        } else if (!a.causal && key0 + BN > a.S_k) {
#pragma unroll
          for (int c = 0; c < BN; ++c)
            if (key0 + c >= a.S_k) s[c] = -INFINITY;
        }
        float m8[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) m8[e] = s[e];
#pragma unroll
        for (int c = 8; c + 16 <= BN; c += 16)
#pragma unroll
          for (int e = 0; e < 8; ++e) m8[e] = fmax3(m8[e], s[c + e], s[c + 8 + e]);
#pragma unroll
        for (int e = 0; e < 8; ++e) m8[e] = fmaxf(m8[e], s[BN - 8 + e]);
        const float mx = fmaxf(fmax3(m8[0], m8[1], m8[2]), fmax3(fmax3(m8[3], m8[4], m8[5]), m8[6], m8[7])) *
                         a.scale_log2;
        const bool need = mx > m_run + kRescaleThreshold;
        float alpha = 1.f;
        if (need) {
          if (i > 0) alpha = fast_exp2(m_run - mx);
          l_run *= alpha;
          m_run = mx;
        }
        uint32_t pr[BN / 2];
        const float2 sl2 = make_float2(a.scale_log2, a.scale_log2);
        const float m_ref = (m_run == -INFINITY) ? 0.f : m_run;  // a row with no visible key yet
        const float2 nm2 = make_float2(-m_ref, -m_ref);
        float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
        for (int c = 0; c < BN / 4; ++c) {
          const float2 x = __ffma2_rn(make_float2(s[2 * c], s[2 * c + 1]), sl2, nm2);
          const float2 pp = make_float2(fast_exp2(x.x), fast_exp2(x.y));
          acc[c & 3] = __fadd2_rn(acc[c & 3], pp);
          pr[c] = pack_bf16x2(pp.x, pp.y);
        }
        tmem_st32(s_addr, pr);
        if (__any_sync(0xffffffffu, need && i > 0)) {  // O rescale before this tile's first P V
#pragma unroll 1
          for (int c = 0; c < DV / 32; ++c) {
            uint32_t orow[32];
            tmem_ld32(o_addr + c * 32, orow);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) orow[e] = __float_as_uint(__uint_as_float(orow[e]) * alpha);
            tmem_st32(o_addr + c * 32, orow);
          }
        }
#pragma unroll
        for (int c = BN / 4; c < BN / 2; ++c) {
          const float2 x = __ffma2_rn(make_float2(s[2 * c], s[2 * c + 1]), sl2, nm2);
          const float2 pp = make_float2(fast_exp2(x.x), fast_exp2(x.y));
          acc[c & 3] = __fadd2_rn(acc[c & 3], pp);
          pr[c] = pack_bf16x2(pp.x, pp.y);
        }
        acc[0] = __fadd2_rn(__fadd2_rn(acc[0], acc[1]), __fadd2_rn(acc[2], acc[3]));
        l_run += acc[0].x + acc[0].y;
        tmem_st32(s_addr + 32, pr + 32);
        tmem_wait_st();
        tc_fence_before();
        warp_arrive(p_full0);
      }
      if (!ok) break;
      const int next_idx = item_at(it + 1);
      uint32_t nxt_qs = cur_qs, nxt_qp = cur_qp;
      q_advance(nxt_qs, nxt_qp, 2);
      if (next_idx < n_items && !prepare_q(nxt_qs, nxt_qp, next_idx)) break;

      // epilogue: O / l -> out (rows past S are computed but not stored)
      if (!warp_wait_cl(&bars->o_done[t], it & 1, wc)) break;
      tc_fence_after();
      const float inv_l = 1.f / l_run;
      const bool store = m < a.S;
      // Each lane of a group of four stores 16-byte pieces of the group's four rows, so that one
      // store instruction writes 64 contiguous bytes of each of eight rows (a row's own lane would
      // write 16 bytes of each of 32 rows 8 KB apart)
      const int lj = lane & 3;
      const int m_base = m - lj;  // first row of this lane's group
      __nv_bfloat16* const og = static_cast<__nv_bfloat16*>(a.out) +
                                ((static_cast<long long>(itm.b) * a.S + m_base) * a.n_h + itm.h) * DV + lj * 8;
      const long long row_step = static_cast<long long>(a.n_h) * DV;
#pragma unroll 1
      for (int c = 0; c < DV / 32; ++c) {
        uint32_t orow[32];
        tmem_ld32(o_addr + c * 32, orow);
        tmem_wait_ld();
        uint4 pc[4];
#pragma unroll
        for (int e = 0; e < 4; ++e)
          pc[e] = make_uint4(pack_bf16x2(__uint_as_float(orow[8 * e]) * inv_l, __uint_as_float(orow[8 * e + 1]) * inv_l),
                             pack_bf16x2(__uint_as_float(orow[8 * e + 2]) * inv_l, __uint_as_float(orow[8 * e + 3]) * inv_l),
                             pack_bf16x2(__uint_as_float(orow[8 * e + 4]) * inv_l, __uint_as_float(orow[8 * e + 5]) * inv_l),
                             pack_bf16x2(__uint_as_float(orow[8 * e + 6]) * inv_l, __uint_as_float(orow[8 * e + 7]) * inv_l));
        // 4 x 4 transpose of the pieces within the group (two exchange rounds): afterwards pc[k] is
        // piece lj of row m_base + k
        {
          const bool b1 = (lj & 2) != 0;
          uint4 s0 = b1 ? pc[0] : pc[2], s1 = b1 ? pc[1] : pc[3];
          uint4 r0 = shfl_xor_u4(s0, 2), r1 = shfl_xor_u4(s1, 2);
          if (b1) { pc[0] = r0; pc[1] = r1; } else { pc[2] = r0; pc[3] = r1; }
          const bool b0 = (lj & 1) != 0;
          s0 = b0 ? pc[0] : pc[1];
          s1 = b0 ? pc[2] : pc[3];
          r0 = shfl_xor_u4(s0, 1);
          r1 = shfl_xor_u4(s1, 1);
          if (b0) { pc[0] = r0; pc[2] = r1; } else { pc[1] = r0; pc[3] = r1; }
        }
#pragma unroll
        for (int k = 0; k < 4; ++k)
          if (m_base + k < a.S) *reinterpret_cast<uint4*>(og + k * row_step + c * 32) = pc[k];
      }
      tc_fence_before();
      warp_arrive(o_empty0);
      if (store && a.lse != nullptr)
        a.lse[(static_cast<long long>(itm.b) * a.n_h + itm.h) * a.S + m] =
            (m_run + log2f(l_run)) * 0.69314718055994530942f;
      idx = next_idx;
      cur_qs = nxt_qs;
      cur_qp = nxt_qp;
      ++it;
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();  // no CTA leaves while the other may still use its shared memory or TMEM
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, 512;" ::"r"(tmem) : "memory");
  }
}

std::atomic<unsigned> g_pair_ready{0};  // one bit per device that has been prepared
std::atomic<int> g_pair_count[32];      // per device: clusters of two CTAs that fit at once (0: not known)

void pair_config(cudaLaunchConfig_t* cfg, cudaLaunchAttribute* attr, int pairs, cudaStream_t st) {
  attr->id = cudaLaunchAttributeClusterDimension;
  attr->val.clusterDim.x = 2;
  attr->val.clusterDim.y = 1;
  attr->val.clusterDim.z = 1;
  cfg->gridDim = dim3(2 * pairs);
  cfg->blockDim = dim3(kThreads);
  cfg->dynamicSmemBytes = kSmemBytes;
  cfg->stream = st;
  cfg->attrs = attr;
  cfg->numAttrs = 1;
}

// Opt in to the shared memory, check the register split against the compiled kernel, and find
// how many pairs are resident at once, once per process and device.
cudaError_t pair_prepare(int* pairs) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned bit = 1u << (dev & 31);
  if (!(g_pair_ready.load(std::memory_order_acquire) & bit)) {
    cudaFuncAttributes fa;
    if ((e = cudaFuncGetAttributes(&fa, prefill_pair_kernel)) != cudaSuccess) return e;
    if (static_cast<long long>(fa.numRegs) * kThreads < kRegsNeeded) return cudaErrorInvalidConfiguration;
    if ((e = cudaFuncSetAttribute(prefill_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes)) !=
        cudaSuccess)
      return e;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr;
    pair_config(&cfg, &attr, 1, nullptr);
    int n = 0;
    if ((e = cudaOccupancyMaxActiveClusters(&n, prefill_pair_kernel, &cfg)) != cudaSuccess) return e;
    if (n < 1) return cudaErrorInvalidConfiguration;
    if (dev < 32) g_pair_count[dev].store(n, std::memory_order_release);
    g_pair_ready.fetch_or(bit, std::memory_order_acq_rel);
  }
  *pairs = dev < 32 ? g_pair_count[dev].load(std::memory_order_acquire) : 1;
  return cudaSuccess;
}
}  // namespace

bool prefill_pair_supported(int D_qk, int D_v, bool bf16, int window) {
  return bf16 && D_qk == DQK && D_v == DV && window == 0;
}

cudaError_t launch_prefill_pair(const PrefillArgs& a, const RopeFreq& rope, const CUtensorMap* maps, cudaStream_t st,
                                int* launches) {
  if (a.D != DQK || a.D_v != DV) return cudaErrorInvalidValue;
  int pairs = 0;
  cudaError_t e = pair_prepare(&pairs);
  if (e != cudaSuccess) return e;
  const int n_qt = (a.S + BM - 1) / BM;
  const long long n_items = static_cast<long long>(a.B) * a.n_h * ((n_qt + 3) / 4);
  if (n_items < pairs) pairs = static_cast<int>(n_items);
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr;
  pair_config(&cfg, &attr, pairs, st);
  e = cudaLaunchKernelEx(&cfg, prefill_pair_kernel, a, rope, maps[0], maps[1], maps[2]);
  *launches += 1;
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace attn

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
//   warps 0, 2  TMA producers: K tiles (warp 0), and the Q tiles of each work
//               item followed by its V tiles (warp 2), through rings of
//               shared-memory stages (128-byte swizzle).
//   warp 1      allocates 512 TMEM columns; lane 0 issues every tcgen05.mma:
//               S_t = Q_t K_j^T (A, B from shared memory) and O_t += P_t V_j
//               (P read from TMEM, V from shared memory as an MN-major operand),
//               each tile's P V and next Q K as one burst.
//   warp 3      idle (gives its registers to the softmax warpgroups)
//   warps 4-7   softmax warpgroup of Q tile 0, warps 8-11 of Q tile 1: each thread
//               owns one query row (TMEM lane), so row max / row sum need no
//               shuffles.  P is written back over S in TMEM as bf16.  The output
//               is rescaled only when the row maximum grows by more than 2^8
//               (exact: l and O always share the same reference maximum).
//   A work item is two Q tiles that read the same K/V tiles: with GQA, one Q tile
//   of two query heads of a K/V group (the tiles then see the same keys), else two
//   adjacent Q tiles of one (batch, head); while one warpgroup computes its softmax,
//   the tensor core runs the other tile's MMAs.  Items are taken heaviest-first
//   (latest Q tiles see the most keys), dealt to the CTAs in waves that alternate
//   direction; a small MHA launch (fewer than four items per CTA) follows a table
//   the host packs instead.
// RoPE: the query tiles are rotated in shared memory right after their TMA load
// (once per item, with hardware sin/cos; for a GQA item both warpgroups rotate
// both tiles, each angle serving the two heads); keys arrive already rotated
// (written once by the rope pass).  The Q tiles cycle through three shared-memory
// slots, so the next item's first tile is in place before the current item ends.
// The epilogue exchanges each row's output among groups of four lanes, so that
// every store instruction writes 64-byte row segments.
// Head dims: (64, 64) and (128, 128); the MLA prefill shape (192, 128) runs on the
// CTA-pair kernel of prefill_pair.cu.
// TMEM columns: [0,128) S/P of tile 0, [128,256) S/P of tile 1,
//               [256, 256+D_v) O of tile 0, [256+D_v, 256+2D_v) O of tile 1.
#include <math.h>

#include <algorithm>
#include <atomic>
#include <memory>
#include <mutex>
#include <utility>
#include <vector>

#include "kernels.h"

namespace attn {
namespace {

constexpr int BM = 128;  // query rows per Q tile
constexpr int BN = 128;  // keys per KV tile
constexpr int kThreads = 384;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

// Register split.  The launch holds 168 registers per thread (384 threads, one
// CTA per SM); the control warpgroup needs fewer, so it drops to kRegsCtl and
// the two softmax warpgroups rise to kRegsSoftmax: a row of 128 fp32 scores
// plus the online-softmax state then fits without spilling.  setmaxnreg.inc
// waits until the pool has the registers, so the split must fit the pool; the
// launcher checks the compiled register count against it before launching.
constexpr int kLaunchRegs = 168;
constexpr int kRegsCtl = 152, kRegsSoftmax = 176;
constexpr int kRegsNeeded = 4 * 32 * kRegsCtl + 8 * 32 * kRegsSoftmax;
static_assert(kRegsNeeded <= kThreads * kLaunchRegs, "register split exceeds the launch's pool");

// Head dims DQK (q, k) and DV (v, out).  Every tile is stored as 64-element
// (128-byte) column blocks of 128 rows with the 128-byte swizzle.  Shared
// memory holds three Q tile slots, kKStages K tiles and kVStages V tiles.
template <int DQK, int DV>
struct Cfg {
  static_assert(BM == BN, "Q, K and V tiles share one row count");
  static constexpr int kQBlocks = DQK / 64;       // column blocks of a Q or K tile
  static constexpr int kVBlocks = DV / 64;        // column blocks of a V tile
  static constexpr int kQKTileBytes = BM * DQK * 2;
  static constexpr int kVTileBytes = BN * DV * 2;
  static constexpr int kBlockBytes = BM * 128;    // one column block of a tile
  static_assert((DQK == 64 && DV == 64) || (DQK == 128 && DV == 128), "head dims");
  static constexpr int kKStages = DQK == 64 ? 3 : 2;
  static constexpr int kVStages = DQK == 64 ? 3 : 2;
  // Q tile slots: the third lets the next item's first Q tile load while the
  // current item still runs
  static constexpr int kQSlots = 3;
  static constexpr int kQOff = 0;
  static constexpr int kKOff = kQOff + kQSlots * kQKTileBytes;
  static constexpr int kVOff = kKOff + kKStages * kQKTileBytes;
  static constexpr int kBarOff = kVOff + kVStages * kVTileBytes;
  static constexpr int kFreqOff = kBarOff + 512;  // the RoPE frequencies, hi then lo words
  static constexpr int kSmemBytes = kFreqOff + 2 * kMaxRopePairs * 4 + 1024;  // + alignment slack
  static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");
  static constexpr uint32_t kOCol0 = 256;         // S of the two tiles in columns [0, 256)
  static_assert(kOCol0 + 2 * DV <= 512, "TMEM columns");
  static constexpr uint32_t kIdescQK = idesc_bf16_f32(BM, BN, false);
  static constexpr uint32_t kIdescPV = idesc_bf16_f32(BM, DV, true);
};

struct Bars {
  uint64_t q_full[3], q_ready[3], q_empty[3];  // per Q slot
  uint64_t s_full[2], p_full[2], o_done[2], o_empty[2];
  uint64_t k_full[3], k_empty[3], v_full[3], v_empty[3];  // up to 3 stages
  uint64_t fin;
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(Bars) <= 512, "barrier block");

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
  int dq, dh;        // Q tile t is tile qt0 + t dq of head h + t dh (adjacent tiles of one head, or one tile
                     // of two heads that share a K/V head)
  TileRange r0, r1;  // the two Q tiles
  int ns_u, n_load;  // loaded tiles: [0, ns_u) then [r0.jl, r1.jh]
  __device__ __forceinline__ int load_at(int v) const { return v < ns_u ? v : r0.jl + v - ns_u; }
};

__host__ __device__ __forceinline__ TileRange tile_range(int qt, const PrefillArgs& a, int n_kt) {
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

// Dealing of work items (a template parameter of the kernel):
constexpr int kDealTiles = 0;      // two adjacent Q tiles of one (batch, head), heaviest-first waves
constexpr int kDealTilesFold = 1;  // the same items, folded (below)
constexpr int kDealHeads = 2;      // one Q tile of two heads of a K/V group, heaviest-first waves
constexpr int kDealTable = 3;      // the items of kDealTiles, dealt by a table the host computes

// The table of a small launch: CTA c takes items item[start[c]], ..., item[start[c + 1] - 1] (item
// indices as kDealTiles numbers them).  It travels with the kernel's parameters.
constexpr int kTableCtas = 256;
constexpr int kTableItems = 1024;
struct DealTable {
  uint16_t start[kTableCtas + 1];
  uint16_t item[kTableItems];
};

// Index of this CTA's k-th work item.  Items are sorted heaviest-first and dealt out in waves
// of gridDim.x, every other wave in reverse CTA order, so that no CTA takes the heaviest item of
// every wave (with one direction only, the busiest CTA of the Llama-3-8B prefill would carry
// 3.5% more key tiles than the mean; alternating brings that to 0.1%).
// Folded dealing instead hands each CTA double items: the tile pairs p and n_pairs - 1 - p of
// one (batch, head), heavy one first, which together always hold the same number of key
// tiles; double items go out head after head, so the CTAs running at one time share few K/V
// heads and their key tiles are re-read from L2 rather than HBM.
// With GQA, an item can instead take one Q tile of two query heads that read the same K/V head:
// both tiles then have the same key tiles, so neither waits at the item's end for the other's
// one extra key tile, and both warpgroups reach the boundary together.
// The dealing is a template parameter: a run-time switch here cost the Llama-3-8B
// prefill 2.7% (register spills in the item loops).
template <int DEAL>
__device__ __forceinline__ int item_at(const DealTable& tbl, int n_items, uint32_t k) {
  const int g = static_cast<int>(gridDim.x), c = static_cast<int>(blockIdx.x);
  if constexpr (DEAL == kDealTable) {
    const int j = tbl.start[c] + static_cast<int>(k);
    return j < tbl.start[c + 1] ? tbl.item[j] : n_items;
  }
  if constexpr (DEAL == kDealTilesFold) return 2 * (static_cast<int>(k >> 1) * g + c) + static_cast<int>(k & 1u);
  return static_cast<int>(k) * g + ((k & 1u) ? g - 1 - c : c);
}

// Items per CTA-independent unit count: tile pairs per (batch, head), or Q tiles per head.
template <int DEAL>
__host__ __device__ __forceinline__ long long n_work_items(int B, int n_h, int n_qt) {
  if constexpr (DEAL == kDealHeads) return static_cast<long long>(B) * (n_h / 2) * n_qt;
  return static_cast<long long>(B) * n_h * ((n_qt + 1) / 2);
}

template <int DEAL>
__device__ __forceinline__ Item decode_item(int idx, const PrefillArgs& a, int n_pairs_q, int n_kt) {
  Item it;
  if constexpr (DEAL == kDealHeads) {
    const int n_qt = (a.S + BM - 1) / BM;
    const int bhp_count = a.B * (a.n_h / 2);
    const int q = n_qt - 1 - idx / bhp_count;  // heaviest (latest) Q tiles first
    const int bhp = idx % bhp_count;
    it.b = bhp / (a.n_h / 2);
    it.h = 2 * (bhp % (a.n_h / 2));
    it.g = it.h / (a.n_h / a.n_kv);
    it.qt0 = q;
    it.dq = 0;
    it.dh = 1;
    it.r0 = tile_range(q, a, n_kt);
    it.r1 = it.r0;
    it.ns_u = it.r0.ns;
    it.n_load = it.ns_u + it.r1.jh - it.r0.jl + 1;
    return it;
  }
  int p, bh;
  if constexpr (DEAL == kDealTilesFold) {  // n_pairs_q is even
    const unsigned half = static_cast<unsigned>(n_pairs_q) >> 1, d = static_cast<unsigned>(idx) >> 1;
    bh = static_cast<int>(d / half);
    const int j = static_cast<int>(d - static_cast<unsigned>(bh) * half);
    p = (idx & 1) ? j : n_pairs_q - 1 - j;
  } else {
    const int bh_count = a.B * a.n_h;
    p = n_pairs_q - 1 - idx / bh_count;  // heaviest (latest) tile pairs first
    bh = idx % bh_count;
  }
  it.b = bh / a.n_h;
  it.h = bh % a.n_h;
  it.g = it.h / (a.n_h / a.n_kv);
  it.qt0 = 2 * p;
  it.dq = 1;
  it.dh = 0;
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

// Rotate the span [rope_offset, rope_offset + 2 * n_pairs) of query row r
// (position pos) of a Q tile in place.  The tile is stored as column blocks of
// 128 rows x 128 bytes with the 128-byte swizzle: the 16-byte chunk c of row r
// sits at chunk (c & 7) ^ (r & 7) of block c >> 3.  rope_offset is a multiple
// of 8 (whole chunks).  Kept out of line: it runs once per tile row, and inlined
// it costs the softmax loop registers.  The frequencies come from shared memory:
// read through a reference to the kernel parameter, out of line, the rotation of
// one tile took ~8000 cycles (a clock trace), about four times its arithmetic.
// Its sin/cos come from rope_sincos_fast:
// with the accurate pair the rotation of each new item's Q tile measured 7% of
// the Llama-3-8B prefill (it runs between two items, while the tensor pipe waits).
template <int DQK>
__device__ __noinline__ void rotate_q_row(uint8_t* row, int r, int pos, int rope_offset, int n_pairs, bool half,
                                        const float* f_hi, const float* f_lo) {
  constexpr int kBlockBytes = BM * 128;
  auto chunk = [&](int c) -> uint8_t* { return row + (c >> 3) * kBlockBytes + (((c & 7) ^ (r & 7)) << 4); };
  const int c0 = rope_offset / 8;
  if (half) {
    // pair j = span dims (j, j + n_pairs): chunk c0 + i holds the first members of
    // pairs 8i..8i+7, chunk c0 + i + n_pairs / 8 their second members
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

// The same rotation for row r of two Q tiles at the same positions (a GQA work item's two
// heads), over loop iterations [i_lo, i_hi): each sin/cos serves both rows.  The two softmax
// warpgroups split the iterations between them, so each computes half the angles.
template <int DQK>
__device__ __noinline__ void rotate_q_rows2(uint8_t* row_a, uint8_t* row_b, int r, int pos, int rope_offset,
                                          int n_pairs, bool half, const float* f_hi, const float* f_lo, int i_lo,
                                          int i_hi) {
  constexpr int kBlockBytes = BM * 128;
  const int sw = r & 7;
  auto off = [&](int c) -> int { return (c >> 3) * kBlockBytes + (((c & 7) ^ sw) << 4); };
  const int c0 = rope_offset / 8;
  if (half) {
    const int hc = n_pairs / 8;
#pragma unroll 1
    for (int i = i_lo; i < i_hi; ++i) {
      const int o0 = off(c0 + i), o1 = off(c0 + i + hc);
      float a0[8], a1[8], b0[8], b1[8];
      bf16x8_to_f32(*reinterpret_cast<const uint4*>(row_a + o0), a0);
      bf16x8_to_f32(*reinterpret_cast<const uint4*>(row_a + o1), a1);
      bf16x8_to_f32(*reinterpret_cast<const uint4*>(row_b + o0), b0);
      bf16x8_to_f32(*reinterpret_cast<const uint4*>(row_b + o1), b1);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        float sn, cs;
        rope_sincos_fast(pos, f_hi[i * 8 + e], f_lo[i * 8 + e], &sn, &cs);
        rotate_pair(a0[e], a1[e], sn, cs);
        rotate_pair(b0[e], b1[e], sn, cs);
      }
      *reinterpret_cast<uint4*>(row_a + o0) = f32_to_bf16x8(a0);
      *reinterpret_cast<uint4*>(row_a + o1) = f32_to_bf16x8(a1);
      *reinterpret_cast<uint4*>(row_b + o0) = f32_to_bf16x8(b0);
      *reinterpret_cast<uint4*>(row_b + o1) = f32_to_bf16x8(b1);
    }
  } else {
#pragma unroll 1
    for (int i = i_lo; i < i_hi; ++i) {
      const int o = off(c0 + i);
      float a[8], b[8];
      bf16x8_to_f32(*reinterpret_cast<const uint4*>(row_a + o), a);
      bf16x8_to_f32(*reinterpret_cast<const uint4*>(row_b + o), b);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float sn, cs;
        rope_sincos_fast(pos, f_hi[i * 4 + e], f_lo[i * 4 + e], &sn, &cs);
        rotate_pair(a[2 * e], a[2 * e + 1], sn, cs);
        rotate_pair(b[2 * e], b[2 * e + 1], sn, cs);
      }
      *reinterpret_cast<uint4*>(row_a + o) = f32_to_bf16x8(a);
      *reinterpret_cast<uint4*>(row_b + o) = f32_to_bf16x8(b);
    }
  }
}

template <int DQK, int DV, int DEAL>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_tc_kernel(const __grid_constant__ PrefillArgs a, const __grid_constant__ RopeFreq f,
                      const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ DealTable tbl) {
  using C = Cfg<DQK, DV>;
  extern __shared__ uint8_t smem_raw[];
  // aligned by pointer arithmetic on the shared array, so that the compiler keeps shared-memory addressing
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  Bars* bars = reinterpret_cast<Bars*>(smem + C::kBarOff);
  float* const f_hi = reinterpret_cast<float*>(smem + C::kFreqOff);
  float* const f_lo = f_hi + kMaxRopePairs;
  for (int i = threadIdx.x; i < f.n_pairs; i += kThreads) {  // made visible by the __syncthreads below
    f_hi[i] = f.hi[i];
    f_lo[i] = f.lo[i];
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const int n_qt = (a.S + BM - 1) / BM;
  const int n_kt = (a.S_k + BN - 1) / BN;
  const int n_pairs_q = (n_qt + 1) / 2;
  const int n_items = static_cast<int>(n_work_items<DEAL>(a.B, a.n_h, n_qt));

  if (threadIdx.x == 0) {
    for (int q = 0; q < C::kQSlots; ++q) {
      mbar_init(&bars->q_full[q], 1);
      // the softmax warpgroup of the tile in the slot; with the GQA dealing both warpgroups,
      // which rotate the item's two tiles together
      mbar_init(&bars->q_ready[q], DEAL == kDealHeads ? 256 : 128);
      mbar_init(&bars->q_empty[q], 128);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&bars->s_full[t], 1);
      mbar_init(&bars->p_full[t], 128);
      mbar_init(&bars->o_done[t], 1);
      mbar_init(&bars->o_empty[t], 128);
    }
    for (int s = 0; s < C::kKStages; ++s) {
      mbar_init(&bars->k_full[s], 1);
      mbar_init(&bars->k_empty[s], 1);
    }
    for (int s = 0; s < C::kVStages; ++s) {
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

  // Q tile t of this CTA's k-th item lives in slot (2k + t) mod kQSlots, at
  // smem + kQOff + slot * kQKTileBytes (arithmetic, not an array: runtime-indexed
  // local arrays would live in local memory); that is the slot's u-th use, u =
  // (2k + t) / kQSlots, whose barrier phases have parity u & 1.
  // Each role walks the positions 2k + t in order, keeping (slot, parity) and advancing
  // them by one or two positions (no division on the hot roles' registers).
  auto q_smem = [&](uint32_t slot) { return smem + C::kQOff + slot * C::kQKTileBytes; };
  auto q_advance = [](uint32_t& slot, uint32_t& par, uint32_t by) {  // by <= kQSlots
    slot += by;
    if (slot >= static_cast<uint32_t>(C::kQSlots)) {
      slot -= C::kQSlots;
      par ^= 1u;
    }
  };

  if (warp < 4) {
    // control warpgroup: TMA producers (warps 0, 2), the MMA issuer (warp 1)
    // and an idle warp; its registers go to the softmax warpgroups
    setmaxnreg_dec<kRegsCtl>();
    if (warp == 0 || warp == 2) {
      // ------------------------------------------------------------ TMA producers
      // Two independent rings, one lane each: warp 0 loads K tiles; warp 2 the
      // two Q tiles of each work item, then its V tiles.  The K ring runs ahead
      // into the next item while the Q loads wait for the current epilogues.
      if (lane == 0) {
        const bool is_v = warp == 2;
        const int n_stages = is_v ? C::kVStages : C::kKStages;
        const int tile_bytes = is_v ? C::kVTileBytes : C::kQKTileBytes;
        const int n_blocks = is_v ? C::kVBlocks : C::kQBlocks;
        uint8_t* const ring = smem + (is_v ? C::kVOff : C::kKOff);
        uint64_t* const full = is_v ? bars->v_full : bars->k_full;
        uint64_t* const empty = is_v ? bars->v_empty : bars->k_empty;
        const CUtensorMap* map = is_v ? &tm_v : &tm_k;
        uint32_t st = 0, ph = 0;
        uint32_t issued = 0, last_ph = 0;  // bit s: stage s had a load issued / its phase parity
        uint32_t q_armed = 0, q_last = 0, it = 0;  // bit q: slot q loaded / parity of its last load
        uint32_t qs = 0, qp = 0;                    // slot and parity of position 2 it + t
        for (int idx = item_at<DEAL>(tbl, n_items, it); idx < n_items; idx = item_at<DEAL>(tbl, n_items, ++it)) {
          const Item itm = decode_item<DEAL>(idx, a, n_pairs_q, n_kt);
          if (is_v) {
            for (int t = 0; t < 2; ++t, q_advance(qs, qp, 1)) {
              if (!mbar_wait(&bars->q_empty[qs], qp ^ 1, wc)) goto load_done;
              mbar_arrive_expect_tx(&bars->q_full[qs], C::kQKTileBytes);
              for (int db = 0; db < C::kQBlocks; ++db)
                tma_load_4d(q_smem(qs) + db * C::kBlockBytes, &tm_q, &bars->q_full[qs], db * 64, itm.h + t * itm.dh,
                            (itm.qt0 + t * itm.dq) * BM, itm.b);
              q_armed |= 1u << qs;
              q_last = (q_last & ~(1u << qs)) | (qp << qs);
            }
          }
          for (int v = 0; v < itm.n_load; ++v) {
            const int j = itm.load_at(v);
            if (!mbar_wait(&empty[st], ph ^ 1, wc)) goto load_done;
            mbar_arrive_expect_tx(&full[st], tile_bytes);
            uint8_t* dst = ring + st * tile_bytes;
            for (int db = 0; db < n_blocks; ++db)
              tma_load_4d(dst + db * C::kBlockBytes, map, &full[st], db * 64, itm.g, j * BN, itm.b);
            issued |= 1u << st;
            last_ph = (last_ph & ~(1u << st)) | (ph << st);
            if (++st == static_cast<uint32_t>(n_stages)) { st = 0; ph ^= 1; }
          }
        }
      load_done:
        if (bars->abort_flag) {  // let every copy in flight land before shared memory goes away
          for (int s2 = 0; s2 < n_stages; ++s2)
            if (issued & (1u << s2)) drain_wait(&full[s2], (last_ph >> s2) & 1, a.wait_limit_ns);
          for (int q = 0; q < C::kQSlots; ++q)
            if (q_armed & (1u << q)) drain_wait(&bars->q_full[q], (q_last >> q) & 1, a.wait_limit_ns);
        }
      }
      __syncwarp();
    } else if (warp == 1) {
      // ------------------------------------------------------------ MMA issuer
      // One lane issues both tiles' MMAs.  Per loaded key tile j: for each Q tile
      // t that needs it, every wait first (P_t(j) ready, K(j+1) landed), then
      // P_t V(j) and Q_t K(j+1) back to back, so the tensor pipe sees one burst.
      // An MMA instruction holds the lane ~53 cycles (measured), nearly the 64 cycles
      // it occupies the pipe, so every other instruction of the lane between bursts is
      // time the pipe may wait.  (One lane per Q tile measured 17% slower: the two tiles'
      // MMAs then interleave in the pipe and each tile's chain through its softmax grows.)
      if (lane == 0) {
        const uint64_t q_desc0 = sdesc_sw128(smem_u32(q_smem(0)), 16, 1024);
        const uint64_t k_desc0 = sdesc_sw128(smem_u32(smem + C::kKOff), 16, 1024);
        const uint64_t v_desc0 = sdesc_sw128(smem_u32(smem + C::kVOff), C::kBlockBytes, 1024);
        uint32_t kst = 0, kph = 0, vst = 0, vph = 0, pph0 = 0, pph1 = 0;
        uint32_t it = 0;
        uint32_t qs0 = 0, qp0 = 0;  // slot and parity of Q tile 0 of the current item
        // Q_t K over the dims [DQK/2 * half, DQK/2 * (half + 1)), or all dims (half < 0)
        auto issue_qk_part = [&](int t, uint32_t qslot, uint32_t stage, int half) {
          const uint64_t a0 = q_desc0 + ((qslot * C::kQKTileBytes) >> 4);
          const uint64_t b0 = k_desc0 + ((stage * C::kQKTileBytes) >> 4);
          const int k_lo = half > 0 ? DQK / 32 : 0, k_hi = half == 0 ? DQK / 32 : DQK / 16;
#pragma unroll
          for (int kk = k_lo; kk < k_hi; ++kk) {
            const uint32_t off = ((kk >> 2) * C::kBlockBytes + (kk & 3) * 32) >> 4;
            mma_ss(tmem + t * 128u, a0 + off, b0 + off, C::kIdescQK, kk > 0 ? 1u : 0u);
          }
        };
        auto issue_qk = [&](int t, uint32_t qslot, uint32_t stage) { issue_qk_part(t, qslot, stage, -1); };
        // P_t V over the tile's 128 keys (P of keys [16 kk, 16 kk + 16) sits in TMEM columns
        // [8 kk, 8 kk + 8) of the tile's S columns, two bf16 per column)
        auto issue_pv = [&](int t, uint32_t stage, bool accumulate) {
          const uint64_t b0 = v_desc0 + ((stage * C::kVTileBytes) >> 4);
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk)
            mma_ts(tmem + C::kOCol0 + t * DV, tmem + t * 128u + kk * 8, b0 + ((kk * 16 * 128) >> 4), C::kIdescPV,
                   (accumulate || kk > 0) ? 1u : 0u);
        };
        for (int idx = item_at<DEAL>(tbl, n_items, it); idx < n_items; idx = item_at<DEAL>(tbl, n_items, ++it)) {
          const Item itm = decode_item<DEAL>(idx, a, n_pairs_q, n_kt);
          bool q_seen0 = false, q_seen1 = false, pv_seen0 = false, pv_seen1 = false;
          uint32_t qs1 = qs0, qp1 = qp0;
          q_advance(qs1, qp1, 1);
          if (!mbar_wait(&bars->k_full[kst], kph, wc)) goto mma_done;
          {
            const int j0 = itm.load_at(0);
            for (int t = 0; t < 2; ++t) {
              if (!(t ? itm.r1 : itm.r0).has(j0)) continue;
              if (!mbar_wait(&bars->q_ready[t ? qs1 : qs0], t ? qp1 : qp0, wc)) goto mma_done;
              (t ? q_seen1 : q_seen0) = true;
              tc_fence_after();
              issue_qk(t, t ? qs1 : qs0, kst);
              mma_commit(&bars->s_full[t]);
            }
          }
          mma_commit(&bars->k_empty[kst]);
          if (++kst == C::kKStages) { kst = 0; kph ^= 1; }
          // Loaded tiles [vs, ve): both Q tiles take P V(j) and Q K(j + 1), neither at its first
          // P V or Q K.  They run through a loop without per-tile decisions: every instruction of
          // the issuing lane between two bursts is time the tensor pipe waits (a clock trace of
          // the general loop showed ~1600 of its ~4200 cycles per key tile spent there).
          // (the window part of the loaded tiles: tile r0.jl + v - ns_u at v >= ns_u; sink tiles, when
          // there are any, are in both Q tiles' ranges and come first)
          const int vs = itm.ns_u + itm.r1.jl - itm.r0.jl + 1;
          const int ve = itm.ns_u + itm.r0.jh - itm.r0.jl;
          for (int v = 0; v < itm.n_load; ++v) {
            if (v == vs && vs < ve) {
              // V(j) and K(j + 1) of the first iteration; each iteration then waits for the next
              // one's while the tensor pipe still holds its own last MMAs
              if (!mbar_wait(&bars->v_full[vst], vph, wc)) goto mma_done;
              if (!mbar_wait(&bars->k_full[kst], kph, wc)) goto mma_done;
              for (; v < ve; ++v) {
                // P of a tile is handed over whole: the softmax finishes it before the issuer
                // asks (a trace of this loop showed every P wait returning at once), so a split
                // hand-off would only add waits and fences between the MMA bursts
                if (!mbar_wait(&bars->p_full[0], pph0, wc)) goto mma_done;
                pph0 ^= 1;
                tc_fence_after();
                issue_pv(0, vst, true);
                issue_qk(0, qs0, kst);
                mma_commit(&bars->s_full[0]);
                if (!mbar_wait(&bars->p_full[1], pph1, wc)) goto mma_done;
                pph1 ^= 1;
                tc_fence_after();
                issue_pv(1, vst, true);
                mma_commit(&bars->v_empty[vst]);
                if (++vst == C::kVStages) { vst = 0; vph ^= 1; }
                issue_qk_part(1, qs1, kst, 0);
                uint32_t kst_n = kst + 1, kph_n = kph;
                if (kst_n == static_cast<uint32_t>(C::kKStages)) { kst_n = 0; kph_n ^= 1; }
                if (v + 1 < ve) {
                  if (!mbar_wait(&bars->v_full[vst], vph, wc)) goto mma_done;
                  if (!mbar_wait(&bars->k_full[kst_n], kph_n, wc)) goto mma_done;
                }
                issue_qk_part(1, qs1, kst, 1);
                mma_commit(&bars->s_full[1]);
                mma_commit(&bars->k_empty[kst]);
                kst = kst_n;
                kph = kph_n;
              }
            }
            const int j = itm.load_at(v);
            const bool next = v + 1 < itm.n_load;
            const int jn = next ? itm.load_at(v + 1) : -1;
            if (!mbar_wait(&bars->v_full[vst], vph, wc)) goto mma_done;
            bool k_ready = false;
            for (int t = 0; t < 2; ++t) {
              const TileRange& r = t ? itm.r1 : itm.r0;
              const bool pv = r.has(j), qk = next && r.has(jn);
              if (pv) {
                if (!mbar_wait(&bars->p_full[t], t ? pph1 : pph0, wc)) goto mma_done;
                if (t) pph1 ^= 1; else pph0 ^= 1;
                if (!(t ? pv_seen1 : pv_seen0) && !mbar_wait(&bars->o_empty[t], (it & 1) ^ 1, wc)) goto mma_done;
              }
              if (qk) {
                if (!k_ready) {
                  if (!mbar_wait(&bars->k_full[kst], kph, wc)) goto mma_done;
                  k_ready = true;
                }
                if (!(t ? q_seen1 : q_seen0) && !mbar_wait(&bars->q_ready[t ? qs1 : qs0], t ? qp1 : qp0, wc))
                  goto mma_done;
                if (t) q_seen1 = true; else q_seen0 = true;
              }
              tc_fence_after();
              if (pv) {
                issue_pv(t, vst, t ? pv_seen1 : pv_seen0);
                if (t) pv_seen1 = true; else pv_seen0 = true;
                if (j == r.jh) mma_commit(&bars->o_done[t]);
              }
              if (t == 1) {
                mma_commit(&bars->v_empty[vst]);
                if (++vst == C::kVStages) { vst = 0; vph ^= 1; }
              }
              if (qk) {
                issue_qk(t, t ? qs1 : qs0, kst);
                mma_commit(&bars->s_full[t]);
              }
            }
            if (next) {
              mma_commit(&bars->k_empty[kst]);
              if (++kst == C::kKStages) { kst = 0; kph ^= 1; }
            }
          }
          q_advance(qs0, qp0, 2);
        }
      mma_done:
        // every MMA issued so far completes before TMEM is released
        mma_commit(&bars->fin);
        drain_wait(&bars->fin, 0, a.wait_limit_ns);
      }
      __syncwarp();
    }
  } else {
    setmaxnreg_inc<kRegsSoftmax>();
    // ------------------------------------------------------------ softmax warpgroups
    const int t = (warp - 4) >> 2;     // Q tile of this warpgroup
    const int quad = warp & 3;         // TMEM lane quadrant
    const int r = quad * 32 + lane;    // query row within the tile
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t s_addr = tmem + lane_off + (t ? 128u : 0u);
    const uint32_t o_addr = tmem + lane_off + C::kOCol0 + (t ? DV : 0);
    uint32_t sph = 0;
    uint32_t it = 0;
    // Q tile t of the k-th item: wait for its load, rotate this thread's row, hand it
    // to the MMA issuer.  The tile is released as soon as its last Q K has completed,
    // and the next item's tile is prepared before this item's epilogue, so that the new
    // item's first Q K overlaps that epilogue (Llama-3-8B prefill 1.92 -> 1.91 ms).
    uint32_t cur_qs = static_cast<uint32_t>(t), cur_qp = 0;  // this tile's Q slot and parity in the current item
    auto prepare_q = [&](uint32_t qs, uint32_t qp, int item_idx) -> bool {
      if constexpr (DEAL == kDealHeads) {
        // the item's two tiles sit in slot qs - t and qs - t + 1 (mod 3) and share their rows'
        // positions: warpgroup t rotates iterations [t n / 2, (t + 1) n / 2) of row r of both
        const uint32_t qa = t ? (qs == 0 ? 2u : qs - 1) : qs, qb = t ? qs : (qs == 2 ? 0u : qs + 1);
        const uint32_t pa = t ? (qs == 0 ? qp ^ 1u : qp) : qp, pb = t ? qp : (qs == 2 ? qp ^ 1u : qp);
        if (!warp_wait(&bars->q_full[qa], pa, wc)) return false;
        if (!warp_wait(&bars->q_full[qb], pb, wc)) return false;
        if (f.n_pairs) {
          const Item nx = decode_item<DEAL>(item_idx, a, n_pairs_q, n_kt);
          const int n_it = f.half ? f.n_pairs / 8 : f.n_pairs / 4;
          rotate_q_rows2<DQK>(q_smem(qa) + r * 128, q_smem(qb) + r * 128, r, a.q_offset + nx.qt0 * BM + r,
                              a.rope_offset, f.n_pairs, f.half != 0, f_hi, f_lo, t * (n_it / 2),
                              t ? n_it : n_it / 2);
          fence_proxy_async_smem();
        }
        mbar_arrive(&bars->q_ready[qa]);
        mbar_arrive(&bars->q_ready[qb]);
      } else {
        if (!warp_wait(&bars->q_full[qs], qp, wc)) return false;
        if (f.n_pairs) {
          const Item nx = decode_item<DEAL>(item_idx, a, n_pairs_q, n_kt);
          rotate_q_row<DQK>(q_smem(qs) + r * 128, r, a.q_offset + (nx.qt0 + t * nx.dq) * BM + r, a.rope_offset,
                            f.n_pairs, f.half != 0, f_hi, f_lo);
          fence_proxy_async_smem();
        }
        mbar_arrive(&bars->q_ready[qs]);
      }
      return true;
    };
    int idx = item_at<DEAL>(tbl, n_items, 0);
    if (idx < n_items && !prepare_q(cur_qs, cur_qp, idx)) idx = n_items;
    while (idx < n_items) {
      const Item itm = decode_item<DEAL>(idx, a, n_pairs_q, n_kt);
      const int qt = itm.qt0 + t * itm.dq;
      const int hd = itm.h + t * itm.dh;  // this tile's query head
      const TileRange rng = t ? itm.r1 : itm.r0;
      const int n_t = rng.count();
      const int m = qt * BM + r;  // query row
      const int pos = a.q_offset + m;  // its absolute position

      float m_run = -INFINITY, l_run = 0.f;
      bool ok = true;
      for (int i = 0; i < n_t; ++i) {
        const int j = rng.at(i);  // key tile
        if (!warp_wait(&bars->s_full[t], sph, wc)) { ok = false; break; }
        sph ^= 1;
        tc_fence_after();
        // the last Q K of this tile has completed: the producer may load the next item's Q
        if (i == n_t - 1) mbar_arrive(&bars->q_empty[cur_qs]);
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
        // row maximum: 8 independent chains of three-input max (two new columns
        // per instruction), then a tree; a single chain of 127 dependent max
        // operations would dominate the warp's latency
        float m8[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) m8[e] = s[e];
        static_assert((BN - 8) % 16 == 8, "chains take 16 columns per round plus one round of 8");
#pragma unroll
        for (int c = 8; c + 16 <= BN; c += 16)
#pragma unroll
          for (int e = 0; e < 8; ++e) m8[e] = fmax3(m8[e], s[c + e], s[c + 8 + e]);
#pragma unroll
        for (int e = 0; e < 8; ++e) m8[e] = fmaxf(m8[e], s[BN - 8 + e]);
        const float mx = fmaxf(fmax3(m8[0], m8[1], m8[2]), fmax3(fmax3(m8[3], m8[4], m8[5]), m8[6], m8[7])) *
                         a.scale_log2;
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
        // sum runs in 4 independent packed accumulators.  P goes back to TMEM in two
        // stores of 64 keys (the first drains while the second half is computed) and is
        // announced once.
        uint32_t pr[BN / 2];
        const float2 sl2 = make_float2(a.scale_log2, a.scale_log2);
        // a row whose tiles so far held no visible key keeps m = -inf: its
        // weights are 0 (reference 0 avoids -inf - -inf)
        const float m_ref = (m_run == -INFINITY) ? 0.f : m_run;
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
        // O rescale before the first P V of this tile accumulates into O.  P V(j-1) has
        // completed (s_full of tile j was committed after it).  TMEM loads/stores are
        // warp-collective: the whole warp rescales when any of its rows needs it (alpha
        // is 1 for the others).
        if (__any_sync(0xffffffffu, need && i > 0)) {
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
        mbar_arrive(&bars->p_full[t]);
      }
      if (!ok) break;
      const int next_idx = item_at<DEAL>(tbl, n_items, it + 1);
      uint32_t nxt_qs = cur_qs, nxt_qp = cur_qp;
      q_advance(nxt_qs, nxt_qp, 2);
      if (next_idx < n_items && !prepare_q(nxt_qs, nxt_qp, next_idx)) break;

      // epilogue: O / l -> out (rows past S are computed but not stored)
      if (!warp_wait(&bars->o_done[t], it & 1, wc)) break;
      tc_fence_after();
      const float inv_l = 1.f / l_run;
      const bool store = m < a.S;
      // Each lane of a group of four stores 16-byte pieces of the group's four rows, so that one
      // store instruction writes 64 contiguous bytes of each of eight rows (a row's own lane would
      // write 16 bytes of each of 32 rows 8 KB apart)
      const int lj = lane & 3;
      const int m_base = m - lj;  // first row of this lane's group
      __nv_bfloat16* const og = static_cast<__nv_bfloat16*>(a.out) +
                                ((static_cast<long long>(itm.b) * a.S + m_base) * a.n_h + hd) * DV + lj * 8;
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
      mbar_arrive(&bars->o_empty[t]);
      if (store && a.lse != nullptr)
        a.lse[(static_cast<long long>(itm.b) * a.n_h + hd) * a.S + m] =
            (m_run + log2f(l_run)) * 0.69314718055994530942f;
      idx = next_idx;
      cur_qs = nxt_qs;
      cur_qp = nxt_qp;
      ++it;
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

namespace {
// Per instantiation, one bit per device that has been prepared.
std::atomic<unsigned> g_ready[6];

// Opt in to the kernel's shared memory and check, once per process and device,
// that the compiled kernel holds enough registers per thread for its register
// split (a split above the pool would leave setmaxnreg.inc waiting forever).
template <typename K>
cudaError_t prepare(K kernel, int smem_bytes, std::atomic<unsigned>* ready) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned bit = 1u << (dev & 31);
  if (ready->load(std::memory_order_acquire) & bit) return cudaSuccess;
  cudaFuncAttributes fa;
  if ((e = cudaFuncGetAttributes(&fa, kernel)) != cudaSuccess) return e;
  if (static_cast<long long>(fa.numRegs) * kThreads < kRegsNeeded) return cudaErrorInvalidConfiguration;
  if ((e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes)) != cudaSuccess)
    return e;
  ready->fetch_or(bit, std::memory_order_acq_rel);
  return cudaSuccess;
}

template <int DQK, int DV, int DEAL = kDealTiles>
cudaError_t launch(const PrefillArgs& a, const RopeFreq& rope, const CUtensorMap* maps, int grid, cudaStream_t st,
                   std::atomic<unsigned>* ready, const DealTable& tbl) {
  auto k = prefill_tc_kernel<DQK, DV, DEAL>;
  const cudaError_t e = prepare(k, Cfg<DQK, DV>::kSmemBytes, ready);
  if (e != cudaSuccess) return e;
  k<<<grid, kThreads, Cfg<DQK, DV>::kSmemBytes, st>>>(a, rope, maps[0], maps[1], maps[2], tbl);
  return cudaGetLastError();
}
}  // namespace

namespace {
// Dealing table of a small launch (fewer than four items per CTA, where the items' sizes are few
// and coarse and heaviest-first waves leave the busiest CTA well above the mean).  An item costs
// its loaded key tiles at 17 units each (a turn of both Q tiles, ~1.7 us) plus 40 for its
// boundary (~4 us).  First-fit decreasing packs the items into at most `grid` CTAs under a cap,
// and a binary search takes the smallest cap that fits; the table is used only when that cap is
// below the busiest CTA of the waves.  Tables are cached per launch shape.
struct TableKey {
  int B, n_h, S, S_k, q_offset, causal, window, n_sink, grid;
  bool operator==(const TableKey& o) const {
    return B == o.B && n_h == o.n_h && S == o.S && S_k == o.S_k && q_offset == o.q_offset && causal == o.causal &&
           window == o.window && n_sink == o.n_sink && grid == o.grid;
  }
};

bool build_table(const PrefillArgs& a, int n_items, int grid, DealTable* t) {
  if (grid > kTableCtas || n_items > kTableItems || n_items >= 4 * grid) return false;
  const int n_qt = (a.S + BM - 1) / BM, n_kt = (a.S_k + BN - 1) / BN;
  const int n_pairs_q = (n_qt + 1) / 2, bh_count = a.B * a.n_h;
  std::vector<int> w(n_items);
  long long total = 0;
  for (int idx = 0; idx < n_items; ++idx) {  // the kDealTiles numbering of decode_item
    const int p = n_pairs_q - 1 - idx / bh_count;
    const TileRange r0 = tile_range(2 * p, a, n_kt), r1 = tile_range(2 * p + 1, a, n_kt);
    w[idx] = 17 * (r0.ns + r1.jh - r0.jl + 1) + 40;
    total += w[idx];
  }
  // busiest CTA of the heaviest-first waves in alternating direction
  std::vector<long long> load(grid, 0);
  for (int idx = 0; idx < n_items; ++idx) {
    const int k = idx / grid, j = idx % grid;
    load[(k & 1) ? grid - 1 - j : j] += w[idx];
  }
  const long long waves_max = *std::max_element(load.begin(), load.end());
  std::vector<int> order(n_items);
  for (int i = 0; i < n_items; ++i) order[i] = i;
  std::stable_sort(order.begin(), order.end(), [&](int x, int y) { return w[x] > w[y]; });
  std::vector<int> bin(n_items);
  auto ffd = [&](long long cap) {
    int used = 0;
    std::fill(load.begin(), load.end(), 0);
    for (int i : order) {
      int b = 0;
      while (b < used && load[b] + w[i] > cap) ++b;
      if (b == used) {
        if (used == grid) return false;
        ++used;
      }
      load[b] += w[i];
      bin[i] = b;
    }
    return true;
  };
  long long lo = std::max<long long>(w[order[0]], (total + grid - 1) / grid), hi = waves_max - 1;
  if (lo > hi || !ffd(hi)) return false;
  while (lo < hi) {
    const long long mid = (lo + hi) / 2;
    if (ffd(mid)) hi = mid; else lo = mid + 1;
  }
  ffd(hi);
  int pos = 0;
  for (int c = 0; c < grid; ++c) {
    t->start[c] = static_cast<uint16_t>(pos);
    for (int i : order)  // heaviest first within a CTA
      if (bin[i] == c) t->item[pos++] = static_cast<uint16_t>(i);
  }
  t->start[grid] = static_cast<uint16_t>(pos);
  return true;
}

// Copies the table for this launch into *out; false: heaviest-first waves.  (A copy, taken under
// the lock: another thread may evict the cached entry before this launch is made.)
bool deal_table(const PrefillArgs& a, int n_items, int grid, DealTable* out) {
  static std::mutex mu;
  static std::vector<std::pair<TableKey, std::unique_ptr<DealTable>>> cache;  // nullptr: no table
  const TableKey key{a.B, a.n_h, a.S, a.S_k, a.q_offset, a.causal, a.window, a.n_sink, grid};
  std::lock_guard<std::mutex> lock(mu);
  const DealTable* t = nullptr;
  bool found = false;
  for (const auto& e : cache)
    if (e.first == key) {
      t = e.second.get();
      found = true;
      break;
    }
  if (!found) {
    std::unique_ptr<DealTable> nt(new DealTable());
    if (!build_table(a, n_items, grid, nt.get())) nt.reset();
    if (cache.size() >= 64) cache.erase(cache.begin());
    cache.emplace_back(key, std::move(nt));
    t = cache.back().second.get();
  }
  if (t == nullptr) return false;
  *out = *t;
  return true;
}
}  // namespace

bool prefill_tc_supported(int D_qk, int D_v, bool bf16) {
  return bf16 && ((D_qk == 64 && D_v == 64) || (D_qk == 128 && D_v == 128));
}

cudaError_t launch_prefill_tc(const PrefillArgs& a, const RopeFreq& rope, const CUtensorMap* maps, int num_sms,
                              cudaStream_t st, int* launches) {
  const int n_qt = (a.S + BM - 1) / BM;
  const bool heads = a.head_pairs && !a.fold && (a.n_h / a.n_kv) % 2 == 0;
  const long long n_items =
      heads ? n_work_items<kDealHeads>(a.B, a.n_h, n_qt) : n_work_items<kDealTiles>(a.B, a.n_h, n_qt);
  const int grid = static_cast<int>(n_items < num_sms ? n_items : num_sms);
  static const DealTable kNoTable{};
  DealTable table;
  const DealTable* tbl = (!heads && !a.fold && deal_table(a, static_cast<int>(n_items), grid, &table)) ? &table
                                                                                                     : nullptr;
  cudaError_t e;
  // folded dealing is built for the two larger head dims (D = 64 prompts whose K/V
  // pass twice the L2 take the plain dealing); the dealing table only for D = 64
  if (a.D == 64)
    e = heads ? launch<64, 64, kDealHeads>(a, rope, maps, grid, st, &g_ready[3], kNoTable)
        : tbl ? launch<64, 64, kDealTable>(a, rope, maps, grid, st, &g_ready[5], *tbl)
              : launch<64, 64>(a, rope, maps, grid, st, &g_ready[0], kNoTable);
  else if (a.D == 128)
    e = a.fold ? launch<128, 128, kDealTilesFold>(a, rope, maps, grid, st, &g_ready[2], kNoTable)
               : heads ? launch<128, 128, kDealHeads>(a, rope, maps, grid, st, &g_ready[4], kNoTable)
                       : launch<128, 128>(a, rope, maps, grid, st, &g_ready[1], kNoTable);
  else
    e = cudaErrorInvalidValue;
  *launches += 1;
  return e;
}

}  // namespace attn

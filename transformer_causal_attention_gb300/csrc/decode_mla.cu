// decode_mla.cu - MLA-absorbed decode on the tensor cores of a CTA pair (sm_103a).
//
// "Transformer 与 LLM" slide 06: after W_UK is folded into the query and W_UV
// into the output, the 128 query heads of a token share one 576-dim latent KV
// head [c^KV (512) ; k^R (64)], V is the first 512 latent dims, and the scores
// use 1/sqrt(192).  Per cached key the work is 128 x (576 + 512) multiply-adds
// against 1152 bytes read - about 242 FLOP per byte, at the ridge of the GPU,
// so both the tensor cores and HBM must run near their peaks.
//
// Mapping.  The two CTAs of a cluster act as one tensor-core unit
// (tcgen05.mma.cta_group::2, issued by the even CTA).  The pair walks its keys in
// rounds of 256; CTA r holds the round's keys [128 r, 128 r + 128) ("its keys").
//   scores   S^T [256 keys x 128 heads] = C [256 x 576] Q^T: M = keys (each CTA
//            supplies its own 128 cache rows as A), N = heads split over the pair
//            (CTA r holds the query rows of heads [64 r, 64 r + 64), 72 KB, as the
//            B half it supplies).  Each CTA receives S^T of its own keys in TMEM.
//   values   O^T [512 dims x 128 heads] += V^T [512 x 256 keys] P^T, as two
//            M = 256 tiles of dims; CTA r supplies (and accumulates) the dims
//            [256 t + 128 r, 256 t + 128 r + 128) of tile t, reading those dims of
//            all 256 keys of the round, and the B half P^T of heads [64 r, +64).
// The value rows of the other CTA's keys come through L2 (the other CTA read them
// from HBM for its scores moments before), so every cache byte leaves HBM once.
//
// TMEM (512 columns, allocated for the pair): two S^T buffers (the scores of the
// next round are computed while the softmax reads the current ones) and O^T
// (256 columns: two tiles of 128 dims x 128 heads).
//
// Softmax.  One thread per (key, half of the heads): it loads 64 scores of its
// key from TMEM.  All keys of a head share one exponent offset per round, agreed
// by the pair before any exponential: each CTA ORs a flag "some score passed the
// offset by 2^8" over its warps and sends it with, only when set, its per-head
// maxima; both CTAs then raise a head's offset to the pair's maximum when that
// passed the old offset by 2^8, rescaling O and the running sums (lazily, as in
// "Transformer架构完全深度解析" §13's online softmax, where the rescale is exact
// because O and l always share one reference maximum).  The probabilities go to
// shared memory as bf16 P^T: the half of the heads this CTA supplies stays local,
// the other half is stored into the other CTA (st.async, counted on its barrier).
// The running sums stay per thread until the end of a piece.
//
// Loads.  Each CTA streams its cache rows through a 3-stage ring of 32 KB units
// (128 keys x 128 dims, two 128-byte-swizzled TMA boxes) plus one 16 KB slot for
// the 64 rotary dims, in the order the MMAs take them: scores of round j + 1, then
// the values of round j.  The odd CTA's copies complete on the even CTA's
// barriers (cp.async.bulk.tensor .cta_group::2), so the issuer sees both halves
// of a unit with one wait.  Rows at or past a sequence's end may hold anything:
// value units that reach past it are cleared by a helper warp in each CTA before
// their MMA.
//
// Keys of all sequences, laid end to end with a gap of kPieceGap virtual keys
// between two sequences, are split evenly over the pairs at whole rounds (a pair's
// range may cross sequence ends; the gap charges a pair that starts a new sequence
// for the new query, its rotation and a pipeline refill); each (pair, sequence) piece writes
// one normalised partial, merged per sequence by mla_combine_kernel with the
// log-sum-exp rule of the online softmax ("Transformer架构完全深度解析" §13).
// Roles (384 threads): warp 0 TMA producer, warp 1 TMEM owner + MMA issuer (even
// CTA), warp 2 key prefix sums, then the value-row fixer, warp 3 query RoPE and
// hand-offs to the even CTA, warps 4-11 softmax (four lane quarters x two halves
// of the heads) and epilogue.
#include <math.h>

#include <atomic>

#include "kernels.h"
#include "pair.cuh"

namespace attn {
namespace {

constexpr int NH = 128;              // query heads
constexpr int HH = 64;               // heads whose query rows one CTA supplies
constexpr int DQK = 576;             // latent + rotary dims
constexpr int DV = 512;              // value dims
constexpr int RK = kMlaTileKeys;     // keys per CTA per round
constexpr int kRoundKeys = 2 * RK;
constexpr int kThreads = 384;
constexpr int kBoxBytes = RK * 128;          // 128 rows x 64 bf16 dims, 128-byte swizzled
constexpr int kUnitBytes = 2 * kBoxBytes;    // one ring stage: 128 keys x 128 dims
constexpr int kStages = 3;
constexpr int kQkUnits = 5;                  // dims [0,128) [128,256) [256,384) [384,512) | [512,576)
constexpr int kQBlockBytes = HH * 128;       // 64 heads x 64 dims
constexpr int kQBlocks = DQK / 64;           // 9
constexpr int kQBytes = kQBlocks * kQBlockBytes;   // 72 KB
constexpr int kPTBytes = kRoundKeys * 128;   // P^T: 256 keys x 64 heads, bf16
constexpr int kMaxB = 256;                   // the batch's key prefix sums live in shared memory
static_assert(RK == 128, "one TMEM lane per key of a CTA");

// shared memory (every MMA operand 1024-byte aligned)
constexpr int kQOff = 0;
constexpr int kRingOff = kQOff + kQBytes;
constexpr int kRopeOff = kRingOff + kStages * kUnitBytes;  // the slot of the 64 rotary dims
constexpr int kPTOff = kRopeOff + kBoxBytes;
constexpr int kMsgWords = NH + 4;                          // per-head maxima, then a flag word
constexpr int kMsgOff = kPTOff + kPTBytes;                 // [2 round parities] messages from the other CTA
constexpr int kRedOff = kMsgOff + 2 * kMsgWords * 4;       // [4 lane quarters][128 heads] partial maxima / sums
constexpr int kMOff = kRedOff + 4 * NH * 4;                // [8 softmax warps][64 heads] offsets, one copy per warp
constexpr int kFacOff = kMOff + 8 * HH * 4;                // [8 softmax warps][64 heads] rescale factors of a round
constexpr int kLOff = kFacOff + 8 * HH * 4;                // [2][128]: this CTA's row sums, the other CTA's
constexpr int kFlagOff = kLOff + 2 * NH * 4;               // [2 round parities][8 warps] exceed flags
constexpr int kPrefOff = kFlagOff + 64;
constexpr int kBarOff = kPrefOff + ((kMaxB + 1) * 4 + 63) / 64 * 64;
constexpr int kUsedBytes = kBarOff + 512;
constexpr int kSmemBytes = kUsedBytes + 1024;  // + slack to align the base to 1024 bytes
static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");
static_assert(kRingOff % 1024 == 0 && kRopeOff % 1024 == 0 && kPTOff % 1024 == 0, "operand alignment");
constexpr uint32_t kMsgBytes = (NH + 1) * 4;   // the maxima and the flag word
constexpr uint32_t kPTPeerBytes = RK * 128;   // the other CTA's 128 key rows of this CTA's P^T

// TMEM columns
constexpr uint32_t kSCol = 0;     // S^T buffers at 0 and 128
constexpr uint32_t kOCol = 256;   // O^T tiles at 256 and 384
constexpr uint32_t kIdescQK = idesc_bf16_f32(256, NH, false);
// O^T = V^T P^T: A (V^T, dims x keys) and B (P^T, keys x heads) are both contiguous along M / N
constexpr uint32_t kIdescPV = idesc_bf16_f32(256, NH, true) | (1u << 15);
constexpr float kRaise = 8.0f;    // a head's offset moves when the pair's maximum passes it by 2^8

// Register split: the launch holds 168 registers per thread (384 threads, one CTA per SM); the
// control warps drop to kRegsCtl, the softmax warps rise to kRegsSoftmax (64 scores, 64 running
// sums and the packed probabilities of a thread).  setmaxnreg.inc waits until the pool has the
// registers, so the split must fit it; the launcher checks the compiled count before launching.
constexpr int kLaunchRegs = 168;
constexpr int kRegsCtl = 104, kRegsSoftmax = 200;
constexpr int kRegsNeeded = 4 * 32 * kRegsCtl + 8 * 32 * kRegsSoftmax;
static_assert(kRegsNeeded <= kThreads * kLaunchRegs, "register split exceeds the launch's pool");
constexpr float kNoOffset = -1e30f;

struct Bars {
  uint64_t kv_full[kStages], kv_fixed[kStages], kv_tofix[kStages], kv_empty[kStages];
  uint64_t rope_full, rope_empty;
  uint64_t q_full, q_ready, q_empty;
  uint64_t s_full[2], s_free[2];
  uint64_t hsync[2];   // among the 8 softmax warps of a CTA: [0] the round's flags, [1] maxima / sums
  uint64_t msg_full[2];
  uint64_t pt_full, pt_ready;
  uint64_t pv_done, o_empty, l_full, fin;
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(Bars) <= 512, "barrier block");

// Three rounds of keys (a pair that starts a second sequence otherwise finishes last): at
// 32 x 32768, with the pair starts rounded to whole rounds, gaps of 256 / 512 / 768 / 1280 / 1792
// keys measured 0.3526 / 0.3498 / 0.3470 / 0.3499 / 0.3531 ms (before the rounding, 0 / 640 /
// 1280 / 2560 keys measured 0.363 / 0.358 / 0.354 / 0.363 ms).
constexpr long long kPieceGap = 768;

// Start of pair p in effective key positions (sequence b's key x sits at prefix[b] + gap b + x;
// Teff = T + gap (B - 1)), and as a real key: inside a sequence, the start is rounded down to a
// whole round of keys, so that only a sequence's last round is partial (a round split between two
// pairs would run its MMAs twice: at 32 x 32768 keys over 76 pairs, 4130 rounds instead of 4096,
// and 0.3517 against 0.3499 ms); in a gap, it is the next sequence's first key.
__device__ __forceinline__ long long pair_start_eff(int p, long long Teff, int P) {
  return static_cast<long long>(p) * Teff / P;
}
__device__ __forceinline__ long long round_down_keys(long long o) {
  return o & ~static_cast<long long>(kRoundKeys - 1);
}
__device__ __forceinline__ long long pair_start_key(int p, long long Teff, int P, const int* prefix, int nb) {
  const long long E = pair_start_eff(p, Teff, P);
  int lo = 0, hi = nb - 1;  // the last sequence starting at or before E
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (prefix[mid] + kPieceGap * mid <= E) lo = mid; else hi = mid - 1;
  }
  const long long o = E - (prefix[lo] + kPieceGap * lo);
  return o < prefix[lo + 1] - prefix[lo] ? prefix[lo] + round_down_keys(o) : prefix[lo + 1];
}

// The keys of pair p as pieces, one per sequence it touches.
struct PieceIter {
  const int* prefix;  // prefix[b] = keys of sequences < b
  int B;
  long long x, end;
  int b;
  __device__ void init(const int* pre, int nb, long long s, long long e) {
    prefix = pre;
    B = nb;
    x = s;
    end = e;
    int lo = 0, hi = nb - 1;  // largest b with prefix[b] <= x
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (prefix[mid] <= x) lo = mid; else hi = mid - 1;
    }
    b = lo;
  }
  __device__ bool next(int* sb, int* lo, int* hi) {
    if (x >= end || b >= B) return false;
    const long long seq_end = prefix[b + 1];
    const long long stop = end < seq_end ? end : seq_end;
    *sb = b;
    *lo = static_cast<int>(x - prefix[b]);
    *hi = static_cast<int>(stop - prefix[b]);
    x = stop;
    ++b;
    return true;
  }
};

// One unit of the load stream: keys [key0, key0 + 128), 64-dim boxes starting at dim d0 (d0 + 64 for the
// second box).  Score units carry this CTA's keys; value units carry the keys of one CTA of the pair and
// this CTA's dims of one O^T tile.
struct Unit {
  int key0, d0, nbox;
  bool rope_slot;  // the 64 rotary dims: its own slot
  bool pv;
};
__device__ __forceinline__ Unit qk_unit(int lo, int j, int r, int u) {
  return Unit{lo + j * kRoundKeys + r * RK, 128 * u, u == kQkUnits - 1 ? 1 : 2, u == kQkUnits - 1, false};
}
__device__ __forceinline__ Unit pv_unit(int lo, int j, int r, int kh, int t) {
  return Unit{lo + j * kRoundKeys + kh * RK, 256 * t + 128 * r, 2, false, true};
}
__device__ __forceinline__ bool needs_fix(const Unit& u, int L) { return u.pv && u.key0 + RK > L; }

// Every unit of a piece with nr rounds in the order the MMAs take them: scores(0), then for
// j = 1 .. nr - 1: scores(j), values(j - 1); then values(nr - 1).
template <typename F>
__device__ __forceinline__ bool for_units(int lo, int nr, int r, F&& f) {
  for (int j = 0; j <= nr; ++j) {
    if (j < nr)
      for (int u = 0; u < kQkUnits; ++u)
        if (!f(qk_unit(lo, j, r, u))) return false;
    if (j >= 1)
      for (int kh = 0; kh < 2; ++kh)
        for (int t = 0; t < 2; ++t)
          if (!f(pv_unit(lo, j - 1, r, kh, t))) return false;
  }
  return true;
}

// ---- pair helpers only this kernel uses
__device__ __forceinline__ void st_async_v4(uint32_t addr, uint32_t x, uint32_t y, uint32_t z, uint32_t w,
                                            uint32_t bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(
                   addr),
               "r"(x), "r"(y), "r"(z), "r"(w), "r"(bar)
               : "memory");
}
__device__ __forceinline__ void st_async_b32(uint32_t addr, uint32_t v, uint32_t bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];" ::"r"(addr), "r"(v),
               "r"(bar)
               : "memory");
}
// columns [col, col + 64) of this thread's TMEM lane (taddr) times the per-column factors f[0..63]
// (shared memory); warp-collective
__device__ __forceinline__ void scale_cols64(uint32_t taddr, const float* f) {
#pragma unroll 1
  for (int c = 0; c < 2; ++c) {
    uint32_t o[32];
    tmem_ld32(taddr + c * 32, o);
    tmem_wait_ld();
#pragma unroll
    for (int e = 0; e < 32; e += 4) {
      const float4 f4 = *reinterpret_cast<const float4*>(f + c * 32 + e);
      o[e] = __float_as_uint(__uint_as_float(o[e]) * f4.x);
      o[e + 1] = __float_as_uint(__uint_as_float(o[e + 1]) * f4.y);
      o[e + 2] = __float_as_uint(__uint_as_float(o[e + 2]) * f4.z);
      o[e + 3] = __float_as_uint(__uint_as_float(o[e + 3]) * f4.w);
    }
    tmem_st32(taddr + c * 32, o);
  }
}

__global__ void __launch_bounds__(kThreads, 1)
    mla_decode_kernel(const __grid_constant__ DecodeArgs a, const __grid_constant__ RopeFreq f,
                      const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_c) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // aligned by pointer arithmetic on the shared array, so that the compiler keeps shared-memory addressing
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  Bars* bars = reinterpret_cast<Bars*>(smem + kBarOff);
  int* prefix = reinterpret_cast<int*>(smem + kPrefOff);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int P = gridDim.x >> 1;   // pairs
  const int p = blockIdx.x >> 1;  // this CTA's pair
  const int r = blockIdx.x & 1;   // rank in the pair; 0 issues the MMAs
  const bool layout_ok = static_cast<int>(smem - smem_raw) + kUsedBytes <= kSmemBytes;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bars->kv_full[s], 1);
      mbar_init(&bars->kv_fixed[s], 2);  // the fixers of both CTAs
      mbar_init(&bars->kv_tofix[s], 1);
      mbar_init(&bars->kv_empty[s], 1);
    }
    mbar_init(&bars->rope_full, 1);
    mbar_init(&bars->rope_empty, 1);
    mbar_init(&bars->q_full, 1);
    mbar_init(&bars->q_ready, 2);   // both CTAs' queries loaded (and rotated)
    mbar_init(&bars->q_empty, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->s_full[i], 1);
      mbar_init(&bars->s_free[i], 16);  // the 8 softmax warps of both CTAs
      mbar_init(&bars->hsync[i], 8);
      mbar_init(&bars->msg_full[i], 1);
    }
    mbar_arrive_expect_tx(&bars->msg_full[0], kMsgBytes);  // rounds 0 and 1, before the other CTA can store
    mbar_arrive_expect_tx(&bars->msg_full[1], kMsgBytes);
    mbar_init(&bars->pt_full, 8);
    mbar_init(&bars->pt_ready, 1);
    mbar_init(&bars->pv_done, 1);
    mbar_init(&bars->o_empty, 16);
    mbar_init(&bars->l_full, 1);
    mbar_arrive_expect_tx(&bars->l_full, NH * 4);  // the first piece's row sums
    mbar_init(&bars->fin, 1);
    bars->abort_flag = layout_ok ? 0 : 1;
    if (!layout_ok) atomicOr(a.status, STATUS_LAYOUT);
    fence_mbar_init();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(
                     smem_u32(&bars->tmem_base))
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  if (warp == 2) {
    // prefix[b] = number of keys of sequences before b (lengths clamped to [1, max_len])
    int carry = 0;
    if (lane == 0) prefix[0] = 0;
    for (int base = 0; base < a.B; base += 32) {
      const int i = base + lane;
      int v = i < a.B ? min(max(a.seqlens[i], 1), a.max_len) : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += t;
      }
      if (i < a.B) prefix[i + 1] = carry + v;
      carry += __shfl_sync(0xffffffffu, v, 31);
    }
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers are initialised before either signals the other
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  const WaitCtl wc{&bars->abort_flag, a.status, a.wait_limit_ns};
  const long long Teff = prefix[a.B] + kPieceGap * (a.B - 1);
  const long long k_begin = pair_start_key(p, Teff, P, prefix, a.B), k_end = pair_start_key(p + 1, Teff, P, prefix, a.B);
  const bool run = !bars->abort_flag;  // false: the shared-memory layout did not fit, touch nothing
  const uint32_t peer = static_cast<uint32_t>(r ^ 1);

  if (warp < 4) {
  setmaxnreg_dec<kRegsCtl>();
  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0 && run) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_c);
      PieceIter it;
      it.init(prefix, a.B, k_begin, k_end);
      uint32_t st = 0, ph = 0, rph = 0, any_issued = 0;
      int sb, lo, hi;
      // L2 hints: a score unit's rows are read again moments later for the values (by both CTAs),
      // a value or rotary unit is their last read (0.368 -> 0.364 ms at 32 x 32768)
      uint64_t pol_keep, pol_drop;
      asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol_keep));
      asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol_drop));
      for (uint32_t n = 0; it.next(&sb, &lo, &hi); ++n) {
        const int L = prefix[sb + 1] - prefix[sb];
        const int nr = (hi - lo + kRoundKeys - 1) / kRoundKeys;
        if (!wait_cl(&bars->q_empty, (n & 1) ^ 1, wc)) break;
        mbar_arrive_expect_tx(&bars->q_full, kQBytes);
        for (int blk = 0; blk < kQBlocks; ++blk)
          tma_load_3d_pair(smem + kQOff + blk * kQBlockBytes, &tm_q, smem_u32(&bars->q_full), blk * 64, HH * r, sb);
        any_issued = 1;
        const bool done = for_units(lo, nr, r, [&](const Unit& u) -> bool {
          if (u.rope_slot) {
            if (!wait_cl(&bars->rope_empty, rph ^ 1, wc)) return false;
            if (r == 0) mbar_arrive_expect_tx(&bars->rope_full, 2 * kBoxBytes);
            tma_load_3d_pair_hint(smem + kRopeOff, &tm_c, cluster_addr(&bars->rope_full, 0), u.d0, u.key0, sb, pol_drop);
            rph ^= 1;
            return true;
          }
          if (!wait_cl(&bars->kv_empty[st], ph ^ 1, wc)) return false;
          uint8_t* dst = smem + kRingOff + st * kUnitBytes;
          if (needs_fix(u, L)) {  // counted locally, cleared by this CTA's fixer, then handed on
            mbar_arrive_expect_tx(&bars->kv_tofix[st], u.nbox * kBoxBytes);
            const uint32_t bar = cluster_addr(&bars->kv_tofix[st], static_cast<uint32_t>(r));
            for (int b = 0; b < u.nbox; ++b)
              tma_load_3d_pair_hint(dst + b * kBoxBytes, &tm_c, bar, u.d0 + 64 * b, u.key0, sb, u.pv ? pol_drop : pol_keep);
          } else {
            if (r == 0) mbar_arrive_expect_tx(&bars->kv_full[st], 2 * u.nbox * kBoxBytes);
            const uint32_t bar = cluster_addr(&bars->kv_full[st], 0);
            for (int b = 0; b < u.nbox; ++b)
              tma_load_3d_pair_hint(dst + b * kBoxBytes, &tm_c, bar, u.d0 + 64 * b, u.key0, sb, u.pv ? pol_drop : pol_keep);
          }
          if (++st == kStages) { st = 0; ph ^= 1; }
          return true;
        });
        if (!done) break;
      }
      if (bars->abort_flag && any_issued) {
        // copies in flight may still land: give them time before the CTA can leave (their barriers may sit
        // in the other CTA, so waiting on them is not always possible here)
        const uint64_t t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < 200000ull) {
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (even CTA)
    if (lane == 0 && run && r == 0) {
      PieceIter it;
      it.init(prefix, a.B, k_begin, k_end);
      const uint32_t q_addr = smem_u32(smem + kQOff);
      const uint32_t pt_addr = smem_u32(smem + kPTOff);
      uint32_t st = 0, fullph = 0, fixph = 0, rph = 0, g = 0, gp = 0;
      int sb, lo, hi, L = 0;
      auto take = [&](const Unit& u) -> bool {
        if (u.rope_slot) {
          if (!wait_cl(&bars->rope_full, rph, wc)) return false;
          rph ^= 1;
        } else if (needs_fix(u, L)) {
          if (!wait_cl(&bars->kv_fixed[st], (fixph >> st) & 1u, wc)) return false;
          fixph ^= 1u << st;
        } else {
          if (!wait_cl(&bars->kv_full[st], (fullph >> st) & 1u, wc)) return false;
          fullph ^= 1u << st;
        }
        tc_fence_after();
        return true;
      };
      auto release = [&](const Unit& u) {
        if (u.rope_slot) {
          commit_both(&bars->rope_empty);
        } else {
          commit_both(&bars->kv_empty[st]);
          if (++st == kStages) st = 0;
        }
      };
      for (uint32_t n = 0; it.next(&sb, &lo, &hi); ++n) {
        L = prefix[sb + 1] - prefix[sb];
        const int nr = (hi - lo + kRoundKeys - 1) / kRoundKeys;
        if (!wait_cl(&bars->q_ready, n & 1, wc)) goto mma_done;
        tc_fence_after();
        for (int j = 0; j <= nr; ++j) {
          if (j < nr) {
            // S^T (+)= C Q^T over the 576 dims: 36 MMAs of 16 dims
            const uint32_t buf = g & 1;
            if (!wait_cl(&bars->s_free[buf], ((g >> 1) & 1) ^ 1, wc)) goto mma_done;
            tc_fence_after();
            for (int u = 0; u < kQkUnits; ++u) {
              const Unit un = qk_unit(lo, j, 0, u);
              if (!take(un)) goto mma_done;
              // descriptors of the unit's first 16 dims; the rest differ only in the start address (+32 bytes
              // per 16 dims = +2 in the descriptor, + one box per 64 dims).  The pair MMA holds the issuing
              // thread until it is handed on, so nothing but the MMAs sits between them.
              const uint64_t a0 = sdesc_sw128(un.rope_slot ? smem_u32(smem + kRopeOff)
                                                           : smem_u32(smem + kRingOff + st * kUnitBytes), 16, 1024);
              const uint64_t b0 = sdesc_sw128(q_addr + 2 * u * kQBlockBytes, 16, 1024);
              const uint32_t dS = tmem + kSCol + 128 * buf;
              mma_pair(dS, a0, b0, kIdescQK, u ? 1u : 0u);
              mma_pair(dS, a0 + 2, b0 + 2, kIdescQK, 1u);
              mma_pair(dS, a0 + 4, b0 + 4, kIdescQK, 1u);
              mma_pair(dS, a0 + 6, b0 + 6, kIdescQK, 1u);
              if (un.nbox == 2) {
                constexpr uint64_t kA = kBoxBytes >> 4, kB = kQBlockBytes >> 4;
                mma_pair(dS, a0 + kA, b0 + kB, kIdescQK, 1u);
                mma_pair(dS, a0 + kA + 2, b0 + kB + 2, kIdescQK, 1u);
                mma_pair(dS, a0 + kA + 4, b0 + kB + 4, kIdescQK, 1u);
                mma_pair(dS, a0 + kA + 6, b0 + kB + 6, kIdescQK, 1u);
              }
              release(un);
            }
            commit_both(&bars->s_full[buf]);
            if (j == nr - 1) commit_both(&bars->q_empty);  // every MMA reading this query is issued
            ++g;
          }
          if (j >= 1) {
            // O^T (+)= V^T P^T over the round's 256 keys, two tiles of 256 dims
            if (!wait_cl(&bars->pt_full, gp & 1, wc)) goto mma_done;
            if (!wait_cl(&bars->pt_ready, gp & 1, wc)) goto mma_done;
            if (j == 1 && !wait_cl(&bars->o_empty, (n & 1) ^ 1, wc)) goto mma_done;
            tc_fence_after();
            fence_proxy_async_smem();
            for (int kh = 0; kh < 2; ++kh) {
              for (int t = 0; t < 2; ++t) {
                const Unit un = pv_unit(lo, j - 1, 0, kh, t);
                if (!take(un)) goto mma_done;
                // 16 keys per MMA: +16 rows of 128 bytes = +128 in both descriptors
                const uint64_t a0 = sdesc_sw128(smem_u32(smem + kRingOff + st * kUnitBytes), kBoxBytes, 1024);
                const uint64_t b0 = sdesc_sw128(pt_addr + kh * RK * 128, kBoxBytes, 1024);
                const uint32_t dO = tmem + kOCol + 128 * t;
                mma_pair(dO, a0, b0, kIdescPV, (j > 1 || kh > 0) ? 1u : 0u);
#pragma unroll
                for (int i = 1; i < RK / 16; ++i) mma_pair(dO, a0 + 128 * i, b0 + 128 * i, kIdescPV, 1u);
                release(un);
              }
            }
            commit_both(&bars->pv_done);
            ++gp;
          }
        }
      }
    mma_done:
      commit_local(&bars->fin);
      drain_wait_cl(&bars->fin, 0, a.wait_limit_ns);
    }
    __syncwarp();
  } else if (warp == 2) {
    // ------------------------------------------------------------ value-row fixer
    if (run) {
      PieceIter it;
      it.init(prefix, a.B, k_begin, k_end);
      uint32_t st = 0, tofixph = 0;
      int sb, lo, hi;
      const uint32_t fixed0 = cluster_addr(&bars->kv_fixed[0], 0);
      for (uint32_t n = 0; it.next(&sb, &lo, &hi); ++n) {
        const int L = prefix[sb + 1] - prefix[sb];
        const int nr = (hi - lo + kRoundKeys - 1) / kRoundKeys;
        const bool done = for_units(lo, nr, r, [&](const Unit& u) -> bool {
          if (u.rope_slot) return true;
          const uint32_t s = st;
          if (++st == kStages) st = 0;
          if (!needs_fix(u, L)) return true;
          if (!warp_wait_cl(&bars->kv_tofix[s], (tofixph >> s) & 1u, wc)) return false;
          tofixph ^= 1u << s;
          // rows [L - key0, 128) of both 64-dim boxes are past the sequence: zero them
          const int r0 = min(max(L - u.key0, 0), RK);
          uint8_t* base = smem + kRingOff + s * kUnitBytes;
          for (int idx = lane; idx < (RK - r0) * 16; idx += 32) {
            const int row = r0 + (idx >> 4), b = (idx >> 3) & 1, c = idx & 7;
            *reinterpret_cast<uint4*>(base + b * kBoxBytes + row * 128 + c * 16) = make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) arrive_cluster(fixed0 + s * 8);
          return true;
        });
        if (!done) break;
      }
    }
  } else if (warp == 3) {
    // ------------------------------------------------------------ query RoPE, hand-offs to the even CTA
    if (run) {
      PieceIter it;
      it.init(prefix, a.B, k_begin, k_end);
      const uint32_t q_ready0 = cluster_addr(&bars->q_ready, 0);
      const uint32_t pt_ready0 = cluster_addr(&bars->pt_ready, 0);
      uint32_t gp = 0;
      int sb, lo, hi;
      for (uint32_t n = 0; it.next(&sb, &lo, &hi); ++n) {
        const int L = prefix[sb + 1] - prefix[sb];
        const int nr = (hi - lo + kRoundKeys - 1) / kRoundKeys;
        if (!warp_wait_cl(&bars->q_full, n & 1, wc)) break;
        if (f.n_pairs) {
          // rotate dims [rope_offset, rope_offset + 2 n_pairs) of this CTA's 64 heads at the new token's position
          const int c0 = a.rope_offset / 8;  // first 8-dim chunk of the span
          for (int hl = lane; hl < HH; hl += 32) {
            uint8_t* row = smem + kQOff + hl * 128;
            auto chunk = [&](int c) {
              return reinterpret_cast<uint4*>(row + (c >> 3) * kQBlockBytes + (((c & 7) ^ (hl & 7)) << 4));
            };
            if (f.half) {
              for (int i = 0; i < f.n_pairs / 8; ++i) {
                uint4* p0 = chunk(c0 + i);
                uint4* p1 = chunk(c0 + i + f.n_pairs / 8);
                float x0[8], x1[8];
                bf16x8_to_f32(*p0, x0);
                bf16x8_to_f32(*p1, x1);
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                  float sn, cs;
                  rope_sincos(L - 1, f.hi[i * 8 + e], f.lo[i * 8 + e], &sn, &cs);
                  rotate_pair(x0[e], x1[e], sn, cs);
                }
                *p0 = f32_to_bf16x8(x0);
                *p1 = f32_to_bf16x8(x1);
              }
            } else {
              for (int i = 0; i < f.n_pairs / 4; ++i) {
                uint4* ptr = chunk(c0 + i);
                float x[8];
                bf16x8_to_f32(*ptr, x);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  float sn, cs;
                  rope_sincos(L - 1, f.hi[i * 4 + e], f.lo[i * 4 + e], &sn, &cs);
                  rotate_pair(x[2 * e], x[2 * e + 1], sn, cs);
                }
                *ptr = f32_to_bf16x8(x);
              }
            }
          }
          fence_proxy_async_smem();
        }
        __syncwarp();
        if (lane == 0) arrive_cluster(q_ready0);
        if (r == 1) {
          // this CTA's P^T of each round is complete (local rows + the even CTA's stores): make the stores
          // visible to the tensor cores' reads and tell the issuer
          bool ok = true;
          for (int j = 0; j < nr; ++j, ++gp) {
            if (!warp_wait_cl(&bars->pt_full, gp & 1, wc)) { ok = false; break; }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) arrive_cluster(pt_ready0);
          }
          if (!ok) break;
        }
      }
    }
  }
  } else {
    // ------------------------------------------------------------ softmax + epilogue (warps 4-11)
    setmaxnreg_inc<kRegsSoftmax>();
    const int sw = warp - 4;            // softmax warp 0..7
    const int qd = warp & 3;            // TMEM lane quarter: keys (S^T) / dims (O^T) 32 qd .. 32 qd + 31
    const int hh = sw >> 2;             // heads [64 hh, 64 hh + 64)
    const int key_l = 32 * qd + lane;   // this thread's key of the CTA's 128
    const uint32_t lane_off = static_cast<uint32_t>(32 * qd) << 16;
    float* red = reinterpret_cast<float*>(smem + kRedOff);        // [4][128]
    float* mw = reinterpret_cast<float*>(smem + kMOff) + sw * HH;  // this warp's copy of the 64 offsets
    float* facw = reinterpret_cast<float*>(smem + kFacOff) + sw * HH;  // this warp's rescale factors
    float* l_cta = reinterpret_cast<float*>(smem + kLOff);
    const float* l_peer = l_cta + NH;
    int* flags = reinterpret_cast<int*>(smem + kFlagOff);          // [2][8]
    const float* msg = reinterpret_cast<const float*>(smem + kMsgOff);
    const uint32_t msg_peer = cluster_addr(smem + kMsgOff, peer);
    const uint32_t msgbar_peer = cluster_addr(&bars->msg_full[0], peer);
    const uint32_t lpeer_addr = cluster_addr(smem + kLOff + NH * 4, peer);
    const uint32_t lbar_peer = cluster_addr(&bars->l_full, peer);
    const uint32_t sfree0 = cluster_addr(&bars->s_free[0], 0);
    const uint32_t oempty0 = cluster_addr(&bars->o_empty, 0);
    // this thread's P^T row (key 128 r + key_l of the round) in the CTA that supplies heads [64 hh, +64)
    const int prow = RK * r + key_l;
    const bool pt_local = hh == r;
    uint8_t* pt_row_local = smem + kPTOff + prow * 128;
    const uint32_t pt_row_peer = cluster_addr(smem + kPTOff + prow * 128, peer);
    const uint32_t ptbar_peer = cluster_addr(&bars->pt_full, peer);
    const float scl = a.scale_log2;
    const bool owner = qd == 0;   // warps 4 and 8: lane owns heads 64 hh + lane and 64 hh + lane + 32
    const bool armer = sw == 0 && lane == 0;
    PieceIter it;
    it.init(prefix, a.B, k_begin, k_end);
    uint32_t g = 0, hs1 = 0, pvw = 0;
    int sb, lo, hi;
    for (uint32_t n = 0; run && it.next(&sb, &lo, &hi); ++n) {
      const int nr = (hi - lo + kRoundKeys - 1) / kRoundKeys;
      float lsum[HH];
#pragma unroll
      for (int c = 0; c < HH; ++c) lsum[c] = 0.f;
      mw[lane] = kNoOffset;
      mw[lane + 32] = kNoOffset;
      __syncwarp();
      bool ok = true;
      for (int j = 0; j < nr; ++j, ++g) {
        const uint32_t buf = g & 1;
        if (!warp_wait_cl(&bars->s_full[buf], (g >> 1) & 1, wc)) { ok = false; break; }
        tc_fence_after();
        uint32_t sr[HH];
        tmem_ld32(tmem + lane_off + kSCol + 128 * buf + HH * hh, sr);
        tmem_ld32(tmem + lane_off + kSCol + 128 * buf + HH * hh + 32, sr + 32);
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) arrive_cluster(sfree0 + buf * 8);
        const bool valid = lo + j * kRoundKeys + RK * r + key_l < hi;
        float x[HH];
        float dmax = -INFINITY;
#pragma unroll
        for (int c = 0; c < HH; c += 4) {
          const float4 m4 = *reinterpret_cast<const float4*>(mw + c);
          const float mm[4] = {m4.x, m4.y, m4.z, m4.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            x[c + e] = valid ? __uint_as_float(sr[c + e]) * scl : -INFINITY;
            dmax = fmaxf(dmax, x[c + e] - mm[e]);
          }
        }
        // does any score of this CTA pass its head's offset by 2^8?
        const bool exceed = __any_sync(0xffffffffu, dmax > kRaise);
        if (lane == 0) flags[buf * 8 + sw] = exceed ? 1 : 0;
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->hsync[0]);  // one arrival per softmax warp
        if (!warp_wait_cl(&bars->hsync[0], g & 1, wc)) { ok = false; break; }
        int cta_exceed = 0;
#pragma unroll
        for (int w = 0; w < 8; ++w) cta_exceed |= flags[buf * 8 + w];
        float* mx_out = red;  // reused: per-quarter maxima, then read back
        if (cta_exceed) {
          // exact per-head maxima of this CTA's keys: over the warp's 32 keys, then the 4 quarters
#pragma unroll
          for (int c = 0; c < HH; ++c) {
            float v = x[c];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
            if ((c & 31) == lane) red[qd * NH + HH * hh + c] = v;
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars->hsync[1]);
          if (!warp_wait_cl(&bars->hsync[1], hs1++ & 1, wc)) { ok = false; break; }
        }
        // the message to the other CTA: the flag, and this CTA's maxima of the owner's two heads
        if (owner) {
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int h = HH * hh + lane + 32 * e;
            float v = -INFINITY;
            if (cta_exceed)
              v = fmaxf(fmaxf(mx_out[h], mx_out[NH + h]), fmaxf(mx_out[2 * NH + h], mx_out[3 * NH + h]));
            st_async_b32(msg_peer + (buf * kMsgWords + h) * 4, __float_as_uint(v), msgbar_peer + buf * 8);
          }
        }
        if (sw == 0 && lane == 0)
          st_async_b32(msg_peer + (buf * kMsgWords + NH) * 4, static_cast<uint32_t>(cta_exceed),
                       msgbar_peer + buf * 8);
        if (!warp_wait_cl(&bars->msg_full[buf], (g >> 1) & 1, wc)) { ok = false; break; }
        const float* pm = msg + buf * kMsgWords;
        const int peer_exceed = __float_as_int(pm[NH]);
        // new offsets: where the pair's maximum passed a head's offset by 2^8, the offset moves to it; each
        // lane decides its two columns, the warp reads them back after a __syncwarp
        bool any_changed = false;
        if (cta_exceed | peer_exceed) {
          bool ch = false;
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int c = lane + 32 * e, h = HH * hh + c;
            float M = pm[h];
            if (cta_exceed) M = fmaxf(M, fmaxf(fmaxf(red[h], red[NH + h]), fmaxf(red[2 * NH + h], red[3 * NH + h])));
            const float mo = mw[c];
            const float mn = M > mo + kRaise ? M : mo;
            facw[c] = mn != mo ? fast_exp2(mo - mn) : 1.f;
            ch |= mn != mo;
            mw[c] = mn;
          }
          any_changed = __any_sync(0xffffffffu, ch);
          __syncwarp();
        }
#pragma unroll
        for (int c = 0; c < HH; c += 4) {
          const float4 m4 = *reinterpret_cast<const float4*>(mw + c);
          x[c] -= m4.x;
          x[c + 1] -= m4.y;
          x[c + 2] -= m4.z;
          x[c + 3] -= m4.w;
        }
        if (any_changed) {
#pragma unroll
          for (int c = 0; c < HH; c += 4) {
            const float4 f4 = *reinterpret_cast<const float4*>(facw + c);
            lsum[c] *= f4.x;
            lsum[c + 1] *= f4.y;
            lsum[c + 2] *= f4.z;
            lsum[c + 3] *= f4.w;
          }
        }
        if (armer) mbar_arrive_expect_tx(&bars->msg_full[buf], kMsgBytes);  // round g + 2's message
        // probabilities (bf16 pairs) and the running sums
        uint32_t pr[HH / 2];
#pragma unroll
        for (int c = 0; c < HH / 2; ++c) {
          const float p0 = fast_exp2(x[2 * c]);
          const float p1 = fast_exp2(x[2 * c + 1]);
          lsum[2 * c] += p0;
          lsum[2 * c + 1] += p1;
          pr[c] = pack_bf16x2(p0, p1);
        }
        // the previous round's P V has completed: P^T may be overwritten and O^T rescaled
        if (j >= 1) {
          if (!warp_wait_cl(&bars->pv_done, pvw & 1, wc)) { ok = false; break; }
          ++pvw;
          tc_fence_after();
          if (any_changed) {
            scale_cols64(tmem + lane_off + kOCol + HH * hh, facw);
            scale_cols64(tmem + lane_off + kOCol + 128 + HH * hh, facw);
            tmem_wait_st();
          }
        }
        // P^T row: heads [64 hh, +64) of this key, 128-byte swizzled, in the CTA that supplies those heads
        if (pt_local) {
#pragma unroll
          for (int i = 0; i < 8; ++i)
            *reinterpret_cast<uint4*>(pt_row_local + ((i ^ (prow & 7)) << 4)) =
                make_uint4(pr[4 * i], pr[4 * i + 1], pr[4 * i + 2], pr[4 * i + 3]);
          fence_proxy_async_smem();
        } else {
#pragma unroll
          for (int i = 0; i < 8; ++i)
            st_async_v4(pt_row_peer + ((i ^ (prow & 7)) << 4), pr[4 * i], pr[4 * i + 1], pr[4 * i + 2],
                        pr[4 * i + 3], ptbar_peer);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if (sw == 0) mbar_arrive_expect_tx(&bars->pt_full, kPTPeerBytes);
          else mbar_arrive(&bars->pt_full);
        }
      }
      if (!__all_sync(0xffffffffu, ok)) break;
      // ---- epilogue: the piece's row sums over both CTAs, then O^T / l -> the partial of (pair, sequence)
      if (!warp_wait_cl(&bars->pv_done, pvw & 1, wc)) break;
      ++pvw;
      tc_fence_after();
#pragma unroll
      for (int c = 0; c < HH; ++c) {
        float v = lsum[c];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if ((c & 31) == lane) red[qd * NH + HH * hh + c] = v;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->hsync[1]);
      if (!warp_wait_cl(&bars->hsync[1], hs1++ & 1, wc)) break;
      if (owner) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int h = HH * hh + lane + 32 * e;
          const float v = (red[h] + red[NH + h]) + (red[2 * NH + h] + red[3 * NH + h]);
          l_cta[h] = v;
          st_async_b32(lpeer_addr + h * 4, __float_as_uint(v), lbar_peer);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->hsync[1]);
      if (!warp_wait_cl(&bars->hsync[1], hs1++ & 1, wc)) break;
      if (!warp_wait_cl(&bars->l_full, n & 1, wc)) break;
      const long long slot = static_cast<long long>(p) + sb;  // unique per (pair, sequence)
#pragma unroll 1
      for (int t = 0; t < 2; ++t) {
        const int dim = 256 * t + 128 * r + key_l;  // this thread's O^T row of tile t
#pragma unroll 1
        for (int cc = 0; cc < 2; ++cc) {
          uint32_t o[32];
          tmem_ld32(tmem + lane_off + kOCol + 128 * t + HH * hh + 32 * cc, o);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const int h = HH * hh + 32 * cc + e;
            const float inv_l = 1.f / (l_cta[h] + l_peer[h]);
            a.ws_o[(slot * a.n_h + h) * DV + dim] = __uint_as_float(o[e]) * inv_l;
          }
        }
      }
      if (r == 0 && owner) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int c = lane + 32 * e, h = HH * hh + c;
          a.ws_lse[slot * a.n_h + h] = mw[c] + log2f(l_cta[h] + l_peer[h]);
        }
      }
      tc_fence_before();
      __syncwarp();
      // the next piece's sums may land once its phase is armed (not before every thread of this CTA has
      // finished this piece's rounds, which the other CTA's next epilogue waits for)
      if (armer) mbar_arrive_expect_tx(&bars->l_full, NH * 4);
      if (lane == 0) arrive_cluster(oempty0);
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

// out[b, h, :] = sum over the pieces of sequence b of 2^(lse_j - lse) O_j.  One warp
// per (b, h), no block-wide step: the lanes find the pairs that hold sequence b's keys,
// reduce the pieces' maximum and weight sum by shuffles, and each lane accumulates 16 of
// the 512 dims with 16-byte loads of the partials.
constexpr int kCombineWarps = 8;

__global__ void __launch_bounds__(kCombineWarps * 32) mla_combine_kernel(DecodeArgs a) {
  const int lane = threadIdx.x & 31;
  const int bh = blockIdx.x * kCombineWarps + (threadIdx.x >> 5);
  if (bh >= a.B * a.n_h) return;  // whole warps only
  const int b = bh / a.n_h, h = bh % a.n_h;
  const int P = a.n_split;  // pairs
  long long before = 0, total = 0;
  for (int i = lane; i < a.B; i += 32) {
    const long long L = min(max(a.seqlens[i], 1), a.max_len);
    total += L;
    if (i < b) before += L;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    before += __shfl_xor_sync(0xffffffffu, before, o);
    total += __shfl_xor_sync(0xffffffffu, total, o);
  }
  const long long Teff = total + kPieceGap * (a.B - 1);
  const long long Lb = min(max(a.seqlens[b], 1), a.max_len);
  const long long e0 = before + kPieceGap * b;  // effective position of
  const long long e1 = e0 + Lb - 1;              // sequence b's first, last key
  // pair holding effective position e: the largest p with floor(p Teff / P) <= e.  Rounding the
  // starts down to whole rounds moves keys of b only between these pairs: no pair before p_lo
  // starts inside b, and a pair after p_hi starts at or after b's end, where nothing is rounded.
  const int p_lo = static_cast<int>(((e0 + 1) * P - 1) / Teff);
  const int p_hi = static_cast<int>(((e1 + 1) * P - 1) / Teff);
  const int np = p_hi - p_lo + 1;
  auto start_in_b = [&](int q) -> long long {  // pair q's first key as an offset into b, clamped to [0, Lb]
    const long long E = pair_start_eff(q, Teff, P);
    if (E <= e0) return 0;
    return E - e0 < Lb ? round_down_keys(E - e0) : Lb;
  };
  auto piece_lse = [&](int j) {  // -inf for a pair that holds no key of b (it wrote nothing for b)
    if (start_in_b(p_lo + j + 1) <= start_in_b(p_lo + j)) return -INFINITY;
    return a.ws_lse[(static_cast<long long>(p_lo + j) + b) * a.n_h + h];
  };
  float M = -INFINITY;
  for (int j = lane; j < np; j += 32) M = fmaxf(M, piece_lse(j));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  float den = 0.f;
  float4 acc[4];
#pragma unroll
  for (int c = 0; c < 4; ++c) acc[c] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int j0 = 0; j0 < np; j0 += 32) {
    const float l = j0 + lane < np ? piece_lse(j0 + lane) : -INFINITY;
    const float wl = l == -INFINITY ? 0.f : exp2f(l - M);
    den += wl;
    const int nj = min(32, np - j0);
    for (int jj = 0; jj < nj; ++jj) {
      const float w = __shfl_sync(0xffffffffu, wl, jj);
      if (w == 0.f) continue;  // uniform across the warp
      const float4* o = reinterpret_cast<const float4*>(
          a.ws_o + ((static_cast<long long>(p_lo + j0 + jj) + b) * a.n_h + h) * DV);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const float4 v = o[c * 32 + lane];
        acc[c].x = fmaf(w, v.x, acc[c].x);
        acc[c].y = fmaf(w, v.y, acc[c].y);
        acc[c].z = fmaf(w, v.z, acc[c].z);
        acc[c].w = fmaf(w, v.w, acc[c].w);
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
  const float inv = 1.f / den;
  __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out) + static_cast<long long>(bh) * DV;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const __nv_bfloat162 lo = __floats2bfloat162_rn(acc[c].x * inv, acc[c].y * inv);
    const __nv_bfloat162 hi = __floats2bfloat162_rn(acc[c].z * inv, acc[c].w * inv);
    uint2 u;
    u.x = *reinterpret_cast<const uint32_t*>(&lo);
    u.y = *reinterpret_cast<const uint32_t*>(&hi);
    *reinterpret_cast<uint2*>(out + (c * 32 + lane) * 4) = u;
  }
  if (a.lse != nullptr && lane == 0) a.lse[bh] = (M + log2f(den)) * 0.69314718055994530942f;
}

}  // namespace

bool decode_mla_supported(int B, int n_h, int n_kv, int D_qk, int D_v, long long v_token_stride, bool v_is_k,
                          bool bf16) {
  return bf16 && n_h == NH && n_kv == 1 && D_qk == DQK && D_v == DV && v_is_k && v_token_stride == DQK &&
         B <= kMaxB;
}

bool decode_mla_rope_ok(int rope_offset, int rope_dims, bool half) {
  // the query lives in shared memory: the rotated span must be whole 8-dim chunks
  return rope_offset % 8 == 0 && rope_dims % (half ? 16 : 8) == 0 && rope_offset + rope_dims <= DQK;
}

namespace {
std::atomic<unsigned> g_mla_ready{0};  // one bit per device whose shared-memory opt-in is done
std::atomic<int> g_mla_pairs[32];      // per device: clusters of two CTAs that fit at once (0: not known)

cudaError_t mla_prepare(int dev) {
  const unsigned bit = 1u << (dev & 31);
  if (g_mla_ready.load(std::memory_order_acquire) & bit) return cudaSuccess;
  // the register split must fit the registers the compiled kernel launches with
  cudaFuncAttributes fa;
  cudaError_t e = cudaFuncGetAttributes(&fa, mla_decode_kernel);
  if (e != cudaSuccess) return e;
  if (static_cast<long long>(fa.numRegs) * kThreads < kRegsNeeded) return cudaErrorInvalidConfiguration;
  e = cudaFuncSetAttribute(mla_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  g_mla_ready.fetch_or(bit, std::memory_order_acq_rel);
  return cudaSuccess;
}

void mla_config(cudaLaunchConfig_t* cfg, cudaLaunchAttribute* attr, int pairs, cudaStream_t st) {
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
}  // namespace

int decode_mla_pairs(int num_sms) {
  int p = num_sms / 2;
  int dev = 0;
  if (cudaGetDevice(&dev) == cudaSuccess && dev < 32) {
    int known = g_mla_pairs[dev].load(std::memory_order_acquire);
    if (known == 0 && mla_prepare(dev) == cudaSuccess) {
      // every pair must be resident at once (the pairs of a GPC pair up its SMs)
      cudaLaunchConfig_t cfg = {};
      cudaLaunchAttribute attr;
      mla_config(&cfg, &attr, p < 1 ? 1 : p, nullptr);
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(&n, mla_decode_kernel, &cfg) == cudaSuccess && n > 0) known = n;
      else (void)cudaGetLastError();
      if (known > 0) g_mla_pairs[dev].store(known, std::memory_order_release);
    }
    if (known > 0 && known < p) p = known;
  }
  return p < 1 ? 1 : (p > kMlaMaxPairs ? kMlaMaxPairs : p);
}

cudaError_t launch_decode_mla(const DecodeArgs& a, const RopeFreq& rope, const CUtensorMap* maps, cudaStream_t st,
                              int* launches) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if ((e = mla_prepare(dev)) != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr;
  mla_config(&cfg, &attr, a.n_split, st);
  e = cudaLaunchKernelEx(&cfg, mla_decode_kernel, a, rope, maps[0], maps[1]);
  *launches += 1;
  if (e != cudaSuccess) return e;
  mla_combine_kernel<<<(a.B * a.n_h + kCombineWarps - 1) / kCombineWarps, kCombineWarps * 32, 0, st>>>(a);
  *launches += 1;
  return cudaGetLastError();
}

}  // namespace attn

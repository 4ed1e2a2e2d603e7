// decode_mla.cu - MLA-absorbed decode on the tensor cores (sm_103a).
//
// "Transformer 与 LLM" slide 06: after W_UK is folded into the query and W_UV
// into the output, the 128 query heads of a token share one 576-dim latent KV
// head [c^KV (512) ; k^R (64)], V is the first 512 latent dims, and the scores
// use 1/sqrt(192).  Per cached key the work is 128 x (576 + 512) multiply-adds
// against 1152 bytes read - about 242 FLOP per byte, at the ridge of the GPU,
// so both the tensor cores and HBM must run near their peaks.
//
// Mapping.  The fp32 output O is 128 heads x 512 dims = all 512 TMEM columns of
// an SM, so the two CTAs of a cluster share it: CTA r accumulates the value
// dims [256 r, 256 r + 256).  The pair walks its keys in rounds of 256; in each
// round CTA r scores its own 128 keys (S = Q C^T, M = 128 heads, N = 128 keys,
// K = 576: full tensor-core rate and no score is computed twice), turns them
// into bf16 probabilities P, keeps P in TMEM for its own P V and writes a copy
// into the other CTA's shared memory (distributed shared memory), so that each
// CTA then accumulates O_half += P_own V_own,half + P_peer V_peer,half
// (M = 128 heads, N = 128 dims per MMA, K = 128 keys).
//
// Softmax offsets.  Each row's exponent offset is shared by the pair and moves
// lazily: a round's probabilities use the offset agreed after the previous
// round, so no round waits for the other CTA before its exponentials.  With the
// probabilities each CTA sends its offset, its row maxima and row sums; both
// CTAs then apply the same rule (raise the offset when a row maximum passes it
// by 2^8) and so stay in step.  A CTA whose scores pass the shared offset by
// 2^64 (fp32/bf16 range) uses its own row maximum instead, and the receiving
// side brings the two halves to the larger offset by scaling O or the peer's P
// down - both factors are at most one.
//
// The copy goes out as asynchronous remote stores that count their bytes on the
// peer's barrier (st.async with complete_tx), so no fence or remote arrive is
// on the sending side.
//
// Loads.  Cache rows stream through a 3-stage ring of 32 KB units (128 keys x
// 128 dims, two 128-byte-swizzled TMA boxes): five units per round for the
// scores (the 576 dims), then two of the own keys and two of the peer's keys
// for P V, restricted to this CTA's value dims (the second read of a row hits
// L2).  No L2 prefetch: requests ahead of the ring (tensor or bulk prefetch
// through the TMA engine, or plain prefetches from an idle warp) measured
// slower or equal.  The query's dims [0, 256) live in TMEM (the score MMA's A
// operand), dims [256, 576) in shared memory.  Rows at or past a sequence's end
// may hold anything, so a helper warp zeroes them in the value units before
// their MMA.  The tensor-core work of round j is issued as P V(own, j), the
// scores of round j + 1, P V(peer, j): the peer's probabilities arrive while the
// next scores run.
//
// Keys of all sequences, laid end to end, are split evenly over the pairs (a
// pair's range may cross sequence boundaries), so every pair does the same
// work; each (pair, sequence) piece writes one normalised partial, merged per
// sequence by mla_combine_kernel with the log-sum-exp rule of the online
// softmax ("Transformer架构完全深度解析" §13).
// Roles (384 threads): warp 0 TMA producer, warp 1 TMEM owner + single-thread
// MMA issuer, warp 2 key prefix sums, then the value-row fixer, warps 4-11
// softmax (two warps per 32 heads = TMEM lanes, 64 keys each) and epilogue.
#include <math.h>

#include <atomic>

#include "kernels.h"

namespace attn {
namespace {

constexpr int NH = 128;              // query heads (MMA M)
constexpr int DQK = 576;             // latent + rotary dims
constexpr int DV = 512;              // value dims
constexpr int DVH = 256;             // value dims per CTA of a pair
constexpr int RK = kMlaTileKeys;     // keys per CTA per round (MMA N of the score tile)
constexpr int kRoundKeys = 2 * RK;
constexpr int kThreads = 384;
constexpr int kBlockBytes = RK * 128;        // 128 rows x 64 bf16 dims, 128-byte swizzled
constexpr int kUnitBytes = 2 * kBlockBytes;  // one ring stage
constexpr int kStages = 3;
constexpr int kQkUnits = 5;                  // dims [0,128) [128,256) [256,384) [384,512) [512,576)
constexpr int kQTmemDims = kMlaQTmemDims;    // query dims [0, 256) live in TMEM
constexpr int kQSmemBlocks = (DQK - kQTmemDims) / 64;  // dims [256, 576) in shared memory: 5 blocks
static_assert(NH == RK, "query blocks and cache blocks share one box shape");
static_assert(kQTmemDims == 256, "the score units 0 and 1 read the query from TMEM");
constexpr int kQSmemBytes = kQSmemBlocks * kBlockBytes;  // 80 KB
constexpr int kMaxB = 256;  // the batch's key prefix sums live in shared memory
constexpr int kQOff = 0;
constexpr int kRingOff = kQOff + kQSmemBytes;
constexpr int kPPOff = kRingOff + kStages * kUnitBytes;  // the peer's P: 2 blocks (keys 0-63, 64-127)
constexpr int kMsgOff = kPPOff + 2 * kBlockBytes;        // the peer's offsets, maxima, row sums
constexpr int kRedOff = kMsgOff + 4 * NH * 4;            // row maxima of the two key halves, 2 rounds; row sums
constexpr int kPrefOff = kRedOff + 6 * NH * 4;
constexpr int kBarOff = kPrefOff + ((kMaxB + 1) * 4 + 63) / 64 * 64;
constexpr int kUsedBytes = kBarOff + 512;
constexpr int kSmemBytes = kUsedBytes + 1024;  // + slack to align the base to 1024 bytes
static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");
// TMEM columns: S (fp32, 128) whose first halves of each 64-key half take P as bf16 pairs,
// O_half (256), the query dims [0, 256) as bf16 pairs (128)
constexpr uint32_t kSCol = 0;
constexpr uint32_t kOCol = 128;
constexpr uint32_t kQCol = 384;
constexpr uint32_t kIdescQK = idesc_bf16_f32(NH, RK, false);
constexpr uint32_t kIdescPV = idesc_bf16_f32(NH, 128, true);
constexpr float kRaise = 8.0f;       // the shared offset moves when a row maximum passes it by 2^8
constexpr float kEmergency = 64.0f;  // a CTA uses its own maximum when its scores pass the offset by 2^64
// bytes the peer stores per round: P (128 heads x 128 keys bf16), offsets, maxima, row sums
constexpr uint32_t kMsgBytes = NH * RK * 2 + 4 * NH * 4;

struct Msg {  // written by the peer CTA each round
  float m_own[NH];  // offset its P used
  float mx[NH];     // its row maxima (log2 domain)
  float rs[2][NH];  // its row sums, per 64-key half
};
static_assert(sizeof(Msg) == 4 * NH * 4, "message layout");

struct Bars {
  uint64_t q_full, q_ready, q_empty;
  uint64_t kv_full[kStages], kv_tofix[kStages], kv_fixed[kStages], kv_empty[kStages];
  uint64_t s_full, p_ready, pvo_done, pp_full, pp_ready, pvp_done, pp_empty;
  uint64_t o_empty, fin;
  uint64_t hsync[4];  // the two softmax warps of 32 heads exchange row maxima / sums (64 arrivals)
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(Bars) <= 512, "barrier block");

// First key (in the concatenation of all sequences) of pair p.
__device__ __forceinline__ long long pair_start(int p, long long T, int P) {
  return static_cast<long long>(p) * T / P;
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
  // next piece: sequence *sb, keys [*lo, *hi) of that sequence
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

// One unit of a piece's load stream: keys [key0, key0 + 128) of the sequence,
// 64-dim blocks [blk0, blk0 + nblk).  Value units are read by P V.
struct Unit {
  int key0, blk0, nblk;
  bool pv;
};
__device__ __forceinline__ Unit qk_unit(int lo, int j, int r, int u) {
  return Unit{lo + j * kRoundKeys + r * RK, 2 * u, u == kQkUnits - 1 ? 1 : 2, false};
}
__device__ __forceinline__ Unit pv_unit(int lo, int j, int owner, int r, int v) {
  return Unit{lo + j * kRoundKeys + owner * RK, 4 * r + 2 * v, 2, true};
}
// A value unit reaching past the sequence (length L) has rows to clear.
__device__ __forceinline__ bool needs_fix(const Unit& u, int L) { return u.pv && u.key0 + RK > L; }

// Every unit of a piece with nr rounds, in the order the MMA issuer takes them:
// scores(0), then per round j: P V(own, j), scores(j + 1), P V(peer, j).
template <typename F>
__device__ __forceinline__ bool for_units(int lo, int nr, int r, F&& f) {
  for (int u = 0; u < kQkUnits; ++u)
    if (!f(qk_unit(lo, 0, r, u), 0)) return false;
  for (int j = 0; j < nr; ++j) {
    for (int v = 0; v < 2; ++v)
      if (!f(pv_unit(lo, j, r, r, v), j)) return false;
    if (j + 1 < nr)
      for (int u = 0; u < kQkUnits; ++u)
        if (!f(qk_unit(lo, j + 1, r, u), j + 1)) return false;
    for (int v = 0; v < 2; ++v)
      if (!f(pv_unit(lo, j, r ^ 1, r, v), j)) return false;
  }
  return true;
}

__device__ __forceinline__ void tma_load_3d(void* smem_dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1,
                                            int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, const WaitCtl& w) {
  const bool ok = mbar_wait(bar, parity, w);
  return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity, unsigned long long limit_ns) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > limit_ns) return;
  }
}

// ---- cluster (distributed shared memory) helpers
__device__ __forceinline__ uint32_t peer_addr(const void* local, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(local)), "r"(rank));
  return r;
}
// Asynchronous stores into the peer CTA's shared memory; each counts its bytes on the
// peer's barrier (complete_tx), so the peer sees them once its barrier phase completes.
__device__ __forceinline__ void st_peer_v4(uint32_t addr, uint32_t x, uint32_t y, uint32_t z, uint32_t w,
                                           uint32_t bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(
                   addr),
               "r"(x), "r"(y), "r"(z), "r"(w), "r"(bar)
               : "memory");
}
__device__ __forceinline__ void st_peer_f32(uint32_t addr, float v, uint32_t bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];" ::"r"(addr),
               "r"(__float_as_uint(v)), "r"(bar)
               : "memory");
}
__device__ __forceinline__ bool try_wait_cluster(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait on a barrier that the other CTA arrives on (acquire at cluster scope).
__device__ __forceinline__ bool wait_cluster(uint64_t* bar, uint32_t parity, const WaitCtl& w) {
  if (try_wait_cluster(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (try_wait_cluster(bar, parity)) return true;
    if ((it & 63u) == 0u) {
      if (*w.abort_flag) return false;
      if (globaltimer_ns() - t0 > w.limit_ns) {
        *w.abort_flag = 1;
        atomicOr(w.status, STATUS_TIMEOUT);
        return false;
      }
    }
  }
}
__device__ __forceinline__ bool warp_wait_cluster(uint64_t* bar, uint32_t parity, const WaitCtl& w) {
  const bool ok = wait_cluster(bar, parity, w);
  return __all_sync(0xffffffffu, ok);
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Arrive once on the barrier at the same offset in the CTAs of mask when every
// tcgen05 operation issued so far by this thread completes.
__device__ __forceinline__ void mma_commit_mc(uint64_t* bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          smem_u32(bar)),
      "h"(mask)
      : "memory");
}

// O_half columns [kOCol + 128 kh, + 128) of this thread's row times f.  The TMEM loads and
// stores are warp-collective: every lane of the warp calls this (f = 1 where nothing moves).
__device__ __forceinline__ void scale_o(uint32_t taddr, float f) {
#pragma unroll 1
  for (int c = 0; c < 4; ++c) {
    uint32_t o[32];
    tmem_ld32(taddr + c * 32, o);
    tmem_wait_ld();
#pragma unroll
    for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * f);
    tmem_st32(taddr + c * 32, o);
  }
  tmem_wait_st();
}

__global__ void __launch_bounds__(kThreads, 1)
    mla_decode_kernel(const __grid_constant__ DecodeArgs a, const __grid_constant__ RopeFreq f,
                      const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_c) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Bars* bars = reinterpret_cast<Bars*>(smem + kBarOff);
  int* prefix = reinterpret_cast<int*>(smem + kPrefOff);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int P = gridDim.x >> 1;           // pairs (clusters of two CTAs)
  const int p = blockIdx.x >> 1;          // this CTA's pair
  const int r = blockIdx.x & 1;           // rank in the cluster = value-dim half
  const bool layout_ok = static_cast<int>(smem - smem_raw) + kUsedBytes <= kSmemBytes;

  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
    mbar_init(&bars->q_ready, 128);
    mbar_init(&bars->q_empty, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bars->kv_full[s], 1);
      mbar_init(&bars->kv_tofix[s], 1);
      mbar_init(&bars->kv_fixed[s], 1);
      mbar_init(&bars->kv_empty[s], 1);
    }
    mbar_init(&bars->s_full, 1);
    mbar_init(&bars->p_ready, 256);
    mbar_init(&bars->pvo_done, 1);
    mbar_init(&bars->pp_full, 1);  // armed locally each round with the message's byte count
    mbar_arrive_expect_tx(&bars->pp_full, kMsgBytes);  // round 0, before the peer can store
    mbar_init(&bars->pp_ready, 256);
    mbar_init(&bars->pvp_done, 1);
    mbar_init(&bars->pp_empty, 1);
    mbar_init(&bars->o_empty, 256);
    mbar_init(&bars->fin, 1);
    for (int i = 0; i < 4; ++i) mbar_init(&bars->hsync[i], 64);
    bars->abort_flag = layout_ok ? 0 : 1;
    if (!layout_ok) atomicOr(a.status, STATUS_LAYOUT);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&bars->tmem_base, 512);
    tmem_relinquish();
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
  cluster_sync();  // both CTAs' barriers are initialised before either arrives remotely
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  const WaitCtl wc{&bars->abort_flag, a.status, a.wait_limit_ns};
  const long long T = prefix[a.B];
  const long long k_begin = pair_start(p, T, P), k_end = pair_start(p + 1, T, P);
  const bool run = !bars->abort_flag;  // false: the shared-memory layout did not fit, touch nothing

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0 && run) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_c);
      PieceIter it;
      it.init(prefix, a.B, k_begin, k_end);
      uint32_t st = 0, ph = 0, q_issued = 0, issued = 0;
      uint64_t* last_bar[kStages] = {};
      uint32_t last_par[kStages] = {};
      uint32_t fullph = 0, fixph = 0;  // bit s: phase of kv_full[s] / kv_tofix[s]
      int sb, lo, hi;
      for (uint32_t n = 0; it.next(&sb, &lo, &hi); ++n) {
        const int L = prefix[sb + 1] - prefix[sb];
        const int nr = (hi - lo + kRoundKeys - 1) / kRoundKeys;
        if (!mbar_wait(&bars->q_empty, (n & 1) ^ 1, wc)) break;
        mbar_arrive_expect_tx(&bars->q_full, kQSmemBytes);
        for (int blk = 0; blk < kQSmemBlocks; ++blk)
          tma_load_3d(smem + kQOff + blk * kBlockBytes, &tm_q, &bars->q_full, kQTmemDims + blk * 64, 0, sb);
        q_issued = n + 1;
        const bool done = for_units(lo, nr, r, [&](const Unit& u, int) -> bool {
          if (!mbar_wait(&bars->kv_empty[st], ph ^ 1, wc)) return false;
          const bool fix = needs_fix(u, L);
          uint64_t* bar = fix ? &bars->kv_tofix[st] : &bars->kv_full[st];
          uint32_t& bits = fix ? fixph : fullph;
          mbar_arrive_expect_tx(bar, u.nblk * kBlockBytes);
          uint8_t* dst = smem + kRingOff + st * kUnitBytes;
          for (int b = 0; b < u.nblk; ++b) tma_load_3d(dst + b * kBlockBytes, &tm_c, bar, (u.blk0 + b) * 64, u.key0, sb);
          last_bar[st] = bar;
          last_par[st] = (bits >> st) & 1u;
          bits ^= 1u << st;
          issued |= 1u << st;
          if (++st == kStages) { st = 0; ph ^= 1; }
          return true;
        });
        if (!done) break;
      }
      if (bars->abort_flag) {  // let every copy in flight land before the CTA may exit
        for (int s = 0; s < kStages; ++s)
          if (issued & (1u << s)) drain_wait(last_bar[s], last_par[s], a.wait_limit_ns);
        if (q_issued) drain_wait(&bars->q_full, (q_issued - 1) & 1, a.wait_limit_ns);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && run) {
      PieceIter it;
      it.init(prefix, a.B, k_begin, k_end);
      const uint32_t q_addr = smem_u32(smem + kQOff);
      const uint32_t pp_addr = smem_u32(smem + kPPOff);
      uint32_t st = 0, fullph = 0, fixph = 0, G = 0;
      int sb, lo, hi, L = 0;
      // wait for the unit in the current stage (cleared value units come through the fixer)
      auto take = [&](const Unit& u) -> bool {
        if (needs_fix(u, L)) {
          if (!mbar_wait(&bars->kv_fixed[st], (fixph >> st) & 1u, wc)) return false;
          fixph ^= 1u << st;
        } else {
          if (!mbar_wait(&bars->kv_full[st], (fullph >> st) & 1u, wc)) return false;
          fullph ^= 1u << st;
        }
        tc_fence_after();
        return true;
      };
      auto release = [&]() {
        mma_commit(&bars->kv_empty[st]);
        if (++st == kStages) st = 0;
      };
      // S (+)= Q[:, dims of unit u] C[keys, dims of unit u]^T
      auto issue_qk = [&](int u) {
        const uint32_t kaddr = smem_u32(smem + kRingOff + st * kUnitBytes);
        const int nb = u == kQkUnits - 1 ? 1 : 2;
        for (int b = 0; b < nb; ++b) {
#pragma unroll
          for (int k4 = 0; k4 < 4; ++k4) {
            const int kk = 8 * u + 4 * b + k4;  // 16-dim step over the 576 dims
            const uint64_t bdesc = sdesc_sw128(kaddr + b * kBlockBytes + k4 * 32, 16, 1024);
            if (kk < kQTmemDims / 16) {
              mma_ts(tmem + kSCol, tmem + kQCol + kk * 8, bdesc, kIdescQK, kk > 0 ? 1u : 0u);
            } else {
              const int kq = kk - kQTmemDims / 16;
              mma_ss(tmem + kSCol, sdesc_sw128(q_addr + (kq >> 2) * kBlockBytes + (kq & 3) * 32, 16, 1024), bdesc,
                     kIdescQK, 1u);
            }
          }
        }
      };
      // O_half[:, 128 v .. 128 v + 128) (+)= P C[keys, value dims]: P from TMEM (own keys) or from
      // the peer's copy in shared memory
      auto issue_pv = [&](int v, bool own, bool accumulate) {
        const uint32_t vaddr = smem_u32(smem + kRingOff + st * kUnitBytes);
#pragma unroll
        for (int kk = 0; kk < RK / 16; ++kk) {
          const uint64_t bdesc = sdesc_sw128(vaddr + kk * 16 * 128, kBlockBytes, 1024);
          const uint32_t acc = (accumulate || kk > 0) ? 1u : 0u;
          if (own)
            mma_ts(tmem + kOCol + 128 * v, tmem + kSCol + (kk >> 2) * 64 + (kk & 3) * 8, bdesc, kIdescPV, acc);
          else
            mma_ss(tmem + kOCol + 128 * v,
                   sdesc_sw128(pp_addr + (kk >> 2) * kBlockBytes + (kk & 3) * 32, 16, 1024), bdesc, kIdescPV, acc);
        }
      };
      auto scores = [&](int j) -> bool {
        for (int u = 0; u < kQkUnits; ++u) {
          if (!take(qk_unit(lo, j, r, u))) return false;
          issue_qk(u);
          release();
        }
        mma_commit(&bars->s_full);
        return true;
      };
      const uint16_t peer_mask = static_cast<uint16_t>(1u << (r ^ 1));
      for (uint32_t n = 0; it.next(&sb, &lo, &hi); ++n) {
        L = prefix[sb + 1] - prefix[sb];
        const int nr = (hi - lo + kRoundKeys - 1) / kRoundKeys;
        if (!mbar_wait(&bars->q_ready, n & 1, wc)) goto mma_done;
        tc_fence_after();
        if (!scores(0)) goto mma_done;
        if (nr == 1) mma_commit(&bars->q_empty);  // every MMA reading this query is issued
        for (int j = 0; j < nr; ++j, ++G) {
          if (!mbar_wait(&bars->p_ready, G & 1, wc)) goto mma_done;
          if (j == 0 && !mbar_wait(&bars->o_empty, (n & 1) ^ 1, wc)) goto mma_done;
          tc_fence_after();
          for (int v = 0; v < 2; ++v) {
            if (!take(pv_unit(lo, j, r, r, v))) goto mma_done;
            issue_pv(v, true, j > 0);
            release();
          }
          mma_commit(&bars->pvo_done);
          if (j + 1 < nr) {
            if (!scores(j + 1)) goto mma_done;
            if (j + 1 == nr - 1) mma_commit(&bars->q_empty);
          }
          if (!mbar_wait(&bars->pp_ready, G & 1, wc)) goto mma_done;
          tc_fence_after();
          fence_proxy_async_smem();
          for (int v = 0; v < 2; ++v) {
            if (!take(pv_unit(lo, j, r ^ 1, r, v))) goto mma_done;
            issue_pv(v, false, true);
            release();
          }
          mma_commit(&bars->pvp_done);
          mma_commit_mc(&bars->pp_empty, peer_mask);  // the peer may write its next P here
        }
      }
    mma_done:
      mma_commit(&bars->fin);
      drain_wait(&bars->fin, 0, a.wait_limit_ns);
    }
    __syncwarp();
  } else if (warp == 2) {
    // ------------------------------------------------------------ value-row fixer
    if (run) {
      PieceIter it;
      it.init(prefix, a.B, k_begin, k_end);
      uint32_t st = 0, tofixph = 0;
      int sb, lo, hi;
      for (uint32_t n = 0; it.next(&sb, &lo, &hi); ++n) {
        const int L = prefix[sb + 1] - prefix[sb];
        const int nr = (hi - lo + kRoundKeys - 1) / kRoundKeys;
        const bool done = for_units(lo, nr, r, [&](const Unit& u, int) -> bool {
          const uint32_t s = st;
          if (++st == kStages) st = 0;
          if (!needs_fix(u, L)) return true;
          if (!warp_wait(&bars->kv_tofix[s], (tofixph >> s) & 1u, wc)) return false;
          tofixph ^= 1u << s;
          // rows [L - key0, 128) of both 64-dim blocks are past the sequence: zero them
          const int r0 = max(L - u.key0, 0);
          uint8_t* base = smem + kRingOff + s * kUnitBytes;
          for (int idx = lane; idx < (RK - r0) * 16; idx += 32) {
            const int row = r0 + (idx >> 4), b = (idx >> 3) & 1, c = idx & 7;
            *reinterpret_cast<uint4*>(base + b * kBlockBytes + row * 128 + c * 16) = make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars->kv_fixed[s]);
          return true;
        });
        if (!done) break;
      }
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax + epilogue
    const int quad = warp & 3;
    const int kh = (warp - 4) >> 2;  // which 64 of the CTA's 128 keys of a round
    const int h = quad * 32 + lane;  // head = TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const Msg* msg = reinterpret_cast<const Msg*>(smem + kMsgOff);
    float* red_mx = reinterpret_cast<float*>(smem + kRedOff);            // [2 rounds][2 halves][NH]
    float* red_l = reinterpret_cast<float*>(smem + kRedOff + 4 * NH * 4);  // [2 halves][NH]
    const uint32_t peer = static_cast<uint32_t>(r ^ 1);
    const uint32_t pp_peer = peer_addr(smem + kPPOff, peer) + kh * kBlockBytes + h * 128;
    const uint32_t msg_peer = peer_addr(smem + kMsgOff, peer);
    const uint32_t ppfull_peer = peer_addr(&bars->pp_full, peer);
    uint8_t* pp_row = smem + kPPOff + kh * kBlockBytes + h * 128;
    const float scl = a.scale_log2;
    PieceIter it;
    it.init(prefix, a.B, k_begin, k_end);
    uint32_t G = 0, pvo_w = 0, pvp_w = 0, hs = 0;  // hs: uses of hsync[quad]
    const bool armer = warp == 4 && lane == 0;  // arms pp_full for each later round's message
    int sb, lo, hi;
    for (uint32_t n = 0; run && it.next(&sb, &lo, &hi); ++n) {
      const int L = prefix[sb + 1] - prefix[sb];
      const int nr = (hi - lo + kRoundKeys - 1) / kRoundKeys;
      if (kh == 0) {
        // query dims [0, 256) of head h -> TMEM columns [kQCol, kQCol + 128) as bf16 pairs (the
        // A-operand layout: row = lane, two consecutive k per 32-bit column); the previous
        // piece's score MMAs must have finished reading them
        if (!warp_wait(&bars->q_empty, (n & 1) ^ 1, wc)) break;
        tc_fence_after();
        const uint4* qrow = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(a.q) +
                                                           (static_cast<long long>(sb) * a.n_h + h) * DQK);
#pragma unroll 1
        for (int c = 0; c < kQTmemDims / 64; ++c) {  // 32 columns = 64 dims per store
          uint32_t rq[32];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const uint4 u = qrow[c * 8 + e];
            rq[4 * e] = u.x;
            rq[4 * e + 1] = u.y;
            rq[4 * e + 2] = u.z;
            rq[4 * e + 3] = u.w;
          }
          tmem_st32(tmem + lane_off + kQCol + c * 32, rq);
        }
        tmem_wait_st();
        if (!warp_wait(&bars->q_full, n & 1, wc)) break;
        if (f.n_pairs) {
          // rotate this head's dims [rope_offset, rope_offset + rope_dims) (all in the shared-memory
          // part) at the new token's position
          uint8_t* row = smem + kQOff + h * 128;
          auto chunk = [&](int c) {
            return reinterpret_cast<uint4*>(row + (c >> 3) * kBlockBytes + (((c & 7) ^ (h & 7)) << 4));
          };
          const int c0 = (a.rope_offset - kQTmemDims) / 8;  // first chunk of the span
          if (f.half) {
            // pair j = span dims (j, j + n_pairs): chunk c0 + i holds first members, chunk c0 + i + n_pairs / 8
            // the second ones (n_pairs % 8 == 0)
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
          fence_proxy_async_smem();
        }
        tc_fence_before();
        mbar_arrive(&bars->q_ready);
      }

      // m_sh: the pair's shared offset for the next round; m_O: the offset O and l are kept at
      float m_sh = -INFINITY, m_O = -INFINITY, l_part = 0.f;
      bool ok = true;
      for (int j = 0; j < nr; ++j, ++G) {
        const int own0 = lo + j * kRoundKeys + r * RK;
        const int n_my = min(max(hi - own0 - 64 * kh, 0), 64);  // valid keys of this thread's 64
        if (!warp_wait(&bars->s_full, G & 1, wc)) { ok = false; break; }
        tc_fence_after();
        uint32_t sr[64];
        tmem_ld32(tmem + lane_off + kSCol + 64 * kh, sr);
        tmem_ld32(tmem + lane_off + kSCol + 64 * kh + 32, sr + 32);
        tmem_wait_ld();
        float s[64];
#pragma unroll
        for (int c = 0; c < 64; ++c) s[c] = (c < n_my) ? __uint_as_float(sr[c]) : -INFINITY;
        // row maximum of this thread's keys: 8 chains of three-input max, then a tree
        float m8[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) m8[i] = fmax3(s[i], s[8 + i], s[16 + i]);
#pragma unroll
        for (int i = 0; i < 8; ++i) m8[i] = fmax3(m8[i], s[24 + i], s[32 + i]);
#pragma unroll
        for (int i = 0; i < 8; ++i) m8[i] = fmax3(m8[i], s[40 + i], s[48 + i]);
#pragma unroll
        for (int i = 0; i < 8; ++i) m8[i] = fmaxf(m8[i], s[56 + i]);
        const float mx_my =
            fmaxf(fmax3(m8[0], m8[1], m8[2]), fmax3(fmax3(m8[3], m8[4], m8[5]), m8[6], m8[7])) * scl;
        // the CTA's row maximum over its 128 keys (the two warps of these heads)
        float* rm = red_mx + (G & 1) * 2 * NH;
        rm[kh * NH + h] = mx_my;
        mbar_arrive(&bars->hsync[quad]);
        if (!warp_wait(&bars->hsync[quad], hs++ & 1, wc)) { ok = false; break; }
        const float mx_cta = fmaxf(rm[h], rm[NH + h]);
        const float m_own = mx_cta > m_sh + kEmergency ? mx_cta : m_sh;
        uint32_t pr[32];
        float rs = 0.f;
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          const float p0 = (2 * c < n_my) ? fast_exp2(fmaf(s[2 * c], scl, -m_own)) : 0.f;
          const float p1 = (2 * c + 1 < n_my) ? fast_exp2(fmaf(s[2 * c + 1], scl, -m_own)) : 0.f;
          rs += p0 + p1;
          pr[c] = pack_bf16x2(p0, p1);
        }
        // P (bf16 pairs) over the first 32 of this thread's 64 score columns
        tmem_st32(tmem + lane_off + kSCol + 64 * kh, pr);
        if (j == 0) {
          m_O = m_own;  // P V(own) of the first round overwrites O
          l_part = 0.f;
        } else {
          const bool resc = m_own > m_O;
          if (__any_sync(0xffffffffu, resc)) {
            // the previous P V(peer) is the last MMA that wrote O: let it finish, then move O to m_own
            if (!warp_wait(&bars->pvp_done, pvp_w & 1, wc)) { ok = false; break; }
            ++pvp_w;
            tc_fence_after();
            const float alpha = resc ? fast_exp2(m_O - m_own) : 1.f;
            scale_o(tmem + lane_off + kOCol + 128 * kh, alpha);
            l_part *= alpha;
            if (resc) m_O = m_own;
          }
        }
        l_part += rs;
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&bars->p_ready);

        // this round's P, offset, maxima and sums -> the peer (its buffer is free once its
        // previous P V(peer) has completed)
        if (!warp_wait_cluster(&bars->pp_empty, (G & 1) ^ 1, wc)) { ok = false; break; }
#pragma unroll
        for (int i = 0; i < 8; ++i)
          st_peer_v4(pp_peer + ((i ^ (h & 7)) << 4), pr[4 * i], pr[4 * i + 1], pr[4 * i + 2], pr[4 * i + 3],
                     ppfull_peer);
        if (kh == 0) {
          st_peer_f32(msg_peer + h * 4, m_own, ppfull_peer);
          st_peer_f32(msg_peer + (NH + h) * 4, mx_cta, ppfull_peer);
        }
        st_peer_f32(msg_peer + ((2 + kh) * NH + h) * 4, rs, ppfull_peer);

        // the peer's round: bring O, l and the peer's P to one offset
        if (!warp_wait_cluster(&bars->pp_full, G & 1, wc)) { ok = false; break; }
        const float m_p = msg->m_own[h], mx_p = msg->mx[h], rs_p = msg->rs[kh][h];
        // the next message may land only after this CTA's P V(peer) of this round has completed,
        // which follows every thread's pp_ready below: arming the next phase here precedes it
        if (armer) mbar_arrive_expect_tx(&bars->pp_full, kMsgBytes);
        if (!warp_wait(&bars->pvo_done, pvo_w & 1, wc)) { ok = false; break; }
        ++pvo_w;
        if (pvp_w < G) {
          if (!warp_wait(&bars->pvp_done, pvp_w & 1, wc)) { ok = false; break; }
          ++pvp_w;
        }
        tc_fence_after();
        const bool up = m_p > m_O;
        if (__any_sync(0xffffffffu, up)) {
          const float alpha = up ? fast_exp2(m_O - m_p) : 1.f;  // 0 when this CTA has no key yet (m_O = -inf)
          scale_o(tmem + lane_off + kOCol + 128 * kh, alpha);
          l_part *= alpha;
          if (up) m_O = m_p;
        }
        float fp = 1.f;
        if (m_p < m_O) {
          fp = m_p == -INFINITY ? 0.f : fast_exp2(m_p - m_O);
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            uint4* c = reinterpret_cast<uint4*>(pp_row + (i << 4));
            float x[8];
            bf16x8_to_f32(*c, x);
#pragma unroll
            for (int e = 0; e < 8; ++e) x[e] *= fp;
            *c = f32_to_bf16x8(x);
          }
          fence_proxy_async_smem();
        }
        l_part += rs_p * fp;
        const float mx_all = fmaxf(mx_cta, mx_p);
        m_sh = mx_all > m_O + kRaise ? mx_all : m_O;
        tc_fence_before();
        mbar_arrive(&bars->pp_ready);
      }
      if (!__all_sync(0xffffffffu, ok)) break;
      // epilogue: this piece's normalised partial for head h, value dims of this thread
      if (!warp_wait(&bars->pvp_done, pvp_w & 1, wc)) break;
      ++pvp_w;
      tc_fence_after();
      red_l[kh * NH + h] = l_part;
      mbar_arrive(&bars->hsync[quad]);
      if (!warp_wait(&bars->hsync[quad], hs++ & 1, wc)) break;
      const float l_tot = red_l[h] + red_l[NH + h];
      const long long slot = static_cast<long long>(p) + sb;  // unique per (pair, sequence)
      float* dst = a.ws_o + (slot * a.n_h + h) * DV + r * DVH + kh * 128;
      const float inv_l = 1.f / l_tot;
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t orow[32];
        tmem_ld32(tmem + lane_off + kOCol + 128 * kh + c * 32, orow);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 8; ++e)
          reinterpret_cast<float4*>(dst + c * 32)[e] =
              make_float4(__uint_as_float(orow[4 * e]) * inv_l, __uint_as_float(orow[4 * e + 1]) * inv_l,
                          __uint_as_float(orow[4 * e + 2]) * inv_l, __uint_as_float(orow[4 * e + 3]) * inv_l);
      }
      if (r == 0 && kh == 0) a.ws_lse[slot * a.n_h + h] = m_O + log2f(l_tot);
      tc_fence_before();
      mbar_arrive(&bars->o_empty);
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();  // no CTA leaves while the other may still write its shared memory
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
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
  const long long x0 = before, T = total;
  const long long x1 = x0 + min(max(a.seqlens[b], 1), a.max_len) - 1;  // last key of sequence b
  // pair holding key x: the largest p with floor(p T / P) <= x
  const int p_lo = static_cast<int>(((x0 + 1) * P - 1) / T);
  const int p_hi = static_cast<int>(((x1 + 1) * P - 1) / T);
  const int np = p_hi - p_lo + 1;
  auto piece_lse = [&](int j) {  // -inf for a pair whose key range is empty (it wrote nothing)
    if (pair_start(p_lo + j + 1, T, P) <= pair_start(p_lo + j, T, P)) return -INFINITY;
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
  // the rotated span lies in the shared-memory part of the query, in whole 8-dim chunks
  return rope_offset >= kQTmemDims && rope_offset % 8 == 0 && rope_dims % (half ? 16 : 8) == 0;
}

namespace {
std::atomic<unsigned> g_mla_ready{0};  // one bit per device whose shared-memory opt-in is done
std::atomic<int> g_mla_pairs[32];      // per device: clusters of two CTAs that fit at once (0: not known)

cudaError_t mla_prepare(int dev) {
  const unsigned bit = 1u << (dev & 31);
  if (g_mla_ready.load(std::memory_order_acquire) & bit) return cudaSuccess;
  const cudaError_t e =
      cudaFuncSetAttribute(mla_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
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

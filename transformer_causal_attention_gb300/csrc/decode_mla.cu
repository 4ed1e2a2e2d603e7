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
// an SM, leaving no room for the scores, so CTAs work in pairs: both CTAs of a
// pair walk the same keys, each computes the full score tile S = Q C^T (M = 128
// heads, N = 64 keys, K = 576) and its own softmax, and each accumulates half of
// the value dims (O_half += P V_half, M = 128, N = 256, K = 64).  The pair
// reads every cache row from L2 twice but from HBM once.  A tcgen05.mma costs
// the same time at N = 64 as at N = 128 (and at N = 32), so the key tile is as
// wide as TMEM allows: two 64-column S/P buffers, O_half (256 columns) and the
// query's first 256 dims (128 columns of bf16 pairs, the MMA's A operand,
// written by the softmax warps) fill the 512 columns; the query's other 320
// dims sit in shared memory (80 KB) beside a 2-stage ring of 64-key cache tiles
// (72 KB each), loaded by TMA with 128-byte swizzle.  (32-key tiles with a
// 4-stage ring ran 1.55x slower.)  The batch's key prefix sums live in shared
// memory too, which caps this kernel at 256 sequences per call.
// Keys of all sequences, laid end to end, are split evenly over the pairs
// (a pair's range may cross sequence boundaries), so every pair does the same
// work; each (pair, sequence) piece writes one normalised partial, merged per
// sequence by mla_combine_kernel with the log-sum-exp rule of the online
// softmax ("Transformer架构完全深度解析" §13).
// Roles (256 threads): warp 0 TMA producer, warp 1 TMEM owner + single-thread
// MMA issuer, warp 2 computes the key prefix sums, warps 4-7 softmax (one
// thread per head = TMEM lane) and epilogue.
#include <math.h>

#include "kernels.h"

namespace attn {
namespace {

constexpr int NH = 128;          // query heads (MMA M)
constexpr int DQK = 576;         // latent + rotary dims
constexpr int DV = 512;          // value dims
constexpr int DVH = 256;         // value dims per CTA of a pair
constexpr int BK = kMlaTileKeys;  // keys per tile (MMA N of the score tile)
constexpr int kStages = BK == 32 ? 4 : (BK == 48 ? 3 : 2);
constexpr int kThreads = 256;
constexpr int kBlocks = DQK / 64;                  // 9 column blocks of 64 dims
constexpr int kQTmemDims = kMlaQTmemDims;          // query dims [0, kQTmemDims) live in TMEM (A operand)
constexpr int kQSmemBlocks = (DQK - kQTmemDims) / 64;  // dims [384, 576) in shared memory: 3 blocks
constexpr int kQBlockBytes = NH * 128;             // 16 KB
constexpr int kQSmemBytes = kQSmemBlocks * kQBlockBytes;  // 48 KB
constexpr int kKBlockBytes = BK * 128;             // 4 KB
constexpr int kTileBytes = kBlocks * kKBlockBytes; // 36 KB
constexpr int kMaxB = BK == 32 ? 1024 : (BK == 48 ? 128 : 256);  // the batch's key prefix sums live in smem
constexpr int kQOff = 0;
constexpr int kKOff = kQOff + kQSmemBytes;
constexpr int kPrefOff = kKOff + kStages * kTileBytes;
constexpr int kBarOff = kPrefOff + (kMaxB + 1) * 4 + 60;
constexpr int kUsedBytes = kBarOff + 160;
// The dynamic shared memory is declared 1024-byte aligned; the slack for aligning it
// by hand is kept wherever it fits (the kernel checks the alignment at run time).
constexpr int kSmemBytes = kUsedBytes + 1024 <= 227 * 1024 ? kUsedBytes + 1024 : kUsedBytes;
static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");
// TMEM columns: S/P buffer b at [BK b, BK b + BK), O_half at [2 BK, 2 BK + 256), then the query dims
// [0, kQTmemDims) as bf16 pairs
__device__ __forceinline__ uint32_t s_col(uint32_t b) { return b * BK; }
constexpr uint32_t kOCol = 2 * BK;
constexpr uint32_t kQCol = kOCol + DVH;
static_assert(kQCol + kQTmemDims / 2 <= 512, "TMEM columns");
constexpr uint32_t kIdescQK = idesc_bf16_f32(NH, BK, false);
constexpr uint32_t kIdescPV = idesc_bf16_f32(NH, DVH, true);
constexpr float kRescaleThreshold = 8.0f;
#ifndef ATTN_MLA_PREFETCH_TILES
#define ATTN_MLA_PREFETCH_TILES 4
#endif
constexpr int kPrefetchTiles = ATTN_MLA_PREFETCH_TILES;  // tiles requested into L2 ahead of the smem loads

struct Bars {
  uint64_t q_full, q_ready, q_empty;
  uint64_t kv_full[kStages], kv_empty[kStages];
  uint64_t s_full[2], p_full[2];
  uint64_t pv_done, o_empty, fin;
  uint32_t tmem_base;
  int abort_flag;
};

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

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t* r) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
               "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
               : "memory");
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

__global__ void __launch_bounds__(kThreads, 1)
    mla_decode_kernel(const __grid_constant__ DecodeArgs a, const __grid_constant__ RopeFreq f,
                      const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_c) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  if (static_cast<int>(smem - smem_raw) + kUsedBytes > kSmemBytes) {  // not enough slack: report, touch nothing
    if (threadIdx.x == 0) atomicOr(a.status, STATUS_LAYOUT);
    return;
  }
  Bars* bars = reinterpret_cast<Bars*>(smem + kBarOff);
  int* prefix = reinterpret_cast<int*>(smem + kPrefOff);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int P = gridDim.x >> 1;       // pairs
  const int p = blockIdx.x >> 1;      // this CTA's pair
  const int half = blockIdx.x & 1;    // value dims [half*256, half*256 + 256)

  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
    mbar_init(&bars->q_ready, 128);
    mbar_init(&bars->q_empty, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bars->kv_full[s], 1);
      mbar_init(&bars->kv_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars->s_full[s], 1);
      mbar_init(&bars->p_full[s], 128);
    }
    mbar_init(&bars->pv_done, 1);
    mbar_init(&bars->o_empty, 128);
    mbar_init(&bars->fin, 1);
    bars->abort_flag = 0;
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
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  const WaitCtl wc{&bars->abort_flag, a.status, a.wait_limit_ns};
  const long long T = prefix[a.B];
  const long long k_begin = pair_start(p, T, P), k_end = pair_start(p + 1, T, P);

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_c);
      PieceIter it;
      it.init(prefix, a.B, k_begin, k_end);
      uint32_t st = 0, ph = 0, issued = 0, last_ph = 0, q_issued = 0;
      int sb, lo, hi;
      for (uint32_t n = 0; it.next(&sb, &lo, &hi); ++n) {
        if (!mbar_wait(&bars->q_empty, (n & 1) ^ 1, wc)) goto producer_done;
        mbar_arrive_expect_tx(&bars->q_full, kQSmemBytes);
        for (int blk = 0; blk < kQSmemBlocks; ++blk)
          tma_load_3d(smem + kQOff + blk * kQBlockBytes, &tm_q, &bars->q_full, kQTmemDims + blk * 64, 0, sb);
        q_issued = n + 1;
        // the 2-stage shared-memory ring is too shallow to cover HBM latency on its
        // own: keep kPrefetchTiles tiles ahead of the loads on their way into L2
        if (half == 0)  // the other CTA of the pair reads the same tiles
          for (int k0 = lo; k0 < hi && k0 < lo + kPrefetchTiles * BK; k0 += BK)
            for (int blk = 0; blk < kBlocks; ++blk) tma_prefetch_l2_3d(&tm_c, blk * 64, k0, sb);
        for (int k0 = lo; k0 < hi; k0 += BK) {
          const int kp = k0 + kPrefetchTiles * BK;
          if (half == 0 && kp < hi)
            for (int blk = 0; blk < kBlocks; ++blk) tma_prefetch_l2_3d(&tm_c, blk * 64, kp, sb);
          if (!mbar_wait(&bars->kv_empty[st], ph ^ 1, wc)) goto producer_done;
          mbar_arrive_expect_tx(&bars->kv_full[st], kTileBytes);
          uint8_t* dst = smem + kKOff + st * kTileBytes;
          for (int blk = 0; blk < kBlocks; ++blk)
            tma_load_3d(dst + blk * kKBlockBytes, &tm_c, &bars->kv_full[st], blk * 64, k0, sb);
          issued |= 1u << st;
          last_ph = (last_ph & ~(1u << st)) | (ph << st);
          if (++st == kStages) { st = 0; ph ^= 1; }
        }
      }
    producer_done:
      if (bars->abort_flag) {
        for (int s = 0; s < kStages; ++s)
          if (issued & (1u << s)) drain_wait(&bars->kv_full[s], (last_ph >> s) & 1, a.wait_limit_ns);
        if (q_issued) drain_wait(&bars->q_full, (q_issued - 1) & 1, a.wait_limit_ns);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      PieceIter it;
      it.init(prefix, a.B, k_begin, k_end);
      const uint32_t q_addr = smem_u32(smem + kQOff);
      uint32_t st = 0, ph = 0, pph = 0u;  // bit b: phase of p_full[b] (bit masks keep it in registers)
      int sb, lo, hi;
      uint32_t tile = 0;  // tiles issued so far (all pieces)
      auto issue_qk = [&](uint32_t stage, uint32_t sbuf) {
        const uint32_t kaddr = smem_u32(smem + kKOff + stage * kTileBytes);
#pragma unroll 4
        for (int kk = 0; kk < kQTmemDims / 16; ++kk) {  // A = query dims [16 kk, 16 kk + 16) from TMEM
          const uint32_t ko = (kk >> 2) * kKBlockBytes + (kk & 3) * 32;
          mma_ts(tmem + s_col(sbuf), tmem + kQCol + kk * 8, sdesc_sw128(kaddr + ko, 16, 1024), kIdescQK,
                 kk > 0 ? 1u : 0u);
        }
#pragma unroll
        for (int kk = kQTmemDims / 16; kk < DQK / 16; ++kk) {  // A from shared memory
          const int kq = kk - kQTmemDims / 16;
          const uint32_t qo = (kq >> 2) * kQBlockBytes + (kq & 3) * 32;
          const uint32_t ko = (kk >> 2) * kKBlockBytes + (kk & 3) * 32;
          mma_ss(tmem + s_col(sbuf), sdesc_sw128(q_addr + qo, 16, 1024), sdesc_sw128(kaddr + ko, 16, 1024),
                 kIdescQK, 1u);
        }
      };
      auto issue_pv = [&](uint32_t stage, uint32_t sbuf, bool accumulate) {
        const uint32_t vaddr = smem_u32(smem + kKOff + stage * kTileBytes + half * 4 * kKBlockBytes);
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk)
          mma_ts(tmem + kOCol, tmem + s_col(sbuf) + kk * 8, sdesc_sw128(vaddr + kk * 16 * 128, kKBlockBytes, 1024),
                 kIdescPV, (accumulate || kk > 0) ? 1u : 0u);
      };
      for (uint32_t n = 0; it.next(&sb, &lo, &hi); ++n) {
        const int nt = (hi - lo + BK - 1) / BK;
        if (!mbar_wait(&bars->q_ready, n & 1, wc)) goto mma_done;
        // Tile j's stage is released by the commit after its P V, so P V(j) must
        // not wait behind the next tile's load: QK(j+1) goes first only when that
        // tile is already resident, otherwise P V(j) is issued first.
        uint32_t cur_stage = st, cur_sbuf = tile & 1;
        if (!mbar_wait(&bars->kv_full[st], ph, wc)) goto mma_done;
        tc_fence_after();
        issue_qk(st, cur_sbuf);
        mma_commit(&bars->s_full[cur_sbuf]);
        if (nt == 1) mma_commit(&bars->q_empty);
        ++tile;
        if (++st == kStages) { st = 0; ph ^= 1; }
        for (int j = 0; j < nt; ++j) {
          bool next_issued = false;
          const uint32_t nstage = st, nsbuf = tile & 1;
          if (j + 1 < nt && mbar_try_wait(&bars->kv_full[st], ph)) {
            tc_fence_after();
            issue_qk(st, nsbuf);
            mma_commit(&bars->s_full[nsbuf]);
            if (j + 1 == nt - 1) mma_commit(&bars->q_empty);  // every MMA reading this query is issued
            next_issued = true;
          }
          if (!mbar_wait(&bars->p_full[cur_sbuf], (pph >> cur_sbuf) & 1u, wc)) goto mma_done;
          pph ^= 1u << cur_sbuf;
          if (j == 0 && !mbar_wait(&bars->o_empty, (n & 1) ^ 1, wc)) goto mma_done;
          tc_fence_after();
          issue_pv(cur_stage, cur_sbuf, j > 0);
          mma_commit(&bars->pv_done);
          mma_commit(&bars->kv_empty[cur_stage]);
          if (j + 1 < nt) {
            if (!next_issued) {
              if (!mbar_wait(&bars->kv_full[st], ph, wc)) goto mma_done;
              tc_fence_after();
              issue_qk(st, nsbuf);
              mma_commit(&bars->s_full[nsbuf]);
              if (j + 1 == nt - 1) mma_commit(&bars->q_empty);
            }
            cur_stage = nstage;
            cur_sbuf = nsbuf;
            ++tile;
            if (++st == kStages) { st = 0; ph ^= 1; }
          }
        }
      }
    mma_done:
      mma_commit(&bars->fin);
      drain_wait(&bars->fin, 0, a.wait_limit_ns);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax + epilogue
    const int quad = warp & 3;
    const int h = quad * 32 + lane;  // head = TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    PieceIter it;
    it.init(prefix, a.B, k_begin, k_end);
    uint32_t sph = 0u, pvph = 0, st = 0, tile = 0;  // sph bit b: phase of s_full[b]
    int sb, lo, hi;
    for (uint32_t n = 0; it.next(&sb, &lo, &hi); ++n) {
      const int nt = (hi - lo + BK - 1) / BK;
      const int L = prefix[sb + 1] - prefix[sb];
      // query dims [0, 384) of head h -> TMEM columns [kQCol, kQCol + 192) as bf16 pairs (the
      // A-operand layout: row = lane, two consecutive k per 32-bit column); the previous
      // piece's QK MMAs must have finished reading them
      if (!warp_wait(&bars->q_empty, (n & 1) ^ 1, wc)) break;
      tc_fence_after();
      {
        const uint4* qrow = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(a.q) +
                                                           (static_cast<long long>(sb) * a.n_h + h) * DQK);
#pragma unroll 1
        for (int c = 0; c < kQTmemDims / 64; ++c) {  // 32 columns = 64 dims per store
          uint32_t r[32];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const uint4 u = qrow[c * 8 + e];
            r[4 * e] = u.x;
            r[4 * e + 1] = u.y;
            r[4 * e + 2] = u.z;
            r[4 * e + 3] = u.w;
          }
          tmem_st32(tmem + lane_off + kQCol + c * 32, r);
        }
        tmem_wait_st();
      }
      if (!warp_wait(&bars->q_full, n & 1, wc)) break;
      if (f.n_pairs) {
        // rotate this head's dims [rope_offset, rope_offset + rope_dims) (all in the shared-memory
        // part) at the new token's position
        uint8_t* row = smem + kQOff + h * 128;
        auto chunk = [&](int c) {
          return reinterpret_cast<uint4*>(row + (c >> 3) * kQBlockBytes + (((c & 7) ^ (h & 7)) << 4));
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

      float m_run = -INFINITY, l_run = 0.f;
      bool ok = true;
      for (int j = 0; j < nt; ++j) {
        const uint32_t sbuf = tile & 1;
        if (!warp_wait(&bars->s_full[sbuf], (sph >> sbuf) & 1u, wc)) { ok = false; break; }
        sph ^= 1u << sbuf;
        tc_fence_after();
        uint32_t sr[BK];
#pragma unroll
        for (int c = 0; c < BK / 32; ++c) tmem_ld32(tmem + lane_off + s_col(sbuf) + c * 32, sr + c * 32);
        if constexpr (BK % 32 == 16) tmem_ld16(tmem + lane_off + s_col(sbuf) + BK - 16, sr + BK - 16);
        tmem_wait_ld();
        const int k0 = lo + j * BK;
        const int n_valid = min(BK, hi - k0);
        float s[BK];
#pragma unroll
        for (int c = 0; c < BK; ++c) s[c] = (c < n_valid) ? __uint_as_float(sr[c]) : -INFINITY;
        // row maximum: 8 chains of three-input max, then a tree
        float m8[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) m8[i] = s[i];
#pragma unroll
        for (int c = 8; c + 16 <= BK; c += 16)
#pragma unroll
          for (int i = 0; i < 8; ++i) m8[i] = fmax3(m8[i], s[c + i], s[c + 8 + i]);
        if ((BK - 8) % 16 == 8) {
#pragma unroll
          for (int i = 0; i < 8; ++i) m8[i] = fmaxf(m8[i], s[BK - 8 + i]);
        }
        float mx = fmaxf(fmax3(m8[0], m8[1], m8[2]), fmax3(fmax3(m8[3], m8[4], m8[5]), m8[6], m8[7]));
        mx *= a.scale_log2;
        const bool need = mx > m_run + kRescaleThreshold;
        float alpha = 1.f;
        if (need) {
          if (j > 0) alpha = fast_exp2(m_run - mx);
          l_run *= alpha;
          m_run = mx;
        }
        uint32_t pr[BK / 2];
        float rs = 0.f;
#pragma unroll
        for (int c = 0; c < BK / 2; ++c) {
          const float p0 = fast_exp2(fmaf(s[2 * c], a.scale_log2, -m_run));
          const float p1 = fast_exp2(fmaf(s[2 * c + 1], a.scale_log2, -m_run));
          rs += p0 + p1;
          pr[c] = pack_bf16x2(p0, p1);
        }
        l_run += rs;
        // P as bf16 pairs: BK / 2 columns
#pragma unroll
        for (int c = 0; c < BK / 64; ++c) tmem_st32(tmem + lane_off + s_col(sbuf) + c * 32, pr + c * 32);
        if constexpr ((BK / 2) % 32 == 16) tmem_st16(tmem + lane_off + s_col(sbuf) + BK / 2 - 16, pr + BK / 2 - 16);
        if constexpr ((BK / 2) % 32 == 24) {
          tmem_st16(tmem + lane_off + s_col(sbuf) + (BK / 64) * 32, pr + (BK / 64) * 32);
          tmem_st8(tmem + lane_off + s_col(sbuf) + (BK / 64) * 32 + 16, pr + (BK / 64) * 32 + 16);
        }
        if (n_valid < BK) {
          // rows past the sequence may hold anything: clear their value dims so that P V stays finite
          uint8_t* tile_smem = smem + kKOff + st * kTileBytes;
          const int rows = BK - n_valid;
          for (int idx = threadIdx.x - 128; idx < rows * 8 * (DV / 64); idx += 128) {
            const int r = n_valid + idx / (8 * (DV / 64));
            const int rem = idx % (8 * (DV / 64));
            const int blk = rem / 8, chunk = rem % 8;
            *reinterpret_cast<uint4*>(tile_smem + blk * kKBlockBytes + r * 128 + (chunk << 4)) =
                make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async_smem();
        }
        tmem_wait_st();
        if (j > 0) {
          // the previous P V has completed: O may be rescaled
          if (!warp_wait(&bars->pv_done, pvph, wc)) { ok = false; break; }
          pvph ^= 1;
          tc_fence_after();
          if (__any_sync(0xffffffffu, need)) {
#pragma unroll 1
            for (int c = 0; c < DVH / 32; ++c) {
              uint32_t orow[32];
              tmem_ld32(tmem + lane_off + kOCol + c * 32, orow);
              tmem_wait_ld();
#pragma unroll
              for (int e = 0; e < 32; ++e) orow[e] = __float_as_uint(__uint_as_float(orow[e]) * alpha);
              tmem_st32(tmem + lane_off + kOCol + c * 32, orow);
            }
            tmem_wait_st();
          }
        }
        tc_fence_before();
        mbar_arrive(&bars->p_full[sbuf]);
        ++tile;
        if (++st == kStages) st = 0;
      }
      if (!__all_sync(0xffffffffu, ok)) break;
      // epilogue: this piece's normalised partial for head h
      if (!warp_wait(&bars->pv_done, pvph, wc)) break;
      pvph ^= 1;
      tc_fence_after();
      const long long slot = static_cast<long long>(p) + sb;  // unique per (pair, sequence)
      float* dst = a.ws_o + (slot * a.n_h + h) * DV + half * DVH;
      const float inv_l = 1.f / l_run;
#pragma unroll 1
      for (int c = 0; c < DVH / 32; ++c) {
        uint32_t orow[32];
        tmem_ld32(tmem + lane_off + kOCol + c * 32, orow);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 8; ++e)
          reinterpret_cast<float4*>(dst + c * 32)[e] =
              make_float4(__uint_as_float(orow[4 * e]) * inv_l, __uint_as_float(orow[4 * e + 1]) * inv_l,
                          __uint_as_float(orow[4 * e + 2]) * inv_l, __uint_as_float(orow[4 * e + 3]) * inv_l);
      }
      if (half == 0) a.ws_lse[slot * a.n_h + h] = m_run + log2f(l_run);
      tc_fence_before();
      mbar_arrive(&bars->o_empty);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// out[b, h, :] = sum over the pieces of sequence b of 2^(lse_j - lse) O_j.
__global__ void __launch_bounds__(128) mla_combine_kernel(DecodeArgs a) {
  __shared__ float w_s[256];
  __shared__ float stat[2];
  __shared__ long long pre[2];
  const int b = blockIdx.x / a.n_h, h = blockIdx.x % a.n_h;
  const int P = a.n_split;  // pairs
  if (threadIdx.x < 32) {
    long long before = 0, total = 0;
    for (int i = threadIdx.x; i < a.B; i += 32) {
      const long long L = min(max(a.seqlens[i], 1), a.max_len);
      total += L;
      if (i < b) before += L;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      before += __shfl_xor_sync(0xffffffffu, before, o);
      total += __shfl_xor_sync(0xffffffffu, total, o);
    }
    if (threadIdx.x == 0) {
      pre[0] = before;
      pre[1] = total;
    }
  }
  __syncthreads();
  const long long x0 = pre[0], T = pre[1];
  const long long x1 = x0 + min(max(a.seqlens[b], 1), a.max_len) - 1;  // last key of sequence b
  // pair holding key x: the largest p with floor(p T / P) <= x
  const int p_lo = static_cast<int>(((x0 + 1) * P - 1) / T);
  const int p_hi = static_cast<int>(((x1 + 1) * P - 1) / T);
  const int np = p_hi - p_lo + 1;
  if (threadIdx.x < 32) {
    // a pair whose key range is empty (fewer keys than pairs) wrote nothing
    float M = -INFINITY;
    for (int j = threadIdx.x; j < np; j += 32)
      if (pair_start(p_lo + j + 1, T, P) > pair_start(p_lo + j, T, P))
        M = fmaxf(M, a.ws_lse[(static_cast<long long>(p_lo + j) + b) * a.n_h + h]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float den = 0.f;
    for (int j = threadIdx.x; j < np; j += 32) {
      float wgt = 0.f;
      if (pair_start(p_lo + j + 1, T, P) > pair_start(p_lo + j, T, P))
        wgt = exp2f(a.ws_lse[(static_cast<long long>(p_lo + j) + b) * a.n_h + h] - M);
      w_s[j] = wgt;
      den += wgt;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
    if (threadIdx.x == 0) {
      stat[0] = M;
      stat[1] = den;
    }
  }
  __syncthreads();
  const float inv = 1.f / stat[1];
  __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out) + (static_cast<long long>(b) * a.n_h + h) * DV;
  for (int d = threadIdx.x; d < DV; d += blockDim.x) {
    float acc = 0.f;
    for (int j = 0; j < np; ++j)
      if (w_s[j] != 0.f) acc = fmaf(w_s[j], a.ws_o[((static_cast<long long>(p_lo + j) + b) * a.n_h + h) * DV + d], acc);
    out[d] = __float2bfloat16_rn(acc * inv);
  }
  if (a.lse != nullptr && threadIdx.x == 0)
    a.lse[static_cast<long long>(b) * a.n_h + h] = (stat[0] + log2f(stat[1])) * 0.69314718055994530942f;
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

int decode_mla_pairs(int num_sms) {
  const int p = num_sms / 2;
  return p < 1 ? 1 : (p > kMlaMaxPairs ? kMlaMaxPairs : p);
}

cudaError_t launch_decode_mla(const DecodeArgs& a, const RopeFreq& rope, const CUtensorMap* maps, cudaStream_t st,
                              int* launches) {
  cudaError_t e = cudaFuncSetAttribute(mla_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  mla_decode_kernel<<<2 * a.n_split, kThreads, kSmemBytes, st>>>(a, rope, maps[0], maps[1]);
  *launches += 1;
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  mla_combine_kernel<<<a.B * a.n_h, 128, 0, st>>>(a);
  *launches += 1;
  return cudaGetLastError();
}

}  // namespace attn

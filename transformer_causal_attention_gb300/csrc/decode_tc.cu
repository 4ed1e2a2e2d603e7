// decode_tc.cu - GQA decode on the tensor cores (bf16, D_qk = D_v = 128,
// up to 16 query heads per KV head).
//
// Decode reads each cached key/value row once ("Transformer架构完全深度解析"
// §9) and does ~2 FLOP per byte, so the goal is HBM speed with as few
// instructions per byte as possible.  The scores of a KV head's query group
// are a tall, thin product - 128 keys x G heads - which the tensor core takes
// with the keys on its M dimension and the heads on N (padded to 16):
//   S^T [keys x heads] = K_tile [keys x d] . Q_g^T [d x heads]      (A = K tile, B = Q_g)
//   O^T [d x heads]   += V_tile^T [d x keys] . P^T [keys x heads]   (A = V tile read MN-major, B = P^T)
// Both operands come straight from the TMA-loaded tiles; only the tiny Q_g
// (2 KB per 64 dims) and P^T (4 KB) tiles are written by threads.  S^T and O^T
// live in TMEM (16 columns each), one TMEM lane per key / per value dim.
//
// The softmax runs over the keys, i.e. across TMEM lanes: each of the 128
// softmax threads owns one key of the tile (and, for O, one value dim).  Per
// tile the block maximum of every head is reduced across the four warps
// through shared memory (online softmax, "Transformer架构完全深度解析" §13,
// with the lazy rescale of the prefill kernel: the reference maximum moves
// only when the row maximum grows by more than 2^8).  The running sums stay
// per thread and are reduced once per work unit.
//
// Roles (256 threads, one persistent CTA per SM): warp 0 TMA producer (K and
// V tiles of 128 keys, two 64-row boxes per 64-dim block, through a 3-stage
// ring of 64 KB; L2 prefetches ahead of the loads measured slower at this
// rate), warp 1 TMEM owner and single-thread MMA issuer, warps 4-7 softmax and
// epilogue.  Work units are (sequence, chunk of keys, KV head) with the KV head
// fastest, as in the CUDA-core streaming kernel; the producer claims them from
// a global counter (sequence lengths differ, so a static split left the
// busiest SM 9% above the mean), longest (sequence, chunk) first, and hands each
// to the consumers through a small shared-memory queue.  Each unit writes one normalised partial per
// head, merged by the combine kernel of decode.cu.  With a sliding window a
// unit keeps only its chunk's keys inside the window or among the sinks (one
// or two key ranges, each tiled from its first key), and chunks with none of
// them are never claimed, so the kernel reads only visible rows (plus the
// rest of the sinks' one tile).
#include <math.h>

#include "kernels.h"

namespace attn {
namespace {

constexpr int D = 128;
constexpr int BK = 128;                       // keys per tile (MMA M)
constexpr int NHP = 16;                       // heads per unit, padded (MMA N)
constexpr int kBox = kStreamTileKeys;         // TMA box rows of the K/V maps
static_assert(BK % kBox == 0, "whole boxes per tile");
constexpr int kStages = 3;
constexpr int kThreads = 256;
constexpr int kBlockBytes = BK * 128;         // one 64-dim column block of a K or V tile (16 KB)
constexpr int kTileBytes = 2 * kBlockBytes;   // one K or V tile (32 KB)
constexpr int kStageBytes = 2 * kTileBytes;   // K + V
constexpr int kQBlockBytes = NHP * 128;       // one 64-dim block of Q_g (2 KB)
constexpr int kPBlockBytes = NHP * 128;       // one 64-key block of P^T (2 KB)
constexpr int kKVOff = 0;
constexpr int kQOff = kKVOff + kStages * kStageBytes;
constexpr int kPOff = kQOff + 2 * kQBlockBytes;           // two P^T buffers of 2 blocks
constexpr int kRedOff = kPOff + 2 * 2 * kPBlockBytes;     // [2][4 warps][NHP] block maxima + [4][NHP] sums
constexpr int kBarOff = kRedOff + (2 * 4 * NHP + 4 * NHP) * 4;
// Claim order: up to kMaxOrder (sequence, chunk) pairs are ranked longest first (below)
constexpr int kMaxOrder = 256;
constexpr int kOrdOff = kBarOff + 256;                    // [kMaxOrder] pair at each rank, then [kMaxOrder] tiles
constexpr int kSmemBytes = kOrdOff + 2 * kMaxOrder * 2 + 1024;
static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");
// TMEM columns: S^T buffer b at [16 b, 16 b + 16), O^T at [32, 48)
constexpr uint32_t kOCol = 2 * NHP;
constexpr uint32_t kTmemCols = 64;
constexpr uint32_t kIdescQK = idesc_bf16_f32(BK, NHP, false);                  // A, B K-major
constexpr uint32_t kIdescPV = idesc_bf16_f32(D, NHP, false) | (1u << 15);     // A (V^T) MN-major
constexpr float kRescaleThreshold = 8.0f;  // log2 units
constexpr int kUnitSlots = 4;               // work units handed from the producer to the consumers

struct Bars {
  uint64_t full[kStages], empty[kStages];
  uint64_t q_ready, q_empty;
  uint64_t s_full[2], p_full[2];
  uint64_t pv_done, o_empty, fin;
  uint64_t red;  // softmax-thread barrier (128 arrivals per phase)
  uint64_t unit_full[kUnitSlots], unit_empty[kUnitSlots];
  int unit_q[kUnitSlots];  // claimed unit index, -1: no more work
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(Bars) <= 256, "barrier block");

// A work unit: the visible keys of one chunk of one sequence for one KV head,
// as one or two key ranges [lo, hi) (two when a chunk holds both the sinks and
// the start of a sliding window).  Tiles of BK keys start at each range's first
// key; keys of a tile past its range's end are masked.
struct Unit {
  int b, g, split, L;
  int lo0, hi0, lo1, hi1;  // the key ranges (the second one empty unless nt > nt0)
  int nt0, nt;             // tiles of the first range, of both
};

// Units enumerate (b, chunk, g) with the KV head fastest.  Chunks past the
// sequence, or with no key inside the window or the sinks, are empty.  (Scalar
// fields, not arrays: a runtime-indexed array would live in local memory.)
__device__ __forceinline__ bool unit_at(int u, const DecodeArgs& a, Unit& w) {
  w.g = u % a.n_kv;
  const int r = u / a.n_kv;
  w.split = r % a.n_split;
  w.b = r / a.n_split;
  w.L = min(max(a.seqlens[w.b], 1), a.max_len);
  const int start = w.split * a.chunk, end = min(w.L, start + a.chunk);
  int n = 0;
  w.lo0 = w.hi0 = w.lo1 = w.hi1 = 0;
  auto add = [&](int vlo, int vhi) {  // keep [vlo, vhi) within the chunk
    const int lo = max(start, vlo), hi = min(end, vhi);
    if (lo >= hi) return;
    if (n == 0) {
      w.lo0 = lo;
      w.hi0 = hi;
    } else {
      w.lo1 = lo;
      w.hi1 = hi;
    }
    ++n;
  };
  // the visible keys of the new token at position L - 1 (decode_visible in kernels.h)
  if (a.window <= 0 || w.L - a.window <= a.n_sink) {
    add(0, w.L);
  } else {
    if (a.n_sink > 0) add(0, a.n_sink);
    add(w.L - a.window, w.L);
  }
  if (n == 0) return false;
  w.nt0 = (w.hi0 - w.lo0 + BK - 1) / BK;
  w.nt = w.nt0 + (n == 2 ? (w.hi1 - w.lo1 + BK - 1) / BK : 0);
  return true;
}

// First key of tile t of a unit, and the end of the range it belongs to.
__device__ __forceinline__ int tile_key0(const Unit& w, int t) {
  return t < w.nt0 ? w.lo0 + t * BK : w.lo1 + (t - w.nt0) * BK;
}
__device__ __forceinline__ int tile_kend(const Unit& w, int t) { return t < w.nt0 ? w.hi0 : w.hi1; }

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, const WaitCtl& w) {
  const bool ok = mbar_wait(bar, parity, w);
  return __all_sync(0xffffffffu, ok);
}

// Barrier over the 128 softmax threads on an mbarrier, so that it is bounded.
__device__ __forceinline__ bool red_sync(uint64_t* bar, uint32_t& phase, const WaitCtl& w) {
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

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

// Byte offset of element (row, k) of a K-major, 128-byte-swizzled operand tile
// whose 64-element column blocks are block_bytes apart (row = MMA M or N index).
__device__ __forceinline__ uint32_t sw128_off(int row, int k, int block_bytes) {
  return (k >> 6) * block_bytes + row * 128 + ((((k & 63) >> 3) ^ (row & 7)) << 4) + (k & 7) * 2;
}

__global__ void __launch_bounds__(kThreads, 1)
    decode_tc_kernel(const __grid_constant__ DecodeArgs a, const __grid_constant__ RopeFreq f,
                     const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v) {
  extern __shared__ uint8_t smem_raw[];
  // aligned by pointer arithmetic on the shared array, so that the compiler keeps shared-memory addressing
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  Bars* bars = reinterpret_cast<Bars*>(smem + kBarOff);
  float* red_m = reinterpret_cast<float*>(smem + kRedOff);  // [2][4][NHP]
  float* red_l = red_m + 2 * 4 * NHP;                        // [4][NHP]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = a.n_h / a.n_kv;
  const int n_units = a.B * a.n_kv * a.n_split;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bars->full[s], 1);
      mbar_init(&bars->empty[s], 1);
    }
    mbar_init(&bars->q_ready, 128);
    mbar_init(&bars->q_empty, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars->s_full[s], 1);
      mbar_init(&bars->p_full[s], 128);
    }
    mbar_init(&bars->pv_done, 1);
    mbar_init(&bars->o_empty, 128);
    mbar_init(&bars->fin, 1);
    mbar_init(&bars->red, 128);
    for (int s = 0; s < kUnitSlots; ++s) {
      mbar_init(&bars->unit_full[s], 1);
      mbar_init(&bars->unit_empty[s], 1 + 128);  // the MMA issuer and every softmax thread
    }
    bars->abort_flag = 0;
    fence_mbar_init();
  }
  // the padding rows (heads G..15) of Q_g and P^T stay zero for the whole kernel
  for (int i = threadIdx.x; i < (2 * kQBlockBytes + 4 * kPBlockBytes) / 16; i += kThreads)
    reinterpret_cast<uint4*>(smem + kQOff)[i] = make_uint4(0, 0, 0, 0);
  fence_proxy_async_smem();
  if (warp == 1) {
    tmem_alloc(&bars->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  // Units are claimed longest first: the (sequence, chunk) pairs are ranked by their number of key
  // tiles (ties by index), so that the last claims of the launch are the shortest units and the
  // SMs finish close together.  Claimed in sequence order, the last claims could be whole
  // 4096-key units; longest first took the 59-sequence decode from 0.244 to 0.233 ms.  The units
  // of one pair (its KV heads) stay consecutive.  More pairs than kMaxOrder keep sequence order.
  const int n_pairs = a.B * a.n_split;
  const bool ordered = n_pairs <= kMaxOrder;
  uint16_t* const ord = reinterpret_cast<uint16_t*>(smem + kOrdOff);
  uint16_t* const pair_tiles = ord + kMaxOrder;
  if (ordered) {
    for (int i = threadIdx.x; i < n_pairs; i += kThreads) {
      Unit w;
      pair_tiles[i] = static_cast<uint16_t>(unit_at(i * a.n_kv, a, w) ? min(w.nt, 0xffff) : 0);
    }
    __syncthreads();
    for (int i = threadIdx.x; i < n_pairs; i += kThreads) {
      const int ti = pair_tiles[i];
      int r = 0;
      for (int j = 0; j < n_pairs; ++j) {
        const int tj = pair_tiles[j];
        r += (tj > ti || (tj == ti && j < i)) ? 1 : 0;
      }
      ord[r] = static_cast<uint16_t>(i);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  const WaitCtl wc{&bars->abort_flag, a.status, a.wait_limit_ns};

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      uint32_t st = 0, ph = 0, issued = 0, last_ph = 0, qs = 0, qph = 0;
      for (;;) {
        Unit w;
        int u;
        do {  // claim the next non-empty unit
          const int k = static_cast<int>(atomicAdd(a.ws_counter, 1u));
          u = (ordered && k < n_units) ? static_cast<int>(ord[k / a.n_kv]) * a.n_kv + k % a.n_kv : k;
        } while (u < n_units && !unit_at(u, a, w));
        if (!mbar_wait(&bars->unit_empty[qs], qph ^ 1, wc)) goto producer_done;
        bars->unit_q[qs] = u < n_units ? u : -1;
        mbar_arrive(&bars->unit_full[qs]);
        if (++qs == kUnitSlots) { qs = 0; qph ^= 1; }
        if (u >= n_units) break;
        for (int t = 0; t < w.nt; ++t) {
          const int k0 = tile_key0(w, t);
          if (!mbar_wait(&bars->empty[st], ph ^ 1, wc)) goto producer_done;
          mbar_arrive_expect_tx(&bars->full[st], kStageBytes);
          uint8_t* kdst = smem + kKVOff + st * kStageBytes;
          for (int db = 0; db < D / 64; ++db)
            for (int hb = 0; hb < BK / kBox; ++hb) {  // rows past max_len read as zero
              tma_load_4d(kdst + db * kBlockBytes + hb * kBox * 128, &tm_k, &bars->full[st], db * 64, w.g,
                          k0 + hb * kBox, w.b);
              tma_load_4d(kdst + kTileBytes + db * kBlockBytes + hb * kBox * 128, &tm_v, &bars->full[st], db * 64,
                          w.g, k0 + hb * kBox, w.b);
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
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint64_t kv_desc0 = sdesc_sw128(smem_u32(smem + kKVOff), 16, 1024);
      const uint64_t v_desc0 = sdesc_sw128(smem_u32(smem + kKVOff + kTileBytes), kBlockBytes, 1024);
      const uint64_t q_desc = sdesc_sw128(smem_u32(smem + kQOff), 16, 1024);
      const uint64_t p_desc0 = sdesc_sw128(smem_u32(smem + kPOff), 16, 1024);
      uint32_t st = 0, ph = 0, pph = 0, tile = 0, n = 0, qs = 0, qph = 0;
      // Descriptors advance by adding offsets in 16-byte units to the start-address
      // field (shared-memory addresses stay below 256 KB: the field never carries).
      auto issue_qk = [&](uint32_t stage, uint32_t sbuf) {
        const uint64_t a0 = kv_desc0 + ((stage * kStageBytes) >> 4);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_ss(tmem + sbuf * NHP, a0 + (((kk >> 2) * kBlockBytes + (kk & 3) * 32) >> 4),
                 q_desc + (((kk >> 2) * kQBlockBytes + (kk & 3) * 32) >> 4), kIdescQK, kk > 0 ? 1u : 0u);
      };
      auto issue_pv = [&](uint32_t stage, uint32_t pbuf, bool accumulate) {
        const uint64_t a0 = v_desc0 + ((stage * kStageBytes) >> 4);
        const uint64_t b0 = p_desc0 + ((pbuf * 2 * kPBlockBytes) >> 4);
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk)
          mma_ss(tmem + kOCol, a0 + ((kk * 16 * 128) >> 4),
                 b0 + (((kk >> 2) * kPBlockBytes + (kk & 3) * 32) >> 4), kIdescPV,
                 (accumulate || kk > 0) ? 1u : 0u);
      };
      for (;;) {
        if (!mbar_wait(&bars->unit_full[qs], qph, wc)) goto mma_done;
        const int u = bars->unit_q[qs];
        mbar_arrive(&bars->unit_empty[qs]);
        if (++qs == kUnitSlots) { qs = 0; qph ^= 1; }
        if (u < 0) break;
        Unit w;
        unit_at(u, a, w);
        const int nt = w.nt;
        if (!mbar_wait(&bars->q_ready, n & 1, wc)) goto mma_done;
        if (!mbar_wait(&bars->full[st], ph, wc)) goto mma_done;
        tc_fence_after();
        issue_qk(st, tile & 1);
        mma_commit(&bars->s_full[tile & 1]);
        if (nt == 1) mma_commit(&bars->q_empty);
        uint32_t cur = st;
        if (++st == kStages) { st = 0; ph ^= 1; }
        for (int t = 0; t < nt; ++t, ++tile) {
          const uint32_t nxt = st;
          if (t + 1 < nt) {
            // S^T buffer (tile + 1) & 1 was read by the softmax of tile - 1, whose P was
            // waited for before the previous P V
            if (!mbar_wait(&bars->full[st], ph, wc)) goto mma_done;
            tc_fence_after();
            issue_qk(st, (tile + 1) & 1);
            mma_commit(&bars->s_full[(tile + 1) & 1]);
            if (t + 1 == nt - 1) mma_commit(&bars->q_empty);
            if (++st == kStages) { st = 0; ph ^= 1; }
          }
          if (!mbar_wait(&bars->p_full[tile & 1], (pph >> (tile & 1)) & 1u, wc)) goto mma_done;
          pph ^= 1u << (tile & 1);
          if (t == 0 && !mbar_wait(&bars->o_empty, (n & 1) ^ 1, wc)) goto mma_done;
          tc_fence_after();
          issue_pv(cur, tile & 1, t > 0);
          mma_commit(&bars->pv_done);
          mma_commit(&bars->empty[cur]);
          cur = nxt;
        }
        ++n;
      }
    mma_done:
      mma_commit(&bars->fin);
      drain_wait(&bars->fin, 0, a.wait_limit_ns);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax + epilogue
    const int sw = warp & 3;             // TMEM lane quadrant
    const int k = sw * 32 + lane;        // key row of a tile / value dim of O^T (TMEM lane)
    const uint32_t lane_off = static_cast<uint32_t>(sw * 32) << 16;
    uint32_t sph = 0, pvph = 0, rph = 0, st = 0, tile = 0, n = 0, qs = 0, qph = 0;
    for (;;) {
      if (!warp_wait(&bars->unit_full[qs], qph, wc)) break;
      const int u = bars->unit_q[qs];
      mbar_arrive(&bars->unit_empty[qs]);
      if (++qs == kUnitSlots) { qs = 0; qph ^= 1; }
      if (u < 0) break;
      Unit w;
      unit_at(u, a, w);
      const int nt = w.nt;
      const int h0 = w.g * G;
      // Q_g into shared memory (rows = heads, K-major, 128-byte swizzle), rotated at
      // the new token's position; the previous unit's QK MMAs must have finished
      // reading it
      if (!warp_wait(&bars->q_empty, (n & 1) ^ 1, wc)) break;
      {
        const __nv_bfloat16* qg =
            static_cast<const __nv_bfloat16*>(a.q) + (static_cast<long long>(w.b) * a.n_h + h0) * D;
        const int pos = w.L - 1;
        // one thread per (head, chunk pair): chunks c and c + 8 hold dims 8c.. and 64 + 8c..
        for (int idx = k; idx < G * 8; idx += 128) {
          const int i = idx >> 3, c = idx & 7;
          float x0[8], x1[8];
          bf16x8_to_f32(*reinterpret_cast<const uint4*>(qg + i * D + c * 8), x0);
          bf16x8_to_f32(*reinterpret_cast<const uint4*>(qg + i * D + 64 + c * 8), x1);
          if (f.n_pairs) {  // the rotated span is the whole head (decode_tc_supported)
            if (f.half) {
#pragma unroll
              for (int e = 0; e < 8; ++e) {
                float sn, cs;
                rope_sincos(pos, f.hi[c * 8 + e], f.lo[c * 8 + e], &sn, &cs);
                rotate_pair(x0[e], x1[e], sn, cs);
              }
            } else {
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                float sn, cs;
                rope_sincos(pos, f.hi[c * 4 + e], f.lo[c * 4 + e], &sn, &cs);
                rotate_pair(x0[2 * e], x0[2 * e + 1], sn, cs);
                rope_sincos(pos, f.hi[32 + c * 4 + e], f.lo[32 + c * 4 + e], &sn, &cs);
                rotate_pair(x1[2 * e], x1[2 * e + 1], sn, cs);
              }
            }
          }
          *reinterpret_cast<uint4*>(smem + kQOff + sw128_off(i, c * 8, kQBlockBytes)) = f32_to_bf16x8(x0);
          *reinterpret_cast<uint4*>(smem + kQOff + sw128_off(i, 64 + c * 8, kQBlockBytes)) = f32_to_bf16x8(x1);
        }
        fence_proxy_async_smem();
      }
      mbar_arrive(&bars->q_ready);

      float m_run[NHP], l_part[NHP];
#pragma unroll
      for (int i = 0; i < NHP; ++i) {
        m_run[i] = -INFINITY;
        l_part[i] = 0.f;
      }
      bool ok = true;
      for (int t = 0; t < nt; ++t, ++tile) {
        const uint32_t sbuf = tile & 1;
        if (!warp_wait(&bars->s_full[sbuf], (sph >> sbuf) & 1u, wc)) { ok = false; break; }
        sph ^= 1u << sbuf;
        tc_fence_after();
        uint32_t sr[NHP];
        tmem_ld16(tmem + lane_off + sbuf * NHP, sr);
        tmem_wait_ld();
        const bool valid = tile_key0(w, t) + k < tile_kend(w, t);
        float x[NHP];
#pragma unroll
        for (int i = 0; i < NHP; ++i) x[i] = valid ? __uint_as_float(sr[i]) * a.scale_log2 : -INFINITY;
        // block maximum of every head over the 128 keys: warp, then the four warps
        float* rm = red_m + (tile & 1) * 4 * NHP;
#pragma unroll
        for (int i = 0; i < NHP; ++i) {
          if (i >= G) break;
          float v = x[i];
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
          if (lane == 0) rm[sw * NHP + i] = v;
        }
        if (!red_sync(&bars->red, rph, wc)) { ok = false; break; }
        bool need = false;
        float alpha[NHP];
#pragma unroll
        for (int i = 0; i < NHP; ++i) {
          alpha[i] = 1.f;
          if (i >= G) continue;
          const float mx = fmaxf(fmaxf(rm[i], rm[NHP + i]), fmaxf(rm[2 * NHP + i], rm[3 * NHP + i]));
          if (mx > m_run[i] + kRescaleThreshold) {
            if (m_run[i] != -INFINITY) alpha[i] = fast_exp2(m_run[i] - mx);
            m_run[i] = mx;
            need = true;
          }
        }
        // P V of the previous tile has completed: O^T may be rescaled and P^T buffer
        // sbuf (last read two tiles ago) rewritten
        if (t > 0) {
          if (!warp_wait(&bars->pv_done, pvph, wc)) { ok = false; break; }
          pvph ^= 1;
          tc_fence_after();
          if (need) {  // uniform across the softmax threads
            uint32_t orow[NHP];
            tmem_ld16(tmem + lane_off + kOCol, orow);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < NHP; ++i) orow[i] = __float_as_uint(__uint_as_float(orow[i]) * alpha[i]);
            tmem_st16(tmem + lane_off + kOCol, orow);
            tmem_wait_st();
          }
        }
        // P^T [key][head] into the K-major B operand (rows = heads, k = key)
        uint8_t* pb = smem + kPOff + sbuf * 2 * kPBlockBytes;
#pragma unroll
        for (int i = 0; i < NHP; ++i) {
          if (i >= G) break;
          l_part[i] *= alpha[i];
          const float m_ref = m_run[i] == -INFINITY ? 0.f : m_run[i];
          const float p = valid ? fast_exp2(x[i] - m_ref) : 0.f;
          l_part[i] += p;
          *reinterpret_cast<__nv_bfloat16*>(pb + sw128_off(i, k, kPBlockBytes)) = __float2bfloat16_rn(p);
        }
        if (!valid) {
          // rows past the range may hold anything (even NaN): zero this key's value row so
          // that P V stays finite
          uint8_t* vt = smem + kKVOff + st * kStageBytes + kTileBytes;
#pragma unroll
          for (int c = 0; c < D / 8; ++c)
            *reinterpret_cast<uint4*>(vt + (c >> 3) * kBlockBytes + k * 128 + ((((c & 7) ^ (k & 7))) << 4)) =
                make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(&bars->p_full[sbuf]);
        if (++st == kStages) st = 0;
      }
      if (!__all_sync(0xffffffffu, ok)) break;
      // epilogue: normaliser of every head over the whole chunk, then O^T / l
      if (!warp_wait(&bars->pv_done, pvph, wc)) break;
      pvph ^= 1;
      tc_fence_after();
#pragma unroll
      for (int i = 0; i < NHP; ++i) {
        if (i >= G) break;
        float v = l_part[i];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (lane == 0) red_l[sw * NHP + i] = v;
      }
      if (!red_sync(&bars->red, rph, wc)) break;
      uint32_t orow[NHP];
      tmem_ld16(tmem + lane_off + kOCol, orow);
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(&bars->o_empty);
      const int split = w.split;
#pragma unroll
      for (int i = 0; i < NHP; ++i) {
        if (i >= G) break;
        const float l = red_l[i] + red_l[NHP + i] + red_l[2 * NHP + i] + red_l[3 * NHP + i];
        const long long slot = (static_cast<long long>(w.b) * a.n_h + h0 + i) * a.n_split + split;
        a.ws_o[slot * D + k] = __uint_as_float(orow[i]) / l;
        if (k == 0) a.ws_lse[slot] = m_run[i] + log2f(l);
      }
      // red_l is rewritten by the next unit only after its first red_sync of a tile,
      // which every thread reaches after this read
      ++n;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

bool decode_tc_supported(int n_h, int n_kv, int D_qk, int D_v, bool bf16, int rope_offset, int rope_dims, bool rope) {
  const int G = n_h / n_kv;
  return bf16 && D_qk == D && D_v == D && G >= 1 && G <= NHP && (!rope || (rope_offset == 0 && rope_dims == D));
}

cudaError_t launch_decode_tc(const DecodeArgs& a, const RopeFreq& rope, const CUtensorMap* maps, int num_sms,
                             cudaStream_t st, int* launches) {
  cudaError_t e = cudaFuncSetAttribute(decode_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  if ((e = cudaMemsetAsync(a.ws_counter, 0, sizeof(unsigned int), st)) != cudaSuccess) return e;  // unit claims
  const long long units = static_cast<long long>(a.B) * a.n_kv * a.n_split;
  const int grid = static_cast<int>(units < num_sms ? units : num_sms);
  decode_tc_kernel<<<grid, kThreads, kSmemBytes, st>>>(a, rope, maps[0], maps[1]);
  *launches += 1;
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_decode_combine(a, true, st, launches);
}

}  // namespace attn

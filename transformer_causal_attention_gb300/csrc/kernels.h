// kernels.h - launch interface between the C ABI (api.cu) and the kernel
// translation units.  Host-side only; nothing here is exported.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>

#include "common.cuh"

namespace attn {

struct PrefillArgs {
  const void* q;
  const void* k;  // keys as the kernels read them: already rotated when RoPE is on
  const void* v;
  void* out;
  float* lse;  // nullable
  int B, S, n_h, n_kv, D;  // S = query rows per sequence; D = head dim of q and k
  float scale_log2;  // score multiplier times log2(e)
  int causal;
  unsigned int* status;
  unsigned long long wait_limit_ns;
  int S_k;           // keys visible per sequence (keys 0 .. S_k-1)
  int q_offset;      // absolute position of query row 0 (a chunk continuing a cache)
  int kv_rows;       // rows per sequence in the K/V buffers (S for a prompt, max_len for a cache)
  int window;        // > 0: a query at position p sees keys n with p - n < window ...
  int n_sink;        // ... plus the first n_sink keys (attention sinks); window 0: no window
  int D_v;           // head dim of v and out
  int rope_offset;   // first rotated dim of q and k (the span holds 2 * n_pairs dims)
  int fold;          // 1: deal work items as (heavy, light) pairs of one head, head after head
  int head_pairs;    // 1: a work item is one Q tile of two query heads of a K/V group (n_h / n_kv even)
};

struct DecodeArgs {
  const void* q;
  const void* kcache;
  const void* vcache;
  long long v_token_stride;  // elements
  const int* seqlens;
  void* out;
  float* lse;  // nullable
  int B, n_h, n_kv, D_qk, D_v, max_len;
  int rope_offset;
  float scale_log2;
  float* ws_o;    // [B, n_h, n_split, D_v] partial outputs (normalised)
  float* ws_lse;  // [B, n_h, n_split] partial log2-normalisers
  int n_split, chunk;
  unsigned int* status;
  unsigned long long wait_limit_ns;
  int window;  // > 0: the new token (position L-1) sees keys n with L-1-n < window, plus n < n_sink
  int n_sink;
  unsigned int* ws_counter;  // scratch counter in the workspace (work claims of the tensor-core GQA decode)
};

// Visible keys of a decode query at position L - 1: [0, L) without a window,
// else [0, min(n_sink, L)) and [max(0, L - window), L).  Returns the number of
// key ranges (1 or 2) in lo/hi.
__host__ __device__ __forceinline__ int decode_visible(int L, int window, int n_sink, int* lo, int* hi) {
  if (window <= 0 || L - window <= n_sink) {  // no window, or window and sinks touch: all keys
    lo[0] = 0;
    hi[0] = L;
    return 1;
  }
  if (n_sink <= 0) {
    lo[0] = L - window;
    hi[0] = L;
    return 1;
  }
  lo[0] = 0;
  hi[0] = n_sink;
  lo[1] = L - window;
  hi[1] = L;
  return 2;
}

struct RopeArgs {
  void* out;
  const void* in;
  int B, S, n_heads, D, rope_offset, rope_dims, pos_offset;
  const int* positions;  // nullable device [B * S]: position of each row; null: pos_offset + s
};

struct KvAppendArgs {
  const void* k_new;  // [B, C, n_kv, D_qk]
  const void* v_new;  // [B, C, n_kv, D_v] or null (values alias the keys)
  void* kcache;       // [B, max_len, n_kv, D_qk]
  void* vcache;       // token stride v_token_stride elements
  long long v_token_stride;
  const int* start;   // device [B]: slot of the first new token of each sequence
  int B, C, n_kv, D_qk, D_v, max_len, rope_offset;
  int head_groups;    // set by the launcher: threads per (token, 8-dim chunk), each owning n_kv / head_groups heads
};

// Each launcher returns the launch error (cudaSuccess when enqueued) and adds
// the number of kernels it enqueued to *launches.
cudaError_t launch_prefill_simt(const PrefillArgs& a, const RopeFreq& rope, bool bf16, cudaStream_t st,
                                int* launches);
bool prefill_tc_supported(int D_qk, int D_v, bool bf16);
// The MLA prefill shape (q/k head dim 192, v head dim 128, bf16, no window) on the tensor cores
// of CTA pairs (prefill_pair.cu); maps: Q and V with 128-row boxes, K with 64-row boxes.
bool prefill_pair_supported(int D_qk, int D_v, bool bf16, int window);
cudaError_t launch_prefill_pair(const PrefillArgs& a, const RopeFreq& rope, const CUtensorMap* maps, cudaStream_t st,
                                int* launches);
cudaError_t launch_prefill_tc(const PrefillArgs& a, const RopeFreq& rope, const CUtensorMap* maps,
                              int num_sms, cudaStream_t st, int* launches);
cudaError_t launch_rope(const RopeArgs& a, const RopeFreq& rope, bool bf16, cudaStream_t st, int* launches);
cudaError_t launch_kv_append(const KvAppendArgs& a, const RopeFreq& rope, bool bf16, cudaStream_t st, int* launches);
int decode_plan_splits(int B, int n_h, int n_kv, int D_qk, int D_v, int max_len, int* chunk);
cudaError_t launch_decode(const DecodeArgs& a, const RopeFreq& rope, bool bf16, cudaStream_t st,
                          int* launches);
cudaError_t launch_decode_combine(const DecodeArgs& a, bool bf16, cudaStream_t st, int* launches);
constexpr int kMlaMaxPairs = 128;  // CTA pairs of the MLA decode kernel (workspace is sized for this)
constexpr int kMlaTileKeys = 128;  // keys per CTA per round (TMA box rows) of the MLA decode kernel
bool decode_mla_supported(int B, int n_h, int n_kv, int D_qk, int D_v, long long v_token_stride, bool v_is_k,
                          bool bf16);
int decode_mla_pairs(int num_sms);
// Whether the MLA kernel can rotate the query span [rope_offset, rope_offset + rope_dims).
bool decode_mla_rope_ok(int rope_offset, int rope_dims, bool half);
cudaError_t launch_decode_mla(const DecodeArgs& a, const RopeFreq& rope, const CUtensorMap* maps, cudaStream_t st,
                              int* launches);
constexpr int kStreamTileKeys = 64;  // keys per TMA box of the streaming GQA decode
constexpr int kDecodeTcMinChunk = 4096;  // keys per work unit of the tensor-core GQA decode, at least
bool decode_tc_supported(int n_h, int n_kv, int D_qk, int D_v, bool bf16, int rope_offset, int rope_dims, bool rope);
cudaError_t launch_decode_tc(const DecodeArgs& a, const RopeFreq& rope, const CUtensorMap* maps, int num_sms,
                             cudaStream_t st, int* launches);
bool decode_stream_supported(int n_h, int n_kv, int D_qk, int D_v, bool bf16);
cudaError_t launch_decode_stream(const DecodeArgs& a, const RopeFreq& rope, const CUtensorMap* maps, int num_sms,
                                 cudaStream_t st, int* launches);

}  // namespace attn

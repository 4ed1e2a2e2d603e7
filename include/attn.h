/*
 * attn.h - C ABI of libattn.so: causal scaled dot-product attention with RoPE
 * and GQA/MQA head sharing on one NVIDIA GB300 (sm_103a).
 *
 * The operation is
 *     O = softmax(Q' K'^T * scale + M) V,   Q' = RoPE(Q), K' = RoPE(K)
 * per head, with M[m, n] = -inf for keys after the query
 * ("Transformer架构从Attention到DecoderBlock" §4.2-§4.5, eq. head_i; the mask of
 * "2.7 Transformer Decoder Block完整解析" §3.2), RoPE rotating each dimension pair
 * (2i, 2i+1) by pos * base^(-2i/D) ("Transformer架构从Attention到DecoderBlock"
 * §8.2-§8.3) and query head h reading KV head floor(h / (n_h / n_kv)) (§6.3).
 *
 * Conventions shared by every entry point:
 *  - Every tensor pointer is a DEVICE pointer owned by the caller; the library
 *    keeps no pointer after a call returns and allocates no device memory.
 *  - Tensors are dense, row-major, innermost dimension last; activations use the
 *    BSHD layout [batch, sequence, heads, head_dim].
 *  - dtype selects the element type of q/k/v/out/caches: ATTN_F32 (float) or
 *    ATTN_BF16 (__nv_bfloat16).  Arithmetic is fp32 in either case; bf16 inputs
 *    feed bf16 tensor-core MMAs with fp32 accumulation.
 *  - stream is a cudaStream_t passed as void*; NULL is the legacy default stream.
 *    Calls only enqueue work: they return before the kernels finish.
 *  - Return value: ATTN_OK (0) or a negative ATTN_ERR_* code.  Argument errors
 *    are detected on the host before anything is launched.  A device-side
 *    bounded wait that expires is reported later by attn_device_status().
 *  - All pointers must be 16-byte aligned (vector and TMA loads), else
 *    ATTN_ERR_ALIGN.
 */
#ifndef ATTN_H
#define ATTN_H

#include <stddef.h>

#if defined(__GNUC__)
#define ATTN_API __attribute__((visibility("default")))
#else
#define ATTN_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/*
 * The dtype argument of every call: the element type in the low byte, with
 * ATTN_ROPE_HALF optionally OR'd in by any call that applies RoPE.  That flag
 * pairs dimension j of the rotated span with j + rope_dims/2 (the split-halves
 * layout of the apply_rope code in "2.7 Transformer Decoder Block完整解析" §4)
 * instead of (2i, 2i+1); pair j still turns by pos * rope_base^(-2j/rope_dims).
 * Either layout is a rotation of 2-d subspaces ("Transformer架构从Attention到
 * DecoderBlock" §8.1 allows both if training and inference agree): keys written
 * to a cache with one pairing must be read back by calls using the same one.
 * With the flag, each half of a rotated span must consist of whole chunks where
 * a call asks for multiples of 8 (16 instead of 8; 4 instead of 2 for ATTN_F32).
 * Any other bit is ATTN_ERR_ARG.
 */
typedef enum {
  ATTN_F32 = 0,
  ATTN_BF16 = 1,
  ATTN_ROPE_HALF = 0x100,
  ATTN_F32_ROPE_HALF = ATTN_F32 | ATTN_ROPE_HALF,
  ATTN_BF16_ROPE_HALF = ATTN_BF16 | ATTN_ROPE_HALF
} attn_dtype_t;

enum {
  ATTN_OK = 0,
  ATTN_ERR_ARG = -1,          /* null pointer, non-positive size, n_h % n_kv != 0, bad span */
  ATTN_ERR_UNSUPPORTED = -2,  /* a head dim / dtype combination no kernel handles */
  ATTN_ERR_ALIGN = -3,        /* a pointer is not 16-byte aligned */
  ATTN_ERR_CUDA = -4,         /* the CUDA runtime rejected a launch (no device, bad stream...) */
  ATTN_ERR_TIMEOUT = -5,      /* a bounded device wait expired (reported by attn_device_status) */
  ATTN_ERR_WORKSPACE = -6     /* the caller's workspace is smaller than required */
};

/* Static, human-readable text for a return code. Never NULL. */
ATTN_API const char* attn_strerror(int code);

/*
 * attn_prefill - attention over whole prompts (prefill), never materialising S.
 *
 * Defined by "Transformer架构从Attention到DecoderBlock" §4.5 (head_i = softmax(
 * Q_i K_i^T / sqrt(D_h) + M) V_i) with §13.1 (prefill: the whole prompt at once);
 * computed tile by tile with the online softmax of "Transformer架构完全深度解析"
 * §13 (running max m and sum l), skipping key tiles that lie wholly after the
 * query tile ("2.7 Transformer Decoder Block完整解析" §3.3).
 *
 *   q      [B, S, n_h,  D_h]  queries, NOT rotated.
 *   k      [B, S, n_kv, D_h]  keys, NOT rotated.
 *   v      [B, S, n_kv, D_h]  values (never rotated).
 *   out    [B, S, n_h,  D_h]  result, same dtype.
 *   k_rot  [B, S, n_kv, D_h]  receives RoPE(K), the rotated keys a KV cache
 *                             stores ("Transformer架构完全深度解析" §7).  Required
 *                             when rope_base > 0, ignored (may be NULL) otherwise.
 *                             It must not overlap k.
 *   lse    [B, n_h, S] fp32   optional (NULL to skip): natural-log normaliser
 *                             log sum_n exp(score[m, n]) of each query row.
 *   rope_base  > 0: rotate Q and K with theta_i = rope_base^(-2i/D_h); <= 0: no RoPE.
 *   scale      > 0: score multiplier; <= 0: 1/sqrt(D_h).
 *   causal     1: mask keys n > m (the diagonal stays visible); 0: no mask.
 * Supported: ATTN_F32 with D_h even, 2 <= D_h <= 256; ATTN_BF16 with D_h a
 * multiple of 8, 8 <= D_h <= 256.  n_h must be a multiple of n_kv.
 */
ATTN_API int attn_prefill(const void* q, const void* k, const void* v, void* out, void* k_rot,
                 float* lse, int B, int S, int n_h, int n_kv, int D_h, float rope_base,
                 float scale, int causal, attn_dtype_t dtype, void* stream);

/*
 * attn_prefill_mla - prefill with separate head dims for q/k and v and RoPE on
 * a span of the q/k dims: the non-absorbed path of Multi-head Latent Attention
 * ("Transformer 与 LLM" slide 06).  There every head scores
 * q . [k^C ; k^R] / sqrt(192): a 128-dim content part (the latent c^KV
 * up-projected per head) and a 64-dim decoupled RoPE part k^R that all heads
 * share, against values of 128 dims; the slide notes that prefill takes this
 * path because absorbing W_UK / W_UV would cost ~3.4x the attention FLOPs.
 * The call is that MHA-like attention for any (D_qk, D_v):
 *
 *   q      [B, S, n_h,  D_qk]  queries, NOT rotated.
 *   k      [B, S, n_kv, D_qk]  keys, NOT rotated (the caller writes k^R into
 *                              the last rope_dims dims of every head).
 *   v      [B, S, n_kv, D_v]   values.
 *   out    [B, S, n_h,  D_v].
 *   k_rot  [B, S, n_kv, D_qk]  receives k with its RoPE span rotated; required
 *                              when rope_base > 0, must not overlap k.
 *   lse    [B, n_h, S] fp32    optional, as attn_prefill.
 *   rope_base > 0 rotates dims [rope_offset, rope_offset + rope_dims) of q and
 *              k at their positions with theta_i = rope_base^(-2i/rope_dims);
 *              <= 0: no RoPE (offset and dims ignored).
 *   scale     > 0: score multiplier; <= 0: 1/sqrt(D_qk) (1/sqrt(192) for MLA).
 *   causal    1: mask keys n > m; 0: no mask.
 * Tensor cores run (D_qk, D_v) = (64, 64), (128, 128) and (192, 128) in bf16;
 * other sizes up to 256 (multiples of 8 in bf16, of 2 in fp32) run on CUDA
 * cores.  rope_offset must be a multiple of 8 (bf16) or 2 (fp32) and
 * rope_dims of 8 or 2 (16 or 4 with ATTN_ROPE_HALF).  Errors as attn_prefill.
 */
ATTN_API int attn_prefill_mla(const void* q, const void* k, const void* v, void* out, void* k_rot, float* lse,
                              int B, int S, int n_h, int n_kv, int D_qk, int D_v, float rope_base, int rope_offset,
                              int rope_dims, float scale, int causal, attn_dtype_t dtype, void* stream);

/*
 * attn_rope - rotate dims [rope_offset, rope_offset + rope_dims) of every row
 * of x_in [B, S, n_heads, D] at position pos_offset + s (s = sequence index),
 * pairing (2i, 2i+1) with theta_i = rope_base^(-2i/rope_dims)
 * ("Transformer架构从Attention到DecoderBlock" §8.2-§8.3).  Dims outside the span
 * are copied unchanged.  x_out may equal x_in (in place) but must not partially
 * overlap it.  rope_offset, rope_dims and D must be multiples of 8 (bf16) or
 * 2 (f32); rope_base must be > 0.  This is the step that fills a cache with
 * rotated keys.
 */
ATTN_API int attn_rope(void* x_out, const void* x_in, int B, int S, int n_heads, int D,
              int rope_offset, int rope_dims, float rope_base, int pos_offset,
              attn_dtype_t dtype, void* stream);

/*
 * attn_rope_at - attn_rope with a position per row instead of consecutive ones:
 * row s of sequence b is rotated at positions[b * S + s].  Each cached key
 * carries its own absolute position ("Transformer架构完全深度解析" §7), so rows
 * whose slots are not consecutive - a batch of requests at different depths,
 * tokens scattered in a cache - are rotated in one call.
 *
 *   positions  DEVICE int32 [B, S] (required, 4-byte aligned); any value is
 *              rotated as given (positions are meant to be in [0, 2^24), where
 *              the angle keeps full fp32 accuracy).
 * Everything else, layouts and errors as attn_rope.
 */
ATTN_API int attn_rope_at(void* x_out, const void* x_in, const int* positions, int B, int S, int n_heads, int D,
                          int rope_offset, int rope_dims, float rope_base, attn_dtype_t dtype, void* stream);

/*
 * attn_prefill_window - attn_prefill with a causal sliding window and
 * attention sinks ("Transformer 与 LLM" slide 07: a window of W keys turns the
 * O(s) KV and compute of each query into O(W); keeping the first few tokens -
 * the sinks - preserves the start of the sequence).  A query at position m sees
 * key n when n <= m and (m - n < window or n < n_sink).  Key tiles that hold no
 * visible key for a query tile are skipped.  window > 0 is required; other
 * arguments as attn_prefill (the mask is always causal).
 */
ATTN_API int attn_prefill_window(const void* q, const void* k, const void* v, void* out, void* k_rot, float* lse,
                                 int B, int S, int n_h, int n_kv, int D_h, float rope_base, float scale, int window,
                                 int n_sink, attn_dtype_t dtype, void* stream);

/*
 * attn_prefill_chunk - a chunk of a prompt whose earlier keys are already in a
 * KV cache (chunked prefill, "Transformer 与 LLM" slide 07: a long prompt is
 * split so that one request does not hold the GPU).  Query row m of the chunk
 * sits at absolute position q_offset + m and, when causal, attends cache keys
 * 0 .. q_offset + m ("2.7 Transformer Decoder Block完整解析" §3.2); without the
 * mask it attends keys 0 .. q_offset + S_q - 1.
 *
 *   q       [B, S_q, n_h, D_h]       the chunk's queries, NOT rotated (rotated here
 *                                    at their absolute positions when rope_base > 0).
 *   kcache  [B, max_len, n_kv, D_h]  rotated keys; rows 0 .. q_offset + S_q - 1 must
 *                                    already hold this chunk's keys too (attn_kv_append).
 *   vcache  [B, max_len, n_kv, D_h]  values, same layout.
 *   out     [B, S_q, n_h, D_h]; lse optional fp32 [B, n_h, S_q].
 * Requires 0 <= q_offset and q_offset + S_q <= max_len.  Other arguments,
 * dtypes and errors as attn_prefill.  Rows past q_offset + S_q are never read.
 */
ATTN_API int attn_prefill_chunk(const void* q, const void* kcache, const void* vcache, void* out, float* lse,
                                int B, int S_q, int q_offset, int max_len, int n_h, int n_kv, int D_h,
                                float rope_base, float scale, int causal, attn_dtype_t dtype, void* stream);

/*
 * attn_kv_append - write C new tokens per sequence into a KV cache: key row c
 * of sequence b is rotated at absolute position start[b] + c (the cache keeps
 * rotated keys, "Transformer架构完全深度解析" §7) and stored in that slot, its value
 * row is copied next to it (§9: K_cache = concat(K_cache, K_new)).
 *
 *   k_new   [B, C, n_kv, D_qk]; v_new [B, C, n_kv, D_v], or NULL when values
 *           alias the keys (MLA: V is the first D_v dims of the stored row).
 *   kcache  [B, max_len, n_kv, D_qk]; vcache with token stride v_token_stride
 *           (0 = n_kv * D_v), as in attn_decode.
 *   start   DEVICE int32 [B]: slot of the first new token of each sequence (for
 *           one decode step: seqlens[b] - 1).  Slots outside [0, max_len) are skipped.
 *   rope_base > 0 rotates dims [rope_offset, rope_offset + rope_dims) of the keys.
 * D_qk, D_v, rope_offset and rope_dims must be multiples of 8.
 */
ATTN_API int attn_kv_append(const void* k_new, const void* v_new, void* kcache, void* vcache, int v_token_stride,
                            const int* start, int B, int C, int n_kv, int D_qk, int D_v, int max_len,
                            float rope_base, int rope_offset, int rope_dims, attn_dtype_t dtype, void* stream);

/*
 * attn_decode_workspace_size - bytes of device scratch attn_decode needs for
 * these sizes (0 is never returned for valid sizes; -1 cast to size_t for
 * invalid ones).  The caller allocates it; it may be reused across calls that
 * do not overlap on the GPU.
 */
ATTN_API size_t attn_decode_workspace_size(int B, int n_h, int n_kv, int D_qk, int D_v, int max_len,
                                  attn_dtype_t dtype);

/*
 * attn_decode - one new query token per sequence against its KV cache.
 *
 * Defined by "Transformer架构完全深度解析" §9 (K_cache = concat(K_cache, K_new),
 * then Attention(Q[t+1], K_cache, V_cache)) and "Transformer架构从Attention到
 * DecoderBlock" §13.2.  The cache holds rotated keys, so only q is rotated, at
 * position seqlens[b] - 1.  The key range is split into chunks processed in
 * parallel; their partial results are merged with the running-max /
 * running-sum rule of the online softmax ("Transformer架构完全深度解析" §13).
 * With n_kv = 1, D_qk = 576, D_v = 512 and vcache aliasing kcache this is the
 * MLA-absorbed decode of "Transformer 与 LLM" slide 06 (128 heads sharing one
 * 576-dim latent head; pass scale = 1/sqrt(192)).
 *
 *   q        [B, n_h, D_qk]          new queries, NOT rotated.
 *   kcache   [B, max_len, n_kv, D_qk] rotated keys; rows >= seqlens[b] are never read.
 *   vcache   values: element (b, t, g, d) at vcache[(b*max_len + t)*v_token_stride + g*D_v + d].
 *   v_token_stride  elements between consecutive tokens of vcache; 0 means n_kv*D_v.
 *                   MLA passes vcache = kcache and v_token_stride = D_qk.
 *   seqlens  DEVICE int32 [B]: valid keys per sequence INCLUDING the new token,
 *            1 <= seqlens[b] <= max_len (out-of-range values are clamped on the device).
 *   out      [B, n_h, D_v]  result, same dtype.
 *   lse      optional fp32 [B, n_h] natural-log normaliser (NULL to skip).
 *   rope_base > 0 rotates q dims [rope_offset, rope_offset + rope_dims); <= 0: no RoPE.
 *   scale     > 0: score multiplier; <= 0: 1/sqrt(D_qk).
 *   workspace device scratch of at least attn_decode_workspace_size(...) bytes,
 *             16-byte aligned, owned by the caller; its contents on entry are ignored.
 * Supported: D_qk, D_v multiples of 8 up to 576 and 512; n_h / n_kv <= 128.
 */
ATTN_API int attn_decode(const void* q, const void* kcache, const void* vcache, int v_token_stride,
                const int* seqlens, void* out, float* lse, int B, int n_h, int n_kv, int D_qk,
                int D_v, int max_len, float rope_base, int rope_offset, int rope_dims,
                float scale, attn_dtype_t dtype, void* workspace, size_t workspace_bytes,
                void* stream);

/*
 * attn_decode_window - attn_decode with a sliding window and attention sinks
 * ("Transformer 与 LLM" slide 07): the new token at position L-1 sees cached
 * keys n with L-1-n < window, plus the first n_sink keys.  Key chunks with no
 * visible key are not read.  window > 0 is required; everything else as
 * attn_decode (same workspace size).
 */
ATTN_API int attn_decode_window(const void* q, const void* kcache, const void* vcache, int v_token_stride,
                                const int* seqlens, void* out, float* lse, int B, int n_h, int n_kv, int D_qk,
                                int D_v, int max_len, float rope_base, int rope_offset, int rope_dims,
                                float scale, int window, int n_sink, attn_dtype_t dtype, void* workspace,
                                size_t workspace_bytes, void* stream);

/*
 * attn_decode_static - attn_decode for callers that cannot allocate device
 * memory.  The pages have no counterpart to this entry point: it exists for
 * callers that are not allowed to call cudaMalloc (or anything that does) when
 * they run a decode step - for example an inference-engine plugin whose
 * per-step hook must not allocate because the engine owns all device memory,
 * a latency-critical token loop that cannot afford the device-wide
 * synchronisation cudaMalloc/cudaFree may cause, or a runtime whose device
 * memory budget is fixed at start-up.  Such a caller cannot provide
 * attn_decode's workspace, so this variant keeps the split-KV partial results
 * in a scratch array compiled into the library instead:
 *  - the array is ATTN_DECODE_STATIC_SCRATCH_BYTES (16 MiB) of device memory
 *    that every GPU holds from the library's first use there (the module is
 *    loaded lazily by default; with CUDA_MODULE_LOADING=EAGER, from the moment
 *    the library is loaded) until the process exits, whether or not this
 *    function is ever called;
 *  - a problem whose attn_decode_workspace_size(...) exceeds that size is
 *    rejected with ATTN_ERR_WORKSPACE before anything is launched (for
 *    example the GQA decode of 59 sequences x 8192 keys, n_h = 32, n_kv = 8,
 *    D = 128 fits; the 32 x 32768-key MLA decode does not);
 *  - the first call on a device looks up the array's device address (once per
 *    device, with that device current); make that first call before any
 *    stream capture;
 *  - every call on a device shares the one array and it keeps whatever the
 *    last call left in it.  Nothing in it needs to start at zero (each call
 *    writes every partial it later reads), but calls whose kernels can overlap
 *    on the GPU - on different streams without ordering between them - race on
 *    the array and give wrong results: order them.
 * Arguments, layouts, results and errors are those of attn_decode, minus the
 * workspace pair.  No device memory is allocated or freed.
 */
#define ATTN_DECODE_STATIC_SCRATCH_BYTES (16u << 20)
ATTN_API int attn_decode_static(const void* q, const void* kcache, const void* vcache, int v_token_stride,
                                const int* seqlens, void* out, float* lse, int B, int n_h, int n_kv, int D_qk,
                                int D_v, int max_len, float rope_base, int rope_offset, int rope_dims,
                                float scale, attn_dtype_t dtype, void* stream);

/*
 * attn_device_status - synchronise the stream, then return ATTN_OK, or
 * ATTN_ERR_TIMEOUT if a kernel of this library gave up on a bounded wait since
 * the last call, or ATTN_ERR_CUDA if the stream reports an error or a kernel
 * found its shared memory laid out other than it requires (and skipped its
 * work); the device flags are cleared.
 */
ATTN_API int attn_device_status(void* stream);

/*
 * attn_check_wait_timeout - exercise the failure path of the bounded device
 * waits: launches one warp that waits on a barrier nothing will ever complete.
 * The wait gives up after the current wait limit (attn_set_wait_limit_ns), sets
 * the status word and returns, so a following attn_device_status() reports
 * ATTN_ERR_TIMEOUT (and clears it) while the CUDA context stays usable.  No
 * other kernel is affected; the launch itself returns ATTN_OK or ATTN_ERR_CUDA.
 */
ATTN_API int attn_check_wait_timeout(void* stream);

/* Number of kernels this library has launched since it was loaded. */
ATTN_API unsigned long long attn_launch_count(void);

/* Set the per-wait limit of device-side bounded waits, in nanoseconds
 * (default 2e9).  Applies to launches made after the call. */
ATTN_API void attn_set_wait_limit_ns(unsigned long long ns);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_H */

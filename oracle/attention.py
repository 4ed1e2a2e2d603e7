"""Plain fp64 CPU oracle for causal scaled dot-product attention.

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the test suite, the package smoke
check and the benchmark's CPU-baseline / reference arm may import this module.
It shares no code, table or constant with the CUDA library: the two sides meet
only through the seeded inputs of the ``workloads`` module.

Everything here is the textbook definition written out, in float64, with the
score matrix S materialised, so that each step can be checked against the
pages by eye:

* RoPE - "Transformer架构从Attention到DecoderBlock" §8.2 (frequency of pair i:
  theta_i = base^(-2i/D_r)) and §8.3 (rotation of the pair (2i, 2i+1) by the
  angle m*theta_i); the half-split pairing (j, j + D/2) is the one printed in
  the PyTorch block of "2.7 Transformer Decoder Block完整解析" §4.
* scores, mask, softmax, weighted sum - "Transformer架构从Attention到DecoderBlock"
  §4.2-§4.5 (S = Q K^T / sqrt(D_h), M[m, n] = -inf for n > m, softmax along
  the key axis, O = A V); "Transformer架构完全深度解析" §5.
* GQA / MQA head sharing - "Transformer架构从Attention到DecoderBlock" §6.3:
  query head h reads KV head floor(h / G), G = n_h / n_kv.
* KV-cache decode - "Transformer架构完全深度解析" §9: the new token's k, v are
  appended first, then Attention(q_new, K_cache, V_cache); the cache holds
  already-rotated K (§7, "cached keys carry their position").
* MLA absorbed decode - "Transformer 与 LLM：结构、实现与算量" slide 06: only
  c^KV (512) and the rotated k^R (64) are cached; W_UK is folded into the
  query and W_UV into the output, so all heads share one 576-dim KV head;
  scores use 1/sqrt(192).

Pins (tests/test_oracle.py) tie every function here to something other than
itself: the printed masks, closed forms, invariants and an independently
written brute-force triple loop.
"""
from __future__ import annotations

import math

import numpy as np

NEG_INF = -np.inf


def _f64(x) -> np.ndarray:
    """Exact float64 copy of an array-like (bf16/fp32 torch tensors included)."""
    if hasattr(x, "detach"):  # a torch tensor: widening to float64 is exact
        x = x.detach().cpu().double().numpy()
    return np.asarray(x, dtype=np.float64)


# --------------------------------------------------------------------------
# mask
# --------------------------------------------------------------------------
def causal_mask(n_q: int, n_k: int | None = None, q_offset: int = 0,
                window: int = 0, n_sink: int = 0) -> np.ndarray:
    """Additive mask M[m, n] (0 = keep, -inf = masked).

    "2.7 Transformer Decoder Block完整解析" §3.2/§3.3: the key n is masked when
    it lies after the query (n > m); the diagonal stays visible.  Query row m
    sits at absolute position q_offset + m (q_offset > 0 is a prefill chunk
    that continues an existing cache, "Transformer 与 LLM" slide 07).
    window > 0 additionally masks keys that are window or more positions
    behind the query, except the first n_sink keys (sliding window with
    attention sinks, "Transformer 与 LLM" slide 07).
    """
    n_k = n_q + q_offset if n_k is None else n_k
    m = (q_offset + np.arange(n_q))[:, None]
    n = np.arange(n_k)[None, :]
    masked = n > m
    if window > 0:
        masked = masked | ((m - n >= window) & (n >= n_sink))
    M = np.zeros((n_q, n_k), dtype=np.float64)
    M[masked] = NEG_INF
    return M


# --------------------------------------------------------------------------
# RoPE
# --------------------------------------------------------------------------
def rope_frequencies(rotary_dims: int, base: float) -> np.ndarray:
    """theta_i = base^(-2i / D_r), i = 0 .. D_r/2 - 1
    ("Transformer架构从Attention到DecoderBlock" §8.2; the exponent starts at 0 as
    in the frequency table of "2.7 Transformer Decoder Block完整解析" §4)."""
    i = np.arange(rotary_dims // 2, dtype=np.float64)
    return np.power(float(base), -2.0 * i / rotary_dims)


def rope_rotate(x, positions, base: float, offset: int = 0, dims: int | None = None,
                pairing: str = "adjacent") -> np.ndarray:
    """Rotate the last axis of x at the given absolute positions.

    positions broadcasts against x.shape[:-1].  Dimensions [offset, offset+dims)
    take part; the rest pass through unchanged (MLA rotates only its last 64
    latent dims).  pairing="adjacent": pair (2i, 2i+1) is rotated by
    pos*theta_i ("Transformer架构从Attention到DecoderBlock" §8.3):
        x'_{2i}   = x_{2i} cos a - x_{2i+1} sin a
        x'_{2i+1} = x_{2i} sin a + x_{2i+1} cos a
    pairing="half": pair (j, j + dims/2) is rotated by pos*theta_j, the form of
    the apply_rope function in "2.7 Transformer Decoder Block完整解析" §4.
    """
    x = _f64(x)
    D = x.shape[-1]
    dims = D - offset if dims is None else dims
    if dims % 2 or offset < 0 or offset + dims > D:
        raise ValueError("rotary span must be even and inside the last axis")
    theta = rope_frequencies(dims, base)
    ang = np.asarray(positions, dtype=np.float64)[..., None] * theta
    c, s = np.cos(ang), np.sin(ang)
    out = x.copy()
    seg = x[..., offset:offset + dims]
    if pairing == "adjacent":
        a, b = seg[..., 0::2], seg[..., 1::2]
        out[..., offset:offset + dims:2] = a * c - b * s
        out[..., offset + 1:offset + dims:2] = a * s + b * c
    elif pairing == "half":
        h = dims // 2
        a, b = seg[..., :h], seg[..., h:]
        out[..., offset:offset + h] = a * c - b * s
        out[..., offset + h:offset + dims] = a * s + b * c
    else:
        raise ValueError(f"unknown pairing {pairing!r}")
    return out


# --------------------------------------------------------------------------
# softmax and one head
# --------------------------------------------------------------------------
def softmax_rows(scores: np.ndarray) -> np.ndarray:
    """Row softmax along the key axis with the row maximum subtracted first
    ("Transformer架构完全深度解析" §5 step 4; "Transformer架构从Attention到DecoderBlock"
    §4.4).  exp(-inf) = 0, so masked keys get weight exactly 0."""
    m = np.max(scores, axis=-1, keepdims=True)
    e = np.exp(scores - m)
    return e / np.sum(e, axis=-1, keepdims=True)


def logsumexp_rows(scores: np.ndarray) -> np.ndarray:
    """log sum_n exp(S[m, n]) per row (the normaliser of softmax_rows)."""
    m = np.max(scores, axis=-1, keepdims=True)
    return (m + np.log(np.sum(np.exp(scores - m), axis=-1, keepdims=True)))[..., 0]


def attention_head(q_rot: np.ndarray, k_rot: np.ndarray, v: np.ndarray, scale: float,
                   mask: np.ndarray | None):
    """One head: A = softmax(scale * Q K^T + M), O = A V.  Returns (O, A, lse)."""
    S = scale * (q_rot @ k_rot.T)
    if mask is not None:
        S = S + mask
    A = softmax_rows(S)
    return A @ v, A, logsumexp_rows(S)


def default_scale(D_h: int, scale: float | None) -> float:
    """scale <= 0 or None selects 1/sqrt(D_h), the per-head dimension
    ("Transformer架构从Attention到DecoderBlock" §4.3)."""
    return 1.0 / math.sqrt(D_h) if (scale is None or scale <= 0) else float(scale)


# --------------------------------------------------------------------------
# prefill
# --------------------------------------------------------------------------
def attention_prefill(q, k, v, *, rope_base: float = 0.0, scale: float | None = None,
                      causal: bool = True, q_offset: int = 0, window: int = 0,
                      n_sink: int = 0, pairing: str = "adjacent", rope_offset: int = 0,
                      rope_dims: int | None = None, return_lse: bool = False):
    """Multi-head causal attention over a whole prompt.

    q [B, S_q, n_h, D_h], k [B, S_k, n_kv, D_h], v [B, S_k, n_kv, D_v] (BSHD, the
    layout the pages' code reaches after .view(batch, seq, heads, d_k)).  Query
    row m sits at position q_offset + m, key row n at position n.  RoPE is
    applied to dims [rope_offset, rope_offset + rope_dims) of q and k (all of
    them by default) when rope_base > 0.  The value head dim D_v may differ
    from D_h (MLA prefill: D_h = 192, D_v = 128).  Returns out [B, S_q, n_h,
    D_v] (float64) and, on request, lse [B, n_h, S_q] (natural log).
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, S_q, n_h, D = q.shape
    S_k, n_kv = k.shape[1], k.shape[2]
    if n_h % n_kv:
        raise ValueError("n_h must be a multiple of n_kv")
    G = n_h // n_kv
    scale = default_scale(D, scale)
    if rope_base > 0:
        q = rope_rotate(q, (q_offset + np.arange(S_q))[None, :, None], rope_base, rope_offset, rope_dims,
                        pairing=pairing)
        k = rope_rotate(k, np.arange(S_k)[None, :, None], rope_base, rope_offset, rope_dims, pairing=pairing)
    mask = None
    if causal or window > 0:
        mask = causal_mask(S_q, S_k, q_offset, window, n_sink)
    out = np.zeros((B, S_q, n_h, v.shape[-1]))
    lse = np.zeros((B, n_h, S_q))
    for b in range(B):
        for h in range(n_h):
            g = h // G
            o, _, l = attention_head(q[b, :, h, :], k[b, :, g, :], v[b, :, g, :], scale, mask)
            out[b, :, h, :] = o
            lse[b, h, :] = l
    return (out, lse) if return_lse else out


def attention_prefill_rows(q, k, v, b: int, h: int, rows, *, rope_base: float = 0.0,
                           scale: float | None = None, causal: bool = True, rope_offset: int = 0,
                           rope_dims: int | None = None):
    """Selected output rows of attention_prefill for one (b, h), computed one
    query at a time so that full-size problems can be sampled.  Returns
    (out [len(rows), D_v], lse [len(rows)])."""
    rows = np.asarray(rows)
    n_h, D = q.shape[2], q.shape[3]
    n_kv = k.shape[2]
    g = h // (n_h // n_kv)
    scale = default_scale(D, scale)
    kk = _f64(k[b, :, g, :])
    vv = _f64(v[b, :, g, :])
    qq = _f64(q[b, rows, h, :])
    if rope_base > 0:
        qq = rope_rotate(qq, rows, rope_base, rope_offset, rope_dims)
        kk = rope_rotate(kk, np.arange(kk.shape[0]), rope_base, rope_offset, rope_dims)
    outs, lses = [], []
    for i, m in enumerate(rows):
        n_vis = int(m) + 1 if causal else kk.shape[0]
        o, _, l = attention_head(qq[i:i + 1], kk[:n_vis], vv[:n_vis], scale, None)
        outs.append(o[0])
        lses.append(l[0])
    return np.stack(outs), np.array(lses)


# --------------------------------------------------------------------------
# decode over a KV cache
# --------------------------------------------------------------------------
def attention_decode(q, kcache, vcache, seqlens, *, rope_base: float = 0.0,
                     rope_offset: int = 0, rope_dims: int | None = None,
                     scale: float | None = None, window: int = 0, n_sink: int = 0,
                     pairing: str = "adjacent", batch_index=None):
    """One new query token per sequence against its cache.

    q [B, n_h, D_qk] un-rotated; kcache [B, L_max, n_kv, D_qk] holding rotated
    keys; vcache [B, L_max, n_kv, D_v]; seqlens[b] keys are valid and already
    include the new token, which therefore sits at position seqlens[b] - 1
    ("Transformer架构完全深度解析" §9: append, then attend).  RoPE (when
    rope_base > 0) rotates dims [rope_offset, rope_offset + rope_dims) of q
    with the given pairing (it must match the one the cache was written with).
    batch_index restricts the work to a subset of sequences.  Returns
    out [B, n_h, D_v] (rows outside batch_index stay 0) and lse [B, n_h].
    """
    q = _f64(q)
    B, n_h, D_qk = q.shape
    n_kv = kcache.shape[2]
    if n_h % n_kv:
        raise ValueError("n_h must be a multiple of n_kv")
    G = n_h // n_kv
    D_v = vcache.shape[-1]
    scale = default_scale(D_qk, scale)
    out = np.zeros((B, n_h, D_v))
    lse = np.zeros((B, n_h))
    todo = range(B) if batch_index is None else batch_index
    for b in todo:
        L = int(seqlens[b])
        if L < 1:
            raise ValueError("every sequence holds at least its new token")
        pos = L - 1
        qb = q[b]
        if rope_base > 0:
            qb = rope_rotate(qb, np.full(n_h, pos), rope_base, rope_offset, rope_dims, pairing=pairing)
        mask = None
        if window > 0:
            mask = causal_mask(1, L, pos, window, n_sink)
        for g in range(n_kv):
            kk = _f64(kcache[b, :L, g, :])
            vv = _f64(vcache[b, :L, g, :])
            # the G query heads of this KV head share K and V; each is one row
            o, _, l = attention_head(qb[g * G:(g + 1) * G], kk, vv, scale, mask)
            out[b, g * G:(g + 1) * G] = o
            lse[b, g * G:(g + 1) * G] = l
    return out, lse


def rope_cache(k, base: float, pairing: str = "adjacent") -> np.ndarray:
    """Rotated keys as a cache stores them: key row n of k [B, S, n_kv, D] is
    rotated at its absolute position n ("Transformer架构完全深度解析" §7)."""
    k = _f64(k)
    return rope_rotate(k, np.arange(k.shape[1])[None, :, None], base, pairing=pairing)


# --------------------------------------------------------------------------
# MLA: the non-absorbed (up-projected) path and the absorption algebra
# --------------------------------------------------------------------------
def mla_decode_unabsorbed(q_c, q_r, c_kv, k_r, w_uk, w_uv, seqlens, scale: float):
    """Multi-head Latent Attention decode without absorption
    ("Transformer 与 LLM" slide 06 diagram).

    q_c [B, n_h, d_c] per-head content query, q_r [B, n_h, d_r] per-head
    rotated query part, c_kv [B, L, d_l] latent cache, k_r [B, L, d_r] rotated
    key part shared by all heads, w_uk / w_uv [n_h, d_l, d_c] up-projections:
    k^C_{n,h} = c_n @ w_uk[h], v_{n,h} = c_n @ w_uv[h].
    score(h, n) = scale * (q_c[h] . k^C_{n,h} + q_r[h] . k_r[n]).
    Returns o [B, n_h, d_c].
    """
    q_c, q_r, c_kv, k_r = _f64(q_c), _f64(q_r), _f64(c_kv), _f64(k_r)
    w_uk, w_uv = _f64(w_uk), _f64(w_uv)
    B, n_h, d_c = q_c.shape
    out = np.zeros((B, n_h, d_c))
    for b in range(B):
        L = int(seqlens[b])
        for h in range(n_h):
            kc = c_kv[b, :L] @ w_uk[h]          # [L, d_c]
            vh = c_kv[b, :L] @ w_uv[h]          # [L, d_c]
            s = scale * (kc @ q_c[b, h] + k_r[b, :L] @ q_r[b, h])
            a = softmax_rows(s[None, :])[0]
            out[b, h] = a @ vh
    return out


def mla_prefill_unabsorbed(q_c, q_r, c_kv, k_r, w_uk, w_uv, *, rope_base: float = 0.0,
                           scale: float | None = None):
    """Multi-head Latent Attention prefill on the non-absorbed path ("Transformer
    与 LLM" slide 06: prefill up-projects instead of absorbing, which would cost
    ~3.4x the attention FLOPs).

    q_c [B, S, n_h, d_c], q_r [B, S, n_h, d_r] (un-rotated), c_kv [B, S, d_l],
    k_r [B, S, d_r] (un-rotated, shared by all heads), w_uk / w_uv [n_h, d_l, d_c].
    Per head h: q = [q_c ; q_r], k = [c_kv @ w_uk[h] ; k_r], v = c_kv @ w_uv[h];
    the d_r dims of q and k are rotated at their positions (decoupled RoPE) when
    rope_base > 0; scale defaults to 1/sqrt(d_c + d_r).  Returns (q, k, v, out):
    the per-head tensors [B, S, n_h, d_c + d_r] / [B, S, n_h, d_c] it built, and
    out [B, S, n_h, d_c] of causal attention over them.
    """
    q_c, q_r, c_kv, k_r = _f64(q_c), _f64(q_r), _f64(c_kv), _f64(k_r)
    w_uk, w_uv = _f64(w_uk), _f64(w_uv)
    n_h, d_c, d_r = q_c.shape[2], q_c.shape[3], q_r.shape[3]
    k_c = np.einsum("bsl,hlc->bshc", c_kv, w_uk)            # [B, S, n_h, d_c]
    v = np.einsum("bsl,hlc->bshc", c_kv, w_uv)
    k_rh = np.broadcast_to(k_r[:, :, None, :], k_r.shape[:2] + (n_h, d_r))
    q = np.concatenate([q_c, q_r], axis=-1)
    k = np.concatenate([k_c, k_rh], axis=-1)
    scale = 1.0 / math.sqrt(d_c + d_r) if scale is None else scale
    out = attention_prefill(q, k, v, rope_base=rope_base, scale=scale, rope_offset=d_c, rope_dims=d_r)
    return q, k, v, out


def mla_absorb_query(q_c, q_r, w_uk) -> np.ndarray:
    """q~_h = [W_UK[h] q_c[h] ; q_r[h]] (d_l + d_r dims): folding W_UK into the
    query lets every head score directly against the cached [c^KV ; k^R]."""
    q_c, q_r, w_uk = _f64(q_c), _f64(q_r), _f64(w_uk)
    absorbed = np.einsum("hlc,bhc->bhl", w_uk, q_c)
    return np.concatenate([absorbed, q_r], axis=-1)


def mla_unabsorb_output(o_latent, w_uv) -> np.ndarray:
    """o_h = W_UV[h]^T applied to the latent output o~_h (d_l -> d_c)."""
    return np.einsum("hlc,bhl->bhc", _f64(w_uv), _f64(o_latent))

"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

This module holds shapes and random draws only - no attention arithmetic - so
that the CUDA library and the fp64 oracle can be fed identical inputs without
sharing any of the method.  Every draw comes from a CPU ``torch.Generator``
seeded explicitly, in a fixed order (Q, K, V; or seqlens, q, K cache, V cache),
as N(0, 1) values in float32 that are then cast to the stated dtype.

The five named configurations stand in for the models the pages discuss; no
dataset is involved:

* ``tiny``        - fp32 causal MHA prefill, B=1 S=16 n_h=n_kv=2 D_h=8, RoPE base 1e4
* ``gpt2``        - GPT-2-small-shaped causal MHA prefill, B=8 S=1024 n_h=n_kv=12 D_h=64, no RoPE
                    ("2.7 Transformer Decoder Block完整解析" §9 model table)
* ``llama3_8b``   - Llama-3-8B-shaped causal GQA prefill, B=4 S=8192 n_h=32 n_kv=8 D_h=128,
                    RoPE base 5e5 ("Transformer架构完全深度解析" §7-§8)
* ``gqa_decode``  - 59 sequences, cached lengths uniform in [4096, 8192], n_h=32 n_kv=8 D_h=128
                    ("Transformer 与 LLM" slide 06: about 59 concurrent 8K sequences fit one card)
* ``mla_decode``  - 32 sequences at 32768 keys, 128 heads sharing one 576-dim latent KV head,
                    V = first 512 latent dims ("Transformer 与 LLM" slide 06)
* ``mla_prefill`` - DeepSeek-V3-shaped MLA prefill on the non-absorbed path: B=1 S=4096,
                    128 heads, q/k head dim 192 (128 content + 64 decoupled RoPE dims,
                    the RoPE part of k shared by all heads), v head dim 128, RoPE base 1e4
                    on dims [128, 192), scale 1/sqrt(192) ("Transformer 与 LLM" slide 06)

The decode caches are drawn directly as the stored (already rotated) keys:
rotating i.i.d. N(0, 1) pairs gives i.i.d. N(0, 1) pairs again, so the draw has
the distribution of a rotated cache.
"""
from __future__ import annotations

import math

import torch

CONFIGS: dict[str, dict] = {
    "tiny": dict(kind="prefill", B=1, S=16, n_h=2, n_kv=2, D_h=8, dtype="f32",
                 rope_base=10000.0, scale=1.0 / math.sqrt(8), causal=True),
    "gpt2": dict(kind="prefill", B=8, S=1024, n_h=12, n_kv=12, D_h=64, dtype="bf16",
                 rope_base=0.0, scale=1.0 / math.sqrt(64), causal=True),
    "llama3_8b": dict(kind="prefill", B=4, S=8192, n_h=32, n_kv=8, D_h=128, dtype="bf16",
                      rope_base=500000.0, scale=1.0 / math.sqrt(128), causal=True),
    "gqa_decode": dict(kind="decode", B=59, max_len=8192, len_lo=4096, len_hi=8192,
                       n_h=32, n_kv=8, D_qk=128, D_v=128, v_aliases_k=False, dtype="bf16",
                       rope_base=500000.0, rope_offset=0, rope_dims=128,
                       scale=1.0 / math.sqrt(128)),
    "mla_decode": dict(kind="decode", B=32, max_len=32768, len_lo=32768, len_hi=32768,
                       n_h=128, n_kv=1, D_qk=576, D_v=512, v_aliases_k=True, dtype="bf16",
                       rope_base=0.0, rope_offset=512, rope_dims=64,
                       scale=1.0 / math.sqrt(192)),
    "mla_prefill": dict(kind="prefill", B=1, S=4096, n_h=128, n_kv=128, D_qk=192, D_v=128, dtype="bf16",
                        rope_base=10000.0, rope_offset=128, rope_dims=64, scale=1.0 / math.sqrt(192),
                        causal=True),
}

TORCH_DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16}


def config(name: str, **overrides) -> dict:
    """A copy of a named configuration with some fields replaced."""
    cfg = dict(CONFIGS[name])
    cfg.update(overrides)
    cfg["name"] = name
    return cfg


def _randn(shape, gen: torch.Generator, dtype: torch.dtype) -> torch.Tensor:
    """N(0, 1) in float32, cast to dtype; drawn in slabs so that a multi-GB
    tensor never needs a second float32 copy."""
    out = torch.empty(shape, dtype=dtype)
    flat = out.view(-1)
    slab = 1 << 26
    for i in range(0, flat.numel(), slab):
        n = min(slab, flat.numel() - i)
        flat[i:i + n] = torch.randn(n, generator=gen, dtype=torch.float32).to(dtype)
    return out


def prefill_inputs(cfg: dict, seed: int = 0):
    """(q, k, v) on the CPU in BSHD layout: q [B,S,n_h,D_h], k, v [B,S,n_kv,D_h]."""
    g = torch.Generator().manual_seed(seed)
    dt = TORCH_DTYPES[cfg["dtype"]]
    B, S, n_h, n_kv, D = cfg["B"], cfg["S"], cfg["n_h"], cfg["n_kv"], cfg["D_h"]
    q = _randn((B, S, n_h, D), g, dt)
    k = _randn((B, S, n_kv, D), g, dt)
    v = _randn((B, S, n_kv, D), g, dt)
    return q, k, v


def mla_prefill_inputs(cfg: dict, seed: int = 0):
    """(q, k, v) on the CPU: q, k [B,S,n_h,D_qk], v [B,S,n_h,D_v].  The last
    rope_dims dims of k are one draw per token copied to every head (the shared
    k^R of MLA); everything else is i.i.d. N(0, 1).  Draw order q, k, k^R, v."""
    g = torch.Generator().manual_seed(seed)
    dt = TORCH_DTYPES[cfg["dtype"]]
    B, S, n_h, D_qk, D_v, r = cfg["B"], cfg["S"], cfg["n_h"], cfg["D_qk"], cfg["D_v"], cfg["rope_dims"]
    q = _randn((B, S, n_h, D_qk), g, dt)
    k = _randn((B, S, n_h, D_qk), g, dt)
    k_r = _randn((B, S, 1, r), g, dt)
    k[..., D_qk - r:] = k_r
    v = _randn((B, S, n_h, D_v), g, dt)
    return q, k, v


def decode_inputs(cfg: dict, seed: int = 0):
    """(q, kcache, vcache, seqlens) on the CPU.

    q [B, n_h, D_qk] (un-rotated new query), kcache [B, max_len, n_kv, D_qk]
    (rotated keys as stored), vcache [B, max_len, n_kv, D_v] or, when the
    configuration says V aliases K (MLA), a view of kcache's first D_v dims.
    seqlens int32 [B], each uniform in [len_lo, len_hi], counts keys including
    the new token.
    """
    g = torch.Generator().manual_seed(seed)
    dt = TORCH_DTYPES[cfg["dtype"]]
    B, L, n_h, n_kv = cfg["B"], cfg["max_len"], cfg["n_h"], cfg["n_kv"]
    D_qk, D_v = cfg["D_qk"], cfg["D_v"]
    seqlens = torch.randint(cfg["len_lo"], cfg["len_hi"] + 1, (B,), generator=g,
                            dtype=torch.int64).to(torch.int32)
    q = _randn((B, n_h, D_qk), g, dt)
    kcache = _randn((B, L, n_kv, D_qk), g, dt)
    if cfg.get("v_aliases_k"):
        vcache = kcache[..., :D_v]
    else:
        vcache = _randn((B, L, n_kv, D_v), g, dt)
    return q, kcache, vcache, seqlens


def mla_factors(B: int, n_h: int, L: int, seed: int = 0, d_c: int = 128, d_r: int = 64,
                d_l: int = 512):
    """Random factors of an MLA layer for the absorbed-vs-unabsorbed check:
    q_c [B,n_h,d_c], q_r [B,n_h,d_r], c_kv [B,L,d_l], k_r [B,L,d_r],
    w_uk, w_uv [n_h,d_l,d_c] (scaled by 1/sqrt(d_l) to keep scores O(1))."""
    g = torch.Generator().manual_seed(seed)
    f = torch.float64
    q_c = torch.randn((B, n_h, d_c), generator=g, dtype=f)
    q_r = torch.randn((B, n_h, d_r), generator=g, dtype=f)
    c_kv = torch.randn((B, L, d_l), generator=g, dtype=f)
    k_r = torch.randn((B, L, d_r), generator=g, dtype=f)
    w_uk = torch.randn((n_h, d_l, d_c), generator=g, dtype=f) / math.sqrt(d_l)
    w_uv = torch.randn((n_h, d_l, d_c), generator=g, dtype=f) / math.sqrt(d_l)
    return q_c, q_r, c_kv, k_r, w_uk, w_uv


def causal_flops(B: int, S: int, n_h: int, D_h: int, D_v: int | None = None) -> float:
    """Causal attention FLOPs as the benchmark counts them: the dense count
    2 * B * n_h * S^2 * (D_h + D_v) (Q K^T plus P V; 4 B n_h S^2 D_h when
    D_v = D_h), halved."""
    D_v = D_h if D_v is None else D_v
    return 2.0 * B * n_h * S * S * (D_h + D_v) / 2.0


def decode_bytes(cfg: dict, seqlens) -> float:
    """Algorithmic KV-cache bytes one decode call must read: every valid key
    row (and value row, unless V aliases K) once, bf16."""
    esize = 2 if cfg["dtype"] == "bf16" else 4
    total_keys = float(sum(int(x) for x in seqlens))
    per_key = cfg["n_kv"] * cfg["D_qk"] * esize
    if not cfg.get("v_aliases_k"):
        per_key += cfg["n_kv"] * cfg["D_v"] * esize
    return total_keys * per_key


def decode_flops(cfg: dict, seqlens) -> float:
    """2 * n_h * (D_qk + D_v) FLOPs per valid key (scores plus weighted sum)."""
    total_keys = float(sum(int(x) for x in seqlens))
    return total_keys * 2.0 * cfg["n_h"] * (cfg["D_qk"] + cfg["D_v"])

"""Chunked prefill over a KV cache and the fused RoPE + KV-cache append.

"Transformer 与 LLM" slide 07: a long prompt is prefilled in chunks so that one
request does not hold the GPU; a chunk's queries sit at positions
q_offset .. q_offset + C - 1 and attend every cached key up to their own
position.  The cache holds rotated keys ("Transformer架构完全深度解析" §7), and
a decode step appends the new token's key and value before attending (§9).
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests.tolerances import BF16_MAX_ABS, assert_parity, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def lib():
    import __graft_entry__
    __graft_entry__.build()
    import transformer_causal_attention_gb300 as attn
    yield attn
    assert attn.device_status() == 0


def make_cache(lib, k, v, max_len, base):
    """Cache [B, max_len, n_kv, D] holding RoPE(k) in its first S rows (written by attn_kv_append)."""
    B, S, n_kv, D = k.shape
    kc = torch.full((B, max_len, n_kv, D), float("nan"), dtype=k.dtype, device=DEV)
    vc = torch.full((B, max_len, n_kv, D), float("nan"), dtype=v.dtype, device=DEV)
    start = torch.zeros(B, dtype=torch.int32, device=DEV)
    lib.kv_append(k.to(DEV), v.to(DEV), kc, vc, start, rope_base=base)
    return kc, vc


@pytest.mark.parametrize("B,S,n_h,n_kv,D,dtype,base", [
    (2, 300, 4, 2, 128, "bf16", 5e5),
    (1, 77, 2, 1, 64, "bf16", 1e4),
    (1, 50, 5, 5, 64, "bf16", 1e4),      # a head count that is not a power of two
    (4, 5000, 8, 8, 128, "bf16", 5e5),   # enough tokens for one thread per (token, chunk) over all heads
    (2, 40, 2, 2, 8, "f32", 1e4),
])
def test_kv_append_writes_rotated_keys(lib, B, S, n_h, n_kv, D, dtype, base):
    cfg = dict(B=B, S=S, n_h=n_h, n_kv=n_kv, D_h=D, dtype=dtype)
    _, k, v = workloads.prefill_inputs(cfg, seed=S)
    kc, vc = make_cache(lib, k, v, S + 16, base)
    want = oracle.rope_cache(k, base)
    if dtype == "f32":
        assert np.max(np.abs(to_np(kc[:, :S]) - want)) <= 1e-5
        assert torch.equal(vc[:, :S].cpu(), v)
    else:
        assert_parity(kc[:, :S], want, "bf16", "appended keys")
        assert torch.equal(vc[:, :S].cpu(), v)
    assert torch.isnan(kc[:, S:]).all()  # slots after the new tokens are untouched


@pytest.mark.parametrize("B,S,split,n_h,n_kv,D,base", [
    (2, 640, 256, 8, 2, 128, 5e5),   # chunk boundary on a tile boundary
    (1, 500, 123, 4, 1, 128, 1e4),   # ragged chunk start, MQA
    (2, 300, 200, 4, 4, 64, 0.0),    # D 64, no RoPE
    (1, 200, 57, 2, 2, 96, 1e4),     # CUDA-core path
])
def test_chunked_prefill_equals_oracle(lib, B, S, split, n_h, n_kv, D, base):
    cfg = dict(B=B, S=S, n_h=n_h, n_kv=n_kv, D_h=D, dtype="bf16")
    q, k, v = workloads.prefill_inputs(cfg, seed=S + split)
    max_len = S + 64
    kc, vc = make_cache(lib, k, v, max_len, base) if base > 0 else (None, None)
    if base <= 0:
        kc = torch.zeros((B, max_len, n_kv, D), dtype=k.dtype, device=DEV)
        vc = torch.zeros((B, max_len, n_kv, D), dtype=v.dtype, device=DEV)
        kc[:, :S] = k.to(DEV)
        vc[:, :S] = v.to(DEV)
    for lo, hi in ((0, split), (split, S)):
        qc = q[:, lo:hi].contiguous()
        out, lse = lib.prefill_chunk(qc.to(DEV), kc, vc, q_offset=lo, rope_base=base, lse=True)
        torch.cuda.synchronize()
        ref, ref_lse = oracle.attention_prefill(qc, k[:, :hi], v[:, :hi], rope_base=base, q_offset=lo,
                                                return_lse=True)
        assert_parity(out, ref, "bf16", f"chunk [{lo},{hi})")
        assert np.max(np.abs(to_np(lse) - ref_lse)) <= BF16_MAX_ABS


def test_chunks_reproduce_the_whole_prompt(lib):
    B, S, n_h, n_kv, D, base = 1, 512, 4, 2, 128, 5e5
    cfg = dict(B=B, S=S, n_h=n_h, n_kv=n_kv, D_h=D, dtype="bf16")
    q, k, v = workloads.prefill_inputs(cfg, seed=4)
    full, _, _ = lib.prefill(q.to(DEV), k.to(DEV), v.to(DEV), rope_base=base)
    kc, vc = make_cache(lib, k, v, S, base)
    parts = []
    for lo in range(0, S, 128):
        out, _ = lib.prefill_chunk(q[:, lo:lo + 128].contiguous().to(DEV), kc, vc, q_offset=lo, rope_base=base)
        parts.append(out)
    torch.cuda.synchronize()
    assert_parity(torch.cat(parts, dim=1), to_np(full), "bf16", "chunked vs whole")


def test_append_then_decode_matches_prefill_last_row(lib):
    # one decode step as the pages describe it: append the new token's k, v, then attend
    B, S, n_h, n_kv, D, base = 3, 200, 8, 2, 128, 5e5
    cfg = dict(B=B, S=S, n_h=n_h, n_kv=n_kv, D_h=D, dtype="bf16")
    q, k, v = workloads.prefill_inputs(cfg, seed=6)
    kc, vc = make_cache(lib, k[:, :S - 1], v[:, :S - 1], S + 8, base)
    start = torch.full((B,), S - 1, dtype=torch.int32, device=DEV)
    lib.kv_append(k[:, S - 1:].contiguous().to(DEV), v[:, S - 1:].contiguous().to(DEV), kc, vc, start,
                  rope_base=base)
    seqlens = torch.full((B,), S, dtype=torch.int32, device=DEV)
    out, _ = lib.decode(q[:, S - 1].contiguous().to(DEV), kc, vc, seqlens, rope_base=base)
    torch.cuda.synchronize()
    ref = oracle.attention_prefill(q, k, v, rope_base=base)[:, S - 1]
    assert_parity(out, ref, "bf16", "append + decode")


@pytest.mark.parametrize("B,S,n_h,n_kv,D,window,sink,dtype", [
    (1, 700, 4, 2, 128, 256, 4, "bf16"),    # window of 2 key tiles, 4 sinks (tensor cores)
    (2, 520, 2, 1, 64, 300, 0, "bf16"),     # unaligned window, no sinks: rows whose first tile is all masked
    (1, 400, 2, 2, 128, 1000, 4, "bf16"),   # window longer than the prompt: plain causal
    (1, 2048, 4, 2, 128, 1024, 4, "bf16"),  # long enough for the issuer's steady loop after a sink tile
    (1, 1536, 2, 1, 64, 512, 130, "bf16"),  # two sink tiles, then the steady loop
    (1, 333, 2, 2, 96, 100, 7, "bf16"),     # CUDA-core path
    (1, 90, 2, 2, 16, 20, 3, "f32"),
])
def test_sliding_window_with_sinks(lib, B, S, n_h, n_kv, D, window, sink, dtype):
    cfg = dict(B=B, S=S, n_h=n_h, n_kv=n_kv, D_h=D, dtype=dtype)
    q, k, v = workloads.prefill_inputs(cfg, seed=window + sink)
    out, _, lse = lib.prefill_window(q.to(DEV), k.to(DEV), v.to(DEV), window=window, n_sink=sink, rope_base=1e4,
                                     lse=True)
    torch.cuda.synchronize()
    ref, ref_lse = oracle.attention_prefill(q, k, v, rope_base=1e4, window=window, n_sink=sink, return_lse=True)
    if dtype == "f32":
        assert np.max(np.abs(to_np(out) - ref)) <= 1e-4
    else:
        assert_parity(out, ref, "bf16", f"window {window} sinks {sink}")
        assert np.max(np.abs(to_np(lse) - ref_lse)) <= BF16_MAX_ABS

"""The split-halves RoPE layout (ATTN_ROPE_HALF) through every kernel that rotates.

"2.7 Transformer Decoder Block完整解析" §4 pairs dimension j with j + D/2 (its
apply_rope code) where "Transformer架构从Attention到DecoderBlock" §8.3 pairs
(2i, 2i+1); §8.1 of the latter allows either as long as training and
inference agree.  Each test runs one entry point with pairing="half" against
the oracle's half-split rotation: the RoPE pass (also at per-row positions,
attn_rope_at, in both pairings), the KV-cache append, the
tensor-core and CUDA-core prefill, chunked prefill over a half-split cache, and
the streaming, generic and MLA decode kernels.
"""
import math

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


@pytest.mark.parametrize("D,off,dims,dtype,pos0", [
    (128, 0, 128, "bf16", 0),
    (128, 64, 64, "bf16", 1000),   # rotate only the second half of the head
    (576, 512, 64, "bf16", 7),     # the MLA layout: RoPE on the last 64 latent dims
    (12, 4, 8, "f32", 3),
])
def test_rope_pass_half_split(lib, D, off, dims, dtype, pos0):
    cfg = dict(B=2, S=37, n_h=3, n_kv=3, D_h=D, dtype=dtype)
    x, _, _ = workloads.prefill_inputs(cfg, seed=D + off)
    y = lib.rope(x.to(DEV), rope_base=1e4, rope_offset=off, rope_dims=dims, pos_offset=pos0, pairing="half")
    torch.cuda.synchronize()
    pos = (pos0 + np.arange(x.shape[1]))[None, :, None]
    want = oracle.rope_rotate(x, pos, 1e4, offset=off, dims=dims, pairing="half")
    if dtype == "f32":
        assert np.max(np.abs(to_np(y) - want)) <= 1e-5
    else:
        assert_parity(y, want, "bf16", "rope half")
    assert torch.equal(y[..., :off].cpu(), x[..., :off])  # dims before the span are copied


@pytest.mark.parametrize("pairing,D,off,dims,dtype", [
    ("adjacent", 128, 0, 128, "bf16"),
    ("half", 128, 0, 128, "bf16"),
    ("adjacent", 576, 512, 64, "bf16"),  # the MLA layout: only the last 64 latent dims turn
    ("adjacent", 12, 4, 8, "f32"),
])
def test_rope_at_per_row_positions(lib, pairing, D, off, dims, dtype):
    # every row at its own absolute position (requests at different depths, tokens scattered in a
    # cache): attn_rope_at against the oracle's rotation at the same positions
    cfg = dict(B=3, S=29, n_h=4, n_kv=4, D_h=D, dtype=dtype)
    x, _, _ = workloads.prefill_inputs(cfg, seed=D + dims)
    g = torch.Generator().manual_seed(11)
    pos = torch.randint(0, 1 << 20, (cfg["B"], cfg["S"]), generator=g, dtype=torch.int64).to(torch.int32)
    pos[0, :4] = torch.tensor([0, 1, 8191, (1 << 24) - 1], dtype=torch.int32)
    y = lib.rope(x.to(DEV), rope_base=5e5, rope_offset=off, rope_dims=dims, positions=pos.to(DEV), pairing=pairing)
    torch.cuda.synchronize()
    want = oracle.rope_rotate(x, pos.numpy()[:, :, None], 5e5, offset=off, dims=dims, pairing=pairing)
    if dtype == "f32":
        assert np.max(np.abs(to_np(y) - want)) <= 1e-5
    else:
        assert_parity(y, want, "bf16", "rope at per-row positions")
    # in place, and equal to attn_rope where the positions are consecutive
    xd = x.to(DEV)
    seq = (7 + torch.arange(cfg["S"], dtype=torch.int32)).repeat(cfg["B"], 1).to(DEV)
    a = lib.rope(xd, rope_base=5e5, rope_offset=off, rope_dims=dims, pos_offset=7, pairing=pairing)
    lib.rope(xd, rope_base=5e5, rope_offset=off, rope_dims=dims, positions=seq, out=xd, pairing=pairing)
    torch.cuda.synchronize()
    assert torch.equal(a, xd)


@pytest.mark.parametrize("B,S,n_h,n_kv,D,dtype", [
    (2, 300, 8, 2, 128, "bf16"),   # tensor cores, D 128
    (1, 200, 4, 4, 64, "bf16"),    # tensor cores, D 64
    (1, 150, 4, 2, 96, "bf16"),    # CUDA-core path
    (1, 40, 2, 1, 12, "f32"),
])
def test_prefill_half_split(lib, B, S, n_h, n_kv, D, dtype):
    cfg = dict(B=B, S=S, n_h=n_h, n_kv=n_kv, D_h=D, dtype=dtype)
    q, k, v = workloads.prefill_inputs(cfg, seed=S + D)
    out, k_rot, lse = lib.prefill(q.to(DEV), k.to(DEV), v.to(DEV), rope_base=5e5, lse=True, pairing="half")
    torch.cuda.synchronize()
    ref, ref_lse = oracle.attention_prefill(q, k, v, rope_base=5e5, pairing="half", return_lse=True)
    kwant = oracle.rope_cache(k, 5e5, pairing="half")
    if dtype == "f32":
        assert np.max(np.abs(to_np(out) - ref)) <= 1e-4
        assert np.max(np.abs(to_np(k_rot) - kwant)) <= 1e-5
    else:
        assert_parity(out, ref, "bf16", "prefill half")
        assert_parity(k_rot, kwant, "bf16", "rotated keys half")
        assert np.max(np.abs(to_np(lse) - ref_lse)) <= BF16_MAX_ABS
    # and the two layouts really differ on these inputs
    adj = oracle.attention_prefill(q, k, v, rope_base=5e5)
    assert np.max(np.abs(to_np(out) - adj)) > 0.05


def test_chunked_prefill_over_half_split_cache(lib):
    B, S, split, n_h, n_kv, D, base = 2, 400, 170, 8, 2, 128, 5e5
    cfg = dict(B=B, S=S, n_h=n_h, n_kv=n_kv, D_h=D, dtype="bf16")
    q, k, v = workloads.prefill_inputs(cfg, seed=12)
    kc = torch.zeros((B, S + 16, n_kv, D), dtype=k.dtype, device=DEV)
    vc = torch.zeros_like(kc)
    start = torch.zeros(B, dtype=torch.int32, device=DEV)
    lib.kv_append(k.to(DEV), v.to(DEV), kc, vc, start, rope_base=base, pairing="half")
    torch.cuda.synchronize()
    assert_parity(kc[:, :S], oracle.rope_cache(k, base, pairing="half"), "bf16", "appended keys half")
    for lo, hi in ((0, split), (split, S)):
        qc = q[:, lo:hi].contiguous()
        out, _ = lib.prefill_chunk(qc.to(DEV), kc, vc, q_offset=lo, rope_base=base, pairing="half")
        torch.cuda.synchronize()
        ref = oracle.attention_prefill(qc, k[:, :hi], v[:, :hi], rope_base=base, q_offset=lo, pairing="half")
        assert_parity(out, ref, "bf16", f"chunk [{lo},{hi}) half")


@pytest.mark.parametrize("B,n_h,n_kv,Dqk,Dv,L,roff,rdims,alias,dtype", [
    (4, 32, 8, 128, 128, 700, 0, 128, False, "bf16"),    # streaming GQA kernel
    (3, 32, 8, 128, 128, 500, 64, 64, False, "bf16"),    # streaming kernel, partial span
    (3, 8, 8, 64, 64, 300, 0, 64, False, "bf16"),        # generic kernel
    (2, 4, 2, 16, 16, 90, 4, 8, False, "f32"),
    (3, 128, 1, 576, 512, 200, 512, 64, True, "bf16"),   # tensor-core MLA kernel
    (2, 16, 1, 576, 512, 150, 512, 64, True, "bf16"),    # MLA layout, generic kernel
])
def test_decode_half_split(lib, B, n_h, n_kv, Dqk, Dv, L, roff, rdims, alias, dtype):
    cfg = dict(B=B, n_h=n_h, n_kv=n_kv, D_qk=Dqk, D_v=Dv, max_len=L, len_lo=1, len_hi=L,
               v_aliases_k=alias, dtype=dtype)
    scale = 1 / math.sqrt(192) if alias else 0.0
    q, kc, vc, sl = workloads.decode_inputs(cfg, seed=L + roff)
    sl[0] = 1
    sl[-1] = L
    kd = kc.to(DEV)
    vd = kd[..., :Dv] if alias else vc.to(DEV)
    out, lse = lib.decode(q.to(DEV), kd, vd, sl.to(DEV), rope_base=1e4, rope_offset=roff, rope_dims=rdims,
                          scale=scale, lse=True, pairing="half")
    torch.cuda.synchronize()
    ref, ref_lse = oracle.attention_decode(q, kc, vc, sl.numpy(), rope_base=1e4, rope_offset=roff,
                                           rope_dims=rdims, scale=scale if scale else None, pairing="half")
    assert_parity(out, ref, dtype, "decode half")
    assert np.max(np.abs(to_np(lse) - ref_lse)) <= (1e-4 if dtype == "f32" else BF16_MAX_ABS)

"""MLA prefill on the non-absorbed path (attn_prefill_mla) against the fp64 oracle.

"Transformer 与 LLM" slide 06: prefill scores q . [k^C ; k^R] / sqrt(192) per
head, with 128 content dims, 64 decoupled RoPE dims whose key part all heads
share, and 128-dim values.  (D_qk, D_v) = (192, 128) runs on the CTA-pair
tensor-core kernel (work items of four 128-row Q tiles), (128, 128) on the
single-CTA one, every other size on the CUDA-core kernel.  Cases cover tiles plus
a ragged tail, items whose later tiles lie past the prompt, a single token, GQA
sharing, both RoPE pairings, no RoPE, the unmasked form, and the full
DeepSeek-V3-shaped configuration at the edge rows of every Q tile of every head.
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


CASES = [
    # B, S, n_h, n_kv, D_qk, D_v, rope_base, rope_offset, rope_dims, causal, pairing, dtype
    (1, 300, 4, 4, 192, 128, 1e4, 128, 64, True, "adjacent", "bf16"),    # tensor cores, ragged tail
    (1, 1, 2, 2, 192, 128, 1e4, 128, 64, True, "adjacent", "bf16"),      # one token: three empty Q tiles
    (1, 64, 2, 1, 192, 128, 1e4, 128, 64, True, "half", "bf16"),         # one partial tile
    (1, 513, 3, 3, 192, 128, 1e4, 128, 64, True, "adjacent", "bf16"),    # a second item of one row
    (2, 1100, 3, 1, 192, 128, 1e4, 128, 64, True, "adjacent", "bf16"),   # several items per pair, MQA
    (2, 257, 4, 2, 192, 128, 1e4, 128, 64, True, "half", "bf16"),        # GQA groups, split halves
    (1, 200, 2, 2, 192, 128, 0.0, 128, 64, True, "adjacent", "bf16"),    # no RoPE
    (1, 190, 2, 1, 192, 128, 1e4, 128, 64, False, "adjacent", "bf16"),   # no mask
    (1, 260, 2, 2, 128, 128, 5e5, 64, 64, True, "adjacent", "bf16"),     # D 128 with a RoPE span
    (1, 150, 2, 2, 96, 64, 1e4, 64, 32, True, "adjacent", "bf16"),       # CUDA cores
    (1, 70, 2, 1, 24, 16, 1e4, 16, 8, True, "half", "f32"),              # CUDA cores, fp32
]


@pytest.mark.parametrize("B,S,n_h,n_kv,Dqk,Dv,base,roff,rdims,causal,pairing,dtype", CASES)
def test_prefill_mla_small(lib, B, S, n_h, n_kv, Dqk, Dv, base, roff, rdims, causal, pairing, dtype):
    g = torch.Generator().manual_seed(S + Dqk)
    dt = workloads.TORCH_DTYPES[dtype]
    q = torch.randn((B, S, n_h, Dqk), generator=g).to(dt)
    k = torch.randn((B, S, n_kv, Dqk), generator=g).to(dt)
    v = torch.randn((B, S, n_kv, Dv), generator=g).to(dt)
    scale = 1.0 / np.sqrt(Dqk)
    out, k_rot, lse = lib.prefill_mla(q.to(DEV), k.to(DEV), v.to(DEV), rope_base=base, rope_offset=roff,
                                      rope_dims=rdims, causal=causal, lse=True, pairing=pairing)
    torch.cuda.synchronize()
    ref, ref_lse = oracle.attention_prefill(q, k, v, rope_base=base, scale=scale, causal=causal,
                                            rope_offset=roff, rope_dims=rdims, pairing=pairing, return_lse=True)
    assert out.shape == (B, S, n_h, Dv)
    if dtype == "f32":
        assert np.max(np.abs(to_np(out) - ref)) <= 1e-4
        assert np.max(np.abs(to_np(lse) - ref_lse)) <= 1e-4
    else:
        assert_parity(out, ref, "bf16", "prefill_mla")
        assert np.max(np.abs(to_np(lse) - ref_lse)) <= BF16_MAX_ABS
    if base > 0:
        kwant = oracle.rope_rotate(k, np.arange(S)[None, :, None], base, roff, rdims, pairing=pairing)
        assert_parity(k_rot, kwant, dtype if dtype == "bf16" else "f32", "rotated keys")
        assert torch.equal(k_rot[..., :roff].cpu(), k[..., :roff])   # the content dims pass through


def test_mla_prefill_from_latent_factors(lib):
    # q, k, v built by the oracle's up-projection of random MLA factors (shared k^R,
    # per-head k^C and v), rounded to bf16, then attended on the GPU
    B, S, n_h, d_c, d_r, d_l = 1, 200, 4, 128, 64, 512
    g = torch.Generator().manual_seed(9)
    f = torch.float64
    q_c = torch.randn((B, S, n_h, d_c), generator=g, dtype=f)
    q_r = torch.randn((B, S, n_h, d_r), generator=g, dtype=f)
    c_kv = torch.randn((B, S, d_l), generator=g, dtype=f)
    k_r = torch.randn((B, S, d_r), generator=g, dtype=f)
    w_uk = torch.randn((n_h, d_l, d_c), generator=g, dtype=f) / np.sqrt(d_l)
    w_uv = torch.randn((n_h, d_l, d_c), generator=g, dtype=f) / np.sqrt(d_l)
    q, k, v, _ = oracle.mla_prefill_unabsorbed(q_c, q_r, c_kv, k_r, w_uk, w_uv, rope_base=1e4)
    qb, kb, vb = (torch.from_numpy(np.ascontiguousarray(x)).to(torch.bfloat16) for x in (q, k, v))
    out, _, _ = lib.prefill_mla(qb.to(DEV), kb.to(DEV), vb.to(DEV), rope_base=1e4, rope_offset=d_c, rope_dims=d_r)
    torch.cuda.synchronize()
    ref = oracle.attention_prefill(qb, kb, vb, rope_base=1e4, scale=1 / np.sqrt(d_c + d_r), rope_offset=d_c,
                                   rope_dims=d_r)
    assert_parity(out, ref, "bf16", "MLA prefill from factors")


def tile_edge_rows(S, tile=128):
    """First and last row of every 128-row query tile."""
    return np.array(sorted({r for t0 in range(0, S, tile) for r in (t0, min(t0 + tile, S) - 1)}))


def check_every_slice(q, k, v, cfg, out, lse, what):
    out_c, lse_c = out.cpu(), lse.cpu()
    rows = tile_edge_rows(cfg["S"])
    got, want, worst_lse = [], [], 0.0
    for b in range(cfg["B"]):
        for h in range(cfg["n_h"]):
            ref, ref_lse = oracle.attention_prefill_rows(q, k, v, b, h, rows, rope_base=cfg["rope_base"],
                                                         scale=cfg["scale"], rope_offset=cfg["rope_offset"],
                                                         rope_dims=cfg["rope_dims"])
            got.append(to_np(out_c[b, rows, h]))
            want.append(ref)
            worst_lse = max(worst_lse, float(np.max(np.abs(to_np(lse_c[b, h, rows]) - ref_lse))))
    assert worst_lse <= BF16_MAX_ABS, f"lse max-abs {worst_lse}"
    assert_parity(np.concatenate(got), np.concatenate(want), "bf16", what)


def test_mla_prefill_config_every_slice(lib):
    # the benchmark's launch (B=1 S=4096, 128 heads: 1024 items of four Q tiles over the CTA pairs);
    # every head at the first and last row of each of its Q tiles, so an item computed for the wrong
    # head or tile, or a pair tile whose CTA 1 half went astray, cannot pass
    cfg = workloads.config("mla_prefill")
    q, k, v = workloads.mla_prefill_inputs(cfg, seed=0)
    out, _, lse = lib.prefill_mla(q.to(DEV), k.to(DEV), v.to(DEV), rope_base=cfg["rope_base"],
                                  rope_offset=cfg["rope_offset"], rope_dims=cfg["rope_dims"], scale=cfg["scale"],
                                  lse=True)
    torch.cuda.synchronize()
    assert bool(torch.isfinite(out).all())
    check_every_slice(q, k, v, cfg, out, lse, "mla prefill, every slice")


def test_mla_prefill_batch_every_slice(lib):
    # 2 sequences x 128 heads x 2048 keys (K/V 335 MB, over twice the L2): 512 items dealt over the
    # pairs in heaviest-first waves; every item of both sequences must be computed once
    cfg = workloads.config("mla_prefill", B=2, S=2048)
    q, k, v = workloads.mla_prefill_inputs(cfg, seed=5)
    out, _, lse = lib.prefill_mla(q.to(DEV), k.to(DEV), v.to(DEV), rope_base=cfg["rope_base"],
                                  rope_offset=cfg["rope_offset"], rope_dims=cfg["rope_dims"], scale=cfg["scale"],
                                  lse=True)
    torch.cuda.synchronize()
    assert bool(torch.isfinite(out).all())
    check_every_slice(q, k, v, cfg, out, lse, "mla prefill over a batch, every slice")

"""Prefill parity: the CUDA library (through the C ABI) against the fp64 oracle.

Covers the tiny fp32 configuration, the GPT-2-shaped configuration in full,
the Llama-3-8B-shaped configuration at full size on the edge rows of every
query tile of every (batch, head) slice (in the launch configuration the
benchmark times), and small cases that span several tiles,
a ragged tail, S = 1, MQA, non-causal masking, the CUDA-core path for other
head sizes, the online-softmax rescale branch and causality.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests.tolerances import BF16_MAX_ABS, assert_parity, errors, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def lib():
    import __graft_entry__
    __graft_entry__.build()
    import transformer_causal_attention_gb300 as attn
    yield attn
    assert attn.device_status() == 0


def gpu_prefill(attn, cfg, q, k, v):
    out, krot, lse = attn.prefill(q.to(DEV), k.to(DEV), v.to(DEV), rope_base=cfg["rope_base"],
                                  scale=cfg["scale"], causal=cfg.get("causal", True), lse=True)
    torch.cuda.synchronize()
    return out, krot, lse


def test_tiny_config(lib):
    cfg = workloads.config("tiny")
    q, k, v = workloads.prefill_inputs(cfg, seed=0)
    out, krot, lse = gpu_prefill(lib, cfg, q, k, v)
    ref, ref_lse = oracle.attention_prefill(q, k, v, rope_base=cfg["rope_base"], scale=cfg["scale"],
                                            return_lse=True)
    assert_parity(out, ref, "f32", "tiny out")
    assert np.max(np.abs(to_np(lse) - ref_lse)) <= 1e-4
    assert np.max(np.abs(to_np(krot) - oracle.rope_cache(k, cfg["rope_base"]))) <= 1e-5


CASES = [
    # B, S, n_h, n_kv, D, rope_base, causal
    (1, 300, 4, 2, 128, 5e5, True),    # tensor cores, GQA, ragged tail (3 tiles)
    (2, 256, 2, 2, 64, 0.0, True),     # tensor cores D=64, exact tile pair
    (1, 77, 4, 1, 128, 1e4, True),     # MQA, one partial tile
    (1, 1, 2, 1, 64, 1e4, True),       # a single token
    (1, 200, 2, 2, 128, 1e4, False),   # no mask, ragged key tile
    (1, 520, 8, 2, 64, 1e4, True),     # five tiles: an odd last pair
    (2, 1024, 4, 4, 128, 1e4, True),   # eight tiles per head
    (1, 130, 2, 2, 96, 1e4, True),     # CUDA-core path (D_h 96)
    (1, 64, 2, 1, 256, 1e4, True),     # CUDA-core path (D_h 256)
    (1, 384, 6, 2, 128, 1e4, True),    # GQA groups of 3: items of two adjacent Q tiles
    (2, 640, 8, 4, 128, 5e5, True),    # GQA groups of 2 over a batch: items of one Q tile of two heads
    (1, 333, 4, 2, 128, 1e4, False),   # GQA head-pair items without the mask, ragged tail
    (4, 1000, 24, 24, 64, 0.0, True),  # fewer than four items per CTA: dealt by a host-computed table
    (3, 1100, 32, 32, 64, 1e4, True),  # the same with RoPE; the table leaves four CTAs without items
]


@pytest.mark.parametrize("B,S,n_h,n_kv,D,rope,causal", CASES)
def test_bf16_prefill_cases(lib, B, S, n_h, n_kv, D, rope, causal):
    cfg = dict(B=B, S=S, n_h=n_h, n_kv=n_kv, D_h=D, dtype="bf16", rope_base=rope, scale=0.0, causal=causal)
    q, k, v = workloads.prefill_inputs(cfg, seed=S + D)
    out, krot, lse = gpu_prefill(lib, cfg, q, k, v)
    ref, ref_lse = oracle.attention_prefill(q, k, v, rope_base=rope, causal=causal, return_lse=True)
    assert_parity(out, ref, "bf16", f"out {cfg}")
    assert np.max(np.abs(to_np(lse) - ref_lse)) <= BF16_MAX_ABS
    if rope > 0:
        assert_parity(krot, oracle.rope_cache(k, rope), "bf16", "k_rot")


def test_gpt2_config_full(lib):
    cfg = workloads.config("gpt2")
    q, k, v = workloads.prefill_inputs(cfg, seed=0)
    out, _, lse = gpu_prefill(lib, cfg, q, k, v)
    ref, ref_lse = oracle.attention_prefill(q, k, v, rope_base=0.0, scale=cfg["scale"], return_lse=True)
    assert_parity(out, ref, "bf16", "gpt2")
    assert np.max(np.abs(to_np(lse) - ref_lse)) <= BF16_MAX_ABS


def tile_edge_rows(S, tile=128):
    """First and last row of every 128-row query tile (the rows a work item starts and ends on)."""
    rows = set()
    for t0 in range(0, S, tile):
        rows.update((t0, min(t0 + tile, S) - 1))
    return sorted(rows)


def test_llama_config_every_slice(lib):
    # the benchmark's launch: B=4 x 32 heads x 32 tile pairs dealt in waves over the persistent CTAs;
    # every (b, h) slice is checked at the first and last row of each of its Q tiles, so an item
    # computed for the wrong slice or tile (or not at all) cannot pass
    cfg = workloads.config("llama3_8b")
    q, k, v = workloads.prefill_inputs(cfg, seed=0)
    out, krot, lse = gpu_prefill(lib, cfg, q, k, v)
    out_c, krot_c, lse_c = out.cpu(), krot.cpu(), lse.cpu()
    del out, krot, lse
    rows = tile_edge_rows(cfg["S"])
    got, want, worst_lse = [], [], 0.0
    for b in range(cfg["B"]):
        for h in range(cfg["n_h"]):
            ref, ref_lse = oracle.attention_prefill_rows(q, k, v, b, h, rows, rope_base=cfg["rope_base"],
                                                         scale=cfg["scale"])
            got.append(to_np(out_c[b, rows, h]))
            want.append(ref)
            worst_lse = max(worst_lse, float(np.max(np.abs(to_np(lse_c[b, h, rows]) - ref_lse))))
    assert worst_lse <= BF16_MAX_ABS, f"lse max-abs {worst_lse}"
    assert_parity(np.concatenate(got), np.concatenate(want), "bf16", "llama every slice")
    # the whole rotated-key tensor the prefill writes (the cache a decode reads)
    for b in range(cfg["B"]):
        assert_parity(krot_c[b], oracle.rope_cache(k[b:b + 1], cfg["rope_base"])[0], "bf16", f"llama k_rot b={b}")


def test_folded_dealing_d128_every_slice(lib):
    # K/V of 3 x 24 heads x 8192 keys (302 MB) is over twice the L2 and there are more than four
    # waves of double items, so the D = 128 kernel deals (heavy, light) tile pairs of one head
    # together; every slice at every Q tile's first and last row must match the oracle
    cfg = dict(B=3, S=8192, n_h=24, n_kv=24, D_h=128, dtype="bf16", rope_base=5e5, scale=0.0)
    q, k, v = workloads.prefill_inputs(cfg, seed=21)
    out, _, lse = gpu_prefill(lib, cfg, q, k, v)
    out_c, lse_c = out.cpu(), lse.cpu()
    del out, lse
    rows = tile_edge_rows(cfg["S"])
    got, want, worst_lse = [], [], 0.0
    for b in range(cfg["B"]):
        for h in range(cfg["n_h"]):
            ref, ref_lse = oracle.attention_prefill_rows(q, k, v, b, h, rows, rope_base=cfg["rope_base"],
                                                         scale=None)
            got.append(to_np(out_c[b, rows, h]))
            want.append(ref)
            worst_lse = max(worst_lse, float(np.max(np.abs(to_np(lse_c[b, h, rows]) - ref_lse))))
    assert worst_lse <= BF16_MAX_ABS, f"lse max-abs {worst_lse}"
    assert_parity(np.concatenate(got), np.concatenate(want), "bf16", "folded D=128 prefill, every slice")


def test_online_softmax_rescale_branch(lib):
    # scores grow by ~17 (log2 units) from one key tile to the next, so the
    # running maximum moves past the lazy-rescale threshold on every tile
    S, D = 640, 64
    q = torch.zeros(1, S, 1, D)
    k = torch.zeros(1, S, 1, D)
    q[..., 0] = 4.0
    k[0, :, 0, 0] = 3.0 * (torch.arange(S) // 128).float()
    v = torch.randn(1, S, 1, D, generator=torch.Generator().manual_seed(5))
    q, k, v = q.bfloat16(), k.bfloat16(), v.bfloat16()
    cfg = dict(rope_base=0.0, scale=1.0)
    out, _, _ = gpu_prefill(lib, cfg, q, k, v)
    ref = oracle.attention_prefill(q, k, v, scale=1.0)
    assert_parity(out, ref, "bf16", "rescale")


def test_causality_future_perturbation_leaves_past_bit_identical(lib):
    cfg = dict(B=1, S=384, n_h=4, n_kv=2, D_h=128, dtype="bf16", rope_base=1e4, scale=0.0)
    q, k, v = workloads.prefill_inputs(cfg, seed=9)
    out, _, _ = gpu_prefill(lib, cfg, q, k, v)
    m = 200
    q2, k2, v2 = q.clone(), k.clone(), v.clone()
    q2[:, m + 1:] = -q2[:, m + 1:]
    k2[:, m + 1:] += 1.0
    v2[:, m + 1:] *= 3.0
    out2, _, _ = gpu_prefill(lib, cfg, q2, k2, v2)
    assert torch.equal(out[:, :m + 1], out2[:, :m + 1])
    assert not torch.equal(out[:, m + 1:], out2[:, m + 1:])


def test_outputs_are_deterministic(lib):
    cfg = dict(B=1, S=512, n_h=4, n_kv=1, D_h=128, dtype="bf16", rope_base=5e5, scale=0.0)
    q, k, v = workloads.prefill_inputs(cfg, seed=3)
    a, _, _ = gpu_prefill(lib, cfg, q, k, v)
    b, _, _ = gpu_prefill(lib, cfg, q, k, v)
    assert torch.equal(a, b)

"""Long-context parity: 131072 positions (a 128K context) through the C ABI against the fp64 oracle.

At this length the Q rotation's angles reach pos * theta_0 = 131071 rad, so the prefill's reduction
of the angle to a fraction of a turn must keep its precision ("Transformer架构完全深度解析" §7: the
rotation of a token depends on its absolute position); a Q tile near the end walks 1024 key tiles;
and a decode over one sequence splits 131072 keys over every SM.  Rows are sampled (the oracle is
O(S) per row); the rotated keys are compared whole.
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
S_LONG = 131072


@pytest.fixture(scope="module", autouse=True)
def lib():
    import __graft_entry__
    __graft_entry__.build()
    import transformer_causal_attention_gb300 as attn
    yield attn
    assert attn.device_status() == 0


def sampled_rows(S, tile=128, n_random=12, seed=0):
    """First and last row of the first three, the middle two and the last two Q tiles, and of a
    few tiles drawn at random."""
    n_t = (S + tile - 1) // tile
    tiles = {0, 1, 2, n_t // 2 - 1, n_t // 2, n_t - 2, n_t - 1}
    tiles.update(np.random.default_rng(seed).integers(0, n_t, n_random).tolist())
    rows = set()
    for t in tiles:
        rows.update((t * tile, min(t * tile + tile, S) - 1))
    return sorted(rows)


def test_prefill_128k_positions(lib):
    # GQA groups of 4 (head-pair work items), RoPE base 5e5 as for Llama 3
    cfg = dict(B=1, S=S_LONG, n_h=4, n_kv=1, D_h=128, dtype="bf16", rope_base=5e5, scale=0.0)
    q, k, v = workloads.prefill_inputs(cfg, seed=128)
    out, krot, lse = lib.prefill(q.to(DEV), k.to(DEV), v.to(DEV), rope_base=cfg["rope_base"], lse=True)
    torch.cuda.synchronize()
    out_c, krot_c, lse_c = out.cpu(), krot.cpu(), lse.cpu()
    del out, krot, lse
    rows = sampled_rows(S_LONG)
    got, want, worst_lse = [], [], 0.0
    for h in range(cfg["n_h"]):
        ref, ref_lse = oracle.attention_prefill_rows(q, k, v, 0, h, rows, rope_base=cfg["rope_base"])
        got.append(to_np(out_c[0, rows, h]))
        want.append(ref)
        worst_lse = max(worst_lse, float(np.max(np.abs(to_np(lse_c[0, h, rows]) - ref_lse))))
    assert worst_lse <= BF16_MAX_ABS, f"lse max-abs {worst_lse}"
    assert_parity(np.concatenate(got), np.concatenate(want), "bf16", "prefill at 128K positions")
    assert_parity(krot_c, oracle.rope_cache(k, cfg["rope_base"]), "bf16", "k_rot at 128K positions")


def test_prefill_128k_positions_theta0_one(lib):
    # RoPE base 1e4 on a 64-dim head: the slowest pair turns by 1e4^(-62/64) rad per position and
    # the fastest by 1 rad, so both extremes of the angle range are exercised at 131071
    cfg = dict(B=1, S=S_LONG, n_h=2, n_kv=2, D_h=64, dtype="bf16", rope_base=1e4, scale=0.0)
    q, k, v = workloads.prefill_inputs(cfg, seed=64)
    out, krot, lse = lib.prefill(q.to(DEV), k.to(DEV), v.to(DEV), rope_base=cfg["rope_base"], lse=True)
    torch.cuda.synchronize()
    out_c, krot_c, lse_c = out.cpu(), krot.cpu(), lse.cpu()
    del out, krot, lse
    rows = sampled_rows(S_LONG, seed=1)
    for h in range(cfg["n_h"]):
        ref, ref_lse = oracle.attention_prefill_rows(q, k, v, 0, h, rows, rope_base=cfg["rope_base"])
        assert_parity(to_np(out_c[0, rows, h]), ref, "bf16", f"prefill D=64 at 128K positions, head {h}")
        assert np.max(np.abs(to_np(lse_c[0, h, rows]) - ref_lse)) <= BF16_MAX_ABS
    assert_parity(krot_c, oracle.rope_cache(k, cfg["rope_base"]), "bf16", "k_rot D=64 at 128K positions")


def decode_one(attn, cfg, q, kc, vc, sl):
    kc_d = kc.to(DEV)
    vc_d = kc_d[..., :cfg["D_v"]] if cfg.get("v_aliases_k") else vc.to(DEV)
    out, lse = attn.decode(q.to(DEV), kc_d, vc_d, sl.to(DEV), rope_base=cfg["rope_base"],
                           rope_offset=cfg["rope_offset"], rope_dims=cfg["rope_dims"], scale=cfg["scale"],
                           lse=True)
    torch.cuda.synchronize()
    ref, ref_lse = oracle.attention_decode(q, kc, vc, sl.numpy(), rope_base=cfg["rope_base"],
                                           rope_offset=cfg["rope_offset"], rope_dims=cfg["rope_dims"],
                                           scale=cfg["scale"])
    return out, lse, ref, ref_lse


def test_gqa_decode_one_128k_sequence(lib):
    # one sequence split over every SM; a second, short one beside it; the query at position 131071
    cfg = workloads.config("gqa_decode", B=2, max_len=S_LONG, len_lo=1, len_hi=S_LONG)
    q, kc, vc, sl = workloads.decode_inputs(cfg, seed=17)
    sl[0], sl[1] = S_LONG, 3
    out, lse, ref, ref_lse = decode_one(lib, cfg, q, kc, vc, sl)
    assert_parity(out, ref, "bf16", "GQA decode over 128K keys")
    assert np.max(np.abs(to_np(lse) - ref_lse)) <= BF16_MAX_ABS


def test_mla_decode_one_128k_sequence(lib):
    # the absorbed MLA decode with a single 131072-key sequence: every CTA pair takes a piece of it
    cfg = workloads.config("mla_decode", B=1, max_len=S_LONG, len_lo=S_LONG, len_hi=S_LONG)
    q, kc, vc, sl = workloads.decode_inputs(cfg, seed=19)
    out, lse, ref, ref_lse = decode_one(lib, cfg, q, kc, vc, sl)
    assert_parity(out, ref, "bf16", "MLA decode over 128K keys")
    assert np.max(np.abs(to_np(lse) - ref_lse)) <= BF16_MAX_ABS
    assert math.isfinite(float(lse.float().sum()))

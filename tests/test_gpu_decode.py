"""Decode parity: split-KV decode (through the C ABI) against the fp64 oracle.

Covers the GQA decode configuration (59 sequences, 4096..8192 cached keys) and
the MLA-absorbed configuration (32 x 32768 keys, one 576-dim latent head, V =
its first 512 dims) in full, small cases with ragged lengths down to a single
key, fp32, RoPE on part of the latent, and the pages' statement that decoding
with a cache reproduces the full prefill token by token.
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


def run_decode(attn, cfg, q, kc, vc, sl):
    kc_d = kc.to(DEV)
    vc_d = kc_d[..., :cfg["D_v"]] if cfg.get("v_aliases_k") else vc.to(DEV)
    out, lse = attn.decode(q.to(DEV), kc_d, vc_d, sl.to(DEV), rope_base=cfg["rope_base"],
                           rope_offset=cfg["rope_offset"], rope_dims=cfg["rope_dims"], scale=cfg["scale"],
                           lse=True)
    torch.cuda.synchronize()
    return out, lse


def oracle_decode(cfg, q, kc, vc, sl, batch_index=None):
    return oracle.attention_decode(q, kc, vc, sl.numpy(), rope_base=cfg["rope_base"],
                                   rope_offset=cfg["rope_offset"], rope_dims=cfg["rope_dims"],
                                   scale=cfg["scale"], batch_index=batch_index)


SMALL = [
    # B, n_h, n_kv, D_qk, D_v, max_len, rope_base, rope_offset, rope_dims, alias, dtype
    (4, 32, 8, 128, 128, 700, 5e5, 0, 128, False, "bf16"),
    (3, 8, 8, 64, 64, 300, 1e4, 0, 64, False, "bf16"),
    (2, 6, 3, 128, 64, 1030, 0.0, 0, 128, False, "bf16"),
    (2, 16, 1, 576, 512, 300, 0.0, 512, 64, True, "bf16"),
    (2, 16, 1, 576, 512, 300, 1e4, 512, 64, True, "bf16"),
    (3, 4, 2, 64, 64, 100, 1e4, 0, 64, False, "f32"),
]


@pytest.mark.parametrize("B,n_h,n_kv,Dqk,Dv,L,rope,roff,rdims,alias,dtype", SMALL)
def test_decode_small(lib, B, n_h, n_kv, Dqk, Dv, L, rope, roff, rdims, alias, dtype):
    cfg = dict(B=B, n_h=n_h, n_kv=n_kv, D_qk=Dqk, D_v=Dv, max_len=L, len_lo=1, len_hi=L,
               v_aliases_k=alias, dtype=dtype, rope_base=rope, rope_offset=roff, rope_dims=rdims,
               scale=1 / math.sqrt(192) if alias else 0.0)
    q, kc, vc, sl = workloads.decode_inputs(cfg, seed=L)
    sl[0] = 1           # a sequence holding only its new token
    sl[-1] = L          # and one filling the cache
    out, lse = run_decode(lib, cfg, q, kc, vc, sl)
    ref, ref_lse = oracle_decode(cfg, q, kc, vc, sl)
    assert_parity(out, ref, dtype, f"decode {cfg}")
    assert np.max(np.abs(to_np(lse) - ref_lse)) <= (1e-4 if dtype == "f32" else BF16_MAX_ABS)


def test_gqa_decode_config_full(lib):
    cfg = workloads.config("gqa_decode")
    q, kc, vc, sl = workloads.decode_inputs(cfg, seed=0)
    out, lse = run_decode(lib, cfg, q, kc, vc, sl)
    ref, ref_lse = oracle_decode(cfg, q, kc, vc, sl)
    assert_parity(out, ref, "bf16", "gqa decode")
    assert np.max(np.abs(to_np(lse) - ref_lse)) <= BF16_MAX_ABS


def test_mla_decode_config_full(lib):
    cfg = workloads.config("mla_decode")
    q, kc, vc, sl = workloads.decode_inputs(cfg, seed=0)
    out, lse = run_decode(lib, cfg, q, kc, vc, sl)
    ref, ref_lse = oracle_decode(cfg, q, kc, vc, sl)
    assert_parity(out, ref, "bf16", "mla decode")
    assert np.max(np.abs(to_np(lse) - ref_lse)) <= BF16_MAX_ABS


def test_decode_with_cache_matches_prefill_token_by_token(lib):
    # "Transformer 与 LLM" slide 02: outputs with and without the KV cache agree token by token
    B, S, n_h, n_kv, D, base = 2, 300, 8, 2, 128, 5e5
    cfg = dict(B=B, S=S, n_h=n_h, n_kv=n_kv, D_h=D, dtype="bf16")
    q, k, v = workloads.prefill_inputs(cfg, seed=11)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    full, krot, _ = lib.prefill(qd, kd, vd, rope_base=base)          # krot is the rotated-K cache
    for t in (0, 1, 127, 128, 299):
        sl = torch.full((B,), t + 1, dtype=torch.int32, device=DEV)
        out, _ = lib.decode(qd[:, t].contiguous(), krot, vd, sl, rope_base=base)
        ref = oracle.attention_prefill(q, k, v, rope_base=base)[:, t]
        assert_parity(out, ref, "bf16", f"decode t={t}")
        assert_parity(out, to_np(full[:, t]), "bf16", f"decode vs prefill t={t}")


MLA_SMALL = [
    # B, max_len, rope_base: 128 heads over one 576-dim latent head, the tensor-core MLA kernel
    (3, 300, 0.0),
    (5, 100, 1e4),      # RoPE on the last 64 latent dims
    (40, 64, 0.0),      # many short sequences: key ranges of CTA pairs cross sequence ends
    (1, 2000, 0.0),     # one sequence split over every pair
    (3, 40000, 1e4),    # several 256-key rounds per pair, with RoPE and a ragged last round
]


@pytest.mark.parametrize("B,L,rope", MLA_SMALL)
def test_mla_shaped_decode(lib, B, L, rope):
    cfg = workloads.config("mla_decode", B=B, max_len=L, len_lo=1, len_hi=L, rope_base=rope)
    q, kc, vc, sl = workloads.decode_inputs(cfg, seed=B * 7 + L)
    sl[0] = 1
    sl[-1] = L
    out, lse = run_decode(lib, cfg, q, kc, vc, sl)
    ref, ref_lse = oracle_decode(cfg, q, kc, vc, sl)
    assert_parity(out, ref, "bf16", f"mla B={B} L={L}")
    assert np.max(np.abs(to_np(lse) - ref_lse)) <= BF16_MAX_ABS


@pytest.mark.parametrize("B", [256, 257])
def test_mla_decode_batch_limit(lib, B):
    # 256 sequences is the most the tensor-core MLA kernel takes (their key prefix sums live in
    # shared memory), with many short sequences per CTA pair; one more runs on the generic kernel
    cfg = workloads.config("mla_decode", B=B, max_len=64, len_lo=1, len_hi=64, rope_base=0.0)
    q, kc, vc, sl = workloads.decode_inputs(cfg, seed=B)
    sl[0] = 1
    sl[-1] = 64
    out, lse = run_decode(lib, cfg, q, kc, vc, sl)
    ref, ref_lse = oracle_decode(cfg, q, kc, vc, sl)
    assert_parity(out, ref, "bf16", f"mla decode B={B}")
    assert np.max(np.abs(to_np(lse) - ref_lse)) <= BF16_MAX_ABS


@pytest.mark.parametrize("lens,rope", [
    ([1], 0.0),              # one key in all: every CTA pair but one has nothing to do
    ([1, 2], 1e4),
    ([3, 1, 1], 0.0),
    ([257], 1e4),            # a second round holding a single valid key
    ([255, 1, 256], 0.0),
    ([4000, 3999, 4001, 4000], 1e4),  # pair starts ~261 keys apart: rounded to whole rounds, some
                                      # pairs hold two rounds and their neighbours none
])
def test_mla_decode_few_keys(lib, lens, rope):
    # far fewer keys than CTA pairs x 256: most pairs get an empty key range, and the partials
    # of the pairs that do get keys must still combine to each sequence's result
    L = max(lens)
    cfg = workloads.config("mla_decode", B=len(lens), max_len=L, len_lo=1, len_hi=L, rope_base=rope)
    q, kc, vc, _ = workloads.decode_inputs(cfg, seed=L + len(lens))
    sl = torch.tensor(lens, dtype=torch.int32)
    out, lse = run_decode(lib, cfg, q, kc, vc, sl)
    ref, ref_lse = oracle_decode(cfg, q, kc, vc, sl)
    assert_parity(out, ref, "bf16", f"mla decode lens={lens}")
    assert np.max(np.abs(to_np(lse) - ref_lse)) <= BF16_MAX_ABS


@pytest.mark.parametrize("roff,rdims,pairing", [
    (0, 64, "adjacent"),     # span at the start of the latent (inside the value dims)
    (256, 128, "half"),
    (504, 72, "adjacent"),   # span across the end of the value dims
    (64, 256, "half"),       # the widest span
])
def test_mla_decode_rope_spans(lib, roff, rdims, pairing):
    # the tensor-core MLA kernel rotates the query in shared memory, any span of whole 8-dim chunks
    cfg = workloads.config("mla_decode", B=3, max_len=600, len_lo=1, len_hi=600, rope_base=1e4)
    q, kc, vc, sl = workloads.decode_inputs(cfg, seed=roff + rdims)
    sl[0] = 1
    sl[-1] = 600
    kd = kc.to(DEV)
    out, lse = lib.decode(q.to(DEV), kd, kd[..., :512], sl.to(DEV), rope_base=1e4, rope_offset=roff,
                          rope_dims=rdims, scale=cfg["scale"], lse=True, pairing=pairing)
    torch.cuda.synchronize()
    ref, ref_lse = oracle.attention_decode(q, kc, vc, sl.numpy(), rope_base=1e4, rope_offset=roff,
                                           rope_dims=rdims, scale=cfg["scale"], pairing=pairing)
    assert_parity(out, ref, "bf16", f"mla decode rope [{roff}, {roff + rdims}) {pairing}")
    assert np.max(np.abs(to_np(lse) - ref_lse)) <= BF16_MAX_ABS


def test_mla_shaped_decode_fp32(lib):
    # the tensor-core MLA kernel is bf16; fp32 inputs of the same shape run on the generic kernel
    cfg = workloads.config("mla_decode", B=2, max_len=200, len_lo=1, len_hi=200, rope_base=1e4, dtype="f32")
    q, kc, vc, sl = workloads.decode_inputs(cfg, seed=13)
    sl[0] = 1
    out, lse = run_decode(lib, cfg, q, kc, vc, sl)
    ref, ref_lse = oracle_decode(cfg, q, kc, vc, sl)
    assert_parity(out, ref, "f32", "mla-shaped fp32 decode")
    assert np.max(np.abs(to_np(lse) - ref_lse)) <= 1e-4


def test_mla_decode_score_spikes(lib):
    """A few cached keys score about 80 (natural log units) above everything else for one head
    each, at positions spread over the sequences, so that most of them arrive after a CTA pair has
    fixed its shared exponent offset: the tensor-core MLA kernel must then move a row's offset
    within a round (its scores pass the old offset by far more than bf16 / fp32 exponents allow)
    and bring the two halves of the pair back to one offset.  Random inputs never take that path."""
    cfg = workloads.config("mla_decode", B=4, max_len=32768, len_lo=32768, len_hi=32768, rope_base=0.0)
    q, kc, vc, sl = workloads.decode_inputs(cfg, seed=5)
    scale = 1.0 / math.sqrt(192.0)
    spikes = [(0, 700, 3), (0, 5000, 77), (0, 17000, 127), (0, 30001, 40), (2, 1500, 0), (2, 20000, 64),
              (3, 32767, 100)]  # (sequence, key, head)
    for b, t, h in spikes:
        qh = q[b, h].double()
        lam = 80.0 / (scale * float(qh @ qh))
        kc[b, t, 0] = (lam * qh).to(kc.dtype)
    out, lse = run_decode(lib, cfg, q, kc, vc, sl)
    idx = sorted({b for b, _, _ in spikes})
    ref, ref_lse = oracle_decode(cfg, q, kc, vc, sl, batch_index=idx)
    got = to_np(out)
    assert_parity(got[idx], ref[idx], "bf16", "mla decode with score spikes")
    assert np.max(np.abs(to_np(lse)[idx] - ref_lse[idx])) <= BF16_MAX_ABS
    for b, t, h in spikes:  # the spiking key takes all of the head's weight
        np.testing.assert_allclose(got[b, h], to_np(kc[b, t, 0, :512]), atol=BF16_MAX_ABS)


@pytest.mark.parametrize("name", ["gqa_decode", "mla_decode"])
def test_rows_past_seqlens_are_never_used(lib, name):
    # cache rows at or after seqlens[b] hold NaN: results must still match the oracle
    if name == "gqa_decode":
        cfg = workloads.config(name, B=4, max_len=300, len_lo=1, len_hi=300)
    else:
        cfg = workloads.config(name, B=4, max_len=200, len_lo=1, len_hi=200)
    q, kc, vc, sl = workloads.decode_inputs(cfg, seed=21)
    sl[0] = 1
    kc_n = kc.clone()
    vc_n = kc_n[..., :cfg["D_v"]] if cfg.get("v_aliases_k") else vc.clone()
    for b in range(cfg["B"]):
        kc_n[b, int(sl[b]):] = float("nan")
        if not cfg.get("v_aliases_k"):
            vc_n[b, int(sl[b]):] = float("nan")
    out, _ = run_decode(lib, cfg, q, kc_n, vc_n, sl)
    assert torch.isfinite(out).all()
    ref, _ = oracle_decode(cfg, q, kc, vc, sl)
    assert_parity(out, ref, "bf16", f"{name} with NaN past seqlens")


@pytest.mark.parametrize("name,window,sink,B,max_len", [
    ("gqa_decode", 1000, 4, 4, 3000),     # one chunk per sequence holding both the sinks and the window
    ("gqa_decode", 300, 0, 4, 3000),
    ("gqa_decode", 4100, 4, 3, 12000),    # several chunks: sinks alone in one, chunks with neither skipped
    ("gqa_decode", 4096, 1, 2, 9000),     # window a multiple of the tile
    ("mla_decode", 500, 4, 2, 1500),
])
def test_decode_sliding_window_with_sinks(lib, name, window, sink, B, max_len):
    # "Transformer 与 LLM" slide 07: keep a window of recent keys plus a few sink tokens
    cfg = workloads.config(name, B=B, max_len=max_len, len_lo=1, len_hi=max_len)
    q, kc, vc, sl = workloads.decode_inputs(cfg, seed=window)
    sl[0] = 2
    sl[-1] = cfg["max_len"]
    kc_d = kc.to(DEV)
    vc_d = kc_d[..., :cfg["D_v"]] if cfg.get("v_aliases_k") else vc.to(DEV)
    out, lse = lib.decode_window(q.to(DEV), kc_d, vc_d, sl.to(DEV), window=window, n_sink=sink,
                                 rope_base=cfg["rope_base"], rope_offset=cfg["rope_offset"],
                                 rope_dims=cfg["rope_dims"], scale=cfg["scale"], lse=True)
    torch.cuda.synchronize()
    ref, ref_lse = oracle.attention_decode(q, kc, vc, sl.numpy(), rope_base=cfg["rope_base"],
                                           rope_offset=cfg["rope_offset"], rope_dims=cfg["rope_dims"],
                                           scale=cfg["scale"], window=window, n_sink=sink)
    assert_parity(out, ref, "bf16", f"{name} window {window}")
    assert np.max(np.abs(to_np(lse) - ref_lse)) <= BF16_MAX_ABS


TC_GQA = [
    # B, n_h, n_kv, max_len, rope_base: head groups of 1..16 on the tensor-core GQA kernel
    (3, 8, 8, 333, 1e4),      # G = 1 (MHA): one real row of the N = 16 operand
    (2, 16, 8, 129, 0.0),     # G = 2, one key past a tile
    (2, 32, 4, 1000, 5e5),    # G = 8
    (2, 64, 4, 260, 1e4),     # G = 16: the whole padded operand
    (2, 32, 8, 9000, 5e5),    # several 4096-key work units per sequence
    (5, 32, 8, 128, 5e5),     # exactly one tile
    (128, 8, 2, 4097, 5e5),   # 256 (sequence, chunk) pairs: the most the kernel ranks longest first
    (300, 8, 2, 700, 1e4),    # 300 pairs: claimed in sequence order
]


@pytest.mark.parametrize("B,n_h,n_kv,L,rope", TC_GQA)
def test_tensor_core_gqa_decode_head_groups(lib, B, n_h, n_kv, L, rope):
    cfg = dict(B=B, n_h=n_h, n_kv=n_kv, D_qk=128, D_v=128, max_len=L, len_lo=1, len_hi=L, v_aliases_k=False,
               dtype="bf16", rope_base=rope, rope_offset=0, rope_dims=128, scale=0.0)
    q, kc, vc, sl = workloads.decode_inputs(cfg, seed=L + n_h)
    sl[0] = 1
    sl[-1] = L
    out, lse = run_decode(lib, cfg, q, kc, vc, sl)
    ref, ref_lse = oracle_decode(cfg, q, kc, vc, sl)
    assert_parity(out, ref, "bf16", f"tensor-core GQA decode {cfg}")
    assert np.max(np.abs(to_np(lse) - ref_lse)) <= BF16_MAX_ABS

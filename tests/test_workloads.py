"""The seeded input generators and the benchmark's work counts (CPU only).

The work counts are checked against figures the pages print for the same
shapes (tests/golden/page_figures.txt).
"""
import math

import torch

import workloads


def test_generators_are_seeded_and_shaped():
    cfg = workloads.config("tiny")
    a = workloads.prefill_inputs(cfg, seed=0)
    b = workloads.prefill_inputs(cfg, seed=0)
    c = workloads.prefill_inputs(cfg, seed=1)
    assert all(torch.equal(x, y) for x, y in zip(a, b))
    assert not torch.equal(a[0], c[0])
    assert a[0].shape == (1, 16, 2, 8) and a[0].dtype == torch.float32


def test_decode_generator_lengths_and_alias():
    cfg = workloads.config("gqa_decode", B=5, max_len=64, len_lo=10, len_hi=64)
    q, kc, vc, sl = workloads.decode_inputs(cfg, seed=0)
    assert q.shape == (5, 32, 128) and kc.shape == (5, 64, 8, 128) and vc.shape == kc.shape
    assert sl.dtype == torch.int32 and int(sl.min()) >= 10 and int(sl.max()) <= 64
    mcfg = workloads.config("mla_decode", B=2, max_len=16, len_lo=16, len_hi=16)
    q, kc, vc, sl = workloads.decode_inputs(mcfg, seed=0)
    assert vc.data_ptr() == kc.data_ptr() and vc.shape[-1] == 512 and kc.shape[-1] == 576


def test_kv_bytes_per_token_match_pages():
    # Llama-3-8B: 32 layers x 2 x n_kv x D_h x 2 B = 128 KiB ("Transformer 与 LLM" slide 02)
    cfg = workloads.config("gqa_decode")
    per_layer = workloads.decode_bytes(cfg, [1])
    assert 32 * per_layer == 128 * 1024
    # DeepSeek-V3: 61 layers of one 576-dim bf16 latent row = 68.6 KiB (slide 06)
    mla = workloads.config("mla_decode")
    per_layer = workloads.decode_bytes(mla, [1])
    assert round(61 * per_layer / 1024, 1) == 68.6


def test_mla_intensity_matches_page():
    # about 242 FLOP per byte of cache for absorbed MLA decode (slide 06)
    mla = workloads.config("mla_decode")
    inten = workloads.decode_flops(mla, [1000]) / workloads.decode_bytes(mla, [1000])
    assert round(inten) == 242


def test_logits_size_matches_page():
    # materialised bf16 S at 8K context, 32 heads = 4 GiB per layer (slide 06)
    assert 8192 * 8192 * 32 * 2 == 4 * 1024 ** 3


def test_causal_flops_halve_dense():
    B, S, n_h, D = 4, 8192, 32, 128
    assert workloads.causal_flops(B, S, n_h, D) == 2 * B * n_h * S * S * D
    assert math.isclose(workloads.causal_flops(B, S, n_h, D), 2.199e12, rel_tol=1e-3)

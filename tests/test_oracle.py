"""Pins of the fp64 oracle against what the pages and the mathematics fix.

Each test ties one oracle function to something other than the oracle itself:
a matrix the pages print (tests/golden), a closed form, an invariant the pages
state, or the independently written brute-force loops of tests/bruteforce.py.
CPU only.
"""
import math
import os

import numpy as np
import pytest

import oracle
from tests import bruteforce
import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def load_golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            rows.append([float(t) if t not in ("-inf",) else -np.inf for t in line.split()])
    return np.array(rows)


def rng_normal(seed, *shape):
    return np.random.default_rng(seed).standard_normal(shape)


# ---------------------------------------------------------------- mask
@pytest.mark.parametrize("S,name", [(5, "causal_mask_5.txt"), (4, "causal_mask_4.txt")])
def test_mask_matches_printed(S, name):
    printed = load_golden(name)
    assert np.array_equal(oracle.causal_mask(S), printed)


def test_visibility_matches_printed():
    printed = load_golden("visibility_5.txt")
    M = oracle.causal_mask(5)
    assert np.array_equal((M == 0).astype(float), printed)


def test_mask_offset_and_window():
    # a chunk of 3 queries at positions 4..6 over 7 keys, window 3, one sink
    M = oracle.causal_mask(3, 7, q_offset=4, window=3, n_sink=1)
    for r in range(3):
        pos = 4 + r
        for n in range(7):
            keep = n <= pos and (pos - n < 3 or n < 1)
            assert (M[r, n] == 0) == keep


# ---------------------------------------------------------------- softmax
def test_softmax_rows_sum_to_one_and_masked_weights_zero():
    S = 37
    scores = rng_normal(1, S, S) * 5 + oracle.causal_mask(S)
    A = oracle.softmax_rows(scores)
    assert np.max(np.abs(A.sum(-1) - 1.0)) < 1e-12
    assert np.all(A[np.triu_indices(S, 1)] == 0.0)
    assert np.all(A[np.tril_indices(S)] > 0.0)


def test_logsumexp_matches_library():
    scipy_special = pytest.importorskip("scipy.special")
    x = rng_normal(2, 5, 40) * 30
    assert np.allclose(oracle.logsumexp_rows(x), scipy_special.logsumexp(x, axis=-1),
                       rtol=1e-14, atol=1e-12)


# ---------------------------------------------------------------- RoPE
def test_rope_first_pair_turns_by_position_in_radians():
    # theta_0 = base^0 = 1: the pair (1, 0) at position p lands on (cos p, sin p)
    for p in (1, 2, 7, 1000):
        out = oracle.rope_rotate(np.array([1.0, 0.0]), p, 10000.0)
        assert np.allclose(out, [math.cos(p), math.sin(p)], atol=1e-12)


def test_rope_frequencies_closed_form():
    th = oracle.rope_frequencies(8, 10000.0)
    assert np.allclose(th, [1.0, 0.1, 0.01, 0.001], rtol=1e-14)
    th = oracle.rope_frequencies(128, 500000.0)
    assert th[0] == 1.0 and abs(th[64 - 1] - 500000.0 ** (-126 / 128)) < 1e-20


def test_rope_position_zero_is_identity_and_norm_is_kept():
    x = rng_normal(3, 6, 16)
    assert np.array_equal(oracle.rope_rotate(x, 0, 10000.0), x)
    y = oracle.rope_rotate(x, np.arange(6) * 37, 10000.0)
    # each 2-D group keeps its length, hence the whole vector too
    assert np.allclose(np.hypot(y[:, 0::2], y[:, 1::2]), np.hypot(x[:, 0::2], x[:, 1::2]), rtol=1e-13)


def test_rope_groups_match_printed_pairs():
    pairs = load_golden("rope_pairs_8.txt").astype(int)
    for grp, d0, d1 in pairs:
        e = np.zeros(8)
        e[d0] = 1.0
        y = oracle.rope_rotate(e, 5, 10000.0)
        touched = set(np.nonzero(np.abs(y) > 1e-15)[0])
        assert touched == {d0, d1}, (grp, touched)


def test_rope_matches_complex_multiplication():
    x = rng_normal(4, 10, 12)
    pos = np.arange(10) * 13 + 3
    y = oracle.rope_rotate(x, pos, 500000.0)
    for r in range(10):
        ref = bruteforce.rotate_complex(list(x[r]), int(pos[r]), 500000.0)
        assert np.allclose(y[r], ref, atol=1e-12)


def test_rope_score_depends_on_relative_position_only():
    q = rng_normal(5, 64)
    k = rng_normal(6, 64)
    base = 10000.0
    ref = oracle.rope_rotate(q, 3, base) @ oracle.rope_rotate(k, 8, base)
    for shift in (10, 500, 4093):
        s = oracle.rope_rotate(q, 3 + shift, base) @ oracle.rope_rotate(k, 8 + shift, base)
        assert abs(s - ref) <= 1e-12 * max(1.0, abs(ref))
    # and it is not constant in the distance itself
    other = oracle.rope_rotate(q, 3, base) @ oracle.rope_rotate(k, 9, base)
    assert abs(other - ref) > 1e-6


def test_rope_half_split_is_adjacent_after_permutation():
    D = 16
    x = rng_normal(7, 5, D)
    pos = np.arange(5) * 11
    half = oracle.rope_rotate(x, pos, 10000.0, pairing="half")
    # dimension j of the half-split layout is dimension perm[j] of the adjacent layout
    perm = np.array([(j % (D // 2)) * 2 + j // (D // 2) for j in range(D)])
    xa = np.empty_like(x)
    xa[:, perm] = x
    adj = oracle.rope_rotate(xa, pos, 10000.0, pairing="adjacent")
    assert np.allclose(adj[:, perm], half, atol=1e-12)


def test_rope_partial_span_leaves_other_dims():
    x = rng_normal(8, 3, 576)
    y = oracle.rope_rotate(x, np.array([0, 5, 9]), 10000.0, offset=512, dims=64)
    assert np.array_equal(y[:, :512], x[:, :512])
    ref = bruteforce.rotate_complex(list(x[2]), 9, 10000.0, offset=512, dims=64)
    assert np.allclose(y[2], ref, atol=1e-12)


# ---------------------------------------------------------------- brute force
@pytest.mark.parametrize("S,n_h,n_kv,D,rope,causal,q_offset,window,sink", [
    (1, 1, 1, 2, 10000.0, True, 0, 0, 0),
    (5, 2, 2, 8, 10000.0, True, 0, 0, 0),
    (7, 4, 2, 6, 500000.0, True, 0, 0, 0),
    (6, 3, 1, 4, 0.0, True, 0, 0, 0),
    (6, 2, 1, 4, 0.0, False, 0, 0, 0),
    (4, 2, 2, 4, 10000.0, True, 3, 0, 0),
    (8, 2, 1, 4, 10000.0, True, 0, 3, 1),
])
def test_prefill_equals_bruteforce(S, n_h, n_kv, D, rope, causal, q_offset, window, sink):
    rng = np.random.default_rng(S * 100 + n_h)
    S_k = S + q_offset
    q = rng.standard_normal((1, S, n_h, D))
    k = rng.standard_normal((1, S_k, n_kv, D))
    v = rng.standard_normal((1, S_k, n_kv, D + 1))     # D_v != D_qk on purpose
    scale = 0.7
    out, lse = oracle.attention_prefill(q, k, v, rope_base=rope, scale=scale, causal=causal,
                                        q_offset=q_offset, window=window, n_sink=sink,
                                        return_lse=True)
    ref, ref_lse = bruteforce.prefill(q[0].tolist(), k[0].tolist(), v[0].tolist(), rope, scale,
                                      causal, q_offset, window, sink)
    assert np.allclose(out[0], np.array(ref), atol=1e-12, rtol=1e-12)
    assert np.allclose(lse[0], np.array(ref_lse), atol=1e-12, rtol=1e-12)


def test_tiny_config_equals_bruteforce():
    cfg = workloads.config("tiny")
    q, k, v = workloads.prefill_inputs(cfg, seed=0)
    out = oracle.attention_prefill(q, k, v, rope_base=cfg["rope_base"], scale=cfg["scale"])
    ref, _ = bruteforce.prefill(q[0].double().tolist(), k[0].double().tolist(),
                                v[0].double().tolist(), cfg["rope_base"], cfg["scale"])
    assert np.allclose(out[0], np.array(ref), atol=1e-12)


def test_default_scale_is_per_head_dim():
    q = rng_normal(9, 1, 3, 2, 16)
    k = rng_normal(10, 1, 3, 2, 16)
    v = rng_normal(11, 1, 3, 2, 16)
    a = oracle.attention_prefill(q, k, v, scale=0)
    b = oracle.attention_prefill(q, k, v, scale=1 / 4.0)
    assert np.array_equal(a, b)


# ---------------------------------------------------------------- closed forms
def test_single_token_returns_its_value():
    v = rng_normal(12, 1, 1, 3, 5)
    out = oracle.attention_prefill(rng_normal(13, 1, 1, 3, 4), rng_normal(14, 1, 1, 3, 4), v,
                                   rope_base=10000.0)
    assert np.allclose(out, v, atol=1e-15)


def test_zero_query_gives_prefix_mean():
    S = 9
    v = rng_normal(15, 1, S, 1, 6)
    out = oracle.attention_prefill(np.zeros((1, S, 1, 6)), rng_normal(16, 1, S, 1, 6), v)
    prefix_mean = np.cumsum(v[0, :, 0, :], axis=0) / np.arange(1, S + 1)[:, None]
    assert np.allclose(out[0, :, 0, :], prefix_mean, atol=1e-13)


def test_dominant_score_selects_that_value():
    S, D = 6, 4
    k = np.zeros((1, S, 1, D))
    k[0, 2, 0, 0] = 1.0
    q = np.zeros((1, S, 1, D))
    q[0, :, 0, 0] = 1.0
    v = rng_normal(17, 1, S, 1, D)
    out = oracle.attention_prefill(q, k, v, scale=200.0)
    # rows 2.. see key 2 with score 200 against 0 elsewhere
    assert np.allclose(out[0, 2:, 0, :], np.broadcast_to(v[0, 2, 0], (S - 2, D)), atol=1e-12)


# ---------------------------------------------------------------- invariants
def test_causality_future_tokens_do_not_leak():
    rng = np.random.default_rng(18)
    q, k, v = (rng.standard_normal((1, 12, 2, 8)) for _ in range(3))
    base = oracle.attention_prefill(q, k, v, rope_base=10000.0)
    m = 6
    q2, k2, v2 = q.copy(), k.copy(), v.copy()
    q2[:, m + 1:] += 3.0
    k2[:, m + 1:] *= -2.0
    v2[:, m + 1:] += 5.0
    pert = oracle.attention_prefill(q2, k2, v2, rope_base=10000.0)
    assert np.array_equal(base[:, :m + 1], pert[:, :m + 1])
    assert not np.allclose(base[:, m + 1:], pert[:, m + 1:])


def test_gqa_with_all_kv_heads_is_mha_and_equals_repeated_kv():
    rng = np.random.default_rng(19)
    B, S, n_h, D = 2, 7, 8, 8
    q = rng.standard_normal((B, S, n_h, D))
    for n_kv in (8, 4, 2, 1):
        k = rng.standard_normal((B, S, n_kv, D))
        v = rng.standard_normal((B, S, n_kv, D))
        G = n_h // n_kv
        gqa = oracle.attention_prefill(q, k, v, rope_base=10000.0)
        mha = oracle.attention_prefill(q, np.repeat(k, G, axis=2), np.repeat(v, G, axis=2),
                                       rope_base=10000.0)
        assert np.allclose(gqa, mha, atol=1e-14)


def test_gqa_groups_match_printed_table():
    rng = np.random.default_rng(20)
    n_h, n_kv, D = 32, 8, 4
    q = rng.standard_normal((1, 3, n_h, D))
    k = rng.standard_normal((1, 3, n_kv, D))
    v = rng.standard_normal((1, 3, n_kv, D))
    base = oracle.attention_prefill(q, k, v)
    for first, last, kv in load_golden("gqa_groups_32_8.txt").astype(int):
        v2 = v.copy()
        v2[:, :, kv - 1, :] += 1.0
        changed = np.nonzero(np.any(oracle.attention_prefill(q, k, v2) != base, axis=(0, 1, 3)))[0]
        assert list(changed) == list(range(first - 1, last))


def test_unmasked_attention_is_permutation_equivariant():
    rng = np.random.default_rng(21)
    S = 10
    q, k, v = (rng.standard_normal((1, S, 2, 6)) for _ in range(3))
    perm = rng.permutation(S)
    out = oracle.attention_prefill(q, k, v, causal=False)
    out_p = oracle.attention_prefill(q[:, perm], k[:, perm], v[:, perm], causal=False)
    assert np.allclose(out_p, out[:, perm], atol=1e-13)


def test_prefill_rows_match_full_prefill():
    rng = np.random.default_rng(22)
    q = rng.standard_normal((2, 40, 4, 8))
    k = rng.standard_normal((2, 40, 2, 8))
    v = rng.standard_normal((2, 40, 2, 8))
    full, lse = oracle.attention_prefill(q, k, v, rope_base=10000.0, return_lse=True)
    rows = [0, 7, 39]
    o, l = oracle.attention_prefill_rows(q, k, v, 1, 3, rows, rope_base=10000.0)
    assert np.allclose(o, full[1, rows, 3], atol=1e-13)
    assert np.allclose(l, lse[1, 3, rows], atol=1e-13)
    # a RoPE span on part of a 12-dim q/k head and 6-dim values
    q2 = rng.standard_normal((1, 30, 2, 12))
    k2 = rng.standard_normal((1, 30, 2, 12))
    v2 = rng.standard_normal((1, 30, 2, 6))
    full2 = oracle.attention_prefill(q2, k2, v2, rope_base=100.0, rope_offset=8, rope_dims=4)
    o2, _ = oracle.attention_prefill_rows(q2, k2, v2, 0, 1, rows[:2], rope_base=100.0, rope_offset=8, rope_dims=4)
    assert np.allclose(o2, full2[0, rows[:2], 1], atol=1e-13)


# ---------------------------------------------------------------- decode
def test_decode_with_cache_equals_prefill_token_by_token():
    rng = np.random.default_rng(23)
    B, S, n_h, n_kv, D = 2, 11, 4, 2, 8
    base = 10000.0
    q = rng.standard_normal((B, S, n_h, D))
    k = rng.standard_normal((B, S, n_kv, D))
    v = rng.standard_normal((B, S, n_kv, D))
    full = oracle.attention_prefill(q, k, v, rope_base=base)
    kc = oracle.rope_cache(k, base)
    for t in range(S):
        seqlens = np.full(B, t + 1)
        out, _ = oracle.attention_decode(q[:, t], kc, v, seqlens, rope_base=base)
        assert np.allclose(out, full[:, t], atol=1e-13)


def test_half_pairing_attention_is_adjacent_attention_on_permuted_dims():
    # a score is a dot product, so permuting the dims of q and k alike changes
    # nothing; the permutation that turns split halves into adjacent pairs
    # therefore carries half-split attention onto adjacent-pair attention
    rng = np.random.default_rng(25)
    B, S, n_h, n_kv, D = 1, 9, 4, 2, 8
    q = rng.standard_normal((B, S, n_h, D))
    k = rng.standard_normal((B, S, n_kv, D))
    v = rng.standard_normal((B, S, n_kv, D))
    perm = np.array([(j % (D // 2)) * 2 + j // (D // 2) for j in range(D)])
    qa, ka = np.empty_like(q), np.empty_like(k)
    qa[..., perm], ka[..., perm] = q, k
    half = oracle.attention_prefill(q, k, v, rope_base=10000.0, pairing="half")
    adj = oracle.attention_prefill(qa, ka, v, rope_base=10000.0, pairing="adjacent")
    assert np.allclose(half, adj, atol=1e-13)
    assert not np.allclose(half, oracle.attention_prefill(q, k, v, rope_base=10000.0), atol=1e-3)


def test_decode_half_pairing_equals_prefill_token_by_token():
    rng = np.random.default_rng(26)
    B, S, n_h, n_kv, D = 2, 7, 4, 1, 8
    q = rng.standard_normal((B, S, n_h, D))
    k = rng.standard_normal((B, S, n_kv, D))
    v = rng.standard_normal((B, S, n_kv, D))
    full = oracle.attention_prefill(q, k, v, rope_base=500.0, pairing="half")
    kc = oracle.rope_cache(k, 500.0, pairing="half")
    for t in range(S):
        out, _ = oracle.attention_decode(q[:, t], kc, v, np.full(B, t + 1), rope_base=500.0, pairing="half")
        assert np.allclose(out, full[:, t], atol=1e-13)


def test_decode_window_matches_prefill_window():
    rng = np.random.default_rng(24)
    S = 12
    q, k, v = (rng.standard_normal((1, S, 2, 4)) for _ in range(3))
    full = oracle.attention_prefill(q, k, v, rope_base=10000.0, window=4, n_sink=2)
    kc = oracle.rope_cache(k, 10000.0)
    out, _ = oracle.attention_decode(q[:, S - 1], kc, v, [S], rope_base=10000.0, window=4, n_sink=2)
    assert np.allclose(out, full[:, S - 1], atol=1e-13)


def test_mla_absorbed_equals_unabsorbed():
    B, n_h, L = 2, 8, 50
    q_c, q_r, c_kv, k_r, w_uk, w_uv = workloads.mla_factors(B, n_h, L, seed=3)
    seqlens = np.array([50, 33])
    scale = 1.0 / math.sqrt(192)
    ref = oracle.mla_decode_unabsorbed(q_c, q_r, c_kv, k_r, w_uk, w_uv, seqlens, scale)
    q_t = oracle.mla_absorb_query(q_c, q_r, w_uk)                     # [B, n_h, 576]
    cache = np.concatenate([c_kv.numpy(), k_r.numpy()], axis=-1)[:, :, None, :]   # one KV head
    o_lat, _ = oracle.attention_decode(q_t, cache, cache[..., :512], seqlens, scale=scale)
    out = oracle.mla_unabsorb_output(o_lat, w_uv)
    assert np.max(np.abs(out - ref)) <= 1e-10 * max(1.0, np.max(np.abs(ref)))


def test_mla_prefill_unabsorbed_equals_absorbed():
    # "Transformer 与 LLM" slide 06: the absorbed form (W_UK folded into the query,
    # W_UV into the output: 128 heads sharing one 576-dim latent KV head) and the
    # up-projected form the slide routes prefill through give the same attention
    rng = np.random.default_rng(27)
    B, S, n_h, d_c, d_r, d_l = 1, 10, 3, 8, 4, 12
    q_c = rng.standard_normal((B, S, n_h, d_c))
    q_r = rng.standard_normal((B, S, n_h, d_r))
    c_kv = rng.standard_normal((B, S, d_l))
    k_r = rng.standard_normal((B, S, d_r))
    w_uk = rng.standard_normal((n_h, d_l, d_c)) / math.sqrt(d_l)
    w_uv = rng.standard_normal((n_h, d_l, d_c)) / math.sqrt(d_l)
    q, k, v, out = oracle.mla_prefill_unabsorbed(q_c, q_r, c_kv, k_r, w_uk, w_uv, rope_base=100.0)
    assert q.shape == (B, S, n_h, d_c + d_r) and v.shape == (B, S, n_h, d_c)
    assert np.array_equal(k[:, :, 0, d_c:], k[:, :, 2, d_c:])   # k^R shared by every head
    q_abs = np.concatenate([np.einsum("hlc,bshc->bshl", w_uk, q_c), q_r], axis=-1)
    latent = np.concatenate([c_kv, k_r], axis=-1)[:, :, None, :]  # one KV head of d_l + d_r dims
    o_lat = oracle.attention_prefill(q_abs, latent, c_kv[:, :, None, :], rope_base=100.0,
                                     scale=1 / math.sqrt(d_c + d_r), rope_offset=d_l, rope_dims=d_r)
    absorbed = np.einsum("hlc,bshl->bshc", w_uv, o_lat)
    assert np.max(np.abs(out - absorbed)) <= 1e-12 * max(1.0, np.max(np.abs(out)))
    # the RoPE span matters: without rotation the result differs
    _, _, _, plain = oracle.mla_prefill_unabsorbed(q_c, q_r, c_kv, k_r, w_uk, w_uv)
    assert np.max(np.abs(out - plain)) > 1e-3


def test_hand_example_rows_sum_to_one():
    # "Transformer 与 LLM" slide 01 works one head by hand (d = 4, T = 3) but does
    # not print its inputs: only the row-sum property can be checked (parity unpinned).
    q, k, v = (rng_normal(25 + i, 1, 3, 1, 4) for i in range(3))
    _, A, _ = oracle.attention_head(q[0, :, 0], k[0, :, 0], v[0, :, 0], 0.5, oracle.causal_mask(3))
    assert np.allclose(A.sum(-1), 1.0, atol=1e-15)


def test_rejects_bad_head_counts():
    with pytest.raises(ValueError):
        oracle.attention_prefill(np.zeros((1, 2, 3, 4)), np.zeros((1, 2, 2, 4)), np.zeros((1, 2, 2, 4)))

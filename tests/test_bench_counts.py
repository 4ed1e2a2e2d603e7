"""The work counts bench.py divides by, checked by brute force on small cases (host logic, no GPU)."""
import itertools

import bench
import workloads


def brute_pairs(q_pos, n_keys, window=None, n_sink=0):
    n = 0
    for m in q_pos:
        for k in range(n_keys):
            if k > m:
                continue
            if window is not None and m - k >= window and k >= n_sink:
                continue
            n += 1
    return n


def test_visible_pairs_matches_brute_force():
    for S, window, sinks in itertools.product((1, 7, 33), (None, 1, 4, 10, 40), (0, 1, 3)):
        if window is None and sinks:
            continue
        assert bench.visible_pairs(range(S), S, window, sinks) == brute_pairs(range(S), S, window, sinks)
    # a chunk of queries at an offset over the keys before and inside it
    assert bench.visible_pairs(range(20, 30), 30) == brute_pairs(range(20, 30), 30)
    assert bench.visible_pairs(range(20, 30), 30, 6, 2) == brute_pairs(range(20, 30), 30, 6, 2)


def test_causal_flops_is_half_the_dense_count():
    B, S, n_h, D = 2, 64, 4, 32
    dense = 4.0 * B * n_h * S * S * D
    assert workloads.causal_flops(B, S, n_h, D) == dense / 2
    # D_v != D_qk: 2 D_qk for the scores and 2 D_v for the weighted sum, per pair
    assert workloads.causal_flops(1, S, n_h, 192, 128) == 2.0 * n_h * S * S * (192 + 128) / 2


def test_windowed_decode_key_count_matches_brute_force():
    # the new token sits at position L - 1 and sees keys n with L - 1 - n < window, plus n < n_sink
    for L, window, sinks in itertools.product((1, 5, 17, 64), (1, 4, 16), (0, 2, 5)):
        brute = sum(1 for n in range(L) if L - 1 - n < window or n < sinks)
        assert bench.window_decode_keys(L, window, sinks) == brute

"""Planted mistakes in the fp64 oracle, for checking that its pins catch them.

Loaded as a pytest plugin (``-p tests.oracle_mutants``) in a child process with
ORACLE_MUTANT naming one mutant: the plugin replaces the named oracle function
(in ``oracle.attention`` and in the ``oracle`` package, so that both the pins
and the oracle's own internal calls see it) by a wrapper that makes one
plausible mistake.  Without ORACLE_MUTANT it does nothing.  Nothing here is
used outside tests/test_oracle_mutations.py.
"""
from __future__ import annotations

import math
import os

import numpy as np

import oracle
import oracle.attention as oa

_orig = {name: getattr(oa, name) for name in (
    "causal_mask", "rope_frequencies", "rope_rotate", "softmax_rows", "logsumexp_rows", "attention_head",
    "default_scale", "attention_prefill", "attention_prefill_rows", "attention_decode", "mla_absorb_query",
    "mla_unabsorb_output", "mla_decode_unabsorbed")}


def _rope_sign(rotary_dims, base):
    # every pair turns the wrong way
    return -_orig["rope_frequencies"](rotary_dims, base)


def _theta_index(rotary_dims, base):
    # theta_i = base^(-2(i+1)/D): the exponent starts at 1
    i = np.arange(1, rotary_dims // 2 + 1, dtype=np.float64)
    return np.power(float(base), -2.0 * i / rotary_dims)


def _mask_diagonal(n_q, n_k=None, q_offset=0, window=0, n_sink=0):
    # the query's own key is masked too (n >= m)
    M = _orig["causal_mask"](n_q, n_k, q_offset, window, n_sink)
    for m in range(n_q):
        if q_offset + m < M.shape[1]:
            M[m, q_offset + m] = oa.NEG_INF
    return M


def _window_off_by_one(n_q, n_k=None, q_offset=0, window=0, n_sink=0):
    # a window of w keys keeps w + 1
    return _orig["causal_mask"](n_q, n_k, q_offset, window + 1 if window > 0 else 0, n_sink)


def _half_is_adjacent(x, positions, base, offset=0, dims=None, pairing="adjacent"):
    # the split-halves pairing silently falls back to adjacent pairs
    return _orig["rope_rotate"](x, positions, base, offset, dims, pairing="adjacent")


def _softmax_axis(scores):
    # normalised over the query axis instead of the key axis
    m = np.max(scores, axis=-1, keepdims=True)
    e = np.exp(scores - m)
    return e / np.sum(e, axis=0, keepdims=True)


def _lse_log2(scores):
    # the normaliser in log2 units
    return _orig["logsumexp_rows"](scores) / math.log(2.0)


def _value_shift(q_rot, k_rot, v, scale, mask):
    # each weight multiplies the value row of the previous key
    S = scale * (q_rot @ k_rot.T)
    if mask is not None:
        S = S + mask
    A = oa.softmax_rows(S)
    return A @ np.roll(v, 1, axis=0), A, oa.logsumexp_rows(S)


def _scale_by_dim(D_h, scale):
    # 1/D_h instead of 1/sqrt(D_h)
    return 1.0 / D_h if (scale is None or scale <= 0) else float(scale)


def _kv_reversed(a):
    return np.ascontiguousarray(oa._f64(a)[:, :, ::-1])


def _head_map_prefill(q, k, v, **kw):
    # query head h reads the K/V head n_kv - 1 - h // G
    return _orig["attention_prefill"](q, _kv_reversed(k), _kv_reversed(v), **kw)


def _head_map_rows(q, k, v, b, h, rows, **kw):
    return _orig["attention_prefill_rows"](q, _kv_reversed(k), _kv_reversed(v), b, h, rows, **kw)


def _head_map_decode(q, kcache, vcache, seqlens, **kw):
    return _orig["attention_decode"](q, _kv_reversed(kcache), _kv_reversed(vcache), seqlens, **kw)


def _decode_position(q, kcache, vcache, seqlens, *, rope_base=0.0, rope_offset=0, rope_dims=None,
                     pairing="adjacent", **kw):
    # the new query is rotated at position seqlens[b] instead of seqlens[b] - 1
    q = oa._f64(q)
    if rope_base > 0:
        q = _orig["rope_rotate"](q, np.ones(q.shape[:-1]), rope_base, rope_offset, rope_dims, pairing=pairing)
    return _orig["attention_decode"](q, kcache, vcache, seqlens, rope_base=rope_base, rope_offset=rope_offset,
                                     rope_dims=rope_dims, pairing=pairing, **kw)


def _absorb_drops_rope(q_c, q_r, w_uk):
    # the decoupled rotary part of the query is left out of the absorbed query
    out = _orig["mla_absorb_query"](q_c, q_r, w_uk)
    out[..., -oa._f64(q_r).shape[-1]:] = 0.0
    return out


def _unabsorb_wrong_head(o_latent, w_uv):
    # head h's output is projected with the next head's W_UV
    return _orig["mla_unabsorb_output"](o_latent, np.roll(oa._f64(w_uv), 1, axis=0))


MUTANTS = {
    "rope_sign": {"rope_frequencies": _rope_sign},
    "theta_index": {"rope_frequencies": _theta_index},
    "mask_diagonal": {"causal_mask": _mask_diagonal},
    "window_off_by_one": {"causal_mask": _window_off_by_one},
    "half_is_adjacent": {"rope_rotate": _half_is_adjacent},
    "softmax_axis": {"softmax_rows": _softmax_axis},
    "lse_log2": {"logsumexp_rows": _lse_log2},
    "value_shift": {"attention_head": _value_shift},
    "scale_by_dim": {"default_scale": _scale_by_dim},
    "head_map": {"attention_prefill": _head_map_prefill, "attention_prefill_rows": _head_map_rows,
                 "attention_decode": _head_map_decode},
    "decode_position": {"attention_decode": _decode_position},
    "absorb_drops_rope": {"mla_absorb_query": _absorb_drops_rope},
    "unabsorb_wrong_head": {"mla_unabsorb_output": _unabsorb_wrong_head},
}


def pytest_configure(config):
    name = os.environ.get("ORACLE_MUTANT", "")
    if not name:
        return
    for fn_name, fn in MUTANTS[name].items():
        setattr(oa, fn_name, fn)
        if hasattr(oracle, fn_name):
            setattr(oracle, fn_name, fn)

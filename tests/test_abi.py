"""The C ABI library without a GPU: it loads, exports every symbol the header
declares, and rejects bad arguments on the host before touching a device.

The pointers passed here are never dereferenced: every call below returns
during host-side validation, before any CUDA call is made.
"""
import ctypes
import os
import re

import pytest

from transformer_causal_attention_gb300 import _binding as B
from transformer_causal_attention_gb300 import build as build_mod

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "attn.h")

FAKE = 1 << 20          # 16-byte aligned, never dereferenced
FAKE2 = 2 << 20
MISALIGNED = (1 << 20) + 4


@pytest.fixture(scope="module")
def lib():
    build_mod.build()
    return B.load()


def declared_symbols():
    text = open(HEADER, encoding="utf-8").read()
    return re.findall(r"ATTN_API\s+[\w\s\*]*?\b(attn_\w+)\s*\(", text)


def test_header_and_binding_agree():
    names = set(declared_symbols())
    assert names == {n for n, _, _ in B.SIGNATURES}
    assert len(names) == 16


def test_library_exports_every_declared_symbol(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name


def test_strerror(lib):
    for code in (0, -1, -2, -3, -4, -5, -6, 12345):
        assert lib.attn_strerror(code)


def prefill(lib, q=FAKE, k=FAKE, v=FAKE, out=FAKE, k_rot=FAKE2, lse=None, B=1, S=16, n_h=2, n_kv=2, D=64,
            rope=0.0, scale=0.0, causal=1, dtype=1):
    return lib.attn_prefill(q, k, v, out, k_rot, lse, B, S, n_h, n_kv, D, rope, scale, causal, dtype, None)


def test_prefill_argument_errors(lib):
    assert prefill(lib, q=None) == -1
    assert prefill(lib, B=0) == -1
    assert prefill(lib, S=-3) == -1
    assert prefill(lib, n_h=6, n_kv=4) == -1
    assert prefill(lib, causal=2) == -1
    assert prefill(lib, dtype=7) == -1
    assert prefill(lib, rope=10000.0, k_rot=None) == -1


def test_prefill_unsupported_and_alignment(lib):
    assert prefill(lib, D=264) == -2
    assert prefill(lib, D=60) == -2            # bf16 needs a multiple of 8
    assert prefill(lib, D=7, dtype=0) == -2
    assert prefill(lib, q=MISALIGNED) == -3
    assert prefill(lib, rope=10000.0, k_rot=MISALIGNED) == -3


def test_prefill_rejects_k_rot_overlapping_k(lib):
    assert prefill(lib, rope=10000.0, k=FAKE, k_rot=FAKE + 64) == -1


def decode(lib, q=FAKE, kc=FAKE, vc=FAKE2, ldv=0, sl=FAKE, out=FAKE, lse=None, B=2, n_h=8, n_kv=2, Dqk=128,
           Dv=128, L=256, rope=0.0, roff=0, rdims=128, scale=0.0, dtype=1, ws=FAKE, ws_bytes=None):
    if ws_bytes is None:
        ws_bytes = lib.attn_decode_workspace_size(B, n_h, n_kv, Dqk, Dv, L, dtype)
    return lib.attn_decode(q, kc, vc, ldv, sl, out, lse, B, n_h, n_kv, Dqk, Dv, L, rope, roff, rdims, scale,
                           dtype, ws, ws_bytes, None)


def test_decode_argument_errors(lib):
    assert decode(lib, sl=None) == -1
    assert decode(lib, ws=None) == -1
    assert decode(lib, n_h=6, n_kv=4) == -1
    assert decode(lib, L=0) == -1
    assert decode(lib, rope=10000.0, roff=64, rdims=128) == -1   # span past D_qk
    assert decode(lib, rope=10000.0, rdims=3) == -1
    assert decode(lib, ldv=-8) == -1


def test_decode_unsupported_alignment_workspace(lib):
    assert decode(lib, Dqk=100) == -2
    assert decode(lib, Dqk=1024) == -2
    assert decode(lib, q=MISALIGNED) == -3
    assert decode(lib, ws_bytes=16) == -6


def test_workspace_size(lib):
    n = lib.attn_decode_workspace_size(59, 32, 8, 128, 128, 8192, 1)
    assert 0 < n < 64 << 20
    bad = lib.attn_decode_workspace_size(0, 32, 8, 128, 128, 8192, 1)
    assert bad == ctypes.c_size_t(-1).value


def test_rope_argument_errors(lib):
    r = lib.attn_rope
    assert r(FAKE, FAKE, 1, 4, 2, 64, 0, 64, 0.0, 0, 1, None) == -1      # base must be > 0
    assert r(FAKE, FAKE, 1, 4, 2, 64, 32, 64, 1e4, 0, 1, None) == -1     # span past D
    assert r(FAKE, FAKE, 1, 4, 2, 64, 4, 8, 1e4, 0, 1, None) == -1       # bf16 offset not a multiple of 8
    assert r(FAKE, FAKE + 32, 1, 4, 2, 64, 0, 64, 1e4, 0, 1, None) == -1  # partial overlap
    assert r(MISALIGNED, FAKE, 1, 4, 2, 64, 0, 64, 1e4, 0, 1, None) == -3
    assert r(FAKE, FAKE, 1, 4, 2, 1024, 0, 1024, 1e4, 0, 1, None) == -2  # more pairs than the table holds


def test_rope_at_argument_errors(lib):
    r = lib.attn_rope_at
    assert r(FAKE, FAKE, None, 1, 4, 2, 64, 0, 64, 1e4, 1, None) == -1        # positions are required
    assert r(FAKE, FAKE, FAKE2, 1, 4, 2, 64, 0, 64, 0.0, 1, None) == -1       # base must be > 0
    assert r(FAKE, FAKE, FAKE2 + 2, 1, 4, 2, 64, 0, 64, 1e4, 1, None) == -3   # positions not 4-byte aligned
    assert r(MISALIGNED, FAKE, FAKE2, 1, 4, 2, 64, 0, 64, 1e4, 1, None) == -3


def test_wait_limit_and_counter(lib):
    before = lib.attn_launch_count()
    lib.attn_set_wait_limit_ns(2_000_000_000)
    assert lib.attn_launch_count() == before


def test_prefill_chunk_argument_errors(lib):
    f = lib.attn_prefill_chunk
    # q, kc, vc, out, lse, B, S_q, q_offset, max_len, n_h, n_kv, D, rope, scale, causal, dtype, stream
    assert f(None, FAKE, FAKE, FAKE, None, 1, 16, 0, 64, 2, 2, 64, 0.0, 0.0, 1, 1, None) == -1
    assert f(FAKE, FAKE, FAKE, FAKE, None, 1, 16, 60, 64, 2, 2, 64, 0.0, 0.0, 1, 1, None) == -1  # past max_len
    assert f(FAKE, FAKE, FAKE, FAKE, None, 1, 16, -1, 64, 2, 2, 64, 0.0, 0.0, 1, 1, None) == -1
    assert f(FAKE, FAKE, FAKE, FAKE, None, 1, 16, 0, 64, 3, 2, 64, 0.0, 0.0, 1, 1, None) == -1
    assert f(FAKE, FAKE, FAKE, FAKE, None, 1, 16, 0, 64, 2, 2, 264, 0.0, 0.0, 1, 1, None) == -2
    assert f(MISALIGNED, FAKE, FAKE, FAKE, None, 1, 16, 0, 64, 2, 2, 64, 0.0, 0.0, 1, 1, None) == -3


def test_kv_append_argument_errors(lib):
    f = lib.attn_kv_append
    # k_new, v_new, kc, vc, ldv, start, B, C, n_kv, D_qk, D_v, max_len, rope, roff, rdims, dtype, stream
    assert f(None, FAKE, FAKE, FAKE, 0, FAKE, 1, 1, 2, 64, 64, 16, 0.0, 0, 64, 1, None) == -1
    assert f(FAKE, FAKE, FAKE, FAKE, 0, None, 1, 1, 2, 64, 64, 16, 0.0, 0, 64, 1, None) == -1
    assert f(FAKE, FAKE, FAKE, None, 0, FAKE, 1, 1, 2, 64, 64, 16, 0.0, 0, 64, 1, None) == -1   # v_new without vcache
    assert f(FAKE, FAKE, FAKE, FAKE, 0, FAKE, 1, 1, 2, 60, 64, 16, 0.0, 0, 64, 1, None) == -1   # D not a multiple of 8
    assert f(FAKE, FAKE, FAKE, FAKE, 0, FAKE, 1, 1, 2, 64, 64, 16, 1e4, 4, 56, 1, None) == -1   # offset not a multiple of 8
    assert f(FAKE, FAKE, FAKE, FAKE, 0, FAKE, 1, 1, 2, 64, 64, 16, 1e4, 32, 64, 1, None) == -1  # span past D_qk
    assert f(MISALIGNED, FAKE, FAKE, FAKE, 0, FAKE, 1, 1, 2, 64, 64, 16, 0.0, 0, 64, 1, None) == -3


def test_rope_half_flag_validation(lib):
    HALF = B.ATTN_ROPE_HALF
    assert HALF == 0x100
    # unknown flag bits or element types are argument errors
    assert prefill(lib, dtype=1 | 0x200) == -1
    assert prefill(lib, dtype=HALF | 2) == -1
    assert decode(lib, dtype=1 | 0x400) == -1
    # split halves need whole 8-element chunks per half in bf16 (D_h a multiple of 16)
    assert prefill(lib, D=8, rope=1e4, dtype=1 | HALF) == -2
    assert prefill(lib, D=6, rope=1e4, dtype=0 | HALF) == -2   # fp32: D_h a multiple of 4
    r = lib.attn_rope
    assert r(FAKE, FAKE, 1, 4, 2, 64, 0, 8, 1e4, 0, 1 | HALF, None) == -1   # a half of 4 bf16 dims
    assert r(FAKE, FAKE, 1, 4, 2, 64, 0, 6, 1e4, 0, 0 | HALF, None) == -1   # a half of 3 fp32 dims
    f = lib.attn_kv_append
    assert f(FAKE, FAKE, FAKE, FAKE, 0, FAKE, 1, 1, 2, 64, 64, 16, 1e4, 0, 8, 1 | HALF, None) == -1
    # the flag does not change the workspace a decode needs
    for dt in (0, 1):
        assert (lib.attn_decode_workspace_size(59, 32, 8, 128, 128, 8192, dt | HALF)
                == lib.attn_decode_workspace_size(59, 32, 8, 128, 128, 8192, dt))


def test_prefill_mla_argument_errors(lib):
    f = lib.attn_prefill_mla
    # q, k, v, out, k_rot, lse, B, S, n_h, n_kv, D_qk, D_v, rope, roff, rdims, scale, causal, dtype, stream
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE2, None, 1, 16, 2, 2, 192, 128, 1e4, 128, 128, 0.0, 1, 1, None) == -1  # span
    assert f(FAKE, FAKE, FAKE, FAKE, None, None, 1, 16, 2, 2, 192, 128, 1e4, 128, 64, 0.0, 1, 1, None) == -1   # k_rot
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE2, None, 1, 16, 2, 2, 192, 0, 1e4, 128, 64, 0.0, 1, 1, None) == -1    # D_v
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE2, None, 1, 16, 2, 2, 192, 264, 0.0, 0, 0, 0.0, 1, 1, None) == -2     # D_v > 256
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE2, None, 1, 16, 2, 2, 192, 128, 1e4, 124, 64, 0.0, 1, 1, None) == -2  # offset % 8
    assert f(FAKE, FAKE, MISALIGNED, FAKE, FAKE2, None, 1, 16, 2, 2, 192, 128, 1e4, 128, 64, 0.0, 1, 1, None) == -3

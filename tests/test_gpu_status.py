"""Failure detection of the bounded device waits, without a GPU fault.

Every wait of the library's kernels (on a TMA copy, an MMA or another warp)
gives up after a time limit, records a status bit and lets the kernel return,
so a stuck pipeline surfaces as ATTN_ERR_TIMEOUT from attn_device_status
instead of a hung GPU.  attn_check_wait_timeout runs one warp whose barrier is
never completed, which makes the wait run out on purpose; the CUDA context must
stay usable afterwards.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    import transformer_causal_attention_gb300 as attn
    return attn


def test_expired_wait_reports_timeout_and_context_survives(lib):
    assert lib.device_status() == 0
    lib.set_wait_limit_ns(50_000_000)          # 50 ms
    try:
        lib.check_wait_timeout()
        assert lib.device_status() == -5        # ATTN_ERR_TIMEOUT
        assert lib.device_status() == 0         # reading clears it
    finally:
        lib.set_wait_limit_ns(2_000_000_000)
    # the context still runs the real kernels correctly
    cfg = dict(B=1, S=200, n_h=2, n_kv=1, D_h=128, dtype="bf16")
    q, k, v = workloads.prefill_inputs(cfg, seed=2)
    out, _, _ = lib.prefill(q.to(DEV), k.to(DEV), v.to(DEV), rope_base=1e4)
    ref = oracle.attention_prefill(q, k, v, rope_base=1e4)
    assert np.max(np.abs(out.float().cpu().numpy() - ref)) <= 2e-2
    assert lib.device_status() == 0

"""attn_decode_static: decode for callers that may not allocate device memory.

Some callers cannot hand attn_decode a workspace because they are not allowed
to allocate at the moment they decode (an engine plugin whose per-step hook
owns no memory, a latency-critical token loop that cannot take the device-wide
synchronisation of cudaMalloc/cudaFree, a runtime with a memory budget fixed at
start-up).  attn_decode_static keeps the split-KV partials in a 16 MiB scratch
array compiled into the library.  This test calls it through the C ABI twice in
a row and compares each result with attn_decode's on the same inputs and with
the fp64 oracle.  The file is named so that pytest collects it last.
"""

import pytest
import torch

import oracle
import workloads
from tests.tolerances import assert_parity, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    import transformer_causal_attention_gb300 as attn
    return attn


def call_static(raw, q, kc, vc, ldv, sl, out, cfg):
    return raw.attn_decode_static(q.data_ptr(), kc.data_ptr(), vc.data_ptr(), ldv, sl.data_ptr(), out.data_ptr(),
                                  None, cfg["B"], cfg["n_h"], cfg["n_kv"], cfg["D_qk"], cfg["D_v"], cfg["max_len"],
                                  float(cfg["rope_base"]), cfg["rope_offset"], cfg["rope_dims"], float(cfg["scale"]),
                                  1, torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("name,overrides", [
    ("gqa_decode", dict(B=59)),                                   # the full GQA decode workload
    ("gqa_decode", dict(B=3, n_h=8, n_kv=8, D_qk=64, D_v=64, max_len=500, len_lo=1, len_hi=500, rope_dims=64)),
])
def test_static_scratch_decode_matches_workspace_decode(lib, name, overrides):
    raw = lib.load()
    cfg = workloads.config(name, **overrides)
    q, kc, vc, sl = workloads.decode_inputs(cfg, seed=5)
    q, kc, vc, sl = q.to(DEV), kc.to(DEV), vc.to(DEV), sl.to(DEV)
    ref, _ = lib.decode(q, kc, vc, sl, rope_base=cfg["rope_base"], rope_offset=cfg["rope_offset"],
                        rope_dims=cfg["rope_dims"], scale=cfg["scale"])
    torch.cuda.synchronize()
    ref_np = to_np(ref)
    want, _ = oracle.attention_decode(q.cpu(), kc.cpu(), vc.cpu(), sl.cpu().numpy(), rope_base=cfg["rope_base"],
                                      rope_offset=cfg["rope_offset"], rope_dims=cfg["rope_dims"],
                                      scale=cfg["scale"])
    for _ in range(2):  # the second call reuses the scratch the first one left behind
        out = torch.full_like(ref, float("nan"))
        assert call_static(raw, q, kc, vc, 0, sl, out, cfg) == 0
        torch.cuda.synchronize()
        assert_parity(out, ref_np, "bf16", "attn_decode_static vs attn_decode")
        assert_parity(out, want, "bf16", "attn_decode_static vs the fp64 oracle")
    assert lib.device_status() == 0


def test_static_scratch_rejects_oversized_problems(lib):
    raw = lib.load()
    cfg = workloads.config("mla_decode")  # needs more partial storage than the 16 MiB scratch
    need = lib.decode_workspace_size(cfg["B"], cfg["n_h"], cfg["n_kv"], cfg["D_qk"], cfg["D_v"], cfg["max_len"])
    assert need > (16 << 20)
    dummy = torch.empty(16, dtype=torch.bfloat16, device=DEV)
    sl = torch.ones(cfg["B"], dtype=torch.int32, device=DEV)
    rc = call_static(raw, dummy, dummy, dummy, 576, sl, dummy, cfg)
    assert rc == -6  # ATTN_ERR_WORKSPACE, before anything is launched
    assert raw.attn_strerror(rc)

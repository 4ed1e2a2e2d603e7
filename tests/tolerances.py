"""Parity bars between the CUDA library and the fp64 oracle.

fp32 inputs: max |gpu - oracle| <= 1e-4.  bf16 inputs: max-abs <= 2e-2 and
relative L2 error <= 5e-3.  The bf16 bar covers the roundings the tensor-core
path makes on purpose - rotated Q/K and the probabilities P are rounded to
bf16 before their MMAs, the output is rounded to bf16 - each a relative
2^-9 effect, inside the 1e-3..1e-2 band that "Transformer 与 LLM" slide 11
gives for a bf16 kernel against an fp32 reference.
"""
import numpy as np

FP32_MAX_ABS = 1e-4
BF16_MAX_ABS = 2e-2
BF16_REL_L2 = 5e-3


def to_np(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def errors(gpu, ref):
    g = to_np(gpu) if hasattr(gpu, "detach") else np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    diff = g - ref
    max_abs = float(np.max(np.abs(diff))) if diff.size else 0.0
    rel = float(np.linalg.norm(diff) / max(np.linalg.norm(ref), 1e-30))
    return max_abs, rel


def assert_parity(gpu, ref, dtype: str, what: str = ""):
    max_abs, rel = errors(gpu, ref)
    if dtype == "f32":
        assert max_abs <= FP32_MAX_ABS, f"{what}: max-abs {max_abs:.3e} > {FP32_MAX_ABS}"
    else:
        assert max_abs <= BF16_MAX_ABS, f"{what}: max-abs {max_abs:.3e} > {BF16_MAX_ABS}"
        assert rel <= BF16_REL_L2, f"{what}: rel-L2 {rel:.3e} > {BF16_REL_L2}"
    return max_abs, rel

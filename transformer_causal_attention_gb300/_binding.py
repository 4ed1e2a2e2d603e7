"""ctypes binding of libattn.so: argument marshalling only.

Every function here checks the torch tensors it is given (device, dtype,
contiguity, shape), allocates outputs with torch when the caller does not pass
them, and forwards raw device pointers to the C ABI declared in
include/attn.h.  All arithmetic runs in the library's CUDA kernels; there is
no CPU or PyTorch fallback - a missing library or GPU raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libattn.so")

ATTN_F32, ATTN_BF16 = 0, 1
ATTN_ROPE_HALF = 0x100  # OR'd into the dtype code: RoPE pairs (j, j + rope_dims/2)
ERRORS = {
    0: "ATTN_OK", -1: "ATTN_ERR_ARG", -2: "ATTN_ERR_UNSUPPORTED", -3: "ATTN_ERR_ALIGN",
    -4: "ATTN_ERR_CUDA", -5: "ATTN_ERR_TIMEOUT", -6: "ATTN_ERR_WORKSPACE",
}

# (name, restype, argtypes) of every exported symbol, mirroring include/attn.h
_vp, _i, _f, _sz, _u64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t, ctypes.c_ulonglong
SIGNATURES = [
    ("attn_strerror", ctypes.c_char_p, [_i]),
    ("attn_prefill", _i, [_vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _f, _i, _i, _vp]),
    ("attn_prefill_window", _i, [_vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _f, _i, _i, _i, _vp]),
    ("attn_prefill_mla", _i, [_vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _f, _i, _i, _f, _i, _i,
                              _vp]),
    ("attn_rope", _i, [_vp, _vp, _i, _i, _i, _i, _i, _i, _f, _i, _i, _vp]),
    ("attn_rope_at", _i, [_vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _f, _i, _vp]),
    ("attn_prefill_chunk", _i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _f, _f, _i, _i, _vp]),
    ("attn_kv_append", _i, [_vp, _vp, _vp, _vp, _i, _vp, _i, _i, _i, _i, _i, _i, _f, _i, _i, _i, _vp]),
    ("attn_decode_workspace_size", _sz, [_i, _i, _i, _i, _i, _i, _i]),
    ("attn_decode", _i, [_vp, _vp, _vp, _i, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _f, _i, _i, _f, _i,
                         _vp, _sz, _vp]),
    ("attn_decode_window", _i, [_vp, _vp, _vp, _i, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _f, _i, _i, _f, _i,
                                _i, _i, _vp, _sz, _vp]),
    ("attn_decode_static", _i, [_vp, _vp, _vp, _i, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _f, _i, _i, _f, _i,
                                _vp]),
    ("attn_device_status", _i, [_vp]),
    ("attn_check_wait_timeout", _i, [_vp]),
    ("attn_launch_count", _u64, []),
    ("attn_set_wait_limit_ns", None, [_u64]),
]


class AttnError(RuntimeError):
    """A non-zero return code of the C ABI."""

    def __init__(self, code: int, where: str):
        self.code = code
        msg = _lib().attn_strerror(code).decode() if _LIB is not None else ERRORS.get(code, "?")
        super().__init__(f"{where}: {ERRORS.get(code, code)} ({msg})")


_LIB = None


def _lib() -> ctypes.CDLL:
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "transformer_causal_attention_gb300.build.build()")
        lib = ctypes.CDLL(LIB_PATH)
        for name, res, args in SIGNATURES:
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _LIB = lib
    return _LIB


def load() -> ctypes.CDLL:
    """Load libattn.so (raises if it has not been built)."""
    return _lib()


def _check(rc: int, where: str) -> None:
    if rc != 0:
        raise AttnError(rc, where)


def _dtype_code(t: torch.Tensor, pairing: str = "adjacent") -> int:
    """Element-type code of t, with ATTN_ROPE_HALF for pairing="half"."""
    if pairing not in ("adjacent", "half"):
        raise ValueError(f"pairing must be 'adjacent' or 'half', not {pairing!r}")
    flag = ATTN_ROPE_HALF if pairing == "half" else 0
    if t.dtype == torch.bfloat16:
        return ATTN_BF16 | flag
    if t.dtype == torch.float32:
        return ATTN_F32 | flag
    raise TypeError(f"unsupported dtype {t.dtype}: bf16 or fp32")


def _dev(t: torch.Tensor, name: str) -> None:
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (the library has no CPU path)")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _stream_ptr(stream) -> int | None:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _ptr(t: torch.Tensor | None):
    return None if t is None else t.data_ptr()


def prefill(q, k, v, *, rope_base: float = 0.0, scale: float = 0.0, causal: bool = True,
            out=None, k_rot=None, lse: bool | torch.Tensor = False, pairing: str = "adjacent", stream=None):
    """Causal (or full) attention over whole prompts via attn_prefill.

    q [B,S,n_h,D], k/v [B,S,n_kv,D] CUDA tensors (bf16 or fp32, contiguous, BSHD).
    Returns out [B,S,n_h,D]; with rope_base > 0 also returns the rotated keys
    k_rot [B,S,n_kv,D] (the KV-cache form), and with lse=True the fp32
    log-sum-exp [B,n_h,S].  Result tuple: (out, k_rot or None, lse or None).
    pairing "adjacent" rotates dims (2i, 2i+1), "half" dims (j, j + D/2).
    """
    for name, t in (("q", q), ("k", k), ("v", v)):
        _dev(t, name)
    if not (q.dtype == k.dtype == v.dtype):
        raise TypeError("q, k and v must share a dtype")
    B, S, n_h, D = q.shape
    n_kv = k.shape[2]
    if k.shape != (B, S, n_kv, D) or v.shape != (B, S, n_kv, D):
        raise ValueError("k and v must be [B, S, n_kv, D] matching q")
    if out is None:
        out = torch.empty_like(q)
    _dev(out, "out")
    if rope_base > 0 and k_rot is None:
        k_rot = torch.empty_like(k)
    if isinstance(lse, torch.Tensor):
        lse_t = lse
    elif lse:
        lse_t = torch.empty((B, n_h, S), dtype=torch.float32, device=q.device)
    else:
        lse_t = None
    rc = _lib().attn_prefill(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(k_rot) if rope_base > 0 else None,
                             _ptr(lse_t), B, S, n_h, n_kv, D, float(rope_base), float(scale),
                             1 if causal else 0, _dtype_code(q, pairing), _stream_ptr(stream))
    _check(rc, "attn_prefill")
    return out, (k_rot if rope_base > 0 else None), lse_t


def prefill_window(q, k, v, *, window: int, n_sink: int = 0, rope_base: float = 0.0, scale: float = 0.0,
                   out=None, k_rot=None, lse: bool = False, pairing: str = "adjacent", stream=None):
    """Causal sliding-window attention with attention sinks via attn_prefill_window.

    Same tensors as prefill(); a query at position m sees keys n <= m with
    m - n < window or n < n_sink.  Returns (out, k_rot or None, lse or None).
    """
    for name, t in (("q", q), ("k", k), ("v", v)):
        _dev(t, name)
    B, S, n_h, D = q.shape
    n_kv = k.shape[2]
    if out is None:
        out = torch.empty_like(q)
    if rope_base > 0 and k_rot is None:
        k_rot = torch.empty_like(k)
    lse_t = torch.empty((B, n_h, S), dtype=torch.float32, device=q.device) if lse else None
    rc = _lib().attn_prefill_window(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(k_rot) if rope_base > 0 else None,
                                    _ptr(lse_t), B, S, n_h, n_kv, D, float(rope_base), float(scale), int(window),
                                    int(n_sink), _dtype_code(q, pairing), _stream_ptr(stream))
    _check(rc, "attn_prefill_window")
    return out, (k_rot if rope_base > 0 else None), lse_t


def prefill_mla(q, k, v, *, rope_base: float = 0.0, rope_offset: int = 0, rope_dims: int | None = None,
                scale: float = 0.0, causal: bool = True, out=None, k_rot=None, lse: bool | torch.Tensor = False,
                pairing: str = "adjacent", stream=None):
    """Prefill with q/k head dim D_qk != v head dim D_v and RoPE on a span (attn_prefill_mla).

    q [B,S,n_h,D_qk], k [B,S,n_kv,D_qk], v [B,S,n_kv,D_v].  For the MLA prefill
    shape D_qk = 192 (content 128 + decoupled RoPE 64, rope_offset=128,
    rope_dims=64) and D_v = 128.  Returns (out [B,S,n_h,D_v], k_rot or None, lse or None).
    """
    for name, t in (("q", q), ("k", k), ("v", v)):
        _dev(t, name)
    if not (q.dtype == k.dtype == v.dtype):
        raise TypeError("q, k and v must share a dtype")
    B, S, n_h, D_qk = q.shape
    n_kv, D_v = k.shape[2], v.shape[3]
    if k.shape != (B, S, n_kv, D_qk) or v.shape != (B, S, n_kv, D_v):
        raise ValueError("k must be [B, S, n_kv, D_qk] and v [B, S, n_kv, D_v]")
    rope_dims = (D_qk - rope_offset) if rope_dims is None else rope_dims
    if out is None:
        out = torch.empty((B, S, n_h, D_v), dtype=q.dtype, device=q.device)
    _dev(out, "out")
    if rope_base > 0 and k_rot is None:
        k_rot = torch.empty_like(k)
    if isinstance(lse, torch.Tensor):
        lse_t = lse
    else:
        lse_t = torch.empty((B, n_h, S), dtype=torch.float32, device=q.device) if lse else None
    rc = _lib().attn_prefill_mla(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(k_rot) if rope_base > 0 else None,
                                 _ptr(lse_t), B, S, n_h, n_kv, D_qk, D_v, float(rope_base), rope_offset, rope_dims,
                                 float(scale), 1 if causal else 0, _dtype_code(q, pairing), _stream_ptr(stream))
    _check(rc, "attn_prefill_mla")
    return out, (k_rot if rope_base > 0 else None), lse_t


def rope(x, *, rope_base: float, rope_offset: int = 0, rope_dims: int | None = None, pos_offset: int = 0,
         positions=None, out=None, pairing: str = "adjacent", stream=None):
    """RoPE of x [B,S,n_heads,D] (out may be x): at positions pos_offset + s via attn_rope, or,
    given positions (int32 [B,S] on the device), row (b, s) at positions[b, s] via attn_rope_at."""
    _dev(x, "x")
    B, S, H, D = x.shape
    rope_dims = D - rope_offset if rope_dims is None else rope_dims
    if out is None:
        out = torch.empty_like(x)
    if positions is not None:
        _dev(positions, "positions")
        if positions.dtype != torch.int32 or tuple(positions.shape) != (B, S):
            raise ValueError("positions must be int32 [B, S]")
        rc = _lib().attn_rope_at(_ptr(out), _ptr(x), _ptr(positions), B, S, H, D, rope_offset, rope_dims,
                                 float(rope_base), _dtype_code(x, pairing), _stream_ptr(stream))
        _check(rc, "attn_rope_at")
        return out
    rc = _lib().attn_rope(_ptr(out), _ptr(x), B, S, H, D, rope_offset, rope_dims, float(rope_base), pos_offset,
                          _dtype_code(x, pairing), _stream_ptr(stream))
    _check(rc, "attn_rope")
    return out


def prefill_chunk(q, kcache, vcache, *, q_offset: int, rope_base: float = 0.0, scale: float = 0.0,
                  causal: bool = True, out=None, lse: bool = False, pairing: str = "adjacent", stream=None):
    """A prompt chunk at positions q_offset.. against a KV cache via attn_prefill_chunk.

    q [B,S_q,n_h,D] (un-rotated), kcache/vcache [B,max_len,n_kv,D] holding rotated keys
    0 .. q_offset+S_q-1 (this chunk's included).  Returns (out [B,S_q,n_h,D], lse or None).
    """
    for name, t in (("q", q), ("kcache", kcache), ("vcache", vcache)):
        _dev(t, name)
    B, S_q, n_h, D = q.shape
    max_len, n_kv = kcache.shape[1], kcache.shape[2]
    if vcache.shape != kcache.shape:
        raise ValueError("vcache must match kcache")
    if out is None:
        out = torch.empty_like(q)
    lse_t = torch.empty((B, n_h, S_q), dtype=torch.float32, device=q.device) if lse else None
    rc = _lib().attn_prefill_chunk(_ptr(q), _ptr(kcache), _ptr(vcache), _ptr(out), _ptr(lse_t), B, S_q, q_offset,
                                   max_len, n_h, n_kv, D, float(rope_base), float(scale), 1 if causal else 0,
                                   _dtype_code(q, pairing), _stream_ptr(stream))
    _check(rc, "attn_prefill_chunk")
    return out, lse_t


def kv_append(k_new, v_new, kcache, vcache, start, *, rope_base: float = 0.0, rope_offset: int = 0,
              rope_dims: int | None = None, pairing: str = "adjacent", stream=None):
    """Write new tokens into a KV cache via attn_kv_append (keys rotated at start[b] + c).

    k_new [B,C,n_kv,D_qk], v_new [B,C,n_kv,D_v] or None (values alias the keys),
    kcache [B,max_len,n_kv,D_qk], vcache contiguous or a leading slice of kcache's
    last dim, start int32 [B] on the device.
    """
    _dev(k_new, "k_new")
    _dev(kcache, "kcache")
    if not start.is_cuda or start.dtype != torch.int32:
        raise ValueError("start must be an int32 CUDA tensor")
    B, C, n_kv, D_qk = k_new.shape
    max_len = kcache.shape[1]
    if v_new is not None:
        _dev(v_new, "v_new")
        D_v = v_new.shape[-1]
        ldv = 0 if vcache.is_contiguous() else vcache.stride(1)
    else:
        D_v = vcache.shape[-1] if vcache is not None else D_qk
        ldv = 0
    rope_dims = (D_qk - rope_offset) if rope_dims is None else rope_dims
    rc = _lib().attn_kv_append(_ptr(k_new), _ptr(v_new), _ptr(kcache), None if vcache is None else vcache.data_ptr(),
                               ldv, _ptr(start), B, C, n_kv, D_qk, D_v, max_len, float(rope_base), rope_offset,
                               rope_dims, _dtype_code(k_new, pairing), _stream_ptr(stream))
    _check(rc, "attn_kv_append")


def decode_workspace_size(B, n_h, n_kv, D_qk, D_v, max_len, dtype=torch.bfloat16) -> int:
    n = _lib().attn_decode_workspace_size(B, n_h, n_kv, D_qk, D_v, max_len,
                                          ATTN_BF16 if dtype == torch.bfloat16 else ATTN_F32)
    if n == ctypes.c_size_t(-1).value:
        raise ValueError("invalid decode sizes")
    return n


def decode(q, kcache, vcache, seqlens, *, rope_base: float = 0.0, rope_offset: int = 0,
           rope_dims: int | None = None, scale: float = 0.0, out=None, lse: bool = False, workspace=None,
           pairing: str = "adjacent", stream=None, _window=None):
    """One new token per sequence against its KV cache via attn_decode.

    q [B,n_h,D_qk] (un-rotated), kcache [B,L,n_kv,D_qk] (rotated keys), vcache
    [B,L,n_kv,D_v] contiguous or a last-dim slice of kcache (MLA: V = the first
    D_v latent dims), seqlens int32 [B] on the device (keys incl. the new one).
    Returns (out [B,n_h,D_v], lse [B,n_h] or None).
    """
    _dev(q, "q")
    _dev(kcache, "kcache")
    if not vcache.is_cuda:
        raise ValueError("vcache must be a CUDA tensor")
    if not seqlens.is_cuda or seqlens.dtype != torch.int32:
        raise ValueError("seqlens must be an int32 CUDA tensor")
    B, n_h, D_qk = q.shape
    _, L, n_kv, _ = kcache.shape
    D_v = vcache.shape[-1]
    if vcache.is_contiguous():
        ldv = 0
    elif vcache.data_ptr() == kcache.data_ptr() and vcache.stride(-1) == 1 and vcache.stride(2) == D_qk:
        ldv = vcache.stride(1)
    else:
        raise ValueError("vcache must be contiguous or a leading slice of kcache's last dim")
    rope_dims = (D_qk - rope_offset) if rope_dims is None else rope_dims
    if out is None:
        out = torch.empty((B, n_h, D_v), dtype=q.dtype, device=q.device)
    lse_t = torch.empty((B, n_h), dtype=torch.float32, device=q.device) if lse else None
    need = decode_workspace_size(B, n_h, n_kv, D_qk, D_v, L, q.dtype)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    common = (_ptr(q), _ptr(kcache), vcache.data_ptr(), ldv, _ptr(seqlens), _ptr(out), _ptr(lse_t), B, n_h, n_kv,
              D_qk, D_v, L, float(rope_base), rope_offset, rope_dims, float(scale))
    tail = (_dtype_code(q, pairing), _ptr(workspace), workspace.numel() * workspace.element_size(), _stream_ptr(stream))
    if _window is None:
        _check(_lib().attn_decode(*common, *tail), "attn_decode")
    else:
        _check(_lib().attn_decode_window(*common, int(_window[0]), int(_window[1]), *tail), "attn_decode_window")
    return out, lse_t


def decode_window(q, kcache, vcache, seqlens, *, window: int, n_sink: int = 0, rope_base: float = 0.0,
                  rope_offset: int = 0, rope_dims: int | None = None, scale: float = 0.0, out=None,
                  lse: bool = False, workspace=None, pairing: str = "adjacent", stream=None):
    """decode() with a sliding window of `window` keys plus `n_sink` sink keys (attn_decode_window)."""
    return decode(q, kcache, vcache, seqlens, rope_base=rope_base, rope_offset=rope_offset, rope_dims=rope_dims,
                  scale=scale, out=out, lse=lse, workspace=workspace, pairing=pairing, stream=stream,
                  _window=(window, n_sink))


def device_status(stream=None) -> int:
    """Synchronise the stream and return (and clear) the library's device status code."""
    return _lib().attn_device_status(_stream_ptr(stream))


def check_wait_timeout(stream=None) -> None:
    """Run the library's bounded-wait failure check (see attn_check_wait_timeout)."""
    _check(_lib().attn_check_wait_timeout(_stream_ptr(stream)), "attn_check_wait_timeout")


def launch_count() -> int:
    return int(_lib().attn_launch_count())


def set_wait_limit_ns(ns: int) -> None:
    _lib().attn_set_wait_limit_ns(int(ns))

"""Python binding of libattn.so (fused online-softmax attention for GB300).

Argument marshalling only: every step of the computation runs in the CUDA
kernels of libattn.so. PyTorch supplies device memory and the current stream.
If the library is not built, importing works but every call raises; there is
no fallback path.

Entry points mirror include/attn.h:
    prefill(q, k, v, causal, scale, alibi_slopes, impl)  -> (O, LSE)
    prefill_host(q, k, v, ...)  (host tensors, pipelined) -> (O, LSE)
    decode_splitk(q, k, v, kv_lens, scale, num_splits)   -> (O_part, LSE_part)
    combine(O_part, LSE_part)                            -> (O, LSE)
    decode(q, k, v, kv_lens, scale, num_splits)          -> (O, LSE)
"""
from __future__ import annotations

import ctypes
import math
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libattn.so")

ATTN_OK = 0
IMPLS = {"auto": 0, "tcgen05": 1, "mma_sync": 2, "tcgen05_1tile": 3}

_c_void_p = ctypes.c_void_p
_c_int = ctypes.c_int
_c_float = ctypes.c_float

class PrefillOptions(ctypes.Structure):
    """Mirror of attn_prefill_options (include/attn.h)."""
    _fields_ = [("causal", ctypes.c_int), ("scale", ctypes.c_float),
                ("alibi_slopes", ctypes.c_void_p), ("softcap", ctypes.c_float),
                ("window_left", ctypes.c_int), ("window_right", ctypes.c_int),
                ("impl", ctypes.c_int)]


# name -> (restype, argtypes); the full exported surface of include/attn.h
SIGNATURES = {
    "attn_prefill": (_c_int, [_c_void_p] * 5 + [_c_int] * 7 + [_c_float, _c_void_p, _c_void_p]),
    "attn_prefill_ex": (_c_int, [_c_void_p] * 5 + [_c_int] * 7 + [_c_float, _c_void_p, _c_int,
                                                                   _c_void_p]),
    "attn_prefill_opts": (_c_int, [_c_void_p] * 5 + [_c_int] * 6 + [ctypes.POINTER(PrefillOptions),
                                                                     _c_void_p]),
    "attn_prefill_host_workspace_bytes": (ctypes.c_size_t, [_c_int] * 6),
    "attn_prefill_host_chunks": (_c_int, [_c_int] * 3),
    "attn_prefill_host": (_c_int, [_c_void_p] * 5 + [_c_int] * 6 + [ctypes.POINTER(PrefillOptions),
                                                                     _c_int, _c_void_p,
                                                                     ctypes.c_size_t, _c_void_p]),
    "attn_prefill_splitkv_workspace_bytes": (ctypes.c_size_t, [_c_int] * 5),
    "attn_prefill_splitkv": (_c_int, [_c_void_p] * 5 + [_c_int] * 7 + [_c_float, _c_void_p, _c_int,
                                                                     _c_void_p, ctypes.c_size_t,
                                                                     _c_void_p]),
    "attn_backward_workspace_bytes": (ctypes.c_size_t, [_c_int] * 4),
    "attn_backward": (_c_int, [_c_void_p] * 9 + [_c_int] * 7 + [_c_float, _c_void_p, _c_void_p,
                                                               ctypes.c_size_t, _c_void_p]),
    "attn_backward_ex": (_c_int, [_c_void_p] * 9 + [_c_int] * 7 + [_c_float, _c_void_p, _c_void_p,
                                                                  ctypes.c_size_t, _c_int,
                                                                  _c_void_p]),
    "attn_rmsnorm_matmul": (_c_int, [_c_void_p] * 5 + [_c_int] * 3 + [_c_float, _c_int,
                                                                     _c_void_p]),
    "attn_rmsnorm_matmul_tiled": (_c_int, [_c_void_p] * 5 + [_c_int] * 3 + [_c_float, _c_int,
                                                                           _c_int, _c_void_p]),
    "attn_rmsnorm_matmul_splits": (_c_int, [_c_int] * 3),
    "attn_rmsnorm_matmul_chained": (_c_int, [_c_void_p] * 5 + [_c_int] * 3 + [_c_float, _c_void_p]),
    "attn_rmsnorm_matmul_ws_bytes": (ctypes.c_size_t, [_c_int] * 2),
    "attn_rmsnorm_matmul_ws": (_c_int, [_c_void_p] * 5 + [_c_int] * 3 + [_c_float, _c_int,
                                                                       _c_void_p, ctypes.c_size_t,
                                                                       _c_void_p]),
    "attn_rmsnorm_matmul_ws_chained": (_c_int, [_c_void_p] * 5 + [_c_int] * 3 +
                                       [_c_float, _c_int, _c_void_p, ctypes.c_size_t, _c_void_p]),
    "attn_decode_num_splits": (_c_int, [_c_int] * 5),
    "attn_decode_split_len": (_c_int, [_c_int] * 2),
    "attn_decode_workspace_bytes": (ctypes.c_size_t, [_c_int] * 4),
    "attn_decode_splitk": (_c_int, [_c_void_p] * 4 + [_c_int] * 5 + [_c_float, _c_int, _c_void_p,
                                                                     _c_void_p, _c_void_p,
                                                                     _c_void_p]),
    "attn_combine": (_c_int, [_c_void_p] * 2 + [_c_int] * 4 + [_c_void_p] * 3),
    "attn_decode": (_c_int, [_c_void_p] * 4 + [_c_int] * 5 + [_c_float, _c_int] + [_c_void_p] * 5),
    "attn_decode_noalloc": (_c_int, [_c_void_p] * 4 + [_c_int] * 5 + [_c_float, _c_int] +
                            [_c_void_p] * 3),
    "attn_status_string": (ctypes.c_char_p, [_c_int]),
    "attn_device_status": (_c_int, [_c_void_p]),
    "attn_version": (_c_int, []),
    "attn_selftest_wait_timeout": (_c_int, [_c_int, _c_void_p]),
    "attn_selftest_prefill_abort": (_c_int, [_c_void_p] * 5 + [_c_int] * 7 + [_c_float, _c_int,
                                                                            _c_int, _c_int,
                                                                            _c_void_p]),
}

_lib = None



class AttnError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = lib().attn_status_string(status).decode() if _lib is not None else str(status)
        super().__init__(f"{where}: {msg} (status {status})")


def lib() -> ctypes.CDLL:
    """The loaded libattn.so; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with "
                "`python -m online_softmax_fusion_gb300.build` (no fallback path exists)")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _check(status: int, where: str):
    if status != ATTN_OK:
        raise AttnError(status, where)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _req(t, name, dtype, dims):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != dims:
        raise ValueError(f"{name} must have {dims} dims, got {t.dim()}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def prefill(q, k, v, causal=False, scale=None, alibi_slopes=None, impl="auto", out=None,
            lse=None, with_lse=True, softcap=0.0, window=(-1, -1)):
    """Fused attention forward. q [B,Hq,Lq,d], k/v [B,Hkv,Lk,d] bf16 CUDA.
    softcap > 0 caps the scaled scores (cap * tanh(x / cap)); window =
    (left, right) limits row i to keys [i' - left, i' + right] (-1 = no limit).
    Returns (O bf16 [B,Hq,Lq,d], LSE fp32 [B,Hq,Lq] or None)."""
    _req(q, "q", torch.bfloat16, 4)
    _req(k, "k", torch.bfloat16, 4)
    _req(v, "v", torch.bfloat16, 4)
    B, Hq, Lq, d = q.shape
    Hkv, Lk = k.shape[1], k.shape[2]
    if tuple(v.shape) != tuple(k.shape) or k.shape[0] != B or k.shape[3] != d:
        raise ValueError("k and v must be [B, Hkv, Lk, d] matching q")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if alibi_slopes is not None:
        _req(alibi_slopes, "alibi_slopes", torch.float32, 1)
    if out is None:
        out = torch.empty_like(q)
    if lse is None and with_lse:
        lse = torch.empty((B, Hq, Lq), dtype=torch.float32, device=q.device)
    if softcap or tuple(window) != (-1, -1):
        opts = PrefillOptions(int(bool(causal)), float(scale),
                              None if alibi_slopes is None else alibi_slopes.data_ptr(),
                              float(softcap), int(window[0]), int(window[1]), IMPLS[impl])
        st = lib().attn_prefill_opts(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, Hq, Hkv,
                                     Lq, Lk, d, ctypes.byref(opts), _stream())
    else:
        st = lib().attn_prefill_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, Hq, Hkv,
                                   Lq, Lk, d, int(bool(causal)), float(scale), _ptr(alibi_slopes),
                                   IMPLS[impl], _stream())
    _check(st, "attn_prefill")
    return out, lse


def _req_host(t, name, dtype, dims):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device.type != "cpu":
        raise ValueError(f"{name} must be a host (CPU) tensor")
    if t.dtype != dtype or t.dim() != dims or not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous {dtype} with {dims} dims")


def prefill_host_workspace(B, Hq, Hkv, Lq, Lk, d, device=None):
    """Device workspace for prefill_host (uint8 tensor of the required size)."""
    n = lib().attn_prefill_host_workspace_bytes(B, Hq, Hkv, Lq, Lk, d)
    if n == 0:
        raise ValueError("invalid sizes")
    return torch.empty(n, dtype=torch.uint8, device=device or "cuda")


def prefill_host(q, k, v, causal=False, scale=None, alibi_slopes=None, impl="auto",
                 softcap=0.0, window=(-1, -1), chunk_kv_heads=0, out=None, lse=None,
                 with_lse=True, workspace=None, synchronize=True):
    """prefill on HOST tensors: q [B,Hq,Lq,d], k/v [B,Hkv,Lk,d] bf16 on the CPU
    (page-locked for the copies to overlap the kernels). The library copies
    chunks of KV heads in, runs the fused prefill per chunk on the current
    stream and copies O / LSE back, the three stages pipelined. alibi_slopes is
    a CUDA tensor. Returns (O, LSE or None) as CPU tensors; with
    synchronize=False they are complete only once the current stream has
    passed the call."""
    _req_host(q, "q", torch.bfloat16, 4)
    _req_host(k, "k", torch.bfloat16, 4)
    _req_host(v, "v", torch.bfloat16, 4)
    B, Hq, Lq, d = q.shape
    Hkv, Lk = k.shape[1], k.shape[2]
    if tuple(v.shape) != tuple(k.shape) or k.shape[0] != B or k.shape[3] != d:
        raise ValueError("k and v must be [B, Hkv, Lk, d] matching q")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if alibi_slopes is not None:
        _req(alibi_slopes, "alibi_slopes", torch.float32, 1)
    pin = q.is_pinned()
    if out is None:
        out = torch.empty(q.shape, dtype=torch.bfloat16, pin_memory=pin)
    if lse is None and with_lse:
        lse = torch.empty((B, Hq, Lq), dtype=torch.float32, pin_memory=pin)
    if out is not None:
        _req_host(out, "out", torch.bfloat16, 4)
    if lse is not None:
        _req_host(lse, "lse", torch.float32, 3)
    if workspace is None:
        workspace = prefill_host_workspace(B, Hq, Hkv, Lq, Lk, d)
    opts = PrefillOptions(int(bool(causal)), float(scale),
                          None if alibi_slopes is None else alibi_slopes.data_ptr(),
                          float(softcap), int(window[0]), int(window[1]), IMPLS[impl])
    st = lib().attn_prefill_host(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, Hq, Hkv, Lq,
                                 Lk, d, ctypes.byref(opts), int(chunk_kv_heads), _ptr(workspace),
                                 workspace.numel() * workspace.element_size(), _stream())
    _check(st, "attn_prefill_host")
    if synchronize:
        torch.cuda.current_stream().synchronize()
    return out, lse


def prefill_splitkv(q, k, v, num_splits, causal=False, scale=None, alibi_slopes=None, out=None,
                    lse=None, with_lse=True, workspace=None):
    """prefill with each CTA's KV range split num_splits ways and merged by
    the log-sum-exp combine. Returns (O, LSE or None)."""
    _req(q, "q", torch.bfloat16, 4)
    _req(k, "k", torch.bfloat16, 4)
    _req(v, "v", torch.bfloat16, 4)
    B, Hq, Lq, d = q.shape
    Hkv, Lk = k.shape[1], k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if alibi_slopes is not None:
        _req(alibi_slopes, "alibi_slopes", torch.float32, 1)
    if out is None:
        out = torch.empty_like(q)
    if lse is None and with_lse:
        lse = torch.empty((B, Hq, Lq), dtype=torch.float32, device=q.device)
    nbytes = lib().attn_prefill_splitkv_workspace_bytes(B, Hq, Lq, d, int(num_splits))
    if workspace is None and nbytes:
        workspace = torch.empty(nbytes // 4, dtype=torch.float32, device=q.device)
    wsb = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib().attn_prefill_splitkv(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, Hq, Hkv,
                                    Lq, Lk, d, int(bool(causal)), float(scale),
                                    _ptr(alibi_slopes), int(num_splits), _ptr(workspace), wsb,
                                    _stream())
    _check(st, "attn_prefill_splitkv")
    return out, lse


def backward(q, k, v, o, lse, dout, causal=False, scale=None, alibi_slopes=None,
             workspace=None, impl="auto", dq=None, dk=None, dv=None):
    """Gradients of prefill: returns (dQ, dK, dV) bf16; dK and dV are per KV
    head (summed over a GQA group). `lse` is the forward's fp32 LSE. impl:
    "auto" (tcgen05 for head dim 128), "tcgen05" or "mma_sync". dq / dk / dv:
    optional output tensors shaped like q / k / v."""
    for t, n in ((q, "q"), (o, "o"), (dout, "dout")):
        _req(t, n, torch.bfloat16, 4)
    _req(k, "k", torch.bfloat16, 4)
    _req(v, "v", torch.bfloat16, 4)
    _req(lse, "lse", torch.float32, 3)
    B, Hq, Lq, d = q.shape
    Hkv, Lk = k.shape[1], k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if alibi_slopes is not None:
        _req(alibi_slopes, "alibi_slopes", torch.float32, 1)
    nbytes = lib().attn_backward_workspace_bytes(B, Hq, Lq, d)
    if workspace is None:
        workspace = torch.empty(nbytes // 4, dtype=torch.float32, device=q.device)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    for t, ref, n in ((dq, q, "dq"), (dk, k, "dk"), (dv, v, "dv")):
        _req(t, n, torch.bfloat16, 4)
        if t.shape != ref.shape:
            raise ValueError(f"{n} must be shaped like its input")
    st = lib().attn_backward_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(lse),
                                _ptr(dq), _ptr(dk), _ptr(dv), B, Hq, Hkv, Lq, Lk, d,
                                int(bool(causal)), float(scale), _ptr(alibi_slopes),
                                _ptr(workspace), workspace.numel() * workspace.element_size(),
                                IMPLS[impl], _stream())
    _check(st, "attn_backward")
    return dq, dk, dv


RMS_FORMS = {"auto": 0, "fused": 1, "two_pass": 2}


def rmsnorm_matmul_ws_bytes(B, H) -> int:
    return int(lib().attn_rmsnorm_matmul_ws_bytes(B, H))


def rmsnorm_matmul(x, g, w, eps=0.0, splits=0, out=None, rms=None, with_rms=False,
                   batch_tile=0, chained=False, form=None, workspace=None):
    """Fused RMSNorm + product: O = ((x * g) @ w) / RMS(x), RMS(x) =
    sqrt(mean(x^2) + eps). x [B,H], g [H], w [H,D] bf16 CUDA. Returns
    (O bf16 [B,D], RMS fp32 [B] or None). batch_tile / splits: 0 = auto.
    form: None = the single fused kernel; "auto" / "fused" / "two_pass" go
    through the workspace entry ("auto": the two-pass form, a separate
    conversion pass then the product); workspace: uint8 CUDA tensor,
    allocated when not given."""
    _req(x, "x", torch.bfloat16, 2)
    _req(g, "g", torch.bfloat16, 1)
    _req(w, "w", torch.bfloat16, 2)
    B, H = x.shape
    D = w.shape[1]
    if g.shape[0] != H or w.shape[0] != H:
        raise ValueError("g must be [H] and w [H, D] matching x [B, H]")
    if out is None:
        out = torch.empty((B, D), dtype=torch.bfloat16, device=x.device)
    if rms is None and with_rms:
        rms = torch.empty((B,), dtype=torch.float32, device=x.device)
    if form is not None:
        if splits or batch_tile:
            raise ValueError("the workspace entry chooses its own tiling")
        if form not in RMS_FORMS:
            raise ValueError(f"form must be one of {sorted(RMS_FORMS)}")
        nbytes = rmsnorm_matmul_ws_bytes(B, H)
        if workspace is None:
            workspace = torch.empty((max(nbytes, 1),), dtype=torch.uint8, device=x.device)
        fn = lib().attn_rmsnorm_matmul_ws_chained if chained else lib().attn_rmsnorm_matmul_ws
        st = fn(_ptr(x), _ptr(g), _ptr(w), _ptr(out), _ptr(rms), B, H, D, float(eps),
                RMS_FORMS[form], _ptr(workspace), workspace.numel() * workspace.element_size(),
                _stream())
    elif chained:
        # launched as a programmatic dependent of the kernel before it on the
        # stream; w must not be written by that kernel (automatic tiling)
        if splits or batch_tile:
            raise ValueError("chained calls choose their own tiling")
        st = lib().attn_rmsnorm_matmul_chained(_ptr(x), _ptr(g), _ptr(w), _ptr(out), _ptr(rms),
                                               B, H, D, float(eps), _stream())
    else:
        st = lib().attn_rmsnorm_matmul_tiled(_ptr(x), _ptr(g), _ptr(w), _ptr(out), _ptr(rms), B,
                                             H, D, float(eps), int(batch_tile), int(splits),
                                             _stream())
    _check(st, "attn_rmsnorm_matmul")
    return out, rms


def resolve_splits(B, Hkv, Lk_max, d, requested=0) -> int:
    s = lib().attn_decode_num_splits(B, Hkv, Lk_max, d, requested)
    if s <= 0:
        raise AttnError(-s, "attn_decode_num_splits")
    return s


def split_len(Lk_max, S) -> int:
    c = lib().attn_decode_split_len(Lk_max, S)
    if c <= 0:
        raise AttnError(-c, "attn_decode_split_len")
    return c


def decode_splitk(q, k, v, kv_lens=None, scale=None, num_splits=0, o_part=None, lse_part=None):
    """Split-K local reductions. q [B,Hq,d], k/v [B,Hkv,Lk_max,d] bf16 CUDA,
    kv_lens int32 [B] CUDA or None. Returns (O_part fp32 [B,Hq,S,d],
    LSE_part fp32 [B,Hq,S])."""
    _req(q, "q", torch.bfloat16, 3)
    _req(k, "k", torch.bfloat16, 4)
    _req(v, "v", torch.bfloat16, 4)
    B, Hq, d = q.shape
    Hkv, Lk_max = k.shape[1], k.shape[2]
    if tuple(v.shape) != tuple(k.shape) or k.shape[0] != B or k.shape[3] != d:
        raise ValueError("k and v must be [B, Hkv, Lk_max, d] matching q")
    if kv_lens is not None:
        _req(kv_lens, "kv_lens", torch.int32, 1)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    S = resolve_splits(B, Hkv, Lk_max, d, num_splits)
    if o_part is None:
        o_part = torch.empty((B, Hq, S, d), dtype=torch.float32, device=q.device)
    if lse_part is None:
        lse_part = torch.empty((B, Hq, S), dtype=torch.float32, device=q.device)
    out_s = ctypes.c_int(0)
    st = lib().attn_decode_splitk(_ptr(q), _ptr(k), _ptr(v), _ptr(kv_lens), B, Hq, Hkv, Lk_max, d,
                                  float(scale), S, ctypes.byref(out_s), _ptr(o_part),
                                  _ptr(lse_part), _stream())
    _check(st, "attn_decode_splitk")
    return o_part, lse_part


def combine(o_part, lse_part, out=None, lse=None, with_lse=True):
    """Log-sum-exp merge of split partials -> (O bf16 [B,Hq,d], LSE fp32 [B,Hq])."""
    _req(o_part, "o_part", torch.float32, 4)
    _req(lse_part, "lse_part", torch.float32, 3)
    B, Hq, S, d = o_part.shape
    if out is None:
        out = torch.empty((B, Hq, d), dtype=torch.bfloat16, device=o_part.device)
    if lse is None and with_lse:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=o_part.device)
    st = lib().attn_combine(_ptr(o_part), _ptr(lse_part), B, Hq, S, d, _ptr(out), _ptr(lse),
                            _stream())
    _check(st, "attn_combine")
    return out, lse


def decode(q, k, v, kv_lens=None, scale=None, num_splits=0, o_part=None, lse_part=None,
           out=None, lse=None):
    """Split-K decode followed by the combine, on the current stream."""
    _req(q, "q", torch.bfloat16, 3)
    B, Hq, d = q.shape
    Hkv, Lk_max = k.shape[1], k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    S = resolve_splits(B, Hkv, Lk_max, d, num_splits)
    if o_part is None:
        o_part = torch.empty((B, Hq, S, d), dtype=torch.float32, device=q.device)
    if lse_part is None:
        lse_part = torch.empty((B, Hq, S), dtype=torch.float32, device=q.device)
    if out is None:
        out = torch.empty((B, Hq, d), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    _req(k, "k", torch.bfloat16, 4)
    _req(v, "v", torch.bfloat16, 4)
    if kv_lens is not None:
        _req(kv_lens, "kv_lens", torch.int32, 1)
    st = lib().attn_decode(_ptr(q), _ptr(k), _ptr(v), _ptr(kv_lens), B, Hq, Hkv, Lk_max, d,
                           float(scale), S, _ptr(o_part), _ptr(lse_part), _ptr(out), _ptr(lse),
                           _stream())
    _check(st, "attn_decode")
    return out, lse


def decode_noalloc(q, k, v, kv_lens=None, scale=None, num_splits=0, out=None, lse=None):
    """Split-K decode + combine with the partials kept in the library's own
    fixed device array (for callers that cannot allocate). Outputs are still
    caller tensors; see attn_decode_noalloc in include/attn.h for the limit."""
    _req(q, "q", torch.bfloat16, 3)
    _req(k, "k", torch.bfloat16, 4)
    _req(v, "v", torch.bfloat16, 4)
    if kv_lens is not None:
        _req(kv_lens, "kv_lens", torch.int32, 1)
    B, Hq, d = q.shape
    Hkv, Lk_max = k.shape[1], k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty((B, Hq, d), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    st = lib().attn_decode_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(kv_lens), B, Hq, Hkv, Lk_max,
                                   d, float(scale), num_splits, _ptr(out), _ptr(lse), _stream())
    _check(st, "attn_decode_noalloc")
    return out, lse


def selftest_wait_timeout(limit_ms: int = 100):
    """Runs the bounded-wait self-test kernel on the current stream; the
    device status word then reads ATTN_ERR_TIMEOUT (see device_status)."""
    _check(lib().attn_selftest_wait_timeout(int(limit_ms), _stream()), "attn_selftest_wait_timeout")


def selftest_prefill_abort(q, k, v, skip_entry, limit_ms=100, causal=False, scale=None,
                           out=None, lse=None, impl="tcgen05"):
    """The tcgen05 prefill (impl "tcgen05" or "tcgen05_1tile") whose first
    CTA's producer stops before K/V ring entry skip_entry, with every wait
    limited to limit_ms: that CTA must record ATTN_ERR_TIMEOUT and return (see
    device_status). Returns (O, LSE)."""
    _req(q, "q", torch.bfloat16, 4)
    _req(k, "k", torch.bfloat16, 4)
    _req(v, "v", torch.bfloat16, 4)
    B, Hq, Lq, d = q.shape
    Hkv, Lk = k.shape[1], k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, Hq, Lq), dtype=torch.float32, device=q.device)
    st = lib().attn_selftest_prefill_abort(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, Hq,
                                           Hkv, Lq, Lk, d, int(bool(causal)), float(scale),
                                           int(skip_entry), int(limit_ms), IMPLS[impl],
                                           _stream())
    _check(st, "attn_selftest_prefill_abort")
    return out, lse


def device_status() -> int:
    """Synchronises the current stream and returns/clears the device status word."""
    return lib().attn_device_status(_stream())

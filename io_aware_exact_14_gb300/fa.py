"""Thin ctypes binding over libfa.so (argument marshalling only).

The same names as the C ABI in ``include/fa.h``.  Tensors are torch CUDA
tensors used only as device memory; every step of the computation runs in the
library's kernels.  There is no fallback: a missing library, a missing GPU or
a non-zero status raises.
"""
from __future__ import annotations

import ctypes
import math
import os
from typing import Optional, Tuple

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libfa.so")

FA_OK = 0
FA_ERR_INVALID_ARG, FA_ERR_UNSUPPORTED, FA_ERR_CUDA, FA_ERR_WORKSPACE, FA_ERR_TIMEOUT = 1, 2, 3, 4, 5
STATUS_NAMES = {0: "FA_OK", 1: "FA_ERR_INVALID_ARG", 2: "FA_ERR_UNSUPPORTED", 3: "FA_ERR_CUDA",
                4: "FA_ERR_WORKSPACE", 5: "FA_ERR_TIMEOUT"}

_lib = None

_P = ctypes.c_void_p
_I = ctypes.c_int
_F = ctypes.c_float
_SZ = ctypes.c_size_t

SIGNATURES = {
    "fa_fwd": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _F, _I, _P]),
    "fa_fwd_strided": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _F, _I, _P]),
    "fa_bwd_strided": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                            _I, _I, _I, _I, _F, _I, _P, _SZ, _P]),
    "fa_fwd_splitkv": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _I, _I, _P, _SZ, _P]),
    "fa_fwd_splitkv_workspace_bytes": (_SZ, [_I, _I, _I, _I, _I, _I]),
    "fa_bwd_workspace_bytes": (_SZ, [_I, _I, _I, _I]),
    "fa_bwd": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _F, _I, _P, _SZ, _P]),
    "fa_fwd_dropout": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _F, _I, _P, _P]),
    "fa_bwd_dropout": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _F, _I, _P, _P, _SZ, _P]),
    "fa_fp8_quantize": (_I, [_P, _P, _P, _I, _I, _I, _I, _I, _I, ctypes.c_ulonglong, _P]),
    "fa_fp8_vt_ld": (_SZ, [_I]),
    "fa_fwd_fp8": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _F, _I, _P]),
    "fa_fwd_fp8_splitkv": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _I, _I, _P, _SZ, _P]),
    "fa_fwd_fp8_splitkv_workspace_bytes": (_SZ, [_I, _I, _I, _I, _I, _I]),
    "fa_bwd_noalloc": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _F, _I, _P]),
    "fa_bwd_preprocess": (_I, [_P, _P, _P, _I, _I, _I, _I, _P]),
    "fa_bwd_dkdv": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _F, _I, _P]),
    "fa_bwd_dq": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _F, _I, _P]),
    "fa_debug_fwd_withhold": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _F, _I, _I, ctypes.c_uint, _P]),
    "fa_status_string": (ctypes.c_char_p, [_I]),
    "fa_debug_status": (_I, [_I]),
    "fa_debug_site": (ctypes.c_uint, []),
    "fa_last_error_detail": (ctypes.c_char_p, []),
}


class FaStrides(ctypes.Structure):
    """fa_strides: element strides (b, h, n) of a [B, H, N, d] view, d contiguous."""
    _fields_ = [("b", ctypes.c_longlong), ("h", ctypes.c_longlong), ("n", ctypes.c_longlong)]


class FaDropout(ctypes.Structure):
    """fa_dropout: drop probability p, Philox key `seed` and counter word `offset`."""
    _fields_ = [("p", ctypes.c_float), ("seed", ctypes.c_ulonglong), ("offset", ctypes.c_uint)]


class FAError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        msg = f"{fn} failed: {status_string(status)}"
        if status == 3:
            try:
                msg += f" [{load().fa_last_error_detail().decode()}]"
            except Exception:
                pass
        super().__init__(msg)


def load(path: str = LIB_PATH):
    """Load libfa.so (once) and declare its signatures.  Raises if absent."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is not built: run `python -c \"import __graft_entry__ as g; g.build()\"`")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def status_string(status: int) -> str:
    try:
        return load().fa_status_string(int(status)).decode()
    except Exception:
        return STATUS_NAMES.get(int(status), f"status {status}")


def _check(fn: str, status: int):
    if status != FA_OK:
        raise FAError(fn, status)


def _stream_ptr(stream: Optional[torch.cuda.Stream]) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return int(s.cuda_stream)


def _bhnd(t: torch.Tensor, name: str) -> Tuple[int, int, int, int]:
    if not isinstance(t, torch.Tensor) or t.dim() != 4:
        raise ValueError(f"{name} must be a 4-D [B, H, N, d] tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (device memory)")
    if t.dtype != torch.bfloat16:
        raise ValueError(f"{name} must be bfloat16")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return tuple(t.shape)


def _same(shape, t: torch.Tensor, name: str):
    if _bhnd(t, name) != shape:
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {shape}")


def _vec(t: torch.Tensor, shape, name: str):
    if not (t.is_cuda and t.dtype == torch.float32 and t.is_contiguous() and tuple(t.shape) == tuple(shape[:3])):
        raise ValueError(f"{name} must be a contiguous fp32 CUDA tensor of shape {tuple(shape[:3])}")


def default_scale(d: int) -> float:
    return 1.0 / math.sqrt(d)


# ---------------------------------------------------------------------------
# Calls
# ---------------------------------------------------------------------------

def fa_fwd(q, k, v, scale: Optional[float] = None, causal: bool = False, out=None, lse=None, stream=None):
    """O, LSE = attention(q, k, v): bf16 [B, H, N, d] in, O bf16 and LSE fp32 [B, H, N] out."""
    shape = _bhnd(q, "q")
    _same(shape, k, "k")
    _same(shape, v, "v")
    B, H, N, d = shape
    scale = default_scale(d) if scale is None else float(scale)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    _same(shape, out, "out")
    _vec(lse, shape, "lse")
    st = load().fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                       B, H, N, d, scale, int(bool(causal)), _stream_ptr(stream))
    _check("fa_fwd", st)
    return out, lse


def _view(t: torch.Tensor, name: str):
    """Shape and fa_strides of a [B, H, N, d] bf16 CUDA view whose last dim is contiguous."""
    if not isinstance(t, torch.Tensor) or t.dim() != 4:
        raise ValueError(f"{name} must be a 4-D [B, H, N, d] view")
    if not t.is_cuda or t.dtype != torch.bfloat16:
        raise ValueError(f"{name} must be a bfloat16 CUDA tensor")
    if t.stride(3) != 1:
        raise ValueError(f"{name} must have a contiguous last (d) dimension")
    sb, sh, sn = t.stride()[:3]
    return tuple(t.shape), FaStrides(sb, sh, sn)


def fa_fwd_strided(q, k, v, scale: Optional[float] = None, causal: bool = False, out=None, lse=None, stream=None):
    """fa_fwd on [B, H, N, d] views of any layout that keeps d contiguous (for example
    x.transpose(1, 2) of a [B, N, H, d] tensor); `out` may be such a view too."""
    shape, qs = _view(q, "q")
    ks, vs = _view(k, "k"), _view(v, "v")
    for (sh, _), n in ((ks, "k"), (vs, "v")):
        if sh != shape:
            raise ValueError(f"{n} has shape {sh}, expected {shape}")
    B, H, N, d = shape
    scale = default_scale(d) if scale is None else float(scale)
    if out is None:
        out = torch.empty(shape, dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    oshape, os_ = _view(out, "out")
    if oshape != shape:
        raise ValueError(f"out has shape {oshape}, expected {shape}")
    _vec(lse, shape, "lse")
    st = load().fa_fwd_strided(q.data_ptr(), ctypes.addressof(qs), k.data_ptr(), ctypes.addressof(ks[1]),
                               v.data_ptr(), ctypes.addressof(vs[1]), out.data_ptr(), ctypes.addressof(os_),
                               lse.data_ptr(), B, H, N, d, scale, int(bool(causal)), _stream_ptr(stream))
    _check("fa_fwd_strided", st)
    return out, lse


def fa_bwd_strided(q, k, v, o, lse, do, scale: Optional[float] = None, causal: bool = False,
                   dq=None, dk=None, dv=None, workspace=None, stream=None):
    """fa_bwd on [B, H, N, d] views (d contiguous); dq, dk, dv may be views into one
    buffer (for example a packed [B, N, 3, H, d] gradient)."""
    shape, qs = _view(q, "q")
    views = {"k": _view(k, "k"), "v": _view(v, "v"), "o": _view(o, "o"), "do": _view(do, "do")}
    for n, (sh, _) in views.items():
        if sh != shape:
            raise ValueError(f"{n} has shape {sh}, expected {shape}")
    _vec(lse, shape, "lse")
    B, H, N, d = shape
    scale = default_scale(d) if scale is None else float(scale)
    grads = []
    for t, n in ((dq, "dq"), (dk, "dk"), (dv, "dv")):
        t = torch.empty(shape, dtype=torch.bfloat16, device=q.device) if t is None else t
        sh, st_ = _view(t, n)
        if sh != shape:
            raise ValueError(f"{n} has shape {sh}, expected {shape}")
        grads.append((t, st_))
    need = fa_bwd_workspace_bytes(B, H, N, d)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    a = ctypes.addressof
    st = load().fa_bwd_strided(q.data_ptr(), a(qs), k.data_ptr(), a(views["k"][1]), v.data_ptr(), a(views["v"][1]),
                               o.data_ptr(), a(views["o"][1]), lse.data_ptr(), do.data_ptr(), a(views["do"][1]),
                               grads[0][0].data_ptr(), a(grads[0][1]), grads[1][0].data_ptr(), a(grads[1][1]),
                               grads[2][0].data_ptr(), a(grads[2][1]), B, H, N, d, scale, int(bool(causal)),
                               workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                               _stream_ptr(stream))
    _check("fa_bwd_strided", st)
    return grads[0][0], grads[1][0], grads[2][0]


def fa_fwd_splitkv_workspace_bytes(B: int, H: int, Nq: int, Nk: int, d: int, num_splits: int = 0) -> int:
    return int(load().fa_fwd_splitkv_workspace_bytes(B, H, Nq, Nk, d, int(num_splits)))


def fa_fwd_splitkv(q, k, v, scale: Optional[float] = None, num_splits: int = 0, out=None, lse=None,
                   workspace=None, stream=None, causal: bool = False):
    """O, LSE for q [B, H, Nq, d] against k, v [B, H, Nk, d], the keys cut into
    `num_splits` chunks (<= 0: the library's choice) merged by their LSE; causal:
    query i sits at position Nk - Nq + i and sees the keys up to it."""
    qs = _bhnd(q, "q")
    ks = _bhnd(k, "k")
    _same(ks, v, "v")
    B, H, Nq, d = qs
    if ks[0] != B or ks[1] != H or ks[3] != d:
        raise ValueError(f"k has shape {ks}, expected [{B}, {H}, Nk, {d}]")
    Nk = ks[2]
    scale = default_scale(d) if scale is None else float(scale)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    _same(qs, out, "out")
    _vec(lse, qs, "lse")
    need = fa_fwd_splitkv_workspace_bytes(B, H, Nq, Nk, d, num_splits)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    st = load().fa_fwd_splitkv(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                               B, H, Nq, Nk, d, scale, int(bool(causal)), int(num_splits), workspace.data_ptr(),
                               workspace.numel() * workspace.element_size(), _stream_ptr(stream))
    _check("fa_fwd_splitkv", st)
    return out, lse


def fa_bwd_workspace_bytes(B: int, H: int, N: int, d: int) -> int:
    return int(load().fa_bwd_workspace_bytes(B, H, N, d))


def fa_bwd(q, k, v, o, lse, do, scale: Optional[float] = None, causal: bool = False,
           dq=None, dk=None, dv=None, workspace=None, stream=None):
    """dQ, dK, dV for upstream gradient `do`, recomputing P from `lse`."""
    shape = _bhnd(q, "q")
    for t, n in ((k, "k"), (v, "v"), (o, "o"), (do, "do")):
        _same(shape, t, n)
    _vec(lse, shape, "lse")
    B, H, N, d = shape
    scale = default_scale(d) if scale is None else float(scale)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(q) if dk is None else dk
    dv = torch.empty_like(q) if dv is None else dv
    for t, n in ((dq, "dq"), (dk, "dk"), (dv, "dv")):
        _same(shape, t, n)
    need = fa_bwd_workspace_bytes(B, H, N, d)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    st = load().fa_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), do.data_ptr(),
                       dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, N, d, scale, int(bool(causal)),
                       workspace.data_ptr(), workspace.numel() * workspace.element_size(), _stream_ptr(stream))
    _check("fa_bwd", st)
    return dq, dk, dv


def fa_fwd_dropout(q, k, v, p: float, seed: int, offset: int = 0, scale: Optional[float] = None,
                   causal: bool = False, out=None, lse=None, stream=None):
    """fa_fwd with dropout on the probabilities: O = (P o M~) V and the plain LSE."""
    shape = _bhnd(q, "q")
    _same(shape, k, "k")
    _same(shape, v, "v")
    B, H, N, d = shape
    scale = default_scale(d) if scale is None else float(scale)
    out = torch.empty_like(q) if out is None else out
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    _same(shape, out, "out")
    _vec(lse, shape, "lse")
    drop = FaDropout(float(p), int(seed), int(offset))
    st = load().fa_fwd_dropout(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                               B, H, N, d, scale, int(bool(causal)), ctypes.addressof(drop), _stream_ptr(stream))
    _check("fa_fwd_dropout", st)
    return out, lse


def fa_bwd_dropout(q, k, v, o, lse, do, p: float, seed: int, offset: int = 0, scale: Optional[float] = None,
                   causal: bool = False, dq=None, dk=None, dv=None, workspace=None, stream=None):
    """fa_bwd for fa_fwd_dropout with the same (p, seed, offset): the same mask."""
    shape = _bhnd(q, "q")
    for t, n in ((k, "k"), (v, "v"), (o, "o"), (do, "do")):
        _same(shape, t, n)
    _vec(lse, shape, "lse")
    B, H, N, d = shape
    scale = default_scale(d) if scale is None else float(scale)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(q) if dk is None else dk
    dv = torch.empty_like(q) if dv is None else dv
    for t, n in ((dq, "dq"), (dk, "dk"), (dv, "dv")):
        _same(shape, t, n)
    need = fa_bwd_workspace_bytes(B, H, N, d)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    drop = FaDropout(float(p), int(seed), int(offset))
    st = load().fa_bwd_dropout(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                               do.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, N, d, scale,
                               int(bool(causal)), ctypes.addressof(drop), workspace.data_ptr(),
                               workspace.numel() * workspace.element_size(), _stream_ptr(stream))
    _check("fa_bwd_dropout", st)
    return dq, dk, dv


def fa_fp8_vt_ld(N: int) -> int:
    return int(load().fa_fp8_vt_ld(N))


def fa_fp8_quantize(x, transpose: bool = False, rotate_seed: Optional[int] = None, out=None, descale=None,
                    stream=None):
    """e4m3 codes (uint8) of a contiguous bf16 [B, H, N, d] tensor, per-(b, h) descale
    (fp32 [B, H]); transpose=True gives [B, H, d, fa_fp8_vt_ld(N)] (the V layout of
    fa_fwd_fp8); rotate_seed applies the random-sign Hadamard rotation first."""
    B, H, N, d = _bhnd(x, "x")
    shape = (B, H, d, fa_fp8_vt_ld(N)) if transpose else (B, H, N, d)
    out = torch.empty(shape, dtype=torch.uint8, device=x.device) if out is None else out
    if tuple(out.shape) != shape or out.dtype != torch.uint8 or not out.is_contiguous() or not out.is_cuda:
        raise ValueError(f"out must be a contiguous uint8 CUDA tensor of shape {shape}")
    descale = torch.empty((B, H), dtype=torch.float32, device=x.device) if descale is None else descale
    if tuple(descale.shape) != (B, H) or descale.dtype != torch.float32 or not descale.is_contiguous():
        raise ValueError("descale must be a contiguous fp32 [B, H] tensor")
    rotate = rotate_seed is not None
    st = load().fa_fp8_quantize(x.data_ptr(), out.data_ptr(), descale.data_ptr(), B, H, N, d, int(transpose),
                                int(rotate), int(rotate_seed or 0), _stream_ptr(stream))
    _check("fa_fp8_quantize", st)
    return out, descale


def fa_fwd_fp8(q8, k8, vt8, descale_q, descale_k, descale_v, scale: Optional[float] = None, causal: bool = False,
               out=None, lse=None, stream=None):
    """Forward on e4m3 codes (uint8): q8, k8 [B, H, N, d], vt8 [B, H, d, fa_fp8_vt_ld(N)],
    descales fp32 [B, H]; returns bf16 O [B, H, N, d] and fp32 LSE [B, H, N]."""
    for t, n in ((q8, "q8"), (k8, "k8"), (vt8, "vt8")):
        if not (isinstance(t, torch.Tensor) and t.is_cuda and t.dtype == torch.uint8 and t.is_contiguous()
                and t.dim() == 4):
            raise ValueError(f"{n} must be a contiguous 4-D uint8 CUDA tensor")
    B, H, N, d = q8.shape
    if tuple(k8.shape) != (B, H, N, d) or tuple(vt8.shape) != (B, H, d, fa_fp8_vt_ld(N)):
        raise ValueError("k8 must match q8 and vt8 must be [B, H, d, fa_fp8_vt_ld(N)]")
    for t, n in ((descale_q, "descale_q"), (descale_k, "descale_k"), (descale_v, "descale_v")):
        if not (t.is_cuda and t.dtype == torch.float32 and t.is_contiguous() and tuple(t.shape) == (B, H)):
            raise ValueError(f"{n} must be a contiguous fp32 CUDA tensor [B, H]")
    scale = default_scale(d) if scale is None else float(scale)
    out = torch.empty((B, H, N, d), dtype=torch.bfloat16, device=q8.device) if out is None else out
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q8.device) if lse is None else lse
    _same((B, H, N, d), out, "out")
    _vec(lse, (B, H, N, d), "lse")
    st = load().fa_fwd_fp8(q8.data_ptr(), k8.data_ptr(), vt8.data_ptr(), descale_q.data_ptr(), descale_k.data_ptr(),
                           descale_v.data_ptr(), out.data_ptr(), lse.data_ptr(), B, H, N, d, scale,
                           int(bool(causal)), _stream_ptr(stream))
    _check("fa_fwd_fp8", st)
    return out, lse


def fa_fwd_fp8_splitkv_workspace_bytes(B: int, H: int, Nq: int, Nk: int, d: int, num_splits: int = 0) -> int:
    return int(load().fa_fwd_fp8_splitkv_workspace_bytes(B, H, Nq, Nk, d, int(num_splits)))


def fa_fwd_fp8_splitkv(q8, k8, vt8, descale_q, descale_k, descale_v, scale: Optional[float] = None,
                       num_splits: int = 0, out=None, lse=None, workspace=None, stream=None, causal: bool = False):
    """Split-KV forward on e4m3 codes (uint8): q8 [B, H, Nq, d], k8 [B, H, Nk, d],
    vt8 [B, H, d, fa_fp8_vt_ld(Nk)], descales fp32 [B, H]; returns bf16 O [B, H, Nq, d] and
    fp32 LSE [B, H, Nq]; causal as in fa_fwd_splitkv."""
    for t, n in ((q8, "q8"), (k8, "k8"), (vt8, "vt8")):
        if not (isinstance(t, torch.Tensor) and t.is_cuda and t.dtype == torch.uint8 and t.is_contiguous()
                and t.dim() == 4):
            raise ValueError(f"{n} must be a contiguous 4-D uint8 CUDA tensor")
    B, H, Nq, d = q8.shape
    Nk = k8.shape[2]
    if tuple(k8.shape) != (B, H, Nk, d) or tuple(vt8.shape) != (B, H, d, fa_fp8_vt_ld(Nk)):
        raise ValueError("k8 must be [B, H, Nk, d] and vt8 [B, H, d, fa_fp8_vt_ld(Nk)]")
    for t, n in ((descale_q, "descale_q"), (descale_k, "descale_k"), (descale_v, "descale_v")):
        if not (t.is_cuda and t.dtype == torch.float32 and t.is_contiguous() and tuple(t.shape) == (B, H)):
            raise ValueError(f"{n} must be a contiguous fp32 CUDA tensor [B, H]")
    scale = default_scale(d) if scale is None else float(scale)
    out = torch.empty((B, H, Nq, d), dtype=torch.bfloat16, device=q8.device) if out is None else out
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q8.device) if lse is None else lse
    _same((B, H, Nq, d), out, "out")
    _vec(lse, (B, H, Nq, d), "lse")
    need = fa_fwd_fp8_splitkv_workspace_bytes(B, H, Nq, Nk, d, num_splits)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q8.device)
    st = load().fa_fwd_fp8_splitkv(q8.data_ptr(), k8.data_ptr(), vt8.data_ptr(), descale_q.data_ptr(),
                                   descale_k.data_ptr(), descale_v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                                   B, H, Nq, Nk, d, scale, int(bool(causal)), int(num_splits), workspace.data_ptr(),
                                   workspace.numel() * workspace.element_size(), _stream_ptr(stream))
    _check("fa_fwd_fp8_splitkv", st)
    return out, lse


def fa_bwd_noalloc(q, k, v, o, lse, do, scale: Optional[float] = None, causal: bool = False,
                   dq=None, dk=None, dv=None, stream=None):
    """fa_bwd for callers that cannot allocate: the library's built-in scratch holds
    the row term, so only the gradients are caller memory (B*H*N <= 2^21)."""
    shape = _bhnd(q, "q")
    for t, n in ((k, "k"), (v, "v"), (o, "o"), (do, "do")):
        _same(shape, t, n)
    _vec(lse, shape, "lse")
    B, H, N, d = shape
    scale = default_scale(d) if scale is None else float(scale)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(q) if dk is None else dk
    dv = torch.empty_like(q) if dv is None else dv
    for t, n in ((dq, "dq"), (dk, "dk"), (dv, "dv")):
        _same(shape, t, n)
    st = load().fa_bwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                               do.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, N, d, scale,
                               int(bool(causal)), _stream_ptr(stream))
    _check("fa_bwd_noalloc", st)
    return dq, dk, dv


def fa_bwd_preprocess(o, do, Dvec=None, stream=None):
    shape = _bhnd(o, "o")
    _same(shape, do, "do")
    B, H, N, d = shape
    if Dvec is None:
        Dvec = torch.empty((B, H, N), dtype=torch.float32, device=o.device)
    _vec(Dvec, shape, "Dvec")
    _check("fa_bwd_preprocess", load().fa_bwd_preprocess(o.data_ptr(), do.data_ptr(), Dvec.data_ptr(),
                                                          B, H, N, d, _stream_ptr(stream)))
    return Dvec


def fa_bwd_dkdv(q, k, v, lse, do, Dvec, scale: Optional[float] = None, causal: bool = False,
                dk=None, dv=None, stream=None):
    shape = _bhnd(q, "q")
    for t, n in ((k, "k"), (v, "v"), (do, "do")):
        _same(shape, t, n)
    _vec(lse, shape, "lse")
    _vec(Dvec, shape, "Dvec")
    B, H, N, d = shape
    scale = default_scale(d) if scale is None else float(scale)
    dk = torch.empty_like(q) if dk is None else dk
    dv = torch.empty_like(q) if dv is None else dv
    _check("fa_bwd_dkdv", load().fa_bwd_dkdv(q.data_ptr(), k.data_ptr(), v.data_ptr(), lse.data_ptr(),
                                              do.data_ptr(), Dvec.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                                              B, H, N, d, scale, int(bool(causal)), _stream_ptr(stream)))
    return dk, dv


def fa_bwd_dq(q, k, v, lse, do, Dvec, scale: Optional[float] = None, causal: bool = False, dq=None,
              stream=None):
    shape = _bhnd(q, "q")
    for t, n in ((k, "k"), (v, "v"), (do, "do")):
        _same(shape, t, n)
    _vec(lse, shape, "lse")
    _vec(Dvec, shape, "Dvec")
    B, H, N, d = shape
    scale = default_scale(d) if scale is None else float(scale)
    dq = torch.empty_like(q) if dq is None else dq
    _check("fa_bwd_dq", load().fa_bwd_dq(q.data_ptr(), k.data_ptr(), v.data_ptr(), lse.data_ptr(),
                                          do.data_ptr(), Dvec.data_ptr(), dq.data_ptr(),
                                          B, H, N, d, scale, int(bool(causal)), _stream_ptr(stream)))
    return dq


def fa_debug_fwd_withhold(q, k, v, withhold_group: int, wait_limit_us: int, scale: Optional[float] = None,
                          causal: bool = False, out=None, lse=None, stream=None):
    """Test hook of the deadlock guard: fa_fwd whose producer withholds K/V group
    `withhold_group` and whose waits give up after `wait_limit_us`.  Returns the
    status code (the launch itself succeeds; the timeout shows in fa_debug_status)."""
    shape = _bhnd(q, "q")
    _same(shape, k, "k")
    _same(shape, v, "v")
    B, H, N, d = shape
    scale = default_scale(d) if scale is None else float(scale)
    out = torch.empty_like(q) if out is None else out
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device) if lse is None else lse
    _same(shape, out, "out")
    _vec(lse, shape, "lse")
    return int(load().fa_debug_fwd_withhold(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                            lse.data_ptr(), B, H, N, d, scale, int(bool(causal)),
                                            int(withhold_group), int(wait_limit_us), _stream_ptr(stream)))


def fa_debug_status(reset: bool = False) -> int:
    """FA_OK, or FA_ERR_TIMEOUT when a kernel gave up on a wait (synchronous)."""
    return int(load().fa_debug_status(int(bool(reset))))


def fa_debug_site() -> int:
    return int(load().fa_debug_site())

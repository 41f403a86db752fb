"""Thin ctypes binding of the C ABI in include/nabla.h (libnabla.so).

Argument marshalling only: every step of the hot path runs in the library's
CUDA kernels.  torch supplies device memory (outputs and the mask-builder
workspace are allocated here with torch when the caller passes none) and the
current CUDA stream.  If the library is missing, every call raises; there is
no fallback.
"""
from __future__ import annotations

import ctypes
import math
import os
from typing import Optional, Tuple

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libnabla.so")

NABLA_OK = 0
NABLA_F32, NABLA_BF16 = 0, 1

_lib = None


class NablaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {nabla_status_string(status)} ({status})")


def load() -> ctypes.CDLL:
    """Load libnabla.so (built by __graft_entry__.build()); raise if it is absent."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: run __graft_entry__.build() first")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    lib.nabla_abi_version.restype = i32
    lib.nabla_abi_version.argtypes = []
    lib.nabla_status_string.restype = ctypes.c_char_p
    lib.nabla_status_string.argtypes = [i32]
    lib.nabla_build_mask_workspace_bytes.restype = sz
    lib.nabla_build_mask_workspace_bytes.argtypes = [i32, i32, i32, i32]
    lib.nabla_build_mask.restype = i32
    lib.nabla_build_mask.argtypes = [vp, vp, i32, i32, i32, i32, i32, vp, ctypes.c_double, vp,
                                     vp, vp, sz, vp]
    lib.nabla_build_mask_noalloc.restype = i32
    lib.nabla_build_mask_noalloc.argtypes = [vp, vp, i32, i32, i32, i32, i32, vp, ctypes.c_double,
                                             vp, vp, vp]
    lib.nabla_build_mask_topk.restype = i32
    lib.nabla_build_mask_topk.argtypes = [vp, vp, i32, i32, i32, i32, i32, ctypes.c_double, vp,
                                          vp, vp, sz, vp]
    lib.nabla_attn_fwd.restype = i32
    lib.nabla_attn_fwd.argtypes = [vp, vp, vp, i32, i32, i32, i32, i32, vp, vp, ctypes.c_float,
                                   vp, vp]
    lib.nabla_attn_bwd_workspace_bytes.restype = sz
    lib.nabla_attn_bwd_workspace_bytes.argtypes = [i32, i32, i32, i32]
    lib.nabla_attn_bwd.restype = i32
    lib.nabla_attn_bwd.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, vp, vp,
                                   ctypes.c_float, vp, vp, vp, vp, sz, vp]
    lib.nabla_attn_fwd_lse.restype = i32
    lib.nabla_attn_fwd_lse.argtypes = [vp, vp, vp, i32, i32, i32, i32, i32, vp, vp,
                                       ctypes.c_float, vp, vp, vp]
    lib.nabla_sta_mask.restype = i32
    lib.nabla_sta_mask.argtypes = [i32, i32, i32, i32, i32, i32, vp, vp]
    for name in ("nabla_fractal_flatten", "nabla_fractal_unflatten"):
        fn = getattr(lib, name)
        fn.restype = i32
        fn.argtypes = [vp, i32, i32, i32, i32, i32, i32, i32, i32, vp, vp]
    lib.nabla_selftest_bounded_wait.restype = i32
    lib.nabla_selftest_bounded_wait.argtypes = [vp]
    lib.nabla_get_last_device_status.restype = i32
    lib.nabla_get_last_device_status.argtypes = [vp]
    _lib = lib
    return lib


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(stream, device: torch.device) -> Optional[int]:
    """The cudaStream_t to launch on: the given one, else torch's current stream of
    the tensors' device (not of whichever device happens to be current)."""
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _call(device: torch.device, fn, *args) -> int:
    """Run one C-ABI call with the tensors' device current: the library launches on,
    and takes its per-device state from, the current device."""
    with torch.cuda.device(device):
        return fn(*args)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return NABLA_BF16
    if t.dtype == torch.float32:
        return NABLA_F32
    raise TypeError(f"unsupported dtype {t.dtype}")


def _check(status: int, where: str) -> None:
    if status != NABLA_OK:
        raise NablaError(status, where)


def _shape(q: torch.Tensor) -> Tuple[int, int, int, int]:
    if q.dim() != 4:
        raise ValueError("q/k/v must be [B, S, h, D]")
    if not q.is_contiguous():
        raise ValueError("q/k/v must be contiguous [B, S, h, D]")
    return tuple(q.shape)


# The C ABI receives bare pointers and cannot see a buffer's size, element type
# or device, so every tensor handed to it is checked here first: a short or
# mistyped buffer, or one in host memory, would otherwise be read or written
# out of bounds by the kernels.
def _on(t: torch.Tensor, name: str, device: torch.device) -> None:
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")


def _buf(t: torch.Tensor, name: str, numel: int, dtype: torch.dtype,
         device: torch.device) -> None:
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if t.numel() < numel:
        raise ValueError(f"{name} holds {t.numel()} elements, needs {numel}")
    _on(t, name, device)


def _cuda(t: torch.Tensor) -> None:
    if not t.is_cuda:
        raise ValueError(f"tensors must be on a CUDA device, got {t.device}")


def _csr(kv_nb: torch.Tensor, kv_inds: torch.Tensor, B: int, h: int, s1: int,
         device: torch.device) -> None:
    _buf(kv_nb, "kv_nb", B * h * s1, torch.int32, device)
    _buf(kv_inds, "kv_inds", B * h * s1 * s1, torch.int32, device)


def nabla_abi_version() -> int:
    return load().nabla_abi_version()


def nabla_status_string(status: int) -> str:
    return load().nabla_status_string(int(status)).decode()


def nabla_build_mask_workspace_bytes(B: int, S: int, h: int, D: int) -> int:
    return load().nabla_build_mask_workspace_bytes(B, S, h, D)


def nabla_build_mask(q: torch.Tensor, k: torch.Tensor, sta: torch.Tensor, thr: float,
                     kv_nb: Optional[torch.Tensor] = None,
                     kv_inds: Optional[torch.Tensor] = None,
                     workspace: Optional[torch.Tensor] = None, stream=None):
    """(q, k [B,S,h,D], sta [s1,s1] uint8, thr) -> (kv_nb [B,h,s1], kv_inds [B,h,s1,s1]) int32."""
    lib = load()
    B, S, h, D = _shape(q)
    if k.shape != q.shape or k.dtype != q.dtype:
        raise ValueError("k must match q")
    s1 = S // 64
    dev = q.device
    if kv_nb is None:
        kv_nb = torch.empty((B, h, s1), dtype=torch.int32, device=dev)
    if kv_inds is None:
        kv_inds = torch.empty((B, h, s1, s1), dtype=torch.int32, device=dev)
    _on(k, "k", dev)
    _buf(sta, "sta", s1 * s1, torch.uint8, dev)
    _csr(kv_nb, kv_inds, B, h, s1, dev)
    need = lib.nabla_build_mask_workspace_bytes(B, S, h, D)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    _on(workspace, "workspace", dev)
    _cuda(q)
    st = _call(dev, lib.nabla_build_mask, _ptr(q), _ptr(k), _dtype_code(q), B, S, h, D, _ptr(sta),
               float(thr), _ptr(kv_nb), _ptr(kv_inds), _ptr(workspace),
               workspace.numel() * workspace.element_size(), _stream(stream, dev))
    _check(st, "nabla_build_mask")
    return kv_nb, kv_inds


def nabla_build_mask_noalloc(q: torch.Tensor, k: torch.Tensor, sta: torch.Tensor, thr: float,
                             kv_nb: torch.Tensor, kv_inds: torch.Tensor, stream=None):
    """nabla_build_mask without a workspace: the library's fixed device scratch is
    used instead (see include/nabla.h); outputs must be preallocated by the caller."""
    B, S, h, D = _shape(q)
    if k.shape != q.shape or k.dtype != q.dtype:
        raise ValueError("k must match q")
    s1 = S // 64
    _on(k, "k", q.device)
    _buf(sta, "sta", s1 * s1, torch.uint8, q.device)
    _csr(kv_nb, kv_inds, B, h, s1, q.device)
    _cuda(q)
    st = _call(q.device, load().nabla_build_mask_noalloc, _ptr(q), _ptr(k), _dtype_code(q), B, S,
               h, D, _ptr(sta), float(thr), _ptr(kv_nb), _ptr(kv_inds), _stream(stream, q.device))
    _check(st, "nabla_build_mask_noalloc")
    return kv_nb, kv_inds


def nabla_build_mask_topk(q: torch.Tensor, k: torch.Tensor, topk_ratio: float,
                          kv_nb: Optional[torch.Tensor] = None,
                          kv_inds: Optional[torch.Tensor] = None,
                          workspace: Optional[torch.Tensor] = None, stream=None):
    """Top-k block selector (sla.get_block_map): (q, k [B,S,h,D], topk_ratio) ->
    (kv_nb [B,h,s1], kv_inds [B,h,s1,s1]) int32, kept blocks ascending."""
    lib = load()
    B, S, h, D = _shape(q)
    if k.shape != q.shape or k.dtype != q.dtype:
        raise ValueError("k must match q")
    s1 = S // 64
    dev = q.device
    if kv_nb is None:
        kv_nb = torch.empty((B, h, s1), dtype=torch.int32, device=dev)
    if kv_inds is None:
        kv_inds = torch.empty((B, h, s1, s1), dtype=torch.int32, device=dev)
    _on(k, "k", dev)
    _csr(kv_nb, kv_inds, B, h, s1, dev)
    need = lib.nabla_build_mask_workspace_bytes(B, S, h, D)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    _on(workspace, "workspace", dev)
    _cuda(q)
    st = _call(dev, lib.nabla_build_mask_topk, _ptr(q), _ptr(k), _dtype_code(q), B, S, h, D,
               float(topk_ratio), _ptr(kv_nb), _ptr(kv_inds), _ptr(workspace),
               workspace.numel() * workspace.element_size(), _stream(stream, dev))
    _check(st, "nabla_build_mask_topk")
    return kv_nb, kv_inds


def nabla_attn_fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, kv_nb: torch.Tensor,
                   kv_inds: torch.Tensor, scale: Optional[float] = None,
                   o: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Block-sparse attention over the kept 64x64 blocks; returns o [B,S,h,D]."""
    lib = load()
    B, S, h, D = _shape(q)
    if k.shape != q.shape or v.shape != q.shape or k.dtype != q.dtype or v.dtype != q.dtype:
        raise ValueError("k, v must match q")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if o is None:
        o = torch.empty_like(q)
    _on(k, "k", q.device)
    _on(v, "v", q.device)
    _csr(kv_nb, kv_inds, B, h, S // 64, q.device)
    _buf(o, "o", q.numel(), q.dtype, q.device)
    _cuda(q)
    st = _call(q.device, lib.nabla_attn_fwd, _ptr(q), _ptr(k), _ptr(v), _dtype_code(q), B, S, h, D,
               _ptr(kv_nb), _ptr(kv_inds), float(scale), _ptr(o), _stream(stream, q.device))
    _check(st, "nabla_attn_fwd")
    return o


def nabla_attn_bwd_workspace_bytes(B: int, S: int, h: int, D: int) -> int:
    return load().nabla_attn_bwd_workspace_bytes(B, S, h, D)


def nabla_attn_fwd_lse(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, kv_nb: torch.Tensor,
                       kv_inds: torch.Tensor, scale: Optional[float] = None,
                       o: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                       stream=None):
    """nabla_attn_fwd that also returns the rows' base-2 log-sum-exp: (o, lse [B,h,S] fp32)."""
    lib = load()
    B, S, h, D = _shape(q)
    if k.shape != q.shape or v.shape != q.shape or k.dtype != q.dtype or v.dtype != q.dtype:
        raise ValueError("k, v must match q")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    o = torch.empty_like(q) if o is None else o
    lse = torch.empty((B, h, S), dtype=torch.float32, device=q.device) if lse is None else lse
    _on(k, "k", q.device)
    _on(v, "v", q.device)
    _csr(kv_nb, kv_inds, B, h, S // 64, q.device)
    _buf(o, "o", q.numel(), q.dtype, q.device)
    _buf(lse, "lse", B * h * S, torch.float32, q.device)
    _cuda(q)
    st = _call(q.device, lib.nabla_attn_fwd_lse, _ptr(q), _ptr(k), _ptr(v), _dtype_code(q), B, S,
               h, D, _ptr(kv_nb), _ptr(kv_inds), float(scale), _ptr(o), _ptr(lse),
               _stream(stream, q.device))
    _check(st, "nabla_attn_fwd_lse")
    return o, lse


def nabla_attn_bwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, o: torch.Tensor,
                   dout: torch.Tensor, kv_nb: torch.Tensor, kv_inds: torch.Tensor,
                   scale: Optional[float] = None, dq: Optional[torch.Tensor] = None,
                   dk: Optional[torch.Tensor] = None, dv: Optional[torch.Tensor] = None,
                   workspace: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                   stream=None):
    """Gradients of nabla_attn_fwd: returns (dq, dk, dv), each [B,S,h,D] in q's dtype.
    lse: the forward's log-sum-exp from nabla_attn_fwd_lse (computed here if None)."""
    lib = load()
    B, S, h, D = _shape(q)
    for t in (k, v, o, dout):
        if t.shape != q.shape or t.dtype != q.dtype or not t.is_contiguous():
            raise ValueError("k, v, o, dout must match q")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(q) if dk is None else dk
    dv = torch.empty_like(q) if dv is None else dv
    for name, t in (("k", k), ("v", v), ("o", o), ("dout", dout)):
        _on(t, name, q.device)
    _csr(kv_nb, kv_inds, B, h, S // 64, q.device)
    for name, t in (("dq", dq), ("dk", dk), ("dv", dv)):
        _buf(t, name, q.numel(), q.dtype, q.device)
    if lse is not None:
        _buf(lse, "lse", B * h * S, torch.float32, q.device)
    need = lib.nabla_attn_bwd_workspace_bytes(B, S, h, D)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    _on(workspace, "workspace", q.device)
    _cuda(q)
    st = _call(q.device, lib.nabla_attn_bwd, _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
               _ptr(dout), _dtype_code(q), B, S, h, D, _ptr(kv_nb), _ptr(kv_inds), float(scale),
               _ptr(dq), _ptr(dk), _ptr(dv), _ptr(workspace),
               workspace.numel() * workspace.element_size(), _stream(stream, q.device))
    _check(st, "nabla_attn_bwd")
    return dq, dk, dv


def nabla_sta_mask(T: int, H: int, W: int, wt: int, wh: int, ww: int, device=None,
                   out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """STA window [s1, s1] uint8 on the (T, H, W) block grid."""
    lib = load()
    s1 = T * H * W
    if out is None:
        out = torch.empty((s1, s1), dtype=torch.uint8, device=device or "cuda")
    _buf(out, "out", s1 * s1, torch.uint8, out.device)
    _cuda(out)
    st = _call(out.device, lib.nabla_sta_mask, T, H, W, wt, wh, ww, _ptr(out),
               _stream(stream, out.device))
    _check(st, "nabla_sta_mask")
    return out


def nabla_fractal_flatten(x: torch.Tensor, P: int = 8, out: Optional[torch.Tensor] = None,
                          stream=None) -> torch.Tensor:
    """x [B, T, H, W, h, D] (raster token order) -> [B, T*H*W, h, D] in fractal order."""
    if x.dim() != 6 or not x.is_contiguous():
        raise ValueError("x must be a contiguous [B, T, H, W, h, D] tensor")
    B, T, H, W, h, D = x.shape
    if out is None:
        out = torch.empty((B, T * H * W, h, D), dtype=x.dtype, device=x.device)
    _buf(out, "out", x.numel(), x.dtype, x.device)
    _cuda(x)
    st = _call(x.device, load().nabla_fractal_flatten, _ptr(x), _dtype_code(x), B, T, H, W, h, D,
               P, _ptr(out), _stream(stream, x.device))
    _check(st, "nabla_fractal_flatten")
    return out


def nabla_fractal_unflatten(y: torch.Tensor, T: int, H: int, W: int, P: int = 8,
                            out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """y [B, T*H*W, h, D] in fractal order -> [B, T, H, W, h, D] in raster order."""
    if y.dim() != 4 or y.shape[1] != T * H * W or not y.is_contiguous():
        raise ValueError("y must be a contiguous [B, T*H*W, h, D] tensor")
    B, _, h, D = y.shape
    if out is None:
        out = torch.empty((B, T, H, W, h, D), dtype=y.dtype, device=y.device)
    _buf(out, "out", y.numel(), y.dtype, y.device)
    _cuda(y)
    st = _call(y.device, load().nabla_fractal_unflatten, _ptr(y), _dtype_code(y), B, T, H, W, h, D,
               P, _ptr(out), _stream(stream, y.device))
    _check(st, "nabla_fractal_unflatten")
    return out


def _stream_device(stream) -> torch.device:
    dev = getattr(stream, "device", None)
    return torch.device(dev) if dev is not None else torch.device(
        "cuda", torch.cuda.current_device())


def nabla_selftest_bounded_wait(stream=None) -> None:
    """Enqueue the bounded-wait probe (it must end as a recorded timeout)."""
    dev = _stream_device(stream)
    st = _call(dev, load().nabla_selftest_bounded_wait, _stream(stream, dev))
    _check(st, "nabla_selftest_bounded_wait")


def nabla_get_last_device_status(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device status code."""
    dev = _stream_device(stream)
    return _call(dev, load().nabla_get_last_device_status, _stream(stream, dev))


def from_storage(a: np.ndarray, device) -> torch.Tensor:
    """numpy storage array (float32, or uint16 bf16 bit patterns) -> device tensor."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(device)
    return torch.from_numpy(a).to(device)

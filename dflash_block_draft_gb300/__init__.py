"""Python binding of the GB300 DFlash draft block-attention library.

Argument marshalling only: every step of the computation runs in the CUDA
kernels of ``libdflash_attn.so`` (C ABI in ``include/dflash_attn.h``).
PyTorch supplies device memory and the current stream.  There is no CPU
fallback: if the shared library has not been built, every call raises.

The functions carry the C names:
  dflash_attn_dense, dflash_attn_anchored, dflash_attn_ragged,
  dflash_attn_dense_backward, dflash_attn_anchored_backward,
  dflash_attn_workspace_size, dflash_build_schedule_host, dflash_scan_mask,
  dflash_last_device_error, dflash_status_string.
"""
from __future__ import annotations

import ctypes
import os
import threading

import numpy as np

from . import build as _build

LIB_PATH = _build.LIB_PATH

DFLASH_BF16, DFLASH_FP32 = 0, 1
MODE_DENSE, MODE_ANCHORED, MODE_RAGGED = 0, 1, 2
MODE_DENSE_BACKWARD, MODE_ANCHORED_BACKWARD = 3, 4
TILE_M = TILE_N = 128
TILE_SKIP, TILE_PARTIAL, TILE_FULL = 0, 1, 2

STATUS = {0: "DFLASH_OK", 1: "DFLASH_ERR_INVALID", 2: "DFLASH_ERR_SHAPE", 3: "DFLASH_ERR_DTYPE",
          4: "DFLASH_ERR_ALIGN", 5: "DFLASH_ERR_UNSUPPORTED", 6: "DFLASH_ERR_WORKSPACE", 7: "DFLASH_ERR_CUDA",
          8: "DFLASH_ERR_TIMEOUT"}

EXPORTS = ("dflash_attn_dense", "dflash_attn_anchored", "dflash_attn_ragged", "dflash_attn_workspace_size",
           "dflash_build_schedule_host", "dflash_scan_mask", "dflash_status_string", "dflash_last_device_error",
           "dflash_kernel_launches", "dflash_attn_dense_noalloc", "dflash_build_mask",
           "dflash_attn_anchored_backward", "dflash_attn_dense_backward", "dflash_test_inject_stall",
           "dflash_test_limit_tile_flags",
           "dflash_attn_latent_ragged", "dflash_attn_latent_workspace_size")


class DFlashError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn}: {STATUS.get(status, status)} ({dflash_status_string(status)})")


class _Dims(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("H", ctypes.c_int), ("S", ctypes.c_int), ("Q", ctypes.c_int),
                ("d_nope", ctypes.c_int), ("d_rope", ctypes.c_int), ("d_v", ctypes.c_int),
                ("scale", ctypes.c_float)]


_lock = threading.Lock()
_lib_handle = None


def load_library(path: str | None = None):
    """Load libdflash_attn.so (built by ``__graft_entry__.build()``); raises if absent."""
    global _lib_handle
    with _lock:
        if _lib_handle is not None:
            return _lib_handle
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(f"DFlash CUDA library not built ({p} missing): run "
                               "`python -c 'import __graft_entry__ as g; g.build()'`")
        lib = ctypes.CDLL(p)
        P, I, F, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        DP = ctypes.POINTER(_Dims)
        lib.dflash_attn_dense.argtypes = [DP, I, P, P, P, P, P, P, P, P, S, P]
        lib.dflash_attn_anchored.argtypes = [DP, I, P, P, P, P, P, I, I, P, P, P, S, P]
        lib.dflash_attn_ragged.argtypes = [I, I, I, I, I, F, I, P, P, P, P, P, P, P, I, I, I, I, P, P, P, S, P]
        lib.dflash_attn_workspace_size.argtypes = [I, DP, I, I, I, I, I, I, I, I, I]
        lib.dflash_attn_workspace_size.restype = S
        lib.dflash_build_schedule_host.argtypes = [I, I, I, P, I, I, P]
        lib.dflash_scan_mask.argtypes = [I, I, I, I, P, P, P]
        lib.dflash_status_string.argtypes = [I]
        lib.dflash_status_string.restype = ctypes.c_char_p
        lib.dflash_last_device_error.argtypes = [P]
        lib.dflash_attn_dense_noalloc.argtypes = [DP, I, P, P, P, P, P, P, P, P]
        lib.dflash_build_mask.argtypes = [I, I, I, P, I, I, I, P, P]
        lib.dflash_build_mask.restype = ctypes.c_int
        lib.dflash_attn_dense_noalloc.restype = ctypes.c_int
        lib.dflash_attn_anchored_backward.argtypes = [DP, I, P, P, P, P, P, I, I, P, P, P, P, P, P, P, P, S, P]
        lib.dflash_attn_dense_backward.argtypes = [DP, I, P, P, P, P, P, P, P, P, P, P, P, P, P, S, P]
        lib.dflash_attn_anchored_backward.restype = ctypes.c_int
        lib.dflash_attn_dense_backward.restype = ctypes.c_int
        lib.dflash_attn_latent_ragged.argtypes = [I, I, I, I, I, I, F, I, P, P, P, P, P, P, P, I, I, I, I, P, P, P,
                                                  S, P]
        lib.dflash_attn_latent_ragged.restype = ctypes.c_int
        lib.dflash_attn_latent_workspace_size.argtypes = [I, I, I, I, I, I, I, I, I, I]
        lib.dflash_attn_latent_workspace_size.restype = S
        lib.dflash_test_inject_stall.argtypes = [ctypes.c_ulonglong, I]
        lib.dflash_test_inject_stall.restype = None
        lib.dflash_test_limit_tile_flags.argtypes = [I]
        lib.dflash_test_limit_tile_flags.restype = None
        lib.dflash_kernel_launches.argtypes = []
        lib.dflash_kernel_launches.restype = ctypes.c_uint64
        for name in ("dflash_attn_dense", "dflash_attn_anchored", "dflash_attn_ragged",
                     "dflash_build_schedule_host", "dflash_scan_mask", "dflash_last_device_error"):
            getattr(lib, name).restype = ctypes.c_int
        _lib_handle = lib
        return lib


# ---------------------------------------------------------------------------
# marshalling helpers
# ---------------------------------------------------------------------------
def _torch():
    import torch
    return torch


def _dtype_code(t) -> int:
    torch = _torch()
    if t.dtype == torch.bfloat16:
        return DFLASH_BF16
    if t.dtype == torch.float32:
        return DFLASH_FP32
    raise TypeError(f"unsupported dtype {t.dtype} (bf16 or fp32)")


def _dev_ptr(t, name, dtype=None):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    torch = _torch()
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _check(fn, st):
    if st != 0:
        raise DFlashError(fn, st)


def _workspace(nbytes, workspace, device):
    torch = _torch()
    if workspace is None:
        workspace = torch.empty(max(int(nbytes), 1), dtype=torch.uint8, device=device)
    elif workspace.numel() * workspace.element_size() < nbytes:
        raise ValueError(f"workspace too small: need {nbytes} bytes")
    return workspace


def _dims(B, H, S, Q, dn, dr, dv, scale):
    return _Dims(B, H, S, Q, dn, dr, dv, float(scale or 0.0))


# ---------------------------------------------------------------------------
# public API
# ---------------------------------------------------------------------------
def dflash_status_string(status: int) -> str:
    try:
        return load_library().dflash_status_string(int(status)).decode()
    except RuntimeError:
        return STATUS.get(status, "unknown")


def dflash_attn_workspace_size(mode, B=0, H=0, S=0, Q=0, d_nope=0, d_rope=0, d_v=0, dtype=DFLASH_BF16, R=0,
                               total_q=0, total_kv=0, max_q_len=0) -> int:
    lib = load_library()
    if mode == MODE_RAGGED:
        return int(lib.dflash_attn_workspace_size(mode, None, dtype, R, H, d_nope, d_rope, d_v, total_q, total_kv,
                                                  max_q_len))
    d = _dims(B, H, S, Q, d_nope, d_rope, d_v, 0.0)
    return int(lib.dflash_attn_workspace_size(mode, ctypes.byref(d), dtype, 0, 0, 0, 0, 0, 0, 0, 0))


def _batched_shapes(q, k_nope, k_rope, v):
    B, Q, H, dqk = q.shape
    K = k_nope.shape[1]
    dn, dr, dv = k_nope.shape[3], k_rope.shape[2], v.shape[3]
    if (k_nope.shape[0], k_nope.shape[2]) != (B, H) or k_rope.shape[:2] != (B, K) or v.shape[:3] != (B, K, H):
        raise ValueError("inconsistent q/k/v shapes")
    if dn + dr != dqk:
        raise ValueError("q head dim must be d_nope + d_rope")
    return B, H, K - Q, Q, dn, dr, dv


def dflash_attn_dense(q, k_nope, k_rope, v, mask, out=None, lse=None, scale=0.0, workspace=None, stream=None):
    """Dense additive-mask block attention.  q [B,Q,H,dn+dr], k_nope [B,S+Q,H,dn],
    k_rope [B,S+Q,dr], v [B,S+Q,H,dv], mask [B,1,Q,S+Q] (q's dtype).
    Returns out [B,Q,H,dv]; fills lse [B,H,Q] fp32 if given."""
    torch = _torch()
    lib = load_library()
    B, H, S, Q, dn, dr, dv = _batched_shapes(q, k_nope, k_rope, v)
    dt = _dtype_code(q)
    if tuple(mask.shape) != (B, 1, Q, S + Q):
        raise ValueError("mask must be [B,1,Q,S+Q]")
    if out is None:
        out = torch.empty((B, Q, H, dv), dtype=q.dtype, device=q.device)
    nbytes = dflash_attn_workspace_size(MODE_DENSE, B, H, S, Q, dn, dr, dv, dt)
    ws = _workspace(nbytes, workspace, q.device)
    d = _dims(B, H, S, Q, dn, dr, dv, scale)
    st = lib.dflash_attn_dense(ctypes.byref(d), dt, _dev_ptr(q, "q"), _dev_ptr(k_nope, "k_nope", q.dtype),
                               _dev_ptr(k_rope, "k_rope", q.dtype), _dev_ptr(v, "v", q.dtype),
                               _dev_ptr(mask, "mask", q.dtype), _dev_ptr(out, "out", q.dtype),
                               _dev_ptr(lse, "lse", torch.float32), _dev_ptr(ws, "workspace"), nbytes,
                               _stream(stream))
    _check("dflash_attn_dense", st)
    return out


def dflash_attn_dense_noalloc(q, k_nope, k_rope, v, mask, out=None, lse=None, scale=0.0, stream=None):
    """dflash_attn_dense without a workspace: the library's own fixed device
    array holds the mask-tile classes (see include/dflash_attn.h).  For callers
    that cannot allocate device scratch memory; concurrent calls on one device
    must not overlap on the GPU."""
    torch = _torch()
    lib = load_library()
    B, H, S, Q, dn, dr, dv = _batched_shapes(q, k_nope, k_rope, v)
    dt = _dtype_code(q)
    if tuple(mask.shape) != (B, 1, Q, S + Q):
        raise ValueError("mask must be [B,1,Q,S+Q]")
    if out is None:
        out = torch.empty((B, Q, H, dv), dtype=q.dtype, device=q.device)
    d = _dims(B, H, S, Q, dn, dr, dv, scale)
    st = lib.dflash_attn_dense_noalloc(ctypes.byref(d), dt, _dev_ptr(q, "q"), _dev_ptr(k_nope, "k_nope", q.dtype),
                                       _dev_ptr(k_rope, "k_rope", q.dtype), _dev_ptr(v, "v", q.dtype),
                                       _dev_ptr(mask, "mask", q.dtype), _dev_ptr(out, "out", q.dtype),
                                       _dev_ptr(lse, "lse", torch.float32), _stream(stream))
    _check("dflash_attn_dense_noalloc", st)
    return out


def dflash_attn_anchored(q, k_nope, k_rope, v, anchors, block_size, out=None, lse=None, scale=0.0, workspace=None,
                         stream=None):
    """Anchored block attention: anchors [B,nb] int32 (device), Q = nb*block_size."""
    torch = _torch()
    lib = load_library()
    B, H, S, Q, dn, dr, dv = _batched_shapes(q, k_nope, k_rope, v)
    dt = _dtype_code(q)
    nb = anchors.shape[1]
    if out is None:
        out = torch.empty((B, Q, H, dv), dtype=q.dtype, device=q.device)
    nbytes = dflash_attn_workspace_size(MODE_ANCHORED, B, H, S, Q, dn, dr, dv, dt)
    ws = _workspace(nbytes, workspace, q.device)
    d = _dims(B, H, S, Q, dn, dr, dv, scale)
    st = lib.dflash_attn_anchored(ctypes.byref(d), dt, _dev_ptr(q, "q"), _dev_ptr(k_nope, "k_nope", q.dtype),
                                  _dev_ptr(k_rope, "k_rope", q.dtype), _dev_ptr(v, "v", q.dtype),
                                  _dev_ptr(anchors, "anchors", torch.int32), nb, int(block_size),
                                  _dev_ptr(out, "out", q.dtype), _dev_ptr(lse, "lse", torch.float32),
                                  _dev_ptr(ws, "workspace"), nbytes, _stream(stream))
    _check("dflash_attn_anchored", st)
    return out


def dflash_attn_ragged(q, k_nope, k_rope, v, q_offsets, kv_offsets, anchors, block_size, max_q_len, out=None,
                       lse=None, scale=0.0, workspace=None, stream=None):
    """Ragged (row-offset) block attention.  q [total_q,H,dn+dr], k_nope
    [total_kv,H,dn], k_rope [total_kv,dr], v [total_kv,H,dv]; offsets int32
    [R+1] and anchors int32 [total_q/block_size] on the device.  lse is [H,total_q]."""
    torch = _torch()
    lib = load_library()
    total_q, H, dqk = q.shape
    total_kv, dn, dr, dv = k_nope.shape[0], k_nope.shape[2], k_rope.shape[1], v.shape[2]
    if dn + dr != dqk:
        raise ValueError("q head dim must be d_nope + d_rope")
    R = q_offsets.shape[0] - 1
    dt = _dtype_code(q)
    if out is None:
        out = torch.empty((total_q, H, dv), dtype=q.dtype, device=q.device)
    nbytes = dflash_attn_workspace_size(MODE_RAGGED, H=H, d_nope=dn, d_rope=dr, d_v=dv, dtype=dt, R=R,
                                        total_q=total_q, total_kv=total_kv, max_q_len=int(max_q_len))
    ws = _workspace(nbytes, workspace, q.device)
    st = lib.dflash_attn_ragged(R, H, dn, dr, dv, float(scale or 0.0), dt, _dev_ptr(q, "q"),
                                _dev_ptr(k_nope, "k_nope", q.dtype), _dev_ptr(k_rope, "k_rope", q.dtype),
                                _dev_ptr(v, "v", q.dtype), _dev_ptr(q_offsets, "q_offsets", torch.int32),
                                _dev_ptr(kv_offsets, "kv_offsets", torch.int32),
                                _dev_ptr(anchors, "anchors", torch.int32), int(block_size), total_q, total_kv,
                                int(max_q_len), _dev_ptr(out, "out", q.dtype), _dev_ptr(lse, "lse", torch.float32),
                                _dev_ptr(ws, "workspace"), nbytes, _stream(stream))
    _check("dflash_attn_ragged", st)
    return out


def dflash_attn_latent_workspace_size(R, H, d_nope, d_rope, d_v, kv_rank, dtype=DFLASH_BF16, total_q=0,
                                      total_kv=0, max_q_len=0) -> int:
    return int(load_library().dflash_attn_latent_workspace_size(R, H, d_nope, d_rope, d_v, kv_rank, dtype, total_q,
                                                                 total_kv, max_q_len))


def dflash_attn_latent_ragged(q, c_kv, k_rope, w_kv_b, q_offsets, kv_offsets, anchors, block_size, max_q_len,
                              out=None, lse=None, scale=0.0, workspace=None, stream=None):
    """Ragged block attention over compressed KV latents.  q [total_q,H,dn+dr],
    c_kv [total_kv,kv_rank], k_rope [total_kv,dr], w_kv_b [H,dn+dv,kv_rank]
    (kv_b_proj per head: key rows, then value rows); offsets int32 [R+1] and
    anchors int32 [total_q/block_size] on the device.  lse is [H,total_q]."""
    torch = _torch()
    lib = load_library()
    total_q, H, dqk = q.shape
    total_kv, rank = c_kv.shape
    dr = k_rope.shape[1]
    dn = dqk - dr
    if w_kv_b.shape[0] != H or w_kv_b.shape[2] != rank or w_kv_b.shape[1] <= dn or k_rope.shape[0] != total_kv:
        raise ValueError("inconsistent q / c_kv / k_rope / w_kv_b shapes")
    dv = w_kv_b.shape[1] - dn
    R = q_offsets.shape[0] - 1
    dt = _dtype_code(q)
    if out is None:
        out = torch.empty((total_q, H, dv), dtype=q.dtype, device=q.device)
    nbytes = dflash_attn_latent_workspace_size(R, H, dn, dr, dv, rank, dt, total_q, total_kv, int(max_q_len))
    ws = _workspace(nbytes, workspace, q.device)
    st = lib.dflash_attn_latent_ragged(R, H, dn, dr, dv, rank, float(scale or 0.0), dt, _dev_ptr(q, "q"),
                                       _dev_ptr(c_kv, "c_kv", q.dtype), _dev_ptr(k_rope, "k_rope", q.dtype),
                                       _dev_ptr(w_kv_b, "w_kv_b", q.dtype),
                                       _dev_ptr(q_offsets, "q_offsets", torch.int32),
                                       _dev_ptr(kv_offsets, "kv_offsets", torch.int32),
                                       _dev_ptr(anchors, "anchors", torch.int32), int(block_size), total_q, total_kv,
                                       int(max_q_len), _dev_ptr(out, "out", q.dtype),
                                       _dev_ptr(lse, "lse", torch.float32), _dev_ptr(ws, "workspace"), nbytes,
                                       _stream(stream))
    _check("dflash_attn_latent_ragged", st)
    return out


def _backward_grads(q, k_nope, k_rope, v, grads):
    torch = _torch()
    if grads is None:
        grads = (torch.empty_like(q), torch.empty_like(k_nope), torch.empty_like(k_rope), torch.empty_like(v))
    dq, dkn, dkr, dvv = grads
    for name, g, ref in (("dq", dq, q), ("dk_nope", dkn, k_nope), ("dk_rope", dkr, k_rope), ("dv", dvv, v)):
        if g.shape != ref.shape or g.dtype != ref.dtype:
            raise ValueError(f"{name} must match its input's shape and dtype")
    return dq, dkn, dkr, dvv


def dflash_attn_anchored_backward(q, k_nope, k_rope, v, anchors, block_size, out, lse, dout, grads=None, scale=0.0,
                                  workspace=None, stream=None):
    """Gradients (dq, dk_nope, dk_rope, dv) of sum(dout * out) for the anchored
    forward; out and lse [B,H,Q] fp32 are that forward's outputs.  grads: optional
    preallocated (dq, dk_nope, dk_rope, dv) shaped like (q, k_nope, k_rope, v)."""
    torch = _torch()
    lib = load_library()
    B, H, S, Q, dn, dr, dv = _batched_shapes(q, k_nope, k_rope, v)
    dt = _dtype_code(q)
    nb = anchors.shape[1]
    dq, dkn, dkr, dvv = _backward_grads(q, k_nope, k_rope, v, grads)
    nbytes = dflash_attn_workspace_size(MODE_ANCHORED_BACKWARD, B, H, S, Q, dn, dr, dv, dt)
    ws = _workspace(nbytes, workspace, q.device)
    d = _dims(B, H, S, Q, dn, dr, dv, scale)
    st = lib.dflash_attn_anchored_backward(
        ctypes.byref(d), dt, _dev_ptr(q, "q"), _dev_ptr(k_nope, "k_nope", q.dtype), _dev_ptr(k_rope, "k_rope", q.dtype),
        _dev_ptr(v, "v", q.dtype), _dev_ptr(anchors, "anchors", torch.int32), nb, int(block_size),
        _dev_ptr(out, "out", q.dtype), _dev_ptr(lse, "lse", torch.float32), _dev_ptr(dout, "dout", q.dtype),
        _dev_ptr(dq, "dq"), _dev_ptr(dkn, "dk_nope"), _dev_ptr(dkr, "dk_rope"), _dev_ptr(dvv, "dv"),
        _dev_ptr(ws, "workspace"), nbytes, _stream(stream))
    _check("dflash_attn_anchored_backward", st)
    return dq, dkn, dkr, dvv


def dflash_attn_dense_backward(q, k_nope, k_rope, v, mask, out, lse, dout, grads=None, scale=0.0, workspace=None,
                               stream=None):
    """Gradients (dq, dk_nope, dk_rope, dv) of sum(dout * out) for the dense
    forward with additive mask [B,1,Q,S+Q] (the mask gets no gradient)."""
    torch = _torch()
    lib = load_library()
    B, H, S, Q, dn, dr, dv = _batched_shapes(q, k_nope, k_rope, v)
    dt = _dtype_code(q)
    if tuple(mask.shape) != (B, 1, Q, S + Q):
        raise ValueError("mask must be [B,1,Q,S+Q]")
    dq, dkn, dkr, dvv = _backward_grads(q, k_nope, k_rope, v, grads)
    nbytes = dflash_attn_workspace_size(MODE_DENSE_BACKWARD, B, H, S, Q, dn, dr, dv, dt)
    ws = _workspace(nbytes, workspace, q.device)
    d = _dims(B, H, S, Q, dn, dr, dv, scale)
    st = lib.dflash_attn_dense_backward(
        ctypes.byref(d), dt, _dev_ptr(q, "q"), _dev_ptr(k_nope, "k_nope", q.dtype), _dev_ptr(k_rope, "k_rope", q.dtype),
        _dev_ptr(v, "v", q.dtype), _dev_ptr(mask, "mask", q.dtype), _dev_ptr(out, "out", q.dtype),
        _dev_ptr(lse, "lse", torch.float32), _dev_ptr(dout, "dout", q.dtype), _dev_ptr(dq, "dq"),
        _dev_ptr(dkn, "dk_nope"), _dev_ptr(dkr, "dk_rope"), _dev_ptr(dvv, "dv"), _dev_ptr(ws, "workspace"), nbytes,
        _stream(stream))
    _check("dflash_attn_dense_backward", st)
    return dq, dkn, dkr, dvv


def dflash_build_schedule_host(B, S, Q, anchors, block_size) -> np.ndarray:
    """Host tile classes [B, ceil(Q/128), ceil((S+Q)/128)] of the anchored rule (numpy in, numpy out)."""
    lib = load_library()
    an = np.ascontiguousarray(anchors, np.int32)
    nb = an.shape[1] if an.ndim == 2 else 0
    out = np.zeros((B, -(-Q // TILE_M), -(-(S + Q) // TILE_N)), np.uint8)
    st = lib.dflash_build_schedule_host(B, S, Q, an.ctypes.data_as(ctypes.c_void_p), nb, int(block_size),
                                        out.ctypes.data_as(ctypes.c_void_p))
    _check("dflash_build_schedule_host", st)
    return out


def dflash_build_mask(anchors, block_size, S, dtype=None, mask=None, stream=None):
    """Device additive mask [B,1,Q,S+Q] (0 visible, -inf hidden) of the anchored
    rule from anchors [B,nb] int32 (CUDA).  dtype: torch.bfloat16 or torch.float32."""
    torch = _torch()
    lib = load_library()
    B, nb = anchors.shape
    Q = nb * int(block_size)
    dtype = dtype or torch.bfloat16
    if mask is None:
        mask = torch.empty((B, 1, Q, S + Q), dtype=dtype, device=anchors.device)
    st = lib.dflash_build_mask(B, S, Q, _dev_ptr(anchors, "anchors", torch.int32), nb, int(block_size),
                               _dtype_code(mask), _dev_ptr(mask, "mask"), _stream(stream))
    _check("dflash_build_mask", st)
    return mask


def dflash_scan_mask(mask, classes=None, stream=None):
    """Device tile classes of a dense mask [B,1,Q,S+Q]; returns a uint8 CUDA tensor."""
    torch = _torch()
    lib = load_library()
    B, _, Q, K = mask.shape
    S = K - Q
    if classes is None:
        classes = torch.empty((B, -(-Q // TILE_M), -(-K // TILE_N)), dtype=torch.uint8, device=mask.device)
    st = lib.dflash_scan_mask(B, S, Q, _dtype_code(mask), _dev_ptr(mask, "mask"),
                              _dev_ptr(classes, "classes", torch.uint8), _stream(stream))
    _check("dflash_scan_mask", st)
    return classes


def dflash_kernel_launches() -> int:
    """Kernels launched by the library in this process so far."""
    return int(load_library().dflash_kernel_launches())


def dflash_last_device_error(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device error word."""
    return int(load_library().dflash_last_device_error(_stream(stream)))


def dflash_test_inject_stall(wait_budget_ns: int = 0, stall_cta: int = -1) -> None:
    """Test export: set the bounded-wait budget (0 = the 2 s default) and the CTA
    whose producer leaves its first work item's key tiles unloaded (-1 = none),
    for every later forward call in this process."""
    load_library().dflash_test_inject_stall(int(wait_budget_ns), int(stall_cta))


def dflash_test_limit_tile_flags(n: int = 0) -> None:
    """Test export: cap the backward kernels' shared-memory table of tile flags
    at n entries (0 = the full table), for every later call in this process."""
    load_library().dflash_test_limit_tile_flags(int(n))

"""fp64 CPU oracle for DFlash draft block attention.

TEST INFRASTRUCTURE ONLY: the test suite, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package; the library's product
path never does.  It shares no code with the CUDA library.

``oracle.c`` holds the plain definition (see its header); this module compiles
it with gcc on first use and wraps it with numpy marshalling.  ``brute.py``
holds an independent numpy brute force used to pin it.

Element types: numpy float32/float64 arrays, or uint16 arrays holding bf16
bit patterns (widened exactly inside the C code).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "_build", "liboracle.so")
_lock = threading.Lock()
_lib = None

TILE_SKIP, TILE_PARTIAL, TILE_FULL = 0, 1, 2

_DT = {np.dtype(np.uint16): 0, np.dtype(np.float32): 1, np.dtype(np.float64): 2}


def build(force: bool = False) -> str:
    """Compile oracle.c into a shared library (gcc, OpenMP).  Returns its path."""
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + f".{os.getpid()}.tmp"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-fno-fast-math",
           "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P, I, D, I64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_double, ctypes.c_int64
            lib.oracle_dense.argtypes = [I, I, I, I, I, I, I, D, I, P, P, P, P, P, I, P, I64, P, P, I]
            lib.oracle_anchored.argtypes = [I, I, I, I, I, I, I, D, I, P, P, P, P, P, I, I, P, I64, P, P, I]
            lib.oracle_ragged.argtypes = [I, I, I, I, I, D, I, P, P, P, P, P, P, P, I, P, I64, P, P, I]
            lib.oracle_anchored_split.argtypes = [I, I, I, I, I, I, I, D, I, P, P, P, P, P, I, I, I, P, P, I]
            lib.oracle_build_mask.argtypes = [I, I, I, P, I, I, P]
            lib.oracle_tile_classes.argtypes = [I, I, I, I, I, P, I, I, P, I, P]
            lib.oracle_max_threads.argtypes = []
            lib.oracle_latent_expand.argtypes = [I, I, I, I, I, P, P, I64, I64, P, P, I]
            lib.oracle_backward.argtypes = [I, I, I, I, I, I, I, D, I, P, P, P, P, P, P, I, I, P, I, P, I64,
                                            P, P, P, P, I]
            for f in (lib.oracle_dense, lib.oracle_anchored, lib.oracle_ragged,
                      lib.oracle_anchored_split, lib.oracle_build_mask, lib.oracle_tile_classes,
                      lib.oracle_max_threads, lib.oracle_backward, lib.oracle_latent_expand):
                f.restype = ctypes.c_int
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _same_dtype(*arrs):
    dts = {a.dtype for a in arrs}
    if len(dts) != 1 or next(iter(dts)) not in _DT:
        raise TypeError(f"q/k/v must share one of uint16(bf16)/float32/float64, got {dts}")
    return _DT[next(iter(dts))]


def _c(a, dtype=None):
    a = np.asarray(a) if dtype is None else np.asarray(a, dtype=dtype)
    return np.ascontiguousarray(a)


def default_scale(d_nope: int, d_rope: int) -> float:
    """scaling = q_head_dim ** -0.5 with q_head_dim = qk_nope + qk_rope."""
    return float((d_nope + d_rope) ** -0.5)


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def _rows_arg(rows):
    if rows is None:
        return None, 0
    r = _c(rows, np.int64)
    return r, r.size


def dense(q, k_nope, k_rope, v, mask, scale=None, rows=None, nthreads=0):
    """Dense additive-mask attention.

    q [B,Q,H,dn+dr], k_nope [B,S+Q,H,dn], k_rope [B,S+Q,dr], v [B,S+Q,H,dv],
    mask [B,1,Q,S+Q].  Returns (out, lse): out [B,Q,H,dv] and lse [B,H,Q] when
    rows is None, else out [n,H,dv] and lse [n,H] for the flat rows b*Q+i.
    """
    q, k_nope, k_rope, v, mask = (_c(x) for x in (q, k_nope, k_rope, v, mask))
    B, Q, H, dqk = q.shape
    S = k_nope.shape[1] - Q
    dn, dr, dv = k_nope.shape[3], k_rope.shape[2], v.shape[3]
    assert dn + dr == dqk and mask.shape == (B, 1, Q, S + Q)
    dt = _same_dtype(q, k_nope, k_rope, v)
    mdt = _DT[mask.dtype]
    scale = default_scale(dn, dr) if scale is None else float(scale)
    r, n = _rows_arg(rows)
    nr = B * Q if r is None else n
    out = np.zeros((nr, H, dv), np.float64)
    lse = np.zeros((nr, H), np.float64)
    rc = _load().oracle_dense(B, H, S, Q, dn, dr, dv, scale, dt, _ptr(q), _ptr(k_nope), _ptr(k_rope),
                              _ptr(v), _ptr(mask), mdt, _ptr(r), n, _ptr(out), _ptr(lse), nthreads)
    if rc:
        raise ValueError(f"oracle_dense failed ({rc})")
    if r is None:
        return out.reshape(B, Q, H, dv), lse.reshape(B, Q, H).transpose(0, 2, 1).copy()
    return out, lse


def anchored(q, k_nope, k_rope, v, anchors, block_size, scale=None, rows=None, nthreads=0):
    """Anchored block attention (block j sees context p < a_j plus its own block).

    anchors [B,nb] int32.  Shapes and returns as for :func:`dense`.
    """
    q, k_nope, k_rope, v = (_c(x) for x in (q, k_nope, k_rope, v))
    anchors = _c(anchors, np.int32)
    B, Q, H, dqk = q.shape
    S = k_nope.shape[1] - Q
    dn, dr, dv = k_nope.shape[3], k_rope.shape[2], v.shape[3]
    nb = anchors.shape[1]
    assert dn + dr == dqk and nb * block_size == Q
    dt = _same_dtype(q, k_nope, k_rope, v)
    scale = default_scale(dn, dr) if scale is None else float(scale)
    r, n = _rows_arg(rows)
    nr = B * Q if r is None else n
    out = np.zeros((nr, H, dv), np.float64)
    lse = np.zeros((nr, H), np.float64)
    rc = _load().oracle_anchored(B, H, S, Q, dn, dr, dv, scale, dt, _ptr(q), _ptr(k_nope), _ptr(k_rope),
                                 _ptr(v), _ptr(anchors), nb, block_size, _ptr(r), n, _ptr(out),
                                 _ptr(lse), nthreads)
    if rc:
        raise ValueError(f"oracle_anchored failed ({rc})")
    if r is None:
        return out.reshape(B, Q, H, dv), lse.reshape(B, Q, H).transpose(0, 2, 1).copy()
    return out, lse


def ragged(q, k_nope, k_rope, v, q_offsets, kv_offsets, anchors, block_size, scale=None, rows=None,
           nthreads=0):
    """Ragged (row-offset) anchored attention.

    q [total_q,H,dn+dr], k_nope [total_kv,H,dn], k_rope [total_kv,dr],
    v [total_kv,H,dv]; offsets int32 [R+1]; anchors int32 [total_q/bs].
    Returns out [total_q,H,dv] and lse [H,total_q] (rows=None) or
    out [n,H,dv], lse [n,H].
    """
    q, k_nope, k_rope, v = (_c(x) for x in (q, k_nope, k_rope, v))
    qo, ko, an = _c(q_offsets, np.int32), _c(kv_offsets, np.int32), _c(anchors, np.int32)
    R = qo.size - 1
    TQ, H, dqk = q.shape
    dn, dr, dv = k_nope.shape[2], k_rope.shape[1], v.shape[2]
    assert dn + dr == dqk
    dt = _same_dtype(q, k_nope, k_rope, v)
    scale = default_scale(dn, dr) if scale is None else float(scale)
    r, n = _rows_arg(rows)
    nr = TQ if r is None else n
    out = np.zeros((nr, H, dv), np.float64)
    lse = np.zeros((nr, H), np.float64)
    rc = _load().oracle_ragged(R, H, dn, dr, dv, scale, dt, _ptr(q), _ptr(k_nope), _ptr(k_rope), _ptr(v),
                               _ptr(qo), _ptr(ko), _ptr(an), block_size, _ptr(r), n, _ptr(out),
                               _ptr(lse), nthreads)
    if rc:
        raise ValueError(f"oracle_ragged failed ({rc})")
    if r is None:
        return out, lse.T.copy()
    return out, lse


def anchored_split(q, k_nope, k_rope, v, anchors, block_size, split, scale=None, nthreads=0):
    """Anchored attention evaluated as key-axis spans of `split` keys merged by
    the log-sum-exp rule.  Same returns as :func:`anchored` (rows=None)."""
    q, k_nope, k_rope, v = (_c(x) for x in (q, k_nope, k_rope, v))
    anchors = _c(anchors, np.int32)
    B, Q, H, dqk = q.shape
    S = k_nope.shape[1] - Q
    dn, dr, dv = k_nope.shape[3], k_rope.shape[2], v.shape[3]
    nb = anchors.shape[1]
    dt = _same_dtype(q, k_nope, k_rope, v)
    scale = default_scale(dn, dr) if scale is None else float(scale)
    out = np.zeros((B * Q, H, dv), np.float64)
    lse = np.zeros((B * Q, H), np.float64)
    rc = _load().oracle_anchored_split(B, H, S, Q, dn, dr, dv, scale, dt, _ptr(q), _ptr(k_nope),
                                       _ptr(k_rope), _ptr(v), _ptr(anchors), nb, block_size, split,
                                       _ptr(out), _ptr(lse), nthreads)
    if rc:
        raise ValueError(f"oracle_anchored_split failed ({rc})")
    return out.reshape(B, Q, H, dv), lse.reshape(B, Q, H).transpose(0, 2, 1).copy()


def backward(q, k_nope, k_rope, v, dout, anchors=None, block_size=0, mask=None, scale=None, pairs=None,
             nthreads=0):
    """Gradients of L = sum(dout * out) for the anchored rule (anchors given) or
    a dense additive mask (mask given; the mask itself gets no gradient).

    Shapes as for :func:`dense`; dout [B,Q,H,dv].  Returns fp64
    (dq [B,Q,H,dn+dr], dk_nope [B,S+Q,H,dn], dk_rope [B,S+Q,dr], dv [B,S+Q,H,dv]).
    pairs: optional flat (b*H + h) subset; other heads' gradients stay 0 and
    dk_rope sums only the listed heads.
    """
    q, k_nope, k_rope, v, dout = (_c(x) for x in (q, k_nope, k_rope, v, dout))
    B, Q, H, dqk = q.shape
    S = k_nope.shape[1] - Q
    dn, dr, dv = k_nope.shape[3], k_rope.shape[2], v.shape[3]
    assert dn + dr == dqk and dout.shape == (B, Q, H, dv)
    dt = _same_dtype(q, k_nope, k_rope, v, dout)
    scale = default_scale(dn, dr) if scale is None else float(scale)
    an, nb, mdt = None, 0, 0
    if mask is None:
        an = _c(anchors, np.int32)
        nb = an.shape[1]
        assert nb * block_size == Q
    else:
        mask = _c(mask)
        assert mask.shape == (B, 1, Q, S + Q)
        mdt = _DT[mask.dtype]
    p, n = _rows_arg(pairs)
    K = S + Q
    dq = np.empty((B, Q, H, dqk), np.float64)
    dkn = np.empty((B, K, H, dn), np.float64)
    dkr = np.empty((B, K, dr), np.float64)
    dvo = np.empty((B, K, H, dv), np.float64)
    rc = _load().oracle_backward(B, H, S, Q, dn, dr, dv, scale, dt, _ptr(q), _ptr(k_nope), _ptr(k_rope),
                                 _ptr(v), _ptr(dout), _ptr(an), nb, block_size, _ptr(mask), mdt, _ptr(p), n,
                                 _ptr(dq), _ptr(dkn), _ptr(dkr), _ptr(dvo), nthreads)
    if rc:
        raise ValueError(f"oracle_backward failed ({rc})")
    return dq, dkn, dkr, dvo


def build_mask(anchors, block_size, S):
    """Additive fp32 mask [B,1,Q,S+Q] (0 visible, -inf hidden) of the anchored rule."""
    an = _c(anchors, np.int32)
    B, nb = an.shape
    Q = nb * block_size
    mask = np.empty((B, 1, Q, S + Q), np.float32)
    rc = _load().oracle_build_mask(B, S, Q, _ptr(an), nb, block_size, _ptr(mask))
    if rc:
        raise ValueError("oracle_build_mask failed")
    return mask


def tile_classes(B, S, Q, tile_m, tile_n, anchors=None, block_size=0, mask=None):
    """Brute-force tile classes uint8 [B, ceil(Q/tile_m), ceil((S+Q)/tile_n)]:
    0 SKIP, 1 PARTIAL, 2 FULL.  Anchored rule when mask is None."""
    nqt, nkt = -(-Q // tile_m), -(-(S + Q) // tile_n)
    out = np.zeros((B, nqt, nkt), np.uint8)
    if mask is not None:
        mask = _c(mask)
        rc = _load().oracle_tile_classes(B, S, Q, tile_m, tile_n, None, 0, 0, _ptr(mask), _DT[mask.dtype],
                                         _ptr(out))
    else:
        an = _c(anchors, np.int32)
        rc = _load().oracle_tile_classes(B, S, Q, tile_m, tile_n, _ptr(an), an.shape[1], block_size, None, 0,
                                         _ptr(out))
    if rc:
        raise ValueError("oracle_tile_classes failed")
    return out


def latent_expand(c_kv, w_kv_b, d_nope, t0=0, t1=None, nthreads=0):
    """Expand compressed KV latents to per-head keys and values (fp64).

    c_kv [T, rank], w_kv_b [H, d_nope + d_v, rank] (the kv_b_proj weight per
    head: key rows first, then value rows).  Returns k_nope [t1-t0, H, d_nope]
    and v [t1-t0, H, d_v] for tokens [t0, t1)."""
    c_kv, w_kv_b = _c(c_kv), _c(w_kv_b)
    T, rank = c_kv.shape
    H, E, rank2 = w_kv_b.shape
    assert rank2 == rank and 0 <= d_nope < E
    dt = _same_dtype(c_kv, w_kv_b)
    t1 = T if t1 is None else int(t1)
    kn = np.empty((t1 - t0, H, d_nope), np.float64)
    v = np.empty((t1 - t0, H, E - d_nope), np.float64)
    rc = _load().oracle_latent_expand(H, d_nope, E - d_nope, rank, dt, _ptr(c_kv), _ptr(w_kv_b), int(t0), t1,
                                      _ptr(kn), _ptr(v), nthreads)
    if rc:
        raise ValueError("oracle_latent_expand failed")
    return kn, v


def _to_f64(a):
    a = np.asarray(a)
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    return a.astype(np.float64)


def latent_ragged(q, c_kv, k_rope, w_kv_b, q_offsets, kv_offsets, anchors, block_size, scale=None,
                  requests=None, nthreads=0):
    """Ragged anchored attention whose per-head keys and values are the
    expansions of compressed KV latents (see oracle_latent_expand): expand,
    then evaluate the ragged definition, all in fp64.

    q [total_q, H, d_nope+d_rope], c_kv [total_kv, rank], k_rope [total_kv, d_rope],
    w_kv_b [H, d_nope+d_v, rank].  scale defaults to (d_nope+d_rope)^-0.5.
    requests: optional subset of request indices (their rows only; others 0).
    Returns out [total_q, H, d_v] and lse [H, total_q] (rows of requests not
    evaluated are 0 and -inf)."""
    qo, ko, an = _c(q_offsets, np.int32), _c(kv_offsets, np.int32), _c(anchors, np.int32)
    R = qo.size - 1
    TQ, H, dqk = np.asarray(q).shape
    d_rope = np.asarray(k_rope).shape[1]
    d_nope = dqk - d_rope
    dv = np.asarray(w_kv_b).shape[1] - d_nope
    scale = default_scale(d_nope, d_rope) if scale is None else float(scale)
    out = np.zeros((TQ, H, dv), np.float64)
    lse = np.full((H, TQ), -np.inf)
    for r in (range(R) if requests is None else requests):
        k0, k1, q0, q1 = int(ko[r]), int(ko[r + 1]), int(qo[r]), int(qo[r + 1])
        kn, v = latent_expand(c_kv, w_kv_b, d_nope, k0, k1, nthreads=nthreads)
        kr = _to_f64(np.asarray(k_rope)[k0:k1])
        qq = _to_f64(np.asarray(q)[q0:q1])
        an_r = an[q0 // block_size:q1 // block_size]
        o, l = ragged(qq, kn, kr, v, np.array([0, q1 - q0], np.int32), np.array([0, k1 - k0], np.int32), an_r,
                      block_size, scale=scale, nthreads=nthreads)
        out[q0:q1] = o
        lse[:, q0:q1] = l
    return out, lse

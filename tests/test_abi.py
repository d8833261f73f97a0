"""C-ABI checks that need no GPU: the library loads, exports every declared
symbol, rejects bad arguments on the host with the documented status codes,
and its host tile schedule matches the oracle's brute-force scan bit for bit."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
import dflash_block_draft_gb300 as dfl
from dflash_block_draft_gb300 import build as dbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    dbuild.build()
    return dfl.load_library()


def _declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            txt = open(os.path.join(ROOT, "include", fn)).read()
            txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
            names.update(re.findall(r"\b(dflash_\w+)\s*\(", txt))
    return sorted(names)


def test_library_exports_every_declared_symbol(lib):
    names = _declared_functions()
    assert {"dflash_attn_dense", "dflash_attn_anchored", "dflash_attn_ragged"} <= set(names)
    raw = ctypes.CDLL(dbuild.LIB_PATH)
    missing = [n for n in names if not hasattr(raw, n)]
    assert not missing, missing
    assert set(dfl.EXPORTS) == set(names) or set(dfl.EXPORTS) <= set(names)


def test_status_strings(lib):
    for code in range(9):
        assert dfl.dflash_status_string(code)
    assert dfl.dflash_status_string(0) == "ok"


def _dims(B=1, H=2, S=8, Q=4, dn=16, dr=8, dv=16, scale=0.0):
    return dfl._Dims(B, H, S, Q, dn, dr, dv, scale)


def test_host_validation_rejects_bad_arguments(lib):
    P = ctypes.c_void_p
    good = P(4096)
    ws = P(1 << 20)
    # null dims
    assert lib.dflash_attn_anchored(None, 0, good, good, good, good, good, 1, 4, good, None, ws, 1 << 20, None) == 1
    # nb * block_size != Q
    d = _dims(Q=4)
    assert lib.dflash_attn_anchored(ctypes.byref(d), 0, good, good, good, good, good, 3, 2, good, None, ws, 1 << 20,
                                    None) == 2
    # unknown dtype
    assert lib.dflash_attn_anchored(ctypes.byref(d), 7, good, good, good, good, good, 1, 4, good, None, ws, 1 << 20,
                                    None) == 3
    # misaligned tensor
    assert lib.dflash_attn_anchored(ctypes.byref(d), 0, P(4098), good, good, good, good, 1, 4, good, None, ws,
                                    1 << 20, None) == 4
    # head dims beyond limits
    big = _dims(dn=400, dr=200)
    assert lib.dflash_attn_anchored(ctypes.byref(big), 0, good, good, good, good, good, 1, 4, good, None, ws,
                                    1 << 20, None) == 5
    # null required pointer
    assert lib.dflash_attn_anchored(ctypes.byref(d), 0, None, good, good, good, good, 1, 4, good, None, ws, 1 << 20,
                                    None) == 1
    # dense: null mask, too small workspace
    assert lib.dflash_attn_dense(ctypes.byref(d), 0, good, good, good, good, None, good, None, ws, 1 << 20,
                                 None) == 1
    assert lib.dflash_attn_dense(ctypes.byref(d), 0, good, good, good, good, good, good, None, ws, 0, None) == 6
    # negative sizes
    neg = _dims(S=-1)
    assert lib.dflash_attn_dense(ctypes.byref(neg), 0, good, good, good, good, good, good, None, ws, 1 << 20,
                                 None) == 2
    # ragged: bad block size, bad heads
    assert lib.dflash_attn_ragged(2, 2, 16, 8, 16, 0.0, 0, good, good, good, good, good, good, good, 0, 8, 40, 4,
                                  good, None, ws, 1 << 20, None) == 2
    assert lib.dflash_attn_ragged(2, 0, 16, 8, 16, 0.0, 0, good, good, good, good, good, good, good, 4, 8, 40, 4,
                                  good, None, ws, 1 << 20, None) == 2
    # NaN scale
    nan = _dims(scale=float("nan"))
    assert lib.dflash_attn_anchored(ctypes.byref(nan), 0, good, good, good, good, good, 1, 4, good, None, ws,
                                    1 << 20, None) == 1


def test_backward_host_validation_rejects_bad_arguments(lib):
    P = ctypes.c_void_p
    good, ws, big = P(4096), P(1 << 20), 1 << 30
    bw = lib.dflash_attn_anchored_backward
    dn = lib.dflash_attn_dense_backward
    d = _dims(B=1, H=2, S=8, Q=4, dn=16, dr=8, dv=16)

    def anch(dims, dtype=0, q=good, lse=good, dq=good, nb=1, bs=4, ws_bytes=big, anchors=good):
        return bw(ctypes.byref(dims) if dims is not None else None, dtype, q, good, good, good, anchors, nb, bs,
                  good, lse, good, dq, good, good, good, ws, ws_bytes, None)

    assert anch(None) == 1                      # null dims
    assert anch(d, dtype=9) == 3                # unknown dtype
    assert anch(d, nb=3, bs=2) == 2             # nb * block_size != Q
    assert anch(d, lse=None) == 1               # lse is required
    assert anch(d, anchors=None) == 1           # anchors are required
    assert anch(d, q=P(4100)) == 4              # misaligned input
    assert anch(d, dq=P(4104)) == 4             # misaligned gradient
    assert anch(d, ws_bytes=16) == 6            # workspace too small
    assert anch(_dims(dn=200, dr=64)) == 5      # d_nope + d_rope beyond the backward limit
    assert anch(_dims(dv=192)) == 5             # d_v beyond the backward limit
    # dense: the mask is required
    assert dn(ctypes.byref(d), 0, good, good, good, good, None, good, good, good, good, good, good, good, ws, big,
              None) == 1
    # nothing to do: no batch rows
    d0 = _dims(B=0)
    assert bw(ctypes.byref(d0), 0, None, None, None, None, good, 1, 4, None, None, None, None, None, None, None,
              None, 0, None) == 0


def test_backward_workspace_size_contract(lib):
    a = dfl.dflash_attn_workspace_size(dfl.MODE_ANCHORED_BACKWARD, 4, 32, 8192, 8192, 128, 64, 128)
    dn = dfl.dflash_attn_workspace_size(dfl.MODE_DENSE_BACKWARD, 4, 32, 8192, 8192, 128, 64, 128)
    # D [B,H,Q] fp32 plus the fp32 dk_rope accumulator [B,S+Q,d_rope]
    assert a >= 4 * 32 * 8192 * 4 + 4 * 16384 * 64 * 4
    assert dn >= a + 4 * 64 * 128  # plus one class byte per 128 x 128 mask tile
    assert dfl.dflash_attn_workspace_size(dfl.MODE_ANCHORED_BACKWARD, -1, 32, 8192, 8192, 128, 64, 128) == 0


def test_empty_problems_return_ok_without_launching(lib):
    P = ctypes.c_void_p
    d0 = _dims(B=0)
    assert lib.dflash_attn_anchored(ctypes.byref(d0), 0, None, None, None, None, None, 1, 4, None, None, None, 0,
                                    None) == 0
    dq = _dims(Q=0)
    assert lib.dflash_attn_anchored(ctypes.byref(dq), 0, None, None, None, None, None, 0, 4, None, None, None, 0,
                                    None) == 0
    assert lib.dflash_attn_ragged(0, 2, 16, 8, 16, 0.0, 0, None, None, None, None, None, None, None, 4, 0, 0, 0,
                                  None, None, None, 0, None) == 0
    del P


def test_workspace_size_contract(lib):
    assert dfl.dflash_attn_workspace_size(dfl.MODE_ANCHORED, 1, 16, 4096, 4096, 128, 64, 128) >= 256
    dense = dfl.dflash_attn_workspace_size(dfl.MODE_DENSE, 4, 32, 8192, 8192, 128, 64, 128)
    assert dense >= 4 * 64 * 128  # one class byte per tile
    assert dfl.dflash_attn_workspace_size(dfl.MODE_DENSE, -1, 32, 8192, 8192, 128, 64, 128) == 0
    assert dfl.dflash_attn_workspace_size(dfl.MODE_RAGGED, H=32, d_nope=128, d_rope=64, d_v=128, R=64,
                                          total_q=1024, total_kv=600000, max_q_len=16) >= 256


@pytest.mark.parametrize("S,nb,bs,B,seed", [
    (64, 4, 4, 1, 0),        # tiny workload shape
    (4096, 256, 16, 1, 1),   # prefill shape
    (300, 23, 8, 2, 2),      # ragged q tail, S not a multiple of 128
    (1000, 30, 12, 2, 3),    # blocks straddle query tiles
    (517, 3, 200, 2, 4),     # blocks larger than a tile
    (0, 5, 16, 1, 5),        # no context at all
    (129, 1, 1, 3, 6),       # single-row blocks
])
def test_host_schedule_bit_exact_vs_bruteforce_scan(lib, S, nb, bs, B, seed):
    rng = np.random.default_rng(seed)
    Q = nb * bs
    an = np.stack([np.sort(rng.choice(np.arange(0, S + 1), size=nb, replace=nb > S + 1)) for _ in range(B)])
    an = an.astype(np.int32)
    an[0, 0] = 0
    an[-1, -1] = S
    got = dfl.dflash_build_schedule_host(B, S, Q, an, bs)
    want = oracle.tile_classes(B, S, Q, 128, 128, anchors=an, block_size=bs)
    np.testing.assert_array_equal(got, want)


def test_host_schedule_rejects_out_of_range_anchor(lib):
    an = np.array([[3, 99]], np.int32)
    with pytest.raises(dfl.DFlashError):
        dfl.dflash_build_schedule_host(1, 50, 8, an, 4)

"""The allocation-free dense entry point (dflash_attn_dense_noalloc).

It serves callers that cannot give the library device scratch memory (memory
planned once at start-up, fixed plugin signatures): the mask-tile classes go to
a fixed array inside the library instead of a caller workspace.  Its results
must match the workspace-based dflash_attn_dense on the same inputs, on two
calls in a row whose masks differ, so that whatever the shared array kept from
the previous call cannot leak into the next result.  This file is collected
last so that a failure here stops a -x run only after every other test ran.
"""
import numpy as np
import pytest

import oracle
from dflash_block_draft_gb300 import synth
from tests.helpers import TOL, bf16_mask, max_abs_err, to_numpy_f64, to_torch

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def dfl():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import dflash_block_draft_gb300 as m
    m.load_library()
    return m


def _case(seed, S, nb, bs):
    d = synth.make("tiny_fp32", seed=seed, dtype="bf16", B=2, H=2, S=S, nb=nb, block_size=bs, d_nope=128,
                   d_rope=64, d_v=128, anchor_lo=0, anchor_hi=S + 1)
    return d, {k: to_torch(d[k], "bf16") for k in ("q", "k_nope", "k_rope", "v")}


def test_noalloc_dense_matches_workspace_dense_on_two_calls(dfl):
    d, t = _case(31, 300, 23, 8)
    rng = np.random.default_rng(4)
    masks = []
    m0 = oracle.build_mask(d["anchors"], 8, 300)
    masks.append(m0)
    m1 = m0.copy()  # second call: a different pattern (extra hidden tiles and a finite bias)
    m1[:, :, :, 128:256] = -np.inf
    m1[1, 0, 3, :5] = rng.normal(size=5)
    masks.append(m1)
    B, Q, H = 2, d["Q"], 2
    for m in masks:
        mk = to_torch(bf16_mask(m), "bf16")
        ref_o = torch.empty((B, Q, H, 128), dtype=torch.bfloat16, device="cuda")
        ref_l = torch.empty((B, H, Q), dtype=torch.float32, device="cuda")
        dfl.dflash_attn_dense(t["q"], t["k_nope"], t["k_rope"], t["v"], mk, out=ref_o, lse=ref_l)
        out = torch.full((B, Q, H, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
        lse = torch.full((B, H, Q), float("nan"), dtype=torch.float32, device="cuda")
        dfl.dflash_attn_dense_noalloc(t["q"], t["k_nope"], t["k_rope"], t["v"], mk, out=out, lse=lse)
        assert dfl.dflash_last_device_error() == 0
        # the same kernels on the same inputs: byte-identical results
        assert torch.equal(out.view(torch.int16), ref_o.view(torch.int16))
        assert torch.equal(lse, ref_l)
        # and both within the bf16 bar of the fp64 oracle on this mask
        want_o, want_l = oracle.dense(d["q"], d["k_nope"], d["k_rope"], d["v"], bf16_mask(m))
        assert max_abs_err(to_numpy_f64(out), want_o) <= TOL["bf16"]
        assert max_abs_err(to_numpy_f64(lse), want_l) <= TOL["bf16"]


def test_noalloc_rejects_problems_beyond_its_fixed_scratch(dfl):
    # 2 x 1024 query tiles x 1024 key tiles > DFLASH_NOALLOC_MAX_TILES: refused before any launch
    big = dfl._Dims(2, 1, 0, 1024 * 128, 128, 64, 128, 0.0)
    import ctypes
    p = ctypes.c_void_p(4096)
    st = dfl.load_library().dflash_attn_dense_noalloc(ctypes.byref(big), 0, p, p, p, p, p, p, None, None)
    assert st == 6  # DFLASH_ERR_WORKSPACE

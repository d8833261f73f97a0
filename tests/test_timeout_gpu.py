"""The bounded-wait failure path of the forward kernels, made to happen on
purpose without faulting the GPU.

Every mbarrier wait of the tensor-core (forward and backward), split-context
decode and latent attention kernels gives up after a budget, records DFLASH_ERR_TIMEOUT in the device error word, and
the CTA winds down (its TMA loads land, its MMAs complete, TMEM is freed).
Here one CTA's producer leaves its first work item's key tiles unloaded (a
phase nothing will complete) under a 20 ms budget; the test checks the error
word, then that a normal call on the same stream is clean and correct.
"""
import time

import numpy as np
import pytest

import oracle
from dflash_block_draft_gb300 import synth
from tests.helpers import TOL, max_abs_err, to_numpy_f64, to_torch

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

DFLASH_ERR_TIMEOUT = 8


@pytest.fixture(scope="module")
def dfl():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import dflash_block_draft_gb300 as m
    m.load_library()
    yield m
    m.dflash_test_inject_stall(0, -1)


def _anchored_case():
    d = synth.make("tiny_fp32", seed=61, dtype="bf16", B=2, H=4, S=1000, nb=40, block_size=16, d_nope=128,
                   d_rope=64, d_v=128, anchor_lo=0, anchor_hi=1001)
    t = {k: to_torch(d[k], "bf16") for k in ("q", "k_nope", "k_rope", "v")}
    return d, t, torch.from_numpy(d["anchors"]).cuda()


def _stalled(dfl, call, stall_cta=0, budget_ns=20_000_000):
    dfl.dflash_test_inject_stall(budget_ns, stall_cta)
    try:
        t0 = time.perf_counter()
        call()
        st = dfl.dflash_last_device_error()
        return st, time.perf_counter() - t0
    finally:
        dfl.dflash_test_inject_stall(0, -1)


@pytest.mark.parametrize("stall_cta", [0, 5])
def test_forward_wait_runs_out_then_context_is_usable(dfl, stall_cta):
    d, t, an = _anchored_case()
    out = torch.empty((2, d["Q"], 4, 128), dtype=torch.bfloat16, device="cuda")
    st, secs = _stalled(dfl, lambda: dfl.dflash_attn_anchored(t["q"], t["k_nope"], t["k_rope"], t["v"], an,
                                                               16, out=out), stall_cta)
    assert st == DFLASH_ERR_TIMEOUT
    assert secs < 1.5  # the call gave up after its short budget, not the 2 s default
    # a normal call on the same stream: no error, results match the oracle
    out2 = torch.full((2, d["Q"], 4, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    dfl.dflash_attn_anchored(t["q"], t["k_nope"], t["k_rope"], t["v"], an, 16, out=out2)
    assert dfl.dflash_last_device_error() == 0
    want, _ = oracle.anchored(d["q"], d["k_nope"], d["k_rope"], d["v"], d["anchors"], 16)
    assert max_abs_err(to_numpy_f64(out2), want) <= TOL["bf16"]


def test_decode_wait_runs_out_then_context_is_usable(dfl):
    d = synth.make("decode_bf16", seed=62, R=6, H=2, ctx_lo=1500, ctx_hi=6000)
    t = {k: to_torch(d[k], "bf16") for k in ("q", "k_nope", "k_rope", "v")}
    qo, ko, an = (torch.from_numpy(d[k]).cuda() for k in ("q_offsets", "kv_offsets", "anchors"))
    out = torch.empty((d["total_q"], 2, 128), dtype=torch.bfloat16, device="cuda")

    def call(o):
        dfl.dflash_attn_ragged(t["q"], t["k_nope"], t["k_rope"], t["v"], qo, ko, an, 16, 16, out=o)

    st, secs = _stalled(dfl, lambda: call(out))
    assert st == DFLASH_ERR_TIMEOUT and secs < 1.5
    out2 = torch.full_like(out, float("nan"))
    call(out2)
    assert dfl.dflash_last_device_error() == 0
    want, _ = oracle.ragged(d["q"], d["k_nope"], d["k_rope"], d["v"], d["q_offsets"], d["kv_offsets"],
                            d["anchors"], 16)
    assert max_abs_err(to_numpy_f64(out2), want) <= TOL["bf16"]


def test_latent_wait_runs_out_then_context_is_usable(dfl, monkeypatch):
    """The absorbed latent attention kernel (bf16 decode shape): one CTA's
    producer leaves its first unit's key tiles unloaded."""
    monkeypatch.delenv("DFLASH_LATENT_EXPAND", raising=False)
    d = synth.make("decode_latent_bf16", seed=63, R=4, H=8, ctx_lo=1500, ctx_hi=5000)
    t = {k: to_torch(d[k], "bf16") for k in ("q", "c_kv", "k_rope", "w_kv_b")}
    qo, ko, an = (torch.from_numpy(d[k]).cuda() for k in ("q_offsets", "kv_offsets", "anchors"))
    out = torch.empty((d["total_q"], 8, 128), dtype=torch.bfloat16, device="cuda")

    def call(o):
        dfl.dflash_attn_latent_ragged(t["q"], t["c_kv"], t["k_rope"], t["w_kv_b"], qo, ko, an, d["block_size"], 16,
                                      out=o)

    st, secs = _stalled(dfl, lambda: call(out))
    assert st == DFLASH_ERR_TIMEOUT and secs < 1.5
    out2 = torch.full_like(out, float("nan"))
    call(out2)
    assert dfl.dflash_last_device_error() == 0
    want, _ = oracle.latent_ragged(d["q"], d["c_kv"], d["k_rope"], d["w_kv_b"], d["q_offsets"], d["kv_offsets"],
                                   d["anchors"], d["block_size"])
    assert max_abs_err(to_numpy_f64(out2), want) <= TOL["bf16"]


def test_backward_wait_runs_out_then_context_is_usable(dfl, monkeypatch):
    """The tensor-core backward kernels (dq and dk/dv): CTA 0 of each grid gets
    no key (dq) or query (dk/dv) tiles."""
    monkeypatch.delenv("DFLASH_FORCE_SIMT", raising=False)
    d = synth.make("tiny_fp32", seed=64, dtype="bf16", B=1, H=2, S=600, nb=20, block_size=16, d_nope=128,
                   d_rope=64, d_v=128, anchor_lo=0, anchor_hi=601)
    d["dout"] = synth.make_dout(d)
    t = {k: to_torch(d[k], "bf16") for k in ("q", "k_nope", "k_rope", "v", "dout")}
    an = torch.from_numpy(d["anchors"]).cuda()
    out = torch.empty((1, d["Q"], 2, 128), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((1, 2, d["Q"]), dtype=torch.float32, device="cuda")
    dfl.dflash_attn_anchored(t["q"], t["k_nope"], t["k_rope"], t["v"], an, 16, out=out, lse=lse)
    assert dfl.dflash_last_device_error() == 0

    def call():
        return dfl.dflash_attn_anchored_backward(t["q"], t["k_nope"], t["k_rope"], t["v"], an, 16, out, lse,
                                                 t["dout"])

    st, secs = _stalled(dfl, call)
    assert st == DFLASH_ERR_TIMEOUT and secs < 1.5
    got = [to_numpy_f64(x) for x in call()]
    assert dfl.dflash_last_device_error() == 0
    want = oracle.backward(d["q"], d["k_nope"], d["k_rope"], d["v"], d["dout"], anchors=d["anchors"],
                           block_size=16)
    for name, g, w in zip(("dq", "dk_nope", "dk_rope", "dv"), got, want):
        np.testing.assert_allclose(g, w, atol=2e-2, rtol=2.0 ** -7, err_msg=name)


def test_no_stall_leaves_the_default_budget(dfl):
    """With the knob cleared, a call is clean (nothing left over from the tests above)."""
    d, t, an = _anchored_case()
    dfl.dflash_attn_anchored(t["q"], t["k_nope"], t["k_rope"], t["v"], an, 16)
    assert dfl.dflash_last_device_error() == 0

"""GPU parity of the backward entry points against the fp64 backward oracle.

Each case runs the library's forward (for out and lse), then its backward,
through the C ABI, and compares every gradient element with oracle.backward
on the same seeded inputs.

Tolerances.  fp32: the forward's bar of 1e-5 absolute, plus 1e-5 relative for
the head-summed dk_rope.  bf16: the gradients accumulate in fp32 and are
rounded once to bf16 (half an ulp is 2^-9 relative); on the tensor-core path P
and dS enter their MMAs as bf16, and D = dout . out uses the forward's
bf16-rounded out.  The bar is 2e-2 absolute (the forward's bar) plus 2^-7
relative, which covers the rounding of gradients larger than 1.
"""
import numpy as np
import pytest

import oracle
from dflash_block_draft_gb300 import synth
from tests.helpers import bf16_mask, to_numpy_f64, to_torch

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

RTOL = {"fp32": 1e-5, "bf16": 2.0 ** -7}
ATOL = {"fp32": 1e-5, "bf16": 2e-2}


@pytest.fixture(params=["default", "simt"])
def kernel(request, monkeypatch):
    """Default dispatch (tensor-core kernels for bf16 with the Kimi K3 MLA head
    dims) or the CUDA-core kernels forced for every shape."""
    if request.param == "simt":
        monkeypatch.setenv("DFLASH_FORCE_SIMT", "1")
    else:
        monkeypatch.delenv("DFLASH_FORCE_SIMT", raising=False)
    return request.param


@pytest.fixture(scope="module")
def dfl():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import dflash_block_draft_gb300 as m
    m.load_library()
    return m


def _case(dtype, B, H, S, nb, bs, dn, dr, dv, seed=321, lo=0):
    d = synth.make("tiny_fp32", seed=seed, dtype=dtype, B=B, H=H, S=S, nb=nb, block_size=bs, d_nope=dn,
                   d_rope=dr, d_v=dv, anchor_lo=lo, anchor_hi=S + 1)
    d["dout"] = synth.make_dout(d)
    return d


def _gpu(dfl, d, dtype, mask=None):
    t = {k: to_torch(d[k], dtype) for k in ("q", "k_nope", "k_rope", "v", "dout")}
    B, Q, H, dv = d["B"], d["Q"], d["H"], d["d_v"]
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    out = torch.empty((B, Q, H, dv), dtype=tdt, device="cuda")
    lse = torch.empty((B, H, Q), dtype=torch.float32, device="cuda")
    # NaN-filled gradients: every element must be written
    grads = tuple(torch.full_like(t[k], float("nan")) for k in ("q", "k_nope", "k_rope", "v"))
    if mask is None:
        an = torch.from_numpy(d["anchors"]).cuda()
        dfl.dflash_attn_anchored(t["q"], t["k_nope"], t["k_rope"], t["v"], an, d["block_size"], out=out, lse=lse)
        g = dfl.dflash_attn_anchored_backward(t["q"], t["k_nope"], t["k_rope"], t["v"], an, d["block_size"], out,
                                              lse, t["dout"], grads=grads)
    else:
        m = to_torch(mask, dtype)
        dfl.dflash_attn_dense(t["q"], t["k_nope"], t["k_rope"], t["v"], m, out=out, lse=lse)
        g = dfl.dflash_attn_dense_backward(t["q"], t["k_nope"], t["k_rope"], t["v"], m, out, lse, t["dout"],
                                           grads=grads)
    assert dfl.dflash_last_device_error() == 0
    return [to_numpy_f64(x) for x in g]


def _oracle(d, mask=None, pairs=None):
    if mask is None:
        return oracle.backward(d["q"], d["k_nope"], d["k_rope"], d["v"], d["dout"], anchors=d["anchors"],
                               block_size=d["block_size"], pairs=pairs)
    return oracle.backward(d["q"], d["k_nope"], d["k_rope"], d["v"], d["dout"], mask=mask, pairs=pairs)


def _compare(got, want, dtype, names=("dq", "dk_nope", "dk_rope", "dv")):
    for name, g, w in zip(names, got, want):
        assert not np.isnan(g).any(), f"{name}: unwritten elements"
        np.testing.assert_allclose(g, w, atol=ATOL[dtype], rtol=RTOL[dtype], err_msg=name)


def _mask(d, dtype, finite_noise=False, seed=5):
    mask = oracle.build_mask(d["anchors"], d["block_size"], d["S"])
    if finite_noise:
        rng = np.random.default_rng(seed)
        vis = mask == 0
        mask = np.where(vis, rng.uniform(-2, 2, mask.shape).astype(np.float32), mask)
    if dtype == "bf16":
        bits = bf16_mask(mask)
        return bits, synth.bf16_bits_to_f32(bits)
    return mask, mask


CASES = [
    # name, dtype, B, H, S, nb, bs, dn, dr, dv
    ("tiny_fp32_workload_shape", "fp32", 1, 2, 64, 4, 4, 16, 8, 16),
    ("fp32_ragged_tails", "fp32", 2, 2, 37, 5, 3, 16, 8, 16),
    ("fp32_general_dims", "fp32", 1, 2, 150, 6, 10, 40, 24, 48),
    ("bf16_mla_multi_tile", "bf16", 1, 2, 300, 20, 16, 128, 64, 128),
    ("bf16_mla_bs8_two_rows", "bf16", 2, 2, 200, 25, 8, 128, 64, 128),
    ("fp32_widest_dims", "fp32", 1, 1, 70, 3, 8, 192, 64, 128),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_anchored_backward_every_element(dfl, case, kernel):
    _, dtype, B, H, S, nb, bs, dn, dr, dv = case
    d = _case(dtype, B, H, S, nb, bs, dn, dr, dv)
    _compare(_gpu(dfl, d, dtype), _oracle(d), dtype)


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
def test_dense_backward_with_finite_mask_values(dfl, dtype, kernel):
    dn, dr, dv = (128, 64, 128) if dtype == "bf16" else (16, 8, 16)
    d = _case(dtype, 2, 2, 140, 9, 16, dn, dr, dv, seed=77)
    dev_mask, ora_mask = _mask(d, dtype, finite_noise=True)
    _compare(_gpu(dfl, d, dtype, mask=dev_mask), _oracle(d, mask=ora_mask), dtype)


def test_dense_backward_row_with_no_visible_key(dfl):
    d = _case("fp32", 1, 2, 40, 4, 4, 16, 8, 16, seed=9)
    mask, _ = _mask(d, "fp32")
    mask[0, 0, 5, :] = -np.inf
    got = _gpu(dfl, d, "fp32", mask=mask)
    _compare(got, _oracle(d, mask=mask), "fp32")
    assert np.all(got[0][0, 5] == 0.0)


def test_dense_from_anchors_equals_anchored_backward(dfl, kernel):
    d = _case("bf16", 1, 2, 260, 10, 16, 128, 64, 128, seed=17)
    dev_mask, _ = _mask(d, "bf16")
    a = _gpu(dfl, d, "bf16")
    b = _gpu(dfl, d, "bf16", mask=dev_mask)
    for x, y in zip(a, b):
        np.testing.assert_allclose(x, y, atol=ATOL["bf16"], rtol=RTOL["bf16"])


def test_keys_no_row_sees_get_zero_gradients(dfl):
    # anchors well below S: context keys past the largest anchor are seen by no row
    d = _case("fp32", 1, 2, 90, 3, 4, 16, 8, 16, seed=4, lo=0)
    d["anchors"][:] = np.array([[5, 9, 20]], np.int32)
    got = _gpu(dfl, d, "fp32")
    _compare(got, _oracle(d), "fp32")
    assert np.all(got[1][0, 20:90] == 0.0) and np.all(got[2][0, 20:90] == 0.0) and np.all(got[3][0, 20:90] == 0.0)


_PREFILL = {}


def _prefill_case():
    if not _PREFILL:
        d = synth.make("prefill_bf16")
        d["dout"] = synth.make_dout(d)
        _PREFILL["d"] = d
        _PREFILL["want"] = _oracle(d)
    return _PREFILL["d"], _PREFILL["want"]


def test_backward_prefill_workload_every_element(dfl, kernel):
    # The bf16 prefill workload at full size (B=1 H=16 S=4096 nb=256
    # block_size=16), every gradient element against the oracle (whose (b, h)
    # pairs run on all host cores).
    d, want = _prefill_case()
    _compare(_gpu(dfl, d, "bf16"), want, "bf16")


def test_backward_training_workload_sampled_heads(dfl):
    """The bf16 training workload at full size (B=4 H=32 S=8192 nb=512
    block_size=16), in the launch configuration the benchmark times: every
    element of dq, dk_nope and dv of two (batch row, head) pairs, the first and
    the last, against the oracle evaluated on those pairs alone (dk_rope sums
    over all heads, so it is left to the every-element tests)."""
    d = synth.make("training_bf16")
    d["dout"] = synth.make_dout(d)
    got = _gpu(dfl, d, "bf16")
    B, H = d["B"], d["H"]
    pairs = [(0, 0), (B - 1, H - 1)]
    want = _oracle(d, pairs=[b * H + h for b, h in pairs])
    for b, h in pairs:
        for name, i in (("dq", 0), ("dk_nope", 1), ("dv", 3)):
            np.testing.assert_allclose(got[i][b, :, h], want[i][b, :, h], atol=ATOL["bf16"], rtol=RTOL["bf16"],
                                       err_msg=f"{name} (b={b}, h={h})")


@pytest.mark.parametrize("shape", [
    # B, H, S, nb, bs: query and key tails that are not multiples of 64 or 128
    (2, 2, 77, 9, 7),
    (1, 3, 0, 1, 16),     # no context: only noise keys
    (3, 1, 130, 1, 16),   # one block per batch row; the next row's keys share a tile
])
def test_tc_backward_tails_every_element(dfl, shape, kernel):
    B, H, S, nb, bs = shape
    d = _case("bf16", B, H, S, nb, bs, 128, 64, 128, seed=sum(shape))
    _compare(_gpu(dfl, d, "bf16"), _oracle(d), "bf16")


def test_backward_without_query_rows_zeroes_key_gradients(dfl):
    # nb = 0 blocks: no query row sees anything, so every key gradient is 0
    B, H, S = 2, 2, 50
    q = torch.empty((B, 0, H, 192), dtype=torch.bfloat16, device="cuda")
    kn = torch.randn((B, S, H, 128), device="cuda").to(torch.bfloat16)
    kr = torch.randn((B, S, 64), device="cuda").to(torch.bfloat16)
    v = torch.randn((B, S, H, 128), device="cuda").to(torch.bfloat16)
    an = torch.empty((B, 0), dtype=torch.int32, device="cuda")
    out = torch.empty((B, 0, H, 128), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((B, H, 0), dtype=torch.float32, device="cuda")
    grads = (torch.empty_like(q), torch.full_like(kn, float("nan")), torch.full_like(kr, float("nan")),
             torch.full_like(v, float("nan")))
    g = dfl.dflash_attn_anchored_backward(q, kn, kr, v, an, 16, out, lse, out, grads=grads)
    torch.cuda.synchronize()
    assert dfl.dflash_last_device_error() == 0
    for x in g[1:]:
        assert torch.all(x == 0)


def test_backward_out_of_range_anchor_is_reported(dfl):
    d = _case("bf16", 1, 2, 100, 4, 16, 128, 64, 128, seed=8)
    t = {k: to_torch(d[k], "bf16") for k in ("q", "k_nope", "k_rope", "v", "dout")}
    out = torch.empty((1, d["Q"], 2, 128), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((1, 2, d["Q"]), dtype=torch.float32, device="cuda")
    an = torch.from_numpy(d["anchors"]).cuda()
    dfl.dflash_attn_anchored(t["q"], t["k_nope"], t["k_rope"], t["v"], an, 16, out=out, lse=lse)
    assert dfl.dflash_last_device_error() == 0
    an[0, 1] = 10_000  # beyond S
    dfl.dflash_attn_anchored_backward(t["q"], t["k_nope"], t["k_rope"], t["v"], an, 16, out, lse, t["dout"])
    assert dfl.dflash_last_device_error() == 1  # DFLASH_ERR_INVALID


def test_bf16_dense_backward_row_with_no_visible_key(dfl, kernel):
    d = _case("bf16", 1, 2, 150, 9, 16, 128, 64, 128, seed=12)
    bits, widened = _mask(d, "bf16", finite_noise=True)
    bits = bits.copy()
    widened = widened.copy()
    neg = synth.f32_to_bf16_bits(np.array([-np.inf], np.float32))[0]
    bits[0, 0, 37, :] = neg
    widened[0, 0, 37, :] = -np.inf
    got = _gpu(dfl, d, "bf16", mask=bits)
    _compare(got, _oracle(d, mask=widened), "bf16")
    assert np.all(got[0][0, 37] == 0.0)


@pytest.mark.parametrize("masked", [False, True], ids=["anchored", "dense"])
@pytest.mark.parametrize("limit", [1, 3])
def test_tc_backward_tiles_past_the_flag_table(dfl, limit, masked, monkeypatch):
    """The tensor-core backward works out once per CTA which tiles it needs (and
    which need no per-pair mask) into a shared-memory table, and the tiles past
    the table when they come up.  With the table capped at `limit` entries most
    tiles (of 10 key tiles for dq, 5 query tiles for dk/dv) take that path: the
    gradients still match the oracle, and dq, dk_nope and dv (no atomics) are
    bit-identical to those of the full table."""
    monkeypatch.delenv("DFLASH_FORCE_SIMT", raising=False)
    d = _case("bf16", 1, 2, 300, 20, 16, 128, 64, 128, seed=41)
    dev_mask, ora_mask = _mask(d, "bf16") if masked else (None, None)
    full = _gpu(dfl, d, "bf16", mask=dev_mask)
    try:
        dfl.dflash_test_limit_tile_flags(limit)
        got = _gpu(dfl, d, "bf16", mask=dev_mask)
    finally:
        dfl.dflash_test_limit_tile_flags(0)
    _compare(got, _oracle(d, mask=ora_mask), "bf16")
    for i in (0, 1, 3):
        np.testing.assert_array_equal(got[i], full[i])

"""GPU parity: the CUDA library (through its C ABI) against the fp64 oracle.

Small cases are compared element by element over every row; the full-size
workloads (in the launch configuration the benchmark times) are compared on a
deterministic sample of rows that the oracle evaluates one by one.  Bars: max
abs error 1e-5 (fp32) and 2e-2 (bf16) on out and lse.
"""
import os

import numpy as np
import pytest

import oracle
from dflash_block_draft_gb300 import synth
from tests.helpers import TOL, bf16_mask, max_abs_err, sample_rows, to_numpy_f64, to_torch

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def dfl():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import dflash_block_draft_gb300 as m
    m.load_library()
    return m


def _mask_for(d, dtype):
    mask = oracle.build_mask(d["anchors"], d["block_size"], d["S"])
    if d.get("pad"):
        mask[:, :, :, d["S"] - d["pad"]:d["S"]] = -np.inf
    return bf16_mask(mask) if dtype == "bf16" else mask


def _dev(d, dtype):
    return {k: to_torch(d[k], dtype) for k in ("q", "k_nope", "k_rope", "v")}


def _run_batched(dfl, d, mode, dtype, mask=None, scale=0.0):
    t = _dev(d, dtype)
    B, Q, H, dv = d["B"], d["Q"], d["H"], d["d_v"]
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    out = torch.full((B, Q, H, dv), float("nan"), dtype=tdt, device="cuda")
    lse = torch.full((B, H, Q), float("nan"), dtype=torch.float32, device="cuda")
    if mode == "anchored":
        an = torch.from_numpy(d["anchors"]).cuda()
        dfl.dflash_attn_anchored(t["q"], t["k_nope"], t["k_rope"], t["v"], an, d["block_size"], out=out, lse=lse,
                                 scale=scale)
    else:
        m = to_torch(mask, dtype)
        dfl.dflash_attn_dense(t["q"], t["k_nope"], t["k_rope"], t["v"], m, out=out, lse=lse, scale=scale)
    assert dfl.dflash_last_device_error() == 0
    return to_numpy_f64(out), to_numpy_f64(lse)


SMALL = [
    # name, dtype, B, H, S, nb, bs, dn, dr, dv
    ("tc_shape_ragged_tails", "bf16", 2, 3, 300, 23, 8, 128, 64, 128),
    ("tc_shape_multi_tile", "bf16", 1, 2, 1024, 40, 16, 128, 64, 128),
    ("tc_shape_bs4", "bf16", 1, 2, 700, 70, 4, 128, 64, 128),
    ("general_dims_fp32", "fp32", 2, 2, 200, 7, 12, 40, 24, 48),
    ("general_dims_bf16", "bf16", 1, 3, 150, 10, 4, 32, 16, 64),
    ("wide_blocks_fp32", "fp32", 1, 2, 90, 2, 150, 16, 8, 16),
    # one block per row: the last key tile is FULL on its clipped extent and runs into the next row's keys
    ("tc_one_block_straddle", "bf16", 3, 2, 300, 1, 16, 128, 64, 128),
]


def _small_case(dtype, B, H, S, nb, bs, dn, dr, dv, seed=123):
    return synth.make("tiny_fp32", seed=seed, dtype=dtype, B=B, H=H, S=S, nb=nb, block_size=bs, d_nope=dn,
                      d_rope=dr, d_v=dv, anchor_lo=0, anchor_hi=S + 1)


@pytest.fixture(params=["default", "simt"])
def kernel(request, monkeypatch):
    """Run a case on the default dispatch (tensor cores for the Kimi K3 MLA bf16
    shape) and with the exact CUDA-core kernel forced."""
    monkeypatch.delenv("DFLASH_FORCE_SIMT", raising=False)
    if request.param == "simt":
        monkeypatch.setenv("DFLASH_FORCE_SIMT", "1")
    return request.param


@pytest.mark.parametrize("case", SMALL, ids=[c[0] for c in SMALL])
@pytest.mark.parametrize("mode", ["anchored", "dense"])
def test_small_cases_every_row(dfl, case, mode, kernel):
    name, dtype, B, H, S, nb, bs, dn, dr, dv = case
    d = _small_case(dtype, B, H, S, nb, bs, dn, dr, dv)
    d["anchors"][0, 0] = 0  # own block only
    d["anchors"][-1, -1] = S  # all context
    want_o, want_l = oracle.anchored(d["q"], d["k_nope"], d["k_rope"], d["v"], d["anchors"], bs)
    mask = _mask_for(d, dtype) if mode == "dense" else None
    got_o, got_l = _run_batched(dfl, d, mode, dtype, mask)
    assert not np.isnan(got_o).any() and not np.isnan(got_l).any()
    assert max_abs_err(got_o, want_o) <= TOL[dtype], name
    assert max_abs_err(got_l, want_l) <= TOL[dtype], name


@pytest.mark.parametrize("shape", ["zero", "all_context", "no_context", "unsorted"])
@pytest.mark.parametrize("mode", ["anchored", "dense"])
def test_degenerate_anchors_every_row(dfl, shape, mode, kernel):
    """The extreme cases of the anchored rule on the tensor-core shape: every
    block sees only itself (all anchors 0), every block sees the whole context
    (all anchors S), there is no context at all (S = 0), and anchors in no
    order with repeats (the schedule uses per-tile min/max, not order)."""
    S = 0 if shape == "no_context" else 500
    d = synth.make("tiny_fp32", seed=321, dtype="bf16", B=2, H=2, S=S, nb=37, block_size=8, d_nope=128, d_rope=64,
                   d_v=128, anchor_lo=0, anchor_hi=S + 38)
    rng = np.random.default_rng(9)
    if shape in ("zero", "no_context"):
        d["anchors"][:] = 0
    elif shape == "all_context":
        d["anchors"][:] = S
    else:
        d["anchors"][:] = rng.integers(0, S + 1, size=d["anchors"].shape).astype(np.int32)
        d["anchors"][:, 5] = d["anchors"][:, 6]
    want_o, want_l = oracle.anchored(d["q"], d["k_nope"], d["k_rope"], d["v"], d["anchors"], d["block_size"])
    mask = _mask_for(d, "bf16") if mode == "dense" else None
    got_o, got_l = _run_batched(dfl, d, mode, "bf16", mask)
    assert not np.isnan(got_o).any() and not np.isnan(got_l).any()
    assert max_abs_err(got_o, want_o) <= TOL["bf16"], shape
    assert max_abs_err(got_l, want_l) <= TOL["bf16"], shape


def test_tiny_fp32_workload_all_entry_points(dfl):
    d = synth.make("tiny_fp32")
    want_o, want_l = oracle.anchored(d["q"], d["k_nope"], d["k_rope"], d["v"], d["anchors"], d["block_size"])
    for mode in ("anchored", "dense"):
        got_o, got_l = _run_batched(dfl, d, mode, "fp32", _mask_for(d, "fp32") if mode == "dense" else None)
        assert max_abs_err(got_o, want_o) <= 1e-5 and max_abs_err(got_l, want_l) <= 1e-5, mode


def test_dense_general_mask_with_finite_values_and_empty_rows(dfl):
    d = _small_case("fp32", 2, 2, 100, 9, 8, 16, 8, 16, seed=5)
    rng = np.random.default_rng(3)
    mask = rng.normal(0, 2, size=(2, 1, d["Q"], d["S"] + d["Q"])).astype(np.float32)
    mask[rng.random(mask.shape) < 0.5] = -np.inf
    mask[:, :, :, 128:200] = -np.inf  # whole -inf tiles on part of the grid
    mask[1, 0, 7, :] = -np.inf  # a row that sees nothing
    want_o, want_l = oracle.dense(d["q"], d["k_nope"], d["k_rope"], d["v"], mask, scale=0.3)
    got_o, got_l = _run_batched(dfl, d, "dense", "fp32", mask, scale=0.3)
    assert max_abs_err(got_o, want_o) <= 1e-5
    assert max_abs_err(got_l, want_l) <= 1e-5
    assert np.all(got_o[1, 7] == 0) and np.all(np.isneginf(got_l[1, :, 7]))


def test_output_only_16_byte_aligned(dfl):
    """The tensor-core kernel writes rows with 32-byte stores when `out` is 32-byte
    aligned and with 16-byte stores otherwise; both give the same bytes."""
    d = _small_case("bf16", 1, 2, 1024, 40, 16, 128, 64, 128)
    t = _dev(d, "bf16")
    an = torch.from_numpy(d["anchors"]).cuda()
    B, Q, H, dv = d["B"], d["Q"], d["H"], d["d_v"]
    ref = dfl.dflash_attn_anchored(t["q"], t["k_nope"], t["k_rope"], t["v"], an, d["block_size"])
    flat = torch.full((B * Q * H * dv + 8,), float("nan"), dtype=torch.bfloat16, device="cuda")
    out = flat[8:].view(B, Q, H, dv)  # 16 bytes past a 32-byte boundary
    assert out.data_ptr() % 32 == 16
    dfl.dflash_attn_anchored(t["q"], t["k_nope"], t["k_rope"], t["v"], an, d["block_size"], out=out)
    assert dfl.dflash_last_device_error() == 0
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    assert torch.isnan(flat[:8]).all()  # nothing written before the output


def test_single_visible_key_returns_value_row_exactly(dfl, kernel):
    d = _small_case("bf16", 1, 2, 200, 20, 8, 128, 64, 128, seed=9)
    Q, K = d["Q"], d["S"] + d["Q"]
    mask = np.full((1, 1, Q, K), -np.inf, np.float32)
    pick = np.random.default_rng(2).integers(0, K, size=Q)
    mask[0, 0, np.arange(Q), pick] = 0.0
    got_o, got_l = _run_batched(dfl, d, "dense", "bf16", bf16_mask(mask))
    vals = synth.bf16_bits_to_f32(d["v"]).astype(np.float64)
    np.testing.assert_array_equal(got_o[0], vals[0, pick])


def test_dense_from_anchors_equals_anchored(dfl, kernel):
    d = _small_case("bf16", 2, 2, 600, 30, 16, 128, 64, 128, seed=11)
    a_o, a_l = _run_batched(dfl, d, "anchored", "bf16")
    d_o, d_l = _run_batched(dfl, d, "dense", "bf16", _mask_for(d, "bf16"))
    assert max_abs_err(a_o, d_o) <= TOL["bf16"] and max_abs_err(a_l, d_l) <= 1e-4


def test_mask_scan_bit_exact_vs_bruteforce(dfl):
    for dtype, (S, nb, bs) in (("bf16", (300, 23, 8)), ("fp32", (1000, 30, 12)), ("bf16", (8192 - 96, 64, 16))):
        d = _small_case(dtype, 2, 1, S, nb, bs, 8, 8, 8, seed=S)
        mask = oracle.build_mask(d["anchors"], bs, S)
        rng = np.random.default_rng(0)
        mask[0, 0, 5, 7] = 0.5  # a finite non-zero entry forces PARTIAL
        mask[1, 0, :, :3] = rng.normal(size=(nb * bs, 3))
        want = oracle.tile_classes(2, S, nb * bs, 128, 128, mask=mask)
        m = to_torch(bf16_mask(mask) if dtype == "bf16" else mask, dtype)
        got = dfl.dflash_scan_mask(m).cpu().numpy()
        np.testing.assert_array_equal(got, want)


@pytest.mark.parametrize("dtype,S,nb,bs", [("bf16", 300, 23, 8), ("fp32", 1000, 30, 12), ("bf16", 4096, 256, 16)])
def test_device_mask_builder_bit_exact_vs_oracle(dfl, dtype, S, nb, bs):
    d = _small_case(dtype, 2, 1, S, nb, bs, 8, 8, 8, seed=S + nb)
    d["anchors"][0, 0] = 0
    d["anchors"][-1, -1] = S
    want = oracle.build_mask(d["anchors"], bs, S)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    got = dfl.dflash_build_mask(torch.from_numpy(d["anchors"]).cuda(), bs, S, dtype=tdt).float().cpu().numpy()
    np.testing.assert_array_equal(got, want)


def test_outputs_fully_written_and_guard_bands_untouched(dfl):
    d = _small_case("bf16", 1, 2, 260, 13, 8, 128, 64, 128, seed=13)
    t = _dev(d, "bf16")
    B, Q, H, dv = 1, d["Q"], 2, 128
    guard = 4096
    buf = torch.full((guard * 2 + B * Q * H * dv,), 7.0, dtype=torch.bfloat16, device="cuda")
    out = buf[guard:guard + B * Q * H * dv].view(B, Q, H, dv)
    out.fill_(float("nan"))
    an = torch.from_numpy(d["anchors"]).cuda()
    dfl.dflash_attn_anchored(t["q"], t["k_nope"], t["k_rope"], t["v"], an, 8, out=out)
    torch.cuda.synchronize()
    assert not torch.isnan(out).any()
    assert torch.all(buf[:guard] == 7.0) and torch.all(buf[guard + B * Q * H * dv:] == 7.0)


def test_out_of_range_anchor_is_reported_on_device(dfl):
    d = _small_case("fp32", 1, 1, 50, 4, 4, 8, 8, 8, seed=17)
    d["anchors"][0, 1] = 51  # > S
    t = _dev(d, "fp32")
    an = torch.from_numpy(d["anchors"]).cuda()
    dfl.dflash_attn_anchored(t["q"], t["k_nope"], t["k_rope"], t["v"], an, 4)
    assert dfl.dflash_last_device_error() == 1
    assert dfl.dflash_last_device_error() == 0  # read clears it


def test_empty_batch_is_a_no_op(dfl):
    q = torch.empty((0, 16, 2, 24), device="cuda")
    kn = torch.empty((0, 40, 2, 16), device="cuda")
    kr = torch.empty((0, 40, 8), device="cuda")
    v = torch.empty((0, 40, 2, 16), device="cuda")
    an = torch.empty((0, 4), dtype=torch.int32, device="cuda")
    out = dfl.dflash_attn_anchored(q, kn, kr, v, an, 4)
    assert out.shape == (0, 16, 2, 16)


# ---------------------------------------------------------------------------
# ragged
# ---------------------------------------------------------------------------
def _run_ragged(dfl, d, dtype, max_q_len=None):
    t = _dev(d, dtype)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    out = torch.full((d["total_q"], d["H"], d["d_v"]), float("nan"), dtype=tdt, device="cuda")
    lse = torch.full((d["H"], d["total_q"]), float("nan"), dtype=torch.float32, device="cuda")
    qo, ko, an = (torch.from_numpy(d[k]).cuda() for k in ("q_offsets", "kv_offsets", "anchors"))
    mq = max_q_len or int(np.diff(d["q_offsets"]).max())
    dfl.dflash_attn_ragged(t["q"], t["k_nope"], t["k_rope"], t["v"], qo, ko, an, d["block_size"], mq, out=out,
                           lse=lse)
    assert dfl.dflash_last_device_error() == 0
    return to_numpy_f64(out), to_numpy_f64(lse)


@pytest.mark.parametrize("dtype,dn,dr,dv", [("bf16", 128, 64, 128), ("fp32", 16, 8, 16)])
def test_ragged_small_every_row(dfl, dtype, dn, dr, dv, kernel):
    d = synth.make("decode_bf16", seed=77, dtype=dtype, R=7, H=3, d_nope=dn, d_rope=dr, d_v=dv, ctx_lo=1,
                   ctx_hi=700, nb=3, block_size=8)
    # vary the anchors inside each request (they need not equal the context length)
    rng = np.random.default_rng(1)
    for r in range(7):
        S_r = int(d["kv_offsets"][r + 1] - d["kv_offsets"][r]) - 24
        d["anchors"][3 * r:3 * r + 3] = np.sort(rng.integers(0, S_r + 1, size=3))
    want_o, want_l = oracle.ragged(d["q"], d["k_nope"], d["k_rope"], d["v"], d["q_offsets"], d["kv_offsets"],
                                   d["anchors"], 8)
    got_o, got_l = _run_ragged(dfl, d, dtype)
    assert max_abs_err(got_o, want_o) <= TOL[dtype]
    assert max_abs_err(got_l, want_l) <= TOL[dtype]


def test_ragged_decode_shape_small(dfl, kernel):
    # decode shape (one block per request, anchor = context length) with short contexts
    d = synth.make("decode_bf16", seed=80, R=9, H=3, ctx_lo=5, ctx_hi=700)
    want_o, want_l = oracle.ragged(d["q"], d["k_nope"], d["k_rope"], d["v"], d["q_offsets"], d["kv_offsets"],
                                   d["anchors"], d["block_size"])
    got_o, got_l = _run_ragged(dfl, d, "bf16")
    assert max_abs_err(got_o, want_o) <= TOL["bf16"]
    assert max_abs_err(got_l, want_l) <= TOL["bf16"]


@pytest.mark.parametrize("bs,nb,seed", [(16, 1, 81), (8, 2, 82), (4, 4, 83)])
def test_ragged_decode_split_context_every_row(dfl, bs, nb, seed):
    # 16 draft rows per request (split-context kernels), contexts that cross the
    # 4096-key split boundaries, anchors anywhere in [0, S_r]
    d = synth.make("decode_bf16", seed=seed, R=6, H=2, ctx_lo=1500, ctx_hi=9000, nb=nb, block_size=bs)
    rng = np.random.default_rng(seed)
    for r in range(6):
        S_r = int(d["kv_offsets"][r + 1] - d["kv_offsets"][r]) - 16
        d["anchors"][nb * r:nb * r + nb] = np.sort(rng.integers(0, S_r + 1, size=nb))
    d["anchors"][0] = 0
    want_o, want_l = oracle.ragged(d["q"], d["k_nope"], d["k_rope"], d["v"], d["q_offsets"], d["kv_offsets"],
                                   d["anchors"], bs)
    got_o, got_l = _run_ragged(dfl, d, "bf16")
    assert max_abs_err(got_o, want_o) <= TOL["bf16"]
    assert max_abs_err(got_l, want_l) <= TOL["bf16"]


@pytest.mark.parametrize("dtype,dn,dr,dv,bs,q_blocks", [
    ("bf16", 128, 64, 128, 16, (1, 2, 3)),     # max_q_len 48: one query tile per request
    ("bf16", 128, 64, 128, 8, (1, 20, 40)),    # up to 320 rows: several query tiles, ragged tails
    ("fp32", 16, 8, 16, 8, (1, 3, 7)),
])
def test_ragged_mixed_lengths_every_row(dfl, dtype, dn, dr, dv, bs, q_blocks, kernel):
    """Requests with different draft lengths (q_offsets[r] != r * q_len), so a
    request's anchors start at its own global block q_offsets[r] / bs."""
    d = synth.make("decode_bf16", seed=90 + bs, dtype=dtype, R=9, H=3, d_nope=dn, d_rope=dr, d_v=dv, ctx_lo=1,
                   ctx_hi=900, block_size=bs, q_blocks=q_blocks)
    assert len(set(np.diff(d["q_offsets"]).tolist())) > 1
    want_o, want_l = oracle.ragged(d["q"], d["k_nope"], d["k_rope"], d["v"], d["q_offsets"], d["kv_offsets"],
                                   d["anchors"], bs)
    got_o, got_l = _run_ragged(dfl, d, dtype)
    assert not np.isnan(got_o).any() and not np.isnan(got_l).any()
    assert max_abs_err(got_o, want_o) <= TOL[dtype]
    assert max_abs_err(got_l, want_l) <= TOL[dtype]


@pytest.mark.parametrize("seed", [95, 96])
def test_ragged_decode_mixed_lengths_split_context_every_row(dfl, seed):
    """The split-context decode path (max_q_len <= 16) with requests of 8 and 16
    rows and contexts that cross the 4096-key split boundaries."""
    d = synth.make("decode_bf16", seed=seed, R=8, H=2, ctx_lo=1500, ctx_hi=9000, block_size=8, q_blocks=(1, 2))
    assert set(np.diff(d["q_offsets"]).tolist()) == {8, 16}
    want_o, want_l = oracle.ragged(d["q"], d["k_nope"], d["k_rope"], d["v"], d["q_offsets"], d["kv_offsets"],
                                   d["anchors"], 8)
    got_o, got_l = _run_ragged(dfl, d, "bf16", max_q_len=16)
    assert not np.isnan(got_o).any() and not np.isnan(got_l).any()
    assert max_abs_err(got_o, want_o) <= TOL["bf16"]
    assert max_abs_err(got_l, want_l) <= TOL["bf16"]


@pytest.mark.parametrize("path", ["decode", "tc", "simt"])
def test_ragged_q_len_beyond_max_q_len_reported(dfl, path, monkeypatch):
    """A request longer than the declared max_q_len is recorded as
    DFLASH_ERR_INVALID and skipped (its rows stay unwritten) on every path; the
    other requests are still computed."""
    monkeypatch.delenv("DFLASH_FORCE_SIMT", raising=False)
    if path == "simt":
        monkeypatch.setenv("DFLASH_FORCE_SIMT", "1")
    bs, declared = (8, 16) if path == "decode" else (16, 32)
    nbr = np.array([1, 3, 1])  # request 1 has more rows than declared
    ctx = np.array([300, 1200, 700])
    qlens = nbr * bs
    qo = np.concatenate([[0], np.cumsum(qlens)]).astype(np.int32)
    ko = np.concatenate([[0], np.cumsum(ctx + qlens)]).astype(np.int32)
    rng = np.random.default_rng(5)
    an = np.concatenate([np.sort(rng.integers(0, ctx[r] + 1, size=nbr[r])) for r in range(3)]).astype(np.int32)
    d2 = dict(q=synth._normal(97, 0, (int(qo[-1]), 2, 192), "bf16"),
              k_nope=synth._normal(97, 1, (int(ko[-1]), 2, 128), "bf16"),
              k_rope=synth._normal(97, 2, (int(ko[-1]), 64), "bf16"),
              v=synth._normal(97, 3, (int(ko[-1]), 2, 128), "bf16"), total_q=int(qo[-1]))
    t = _dev(d2, "bf16")
    out = torch.full((d2["total_q"], 2, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    qo_t, ko_t, an_t = (torch.from_numpy(x).cuda() for x in (qo, ko, an))
    dfl.dflash_attn_ragged(t["q"], t["k_nope"], t["k_rope"], t["v"], qo_t, ko_t, an_t, bs, declared, out=out)
    assert dfl.dflash_last_device_error() == 1  # DFLASH_ERR_INVALID
    got = to_numpy_f64(out)
    assert np.isnan(got[qo[1]:qo[2]]).all()  # the long request is skipped
    want_o, _ = oracle.ragged(d2["q"], d2["k_nope"], d2["k_rope"], d2["v"], qo, ko, an, bs)
    for r in (0, 2):
        assert max_abs_err(got[qo[r]:qo[r + 1]], want_o[qo[r]:qo[r + 1]]) <= TOL["bf16"]


def test_ragged_split_equals_unsplit(dfl, monkeypatch):
    d = synth.make("decode_bf16", seed=84, R=5, H=2, ctx_lo=100, ctx_hi=6000)
    split_o, split_l = _run_ragged(dfl, d, "bf16")
    monkeypatch.setenv("DFLASH_NO_SPLIT", "1")  # one pass over each request's whole context
    full_o, full_l = _run_ragged(dfl, d, "bf16")
    assert max_abs_err(split_o, full_o) <= TOL["bf16"]
    assert max_abs_err(split_l, full_l) <= 1e-3


def test_ragged_equals_per_request_anchored(dfl):
    d = synth.make("decode_bf16", seed=78, R=4, H=2, ctx_lo=100, ctx_hi=900, nb=2, block_size=16)
    got_o, _ = _run_ragged(dfl, d, "bf16")
    qo, ko = d["q_offsets"], d["kv_offsets"]
    for r in range(4):
        sub = dict(d, B=1, Q=int(qo[r + 1] - qo[r]), S=int(ko[r + 1] - ko[r] - (qo[r + 1] - qo[r])),
                   q=d["q"][None, qo[r]:qo[r + 1]], k_nope=d["k_nope"][None, ko[r]:ko[r + 1]],
                   k_rope=d["k_rope"][None, ko[r]:ko[r + 1]], v=d["v"][None, ko[r]:ko[r + 1]],
                   anchors=d["anchors"][None, qo[r] // 16:qo[r + 1] // 16])
        o, _ = _run_batched(dfl, sub, "anchored", "bf16")
        assert max_abs_err(got_o[qo[r]:qo[r + 1]], o[0]) <= TOL["bf16"]


def test_ragged_bad_offsets_reported(dfl):
    d = synth.make("decode_bf16", seed=79, R=2, H=1, ctx_lo=10, ctx_hi=20, d_nope=8, d_rope=8, d_v=8)
    d["q_offsets"] = np.array([0, 8, 16], np.int32)  # q_len 8 < block_size 16
    _run_ragged_err = None
    t = _dev(d, "bf16")
    qo, ko, an = (torch.from_numpy(d[k]).cuda() for k in ("q_offsets", "kv_offsets", "anchors"))
    dfl.dflash_attn_ragged(t["q"], t["k_nope"], t["k_rope"], t["v"], qo, ko, an, 16, 16)
    assert dfl.dflash_last_device_error() == 1
    del _run_ragged_err


# ---------------------------------------------------------------------------
# full-size workloads, sampled rows
# ---------------------------------------------------------------------------
def _check_sampled(got_o, got_l_rows, d, rows, mode, mask=None):
    flat_o = got_o.reshape(-1, d["H"], d["d_v"])[rows]
    if mode == "ragged":
        want_o, want_l = oracle.ragged(d["q"], d["k_nope"], d["k_rope"], d["v"], d["q_offsets"], d["kv_offsets"],
                                       d["anchors"], d["block_size"], rows=rows)
    elif mode == "dense":
        want_o, want_l = oracle.dense(d["q"], d["k_nope"], d["k_rope"], d["v"], mask, rows=rows)
    else:
        want_o, want_l = oracle.anchored(d["q"], d["k_nope"], d["k_rope"], d["v"], d["anchors"], d["block_size"],
                                         rows=rows)
    e_o, e_l = max_abs_err(flat_o, want_o), max_abs_err(got_l_rows, want_l)
    return e_o, e_l


def _lse_rows_batched(got_l, d, rows):
    # got_l [B,H,Q] -> [n,H] for flat rows b*Q+i
    b, i = rows // d["Q"], rows % d["Q"]
    return got_l[b, :, i]


@pytest.mark.parametrize("name", ["prefill_bf16", "training_bf16", "long_bf16"])
def test_full_workload_anchored_sampled(dfl, name):
    d = synth.make(name)
    got_o, got_l = _run_batched(dfl, d, "anchored", "bf16")
    assert not np.isnan(got_o).any()
    rows = sample_rows(d["B"] * d["Q"], 96, seed=1, segment_len=d["Q"])
    e_o, e_l = _check_sampled(got_o, _lse_rows_batched(got_l, d, rows), d, rows, "anchored")
    assert e_o <= TOL["bf16"] and e_l <= TOL["bf16"], (e_o, e_l)


@pytest.mark.parametrize("name", ["training_bf16", "long_bf16"])
def test_full_workload_dense_sampled(dfl, name):
    d = synth.make(name)
    mask = _mask_for(d, "bf16")
    got_o, got_l = _run_batched(dfl, d, "dense", "bf16", mask)
    assert not np.isnan(got_o).any()
    rows = sample_rows(d["B"] * d["Q"], 64, seed=2, segment_len=d["Q"])
    e_o, e_l = _check_sampled(got_o, _lse_rows_batched(got_l, d, rows), d, rows, "dense", mask=mask)
    assert e_o <= TOL["bf16"] and e_l <= TOL["bf16"], (e_o, e_l)


def test_full_workload_ragged_decode_sampled(dfl):
    d = synth.make("decode_bf16")
    got_o, got_l = _run_ragged(dfl, d, "bf16")
    assert not np.isnan(got_o).any()
    rows = sample_rows(d["total_q"], 160, seed=3, segment_len=16)
    e_o, e_l = _check_sampled(got_o, got_l[:, rows].T, d, rows, "ragged")
    assert e_o <= TOL["bf16"] and e_l <= TOL["bf16"], (e_o, e_l)

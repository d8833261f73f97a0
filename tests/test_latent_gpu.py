"""GPU parity of the compressed-latent ragged entry point (dflash_attn_latent_ragged)
against the fp64 oracle (kv_b_proj expansion, then the ragged definition).

Both ways the library computes it are checked: the absorbed tensor-core path
(bf16, Kimi K3 MLA dims, kv_lora_rank 512, decode-shaped requests) and the
expanded path (any dims, fp32 or bf16).  Bars: 1e-5 (fp32) and 2e-2 (bf16)
max abs error on out and lse.
"""
import numpy as np
import pytest

import oracle
from dflash_block_draft_gb300 import synth
from tests.helpers import TOL, max_abs_err, sample_rows, to_numpy_f64, to_torch

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def dfl():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import dflash_block_draft_gb300 as m
    m.load_library()
    return m


def _run(dfl, d, dtype, max_q_len=None):
    t = {k: to_torch(d[k], dtype) for k in ("q", "c_kv", "k_rope", "w_kv_b")}
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    dv = d["w_kv_b"].shape[1] - d["d_nope"]
    out = torch.full((d["total_q"], d["H"], dv), float("nan"), dtype=tdt, device="cuda")
    lse = torch.full((d["H"], d["total_q"]), float("nan"), dtype=torch.float32, device="cuda")
    qo, ko, an = (torch.from_numpy(d[k]).cuda() for k in ("q_offsets", "kv_offsets", "anchors"))
    mq = max_q_len or int(np.diff(d["q_offsets"]).max())
    dfl.dflash_attn_latent_ragged(t["q"], t["c_kv"], t["k_rope"], t["w_kv_b"], qo, ko, an, d["block_size"], mq,
                                  out=out, lse=lse)
    assert dfl.dflash_last_device_error() == 0
    return to_numpy_f64(out), to_numpy_f64(lse)


def _want(d, requests=None):
    return oracle.latent_ragged(d["q"], d["c_kv"], d["k_rope"], d["w_kv_b"], d["q_offsets"], d["kv_offsets"],
                                d["anchors"], d["block_size"], requests=requests)


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
def test_expanded_path_general_dims_every_row(dfl, dtype):
    d = synth.make("decode_latent_bf16", seed=201, dtype=dtype, R=7, H=3, d_nope=16, d_rope=8, d_v=12, kv_rank=40,
                   ctx_lo=1, ctx_hi=500, block_size=4, q_blocks=(1, 3, 5))
    want_o, want_l = _want(d)
    got_o, got_l = _run(dfl, d, dtype)
    assert not np.isnan(got_o).any()
    assert max_abs_err(got_o, want_o) <= TOL[dtype]
    assert max_abs_err(got_l, want_l) <= TOL[dtype]


@pytest.mark.parametrize("bs,q_blocks,seed", [(16, (1,), 202), (8, (1, 2), 203), (4, (2, 4), 204)])
def test_absorbed_path_decode_shape_every_row(dfl, bs, q_blocks, seed):
    """Kimi K3 MLA dims, kv_lora_rank 512, at most 16 rows per request; contexts
    that cross split boundaries (at most 3072 keys per split); anchors anywhere in [0, S_r]."""
    d = synth.make("decode_latent_bf16", seed=seed, R=6, H=8, ctx_lo=200, ctx_hi=14000, block_size=bs,
                   q_blocks=q_blocks)
    rng = np.random.default_rng(seed)
    qo = d["q_offsets"]
    for r in range(d["R"]):
        nbr = int(qo[r + 1] - qo[r]) // bs
        S_r = int(d["kv_offsets"][r + 1] - d["kv_offsets"][r]) - nbr * bs
        d["anchors"][qo[r] // bs:qo[r + 1] // bs] = np.sort(rng.integers(0, S_r + 1, size=nbr))
    want_o, want_l = _want(d)
    got_o, got_l = _run(dfl, d, "bf16", max_q_len=16)
    assert not np.isnan(got_o).any() and not np.isnan(got_l).any()
    assert max_abs_err(got_o, want_o) <= TOL["bf16"]
    assert max_abs_err(got_l, want_l) <= TOL["bf16"]


def test_absorbed_equals_expanded(dfl, monkeypatch):
    d = synth.make("decode_latent_bf16", seed=205, R=5, H=4, ctx_lo=100, ctx_hi=7000)
    a_o, a_l = _run(dfl, d, "bf16", max_q_len=16)
    monkeypatch.setenv("DFLASH_LATENT_EXPAND", "1")  # expand k_nope / v, then the ragged kernels
    e_o, e_l = _run(dfl, d, "bf16", max_q_len=16)
    assert max_abs_err(a_o, e_o) <= TOL["bf16"]
    assert max_abs_err(a_l, e_l) <= TOL["bf16"]


def test_full_latent_decode_workload_sampled(dfl):
    """The full latent decode workload (64 requests, contexts log-uniform in
    [1024, 32768], H = 32) in the benchmark's launch configuration; the oracle
    evaluates every row of a short, a median and the longest request."""
    d = synth.make("decode_latent_bf16")
    got_o, got_l = _run(dfl, d, "bf16", max_q_len=16)
    assert not np.isnan(got_o).any()
    ctx = d["context_lens"]
    reqs = sorted({int(np.argmin(ctx)), int(np.argsort(ctx)[len(ctx) // 2]), int(np.argmax(ctx))})
    want_o, want_l = _want(d, requests=reqs)
    qo = d["q_offsets"]
    for r in reqs:
        sl = slice(int(qo[r]), int(qo[r + 1]))
        assert max_abs_err(got_o[sl], want_o[sl]) <= TOL["bf16"], r
        assert max_abs_err(got_l[:, sl], want_l[:, sl]) <= TOL["bf16"], r

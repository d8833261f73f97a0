"""Host-side measurement arithmetic of the benchmark (CPU only): the FLOP and
byte accounting the bench line reports, the whole-job value, and the rule that
recorded DRAM traffic is only reported for the kernel source it was captured on."""
import hashlib
import json
import os

import numpy as np
import pytest

import bench
import oracle
from dflash_block_draft_gb300 import metrics, synth


def test_flops_per_visible_pair():
    # forward: QK^T (2 d_qk) and PV (2 d_v); backward: S, dP, dV, dK, dQ
    assert metrics.flops_per_pair(128, 64, 128) == 2 * (192 + 128) == 640
    assert metrics.backward_flops_per_pair(128, 64, 128) == 2 * (3 * 192 + 2 * 128) == 1664


@pytest.mark.parametrize("S,nb,bs,B", [(37, 5, 3, 2), (64, 4, 4, 1), (0, 3, 5, 1), (200, 7, 16, 2)])
def test_visible_counts_equal_the_oracle_mask(S, nb, bs, B):
    rng = np.random.default_rng(S + nb)
    Q = nb * bs
    an = np.stack([np.sort(rng.choice(np.arange(0, S + 1), nb, replace=nb > S + 1)) for _ in range(B)])
    an = an.astype(np.int32)
    mask = oracle.build_mask(an, bs, S)
    want = (mask[:, 0] == 0).sum(axis=-1)
    np.testing.assert_array_equal(metrics.anchored_visible_counts(an, S, Q, bs), want)


def test_anchored_work_counts_pairs_and_bytes():
    d = synth.make("tiny_fp32")
    S, Q, H, bs = d["S"], d["Q"], d["H"], d["block_size"]
    w = metrics.anchored_work(d["anchors"], S, Q, H, bs, 16, 8, 16, esize=4)
    mask = oracle.build_mask(d["anchors"], bs, S)
    pairs = int((mask == 0).sum()) * H
    assert w["pairs"] == pairs and w["flops"] == pairs * 2 * (24 + 16)
    keys = int(min(d["anchors"].max(), S)) + Q  # keys some row sees: below the largest anchor, plus noise
    assert w["keys_read"] == keys
    expect = Q * H * 24 * 4 + keys * (H * 32 * 4 + 8 * 4) + Q * H * 16 * 4 + d["anchors"].size * 4
    assert w["bytes"] == expect


def test_job_value_is_all_ranks_units_over_slowest_time():
    assert bench.job_value(1e12, 1, 1000.0) == pytest.approx(1e12)
    assert bench.job_value(1e12, 4, 2000.0) == pytest.approx(2e12)


def _fake_root(tmp_path, source_text, entry):
    (tmp_path / "profiles").mkdir()
    (tmp_path / "k.cu").write_text(source_text)
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps({"w": entry}))
    return str(tmp_path)


def test_traffic_reported_only_for_the_captured_source(tmp_path, monkeypatch):
    src = "// kernel source\\n"
    md5 = hashlib.md5(src.encode()).hexdigest()
    root = _fake_root(tmp_path, src, {"source": "k.cu", "source_md5": md5, "bytes_per_launch": 12345})
    monkeypatch.setattr(bench, "ROOT", root)
    assert bench.load_traffic("w") == 12345
    (tmp_path / "k.cu").write_text(src + "// changed\\n")
    assert bench.load_traffic("w") is None
    assert bench.load_traffic("absent") is None


def test_traffic_of_a_smaller_capture_scales_with_algorithmic_bytes(tmp_path, monkeypatch):
    src = "x"
    md5 = hashlib.md5(src.encode()).hexdigest()
    root = _fake_root(tmp_path, src, {"source": "k.cu", "source_md5": md5, "bytes_per_launch": 1000,
                                      "algorithmic_bytes_of_capture": 500})
    monkeypatch.setattr(bench, "ROOT", root)
    assert bench.load_traffic("w", alg_bytes=2000) == 4000
    assert bench.load_traffic("w") is None  # a scaled figure needs this launch's algorithmic bytes


def test_committed_traffic_entries_name_existing_sources():
    with open(os.path.join(bench.ROOT, "profiles", "traffic.json")) as f:
        entries = json.load(f)
    for key, t in entries.items():
        assert os.path.exists(os.path.join(bench.ROOT, t["source"])), key
        assert len(t["source_md5"]) == 32 and t["bytes_per_launch"] > 0


def test_latent_work_counts():
    d = synth.make("decode_latent_bf16", R=3, H=4, ctx_lo=10, ctx_hi=300)
    w = metrics.latent_work(d["q_offsets"], d["kv_offsets"], d["anchors"], 4, 16, 128, 64, 128, 512)
    r = metrics.ragged_work(d["q_offsets"], d["kv_offsets"], d["anchors"], 4, 16, 128, 64, 128)
    assert w["pairs"] == r["pairs"] and w["keys_read"] == r["keys_read"]
    assert metrics.latent_flops_per_pair(512, 64) == 2 * 576 + 2 * 512
    tq = d["total_q"]
    assert w["flops"] == r["pairs"] * 2176 + tq * 4 * 2 * 512 * 256
    # per key 1152 bytes of latent + rope key instead of 4 heads x 512 + 128 expanded bytes
    expect = tq * 4 * 192 * 2 + r["keys_read"] * 576 * 2 + 4 * 256 * 512 * 2 + tq * 4 * 128 * 2 + (4 + 4 + tq // 16) * 4
    assert w["bytes"] == expect

"""Pins for the fp64 oracle (CPU only).

Each test ties the oracle to something other than itself: a hand-worked
visibility fixture, an independent numpy brute force, torch's fp64 SDPA (the
prior-art formulation of the attention on the DFlash Kimi K3 draft page,
KimiK3DFlashAttention.forward), closed forms, and invariants.
"""
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import brute
from dflash_block_draft_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
TOL = 1e-12


def _tiny(dtype="fp32", seed=7, B=2, H=3, S=37, nb=5, bs=3, dn=6, dr=4, dv=5, lo=0):
    rng = np.random.default_rng(seed)
    Q = nb * bs
    K = S + Q
    anchors = np.stack([np.sort(rng.choice(np.arange(lo, S + 1), nb, replace=False)) for _ in range(B)])

    def n(*shape):
        a = rng.standard_normal(shape).astype(np.float32)
        return synth.f32_to_bf16_bits(a) if dtype == "bf16" else (a.astype(np.float64) if dtype == "fp64" else a)

    return dict(q=n(B, Q, H, dn + dr), k_nope=n(B, K, H, dn), k_rope=n(B, K, dr), v=n(B, K, H, dv),
                anchors=anchors.astype(np.int32), bs=bs, S=S, Q=Q, B=B, H=H, dn=dn, dr=dr, dv=dv)


def _read_golden_visibility(name):
    rows, meta = [], {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            tok = line.split()
            if tok[0] in ("S", "block_size"):
                meta[tok[0]] = int(tok[1])
            elif tok[0] == "anchors":
                meta["anchors"] = [int(t) for t in tok[1:]]
            else:
                rows.append([int(t) for t in tok])
    return meta, np.array(rows, dtype=bool)


# --------------------------------------------------------------------------
# visibility rule
# --------------------------------------------------------------------------
def test_mask_matches_hand_worked_fixture():
    meta, vis = _read_golden_visibility("anchored_visibility_S5_nb3_bs2.txt")
    an = np.array([meta["anchors"]], np.int32)
    mask = oracle.build_mask(an, meta["block_size"], meta["S"])
    assert mask.shape == (1, 1, 6, 11)  # [batch, 1, blocks*block_size, sequence+blocks*block_size]
    np.testing.assert_array_equal(mask[0, 0] == 0, vis)
    np.testing.assert_array_equal(np.isneginf(mask[0, 0]), ~vis)


def test_anchored_output_uses_exactly_the_fixture_keys():
    # With v = one-hot of the key index, out[i] is the softmax weight row, so its
    # support must be exactly the fixture's visible set.
    meta, vis = _read_golden_visibility("anchored_visibility_S5_nb3_bs2.txt")
    S, bs = meta["S"], meta["block_size"]
    Q, K, H = 6, 11, 1
    rng = np.random.default_rng(3)
    q = rng.standard_normal((1, Q, H, 3))
    kn = rng.standard_normal((1, K, H, 2))
    kr = rng.standard_normal((1, K, 1))
    v = np.eye(K).reshape(1, K, H, K)
    out, _ = oracle.anchored(q, kn, kr, v, np.array([meta["anchors"]], np.int32), bs)
    np.testing.assert_array_equal(out[0, :, 0, :] > 0, vis)
    np.testing.assert_allclose(out[0, :, 0, :].sum(-1), 1.0, atol=1e-15)


# --------------------------------------------------------------------------
# brute force and library cross-checks
# --------------------------------------------------------------------------
@pytest.mark.parametrize("dtype", ["fp32", "bf16", "fp64"])
def test_dense_and_anchored_match_brute_force(dtype):
    t = _tiny(dtype)
    mask = oracle.build_mask(t["anchors"], t["bs"], t["S"])
    scale = oracle.default_scale(t["dn"], t["dr"])
    ob, lb = brute.dense(t["q"], t["k_nope"], t["k_rope"], t["v"], mask, scale)
    od, ld = oracle.dense(t["q"], t["k_nope"], t["k_rope"], t["v"], mask)
    oa, la = oracle.anchored(t["q"], t["k_nope"], t["k_rope"], t["v"], t["anchors"], t["bs"])
    for o, l in ((od, ld), (oa, la)):
        np.testing.assert_allclose(o, ob, atol=TOL, rtol=0)
        np.testing.assert_allclose(l, lb, atol=TOL, rtol=0)


def test_random_dense_mask_matches_brute_force():
    # A general additive mask: finite values of both signs, -inf holes, and one fully masked row.
    t = _tiny("fp32", seed=11)
    rng = np.random.default_rng(12)
    mask = rng.normal(0, 3, size=(t["B"], 1, t["Q"], t["S"] + t["Q"])).astype(np.float32)
    mask[rng.random(mask.shape) < 0.4] = -np.inf
    mask[1, 0, 4, :] = -np.inf
    scale = 0.37
    ob, lb = brute.dense(t["q"], t["k_nope"], t["k_rope"], t["v"], mask, scale)
    od, ld = oracle.dense(t["q"], t["k_nope"], t["k_rope"], t["v"], mask, scale=scale)
    np.testing.assert_allclose(od, ob, atol=TOL, rtol=0)
    np.testing.assert_allclose(ld, lb, atol=TOL, rtol=0)
    assert np.all(od[1, 4] == 0.0) and np.all(np.isneginf(ld[1, :, 4]))


def test_dense_matches_torch_sdpa_fp64():
    """The pages route this attention through SDPA with the dense additive mask;
    torch's fp64 CPU SDPA with keys cat(k_nope[h], k_rope) and its default scale
    1/sqrt(qk_nope+qk_rope) must agree."""
    t = _tiny("fp64", seed=5, B=2, H=4, S=50, nb=6, bs=4, dn=12, dr=6, dv=10, lo=1)
    mask = oracle.build_mask(t["anchors"], t["bs"], t["S"]).astype(np.float64)
    B, Q, H = t["B"], t["Q"], t["H"]
    K = t["S"] + Q
    q = torch.from_numpy(t["q"]).permute(0, 2, 1, 3)  # [B,H,Q,E]
    kn = torch.from_numpy(t["k_nope"]).permute(0, 2, 1, 3)  # [B,H,K,dn]
    kr = torch.from_numpy(t["k_rope"])[:, None].expand(B, H, K, t["dr"])
    k = torch.cat([kn, kr], dim=-1)
    v = torch.from_numpy(t["v"]).permute(0, 2, 1, 3)
    ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, attn_mask=torch.from_numpy(mask))
    ref = ref.permute(0, 2, 1, 3).numpy()
    od, _ = oracle.dense(t["q"], t["k_nope"], t["k_rope"], t["v"], mask)
    np.testing.assert_allclose(od, ref, atol=TOL, rtol=0)


# --------------------------------------------------------------------------
# closed forms
# --------------------------------------------------------------------------
def test_single_visible_key_returns_that_value_row_exactly():
    t = _tiny("fp32", seed=2)
    B, Q, K = t["B"], t["Q"], t["S"] + t["Q"]
    mask = np.full((B, 1, Q, K), -np.inf, np.float32)
    rng = np.random.default_rng(1)
    pick = rng.integers(0, K, size=(B, Q))
    for b in range(B):
        for i in range(Q):
            mask[b, 0, i, pick[b, i]] = 0.0
    out, lse = oracle.dense(t["q"], t["k_nope"], t["k_rope"], t["v"], mask)
    scale = oracle.default_scale(t["dn"], t["dr"])
    for b in range(B):
        for i in range(Q):
            k = pick[b, i]
            np.testing.assert_array_equal(out[b, i], t["v"][b, k].astype(np.float64))
            for h in range(t["H"]):
                s = scale * (t["q"][b, i, h, :t["dn"]].astype(np.float64) @ t["k_nope"][b, k, h].astype(np.float64)
                             + t["q"][b, i, h, t["dn"]:].astype(np.float64) @ t["k_rope"][b, k].astype(np.float64))
                assert abs(lse[b, h, i] - s) < 1e-13


def test_zero_query_gives_mean_of_visible_values():
    t = _tiny("fp32", seed=4)
    t["q"][:] = 0
    out, lse = oracle.anchored(t["q"], t["k_nope"], t["k_rope"], t["v"], t["anchors"], t["bs"])
    S, bs, Q = t["S"], t["bs"], t["Q"]
    for b in range(t["B"]):
        for i in range(Q):
            a = t["anchors"][b, i // bs]
            blk = i // bs
            keys = list(range(min(a, S))) + [S + blk * bs + u for u in range(bs)]
            mean = t["v"][b, keys].astype(np.float64).mean(axis=0)
            np.testing.assert_allclose(out[b, i], mean, atol=1e-14, rtol=0)
            np.testing.assert_allclose(lse[b, :, i], np.log(len(keys)), atol=1e-14, rtol=0)


def test_two_visible_keys_sigmoid_closed_form():
    rng = np.random.default_rng(9)
    H, dn, dr, dv = 2, 5, 3, 4
    q = rng.standard_normal((1, 1, H, dn + dr))
    kn = rng.standard_normal((1, 3, H, dn))
    kr = rng.standard_normal((1, 3, dr))
    v = rng.standard_normal((1, 3, H, dv))
    mask = np.array([[[[0.0, -np.inf, 0.5]]]])  # keys 0 and 2 visible, key 2 biased by +0.5
    out, lse = oracle.dense(q, kn, kr, v, mask, scale=0.8)
    for h in range(H):
        s0 = 0.8 * (q[0, 0, h, :dn] @ kn[0, 0, h] + q[0, 0, h, dn:] @ kr[0, 0])
        s2 = 0.8 * (q[0, 0, h, :dn] @ kn[0, 2, h] + q[0, 0, h, dn:] @ kr[0, 2]) + 0.5
        sig = 1.0 / (1.0 + np.exp(s2 - s0))
        np.testing.assert_allclose(out[0, 0, h], sig * v[0, 0, h] + (1 - sig) * v[0, 2, h], atol=1e-14)
        np.testing.assert_allclose(lse[0, h, 0], np.logaddexp(s0, s2), atol=1e-14)


# --------------------------------------------------------------------------
# invariants
# --------------------------------------------------------------------------
def test_permuting_commonly_visible_context_keys_leaves_output_unchanged():
    t = _tiny("fp64", seed=21, lo=10)
    base, lb = oracle.anchored(t["q"], t["k_nope"], t["k_rope"], t["v"], t["anchors"], t["bs"])
    amin = int(t["anchors"].min())
    perm = np.random.default_rng(0).permutation(amin)
    kn, kr, v = t["k_nope"].copy(), t["k_rope"].copy(), t["v"].copy()
    kn[:, :amin], kr[:, :amin], v[:, :amin] = kn[:, perm], kr[:, perm], v[:, perm]
    out, lo = oracle.anchored(t["q"], kn, kr, v, t["anchors"], t["bs"])
    np.testing.assert_allclose(out, base, atol=TOL, rtol=0)
    np.testing.assert_allclose(lo, lb, atol=TOL, rtol=0)


def test_permuting_heads_permutes_output():
    t = _tiny("fp64", seed=22)
    base, _ = oracle.anchored(t["q"], t["k_nope"], t["k_rope"], t["v"], t["anchors"], t["bs"])
    p = np.array([2, 0, 1])
    out, _ = oracle.anchored(t["q"][:, :, p], t["k_nope"][:, :, p], t["k_rope"], t["v"][:, :, p],
                             t["anchors"], t["bs"])
    np.testing.assert_allclose(out, base[:, :, p], atol=TOL, rtol=0)


def test_mask_row_shift_and_value_affine():
    t = _tiny("fp64", seed=23)
    mask = oracle.build_mask(t["anchors"], t["bs"], t["S"]).astype(np.float64)
    base, lb = oracle.dense(t["q"], t["k_nope"], t["k_rope"], t["v"], mask)
    shift = np.random.default_rng(1).normal(size=(t["B"], 1, t["Q"], 1))  # per-row constant
    out, lo = oracle.dense(t["q"], t["k_nope"], t["k_rope"], t["v"], mask + shift)
    np.testing.assert_allclose(out, base, atol=TOL, rtol=0)
    d = shift[:, 0, :, 0]  # [B,Q]
    np.testing.assert_allclose(lo, lb + d[:, None, :], atol=TOL, rtol=0)
    out2, _ = oracle.dense(t["q"], t["k_nope"], t["k_rope"], 2.5 * t["v"] - 0.75, mask)
    np.testing.assert_allclose(out2, 2.5 * base - 0.75, atol=1e-12, rtol=0)


def test_rope_key_is_head_shared_and_irrelevant_when_q_rope_is_zero():
    t = _tiny("fp64", seed=24)
    q = t["q"].copy()
    q[..., t["dn"]:] = 0
    a, _ = oracle.anchored(q, t["k_nope"], t["k_rope"], t["v"], t["anchors"], t["bs"])
    b, _ = oracle.anchored(q, t["k_nope"], np.random.default_rng(5).normal(size=t["k_rope"].shape),
                           t["v"], t["anchors"], t["bs"])
    np.testing.assert_allclose(a, b, atol=TOL, rtol=0)
    # head-shared rope key == a per-head rope key replicated over heads (brute force on the concatenated key)
    full, _ = oracle.anchored(t["q"], t["k_nope"], t["k_rope"], t["v"], t["anchors"], t["bs"])
    kcat = np.concatenate([t["k_nope"], np.repeat(t["k_rope"][:, :, None], t["H"], axis=2)], axis=-1)
    mask = oracle.build_mask(t["anchors"], t["bs"], t["S"])
    dn = t["dn"] + t["dr"]
    ref, _ = brute.dense(t["q"], kcat, np.zeros(t["k_rope"].shape[:2] + (0,)), t["v"], mask, dn ** -0.5)
    np.testing.assert_allclose(full, ref, atol=TOL, rtol=0)


# --------------------------------------------------------------------------
# entry-point equivalences
# --------------------------------------------------------------------------
def test_dense_from_anchors_with_padding_equals_anchored():
    # Long-context recipe at small scale: trailing context columns are padding (-inf in
    # the dense mask) and anchors never reach past the valid context.
    S, pad, bs, nb = 40, 2, 2, 6
    t = _tiny("fp32", seed=31, S=S, nb=nb, bs=bs)
    rng = np.random.default_rng(3)
    an = np.stack([np.sort(rng.choice(np.arange(1, S - pad + 1), nb, replace=False)) for _ in range(t["B"])])
    an = an.astype(np.int32)
    mask = oracle.build_mask(an, bs, S)
    mask[:, :, :, S - pad:S] = -np.inf
    od, ld = oracle.dense(t["q"], t["k_nope"], t["k_rope"], t["v"], mask)
    oa, la = oracle.anchored(t["q"], t["k_nope"], t["k_rope"], t["v"], an, bs)
    np.testing.assert_allclose(od, oa, atol=TOL, rtol=0)
    np.testing.assert_allclose(ld, la, atol=TOL, rtol=0)


@pytest.mark.parametrize("q_blocks", [(), (1, 2, 3)], ids=["uniform", "mixed"])
def test_ragged_equals_per_request_loop(q_blocks):
    """Ragged == a B=1 anchored call per request on that request's slices.  With
    mixed draft lengths a request's first global block q_offsets[r]/bs differs
    from r*nb, so a mistake in how anchors are indexed across requests fails."""
    R = 9 if q_blocks else 5
    d = synth.make("decode_bf16", R=R, H=2, d_nope=8, d_rope=4, d_v=6, ctx_lo=3, ctx_hi=40, block_size=4,
                   nb=2, q_blocks=q_blocks)
    out, lse = oracle.ragged(d["q"], d["k_nope"], d["k_rope"], d["v"], d["q_offsets"], d["kv_offsets"],
                             d["anchors"], d["block_size"])
    qo, ko = d["q_offsets"], d["kv_offsets"]
    qlens = np.diff(qo)
    if q_blocks:
        assert len(set(qlens.tolist())) > 1 and np.any(qo[:-1] != np.arange(R) * qlens[0])
    else:
        assert np.all(qlens == 8)
    for r in range(R):
        sl = slice(ko[r], ko[r + 1])
        an = d["anchors"][qo[r] // 4:qo[r + 1] // 4][None]
        o, l = oracle.anchored(d["q"][None, qo[r]:qo[r + 1]], d["k_nope"][None, sl], d["k_rope"][None, sl],
                               d["v"][None, sl], an, 4)
        np.testing.assert_allclose(out[qo[r]:qo[r + 1]], o[0], atol=TOL, rtol=0)
        np.testing.assert_allclose(lse[:, qo[r]:qo[r + 1]], l[0], atol=TOL, rtol=0)


def test_ragged_mixed_lengths_against_brute_force():
    """Mixed draft lengths against the numpy brute force, one request at a time:
    its own keys and a mask built by hand from its anchors (context p < a_j, own
    block only)."""
    d = synth.make("decode_bf16", seed=7, R=6, H=2, d_nope=8, d_rope=4, d_v=6, ctx_lo=2, ctx_hi=30,
                   block_size=3, nb=1, q_blocks=(1, 2, 4), dtype="fp32")
    out, lse = oracle.ragged(d["q"], d["k_nope"], d["k_rope"], d["v"], d["q_offsets"], d["kv_offsets"],
                             d["anchors"], 3)
    qo, ko = d["q_offsets"], d["kv_offsets"]
    for r in range(6):
        ql, kl = int(qo[r + 1] - qo[r]), int(ko[r + 1] - ko[r])
        S_r = kl - ql
        mask = np.full((1, 1, ql, kl), -np.inf)
        for i in range(ql):
            j = i // 3
            a = int(d["anchors"][qo[r] // 3 + j])
            mask[0, 0, i, :a] = 0.0
            mask[0, 0, i, S_r + 3 * j:S_r + 3 * j + 3] = 0.0
        sl = slice(ko[r], ko[r + 1])
        o, l = brute.dense(d["q"][None, qo[r]:qo[r + 1]], d["k_nope"][None, sl], d["k_rope"][None, sl],
                           d["v"][None, sl], mask, oracle.default_scale(8, 4))
        np.testing.assert_allclose(out[qo[r]:qo[r + 1]], o[0], atol=TOL, rtol=0)
        np.testing.assert_allclose(lse[:, qo[r]:qo[r + 1]], l[0], atol=TOL, rtol=0)


@pytest.mark.parametrize("split", [1, 7, 16, 1000])
def test_split_context_merge_equals_unsplit(split):
    t = _tiny("fp32", seed=41)
    oa, la = oracle.anchored(t["q"], t["k_nope"], t["k_rope"], t["v"], t["anchors"], t["bs"])
    os_, ls = oracle.anchored_split(t["q"], t["k_nope"], t["k_rope"], t["v"], t["anchors"], t["bs"], split)
    np.testing.assert_allclose(os_, oa, atol=TOL, rtol=0)
    np.testing.assert_allclose(ls, la, atol=TOL, rtol=0)


def test_rows_subset_matches_full_evaluation():
    t = _tiny("bf16", seed=51)
    full, lf = oracle.anchored(t["q"], t["k_nope"], t["k_rope"], t["v"], t["anchors"], t["bs"])
    rows = np.array([0, 3, t["Q"] + 2, 2 * t["Q"] - 1])
    sub, ls = oracle.anchored(t["q"], t["k_nope"], t["k_rope"], t["v"], t["anchors"], t["bs"], rows=rows)
    flat = full.reshape(-1, t["H"], t["dv"])
    np.testing.assert_array_equal(sub, flat[rows])
    np.testing.assert_array_equal(ls, lf.transpose(0, 2, 1).reshape(-1, t["H"])[rows])


def test_anchor_zero_and_full_context_edges():
    t = _tiny("fp64", seed=61, S=9, nb=3, bs=2)
    an = np.array([[0, 9, 4], [9, 0, 0]], np.int32)
    mask = oracle.build_mask(an, 2, 9)
    ob, lb = brute.dense(t["q"], t["k_nope"], t["k_rope"], t["v"], mask, oracle.default_scale(t["dn"], t["dr"]))
    oa, la = oracle.anchored(t["q"], t["k_nope"], t["k_rope"], t["v"], an, 2)
    np.testing.assert_allclose(oa, ob, atol=TOL, rtol=0)
    np.testing.assert_allclose(la, lb, atol=TOL, rtol=0)


# --------------------------------------------------------------------------
# brute-force tile scan
# --------------------------------------------------------------------------
def test_tile_scan_from_rule_equals_scan_from_mask():
    rng = np.random.default_rng(71)
    for S, nb, bs, tm, tn in ((37, 5, 3, 4, 8), (64, 4, 4, 8, 16), (100, 12, 8, 32, 16)):
        an = np.stack([np.sort(rng.choice(np.arange(0, S + 1), nb, replace=False)) for _ in range(2)])
        an = an.astype(np.int32)
        mask = oracle.build_mask(an, bs, S)
        a = oracle.tile_classes(2, S, nb * bs, tm, tn, anchors=an, block_size=bs)
        b = oracle.tile_classes(2, S, nb * bs, tm, tn, mask=mask)
        np.testing.assert_array_equal(a, b)
        assert set(np.unique(a)) <= {0, 1, 2}


def test_tile_scan_small_hand_case():
    # Fixture case with 2x4 tiles: rows {0,1} see ctx {0,1} + noise {5,6}, etc.
    meta, vis = _read_golden_visibility("anchored_visibility_S5_nb3_bs2.txt")
    cls = oracle.tile_classes(1, 5, 6, 2, 4, anchors=np.array([meta["anchors"]], np.int32), block_size=2)
    expect = np.zeros((3, 3), np.uint8)
    for tq in range(3):
        for tk in range(3):
            blk = vis[2 * tq:2 * tq + 2, 4 * tk:min(4 * tk + 4, 11)]
            expect[tq, tk] = 0 if not blk.any() else (2 if blk.all() else 1)
    np.testing.assert_array_equal(cls[0], expect)
    assert cls[0, 0, 0] == 1 and cls[0, 2, 0] == 2 and cls[0, 1, 0] == 0


def test_fully_masked_dense_rows_give_zero_and_neg_inf():
    t = _tiny("fp32", seed=81)
    mask = np.full((t["B"], 1, t["Q"], t["S"] + t["Q"]), -np.inf, np.float32)
    out, lse = oracle.dense(t["q"], t["k_nope"], t["k_rope"], t["v"], mask)
    assert np.all(out == 0) and np.all(np.isneginf(lse))

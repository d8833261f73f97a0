"""Pins for the fp64 backward oracle (CPU only).

The backward oracle differentiates the forward definition by hand.  It is tied
to things other than itself:
  - central finite differences of the (separately pinned) forward oracle, for
    every input element of small anchored and dense cases;
  - torch's fp64 autograd through scaled_dot_product_attention, the library
    routine the DFlash Kimi K3 draft page routes the attention through
    (KimiK3DFlashAttention.forward), with the head-shared k_rope broadcast by
    expand so that autograd sums its gradient over heads;
  - closed forms (one visible key) and invariants that hold for any input.
"""
import numpy as np
import pytest
import torch

import oracle

TOL = 1e-12


def _case(seed=11, B=1, H=2, S=9, nb=3, bs=2, dn=4, dr=3, dv=3, lo=0):
    rng = np.random.default_rng(seed)
    Q = nb * bs
    K = S + Q
    anchors = np.stack([np.sort(rng.choice(np.arange(lo, S + 1), nb, replace=False)) for _ in range(B)])
    n = lambda *shape: rng.standard_normal(shape)
    return dict(q=n(B, Q, H, dn + dr), k_nope=n(B, K, H, dn), k_rope=n(B, K, dr), v=n(B, K, H, dv),
                dout=n(B, Q, H, dv), anchors=anchors.astype(np.int32), bs=bs, S=S, Q=Q, B=B, H=H)


def _loss(c, mask=None, scale=None):
    if mask is None:
        out, _ = oracle.anchored(c["q"], c["k_nope"], c["k_rope"], c["v"], c["anchors"], c["bs"], scale=scale)
    else:
        out, _ = oracle.dense(c["q"], c["k_nope"], c["k_rope"], c["v"], mask, scale=scale)
    return float(np.sum(c["dout"] * out))


def _finite_diff(c, mask=None, scale=None, eps=1e-6):
    grads = {}
    for name in ("q", "k_nope", "k_rope", "v"):
        x = c[name]
        g = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            old = x[idx]
            x[idx] = old + eps
            lp = _loss(c, mask, scale)
            x[idx] = old - eps
            lm = _loss(c, mask, scale)
            x[idx] = old
            g[idx] = (lp - lm) / (2 * eps)
        grads[name] = g
    return grads


def _bwd(c, mask=None, scale=None, pairs=None):
    if mask is None:
        return oracle.backward(c["q"], c["k_nope"], c["k_rope"], c["v"], c["dout"], anchors=c["anchors"],
                               block_size=c["bs"], scale=scale, pairs=pairs)
    return oracle.backward(c["q"], c["k_nope"], c["k_rope"], c["v"], c["dout"], mask=mask, scale=scale,
                           pairs=pairs)


def _check_fd(c, mask=None, scale=None):
    fd = _finite_diff(c, mask, scale)
    dq, dkn, dkr, dv = _bwd(c, mask, scale)
    for name, got in (("q", dq), ("k_nope", dkn), ("k_rope", dkr), ("v", dv)):
        np.testing.assert_allclose(got, fd[name], atol=2e-8, rtol=1e-6, err_msg=name)


def test_backward_matches_finite_differences_anchored():
    # anchors include 0 (a block that sees only its own noise keys) and S
    c = _case(seed=11)
    c["anchors"][0, 0] = 0
    c["anchors"][0, -1] = c["S"]
    _check_fd(c)


def test_backward_matches_finite_differences_anchored_two_rows_custom_scale():
    c = _case(seed=12, B=2, H=1, S=7, nb=2, bs=3, dn=3, dr=2, dv=2)
    _check_fd(c, scale=0.37)


def test_backward_matches_finite_differences_dense_with_finite_mask_values():
    c = _case(seed=13)
    rng = np.random.default_rng(99)
    B, Q, K = c["B"], c["Q"], c["S"] + c["Q"]
    mask = rng.standard_normal((B, 1, Q, K)) * 0.5
    mask[rng.random((B, 1, Q, K)) < 0.4] = -np.inf
    mask[0, 0, 1, :] = -np.inf  # a row with no visible key contributes nothing
    _check_fd(c, mask=mask)
    dq = _bwd(c, mask=mask)[0]
    assert np.all(dq[0, 1] == 0.0)


def _torch_sdpa_grads(c, mask):
    q = torch.tensor(c["q"], requires_grad=True)
    kn = torch.tensor(c["k_nope"], requires_grad=True)
    kr = torch.tensor(c["k_rope"], requires_grad=True)
    v = torch.tensor(c["v"], requires_grad=True)
    H = q.shape[2]
    k = torch.cat([kn, kr[:, :, None, :].expand(-1, -1, H, -1)], dim=-1)
    out = torch.nn.functional.scaled_dot_product_attention(
        q.transpose(1, 2), k.transpose(1, 2), v.transpose(1, 2), attn_mask=torch.tensor(mask))
    loss = (out.transpose(1, 2) * torch.tensor(c["dout"])).sum()
    loss.backward()
    return q.grad.numpy(), kn.grad.numpy(), kr.grad.numpy(), v.grad.numpy()


def test_backward_matches_torch_sdpa_autograd_fp64():
    c = _case(seed=21, B=2, H=3, S=40, nb=4, bs=4, dn=8, dr=4, dv=6, lo=1)
    mask = oracle.build_mask(c["anchors"], c["bs"], c["S"]).astype(np.float64)
    ref = _torch_sdpa_grads(c, mask)
    got = _bwd(c)
    for name, g, r in zip(("dq", "dk_nope", "dk_rope", "dv"), got, ref):
        np.testing.assert_allclose(g, r, atol=1e-11, rtol=1e-10, err_msg=name)
    # the dense form with the same mask gives the same gradients
    got_d = _bwd(c, mask=mask)
    for g, r in zip(got_d, got):
        np.testing.assert_allclose(g, r, atol=TOL)


def test_single_visible_key_closed_form():
    # A row that sees one key has P = 1, so dS = 0: no gradient reaches q or k,
    # and that key's v receives exactly the row's dout.
    c = _case(seed=31, B=1, H=2, S=5, nb=2, bs=2)
    B, Q, K = 1, c["Q"], c["S"] + c["Q"]
    mask = np.full((B, 1, Q, K), -np.inf)
    for i in range(Q):
        mask[0, 0, i, i] = 0.0  # row i sees key i only
    dq, dkn, dkr, dv = _bwd(c, mask=mask)
    assert np.all(dq == 0.0) and np.all(dkn == 0.0) and np.all(dkr == 0.0)
    np.testing.assert_array_equal(dv[0, :Q], c["dout"][0])
    assert np.all(dv[0, Q:] == 0.0)


@pytest.mark.parametrize("seed", [41, 42])
def test_gradient_sums_over_keys(seed):
    # sum_k dS_k = 0 for every row, so the key gradients sum to zero over the
    # key axis; sum_k P_k = 1, so the v gradients sum to the rows' douts.
    c = _case(seed=seed, B=2, H=3, S=30, nb=5, bs=3, dn=5, dr=3, dv=4)
    dq, dkn, dkr, dv = _bwd(c)
    np.testing.assert_allclose(dkn.sum(axis=1), 0.0, atol=1e-12)
    np.testing.assert_allclose(dkr.sum(axis=1), 0.0, atol=1e-12)
    np.testing.assert_allclose(dv.sum(axis=1), c["dout"].sum(axis=1), atol=1e-12)


def test_rope_gradient_is_the_sum_of_per_head_gradients():
    # Evaluating head by head (pairs) and summing dk_rope reproduces the full
    # call; the per-head outputs of the subset equal the full call's.
    c = _case(seed=51, B=2, H=3, S=12, nb=3, bs=2)
    full = _bwd(c)
    acc = np.zeros_like(full[2])
    for p in range(c["B"] * c["H"]):
        b, h = divmod(p, c["H"])
        dq, dkn, dkr, dv = _bwd(c, pairs=[p])
        np.testing.assert_array_equal(dq[b, :, h], full[0][b, :, h])
        np.testing.assert_array_equal(dkn[b, :, h], full[1][b, :, h])
        np.testing.assert_array_equal(dv[b, :, h], full[3][b, :, h])
        acc += dkr
    np.testing.assert_allclose(acc, full[2], atol=1e-13)


def test_per_head_rope_replicated_equals_shared():
    # Replacing the shared k_rope by per-head copies (folded into k_nope) gives
    # per-head rope gradients whose head sum is the shared gradient.
    c = _case(seed=61, B=1, H=3, S=10, nb=2, bs=3, dn=4, dr=2, dv=3)
    H, dn, dr = c["H"], 4, 2
    kn2 = np.concatenate([c["k_nope"], np.repeat(c["k_rope"][:, :, None, :], H, axis=2)], axis=-1)
    kr2 = np.zeros(c["k_rope"].shape[:2] + (0,))
    scale = (dn + dr) ** -0.5
    dq, dkn, dkr, dv = _bwd(c)
    dq2, dkn2, _, dv2 = oracle.backward(c["q"], kn2, kr2, c["v"], c["dout"], anchors=c["anchors"],
                                        block_size=c["bs"], scale=scale)
    np.testing.assert_allclose(dq2, dq, atol=TOL)
    np.testing.assert_allclose(dkn2[..., :dn], dkn, atol=TOL)
    np.testing.assert_allclose(dkn2[..., dn:].sum(axis=2), dkr, atol=TOL)
    np.testing.assert_allclose(dv2, dv, atol=TOL)


def test_bf16_inputs_widen_exactly():
    c = _case(seed=71, B=1, H=2, S=8, nb=2, bs=2)
    from dflash_block_draft_gb300 import synth
    bits = {k: synth.f32_to_bf16_bits(c[k].astype(np.float32)) for k in ("q", "k_nope", "k_rope", "v", "dout")}
    wide = {k: synth.bf16_bits_to_f32(bits[k]).astype(np.float64) for k in bits}
    g16 = oracle.backward(bits["q"], bits["k_nope"], bits["k_rope"], bits["v"], bits["dout"],
                          anchors=c["anchors"], block_size=c["bs"])
    g64 = oracle.backward(wide["q"], wide["k_nope"], wide["k_rope"], wide["v"], wide["dout"],
                          anchors=c["anchors"], block_size=c["bs"])
    for a, b in zip(g16, g64):
        np.testing.assert_array_equal(a, b)

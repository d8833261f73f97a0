"""Pins of the compressed-latent (MLA kv_b_proj) oracle, CPU only.

The oracle expands each token's KV latent c_kv to per-head keys and values
with the kv_b_proj weight w_kv_b [H, d_nope + d_v, rank] (key rows first) and
then evaluates the ragged attention definition.  It is pinned here by:
  - elementary weights (a single 1 at [h, e, c]) whose expansion is known
    element by element, with rank != d_nope so that a transposed weight fails;
  - identity weights, which reduce the latent form to the plain ragged
    attention with k_nope = v = c_kv in every head;
  - the absorbed form (scores from W_UK^T q against c_kv, output W_UV applied
    after the softmax-weighted latent sum), a different evaluation order of
    the same algebra, written out here in numpy;
  - torch's fp64 scaled_dot_product_attention on keys expanded with einsum.
"""
import numpy as np
import pytest
import torch

import oracle
from dflash_block_draft_gb300 import synth

TOL = 1e-11


def _case(seed=3, R=4, H=3, dn=6, dr=4, dv=5, rank=9, bs=4, q_blocks=(1, 2)):
    d = synth.make("decode_latent_bf16", seed=seed, R=R, H=H, d_nope=dn, d_rope=dr, d_v=dv, kv_rank=rank,
                   ctx_lo=3, ctx_hi=30, block_size=bs, q_blocks=q_blocks, dtype="fp32")
    assert d["c_kv"].shape == (d["total_kv"], rank) and d["w_kv_b"].shape == (H, dn + dv, rank)
    return d


def test_expansion_of_elementary_weights():
    rng = np.random.default_rng(0)
    H, dn, dv, rank, T = 2, 3, 4, 7, 5
    c = rng.normal(size=(T, rank))
    for h, e, col in [(0, 1, 5), (1, 0, 2), (1, dn + 2, 6), (0, dn, 0)]:
        w = np.zeros((H, dn + dv, rank))
        w[h, e, col] = 1.0
        kn, v = oracle.latent_expand(c, w, dn)
        want_k = np.zeros((T, H, dn))
        want_v = np.zeros((T, H, dv))
        if e < dn:
            want_k[:, h, e] = c[:, col]
        else:
            want_v[:, h, e - dn] = c[:, col]
        np.testing.assert_array_equal(kn, want_k)
        np.testing.assert_array_equal(v, want_v)


def test_expansion_token_range():
    d = _case()
    kn, v = oracle.latent_expand(d["c_kv"], d["w_kv_b"], 6)
    kn2, v2 = oracle.latent_expand(d["c_kv"], d["w_kv_b"], 6, t0=3, t1=11)
    np.testing.assert_array_equal(kn2, kn[3:11])
    np.testing.assert_array_equal(v2, v[3:11])


def test_identity_weights_reduce_to_plain_ragged():
    d = _case(dn=5, dv=5, rank=5)
    H = d["H"]
    w = np.zeros((H, 10, 5), np.float32)
    for h in range(H):
        w[h, :5] = np.eye(5)
        w[h, 5:] = np.eye(5)
    got_o, got_l = oracle.latent_ragged(d["q"], d["c_kv"], d["k_rope"], w, d["q_offsets"], d["kv_offsets"],
                                        d["anchors"], d["block_size"])
    kv = np.repeat(d["c_kv"][:, None, :], H, axis=1)
    want_o, want_l = oracle.ragged(d["q"], kv, d["k_rope"], kv, d["q_offsets"], d["kv_offsets"], d["anchors"],
                                   d["block_size"])
    np.testing.assert_allclose(got_o, want_o, atol=TOL, rtol=0)
    np.testing.assert_allclose(got_l, want_l, atol=TOL, rtol=0)


def test_absorbed_order_gives_the_same_result():
    """Scores as (W_UK^T q_nope) . c + q_rope . k_rope and outputs as
    W_UV (sum_k p_k c_k) / sum_k p_k: the absorbed evaluation order."""
    d = _case(seed=5)
    H, dn, dr = d["H"], 6, 4
    q = d["q"].astype(np.float64)
    c = d["c_kv"].astype(np.float64)
    kr = d["k_rope"].astype(np.float64)
    w = d["w_kv_b"].astype(np.float64)
    w_uk, w_uv = w[:, :dn, :], w[:, dn:, :]
    scale = (dn + dr) ** -0.5
    qo, ko, an, bs = d["q_offsets"], d["kv_offsets"], d["anchors"], d["block_size"]
    want_o = np.zeros((d["total_q"], H, w_uv.shape[1]))
    want_l = np.zeros((H, d["total_q"]))
    for r in range(d["R"]):
        S_r = int(ko[r + 1] - ko[r]) - int(qo[r + 1] - qo[r])
        for i in range(int(qo[r + 1] - qo[r])):
            row = int(qo[r]) + i
            j = i // bs
            a = int(an[int(qo[r]) // bs + j])
            keys = [int(ko[r]) + p for p in range(min(a, S_r))]
            keys += [int(ko[r]) + S_r + j * bs + t for t in range(bs)]
            for h in range(H):
                q_lat = w_uk[h].T @ q[row, h, :dn]                      # [rank]
                s = scale * (c[keys] @ q_lat + kr[keys] @ q[row, h, dn:])
                m = s.max()
                p = np.exp(s - m)
                o_lat = p @ c[keys] / p.sum()                           # [rank]
                want_o[row, h] = w_uv[h] @ o_lat
                want_l[h, row] = m + np.log(p.sum())
    got_o, got_l = oracle.latent_ragged(d["q"], d["c_kv"], d["k_rope"], d["w_kv_b"], qo, ko, an, bs)
    np.testing.assert_allclose(got_o, want_o, atol=TOL, rtol=0)
    np.testing.assert_allclose(got_l, want_l, atol=TOL, rtol=0)


def test_matches_sdpa_on_expanded_keys():
    d = _case(seed=8, q_blocks=(2,))
    H, dn = d["H"], 6
    w = torch.from_numpy(d["w_kv_b"].astype(np.float64))
    c = torch.from_numpy(d["c_kv"].astype(np.float64))
    k_nope = torch.einsum("hec,tc->the", w[:, :dn], c)
    v = torch.einsum("hec,tc->the", w[:, dn:], c)
    got_o, _ = oracle.latent_ragged(d["q"], d["c_kv"], d["k_rope"], d["w_kv_b"], d["q_offsets"], d["kv_offsets"],
                                    d["anchors"], d["block_size"])
    qo, ko, an, bs = d["q_offsets"], d["kv_offsets"], d["anchors"], d["block_size"]
    q = torch.from_numpy(d["q"].astype(np.float64))
    kr = torch.from_numpy(d["k_rope"].astype(np.float64))
    for r in range(d["R"]):
        q0, q1, k0, k1 = int(qo[r]), int(qo[r + 1]), int(ko[r]), int(ko[r + 1])
        S_r = (k1 - k0) - (q1 - q0)
        K = torch.cat([k_nope[k0:k1], kr[k0:k1, None, :].expand(-1, H, -1)], dim=-1)   # [keys, H, dn+dr]
        mask = torch.full((q1 - q0, k1 - k0), float("-inf"), dtype=torch.float64)
        for i in range(q1 - q0):
            j = i // bs
            mask[i, :min(int(an[q0 // bs + j]), S_r)] = 0
            mask[i, S_r + j * bs:S_r + (j + 1) * bs] = 0
        o = torch.nn.functional.scaled_dot_product_attention(q[q0:q1].transpose(0, 1), K.transpose(0, 1),
                                                             v[k0:k1].transpose(0, 1), attn_mask=mask)
        np.testing.assert_allclose(got_o[q0:q1], o.transpose(0, 1).numpy(), atol=1e-10, rtol=0)


def test_latent_workload_recipe():
    d = synth.make("decode_latent_bf16", R=3, H=2)
    assert d["c_kv"].dtype == np.uint16 and d["c_kv"].shape == (d["total_kv"], 512)
    assert d["w_kv_b"].shape == (2, 256, 512) and "k_nope" not in d and "v" not in d
    w = synth.bf16_bits_to_f32(d["w_kv_b"])
    assert abs(w.std() * 512 ** 0.5 - 1.0) < 0.02  # kv_rank^-0.5 scaling: expanded keys have unit variance
    np.testing.assert_array_equal(d["anchors"], d["context_lens"])

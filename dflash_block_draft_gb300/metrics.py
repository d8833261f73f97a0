"""Work accounting for the benchmark: unmasked FLOPs and algorithmic bytes.

Unmasked FLOPs count 2*(d_qk + d_v) per visible (query row, key, head)
triple -- the two matrix products QK^T and PV restricted to the pairs the
mask lets through; exp, scaling and the softmax sums are not counted.  The
backward pass counts its five products the same way, 2*(3*d_qk + 2*d_v).
Algorithmic bytes are what the operation must move at minimum: q once, the
k_nope/v of every key that some row of the batch row sees once, the
head-shared k_rope of those keys once (not per head), the mask once (dense),
out once, and the optional lse.
"""
from __future__ import annotations

import numpy as np


def flops_per_pair(d_nope: int, d_rope: int, d_v: int) -> int:
    return 2 * (d_nope + d_rope + d_v)


def backward_flops_per_pair(d_nope: int, d_rope: int, d_v: int) -> int:
    """Backward: the five products S = QK^T (recomputed), dP = dO V^T, dV = P^T dO,
    dK = dS^T Q and dQ = dS K over the visible pairs, 2*(3*d_qk + 2*d_v) FLOPs."""
    return 2 * (3 * (d_nope + d_rope) + 2 * d_v)


def anchored_visible_counts(anchors: np.ndarray, S: int, Q: int, block_size: int) -> np.ndarray:
    """|visible keys| per query row [B, Q]: min(a_j, S) context keys plus the
    row's own block clipped to Q."""
    an = np.minimum(np.asarray(anchors, np.int64), S)
    rows = np.arange(Q)
    blk = rows // block_size
    own = np.minimum((blk + 1) * block_size, Q) - blk * block_size
    return an[:, blk] + own[None, :]


def anchored_work(anchors, S, Q, H, block_size, d_nope, d_rope, d_v, esize=2, lse=False):
    an = np.asarray(anchors)
    B = an.shape[0]
    pairs = int(anchored_visible_counts(an, S, Q, block_size).sum()) * H
    flops = pairs * flops_per_pair(d_nope, d_rope, d_v)
    keys = int((np.minimum(an.max(axis=1), S) + Q).sum()) if an.size else 0
    per_key = H * (d_nope + d_v) * esize + d_rope * esize
    nbytes = (B * Q * H * (d_nope + d_rope) * esize + keys * per_key + B * Q * H * d_v * esize + an.size * 4
              + (B * H * Q * 4 if lse else 0))
    return dict(pairs=pairs, flops=flops, bytes=nbytes, keys_read=keys)


def dense_work(visible_per_row: np.ndarray, keys_read_per_batch: np.ndarray, S, Q, H, d_nope, d_rope, d_v,
               esize=2, lse=False):
    """visible_per_row [B,Q] (entries != -inf), keys_read_per_batch [B] (keys any row sees)."""
    B = visible_per_row.shape[0]
    pairs = int(visible_per_row.sum()) * H
    per_key = H * (d_nope + d_v) * esize + d_rope * esize
    nbytes = (B * Q * H * (d_nope + d_rope) * esize + int(keys_read_per_batch.sum()) * per_key
              + B * Q * (S + Q) * esize + B * Q * H * d_v * esize + (B * H * Q * 4 if lse else 0))
    return dict(pairs=pairs, flops=pairs * flops_per_pair(d_nope, d_rope, d_v), bytes=nbytes)


def ragged_work(q_offsets, kv_offsets, anchors, H, block_size, d_nope, d_rope, d_v, esize=2, lse=False):
    qo, ko, an = (np.asarray(x, np.int64) for x in (q_offsets, kv_offsets, anchors))
    pairs = 0
    keys = 0
    for r in range(qo.size - 1):
        ql = int(qo[r + 1] - qo[r])
        S_r = int(ko[r + 1] - ko[r]) - ql
        a = an[qo[r] // block_size:qo[r + 1] // block_size]
        pairs += int(anchored_visible_counts(a[None], S_r, ql, block_size).sum())
        keys += min(int(a.max()), S_r) + ql
    total_q = int(qo[-1])
    per_key = H * (d_nope + d_v) * esize + d_rope * esize
    nbytes = (total_q * H * (d_nope + d_rope) * esize + keys * per_key + total_q * H * d_v * esize
              + (qo.size + ko.size + an.size) * 4 + (H * total_q * 4 if lse else 0))
    return dict(pairs=pairs * H, flops=pairs * H * flops_per_pair(d_nope, d_rope, d_v), bytes=nbytes,
                keys_read=keys)


def latent_flops_per_pair(kv_rank: int, d_rope: int) -> int:
    """Compressed-latent attention in absorbed form: the score over the latent
    and the rope key, 2*(kv_rank + d_rope), and the latent output, 2*kv_rank,
    per visible (query row, key, head)."""
    return 2 * (kv_rank + d_rope) + 2 * kv_rank


def latent_work(q_offsets, kv_offsets, anchors, H, block_size, d_nope, d_rope, d_v, kv_rank, esize=2):
    """Work of the compressed-latent ragged call: the attention over the latents
    (latent_flops_per_pair per visible pair) plus the query absorption and the
    output projection, 2*d_nope*kv_rank and 2*kv_rank*d_v per (row, head).
    Bytes: q once, the latent and rope key of every key some row sees once (not
    per head), the projection weight once, out once."""
    w = ragged_work(q_offsets, kv_offsets, anchors, H, block_size, d_nope, d_rope, d_v, esize=esize)
    pairs = w["pairs"]
    total_q = int(np.asarray(q_offsets)[-1])
    flops = pairs * latent_flops_per_pair(kv_rank, d_rope) + total_q * H * 2 * kv_rank * (d_nope + d_v)
    qo, ko, an = (np.asarray(x, np.int64) for x in (q_offsets, kv_offsets, anchors))
    nbytes = (total_q * H * (d_nope + d_rope) * esize + w["keys_read"] * (kv_rank + d_rope) * esize
              + H * (d_nope + d_v) * kv_rank * esize + total_q * H * d_v * esize + (qo.size + ko.size + an.size) * 4)
    return dict(pairs=pairs, flops=flops, bytes=nbytes, keys_read=w["keys_read"])

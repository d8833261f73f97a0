"""Independent numpy brute force for tiny inputs (TEST INFRASTRUCTURE ONLY).

Materialises the whole [Q, S+Q] score matrix per (batch row, head) from a
dense additive mask, exactly as the prior-art formulation does (SDPA with a
dense additive mask: nemo_automodel.components.speculative.dflash.draft_kimi_k3,
KimiK3DFlashAttention.forward), and applies a row softmax.  Written
separately from oracle.c so that each can catch a mistake in the other.
"""
from __future__ import annotations

import numpy as np


def bf16_bits_to_f64(a: np.ndarray) -> np.ndarray:
    """Widen uint16 bf16 bit patterns to float64 exactly."""
    return (np.asarray(a, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def as_f64(a: np.ndarray) -> np.ndarray:
    a = np.asarray(a)
    return bf16_bits_to_f64(a) if a.dtype == np.uint16 else a.astype(np.float64)


def dense(q, k_nope, k_rope, v, mask, scale):
    """q [B,Q,H,dn+dr], k_nope [B,K,H,dn], k_rope [B,K,dr], v [B,K,H,dv],
    mask [B,1,Q,K].  Returns out [B,Q,H,dv], lse [B,H,Q] (fully masked rows:
    out 0, lse -inf)."""
    q, kn, kr, v, mask = (as_f64(x) for x in (q, k_nope, k_rope, v, mask))
    B, Q, H, _ = q.shape
    K = kn.shape[1]
    dn = kn.shape[3]
    out = np.zeros((B, Q, H, v.shape[3]))
    lse = np.full((B, H, Q), -np.inf)
    for b in range(B):
        for h in range(H):
            # Keys of head h: per-head nope part next to the head-shared rope part.
            keys = np.concatenate([kn[b, :, h, :], kr[b]], axis=1)  # [K, dn+dr]
            scores = (q[b, :, h, :] @ keys.T) * scale + mask[b, 0]  # [Q, K]
            for i in range(Q):
                row = scores[i]
                vis = np.isfinite(mask[b, 0, i])
                if not vis.any():
                    continue
                m = row[vis].max()
                w = np.where(vis, np.exp(np.where(vis, row, m) - m), 0.0)
                out[b, i, h] = (w @ v[b, :, h, :]) / w.sum()
                lse[b, h, i] = m + np.log(w.sum())
    del dn, K
    return out, lse

"""Seeded synthetic inputs for the five DFlash block-attention workloads.

This module only draws random numbers and casts them; it holds none of the
attention arithmetic and no visibility rule, so that both the CUDA library's
tests and the fp64 oracle can take their inputs from it.

Recipe (shared by every workload):
  seed = 1000 + workload index;
  anchors (or, for the ragged workload, the context lengths) come from
  numpy.random.default_rng(seed);
  q, k_nope, k_rope, v (tensor ids 0..3) are float32 standard normals drawn in
  flat chunks of 2**22 elements, chunk c of tensor t from its own stream
  Generator(PCG64(SeedSequence(seed, spawn_key=(t, c)))) so that chunks can be
  drawn on several threads with a result that does not depend on the thread
  count; bf16 workloads round them to bf16 (nearest, ties to even).
Anchors are sorted, distinct and uniform without replacement over the stated
range.  bf16 tensors are carried as uint16 bit patterns.  The backward pass
takes its output gradient dout from the same recipe as tensor id 4.  The
compressed-latent decode workload draws the per-token KV latent c_kv as tensor
id 5 and the per-head expansion weight w_kv_b (kv_b_proj viewed as
[H, d_nope + d_v, kv_rank]) as tensor id 6, standard normals scaled by
kv_rank^-0.5 in fp32 before the bf16 rounding, so that the expanded keys and
values have unit variance like the other workloads' inputs.
"""
from __future__ import annotations

import concurrent.futures as cf
import dataclasses
import math
import os

import numpy as np


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    index: int
    dtype: str  # "fp32" | "bf16"
    H: int
    d_nope: int
    d_rope: int
    d_v: int
    # batched (dense / anchored) workloads
    B: int = 0
    S: int = 0
    nb: int = 0
    block_size: int = 0
    anchor_lo: int = 1  # anchors drawn from [anchor_lo, anchor_hi)
    anchor_hi: int = 0
    pad: int = 0  # trailing context columns that are padding (masked -inf in the dense mask)
    # ragged workload
    R: int = 0
    ctx_lo: int = 0
    ctx_hi: int = 0
    # ragged only: when set, request r has nb_r blocks drawn uniformly from these
    # counts (instead of nb each), and its anchors are drawn inside its context
    q_blocks: tuple = ()
    # ragged only: when > 0, keys and values come as compressed latents
    # c_kv [total_kv, kv_rank] plus the per-head expansion weight
    # w_kv_b [H, d_nope + d_v, kv_rank] instead of k_nope and v
    kv_rank: int = 0

    @property
    def Q(self) -> int:
        return self.nb * self.block_size

    @property
    def seed(self) -> int:
        return 1000 + self.index

    @property
    def ragged(self) -> bool:
        return self.R > 0


_LONG_S = 32768
_LONG_PAD = int(math.floor(0.05 * _LONG_S))  # 1638 padding columns, 31130 valid

WORKLOADS = {
    w.name: w
    for w in (
        Workload("tiny_fp32", 0, "fp32", H=2, d_nope=16, d_rope=8, d_v=16, B=1, S=64, nb=4,
                 block_size=4, anchor_lo=1, anchor_hi=64),
        Workload("prefill_bf16", 1, "bf16", H=16, d_nope=128, d_rope=64, d_v=128, B=1, S=4096,
                 nb=256, block_size=16, anchor_lo=1, anchor_hi=4096),
        Workload("training_bf16", 2, "bf16", H=32, d_nope=128, d_rope=64, d_v=128, B=4, S=8192,
                 nb=512, block_size=16, anchor_lo=1, anchor_hi=8192),
        Workload("long_bf16", 3, "bf16", H=16, d_nope=128, d_rope=64, d_v=128, B=2, S=_LONG_S,
                 nb=2048, block_size=8, anchor_lo=1, anchor_hi=_LONG_S - _LONG_PAD + 1,
                 pad=_LONG_PAD),
        Workload("decode_bf16", 4, "bf16", H=32, d_nope=128, d_rope=64, d_v=128, R=64,
                 block_size=16, nb=1, ctx_lo=1024, ctx_hi=32768),
        # the decode workload with the keys and values in compressed-latent form
        Workload("decode_latent_bf16", 5, "bf16", H=32, d_nope=128, d_rope=64, d_v=128, R=64,
                 block_size=16, nb=1, ctx_lo=1024, ctx_hi=32768, kv_rank=512),
    )
}


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 (nearest, ties to even); returns uint16 patterns."""
    u = np.ascontiguousarray(x, np.float32).view(np.uint32)
    out = np.empty(u.shape, np.uint16)
    flat_u, flat_o = u.reshape(-1), out.reshape(-1)
    step = 1 << 24
    for s in range(0, flat_u.size, step):
        c = flat_u[s:s + step]
        lsb = (c >> np.uint32(16)) & np.uint32(1)
        flat_o[s:s + step] = ((c + np.uint32(0x7FFF) + lsb) >> np.uint32(16)).astype(np.uint16)
    return out


def bf16_bits_to_f32(x: np.ndarray) -> np.ndarray:
    return (np.asarray(x, np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


_CHUNK = 1 << 22


def _normal(seed: int, tensor_id: int, shape, dtype: str, scale: float = 1.0) -> np.ndarray:
    n = int(np.prod(shape))
    out = np.empty(n, np.uint16 if dtype == "bf16" else np.float32)

    def fill(c):
        lo, hi = c * _CHUNK, min(n, (c + 1) * _CHUNK)
        g = np.random.Generator(np.random.PCG64(np.random.SeedSequence(seed, spawn_key=(tensor_id, c))))
        a = g.standard_normal(size=hi - lo, dtype=np.float32)
        if scale != 1.0:
            a = a * np.float32(scale)
        out[lo:hi] = f32_to_bf16_bits(a) if dtype == "bf16" else a

    nchunks = -(-n // _CHUNK)
    if nchunks <= 1:
        for c in range(nchunks):
            fill(c)
    else:
        with cf.ThreadPoolExecutor(max_workers=min(nchunks, os.cpu_count() or 4)) as ex:
            list(ex.map(fill, range(nchunks)))
    return out.reshape(shape)


def sorted_distinct(rng, lo: int, hi: int, n: int) -> np.ndarray:
    """n sorted distinct integers uniform without replacement over [lo, hi)."""
    if n > hi - lo:
        raise ValueError("range too small for distinct anchors")
    return np.sort(rng.choice(np.arange(lo, hi, dtype=np.int64), size=n, replace=False)).astype(np.int32)


def make(w: Workload | str, seed: int | None = None, **override) -> dict:
    """Draw the inputs of workload `w` (a Workload or its name).

    `override` replaces Workload fields (to make smaller cases with the same
    recipe).  Returns a dict of numpy arrays plus the integer dims.
    Batched: q [B,Q,H,dn+dr], k_nope [B,S+Q,H,dn], k_rope [B,S+Q,dr],
    v [B,S+Q,H,dv], anchors [B,nb] int32.
    Ragged: q [total_q,H,dqk], k_nope [total_kv,H,dn], k_rope [total_kv,dr],
    v [total_kv,H,dv], q_offsets/kv_offsets [R+1] int32, anchors [total_q/bs]
    int32 (each request's anchors equal its context length; with q_blocks, the
    requests' block counts differ and their anchors lie inside their contexts).
    """
    if isinstance(w, str):
        w = WORKLOADS[w]
    if override:
        w = dataclasses.replace(w, **override)
    seed = w.seed if seed is None else seed
    rng = np.random.default_rng(seed)
    dqk = w.d_nope + w.d_rope
    d = dict(workload=w, seed=seed, H=w.H, d_nope=w.d_nope, d_rope=w.d_rope, d_v=w.d_v,
             block_size=w.block_size, dtype=w.dtype)
    if w.ragged:
        lo, hi = math.log(w.ctx_lo), math.log(w.ctx_hi)
        ctx = np.rint(np.exp(rng.uniform(lo, hi, size=w.R))).astype(np.int64)
        if w.q_blocks:
            # Mixed draft lengths: nb_r blocks per request; anchors sorted uniform
            # in [0, ctx_r], the last block's anchor the whole context.
            nbr = rng.choice(np.asarray(w.q_blocks, np.int64), size=w.R)
            q_lens = nbr * w.block_size
            anchors = []
            for r in range(w.R):
                a = np.sort(rng.integers(0, ctx[r] + 1, size=nbr[r]))
                a[-1] = ctx[r]
                anchors.append(a)
            anchors = np.concatenate(anchors).astype(np.int32)
        else:
            q_lens = np.full(w.R, w.nb * w.block_size, np.int64)
            # One block per request in the decode shape: its anchor is its context length.
            anchors = np.repeat(ctx, w.nb).astype(np.int32)
        q_off = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int64)
        kv_off = np.concatenate([[0], np.cumsum(ctx + q_lens)])
        total_q, total_kv = int(q_off[-1]), int(kv_off[-1])
        d.update(R=w.R, q_offsets=q_off.astype(np.int32), kv_offsets=kv_off.astype(np.int32),
                 anchors=anchors, context_lens=ctx.astype(np.int32), total_q=total_q, total_kv=total_kv,
                 q=_normal(seed, 0, (total_q, w.H, dqk), w.dtype),
                 k_rope=_normal(seed, 2, (total_kv, w.d_rope), w.dtype))
        if w.kv_rank:
            d.update(kv_rank=w.kv_rank, c_kv=_normal(seed, 5, (total_kv, w.kv_rank), w.dtype),
                     w_kv_b=_normal(seed, 6, (w.H, w.d_nope + w.d_v, w.kv_rank), w.dtype,
                                    scale=w.kv_rank ** -0.5))
        else:
            d.update(k_nope=_normal(seed, 1, (total_kv, w.H, w.d_nope), w.dtype),
                     v=_normal(seed, 3, (total_kv, w.H, w.d_v), w.dtype))
        return d
    K = w.S + w.Q
    anchors = np.stack([sorted_distinct(rng, w.anchor_lo, w.anchor_hi, w.nb) for _ in range(w.B)])
    d.update(B=w.B, S=w.S, Q=w.Q, nb=w.nb, pad=w.pad, anchors=anchors,
             q=_normal(seed, 0, (w.B, w.Q, w.H, dqk), w.dtype),
             k_nope=_normal(seed, 1, (w.B, K, w.H, w.d_nope), w.dtype),
             k_rope=_normal(seed, 2, (w.B, K, w.d_rope), w.dtype),
             v=_normal(seed, 3, (w.B, K, w.H, w.d_v), w.dtype))
    return d


def make_dout(d: dict, seed: int | None = None) -> np.ndarray:
    """Output gradient dout [B,Q,H,dv] (batched) for the inputs `d` of :func:`make`:
    standard normals of tensor id 4 under the same seed, in d's dtype."""
    seed = d["seed"] if seed is None else seed
    return _normal(seed, 4, (d["B"], d["Q"], d["H"], d["d_v"]), d["dtype"])

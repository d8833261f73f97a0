"""Shared test helpers: moving seeded numpy inputs onto the GPU and comparing."""
from __future__ import annotations

import numpy as np

# Parity bars: max abs error vs the fp64 oracle for unit-normal inputs.
TOL = {"fp32": 1e-5, "bf16": 2e-2}


def to_torch(a: np.ndarray, dtype: str, device="cuda"):
    import torch
    a = np.ascontiguousarray(a)
    if dtype == "bf16":
        assert a.dtype == np.uint16
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(device)
    return torch.from_numpy(a).to(device)


def to_numpy_f64(t) -> np.ndarray:
    import torch
    return t.detach().to(torch.float64).cpu().numpy()


def bf16_mask(mask_f32: np.ndarray) -> np.ndarray:
    """0/-inf (or any bf16-representable) fp32 mask -> bf16 bit patterns."""
    from dflash_block_draft_gb300.synth import f32_to_bf16_bits
    return f32_to_bf16_bits(mask_f32)


def max_abs_err(got: np.ndarray, want: np.ndarray) -> float:
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    both_ninf = np.isneginf(got) & np.isneginf(want)
    with np.errstate(invalid="ignore"):
        diff = np.where(both_ninf, 0.0, np.abs(got - want))
    return float(np.nanmax(np.where(np.isnan(diff), np.inf, diff))) if diff.size else 0.0


def sample_rows(total_rows: int, n: int, seed: int = 0, per_segment: int | None = None,
                segment_len: int | None = None) -> np.ndarray:
    """Deterministic row sample: first/last rows of every segment plus uniform picks."""
    rng = np.random.default_rng(seed)
    rows = set()
    if segment_len:
        for s0 in range(0, total_rows, segment_len):
            rows.update({s0, s0 + 1, s0 + segment_len - 1, s0 + segment_len // 2})
    rows.update(rng.choice(total_rows, size=min(n, total_rows), replace=False).tolist())
    return np.array(sorted(r for r in rows if 0 <= r < total_rows), np.int64)

"""Pins for the seeded input generators (CPU only).

The generators are shared by the oracle and the CUDA path, so they hold no
attention arithmetic; these tests tie them to the stated workload
configurations and to independent restatements of their recipe.
"""
import math
from fractions import Fraction

import numpy as np

from dflash_block_draft_gb300 import synth


def test_workload_shapes_match_the_stated_configurations():
    W = synth.WORKLOADS
    tiny = W["tiny_fp32"]
    assert (tiny.dtype, tiny.B, tiny.H, tiny.S, tiny.nb, tiny.block_size, tiny.Q) == ("fp32", 1, 2, 64, 4, 4, 16)
    assert (tiny.d_nope, tiny.d_rope, tiny.d_v) == (16, 8, 16)
    for name, B, H, S, nb, bs in (("prefill_bf16", 1, 16, 4096, 256, 16), ("training_bf16", 4, 32, 8192, 512, 16),
                                  ("long_bf16", 2, 16, 32768, 2048, 8)):
        w = W[name]
        assert (w.dtype, w.B, w.H, w.S, w.nb, w.block_size) == ("bf16", B, H, S, nb, bs), name
        assert (w.d_nope, w.d_rope, w.d_v) == (128, 64, 128), name
    assert W["prefill_bf16"].Q == 4096 and W["training_bf16"].Q == 8192 and W["long_bf16"].Q == 16384
    # the last 5 % of the long context is padding: floor(0.05 * 32768) columns
    assert W["long_bf16"].pad == 1638
    dec = W["decode_bf16"]
    assert (dec.R, dec.H, dec.nb * dec.block_size, dec.ctx_lo, dec.ctx_hi) == (64, 32, 16, 1024, 32768)
    assert [W[n].seed for n in ("tiny_fp32", "prefill_bf16", "training_bf16", "long_bf16", "decode_bf16")] == \
        [1000, 1001, 1002, 1003, 1004]


def _bf16_reference(x: float) -> int:
    """Round-to-nearest-even to bf16 by exact rational arithmetic (finite inputs)."""
    if x == 0.0:
        return 0x8000 if math.copysign(1.0, x) < 0 else 0
    sign = 0x8000 if x < 0 else 0
    a = Fraction(abs(x))
    # bf16 keeps 8 significant bits; exponent range as float32
    e = math.floor(math.log2(abs(x)))
    if Fraction(2) ** e > a:
        e -= 1
    elif Fraction(2) ** (e + 1) <= a:
        e += 1
    e = max(e, -126)  # subnormal spacing below 2^-126
    ulp = Fraction(2) ** (e - 7)
    q, r = divmod(a, ulp)
    if r * 2 > ulp or (r * 2 == ulp and q % 2 == 1):
        q += 1
    v = q * ulp
    if v >= Fraction(2) ** 128:
        return sign | 0x7F80
    bits = int(np.array([float(v)], np.float32).view(np.uint32)[0]) >> 16
    return sign | bits


def test_bf16_rounding_is_nearest_even():
    cases = [1.0, 1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, 1.0 + 2.0 ** -8 + 2.0 ** -20, -1.5, 2.0 ** -130,
             3.0e38, -0.0, 65504.0, 1.0 / 3.0]
    rng = np.random.default_rng(0)
    cases += [float(v) for v in rng.standard_normal(200).astype(np.float32)]
    cases += [float(v) for v in (rng.standard_normal(50) * 1e-39).astype(np.float32)]
    x = np.array(cases, np.float32)
    got = synth.f32_to_bf16_bits(x)
    want = np.array([_bf16_reference(float(v)) for v in x], np.uint16)
    np.testing.assert_array_equal(got, want)
    # ties: halfway values go to the even neighbour
    assert synth.f32_to_bf16_bits(np.array([1.0 + 2.0 ** -8], np.float32))[0] == 0x3F80
    assert synth.f32_to_bf16_bits(np.array([1.0 + 3 * 2.0 ** -8], np.float32))[0] == 0x3F82
    assert synth.f32_to_bf16_bits(np.array([np.inf, -np.inf], np.float32)).tolist() == [0x7F80, 0xFF80]
    np.testing.assert_array_equal(synth.bf16_bits_to_f32(got).view(np.uint32) >> 16, got)


def test_chunked_normals_equal_their_streams_drawn_one_by_one():
    # more than one 2^22-element chunk, drawn on threads; each chunk must equal
    # the output of its own PCG64(SeedSequence(seed, spawn_key=(tensor, chunk)))
    n = (1 << 22) + 12345
    got = synth._normal(77, 3, (n,), "fp32")
    for c in range(2):
        lo, hi = c << 22, min(n, (c + 1) << 22)
        g = np.random.Generator(np.random.PCG64(np.random.SeedSequence(77, spawn_key=(3, c))))
        np.testing.assert_array_equal(got[lo:hi], g.standard_normal(size=hi - lo, dtype=np.float32))
    again = synth._normal(77, 3, (n,), "fp32")
    np.testing.assert_array_equal(got, again)
    bf = synth._normal(77, 3, (n,), "bf16")
    np.testing.assert_array_equal(bf, synth.f32_to_bf16_bits(got))


def test_anchor_recipe_sorted_distinct_in_range():
    # tiny head dims keep the tensors small; the anchors are drawn first, so
    # they are the workloads' own anchors
    for name in ("tiny_fp32", "prefill_bf16", "training_bf16", "long_bf16"):
        w = synth.WORKLOADS[name]
        d = synth.make(name, H=1, d_nope=1, d_rope=1, d_v=1)
        an = d["anchors"]
        assert an.shape == (w.B, w.nb) and an.dtype == np.int32
        assert np.all(np.diff(an, axis=1) > 0), name
        assert an.min() >= w.anchor_lo and an.max() < w.anchor_hi, name
        if name == "long_bf16":
            assert an.max() <= w.S - w.pad  # anchored rows never see padding
        full = synth.make(name, H=1, d_nope=1, d_rope=1, d_v=1)
        np.testing.assert_array_equal(full["anchors"], an)


def test_decode_recipe():
    d = synth.make("decode_bf16", H=1, d_nope=1, d_rope=1, d_v=1)
    ctx = d["context_lens"].astype(np.int64)
    assert ctx.size == 64 and ctx.min() >= 1024 and ctx.max() <= 32768
    np.testing.assert_array_equal(d["q_offsets"], np.arange(65) * 16)
    np.testing.assert_array_equal(np.diff(d["kv_offsets"]), ctx + 16)
    np.testing.assert_array_equal(d["anchors"], ctx)  # one block per request, anchored at its context length
    # log-uniform: the mean of log(ctx) sits near the middle of [log 1024, log 32768]
    mid = 0.5 * (math.log(1024) + math.log(32768))
    assert abs(np.log(ctx).mean() - mid) < 0.5


def test_mixed_draft_length_recipe():
    d = synth.make("decode_bf16", R=40, H=1, d_nope=1, d_rope=1, d_v=1, block_size=8, q_blocks=(1, 2, 3))
    qo, ko = d["q_offsets"].astype(np.int64), d["kv_offsets"].astype(np.int64)
    ctx = d["context_lens"].astype(np.int64)
    qlens = np.diff(qo)
    assert set(qlens.tolist()) == {8, 16, 24}  # every count drawn at least once among 40 requests
    assert qo[0] == 0 and np.all(qo % 8 == 0) and d["total_q"] == qo[-1]
    np.testing.assert_array_equal(np.diff(ko), ctx + qlens)
    assert d["anchors"].size == qo[-1] // 8
    for r in range(40):
        a = d["anchors"][qo[r] // 8:qo[r + 1] // 8]
        assert np.all(np.diff(a) >= 0) and a.min() >= 0 and a[-1] == ctx[r]
    assert d["q"].shape == (qo[-1], 1, 2) and d["k_nope"].shape == (ko[-1], 1, 1)


def test_dout_is_its_own_stream():
    d = synth.make("tiny_fp32")
    g1, g2 = synth.make_dout(d), synth.make_dout(d)
    np.testing.assert_array_equal(g1, g2)
    assert g1.shape == (1, 16, 2, 16) and g1.dtype == np.float32
    assert not np.array_equal(g1.reshape(-1)[:64], d["q"].reshape(-1)[:64])
    g = np.random.Generator(np.random.PCG64(np.random.SeedSequence(1000, spawn_key=(4, 0))))
    np.testing.assert_array_equal(g1.reshape(-1), g.standard_normal(size=g1.size, dtype=np.float32))

"""The token format a block-scaled tensor-core path (MXFP8 tokens x MXFP4 experts, the
E8M0 scales applied by the MMA) would need, checked on the CPU before any such kernel.

An e4m3 element holds 4 significant bits, a bf16 token element 8, so one e4m3 copy of a
token loses precision far beyond the layer's 5e-3 bar.  Two terms do not: every
32-element block of a token row becomes hi * 2^a + lo * 2^b, hi and lo e4m3 (round to
nearest even), 2^a the smallest power of two that brings the block's largest magnitude
to 448 (the largest e4m3) or below, lo the same for the remainder x - hi * 2^a.  The test
checks on every workload's tokens (unit normal rows, the 1% of rows scaled by 8) that
the two terms rebuild every element within 2^-12 of its block's largest magnitude bit
for bit; the few smaller elements (an element 2^-17 below its block's largest keeps
about 4 of its 8 significant bits in the remainder's e4m3) leave the rebuilt tokens
within 1e-8 (relative L2) of the originals, against the layer's 5e-3 bar.  It also
measures the split on heavier-tailed tokens, which the workloads do not have.
"""
import numpy as np
import pytest

import k3moe_inputs as ki

E4M3_MAX = 448.0


def e4m3_rne(v):
    """v (float64, |v| <= 448) rounded to the nearest e4m3 value, ties to even: 3 stored
    mantissa bits, exponents -6..8, subnormal steps of 2^-9."""
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(e, -6.0)                       # below 2^-6: the subnormal step
    q = np.exp2(e - 3.0)
    r = np.round(v / q) * q                       # numpy rounds halves to even
    assert np.all(np.abs(r) <= E4M3_MAX)
    return r


def block_scale(a):
    """Smallest power of two s with a / s <= 448 (1 where the block is all zero)."""
    a = np.asarray(a, dtype=np.float64)
    return np.where(a > 0, np.exp2(np.ceil(np.log2(np.where(a > 0, a, 1.0) / E4M3_MAX))), 1.0)


def split_two_term(x):
    """x [rows, cols] float64 (cols a multiple of 32) -> the rebuilt hi*s_hi + lo*s_lo."""
    rows, cols = x.shape
    xb = x.reshape(rows, cols // 32, 32)
    s_hi = block_scale(np.abs(xb).max(axis=2, keepdims=True))
    hi = e4m3_rne(xb / s_hi)
    r = xb - hi * s_hi                            # exact in float64
    s_lo = block_scale(np.abs(r).max(axis=2, keepdims=True))
    lo = e4m3_rne(r / s_lo)
    return (hi * s_hi + lo * s_lo).reshape(rows, cols)


def test_e4m3_rounding_on_its_own_grid():
    # every e4m3 magnitude maps to itself, and the midpoints round to even mantissas
    grid = [m * 2.0 ** -9 for m in range(8)] + [(8 + m) * 2.0 ** (e - 3) for e in range(-6, 9) for m in range(8)]
    grid = np.array([g for g in grid if g <= E4M3_MAX])
    np.testing.assert_array_equal(e4m3_rne(grid), grid)
    np.testing.assert_array_equal(e4m3_rne(-grid), -grid)
    assert e4m3_rne(1.0 + 1.0 / 16) == 1.0        # halfway between 1 and 1.125: even
    assert e4m3_rne(1.0 + 3.0 / 16) == 1.25       # halfway between 1.125 and 1.25: even
    assert e4m3_rne(2.0 ** -10) == 0.0            # half the smallest subnormal: even (zero)


@pytest.mark.parametrize("name", ["tiny", "decode_t1", "decode_t64", "prefill_t4096", "prefill_t16k"])
def test_two_term_split_rebuilds_every_workload_token(name):
    w = ki.WORKLOADS[name]
    x = ki.bf16_to_f32(ki.make_x(w)).astype(np.float64)
    got = split_two_term(x)
    amax = np.repeat(np.abs(x.reshape(x.shape[0], -1, 32)).max(axis=2), 32, axis=1)
    big = np.abs(x) >= amax * 2.0 ** -12
    np.testing.assert_array_equal(got[big], x[big])
    rel = np.linalg.norm(got - x) / np.linalg.norm(x)
    print(f"[{name}] inexact {np.count_nonzero(got != x)} of {x.size} "
          f"(all below 2^-12 of their block's largest), rel-L2 {rel:.2e}")
    assert rel < 1e-8


def test_two_term_split_on_heavier_tails():
    """Not the workloads: Student-t(3) tokens (rounded to bf16) lose bits only where an
    element sits far below its block's largest; the rebuilt tokens stay within 1e-6
    (relative L2) of the originals, against the layer's 5e-3 bar."""
    rng = np.random.default_rng(11)
    t = rng.standard_t(3, size=(512, 3584))
    x = ki.bf16_to_f32(ki.f32_to_bf16(t.astype(np.float32))).astype(np.float64)
    got = split_two_term(x)
    rel = np.linalg.norm(got - x) / np.linalg.norm(x)
    print(f"student-t(3): {np.count_nonzero(got != x)} of {x.size} inexact, rel-L2 {rel:.2e}")
    assert rel < 1e-6

"""The seeded input generator: determinism, slicing, ranges and distributions."""
import math

import numpy as np

import k3moe_inputs as ki


def test_counter_based_slices_regenerate():
    a = ki.random_bytes(4096, 3, 17)
    b = ki.random_bytes(1024, 3, 17, offset=2048)
    np.testing.assert_array_equal(a[2048:3072], b)
    n = ki.bf16_normal(1000, 3, 18, 1.0)
    m = ki.bf16_normal(100, 3, 18, 1.0, offset=450)
    np.testing.assert_array_equal(n[450:550], m)
    assert not np.array_equal(ki.random_bytes(64, 3, 17), ki.random_bytes(64, 4, 17))


def test_expert_draws_are_per_expert_and_in_range():
    w = ki.WORKLOADS["tiny"]
    e0, e1 = ki.make_expert(w, 0), ki.make_expert(w, 1)
    assert e0["w1_packed"].shape == (w.f, w.d // 2) and e0["w2_scale"].shape == (w.d, w.f // 32)
    assert not np.array_equal(e0["w1_packed"], e1["w1_packed"])
    for name in ("w1_scale", "w3_scale", "w2_scale"):
        assert e0[name].min() >= w.scale_lo and e0[name].max() <= w.scale_hi
    blk = ki.make_experts_block(w, 0, 2)
    np.testing.assert_array_equal(blk["w3_packed"][1], e1["w3_packed"])


def test_codes_uniform_and_normals_standard():
    b = ki.random_bytes(1 << 20, 9, 1)
    counts = np.bincount(np.concatenate([b & 15, b >> 4]), minlength=16)
    assert counts.min() > 0.97 * counts.mean() and counts.max() < 1.03 * counts.mean()
    z = ki.bf16_to_f32(ki.bf16_normal(1 << 18, 9, 2, 1.0)).astype(np.float64)
    assert abs(z.mean()) < 0.01 and abs(z.std() - 1.0) < 0.01
    assert abs(np.mean(z ** 4) - 3.0) < 0.05


def test_bf16_round_to_nearest_even():
    f = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 3.0e38], dtype=np.float32)
    got = ki.f32_to_bf16(f)
    assert got.tolist() == [0x3F80, 0x3F80, 0x3F82, 0xC020, 0x7F62]
    for v in f:
        assert ki._load().k3g_f32_to_bf16(float(v)) == ki.f32_to_bf16(np.array([v]))[0]


def test_workload_recipes():
    w = ki.WORKLOADS["prefill_t4096"]
    rows = ki.outlier_rows(w)
    assert len(rows) == 41 and len(set(rows.tolist())) == 41
    x = ki.make_x(w.with_(outlier_frac=0.0))
    xo = ki.make_x(w)
    np.testing.assert_array_equal(ki.bf16_to_f32(xo[rows]), 8 * ki.bf16_to_f32(x[rows]))
    others = np.setdiff1d(np.arange(w.T), rows)
    np.testing.assert_array_equal(xo[others], x[others])
    zb = ki.WORKLOADS["prefill_t16k"]
    bias = ki.make_bias(zb)
    ranks = ki.permutation(zb.E, zb.seed, ki.STREAM_BIAS_RANKS)
    for r in (1, 2, 10, 896):
        assert abs(bias[ranks[r - 1]] - (-0.11 * math.log(r))) < 1e-6
    assert ki.make_bias(ki.WORKLOADS["decode_t1"]) is None
    assert abs(ki.WORKLOADS["decode_t1"].shared_sigma - 0.0236) < 1e-4

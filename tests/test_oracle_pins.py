"""Pins of the CPU oracle to facts fixed outside it.

Each test checks the oracle against something other than its own code: values
printed on the pages (``tests/golden/``), closed forms, invariants, textbook
special cases, library routines used as an independent method (a full
lexicographic sort, a dense numpy mat-vec), or an independent brute force.
Each is chosen so that a plausible mistake in the oracle -- a swapped nibble,
a missing scale, the bias leaking into the weights, the capped gate fed to the
sigmoid, a transposed operand -- fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest

import k3moe_inputs as ki
import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def golden(name):
    with open(os.path.join(GOLDEN, name)) as fh:
        return json.load(fh)


FMT = golden("mxfp4_format.json")
LUT = np.array(FMT["e2m1_lut"], dtype=np.float64)


# ----------------------------------------------------------------------------- independent dense decode

def dense_mxfp4(packed: np.ndarray, scales: np.ndarray, group: int = 32) -> np.ndarray:
    """Dense fp64 decode written from the format note alone (LUT, 2^(b-127),
    255 -> 0, low nibble = even column); vectorised numpy, not the oracle."""
    rows, half = packed.shape
    codes = np.empty((rows, 2 * half), dtype=np.int64)
    codes[:, 0::2] = packed & 15
    codes[:, 1::2] = packed >> 4
    s = np.where(scales == 255, 0.0, np.ldexp(1.0, scales.astype(np.int64) - 127))
    return LUT[codes] * np.repeat(s, group, axis=1)


def dense_bf16(bits: np.ndarray) -> np.ndarray:
    return ki.bf16_to_f32(bits).astype(np.float64)


# ----------------------------------------------------------------------------- MXFP4 format

def test_expert_size_matches_census():
    shp = FMT["expert_shape"]
    d, f = shp["d_latent"], shp["f_moe_inter"]
    assert 3 * d * f == FMT["expert_params"]
    assert FMT["expert_params"] * FMT["bytes_per_weight"] == FMT["expert_bytes"]
    w = ki.WORKLOADS["decode_t1"]
    assert w.expert_bytes == FMT["expert_bytes"]
    # the checkpoint sample's layout: two nibbles per byte, one scale per 32 columns
    smp = FMT["sample_tensor"]
    assert smp["packed_cols"] * 2 == smp["logical_width"]
    assert smp["scale_cols"] * FMT["group_size"] == smp["logical_width"]


def test_e2m1_table_matches_page():
    for code in range(16):
        v = oracle.e2m1(code)
        assert v == LUT[code]
        assert math.copysign(1.0, v) == math.copysign(1.0, LUT[code])  # code 8 is -0.0


def test_e8m0_closed_form_all_bytes():
    for b in range(255):
        assert oracle.e8m0(b) == 2.0 ** (b - FMT["scale_bias"])
    assert oracle.e8m0(FMT["nan_scale_byte"]) == FMT["nan_scale_value"]


def test_mxfp4_decode_exhaustive_codes_and_scales():
    """Every (code, scale byte) pair, at both nibble positions, against the closed form."""
    G = 32
    for b in range(256):
        packed = np.zeros((16, 16), dtype=np.uint8)        # 16 rows x 32 columns
        for code in range(16):
            packed[code, :] = code | (((code + 5) & 15) << 4)
        scales = np.full((16, 1), b, dtype=np.uint8)
        s = 0.0 if b == 255 else 2.0 ** (b - 127)
        for code in range(16):
            even = oracle.mxfp4_weight(packed, scales, G, G, code, 4)
            odd = oracle.mxfp4_weight(packed, scales, G, G, code, 5)
            assert even == LUT[code] * s
            assert odd == LUT[(code + 5) & 15] * s


def test_nibble_order_is_positional():
    """Distinct codes at every position: only the low-nibble-is-even reading decodes them."""
    G = 32
    codes = np.array([(3 * i + 1) % 16 for i in range(G)], dtype=np.uint8)
    packed = (codes[0::2] | (codes[1::2] << 4)).reshape(1, G // 2).astype(np.uint8)
    scales = np.array([[127]], dtype=np.uint8)
    got = [oracle.mxfp4_weight(packed, scales, G, G, 0, c) for c in range(G)]
    assert got == [LUT[c] for c in codes]
    swapped = [LUT[c] for c in np.stack([codes[1::2], codes[0::2]], 1).ravel()]
    assert got != swapped
    # the same through the mat-vec: unit vectors pick single columns
    for c in range(G):
        x = np.zeros(G)
        x[c] = 1.0
        assert oracle.mxfp4_matvec(x, packed, scales, G)[0] == LUT[codes[c]]
    # identical statistics under the swap, so only a positional test can tell
    assert sorted(got) == sorted(swapped)


def test_mxfp4_matvec_matches_dense_fp64():
    rng = np.random.default_rng(7)
    rows, cols = 48, 256
    packed = ki.random_bytes(rows * cols // 2, 11, 99).reshape(rows, cols // 2)
    scales = ki.uniform_bytes(rows * cols // 32, 11, 98, 100, 140).reshape(rows, cols // 32)
    scales[3, 2] = 255              # a NaN scale byte zeroes exactly its group
    scales[7, :] = 255
    x = rng.standard_normal(cols)
    y = oracle.mxfp4_matvec(x, packed, scales)
    W = dense_mxfp4(packed, scales)
    ref = W @ x
    mag = np.abs(W) @ np.abs(x)
    assert np.all(np.abs(y - ref) <= 1e-13 * mag + 1e-300)
    assert y[7] == 0.0
    # a transposed reading or a dropped scale would miss by O(1)
    assert np.max(np.abs(y - (W * 2.0) @ x)) > 1e-3 * np.max(mag)


def test_bf16_matvec_matches_dense_fp64():
    rows, cols = 40, 192
    W = ki.bf16_normal(rows * cols, 3, 5, 0.05).reshape(rows, cols)
    x = np.random.default_rng(1).standard_normal(cols)
    y = oracle.bf16_matvec(x, W)
    Wd = dense_bf16(W)
    ref = Wd @ x
    assert np.all(np.abs(y - ref) <= 1e-13 * (np.abs(Wd) @ np.abs(x)))


# ----------------------------------------------------------------------------- SiTU

SITU = golden("situ_fixture.json")


def sigmoid(z):
    return 1.0 / (1.0 + math.exp(-z))


def test_situ_reaches_the_printed_cap():
    b1, b2 = SITU["b1"], SITU["b2"]
    lo, hi = SITU["input_span"]
    top = oracle.situ(hi, hi, b1, b2)
    assert f"{abs(top):.3f}" == SITU["printed_cap_3dp"]
    assert abs(top) <= SITU["cap"]
    for g in np.geomspace(lo, hi, 41):
        for u in np.geomspace(lo, hi, 41):
            for sg, su in ((1, 1), (-1, 1), (1, -1), (-1, -1)):
                assert abs(oracle.situ(sg * g, su * u, b1, b2)) <= SITU["cap"]


def test_situ_small_input_limit_is_swiglu():
    """For |g| << b1, |u| << b2 the caps vanish: situ -> SiLU(g) * u (SwiGLU)."""
    b1, b2 = SITU["b1"], SITU["b2"]
    for g, u in ((1e-3, 2e-3), (-3e-3, 1e-3), (1e-4, -5e-4)):
        silu_u = g * sigmoid(g) * u
        assert abs(oracle.situ(g, u, b1, b2) / silu_u - 1.0) < 1e-6


def test_situ_sigmoid_reads_uncapped_gate():
    """At g = 10 the capped gate b1*tanh(g/b1) = 3.95; sigma(3.95) and sigma(10)
    differ by 2%, so feeding the capped value is caught."""
    b1, b2 = SITU["b1"], SITU["b2"]
    g, u = 10.0, 7.0
    caps = b1 * math.tanh(g / b1) * b2 * math.tanh(u / b2)
    ratio = oracle.situ(g, u, b1, b2) / caps
    assert abs(ratio - sigmoid(g)) < 1e-12
    assert abs(ratio - sigmoid(b1 * math.tanh(g / b1))) > 1e-2


def test_situ_odd_in_up_and_zero_at_zero():
    for g in (-3.0, 0.5, 40.0):
        for u in (0.1, 2.0, 300.0):
            assert oracle.situ(g, -u) == -oracle.situ(g, u)
    assert oracle.situ(0.0, 5.0) == 0.0
    assert oracle.situ(5.0, 0.0) == 0.0


# ----------------------------------------------------------------------------- router

def lexsort_topk(ch_row: np.ndarray, k: int):
    """Independent method: full sort by (ch descending, index ascending)."""
    order = np.lexsort((np.arange(ch_row.size), -ch_row.astype(np.float64)))
    return order[:k], order


def test_topk_equals_full_sort_with_ties():
    rng = np.random.default_rng(3)
    T, E, k = 64, 96, 16
    # coarse grid -> many exact ties; ties must go to the lower index
    sc = (np.round(rng.random((T, E)) * 40) / 40).astype(np.float32)
    ch = sc.copy()
    c = oracle.cfg(d=32, f=32, n_experts=E, top_k=k, n_shared=0)
    idx, w, gap = oracle.select(c, sc, ch)
    for t in range(T):
        want, order = lexsort_topk(ch[t], k)
        assert list(idx[t]) == list(want)
        assert gap[t] == ch[t][order[k - 1]] - ch[t][order[k]]


def test_router_bias_fixture_selection_only():
    fx = golden("router_bias_fixture.json")
    sc = np.array(fx["sc"], dtype=np.float32)
    bias = np.array(fx["bias"], dtype=np.float32)
    ch = sc + bias
    T, E = sc.shape
    k = fx["top_k"]
    c = oracle.cfg(d=32, f=32, n_experts=E, top_k=k, n_shared=0)
    idx, w, _ = oracle.select(c, sc, ch)
    assert idx.tolist() == fx["expected_idx"]
    reordered = sum(a != b for a, b in zip(fx["expected_idx"], fx["unbiased_idx"]))
    assert reordered == 5
    # weights come from the UNBIASED scores of the chosen experts, renormalised
    for t in range(T):
        s_sel = sc[t, idx[t]]
        np.testing.assert_allclose(w[t], s_sel / s_sel.sum(), rtol=1e-6)
        c_sel = ch[t, idx[t]]
        if reordered and not np.allclose(s_sel / s_sel.sum(), c_sel / c_sel.sum()):
            assert not np.allclose(w[t], c_sel / c_sel.sum(), rtol=1e-4)
    # without renorm the weights are the raw unbiased scores times routed_scale
    c2 = oracle.cfg(d=32, f=32, n_experts=E, top_k=k, n_shared=0, renorm=0, routed_scale=2.5)
    idx2, w2, _ = oracle.select(c2, sc, ch)
    assert idx2.tolist() == fx["expected_idx"]
    for t in range(T):
        np.testing.assert_array_equal(w2[t], sc[t, idx2[t]] * np.float32(2.5))


def test_renorm_guard_zero_sum():
    """Renormalisation only when the chosen scores sum to a positive number."""
    sc = np.zeros((1, 8), dtype=np.float32)
    ch = np.zeros((1, 8), dtype=np.float32)
    c = oracle.cfg(d=32, f=32, n_experts=8, top_k=3, n_shared=0)
    idx, w, _ = oracle.select(c, sc, ch)
    assert idx.tolist() == [[0, 1, 2]]          # all tied: lowest indices, in order
    assert np.all(w == 0.0) and np.all(np.isfinite(w))


@pytest.mark.parametrize("name", ["tiny", "decode_t64"])
def test_route_invariants_and_scores(name):
    wl = ki.WORKLOADS[name]
    if name == "decode_t64":
        wl = wl.with_(T=8)
    x, Wr, bias = ki.make_x(wl), ki.make_router(wl), ki.make_bias(wl)
    c = oracle.cfg(**wl.config_kwargs())
    idx, w, gap, sc, ch = oracle.route(c, x, Wr, bias, want_scores=True)
    T, E, k = wl.T, wl.E, wl.k
    assert idx.shape == (T, k)
    for t in range(T):
        assert len(set(idx[t].tolist())) == k                       # k distinct experts
        assert idx[t].min() >= 0 and idx[t].max() < E
        assert abs(float(w[t].astype(np.float64).sum()) - 1.0) <= 1e-6 * k   # weights sum to 1
        want, _ = lexsort_topk(ch[t], k)
        assert list(idx[t]) == list(want)
    # the scores: sigmoid of the float-rounded fp64 logit (independent numpy matmul)
    logit = (dense_bf16(x) @ dense_bf16(Wr).T).astype(np.float32)
    ref = (1.0 / (1.0 + np.exp(-logit.astype(np.float64)))).astype(np.float32)
    ulp = np.spacing(np.maximum(np.abs(ref), np.float32(1e-30)))
    assert np.all(np.abs(sc - ref) <= 4 * ulp)
    np.testing.assert_array_equal(ch, sc + (bias if bias is not None else np.float32(0)))


def test_route_bias_changes_selection_not_weights_source():
    """With a bias the chosen set changes, and weights are sc of the chosen."""
    wl = ki.WORKLOADS["prefill_t16k"].with_(T=6)
    x, Wr, bias = ki.make_x(wl), ki.make_router(wl), ki.make_bias(wl)
    c = oracle.cfg(**wl.config_kwargs())
    idx_b, w_b, _, sc, _ = oracle.route(c, x, Wr, bias, want_scores=True)
    idx_u, _, _ = oracle.route(c, x, Wr, None)
    assert any(set(a) != set(b) for a, b in zip(idx_b.tolist(), idx_u.tolist()))
    for t in range(wl.T):
        s = sc[t, idx_b[t]]
        np.testing.assert_allclose(w_b[t], s / s.sum(), rtol=1e-6)


# ----------------------------------------------------------------------------- permutation

def test_perm_is_stable_counting_sort():
    rng = np.random.default_rng(5)
    T, E, k = 37, 20, 4
    idx = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
    offsets, perm = oracle.perm(idx, E)
    counts = np.bincount(idx.ravel(), minlength=E)
    assert offsets[0] == 0 and offsets[-1] == T * k
    np.testing.assert_array_equal(np.diff(offsets), counts)
    np.testing.assert_array_equal(perm, np.argsort(idx.ravel(), kind="stable"))
    assert sorted(perm.tolist()) == list(range(T * k))


# ----------------------------------------------------------------------------- whole layer vs brute force

def brute_force_layer(wl, x, Wr, bias, experts, shared):
    """Independent dense fp64 restatement: float32 router scores, full-sort
    top-k, dense decoded weights, numpy tanh/exp, fp64 accumulation."""
    T, E, k, S = wl.T, wl.E, wl.k, wl.S
    xd = dense_bf16(x)
    logit = (xd @ dense_bf16(Wr).T).astype(np.float32)
    sc = (np.float32(1) / (np.float32(1) + np.exp(-logit))).astype(np.float32)
    ch = sc + (bias if bias is not None else np.float32(0))
    b1, b2 = wl.situ_b1, wl.situ_b2

    def situ(g, u):
        return b1 * np.tanh(g / b1) / (1.0 + np.exp(-g)) * (b2 * np.tanh(u / b2))

    dense = {}
    out = np.zeros((T, wl.d))
    idx_all = np.zeros((T, k), dtype=np.int64)
    for t in range(T):
        sel, _ = lexsort_topk(ch[t], k)
        idx_all[t] = sel
        wsel = sc[t, sel].astype(np.float32)
        if wl.renorm:
            s = np.float32(0)
            for v in wsel:
                s = np.float32(s + v)
            if s > 0:
                wsel = (wsel / s).astype(np.float32)
        wsel = (wsel * np.float32(wl.routed_scale)).astype(np.float32)
        for e, wt in zip(sel, wsel):
            if e not in dense:
                q = experts[e]
                dense[e] = tuple(dense_mxfp4(q[f"{m}_packed"], q[f"{m}_scale"]) for m in ("w1", "w3", "w2"))
            W1, W3, W2 = dense[e]
            out[t] += float(wt) * (W2 @ situ(W1 @ xd[t], W3 @ xd[t]))
        for s in range(S):
            W1, W3, W2 = (dense_bf16(shared[m][s]) for m in ("w1", "w3", "w2"))
            out[t] += W2 @ situ(W1 @ xd[t], W3 @ xd[t])
    return out, idx_all, sc, ch


def _layer_case(wl):
    x, Wr, bias = ki.make_x(wl), ki.make_router(wl), ki.make_bias(wl)
    experts = {e: ki.make_expert(wl, e) for e in range(wl.E)}
    shared = ki.make_shared(wl) if wl.S else None
    return x, Wr, bias, experts, shared


MICRO = ki.Workload("micro", T=5, d=64, f=32, E=8, k=2, S=1, exp_lo=-6, exp_hi=-2, seed=21)


@pytest.mark.parametrize("wl", [
    ki.WORKLOADS["tiny"],
    MICRO,
    MICRO.with_(name="micro_bias", zipf_bias=True, seed=22, E=12, k=3),
    MICRO.with_(name="micro_k_eq_E", k=8, seed=23),                 # every expert chosen
    MICRO.with_(name="micro_one_expert", E=1, k=1, seed=24),        # out = FFN(x) + shared(x)
    MICRO.with_(name="micro_no_renorm", renorm=0, routed_scale=0.75, seed=25),
    MICRO.with_(name="micro_no_shared", S=0, seed=26),
], ids=lambda w: w.name)
def test_layer_matches_brute_force(wl):
    x, Wr, bias, experts, shared = _layer_case(wl)
    c = oracle.cfg(**wl.config_kwargs())
    idx, w, gap = oracle.route(c, x, Wr, bias)
    out = oracle.forward(c, x, idx, w, experts, shared)
    ref, ref_idx, sc, ch = brute_force_layer(wl, x, Wr, bias, experts, shared)
    for t in range(wl.T):
        if gap[t] >= 1e-6:
            assert list(idx[t]) == list(ref_idx[t])
    scale = np.max(np.abs(ref))
    assert np.max(np.abs(out - ref)) <= 1e-6 * scale
    if wl.E == wl.k:
        np.testing.assert_allclose(w.sum(axis=1), 1.0, rtol=1e-6)
        assert all(sorted(r) == list(range(wl.E)) for r in idx.tolist())


def test_one_expert_layer_is_ffn_plus_shared():
    wl = MICRO.with_(E=1, k=1, seed=31)
    x, Wr, bias, experts, shared = _layer_case(wl)
    c = oracle.cfg(**wl.config_kwargs())
    idx, w, _ = oracle.route(c, x, Wr, None)
    assert np.all(idx == 0) and np.all(w == 1.0)
    out = oracle.forward(c, x, idx, w, experts, shared)
    nosh = oracle.forward(oracle.cfg(**wl.with_(S=0).config_kwargs()), x, idx, w, experts, None)
    shonly = out - nosh
    # the shared part equals the layer of a single routed expert whose weights are the shared ones
    assert np.max(np.abs(shonly)) > 0


def test_shared_output_independent_of_routing():
    wl = ki.WORKLOADS["tiny"]
    x, Wr, bias, experts, shared = _layer_case(wl)
    c = oracle.cfg(**wl.config_kwargs())
    idx, w, _ = oracle.route(c, x, Wr, None)
    _, sh1 = oracle.forward(c, x, idx, w, experts, shared, want_shared=True)
    idx2 = np.roll(idx, 1, axis=1)[:, ::-1].copy()
    idx2[:, 0] = (idx2[:, 0] + 7) % wl.E
    idx2 = np.stack([r if len(set(r)) == len(r) else idx[i] for i, r in enumerate(idx2)])
    w2 = np.full_like(w, 0.3)
    out2, sh2 = oracle.forward(c, x, idx2, w2, experts, shared, want_shared=True)
    np.testing.assert_array_equal(sh1, sh2)
    out1 = oracle.forward(c, x, idx, w, experts, shared)
    assert np.max(np.abs(out1 - out2)) > 0


def test_missing_expert_is_an_error_not_a_skip():
    wl = ki.WORKLOADS["tiny"]
    x, Wr, bias, experts, shared = _layer_case(wl)
    c = oracle.cfg(**wl.config_kwargs())
    idx, w, _ = oracle.route(c, x, Wr, None)
    missing = dict(experts)
    del missing[int(idx[0, 0])]
    with pytest.raises(RuntimeError):
        oracle.forward(c, x, idx, w, missing, shared)


def test_invalid_configs_rejected():
    bad = [
        dict(d=0, f=32, n_experts=4, top_k=2, n_shared=0),
        dict(d=64, f=32, n_experts=4, top_k=5, n_shared=0),
        dict(d=48, f=32, n_experts=4, top_k=2, n_shared=0),
        dict(d=64, f=32, n_experts=4, top_k=2, n_shared=0, situ_b1=0.0),
        dict(d=64, f=32, n_experts=4, top_k=2, n_shared=0, renorm=2),
    ]
    lib = oracle.lib()
    import ctypes
    for kw in bad:
        assert lib.k3o_check_cfg(ctypes.byref(oracle.cfg(**kw))) != 0


# ----------------------------------------------------------------------------- full-width block

def _full_case(wl):
    h, Wr, bias = ki.make_h(wl), ki.make_full_router(wl), ki.make_bias(wl)
    experts = {e: ki.make_expert(wl, e) for e in range(wl.E)}
    full = ki.make_full(wl)
    shared = {"w1": full["sh1"], "w3": full["sh3"], "w2": full["sh2"]} if wl.S else None
    return h, Wr, bias, experts, full, shared


def _full_oracle(wl, h, Wr, bias, experts, full, shared, route=None):
    c_route = oracle.cfg(**dict(wl.config_kwargs(), d=wl.hidden))
    idx, w, gap = route if route is not None else oracle.route(c_route, h, Wr, bias)
    out = oracle.forward_full(oracle.cfg(**wl.config_kwargs()), wl.hidden, wl.latent_norm,
                              wl.rms_eps, h, idx, w, full["down"], experts, full["gain"],
                              full["up"], shared)
    return out, idx, w, gap


def brute_force_full(wl, h, Wr, bias, experts, full, shared):
    """Independent dense fp64 restatement of the block's six steps: float32 router
    scores on the full-width token, full-sort top-k, dense decoded weights, numpy
    tanh/exp, the RMSNorm of the weighted sum written out, fp64 throughout."""
    T, k = wl.T, wl.k
    hd = dense_bf16(h)
    logit = (hd @ dense_bf16(Wr).T).astype(np.float32)
    sc = (np.float32(1) / (np.float32(1) + np.exp(-logit))).astype(np.float32)
    ch = sc + (bias if bias is not None else np.float32(0))
    b1, b2 = wl.situ_b1, wl.situ_b2

    def situ(g, u):
        return b1 * np.tanh(g / b1) / (1.0 + np.exp(-g)) * (b2 * np.tanh(u / b2))

    Wd, Wu = dense_bf16(full["down"]), dense_bf16(full["up"])
    dense = {e: tuple(dense_mxfp4(q[f"{m}_packed"], q[f"{m}_scale"]) for m in ("w1", "w3", "w2"))
             for e, q in experts.items()}
    out = np.zeros((T, wl.hidden))
    idx_all = np.zeros((T, k), dtype=np.int64)
    for t in range(T):
        sel, _ = lexsort_topk(ch[t], k)
        idx_all[t] = sel
        wsel = sc[t, sel].astype(np.float32)
        if wl.renorm:
            s = np.float32(0)
            for v in wsel:
                s = np.float32(s + v)
            if s > 0:
                wsel = (wsel / s).astype(np.float32)
        wsel = (wsel * np.float32(wl.routed_scale)).astype(np.float32)
        z = Wd @ hd[t]
        a = np.zeros(wl.d)
        for e, wt in zip(sel, wsel):
            W1, W3, W2 = dense[e]
            a += float(wt) * (W2 @ situ(W1 @ z, W3 @ z))
        if wl.latent_norm:
            a = a / np.sqrt(np.mean(a * a) + wl.rms_eps) * full["gain"].astype(np.float64)
        out[t] = Wu @ a
        if shared is not None:
            S1, S3, S2 = (dense_bf16(shared[m]) for m in ("w1", "w3", "w2"))
            out[t] += S2 @ situ(S1 @ hd[t], S3 @ hd[t])
    return out, idx_all


FULL = ki.WORKLOADS["full_tiny"]


@pytest.mark.parametrize("wl", [
    FULL,
    FULL.with_(name="full_no_norm", latent_norm=0, seed=31),
    FULL.with_(name="full_no_shared", S=0, seed=32),
    FULL.with_(name="full_two_shared", S=2, seed=33, T=3),
    FULL.with_(name="full_bias", zipf_bias=True, E=12, k=3, seed=34),
    FULL.with_(name="full_wide_latent", d=256, hidden=128, seed=35, T=2),
], ids=lambda w: w.name)
def test_full_block_matches_brute_force(wl):
    case = _full_case(wl)
    out, idx, w, gap = _full_oracle(wl, *case)
    ref, ref_idx = brute_force_full(wl, *case)
    for t in range(wl.T):
        if gap[t] >= 1e-6:
            assert list(idx[t]) == list(ref_idx[t])
    assert np.max(np.abs(out - ref)) <= 1e-6 * np.max(np.abs(ref))


def test_full_block_reduces_to_latent_layer():
    """Identity down and up projections, no norm, and the shared experts' fused
    weights stacked from the latent layer's: the block is the latent layer."""
    wl = FULL.with_(name="full_identity", hidden=128, d=128, S=2, latent_norm=0, seed=36)
    h, Wr, bias, experts, full, _ = _full_case(wl)
    eye = np.where(np.eye(wl.d, dtype=bool), np.uint16(0x3F80), np.uint16(0))   # bf16 1.0
    full = dict(full, down=eye, up=eye.copy())
    sh = ki.make_shared(wl)                                  # [S,f,d], [S,d,f]
    fused = {"w1": sh["w1"].reshape(wl.S * wl.f, wl.d), "w3": sh["w3"].reshape(wl.S * wl.f, wl.d),
             "w2": np.ascontiguousarray(np.concatenate(list(sh["w2"]), axis=1))}
    out, idx, w, _ = _full_oracle(wl, h, Wr, bias, experts, full, fused)
    lat = oracle.forward(oracle.cfg(**wl.config_kwargs()), h, idx, w, experts, sh)
    assert np.max(np.abs(out - lat)) <= 1e-6 * np.max(np.abs(lat))
    # the identity case still routes on the full-width token: same scores as the layer's router
    idx_l, w_l, _ = oracle.route(oracle.cfg(**wl.config_kwargs()), h, Wr, bias)
    np.testing.assert_array_equal(idx, idx_l)


def test_full_block_norms_the_aggregate_not_each_expert():
    """Doubling every expert's down weights (scale bytes + 1) leaves the normed block
    unchanged; doubling ONE chosen expert's changes it, which a per-expert norm would
    not; without the norm, doubling all changes the routed part."""
    wl = FULL.with_(name="full_norm", S=0, seed=37, T=3, rms_eps=1e-12)   # eps out of the way
    h, Wr, bias, experts, full, shared = _full_case(wl)
    base, idx, w, gap = _full_oracle(wl, h, Wr, bias, experts, full, shared)
    route = (idx, w, gap)

    def doubled(which):
        return {e: (dict(q, w2_scale=q["w2_scale"] + 1) if e in which else q) for e, q in experts.items()}

    scale = np.max(np.abs(base))
    all2 = _full_oracle(wl, h, Wr, bias, doubled(set(experts)), full, shared, route)[0]
    assert np.max(np.abs(all2 - base)) <= 1e-6 * scale
    one2 = _full_oracle(wl, h, Wr, bias, doubled({int(idx[0, 0])}), full, shared, route)[0]
    assert np.max(np.abs(one2[0] - base[0])) > 1e-2 * scale
    raw = wl.with_(latent_norm=0)
    r1 = _full_oracle(raw, h, Wr, bias, experts, full, shared, route)[0]
    r2 = _full_oracle(raw, h, Wr, bias, doubled(set(experts)), full, shared, route)[0]
    np.testing.assert_allclose(r2, 2.0 * r1, rtol=1e-9, atol=1e-9 * np.max(np.abs(r1)))

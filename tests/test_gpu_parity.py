"""GPU parity: every call of the C ABI against the CPU oracle on the same seeded inputs.

Router: the device's exact scores within SCORE_ULPS ulps of the oracle's; its selection
and weights bit-exact against the oracle's selection step on those scores; indices,
offsets and perm bit-exact against the oracle's own routing except on tokens whose
k-th and (k+1)-th oracle choice scores differ by less than NEAR_TIE = 1e-6 without being
equal (counted, checked for validity).  Outputs: rel-L2 <= 5e-3 and max error <=
2e-2 max|ref|.
"""
import numpy as np
import pytest

import k3moe_inputs as ki
import oracle
from gpu_util import (NEAR_TIE, SCORE_ULPS, assert_out_close, ocfg, oracle_experts,
                      oracle_forward_expert_major, ulp32)

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def k3():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_moe_expert_k3moe_gb300 import build as kbuild
    kbuild.build()
    import sparse_moe_expert_k3moe_gb300 as k3
    return k3


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def dev16(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda()


def host(t):
    return t.cpu().numpy()


def run_route(k3, layer, x_dev, T, rows=None):
    """idx, weight, offsets, perm from k3moe_route, plus the router's exact scores (sc, ch)
    from k3moe_router_scores for the token rows `rows` (all when None)."""
    layer.route(x_dev)
    xs = x_dev if rows is None else x_dev[torch.as_tensor(rows, device=x_dev.device)].contiguous()
    gsc, gch = layer.scores(xs)
    torch.cuda.synchronize()
    k = layer.cfg.top_k
    return (host(layer.idx[:T]), host(layer.weight[:T]), host(layer.offsets),
            host(layer.perm[:T * k]), host(gsc), host(gch))


def check_route(w, x, gidx, gw, goff, gperm, gsc, gch, rows=None):
    """(1) The device's exact scores (for `rows`, all tokens when None) against the
    oracle's, within SCORE_ULPS ulps.  (2) The device's selection and weights bit-exact
    against the oracle's selection step run on those scores.  (3) Against the oracle's own
    routing, every token: the indices in rank order and the weights (to a few ulps) where
    the oracle's k-th and (k+1)-th choice scores are equal (an exact tie, decided by the
    lower index on both sides) or differ by at least NEAR_TIE; below that a boundary
    near-tie, checked for validity; two adjacent chosen scores closer than NEAR_TIE but not
    equal make an order near-tie (the set compared exactly).  Offsets depend only on the
    sets; perm is checked exactly against the oracle's counting sort of the device's
    indices, and against the oracle's own when no near-tie touches it."""
    c = ocfg(w)
    wr = ki.make_router(w)
    oidx, ow, gap, sc, ch = oracle.route(c, x, wr, ki.make_bias(w), want_scores=True)
    k = w.k
    rr = np.arange(w.T) if rows is None else np.asarray(rows)
    osc, och_r = sc[rr].astype(np.float64), ch[rr].astype(np.float64)
    usc = np.abs(gsc.astype(np.float64) - osc) / ulp32(osc)
    ech = np.abs(gch.astype(np.float64) - och_r)
    print(f"[{w.name}] scores of {len(rr)} tokens: {int((usc > 0).sum())} of {usc.size} differ, "
          f"max {usc.max():.0f} ulp")
    assert np.all(usc <= SCORE_ULPS)
    assert np.all(ech <= SCORE_ULPS * ulp32(osc) + ulp32(och_r))
    sidx, sw, _ = oracle.select(c, gsc, gch)
    np.testing.assert_array_equal(gidx[rr], sidx)
    np.testing.assert_array_equal(gw[rr], sw)
    och = np.take_along_axis(ch, oidx.astype(np.int64), axis=1)
    inner = (np.min(np.where(och[:, :-1] > och[:, 1:], och[:, :-1] - och[:, 1:], np.inf), axis=1)
             if k > 1 else np.full(w.T, np.inf, dtype=np.float32))
    boundary = (gap > 0) & (gap < NEAR_TIE)
    order = ~boundary & (inner < NEAR_TIE)
    exact = ~boundary & ~order
    np.testing.assert_array_equal(gidx[exact], oidx[exact])
    np.testing.assert_allclose(gw[exact], ow[exact], rtol=1e-6, atol=0)
    for t in np.nonzero(order)[0]:
        assert sorted(gidx[t].tolist()) == sorted(oidx[t].tolist())
        gmap = dict(zip(gidx[t].tolist(), gw[t].tolist()))
        omap = dict(zip(oidx[t].tolist(), ow[t].tolist()))
        for e in omap:
            assert abs(gmap[e] - omap[e]) <= 1e-6 * abs(omap[e])
    for t in np.nonzero(boundary)[0]:
        assert len(set(gidx[t].tolist())) == k and gidx[t].min() >= 0 and gidx[t].max() < w.E
    # the map is a pure function of idx: exact against the oracle's counting sort of the GPU's idx
    ooff, operm = oracle.perm(gidx, w.E)
    np.testing.assert_array_equal(goff, ooff)
    np.testing.assert_array_equal(gperm, operm)
    if not boundary.any():
        np.testing.assert_array_equal(goff, oracle.perm(oidx, w.E)[0])
        if not order.any():
            np.testing.assert_array_equal(gperm, oracle.perm(oidx, w.E)[1])
    print(f"[{w.name}] tokens={w.T} boundary_near_ties={int(boundary.sum())} "
          f"order_near_ties={int(order.sum())} exact_tie_tokens={int((gap == 0).sum())} "
          f"(compared exactly)")
    return oidx, ow, gap


# ----------------------------------------------------------------------------- pack / unpack

def test_pack_roundtrip_every_code_and_scale(k3):
    w = ki.Workload("rt", T=1, d=256, f=128, E=3, k=1, S=0, exp_lo=-8, exp_hi=-4, seed=5)
    cfg = k3.k3moe_config(**w.config_kwargs())
    blk = ki.make_experts_block(w, 0, w.E)
    # every scale byte 0..255 and every code at every nibble position appears
    for name in ("w1_scale", "w3_scale", "w2_scale"):
        flat = blk[name].reshape(-1)
        flat[:] = np.arange(flat.size) % 256
    blk["w1_packed"].reshape(-1)[:256] = np.arange(256, dtype=np.uint8)
    table = torch.empty(k3.k3moe_packed_bytes(cfg), dtype=torch.uint8, device="cuda")
    d_in = {kname: dev(v) for kname, v in blk.items()}
    ws = torch.zeros(k3.k3moe_workspace_bytes(cfg, 1), dtype=torch.uint8, device="cuda")
    k3.k3moe_pack_mxfp4(cfg, 0, w.E, *(d_in[n] for n in ki.EXPERT_TENSORS), table, ws=ws)
    d_out = {kname: torch.zeros_like(v) for kname, v in d_in.items()}
    k3.k3moe_unpack_mxfp4(cfg, 0, w.E, table, *(d_out[n] for n in ki.EXPERT_TENSORS))
    torch.cuda.synchronize()
    for n in ki.EXPERT_TENSORS:
        np.testing.assert_array_equal(host(d_out[n]), blk[n])
    rc, code = k3.k3moe_device_status(ws)
    assert rc == 0 and code & k3.DEV_NAN_SCALE      # byte 255 present: warning, not error
    # per expert: the tiles, the trailer, and the block-scaled section (the same codes and
    # scales again, row-major and in scale blocks)
    assert table.numel() == w.E * (2 * w.expert_bytes + 1024)


def test_pack_records_block_scale_maxima(k3):
    """The table's trailer: per expert, matrix and 128-row block, the largest scale byte
    other than 255; and in its last word a flag for a scale byte 0 or 255 in the expert."""
    w = ki.Workload("trail", T=1, d=256, f=256, E=4, k=1, S=0, exp_lo=-9, exp_hi=-1, seed=9)
    cfg = k3.k3moe_config(**w.config_kwargs())
    blk = ki.make_experts_block(w, 0, w.E)
    blk["w1_scale"][1, 5, 3] = 255                 # a NaN byte never counts as the maximum
    blk["w2_scale"][0, 130, 0] = 140
    blk["w3_scale"][2, 200, 7] = 0                 # the subnormal byte also sets the flag
    table = torch.zeros(k3.k3moe_packed_bytes(cfg), dtype=torch.uint8, device="cuda")
    k3.k3moe_pack_mxfp4(cfg, 0, w.E, *(dev(blk[n]) for n in ki.EXPERT_TENSORS), table)
    torch.cuda.synchronize()
    tb = host(table)
    trailer = tb[w.E * w.expert_bytes:w.E * (w.expert_bytes + 1024)].view(np.uint32).reshape(w.E, 256)
    for e in range(w.E):
        col = 0
        for m in ("w1", "w3", "w2"):
            sc = blk[f"{m}_scale"][e]
            for rb in range(sc.shape[0] // 128):
                blkv = sc[rb * 128:(rb + 1) * 128]
                assert trailer[e, col] == blkv[blkv != 255].max()
                col += 1
        special = any(((blk[f"{m}_scale"][e] == 0) | (blk[f"{m}_scale"][e] == 255)).any()
                      for m in ("w1", "w3", "w2"))
        assert (trailer[e, 255] != 0) == special
        assert not trailer[e, col:255].any()
    assert [trailer[e, 255] != 0 for e in range(w.E)] == [False, True, True, False]


def test_pack_roundtrip_full_shape(k3):
    w = ki.WORKLOADS["decode_t1"]
    cfg = k3.k3moe_config(**w.config_kwargs())
    cfg_small = k3.k3moe_config(**w.with_(E=3, k=1).config_kwargs())
    blk = ki.make_experts_block(w, 10, 3)
    table = torch.empty(k3.k3moe_packed_bytes(cfg_small), dtype=torch.uint8, device="cuda")
    d_in = {kname: dev(v) for kname, v in blk.items()}
    k3.k3moe_pack_mxfp4(cfg_small, 0, 3, *(d_in[n] for n in ki.EXPERT_TENSORS), table)
    d_out = {kname: torch.zeros_like(v) for kname, v in d_in.items()}
    k3.k3moe_unpack_mxfp4(cfg_small, 0, 3, table, *(d_out[n] for n in ki.EXPERT_TENSORS))
    torch.cuda.synchronize()
    for n in ki.EXPERT_TENSORS:
        np.testing.assert_array_equal(host(d_out[n]), blk[n])
    assert k3.k3moe_packed_bytes(cfg) == 896 * (2 * 17547264 + 1024)


# ----------------------------------------------------------------------------- small layers, all outputs

MICRO = ki.Workload("micro", T=37, d=384, f=256, E=16, k=4, S=2, exp_lo=-7, exp_hi=-3, seed=40)
SMALL_CASES = [
    ki.WORKLOADS["tiny"],
    MICRO,
    MICRO.with_(name="micro_bias", zipf_bias=True, seed=41, T=70),        # two chunks
    MICRO.with_(name="micro_k_eq_E", E=8, k=8, seed=42, T=9),
    MICRO.with_(name="micro_one_expert", E=1, k=1, seed=43, T=5),
    MICRO.with_(name="micro_no_renorm", renorm=0, routed_scale=0.75, seed=44),
    MICRO.with_(name="micro_no_shared", S=0, seed=45, T=130),             # ragged third chunk
    MICRO.with_(name="micro_wide", d=1024, f=640, E=40, k=16, S=1, seed=46, T=23),
    # one token: the shared gate/up items are cut into K parts (d = 512: 4 tiles of K)
    MICRO.with_(name="micro_t1_split", d=512, f=256, E=32, k=4, S=2, seed=47, T=1),
]


# Cases on the tensor-core path (average >= 8 tokens per expert and T >= 32): several
# 256-token tiles per expert with ragged tails, skewed routing, several row blocks.
GEMM_CASES = [
    ki.Workload("gemm_multi_tile", T=1100, d=256, f=256, E=8, k=2, S=1, exp_lo=-7, exp_hi=-3, seed=70),
    ki.Workload("gemm_bias", T=300, d=384, f=256, E=12, k=3, S=2, exp_lo=-9, exp_hi=-5, seed=71,
                zipf_bias=True),
    ki.Workload("gemm_wide", T=64, d=1024, f=640, E=40, k=16, S=1, exp_lo=-10, exp_hi=-6, seed=72),
    ki.Workload("gemm_outliers", T=520, d=256, f=384, E=16, k=4, S=2, exp_lo=-8, exp_hi=-4, seed=73,
                outlier_frac=0.05),
    # router scores on the tensor cores (T >= 32, E >= 128): a ragged second block of 128
    # experts and a ragged last token tile (300 = 256 + 44)
    ki.Workload("gemm_router_ragged", T=300, d=384, f=128, E=200, k=8, S=1, exp_lo=-8, exp_hi=-4,
                seed=74, zipf_bias=True),
]
# the decode path with the tensor-core router (T >= 32, fewer than 8 tokens per expert)
SMALL_CASES.append(ki.Workload("decode_router_tc", T=40, d=256, f=128, E=160, k=4, S=1, exp_lo=-8,
                               exp_hi=-4, seed=75))


@pytest.mark.parametrize("w", SMALL_CASES + GEMM_CASES, ids=lambda w: w.name)
def test_small_layer_parity(k3, w):
    from k3moe_inputs.device import build_layer
    layer = build_layer(w)
    x = ki.make_x(w)
    xd = dev16(x)
    gidx, gw, goff, gperm, gsc, gch = run_route(k3, layer, xd, w.T)
    check_route(w, x, gidx, gw, goff, gperm, gsc, gch)
    out = torch.empty((w.T, w.d), dtype=torch.float32, device="cuda")
    layer.forward(xd, out)
    rc, code = k3.k3moe_device_status(layer.ws)
    assert rc == 0 and code == 0
    ref = oracle.forward(ocfg(w), x, gidx, gw, oracle_experts(w, range(w.E)),
                         ki.make_shared(w) if w.S else None)
    rel, mx = assert_out_close(host(out), ref, w.name)
    print(f"[{w.name}] rel_l2={rel:.2e} max_rel={mx:.2e}")


def test_alternating_shapes(k3):
    """Calls whose kernels need different shared-memory sizes, large -> small -> large:
    a launch setting left by a smaller call must not break a later larger one."""
    from k3moe_inputs.device import build_layer
    cases = [MICRO.with_(name="alt_big", T=11, seed=49),
             ki.Workload("alt_small", T=12, d=256, f=128, E=8, k=2, S=1, exp_lo=-8, exp_hi=-4, seed=50)]
    layers = [(w, build_layer(w)) for w in cases]
    for w, layer in layers + layers:
        x = ki.make_x(w)
        xd = dev16(x)
        layer.route(xd)
        out = torch.empty((w.T, w.d), dtype=torch.float32, device="cuda")
        layer.forward(xd, out)
        rc, code = k3.k3moe_device_status(layer.ws)
        assert rc == 0 and code == 0
        ref = oracle.forward(ocfg(w), x, host(layer.idx), host(layer.weight),
                             oracle_experts(w, range(w.E)), ki.make_shared(w))
        assert_out_close(host(out), ref, w.name)


def test_workspace_reuse_across_paths(k3):
    """One workspace for calls whose T takes different paths: the tensor-core GEMMs
    (T = 64, 40), the streamed mat-vecs whose down items start per unit (T = 1, 2, 3;
    at T = 1 with the shared expert's gate/up split in K), and those whose down waits for
    all of gate/up (T = 4).  The counters the kernels keep at zero between calls sit in a
    block at a fixed offset, so no buffer of a call with another T overwrites them, and
    each schedule leaves them at zero for the next."""
    from k3moe_inputs.device import build_layer
    big = ki.Workload("reuse", T=64, d=256, f=256, E=8, k=2, S=1, exp_lo=-8, exp_hi=-4, seed=87)
    layer = build_layer(big)
    for T in (64, 1, 64, 1, 4, 2, 40, 3, 1, 4, 1):
        w = big.with_(name=f"reuse_T{T}", T=T)
        x = ki.make_x(w)
        xd = dev16(x)
        layer.route(xd)
        out = torch.full((T, w.d), float("nan"), dtype=torch.float32, device="cuda")
        layer.forward(xd, out)
        rc, code = k3.k3moe_device_status(layer.ws)
        assert rc == 0 and code == 0
        ref = oracle.forward(ocfg(w), x, host(layer.idx)[:T], host(layer.weight)[:T],
                             oracle_experts(w, range(w.E)), ki.make_shared(w))
        assert_out_close(host(out), ref, w.name)


@pytest.mark.parametrize("T,bitwise", [(1, True), (4, True), (40, False)])
def test_graph_replay(k3, T, bitwise):
    """route + forward captured as one CUDA graph: a replay gives the eager call's routing
    and output, and a replay on new tokens copied into the same input buffer matches the
    oracle.  T = 1 and 4 take the streamed mat-vecs, whose combine is a fixed-order
    gather, so the output repeats bit for bit; T = 40 takes the tensor-core path, whose
    down epilogue adds into the output with fp32 atomics (order varies run to run)."""
    from k3moe_inputs.device import build_layer
    w = MICRO.with_(name=f"graph_t{T}", T=T, seed=60 + T)
    layer = build_layer(w)
    xd = dev16(ki.make_x(w))
    out_eager = torch.empty((T, w.d), dtype=torch.float32, device="cuda")
    layer(xd, out_eager)
    idx_eager = host(layer.idx).copy()
    out = torch.zeros_like(out_eager)
    graph = layer.capture(xd, out)
    out.zero_()
    layer.idx.zero_()
    graph.replay()
    torch.cuda.synchronize()
    np.testing.assert_array_equal(host(layer.idx), idx_eager)
    if bitwise:
        np.testing.assert_array_equal(host(out), host(out_eager))
    else:
        ref_scale = float(np.abs(host(out_eager)).max())
        np.testing.assert_allclose(host(out), host(out_eager), rtol=1e-5, atol=1e-6 * ref_scale)
    x2 = ki.make_x(w.with_(seed=w.seed + 1000))
    xd.copy_(dev16(x2))
    graph.replay()
    torch.cuda.synchronize()
    rc, code = k3.k3moe_device_status(layer.ws)
    assert rc == 0 and code == 0
    assert not np.array_equal(host(layer.idx), idx_eager)
    ref = oracle.forward(ocfg(w), x2, host(layer.idx), host(layer.weight),
                         oracle_experts(w, range(w.E)), ki.make_shared(w))
    assert_out_close(host(out), ref, w.name + " replayed on new tokens")


def test_forward_with_injected_oracle_routing(k3):
    """Routing computed by the oracle, uploaded, consumed by k3moe_forward."""
    from k3moe_inputs.device import build_layer
    w = MICRO.with_(name="inject", seed=47)
    layer = build_layer(w)
    x = ki.make_x(w)
    oidx, ow, _ = oracle.route(ocfg(w), x, ki.make_router(w), ki.make_bias(w))
    ooff, operm = oracle.perm(oidx, w.E)
    routing = (dev(oidx), dev(ow), dev(ooff), dev(operm))
    out = torch.empty((w.T, w.d), dtype=torch.float32, device="cuda")
    layer.forward(dev16(x), out, routing=routing)
    ref = oracle.forward(ocfg(w), x, oidx, ow, oracle_experts(w, range(w.E)), ki.make_shared(w))
    assert_out_close(host(out), ref, "injected")


def test_zero_tokens(k3):
    from k3moe_inputs.device import build_layer
    w = ki.WORKLOADS["tiny"]
    layer = build_layer(w)
    layer.offsets.fill_(7)
    x0 = torch.empty((0, w.d), dtype=torch.int16, device="cuda")
    layer.route(x0)
    torch.cuda.synchronize()
    assert host(layer.offsets).tolist() == [0] * (w.E + 1)
    out = torch.empty((0, w.d), dtype=torch.float32, device="cuda")
    layer.forward(x0, out)


def test_bad_routing_sets_status_without_fault(k3):
    from k3moe_inputs.device import build_layer
    w = ki.WORKLOADS["tiny"]
    layer = build_layer(w)
    x = dev16(ki.make_x(w))
    out = torch.empty((w.T, w.d), dtype=torch.float32, device="cuda")
    layer.route(x)
    good = (layer.idx.clone(), layer.weight.clone(), layer.offsets.clone(), layer.perm.clone())
    # offsets that do not describe the routing
    off = good[2].clone()
    off[3] += 1
    layer.forward(x, out, routing=(good[0], good[1], off, good[3]))
    rc, code = k3.k3moe_device_status(layer.ws)
    assert rc == 6 and code & k3.DEV_BAD_OFFSETS
    assert torch.all(out == 0)
    # an expert index out of range
    bad_idx = good[0].clone()
    bad_idx[0, 0] = w.E + 5
    layer.forward(x, out, routing=(bad_idx, good[1], good[2], good[3]))
    rc, code = k3.k3moe_device_status(layer.ws)
    assert rc == 6 and code & k3.DEV_BAD_INDEX
    # the next valid call is clean again
    layer.forward(x, out, routing=good)
    rc, code = k3.k3moe_device_status(layer.ws)
    assert rc == 0 and code == 0
    assert torch.isfinite(out).all() and out.abs().max() > 0


@pytest.mark.parametrize("T", [1, 11, 40])
def test_nan_scale_groups_read_as_zero(k3, T):
    """Scale byte 255 reads as zero and byte 0 as 2^-127; experts holding either take
    the exact scale path of the streamed mat-vecs, the others the fast one, in the same
    launch; T = 40 takes the tensor-core path."""
    w = MICRO.with_(name="nanscale", seed=48, T=T)
    cfg = k3.k3moe_config(**w.config_kwargs())
    from sparse_moe_expert_k3moe_gb300 import MoELayer
    from k3moe_inputs.device import to_device_u16
    layer = MoELayer(cfg, w.T)
    layer.w_router = to_device_u16(ki.make_router(w), "cuda")
    sh = ki.make_shared(w)
    layer.sh_w1, layer.sh_w3, layer.sh_w2 = (to_device_u16(sh[m], "cuda") for m in ("w1", "w3", "w2"))
    experts = {e: ki.make_expert(w, e) for e in range(w.E)}
    for e in range(w.E):
        for name in ("w1_scale", "w3_scale", "w2_scale"):
            if e % 3 == 0:
                experts[e][name][::7, 1] = 255
            elif e % 3 == 1:
                experts[e][name][::11, 2] = 0
    blk = {n: np.stack([experts[e][n] for e in range(w.E)]) for n in ki.EXPERT_TENSORS}
    layer.pack_experts(0, w.E, *(dev(blk[n]) for n in ki.EXPERT_TENSORS))
    x = ki.make_x(w)
    xd = dev16(x)
    layer.route(xd)
    out = torch.empty((w.T, w.d), dtype=torch.float32, device="cuda")
    layer.forward(xd, out)
    rc, code = k3.k3moe_device_status(layer.ws)
    assert rc == 0 and code == k3.DEV_NAN_SCALE
    gidx, gw = host(layer.idx), host(layer.weight)
    ref = oracle.forward(ocfg(w), x, gidx, gw, experts, sh)
    assert_out_close(host(out), ref, "nan-scale")


def test_launch_count_and_timing(k3):
    from k3moe_inputs.device import build_layer
    w = ki.WORKLOADS["tiny"]
    layer = build_layer(w)
    x = dev16(ki.make_x(w))
    out = torch.empty((w.T, w.d), dtype=torch.float32, device="cuda")
    n0 = k3.k3moe_launch_count()
    k3.k3moe_timing_reset()
    k3.k3moe_timing_enable(True)
    layer(x, out)
    torch.cuda.synchronize()
    k3.k3moe_timing_enable(False)
    tm = k3.k3moe_timing_read()
    assert k3.k3moe_launch_count() > n0
    assert sum(v[0] for v in tm.values()) == k3.k3moe_launch_count() - n0
    assert all(v[1] >= 0 for v in tm.values())


# ----------------------------------------------------------------------------- full-size workloads

@pytest.fixture(scope="module")
def full_layers():
    cache = {}
    yield cache
    cache.clear()


def full_layer(cache, name):
    from k3moe_inputs.device import build_layer
    if name not in cache:
        cache.clear()
        torch.cuda.empty_cache()
        w = ki.WORKLOADS[name]
        cache[name] = (w, build_layer(w))
    return cache[name]


@pytest.mark.parametrize("name", ["decode_t1", "decode_t64", "prefill_t4096", "prefill_t16k"])
def test_full_route_parity(k3, full_layers, name):
    """Every token's routing against the oracle's.  The device's exact scores (scored pair
    by pair, far slower than the routing) are taken for every token up to T = 4096, and at
    T = 16384 for 2048 tokens: every outlier row and a seeded sample of the rest."""
    w, layer = full_layer(full_layers, name)
    x = ki.make_x(w)
    rows = None
    if w.T > 4096:
        rng = np.random.default_rng(w.seed)
        out_rows = set(int(r) for r in ki.outlier_rows(w))
        rest = np.array(sorted(set(range(w.T)) - out_rows))
        rows = sorted(out_rows | set(int(r) for r in rng.choice(rest, 2048 - len(out_rows), replace=False)))
    gidx, gw, goff, gperm, gsc, gch = run_route(k3, layer, dev16(x), w.T, rows)
    check_route(w, x, gidx, gw, goff, gperm, gsc, gch, rows)
    rc, code = k3.k3moe_device_status(layer.ws)
    assert rc == 0 and code == 0


@pytest.mark.parametrize("name,rows", [
    ("decode_t1", None),                   # every output
    ("decode_t64", None),                  # every output
    ("prefill_t4096", None),               # every output
    ("prefill_t16k", "tiles"),             # >= 1024 rows covering every expert's tiles
])
def test_full_forward_parity(k3, full_layers, name, rows):
    """The layer's output on the device's routing against the oracle's, element by element.
    Every row up to T = 4096 (the oracle expert by expert, one expert's weights at a time).
    At T = 16384: for every expert touched, the first and last token of its last (ragged)
    128-token tile and of its first tile; the first and last row; every outlier row; then
    a seeded sample of the rest up to 1024 rows."""
    w, layer = full_layer(full_layers, name)
    x = ki.make_x(w)
    xd = dev16(x)
    layer.route(xd)
    out = torch.empty((w.T, w.d), dtype=torch.float32, device="cuda")
    layer.forward(xd, out)
    rc, code = k3.k3moe_device_status(layer.ws)
    assert rc == 0 and code == 0
    gidx, gw = host(layer.idx[:w.T]), host(layer.weight[:w.T])
    if rows is None:
        sel = np.arange(w.T)
    else:
        goff = host(layer.offsets)
        gperm = host(layer.perm[:w.T * w.k])
        pick = {0, w.T - 1} | set(int(r) for r in ki.outlier_rows(w))
        for e in range(w.E):
            lo, hi = int(goff[e]), int(goff[e + 1])
            if hi == lo:
                continue
            last0 = lo + 128 * ((hi - lo - 1) // 128)
            for p in (lo, min(lo + 127, hi - 1), last0, hi - 1):
                pick.add(int(gperm[p]) // w.k)
        rng = np.random.default_rng(w.seed)
        rest = np.array(sorted(set(range(w.T)) - pick))
        if len(pick) < 1024:
            pick |= set(int(r) for r in rng.choice(rest, 1024 - len(pick), replace=False))
        sel = np.array(sorted(pick))
    ref = oracle_forward_expert_major(w, x, gidx, gw, sel)
    got = host(out)[sel]
    rel, mx = assert_out_close(got, ref, name)
    print(f"[{name}] rows={len(sel)} of {w.T} rel_l2={rel:.2e} max_rel={mx:.2e}")


# ----------------------------------------------------------------------------- full-width block

FULL_CASES = [
    ki.WORKLOADS["full_tiny"],                                                  # mat-vecs, S = 1
    ki.WORKLOADS["full_tiny"].with_(name="full_tiny_t1", T=1, seed=80),
    ki.WORKLOADS["full_tiny"].with_(name="full_tiny_gemm", T=40, seed=81),      # tensor-core path
    ki.WORKLOADS["full_tiny"].with_(name="full_tiny_raw", T=6, S=2, latent_norm=0, seed=82),
    ki.WORKLOADS["full_tiny"].with_(name="full_tiny_no_shared", T=5, S=0, seed=83),
    ki.Workload("full_mid", T=3, d=512, f=256, E=32, k=4, S=2, exp_lo=-9, exp_hi=-5, seed=84,
                hidden=1024, zipf_bias=True),
    # the dense projections over several token tiles with a ragged last one (256 + 44;
    # the gated shared projection in tiles of 128), K not split
    ki.Workload("full_tiles", T=300, d=256, f=256, E=16, k=4, S=2, exp_lo=-8, exp_hi=-4, seed=86,
                hidden=512),
]


@pytest.mark.parametrize("w", FULL_CASES, ids=lambda w: w.name)
def test_full_block_parity(k3, w):
    """k3moe_full_forward against the oracle's full-width block: routing on the
    full-width token bit-exact away from near-ties, offsets and perm exact, and the
    output within the layer's tolerance on the GPU's routing.  The block rounds z, the
    normed aggregate and the shared SiTU output to bf16 (the dense GEMMs' operand
    type), about 2^-9 relative each, which the tolerance covers."""
    from k3moe_inputs.device import build_block
    blk = build_block(w)
    h = ki.make_h(w)
    out = torch.full((w.T, w.hidden), float("nan"), dtype=torch.float32, device="cuda")
    blk.forward(dev16(h), out)
    rc, code = k3.k3moe_device_status(blk.ws)
    assert rc == 0 and code == 0
    Wr = ki.make_full_router(w)
    c_route = oracle.cfg(**dict(w.config_kwargs(), d=w.hidden))
    oidx, ow, gap = oracle.route(c_route, h, Wr, ki.make_bias(w))
    gidx, gw = host(blk.idx)[:w.T], host(blk.weight)[:w.T]
    for t in range(w.T):
        if not (0 < gap[t] < NEAR_TIE):
            np.testing.assert_array_equal(gidx[t], oidx[t])
            # weights: the same selection on scores equal to the oracle's within a few ulps
            np.testing.assert_allclose(gw[t], ow[t], rtol=1e-6, atol=0)
        else:
            assert len(set(gidx[t].tolist())) == w.k and gidx[t].min() >= 0 and gidx[t].max() < w.E
    offs, pm = oracle.perm(gidx, w.E)
    np.testing.assert_array_equal(host(blk.offsets), offs)
    np.testing.assert_array_equal(host(blk.perm)[:w.T * w.k], pm)
    full = ki.make_full(w)
    shared = {"w1": full["sh1"], "w3": full["sh3"], "w2": full["sh2"]} if w.S else None
    ref = oracle.forward_full(ocfg(w), w.hidden, w.latent_norm, w.rms_eps, h, gidx, gw, full["down"],
                              oracle_experts(w, gidx.ravel()), full["gain"], full["up"], shared)
    rel_l2, max_rel = assert_out_close(host(out), ref, w.name)
    print(f"[{w.name}] rel_l2={rel_l2:.2e} max_rel={max_rel:.2e}")
    # no tokens: the routing is left empty and nothing else is touched
    blk.offsets.fill_(7)
    blk.forward(dev16(h[:0]), out[:0])
    torch.cuda.synchronize()
    assert not host(blk.offsets).any()


def test_block_workspace_reuse_across_paths(k3):
    """One block workspace for T = 200 (latent experts on the GEMMs, dense projections
    split in K over token tiles), T = 40 (mat-vecs, split dense projections) and T = 1
    (row-streaming projections): the dense split-K counters and the layer's counters stay
    consistent from call to call."""
    from k3moe_inputs.device import build_block
    big = ki.Workload("full_reuse", T=200, d=512, f=256, E=32, k=4, S=2, exp_lo=-9, exp_hi=-5, seed=89,
                      hidden=1024)
    blk = build_block(big)
    for T in (200, 40, 200, 40, 1):
        w = big.with_(name=f"full_reuse_T{T}", T=T)
        h = ki.make_h(w)
        out = torch.full((T, w.hidden), float("nan"), dtype=torch.float32, device="cuda")
        blk.forward(dev16(h), out)
        rc, code = k3.k3moe_device_status(blk.ws)
        assert rc == 0 and code == 0
        gidx, gw = host(blk.idx)[:T], host(blk.weight)[:T]
        full = ki.make_full(w)
        shared = {"w1": full["sh1"], "w3": full["sh3"], "w2": full["sh2"]}
        ref = oracle.forward_full(ocfg(w), w.hidden, w.latent_norm, w.rms_eps, h, gidx, gw, full["down"],
                                  oracle_experts(w, gidx.ravel()), full["gain"], full["up"], shared)
        assert_out_close(host(out), ref, w.name)


def test_block_graph_replay(k3):
    """The full-width block (its dense projections included) captured as one CUDA graph:
    a replay repeats the eager call, and a replay on new tokens copied into the same
    input buffer matches the oracle's block."""
    from k3moe_inputs.device import build_block
    w = ki.WORKLOADS["full_tiny"].with_(name="full_graph", T=3, seed=85)
    blk = build_block(w)
    hd = dev16(ki.make_h(w))
    out_eager = torch.empty((w.T, w.hidden), dtype=torch.float32, device="cuda")
    blk(hd, out_eager)
    out = torch.zeros_like(out_eager)
    graph = blk.capture(hd, out)
    out.zero_()
    graph.replay()
    torch.cuda.synchronize()
    np.testing.assert_allclose(host(out), host(out_eager), rtol=1e-6,
                               atol=1e-6 * float(np.abs(host(out_eager)).max()))
    h2 = ki.make_h(w.with_(seed=w.seed + 1000))
    hd.copy_(dev16(h2))
    graph.replay()
    torch.cuda.synchronize()
    rc, code = k3.k3moe_device_status(blk.ws)
    assert rc == 0 and code == 0
    gidx, gw = host(blk.idx)[:w.T], host(blk.weight)[:w.T]
    full = ki.make_full(w)
    shared = {"w1": full["sh1"], "w3": full["sh3"], "w2": full["sh2"]}
    ref = oracle.forward_full(ocfg(w), w.hidden, w.latent_norm, w.rms_eps, h2, gidx, gw, full["down"],
                              oracle_experts(w, gidx.ravel()), full["gain"], full["up"], shared)
    assert_out_close(host(out), ref, w.name + " replayed on new tokens")

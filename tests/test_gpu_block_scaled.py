"""GPU parity of the block-scaled prefill GEMM (k3moe_set_prefill_gemm(2): the routed
experts' gate/up projection on tcgen05 kind::mxf8f6f4 MMAs, the E2M1 codes and E8M0
scales of the packed table read by the tensor core, the tokens as two e4m3 planes with
their own E8M0 scales per 32 elements).

Same bar as the other output tests: rel-L2 <= 5e-3 and max error <= 2e-2 max|ref|
against the oracle's forward on the device's routing.  The cases span several 128-token
tiles with ragged tails, skewed routing, K of 2 to 8 stages, outlier token rows (x8)
whose 32-element blocks take larger scales, no shared experts, scale bytes 0 and 255,
and the K3 shape at T = 4096.
"""
import numpy as np
import pytest

import k3moe_inputs as ki
import oracle
from gpu_util import assert_out_close, ocfg, oracle_experts, oracle_forward_expert_major

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def k3():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_moe_expert_k3moe_gb300 import build as kbuild
    kbuild.build()
    import sparse_moe_expert_k3moe_gb300 as k3
    yield k3
    k3.k3moe_set_prefill_gemm(k3.PREFILL_GEMM_DEFAULT)


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def dev16(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda()


def host(t):
    return t.cpu().numpy()


CASES = [
    ki.Workload("mx_multi_tile", T=1100, d=256, f=256, E=8, k=2, S=1, exp_lo=-7, exp_hi=-3, seed=90),
    ki.Workload("mx_bias", T=300, d=384, f=256, E=12, k=3, S=2, exp_lo=-9, exp_hi=-5, seed=91,
                zipf_bias=True),
    ki.Workload("mx_wide", T=64, d=1024, f=640, E=40, k=16, S=1, exp_lo=-10, exp_hi=-6, seed=92),
    ki.Workload("mx_outliers", T=520, d=256, f=384, E=16, k=4, S=2, exp_lo=-8, exp_hi=-4, seed=93,
                outlier_frac=0.05),
    ki.Workload("mx_no_shared", T=400, d=512, f=256, E=16, k=4, S=0, exp_lo=-8, exp_hi=-4, seed=94),
    ki.Workload("mx_router_ragged", T=300, d=384, f=128, E=200, k=8, S=1, exp_lo=-8, exp_hi=-4,
                seed=95, zipf_bias=True),
]


def run_both(k3, layer, xd, T):
    """The layer's output with the f16 GEMM and with the block-scaled GEMM, on one routing."""
    layer.route(xd)
    outs = {}
    for v in (k3.PREFILL_GEMM_F16, k3.PREFILL_GEMM_BLOCK_SCALED):
        k3.k3moe_set_prefill_gemm(v)
        out = torch.empty((T, layer.cfg.d), dtype=torch.float32, device="cuda")
        layer.forward(xd, out)
        rc, code = k3.k3moe_device_status(layer.ws)
        assert rc == 0 and code == 0, (v, rc, code)
        outs[v] = host(out)
    k3.k3moe_set_prefill_gemm(k3.PREFILL_GEMM_DEFAULT)
    return outs[k3.PREFILL_GEMM_F16], outs[k3.PREFILL_GEMM_BLOCK_SCALED]


def test_pack_writes_block_scaled_section(k3):
    """The packed table's block-scaled section, which the block-scaled GEMM loads by
    tensor map: the codes row-major exactly as the checkpoint holds them, and every scale
    byte in its 512-byte block (rows 128 rb.., K groups of 128 kc..: row r's 4 bytes at
    16 (r % 32) + 4 (r / 32)), byte 255 stored as 0."""
    w = ki.Workload("mx_pack", T=1, d=384, f=256, E=3, k=1, S=0, exp_lo=-9, exp_hi=-1, seed=97)
    cfg = k3.k3moe_config(**w.config_kwargs())
    blk = ki.make_experts_block(w, 0, w.E)
    blk["w1_scale"][1, 5, 3] = 255
    blk["w2_scale"][2, 7, 1] = 0
    blk["w3_scale"][0, 130, 11] = 255
    table = torch.zeros(k3.k3moe_packed_bytes(cfg), dtype=torch.uint8, device="cuda")
    k3.k3moe_pack_mxfp4(cfg, 0, w.E, *(dev(blk[n]) for n in ki.EXPERT_TENSORS), table)
    torch.cuda.synchronize()
    tb = host(table)
    E, d, f = w.E, w.d, w.f
    o = E * (w.expert_bytes + 1024)
    for name, rows, cols in (("w1", f, d), ("w3", f, d), ("w2", d, f)):
        n = E * rows * cols // 2
        np.testing.assert_array_equal(tb[o:o + n].reshape(E, rows, cols // 2), blk[name + "_packed"])
        o += n

    def blocks(sc, rows, cols):
        s = np.where(sc == 255, 0, sc).astype(np.uint8)
        s = s.reshape(E, rows // 128, 4, 32, cols // 128, 4)         # e, rb, j, i, kc, kb (r = i + 32 j)
        return s.transpose(0, 1, 4, 3, 2, 5).reshape(E, rows // 128, cols // 128, 512)
    n = E * (f // 128) * (d // 128) * 1024
    gu = tb[o:o + n].reshape(E, f // 128, d // 128, 2, 512)
    np.testing.assert_array_equal(gu[:, :, :, 0], blocks(blk["w1_scale"], f, d))
    np.testing.assert_array_equal(gu[:, :, :, 1], blocks(blk["w3_scale"], f, d))
    o += n
    n = E * (d // 128) * (f // 128) * 512
    np.testing.assert_array_equal(tb[o:o + n].reshape(E, d // 128, f // 128, 512), blocks(blk["w2_scale"], d, f))
    assert o + n == tb.size


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_block_scaled_gemm_parity(k3, w):
    from k3moe_inputs.device import build_layer
    assert w.T >= 32 and w.T * w.k >= 8 * w.E          # the tensor-core path
    layer = build_layer(w)
    x = ki.make_x(w)
    xd = dev16(x)
    f16, mx = run_both(k3, layer, xd, w.T)
    gidx, gw = host(layer.idx[:w.T]), host(layer.weight[:w.T])
    ref = oracle.forward(ocfg(w), x, gidx, gw, oracle_experts(w, range(w.E)),
                         ki.make_shared(w) if w.S else None)
    rel, mxe = assert_out_close(mx, ref, w.name + " block-scaled")
    rel16, _ = assert_out_close(f16, ref, w.name + " f16")
    print(f"[{w.name}] block-scaled rel_l2={rel:.2e} max_rel={mxe:.2e} (f16 GEMM rel_l2={rel16:.2e})")


def test_block_scaled_tile_edges(k3):
    """Injected routing that puts experts exactly on the 128-token tile edges: 0, 1, 63, 64,
    65, 127, 128, 129, 192 and 256 tokens, both kernels against the oracle (every row)."""
    from k3moe_inputs.device import build_layer
    w = ki.Workload("mx_edges", T=600, d=256, f=256, E=12, k=2, S=1, exp_lo=-8, exp_hi=-4, seed=98)
    counts = [128, 129, 1, 0, 256, 127, 64, 65, 192, 63, 175, 0]
    assert sum(counts) == w.T * w.k and max(counts) < w.T
    # slot list sorted by expert; token t takes entries t and t + T (distinct: no count reaches T)
    lst = np.repeat(np.arange(w.E, dtype=np.int32), counts)
    idx = np.stack([lst[:w.T], lst[w.T:]], axis=1).astype(np.int32)
    assert (idx[:, 0] != idx[:, 1]).all()
    rng = np.random.default_rng(w.seed)
    wt = rng.uniform(0.2, 1.0, size=idx.shape).astype(np.float32)
    wt /= wt.sum(axis=1, keepdims=True)
    off, perm = oracle.perm(idx, w.E)
    assert list(np.diff(off)) == counts
    layer = build_layer(w)
    x = ki.make_x(w)
    xd = dev16(x)
    routing = (dev(idx), dev(wt), dev(off), dev(perm))
    ref = oracle.forward(ocfg(w), x, idx, wt, oracle_experts(w, range(w.E)), ki.make_shared(w))
    for v in (k3.PREFILL_GEMM_F16, k3.PREFILL_GEMM_BLOCK_SCALED):
        k3.k3moe_set_prefill_gemm(v)
        out = torch.empty((w.T, w.d), dtype=torch.float32, device="cuda")
        layer.forward(xd, out, routing=routing)
        rc, code = k3.k3moe_device_status(layer.ws)
        assert rc == 0 and code == 0, (v, rc, code)
        rel, mxe = assert_out_close(host(out), ref, f"tile edges, variant {v}")
        print(f"[mx_edges variant {v}] rel_l2={rel:.2e} max_rel={mxe:.2e}")
    k3.k3moe_set_prefill_gemm(k3.PREFILL_GEMM_DEFAULT)


def test_block_scaled_repeats_bit_for_bit(k3):
    """Two calls on the same routing give the same output (the gate/up GEMM has no atomics;
    the down GEMM's fp32 atomics may reorder additions, so the comparison is at 1e-6)."""
    from k3moe_inputs.device import build_layer
    w = CASES[0]
    layer = build_layer(w)
    xd = dev16(ki.make_x(w))
    layer.route(xd)
    k3.k3moe_set_prefill_gemm(k3.PREFILL_GEMM_BLOCK_SCALED)
    outs = []
    for _ in range(2):
        out = torch.empty((w.T, w.d), dtype=torch.float32, device="cuda")
        layer.forward(xd, out)
        outs.append(host(out))
    k3.k3moe_set_prefill_gemm(k3.PREFILL_GEMM_DEFAULT)
    rc, code = k3.k3moe_device_status(layer.ws)
    assert rc == 0 and code == 0
    d = np.abs(outs[0] - outs[1]).max() / np.abs(outs[0]).max()
    assert d <= 1e-6, d


def test_block_scaled_scale_bytes_0_and_255(k3):
    """Scale byte 255 reads as zero in the oracle; the block-scaled GEMM takes it as 2^-127
    (the tensor core has no zero scale), a difference far below the bar.  Byte 0 is 2^-127
    on both sides."""
    w = ki.Workload("mx_nanscale", T=200, d=384, f=256, E=16, k=4, S=2, exp_lo=-7, exp_hi=-3, seed=96)
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
    k3.k3moe_set_prefill_gemm(k3.PREFILL_GEMM_BLOCK_SCALED)
    out = torch.empty((w.T, w.d), dtype=torch.float32, device="cuda")
    layer.forward(xd, out)
    k3.k3moe_set_prefill_gemm(k3.PREFILL_GEMM_DEFAULT)
    rc, code = k3.k3moe_device_status(layer.ws)
    assert rc == 0 and code == k3.DEV_NAN_SCALE
    ref = oracle.forward(ocfg(w), x, host(layer.idx), host(layer.weight), experts, sh)
    rel, mxe = assert_out_close(host(out), ref, "block-scaled nan-scale")
    print(f"[mx_nanscale] rel_l2={rel:.2e} max_rel={mxe:.2e}")


def test_block_scaled_k3_prefill(k3):
    """The K3 shape at T = 4096 (896 experts, top 16, 2 shared): 1024 rows against the
    oracle, among them the first and last token of every expert's first and last
    128-token tile, the first and last row and every outlier row; and every row against
    the f16 GEMM's output, at the same bar."""
    from k3moe_inputs.device import build_layer
    w = ki.WORKLOADS["prefill_t4096"]
    torch.cuda.empty_cache()
    layer = build_layer(w)
    x = ki.make_x(w)
    xd = dev16(x)
    f16, mx = run_both(k3, layer, xd, w.T)
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
    gidx, gw = host(layer.idx[:w.T]), host(layer.weight[:w.T])
    ref = oracle_forward_expert_major(w, x, gidx, gw, sel)
    rel, mxe = assert_out_close(mx[sel], ref, "prefill_t4096 block-scaled")
    relf, mxf = assert_out_close(mx, f16, "prefill_t4096 block-scaled vs f16")
    print(f"[prefill_t4096 block-scaled] rows={len(sel)} rel_l2={rel:.2e} max_rel={mxe:.2e}; "
          f"vs the f16 GEMM on every row rel_l2={relf:.2e}")
    del layer
    torch.cuda.empty_cache()

"""Helpers shared by the GPU parity tests: device setup, oracle comparisons, tolerances."""
import numpy as np

import k3moe_inputs as ki
import oracle

# Output tolerance: relative L2 <= 5e-3 and max |err| <= 2e-2 * max |ref| (the layer's
# acceptance bar).  Indices, offsets and permutations are compared bit-exactly.
REL_L2 = 5e-3
MAX_REL = 2e-2
# Router scores: the device accumulates each logit's d exact bf16 products in fp32 in
# its own order (the oracle: exactly, then one rounding), so its scores differ from the
# oracle's by accumulation rounding only.  That rounding grows with the size of the
# token's logits, |x_t| * rms(Wr) (about 1.2 at the K3 shapes with unit-variance x):
# the per-token kernel stays within 2e-7 of the oracle; the tensor-core path (T >= 32),
# whose accumulation is coarser, was measured at 3.7e-6 max over 14.7M scores of unit
# scale and 1.3e-5 on tokens scaled by 8.  score_tol(t) = SCORE_TOL_REL * max(1, scale_t)
# bounds |sc_dev - sc_oracle| (plus one rounding of the bias add for ch).  A selection can
# only differ from the oracle's where two compared choice scores lie within twice that of
# each other: the token's near-tie threshold.
SCORE_TOL_REL = 6e-6
BIAS_ADD_TOL = 2.5e-7


def score_tol(x_bf16, wr_bf16):
    """Per-token score tolerance [T] (see above)."""
    x = ki.bf16_to_f32(x_bf16)
    wr = ki.bf16_to_f32(wr_bf16).astype(np.float64)
    scale = np.linalg.norm(x, axis=1).astype(np.float64) * np.sqrt(np.mean(wr * wr))
    return SCORE_TOL_REL * np.maximum(1.0, scale)


def near_tie(x_bf16, wr_bf16):
    return 2.0 * (score_tol(x_bf16, wr_bf16) + BIAS_ADD_TOL)


def out_errors(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    rel_l2 = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300)
    max_rel = np.max(np.abs(got - ref)) / max(np.max(np.abs(ref)), 1e-300)
    return rel_l2, max_rel


def assert_out_close(got, ref, what=""):
    rel_l2, max_rel = out_errors(got, ref)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    assert rel_l2 <= REL_L2 and max_rel <= MAX_REL, f"{what}: rel_l2={rel_l2:.3e} max_rel={max_rel:.3e}"
    return rel_l2, max_rel


def ocfg(w):
    return oracle.cfg(**w.config_kwargs())


def oracle_experts(w, ids):
    return {int(e): ki.make_expert(w, int(e)) for e in sorted(set(int(v) for v in ids))}


def oracle_forward_rows(w, x, idx, weight, rows, batch=8):
    """Oracle output for the given token rows (routing taken as given)."""
    shared = ki.make_shared(w) if w.S else None
    c = ocfg(w)
    outs = []
    rows = list(rows)
    for i in range(0, len(rows), batch):
        r = rows[i:i + batch]
        xi = np.ascontiguousarray(x[r])
        ii = np.ascontiguousarray(idx[r])
        wi = np.ascontiguousarray(weight[r])
        outs.append(oracle.forward(c, xi, ii, wi, oracle_experts(w, ii.ravel()), shared))
    return np.concatenate(outs, axis=0)

"""Helpers shared by the GPU parity tests: device setup, oracle comparisons, tolerances."""
import numpy as np

import k3moe_inputs as ki
import oracle

# Output tolerance: relative L2 <= 5e-3 and max |err| <= 2e-2 * max |ref| (the layer's
# acceptance bar).  Indices, offsets and permutations are compared bit-exactly.
REL_L2 = 5e-3
MAX_REL = 2e-2
# Router: the device computes every logit it selects with as the exact sum of the d bf16
# products rounded once to float, and sc = 1/(1+expf(-logit)) with the correctly rounded
# float exponential; the oracle sums in double, rounds once, and calls the host's expf.
# They agree bit for bit except where the host's expf misrounds (its error bound is a
# little over half an ulp) or the exact sum sits within ~1e-12 (relative) of a rounding
# boundary, and then by an ulp or two: SCORE_ULPS bounds |sc_dev - sc_oracle| in ulps of
# sc (ch: plus one rounding of the bias add).
SCORE_ULPS = 4
# The acceptance rule's near-tie: a token whose k-th and (k+1)-th oracle choice scores
# differ by less than this (but are not equal) may take either expert; such tokens are
# counted and checked for validity only.
NEAR_TIE = 1e-6


def ulp32(v):
    """Spacing of float32 at |v| (the ulp), as float64."""
    return np.spacing(np.abs(np.asarray(v, dtype=np.float32))).astype(np.float64)


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


def oracle_forward_expert_major(w, x, idx, weight, rows):
    """Oracle output for the token rows `rows` (routing taken as given), expert by expert,
    so that only one routed expert's weights are held at a time: each expert's weighted
    output for the rows routed to it comes from the oracle's forward with that single
    expert (k = 1, the row's weight), the shared experts' from the oracle's forward as its
    shared part alone; the per-expert float results are summed in double.  The oracle's
    own forward sums the same terms in double before one rounding, so the two differ by
    about k float roundings (~1e-7 relative), far inside the output tolerance."""
    rows = np.asarray(rows)
    xr = np.ascontiguousarray(x[rows])
    ir, wr = idx[rows], weight[rows]
    acc = np.zeros((len(rows), w.d), dtype=np.float64)
    c1 = oracle.cfg(**dict(w.config_kwargs(), top_k=1, n_shared=0))
    for e in np.unique(ir):
        r, j = np.nonzero(ir == e)
        got = oracle.forward(c1, np.ascontiguousarray(xr[r]), np.full((len(r), 1), e, dtype=np.int32),
                             np.ascontiguousarray(wr[r, j].reshape(-1, 1)), {int(e): ki.make_expert(w, int(e))},
                             None)
        acc[r] += got
    if w.S:
        cs = oracle.cfg(**dict(w.config_kwargs(), top_k=1))
        e0 = int(ir[0, 0])
        _, sh = oracle.forward(cs, xr, np.full((len(rows), 1), e0, dtype=np.int32),
                               np.zeros((len(rows), 1), dtype=np.float32), {e0: ki.make_expert(w, e0)},
                               ki.make_shared(w), want_shared=True)
        acc += sh
    return acc

"""The test helpers' own arithmetic, pinned on the CPU: the expert-by-expert assembly of
the oracle's output (used where the oracle checks every row of a large workload) equals
the oracle's own forward on the same routing."""
import numpy as np

import k3moe_inputs as ki
import oracle
from gpu_util import oracle_forward_expert_major, out_errors


def test_expert_major_assembly_equals_oracle_forward():
    w = ki.Workload("helper", T=37, d=384, f=256, E=16, k=4, S=2, exp_lo=-7, exp_hi=-3, seed=40)
    x = ki.make_x(w)
    idx, wt, _ = oracle.route(oracle.cfg(**w.config_kwargs()), x, ki.make_router(w), None)
    rows = [0, 3, 4, 17, 36]
    got = oracle_forward_expert_major(w, x, idx, wt, rows)
    ref = oracle.forward(oracle.cfg(**w.config_kwargs()), np.ascontiguousarray(x[rows]),
                         np.ascontiguousarray(idx[rows]), np.ascontiguousarray(wt[rows]),
                         {e: ki.make_expert(w, e) for e in range(w.E)}, ki.make_shared(w))
    rel_l2, max_rel = out_errors(got, ref)
    # k float roundings of the per-expert terms apart, nothing more
    assert rel_l2 < 1e-6 and max_rel < 1e-6

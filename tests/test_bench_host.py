"""The benchmark's CPU restatement of the pages' method (gather + einsum
attention in fp32) computes the same attention as the oracle."""
import numpy as np
import pytest

import bench
import oracle
from gpu_step import raw
from workloads import draw_plan, make_layer


@pytest.mark.parametrize("name", ["toy", "smollm2-135m"])
def test_pages_method_matches_oracle(name):
    plan = draw_plan(name)
    layer = make_layer(plan, 0)
    nd = plan.n_decode
    outs = []
    bench.pages_method_sample(plan, layer, range(nd), outputs=outs)
    r = {n: raw(layer[n]) for n in ("q", "k_pool", "v_pool")}
    ref = oracle.paged_attention_decode(r["q"][:nd], r["k_pool"], r["v_pool"], plan.block_tables[:nd],
                                        plan.seq_lens[:nd], plan.shape.scale, plan.shape.dtype)
    got = np.stack([o.double().numpy() for o in outs])
    assert np.max(np.abs(got - ref)) < 1e-5

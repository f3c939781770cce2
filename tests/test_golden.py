"""Fixtures under tests/golden/: printed workload shapes and stored oracle values."""
import json
import os

import numpy as np

import ssd_inputs

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def test_workload_shapes_match_the_printed_shapes():
    spec = json.load(open(os.path.join(GOLDEN, "workloads.json")))
    for name, w in ssd_inputs.WORKLOADS.items():
        assert w.shape_tuple() == spec[name]["shape"], name
        assert w.return_final_state == spec[name]["final_state"], name


def test_tiny_workload_is_the_readme_demo():
    """README "Usage": x, B, C ~ randn, dt ~ rand, A = -rand [H], chunk 128,
    dt_softplus, final state returned, fp32."""
    w = ssd_inputs.WORKLOADS["tiny"]
    inp = ssd_inputs.make(w)
    assert inp["x"].dtype == inp["B"].dtype == inp["C"].dtype == inp["dt"].dtype
    assert str(inp["x"].dtype) == "torch.float32"
    assert float(inp["dt"].min()) >= 0.0 and float(inp["dt"].max()) <= 1.0
    assert float(inp["A"].max()) <= 0.0 and float(inp["A"].min()) >= -1.0
    assert inp["D"] is None and inp["z"] is None and inp["initial_states"] is None


def test_oracle_reproduces_stored_tiny_values(oracle_mod):
    ref = json.load(open(os.path.join(GOLDEN, "tiny_oracle.json")))
    inp = ssd_inputs.make(ssd_inputs.WORKLOADS["tiny"])
    prob = oracle_mod.Problem(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], dt_softplus=True)
    y, fin = oracle_mod.forward(prob)
    for idx, v in ref["y_samples"]:
        assert abs(y[tuple(idx)] - v) <= 1e-12 * max(1.0, abs(v))
    for idx, v in ref["final_samples"]:
        assert abs(fin[tuple(idx)] - v) <= 1e-12 * max(1.0, abs(v))
    assert abs(np.linalg.norm(y.ravel()) - ref["y_l2"]) <= 1e-10 * ref["y_l2"]
    assert abs(np.linalg.norm(fin.ravel()) - ref["final_l2"]) <= 1e-10 * ref["final_l2"]

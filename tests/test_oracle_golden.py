"""The oracle still reproduces its stored regression fixture."""
import json
import os
import sys

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.join(HERE, "golden"))


def _unhex(rows):
    return torch.tensor([[float.fromhex(v) for v in r] for r in rows],
                        dtype=torch.float64)


def test_oracle_reproduces_tiny_layer_fixture(oracle_lib):
    import make_golden
    doc = json.load(open(os.path.join(HERE, "golden", "tiny_layer.json")))
    L = make_golden.grid_layer()
    ids, w, out, logits = oracle_lib.forward(L, want_logits=True)
    # logits are sums of exact products on a power-of-two grid: exact
    assert torch.equal(logits.double(), _unhex(doc["logits"]))
    assert ids.tolist() == doc["topk_ids"]
    # softmax / sigmoid go through the host libm's expf: allow 1e-6 relative
    ref_w, ref_out = _unhex(doc["topk_w"]), _unhex(doc["out"])
    assert (w.double() - ref_w).abs().max() <= 1e-6
    assert (out.double() - ref_out).abs().max() <= 1e-6 * ref_out.abs().max()

"""Write tests/golden/tiny_layer.json: a regression fixture of the oracle.

The layer's inputs are a closed-form integer grid (every value a small integer
over a power of two, so exact in bf16); the expected outputs are what the
oracle computes for them.  This script calls only oracle/ (and torch for
containers).  It guards the oracle against later drift; the pins in
tests/test_oracle_pins.py are what tie it to the page.

Usage: python tests/golden/make_golden.py
"""
import json
import os
import sys

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

SPEC = dict(T=3, H=32, I=32, E=4, top_k=2)


def grid_layer():
    """The fixture's inputs, as a synth.Layer-like object."""
    from types import SimpleNamespace
    T, H, I, E = SPEC["T"], SPEC["H"], SPEC["I"], SPEC["E"]

    def bf(f, shape):
        idx = torch.stack(torch.meshgrid(*[torch.arange(s) for s in shape],
                                         indexing="ij"), dim=-1)
        vals = f(*[idx[..., d] for d in range(len(shape))]).to(torch.float32)
        return vals.to(torch.bfloat16).contiguous()

    x = bf(lambda t, h: ((t * 13 + h * 7) % 17 - 8) / 8.0, (T, H))
    wr = bf(lambda e, h: ((e * 5 + h * 3) % 11 - 5) / 64.0, (E, H))
    br = bf(lambda e: ((e * 3) % 5 - 2) / 256.0, (E,))
    w_gu = bf(lambda e, n, k: ((e * 31 + n * 17 + k * 5) % 23 - 11) / 128.0,
              (E, 2 * I, H))
    b_gu = bf(lambda e, n: ((e + n * 3) % 7 - 3) / 64.0, (E, 2 * I))
    w_d = bf(lambda e, n, k: ((e * 7 + n * 11 + k * 13) % 19 - 9) / 128.0,
             (E, H, I))
    b_d = bf(lambda e, n: ((e * 2 + n) % 5 - 2) / 64.0, (E, H))
    return SimpleNamespace(T=T, H=H, I=I, E=E, top_k=SPEC["top_k"],
                           wfmt="bf16", x=x, wr=wr, br=br, w_gu=w_gu,
                           b_gu=b_gu, w_d=w_d, b_d=b_d, s_gu=None, s_d=None)


def main():
    import oracle
    L = grid_layer()
    ids, w, out, logits = oracle.forward(L, want_logits=True)
    doc = {
        "what": "oracle regression fixture, gpt-oss MoE layer on a closed-form "
                "integer grid (see make_golden.py: grid_layer)",
        "source": "xserv docs/19-gpt-oss-moe.md, 'Phase 19: gpt-oss-20b', "
                  "section 1 table (MoE and activation rows), section 2 "
                  "(MoE forward)",
        "spec": SPEC,
        "logits": [[float.hex(float(v)) for v in r] for r in logits.tolist()],
        "topk_ids": ids.tolist(),
        "topk_w": [[float.hex(float(v)) for v in r] for r in w.tolist()],
        "out": [[float.hex(float(v)) for v in r] for r in out.tolist()],
    }
    with open(os.path.join(HERE, "tiny_layer.json"), "w") as f:
        json.dump(doc, f, indent=1)


if __name__ == "__main__":
    main()

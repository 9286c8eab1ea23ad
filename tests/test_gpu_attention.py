"""Attention with sinks on the GPU against the fp64 CPU oracle (the other
half of a gpt-oss block: sliding-window / full layers, per-head sinks, GQA)."""
import pytest
import torch

pytestmark = pytest.mark.gpu

TOL = 1e-2      # P is rounded to bf16 for the second MMA


@pytest.fixture(scope="module")
def moe():
    from gpt_oss_moe_gb300 import _build
    _build.build()
    import gpt_oss_moe_gb300 as m
    return m


CASES = [
    # Tq, Tkv, Hq, Hkv, window, sinks ("n": N(0,1), "none": -inf, "big": +20)
    (1, 1, 8, 1, 0, "n"),
    (70, 70, 8, 2, 0, "n"),              # ragged query and key tails
    (300, 300, 8, 1, 128, "n"),          # tiles that slid out of the window
    (300, 300, 8, 1, 128, "none"),       # ... with no sink: the running max starts at -inf
    (200, 200, 4, 4, 1, "n"),            # window of one key
    (512, 512, 64, 8, 128, "n"),         # gpt-oss sliding layer
    (512, 512, 64, 8, 0, "n"),           # gpt-oss full layer
    (130, 130, 8, 2, 0, "big"),          # the sink takes almost all the mass
    (1, 1000, 64, 8, 128, "n"),          # decode step, sliding
    (1, 1000, 64, 8, 0, "n"),            # decode step, full
    (5, 700, 16, 2, 128, "none"),        # several new queries at the end of a cache
    (64, 2048, 8, 1, 0, "n"),            # keys split over 16 CTAs, merged
    (200, 3000, 8, 2, 0, "none"),        # split keys, no sink, four query blocks
    (100, 100, 12, 4, 0, "n"),           # 3 heads per KV head: one head per CTA
    (1, 500, 12, 4, 128, "n"),           # ... decode
    (1024, 1024, 64, 8, 0, "n"),         # prefill-sized: several 128-query blocks
    (1024, 1024, 64, 8, 128, "n"),       # ... sliding: tiles before the window skipped
    (600, 4096, 8, 1, 0, "none"),        # queries at the end of a longer cache
]

# "attn_tc": 1 = the 64-row mma.sync kernel (with key splits), 2 = the
# tcgen05 kernel (128-query blocks; TMEM scores, P back through TMEM) with
# suspending hand-off waits (the default), 3 = the tcgen05 kernel with
# polling waits ("attn_poll" 1)
MODES = [1, 2, 3]


@pytest.mark.parametrize("mode", MODES, ids=["mma_sync", "tcgen05", "tcgen05_poll"])
@pytest.mark.parametrize("case", CASES, ids=lambda c: "Tq{}Tkv{}Hq{}Hkv{}W{}{}".format(*c))
def test_attention_sinks_matches_oracle(moe, oracle_lib, synth_lib, case, mode):
    Tq, Tkv, Hq, Hkv, W, sk = case
    a = synth_lib.make_attention(Tkv, Tkv, Hq=Hq, Hkv=Hkv, D=64, seed=Tq + Tkv + W)
    q = a["q"][Tkv - Tq:]
    sinks = a["sinks"]
    if sk == "none":
        sinks = torch.full_like(sinks, float("-inf"))
    elif sk == "big":
        sinks = torch.full_like(sinks, 20.0)
    ref = oracle_lib.attention_sinks(q, a["k"], a["v"], sinks, window=W)
    tc = mode >= 2
    moe.moe_set_tuning("attn_tc", 2 if tc else 1)
    moe.moe_set_tuning("attn_poll", 1 if mode == 3 else 0)
    try:
        ws = torch.zeros(4096, dtype=torch.uint8, device="cuda")
        if tc:
            ws = torch.full((256,), 0x55, dtype=torch.uint8, device="cuda")   # cleared by the call
        out = moe.attention_sinks(q.cuda(), a["k"].cuda(), a["v"].cuda(), sinks.cuda(), window=W,
                                  workspace=ws if tc else None)
        torch.cuda.synchronize()
        if tc:
            assert moe.moe_get_device_status(ws) == 0
    finally:
        moe.moe_set_tuning("attn_tc", 0)
        moe.moe_set_tuning("attn_poll", 0)
    got = out.cpu()
    assert torch.isfinite(got).all()
    err = (got - ref).abs().max().item()
    assert err <= TOL * max(ref.abs().max().item(), 1e-30), err


def test_attention_rejects_bad_shapes(moe):
    q = torch.zeros((4, 8, 32), dtype=torch.bfloat16, device="cuda")
    k = torch.zeros((4, 2, 32), dtype=torch.bfloat16, device="cuda")
    s = torch.zeros(8, device="cuda")
    with pytest.raises(Exception):
        moe.attention_sinks(q, k, k, s)                     # D = 32
    q = torch.zeros((4, 6, 64), dtype=torch.bfloat16, device="cuda")
    k = torch.zeros((4, 4, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(Exception):
        moe.attention_sinks(q, k, k, torch.zeros(6, device="cuda"))   # 6 % 4 != 0

"""Failure detection, determinism and the debugging switches, on the GPU.

Every fault here is made on purpose through the library's test switches
(moe_set_tuning "inject") and must come back as a bit of the device status
word; none of them faults, traps or hangs the GPU:
  * a routed expert id out of range  -> MOE_DEV_BAD_EXPERT_ID,
  * a GEMM tile naming an expert out of range -> MOE_DEV_BAD_TILE,
  * a pipeline wait on a barrier nothing arrives on -> MOE_DEV_WAIT_TIMEOUT
    after the kernel's ~1 s bound (every role leaves, TMEM is freed).
After each, the same workspace, cleared, serves a normal call that matches
the oracle.  The environment switches (MOE_CHECK_STAGES, MOE_NVTX) are read
once per process, so their tests run a child process.
"""
import os
import subprocess
import sys

import pytest
import torch

from parity_util import TOL_BF16, TOL_MXFP4, compare_output, gpu_forward, to_device

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a GPU")]

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def moe():
    from gpt_oss_moe_gb300 import _build
    _build.build()
    import gpt_oss_moe_gb300 as m
    m.lib()
    return m


def _oracle_ok(oracle_lib, L, out, tol=TOL_BF16):
    _, _, o_out = oracle_lib.forward(L)
    compare_output(out.float(), o_out, slice(None), tol)


# ---------------------------------------------------------------- determinism

DET_CASES = [
    # name, E, k, H, I, T, wfmt
    ("small", 8, 4, 320, 192, 37, "bf16"),
    ("ksplit", 8, 4, 1024, 512, 3, "bf16"),       # down would split K
    ("fp8", 8, 4, 256, 256, 200, "fp8"),
    ("mxfp4", 8, 4, 256, 192, 45, "mxfp4"),
    ("mx", 8, 4, 320, 192, 37, "mxfp4_mxfp8"),
]


@pytest.mark.parametrize("case", DET_CASES, ids=lambda c: c[0])
def test_deterministic_combine_is_bitwise_reproducible(moe, oracle_lib, synth_lib, case):
    _, E, k, H, I, T, wfmt = case
    L = synth_lib.make_layer(E=E, T=T, H=H, I=I, top_k=k, seed=1200 + T, wfmt=wfmt,
                             router_w_std=0.05)
    dev = to_device(L)
    _, _, o_atomic, _ = gpu_forward(moe, L, dev=dev)
    moe.moe_set_tuning("deterministic", 1)
    try:
        runs = [gpu_forward(moe, L, dev=dev) for _ in range(3)]
        runs16 = [gpu_forward(moe, L, dev=dev, out_dtype=torch.bfloat16) for _ in range(2)]
    finally:
        moe.moe_set_tuning("deterministic", 0)
    for ids, w, out, ws in runs + runs16:
        assert moe.moe_get_device_status(ws) == 0
    assert all(torch.equal(r[2], runs[0][2]) for r in runs[1:])
    assert torch.equal(runs16[0][2], runs16[1][2])
    # the bf16 output is the rounded fp32 output of the same sums
    assert torch.equal(runs16[0][2], runs[0][2].to(torch.bfloat16))
    # the same sums as the atomic combine, up to the order of the k terms
    scale = o_atomic.abs().max().item()
    assert (runs[0][2] - o_atomic).abs().max().item() <= 1e-5 * scale
    _oracle_ok(oracle_lib, L, runs[0][2], TOL_MXFP4 if wfmt == "mxfp4" else TOL_BF16)


def test_deterministic_gpt_oss_decode(moe, oracle_lib, synth_lib):
    L = synth_lib.make_workload("20b_decode", 64)
    dev = to_device(L)
    moe.moe_set_tuning("deterministic", 1)
    try:
        a = gpu_forward(moe, L, dev=dev)
        b = gpu_forward(moe, L, dev=dev)
    finally:
        moe.moe_set_tuning("deterministic", 0)
    assert torch.equal(a[2], b[2]) and torch.equal(a[0], b[0])
    _oracle_ok(oracle_lib, L, a[2])


def test_deterministic_expert_parallel_partials(moe, oracle_lib, synth_lib):
    L = synth_lib.make_layer(E=8, T=40, H=256, I=192, top_k=3, seed=1290, router_w_std=0.05)
    dev = to_device(L)
    shape = moe.layer_shape(L)
    moe.moe_set_tuning("deterministic", 1)
    try:
        outs = []
        for _ in range(2):
            out = torch.empty((L.T, L.H), dtype=torch.float32, device="cuda")
            ws = moe.moe_forward_ep(shape, 3, 4, dev["x"], dev["wr"], dev["br"],
                                    dev["w_gu"][3:7], dev["b_gu"][3:7], dev["w_d"][3:7],
                                    dev["b_d"][3:7], out)
            assert moe.moe_get_device_status(ws) == 0
            outs.append(out)
    finally:
        moe.moe_set_tuning("deterministic", 0)
    assert torch.equal(outs[0], outs[1])
    o_part = oracle_lib.forward_ep(L, 3, 4)
    _, _, full = oracle_lib.forward(L)
    assert (outs[0].cpu() - o_part).abs().max().item() <= TOL_BF16 * full.abs().max().item()


def test_deterministic_needs_its_workspace(moe, synth_lib):
    """The ordered combine's rows are part of the workspace only while the
    switch is on: a workspace sized before is refused, not overrun."""
    L = synth_lib.make_layer(E=8, T=20, H=128, I=128, top_k=2, seed=1291)
    dev = to_device(L)
    small = moe.alloc_workspace(moe.layer_shape(L))
    moe.moe_set_tuning("deterministic", 1)
    try:
        assert moe.moe_workspace_bytes(moe.layer_shape(L)) > small.numel()
        out = torch.empty((L.T, L.H), device="cuda")
        with pytest.raises(moe.MoEError) as e:
            moe.moe_forward(moe.layer_shape(L), dev["x"], dev["wr"], dev["br"], dev["w_gu"],
                            dev["b_gu"], dev["w_d"], dev["b_d"], out, workspace=small)
        assert e.value.code == -4
    finally:
        moe.moe_set_tuning("deterministic", 0)


# ---------------------------------------------------------------- injected faults

@pytest.mark.parametrize("bit,expect", [(1, 0x1), (2, 0x4), (4, 0x2)],
                         ids=["bad_expert_id", "bad_tile", "wait_timeout"])
def test_injected_fault_is_reported_and_the_workspace_recovers(moe, oracle_lib, synth_lib,
                                                               bit, expect):
    L = synth_lib.make_layer(E=8, T=37, H=320, I=192, top_k=4, seed=1300 + bit,
                             router_w_std=0.05)
    dev = to_device(L)
    ws = moe.alloc_workspace(moe.layer_shape(L))
    moe.moe_set_tuning("inject", bit)
    try:
        gpu_forward(moe, L, dev=dev, workspace=ws)
    finally:
        moe.moe_set_tuning("inject", 0)
    status = moe.moe_get_device_status(ws)
    assert status & expect, hex(status)
    # the context is intact: the cleared workspace serves a correct call
    moe.moe_clear_device_status(ws)
    ids, w, out, _ = gpu_forward(moe, L, dev=dev, workspace=ws)
    assert moe.moe_get_device_status(ws) == 0
    _oracle_ok(oracle_lib, L, out)


def test_injected_fault_in_routing_only(moe, synth_lib):
    """moe_route reports a bad id from the router the same way."""
    L = synth_lib.make_layer(E=32, T=40, H=128, I=128, top_k=4, seed=1310, with_experts=False)
    moe.moe_set_tuning("inject", 1)
    try:
        ws = moe.moe_route(moe.make_shape(40, 128, 128, 32, 4), L.x.cuda(), L.wr.cuda(),
                           L.br.cuda())
    finally:
        moe.moe_set_tuning("inject", 0)
    assert moe.moe_get_device_status(ws) & 0x1


# ---------------------------------------------------------------- environment switches

_CHILD = r'''
import json, os, sys
sys.path.insert(0, {root!r}); sys.path.insert(0, os.path.join({root!r}, "tests"))
import torch, synth, oracle
import gpt_oss_moe_gb300 as moe
from parity_util import gpu_forward, to_device
synth.build(); oracle.build(); moe.lib()
res = {{"lib": moe.LIB_PATH}}
L = synth.make_layer(E=8, T=37, H=320, I=192, top_k=4, seed=1400, router_w_std=0.05)
dev = to_device(L)
ids, w, out, ws = gpu_forward(moe, L, dev=dev)
res["status"] = moe.moe_get_device_status(ws)
res["stats"] = moe.moe_stage_stats(ws)
_, _, o = oracle.forward(L)
res["err"] = (out.cpu() - o).abs().max().item() / o.abs().max().item()
res["max_out"] = out.abs().max().item()
# K split and the MXFP4 path as well
L2 = synth.make_layer(E=4, T=3, H=1024, I=512, top_k=2, seed=1401, wfmt="mxfp4", router_w_std=0.05)
_, _, out2, ws2 = gpu_forward(moe, L2)
_, _, o2 = oracle.forward(L2)
res["status2"] = moe.moe_get_device_status(ws2)
res["err2"] = (out2.cpu() - o2).abs().max().item() / o2.abs().max().item()
# a NaN in one activation: the first stage's check must see it (in the
# gathered rows of the permutation path: the token's four copies; in the
# layer input for the small-batch path, which stores no copies: once)
if os.environ.get("MOE_CHECK_STAGES") == "1":
    L.x = L.x.clone(); L.x[5, 7] = float("nan")
    dev["x"] = L.x.cuda()
    for small in (0, 1):
        moe.moe_set_tuning("small_path", small)
        L8 = synth.make_layer(E=8, T=24, H=320, I=192, top_k=4, seed=1400, router_w_std=0.05)
        LL = L if small == 0 else L8
        if small:
            LL.x = LL.x.clone(); LL.x[5, 7] = float("nan")
        _, _, out3, ws3 = gpu_forward(moe, LL)
        res[f"nan_status{{small}}"] = moe.moe_get_device_status(ws3)
        res[f"nan_stats{{small}}"] = moe.moe_stage_stats(ws3)
    moe.moe_set_tuning("small_path", 1)
print("RESULT " + json.dumps(res))
'''


def _child(env_extra):
    env = dict(os.environ)
    env.update(env_extra)
    r = subprocess.run([sys.executable, "-c", _CHILD.format(root=ROOT)], env=env,
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-2000:]
    import json
    line = [l for l in r.stdout.splitlines() if l.startswith("RESULT ")][-1]
    return json.loads(line[len("RESULT "):])


def test_stage_checks_count_nonfinite_values_per_stage(moe):
    res = _child({"MOE_CHECK_STAGES": "1"})
    assert res["status"] == 0 and res["status2"] == 0
    assert res["err"] <= TOL_BF16 and res["err2"] <= TOL_MXFP4
    (nf0, m0), (nf1, m1), (nf2, m2) = res["stats"]
    assert nf0 == nf1 == nf2 == 0
    assert 0 < m0 < 10 and 0 < m1 < 56 and abs(m2 - res["max_out"]) <= 1e-6 * res["max_out"]
    # the planted NaN shows from the first stage on, and sets its status bit
    assert res["nan_status0"] & 0x8 and res["nan_status1"] & 0x8
    assert res["nan_stats0"][0][0] == 4      # the token's row, gathered for 4 experts
    assert res["nan_stats1"][0][0] == 1      # the layer input (small batches)


def test_nvtx_ranges_switch(moe):
    res = _child({"MOE_NVTX": "1"})
    assert res["status"] == 0 and res["err"] <= TOL_BF16 and res["err2"] <= TOL_MXFP4
    assert res["stats"] == [[0, 0.0], [0, 0.0], [0, 0.0]]      # checks off


def test_debug_bounds_build(moe):
    """The MOE_DEBUG_BOUNDS variant: every store index checked; a clean run
    reports nothing and matches the oracle."""
    from gpt_oss_moe_gb300 import _build
    lib = _build.build(variant="debug_bounds")
    res = _child({"GPT_OSS_MOE_LIB": lib})
    assert res["lib"] == lib
    assert res["status"] == 0 and res["status2"] == 0
    assert res["err"] <= TOL_BF16 and res["err2"] <= TOL_MXFP4

"""moe_forward_noalloc against moe_forward, through the C ABI.

moe_forward_noalloc serves callers that cannot allocate device memory: hosts
that hand a plugin only its inputs and outputs and plan every other byte of
device memory themselves, or that cannot afford cudaMalloc's implicit
synchronisation.  It keeps its scratch in the library's own static device
array instead of a caller workspace.  This file is collected last, so a run
that stops at the first failure has already run every other test; it also
passes alone in a fresh process.
"""
import ctypes

import pytest
import torch

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a GPU")]

NOALLOC_BYTES = 8 << 20          # MOE_NOALLOC_SCRATCH_BYTES
REL_TOL = 1e-5                   # the two paths differ only in the fp32 combine order


@pytest.fixture(scope="module")
def moe():
    from gpt_oss_moe_gb300 import _build
    _build.build()
    import gpt_oss_moe_gb300 as m
    m.lib()
    return m


def _call_noalloc(moe, shape, dev, x, out, ids, w, status):
    gu = moe.moe_weight(dev["w_gu"].data_ptr(), None, dev["b_gu"].data_ptr())
    dn = moe.moe_weight(dev["w_d"].data_ptr(), None, dev["b_d"].data_ptr())
    return moe.lib().moe_forward_noalloc(
        ctypes.byref(shape), x.data_ptr(), dev["wr"].data_ptr(), dev["br"].data_ptr(),
        gu, dn, out.data_ptr(), 1 if out.dtype == torch.float32 else 0,
        ids.data_ptr(), w.data_ptr(), status.data_ptr(),
        torch.cuda.current_stream().cuda_stream)


def _reference(moe, shape, dev, x, dtype):
    T, H = x.shape
    out = torch.empty((T, H), dtype=dtype, device="cuda")
    ids = torch.empty((T, shape.top_k), dtype=torch.int32, device="cuda")
    moe.moe_forward(shape, x, dev["wr"], dev["br"], dev["w_gu"], dev["b_gu"],
                    dev["w_d"], dev["b_d"], out, topk_ids_out=ids)
    return out, ids


def _noalloc(moe, shape, dev, x, dtype):
    T, H = x.shape
    out = torch.full((T, H), float("nan"), dtype=dtype, device="cuda")
    ids = torch.full((T, shape.top_k), -1, dtype=torch.int32, device="cuda")
    w = torch.empty((T, shape.top_k), dtype=torch.float32, device="cuda")
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    code = _call_noalloc(moe, shape, dev, x, out, ids, w, status)
    return code, out, ids, status


def _same(ref, got):
    (ref_out, ref_ids), (code, out, ids, status) = ref, got
    assert code == 0
    assert int(status.item()) == 0
    assert torch.equal(ids, ref_ids)
    err = (out.float() - ref_out.float()).abs().max().item()
    scale = ref_out.float().abs().max().item()
    # bf16 outputs: one rounding of sums that may differ in the last fp32 bit
    tol = REL_TOL if out.dtype == torch.float32 else 2.0 ** -7
    assert err <= tol * scale, (err, scale)


def _random_layer(E, H, I, seed):
    """Seeded synthetic bf16 layer drawn on the device (no oracle is involved:
    the two entry points are compared with each other)."""
    g = torch.Generator(device="cuda").manual_seed(seed)
    rn = lambda *s, std: (torch.randn(*s, generator=g, device="cuda") * std).to(torch.bfloat16)
    return {"wr": rn(E, H, std=0.02), "br": rn(E, std=0.01),
            "w_gu": rn(E, 2 * I, H, std=0.02), "b_gu": rn(E, 2 * I, std=0.01),
            "w_d": rn(E, H, I, std=0.02), "b_d": rn(E, H, std=0.01)}, g


def test_noalloc_matches_workspace_entry_point_on_two_calls_in_a_row(moe, synth_lib):
    L = synth_lib.make_workload("20b_decode", 64)
    dev = {n: getattr(L, n).cuda() for n in ("x", "wr", "br", "w_gu", "b_gu", "w_d", "b_d")}
    x2 = synth_lib.make_x(16, L.H, seed=77).cuda()        # second call: other tokens
    calls = [(dev["x"], torch.float32), (x2, torch.bfloat16)]
    shapes = [moe.make_shape(x.shape[0], L.H, L.I, L.E, L.top_k) for x, _ in calls]
    refs = [_reference(moe, s, dev, x, dt) for s, (x, dt) in zip(shapes, calls)]
    # the same two calls, back to back, through the no-allocation entry point
    got = [_noalloc(moe, s, dev, x, dt) for s, (x, dt) in zip(shapes, calls)]
    torch.cuda.synchronize()
    for r, g in zip(refs, got):
        _same(r, g)


def test_noalloc_clears_counters_left_by_a_failed_call(moe, synth_lib):
    """A call that gives up on the device can leave the completion counters
    after the status word non-zero.  The test switch fills them (and the
    status word) with non-zero bytes before the next call; the call must
    clear them itself and still match moe_forward, twice in a row."""
    L = synth_lib.make_workload("20b_decode", 64)
    dev = {n: getattr(L, n).cuda() for n in ("x", "wr", "br", "w_gu", "b_gu", "w_d", "b_d")}
    for T in (64, 3):          # 3 tokens: K-split tickets in use as well
        x = dev["x"][:T].contiguous()
        shape = moe.make_shape(T, L.H, L.I, L.E, L.top_k)
        ref = _reference(moe, shape, dev, x, torch.float32)
        moe.moe_set_tuning("noalloc_poison", 1)
        try:
            got = _noalloc(moe, shape, dev, x, torch.float32)
        finally:
            moe.moe_set_tuning("noalloc_poison", 0)
        again = _noalloc(moe, shape, dev, x, torch.float32)
        torch.cuda.synchronize()
        _same(ref, got)
        _same(ref, again)


def _limits(moe, E):
    """Largest accepted and smallest rejected T at gpt-oss widths, top-4."""
    acc = [T for T in range(1, 1024)
           if moe.moe_workspace_bytes(moe.make_shape(T, 2880, 2880, E, 4)) <= NOALLOC_BYTES]
    return max(acc), max(acc) + 1


@pytest.mark.parametrize("E", [32, 128])
def test_noalloc_size_limit(moe, E):
    """The largest shape that fits the static scratch runs and matches
    moe_forward; the next one is rejected with MOE_ERR_WORKSPACE before
    anything is enqueued."""
    t_ok, t_bad = _limits(moe, E)
    assert moe.moe_workspace_bytes(moe.make_shape(t_bad, 2880, 2880, E, 4)) > NOALLOC_BYTES
    dev, g = _random_layer(E, 2880, 2880, seed=1000 + E)
    x = torch.randn(t_ok, 2880, generator=g, device="cuda").to(torch.bfloat16)
    shape = moe.make_shape(t_ok, 2880, 2880, E, 4)
    ref = _reference(moe, shape, dev, x, torch.float32)
    got = _noalloc(moe, shape, dev, x, torch.float32)
    torch.cuda.synchronize()
    _same(ref, got)
    big = moe.make_shape(t_bad, 2880, 2880, E, 4)
    code = moe.lib().moe_forward_noalloc(ctypes.byref(big), 16, 32, 48, moe.moe_weight(),
                                         moe.moe_weight(), 64, 1, None, None, None, None)
    assert code == -4                                    # MOE_ERR_WORKSPACE

"""moe_forward_noalloc against moe_forward, through the C ABI.

moe_forward_noalloc serves callers that cannot allocate device memory (hosts
that hand a plugin only its inputs and outputs): it keeps its scratch in the
library's own static device array instead of a caller workspace.  This file
is collected last, so a run that stops at the first failure has already run
every other test; it also passes alone in a fresh process.
"""
import ctypes

import pytest
import torch

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a GPU")]


def _call_noalloc(moe, shape, dev, x, out, ids, w, status):
    gu = moe.moe_weight(dev["w_gu"].data_ptr(), None, dev["b_gu"].data_ptr())
    dn = moe.moe_weight(dev["w_d"].data_ptr(), None, dev["b_d"].data_ptr())
    return moe.lib().moe_forward_noalloc(
        ctypes.byref(shape), x.data_ptr(), dev["wr"].data_ptr(), dev["br"].data_ptr(),
        gu, dn, out.data_ptr(), 1 if out.dtype == torch.float32 else 0,
        ids.data_ptr(), w.data_ptr(), status.data_ptr(),
        torch.cuda.current_stream().cuda_stream)


def test_noalloc_matches_workspace_entry_point_on_two_calls_in_a_row(synth_lib):
    from gpt_oss_moe_gb300 import _build
    _build.build()
    import gpt_oss_moe_gb300 as moe

    L = synth_lib.make_workload("20b_decode", 64)
    dev = {n: getattr(L, n).cuda() for n in ("x", "wr", "br", "w_gu", "b_gu", "w_d", "b_d")}
    x2 = synth_lib.make_x(16, L.H, seed=77).cuda()        # second call: other tokens
    calls = [(64, dev["x"], torch.float32), (16, x2, torch.bfloat16)]

    # reference results from the workspace entry point
    refs = []
    for T, x, dt in calls:
        shape = moe.make_shape(T, L.H, L.I, L.E, L.top_k)
        out = torch.empty((T, L.H), dtype=dt, device="cuda")
        ids = torch.empty((T, 4), dtype=torch.int32, device="cuda")
        moe.moe_forward(shape, x, dev["wr"], dev["br"], dev["w_gu"], dev["b_gu"],
                        dev["w_d"], dev["b_d"], out, topk_ids_out=ids)
        refs.append((out, ids))

    # the same two calls, back to back, through the no-allocation entry point
    got = []
    for T, x, dt in calls:
        shape = moe.make_shape(T, L.H, L.I, L.E, L.top_k)
        out = torch.full((T, L.H), float("nan"), dtype=dt, device="cuda")
        ids = torch.full((T, 4), -1, dtype=torch.int32, device="cuda")
        w = torch.empty((T, 4), dtype=torch.float32, device="cuda")
        status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
        assert _call_noalloc(moe, shape, dev, x, out, ids, w, status) == 0
        got.append((out, ids, status))
    torch.cuda.synchronize()

    for (ref_out, ref_ids), (out, ids, status) in zip(refs, got):
        assert int(status.item()) == 0
        assert torch.equal(ids, ref_ids)
        err = (out.float() - ref_out.float()).abs().max().item()
        scale = ref_out.float().abs().max().item()
        assert err <= 1e-2 * scale, (err, scale)


def test_noalloc_rejects_shapes_beyond_its_scratch():
    from gpt_oss_moe_gb300 import _build
    _build.build()
    import gpt_oss_moe_gb300 as moe
    big = moe.make_shape(4096, 2880, 2880, 32, 4)
    assert moe.moe_workspace_bytes(big) > (8 << 20)
    code = moe.lib().moe_forward_noalloc(ctypes.byref(big), 16, 32, 48, moe.moe_weight(),
                                         moe.moe_weight(), 64, 1, None, None, None, None)
    assert code == -4                                    # MOE_ERR_WORKSPACE

"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Small shapes span several tiles and every ragged tail (token counts, the
128-row weight blocks, expert counts, forced token-tile sizes); the
full-size gpt-oss shapes are checked on every token's routing and on every
output row (tokens whose k-th and (k+1)-th router logits nearly tie are
excluded and counted).  The oracle runs once per full-size workload, on its
largest batch: a smaller batch's activations are a prefix of the larger
one's, and the layer computes every token on its own.
"""
import dataclasses

import pytest
import torch

from parity_util import (TOL_BF16, compare_output, compare_routing, gpu_forward,
                         tie_masks, to_device)

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a GPU")]


@pytest.fixture(scope="module")
def moe():
    from gpt_oss_moe_gb300 import _build
    _build.build()
    import gpt_oss_moe_gb300 as m
    m.lib()
    return m


def _prefix(layer, T):
    return dataclasses.replace(layer, T=T, x=layer.x[:T].contiguous())


# Oracle results of the full-size workloads: id(layer) -> (layer, logits,
# ids, weights, outputs) over all of the layer's tokens.
_ORACLE_FULL = {}


def _oracle_all(oracle_lib, layer):
    hit = _ORACLE_FULL.get(id(layer))
    if hit is None or hit[0] is not layer:
        logits = oracle_lib.router_logits(layer)
        o_ids, o_w = oracle_lib.topk_softmax(logits, layer.top_k)
        _, _, o_out = oracle_lib.forward(layer)
        hit = (layer, logits, o_ids, o_w, o_out)
        _ORACLE_FULL[id(layer)] = hit
    return hit[1:]


def _check(moe, oracle_lib, layer, dev=None, T=None, tol=TOL_BF16,
           out_dtype=torch.float32, report=None, full_oracle=False):
    """GPU forward of the first T tokens vs the oracle, every output row.
    full_oracle: take the oracle's results from one run over all of the
    layer's tokens (shared by the tests of one full-size workload)."""
    T = layer.T if T is None else T
    ids, w, out, ws = gpu_forward(moe, layer, dev=dev, T=T, out_dtype=out_dtype)
    assert moe.moe_get_device_status(ws) == 0
    if full_oracle:
        logits, o_ids, o_w, o_out = (t[:T] for t in _oracle_all(oracle_lib, layer))
        k = layer.top_k
    else:
        L = _prefix(layer, T) if T != layer.T else layer
        logits = oracle_lib.router_logits(L)
        o_ids, o_w = oracle_lib.topk_softmax(logits, L.top_k)
        o_out = None
        k = L.top_k
    # routing of every token
    rep = compare_routing(ids, w, o_ids, o_w, logits, k)
    excluded, _ = tie_masks(logits, k)
    keep = [t for t in range(T) if not excluded[t]]
    if o_out is None:
        _, _, o_out = oracle_lib.forward(L, tokens=keep)
    else:
        o_out = o_out[keep]
    err, ref = compare_output(out.float()[keep], o_out, slice(None), tol)
    if report is not None:
        report(rep, err, ref)
    return rep, err, ref, ids


SMALL_CASES = [
    # E, k, H, I, T, w_std, token_tile
    (8, 2, 128, 128, 1, 0.05, 0),
    (8, 4, 320, 192, 37, 0.05, 0),      # 320 = 2*128 + 64: weight-row tail
    (16, 4, 256, 384, 300, 0.05, 0),
    (4, 2, 192, 64, 700, 0.05, 0),      # several token tiles per expert
    (8, 4, 256, 256, 200, 0.2, 16),     # clamps active, forced token tiles
    (8, 4, 256, 256, 200, 0.2, 48),
    (8, 4, 256, 256, 200, 0.2, 128),
    (8, 4, 256, 256, 200, 0.2, 256),
    (8, 1, 128, 128, 64, 0.05, 0),      # top-1
    (256, 8, 128, 128, 40, 0.05, 0),    # most experts, largest top_k
    (5, 3, 64, 64, 19, 0.1, 0),         # E not a multiple of 8, 64-wide
    (32, 4, 2880, 2880, 3, 0.02, 0),    # gpt-oss widths, tiny T
]


@pytest.mark.parametrize("case", SMALL_CASES, ids=lambda c: "E{}k{}H{}I{}T{}s{}tile{}".format(*c))
def test_forward_small_shapes(moe, oracle_lib, synth_lib, case):
    E, k, H, I, T, wstd, tile = case
    L = synth_lib.make_layer(E=E, T=T, H=H, I=I, top_k=k, seed=100 + T, w_std=wstd,
                             router_w_std=0.05)
    moe.moe_set_tuning("token_tile", tile)
    try:
        _check(moe, oracle_lib, L)
    finally:
        moe.moe_set_tuning("token_tile", 0)


def test_clamps_are_exercised(oracle_lib, synth_lib):
    L = synth_lib.make_layer(E=8, T=200, H=256, I=256, top_k=4, seed=300, w_std=0.2,
                             router_w_std=0.05)
    x = L.x[:16].float()
    gu = torch.einsum("nh,th->tn", L.w_gu[0].float(), x) + L.b_gu[0].float()
    assert (gu[:, 0::2] > 7).any() and (gu[:, 1::2].abs() > 7).any()


def test_bf16_output_is_rounded_fp32_output(moe, synth_lib):
    L = synth_lib.make_layer(E=8, T=50, H=256, I=256, top_k=4, seed=7, w_std=0.05)
    dev = to_device(L)
    _, _, o32, _ = gpu_forward(moe, L, dev=dev)
    _, _, o16, _ = gpu_forward(moe, L, dev=dev, out_dtype=torch.bfloat16)
    # the fp32 combine order may differ between the runs in the last bit
    diff = (o16.float() - o32.to(torch.bfloat16).float()).abs()
    ulp = o32.abs().clamp_min(1e-30) * 2.0 ** -7
    assert (diff <= ulp).all()


def test_zero_tokens_enqueues_nothing(moe, synth_lib):
    L = synth_lib.make_layer(E=8, T=4, H=128, I=128, top_k=2, seed=1)
    dev = to_device(L)
    shape = moe.layer_shape(L, 0)
    out = torch.full((1, 128), 3.0, device="cuda")
    moe.moe_forward(shape, dev["x"], dev["wr"], dev["br"], dev["w_gu"], dev["b_gu"],
                    dev["w_d"], dev["b_d"], out,
                    workspace=torch.zeros(1024, dtype=torch.uint8, device="cuda"))
    torch.cuda.synchronize()
    assert (out == 3.0).all()


def test_outputs_stay_inside_their_buffers(moe, synth_lib):
    """Canary rows around out/topk buffers must be untouched."""
    L = synth_lib.make_layer(E=16, T=45, H=320, I=192, top_k=4, seed=5, w_std=0.05)
    dev = to_device(L)
    shape = moe.layer_shape(L)
    pad = 8
    big = torch.full((L.T + 2 * pad, L.H), float("nan"), device="cuda")
    ids_big = torch.full((L.T + 2 * pad, 4), -7, dtype=torch.int32, device="cuda")
    w_big = torch.full((L.T + 2 * pad, 4), -7.0, device="cuda")
    ws = moe.alloc_workspace(shape)
    moe.moe_forward(shape, dev["x"], dev["wr"], dev["br"], dev["w_gu"], dev["b_gu"],
                    dev["w_d"], dev["b_d"], big[pad:pad + L.T], topk_ids_out=ids_big[pad:pad + L.T],
                    topk_w_out=w_big[pad:pad + L.T], workspace=ws)
    torch.cuda.synchronize()
    assert torch.isnan(big[:pad]).all() and torch.isnan(big[pad + L.T:]).all()
    assert torch.isfinite(big[pad:pad + L.T]).all()
    assert (ids_big[:pad] == -7).all() and (ids_big[pad + L.T:] == -7).all()
    assert (w_big[:pad] == -7).all() and (w_big[pad + L.T:] == -7).all()


# ---------------------------------------------------------------- routing


ROUTE_CASES = [("20b_t8", 8), ("20b_decode", 1), ("20b_decode", 64),
               ("20b_prefill_skewed", 4096), ("120b_shape", 512), ("120b_shape", 8192)]


@pytest.mark.parametrize("name,T", ROUTE_CASES, ids=lambda v: str(v))
def test_route_full_size(moe, oracle_lib, synth_lib, name, T):
    L = synth_lib.make_workload(name, T, with_experts=False)
    k, E = L.top_k, L.E
    x, wr, br = (t.cuda() for t in (L.x, L.wr, L.br))
    ids = torch.empty((T, k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, k), dtype=torch.float32, device="cuda")
    off = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    sa = torch.empty(T * k, dtype=torch.int32, device="cuda")
    shape = moe.make_shape(T, L.H, 2880, E, k)
    ws = moe.moe_route(shape, x, wr, br, ids, w, off, sa)
    torch.cuda.synchronize()
    assert moe.moe_get_device_status(ws) == 0
    logits = oracle_lib.router_logits(L)
    o_ids, o_w = oracle_lib.topk_softmax(logits, k)
    rep = compare_routing(ids, w, o_ids, o_w, logits, k)
    # the permutation is the oracle's stable sort of the GPU's ids, bit-exact
    o_off, o_sa, _ = oracle_lib.permute(ids.cpu(), E)
    assert torch.equal(off.cpu(), o_off) and torch.equal(sa.cpu(), o_sa)
    assert rep.n_near_tie <= max(2, T // 500)
    # a second run gives bit-identical routing
    ids2, w2 = torch.empty_like(ids), torch.empty_like(w)
    off2, sa2 = torch.empty_like(off), torch.empty_like(sa)
    moe.moe_route(shape, x, wr, br, ids2, w2, off2, sa2, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(ids, ids2) and torch.equal(w, w2)
    assert torch.equal(off, off2) and torch.equal(sa, sa2)


@pytest.mark.parametrize("E,k", [(8, 4), (32, 4), (128, 4), (40, 8), (6, 3)])
def test_route_exact_ties_go_to_the_lower_index(moe, oracle_lib, synth_lib, E, k):
    """Router weights zero: every logit equals its bias exactly, and the
    biases repeat, so the selection is decided by the tie rule alone."""
    T = 40
    L = synth_lib.make_layer(E=E, T=T, H=128, I=128, top_k=k, seed=3, with_experts=False)
    L.wr.zero_()
    L.br.copy_(torch.tensor([float((e * 7) % 3) * 0.5 for e in range(E)]).to(torch.bfloat16))
    ids = torch.empty((T, k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, k), dtype=torch.float32, device="cuda")
    shape = moe.make_shape(T, 128, 128, E, k)
    moe.moe_route(shape, L.x.cuda(), L.wr.cuda(), L.br.cuda(), ids, w)
    torch.cuda.synchronize()
    o_ids, o_w = oracle_lib.topk_softmax(oracle_lib.router_logits(L), k)
    assert torch.equal(ids.cpu(), o_ids)
    assert (w.cpu() - o_w).abs().max() <= 1e-6


def test_hot_experts_take_a_large_share(moe, synth_lib):
    L = synth_lib.make_workload("20b_prefill_skewed", 4096, with_experts=False)
    shape = moe.make_shape(4096, L.H, 2880, L.E, 4)
    off = torch.empty(L.E + 1, dtype=torch.int32, device="cuda")
    moe.moe_route(shape, L.x.cuda(), L.wr.cuda(), L.br.cuda(), expert_offsets=off)
    counts = off.diff().cpu()
    share = counts[:4].sum().item() / counts.sum().item()
    assert 0.2 < share < 0.7


# ---------------------------------------------------------------- full size


@pytest.fixture(scope="module")
def layer_20b_decode(synth_lib):
    L = synth_lib.make_workload("20b_decode", 64)
    return L, to_device(L)


@pytest.mark.parametrize("T", [1, 16, 64])
def test_forward_20b_decode(moe, oracle_lib, layer_20b_decode, parity_report, T):
    L, dev = layer_20b_decode
    _check(moe, oracle_lib, L, dev=dev, T=T, report=parity_report(f"20b_decode bf16 T={T}"))


def test_forward_20b_t8(moe, oracle_lib, synth_lib, parity_report):
    L = synth_lib.make_workload("20b_t8", 8)
    _check(moe, oracle_lib, L, report=parity_report("20b_t8 bf16 T=8"))


def test_forward_20b_prefill_skewed(moe, oracle_lib, synth_lib, parity_report):
    L = synth_lib.make_workload("20b_prefill_skewed", 4096)
    _check(moe, oracle_lib, L, full_oracle=True,
           report=parity_report("20b_prefill_skewed bf16 T=4096"))


@pytest.fixture(scope="module")
def layer_120b(synth_lib):
    L = synth_lib.make_workload("120b_shape", 8192)
    return L, to_device(L)


@pytest.mark.parametrize("T", [1, 8, 64, 512, 4096, 8192])
def test_forward_120b_shape(moe, oracle_lib, layer_120b, parity_report, T):
    L, dev = layer_120b
    _check(moe, oracle_lib, L, dev=dev, T=T, full_oracle=T > 64,
           report=parity_report(f"120b_shape bf16 T={T}"))


# ---------------------------------------------------------------- K split

# Few routed rows and a long K range: the units (token tiles x 128-row weight
# blocks) cannot fill two waves of the GPU, so the GEMMs split each unit's K
# range into parts (down: added by the output atomics; gate_up: partial tiles
# summed by the last part before the GLU).  R = T*k rows; parts per unit:
KSPLIT_CASES = [
    # E, k, H, I, T, wfmt      gate_up parts x slots / down parts
    (4, 2, 512, 256, 3, "bf16"),     # 4 x 2 of 8 k-blocks / 2 x 2 of 4
    (8, 4, 320, 192, 1, "bf16"),     # 2 parts of 3 + 2 k-blocks (uneven); W_d tail
    (4, 1, 1024, 512, 2, "bf16"),    # 8 x 2 of 16 / 4 x 2 of 8
    (4, 2, 1024, 512, 3, "mxfp4"),   # 2 parts of 2 ring slots (4 k-blocks each)
    (8, 4, 2048, 384, 1, "mxfp4"),   # 4 parts of 2 ring slots / down unsplit (2 slots)
]


@pytest.mark.parametrize("case", KSPLIT_CASES, ids=lambda c: "E{}k{}H{}I{}T{}{}".format(*c))
def test_forward_ksplit(moe, oracle_lib, synth_lib, case):
    from parity_util import TOL_MXFP4
    E, k, H, I, T, wfmt = case
    L = synth_lib.make_layer(E=E, T=T, H=H, I=I, top_k=k, seed=700 + T + H, wfmt=wfmt,
                             router_w_std=0.05)
    tol = TOL_MXFP4 if wfmt == "mxfp4" else TOL_BF16
    _check(moe, oracle_lib, L, tol=tol)


@pytest.mark.parametrize("parts", [3, 8])
def test_forward_fixed_ksplit(moe, oracle_lib, synth_lib, parts):
    """The K split forced to 3 and 8 parts ("ksplit" 2..8), beside the
    automatic choice the cases above use (gate_up takes as many parts as
    the partial-tile region holds)."""
    L = synth_lib.make_layer(E=8, T=3, H=1024, I=512, top_k=2, seed=733, router_w_std=0.05)
    moe.moe_set_tuning("ksplit", parts)
    try:
        _check(moe, oracle_lib, L)
    finally:
        moe.moe_set_tuning("ksplit", 0)


def test_ksplit_tickets_reset(moe, oracle_lib, synth_lib):
    """The gate_up part tickets are left at zero: the same workspace serves a
    second split call, and a call of another shape, with the same results."""
    L = synth_lib.make_layer(E=4, T=3, H=512, I=256, top_k=2, seed=7, router_w_std=0.05)
    L2 = synth_lib.make_layer(E=8, T=1, H=320, I=192, top_k=4, seed=8, router_w_std=0.05)
    shape = moe.layer_shape(L)
    shape2 = moe.layer_shape(L2)
    ws = moe.alloc_workspace(shape) if moe.moe_workspace_bytes(shape) >= moe.moe_workspace_bytes(shape2) \
        else moe.alloc_workspace(shape2)
    i1, w1, o1, _ = gpu_forward(moe, L, workspace=ws)
    i2, w2, o2, _ = gpu_forward(moe, L2, workspace=ws)
    i3, w3, o3, _ = gpu_forward(moe, L, workspace=ws)
    assert moe.moe_get_device_status(ws) == 0
    assert torch.equal(i1, i3) and torch.equal(w1, w3)
    assert torch.allclose(o1, o3, rtol=0, atol=1e-6 * float(o1.abs().max()))
    _check(moe, oracle_lib, L2)


PAIR_CASES = [
    # E, k, H, I, T, token_tile   (bf16 GEMMs forced onto CTA pairs)
    (8, 2, 128, 128, 1, 0),          # one 16-column tile: 8 token rows per CTA
    (8, 4, 320, 192, 37, 0),         # 2I = 384: the odd CTA's rows of the last
                                     # gate_up block are all past the matrix;
                                     # H = 320: down's last block has 64 rows
    (8, 4, 448, 256, 200, 48),       # H = 448: the odd CTA holds 64 rows of
                                     # down's last block; 24 token rows per CTA
    (4, 2, 192, 64, 700, 0),         # several 256-row token tiles per expert
    (8, 4, 256, 256, 200, 16),       # smallest box: 8 token rows per CTA
    (16, 4, 256, 384, 300, 0),
]


@pytest.mark.parametrize("case", PAIR_CASES, ids=lambda c: "E{}k{}H{}I{}T{}tile{}".format(*c))
def test_forward_cta_pairs(moe, oracle_lib, synth_lib, case):
    E, k, H, I, T, tile = case
    L = synth_lib.make_layer(E=E, T=T, H=H, I=I, top_k=k, seed=800 + T + H, router_w_std=0.05)
    moe.moe_set_tuning("pair", 2)
    moe.moe_set_tuning("token_tile", tile)
    try:
        _check(moe, oracle_lib, L)
    finally:
        moe.moe_set_tuning("pair", 0)
        moe.moe_set_tuning("token_tile", 0)


def test_cta_pairs_match_single(moe, synth_lib):
    """Pairs and single CTAs sum every output over K in the same order: the
    routing is identical and the outputs agree to fp32 rounding of the
    combine's atomics."""
    L = synth_lib.make_layer(E=32, T=256, H=2880, I=2880, top_k=4, seed=811, router_w_std=0.05)
    outs = []
    for mode in (1, 2):
        moe.moe_set_tuning("pair", mode)
        try:
            outs.append(gpu_forward(moe, L))
        finally:
            moe.moe_set_tuning("pair", 0)
    (i1, w1, o1, ws1), (i2, w2, o2, ws2) = outs
    assert moe.moe_get_device_status(ws1) == 0 and moe.moe_get_device_status(ws2) == 0
    assert torch.equal(i1, i2) and torch.equal(w1, w2)
    assert torch.allclose(o1, o2, rtol=0, atol=1e-5 * float(o1.abs().max()))


# ---------------------------------------------------------------- MXFP4

MXFP4_CASES = [
    # E, k, H, I, T, token_tile
    (8, 2, 128, 128, 1, 0),
    (8, 4, 320, 192, 37, 0),        # weight-row tail in the down projection
    (4, 2, 192, 128, 700, 0),       # several token tiles per expert
    (8, 4, 256, 256, 200, 48),
    (32, 4, 2880, 2880, 5, 0),
]


@pytest.mark.parametrize("case", MXFP4_CASES, ids=lambda c: "E{}k{}H{}I{}T{}tile{}".format(*c))
def test_forward_mxfp4_small_shapes(moe, oracle_lib, synth_lib, case):
    from parity_util import TOL_MXFP4
    E, k, H, I, T, tile = case
    L = synth_lib.make_layer(E=E, T=T, H=H, I=I, top_k=k, seed=400 + T, wfmt="mxfp4",
                             router_w_std=0.05)
    moe.moe_set_tuning("token_tile", tile)
    try:
        _check(moe, oracle_lib, L, tol=TOL_MXFP4)
    finally:
        moe.moe_set_tuning("token_tile", 0)


@pytest.mark.parametrize("T,scale_lo,scale_hi", [(3, 116, 126), (300, 116, 126), (300, 124, 136)])
def test_mxfp4_dequant_is_exact(moe, oracle_lib, synth_lib, T, scale_lo, scale_hi):
    """In-kernel dequantisation is exact: with top-1 routing each output
    element is a single combine term (weight 1), so the MXFP4 path must equal
    bit for bit the bf16 path run on the oracle's dequantised weights.  Scale
    bytes above 128 (factors above 2) take the kernel's two-multiply path,
    mixed with one-multiply lanes in the same warps."""
    Lq = synth_lib.make_layer(E=4, T=T, H=320, I=192, top_k=1, seed=9, wfmt="mxfp4",
                              scale_lo=scale_lo, scale_hi=scale_hi)
    Lb = dataclasses.replace(
        Lq, wfmt="bf16", s_gu=None, s_d=None,
        w_gu=oracle_lib.dequant_mxfp4(Lq.w_gu, Lq.s_gu).to(torch.bfloat16).contiguous(),
        w_d=oracle_lib.dequant_mxfp4(Lq.w_d, Lq.s_d).to(torch.bfloat16).contiguous())
    # one K order in both paths: no K split (it would differ between the
    # 4-k-block MXFP4 ring and the 1-k-block bf16 ring); bf16 operands (the
    # f16 mode rounds the activations and h to f16 instead)
    moe.moe_set_tuning("ksplit", 1)
    moe.moe_set_tuning("mxfp4_f16", 0)
    try:
        iq, wq, oq, wsq = gpu_forward(moe, Lq)
        ib, wb, ob, wsb = gpu_forward(moe, Lb)
    finally:
        moe.moe_set_tuning("ksplit", 0)
        moe.moe_set_tuning("mxfp4_f16", 1)
    assert moe.moe_get_device_status(wsq) == 0
    assert torch.equal(iq, ib) and torch.equal(wq, wb)
    assert torch.equal(oq, ob)


@pytest.mark.parametrize("lo,hi,flag", [(104, 110, False), (134, 140, False), (103, 110, True),
                                         (134, 141, True)])
def test_mxfp4_f16_mode_scale_range(moe, oracle_lib, synth_lib, lo, hi, flag):
    """The f16 mode expands E2M1 codes exactly for scale bytes 104..140 (its
    operands then differ from the oracle's only by the rounding of the
    activations and h to f16, well inside 2e-3 of the output's magnitude); a
    scale byte outside is clamped and reported as MOE_DEV_RANGE, and the
    bf16 mode computes the same layer exactly with no report."""
    L = synth_lib.make_layer(E=4, T=40, H=320, I=192, top_k=2, seed=17 + lo + hi, wfmt="mxfp4",
                             scale_lo=lo, scale_hi=hi, router_w_std=0.05)
    if lo < 110:
        # small scales: activations large enough that the products matter
        L.x = (L.x.float() * 64).to(torch.bfloat16)
    _, _, o_out = oracle_lib.forward(L)
    ref = o_out.abs().max().item()
    ids, w, out, ws = gpu_forward(moe, L)
    status = moe.moe_get_device_status(ws)
    if flag:
        assert status == moe.MOE_DEV_RANGE
    else:
        assert status == 0
        assert (out.cpu() - o_out).abs().max().item() <= 2e-3 * ref
    moe.moe_set_tuning("mxfp4_f16", 0)
    try:
        ids, w, out, ws = gpu_forward(moe, L)
    finally:
        moe.moe_set_tuning("mxfp4_f16", 1)
    assert moe.moe_get_device_status(ws) == 0
    assert (out.cpu() - o_out).abs().max().item() <= 1e-2 * ref


def test_mxfp4_f16_mode_activation_range(moe, oracle_lib, synth_lib):
    """An activation beyond the f16 range is reported (MOE_DEV_RANGE)."""
    L = synth_lib.make_layer(E=4, T=10, H=128, I=128, top_k=2, seed=23, wfmt="mxfp4",
                             router_w_std=0.05)
    L.x = L.x.clone()
    L.x[2, 5] = 1e6
    ids, w, out, ws = gpu_forward(moe, L)
    assert moe.moe_get_device_status(ws) & moe.MOE_DEV_RANGE


@pytest.mark.parametrize("ksplit", [1, 0])
def test_mxfp4_odd_ring_slots_per_unit(moe, oracle_lib, synth_lib, ksplit):
    """K = 640 is 10 k-blocks, 3 ring slots per unit (down: K = 320, 2
    slots): consecutive units start at ring uses of both parities, and the
    two MMA issuers must still each keep their own A slot.  ksplit 1 runs
    whole units, 0 the automatic K split."""
    from parity_util import TOL_MXFP4
    L = synth_lib.make_layer(E=8, T=37, H=640, I=320, top_k=4, seed=640, wfmt="mxfp4",
                             router_w_std=0.05)
    moe.moe_set_tuning("ksplit", ksplit)
    try:
        _check(moe, oracle_lib, L, tol=TOL_MXFP4)
    finally:
        moe.moe_set_tuning("ksplit", 0)


# ---------------------------------------------------------------- FP8 W8A8

FP8_CASES = [
    # E, k, H, I, T, token_tile
    (8, 2, 128, 128, 1, 0),
    (8, 4, 320, 192, 37, 0),        # K tails: 320 = 2.5 and 192 = 1.5 k-blocks of 128
    (4, 2, 192, 64, 700, 0),        # several token tiles per expert
    (8, 4, 256, 256, 200, 48),
    (32, 4, 2880, 2880, 5, 0),      # 2880 = 22.5 k-blocks
]


@pytest.mark.parametrize("case", FP8_CASES, ids=lambda c: "E{}k{}H{}I{}T{}tile{}".format(*c))
def test_forward_fp8_small_shapes(moe, oracle_lib, synth_lib, case):
    E, k, H, I, T, tile = case
    L = synth_lib.make_layer(E=E, T=T, H=H, I=I, top_k=k, seed=500 + T, wfmt="fp8",
                             router_w_std=0.05)
    moe.moe_set_tuning("token_tile", tile)
    try:
        _check(moe, oracle_lib, L)
    finally:
        moe.moe_set_tuning("token_tile", 0)


@pytest.mark.parametrize("case", PAIR_CASES, ids=lambda c: "E{}k{}H{}I{}T{}tile{}".format(*c))
def test_forward_fp8_cta_pairs(moe, oracle_lib, synth_lib, case):
    """FP8 GEMMs forced onto CTA pairs (M = 256 kind::f8f6f4 MMAs)."""
    E, k, H, I, T, tile = case
    L = synth_lib.make_layer(E=E, T=T, H=H, I=I, top_k=k, seed=820 + T + H, wfmt="fp8",
                             router_w_std=0.05)
    moe.moe_set_tuning("pair", 2)
    moe.moe_set_tuning("token_tile", tile)
    try:
        _check(moe, oracle_lib, L)
    finally:
        moe.moe_set_tuning("pair", 0)
        moe.moe_set_tuning("token_tile", 0)


def test_fp8_outliers_and_zero_rows(moe, oracle_lib, synth_lib):
    """Per-token scales: a token with 20x outliers and an all-zero token
    (scale 1, every code 0) beside ordinary ones."""
    L = synth_lib.make_layer(E=8, T=20, H=256, I=128, top_k=2, seed=511, wfmt="fp8",
                             router_w_std=0.05, p_outlier=0.05)
    L.x = L.x.clone()
    L.x[3] = 0
    _check(moe, oracle_lib, L)


@pytest.fixture(scope="module")
def layer_20b_fp8(synth_lib):
    L = synth_lib.make_workload("20b_fp8", 4096)
    return L, to_device(L)


@pytest.mark.parametrize("T", [1, 64, 512, 4096])
def test_forward_20b_fp8(moe, oracle_lib, layer_20b_fp8, parity_report, T):
    L, dev = layer_20b_fp8
    _check(moe, oracle_lib, L, dev=dev, T=T, full_oracle=T > 64,
           report=parity_report(f"20b_fp8 fp8 T={T}"))


@pytest.fixture(scope="module")
def layer_20b_mxfp4(synth_lib):
    L = synth_lib.make_workload("20b_mxfp4", 4096)
    return L, to_device(L)


@pytest.mark.parametrize("T", [1, 64, 512, 4096])
def test_forward_20b_mxfp4(moe, oracle_lib, layer_20b_mxfp4, parity_report, T):
    from parity_util import TOL_MXFP4
    L, dev = layer_20b_mxfp4
    _check(moe, oracle_lib, L, dev=dev, T=T, full_oracle=T > 64, tol=TOL_MXFP4,
           report=parity_report(f"20b_mxfp4 mxfp4 T={T}"))


# ------------------------------------------- MXFP4 weights, MXFP8 activations

MX_CASES = [
    # E, k, H, I, T, token_tile
    (8, 2, 128, 128, 1, 0),
    (8, 4, 320, 192, 37, 0),        # K = 128 m + 64 on both GEMMs: the chunk view's tail
    (4, 2, 192, 128, 700, 0),       # several token tiles per expert
    (8, 4, 256, 256, 200, 48),
    (8, 4, 256, 256, 200, 16),
    (8, 4, 448, 320, 130, 128),     # widest MX token box
    (32, 4, 2880, 2880, 5, 0),      # 2880 = 22.5 k-blocks of 128
]


@pytest.mark.parametrize("case", MX_CASES, ids=lambda c: "E{}k{}H{}I{}T{}tile{}".format(*c))
def test_forward_mxfp8_small_shapes(moe, oracle_lib, synth_lib, case):
    E, k, H, I, T, tile = case
    L = synth_lib.make_layer(E=E, T=T, H=H, I=I, top_k=k, seed=600 + T, wfmt="mxfp4_mxfp8",
                             router_w_std=0.05)
    moe.moe_set_tuning("token_tile", tile)
    try:
        _check(moe, oracle_lib, L)
    finally:
        moe.moe_set_tuning("token_tile", 0)


@pytest.mark.parametrize("parts", [3, 8])
def test_mxfp8_fixed_ksplit(moe, oracle_lib, synth_lib, parts):
    L = synth_lib.make_layer(E=8, T=9, H=1024, I=768, top_k=2, seed=640 + parts,
                             wfmt="mxfp4_mxfp8", router_w_std=0.05)
    moe.moe_set_tuning("ksplit", parts)
    try:
        _check(moe, oracle_lib, L)
    finally:
        moe.moe_set_tuning("ksplit", 0)


def test_mxfp8_outliers_and_zero_rows(moe, oracle_lib, synth_lib):
    """Per-block scales: 20x outliers, an all-zero token and a token whose
    blocks span many binades."""
    L = synth_lib.make_layer(E=8, T=20, H=256, I=192, top_k=2, seed=611, wfmt="mxfp4_mxfp8",
                             router_w_std=0.05, p_outlier=0.05)
    L.x = L.x.clone()
    L.x[3] = 0
    L.x[5] = (L.x[5].float() * torch.exp2(torch.arange(256).float() / 16 - 8)).to(torch.bfloat16)
    _check(moe, oracle_lib, L)


@pytest.fixture(scope="module")
def layer_20b_mxfp8(synth_lib):
    L = synth_lib.make_workload("20b_mxfp4_mxfp8", 4096)
    return L, to_device(L)


@pytest.mark.parametrize("T", [1, 64, 512, 4096])
def test_forward_20b_mxfp4_mxfp8(moe, oracle_lib, layer_20b_mxfp8, parity_report, T):
    L, dev = layer_20b_mxfp8
    _check(moe, oracle_lib, L, dev=dev, T=T, full_oracle=T > 64,
           report=parity_report(f"20b_mxfp4_mxfp8 mxfp4xmxfp8 T={T}"))


# ------------------------------------------------ expert-parallel partial form

def _ep_partials(moe, L, dev, world, tokens=None):
    """Partial outputs of `world` devices (run one after another on this
    GPU) that partition the experts, each given its slice of the banks."""
    shape = moe.layer_shape(L)
    parts = []
    for r in range(world):
        lo, n = moe.ep_expert_range(r, world, L.E)
        sl = lambda t: None if t is None else t[lo:lo + n]
        out = torch.empty((L.T, L.H), dtype=torch.float32, device="cuda")
        ws = moe.moe_forward_ep(shape, lo, n, dev["x"], dev["wr"], dev["br"], sl(dev["w_gu"]),
                                sl(dev["b_gu"]), sl(dev["w_d"]), sl(dev["b_d"]), out,
                                s_gu=sl(dev["s_gu"]), s_d=sl(dev["s_d"]))
        assert moe.moe_get_device_status(ws) == 0
        parts.append((lo, n, out.cpu()))
    return parts


@pytest.mark.parametrize("wfmt", ["bf16", "fp8", "mxfp4", "mxfp4_mxfp8"])
def test_forward_ep_partials_match_and_sum_to_the_layer(moe, oracle_lib, synth_lib, wfmt):
    from parity_util import TOL_MXFP4
    L = synth_lib.make_layer(E=8, T=40, H=256, I=192, top_k=3, seed=900, wfmt=wfmt,
                             router_w_std=0.05)
    tol = TOL_MXFP4 if wfmt == "mxfp4" else TOL_BF16
    _, _, full = oracle_lib.forward(L)
    ref = full.abs().max().item()
    total = torch.zeros_like(full)
    for lo, n, part in _ep_partials(moe, L, to_device(L), 3):
        o_part = oracle_lib.forward_ep(L, lo, n)
        assert (part - o_part).abs().max().item() <= tol * ref, (lo, n)
        total += part
    assert (total - full).abs().max().item() <= tol * ref


def test_forward_ep_rank_without_tokens_outputs_zero(moe, oracle_lib, synth_lib):
    """+20 on the router bias of experts 0 and 1 with top-2 routes every
    token there: the rank holding experts 4..7 has no tile at all and must
    write an all-zero partial; the rank holding 0..3 carries the layer."""
    L = synth_lib.make_layer(E=8, T=50, H=256, I=128, top_k=2, seed=905, hot=(0, 1),
                             hot_bias=20.0, router_w_std=0.05)
    parts = _ep_partials(moe, L, to_device(L), 2)
    assert parts[1][2].eq(0).all()
    _, _, full = oracle_lib.forward(L)
    assert (parts[0][2] - full).abs().max().item() <= TOL_BF16 * full.abs().max().item()


def test_empty_calls_enqueue_nothing(moe, synth_lib):
    L = synth_lib.make_layer(E=8, T=4, H=128, I=128, top_k=2, seed=906)
    dev = to_device(L)
    shape = moe.make_shape(0, 128, 128, 8, 2)
    out = torch.empty((1, 128), device="cuda")
    moe.moe_forward_ep(shape, 2, 3, dev["x"], dev["wr"], dev["br"], dev["w_gu"][2:5],
                       dev["b_gu"][2:5], dev["w_d"][2:5], dev["b_d"][2:5], out)
    a = synth_lib.make_attention(4, 4, Hq=8, Hkv=1, D=64)
    o = moe.attention_sinks(a["q"][:0].cuda(), a["k"].cuda(), a["v"].cuda(),
                            a["sinks"].cuda())
    torch.cuda.synchronize()
    assert o.shape == (0, 8, 64)


def test_forward_ep_20b_four_ranks(moe, oracle_lib, layer_20b_decode):
    """gpt-oss-20b widths, T = 64, four ranks of 8 experts."""
    L64, dev64 = layer_20b_decode
    assert L64.T == 64
    parts = _ep_partials(moe, L64, dev64, 4)
    sample = list(range(0, 64, 4))
    _, _, full = oracle_lib.forward(L64, tokens=sample)
    ref = full.abs().max().item()
    total = sum(p for _, _, p in parts)[sample]
    assert (total - full).abs().max().item() <= TOL_BF16 * ref
    lo, n, part = parts[1]
    o_part = oracle_lib.forward_ep(L64, lo, n, tokens=sample)
    assert (part[sample] - o_part).abs().max().item() <= TOL_BF16 * ref


def test_one_workspace_serves_successive_shapes(moe, synth_lib):
    """A workspace sized for the largest call is reused for smaller ones
    (other token counts shift every region but the status word and the
    completion counters); each call must match a call on a fresh workspace."""
    L = synth_lib.make_layer(E=64, T=300, H=256, I=256, top_k=4, seed=77, w_std=0.05,
                             router_w_std=0.05)
    dev = to_device(L)
    big = moe.alloc_workspace(moe.layer_shape(L, 300))
    for T in (300, 33, 1, 300, 64):
        ids_a, w_a, out_a, _ = gpu_forward(moe, L, dev=dev, T=T, workspace=big)
        ids_b, w_b, out_b, _ = gpu_forward(moe, L, dev=dev, T=T)
        assert moe.moe_get_device_status(big) == 0
        assert torch.equal(ids_a, ids_b) and torch.equal(w_a, w_b)
        assert (out_a - out_b).abs().max().item() <= 1e-5 * out_b.abs().max().item()


# ------------------------------------------- small batches without a permutation kernel

SMALL_PATH_CASES = [
    # E, k, H, I, T     (bf16 weights, T * k <= 256 and T <= 64: the router
    #                    permutes and gate_up gathers the token rows itself;
    #                    T <= 8: the single-block router)
    (32, 4, 2880, 2880, 1),
    (32, 4, 2880, 2880, 8),
    (32, 4, 2880, 2880, 16),
    (16, 2, 6400, 128, 8),       # wide rows (five load batches per row in the single-block router)
    (128, 4, 2880, 2880, 3),
    (8, 4, 320, 192, 37),        # weight-row tail, 48-row token tiles
    (8, 1, 128, 128, 64),        # top-1, 64-row tiles (rows 32..63 of a tile)
    (256, 8, 128, 128, 32),      # R = 256, most experts
    (5, 3, 64, 64, 19),
    (128, 4, 2880, 2880, 2),     # single-block router with 128 experts (matrix read from global)
    (20, 4, 64, 64, 5),          # single-block router, matrix staged: a partial 16-expert tile
    (32, 4, 2880, 2880, 48),     # grid of 4-token router blocks beside the permutation kernel
    (64, 4, 128, 128, 8),        # ... four 16-expert tiles, eight tokens
]


@pytest.mark.parametrize("case", SMALL_PATH_CASES, ids=lambda c: "E{}k{}H{}I{}T{}".format(*c))
def test_small_path_matches_the_permutation_kernel(moe, oracle_lib, synth_lib, case):
    E, k, H, I, T = case
    L = synth_lib.make_layer(E=E, T=T, H=H, I=I, top_k=k, seed=1500 + T + E, router_w_std=0.05)
    dev = to_device(L)
    runs = []
    for small, tiny in ((1, 1), (1, 0), (0, 1)):
        moe.moe_set_tuning("small_path", small)
        moe.moe_set_tuning("tiny_router", tiny)
        try:
            runs.append(gpu_forward(moe, L, dev=dev))
        finally:
            moe.moe_set_tuning("small_path", 1)
            moe.moe_set_tuning("tiny_router", 1)
    (i0, w0, o0, ws0) = runs[-1]
    logits = oracle_lib.router_logits(L)
    excluded, inner = tie_masks(logits, k)
    exact = ~excluded & ~inner
    for ids, w, out, ws in runs:
        assert moe.moe_get_device_status(ws) == 0
        # the single-block router sums the logits in another order: ids may
        # differ only where the oracle's logits nearly tie
        assert torch.equal(ids.cpu()[exact], i0.cpu()[exact])
        assert (w.cpu()[exact] - w0.cpu()[exact]).abs().max().item() <= 2e-5 if exact.any() else True
        keep = exact.nonzero().flatten().cuda()
        assert (out[keep] - o0[keep]).abs().max().item() <= 1e-5 * o0.abs().max().item()
    _check(moe, oracle_lib, L, dev=dev)

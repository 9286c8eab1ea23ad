"""Helpers for comparing the CUDA path with the CPU oracle.

Parity rules (the layer's tolerance statement):
  * routing ids: bit-exact, except tokens whose k-th and (k+1)-th oracle
    logits are closer than 1e-5 ("near ties"), which are excluded and
    counted; tokens with a gap < 1e-5 *inside* the top k may list the same
    experts in another order, so their ids are compared as sets;
  * routing weights: |gpu - oracle| <= 2e-5 (both take the softmax of fp32
    logits that differ only by summation order);
  * permutation: bit-exact against the oracle's stable sort of the GPU ids;
  * outputs: max |gpu - oracle| <= tol * max |oracle| over the rows of
    non-excluded tokens, tol = 1e-2 for bf16 weights and 3e-2 for MXFP4.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

TIE_GAP = 1e-5
W_ATOL = 2e-5
TOL_BF16 = 1e-2
TOL_MXFP4 = 3e-2


@dataclass
class RoutingReport:
    n_tokens: int
    n_near_tie: int
    n_inner_tie: int


def tie_masks(logits: torch.Tensor, k: int):
    """(excluded, inner) boolean masks over tokens from oracle logits [n, E]."""
    srt = torch.sort(logits.double(), dim=1, descending=True).values
    n, E = srt.shape
    if k < E:
        excluded = (srt[:, k - 1] - srt[:, k]) < TIE_GAP
    else:
        excluded = torch.zeros(n, dtype=torch.bool)
    if k > 1:
        inner = ((srt[:, : k - 1] - srt[:, 1:k]) < TIE_GAP).any(dim=1) & ~excluded
    else:
        inner = torch.zeros(n, dtype=torch.bool)
    return excluded, inner


def compare_routing(g_ids, g_w, o_ids, o_w, logits, k) -> RoutingReport:
    g_ids, g_w = g_ids.cpu(), g_w.cpu().double()
    o_w = o_w.double()
    excluded, inner = tie_masks(logits, k)
    exact = ~excluded & ~inner
    assert torch.equal(g_ids[exact], o_ids[exact]), "routing ids differ"
    assert (g_w[exact] - o_w[exact]).abs().max().item() <= W_ATOL if exact.any() else True
    for t in torch.nonzero(inner).flatten().tolist():
        gi, oi = g_ids[t].tolist(), o_ids[t].tolist()
        assert sorted(gi) == sorted(oi), f"token {t}: expert sets differ"
        gw = dict(zip(gi, g_w[t].tolist()))
        for e, w in zip(oi, o_w[t].tolist()):
            assert abs(gw[e] - w) <= W_ATOL
    # every token, excluded or not, still has k distinct in-range ids
    assert all(len(set(r)) == k for r in g_ids.tolist())
    assert ((g_w.sum(dim=1) - 1).abs() <= 1e-5).all()
    return RoutingReport(int(g_ids.shape[0]), int(excluded.sum()), int(inner.sum()))


def compare_output(g_out, o_out, keep_rows, tol):
    """Returns (max abs err, max |oracle|); asserts the bound."""
    g = g_out.cpu().double()[keep_rows]
    o = o_out.double()[keep_rows]
    assert torch.isfinite(g).all(), "non-finite GPU output"
    err = (g - o).abs().max().item()
    ref = o.abs().max().item()
    assert err <= tol * ref, f"max err {err:.3e} > {tol} * {ref:.3e}"
    return err, ref


def to_device(layer, device="cuda"):
    d = {}
    for name in ("x", "wr", "br", "w_gu", "b_gu", "w_d", "b_d", "s_gu", "s_d"):
        t = getattr(layer, name)
        d[name] = None if t is None else t.to(device, non_blocking=True)
    torch.cuda.synchronize()
    return d


def gpu_forward(moe, layer, dev=None, T=None, out_dtype=torch.float32,
                workspace=None):
    """Run moe_forward on the first T tokens; returns (ids, w, out, ws)."""
    T = layer.T if T is None else T
    dev = dev or to_device(layer)
    shape = moe.layer_shape(layer, T)
    x = dev["x"][:T].contiguous()
    out = torch.empty((T, layer.H), dtype=out_dtype, device="cuda")
    ids = torch.empty((T, layer.top_k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, layer.top_k), dtype=torch.float32, device="cuda")
    ws = workspace if workspace is not None else moe.alloc_workspace(shape)
    moe.moe_forward(shape, x, dev["wr"], dev["br"], dev["w_gu"], dev["b_gu"],
                    dev["w_d"], dev["b_d"], out, s_gu=dev["s_gu"],
                    s_d=dev["s_d"], topk_ids_out=ids, topk_w_out=w,
                    workspace=ws)
    torch.cuda.synchronize()
    return ids, w, out, ws

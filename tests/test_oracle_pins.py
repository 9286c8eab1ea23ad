"""Pins of the CPU oracle against the page and against mathematics.

Each test checks the oracle against something other than itself: closed
forms, identities of the activation, brute force over all k-subsets, an
independent fp64 brute force of the whole layer, and the published E2M1/E8M0
tables.  Source of the definitions: xserv docs/19-gpt-oss-moe.md ("Phase 19:
gpt-oss-20b"), §1 model-architecture table ("MoE" and "激活" rows), §2 "MoE
前向" and §5 "量化".
"""
import itertools
import math

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.filterwarnings("ignore")


def _tiny(synth_lib, E=4, T=6, H=64, I=64, k=2, seed=0, **kw):
    return synth_lib.make_layer(E=E, T=T, H=H, I=I, top_k=k, seed=seed, **kw)


def _bf16(a):
    return torch.as_tensor(np.asarray(a, dtype=np.float32)).to(torch.bfloat16)


# --------------------------------------------------------------------------
# top-k + softmax (§2 "topk_softmax"; ties go to the lower expert index)


def test_topk_brute_force_over_all_subsets(oracle_lib):
    rng = np.random.default_rng(11)
    for E, k in [(4, 2), (6, 3), (8, 4), (8, 1), (5, 5)]:
        # small integer logits force many exact ties
        logits = rng.integers(-3, 4, size=(64, E)).astype(np.float32)
        ids, w = oracle_lib.topk_softmax(torch.from_numpy(logits), k)
        for t in range(logits.shape[0]):
            l = logits[t].astype(np.float64)
            sel = ids[t].tolist()
            # the chosen set maximises the sum of logits over all k-subsets
            best = max(sum(l[list(c)]) for c in itertools.combinations(range(E), k))
            assert sum(l[sel]) == best
            # among equal logits, the lower index is taken
            for e in sel:
                for f in range(E):
                    if f not in sel:
                        assert l[e] > l[f] or (l[e] == l[f] and e < f)
            # slot order: descending logit, lower index first on ties
            for a, b in zip(sel, sel[1:]):
                assert l[a] > l[b] or (l[a] == l[b] and a < b)


def test_topk_all_equal_logits_closed_form(oracle_lib):
    # router W = 0, b = 0: every logit is 0 -> ids 0..k-1 and w = 1/k exactly
    for E, k in [(32, 4), (128, 4), (8, 3)]:
        ids, w = oracle_lib.topk_softmax(torch.zeros(5, E), k)
        assert ids.tolist() == [list(range(k))] * 5
        assert torch.equal(w, torch.full((5, k), np.float32(1.0) / np.float32(k)))


def test_topk_zero_router_through_layer(oracle_lib, synth_lib):
    L = _tiny(synth_lib, E=8, T=3, k=4)
    L.wr.zero_()
    L.br.zero_()
    ids, w, _ = oracle_lib.forward(L)
    assert ids.tolist() == [[0, 1, 2, 3]] * 3
    assert torch.equal(w, torch.full((3, 4), 0.25))


def test_top1_weight_is_one(oracle_lib):
    logits = torch.randn(20, 32, generator=torch.Generator().manual_seed(1))
    ids, w = oracle_lib.topk_softmax(logits, 1)
    assert torch.equal(w, torch.ones(20, 1))
    assert torch.equal(ids[:, 0].long(), logits.argmax(dim=1))


def test_topk_equal_to_E_is_full_softmax(oracle_lib):
    g = torch.Generator().manual_seed(2)
    logits = torch.randn(10, 8, generator=g) * 3
    ids, w = oracle_lib.topk_softmax(logits, 8)
    l64 = logits.double()
    full = torch.exp(l64 - l64.max(dim=1, keepdim=True).values)
    full = full / full.sum(dim=1, keepdim=True)
    got = torch.zeros(10, 8, dtype=torch.float64)
    got.scatter_(1, ids.long(), w.double())
    assert torch.allclose(got, full, rtol=0, atol=2e-7)


def test_topk_invariants(oracle_lib):
    g = torch.Generator().manual_seed(3)
    logits = torch.randn(500, 32, generator=g)
    ids, w = oracle_lib.topk_softmax(logits, 4)
    assert torch.all((w.sum(dim=1) - 1).abs() <= 1e-6)
    assert torch.all(w[:, :-1] >= w[:, 1:])
    assert torch.all((ids >= 0) & (ids < 32))
    for row in ids.tolist():
        assert len(set(row)) == 4


def test_topk_rejects_bad_k(oracle_lib):
    with pytest.raises(ValueError):
        oracle_lib.topk_softmax(torch.zeros(2, 4), 5)
    with pytest.raises(ValueError):
        oracle_lib.topk_softmax(torch.zeros(2, 4), 0)


# --------------------------------------------------------------------------
# permutation (§2: expert ids stay on the device; dispatch by expert)


def test_permutation_brute_force_and_invariants(oracle_lib):
    rng = np.random.default_rng(5)
    for T, k, E in [(1, 4, 32), (7, 4, 32), (100, 2, 8), (257, 4, 128)]:
        ids = rng.integers(0, E, size=(T, k)).astype(np.int32)
        off, sa, ar = oracle_lib.permute(torch.from_numpy(ids), E)
        flat = ids.reshape(-1)
        expect = sorted(range(T * k), key=lambda a: (flat[a], a))
        assert sa.tolist() == expect
        assert off[0] == 0 and off[-1] == T * k
        assert np.array_equal(np.diff(off.numpy()), np.bincount(flat, minlength=E))
        assert sorted(sa.tolist()) == list(range(T * k))         # bijection
        assert np.array_equal(ar.numpy()[sa.numpy()], np.arange(T * k))


def test_permutation_structured_closed_forms(oracle_lib):
    T, k, E = 9, 4, 32
    # every assignment to one expert: identity order
    ids = torch.full((T, k), 17, dtype=torch.int32)
    off, sa, _ = oracle_lib.permute(ids, E)
    assert sa.tolist() == list(range(T * k))
    assert off.tolist() == [0] * 18 + [T * k] * 15
    # slot j goes to expert j: rows are grouped by slot, tokens ascending
    ids = torch.arange(k, dtype=torch.int32).repeat(T, 1)
    off, sa, _ = oracle_lib.permute(ids, E)
    assert sa.tolist() == [t * k + j for j in range(k) for t in range(T)]
    assert off.tolist()[: k + 1] == [j * T for j in range(k + 1)]
    # id = (7t + j) mod E: row of (t, j) is offsets[id] + #earlier same-id
    ids = torch.tensor([[(7 * t + j) % E for j in range(k)] for t in range(T)],
                       dtype=torch.int32)
    off, sa, ar = oracle_lib.permute(ids, E)
    seen = {}
    for a in range(T * k):
        e = int(ids.view(-1)[a])
        assert ar[a] == off[e] + seen.get(e, 0)
        seen[e] = seen.get(e, 0) + 1


def test_permutation_rejects_out_of_range(oracle_lib):
    with pytest.raises(ValueError):
        oracle_lib.permute(torch.tensor([[0, 32]], dtype=torch.int32), 32)


# --------------------------------------------------------------------------
# clamped interleaved GLU (§1 table, activation row)


def test_glu_zeros():
    import oracle
    for up in [-7.0, -1.5, 0.0, 3.0, 9.0]:
        assert oracle.glu(0.0, up) == 0.0                  # gate = 0 -> h = 0
    for gate in [-3.0, 0.5, 2.0, 7.0, 12.0]:
        assert oracle.glu(gate, -1.0) == 0.0               # up = -1 -> h = 0


def test_glu_clamps():
    import oracle
    for up in [-2.0, 0.0, 1.25]:
        assert oracle.glu(10.0, up) == oracle.glu(7.0, up)   # gate <= 7
        assert oracle.glu(1e6, up) == oracle.glu(7.0, up)
    for gate in [-1.0, 0.5, 3.0]:
        assert oracle.glu(gate, 9.0) == oracle.glu(gate, 7.0)    # up <= 7
        assert oracle.glu(gate, -9.0) == oracle.glu(gate, -7.0)  # up >= -7
    # the gate has no lower clamp: far below -7 the gate term keeps shrinking
    assert abs(oracle.glu(-8.0, 0.0)) < abs(oracle.glu(-7.0, 0.0))


def test_glu_identities_pin_the_sigmoid_form():
    import oracle
    # glu(g) = g*sigma(a g): odd part glu(g) - glu(-g) = g since
    # sigma(z) + sigma(-z) = 1, for any a.
    for g in [0.125, 0.5, 1.0, 2.5, 4.0, 6.75]:
        d = oracle.glu(g, 0.0) - oracle.glu(-g, 0.0)
        assert abs(d - g) <= 4e-7 * max(1.0, g)
    # logit of the gate fraction recovers the constant: ln(s / (1 - s)) = a g
    for g in [0.25, 0.5, 1.0, 1.5]:
        s = np.float64(oracle.glu(g, 0.0)) / g
        assert abs(math.log(s / (1 - s)) / g - 1.702) < 2e-5
    # sigma(0) = 1/2: slope of glu at 0 is 1/2
    eps = 1.0 / 1024
    assert abs(oracle.glu(eps, 0.0) / eps - 0.5) < 1e-3
    # (up + 1) multiplies the gate term (exact in fp32)
    for g, u in [(0.75, 2.0), (-1.5, -3.0), (5.0, 6.5)]:
        assert oracle.glu(g, u) == np.float32(u + 1) * np.float32(oracle.glu(g, 0.0))


def test_glu_range():
    import oracle
    rng = np.random.default_rng(7)
    vals = [oracle.glu(float(g), float(u))
            for g, u in rng.uniform(-60, 60, size=(4000, 2))]
    # glu in [-0.2785/1.702, 7) and (up + 1) in [-6, 8]  =>  h in [-42, 56]
    assert min(vals) >= -42.0 and max(vals) <= 56.0
    assert oracle.glu(7.0, 7.0) <= 56.0 and oracle.glu(7.0, -7.0) >= -42.0


def test_interleave_axis_via_bias_only(oracle_lib, synth_lib):
    # W_gu = 0 -> gu = b_gu, so h_j = glu(b_gu[2j], b_gu[2j+1]) in closed form
    L = _tiny(synth_lib, E=2, T=1, H=64, I=64, k=1)
    L.w_gu.zero_()
    gate = np.linspace(-3, 3, 64).astype(np.float32)
    up = np.linspace(2, -2, 64).astype(np.float32)
    b = np.empty(128, dtype=np.float32)
    b[0::2], b[1::2] = gate, up
    L.b_gu[1] = _bf16(b)
    import oracle
    h, _ = oracle_lib.expert_ffn(L, 1, 0)
    gb = L.b_gu[1].float().numpy()
    expect = [oracle.glu(float(gb[2 * j]), float(gb[2 * j + 1])) for j in range(64)]
    assert h.tolist() == expect
    # swapped roles would differ: glu(1, 0) != glu(0, 1)
    assert oracle.glu(1.0, 0.0) != oracle.glu(0.0, 1.0)


def test_identity_down_projection_returns_h(oracle_lib, synth_lib):
    L = _tiny(synth_lib, E=2, T=2, H=64, I=64, k=1, w_std=0.3)
    L.w_d[0] = torch.eye(64, dtype=torch.bfloat16)
    L.b_d[0].zero_()
    h, y = oracle_lib.expert_ffn(L, 0, 1)
    assert torch.equal(h, y)


# --------------------------------------------------------------------------
# whole layer


def _fp64_layer(L):
    """Independent fp64 brute force of the routed layer (tiny shapes)."""
    f = lambda t: t.float().double().numpy()
    x, wr, br = f(L.x), f(L.wr), f(L.br)
    wgu, bgu, wd, bd = f(L.w_gu), f(L.b_gu), f(L.w_d), f(L.b_d)
    logits = x @ wr.T + br
    out = np.zeros((L.T, L.H))
    sels = []
    for t in range(L.T):
        order = sorted(range(L.E), key=lambda e: (-logits[t, e], e))
        sel = order[: L.top_k]
        gap = logits[t, order[L.top_k - 1]] - logits[t, order[L.top_k]] \
            if L.top_k < L.E else 1.0
        assert gap > 1e-4, "fixture too close to a routing tie"
        z = np.exp(logits[t, sel] - logits[t, sel[0]])
        w = z / z.sum()
        for j, e in enumerate(sel):
            gu = wgu[e] @ x[t] + bgu[e]
            gate, up = np.minimum(gu[0::2], 7.0), np.clip(gu[1::2], -7.0, 7.0)
            h = (up + 1.0) * gate / (1.0 + np.exp(-1.702 * gate))
            out[t] += w[j] * (wd[e] @ h + bd[e])
        sels.append(sel)
    return sels, out


@pytest.mark.parametrize("w_std", [0.02, 0.5])
def test_layer_matches_fp64_brute_force(oracle_lib, synth_lib, w_std):
    # E=4, top-2, H=I=64; w_std=0.5 drives many gate/up values into the clamps
    L = _tiny(synth_lib, E=4, T=8, H=64, I=64, k=2, seed=21, w_std=w_std,
              router_w_std=0.3)
    sels, ref = _fp64_layer(L)
    ids, w, out = oracle_lib.forward(L)
    assert ids.tolist() == sels
    err = np.abs(out.double().numpy() - ref).max()
    assert err <= 1e-5 * np.abs(ref).max()


def test_clamps_are_active_in_the_fp64_fixture(oracle_lib, synth_lib):
    L = _tiny(synth_lib, E=4, T=8, H=64, I=64, k=2, seed=21, w_std=0.5)
    x = L.x.float().double().numpy()
    gu = L.w_gu[0].float().double().numpy() @ x.T
    assert (gu[0::2] > 7).any() and (gu[1::2] > 7).any() and (gu[1::2] < -7).any()


def test_routed_equals_dense_bit_exact(oracle_lib, synth_lib):
    for E, k in [(4, 2), (8, 4), (6, 1)]:
        L = _tiny(synth_lib, E=E, T=5, H=64, I=64, k=k, seed=E * 10 + k)
        i1, w1, o1 = oracle_lib.forward(L)
        i2, w2, o2 = oracle_lib.forward_dense(L)
        assert torch.equal(i1, i2) and torch.equal(w1, w2) and torch.equal(o1, o2)


def test_dense_form_skips_unselected_experts(oracle_lib, synth_lib):
    # A non-selected expert with non-finite weights must not leak into the
    # output: §2 requires a skip, and 0 * inf would give NaN.
    L = _tiny(synth_lib, E=4, T=3, H=64, I=64, k=2, seed=3)
    L.wr.zero_()
    L.br.copy_(_bf16([1.0, 0.5, -1.0, -2.0]))    # experts 0, 1 always selected
    L.w_d[3, 0, 0] = float("inf")
    ids, _, out = oracle_lib.forward_dense(L)
    assert ids.tolist() == [[0, 1]] * 3
    assert torch.isfinite(out).all()


def test_output_is_weighted_sum_of_expert_outputs(oracle_lib, synth_lib):
    L = _tiny(synth_lib, E=4, T=4, H=64, I=64, k=2, seed=9)
    ids, w, out = oracle_lib.forward(L)
    for t in range(L.T):
        acc = torch.zeros(L.H)
        for j in range(2):
            acc += w[t, j] * oracle_lib.expert_ffn(L, int(ids[t, j]), t)[1]
        assert torch.equal(acc, out[t])


def test_token_subset_matches_full_forward(oracle_lib, synth_lib):
    L = _tiny(synth_lib, E=8, T=9, H=64, I=64, k=4, seed=4)
    ids, w, out = oracle_lib.forward(L)
    sel = [8, 0, 5]
    i2, w2, o2 = oracle_lib.forward(L, tokens=sel)
    assert torch.equal(i2, ids[sel]) and torch.equal(w2, w[sel])
    assert torch.equal(o2, out[sel])


def test_thread_count_does_not_change_results(oracle_lib, synth_lib):
    L = _tiny(synth_lib, E=8, T=6, H=64, I=64, k=4, seed=8)
    a = oracle_lib.forward(L, threads=1)
    b = oracle_lib.forward(L, threads=4)
    assert all(torch.equal(p, q) for p, q in zip(a, b))


# --------------------------------------------------------------------------
# MXFP4 (§5: E2M1 values, one UE8M0 scale per 32 elements)

# OCP Microscaling Formats (MX) v1.0, FP4 E2M1 value table, codes 0..15.
E2M1_TABLE = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0,
              -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0]


def test_e2m1_and_e8m0_tables():
    import oracle
    for c in range(16):
        assert oracle.e2m1(c) == E2M1_TABLE[c]
    for s, v in [(127, 1.0), (119, 2.0 ** -8), (123, 2.0 ** -4), (128, 2.0),
                 (0, 2.0 ** -127)]:
        assert oracle.e8m0(s) == v


def test_mxfp4_dequant_all_codes_and_scales(oracle_lib):
    # one row of 32 elements per scale: codes 0..15 twice, low nibble first
    codes = torch.tensor([(2 * i + 1) % 16 << 4 | (2 * i) % 16 for i in range(16)],
                         dtype=torch.uint8)
    for s in range(119, 124):
        deq = oracle_lib.dequant_mxfp4(codes.view(1, 16),
                                       torch.tensor([[s]], dtype=torch.uint8))
        expect = [E2M1_TABLE[i % 16] * 2.0 ** (s - 127) for i in range(32)]
        assert deq.view(-1).tolist() == expect


def test_mxfp4_scale_blocks_run_along_k(oracle_lib):
    codes = torch.full((2, 32), 0x22, dtype=torch.uint8)      # every value 1.0
    scales = torch.tensor([[127, 128], [126, 127]], dtype=torch.uint8)
    deq = oracle_lib.dequant_mxfp4(codes, scales)
    assert deq[0, :32].eq(1.0).all() and deq[0, 32:].eq(2.0).all()
    assert deq[1, :32].eq(0.5).all() and deq[1, 32:].eq(1.0).all()


def test_mxfp4_layer_equals_bf16_layer_on_dequantised_weights(oracle_lib, synth_lib):
    Lq = _tiny(synth_lib, E=4, T=5, H=64, I=64, k=2, seed=13, wfmt="mxfp4")
    wgu = oracle_lib.dequant_mxfp4(Lq.w_gu, Lq.s_gu)
    wd = oracle_lib.dequant_mxfp4(Lq.w_d, Lq.s_d)
    # dequantised values are exact in bf16 (2-bit significand, power-2 scale)
    assert torch.equal(wgu.to(torch.bfloat16).float(), wgu)
    assert torch.equal(wd.to(torch.bfloat16).float(), wd)
    Lb = _tiny(synth_lib, E=4, T=5, H=64, I=64, k=2, seed=13)
    Lb.w_gu = wgu.to(torch.bfloat16).contiguous()
    Lb.w_d = wd.to(torch.bfloat16).contiguous()
    a, b = oracle_lib.forward(Lq), oracle_lib.forward(Lb)
    assert all(torch.equal(p, q) for p, q in zip(a, b))


# --------------------------------------------------------------------------
# FP8 W8A8 (E4M3 weights with per-expert scales, per-token E4M3 activations)


def _torch_e4m3_codes(v: torch.Tensor) -> torch.Tensor:
    """Library rounding to e4m3 (round to nearest even; NaN past 464)."""
    return v.to(torch.float32).to(torch.float8_e4m3fn).view(torch.uint8)


def test_e4m3_decode_matches_library_for_all_codes():
    import oracle
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float32)
    for c in range(256):
        v = oracle.e4m3(c)
        if c in (0x7F, 0xFF):
            assert v != v                          # NaN
        else:
            assert v == ref[c].item(), hex(c)
    # the format's landmarks
    assert oracle.e4m3(0x7E) == 448.0 and oracle.e4m3(0x01) == 2.0 ** -9
    assert oracle.e4m3(0x08) == 2.0 ** -6 and oracle.e4m3(0x38) == 1.0


def test_e4m3_rounding_matches_library_within_range():
    import oracle
    g = torch.Generator().manual_seed(8)
    # magnitudes from the subnormal range to 464, both signs
    mag = torch.exp2(torch.rand(4000, generator=g) * 18.0 - 12.0).clamp(max=464.0)
    sgn = torch.where(torch.rand(4000, generator=g) < 0.5, -1.0, 1.0)
    vals = (mag * sgn).to(torch.float32)
    # plus every midpoint between adjacent codes (ties go to the even code)
    pos = torch.tensor([oracle.e4m3(c) for c in range(0x7F)], dtype=torch.float64)
    mids = ((pos[:-1] + pos[1:]) / 2).to(torch.float32)
    vals = torch.cat([vals, mids, -mids])
    ref = _torch_e4m3_codes(vals)
    got = torch.tensor([oracle.e4m3_round(v) for v in vals.tolist()], dtype=torch.uint8)
    assert torch.equal(got, ref)


def test_e4m3_rounding_saturates_beyond_448():
    import oracle
    for v in (464.0, 470.0, 480.0, 1.0e4, 3.0e38):
        assert oracle.e4m3_round(v) == 0x7E and oracle.e4m3_round(-v) == 0xFE


def test_fp8_row_quantisation_rules(oracle_lib):
    g = torch.Generator().manual_seed(3)
    x = (torch.randn(200, generator=g) * 3).to(torch.bfloat16)
    x[17] = -25.0                                   # the row's largest magnitude
    codes, scale = oracle_lib.fp8_quantize_row(x)
    xf = x.float()
    amax = xf.abs().max()
    assert scale == (amax / 448.0).item()
    assert codes[17].item() == 0xFE                 # -448 exactly
    # every code is the library rounding of x * (448 / max|x|)
    assert torch.equal(codes, _torch_e4m3_codes(xf * (448.0 / amax)))
    zero_codes, zero_scale = oracle_lib.fp8_quantize_row(torch.zeros(8, dtype=torch.bfloat16))
    assert zero_scale == 1.0 and zero_codes.eq(0).all()


def _fp64_fp8_layer(L):
    """Independent fp64 brute force of the FP8 W8A8 layer: e4m3 decoding and
    rounding by the library, scales applied after the product."""
    dec = lambda c: c.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    x = L.x.float()
    wr, br = L.wr.float().double().numpy(), L.br.float().double().numpy()
    logits = x.double().numpy() @ wr.T + br
    wgu, wd = dec(L.w_gu), dec(L.w_d)
    sgu, sd = L.s_gu.double().numpy(), L.s_d.double().numpy()
    bgu, bd = L.b_gu.float().double().numpy(), L.b_d.float().double().numpy()
    out = np.zeros((L.T, L.H))
    sels = []
    for t in range(L.T):
        order = sorted(range(L.E), key=lambda e: (-logits[t, e], e))
        sel = order[: L.top_k]
        z = np.exp(logits[t, sel] - logits[t, sel[0]])
        w = z / z.sum()
        amax = x[t].abs().max()
        xq = dec(_torch_e4m3_codes(x[t] * (448.0 / amax)))
        xs = float(amax) / 448.0
        for j, e in enumerate(sel):
            gu = (wgu[e] @ xq) * (sgu[e] * xs) + bgu[e]
            gate, up = np.minimum(gu[0::2], 7.0), np.clip(gu[1::2], -7.0, 7.0)
            h = (up + 1.0) * gate / (1.0 + np.exp(-1.702 * gate))
            hq = dec(_torch_e4m3_codes(torch.from_numpy(h * 8.0)))
            out[t] += w[j] * ((wd[e] @ hq) * (sd[e] * 0.125) + bd[e])
        sels.append(sel)
    return sels, out


def test_fp8_layer_matches_fp64_brute_force(oracle_lib, synth_lib):
    L = synth_lib.make_layer(E=4, T=6, H=64, I=64, top_k=2, seed=31, wfmt="fp8",
                             router_w_std=0.3)
    sels, ref = _fp64_fp8_layer(L)
    ids, w, out = oracle_lib.forward(L)
    assert ids.tolist() == sels
    # fp32 vs fp64 sums can move an h value across an e4m3 rounding boundary;
    # one such flip changes an output by ~|w_d| * |h| / 16
    err = np.abs(out.double().numpy() - ref).max()
    assert err <= 2e-3 * np.abs(ref).max()


def test_fp8_scales_apply_after_the_product(oracle_lib, synth_lib):
    """The expert scale multiplies the finished sum: with zero biases,
    doubling one expert's down scale doubles its output exactly (a power-of-
    two factor applied to an fp32 sum), and h does not change."""
    L = synth_lib.make_layer(E=2, T=2, H=64, I=64, top_k=1, seed=5, wfmt="fp8")
    L.b_gu = torch.zeros_like(L.b_gu)
    L.b_d = torch.zeros_like(L.b_d)
    h1, y1 = oracle_lib.expert_ffn(L, 1, 0)
    L.s_d = L.s_d.clone()
    L.s_d[1] *= 2.0
    h2, y2 = oracle_lib.expert_ffn(L, 1, 0)
    assert torch.equal(h1, h2)
    assert torch.equal(y2, 2.0 * y1) and y1.abs().max() > 0


# ------------------------------------------- MXFP4 weights, MXFP8 activations

def _mx_expected(block: torch.Tensor):
    """OCP MX v1.0 conversion of one bf16 block of 32, written with torch ops:
    shared exponent floor(log2 max|x|) - 8 clamped to [-127, 127] (-127 for
    a zero block), elements by the library's e4m3 rounding, saturated."""
    xf = block.double()
    amax = xf.abs().max().item()
    shared = -127 if amax == 0 else max(-127, min(127, math.floor(math.log2(amax)) - 8))
    v = (xf * 2.0 ** (-shared)).clamp(-448.0, 448.0).float()
    return _torch_e4m3_codes(v), shared + 127


def test_mx_quantisation_closed_forms(oracle_lib):
    def q(vals):
        x = torch.zeros(32, dtype=torch.bfloat16)
        x[: len(vals)] = torch.tensor(vals, dtype=torch.float32).to(torch.bfloat16)
        return oracle_lib.mx_quantize_row(x)
    codes, scales = q([1.0])                 # 1 = 2^0: scale 2^-8, 1 -> 256
    assert scales.tolist() == [119] and codes[0].item() == 0x78
    codes, scales = q([480.0, -3.0])         # floor(log2 480) = 8: scale 1; 480 saturates
    assert scales.tolist() == [127] and codes[0].item() == 0x7E and codes[1].item() == 0xC4
    codes, scales = q([])                    # all zero: smallest scale, zero codes
    assert scales.tolist() == [0] and codes.eq(0).all()
    codes, scales = q([2.0 ** -130])         # scale clamps at 2^-127: 2^-130 -> 2^-3
    assert scales.tolist() == [0] and codes[0].item() == 0x20
    codes, scales = q([0.75, 0.5])           # floor(log2 0.75) = -1: scale 2^-9
    assert scales.tolist() == [118] and codes[0].item() == 0x7C and codes[1].item() == 0x78


def test_mx_quantisation_matches_library_rounding(oracle_lib):
    g = torch.Generator().manual_seed(12)
    x = (torch.randn(32 * 40, generator=g) * torch.exp(torch.randn(32 * 40, generator=g) * 3))
    x[5 * 32: 6 * 32] = 0.0
    x = x.to(torch.bfloat16)
    codes, scales = oracle_lib.mx_quantize_row(x)
    for b in range(40):
        ec, es = _mx_expected(x[32 * b: 32 * (b + 1)])
        assert scales[b].item() == es, b
        assert torch.equal(codes[32 * b: 32 * (b + 1)], ec), b


def _fp64_mx_layer(L):
    """Independent fp64 brute force of the MXFP4-weight / MXFP8-activation
    layer: MXFP4 weights from the E2M1 table, activations by the MX rule above,
    h as e4m3 of h * 8."""
    dec = lambda c: c.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    tab = np.array(E2M1_TABLE)

    def dequant(codes, scales, K):
        lo, hi = codes & 0xF, codes >> 4
        q = torch.stack([lo, hi], dim=-1).reshape(*codes.shape[:-1], K).long().numpy()
        s = np.repeat(2.0 ** (scales.double().numpy() - 127), 32, axis=-1)
        return tab[q] * s

    x = L.x.float()
    wr, br = L.wr.float().double().numpy(), L.br.float().double().numpy()
    logits = x.double().numpy() @ wr.T + br
    wgu, wd = dequant(L.w_gu, L.s_gu, L.H), dequant(L.w_d, L.s_d, L.I)
    bgu, bd = L.b_gu.float().double().numpy(), L.b_d.float().double().numpy()
    out = np.zeros((L.T, L.H))
    sels = []
    for t in range(L.T):
        order = sorted(range(L.E), key=lambda e: (-logits[t, e], e))
        sel = order[: L.top_k]
        z = np.exp(logits[t, sel] - logits[t, sel[0]])
        w = z / z.sum()
        xq = np.zeros(L.H)
        for b in range(L.H // 32):
            c, s = _mx_expected(L.x[t, 32 * b: 32 * (b + 1)])
            xq[32 * b: 32 * (b + 1)] = dec(c) * 2.0 ** (s - 127)
        for j, e in enumerate(sel):
            gu = wgu[e] @ xq + bgu[e]
            gate, up = np.minimum(gu[0::2], 7.0), np.clip(gu[1::2], -7.0, 7.0)
            h = (up + 1.0) * gate / (1.0 + np.exp(-1.702 * gate))
            hq = dec(_torch_e4m3_codes(torch.from_numpy(h * 8.0))) * 0.125
            out[t] += w[j] * (wd[e] @ hq + bd[e])
        sels.append(sel)
    return sels, out


def test_mx_layer_matches_fp64_brute_force(oracle_lib, synth_lib):
    L = synth_lib.make_layer(E=4, T=6, H=64, I=64, top_k=2, seed=33, wfmt="mxfp4_mxfp8",
                             router_w_std=0.3)
    sels, ref = _fp64_mx_layer(L)
    ids, w, out = oracle_lib.forward(L)
    assert ids.tolist() == sels
    err = np.abs(out.double().numpy() - ref).max()
    assert err <= 2e-3 * np.abs(ref).max()


def test_mx_layer_with_exact_activations_equals_mxfp4_layer(oracle_lib, synth_lib):
    """Activations that MXFP8 holds exactly give the MXFP4 (bf16-activation)
    layer's h bit for bit: x = m / 8 with |m| <= 14 and every block's largest
    magnitude 1.75, so the block scale is 2^-8 and x / scale = 32 m, at most
    448 and within e4m3's 4 significant bits."""
    L = synth_lib.make_layer(E=2, T=2, H=64, I=64, top_k=1, seed=9, wfmt="mxfp4_mxfp8")
    g = torch.Generator().manual_seed(4)
    x = torch.randint(-14, 15, (2, 64), generator=g).float() * 0.125
    x[:, 0] = 1.75
    x[:, 32] = -1.75
    L.x = x.to(torch.bfloat16)
    codes, scales = oracle_lib.mx_quantize_row(L.x[0])
    assert scales.tolist() == [119, 119]
    h_mx, _ = oracle_lib.expert_ffn(L, 1, 0)
    L4 = synth_lib.make_layer(E=2, T=2, H=64, I=64, top_k=1, seed=9, wfmt="mxfp4")
    L4.x = L.x
    h_4, _ = oracle_lib.expert_ffn(L4, 1, 0)
    assert torch.equal(h_mx, h_4)


# ------------------------------------------------ expert-parallel partial form

def test_ep_full_range_is_the_forward(oracle_lib, synth_lib):
    L = _tiny(synth_lib, E=8, T=10, k=3, seed=41)
    _, _, out = oracle_lib.forward(L)
    assert torch.equal(oracle_lib.forward_ep(L, 0, 8), out)


def test_ep_single_expert_is_weight_times_expert_output(oracle_lib, synth_lib):
    """A device holding expert e alone outputs w[t, j] * y(e, t) for the
    tokens that chose e (ids are distinct, so one slot at most) and zero rows
    for the others."""
    L = _tiny(synth_lib, E=6, T=12, k=2, seed=43)
    ids, w, _ = oracle_lib.forward(L)
    for e in range(6):
        part = oracle_lib.forward_ep(L, e, 1)
        for t in range(12):
            hit = (ids[t] == e).nonzero()
            if len(hit) == 0:
                assert part[t].eq(0).all()
            else:
                _, y = oracle_lib.expert_ffn(L, e, t)
                assert torch.equal(part[t], w[t, hit[0, 0]] * y)


def test_ep_partition_sums_to_the_forward(oracle_lib, synth_lib):
    L = _tiny(synth_lib, E=8, T=10, k=3, seed=45)
    _, _, out = oracle_lib.forward(L)
    parts = [oracle_lib.forward_ep(L, lo, n) for lo, n in ((0, 3), (3, 1), (4, 4))]
    total = parts[0] + parts[1] + parts[2]
    assert (total - out).abs().max() <= 1e-6 * out.abs().max()
    assert oracle_lib.forward_ep(L, 2, 0).eq(0).all()


# ------------------------------------------------ attention with sinks (f4)

def _att(synth_lib, Tq, Tkv, Hq=4, Hkv=2, D=16, seed=0, **kw):
    return synth_lib.make_attention(Tq, Tkv, Hq=Hq, Hkv=Hkv, D=D, seed=seed, **kw)


def test_attention_without_sink_is_library_causal_attention(oracle_lib, synth_lib):
    a = _att(synth_lib, 9, 9, seed=1)
    out = oracle_lib.attention_sinks(a["q"], a["k"], a["v"],
                                     torch.full((4,), float("-inf")))
    q = a["q"].double().permute(1, 0, 2)
    k = a["k"].double().repeat_interleave(2, dim=1).permute(1, 0, 2)
    v = a["v"].double().repeat_interleave(2, dim=1).permute(1, 0, 2)
    ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=True)
    assert torch.allclose(out.double(), ref.permute(1, 0, 2), rtol=0, atol=1e-6)


def test_attention_window_of_one_closed_form(oracle_lib, synth_lib):
    """W = 1: each query sees its own key only, against the sink:
    out_i = v_i / (1 + exp(sink - s_ii))."""
    a = _att(synth_lib, 6, 6, seed=2)
    out = oracle_lib.attention_sinks(a["q"], a["k"], a["v"], a["sinks"], window=1)
    for i in range(6):
        for h in range(4):
            s = float((a["q"][i, h].double() * a["k"][i, h // 2].double()).sum()) / 4.0
            w = 1.0 / (1.0 + math.exp(float(a["sinks"][h]) - s))
            assert torch.allclose(out[i, h].double(), w * a["v"][i, h // 2].double(),
                                  rtol=1e-6, atol=1e-7)


def test_attention_large_sink_takes_all_mass(oracle_lib, synth_lib):
    a = _att(synth_lib, 5, 5, seed=3, qk_std=0.1)
    out = oracle_lib.attention_sinks(a["q"], a["k"], a["v"], torch.full((4,), 60.0))
    assert out.abs().max() < 1e-20


def test_attention_window_covering_everything_is_full(oracle_lib, synth_lib):
    a = _att(synth_lib, 12, 12, seed=4)
    full = oracle_lib.attention_sinks(a["q"], a["k"], a["v"], a["sinks"])
    assert torch.equal(oracle_lib.attention_sinks(a["q"], a["k"], a["v"], a["sinks"],
                                                  window=12), full)
    w3 = oracle_lib.attention_sinks(a["q"], a["k"], a["v"], a["sinks"], window=3)
    assert torch.equal(w3[:3], full[:3]) and not torch.equal(w3[3:], full[3:])


def test_attention_decode_rows_equal_prefill_rows(oracle_lib, synth_lib):
    """A query at position p over the cache [0, p] (decode) equals row p of
    the prefill over the same keys."""
    a = _att(synth_lib, 10, 10, seed=5)
    full = oracle_lib.attention_sinks(a["q"], a["k"], a["v"], a["sinks"], window=4)
    for p in (0, 3, 9):
        one = oracle_lib.attention_sinks(a["q"][p:p + 1], a["k"][:p + 1], a["v"][:p + 1],
                                         a["sinks"], window=4)
        assert torch.equal(one[0], full[p])


def test_attention_gqa_heads_share_their_kv_head(oracle_lib, synth_lib):
    a = _att(synth_lib, 7, 7, Hq=6, Hkv=3, seed=6)
    q = a["q"].clone()
    q[:, 1] = q[:, 0]                       # heads 0 and 1 read KV head 0
    q[:, 2] = q[:, 0]                       # head 2 reads KV head 1
    sinks = torch.zeros(6)
    out = oracle_lib.attention_sinks(q, a["k"], a["v"], sinks)
    assert torch.equal(out[:, 0], out[:, 1]) and not torch.equal(out[:, 0], out[:, 2])

"""The C-ABI library builds, loads and exports every symbol include/moe.h
declares; host-side argument checks reject bad calls before touching a GPU.

No test here launches work: with no GPU present, only calls that fail
validation (or never reach CUDA) are made.
"""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def moe():
    from gpt_oss_moe_gb300 import _build
    _build.build()
    import gpt_oss_moe_gb300 as m
    return m


def _declared_functions():
    names = []
    for hdr in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if not hdr.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", hdr)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\**\s*"
                            r"(moe_[a-z0-9_]+)\s*\(", text, flags=re.M)
    return names


def test_header_declares_the_binding_names(moe):
    declared = _declared_functions()
    assert sorted(declared) == sorted(moe.EXPORTS)
    assert "moe_route" in declared and "moe_forward" in declared


def test_library_exports_every_declared_symbol(moe):
    L = ctypes.CDLL(moe.LIB_PATH)
    for name in _declared_functions():
        assert hasattr(L, name), name


def test_status_strings(moe):
    for code in range(-7, 1):
        assert moe.moe_status_str(code) != "unknown status"
    assert moe.moe_status_str(-99) == "unknown status"


def _shape(moe, **kw):
    d = dict(T=8, H=2880, I=2880, E=32, top_k=4, wfmt=0)
    d.update(kw)
    return moe.make_shape(**d)


def test_workspace_bytes(moe):
    small = moe.moe_workspace_bytes(_shape(moe, T=8))
    big = moe.moe_workspace_bytes(_shape(moe, T=4096))
    assert 0 < small < big
    # T * k rows of activations and of h, T rows of fp32 output
    assert big >= 4096 * 4 * 2880 * 2 * 2 + 4096 * 2880 * 4
    assert moe.moe_workspace_bytes(_shape(moe, T=0)) > 0
    for bad in [dict(H=2880 + 32), dict(I=100), dict(E=0), dict(E=257),
                dict(top_k=0), dict(top_k=9), dict(E=2, top_k=3), dict(T=-1),
                dict(T=(1 << 20) + 1)]:
        assert moe.moe_workspace_bytes(_shape(moe, **bad)) == 0, bad


def _fwd(moe, shape, ptrs, ws_bytes=1 << 30):
    L = moe.lib()
    gu = moe.moe_weight(ptrs.get("wgu", 256), ptrs.get("sgu"), ptrs.get("bgu", 512))
    dn = moe.moe_weight(ptrs.get("wd", 768), ptrs.get("sd"), ptrs.get("bd", 1024))
    return L.moe_forward(ctypes.byref(shape), ptrs.get("x", 16), ptrs.get("wr", 32),
                         ptrs.get("br", 48), gu, dn, ptrs.get("out", 64), 1,
                         None, None, ptrs.get("ws", 4096), ws_bytes, None)


def test_forward_rejects_bad_arguments_on_the_host(moe):
    s = _shape(moe)
    assert _fwd(moe, _shape(moe, H=100), {}) == -2          # MOE_ERR_SHAPE
    assert _fwd(moe, _shape(moe, wfmt=7), {}) == -1         # MOE_ERR_ARG
    assert _fwd(moe, s, {"x": 0}) == -1                     # null hidden
    assert _fwd(moe, s, {"out": 0}) == -1                   # null out
    assert _fwd(moe, s, {"wd": 0}) == -1                    # null down weights
    assert _fwd(moe, s, {"x": 24}) == -3                    # misaligned
    assert _fwd(moe, s, {"wgu": 520}) == -3
    assert _fwd(moe, s, {}, ws_bytes=100) == -4             # workspace too small
    assert moe.lib().moe_forward(None, 16, 32, 48, moe.moe_weight(), moe.moe_weight(),
                                 64, 1, None, None, 4096, 1 << 30, None) == -1
    # T == 0 is valid and enqueues nothing (no device needed)
    assert _fwd(moe, _shape(moe, T=0), {"x": 0, "out": 0}) == 0


def test_forward_ep_rejects_bad_expert_ranges_on_the_host(moe):
    L = moe.lib()
    s = _shape(moe, E=32)

    def ep(start, n, wfmt=None):
        sh = s if wfmt is None else _shape(moe, E=32, wfmt=wfmt)
        gu = moe.moe_weight(256, 1024 if wfmt else None, 512)
        dn = moe.moe_weight(768, 1024 if wfmt else None, 1024)
        return L.moe_forward_ep(ctypes.byref(sh), start, n, 16, 32, 48, gu, dn, 64, 1,
                                None, None, 4096, 1 << 30, None)
    for start, n in [(-1, 4), (0, 0), (30, 3), (32, 1), (0, 33)]:
        assert ep(start, n) == -1, (start, n)                 # MOE_ERR_ARG
    # MXFP4 x MXFP8 codes must be 32-byte aligned: 16 + 256 is not
    gu = moe.moe_weight(272, 1024, 512)
    dn = moe.moe_weight(768, 1024, 1024)
    sh = _shape(moe, E=32, wfmt=moe.MOE_W_MXFP4_MXFP8)
    assert L.moe_forward_ep(ctypes.byref(sh), 0, 32, 16, 32, 48, gu, dn, 64, 1,
                            None, None, 4096, 1 << 30, None) == -3
    assert L.moe_forward_ep(None, 0, 1, 16, 32, 48, gu, dn, 64, 1, None, None, 4096,
                            1 << 30, None) == -1


def test_noalloc_maps_bad_shapes_for_every_format(moe):
    L = moe.lib()
    for wfmt in (moe.MOE_W_BF16, moe.MOE_W_MXFP4, moe.MOE_W_FP8, moe.MOE_W_MXFP4_MXFP8):
        bad = _shape(moe, H=100, wfmt=wfmt)
        code = L.moe_forward_noalloc(ctypes.byref(bad), 16, 32, 48, moe.moe_weight(),
                                     moe.moe_weight(), 64, 1, None, None, None, None)
        assert code == -2, wfmt                                # MOE_ERR_SHAPE
    # MXFP4 x MXFP8 needs H, I >= 128
    assert moe.moe_workspace_bytes(_shape(moe, H=64, wfmt=moe.MOE_W_MXFP4_MXFP8)) == 0
    bad = _shape(moe, wfmt=9)
    assert L.moe_forward_noalloc(ctypes.byref(bad), 16, 32, 48, moe.moe_weight(),
                                 moe.moe_weight(), 64, 1, None, None, None, None) == -1


def test_ep_expert_ranges_partition_the_experts(moe):
    for E in (1, 7, 32, 128):
        for world in range(1, min(E, 9) + 1):
            got = [moe.ep_expert_range(r, world, E) for r in range(world)]
            assert got[0][0] == 0 and sum(n for _, n in got) == E
            assert all(a + n == b for (a, n), (b, _) in zip(got, got[1:]))
            assert max(n for _, n in got) - min(n for _, n in got) <= 1
    with pytest.raises(ValueError):
        moe.ep_expert_range(0, 5, 4)


def test_attention_workspace_and_argument_checks_on_the_host(moe):
    L = moe.lib()

    def shape(**kw):
        d = dict(Tq=4, Tkv=4, Hq=8, Hkv=1, D=64, window=0, q_start=0)
        d.update(kw)
        return moe.moe_attn_shape(*[d[n] for n, _ in moe.moe_attn_shape._fields_])
    ws = L.moe_attention_workspace_bytes
    assert ws(ctypes.byref(shape(Tq=0, q_start=4))) == 0          # nothing to split
    assert ws(ctypes.byref(shape(D=32))) == 0                     # invalid shape
    assert ws(ctypes.byref(shape(Tq=1, Tkv=4096, q_start=4095))) > 0   # decode splits
    call = lambda s, q=16, sinks=32: L.moe_attention_sinks(ctypes.byref(s), q, 48, 64, sinks,
                                                           80, None, 0, None)
    assert call(shape(D=32)) == -2
    assert call(shape(Hq=6, Hkv=4)) == -2
    assert call(shape(Tq=5)) == -2                                # q_start + Tq > Tkv
    assert call(shape(), q=24) == -3                              # misaligned q
    assert call(shape(), sinks=34) == -3                          # misaligned sinks
    assert call(shape(), q=0) == -1
    assert call(shape(Tq=0, q_start=4)) == 0                      # empty: enqueues nothing
    assert call(shape(Tq=0, q_start=4), q=0) == 0                 # ... even with null pointers
    assert call(shape(Tq=1, Tkv=4096, q_start=4095)) == -4        # decode needs a workspace


def test_route_rejects_bad_arguments_on_the_host(moe):
    L = moe.lib()
    s = _shape(moe)
    assert L.moe_route(ctypes.byref(s), 0, 32, 48, None, None, None, None, 4096,
                       1 << 30, None) == -1
    assert L.moe_route(ctypes.byref(s), 16, 32, 48, 8, None, None, None, 4096,
                       1 << 30, None) == -3
    assert L.moe_route(ctypes.byref(s), 16, 32, 48, None, None, None, None, 4096,
                       10, None) == -4
    s0 = _shape(moe, T=0)
    assert L.moe_route(ctypes.byref(s0), 0, 0, 0, None, None, None, None, 0, 0,
                       None) == 0


def test_tuning_switches(moe):
    with pytest.raises(moe.MoEError):
        moe.moe_set_tuning("token_tile", 24)
    with pytest.raises(moe.MoEError):
        moe.moe_set_tuning("token_tile", 512)
    with pytest.raises(moe.MoEError):
        moe.moe_set_tuning("no_such_key", 1)
    moe.moe_set_tuning("token_tile", 64)
    moe.moe_set_tuning("token_tile", 0)
    moe.moe_set_tuning("pdl", 0)
    moe.moe_set_tuning("pdl", 1)
    moe.moe_set_tuning("ksplit", 1)
    moe.moe_set_tuning("ksplit", 0)
    moe.moe_set_tuning("ksplit", 3)
    moe.moe_set_tuning("ksplit", 0)
    with pytest.raises(moe.MoEError):
        moe.moe_set_tuning("ksplit", 9)
    for v in (1, 2, 0):
        moe.moe_set_tuning("pair", v)
    for v in (-1, 3):
        with pytest.raises(moe.MoEError):
            moe.moe_set_tuning("pair", v)


# every switch with its accepted values (the default last) and values the
# library must refuse without changing anything
SWITCHES = {
    "mxfp4_f16": ((0, 1), (-1, 2)),
    "attn_tc": ((1, 2, 0), (-1, 3)),
    "attn_poll": ((1, 0), (-1, 2)),
    "tiny_router": ((0, 1), (-1, 2)),
    "small_path": ((0, 1), (-1, 2)),
    "inject": ((7, 1, 0), (-1, 8)),
    "deterministic": ((1, 0), (-1, 2)),
    "noalloc_poison": ((1, 0), (-1, 2)),
}


@pytest.mark.parametrize("key", sorted(SWITCHES))
def test_switch_values(moe, key):
    good, bad = SWITCHES[key]
    for v in bad:
        with pytest.raises(moe.MoEError):
            moe.moe_set_tuning(key, v)
    for v in good:
        moe.moe_set_tuning(key, v)


def test_attention_workspace_follows_the_kernel_choice(moe):
    """The tcgen05 kernel (calls of 512 queries or more, or attn_tc 2) needs
    only the 256-byte status word; the key-split kernel's workspace holds
    its partial rows."""
    L = moe.lib()

    def ws(**kw):
        d = dict(Tq=4, Tkv=4, Hq=8, Hkv=1, D=64, window=0, q_start=0)
        d.update(kw)
        sh = moe.moe_attn_shape(*[d[n] for n, _ in moe.moe_attn_shape._fields_])
        return L.moe_attention_workspace_bytes(ctypes.byref(sh))
    decode = dict(Tq=1, Tkv=4096, Hq=64, Hkv=8, q_start=4095)
    prefill = dict(Tq=4096, Tkv=4096, Hq=64, Hkv=8)
    try:
        moe.moe_set_tuning("attn_tc", 0)
        assert ws(**prefill) == 256
        assert ws(**decode) > 256
        moe.moe_set_tuning("attn_tc", 2)
        assert ws(**decode) == 256
        assert ws(Tq=0, Tkv=4, q_start=4) == 256
        moe.moe_set_tuning("attn_tc", 1)
        assert ws(**prefill) == 0          # the key-split kernel: no split at this size
    finally:
        moe.moe_set_tuning("attn_tc", 0)


def test_binding_fails_loudly_without_library(tmp_path, monkeypatch):
    import gpt_oss_moe_gb300 as m
    monkeypatch.setattr(m, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(m, "_lib", None)
    with pytest.raises(ImportError):
        m.lib()

"""Seeded synthetic inputs for the gpt-oss MoE layer.

This module holds none of the layer's arithmetic: it draws seeded random
numbers (``synth.c``, splitmix64 in counter mode, Box-Muller normals) and
rounds them to the storage formats (bf16, MXFP4 codes and E8M0 block scales).
The CPU oracle and the CUDA library are both fed from the buffers it fills.

Workload recipes (shapes from the xserv page "Phase 19: gpt-oss-20b", §1
model-architecture table: hidden 2880, 32 experts top-4, expert inter 2880;
the 120b-shaped layer keeps the same widths with 128 experts):

* expert and router weights ~ N(0, 0.02), biases ~ N(0, 0.01), activations
  ~ N(0, 1), all rounded to bf16;
* "hot experts": +2.0 added to the router bias of experts 0-3 (skewed load);
* outliers: each activation element independently, with probability 0.01,
  is multiplied by 20 before rounding;
* MXFP4: e2m1 codes uniform over the 16 nibble values, two per byte, and one
  E8M0 scale byte per 32 consecutive input elements with exponent uniform in
  [-8, -4] (bytes 119..123).
* FP8 (W8A8 weights): e4m3 codes drawn field by field -- sign uniform,
  exponent field uniform in [5, 9] (magnitudes 0.25 .. 7.5), mantissa
  uniform over its 8 values -- and one fp32 scale per expert and matrix,
  w_std / 3 times a factor uniform in [0.75, 1.25], so that the weights'
  spread matches the bf16 recipe.  Activations stay bf16 here; the layer
  quantises them itself.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass, field
from typing import Optional, Sequence

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libsynth.so")
_lock = threading.Lock()
_lib = None

# Stream ids: one independent random stream per tensor.
S_X, S_WR, S_BR, S_WGU, S_BGU, S_WD, S_BD = 1, 2, 3, 4, 5, 6, 7
S_GU_CODES, S_GU_SCALES, S_D_CODES, S_D_SCALES = 8, 9, 10, 11
# FP8 code fields (sign, exponent, mantissa) and per-expert scales
S_F8_GU_SIGN, S_F8_GU_EXP, S_F8_GU_MAN, S_F8_GU_SCALE = 12, 13, 14, 15
S_F8_D_SIGN, S_F8_D_EXP, S_F8_D_MAN, S_F8_D_SCALE = 16, 17, 18, 19
S_ATT_Q, S_ATT_K, S_ATT_V, S_ATT_SINK = 20, 21, 22, 23


def build(force: bool = False) -> str:
    """Compile ``libsynth.so`` next to this file (gcc, OpenMP)."""
    src = os.path.join(_HERE, "synth.c")
    if force or not os.path.exists(_LIB_PATH) or \
            os.path.getmtime(_LIB_PATH) < os.path.getmtime(src):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared",
                               "-ffp-contract=off", src, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB_PATH)
            vp, sz, u64, d, u32 = (ctypes.c_void_p, ctypes.c_size_t,
                                   ctypes.c_uint64, ctypes.c_double,
                                   ctypes.c_uint32)
            L.synth_normal_f32.argtypes = [vp, sz, u64, u64, d, d]
            L.synth_normal_bf16.argtypes = [vp, sz, u64, u64, d, d, d, d]
            L.synth_uniform_u8.argtypes = [vp, sz, u64, u64, u32, u32]
            L.synth_round_bf16.argtypes = [vp, vp, sz]
            L.synth_f32_to_bf16.argtypes = [ctypes.c_float]
            L.synth_f32_to_bf16.restype = ctypes.c_uint16
            _lib = L
    return _lib


def _empty(shape, dtype, pin):
    return torch.empty(shape, dtype=dtype, pin_memory=pin)


def normal_bf16(shape, seed, stream, mean=0.0, std=1.0, p_outlier=0.0,
                outlier_scale=20.0, pin=False) -> torch.Tensor:
    t = _empty(shape, torch.bfloat16, pin)
    lib().synth_normal_bf16(t.data_ptr(), t.numel(), seed, stream, mean, std,
                            p_outlier, outlier_scale)
    return t


def normal_f32(shape, seed, stream, mean=0.0, std=1.0, pin=False):
    t = _empty(shape, torch.float32, pin)
    lib().synth_normal_f32(t.data_ptr(), t.numel(), seed, stream, mean, std)
    return t


def uniform_u8(shape, seed, stream, lo, hi, pin=False) -> torch.Tensor:
    t = _empty(shape, torch.uint8, pin)
    lib().synth_uniform_u8(t.data_ptr(), t.numel(), seed, stream, lo, hi)
    return t


def round_bf16(t: torch.Tensor, pin=False) -> torch.Tensor:
    t = t.contiguous().to(torch.float32)
    out = _empty(tuple(t.shape), torch.bfloat16, pin)
    lib().synth_round_bf16(t.data_ptr(), out.data_ptr(), t.numel())
    return out


@dataclass
class Layer:
    """Host copies of one MoE layer's inputs (torch CPU tensors).

    bf16 tensors are ``torch.bfloat16``; MXFP4 codes and scales are
    ``torch.uint8``.  ``w_gu`` rows alternate gate/up features (row 2j is
    gate_j, row 2j+1 is up_j).
    """
    T: int
    H: int
    I: int
    E: int
    top_k: int
    wfmt: str                      # "bf16", "mxfp4", "fp8" or "mxfp4_mxfp8"
    x: torch.Tensor                # [T, H] bf16
    wr: torch.Tensor               # [E, H] bf16
    br: torch.Tensor               # [E] bf16
    w_gu: torch.Tensor             # [E, 2I, H] bf16 | [E, 2I, H/2] u8 | [E, 2I, H] u8 e4m3
    b_gu: torch.Tensor             # [E, 2I] bf16
    w_d: torch.Tensor              # [E, H, I] bf16 | [E, H, I/2] u8 | [E, H, I] u8 e4m3
    b_d: torch.Tensor              # [E, H] bf16
    s_gu: Optional[torch.Tensor] = None   # [E, 2I, H/32] u8 (mxfp4) | [E] fp32 (fp8)
    s_d: Optional[torch.Tensor] = None    # [E, H, I/32] u8 (mxfp4) | [E] fp32 (fp8)
    meta: dict = field(default_factory=dict)


def fp8_codes(shape, seed, streams, exp_lo=5, exp_hi=9, pin=False) -> torch.Tensor:
    """e4m3 bytes: sign, exponent field and mantissa drawn independently
    (the exponent range keeps clear of the NaN code 0x7F/0xFF)."""
    sign = uniform_u8(shape, seed, streams[0], 0, 1)
    ex = uniform_u8(shape, seed, streams[1], exp_lo, exp_hi)
    man = uniform_u8(shape, seed, streams[2], 0, 7)
    out = _empty(shape, torch.uint8, pin)
    out.copy_((sign << 7) | (ex << 3) | man)
    return out


def fp8_expert_scales(E, seed, stream, w_std, pin=False) -> torch.Tensor:
    """One fp32 scale per expert: w_std / 3 times a factor in [0.75, 1.25]."""
    u = uniform_u8((E,), seed, stream, 0, 255).to(torch.float32)
    out = _empty((E,), torch.float32, pin)
    out.copy_((w_std / 3.0) * (0.75 + 0.5 * u / 255.0))
    return out


def make_x(T, H, seed, p_outlier=0.0, outlier_scale=20.0, pin=False):
    """Activations: element i of stream S_X, so a smaller T is a prefix."""
    return normal_bf16((T, H), seed, S_X, 0.0, 1.0, p_outlier, outlier_scale,
                       pin)


def make_layer(E: int, T: int, H: int = 2880, I: int = 2880, top_k: int = 4,
               seed: int = 0, wfmt: str = "bf16",
               hot: Sequence[int] = (), hot_bias: float = 0.0,
               p_outlier: float = 0.0, outlier_scale: float = 20.0,
               w_std: float = 0.02, b_std: float = 0.01,
               router_w_std: Optional[float] = None,
               scale_lo: int = 119, scale_hi: int = 123,
               pin: bool = False, with_experts: bool = True) -> Layer:
    if wfmt not in ("bf16", "mxfp4", "fp8", "mxfp4_mxfp8"):
        raise ValueError(f"unknown weight format {wfmt!r}")
    rws = w_std if router_w_std is None else router_w_std
    x = make_x(T, H, seed, p_outlier, outlier_scale, pin)
    wr = normal_bf16((E, H), seed, S_WR, 0.0, rws, pin=pin)
    br32 = normal_f32((E,), seed, S_BR, 0.0, b_std)
    for e in hot:
        br32[e] += hot_bias
    br = round_bf16(br32, pin)
    s_gu = s_d = None
    b_gu = w_gu = b_d = w_d = None       # routing-only inputs keep these empty
    if with_experts:
        b_gu = normal_bf16((E, 2 * I), seed, S_BGU, 0.0, b_std, pin=pin)
        b_d = normal_bf16((E, H), seed, S_BD, 0.0, b_std, pin=pin)
    if not with_experts:
        pass
    elif wfmt == "bf16":
        w_gu = normal_bf16((E, 2 * I, H), seed, S_WGU, 0.0, w_std, pin=pin)
        w_d = normal_bf16((E, H, I), seed, S_WD, 0.0, w_std, pin=pin)
    elif wfmt == "fp8":
        w_gu = fp8_codes((E, 2 * I, H), seed, (S_F8_GU_SIGN, S_F8_GU_EXP, S_F8_GU_MAN), pin=pin)
        s_gu = fp8_expert_scales(E, seed, S_F8_GU_SCALE, w_std, pin)
        w_d = fp8_codes((E, H, I), seed, (S_F8_D_SIGN, S_F8_D_EXP, S_F8_D_MAN), pin=pin)
        s_d = fp8_expert_scales(E, seed, S_F8_D_SCALE, w_std, pin)
    else:
        if H % 32 or I % 32:
            raise ValueError("MXFP4 needs H and I multiples of 32")
        w_gu = uniform_u8((E, 2 * I, H // 2), seed, S_GU_CODES, 0, 255, pin)
        s_gu = uniform_u8((E, 2 * I, H // 32), seed, S_GU_SCALES, scale_lo,
                          scale_hi, pin)
        w_d = uniform_u8((E, H, I // 2), seed, S_D_CODES, 0, 255, pin)
        s_d = uniform_u8((E, H, I // 32), seed, S_D_SCALES, scale_lo,
                         scale_hi, pin)
    return Layer(T=T, H=H, I=I, E=E, top_k=top_k, wfmt=wfmt, x=x, wr=wr,
                 br=br, w_gu=w_gu, b_gu=b_gu, w_d=w_d, b_d=b_d, s_gu=s_gu,
                 s_d=s_d,
                 meta=dict(seed=seed, hot=tuple(hot), hot_bias=hot_bias,
                           p_outlier=p_outlier, outlier_scale=outlier_scale,
                           w_std=w_std, b_std=b_std))


# The five workload families.  Each is (E, seed, token counts, extra recipe).
WORKLOADS = {
    "20b_t8": dict(E=32, seed=0, Ts=(8,), wfmt="bf16"),
    "20b_decode": dict(E=32, seed=1, Ts=(1, 16, 64), wfmt="bf16"),
    "20b_prefill_skewed": dict(E=32, seed=2, Ts=(4096,), wfmt="bf16",
                               hot=(0, 1, 2, 3), hot_bias=2.0,
                               p_outlier=0.01, outlier_scale=20.0),
    "120b_shape": dict(E=128, seed=3, Ts=(1, 8, 64, 512, 4096, 8192),
                       wfmt="bf16"),
    "20b_mxfp4": dict(E=32, seed=4, Ts=(1, 64, 512), wfmt="mxfp4"),
    # FP8 W8A8 (the pages' quantised serving path, next after the five above)
    "20b_fp8": dict(E=32, seed=5, Ts=(1, 64, 512, 4096), wfmt="fp8"),
    # MXFP4 weights (the same as 20b_mxfp4: seed 4) with MXFP8 activations
    "20b_mxfp4_mxfp8": dict(E=32, seed=4, Ts=(1, 64, 512, 4096), wfmt="mxfp4_mxfp8"),
}


def make_workload(name: str, T: int, pin: bool = False, **over) -> Layer:
    """Full-size gpt-oss layer for one of the named workloads at T tokens."""
    w = dict(WORKLOADS[name])
    w.pop("Ts")
    w.update(over)
    return make_layer(T=T, pin=pin, **w)


def make_attention(Tq: int, Tkv: int, Hq: int = 64, Hkv: int = 8, D: int = 64, seed: int = 0,
                   qk_std: float = 1.0, sink_std: float = 1.0, pin: bool = False) -> dict:
    """Attention inputs of the gpt-oss block's shape (64 query heads, 8 KV
    heads, head_dim 64): q [Tq, Hq, D], k / v [Tkv, Hkv, D] bf16 ~ N(0, std)
    (q and k post-rotary stand-ins), sinks [Hq] fp32 ~ N(0, sink_std)."""
    return dict(q=normal_bf16((Tq, Hq, D), seed, S_ATT_Q, 0.0, qk_std, pin=pin),
                k=normal_bf16((Tkv, Hkv, D), seed, S_ATT_K, 0.0, qk_std, pin=pin),
                v=normal_bf16((Tkv, Hkv, D), seed, S_ATT_V, 0.0, 1.0, pin=pin),
                sinks=normal_f32((Hq,), seed, S_ATT_SINK, 0.0, sink_std))

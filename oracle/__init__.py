"""ctypes wrapper of the CPU oracle (``liboracle.so``).

TEST INFRASTRUCTURE ONLY: only tests/, ``__graft_entry__.smoke()`` and the
cpu_baseline / reference legs of ``bench.py`` may import this package.  It
shares no code with the CUDA library; the layer it computes is defined in
``moe_oracle.cpp`` (xserv docs/19-gpt-oss-moe.md, "Phase 19: gpt-oss-20b",
§1 model-architecture table and §2 MoE forward).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_DEFAULT_LIB = os.path.join(_HERE, "liboracle.so")
# A test may point the wrapper at a separately built copy (mutation tests).
_LIB_PATH = os.environ.get("GPT_OSS_ORACLE_LIB") or _DEFAULT_LIB
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``liboracle.so`` (g++, OpenMP, no FP contraction)."""
    if _LIB_PATH != _DEFAULT_LIB:
        return _LIB_PATH
    src = os.path.join(_HERE, "moe_oracle.cpp")
    hdr = os.path.join(_HERE, "moe_oracle.h")
    newest = max(os.path.getmtime(src), os.path.getmtime(hdr))
    if force or not os.path.exists(_LIB_PATH) or \
            os.path.getmtime(_LIB_PATH) < newest:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["g++", "-O2", "-std=c++17", "-fopenmp", "-fPIC",
                               "-shared", "-ffp-contract=off", src, "-o", tmp])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class OracleLayer(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int), ("H", ctypes.c_int), ("I", ctypes.c_int),
                ("E", ctypes.c_int), ("top_k", ctypes.c_int),
                ("wfmt", ctypes.c_int),
                ("x", ctypes.c_void_p), ("wr", ctypes.c_void_p),
                ("br", ctypes.c_void_p), ("w_gu", ctypes.c_void_p),
                ("s_gu", ctypes.c_void_p), ("b_gu", ctypes.c_void_p),
                ("w_d", ctypes.c_void_p), ("s_d", ctypes.c_void_p),
                ("b_d", ctypes.c_void_p)]


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB_PATH)
            vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
            P = ctypes.POINTER(OracleLayer)
            L.oracle_max_threads.restype = i
            L.oracle_glu.argtypes = [f, f]
            L.oracle_glu.restype = f
            L.oracle_e2m1.argtypes = [ctypes.c_uint]
            L.oracle_e2m1.restype = f
            L.oracle_e8m0.argtypes = [ctypes.c_uint8]
            L.oracle_e8m0.restype = f
            L.oracle_e4m3.argtypes = [ctypes.c_uint8]
            L.oracle_e4m3.restype = f
            L.oracle_e4m3_round.argtypes = [f]
            L.oracle_e4m3_round.restype = ctypes.c_uint8
            L.oracle_fp8_quantize_row.argtypes = [vp, i, vp, vp]
            L.oracle_mx_quantize_row.argtypes = [vp, i, vp, vp]
            L.oracle_router_logits.argtypes = [P, vp, i]
            L.oracle_topk_softmax.argtypes = [vp, i, i, i, vp, vp]
            L.oracle_permute.argtypes = [vp, i, i, i, vp, vp, vp]
            L.oracle_expert_ffn.argtypes = [P, i, i, vp, vp]
            L.oracle_forward_tokens.argtypes = [P, vp, i, vp, vp, vp, vp, i]
            L.oracle_moe_forward.argtypes = [P, vp, vp, vp, i]
            L.oracle_moe_forward_dense.argtypes = [P, vp, vp, vp, i]
            L.oracle_moe_forward_ep.argtypes = [P, i, i, vp, i, vp, i]
            L.oracle_attention_sinks.argtypes = [vp, vp, vp, vp, i, i, i, i, i, i, i, vp, i]
            L.oracle_dequant_mxfp4.argtypes = [vp, vp, i, i, vp]
            _lib = L
    return _lib


def _ptr(t):
    if t is None:
        return None
    assert t.device.type == "cpu" and t.is_contiguous()
    return t.data_ptr()


def _layer_struct(layer):
    """Build the C struct from a synth.Layer (keeps the tensors alive)."""
    s = OracleLayer(layer.T, layer.H, layer.I, layer.E, layer.top_k,
                    {"bf16": 0, "mxfp4": 1, "fp8": 2, "mxfp4_mxfp8": 3}[layer.wfmt],
                    _ptr(layer.x), _ptr(layer.wr), _ptr(layer.br),
                    _ptr(layer.w_gu), _ptr(layer.s_gu), _ptr(layer.b_gu),
                    _ptr(layer.w_d), _ptr(layer.s_d), _ptr(layer.b_d))
    return s


def max_threads() -> int:
    return lib().oracle_max_threads()


def glu(gate: float, up: float) -> float:
    return lib().oracle_glu(gate, up)


def e2m1(code: int) -> float:
    return lib().oracle_e2m1(code)


def e8m0(s: int) -> float:
    return lib().oracle_e8m0(s)


def e4m3(code: int) -> float:
    return lib().oracle_e4m3(code)


def e4m3_round(v: float) -> int:
    return lib().oracle_e4m3_round(v)


def fp8_quantize_row(x: torch.Tensor):
    """One token's bf16 activations -> (e4m3 codes uint8[n], scale)."""
    x = x.contiguous()
    assert x.dtype == torch.bfloat16 and x.dim() == 1
    codes = torch.empty(x.numel(), dtype=torch.uint8)
    scale = ctypes.c_float(0.0)
    lib().oracle_fp8_quantize_row(x.data_ptr(), x.numel(), codes.data_ptr(),
                                  ctypes.byref(scale))
    return codes, scale.value


def mx_quantize_row(x: torch.Tensor):
    """One token's bf16 activations (a multiple of 32) -> MXFP8 (e4m3 codes
    uint8[n], UE8M0 block scales uint8[n / 32])."""
    x = x.contiguous()
    assert x.dtype == torch.bfloat16 and x.dim() == 1 and x.numel() % 32 == 0
    codes = torch.empty(x.numel(), dtype=torch.uint8)
    scales = torch.empty(x.numel() // 32, dtype=torch.uint8)
    rc = lib().oracle_mx_quantize_row(x.data_ptr(), x.numel(), codes.data_ptr(),
                                      scales.data_ptr())
    assert rc == 0
    return codes, scales


def router_logits(layer, threads: int = 0) -> torch.Tensor:
    out = torch.empty((layer.T, layer.E), dtype=torch.float32)
    s = _layer_struct(layer)
    rc = lib().oracle_router_logits(ctypes.byref(s), out.data_ptr(), threads)
    assert rc == 0
    return out


def topk_softmax(logits: torch.Tensor, k: int):
    logits = logits.contiguous().to(torch.float32)
    T, E = logits.shape
    ids = torch.empty((T, k), dtype=torch.int32)
    w = torch.empty((T, k), dtype=torch.float32)
    rc = lib().oracle_topk_softmax(logits.data_ptr(), T, E, k, ids.data_ptr(),
                                   w.data_ptr())
    if rc != 0:
        raise ValueError("top_k must lie in [1, E]")
    return ids, w


def permute(ids: torch.Tensor, E: int):
    ids = ids.contiguous().to(torch.int32)
    T, k = ids.shape
    offsets = torch.empty(E + 1, dtype=torch.int32)
    sorted_assign = torch.empty(T * k, dtype=torch.int32)
    assign_row = torch.empty(T * k, dtype=torch.int32)
    rc = lib().oracle_permute(ids.data_ptr(), T, k, E, offsets.data_ptr(),
                              sorted_assign.data_ptr(), assign_row.data_ptr())
    if rc != 0:
        raise ValueError("expert id out of range")
    return offsets, sorted_assign, assign_row


def expert_ffn(layer, e: int, t: int):
    h = torch.empty(layer.I, dtype=torch.float32)
    y = torch.empty(layer.H, dtype=torch.float32)
    s = _layer_struct(layer)
    lib().oracle_expert_ffn(ctypes.byref(s), e, t, h.data_ptr(), y.data_ptr())
    return h, y


def forward(layer, tokens=None, threads: int = 0, want_logits: bool = False):
    """Routed forward.  Returns (ids[n,k], w[n,k], out[n,H] fp32[, logits])."""
    s = _layer_struct(layer)
    if tokens is None:
        n, tok_ptr = layer.T, None
    else:
        tokens = torch.as_tensor(tokens, dtype=torch.int32).contiguous()
        n, tok_ptr = tokens.numel(), tokens.data_ptr()
    k = layer.top_k
    ids = torch.empty((n, k), dtype=torch.int32)
    w = torch.empty((n, k), dtype=torch.float32)
    out = torch.empty((n, layer.H), dtype=torch.float32)
    logits = torch.empty((n, layer.E), dtype=torch.float32) if want_logits \
        else None
    rc = lib().oracle_forward_tokens(ctypes.byref(s), tok_ptr, n,
                                     ids.data_ptr(), w.data_ptr(),
                                     _ptr(logits), out.data_ptr(), threads)
    if rc != 0:
        raise ValueError("top_k must lie in [1, E]")
    if want_logits:
        return ids, w, out, logits
    return ids, w, out


def forward_ep(layer, ex_lo: int, ex_n: int, tokens=None, threads: int = 0) -> torch.Tensor:
    """Partial output [n, H] fp32 of the experts [ex_lo, ex_lo + ex_n)."""
    s = _layer_struct(layer)
    if tokens is None:
        n, tok_ptr = layer.T, None
    else:
        tokens = torch.as_tensor(tokens, dtype=torch.int32).contiguous()
        n, tok_ptr = tokens.numel(), tokens.data_ptr()
    out = torch.empty((n, layer.H), dtype=torch.float32)
    rc = lib().oracle_moe_forward_ep(ctypes.byref(s), ex_lo, ex_n, tok_ptr, n,
                                     out.data_ptr(), threads)
    assert rc == 0
    return out


def attention_sinks(q, k, v, sinks, window: int = 0, q_start=None, threads: int = 0):
    """q [Tq, Hq, D], k / v [Tkv, Hkv, D] bf16, sinks [Hq] fp32 -> out
    [Tq, Hq, D] fp32 (fp64 inside).  q_start defaults to Tkv - Tq."""
    q, k, v = q.contiguous(), k.contiguous(), v.contiguous()
    sinks = sinks.to(torch.float32).contiguous()
    assert q.dtype == k.dtype == v.dtype == torch.bfloat16
    Tq, Hq, D = q.shape
    Tkv, Hkv, _ = k.shape
    if q_start is None:
        q_start = Tkv - Tq
    out = torch.empty((Tq, Hq, D), dtype=torch.float32)
    rc = lib().oracle_attention_sinks(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                      sinks.data_ptr(), Tq, Tkv, Hq, Hkv, D, window,
                                      q_start, out.data_ptr(), threads)
    assert rc == 0
    return out


def forward_dense(layer, threads: int = 0):
    s = _layer_struct(layer)
    k = layer.top_k
    ids = torch.empty((layer.T, k), dtype=torch.int32)
    w = torch.empty((layer.T, k), dtype=torch.float32)
    out = torch.empty((layer.T, layer.H), dtype=torch.float32)
    rc = lib().oracle_moe_forward_dense(ctypes.byref(s), ids.data_ptr(),
                                        w.data_ptr(), out.data_ptr(), threads)
    if rc != 0:
        raise ValueError("top_k must lie in [1, E]")
    return ids, w, out


def dequant_mxfp4(codes: torch.Tensor, scales: torch.Tensor) -> torch.Tensor:
    codes = codes.contiguous()
    scales = scales.contiguous()
    K = codes.shape[-1] * 2
    rows = codes.numel() // codes.shape[-1]
    out = torch.empty(tuple(codes.shape[:-1]) + (K,), dtype=torch.float32)
    rc = lib().oracle_dequant_mxfp4(codes.data_ptr(), scales.data_ptr(), rows,
                                    K, out.data_ptr())
    assert rc == 0
    return out

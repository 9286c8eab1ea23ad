"""Python binding of the gpt-oss MoE layer library (``include/moe.h``).

Argument marshalling only: every step of the layer runs in the CUDA kernels
of ``libgpt_oss_moe.so``.  PyTorch supplies device memory and streams.  The
names mirror the C ABI (``moe_route``, ``moe_forward``, ...).  There is no
fallback: if the library has not been built, importing the binding's calls
raises.

Build the library with ``python -c "import __graft_entry__ as g; g.build()"``
or ``python gpt_oss_moe_gb300/_build.py``.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
# GPT_OSS_MOE_LIB selects another build of the same library (the
# MOE_DEBUG_BOUNDS variant, libgpt_oss_moe_debug_bounds.so)
LIB_PATH = os.environ.get("GPT_OSS_MOE_LIB") or os.path.join(_PKG, "libgpt_oss_moe.so")

MOE_W_BF16, MOE_W_MXFP4, MOE_W_FP8, MOE_W_MXFP4_MXFP8 = 0, 1, 2, 3
MOE_DEV_BAD_EXPERT_ID, MOE_DEV_WAIT_TIMEOUT, MOE_DEV_BAD_TILE = 0x1, 0x2, 0x4
MOE_DEV_NONFINITE, MOE_DEV_BOUNDS, MOE_DEV_RANGE = 0x8, 0x10, 0x20

# Every function the C header declares, in order (checked by the tests).
EXPORTS = ("moe_workspace_bytes", "moe_route", "moe_forward", "moe_forward_ep",
           "moe_forward_noalloc", "moe_get_device_status",
           "moe_clear_device_status", "moe_stage_stats", "moe_trace_read",
           "moe_set_tuning", "moe_profile_enable", "moe_profile_read",
           "moe_status_str", "moe_attention_sinks", "moe_attention_workspace_bytes")


class MoEError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {moe_status_str(code)} (status {code})")


class moe_shape(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int), ("H", ctypes.c_int), ("I", ctypes.c_int),
                ("E", ctypes.c_int), ("top_k", ctypes.c_int),
                ("wfmt", ctypes.c_int)]


class moe_attn_shape(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in ("Tq", "Tkv", "Hq", "Hkv", "D", "window",
                                            "q_start")]


class moe_weight(ctypes.Structure):
    _fields_ = [("w", ctypes.c_void_p), ("scale", ctypes.c_void_p),
                ("bias", ctypes.c_void_p)]


_lib = None
_lock = threading.Lock()


def lib():
    """The loaded library; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise ImportError(
                    f"{LIB_PATH} is missing: build it first "
                    "(python gpt_oss_moe_gb300/_build.py)")
            L = ctypes.CDLL(LIB_PATH)
            vp, i, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
            S = ctypes.POINTER(moe_shape)
            L.moe_workspace_bytes.argtypes = [S]
            L.moe_workspace_bytes.restype = sz
            L.moe_route.argtypes = [S, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
            L.moe_route.restype = i
            L.moe_forward.argtypes = [S, vp, vp, vp, moe_weight, moe_weight, vp, i,
                                      vp, vp, vp, sz, vp]
            L.moe_forward.restype = i
            L.moe_forward_ep.argtypes = [S, i, i, vp, vp, vp, moe_weight, moe_weight, vp, i,
                                         vp, vp, vp, sz, vp]
            L.moe_forward_ep.restype = i
            L.moe_attention_sinks.argtypes = [ctypes.POINTER(moe_attn_shape), vp, vp, vp, vp,
                                              vp, vp, sz, vp]
            L.moe_attention_sinks.restype = i
            L.moe_attention_workspace_bytes.argtypes = [ctypes.POINTER(moe_attn_shape)]
            L.moe_attention_workspace_bytes.restype = sz
            L.moe_forward_noalloc.argtypes = [S, vp, vp, vp, moe_weight, moe_weight,
                                              vp, i, vp, vp, vp, vp]
            L.moe_forward_noalloc.restype = i
            L.moe_get_device_status.argtypes = [vp, ctypes.POINTER(ctypes.c_int32)]
            L.moe_get_device_status.restype = i
            L.moe_clear_device_status.argtypes = [vp, vp]
            L.moe_clear_device_status.restype = i
            L.moe_stage_stats.argtypes = [vp, ctypes.POINTER(ctypes.c_int32),
                                          ctypes.POINTER(ctypes.c_float)]
            L.moe_stage_stats.restype = i
            L.moe_trace_read.argtypes = [ctypes.POINTER(ctypes.c_uint64), sz,
                                         ctypes.POINTER(sz)]
            L.moe_trace_read.restype = i
            L.moe_set_tuning.argtypes = [ctypes.c_char_p, i]
            L.moe_set_tuning.restype = i
            L.moe_profile_enable.argtypes = [i]
            L.moe_profile_enable.restype = i
            L.moe_profile_read.argtypes = [ctypes.POINTER(ctypes.c_char_p),
                                           ctypes.POINTER(ctypes.c_float), i,
                                           ctypes.POINTER(ctypes.c_int)]
            L.moe_profile_read.restype = i
            L.moe_status_str.argtypes = [i]
            L.moe_status_str.restype = ctypes.c_char_p
            _lib = L
    return _lib


def _p(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensors passed to the library must live on the GPU")
    if not t.is_contiguous():
        raise ValueError("tensors passed to the library must be contiguous")
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _check(code: int, where: str):
    if code != 0:
        raise MoEError(code, where)


def make_shape(T, H, I, E, top_k, wfmt=MOE_W_BF16) -> moe_shape:
    return moe_shape(int(T), int(H), int(I), int(E), int(top_k), int(wfmt))


def moe_status_str(code: int) -> str:
    return lib().moe_status_str(int(code)).decode()


def moe_workspace_bytes(shape: moe_shape) -> int:
    return lib().moe_workspace_bytes(ctypes.byref(shape))


def alloc_workspace(shape: moe_shape, device=None) -> torch.Tensor:
    """Zeroed device workspace (status word cleared) for ``shape``."""
    n = moe_workspace_bytes(shape)
    if n == 0:
        raise MoEError(-2, "moe_workspace_bytes")
    return torch.zeros(n, dtype=torch.uint8, device=device or "cuda")


def moe_route(shape, hidden, router_w, router_b, topk_ids=None, topk_w=None,
              expert_offsets=None, sorted_assign=None, workspace=None,
              stream=None):
    ws = workspace if workspace is not None else alloc_workspace(shape, hidden.device)
    code = lib().moe_route(ctypes.byref(shape), _p(hidden), _p(router_w),
                           _p(router_b), _p(topk_ids), _p(topk_w),
                           _p(expert_offsets), _p(sorted_assign), _p(ws),
                           ws.numel(), _stream(stream))
    _check(code, "moe_route")
    return ws


def moe_forward(shape, hidden, router_w, router_b, w_gu, b_gu, w_d, b_d,
                out, s_gu=None, s_d=None, topk_ids_out=None, topk_w_out=None,
                workspace=None, stream=None):
    """Enqueue the layer forward; ``out`` is fp32 or bf16 [T, H]."""
    ws = workspace if workspace is not None else alloc_workspace(shape, hidden.device)
    gu = moe_weight(_p(w_gu), _p(s_gu), _p(b_gu))
    dn = moe_weight(_p(w_d), _p(s_d), _p(b_d))
    out_f32 = 1 if out.dtype == torch.float32 else 0
    if not out_f32 and out.dtype != torch.bfloat16:
        raise ValueError("out must be float32 or bfloat16")
    code = lib().moe_forward(ctypes.byref(shape), _p(hidden), _p(router_w),
                             _p(router_b), gu, dn, _p(out), out_f32,
                             _p(topk_ids_out), _p(topk_w_out), _p(ws),
                             ws.numel(), _stream(stream))
    _check(code, "moe_forward")
    return ws


def moe_forward_ep(shape, expert_start, local_experts, hidden, router_w, router_b,
                   w_gu, b_gu, w_d, b_d, out, s_gu=None, s_d=None, topk_ids_out=None,
                   topk_w_out=None, workspace=None, stream=None):
    """Expert-parallel forward: this device's partial output over the experts
    [expert_start, expert_start + local_experts), whose banks alone are given
    (w_gu, b_gu, w_d, b_d, s_gu, s_d hold local_experts experts); routing uses
    the router of all shape.E experts.  Sum the devices' partial outputs
    (ep_all_reduce) for the layer's output."""
    ws = workspace if workspace is not None else alloc_workspace(shape, hidden.device)
    gu = moe_weight(_p(w_gu), _p(s_gu), _p(b_gu))
    dn = moe_weight(_p(w_d), _p(s_d), _p(b_d))
    out_f32 = 1 if out.dtype == torch.float32 else 0
    if not out_f32 and out.dtype != torch.bfloat16:
        raise ValueError("out must be float32 or bfloat16")
    code = lib().moe_forward_ep(ctypes.byref(shape), int(expert_start), int(local_experts),
                                _p(hidden), _p(router_w), _p(router_b), gu, dn, _p(out),
                                out_f32, _p(topk_ids_out), _p(topk_w_out), _p(ws),
                                ws.numel(), _stream(stream))
    _check(code, "moe_forward_ep")
    return ws


def attention_sinks(q, k, v, sinks, out=None, window: int = 0, q_start=None, workspace=None,
                    stream=None):
    """Attention with sinks on the GPU: q [Tq, Hq, 64], k / v [Tkv, Hkv, 64]
    bf16, sinks [Hq] fp32 -> out [Tq, Hq, 64] fp32 (see moe_attention_sinks)."""
    Tq, Hq, D = q.shape
    Tkv, Hkv, _ = k.shape
    if out is None:
        out = torch.empty((Tq, Hq, D), dtype=torch.float32, device=q.device)
    shape = moe_attn_shape(int(Tq), int(Tkv), int(Hq), int(Hkv), int(D), int(window),
                           int(Tkv - Tq if q_start is None else q_start))
    need = lib().moe_attention_workspace_bytes(ctypes.byref(shape))
    if need and (workspace is None or workspace.numel() < need):
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    code = lib().moe_attention_sinks(ctypes.byref(shape), _p(q), _p(k), _p(v), _p(sinks),
                                     _p(out), _p(workspace) if need else None,
                                     workspace.numel() if need else 0, _stream(stream))
    _check(code, "moe_attention_sinks")
    return out


def ep_expert_range(rank: int, world: int, num_experts: int):
    """Contiguous expert range (start, count) of one rank: E / world each,
    the first E % world ranks one more."""
    if world < 1 or not 0 <= rank < world or num_experts < world:
        raise ValueError("need 0 <= rank < world <= num_experts")
    base, extra = divmod(num_experts, world)
    start = rank * base + min(rank, extra)
    return start, base + (1 if rank < extra else 0)


def ep_all_reduce(partial: torch.Tensor, group=None) -> torch.Tensor:
    """Sums the ranks' partial outputs in place (torch.distributed: NCCL
    for device tensors, gloo for host tensors) and returns them."""
    import torch.distributed as dist
    dist.all_reduce(partial, op=dist.ReduceOp.SUM, group=group)
    return partial


def moe_forward_noalloc(shape, hidden, router_w, router_b, w_gu, b_gu, w_d, b_d,
                        out, s_gu=None, s_d=None, topk_ids_out=None,
                        topk_w_out=None, device_status_out=None, stream=None):
    """The layer forward without a workspace, for callers that cannot
    allocate device memory: the scratch is the library's own static device
    array (shapes up to MOE_NOALLOC_SCRATCH_BYTES of scratch).  Calls share
    that array, so calls that overlap on the GPU race."""
    gu = moe_weight(_p(w_gu), _p(s_gu), _p(b_gu))
    dn = moe_weight(_p(w_d), _p(s_d), _p(b_d))
    out_f32 = 1 if out.dtype == torch.float32 else 0
    if not out_f32 and out.dtype != torch.bfloat16:
        raise ValueError("out must be float32 or bfloat16")
    code = lib().moe_forward_noalloc(ctypes.byref(shape), _p(hidden), _p(router_w),
                                     _p(router_b), gu, dn, _p(out), out_f32,
                                     _p(topk_ids_out), _p(topk_w_out),
                                     _p(device_status_out), _stream(stream))
    _check(code, "moe_forward_noalloc")


def moe_get_device_status(workspace: torch.Tensor) -> int:
    """Synchronising read of the device status word (0 = no error)."""
    v = ctypes.c_int32(0)
    code = lib().moe_get_device_status(_p(workspace), ctypes.byref(v))
    if code not in (0, -7):
        _check(code, "moe_get_device_status")
    return v.value


def moe_stage_stats(workspace: torch.Tensor):
    """Synchronising read of the stage checks (MOE_CHECK_STAGES=1):
    [(non-finite count, largest finite magnitude)] for the gathered
    activations, h and the output of the last checked call."""
    nf = (ctypes.c_int32 * 3)()
    mx = (ctypes.c_float * 3)()
    _check(lib().moe_stage_stats(_p(workspace), nf, mx), "moe_stage_stats")
    return [(int(nf[i]), float(mx[i])) for i in range(3)]


def moe_trace_read():
    """Phase timestamps of the last call (trace build only): a dict of
    int64 tensors router [512, 8], permute [512, 8], gemm [2, 512, 8],
    attn [2, 512, 8]."""
    cap = 6 * 512 * 8
    buf = (ctypes.c_uint64 * cap)()
    n = ctypes.c_size_t(0)
    _check(lib().moe_trace_read(buf, cap, ctypes.byref(n)), "moe_trace_read")
    t = torch.tensor(list(buf[:n.value]), dtype=torch.int64)
    return {"router": t[:4096].view(512, 8), "permute": t[4096:8192].view(512, 8),
            "gemm": t[8192:16384].view(2, 512, 8), "attn": t[16384:].view(2, 512, 8)}


def moe_clear_device_status(workspace: torch.Tensor, stream=None):
    _check(lib().moe_clear_device_status(_p(workspace), _stream(stream)),
           "moe_clear_device_status")


def moe_set_tuning(key: str, value: int):
    _check(lib().moe_set_tuning(key.encode(), int(value)), "moe_set_tuning")


def moe_profile_enable(calls: int):
    """Record per-kernel events for the next ``calls`` calls (0 = off)."""
    _check(lib().moe_profile_enable(int(calls)), "moe_profile_enable")


def moe_profile_read(cap: int = 8):
    """[(kernel name, mean milliseconds over the recorded calls)]."""
    names = (ctypes.c_char_p * cap)()
    ms = (ctypes.c_float * cap)()
    n = ctypes.c_int(0)
    _check(lib().moe_profile_read(names, ms, cap, ctypes.byref(n)),
           "moe_profile_read")
    return [(names[i].decode(), float(ms[i])) for i in range(n.value)]


def layer_shape(layer, T=None) -> moe_shape:
    """Shape of a synthetic layer object (fields T, H, I, E, top_k, wfmt)."""
    return make_shape(layer.T if T is None else T, layer.H, layer.I, layer.E,
                      layer.top_k,
                      {"bf16": MOE_W_BF16, "mxfp4": MOE_W_MXFP4, "fp8": MOE_W_FP8,
                       "mxfp4_mxfp8": MOE_W_MXFP4_MXFP8}[layer.wfmt])

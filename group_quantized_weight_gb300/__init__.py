"""Python binding of libgq, the GB300 group-quantized weight-only GEMM.

Argument marshalling only: every function forwards to the C ABI of ``include/gq.h`` with
the same name; all computation happens in the library's CUDA kernels.  The library must
have been built (``group_quantized_weight_gb300.build.build()``); importing this module
without it raises ImportError — there is no fallback.

Tensors are passed as raw device pointers; the ``*_t`` helpers accept torch tensors and
pass ``tensor.data_ptr()`` and torch's current CUDA stream.
"""
from __future__ import annotations

import ctypes
import os

from .constants import (GQ_W4, GQ_ZP, GQ_ACT_F32, GQ_SC_BF16, GQ_SC_F32, GQ_OUT_F32,  # noqa: F401
                        GQ_OK, STATUS_NAMES, GqError, algorithmic_bytes, gemm_flops, prec_flags)

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_lib", "libgq.so")

if not os.path.exists(_LIB_PATH):
    raise ImportError(f"libgq.so is not built ({_LIB_PATH}); run "
                      "group_quantized_weight_gb300.build.build() first")

_lib = ctypes.CDLL(_LIB_PATH)
LIB_PATH = _LIB_PATH

_i, _p, _sz = ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t


class gq_plan_t(ctypes.Structure):
    _fields_ = [("path", _i), ("nsplit", _i), ("m_tile", _i), ("n_tile", _i),
                ("grid_x", _i), ("grid_y", _i), ("grid_z", _i), ("block_threads", _i),
                ("smem_bytes", _sz), ("workspace_bytes", _sz)]


class gq_bench_args(ctypes.Structure):
    _fields_ = [("M", _i), ("K", _i), ("N", _i), ("G", _i), ("prec", _i), ("A", _p),
                ("Wq", ctypes.POINTER(_p)), ("scales", ctypes.POINTER(_p)),
                ("zeros", ctypes.POINTER(_p)), ("n_copies", _i), ("out", _p),
                ("warmup", _i), ("iters", _i), ("use_graph", _i), ("stream", _p),
                ("a_scales", _p)]


class gq_bench_result(ctypes.Structure):
    _fields_ = [("us_per_call", ctypes.c_double), ("launches_per_call", _i)]


_SIGS = {
    "gq_packed_bytes": [_i, _i, _i, _i, ctypes.POINTER(_sz)],
    "gq_pack_weights": [_i, _i, _i, _i, _p, _p, _p],
    "gq_workspace_size": [_i, _i, _i, _i, _i, ctypes.POINTER(_sz)],
    "gq_set_workspace": [_p, _sz],
    "gq_gemm": [_i, _i, _i, _i, _i, _p, _p, _p, _p, _p, _p],
    "gq_gemm_host": [_i, _i, _i, _i, _i, _p, _p, _p, _p, _p, _p, _p, _p],
    "gq_gemm_static_scratch": [_i, _i, _i, _i, _i, _p, _p, _p, _p, _p, _p],
    "gq_gemm_a8": [_i, _i, _i, _i, _i, _p, _p, _p, _p, _p, _p],
    "gq_quantize_act": [_i, _i, _i, _i, _p, _p, _p, _p],
    "gq_gemm_fp8_block": [_i, _i, _i, _i, _p, _p, _p, _p, _p, _p],
    "gq_quantize_act_fp8": [_i, _i, _i, _p, _p, _p, _p],
    "gq_bench_calls": [ctypes.POINTER(gq_bench_args), ctypes.POINTER(gq_bench_result)],
    "gq_bench": [ctypes.c_char_p, ctypes.c_char_p, _sz],
    "gq_plan": [_i, _i, _i, _i, _i, _i, ctypes.POINTER(gq_plan_t)],
    "gq_zsplit": [_i, _i, _i, ctypes.POINTER(_i), ctypes.POINTER(_i)],
    "gq_set_split_override": [_i],
    "gq_set_wait_limit": [ctypes.c_longlong],
    "gq_set_fault_injection": [_i],
    "gq_device_error": [_i],
    "gq_status_string": [_i],
    "gq_last_error_detail": [],
}
for _name, _args in _SIGS.items():
    _f = getattr(_lib, _name)
    _f.argtypes = _args
    _f.restype = ctypes.c_char_p if _name in ("gq_status_string", "gq_last_error_detail") else _i

EXPORTED = tuple(_SIGS)


def _check(st: int, what: str) -> None:
    if st != GQ_OK:
        msg = f"{what}: {_lib.gq_status_string(st).decode()}"
        if st == 5:
            msg += f" ({_lib.gq_last_error_detail().decode()})"
        raise GqError(st, msg)


def gq_status_string(status: int) -> str:
    return _lib.gq_status_string(status).decode()


def gq_last_error_detail() -> str:
    return _lib.gq_last_error_detail().decode()


def gq_packed_bytes(K: int, N: int, G: int, prec: int) -> int:
    out = _sz()
    _check(_lib.gq_packed_bytes(K, N, G, prec, ctypes.byref(out)), "gq_packed_bytes")
    return out.value


def gq_pack_weights(K, N, G, prec, codes_ptr, packed_ptr, stream=None) -> int:
    """Raw call; returns the status."""
    return _lib.gq_pack_weights(K, N, G, prec, codes_ptr, packed_ptr, stream)


def gq_workspace_size(M: int, K: int, N: int, G: int, prec: int) -> int:
    out = _sz()
    _check(_lib.gq_workspace_size(M, K, N, G, prec, ctypes.byref(out)), "gq_workspace_size")
    return out.value


def gq_set_workspace(ptr, nbytes: int) -> int:
    return _lib.gq_set_workspace(ptr, nbytes)


def gq_gemm(M, K, N, G, prec, A_ptr, Wq_ptr, scales_ptr, zeros_ptr, out_ptr, stream=None) -> int:
    """Raw call; returns the status."""
    return _lib.gq_gemm(M, K, N, G, prec, A_ptr, Wq_ptr, scales_ptr, zeros_ptr, out_ptr, stream)


def gq_gemm_host(M, K, N, G, prec, A_host_ptr, A_dev_ptr, Wq_ptr, scales_ptr, zeros_ptr,
                 out_dev_ptr, out_host_ptr, stream=None) -> int:
    """gq_gemm on host activations and output (copied in and out on the stream).  Raw call;
    returns the status."""
    return _lib.gq_gemm_host(M, K, N, G, prec, A_host_ptr, A_dev_ptr, Wq_ptr, scales_ptr,
                             zeros_ptr, out_dev_ptr, out_host_ptr, stream)


def gq_gemm_a8(M, K, N, G, prec, Aq_ptr, a_scales_ptr, Wq_ptr, scales_ptr, out_ptr,
               stream=None) -> int:
    """W8A8 group GEMM (GQ_ACT_I8).  Raw call; returns the status."""
    return _lib.gq_gemm_a8(M, K, N, G, prec, Aq_ptr, a_scales_ptr, Wq_ptr, scales_ptr, out_ptr,
                           stream)


def gq_quantize_act(M, K, G, prec, A_ptr, Aq_ptr, a_scales_ptr, stream=None) -> int:
    """Dynamic per-group INT8 quantization of activations.  Raw call; returns the status."""
    return _lib.gq_quantize_act(M, K, G, prec, A_ptr, Aq_ptr, a_scales_ptr, stream)


def gq_gemm_fp8_block(M, K, N, prec, A_ptr, a_scales_ptr, W_ptr, w_scales_ptr, out_ptr,
                      stream=None) -> int:
    """FP8 W8A8 GEMM with 1 x 128 activation and 128 x 128 weight block scales.  Raw call;
    returns the status."""
    return _lib.gq_gemm_fp8_block(M, K, N, prec, A_ptr, a_scales_ptr, W_ptr, w_scales_ptr,
                                  out_ptr, stream)


def gq_quantize_act_fp8(M, K, prec, A_ptr, Aq_ptr, a_scales_ptr, stream=None) -> int:
    """Dynamic FP8 (E4M3) quantization of activations per 1 x 128 block.  Raw call."""
    return _lib.gq_quantize_act_fp8(M, K, prec, A_ptr, Aq_ptr, a_scales_ptr, stream)


def gq_gemm_static_scratch(M, K, N, G, prec, A_ptr, Wq_ptr, scales_ptr, zeros_ptr, out_ptr,
                           stream=None) -> int:
    """gq_gemm that never allocates: scratch comes from a fixed array inside the library
    (GQ_STATIC_SCRATCH_BYTES).  Raw call; returns the status."""
    return _lib.gq_gemm_static_scratch(M, K, N, G, prec, A_ptr, Wq_ptr, scales_ptr, zeros_ptr,
                                       out_ptr, stream)


GQ_STATIC_SCRATCH_BYTES = 4 << 20


def gq_plan(M: int, K: int, N: int, G: int, prec: int, sm_count: int = 0) -> dict:
    p = gq_plan_t()
    _check(_lib.gq_plan(M, K, N, G, prec, sm_count, ctypes.byref(p)), "gq_plan")
    return {f: getattr(p, f) for f, _ in gq_plan_t._fields_}


def gq_zsplit(units: int, nsplit: int, z: int):
    b, e = _i(), _i()
    _check(_lib.gq_zsplit(units, nsplit, z, ctypes.byref(b), ctypes.byref(e)), "gq_zsplit")
    return b.value, e.value


def gq_set_split_override(n: int) -> int:
    """Force the K-slice count of the split-K paths (0 = planner's choice, -1 = the largest);
    returns the previous setting."""
    return _lib.gq_set_split_override(n)


def gq_set_wait_limit(cycles: int) -> int:
    """SM clock cycles after which a bounded device-side wait gives up (0 = the default);
    returns the status."""
    return _lib.gq_set_wait_limit(cycles)


def gq_set_fault_injection(fault: int) -> int:
    """Inject a failure (GQ_FAULT_* of gq.h; 0 = none); returns the previous setting."""
    return _lib.gq_set_fault_injection(fault)


def gq_device_error(clear: bool = False) -> int:
    return _lib.gq_device_error(1 if clear else 0)


def gq_bench(config: str, cap: int = 1 << 16):
    """Self-contained benchmark of a named workload ("all" for every one); returns the parsed
    JSON the library writes (a dict, or a list for "all")."""
    import json
    buf = ctypes.create_string_buffer(cap)
    _check(_lib.gq_bench(config.encode(), buf, cap), "gq_bench")
    return json.loads(buf.value.decode())


def gq_bench_calls(M, K, N, G, prec, A_ptr, Wq_ptrs, scales_ptrs, zeros_ptrs, out_ptr, *,
                   warmup=3, iters=100, use_graph=True, stream=None, a_scales_ptr=None) -> dict:
    n = len(Wq_ptrs)
    arr = _p * n
    args = gq_bench_args(M, K, N, G, prec, A_ptr, arr(*Wq_ptrs), arr(*scales_ptrs),
                         arr(*zeros_ptrs) if zeros_ptrs else None, n, out_ptr, warmup, iters,
                         1 if use_graph else 0, stream, a_scales_ptr)
    res = gq_bench_result()
    _check(_lib.gq_bench_calls(ctypes.byref(args), ctypes.byref(res)), "gq_bench_calls")
    return {"us_per_call": res.us_per_call, "launches_per_call": res.launches_per_call}


# ------------------------------------------------------------------ torch conveniences

def _stream_ptr(stream):
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def pack_weights_t(codes, K: int, N: int, G: int, prec: int, stream=None):
    """codes: device tensor in the canonical layout -> packed device tensor (uint8)."""
    import torch
    packed = torch.empty(gq_packed_bytes(K, N, G, prec), dtype=torch.uint8, device=codes.device)
    _check(gq_pack_weights(K, N, G, prec, codes.data_ptr(), packed.data_ptr(),
                           _stream_ptr(stream)), "gq_pack_weights")
    return packed


def quantize_act_t(A, K: int, G: int, prec: int = 0, stream=None):
    """A [M][K] (bf16 bits as int16/bfloat16, or fp32 with GQ_ACT_F32) -> (Aq int8 [M][K],
    a_scales fp32 [M][K/G]) on torch's current stream."""
    import torch
    M = A.shape[0]
    Aq = torch.empty((M, K), dtype=torch.int8, device=A.device)
    As = torch.empty((M, K // G), dtype=torch.float32, device=A.device)
    _check(gq_quantize_act(M, K, G, prec, A.data_ptr(), Aq.data_ptr(), As.data_ptr(),
                           _stream_ptr(stream)), "gq_quantize_act")
    return Aq, As


def gemm_a8_t(Aq, As, Wq, scales, out, M: int, K: int, N: int, G: int, prec: int, stream=None):
    """out <- gq_gemm_a8(...) on torch's current stream; raises GqError on a bad status."""
    _check(gq_gemm_a8(M, K, N, G, prec, Aq.data_ptr(), As.data_ptr(), Wq.data_ptr(),
                      scales.data_ptr(), out.data_ptr(), _stream_ptr(stream)), "gq_gemm_a8")
    return out


def quantize_act_fp8_t(A, K: int, prec: int = 0, stream=None):
    """A [M][K] (bf16 bits, or fp32 with GQ_ACT_F32) -> (Aq uint8 E4M3 [M][K], a_scales fp32
    [K/128][M]) on torch's current stream."""
    import torch
    M = A.shape[0]
    Aq = torch.empty((M, K), dtype=torch.uint8, device=A.device)
    As = torch.empty((K // 128, M), dtype=torch.float32, device=A.device)
    _check(gq_quantize_act_fp8(M, K, prec, A.data_ptr(), Aq.data_ptr(), As.data_ptr(),
                               _stream_ptr(stream)), "gq_quantize_act_fp8")
    return Aq, As


def gemm_fp8_t(A, a_scales, W, w_scales, out, M: int, K: int, N: int, prec: int = 0,
               stream=None):
    """out <- gq_gemm_fp8_block(...) on torch's current stream; raises GqError on a bad status."""
    _check(gq_gemm_fp8_block(M, K, N, prec, A.data_ptr(), a_scales.data_ptr(), W.data_ptr(),
                             w_scales.data_ptr(), out.data_ptr(), _stream_ptr(stream)),
           "gq_gemm_fp8_block")
    return out


def gemm_t(A, Wq, scales, zeros, out, M: int, K: int, N: int, G: int, prec: int, stream=None):
    """out <- gq_gemm(...) on torch's current stream; raises GqError on a bad status."""
    _check(gq_gemm(M, K, N, G, prec, A.data_ptr(), Wq.data_ptr(), scales.data_ptr(),
                   zeros.data_ptr() if zeros is not None else None, out.data_ptr(),
                   _stream_ptr(stream)), "gq_gemm")
    return out

"""Shared test plumbing: build/load the library, move generator inputs to the device,
decode outputs.  No arithmetic of the method lives here."""
from __future__ import annotations

import importlib.util
import os

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def ensure_built():
    spec = importlib.util.spec_from_file_location(
        "_gq_build", os.path.join(ROOT, "group_quantized_weight_gb300", "build.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod.build()


def load():
    ensure_built()
    import group_quantized_weight_gb300 as gq
    return gq


def prec_of(cfg) -> int:
    from group_quantized_weight_gb300.constants import prec_flags
    return prec_flags(cfg.w4, cfg.zp, cfg.act, cfg.sc, cfg.out, zf=cfg.zf)


def np_to_dev(a: np.ndarray):
    import torch
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        t = torch.from_numpy(a.view(np.int16))
    elif a.dtype == np.uint32:
        t = torch.from_numpy(a.view(np.int32))
    else:
        t = torch.from_numpy(a)
    return t.cuda()


def out_to_f64(out, out_dtype: str) -> np.ndarray:
    import oracle
    import torch
    if out_dtype == "bf16":
        return oracle.bf16_bits_to_f64(out.view(torch.int16).cpu().numpy().view(np.uint16))
    return out.cpu().numpy().astype(np.float64)


def alloc_out(M: int, N: int, out_dtype: str, fill: float = float("nan")):
    import torch
    if out_dtype == "bf16":
        t = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    else:
        t = torch.empty((M, N), dtype=torch.float32, device="cuda")
    t.fill_(fill)
    return t


def run_gemm(gq, cfg, inp, M=None):
    """Pack on the device, run gq_gemm, return (out tensor, packed tensor)."""
    import torch
    M = cfg.M if M is None else M
    prec = prec_of(cfg)
    codes = np_to_dev(inp["codes"])
    packed = gq.pack_weights_t(codes, cfg.K, cfg.N, cfg.G, prec)
    A = np_to_dev(inp["A"])
    S = np_to_dev(inp["scales"])
    Z = np_to_dev(inp["zeros"]) if inp["zeros"] is not None else None
    out = alloc_out(M, cfg.N, cfg.out)
    gq.gemm_t(A, packed, S, Z, out, M, cfg.K, cfg.N, cfg.G, prec)
    torch.cuda.synchronize()
    return out, packed

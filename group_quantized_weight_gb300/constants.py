"""Flags, status codes and the work model of the GEMM (host-side, no device needed)."""
from __future__ import annotations

# prec bit field (include/gq.h)
GQ_W4 = 0x01
GQ_ZP = 0x02
GQ_ACT_F32 = 0x04
GQ_SC_BF16 = 0x08
GQ_SC_F32 = 0x10
GQ_OUT_F32 = 0x20
GQ_STATIC_W = 0x40
GQ_GATE_UP = 0x80
GQ_ACT_I8 = 0x100
GQ_ZP_FLOAT = 0x200

GQ_OK = 0
STATUS_NAMES = {0: "GQ_OK", 1: "GQ_ERR_INVALID_ARG", 2: "GQ_ERR_UNSUPPORTED",
                3: "GQ_ERR_ALIGNMENT", 4: "GQ_ERR_WORKSPACE", 5: "GQ_ERR_CUDA",
                6: "GQ_ERR_TIMEOUT", 7: "GQ_ERR_NO_DEVICE"}

_SIZE = {"bf16": 2, "fp16": 2, "f32": 4}


class GqError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"[{STATUS_NAMES.get(status, status)}] {msg}")
        self.status = status


def prec_flags(w4: bool, zp: bool, act: str, sc: str, out: str, zf: bool = False) -> int:
    p = GQ_ZP_FLOAT if zf else 0
    if w4:
        p |= GQ_W4
    if zp:
        p |= GQ_ZP
    if act == "f32":
        p |= GQ_ACT_F32
    if sc == "bf16":
        p |= GQ_SC_BF16
    elif sc == "f32":
        p |= GQ_SC_F32
    if out == "f32":
        p |= GQ_OUT_F32
    return p


def algorithmic_bytes(M: int, K: int, N: int, G: int, w4: bool, zp: bool, act: str, sc: str,
                      out: str, zf: bool = False) -> int:
    """Bytes the GEMM must move at least once: the codes (0.5 or 1 byte per weight), one
    scale and (optionally) one INT4 or float zero point per group and column, the activations read
    once and the output written once.  This is the memory term of the weight-only GEMM
    roofline of "GPU Kernel 工程（09）：量化与融合 kernel", section 3.2 (weights K·N·b_w plus
    activations M·K and outputs M·N), with the group metadata of section 3.1 added."""
    ng = K // G
    codes = K * N // 2 if w4 else K * N
    scales = ng * N * _SIZE[sc]
    zeros = ng * (N // 8) * 4 if zp else ng * N * _SIZE[sc] if zf else 0
    return codes + scales + zeros + M * K * _SIZE[act] + M * N * _SIZE[out]


def gemm_flops(M: int, K: int, N: int) -> int:
    """2·M·K·N (section 3.2 of the same page): the scale and zero-point work is not counted."""
    return 2 * M * K * N

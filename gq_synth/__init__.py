"""Seeded synthetic inputs for the group-quantized weight-only GEMM.

This module is shared by the tests, the benchmark and the oracle's checks.  It holds
no arithmetic of the method: it draws random numbers, rounds them to the storage
dtypes with library conversions (torch / numpy), and writes integer codes into the
canonical packed layouts that the library accepts as input.

Canonical layouts (row-major, as the library's public header states them):
  * INT4 codes  ``uint32 [K/8][N]``: word (r, n) holds k = 8r..8r+7 of column n,
    element j at bits 4j..4j+3 (the INT4 packing of "quantization-and-fused-kernels",
    section 2.4, and its INT4 GEMV teaching kernel, section 9.4).
  * INT8 codes  ``int8 [K][N]`` in [-127, 127] (the int8 code range of the
    group-wise GEMM blog "04 · 分组量化 GEMM 内核", section 2).
  * scales      ``[K/G][N]`` as fp16 / bf16 bit patterns (uint16) or fp32.
  * zero points ``uint32 [K/G][N/8]``: word (g, c) holds n = 8c..8c+7, element j at
    bits 4j (the "[K/g, N/8] INT4" zero-point matrix of section 3.1 of the first page).
  * activations ``[M][K]`` as bf16 bit patterns (uint16) or fp32.

Input recipe (seed 0 unless stated): one independent numpy PCG64 stream per tensor,
seeded by ``SeedSequence([seed, tensor_id])``; reals are drawn in float64, rounded to
fp32, then to the storage dtype with round-to-nearest-even; integers are drawn
uniformly with ``Generator.integers`` (no modulo bias).
"""
from __future__ import annotations

import dataclasses
import numpy as np
import torch

# tensor ids for the per-tensor random streams
_T_A, _T_Q, _T_S, _T_Z, _T_OUTLIER = 1, 2, 3, 4, 5


@dataclasses.dataclass(frozen=True)
class Config:
    """One synthetic workload.  ``w4`` False means INT8 codes."""
    name: str
    M: int
    K: int
    N: int
    G: int
    w4: bool = True
    zp: bool = False            # per-group packed INT4 zero points (else z = 8 for W4, 0 for W8)
    zf: bool = False            # per-group float zero points [K/G][N] in the scales' format
    act: str = "bf16"           # "bf16" | "f32"
    sc: str = "fp16"            # "fp16" | "bf16" | "f32"
    out: str = "bf16"           # "bf16" | "f32"
    s_lo: float = 0.005
    s_hi: float = 0.02
    z_lo: int = 4
    z_hi: int = 11
    outlier_frac: float = 0.0   # fraction of each activation row multiplied by outlier_mult
    outlier_mult: float = 50.0
    a_kind: str = "normal"      # "normal" | "int" (integers in [-8, 8]) | "wide" (see a_spread)
    a_spread: int = 0           # "wide": N(0,1) times 2^U{-a_spread..a_spread} per element
    pow2_scales: bool = False   # scales drawn from {2^-8 .. 2^-5} (exact-arithmetic cases)

    def replace(self, **kw) -> "Config":
        return dataclasses.replace(self, **kw)

    @property
    def ng(self) -> int:
        return self.K // self.G


# The workloads: gate+up shapes of an 8B-class decoder (d = 4096, d_ff = 14336, fused
# N = 2 * d_ff), the 2B-class Q8_0 shapes (N = 2 * 6144), and a 4096-token prefill.
CONFIGS = {
    "tiny_gemv": Config("tiny_gemv", M=1, K=512, N=512, G=128),
    "decode_gateup": Config("decode_gateup", M=1, K=4096, N=28672, G=128,
                            outlier_frac=0.001, outlier_mult=50.0),
    "q8_m1": Config("q8_m1", M=1, K=2048, N=12288, G=32, w4=False, act="f32", sc="f32",
                    out="f32", s_lo=1e-3, s_hi=1e-2),
    "q8_m32": Config("q8_m32", M=32, K=2048, N=12288, G=32, w4=False, act="f32", sc="f32",
                     out="f32", s_lo=1e-3, s_hi=1e-2),
    "asym_m16": Config("asym_m16", M=16, K=8192, N=28672, G=128, zp=True, sc="bf16"),
    "prefill": Config("prefill", M=4096, K=4096, N=14336, G=128),
}


def _rng(seed: int, tensor_id: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, tensor_id])))


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 (RNE) bit patterns as uint16, by torch's conversion."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def f32_to_fp16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> fp16 (RNE) bit patterns as uint16, by numpy's conversion."""
    return np.ascontiguousarray(x, dtype=np.float32).astype(np.float16).view(np.uint16)


def pack_int4_along_k(q: np.ndarray) -> np.ndarray:
    """codes uint8 [K][N] in [0,15] -> uint32 [K/8][N], k = 8r + j at bits 4j."""
    K, N = q.shape
    assert K % 8 == 0
    q3 = q.reshape(K // 8, 8, N).astype(np.uint32)
    w = np.zeros((K // 8, N), dtype=np.uint32)
    for j in range(8):
        w |= q3[:, j, :] << np.uint32(4 * j)
    return w


def pack_int4_along_n(z: np.ndarray) -> np.ndarray:
    """codes uint8 [R][N] in [0,15] -> uint32 [R][N/8], n = 8c + j at bits 4j."""
    R, N = z.shape
    assert N % 8 == 0
    z3 = z.reshape(R, N // 8, 8).astype(np.uint32)
    w = np.zeros((R, N // 8), dtype=np.uint32)
    for j in range(8):
        w |= z3[:, :, j] << np.uint32(4 * j)
    return w


def make_activations(cfg: Config, seed: int = 0, M: int | None = None) -> np.ndarray:
    """Activations [M][K]: bf16 bits (uint16) or float32."""
    M = cfg.M if M is None else M
    rng = _rng(seed, _T_A)
    if cfg.a_kind == "int":
        a = rng.integers(-8, 9, size=(M, cfg.K)).astype(np.float32)
    elif cfg.a_kind == "wide":
        e = rng.integers(-cfg.a_spread, cfg.a_spread + 1, size=(M, cfg.K))
        a = np.ldexp(rng.standard_normal((M, cfg.K)), e).astype(np.float32)
    else:
        a = rng.standard_normal((M, cfg.K)).astype(np.float32)
    if cfg.outlier_frac > 0:
        orng = _rng(seed, _T_OUTLIER)
        n_out = int(round(cfg.outlier_frac * cfg.K))
        for m in range(M):
            ks = orng.choice(cfg.K, size=n_out, replace=False)
            a[m, ks] *= np.float32(cfg.outlier_mult)
    if cfg.act == "bf16":
        return f32_to_bf16_bits(a)
    return a


def make_weights(cfg: Config, seed: int = 0) -> dict:
    """Codes, scales and zero points in the canonical layouts.

    Returns a dict with the packed inputs (``codes``, ``scales``, ``zeros``) and the
    raw integer codes they were packed from (``q`` uint8/int8 [K][N], ``z`` uint8
    [K/G][N] or None) for the layout checks.
    """
    K, N, G = cfg.K, cfg.N, cfg.G
    assert K % G == 0
    ng = K // G
    rq, rs, rz = _rng(seed, _T_Q), _rng(seed, _T_S), _rng(seed, _T_Z)
    if cfg.w4:
        q = rq.integers(0, 16, size=(K, N), dtype=np.uint8)
        codes = pack_int4_along_k(q)
    else:
        q = rq.integers(-127, 128, size=(K, N), dtype=np.int8)
        codes = q
    if cfg.pow2_scales:
        s = np.ldexp(1.0, rs.integers(-8, -4, size=(ng, N))).astype(np.float32)
    else:
        s = rs.uniform(cfg.s_lo, cfg.s_hi, size=(ng, N)).astype(np.float32)
    if cfg.sc == "fp16":
        scales = f32_to_fp16_bits(s)
    elif cfg.sc == "bf16":
        scales = f32_to_bf16_bits(s)
    else:
        scales = s
    z = zeros = None
    if cfg.zf:
        # float zero points near s·z for z in [z_lo, z_hi] (a real z; an integer one with
        # power-of-two scales, so that s·z is exact in every format)
        assert cfg.w4 and not cfg.zp, "float zero points replace the packed INT4 ones"
        if cfg.pow2_scales:
            zr = rz.integers(cfg.z_lo, cfg.z_hi + 1, size=(ng, N)).astype(np.float64)
        else:
            zr = rz.uniform(cfg.z_lo, cfg.z_hi, size=(ng, N))
        zf = (s.astype(np.float64) * zr).astype(np.float32)
        if cfg.sc == "fp16":
            zeros = f32_to_fp16_bits(zf)
        elif cfg.sc == "bf16":
            zeros = f32_to_bf16_bits(zf)
        else:
            zeros = zf
    if cfg.zp:
        assert cfg.w4, "zero points are INT4-packed"
        z = rz.integers(cfg.z_lo, cfg.z_hi + 1, size=(ng, N), dtype=np.uint8)
        zeros = pack_int4_along_n(z)
    return dict(codes=codes, scales=scales, zeros=zeros, q=q, z=z)


def make_inputs(cfg: Config, seed: int = 0, M: int | None = None) -> dict:
    d = make_weights(cfg, seed)
    d["A"] = make_activations(cfg, seed, M)
    return d


def real_weights(N: int, K: int, seed: int = 0, outlier_frac: float = 0.01) -> np.ndarray:
    """Real-valued weights [N][K] fp32 (normal, a few x100 outliers) for quantizer checks."""
    rng = _rng(seed, 17)
    w = rng.standard_normal((N, K)).astype(np.float32)
    n_out = max(1, int(outlier_frac * w.size))
    idx = rng.choice(w.size, size=n_out, replace=False)
    w.reshape(-1)[idx] *= np.float32(100.0)
    return w

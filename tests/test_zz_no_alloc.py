"""gq_gemm_static_scratch: the entry point for callers that cannot allocate device memory
(serving runtimes that reserve all memory up front, latency-critical loops, embedders with
their own allocator).  It must give the same result as gq_gemm, call after call, while its
scratch comes from a fixed array inside the library; both are checked against the float64
oracle.

This file is collected last on purpose, so that a run stopping at the first failure has
already run every other test.
"""
import numpy as np
import pytest

import gq_synth
import oracle
from helpers import alloc_out, load, np_to_dev, out_to_f64, prec_of

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def gq():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return load()


@pytest.mark.parametrize("cfg", [
    gq_synth.Config("nsa_stripe_m1", M=1, K=4096, N=2048, G=128),   # striped decode, CTAs share tiles
    gq_synth.Config("nsa_asym_m3", M=3, K=2048, N=1032, G=128, zp=True, sc="bf16"),
    gq_synth.Config("nsa_q8_m16", M=16, K=2048, N=1024, G=32, w4=False, act="f32", sc="f32",
                    out="f32", s_lo=1e-3, s_hi=1e-2),        # INT8 CUDA-core kernel, K split
    gq_synth.Config("nsa_zf_m12", M=12, K=4096, N=520, G=64, zf=True, sc="bf16"),  # float zeros, K split
    gq_synth.Config("nsa_q8g_m2", M=2, K=2048, N=1024, G=32, w4=False, act="f32", sc="f32",
                    out="f32", s_lo=1e-3, s_hi=1e-2),        # INT8 decode kernel, CTAs share blocks
], ids=lambda c: c.name)
def test_static_scratch_matches_gq_gemm_twice(gq, cfg):
    inp = gq_synth.make_inputs(cfg, seed=4)
    prec = prec_of(cfg)
    packed = gq.pack_weights_t(np_to_dev(inp["codes"]), cfg.K, cfg.N, cfg.G, prec)
    A, S = np_to_dev(inp["A"]), np_to_dev(inp["scales"])
    Z = np_to_dev(inp["zeros"]) if inp["zeros"] is not None else None
    need = gq.gq_workspace_size(cfg.M, cfg.K, cfg.N, cfg.G, prec)
    assert 0 < need <= gq.GQ_STATIC_SCRATCH_BYTES
    ref = alloc_out(cfg.M, cfg.N, cfg.out)
    gq.gemm_t(A, packed, S, Z, ref, cfg.M, cfg.K, cfg.N, cfg.G, prec)
    stream = torch.cuda.current_stream().cuda_stream
    want, mag = oracle.reference(inp["A"], inp["codes"], inp["scales"], inp["zeros"], K=cfg.K,
                                 N=cfg.N, G=cfg.G, w4=cfg.w4, act=cfg.act, sc=cfg.sc,
                                 zp_float=cfg.zf)
    bad, ratio = oracle.check(out_to_f64(ref, cfg.out), want, mag, cfg.out)
    assert bad == 0, f"gq_gemm: {bad} elements out of tolerance against the oracle ({ratio:.3g})"
    for _ in range(2):
        got = alloc_out(cfg.M, cfg.N, cfg.out)
        st = gq.gq_gemm_static_scratch(cfg.M, cfg.K, cfg.N, cfg.G, prec, A.data_ptr(),
                                       packed.data_ptr(), S.data_ptr(),
                                       Z.data_ptr() if Z is not None else None,
                                       got.data_ptr(), stream)
        assert st == 0, gq.gq_status_string(st)
        torch.cuda.synchronize()
        # against the oracle first (a fault shared by both entry points must not pass), then
        # bit for bit against gq_gemm (the same kernels, so the same bits)
        bad, ratio = oracle.check(out_to_f64(got, cfg.out), want, mag, cfg.out)
        assert bad == 0, f"{bad} elements out of tolerance against the oracle ({ratio:.3g})"
        view = torch.int16 if cfg.out == "bf16" else torch.int32
        assert torch.equal(got.view(view), ref.view(view))


def test_static_scratch_rejects_problems_larger_than_the_array(gq):
    cfg = gq_synth.CONFIGS["asym_m16"]
    prec = prec_of(cfg)
    need = gq.gq_workspace_size(cfg.M, cfg.K, cfg.N, cfg.G, prec)
    assert need > gq.GQ_STATIC_SCRATCH_BYTES
    d = torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")
    p = d.data_ptr()
    st = gq.gq_gemm_static_scratch(cfg.M, cfg.K, cfg.N, cfg.G, prec, p, p, p, p, p, None)
    assert st == 4                                             # GQ_ERR_WORKSPACE

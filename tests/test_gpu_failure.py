"""Failure detection on the GPU without a GPU fault: every device-side wait is bounded, and a
wait that runs out is reported through gq_device_error while the context stays usable; host
failures (scratch allocation, kernel launch) are injected and must surface as GQ_ERR_CUDA
with nothing launched.  Nothing here traps, faults or hangs a GPU."""
import numpy as np
import pytest

import gq_synth
import oracle
from helpers import alloc_out, load, np_to_dev, out_to_f64, prec_of

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

GQ_FAULT_NONE, GQ_FAULT_WORKSPACE, GQ_FAULT_LAUNCH, GQ_FAULT_DEVICE_WAIT = 0, 1, 2, 3


@pytest.fixture(scope="module")
def gq():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return load()


def _setup(gq, cfg, seed=3):
    inp = gq_synth.make_inputs(cfg, seed=seed)
    prec = prec_of(cfg)
    packed = gq.pack_weights_t(np_to_dev(inp["codes"]), cfg.K, cfg.N, cfg.G, prec)
    A, S = np_to_dev(inp["A"]), np_to_dev(inp["scales"])
    Z = np_to_dev(inp["zeros"]) if inp["zeros"] is not None else None
    ref, mag = oracle.reference(inp["A"], inp["codes"], inp["scales"], inp["zeros"], K=cfg.K,
                                N=cfg.N, G=cfg.G, w4=cfg.w4, act=cfg.act, sc=cfg.sc)
    return prec, (A, packed, S, Z), ref, mag


def _call(gq, cfg, prec, bufs, out):
    A, packed, S, Z = bufs
    return gq.gq_gemm(cfg.M, cfg.K, cfg.N, cfg.G, prec, A.data_ptr(), packed.data_ptr(),
                      S.data_ptr(), Z.data_ptr() if Z is not None else None, out.data_ptr(),
                      torch.cuda.current_stream().cuda_stream)


def test_a_bounded_device_wait_that_runs_out_is_reported_and_the_context_stays_usable(gq):
    # fewer 16-column tiles than SMs: the warp-specialized decode kernel, whose producer can be
    # told to withhold a slot (a barrier nothing completes)
    cfg = gq_synth.Config("wait_m1", M=1, K=4096, N=2048, G=128)
    prec, bufs, ref, mag = _setup(gq, cfg)
    assert gq.gq_plan(cfg.M, cfg.K, cfg.N, cfg.G, prec)["path"] == 8
    torch.cuda.synchronize()
    gq.gq_device_error(True)
    assert gq.gq_set_wait_limit(2_000_000) == 0            # about a millisecond
    try:
        assert gq.gq_set_fault_injection(GQ_FAULT_DEVICE_WAIT) == GQ_FAULT_NONE
        out = alloc_out(cfg.M, cfg.N, cfg.out)
        assert _call(gq, cfg, prec, bufs, out) == 0
        torch.cuda.synchronize()
        assert gq.gq_device_error(True) == 6               # GQ_ERR_TIMEOUT
    finally:
        gq.gq_set_fault_injection(GQ_FAULT_NONE)
        gq.gq_set_wait_limit(0)
    # the next plain call on the same context is correct and raises nothing
    out = alloc_out(cfg.M, cfg.N, cfg.out)
    assert _call(gq, cfg, prec, bufs, out) == 0
    torch.cuda.synchronize()
    bad, ratio = oracle.check(out_to_f64(out, cfg.out), ref, mag, cfg.out)
    assert bad == 0, f"{bad} elements out of tolerance after the timeout ({ratio:.3g})"
    assert gq.gq_device_error(False) == 0


@pytest.mark.parametrize("fault,detail", [(GQ_FAULT_WORKSPACE, "workspace allocation (injected)"),
                                          (GQ_FAULT_LAUNCH, "launch (injected)")])
def test_injected_host_failures_return_cuda_error_and_launch_nothing(gq, fault, detail):
    # a split-K shape, so the call needs the library-owned scratch
    cfg = gq_synth.Config("inj_m16", M=16, K=8192, N=1024, G=128, zp=True, sc="bf16")
    prec, bufs, ref, mag = _setup(gq, cfg)
    assert gq.gq_workspace_size(cfg.M, cfg.K, cfg.N, cfg.G, prec) > 0
    assert gq.gq_set_workspace(None, 0) == 0              # the library-owned scratch
    out = alloc_out(cfg.M, cfg.N, cfg.out)                 # NaN-filled
    torch.cuda.synchronize()
    try:
        gq.gq_set_fault_injection(fault)
        assert _call(gq, cfg, prec, bufs, out) == 5        # GQ_ERR_CUDA
        assert gq.gq_last_error_detail().startswith(detail)
        if fault == GQ_FAULT_LAUNCH:
            st = gq.gq_gemm_static_scratch(cfg.M, cfg.K, cfg.N, cfg.G, prec,
                                           bufs[0].data_ptr(), bufs[1].data_ptr(),
                                           bufs[2].data_ptr(), bufs[3].data_ptr(),
                                           out.data_ptr(), None)
            assert st == 5
    finally:
        gq.gq_set_fault_injection(GQ_FAULT_NONE)
    torch.cuda.synchronize()
    assert torch.isnan(out.float()).all()                  # nothing was written
    assert _call(gq, cfg, prec, bufs, out) == 0
    torch.cuda.synchronize()
    bad, _ = oracle.check(out_to_f64(out, cfg.out), ref, mag, cfg.out)
    assert bad == 0

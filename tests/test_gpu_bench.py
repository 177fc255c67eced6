"""gq_bench(config, json_out, cap): the library's self-contained benchmark of a named
workload, called through the C ABI on the GPU."""
import pytest

from helpers import load, prec_of
import gq_synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def gq():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return load()


def test_config_benchmark_reports_the_tiny_gemv(gq):
    r = gq.gq_bench("tiny_gemv")
    cfg = gq_synth.CONFIGS["tiny_gemv"]
    assert r["config"] == "tiny_gemv" and (r["M"], r["K"], r["N"], r["G"]) == (1, 512, 512, 128)
    assert r["path"] == gq.gq_plan(cfg.M, cfg.K, cfg.N, cfg.G, prec_of(cfg))["path"]
    assert 0 < r["us_p10"] <= r["us_median"] <= r["us_p90"]
    assert r["us_single_call"] > 0 and r["repeats"] == 5 and r["graph"] is True
    # 512·512/2 codes + 4·512 fp16 scales + 512 bf16 activations + 512 bf16 outputs
    assert r["algorithmic_bytes"] == 131072 + 4096 + 1024 + 1024
    assert r["GB/s"] == pytest.approx(r["algorithmic_bytes"] / r["us_median"] / 1e3, rel=1e-3)
    assert r["bound"] == "hbm" and r["peak"] > 1000 and 0 < r["frac"] < 2
    assert r["launches_per_call"] == 1 and r["deterministic"] is True
    assert r["weight_copies"] == 16          # a 0.14 MB problem: the cap of the rotation


def test_config_benchmark_rejects_a_buffer_too_small(gq):
    import ctypes
    buf = ctypes.create_string_buffer(16)
    assert gq._lib.gq_bench(b"tiny_gemv", buf, 16) == 1
    assert buf.value == b""

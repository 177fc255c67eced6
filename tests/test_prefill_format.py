"""Why the prefill kernel's tensor-core operand holds the exact integer (q − z) and applies
the scale per group in FP32, rather than holding bf16-rounded dequantized weights s·(q − z).

The pages only say the prefill path dequantizes into BF16 tiles; where the scale goes is
open. On a 256 x 2048 output slice of the M=4096 K=4096 N=14336 G=128 prefill workload
(its own distributions), an FP32-accumulation model of each choice is compared with the
float64 oracle under the bf16-output tolerance: rounding s·(q − 8) to bf16 puts hundreds of
elements out of tolerance, while exact integer tiles with an FP32 per-group scale put none.
Both models use library arithmetic only (torch's bf16 rounding, numpy float32 matmuls).
"""
import numpy as np
import pytest

import gq_synth
import oracle

torch = pytest.importorskip("torch")


def _to_bf16(x):
    return torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(torch.bfloat16).float().numpy()


def test_integer_tiles_with_fp32_group_scales_meet_the_tolerance_and_bf16_weights_do_not():
    cfg = gq_synth.CONFIGS["prefill"].replace(name="prefill_slice", M=256, N=2048)
    inp = gq_synth.make_inputs(cfg, seed=0)
    ref, mag = oracle.reference(inp["A"], inp["codes"], inp["scales"], None, K=cfg.K, N=cfg.N,
                                G=cfg.G, w4=True, act="bf16", sc="fp16")
    A = torch.from_numpy(inp["A"].view(np.int16)).view(torch.bfloat16).float().numpy()
    s = inp["scales"].view(np.float16).astype(np.float32)
    qz = inp["q"].astype(np.float32) - 8.0                 # symmetric zero point
    G, ng = cfg.G, cfg.K // cfg.G

    # bf16-rounded dequantized weights, one FP32-accumulated product, bf16 output
    W = _to_bf16(qz.reshape(ng, G, -1) * s[:, None, :]).reshape(cfg.K, -1)
    bad_w, _ = oracle.check(_to_bf16(A @ W).astype(np.float64), ref, mag, "bf16")

    # exact integer tiles: each group's FP32 dot, then its FP32 scale, bf16 output
    acc = np.zeros((cfg.M, cfg.N), np.float32)
    for g in range(ng):
        acc = acc + s[g][None, :] * (A[:, g * G:(g + 1) * G] @ qz[g * G:(g + 1) * G])
    bad_i, worst_i = oracle.check(_to_bf16(acc).astype(np.float64), ref, mag, "bf16")

    assert bad_i == 0 and worst_i < 1.0
    assert bad_w > 100                                     # about 0.17% of the slice

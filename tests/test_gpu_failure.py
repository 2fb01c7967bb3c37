"""Failure detection on the GPU without a fault: a kernel whose bounded
pipeline wait can never complete must give up, report USP_ERR_TIMEOUT through
usp_device_status, and leave the device usable for the next call."""
import time

import numpy as np
import pytest
import torch

import sequence_long_context_gb300 as usp
from oracle import attention
from sequence_long_context_gb300.workloads import WORKLOADS, make_inputs
from tests._gpu import TOL, device

pytestmark = pytest.mark.gpu


def test_wait_times_out_and_device_stays_usable():
    dev = device()
    usp.usp_device_status()  # nothing pending from earlier tests
    t0 = time.perf_counter()
    usp.usp_selftest_wait_timeout(20000)  # 20 ms
    with pytest.raises(usp.UspError, match="USP_ERR_TIMEOUT"):
        usp.usp_device_status()
    assert time.perf_counter() - t0 >= 0.02
    usp.usp_device_status()  # reported once, then cleared
    # the context still computes correctly
    w = WORKLOADS["tiny_zigzag_cp4"].replace(dtype="bf16", D=128, S=512)
    x = make_inputs(w, seed=3, with_grad=False)
    qp, kp, vp = (usp.permute(x[n].to(dev), "extract", w.layout, w.cp) for n in "qkv")
    out, _ = usp.attn_forward(qp, kp, vp, causal=True, cp=w.cp, layout=w.layout)
    o_nat = usp.permute(out, "restore", w.layout, w.cp).float().cpu().numpy()
    O, _ = attention.attn_fwd(x["q"], x["k"], x["v"], w.scale, True)
    assert np.abs(o_nat - O).max() <= TOL["bf16"]["o"]
    usp.usp_device_status()

"""usp_attn_bwd_noalloc: the backward entry point for callers that cannot
allocate a workspace (its scratch is the library's fixed 64 MiB device
array). It must give what usp_attn_bwd gives, call after call, and refuse
problems whose scratch would not fit.

This file is collected last on purpose, so a run that stops at the first
failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import sequence_long_context_gb300 as usp
from sequence_long_context_gb300 import _lib
from sequence_long_context_gb300.workloads import WORKLOADS, make_inputs
from tests._gpu import TOL, device, rel_fro, to_np

pytestmark = pytest.mark.gpu


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


@pytest.mark.parametrize("dtype,layout,cp", [("bf16", "zigzag", 4), ("fp32", "stripe", 2)])
def test_noalloc_matches_workspace_backward_twice(dtype, layout, cp):
    dev = device()
    w = WORKLOADS["tiny_zigzag_cp4"].replace(B=2, S=1024, Hq=4, Hkv=2, D=128, dtype=dtype,
                                             layout=layout, cp=cp)
    x = make_inputs(w, seed=21)
    qp, kp, vp, dop = (usp.permute(x[n].to(dev), "extract", w.layout, w.cp)
                       for n in ("q", "k", "v", "dout"))
    kw = dict(causal=True, cp=w.cp, layout=w.layout)
    out, lse = usp.attn_forward(qp, kp, vp, **kw)
    ref = usp.attn_backward(qp, kp, vp, out, lse, dop, **kw)
    lib = _lib.load()
    for call in range(2):
        dq, dk, dv = torch.empty_like(qp), torch.empty_like(kp), torch.empty_like(vp)
        for g in (dq, dk, dv):
            g.fill_(float("nan"))
        st = lib.usp_attn_bwd_noalloc(
            _ptr(qp), _ptr(kp), _ptr(vp), _ptr(out), _ptr(lse), _ptr(dop), _ptr(dq),
            _ptr(dk), _ptr(dv), w.B, w.S, w.Hq, w.Hkv, w.D, 0.0, 1, 0, 0, None, w.cp, 1,
            usp.LAYOUT[w.layout], usp.DTYPE[qp.dtype], 0,
            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
        assert st == 0, lib.usp_status_string(st)
        torch.cuda.synchronize()
        for got, want in zip((dq, dk, dv), ref):
            e = rel_fro(to_np(got), to_np(want))
            assert np.isfinite(to_np(got)).all()
            assert e <= TOL[dtype]["grad"], (call, e)


def test_noalloc_rejects_problem_beyond_the_scratch_limit():
    device()
    lib = _lib.load()
    fake = ctypes.c_void_p(1 << 20)  # never dereferenced: rejected before launch
    # B=1, S=65536, 32 heads, D=128: the dQ accumulator alone is 1 GiB
    st = lib.usp_attn_bwd_noalloc(fake, fake, fake, fake, fake, fake, fake, fake, fake,
                                  1, 65536, 32, 8, 128, 0.0, 1, 0, 0, None, 8, 1, 1, 0, 0,
                                  None)
    assert lib.usp_status_string(st).decode() == "USP_ERR_WORKSPACE"
    assert b"64 MiB" in lib.usp_last_error_detail()

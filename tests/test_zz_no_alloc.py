"""usp_attn_bwd_noalloc: the backward entry point for callers that cannot
allocate a workspace (a runtime whose device memory already belongs to its
own pools, or a path where cudaMalloc is not allowed). Its scratch is the
library's fixed 64 MiB device array. It must give what usp_attn_bwd gives,
call after call (the array keeps the previous call's contents), match the
oracle, and refuse problems whose scratch would not fit.

This file is collected last on purpose, so a run that stops at the first
failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import sequence_long_context_gb300 as usp
from oracle import attention
from sequence_long_context_gb300 import _lib
from sequence_long_context_gb300.workloads import WORKLOADS, make_inputs
from tests._gpu import TOL, device, rel_fro, to_np

pytestmark = pytest.mark.gpu


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


# (dtype, layout, cp, ulysses degree, packed): the tensor-core path, the fp32
# path, the Ulysses exchange buffers carved from the array, and a packed batch
CASES = [("bf16", "zigzag", 4, 1, False), ("fp32", "stripe", 2, 1, False),
         ("bf16", "zigzag", 2, 2, False), ("bf16", "zigzag", 2, 1, True)]


@pytest.mark.parametrize("dtype,layout,cp,ud,packed", CASES)
def test_noalloc_matches_workspace_backward_twice(dtype, layout, cp, ud, packed):
    dev = device()
    w = WORKLOADS["tiny_zigzag_cp4"].replace(B=2, S=1024, Hq=4, Hkv=2, D=128, dtype=dtype,
                                             layout=layout, cp=cp, ud=ud)
    x = make_inputs(w, seed=21)
    cu = None
    if packed:  # two sequences of 400 and 624 tokens in one packed batch
        x = {n: t[0] for n, t in x.items()}
        cu = torch.tensor([0, 400, 1024], dtype=torch.int32)
    cu_dev = cu.to(dev) if cu is not None else None
    nseq = 2 if packed else w.B
    qp, kp, vp, dop = (usp.permute(x[n].to(dev), "extract", w.layout, w.cp)
                       for n in ("q", "k", "v", "dout"))
    kw = dict(causal=True, cp=w.cp, ud=w.ud, layout=w.layout, cu_seqlens=cu_dev)
    out, lse = usp.attn_forward(qp, kp, vp, **kw)
    ref = usp.attn_backward(qp, kp, vp, out, lse, dop, **kw)
    lib = _lib.load()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call in range(2):
        dq, dk, dv = torch.empty_like(qp), torch.empty_like(kp), torch.empty_like(vp)
        for g in (dq, dk, dv):
            g.fill_(float("nan"))
        st = lib.usp_attn_bwd_noalloc(
            _ptr(qp), _ptr(kp), _ptr(vp), _ptr(out), _ptr(lse), _ptr(dop), _ptr(dq),
            _ptr(dk), _ptr(dv), nseq, w.S, w.Hq, w.Hkv, w.D, 0.0, 1, 0, 0, _ptr(cu_dev),
            w.cp, w.ud, usp.LAYOUT[w.layout], usp.DTYPE[qp.dtype], 0, stream)
        assert st == 0, lib.usp_status_string(st)
        torch.cuda.synchronize()
        for got, want in zip((dq, dk, dv), ref):
            e = rel_fro(to_np(got), to_np(want))
            assert np.isfinite(to_np(got)).all()
            assert e <= TOL[dtype]["grad"], (call, e)
    # the second call's gradients against the oracle, in natural order
    want = attention.attn_bwd(x["q"], x["k"], x["v"], x["dout"], w.scale, True,
                              cu_seqlens=cu.numpy() if cu is not None else None)
    for got, ref_g in zip((dq, dk, dv), want):
        g = usp.permute(got, "restore", w.layout, w.cp)
        assert rel_fro(to_np(g), ref_g) <= TOL[dtype]["grad"]


def test_noalloc_setup_call_launches_nothing():
    device()
    lib = _lib.load()
    n0 = lib.usp_launch_count()
    # valid sizes with S = 0 (tensors may then be NULL): only the per-device
    # set-up runs
    st = lib.usp_attn_bwd_noalloc(None, None, None, None, None, None, None, None, None,
                                  1, 0, 4, 2, 128, 0.0, 1, 0, 0, None, 2, 1, 1, 0, 0, None)
    assert st == 0, lib.usp_status_string(st)
    assert lib.usp_launch_count() == n0


def test_noalloc_rejects_problem_beyond_the_scratch_limit():
    device()
    lib = _lib.load()
    fake = ctypes.c_void_p(1 << 20)  # never dereferenced: rejected before launch
    # B=1, S=65536, 32 heads, D=128: the dQ accumulator alone is 1 GiB
    n0 = lib.usp_launch_count()
    st = lib.usp_attn_bwd_noalloc(fake, fake, fake, fake, fake, fake, fake, fake, fake,
                                  1, 65536, 32, 8, 128, 0.0, 1, 0, 0, None, 8, 1, 1, 0, 0,
                                  None)
    assert lib.usp_status_string(st).decode() == "USP_ERR_WORKSPACE"
    assert b"64 MiB" in lib.usp_last_error_detail()
    assert lib.usp_launch_count() == n0

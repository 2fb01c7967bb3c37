"""GPU parity of ring attention (forward + backward) against the oracle on
small seeded problems: every layout, ring degree and Ulysses degree, causal
and non-causal, sliding window with and without sinks, GQA, packed varlen,
fp32 and bf16, through both kernel families."""
import numpy as np
import pytest
import torch

import sequence_long_context_gb300 as usp
from oracle import attention
from sequence_long_context_gb300.workloads import WORKLOADS, make_inputs
from tests._gpu import (TOL, device, lse_to_natural, rel_fro, run_backward,
                        run_forward, to_np)

pytestmark = pytest.mark.gpu

BASE = WORKLOADS["tiny_zigzag_cp4"]


def check(w, flags=0, seed=0, backward=True):
    dev = device()
    x = make_inputs(w, seed=seed, with_grad=backward)
    cu = x.get("cu_seqlens")
    fwd = run_forward(usp, w, x, dev, flags)
    O, L = attention.attn_fwd(x["q"], x["k"], x["v"], w.scale, w.causal,
                              w.window, w.sink_tokens, cu_seqlens=cu)
    tol = TOL[w.dtype]
    o = to_np(fwd[0])
    lse = lse_to_natural(to_np(fwd[1]), w)
    assert np.isfinite(o).all()
    err_o = np.abs(o - O).max()
    err_l = np.abs(lse - L).max()
    assert err_o <= tol["o"], err_o
    assert err_l <= tol["lse"], err_l
    if not backward:
        return
    grads = run_backward(usp, w, x, dev, fwd, flags)
    ref = attention.attn_bwd(x["q"], x["k"], x["v"], x["dout"], w.scale,
                             w.causal, w.window, w.sink_tokens, cu_seqlens=cu)
    for name, g, r in zip("qkv", grads, ref):
        e = rel_fro(to_np(g), r)
        assert e <= tol["grad"], (name, e)


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
def test_tiny_zigzag_config(dtype):
    """The tiny oracle-check workload: S=256, 2 heads, D=64, zigzag cp=4."""
    check(BASE.replace(dtype=dtype))


@pytest.mark.parametrize("layout", ["contiguous", "zigzag", "stripe"])
@pytest.mark.parametrize("cp,ud", [(1, 1), (2, 1), (3, 1), (4, 1), (8, 1), (2, 2), (4, 2), (3, 2)])
def test_layouts_and_degrees(layout, cp, ud):
    w = BASE.replace(B=2, S=384, Hq=4, Hkv=2, D=64, dtype="fp32", layout=layout, cp=cp, ud=ud)
    check(w)


@pytest.mark.parametrize("flags", [0, usp.FLAG_FORCE_SIMT])
@pytest.mark.parametrize("case", [
    dict(layout="zigzag", cp=8, S=2048, Hq=4, Hkv=2),
    dict(layout="stripe", cp=8, S=2048, Hq=8, Hkv=2),
    dict(layout="contiguous", cp=4, S=1024, Hq=4, Hkv=4, window=200),
    dict(layout="contiguous", cp=4, S=1024, Hq=4, Hkv=4, window=200, sink_tokens=4),
    dict(layout="zigzag", cp=2, S=1024, Hq=4, Hkv=1, ud=1, causal=False),
    dict(layout="zigzag", cp=4, S=1024, Hq=4, Hkv=2, ud=2),
    # windows through the one-tile-per-CTA forward, on every layout
    dict(layout="stripe", cp=4, S=1024, Hq=4, Hkv=2, window=300),
    dict(layout="zigzag", cp=2, S=1024, Hq=8, Hkv=2, window=250, sink_tokens=2),
    dict(layout="zigzag", cp=2, S=1024, Hq=4, Hkv=2, ud=2, window=333),
    # 128-token zigzag chunks and stripe shards (one query tile per chunk)
    dict(layout="zigzag", cp=4, S=1024, Hq=4, Hkv=2),
    dict(layout="stripe", cp=4, S=512, Hq=4, Hkv=2),
    dict(layout="contiguous", cp=8, S=1024, Hq=4, Hkv=2, ud=1, window=100),
])
def test_bf16_d128(case, flags):
    w = BASE.replace(B=2, D=128, dtype="bf16", **case)
    check(w, flags=flags)


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
@pytest.mark.parametrize("window,sink", [(0, 0), (300, 0), (300, 3)])
def test_varlen(dtype, window, sink):
    w = BASE.replace(B=0, S=2048, Hq=4, Hkv=2, D=128, dtype=dtype, cp=8, layout="zigzag",
                     varlen=True, seg_lo=1, seg_hi=700, window=window, sink_tokens=sink)
    check(w)


@pytest.mark.parametrize("window,sink", [(0, 0), (400, 2)])
def test_bf16_varlen_tensor_core(window, sink):
    # 256-token zigzag chunks: the tensor-core kernels (the forward with one
    # query tile per CTA) on a packed batch
    w = BASE.replace(B=0, S=4096, Hq=4, Hkv=2, D=128, dtype="bf16", cp=8, layout="zigzag",
                     varlen=True, seg_lo=100, seg_hi=1500, window=window, sink_tokens=sink)
    check(w)


def test_bf16_d64_window():
    w = BASE.replace(B=2, S=1024, Hq=4, Hkv=2, D=64, dtype="bf16", cp=4, layout="contiguous",
                     window=200)
    check(w)


def test_varlen_empty_and_single_token_segments():
    dev = device()
    w = BASE.replace(B=0, S=256, Hq=2, Hkv=1, D=64, dtype="fp32", cp=4, layout="stripe",
                     varlen=True)
    x = make_inputs(w.replace(varlen=False, B=1), seed=3)
    x = {n: t[0] for n, t in x.items()}
    x["cu_seqlens"] = torch.tensor([0, 1, 1, 2, 100, 256], dtype=torch.int32)
    fwd = run_forward(usp, w, x, dev)
    O, L = attention.attn_fwd(x["q"], x["k"], x["v"], w.scale, True,
                              cu_seqlens=x["cu_seqlens"])
    assert np.abs(to_np(fwd[0]) - O).max() <= 1e-5
    grads = run_backward(usp, w, x, dev, fwd)
    ref = attention.attn_bwd(x["q"], x["k"], x["v"], x["dout"], w.scale, True,
                             cu_seqlens=x["cu_seqlens"])
    for g, r in zip(grads, ref):
        assert rel_fro(to_np(g), r) <= 1e-5


def test_custom_scale_and_window_wider_than_sequence():
    w = BASE.replace(S=512, window=4096, dtype="fp32", layout="stripe")
    dev = device()
    x = make_inputs(w, seed=4)
    qp, kp, vp = (usp.permute(x[n].to(dev), "extract", w.layout, w.cp) for n in "qkv")
    out, lse = usp.attn_forward(qp, kp, vp, causal=True, window=4096, cp=w.cp,
                                layout=w.layout, softmax_scale=0.05)
    O, _ = attention.attn_fwd(x["q"], x["k"], x["v"], 0.05, True, 0)
    o = to_np(usp.permute(out, "restore", w.layout, w.cp))
    assert np.abs(o - O).max() <= 1e-5


def test_simt_and_tensor_core_paths_agree():
    """The two kernel families compute the same ring schedule."""
    dev = device()
    w = BASE.replace(B=1, S=2048, Hq=4, Hkv=2, D=128, dtype="bf16", cp=8)
    x = make_inputs(w, seed=9)
    a = run_forward(usp, w, x, dev, 0)
    b = run_forward(usp, w, x, dev, usp.FLAG_FORCE_SIMT)
    assert np.abs(to_np(a[0]) - to_np(b[0])).max() <= 2e-2
    assert np.abs(to_np(a[1]) - to_np(b[1])).max() <= 1e-3


# Edge cases of the visibility rule on the tensor-core kernels (bf16, D=128,
# ring chunks of 128 tokens or more).
EDGE = {
    "window1_sinks5": dict(layout="contiguous", cp=4, S=1024, Hq=4, Hkv=2, window=1,
                           sink_tokens=5),
    "sinks_past_window": dict(layout="stripe", cp=4, S=1024, Hq=4, Hkv=2, window=64,
                              sink_tokens=200),
    "window_wider_than_sequence": dict(layout="zigzag", cp=4, S=1024, Hq=4, Hkv=2,
                                       window=5000),
    "window_equal_to_sequence": dict(layout="zigzag", cp=2, S=1024, Hq=4, Hkv=2, window=1024),
    "multi_query_ring8": dict(layout="zigzag", cp=8, S=2048, Hq=8, Hkv=1),
    "one_head_per_ulysses_rank": dict(layout="zigzag", cp=2, S=1024, Hq=4, Hkv=4, ud=4),
    "non_causal_window": dict(layout="contiguous", cp=4, S=1024, Hq=4, Hkv=2, window=200,
                              causal=False),
}


@pytest.mark.parametrize("name", sorted(EDGE))
def test_bf16_visibility_edge_cases(name):
    check(BASE.replace(B=2, D=128, dtype="bf16", **EDGE[name]))


def test_window_of_one_returns_own_value():
    """A window of one key (the query's own): the softmax over a single score
    is 1, so O_i = v_i and dV = dO bit for bit, LSE_i = scale * q_i . k_i,
    and dQ, dK vanish up to the rounding of dP - Delta (two fp32 sums of the
    same 128 products, in different orders)."""
    dev = device()
    w = BASE.replace(B=2, S=1024, Hq=4, Hkv=4, D=128, dtype="bf16", cp=4, layout="zigzag",
                     window=1)
    x = make_inputs(w, seed=11, with_grad=True)
    fwd = run_forward(usp, w, x, dev)
    assert torch.equal(fwd[0].cpu(), x["v"])
    q, k = to_np(x["q"]), to_np(x["k"])
    lse = lse_to_natural(to_np(fwd[1]), w)
    assert np.abs(lse - w.scale * np.einsum("bshd,bshd->bhs", q, k)).max() <= 1e-3
    dq, dk, dv = run_backward(usp, w, x, dev, fwd)
    assert torch.equal(dv.cpu(), x["dout"])
    assert float(dq.abs().max()) <= 2e-3 and float(dk.abs().max()) <= 2e-3

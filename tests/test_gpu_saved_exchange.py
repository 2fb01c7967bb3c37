"""GPU parity of the backward that reuses the forward's Ulysses exchange
(FLAG_SAVED_EXCHANGE): the method's backward keeps the head-sharded q, k, v,
output and LSE of the forward ("Long Context Attention" notes,
"Motivation"), so only dout is exchanged on the way in.

The saved-exchange call is handed zeroed q, k, v, out: it must take them from
the workspace, and give the ordinary backward's dK, dV bit for bit (dQ is
reduced in hardware order, so it is checked against the oracle)."""
import numpy as np
import pytest
import torch

import sequence_long_context_gb300 as usp
from oracle import attention
from sequence_long_context_gb300.workloads import WORKLOADS, make_inputs
from tests._gpu import TOL, device, rel_fro

pytestmark = pytest.mark.gpu

CASES = [
    dict(dtype="bf16", D=128, S=1024, Hq=4, Hkv=4, cp=2, ud=2, layout="zigzag"),
    dict(dtype="bf16", D=128, S=2048, Hq=8, Hkv=2, cp=2, ud=2, layout="stripe"),
    dict(dtype="bf16", D=64, S=1024, Hq=4, Hkv=4, cp=1, ud=4, layout="contiguous", window=200,
         sink_tokens=3),
    dict(dtype="fp32", D=64, S=512, Hq=4, Hkv=2, cp=2, ud=2, layout="zigzag"),
    dict(dtype="bf16", D=128, S=1024, Hq=4, Hkv=4, cp=2, ud=2, layout="zigzag", varlen=True,
         seg_lo=100, seg_hi=600),
    dict(dtype="bf16", D=128, S=512, Hq=4, Hkv=4, cp=4, ud=1, layout="zigzag"),  # flag is a no-op
]


def _oracle_check(w, x, cu, grads, unperm):
    ref = attention.attn_bwd(x["q"], x["k"], x["v"], x["dout"], w.scale, w.causal, w.window,
                             w.sink_tokens, cu_seqlens=cu)
    for i, (g, r) in enumerate(zip(grads, ref)):
        e = rel_fro(unperm(g).double().cpu().numpy(), r)
        assert np.isfinite(e) and e <= TOL[w.dtype]["grad"], (i, e)


@pytest.mark.parametrize("case", CASES, ids=lambda c: "-".join(f"{k}{v}" for k, v in c.items()))
def test_saved_exchange_backward(case):
    dev = device()
    w = WORKLOADS["tiny_zigzag_cp4"].replace(**case)
    x = make_inputs(w, seed=23, with_grad=True)
    cu = x.get("cu_seqlens")
    cu_dev = cu.to(dev) if cu is not None else None
    perm = lambda t: usp.permute(t.to(dev), "extract", w.layout, w.cp)  # noqa: E731
    unperm = lambda t: usp.permute(t, "restore", w.layout, w.cp)  # noqa: E731
    kw = dict(causal=w.causal, window=w.window, sink_tokens=w.sink_tokens,
              cu_seqlens=cu_dev, cp=w.cp, ud=w.ud, layout=w.layout)
    qp, kp, vp, dop = perm(x["q"]), perm(x["k"]), perm(x["v"]), perm(x["dout"])
    ws = usp.attn_workspace(qp, kp, cu_seqlens=cu_dev, cp=w.cp, ud=w.ud)
    ws.fill_(0x7F)  # stale contents must not matter to the forward
    out, lse = usp.attn_forward(qp, kp, vp, workspace=ws, **kw)
    out_ref, lse_ref = usp.attn_forward(qp, kp, vp, **kw)
    assert torch.equal(out, out_ref) and torch.equal(lse, lse_ref)
    ref = usp.attn_backward(qp, kp, vp, out, lse, dop, **kw)
    zq, zk, zo = torch.zeros_like(qp), torch.zeros_like(kp), torch.zeros_like(out)
    if w.ud == 1:  # nothing saved: the tensors are read as usual
        zq, zk, zo = qp, kp, out
    for _ in range(2):  # the backward leaves the saved exchange intact
        got = usp.attn_backward(zq, zk, zk if w.ud > 1 else vp, zo, lse, dop, workspace=ws,
                                saved_exchange=True, **kw)
        assert torch.equal(got[1], ref[1]) and torch.equal(got[2], ref[2])
        _oracle_check(w, x, cu, got, unperm)


def test_saved_exchange_packed():
    dev = device()
    w = WORKLOADS["tiny_zigzag_cp4"].replace(dtype="bf16", D=128, S=1024, Hq=4, Hkv=4, cp=2,
                                              ud=2, layout="zigzag")
    x = make_inputs(w, seed=29, with_grad=True)
    perm = lambda t: usp.permute(t.to(dev), "extract", w.layout, w.cp)  # noqa: E731
    unperm = lambda t: usp.permute(t, "restore", w.layout, w.cp)  # noqa: E731
    kw = dict(causal=w.causal, cp=w.cp, ud=w.ud, layout=w.layout)
    qp, kp, vp, dop = perm(x["q"]), perm(x["k"]), perm(x["v"]), perm(x["dout"])
    qkv = torch.stack([qp, kp, vp], dim=-3).contiguous()
    ws = usp.attn_workspace(qp, kp, cp=w.cp, ud=w.ud)
    out, lse = usp.attn_forward_qkvpacked(qkv, workspace=ws, **kw)
    ref = usp.attn_backward_qkvpacked(qkv, out, lse, dop, **kw)
    got = usp.attn_backward_qkvpacked(torch.zeros_like(qkv), torch.zeros_like(out), lse, dop,
                                      workspace=ws, saved_exchange=True, **kw)
    assert torch.equal(got[..., 1, :, :], ref[..., 1, :, :])
    assert torch.equal(got[..., 2, :, :], ref[..., 2, :, :])
    _oracle_check(w, x, None, [got[..., i, :, :].contiguous() for i in range(3)], unperm)

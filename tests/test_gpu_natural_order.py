"""GPU parity of the natural-order calls (FLAG_NATURAL_ORDER): q, k, v, out,
dout, dq, dk, dv in natural sequence order, read and written in place by the
tensor-core kernels (contiguous and zigzag layouts), or with the layout's
extract and restore done inside the call (stripe, the CUDA-core kernels:
fused into the Ulysses exchange when ulysses_degree > 1). The result must
equal extracting the inputs, calling in rank-major order and restoring the
outputs (YunChang README, "2. Usage": the inputs are reordered by the
extract function before the attention):
out, lse, dk, dv bit for bit; dq is reduced in hardware order, so it is
checked against the oracle."""
import numpy as np
import pytest
import torch

import sequence_long_context_gb300 as usp
from oracle import attention
from sequence_long_context_gb300.workloads import WORKLOADS, make_inputs
from tests._gpu import TOL, device, rel_fro

pytestmark = pytest.mark.gpu

CASES = [
    dict(dtype="bf16", D=128, S=2048, Hq=4, Hkv=4, cp=4, ud=2, layout="zigzag"),
    dict(dtype="bf16", D=128, S=2048, Hq=8, Hkv=2, cp=2, ud=2, layout="stripe"),
    dict(dtype="bf16", D=128, S=1024, Hq=4, Hkv=2, cp=4, ud=1, layout="zigzag"),
    dict(dtype="bf16", D=64, S=1024, Hq=4, Hkv=4, cp=2, ud=2, layout="contiguous", window=200,
         sink_tokens=3),
    dict(dtype="fp32", D=64, S=512, Hq=4, Hkv=2, cp=2, ud=2, layout="zigzag"),
    dict(dtype="fp32", D=64, S=512, Hq=4, Hkv=2, cp=4, ud=1, layout="stripe"),
    dict(dtype="bf16", D=128, S=2048, Hq=4, Hkv=4, cp=2, ud=2, layout="zigzag", varlen=True,
         seg_lo=100, seg_hi=900),
]


@pytest.mark.parametrize("saved", [False, True])
@pytest.mark.parametrize("case", CASES, ids=lambda c: "-".join(f"{k}{v}" for k, v in c.items()))
def test_natural_order_matches_extract_call_restore(case, saved):
    dev = device()
    w = WORKLOADS["tiny_zigzag_cp4"].replace(**case)
    x = make_inputs(w, seed=31, with_grad=True)
    cu = x.get("cu_seqlens")
    cu_dev = cu.to(dev) if cu is not None else None
    nat = {n: x[n].to(dev) for n in ("q", "k", "v", "dout")}
    perm = lambda t: usp.permute(t, "extract", w.layout, w.cp)  # noqa: E731
    unperm = lambda t: usp.permute(t, "restore", w.layout, w.cp)  # noqa: E731
    kw = dict(causal=w.causal, window=w.window, sink_tokens=w.sink_tokens,
              cu_seqlens=cu_dev, cp=w.cp, ud=w.ud, layout=w.layout)
    # the reference: extract, call in rank-major order, restore
    qp, kp, vp, dop = (perm(nat[n]) for n in ("q", "k", "v", "dout"))
    out_p, lse_ref = usp.attn_forward(qp, kp, vp, **kw)
    ref_grads = usp.attn_backward(qp, kp, vp, out_p, lse_ref, dop, **kw)
    out_ref = unperm(out_p)
    # the natural-order calls, sharing one workspace
    ws = usp.attn_workspace(nat["q"], nat["k"], cu_seqlens=cu_dev, cp=w.cp, ud=w.ud,
                            natural=True)
    ws.fill_(0x7F)  # stale contents must not matter
    out, lse = usp.attn_forward(nat["q"], nat["k"], nat["v"], workspace=ws, natural=True, **kw)
    assert torch.equal(out, out_ref) and torch.equal(lse, lse_ref)
    # saved: the copy path reuses the forward's copies of q, k, v, out; the
    # in-place path (tensor-core kernels, contiguous / zigzag) reads them
    grads = usp.attn_backward(nat["q"], nat["k"], nat["v"], out, lse, nat["dout"], workspace=ws,
                              natural=True, saved_exchange=saved, **kw)
    assert torch.equal(grads[1], unperm(ref_grads[1]))
    assert torch.equal(grads[2], unperm(ref_grads[2]))
    ref = attention.attn_bwd(x["q"], x["k"], x["v"], x["dout"], w.scale, w.causal, w.window,
                             w.sink_tokens, cu_seqlens=cu)
    for i, (g, r) in enumerate(zip(grads, ref)):
        e = rel_fro(g.double().cpu().numpy(), r)
        assert np.isfinite(e) and e <= TOL[w.dtype]["grad"], (i, e)

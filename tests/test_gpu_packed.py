"""GPU parity of the packed entry points (one [B,S,3,H,D] tensor): against
the unpacked calls on the same values (bit for bit where the computation is
deterministic) and against the oracle."""
import numpy as np
import pytest
import torch

import sequence_long_context_gb300 as usp
from oracle import attention
from sequence_long_context_gb300.workloads import WORKLOADS, make_inputs
from tests._gpu import TOL, device, rel_fro

pytestmark = pytest.mark.gpu

CASES = [
    dict(dtype="bf16", D=128, S=1024, Hq=4, Hkv=4, cp=4, ud=1, layout="zigzag"),
    dict(dtype="bf16", D=128, S=1024, Hq=4, Hkv=4, cp=2, ud=2, layout="zigzag"),
    dict(dtype="bf16", D=64, S=512, Hq=2, Hkv=2, cp=2, ud=1, layout="stripe", window=100, sink_tokens=2),
    dict(dtype="fp32", D=64, S=256, Hq=2, Hkv=2, cp=4, ud=1, layout="zigzag"),
    dict(dtype="bf16", D=128, S=1024, Hq=4, Hkv=4, cp=2, ud=1, layout="zigzag", varlen=True,
         seg_lo=100, seg_hi=600),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "-".join(f"{k}{v}" for k, v in c.items()))
def test_packed_matches_unpacked_and_oracle(case):
    dev = device()
    w = WORKLOADS["tiny_zigzag_cp4"].replace(**case)
    x = make_inputs(w, seed=11, with_grad=True)
    cu = x.get("cu_seqlens")
    cu_dev = cu.to(dev) if cu is not None else None
    perm = lambda t: usp.permute(t.to(dev), "extract", w.layout, w.cp)  # noqa: E731
    unperm = lambda t: usp.permute(t, "restore", w.layout, w.cp)  # noqa: E731
    kw = dict(causal=w.causal, window=w.window, sink_tokens=w.sink_tokens,
              cu_seqlens=cu_dev, cp=w.cp, ud=w.ud, layout=w.layout)
    qp, kp, vp, dop = perm(x["q"]), perm(x["k"]), perm(x["v"]), perm(x["dout"])
    qkv = torch.stack([qp, kp, vp], dim=-3).contiguous()  # [.., S, 3, H, D]
    out_p, lse_p = usp.attn_forward_qkvpacked(qkv, **kw)
    out_u, lse_u = usp.attn_forward(qp, kp, vp, **kw)
    assert torch.equal(out_p, out_u) and torch.equal(lse_p, lse_u)
    dqkv = usp.attn_backward_qkvpacked(qkv, out_p, lse_p, dop, **kw)
    dq_u, dk_u, dv_u = usp.attn_backward(qp, kp, vp, out_u, lse_u, dop, **kw)
    assert torch.equal(dqkv[..., 1, :, :], dk_u) and torch.equal(dqkv[..., 2, :, :], dv_u)
    tol = TOL[w.dtype]
    O, _ = attention.attn_fwd(x["q"], x["k"], x["v"], w.scale, w.causal, w.window,
                              w.sink_tokens, cu_seqlens=cu)
    assert np.abs(unperm(out_p).double().cpu().numpy() - O).max() <= tol["o"]
    ref = attention.attn_bwd(x["q"], x["k"], x["v"], x["dout"], w.scale, w.causal, w.window,
                             w.sink_tokens, cu_seqlens=cu)
    for i, r in enumerate(ref):
        g = unperm(dqkv[..., i, :, :].contiguous()).double().cpu().numpy()
        assert rel_fro(g, r) <= tol["grad"], i

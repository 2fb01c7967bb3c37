"""Helpers shared by the GPU parity tests: run the CUDA path end to end
(extract -> attention -> restore, all through the C ABI) and compare with the
oracle in natural token order."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import __graft_entry__

# Tolerances. bf16 inputs with fp32 accumulation: max|dO| <= 2e-2,
# max|dLSE| <= 1e-3, gradients <= 5e-2 relative Frobenius; fp32 inputs:
# max|dO| <= 1e-5 (and, derived from it, LSE <= 1e-5 and gradients <= 1e-5
# relative Frobenius: fp32 arithmetic over <= 1e5 keys).
TOL = {
    "bf16": dict(o=2e-2, lse=1e-3, grad=5e-2),
    "fp32": dict(o=1e-5, lse=1e-5, grad=1e-5),
}


def device():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    __graft_entry__.build()
    return torch.device("cuda:0")


def to_np(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def run_forward(usp, w, x, dev, flags=0):
    """Natural-order inputs -> natural-order (O, LSE permuted-order) via the
    library. Returns (o_nat fp64, lse in rank-major order fp64)."""
    cu = x.get("cu_seqlens")
    cu_dev = cu.to(dev) if cu is not None else None
    qp, kp, vp = (usp.permute(x[n].to(dev), "extract", w.layout, w.cp)
                  for n in ("q", "k", "v"))
    out, lse = usp.attn_forward(qp, kp, vp, causal=w.causal, window=w.window,
                                sink_tokens=w.sink_tokens, cu_seqlens=cu_dev,
                                cp=w.cp, ud=w.ud, layout=w.layout, flags=flags)
    o_nat = usp.permute(out, "restore", w.layout, w.cp)
    return o_nat, lse, (qp, kp, vp, out, cu_dev)


def run_backward(usp, w, x, dev, fwd_state, flags=0):
    qp, kp, vp, out, cu_dev = fwd_state[2]
    lse = fwd_state[1]
    dop = usp.permute(x["dout"].to(dev), "extract", w.layout, w.cp)
    dq, dk, dv = usp.attn_backward(qp, kp, vp, out, lse, dop, causal=w.causal,
                                   window=w.window, sink_tokens=w.sink_tokens,
                                   cu_seqlens=cu_dev, cp=w.cp, ud=w.ud,
                                   layout=w.layout, flags=flags)
    return tuple(usp.permute(g, "restore", w.layout, w.cp) for g in (dq, dk, dv))


def lse_to_natural(lse_perm: np.ndarray, w) -> np.ndarray:
    from oracle import layouts
    return layouts.restore(lse_perm, w.layout, w.cp, axis=lse_perm.ndim - 1)


def rel_fro(a: np.ndarray, b: np.ndarray) -> float:
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))

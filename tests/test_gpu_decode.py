"""GPU parity of the decode step (split-KV partials over a sharded cache and
their log-sum-exp merge) against the decode oracle."""
import numpy as np
import pytest
import torch

import sequence_long_context_gb300 as usp
from oracle import decode
from sequence_long_context_gb300.workloads import DECODE_WORKLOADS, make_decode_inputs
from tests._gpu import TOL, device

pytestmark = pytest.mark.gpu

CASES = [
    # B, Tq, S, Hq, Hkv, D, cp, splits, causal, tree
    (2, 1, 512, 8, 2, 128, 2, 2, True, True),
    (1, 3, 1024, 8, 2, 128, 4, 1, True, False),
    (3, 1, 768, 4, 4, 64, 3, 1, True, True),
    (1, 4, 640, 16, 4, 128, 1, 5, False, True),
    (2, 2, 256, 2, 1, 64, 1, 1, True, False),
    (1, 16, 4096, 1, 1, 128, 8, 8, True, True),  # 64 partials, 16 rows per KV head
    (1, 16, 128, 1, 1, 64, 1, 2, True, True),    # the last piece partly masked
    (2, 2, 1024, 8, 2, 128, 2, 2, True, True),   # 8 rows per KV head (five stages)
]


@pytest.mark.parametrize("B,Tq,S,Hq,Hkv,D,cp,splits,causal,tree", CASES)
def test_decode_matches_oracle(B, Tq, S, Hq, Hkv, D, cp, splits, causal, tree):
    if Tq * Hq // Hkv > 16:
        pytest.skip("more than 16 query rows per KV head")
    dev = device()
    g = torch.Generator().manual_seed(B * 1000 + S + Tq)
    q = torch.randn(B, Tq, Hq, D, generator=g).to(torch.bfloat16)
    k = torch.randn(B, S, Hkv, D, generator=g).to(torch.bfloat16)
    v = torch.randn(B, S, Hkv, D, generator=g).to(torch.bfloat16)
    scale = 1.0 / np.sqrt(D)
    out, lse = usp.attn_decode(q.to(dev), k.to(dev), v.to(dev), causal=causal, cp=cp,
                               splits=splits, tree_order=tree)
    O, L = decode.decode_fwd(q, k, v, scale, causal)
    tol = TOL["bf16"]
    got_o = out.float().cpu().numpy()
    got_l = lse.cpu().numpy()
    assert np.isfinite(got_o).all()
    assert np.abs(got_o - O).max() <= tol["o"]
    assert np.abs(got_l - L).max() <= tol["lse"]


def test_decode_rows_beyond_limit_rejected():
    dev = device()
    q = torch.zeros(1, 5, 8, 64, dtype=torch.bfloat16, device=dev)
    k = torch.zeros(1, 256, 2, 64, dtype=torch.bfloat16, device=dev)
    with pytest.raises(usp.UspError, match="UNSUPPORTED"):
        usp.attn_decode(q, k, k)


def test_decode_full_workload_sampled():
    """The benchmark's decode step at full size, checked on sampled KV groups
    of sampled sequences (every query head of the group)."""
    w = DECODE_WORKLOADS["decode_gqa_b8_s128k_cp8"]
    dev = device()
    x = make_decode_inputs(w, seed=0, device="cuda")
    out, lse = usp.attn_decode(x["q"], x["k"], x["v"], causal=w.causal, cp=w.cp,
                               splits=w.splits, tree_order=True)
    torch.cuda.synchronize()
    rng = np.random.default_rng(5)
    G = w.Hq // w.Hkv
    tol = TOL["bf16"]
    for b in rng.choice(w.B, 2, replace=False):
        g = int(rng.integers(w.Hkv))
        hs = slice(g * G, (g + 1) * G)
        qc = x["q"][b:b + 1, :, hs].cpu()
        kc = x["k"][b:b + 1, :, g:g + 1].cpu()
        vc = x["v"][b:b + 1, :, g:g + 1].cpu()
        O, L = decode.decode_fwd(qc, kc, vc, w.scale, w.causal)
        got_o = out[b:b + 1, :, hs].float().cpu().numpy()
        got_l = lse[b:b + 1, :, hs].cpu().numpy()
        assert np.abs(got_o - O).max() <= tol["o"]
        assert np.abs(got_l - L).max() <= tol["lse"]

"""GPU parity at the full problem sizes, in the benchmark's launch
configuration: the benchmark's own training step (natural-order forward and
backward sharing one workspace, tensor-core kernels where they apply).

The oracle cannot redo a full problem in seconds, so outputs are checked on
seeded samples it computes one by one from the definition: O and LSE rows of
sampled (batch, head, position) triples, dQ rows of every query head of a
sampled KV group, and dK/dV rows of sampled keys of that group. Sampled
positions include chunk and shard boundaries, the first and the last token.
"""
import zlib

import numpy as np
import pytest
import torch

import bench
import sequence_long_context_gb300 as usp
from oracle import attention
from sequence_long_context_gb300.workloads import WORKLOADS, make_inputs
from tests._gpu import TOL, device, lse_to_natural, rel_fro

pytestmark = pytest.mark.gpu

# the five problem statements, the sliding-window training step, and the
# zigzag sweep points that carry the throughput gate (S = 32K) and the end of
# the measured range (S = 128K: a 2 GiB fp32 dQ accumulator)
CONFIGS = ["usp_ud2_ring4_s8k", "gqa_stripe_cp8_s32k", "swa_w1000_cp8_s8k",
           "swa_w1000_sink4_cp8_s8k", "swa_w1000_sink4_cp8_s8k_train",
           "varlen_zigzag_cp8_t128k", "sweep_zigzag_cp8_s32k", "sweep_zigzag_cp8_s128k"]


def sample_positions(w, rng, n=40):
    C = w.S // (2 * w.cp)
    special = [0, 1, C - 1, C, w.S // w.cp, w.S // 2, w.S - 2, w.S - 1]
    return sorted(set(special) | set(rng.choice(w.S, n, replace=False).tolist()))


@pytest.mark.parametrize("name", CONFIGS)
def test_full_config(name):
    w = WORKLOADS[name]
    dev = device()
    rng = np.random.default_rng(zlib.crc32(name.encode()))
    x = make_inputs(w, seed=0, device="cuda")
    cu_dev = x.get("cu_seqlens")
    kept = {}
    res = bench.make_step(usp, w, x, cu_dev.to(dev) if cu_dev is not None else None,
                          keep=kept)(x)
    o_nat = res[0]
    grads = tuple(res[1:]) if w.backward else None
    torch.cuda.synchronize()
    xc = {k: v.cpu() for k, v in x.items()}
    cu = xc.get("cu_seqlens")
    tol = TOL[w.dtype]
    lse_nat = lse_to_natural(kept["lse"].cpu().numpy().astype(np.float64), w)
    rows = sample_positions(w, rng)
    G = w.Hq // w.Hkv
    g = int(rng.integers(w.Hkv))
    heads = sorted(set(range(g * G, (g + 1) * G)) | {int(rng.integers(w.Hq))})
    batches = [0] if w.varlen else list(range(w.B))
    for b in batches:
        for h in heads:
            O, L = attention.attn_fwd_rows(xc["q"], xc["k"], xc["v"], w.scale, b, h, rows,
                                           w.causal, w.window, w.sink_tokens, cu_seqlens=cu)
            if w.varlen:
                o = o_nat[rows, h].float().cpu().numpy()
                lse = lse_nat[h, rows]
            else:
                o = o_nat[b, rows, h].float().cpu().numpy()
                lse = lse_nat[b, h, rows]
            assert np.abs(o - O).max() <= tol["o"], (b, h)
            assert np.abs(lse - L).max() <= tol["lse"], (b, h)
    if grads is None:
        return
    b = batches[-1]
    if w.S >= 131072:
        # at S = 128K the dK/dV rows are keys of the last 4096 positions: the
        # oracle needs the forward of every query that sees a sampled key,
        # and these are seen by at most 4096 queries each (the dQ rows above
        # still span the whole sequence)
        lo = w.S - 4096
        keys = sorted({lo, lo + 1, w.S - 129, w.S - 128, w.S - 1}
                      | set(rng.choice(np.arange(lo, w.S), 19, replace=False).tolist()))
    else:
        keys = sample_positions(w, rng, 24)
    dq_ref, dk_ref, dv_ref = attention.attn_bwd_sampled(
        xc["q"], xc["k"], xc["v"], xc["dout"], w.scale, b, g, rows, keys,
        w.causal, w.window, w.sink_tokens, cu_seqlens=cu)
    sel = (lambda t: t) if w.varlen else (lambda t: t[b])
    dq = sel(grads[0])[rows][:, g * G:(g + 1) * G].float().cpu().numpy().transpose(1, 0, 2)
    dk = sel(grads[1])[keys, g].float().cpu().numpy()
    dv = sel(grads[2])[keys, g].float().cpu().numpy()
    for nm, got, ref in (("dq", dq, dq_ref), ("dk", dk, dk_ref), ("dv", dv, dv_ref)):
        e = rel_fro(got, ref)
        assert e <= tol["grad"], (nm, e)

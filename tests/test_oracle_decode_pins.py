"""Pins for the decode-step oracle (oracle/decode.py), on the CPU.

Each check ties the oracle to something other than itself: torch's fp64
scaled_dot_product_attention with a mask cut from torch.tril, the full
attention oracle's last rows (itself pinned to SDPA), the merge of per-shard
partials (the pages' flash-decoding / tree-reduction claim, "Long Context
Attention" notes, "Ring Attention" and "Tree Attention"), a closed-form
special case, and a planted mistake that must fail.
"""
import math

import numpy as np
import pytest
import torch

from oracle import attention, decode, merge


def rnd(shape, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(shape, generator=g, dtype=torch.float64)


def lib_decode(q, k, v, causal, scale):
    """SDPA over the newest Tq rows of a causal S x S mask (torch.tril)."""
    B, Tq, Hq, D = q.shape
    S = k.shape[1]
    G = Hq // k.shape[2]
    mask = torch.tril(torch.ones(S, S, dtype=torch.bool))[S - Tq:]
    if not causal:
        mask = torch.ones(Tq, S, dtype=torch.bool)
    kr, vr = k.repeat_interleave(G, dim=2), v.repeat_interleave(G, dim=2)
    qt, kt, vt = (x.transpose(1, 2) for x in (q, kr, vr))
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask,
                                                         scale=scale)
    s = torch.matmul(qt, kt.transpose(-1, -2)) * scale
    lse = torch.logsumexp(s.masked_fill(~mask, -math.inf), dim=-1)  # [B,Hq,Tq]
    return o.transpose(1, 2).numpy(), lse.transpose(1, 2).numpy()


CASES = [(1, 1, 40, 4, 1, 8, True), (2, 3, 40, 4, 2, 8, True), (1, 5, 33, 2, 2, 16, False),
         (2, 1, 64, 8, 2, 8, False)]


@pytest.mark.parametrize("B,Tq,S,Hq,Hkv,D,causal", CASES)
def test_decode_matches_library_sdpa(B, Tq, S, Hq, Hkv, D, causal):
    q, k, v = rnd((B, Tq, Hq, D), 1), rnd((B, S, Hkv, D), 2), rnd((B, S, Hkv, D), 3)
    O, L = decode.decode_fwd(q, k, v, 0.35, causal)
    o_ref, l_ref = lib_decode(q, k, v, causal, 0.35)
    np.testing.assert_allclose(O, o_ref, atol=1e-12, rtol=0)
    np.testing.assert_allclose(L, l_ref, atol=1e-12, rtol=0)


def test_decode_equals_tail_of_full_attention():
    B, Tq, S, Hq, Hkv, D = 2, 4, 30, 4, 2, 8
    q, k, v = rnd((B, Tq, Hq, D), 4), rnd((B, S, Hkv, D), 5), rnd((B, S, Hkv, D), 6)
    qfull = rnd((B, S, Hq, D), 7)
    qfull[:, S - Tq:] = q
    O_full, L_full = attention.attn_fwd(qfull, k, v, 0.4, causal=True)
    O, L = decode.decode_fwd(q, k, v, 0.4, causal=True)
    np.testing.assert_allclose(O, O_full[:, S - Tq:], atol=1e-12, rtol=0)
    np.testing.assert_allclose(L, L_full[:, :, S - Tq:].transpose(0, 2, 1), atol=1e-12, rtol=0)


@pytest.mark.parametrize("n_parts", [1, 2, 4, 8])
@pytest.mark.parametrize("Tq", [1, 3, 20])
@pytest.mark.parametrize("tree", [False, True])
def test_shard_partials_merge_to_decode(n_parts, Tq, tree):
    # Tq = 20 > piece length 4 at n_parts = 8: whole pieces are invisible to
    # the earliest queries, so empty partials (LSE = -inf) take part
    B, S, Hq, Hkv, D = 1, 32, 4, 2, 8
    q, k, v = rnd((B, Tq, Hq, D), 8), rnd((B, S, Hkv, D), 9), rnd((B, S, Hkv, D), 10)
    parts = decode.decode_partials(q, k, v, 0.3, True, n_parts)
    O, L = (merge.merge_tree if tree else merge.merge_linear)(parts)
    O_ref, L_ref = decode.decode_fwd(q, k, v, 0.3, True)
    np.testing.assert_allclose(O, O_ref, atol=1e-12, rtol=0)
    np.testing.assert_allclose(L, L_ref, atol=1e-12, rtol=0)
    if Tq == 20 and n_parts == 8:
        assert np.isneginf(parts[-1][1][0, 0]).all()  # the last piece is empty for t=0


def test_single_key_cache():
    q, k, v = rnd((1, 1, 2, 4), 11), rnd((1, 1, 2, 4), 12), rnd((1, 1, 2, 4), 13)
    O, L = decode.decode_fwd(q, k, v, 0.5)
    np.testing.assert_allclose(O[0, 0], v[0, 0].numpy(), atol=1e-15)
    np.testing.assert_allclose(L[0, 0], 0.5 * (q[0, 0] * k[0, 0]).sum(-1).numpy(), atol=1e-15)


def test_pin_catches_planted_off_by_one(monkeypatch):
    B, Tq, S, Hq, Hkv, D = 1, 3, 20, 2, 1, 8
    q, k, v = rnd((B, Tq, Hq, D), 14), rnd((B, S, Hkv, D), 15), rnd((B, S, Hkv, D), 16)
    o_ref, _ = lib_decode(q, k, v, True, 0.3)
    real = decode.softmax_rows

    def hides_own_key(qq, kk, vv, vis, scale):
        vis = vis.copy()
        vis[np.arange(vis.shape[0]), vis.shape[1] - vis.shape[0] + np.arange(vis.shape[0])] = False
        return real(qq, kk, vv, vis, scale)

    monkeypatch.setattr(decode, "softmax_rows", hides_own_key)
    O, _ = decode.decode_fwd(q, k, v, 0.3, True)
    assert np.abs(O - o_ref).max() > 1e-3

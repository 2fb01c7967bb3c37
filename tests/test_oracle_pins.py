"""Pins for the CPU oracle: each check ties it to something other than itself.

Library routines (torch's fp64 scaled_dot_product_attention, logsumexp and
autograd, with masks built from tril/triu/block_diag), central finite
differences, closed-form pair counts, and the worked examples the pages
print. None of these re-types the oracle's own formula.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import attention, layouts, merge, ring

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "worked_examples.json")
LAYOUTS = ("contiguous", "zigzag", "stripe")


def rnd(shape, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(shape, generator=g, dtype=torch.float64)


def lib_mask(S, causal, window, sink):
    """Visibility built from library band/triangle primitives."""
    m = torch.ones(S, S, dtype=torch.bool)
    if causal:
        m = torch.tril(m)
    if window > 0:
        band = torch.triu(torch.ones(S, S, dtype=torch.bool), diagonal=-(window - 1))
        sinks = torch.zeros(S, S, dtype=torch.bool)
        sinks[:, :sink] = True
        m = m & (band | sinks)
    return m


def lib_attention(q, k, v, mask, scale):
    """torch SDPA (fp64) and torch.logsumexp on [B,S,H,D] inputs, GQA by repeat."""
    G = q.shape[2] // k.shape[2]
    kr = k.repeat_interleave(G, dim=2)
    vr = v.repeat_interleave(G, dim=2)
    qt, kt, vt = (x.transpose(1, 2) for x in (q, kr, vr))
    o = torch.nn.functional.scaled_dot_product_attention(
        qt, kt, vt, attn_mask=mask, scale=scale)
    s = torch.matmul(qt, kt.transpose(-1, -2)) * scale
    lse = torch.logsumexp(s.masked_fill(~mask, -math.inf), dim=-1)
    return o.transpose(1, 2), lse


CASES = [
    # S, Hq, Hkv, D, causal, window, sink
    (13, 2, 2, 8, True, 0, 0),
    (13, 4, 2, 8, False, 0, 0),
    (24, 4, 1, 16, True, 5, 0),
    (24, 2, 2, 8, True, 5, 2),
    (17, 2, 2, 8, False, 4, 0),
    (9, 2, 2, 4, True, 100, 0),
]


@pytest.mark.parametrize("S,Hq,Hkv,D,causal,window,sink", CASES)
def test_fwd_matches_library_sdpa(S, Hq, Hkv, D, causal, window, sink):
    q, k, v = rnd((2, S, Hq, D), 1), rnd((2, S, Hkv, D), 2), rnd((2, S, Hkv, D), 3)
    scale = 1 / math.sqrt(D)
    O, L = attention.attn_fwd(q, k, v, scale, causal, window, sink)
    mask = lib_mask(S, causal, window, sink)
    o_ref, l_ref = lib_attention(q, k, v, mask, scale)
    np.testing.assert_allclose(O, o_ref.numpy(), atol=1e-12, rtol=0)
    np.testing.assert_allclose(L, l_ref.numpy(), atol=1e-12, rtol=0)


@pytest.mark.parametrize("S,Hq,Hkv,D,causal,window,sink", CASES)
def test_bwd_matches_torch_autograd(S, Hq, Hkv, D, causal, window, sink):
    q, k, v = rnd((1, S, Hq, D), 4), rnd((1, S, Hkv, D), 5), rnd((1, S, Hkv, D), 6)
    do = rnd((1, S, Hq, D), 7)
    scale = 1 / math.sqrt(D)
    dq, dk, dv = attention.attn_bwd(q, k, v, do, scale, causal, window, sink)
    qq, kk, vv = (x.clone().requires_grad_(True) for x in (q, k, v))
    o, _ = lib_attention(qq, kk, vv, lib_mask(S, causal, window, sink), scale)
    (o * do).sum().backward()
    np.testing.assert_allclose(dq, qq.grad.numpy(), atol=1e-11)
    np.testing.assert_allclose(dk, kk.grad.numpy(), atol=1e-11)
    np.testing.assert_allclose(dv, vv.grad.numpy(), atol=1e-11)


def test_bwd_matches_finite_differences():
    S, Hq, Hkv, D = 11, 2, 1, 4
    q, k, v = (rnd(s, i).numpy() for i, s in
               enumerate([(1, S, Hq, D), (1, S, Hkv, D), (1, S, Hkv, D)]))
    do = rnd((1, S, Hq, D), 9).numpy()
    scale = 0.37
    kw = dict(causal=True, window=6, sink_tokens=1)
    dq, dk, dv = attention.attn_bwd(q, k, v, do, scale, **kw)

    def f(q_, k_, v_):
        return float((attention.attn_fwd(q_, k_, v_, scale, **kw)[0] * do).sum())

    eps = 1e-6
    for grad, which in ((dq, 0), (dk, 1), (dv, 2)):
        args = [q, k, v]
        fd = np.zeros_like(args[which])
        it = np.nditer(args[which], flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            plus = [a.copy() for a in args]
            minus = [a.copy() for a in args]
            plus[which][idx] += eps
            minus[which][idx] -= eps
            fd[idx] = (f(*plus) - f(*minus)) / (2 * eps)
        rel = np.linalg.norm(fd - grad) / np.linalg.norm(grad)
        assert rel < 1e-6, (which, rel)


def test_varlen_matches_block_diagonal_sdpa():
    cu = [0, 5, 6, 19, 32]
    T, Hq, Hkv, D = 32, 4, 2, 8
    q, k, v = rnd((T, Hq, D), 11), rnd((T, Hkv, D), 12), rnd((T, Hkv, D), 13)
    scale = 0.3
    for causal, window, sink in ((True, 0, 0), (True, 4, 2), (False, 0, 0)):
        O, L = attention.attn_fwd(q, k, v, scale, causal, window, sink,
                                  cu_seqlens=cu)
        blocks = [lib_mask(cu[i + 1] - cu[i], causal, window, sink)
                  for i in range(len(cu) - 1)]
        mask = torch.block_diag(*blocks)
        o_ref, l_ref = lib_attention(q[None], k[None], v[None], mask, scale)
        np.testing.assert_allclose(O, o_ref[0].numpy(), atol=1e-12)
        np.testing.assert_allclose(L, l_ref[0].numpy(), atol=1e-12)


def test_special_cases():
    D = 8
    q, k, v = rnd((1, 1, 1, D), 20), rnd((1, 1, 1, D), 21), rnd((1, 1, 1, D), 22)
    O, L = attention.attn_fwd(q, k, v, 0.5)
    np.testing.assert_allclose(O[0, 0, 0], v[0, 0, 0].numpy(), atol=1e-15)
    np.testing.assert_allclose(L[0, 0, 0], 0.5 * float((q * k).sum()), atol=1e-14)
    # window >= S is plain causal
    q, k, v = rnd((1, 20, 2, D), 23), rnd((1, 20, 2, D), 24), rnd((1, 20, 2, D), 25)
    a = attention.attn_fwd(q, k, v, 0.3, True, 0)
    b = attention.attn_fwd(q, k, v, 0.3, True, 20)
    np.testing.assert_allclose(a[0], b[0], atol=1e-15)
    # GQA equals repeated KV heads
    q, k, v = rnd((1, 20, 8, D), 26), rnd((1, 20, 2, D), 27), rnd((1, 20, 2, D), 28)
    g = attention.attn_fwd(q, k, v, 0.3, True)
    r = attention.attn_fwd(q, k.repeat_interleave(4, 2), v.repeat_interleave(4, 2), 0.3, True)
    np.testing.assert_allclose(g[0], r[0], atol=1e-15)
    np.testing.assert_allclose(g[1], r[1], atol=1e-15)
    # rows outside every window (fully masked): O = 0, LSE = -inf, via partials
    vis = np.zeros((3, 4), bool)
    o, lse = attention.softmax_rows(np.ones((3, D)), np.ones((4, D)), np.ones((4, D)), vis, 1.0)
    assert np.all(o == 0) and np.all(np.isneginf(lse))


def test_rows_match_full():
    S, Hq, Hkv, D = 40, 4, 2, 8
    q, k, v = rnd((2, S, Hq, D), 30), rnd((2, S, Hkv, D), 31), rnd((2, S, Hkv, D), 32)
    O, L = attention.attn_fwd(q, k, v, 0.3, True, 7, 2)
    rows = [0, 3, 17, 39]
    o, lse = attention.attn_fwd_rows(q, k, v, 0.3, 1, 3, rows, True, 7, 2)
    np.testing.assert_allclose(o, O[1, rows, 3], atol=1e-13)
    np.testing.assert_allclose(lse, L[1, 3, rows], atol=1e-13)
    cu = [0, 9, 40]
    O, L = attention.attn_fwd(q[0], k[0], v[0], 0.3, True, cu_seqlens=cu)
    o, lse = attention.attn_fwd_rows(q[0], k[0], v[0], 0.3, 0, 1, [8, 9, 30],
                                     True, cu_seqlens=cu)
    np.testing.assert_allclose(o, O[[8, 9, 30], 1], atol=1e-13)


# ----------------------------------------------------------------------------
# layouts


def test_layout_worked_examples():
    gold = json.load(open(GOLDEN))
    ex = gold["stripe_16_tokens_4_ranks"]
    assert layouts.shard_positions("stripe", ex["S"], ex["cp"], ex["rank"]).tolist() == ex["positions"]
    ex = gold["zigzag_tiny_S256_cp4"]
    C = ex["chunk"]
    for r, chunks in enumerate(ex["rank_chunks"]):
        want = np.concatenate([np.arange(c * C, (c + 1) * C) for c in chunks])
        assert layouts.shard_positions("zigzag", ex["S"], ex["cp"], r).tolist() == want.tolist()


@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("cp", [1, 2, 3, 4, 8])
def test_restore_extract_identity(layout, cp):
    S = 2 * cp * 6
    x = np.arange(2 * S * 3).reshape(2, S, 3)
    perm = layouts.permutation(layout, S, cp)
    assert sorted(perm.tolist()) == list(range(S))
    y = layouts.extract(x, layout, cp)
    assert not (layout != "contiguous" and cp > 1 and np.array_equal(x, y))
    assert np.array_equal(layouts.restore(y, layout, cp), x)


@pytest.mark.parametrize("cp,ud", [(1, 2), (4, 2), (2, 4), (3, 2)])
def test_ulysses_roundtrip_and_head_slices(cp, ud):
    B, S, H, D = 2, cp * ud * 4, 8, 3
    x = np.arange(B * S * H * D).reshape(B, S, H, D)
    y = layouts.ulysses_seq2head(x, cp, ud)
    assert y.shape == (ud, B, S, H // ud, D)
    # after the exchange, group u holds heads u*H/ud.. of every token
    for u in range(ud):
        assert np.array_equal(y[u], x[:, :, u * (H // ud):(u + 1) * (H // ud)])
    assert np.array_equal(layouts.ulysses_head2seq(y, cp, ud), x)


def test_stripe_round_rule():
    """Round r: host h receives KV of host (h - r) mod cp; the pair is strictly
    causal (first query and last key dropped) exactly when h < r."""
    S, cp = 16, 4
    n = S // cp
    lower_incl = np.tril(np.ones((n, n), bool))
    lower_strict = np.tril(np.ones((n, n), bool), -1)
    for h in range(cp):
        for r in range(cp):
            kap = (h - r) % cp
            qn = layouts.shard_positions("stripe", S, cp, h)
            kn = layouts.shard_positions("stripe", S, cp, kap)
            vis = attention.visibility(qn, kn, True, 0, 0)
            want = lower_strict if h < r else lower_incl
            assert np.array_equal(vis, want), (h, r)


@pytest.mark.parametrize("cp", [2, 4, 8])
def test_zigzag_squares_and_balance(cp):
    S = 2 * cp * 16
    C = S // (2 * cp)
    for qc in range(2 * cp):
        for kc in range(2 * cp):
            if qc == kc:
                continue
            vis = attention.visibility(np.arange(qc * C, (qc + 1) * C),
                                       np.arange(kc * C, (kc + 1) * C), True, 0, 0)
            assert vis.all() or not vis.any()
    counts = ring.step_pair_counts("zigzag", S, cp).sum(axis=1)
    assert set(counts.tolist()) == {(2 * cp - 1) * C * C + C * (C + 1)}


def test_tiny_config_pair_counts():
    # zigzag cp=4, S=256: (2cp-1)C^2 + C(C+1) = 8224 pairs per rank
    assert ring.step_pair_counts("zigzag", 256, 4).sum(axis=1).tolist() == [8224] * 4
    # stripe: rank r holds 4i + r: sum_{i<64} (4i + r + 1) = 8064 + 64(r+1)
    assert ring.step_pair_counts("stripe", 256, 4).sum(axis=1).tolist() == [8128, 8192, 8256, 8320]


def test_window_steps_and_pair_counts():
    S, cp, W = 8192, 8, 1000
    c = ring.step_pair_counts("contiguous", S, cp, True, W, 0)
    assert np.all(c[:, 2:] == 0) and np.all(c[1:, :2] > 0) and c[0, 1] == 0
    # closed form: sum_i min(i+1, W) = W(W-1)/2 + (S-W+1)W ... per head
    assert c.sum() == attention.count_visible_pairs(S, True, W, 0) == 7692500
    c4 = ring.step_pair_counts("contiguous", S, cp, True, W, 4)
    for rho in range(cp):
        for s in range(cp):
            expect_nonzero = s in (0, 1) or s == rho
            if rho == 0 and s == 1:
                expect_nonzero = False
            assert (c4[rho, s] > 0) == expect_nonzero, (rho, s)
    # extra sink pairs: sum_{i>=1000} min(4, i-999) = 6 + 4*7189 = 28762
    assert c4.sum() == attention.count_visible_pairs(S, True, W, 4) == 7721262


# ----------------------------------------------------------------------------
# merge and ring


def _random_partials(n, rows, D, seed):
    g = np.random.default_rng(seed)
    parts = [(g.standard_normal((rows, D)), g.standard_normal(rows) * 3) for _ in range(n)]
    parts[1][1][::5] = -np.inf
    parts[1][0][::5] = 0.0
    return parts


def test_merge_matches_library_logsumexp():
    parts = _random_partials(5, 33, 7, 1)
    O, L = merge.merge_linear(parts)
    Ls = torch.tensor(np.stack([p[1] for p in parts]))
    np.testing.assert_allclose(L, torch.logsumexp(Ls, 0).numpy(), atol=1e-13)
    w = torch.softmax(Ls, 0).numpy()
    np.testing.assert_allclose(O, sum(w[i][:, None] * parts[i][0] for i in range(5)), atol=1e-13)


@pytest.mark.parametrize("n", [1, 2, 3, 4, 7, 8])
def test_merge_order_independence(n):
    parts = _random_partials(max(n, 2), 40, 16, n)[:n]
    a = merge.merge_linear(parts)
    b = merge.merge_tree(parts)
    rng = np.random.default_rng(n)
    c = merge.merge_linear([parts[i] for i in rng.permutation(n)])
    for x in (b, c):
        np.testing.assert_allclose(x[0], a[0], atol=1e-12)
        np.testing.assert_allclose(x[1], a[1], atol=1e-12)


def test_merge_empty_is_identity():
    o = np.random.default_rng(0).standard_normal((4, 3))
    l = np.array([0.1, -2.0, 5.0, -np.inf])
    empty = (np.zeros((4, 3)), np.full(4, -np.inf))
    for x in (merge.merge_pair(empty, (o, l)), merge.merge_pair((o, l), empty)):
        assert np.array_equal(x[1], l)
        np.testing.assert_allclose(x[0][:3], o[:3], atol=0)
        assert np.all(x[0][3] == 0)


RING_CASES = [
    # causal, window, sink, varlen
    (True, 0, 0, False),
    (False, 0, 0, False),
    (True, 13, 0, False),
    (True, 13, 3, False),
    (True, 0, 0, True),
    (True, 9, 2, True),
]


@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("cp,ud", [(1, 1), (2, 1), (3, 1), (4, 1), (8, 1), (1, 2), (2, 2), (4, 2), (3, 2)])
@pytest.mark.parametrize("causal,window,sink,varlen", RING_CASES)
def test_ring_chunk_merge_equals_full(layout, cp, ud, causal, window, sink, varlen):
    S = 96
    Hq, Hkv, D = 4, 2, 8
    if varlen:
        cu = [0, 7, 40, 41, 96]
        q, k, v = rnd((S, Hq, D), 40), rnd((S, Hkv, D), 41), rnd((S, Hkv, D), 42)
    else:
        cu = None
        q, k, v = rnd((2, S, Hq, D), 40), rnd((2, S, Hkv, D), 41), rnd((2, S, Hkv, D), 42)
    scale = 0.35
    O, L = attention.attn_fwd(q, k, v, scale, causal, window, sink, cu_seqlens=cu)
    for order in ("ring", "tree"):
        Or, Lr = ring.ring_attn_fwd(q, k, v, scale, layout, cp, ud, causal,
                                    window, sink, cu_seqlens=cu, order=order)
        np.testing.assert_allclose(Or, O, atol=1e-12)
        np.testing.assert_allclose(Lr, L, atol=1e-12)


@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("cp,ud", [(1, 1), (4, 1), (3, 1), (2, 2), (4, 2)])
@pytest.mark.parametrize("window,sink,varlen", [(0, 0, False), (11, 2, False), (0, 0, True)])
def test_ring_bwd_equals_full(layout, cp, ud, window, sink, varlen):
    S, Hq, Hkv, D = 48, 4, 2, 8
    if varlen:
        cu = [0, 20, 21, 48]
        shp_q, shp_k = (S, Hq, D), (S, Hkv, D)
    else:
        cu = None
        shp_q, shp_k = (1, S, Hq, D), (1, S, Hkv, D)
    q, k, v, do = rnd(shp_q, 50), rnd(shp_k, 51), rnd(shp_k, 52), rnd(shp_q, 53)
    full = attention.attn_bwd(q, k, v, do, 0.3, True, window, sink, cu_seqlens=cu)
    rg = ring.ring_attn_bwd(q, k, v, do, 0.3, layout, cp, ud, True, window, sink, cu_seqlens=cu)
    for a, b in zip(rg, full):
        np.testing.assert_allclose(a, b, atol=1e-12)


def test_pin_catches_planted_mistakes(monkeypatch):
    """A wrong window bound or a transposed GQA map must fail a pin."""
    S, D = 24, 8
    q, k, v = rnd((1, S, 4, D), 60), rnd((1, S, 2, D), 61), rnd((1, S, 2, D), 62)
    o_ref, _ = lib_attention(q, k, v, lib_mask(S, True, 5, 0), 0.3)
    real = attention.visibility

    def off_by_one(qpos, kpos, causal, window, sink):
        return real(qpos, kpos, causal, window + 1, sink)

    monkeypatch.setattr(attention, "visibility", off_by_one)
    O, _ = attention.attn_fwd(q, k, v, 0.3, True, 5, 0)
    assert np.abs(O - o_ref.numpy()).max() > 1e-3


@pytest.mark.parametrize("varlen", [False, True])
def test_sampled_bwd_matches_full(varlen):
    S, Hq, Hkv, D = 40, 6, 2, 8
    cu = [0, 13, 14, 40] if varlen else None
    if varlen:
        q, k, v, do = rnd((S, Hq, D), 70), rnd((S, Hkv, D), 71), rnd((S, Hkv, D), 72), rnd((S, Hq, D), 73)
    else:
        q, k, v, do = rnd((2, S, Hq, D), 70), rnd((2, S, Hkv, D), 71), rnd((2, S, Hkv, D), 72), rnd((2, S, Hq, D), 73)
    kw = dict(causal=True, window=9, sink_tokens=2, cu_seqlens=cu)
    dq, dk, dv = attention.attn_bwd(q, k, v, do, 0.4, **kw)
    b = 0 if varlen else 1
    rows, keys = [0, 5, 13, 14, 39], [0, 1, 12, 20, 39]
    sq, sk, sv = attention.attn_bwd_sampled(q, k, v, do, 0.4, b, 1, rows, keys, **kw)
    sel = (lambda t: t) if varlen else (lambda t: t[b])
    np.testing.assert_allclose(sq, np.transpose(sel(dq)[rows][:, 3:6], (1, 0, 2)), atol=1e-12)
    np.testing.assert_allclose(sk, sel(dk)[keys, 1], atol=1e-12)
    np.testing.assert_allclose(sv, sel(dv)[keys, 1], atol=1e-12)


@pytest.mark.parametrize("varlen", [False, True])
def test_sampled_bwd_late_keys_matches_full(varlen):
    # keys late in their sequences are seen by few queries, so the sampled
    # backward computes the forward of only those rows (and of the dq rows):
    # the skipped rows must not matter
    S, Hq, Hkv, D = 48, 4, 2, 8
    cu = [0, 20, 21, 48] if varlen else None
    if varlen:
        q, k, v, do = rnd((S, Hq, D), 80), rnd((S, Hkv, D), 81), rnd((S, Hkv, D), 82), rnd((S, Hq, D), 83)
    else:
        q, k, v, do = rnd((1, S, Hq, D), 80), rnd((1, S, Hkv, D), 81), rnd((1, S, Hkv, D), 82), rnd((1, S, Hq, D), 83)
    for kw in (dict(causal=True), dict(causal=True, window=6, sink_tokens=1)):
        dq, dk, dv = attention.attn_bwd(q, k, v, do, 0.35, cu_seqlens=cu, **kw)
        rows, keys = [3, 19, 33], [17, 19, 20, 44, 47]
        sq, sk, sv = attention.attn_bwd_sampled(q, k, v, do, 0.35, 0, 1, rows, keys,
                                                cu_seqlens=cu, **kw)
        sel = (lambda t: t) if varlen else (lambda t: t[0])
        np.testing.assert_allclose(sq, np.transpose(sel(dq)[rows][:, 2:4], (1, 0, 2)), atol=1e-12)
        np.testing.assert_allclose(sk, sel(dk)[keys, 1], atol=1e-12)
        np.testing.assert_allclose(sv, sel(dv)[keys, 1], atol=1e-12)

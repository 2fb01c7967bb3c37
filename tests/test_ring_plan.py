"""The multi-device ring plan (sequence_long_context_gb300.ring_plan), checked on
the host: its invariants, then executed by gloo ranks on the CPU (2 and 4
ranks, 127.0.0.1) that send the KV shards (and, backward, their dK/dV) to the
peers the plan names, compute each step's partial with the oracle's plain
softmax over the pair's visible keys, merge with the oracle's log-sum-exp rule
and compare the gathered result with the oracle's full attention. A wrong
peer, owner, buffer or return hop shows up as a wrong result (or a timeout of
the process group)."""
import datetime
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from sequence_long_context_gb300 import ring_plan as rp


@pytest.mark.parametrize("layout", rp.LAYOUTS)
@pytest.mark.parametrize("cp", [1, 2, 3, 4, 8])
def test_every_rank_sees_every_shard_once_and_peers_agree(layout, cp):
    plans = [rp.forward_plan(r, cp, layout) for r in range(cp)]
    for r, plan in enumerate(plans):
        assert sorted(st.kv_owner for st in plan) == list(range(cp))
        assert plan[0].kv_owner == r  # a rank starts on its own shard
        for s, st in enumerate(plan[:-1]):
            # what r sends at step s is what r + 1 uses at step s + 1, and it
            # lands in the other buffer
            nxt = plans[st.send_to][s + 1]
            assert st.send_to == (r + 1) % cp and nxt.kv_owner == st.kv_owner
            assert plans[st.send_to][s].recv_from == r
            assert nxt.buf != st.buf
        assert plan[-1].send_to is None and plan[-1].recv_from is None
    dest, src = rp.backward_plan(0, cp, layout)[1]
    assert dest == 1 % cp and src == (cp - 1) % cp


@pytest.mark.parametrize("cp", [2, 4, 8])
def test_zigzag_steps_are_balanced(cp):
    # "Zig-Zag Attention": after the first step every rank meets exactly two
    # full chunk squares per step; the first step is the two diagonals and
    # one full square on every rank
    for r in range(cp):
        plan = rp.forward_plan(r, cp, "zigzag")
        classes0 = sorted(c for _, _, c in plan[0].pairs)
        assert classes0 == sorted([rp.DIAGONAL, rp.DIAGONAL, rp.FULL, rp.EMPTY])
        for st in plan[1:]:
            assert sorted(c for _, _, c in st.pairs).count(rp.FULL) == 2
            assert all(c in (rp.FULL, rp.EMPTY) for _, _, c in st.pairs)


def test_stripe_rule_drops_the_diagonal_when_the_host_is_below_the_round():
    # round s: rank h holds shard (h - s) mod cp; strict exactly when h < s
    cp = 4
    for h in range(cp):
        for st in rp.forward_plan(h, cp, "stripe"):
            (_, _, cls), = st.pairs
            assert (cls == rp.STRICT) == (h < st.step)


def test_ulysses_groups_and_ring_peers():
    cp, ud = 4, 2
    assert rp.ulysses_group(5, ud) == [4, 5]
    assert rp.ring_peers(5, cp, ud) == (7, 3)
    assert rp.ring_peers(7, cp, ud) == (1, 5)


# ---------------------------------------------------------------- gloo ranks

def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _inputs(S, H, D, seed):
    g = torch.Generator().manual_seed(seed)
    return [torch.randn(1, S, H, D, generator=g, dtype=torch.float64) for _ in range(4)]


def _rank_main(rank, cp, layout, port, S, H, D, results):
    from oracle import attention, layouts, merge
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=cp,
                            timeout=datetime.timedelta(seconds=60))
    try:
        q, k, v, do = (t.numpy() for t in _inputs(S, H, D, 11))
        scale = 0.3
        n = S // cp
        perm = layouts.permutation(layout, S, cp)
        mine = slice(rank * n, (rank + 1) * n)
        qn = perm[mine]                                 # natural positions of my queries
        ql, dol = (layouts.extract(t, layout, cp)[0, mine] for t in (q, do))
        kv = np.stack([layouts.extract(t, layout, cp)[0, mine] for t in (k, v)])  # [2, n, H, D]

        def vis(kown):
            return attention.visibility(qn, perm[kown * n:(kown + 1) * n], True, 0, 0)

        def exchange(st, send, shape):
            """Send `send` to st.send_to, receive the next piece from st.recv_from."""
            recv = torch.empty(shape, dtype=torch.float64)
            reqs = [dist.isend(torch.from_numpy(np.ascontiguousarray(send)), st.send_to),
                    dist.irecv(recv, st.recv_from)]
            for rq in reqs:
                rq.wait()
            return recv.numpy()

        # forward: partials of every step, merged in ring order
        plan = rp.forward_plan(rank, cp, layout)
        bufs = [kv, None]
        parts = []
        for st in plan:
            cur = bufs[st.buf]
            m = vis(st.kv_owner)
            # the plan's chunk classes say whether the step has visible pairs
            assert (m.sum() > 0) == st.has_work
            parts.append([attention.softmax_rows(ql[:, h], cur[0, :, h], cur[1, :, h], m, scale)
                          for h in range(H)])
            if st.send_to is not None:
                bufs[1 - st.buf] = exchange(st, cur, cur.shape)
        O = np.zeros((n, H, D))
        L = np.zeros((H, n))
        for h in range(H):
            O[:, h], L[h] = merge.merge_linear([p[h] for p in parts])
        # backward: dQ stays, each shard's dK/dV travels with it, then home
        plan, (home_to, home_from) = rp.backward_plan(rank, cp, layout)
        delta = np.einsum("nhd,nhd->hn", O, dol)
        dq = np.zeros_like(ql)
        bufs = [np.concatenate([kv, np.zeros_like(kv)]), None]  # [k, v, dk, dv]
        for st in plan:
            cur = bufs[st.buf]
            m = vis(st.kv_owner)
            for h in range(H):
                s_ = scale * ql[:, h] @ cur[0, :, h].T
                P = np.where(m, np.exp(s_ - L[h][:, None]), 0.0)
                dP = dol[:, h] @ cur[1, :, h].T
                dS = P * (dP - delta[h][:, None])
                dq[:, h] += scale * dS @ cur[0, :, h]
                cur[2, :, h] += scale * dS.T @ ql[:, h]
                cur[3, :, h] += P.T @ dol[:, h]
            if st.send_to is not None:
                bufs[1 - st.buf] = exchange(st, cur, cur.shape)
        last = bufs[plan[-1].buf]
        home = exchange(rp.RingStep(cp, -1, 0, home_to, home_from, ()), last[2:], last[2:].shape)
        results[rank] = (O, L, dq, home[0], home[1])
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("cp,layout", [(2, "zigzag"), (4, "zigzag"), (4, "stripe"),
                                       (4, "contiguous")])
def test_gloo_ranks_running_the_plan_reproduce_full_attention(cp, layout):
    from oracle import attention, layouts
    S, H, D = 16 * cp, 2, 8
    port = _free_port()
    results = mp.get_context("spawn").Manager().dict()
    mp.start_processes(_rank_main, args=(cp, layout, port, S, H, D, results), nprocs=cp,
                       start_method="spawn", join=True)
    q, k, v, do = (t.numpy() for t in _inputs(S, H, D, 11))
    O_ref, L_ref = attention.attn_fwd(q, k, v, 0.3, True)
    dq_ref, dk_ref, dv_ref = attention.attn_bwd(q, k, v, do, 0.3, True)
    got = [results[r] for r in range(cp)]
    cat = lambda i: np.concatenate([g[i] for g in got], axis=0)[None]  # noqa: E731
    O = layouts.restore(cat(0), layout, cp, axis=1)
    L = layouts.restore(np.concatenate([g[1] for g in got], axis=1)[None], layout, cp, axis=2)
    np.testing.assert_allclose(O, O_ref, atol=1e-12)
    np.testing.assert_allclose(L, L_ref, atol=1e-12)
    for i, ref in ((2, dq_ref), (3, dk_ref), (4, dv_ref)):
        np.testing.assert_allclose(layouts.restore(cat(i), layout, cp, axis=1), ref, atol=1e-11)

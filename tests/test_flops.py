"""The benchmark's closed-form pair counts against the oracle's brute force."""
import pytest

from oracle import attention
from sequence_long_context_gb300 import flops
from sequence_long_context_gb300.workloads import WORKLOADS, draw_cu_seqlens


@pytest.mark.parametrize("L", [1, 2, 7, 64, 300])
@pytest.mark.parametrize("causal,window,sink", [(True, 0, 0), (False, 0, 0), (True, 5, 0),
                                                (True, 5, 3), (False, 7, 2), (True, 400, 1)])
def test_pairs_closed_form(L, causal, window, sink):
    assert flops.visible_pairs_segment(L, causal, window, sink) == \
        attention.count_visible_pairs(L, causal, window, sink)


def test_pairs_varlen():
    cu = draw_cu_seqlens(3000, 1, 900, 3).tolist()
    assert flops.visible_pairs(3000, True, 50, 2, cu) == \
        attention.count_visible_pairs(3000, True, 50, 2, cu_seqlens=cu)


def test_workload_flops_match_stated_figures():
    # forward useful FLOPs of the stated workloads
    f = flops.attention_flops
    assert f(WORKLOADS["tiny_zigzag_cp4"])["fwd"] == 4 * 64 * (256 * 257 // 2) * 2
    assert abs(f(WORKLOADS["usp_ud2_ring4_s8k"])["fwd"] - 1.0996e12) < 1e9
    assert abs(f(WORKLOADS["gqa_stripe_cp8_s32k"])["fwd"] - 8.796e12) < 1e10
    assert f(WORKLOADS["swa_w1000_cp8_s8k"])["pairs_per_head"] == 7692500
    assert f(WORKLOADS["swa_w1000_sink4_cp8_s8k"])["pairs_per_head"] == 7721262

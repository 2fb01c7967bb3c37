"""A training step captured in a CUDA graph: the attention calls take their
scratch from a caller workspace, never synchronise and never allocate, so a
natural-order forward + backward (and the e4m3 forward) can be captured once
and replayed. Replays must give what the calls give when launched one by
one: out, lse, dk, dv bit for bit; dq (added into its fp32 accumulator by
the TMA unit in hardware order) to rounding."""
import pytest
import torch

import bench
import sequence_long_context_gb300 as usp
from sequence_long_context_gb300.workloads import WORKLOADS, make_inputs
from tests._gpu import device

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name,over", [
    ("tiny_zigzag_cp4", dict(S=2048, Hq=4, Hkv=2, D=128, dtype="bf16", ud=2)),
    ("tiny_zigzag_cp4", dict(S=2048, Hq=4, Hkv=4, D=128, dtype="bf16", layout="contiguous",
                             cp=2, window=300, sink_tokens=2)),
])
def test_captured_training_step_replays_exactly(name, over):
    dev = device()
    w = WORKLOADS[name].replace(B=2, **over)
    x = make_inputs(w, seed=5, with_grad=True, device="cuda")
    step = bench.make_step(usp, w, x, None)
    eager = [t.clone() for t in step(x)]
    torch.cuda.synchronize()
    # static inputs: the graph reads these buffers on every replay
    inp = {n: x[n].clone() for n in ("q", "k", "v", "dout")}
    s = torch.cuda.Stream(device=dev)
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step(inp)  # warm-up on the capture stream
    torch.cuda.current_stream().wait_stream(s)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        outs = step(inp)
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    usp.usp_device_status()
    o, dq, dk, dv = outs
    assert torch.equal(o, eager[0])
    assert torch.equal(dk, eager[2]) and torch.equal(dv, eager[3])
    err = (dq.float() - eager[1].float()).norm() / eager[1].float().norm()
    assert float(err) < 1e-2
    # new inputs copied into the static buffers are picked up by a replay
    for n in inp:
        inp[n].copy_(x[n] * 0.5)
    graph.replay()
    torch.cuda.synchronize()
    half = {n: x[n] * 0.5 for n in inp}
    ref = step(half)
    torch.cuda.synchronize()
    assert torch.equal(outs[0], ref[0]) and torch.equal(outs[3], ref[3])


def test_captured_fp8_forward_replays_exactly():
    dev = device()
    w = WORKLOADS["tiny_zigzag_cp4"].replace(B=2, S=2048, Hq=4, Hkv=2, D=128, dtype="bf16")
    x = make_inputs(w, seed=6, device="cuda")
    codes = []
    for n in "qkv":
        t = usp.permute(x[n], "extract", w.layout, w.cp)
        inv = 256.0 / float(t.float().abs().max())
        codes.append((usp.quantize_e4m3(t, inv), 1.0 / inv))
    (q8, qd), (k8, kd), (v8, vd) = codes
    ws = torch.empty(usp.usp_attn_fwd_fp8_workspace_size(w.B, w.S, w.Hq, w.Hkv, w.D, w.cp, w.ud),
                     dtype=torch.uint8, device=dev)

    def fwd():
        return usp.attn_forward_fp8(q8, k8, v8, qd, kd, vd, causal=True, cp=w.cp,
                                    layout=w.layout, workspace=ws)

    eager = [t.clone() for t in fwd()]
    s = torch.cuda.Stream(device=dev)
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fwd()
    torch.cuda.current_stream().wait_stream(s)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        out, lse = fwd()
    graph.replay()
    torch.cuda.synchronize()
    usp.usp_device_status()
    assert torch.equal(out, eager[0]) and torch.equal(lse, eager[1])

"""GPU parity of the e4m3 path: usp_quantize_e4m3 against the oracle's codes
(bit for bit) and usp_attn_fwd_fp8 against the oracle's attention of the real
values of the same codes.

Tolerance (derived from the arithmetic): the kernel rounds each probability
to an E4M3 code of 16 p before the P V product (3 mantissa bits: relative
error <= 2^-4; below 16 p = 2^-6 an absolute error <= 2^-14 in p) and the
output to bf16 (<= 2^-9 relative), with fp32 everywhere else. With A_rd =
sum_j P_rj |v_jd| (the oracle's attention of |v|), every element obeys
    |O - O_ref| <= 2^-4 A_rd + 2^-8 |O_ref| + 2e-3
(the constant covers the subnormal range and fp32 rounding). The rounding
errors have random signs, so their root mean square is far below that bound:
the test asks for RMS(err) <= RMS(bound) / 2. LSE is computed from the
unrounded fp32 probabilities: |LSE - LSE_ref| <= 1e-3.
"""
import numpy as np
import pytest
import torch

import sequence_long_context_gb300 as usp
from oracle import attention, fp8
from sequence_long_context_gb300.workloads import WORKLOADS, make_inputs
from tests._gpu import device, lse_to_natural

pytestmark = pytest.mark.gpu


def quantize(x, dev):
    """Codes and descale of a bf16 tensor, scaled so that amax maps to 256."""
    amax = float(x.float().abs().max())
    inv = 256.0 / amax
    codes = usp.quantize_e4m3(x.to(dev).contiguous(), inv)
    return codes, 1.0 / inv, inv


def check_against_oracle(w, x, q8, k8, v8, ds, out, lse, cu, heads=None):
    qd, kd, vd = ds
    unperm = lambda t: usp.permute(t, "restore", w.layout, w.cp)  # noqa: E731
    qn, kn, vn = (unperm(t).cpu().numpy() for t in (q8, k8, v8))
    O_ref, L_ref = fp8.attn_fwd_fp8(qn, kn, vn, qd, kd, vd, w.scale, w.causal, w.window,
                                    w.sink_tokens, cu_seqlens=cu, heads=heads)
    A, _ = attention.attn_fwd(fp8.dequantize(qn, qd), fp8.dequantize(kn, kd),
                              np.abs(fp8.dequantize(vn, vd)), w.scale, w.causal, w.window,
                              w.sink_tokens, cu_seqlens=cu, heads=heads)
    o = unperm(out).double().cpu().numpy()
    sel = (slice(None),) * (o.ndim - 2) + (list(heads) if heads is not None else slice(None),)
    o, O_ref, A = o[sel], O_ref[sel], A[sel]
    err = np.abs(o - O_ref)
    bound = 2.0 ** -4 * A + 2.0 ** -8 * np.abs(O_ref) + 2e-3
    assert np.isfinite(o).all()
    assert (err <= bound).all(), float((err - bound).max())
    assert np.sqrt((err ** 2).mean()) <= 0.5 * np.sqrt((bound ** 2).mean())
    lse_nat = lse_to_natural(lse.double().cpu().numpy(), w)
    lsel = lse_nat if heads is None else lse_nat[..., list(heads), :]
    lref = L_ref if heads is None else L_ref[..., list(heads), :]
    fin = np.isfinite(lref)
    assert np.array_equal(fin, np.isfinite(lsel))
    assert np.abs(lsel[fin] - lref[fin]).max() <= 1e-3


def test_quantize_matches_oracle_codes_bit_for_bit():
    dev = device()
    g = torch.Generator().manual_seed(5)
    x = (torch.randn(3, 1001, 7, generator=g) * 40).to(torch.bfloat16)  # tail of 5
    x.view(-1)[:6] = torch.tensor([0.0, -0.0, 1e30, -1e30, float("nan"), 3.0e-3],
                                  dtype=torch.bfloat16)
    for inv in (1.0, 3.7, 1.0 / 64):
        got = usp.quantize_e4m3(x.to(dev), inv).cpu().numpy()
        ref = fp8.quantize(x.float().numpy(), inv)
        assert np.array_equal(got, ref)


CASES = [
    dict(layout="zigzag", cp=4, S=2048, Hq=4, Hkv=4),
    dict(layout="stripe", cp=2, S=2048, Hq=8, Hkv=2),
    dict(layout="contiguous", cp=2, S=1024, Hq=4, Hkv=2, window=300, sink_tokens=3),
    dict(layout="zigzag", cp=2, S=1024, Hq=4, Hkv=1, causal=False),
    dict(layout="zigzag", cp=2, S=2048, Hq=4, Hkv=2, ud=2),
    # 128-token zigzag chunks and stripe shards: one query tile per chunk
    dict(layout="zigzag", cp=4, S=1024, Hq=4, Hkv=2),
    dict(layout="stripe", cp=4, S=512, Hq=4, Hkv=2),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "-".join(f"{k}{v}" for k, v in c.items()))
def test_fp8_forward_matches_oracle(case):
    dev = device()
    w = WORKLOADS["tiny_zigzag_cp4"].replace(B=2, D=128, dtype="bf16", **case)
    x = make_inputs(w, seed=31)
    perm = lambda t: usp.permute(t.to(dev), "extract", w.layout, w.cp)  # noqa: E731
    (q8, qd, _), (k8, kd, _), (v8, vd, _) = (quantize(perm(x[n]), dev) for n in "qkv")
    out, lse = usp.attn_forward_fp8(q8, k8, v8, qd, kd, vd, causal=w.causal, window=w.window,
                                    sink_tokens=w.sink_tokens, cp=w.cp, ud=w.ud,
                                    layout=w.layout)
    check_against_oracle(w, x, q8, k8, v8, (qd, kd, vd), out, lse, None)


def test_fp8_varlen_with_window_and_sinks():
    dev = device()
    w = WORKLOADS["tiny_zigzag_cp4"].replace(B=0, S=2048, Hq=4, Hkv=2, D=128, dtype="bf16",
                                              cp=2, layout="zigzag", varlen=True, seg_lo=1,
                                              seg_hi=700, window=300, sink_tokens=2)
    x = make_inputs(w, seed=37)
    cu = x["cu_seqlens"]
    perm = lambda t: usp.permute(t.to(dev), "extract", w.layout, w.cp)  # noqa: E731
    (q8, qd, _), (k8, kd, _), (v8, vd, _) = (quantize(perm(x[n]), dev) for n in "qkv")
    out, lse = usp.attn_forward_fp8(q8, k8, v8, qd, kd, vd, causal=True, window=w.window,
                                    sink_tokens=w.sink_tokens, cu_seqlens=cu.to(dev),
                                    cp=w.cp, layout=w.layout)
    check_against_oracle(w, x, q8, k8, v8, (qd, kd, vd), out, lse, cu)


def test_fp8_ulysses_is_bit_identical_to_plain_ring():
    dev = device()
    w = WORKLOADS["tiny_zigzag_cp4"].replace(B=1, S=2048, Hq=8, Hkv=4, D=128, dtype="bf16",
                                              cp=2, layout="zigzag")
    x = make_inputs(w, seed=41)
    perm = lambda t: usp.permute(t.to(dev), "extract", w.layout, w.cp)  # noqa: E731
    (q8, qd, _), (k8, kd, _), (v8, vd, _) = (quantize(perm(x[n]), dev) for n in "qkv")
    kw = dict(causal=True, cp=w.cp, layout=w.layout)
    o1, l1 = usp.attn_forward_fp8(q8, k8, v8, qd, kd, vd, ud=1, **kw)
    o2, l2 = usp.attn_forward_fp8(q8, k8, v8, qd, kd, vd, ud=2, **kw)
    o4, l4 = usp.attn_forward_fp8(q8, k8, v8, qd, kd, vd, ud=4, **kw)
    assert torch.equal(o1, o2) and torch.equal(o1, o4)
    assert torch.equal(l1, l2) and torch.equal(l1, l4)


def test_fp8_rejections():
    dev = device()
    z = torch.zeros(1, 512, 2, 64, dtype=torch.uint8, device=dev)
    with pytest.raises(usp.UspError, match="UNSUPPORTED"):
        usp.attn_forward_fp8(z, z, z, 1.0, 1.0, 1.0, cp=1)          # D = 64
    z = torch.zeros(1, 512, 2, 128, dtype=torch.uint8, device=dev)
    with pytest.raises(usp.UspError, match="INVALID_ARG"):
        usp.attn_forward_fp8(z, z, z, 0.0, 1.0, 1.0, cp=1)          # descale 0
    with pytest.raises(usp.UspError, match="UNSUPPORTED"):
        usp.attn_forward_fp8(z, z, z, 1.0, 1.0, 1.0, cp=8)          # 64-token shards


def test_fp8_full_size_sampled_rows():
    # the bench's fp8 workload (S = 32K zigzag ring of 8, 32 query / 8 KV
    # heads) in the launch configuration it times, checked on sampled rows
    dev = device()
    w = WORKLOADS["sweep_zigzag_cp8_s32k"]
    x = make_inputs(w, seed=0, device=str(dev))
    perm = lambda t: usp.permute(t, "extract", w.layout, w.cp)  # noqa: E731
    (q8, qd, _), (k8, kd, _), (v8, vd, _) = (quantize(perm(x[n]), dev) for n in "qkv")
    out, lse = usp.attn_forward_fp8(q8, k8, v8, qd, kd, vd, causal=True, cp=w.cp,
                                    layout=w.layout)
    unperm = lambda t: usp.permute(t, "restore", w.layout, w.cp)  # noqa: E731
    on = unperm(out)
    g = np.random.default_rng(7)
    rows = sorted(set(g.integers(0, w.S, 24).tolist()) | {0, 1, w.S - 1})
    heads = (0, 13, 31)
    # only the sampled query rows and the KV heads they read are needed
    qs = fp8.dequantize(unperm(q8)[:, rows][:, :, list(heads)].cpu().numpy(), qd)
    kr = fp8.dequantize(unperm(k8)[:, :, [h // (w.Hq // w.Hkv) for h in heads]].cpu().numpy(), kd)
    vr = fp8.dequantize(unperm(v8)[:, :, [h // (w.Hq // w.Hkv) for h in heads]].cpu().numpy(), vd)
    for n, h in enumerate(heads):
        # rows of qs are the sampled ones: place them at their positions
        qf = np.zeros((1, w.S, 1, w.D))
        qf[0, rows, 0] = qs[0, :, n]
        kk, vv = kr[:, :, n:n + 1], vr[:, :, n:n + 1]
        o_ref, _ = attention.attn_fwd_rows(qf, kk, vv, w.scale, 0, 0, rows, causal=True)
        a_ref, _ = attention.attn_fwd_rows(qf, kk, np.abs(vv), w.scale, 0, 0, rows,
                                           causal=True)
        got = on[0, rows, h].double().cpu().numpy()
        bound = 2.0 ** -4 * a_ref + 2.0 ** -8 * np.abs(o_ref) + 2e-3
        assert (np.abs(got - o_ref) <= bound).all()

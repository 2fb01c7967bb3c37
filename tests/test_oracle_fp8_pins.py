"""Pins for the fp8 oracle (oracle/fp8.py), on the CPU.

E4M3 codes are tied to torch's float8_e4m3fn conversion (a library routine)
inside the range where both saturate alike, and to closed forms of the
format (largest finite value, smallest subnormal, ties to the even code,
saturation, NaN). The attention of e4m3 inputs is tied to a case whose
answer is known without the oracle (constant values) and to the bf16 / fp64
attention of the same real values; planted mistakes must fail.
"""
import math

import numpy as np
import pytest
import torch

from oracle import attention, fp8


def test_decode_matches_torch_for_every_code():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = fp8.e4m3_decode(codes)
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])


def test_encode_matches_torch_below_the_saturation_point():
    g = np.random.default_rng(0)
    x = np.concatenate([
        g.standard_normal(20000) * s for s in (1e-3, 0.05, 1.0, 30.0, 150.0)] + [
        # every midpoint between neighbouring codes (the ties) and the codes
        (fp8._MAG[1:] + fp8._MAG[:-1]) / 2, fp8._MAG, -fp8._MAG])
    x = x[np.abs(x) < 464.0].astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(fp8.e4m3_encode(x), ref)


def test_closed_forms():
    enc = fp8.e4m3_encode
    assert fp8.e4m3_decode(np.uint8(0x7E)) == 448.0
    assert fp8.e4m3_decode(np.uint8(0x01)) == 2.0 ** -9          # smallest subnormal
    assert fp8.e4m3_decode(np.uint8(0x08)) == 2.0 ** -6          # smallest normal
    assert fp8.e4m3_decode(np.uint8(0x38)) == 1.0
    assert enc(448.0) == 0x7E and enc(-448.0) == 0xFE
    assert enc(1e6) == 0x7E and enc(-1e6) == 0xFE and enc(470.0) == 0x7E  # saturate
    assert (enc(np.nan) & 0x7F) == 0x7F
    assert enc(2.0 ** -10) == 0x00           # tie between 0 and 2^-9: even code 0
    assert enc(3 * 2.0 ** -10) == 0x02       # tie between 2^-9 and 2^-8: even code 2
    assert enc(1.0625) == 0x38               # tie between 1 and 1.125: even code 0x38
    assert enc(1.1875) == 0x3A               # tie between 1.125 and 1.25: even code 0x3A
    assert enc(0.0) == 0x00 and enc(-0.0) == 0x80


def test_round_trip_error_bound():
    # |decode(encode(x)) - x| <= 2^-4 |x| in the normal range, <= 2^-10 below
    g = np.random.default_rng(1)
    x = g.standard_normal(50000) * 20.0
    x = x[np.abs(x) < 448.0]
    err = np.abs(fp8.e4m3_decode(fp8.e4m3_encode(x)) - x)
    bound = np.where(np.abs(x) >= 2.0 ** -6, 2.0 ** -4 * np.abs(x), 2.0 ** -10)
    assert (err <= bound + 1e-300).all()


def test_quantize_takes_the_product_in_fp32():
    x = np.array([1.0 / 3.0, 7.3, -0.011], dtype=np.float32)
    inv = 13.7
    prod = (x * np.float32(inv)).astype(np.float32)
    assert np.array_equal(fp8.quantize(x, inv), fp8.e4m3_encode(prod))
    ref = torch.from_numpy(prod).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(fp8.quantize(x, inv), ref)


def test_attention_of_constant_values():
    # every visible value row is the same vector: O is that vector exactly
    B, S, Hq, Hkv, D = 1, 40, 4, 2, 16
    g = np.random.default_rng(2)
    q8 = fp8.e4m3_encode(g.standard_normal((B, S, Hq, D)))
    k8 = fp8.e4m3_encode(g.standard_normal((B, S, Hkv, D)))
    row = fp8.e4m3_encode(g.standard_normal(D))
    v8 = np.broadcast_to(row, (B, S, Hkv, D)).copy()
    O, L = fp8.attn_fwd_fp8(q8, k8, v8, 0.5, 0.25, 2.0, 0.3, causal=True, window=7,
                            sink_tokens=2)
    np.testing.assert_allclose(O, np.broadcast_to(fp8.e4m3_decode(row) * 2.0, O.shape),
                               atol=1e-12, rtol=0)
    # LSE of row 0 (only key 0 visible): s = scale * <q, k> in real values
    s00 = 0.3 * float((fp8.e4m3_decode(q8[0, 0, 0]) * 0.5) @ (fp8.e4m3_decode(k8[0, 0, 0]) * 0.25))
    assert math.isclose(L[0, 0, 0], s00, abs_tol=1e-12)


def test_attention_equals_torch_sdpa_of_the_real_values():
    B, S, Hq, Hkv, D = 2, 48, 4, 1, 32
    g = np.random.default_rng(3)
    q8, k8, v8 = (fp8.quantize(g.standard_normal(sh), 4.0) for sh in
                  ((B, S, Hq, D), (B, S, Hkv, D), (B, S, Hkv, D)))
    O, _ = fp8.attn_fwd_fp8(q8, k8, v8, 0.25, 0.25, 0.25, 0.2, causal=True)
    qt, kt, vt = (torch.from_numpy(fp8.e4m3_decode(t) * 0.25).transpose(1, 2)
                  for t in (q8, k8, v8))
    kt, vt = kt.repeat_interleave(Hq // Hkv, 1), vt.repeat_interleave(Hq // Hkv, 1)
    ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, is_causal=True,
                                                           scale=0.2)
    np.testing.assert_allclose(O, ref.transpose(1, 2).numpy(), atol=1e-12, rtol=0)


def test_planted_mistakes_fail(monkeypatch):
    # ties away from zero instead of to even
    x = np.array([3 * 2.0 ** -10, 1.0625], dtype=np.float32)
    away = np.where(x > 0, np.array([0x02 + 1, 0x39]), 0)
    assert not np.array_equal(fp8.e4m3_encode(x), away)
    # a descale applied to the wrong tensor changes the result
    B, S, H, D = 1, 16, 1, 8
    g = np.random.default_rng(4)
    q8, k8, v8 = (fp8.e4m3_encode(g.standard_normal((B, S, H, D))) for _ in range(3))
    good, _ = fp8.attn_fwd_fp8(q8, k8, v8, 1.0, 0.5, 2.0, 0.3)
    swapped, _ = fp8.attn_fwd_fp8(q8, k8, v8, 1.0, 2.0, 0.5, 0.3)
    assert np.abs(good - swapped).max() > 1e-3
    # a decode that drops the subnormals is caught by the torch pin
    real = fp8._MAG.copy()
    monkeypatch.setattr(fp8, "_MAG", np.where(np.arange(real.size) < 8, 0.0, real))
    codes = np.arange(1, 8, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert not np.array_equal(fp8.e4m3_decode(codes), ref)

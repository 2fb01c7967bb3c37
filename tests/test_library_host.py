"""Host-side checks of the C ABI (no GPU): the library loads, exports every
symbol include/usp.h declares, and rejects invalid arguments before any
launch."""
import ctypes
import os
import re

import pytest
import torch

import __graft_entry__
import sequence_long_context_gb300 as usp
from sequence_long_context_gb300 import _lib

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "usp.h")


@pytest.fixture(scope="module")
def lib():
    __graft_entry__.build()
    return _lib.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(usp_[a-z_0-9]+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert len(names) >= 8
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(_lib.SIGNATURES) == names


def test_status_strings(lib):
    for code, name in enumerate(["USP_OK", "USP_ERR_INVALID_ARG", "USP_ERR_UNSUPPORTED",
                                 "USP_ERR_ALIGNMENT", "USP_ERR_WORKSPACE", "USP_ERR_CUDA",
                                 "USP_ERR_TIMEOUT"]):
        assert lib.usp_status_string(code).decode() == name


def test_workspace_sizes(lib):
    # ud=1 forward needs no scratch; ud=2 holds q,k,v,o in head-grouped form
    assert usp.usp_attn_fwd_workspace_size(2, 8192, 32, 32, 128, 4, 1, 0) == 0
    n = usp.usp_attn_fwd_workspace_size(2, 8192, 32, 32, 128, 4, 2, 0)
    assert n == 4 * 2 * 8192 * 32 * 128 * 2
    b = usp.usp_attn_bwd_workspace_size(1, 1024, 8, 2, 64, 2, 1, 1)
    assert b >= 8 * 1024 * 4


FAKE = 1 << 20  # a 16-byte aligned non-null address; never dereferenced


def fwd(lib, **over):
    a = dict(q=FAKE, k=FAKE, v=FAKE, out=FAKE, lse=FAKE, B=1, S=256, Hq=4, Hkv=2,
             D=64, scale=0.0, causal=1, window=0, sink=0, cu=None, cp=4, ud=1,
             layout=1, dtype=1, flags=0, ws=None, wsb=0, stream=None)
    a.update(over)
    return lib.usp_attn_fwd(a["q"], a["k"], a["v"], a["out"], a["lse"], a["B"], a["S"],
                            a["Hq"], a["Hkv"], a["D"], a["scale"], a["causal"],
                            a["window"], a["sink"], a["cu"], a["cp"], a["ud"],
                            a["layout"], a["dtype"], a["flags"], a["ws"], a["wsb"],
                            a["stream"])


@pytest.mark.parametrize("over,code", [
    (dict(Hq=3), 1),               # Hq % Hkv
    (dict(S=250), 1),              # zigzag needs S % (2 cp) == 0
    (dict(layout=0, S=254), 1),    # contiguous needs S % cp == 0
    (dict(D=96), 2),               # head dim not supported
    (dict(cp=0), 1),
    (dict(ud=4), 1),               # Hkv=2 not divisible by ud=4
    (dict(layout=7), 1),
    (dict(sink=-1), 1),
    (dict(q=FAKE + 8), 3),         # misaligned
    (dict(q=None), 1),             # null tensor
    (dict(ud=2), 4),               # Ulysses needs workspace
])
def test_fwd_rejects_before_launch(lib, over, code):
    assert fwd(lib, **over) == code


def test_permute_and_merge_reject(lib):
    # elem_bytes, layout, divisibility, alignment
    assert lib.usp_permute(FAKE, FAKE, 0, 1, 1, 100, 2, 64, 4, 1, 3, None) == 1
    # 1-byte codes: the row (H*D bytes) must still be a multiple of 16
    assert lib.usp_permute(FAKE, FAKE, 0, 1, 1, 128, 1, 8, 4, 1, 1, None) == 1
    assert lib.usp_permute(FAKE, FAKE, 0, 9, 1, 128, 2, 64, 4, 1, 2, None) == 1
    assert lib.usp_permute(FAKE, FAKE, 0, 1, 1, 100, 2, 64, 4, 1, 2, None) == 1
    assert lib.usp_permute(FAKE + 4, FAKE, 0, 1, 1, 128, 2, 64, 4, 1, 2, None) == 3
    assert lib.usp_permute(FAKE, FAKE, 2, 1, 1, 128, 3, 64, 4, 2, 2, None) == 1
    assert lib.usp_merge_partials(FAKE, FAKE, 0, 10, 128, 0, FAKE, 1, FAKE, None) == 1
    assert lib.usp_merge_partials(FAKE, FAKE, 65, 10, 128, 1, FAKE, 1, FAKE, None) == 1
    assert lib.usp_merge_partials(FAKE, FAKE, 2, 10, 96, 0, FAKE, 1, FAKE, None) == 1
    assert lib.usp_merge_partials(FAKE, FAKE + 4, 2, 10, 128, 0, FAKE, 1, FAKE, None) == 3


def test_empty_problem_is_a_no_op(lib):
    # S == 0 validates and returns OK without touching the device
    assert fwd(lib, S=0, q=None, k=None, v=None, out=None, lse=None) == 0


def test_python_binding_raises(lib):
    with pytest.raises(usp.UspError, match="USP_ERR_INVALID_ARG"):
        usp._check(1)


def decode(lib, **over):
    a = dict(q=FAKE, k=FAKE, v=FAKE, out=FAKE, lse=FAKE, B=2, Tq=1, S=1024, Hq=8,
             Hkv=2, D=128, scale=0.0, causal=1, cp=4, splits=2, tree=1, dtype=0,
             ws=FAKE, wsb=1 << 30, stream=None)
    a.update(over)
    return lib.usp_attn_decode(a["q"], a["k"], a["v"], a["out"], a["lse"], a["B"],
                               a["Tq"], a["S"], a["Hq"], a["Hkv"], a["D"], a["scale"],
                               a["causal"], a["cp"], a["splits"], a["tree"], a["dtype"],
                               a["ws"], a["wsb"], a["stream"])


@pytest.mark.parametrize("over,code", [
    (dict(Hq=7), 1),                  # Hq % Hkv
    (dict(Tq=5), 2),                  # G * Tq = 20 rows > 16
    (dict(S=1000), 1),                # S % (cp * splits)
    (dict(S=256), 1),                 # pieces of 32 keys, not a multiple of 64
    (dict(D=96), 1),
    (dict(dtype=1), 2),               # fp32 cache: unsupported
    (dict(cp=16, splits=8, S=8192), 1),  # tree order over more than 64 partials
    (dict(q=FAKE + 4), 3),
    (dict(ws=None), 4),               # no workspace
    (dict(wsb=16), 4),                # workspace too small
    (dict(Tq=2000), 1),               # more new tokens than cached keys
])
def test_decode_rejects_before_launch(lib, over, code):
    assert decode(lib, **over) == code


def test_decode_workspace_and_empty_batch(lib):
    n = usp.usp_attn_decode_workspace_size(2, 1, 1024, 8, 2, 128, 4, 2)
    rows = 2 * 1 * 8
    assert n >= 8 * rows * 128 * 4 + 8 * rows * 4
    assert decode(lib, B=0, q=None, k=None, v=None, out=None, lse=None) == 0


def test_selftest_rejects_limits(lib):
    assert lib.usp_selftest_wait_timeout(0, None) == 1
    assert lib.usp_selftest_wait_timeout(2_000_000, None) == 1


def test_packed_entry_points_reject_before_launch(lib):
    # H = 0, a misaligned packed tensor, a missing workspace under Ulysses
    assert lib.usp_attn_fwd_qkvpacked(FAKE, FAKE, FAKE, 1, 256, 0, 64, 0.0, 1, 0, 0, None, 4, 1,
                                      1, 1, 0, None, 0, None) == 1
    assert lib.usp_attn_fwd_qkvpacked(FAKE + 8, FAKE, FAKE, 1, 256, 2, 64, 0.0, 1, 0, 0, None, 4,
                                      1, 1, 1, 0, None, 0, None) == 3
    assert lib.usp_attn_fwd_qkvpacked(FAKE, FAKE, FAKE, 1, 256, 2, 64, 0.0, 1, 0, 0, None, 2, 2,
                                      1, 1, 0, None, 0, None) == 4
    assert lib.usp_attn_bwd_qkvpacked(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 256, 2, 64, 0.0, 1, 0, 0,
                                      None, 4, 1, 1, 1, 0, None, 0, None) == 4


def bwd(lib, **over):
    a = dict(q=FAKE, k=FAKE, v=FAKE, out=FAKE, lse=FAKE, dout=FAKE, dq=FAKE, dk=FAKE, dv=FAKE,
             B=1, S=256, Hq=4, Hkv=2, D=64, scale=0.0, causal=1, window=0, sink=0, cu=None,
             cp=2, ud=2, layout=1, dtype=1, flags=0, ws=None, wsb=0, stream=None)
    a.update(over)
    return lib.usp_attn_bwd(a["q"], a["k"], a["v"], a["out"], a["lse"], a["dout"], a["dq"],
                            a["dk"], a["dv"], a["B"], a["S"], a["Hq"], a["Hkv"], a["D"],
                            a["scale"], a["causal"], a["window"], a["sink"], a["cu"], a["cp"],
                            a["ud"], a["layout"], a["dtype"], a["flags"], a["ws"], a["wsb"],
                            a["stream"])


def test_saved_exchange_flag_host_checks(lib):
    F = usp.FLAG_SAVED_EXCHANGE
    none = dict(q=None, k=None, v=None, out=None)
    # with the flag under Ulysses, q/k/v/out are not needed: the call gets as
    # far as the (missing) workspace
    assert bwd(lib, flags=F, **none) == 4
    # without Ulysses the flag does nothing, so the null tensors are an error
    assert bwd(lib, flags=F, ud=1, **none) == 1
    assert bwd(lib, flags=0, **none) == 1
    # the no-alloc call has no forward workspace to read from
    st = lib.usp_attn_bwd_noalloc(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                                  1, 256, 4, 2, 64, 0.0, 1, 0, 0, None, 2, 2, 1, 1, F, None)
    assert st == 1
    assert b"SAVED_EXCHANGE" in lib.usp_last_error_detail()


@pytest.mark.parametrize("B,S,Hq,Hkv,D,cp,ud,dtype", [
    (2, 8192, 32, 32, 128, 4, 2, 1), (1, 4096, 32, 8, 128, 2, 4, 1), (1, 512, 4, 2, 64, 2, 2, 0),
    (3, 1000, 8, 8, 64, 1, 8, 0)])
def test_backward_workspace_holds_the_forward_exchange(lib, B, S, Hq, Hkv, D, cp, ud, dtype):
    # the saved-exchange flag relies on the forward's workspace being a
    # prefix of the backward's (same q, k, v, o slices at the same offsets)
    f = usp.usp_attn_fwd_workspace_size(B, S, Hq, Hkv, D, cp, ud, dtype)
    b = usp.usp_attn_bwd_workspace_size(B, S, Hq, Hkv, D, cp, ud, dtype)
    el = 2 if dtype == 0 else 4
    assert f == 2 * B * S * (Hq + Hkv) * D * el
    assert b >= f


def test_python_saved_exchange_needs_the_workspace():
    q = torch.zeros(1, 256, 4, 64, dtype=torch.bfloat16)
    k = torch.zeros(1, 256, 2, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        usp.attn_backward(q, k, k, q, None, q, cp=2, ud=2, saved_exchange=True)


def fp8_fwd(lib, **over):
    # zigzag, ring of 2, S = 1024: 256-token chunks (the kernel takes multiples of 128)
    a = dict(q=FAKE, k=FAKE, v=FAKE, qd=1.0, kd=1.0, vd=1.0, out=FAKE, lse=FAKE, B=1, S=1024,
             Hq=4, Hkv=2, D=128, scale=0.0, causal=1, window=0, sink=0, cu=None, cp=2, ud=1,
             layout=1, flags=0, ws=None, wsb=0, stream=None)
    a.update(over)
    return lib.usp_attn_fwd_fp8(a["q"], a["k"], a["v"], a["qd"], a["kd"], a["vd"], a["out"],
                                a["lse"], a["B"], a["S"], a["Hq"], a["Hkv"], a["D"], a["scale"],
                                a["causal"], a["window"], a["sink"], a["cu"], a["cp"], a["ud"],
                                a["layout"], a["flags"], a["ws"], a["wsb"], a["stream"])


@pytest.mark.parametrize("over,code", [
    (dict(), 4),                    # the V^T scratch is always needed
    (dict(D=64), 2),                # head dim 128 only
    (dict(qd=0.0), 1), (dict(vd=-1.0), 1), (dict(kd=float("inf")), 1),
    (dict(q=FAKE + 8), 3),
    (dict(v=None), 1),
    (dict(cp=8), 2),                # 64-token chunks are below the 128-token tile
    (dict(Hq=3), 1),
])
def test_fp8_forward_rejects_before_launch(lib, over, code):
    assert fp8_fwd(lib, **over) == code


def test_fp8_workspace_and_quantize_checks(lib):
    # V^T always; with Ulysses also the e4m3 head groups and the bf16 output
    assert usp.usp_attn_fwd_fp8_workspace_size(2, 1024, 8, 2, 128, 2, 1) == 2 * 1024 * 2 * 128
    assert usp.usp_attn_fwd_fp8_workspace_size(2, 1024, 8, 2, 128, 2, 2) == \
        2 * 1024 * 128 * (2 + 8 + 2 + 2 + 2 * 8)
    assert usp.usp_attn_fwd_fp8_workspace_size(-1, 1024, 8, 2, 128, 2, 1) == 0
    assert lib.usp_quantize_e4m3(FAKE, FAKE, -1, 1.0, None) == 1
    assert lib.usp_quantize_e4m3(None, FAKE, 16, 1.0, None) == 1
    assert lib.usp_quantize_e4m3(FAKE, FAKE, 16, float("inf"), None) == 1
    assert lib.usp_quantize_e4m3(FAKE + 4, FAKE, 16, 1.0, None) == 3
    assert lib.usp_quantize_e4m3(FAKE, FAKE, 0, 1.0, None) == 0  # nothing to do


@pytest.mark.parametrize("over,code", [
    (dict(B=-1), 1), (dict(Hq=3), 1), (dict(D=96), 2), (dict(S=255), 1), (dict(cp=0), 1),
    (dict(q=FAKE + 8), 3)])
def test_noalloc_checks_arguments_first(lib, over, code):
    # argument errors come back as usp_attn_bwd reports them, before the
    # scratch array is looked up (no device is needed to get them)
    a = dict(q=FAKE, B=1, S=256, Hq=4, D=64, cp=2)
    a.update(over)
    st = lib.usp_attn_bwd_noalloc(a["q"], FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                                  a["B"], a["S"], a["Hq"], 2, a["D"], 0.0, 1, 0, 0, None,
                                  a["cp"], 1, 1, 0, 0, None)
    assert st == code, lib.usp_status_string(st)


def test_natural_order_flag_host_checks(lib):
    N = usp.FLAG_NATURAL_ORDER
    # ud = 1: the kernels' rank-major copies of q, k, v, out need scratch
    assert usp.usp_attn_fwd_workspace_size(2, 8192, 32, 8, 128, 4, 1, 0) == 0
    assert usp.usp_attn_fwd_workspace_size(2, 8192, 32, 8, 128, 4, 1, 0, N) == \
        2 * 2 * 8192 * (32 + 8) * 128 * 2
    # ud > 1: the exchange buffers serve as those copies, no extra scratch
    for fn in (usp.usp_attn_fwd_workspace_size, usp.usp_attn_bwd_workspace_size):
        assert fn(2, 8192, 32, 8, 128, 4, 2, 0, N) == fn(2, 8192, 32, 8, 128, 4, 2, 0)
    # the backward's scratch still starts with the forward's (saved copies)
    assert usp.usp_attn_bwd_workspace_size(1, 4096, 8, 2, 64, 2, 1, 1, N) >= \
        usp.usp_attn_fwd_workspace_size(1, 4096, 8, 2, 64, 2, 1, 1, N)
    # ud = 1 with the flag: the call gets as far as the missing workspace
    assert fwd(lib, flags=N) == 4
    assert bwd(lib, ud=1, flags=N) == 4
    # natural-order backward calls may read q, k, v, out in place: they are
    # needed even with the saved-exchange flag
    assert bwd(lib, ud=1, flags=N | usp.FLAG_SAVED_EXCHANGE, q=None, k=None, v=None,
               out=None) == 1
    assert bwd(lib, flags=N | usp.FLAG_SAVED_EXCHANGE, q=None, k=None, v=None,
               out=None) == 1
    # the packed entry points and the e4m3 forward do not take it
    assert lib.usp_attn_fwd_qkvpacked(FAKE, FAKE, FAKE, 1, 256, 2, 64, 0.0, 1, 0, 0, None, 4,
                                      1, 1, 1, N, None, 0, None) == 2
    assert lib.usp_attn_bwd_qkvpacked(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 256, 2, 64, 0.0, 1, 0,
                                      0, None, 4, 1, 1, 1, N, None, 0, None) == 2
    assert fp8_fwd(lib, flags=N) == 2


@pytest.mark.parametrize("cu,total,ok,detail", [
    ([0, 128], 128, True, None),
    ([0, 100, 100, 512], 512, True, None),   # an empty sequence is allowed
    ([0, 0], 0, True, None),
    ([1, 128], 128, False, b"cu_seqlens[0]"),
    ([0, 300, 200, 512], 512, False, b"cu_seqlens[2] = 200"),
    ([0, 100, 500], 512, False, b"not the 512 tokens"),
    ([0, 100, 600], 512, False, b"not the 512 tokens"),
])
def test_check_cu_seqlens(lib, cu, total, ok, detail):
    arr = (ctypes.c_int32 * len(cu))(*cu)
    st = lib.usp_check_cu_seqlens(ctypes.addressof(arr), len(cu) - 1, total)
    assert st == (0 if ok else 1)
    if detail is not None:
        assert detail in lib.usp_last_error_detail()
    t = torch.tensor(cu, dtype=torch.int32)
    if ok:
        usp.check_cu_seqlens(t, total)
    else:
        with pytest.raises(usp.UspError, match="INVALID_ARG"):
            usp.check_cu_seqlens(t, total)


def test_check_cu_seqlens_rejects_bad_arguments(lib):
    arr = (ctypes.c_int32 * 2)(0, 8)
    assert lib.usp_check_cu_seqlens(None, 1, 8) == 1
    assert lib.usp_check_cu_seqlens(ctypes.addressof(arr), 0, 8) == 1
    assert lib.usp_check_cu_seqlens(ctypes.addressof(arr), 1, -1) == 1
    with pytest.raises(usp.UspError):
        usp.check_cu_seqlens(torch.tensor([0], dtype=torch.int32), 0)

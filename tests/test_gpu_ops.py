"""GPU parity of the permute (bit-exact) and merge kernels against the oracle."""
import numpy as np
import pytest
import torch

import sequence_long_context_gb300 as usp
from oracle import layouts, merge
from tests._gpu import device

pytestmark = pytest.mark.gpu


def bits(t: torch.Tensor) -> np.ndarray:
    t = t.detach().cpu()
    return t.view(torch.int16 if t.element_size() == 2 else torch.int32).numpy()


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("layout", ["contiguous", "zigzag", "stripe"])
@pytest.mark.parametrize("cp", [1, 2, 3, 4, 8])
def test_extract_restore_bit_exact(dtype, layout, cp):
    dev = device()
    B, S, H, D = 2, 2 * cp * 24, 4, 64
    g = torch.Generator().manual_seed(cp)
    x = torch.randn(B, S, H, D, generator=g).to(dtype)
    y = usp.permute(x.to(dev), "extract", layout, cp)
    want = layouts.extract(bits(x), layout, cp, axis=1)
    assert np.array_equal(bits(y), want)
    z = usp.permute(y, "restore", layout, cp)
    assert np.array_equal(bits(z), bits(x))


def test_extract_packed_sequence():
    dev = device()
    T, H, D, cp = 8 * 2 * 40, 3, 128, 8
    x = torch.randn(T, H, D, generator=torch.Generator().manual_seed(5)).to(torch.bfloat16)
    y = usp.permute(x.to(dev), "extract", "zigzag", cp)
    assert np.array_equal(bits(y), layouts.extract(bits(x), "zigzag", cp, axis=0))


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("cp,ud", [(1, 2), (4, 2), (2, 4), (3, 2)])
def test_ulysses_bit_exact(dtype, cp, ud):
    dev = device()
    B, S, H, D = 2, cp * ud * 16, 8, 128
    x = torch.randn(B, S, H, D, generator=torch.Generator().manual_seed(ud)).to(dtype)
    y = usp.permute(x.to(dev), "seq2head", cp=cp, ud=ud)
    assert np.array_equal(bits(y), layouts.ulysses_seq2head(bits(x), cp, ud))
    z = usp.permute(y, "head2seq", cp=cp, ud=ud)
    assert np.array_equal(bits(z), bits(x))


def _partials(n, rows, D, seed):
    g = torch.Generator().manual_seed(seed)
    o = torch.randn(n, rows, D, generator=g)
    lse = torch.randn(n, rows, generator=g) * 4
    if n > 1:
        lse[1, ::7] = -float("inf")
        o[1, ::7] = float("nan")  # an empty partial's O must never be read
    lse[:, 5] = -float("inf")     # a row empty in every partial
    return o, lse


@pytest.mark.parametrize("n", [1, 2, 3, 4, 5, 6, 7, 8, 9, 17, 64])
@pytest.mark.parametrize("tree", [False, True])
@pytest.mark.parametrize("D", [64, 128])
def test_merge_matches_oracle(n, tree, D):
    dev = device()
    rows = 1000
    o, lse = _partials(n, rows, D, n * 3 + D)
    oo, ll = usp.merge_partials(o.to(dev), lse.to(dev), tree_order=tree)
    parts = [(np.nan_to_num(o[i].double().numpy()), lse[i].double().numpy()) for i in range(n)]
    O, L = (merge.merge_tree if tree else merge.merge_linear)(parts)
    got_o, got_l = oo.cpu().double().numpy(), ll.cpu().double().numpy()
    fin = np.isfinite(L)
    assert np.array_equal(np.isneginf(got_l), ~fin)
    np.testing.assert_allclose(got_l[fin], L[fin], rtol=1e-5, atol=1e-5)
    np.testing.assert_allclose(got_o[fin], O[fin], rtol=1e-5, atol=1e-5)
    assert np.all(got_o[~fin] == 0)


def test_merge_bf16_output():
    dev = device()
    o, lse = _partials(4, 513, 128, 1)
    oo, ll = usp.merge_partials(o.to(dev), lse.to(dev), out_dtype=torch.bfloat16)
    parts = [(np.nan_to_num(o[i].double().numpy()), lse[i].double().numpy()) for i in range(4)]
    O, _ = merge.merge_linear(parts)
    np.testing.assert_allclose(oo.cpu().double().numpy(), O, atol=2e-2)


def _merge_check_all_rows(oo, ll, o, lse, tree, rtol_o):
    """Every output row against the oracle, in row chunks (rows are independent)."""
    n, rows = lse.shape
    fn = merge.merge_tree if tree else merge.merge_linear
    step = 1 << 15
    for r0 in range(0, rows, step):
        r1 = min(rows, r0 + step)
        parts = [(np.nan_to_num(o[i, r0:r1].double().numpy()), lse[i, r0:r1].double().numpy())
                 for i in range(n)]
        O, L = fn(parts)
        got_o = oo[r0:r1].double().numpy()
        got_l = ll[r0:r1].double().numpy()
        fin = np.isfinite(L)
        assert np.array_equal(np.isneginf(got_l), ~fin), r0
        np.testing.assert_allclose(got_l[fin], L[fin], rtol=1e-5, atol=1e-5)
        np.testing.assert_allclose(got_o[fin], O[fin], rtol=rtol_o, atol=1e-5)
        assert np.all(got_o[~fin] == 0), r0


# The benchmark's merge workload (n partials of B*S*Hq = 524288 rows, D = 128)
# at full size: every row is compared, so every iteration of the kernels'
# grid-stride loops (a persistent one-wave grid) and the last, partial pass
# are covered. n = 17 runs the kernels for more than eight partials.
@pytest.mark.parametrize("n,rows", [(4, 524288), (8, 524288), (17, 131072 + 77)])
@pytest.mark.parametrize("tree", [False, True])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_merge_full_size(n, rows, tree, out_dtype):
    dev = device()
    o, lse = _partials(n, rows, 128, 1000 + n)
    oo, ll = usp.merge_partials(o.to(dev), lse.to(dev), tree_order=tree, out_dtype=out_dtype)
    torch.cuda.synchronize()
    # bf16 output: the fp32 result rounded once to nearest, which is within
    # one bf16 ulp (2^-7 relative) even after the fp32 arithmetic
    _merge_check_all_rows(oo.cpu(), ll.cpu(), o, lse, tree,
                          2.0 ** -7 if out_dtype == torch.bfloat16 else 1e-5)


def test_merge_empty_rows_ok():
    dev = device()
    o = torch.zeros(3, 0, 128, device=dev)
    lse = torch.zeros(3, 0, device=dev)
    oo, ll = usp.merge_partials(o, lse)
    assert oo.shape == (0, 128)

"""GPU parity of the standalone row softmax and row sum against the fp64
oracle (through the C ABI), across single-pass and two-pass row lengths,
ragged and misaligned widths, both element types, in place, and empty."""
import numpy as np
import pytest
import torch

import oracle
from tiled_online_softmax_fwd_gb300 import fattn

pytestmark = pytest.mark.gpu

# Tolerances.  fp32 softmax: exp2 with a ~2 ulp MUFU and the rounding of
# x*log2(e) and max*log2(e) (|x| <= ~40 here) give a relative error of a few
# 1e-6; held to 1e-5 relative.  bf16 output: the final rounding, 2^-8
# relative.  Row sums: fp32 accumulation over N terms, held to 1e-6 of
# sum |x| (plus 1e-6 absolute).
SIZES = [(1, 1), (3, 5), (7, 255), (5, 1024), (4, 1025), (9, 4000), (3, 16384), (2, 16385),
         (2, 50001), (1, 131072), (33, 2048)]


def _x(M, N, dtype, seed, scale=4.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(M, N, generator=g) * scale).to(dtype)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("M,N", SIZES)
def test_softmax_rows_matches_oracle(M, N, dtype):
    x = _x(M, N, dtype, seed=M * 7 + N)
    y = fattn.softmax_rows(x.cuda())
    torch.cuda.synchronize()
    ref = oracle.softmax_rows(x)
    got = y.cpu().double().numpy()
    rtol = 1e-5 if dtype == torch.float32 else 2 ** -8
    err = np.abs(got - ref) / np.maximum(np.abs(ref), 1e-30)
    assert np.all(np.isfinite(got))
    assert np.all(np.abs(got - ref) <= rtol * np.abs(ref) + 1e-30), err.max()
    # rows sum to 1 up to the output rounding (one dominant bf16 element can
    # be off by 2^-8 of itself)
    np.testing.assert_allclose(got.sum(axis=1), 1.0, rtol=0,
                               atol=1e-5 if dtype == torch.float32 else 2 ** -8)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("M,N", SIZES)
def test_row_sum_matches_oracle(M, N, dtype):
    x = _x(M, N, dtype, seed=M * 11 + N, scale=1.0)
    s = fattn.row_sum(x.cuda())
    torch.cuda.synchronize()
    ref = oracle.row_sum(x)
    bound = 1e-6 * oracle.row_sum(x.abs()) + 1e-6
    assert np.all(np.abs(s.cpu().double().numpy() - ref) <= bound)


def test_softmax_in_place_and_misaligned():
    x = _x(6, 3000, torch.float32, seed=3).cuda()
    ref = fattn.softmax_rows(x.clone())
    y = x.clone()
    fattn.softmax_rows(y, out=y)
    torch.cuda.synchronize()
    assert torch.equal(y, ref)
    # a view that starts 4 bytes into an allocation: scalar path, same results
    buf = torch.empty(6 * 3000 + 1, device="cuda")
    view = buf[1:].view(6, 3000)
    view.copy_(x)
    out = torch.empty(6 * 3000 + 1, device="cuda")[1:].view(6, 3000)
    fattn.softmax_rows(view, out=out)
    torch.cuda.synchronize()
    assert torch.allclose(out, ref, rtol=1e-6, atol=0)


def test_rowops_empty():
    e = torch.empty(0, 7, device="cuda")
    assert fattn.softmax_rows(e).shape == (0, 7)
    z = torch.empty(3, 0, device="cuda")
    assert fattn.row_sum(z).tolist() == [0.0, 0.0, 0.0]

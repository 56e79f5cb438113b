"""GPU test of attn_fwd_split_noalloc, the split-KV entry point for callers that
cannot allocate device memory on their execution path (a serving runtime that
plans all device memory before it starts, a plugin whose host framework owns
every allocation).  Its scratch is a fixed 32 MiB array inside the library.

Called through the C ABI and checked two ways on two calls in a row (the
second call finds the first call's leftovers in the shared scratch):
  * against attn_fwd_split given a caller-allocated workspace: the same
    kernels, split count and merge order, so the bits must be identical;
  * against the fp64 oracle, with the tolerances of every parity test.
Also: one split (no scratch at all, attn_fwd's bits, also where attn_fwd
itself would round V in a pre-pass that needs memory), the largest shape whose
scratch fits the array (32 bytes short of 32 MiB) and the next one up, which
is refused.

Kept in its own file, named to be collected last."""
import ctypes
import os

import pytest
import torch

import oracle
from tests.parity import assert_parity, compare
from tiled_online_softmax_fwd_gb300 import build as fbuild
from tiled_online_softmax_fwd_gb300 import fattn
from tiled_online_softmax_fwd_gb300.inputs import make_qkv

pytestmark = pytest.mark.gpu

OK, UNSUPPORTED = 0, 2
SCRATCH_BYTES = 32 << 20


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(fattn.library_path()):
        fbuild.build()
    return fattn.load()


def _noalloc(lib, q, k, v, o, lse, causal, scale, splits):
    B, H, N, d = q.shape
    return lib.attn_fwd_split_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                      lse.data_ptr(), B, H, N, d, ctypes.c_float(scale),
                                      1 if causal else 0, splits,
                                      torch.cuda.current_stream().cuda_stream)


def _outputs(q):
    B, H, N, _ = q.shape
    return (torch.full_like(q, float("nan")),
            torch.full((B, H, N), float("nan"), device=q.device))


@pytest.mark.parametrize("B,H,N,d,causal,splits", [(1, 1, 4096, 64, False, 10),
                                                   (1, 2, 2000, 128, True, 6),
                                                   (2, 3, 700, 96, True, 3)])
def test_noalloc_matches_workspace_entry_point_and_oracle_twice(lib, B, H, N, d, causal, splits):
    scale = fattn.default_scale(d)
    for call in range(2):
        q, k, v = make_qkv(B, H, N, d, seed=900 + call, sigma_qk=2.0)
        dq, dk, dv = q.cuda(), k.cuda(), v.cuda()
        ref_o, ref_l = fattn.attn_fwd_split(dq, dk, dv, causal=causal, scale=scale,
                                            num_splits=splits)
        o, lse = _outputs(dq)
        assert _noalloc(lib, dq, dk, dv, o, lse, causal, scale, splits) == OK
        torch.cuda.synchronize()
        assert torch.equal(o, ref_o) and torch.equal(lse, ref_l), "call %d" % call
        o_ref, lse_ref = oracle.attn_fwd(q, k, v, scale, causal)
        r = compare(o.cpu().reshape(-1, d), lse.cpu().reshape(-1), o_ref, lse_ref)
        assert_parity(r, "noalloc call %d" % call)


@pytest.mark.parametrize("B,H,N,d", [(2, 2, 1000, 128), (1, 2, 3072, 256)])
def test_noalloc_single_split_is_attn_fwd(lib, B, H, N, d):
    """The no-allocation call always rounds V on chip; at d = 256 with 3072
    queries attn_fwd takes the V pre-pass instead.  Same bits either way."""
    q, k, v = make_qkv(B, H, N, d, seed=911)
    dq, dk, dv = q.cuda(), k.cuda(), v.cuda()
    scale = fattn.default_scale(d)
    with fattn.v_conversion("auto"):
        assert (fattn.v_conversion_route(N, d, True) == "prepass") == (d == 256)
        ref_o, ref_l = fattn.attn_fwd(dq, dk, dv, causal=True, scale=scale)
        o, lse = _outputs(dq)
        assert _noalloc(lib, dq, dk, dv, o, lse, True, scale, 1) == OK
        torch.cuda.synchronize()
    assert torch.equal(o, ref_o) and torch.equal(lse, ref_l)


def test_noalloc_largest_shape_that_fits(lib):
    """Two splits of one head of 63550 rows at d = 64 need 2 * 63550 *
    (4 * 64 + 8) = 33554400 bytes, 32 short of the array; 63551 rows do not
    fit and are refused without a launch."""
    B, H, N, d, splits = 1, 1, 63550, 64, 2
    assert fattn.split_workspace_size(B, H, N, d, splits) <= SCRATCH_BYTES
    assert fattn.split_workspace_size(B, H, N + 1, d, splits) > SCRATCH_BYTES
    scale = fattn.default_scale(d)
    for call in range(2):
        q, k, v = make_qkv(B, H, N, d, seed=920 + call)
        dq, dk, dv = q.cuda(), k.cuda(), v.cuda()
        ref_o, ref_l = fattn.attn_fwd_split(dq, dk, dv, causal=bool(call), scale=scale,
                                            num_splits=splits)
        o, lse = _outputs(dq)
        assert _noalloc(lib, dq, dk, dv, o, lse, bool(call), scale, splits) == OK
        torch.cuda.synchronize()
        assert torch.equal(o, ref_o) and torch.equal(lse, ref_l), "call %d" % call
        # The last rows' partials sit at the end of the array: check them,
        # and a seeded sample of the rest, against the oracle.
        g = torch.Generator().manual_seed(930 + call)
        rows = torch.cat([torch.randperm(N - 256, generator=g)[:256],
                          torch.arange(N - 256, N)]).sort().values
        o_ref, lse_ref = oracle.attn_fwd(q, k, v, scale, bool(call), rows=rows.numpy())
        r = compare(o.cpu().reshape(-1, d)[rows], lse.cpu().reshape(-1)[rows], o_ref, lse_ref)
        assert_parity(r, "largest noalloc shape, call %d" % call)
    q = torch.zeros(B, H, N + 1, d, dtype=torch.bfloat16, device="cuda")
    o, lse = _outputs(q)
    assert _noalloc(lib, q, q, q, o, lse, False, scale, splits) == UNSUPPORTED
    torch.cuda.synchronize()
    assert torch.isnan(o).all()  # nothing was enqueued


def test_noalloc_rejects_shapes_beyond_its_scratch(lib):
    # 16 splits of 8 heads x 16384 rows x d=128 need far more than 32 MiB.
    q = torch.zeros(1, 8, 16384, 128, dtype=torch.bfloat16, device="cuda")
    o = torch.empty_like(q)
    lse = torch.empty(1, 8, 16384, device="cuda")
    assert _noalloc(lib, q, q, q, o, lse, False, 0.088, 16) == UNSUPPORTED

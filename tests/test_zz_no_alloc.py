"""GPU test of attn_fwd_split_noalloc, the split-KV entry point for callers that
cannot allocate device memory on their execution path (its scratch is a fixed
array inside the library).  Called through the C ABI and compared with
attn_fwd_split given a caller-allocated workspace, on two calls in a row (the
second call finds the first call's leftovers in the shared scratch).

Kept in its own file, named to be collected last."""
import ctypes
import os

import pytest
import torch

from tests.parity import assert_parity, compare
from tiled_online_softmax_fwd_gb300 import build as fbuild
from tiled_online_softmax_fwd_gb300 import fattn
from tiled_online_softmax_fwd_gb300.inputs import make_qkv

pytestmark = pytest.mark.gpu

OK, UNSUPPORTED = 0, 2


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


@pytest.mark.parametrize("B,H,N,d,causal,splits", [(1, 1, 4096, 64, False, 10),
                                                   (1, 2, 2000, 128, True, 6)])
def test_noalloc_matches_workspace_entry_point_twice(lib, B, H, N, d, causal, splits):
    scale = fattn.default_scale(d)
    for call in range(2):
        q, k, v = make_qkv(B, H, N, d, seed=900 + call, sigma_qk=2.0)
        dq, dk, dv = q.cuda(), k.cuda(), v.cuda()
        ref_o, ref_l = fattn.attn_fwd_split(dq, dk, dv, causal=causal, scale=scale,
                                            num_splits=splits)
        o = torch.full_like(dq, float("nan"))
        lse = torch.full((B, H, N), float("nan"), device="cuda")
        assert _noalloc(lib, dq, dk, dv, o, lse, causal, scale, splits) == OK
        torch.cuda.synchronize()
        r = compare(o.cpu().reshape(-1, d), lse.cpu().reshape(-1),
                    ref_o.cpu().double().reshape(-1, d).numpy(),
                    ref_l.cpu().double().reshape(-1).numpy(), mean_rule="floor")
        assert_parity(r, "noalloc call %d" % call)


def test_noalloc_rejects_shapes_beyond_its_scratch(lib):
    # 16 splits of 8 heads x 16384 rows x d=128 need far more than 32 MiB.
    q = torch.zeros(1, 8, 16384, 128, dtype=torch.bfloat16, device="cuda")
    o = torch.empty_like(q)
    lse = torch.empty(1, 8, 16384, device="cuda")
    assert _noalloc(lib, q, q, q, o, lse, False, 0.088, 16) == UNSUPPORTED

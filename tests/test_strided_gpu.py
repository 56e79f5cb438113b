"""GPU parity tests of attn_fwd_strided (any (batch, head, row) strides with a
contiguous last dimension) through the C ABI against the fp64 oracle on
contiguous copies of the same seeded inputs."""
import os

import pytest
import torch

import oracle
from tests.parity import assert_parity, compare
from tiled_online_softmax_fwd_gb300 import build as fbuild
from tiled_online_softmax_fwd_gb300 import fattn
from tiled_online_softmax_fwd_gb300.inputs import make_qkv, make_qkv_kv

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not os.path.exists(fattn.library_path()):
        fbuild.build()
    lib = fattn.load()
    yield lib
    torch.cuda.synchronize()
    assert fattn.device_status() == 0, "a kernel reported a pipeline timeout"


def packed_views(q, k, v):
    """q, k, v [B,H,N,d] copied into one [B, N, 3, H, d] device buffer and
    returned as strided [B,H,N,d] views of it."""
    B, H, N, d = q.shape
    buf = torch.empty((B, N, 3, H, d), dtype=torch.bfloat16, device="cuda")
    for i, t in enumerate((q, k, v)):
        buf[:, :, i] = t.permute(0, 2, 1, 3).cuda()
    return [buf[:, :, i].permute(0, 2, 1, 3) for i in range(3)]


PACKED_CASES = [(2, 3, 200, 64, False), (2, 3, 200, 64, True), (1, 4, 513, 128, True),
                (2, 2, 128, 128, False), (1, 1, 1, 64, True), (3, 2, 1000, 64, True)]


@pytest.mark.parametrize("B,H,N,d,causal", PACKED_CASES,
                         ids=["B%dH%dN%dd%d%s" % (b, h, n, d, "c" if c else "")
                              for b, h, n, d, c in PACKED_CASES])
def test_packed_qkv_and_interleaved_output(B, H, N, d, causal):
    """q, k, v sliced from one packed [B, N, 3, H, d] projection output; o
    written into a [B, N, H, d] buffer, whose padding stays untouched."""
    q, k, v = make_qkv(B, H, N, d, seed=70 + N + d, sigma_qk=2.0)
    dq, dk, dv = packed_views(q, k, v)
    assert H * N == 1 or not dq.is_contiguous()
    obuf = torch.full((B, N, H, d + 8), 7.0, dtype=torch.bfloat16, device="cuda")
    o_view = obuf[..., :d].permute(0, 2, 1, 3)
    o, lse = fattn.attn_fwd_strided(dq, dk, dv, causal=causal, out=o_view)
    torch.cuda.synchronize()
    assert (obuf[..., d:] == 7.0).all(), "the kernel wrote outside o"
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, fattn.default_scale(d), causal)
    r = compare(o_view.contiguous().cpu().reshape(-1, d), lse.cpu().reshape(-1), o_ref, lse_ref)
    assert_parity(r, "packed B%dH%dN%dd%d" % (B, H, N, d))


@pytest.mark.parametrize("d", [64, 128])
def test_dense_strides_match_attn_fwd(d):
    q, k, v = make_qkv(2, 3, 300, d, seed=5)
    dq, dk, dv = q.cuda(), k.cuda(), v.cuda()
    a = fattn.attn_fwd_strided(dq, dk, dv, causal=True, num_splits=1)
    b = fattn.attn_fwd(dq, dk, dv, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


@pytest.mark.parametrize("Nq,Nk,splits", [(1, 3000, 0), (1, 20000, 0), (100, 2500, 0),
                                          (100, 2500, 4), (256, 700, 1)])
def test_decode_from_a_cache_with_spare_rows(Nq, Nk, splits):
    """Keys and values are the first Nk rows of a [B, H, 24576, d] cache
    (head stride 24576*d); queries have a padded row stride."""
    B, H, d, cap = 2, 4, 128, 24576
    q, k, v = make_qkv_kv(B, H, Nq, Nk, d, seed=Nq + Nk + splits, sigma_qk=2.0)
    kc = torch.zeros((B, H, cap, d), dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    kc[:, :, :Nk] = k.cuda()
    vc[:, :, :Nk] = v.cuda()
    qpad = torch.zeros((B, H, Nq, d + 64), dtype=torch.bfloat16, device="cuda")
    qpad[..., :d] = q.cuda()
    o, lse = fattn.attn_fwd_strided(qpad[..., :d], kc[:, :, :Nk], vc[:, :, :Nk], causal=True,
                                    num_splits=splits)
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle.attn_fwd_kv(q, k, v, fattn.default_scale(d), True)
    r = compare(o.cpu().reshape(-1, d), lse.cpu().reshape(-1), o_ref, lse_ref)
    assert_parity(r, "cache Nq%d Nk%d s%d" % (Nq, Nk, splits))


def test_head_major_batch_minor_layout():
    """Batch stride smaller than head stride ([H, B, N, d] storage)."""
    B, H, N, d = 3, 2, 257, 64
    q, k, v = make_qkv(B, H, N, d, seed=9)
    views = [t.permute(1, 0, 2, 3).contiguous().cuda().permute(1, 0, 2, 3) for t in (q, k, v)]
    o_store = torch.empty((H, B, N, d), dtype=torch.bfloat16, device="cuda")
    o, lse = fattn.attn_fwd_strided(*views, causal=False, out=o_store.permute(1, 0, 2, 3))
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, fattn.default_scale(d), False)
    r = compare(o.contiguous().cpu().reshape(-1, d), lse.cpu().reshape(-1), o_ref, lse_ref)
    assert_parity(r, "head-major")


@pytest.mark.parametrize("d", [64, 128, 256])
def test_fp16_strided_kv_and_splits(d):
    """fp16 through the general entry: packed q/k/v views, decode-shaped
    queries against a longer key sequence, the automatic schedule."""
    B, H, Nq, Nk = 1, 3, 100, 3000
    q, k, v = make_qkv_kv(B, H, Nq, Nk, d, seed=d, dtype=torch.float16)
    kv = torch.empty((B, Nk, 2, H, d), dtype=torch.float16, device="cuda")
    kv[:, :, 0] = k.permute(0, 2, 1, 3).cuda()
    kv[:, :, 1] = v.permute(0, 2, 1, 3).cuda()
    dk, dv = kv[:, :, 0].permute(0, 2, 1, 3), kv[:, :, 1].permute(0, 2, 1, 3)
    o, lse = fattn.attn_fwd_strided(q.cuda(), dk, dv, causal=True)
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle.attn_fwd_kv(q, k, v, fattn.default_scale(d), True)
    r = compare(o.float().cpu().reshape(-1, d), lse.cpu().reshape(-1), o_ref, lse_ref)
    assert_parity(r, "fp16 strided d%d" % d)

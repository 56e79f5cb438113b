"""GPU parity tests of attn_fwd_kv (queries against a longer key sequence, the
decode shape) through the C ABI against the fp64 oracle on the same seeded
inputs, element by element; the full-size decode and chunk workloads against
oracle rows; the square case against attn_fwd."""
import os

import pytest
import torch

import oracle
from tests.parity import assert_parity, compare
from tiled_online_softmax_fwd_gb300 import build as fbuild
from tiled_online_softmax_fwd_gb300 import fattn
from tiled_online_softmax_fwd_gb300.inputs import KV_WORKLOADS, make_qkv_kv, sample_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not os.path.exists(fattn.library_path()):
        fbuild.build()
    lib = fattn.load()
    yield lib
    torch.cuda.synchronize()
    assert fattn.device_status() == 0, "a kernel reported a pipeline timeout"


# (B, H, Nq, Nk, d, causal, num_splits); num_splits 0 = the library's choice.
# Offsets Nk - Nq that are and are not multiples of 128, one and several
# query tiles, ragged key tails, and splits that start on a key tile where
# some rows see no key (Nq 256, Nk 320, 3 splits: rows 0..63 of the first
# query tile see no key of the second key tile, the second split's only one).
KV_CASES = [
    (1, 2, 1, 1, 64, True, 1), (2, 3, 1, 300, 128, True, 0), (1, 2, 1, 4099, 64, False, 0),
    (1, 1, 7, 7, 128, True, 1), (1, 2, 128, 1000, 64, True, 1), (1, 2, 129, 1000, 128, True, 3),
    (2, 2, 300, 1037, 64, True, 0), (1, 1, 200, 3000, 128, False, 5),
    (1, 1, 64, 448, 128, True, 1), (1, 3, 1, 16384, 128, True, 0), (1, 1, 255, 256, 64, True, 2),
    (1, 1, 256, 320, 64, True, 3), (1, 1, 256, 320, 128, True, 3), (1, 1, 130, 2000, 64, True, 16),
    (1, 1, 16, 5000, 128, False, 64), (3, 1, 2, 129, 64, True, 2),
    # The automatic schedule deals (head, key tile) steps over the SMs
    # (stream-K) for these: one or two query tiles per head, few heads, long
    # keys; the last one has ranges of two key tiles, some starting on a key
    # tile that rows 0..63 of the first query tile cannot see.
    (1, 5, 200, 9000, 64, True, 0), (2, 3, 256, 20000, 128, True, 0),
    (1, 1, 1, 50000, 128, False, 0), (1, 2, 256, 19520, 64, True, 0),
    (1, 2, 256, 19520, 128, True, 0),
]


def case_id(c):
    B, H, Nq, Nk, d, causal, s = c
    return "B%dH%dNq%dNk%dd%d%s_s%d" % (B, H, Nq, Nk, d, "c" if causal else "", s)


@pytest.mark.parametrize("B,H,Nq,Nk,d,causal,splits", KV_CASES, ids=[case_id(c) for c in KV_CASES])
def test_kv_matches_oracle(B, H, Nq, Nk, d, causal, splits):
    q, k, v = make_qkv_kv(B, H, Nq, Nk, d, seed=900 + Nq + Nk + d, sigma_qk=2.0)
    scale = fattn.default_scale(d)
    o, lse = fattn.attn_fwd_kv(q.cuda(), k.cuda(), v.cuda(), causal=causal, scale=scale,
                               num_splits=splits)
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle.attn_fwd_kv(q, k, v, scale, causal)
    r = compare(o.cpu().reshape(-1, d), lse.cpu().reshape(-1), o_ref, lse_ref)
    assert_parity(r, case_id((B, H, Nq, Nk, d, causal, splits)))


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
def test_square_kv_is_attn_fwd(causal, d):
    """Nq == Nk with one split runs the same kernel with the same schedule as
    attn_fwd: the results are bit-identical."""
    q, k, v = make_qkv_kv(2, 3, 700, 700, d, seed=31 + d)
    dq, dk, dv = q.cuda(), k.cuda(), v.cuda()
    o1, l1 = fattn.attn_fwd_kv(dq, dk, dv, causal=causal, num_splits=1)
    o2, l2 = fattn.attn_fwd(dq, dk, dv, causal=causal)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_decode_row_ignores_the_mask():
    """A single query row is the last key position: the mask hides nothing."""
    q, k, v = make_qkv_kv(2, 4, 1, 3000, 128, seed=5)
    dq, dk, dv = q.cuda(), k.cuda(), v.cuda()
    a = fattn.attn_fwd_kv(dq, dk, dv, causal=True, num_splits=4)
    b = fattn.attn_fwd_kv(dq, dk, dv, causal=False, num_splits=4)
    torch.cuda.synchronize()
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_splits_agree():
    """Different key-range splits give the same result up to the merge's
    rounding (the partial outputs are fp32)."""
    q, k, v = make_qkv_kv(1, 2, 64, 8192, 128, seed=8, sigma_qk=2.0)
    dq, dk, dv = q.cuda(), k.cuda(), v.cuda()
    o1, l1 = fattn.attn_fwd_kv(dq, dk, dv, causal=True, num_splits=1)
    for s in (2, 9, 32):
        o, lse = fattn.attn_fwd_kv(dq, dk, dv, causal=True, num_splits=s)
        torch.cuda.synchronize()
        assert (o.float() - o1.float()).abs().max().item() <= 2 ** -5
        assert (lse - l1).abs().max().item() <= 1e-4


def test_kv_workspace_query_matches_the_auto_choice():
    need = fattn.kv_workspace_size(8, 32, 1, 32768, 128, True, 0)
    assert need >= 0
    q, k, v = make_qkv_kv(1, 1, 1, 256, 64, seed=2)
    ws = torch.empty(max(fattn.kv_workspace_size(1, 1, 1, 256, 64, True, 0), 1),
                     dtype=torch.uint8, device="cuda")
    o, _ = fattn.attn_fwd_kv(q.cuda(), k.cuda(), v.cuda(), causal=True, workspace=ws)
    torch.cuda.synchronize()
    assert torch.isfinite(o.float()).all()


@pytest.mark.parametrize("name", list(KV_WORKLOADS))
def test_kv_workload_matches_oracle(name):
    """Full-size decode / chunk workloads in the launch configuration the
    benchmark times (the library's split choice), on oracle rows: every row
    of the decode workload, 64 rows of every head of the chunk workload."""
    w = KV_WORKLOADS[name]
    q, k, v = make_qkv_kv(w.B, w.H, w.Nq, w.Nk, w.d, w.seed, w.sigma_qk)
    o, lse = fattn.attn_fwd_kv(q.cuda(), k.cuda(), v.cuda(), causal=w.causal, scale=w.scale)
    torch.cuda.synchronize()
    rows = None
    if w.Nq > 64:
        rows = sample_rows(w.B, w.H, w.Nq, 64, torch.Generator("cpu").manual_seed(w.seed + 1))
    o_ref, lse_ref = oracle.attn_fwd_kv(q, k, v, w.scale, w.causal, rows=rows)
    o_g, l_g = o.cpu().reshape(-1, w.d), lse.cpu().reshape(-1)
    if rows is not None:
        o_g, l_g = o_g[rows], l_g[rows]
    assert_parity(compare(o_g, l_g, o_ref, lse_ref), name)

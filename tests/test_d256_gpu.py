"""GPU parity tests of head dimension 256 (one Q tile per CTA, two S buffers
in TMEM, O in 256 columns) through the C ABI against the fp64 oracle on the
same seeded inputs."""
import os

import pytest
import torch

import oracle
from tests.parity import assert_parity, compare
from tiled_online_softmax_fwd_gb300 import build as fbuild
from tiled_online_softmax_fwd_gb300 import fattn
from tiled_online_softmax_fwd_gb300.inputs import (VARIANT_WORKLOADS, make_qkv, make_qkv_kv,
                                                   make_workload)

pytestmark = pytest.mark.gpu
D = 256


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not os.path.exists(fattn.library_path()):
        fbuild.build()
    lib = fattn.load()
    yield lib
    torch.cuda.synchronize()
    assert fattn.device_status() == 0, "a kernel reported a pipeline timeout"


CASES = [(2, 3, N, c) for N in (1, 17, 127, 128, 129, 256, 383, 513, 1000) for c in (False, True)]


@pytest.mark.parametrize("B,H,N,causal", CASES,
                         ids=["B%dH%dN%d%s" % (b, h, n, "c" if c else "") for b, h, n, c in CASES])
def test_d256_matches_oracle(B, H, N, causal):
    q, k, v = make_qkv(B, H, N, D, seed=3000 + N + causal, sigma_qk=1.5)
    o, lse = fattn.attn_fwd(q.cuda(), k.cuda(), v.cuda(), causal=causal)
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, fattn.default_scale(D), causal)
    r = compare(o.cpu().reshape(-1, D), lse.cpu().reshape(-1), o_ref, lse_ref)
    assert_parity(r, "d256 N%d" % N)


@pytest.mark.parametrize("N,causal", [(300, True), (1000, False)])
def test_d256_fp16(N, causal):
    q, k, v = make_qkv(2, 2, N, D, seed=11 + N, dtype=torch.float16)
    o, lse = fattn.attn_fwd_fp16(q.cuda(), k.cuda(), v.cuda(), causal=causal)
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, fattn.default_scale(D), causal)
    r = compare(o.float().cpu().reshape(-1, D), lse.cpu().reshape(-1), o_ref, lse_ref)
    assert_parity(r, "d256 fp16 N%d" % N)


@pytest.mark.parametrize("Nq,Nk,splits", [(1, 9000, 0), (64, 3000, 0), (200, 1500, 3),
                                          (256, 320, 3)])
def test_d256_kv_and_splits(Nq, Nk, splits):
    q, k, v = make_qkv_kv(1, 3, Nq, Nk, D, seed=Nq + Nk, sigma_qk=2.0)
    o, lse = fattn.attn_fwd_kv(q.cuda(), k.cuda(), v.cuda(), causal=True, num_splits=splits)
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle.attn_fwd_kv(q, k, v, fattn.default_scale(D), True)
    r = compare(o.cpu().reshape(-1, D), lse.cpu().reshape(-1), o_ref, lse_ref)
    assert_parity(r, "d256 kv Nq%d Nk%d" % (Nq, Nk))


def test_d256_strided_output_leaves_padding():
    B, H, N = 2, 3, 333
    q, k, v = make_qkv(B, H, N, D, seed=4)
    obuf = torch.full((B, H, N, D + 32), 5.0, dtype=torch.bfloat16, device="cuda")
    o, lse = fattn.attn_fwd_strided(q.cuda(), k.cuda(), v.cuda(), causal=True,
                                    out=obuf[..., :D])
    torch.cuda.synchronize()
    assert (obuf[..., D:] == 5.0).all()
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, fattn.default_scale(D), True)
    r = compare(o.contiguous().cpu().reshape(-1, D), lse.cpu().reshape(-1), o_ref, lse_ref)
    assert_parity(r, "d256 strided")


def test_d256_workload_matches_oracle():
    """B=2, H=16, N=8192, d=256, causal: 128 seeded rows per head against the
    oracle (the SIMT cross-check kernel has no d = 256 instance)."""
    w = VARIANT_WORKLOADS["B2_H16_N8192_d256_causal"]
    q, k, v, rows = make_workload(w)
    o, lse = fattn.attn_fwd(q.cuda(), k.cuda(), v.cuda(), causal=True, scale=w.scale)
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, w.scale, True, rows=rows.numpy())
    r = compare(o.cpu().reshape(-1, D)[rows], lse.cpu().reshape(-1)[rows], o_ref, lse_ref)
    assert_parity(r, w.name)


def test_d256_many_units_and_splits():
    """Several Q tiles per CTA (units over 152 SMs) and a fixed split."""
    q, k, v = make_qkv(3, 20, 700, D, seed=21, sigma_qk=2.0)
    dq, dk, dv = q.cuda(), k.cuda(), v.cuda()
    o, lse = fattn.attn_fwd(dq, dk, dv, causal=True)
    o2, lse2 = fattn.attn_fwd_split(dq, dk, dv, causal=True, num_splits=3)
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, fattn.default_scale(D), True)
    for a, b in ((o, lse), (o2, lse2)):
        r = compare(a.cpu().reshape(-1, D), b.cpu().reshape(-1), o_ref, lse_ref)
        assert_parity(r, "d256 units")


def test_d256_backward_is_refused():
    q, k, v = make_qkv(1, 1, 128, D, seed=1)
    dq = q.cuda()
    o, lse = fattn.attn_fwd(dq, dq, dq)
    with pytest.raises(ValueError):
        fattn.attn_bwd(dq, dq, dq, o, lse, o)

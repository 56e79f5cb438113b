"""GPU parity tests of head dimension 96 (two 64-column tensor-map boxes, the
second half zero-filled; S over K = 96, P V with N = 96) through the C ABI
against the fp64 oracle on the same seeded inputs."""
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
D = 96


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
def test_d96_matches_oracle(B, H, N, causal):
    q, k, v = make_qkv(B, H, N, D, seed=3000 + N + causal, sigma_qk=1.5)
    o, lse = fattn.attn_fwd(q.cuda(), k.cuda(), v.cuda(), causal=causal)
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, fattn.default_scale(D), causal)
    r = compare(o.cpu().reshape(-1, D), lse.cpu().reshape(-1), o_ref, lse_ref)
    assert_parity(r, "d96 N%d" % N)


@pytest.mark.parametrize("N,causal", [(300, True), (1000, False)])
def test_d96_fp16(N, causal):
    q, k, v = make_qkv(2, 2, N, D, seed=11 + N, dtype=torch.float16)
    o, lse = fattn.attn_fwd_fp16(q.cuda(), k.cuda(), v.cuda(), causal=causal)
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, fattn.default_scale(D), causal)
    r = compare(o.float().cpu().reshape(-1, D), lse.cpu().reshape(-1), o_ref, lse_ref)
    assert_parity(r, "d96 fp16 N%d" % N)


@pytest.mark.parametrize("Nq,Nk,splits", [(1, 9000, 0), (64, 3000, 0), (200, 1500, 3),
                                          (256, 320, 3)])
def test_d96_kv_and_splits(Nq, Nk, splits):
    q, k, v = make_qkv_kv(1, 3, Nq, Nk, D, seed=Nq + Nk, sigma_qk=2.0)
    o, lse = fattn.attn_fwd_kv(q.cuda(), k.cuda(), v.cuda(), causal=True, num_splits=splits)
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle.attn_fwd_kv(q, k, v, fattn.default_scale(D), True)
    r = compare(o.cpu().reshape(-1, D), lse.cpu().reshape(-1), o_ref, lse_ref)
    assert_parity(r, "d96 kv Nq%d Nk%d" % (Nq, Nk))


def test_d96_strided_output_leaves_padding():
    B, H, N = 2, 3, 333
    q, k, v = make_qkv(B, H, N, D, seed=4)
    obuf = torch.full((B, H, N, D + 32), 5.0, dtype=torch.bfloat16, device="cuda")
    o, lse = fattn.attn_fwd_strided(q.cuda(), k.cuda(), v.cuda(), causal=True,
                                    out=obuf[..., :D])
    torch.cuda.synchronize()
    assert (obuf[..., D:] == 5.0).all()
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, fattn.default_scale(D), True)
    r = compare(o.contiguous().cpu().reshape(-1, D), lse.cpu().reshape(-1), o_ref, lse_ref)
    assert_parity(r, "d96 strided")


def test_d96_workload_matches_oracle_and_simt():
    """B=4, H=16, N=4096, d=96, causal: 256 seeded rows per head against the
    oracle, every row against the SIMT kernel."""
    w = VARIANT_WORKLOADS["B4_H16_N4096_d96_causal"]
    q, k, v, rows = make_workload(w)
    dq, dk, dv = q.cuda(), k.cuda(), v.cuda()
    o, lse = fattn.attn_fwd(dq, dk, dv, causal=True, scale=w.scale)
    o2, lse2 = fattn.attn_fwd_simt(dq, dk, dv, causal=True, scale=w.scale)
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, w.scale, True, rows=rows.numpy())
    r = compare(o.cpu().reshape(-1, D)[rows], lse.cpu().reshape(-1)[rows], o_ref, lse_ref)
    assert_parity(r, w.name)
    assert (o.float() - o2.float()).abs().max().item() <= 2e-2
    assert (lse - lse2).abs().max().item() <= 1e-3


def test_d96_backward_is_refused():
    q, k, v = make_qkv(1, 1, 128, D, seed=1)
    dq = q.cuda()
    o, lse = fattn.attn_fwd(dq, dq, dq)
    with pytest.raises(ValueError):
        fattn.attn_bwd(dq, dq, dq, o, lse, o)

"""GPU parity of the fp16 variant (attn_fwd_fp16) against the fp64 oracle.

fp16 outputs have a rounding step of at most 2^-7 below |O| = 16, so the
stated bounds apply to every element as they stand: max |dO| <= 1e-2,
mean |dO| <= 1e-3, max |dlse| <= 1e-3."""
import numpy as np
import pytest
import torch

import oracle
from tiled_online_softmax_fwd_gb300 import fattn
from tiled_online_softmax_fwd_gb300.inputs import WORKLOADS, make_qkv, make_workload

pytestmark = pytest.mark.gpu


def _check(o, lse, o_ref, lse_ref):
    d = np.abs(o.cpu().double().numpy().reshape(o_ref.shape) - o_ref)
    dl = np.abs(lse.cpu().double().numpy().reshape(lse_ref.shape) - lse_ref)
    assert np.all(np.isfinite(d)) and np.all(np.isfinite(dl))
    assert d.max() <= 1e-2 and d.mean() <= 1e-3 and dl.max() <= 1e-3, (d.max(), d.mean(), dl.max())


CASES = [(2, 3, N, d, c) for N in (1, 127, 129, 300, 1000) for d in (64, 128) for c in (False, True)]


@pytest.mark.parametrize("B,H,N,d,causal", CASES,
                         ids=["B%dH%dN%dd%d%s" % (b, h, n, d, "c" if c else "") for b, h, n, d, c in CASES])
def test_fp16_matches_oracle(B, H, N, d, causal):
    q, k, v = make_qkv(B, H, N, d, seed=4000 + N + d, sigma_qk=2.0, dtype=torch.float16)
    scale = fattn.default_scale(d)
    o, lse = fattn.attn_fwd_fp16(q.cuda(), k.cuda(), v.cuda(), causal=causal, scale=scale)
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, scale, causal)
    _check(o, lse, o_ref, lse_ref)


@pytest.mark.parametrize("name", ["B4_H16_N4096_d128_causal", "B1_H32_N16384_d128_causal_sigma3"])
def test_fp16_workload_sampled(name):
    w = WORKLOADS[name]
    q, k, v, rows = make_workload(w, dtype=torch.float16, sample_per_head=512)
    o, lse = fattn.attn_fwd_fp16(q.cuda(), k.cuda(), v.cuda(), causal=w.causal, scale=w.scale)
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, w.scale, w.causal, rows=rows.numpy())
    idx = rows.cuda()
    _check(o.reshape(-1, w.d)[idx], lse.reshape(-1)[idx], o_ref, lse_ref)


def test_fp16_rejects_bf16_tensors():
    q = torch.zeros(1, 1, 8, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ValueError):
        fattn.attn_fwd_fp16(q, q, q)

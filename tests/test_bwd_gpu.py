"""GPU parity of the backward pass (attn_bwd, through the C ABI) against the
fp64 oracle's gradients.  The forward's o and lse come from attn_fwd, as a
user's autograd wrapper would save them.

Tolerances (derived from the arithmetic; the pages state none for the
backward): every gradient is stored in bf16 (rounding 2^-9 relative) and is
computed from P and dS rounded to bf16 (2^-9 relative each) with fp32
accumulation.  D = dO . O uses the forward's bf16-rounded O, and where P is
peaked, dS = P (dP - D) cancels, so D's rounding shows up relative to a small
dQ: a CPU simulation of exactly this arithmetic on the N=16384 causal sigma=3
workload gives mean |delta| = 0.62% of mean |dQ| (0.22% with exact D).  Per
tensor: max |delta| <= 2e-2 * max |ref| + 1e-5 and mean |delta| <=
1e-2 * mean |ref| + 1e-6 (the absolute floors cover references that are
exactly zero, e.g. dQ with a single key)."""
import numpy as np
import pytest
import torch

import oracle
from tiled_online_softmax_fwd_gb300 import fattn
from tiled_online_softmax_fwd_gb300.inputs import WORKLOADS, make_qkv, make_workload

pytestmark = pytest.mark.gpu

MAX_REL, MEAN_REL = 2e-2, 1e-2
MAX_ABS, MEAN_ABS = 1e-5, 1e-6


def _dout(shape, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(shape, generator=g).to(torch.bfloat16)


def _check(name, got, ref):
    got = got.cpu().double().numpy().reshape(ref.shape)
    assert np.all(np.isfinite(got)), name
    err = np.abs(got - ref)
    scale_max, scale_mean = np.abs(ref).max(), np.abs(ref).mean()
    assert err.max() <= MAX_REL * scale_max + MAX_ABS, (name, err.max(), scale_max)
    assert err.mean() <= MEAN_REL * scale_mean + MEAN_ABS, (name, err.mean(), scale_mean)
    return err.max() / max(scale_max, 1e-30), err.mean() / max(scale_mean, 1e-30)


CASES = []
for N in (1, 17, 128, 129, 300, 513):
    for d in (64, 128):
        for causal in (False, True):
            CASES.append((1, 2, N, d, causal))
CASES += [(2, 3, 256, 128, True), (1, 1, 1024, 64, False), (3, 2, 700, 128, True)]
# Several work units per CTA (640 key tiles and 640 query tiles over the
# SMs), so every pipeline crosses unit boundaries, checked element by element.
CASES += [(8, 20, 512, 64, True), (4, 40, 384, 128, True), (4, 40, 300, 128, False)]


@pytest.mark.parametrize("B,H,N,d,causal", CASES,
                         ids=["B%dH%dN%dd%d%s" % (b, h, n, d, "c" if c else "") for b, h, n, d, c in CASES])
def test_bwd_matches_oracle(B, H, N, d, causal):
    q, k, v = make_qkv(B, H, N, d, seed=2000 + N + d, sigma_qk=1.5)
    g = _dout(q.shape, seed=3000 + N)
    scale = fattn.default_scale(d)
    dq_, dk_, dv_, dg = q.cuda(), k.cuda(), v.cuda(), g.cuda()
    o, lse = fattn.attn_fwd(dq_, dk_, dv_, causal=causal, scale=scale)
    gq, gk, gv = fattn.attn_bwd(dq_, dk_, dv_, o, lse, dg, causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert fattn.device_status() == 0
    rq, rk, rv = oracle.attn_bwd(q, k, v, g, scale, causal)
    _check("dq", gq, rq)
    _check("dk", gk, rk)
    _check("dv", gv, rv)


# Full-size workloads: (name, heads whose key rows dK/dV are checked).  Each
# checked head costs the oracle one pass over all of its query rows.
BWD_WORKLOADS = [("B4_H16_N4096_d128_causal", 4), ("B1_H32_N16384_d128_causal_sigma3", 2),
                 ("B2_H8_N65536_d64", 1)]


def _key_rows(w, heads, per_head, seed):
    """Seeded key rows of `heads` seeded heads: the first and last key of
    each (the last is seen by the fewest queries under the mask) and
    per_head - 2 random others; global ids (b*H + h)*N + j."""
    g = torch.Generator().manual_seed(seed)
    hs = torch.randperm(w.B * w.H, generator=g)[:heads]
    out = []
    for h in hs.tolist():
        js = torch.randperm(w.N - 2, generator=g)[:per_head - 2] + 1
        out.append(torch.cat([torch.tensor([0, w.N - 1]), js]).sort().values + h * w.N)
    return torch.cat(out)


@pytest.mark.parametrize("name,heads", BWD_WORKLOADS, ids=[n for n, _ in BWD_WORKLOADS])
def test_bwd_full_size_sampled(name, heads):
    """Full-size workloads in the benchmark's launch configuration: dQ on 64
    seeded query rows per head, and dK, dV on 64 seeded key rows of a few
    seeded heads, element by element against the oracle; plus the
    invariants that hold at any size over every head (each row of dS sums
    to zero, so sum_j dK_j = 0; rows of P sum to one, so
    sum_j dV_j = sum_i dO_i), relative to the tensors' own magnitude."""
    w = WORKLOADS[name]
    q, k, v, rows = make_workload(w, sample_per_head=64)
    g = _dout(q.shape, seed=77)
    dq_, dk_, dv_, dg = q.cuda(), k.cuda(), v.cuda(), g.cuda()
    o, lse = fattn.attn_fwd(dq_, dk_, dv_, causal=w.causal, scale=w.scale)
    gq, gk, gv = fattn.attn_bwd(dq_, dk_, dv_, o, lse, dg, causal=w.causal, scale=w.scale)
    torch.cuda.synchronize()
    assert fattn.device_status() == 0
    ref = oracle.attn_bwd_dq_rows(q, k, v, g, w.scale, w.causal, rows.numpy())
    _check("dq rows", gq.reshape(-1, w.d)[rows.cuda()], ref)
    keys = _key_rows(w, heads, 64, seed=78)
    rk, rv = oracle.attn_bwd_dkv_rows(q, k, v, g, w.scale, w.causal, keys.numpy())
    _check("dk rows", gk.reshape(-1, w.d)[keys.cuda()], rk)
    _check("dv rows", gv.reshape(-1, w.d)[keys.cuda()], rv)
    sk = gk.double().sum(dim=2)
    assert (sk.abs().max() / gk.double().abs().sum(dim=2).max()).item() <= 1e-2
    sv = gv.double().sum(dim=2)
    ref_sv = dg.double().sum(dim=2)
    assert ((sv - ref_sv).abs().max() / ref_sv.abs().max()).item() <= 2e-2


@pytest.mark.parametrize("B,H,N,d,causal", [(4, 16, 4096, 128, True), (2, 8, 16384, 64, False)])
def test_bwd_is_deterministic(B, H, N, d, causal):
    """Repeated backward calls on the same inputs give identical, finite bits.
    (The dQ kernel releases dP of a key tile early, so its warps can be a
    tile apart; a hand-off of dS that mixed two tiles' arrivals once let the
    dQ product read a slow warp's rows before they were written, in a few
    percent of calls.)"""
    q, k, v = make_qkv(B, H, N, d, seed=5000 + N + d, sigma_qk=1.5)
    g = _dout(q.shape, seed=5100 + N)
    dq_, dk_, dv_, dg = q.cuda(), k.cuda(), v.cuda(), g.cuda()
    scale = fattn.default_scale(d)
    o, lse = fattn.attn_fwd(dq_, dk_, dv_, causal=causal, scale=scale)
    ref = fattn.attn_bwd(dq_, dk_, dv_, o, lse, dg, causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert all(torch.isfinite(t.float()).all() for t in ref)
    for _ in range(30):
        got = fattn.attn_bwd(dq_, dk_, dv_, o, lse, dg, causal=causal, scale=scale)
        torch.cuda.synchronize()
        assert all(torch.equal(a, b) for a, b in zip(got, ref))
    assert fattn.device_status() == 0

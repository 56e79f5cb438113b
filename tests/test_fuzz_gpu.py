"""Seeded random sweep over the forward's parameters through the general
entry point (attn_fwd_strided): head dims 64/96/128/256, bf16 and fp16,
queries against equal or longer key sequences, causal or not, fixed or
automatic splits, contiguous or packed strided layouts; each case against
the fp64 oracle element by element, and the bf16 cases once more on both
places V can be rounded to fp16 (same bits)."""
import os
import random
import zlib

import pytest
import torch

import oracle
from tests.parity import assert_parity, compare
from tiled_online_softmax_fwd_gb300 import build as fbuild
from tiled_online_softmax_fwd_gb300 import fattn
from tiled_online_softmax_fwd_gb300.inputs import make_qkv_kv

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not os.path.exists(fattn.library_path()):
        fbuild.build()
    lib = fattn.load()
    yield lib
    torch.cuda.synchronize()
    assert fattn.device_status() == 0, "a kernel reported a pipeline timeout"


def draw(seed):
    rng = random.Random(seed)
    d = rng.choice([64, 96, 128, 256])
    B, H = rng.randint(1, 3), rng.randint(1, 4)
    causal = rng.random() < 0.6
    Nq = rng.choice([1, rng.randint(2, 130), rng.randint(131, 700)])
    Nk = Nq if rng.random() < 0.4 else Nq + rng.randint(0, 2500)
    # keep the oracle's work small
    while B * H * Nq * Nk * d > 1.5e8 and Nk > Nq:
        Nk = max(Nq, Nk // 2)
    while B * H * Nq * Nk * d > 1.5e8:
        Nq, Nk = max(1, Nq // 2), max(1, Nk // 2) if not causal else max(Nq // 2, Nk // 2)
    if causal and Nk < Nq:
        Nk = Nq
    splits = rng.choice([0, 1, rng.randint(2, 8)])
    dtype = rng.choice([torch.bfloat16, torch.float16])
    packed = rng.random() < 0.5
    sigma = rng.choice([1.0, 2.0, 3.0])
    return dict(B=B, H=H, Nq=Nq, Nk=Nk, d=d, causal=causal, splits=splits, dtype=dtype,
                packed=packed, sigma=sigma)


CASES = [draw(1000 + i) for i in range(40)]


def case_id(c):
    return "B%dH%dNq%dNk%dd%d%s_s%d_%s%s" % (c["B"], c["H"], c["Nq"], c["Nk"], c["d"],
                                             "c" if c["causal"] else "", c["splits"],
                                             "f16" if c["dtype"] == torch.float16 else "bf16",
                                             "_packed" if c["packed"] else "")


@pytest.mark.parametrize("case", CASES, ids=[case_id(c) for c in CASES])
def test_fuzz_matches_oracle(case):
    B, H, Nq, Nk, d = case["B"], case["H"], case["Nq"], case["Nk"], case["d"]
    q, k, v = make_qkv_kv(B, H, Nq, Nk, d, seed=zlib.crc32(case_id(case).encode()) % 100000,
                          sigma_qk=case["sigma"], dtype=case["dtype"])
    if case["packed"]:  # k and v interleaved in one [B, Nk, 2, H, d] buffer
        kv = torch.empty((B, Nk, 2, H, d), dtype=case["dtype"], device="cuda")
        kv[:, :, 0] = k.permute(0, 2, 1, 3).cuda()
        kv[:, :, 1] = v.permute(0, 2, 1, 3).cuda()
        dk, dv = kv[:, :, 0].permute(0, 2, 1, 3), kv[:, :, 1].permute(0, 2, 1, 3)
    else:
        dk, dv = k.cuda(), v.cuda()
    o, lse = fattn.attn_fwd_strided(q.cuda(), dk, dv, causal=case["causal"],
                                    num_splits=case["splits"])
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle.attn_fwd_kv(q, k, v, fattn.default_scale(d), case["causal"])
    r = compare(o.float().cpu().reshape(-1, d), lse.cpu().reshape(-1), o_ref, lse_ref)
    assert_parity(r, case_id(case))


BF16_CASES = [c for c in CASES if c["dtype"] == torch.bfloat16]


@pytest.mark.parametrize("case", BF16_CASES, ids=[case_id(c) for c in BF16_CASES])
def test_fuzz_v_rounding_routes_agree(case):
    """The same bf16 cases with V rounded on chip and by the pre-pass (which
    also gathers the packed layout): the bits must agree."""
    B, H, Nq, Nk, d = case["B"], case["H"], case["Nq"], case["Nk"], case["d"]
    q, k, v = make_qkv_kv(B, H, Nq, Nk, d, seed=zlib.crc32(case_id(case).encode()) % 100000,
                          sigma_qk=case["sigma"], dtype=case["dtype"])
    if case["packed"]:
        kv = torch.empty((B, Nk, 2, H, d), dtype=case["dtype"], device="cuda")
        kv[:, :, 0] = k.permute(0, 2, 1, 3).cuda()
        kv[:, :, 1] = v.permute(0, 2, 1, 3).cuda()
        dk, dv = kv[:, :, 0].permute(0, 2, 1, 3), kv[:, :, 1].permute(0, 2, 1, 3)
    else:
        dk, dv = k.cuda(), v.cuda()
    dq = q.cuda()
    outs = []
    for mode in ("on_chip", "prepass"):
        with fattn.v_conversion(mode):
            o, lse = fattn.attn_fwd_strided(dq, dk, dv, causal=case["causal"],
                                            num_splits=case["splits"])
            torch.cuda.synchronize()
        outs.append((o, lse))
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])


# ---------------------------------------------------------------- backward
def draw_bwd(seed):
    rng = random.Random(seed)
    d = rng.choice([64, 128])
    B, H = rng.randint(1, 3), rng.randint(1, 3)
    N = rng.choice([1, rng.randint(2, 130), rng.randint(131, 600)])
    while B * H * N * N * d > 6e7:
        N = max(1, N // 2)
    return dict(B=B, H=H, N=N, d=d, causal=rng.random() < 0.6, sigma=rng.choice([0.5, 1.0, 2.0]))


BWD_CASES = [draw_bwd(5000 + i) for i in range(20)]


@pytest.mark.parametrize("case", BWD_CASES,
                         ids=["B%dH%dN%dd%d%s_sig%g" % (c["B"], c["H"], c["N"], c["d"],
                                                        "c" if c["causal"] else "", c["sigma"])
                              for c in BWD_CASES])
def test_fuzz_backward_matches_oracle(case):
    """Random shapes through attn_bwd against the oracle's gradients, with the
    backward tests' tolerances (max |delta| <= 2e-2 max |ref| + 1e-5, mean
    |delta| <= 1e-2 mean |ref| + 1e-6 per tensor)."""
    import numpy as np
    B, H, N, d = case["B"], case["H"], case["N"], case["d"]
    q, k, v = make_qkv_kv(B, H, N, N, d, seed=zlib.crc32(repr(case).encode()) % 100000,
                          sigma_qk=case["sigma"])
    g = torch.Generator("cpu").manual_seed(N + d)
    dout = torch.randn(q.shape, generator=g).to(torch.bfloat16)
    scale = fattn.default_scale(d)
    dq_, dk_, dv_ = q.cuda(), k.cuda(), v.cuda()
    o, lse = fattn.attn_fwd(dq_, dk_, dv_, causal=case["causal"], scale=scale)
    grads = fattn.attn_bwd(dq_, dk_, dv_, o, lse, dout.cuda(), causal=case["causal"], scale=scale)
    torch.cuda.synchronize()
    refs = oracle.attn_bwd(q, k, v, dout, scale, case["causal"])
    for name, got, ref in zip(("dq", "dk", "dv"), grads, refs):
        got = got.cpu().double().numpy().reshape(ref.shape)
        assert np.all(np.isfinite(got)), name
        err = np.abs(got - ref)
        assert err.max() <= 2e-2 * np.abs(ref).max() + 1e-5, (name, err.max(), np.abs(ref).max())
        assert err.mean() <= 1e-2 * np.abs(ref).mean() + 1e-6, (name, err.mean(), np.abs(ref).mean())

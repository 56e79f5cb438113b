"""GPU regression tests for specific failure modes found earlier, each against
the fp64 oracle."""
import os

import pytest
import torch

import oracle
from tests.parity import assert_parity, compare
from tiled_online_softmax_fwd_gb300 import build as fbuild
from tiled_online_softmax_fwd_gb300 import fattn
from tiled_online_softmax_fwd_gb300.inputs import make_qkv

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not os.path.exists(fattn.library_path()):
        fbuild.build()
    lib = fattn.load()
    yield lib
    torch.cuda.synchronize()
    assert fattn.device_status() == 0, "a kernel reported a pipeline timeout"


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("d", [64, 96, 128, 256])
@pytest.mark.parametrize("causal", [False, True])
def test_all_scores_very_negative(dtype, d, causal):
    """Every score of every row is about -60 (natural log): the running max
    must be the row's own maximum, not a value clamped at 0 (with a base of 0
    the probabilities 2^(s*log2e) underflow fp16 and O collapses).  The row
    max once read four columns past the end of the score row."""
    B, H, N = 1, 2, 300
    g = torch.Generator("cpu").manual_seed(d)
    u = torch.rand(d, generator=g) + 0.5
    u = u / u.norm()
    jitter = 0.02 * torch.randn((B, H, N, d), generator=g)
    q = (-u * (60.0 * d) ** 0.5 + jitter).to(dtype)
    k = (u * (d ** 0.5 / 1.0) ** 0.5 * (d ** 0.25) + jitter).to(dtype)
    v = torch.randn((B, H, N, d), generator=g).to(dtype)
    o, lse = fattn.attn_fwd_strided(q.cuda(), k.cuda(), v.cuda(), causal=causal)
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, fattn.default_scale(d), causal)
    assert float(lse_ref.max()) < -20.0   # the scores really are very negative
    r = compare(o.float().cpu().reshape(-1, d), lse.cpu().reshape(-1), o_ref, lse_ref)
    assert_parity(r, "negative scores d%d" % d)


@pytest.mark.parametrize("d", [64, 128, 256])
def test_fp16_causal_first_row_wide_logits(d):
    """fp16, causal, Q/K ~ N(0, 9): row 0 of each head sees one key and must
    equal v_0 (the case the random sweep caught)."""
    q, k, v = make_qkv(3, 4, 26, d, seed=8, sigma_qk=3.0, dtype=torch.float16)
    o, lse = fattn.attn_fwd_fp16(q.cuda(), k.cuda(), v.cuda(), causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o[:, :, 0].cpu(), v[:, :, 0])
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, fattn.default_scale(d), True)
    assert_parity(compare(o.float().cpu().reshape(-1, d), lse.cpu().reshape(-1), o_ref, lse_ref), "fp16 first row d%d" % d)

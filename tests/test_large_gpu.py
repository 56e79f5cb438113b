"""GPU parity at sizes far past the other tests: one head of a million
queries, tensors of 2^31 elements (element offsets past the 32-bit range,
checked on the last heads), and a decode row against four million cached keys.
The inputs are drawn on the device from seeded generators; the oracle gets the
same bytes of the heads it checks, and checks sampled rows of them.

Every index these sizes reach was checked by reading to be 64-bit on both the
host and the device side (row pointers, lse offsets, partial-result slots)."""
import os

import pytest
import torch

import oracle
from tests.parity import assert_parity, compare
from tiled_online_softmax_fwd_gb300 import build as fbuild
from tiled_online_softmax_fwd_gb300 import fattn

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not os.path.exists(fattn.library_path()):
        fbuild.build()
    lib = fattn.load()
    yield lib
    torch.cuda.synchronize()
    assert fattn.device_status() == 0, "a kernel reported a pipeline timeout"


def device_qkv(shape_q, shape_kv, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    q = torch.randn(shape_q, generator=g, device="cuda", dtype=torch.bfloat16)
    k = torch.randn(shape_kv, generator=g, device="cuda", dtype=torch.bfloat16)
    v = torch.randn(shape_kv, generator=g, device="cuda", dtype=torch.bfloat16)
    return q, k, v


def check_heads(name, q, k, v, o, lse, heads, rows, causal, scale):
    """Compare rows `rows` (query indices) of the listed (b, h) heads with the
    oracle run on those heads alone."""
    d = q.shape[-1]
    for b, h in heads:
        qh, kh, vh = (t[b:b + 1, h:h + 1].cpu() for t in (q, k, v))
        if kh.shape[2] == qh.shape[2]:
            o_ref, lse_ref = oracle.attn_fwd(qh, kh, vh, scale, causal, rows=rows)
        else:
            o_ref, lse_ref = oracle.attn_fwd_kv(qh, kh, vh, scale, causal, rows=rows)
        idx = torch.as_tensor(rows, dtype=torch.int64)
        og = o[b, h].cpu().reshape(-1, d)[idx]
        lg = lse[b, h].cpu().reshape(-1)[idx]
        assert_parity(compare(og, lg, o_ref, lse_ref),
                      "%s head (%d, %d)" % (name, b, h))


@pytest.mark.parametrize("d,causal", [(64, False), (128, True)])
def test_one_head_of_a_million_queries(d, causal):
    N = 1 << 20
    q, k, v = device_qkv((1, 1, N, d), (1, 1, N, d), seed=11 + d)
    scale = fattn.default_scale(d)
    o, lse = fattn.attn_fwd(q, k, v, causal=causal, scale=scale)
    torch.cuda.synchronize()
    g = torch.Generator("cpu").manual_seed(5)
    rows = sorted(set([0, 1, 127, 128, N - 129, N - 1] +
                      torch.randint(0, N, (10,), generator=g).tolist()))
    check_heads("N=2^20 d%d" % d, q, k, v, o, lse, [(0, 0)], rows, causal, scale)
    del q, k, v, o, lse
    torch.cuda.empty_cache()


@pytest.mark.parametrize("B,H,N,d", [(256, 64, 2048, 64), (1, 8192, 2048, 128)])
def test_tensors_of_two_to_the_31_elements(B, H, N, d):
    assert B * H * N * d == 1 << 31
    q, k, v = device_qkv((B, H, N, d), (B, H, N, d), seed=B + H)
    scale = fattn.default_scale(d)
    o, lse = fattn.attn_fwd(q, k, v, causal=True, scale=scale)
    torch.cuda.synchronize()
    # The first head and the last ones (element offsets past 2^31).
    heads = [(0, 0), (B - 1, H - 1), (B - 1, H - 2)]
    rows = [0, 1, 200, 1023, 1024, N - 2, N - 1]
    check_heads("B%dH%dN%dd%d" % (B, H, N, d), q, k, v, o, lse, heads, rows, True, scale)
    del q, k, v, o, lse
    torch.cuda.empty_cache()


def test_decode_row_against_four_million_keys():
    Nk = 1 << 22
    q, k, v = device_qkv((1, 2, 1, 128), (1, 2, Nk, 128), seed=3)
    scale = fattn.default_scale(128)
    o, lse = fattn.attn_fwd_kv(q, k, v, causal=True, scale=scale)
    torch.cuda.synchronize()
    check_heads("decode Nk=2^22", q, k, v, o, lse, [(0, 0), (0, 1)], [0], True, scale)
    del q, k, v, o, lse
    torch.cuda.empty_cache()

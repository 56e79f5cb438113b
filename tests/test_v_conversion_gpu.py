"""GPU tests of the two places V is rounded to fp16 for bf16 inputs (P in
fp16): on chip by the forward kernel's converter warps, or once per call by
the pre-pass kernel into pooled scratch.  Both use the same rounding, so:
  * every entry point gives the same bits on either route (contiguous and
    strided V, split and unsplit, every head dimension);
  * repeated calls with new V each time (the pool hands the same scratch
    back) keep giving the on-chip route's bits;
  * the pre-pass route meets the oracle bounds on its own;
  * a V element beyond the fp16 range is reported as FATTN_ERR_RANGE on the
    pre-pass route too;
  * a call captured into a CUDA graph takes no scratch (it converts on chip)
    and replays to the same bits;
  * the scratch pool can be trimmed between calls.
"""
import os

import pytest
import torch

import oracle
from tests.parity import assert_parity, compare
from tiled_online_softmax_fwd_gb300 import build as fbuild
from tiled_online_softmax_fwd_gb300 import fattn
from tiled_online_softmax_fwd_gb300.inputs import make_qkv

pytestmark = pytest.mark.gpu

RANGE, ROLE_EPILOGUE = 5, 4


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not os.path.exists(fattn.library_path()):
        fbuild.build()
    lib = fattn.load()
    torch.cuda.synchronize()
    fattn.device_status()  # start from a clear status word
    yield lib


ROUTES = ("on_chip", "prepass")


def _routes(fn):
    """fn's (o, lse) on each route, asserted bit-identical."""
    outs = []
    for mode in ROUTES:
        with fattn.v_conversion(mode):
            o, lse = fn()
            torch.cuda.synchronize()
        outs.append((o.clone(), lse.clone()))
    assert fattn.device_status() == 0
    for mode, (o, lse) in zip(ROUTES[1:], outs[1:]):
        assert torch.equal(o, outs[0][0]) and torch.equal(lse, outs[0][1]), mode
    return outs


SHAPES = [(1, 2, 1000, 256, True), (2, 1, 777, 256, False), (2, 3, 700, 128, False),
          (1, 4, 640, 96, True), (1, 2, 4096, 64, False), (1, 1, 130, 128, True)]


@pytest.mark.parametrize("B,H,N,d,causal", SHAPES)
def test_routes_give_the_same_bits_and_meet_the_oracle(B, H, N, d, causal):
    q, k, v = make_qkv(B, H, N, d, seed=1300 + d + N, sigma_qk=2.0)
    dq, dk, dv = q.cuda(), k.cuda(), v.cuda()
    scale = fattn.default_scale(d)
    (o1, l1), (o2, l2) = _routes(
        lambda: fattn.attn_fwd(dq, dk, dv, causal=causal, scale=scale))
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, scale, causal)
    r = compare(o2.cpu().reshape(-1, d), l2.cpu().reshape(-1), o_ref, lse_ref)
    assert_parity(r, "pre-pass route B%d H%d N%d d%d" % (B, H, N, d))


@pytest.mark.parametrize("d,splits", [(256, 3), (128, 4), (64, 8)])
def test_split_calls_give_the_same_bits(d, splits):
    q, k, v = make_qkv(1, 2, 2048, d, seed=1400 + d)
    dq, dk, dv = q.cuda(), k.cuda(), v.cuda()
    (o1, l1), (o2, l2) = _routes(
        lambda: fattn.attn_fwd_split(dq, dk, dv, causal=True, num_splits=splits))
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    # A split changes the merge, not the rounding of V: attn_fwd's bits are
    # not expected, the oracle's bounds are.
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, fattn.default_scale(d), True)
    r = compare(o2.cpu().reshape(-1, d), l2.cpu().reshape(-1), o_ref, lse_ref)
    assert_parity(r, "pre-pass split d%d" % d)


@pytest.mark.parametrize("d", [256, 128])
def test_strided_v_gives_the_same_bits(d):
    """q, k, v sliced from one packed [B, N, 3, H, d] projection output: V's
    row stride is 3*H*d and its head stride d, so the pre-pass gathers."""
    B, H, N = 2, 3, 600
    g = torch.Generator().manual_seed(1500 + d)
    packed = torch.randn(B, N, 3, H, d, generator=g).to(torch.bfloat16).cuda()
    q, k, v = (packed[:, :, i].permute(0, 2, 1, 3) for i in range(3))
    assert not v.is_contiguous()
    (o1, l1), (o2, l2) = _routes(lambda: fattn.attn_fwd_strided(q, k, v, causal=True))
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    qc, kc, vc = (t.contiguous().cpu() for t in (q, k, v))
    o_ref, lse_ref = oracle.attn_fwd(qc, kc, vc, fattn.default_scale(d), True)
    r = compare(o2.cpu().reshape(-1, d), l2.cpu().reshape(-1), o_ref, lse_ref)
    assert_parity(r, "pre-pass strided d%d" % d)


def test_kv_and_host_entry_points_give_the_same_bits():
    q, k, v = make_qkv(1, 2, 1024, 256, seed=1600)
    dq, dk, dv = q.cuda(), k.cuda(), v.cuda()
    (o1, l1), (o2, l2) = _routes(lambda: fattn.attn_fwd_kv(dq[:, :, -300:].contiguous(),
                                                                dk, dv, causal=True))
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    hq, hk, hv = q.pin_memory(), k.pin_memory(), v.pin_memory()
    outs = []
    for mode in ROUTES:
        ho = torch.empty_like(q).pin_memory()
        hl = torch.empty(q.shape[:3], dtype=torch.float32).pin_memory()
        with fattn.v_conversion(mode):
            fattn.attn_fwd_host(hq, hk, hv, ho, hl, dq.clone(), dk.clone(), dv.clone(),
                                torch.empty_like(dq), torch.empty(q.shape[:3], device="cuda"),
                                causal=False)
        outs.append((ho, hl))
    for o, lse in outs[1:]:
        assert torch.equal(outs[0][0], o) and torch.equal(outs[0][1], lse)


@pytest.mark.parametrize("B,H,N,d,causal", [(2, 8, 4096, 128, True), (2, 4, 2048, 256, True)])
def test_prepass_scratch_is_never_stale(B, H, N, d, causal):
    """Eight calls in a row, each with new V: the pool hands the same scratch
    back, so a forward launch that read the copy before the pre-pass wrote it
    would see the previous call's values."""
    q, k, _ = make_qkv(B, H, N, d, seed=2000 + d)
    dq, dk = q.cuda(), k.cuda()
    for call in range(8):
        dv = make_qkv(B, H, N, d, seed=2100 + call)[2].cuda()
        with fattn.v_conversion("on_chip"):
            ref_o, ref_l = fattn.attn_fwd(dq, dk, dv, causal=causal)
        with fattn.v_conversion("prepass"):
            o, lse = fattn.attn_fwd(dq, dk, dv, causal=causal)
        torch.cuda.synchronize()
        assert torch.equal(o, ref_o) and torch.equal(lse, ref_l), "call %d" % call
    assert fattn.device_status() == 0


def test_auto_takes_the_prepass_where_planned():
    with fattn.v_conversion("auto"):
        assert fattn.v_conversion_route(16384, 128, True) == "prepass"  # the headline shape
        assert fattn.v_conversion_route(4096, 128, True) != "prepass"   # 4 x 16 heads of 4096
        assert fattn.v_conversion_route(65536, 64, False) == "prepass"
        assert fattn.v_conversion_route(4096, 64, False) != "prepass"
        assert fattn.v_conversion_route(8192, 256, True) == "prepass"
    with fattn.v_conversion("prepass"):
        assert fattn.v_conversion_route(1, 64, False) == "prepass"
    with fattn.v_conversion("on_chip"):
        assert fattn.v_conversion_route(1 << 20, 256, False) == "on_chip"


@pytest.mark.parametrize("d", [256, 128])
def test_out_of_range_v_is_reported_on_the_prepass_route(d):
    q, k, v = make_qkv(1, 1, 512, d, seed=1700 + d)
    v[0, 0, 100, 7] = 7.0e4
    with fattn.v_conversion("prepass"):
        fattn.attn_fwd(q.cuda(), k.cuda(), v.cuda(), causal=False)
        torch.cuda.synchronize()
    word = fattn.device_status()
    assert word & 0xff == RANGE and (word >> 8) & 0xff == ROLE_EPILOGUE, hex(word)
    assert fattn.device_status() == 0  # read and cleared


def test_graph_capture_converts_on_chip_and_replays():
    q, k, v = make_qkv(1, 2, 1024, 256, seed=1800)
    dq, dk, dv = q.cuda(), k.cuda(), v.cuda()
    o = torch.empty_like(dq)
    lse = torch.empty(dq.shape[:3], device="cuda")
    with fattn.v_conversion("prepass"):
        ref_o, ref_l = fattn.attn_fwd(dq, dk, dv, causal=True)
        torch.cuda.synchronize()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):  # warm-up on the capture stream
            fattn.attn_fwd(dq, dk, dv, causal=True, out=o, lse=lse, stream=s)
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        o.fill_(float("nan"))
        with torch.cuda.graph(graph):
            fattn.attn_fwd(dq, dk, dv, causal=True, out=o, lse=lse,
                           stream=torch.cuda.current_stream())
        graph.replay()
        torch.cuda.synchronize()
    assert torch.equal(o, ref_o) and torch.equal(lse, ref_l)


def test_trim_between_calls():
    q, k, v = make_qkv(1, 2, 1024, 256, seed=1900)
    dq, dk, dv = q.cuda(), k.cuda(), v.cuda()
    with fattn.v_conversion("prepass"):
        a, la = fattn.attn_fwd(dq, dk, dv, causal=True)
        torch.cuda.synchronize()
        fattn.trim_scratch()
        b, lb = fattn.attn_fwd(dq, dk, dv, causal=True)
        fattn.trim_scratch()  # with the call possibly still in flight
        torch.cuda.synchronize()
    assert torch.equal(a, b) and torch.equal(la, lb)

"""GPU parity tests: libfattn (through its C ABI) against the fp64 oracle on
the same seeded inputs, element by element, plus the exactness probes the
method fixes (identical value rows, zero queries, the causal first row, N=1)
and the edge cases (empty, ragged, many heads, streams, host entry point).

Set FATTN_PARITY_REPORT=<path> to append one JSON line per compared case."""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from tests.parity import assert_parity, compare
from tiled_online_softmax_fwd_gb300 import build as fbuild
from tiled_online_softmax_fwd_gb300 import fattn
from tiled_online_softmax_fwd_gb300.inputs import WORKLOADS, WORKLOAD_ORDER, make_qkv, make_workload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not os.path.exists(fattn.library_path()):
        fbuild.build()
    lib = fattn.load()
    yield lib
    torch.cuda.synchronize()
    assert fattn.device_status() == 0, "a kernel reported a pipeline timeout"


def report(case: str, r: dict):
    path = os.environ.get("FATTN_PARITY_REPORT")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps({"case": case, **r}) + "\n")


def gpu_run(q, k, v, causal, scale, entry=fattn.attn_fwd):
    dq, dk, dv = q.cuda(), k.cuda(), v.cuda()
    o, lse = entry(dq, dk, dv, causal=causal, scale=scale)
    torch.cuda.synchronize()
    return o.cpu(), lse.cpu()


def check_case(name, q, k, v, causal, scale, rows=None, entry=fattn.attn_fwd):
    o, lse = gpu_run(q, k, v, causal, scale, entry)
    B, H, N, d = q.shape
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, scale, causal, rows=rows)
    of, lf = o.reshape(-1, d), lse.reshape(-1)
    if rows is not None:
        idx = torch.as_tensor(rows, dtype=torch.int64)
        of, lf = of[idx], lf[idx]
    r = compare(of, lf, o_ref, lse_ref)
    report(name, r)
    assert_parity(r, name)
    return o, lse


# ----------------------------------------------------------------- small cases
SMALL = []
for N in (1, 2, 17, 64, 127, 128, 129, 200, 255, 256, 257, 383, 384, 513, 1000):
    for d in (64, 128):
        for causal in (False, True):
            SMALL.append((2, 3, N, d, causal))


@pytest.mark.parametrize("B,H,N,d,causal", SMALL,
                         ids=["B%dH%dN%dd%d%s" % (b, h, n, d, "c" if c else "") for b, h, n, d, c in SMALL])
def test_small_cases_match_oracle(B, H, N, d, causal):
    q, k, v = make_qkv(B, H, N, d, seed=1000 + N * 4 + d + causal)
    check_case("small_B%dH%dN%dd%d_c%d" % (B, H, N, d, causal), q, k, v, causal,
               fattn.default_scale(d))


@pytest.mark.parametrize("B,H,N,d,causal", [(3, 50, 384, 128, True), (2, 160, 256, 64, False),
                                            (1, 7, 1280, 64, True), (5, 3, 700, 128, False)])
def test_many_units_per_cta(B, H, N, d, causal):
    """More work units than SMs: every CTA loops over several units."""
    q, k, v = make_qkv(B, H, N, d, seed=77 + N)
    check_case("units_B%dH%dN%dd%d_c%d" % (B, H, N, d, causal), q, k, v, causal,
               fattn.default_scale(d))


@pytest.mark.parametrize("sigma", [3.0, 6.0])
def test_wide_logit_range(sigma):
    """Large logits: the running max moves a lot and the rescale path runs."""
    q, k, v = make_qkv(2, 4, 1024, 128, seed=5, sigma_qk=sigma)
    check_case("wide_sigma%g" % sigma, q, k, v, True, fattn.default_scale(128))


def test_other_scales():
    q, k, v = make_qkv(1, 2, 300, 64, seed=9)
    for scale in (1.0, 0.01, 0.3):
        check_case("scale%g" % scale, q, k, v, False, scale)


# ----------------------------------------------------------------- workloads
@pytest.mark.parametrize("name", WORKLOAD_ORDER)
def test_workload_matches_oracle(name):
    """The five workloads at full size, in the launch configuration the
    benchmark times.  The oracle checks every row of the first four (about a
    minute of host-core time for the 16K-token causal one) and, for the
    2 x 8 x 65536-row workload, 1024 seeded rows per head, each against all
    of its keys."""
    w = WORKLOADS[name]
    q, k, v, rows = make_workload(w)
    check_case("workload_" + name, q, k, v, w.causal, w.scale,
               rows=None if rows is None else rows.numpy())


@pytest.mark.parametrize("name", WORKLOAD_ORDER)
def test_workload_matches_simt_kernel(name):
    """Every row at full size against the independent SIMT kernel (fp32 P):
    the two GPU paths must agree within the sum of their tolerances."""
    w = WORKLOADS[name]
    q, k, v, _ = make_workload(w)
    dq, dk, dv = q.cuda(), k.cuda(), v.cuda()
    o1, l1 = fattn.attn_fwd(dq, dk, dv, causal=w.causal, scale=w.scale)
    o2, l2 = fattn.attn_fwd_simt(dq, dk, dv, causal=w.causal, scale=w.scale)
    torch.cuda.synchronize()
    do = (o1.float() - o2.float()).abs()
    dl = (l1 - l2).abs()
    r = {"o_max": float(do.max()), "o_mean": float(do.mean()), "lse_max": float(dl.max())}
    report("simt_vs_tcgen05_" + name, r)
    assert torch.isfinite(o1.float()).all() and torch.isfinite(l1).all()
    assert r["o_max"] <= 4e-2 and r["o_mean"] <= 2e-3 and r["lse_max"] <= 2e-3, r


# ----------------------------------------------------------------- exactness probes
@pytest.mark.parametrize("causal", [False, True])
def test_identical_value_rows(causal):
    """All V rows equal w  =>  every output row equals w."""
    B, H, N, d = 2, 2, 700, 128
    q, k, _ = make_qkv(B, H, N, d, seed=11, sigma_qk=3.0)
    w = torch.randn(B, H, 1, d, generator=torch.Generator().manual_seed(12)).to(torch.bfloat16)
    v = w.expand(B, H, N, d).contiguous()
    o, _ = gpu_run(q, k, v, causal, fattn.default_scale(d))
    err = (o.float() - w.float()).abs().max().item()
    assert err <= 1e-2, err


@pytest.mark.parametrize("causal", [False, True])
def test_zero_queries(causal):
    """Q = 0  =>  uniform weights: O_i = mean of visible V rows, lse_i = ln(#visible)."""
    B, H, N, d = 1, 2, 640, 64
    _, k, v = make_qkv(B, H, N, d, seed=13)
    q = torch.zeros_like(k)
    o, lse = gpu_run(q, k, v, causal, fattn.default_scale(d))
    vd = v.double()
    if causal:
        ref = vd.cumsum(dim=2) / torch.arange(1, N + 1, dtype=torch.float64)[None, None, :, None]
        ref_lse = torch.log(torch.arange(1, N + 1, dtype=torch.float64))[None, None, :].expand(B, H, N)
    else:
        ref = vd.mean(dim=2, keepdim=True).expand(B, H, N, d)
        ref_lse = torch.full((B, H, N), float(np.log(N)), dtype=torch.float64)
    r = compare(o.reshape(-1, d), lse.reshape(-1), ref.reshape(-1, d).numpy(),
                ref_lse.reshape(-1).numpy())
    report("zero_queries_c%d" % causal, r)
    assert_parity(r, "zero queries")


def test_causal_first_row_is_exact():
    """Causal row 0 sees only key 0: o_0 == v_0 exactly, lse_0 = scale q_0.k_0."""
    B, H, N, d = 2, 3, 512, 128
    q, k, v = make_qkv(B, H, N, d, seed=17, sigma_qk=3.0)
    scale = fattn.default_scale(d)
    o, lse = gpu_run(q, k, v, True, scale)
    assert torch.equal(o[:, :, 0], v[:, :, 0])
    ref = scale * (q[:, :, 0].double() * k[:, :, 0].double()).sum(-1)
    assert (lse[:, :, 0].double() - ref).abs().max().item() <= 1e-3


@pytest.mark.parametrize("causal", [False, True])
def test_single_key(causal):
    """N = 1: O = v_0 exactly and lse = scale q.k."""
    q, k, v = make_qkv(4, 5, 1, 64, seed=19)
    scale = fattn.default_scale(64)
    o, lse = gpu_run(q, k, v, causal, scale)
    assert torch.equal(o, v)
    ref = scale * (q.double() * k.double()).sum(-1)
    assert (lse.double() - ref).abs().max().item() <= 1e-3


# ----------------------------------------------------------------- edge cases / API
def test_empty_inputs_are_noops():
    for shape in ((1, 2, 0, 64), (0, 2, 16, 64), (2, 0, 16, 128)):
        q = torch.empty(shape, dtype=torch.bfloat16, device="cuda")
        o, lse = fattn.attn_fwd(q, q, q, causal=True)
        torch.cuda.synchronize()
        assert o.shape == shape and lse.shape == shape[:3]


def test_deterministic():
    q, k, v = make_qkv(2, 8, 1500, 128, seed=23)
    dq, dk, dv = q.cuda(), k.cuda(), v.cuda()
    o1, l1 = fattn.attn_fwd(dq, dk, dv, causal=True)
    o2, l2 = fattn.attn_fwd(dq, dk, dv, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_side_stream_and_preallocated_outputs():
    q, k, v = make_qkv(1, 4, 777, 64, seed=29)
    dq, dk, dv = q.cuda(), k.cuda(), v.cuda()
    ref_o, ref_l = fattn.attn_fwd(dq, dk, dv)
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    out = torch.full_like(dq, float("nan"))
    lse = torch.full((1, 4, 777), float("nan"), device="cuda")
    with torch.cuda.stream(s):
        fattn.attn_fwd(dq, dk, dv, out=out, lse=lse, stream=s)
    s.synchronize()
    assert torch.equal(out, ref_o) and torch.equal(lse, ref_l)


@pytest.mark.parametrize("B,H,N,d", [(1, 4, 1000, 128), (2, 5, 700, 64), (3, 1, 300, 128),
                                     (1, 1, 129, 64), (2, 16, 256, 128), (1, 24, 4096, 64),
                                     (1, 24, 38912, 64)])
def test_host_entry_point_matches_device_path(B, H, N, d):
    """The pipelined host entry (copies and compute overlapped over chunks of
    heads, each chunk at least enough heads for one work unit per SM; on 152
    SMs: one chunk for the small shapes, three equal chunks of 8 heads for
    24 x 4096, and 1, 1, 4, 4, 3, 3, 3, 3, 1, 1 heads for 24 x 38912) gives
    the device path's bits."""
    q, k, v = make_qkv(B, H, N, d, seed=31 + B * H)
    hq, hk, hv = q.pin_memory(), k.pin_memory(), v.pin_memory()
    ho = torch.empty_like(hq).pin_memory()
    hl = torch.empty((B, H, N), dtype=torch.float32).pin_memory()
    dq, dk, dv = torch.empty_like(q, device="cuda"), torch.empty_like(k, device="cuda"), \
        torch.empty_like(v, device="cuda")
    do = torch.empty_like(dq)
    dl = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    fattn.attn_fwd_host(hq, hk, hv, ho, hl, dq, dk, dv, do, dl, causal=True)
    ref_o, ref_l = gpu_run(q, k, v, True, fattn.default_scale(d))
    assert torch.equal(ho, ref_o) and torch.equal(hl, ref_l)


def test_rejects_host_pointer_for_device_buffer():
    """A pinned host buffer passed as a device operand is refused, not read."""
    q = torch.zeros(1, 1, 64, 64, dtype=torch.bfloat16, device="cuda")
    hq = torch.zeros(1, 1, 64, 64, dtype=torch.bfloat16).pin_memory()
    o = torch.empty_like(q)
    lse = torch.empty(1, 1, 64, device="cuda")
    st = fattn.raw_call("attn_fwd", hq.data_ptr(), q.data_ptr(), q.data_ptr(), o.data_ptr(),
                        lse.data_ptr(), 1, 1, 64, 64, 0.125, 0, None)
    assert st == 1


def test_stalled_wait_reports_timeout_and_context_survives():
    """A pipeline wait that nothing satisfies gives up after its limit, records
    FATTN_ERR_TIMEOUT (role 5) in the device status word, and the context stays
    usable: a forward call afterwards is correct and leaves the word clear."""
    assert fattn.device_status() == 0
    fattn.selftest_wait_timeout(limit_us=20000)
    torch.cuda.synchronize()
    word = fattn.device_status()
    assert word & 0xff == 4 and (word >> 8) & 0xff == 5, hex(word)
    assert fattn.device_status() == 0  # reading clears it
    q, k, v = make_qkv(1, 2, 300, 128, seed=41)
    check_case("after_selftest", q, k, v, True, fattn.default_scale(128))
    assert fattn.device_status() == 0


# ----------------------------------------------------------------- key-range split
SPLIT_CASES = [(1, 1, 4096, 64, False, None), (1, 1, 4096, 64, True, None),
               (1, 2, 1000, 128, True, 3), (2, 1, 777, 64, False, 5),
               (1, 1, 300, 128, True, 2), (1, 3, 2048, 128, False, 16),
               (1, 1, 128, 64, False, 2), (1, 1, 4096, 128, True, 7), (3, 2, 513, 64, True, 64)]


@pytest.mark.parametrize("B,H,N,d,causal,splits", SPLIT_CASES,
                         ids=["B%dH%dN%dd%d%s_s%s" % (b, h, n, d, "c" if c else "", s)
                              for b, h, n, d, c, s in SPLIT_CASES])
def test_split_matches_oracle(B, H, N, d, causal, splits):
    """Key-range split + combine against the oracle (and close to the
    unsplit kernel)."""
    q, k, v = make_qkv(B, H, N, d, seed=500 + N + d, sigma_qk=2.0)
    scale = fattn.default_scale(d)
    dq, dk, dv = q.cuda(), k.cuda(), v.cuda()
    o, lse = fattn.attn_fwd_split(dq, dk, dv, causal=causal, scale=scale, num_splits=splits)
    o1, l1 = fattn.attn_fwd(dq, dk, dv, causal=causal, scale=scale)
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, scale, causal)
    r = compare(o.cpu().reshape(-1, d), lse.cpu().reshape(-1), o_ref, lse_ref)
    report("split_B%dH%dN%dd%d_c%d_s%s" % (B, H, N, d, causal, splits), r)
    assert_parity(r, "split")
    assert (o.float() - o1.float()).abs().max().item() <= 2 ** -5
    assert (lse - l1).abs().max().item() <= 1e-4


def test_split_count_fills_the_device():
    """The split count minimises the estimated time in key-tile steps:
    ceil(units * s / SMs) rounds of ceil(key tiles / s) + 3 steps, plus 6
    steps for the partials and their merge when s > 1."""
    n_sm = torch.cuda.get_device_properties(0).multi_processor_count
    units, tiles = 16, 32                      # B=1, H=1, N=4096: 16 pairs, 32 key tiles

    def est(s):
        return -(-units * s // n_sm) * (-(-tiles // s) + 3) + (6 if s > 1 else 0)
    s = fattn.split_count(1, 1, 4096, 64, False)
    assert 1 < s <= 16 and est(s) == min(est(x) for x in range(1, 17))
    assert fattn.split_count(1, 32, 16384, 128, True) == 1   # already more units than SMs


def test_split_workload_single_head():
    """The single-head N=4096 workload through the automatic split."""
    w = WORKLOADS["B1_H1_N4096_d64"]
    q, k, v, _ = make_workload(w)
    o, lse = fattn.attn_fwd_split(q.cuda(), k.cuda(), v.cuda(), causal=w.causal, scale=w.scale)
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, w.scale, w.causal)
    r = compare(o.cpu().reshape(-1, w.d), lse.cpu().reshape(-1), o_ref, lse_ref)
    report("split_workload_" + w.name, r)
    assert_parity(r, w.name)

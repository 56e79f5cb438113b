"""CPU tests of the C-ABI boundary: the library loads, exports every function
that include/*.h declares, and rejects bad arguments synchronously (these
checks run before any device call, so no GPU is needed)."""
import ctypes
import glob
import os
import re

import pytest

from tiled_online_softmax_fwd_gb300 import build as fbuild
from tiled_online_softmax_fwd_gb300 import fattn

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
OK, INVALID, UNSUPPORTED = 0, 1, 2


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(fattn.library_path()):
        fbuild.build()
    return fattn.load()


def declared_functions():
    names = []
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b([A-Za-z_]\w*)\s*\(", text, re.M)
    return sorted(set(n for n in names if n not in ("if", "defined")))


def test_header_declares_the_api():
    names = declared_functions()
    for n in ("attn_fwd", "attn_fwd_host", "attn_fwd_simt", "fattn_status_string",
              "fattn_last_cuda_error", "fattn_get_device_status", "fattn_version"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), "libfattn.so does not export %s" % name


def test_library_exports_nothing_else():
    nm = os.popen("nm -D --defined-only %s" % fattn.library_path()).read().split("\n")
    funcs = sorted(l.split()[-1] for l in nm if " T " in l)
    assert funcs == declared_functions(), funcs


def test_status_strings_and_version(lib):
    assert lib.fattn_status_string(0) == b"FATTN_OK"
    assert lib.fattn_status_string(1) == b"FATTN_ERR_INVALID_ARG"
    assert lib.fattn_status_string(4) == b"FATTN_ERR_TIMEOUT"
    assert lib.fattn_status_string(5) == b"FATTN_ERR_RANGE"
    assert lib.fattn_status_string(99) == b"FATTN_UNKNOWN_STATUS"
    assert fattn.version().startswith("libfattn")


A = 1 << 20  # a fake, 16-byte aligned address: never dereferenced by these calls


def call(lib, q=A, k=A + (1 << 24), v=A + (2 << 24), o=A + (3 << 24), lse=A + (4 << 24),
         B=1, H=2, N=64, d=64, scale=0.125, causal=0):
    return lib.attn_fwd(q, k, v, o, lse, B, H, N, d, scale, causal, None)


def test_empty_problems_are_noops(lib):
    # Nothing to do: OK without touching pointers or the device.
    assert call(lib, q=0, k=0, v=0, o=0, lse=0, N=0) == OK
    assert call(lib, q=0, k=0, v=0, o=0, lse=0, B=0) == OK
    assert call(lib, q=0, k=0, v=0, o=0, lse=0, H=0) == OK


@pytest.mark.parametrize("kw,expect", [
    (dict(B=-1), INVALID), (dict(H=-1), INVALID), (dict(N=-5), INVALID),
    (dict(d=80), UNSUPPORTED), (dict(d=0), UNSUPPORTED), (dict(d=512), UNSUPPORTED),
    (dict(scale=0.0), INVALID), (dict(scale=-1.0), INVALID),
    (dict(scale=float("nan")), INVALID), (dict(scale=float("inf")), INVALID),
    (dict(causal=2), INVALID), (dict(causal=-1), INVALID),
    (dict(q=0), INVALID), (dict(k=0), INVALID), (dict(v=0), INVALID), (dict(o=0), INVALID),
    (dict(lse=0), INVALID),
    (dict(q=A + 8), INVALID), (dict(o=A + (3 << 24) + 2), INVALID), (dict(lse=A + (4 << 24) + 4), INVALID),
    (dict(o=A), INVALID),                         # output aliases q
    (dict(o=A + 4096), INVALID),                  # output overlaps q
    (dict(lse=A + (3 << 24) + 4096), INVALID),    # lse inside o
    (dict(lse=A + (2 << 24)), INVALID),           # lse aliases v
    (dict(B=1 << 20, H=1 << 12, N=1), UNSUPPORTED),        # B*H beyond the tensor-map range
    (dict(B=1024, H=1024, N=1 << 20, d=128), UNSUPPORTED),  # tensor beyond 2^39 bytes
])
def test_bad_arguments_are_rejected(lib, kw, expect):
    assert call(lib, **kw) == expect


def test_inputs_may_alias_each_other_but_not_outputs(lib):
    # q == k == v is legal (self-attention on one buffer); validation then
    # proceeds to the device query, which is not reached for the output cases.
    assert call(lib, k=A, v=A, o=A) == INVALID


def test_host_entry_validates_before_copying(lib):
    f = lib.attn_fwd_host
    dev = [A, A + (1 << 24), A + (2 << 24), A + (3 << 24), A + (4 << 24)]
    host = [A + (10 << 24), A + (11 << 24), A + (12 << 24), A + (13 << 24), A + (14 << 24)]
    # a bad device buffer is reported before any copy
    assert f(*host, 0, *dev[1:], 1, 1, 64, 64, 0.125, 0, None) == INVALID
    # unsupported head dim
    assert f(*host, *dev, 1, 1, 64, 80, 0.125, 0, None) == UNSUPPORTED
    # empty problem
    assert f(0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 1, 1, 0, 64, 0.125, 0, None) == OK


def test_python_binding_checks(lib):
    import torch
    q = torch.zeros(1, 1, 8, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        fattn.attn_fwd(q, q, q)  # CPU tensors
    with pytest.raises(TypeError):
        fattn.attn_fwd(None, q, q)


def test_device_status_argument_check(lib):
    assert lib.fattn_get_device_status(ctypes.POINTER(ctypes.c_int)(), None) == INVALID


def test_selftest_limit_is_checked_before_any_device_call(lib):
    assert lib.fattn_selftest_wait_timeout(0, None) == INVALID
    assert lib.fattn_selftest_wait_timeout(2000001, None) == INVALID


def test_split_workspace_size(lib):
    f = lib.attn_fwd_split_workspace_size
    f.restype = ctypes.c_size_t
    assert f(1, 1, 4096, 64, 1) == 0                  # no split, no scratch
    rows = 4096
    o_bytes = 10 * rows * 64 * 4
    aligned = (o_bytes + 255) // 256 * 256
    assert f(1, 1, 4096, 64, 10) == aligned + 10 * rows * 8
    assert f(1, 1, 4096, 80, 2) == 0 and f(1, 1, 4096, 64, 0) == 0 and f(1, 1, 4096, 64, 65) == 0


def test_split_arguments_are_checked(lib):
    f = lib.attn_fwd_split
    base = [A, A + (1 << 24), A + (2 << 24), A + (3 << 24), A + (4 << 24), 1, 1, 4096, 64, 0.125, 0]
    ws = A + (8 << 24)
    assert f(*base, 0, ws, 1 << 30, None) == INVALID       # num_splits out of range
    assert f(*base, 65, ws, 1 << 30, None) == INVALID
    assert f(*base[:5], 1, 1, 4096, 80, 0.125, 0, 4, ws, 1 << 30, None) == UNSUPPORTED
    assert f(*base[:5], 1, 1, 0, 64, 0.125, 0, 4, 0, 0, None) == OK   # empty: no-op


def test_kv_workspace_size(lib):
    f = lib.attn_fwd_kv_workspace_size
    rows = 2 * 3 * 5                                   # B*H*Nq: the scratch follows the queries
    o_bytes = 7 * rows * 128 * 4
    assert f(2, 3, 5, 9000, 128, 1, 7) == (o_bytes + 255) // 256 * 256 + 7 * rows * 8
    assert f(2, 3, 5, 9000, 128, 0, 1) == 0
    assert f(2, 3, 5, 9000, 80, 0, 7) == 0 and f(2, 3, 5, 9000, 128, 0, 65) == 0
    assert f(2, 3, 5, 9000, 128, 0, -1) == 0 and f(2, 3, 5, 0, 128, 0, 7) == 0   # no keys
    assert f(2, 3, 5, -1, 128, 0, 7) == 0 and f(1, 1, 9, 5, 64, 1, 2) == 0   # Nq > Nk, causal


def test_kv_arguments_are_checked(lib):
    f = lib.attn_fwd_kv
    ptrs = [A, A + (1 << 24), A + (2 << 24), A + (3 << 24), A + (4 << 24)]
    ws = A + (8 << 24)

    def call(B, H, Nq, Nk, d, causal=0, splits=1, scale=0.125, p=ptrs):
        return f(*p, B, H, Nq, Nk, d, scale, causal, splits, ws, 1 << 30, None)
    assert call(1, 1, 10, 5, 64, causal=1) == INVALID      # more queries than keys under the mask
    assert call(1, 1, 10, 0, 64) == INVALID                # queries without keys
    assert call(1, 1, 10, -3, 64) == INVALID
    assert call(1, 1, 4, 8, 64, splits=-1) == INVALID
    assert call(1, 1, 4, 8, 64, splits=65) == INVALID
    assert call(1, 1, 4, 8, 64, causal=2) == INVALID
    assert call(1, 1, 4, 8, 64, scale=0.0) == INVALID
    assert call(1, 1, 4, 8, 80) == UNSUPPORTED
    assert call(1, 1, 4, 8, 64, p=[0] + ptrs[1:]) == INVALID
    assert call(1, 1, 4, 8, 64, p=ptrs[:3] + [A + 8] + ptrs[4:]) == INVALID   # misaligned o
    # o (4 rows) overlapping the end of k (8 rows of 64 bf16) is caught with k's own size
    assert call(1, 1, 4, 8, 64, p=ptrs[:3] + [ptrs[1] + 8 * 64 * 2 - 16] + ptrs[4:]) == INVALID
    assert call(1, 1, 0, 8, 64) == OK                      # no queries: no-op
    assert call(1, 1, 0, 0, 64, causal=1) == OK


def test_strided_arguments_are_checked(lib):
    f = lib.attn_fwd_strided
    L3 = ctypes.c_longlong * 3
    ptrs = [A, A + (1 << 24), A + (2 << 24), A + (3 << 24), A + (4 << 24)]
    B, H, N, d = 2, 3, 40, 64
    dense = L3(H * N * d, N * d, d)

    def call(qs=dense, ks=dense, vs=dense, os_=dense, p=ptrs, causal=0, dtype=0):
        return f(*p, B, H, N, N, d, qs, ks, vs, os_, 0.125, causal, 1, None, 0, dtype, None)
    assert call(qs=None) == INVALID
    assert call(dtype=3) == INVALID and call(dtype=-1) == INVALID
    assert call(os_=L3(H * N * d, N * d, d + 4)) == INVALID       # not a multiple of 8
    assert call(ks=L3(H * N * d, 0, d)) == INVALID                # zero stride, extent 3
    assert call(os_=L3(H * N * d, N * d, 32)) == INVALID          # o rows overlap (32 < d)
    assert call(os_=L3(N * d, N * d, d)) == INVALID               # o heads alias batches
    # o's span reaching into k's span
    assert call(p=ptrs[:3] + [ptrs[1] + 64] + ptrs[4:]) == INVALID
    # The layouts below pass the layout checks; with no device the call then
    # fails on the device query (with one, on the fake pointers).
    import torch
    if torch.cuda.is_available():
        return
    # q, k, v may overlap each other: one packed buffer [B][N][3][H][d]
    packed = L3(N * 3 * H * d, d, 3 * H * d)
    q0 = A
    p_packed = [q0, q0 + H * d * 2, q0 + 2 * H * d * 2, A + (5 << 24), A + (6 << 24)]
    assert call(qs=packed, ks=packed, vs=packed, p=p_packed) not in (INVALID, UNSUPPORTED)
    # o interleaved as [B][N][H][d] is a valid nesting
    assert call(os_=L3(N * H * d, d, H * d)) not in (INVALID, UNSUPPORTED)


def test_rowop_arguments_are_checked(lib):
    for f in (lib.fattn_softmax_rows, lib.fattn_row_sum):
        assert f(A, A + (1 << 24), -1, 4, 0, None) == INVALID      # negative M
        assert f(A, A + (1 << 24), 4, -1, 0, None) == INVALID      # negative N
        assert f(A, A + (1 << 24), 4, 4, 2, None) == INVALID       # unknown dtype
        assert f(0, A, 4, 4, 0, None) == INVALID                   # null input
        assert f(A + 2, A + (1 << 24), 4, 4, 0, None) == INVALID   # misaligned fp32
        assert f(0, 0, 0, 16, 0, None) == OK                       # empty: no-op
    assert lib.fattn_softmax_rows(A, A + 8, 4, 4, 0, None) == INVALID   # partial overlap
    assert lib.fattn_row_sum(A, A + 8, 4, 4, 0, None) == INVALID        # sums inside input


def test_v_conversion_setting(lib):
    """Host-only: the setting is a process-wide integer, no device call."""
    prev = lib.fattn_set_v_conversion(1)
    assert prev in (0, 1, 2)
    try:
        assert lib.fattn_set_v_conversion(3) == -1 and lib.fattn_set_v_conversion(-1) == -1
        assert lib.fattn_set_v_conversion(2) == 1  # the invalid calls changed nothing
        ON_CHIP, PREPASS = 1, 2
        assert lib.fattn_v_conversion_route(128, 64, 0) == PREPASS
        assert lib.fattn_v_conversion_route(0, 64, 0) == ON_CHIP  # nothing to convert
        assert lib.fattn_set_v_conversion(0) == 2
        # Automatic: visits = units per head (halved under the causal mask)
        # against 24 / 8 / 16 / 12 for d = 64 / 96 / 128 / 256.
        # The first N that takes the pre-pass, per (d, causal): e.g. d = 64
        # without the mask needs ceil(T/2) >= 24, T = ceil(N/128) >= 47.
        first = {(64, 0): 46 * 128 + 1, (64, 1): 94 * 128 + 1, (96, 0): 14 * 128 + 1,
                 (96, 1): 30 * 128 + 1, (128, 0): 30 * 128 + 1, (128, 1): 62 * 128 + 1,
                 (256, 0): 11 * 128 + 1, (256, 1): 23 * 128 + 1}
        for (d, causal), n in first.items():
            assert lib.fattn_v_conversion_route(n, d, causal) == PREPASS, (n, d, causal)
            assert lib.fattn_v_conversion_route(n - 1, d, causal) == ON_CHIP, (n - 1, d, causal)
        for n, d, causal, want in [(16384, 128, 1, 1), (4096, 128, 1, 0), (256, 64, 0, 0),
                                   (4096, 64, 0, 0), (65536, 64, 0, 1), (4096, 96, 1, 1),
                                   (8192, 256, 1, 1)]:
            assert lib.fattn_v_conversion_route(n, d, causal) == (PREPASS if want else ON_CHIP), (n, d)
        assert lib.fattn_v_conversion_route(512, 80, 0) == -1
        assert lib.fattn_v_conversion_route(-1, 128, 0) == -1
        assert lib.fattn_v_conversion_route(512, 128, 2) == -1
        assert fattn.set_v_conversion("on_chip") == "auto"
        with pytest.raises(ValueError):
            fattn.set_v_conversion("gpu")
    finally:
        lib.fattn_set_v_conversion(prev)


def test_trim_scratch_without_pools(lib):
    """No call has taken pre-pass scratch in this process (no GPU here), so
    there is no pool to trim: FATTN_OK without touching CUDA."""
    assert lib.fattn_trim_scratch() == OK


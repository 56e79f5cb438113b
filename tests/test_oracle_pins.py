"""CPU tests: the fp64 oracle against its pins, and planted mistakes in copies
of the oracle that the pins must catch."""
import ctypes
import os
import subprocess

import numpy as np
import pytest
import torch

import oracle
from tests import oracle_pins as pins


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda f: f.__name__)
def test_oracle_meets_pin(pin):
    pin(oracle.attn_fwd)


# Each planted mistake is a one-line edit of the oracle's C source (built into
# a temporary library on the CPU); at least one pin must reject it.
MUTANTS = {
    "kv_causal_offset_dropped": ("jb->causal ? i + (Nk - Nq) + 1 : Nk", "jb->causal ? i + 1 : Nk"),
    "kv_values_of_wrong_head": ("const double *vh = jb->v + head * Nk * d;",
                                "const double *vh = jb->v;"),
    "dropped_scale": ("s[j] = job->scale * dot;", "s[j] = dot;"),
    "causal_excludes_diagonal": ("job->causal ? i + 1 : N", "job->causal ? i : N"),
    "exp_sign_flipped": ("exp(s[j] - m)", "exp(m - s[j])"),
    "lse_log2": ("m + log(l)", "m + log2(l)"),
    "lse_without_max": ("job->lse[out_idx] = m + log(l);", "job->lse[out_idx] = log(l);"),
    "no_normalisation": ("oi[c] /= l;", "oi[c] /= 1.0;"),
    "values_reversed": ("const double *vj = vh + j * d;",
                        "const double *vj = vh + (n_keys - 1 - j) * d;"),
    "max_not_subtracted_in_exp": ("exp(s[j] - m)", "exp(s[j])"),
    "query_of_wrong_row": ("const double *qi = job->q + grow * d;",
                           "const double *qi = job->q + (head * N) * d;"),
}


@pytest.fixture(scope="module")
def mutant_dir(tmp_path_factory):
    return tmp_path_factory.mktemp("oracle_mutants")


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name, mutant_dir):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "attn_oracle.c")).read()
    old, new = MUTANTS[name]
    assert src.count(old) >= 1, "mutation anchor vanished: %r" % old
    c_path = os.path.join(mutant_dir, name + ".c")
    so_path = os.path.join(mutant_dir, name + ".so")
    with open(c_path, "w") as f:
        f.write(src.replace(old, new))
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-o", so_path,
                    c_path, "-lm"], check=True)
    fn = oracle.bind(so_path)
    failed = []
    lib = oracle._open(so_path)

    def fwd_kv(q, k, v, scale, causal, rows=None):
        qd, kd, vd = (oracle._as_f64(t) for t in (q, k, v))
        B, H, Nq, d = qd.shape
        o = np.zeros((B * H * Nq, d))
        lse = np.zeros(B * H * Nq)
        rc = lib.oracle_attn_fwd_kv(*(oracle._ptr(t) for t in (qd, kd, vd, o, lse)), B, H, Nq,
                                    kd.shape[2], d, float(scale), int(causal), None, B * H * Nq, 1)
        assert rc == 0
        return o, lse
    with np.errstate(all="ignore"):
        for pin in pins.ALL_PINS:
            try:
                pin(fn)
            except AssertionError:
                failed.append(pin.__name__)
        try:
            pins.pin_fwd_kv(fwd_kv, fn)
        except AssertionError:
            failed.append("pin_fwd_kv")
    assert failed, "planted mistake %s passed every pin" % name


def test_fwd_kv_oracle_meets_pins():
    pins.pin_fwd_kv(oracle.attn_fwd_kv, oracle.attn_fwd)


def test_bwd_oracle_meets_pins():
    pins.pin_bwd_autograd(oracle.attn_bwd)
    pins.pin_bwd_finite_difference(oracle.attn_bwd, oracle.attn_fwd)
    pins.pin_bwd_invariants(oracle.attn_bwd, oracle.attn_bwd_dq_rows, oracle.attn_bwd_dkv_rows)


BWD_MUTANTS = {
    "dq_without_scale": ("dqh[i * d + c] += jb->scale * ds * kh[j * d + c];",
                         "dqh[i * d + c] += ds * kh[j * d + c];"),
    "ds_without_D": ("const double ds = p[j] * (dp[j] - D);\n                for",
                     "const double ds = p[j] * dp[j];\n                for"),
    "dk_uses_k": ("dkh[j * d + c] += jb->scale * ds * qh[i * d + c];",
                  "dkh[j * d + c] += jb->scale * ds * kh[i * d + c];"),
    "dv_uses_ds": ("dvh[j * d + c] += p[j] * doh[i * d + c];",
                   "dvh[j * d + c] += (p[j] - 0.5 * p[j] * p[j]) * doh[i * d + c];"),
    "dp_wrong_operand": ("dot += doi[c] * vh[j * d + c];", "dot += doi[c] * kh[j * d + c];"),
    # the dk/dv rows mode
    "dkv_ds_without_D": ("const double ds = p * (dp - jb->D[i]);", "const double ds = p * dp;"),
    "dkv_D_unnormalised": ("jb->D[i] = acc / l;", "jb->D[i] = acc;"),
    "dkv_causal_skips_diagonal": ("for (int64_t i = jb->causal ? j : 0; i < N; ++i) {",
                                  "for (int64_t i = jb->causal ? j + 1 : 0; i < N; ++i) {"),
    "dkv_dv_weight_unnormalised": ("const double p = exp(jb->scale * dot - jb->m[i]) / jb->l[i];",
                                   "const double p = exp(jb->scale * dot - jb->m[i]);"),
}


@pytest.mark.parametrize("name", sorted(BWD_MUTANTS))
def test_bwd_planted_mistake_is_caught(name, mutant_dir):
    here = os.path.dirname(oracle.__file__)
    src = open(os.path.join(here, "attn_bwd_oracle.c")).read()
    old, new = BWD_MUTANTS[name]
    assert src.count(old) >= 1, "mutation anchor vanished: %r" % old
    c_path = os.path.join(mutant_dir, "bwd_" + name + ".c")
    so_path = os.path.join(mutant_dir, "bwd_" + name + ".so")
    with open(c_path, "w") as f:
        f.write(src.replace(old, new))
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-o", so_path,
                    os.path.join(here, "attn_oracle.c"), os.path.join(here, "rowops_oracle.c"),
                    c_path, "-lm"], check=True)
    lib = oracle._open(so_path)

    def attn_bwd(q, k, v, dout, scale, causal):
        qd, kd, vd, dd = (oracle._as_f64(t) for t in (q, k, v, dout))
        B, H, N, d = qd.shape
        outs = [np.zeros_like(qd) for _ in range(3)]
        assert lib.oracle_attn_bwd(*(oracle._ptr(t) for t in (qd, kd, vd, dd, *outs)), B, H, N, d,
                                   float(scale), int(causal), 1) == 0
        return outs

    def dq_rows(q, k, v, dout, scale, causal, rows):
        qd, kd, vd, dd = (oracle._as_f64(t) for t in (q, k, v, dout))
        B, H, N, d = qd.shape
        r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        out = np.zeros((r.size, d))
        assert lib.oracle_attn_bwd_dq_rows(*(oracle._ptr(t) for t in (qd, kd, vd, dd, out)), B, H,
                                           N, d, float(scale), int(causal),
                                           r.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
                                           r.size, 1) == 0
        return out

    def dkv_rows(q, k, v, dout, scale, causal, rows):
        qd, kd, vd, dd = (oracle._as_f64(t) for t in (q, k, v, dout))
        B, H, N, d = qd.shape
        r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        dk, dv = np.zeros((r.size, d)), np.zeros((r.size, d))
        assert lib.oracle_attn_bwd_dkv_rows(*(oracle._ptr(t) for t in (qd, kd, vd, dd, dk, dv)),
                                            B, H, N, d, float(scale), int(causal),
                                            r.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
                                            r.size, 1) == 0
        return dk, dv
    failed = 0
    with np.errstate(all="ignore"):
        for run in (lambda: pins.pin_bwd_autograd(attn_bwd),
                    lambda: pins.pin_bwd_finite_difference(attn_bwd, oracle.attn_fwd),
                    lambda: pins.pin_bwd_invariants(attn_bwd, dq_rows, dkv_rows)):
            try:
                run()
            except AssertionError:
                failed += 1
    assert failed, "planted mistake %s passed every pin" % name


def test_rowops_oracle_meets_pins():
    pins.pin_softmax_rows(oracle.softmax_rows)
    pins.pin_row_sum(oracle.row_sum)


ROWOPS_MUTANTS = {
    "softmax_no_max_shift": ("yi[j] = exp(xi[j] - m);", "yi[j] = exp(xi[j] - m) * exp(m - 1.0);"),
    "softmax_not_normalised": ("yi[j] /= z;", "yi[j] /= 1.0;"),
    "softmax_exp_sign": ("yi[j] = exp(xi[j] - m);", "yi[j] = exp(m - xi[j]);"),
    "row_sum_drops_last": ("for (int64_t j = 0; j < N; ++j)\n            acc += xi[j];",
                           "for (int64_t j = 0; j + 1 < N; ++j)\n            acc += xi[j];"),
}


@pytest.mark.parametrize("name", sorted(ROWOPS_MUTANTS))
def test_rowops_planted_mistake_is_caught(name, mutant_dir):
    here = os.path.dirname(oracle.__file__)
    src = open(os.path.join(here, "rowops_oracle.c")).read()
    old, new = ROWOPS_MUTANTS[name]
    assert src.count(old) >= 1, "mutation anchor vanished: %r" % old
    c_path = os.path.join(mutant_dir, name + ".c")
    so_path = os.path.join(mutant_dir, name + ".so")
    with open(c_path, "w") as f:
        f.write(src.replace(old, new))
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-o", so_path,
                    os.path.join(here, "attn_oracle.c"), c_path, "-lm"], check=True)
    lib = oracle._open(so_path)

    def softmax_rows(x):
        xd = oracle._as_f64(x)
        y = np.zeros_like(xd)
        assert lib.oracle_softmax_rows(oracle._ptr(xd), oracle._ptr(y), *xd.shape) == 0
        return y

    def row_sum(x):
        xd = oracle._as_f64(x)
        out = np.zeros(xd.shape[0])
        assert lib.oracle_row_sum(oracle._ptr(xd), oracle._ptr(out), *xd.shape) == 0
        return out
    failed = 0
    with np.errstate(all="ignore"):
        for pin, fn in ((pins.pin_softmax_rows, softmax_rows), (pins.pin_row_sum, row_sum)):
            try:
                pin(fn)
            except AssertionError:
                failed += 1
    assert failed, "planted mistake %s passed every pin" % name


def test_oracle_rejects_bad_arguments():
    q = torch.zeros(1, 1, 4, 2, dtype=torch.float64)
    with pytest.raises(RuntimeError):
        oracle.attn_fwd(q, q, q, 1.0, False, rows=[4])  # row id out of range
    with pytest.raises(RuntimeError):
        oracle.attn_fwd(q, q, q, 1.0, False, rows=[-1])
    with pytest.raises(ValueError):
        oracle.attn_fwd(q, q[:, :, :3], q, 1.0, False)


def test_oracle_empty_inputs():
    q = torch.zeros(1, 1, 0, 8, dtype=torch.float64)
    o, lse = oracle.attn_fwd(q, q, q, 1.0, True)
    assert o.shape == (0, 8) and lse.shape == (0,)
    q = torch.zeros(0, 3, 5, 8, dtype=torch.float64)
    o, lse = oracle.attn_fwd(q, q, q, 1.0, False)
    assert o.shape == (0, 8)


def test_oracle_threads_do_not_change_results():
    g = torch.Generator().manual_seed(5)
    q, k, v = (torch.randn(2, 2, 70, 8, generator=g, dtype=torch.float64) for _ in range(3))
    o1, l1 = oracle.attn_fwd(q, k, v, 0.3, True, threads=1)
    o7, l7 = oracle.attn_fwd(q, k, v, 0.3, True, threads=7)
    assert np.array_equal(o1, o7) and np.array_equal(l1, l7)

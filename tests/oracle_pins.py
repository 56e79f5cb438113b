"""Pins for the fp64 oracle: checks against what the method and the mathematics
fix, independent of the oracle's own code.

Each ``pin_*`` takes an oracle callable with the signature of
``oracle.attn_fwd`` and raises AssertionError when the oracle is wrong.  The
tests run them on the real oracle (all must pass) and on deliberately broken
copies of it (each copy must fail at least one), which shows that a plausible
slip -- a dropped scale, a wrong sign, an off-by-one mask, a wrong log base, a
missing normalisation, a mis-indexed operand -- cannot pass unnoticed.

Sources of the facts pinned here:
  * the definition itself: "OpenAI Triton: from introduction to model
    practice", section 3 (standard attention in the decoder layer) and section
    5 (Figure 5 / Source 2: output plus lse = m + log l);
  * the online recurrence (running max m_i, running sum l_i, rescaled
    accumulator): "Triton hand-written kernels: vector add -> tiled GEMM ->
    FlashAttention core", section 4;
  * the causal mask keeps keys j <= i: the same page's note that a real
    implementation needs the causal mask, and the decoder layer's masked_fill.
"""
from __future__ import annotations

import math

import numpy as np
import torch

TOL = 1e-12


def _rand(shape, seed, scale=1.0):
    g = torch.Generator("cpu").manual_seed(seed)
    return (torch.randn(shape, generator=g, dtype=torch.float64) * scale)


def _bf16_exact(shape, seed, scale=1.0):
    """Random values that are exactly representable in bf16, as float64."""
    return _rand(shape, seed, scale).to(torch.bfloat16).to(torch.float64)


def _close(a, b, tol=TOL, what=""):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    assert a.shape == b.shape, (what, a.shape, b.shape)
    assert np.all(np.isfinite(a)), "%s: non-finite values" % what
    err = np.max(np.abs(a - b) / np.maximum(1.0, np.abs(b))) if a.size else 0.0
    assert err <= tol, "%s: max relative error %.3e > %.1e" % (what, err, tol)


# --------------------------------------------------------------------------- P1
def _direct_row(qi, K, V, scale, n_keys):
    """Softmax straight from its definition in Python floats, with exactly
    rounded sums and without the max shift: p_j = e^{s_j} / sum_k e^{s_k}."""
    s = [scale * math.fsum(qi[c] * K[j][c] for c in range(len(qi))) for j in range(n_keys)]
    e = [math.exp(x) for x in s]
    z = math.fsum(e)
    o = [math.fsum(e[j] * V[j][c] for j in range(n_keys)) / z for c in range(len(V[0]))]
    return o, math.log(z)


def pin_brute_force(oracle):
    """P1: tiny cases against a direct evaluation and against torch.softmax."""
    for (B, H, N, d, causal, seed) in [(1, 1, 1, 1, False, 1), (1, 2, 5, 3, False, 2),
                                       (2, 1, 8, 4, True, 3), (1, 1, 7, 2, True, 4),
                                       (2, 2, 6, 4, False, 5)]:
        q = _bf16_exact((B, H, N, d), seed)
        k = _bf16_exact((B, H, N, d), seed + 100)
        v = _bf16_exact((B, H, N, d), seed + 200)
        scale = 0.7
        o, lse = oracle(q, k, v, scale, causal)
        o = o.reshape(B, H, N, d)
        lse = lse.reshape(B, H, N)
        # (a) direct definition, row by row
        for b in range(B):
            for h in range(H):
                Q, K, V = q[b, h].tolist(), k[b, h].tolist(), v[b, h].tolist()
                for i in range(N):
                    n_keys = i + 1 if causal else N
                    ro, rl = _direct_row(Q[i], K, V, scale, n_keys)
                    _close(o[b, h, i], ro, 1e-13, "P1 direct O")
                    _close(lse[b, h, i], rl, 1e-13, "P1 direct lse")
        # (b) a library softmax of the masked score matrix
        s = torch.einsum("bhic,bhjc->bhij", q, k) * scale
        if causal:
            mask = torch.ones(N, N, dtype=torch.bool).tril()
            s = s.masked_fill(~mask, float("-inf"))
        ref_o = torch.softmax(s, dim=-1) @ v
        ref_lse = torch.logsumexp(s, dim=-1)
        _close(o, ref_o.numpy(), 1e-13, "P1 torch O")
        _close(lse, ref_lse.numpy(), 1e-13, "P1 torch lse")


# --------------------------------------------------------------------------- P2
def online_reference(q, k, v, scale, causal, tile):
    """The method's own recurrence, tile by tile over the keys, in fp64:
    m_new = max(m, rowmax S); alpha = exp(m - m_new); l = alpha*l + rowsum P;
    acc = alpha*acc + P V; finally O = acc / l and lse = m + log l."""
    q = q.numpy()
    k = k.numpy()
    v = v.numpy()
    B, H, N, d = q.shape
    O = np.zeros((B, H, N, d))
    L = np.zeros((B, H, N))
    rows = np.arange(N)[:, None]
    for b in range(B):
        for h in range(H):
            m = np.full(N, -np.inf)
            l = np.zeros(N)
            acc = np.zeros((N, d))
            for j0 in range(0, N, tile):
                cols = np.arange(j0, min(j0 + tile, N))[None, :]
                S = scale * (q[b, h] @ k[b, h, j0:j0 + tile].T)
                if causal:
                    S = np.where(cols <= rows, S, -np.inf)
                m_new = np.maximum(m, S.max(axis=1))
                live = np.isfinite(m_new)
                alpha = np.where(live, np.exp(np.where(live, m - m_new, 0.0)), 1.0)
                P = np.where(np.isfinite(S), np.exp(S - np.where(live, m_new, 0.0)[:, None]), 0.0)
                l = alpha * l + P.sum(axis=1)
                acc = alpha[:, None] * acc + P @ v[b, h, j0:j0 + tile]
                m = m_new
            O[b, h] = acc / l[:, None]
            L[b, h] = m + np.log(l)
    return O, L


def pin_online_equals_two_pass(oracle):
    """P2: the tiled online softmax reaches the full-softmax result."""
    for causal in (False, True):
        B, H, N, d = 1, 2, 150, 8
        q = _bf16_exact((B, H, N, d), 11, 2.0)
        k = _bf16_exact((B, H, N, d), 12, 2.0)
        v = _bf16_exact((B, H, N, d), 13)
        o, lse = oracle(q, k, v, 0.35, causal)
        for tile in (1, 3, 7, 128):
            ro, rl = online_reference(q, k, v, 0.35, causal, tile)
            _close(o, ro.reshape(-1, d), 1e-12, "P2 O tile=%d" % tile)
            _close(lse, rl.reshape(-1), 1e-12, "P2 lse tile=%d" % tile)


# --------------------------------------------------------------------------- P3
def pin_rows_sum_to_one(oracle):
    """P3: every softmax row sums to 1; masked probabilities are exactly 0."""
    for causal in (False, True):
        B, H, N, d = 1, 1, 33, 16
        q = _bf16_exact((B, H, N, d), 21, 3.0)
        k = _bf16_exact((B, H, N, d), 22, 3.0)
        v = _bf16_exact((B, H, N, d), 23)
        o, lse, p = oracle(q, k, v, 0.25, causal, with_probs=True)
        _close(p.sum(axis=1), np.ones(N), 1e-12, "P3 row sums")
        assert np.all(p >= 0.0)
        if causal:
            upper = np.triu(np.ones((N, N), dtype=bool), k=1)
            assert np.all(p[upper] == 0.0), "P3: masked keys carry weight"
        # O is the probability-weighted sum of V rows
        _close(o, p @ v[0, 0].numpy(), 1e-12, "P3 O = P V")


# --------------------------------------------------------------------------- P4
def pin_shift_invariance(oracle):
    """P4: adding one vector u to every key row shifts row i's scores by
    c_i = scale * q_i . u; O is unchanged and lse moves by exactly c_i."""
    for causal in (False, True):
        B, H, N, d = 2, 1, 40, 8
        q = _bf16_exact((B, H, N, d), 31)
        k = _bf16_exact((B, H, N, d), 32)
        v = _bf16_exact((B, H, N, d), 33)
        u = torch.tensor([0.5, -1.25, 2.0, 0.125, -0.75, 1.5, 0.0, -2.5], dtype=torch.float64)
        scale = 0.5
        o, lse = oracle(q, k, v, scale, causal)
        o2, lse2 = oracle(q, k + u, v, scale, causal)
        c = (scale * (q @ u)).reshape(-1).numpy()
        _close(o2, o, 1e-12, "P4 O")
        _close(lse2, lse + c, 1e-12, "P4 lse")


# --------------------------------------------------------------------------- P5
def pin_identical_values(oracle):
    """P5: if all value rows equal w, every output row equals w."""
    for causal in (False, True):
        B, H, N, d = 1, 3, 50, 6
        q = _bf16_exact((B, H, N, d), 41, 3.0)
        k = _bf16_exact((B, H, N, d), 42, 3.0)
        w = _bf16_exact((B, H, 1, d), 43)
        v = w.expand(B, H, N, d).contiguous()
        o, _ = oracle(q, k, v, 0.4, causal)
        _close(o, w.expand(B, H, N, d).reshape(-1, d).numpy(), 1e-13, "P5")


# --------------------------------------------------------------------------- P6
def pin_zero_queries(oracle):
    """P6: Q = 0 gives uniform weights: O_i = mean of the visible V rows and
    lse_i = ln(number of visible keys)."""
    B, H, N, d = 1, 2, 37, 5
    q = torch.zeros((B, H, N, d), dtype=torch.float64)
    k = _bf16_exact((B, H, N, d), 51)
    v = _bf16_exact((B, H, N, d), 52)
    o, lse = oracle(q, k, v, 0.3, False)
    _close(o.reshape(B, H, N, d), v.mean(dim=2, keepdim=True).expand(B, H, N, d).numpy(),
           1e-13, "P6 O")
    _close(lse, np.full(B * H * N, math.log(N)), 1e-13, "P6 lse")
    o, lse = oracle(q, k, v, 0.3, True)
    counts = torch.arange(1, N + 1, dtype=torch.float64)[None, None, :, None]
    _close(o.reshape(B, H, N, d), (v.cumsum(dim=2) / counts).numpy(), 1e-13, "P6 causal O")
    _close(lse.reshape(B, H, N), np.log(np.arange(1, N + 1))[None, None, :].repeat(H, 1),
           1e-13, "P6 causal lse")


# --------------------------------------------------------------------------- P7/P8
def pin_single_key_rows(oracle):
    """P7: under the causal mask row 0 sees only key 0, so o_0 = v_0 and
    lse_0 = scale * q_0 . k_0.  P8: with N = 1 the same holds without a mask."""
    B, H, N, d = 2, 2, 9, 4
    q = _bf16_exact((B, H, N, d), 61)
    k = _bf16_exact((B, H, N, d), 62)
    v = _bf16_exact((B, H, N, d), 63)
    o, lse = oracle(q, k, v, 0.5, True)
    o = o.reshape(B, H, N, d)
    lse = lse.reshape(B, H, N)
    assert np.array_equal(o[:, :, 0], v[:, :, 0].numpy()), "P7 o_0 != v_0"
    _close(lse[:, :, 0], (0.5 * (q[:, :, 0] * k[:, :, 0]).sum(-1)).numpy(), 1e-15, "P7 lse_0")
    for causal in (False, True):
        q1, k1, v1 = q[:, :, :1].contiguous(), k[:, :, :1].contiguous(), v[:, :, :1].contiguous()
        o1, l1 = oracle(q1, k1, v1, 0.5, causal)
        assert np.array_equal(o1, v1.reshape(-1, d).numpy()), "P8 O != v_0"
        _close(l1, (0.5 * (q1 * k1).sum(-1)).reshape(-1).numpy(), 1e-15, "P8 lse")


# --------------------------------------------------------------------------- P9
def pin_permutations(oracle):
    """P9 (no mask): permuting key/value rows jointly leaves O unchanged;
    permuting query rows permutes the output rows the same way."""
    B, H, N, d = 1, 1, 31, 6
    q = _bf16_exact((B, H, N, d), 71, 2.0)
    k = _bf16_exact((B, H, N, d), 72, 2.0)
    v = _bf16_exact((B, H, N, d), 73)
    o, lse = oracle(q, k, v, 0.45, False)
    perm = torch.randperm(N, generator=torch.Generator().manual_seed(7))
    o2, lse2 = oracle(q, k[:, :, perm], v[:, :, perm], 0.45, False)
    _close(o2, o, 1e-12, "P9 kv permutation O")
    _close(lse2, lse, 1e-12, "P9 kv permutation lse")
    o3, lse3 = oracle(q[:, :, perm], k, v, 0.45, False)
    _close(o3, o[perm.numpy()], 1e-13, "P9 q permutation O")
    _close(lse3, lse[perm.numpy()], 1e-13, "P9 q permutation lse")


def pin_row_selection(oracle):
    """Selected rows (the sampled mode) equal the same rows of the full run."""
    for causal in (False, True):
        B, H, N, d = 2, 3, 20, 4
        q = _bf16_exact((B, H, N, d), 81)
        k = _bf16_exact((B, H, N, d), 82)
        v = _bf16_exact((B, H, N, d), 83)
        o, lse = oracle(q, k, v, 0.5, causal)
        rows = np.array([0, 5, 19, 20, 37, 59, 119], dtype=np.int64)
        os_, ls_ = oracle(q, k, v, 0.5, causal, rows=rows)
        assert np.array_equal(os_, o[rows]) and np.array_equal(ls_, lse[rows]), "row selection"


ALL_PINS = [pin_brute_force, pin_online_equals_two_pass, pin_rows_sum_to_one,
            pin_shift_invariance, pin_identical_values, pin_zero_queries,
            pin_single_key_rows, pin_permutations, pin_row_selection]


# --------------------------------------------------------------------------- row ops
def pin_softmax_rows(softmax_rows):
    """Row softmax: matches torch.softmax in fp64, rows sum to 1, invariant to a
    per-row shift, uniform for a constant row, one-hot in the large-gap limit."""
    g = torch.Generator().manual_seed(101)
    x = torch.randn(7, 33, generator=g, dtype=torch.float64) * 4
    y = softmax_rows(x)
    _close(y, torch.softmax(x, dim=1).numpy(), 1e-14, "softmax vs torch")
    _close(y.sum(axis=1), np.ones(7), 1e-14, "softmax row sums")
    shift = torch.tensor([[-3.5], [0.25], [100.0], [-1e3], [7.0], [0.0], [12.5]], dtype=torch.float64)
    _close(softmax_rows(x + shift), y, 1e-13, "softmax shift invariance")
    _close(softmax_rows(torch.full((2, 9), 3.0, dtype=torch.float64)), np.full((2, 9), 1 / 9), 1e-15,
           "softmax of a constant row")
    z = torch.zeros(1, 5, dtype=torch.float64)
    z[0, 2] = 800.0
    assert np.array_equal(softmax_rows(z), np.array([[0.0, 0.0, 1.0, 0.0, 0.0]])), "one-hot limit"
    # direct definition without the max shift, exactly rounded sums
    for row in x.tolist()[:3]:
        e = [math.exp(a) for a in row]
        zsum = math.fsum(e)
        ref = [a / zsum for a in e]
        _close(softmax_rows(torch.tensor([row], dtype=torch.float64))[0], ref, 1e-14, "softmax direct")


def pin_row_sum(row_sum):
    """Row sum: equals math.fsum of each row (exactly rounded), and is linear."""
    g = torch.Generator().manual_seed(102)
    x = torch.randn(6, 1000, generator=g, dtype=torch.float64)
    s = row_sum(x)
    ref = [math.fsum(r) for r in x.tolist()]
    _close(s, ref, 1e-12, "row sum vs fsum")
    _close(row_sum(2.0 * x + 1.0), 2.0 * np.asarray(ref) + 1000.0, 1e-12, "row sum linearity")
    assert row_sum(torch.zeros(3, 0, dtype=torch.float64)).tolist() == [0.0, 0.0, 0.0]


# --------------------------------------------------------------------------- backward
def _torch_attn(q, k, v, scale, causal):
    s = torch.einsum("bhic,bhjc->bhij", q, k) * scale
    if causal:
        N = q.shape[2]
        s = s.masked_fill(~torch.ones(N, N, dtype=torch.bool).tril(), float("-inf"))
    return torch.softmax(s, dim=-1) @ v


def pin_bwd_autograd(attn_bwd):
    """Gradients equal torch.autograd of the standard attention in fp64."""
    for (B, H, N, d, causal, seed) in [(1, 1, 1, 2, False, 1), (1, 2, 6, 3, False, 2),
                                       (2, 1, 9, 4, True, 3), (1, 1, 17, 8, True, 4)]:
        q = _bf16_exact((B, H, N, d), seed, 2.0).requires_grad_()
        k = _bf16_exact((B, H, N, d), seed + 10, 2.0).requires_grad_()
        v = _bf16_exact((B, H, N, d), seed + 20).requires_grad_()
        g = _bf16_exact((B, H, N, d), seed + 30)
        _torch_attn(q, k, v, 0.6, causal).backward(g)
        dq, dk, dv = attn_bwd(q.detach(), k.detach(), v.detach(), g, 0.6, causal)
        _close(dq, q.grad.numpy(), 1e-12, "bwd dq vs autograd")
        _close(dk, k.grad.numpy(), 1e-12, "bwd dk vs autograd")
        _close(dv, v.grad.numpy(), 1e-12, "bwd dv vs autograd")


def pin_bwd_finite_difference(attn_bwd, attn_fwd):
    """Central differences of L = sum(O * g) through the forward oracle."""
    B, H, N, d = 1, 1, 5, 3
    q = _bf16_exact((B, H, N, d), 41)
    k = _bf16_exact((B, H, N, d), 42)
    v = _bf16_exact((B, H, N, d), 43)
    g = _bf16_exact((B, H, N, d), 44)
    for causal in (False, True):
        grads = dict(zip("qkv", attn_bwd(q, k, v, g, 0.8, causal)))
        for name, t in (("q", q), ("k", k), ("v", v)):
            for idx in [(0, 0, 0, 0), (0, 0, 2, 1), (0, 0, 4, 2)]:
                eps = 1e-5
                tp, tm = t.clone(), t.clone()
                tp[idx] += eps
                tm[idx] -= eps
                args_p = {"q": q, "k": k, "v": v, name: tp}
                args_m = {"q": q, "k": k, "v": v, name: tm}
                lp = (attn_fwd(args_p["q"], args_p["k"], args_p["v"], 0.8, causal)[0] *
                      g.reshape(-1, d).numpy()).sum()
                lm = (attn_fwd(args_m["q"], args_m["k"], args_m["v"], 0.8, causal)[0] *
                      g.reshape(-1, d).numpy()).sum()
                fd = (lp - lm) / (2 * eps)
                assert abs(fd - grads[name][idx]) <= 1e-7 * max(1.0, abs(fd)), (name, idx, fd,
                                                                                 grads[name][idx])


def pin_bwd_invariants(attn_bwd, attn_bwd_dq_rows, attn_bwd_dkv_rows=None):
    """Each row of dS sums to zero, so the key gradients sum to zero over the
    keys; the value gradients sum to the sum of dO over the rows (rows of P
    sum to one); and the dq rows and dk/dv rows modes equal the full rows."""
    for causal in (False, True):
        B, H, N, d = 2, 2, 23, 4
        q = _bf16_exact((B, H, N, d), 51, 2.0)
        k = _bf16_exact((B, H, N, d), 52, 2.0)
        v = _bf16_exact((B, H, N, d), 53)
        g = _bf16_exact((B, H, N, d), 54)
        dq, dk, dv = attn_bwd(q, k, v, g, 0.4, causal)
        assert np.max(np.abs(dk.sum(axis=2))) <= 1e-12, "sum_j dK_j != 0"
        _close(dv.sum(axis=2), g.sum(dim=2).numpy(), 1e-12, "sum_j dV_j")
        rows = np.array([0, 7, 22, 23, 50, 91], dtype=np.int64)
        _close(attn_bwd_dq_rows(q, k, v, g, 0.4, causal, rows), dq.reshape(-1, d)[rows], 1e-13,
               "dq rows mode")
        if attn_bwd_dkv_rows is not None:
            # Keys of several heads, out of order and repeated.
            keys = np.array([91, 0, 22, 45, 23, 7, 68, 91, 46], dtype=np.int64)
            dk_r, dv_r = attn_bwd_dkv_rows(q, k, v, g, 0.4, causal, keys)
            _close(dk_r, dk.reshape(-1, d)[keys], 1e-13, "dk rows mode")
            _close(dv_r, dv.reshape(-1, d)[keys], 1e-13, "dv rows mode")


# --------------------------------------------------------------------------- Nq != Nk
def pin_fwd_kv(attn_fwd_kv, attn_fwd):
    """Queries against a longer key sequence: brute force against torch.softmax
    with the bottom-right causal mask; the square case equals the main oracle;
    a single query (decode) sees every key with or without the mask; a query
    block at the end of the sequence equals those rows of the square problem."""
    for (B, H, Nq, Nk, d, causal, seed) in [(1, 2, 3, 7, 4, True, 1), (2, 1, 5, 5, 3, True, 2),
                                            (1, 1, 4, 9, 2, False, 3), (1, 1, 1, 6, 4, True, 4)]:
        q = _bf16_exact((B, H, Nq, d), seed, 2.0)
        k = _bf16_exact((B, H, Nk, d), seed + 50, 2.0)
        v = _bf16_exact((B, H, Nk, d), seed + 60)
        o, lse = attn_fwd_kv(q, k, v, 0.5, causal)
        s = torch.einsum("bhic,bhjc->bhij", q, k) * 0.5
        if causal:
            i = torch.arange(Nq)[:, None]
            j = torch.arange(Nk)[None, :]
            s = s.masked_fill(j > i + (Nk - Nq), float("-inf"))
        _close(o, (torch.softmax(s, -1) @ v).reshape(-1, d).numpy(), 1e-13, "kv vs torch")
        _close(lse, torch.logsumexp(s, -1).reshape(-1).numpy(), 1e-13, "kv lse vs torch")
    q = _bf16_exact((2, 2, 11, 4), 7)
    k = _bf16_exact((2, 2, 11, 4), 8)
    v = _bf16_exact((2, 2, 11, 4), 9)
    for causal in (False, True):
        a = attn_fwd_kv(q, k, v, 0.3, causal)
        b = attn_fwd(q, k, v, 0.3, causal)
        assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1]), "square case"
        tail = attn_fwd_kv(q[:, :, 8:].contiguous(), k, v, 0.3, causal)
        rows = np.array([h * 11 + i for h in range(4) for i in range(8, 11)])
        _close(tail[0], b[0][rows], 1e-14, "query block at the end")
    one_q = q[:, :, -1:].contiguous()
    assert np.array_equal(attn_fwd_kv(one_q, k, v, 0.3, True)[0],
                          attn_fwd_kv(one_q, k, v, 0.3, False)[0]), "decode row sees all keys"

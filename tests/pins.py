"""Checks that pin the FP64 oracle to facts fixed outside it.

Each ``pin_*`` function takes an ``oracle.Oracle`` and raises AssertionError
if the oracle disagrees with a closed form, a brute-force evaluation, an
identity the pages state, or an independent library evaluation.  The test
suite runs every pin on the real oracle (all must pass) and on deliberately
broken builds of the oracle (each must be caught by at least one pin).
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "closed_form_fwd.json")

_EXPR_NAMES = {"log": math.log, "exp": math.exp, "sqrt": math.sqrt}


def _expr(x) -> float:
    """Evaluate a fixture entry: a number, or an expression in log/exp/sqrt."""
    if isinstance(x, (int, float)):
        return float(x)
    return float(eval(str(x), {"__builtins__": {}}, dict(_EXPR_NAMES)))


def _arr(rows):
    return np.array([[_expr(x) for x in r] for r in rows], dtype=np.float64)


def _close(a, b, tol, what):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    assert a.shape == b.shape, f"{what}: shape {a.shape} vs {b.shape}"
    assert np.all(np.isfinite(a)), f"{what}: non-finite values"
    err = np.max(np.abs(a - b) / np.maximum(1.0, np.abs(b))) if a.size else 0.0
    assert err <= tol, f"{what}: error {err:.3e} > {tol:.1e}"


# ---------------------------------------------------------------------------
# forward pins


def pin_golden_closed_forms(orc):
    """Hand-derived cases (tests/golden/closed_form_fwd.json)."""
    cases = json.load(open(GOLDEN))["cases"]
    for c in cases:
        q, k, v = _arr(c["q"]), _arr(c["k"]), _arr(c["v"])
        o, lse = orc.attn_fwd(q, k, v, c["causal"], c["scale"])
        _close(o, _arr(c["o"]), 1e-12, c["name"] + " O")
        _close(lse, np.array([_expr(x) for x in c["lse"]]), 1e-12, c["name"] + " LSE")


def brute_force_fwd(q, k, v, causal, scale):
    """exp(S)/sum exp(S) with Python floats, no max subtraction (small scores only).
    Causal with Nk >= N keys: query i sees keys j <= i + Nk - N."""
    N, d = len(q), len(q[0])
    o, lse = [], []
    for i in range(N):
        keys = range(i + len(k) - N + 1) if causal else range(len(k))
        w = {}
        for j in keys:
            w[j] = math.exp(scale * math.fsum(q[i][t] * k[j][t] for t in range(d)))
        z = math.fsum(w.values())
        o.append([math.fsum(w[j] * v[j][t] for j in keys) / z for t in range(len(v[0]))])
        lse.append(math.log(z))
    return np.array(o), np.array(lse)


def pin_brute_force(orc):
    """Direct softmax on tiny inputs in pure-Python float64."""
    rng = np.random.default_rng(11)
    for (N, Nk, d, causal) in [(4, 4, 4, False), (4, 4, 4, True), (5, 3, 2, False),
                               (6, 6, 3, True), (1, 1, 5, True), (3, 7, 1, False),
                               (3, 7, 2, True), (1, 5, 3, True)]:
        q = rng.uniform(-1.5, 1.5, (N, d))
        k = rng.uniform(-1.5, 1.5, (Nk, d))
        v = rng.uniform(-2, 2, (Nk, d))
        scale = 1.0 / math.sqrt(d)
        o_ref, lse_ref = brute_force_fwd(q.tolist(), k.tolist(), v.tolist(), causal, scale)
        o, lse = orc.attn_fwd(q, k, v, causal, scale)
        _close(o, o_ref, 1e-12, f"brute force O {N}x{Nk}x{d} causal={causal}")
        _close(lse, lse_ref, 1e-12, f"brute force LSE {N}x{Nk}x{d} causal={causal}")


def pin_rows_sum_to_one(orc):
    """With V = I the output is P itself: rows sum to 1, entries >= 0, masked ones exactly 0."""
    rng = np.random.default_rng(12)
    for causal in (False, True):
        N = d = 9
        q = rng.normal(size=(N, d)) * 3
        k = rng.normal(size=(N, d)) * 3
        P, _ = orc.attn_fwd(q, k, np.eye(N), causal, 0.7)
        _close(P.sum(axis=1), np.ones(N), 1e-12, "row sums of P")
        assert np.all(P >= 0.0), "P has negative entries"
        if causal:
            assert np.all(np.triu(P, 1) == 0.0), "causal P has weight above the diagonal"


def pin_equal_scores(orc):
    """Q = 0: every score is 0, so O_i is the mean of the visible V rows and LSE_i = ln(#visible)."""
    rng = np.random.default_rng(13)
    N, d = 23, 6
    k = rng.normal(size=(N, d))
    v = rng.normal(size=(N, d))
    o, lse = orc.attn_fwd(np.zeros((N, d)), k, v, False, 0.3)
    _close(o, np.broadcast_to(v.mean(axis=0), (N, d)), 1e-12, "Q=0 non-causal O")
    _close(lse, np.full(N, math.log(N)), 1e-12, "Q=0 non-causal LSE")
    o, lse = orc.attn_fwd(np.zeros((N, d)), k, v, True, 0.3)
    mean_prefix = np.cumsum(v, axis=0) / np.arange(1, N + 1)[:, None]
    _close(o, mean_prefix, 1e-12, "Q=0 causal O")
    _close(lse, np.log(np.arange(1, N + 1)), 1e-12, "Q=0 causal LSE")


def merge_states(a, b):
    """Two-block merge of (m, l, O) with O normalised, as the huaweicloud page's section two
    states it: m = max(mA, mB); l = e^(mA-m) lA + e^(mB-m) lB;
    O = (lA e^(mA-m) OA + lB e^(mB-m) OB) / l."""
    (ma, la, oa), (mb, lb, ob) = a, b
    m = np.maximum(ma, mb)
    ea = np.where(np.isneginf(ma), 0.0, np.exp(ma - m))
    eb = np.where(np.isneginf(mb), 0.0, np.exp(mb - m))
    l = ea * la + eb * lb
    o = ((la * ea)[:, None] * oa + (lb * eb)[:, None] * ob) / l[:, None]
    return m, l, o


def pin_merge_rule(orc):
    """Oracle on key blocks, merged by the page's rule, equals the oracle on all keys
    (two blocks, and k blocks merged one after another as in the induction argument)."""
    rng = np.random.default_rng(14)
    N, Nk, d = 17, 41, 8
    q = rng.normal(size=(N, d)) * 2
    k = rng.normal(size=(Nk, d)) * 2
    v = rng.normal(size=(Nk, d))
    scale = 1 / math.sqrt(d)
    o_full, lse_full = orc.attn_fwd(q, k, v, False, scale)

    def state(lo, hi):
        o, lse = orc.attn_fwd(q, k[lo:hi], v[lo:hi], False, scale)
        return lse, np.ones(N), o          # (m, l) = (LSE, 1) represents the same block

    for cut in (1, 16, 40):
        m, l, o = merge_states(state(0, cut), state(cut, Nk))
        _close(o, o_full, 1e-12, f"two-block merge O (cut {cut})")
        _close(m + np.log(l), lse_full, 1e-12, f"two-block merge LSE (cut {cut})")
    # k blocks, starting from the initial state O = 0, l = 0, m = -inf
    st = (np.full(N, -np.inf), np.zeros(N), np.zeros((N, d)))
    for lo in range(0, Nk, 7):
        st = merge_states(st, state(lo, min(lo + 7, Nk)))
    _close(st[2], o_full, 1e-12, "k-block merge O")
    _close(st[0] + np.log(st[1]), lse_full, 1e-12, "k-block merge LSE")


def online_simulator(q, k, v, causal, scale, br, bc, deferred):
    """FP64 restatement of the tiled forward that the huaweicloud page's section three
    simulates: K/V blocks outer, Q blocks inner, running (m, l, O) per row with the
    rescale factor exp(m_prev - m_new).  deferred=False keeps O normalised after every
    block (the page's simulator); deferred=True keeps it unnormalised and divides by l
    once at the end (the second-generation ordering)."""
    N, d = q.shape
    Nk = k.shape[0]
    O = np.zeros((N, d))
    l = np.zeros(N)
    m = np.full(N, -np.inf)
    for j in range(0, Nk, bc):
        for i in range(0, N, br):
            s = scale * q[i:i + br] @ k[j:j + bc].T
            if causal:
                rows = np.arange(i, min(i + br, N))[:, None]
                cols = np.arange(j, min(j + bc, Nk))[None, :]
                s = np.where(cols > rows, -np.inf, s)
            m_prev, l_prev = m[i:i + br], l[i:i + br]
            m_new = np.maximum(m_prev, s.max(axis=1))
            p = np.exp(s - m_new[:, None])
            alpha = np.where(np.isneginf(m_prev), 0.0, np.exp(m_prev - m_new))
            l_new = alpha * l_prev + p.sum(axis=1)
            if deferred:
                O[i:i + br] = alpha[:, None] * O[i:i + br] + p @ v[j:j + bc]
            else:
                O[i:i + br] = ((alpha * l_prev)[:, None] * O[i:i + br] + p @ v[j:j + bc]) / l_new[:, None]
            m[i:i + br], l[i:i + br] = m_new, l_new
    if deferred:
        O = O / l[:, None]
    return O, m + np.log(l)


def pin_online_recurrence(orc):
    """The online-softmax recurrence, run block by block, reaches the oracle's exact result."""
    rng = np.random.default_rng(15)
    for (N, d, br, bc, causal) in [(37, 8, 8, 16, False), (37, 8, 16, 8, True), (64, 4, 64, 1, True)]:
        q = rng.normal(size=(N, d)) * 3
        k = rng.normal(size=(N, d)) * 3
        v = rng.normal(size=(N, d))
        o_ref, lse_ref = orc.attn_fwd(q, k, v, causal, 0.5)
        for deferred in (False, True):
            o, lse = online_simulator(q, k, v, causal, 0.5, br, bc, deferred)
            _close(o_ref, o, 1e-12, f"online recurrence O (deferred={deferred}, causal={causal})")
            _close(lse_ref, lse, 1e-12, f"online recurrence LSE (deferred={deferred}, causal={causal})")


def pin_one_hot_large_scores(orc):
    """A key boosted by ~1000 wins every row outright: O_i = V_j* and LSE_i = S_ij* exactly
    in float64 (every other term is below e^-900, which underflows to 0 next to 1)."""
    rng = np.random.default_rng(16)
    N, d = 33, 16
    q = rng.normal(size=(N, d))
    k = rng.normal(size=(N, d))
    v = rng.normal(size=(N, d))
    q[:, d - 1] = 1.0
    js = N - 1
    k[js, d - 1] = 1000.0 * math.sqrt(d)
    scale = 1 / math.sqrt(d)
    o, lse = orc.attn_fwd(q, k, v, False, scale)
    _close(o, np.broadcast_to(v[js], (N, d)), 1e-12, "one-hot O")
    s_star = np.array([scale * math.fsum(q[i] * k[js]) for i in range(N)])
    _close(lse, s_star, 1e-12, "one-hot LSE")
    # scores of several hundred both ways stay finite
    o, lse = orc.attn_fwd(q * 20, k * 20, v, False, scale)
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse)), "large scores overflowed"
    assert np.max(np.abs(lse)) > 300, "the large-score case did not reach large scores"


def pin_causal_first_row(orc):
    """Causal row 0 sees only key 0: O_0 = V_0, LSE_0 = S_00; N = 1 gives O = V."""
    rng = np.random.default_rng(17)
    N, d = 12, 5
    q, k, v = (rng.normal(size=(N, d)) for _ in range(3))
    o, lse = orc.attn_fwd(q, k, v, True, 0.9)
    _close(o[0], v[0], 1e-12, "causal O_0")
    _close(lse[0], 0.9 * math.fsum(q[0] * k[0]), 1e-12, "causal LSE_0")
    o, lse = orc.attn_fwd(q[:1], k[:1], v[:1], False, 0.9)
    _close(o, v[:1], 1e-12, "N=1 O")


def pin_permutation_symmetry(orc):
    """Non-causal attention does not depend on the order of the (key, value) pairs."""
    rng = np.random.default_rng(18)
    N, d = 19, 7
    q, k, v = (rng.normal(size=(N, d)) for _ in range(3))
    perm = rng.permutation(N)
    o1, l1 = orc.attn_fwd(q, k, v, False, 0.4)
    o2, l2 = orc.attn_fwd(q, k[perm], v[perm], False, 0.4)
    _close(o1, o2, 1e-12, "permuted K/V O")
    _close(l1, l2, 1e-12, "permuted K/V LSE")


def pin_sampled_rows(orc):
    """Asking for a subset of rows or keys returns exactly those rows of the full result."""
    rng = np.random.default_rng(19)
    BH, N, d = 2, 21, 4
    q, k, v, do = (rng.normal(size=(BH, N, d)) for _ in range(4))
    rows = [20, 0, 7, 7]
    for causal in (False, True):
        o, lse = orc.attn_fwd(q, k, v, causal, 0.5)
        os_, ls_ = orc.attn_fwd(q, k, v, causal, 0.5, rows=rows)
        assert np.array_equal(os_, o[:, rows]) and np.array_equal(ls_, lse[:, rows])
        dq, dk, dv = orc.attn_bwd(q, k, v, do, causal, 0.5)
        dqs, dks, dvs = orc.attn_bwd(q, k, v, do, causal, 0.5, qrows=rows, kcols=[3, 20])
        assert np.array_equal(dqs, dq[:, rows])
        assert np.array_equal(dks, dk[:, [3, 20]]) and np.array_equal(dvs, dv[:, [3, 20]])


# ---------------------------------------------------------------------------
# backward pins


def pin_bwd_finite_differences(orc):
    """Central differences of L = sum(dO * O), O from the oracle's forward, match the gradients."""
    rng = np.random.default_rng(20)
    for causal, N, Nk in ((False, 6, 6), (True, 6, 6), (False, 4, 7), (True, 4, 7)):
        d = 3
        q, do = (rng.normal(size=(N, d)) for _ in range(2))
        k, v = (rng.normal(size=(Nk, d)) for _ in range(2))
        scale = 0.8
        dq, dk, dv = orc.attn_bwd(q, k, v, do, causal, scale)
        h = 1e-6
        for name, x, g in (("dQ", q, dq), ("dK", k, dk), ("dV", v, dv)):
            num = np.zeros_like(x)
            for idx in np.ndindex(*x.shape):
                xp, xm = x.copy(), x.copy()
                xp[idx] += h
                xm[idx] -= h
                args_p = {"dQ": (xp, k, v), "dK": (q, xp, v), "dV": (q, k, xp)}[name]
                args_m = {"dQ": (xm, k, v), "dK": (q, xm, v), "dV": (q, k, xm)}[name]
                lp = np.sum(do * orc.attn_fwd(*args_p, causal, scale)[0])
                lm = np.sum(do * orc.attn_fwd(*args_m, causal, scale)[0])
                num[idx] = (lp - lm) / (2 * h)
            err = np.max(np.abs(num - g)) / max(1e-3, np.max(np.abs(g)))
            assert err < 1e-6, f"{name} vs finite differences (causal={causal}, {N}x{Nk}): {err:.2e}"


def pin_bwd_invariants(orc):
    """Rows of P sum to 1, so sum_j dV_j = sum_i dO_i; rows of dS sum to 0, so sum_j dK_j = 0."""
    rng = np.random.default_rng(21)
    for causal in (False, True):
        N, d = 29, 8
        q, k, v, do = (rng.normal(size=(N, d)) * 2 for _ in range(4))
        dq, dk, dv = orc.attn_bwd(q, k, v, do, causal, 0.35)
        _close(dv.sum(axis=0), do.sum(axis=0), 1e-11, f"sum dV = sum dO (causal={causal})")
        assert np.max(np.abs(dk.sum(axis=0))) < 1e-11 * max(1.0, np.abs(dk).max()), \
            f"sum dK != 0 (causal={causal})"


def pin_bwd_autograd(orc):
    """FP64 torch autograd through an explicit softmax formula (an independent library path)."""
    rng = np.random.default_rng(22)
    for causal in (False, True):
        N, d = 13, 6
        arrs = [rng.normal(size=(2, N, d)) for _ in range(4)]
        q, k, v = (torch.tensor(a, requires_grad=True) for a in arrs[:3])
        do = torch.tensor(arrs[3])
        s = 0.45 * q @ k.transpose(-1, -2)
        if causal:
            s = s.masked_fill(torch.ones(N, N, dtype=torch.bool).triu(1), float("-inf"))
        o = torch.softmax(s, dim=-1) @ v
        (o * do).sum().backward()
        dq, dk, dv = orc.attn_bwd(arrs[0], arrs[1], arrs[2], arrs[3], causal, 0.45)
        _close(dq, q.grad.numpy(), 1e-10, "dQ vs autograd")
        _close(dk, k.grad.numpy(), 1e-10, "dK vs autograd")
        _close(dv, v.grad.numpy(), 1e-10, "dV vs autograd")


# ---------------------------------------------------------------------------
# FP8 (E4M3) decoding and block dequantisation

# Codes worked out by hand from the E4M3 definition (sign, 4 exponent bits with bias 7,
# 3 mantissa bits; E = 0 subnormal 2^-6 * M/8; S.1111.111 NaN, no infinities).
E4M3_CLOSED_FORMS = [
    (0x00, 0.0),                  # +0
    (0x01, 2.0 ** -9),            # smallest subnormal: 2^-6 * 1/8
    (0x07, 7 * 2.0 ** -9),        # largest subnormal
    (0x08, 2.0 ** -6),            # smallest normal: E = 1, M = 0
    (0x38, 1.0),                  # E = 7
    (0x3C, 1.5),                  # E = 7, M = 4
    (0x40, 2.0),                  # E = 8
    (0x77, 240.0),                # E = 14, M = 7: 2^7 * 15/8
    (0x7E, 448.0),                # E = 15, M = 6: the largest finite value
    (0xB8, -1.0),
    (0xFE, -448.0),
]


def pin_e4m3_closed_forms(orc):
    """E4M3 codes against values derived by hand from the format definition."""
    for code, val in E4M3_CLOSED_FORMS:
        got = orc.e4m3_value(code)
        assert got == val, f"e4m3 code {code:#04x}: {got!r} != {val!r}"
    assert math.copysign(1.0, orc.e4m3_value(0x80)) == -1.0 and orc.e4m3_value(0x80) == 0.0, "-0"
    assert math.isnan(orc.e4m3_value(0x7F)) and math.isnan(orc.e4m3_value(0xFF)), "NaN codes"


def _torch_e4m3_table():
    return torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).double().numpy()


def pin_e4m3_all_codes_vs_torch(orc):
    """All 256 codes against PyTorch's float8_e4m3fn conversion (an independent library)."""
    ref = _torch_e4m3_table()
    got = np.array([orc.e4m3_value(c) for c in range(256)])
    assert np.array_equal(np.isnan(got), np.isnan(ref)), "NaN codes differ from float8_e4m3fn"
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok]), "decoded values differ from float8_e4m3fn"


def pin_dequant_brute_force(orc):
    """Block dequantisation against a Python loop over rows with the PyTorch decode table."""
    rng = np.random.default_rng(30)
    table = _torch_e4m3_table()
    for N, block in ((300, 128), (23, 7), (5, 128)):
        BH, d = 2, 3
        codes = rng.integers(0, 256, size=(BH, N, d)).astype(np.uint8)
        codes[np.isnan(table[codes])] = 0x38
        nblk = -(-N // block)
        scales = (2.0 ** rng.uniform(-8, 8, size=(BH, nblk))).astype(np.float32)
        got = orc.dequant_e4m3(codes, scales, block)
        for bh in range(BH):
            for n in range(N):
                for c in range(d):
                    want = table[codes[bh, n, c]] * float(scales[bh, n // block])
                    assert got[bh, n, c] == want, f"dequant [{bh},{n},{c}] (block {block})"


def pin_fp8_attention_brute_force(orc):
    """attn_fwd_fp8 on tiny inputs against brute force over the hand-dequantised values."""
    rng = np.random.default_rng(31)
    table = _torch_e4m3_table()
    N, d, block = 9, 4, 4
    nblk = -(-N // block)
    arrs, deq = [], []
    for t in range(3):
        codes = rng.integers(0, 256, size=(1, N, d)).astype(np.uint8)
        codes[np.isnan(table[codes])] = 0x30
        codes[np.abs(table[codes]) > 4] = 0x38  # keep scores small for the brute force
        sc = np.array([[0.25, 0.5, 1.0]], np.float32) * (t + 1)  # one scale per 4-row block
        arrs.append((codes, sc))
        deq.append([[table[codes[0, n, c]] * float(sc[0, n // block]) for c in range(d)] for n in range(N)])
    for causal in (False, True):
        o, lse = orc.attn_fwd_fp8(arrs[0][0], arrs[1][0], arrs[2][0], arrs[0][1], arrs[1][1], arrs[2][1],
                                  causal, 0.3, block_rows=block)
        bo, bl = brute_force_fwd(deq[0], deq[1], deq[2], causal, 0.3)
        _close(o[0], bo, 1e-12, f"fp8 O (causal={causal})")
        _close(lse[0], bl, 1e-12, f"fp8 LSE (causal={causal})")


def pin_rect_causal_is_a_suffix(orc):
    """Nq < Nk causal = the last Nq query rows of the square causal problem over all Nk
    positions: forward rows, dQ rows, and dK/dV with dO zero on the first Nk - Nq rows."""
    rng = np.random.default_rng(32)
    Nk, Nq, d = 9, 4, 3
    qf, k, v, dof = (rng.normal(size=(Nk, d)) for _ in range(4))
    dof[:Nk - Nq] = 0.0
    q, do = qf[Nk - Nq:], dof[Nk - Nq:]
    o_sq, lse_sq = orc.attn_fwd(qf, k, v, True, 0.7)
    o, lse = orc.attn_fwd(q, k, v, True, 0.7)
    _close(o, o_sq[Nk - Nq:], 1e-13, "rect causal O = suffix of square")
    _close(lse, lse_sq[Nk - Nq:], 1e-13, "rect causal LSE = suffix of square")
    dq_sq, dk_sq, dv_sq = orc.attn_bwd(qf, k, v, dof, True, 0.7)
    dq, dk, dv = orc.attn_bwd(q, k, v, do, True, 0.7)
    _close(dq, dq_sq[Nk - Nq:], 1e-12, "rect causal dQ = suffix of square")
    _close(dk, dk_sq, 1e-12, "rect causal dK = square with dO zero on the prefix")
    _close(dv, dv_sq, 1e-12, "rect causal dV = square with dO zero on the prefix")


# ---------------------------------------------------------------------------
# dropout

PHILOX_KAT = os.path.join(os.path.dirname(__file__), "golden", "philox4x32_10_kat.json")


def pin_philox_known_answers(orc):
    """Philox4x32-10 against the generator's published known-answer vectors."""
    for vec in json.load(open(PHILOX_KAT))["vectors"]:
        ctr = [int(x, 16) for x in vec["counter"]]
        key = [int(x, 16) for x in vec["key"]]
        want = [int(x, 16) for x in vec["output"]]
        got = [int(x) for x in orc.philox(ctr, key)]
        assert got == want, f"philox({vec['counter']}, {vec['key']}) = {[hex(g) for g in got]}"


def pin_dropout_mask_definition(orc):
    """The keep factor follows its definition: byte j mod 16 (little-endian over the four
    words) of Philox((j // 16, i, bh, 0), seed) compared with t, kept ones scaled by
    256 / (256 - t); t = 0 keeps everything with factor 1."""
    seed = 0x0123456789ABCDEF
    key = [seed & 0xFFFFFFFF, seed >> 32]
    rng = np.random.default_rng(37)
    cases = [(0, 0, 0), (3, 17, 40), (1, 1000, 4095), (2, 5, 15)]
    cases += [tuple(int(x) for x in (rng.integers(0, 64), rng.integers(0, 5000), rng.integers(0, 5000)))
              for _ in range(60)]
    for (bh, i, j) in cases:
        w = orc.philox([j // 16, i, bh, 0], key)
        b = j % 16
        byte = (int(w[b // 4]) >> (8 * (b % 4))) & 0xFF
        for t in (0, 1, 64, 128, 200, 255):
            want = 1.0 if t == 0 else (256.0 / (256 - t) if byte >= t else 0.0)
            assert orc.dropout_factor(bh, i, j, t, seed) == want, f"dropout factor at {(bh, i, j, t)}"


def pin_dropout_rate_and_unbiased(orc):
    """The dropped fraction is t/256 within a binomial bound, and averaging O over many
    seeds gives the plain attention (the 256 / (256 - t) scale makes dropout unbiased)."""
    t = 77
    n = 0
    dropped = 0
    for bh in range(2):
        for i in range(40):
            for j in range(64):
                n += 1
                dropped += orc.dropout_factor(bh, i, j, t, 99) == 0.0
    p = t / 256
    assert abs(dropped / n - p) < 4 * math.sqrt(p * (1 - p) / n), f"dropped fraction {dropped / n:.4f} vs {p:.4f}"
    rng = np.random.default_rng(33)
    q, k, v = (rng.normal(size=(6, 4)) for _ in range(3))
    o_ref, _ = orc.attn_fwd(q, k, v, False, 0.5)
    S = 400
    acc = np.zeros_like(o_ref)
    acc2 = np.zeros_like(o_ref)
    for seed in range(S):
        o, _ = orc.attn_fwd_dropout(q, k, v, False, 0.5, t, seed)
        acc += o
        acc2 += o * o
    mean = acc / S
    sd = np.sqrt(np.maximum(acc2 / S - mean ** 2, 1e-30) / S)
    assert np.all(np.abs(mean - o_ref) < 5 * sd + 1e-12), "dropout output is biased"


def pin_dropout_t0_is_plain(orc):
    """t = 0 keeps every probability: forward and backward equal the plain oracle's bits."""
    rng = np.random.default_rng(34)
    q, k, v, do = (rng.normal(size=(2, 9, 3)) for _ in range(4))
    for causal in (False, True):
        o, lse = orc.attn_fwd(q, k, v, causal, 0.6)
        od, lsed = orc.attn_fwd_dropout(q, k, v, causal, 0.6, 0, 5)
        assert np.array_equal(o, od) and np.array_equal(lse, lsed)
        g = orc.attn_bwd(q, k, v, do, causal, 0.6)
        gd = orc.attn_bwd_dropout(q, k, v, do, causal, 0.6, 0, 5)
        for a, b in zip(g, gd):
            assert np.array_equal(a, b)


def pin_dropout_brute_force(orc):
    """Tiny inputs: O = sum_j softmax_ij Z_ij V_j with Python floats and the keep factors;
    the logsumexp is the plain one."""
    rng = np.random.default_rng(35)
    for (N, Nk, causal) in [(5, 5, False), (5, 5, True), (3, 20, True)]:
        q = rng.uniform(-1, 1, (N, 3))
        k = rng.uniform(-1, 1, (Nk, 3))
        v = rng.uniform(-2, 2, (Nk, 3))
        t, seed = 100, 0xDEADBEEF12345
        o, lse = orc.attn_fwd_dropout(q, k, v, causal, 0.7, t, seed)
        for i in range(N):
            keys = range(i + Nk - N + 1) if causal else range(Nk)
            w = {j: math.exp(0.7 * math.fsum(q[i][x] * k[j][x] for x in range(3))) for j in keys}
            z = math.fsum(w.values())
            for c in range(3):
                ref = math.fsum(w[j] / z * orc.dropout_factor(0, i, j, t, seed) * v[j][c] for j in keys)
                assert abs(o[i][c] - ref) <= 1e-12 * max(1.0, abs(ref)), f"dropout brute force O[{i},{c}]"
            assert abs(lse[i] - math.log(z)) <= 1e-12 * max(1.0, abs(math.log(z)))


def pin_dropout_bwd_finite_differences(orc):
    """Central differences of sum(dO * O_dropout) with the mask fixed by the seed."""
    rng = np.random.default_rng(36)
    t, seed = 90, 4242
    for causal, N, Nk in ((False, 5, 5), (True, 5, 7)):
        q, do = (rng.normal(size=(N, 3)) for _ in range(2))
        k, v = (rng.normal(size=(Nk, 3)) for _ in range(2))
        dq, dk, dv = orc.attn_bwd_dropout(q, k, v, do, causal, 0.8, t, seed)
        h = 1e-6
        for name, x, g in (("dQ", q, dq), ("dK", k, dk), ("dV", v, dv)):
            num = np.zeros_like(x)
            for idx in np.ndindex(*x.shape):
                xp, xm = x.copy(), x.copy()
                xp[idx] += h
                xm[idx] -= h
                ap = {"dQ": (xp, k, v), "dK": (q, xp, v), "dV": (q, k, xp)}[name]
                am = {"dQ": (xm, k, v), "dK": (q, xm, v), "dV": (q, k, xm)}[name]
                lp = np.sum(do * orc.attn_fwd_dropout(*ap, causal, 0.8, t, seed)[0])
                lm = np.sum(do * orc.attn_fwd_dropout(*am, causal, 0.8, t, seed)[0])
                num[idx] = (lp - lm) / (2 * h)
            err = np.max(np.abs(num - g)) / max(1e-3, np.max(np.abs(g)))
            assert err < 1e-6, f"dropout {name} vs finite differences (causal={causal}): {err:.2e}"


def pin_dropout_head_offset(orc):
    """Several heads with a head offset bh0: head h of the arrays draws the mask of head
    bh0 + h.  Forward by brute force with the keep factors of those heads; backward by
    central differences of sum(dO * O) at the same offset (a packed batch's sequence b
    is computed as heads b*H .. b*H + H - 1 this way)."""
    rng = np.random.default_rng(39)
    H, N, Nk, d, t, seed, bh0, sc = 3, 4, 6, 3, 77, 0xABC0123, 5, 0.9
    q = rng.uniform(-1, 1, (H, N, d))
    k = rng.uniform(-1, 1, (H, Nk, d))
    v = rng.uniform(-2, 2, (H, Nk, d))
    o, _ = orc.attn_fwd_dropout(q, k, v, True, sc, t, seed, bh0=bh0)
    for h in range(H):
        for i in range(N):
            keys = range(i + Nk - N + 1)
            w = {j: math.exp(sc * math.fsum(q[h][i][x] * k[h][j][x] for x in range(d))) for j in keys}
            z = math.fsum(w.values())
            for c in range(d):
                ref = math.fsum(w[j] / z * orc.dropout_factor(bh0 + h, i, j, t, seed) * v[h][j][c] for j in keys)
                assert abs(o[h][i][c] - ref) <= 1e-12 * max(1.0, abs(ref)), f"head offset O[{h},{i},{c}]"
    H, N, Nk, d = 2, 3, 4, 2
    q, do = (rng.normal(size=(H, N, d)) for _ in range(2))
    k, v = (rng.normal(size=(H, Nk, d)) for _ in range(2))
    grads = orc.attn_bwd_dropout(q, k, v, do, True, sc, t, seed, bh0=bh0)
    hstep = 1e-6
    for name, x, g in zip(("dQ", "dK", "dV"), (q, k, v), grads):
        num = np.zeros_like(x)
        for idx in np.ndindex(*x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += hstep
            xm[idx] -= hstep
            ap = {"dQ": (xp, k, v), "dK": (q, xp, v), "dV": (q, k, xp)}[name]
            am = {"dQ": (xm, k, v), "dK": (q, xm, v), "dV": (q, k, xm)}[name]
            lp = np.sum(do * orc.attn_fwd_dropout(*ap, True, sc, t, seed, bh0=bh0)[0])
            lm = np.sum(do * orc.attn_fwd_dropout(*am, True, sc, t, seed, bh0=bh0)[0])
            num[idx] = (lp - lm) / (2 * hstep)
        err = np.max(np.abs(num - g)) / max(1e-3, np.max(np.abs(g)))
        assert err < 1e-6, f"head-offset dropout {name} vs finite differences: {err:.2e}"


# ---------------------------------------------------------------------------
# variable-length packed sequences


def pin_varlen_brute_force(orc):
    """Packed sequences [tokens, H, d] with offsets: brute force per sequence and head with
    Python floats, including an empty sequence and, with causal, Nk > Nq per sequence; a
    sequence with no keys (and, causal, one with fewer keys than queries) gives O = 0 and
    lse = -inf on its rows."""
    rng = np.random.default_rng(38)
    H, d = 2, 3
    cu_q, cu_k = [0, 3, 3, 8, 10, 13], [0, 5, 7, 13, 13, 15]
    q = rng.uniform(-1, 1, (cu_q[-1], H, d))
    k = rng.uniform(-1, 1, (cu_k[-1], H, d))
    v = rng.uniform(-2, 2, (cu_k[-1], H, d))
    for causal in (False, True):
        o, lse = orc.attn_fwd_varlen(q, k, v, cu_q, cu_k, causal, 0.8)
        for b in range(len(cu_q) - 1):
            nq, nk = cu_q[b + 1] - cu_q[b], cu_k[b + 1] - cu_k[b]
            for h in range(H):
                qb = q[cu_q[b]:cu_q[b + 1], h].tolist()
                if not qb:
                    continue
                if nk == 0 or (causal and nk < nq):
                    assert np.all(o[cu_q[b]:cu_q[b + 1], h] == 0.0), f"degenerate seq {b}: O not zero"
                    assert np.all(np.isneginf(lse[h, cu_q[b]:cu_q[b + 1]])), f"degenerate seq {b}: lse not -inf"
                    continue
                kb, vb = k[cu_k[b]:cu_k[b + 1], h].tolist(), v[cu_k[b]:cu_k[b + 1], h].tolist()
                bo, bl = brute_force_fwd(qb, kb, vb, causal, 0.8)
                _close(o[cu_q[b]:cu_q[b + 1], h], bo, 1e-12, f"varlen O seq {b} head {h} causal={causal}")
                _close(lse[h, cu_q[b]:cu_q[b + 1]], bl, 1e-12, f"varlen LSE seq {b} head {h}")


def pin_varlen_bwd_finite_differences(orc):
    """Central differences of L = sum(dO * O) over every element of the packed q, k and v,
    O from the packed forward (itself pinned by brute force above), match the packed
    backward.  The batch holds a sequence with Nk > Nq, one without queries, a square one,
    one without keys and one with fewer keys than queries (degenerate when causal), so a
    gradient written to the wrong slice, a sequence skipped or a mask misaligned shows up
    as a mismatch ("Understanding FlashAttention, Part 2", section 2.4: the backward is the
    chain rule of the forward)."""
    rng = np.random.default_rng(44)
    H, d = 2, 3
    cu_q, cu_k = [0, 3, 3, 7, 9, 12], [0, 5, 7, 11, 11, 13]
    Tq, Tk = cu_q[-1], cu_k[-1]
    q, do = rng.normal(size=(Tq, H, d)), rng.normal(size=(Tq, H, d))
    k, v = rng.normal(size=(Tk, H, d)), rng.normal(size=(Tk, H, d))
    scale, h = 0.7, 1e-6
    for causal in (False, True):
        dq, dk, dv = orc.attn_bwd_varlen(q, k, v, do, cu_q, cu_k, causal, scale)
        for name, x, g in (("dQ", q, dq), ("dK", k, dk), ("dV", v, dv)):
            num = np.zeros_like(x)
            for idx in np.ndindex(*x.shape):
                vals = []
                for sgn in (1.0, -1.0):
                    xs = x.copy()
                    xs[idx] += sgn * h
                    args = {"dQ": (xs, k, v), "dK": (q, xs, v), "dV": (q, k, xs)}[name]
                    vals.append(np.sum(do * orc.attn_fwd_varlen(*args, cu_q, cu_k, causal, scale)[0]))
                num[idx] = (vals[0] - vals[1]) / (2 * h)
            err = np.max(np.abs(num - g)) / max(1e-3, np.max(np.abs(g)))
            assert err < 1e-6, f"packed {name} vs finite differences (causal={causal}): {err:.2e}"


ALL_PINS = [
    pin_golden_closed_forms, pin_brute_force, pin_rows_sum_to_one, pin_equal_scores,
    pin_merge_rule, pin_online_recurrence, pin_one_hot_large_scores, pin_causal_first_row,
    pin_permutation_symmetry, pin_sampled_rows, pin_bwd_finite_differences,
    pin_bwd_invariants, pin_bwd_autograd,
    pin_e4m3_closed_forms, pin_e4m3_all_codes_vs_torch, pin_dequant_brute_force,
    pin_fp8_attention_brute_force, pin_rect_causal_is_a_suffix,
    pin_philox_known_answers, pin_dropout_mask_definition, pin_dropout_rate_and_unbiased,
    pin_dropout_t0_is_plain, pin_dropout_brute_force, pin_dropout_bwd_finite_differences,
    pin_dropout_head_offset, pin_varlen_brute_force, pin_varlen_bwd_finite_differences,
]

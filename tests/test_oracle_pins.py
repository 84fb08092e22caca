"""Pins for the CPU oracle: what the definition of attention fixes, checked
without trusting the oracle itself (closed forms, invariants, brute force,
finite differences, an independent numpy restatement, a worked example).

CPU only; the shapes keep the whole file to a few seconds.
"""
import json
import math
import os

import numpy as np
import pytest

from oracle import np_ref

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rnd(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def qkv(B, N, H, Hkv, d, seed):
    return rnd((B, N, H, d), seed), rnd((B, N, Hkv, d), seed + 1), rnd((B, N, Hkv, d), seed + 2)


# ---------------------------------------------------------------- worked example
@pytest.mark.parametrize("causal", [False, True])
def test_golden_two_token(oracle_mod, causal):
    with open(os.path.join(GOLDEN, "two_token.json")) as f:
        g = json.load(f)
    inp = g["inputs"]
    env = {"e": math.e, "log": math.log}
    ev = lambda a: np.array([[eval(x, env) for x in r] for r in a], dtype=np.float64)
    q = np.array(inp["q"], float)[None, :, None, :]
    k = np.array(inp["k"], float)[None, :, None, :]
    v = np.array(inp["v"], float)[None, :, None, :]
    dO = np.array(inp["dO"], float)[None, :, None, :]
    exp = g["causal" if causal else "noncausal"]
    o, lse = oracle_mod.attention_fwd(q, k, v, inp["scale"], causal)
    np.testing.assert_allclose(o[0, :, 0, :], ev(exp["O"]), rtol=0, atol=1e-14)
    np.testing.assert_allclose(lse[0, 0], [eval(x, env) for x in exp["LSE"]], rtol=0, atol=1e-14)
    dq, dk, dv = oracle_mod.attention_bwd(q, k, v, dO, inp["scale"], causal)
    np.testing.assert_allclose(dq[0, :, 0, :], ev(exp["dQ"]), rtol=0, atol=1e-14)
    np.testing.assert_allclose(dk[0, :, 0, :], ev(exp["dK"]), rtol=0, atol=1e-14)
    np.testing.assert_allclose(dv[0, :, 0, :], ev(exp["dV"]), rtol=0, atol=1e-14)


# ---------------------------------------------------------------- closed forms
@pytest.mark.parametrize("causal", [False, True])
def test_constant_v_gives_constant_o(oracle_mod, causal):
    """Rows of P sum to 1: with every V row equal to u, every O row is u."""
    q, k, _ = qkv(2, 33, 4, 2, 16, 10)
    u = rnd((16,), 3)
    v = np.broadcast_to(u, (2, 33, 2, 16)).copy()
    o, _ = oracle_mod.attention_fwd(q, k, v, 0.3, causal)
    np.testing.assert_allclose(o, np.broadcast_to(u, o.shape), rtol=0, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_zero_q_gives_mean_of_visible_v(oracle_mod, causal):
    B, N, H, d = 1, 17, 2, 8
    _, k, v = qkv(B, N, H, H, d, 20)
    q = np.zeros((B, N, H, d))
    o, lse = oracle_mod.attention_fwd(q, k, v, 0.125, causal)
    for i in range(N):
        nvis = i + 1 if causal else N
        np.testing.assert_allclose(o[0, i], v[0, :nvis].mean(axis=0), rtol=0, atol=1e-13)
        np.testing.assert_allclose(lse[0, :, i], math.log(nvis), rtol=0, atol=1e-13)


def test_causal_row0_is_v0(oracle_mod):
    q, k, v = qkv(2, 9, 3, 3, 8, 30)
    o, lse = oracle_mod.attention_fwd(q, k, v, 0.7, True)
    np.testing.assert_allclose(o[:, 0], v[:, 0], rtol=0, atol=1e-14)
    expect = 0.7 * np.einsum("bhc,bhc->bh", q[:, 0], k[:, 0])
    np.testing.assert_allclose(lse[:, :, 0], expect, rtol=0, atol=1e-13)


def test_single_key_gives_o_equals_v(oracle_mod):
    q, k, v = qkv(3, 1, 2, 2, 8, 40)
    o, lse = oracle_mod.attention_fwd(q, k, v, 0.5, False)
    np.testing.assert_allclose(o, v, rtol=0, atol=1e-14)
    np.testing.assert_allclose(lse, 0.5 * np.einsum("bnhc,bnhc->bhn", q, k), rtol=0, atol=1e-13)


def test_dominant_key_gives_one_hot(oracle_mod):
    """A key aligned with q and scaled far beyond the rest makes P one-hot."""
    B, N, H, d = 1, 12, 1, 4
    q = np.zeros((B, N, H, d)); q[..., 0] = 1.0
    k = rnd((B, N, H, d), 50) * 0.01
    k[0, 5, 0, 0] = 2000.0
    v = rnd((B, N, H, d), 51)
    o, _ = oracle_mod.attention_fwd(q, k, v, 1.0, False)
    np.testing.assert_allclose(o[0, :, 0], np.broadcast_to(v[0, 5, 0], (N, d)), rtol=0, atol=1e-12)


# ---------------------------------------------------------------- invariants
@pytest.mark.parametrize("causal", [False, True])
def test_key_shift_invariance(oracle_mod, causal):
    """Adding u to every key row leaves O unchanged and shifts LSE_i by scale q_i.u."""
    B, N, H, d = 2, 21, 2, 8
    q, k, v = qkv(B, N, H, H, d, 60)
    u = rnd((d,), 61)
    s = 0.4
    o1, l1 = oracle_mod.attention_fwd(q, k, v, s, causal)
    o2, l2 = oracle_mod.attention_fwd(q, k + u, v, s, causal)
    np.testing.assert_allclose(o2, o1, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l2 - l1, s * np.einsum("bnhc,c->bhn", q, u), rtol=0, atol=1e-12)
    # dQ depends on keys only through differences k_j - k_j' (rows of dS sum to 0)
    dO = rnd(q.shape, 62)
    dq1, dk1, dv1 = oracle_mod.attention_bwd(q, k, v, dO, s, causal)
    dq2, dk2, dv2 = oracle_mod.attention_bwd(q, k + u, v, dO, s, causal)
    np.testing.assert_allclose(dq2, dq1, rtol=0, atol=1e-12)
    np.testing.assert_allclose(dk2, dk1, rtol=0, atol=1e-12)
    np.testing.assert_allclose(dv2, dv1, rtol=0, atol=1e-12)


def test_kv_permutation_invariance(oracle_mod):
    B, N, H, d = 1, 19, 2, 8
    q, k, v = qkv(B, N, H, H, d, 70)
    perm = np.random.default_rng(71).permutation(N)
    o1, l1 = oracle_mod.attention_fwd(q, k, v, 0.3, False)
    o2, l2 = oracle_mod.attention_fwd(q, k[:, perm], v[:, perm], 0.3, False)
    np.testing.assert_allclose(o2, o1, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l2, l1, rtol=0, atol=1e-12)
    dO = rnd(q.shape, 72)
    dq1, dk1, dv1 = oracle_mod.attention_bwd(q, k, v, dO, 0.3, False)
    dq2, dk2, dv2 = oracle_mod.attention_bwd(q, k[:, perm], v[:, perm], dO, 0.3, False)
    np.testing.assert_allclose(dq2, dq1, rtol=0, atol=1e-12)
    np.testing.assert_allclose(dk2, dk1[:, perm], rtol=0, atol=1e-12)
    np.testing.assert_allclose(dv2, dv1[:, perm], rtol=0, atol=1e-12)


def test_causal_row_is_prefix_attention(oracle_mod):
    """Brute force: causal row i equals non-causal attention over keys 0..i."""
    B, N, H, d = 1, 13, 2, 8
    q, k, v = qkv(B, N, H, H, d, 80)
    o, lse = oracle_mod.attention_fwd(q, k, v, 0.5, True)
    for i in range(N):
        oi, li = oracle_mod.attention_fwd(q[:, : i + 1], k[:, : i + 1], v[:, : i + 1], 0.5, False)
        np.testing.assert_allclose(o[:, i], oi[:, i], rtol=0, atol=1e-13)
        np.testing.assert_allclose(lse[:, :, i], li[:, :, i], rtol=0, atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_gqa_equals_repeated_kv(oracle_mod, causal):
    """Query head h reads kv head h // (H/Hkv); the gradient of a shared kv head
    is the sum over its query heads."""
    B, N, H, Hkv, d = 2, 11, 6, 2, 8
    q, k, v = qkv(B, N, H, Hkv, d, 90)
    dO = rnd(q.shape, 91)
    kr, vr = np.repeat(k, 3, axis=2), np.repeat(v, 3, axis=2)
    o1, l1 = oracle_mod.attention_fwd(q, k, v, 0.3, causal)
    o2, l2 = oracle_mod.attention_fwd(q, kr, vr, 0.3, causal)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-13)
    np.testing.assert_allclose(l1, l2, rtol=0, atol=1e-13)
    dq1, dk1, dv1 = oracle_mod.attention_bwd(q, k, v, dO, 0.3, causal)
    dq2, dk2, dv2 = oracle_mod.attention_bwd(q, kr, vr, dO, 0.3, causal)
    np.testing.assert_allclose(dq1, dq2, rtol=0, atol=1e-12)
    np.testing.assert_allclose(dk1, dk2.reshape(B, N, Hkv, 3, d).sum(3), rtol=0, atol=1e-12)
    np.testing.assert_allclose(dv1, dv2.reshape(B, N, Hkv, 3, d).sum(3), rtol=0, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_backward_linearity_in_v(oracle_mod, causal):
    """O is linear in V: dV does not change with V -> cV, dQ and dK scale by c;
    and the key gradients of one head sum to zero over the keys."""
    q, k, v = qkv(1, 15, 2, 2, 8, 100)
    dO = rnd(q.shape, 101)
    dq1, dk1, dv1 = oracle_mod.attention_bwd(q, k, v, dO, 0.35, causal)
    dq2, dk2, dv2 = oracle_mod.attention_bwd(q, k, 2.5 * v, dO, 0.35, causal)
    np.testing.assert_allclose(dv2, dv1, rtol=0, atol=1e-12)
    np.testing.assert_allclose(dq2, 2.5 * dq1, rtol=0, atol=1e-12)
    np.testing.assert_allclose(dk2, 2.5 * dk1, rtol=0, atol=1e-12)
    np.testing.assert_allclose(dk1.sum(axis=1), 0.0, rtol=0, atol=1e-12)


# ---------------------------------------------------------------- finite differences
@pytest.mark.parametrize("H,Hkv,causal", [(1, 1, False), (2, 2, True), (2, 1, False), (2, 1, True)])
def test_backward_matches_finite_differences(oracle_mod, H, Hkv, causal):
    B, N, d = 1, 6, 5
    q, k, v = qkv(B, N, H, Hkv, d, 110 + H + 3 * Hkv + causal)
    dO = rnd(q.shape, 120)
    s = 0.6
    dq, dk, dv = oracle_mod.attention_bwd(q, k, v, dO, s, causal)

    def loss(q_, k_, v_):
        o, _ = oracle_mod.attention_fwd(q_, k_, v_, s, causal)
        return float((o * dO).sum())

    h = 1e-5
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            args_p = {"q": q, "k": k, "v": v}
            args_m = dict(args_p)
            args_p[name], args_m[name] = xp, xm
            num[idx] = (loss(**{f"{a}_": b for a, b in args_p.items()})
                        - loss(**{f"{a}_": b for a, b in args_m.items()})) / (2 * h)
        err = np.abs(num - g).max() / max(np.abs(g).max(), 1e-30)
        assert err < 1e-6, (name, err)


# ---------------------------------------------------------------- independent restatement
@pytest.mark.parametrize("B,N,H,Hkv,d,causal", [(1, 128, 2, 2, 64, False), (2, 37, 4, 2, 16, True),
                                                (1, 50, 3, 1, 32, False), (1, 64, 2, 2, 8, True)])
def test_c_oracle_matches_numpy_restatement(oracle_mod, B, N, H, Hkv, d, causal):
    q, k, v = qkv(B, N, H, Hkv, d, 130 + N)
    dO = rnd(q.shape, 131)
    s = 1.0 / math.sqrt(d)
    o1, l1 = oracle_mod.attention_fwd(q, k, v, s, causal)
    o2, l2 = np_ref.fwd(q, k, v, s, causal)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l1, l2, rtol=0, atol=1e-12)
    g1 = oracle_mod.attention_bwd(q, k, v, dO, s, causal)
    g2 = np_ref.bwd(q, k, v, dO, s, causal)
    for a, b in zip(g1, g2):
        np.testing.assert_allclose(a, b, rtol=0, atol=1e-11)


@pytest.mark.parametrize("causal", [False, True])
def test_row_selection_matches_full(oracle_mod, causal):
    B, N, H, Hkv, d = 2, 40, 4, 2, 8
    q, k, v = qkv(B, N, H, Hkv, d, 140)
    dO = rnd(q.shape, 141)
    rows = np.array([39, 0, 17, 5])
    o, l = oracle_mod.attention_fwd(q, k, v, 0.3, causal)
    os_, ls_ = oracle_mod.attention_fwd(q, k, v, 0.3, causal, rows=rows)
    np.testing.assert_array_equal(os_, o[:, rows])
    np.testing.assert_array_equal(ls_, l[:, :, rows])
    dq, dk, dv = oracle_mod.attention_bwd(q, k, v, dO, 0.3, causal)
    dqs, dks, dvs = oracle_mod.attention_bwd(q, k, v, dO, 0.3, causal, qrows=rows, kvrows=rows[::-1])
    np.testing.assert_array_equal(dqs, dq[:, rows])
    np.testing.assert_array_equal(dks, dk[:, rows[::-1]])
    np.testing.assert_array_equal(dvs, dv[:, rows[::-1]])


# ---------------------------------------------------------------- packed variable-length batches
def test_varlen_single_row_sequences_are_closed_form(oracle_mod):
    # every sequence has one row: softmax over one key, so O = v and LSE = scale q.k
    total, H, Hkv, d, scale = 5, 4, 2, 8, 0.3
    q, k, v = rnd((total, H, d), 1), rnd((total, Hkv, d), 2), rnd((total, Hkv, d), 3)
    cu = np.arange(total + 1)
    for causal in (False, True):
        o, lse = oracle_mod.attention_fwd_varlen(q, k, v, cu, scale, causal)
        kv = np.repeat(np.arange(Hkv), H // Hkv)
        np.testing.assert_allclose(o, v[:, kv, :], rtol=0, atol=1e-15)
        np.testing.assert_allclose(lse, scale * np.einsum("thd,thd->ht", q, k[:, kv, :]), rtol=1e-14, atol=1e-14)


def test_varlen_equal_lengths_match_the_batched_problem(oracle_mod):
    B, N, H, Hkv, d = 3, 7, 4, 2, 8
    q, k, v = qkv(B, N, H, Hkv, d, 40)
    dO = rnd((B, N, H, d), 44)
    cu = np.arange(B + 1) * N
    for causal in (False, True):
        o, lse = oracle_mod.attention_fwd(q, k, v, 0.4, causal)
        ov, lv = oracle_mod.attention_fwd_varlen(q.reshape(B * N, H, d), k.reshape(B * N, Hkv, d),
                                                 v.reshape(B * N, Hkv, d), cu, 0.4, causal)
        np.testing.assert_array_equal(ov, o.reshape(B * N, H, d))
        np.testing.assert_array_equal(lv, lse.transpose(1, 0, 2).reshape(H, B * N))
        g = oracle_mod.attention_bwd(q, k, v, dO, 0.4, causal)
        gv = oracle_mod.attention_bwd_varlen(q.reshape(B * N, H, d), k.reshape(B * N, Hkv, d),
                                             v.reshape(B * N, Hkv, d), dO.reshape(B * N, H, d), cu, 0.4, causal)
        for a, b in zip(gv, g):
            np.testing.assert_array_equal(a, b.reshape(a.shape))


def test_varlen_sequences_do_not_see_each_other(oracle_mod):
    # changing sequence 1 leaves sequence 0's outputs and gradients unchanged
    H, Hkv, d = 2, 1, 8
    cu = np.array([0, 5, 9])
    q, k, v = rnd((9, H, d), 50), rnd((9, Hkv, d), 51), rnd((9, Hkv, d), 52)
    dO = rnd((9, H, d), 53)
    o1, l1 = oracle_mod.attention_fwd_varlen(q, k, v, cu, 0.5, False)
    g1 = oracle_mod.attention_bwd_varlen(q, k, v, dO, cu, 0.5, False)
    k2, v2 = k.copy(), v.copy()
    k2[5:] += 3.0
    v2[5:] -= 2.0
    o2, l2 = oracle_mod.attention_fwd_varlen(q, k2, v2, cu, 0.5, False)
    g2 = oracle_mod.attention_bwd_varlen(q, k2, v2, dO, cu, 0.5, False)
    np.testing.assert_array_equal(o1[:5], o2[:5])
    np.testing.assert_array_equal(l1[:, :5], l2[:, :5])
    for a, b in zip(g1, g2):
        np.testing.assert_array_equal(a[:5], b[:5])
    assert not np.allclose(o1[5:], o2[5:])


def test_oracle_results_do_not_depend_on_its_thread_count(oracle_mod):
    # rows are split across OpenMP threads, each computed in a fixed order: the
    # one-thread run the CPU baseline times gives the same numbers
    q, k, v = qkv(1, 128, 2, 2, 64, 4400)
    dO = rnd((1, 128, 2, 64), 4404)
    scale = 1.0 / math.sqrt(64)
    full = oracle_mod.attention_fwd(q, k, v, scale, False)
    grads = oracle_mod.attention_bwd(q, k, v, dO, scale, False)
    n = oracle_mod.num_threads()
    oracle_mod.set_threads(1)
    try:
        assert oracle_mod.num_threads() == 1
        one = oracle_mod.attention_fwd(q, k, v, scale, False)
        grads1 = oracle_mod.attention_bwd(q, k, v, dO, scale, False)
    finally:
        oracle_mod.set_threads(n)
    for a, b in zip(full + tuple(grads), one + tuple(grads1)):
        assert np.array_equal(a, b)


# ---------------------------------------------------------------- automatic differentiation
@pytest.mark.parametrize("B,N,H,Hkv,d,causal", [(2, 37, 4, 2, 16, False), (2, 37, 4, 2, 16, True),
                                                (1, 64, 2, 1, 32, True), (1, 1, 1, 1, 8, True)])
def test_backward_matches_autograd_of_the_definition(oracle_mod, B, N, H, Hkv, d, causal):
    """The oracle's backward (row terms D = rowsum(dO o O), dS = P o (dP - D)) against
    torch's automatic differentiation of softmax(scale Q K^T + mask) V in float64, and its
    LSE against torch.logsumexp: two computations that share nothing with the oracle."""
    torch = pytest.importorskip("torch")
    q, k, v = qkv(B, N, H, Hkv, d, 150 + N + causal)
    dO = rnd(q.shape, 151)
    s = 1.0 / math.sqrt(d)
    tq, tk, tv = (torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (q, k, v))
    g = H // Hkv
    kk = tk.repeat_interleave(g, dim=2)  # query head h reads kv head h // g
    vv = tv.repeat_interleave(g, dim=2)
    scores = torch.einsum("bihc,bjhc->bhij", tq, kk) * s
    if causal:
        scores = scores.masked_fill(torch.ones(N, N, dtype=torch.bool).triu(1), float("-inf"))
    o = torch.einsum("bhij,bjhc->bihc", torch.softmax(scores, dim=-1), vv)
    (o * torch.tensor(dO)).sum().backward()
    o1, l1 = oracle_mod.attention_fwd(q, k, v, s, causal)
    np.testing.assert_allclose(o1, o.detach().numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(l1, torch.logsumexp(scores, dim=-1).detach().numpy(), rtol=0, atol=1e-12)
    dq, dk, dv = oracle_mod.attention_bwd(q, k, v, dO, s, causal)
    for name, a, t in (("dq", dq, tq), ("dk", dk, tk), ("dv", dv, tv)):
        np.testing.assert_allclose(a, t.grad.numpy(), rtol=0, atol=1e-11, err_msg=name)

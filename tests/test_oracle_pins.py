"""Pins of the FP64 oracle to facts other than itself.

Each test checks the oracle against a closed form, an invariant of the gated
delta rule, a hand-worked golden case, a special case that reduces to a
known value, or a second algorithm (the chunk form).  They run on the CPU.

Phase contracts exercised here come from the pages:
  * "PR #35197 report: fix(kernel) Fix Helion small-token prefill bug",
    implementation steps 1-2 and the kda_prefill.py / kda_decode.py snippets
    (indexed pool required, padded gate/beta rows trimmed, T=1 prefill).
  * "[KDA] Support Helion MTP verification and harden prefill, decode"
    (sglang PR #42857), Modifications and the review thread (chain/tree
    verify with per-candidate snapshots, commit of an accepted prefix).
"""
import os

import numpy as np
import pytest

from oracle import kda_oracle as ko
from linear_attention_serving_gated_gb300 import inputs
from tests.chunk_form import chunk_prefill

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
RNG = np.random.default_rng(1234)


def _read_golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *nums = line.split()
            vals[key] = np.array([float(x) for x in nums])
    return vals


def _plain_gate(H, K, V, scale=None):
    """No fold: g is the log-decay, beta used as given, no q/k norm."""
    return ko.Gate(H, K, V, A_log=None, beta_is_raw=False, use_qk_l2norm=False,
                   scale=scale if scale is not None else 1.0)


def _one_seq(gate, q, k, v, g, beta, S0, **kw):
    """Prefill one sequence of one head from S0 ([K,V]); returns o, S_T."""
    T, K = q.shape
    V = v.shape[1]
    pool = np.ascontiguousarray(S0.T[None, None], dtype=np.float64)  # [1,1,V,K]
    o = ko.prefill(gate, q.reshape(T, 1, K).astype(np.float32), k.reshape(T, 1, K).astype(np.float32),
                   v.reshape(T, 1, V).astype(np.float32), g.reshape(T, 1, K).astype(np.float32),
                   np.asarray(beta, np.float32).reshape(T, 1), pool, [0], **kw)
    return o[:, 0, :], pool[0, 0].T.copy()


# --------------------------------------------------------------------------- #
# Hand-worked scalar case.

def test_scalar_three_steps_golden():
    gd = _read_golden("scalar_gated_delta_3step.txt")
    gate = _plain_gate(1, 1, 1, scale=gd["scale"][0])
    S0 = np.array([[gd["S0"][0]]])
    col = lambda x: x.reshape(-1, 1)
    o, S = _one_seq(gate, col(gd["q"]), col(gd["k"]), col(gd["v"]), col(gd["g"]), gd["beta"], S0)
    np.testing.assert_allclose(o[:, 0], gd["o"], rtol=0, atol=1e-7)
    np.testing.assert_allclose(S[0, 0], gd["S"][-1], rtol=0, atol=1e-7)
    # per-step states through the chain verify (snapshot i = state after token i)
    x = np.zeros((3, 3), np.float32)
    x[:, 0], x[:, 1], x[:, 2] = gd["q"], gd["k"], gd["v"]
    pool = np.array([[[[gd["S0"][0]]]]])
    o2, snaps = ko.verify(gate, x, gd["g"].reshape(3, 1).astype(np.float32),
                          gd["beta"].reshape(3, 1).astype(np.float32), 1, 3, pool, [0])
    np.testing.assert_allclose(snaps[0, :, 0, 0, 0], gd["S"], atol=1e-7)
    np.testing.assert_allclose(o2[0, :, 0, 0], gd["o"], atol=1e-7)


# --------------------------------------------------------------------------- #
# Fold: gate, beta and the L2 norm reduce to known values at special inputs.

def _decay_ratio(a_val, A_log, dt, lb=-5.0, K=2, V=2):
    """Observe exp(g) through a pure-decay step (beta = 0)."""
    gate = ko.Gate(1, K, V, A_log=np.array([A_log], np.float32),
                   dt_bias=np.full((1, K), dt, np.float32), lower_bound=lb, beta_is_raw=False,
                   use_qk_l2norm=False, scale=1.0)
    pool = np.ones((1, 1, V, K))
    x = np.zeros((1, 2 * K + V), np.float32)
    x[0, :K] = 1.0
    x[0, K:2 * K] = 1.0
    a = np.full((1, K), a_val, np.float32)
    ko.decode(gate, x, a, np.zeros((1, 1), np.float32), pool, [0])
    return pool[0, 0, 0, 0]


def test_gate_special_values():
    lb = -5.0
    # sigmoid(0) = 1/2: a + dt_bias = 0 gives g = lb/2 whatever A_log is
    assert _decay_ratio(0.25, 0.7, -0.25) == pytest.approx(np.exp(lb / 2), rel=1e-12)
    # exp(A_log) -> 0 also gives g = lb/2
    assert _decay_ratio(3.0, -200.0, 0.0) == pytest.approx(np.exp(lb / 2), rel=1e-12)
    # a -> +inf saturates at the bound, a -> -inf gives no decay
    assert _decay_ratio(1e4, 0.0, 0.0) == pytest.approx(np.exp(lb), rel=1e-12)
    assert _decay_ratio(-1e4, 0.0, 0.0) == pytest.approx(1.0, rel=1e-12)
    # the bound scales g linearly
    assert _decay_ratio(0.0, 0.0, 0.0, lb=-2.0) == pytest.approx(np.exp(-1.0), rel=1e-12)
    # exp(A_log) multiplies (a + dt_bias): A_log = ln 2, a + dt = 1 -> sigmoid(2)
    r = _decay_ratio(0.75, float(np.float32(np.log(2.0))), 0.25)
    A = float(np.float32(np.log(2.0)))
    assert np.log(r) == pytest.approx(lb / (1 + np.exp(-np.exp(A) * 1.0)), rel=1e-12)


def test_gate_range_random():
    lb = -5.0
    K = V = 16
    gate = ko.Gate(1, K, V, A_log=np.array([0.3], np.float32),
                   dt_bias=RNG.normal(0, 0.1, (1, K)).astype(np.float32), lower_bound=lb,
                   beta_is_raw=False, use_qk_l2norm=False)
    pool = np.ones((1, 1, V, K))
    x = RNG.standard_normal((1, 2 * K + V)).astype(np.float32)
    a = (RNG.standard_normal((1, K)) * 4).astype(np.float32)
    ko.decode(gate, x, a, np.zeros((1, 1), np.float32), pool, [0])
    ratios = pool[0, 0, 0]
    assert np.all(ratios <= 1.0) and np.all(ratios >= np.exp(lb))


def test_beta_sigmoid_and_l2norm():
    K, V = 2, 3
    gate = ko.Gate(1, K, V, A_log=None, beta_is_raw=True, use_qk_l2norm=True, scale=0.5)
    pool = np.zeros((1, 1, V, K))
    x = np.zeros((1, 2 * K + V), np.float32)
    x[0, :K] = [6.0, 8.0]          # q parallel to k
    x[0, K:2 * K] = [3.0, 4.0]     # k, |k| = 5
    x[0, 2 * K:] = [1.0, -2.0, 4.0]
    o = ko.decode(gate, x, np.zeros((1, K), np.float32), np.zeros((1, 1), np.float32), pool, [0])
    # S1 = beta k^ v^T with beta = sigmoid(0) = 1/2 and k^ = (0.6, 0.8)
    expect = 0.5 * np.outer([0.6, 0.8], [1.0, -2.0, 4.0])
    np.testing.assert_allclose(pool[0, 0].T, expect, atol=1e-7)
    # o = scale * S1^T q^ = 0.5 * 0.5 * v (q^ = k^)
    np.testing.assert_allclose(o[0, 0], 0.25 * np.array([1.0, -2.0, 4.0]), atol=1e-7)
    # q orthogonal to k reads nothing; a large raw beta saturates at 1
    pool[:] = 0
    x[0, :K] = [-4.0, 3.0]
    o = ko.decode(gate, x, np.zeros((1, K), np.float32), np.full((1, 1), 1e4, np.float32),
                  pool, [0])
    np.testing.assert_allclose(o[0, 0], 0.0, atol=1e-7)
    np.testing.assert_allclose(pool[0, 0].T, np.outer([0.6, 0.8], [1.0, -2.0, 4.0]), atol=1e-7)


# --------------------------------------------------------------------------- #
# Invariants of the update rule.

def test_beta0_g0_leaves_state_unchanged():
    K, V, T = 16, 12, 5
    S0 = RNG.standard_normal((K, V))
    q = RNG.standard_normal((T, K))
    o, S = _one_seq(_plain_gate(1, K, V, scale=0.3), q, RNG.standard_normal((T, K)),
                    RNG.standard_normal((T, V)), np.zeros((T, K)), np.zeros(T), S0)
    assert np.array_equal(S, S0)  # bit for bit
    np.testing.assert_allclose(o, 0.3 * q.astype(np.float32).astype(np.float64) @ S0, atol=1e-12)


def test_projection_with_unit_key():
    """g = 0, beta = 1, |k| = 1: the new state maps k to v exactly."""
    K, V = 8, 5
    S0 = RNG.standard_normal((K, V))
    k = RNG.standard_normal(K)
    k /= np.linalg.norm(k)
    k = k.astype(np.float32).astype(np.float64)
    k /= np.linalg.norm(k)
    v = RNG.standard_normal(V).astype(np.float32)
    gate = _plain_gate(1, K, V, scale=1.0)
    o, S = _one_seq(gate, k[None], k[None], v[None], np.zeros((1, K)), [1.0], S0)
    kf = k.astype(np.float32).astype(np.float64)
    # k is passed through float32, so S^T k = v up to |k|^2 - 1 ~ 1e-7
    np.testing.assert_allclose(S.T @ kf, v, atol=2e-6)
    # reading with q = k returns scale * S^T k = v (output uses the updated state)
    np.testing.assert_allclose(o[0], v, atol=2e-6)


def test_orthonormal_keys_closed_form():
    """g = 0, beta = 1, mutually orthonormal keys: S_m = (I - sum k k^T) S0 + sum k v^T."""
    K, V, m = 6, 4, 4
    Q, _ = np.linalg.qr(RNG.standard_normal((K, K)))
    keys = Q[:, :m].T
    gate = ko.Gate(1, K, V, A_log=None, beta_is_raw=False, use_qk_l2norm=True, scale=1.0)
    S0 = RNG.standard_normal((K, V))
    vals = RNG.standard_normal((m, V)).astype(np.float32)
    kf = keys.astype(np.float32)
    o, S = _one_seq(gate, kf, kf, vals, np.zeros((m, K)), np.ones(m), S0)
    kn = kf.astype(np.float64) / np.sqrt((kf.astype(np.float64) ** 2).sum(1, keepdims=True) + 1e-6)
    expect = (np.eye(K) - kn.T @ kn) @ S0 + kn.T @ vals
    np.testing.assert_allclose(S, expect, atol=2e-6)


def test_pure_decay_closed_form():
    K, V, T = 8, 7, 37
    S0 = RNG.standard_normal((K, V))
    g = -RNG.uniform(0, 0.5, (T, K)).astype(np.float32)
    o, S = _one_seq(_plain_gate(1, K, V), RNG.standard_normal((T, K)), RNG.standard_normal((T, K)),
                    RNG.standard_normal((T, V)), g, np.zeros(T), S0)
    expect = np.exp(g.astype(np.float64).sum(0))[:, None] * S0
    np.testing.assert_allclose(S, expect, rtol=1e-12, atol=0)


def test_affine_in_initial_state():
    K, V, T = 8, 6, 20
    args = (RNG.standard_normal((T, K)), RNG.standard_normal((T, K)), RNG.standard_normal((T, V)),
            -RNG.uniform(0, 1, (T, K)), RNG.uniform(0, 1, T))
    gate = _plain_gate(1, K, V, scale=0.7)
    Sa, Sb = RNG.standard_normal((K, V)), RNG.standard_normal((K, V))
    oa, Ta = _one_seq(gate, *args, Sa)
    ob, Tb = _one_seq(gate, *args, Sb)
    oz, Tz = _one_seq(gate, *args, np.zeros((K, V)))
    os_, Ts = _one_seq(gate, *args, Sa + Sb)
    np.testing.assert_allclose(Ts, Ta + Tb - Tz, atol=1e-12)
    np.testing.assert_allclose(os_, oa + ob - oz, atol=1e-12)


def test_dense_matrix_restatement_tiny():
    """Explicit (I - beta k k^T) Diag(e^g) S + beta k v^T with dense numpy matrices
    (catches a transposed state layout in the C loops)."""
    K, V, T = 4, 3, 6
    q, k = RNG.standard_normal((T, K)), RNG.standard_normal((T, K))
    v, g, b = RNG.standard_normal((T, V)), -RNG.uniform(0, 1, (T, K)), RNG.uniform(0, 1, T)
    S0 = RNG.standard_normal((K, V))
    f = lambda x: np.asarray(x, np.float32).astype(np.float64)
    o, S = _one_seq(_plain_gate(1, K, V, scale=0.9), q, k, v, g, b, S0)
    St = S0.copy()
    for t in range(T):
        kt = f(k[t])
        St = (np.eye(K) - f(b[t]) * np.outer(kt, kt)) @ np.diag(np.exp(f(g[t]))) @ St \
            + f(b[t]) * np.outer(kt, f(v[t]))
        np.testing.assert_allclose(o[t], 0.9 * St.T @ f(q[t]), atol=1e-12)
    np.testing.assert_allclose(S, St, atol=1e-12)


def test_chunk_form_agrees_with_token_recurrence():
    """The chunk form (a different algorithm) reproduces the oracle over several
    chunks with a ragged tail, including strong decay."""
    K, V, T = 16, 12, 150
    f = lambda x: np.asarray(x, np.float32).astype(np.float64)
    q = RNG.standard_normal((T, K))
    q /= np.linalg.norm(q, axis=1, keepdims=True)
    k = RNG.standard_normal((T, K))
    k /= np.linalg.norm(k, axis=1, keepdims=True)
    v = RNG.standard_normal((T, V))
    g = -5.0 / (1 + np.exp(-RNG.standard_normal((T, K)) * 2))
    b = RNG.uniform(0, 1, T)
    S0 = RNG.standard_normal((K, V)) * 0.1
    o, S = _one_seq(_plain_gate(1, K, V, scale=K ** -0.5), q, k, v, g, b, S0)
    oc, Sc, _ = chunk_prefill(f(q), f(k), f(v), f(g), f(b), S0, K ** -0.5)
    np.testing.assert_allclose(oc, o, atol=1e-10)
    np.testing.assert_allclose(Sc, S, atol=1e-10)


# --------------------------------------------------------------------------- #
# Phase relations (verify, tree, commit, T=1, padding, varlen, carry-over).

H, K, V = 2, 16, 16


def _gate():
    rng = np.random.default_rng(7)
    A_log, dt = inputs.gate_params(rng, H, K)
    return ko.Gate(H, K, V, A_log=A_log, dt_bias=dt, lower_bound=-5.0)


def test_verify_snapshot_i_equals_i_plus_1_decode_steps():
    gate = _gate()
    d = inputs.verify_inputs(seed=3, B=3, T=5, H=H, K=K, V=V, slots=6)
    pool = d["pool"].astype(np.float64)
    o, snaps = ko.verify(gate, d["mixed_qkv"], d["a"], d["b"], 3, 5, pool, d["state_idx"])
    dec_pool = pool.copy()
    x = d["mixed_qkv"].reshape(3, 5, -1)
    a = d["a"].reshape(3, 5, -1)
    b = d["b"].reshape(3, 5, -1)
    for i in range(5):
        od = ko.decode(gate, x[:, i], a[:, i], b[:, i], dec_pool, d["state_idx"])
        np.testing.assert_allclose(od, o[:, i], atol=1e-13)
        np.testing.assert_allclose(dec_pool[d["state_idx"]], snaps[:, i], atol=1e-13)
    assert np.array_equal(pool, d["pool"].astype(np.float64))  # verify leaves the pool alone


def test_tree_with_chain_parents_equals_chain():
    gate = _gate()
    d = inputs.verify_inputs(seed=4, B=2, T=6, H=H, K=K, V=V, slots=4)
    pool = d["pool"].astype(np.float64)
    chain = np.tile(np.arange(-1, 5, dtype=np.int32), (2, 1))
    o1, s1 = ko.verify(gate, d["mixed_qkv"], d["a"], d["b"], 2, 6, pool, d["state_idx"])
    o2, s2 = ko.verify(gate, d["mixed_qkv"], d["a"], d["b"], 2, 6, pool, d["state_idx"], parent=chain)
    assert np.array_equal(o1, o2) and np.array_equal(s1, s2)


def test_tree_node_equals_chain_along_its_root_path():
    gate = _gate()
    B, T = 3, 6
    d = inputs.verify_inputs(seed=5, B=B, T=T, H=H, K=K, V=V, slots=5)
    pool = d["pool"].astype(np.float64)
    par = d["parent"]
    o, snaps = ko.verify(gate, d["mixed_qkv"], d["a"], d["b"], B, T, pool, d["state_idx"], parent=par)
    for r in range(B):
        for i in range(T):
            path = []
            n = i
            while n >= 0:
                path.append(n)
                n = par[r, n]
            path = path[::-1]
            rows = [r * T + n for n in path]
            oc, sc = ko.verify(gate, d["mixed_qkv"][rows], d["a"][rows], d["b"][rows], 1, len(path),
                               pool, d["state_idx"][r:r + 1])
            np.testing.assert_allclose(oc[0, -1], o[r, i], atol=1e-13)
            np.testing.assert_allclose(sc[0, -1], snaps[r, i], atol=1e-13)


def test_commit_copies_accepted_snapshot():
    gate = _gate()
    B, T = 3, 4
    d = inputs.verify_inputs(seed=6, B=B, T=T, H=H, K=K, V=V, slots=7)
    pool = d["pool"].astype(np.float64)
    before = pool.copy()
    _, snaps = ko.verify(gate, d["mixed_qkv"], d["a"], d["b"], B, T, pool, d["state_idx"])
    acc = np.array([2, -1, 0], np.int32)
    ko.commit(snaps, acc, pool, d["state_idx"])
    idx = d["state_idx"]
    assert np.array_equal(pool[idx[0]], snaps[0, 2])
    assert np.array_equal(pool[idx[1]], before[idx[1]])
    assert np.array_equal(pool[idx[2]], snaps[2, 0])
    untouched = np.setdiff1d(np.arange(7), idx[[0, 2]])
    assert np.array_equal(pool[untouched], before[untouched])


def test_T1_prefill_equals_one_decode_step():
    gate = _gate()
    d = inputs.prefill_inputs(seed=8, lengths=[1], H=H, K=K, V=V, slots=3, gb_rows=4)
    pool_p = d["pool"].astype(np.float64)
    pool_d = pool_p.copy()
    o = ko.prefill(gate, d["q"], d["k"], d["v"], d["g"], d["beta"], pool_p, d["state_idx"],
                   d["cu_seqlens"])
    x = np.concatenate([d["q"].reshape(1, -1), d["k"].reshape(1, -1), d["v"].reshape(1, -1)], 1)
    od = ko.decode(gate, x, d["g"][:1].reshape(1, -1), d["beta"][:1], pool_d, d["state_idx"])
    np.testing.assert_allclose(o, od, atol=1e-14)
    np.testing.assert_allclose(pool_p, pool_d, atol=1e-14)


def test_padding_rows_are_never_read():
    gate = _gate()
    d = inputs.prefill_inputs(seed=9, lengths=[40, 1, 25], H=H, K=K, V=V, slots=5, gb_rows=100)
    assert np.isnan(ko.bf16_to_f32(d["g"][66:])).any()
    p1 = d["pool"].astype(np.float64)
    p2 = p1.copy()
    o1 = ko.prefill(gate, d["q"], d["k"], d["v"], d["g"], d["beta"], p1, d["state_idx"], d["cu_seqlens"])
    o2 = ko.prefill(gate, d["q"], d["k"], d["v"], d["g"][:66].copy(), d["beta"][:66].copy(), p2,
                    d["state_idx"], d["cu_seqlens"])
    assert np.isfinite(o1).all()
    assert np.array_equal(o1, o2) and np.array_equal(p1, p2)
    with pytest.raises(ko.OracleError):  # gate/beta must cover every q token
        ko.prefill(gate, d["q"], d["k"], d["v"], d["g"][:65], d["beta"][:65], p2, d["state_idx"],
                   d["cu_seqlens"])


def test_varlen_equals_separate_calls_and_fixed_layout():
    gate = _gate()
    lens = [70, 1, 0, 64, 33]
    d = inputs.prefill_inputs(seed=10, lengths=lens, H=H, K=K, V=V, slots=8)
    pool = d["pool"].astype(np.float64)
    ref_pool = pool.copy()
    o = ko.prefill(gate, d["q"], d["k"], d["v"], d["g"], d["beta"], pool, d["state_idx"], d["cu_seqlens"])
    cu = d["cu_seqlens"]
    for n in range(len(lens)):
        s, e = cu[n], cu[n + 1]
        on = ko.prefill(gate, d["q"][s:e], d["k"][s:e], d["v"][s:e], d["g"][s:e], d["beta"][s:e],
                        ref_pool, d["state_idx"][n:n + 1], np.array([0, e - s], np.int32))
        np.testing.assert_array_equal(on, o[s:e])
    np.testing.assert_array_equal(pool, ref_pool)
    # fixed layout (no cu_seqlens) with equal lengths equals the varlen call
    d2 = inputs.prefill_inputs(seed=11, lengths=[48, 48], H=H, K=K, V=V, slots=4)
    pa, pb = d2["pool"].astype(np.float64), d2["pool"].astype(np.float64)
    oa = ko.prefill(gate, d2["q"], d2["k"], d2["v"], d2["g"], d2["beta"], pa, d2["state_idx"],
                    d2["cu_seqlens"])
    ob = ko.prefill(gate, d2["q"], d2["k"], d2["v"], d2["g"], d2["beta"], pb, d2["state_idx"], None,
                    num_seqs=2)
    assert np.array_equal(oa, ob) and np.array_equal(pa, pb)


def test_chunked_prefill_across_calls():
    """prefill(T1) then prefill(T2) from the scattered state == prefill(T1 + T2)."""
    gate = _gate()
    d = inputs.prefill_inputs(seed=12, lengths=[150], H=H, K=K, V=V, slots=2)
    p_full = d["pool"].astype(np.float64)
    p_split = p_full.copy()
    o_full = ko.prefill(gate, d["q"], d["k"], d["v"], d["g"], d["beta"], p_full, d["state_idx"],
                        d["cu_seqlens"])
    sl = lambda x, a, b: x[a:b].copy()
    o1 = ko.prefill(gate, *(sl(d[n], 0, 90) for n in ("q", "k", "v", "g", "beta")), p_split,
                    d["state_idx"], np.array([0, 90], np.int32))
    o2 = ko.prefill(gate, *(sl(d[n], 90, 150) for n in ("q", "k", "v", "g", "beta")), p_split,
                    d["state_idx"], np.array([0, 60], np.int32))
    np.testing.assert_allclose(np.concatenate([o1, o2]), o_full, atol=1e-13)
    np.testing.assert_allclose(p_split, p_full, atol=1e-13)


def test_intermediate_states_are_chunk_start_states():
    gate = _gate()
    lens = [130, 64, 5]
    d = inputs.prefill_inputs(seed=13, lengths=lens, H=H, K=K, V=V, slots=4)
    pool = d["pool"].astype(np.float64)
    start_pool = pool.copy()
    _, inter = ko.prefill(gate, d["q"], d["k"], d["v"], d["g"], d["beta"], pool, d["state_idx"],
                          d["cu_seqlens"], intermediate=True)
    assert inter.shape[0] == 3 + 1 + 1
    cu = d["cu_seqlens"]
    ci = 0
    for n, L in enumerate(lens):
        for c0 in range(0, L, 64):
            p = start_pool.copy()
            s = cu[n]
            if c0:
                ko.prefill(gate, *(d[x][s:s + c0].copy() for x in ("q", "k", "v", "g", "beta")), p,
                           d["state_idx"][n:n + 1], np.array([0, c0], np.int32))
            np.testing.assert_allclose(inter[ci], p[d["state_idx"][n]], atol=1e-13)
            ci += 1


def test_pool_indexing_and_padding_requests():
    gate = _gate()
    d = inputs.decode_inputs(seed=14, B=4, H=H, K=K, V=V, slots=9)
    pool = d["pool"].astype(np.float64)
    before = pool.copy()
    idx = d["state_idx"].copy()
    idx[2] = -1  # padding request
    o = ko.decode(gate, d["mixed_qkv"], d["a"], d["b"], pool, idx)
    assert np.all(o[2] == 0)
    untouched = np.setdiff1d(np.arange(9), idx[idx >= 0])
    assert np.array_equal(pool[untouched], before[untouched])
    for r in (0, 1, 3):
        assert not np.array_equal(pool[idx[r]], before[idx[r]])


def test_invalid_inputs_are_rejected():
    gate = _gate()
    d = inputs.verify_inputs(seed=15, B=2, T=3, H=H, K=K, V=V, slots=4)
    pool = d["pool"].astype(np.float64)
    with pytest.raises(ko.OracleError):
        ko.verify(gate, d["mixed_qkv"], d["a"], d["b"], 2, 3, pool, np.array([1, 1], np.int32))
    bad = np.array([[-1, 1, 0], [-1, 0, 1]], np.int32)  # parent[1] = 1 is not < 1
    with pytest.raises(ko.OracleError):
        ko.verify(gate, d["mixed_qkv"], d["a"], d["b"], 2, 3, pool, d["state_idx"], parent=bad)
    with pytest.raises(ko.OracleError):
        ko.verify(gate, d["mixed_qkv"], d["a"], d["b"], 2, 3, pool, np.array([0, 4], np.int32))


# --------------------------------------------------------------------------- #
# Grouped value heads: HV = G * H, value head h reading q/k head h // G.  The
# same call with every q/k head repeated G times (H' = HV) takes the plain
# one-q/k-head-per-value-head path and must give the same bits.

G_GROUP = 2


def _group_gate(Hq, HV, A_log, dt_bias):
    return ko.Gate(Hq, K, V, HV=HV, A_log=A_log, dt_bias=dt_bias, lower_bound=-5.0)


def _repeat_packed_qk(x, Hq):
    """Packed rows [q (Hq*K) | k (Hq*K) | v] -> [q repeated | k repeated | v]."""
    rows = x.shape[0]
    q = np.repeat(x[:, :Hq * K].reshape(rows, Hq, K), G_GROUP, axis=1).reshape(rows, -1)
    k = np.repeat(x[:, Hq * K:2 * Hq * K].reshape(rows, Hq, K), G_GROUP, axis=1).reshape(rows, -1)
    return np.ascontiguousarray(np.concatenate([q, k, x[:, 2 * Hq * K:]], axis=1))


def test_grouped_value_heads_prefill_equals_repeated_qk():
    Hq, HV = 2, 2 * G_GROUP
    d = inputs.prefill_inputs(seed=21, lengths=[70, 33], H=Hq, HV=HV, K=K, V=V, slots=4)
    pool_g = d["pool"].astype(np.float64)
    pool_p = pool_g.copy()
    o_g, st_g = ko.prefill(_group_gate(Hq, HV, d["A_log"], d["dt_bias"]), d["q"], d["k"], d["v"], d["g"],
                           d["beta"], pool_g, d["state_idx"], d["cu_seqlens"], intermediate=True)
    o_p, st_p = ko.prefill(_group_gate(HV, HV, d["A_log"], d["dt_bias"]), np.repeat(d["q"], G_GROUP, axis=1),
                           np.repeat(d["k"], G_GROUP, axis=1), d["v"], d["g"], d["beta"], pool_p,
                           d["state_idx"], d["cu_seqlens"], intermediate=True)
    assert np.array_equal(o_g, o_p) and np.array_equal(st_g, st_p) and np.array_equal(pool_g, pool_p)
    # value heads of one group read the same q/k but their own v, gate and state
    assert not np.array_equal(o_g[:, 0], o_g[:, 1])


def test_grouped_value_heads_decode_and_verify_equal_repeated_qk():
    Hq, HV = 2, 2 * G_GROUP
    d = inputs.decode_inputs(seed=22, B=3, H=Hq, HV=HV, K=K, V=V, slots=5)
    pool_g = d["pool"].astype(np.float64)
    pool_p = pool_g.copy()
    o_g = ko.decode(_group_gate(Hq, HV, d["A_log"], d["dt_bias"]), d["mixed_qkv"], d["a"], d["b"], pool_g,
                    d["state_idx"])
    o_p = ko.decode(_group_gate(HV, HV, d["A_log"], d["dt_bias"]), _repeat_packed_qk(d["mixed_qkv"], Hq),
                    d["a"], d["b"], pool_p, d["state_idx"])
    assert np.array_equal(o_g, o_p) and np.array_equal(pool_g, pool_p)

    v = inputs.verify_inputs(seed=23, B=2, T=4, H=Hq, HV=HV, K=K, V=V, slots=5)
    pool = v["pool"].astype(np.float64)
    for parent in (None, v["parent"]):
        og, sg = ko.verify(_group_gate(Hq, HV, v["A_log"], v["dt_bias"]), v["mixed_qkv"], v["a"], v["b"], 2, 4,
                           pool, v["state_idx"], parent=parent)
        op, sp = ko.verify(_group_gate(HV, HV, v["A_log"], v["dt_bias"]), _repeat_packed_qk(v["mixed_qkv"], Hq),
                           v["a"], v["b"], 2, 4, pool, v["state_idx"], parent=parent)
        assert np.array_equal(og, op) and np.array_equal(sg, sp)


def test_head_counts_must_group():
    d = inputs.prefill_inputs(seed=24, lengths=[8], H=2, HV=3, K=K, V=V, slots=2)
    with pytest.raises(ko.OracleError):
        ko.prefill(_group_gate(2, 3, d["A_log"], d["dt_bias"]), d["q"], d["k"], d["v"], d["g"], d["beta"],
                   d["pool"].astype(np.float64), d["state_idx"], d["cu_seqlens"])


def test_fp16_token_inputs_widen_exactly():
    """The second token precision, FP16: values that FP16 holds exactly come
    back unchanged from the seeded encoder and the oracle's widening, and
    others round to nearest even (IEEE binary16: 10 fraction bits)."""
    exact = np.array([0.0, 1.0, -2.5, 1.0 + 2.0 ** -10, 65504.0, 2.0 ** -14, 6.103515625e-05,
                      -3.0517578125e-05], np.float32)
    f16 = inputs.encode16(exact, "f16")
    assert f16.dtype == np.float16
    assert np.array_equal(ko.bf16_to_f32(f16), exact)
    # halfway between 1 and 1 + 2^-10 rounds to the even neighbour 1; just above it rounds up
    assert ko.bf16_to_f32(inputs.encode16(np.float32([1.0 + 2.0 ** -11]), "f16"))[0] == 1.0
    assert ko.bf16_to_f32(inputs.encode16(np.float32([1.0 + 3 * 2.0 ** -12]), "f16"))[0] == 1.0 + 2.0 ** -10

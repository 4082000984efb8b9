"""Pins for the fp64 oracle: each test checks it against something other than
itself -- a hand-worked example, a closed form, an invariant, brute force on
tiny inputs, or the independent chunk-form evaluation.  CPU only."""
import math
import os

import numpy as np
import pytest

import oracle
from chunk_mirror import chunk_prefill

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


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


def _rand_inputs(rng, T, H, dk, dv, *, unit=True):
    q = rng.standard_normal((T, H, dk))
    k = rng.standard_normal((T, H, dk))
    if unit:
        q /= np.linalg.norm(q, axis=-1, keepdims=True)
        k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((T, H, dv))
    g = -np.log1p(np.exp(rng.standard_normal((T, H, dk))))
    beta = 1 / (1 + np.exp(-rng.standard_normal((T, H))))
    return q, k, v, g, beta


def _one_seq(T):
    return np.array([0, T], np.int32), np.array([0], np.int32)


# ---------------------------------------------------------------- worked example
def test_hand_worked_example_d2():
    gd = _read_golden("worked_example_d2.txt")
    q = np.stack([gd["q1"], gd["q2"]])[:, None, :]
    k = np.stack([gd["k1"], gd["k2"]])[:, None, :]
    v = np.stack([gd["v1"], gd["v2"]])[:, None, :]
    g = np.stack([gd["g1"], gd["g2"]])[:, None, :]
    beta = np.array([gd["b1"][0], gd["b2"][0]])[:, None]
    pool = gd["s0"].reshape(1, 1, 2, 2)
    cu, idx = _one_seq(2)
    out, pool_after, ck, offs = oracle.prefill(q, k, v, g, beta, cu, idx, pool,
                                               checkpoint_every=1, scale=1.0)
    np.testing.assert_allclose(out[0, 0], gd["o1"], atol=1e-12)
    np.testing.assert_allclose(out[1, 0], gd["o2"], atol=1e-12)
    np.testing.assert_allclose(ck[0, 0].ravel(), gd["s1"], atol=1e-12)
    np.testing.assert_allclose(ck[1, 0].ravel(), gd["s2"], atol=1e-12)
    np.testing.assert_allclose(pool_after[0, 0].ravel(), gd["s2"], atol=1e-12)
    assert offs.tolist() == [0, 2]


def test_hand_worked_norm_gate():
    gd = _read_golden("norm_gate_example.txt")
    y = oracle.norm_gate(gd["o"][None], gd["gate"][None], gd["w"], eps=gd["eps"][0])
    np.testing.assert_allclose(y[0], gd["y"], atol=1e-12)


# ---------------------------------------------------------------- brute force
def _brute_force(q, k, v, g, beta, S0, scale):
    """Materialise each transition M_t = (I - b k k^T) Diag(exp g) as a dense
    matrix and multiply: S_t = M_t S_{t-1} + b k v^T, o_t = scale S_t^T q_t."""
    T, dk = q.shape
    S = S0.copy()
    outs, states = [], []
    for t in range(T):
        M = (np.eye(dk) - beta[t] * np.outer(k[t], k[t])) @ np.diag(np.exp(g[t]))
        S = M @ S + beta[t] * np.outer(k[t], v[t])
        outs.append(scale * S.T @ q[t])
        states.append(S.copy())
    return np.array(outs), states


@pytest.mark.parametrize("dk,dv,T", [(1, 1, 5), (2, 3, 6), (4, 4, 8), (3, 2, 7)])
def test_brute_force_tiny(dk, dv, T):
    rng = np.random.default_rng(100 + dk * 10 + dv)
    H = 2
    q, k, v, g, beta = _rand_inputs(rng, T, H, dk, dv, unit=False)
    pool = rng.standard_normal((3, H, dk, dv))
    cu, idx = np.array([0, T], np.int32), np.array([2], np.int32)
    out, pool_after, ck, _ = oracle.prefill(q, k, v, g, beta, cu, idx, pool, checkpoint_every=2,
                                            scale=0.7)
    for h in range(H):
        o_bf, states = _brute_force(q[:, h], k[:, h], v[:, h], g[:, h], beta[:, h], pool[2, h], 0.7)
        np.testing.assert_allclose(out[:, h], o_bf, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(pool_after[2, h], states[-1], rtol=1e-12, atol=1e-12)
        for m in range(T // 2):
            np.testing.assert_allclose(ck[m, h], states[2 * m + 1], rtol=1e-12, atol=1e-12)
    # untouched slots stay bit-identical
    assert np.array_equal(pool_after[:2], pool[:2])


# ---------------------------------------------------------------- closed forms
def test_single_token_from_zero_state():
    rng = np.random.default_rng(1)
    dk, dv, H = 8, 5, 3
    q, k, v, g, beta = _rand_inputs(rng, 1, H, dk, dv)
    pool = np.zeros((1, H, dk, dv))
    cu, idx = _one_seq(1)
    out, pool_after, _, _ = oracle.prefill(q, k, v, g, beta, cu, idx, pool, scale=0.3)
    for h in range(H):
        S = beta[0, h] * np.outer(k[0, h], v[0, h])
        np.testing.assert_allclose(pool_after[0, h], S, atol=1e-14)
        np.testing.assert_allclose(out[0, h], 0.3 * beta[0, h] * (q[0, h] @ k[0, h]) * v[0, h],
                                   atol=1e-14)


def test_beta0_g0_leaves_state_unchanged():
    rng = np.random.default_rng(2)
    T, H, dk, dv = 9, 2, 6, 4
    q, k, v, _, _ = _rand_inputs(rng, T, H, dk, dv)
    g = np.zeros((T, H, dk))
    beta = np.zeros((T, H))
    pool = rng.standard_normal((2, H, dk, dv))
    cu, idx = np.array([0, T], np.int32), np.array([1], np.int32)
    out, pool_after, _, _ = oracle.prefill(q, k, v, g, beta, cu, idx, pool, scale=0.5)
    assert np.array_equal(pool_after, pool)
    for h in range(H):
        np.testing.assert_allclose(out[:, h], 0.5 * q[:, h] @ pool[1, h], atol=1e-14)


def test_infinite_decay_erases_history():
    rng = np.random.default_rng(3)
    T, H, dk, dv = 6, 2, 4, 4
    q, k, v, _, beta = _rand_inputs(rng, T, H, dk, dv)
    g = np.full((T, H, dk), -1e30)  # exp(-1e30) == 0 exactly in fp64
    pool = rng.standard_normal((1, H, dk, dv))
    cu, idx = _one_seq(T)
    out, pool_after, _, _ = oracle.prefill(q, k, v, g, beta, cu, idx, pool, scale=1.0)
    for h in range(H):
        for t in range(T):
            np.testing.assert_allclose(out[t, h], beta[t, h] * (q[t, h] @ k[t, h]) * v[t, h],
                                       atol=1e-14)
        np.testing.assert_allclose(pool_after[0, h], beta[-1, h] * np.outer(k[-1, h], v[-1, h]),
                                   atol=1e-14)


def test_delta_rule_retrieval_beta1_g0():
    """beta = 1, no decay, unit k: after writing (k_t, v_t) the state maps k_t
    to v_t exactly, so reading with q = k returns v."""
    rng = np.random.default_rng(4)
    T, H, dk, dv = 10, 2, 6, 3
    _, k, v, _, _ = _rand_inputs(rng, T, H, dk, dv)
    g = np.zeros((T, H, dk))
    beta = np.ones((T, H))
    pool = rng.standard_normal((1, H, dk, dv))
    cu, idx = _one_seq(T)
    out, _, _, _ = oracle.prefill(k, k, v, g, beta, cu, idx, pool, scale=1.0)
    np.testing.assert_allclose(out, v, atol=1e-12)


def test_scalar_geometric_closed_form():
    """dk = dv = 1, k = 1, v = 1, beta = 1/2, alpha = 1/2, s0 = 0:
    s_t = (1/4) s_{t-1} + 1/2, whose closed form is s_t = (2/3)(1 - 4^-t)."""
    T = 12
    q = np.ones((T, 1, 1))
    k = np.ones((T, 1, 1))
    v = np.ones((T, 1, 1))
    g = np.full((T, 1, 1), math.log(0.5))
    beta = np.full((T, 1), 0.5)
    pool = np.zeros((1, 1, 1, 1))
    cu, idx = _one_seq(T)
    out, _, _, _ = oracle.prefill(q, k, v, g, beta, cu, idx, pool, scale=1.0)
    t = np.arange(1, T + 1)
    np.testing.assert_allclose(out[:, 0, 0], (2 / 3) * (1 - 4.0 ** (-t)), rtol=1e-14)


# ---------------------------------------------------------------- invariants
def test_split_invariance_and_checkpoint_placement():
    rng = np.random.default_rng(5)
    T, H, dk, dv, I = 96, 2, 8, 6, 16
    q, k, v, g, beta = _rand_inputs(rng, T, H, dk, dv)
    pool = rng.standard_normal((4, H, dk, dv))
    idx = np.array([3], np.int32)
    out1, pool1, ck1, _ = oracle.prefill(q, k, v, g, beta, [0, T], idx, pool, checkpoint_every=I)
    a = 48
    outa, poola, cka, _ = oracle.prefill(q[:a], k[:a], v[:a], g[:a], beta[:a], [0, a], idx, pool,
                                         checkpoint_every=I)
    outb, poolb, ckb, _ = oracle.prefill(q[a:], k[a:], v[a:], g[a:], beta[a:], [0, T - a], idx,
                                         poola, checkpoint_every=I)
    np.testing.assert_allclose(np.concatenate([outa, outb]), out1, atol=1e-12)
    np.testing.assert_allclose(poolb, pool1, atol=1e-12)
    assert ck1.shape[0] == T // I and cka.shape[0] + ckb.shape[0] == T // I
    np.testing.assert_allclose(np.concatenate([cka, ckb]), ck1, atol=1e-12)
    # checkpoint m equals the final state of a prefill over the first (m+1)*I tokens
    for m in range(T // I):
        n = (m + 1) * I
        _, pm, _, _ = oracle.prefill(q[:n], k[:n], v[:n], g[:n], beta[:n], [0, n], idx, pool)
        np.testing.assert_allclose(ck1[m], pm[3], atol=1e-12)


def test_packing_equals_separate_calls_and_offsets():
    rng = np.random.default_rng(6)
    lens = [37, 0, 64, 5, 130]
    T, H, dk, dv, I = sum(lens), 2, 4, 4, 32
    q, k, v, g, beta = _rand_inputs(rng, T, H, dk, dv)
    pool = rng.standard_normal((8, H, dk, dv))
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    idx = np.array([5, 1, 7, -1, 2], np.int32)
    out, pool_after, ck, offs = oracle.prefill(q, k, v, g, beta, cu, idx, pool, checkpoint_every=I)
    assert offs.tolist() == [0, 1, 1, 3, 3, 7]
    assert ck.shape[0] == 7
    for i, L in enumerate(lens):
        t0 = cu[i]
        sl = slice(t0, t0 + L)
        if idx[i] < 0:
            assert np.all(out[sl] == 0)  # padding rows are zeroed
            continue
        o_i, p_i, ck_i, _ = oracle.prefill(q[sl], k[sl], v[sl], g[sl], beta[sl], [0, L],
                                           [idx[i]], pool, checkpoint_every=I)
        np.testing.assert_allclose(out[sl], o_i, atol=1e-13)
        np.testing.assert_allclose(pool_after[idx[i]], p_i[idx[i]], atol=1e-13)
        np.testing.assert_allclose(ck[offs[i]:offs[i + 1]], ck_i, atol=1e-13)
    # slot 1 belongs to a zero-length segment: untouched; slots 0,3,4,6 untouched
    for s in (0, 1, 3, 4, 6):
        assert np.array_equal(pool_after[s], pool[s])


def test_linearity_in_state_and_values():
    rng = np.random.default_rng(7)
    T, H, dk, dv = 20, 1, 5, 4
    q, k, v1, g, beta = _rand_inputs(rng, T, H, dk, dv)
    v2 = rng.standard_normal(v1.shape)
    p1, p2 = rng.standard_normal((2, 1, H, dk, dv))
    cu, idx = _one_seq(T)
    a, b = 0.75, -1.5
    o1, s1, _, _ = oracle.prefill(q, k, v1, g, beta, cu, idx, p1)
    o2, s2, _, _ = oracle.prefill(q, k, v2, g, beta, cu, idx, p2)
    o3, s3, _, _ = oracle.prefill(q, k, a * v1 + b * v2, g, beta, cu, idx, a * p1 + b * p2)
    np.testing.assert_allclose(o3, a * o1 + b * o2, atol=1e-12)
    np.testing.assert_allclose(s3, a * s1 + b * s2, atol=1e-12)


def test_value_columns_are_independent():
    rng = np.random.default_rng(8)
    T, H, dk, dv = 15, 2, 4, 6
    q, k, v, g, beta = _rand_inputs(rng, T, H, dk, dv)
    pool = rng.standard_normal((1, H, dk, dv))
    perm = rng.permutation(dv)
    cu, idx = _one_seq(T)
    o, s, _, _ = oracle.prefill(q, k, v, g, beta, cu, idx, pool)
    op, sp, _, _ = oracle.prefill(q, k, v[..., perm], g, beta, cu, idx, pool[..., perm])
    np.testing.assert_allclose(op, o[..., perm], atol=1e-13)
    np.testing.assert_allclose(sp, s[..., perm], atol=1e-13)


def test_decode_equals_one_token_prefill():
    rng = np.random.default_rng(9)
    N, H, dk, dv = 5, 2, 8, 8
    q, k, v, g, beta = _rand_inputs(rng, N, H, dk, dv)
    gate = rng.standard_normal((N, H, dv))
    w = 1 + 0.02 * rng.standard_normal(dv)
    pool = rng.standard_normal((9, H, dk, dv))
    idx = np.array([4, -1, 0, 8, 2], np.int32)
    o, p = oracle.decode(q, k, v, g, beta, idx, pool, gate=gate, norm_w=w)
    for i in range(N):
        if idx[i] < 0:
            assert np.all(o[i] == 0)
            continue
        S = pool[idx[i]]
        for h in range(H):
            # single-token recurrence written via the expanded transition
            Sn = (np.eye(dk) - beta[i, h] * np.outer(k[i, h], k[i, h])) @ (
                np.exp(g[i, h])[:, None] * S[h]) + beta[i, h] * np.outer(k[i, h], v[i, h])
            np.testing.assert_allclose(p[idx[i], h], Sn, atol=1e-12)
            oh = Sn.T @ q[i, h] / math.sqrt(dk)
            yh = oh / math.sqrt(np.mean(oh ** 2) + 1e-6) * w / (1 + np.exp(-gate[i, h]))
            np.testing.assert_allclose(o[i, h], yh, atol=1e-12)


def test_norm_gate_constant_row_and_scale_invariance():
    rng = np.random.default_rng(10)
    dv = 16
    gate = rng.standard_normal((3, dv))
    w = 1 + 0.02 * rng.standard_normal(dv)
    c = np.array([[2.0] * dv, [-0.5] * dv, [1e-3] * dv])
    y = oracle.norm_gate(c, gate, w, eps=1e-6)
    sig = 1 / (1 + np.exp(-gate))
    expect = (c / np.sqrt(c ** 2 + 1e-6)) * w * sig
    np.testing.assert_allclose(y, expect, rtol=1e-12)
    o = rng.standard_normal((4, dv))
    np.testing.assert_allclose(oracle.norm_gate(1e3 * o, np.zeros((4, dv)), np.ones(dv), eps=0.0),
                               oracle.norm_gate(o, np.zeros((4, dv)), np.ones(dv), eps=0.0),
                               rtol=1e-12)


def test_bad_index_rejected():
    q = np.zeros((2, 1, 2, 2))[:, :, 0]
    with pytest.raises(oracle.OracleError):
        oracle.prefill(q, q, q, q, np.zeros((2, 1)), [0, 2], [5], np.zeros((2, 1, 2, 2)))


# ---------------------------------------------------------------- chunk form
@pytest.mark.parametrize("chunk,lens", [(16, [64]), (16, [37, 5, 16]), (64, [37, 128, 200]),
                                        (64, [1, 63, 65, 64])])
def test_chunk_form_matches_oracle(chunk, lens):
    rng = np.random.default_rng(11 + chunk + len(lens))
    T, H, dk, dv = sum(lens), 2, 16, 8
    q, k, v, g, beta = _rand_inputs(rng, T, H, dk, dv)
    pool = 0.1 * rng.standard_normal((6, H, dk, dv))
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    idx = rng.permutation(6)[:len(lens)].astype(np.int32)
    I = chunk * 2
    out, pool_o, ck_o, _ = oracle.prefill(q, k, v, g, beta, cu, idx, pool, checkpoint_every=I)
    out_c, pool_c, ck_c = chunk_prefill(q, k, v, g, beta, cu, idx, pool, chunk=chunk,
                                        checkpoint_every=I)
    np.testing.assert_allclose(out_c, out, atol=1e-10)
    np.testing.assert_allclose(pool_c, pool_o, atol=1e-10)
    np.testing.assert_allclose(ck_c, ck_o, atol=1e-10)


# ---------------------------------------------------------------- planted mistakes
def test_pins_catch_planted_mistakes():
    """The closed forms above distinguish the recurrence from its plausible
    mis-readings: reading the state before the write, applying the decay after
    the delta-rule residual, or dropping beta from the write."""
    rng = np.random.default_rng(12)
    T, dk, dv = 6, 4, 3
    q, k, v, g, beta = (x[:, 0] for x in _rand_inputs(rng, T, 1, dk, dv))
    S0 = rng.standard_normal((dk, dv))

    def variant(mode):
        S = S0.copy()
        outs = []
        for t in range(T):
            a = np.exp(g[t])
            if mode == "read_before_write":
                Sd = a[:, None] * S
                u = beta[t] * (v[t] - Sd.T @ k[t])
                outs.append(Sd.T @ q[t])
                S = Sd + np.outer(k[t], u)
            elif mode == "decay_after_residual":
                u = beta[t] * (v[t] - S.T @ k[t])
                S = a[:, None] * (S + np.outer(k[t], u))
                outs.append(S.T @ q[t])
            elif mode == "no_beta_write":
                Sd = a[:, None] * S
                u = v[t] - Sd.T @ k[t]
                S = Sd + np.outer(k[t], u)
                outs.append(S.T @ q[t])
        return np.array(outs)

    o_ref, _ = _brute_force(q, k, v, g, beta, S0, 1.0)
    out, _, _, _ = oracle.prefill(q[:, None], k[:, None], v[:, None], g[:, None], beta[:, None],
                                  [0, T], [0], S0[None, None], scale=1.0)
    np.testing.assert_allclose(out[:, 0], o_ref, atol=1e-12)
    for mode in ("read_before_write", "decay_after_residual", "no_beta_write"):
        assert np.max(np.abs(variant(mode) - o_ref)) > 1e-3, mode


def test_hand_worked_norm_gate_silu():
    gd = _read_golden("norm_gate_silu_example.txt")
    y = oracle.norm_gate(gd["o"][None], gd["gate"][None], gd["w"], eps=gd["eps"][0],
                         gate_act="silu")
    np.testing.assert_allclose(y[0], gd["y"], atol=1e-12)


def test_no_initial_state_starts_from_zero():
    """A sequence flagged without initial state computes exactly what the same
    sequence computes from a zeroed slot, whatever the slot held; flagged-with
    sequences are unaffected, and the final state still lands in the slot."""
    rng = np.random.default_rng(13)
    lens = [9, 14, 5]
    T, H, dk, dv = sum(lens), 2, 4, 3
    q, k, v, g, beta = _rand_inputs(rng, T, H, dk, dv)
    pool = rng.standard_normal((5, H, dk, dv))
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    idx = np.array([4, 0, 2], np.int32)
    flags = np.array([1, 0, 1], np.int32)
    out, pool_a, _, _ = oracle.prefill(q, k, v, g, beta, cu, idx, pool, has_initial_state=flags)
    zeroed = pool.copy()
    zeroed[0] = 0.0
    out_z, pool_z, _, _ = oracle.prefill(q, k, v, g, beta, cu, idx, zeroed)
    np.testing.assert_allclose(out, out_z, atol=1e-14)
    np.testing.assert_allclose(pool_a, pool_z, atol=1e-14)
    out_all, _, _, _ = oracle.prefill(q, k, v, g, beta, cu, idx, pool)
    np.testing.assert_allclose(out[:9], out_all[:9], atol=1e-14)
    assert np.max(np.abs(out[9:23] - out_all[9:23])) > 1e-6  # the flag did change seq 1


def test_multi_token_decode_equals_prefill_with_per_token_checkpoints():
    """K decode steps per sequence are the prefill of those K tokens: the
    outputs agree, and the state after token t is the prefill's checkpoint
    t when a checkpoint is taken after every token.  Committing a_i accepted
    tokens leaves the slot at checkpoint a_i - 1 (unchanged for a_i = 0)."""
    rng = np.random.default_rng(21)
    N, K, H, dk, dv = 4, 5, 2, 6, 4
    q, k, v, g, beta = _rand_inputs(rng, N * K, H, dk, dv)
    gate = rng.standard_normal((N * K, H, dv))
    w = 1 + 0.1 * rng.standard_normal(dv)
    pool = rng.standard_normal((7, H, dk, dv))
    idx = np.array([3, -1, 0, 6], np.int32)
    sh = lambda x: x.reshape((N, K) + x.shape[1:])
    out, ts, pool_k = oracle.decode_multi(sh(q), sh(k), sh(v), sh(g), sh(beta), idx, pool,
                                          gate=sh(gate), norm_w=w, gate_act="silu")
    live = [i for i in range(N) if idx[i] >= 0]
    cu = np.arange(len(live) + 1, dtype=np.int32) * K
    rows = np.concatenate([np.arange(i * K, (i + 1) * K) for i in live])
    o_p, pool_p, ck, _ = oracle.prefill(q[rows], k[rows], v[rows], g[rows], beta[rows], cu,
                                        idx[live], pool, checkpoint_every=1, gate=gate[rows],
                                        norm_w=w, gate_act="silu")
    np.testing.assert_allclose(out[live].reshape(-1, H, dv), o_p, atol=1e-12)
    np.testing.assert_allclose(ts[live].reshape(-1, H, dk, dv), ck, atol=1e-12)
    np.testing.assert_allclose(pool_k, pool_p, atol=1e-12)
    assert np.all(out[1] == 0) and np.all(np.isnan(ts[1]))
    acc = np.array([2, 3, 0, K], np.int32)
    committed = oracle.commit_accepted(ts, acc, idx, pool)
    np.testing.assert_allclose(committed[3], ck[1], atol=1e-12)
    np.testing.assert_array_equal(committed[0], pool[0])
    np.testing.assert_allclose(committed[6], pool_p[6], atol=1e-12)
    untouched = [s for s in range(7) if s not in (3, 0, 6)]
    np.testing.assert_array_equal(committed[untouched], pool[untouched])
    # one step of the expanded transition pins token 0 independently of both routines
    S = pool[3, 1]
    i0 = 0
    Sn = (np.eye(dk) - beta[i0, 1] * np.outer(k[i0, 1], k[i0, 1])) @ (
        np.exp(g[i0, 1])[:, None] * S) + beta[i0, 1] * np.outer(k[i0, 1], v[i0, 1])
    np.testing.assert_allclose(ts[0, 0, 1], Sn, atol=1e-12)


def test_hand_worked_norm_gate_ex():
    """Residual + affine weight + bias, both activations, against the values
    worked by hand in the fixture; the prenorm output is x = o + residual."""
    gd = _read_golden("norm_gate_ex_example.txt")
    sh = lambda a: a.reshape(1, 1, -1)
    for act, key in (("sigmoid", "y_sigmoid"), ("silu", "y_silu")):
        y, x = oracle.norm_gate_ex(sh(gd["o"]), sh(gd["gate"]), residual=sh(gd["residual"]),
                                   w=gd["w"], b=gd["b"], eps=gd["eps"][0], gate_act=act)
        np.testing.assert_allclose(y[0, 0], gd[key], atol=1e-12)
        np.testing.assert_allclose(x[0, 0], gd["x"], atol=0)


def test_norm_gate_ex_reductions():
    """Special cases that pin each option of the variant entry: no residual,
    unit weight and zero bias reduce to the plain norm-gate; no weight equals
    unit weight; the bias enters as b * act(gate); a packed gate row (stride
    > H*dv, heads at their offsets) equals the contiguous gate; the residual
    path equals the plain norm-gate of o + residual."""
    rng = np.random.default_rng(31)
    rows, H, dv = 5, 3, 8
    o = rng.standard_normal((rows, H, dv))
    res = rng.standard_normal((rows, H, dv))
    gate = rng.standard_normal((rows, H, dv))
    w = 1 + 0.1 * rng.standard_normal(dv)
    b = 0.3 * rng.standard_normal(dv)
    for act in ("sigmoid", "silu"):
        ref = oracle.norm_gate(o, gate, w, eps=1e-6, gate_act=act)
        y, x = oracle.norm_gate_ex(o, gate, w=w, gate_act=act)
        np.testing.assert_allclose(y, ref, atol=1e-14)
        np.testing.assert_array_equal(x, o)
        y1, _ = oracle.norm_gate_ex(o, gate, w=np.ones(dv), gate_act=act)
        y0, _ = oracle.norm_gate_ex(o, gate, gate_act=act)
        np.testing.assert_allclose(y0, y1, atol=1e-14)
        yb, _ = oracle.norm_gate_ex(o, gate, w=w, b=b, gate_act=act)
        sig = 1 / (1 + np.exp(-gate))
        a = sig if act == "sigmoid" else gate * sig
        np.testing.assert_allclose(yb - ref, b * a, atol=1e-13)
        packed = rng.standard_normal((rows, H * dv + 40))
        packed[:, 16:16 + H * dv] = gate.reshape(rows, -1)
        yp, _ = oracle.norm_gate_ex(o, packed[:, 16:].copy(), w=w, gate_act=act,
                                    gate_row_stride=H * dv + 24)
        np.testing.assert_allclose(yp, ref, atol=1e-14)
        yr, xr = oracle.norm_gate_ex(o, gate, residual=res, w=w, gate_act=act)
        np.testing.assert_allclose(xr, o + res, atol=1e-15)
        np.testing.assert_allclose(yr, oracle.norm_gate(o + res, gate, w, eps=1e-6, gate_act=act),
                                   atol=1e-14)


# ------------------------------------------------------------ short causal conv
def test_hand_worked_conv():
    gd = _read_golden("conv_example.txt")
    x = gd["x"].reshape(-1, 1)
    pool = gd["cache"].reshape(1, 2, 1)
    cu, idx = np.array([0, len(x)], np.int32), np.array([0], np.int32)
    y, p = oracle.conv_prefill(x, gd["w"].reshape(1, 3), cu, idx, pool, act="none")
    np.testing.assert_allclose(y[:, 0], gd["y"], atol=0)
    np.testing.assert_allclose(p[0, :, 0], gd["cache_after"], atol=0)
    ys, _ = oracle.conv_prefill(x, gd["w"].reshape(1, 3), cu, idx, pool, act="silu")
    np.testing.assert_allclose(ys[2, 0], gd["silu_y2"][0], atol=1e-13)


def _conv_inputs(rng, lens, C, W, slots=9):
    T = sum(lens)
    x = rng.standard_normal((T, C))
    w = rng.standard_normal((C, W))
    b = rng.standard_normal(C)
    pool = rng.standard_normal((slots, W - 1, C))
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    return x, w, b, pool, cu


@pytest.mark.parametrize("W", [1, 2, 4])
def test_conv_matches_numpy_convolve(W):
    """Each channel of each sequence is numpy's full convolution of the
    extended sequence (cache then inputs) with the reversed taps, shifted so
    that only past and current inputs enter."""
    rng = np.random.default_rng(40 + W)
    lens, C = [7, 1, 0, 12], 5
    x, w, b, pool, cu = _conv_inputs(rng, lens, C, W)
    idx = np.array([3, 0, 5, 8], np.int32)
    y, p = oracle.conv_prefill(x, w, cu, idx, pool, bias=b, act="none")
    for i, L in enumerate(lens):
        if L == 0:
            continue
        for c in range(C):
            xe = np.concatenate([pool[idx[i], :, c], x[cu[i]:cu[i + 1], c]])
            full = np.convolve(xe, w[c, ::-1])       # full[n] = sum_k w[c, W-1-k'] ...
            ref = full[W - 1:W - 1 + L] + b[c]        # outputs aligned to the current input
            np.testing.assert_allclose(y[cu[i]:cu[i + 1], c], ref, atol=1e-12)
            if W > 1:
                np.testing.assert_allclose(p[idx[i], :, c], xe[-(W - 1):], atol=0)
    np.testing.assert_array_equal(p[5], pool[5])  # the empty sequence leaves its slot


def test_conv_split_decode_and_flags():
    """Two calls carrying the cache through the pool equal one call; K decode
    steps equal the prefill of those K tokens; a sequence without initial
    state equals one whose cache is zero; padding rows are zero and leave the
    pool alone; SiLU is applied to the pre-activation."""
    rng = np.random.default_rng(77)
    C, W = 6, 4
    x, w, b, pool, cu = _conv_inputs(rng, [11], C, W)
    idx = np.array([2], np.int32)
    y, p = oracle.conv_prefill(x, w, cu, idx, pool, bias=b)
    y1, p1 = oracle.conv_prefill(x[:5], w, np.array([0, 5], np.int32), idx, pool, bias=b)
    y2, p2 = oracle.conv_prefill(x[5:], w, np.array([0, 6], np.int32), idx, p1, bias=b)
    np.testing.assert_allclose(np.concatenate([y1, y2]), y, atol=1e-13)
    np.testing.assert_allclose(p2, p, atol=0)
    pd, ys = pool, []
    for t in range(11):
        yt, pd = oracle.conv_decode(x[t:t + 1], w, idx, pd, bias=b)
        ys.append(yt[0])
    np.testing.assert_allclose(np.array(ys), y, atol=1e-13)
    np.testing.assert_allclose(pd, p, atol=0)
    zeroed = pool.copy()
    zeroed[2] = 0
    yz, _ = oracle.conv_prefill(x, w, cu, idx, zeroed, bias=b)
    yf, _ = oracle.conv_prefill(x, w, cu, idx, pool, bias=b, has_initial_state=np.array([0], np.int32))
    np.testing.assert_allclose(yf, yz, atol=0)
    yp, pp = oracle.conv_prefill(x, w, cu, np.array([-1], np.int32), pool, bias=b)
    assert np.all(yp == 0) and np.array_equal(pp, pool)
    ya, _ = oracle.conv_prefill(x, w, cu, idx, pool, bias=b, act="none")
    np.testing.assert_allclose(y, ya / (1 + np.exp(-ya)), atol=1e-14)


def test_l2_normalize_hand_worked_and_invariants():
    """x / sqrt(sum x^2 + eps): [3, 4] -> [0.6, 0.8] (eps = 0), a zero row
    stays zero, and rows of any scale come out with norm sqrt(s / (s + eps))."""
    np.testing.assert_allclose(oracle.l2_normalize(np.array([[3.0, 4.0]]), eps=0.0), [[0.6, 0.8]],
                               rtol=0, atol=1e-15)
    assert not np.any(oracle.l2_normalize(np.zeros((2, 5))))
    rng = np.random.default_rng(5)
    x = rng.standard_normal((7, 3, 16)) * rng.uniform(1e-2, 1e2, (7, 3, 1))
    y = oracle.l2_normalize(x, eps=1e-6)
    s = np.sum(x * x, axis=-1)
    np.testing.assert_allclose(np.linalg.norm(y, axis=-1), np.sqrt(s / (s + 1e-6)), rtol=1e-13)
    # direction unchanged: y is a positive multiple of x
    np.testing.assert_allclose(y * np.linalg.norm(x, axis=-1, keepdims=True),
                               x * np.linalg.norm(y, axis=-1, keepdims=True), rtol=1e-12, atol=1e-12)


def test_prefill_conv_with_identity_taps_is_the_plain_prefill():
    """A convolution whose only tap is the current token (taps [0, 0, 0, 1], no
    bias, no activation) passes x through, so on q, k rows that already have
    unit norm the composed operator is the plain prefill; v is passed through
    unnormalised; the cache afterwards holds each sequence's last 3 inputs."""
    rng = np.random.default_rng(21)
    T, H, dd = 16, 2, 8
    q, k, v, g, beta = _rand_inputs(rng, T, H, dd, dd)
    cu = np.array([0, 5, 16], np.int32)
    idx = np.array([3, 1], np.int32)
    pool = rng.standard_normal((4, H, dd, dd)) * 0.1
    C = 3 * H * dd
    taps = np.zeros((C, 4))
    taps[:, 3] = 1.0
    conv_pool = rng.standard_normal((4, 3, C))
    out_c, pool_c, _, _, conv_after = oracle.prefill_conv(
        q, k, v, taps, cu, idx, pool, conv_pool, conv_act="none", l2_eps=0.0, g=g, beta=beta)
    out_p, pool_p, _, _ = oracle.prefill(q, k, v, g, beta, cu, idx, pool)
    np.testing.assert_allclose(out_c, out_p, rtol=0, atol=1e-12)
    np.testing.assert_allclose(pool_c, pool_p, rtol=0, atol=1e-12)
    x = np.concatenate([a.reshape(T, H * dd) for a in (q, k, v)], axis=1)
    for i, slot in enumerate(idx.tolist()):
        np.testing.assert_array_equal(conv_after[slot], x[cu[i + 1] - 3:cu[i + 1]])


def test_prefill_conv_order_of_stages():
    """Swapping the q and k channel blocks, or normalising v as well, changes
    the result: the composition reads the blocks in the order q, k, v and
    normalises q and k only."""
    rng = np.random.default_rng(33)
    _, _, _, g, beta = _rand_inputs(rng, 9, 1, 4, 4)
    cu, idx = _one_seq(9)
    pool = rng.standard_normal((1, 1, 4, 4)) * 0.1
    C = 12
    taps = rng.standard_normal((C, 4)) * 0.5
    conv_pool = rng.standard_normal((1, 3, C))
    xq, xk, xv = (rng.standard_normal((9, 1, 4)) for _ in range(3))
    kw = dict(conv_act="silu", g=g, beta=beta)
    ref = oracle.prefill_conv(xq, xk, xv, taps, cu, idx, pool, conv_pool, **kw)[0]
    perm = [*range(4, 8), *range(4), *range(8, 12)]
    swapped = oracle.prefill_conv(xk, xq, xv, taps[perm], cu, idx, pool, conv_pool[:, :, perm], **kw)[0]
    assert np.max(np.abs(ref - swapped)) > 1e-3
    y, _ = oracle.conv_prefill(np.concatenate([xq[:, 0], xk[:, 0], xv[:, 0]], axis=1), taps, cu, idx,
                               conv_pool, act="silu")
    q, k, v = (y[:, 4 * i:4 * i + 4].reshape(9, 1, 4) for i in range(3))
    # v normalised as well (a plausible mistake) gives another answer
    wrong = oracle.prefill(oracle.l2_normalize(q), oracle.l2_normalize(k), oracle.l2_normalize(v), g,
                           beta, cu, idx, pool)[0]
    assert np.max(np.abs(ref - wrong)) > 1e-3
    right = oracle.prefill(oracle.l2_normalize(q), oracle.l2_normalize(k), v, g, beta, cu, idx, pool)[0]
    np.testing.assert_allclose(ref, right, rtol=0, atol=1e-12)

"""Pins for the oracle: checks of the fp64 token recurrence (and of the chunked
algebra beside it) against what the pages and the mathematics fix — values
the TPU report prints, closed forms, invariants and brute force on tiny
inputs. Nothing here touches the CUDA path. Runs with ``-m "not gpu"``.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
from oracle import chunked

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "page_constants.json")


def rand_case(rng, seqlens, H, K, V, state=True, g_lo=-5.0):
    T = sum(seqlens)
    q = rng.standard_normal((T, H, K))
    k = rng.standard_normal((T, H, K))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    q /= np.linalg.norm(q, axis=-1, keepdims=True)
    v = rng.standard_normal((T, H, V))
    g = g_lo * rng.random((T, H, K))
    beta = rng.random((T, H))
    cu = np.concatenate([[0], np.cumsum(seqlens)]).astype(np.int64)
    s0 = rng.standard_normal((len(seqlens), H, K, V)) * 0.5 if state else None
    return q, k, v, g, beta, cu, s0


def seq_cumsum(g, cu):
    """Inclusive per-sequence prefix sum of g over tokens (test-side helper)."""
    G = np.zeros_like(g)
    for n in range(len(cu) - 1):
        G[cu[n]:cu[n + 1]] = np.cumsum(g[cu[n]:cu[n + 1]], axis=0)
    return G


# ----------------------------------------------------------------- page values

def test_exponent_budget_matches_printed_value():
    gold = json.load(open(GOLDEN))["exponent_budget"]
    b = chunked.exponent_budget(gold["sb"], gold["lower_bound"])
    assert round(b, gold["printed_digits"]) == gold["printed_value"]
    assert b < gold["bf16_exponent_limit_printed"]


def test_strip_factors_reach_but_stay_within_budget():
    # g pinned at lower_bound everywhere: the largest factor a strip forms is
    # exp(8*5) = 2^57.7, exactly the printed budget.
    rng = np.random.default_rng(3)
    n, K = 64, 8
    g = np.full((n, K), -5.0)
    G = chunked.gate_cumsum(g)
    a, b = rng.standard_normal((n, K)), rng.standard_normal((n, K))
    _, worst = chunked.decay_scores_strips(a, b, G, strict=False)
    assert abs(worst - chunked.exponent_budget()) < 1e-9


def test_chunk_table_matches_page_address_example():
    gold = json.load(open(GOLDEN))["unified_addressing_example"]
    cu = np.concatenate([[0], np.cumsum(gold["seqlens"])])
    tab = chunked.chunk_table(cu, gold["chunk_size"])
    assert tab["aligned_cu_seqlens"].tolist() == gold["aligned_cu_seqlens"]
    assert np.diff(tab["aligned_cu_seqlens"]).tolist() == gold["aligned_lengths"]
    pairs = [[int(a), int(b)] for a, b in zip(tab["seq_id"], tab["local_chunk"])]
    assert pairs == gold["chunk_indices"]
    assert tab["aligned_start"].tolist() == gold["starts"]
    # the same starts through the indices: aligned_cu[seq] + local*chunk
    via_idx = [gold["aligned_cu_seqlens"][s] + c * gold["chunk_size"] for s, c in pairs]
    assert via_idx == gold["starts"]
    assert tab["start_flag"].tolist() == [1, 0, 1, 0, 0]
    assert tab["end_flag"].tolist() == [0, 1, 0, 0, 1]
    assert tab["length"].tolist() == [64, 6, 64, 64, 2]


# ---------------------------------------------------------------- closed forms

def test_beta_zero_is_pure_decay_of_initial_state():
    """beta = 0 removes both the erase and the write: S_t = Diag(e^{G_t}) S_0
    with G the inclusive prefix of g, o_t = scale (e^{G_t} * q_t)^T S_0."""
    rng = np.random.default_rng(0)
    q, k, v, g, beta, cu, s0 = rand_case(rng, [37, 0, 70], 2, 8, 6)
    beta[:] = 0.0
    scale = 0.3
    o, sT = oracle.kda_recurrence(q, k, v, g, beta, cu, s0, scale)
    G = seq_cumsum(g, cu)
    for n in range(len(cu) - 1):
        sl = slice(cu[n], cu[n + 1])
        ref_o = scale * np.einsum("thk,hkv->thv", q[sl] * np.exp(G[sl]), s0[n])
        np.testing.assert_allclose(o[sl], ref_o, rtol=1e-12, atol=1e-14)
        Glast = G[cu[n + 1] - 1] if cu[n + 1] > cu[n] else np.zeros_like(G[0])
        np.testing.assert_allclose(sT[n], np.exp(Glast)[:, :, None] * s0[n], rtol=1e-12, atol=1e-15)


def test_g_zero_beta_zero_keeps_state_exactly():
    rng = np.random.default_rng(1)
    q, k, v, g, beta, cu, s0 = rand_case(rng, [20, 9], 3, 8, 8)
    g[:] = 0.0
    beta[:] = 0.0
    o, sT = oracle.kda_recurrence(q, k, v, g, beta, cu, s0, 1.0)
    assert np.array_equal(sT, s0)
    for n in range(2):
        sl = slice(cu[n], cu[n + 1])
        np.testing.assert_allclose(o[sl], np.einsum("thk,hkv->thv", q[sl], s0[n]), rtol=1e-13, atol=1e-15)


def test_beta_one_self_query_reads_back_value():
    """With beta = 1 and a unit key, the delta rule writes exactly: S_t^T k_t = v_t.
    So q_t = k_t gives o_t = scale * v_t for any decay and any state."""
    rng = np.random.default_rng(2)
    q, k, v, g, beta, cu, s0 = rand_case(rng, [50, 31], 2, 16, 12)
    beta[:] = 1.0
    q = k.copy()
    o, _ = oracle.kda_recurrence(q, k, v, g, beta, cu, s0, 0.7)
    np.testing.assert_allclose(o, 0.7 * v, rtol=0, atol=1e-11)


def basis_key_closed_form(q, ch, v, g, beta, scale):
    """Decayed linear attention with a per-channel decay, for keys that are the
    standard basis vectors e_{ch[t]} (distinct within the sequence):
    o_t = scale * sum_{s<=t} beta_s q_t[c_s] exp(G_t[c_s] - G_s[c_s]) v_s and
    S_T = sum_s beta_s exp(G_T[c_s] - G_s[c_s]) e_{c_s} v_s^T. Shapes: q, g [T,K],
    ch [T], v [T,V], beta [T]."""
    T, K = q.shape
    G = np.cumsum(g, axis=0)
    idx = np.arange(T)
    o = np.zeros((T, v.shape[1]))
    for t in range(T):
        c = ch[: t + 1]
        w = beta[: t + 1] * q[t, c] * np.exp(G[t, c] - G[idx[: t + 1], c])
        o[t] = scale * w @ v[: t + 1]
    S = np.zeros((K, v.shape[1]))
    for s in range(T):
        S[ch[s]] += beta[s] * np.exp(G[T - 1, ch[s]] - G[s, ch[s]]) * v[s]
    return o, S


def test_basis_keys_give_decayed_linear_attention():
    """Keys that are distinct standard basis vectors stay orthogonal under any
    diagonal decay, so the erase term vanishes and KDA reduces to decayed
    linear attention with a per-channel decay (closed form above)."""
    rng = np.random.default_rng(4)
    T, H, K, V = 24, 2, 32, 5
    ch = np.stack([rng.permutation(K)[:T] for _ in range(H)], axis=1)  # [T,H]
    k = np.zeros((T, H, K))
    for t in range(T):
        for h in range(H):
            k[t, h, ch[t, h]] = 1.0
    q = rng.standard_normal((T, H, K))
    v = rng.standard_normal((T, H, V))
    g = -5.0 * rng.random((T, H, K))
    beta = rng.random((T, H))
    o, sT = oracle.kda_recurrence(q, k, v, g, beta, [0, T], None, 0.5)
    for h in range(H):
        ref_o, ref_s = basis_key_closed_form(q[:, h], ch[:, h], v[:, h], g[:, h], beta[:, h], 0.5)
        np.testing.assert_allclose(o[:, h], ref_o, rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(sT[0, h], ref_s, rtol=1e-12, atol=1e-14)


def test_orthonormal_keys_scalar_decay_is_masked_matmul():
    """Orthonormal keys and a channel-uniform decay: the erase term vanishes
    and o = scale * (tril(Q K^T * exp(G_t - G_s)) * beta_s) V, one library matmul."""
    rng = np.random.default_rng(5)
    T, K, V = 40, 64, 16
    Qm, _ = np.linalg.qr(rng.standard_normal((K, K)))
    k = Qm[:T][:, None, :]
    q = rng.standard_normal((T, 1, K))
    v = rng.standard_normal((T, 1, V))
    gam = -5.0 * rng.random(T)
    g = np.repeat(gam[:, None, None], K, axis=2)
    beta = rng.random((T, 1))
    o, _ = oracle.kda_recurrence(q, k, v, g, beta, np.array([0, T]), None, 0.25)
    G = np.cumsum(gam)
    M = np.tril((q[:, 0] @ k[:, 0].T) * np.exp(G[:, None] - G[None, :])) * beta[None, :, 0]
    np.testing.assert_allclose(o[:, 0], 0.25 * M @ v[:, 0], rtol=1e-11, atol=1e-13)


# ------------------------------------------------------------------ invariants

def test_packed_varlen_equals_independent_runs():
    rng = np.random.default_rng(6)
    lens = [33, 0, 64, 1, 90]
    q, k, v, g, beta, cu, s0 = rand_case(rng, lens, 2, 8, 8)
    o, sT = oracle.kda_recurrence(q, k, v, g, beta, cu, s0, 0.35)
    for n, L in enumerate(lens):
        sl = slice(cu[n], cu[n + 1])
        oi, si = oracle.kda_recurrence(q[sl], k[sl], v[sl], g[sl], beta[sl], [0, L], s0[n:n + 1], 0.35)
        assert np.array_equal(o[sl], oi)
        assert np.array_equal(sT[n], si[0])


@pytest.mark.parametrize("cut", [64, 128, 37, 1])
def test_split_and_carry_state_equals_full_run(cut):
    rng = np.random.default_rng(7)
    q, k, v, g, beta, cu, s0 = rand_case(rng, [200], 2, 8, 8)
    o, sT = oracle.kda_recurrence(q, k, v, g, beta, cu, s0, 0.35)
    a = slice(0, cut)
    b = slice(cut, 200)
    oa, sa = oracle.kda_recurrence(q[a], k[a], v[a], g[a], beta[a], [0, cut], s0, 0.35)
    ob, sb = oracle.kda_recurrence(q[b], k[b], v[b], g[b], beta[b], [0, 200 - cut], sa, 0.35)
    np.testing.assert_allclose(np.concatenate([oa, ob]), o, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(sb, sT, rtol=1e-13, atol=1e-14)


def test_segment_exit_state_is_affine_in_its_entry_state():
    """The reading behind the split-sequence scan: a segment maps its entry
    state S to Phi S + N, with N its exit state from a zero entry state and
    Phi + N its exit state from the identity; chaining three segments this way
    reproduces the full run's final state, and each segment's o from its
    composed entry state reproduces the full run's o. Computed on the oracle
    with K = V = 12 (the identity needs K = V)."""
    rng = np.random.default_rng(21)
    K = 12
    q, k, v, g, beta, cu, s0 = rand_case(rng, [150], 2, K, K)
    o, sT = oracle.kda_recurrence(q, k, v, g, beta, cu, s0, 0.3)
    eye = np.broadcast_to(np.eye(K), (1, 2, K, K)).copy()
    cuts = [0, 64, 128, 150]
    S = s0
    for a, b in zip(cuts[:-1], cuts[1:]):
        sl = slice(a, b)
        args = (q[sl], k[sl], v[sl], g[sl], beta[sl], [0, b - a])
        _, n0 = oracle.kda_recurrence(*args, None, 0.3)
        _, fi = oracle.kda_recurrence(*args, eye, 0.3)
        phi = fi - n0
        o_seg, s_seg = oracle.kda_recurrence(*args, S, 0.3)
        np.testing.assert_allclose(o_seg, o[sl], rtol=1e-12, atol=1e-13)
        S_next = np.einsum("nhij,nhjc->nhic", phi, S) + n0
        np.testing.assert_allclose(S_next, s_seg, rtol=1e-12, atol=1e-13)
        S = S_next
    np.testing.assert_allclose(S, sT, rtol=1e-12, atol=1e-13)


def test_linear_in_value_and_state_jointly():
    rng = np.random.default_rng(8)
    q, k, v, g, beta, cu, s0 = rand_case(rng, [45, 19], 2, 8, 8)
    _, _, v2, _, _, _, s2 = rand_case(rng, [45, 19], 2, 8, 8)
    o1, f1 = oracle.kda_recurrence(q, k, v, g, beta, cu, s0, 0.4)
    o2, f2 = oracle.kda_recurrence(q, k, v2, g, beta, cu, s2, 0.4)
    o3, f3 = oracle.kda_recurrence(q, k, 2.0 * v - 3.0 * v2, g, beta, cu, 2.0 * s0 - 3.0 * s2, 0.4)
    np.testing.assert_allclose(o3, 2.0 * o1 - 3.0 * o2, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(f3, 2.0 * f1 - 3.0 * f2, rtol=1e-11, atol=1e-12)


def test_heads_independent_and_permutation_equivariant():
    rng = np.random.default_rng(9)
    q, k, v, g, beta, cu, s0 = rand_case(rng, [30, 41], 4, 8, 8)
    p = np.array([2, 0, 3, 1])
    o, sT = oracle.kda_recurrence(q, k, v, g, beta, cu, s0, 0.3)
    op, sp = oracle.kda_recurrence(q[:, p], k[:, p], v[:, p], g[:, p], beta[:, p], cu, s0[:, p], 0.3)
    assert np.array_equal(op, o[:, p])
    assert np.array_equal(sp, sT[:, p])


def test_empty_sequence_passes_state_through():
    rng = np.random.default_rng(10)
    q, k, v, g, beta, cu, s0 = rand_case(rng, [0, 5, 0], 2, 8, 8)
    _, sT = oracle.kda_recurrence(q, k, v, g, beta, cu, s0, 0.3)
    assert np.array_equal(sT[0], s0[0]) and np.array_equal(sT[2], s0[2])
    _, sZ = oracle.kda_recurrence(q, k, v, g, beta, cu, None, 0.3)
    assert np.all(sZ[0] == 0) and np.all(sZ[2] == 0)


def test_result_independent_of_thread_count():
    rng = np.random.default_rng(11)
    q, k, v, g, beta, cu, s0 = rand_case(rng, [17, 40, 3], 3, 8, 8)
    o1, s1 = oracle.kda_recurrence(q, k, v, g, beta, cu, s0, 0.3, num_threads=1)
    o4, s4, used = oracle.kda_recurrence(q, k, v, g, beta, cu, s0, 0.3, num_threads=4, return_threads=True)
    assert used == 4
    assert np.array_equal(o1, o4) and np.array_equal(s1, s4)


# ------------------------------------------- brute force: chunked algebra (§4, §6)

@pytest.mark.parametrize("solver", ["blocked", "neumann", "solve"])
def test_chunked_algebra_matches_token_recurrence(solver):
    """The page's chunked method (cumsum, midpoint strips, (I+L) solve, WY
    form, entry-state recurrence) and the token recurrence are two
    derivations of one result: they must agree to fp64 rounding. Lengths
    follow the report's unaligned varlen case [130, 64, 210], plus an empty
    and a sub-block-short sequence."""
    rng = np.random.default_rng(12)
    lens = [130, 64, 0, 5, 210]
    q, k, v, g, beta, cu, s0 = rand_case(rng, lens, 2, 16, 12)
    o_ref, s_ref = oracle.kda_recurrence(q, k, v, g, beta, cu, s0, 0.25)
    o, sT = chunked.kda_chunked(q, k, v, g, beta, cu, s0, 0.25, solver=solver)
    err_o = np.max(np.abs(o - o_ref)) / np.max(np.abs(o_ref))
    err_s = np.max(np.abs(sT - s_ref)) / np.max(np.abs(s_ref))
    assert err_o < 1e-11 and err_s < 1e-11, (err_o, err_s)


def test_strip_products_equal_direct_decay_tensor():
    rng = np.random.default_rng(13)
    for n in (64, 50, 16, 7):
        a, b = rng.standard_normal((n, 12)), rng.standard_normal((n, 12))
        G = chunked.gate_cumsum(-5.0 * rng.random((n, 12)))
        for strict in (False, True):
            A1 = chunked.decay_scores_direct(a, b, G, strict)
            A2, _ = chunked.decay_scores_strips(a, b, G, strict)
            np.testing.assert_allclose(A2, A1, rtol=1e-12, atol=1e-13)


def test_neumann_chain_and_blocked_substitution_equal_inverse():
    rng = np.random.default_rng(14)
    for n in (64, 48, 33, 16, 3):
        L = np.tril(rng.standard_normal((n, n)) * 0.3, -1)
        R = rng.standard_normal((n, 20))
        ref = np.linalg.solve(np.eye(n) + L, R)
        np.testing.assert_allclose(chunked.neumann_apply(L, R), ref, rtol=1e-10, atol=1e-11)
        np.testing.assert_allclose(chunked.blocked_solve(L, R), ref, rtol=1e-10, atol=1e-11)


# ------------------------------------------ the pins reject plausible mistakes

def _mutant_recurrence(q, k, v, g, beta, scale, kind):
    """A deliberately wrong recurrence, one mistake per kind, used only to show
    that the closed-form pins above reject it."""
    T, K = q.shape
    V = v.shape[1]
    S = np.zeros((K, V))
    o = np.zeros((T, V))
    for t in range(T):
        D = np.exp(-g[t] if kind == "sign" else g[t])[:, None]
        if kind == "decay_after_erase":
            S = S - beta[t] * np.outer(k[t], k[t] @ S)
            S = D * S + beta[t] * np.outer(k[t], v[t])
        elif kind == "no_decay":
            S = S + beta[t] * np.outer(k[t], v[t] - k[t] @ S)
        else:
            S = D * S
            prev = S.copy()
            S = S + beta[t] * np.outer(k[t], v[t] - k[t] @ S)
        if kind == "output_before_update":
            o[t] = scale * prev.T @ q[t]
        elif kind == "transposed_read":
            o[t] = scale * S @ q[t]
        else:
            o[t] = scale * S.T @ q[t]
    return o


@pytest.mark.parametrize("kind", ["decay_after_erase", "no_decay", "sign",
                                  "output_before_update", "transposed_read"])
def test_pins_reject_planted_mistakes(kind):
    rng = np.random.default_rng(15)
    T, K = 20, 8
    k = rng.standard_normal((T, K))
    k /= np.linalg.norm(k, axis=1, keepdims=True)
    v = rng.standard_normal((T, K))
    g = -2.0 * rng.random((T, K))
    beta = np.ones(T)
    o = _mutant_recurrence(k, k, v, g, beta, 1.0, kind)      # beta=1, q=k pin
    bad1 = not np.allclose(o, v, atol=1e-9)
    # basis-key pin with per-channel decay, checked against its closed form
    Tb = 6
    ch = rng.permutation(K)[:Tb]
    kb = np.eye(K)[ch]
    qb = rng.standard_normal((Tb, K))
    vb = rng.standard_normal((Tb, K))
    gb = -2.0 * rng.random((Tb, K))
    bb = rng.random(Tb)
    ob = _mutant_recurrence(qb, kb, vb, gb, bb, 1.0, kind)
    ref, _ = basis_key_closed_form(qb, ch, vb, gb, bb, 1.0)
    bad2 = not np.allclose(ob, ref, atol=1e-9)
    assert bad1 or bad2


# ---- gate and beta activations (the raw-gate entry point; a stated reading)
def test_gate_activation_closed_forms():
    """The restated activation against closed forms of the logistic function:
    sigma(0) = 1/2, sigma(ln 3) = 3/4, sigma(x) + sigma(-x) = 1, the limits, and
    the per-head scale e^A_log and per-channel shift dt_bias entering as
    e^A_log * (x + dt_bias)."""
    from oracle import gates
    lb = -5.0
    x = np.zeros((2, 3, 4))
    assert np.allclose(gates.activate_gate(x, lb), lb / 2, rtol=0, atol=0)
    assert abs(gates.sigmoid(math.log(3.0)) - 0.75) < 1e-15
    r = np.random.default_rng(0).normal(size=(5, 2, 4)) * 4
    assert np.allclose(gates.activate_gate(r, lb) + gates.activate_gate(-r, lb), lb, atol=1e-13)
    big = np.full((1, 1, 2), 800.0)
    assert np.all(gates.activate_gate(big, lb) == lb) and np.all(gates.activate_gate(-big, lb) == 0.0)
    g = gates.activate_gate(r, lb)
    assert np.all((g >= lb) & (g <= 0))
    # e^A_log = 2 doubles the argument; dt_bias = -x brings it back to sigma(0)
    A = np.array([math.log(2.0), 0.0])
    dt = np.zeros((2, 4))
    g2 = gates.activate_gate(r, lb, A_log=A, dt_bias=dt)
    assert np.allclose(g2[:, 0], lb * (1 / (1 + np.exp(-2 * r[:, 0]))), atol=1e-13)
    assert np.allclose(g2[:, 1], g[:, 1], atol=0)
    shift = gates.activate_gate(r, lb, dt_bias=-r[0])
    assert np.allclose(shift[0], lb / 2, atol=1e-15)


def test_beta_activation_closed_forms():
    from oracle import gates
    assert gates.activate_beta(np.zeros(3)).tolist() == [0.5, 0.5, 0.5]
    x = np.linspace(-30, 30, 61)
    b = gates.activate_beta(x)
    assert np.all((b > 0) & (b < 1)) and np.all(np.diff(b) > 0)
    assert np.allclose(b + gates.activate_beta(-x), 1.0, atol=1e-15)



def _gated_norm_pins(fn):
    """The gated-RMSNorm pins, worked by hand, as a list of the ones `fn`
    (o, gate, weight, eps) -> y fails (an exception counts as failing): the
    mean (not the sum) of squares over the value channels of one (token, head)
    row, eps inside the square root, the weight on the channel axis, and a
    sigmoid (not a swish) gate."""
    big = lambda shape: np.full(shape, 800.0)  # sigmoid(800) == 1 in fp64
    r = np.random.default_rng(1).normal(size=(4, 3, 8)) * np.array([1e-3, 1.0, 50.0])[None, :, None]
    o = np.random.default_rng(2).normal(size=(2, 3, 3))
    w = np.array([1.0, 2.0, -3.0])

    def unit(eps=0.0):
        return fn(r, big(r.shape), np.ones(8), eps)

    def eps_case():
        y = fn(np.array([[[1e-3, 1e-3], [0.0, 0.0]]]), big((1, 2, 2)), np.ones(2), 1e-6)
        return np.allclose(y[0, 0], 1e-3 / math.sqrt(2e-6), rtol=1e-14) and np.all(y[0, 1] == 0.0)

    pins = {
        "worked example [3, 4]": lambda: np.allclose(fn(np.array([[[3.0, 4.0]]]), big((1, 1, 2)), np.ones(2), 0.0),
                                                     [[[3 / math.sqrt(12.5), 4 / math.sqrt(12.5)]]], rtol=1e-15, atol=0),
        # every row normalised on its own: unit RMS whatever the row's scale
        "unit RMS per row": lambda: np.allclose(np.sqrt(np.mean(unit() ** 2, axis=-1)), 1.0, atol=1e-14),
        "scale invariance": lambda: np.allclose(fn(7.5 * r, big(r.shape), np.ones(8), 0.0), unit(), atol=1e-14),
        # gate 0 halves the output, gate ln 3 keeps three quarters
        "sigmoid gate": lambda: (np.allclose(fn(r, np.zeros(r.shape), np.ones(8), 0.0), 0.5 * unit(), atol=1e-15)
                                 and np.allclose(fn(r, np.full(r.shape, math.log(3.0)), np.ones(8), 0.0),
                                                 0.75 * unit(), atol=1e-14)),
        # the weight scales value channel c (V == H here, so a head-axis weight still broadcasts)
        "weight on channels": lambda: np.allclose(fn(o, big(o.shape), w, 1e-6),
                                                  fn(o, big(o.shape), np.ones(3), 1e-6) * w[None, None, :], atol=1e-15),
        # eps inside the root: [1e-3, 1e-3] with eps 1e-6 gives 1e-3 / sqrt(2e-6); an all-zero row stays 0
        "eps inside the root": eps_case,
    }
    bad = []
    for name, check in pins.items():
        try:
            good = bool(check())
        except (ValueError, IndexError):
            good = False
        if not good:
            bad.append(name)
    return bad


def test_gated_rmsnorm_closed_forms():
    from oracle import norm
    assert _gated_norm_pins(norm.gated_rmsnorm) == []


def _mutant_norm(kind):
    """A deliberately wrong gated RMSNorm, one mistake per kind, used only to
    show that the pins above reject it."""
    from oracle import gates

    def fn(o, gate, weight, eps):
        o, gate, weight = (np.asarray(x, dtype=np.float64) for x in (o, gate, weight))
        axis = 1 if kind == "norm_over_heads" else -1
        ms = np.sum(o * o, axis=-1, keepdims=True) if kind == "sum" else np.mean(o * o, axis=axis, keepdims=True)
        n = o / (np.sqrt(ms) + eps) if kind == "eps_outside" else o / np.sqrt(ms + eps)
        gg = gate * gates.sigmoid(gate) if kind == "swish" else gates.sigmoid(gate)
        ww = weight[None, :, None] if kind == "weight_on_heads" else weight
        return n * ww * gg
    return fn


@pytest.mark.parametrize("kind", ["sum", "eps_outside", "swish", "weight_on_heads", "norm_over_heads"])
def test_norm_pins_reject_planted_mistakes(kind):
    assert _gated_norm_pins(_mutant_norm(kind)) != []

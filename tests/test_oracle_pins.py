"""Pins of the fp64 oracle to facts other than itself.

Each test checks the oracle against something the pages or the mathematics fix:
closed forms, exact rational brute force of the matrix recurrence, invariants
of the recurrence, and the chunkwise-parallel form.  Together they are chosen so
that a dropped term, a wrong sign, an off-by-one in the gate or a transposed
operand in the oracle fails at least one of them.

The recurrence: "Qwen3.5-9B: Giai ma kien truc Gated DeltaNet", section
"Gated DeltaNet" (S_t = alpha_t (I - beta_t k_t k_t^T) S_{t-1} + beta_t k_t v_t^T),
and the per-token Loop of the Qwen3.5-9B NPU model card, section "How it works"
(decay, recall S^T k, delta correction, read-out S^T q from the updated state).
"""

from fractions import Fraction

import numpy as np
import pytest

import oracle
from tests.chunk_form import (chunk_form_factored, chunk_form_lookahead, chunk_form_pages, commit_from_deltas,
                               verify_deltas)


def _rng(seed):
    return np.random.default_rng(seed)


def _unit(x):
    return x / np.linalg.norm(x, axis=-1, keepdims=True)


def _single(q, k, v, g, beta, S0, threads=1):
    """Oracle on one sequence with one QK head and one V head."""
    T = q.shape[0]
    o, S = oracle.gdr_sequential(
        [0, T], q[:, None, :], k[:, None, :], v[:, None, :], g[:, None], beta[:, None],
        S0[None, None], threads=threads,
    )
    return o[:, 0, :], S[0, 0]


def _rand_case(seed, T=12, dk=6, dv=5, unit_keys=True):
    r = _rng(seed)
    q = _unit(r.standard_normal((T, dk)))
    k = r.standard_normal((T, dk))
    k = _unit(k) if unit_keys else k
    v = r.standard_normal((T, dv))
    g = r.uniform(-2.0, -0.01, T)
    beta = 1.0 / (1.0 + np.exp(-r.standard_normal(T)))
    S0 = 0.3 * r.standard_normal((dk, dv))
    return q, k, v, g, beta, S0


# --- closed forms --------------------------------------------------------------


def test_beta_zero_is_pure_geometric_decay():
    """beta = 0 writes nothing: S_t = exp(G_t) S0 and o_t = exp(G_t) S0^T q_t."""
    q, k, v, g, beta, S0 = _rand_case(1, T=20)
    beta[:] = 0.0
    o, S = _single(q, k, v, g, beta, S0)
    G = np.cumsum(g)
    np.testing.assert_allclose(S, np.exp(G[-1]) * S0, rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(o, np.exp(G)[:, None] * (q @ S0), rtol=1e-12, atol=1e-15)


def test_alpha_one_beta_zero_freezes_state():
    """alpha = 1 (g = 0) and beta = 0: S_t = S0 and o_t = S0^T q_t for every t."""
    q, k, v, g, beta, S0 = _rand_case(2)
    g[:] = 0.0
    beta[:] = 0.0
    o, S = _single(q, k, v, g, beta, S0)
    np.testing.assert_array_equal(S, S0)
    np.testing.assert_allclose(o, q @ S0, rtol=1e-13, atol=1e-15)


def test_orthogonal_keys_give_cumulative_linear_attention():
    """alpha = 1, S0 = 0 and mutually orthogonal keys: nothing is recalled, so
    S_t = sum_{j<=t} beta_j k_j v_j^T and o_t = sum_{j<=t} beta_j (q_t . k_j) v_j."""
    r = _rng(3)
    dk, dv, T = 16, 7, 12
    basis, _ = np.linalg.qr(r.standard_normal((dk, dk)))
    k = basis[:, :T].T * r.uniform(0.5, 2.0, (T, 1))  # orthogonal, not unit
    q = r.standard_normal((T, dk))
    v = r.standard_normal((T, dv))
    g = np.zeros(T)
    beta = r.uniform(0.1, 0.9, T)
    o, S = _single(q, k, v, g, beta, np.zeros((dk, dv)))
    S_ref = sum(beta[j] * np.outer(k[j], v[j]) for j in range(T))
    np.testing.assert_allclose(S, S_ref, rtol=1e-12, atol=1e-13)
    o_ref = np.array([sum(beta[j] * (q[t] @ k[j]) * v[j] for j in range(t + 1)) for t in range(T)])
    np.testing.assert_allclose(o, o_ref, rtol=1e-12, atol=1e-13)


def test_orthonormal_keys_beta_one_overwrite_slots():
    """alpha = 1, beta = 1, orthonormal keys: writing (k_i, v) sets k_i^T S = v^T
    exactly, re-writing overwrites, and directions orthogonal to every written key
    keep what S0 held."""
    r = _rng(4)
    dk, dv = 8, 5
    basis, _ = np.linalg.qr(r.standard_normal((dk, dk)))
    keys = basis.T  # rows orthonormal
    seq = [0, 1, 0, 2, 1]
    k = keys[seq]
    v = r.standard_normal((len(seq), dv))
    q = r.standard_normal((len(seq), dk))
    S0 = r.standard_normal((dk, dv))
    o, S = _single(q, k, v, np.zeros(len(seq)), np.ones(len(seq)), S0)
    np.testing.assert_allclose(keys[0] @ S, v[2], atol=1e-13)
    np.testing.assert_allclose(keys[1] @ S, v[4], atol=1e-13)
    np.testing.assert_allclose(keys[2] @ S, v[3], atol=1e-13)
    for i in range(3, dk):
        np.testing.assert_allclose(keys[i] @ S, keys[i] @ S0, atol=1e-13)


def test_scalar_case_by_hand():
    """d_k = d_v = 1: s_t = alpha_t (1 - beta_t k_t^2) s_{t-1} + beta_t k_t v_t, o_t = s_t q_t."""
    r = _rng(5)
    T = 30
    q, k, v = r.standard_normal((3, T))
    g = r.uniform(-1.5, 0.0, T)
    beta = r.uniform(0, 1, T)
    s = 0.7
    o_ref, s_ref = [], s
    for t in range(T):
        s_ref = np.exp(g[t]) * (1.0 - beta[t] * k[t] ** 2) * s_ref + beta[t] * k[t] * v[t]
        o_ref.append(s_ref * q[t])
    o, S = _single(q[:, None], k[:, None], v[:, None], g, beta, np.array([[s]]))
    np.testing.assert_allclose(o[:, 0], o_ref, rtol=1e-12)
    assert abs(S[0, 0] - s_ref) <= 1e-12 * max(1.0, abs(s_ref))


def _frac_matrix_product_reference(q, k, v, alpha, beta, S0):
    """Exact rational S_T and o_t from the matrix form M_t = alpha_t (I - beta_t k_t k_t^T):
    S_t = M_t S_{t-1} + beta_t k_t v_t^T, expanded as explicit products."""
    T, dk = len(k), len(k[0])
    dv = len(v[0])
    I = [[Fraction(int(i == j)) for j in range(dk)] for i in range(dk)]

    def matmul(A, B):
        return [[sum(A[i][m] * B[m][j] for m in range(len(B))) for j in range(len(B[0]))] for i in range(len(A))]

    def outer(a, b, s):
        return [[s * a[i] * b[j] for j in range(len(b))] for i in range(len(a))]

    M = []
    for t in range(T):
        kk = outer(k[t], k[t], beta[t])
        M.append([[alpha[t] * (I[i][j] - kk[i][j]) for j in range(dk)] for i in range(dk)])
    states = []
    for t in range(T):
        # S_t = (M_t ... M_1) S0 + sum_j (M_t ... M_{j+1}) beta_j k_j v_j^T
        prod = I
        for m in range(t, -1, -1):
            prod = matmul(prod, M[m])
        acc = matmul(prod, S0)
        for j in range(t + 1):
            P = I
            for m in range(t, j, -1):
                P = matmul(P, M[m])
            term = matmul(P, outer(k[j], v[j], beta[j]))
            acc = [[acc[i][c] + term[i][c] for c in range(dv)] for i in range(dk)]
        states.append(acc)
    outs = [[sum(states[t][i][c] * q[t][i] for i in range(dk)) for c in range(dv)] for t in range(T)]
    return outs, states[-1]


def test_exact_rational_brute_force_matrix_products():
    """Tiny case (d_k = 3, d_v = 2, T = 5) against exact rational arithmetic of the
    product form; alphas are exact rationals, passed to the oracle as log(alpha)."""
    r = _rng(6)
    T, dk, dv = 5, 3, 2

    def rat(x, den=8):
        return Fraction(int(round(x * den)), den)

    k = [[rat(x) for x in row] for row in r.uniform(-1, 1, (T, dk))]
    q = [[rat(x) for x in row] for row in r.uniform(-1, 1, (T, dk))]
    v = [[rat(x) for x in row] for row in r.uniform(-2, 2, (T, dv))]
    alpha = [Fraction(n, 16) for n in r.integers(4, 17, T)]
    beta = [Fraction(n, 8) for n in r.integers(0, 9, T)]
    S0 = [[rat(x) for x in row] for row in r.uniform(-1, 1, (dk, dv))]
    o_ref, S_ref = _frac_matrix_product_reference(q, k, v, alpha, beta, S0)

    f = lambda a: np.array(a, dtype=np.float64)
    o, S = _single(f(q), f(k), f(v), np.log(f(alpha)), f(beta), f(S0))
    np.testing.assert_allclose(o, f(o_ref), rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(S, f(S_ref), rtol=1e-13, atol=1e-14)


# --- invariants ----------------------------------------------------------------


def test_superposition_in_state_and_values():
    """For fixed K, g, beta the map (S0, V) -> (S_T, O) is linear."""
    q, k, v1, g, beta, S1 = _rand_case(7, T=25)
    _, _, v2, _, _, S2 = _rand_case(8, T=25)
    a, b = 0.7, -1.3
    o1, T1 = _single(q, k, v1, g, beta, S1)
    o2, T2 = _single(q, k, v2, g, beta, S2)
    o12, T12 = _single(q, k, a * v1 + b * v2, g, beta, a * S1 + b * S2)
    np.testing.assert_allclose(o12, a * o1 + b * o2, rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(T12, a * T1 + b * T2, rtol=1e-11, atol=1e-13)


def test_output_linear_in_query_state_independent_of_query():
    q, k, v, g, beta, S0 = _rand_case(9)
    o1, T1 = _single(q, k, v, g, beta, S0)
    o2, T2 = _single(-2.5 * q, k, v, g, beta, S0)
    np.testing.assert_array_equal(T1, T2)
    np.testing.assert_allclose(o2, -2.5 * o1, rtol=1e-13, atol=1e-15)


def test_scale_multiplies_output_only():
    q, k, v, g, beta, S0 = _rand_case(10)
    T = q.shape[0]
    args = ([0, T], q[:, None], k[:, None], v[:, None], g[:, None], beta[:, None], S0[None, None])
    o1, T1 = oracle.gdr_sequential(*args, scale=1.0)
    o2, T2 = oracle.gdr_sequential(*args, scale=0.125)
    np.testing.assert_array_equal(T1, T2)
    np.testing.assert_allclose(o2, 0.125 * o1, rtol=1e-14)


def test_padding_rows_are_a_no_op():
    """Rows with g = 0 and beta = 0 (the model card's token_valid padding) leave
    the state exactly as after the last real token."""
    q, k, v, g, beta, S0 = _rand_case(11, T=10)
    _, S_a = _single(q, k, v, g, beta, S0)
    r = _rng(12)
    pad = 6
    qp = np.vstack([q, _unit(r.standard_normal((pad, q.shape[1])))])
    kp = np.vstack([k, _unit(r.standard_normal((pad, k.shape[1])))])
    vp = np.vstack([v, r.standard_normal((pad, v.shape[1]))])
    o_b, S_b = _single(qp, kp, vp, np.r_[g, np.zeros(pad)], np.r_[beta, np.zeros(pad)], S0)
    np.testing.assert_array_equal(S_a, S_b)
    np.testing.assert_allclose(o_b[10:], qp[10:] @ S_a, rtol=1e-13, atol=1e-15)


def test_prefill_then_decode_handoff():
    """Running T1 tokens, then T2 more from the returned state, equals T1 + T2 at once."""
    q, k, v, g, beta, S0 = _rand_case(13, T=40)
    o_all, S_all = _single(q, k, v, g, beta, S0)
    o1, S1 = _single(q[:25], k[:25], v[:25], g[:25], beta[:25], S0)
    outs = [o1]
    S = S1
    for t in range(25, 40):  # one-token "decode" calls
        o_t, S = _single(q[t:t + 1], k[t:t + 1], v[t:t + 1], g[t:t + 1], beta[t:t + 1], S)
        outs.append(o_t)
    np.testing.assert_array_equal(np.vstack(outs), o_all)
    np.testing.assert_array_equal(S, S_all)


def test_varlen_packing_equals_separate_sequences_and_threads_agree():
    r = _rng(14)
    lens = [5, 0, 17, 1, 9]
    T = sum(lens)
    cu = np.r_[0, np.cumsum(lens)]
    hqk, hv, dk, dv = 2, 4, 6, 5
    q = _unit(r.standard_normal((T, hqk, dk)))
    k = _unit(r.standard_normal((T, hqk, dk)))
    v = r.standard_normal((T, hv, dv))
    g = r.uniform(-3, -0.01, (T, hv))
    beta = r.uniform(0, 1, (T, hv))
    S0 = r.standard_normal((len(lens), hv, dk, dv))
    o, S = oracle.gdr_sequential(cu, q, k, v, g, beta, S0, threads=1)
    o8, S8 = oracle.gdr_sequential(cu, q, k, v, g, beta, S0, threads=8)
    np.testing.assert_array_equal(o, o8)
    np.testing.assert_array_equal(S, S8)
    for s, L in enumerate(lens):
        a, b = cu[s], cu[s + 1]
        os_, Ss = oracle.gdr_sequential([0, L], q[a:b], k[a:b], v[a:b], g[a:b], beta[a:b], S0[s:s + 1])
        np.testing.assert_array_equal(o[a:b], os_)
        np.testing.assert_array_equal(S[s], Ss[0])


def test_qk_head_shared_by_contiguous_pair_of_v_heads():
    """V heads 2i and 2i+1 read QK head i: identical v/g/beta on a pair gives
    identical outputs, and changing QK head i changes only V heads 2i, 2i+1."""
    r = _rng(15)
    T, hqk, hv, dk, dv = 9, 3, 6, 5, 4
    q = _unit(r.standard_normal((T, hqk, dk)))
    k = _unit(r.standard_normal((T, hqk, dk)))
    v = r.standard_normal((T, hv, dv))
    g = r.uniform(-2, -0.01, (T, hv))
    beta = r.uniform(0, 1, (T, hv))
    for i in range(hqk):
        v[:, 2 * i + 1], g[:, 2 * i + 1], beta[:, 2 * i + 1] = v[:, 2 * i], g[:, 2 * i], beta[:, 2 * i]
    S0 = np.zeros((1, hv, dk, dv))
    o, S = oracle.gdr_sequential([0, T], q, k, v, g, beta, S0)
    for i in range(hqk):
        np.testing.assert_array_equal(o[:, 2 * i], o[:, 2 * i + 1])
    k2 = k.copy()
    k2[:, 1] = _unit(r.standard_normal((T, dk)))
    o2, _ = oracle.gdr_sequential([0, T], q, k2, v, g, beta, S0)
    changed = [h for h in range(hv) if not np.array_equal(o[:, h], o2[:, h])]
    assert changed == [2, 3]


def test_contraction_bound_per_step():
    """Unit keys, beta in [0, 1], alpha <= 1: (I - beta k k^T) has spectral norm <= 1,
    so ||S_t||_2 <= alpha_t ||S_{t-1}||_2 + beta_t ||v_t||."""
    q, k, v, g, beta, S = _rand_case(16, T=30, dk=8, dv=6)
    for t in range(30):
        _, S_next = _single(q[t:t + 1], k[t:t + 1], v[t:t + 1], g[t:t + 1], beta[t:t + 1], S)
        lhs = np.linalg.norm(S_next, 2)
        rhs = np.exp(g[t]) * np.linalg.norm(S, 2) + beta[t] * np.linalg.norm(v[t])
        assert lhs <= rhs * (1 + 1e-12)
        S = S_next


# --- the chunkwise-parallel form -------------------------------------------------


@pytest.mark.parametrize("C", [16, 64])
@pytest.mark.parametrize("T", [1, 15, 16, 17, 63, 64, 65, 128, 200])
def test_chunk_forms_match_sequential(C, T):
    """The model card's chunk form, and the kernels' regroupings of it (the factored
    form, and the chunk scan's lookahead), equal the sequential recurrence for every
    length around the chunk boundary."""
    r = _rng(100 + T + C)
    dk = dv = 32
    q = _unit(r.standard_normal((T, dk)))
    k = _unit(r.standard_normal((T, dk)))
    v = r.standard_normal((T, dv))
    g = r.uniform(-8.0, -0.01, T)
    beta = 1.0 / (1.0 + np.exp(-r.standard_normal(T)))
    S0 = 0.02 * r.standard_normal((dk, dv))
    o, S = _single(q, k, v, g, beta, S0)
    for form in (chunk_form_pages, chunk_form_factored, chunk_form_lookahead):
        oc, Sc = form(q, k, v, g, beta, S0, C)
        scale_o = np.sqrt(np.mean(o * o))
        assert np.max(np.abs(oc - o)) <= 1e-10 * max(scale_o, 1e-30), form.__name__
        assert np.linalg.norm(Sc - S) <= 1e-10 * np.linalg.norm(S), form.__name__


def test_chunk_form_strong_decay_stays_finite():
    """log alpha = -6.72 for every token (the Candle PR's overflow regression): with
    the log-space mask the chunk form is finite and equals the sequential result."""
    r = _rng(17)
    T, dk, dv, C = 130, 16, 8, 64
    q = _unit(r.standard_normal((T, dk)))
    k = _unit(r.standard_normal((T, dk)))
    v = r.standard_normal((T, dv))
    g = np.full(T, -6.72)
    beta = 1.0 / (1.0 + np.exp(-r.standard_normal(T)))
    S0 = 0.02 * r.standard_normal((dk, dv))
    o, S = _single(q, k, v, g, beta, S0)
    for form in (chunk_form_factored, chunk_form_lookahead):
        oc, Sc = form(q, k, v, g, beta, S0, C)
        assert np.all(np.isfinite(oc)) and np.all(np.isfinite(Sc)), form.__name__
        assert np.max(np.abs(oc - o)) <= 1e-10 * np.sqrt(np.mean(o * o)), form.__name__
        assert np.linalg.norm(Sc - S) <= 1e-10 * np.linalg.norm(S), form.__name__
    # With the same decay, the unmasked factorisation exp(G_t) * exp(-G_j)
    # overflows fp32 within a chunk: exp(-G_j) passes FLT_MAX at j = 14.
    with np.errstate(over="ignore"):
        G = np.cumsum(g[:C]).astype(np.float32)
        inv = np.exp(-G)
    assert np.isfinite(inv[12]) and not np.isfinite(inv[13])


# --- verify commit from cached corrections ------------------------------------------


@pytest.mark.parametrize("n_tok", [1, 7, 16])
def test_verify_commit_from_deltas_equals_sequential_prefix(n_tok):
    """A verify block's corrections u_t are the recurrence's own u_t = beta_t (v_t -
    e^{g_t} S_{t-1}^T k_t), and the state formed from them for any accepted prefix a
    (the formula gdr_verify_commit evaluates) equals the sequential state after those
    a tokens."""
    q, k, v, g, beta, S0 = _rand_case(200 + n_tok, T=n_tok, dk=8, dv=6)
    D = verify_deltas(k, v, g, beta, S0)
    S = S0.copy()
    for t in range(n_tok):
        u = beta[t] * (v[t] - np.exp(g[t]) * (S.T @ k[t]))
        assert np.allclose(D[t], u, rtol=0, atol=1e-12 * max(1.0, np.abs(u).max()))
        _, S = _single(q[t:t + 1], k[t:t + 1], v[t:t + 1], g[t:t + 1], beta[t:t + 1], S)
    for a in range(n_tok + 1):
        S_ref = S0 if a == 0 else _single(q[:a], k[:a], v[:a], g[:a], beta[:a], S0)[1]
        S_c = commit_from_deltas(k, g, D, S0, a)
        assert np.linalg.norm(S_c - S_ref) <= 1e-12 * np.linalg.norm(S_ref)


@pytest.mark.parametrize("g_fixed", [None, -6.72])
def test_kernel_operand_rounding_stays_inside_the_tolerances(g_fixed):
    """The tensor-core scan's operand roundings (fp16 Tw, PTw, X, R and D~ in
    MMA2 and MMA_X; bf16 hi/lo S' and D~ in MMA1' and MMA3), applied to the
    lookahead grouping with exact fp64 products, against the sequential oracle on
    one Qwen3.5-9B-sized head (d = 128, 16 chunks of 64, bf16 q/k/v values, state
    ~ N(0, 0.02)): the error budget of that design is inside the stated
    tolerances (2e-2 max-abs / RMS, 1e-3 relative Frobenius) with a margin of
    two, and a single bf16 term in place of fp16 is markedly worse.  (The
    kernel's fp32 accumulation is not modelled.)"""
    from tests.chunk_form import round_bf16
    r = _rng(29)
    T, d, C = 1024, 128, 64
    q = round_bf16(_unit(r.standard_normal((T, d))))
    k = round_bf16(_unit(r.standard_normal((T, d))))
    v = round_bf16(r.standard_normal((T, d)))
    g = np.full(T, g_fixed) if g_fixed is not None else r.uniform(-8.0, -0.01, T)
    beta = 1.0 / (1.0 + np.exp(-r.standard_normal(T)))
    S0 = 0.02 * r.standard_normal((d, d))
    o, S = _single(q, k, v, g, beta, S0)
    rms = np.sqrt(np.mean(o * o))
    err = {}
    for name in ("kernel", "bf16_single"):
        oc, Sc = chunk_form_lookahead(q, k, v, g, beta, S0, C, operands=name)
        err[name] = (np.max(np.abs(oc - o)) / rms, np.linalg.norm(Sc - S) / np.linalg.norm(S))
    eo, es = err["kernel"]
    assert eo <= 1e-2 and es <= 5e-4, err
    # fp16 keeps 3 more significand bits; under strong decay part of the fp16
    # error is the underflow of the most decayed Tw rows, which bf16 keeps
    assert err["bf16_single"][0] >= 4 * eo and err["bf16_single"][1] >= 2 * es, err


# --- two-level (segment-parallel) scan -----------------------------------------------


def _gates(r, T, regime):
    if regime == "slow":  # the start state's influence survives a whole segment
        return r.uniform(-0.05, -0.001, T)
    if regime == "fixed":
        return np.full(T, -6.72)
    return r.uniform(-8.0, -0.01, T)


@pytest.mark.parametrize("T,P,regime", [(128, 2, "slow"), (1000, 3, "slow"), (1000, 4, "uniform"),
                                        (4096, 4, "slow"), (4096, 2, "fixed"), (200, 3, "slow")])
def test_segment_composition_equals_sequential(T, P, regime):
    """Segments composed through their affine transitions (start state I with
    zero values for the transition and the output maps, start state 0 for the
    offsets, a sequential combine, then the per-token fix-up) reproduce the
    sequential recurrence, for segment cuts at chunk boundaries with a ragged
    last chunk.  With slow decay the transitions carry the start state across
    whole segments (checked), so the combine and the fix-up are exercised; under
    the strong -6.72 decay they vanish and the segments decouple."""
    from tests.chunk_form import segment_compose

    r = _rng(400 + T + P)
    dk = dv = 32 if T > 1000 else 16
    q = _unit(r.standard_normal((T, dk)))
    k = _unit(r.standard_normal((T, dk)))
    v = r.standard_normal((T, dv))
    g = _gates(r, T, regime)
    beta = 1.0 / (1.0 + np.exp(-r.standard_normal(T)))
    S0 = 0.02 * r.standard_normal((dk, dv))
    o, S = _single(q, k, v, g, beta, S0)
    oc, Sc = segment_compose(q, k, v, g, beta, S0, 64, P)
    assert np.max(np.abs(oc - o)) <= 1e-10 * np.sqrt(np.mean(o * o))
    assert np.linalg.norm(Sc - S) <= 1e-10 * np.linalg.norm(S)
    if regime == "slow":
        bad, _ = segment_compose(q, k, v, g, beta, S0, 64, P, mutate="no_fixup")
        assert np.max(np.abs(bad - o)) > 1e-3 * np.sqrt(np.mean(o * o))


def test_segment_composition_is_pinned_by_the_oracle_too():
    """The same composition with every segment run by the oracle itself (the
    sequential recurrence from X = I with zero values gives the transition and the
    output maps): its arithmetic alone, independent of any chunk form."""
    from tests.chunk_form import segment_compose

    r = _rng(471)
    T, dk, dv, P = 333, 8, 8, 3
    q = _unit(r.standard_normal((T, dk)))
    k = _unit(r.standard_normal((T, dk)))
    v = r.standard_normal((T, dv))
    g = _gates(r, T, "slow")
    beta = 1.0 / (1.0 + np.exp(-r.standard_normal(T)))
    S0 = 0.02 * r.standard_normal((dk, dv))
    o, S = _single(q, k, v, g, beta, S0)
    oc, Sc = segment_compose(q, k, v, g, beta, S0, 64, P, run=lambda *a: _single(*a))
    assert np.max(np.abs(oc - o)) <= 1e-11 * np.sqrt(np.mean(o * o))
    assert np.linalg.norm(Sc - S) <= 1e-11 * np.linalg.norm(S)
    # plausible mistakes: combining with the transposed transition, dropping the fix-up
    bad_t = segment_compose(q, k, v, g, beta, S0, 64, P, run=lambda *a: _single(*a), mutate="transpose")
    assert np.linalg.norm(bad_t[1] - S) > 1e-6 * np.linalg.norm(S)
    bad_f = segment_compose(q, k, v, g, beta, S0, 64, P, run=lambda *a: _single(*a), mutate="no_fixup")
    assert np.max(np.abs(bad_f[0] - o)) > 1e-6 * np.sqrt(np.mean(o * o))


# --- steps on either side of the rule (q/k L2 norm, beta from logits, gated RMSNorm) ---


def test_l2norm_rows_closed_forms():
    """(3, 4) -> (3, 4) / sqrt(25 + 1e-6); a zero row stays zero; every row of
    random input comes out with unit norm up to the epsilon; positive scaling of a
    row does not change it (up to the epsilon)."""
    y = oracle.l2norm_rows(np.array([[3.0, 4.0], [0.0, 0.0]]))
    assert np.allclose(y[0], np.array([3.0, 4.0]) / np.sqrt(25.0 + 1e-6), rtol=0, atol=1e-15)
    assert np.all(y[1] == 0.0)
    r = _rng(501)
    x = r.standard_normal((40, 128)) * r.uniform(0.1, 10.0, (40, 1))
    y = oracle.l2norm_rows(x)
    n2 = np.sum(x * x, axis=1)
    assert np.allclose(np.linalg.norm(y, axis=1), np.sqrt(n2 / (n2 + 1e-6)), rtol=1e-14)
    assert np.allclose(oracle.l2norm_rows(7.5 * x), y, rtol=1e-7, atol=0)
    assert np.allclose(oracle.l2norm_rows(x, eps=0.0), x / np.sqrt(n2)[:, None], rtol=1e-14)


def test_sigmoid_closed_forms():
    b = np.array([0.0, np.log(3.0), -np.log(3.0), 30.0, -30.0])
    s = oracle.sigmoid(b)
    assert s[0] == 0.5 and abs(s[1] - 0.75) < 1e-15 and abs(s[2] - 0.25) < 1e-15
    r = _rng(502).standard_normal(100)
    assert np.allclose(oracle.sigmoid(r) + oracle.sigmoid(-r), 1.0, rtol=0, atol=1e-15)


def test_gated_rmsnorm_by_hand_and_invariants():
    """Row (1, -1, 1, -1) has mean square 1: y_j = w_j o_j silu(z_j) / sqrt(1 + eps),
    with silu(z) = z / (1 + e^-z) written out here for z = 0, 1, 2, -3.  The norm is
    invariant to scaling o (up to the epsilon), linear in the weights, zero where
    z = 0, and silu(z) - silu(-z) = z."""
    o = np.array([[1.0, -1.0, 1.0, -1.0]])
    z = np.array([[0.0, 1.0, 2.0, -3.0]])
    w = np.array([1.0, 2.0, 3.0, 4.0])
    silu = np.array([0.0, 1.0 / (1.0 + np.exp(-1.0)), 2.0 / (1.0 + np.exp(-2.0)), -3.0 / (1.0 + np.exp(3.0))])
    want = w * o[0] * silu / np.sqrt(1.0 + 1e-6)
    assert np.allclose(oracle.gated_rmsnorm(o, z, w)[0], want, rtol=1e-15, atol=0)
    r = _rng(503)
    o = r.standard_normal((20, 128))
    z = r.standard_normal((20, 128))
    w = r.uniform(0.5, 1.5, 128)
    y = oracle.gated_rmsnorm(o, z, w)
    assert np.allclose(oracle.gated_rmsnorm(4.0 * o, z, w), y, rtol=1e-6)
    assert np.allclose(oracle.gated_rmsnorm(o, z, 2.0 * w), 2.0 * y, rtol=1e-15)
    assert np.all(oracle.gated_rmsnorm(o, np.zeros_like(z), w) == 0.0)
    ones = np.ones(128)
    unit = o / np.sqrt(np.mean(o * o, axis=1, keepdims=True) + 1e-6)
    assert np.allclose(oracle.gated_rmsnorm(o, z, ones) - oracle.gated_rmsnorm(o, -z, ones), unit * z, rtol=1e-12)
    # the epsilon sits inside the square root: a row of tiny values is scaled by ~1/sqrt(eps)
    tiny = np.full((1, 128), 1e-5)
    assert np.allclose(oracle.gated_rmsnorm(tiny, np.full((1, 128), 50.0), ones),
                       1e-5 * 50.0 / np.sqrt(1e-10 + 1e-6), rtol=1e-12)


def test_fused_steps_compose_around_the_rule():
    """Normalising raw q and k and forming beta from logits before the rule, then
    the gated norm after it, equals doing those steps by hand around the plain
    oracle; the normalisation makes the rule invariant to q and k scaling."""
    r = _rng(504)
    T, dk, dv = 30, 16, 16
    q = r.standard_normal((T, 1, dk)) * 3.0
    k = r.standard_normal((T, 1, dk)) * 0.2
    v = r.standard_normal((T, 1, dv))
    g = r.uniform(-2.0, -0.01, (T, 1))
    b = r.standard_normal((T, 1))
    S0 = 0.02 * r.standard_normal((1, 1, dk, dv))
    z = r.standard_normal((T, 1, dv))
    w = r.uniform(0.5, 1.5, dv)
    y, S = oracle.gdr_fused([0, T], q, k, v, g, b, S0, qk_l2norm=True, beta_logits=True, z=z, norm_weight=w)
    qn = q / np.sqrt(np.sum(q * q, -1, keepdims=True) + 1e-6)
    kn = k / np.sqrt(np.sum(k * k, -1, keepdims=True) + 1e-6)
    o2, S2 = oracle.gdr_sequential([0, T], qn, kn, v, g, 1 / (1 + np.exp(-b)), S0)
    y2 = w * o2 / np.sqrt(np.mean(o2 * o2, -1, keepdims=True) + 1e-6) * (z / (1 + np.exp(-z)))
    assert np.allclose(y, y2, rtol=1e-12, atol=1e-15) and np.allclose(S, S2, rtol=1e-12, atol=1e-15)
    y3, S3 = oracle.gdr_fused([0, T], 5.0 * q, 0.5 * k, v, g, b, S0, qk_l2norm=True, beta_logits=True, z=z,
                              norm_weight=w)
    # up to the epsilon's share of |k|^2 (~1e-5 here)
    assert np.linalg.norm(S3 - S) <= 1e-4 * np.linalg.norm(S)
    assert np.max(np.abs(y3 - y)) <= 1e-4 * np.sqrt(np.mean(y * y))

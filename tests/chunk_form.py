"""Test-only fp64 models of the chunkwise-parallel form (numpy).

These are NOT the oracle.  They restate, in plain numpy, the block form that
the CUDA kernels use, so the tests can check that algebra against the
sequential oracle on the CPU (to ~1e-12) before any kernel runs.

``chunk_form_pages`` follows the chunk form written out on the Qwen3.5-9B NPU
model card ("How it works": N, D, O and S_T in terms of G = cumsum(g) and the
incoming state S0), with the upper triangle of G_t - G_j masked to -inf in log
space before exp (the Candle pull request's "Float32 overflow fix").

``chunk_form_factored`` regroups the same products the way the tcgen05 prefill
kernel does: everything that does not depend on the state is folded into
    W  = T diag(beta e^G) K,   U  = T diag(beta) V,
    Q' = diag(e^G) Q - P W,    U' = P U,      with T = (I + N)^-1,
so that one chunk of the sequential pass is
    D = U - W S,   O = Q' S + U',   S <- e^{G_C} S + K^T diag(e^{G_C - G}) D.
T is formed by 16x16 diagonal-block forward substitution followed by blocked
off-diagonal solves, as in the kernel.

``chunk_form_lookahead`` is the grouping of the tcgen05 chunk scan: with
Tw = diag(e^{G_C - G}) T diag(beta) and PTw = P T diag(beta), a chunk is
    R = V - diag(e^G) K S,  D~ = Tw R,  O = diag(e^G) Q S + PTw R,
    S <- e^{G_C} S + K^T D~,
and the next chunk's [K S; Q S] is formed without the new S as
    [K; Q]_{c+1} (e^{G_C} S_c) + X_c D~_c,   X_c = [K; Q]_{c+1} K_c^T.
"""

from __future__ import annotations

import numpy as np


def _decay_matrix(G: np.ndarray, strict: bool) -> np.ndarray:
    """exp(G_t - G_j) on the lower triangle (strict or inclusive), 0 above.

    The exponent is masked in log space first, so large positive differences
    above the diagonal never reach exp."""
    C = G.shape[0]
    diff = G[:, None] - G[None, :]
    keep = np.tril(np.ones((C, C), dtype=bool), -1 if strict else 0)
    diff = np.where(keep, diff, -np.inf)
    return np.exp(diff)


def _pad(x: np.ndarray, C: int) -> np.ndarray:
    L = x.shape[0]
    if L == C:
        return x
    out = np.zeros((C,) + x.shape[1:], dtype=x.dtype)
    out[:L] = x
    return out


def chunk_form_pages(q, k, v, g, beta, S0, C):
    """One head, one sequence: q, k [T, d_k], v [T, d_v], g, beta [T], S0 [d_k, d_v]."""
    T = q.shape[0]
    S = np.array(S0, dtype=np.float64)
    O = np.zeros((T, v.shape[1]))
    for c0 in range(0, T, C):
        L = min(C, T - c0)
        Q, K, V = (_pad(np.asarray(x[c0:c0 + L], np.float64), C) for x in (q, k, v))
        gc = _pad(np.asarray(g[c0:c0 + L], np.float64), C)  # padding: g = 0
        bc = _pad(np.asarray(beta[c0:c0 + L], np.float64), C)  # padding: beta = 0
        G = np.cumsum(gc)
        eG = np.exp(G)
        N = bc[:, None] * _decay_matrix(G, strict=True) * (K @ K.T)
        D = np.linalg.solve(np.eye(C) + N, bc[:, None] * (V - eG[:, None] * (K @ S)))
        Oc = eG[:, None] * (Q @ S) + (_decay_matrix(G, strict=False) * (Q @ K.T)) @ D
        S = np.exp(G[-1]) * S + K.T @ (np.exp(G[-1] - G)[:, None] * D)
        O[c0:c0 + L] = Oc[:L]
    return O, S


def unit_lower_inverse_blocked(N: np.ndarray, b: int = 16) -> np.ndarray:
    """(I + N)^-1 for strictly lower N: forward substitution inside each b x b
    diagonal block, then blocked solves for the blocks below the diagonal:
        T_ii = (I + N_ii)^-1,   T_ij = -T_ii * sum_{j <= m < i} N_im T_mj."""
    C = N.shape[0]
    nb = C // b
    T = np.zeros_like(N)
    for i in range(nb):
        sl = slice(i * b, (i + 1) * b)
        Nii = N[sl, sl]
        Tii = np.eye(b)
        for r in range(b):  # row r of T_ii: e_r - sum_{m<r} N_rm T_m
            Tii[r] = np.eye(b)[r] - Nii[r, :r] @ Tii[:r]
        T[sl, sl] = Tii
    for i in range(nb):
        si = slice(i * b, (i + 1) * b)
        for j in range(i - 1, -1, -1):
            sj = slice(j * b, (j + 1) * b)
            acc = np.zeros((b, b))
            for m in range(j, i):
                sm = slice(m * b, (m + 1) * b)
                acc += N[si, sm] @ T[sm, sj]
            T[si, sj] = -T[si, si] @ acc
    return T


def chunk_form_factored(q, k, v, g, beta, S0, C):
    """Same contract as ``chunk_form_pages``, regrouped as the kernel computes it."""
    T_len = q.shape[0]
    S = np.array(S0, dtype=np.float64)
    O = np.zeros((T_len, v.shape[1]))
    for c0 in range(0, T_len, C):
        L = min(C, T_len - c0)
        Q, K, V = (_pad(np.asarray(x[c0:c0 + L], np.float64), C) for x in (q, k, v))
        gc = _pad(np.asarray(g[c0:c0 + L], np.float64), C)
        bc = _pad(np.asarray(beta[c0:c0 + L], np.float64), C)
        G = np.cumsum(gc)
        eG = np.exp(G)
        A_kk = K @ K.T
        A_qk = Q @ K.T
        N = bc[:, None] * _decay_matrix(G, strict=True) * A_kk
        P = _decay_matrix(G, strict=False) * A_qk
        Tm = unit_lower_inverse_blocked(N, 16 if C % 16 == 0 else C)
        W = Tm @ ((bc * eG)[:, None] * K)
        U = Tm @ (bc[:, None] * V)
        Qp = eG[:, None] * Q - P @ W
        Up = P @ U
        # sequential part
        D = U - W @ S
        Oc = Qp @ S + Up
        S = np.exp(G[-1]) * S + K.T @ (np.exp(G[-1] - G)[:, None] * D)
        O[c0:c0 + L] = Oc[:L]
    return O, S


def verify_deltas(k, v, g, beta, S0):
    """Corrections u_t of one verify block (all rows real, one chunk), the rows of
    D = (I + N)^-1 diag(beta) (V - diag(e^G) K S0) on the model card's chunk form."""
    K, V = np.asarray(k, np.float64), np.asarray(v, np.float64)
    G = np.cumsum(np.asarray(g, np.float64))
    b = np.asarray(beta, np.float64)
    n = K.shape[0]
    N = b[:, None] * _decay_matrix(G, strict=True) * (K @ K.T)
    return np.linalg.solve(np.eye(n) + N, b[:, None] * (V - np.exp(G)[:, None] * (K @ S0)))


def commit_from_deltas(k, g, D, S0, a):
    """State after the first a tokens of a block from its corrections:
    e^{G_a} S0 + sum_{j < a} e^{G_a - G_j} k_j u_j^T, G_a = G_{a-1} (0 for a = 0)."""
    S0 = np.asarray(S0, np.float64)
    if a == 0:
        return S0.copy()
    G = np.cumsum(np.asarray(g[:a], np.float64))
    w = np.exp(G[-1] - G)
    return np.exp(G[-1]) * S0 + np.asarray(k[:a], np.float64).T @ (w[:, None] * np.asarray(D[:a], np.float64))


def _f32(x):
    return np.asarray(x, np.float64).astype(np.float32)


def round_bf16(x):
    """fp64 -> fp32 -> bf16 (round to nearest even), back to fp64."""
    u = _f32(x).view(np.uint32).astype(np.uint64)
    r = ((u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000).astype(np.uint32)
    return r.view(np.float32).astype(np.float64)


def round_f16(x):
    """fp64 -> fp32 -> fp16 (round to nearest even, IEEE subnormals), back to fp64."""
    with np.errstate(over="ignore", under="ignore"):
        return _f32(x).astype(np.float16).astype(np.float64)


def hilo_bf16(x):
    """hi = the fp32 value with its low 16 bits dropped, lo = bf16(x - hi); returns hi + lo."""
    f = _f32(x)
    hi = (f.view(np.uint32) & np.uint32(0xFFFF0000)).view(np.float32).astype(np.float64)
    return hi + round_bf16(f.astype(np.float64) - hi)


# Operand roundings of the chunk scan's products: the operands the kernel
# rounds to fp16 (Tw, PTw, X, R and D~ for MMA_X) and the ones it splits into
# bf16 hi/lo (S' for MMA1', D~ for MMA3).  "bf16_single" puts a single bf16
# term where the kernel has fp16, for comparison.
OPERANDS = {
    "kernel": (round_f16, hilo_bf16),
    "bf16_single": (round_bf16, hilo_bf16),
}


def chunk_form_lookahead(q, k, v, g, beta, S0, C, operands=None):
    """Same contract as ``chunk_form_pages``, in the tcgen05 chunk scan's grouping.

    ``operands`` names an entry of OPERANDS to round the products' operands the
    way the kernel does (the products themselves stay in fp64); None keeps
    every operand exact."""
    rnd, split = OPERANDS[operands] if operands else ((lambda x: x), (lambda x: x))
    T_len = q.shape[0]
    n = (T_len + C - 1) // C
    chunks = []
    for c in range(n):
        c0 = c * C
        L = min(C, T_len - c0)
        Q, K, V = (_pad(np.asarray(x[c0:c0 + L], np.float64), C) for x in (q, k, v))
        gc = _pad(np.asarray(g[c0:c0 + L], np.float64), C)
        bc = _pad(np.asarray(beta[c0:c0 + L], np.float64), C)
        G = np.cumsum(gc)
        N = bc[:, None] * _decay_matrix(G, strict=True) * (K @ K.T)
        P = _decay_matrix(G, strict=False) * (Q @ K.T)
        Tm = unit_lower_inverse_blocked(N, 16 if C % 16 == 0 else C)
        Tw = np.exp(G[-1] - G)[:, None] * Tm * bc[None, :]
        PTw = P @ Tm * bc[None, :]
        chunks.append((c0, L, np.vstack([K, Q]), K, V, G, Tw, PTw))
    S = np.array(S0, dtype=np.float64)
    O = np.zeros((T_len, v.shape[1]))
    dk = q.shape[1]
    A = chunks[0][2] @ split(S)  # [K S; Q S] of chunk 0
    for c, (c0, L, KQ, K, V, G, Tw, PTw) in enumerate(chunks):
        KS, QS = A[:C], A[C:]
        eG = np.exp(G)[:, None]
        R = rnd(V - eG * KS)
        Dt = rnd(Tw) @ R
        O[c0:c0 + L] = (eG * QS + rnd(PTw) @ R)[:L]
        eGC = np.exp(G[-1])
        if c + 1 < n:
            KQn = chunks[c + 1][2]
            X = KQn @ K.T
            A = KQn @ split(eGC * S) + rnd(X) @ rnd(Dt)
        S = eGC * S + K.T @ split(Dt)
    assert S.shape == (dk, v.shape[1])
    return O, S


def segment_bounds(n_chunks: int, P: int, C: int, T: int):
    """Token ranges of P segments over a sequence of T tokens: consecutive runs of
    whole chunks, as even as possible (the last may end in a partial chunk)."""
    cuts = [(n_chunks * p) // P * C for p in range(P + 1)]
    cuts[-1] = T
    return [(cuts[p], cuts[p + 1]) for p in range(P)]


def segment_compose(q, k, v, g, beta, S0, C, P, run=None, mutate=None):
    """The two-level (segment-parallel) form of one head's recurrence.

    Over a segment the recurrence is affine in its start state X (the model card's
    closed form of S_T after a chunk, "How it works", applied chunk after chunk):
        S_t = Phi_t X + S0_t,     o_t = X^T m_t + o0_t,
    where (S0_t, o0_t) is the run from X = 0 with the segment's values, and
    (Phi_t, m_t) the run from X = I with all values 0 (so Phi_t = S_t and
    m_t = Phi_t^T q_t are its state and outputs).  Segment 0 runs from the real
    state; the others give (Phi, B = S0_end, m, o0) independently; a short
    sequential combine X_{p+1} = Phi_p X_p + B_p yields every segment's start;
    then each later output is o_t = o0_t + X_p^T m_t.  ``run`` computes one
    segment from a start state (default: the model card's chunk form).
    ``mutate`` plants a mistake for the tests that check the pins catch it:
    "transpose" combines with Phi^T, "no_fixup" drops the X^T m_t term."""
    run = run or (lambda q_, k_, v_, g_, b_, S_: chunk_form_pages(q_, k_, v_, g_, b_, S_, C))
    T = q.shape[0]
    n_chunks = (T + C - 1) // C
    bounds = segment_bounds(n_chunks, P, C, T)
    dk = k.shape[1]
    O = np.zeros((T, v.shape[1]))
    a, b = bounds[0]
    O[a:b], X = run(q[a:b], k[a:b], v[a:b], g[a:b], beta[a:b], np.asarray(S0, np.float64))
    trans = []
    for a, b in bounds[1:]:
        o0, B = run(q[a:b], k[a:b], v[a:b], g[a:b], beta[a:b], np.zeros_like(X))
        m, Phi = run(q[a:b], k[a:b], np.zeros((b - a, dk)), g[a:b], beta[a:b], np.eye(dk))
        trans.append((a, b, o0, B, m, Phi))
    for a, b, o0, B, m, Phi in trans:
        O[a:b] = o0 + (0.0 if mutate == "no_fixup" else m @ X)
        X = (Phi.T if mutate == "transpose" else Phi) @ X + B
    return O, X

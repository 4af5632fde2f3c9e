"""Pins of the oracle's gated delta-rule decode step ("All the attentions", sections 6 Gated
DeltaNet and 7 KDA; "Attention Optimizations", KDA and its chunk-wise form).

Each pin checks the oracle against something other than its own formula:
* the delta rule's stated purpose: with beta = 1 and a unit key, the memory afterwards
  returns exactly v for that key; when the faded memory already predicts v, nothing is
  written;
* special cases: beta = 0 is a pure fade, a zero state gets beta v k^T, a per-channel gate
  with equal channels is the per-head gate;
* the chunk-wise form of the same recurrence (a triangular solve over a chunk of tokens,
  the state carried between chunks) run over several tokens gives the same outputs and the
  same final state as that many single steps;
* a row/column transposition (dv != dk) or a gate applied to rows instead of key channels
  fails these pins.
"""
import numpy as np

import oracle


def _rand(seed, n, dk, dv, per_channel=True):
    rng = np.random.default_rng(seed)
    f = np.float32
    S = rng.standard_normal((n, dv, dk)).astype(f)
    q = rng.standard_normal((n, dk)).astype(f)
    k = rng.standard_normal((n, dk)).astype(f)
    v = rng.standard_normal((n, dv)).astype(f)
    a = rng.uniform(0.5, 1.0, (n, dk) if per_channel else (n,)).astype(f)
    beta = rng.uniform(0.1, 1.0, n).astype(f)
    return S, q, k, v, a, beta


def test_unit_key_full_write_stores_v():
    # beta = 1 and |k| = 1: the corrected memory maps k to v exactly
    S, q, k, v, a, beta = _rand(1, 4, 8, 6)
    k = (k / np.linalg.norm(k, axis=1, keepdims=True)).astype(np.float32)
    k64 = k.astype(np.float64)
    beta[:] = 1.0
    S2, _ = oracle.delta_step(S, q, k, v, a, beta)
    recalled = np.einsum("nij,nj->ni", S2, k64)
    # |k|^2 is 1 up to the float32 rounding of k, so the recall is v up to that rounding
    err = recalled - v.astype(np.float64)
    assert np.abs(err).max() < 1e-5 * (1 + np.abs(v).max())


def test_known_fact_is_not_rewritten():
    # if the faded memory already returns v for k, the write adds nothing
    S, q, k, v, a, beta = _rand(2, 3, 8, 5)
    faded = S.astype(np.float64) * a.astype(np.float64)[:, None, :]
    v_exact = np.einsum("nij,nj->ni", faded, k.astype(np.float64))
    v32 = v_exact.astype(np.float32)
    S2, o = oracle.delta_step(S, q, k, v32, a, beta)
    # the only change left is the float32 rounding of v times beta k
    resid = (v32.astype(np.float64) - v_exact)
    bound = np.abs(resid).max() * np.abs(k).max() * 1.01 + 1e-12
    assert np.abs(S2 - faded).max() <= bound
    assert np.allclose(o, np.einsum("nij,nj->ni", S2, q.astype(np.float64)), rtol=1e-12, atol=1e-12)


def test_zero_write_strength_is_a_pure_fade():
    S, q, k, v, a, beta = _rand(3, 2, 6, 7)
    beta[:] = 0.0
    S2, o = oracle.delta_step(S, q, k, v, a, beta)
    faded = S.astype(np.float64) * a.astype(np.float64)[:, None, :]
    assert np.array_equal(S2, faded)
    assert np.allclose(o, np.einsum("nij,nj->ni", faded, q.astype(np.float64)), rtol=1e-13,
                       atol=1e-13)
    # a = 1, beta = 0: the state is untouched and the read is S q
    a1 = np.ones_like(a)
    S3, o3 = oracle.delta_step(S, q, k, v, a1, beta)
    assert np.array_equal(S3, S.astype(np.float64))


def test_empty_memory_gets_beta_v_k():
    S, q, k, v, a, beta = _rand(4, 3, 5, 4)
    S[:] = 0
    S2, o = oracle.delta_step(S, q, k, v, a, beta)
    b, k64, v64, q64 = beta.astype(np.float64), k.astype(np.float64), v.astype(np.float64), q.astype(np.float64)
    exp_S = b[:, None, None] * v64[:, :, None] * k64[:, None, :]
    assert np.allclose(S2, exp_S, rtol=1e-14, atol=0)
    assert np.allclose(o, b[:, None] * v64 * (k64 * q64).sum(1)[:, None], rtol=1e-12, atol=1e-14)


def test_head_gate_equals_equal_channel_gates():
    S, q, k, v, a, beta = _rand(5, 3, 8, 8, per_channel=False)
    S2, o2 = oracle.delta_step(S, q, k, v, a, beta)
    a_ch = np.repeat(a[:, None], 8, axis=1)
    S3, o3 = oracle.delta_step(S, q, k, v, a_ch, beta)
    assert np.array_equal(S2, S3) and np.array_equal(o2, o3)


def test_gate_acts_on_key_channels():
    # a decay on key channel 2 alone changes column 2 of the state and nothing else
    S, q, k, v, a, beta = _rand(6, 1, 6, 4)
    a[:] = 1.0
    a[0, 2] = 0.25
    beta[:] = 0.0
    S2, _ = oracle.delta_step(S, q, k, v, a, beta)
    d = S2 - S.astype(np.float64)
    assert np.allclose(d[0][:, 2], -0.75 * S[0][:, 2])           # the column of channel 2
    assert np.count_nonzero(np.delete(d[0], 2, axis=1)) == 0     # every other column intact


def _chunked(M0, Q, K, V, A, Bt):
    """The chunk-wise form of the same recurrence over one chunk, written from its algebra:
    M (dk x dv) is the transposed state, g the cumulative product of the per-channel decays.
    The corrections D solve (I + L) D = diag(beta) (V - (K*g) M0) with L strictly lower
    triangular, L[t, s] = beta_t (k_t * g_t) . (k_s / g_s); outputs and the carried state
    follow from D without a per-token loop over the state."""
    g = np.cumprod(A, axis=0)                                    # (C, dk)
    C = K.shape[0]
    L = np.tril(Bt[:, None] * ((K * g) @ (K / g).T), -1)
    D = np.linalg.solve(np.eye(C) + L, Bt[:, None] * (V - (K * g) @ M0))
    Aqk = np.tril((Q * g) @ (K / g).T)                           # diagonal included
    O = (Q * g) @ M0 + Aqk @ D
    M1 = g[-1][:, None] * M0 + (K * (g[-1] / g)).T @ D
    return O, M1


def test_chunked_form_matches_single_steps():
    rng = np.random.default_rng(7)
    dk, dv, C, n_chunks = 8, 6, 5, 3
    T = C * n_chunks
    Q = rng.standard_normal((T, dk))
    K = rng.standard_normal((T, dk))
    K /= np.linalg.norm(K, axis=1, keepdims=True)
    V = rng.standard_normal((T, dv))
    A = rng.uniform(0.6, 1.0, (T, dk))
    Bt = rng.uniform(0.1, 0.9, T)
    S0 = rng.standard_normal((dv, dk))
    # float32 round trip of every input, so that the oracle (which reads float32) and the
    # chunk form (fp64) see the same numbers
    Q, K, V, A, Bt, S0 = (x.astype(np.float32).astype(np.float64) for x in (Q, K, V, A, Bt, S0))
    S = S0.copy()
    outs = []
    for t in range(T):
        S, o = oracle.delta_step(S[None].astype(np.float32), Q[t][None].astype(np.float32),
                                 K[t][None].astype(np.float32), V[t][None].astype(np.float32),
                                 A[t][None].astype(np.float32), Bt[t:t + 1].astype(np.float32))
        S, o = S[0], o[0]
        outs.append(o)
        # the oracle reads float32; the chunk form below carries fp64 state, so both runs
        # are compared through a state rounded to float32 after every step
        S = S.astype(np.float32).astype(np.float64)
    O_steps = np.array(outs)
    M = S0.T.copy()
    O_chunk = []
    Mr = M
    for c in range(n_chunks):
        sl = slice(c * C, (c + 1) * C)
        O, Mr = _chunked(Mr, Q[sl], K[sl], V[sl], A[sl], Bt[sl])
        O_chunk.append(O)
    O_chunk = np.concatenate(O_chunk)
    # the step-by-step run rounds the state to float32 between steps; the chunk form does not
    assert np.abs(O_steps - O_chunk).max() < 1e-5 * (1 + np.abs(O_chunk).max())
    assert np.abs(S - Mr.T).max() < 1e-5 * (1 + np.abs(Mr).max())

"""Pins for the float64 oracle. Each check uses something other than the
oracle's own formula:
  * the unrolled closed form of the Mamba-2 recurrence, and the replay output
    formula (decay products times checkpoint plus weighted buffered inputs);
  * explicit d_k x d_k transition matrices for Gated DeltaNet (brute force);
  * the WY/UT (forward substitution) form of the Gated DeltaNet window;
  * special cases with exact answers (no input, no decay, unit keys);
  * error bounds for the low-precision read copies.
A plausible slip in the oracle (a dropped term, a wrong group index, a
transposed state, a pre-update read) fails at least one of them.
"""
import numpy as np
import pytest

import oracle

RTOL = 1e-12


def _rel(a, b):
    return np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300)


def _m2_problem(rng, B=2, H=4, P=3, N=5, G=2, S=7, scale_dt=1.0):
    h0 = 0.1 * rng.standard_normal((B, H, P, N))
    A = -np.exp(rng.uniform(0, np.log(16), H))
    D = rng.standard_normal(H)
    x = rng.standard_normal((S, B, H, P))
    Bm = rng.standard_normal((S, B, G, N)) / np.sqrt(N)
    C = rng.standard_normal((S, B, G, N)) / np.sqrt(N)
    dt = scale_dt * np.logaddexp(0, rng.standard_normal((S, B, H)) - 2)
    return h0, A, D, x, Bm, C, dt


# ----------------------------------------------------------------------------
# Mamba-2
# ----------------------------------------------------------------------------
def _m2_unrolled_state(h0, A, x, Bm, dt, t, b, h, G):
    """h_t = (prod_{j<=t} a_j) h0 + sum_{i<=t} (prod_{i<j<=t} a_j) dt_i x_i (outer) B_i,
    with explicit products (t is 0-based: tokens 0..t)."""
    H = h0.shape[1]
    g = h // (H // G)
    a = np.exp(dt[: t + 1, b, h] * A[h])
    state = np.prod(a) * h0[b, h]
    for i in range(t + 1):
        state = state + np.prod(a[i + 1:]) * dt[i, b, h] * np.outer(x[i, b, h], Bm[i, b, g])
    return state


def test_m2_matches_unrolled_closed_form():
    rng = np.random.default_rng(1)
    h0, A, D, x, Bm, C, dt = _m2_problem(rng)
    y, hT = oracle.m2_recurrence(h0, A, D, x, Bm, C, dt)
    S, B, H, P = x.shape
    G = Bm.shape[2]
    for b in range(B):
        for h in range(H):
            g = h // (H // G)
            for t in range(S):
                st = _m2_unrolled_state(h0, A, x, Bm, dt, t, b, h, G)
                ref = st @ C[t, b, g] + D[h] * x[t, b, h]
                assert _rel(y[t, b, h], ref) < RTOL
            assert _rel(hT[b, h], _m2_unrolled_state(h0, A, x, Bm, dt, S - 1, b, h, G)) < RTOL


def test_m2_matches_replay_output_formula():
    """y_t = (prod a) h_ckpt C_t + sum_i (prod_{j>i} a_j) dt_i (B_i . C_t) x_i + D x_t,
    the output-from-checkpoint-and-buffer formula, evaluated with scalar weights."""
    rng = np.random.default_rng(2)
    h0, A, D, x, Bm, C, dt = _m2_problem(rng, B=1, H=2, P=4, N=6, G=1, S=16)
    y, _ = oracle.m2_recurrence(h0, A, D, x, Bm, C, dt)
    for h in range(2):
        a = np.exp(dt[:, 0, h] * A[h])
        for t in range(16):
            Ct = C[t, 0, 0]
            out = np.prod(a[: t + 1]) * (h0[0, h] @ Ct) + D[h] * x[t, 0, h]
            for i in range(t + 1):
                w = np.prod(a[i + 1: t + 1]) * dt[i, 0, h] * np.dot(Bm[i, 0, 0], Ct)
                out = out + w * x[i, 0, h]
            assert _rel(y[t, 0, h], out) < RTOL


def test_m2_group_map_is_contiguous_heads():
    """Heads h use group h // (H/G): heads 0,1 -> group 0 and 2,3 -> group 1
    for H=4, G=2. Compare with single-group runs of each head pair."""
    rng = np.random.default_rng(3)
    h0, A, D, x, Bm, C, dt = _m2_problem(rng, B=1, H=4, P=3, N=4, G=2, S=5)
    y, _ = oracle.m2_recurrence(h0, A, D, x, Bm, C, dt)
    for g, heads in ((0, [0, 1]), (1, [2, 3])):
        ys, _ = oracle.m2_recurrence(h0[:, heads], A[heads], D[heads], x[:, :, heads],
                                     Bm[:, :, g:g + 1], C[:, :, g:g + 1], dt[:, :, heads])
        np.testing.assert_array_equal(ys, y[:, :, heads])


def test_m2_no_input_is_pure_decay():
    rng = np.random.default_rng(4)
    h0, A, D, x, Bm, C, dt = _m2_problem(rng)
    Bm = np.zeros_like(Bm)
    y, hT = oracle.m2_recurrence(h0, A, D, x, Bm, C, dt)
    S, B, H, P = x.shape
    for b in range(B):
        for h in range(H):
            g = h // (H // Bm.shape[2])
            for t in range(S):
                gam = np.exp(A[h] * np.sum(dt[: t + 1, b, h]))
                assert _rel(y[t, b, h], gam * (h0[b, h] @ C[t, b, g]) + D[h] * x[t, b, h]) < 1e-12


def test_m2_zero_state_zero_input_is_skip_connection_exactly():
    rng = np.random.default_rng(5)
    h0, A, D, x, Bm, C, dt = _m2_problem(rng)
    y, hT = oracle.m2_recurrence(np.zeros_like(h0), A, D, x, np.zeros_like(Bm), C, dt)
    np.testing.assert_array_equal(y, D[None, None, :, None] * x)
    assert not hT.any()


def test_m2_dt_to_zero_freezes_state():
    rng = np.random.default_rng(6)
    h0, A, D, x, Bm, C, dt = _m2_problem(rng)
    y, hT = oracle.m2_recurrence(h0, A, D, x, Bm, C, np.zeros_like(dt))
    np.testing.assert_array_equal(hT, h0)


def test_m2_nsteps_truncates_each_sequence():
    rng = np.random.default_rng(7)
    h0, A, D, x, Bm, C, dt = _m2_problem(rng, B=3, S=6)
    ns = np.array([0, 2, 6], np.int32)
    y, h = oracle.m2_recurrence(h0, A, D, x, Bm, C, dt, nsteps=ns)
    for b in range(3):
        yb, hb = oracle.m2_recurrence(h0[b:b + 1], A, D, x[: ns[b], b:b + 1], Bm[: ns[b], b:b + 1],
                                      C[: ns[b], b:b + 1], dt[: ns[b], b:b + 1])
        np.testing.assert_array_equal(h[b], hb[0])
        np.testing.assert_array_equal(y[: ns[b], b], yb[:, 0])
        assert np.isnan(y[ns[b]:, b]).all()


def test_m2_speculative_commits_only_accepted_prefix():
    """Draft outputs continue the committed state; the committed state after
    each round equals a plain run over the accepted tokens only."""
    rng = np.random.default_rng(8)
    R, T, B = 4, 3, 2
    h0, A, D, x, Bm, C, dt = _m2_problem(rng, B=B, S=R * T)
    rs = lambda a: a.reshape((R, T) + a.shape[1:])
    acc = np.array([[0, 3], [2, 1], [3, 0], [1, 2]], np.int32)
    y, hc = oracle.m2_speculative(h0, A, D, rs(x), rs(Bm), rs(C), rs(dt), acc)
    for b in range(B):
        keep = [r * T + j for r in range(R) for j in range(acc[r, b])]
        _, hb = oracle.m2_recurrence(h0[b:b + 1], A, D, x[keep][:, b:b + 1], Bm[keep][:, b:b + 1],
                                     C[keep][:, b:b + 1], dt[keep][:, b:b + 1])
        assert _rel(hc[b], hb[0]) < 1e-13
        # round r's draft outputs: from the committed prefix of rounds < r
        for r in range(R):
            pre = [rr * T + j for rr in range(r) for j in range(acc[rr, b])]
            idx = pre + [r * T + j for j in range(T)]
            yb, _ = oracle.m2_recurrence(h0[b:b + 1], A, D, x[idx][:, b:b + 1], Bm[idx][:, b:b + 1],
                                         C[idx][:, b:b + 1], dt[idx][:, b:b + 1])
            assert _rel(y[r, :, b], yb[len(pre):, 0]) < 1e-13


# ----------------------------------------------------------------------------
# Gated DeltaNet
# ----------------------------------------------------------------------------
def _gdn_problem(rng, B=2, H=2, DK=4, DV=3, S=6):
    S0 = 0.1 * rng.standard_normal((B, H, DV, DK))
    q = rng.standard_normal((S, B, H, DK)); q /= np.linalg.norm(q, axis=-1, keepdims=True)
    k = rng.standard_normal((S, B, H, DK)); k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((S, B, H, DV))
    beta = 1 / (1 + np.exp(-rng.standard_normal((S, B, H))))
    alpha = np.exp(-np.logaddexp(0, rng.standard_normal((S, B, H)) - 3))
    return S0, q, k, v, alpha, beta


def test_gdn_matches_explicit_transition_matrices():
    """S_t = S_{t-1} M_t + beta_t v_t k_t^T with M_t = alpha_t (I - beta_t k_t k_t^T),
    multiplied out as d_k x d_k matrices; o_t = S_t (scale q_t)."""
    rng = np.random.default_rng(10)
    S0, q, k, v, alpha, beta = _gdn_problem(rng)
    scale = 0.7
    o, ST = oracle.gdn_recurrence(S0, q, k, v, alpha, beta, scale=scale)
    St_, B, H, DK = q.shape
    for b in range(B):
        for h in range(H):
            Sm = S0[b, h].copy()
            for t in range(St_):
                kt = k[t, b, h]
                M = alpha[t, b, h] * (np.eye(DK) - beta[t, b, h] * np.outer(kt, kt))
                Sm = Sm @ M + beta[t, b, h] * np.outer(v[t, b, h], kt)
                assert _rel(o[t, b, h], Sm @ (scale * q[t, b, h])) < RTOL
            assert _rel(ST[b, h], Sm) < RTOL


def test_gdn_matches_wy_ut_window_form():
    """Over a window of m tokens after a checkpoint S0:
        gamma_i = prod_{j<=i} alpha_j,  A[i,j] = (gamma_i/gamma_j)(k_i . k_j) for j<i,
        T = (I + diag(beta) A)^-1 diag(beta),  U = T (V - diag(gamma) K S0^T),
        S_m = gamma_m S0 + sum_i (gamma_m/gamma_i) u_i k_i^T,
        o_m = gamma_m S0 q_m + sum_i (gamma_m/gamma_i)(k_i . q_m) u_i.
    This is the window algebra the replay kernels evaluate."""
    rng = np.random.default_rng(11)
    m = 9
    S0, q, k, v, alpha, beta = _gdn_problem(rng, B=1, H=1, DK=5, DV=4, S=m)
    o, Sm = oracle.gdn_recurrence(S0, q, k, v, alpha, beta)
    K, V, Q = k[:, 0, 0], v[:, 0, 0], q[:, 0, 0]
    al, be = alpha[:, 0, 0], beta[:, 0, 0]
    S_0 = S0[0, 0]
    gam = np.cumprod(al)
    Amat = np.zeros((m, m))
    for i in range(m):
        for j in range(i):
            Amat[i, j] = gam[i] / gam[j] * (K[i] @ K[j])
    T = np.linalg.solve(np.eye(m) + np.diag(be) @ Amat, np.diag(be))
    U = T @ (V - np.diag(gam) @ K @ S_0.T)
    for t in range(m):
        ot = gam[t] * S_0 @ Q[t] + sum(gam[t] / gam[i] * (K[i] @ Q[t]) * U[i] for i in range(t + 1))
        assert _rel(o[t, 0, 0], ot) < 1e-11
    Sref = gam[-1] * S_0 + sum(gam[-1] / gam[i] * np.outer(U[i], K[i]) for i in range(m))
    assert _rel(Sm[0, 0], Sref) < 1e-11


def test_gdn_beta_zero_is_pure_decay():
    rng = np.random.default_rng(12)
    S0, q, k, v, alpha, beta = _gdn_problem(rng)
    o, ST = oracle.gdn_recurrence(S0, q, k, v, alpha, np.zeros_like(beta))
    gam = np.prod(alpha, axis=0)
    assert _rel(ST, gam[:, :, None, None] * S0) < 1e-13


def test_gdn_unit_gates_store_value_under_key():
    """alpha=1, beta=1, |k|=1: S_t k_t = v_t, so querying with q_t = k_t returns v_t."""
    rng = np.random.default_rng(13)
    S0, q, k, v, alpha, beta = _gdn_problem(rng, DK=6, DV=4)
    o, _ = oracle.gdn_recurrence(S0, k, k, v, np.ones_like(alpha), np.ones_like(beta))
    assert np.max(np.abs(o - v)) < 1e-13


def test_gdn_nsteps_truncates():
    rng = np.random.default_rng(14)
    S0, q, k, v, alpha, beta = _gdn_problem(rng, B=2)
    ns = np.array([1, 4], np.int32)
    o, S = oracle.gdn_recurrence(S0, q, k, v, alpha, beta, nsteps=ns)
    for b in range(2):
        _, Sb = oracle.gdn_recurrence(S0[b:b + 1], q[: ns[b], b:b + 1], k[: ns[b], b:b + 1],
                                      v[: ns[b], b:b + 1], alpha[: ns[b], b:b + 1],
                                      beta[: ns[b], b:b + 1])
        np.testing.assert_array_equal(S[b], Sb[0])


# ----------------------------------------------------------------------------
# Read-copy emulation
# ----------------------------------------------------------------------------
def test_readcopy_flush_outputs_are_exact_and_others_bounded():
    rng = np.random.default_rng(20)
    h0, A, D, x, Bm, C, dt = _m2_problem(rng, B=2, H=2, P=4, N=32, G=1, S=40)
    y, _ = oracle.m2_recurrence(h0, A, D, x, Bm, C, dt)
    k = 8
    for fmt, rel_bound in (("fp8", 2.0 ** -4), ("nvfp4", 17.0 / 96.0)):
        yr = oracle.m2_readcopy(h0, A, D, x, Bm, C, dt, k, fmt)
        flush = [t for t in range(40) if (t + 1) % k == 0]
        np.testing.assert_array_equal(yr[flush], y[flush])
        # non-flush: |err| <= gamma * sum|C| * max|copy - ckpt|, and the copy's
        # error is bounded by rel_bound * amax(ckpt) (fp8: half ulp of 3 mantissa
        # bits; nvfp4: one element quantum at the block scale).
        for b in range(2):
            for h in range(2):
                for t in range(40):
                    if t in flush:
                        continue
                    last = ((t + 1) // k) * k  # tokens folded into the checkpoint
                    ck = _m2_unrolled_state(h0, A, x, Bm, dt, last - 1, b, h, 1) if last else h0[b, h]
                    gam = np.exp(A[h] * np.sum(dt[last: t + 1, b, h]))
                    bound = gam * np.sum(np.abs(C[t, b, 0])) * rel_bound * np.max(np.abs(ck))
                    err = np.max(np.abs(yr[t, b, h] - y[t, b, h]))
                    assert err <= bound * (1 + 1e-9) + 1e-15, (fmt, t, err, bound)


def test_readcopy_is_exact_while_checkpoint_is_representable():
    """A start state on the FP8 grid (scale 1, amax 448) is copied exactly, so
    the first window's outputs equal the exact recurrence."""
    rng = np.random.default_rng(21)
    h0, A, D, x, Bm, C, dt = _m2_problem(rng, B=1, H=2, P=4, N=16, G=1, S=12)
    grid = np.array([0, 0.5, 1.0, 1.5, 2, 3, 24, 448, -448, -0.25, -7], np.float64)
    h0 = rng.choice(grid, size=h0.shape)
    h0[:, :, 0, 0] = 448.0
    y, _ = oracle.m2_recurrence(h0, A, D, x, Bm, C, dt)
    yr = oracle.m2_readcopy(h0, A, D, x, Bm, C, dt, 16, "fp8")
    np.testing.assert_array_equal(yr, y)


def _spec_rounds(rng, R, T, B, H, P, N, G, scale_dt=1.0):
    h0, A, D, x, Bm, C, dt = _m2_problem(rng, B=B, H=H, P=P, N=N, G=G, S=R * T, scale_dt=scale_dt)
    rs = lambda a: a.reshape((R, T) + a.shape[1:])
    return h0, A, D, rs(x), rs(Bm), rs(C), rs(dt)


@pytest.mark.parametrize("fmt", ["fp8", "nvfp4"])
def test_spec_readcopy_state_is_the_plain_speculative_state(fmt):
    """The copy serves reads only: the committed state is m2_speculative's, and
    the checkpoint is that state at the last fold."""
    rng = np.random.default_rng(40)
    R, T, B, k = 7, 3, 3, 5
    h0, A, D, x, Bm, C, dt = _spec_rounds(rng, R, T, B, 2, 4, 16, 1)
    acc = rng.integers(0, T + 1, size=(R, B)).astype(np.int32)
    _, h_ref = oracle.m2_speculative(h0, A, D, x, Bm, C, dt, acc)
    _, h, ck = oracle.m2_speculative_readcopy(h0, A, D, x, Bm, C, dt, acc, k, fmt)
    np.testing.assert_array_equal(h, h_ref)
    for b in range(B):
        n, last = 0, 0
        for r in range(R):                     # tokens committed at the last fold
            n += acc[r, b]
            if n >= k:
                last, n = last + n, 0
        keep = [r * T + j for r in range(R) for j in range(acc[r, b])][:last]
        flat = lambda a: a.reshape((R * T,) + a.shape[2:])
        _, hb = oracle.m2_recurrence(h0[b:b + 1], A, D, flat(x)[keep][:, b:b + 1], flat(Bm)[keep][:, b:b + 1],
                                     flat(C)[keep][:, b:b + 1], flat(dt)[keep][:, b:b + 1])
        assert _rel(ck[b], hb[0]) < 1e-13


def test_spec_readcopy_single_drafts_are_the_readcopy_decode_off_the_flush_token():
    """Rounds of one draft, all accepted, are plain decode. Outputs of tokens
    that do not complete a window equal m2_readcopy's; the token that does
    reads the copy here (the fold comes with the verify), where plain decode
    reads the checkpoint itself."""
    rng = np.random.default_rng(41)
    R, T, B, k = 20, 1, 2, 6
    h0, A, D, x, Bm, C, dt = _spec_rounds(rng, R, T, B, 2, 4, 32, 2)
    acc = np.ones((R, B), np.int32)
    for fmt in ("fp8", "nvfp4"):
        y, _, _ = oracle.m2_speculative_readcopy(h0, A, D, x, Bm, C, dt, acc, k, fmt)
        yr = oracle.m2_readcopy(h0, A, D, x[:, 0], Bm[:, 0], C[:, 0], dt[:, 0], k, fmt)
        ye, _ = oracle.m2_recurrence(h0, A, D, x[:, 0], Bm[:, 0], C[:, 0], dt[:, 0])
        non = [t for t in range(R) if (t + 1) % k != 0]
        assert _rel(y[non, 0], yr[non]) < 1e-13
        flush = [t for t in range(R) if (t + 1) % k == 0]
        np.testing.assert_array_equal(yr[flush], ye[flush])
        assert _rel(y[flush, 0], ye[flush]) > 1e-9      # the copy's error shows there


def test_spec_readcopy_is_exact_while_the_checkpoint_is_representable():
    """A start state on the FP8 grid is copied exactly: until the first fold
    every draft's output is m2_speculative's."""
    rng = np.random.default_rng(42)
    R, T, B, k = 3, 4, 2, 16
    h0, A, D, x, Bm, C, dt = _spec_rounds(rng, R, T, B, 2, 4, 16, 1)
    grid = np.array([0, 0.5, 1.0, 1.5, 2, 3, 24, 448, -448, -0.25, -7], np.float64)
    h0 = rng.choice(grid, size=h0.shape)
    h0[:, :, 0, 0] = 448.0
    acc = np.array([[1, 4], [4, 0], [2, 3]], np.int32)
    y_ref, _ = oracle.m2_speculative(h0, A, D, x, Bm, C, dt, acc)
    y, _, _ = oracle.m2_speculative_readcopy(h0, A, D, x, Bm, C, dt, acc, k, "fp8")
    np.testing.assert_array_equal(y, y_ref)


def test_spec_readcopy_error_is_bounded_by_the_copy_error():
    """|y - y_exact| <= gamma sum|C| * max|copy - ckpt| for every draft, where
    gamma is the decay since the checkpoint (through the draft)."""
    rng = np.random.default_rng(43)
    R, T, B, k = 6, 3, 2, 4
    h0, A, D, x, Bm, C, dt = _spec_rounds(rng, R, T, B, 2, 4, 32, 1)
    acc = rng.integers(0, T + 1, size=(R, B)).astype(np.int32)
    for fmt, rel_bound in (("fp8", 2.0 ** -4), ("nvfp4", 17.0 / 96.0)):
        y, _, _ = oracle.m2_speculative_readcopy(h0, A, D, x, Bm, C, dt, acc, k, fmt)
        ye, _ = oracle.m2_speculative(h0, A, D, x, Bm, C, dt, acc)
        # replay the checkpoint bookkeeping independently
        ck = h0.copy()
        h = h0.copy()
        since = np.zeros((B, 2))
        n = np.zeros(B, np.int64)
        for r in range(R):
            cum = since[None] + np.cumsum(dt[r], axis=0)
            for b in range(B):
                for hh in range(2):
                    for t in range(T):
                        gam = np.exp(A[hh] * cum[t, b, hh])
                        bound = gam * np.sum(np.abs(C[r, t, b, 0])) * rel_bound * np.max(np.abs(ck[b, hh]))
                        err = np.max(np.abs(y[r, t, b, hh] - ye[r, t, b, hh]))
                        assert err <= bound * (1 + 1e-9) + 1e-15, (fmt, r, t, err, bound)
            _, h = oracle.m2_recurrence(h, A, D, x[r], Bm[r], C[r], dt[r], nsteps=acc[r])
            for b in range(B):
                since[b] += dt[r, : acc[r, b], b].sum(axis=0)
            n = n + acc[r]
            f = n >= k
            ck[f], since[f], n[f] = h[f], 0.0, 0


# ----------------------------------------------------------------------------
# Quantised-recurrence baseline
# ----------------------------------------------------------------------------
@pytest.mark.parametrize("fmt", ["fp8", "nvfp4"])
def test_qrecurrence_commutes_with_power_of_two_scaling(fmt):
    """Scaling the start state and the inputs x by 2^5 scales every output by
    exactly 2^5: the tile scales absorb the factor and the codes do not move."""
    rng = np.random.default_rng(30)
    h0, A, D, x, Bm, C, dt = _m2_problem(rng, B=2, H=4, P=8, N=32, G=2, S=10)
    y1 = oracle.m2_qrecurrence(h0, A, D, x, Bm, C, dt, fmt)
    y2 = oracle.m2_qrecurrence(h0 * 32.0, A, D, x * 32.0, Bm, C, dt, fmt)
    np.testing.assert_array_equal(y2, y1 * 32.0)


@pytest.mark.parametrize("fmt", ["fp8", "nvfp4"])
def test_qrecurrence_is_odd(fmt):
    """The quantisers are symmetric, so negating the state and x negates y."""
    rng = np.random.default_rng(31)
    h0, A, D, x, Bm, C, dt = _m2_problem(rng, B=1, H=2, P=8, N=32, G=1, S=8)
    y1 = oracle.m2_qrecurrence(h0, A, D, x, Bm, C, dt, fmt)
    y2 = oracle.m2_qrecurrence(-h0, A, D, -x, Bm, C, dt, fmt)
    np.testing.assert_array_equal(y2, -y1)


@pytest.mark.parametrize("fmt,rel", [("fp8", 2.0 ** -4), ("nvfp4", 17.0 / 96.0)])
def test_qrecurrence_first_token_error_is_the_start_quantisation(fmt, rel):
    """The first token reads the quantised start state: y_1 - y_1(exact) =
    a_1 (Q(h0) - h0) C_1, bounded by a_1 * sum|C| * rel * amax(h0) per row
    (rel: half an FP8 ulp, or one NVFP4 quantum at the block scale)."""
    rng = np.random.default_rng(32)
    h0, A, D, x, Bm, C, dt = _m2_problem(rng, B=2, H=2, P=4, N=32, G=1, S=1)
    y, _ = oracle.m2_recurrence(h0, A, D, x, Bm, C, dt)
    yq = oracle.m2_qrecurrence(h0, A, D, x, Bm, C, dt, fmt)
    for b in range(2):
        for h in range(2):
            a = np.exp(dt[0, b, h] * A[h])
            bound = a * np.sum(np.abs(C[0, b, 0])) * rel * np.max(np.abs(h0[b, h]))
            assert np.max(np.abs(yq[0, b, h] - y[0, b, h])) <= bound * (1 + 1e-9)
            assert np.max(np.abs(yq[0, b, h] - y[0, b, h])) > 0


def test_qrecurrence_error_grows_where_the_read_copy_does_not():
    """Over 12 windows the quantised recurrence drifts from the exact one by
    more than the read copy ever does (its copy is refreshed from the exact
    checkpoint at every flush)."""
    rng = np.random.default_rng(33)
    h0, A, D, x, Bm, C, dt = _m2_problem(rng, B=2, H=2, P=8, N=32, G=1, S=96)
    dt = dt * 0.05                      # slow decay: the state remembers its errors
    y, _ = oracle.m2_recurrence(h0, A, D, x, Bm, C, dt)
    yq = oracle.m2_qrecurrence(h0, A, D, x, Bm, C, dt, "nvfp4")
    yr = oracle.m2_readcopy(h0, A, D, x, Bm, C, dt, 8, "nvfp4")
    eq = np.max(np.abs(yq - y), axis=(1, 2, 3))
    er = np.max(np.abs(yr - y), axis=(1, 2, 3))
    assert eq[-16:].mean() > 2 * er[-16:].mean()


# ----------------------------------------------------------------------------
# Gated DeltaNet speculative rounds
# ----------------------------------------------------------------------------
def _gdn_rounds(rng, R, T, B, H, DK, DV):
    def unit(a):
        return a / np.linalg.norm(a, axis=-1, keepdims=True)
    S0 = 0.1 * rng.standard_normal((B, H, DV, DK))
    q = unit(rng.standard_normal((R, T, B, H, DK)))
    k = unit(rng.standard_normal((R, T, B, H, DK)))
    v = rng.standard_normal((R, T, B, H, DV))
    alpha = np.exp(-np.logaddexp(0, rng.standard_normal((R, T, B, H)) - 3))
    beta = 1 / (1 + np.exp(-rng.standard_normal((R, T, B, H))))
    return S0, q, k, v, alpha, beta


def test_gdn_speculative_all_accepted_is_the_plain_recurrence():
    rng = np.random.default_rng(40)
    R, T, B, H = 5, 3, 2, 2
    S0, q, k, v, al, be = _gdn_rounds(rng, R, T, B, H, 8, 6)
    o, S = oracle.gdn_speculative(S0, q, k, v, al, be, np.full((R, B), T))
    flat = [a.reshape((R * T,) + a.shape[2:]) for a in (q, k, v, al, be)]
    o_ref, S_ref = oracle.gdn_recurrence(S0, *flat)
    np.testing.assert_allclose(o.reshape(o_ref.shape), o_ref, rtol=0, atol=1e-13)
    np.testing.assert_allclose(S, S_ref, rtol=0, atol=1e-13)


def test_gdn_speculative_per_sequence_prefixes():
    """Sequence b's committed state is the recurrence over the accepted
    prefixes of its rounds only, and every round's drafts start from it."""
    rng = np.random.default_rng(41)
    R, T, B, H = 4, 4, 3, 2
    S0, q, k, v, al, be = _gdn_rounds(rng, R, T, B, H, 8, 4)
    acc = np.array([[0, 4, 2], [1, 0, 4], [3, 3, 0], [2, 1, 1]])
    o, S = oracle.gdn_speculative(S0, q, k, v, al, be, acc)
    for b in range(B):
        Sb = S0[b:b + 1]
        for r in range(R):
            sl = (r, slice(None), slice(b, b + 1))
            o_r, _ = oracle.gdn_recurrence(Sb, q[sl], k[sl], v[sl], al[sl], be[sl])
            np.testing.assert_allclose(o[r, :, b], o_r[:, 0], rtol=0, atol=1e-13)
            a = acc[r, b]
            if a:
                pre = (r, slice(0, a), slice(b, b + 1))
                _, Sb = oracle.gdn_recurrence(Sb, q[pre], k[pre], v[pre], al[pre], be[pre])
        np.testing.assert_allclose(S[b], Sb[0], rtol=0, atol=1e-13)


# ----------------------------------------------------------------------------
# FP16 checkpoint
# ----------------------------------------------------------------------------
def test_round_f16_follows_ieee_binary16():
    """Round to nearest, ties to even, gradual underflow, overflow to inf."""
    u = 2.0 ** -10                                # ulp of binary16 at 1
    cases = [(1 + u / 2, 1.0), (1 + 3 * u / 2, 1 + 2 * u), (1 + 0.74 * u, 1 + u),
             (65504.0, 65504.0), (65519.0, 65504.0), (65520.0, np.inf),
             (2.0 ** -25, 0.0), (3 * 2.0 ** -26, 2.0 ** -24), (-(1 + u / 2), -1.0),
             (2.0 ** -14 * (1 + u), 2.0 ** -14 * (1 + u))]
    for v, want in cases:
        assert oracle.round_f16(v) == want, (v, want)


def _ckpt16_scalar_problem(S):
    """One scalar state (B=H=G=P=N=1) with no decay (A = 0), no skip (D = 0),
    C = B = dt = 1 and x = 3 * 2^-13: each token adds exactly 3 * 2^-13."""
    h0 = np.full((1, 1, 1, 1), 1 + 2.0 ** -12)
    A, D = np.zeros(1), np.zeros(1)
    x = np.full((S, 1, 1, 1), 3 * 2.0 ** -13)
    Bm, C = np.ones((S, 1, 1, 1)), np.ones((S, 1, 1, 1))
    dt = np.ones((S, 1, 1))
    return h0, A, D, x, Bm, C, dt


def test_ckpt16_hand_computed_scalar_windows():
    """Worked by hand from the binary16 grid near 1 (ulp 2^-10 = 8 * 2^-13):
    the start 1 + 2^-12 rounds to 1; k = 2 commits after tokens 2 and 4, at
    1 + 6*2^-13 (-> 1 + 2^-10) and 1 + 14*2^-13 (-> 1 + 2^-9); token 5 is
    left uncommitted."""
    e = 2.0 ** -13
    h0, A, D, x, Bm, C, dt = _ckpt16_scalar_problem(5)
    y, ck = oracle.m2_ckpt16(h0, A, D, x, Bm, C, dt, k=2)
    want = [1 + 3 * e, 1 + 6 * e, 1 + 11 * e, 1 + 14 * e, 1 + 19 * e]
    np.testing.assert_array_equal(y.ravel(), want)
    assert ck.item() == 1 + 2.0 ** -9
    # explicit windows 1, 2, 2: commits at 1 + 3e (-> 1), 1 + 6e (-> 1 + 8e),
    # 1 + 14e (-> 1 + 16e)
    y, ck = oracle.m2_ckpt16(h0, A, D, x, Bm, C, dt, k=2, windows=[1, 2, 2])
    np.testing.assert_array_equal(y.ravel(), [1 + 3 * e, 1 + 3 * e, 1 + 6 * e, 1 + 11 * e, 1 + 14 * e])
    assert ck.item() == 1 + 2.0 ** -9
    # the FP8 read copy of a one-element tile is the value itself up to the
    # float32 tile scale, so the outputs are those above within 2^-20; a copy
    # made from the unrounded start would be off by 2^-12 on token 1
    y8, _ = oracle.m2_ckpt16(h0, A, D, x, Bm, C, dt, k=2, fmt="fp8")
    np.testing.assert_allclose(y8.ravel(), want, rtol=0, atol=2.0 ** -20)


def test_ckpt16_is_exact_on_the_binary16_grid():
    """Integer states, inputs and steps with no decay stay on the binary16
    grid, so rounding the checkpoint changes nothing."""
    rng = np.random.default_rng(40)
    B, H, P, N, G, S = 2, 2, 3, 4, 1, 9
    h0 = rng.integers(-20, 20, (B, H, P, N)).astype(np.float64)
    A, D = np.zeros(H), rng.integers(-3, 3, H).astype(np.float64)
    x = rng.integers(-4, 4, (S, B, H, P)).astype(np.float64)
    Bm = rng.integers(-2, 3, (S, B, G, N)).astype(np.float64)
    C = rng.integers(-2, 3, (S, B, G, N)).astype(np.float64)
    dt = rng.integers(1, 3, (S, B, H)).astype(np.float64)
    y, h = oracle.m2_recurrence(h0, A, D, x, Bm, C, dt)
    y16, ck = oracle.m2_ckpt16(h0, A, D, x, Bm, C, dt, k=3)
    np.testing.assert_array_equal(y16, y)
    np.testing.assert_array_equal(ck, h)


def test_ckpt16_error_is_the_propagated_rounding():
    """The recurrence is linear, so the output error at token t is the sum over
    earlier commits f of gamma(f -> t) * (rounding error at f) . C_t. Each
    rounding is at most 2^-11 (+2^-24 for the float32 step) of the value,
    giving a per-row bound; the bound holds, the error is not zero, and every
    returned checkpoint value is on the binary16 grid."""
    rng = np.random.default_rng(41)
    h0, A, D, x, Bm, C, dt = _m2_problem(rng, B=2, H=2, P=4, N=8, G=1, S=23)
    k = 5
    y, _ = oracle.m2_recurrence(h0, A, D, x, Bm, C, dt)
    y16, ck = oracle.m2_ckpt16(h0, A, D, x, Bm, C, dt, k=k)
    np.testing.assert_array_equal(oracle.round_f16(ck), ck)
    u = 2.0 ** -11 + 2.0 ** -24
    commits = [0] + list(range(k, 23, k))           # tokens folded before each rounding
    assert np.max(np.abs(y16 - y)) > 0
    for b in range(2):
        for h in range(2):
            for t in range(23):
                bound = 0.0
                for f in commits:
                    if f > t:
                        break
                    hf = _m2_unrolled_state(h0, A, x, Bm, dt, f - 1, b, h, 1) if f else h0[b, h]
                    gam = np.exp(A[h] * np.sum(dt[f: t + 1, b, h]))
                    bound += gam * (np.abs(hf) * u + 2.0 ** -25) @ np.abs(C[t, b, 0])
                err = np.abs(y16[t, b, h] - y[t, b, h])
                assert np.all(err <= bound * 1.01 + 1e-15), (t, err, bound)


# ----------------------------------------------------------------------------
# Synthetic decode stack
# ----------------------------------------------------------------------------
def test_round_bf16_follows_round_to_nearest_even():
    u = 2.0 ** -7                                 # ulp of bfloat16 at 1
    for v, want in [(1 + u / 2, 1.0), (1 + 3 * u / 2, 1 + 2 * u), (1 + u / 2 + 2.0 ** -20, 1 + u),
                    (-(1 + u / 2), -1.0), (3.0, 3.0), (0.1, 0.10009765625)]:
        assert oracle.round_bf16(v) == want, (v, want)


def _stack_problem(rng, L=2, Bsz=3, H=4, P=4, N=8, G=2, S=3):
    dm, di = H * P // 2, H * P

    def w(r, c):
        return oracle.round_bf16(rng.standard_normal((r, c)) / np.sqrt(r))
    weights = [{"x": w(dm, di), "z": w(dm, di), "B": w(dm, G * N), "C": w(dm, G * N), "dt": w(dm, H),
                "out": w(di, dm), "dt_bias": rng.uniform(-4, -2, H)} for _ in range(L)]
    params = [(-np.exp(rng.uniform(0, 2, H)), rng.standard_normal(H)) for _ in range(L)]
    states = [0.1 * rng.standard_normal((Bsz, H, P, N)) for _ in range(L)]
    u = oracle.round_bf16(rng.standard_normal((S, Bsz, dm)))
    return u, weights, params, states


def test_stack_without_out_projection_is_the_identity():
    rng = np.random.default_rng(50)
    u, weights, params, states = _stack_problem(rng)
    for w in weights:
        w["out"] = np.zeros_like(w["out"])
    out, deltas, _ = oracle.m2_stack(u, weights, params, states)
    np.testing.assert_array_equal(out, u)
    assert not deltas.any()


def test_stack_closed_gate_adds_nothing():
    """silu(0) = 0: with W_z = 0 the gate closes and no layer changes u, while
    the SSM states still advance."""
    rng = np.random.default_rng(51)
    u, weights, params, states = _stack_problem(rng)
    for w in weights:
        w["z"] = np.zeros_like(w["z"])
    out, deltas, st = oracle.m2_stack(u, weights, params, states)
    np.testing.assert_array_equal(out, u)
    assert not deltas.any()
    assert all(np.max(np.abs(a - b)) > 0 for a, b in zip(st, states))


def test_stack_layer_input_is_scale_free():
    """RMS normalisation: scaling the embedding by 2^3 scales n by nothing, so
    the first layer's delta is unchanged bit for bit."""
    rng = np.random.default_rng(52)
    u, weights, params, states = _stack_problem(rng, L=1, S=1)
    _, d1, _ = oracle.m2_stack(u, weights, params, states)
    _, d2, _ = oracle.m2_stack(u * 8.0, weights, params, states)
    np.testing.assert_array_equal(d1, d2)
    assert d1.any()


# ----------------------------------------------------------------------------
# Gated DeltaNet read copies
# ----------------------------------------------------------------------------
def test_gdn_readcopy_flush_outputs_and_checkpoint_are_exact():
    rng = np.random.default_rng(60)
    S0, q, k, v, alpha, beta = _gdn_problem(rng, B=2, H=2, DK=16, DV=64, S=11)
    o, S = oracle.gdn_recurrence(S0, q, k, v, alpha, beta, scale=0.5)
    for fmt in ("fp8", "nvfp4"):
        orc, Sr = oracle.gdn_readcopy(S0, q, k, v, alpha, beta, 4, fmt, scale=0.5)
        np.testing.assert_array_equal(orc[[3, 7]], o[[3, 7]])
        _, S8 = oracle.gdn_recurrence(S0, q[:8], k[:8], v[:8], alpha[:8], beta[:8], scale=0.5)
        np.testing.assert_array_equal(Sr, S8)          # tokens 9..11 are left uncommitted
        assert np.max(np.abs(orc - o)) > 0


def test_gdn_readcopy_is_exact_while_the_state_is_representable():
    """Each 64-row half on the FP8 grid with amax 448: the copy is the state."""
    rng = np.random.default_rng(61)
    S0, q, k, v, alpha, beta = _gdn_problem(rng, B=1, H=2, DK=16, DV=128, S=5)
    grid = np.array([0, 0.5, 1.0, 1.5, 2, 3, 24, 448, -448, -0.25, -7], np.float64)
    S0 = rng.choice(grid, size=S0.shape)
    S0[:, :, 0, 0] = 448.0
    S0[:, :, 64, 0] = -448.0
    o, _ = oracle.gdn_recurrence(S0, q, k, v, alpha, beta)
    orc, _ = oracle.gdn_readcopy(S0, q, k, v, alpha, beta, 8, "fp8")
    np.testing.assert_array_equal(orc, o)


@pytest.mark.parametrize("fmt", ["fp8", "nvfp4"])
def test_gdn_readcopy_error_per_row_is_bounded_by_the_copy_error(fmt):
    """Rows of S evolve independently (S_t = S_{t-1} M_t + ...), and with unit
    keys and beta in [0, 1] each M_t = alpha_t (I - beta_t k_t k_t^T) has
    spectral norm alpha_t. So row r of a non-flush output moves by at most
    gamma ||row r of (copy - S_ckpt)||_2 ||scale q||_2. The two halves of each
    tile differ in magnitude by 10^3: a copy with one scale per tile instead of
    per half fails the bound on the small half."""
    rng = np.random.default_rng(62)
    S0, q, k, v, alpha, beta = _gdn_problem(rng, B=2, H=2, DK=32, DV=128, S=6)
    S0[:, :, :64] *= 1e-3
    scale = 0.7
    o, _ = oracle.gdn_recurrence(S0, q, k, v, alpha, beta, scale=scale)
    orc, _ = oracle.gdn_readcopy(S0, q, k, v, alpha, beta, 16, fmt, scale=scale)
    halves = S0.reshape(-1, 64, 32).astype(np.float32)
    if fmt == "fp8":
        copy = oracle.dequant_fp8(*oracle.quant_fp8(halves))
    else:
        copy = oracle.dequant_nvfp4(*oracle.quant_nvfp4(halves))
    dS = np.linalg.norm(copy.reshape(S0.shape) - S0, axis=-1)        # [B][H][DV]
    gam = np.cumprod(alpha, axis=0)                                    # [S][B][H]
    bound = gam[..., None] * dS[None] * scale * np.linalg.norm(q, axis=-1)[..., None]
    err = np.abs(orc - o)
    assert np.all(err <= bound * (1 + 1e-9) + 1e-15)
    assert err[:, :, :, :64].max() > 0 and err[:, :, :, :64].max() < 1e-3 * err[:, :, :, 64:].max()


def test_gdn_readcopy_explicit_windows():
    """Windows 3 then 4 (k = 4): the first ends in an explicit flush, so none of
    its outputs is exact; the second window's copy is made from the state
    after 3 tokens."""
    rng = np.random.default_rng(63)
    S0, q, k, v, alpha, beta = _gdn_problem(rng, B=1, H=2, DK=16, DV=64, S=8)
    o, _ = oracle.gdn_recurrence(S0, q, k, v, alpha, beta)
    orc, S7 = oracle.gdn_readcopy(S0, q, k, v, alpha, beta, 4, "fp8", windows=[3, 4])
    assert np.all(np.max(np.abs(orc[:3] - o[:3]), axis=(1, 2, 3)) > 0)
    np.testing.assert_array_equal(orc[6], o[6])
    _, S3 = oracle.gdn_recurrence(S0, q[:3], k[:3], v[:3], alpha[:3], beta[:3])
    o2, _ = oracle.gdn_recurrence(oracle.gdn_copy(S3, "fp8"), q[3:6], k[3:6], v[3:6], alpha[3:6], beta[3:6])
    np.testing.assert_array_equal(orc[3:6], o2)
    _, S_ref = oracle.gdn_recurrence(S0, q[:7], k[:7], v[:7], alpha[:7], beta[:7])
    np.testing.assert_array_equal(S7, S_ref)


# ----------------------------------------------------------------------------
# FP8 / NVFP4 checkpoints
# ----------------------------------------------------------------------------
def _tile_scalar_problem(h0_row, add, S):
    """One sequence, one head, P = 1: no decay (A = 0), no skip (D = 0), x = dt = 1,
    B = e_1 (each token adds `add` to element 1), C = e_1 (y reads element 1)."""
    N = len(h0_row)
    h0 = np.array(h0_row, np.float64).reshape(1, 1, 1, N)
    A, D = np.zeros(1), np.zeros(1)
    x = np.full((S, 1, 1, 1), add)
    e1 = np.zeros(N)
    e1[1] = 1.0
    Bm = np.tile(e1, (S, 1, 1, 1))
    C = np.tile(e1, (S, 1, 1, 1))
    dt = np.ones((S, 1, 1))
    return h0, A, D, x, Bm, C, dt


def test_fp8_checkpoint_hand_computed():
    """Tile [448, v]: the tile scale is 1, so v is stored as E4M3(v) (spacing 8 on
    [64, 128), 16 on [128, 256)). 100 -> 96 (tie, even), 110 -> 112, 126 -> 128."""
    h0, A, D, x, Bm, C, dt = _tile_scalar_problem([448.0, 100.0], 7.0, 5)
    y, ck = oracle.m2_ckpt_lowp(h0, A, D, x, Bm, C, dt, 2, "fp8")
    np.testing.assert_array_equal(y.ravel(), [103, 110, 119, 126, 135])
    np.testing.assert_array_equal(ck.ravel(), [448, 128])


def test_nvfp4_checkpoint_hand_computed():
    """Tile [6, v, 0 x 14]: the block scale decodes to 448 and the element step to
    1 (up to float32 rounding), so v is stored as E2M1(v) on {..., 2, 3, 4, 6}:
    2.6 -> 3, 3.6 -> 4, 4.6 -> 4."""
    h0, A, D, x, Bm, C, dt = _tile_scalar_problem([6.0, 2.6] + [0.0] * 14, 0.3, 5)
    y, ck = oracle.m2_ckpt_lowp(h0, A, D, x, Bm, C, dt, 2, "nvfp4")
    np.testing.assert_allclose(y.ravel(), [3.3, 3.6, 4.3, 4.6, 4.3], rtol=1e-6)
    np.testing.assert_allclose(ck.ravel()[:2], [6, 4], rtol=1e-6)


@pytest.mark.parametrize("store,rel", [("fp8", 2.0 ** -4), ("nvfp4", 17.0 / 96.0)])
def test_tile_checkpoint_error_is_the_propagated_rounding(store, rel):
    """Each store moves an element by at most rel * amax of its tile (half an
    FP8 ulp; one NVFP4 quantum at the block scale), and the recurrence is
    linear: the output error at token t is bounded by the sum over earlier
    stores f of gamma(f -> t) * rel * amax(h_f) * sum|C_t|."""
    rng = np.random.default_rng(70)
    h0, A, D, x, Bm, C, dt = _m2_problem(rng, B=2, H=2, P=4, N=32, G=1, S=21)
    k = 5
    y, _ = oracle.m2_recurrence(h0, A, D, x, Bm, C, dt)
    yl, _ = oracle.m2_ckpt_lowp(h0, A, D, x, Bm, C, dt, k, store)
    commits = [0] + list(range(k, 21, k))
    assert np.max(np.abs(yl - y)) > 0
    for b in range(2):
        for h in range(2):
            for t in range(21):
                bound = 0.0
                for f in commits:
                    if f > t:
                        break
                    hf = _m2_unrolled_state(h0, A, x, Bm, dt, f - 1, b, h, 1) if f else h0[b, h]
                    gam = np.exp(A[h] * np.sum(dt[f: t + 1, b, h]))
                    bound += gam * rel * np.max(np.abs(hf)) * np.sum(np.abs(C[t, b, 0]))
                err = np.max(np.abs(yl[t, b, h] - y[t, b, h]))
                assert err <= bound * 1.05 + 1e-15, (store, t, err, bound)


@pytest.mark.parametrize("store", ["fp8", "nvfp4"])
def test_tile_checkpoint_drifts_less_than_the_per_token_quantised_recurrence(store):
    """The same format, rounded once per window of 8 instead of at every token:
    both read a state rounded once since its last store, but the per-token
    scheme also carries every earlier token's rounding (about 1.6x to 1.8x the
    late error on this slowly decaying case)."""
    rng = np.random.default_rng(71)
    h0, A, D, x, Bm, C, dt = _m2_problem(rng, B=2, H=2, P=8, N=32, G=1, S=96)
    dt = dt * 0.05
    y, _ = oracle.m2_recurrence(h0, A, D, x, Bm, C, dt)
    yq = oracle.m2_qrecurrence(h0, A, D, x, Bm, C, dt, store)
    yl, _ = oracle.m2_ckpt_lowp(h0, A, D, x, Bm, C, dt, 8, store)
    eq = np.max(np.abs(yq - y), axis=(1, 2, 3))
    el = np.max(np.abs(yl - y), axis=(1, 2, 3))
    assert el[-16:].mean() < 0.75 * eq[-16:].mean()


def test_stack_hand_computed_layer():
    """One layer worked by hand (d_model 2, two heads of P = 2, N = 2, G = 1):
    u = [1, 7] has RMS 5, so n = [0.2, 1.4]; x = [n0, n1, n0, n1];
    z = 40 [n0, n1, n0, -n1], so SiLU passes the first three channels (z >= 8)
    and closes the last (z = -56); B = C = [n0, 0], so B.C = n0^2; W_dt = 0, so
    dt = softplus(bias) = softplus(-3) = log(1 + e^-3); zero start state, no decay
    or skip, so y_p = dt x_p n0^2; W_out routes channel 0 to u_0 and channel 3 to
    u_1. Hence delta_0 = 40 softplus(-3) n0^4 and delta_1 = 0 (up to the bf16
    storage points, within 3 %)."""
    W = lambda rows: np.array(rows, np.float64)
    w = {"x": W([[1, 0, 1, 0], [0, 1, 0, 1]]), "z": W([[40, 0, 40, 0], [0, 40, 0, -40]]),
         "B": W([[1, 0], [0, 0]]), "C": W([[1, 0], [0, 0]]), "dt": np.zeros((2, 2)),
         "out": W([[1, 0], [0, 0], [0, 0], [0, 1]]), "dt_bias": np.array([-3.0, -3.0])}
    params = [(np.zeros(2), np.zeros(2))]
    states = [np.zeros((1, 2, 2, 2))]
    u = np.array([[[1.0, 7.0]]])
    _, deltas, _ = oracle.m2_stack(u, [w], params, states)
    want0 = 40 * np.log1p(np.exp(-3.0)) * 0.2 ** 4
    assert abs(deltas[0, 0, 0, 0] - want0) <= 0.03 * want0
    assert abs(deltas[0, 0, 0, 1]) <= 1e-9


# ----------------------------------------------------------------------------
# Gated DeltaNet quantised-recurrence baseline
# ----------------------------------------------------------------------------
@pytest.mark.parametrize("fmt", ["fp8", "nvfp4"])
def test_gdn_qrecurrence_commutes_with_power_of_two_scaling(fmt):
    """The recurrence is linear in (S, v): scaling the start state and v by
    2^5 scales every output by exactly 2^5 (the half-tile scales absorb the
    factor and the codes do not move)."""
    rng = np.random.default_rng(70)
    S0, q, k, v, alpha, beta = _gdn_problem(rng, B=2, H=2, DK=16, DV=128, S=7)
    o1 = oracle.gdn_qrecurrence(S0, q, k, v, alpha, beta, fmt, scale=0.5)
    o2 = oracle.gdn_qrecurrence(S0 * 32.0, q, k, v * 32.0, alpha, beta, fmt, scale=0.5)
    np.testing.assert_array_equal(o2, o1 * 32.0)


@pytest.mark.parametrize("fmt", ["fp8", "nvfp4"])
def test_gdn_qrecurrence_is_odd(fmt):
    """The quantisers are symmetric: negating the state and v negates o."""
    rng = np.random.default_rng(71)
    S0, q, k, v, alpha, beta = _gdn_problem(rng, B=1, H=2, DK=16, DV=64, S=6)
    o1 = oracle.gdn_qrecurrence(S0, q, k, v, alpha, beta, fmt)
    o2 = oracle.gdn_qrecurrence(-S0, q, k, -v, alpha, beta, fmt)
    np.testing.assert_array_equal(o2, -o1)


@pytest.mark.parametrize("fmt", ["fp8", "nvfp4"])
def test_gdn_qrecurrence_first_token_error_is_the_start_quantisation(fmt):
    """The first token reads the quantised start state. Rows of S evolve
    independently through M_1 = alpha_1 (I - beta_1 k_1 k_1^T), of spectral
    norm alpha_1 for a unit key, so row r of o_1 moves by at most
    alpha_1 ||row r of (Q(S0) - S0)||_2 ||scale q_1||_2 (Q per 64-row half)."""
    rng = np.random.default_rng(72)
    S0, q, k, v, alpha, beta = _gdn_problem(rng, B=2, H=2, DK=32, DV=128, S=1)
    scale = 0.7
    o, _ = oracle.gdn_recurrence(S0, q, k, v, alpha, beta, scale=scale)
    oq = oracle.gdn_qrecurrence(S0, q, k, v, alpha, beta, fmt, scale=scale)
    halves = S0.reshape(-1, 64, 32).astype(np.float32)
    if fmt == "fp8":
        stored = oracle.dequant_fp8(*oracle.quant_fp8(halves))
    else:
        stored = oracle.dequant_nvfp4(*oracle.quant_nvfp4(halves))
    dS = np.linalg.norm(stored.reshape(S0.shape) - S0, axis=-1)           # [B][H][DV]
    bound = alpha[0][..., None] * dS * scale * np.linalg.norm(q[0], axis=-1)[..., None]
    err = np.abs(oq[0] - o[0])
    assert np.all(err <= bound * (1 + 1e-9) + 1e-15)
    assert err.max() > 0


def test_gdn_qrecurrence_first_output_is_exact_on_the_grid():
    """Each 64-row half on the FP8 grid with amax 448 quantises to itself, so
    the first output is the exact recurrence's; later ones are not (the
    updated state leaves the grid)."""
    rng = np.random.default_rng(73)
    S0, q, k, v, alpha, beta = _gdn_problem(rng, B=1, H=2, DK=16, DV=128, S=4)
    grid = np.array([0, 0.5, 1.0, 1.5, 2, 3, 24, 448, -448, -0.25, -7], np.float64)
    S0 = rng.choice(grid, size=S0.shape)
    S0[:, :, 0, 0] = 448.0
    S0[:, :, 64, 0] = -448.0
    o, _ = oracle.gdn_recurrence(S0, q, k, v, alpha, beta)
    oq = oracle.gdn_qrecurrence(S0, q, k, v, alpha, beta, "fp8")
    np.testing.assert_array_equal(oq[0], o[0])
    assert np.max(np.abs(oq[1:] - o[1:])) > 0


def test_gdn_qrecurrence_error_grows_where_the_read_copy_does_not():
    """With slow decay (alpha near 1) the quantised recurrence drifts from the
    exact one by more than the read copy ever does over 12 windows (the copy
    is remade from the exact checkpoint at every flush)."""
    rng = np.random.default_rng(74)
    S0, q, k, v, alpha, beta = _gdn_problem(rng, B=1, H=2, DK=16, DV=64, S=96)
    alpha = 1.0 - 0.01 * (1.0 - alpha)
    beta = 0.1 * beta
    o, _ = oracle.gdn_recurrence(S0, q, k, v, alpha, beta)
    oq = oracle.gdn_qrecurrence(S0, q, k, v, alpha, beta, "nvfp4")
    orc, _ = oracle.gdn_readcopy(S0, q, k, v, alpha, beta, 8, "nvfp4")
    eq = np.max(np.abs(oq - o), axis=(1, 2, 3))
    er = np.max(np.abs(orc - o), axis=(1, 2, 3))
    assert eq[-16:].mean() > 2 * er[-16:].mean()


# ----------------------------------------------------------------------------
# Gated DeltaNet FP16 checkpoint
# ----------------------------------------------------------------------------
def test_gdn_ckpt16_commutes_with_power_of_two_scaling():
    """Binary16 rounding commutes with a 2^5 scaling in the normal range, and
    the recurrence is linear in (S, v). The state is scaled up 100-fold so
    that no stored value is a binary16 subnormal, whose rounding does not
    commute."""
    rng = np.random.default_rng(80)
    S0, q, k, v, alpha, beta = _gdn_problem(rng, B=2, H=2, DK=16, DV=64, S=11)
    S0, v = S0 * 100.0, v * 100.0
    o1, S1 = oracle.gdn_ckpt16(S0, q, k, v, alpha, beta, 4, scale=0.5)
    o2, S2 = oracle.gdn_ckpt16(S0 * 32.0, q, k, v * 32.0, alpha, beta, 4, scale=0.5)
    np.testing.assert_array_equal(o2, o1 * 32.0)
    np.testing.assert_array_equal(S2, S1 * 32.0)


def test_gdn_ckpt16_is_exact_for_a_representable_start():
    """A start state of binary16 values is stored as it is: the first window's
    outputs are the exact recurrence's, and the checkpoint after it is the
    exact end state rounded to binary16 (which moves it)."""
    rng = np.random.default_rng(81)
    S0, q, k, v, alpha, beta = _gdn_problem(rng, B=1, H=2, DK=16, DV=64, S=6)
    S0 = S0.astype(np.float16).astype(np.float64)
    o, S_end = oracle.gdn_recurrence(S0, q[:4], k[:4], v[:4], alpha[:4], beta[:4])
    o16, S16 = oracle.gdn_ckpt16(S0, q, k, v, alpha, beta, 4, windows=[4])
    np.testing.assert_array_equal(o16[:4], o)
    assert np.max(np.abs(S16 - S_end)) > 0
    assert np.max(np.abs(S16 - S_end) / np.maximum(np.abs(S_end), 2.0 ** -14)) <= 2.0 ** -11


def test_gdn_ckpt16_first_window_error_is_bounded_by_the_rounding():
    """Row r of S evolves through M_t = alpha_t (I - beta_t k_t k_t^T), of
    spectral norm alpha_t for unit keys, so in the first window row r of
    o_t moves by at most gamma_t ||row r of (f16(S0) - S0)||_2 ||scale q_t||_2,
    and ||f16(s) - s|| <= 2^-11 |s| elementwise in the normal range."""
    rng = np.random.default_rng(82)
    S0, q, k, v, alpha, beta = _gdn_problem(rng, B=2, H=2, DK=32, DV=64, S=6)
    scale = 0.7
    o, _ = oracle.gdn_recurrence(S0, q, k, v, alpha, beta, scale=scale)
    o16, _ = oracle.gdn_ckpt16(S0, q, k, v, alpha, beta, 16, scale=scale)
    dS = np.linalg.norm(S0, axis=-1) * 2.0 ** -11                        # [B][H][DV]
    gam = np.cumprod(alpha, axis=0)
    bound = gam[..., None] * dS[None] * scale * np.linalg.norm(q, axis=-1)[..., None]
    err = np.abs(o16 - o)
    assert np.all(err <= bound * (1 + 1e-9))
    assert err.max() > 0


def test_gdn_ckpt16_with_k1_rounds_the_state_after_every_token():
    """k = 1: every token is a flush, so the stored state is the FP16-rounded
    state after every token (a plain loop over single tokens)."""
    rng = np.random.default_rng(83)
    S0, q, k, v, alpha, beta = _gdn_problem(rng, B=1, H=2, DK=16, DV=64, S=5)
    o16, S16 = oracle.gdn_ckpt16(S0, q, k, v, alpha, beta, 1)
    S = S0.astype(np.float32).astype(np.float16).astype(np.float64)
    for t in range(5):
        sl = slice(t, t + 1)
        o, S = oracle.gdn_recurrence(S, q[sl], k[sl], v[sl], alpha[sl], beta[sl])
        np.testing.assert_array_equal(o16[t], o[0])
        S = S.astype(np.float32).astype(np.float16).astype(np.float64)
    np.testing.assert_array_equal(S16, S)


# ----------------------------------------------------------------------------
# Gated DeltaNet speculative rounds that read the copy
# ----------------------------------------------------------------------------
@pytest.mark.parametrize("fmt", ["fp8", "nvfp4"])
def test_gdn_spec_readcopy_state_is_the_plain_speculative_state(fmt):
    """The copy serves reads only: the committed state is gdn_speculative's,
    and the checkpoint is that state at the sequence's last fold."""
    rng = np.random.default_rng(90)
    R, T, B, k = 6, 3, 3, 4
    S0, q, kk, v, al, be = _gdn_rounds(rng, R, T, B, 2, 16, 64)
    acc = rng.integers(0, T + 1, size=(R, B))
    o, S_plain = oracle.gdn_speculative(S0, q, kk, v, al, be, acc)
    _, S, ck = oracle.gdn_speculative_readcopy(S0, q, kk, v, al, be, acc, k, fmt)
    np.testing.assert_allclose(S, S_plain, rtol=0, atol=1e-13)
    # each sequence's checkpoint is its state after its last fold
    for b in range(B):
        n, last = 0, None
        for r in range(R):
            n += acc[r, b]
            if n >= k:
                n, last = 0, r
        if last is None:
            np.testing.assert_array_equal(ck[b], S0[b])
        else:
            _, Sb = oracle.gdn_speculative(S0[b:b + 1], q[: last + 1, :, b:b + 1], kk[: last + 1, :, b:b + 1],
                                           v[: last + 1, :, b:b + 1], al[: last + 1, :, b:b + 1],
                                           be[: last + 1, :, b:b + 1], acc[: last + 1, b:b + 1])
            np.testing.assert_allclose(ck[b], Sb[0], rtol=0, atol=1e-13)


@pytest.mark.parametrize("fmt", ["fp8", "nvfp4"])
def test_gdn_spec_readcopy_single_drafts_are_the_readcopy_decode_off_the_flush_token(fmt):
    """Rounds of one draft, each accepted, walk the plain decode: every output
    is the read-copy decode's, bit for bit, except the flush token, which in
    plain decode reads the checkpoint itself."""
    rng = np.random.default_rng(91)
    R, k = 11, 4
    S0, q, kk, v, al, be = _gdn_rounds(rng, R, 1, 2, 2, 16, 64)
    acc = np.ones((R, 2), np.int64)
    o, _, _ = oracle.gdn_speculative_readcopy(S0, q, kk, v, al, be, acc, k, fmt, scale=0.5)
    flat = [a[:, 0] for a in (q, kk, v, al, be)]
    o_rc, _ = oracle.gdn_readcopy(S0, *flat, k, fmt, scale=0.5)
    keep = [t for t in range(R) if (t + 1) % k]
    np.testing.assert_array_equal(o[keep, 0], o_rc[keep])
    flush = [t for t in range(R) if (t + 1) % k == 0]
    assert np.max(np.abs(o[flush, 0] - o_rc[flush])) > 0


def test_gdn_spec_readcopy_is_exact_while_the_checkpoint_is_representable():
    """Each 64-row half on the FP8 grid with amax 448: until the first fold
    the copy is the checkpoint, so the drafts are the exact rounds'."""
    rng = np.random.default_rng(92)
    R, T, B = 2, 3, 2
    S0, q, kk, v, al, be = _gdn_rounds(rng, R, T, B, 2, 16, 128)
    grid = np.array([0, 0.5, 1.0, 1.5, 2, 3, 24, 448, -448, -0.25, -7], np.float64)
    S0 = rng.choice(grid, size=S0.shape)
    S0[:, :, 0, 0] = 448.0
    S0[:, :, 64, 0] = -448.0
    acc = np.array([[1, 2], [3, 0]])
    o, _ = oracle.gdn_speculative(S0, q, kk, v, al, be, acc)
    o_rc, _, _ = oracle.gdn_speculative_readcopy(S0, q, kk, v, al, be, acc, 8, "fp8")
    np.testing.assert_array_equal(o_rc, o)


@pytest.mark.parametrize("fmt", ["fp8", "nvfp4"])
def test_gdn_spec_readcopy_first_round_error_is_bounded_by_the_copy_error(fmt):
    """Before any fold, draft tau's row r moves by at most
    gamma_tau ||row r of (copy - S0)||_2 ||scale q_tau||_2 (each transition
    has spectral norm alpha for unit keys and beta in [0, 1])."""
    rng = np.random.default_rng(93)
    R, T, B = 1, 4, 2
    S0, q, kk, v, al, be = _gdn_rounds(rng, R, T, B, 2, 32, 128)
    scale = 0.7
    acc = np.zeros((R, B), np.int64)
    o, _ = oracle.gdn_speculative(S0, q, kk, v, al, be, acc, scale=scale)
    o_rc, _, _ = oracle.gdn_speculative_readcopy(S0, q, kk, v, al, be, acc, 16, fmt, scale=scale)
    halves = S0.reshape(-1, 64, 32).astype(np.float32)
    if fmt == "fp8":
        copy = oracle.dequant_fp8(*oracle.quant_fp8(halves))
    else:
        copy = oracle.dequant_nvfp4(*oracle.quant_nvfp4(halves))
    dS = np.linalg.norm(copy.reshape(S0.shape) - S0, axis=-1)            # [B][H][DV]
    gam = np.cumprod(al[0], axis=0)                                       # [T][B][H]
    bound = gam[..., None] * dS[None] * scale * np.linalg.norm(q[0], axis=-1)[..., None]
    err = np.abs(o_rc[0] - o[0])
    assert np.all(err <= bound * (1 + 1e-9) + 1e-15)
    assert err.max() > 0

"""The chunked SSD decomposition equals the sequential selective recurrence.

soft186.com, "Mamba选择性状态空间机制", section "状态空间对偶性算法突破": Mamba-2
computes the scan as a block decomposition of its semiseparable matrix. Read
with a scalar decay a per head, dt shared by the head's channels and B, C shared
by the heads, a chunk of Q steps contributes
    y_t = sum_{s<=t} (C_t . B_s) exp(cum_t - cum_s) dt_s x_s + exp(cum_t) C_t S + D x_t
    S  <- exp(cum_last) S + sum_s B_s (x_s exp(cum_last - cum_s) dt_s)
with cum the running sum of dt a inside the chunk and S the (N x P) state
entering it. This file writes that decomposition out in fp64 numpy for any Q
and checks it against the fp64 scan oracle on the same numbers: the GPU SSD
kernels compute this decomposition, so their agreement with the oracle rests
on this identity. CPU only."""
import numpy as np
import pytest

import oracle


def _softplus(x):
    return np.where(x > 0, x + np.log1p(np.exp(-x)), np.log1p(np.exp(x)))


def _chunked_ssd(x, dt, a, B, C, D, S0, Q):
    """One (batch, head): x (L, P), dt (L,) after softplus, a scalar, B, C (L, N),
    D scalar, S0 (N, P). Returns y (L, P) and the final state (N, P)."""
    L = x.shape[0]
    S = S0.copy()
    y = np.empty_like(x)
    for l0 in range(0, L, Q):
        sl = slice(l0, min(l0 + Q, L))
        xc, dc, Bc, Cc = x[sl], dt[sl], B[sl], C[sl]
        cum = np.cumsum(dc * a)
        q = len(dc)
        causal = np.tril(np.ones((q, q), dtype=bool))
        M = (Cc @ Bc.T) * np.exp(cum[:, None] - cum[None, :]) * dc[None, :]
        M = np.where(causal, M, 0.0)
        y[sl] = M @ xc + np.exp(cum)[:, None] * (Cc @ S) + D * xc
        S = np.exp(cum[-1]) * S + Bc.T @ (xc * (np.exp(cum[-1] - cum) * dc)[:, None])
    return y, S


@pytest.mark.parametrize("Q", [1, 3, 16, 64])
@pytest.mark.parametrize("with_h0", [False, True])
def test_chunked_decomposition_equals_scan_oracle(Q, with_h0):
    g = np.random.default_rng(300 + Q)
    batch, L, H, P, N = 2, 64, 3, 4, 8
    x = g.standard_normal((batch, L, H, P)).astype(np.float32)
    dt_raw = (g.standard_normal((batch, L, H)) * 0.5 - 1.0).astype(np.float32)
    B = (g.standard_normal((batch, L, N)) * 0.3).astype(np.float32)
    C = (g.standard_normal((batch, L, N)) * 0.3).astype(np.float32)
    A = -g.uniform(0.5, 4.0, H).astype(np.float32)
    D = g.standard_normal(H).astype(np.float32)
    bias = g.uniform(-2.0, 0.0, H).astype(np.float32)
    h0 = g.standard_normal((batch, H, P, N)).astype(np.float32)

    # the oracle: a selective scan over channels d = h * P + p
    u = np.ascontiguousarray(x.transpose(0, 2, 3, 1).reshape(batch, H * P, L))
    delta = np.ascontiguousarray(np.repeat(dt_raw.transpose(0, 2, 1), P, axis=1))
    A_full = np.repeat(A, P)[:, None].repeat(N, axis=1).astype(np.float32)
    y_ref, h_ref = oracle.scan_fwd(
        u, delta, A_full, np.ascontiguousarray(B.transpose(0, 2, 1)),
        np.ascontiguousarray(C.transpose(0, 2, 1)), D=np.repeat(D, P),
        delta_bias=np.repeat(bias, P), z=None,
        h0=h0.reshape(batch, H * P, N).astype(np.float64) if with_h0 else None)
    y_ref = y_ref.reshape(batch, H, P, L)
    h_ref = h_ref.reshape(batch, H, P, N)

    for b in range(batch):
        for h in range(H):
            dt = _softplus(dt_raw[b, :, h].astype(np.float64) + float(bias[h]))
            S0 = h0[b, h].T.astype(np.float64) if with_h0 else np.zeros((N, P))
            y, S = _chunked_ssd(x[b, :, h].astype(np.float64), dt, float(A[h]),
                                B[b].astype(np.float64), C[b].astype(np.float64),
                                float(D[h]), S0, Q)
            scale = np.max(np.abs(y_ref[b, h]))
            assert np.max(np.abs(y.T - y_ref[b, h])) <= 1e-11 * scale, (b, h)
            assert np.max(np.abs(S.T - h_ref[b, h])) <= 1e-11 * np.max(np.abs(h_ref[b, h]))


def test_decomposition_catches_a_missing_decay():
    """The comparison is sharp: dropping the carried state's decay breaks it."""
    g = np.random.default_rng(310)
    L, P, N = 32, 2, 4
    x = g.standard_normal((L, P))
    dt = _softplus(g.standard_normal(L) * 0.5 - 1.0)
    B, C = g.standard_normal((L, N)) * 0.3, g.standard_normal((L, N)) * 0.3
    S0 = g.standard_normal((N, P))
    y_whole, _ = _chunked_ssd(x, dt, -1.5, B, C, 0.3, S0, L)
    y_chunks, _ = _chunked_ssd(x, dt, -1.5, B, C, 0.3, S0, 8)
    assert np.max(np.abs(y_whole - y_chunks)) <= 1e-12 * np.max(np.abs(y_whole))

    def no_decay(x, dt, a, B, C, D, S, Q):
        y = np.empty_like(x)
        for l0 in range(0, len(dt), Q):
            sl = slice(l0, l0 + Q)
            cum = np.cumsum(dt[sl] * a)
            M = np.where(np.tril(np.ones((Q, Q), dtype=bool)),
                         (C[sl] @ B[sl].T) * np.exp(cum[:, None] - cum[None, :]) * dt[sl][None, :], 0)
            y[sl] = M @ x[sl] + np.exp(cum)[:, None] * (C[sl] @ S) + D * x[sl]
            S = S + B[sl].T @ (x[sl] * (np.exp(cum[-1] - cum) * dt[sl])[:, None])  # decay dropped
        return y
    y_bad = no_decay(x, dt, -1.5, B, C, 0.3, S0, 8)
    assert np.max(np.abs(y_bad - y_whole)) > 1e-3 * np.max(np.abs(y_whole))

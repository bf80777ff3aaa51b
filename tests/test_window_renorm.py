"""The windowed state rescale of the head-gated (retention) chunk kernel, restated
in fp64 and checked against the per-token recurrence S_t = gamma S_{t-1} + k_t v_t^T,
o_t = q_t^T S_t (the recurrent form of retention).

Inside a window of R chunks, m chunks in, the kernel keeps A = S / gamma^(C m) in
its accumulator: q rows carry gamma^(t+1) gamma^(C m), k rows gamma^-(s+1)
gamma^-(C m), and the accumulator is multiplied by gamma^(c + C m) only at a
window's last chunk (c = that chunk's length); the final state takes the same
factor. R = floor(40 / (C |ln gamma|)) in the kernel (C = 64); here C = 8 and
the bound is scaled so that windows of several chunks occur.
"""
import numpy as np
import pytest


def _windowed(q, k, v, gamma, C, bound):
    L, d = q.shape
    lg = np.log(gamma)
    rl = -C * lg
    R = max(1, int(min(bound / rl, 2 ** 20))) if rl > 0 else 2 ** 20
    N = (L + C - 1) // C
    A = np.zeros((d, v.shape[1]))
    out = np.zeros((L, v.shape[1]))
    m = 0
    for n in range(N):
        t0 = n * C
        c = min(C, L - t0)
        m = n % R
        fq = gamma ** (np.arange(c) + 1.0) * np.exp(C * m * lg)
        fk = gamma ** -(np.arange(c) + 1.0) * np.exp(-C * m * lg)
        qt, kt = q[t0:t0 + c] * fq[:, None], k[t0:t0 + c] * fk[:, None]
        out[t0:t0 + c] = np.tril(qt @ kt.T) @ v[t0:t0 + c] + qt @ A
        A = A + kt.T @ v[t0:t0 + c]
        if n < N - 1 and m == R - 1:
            A = np.exp((c + C * m) * lg) * A
    c_last = L - (N - 1) * C
    return out, np.exp((c_last + C * m) * lg) * A, R


@pytest.mark.parametrize("gamma", [0.5, 0.9, 0.99, 1.0])
@pytest.mark.parametrize("L", [1, 7, 8, 37, 70])
def test_windowed_rescale_equals_recurrence(gamma, L):
    rng = np.random.default_rng(L)
    q, k, v = rng.standard_normal((3, L, 4))
    S = np.zeros((4, 4))
    ref = np.zeros((L, 4))
    for t in range(L):
        S = gamma * S + np.outer(k[t], v[t])
        ref[t] = q[t] @ S
    out, S_end, R = _windowed(q, k, v, gamma, C=8, bound=3.0)
    if 0.85 < gamma < 1.0:
        assert R > 1  # the case the window exists for
    assert np.abs(out - ref).max() <= 1e-12 * np.abs(ref).max()
    assert np.abs(S_end - S).max() <= 1e-12 * np.abs(S).max()

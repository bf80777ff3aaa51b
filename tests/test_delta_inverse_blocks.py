"""The blocked triangular inverse of the chunked delta-rule kernel, restated in
fp64 with the kernel's thread mapping and checked against a library inverse.

Inside a chunk of 64 tokens the kernel needs T = (I + A)^-1 diag(beta), with
A[t, s] = beta_t k_t . k_s for s < t (the pseudo-values' unit lower-triangular
system). 128 solver threads form L^-1 by 16 x 16 blocks in place over A:
  1. threads s < 64 take column s % 16 of diagonal block s / 16 and solve it
     right-looking: once x_r is final, x_j -= A[j, r] x_r for every later j;
  2. block rows I = 1, 2, 3 in turn: thread s makes the outputs u < 2I with
     block J = u / 2, row s / 16 + 8 (u % 2) and column s % 16, first
     Z_J = sum_{J <= K < I} A_IK X_KJ (kept aside), then X_IJ = -X_II Z_J;
  3. T goes out by 16-byte groups: thread s takes row s / 2 and the groups
     (s % 2) + 2 u, u < 4, that lie in blocks at or left of the diagonal.
A mistake in any of the index maps (a transposed block, a missed row, a group
written twice or never) changes the inverse, so the restatement is checked
element by element against numpy's inverse, on inputs shaped like the delta
workload's (unit keys, beta = sigmoid of a normal draw).
"""
import numpy as np
import pytest


def _a_matrix(rng):
    k = rng.standard_normal((64, 128))
    k /= np.linalg.norm(k, axis=1, keepdims=True)
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal(64)))
    return np.tril(beta[:, None] * (k @ k.T), -1), beta


def _kernel_inverse(A):
    M = A.copy()  # the kernel's fp32 [64][68] array, here fp64 [64][64]
    # 1. diagonal blocks: every thread reads its block before any block is written
    cols = {}
    for s in range(64):
        b, c = s >> 4, s & 15
        o = 16 * b
        x = np.array([1.0 if r == c else 0.0 for r in range(16)])
        for r in range(16):
            for j in range(r + 1, 16):
                x[j] -= M[o + j, o + r] * x[r]
        cols[s] = x
    for s, x in cols.items():
        b, c = s >> 4, s & 15
        M[16 * b:16 * b + 16, 16 * b + c] = x
    # 2. block rows 1..3, each in two barrier-separated steps
    for I in (1, 2, 3):
        Z = {}
        for s in range(128):
            r0, col = s >> 4, s & 15
            for u in range(2 * I):
                J, r = u >> 1, r0 + 8 * (u & 1)
                Z[(J, r, col)] = sum(M[16 * I + r, kk] * M[kk, 16 * J + col] for kk in range(16 * J, 16 * I))
        for s in range(128):
            r0, col = s >> 4, s & 15
            for u in range(2 * I):
                J, r = u >> 1, r0 + 8 * (u & 1)
                M[16 * I + r, 16 * J + col] = -sum(M[16 * I + r, 16 * I + kk] * Z[(J, kk, col)] for kk in range(16))
    return M


def _kernel_t(M, beta):
    T = np.zeros((64, 64))
    written = np.zeros((64, 8), int)
    for s in range(128):
        i, lastg = s >> 1, 2 * ((s >> 1) >> 4) + 1
        for u in range(4):
            c8 = (s & 1) + 2 * u
            if c8 <= lastg:
                T[i, 8 * c8:8 * c8 + 8] = M[i, 8 * c8:8 * c8 + 8] * beta[8 * c8:8 * c8 + 8]
                written[i, c8] += 1
    return T, written


@pytest.mark.parametrize("seed", range(4))
def test_blocked_inverse_matches_library_inverse(seed):
    A, beta = _a_matrix(np.random.default_rng(seed))
    X = _kernel_inverse(A)
    ref = np.linalg.inv(np.eye(64) + A)
    low = np.kron(np.tril(np.ones((4, 4))), np.ones((16, 16))).astype(bool)  # blocks at or left of the diagonal
    assert np.max(np.abs(np.where(low, X, 0.0) - ref)) < 1e-12 * max(1.0, np.max(np.abs(ref)))


@pytest.mark.parametrize("seed", range(2))
def test_t_groups_cover_the_lower_blocks_once(seed):
    A, beta = _a_matrix(np.random.default_rng(10 + seed))
    T, written = _kernel_t(_kernel_inverse(A), beta)
    ref = np.linalg.inv(np.eye(64) + A) * beta[None, :]
    assert np.max(np.abs(T - ref)) < 1e-12 * max(1.0, np.max(np.abs(ref)))
    # each 16-byte group of a block at or left of the diagonal exactly once, none to its right
    for i in range(64):
        for c8 in range(8):
            assert written[i, c8] == (1 if c8 // 2 <= i // 16 else 0), (i, c8)

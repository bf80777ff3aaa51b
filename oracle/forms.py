"""Independent numpy restatements of the same function, in fp64, one sequence
at a time (q, k: [L, dk]; v: [L, dv]).

TEST INFRASTRUCTURE ONLY (see the package docstring). They pin the C oracle:
each form is a different formula for the same outputs, written from the pages:

* ``recurrent``  -- the running-state loop (linear_sparse_attention.py,
  linear_attn_recurrent; learnllm m22 "The Math: Linear Attention"); a numpy
  twin of the C definition for tiny cases.
* ``parallel``   -- the masked matmul (QK^T * D) V with D the lower-triangular
  decay matrix (learnllm m22 "Code: The Two Faces", "The Three Faces of
  Retention"), rows divided by their sums when normalised.
* ``brute_force`` -- the explicit double sum over j <= t and channels, with
  the decay written as a product of per-step gates; pure Python loops.
* ``chunkwise``  -- intra-chunk parallel term plus cross-chunk carried state R
  (linear_sparse_attention.py, linear_attn_chunkwise; learnllm m22 "The Three
  Faces of Retention"), with the decay factors written as explicit products
  of per-step gates, so gamma^(t-s), gamma^(t+1), gamma^B, gamma^(B-1-s) and
  their per-channel generalisation all come from one rule.

``a`` is the per-step, per-key-channel gate A_t as an [L, dk] array (ones for
linear attention, gamma for retention, alpha_t for the gated form).
"""
import numpy as np


def phi(x, elu1):
    """elu(x)+1 (x+1 for x>0, e^x otherwise) or the identity."""
    x = np.asarray(x, dtype=np.float64)
    if not elu1:
        return x.copy()
    return np.where(x > 0, x + 1.0, np.exp(np.minimum(x, 0.0)))


def log_sigmoid(x):
    x = np.asarray(x, dtype=np.float64)
    return np.where(x >= 0, -np.log1p(np.exp(-np.abs(x))), x - np.log1p(np.exp(-np.abs(x))))


def gate_channel(g):
    """alpha = exp(logsigmoid(g) / 16), elementwise."""
    return np.exp(log_sigmoid(g) / 16.0)


def step_gates(L, dk, gamma=None, g=None):
    """The per-step gate A_t as an [L, dk] array."""
    if g is not None:
        return gate_channel(np.asarray(g, dtype=np.float64).reshape(L, dk))
    if gamma is not None:
        return np.full((L, dk), float(gamma))
    return np.ones((L, dk))


def recurrent(q, k, v, a, elu1=False, normalize=False, S0=None, z0=None):
    """Returns (out [L,dv], S [dk,dv], z [dk])."""
    q = phi(q, elu1)
    k = phi(k, elu1)
    v = np.asarray(v, dtype=np.float64)
    L, dk = q.shape
    dv = v.shape[1]
    S = np.zeros((dk, dv)) if S0 is None else np.array(S0, dtype=np.float64)
    z = np.zeros(dk) if z0 is None else np.array(z0, dtype=np.float64)
    out = np.zeros((L, dv))
    for t in range(L):
        S = a[t][:, None] * S + np.outer(k[t], v[t])
        z = a[t] * z + k[t]
        num = q[t] @ S
        out[t] = num / (q[t] @ z) if normalize else num
    return out, S, z


def decay_tensor(a):
    """D[i, j, d] = prod_{r=j+1..i} a[r, d] for j <= i, else 0 (an empty
    product is 1, so the diagonal is 1 even when a gate is 0)."""
    L, dk = a.shape
    D = np.zeros((L, L, dk))
    for j in range(L):
        p = np.ones(dk)
        D[j, j] = p
        for i in range(j + 1, L):
            p = p * a[i]
            D[i, j] = p
    return D


def parallel(q, k, v, a, elu1=False, normalize=False):
    """(Q K^T (.) D) V with the per-channel decay inside the score."""
    qf = phi(q, elu1)
    kf = phi(k, elu1)
    v = np.asarray(v, dtype=np.float64)
    D = decay_tensor(a)
    A = np.einsum("id,ijd,jd->ij", qf, D, kf)
    num = A @ v
    if normalize:
        return num / A.sum(axis=1, keepdims=True)
    return num


def brute_force(q, k, v, a, elu1=False, normalize=False):
    """o_t = sum_{j<=t} sum_i qf_t[i] (prod_{r=j+1..t} a_r[i]) kf_j[i] v_j."""
    qf = phi(q, elu1)
    kf = phi(k, elu1)
    v = np.asarray(v, dtype=np.float64)
    L, dk = qf.shape
    dv = v.shape[1]
    out = np.zeros((L, dv))
    for t in range(L):
        num = [0.0] * dv
        den = 0.0
        for j in range(t + 1):
            w = 0.0
            for i in range(dk):
                p = 1.0
                for r in range(j + 1, t + 1):
                    p *= float(a[r, i])
                w += float(qf[t, i]) * p * float(kf[j, i])
            for c in range(dv):
                num[c] += w * float(v[j, c])
            den += w
        for c in range(dv):
            out[t, c] = num[c] / den if normalize else num[c]
    return out


def chunkwise(q, k, v, a, C, elu1=False, normalize=False):
    """Chunks of C tokens (the last one ragged). Per chunk, local index t:
    intra_t = sum_{s<=t} (decay s->t) (q_t . k_s) v_s,
    cross_t = q_t (decay chunk start->t) R,
    R <- (decay over the whole chunk) R + sum_s (decay s->chunk end) k_s v_s^T.
    Returns (out, R, zR)."""
    qf = phi(q, elu1)
    kf = phi(k, elu1)
    v = np.asarray(v, dtype=np.float64)
    L, dk = qf.shape
    dv = v.shape[1]
    R = np.zeros((dk, dv))
    zR = np.zeros(dk)
    out = np.zeros((L, dv))
    for s0 in range(0, L, C):
        e = min(s0 + C, L)
        c = e - s0
        ac = a[s0:e]
        # cum[t] = prod_{r=0..t} ac[r]  (decay from the chunk start through t)
        cum = np.cumprod(ac, axis=0)
        for t in range(c):
            num = (qf[s0 + t] * cum[t]) @ R
            den = (qf[s0 + t] * cum[t]) @ zR
            for s in range(t + 1):
                w = np.prod(ac[s + 1:t + 1], axis=0) if t > s else np.ones(dk)
                sc = np.sum(qf[s0 + t] * w * kf[s0 + s])
                num = num + sc * v[s0 + s]
                den = den + sc
            out[s0 + t] = num / den if normalize else num
        newR = cum[c - 1][:, None] * R
        newz = cum[c - 1] * zR
        for s in range(c):
            w = np.prod(ac[s + 1:c], axis=0) if s < c - 1 else np.ones(dk)
            newR = newR + np.outer(w * kf[s0 + s], v[s0 + s])
            newz = newz + w * kf[s0 + s]
        R, zR = newR, newz
    return out, R, zR


def delta_recurrent(K, V, beta, Q=None, use_delta=True, S0=None):
    """The delta rule as matrix products, one token at a time
    (linear_sparse_attention.py, "delta_rule_recurrent"): S is d_v x d_k,
        S <- S (I - beta_t k_t k_t^T)   (skipped when use_delta is False)
        S <- S + beta_t v_t k_t^T
    and, with queries, out_t = S q_t after the update. K, Q: [L, dk]; V: [L, dv];
    beta: [L]. Returns (states [L, dv, dk], out [L, dv] or None)."""
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    beta = np.asarray(beta, dtype=np.float64)
    L, dk = K.shape
    dv = V.shape[1]
    S = np.zeros((dv, dk)) if S0 is None else np.array(S0, dtype=np.float64).reshape(dv, dk)
    eye = np.eye(dk)
    states = np.zeros((L, dv, dk))
    out = None if Q is None else np.zeros((L, dv))
    for t in range(L):
        k = K[t]
        if use_delta:
            S = S @ (eye - beta[t] * np.outer(k, k))
        S = S + beta[t] * np.outer(V[t], k)
        states[t] = S
        if Q is not None:
            out[t] = S @ np.asarray(Q[t], dtype=np.float64)
    return states, out


def delta_chunkwise(K, V, beta, Q, C, S0=None):
    """The delta rule over chunks of C tokens (the last one ragged), the form a
    chunked kernel computes. No page gives it; it follows from the recurrence.
    Write each step as S_t = S_{t-1} + u_t k_t^T with the pseudo-value
    u_t = beta_t (v_t - S_{t-1} k_t). Inside a chunk starting from S0,
    S_{t-1} = S0 + sum_{s<t} u_s k_s^T, so
        u_t + beta_t sum_{s<t} (k_t . k_s) u_s = beta_t (v_t - S0 k_t),
    a unit lower-triangular system: (I + A) Ut = diag(beta) (V - K S0^T) with
    A[t, s] = beta_t k_t . k_s for s < t. With T = (I + A)^-1 diag(beta),
    W = T K and U = T V (both free of the state):
        Ut  = U - W S0^T
        out = Q S0^T + tril(Q K^T) Ut        (diagonal included: read after the update)
        S   = S0 + Ut^T K
    K, Q: [L, dk]; V: [L, dv]; beta: [L]. Returns (out [L, dv], S [dv, dk])."""
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    Q = np.asarray(Q, dtype=np.float64)
    beta = np.asarray(beta, dtype=np.float64)
    L, dk = K.shape
    dv = V.shape[1]
    S = np.zeros((dv, dk)) if S0 is None else np.array(S0, dtype=np.float64).reshape(dv, dk)
    out = np.zeros((L, dv))
    for c0 in range(0, L, C):
        k, v, q, b = K[c0:c0 + C], V[c0:c0 + C], Q[c0:c0 + C], beta[c0:c0 + C]
        n = k.shape[0]
        A = np.tril(b[:, None] * (k @ k.T), -1)
        T = np.linalg.solve(np.eye(n) + A, np.diag(b))
        W, U = T @ k, T @ v
        Ut = U - W @ S.T
        out[c0:c0 + n] = q @ S.T + np.tril(q @ k.T) @ Ut
        S = S + Ut.T @ k
    return out, S

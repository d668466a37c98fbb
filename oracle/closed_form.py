"""The closed form of the tree recurrence (Bole's Theorem 1 as the canopy page
states it), with every solver the page names.

canopy page, "The tree closed form", for one stream and one head, in the
library's (dv, dk) orientation:
    l_i    = log alpha_i + l_parent(i)                 (root's parent: 0)
    P_i    = exp(l_i)
    Gam_ij = exp(l_i - l_j)        if j in path(i), else 0
    G_ij   = beta_i Gam_ij k_i.k_j  if j in A(i),   else 0   (strictly lower)
    R_i    = beta_i (v_i - P_i S0 k_i)
    (I + G) U = R
    C_ij   = Gam_ij q_i.k_j         if j in path(i), else 0
    O      = diag(P) Q S0^T + C U
Ratios are taken in log space only ("Hard constraints", log-space gates); the
naive-ratio twin below exists solely for the stability pin.

Solvers for (I + G) U = R (page: "The tree closed form" and "Design
decisions"):
  dense     a library LU solve of I + G
  fwdsub    row-by-row forward substitution
  blocked   forward substitution by blocks of 64 nodes:
            (I + G_bb) U_b = R_b - sum_{c<b} G_bc U_c
  neumann   U = sum_{m=0..d} (-G)^m R, as Z <- -G Z, U <- U + Z for d rounds
  squaring  U = (I - G)(I + G^2)(I + G^4)... R with ceil(log2(d+1)) factors
  level     per depth level L in order: U_L = R_L - G_{L,:} U
  split     the split design: W = (I + G)^-1 formed once (row i: W_i = e_i -
            G_i W, rows in order), then U = W R
"""

from __future__ import annotations

import math

import numpy as np

from .tree import cumulative_log_gate, depths, strict_ancestor_mask, validate_parent


def build_G_C(parent, q, k, alpha, beta, dtype=np.float64):
    """G, C, l and P for one stream and one head, in the given float dtype.

    q, k [T, dk]; alpha, beta [T]."""
    p = validate_parent(parent)
    T = p.size
    Ms = strict_ancestor_mask(p)
    Mp = Ms | np.eye(T, dtype=bool)
    if dtype == np.float64:
        l = cumulative_log_gate(p, alpha)
    else:
        la = np.log(np.asarray(alpha, dtype))
        l = np.zeros(T, dtype)
        for i in range(T):
            l[i] = la[i] + (l[p[i]] if p[i] >= 0 else dtype(0))
    q = np.asarray(q, dtype)
    k = np.asarray(k, dtype)
    b = np.asarray(beta, dtype)
    diff = np.where(Mp, l[:, None] - l[None, :], dtype(0))
    Gam = np.where(Mp, np.exp(diff), dtype(0)).astype(dtype)
    KK = k @ k.T
    QK = q @ k.T
    G = np.where(Ms, b[:, None] * Gam * KK, dtype(0)).astype(dtype)
    C = np.where(Mp, Gam * QK, dtype(0)).astype(dtype)
    return G, C, l, np.exp(l).astype(dtype)


def naive_ratio_gamma(parent, alpha, flush_subnormals: bool):
    """Gam from cumulative products P and the naive ratio P_i / P_j, in fp32.

    The form the page warns against ("What might go wrong" and "Verification
    of the formulas"); with flush_subnormals the products are flushed to zero
    below the smallest normal fp32, as flush-to-zero arithmetic does."""
    p = validate_parent(parent)
    T = p.size
    a = np.asarray(alpha, np.float32)
    tiny = np.finfo(np.float32).tiny
    P = np.zeros(T, np.float32)
    for i in range(T):
        P[i] = a[i] * (P[p[i]] if p[i] >= 0 else np.float32(1))
        if flush_subnormals and abs(P[i]) < tiny:
            P[i] = np.float32(0)
    Mp = strict_ancestor_mask(p) | np.eye(T, dtype=bool)
    with np.errstate(divide="ignore", invalid="ignore", over="ignore"):
        ratio = P[:, None] / P[None, :]
    return np.where(Mp, ratio, np.float32(0)), Mp


# ----------------------------------------------------------------------------
# solvers: (I + G) U = R, G strictly lower triangular in a topological order

def solve_dense(G, R, parent=None):
    return np.linalg.solve(np.eye(G.shape[0], dtype=G.dtype) + G, R)


def solve_fwdsub(G, R, parent=None):
    U = np.zeros_like(R)
    for i in range(G.shape[0]):
        U[i] = R[i] - G[i, :i] @ U[:i]
    return U


def solve_blocked(G, R, parent=None, block: int = 64):
    T = G.shape[0]
    U = np.zeros_like(R)
    for s in range(0, T, block):
        e = min(T, s + block)
        Rb = R[s:e] - G[s:e, :s] @ U[:s]
        Gb = G[s:e, s:e]
        for r in range(e - s):
            U[s + r] = Rb[r] - Gb[r, :r] @ U[s:s + r]
    return U


def solve_neumann(G, R, parent):
    d = int(depths(parent).max())
    Z = R.copy()
    U = R.copy()
    for _ in range(d):
        Z = -(G @ Z)
        U = U + Z
    return U


def solve_squaring(G, R, parent):
    d = int(depths(parent).max())
    nfac = math.ceil(math.log2(d + 1)) if d > 0 else 0
    if nfac == 0:
        return R.copy()
    U = R - G @ R                       # factor (I - G)
    Gp = G
    for _ in range(1, nfac):
        Gp = Gp @ Gp                    # G^(2^m)
        U = U + Gp @ U                  # factor (I + G^(2^m))
    return U


def solve_level(G, R, parent):
    dep = depths(parent)
    U = np.zeros_like(R)
    for L in range(int(dep.max()) + 1):
        rows = np.nonzero(dep == L)[0]
        U[rows] = R[rows] - G[rows, :] @ U
    return U


def solve_split(G, R, parent=None):
    T = G.shape[0]
    W = np.zeros_like(G)
    for i in range(T):
        W[i] = -(G[i, :i] @ W[:i])
        W[i, i] += 1.0
    return W @ R


SOLVERS = {
    "dense": solve_dense,
    "fwdsub": solve_fwdsub,
    "blocked": solve_blocked,
    "neumann": solve_neumann,
    "squaring": solve_squaring,
    "level": solve_level,
    "split": solve_split,
}


def closed_form(parent, q, k, v, alpha, beta, S0, solver: str = "fwdsub",
                dtype=np.float64):
    """One stream, one head.  q, k [T, dk]; v [T, dv]; alpha, beta [T];
    S0 [dv, dk].  Returns (O [T, dv], U [T, dv], l [T])."""
    G, C, l, P = build_G_C(parent, q, k, alpha, beta, dtype)
    q = np.asarray(q, dtype)
    k = np.asarray(k, dtype)
    v = np.asarray(v, dtype)
    b = np.asarray(beta, dtype)
    S0 = np.asarray(S0, dtype)
    R = b[:, None] * (v - P[:, None] * (k @ S0.T))
    U = SOLVERS[solver](G, R, np.asarray(parent))
    O = P[:, None] * (q @ S0.T) + C @ U
    return O, U, l


def closed_form_batch(parent, q, k, v, alpha, beta, S0, solver: str = "fwdsub",
                      dtype=np.float64):
    """B streams, H heads.  Returns O, U [B, T, H, dv] and l [B, T, H]."""
    B, T, H, _ = np.shape(q)
    dv = np.shape(v)[-1]
    O = np.zeros((B, T, H, dv), dtype)
    U = np.zeros((B, T, H, dv), dtype)
    L = np.zeros((B, T, H), dtype)
    for b in range(B):
        for h in range(H):
            O[b, :, h], U[b, :, h], L[b, :, h] = closed_form(
                parent[b], q[b, :, h], k[b, :, h], v[b, :, h], alpha[b, :, h],
                beta[b, :, h], S0[b, h], solver, dtype)
    return O, U, L


def closed_form_heads(parent, q, k, v, alpha, beta, S0, scale: float = 1.0):
    """The same closed form for one stream and all heads at once (fp64), with
    the forward-substitution solve; the head axis is carried through every
    step, nothing else changes.  q, k [T, H, dk] (key heads); v [T, HV, dv];
    alpha, beta [T, HV]; S0 [HV, dv, dk]; value head j reads key head
    j // (HV / H) and q is multiplied by ``scale``, as in ``replay``.
    Returns (O [T, HV, dv], U [T, HV, dv], l [T, HV])."""
    from .replay import value_heads
    p = validate_parent(parent)
    T = p.size
    v = np.asarray(v, np.float64).transpose(1, 0, 2)              # [HV, T, dv]
    HV = v.shape[0]
    q = (value_heads(q, HV) * float(scale)).transpose(1, 0, 2)    # [HV, T, dk]
    k = value_heads(k, HV).transpose(1, 0, 2)
    a = np.asarray(alpha, np.float64)
    b = np.asarray(beta, np.float64).T                            # [HV, T]
    S0 = np.asarray(S0, np.float64)
    Ms = strict_ancestor_mask(p)
    Mp = Ms | np.eye(T, dtype=bool)
    l = cumulative_log_gate(p, a)                                 # [T, HV]
    lt = l.T
    P = np.exp(lt)                                                # [HV, T]
    diff = np.where(Mp[None], lt[:, :, None] - lt[:, None, :], 0.0)
    Gam = np.where(Mp[None], np.exp(diff), 0.0)                   # [HV, T, T]
    KT = k.transpose(0, 2, 1)
    G = np.where(Ms[None], b[:, :, None] * Gam * (k @ KT), 0.0)
    C = np.where(Mp[None], Gam * (q @ KT), 0.0)
    S0T = S0.transpose(0, 2, 1)
    R = b[:, :, None] * (v - P[:, :, None] * (k @ S0T))           # [HV, T, dv]
    U = np.zeros_like(R)
    for i in range(T):
        U[:, i] = R[:, i] - (G[:, i, None, :i] @ U[:, :i])[:, 0]
    O = P[:, :, None] * (q @ S0T) + C @ U
    return O.transpose(1, 0, 2), U.transpose(1, 0, 2), l

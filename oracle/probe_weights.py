"""LoKA Probe: online learning of a layer's weight distribution, and sampling.

TEST INFRASTRUCTURE ONLY (see the package docstring).

LoKA page, section III-A 1 "Online Distribution Learning", paragraph
"Optimized Weight Distribution Modeling", and "Sampling learned
distributions" (b).  A weight matrix W [R, C] (the page's M x N) has no
independent dimension, so it is modeled as matrix-normal,
W ~ MN(M, U, V): mean M [R, C], row covariance U [R, R], column covariance
V [C, C], i.e. vec(W) ~ N(vec(M), V (x) U).  (U, V) are tracked online by a
Kronecker-factor ("flip-flop") update smoothed by an exponential moving
average, with linear solves against regularized Cholesky factors instead of
inverses.  One update with the current (M, U, V) and a new W:

  Wc    = W - M
  L_V L_V^T = V + eps_V I,   W_V = Wc L_V^{-T},   U' = W_V W_V^T / C   [R, R]
  L_U L_U^T = U + eps_U I,   W_U = L_U^{-1} Wc,   V' = W_U^T W_U / R   [C, C]
  U'' = m U + (1 - m) U',    V'' = m V + (1 - m) V'
  U   = (U'' + U''^T) / 2 + eps_U I,   V = (V'' + V''^T) / 2 + eps_V I
  s   = trace(U) / R,   U <- U / s,   V <- s V      (V (x) U is unchanged)

Sampling: Z ~ N(0, I) [R, C], W' = M + L_U Z L_V^T with L_U L_U^T = U + eps_U I
and L_V L_V^T = V + eps_V I.

Readings (the page leaves these open):
  * Both per-update estimates use the (U, V) held before the update: the
    page writes the two solves side by side and the averages after them.
  * eps_U = eps_rel * trace(U) / R and eps_V = eps_rel * trace(V) / C, the
    page's "10^-6 x trace(U) / M" with its counterpart for V, each taken on
    the matrix it regularizes (for the jitter after the average: on the
    symmetrized average).
  * The mean M follows the same moving average, after the covariances (Wc
    uses the mean held before the update).  The first update starts the
    model: M = W, U = I, V = I.
  * The sampler's normals are the counter-based stream of probe_stats
    (Z[r, c] is normal r C + c of the seed).

Float64 throughout; numpy's Cholesky and triangular solves are the library
steps.
"""
from __future__ import annotations

import dataclasses

import numpy as np

from .probe_stats import normals


@dataclasses.dataclass
class WeightStats:
    n: int                  # updates merged
    M: np.ndarray           # [R, C]
    U: np.ndarray           # [R, R]
    V: np.ndarray           # [C, C]


def eps_of(A: np.ndarray, eps_rel: float) -> float:
    """The page's jitter: eps_rel * trace(A) / dim(A)."""
    return eps_rel * float(np.trace(A)) / A.shape[0]


def reg_cholesky(A: np.ndarray, eps_rel: float) -> np.ndarray:
    """Lower L with L L^T = A + eps I."""
    return np.linalg.cholesky(A + eps_of(A, eps_rel) * np.eye(A.shape[0]))


def forward_solve(L: np.ndarray, B: np.ndarray) -> np.ndarray:
    """X with L X = B for lower-triangular L (column by column, in order)."""
    n = L.shape[0]
    X = np.zeros_like(B, dtype=np.float64)
    for j in range(n):
        X[j] = (B[j] - L[j, :j] @ X[:j]) / L[j, j]
    return X


def weight_update(st: WeightStats | None, w, m: float, eps_rel: float) -> WeightStats:
    """One online update of the matrix-normal model with the weight w [R, C]."""
    W = np.asarray(w, dtype=np.float64)
    R, C = W.shape
    if st is None or st.n == 0:
        return WeightStats(1, W.copy(), np.eye(R), np.eye(C))
    Wc = W - st.M
    L_V = reg_cholesky(st.V, eps_rel)
    W_V = forward_solve(L_V, Wc.T).T          # Wc L_V^{-T}: row r solves L_V y = Wc[r]^T
    U1 = W_V @ W_V.T / C
    L_U = reg_cholesky(st.U, eps_rel)
    W_U = forward_solve(L_U, Wc)              # L_U^{-1} Wc: column c solves L_U z = Wc[:, c]
    V1 = W_U.T @ W_U / R
    U2 = m * st.U + (1.0 - m) * U1
    V2 = m * st.V + (1.0 - m) * V1
    Us = 0.5 * (U2 + U2.T)
    Vs = 0.5 * (V2 + V2.T)
    U = Us + eps_of(Us, eps_rel) * np.eye(R)
    V = Vs + eps_of(Vs, eps_rel) * np.eye(C)
    s = float(np.trace(U)) / R
    U = U / s
    V = V * s
    M = m * st.M + (1.0 - m) * W
    return WeightStats(st.n + 1, M, U, V)


def weight_sample(st: WeightStats, eps_rel: float, seed: int) -> tuple:
    """W' = M + L_U Z L_V^T; returns (Z, W') in float64."""
    R, C = st.M.shape
    Z = normals(seed, R * C).reshape(R, C)
    L_U = reg_cholesky(st.U, eps_rel)
    L_V = reg_cholesky(st.V, eps_rel)
    return Z, st.M + L_U @ Z @ L_V.T

"""LoKA Probe: online learning of a layer's input distribution, and sampling.

TEST INFRASTRUCTURE ONLY (see the package docstring).

LoKA page, section III-A 1 "Online Distribution Learning":
  * Activations are modeled per feature (the batch dimension is independent),
    by their mean and covariance, tracked in streaming form with a batched
    Welford / Chan update.  With the running summary (n_old, mu_old, S_old),
    S the unnormalized scatter matrix, and a batch X [B, K] of mean mu_b and
    scatter S_b = (X - mu_b)^T (X - mu_b):
        n_new  = n_old + B,   delta = mu_b - mu_old,
        mu_new = mu_old + (B / n_new) delta,
        S_new  = S_old + S_b + (n_old B / n_new) delta delta^T,
    and the unbiased covariance is S / (n - 1).
  * Sampling: T' = 1_B mu^T + Z L^T with Z ~ N(0, I_K) and L L^T = Sigma + eps I
    (the Cholesky factor of the regularized covariance).

Random normals.  The sampler draws its normals on the device; both sides
implement the same counter-based generator from its published definition:
SplitMix64 (the output function of Steele, Lea and Flood's SplittableRandom:
add the golden-ratio increment 0x9E3779B97F4A7C15, then the two
xor-shift-multiply rounds with 0xBF58476D1CE4E5B9 and 0x94D049BB133111EB and
shifts 30, 27, 31).  Random number i of a seed is the SplitMix64 output of
state seed + (i + 1) * 0x9E3779B97F4A7C15.  Normal pair j (elements 2j and
2j + 1) is Box-Muller on u1 = (r_{2j} >> 40 + 1) 2^-24 in (0, 1] and
u2 = (r_{2j+1} >> 40) 2^-24: z_{2j} = sqrt(-2 ln u1) cos(2 pi u2),
z_{2j+1} = sqrt(-2 ln u1) sin(2 pi u2).  Z[b, k] is normal b K + k.  Here in
float64; the device evaluates the same formula in float32.
"""
from __future__ import annotations

import numpy as np

GAMMA = np.uint64(0x9E3779B97F4A7C15)
MIX1 = np.uint64(0xBF58476D1CE4E5B9)
MIX2 = np.uint64(0x94D049BB133111EB)


def stats_update(n: int, mu: np.ndarray, S: np.ndarray, x) -> tuple:
    """One batched Chan update of (n, mu [K], S [K,K]) with the rows of x."""
    xf = np.asarray(x, dtype=np.float64)
    B = xf.shape[0]
    if B == 0:
        return n, mu.copy(), S.copy()
    mu_b = xf.mean(axis=0)
    xc = xf - mu_b[None, :]
    S_b = xc.T @ xc
    n_new = n + B
    delta = mu_b - mu
    mu_new = mu + (B / n_new) * delta
    S_new = S + S_b + (n * B / n_new) * np.outer(delta, delta)
    return n_new, mu_new, S_new


def covariance(n: int, S: np.ndarray) -> np.ndarray:
    """The unbiased covariance S / (n - 1) (n > 1)."""
    return S / (n - 1)


def cholesky_factor(n: int, S: np.ndarray, eps_rel: float) -> np.ndarray:
    """L with L L^T = S / (n - 1) + eps I, eps = eps_rel * trace(S / (n - 1)) / K."""
    sigma = covariance(n, S)
    K = sigma.shape[0]
    return np.linalg.cholesky(sigma + eps_rel * np.trace(sigma) / K * np.eye(K))


def splitmix64(seed: int, index: np.ndarray) -> np.ndarray:
    """Random numbers `index` (uint64 array) of the counter-based stream."""
    with np.errstate(over="ignore"):
        z = np.uint64(seed) + (index.astype(np.uint64) + np.uint64(1)) * GAMMA
        z = (z ^ (z >> np.uint64(30))) * MIX1
        z = (z ^ (z >> np.uint64(27))) * MIX2
        return z ^ (z >> np.uint64(31))


def normals(seed: int, count: int) -> np.ndarray:
    """The first `count` (even) normals of the seed's stream, float64."""
    assert count % 2 == 0
    r = splitmix64(seed, np.arange(count, dtype=np.uint64))
    top = (r >> np.uint64(40)).astype(np.float64)
    u1 = (top[0::2] + 1.0) * 2.0 ** -24
    u2 = top[1::2] * 2.0 ** -24
    rad = np.sqrt(-2.0 * np.log(u1))
    z = np.empty(count, dtype=np.float64)
    z[0::2] = rad * np.cos(2.0 * np.pi * u2)
    z[1::2] = rad * np.sin(2.0 * np.pi * u2)
    return z


def sample_inputs(mu, L, B: int, seed: int) -> tuple:
    """T' = 1 mu^T + Z L^T with the stream's normals; returns (Z, T') in
    float64 (mu [K], L [K, K] lower triangular)."""
    mu = np.asarray(mu, dtype=np.float64)
    L = np.asarray(L, dtype=np.float64)
    K = mu.shape[0]
    Z = normals(seed, B * K).reshape(B, K)
    return Z, mu[None, :] + Z @ L.T

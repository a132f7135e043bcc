"""Neumann power doubling vs the direct triangular solve, in fp32: a documented experiment.

PR #164 "Fused DeltaNet Direct-Solve Follow-Up" ("Why This Exists", "Implementation
Details") replaced a Neumann power-doubling solve of the chunk's (I + A) system by a direct
triangular solve, because forming full matrix powers amplified rounding error at realistic
gate values.  This study measures that on the CPU, for one 64-token chunk:

  * A_rs = beta_r exp(G_r - G_s) (k_r . k_s) for s < r (the chunk's strictly lower matrix);
  * the exact inverse (I + A)^-1 in fp64 (the oracle's forward substitution);
  * in fp32: forward substitution (what the kernels do), and Neumann power doubling
    (I - A)(I + A^2)(I + A^4)...(I + A^32) = sum_{k < 64} (-A)^k, exact in exact
    arithmetic because A^64 = 0;
  * the relative error of each in the chunk's U = (I + A)^-1 (diag(beta) V), the quantity the
    recurrence carries on.

Keys are made correlated (a shared direction with weight rho), since correlated keys and
weak decay are where the powers of A grow.  The direct solve stays at fp32 rounding
everywhere; Neumann doubling degrades by orders of magnitude as keys correlate and decay
weakens.  The solve the kernels use is the direct one; Neumann is not built.

Run with -s to print the table.
"""
import numpy as np
import pytest

import oracle

C, D = 64, 128


def _chunk(rng, rho, decay_scale, beta_mu):
    shared = rng.standard_normal(D)
    k = rho * shared + (1 - rho) * rng.standard_normal((C, D))
    k /= np.linalg.norm(k, axis=1, keepdims=True)
    beta = 1 / (1 + np.exp(-(beta_mu + rng.standard_normal(C))))
    g = -decay_scale * rng.uniform(0.0, 1.0, C)
    G = np.cumsum(g)
    A = np.tril(beta[:, None] * np.exp(G[:, None] - G[None, :]) * (k @ k.T), -1)
    v = rng.standard_normal((C, D))
    return A, beta, v


def _forward_subst_f32(A):
    n = A.shape[0]
    A = A.astype(np.float32)
    T = np.zeros((n, n), np.float32)
    for r in range(n):
        row = np.zeros(n, np.float32)
        row[r] = 1.0
        for s in range(r):
            row -= A[r, s] * T[s]
        T[r] = row
    return T


def _neumann_doubling_f32(A):
    n = A.shape[0]
    A = A.astype(np.float32)
    eye = np.eye(n, dtype=np.float32)
    T = eye - A
    P = A
    k = 2
    while k < n:
        P = P @ P                                   # A^k
        T = T @ (eye + P)
        k *= 2
    return T


def _errors(rho, decay_scale, beta_mu, seeds=4):
    e_dir, e_neu = 0.0, 0.0
    for sd in range(seeds):
        A, beta, v = _chunk(np.random.default_rng(1000 * sd + 7), rho, decay_scale, beta_mu)
        rhs = beta[:, None] * v
        U = oracle.unit_lower_inverse(A) @ rhs
        nU = np.linalg.norm(U)
        e_dir = max(e_dir, np.linalg.norm(_forward_subst_f32(A).astype(np.float64) @ rhs - U) / nU)
        e_neu = max(e_neu, np.linalg.norm(_neumann_doubling_f32(A).astype(np.float64) @ rhs - U) / nU)
    return e_dir, e_neu


GRID = [(0.0, 1.0, 0.0), (0.5, 1.0, 0.0), (0.8, 0.1, 2.0), (0.9, 0.01, 2.0), (0.95, 0.0, 3.0)]


def test_neumann_vs_direct_study():
    rows = []
    for rho, ds, bm in GRID:
        e_dir, e_neu = _errors(rho, ds, bm)
        rows.append((rho, ds, bm, e_dir, e_neu))
    print("\n  key corr | decay scale | beta mean | direct fp32 | Neumann fp32")
    for rho, ds, bm, e_dir, e_neu in rows:
        print(f"  {rho:8.2f} | {ds:11.2f} | {bm:9.1f} | {e_dir:11.2e} | {e_neu:12.2e}")
    # the direct solve stays at fp32 rounding on every case
    assert all(r[3] < 1e-4 for r in rows)
    # Neumann doubling is no better than the direct solve anywhere, and on the correlated,
    # weakly decayed chunks it is orders of magnitude worse
    assert all(r[4] >= 0.5 * r[3] for r in rows)
    assert rows[-1][4] > 100 * rows[-1][3]

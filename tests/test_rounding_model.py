"""A numpy model of the bf16 operand roundings in the tensor-core backward.

The forward-sweep kernel computes dq chunk by chunk from bf16 operands with
fp32 accumulation.  When phi(k) varies little (q, k ~ N(0,1)/sqrt(128)), dq is
a small difference of large terms and bf16 rounding is amplified.  This test
models the kernel's arithmetic in fp64 with bf16 rounding applied exactly where
the kernel rounds, and checks that the chosen scheme (D and phi(K) as hi + lo
pairs in D K~, g taken from the rounded P) stays inside the 2e-2 bound while
single bf16 copies do not.  CPU only; no GPU code involved.
"""
import numpy as np
import pytest
import torch


def bf(x):
    return torch.as_tensor(x, dtype=torch.float32).to(torch.bfloat16).to(torch.float64).numpy()


def split(x):
    h = bf(x)
    return h + bf(x - h)


def phi(x):
    return np.where(x > 0, x + 1, np.exp(x))


def dphi(x):
    return np.where(x > 0, 1.0, np.exp(x))


N, D, C = 4096, 128, 128


@pytest.fixture(scope="module")
def data():
    rng = np.random.default_rng(0)
    q = bf(rng.standard_normal((N, D)) / np.sqrt(128))
    k = bf(rng.standard_normal((N, D)) / np.sqrt(128))
    v = bf(rng.standard_normal((N, D)))
    dO = bf(rng.standard_normal((N, D)))
    qt, kt = phi(q), phi(k)
    # exact dq by the recurrence written chunk-wise in fp64
    S, z, dq = np.zeros((D, D)), np.zeros(D), np.zeros((N, D))
    for c0 in range(0, N, C):
        Q, K, V, G = qt[c0:c0 + C], kt[c0:c0 + C], v[c0:c0 + C], dO[c0:c0 + C]
        A = np.tril(Q @ K.T)
        num, den = Q @ S + A @ V, Q @ z + A.sum(1)
        P = G / den[:, None]
        g = -(P * num / den[:, None]).sum(1)
        Dm = np.tril(P @ V.T + g[:, None])
        dq[c0:c0 + C] = (P @ S.T + g[:, None] * z[None] + Dm @ K) * dphi(q[c0:c0 + C])
        S += K.T @ V
        z += K.sum(0)
    return q, qt, kt, v, dO, dq


def modelled_dq(data, d_split, k_split):
    q, qt, kt, v, dO, _ = data
    Qb, Kb = bf(qt), bf(kt)
    Kd = split(kt) if k_split else Kb
    S, z, out = np.zeros((D, D)), np.zeros(D), np.zeros((N, D))
    for c0 in range(0, N, C):
        sl = slice(c0, c0 + C)
        Q, K, V, G = Qb[sl], Kb[sl], v[sl], dO[sl]
        Sp = bf(S)                                   # S_prev as one bf16 operand
        A = bf(np.tril(Q @ K.T))                     # masked A, bf16 operand of A V
        num, den = Q @ Sp + A @ V, Q @ z + A.sum(1)  # fp32-accumulated products; z in fp32
        P = bf(G / den[:, None])                     # bf16 P
        g = -(P * num / den[:, None]).sum(1)         # g from that P
        Dm = np.tril(P @ V.T + g[:, None])
        Dm = split(Dm) if d_split else bf(Dm)
        out[sl] = (P @ Sp.T + g[:, None] * z[None] + Dm @ Kd[sl]) * dphi(q[sl])
        S += K.T @ V
        z += K.sum(0)
    return out


def rel(a, b):
    return float(np.abs(a - b).max() / np.abs(b).max())


def test_single_bf16_copies_exceed_the_bound(data):
    assert rel(modelled_dq(data, d_split=False, k_split=False), data[-1]) > 2e-2


def test_chosen_scheme_meets_the_bound(data):
    assert rel(modelled_dq(data, d_split=True, k_split=True), data[-1]) < 1.2e-2

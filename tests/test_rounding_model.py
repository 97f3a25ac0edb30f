"""A numpy model of the bf16 operand roundings in the tensor-core backward.

The forward-sweep kernel computes dq chunk by chunk from bf16 operands with
fp32 accumulation.  When phi(k) varies little (q, k ~ N(0,1)/sqrt(128)), dq is
a small difference of large terms and bf16 rounding is amplified.  This test
models the kernel's arithmetic in fp64 with bf16 rounding applied exactly where
the kernel rounds, and checks that the scheme the kernel uses stays well inside
the 2e-2 bound while single bf16 copies do not:
  - A = tril(phi(Q) phi(K)^T) enters A V as a hi + lo pair (its entries sit near
    the head size, so one bf16 copy keeps little of their variation; this is the
    largest error source at long N),
  - D K~ is formed as rowsum(D) 1^T (fp32) + bf16(D) bf16(phi(K) - 1),
  - g is taken from the rounded P.
The non-causal gradient has the same cancellation with the whole sequence in
every row; its model checks the scheme of the non-causal kernels (phi(K) as
hi + lo in the sums S and z, S as hi + lo in num and dQ~, phi(Q) one bf16 copy
in num and den, den in fp32, g from the rounded P).  CPU only; no GPU code
involved.
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


def make_case(n, seed):
    """Inputs of the long-context recipe (q, k ~ N(0,1)/sqrt(128), v, dO ~ N(0,1), bf16) and
    the exact dq by the recurrence written chunk-wise in fp64."""
    rng = np.random.default_rng(seed)
    q = bf(rng.standard_normal((n, D)) / np.sqrt(128))
    k = bf(rng.standard_normal((n, D)) / np.sqrt(128))
    v = bf(rng.standard_normal((n, D)))
    dO = bf(rng.standard_normal((n, D)))
    qt, kt = phi(q), phi(k)
    S, z, dq = np.zeros((D, D)), np.zeros(D), np.zeros((n, D))
    for c0 in range(0, n, C):
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


@pytest.fixture(scope="module")
def data():
    return make_case(N, 0)


def modelled_dq(data, a_split, dk):
    """dk: 'single' (bf16 D times bf16 phi(K)), 'hilo' (D_hi K_hi + D_lo K_hi + D_hi K_lo) or
    'minus_one' (fp32 rowsum(D) plus bf16 D times bf16(phi(K) - 1))."""
    q, qt, kt, v, dO, _ = data
    n = q.shape[0]
    Qb, Kb = bf(qt), bf(kt)
    Kl, Km1 = bf(kt - Kb), bf(kt - 1.0)
    S, z, out = np.zeros((D, D)), np.zeros(D), np.zeros((n, D))
    for c0 in range(0, n, C):
        sl = slice(c0, c0 + C)
        Q, K, V, G = Qb[sl], Kb[sl], v[sl], dO[sl]
        Sp = bf(S)                                   # S_prev as one bf16 operand
        Af = np.tril(Q @ K.T)                        # fp32-accumulated, masked
        A = split(Af) if a_split else bf(Af)         # the A operand(s) of A V
        num, den = Q @ Sp + A @ V, Q @ z + A.sum(1)  # row sums of the operands A V uses; z in fp32
        P = bf(G / den[:, None])                     # bf16 P
        g = -(P * num / den[:, None]).sum(1)         # g from that P
        Dm = np.tril(P @ V.T + g[:, None])
        if dk == "single":
            DK = bf(Dm) @ K
        elif dk == "hilo":
            Dh = bf(Dm)
            DK = Dh @ K + bf(Dm - Dh) @ K + Dh @ Kl[sl]
        else:
            DK = Dm.sum(1)[:, None] + bf(Dm) @ Km1[sl]
        out[sl] = (P @ Sp.T + g[:, None] * z[None] + DK) * dphi(q[sl])
        S += K.T @ V
        z += K.sum(0)
    return out


def rel(a, b):
    return float(np.abs(a - b).max() / np.abs(b).max())


def test_single_bf16_copies_exceed_the_bound(data):
    assert rel(modelled_dq(data, a_split=False, dk="single"), data[-1]) > 2e-2


def test_kernel_scheme_meets_the_bound(data):
    assert rel(modelled_dq(data, a_split=True, dk="minus_one"), data[-1]) < 1e-2


def test_long_sequence_needs_the_a_split():
    """At N = 16384 (seed 0) the rounding of A dominates: with one bf16 copy of A the error
    comes within a few percent of the bound whatever D K~ does, with A as hi + lo it is
    under a third of it."""
    case = make_case(16384, 0)
    for dk in ("hilo", "minus_one"):
        assert rel(modelled_dq(case, a_split=False, dk=dk), case[-1]) > 1.8e-2
    assert rel(modelled_dq(case, a_split=True, dk="minus_one"), case[-1]) < 7e-3


# ---------------------------------------------------------------- non-causal gradient
# dphi(q)_i = S P_i - z (P_i . num_i) / den_i with P_i = dO_i / den_i, S = phi(K)^T V,
# z = phi(K)^T 1 over the whole sequence: the non-causal form of "Transformers은 RNN이다"
# (irregular6612 blog digest), 핵심 구성요소 2, differentiated.
NC_N = 1024


@pytest.fixture(scope="module")
def nc_data():
    rng = np.random.default_rng(1)
    q = bf(rng.standard_normal((NC_N, D)) / np.sqrt(128))
    k = bf(rng.standard_normal((NC_N, D)) / np.sqrt(128))
    v = bf(rng.standard_normal((NC_N, D)))
    dO = bf(rng.standard_normal((NC_N, D)))
    qt, kt = phi(q), phi(k)
    # exact dq from the direct pairwise weights w_ij = phi(q_i) . phi(k_j), in fp64
    w = qt @ kt.T
    den = w.sum(1)
    o = (w @ v) / den[:, None]
    dw = (dO @ v.T - (dO * o).sum(1)[:, None]) / den[:, None]   # d loss / d w_ij
    dq = (dw @ kt) * dphi(q)
    return q, qt, kt, v, dO, dq


def nc_modelled_dq(data, k_split, s_split, q_split):
    q, qt, kt, v, dO, _ = data
    Ks = split(kt) if k_split else bf(kt)          # phi(K) operand(s) of the sums
    S, z = Ks.T @ v, Ks.sum(0)                     # fp32-accumulated sums
    Sh = bf(S)
    Sl = bf(S - Sh) if s_split else 0 * S
    Qh = bf(qt)
    Ql = bf(qt - Qh) if q_split else 0 * qt
    num = Qh @ Sh + Qh @ Sl + Ql @ Sh
    den = (Qh + Ql) @ z                            # fp32, from the same parts
    P = bf(dO / den[:, None])                      # bf16 P
    g = -(P * num).sum(1) / den                    # g from that P
    return (P @ (Sh + Sl).T + g[:, None] * z[None]) * dphi(q)


def test_noncausal_exact_gradient_is_the_state_form(nc_data):
    # the fixture's pairwise form against the state form in fp64 (no rounding)
    q, qt, kt, v, dO, dq = nc_data
    S, z = kt.T @ v, kt.sum(0)
    num, den = qt @ S, qt @ z
    P = dO / den[:, None]
    ref = (P @ S.T - ((P * num).sum(1) / den)[:, None] * z[None]) * dphi(q)
    assert rel(ref, dq) < 1e-10


@pytest.mark.parametrize("k_split,s_split,q_split", [(False, False, False), (True, False, False),
                                                     (False, True, True)])
def test_noncausal_partial_schemes_exceed_the_bound(nc_data, k_split, s_split, q_split):
    assert rel(nc_modelled_dq(nc_data, k_split, s_split, q_split), nc_data[-1]) > 2e-2


def test_noncausal_chosen_scheme_meets_the_bound(nc_data):
    assert rel(nc_modelled_dq(nc_data, True, True, False), nc_data[-1]) < 5e-3


def test_noncausal_splitting_phi_q_adds_nothing(nc_data):
    # phi(q) rounding scales every key's weight alike and num, den share it: splitting it
    # as well changes dq by far less than the bound
    a = rel(nc_modelled_dq(nc_data, True, True, False), nc_data[-1])
    b = rel(nc_modelled_dq(nc_data, True, True, True), nc_data[-1])
    assert abs(a - b) < 5e-4

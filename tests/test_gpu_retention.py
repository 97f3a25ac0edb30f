"""GPU parity of retention (constant decay per head) against the fp64 oracle.

Same comparison as the other parity tests: per (b, h) head slice,
max|gpu - oracle| / max|oracle|, bounded by 1e-4 for fp32 inputs and 2e-2 for
bf16 inputs.  The oracle reads the same seeded inputs after the cast.
"""
import numpy as np
import pytest
import torch

import oracle
from causal_linear_attention_phi_gb300 import workloads as W
from util import rel_per_head, tol_for, to_np

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module")
def la():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import causal_linear_attention_phi_gb300 as la
    la.build.build_library()
    la.library()
    la.clear_error()
    yield la
    assert la.last_error() == 0


def check(name, gpu, ref, tol):
    e = rel_per_head(gpu, ref)
    assert e <= tol, "%s: max rel err %.3e > %.1e" % (name, e, tol)
    return e


# the special values 0 and 1 and the workload's range, cycled over the heads
GAMMA_POOL = [0.9, 1.0, 0.0, 0.5, 0.999, 0.97]


def gammas(H):
    return torch.tensor([GAMMA_POOL[h % len(GAMMA_POOL)] for h in range(H)], dtype=torch.float32)


CASES = [
    # (B, H, N, Dk, Dv, dtype)
    (1, 1, 1, 16, 16, torch.float32),        # a single position: o = (q . k) v
    (1, 3, 63, 32, 16, torch.float32),       # one short chunk
    (2, 2, 64, 16, 32, torch.float32),       # exactly one chunk
    (1, 3, 65, 64, 128, torch.float32),      # one position past a chunk
    (2, 3, 200, 128, 64, torch.float32),     # several chunks, ragged tail
    (1, 6, 1000, 128, 128, torch.float32),   # many segments: the decayed scan in use
    (3, 2, 777, 32, 32, torch.bfloat16),
    (1, 4, 4097, 64, 64, torch.bfloat16),
    (2, 3, 1500, 128, 128, torch.bfloat16),
]


@pytest.mark.parametrize("B,H,N,Dk,Dv,dtype", CASES)
def test_retention_fwd_cases(la, B, H, N, Dk, Dv, dtype):
    q, k, v = W.random_case(900 + N, B, H, N, Dk, Dv, dtype=dtype, scale=Dk ** -0.25)
    g = gammas(H)
    o, S = la.retention_fwd(q.to(DEV), k.to(DEV), v.to(DEV), g.to(DEV), return_state=True)
    assert o.dtype == dtype and S.dtype == torch.float32
    ref = oracle.retention_direct(q, k, v, g) if N <= 1000 else oracle.retention_chunked(q, k, v, g, 128)
    check("retention o", o, ref, tol_for(dtype))
    # the state after position N: sum_j gamma^(N-1-j) k_j v_j^T, from the oracle's decode steps
    if N <= 200:
        Sref = np.zeros((B, H, Dk, Dv))
        for t in range(N):
            _, Sref = oracle.retention_step(q[:, :, t], k[:, :, t], v[:, :, t], g, Sref)
        check("retention S", S, Sref, 1e-4 if dtype == torch.float32 else 1e-3)


# bf16 heads of 128 (or 64, padded on chip) run on the tensor-core kernels (chunks of 128)
TC_CASES = [
    (1, 3, 1, 128, 128),      # a single position
    (1, 2, 127, 128, 128),    # one short chunk
    (2, 3, 128, 128, 128),    # exactly one chunk
    (1, 3, 129, 64, 64),      # one position past a chunk, padded head
    (1, 6, 1000, 128, 128),   # several chunks and segments, ragged tail
    (2, 6, 3001, 64, 64),
    (1, 2, 8192, 128, 128),   # long segments: the reverse-walk sums over many chunks
]


@pytest.mark.parametrize("B,H,N,Dk,Dv", TC_CASES)
def test_retention_tensor_core_cases(la, B, H, N, Dk, Dv):
    q, k, v = W.random_case(1900 + N, B, H, N, Dk, Dv, dtype=torch.bfloat16, scale=Dk ** -0.25)
    g = gammas(H)
    la.timing_reset()
    la.timing_enable(True)
    try:
        o, S = la.retention_fwd(q.to(DEV), k.to(DEV), v.to(DEV), g.to(DEV), return_state=True)
        torch.cuda.synchronize()
    finally:
        la.timing_enable(False)
    assert "tc_retention_out" in la.timing_read()
    ref = oracle.retention_direct(q, k, v, g) if N <= 1000 else oracle.retention_chunked(q, k, v, g, 128)
    check("retention o (tensor cores)", o, ref, 2e-2)
    # the final state against the oracle's decode recurrence (bf16 K' and V products, fp32 sums)
    if N <= 300:
        Sref = np.zeros((B, H, Dk, Dv))
        for t in range(N):
            _, Sref = oracle.retention_step(q[:, :, t], k[:, :, t], v[:, :, t], g, Sref)
        check("retention S (tensor cores)", S, Sref, 1e-2)


@pytest.mark.parametrize("Dk,dtype", [(32, torch.float32), (64, torch.bfloat16), (128, torch.bfloat16)])
def test_decay_outside_unit_interval(la, Dk, dtype):
    """Any real gamma is computed as written: negative decays alternate the signs of older
    terms (the powers come from repeated squaring, not a logarithm), and a decay above 1
    grows them (here 1.01^300, about 20)."""
    q, k, v = W.random_case(2300 + Dk, 1, 3, 300, Dk, Dk, dtype=dtype, scale=Dk ** -0.25)
    g = torch.tensor([-0.5, 1.01, -1.0])
    o, S = la.retention_fwd(q.to(DEV), k.to(DEV), v.to(DEV), g.to(DEV), return_state=True)
    check("o", o, oracle.retention_direct(q, k, v, g), tol_for(dtype))
    Sref = np.zeros((1, 3, Dk, Dk))
    for t in range(300):
        _, Sref = oracle.retention_step(q[:, :, t], k[:, :, t], v[:, :, t], g, Sref)
    check("S", S, Sref, 1e-4 if dtype == torch.float32 else 1e-2)


def test_gamma_one_is_the_masked_product(la):
    """gamma = 1: o = tril(Q K^T) V, checked against a float64 matrix product."""
    q, k, v = W.random_case(31, 1, 2, 300, 64, 32, dtype=torch.float32, scale=64 ** -0.25)
    o = la.retention_fwd(q.to(DEV), k.to(DEV), v.to(DEV), torch.ones(2, device=DEV))
    qd, kd, vd = to_np(q), to_np(k), to_np(v)
    ref = np.tril(qd @ np.swapaxes(kd, -1, -2)) @ vd
    check("gamma=1", o, ref, 1e-4)


def test_gamma_zero_keeps_the_diagonal(la):
    q, k, v = W.random_case(32, 2, 2, 130, 32, 64, dtype=torch.float32)
    o = la.retention_fwd(q.to(DEV), k.to(DEV), v.to(DEV), torch.zeros(2, device=DEV))
    ref = (to_np(q) * to_np(k)).sum(-1, keepdims=True) * to_np(v)
    check("gamma=0", o, ref, 1e-5)


@pytest.mark.parametrize("B,H,N,Dk,Dv,dtype", [
    (1, 3, 333, 64, 64, torch.float32),
    (2, 2, 1000, 128, 128, torch.float32),   # prefill over several segments
    (1, 4, 700, 128, 128, torch.bfloat16),
])
def test_prefill_state_then_decode(la, B, H, N, Dk, Dv, dtype):
    """retention_fwd's state, continued by retention_step, reproduces the recurrence."""
    T = 40
    q, k, v = W.random_case(1200 + N, B, H, N + T, Dk, Dv, dtype=dtype, scale=Dk ** -0.25)
    g = gammas(H)
    gd = g.to(DEV)
    o_pre, S = la.retention_fwd(q[:, :, :N].contiguous().to(DEV), k[:, :, :N].contiguous().to(DEV),
                                v[:, :, :N].contiguous().to(DEV), gd, return_state=True)
    outs = []
    for t in range(N, N + T):
        outs.append(la.retention_step(q[:, :, t].contiguous().to(DEV), k[:, :, t].contiguous().to(DEV),
                                      v[:, :, t].contiguous().to(DEV), gd, S))
    ref = oracle.retention_recurrent(q, k, v, g)
    tol = tol_for(dtype)
    check("prefill o", o_pre, ref[:, :, :N], tol)
    check("decode o", torch.stack(outs, 2), ref[:, :, N:], tol)


def test_decode_from_zero_matches_oracle_steps(la):
    B, H, Dk, Dv, T = 8, 4, 32, 16, 50
    q, k, v = W.random_case(77, B, H, T, Dk, Dv, dtype=torch.float32)
    g = gammas(H)
    S = torch.zeros(B, H, Dk, Dv, device=DEV)
    Sref = np.zeros((B, H, Dk, Dv))
    for t in range(T):
        o = la.retention_step(q[:, :, t].contiguous().to(DEV), k[:, :, t].contiguous().to(DEV),
                              v[:, :, t].contiguous().to(DEV), g.to(DEV), S)
        oref, Sref = oracle.retention_step(q[:, :, t], k[:, :, t], v[:, :, t], g, Sref)
        check("step %d o" % t, o, oref, 1e-4)
    check("final S", S, Sref, 1e-4)


def test_decode_cifar_shape_all_steps_graph(la):
    """The retention step over all 3072 steps of the CIFAR-shaped decode workload (B=64 H=8
    D=32 fp32), captured in one CUDA graph as the bench runs it: every output and the final
    state against the oracle's recurrence."""
    w = W.DECODE_CIFAR
    q, k, v = W.make_decode_inputs(w)
    g = W.retention_gammas(w.H)
    qd, kd, vd, gd = (t.to(DEV) for t in (q, k, v, g))
    S = torch.zeros(w.B, w.H, w.Dk, w.Dv, device=DEV)
    outs = torch.empty(w.steps, w.B, w.H, w.Dv, device=DEV)
    st = torch.cuda.Stream()
    st.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(st):
        la.retention_step(qd[0], kd[0], vd[0], gd, S, out=outs[0])
    torch.cuda.synchronize()
    S.zero_()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=st):
        for t in range(w.steps):
            la.retention_step(qd[t], kd[t], vd[t], gd, S, out=outs[t])
    graph.replay()
    torch.cuda.synchronize()
    to_seq = lambda x: x.permute(1, 2, 0, 3).contiguous()
    ref = oracle.retention_recurrent(to_seq(q), to_seq(k), to_seq(v), g)
    check("retention decode, 3072 steps", to_seq(outs.cpu()), ref, 1e-4)
    decay = g.double().numpy()[:, None] ** np.arange(w.steps - 1, -1, -1, dtype=np.float64)[None, :]  # [H, T]
    Sref = np.einsum("hn,bhnd,bhnm->bhdm", decay, to_np(to_seq(k)), to_np(to_seq(v)))
    check("final S", S.cpu(), Sref, 1e-4)


@pytest.mark.parametrize("Dk,Dv", [(16, 128), (128, 16), (64, 32)])
def test_decode_head_sizes(la, Dk, Dv):
    B, H, T = 3, 2, 20
    q, k, v = W.random_case(78 + Dk, B, H, T, Dk, Dv, dtype=torch.bfloat16)
    g = gammas(H)
    S = torch.zeros(B, H, Dk, Dv, device=DEV)
    outs = [la.retention_step(q[:, :, t].contiguous().to(DEV), k[:, :, t].contiguous().to(DEV),
                              v[:, :, t].contiguous().to(DEV), g.to(DEV), S) for t in range(T)]
    check("decode", torch.stack(outs, 2), oracle.retention_recurrent(q, k, v, g), 2e-2)


def test_empty_sequence_state_is_zero(la):
    q = torch.empty(2, 3, 0, 32, device=DEV)
    o, S = la.retention_fwd(q, q, q, torch.ones(3, device=DEV), return_state=True)
    assert o.numel() == 0 and S.shape == (2, 3, 32, 32) and torch.count_nonzero(S).item() == 0


def test_bad_gamma_is_refused(la):
    q, k, v = W.random_case(3, 1, 2, 64, 16, 16)
    with pytest.raises(ValueError):
        la.retention_fwd(q.to(DEV), k.to(DEV), v.to(DEV), torch.ones(3, device=DEV))   # wrong length
    lib = la.library()
    qd = q.to(DEV)
    o = torch.empty_like(qd)
    s = la.Shape(1, 2, 64, 16, 16, 0)
    host_gamma = torch.ones(2)
    import ctypes
    st = lib.la_retention_fwd(la._ptr(qd), la._ptr(qd), la._ptr(qd), ctypes.c_void_p(host_gamma.data_ptr()),
                              la._ptr(o), None, s, None, 0, None)
    assert st == 1   # a host pointer for gamma: LA_ERR_INVALID_ARG before any launch


def test_full_size_sampled_heads(la):
    """The bench workload (B=2 H=16 N=65536 D=128 bf16) through the same call the
    bench times; two heads checked against the oracle's chunked form."""
    w = W.RETENTION_BF16
    q, k, v = W.make_inputs(w)
    g = W.retention_gammas(w.H)
    o = la.retention_fwd(q.to(DEV), k.to(DEV), v.to(DEV), g.to(DEV)).cpu()
    for b, h in [(0, 0), (1, 15)]:
        sl = (slice(b, b + 1), slice(h, h + 1))
        ref = oracle.retention_chunked(q[sl], k[sl], v[sl], g[h:h + 1], 256)
        check("head (%d,%d)" % (b, h), o[sl], ref, 2e-2)

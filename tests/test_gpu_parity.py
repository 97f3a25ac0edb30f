"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Every comparison is per (b, h) head slice, max|gpu - oracle| / max|oracle|,
bounded by 1e-4 for fp32 inputs and 2e-2 for bf16 inputs (fp32 accumulation).
The oracle consumes the same seeded inputs after the cast to the input dtype.
"""
import ctypes

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


def dev(*ts):
    return [t.to(DEV) for t in ts]


def check(name, gpu, ref, tol):
    e = rel_per_head(gpu, ref)
    assert e <= tol, "%s: max rel err %.3e > %.1e" % (name, e, tol)
    return e


def check_all(pairs, tol):
    """Compare several tensors, reporting every error before failing on any."""
    errs = {name: rel_per_head(a, b) for name, a, b in pairs}
    bad = {n: e for n, e in errs.items() if not e <= tol}
    assert not bad, "max rel errs %s (bound %.1e)" % ({n: "%.3e" % e for n, e in errs.items()}, tol)
    return errs


# ---------------------------------------------------------------- forward, small fp32 workload
def test_small_f32_causal_fwd(la):
    q, k, v = W.make_inputs(W.SMALL_F32)
    o = la.causal_fwd(*dev(q, k, v))
    check("o vs direct", o, oracle.causal_direct(q, k, v), 1e-4)
    check("o vs recurrent", o, oracle.causal_recurrent(q, k, v), 1e-4)


# ---------------------------------------------------------------- forward, bf16 B=4 H=8 N=1024 D=64
def test_fwd_bf16_noncausal_and_causal(la):
    q, k, v = W.make_inputs(W.FWD_BF16)
    qd, kd, vd = dev(q, k, v)
    onc = la.noncausal_fwd(qd, kd, vd)
    oc = la.causal_fwd(qd, kd, vd)
    assert onc.dtype == torch.bfloat16 and oc.dtype == torch.bfloat16
    check("noncausal", onc, oracle.noncausal_assoc(q, k, v), 2e-2)
    check("causal", oc, oracle.causal_recurrent(q, k, v), 2e-2)


# ---------------------------------------------------------------- edge cases of the forward
FWD_CASES = [
    # (B, H, N, Dk, Dv, dtype)
    (1, 1, 1, 16, 16, torch.float32),      # a single position: o = v
    (1, 2, 63, 32, 16, torch.float32),     # one short chunk
    (1, 1, 64, 16, 32, torch.float32),     # exactly one chunk
    (2, 1, 65, 64, 128, torch.float32),    # one position past a chunk
    (1, 3, 200, 128, 64, torch.float32),   # several chunks and a ragged tail
    (1, 2, 1000, 128, 128, torch.float32), # many segments (segment scan in use)
    (3, 1, 777, 32, 32, torch.bfloat16),
    (1, 1, 4097, 64, 64, torch.bfloat16),
    (2, 2, 130, 16, 128, torch.bfloat16),
    # bf16 with Dk = Dv = 128 runs on the tensor-core kernels (chunks of 128)
    (1, 1, 1, 128, 128, torch.bfloat16),
    (1, 1, 128, 128, 128, torch.bfloat16),
    (2, 1, 129, 128, 128, torch.bfloat16),
    (1, 2, 1000, 128, 128, torch.bfloat16),
    (1, 3, 4097, 128, 128, torch.bfloat16),
]


@pytest.mark.parametrize("B,H,N,Dk,Dv,dtype", FWD_CASES)
def test_causal_fwd_cases(la, B, H, N, Dk, Dv, dtype):
    scale = 1.0 if dtype == torch.float32 else 0.5
    q, k, v = W.random_case(100 + N, B, H, N, Dk, Dv, dtype=dtype, scale=scale)
    o = la.causal_fwd(*dev(q, k, v))
    ref = oracle.causal_direct(q, k, v) if N <= 1000 else oracle.causal_recurrent(q, k, v)
    check("causal o", o, ref, tol_for(dtype))
    onc = la.noncausal_fwd(*dev(q, k, v))
    check("noncausal o", onc, oracle.noncausal_assoc(q, k, v), tol_for(dtype))
    if N == 1:
        assert torch.allclose(o.cpu(), v, rtol=1e-6, atol=0)


@pytest.mark.parametrize("B,H,N,Dk,Dv,dtype", [
    (1, 2, 1000, 128, 128, torch.bfloat16),   # segment sums on the tensor cores
    (2, 3, 777, 64, 64, torch.bfloat16),      # the same with a padded head
    (1, 2, 300, 32, 16, torch.float32),       # CUDA cores throughout
])
def test_noncausal_fwd_cases(la, B, H, N, Dk, Dv, dtype):
    q, k, v = W.random_case(700 + N, B, H, N, Dk, Dv, dtype=dtype, scale=Dk ** -0.5)
    o = la.noncausal_fwd(*dev(q, k, v))
    check("non-causal o", o, oracle.noncausal_assoc(q, k, v), tol_for(dtype))


def test_constant_v_gives_constant_output(la):
    q, k, _ = W.random_case(5, 1, 2, 333, 64, 32, dtype=torch.float32)
    c = torch.linspace(-2, 2, 32)
    v = c.expand(1, 2, 333, 32).contiguous()
    o = la.causal_fwd(*dev(q, k, v)).cpu()
    assert torch.max(torch.abs(o - c)) < 1e-5


def test_empty_is_noop(la):
    z = torch.empty(1, 2, 0, 16, device=DEV)
    o = la.causal_fwd(z, z, z)
    assert o.shape == (1, 2, 0, 16)


# ---------------------------------------------------------------- backward
BWD_CASES = [
    (1, 2, 50, 16, 32, torch.float32),     # the itwiki check's shapes
    (2, 1, 129, 32, 16, torch.float32),
    (1, 2, 700, 64, 64, torch.float32),    # multiple segments
    (1, 1, 300, 128, 128, torch.float32),
    (1, 2, 1000, 64, 64, torch.bfloat16),
    (2, 1, 515, 128, 128, torch.bfloat16),
]


@pytest.mark.parametrize("B,H,N,Dk,Dv,dtype", BWD_CASES)
def test_causal_bwd_cases(la, B, H, N, Dk, Dv, dtype):
    scale = 1.0 if dtype == torch.float32 else 0.5
    q, k, v, dO = W.random_case(200 + N, B, H, N, Dk, Dv, dtype=dtype, scale=scale, with_grad=True)
    dq, dk, dv = la.causal_bwd(*dev(q, k, v, dO))
    ref = oracle.causal_bwd_recurrent(q, k, v, dO)
    check_all([(n, a, b) for n, a, b in zip(("dq", "dk", "dv"), (dq, dk, dv), ref)], tol_for(dtype))


@pytest.mark.parametrize("B,H,N,Dk,Dv,dtype", [
    (1, 2, 64, 16, 16, torch.float32),
    (2, 3, 1000, 32, 64, torch.float32),       # several chunks and segments, ragged tail
    (4, 8, 1024, 64, 64, torch.bfloat16),      # the non-causal forward workload's shape
    (1, 2, 300, 128, 128, torch.bfloat16),
    (1, 2, 2049, 128, 128, torch.bfloat16),    # tensor cores: many chunks, a one-row tail
    (2, 1, 1500, 64, 64, torch.bfloat16),      # tensor cores, padded head, several segments
    (1, 1, 1, 32, 16, torch.float32),          # a single position
])
def test_noncausal_bwd_cases(la, B, H, N, Dk, Dv, dtype):
    q, k, v, dO = W.random_case(500 + N, B, H, N, Dk, Dv, dtype=dtype, scale=Dk ** -0.5, with_grad=True)
    dq, dk, dv = la.noncausal_bwd(*dev(q, k, v, dO))
    ref = oracle.noncausal_bwd_direct(q, k, v, dO)
    if N == 1:  # o = v: no dependence on q or k, dv = dO
        assert float(dq.abs().max()) < 1e-5 and float(dk.abs().max()) < 1e-5
        check("dv", dv, ref[2], tol_for(dtype))
        return
    check_all([(n, a, b) for n, a, b in zip(("dq", "dk", "dv"), (dq, dk, dv), ref)], tol_for(dtype))


def test_noncausal_bwd_sums_match_forward_invariants(la):
    """sum_j dv_j = sum_i dO_i per head and column (the weights of each o_i sum to one)."""
    q, k, v, dO = W.random_case(77, 2, 2, 513, 32, 32, dtype=torch.float32, with_grad=True)
    _, _, dv = la.noncausal_bwd(*dev(q, k, v, dO))
    np.testing.assert_allclose(to_np(dv.sum(2).cpu()), to_np(dO.sum(2)), rtol=1e-4, atol=1e-4)


@pytest.mark.parametrize("B,H,N,Dk,Dv,dtype,G", [
    (2, 3, 1000, 128, 128, torch.bfloat16, 4),   # tensor-core kernels; 6 heads in groups of 4 and 2
    (1, 5, 700, 32, 64, torch.float32, 2),       # CUDA-core kernels; groups of 2, 2, 1
    (1, 2, 300, 64, 64, torch.bfloat16, 8),      # one group
])
def test_step_host_matches_oracle(la, B, H, N, Dk, Dv, dtype, G):
    q, k, v, dO = W.random_case(600 + N, B, H, N, Dk, Dv, dtype=dtype, scale=Dk ** -0.5, with_grad=True)
    hin = [t.contiguous().pin_memory() for t in (q, k, v, dO)]
    hout = [torch.empty(t.shape, dtype=dtype).pin_memory() for t in (v, q, k, v)]
    la.causal_step_host(*hin, *hout, group_heads=G)
    torch.cuda.synchronize()
    o, dq, dk, dv = hout
    tol = tol_for(dtype)
    check("o", o, oracle.causal_recurrent(q, k, v), tol)
    ref = oracle.causal_bwd_recurrent(q, k, v, dO)
    check_all([(n, a, b) for n, a, b in zip(("dq", "dk", "dv"), (dq, dk, dv), ref)], tol)


def test_step_host_refuses_pageable_memory(la):
    q = torch.randn(1, 2, 64, 32)
    with pytest.raises(ValueError):
        la.causal_step_host(q, q, q, q, q.clone(), q.clone(), q.clone(), q.clone())
    # through the C ABI directly: pageable buffers are refused before anything is queued
    s = la.Shape(1, 2, 64, 32, 32, la.LA_F32)
    dev_buf = torch.empty(la.host_step_bytes(1, 2, 64, 32, 32, torch.float32, 2), dtype=torch.uint8, device=DEV)
    p = ctypes.c_void_p(q.data_ptr())
    st = la.library().la_causal_step_host(p, p, p, p, p, p, p, p, s, 2, ctypes.c_void_p(dev_buf.data_ptr()),
                                          dev_buf.numel(), None)
    assert st == 1


def test_bwd_single_position(la):
    # N = 1: o_1 = v_1 whatever q and k are, so dq = dk = 0 exactly and dv = dO.
    q, k, v, dO = W.random_case(30, 2, 3, 1, 16, 32, dtype=torch.float32, with_grad=True)
    dq, dk, dv = la.causal_bwd(*dev(q, k, v, dO))
    assert float(dq.abs().max()) < 1e-5 and float(dk.abs().max()) < 1e-5
    assert torch.allclose(dv.cpu(), dO, rtol=1e-5, atol=1e-6)


def test_bwd_invariants(la):
    q, k, v, dO = W.random_case(31, 1, 2, 257, 32, 32, dtype=torch.float32, with_grad=True)
    dq, dk, dv = la.causal_bwd(*dev(q, k, v, dO))
    # sum_j dv_j = sum_i dO_i per head and column
    assert rel_per_head(dv.sum(2, keepdim=True).cpu(), dO.sum(2, keepdim=True)) < 1e-4
    # constant v: the output ignores q and k
    vc = torch.linspace(-1, 1, 32).expand_as(v).contiguous()
    dq, dk, _ = la.causal_bwd(*dev(q, k, vc, dO))
    assert float(dq.abs().max()) < 1e-4 and float(dk.abs().max()) < 1e-4


# ---------------------------------------------------------------- length sweep, bf16 B=1 H=8 D=64
@pytest.mark.parametrize("N", [n for n in W.SWEEP_NS if n <= 4096])
def test_sweep_fwd_bwd_full(la, N):
    w = W.sweep(N)
    q, k, v, dO = W.make_inputs(w, with_grad=True)
    qd, kd, vd, dOd = dev(q, k, v, dO)
    o = la.causal_fwd(qd, kd, vd)
    dq, dk, dv = la.causal_bwd(qd, kd, vd, dOd)
    check_all([("o", o, oracle.causal_recurrent(q, k, v))] +
              [(n, a, b) for n, a, b in zip(("dq", "dk", "dv"), (dq, dk, dv), oracle.causal_bwd_recurrent(q, k, v, dO))],
              2e-2)


def _sampled_heads(la, w, heads, tensors=None):
    """Full-size run on the GPU, oracle on a few whole heads (heads are independent)."""
    q, k, v, dO = W.make_inputs(w, with_grad=True) if tensors is None else tensors
    qd, kd, vd, dOd = dev(q, k, v, dO)
    o = la.causal_fwd(qd, kd, vd)
    dq, dk, dv = la.causal_bwd(qd, kd, vd, dOd)
    torch.cuda.synchronize()
    sel = lambda t: torch.stack([t[b, h] for b, h in heads])[None]
    qs, ks, vs, dOs = (sel(t) for t in (q, k, v, dO))
    ref = oracle.causal_bwd_recurrent(qs, ks, vs, dOs)
    check_all([("o", sel(o.cpu()), oracle.causal_recurrent(qs, ks, vs))] +
              [(n, sel(a.cpu()), b) for n, a, b in zip(("dq", "dk", "dv"), (dq, dk, dv), ref)], 2e-2)


@pytest.mark.parametrize("N", [n for n in W.SWEEP_NS if n > 4096])
def test_sweep_long_sampled_heads(la, N):
    """Every length of the sweep above 4096 (8192 .. 65536): the whole batch on the GPU,
    two whole heads against the oracle."""
    _sampled_heads(la, W.sweep(N), [(0, 0), (0, 5)])


def test_long_bf16_full_size_sampled_heads(la):
    _sampled_heads(la, W.LONG_BF16, [(0, 0), (1, 15)])


def test_bf16_d128_many_chunks_and_segments(la):
    # B*H = 64, N = 20000: 157 chunks of 128 per head, several chunks per segment and
    # several segments per head, ragged tail (20000 = 156 * 128 + 32)
    t = W.random_case(77, 4, 16, 20000, 128, 128, dtype=torch.bfloat16, scale=128 ** -0.5, with_grad=True)
    _sampled_heads(la, None, [(0, 0), (2, 7), (3, 15)], tensors=t)


@pytest.mark.parametrize("B,H,N,Dk,Dv,dtype", [
    (1, 4, 4096, 128, 128, torch.bfloat16),   # tensor-core path, several segments
    (1, 2, 100, 128, 128, torch.bfloat16),    # tensor-core path, one segment
    (2, 2, 3000, 64, 64, torch.bfloat16),     # tensor-core path, head of 64 padded on chip
    (2, 3, 1500, 32, 64, torch.float32),      # CUDA-core path
])
def test_bwd_after_fwd_is_bit_identical(la, B, H, N, Dk, Dv, dtype):
    """The backward that reads the forward's segment states gives exactly la_causal_bwd's gradients."""
    q, k, v, dO = dev(*W.random_case(300 + N, B, H, N, Dk, Dv, dtype=dtype, scale=Dk ** -0.5, with_grad=True))
    ws_f = torch.empty(la.workspace_bytes(la.OP_CAUSAL_FWD, B, H, N, Dk, Dv, dtype), dtype=torch.uint8, device=DEV)
    la.causal_fwd(q, k, v, workspace=ws_f)
    ref = la.causal_bwd(q, k, v, dO)
    got = la.causal_bwd(q, k, v, dO, fwd_workspace=ws_f)
    torch.cuda.synchronize()
    for name, a, b in zip(("dq", "dk", "dv"), got, ref):
        assert torch.equal(a, b), name
    with pytest.raises(la.LaError):  # a forward workspace one byte short is refused
        la.causal_bwd(q, k, v, dO, fwd_workspace=ws_f[:-1])


def test_bf16_d128_single_position(la):
    q, k, v, dO = W.random_case(78, 1, 2, 1, 128, 128, dtype=torch.bfloat16, with_grad=True)
    qd, kd, vd, dOd = dev(q, k, v, dO)
    o = la.causal_fwd(qd, kd, vd)
    assert torch.equal(o.cpu(), v)
    dq, dk, dv = la.causal_bwd(qd, kd, vd, dOd)
    assert float(dq.float().abs().max()) < 1e-2 and float(dk.float().abs().max()) < 1e-2
    assert rel_per_head(dv.cpu(), dO) < 2e-2


# ---------------------------------------------------------------- decode
def test_decode_mnist_shape_all_steps(la):
    w = W.DECODE_MNIST
    q, k, v = W.make_decode_inputs(w)
    qd, kd, vd = dev(q, k, v)
    S = torch.zeros(w.B, w.H, w.Dk, w.Dv, device=DEV)
    z = torch.zeros(w.B, w.H, w.Dk, device=DEV)
    outs = torch.empty(w.steps, w.B, w.H, w.Dv, device=DEV)
    for t in range(w.steps):
        la.recurrent_step(qd[t], kd[t], vd[t], S, z, out=outs[t])
    torch.cuda.synchronize()
    # the causal form over the step sequence, computed by the oracle
    to_seq = lambda x: x.permute(1, 2, 0, 3).contiguous()
    ref = oracle.causal_recurrent(to_seq(q), to_seq(k), to_seq(v))
    check("decode outputs", to_seq(outs.cpu()), ref, 1e-4)
    phk = oracle.phi(to_seq(k))
    check("final S", S.cpu(), np.einsum("bhnd,bhnm->bhdm", phk, to_np(to_seq(v))), 1e-4)
    assert rel_per_head(z.cpu()[..., None], phk.sum(axis=2)[..., None]) < 1e-4


def _graph_decode(la, w, q, k, v):
    """All steps of the decode workload captured in one CUDA graph of single-step launches
    and replayed once, as the benchmark runs them; returns (outputs [T,B,H,Dv], S, z)."""
    qd, kd, vd = dev(q, k, v)
    S = torch.zeros(w.B, w.H, w.Dk, w.Dv, device=DEV)
    z = torch.zeros(w.B, w.H, w.Dk, device=DEV)
    outs = torch.empty(w.steps, w.B, w.H, w.Dv, device=DEV)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):  # first launch outside the capture
        la.recurrent_step(qd[0], kd[0], vd[0], S, z, out=outs[0])
    torch.cuda.synchronize()
    S.zero_()
    z.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for t in range(w.steps):
            la.recurrent_step(qd[t], kd[t], vd[t], S, z, out=outs[t])
    g.replay()
    torch.cuda.synchronize()
    return outs.cpu(), S.cpu(), z.cpu()


def test_decode_cifar_shape_all_steps_graph(la):
    """The 3072-step decode at B=64 H=8 D=32 (CIFAR-shaped pixel sequences), every step's
    output and the final (S, z) against the oracle, through the graph replay the bench times."""
    w = W.DECODE_CIFAR
    q, k, v = W.make_decode_inputs(w)
    outs, S, z = _graph_decode(la, w, q, k, v)
    to_seq = lambda x: x.permute(1, 2, 0, 3).contiguous()
    ref = oracle.causal_recurrent(to_seq(q), to_seq(k), to_seq(v))
    check("decode outputs, 3072 steps", to_seq(outs), ref, 1e-4)
    phk = oracle.phi(to_seq(k))
    check("final S", S, np.einsum("bhnd,bhnm->bhdm", phk, to_np(to_seq(v))), 1e-4)
    assert rel_per_head(z[..., None], phk.sum(axis=2)[..., None]) < 1e-4


def test_decode_resume_is_bit_exact(la):
    q, k, v = (t[:, :4] for t in W.make_decode_inputs(W.DECODE_MNIST, steps=40))
    qd, kd, vd = dev(q.contiguous(), k.contiguous(), v.contiguous())
    S = torch.zeros(4, 8, 32, 32, device=DEV)
    z = torch.zeros(4, 8, 32, device=DEV)
    full = [la.recurrent_step(qd[t], kd[t], vd[t], S, z).clone() for t in range(40)]
    S2 = torch.zeros_like(S)
    z2 = torch.zeros_like(z)
    for t in range(25):
        la.recurrent_step(qd[t], kd[t], vd[t], S2, z2)
    saved_S, saved_z = S2.cpu(), z2.cpu()          # checkpoint to the host and back
    S3, z3 = saved_S.to(DEV), saved_z.to(DEV)
    for t in range(25, 40):
        o = la.recurrent_step(qd[t], kd[t], vd[t], S3, z3)
        assert torch.equal(o, full[t])
    assert torch.equal(S3, S) and torch.equal(z3, z)


@pytest.mark.parametrize("B,H,N,Dk,Dv,dtype", [
    (1, 2, 4096, 128, 128, torch.bfloat16),   # tensor-core forward, several segments
    (1, 3, 100, 128, 128, torch.bfloat16),    # tensor-core forward, one segment
    (2, 2, 1500, 64, 64, torch.bfloat16),     # tensor-core forward, padded state records
    (2, 3, 700, 32, 64, torch.float32),       # CUDA-core forward
])
def test_prefill_state_then_decode(la, B, H, N, Dk, Dv, dtype):
    """The forward's final (S, z) is phi(K)^T V, phi(K)^T 1; decoding on from it continues the causal form."""
    T = 12
    q, k, v = W.random_case(400 + N, B, H, N + T, Dk, Dv, dtype=dtype, scale=Dk ** -0.5)
    qd, kd, vd = dev(q, k, v)
    pre = lambda x: x[:, :, :N].contiguous()
    o, S, z = la.causal_fwd(pre(qd), pre(kd), pre(vd), return_state=True)
    torch.cuda.synchronize()
    tol = tol_for(dtype)
    phk = oracle.phi(pre(k))
    check("final S", S.cpu(), np.einsum("bhnd,bhnm->bhdm", phk, to_np(pre(v))), tol)
    assert rel_per_head(z.cpu()[..., None], phk.sum(axis=2)[..., None]) < tol
    assert torch.equal(o, la.causal_fwd(pre(qd), pre(kd), pre(vd)))  # same output as without the state
    outs = [la.recurrent_step(qd[:, :, t].contiguous(), kd[:, :, t].contiguous(), vd[:, :, t].contiguous(), S, z)
            for t in range(N, N + T)]
    ref = oracle.causal_recurrent(q, k, v)[:, :, N:]
    check("decode after prefill", torch.stack(outs, 2), ref, tol)


def test_prefill_state_of_empty_sequence_is_zero(la):
    q = torch.randn(2, 3, 0, 32, device=DEV)
    o, S, z = la.causal_fwd(q, q, q, return_state=True)
    torch.cuda.synchronize()
    assert o.shape == (2, 3, 0, 32) and float(S.abs().max()) == 0.0 and float(z.abs().max()) == 0.0


@pytest.mark.parametrize("Dk,Dv,dtype", [(16, 16, torch.float32), (64, 32, torch.float32), (128, 128, torch.float32),
                                         (32, 64, torch.bfloat16), (128, 16, torch.bfloat16)])
def test_decode_head_sizes(la, Dk, Dv, dtype):
    B, H, T = 3, 5, 9
    q, k, v = W.random_case(41, B, H, T, Dk, Dv, dtype=dtype)
    S = torch.zeros(B, H, Dk, Dv, device=DEV)
    z = torch.zeros(B, H, Dk, device=DEV)
    qd, kd, vd = dev(q, k, v)
    outs = [la.recurrent_step(qd[:, :, t].contiguous(), kd[:, :, t].contiguous(), vd[:, :, t].contiguous(), S, z)
            for t in range(T)]
    o = torch.stack(outs, 2)
    check("decode", o, oracle.causal_recurrent(q, k, v), tol_for(dtype))


# ---------------------------------------------------------------- maximum sizes
SAMPLE_HEADS = [0, 1, 32767, 65534]


@pytest.mark.parametrize("N,D,dtype", [(70, 16, torch.float32), (129, 64, torch.bfloat16)])
def test_maximum_head_count(la, N, D, dtype):
    """B*H = 65535 (the largest head count, one grid row per head): forward and backward
    on the CUDA cores (fp32) and on the padded tensor-core path (bf16, D = 64); sampled
    heads against the oracle."""
    B = 65535
    q, k, v, dO = W.random_case(4242 + N, B, 1, N, D, D, dtype=dtype, scale=D ** -0.5, with_grad=True)
    qd, kd, vd, dOd = dev(q, k, v, dO)
    o = la.causal_fwd(qd, kd, vd)
    dq, dk, dv = la.causal_bwd(qd, kd, vd, dOd)
    torch.cuda.synchronize()
    idx = torch.tensor(SAMPLE_HEADS)
    sq, sk, sv, sdo = (t[idx] for t in (q, k, v, dO))
    tol = tol_for(dtype)
    check("o", o.cpu()[idx], oracle.causal_recurrent(sq, sk, sv), tol)
    ref = oracle.causal_bwd_recurrent(sq, sk, sv, sdo)
    check_all([("dq", dq.cpu()[idx], ref[0]), ("dk", dk.cpu()[idx], ref[1]), ("dv", dv.cpu()[idx], ref[2])], tol)


@pytest.mark.parametrize("N,D,dtype", [(70, 16, torch.float32), (129, 64, torch.bfloat16)])
def test_maximum_head_count_noncausal_and_retention(la, N, D, dtype):
    """B*H = 65535 for the non-causal forward and gradient and the retention forward (CUDA
    cores for fp32, the padded tensor-core path for bf16 D = 64); sampled heads against the
    oracle."""
    B = 65535
    q, k, v, dO = W.random_case(4545 + N, B, 1, N, D, D, dtype=dtype, scale=D ** -0.5, with_grad=True)
    qd, kd, vd, dOd = dev(q, k, v, dO)
    o = la.noncausal_fwd(qd, kd, vd).cpu()
    dq, dk, dv = (t.cpu() for t in la.noncausal_bwd(qd, kd, vd, dOd))
    del dOd
    gam = torch.tensor([0.95])
    orr = la.retention_fwd(qd, kd, vd, gam.to(DEV)).cpu()
    idx = torch.tensor(SAMPLE_HEADS)
    sq, sk, sv, sdo = (t[idx] for t in (q, k, v, dO))
    tol = tol_for(dtype)
    check("noncausal o", o[idx], oracle.noncausal_direct(sq, sk, sv), tol)
    ref = oracle.noncausal_bwd_direct(sq, sk, sv, sdo)
    check_all([("dq", dq[idx], ref[0]), ("dk", dk[idx], ref[1]), ("dv", dv[idx], ref[2])], tol)
    check("retention o", orr[idx], oracle.retention_recurrent(sq, sk, sv, gam), tol)


def test_maximum_head_count_decode(la):
    B, Dk, Dv = 65535, 16, 32
    q, k, v = W.random_case(4343, B, 1, 2, Dk, Dv)
    S = torch.zeros(B, 1, Dk, Dv, device=DEV)
    z = torch.zeros(B, 1, Dk, device=DEV)
    for t in range(2):
        out = la.recurrent_step(q[:, :, t].contiguous().to(DEV), k[:, :, t].contiguous().to(DEV),
                                v[:, :, t].contiguous().to(DEV), S, z)
    idx = torch.tensor(SAMPLE_HEADS)
    ref = oracle.causal_recurrent(q[idx], k[idx], v[idx])[:, :, 1]
    check("decode", out.cpu()[idx], ref, 1e-4)


def test_long_single_head_bf16(la):
    """One head of N = 2^19 positions (4096 chunks: the tensor-core planner gives 152
    segments of 27 chunks, one wave, and the scan runs over 152 records of one head): the
    forward against the oracle."""
    q, k, v = W.random_case(4444, 1, 1, 1 << 19, 64, 64, dtype=torch.bfloat16, scale=64 ** -0.5)
    o = la.causal_fwd(*dev(q, k, v))
    check("o", o, oracle.causal_recurrent(q, k, v), 2e-2)


def test_noncausal_fwd_long_sampled_heads(la):
    """The non-causal forward at B=2 H=16 N=65536 D=128 bf16 (segment sums and apply on the
    tensor cores): two heads against the oracle's associative form."""
    w = W.LONG_BF16
    q, k, v = W.make_inputs(w)
    o = la.noncausal_fwd(*dev(q, k, v)).cpu()
    for b, h in [(0, 0), (1, 15)]:
        sl = (slice(b, b + 1), slice(h, h + 1))
        check("head (%d,%d)" % (b, h), o[sl], oracle.noncausal_assoc(q[sl], k[sl], v[sl]), 2e-2)


def test_noncausal_bwd_long_sampled_heads(la):
    """The non-causal gradient at B=2 H=16 N=65536 D=128 bf16 (split segment sums, query and
    key passes on the tensor cores, the launch the bench times): two whole heads against the
    oracle's associative form of the same gradient."""
    w = W.LONG_BF16
    q, k, v, dO = W.make_inputs(w, with_grad=True)
    dq, dk, dv = (t.cpu() for t in la.noncausal_bwd(*dev(q, k, v, dO)))
    heads = [(0, 0), (1, 15)]
    sel = lambda t: torch.stack([t[b, h] for b, h in heads])[None]
    ref = oracle.noncausal_bwd_assoc(sel(q), sel(k), sel(v), sel(dO))
    check_all([(n, sel(a), b) for n, a, b in zip(("dq", "dk", "dv"), (dq, dk, dv), ref)], 2e-2)


# ---------------------------------------------------------------- one-launch forward (chained scan)
@pytest.mark.parametrize("B,H,N,D", [(1, 3, 4097, 128), (2, 2, 3000, 64), (1, 2, 1000, 128), (4, 8, 1024, 64),
                                     (1, 1, 1 << 16, 128)])
def test_one_launch_forward_matches_oracle_and_feeds_the_backward(la, B, H, N, D):
    """la_causal_fwd_fused against the oracle; the backward that reads its workspace gives
    la_causal_bwd's gradients bit for bit (its segment prefixes are the scan's exactly)."""
    q, k, v, dO = W.random_case(800 + N, B, H, N, D, D, dtype=torch.bfloat16, scale=D ** -0.5, with_grad=True)
    qd, kd, vd, dOd = dev(q, k, v, dO)
    ws_f = torch.empty(la.workspace_bytes(la.OP_CAUSAL_FWD, B, H, N, D, D, torch.bfloat16), dtype=torch.uint8,
                       device=DEV)
    o = la.causal_fwd(qd, kd, vd, workspace=ws_f, one_launch=True)
    got = la.causal_bwd(qd, kd, vd, dOd, fwd_workspace=ws_f)
    ref_b = la.causal_bwd(qd, kd, vd, dOd)
    torch.cuda.synchronize()
    check("o", o, oracle.causal_recurrent(q, k, v), 2e-2)
    for name, a, b in zip(("dq", "dk", "dv"), got, ref_b):
        assert torch.equal(a, b), name


def test_one_launch_forward_long_sampled_heads(la):
    """The one-launch forward at B=2 H=16 N=65536 D=128 (19 segments per head, four waves):
    two whole heads against the oracle."""
    w = W.LONG_BF16
    q, k, v = W.make_inputs(w)
    o = la.causal_fwd(*dev(q, k, v), one_launch=True).cpu()
    for b, h in [(0, 0), (1, 15)]:
        sl = (slice(b, b + 1), slice(h, h + 1))
        check("head (%d,%d)" % (b, h), o[sl], oracle.causal_recurrent(q[sl], k[sl], v[sl]), 2e-2)

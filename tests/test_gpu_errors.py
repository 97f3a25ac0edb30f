"""Error behaviour of the C ABI on a GPU: bad pointers and short workspaces are
refused before anything is launched, and the sticky device word stays clear."""
import ctypes

import pytest
import torch

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module")
def la():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import causal_linear_attention_phi_gb300 as la
    la.build.build_library()
    la.clear_error()
    return la


def _raw_fwd(la, q, k, v, o, ws, nbytes):
    s = la.Shape(*k.shape, v.shape[-1], la.LA_F32)
    p = lambda t: ctypes.c_void_p(t.data_ptr()) if isinstance(t, torch.Tensor) else ctypes.c_void_p(t)
    return la.library().la_causal_fwd(p(q), p(k), p(v), p(o), s, p(ws), nbytes, None)


def test_workspace_too_small(la):
    q = torch.randn(1, 2, 300, 32, device=DEV)
    need = la.workspace_bytes(la.OP_CAUSAL_FWD, 1, 2, 300, 32, 32, torch.float32)
    ws = torch.empty(need, dtype=torch.uint8, device=DEV)
    o = torch.empty_like(q)
    assert _raw_fwd(la, q, q, q, o, ws, need - 1) == 3
    assert _raw_fwd(la, q, q, q, o, 0, need) == 3
    assert _raw_fwd(la, q, q, q, o, ws, need) == 0


def test_binding_passes_real_workspace_size(la):
    q = torch.randn(1, 2, 300, 32, device=DEV)
    need = la.workspace_bytes(la.OP_CAUSAL_FWD, 1, 2, 300, 32, 32, torch.float32)
    short = torch.empty(need - 1, dtype=torch.uint8, device=DEV)
    with pytest.raises(la.LaError):
        la.causal_fwd(q, q, q, workspace=short)
    torch.cuda.synchronize()
    assert la.last_error() == 0


def test_bad_pointers(la):
    q = torch.randn(1, 2, 100, 32, device=DEV)
    o = torch.empty_like(q)
    need = la.workspace_bytes(la.OP_CAUSAL_FWD, 1, 2, 100, 32, 32, torch.float32)
    ws = torch.empty(need, dtype=torch.uint8, device=DEV)
    host = torch.randn(1, 2, 100, 32)
    assert _raw_fwd(la, host, q, q, o, ws, need) == 1            # host memory refused
    assert _raw_fwd(la, q, q, q, 0, ws, need) == 1               # NULL output
    assert _raw_fwd(la, q.data_ptr() + 4, q, q, o, ws, need) == 1  # misaligned
    with pytest.raises(la.LaError):
        la.causal_fwd(q, q, torch.randn(1, 2, 100, 48, device=DEV))  # unsupported Dv
    torch.cuda.synchronize()
    assert la.last_error() == 0


def test_timing_hooks(la):
    q = torch.randn(1, 2, 640, 64, device=DEV)
    la.timing_reset()
    la.timing_enable(True)
    try:
        la.causal_fwd(q, q, q)
        t = la.timing_read()
    finally:
        la.timing_enable(False)
    assert any(n.startswith("simt_causal_fwd") or n.startswith("tc_") for n in t)
    assert all(v[0] >= 1 and v[1] >= 0 for v in t.values())


def test_bounded_wait_times_out_and_the_context_stays_usable(la):
    """A device wait on a barrier that nothing completes gives up after its limit (about a
    second), records LA_ERR_TIMEOUT in the sticky word and lets the kernel end; no fault."""
    la.clear_error()
    la.selftest_bounded_wait()
    torch.cuda.synchronize()
    assert la.last_error() == 5  # LA_ERR_TIMEOUT
    la.clear_error()
    assert la.last_error() == 0
    q = torch.randn(1, 2, 200, 32, device=DEV)
    o = la.causal_fwd(q, q, q)
    torch.cuda.synchronize()
    assert torch.isfinite(o).all() and la.last_error() == 0


def test_chained_scan_wait_times_out_and_the_context_stays_usable(la):
    """The one-launch causal forward with segment 0 of head 0 withholding its sums (a
    test-only switch of the self-test entry point): the later segments of head 0 give up
    waiting after about a second and record LA_ERR_TIMEOUT; head 1 is complete and right;
    after clearing the word the same call without the switch is right for both heads."""
    import oracle
    from causal_linear_attention_phi_gb300 import workloads as W
    q, k, v = W.random_case(61, 1, 2, 1024, 128, 128, dtype=torch.bfloat16, scale=128 ** -0.5)
    qd, kd, vd = (t.to(DEV) for t in (q, k, v))
    la.clear_error()
    o = la.selftest_lookback_timeout(qd, kd, vd)
    torch.cuda.synchronize()
    assert la.last_error() == 5  # LA_ERR_TIMEOUT
    ref = oracle.causal_recurrent(q, k, v)
    from util import rel_per_head
    assert rel_per_head(o.cpu()[:, 1:], ref[:, 1:]) < 2e-2
    la.clear_error()
    o = la.causal_fwd(qd, kd, vd)
    torch.cuda.synchronize()
    assert la.last_error() == 0 and rel_per_head(o.cpu(), ref) < 2e-2


def test_lookback_selftest_refuses_shapes_without_a_chained_scan(la):
    q = torch.randn(1, 2, 1024, 64, device=DEV)          # fp32: the three-launch CUDA-core path
    with pytest.raises(la.LaError):
        la.selftest_lookback_timeout(q, q, q)
    qb = torch.randn(1, 2, 100, 128, device=DEV).bfloat16()  # one chunk: a single segment
    with pytest.raises(la.LaError):
        la.selftest_lookback_timeout(qb, qb, qb)


def test_tensor_core_fused_forward_is_one_kernel(la):
    """bf16 heads of 64 and 128: la_causal_fwd_fused launches one kernel (after a memset of its
    flags) and gives la_causal_fwd's outputs and segment records bit for bit."""
    for D in (64, 128):
        q, k, v = (torch.randn(2, 3, 3000, D, device=DEV).bfloat16() * 0.1 for _ in range(3))
        wsf = torch.empty(la.workspace_bytes(la.OP_CAUSAL_FWD, 2, 3, 3000, D, D, torch.bfloat16), dtype=torch.uint8,
                          device=DEV)
        ws3 = torch.empty_like(wsf)
        la.timing_reset()
        la.timing_enable(True)
        try:
            o1 = la.causal_fwd(q, k, v, workspace=wsf, one_launch=True)
            t = la.timing_read()
        finally:
            la.timing_enable(False)
        assert list(t) == ["tc_causal_fwd_fused"] and t["tc_causal_fwd_fused"][0] == 1, t
        o3 = la.causal_fwd(q, k, v, workspace=ws3)
        torch.cuda.synchronize()
        assert torch.equal(o1, o3)
        # the segment prefix records (the first region of the workspace) match bit for bit
        rec = _segment_records_bytes(la, 2, 3, 3000, D)
        assert torch.equal(wsf[:rec], ws3[:rec])


def _segment_records_bytes(la, B, H, N, D):
    """Bytes of the forward workspace's prefix records: B*H*P padded (128 x 128 + 128) fp32
    records, P read back from the retention workspace (same planner)."""
    P = la.workspace_bytes(la.OP_RETENTION_FWD, B, H, N, D, D, torch.bfloat16) // (B * H * 128 * 128 * 4)
    return B * H * P * (128 * 128 + 128) * 4

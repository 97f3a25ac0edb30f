"""la_causal_fwd_noalloc: the causal forward for callers that cannot allocate
device memory at call time (it keeps its scratch in a static device array).
Checked through the C ABI against la_causal_fwd, which takes a caller
workspace, on two calls in a row.  Collected last (file name) so that a run
stopping at the first failure has already run every other test."""
import ctypes

import pytest
import torch

from causal_linear_attention_phi_gb300 import workloads as W
from util import rel_per_head, tol_for

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module")
def la():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import causal_linear_attention_phi_gb300 as la
    la.build.build_library()
    lib = la.library()
    lib.la_causal_fwd_noalloc.argtypes = [ctypes.c_void_p] * 4 + [la.Shape, ctypes.c_void_p]
    lib.la_causal_fwd_noalloc.restype = ctypes.c_int
    return la


def _noalloc(la, q, k, v, o):
    s = la.Shape(*q.shape, v.shape[-1], la.LA_BF16 if q.dtype == torch.bfloat16 else la.LA_F32)
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return la.library().la_causal_fwd_noalloc(p(q), p(k), p(v), p(o), s, st)


@pytest.mark.parametrize("B,H,N,D,dtype", [(2, 16, 8192, 128, torch.bfloat16),   # tensor-core path, segments capped
                                           (2, 8, 5000, 64, torch.bfloat16),     # tensor-core path, padded head
                                           (1, 2, 1000, 64, torch.float32)])      # CUDA-core path
def test_noalloc_matches_workspace_entry_twice(la, B, H, N, D, dtype):
    scale = 128 ** -0.5 if dtype == torch.bfloat16 else 1.0
    for call, seed in enumerate((11, 12)):  # two calls in a row, different inputs
        q, k, v = (t.to(DEV) for t in W.random_case(seed, B, H, N, D, D, dtype=dtype, scale=scale))
        ref = la.causal_fwd(q, k, v)
        out = torch.full_like(v, float("nan"))
        assert _noalloc(la, q, k, v, out) == 0, la.library().la_error_detail()
        torch.cuda.synchronize()
        e = rel_per_head(out.cpu(), ref.cpu())
        assert e <= tol_for(dtype), "call %d: rel err %.3e" % (call, e)
    assert la.last_error() == 0


def test_noalloc_rejects_sizes_beyond_its_scratch(la):
    # B*H = 256 heads of 128 x 128 fp32 states need 256 * 16512 * 4 bytes > 16 MiB
    q = torch.zeros(4, 64, 4, 128, dtype=torch.bfloat16, device=DEV)
    o = torch.empty_like(q)
    assert _noalloc(la, q, q, q, o) == 3
    assert b"16 MiB" in la.library().la_error_detail()

"""la_causal_fwd_noalloc: the causal forward for callers that cannot allocate
device memory at call time (it keeps its scratch in a static device array).
Checked through the C ABI against la_causal_fwd, which takes a caller
workspace, on two calls in a row, and on one sampled head against the fp64
oracle.  Collected last (file name) so that a run stopping at the first
failure has already run every other test."""
import ctypes

import pytest
import torch

import oracle
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


# The regular plan of the first two cases does not fit the 16 MiB array: (2,16,8192,128) has
# 32 segments of 32 records of 66048 bytes (2.1 MB per segment), capped to 7; (1,16,65536,128)
# has 19 segments, capped to 15.  The padded head of 64 keeps 128-wide records as well.
@pytest.mark.parametrize("B,H,N,D,dtype", [(2, 16, 8192, 128, torch.bfloat16),   # tensor-core path, segments capped
                                           (1, 16, 65536, 128, torch.bfloat16),  # the same at the long length
                                           (2, 8, 5000, 64, torch.bfloat16),     # tensor-core path, padded head
                                           (1, 2, 1000, 64, torch.float32)])      # CUDA-core path
def test_noalloc_matches_workspace_entry_twice(la, B, H, N, D, dtype):
    scale = 128 ** -0.5 if dtype == torch.bfloat16 else 1.0
    for call, seed in enumerate((11, 12)):  # two calls in a row, different inputs
        qc, kc, vc = W.random_case(seed, B, H, N, D, D, dtype=dtype, scale=scale)
        q, k, v = (t.to(DEV) for t in (qc, kc, vc))
        ref = la.causal_fwd(q, k, v)
        out = torch.full_like(v, float("nan"))
        assert _noalloc(la, q, k, v, out) == 0, la.library().la_error_detail()
        torch.cuda.synchronize()
        out = out.cpu()
        e = rel_per_head(out, ref.cpu())
        assert e <= tol_for(dtype), "call %d: rel err %.3e against la_causal_fwd" % (call, e)
        b, h = B - 1, H - 1  # the last head: its state crosses every segment boundary of the plan
        sl = (slice(b, b + 1), slice(h, h + 1))
        e = rel_per_head(out[sl], oracle.causal_recurrent(qc[sl], kc[sl], vc[sl]))
        assert e <= tol_for(dtype), "call %d: rel err %.3e against the oracle" % (call, e)
    assert la.last_error() == 0


@pytest.mark.parametrize("shape,dtype", [((4, 64, 4, 128), torch.bfloat16),   # B*H = 256 records of 66048 bytes
                                         ((5, 51, 4, 64), torch.bfloat16),    # B*H = 255, padded 128-wide records
                                         ((1, 1009, 4, 64), torch.float32)])  # B*H = 1009 records of 16640 bytes
def test_noalloc_rejects_sizes_beyond_its_scratch(la, shape, dtype):
    q = torch.zeros(*shape, dtype=dtype, device=DEV)
    o = torch.empty_like(q)
    assert _noalloc(la, q, q, q, o) == 3
    assert b"16 MiB" in la.library().la_error_detail()


@pytest.mark.parametrize("shape,dtype", [((2, 127, 4, 64), torch.bfloat16),   # B*H = 254: the largest that fits
                                         ((1, 1008, 4, 64), torch.float32)])
def test_noalloc_accepts_the_largest_size_that_fits(la, shape, dtype):
    qc, kc, vc = W.random_case(13, *shape, shape[-1], dtype=dtype, scale=0.25)
    q, k, v = (t.to(DEV) for t in (qc, kc, vc))
    out = torch.full_like(v, float("nan"))
    assert _noalloc(la, q, k, v, out) == 0, la.library().la_error_detail()
    torch.cuda.synchronize()
    assert rel_per_head(out.cpu(), la.causal_fwd(q, k, v).cpu()) <= tol_for(dtype)

"""The debug build (device-side index checks, the stand-in for a memory checker):
the small parity cases run under it with the sticky error word still clear.

The debug library is loaded in a child process (LA_DEBUG=1 selects it there), so
this process keeps the regular build."""
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu
HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def run_debug_cases():
    """Runs in the child: causal forward and backward (CUDA-core fp32, tensor-core bf16 at
    heads of 64 and 128, several segments and ragged tails), the non-causal forward and
    gradient, retention and both decode steps, each against the oracle, then the error word."""
    import numpy as np
    import oracle
    import causal_linear_attention_phi_gb300 as la
    from causal_linear_attention_phi_gb300 import workloads as W
    from util import rel_per_head, tol_for
    assert la.version().endswith("-debug"), la.version()
    la.clear_error()
    dev = "cuda:0"
    d = lambda *ts: [t.to(dev) for t in ts]
    for (B, H, N, D, dt) in [(1, 2, 200, 32, torch.float32), (1, 2, 1000, 64, torch.bfloat16),
                             (2, 1, 1300, 128, torch.bfloat16), (1, 3, 129, 128, torch.bfloat16)]:
        q, k, v, dO = W.random_case(900 + N, B, H, N, D, D, dtype=dt, scale=D ** -0.5, with_grad=True)
        o = la.causal_fwd(*d(q, k, v))
        dq, dk, dv = la.causal_bwd(*d(q, k, v, dO))
        onc = la.noncausal_fwd(*d(q, k, v))
        ndq, ndk, ndv = la.noncausal_bwd(*d(q, k, v, dO))
        g = torch.linspace(0.9, 1.0, H)
        orr = la.retention_fwd(*d(q, k, v), g.to(dev))
        torch.cuda.synchronize()
        tol = tol_for(dt)
        ref = oracle.causal_bwd_recurrent(q, k, v, dO)
        nref = oracle.noncausal_bwd_direct(q, k, v, dO)
        pairs = [(o, oracle.causal_recurrent(q, k, v)), (dq, ref[0]), (dk, ref[1]), (dv, ref[2]),
                 (onc, oracle.noncausal_assoc(q, k, v)), (ndq, nref[0]), (ndk, nref[1]), (ndv, nref[2]),
                 (orr, oracle.retention_recurrent(q, k, v, g))]
        for i, (a, b) in enumerate(pairs):
            e = rel_per_head(a.cpu(), b)
            assert e <= tol, "case %s output %d: rel err %.3e" % ((B, H, N, D, dt), i, e)
        assert la.last_error() == 0, la.library().la_error_detail()
    # decode steps (causal and retention) from zero states
    q, k, v = W.random_case(5, 3, 4, 6, 32, 32)
    S = torch.zeros(3, 4, 32, 32, device=dev)
    z = torch.zeros(3, 4, 32, device=dev)
    Sr = torch.zeros_like(S)
    g = torch.full((4,), 0.9)
    outs, routs = [], []
    for t in range(6):
        qt, kt, vt = (x[:, :, t].contiguous().to(dev) for x in (q, k, v))
        outs.append(la.recurrent_step(qt, kt, vt, S, z))
        routs.append(la.retention_step(qt, kt, vt, g.to(dev), Sr))
    assert rel_per_head(torch.stack(outs, 2).cpu(), oracle.causal_recurrent(q, k, v)) < 1e-4
    assert rel_per_head(torch.stack(routs, 2).cpu(), oracle.retention_recurrent(q, k, v, g)) < 1e-4
    st = la.last_error()
    assert st == 0, "sticky status %d: %s" % (st, la.library().la_error_detail())
    print("debug build cases ok")


def test_parity_cases_under_the_debug_build():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from causal_linear_attention_phi_gb300 import build
    build.build_library(debug=True)
    env = dict(os.environ, LA_DEBUG="1")
    code = "import sys; sys.path[:0] = [%r, %r]; import test_gpu_debug_build as t; t.run_debug_cases()" % (HERE, ROOT)
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env, timeout=900)
    assert r.returncode == 0 and "debug build cases ok" in r.stdout, r.stdout[-2000:] + r.stderr[-4000:]

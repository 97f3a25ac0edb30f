"""The C ABI on the CPU: the library builds, loads, exports every symbol that
include/la.h declares, and rejects bad arguments before touching a GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", f) for f in os.listdir(os.path.join(ROOT, "include")) if f.endswith(".h")]


@pytest.fixture(scope="module")
def la():
    from causal_linear_attention_phi_gb300 import build
    build.build_library()
    import causal_linear_attention_phi_gb300 as la
    la.library()
    return la


def declared_functions():
    names = set()
    for h in HEADERS:
        src = open(h).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        src = re.sub(r"//[^\n]*", "", src)
        for m in re.finditer(r"^\s*[A-Za-z_][\w\s\*]*?\b(la_\w+)\s*\(", src, flags=re.M):
            names.add(m.group(1))
    return sorted(names)


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("la_noncausal_fwd", "la_causal_fwd", "la_causal_bwd", "la_recurrent_step",
                     "la_retention_fwd", "la_retention_step",
                     "la_workspace_bytes", "la_last_error", "la_status_string"):
        assert required in names


def test_every_declared_symbol_is_exported(la):
    lib = ctypes.CDLL(la.build.LIB_PATH)
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_static_strings(la):
    lib = la.library()
    assert lib.la_status_string(0) == b"LA_OK"
    assert b"WORKSPACE" in lib.la_status_string(3)
    assert lib.la_version().decode().count(".") == 2


def test_workspace_bytes_is_pure(la):
    import torch
    ws = la.workspace_bytes(la.OP_CAUSAL_FWD, 2, 16, 65536, 128, 128, torch.bfloat16)
    assert ws > 0 and ws == la.workspace_bytes(la.OP_CAUSAL_FWD, 2, 16, 65536, 128, 128, torch.bfloat16)
    assert la.workspace_bytes(la.OP_CAUSAL_BWD, 2, 16, 65536, 128, 128, torch.bfloat16) > ws
    assert la.workspace_bytes(la.OP_CAUSAL_FWD, 2, 16, 0, 128, 128, torch.bfloat16) == 0
    assert la.workspace_bytes(la.OP_CAUSAL_FWD, 2, 16, 64, 48, 128, torch.bfloat16) == 0   # unsupported size
    assert la.workspace_bytes(99, 2, 16, 64, 64, 64, torch.bfloat16) == 0                   # bad op
    # retention records hold S only: smaller than the CUDA-core causal forward's (S, z) records
    rw = la.workspace_bytes(la.OP_RETENTION_FWD, 2, 16, 65536, 128, 128, torch.float32)
    assert 0 < rw < la.workspace_bytes(la.OP_CAUSAL_FWD, 2, 16, 65536, 128, 128, torch.float32)


def _call_fwd(la, shape, ptr=0):
    lib = la.library()
    s = la.Shape(*shape)
    p = ctypes.c_void_p(ptr)
    return lib.la_causal_fwd(p, p, p, p, s, p, 0, None)


def test_host_side_rejections(la):
    # each of these returns before any device call, so it runs without a GPU
    assert _call_fwd(la, (-1, 1, 8, 16, 16, 0)) == 1        # negative size
    assert _call_fwd(la, (1, 1, 8, 16, 16, 7)) == 1         # bad dtype
    assert _call_fwd(la, (1, 1, 8, 48, 16, 0)) == 2         # head size not in {16,32,64,128}
    assert _call_fwd(la, (1, 1, 8, 16, 256, 0)) == 2
    assert _call_fwd(la, (256, 256, 8, 16, 16, 0)) == 2     # B*H > 65535
    assert _call_fwd(la, (1, 1, 0, 16, 16, 0)) == 0         # empty: a no-op
    assert _call_fwd(la, (0, 4, 8, 16, 16, 1)) == 0
    lib = la.library()
    assert b"head sizes" in lib.la_error_detail() or True


def test_retention_host_side_rejections(la):
    # shape checks come before any device call, so these run without a GPU
    lib = la.library()
    p = ctypes.c_void_p(0)

    def fwd(shape):
        return lib.la_retention_fwd(p, p, p, p, p, p, la.Shape(*shape), p, 0, None)

    def step(shape):
        return lib.la_retention_step(p, p, p, p, p, p, la.Shape(*shape), None)

    assert fwd((-1, 1, 8, 16, 16, 0)) == 1      # negative size
    assert fwd((1, 1, 8, 16, 16, 9)) == 1       # bad dtype
    assert fwd((1, 1, 8, 48, 16, 0)) == 2       # head size not in {16, 32, 64, 128}
    assert fwd((0, 4, 8, 16, 16, 1)) == 0       # no heads: a no-op
    assert step((1, 1, 1, 16, 256, 0)) == 2
    assert step((0, 2, 1, 16, 16, 0)) == 0
    assert step((-2, 2, 1, 16, 16, 0)) == 1


def test_retention_workspace_is_pure(la):
    import torch
    a = la.workspace_bytes(la.OP_RETENTION_FWD, 2, 16, 65536, 128, 128, torch.bfloat16)
    assert a > 0 and a == la.workspace_bytes(la.OP_RETENTION_FWD, 2, 16, 65536, 128, 128, torch.bfloat16)
    assert la.workspace_bytes(la.OP_RETENTION_FWD, 2, 16, 0, 128, 128, torch.bfloat16) == 0
    # same planner as the causal forward, records of S only (no z): strictly smaller
    assert a < la.workspace_bytes(la.OP_CAUSAL_FWD, 2, 16, 65536, 128, 128, torch.bfloat16)


def test_product_path_fails_loudly_without_library(tmp_path):
    import causal_linear_attention_phi_gb300 as la
    saved = la._lib
    try:
        la._lib = None
        with pytest.raises(RuntimeError):
            la.library(str(tmp_path / "missing.so"))
    finally:
        la._lib = saved


def _segments(la, B, H, N, D=128):
    """Segments per head of the tensor-core plan, read back from the retention forward's
    workspace (the same planner; one padded 128 x 128 fp32 state record per segment and head)."""
    import torch
    rec = 128 * 128 * 4
    ws = la.workspace_bytes(la.OP_RETENTION_FWD, B, H, N, D, D, torch.bfloat16)
    assert ws % (B * H * rec) == 0
    return ws // (B * H * rec)


def test_causal_forward_workspace_holds_the_chained_scan(la):
    """The one-launch forward's workspace: the segment prefixes, the segments' own sums (both
    B*H*P padded records) and B*H*P + 1 flag words, each region 256-byte aligned."""
    import torch
    for B, H, N in [(2, 16, 65536), (1, 8, 1024), (65535, 1, 129)]:
        P = _segments(la, B, H, N)
        seg = -(-(B * H * P * (128 * 128 + 128) * 4) // 256) * 256
        flags = -(-((B * H * P + 1) * 4) // 256) * 256
        assert la.workspace_bytes(la.OP_CAUSAL_FWD, B, H, N, 128, 128, torch.bfloat16) == 2 * seg + flags


@pytest.mark.parametrize("B,H,N", [(2, 16, 65536), (1, 16, 32768), (1, 8, 65536), (1, 1, 1 << 19),
                                   (4, 8, 1024), (65535, 1, 129), (1, 1, 1)])
def test_planner_segments(la, B, H, N):
    # host logic only: every segment gets the same chunk count but possibly the last, none is
    # empty, and the grid stays within 8 waves of the 152 SMs (one CTA per SM)
    BH, nchunks = B * H, -(-N // 128)
    P = _segments(la, B, H, N)
    cps = -(-nchunks // P)
    assert 1 <= P <= nchunks and -(-nchunks // cps) == P
    assert BH * P <= 8 * 152 or P == 1


def test_planner_fills_whole_waves_at_the_long_shape(la):
    # B=2 H=16 N=65536: 512 chunks per head as 19 segments of 27 (the last 26), 608 CTAs,
    # exactly 4 waves of 152; one head of 2^19 positions: 152 segments of 27, one wave
    assert _segments(la, 2, 16, 65536) == 19
    assert _segments(la, 1, 1, 1 << 19) == 152


def test_bench_refuses_a_gpu_count_it_was_not_launched_with():
    """bench.py --gpus N runs one process per GPU: without N ranks it exits non-zero
    instead of timing one GPU under another GPU count."""
    import subprocess
    import sys
    env = dict(os.environ)
    env.pop("WORLD_SIZE", None)
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--gpus", "2", "--steps", "1"],
                       capture_output=True, text=True, env=env, timeout=300)
    assert r.returncode != 0 and "WORLD_SIZE=1" in r.stderr


def test_debug_build_flag_reaches_nvcc_and_the_library():
    """build_library(debug=True) compiles with -DLA_DEBUG (and relocatable device code, so the
    checks of every translation unit reach one error word) into a library that reports a
    '-debug' version; the regular library does not."""
    from causal_linear_attention_phi_gb300 import build
    cmd = build.nvcc_command("x.cu", "x.o", debug=True)
    assert "-DLA_DEBUG" in cmd and "-rdc=true" in cmd
    assert "-DLA_DEBUG" not in build.nvcc_command("x.cu", "x.o")
    path = build.build_library(debug=True)
    lib = ctypes.CDLL(path)
    lib.la_version.restype = ctypes.c_char_p
    assert lib.la_version().decode().endswith("-debug")
    reg = ctypes.CDLL(build.build_library())
    reg.la_version.restype = ctypes.c_char_p
    assert not reg.la_version().decode().endswith("-debug")
    lib.la_status_string.restype = ctypes.c_char_p
    assert b"LA_ERR_BOUNDS" in lib.la_status_string(6)

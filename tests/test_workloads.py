"""The seeded input generators: deterministic, right shapes and dtypes."""
import torch

from causal_linear_attention_phi_gb300 import workloads as W


def test_deterministic_and_shaped():
    a = W.make_inputs(W.SMALL_F32)
    b = W.make_inputs(W.SMALL_F32)
    for x, y in zip(a, b):
        assert torch.equal(x, y)
    assert a[0].shape == (1, 2, 64, 16) and a[0].dtype == torch.float32
    q, k, v, dO = W.make_inputs(W.FWD_BF16, with_grad=True, N=128)
    assert q.dtype == torch.bfloat16 and q.shape == (4, 8, 128, 64) and dO.shape == v.shape
    # the N(0,1)/8 scale of the bf16 forward workload
    assert 0.08 < float(q.float().std()) < 0.17
    q, k, v = W.make_decode_inputs(W.DECODE_MNIST, steps=3)
    assert q.shape == (3, 64, 8, 32)


def test_sweep_lengths():
    assert W.SWEEP_NS[0] == 512 and W.SWEEP_NS[-1] == 65536
    assert W.sweep(4096).N == 4096 and W.sweep(4096).Dk == 64

"""GPU parity of the attention backward (dQ, dK, dV through the C ABI) against
the fp64 oracle's chain-rule gradients on the same bf16/fp16 inputs.

Tolerance. The GPU rounds P and dS to the input dtype before the three
gradient GEMMs (bf16: relative 2^-9 per element, fp16: 2^-12), uses the
forward's rounded O in D = rowsum(dO * O), and rounds the outputs; all sums
run in fp32. Independent element roundings of relative size u give gradient
errors of order u times the gradient's own scale, so the test bounds the
RMS error by 8u * RMS(reference) and the largest error by 64u * max|reference|
per tensor (u = 2^-9 for bf16, 2^-12 for fp16), plus absolute floors of 1e-5
(RMS) and 1e-4 (max) for gradients that vanish exactly (a single key gives
dS = 0 while D is formed from the rounded O)."""
import numpy as np
import pytest
import torch

import attn_inputs as gen
import oracle as O

pytestmark = pytest.mark.gpu


def _check_grads(got3, ref3, u, what=""):
    for name, g, want in zip(("dq", "dk", "dv"), got3, ref3):
        err = g - want
        rms_ref = float(np.sqrt((want ** 2).mean()))
        rms = float(np.sqrt((err ** 2).mean()))
        mx = float(np.abs(err).max())
        assert np.isfinite(g).all(), name
        assert rms <= 8 * u * rms_ref + 1e-5 and mx <= 64 * u * float(np.abs(want).max()) + 1e-4, \
            f"{what} {name}: rms {rms:.3e} (ref rms {rms_ref:.3e}), max {mx:.3e} (ref max {np.abs(want).max():.3e})"


def _gpu_grads(q, k, v, do, causal):
    import exact_attention_45_gb300 as A
    dq_, dk_, dv_ = (t.cuda() for t in (q, k, v))
    o, lse = A.attn_fwd(dq_, dk_, dv_, causal=causal)
    dq, dk, dv = A.attn_bwd(dq_, dk_, dv_, o, lse, do.cuda(), causal=causal)
    torch.cuda.synchronize()
    assert A.attn_get_device_error() == 0
    return tuple(t.float().cpu().numpy() for t in (dq, dk, dv))


def _run(B, N, H, Hkv, d, causal, dtype="bf16", seed=0):
    q, k, v = gen.qkv_fixed(B, N, H, Hkv, d, seed=seed, dtype=dtype)
    do = gen.qkv_fixed(B, N, H, H, d, seed=seed + 100, dtype=dtype)[0]
    got = _gpu_grads(q, k, v, do, causal)
    ref = O.attention_backward(q, k, v, do, causal=causal)
    _check_grads(got, ref, 2.0 ** -9 if dtype == "bf16" else 2.0 ** -12)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 77, 128, 300, 513])
def test_bwd_shapes_with_ragged_tails(d, causal, N):
    _run(2, N, 4, 2, d, causal, seed=N + d)


@pytest.mark.parametrize("d", [64, 128])
def test_bwd_fp16(d):
    _run(1, 260, 2, 1, d, True, dtype="fp16", seed=3)
    _run(1, 200, 2, 2, d, False, dtype="fp16", seed=4)


def test_bwd_mqa_and_longer_sequence():
    _run(1, 2048, 4, 1, 128, True, seed=9)
    _run(1, 1024, 2, 2, 128, False, seed=10)


@pytest.mark.parametrize("causal", [False, True])
def test_bwd_benchmark_shape_sampled_heads(causal):
    # the benchmarked shape (B=4, N=4096, H=16, d=128) runs whole on the GPU;
    # with H = Hkv the gradients of one (batch, head) depend on that head
    # only, so the oracle checks three whole heads of it
    B, N, H, d = 4, 4096, 16, 128
    q, k, v = gen.qkv_fixed(B, N, H, H, d, seed=21)
    do = gen.qkv_fixed(B, N, H, H, d, seed=121)[0]
    got = _gpu_grads(q, k, v, do, causal)
    for b, h in ((0, 0), (2, 7), (3, 15)):
        sl = (slice(b, b + 1), slice(None), slice(h, h + 1))
        ref = O.attention_backward(q[sl], k[sl], v[sl], do[sl], causal=causal)
        _check_grads(tuple(g[sl] for g in got), ref, 2.0 ** -9, what=f"b{b} h{h}")

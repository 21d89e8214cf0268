"""Helpers shared by the GPU parity tests: run the CUDA path, run the oracle
on the same host inputs, compare with the stated tolerances."""
from __future__ import annotations

import numpy as np
import torch

import attn_inputs as gen
import oracle as O

# Tolerances for BF16/FP16 with N(0,1) inputs (stated for the fp64 oracle):
# max |err| <= 1e-2, RMS err <= 2e-3 on O; |err| <= 1e-3 on the logsumexp.
TOL_MAX, TOL_RMS, TOL_LSE = 1e-2, 2e-3, 1e-3


def errors(o_gpu: np.ndarray, o_ref: np.ndarray, l_gpu: np.ndarray, l_ref: np.ndarray):
    d = o_gpu.astype(np.float64) - o_ref
    return (float(np.abs(d).max()) if d.size else 0.0,
            float(np.sqrt((d ** 2).mean())) if d.size else 0.0,
            float(np.abs(l_gpu.astype(np.float64) - l_ref).max()) if l_ref.size else 0.0)


def assert_close(o_gpu, o_ref, l_gpu, l_ref, tol=(TOL_MAX, TOL_RMS, TOL_LSE), what=""):
    mx, rms, le = errors(o_gpu, o_ref, l_gpu, l_ref)
    assert np.all(np.isfinite(o_gpu)), f"{what}: non-finite output"
    assert mx <= tol[0] and rms <= tol[1] and le <= tol[2], \
        f"{what}: max {mx:.3e} (<= {tol[0]}), rms {rms:.3e} (<= {tol[1]}), lse {le:.3e} (<= {tol[2]})"
    return mx, rms, le


def run_fixed(q, k, v, causal, scale=None):
    import exact_attention_45_gb300 as A
    dq, dk, dv = (t.cuda() for t in (q, k, v))
    o, lse = A.attn_fwd(dq, dk, dv, causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert A.attn_get_device_error() == 0
    return o, lse


def run_varlen(q, k, v, cu, causal, scale=None):
    import exact_attention_45_gb300 as A
    dq, dk, dv = (t.cuda() for t in (q, k, v))
    dcu = torch.as_tensor(cu, dtype=torch.int32).cuda()
    o, lse = A.attn_fwd_varlen(dq, dk, dv, dcu, causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert A.attn_get_device_error() == 0
    return o, lse


def check_fixed_full(B, N, H, Hkv, d, causal, dtype="bf16", seed=0):
    q, k, v = gen.qkv_fixed(B, N, H, Hkv, d, seed=seed, dtype=dtype)
    o, lse = run_fixed(q, k, v, causal)
    o_ref, l_ref = O.attention(q, k, v, causal=causal)
    return assert_close(o.float().cpu().numpy(), o_ref, lse.cpu().numpy(), l_ref,
                        what=f"B{B} N{N} H{H}/{Hkv} d{d} causal={causal} {dtype}")


def check_fixed_sampled(B, N, H, Hkv, d, causal, count=256, seed=0, dtype="bf16"):
    """Full-size launch; the oracle computes a seeded sample of rows."""
    q, k, v = gen.qkv_fixed(B, N, H, Hkv, d, seed=seed, dtype=dtype)
    o, lse = run_fixed(q, k, v, causal)
    o_h = o.float().cpu().numpy()
    l_h = lse.cpu().numpy()
    assert np.isfinite(o_h).all() and np.isfinite(l_h).all()
    rs, rh, ri = gen.sample_rows([N] * B, H, count, seed=seed)
    o_ref, l_ref = O.attention(q, k, v, causal=causal, rows=(rs, rh, ri))
    return assert_close(o_h[rs, ri, rh], o_ref, l_h[rs, rh, ri], l_ref,
                        what=f"sampled B{B} N{N} H{H}/{Hkv} d{d} causal={causal}")

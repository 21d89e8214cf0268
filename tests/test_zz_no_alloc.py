"""GPU test of attn_fwd_fp8_auto_noalloc, the FP8 entry point for callers that
may not allocate device memory (hosts that own all device memory through
their own pool and forbid cudaMalloc/cudaFree, whose device-wide
synchronisation and possible out-of-memory failure they cannot accept on the
request path). It keeps its quantised tensors in a fixed 16 MiB scratch array
inside the library instead of a caller workspace.

Called through the C ABI with raw pointers; two calls in a row must give the
same output as attn_fwd_fp8_auto with a caller-provided workspace. This file
is named so pytest collects it last.
"""
import math

import pytest
import torch

import attn_inputs as gen

pytestmark = pytest.mark.gpu

B, N, H, HKV, D = 2, 384, 4, 2, 128


def _run_noalloc(lib, q, k, v, causal, mode, rotate, seed):
    o = torch.empty((B, N, H, D), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    rc = lib.attn_fwd_fp8_auto_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                       B, H, HKV, N, D, int(causal), 1.0 / math.sqrt(D), mode, int(rotate), seed,
                                       torch.cuda.current_stream().cuda_stream)
    assert rc == 0, lib.attn_last_error_message()
    return o, lse


@pytest.mark.parametrize("causal", [False, True])
def test_noalloc_matches_workspace_entry_point(causal):
    import exact_attention_45_gb300 as A
    lib = A.capi()
    q, k, v = (t.cuda() for t in gen.qkv_fixed(B, N, H, HKV, D, seed=11, dist="outlier"))
    assert A.attn_fp8_workspace_size(B, H, HKV, N, D, "block") <= 16 << 20
    o_ref, l_ref = A.attn_fwd_fp8_auto(q, k, v, causal=causal, mode="block", rotate=True, hadamard_seed=7)
    for _ in range(2):                      # the scratch keeps the previous call's contents
        o, lse = _run_noalloc(lib, q, k, v, causal, 1, True, 7)
        torch.cuda.synchronize()
        assert A.attn_get_device_error() == 0
        # same kernels on the same inputs: identical up to the tolerance the
        # FP8 parity tests use (bitwise equality is expected and checked first)
        if not torch.equal(o, o_ref):
            err = (o.float() - o_ref.float()).abs()
            assert float((err / (1e-2 + 4e-3 * o_ref.float().abs())).max()) <= 1.0
        assert torch.allclose(lse, l_ref, atol=2e-3, rtol=0)


def test_noalloc_rejects_shapes_beyond_the_scratch():
    import exact_attention_45_gb300 as A
    lib = A.capi()
    # 16 sequences of 4096 tokens x 16 heads x d=128 needs far more than 16 MiB;
    # the size check happens on the host before anything touches the pointers
    rc = lib.attn_fwd_fp8_auto_noalloc(None, None, None, None, None, 16, 16, 16, 4096, 128, 0, 0.088, 1, 1, 0,
                                       None)
    assert rc == A.ATTN_ERR_INVALID_ARG
    assert b"16777216" in lib.attn_last_error_message()

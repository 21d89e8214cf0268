"""GPU parity of the FP8 path through the C ABI.

* pre-pass (rotation + quantisation): bit-exact codes and scales against the
  oracle's statement of the same definition;
* FP8 forward on those codes: against the oracle's fp64 emulation of the
  method's steps (online softmax over 128-key blocks with a lazy running
  maximum, margin 2^8; p = 2^(t - m) <= 2^8 rounded to e4m3 with multiplier 1
  for P V; the normaliser from the unrounded p);
* the error gate on the outlier distribution (RMS against exact fp64
  attention, all four quantisation variants) is in test_gpu_fp8_fullsize.py.
"""
import numpy as np
import pytest
import torch

import attn_inputs as gen
import oracle as O

pytestmark = pytest.mark.gpu

# Where the kernel's fp32 scores and the oracle's fp64 ones put some p on
# opposite sides of an e4m3 rounding midpoint, both roundings are the method's
# result: the oracle reports, per output element, what rounding each p within
# FLIP_TOL (relative) of a midpoint the other way would change, and the bound
# grants that. 2^-12 is far above the fp32 score error at these sizes (the
# straddles seen were within 2^-22) and covers well under 1% of the p values.
FLIP_TOL = 2.0 ** -12


def _prepass_gpu(q, k, v, mode, rotate, seed):
    import exact_attention_45_gb300 as A
    pre = A.attn_fp8_prepass(q.cuda(), k.cuda(), v.cuda(), mode=mode, rotate=rotate, hadamard_seed=seed)
    torch.cuda.synchronize()
    assert A.attn_get_device_error() == 0
    return pre


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("mode", ["block", "tensor"])
@pytest.mark.parametrize("rotate", [True, False])
def test_prepass_bit_exact(d, mode, rotate):
    B, N, H, Hkv = 2, 300, 4, 2
    q, k, v = gen.qkv_fixed(B, N, H, Hkv, d, seed=d, dist="outlier")
    pre = _prepass_gpu(q, k, v, mode, rotate, seed=5)
    ref = O.fp8_prepass(q, k, v, mode=mode, rotate=rotate, seed=5)
    assert np.array_equal(pre["q8"].cpu().numpy(), ref["q8"])
    assert np.array_equal(pre["k8"].cpu().numpy(), ref["k8"])
    vt = pre["vt8"].cpu().numpy()
    assert np.array_equal(vt[..., :N], ref["vt8"])
    assert np.all(vt[..., N:] == 0)
    for name in ("sq", "sk", "sv"):
        assert np.array_equal(pre[name].cpu().numpy(), ref[name]), name


@pytest.mark.parametrize("d,B", [(64, 8), (128, 4), (256, 2)])
def test_prepass_persistent_many_tiles_bit_exact(d, B):
    # block scales at head dims 64, 128 and 256 run on persistent kernels fed by a
    # ring of TMA copies: enough 128-row tiles that every CTA goes around the
    # ring more than once, the last block of each sequence ragged (2000 rows)
    N, H, Hkv = 2000, 8, 4
    q, k, v = gen.qkv_fixed(B, N, H, Hkv, d, seed=20 + d, dist="outlier")
    pre = _prepass_gpu(q, k, v, "block", True, seed=6)
    ref = O.fp8_prepass(q, k, v, mode="block", rotate=True, seed=6)
    for name in ("q8", "k8", "sq", "sk", "sv"):
        assert np.array_equal(pre[name].cpu().numpy(), ref[name]), name
    vt = pre["vt8"].cpu().numpy()
    assert np.array_equal(vt[..., :N], ref["vt8"])
    assert np.all(vt[..., N:] == 0)


def _emulated_check(B, N, H, Hkv, causal, mode, rotate, seed, rows=None, d=128):
    import exact_attention_45_gb300 as A
    q, k, v = gen.qkv_fixed(B, N, H, Hkv, d, seed=seed, dist="outlier")
    pre = _prepass_gpu(q, k, v, mode, rotate, seed=seed)
    o, lse = A.attn_fwd_fp8(pre, causal=causal)
    torch.cuda.synchronize()
    assert A.attn_get_device_error() == 0
    ref_pre = O.fp8_prepass(q, k, v, mode=mode, rotate=rotate, seed=seed)
    o_ref, l_ref, flip = O.fp8_attention_emulated(ref_pre, causal=causal, block_n=128, rows=rows, flip_tol=FLIP_TOL)
    o_h = o.float().cpu().numpy()
    l_h = lse.cpu().numpy()
    if rows is None:
        o_g = o_h.transpose(0, 2, 1, 3).reshape(-1, d)
        l_g = l_h.reshape(-1)
    else:
        o_g = o_h[rows[0], rows[2], rows[1]]
        l_g = l_h[rows[0], rows[1], rows[2]]
    err = o_g - o_ref
    assert np.isfinite(o_h).all()
    # bf16 output rounding (relative, up to 2^-9 |O|; outlier V makes |O| large)
    # plus the e4m3 rounding of any p that sits on a midpoint (see FLIP_TOL)
    bound = 1e-2 + 4e-3 * np.abs(o_ref) + flip
    worst = float((np.abs(err) / bound).max())
    rms = float(np.sqrt((err ** 2).mean()))
    assert worst <= 1.0 and rms <= 2e-3, (worst, rms)
    assert np.abs(l_g - l_ref).max() <= 2e-3


@pytest.mark.parametrize("mode", ["block", "tensor"])
@pytest.mark.parametrize("causal", [False, True])
def test_fp8_forward_matches_emulation(mode, causal):
    _emulated_check(2, 300, 4, 2, causal, mode, True, seed=1)


def test_fp8_forward_no_rotation_and_gqa():
    _emulated_check(1, 513, 8, 2, False, "block", False, seed=2)


# head dim 256: CTA pairs (two CTAs share each product; one 256-row unit per
# pair, the odd CTA's rows past the end of a ragged tail)
@pytest.mark.parametrize("mode", ["block", "tensor"])
@pytest.mark.parametrize("causal", [False, True])
def test_fp8_forward_d256_matches_emulation(mode, causal):
    _emulated_check(2, 300, 4, 2, causal, mode, True, seed=11, d=256)


def test_fp8_forward_d256_no_rotation_gqa_several_units():
    # 4 query heads per KV head, 1000 rows: 4 units per head, ragged last one
    _emulated_check(1, 1000, 8, 2, True, "block", False, seed=12, d=256)


def test_fp8_forward_d256_short():
    # fewer rows than one CTA's tile: the odd CTA of each pair has no valid row
    _emulated_check(3, 77, 2, 1, False, "block", True, seed=13, d=256)


# head dim 64: the head-dim-128 kernel, whose copies zero-fill channels 64-127
# of Q, K and V^T; only the 64 real output channels are stored
@pytest.mark.parametrize("mode", ["block", "tensor"])
@pytest.mark.parametrize("causal", [False, True])
def test_fp8_forward_d64_matches_emulation(mode, causal):
    _emulated_check(2, 300, 4, 2, causal, mode, True, seed=21, d=64)


def test_fp8_forward_d64_no_rotation_gqa_several_units():
    _emulated_check(1, 1000, 8, 2, True, "block", False, seed=22, d=64)


def test_fp8_d64_output_rows_are_exactly_64_channels():
    # the output tensor's neighbours are untouched (nothing is stored past
    # channel 63 of a row)
    import exact_attention_45_gb300 as A
    B, N, H, d = 1, 200, 2, 64
    q, k, v = (t.cuda() for t in gen.qkv_fixed(B, N, H, H, d, seed=23, dist="outlier"))
    pre = A.attn_fp8_prepass(q, k, v, mode="block", rotate=True, hadamard_seed=3)
    buf = torch.full((B * N * H * d + 4096,), 7.0, dtype=torch.bfloat16, device="cuda")
    out = buf[:B * N * H * d].view(B, N, H, d)
    o, _ = A.attn_fwd_fp8(pre, out=out)
    torch.cuda.synchronize()
    assert A.attn_get_device_error() == 0
    assert torch.isfinite(o.float()).all()
    assert torch.all(buf[B * N * H * d:] == 7.0)


def test_fp8_auto_equals_two_calls():
    import exact_attention_45_gb300 as A
    q, k, v = (t.cuda() for t in gen.qkv_fixed(2, 640, 4, 4, 128, seed=3, dist="outlier"))
    pre = A.attn_fp8_prepass(q, k, v, mode="block", rotate=True, hadamard_seed=9)
    o1, l1 = A.attn_fwd_fp8(pre, causal=True)
    o2, l2 = A.attn_fwd_fp8_auto(q, k, v, causal=True, mode="block", rotate=True, hadamard_seed=9)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)

"""GPU parity of the FP8 path at the full benchmark sizes, and the FP8 error
study of the pages' claim.

* The FP8 forward at B=4, N=4096, H=16, d=128 (block scales + rotation,
  outlier inputs), causal and not, at B=4, N=4096, H=8, d=256 (CTA pairs), and
  over the packed GQA configuration (8 sequences of 1k-32k tokens, H=32,
  Hkv=8, causal), against the oracle's FP8 emulation on >= 512 sampled rows
  with the bounds of the small FP8 tests.
  Block-mode scales belong to one (batch or sequence, head), so the oracle
  quantises only the (batch, KV head) slices the sampled rows need; their codes
  and scales are those of the whole tensor.
* The error study ("FlashAttention-3: Fast and Accurate Attention with
  Asynchrony and Low-precision", abstract and core claim: block quantization
  and incoherent processing give 2.6x lower numerical error than a baseline
  FP8 attention; "What would settle it": compare FP8 error against standard
  FP8 attention): RMS error against exact fp64 attention of the bf16 inputs
  for the four variants {per-block, per-tensor} x {rotation, none} at
  N = 1k..16k (B*N = 16384, H = 16, d = 128, outlier inputs). Asserts the
  gate (block + rotation <= 2.5e-2), that it beats the plain per-tensor path,
  and that the rotation alone helps (block + rotation below block without).
  Each row of the table is printed with the prefix FP8-ERROR-STUDY.
"""
import json

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

SEED = 0


def _within_emulation_bounds(o_g, l_g, o_ref, l_ref, flip, what):
    # the bounds of the small-shape FP8 tests: bf16 output rounding (relative)
    # plus the e4m3 rounding of any p that sits on a midpoint (see FLIP_TOL)
    err = o_g - o_ref
    bound = 1e-2 + 4e-3 * np.abs(o_ref) + flip
    worst = float((np.abs(err) / bound).max())
    rms = float(np.sqrt((err ** 2).mean()))
    lerr = float(np.abs(l_g - l_ref).max())
    assert worst <= 1.0 and rms <= 2e-3 and lerr <= 2e-3, f"{what}: worst {worst:.3f} rms {rms:.3e} lse {lerr:.3e}"


def _emulate_fixed_rows(q, k, v, rows, causal, seed):
    """Oracle FP8 emulation of the sampled rows (b, h, i), block scales with
    rotation, pre-pass run per (batch, KV head) slice."""
    rb, rh, ri = rows
    H, Hkv, d = q.shape[2], k.shape[2], q.shape[3]
    g = H // Hkv
    o = np.zeros((rb.size, d))
    lse = np.zeros(rb.size)
    flip = np.zeros((rb.size, d))
    for b in np.unique(rb):
        for hk in np.unique(rh[rb == b] // g):
            sel = np.nonzero((rb == b) & (rh // g == hk))[0]
            pre = O.fp8_prepass(q[b:b + 1, :, hk * g:(hk + 1) * g], k[b:b + 1, :, hk:hk + 1],
                                v[b:b + 1, :, hk:hk + 1], mode="block", rotate=True, seed=seed)
            o[sel], lse[sel], flip[sel] = O.fp8_attention_emulated(
                pre, causal=causal, rows=(np.zeros(sel.size, np.int64), rh[sel] - hk * g, ri[sel]),
                flip_tol=FLIP_TOL)
    return o, lse, flip


@pytest.mark.parametrize("causal", [False, True])
def test_fp8_forward_full_size_matches_emulation(causal):
    import exact_attention_45_gb300 as A
    B, N, H, d = 4, 4096, 16, 128
    q, k, v = gen.qkv_fixed(B, N, H, H, d, seed=SEED, dist="outlier")
    o, lse = A.attn_fwd_fp8_auto(q.cuda(), k.cuda(), v.cuda(), causal=causal, mode="block", rotate=True,
                                 hadamard_seed=SEED)
    torch.cuda.synchronize()
    assert A.attn_get_device_error() == 0
    o_h, l_h = o.float().cpu().numpy(), lse.cpu().numpy()
    assert np.isfinite(o_h).all() and np.isfinite(l_h).all()
    rb, rh, ri = gen.sample_rows([N] * B, H, 512, seed=1 + causal)
    assert rb.size >= 512
    o_ref, l_ref, flip = _emulate_fixed_rows(q, k, v, (rb, rh, ri), causal, SEED)
    _within_emulation_bounds(o_h[rb, ri, rh], l_h[rb, rh, ri], o_ref, l_ref, flip,
                             f"FP8 B{B} N{N} H{H} causal={causal}")


def test_fp8_forward_d256_full_size_matches_emulation():
    # head dim 256 (CTA pairs) at the FP8 sweep's N = 4096 point: B = 4, H = 8,
    # per-block scales + rotation, outlier inputs, non-causal
    import exact_attention_45_gb300 as A
    B, N, H, d = 4, 4096, 8, 256
    q, k, v = gen.qkv_fixed(B, N, H, H, d, seed=SEED, dist="outlier")
    o, lse = A.attn_fwd_fp8_auto(q.cuda(), k.cuda(), v.cuda(), causal=False, mode="block", rotate=True,
                                 hadamard_seed=SEED)
    torch.cuda.synchronize()
    assert A.attn_get_device_error() == 0
    o_h, l_h = o.float().cpu().numpy(), lse.cpu().numpy()
    assert np.isfinite(o_h).all() and np.isfinite(l_h).all()
    rb, rh, ri = gen.sample_rows([N] * B, H, 512, seed=5)
    assert rb.size >= 512
    o_ref, l_ref, flip = _emulate_fixed_rows(q, k, v, (rb, rh, ri), False, SEED)
    _within_emulation_bounds(o_h[rb, ri, rh], l_h[rb, rh, ri], o_ref, l_ref, flip, f"FP8 d256 B{B} N{N} H{H}")


def _varlen_pair_rows(lengths, g, pairs, per_pair, seed):
    """Rows (sequence, query head, local row) of the given (sequence, KV head)
    pairs: first, 127th, 128th and last rows plus uniform ones, over the pair's
    query heads."""
    rng = np.random.default_rng(seed)
    rs, rh, ri = [], [], []
    for s, hk in pairs:
        n = int(lengths[s])
        fixed = [r for r in (0, 127, 128, n - 1) if 0 <= r < n]
        rr = fixed + rng.integers(0, n, size=per_pair - len(fixed)).tolist()
        rs += [s] * len(rr)
        rh += (hk * g + rng.integers(0, g, size=len(rr))).tolist()
        ri += rr
    trip = np.unique(np.stack([rs, rh, ri], axis=1), axis=0)
    return trip[:, 0].astype(np.int64), trip[:, 1].astype(np.int64), trip[:, 2].astype(np.int64)


def test_fp8_varlen_gqa_full_size_matches_emulation():
    import exact_attention_45_gb300 as A
    lengths = gen.varlen_lengths(8, 1024, 32768, seed=SEED)
    H, Hkv, d = 32, 8, 128
    g = H // Hkv
    q, k, v, cu = gen.qkv_varlen(lengths, H, Hkv, d, seed=SEED, dist="outlier")
    dcu = torch.as_tensor(cu, dtype=torch.int32).cuda()
    pre = A.attn_fp8_prepass_varlen(q.cuda(), k.cuda(), v.cuda(), dcu, mode="block", rotate=True,
                                    hadamard_seed=SEED)
    o, lse = A.attn_fwd_fp8_varlen(pre, causal=True)
    torch.cuda.synchronize()
    assert A.attn_get_device_error() == 0
    o_h, l_h = o.float().cpu().numpy(), lse.cpu().numpy()
    assert np.isfinite(o_h).all() and np.isfinite(l_h).all()
    order = np.argsort(lengths)
    # the longest and the shortest sequence, the first and the last one
    pairs = [(int(order[-1]), 0), (int(order[0]), Hkv - 1), (0, 3), (len(lengths) - 1, 5)]
    rs, rh, ri = _varlen_pair_rows(lengths, g, pairs, 130, seed=3)
    assert rs.size >= 512
    o_ref = np.zeros((rs.size, d))
    l_ref = np.zeros(rs.size)
    flip = np.zeros((rs.size, d))
    for s, hk in set(pairs):
        a, b = int(cu[s]), int(cu[s + 1])
        sel = np.nonzero((rs == s) & (rh // g == hk))[0]
        # one sequence of the packed batch is its own block-quantised problem
        pre_s = O.fp8_prepass(q[None, a:b, hk * g:(hk + 1) * g], k[None, a:b, hk:hk + 1], v[None, a:b, hk:hk + 1],
                              mode="block", rotate=True, seed=SEED)
        o_ref[sel], l_ref[sel], flip[sel] = O.fp8_attention_emulated(
            pre_s, causal=True, rows=(np.zeros(sel.size, np.int64), rh[sel] - hk * g, ri[sel]), flip_tol=FLIP_TOL)
    tok = np.asarray(cu)[rs] + ri
    _within_emulation_bounds(o_h[tok, rh], l_h[rh, tok], o_ref, l_ref, flip, "FP8 GQA varlen causal")


VARIANTS = (("block", True), ("block", False), ("tensor", True), ("tensor", False))


@pytest.mark.parametrize("N", [1024, 2048, 4096, 8192, 16384])
def test_fp8_error_study(N):
    import exact_attention_45_gb300 as A
    B, H, d = 16384 // N, 16, 128
    q, k, v = gen.qkv_fixed(B, N, H, H, d, seed=SEED, dist="outlier")
    rs, rh, ri = gen.sample_rows([N] * B, H, 512, seed=SEED)
    o_ref, _ = O.attention(q, k, v, rows=(rs, rh, ri))
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    rms = {}
    for mode, rotate in VARIANTS:
        o, _ = A.attn_fwd_fp8_auto(qd, kd, vd, mode=mode, rotate=rotate, hadamard_seed=SEED)
        torch.cuda.synchronize()
        assert A.attn_get_device_error() == 0
        o_h = o.float().cpu().numpy()
        assert np.isfinite(o_h).all()
        rms[(mode, rotate)] = float(np.sqrt(((o_h[rs, ri, rh] - o_ref) ** 2).mean()))
    best, no_rot, plain = rms[("block", True)], rms[("block", False)], rms[("tensor", False)]
    print("FP8-ERROR-STUDY " + json.dumps({
        "N": N, "B": B, "H": H, "d": d, "rows": int(rs.size),
        "rms_block_rot": best, "rms_block_norot": no_rot, "rms_tensor_rot": rms[("tensor", True)],
        "rms_tensor_norot": plain, "ratio_plain_over_block_rot": plain / best,
        "ratio_block_norot_over_block_rot": no_rot / best}), flush=True)
    assert best <= 2.5e-2
    assert best < plain
    assert best < no_rot

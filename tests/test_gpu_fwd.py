"""GPU parity of the BF16/FP16 forward (through the C ABI) against the fp64
oracle, element by element on small shapes and on sampled rows at the full
benchmark sizes."""
import numpy as np
import pytest
import torch

import attn_inputs as gen
import oracle as O
from _attn_util import (assert_close, check_fixed_full, check_fixed_sampled, run_fixed, run_varlen)

pytestmark = pytest.mark.gpu


def test_tiny_config():
    # B=1, H=1, N=128, d=64, non-causal, seed 0, scale 1/sqrt(d)
    check_fixed_full(1, 128, 1, 1, 64, False)


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 77, 300, 513])
def test_shapes_with_ragged_tails(d, causal, N):
    check_fixed_full(2, N, 4, 2, d, causal, seed=N + d)


@pytest.mark.parametrize("d", [64, 128, 256])
def test_fp16(d):
    check_fixed_full(1, 257, 2, 1, d, True, dtype="fp16")
    check_fixed_full(1, 200, 2, 2, d, False, dtype="fp16")


def test_mqa_single_kv_head():
    check_fixed_full(2, 300, 8, 1, 128, True)


def test_single_key_is_v_exactly():
    for d in (64, 128, 256):
        q, k, v = gen.qkv_fixed(3, 1, 4, 2, d, seed=d)
        o, lse = run_fixed(q, k, v, False)
        ref = v.repeat_interleave(2, dim=2)
        assert torch.equal(o.cpu(), ref)
        o_ref, l_ref = O.attention(q, k, v)
        assert np.abs(lse.cpu().numpy() - l_ref).max() <= 1e-3


def test_first_causal_row_is_v0_exactly():
    for d in (64, 128, 256):
        q, k, v = gen.qkv_fixed(2, 190, 4, 4, d, seed=1)
        o, _ = run_fixed(q, k, v, True)
        assert torch.equal(o[:, 0].cpu(), v[:, 0])


def test_uniform_scores_give_mean_of_v():
    q = torch.zeros(1, 300, 2, 128, dtype=torch.bfloat16)
    _, k, v = gen.qkv_fixed(1, 300, 2, 1, 128, seed=4)
    o, lse = run_fixed(q, k, v, True)
    o_ref, l_ref = O.attention(q, k, v, causal=True)
    assert_close(o.float().cpu().numpy(), o_ref, lse.cpu().numpy(), l_ref)
    assert np.abs(lse.cpu().numpy()[0, 0] - np.log(np.arange(1, 301))).max() <= 1e-3


def test_deterministic():
    q, k, v = gen.qkv_fixed(2, 700, 4, 2, 128, seed=5)
    o1, l1 = run_fixed(q, k, v, True)
    o2, l2 = run_fixed(q, k, v, True)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_varlen_small():
    lengths = [1, 130, 257, 64, 0, 500]
    for d in (64, 128, 256):
        for causal in (False, True):
            q, k, v, cu = gen.qkv_varlen(lengths, 4, 2, d, seed=d + causal)
            o, lse = run_varlen(q, k, v, cu, causal)
            o_ref, l_ref = O.attention(q, k, v, causal=causal, cu_seqlens=cu)
            assert_close(o.float().cpu().numpy(), o_ref, lse.cpu().numpy(), l_ref,
                         what=f"varlen d{d} causal={causal}")


def test_varlen_matches_fixed_when_equal_lengths():
    q, k, v = gen.qkv_fixed(3, 200, 4, 2, 128, seed=8)
    o_f, l_f = run_fixed(q, k, v, True)
    cu = np.array([0, 200, 400, 600], dtype=np.int32)
    o_v, l_v = run_varlen(q.reshape(600, 4, 128), k.reshape(600, 2, 128), v.reshape(600, 2, 128), cu, True)
    assert torch.equal(o_v.reshape(3, 200, 4, 128), o_f)
    assert torch.equal(l_v.reshape(4, 3, 200).permute(1, 0, 2), l_f)


def test_timeout_probe_reports_and_recovers():
    import exact_attention_45_gb300 as A
    A.attn_debug_timeout_probe(2_000_000)          # 2 ms bound, nothing ever arrives
    assert A.attn_get_device_error() == A.ATTN_ERR_TIMEOUT
    assert A.attn_get_device_error() == 0          # cleared
    check_fixed_full(1, 128, 1, 1, 64, False)      # context still usable


def test_invalid_arguments_raise():
    import exact_attention_45_gb300 as A
    q, k, v = (t.cuda() for t in gen.qkv_fixed(1, 64, 2, 2, 96, seed=0))
    with pytest.raises(A.AttnError) as e:
        A.attn_fwd(q, k, v)
    assert e.value.status == A.ATTN_ERR_UNSUPPORTED
    q, k, v = (t.cuda() for t in gen.qkv_fixed(1, 64, 3, 2, 64, seed=0))
    with pytest.raises(A.AttnError):
        A.attn_fwd(q, k, v)


# ---- every output element at a size where each persistent CTA walks several
# work units (ring phases, TMEM reuse and the epilogue staging of later units):
# 4 x 2048 tokens, hidden 2048 -> 512 units of 256 rows (d = 64, 128) or 1024
# units of 128 rows (d = 256) over at most 152 CTAs
@pytest.mark.parametrize("d,H", [(128, 16), (64, 32), (256, 8)])
@pytest.mark.parametrize("causal", [False, True])
def test_multi_unit_per_cta_every_element(d, H, causal):
    check_fixed_full(4, 2048, H, H, d, causal, seed=17 + d)


# ---- full benchmark sizes: BF16 sweep (hidden 2048, B*N = 16384 tokens)
SWEEP = [(d, H, N, causal) for d, H in ((64, 32), (128, 16)) for N in (512, 1024, 2048, 4096, 8192, 16384)
         for causal in (False, True)]


@pytest.mark.parametrize("d,H,N,causal", SWEEP)
def test_bf16_sweep_sampled(d, H, N, causal):
    check_fixed_sampled(16384 // N, N, H, H, d, causal, count=192)


@pytest.mark.parametrize("N", [1024, 2048, 4096, 8192, 16384])
@pytest.mark.parametrize("causal", [False, True])
def test_d256_sampled(N, causal):
    check_fixed_sampled(16384 // N, N, 8, 8, 256, causal, count=128)


def test_gqa_varlen_causal_full_size():
    lengths = gen.varlen_lengths(8, 1024, 32768, seed=0)
    q, k, v, cu = gen.qkv_varlen(lengths, 32, 8, 128, seed=0)
    o, lse = run_varlen(q, k, v, cu, True)
    o_h, l_h = o.float().cpu().numpy(), lse.cpu().numpy()
    assert np.isfinite(o_h).all() and np.isfinite(l_h).all()
    rs, rh, ri = gen.sample_rows(lengths, 32, 160, seed=0)
    o_ref, l_ref = O.attention(q, k, v, causal=True, cu_seqlens=cu, rows=(rs, rh, ri))
    tok = cu[rs] + ri
    assert_close(o_h[tok, rh], o_ref, l_h[rh, tok], l_ref, what="GQA varlen causal")

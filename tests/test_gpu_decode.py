"""GPU parity of split-KV decode and the partial-result combine (through the
C ABI) against the fp64 oracle."""
import math

import numpy as np
import pytest
import torch

import attn_inputs as gen
import oracle as O
from _attn_util import assert_close

pytestmark = pytest.mark.gpu


def _inputs(B, H, Hkv, nmax, d, seed, dtype="bf16"):
    q, _, _ = gen.qkv_fixed(B, 1, H, Hkv, d, seed=seed, dtype=dtype)
    _, k, v = gen.qkv_fixed(B, nmax, Hkv, Hkv, d, seed=seed + 1, dtype=dtype)
    return q[:, 0].contiguous(), k, v


def _run(q, k, v, seqlens, splits):
    import exact_attention_45_gb300 as A
    sl = torch.as_tensor(np.asarray(seqlens), dtype=torch.int32).cuda()
    o, lse = A.attn_decode(q.cuda(), k.cuda(), v.cuda(), sl, num_splits=splits)
    torch.cuda.synchronize()
    assert A.attn_get_device_error() == 0
    return o.float().cpu().numpy(), lse.cpu().numpy()


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("splits", [1, 3, 0, 40])
def test_decode_matches_oracle(d, splits):
    B, H, Hkv, nmax = 5, 8, 2, 1000
    seqlens = [1, 127, 128, 129, 1000]
    q, k, v = _inputs(B, H, Hkv, nmax, d, seed=d + splits)
    o, lse = _run(q, k, v, seqlens, splits)
    o_ref, l_ref = O.attention_decode(q, k, v, seqlens)
    assert_close(o, o_ref, lse, l_ref, what=f"decode d{d} splits={splits}")


@pytest.mark.parametrize("d", [64, 128])
def test_decode_fp16_and_mha(d):
    q, k, v = _inputs(3, 4, 4, 300, d, seed=7, dtype="fp16")
    seqlens = [300, 2, 257]
    o, lse = _run(q, k, v, seqlens, 2)
    o_ref, l_ref = O.attention_decode(q, k, v, seqlens)
    assert_close(o, o_ref, lse, l_ref, what="decode fp16 MHA")


def test_decode_single_key_and_empty_cache():
    q, k, v = _inputs(2, 4, 1, 256, 128, seed=3)
    o, lse = _run(q, k, v, [1, 0], 3)
    assert np.array_equal(o[0], np.repeat(v[0, 0].float().numpy(), 4, axis=0))
    assert np.all(o[1] == 0) and np.all(lse[1] == -np.inf)
    o_ref, l_ref = O.attention_decode(q, k, v, [1, 0])
    assert np.abs(lse[0] - l_ref[0]).max() <= 1e-3


def test_decode_gqa_long_cache_full_size():
    # 8 sequences with cached lengths uniform in [1k, 32k], H=32, Hkv=8, d=128
    seqlens = gen.varlen_lengths(8, 1024, 32768, seed=0)
    nmax = 32768
    q, k, v = _inputs(8, 32, 8, nmax, 128, seed=11)
    o, lse = _run(q, k, v, seqlens, 0)
    o_ref, l_ref = O.attention_decode(q, k, v, seqlens)
    assert_close(o, o_ref, lse, l_ref, what="decode GQA 32k")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("H,Hkv", [(2, 2), (8, 4), (16, 2), (24, 2), (32, 2), (48, 2), (64, 2), (40, 2)])
def test_decode_query_groups(H, Hkv, d):
    # groups of 1, 2, 8, 12, 16 (keys-as-rows kernel, N = 16), 24 and 32 (N =
    # 32) query heads per KV head, and 20 (units with the query heads as
    # rows), over several splits
    B, nmax = 3, 700
    seqlens = [700, 1, 385]
    q, k, v = _inputs(B, H, Hkv, nmax, d, seed=H * 10 + Hkv + d)
    o, lse = _run(q, k, v, seqlens, 3)
    o_ref, l_ref = O.attention_decode(q, k, v, seqlens)
    assert_close(o, o_ref, lse, l_ref, what=f"decode group {H // Hkv}")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("H,Hkv", [(4, 4), (8, 2), (48, 4), (48, 2), (64, 2)])
def test_decode_ignores_cache_rows_past_length(H, Hkv, d):
    # groups 1, 4 and 12 (keys-as-rows kernel with 16 columns), 24 and 32 (32
    # columns): rows at or past a sequence's length are cleared, so NaN there
    # must not reach O
    B, nmax = 2, 512
    seqlens = [200, 333]
    q, k, v = _inputs(B, H, Hkv, nmax, d, seed=31 + H + d)
    kn, vn = k.clone(), v.clone()
    for b, n in enumerate(seqlens):
        kn[b, n:] = float("nan")
        vn[b, n:] = float("nan")
    o, lse = _run(q, kn, vn, seqlens, 2)
    o_ref, l_ref = O.attention_decode(q, k, v, seqlens)
    assert np.isfinite(o).all() and np.isfinite(lse).all()
    assert_close(o, o_ref, lse, l_ref, what="decode with NaN past the length")


@pytest.mark.parametrize("d,splits,H", [(128, 1, 8), (128, 0, 8), (64, 0, 8), (128, 0, 32), (64, 0, 24)])
def test_decode_many_short_sequences(d, splits, H):
    # 300 sequences (some empty) on one KV head each: more units than SMs, so
    # a CTA's range crosses several units and leaves several partials; groups
    # of 8 (16-column kernel), 24 and 32 (32-column kernel)
    rng = np.random.default_rng(4)
    B, Hkv, nmax = 300, 1, 300
    seqlens = rng.integers(0, nmax + 1, size=B)
    seqlens[::37] = 0
    q, k, v = _inputs(B, H, Hkv, nmax, d, seed=41 + d + H)
    o, lse = _run(q, k, v, seqlens, splits)
    o_ref, l_ref = O.attention_decode(q, k, v, seqlens)
    empty = seqlens == 0
    assert np.all(o[empty] == 0) and np.all(lse[empty] == -np.inf)
    assert_close(o[~empty], o_ref[~empty], lse[~empty], l_ref[~empty], what="decode, 300 short sequences")


def test_decode_dirty_workspace_reused():
    # the per-pair merge counters carry a per-call epoch: a workspace full of
    # arbitrary bytes needs no initialisation, and reusing it gives the same
    # result bit for bit
    import exact_attention_45_gb300 as A
    B, H, Hkv, nmax, splits = 3, 8, 2, 2000, 2
    seqlens = [2000, 700, 1500]
    q, k, v = _inputs(B, H, Hkv, nmax, 128, seed=53)
    ws = torch.full((A.attn_decode_workspace_size(B, H, 128, splits),), 0xFF, dtype=torch.uint8, device="cuda")
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    sl = torch.as_tensor(seqlens, dtype=torch.int32).cuda()
    outs = [A.attn_decode(qd, kd, vd, sl, num_splits=splits, workspace=ws) for _ in range(2)]
    torch.cuda.synchronize()
    assert A.attn_get_device_error() == 0
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])
    o_ref, l_ref = O.attention_decode(q, k, v, seqlens)
    assert_close(outs[0][0].float().cpu().numpy(), o_ref, outs[0][1].cpu().numpy(), l_ref, what="decode, dirty workspace")


def test_combine_matches_oracle():
    import exact_attention_45_gb300 as A
    rng = np.random.default_rng(5)
    S, rows, d = 6, 37, 128
    o_parts = rng.standard_normal((S, rows, d)).astype(np.float32)
    lse_parts = (rng.standard_normal((S, rows)) * 4).astype(np.float32)
    lse_parts[2, :] = -np.inf
    lse_parts[:, 5] = -np.inf              # a row with no keys at all
    o_parts[2, :] = np.nan                 # never read: its lse is -inf
    o, lse = A.attn_combine(torch.from_numpy(o_parts).cuda(), torch.from_numpy(lse_parts).cuda())
    torch.cuda.synchronize()
    op = o_parts.astype(np.float64)
    op[2] = 0.0
    o_ref, l_ref = O.combine_partials(op, lse_parts)
    o_h, l_h = o.float().cpu().numpy(), lse.cpu().numpy()
    assert np.all(o_h[5] == 0) and l_h[5] == -np.inf
    ok = np.isfinite(l_ref)
    assert np.abs(o_h - o_ref).max() <= 1e-2
    assert np.abs(l_h[ok] - l_ref[ok]).max() <= 1e-4


def test_decode_invalid_arguments():
    import exact_attention_45_gb300 as A
    q, k, v = _inputs(1, 2, 1, 128, 256, seed=0)
    sl = torch.tensor([128], dtype=torch.int32).cuda()
    with pytest.raises(A.AttnError) as e:
        A.attn_decode(q.cuda(), k.cuda(), v.cuda(), sl)
    assert e.value.status == A.ATTN_ERR_UNSUPPORTED

"""CPU checks of the C ABI: the library builds, loads and exports every
function include/attn45.h declares; host-side argument checks answer without
touching a GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _header_functions():
    src = open(os.path.join(ROOT, "include", "attn45.h")).read()
    return sorted(set(re.findall(r"ATTN45_API\s+[\w\s\*]+?\b(attn_\w+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    import exact_attention_45_gb300 as A
    return A.capi()


def test_every_declared_symbol_is_exported(lib):
    import exact_attention_45_gb300 as A
    declared = _header_functions()
    assert len(declared) >= 13
    assert sorted(A.EXPORTED_SYMBOLS) == declared
    for name in declared:
        assert hasattr(lib, name), name


def test_status_strings(lib):
    assert lib.attn_status_string(0) == b"ok"
    assert lib.attn_status_string(4) == b"device wait timed out"
    assert lib.attn_version() >= 1


def test_host_checks_need_no_gpu(lib):
    # rejected before any CUDA call is made
    rc = lib.attn_fwd(None, None, None, None, None, 1, 2, 2, 128, 96, 0, 0.1, 0, None)
    assert rc == 2 and b"head dim" in lib.attn_last_error_message()
    rc = lib.attn_fwd(None, None, None, None, None, 1, 3, 2, 128, 64, 0, 0.1, 0, None)
    assert rc == 1
    rc = lib.attn_fwd(None, None, None, None, None, 1, 2, 2, 128, 64, 0, -1.0, 0, None)
    assert rc == 1 and b"scale" in lib.attn_last_error_message()
    rc = lib.attn_fwd(None, None, None, None, None, 1, 2, 2, 128, 64, 2, 0.1, 0, None)
    assert rc == 1
    rc = lib.attn_fwd(None, None, None, None, None, 0, 2, 2, 128, 64, 0, 0.1, 0, None)
    assert rc == 1
    rc = lib.attn_fwd(None, None, None, None, None, 1, 2, 2, 128, 64, 0, 0.1, 0, None)
    assert rc == 1 and b"null" in lib.attn_last_error_message()
    rc = lib.attn_fwd_varlen(None, None, None, None, None, None, 0, 0, 10, 2, 2, 64, 0, 0.1, 0, None)
    assert rc == 1
    assert lib.attn_set_wait_timeout_ns(10) == 1
    assert lib.attn_set_wait_timeout_ns(2_000_000_000) == 0


def _pad256(x):
    return (x + 255) // 256 * 256


def test_workspace_sizes_and_block_bounds(lib):
    # decode: fp32 partial O and lse for (splits + 1) rows per output row, then
    # one 8-byte merge counter per (sequence, head)
    B, H, d, S = 3, 8, 128, 4
    rows = (S + 1) * B * H
    assert lib.attn_decode_workspace_size(B, H, d, S) == _pad256(rows * d * 4) + _pad256(rows * 4) + _pad256(B * H * 8)
    assert lib.attn_decode_workspace_size(0, H, d, S) == 0 and lib.attn_decode_workspace_size(B, H, d, 0) == 0
    # backward: fp32 dQ accumulator and the row sums D
    B, H, N = 2, 4, 300
    r = B * N * H
    assert lib.attn_bwd_workspace_size(B, H, N, 64) == _pad256(r * 64 * 4) + _pad256(r * 4)
    assert lib.attn_bwd_workspace_size(B, H, 0, 64) == 0
    # packed FP8: 128-row blocks over all sequences never exceed ceil(T/128) + nseq
    assert lib.attn_fp8_varlen_tmax(0, 3) == 3
    assert lib.attn_fp8_varlen_tmax(1000, 3) == 8 + 3
    assert lib.attn_fp8_varlen_tmax(10, 0) == 0


def test_host_checks_of_decode_backward_and_packed_fp8(lib):
    # rejected before any CUDA call is made
    args = [None] * 7 + [0]
    rc = lib.attn_decode(*args, 1, 2, 1, 128, 256, 2, 0.1, 0, None)
    assert rc == 2 and b"head dim" in lib.attn_last_error_message()
    assert lib.attn_decode(*args, 1, 3, 2, 128, 128, 2, 0.1, 0, None) == 1      # H % Hkv != 0
    assert lib.attn_decode(*args, 1, 256, 1, 128, 128, 2, 0.1, 0, None) == 2    # more than 128 heads per KV head
    assert lib.attn_decode(*args, 0, 2, 1, 128, 128, 2, 0.1, 0, None) == 1      # B = 0
    rc = lib.attn_decode(*args, 1, 2, 1, 128, 128, 2, 0.1, 0, None)
    assert rc == 1 and b"null" in lib.attn_last_error_message()
    assert lib.attn_combine(None, None, None, None, 0, 4, 64, 0, None) == 1     # no splits
    assert lib.attn_combine(None, None, None, None, 2, 0, 64, 0, None) == 0     # no rows: nothing to do
    bargs = [None] * 10 + [0]
    assert lib.attn_bwd(*bargs, 1, 2, 2, 128, 256, 0, 0.1, 0, None) == 2          # head dim 256
    assert lib.attn_bwd(*bargs, 1, 2, 2, 128, 64, 2, 0.1, 0, None) == 1           # causal must be 0 or 1
    rc = lib.attn_bwd(*bargs, 1, 2, 2, 128, 64, 0, 0.1, 0, None)
    assert rc == 1 and b"null" in lib.attn_last_error_message()
    vargs = [None] * 11
    assert lib.attn_fp8_prepass_varlen(*vargs, 0, 10, 2, 2, 128, 1, 1, 0, None) == 1   # no sequences
    assert lib.attn_fp8_prepass_varlen(*vargs, 2, 10, 2, 2, 96, 1, 1, 0, None) == 2    # head dim 96
    assert lib.attn_fp8_prepass_varlen(*vargs, 2, 10, 2, 2, 128, 7, 1, 0, None) == 1   # unknown mode


def test_fp8_combined_calls_reject_forward_arguments_before_the_prepass(lib):
    # the combined calls check what the forward step would reject before the
    # pre-pass runs, so a rejected call writes nothing; the pointers are never
    # dereferenced, so None is enough here. Head dims 64, 128 and 256 get as
    # far as the pointer check.
    for d in (64, 128, 256):
        rc = lib.attn_fwd_fp8_auto(None, None, None, None, None, None, 0, 1, 2, 2, 256, d, 0, 0.1, 1, 1, 0, None)
        assert rc == 1 and b"null" in lib.attn_last_error_message()
    rc = lib.attn_fwd_fp8_auto(None, None, None, None, None, None, 0, 1, 2, 2, 256, 96, 0, 0.1, 1, 1, 0, None)
    assert rc == 2                                                  # head dim 96
    rc = lib.attn_fwd_fp8_auto_noalloc(None, None, None, None, None, 1, 2, 2, 256, 128, 2, 0.1, 1, 1, 0, None)
    assert rc == 1 and b"causal" in lib.attn_last_error_message()
    rc = lib.attn_fwd_fp8_auto_noalloc(None, None, None, None, None, 1, 2, 2, 256, 64, 0, 0.1, 1, 1, 0, None)
    assert rc == 1 and b"null" in lib.attn_last_error_message()


def test_vt_ld(lib):
    assert lib.attn_fp8_vt_ld(1) == 128 and lib.attn_fp8_vt_ld(128) == 128 and lib.attn_fp8_vt_ld(129) == 256


def test_oracle_and_product_share_no_code():
    # neither side imports the other
    for path in ("exact_attention_45_gb300/__init__.py", "exact_attention_45_gb300/build.py"):
        assert "oracle" not in open(os.path.join(ROOT, path)).read()
    src = open(os.path.join(ROOT, "oracle", "__init__.py")).read()
    assert "exact_attention_45_gb300" not in src.split('"""', 2)[2]
    assert "exact_attention_45_gb300" not in open(os.path.join(ROOT, "oracle", "attn_oracle.c")).read()

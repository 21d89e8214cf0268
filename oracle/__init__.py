"""CPU oracle for the fused exact attention forward pass -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The product path (the CUDA library and
its Python binding) never imports it, and this package never imports the
product path: the two share no code. Both are fed from ``attn_inputs``, which
only draws seeded random numbers.

Contents
--------
* ``attention`` -- fp64 exact attention (the plain definition) via the C core
  in ``attn_oracle.c``; any subset of rows, fixed-length or packed varlen.
* ``attention_bruteforce`` -- an independent numpy float64 statement that
  materialises the whole score matrix; for tiny shapes only.
* ``attention_backward`` -- fp64 gradients dQ, dK, dV of sum(dO * O).
* ``attention_decode`` / ``combine_partials`` / ``decode_split_ranges`` --
  one query token per (sequence, head) over a key/value cache, and the merge
  of results computed over disjoint key ranges (split-KV decode).
* FP8 pieces, each following the FP8 technique of "FlashAttention-3: Fast and
  Accurate Attention with Asynchrony and Low-precision" (abstract, technique
  (3): block quantization and incoherent processing):
  ``splitmix64``, ``hadamard_signs``, ``sylvester``, ``fwht_f32``,
  ``rotate_f32``, ``e4m3_decode``, ``e4m3_encode``, ``fp8_prepass`` and
  ``fp8_attention_emulated``.

Readings where the pages are silent are stated beside each function.
Parity status: every function here is pinned by ``tests/test_oracle.py``
except ``fp8_attention_emulated``, whose P-quantisation step is a reading of
the pages that no printed value fixes; it is pinned only through its special
cases (single key block, uniform scores) -- see that function's docstring.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
import threading

import numpy as np

__all__ = [
    "build", "attention", "attention_bruteforce", "attention_flops",
    "attention_decode", "combine_partials", "decode_split_ranges", "attention_backward",
    "splitmix64", "hadamard_signs", "sylvester", "fwht_f32", "rotate_f32",
    "E4M3_MAX", "e4m3_decode", "e4m3_encode", "e4m3_table",
    "fp8_quant_block_rows", "fp8_prepass", "fp8_attention_emulated",
    "fp8_varlen_block_offsets", "fp8_prepass_varlen", "fp8_attention_emulated_varlen",
    "P_FP8_MULT", "P_FP8_LAZY_LOG2", "Q_BLOCK", "K_BLOCK",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_LIB = os.path.join(_HERE, "_build", "liboracle_attn.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the C core with gcc (plain C, -O2, no fast-math)."""
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                        "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp, "-lm"],
                       check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            p = ctypes.c_void_p
            lib.oracle_attn_rows.argtypes = [p, p, p, ctypes.c_int64, ctypes.c_int64,
                                             ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                             p, p, ctypes.c_int64, p, p, p,
                                             ctypes.c_int, ctypes.c_double, p, p, ctypes.c_int]
            lib.oracle_attn_rows.restype = ctypes.c_int
            _lib = lib
    return _lib


def _f32(x) -> np.ndarray:
    """Exact widening of a bf16/fp16/fp32 tensor (torch or numpy) to fp32."""
    if hasattr(x, "detach"):
        x = x.detach().cpu().float().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float32))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def attention(q, k, v, causal: bool = False, scale: float | None = None,
              cu_seqlens=None, rows=None, nthreads: int | None = None):
    """fp64 exact attention on the values stored in q, k, v.

    Fixed length: q [B,N,H,d], k/v [B,N,Hkv,d]; full output o [B,N,H,d] and
    lse [B,H,N]. Packed varlen (``cu_seqlens`` given): q [T,H,d], k/v
    [T,Hkv,d]; full output o [T,H,d] and lse [H,T].
    ``rows=(seq, head, i)`` (i local to the sequence; seq = batch index for
    fixed length) computes only those rows: o [R,d], lse [R].
    ``scale`` defaults to 1/sqrt(d). lse is the natural log of the softmax
    normaliser of the scaled scores.
    """
    qf, kf, vf = _f32(q), _f32(k), _f32(v)
    if cu_seqlens is None:
        B, N, H, d = qf.shape
        Hkv = kf.shape[2]
        starts = np.arange(B, dtype=np.int64) * N
        lens = np.full(B, N, dtype=np.int64)
    else:
        cu = np.asarray(cu_seqlens, dtype=np.int64)
        _, H, d = qf.shape
        Hkv = kf.shape[1]
        starts = cu[:-1].copy()
        lens = (cu[1:] - cu[:-1]).astype(np.int64)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    full = rows is None
    if full:
        seq_l, head_l, row_l = [], [], []
        for s, n in enumerate(lens):
            hh, ii = np.meshgrid(np.arange(H, dtype=np.int64), np.arange(n, dtype=np.int64), indexing="ij")
            seq_l.append(np.full(hh.size, s, dtype=np.int64))
            head_l.append(hh.ravel())
            row_l.append(ii.ravel())
        rs = np.concatenate(seq_l) if seq_l else np.zeros(0, np.int64)
        rh = np.concatenate(head_l) if head_l else np.zeros(0, np.int64)
        ri = np.concatenate(row_l) if row_l else np.zeros(0, np.int64)
    else:
        rs, rh, ri = (np.ascontiguousarray(np.asarray(a, dtype=np.int64)) for a in rows)
    R = rs.size
    o = np.zeros((R, d), dtype=np.float64)
    lse = np.zeros(R, dtype=np.float64)
    if nthreads is None:
        nthreads = os.cpu_count() or 1
    lib = _load()
    rc = lib.oracle_attn_rows(_ptr(qf), _ptr(kf), _ptr(vf), H * d, Hkv * d, H, Hkv, d,
                              _ptr(starts), _ptr(lens), R, _ptr(rs), _ptr(rh), _ptr(ri),
                              int(bool(causal)), float(scale), _ptr(o), _ptr(lse), int(nthreads))
    if rc != 0:
        raise RuntimeError("oracle_attn_rows failed")
    if not full:
        return o, lse
    if cu_seqlens is None:
        # rows were enumerated as (b, h, i) with i fastest
        o_full = o.reshape(B, H, N, d).transpose(0, 2, 1, 3).copy()
        return o_full, lse.reshape(B, H, N)
    T = int(lens.sum())
    o_full = np.zeros((T, H, d))
    lse_full = np.zeros((H, T))
    pos = 0
    for s, n in enumerate(lens):
        blk = o[pos:pos + H * n].reshape(H, n, d)
        o_full[starts[s]:starts[s] + n] = blk.transpose(1, 0, 2)
        lse_full[:, starts[s]:starts[s] + n] = lse[pos:pos + H * n].reshape(H, n)
        pos += H * n
    return o_full, lse_full


def attention_bruteforce(q, k, v, causal: bool = False, scale: float | None = None):
    """Materialised softmax(scale * Q K^T [+ causal mask]) V in numpy float64.

    Fixed-length BSHD only; meant for tiny shapes (it builds N x N matrices).
    Independent of the C core: matrix products and exp come from numpy.
    """
    qf = _f32(q).astype(np.float64)
    kf = _f32(k).astype(np.float64)
    vf = _f32(v).astype(np.float64)
    B, N, H, d = qf.shape
    Hkv = kf.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    g = H // Hkv
    o = np.zeros_like(qf)
    lse = np.zeros((B, H, N))
    keep = np.tril(np.ones((N, N), dtype=bool)) if causal else np.ones((N, N), dtype=bool)
    for b in range(B):
        for h in range(H):
            S = scale * (qf[b, :, h, :] @ kf[b, :, h // g, :].T)
            S = np.where(keep, S, -np.inf)
            mx = S.max(axis=1, keepdims=True)
            W = np.exp(S - mx)
            Z = W.sum(axis=1, keepdims=True)
            o[b, :, h, :] = (W / Z) @ vf[b, :, h // g, :]
            lse[b, h, :] = (mx + np.log(Z))[:, 0]
    return o, lse


def attention_backward(q, k, v, do, causal: bool = False, scale: float | None = None):
    """fp64 gradients of the loss sum(dO * O) with O = softmax(scale Q K^T [+ causal mask]) V.

    The backward pass of the FlashAttention papers (FA1, "trains Transformers
    faster", consumes the forward's logsumexp); written here as the plain
    chain rule, one (b, h) at a time:
        P  = softmax(S),  S = scale Q K^T (masked keys: P = 0)
        dV = P^T dO                     dP = dO V^T
        D_i = sum_c dO_ic O_ic          dS = P * (dP - D)   (row-wise D)
        dQ = scale dS K                 dK = scale dS^T Q
    With grouped-query attention, dK and dV of a KV head sum over the query
    heads that share it. Inputs BSHD (q, do [B,N,H,d]; k, v [B,N,Hkv,d]);
    returns dq, dk, dv in fp64 with the same shapes.
    """
    qf = _f32(q).astype(np.float64)
    kf = _f32(k).astype(np.float64)
    vf = _f32(v).astype(np.float64)
    gf = _f32(do).astype(np.float64)
    B, N, H, d = qf.shape
    Hkv = kf.shape[2]
    g = H // Hkv
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dq = np.zeros_like(qf)
    dk = np.zeros_like(kf)
    dv = np.zeros_like(vf)
    mask = np.tril(np.ones((N, N), dtype=bool)) if causal else np.ones((N, N), dtype=bool)
    for b in range(B):
        for h in range(H):
            hk = h // g
            Q, K, V, G = qf[b, :, h], kf[b, :, hk], vf[b, :, hk], gf[b, :, h]
            S = np.where(mask, scale * (Q @ K.T), -np.inf)
            P = np.exp(S - S.max(axis=1, keepdims=True))
            P /= P.sum(axis=1, keepdims=True)
            O = P @ V
            dv[b, :, hk] += P.T @ G
            dP = G @ V.T
            D = (G * O).sum(axis=1, keepdims=True)
            dS = P * (dP - D)
            dq[b, :, h] = scale * (dS @ K)
            dk[b, :, hk] += scale * (dS.T @ Q)
    return dq, dk, dv


def attention_decode(q, k_cache, v_cache, seqlens, scale: float | None = None):
    """fp64 attention of one query token per (sequence b, query head h) over
    the first ``seqlens[b]`` keys of its KV head's cache (decode phase: the
    FlashAttention-3 page's references [49] "Lean attention ... decode-phase
    of transformers" and [51] "Fast Transformer Decoding: One Write-Head is
    All You Need"). The plain definition, one row at a time:
        s_j = scale * q[b,h] . k[b,j,hk];  m = max_j s_j;  w_j = exp(s_j - m)
        o[b,h] = sum_j w_j v[b,j,hk] / sum_j w_j;  lse[b,h] = m + ln sum_j w_j
    with hk = h // (H / Hkv). q [B,H,d]; caches [B,Nmax,Hkv,d]; an empty
    cache (seqlens[b] == 0) gives o = 0 and lse = -inf (an empty sum).
    Returns o [B,H,d] and lse [B,H] (natural log, scale included), fp64.
    """
    qf = _f32(q).astype(np.float64)
    kf = _f32(k_cache).astype(np.float64)
    vf = _f32(v_cache).astype(np.float64)
    B, H, d = qf.shape
    Hkv = kf.shape[2]
    g = H // Hkv
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    o = np.zeros((B, H, d))
    lse = np.full((B, H), -np.inf)
    for b in range(B):
        n = int(seqlens[b])
        if n == 0:
            continue
        for h in range(H):
            hk = h // g
            s = scale * (kf[b, :n, hk, :] @ qf[b, h])
            m = s.max()
            w = np.exp(s - m)
            o[b, h] = (w @ vf[b, :n, hk, :]) / w.sum()
            lse[b, h] = m + math.log(w.sum())
    return o, lse


def combine_partials(o_parts, lse_parts):
    """Merge attention results over disjoint key subsets into the result over
    their union. The online softmax's rescaling step ("Related papers:
    FlashAttention-4" page, online-softmax teaser: a running maximum and
    normaliser let partial results be rescaled and summed), applied once
    across subsets: with L = ln sum_s exp(lse_s),
        lse = L,   o = sum_s exp(lse_s - L) o_s.
    Computed as L = m + ln sum_s exp(lse_s - m), m = max_s lse_s. Subsets with
    lse_s = -inf (no keys) weigh 0; if every subset is empty, o = 0 and
    lse = -inf. o_parts [S, ..., d], lse_parts [S, ...]; fp64 results.
    """
    op = np.asarray(o_parts, np.float64)
    lp = np.asarray(lse_parts, np.float64)
    m = lp.max(axis=0)
    mm = np.where(np.isfinite(m), m, 0.0)
    w = np.exp(lp - mm)                       # exp(-inf) = 0 for empty subsets
    tot = w.sum(axis=0)
    with np.errstate(divide="ignore", invalid="ignore"):
        lse = np.where(tot > 0, mm + np.log(np.where(tot > 0, tot, 1.0)), -np.inf)
        o = np.where(tot[..., None] > 0, (w[..., None] * op).sum(axis=0) / np.where(tot > 0, tot, 1.0)[..., None], 0.0)
    return o, lse


def decode_split_ranges(seqlen: int, nmax: int, num_splits: int, block: int = 128):
    """Key ranges [s0, s1) of the ``num_splits`` splits of one sequence: the
    cache length ``nmax`` is cut into equal chunks of ceil(nmax / num_splits)
    keys rounded up to ``block``; split s covers [s*chunk, (s+1)*chunk)
    clipped to [0, seqlen) and is empty past the sequence end (our reading:
    the pages fix no split rule)."""
    chunk = -(-nmax // num_splits)
    chunk = -(-chunk // block) * block
    return [(min(s * chunk, seqlen), min((s + 1) * chunk, seqlen)) for s in range(num_splits)]


def attention_flops(B: int, H: int, N: int, d: int, causal: bool) -> float:
    """The headline work count: 4*B*H*N^2*d, halved for causal."""
    f = 4.0 * B * H * N * N * d
    return f / 2 if causal else f


# --------------------------------------------------------------------------
# FP8 pieces. "FlashAttention-3: Fast and Accurate Attention with Asynchrony
# and Low-precision", abstract / core claim: FP8 with block quantization and
# incoherent processing (multiplying Q and K by a random orthogonal matrix so
# outliers spread out; the product Q K^T is unchanged). The pages fix neither
# the orthogonal matrix nor the block shape; the readings below are ours.
# --------------------------------------------------------------------------

_M64 = (1 << 64) - 1
Q_BLOCK = 128      # rows of Q per quantisation block (one scale per block)
K_BLOCK = 128      # rows of K per quantisation block
P_FP8_LAZY_LOG2 = 8.0  # FP8 P: the running maximum is raised only when a block
                       # maximum exceeds it by more than this (log2 units)
P_FP8_MULT = 1.0       # = 2^(8 - P_FP8_LAZY_LOG2): P <= 2^8 maps to codes <= 256


def splitmix64(x: int) -> int:
    """First output of Vigna's SplitMix64 generator whose state is ``x``.

    Published definition: state += 0x9E3779B97F4A7C15; z = state;
    z = (z ^ z>>30) * 0xBF58476D1CE4E5B9; z = (z ^ z>>27) * 0x94D049BB133111EB;
    return z ^ z>>31 (all mod 2^64).
    """
    z = (x + 0x9E3779B97F4A7C15) & _M64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _M64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _M64
    return z ^ (z >> 31)


def hadamard_signs(seed: int, d: int) -> np.ndarray:
    """Diagonal of the random sign matrix D: sigma_c = 1 - 2*(splitmix64(seed+c) & 1)."""
    return np.array([1.0 - 2.0 * (splitmix64((seed + c) & _M64) & 1) for c in range(d)],
                    dtype=np.float32)


def sylvester(d: int) -> np.ndarray:
    """Sylvester Hadamard matrix: H_1 = [1], H_2k = [[H_k, H_k], [H_k, -H_k]]."""
    Hm = np.ones((1, 1), dtype=np.int64)
    while Hm.shape[0] < d:
        Hm = np.block([[Hm, Hm], [Hm, -Hm]])
    if Hm.shape[0] != d:
        raise ValueError("d must be a power of two")
    return Hm


def fwht_f32(x: np.ndarray) -> np.ndarray:
    """x @ H_d along the last axis by the fast Walsh-Hadamard butterflies, in fp32.

    Stages run with span h = 1, 2, 4, ..., d/2; each replaces the pair
    (a = x[i], b = x[i+h]) (bit h of i clear) by (a + b, a - b). Every add and
    subtract is one fp32 rounding, so the stage order is part of the definition.
    """
    y = np.array(x, dtype=np.float32, copy=True)
    d = y.shape[-1]
    lead = y.shape[:-1]
    h = 1
    while h < d:
        y = y.reshape(*lead, d // (2 * h), 2, h)
        a = y[..., 0, :]
        b = y[..., 1, :]
        y = np.stack([a + b, a - b], axis=-2).reshape(*lead, d)
        h *= 2
    return y


def rotate_f32(x: np.ndarray, signs: np.ndarray) -> np.ndarray:
    """Incoherent processing of rows: x -> (x * sigma) @ H_d * fl32(1/sqrt(d)), in fp32."""
    d = x.shape[-1]
    c = np.float32(1.0 / math.sqrt(d))
    return (fwht_f32(np.asarray(x, np.float32) * signs) * c).astype(np.float32)


# e4m3 ("FP8 Formats for Deep Learning", cited by the FlashAttention-3 page as
# its FP8 reference): 1 sign, 4 exponent (bias 7), 3 mantissa bits; no
# infinities; S.1111.111 is NaN; largest finite magnitude 448.
E4M3_MAX = 448.0


def e4m3_decode(code) -> np.ndarray:
    code = np.asarray(code, dtype=np.int64)
    s = np.where((code >> 7) & 1, -1.0, 1.0)
    e = (code >> 3) & 0xF
    m = code & 0x7
    mag = np.where(e == 0, (m / 8.0) * 2.0 ** (1 - 7), (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7))
    val = s * mag
    return np.where((e == 15) & (m == 7), np.nan, val)


def e4m3_table() -> np.ndarray:
    """Decoded value of every byte 0..255."""
    return e4m3_decode(np.arange(256))


_POS_CODES = np.arange(0, 0x7F)          # 0x00 .. 0x7E: all non-negative finite values
_POS_VALS = e4m3_decode(_POS_CODES)      # strictly increasing, 0 .. 448


def e4m3_encode(x) -> np.ndarray:
    """Round to nearest e4m3, ties to even code, saturating to +-448 (satfinite).

    NaN maps to 0x7F (with the sign bit of the input); +-inf saturate to +-448.
    The decision is made exactly (fp64 comparisons of an fp32 input).
    """
    x = np.asarray(x, dtype=np.float64)
    sign = np.signbit(x)
    a = np.abs(x)
    a_c = np.minimum(a, E4M3_MAX)
    hi = np.clip(np.searchsorted(_POS_VALS, a_c, side="left"), 0, len(_POS_VALS) - 1)
    lo = np.clip(hi - 1, 0, None)
    dlo = np.abs(a_c - _POS_VALS[lo])
    dhi = np.abs(_POS_VALS[hi] - a_c)
    pick_hi = (dhi < dlo) | ((dhi == dlo) & ((_POS_CODES[hi] & 1) == 0))
    code = np.where(pick_hi, _POS_CODES[hi], _POS_CODES[lo]).astype(np.int64)
    code = np.where(np.isnan(x), 0x7F, code)
    code = code | (sign.astype(np.int64) << 7)
    return code.astype(np.uint8)


def _scale_from_amax(amax: np.ndarray) -> np.ndarray:
    """scale = fl32(amax / 448), or 1 where amax == 0 (the block is all zeros)."""
    amax = np.asarray(amax, dtype=np.float32)
    s = (amax / np.float32(E4M3_MAX)).astype(np.float32)
    return np.where(amax == 0, np.float32(1.0), s).astype(np.float32)


def _quant(y_f32: np.ndarray, s_f32) -> np.ndarray:
    """code = e4m3(fl32(y / s)) with the division one fp32 rounding."""
    return e4m3_encode((np.asarray(y_f32, np.float32) / np.asarray(s_f32, np.float32)).astype(np.float32))


def fp8_quant_block_rows(x_f32: np.ndarray, block: int):
    """Quantise x [B, N, Hx, d] with one scale per (b, head, block of rows).

    Returns codes (uint8, same shape) and scales [B, Hx, ceil(N/block)].
    """
    B, N, Hx, d = x_f32.shape
    nb = (N + block - 1) // block
    codes = np.zeros(x_f32.shape, dtype=np.uint8)
    scales = np.zeros((B, Hx, nb), dtype=np.float32)
    for ib in range(nb):
        sl = slice(ib * block, min(N, (ib + 1) * block))
        amax = np.abs(x_f32[:, sl]).max(axis=(1, 3))       # [B, Hx]
        s = _scale_from_amax(amax)
        scales[:, :, ib] = s
        codes[:, sl] = _quant(x_f32[:, sl], s[:, None, :, None])
    return codes, scales


def fp8_prepass(q, k, v, mode: str = "block", rotate: bool = True, seed: int = 0):
    """Quantise bf16/fp16 Q, K, V (BSHD) to e4m3 codes plus fp32 scales.

    Reading of the pages' "block quantization" + "incoherent processing":
      * rotate (optional): Q' = rotate_f32(Q), K' = rotate_f32(K) with the same
        signs for every (b, head); V is never rotated.
      * mode "block":  Q', K' one scale per (b, head, 128-row block);
                       V one scale per (b, kv head, channel) over all rows.
      * mode "tensor": one scale per tensor for each of Q', K', V (the plain
                       FP8 baseline when ``rotate`` is False).
      * scale = fl32(amax/448) (1 if amax == 0); code = e4m3(fl32(x/scale)).
    Returns dict: q8 [B,N,H,d], k8 [B,N,Hkv,d], vt8 [B,Hkv,d,N] (V codes
    transposed so keys are contiguous), sq, sk, sv (fp32 arrays).
    """
    qf, kf, vf = _f32(q), _f32(k), _f32(v)
    B, N, H, d = qf.shape
    Hkv = kf.shape[2]
    if rotate:
        signs = hadamard_signs(seed, d)
        qf = rotate_f32(qf, signs)
        kf = rotate_f32(kf, signs)
    if mode == "block":
        q8, sq = fp8_quant_block_rows(qf, Q_BLOCK)
        k8, sk = fp8_quant_block_rows(kf, K_BLOCK)
        sv = _scale_from_amax(np.abs(vf).max(axis=1))      # [B, Hkv, d]
        v8 = _quant(vf, sv[:, None, :, :])
    elif mode == "tensor":
        sq = _scale_from_amax(np.abs(qf).max()).reshape(1)
        sk = _scale_from_amax(np.abs(kf).max()).reshape(1)
        sv = _scale_from_amax(np.abs(vf).max()).reshape(1)
        q8, k8, v8 = _quant(qf, sq[0]), _quant(kf, sk[0]), _quant(vf, sv[0])
    else:
        raise ValueError(mode)
    vt8 = np.ascontiguousarray(v8.transpose(0, 2, 3, 1))
    return {"q8": q8, "k8": k8, "vt8": vt8, "sq": sq, "sk": sk, "sv": sv,
            "mode": mode, "rotate": rotate, "seed": seed}


def fp8_attention_emulated(pre: dict, causal: bool = False, scale: float | None = None,
                           block_n: int = 128, rows=None, quantize_p: bool = True, flip_tol: float | None = None):
    """FP8 attention on pre-pass codes, following the method's own steps.

    Online softmax ("Related papers: FlashAttention-4" page, teaser on online
    softmax: stream score tiles, keep a running maximum and normaliser), over
    key blocks of ``block_n`` in order, in fp64:
      t_j   = (Q8 K8^T)_ij * scale * log2(e) * sq(row block) * sk(key block)
      b     = max_j t_j;  m' = b if b > m + tau else m     (tau = P_FP8_LAZY_LOG2)
      p_j   = 2^(t_j - m')                               (so p_j <= 2^tau)
      l     = l * 2^(m - m') + sum_j p_j                 (l from unquantised p)
      acc   = acc * 2^(m - m') + sum_j e4m3(M p_j) * V8_j  (M = P_FP8_MULT = 2^(8-tau))
      O     = acc * sv / (M l),  lse = (m + log2 l) * ln 2
    The lazy maximum is the same online softmax with a stale reference point:
    O and lse do not depend on m in exact arithmetic, only the e4m3 grid P
    lands on does. The P quantisation (lazy margin 2^8, the same as the 16-bit
    path's, multiplier 1, l from unquantised p) is our reading; parity unpinned beyond the special cases
    tested (a single key block equals a direct evaluation; blocks after one
    that holds the row maximum reproduce the single-block result; uniform
    scores give the mean of dequantised V).
    ``rows`` = (b, h, i) arrays; default all rows. Returns o [R,d], lse [R].
    ``quantize_p=False`` keeps p unquantised (then the result is the exact
    softmax attention of the dequantised inputs, for any ``block_n``).

    ``flip_tol`` (a relative distance) adds a third output ``flip`` [R, d]:
    for every p whose M p lies within ``flip_tol`` of a midpoint between two
    neighbouring e4m3 values, the change in O that rounding it the other way
    would make, |one e4m3 step| * 2^(m_block - m_final) * |V8_j| * sv / (M l),
    summed over such p. Both roundings of such a p are the method's result:
    which one a computation takes depends on the last bits of its score
    arithmetic (fp32 against fp64 here). o and lse are unchanged.
    """
    q8 = e4m3_decode(pre["q8"])
    k8 = e4m3_decode(pre["k8"])
    vt8 = e4m3_decode(pre["vt8"])
    sq, sk, sv = (np.asarray(pre[n], np.float64) for n in ("sq", "sk", "sv"))
    block = pre["mode"] == "block"
    B, N, H, d = q8.shape
    Hkv = k8.shape[2]
    g = H // Hkv
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    log2e = 1.0 / math.log(2.0)
    if rows is None:
        bb, hh, ii = np.meshgrid(np.arange(B), np.arange(H), np.arange(N), indexing="ij")
        rows = (bb.ravel(), hh.ravel(), ii.ravel())
    rb, rh, ri = (np.asarray(a, dtype=np.int64) for a in rows)
    R = rb.size
    o = np.zeros((R, d))
    lse = np.zeros(R)
    flip = np.zeros((R, d)) if flip_tol is not None else None
    for r in range(R):
        b, h, i = int(rb[r]), int(rh[r]), int(ri[r])
        hk = h // g
        nk = i + 1 if causal else N
        qs = sq[b, h, i // Q_BLOCK] if block else sq[0]
        svec = sv[b, hk, :] if block else np.full(d, sv[0])
        m, l = -np.inf, 0.0
        acc = np.zeros(d)
        facc = np.zeros(d)
        for j0 in range(0, nk, block_n):
            j1 = min(nk, j0 + block_n)
            keys = np.arange(j0, j1)
            ks = np.array([sk[b, hk, j // K_BLOCK] if block else sk[0] for j in keys])
            raw = k8[b, j0:j1, hk, :] @ q8[b, i, h, :]
            t = raw * scale * log2e * qs * ks
            bmax = t.max()
            m_new = bmax if bmax > m + P_FP8_LAZY_LOG2 else m
            alpha = 2.0 ** (m - m_new) if m != -np.inf else 0.0
            p = 2.0 ** (t - m_new)
            l = l * alpha + p.sum()
            if quantize_p:
                p8 = e4m3_decode(e4m3_encode((p * P_FP8_MULT).astype(np.float32)))
            else:
                p8 = p * P_FP8_MULT
            acc = acc * alpha + p8 @ vt8[b, hk, :, j0:j1].T
            if flip_tol is not None:
                pm = p * P_FP8_MULT
                # e4m3 spacing at pm: 2^(e-3) in the normal range [2^e, 2^(e+1)),
                # 2^-9 below 2^-6 (subnormals, and the step from 0 to 2^-9)
                step = np.where(pm >= 2.0 ** -6, 2.0 ** (np.floor(np.log2(np.maximum(pm, 2.0 ** -6))) - 3), 2.0 ** -9)
                frac = pm / step - np.floor(pm / step)
                dist = np.abs(frac - 0.5) * step / np.maximum(pm, 1e-300)
                facc = facc * alpha + np.where(dist <= flip_tol, step, 0.0) @ np.abs(vt8[b, hk, :, j0:j1]).T
            m = m_new
        o[r] = acc * svec / (P_FP8_MULT * l)
        lse[r] = (m + math.log2(l)) * math.log(2.0)
        if flip_tol is not None:
            flip[r] = facc * np.abs(svec) / (P_FP8_MULT * l)
    if flip_tol is not None:
        return o, lse, flip
    return o, lse


# ------------------------------------------------------------------ FP8, packed variable-length sequences
def fp8_varlen_block_offsets(cu_seqlens) -> np.ndarray:
    """blk_off[s] = sum over earlier sequences of ceil(n/128): the first
    128-row quantisation block (and 128-key V column block) of sequence s."""
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    n = cu[1:] - cu[:-1]
    return np.concatenate([[0], np.cumsum((n + Q_BLOCK - 1) // Q_BLOCK)]).astype(np.int32)


def fp8_prepass_varlen(q, k, v, cu_seqlens, mode: str = "block", rotate: bool = True, seed: int = 0):
    """The FP8 pre-pass of packed sequences (THD: q [T,H,d], k, v [T,Hkv,d]).

    Reading: every sequence is quantised as its own batch element of
    ``fp8_prepass`` (blocks of 128 rows never cross a sequence boundary, V's
    channel scales are per (sequence, KV head)); in "tensor" mode the three
    scales cover the whole packed tensors. Layout (tmax = ceil(T/128) + nseq
    bounds the number of blocks): q8 [T,H,d], k8 [T,Hkv,d]; vt8 [Hkv, d,
    128*tmax] with sequence s's keys from column 128*blk_off[s] (pad keys of
    its last block hold code 0); block mode sq [H, tmax], sk [Hkv, tmax] with
    sequence s's block b at column blk_off[s] + b (other columns 0 here, not
    written by the GPU), sv [nseq, Hkv, d]; tensor mode one value each.
    """
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    nseq = cu.size - 1
    qf, kf, vf = _f32(q), _f32(k), _f32(v)
    T, H, d = qf.shape
    Hkv = kf.shape[1]
    boff = fp8_varlen_block_offsets(cu)
    tmax = -(-T // Q_BLOCK) + nseq
    q8 = np.zeros((T, H, d), np.uint8)
    k8 = np.zeros((T, Hkv, d), np.uint8)
    vt8 = np.zeros((Hkv, d, Q_BLOCK * tmax), np.uint8)
    if mode == "tensor":
        whole = fp8_prepass(qf[None], kf[None], vf[None], mode="tensor", rotate=rotate, seed=seed)
        q8[:] = whole["q8"][0]
        k8[:] = whole["k8"][0]
        for s in range(nseq):
            a, b = int(cu[s]), int(cu[s + 1])
            vt8[:, :, Q_BLOCK * boff[s]:Q_BLOCK * boff[s] + (b - a)] = whole["vt8"][0, :, :, a:b]
        sq, sk, sv = whole["sq"], whole["sk"], whole["sv"]
    elif mode == "block":
        sq = np.zeros((H, tmax), np.float32)
        sk = np.zeros((Hkv, tmax), np.float32)
        sv = np.zeros((nseq, Hkv, d), np.float32)
        for s in range(nseq):
            a, b = int(cu[s]), int(cu[s + 1])
            if b == a:
                # no rows: the channel amax over an empty set is 0, whose scale is 1
                sv[s] = _scale_from_amax(np.zeros((Hkv, d), np.float32))
                continue
            ps = fp8_prepass(qf[None, a:b], kf[None, a:b], vf[None, a:b], mode="block", rotate=rotate, seed=seed)
            q8[a:b], k8[a:b] = ps["q8"][0], ps["k8"][0]
            vt8[:, :, Q_BLOCK * boff[s]:Q_BLOCK * boff[s] + (b - a)] = ps["vt8"][0]
            nb = ps["sq"].shape[2]
            sq[:, boff[s]:boff[s] + nb] = ps["sq"][0]
            sk[:, boff[s]:boff[s] + nb] = ps["sk"][0]
            sv[s] = ps["sv"][0]
    else:
        raise ValueError(mode)
    return {"q8": q8, "k8": k8, "vt8": vt8, "sq": sq, "sk": sk, "sv": sv, "blk_off": boff, "tmax": tmax,
            "mode": mode, "rotate": rotate, "seed": seed}


def fp8_attention_emulated_varlen(pre: dict, cu_seqlens, causal: bool = False, scale: float | None = None,
                                  rows=None, flip_tol: float | None = None):
    """``fp8_attention_emulated`` of every sequence of a packed pre-pass result
    (each sequence is its own problem; causal masking is per sequence).
    ``rows`` = (sequence, head, local row) arrays; default every row. Returns
    o [R, d] and lse [R] in that row order (and ``flip`` [R, d] when
    ``flip_tol`` is given)."""
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    nseq = cu.size - 1
    boff = pre["blk_off"]
    H, d = pre["q8"].shape[1], pre["q8"].shape[2]
    if rows is None:
        rs, rh, ri = [], [], []
        for s in range(nseq):
            n = int(cu[s + 1] - cu[s])
            for h in range(H):
                rs += [s] * n
                rh += [h] * n
                ri += list(range(n))
        rows = (np.array(rs, np.int64), np.array(rh, np.int64), np.array(ri, np.int64))
    rs, rh, ri = (np.asarray(x, np.int64) for x in rows)
    o = np.zeros((rs.size, d))
    lse = np.zeros(rs.size)
    flip = np.zeros((rs.size, d))
    for s in np.unique(rs):
        a, b = int(cu[s]), int(cu[s + 1])
        n = b - a
        nb = -(-n // Q_BLOCK)
        sel = np.nonzero(rs == s)[0]
        blk = pre["mode"] == "block"
        ps = {"q8": pre["q8"][None, a:b], "k8": pre["k8"][None, a:b],
              "vt8": pre["vt8"][None, :, :, Q_BLOCK * boff[s]:Q_BLOCK * boff[s] + n],
              "sq": pre["sq"][None, :, boff[s]:boff[s] + nb] if blk else pre["sq"],
              "sk": pre["sk"][None, :, boff[s]:boff[s] + nb] if blk else pre["sk"],
              "sv": pre["sv"][s:s + 1] if blk else pre["sv"], "mode": pre["mode"]}
        res = fp8_attention_emulated(ps, causal=causal, scale=scale,
                                     rows=(np.zeros(sel.size, np.int64), rh[sel], ri[sel]), flip_tol=flip_tol)
        o[sel], lse[sel] = res[0], res[1]
        if flip_tol is not None:
            flip[sel] = res[2]
    if flip_tol is not None:
        return o, lse, flip
    return o, lse

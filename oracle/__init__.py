"""Float64 CPU oracle for speculative-decoding verification (ctypes wrapper).

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
benchmark's ``cpu_baseline`` / reference leg may import this package.  It
shares no code with the CUDA library; the C source states what each function
computes and which passage of the pages it follows:

* ``verify_attn`` / ``attn_rows`` -- multi-query causal attention of the k
  draft queries over the paged cache ("Decoding Speculative Decoding from
  First Principles", "Parallelizing method 2: sequence parallel"), with the
  INT8 dequantiser that inverts CXL-SpecKV's "Algorithm 2 KV-Cache
  Compression".
* ``accept_greedy`` -- first-disagreement acceptance plus bonus token (same
  blog, "Speculating to get sequence parallelism during decode").
* ``verify_attn_tree`` / ``accept_tree`` -- the same over a tree of drafts
  (same blog, "Advances in speculators": token trees verified in one pass).
* ``kv_append`` / ``quantize_rows`` / ``commit`` -- the drafts' K/V rows
  written into the paged cache (INT8: CXL-SpecKV's "Algorithm 2 KV-Cache
  Compression", per (token, kv-head) row) and HeteroReason's KVMU Accept
  pointer move.
* ``accept_rejection`` -- lossless rejection-sampling acceptance (same blog,
  "How does this drafter maintain the same distribution of the target?"),
  with its draws from the counter-based generator SplitMix64.
* ``codec_encode`` / ``codec_decode`` -- the delta + run-length coding of a
  page's INT8 codes (CXL-SpecKV, observation (5) and "Algorithm 2 KV-Cache
  Compression"), in the byte format the C source defines.

Arrays are numpy; 16-bit float types travel as their raw ``uint16`` bits.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

# The oracle's own element-type codes (mirrors the enum in spec_oracle.c only).
DTYPES = {"f32": 0, "bf16": 1, "f16": 2, "i8": 3}

_lib = None


def _load():
    global _lib
    if _lib is None:
        path = _build.build()
        lib = ctypes.CDLL(path)
        P = ctypes.c_void_p
        i32 = ctypes.c_int
        attn_common = [P, i32, P, P, i32, P, P, P, P, i32, i32, i32, i32, i32, i32, i32, i32,
                       ctypes.c_double]
        lib.oracle_verify_attn.argtypes = attn_common + [P, P]
        lib.oracle_verify_attn.restype = i32
        lib.oracle_attn_rows.argtypes = attn_common + [P, i32, P, P]
        lib.oracle_attn_rows.restype = i32
        lib.oracle_accept_greedy.argtypes = [P, i32, P, i32, i32, ctypes.c_int64, P, P, P]
        lib.oracle_accept_greedy.restype = i32
        u64 = ctypes.c_uint64
        lib.oracle_accept_rejection.argtypes = [P, P, i32, P, i32, i32, ctypes.c_int64,
                                                ctypes.c_double, u64, P, P, P, P, P]
        lib.oracle_accept_rejection.restype = i32
        lib.oracle_splitmix64.argtypes = [u64, u64]
        lib.oracle_splitmix64.restype = u64
        lib.oracle_accept_uniform.argtypes = [u64, i32, i32]
        lib.oracle_accept_uniform.restype = ctypes.c_double
        lib.oracle_gumbel.argtypes = [u64, i32, ctypes.c_int64]
        lib.oracle_gumbel.restype = ctypes.c_double
        lib.oracle_quantize_rows.argtypes = [P, i32, ctypes.c_int64, i32, P, P]
        lib.oracle_quantize_rows.restype = i32
        lib.oracle_kv_append.argtypes = [P, P, i32, P, P, P, P, i32, P, P, i32, i32, i32, i32,
                                         i32, i32, i32]
        lib.oracle_kv_append.restype = i32
        lib.oracle_commit.argtypes = [P, P, i32, i32]
        lib.oracle_commit.restype = i32
        lib.oracle_verify_attn_tree.argtypes = attn_common + [P, P, P]
        lib.oracle_verify_attn_tree.restype = i32
        lib.oracle_accept_tree.argtypes = [P, i32, P, P, i32, i32, ctypes.c_int64, P, P, P]
        lib.oracle_accept_tree.restype = i32
        lib.oracle_codec_encode.argtypes = [P, ctypes.c_int64, i32, i32, P, P]
        lib.oracle_codec_encode.restype = i32
        lib.oracle_codec_decode.argtypes = [P, P, ctypes.c_int64, i32, i32, P]
        lib.oracle_codec_decode.restype = i32
        lib.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
        lib.oracle_bf16_to_f64.restype = ctypes.c_double
        lib.oracle_f16_to_f64.argtypes = [ctypes.c_uint16]
        lib.oracle_f16_to_f64.restype = ctypes.c_double
        _lib = lib
    return _lib


def _ptr(a):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def _attn_common(q, q_dtype, k_cache, v_cache, kv_dtype, k_scale, v_scale, block_table,
                 ctx_lens, scale):
    B, k, Hq, D = q.shape
    NP, Hkv, P, D2 = k_cache.shape
    assert D2 == D and v_cache.shape == k_cache.shape
    assert block_table.dtype == np.int32 and ctx_lens.dtype == np.int32
    if kv_dtype == "i8":
        assert k_scale is not None and v_scale is not None
        assert k_scale.dtype == np.uint16 and k_scale.shape == (NP, Hkv, P)
    keep = (q, k_cache, v_cache, k_scale, v_scale, block_table, ctx_lens)
    args = [_ptr(q), DTYPES[q_dtype], _ptr(k_cache), _ptr(v_cache), DTYPES[kv_dtype],
            _ptr(k_scale), _ptr(v_scale), _ptr(block_table), _ptr(ctx_lens),
            B, k, Hq, Hkv, D, P, NP, block_table.shape[1], float(scale)]
    return keep, args, (B, k, Hq, D)


def verify_attn(q, q_dtype, k_cache, v_cache, kv_dtype, k_scale, v_scale, block_table,
                ctx_lens, scale):
    """Return (out[B,k,Hq,D], lse[B,k,Hq]) in float64."""
    keep, args, (B, k, Hq, D) = _attn_common(q, q_dtype, k_cache, v_cache, kv_dtype, k_scale,
                                             v_scale, block_table, ctx_lens, scale)
    out = np.zeros((B, k, Hq, D), np.float64)
    lse = np.zeros((B, k, Hq), np.float64)
    rc = _load().oracle_verify_attn(*args, _ptr(out), _ptr(lse))
    if rc:
        raise ValueError("oracle_verify_attn failed (%d): bad shape or page reference" % rc)
    del keep
    return out, lse


def attn_rows(q, q_dtype, k_cache, v_cache, kv_dtype, k_scale, v_scale, block_table, ctx_lens,
              scale, rows):
    """rows: int array [n, 3] of (b, i, h).  Return (out[n,D], lse[n]) in float64."""
    keep, args, (B, k, Hq, D) = _attn_common(q, q_dtype, k_cache, v_cache, kv_dtype, k_scale,
                                             v_scale, block_table, ctx_lens, scale)
    rows = np.ascontiguousarray(np.asarray(rows, np.int32).reshape(-1, 3))
    out = np.zeros((rows.shape[0], D), np.float64)
    lse = np.zeros((rows.shape[0],), np.float64)
    rc = _load().oracle_attn_rows(*args, _ptr(rows), rows.shape[0], _ptr(out), _ptr(lse))
    if rc:
        raise ValueError("oracle_attn_rows failed (%d)" % rc)
    del keep
    return out, lse


def verify_attn_tree(q, q_dtype, k_cache, v_cache, kv_dtype, k_scale, v_scale, block_table,
                     ctx_lens, scale, tree_mask):
    """Attention where draft query i sees the context and the drafts set in
    tree_mask[b, i] (uint64 [B, k]); returns (out, lse) float64."""
    keep, args, (B, k, Hq, D) = _attn_common(q, q_dtype, k_cache, v_cache, kv_dtype, k_scale,
                                             v_scale, block_table, ctx_lens, scale)
    tree_mask = np.ascontiguousarray(tree_mask, np.uint64)
    assert tree_mask.shape == (B, k)
    out = np.zeros((B, k, Hq, D), np.float64)
    lse = np.zeros((B, k, Hq), np.float64)
    rc = _load().oracle_verify_attn_tree(*args, _ptr(tree_mask), _ptr(out), _ptr(lse))
    if rc:
        raise ValueError("oracle_verify_attn_tree failed (%d)" % rc)
    return out, lse


def accept_tree(logits, dtype, draft_tokens, parents):
    """Greedy acceptance over a tree of drafts; returns (accepted_len, next_token, path [B, k])."""
    B, k1, V = logits.shape
    k = k1 - 1
    draft_tokens = np.ascontiguousarray(draft_tokens, np.int32)
    parents = np.ascontiguousarray(parents, np.int32)
    assert draft_tokens.shape == (B, k) and parents.shape == (B, k)
    acc = np.zeros(B, np.int32)
    nxt = np.zeros(B, np.int32)
    path = np.zeros((B, k), np.int32)
    rc = _load().oracle_accept_tree(_ptr(logits), DTYPES[dtype], _ptr(draft_tokens), _ptr(parents),
                                    B, k, V, _ptr(acc), _ptr(nxt), _ptr(path))
    if rc:
        raise ValueError("oracle_accept_tree failed (%d)" % rc)
    return acc, nxt, path


def accept_greedy(logits, dtype, draft_tokens):
    """logits [B, k+1, V]; draft_tokens int32 [B, k].

    Return (accepted_len[B], next_token[B], argmax_rows[B, k+1]) as int32.
    """
    B, k1, V = logits.shape
    k = k1 - 1
    draft_tokens = np.ascontiguousarray(draft_tokens, np.int32)
    assert draft_tokens.shape == (B, k)
    acc = np.zeros(B, np.int32)
    nxt = np.zeros(B, np.int32)
    am = np.zeros((B, k1), np.int32)
    rc = _load().oracle_accept_greedy(_ptr(logits), DTYPES[dtype], _ptr(draft_tokens), B, k, V,
                                      _ptr(acc), _ptr(nxt), _ptr(am))
    if rc:
        raise ValueError("oracle_accept_greedy failed (%d)" % rc)
    return acc, nxt, am


def accept_rejection(target_logits, draft_logits, dtype, draft_tokens, temperature, seed):
    """target_logits [B, k+1, V]; draft_logits [B, k, V]; draft_tokens int32 [B, k].

    Return (accepted_len[B] int32, next_token[B] int32, ratio[B, k],
    unif[B, k], key_gap[B]): p(x)/q(x) and the acceptance uniform at every
    position up to the first rejection (NaN after it), and the gap between
    the two best Gumbel keys of the final draw.
    """
    B, k1, V = target_logits.shape
    k = k1 - 1
    assert draft_logits.shape == (B, k, V)
    draft_tokens = np.ascontiguousarray(draft_tokens, np.int32)
    assert draft_tokens.shape == (B, k)
    acc = np.zeros(B, np.int32)
    nxt = np.zeros(B, np.int32)
    ratio = np.zeros((B, k), np.float64)
    unif = np.zeros((B, k), np.float64)
    gap = np.zeros(B, np.float64)
    rc = _load().oracle_accept_rejection(_ptr(target_logits), _ptr(draft_logits), DTYPES[dtype],
                                         _ptr(draft_tokens), B, k, V, float(temperature),
                                         int(seed) & (2**64 - 1), _ptr(acc), _ptr(nxt),
                                         _ptr(ratio), _ptr(unif), _ptr(gap))
    if rc:
        raise ValueError("oracle_accept_rejection failed (%d)" % rc)
    return acc, nxt, ratio, unif, gap


def quantize_rows(x, dtype):
    """Rows x [..., D] (f32 array or bf16 bits) -> (codes int8 [..., D], scale fp16 bits [...])."""
    x = np.ascontiguousarray(x)
    D = x.shape[-1]
    n = x.size // D
    codes = np.zeros(x.shape, np.int8)
    scales = np.zeros(x.shape[:-1], np.uint16)
    rc = _load().oracle_quantize_rows(_ptr(x), DTYPES[dtype], n, D, _ptr(codes), _ptr(scales))
    if rc:
        raise ValueError("oracle_quantize_rows failed (%d)" % rc)
    return codes, scales


def kv_append(k_new, v_new, src_dtype, k_cache, v_cache, k_scale, v_scale, cache_dtype,
              block_table, ctx_lens):
    """Return copies of (k_cache, v_cache, k_scale, v_scale) with the rows
    k_new / v_new [B, n, Hkv, D] written at positions ctx_b .. ctx_b + n - 1."""
    B, n, Hkv, D = k_new.shape
    NP, Hkv2, P, D2 = k_cache.shape
    assert (Hkv2, D2) == (Hkv, D) and v_new.shape == k_new.shape
    kc, vc = k_cache.copy(), v_cache.copy()
    ks = None if k_scale is None else k_scale.copy()
    vs = None if v_scale is None else v_scale.copy()
    rc = _load().oracle_kv_append(_ptr(np.ascontiguousarray(k_new)), _ptr(np.ascontiguousarray(v_new)),
                                  DTYPES[src_dtype], _ptr(kc), _ptr(vc), _ptr(ks), _ptr(vs),
                                  DTYPES[cache_dtype], _ptr(block_table), _ptr(ctx_lens), B, n,
                                  Hkv, D, P, NP, block_table.shape[1])
    if rc:
        raise ValueError("oracle_kv_append failed (%d)" % rc)
    return kc, vc, ks, vs


def commit(ctx_lens, accepted_len, extra=1):
    out = np.ascontiguousarray(ctx_lens, np.int32).copy()
    acc = np.ascontiguousarray(accepted_len, np.int32)
    _load().oracle_commit(_ptr(out), _ptr(acc), len(out), int(extra))
    return out


def splitmix64(seed: int, n: int) -> int:
    """The n-th (0-based) output of SplitMix64 seeded with `seed`."""
    return int(_load().oracle_splitmix64(int(seed) & (2**64 - 1), int(n)))


def accept_uniform(seed: int, b: int, i: int) -> float:
    return float(_load().oracle_accept_uniform(int(seed) & (2**64 - 1), int(b), int(i)))


def gumbel(seed: int, b: int, x: int) -> float:
    return float(_load().oracle_gumbel(int(seed) & (2**64 - 1), int(b), int(x)))


def bf16_bits_to_f64(bits: int) -> float:
    return _load().oracle_bf16_to_f64(int(bits))


def f16_bits_to_f64(bits: int) -> float:
    return _load().oracle_f16_to_f64(int(bits))


__all__ = ["verify_attn", "attn_rows", "verify_attn_tree", "accept_tree", "accept_greedy",
           "accept_rejection", "quantize_rows",
           "kv_append", "commit", "splitmix64",
           "accept_uniform", "gumbel", "bf16_bits_to_f64", "f16_bits_to_f64", "DTYPES"]


def codec_encode(codes):
    """codes int8 [nblk, P, D] -> (pairs uint8 [nblk, 2*P*D], npairs int32 [nblk])."""
    codes = np.ascontiguousarray(codes, dtype=np.int8)
    nblk, P, D = codes.shape
    pairs = np.zeros((nblk, 2 * P * D), np.uint8)
    npairs = np.zeros(nblk, np.int32)
    if _load().oracle_codec_encode(_ptr(codes), nblk, P, D, _ptr(pairs), _ptr(npairs)) != 0:
        raise MemoryError("oracle_codec_encode")
    return pairs, npairs


def codec_decode(pairs, npairs, P, D):
    """Inverse of codec_encode; ValueError on a malformed block."""
    pairs = np.ascontiguousarray(pairs, dtype=np.uint8)
    npairs = np.ascontiguousarray(npairs, dtype=np.int32)
    nblk = npairs.shape[0]
    codes = np.zeros((nblk, P, D), np.int8)
    if _load().oracle_codec_decode(_ptr(pairs), _ptr(npairs), nblk, P, D, _ptr(codes)) != 0:
        raise ValueError("malformed codec block")
    return codes

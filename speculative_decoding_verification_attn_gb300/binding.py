"""Thin ctypes binding of ``libspecverify.so`` (see ``include/spec_verify.h``).

Argument marshalling only: torch tensors supply device pointers, shapes,
dtypes and the current CUDA stream; every step of the computation runs in
the library's kernels.  There is no fallback: if the library has not been
built (``python -c "import __graft_entry__ as g; g.build()"``) or fails to
load, every call raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import numpy as np
import torch

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libspecverify.so")

SPEC_DTYPE_F32, SPEC_DTYPE_BF16, SPEC_DTYPE_F16, SPEC_DTYPE_I8, SPEC_DTYPE_I32 = 0, 1, 2, 3, 4
SPEC_OK, SPEC_ERR_INVALID, SPEC_ERR_UNSUPPORTED, SPEC_ERR_CUDA = 0, -1, -2, -3
SPEC_OPT_ATTN_PATH, SPEC_OPT_NUM_CTAS, SPEC_OPT_VALIDATE, SPEC_OPT_SIMT_CHUNK = 0, 1, 2, 3
SPEC_OPT_SPLIT_WEIGHT = 4
SPEC_OPT_SMALL_CLUSTER = 5
NUM_OPTIONS = 6
SPEC_DEVERR_PAGE, SPEC_DEVERR_CTX, SPEC_DEVERR_TIMEOUT, SPEC_DEVERR_TOKEN = 1, 2, 4, 8
SPEC_DEVERR_TREE = 16
SPEC_DEVERR_CODEC = 32

# every symbol the public header declares
EXPORTED = ["spec_version", "spec_last_error", "spec_set_option", "spec_verify_attn",
            "spec_accept_greedy", "spec_verify_attn_tensors", "spec_accept_greedy_tensors",
            "spec_accept_greedy_noalloc", "spec_accept_rejection",
            "spec_kv_append", "spec_commit", "spec_verify_attn_tree", "spec_accept_tree",
            "spec_codec_encode", "spec_codec_decode", "spec_device_error", "spec_release"]
SPEC_NOALLOC_MAX_PARTIALS, SPEC_NOALLOC_MAX_BATCH = 65536, 4096

_TORCH_DT = {torch.float32: SPEC_DTYPE_F32, torch.bfloat16: SPEC_DTYPE_BF16,
             torch.float16: SPEC_DTYPE_F16, torch.int8: SPEC_DTYPE_I8,
             torch.int32: SPEC_DTYPE_I32}


class SpecTensor(ctypes.Structure):
    """spec_tensor_t: data pointer, element type, rank, shape, strides (elements)."""
    _fields_ = [("data", ctypes.c_void_p), ("dtype", ctypes.c_int32), ("ndim", ctypes.c_int32),
                ("shape", ctypes.c_int64 * 4), ("stride", ctypes.c_int64 * 4)]


def tensor_desc(t: Optional[torch.Tensor]):
    """The spec_tensor_t of a torch tensor (any strides; None stays None)."""
    if t is None:
        return None
    if t.dim() > 4:
        raise ValueError("descriptors hold at most 4 dimensions")
    d = SpecTensor()
    d.data = t.data_ptr()
    d.dtype = _TORCH_DT[t.dtype]
    d.ndim = t.dim()
    for i, (n, st) in enumerate(zip(t.shape, t.stride())):
        d.shape[i] = n
        d.stride[i] = st
    return d

_lib = None


class SpecError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__("spec call failed (%d): %s" % (code, msg))
        self.code = code


def load():
    """Load the in-tree library (once).  Raises if it is missing."""
    global _lib
    if _lib is None:
        _lib = _open(LIB_PATH)
    return _lib


def _open(path: str):
    if not os.path.exists(path):
        raise RuntimeError("libspecverify.so not built at %s; run __graft_entry__.build()" % path)
    lib = ctypes.CDLL(path)
    P, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    lib.spec_version.restype = ctypes.c_int
    lib.spec_last_error.restype = ctypes.c_char_p
    lib.spec_set_option.argtypes = [i32, i64]
    lib.spec_set_option.restype = ctypes.c_int
    lib.spec_verify_attn.argtypes = [P, P, P, P, P, P, P, i32, i32, i32, i32, i32, i32, i32, i32,
                                     i32, i32, ctypes.c_float, P, P, P]
    lib.spec_verify_attn.restype = ctypes.c_int
    lib.spec_accept_greedy.argtypes = [P, i32, P, i32, i32, i64, P, P, P]
    lib.spec_accept_greedy.restype = ctypes.c_int
    lib.spec_accept_greedy_noalloc.argtypes = [P, i32, P, i32, i32, i64, P, P, P]
    lib.spec_accept_greedy_noalloc.restype = ctypes.c_int
    lib.spec_accept_rejection.argtypes = [P, P, i32, P, i32, i32, i64, ctypes.c_float,
                                          ctypes.c_uint64, P, P, P]
    lib.spec_accept_rejection.restype = ctypes.c_int
    lib.spec_kv_append.argtypes = [P, P, i32, P, P, P, P, i32, P, P, i32, i32, i32, i32, i32, i32,
                                   i32, P]
    lib.spec_kv_append.restype = ctypes.c_int
    lib.spec_commit.argtypes = [P, P, i32, i32, P]
    lib.spec_commit.restype = ctypes.c_int
    lib.spec_codec_encode.argtypes = [P, ctypes.c_int64, i32, i32, P, P, P]
    lib.spec_codec_encode.restype = ctypes.c_int
    lib.spec_codec_decode.argtypes = [P, P, ctypes.c_int64, i32, i32, P, P]
    lib.spec_codec_decode.restype = ctypes.c_int
    lib.spec_verify_attn_tree.argtypes = [P, P, P, P, P, P, P, P, i32, i32, i32, i32, i32, i32, i32,
                                          i32, i32, i32, ctypes.c_float, P, P, P]
    lib.spec_verify_attn_tree.restype = ctypes.c_int
    lib.spec_accept_tree.argtypes = [P, i32, P, P, i32, i32, i64, P, P, P, P]
    lib.spec_accept_tree.restype = ctypes.c_int
    T = ctypes.POINTER(SpecTensor)
    lib.spec_verify_attn_tensors.argtypes = [T, T, T, T, T, T, T, i32, ctypes.c_float, T, T, P]
    lib.spec_verify_attn_tensors.restype = ctypes.c_int
    lib.spec_accept_greedy_tensors.argtypes = [T, T, i32, T, T, P]
    lib.spec_accept_greedy_tensors.restype = ctypes.c_int
    lib.spec_device_error.argtypes = [ctypes.POINTER(ctypes.c_int32)]
    lib.spec_device_error.restype = ctypes.c_int
    lib.spec_release.restype = ctypes.c_int
    return lib


def _check(rc: int):
    if rc != SPEC_OK:
        raise SpecError(rc, load().spec_last_error().decode())


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def spec_version() -> int:
    return load().spec_version()


def spec_last_error() -> str:
    return load().spec_last_error().decode()


def spec_set_option(option: int, value: int) -> None:
    _check(load().spec_set_option(option, int(value)))


def spec_verify_attn(q, k_cache, v_cache, block_table, ctx_lens, num_draft: int, scale: float,
                     out, lse=None, k_scale=None, v_scale=None, stream=None) -> None:
    """Verification attention; writes ``out`` (and ``lse`` if given).

    q [B, k, Hq, D]; k_cache / v_cache [NP, Hkv, P, D]; block_table
    [B, max_pages] int32; ctx_lens [B] int32; out like q; lse [B, k, Hq] f32;
    k_scale / v_scale [NP, Hkv, P] fp16 for an int8 cache.
    """
    B, k, Hq, D = q.shape
    NP, Hkv, P, D2 = k_cache.shape
    if k != num_draft or D2 != D:
        raise ValueError("shape mismatch between q, num_draft and the cache")
    if block_table.dtype != torch.int32 or ctx_lens.dtype != torch.int32:
        raise ValueError("block_table and ctx_lens must be int32")
    _check(load().spec_verify_attn(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale), _ptr(block_table),
        _ptr(ctx_lens), B, k, Hq, Hkv, D, P, NP, block_table.shape[1], _TORCH_DT[q.dtype],
        _TORCH_DT[k_cache.dtype], float(scale), _ptr(out), _ptr(lse), _stream(stream)))


def _ref(d):
    return None if d is None else ctypes.byref(d)


def spec_verify_attn_tensors(q, k_cache, v_cache, block_table, ctx_lens, num_draft: int,
                             scale: float, out, lse=None, k_scale=None, v_scale=None,
                             stream=None) -> None:
    """spec_verify_attn through the descriptor form (sizes and strides are
    read from the tensors; the library checks them)."""
    descs = [tensor_desc(t) for t in (q, k_cache, v_cache, k_scale, v_scale, block_table,
                                      ctx_lens, out, lse)]
    _check(load().spec_verify_attn_tensors(*[_ref(d) for d in descs[:7]], int(num_draft),
                                           float(scale), _ref(descs[7]), _ref(descs[8]),
                                           _stream(stream)))


def spec_accept_greedy_tensors(logits, draft_tokens, num_draft: int, accepted_len, next_token,
                               stream=None) -> None:
    """spec_accept_greedy through the descriptor form."""
    descs = [tensor_desc(t) for t in (logits, draft_tokens, accepted_len, next_token)]
    _check(load().spec_accept_greedy_tensors(_ref(descs[0]), _ref(descs[1]), int(num_draft),
                                             _ref(descs[2]), _ref(descs[3]), _stream(stream)))


def spec_verify_attn_tree(q, k_cache, v_cache, block_table, ctx_lens, tree_mask, num_draft: int,
                          scale: float, out, lse=None, k_scale=None, v_scale=None,
                          stream=None) -> None:
    """spec_verify_attn with draft visibility from ``tree_mask`` (64-bit [B, k],
    bit t of row i: query i sees draft t; int64 or uint64 tensor)."""
    B, k, Hq, D = q.shape
    NP, Hkv, P, D2 = k_cache.shape
    if k != num_draft or D2 != D or tuple(tree_mask.shape) != (B, k):
        raise ValueError("q must be [B, num_draft, Hq, D], tree_mask [B, num_draft]")
    if tree_mask.element_size() != 8:
        raise ValueError("tree_mask must hold 64-bit words")
    _check(load().spec_verify_attn_tree(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale), _ptr(block_table),
        _ptr(ctx_lens), _ptr(tree_mask), B, k, Hq, Hkv, D, P, NP, block_table.shape[1],
        _TORCH_DT[q.dtype], _TORCH_DT[k_cache.dtype], float(scale), _ptr(out), _ptr(lse),
        _stream(stream)))


def spec_accept_tree(logits, draft_tokens, parents, num_draft: int, accepted_len, next_token,
                     path=None, stream=None) -> None:
    """Greedy acceptance over a tree of drafts (parents int32 [B, k] in [-1, i))."""
    B, k1, V = logits.shape
    if (k1 != num_draft + 1 or tuple(draft_tokens.shape) != (B, num_draft)
            or tuple(parents.shape) != (B, num_draft)):
        raise ValueError("logits [B, k+1, V], drafts and parents [B, k]")
    _check(load().spec_accept_tree(_ptr(logits), _TORCH_DT[logits.dtype], _ptr(draft_tokens),
                                   _ptr(parents), B, num_draft, V, _ptr(accepted_len),
                                   _ptr(next_token), _ptr(path), _stream(stream)))


def spec_accept_greedy(logits, draft_tokens, num_draft: int, accepted_len, next_token,
                       stream=None) -> None:
    """Greedy acceptance; writes ``accepted_len`` and ``next_token`` (int32 [B])."""
    B, k1, V = logits.shape
    if k1 != num_draft + 1 or tuple(draft_tokens.shape) != (B, num_draft):
        raise ValueError("logits must be [B, num_draft+1, V] and drafts [B, num_draft]")
    _check(load().spec_accept_greedy(_ptr(logits), _TORCH_DT[logits.dtype], _ptr(draft_tokens), B,
                                     num_draft, V, _ptr(accepted_len), _ptr(next_token),
                                     _stream(stream)))


def spec_accept_greedy_noalloc(logits, draft_tokens, num_draft: int, accepted_len, next_token,
                               stream=None) -> None:
    """spec_accept_greedy without any device allocation (fixed library scratch).

    For callers that cannot allocate device memory, e.g. a serving loop whose
    GPU memory is reserved up front by its own allocator.  Sizes are limited
    (see include/spec_verify.h); calls that overlap on the GPU share the
    scratch and race.
    """
    B, k1, V = logits.shape
    if k1 != num_draft + 1 or tuple(draft_tokens.shape) != (B, num_draft):
        raise ValueError("logits must be [B, num_draft+1, V] and drafts [B, num_draft]")
    _check(load().spec_accept_greedy_noalloc(_ptr(logits), _TORCH_DT[logits.dtype],
                                             _ptr(draft_tokens), B, num_draft, V,
                                             _ptr(accepted_len), _ptr(next_token),
                                             _stream(stream)))


def spec_accept_rejection(target_logits, draft_logits, draft_tokens, num_draft: int,
                          temperature: float, seed: int, accepted_len, next_token,
                          stream=None) -> None:
    """Rejection-sampling acceptance; writes ``accepted_len`` and ``next_token``.

    target_logits [B, k+1, V], draft_logits [B, k, V] (same dtype), drafts
    int32 [B, k]; draws from SplitMix64 keyed by ``seed``.
    """
    B, k1, V = target_logits.shape
    if (k1 != num_draft + 1 or tuple(draft_logits.shape) != (B, num_draft, V)
            or tuple(draft_tokens.shape) != (B, num_draft)):
        raise ValueError("target_logits must be [B, k+1, V], draft_logits [B, k, V], drafts [B, k]")
    if draft_logits.dtype != target_logits.dtype:
        raise ValueError("target and draft logits must share a dtype")
    _check(load().spec_accept_rejection(_ptr(target_logits), _ptr(draft_logits),
                                        _TORCH_DT[target_logits.dtype], _ptr(draft_tokens), B,
                                        num_draft, V, float(temperature),
                                        int(seed) & (2**64 - 1), _ptr(accepted_len),
                                        _ptr(next_token), _stream(stream)))


def spec_kv_append(k_new, v_new, k_cache, v_cache, block_table, ctx_lens, k_scale=None,
                   v_scale=None, stream=None) -> None:
    """Write k_new / v_new [B, n, Hkv, D] at positions ctx_b .. ctx_b + n - 1 of
    the paged caches (INT8 caches are quantised into k_scale / v_scale)."""
    B, n, Hkv, D = k_new.shape
    NP, Hkv2, P, D2 = k_cache.shape
    if (Hkv2, D2) != (Hkv, D) or tuple(v_new.shape) != tuple(k_new.shape):
        raise ValueError("k_new / v_new must be [B, n, Hkv, D] matching the cache")
    _check(load().spec_kv_append(_ptr(k_new), _ptr(v_new), _TORCH_DT[k_new.dtype], _ptr(k_cache),
                                 _ptr(v_cache), _ptr(k_scale), _ptr(v_scale),
                                 _TORCH_DT[k_cache.dtype], _ptr(block_table), _ptr(ctx_lens), B,
                                 n, Hkv, D, P, NP, block_table.shape[1], _stream(stream)))


def spec_codec_encode(codes, pairs, num_pairs, stream=None) -> None:
    """codes int8 [num_blocks, P, D] -> pairs uint8 [num_blocks, 2*P*D], num_pairs int32."""
    nblk, P, D = codes.shape
    _check(load().spec_codec_encode(_ptr(codes), nblk, P, D, _ptr(pairs), _ptr(num_pairs),
                                    _stream(stream)))


def spec_codec_decode(pairs, num_pairs, codes, stream=None) -> None:
    """pairs uint8 [num_blocks, 2*P*D], num_pairs int32 -> codes int8 [num_blocks, P, D]."""
    nblk, P, D = codes.shape
    _check(load().spec_codec_decode(_ptr(pairs), _ptr(num_pairs), nblk, P, D, _ptr(codes),
                                    _stream(stream)))


def spec_commit(ctx_lens, accepted_len, extra: int = 1, stream=None) -> None:
    """ctx_lens[b] += accepted_len[b] + extra, on the device."""
    _check(load().spec_commit(_ptr(ctx_lens), _ptr(accepted_len), ctx_lens.shape[0], int(extra),
                              _stream(stream)))


def spec_device_error() -> int:
    v = ctypes.c_int32(0)
    _check(load().spec_device_error(ctypes.byref(v)))
    return v.value


def spec_release() -> None:
    _check(load().spec_release())


# ---------------------------------------------------------------- plumbing

def _np_to_torch(a: np.ndarray, kind: str) -> torch.Tensor:
    if kind == "bf16":
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
    if kind == "f16":
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.float16)
    return torch.from_numpy(np.ascontiguousarray(a))


def inputs_to_torch(inp, device="cuda", pin: bool = False) -> dict:
    """Generator output (numpy) -> torch tensors on `device` (or pinned host)."""
    s = inp.spec
    t = {
        "q": _np_to_torch(inp.q, s.q_dtype),
        "k_cache": _np_to_torch(inp.k_cache, s.kv_dtype),
        "v_cache": _np_to_torch(inp.v_cache, s.kv_dtype),
        "block_table": torch.from_numpy(inp.block_table),
        "ctx_lens": torch.from_numpy(inp.ctx_lens),
        "logits": _np_to_torch(inp.logits, s.logits_dtype),
        "draft_tokens": torch.from_numpy(inp.draft_tokens),
    }
    if inp.k_scale is not None:
        t["k_scale"] = _np_to_torch(inp.k_scale, "f16")
        t["v_scale"] = _np_to_torch(inp.v_scale, "f16")
    if pin:
        return {n: v.pin_memory() for n, v in t.items()}
    return {n: v.to(device) for n, v in t.items()}


def alloc_outputs(inp, device="cuda") -> dict:
    s = inp.spec
    qdt = torch.float32 if s.q_dtype == "f32" else torch.bfloat16
    B, k = s.batch, s.num_draft
    return {
        "out": torch.empty((B, k, s.num_q_heads, s.head_dim), dtype=qdt, device=device),
        "lse": torch.empty((B, k, s.num_q_heads), dtype=torch.float32, device=device),
        "accepted_len": torch.empty((B,), dtype=torch.int32, device=device),
        "next_token": torch.empty((B,), dtype=torch.int32, device=device),
    }


def run_verify(t: dict, o: dict, num_draft: int, scale: float, stream=None) -> None:
    """One verification step: attention, then acceptance, on one stream."""
    spec_verify_attn(t["q"], t["k_cache"], t["v_cache"], t["block_table"], t["ctx_lens"],
                     num_draft, scale, o["out"], o["lse"], t.get("k_scale"), t.get("v_scale"),
                     stream=stream)
    spec_accept_greedy(t["logits"], t["draft_tokens"], num_draft, o["accepted_len"],
                       o["next_token"], stream=stream)

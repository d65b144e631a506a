"""Seeded synthetic inputs for speculative-decoding verification.

This module only makes inputs: it holds none of the verification arithmetic
(no attention, no acceptance).  Both the CUDA path and the CPU oracle consume
what it returns, so it depends on numpy alone and returns host arrays; 16-bit
float tensors are returned as their raw ``uint16`` bits.

Recipe (one ``numpy.random.SeedSequence`` per call, spawned into fixed
streams so every array is reproducible on any platform):

* ``ctx_lens``: fixed, or uniform integers in ``[lo, hi]`` per sequence.
* paged cache ``[num_pages, Hkv, P, D]``: every sequence owns
  ``ceil((ctx_b + k) / P)`` pages; physical page ids are a random
  permutation of all pages, so consecutive logical pages are scattered.
* q, K, V ~ N(0, 1), rounded (to nearest even) to the stored dtype.
* INT8 cache: each (token, kv-head) row of D bf16 values is quantised as in
  CXL-SpecKV's "Algorithm 2 KV-Cache Compression" (s = max|x| / 127,
  c = round(x / s)), with s stored as fp16 and c clamped to [-127, 127];
  rounding is to nearest even.
* cache slots past ``ctx_b + k`` in a sequence's last page are canaries:
  NaN (float caches) or a NaN fp16 scale (INT8 caches), or zeros when
  ``canary=False``.
* logits ``[B, k+1, V]`` ~ N(0, sigma) rounded to the logits dtype.
* drafts: with probability ``match_prob`` a position copies the target's
  argmax (first index of the row maximum, found with ``numpy.argmax`` on
  the stored values); otherwise it draws a token per ``draft_mode``:
  ``"uniform"`` (any token, may coincide with the argmax), ``"mismatch"``
  (uniform over the other V-1 tokens) or ``"geometric_break"`` (positions
  match independently until the first miss, and every later position is a
  forced mismatch).
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional, Sequence, Tuple, Union

import numpy as np

Ctx = Union[int, Tuple[int, int], Sequence[int]]


@dataclasses.dataclass(frozen=True)
class WorkloadSpec:
    name: str
    batch: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    ctx: Ctx                # int: fixed; (lo, hi): uniform inclusive; list: explicit per sequence
    num_draft: int
    page_size: int
    vocab: int
    q_dtype: str = "bf16"   # "f32" | "bf16"
    kv_dtype: str = "bf16"  # "f32" | "bf16" | "i8"
    logits_dtype: str = "bf16"
    logit_sigma: float = math.sqrt(2.0)
    match_prob: float = 0.75
    draft_mode: str = "mismatch"

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads


# The five named workloads: shapes of real verification calls.
WORKLOADS = {
    "tiny_fp32": WorkloadSpec(
        "tiny_fp32", batch=1, num_q_heads=2, num_kv_heads=2, head_dim=64, ctx=128,
        num_draft=4, page_size=16, vocab=1000, q_dtype="f32", kv_dtype="f32",
        logits_dtype="f32", logit_sigma=1.0, match_prob=0.8, draft_mode="uniform"),
    "mha7b_bf16": WorkloadSpec(
        "mha7b_bf16", batch=8, num_q_heads=32, num_kv_heads=32, head_dim=128, ctx=2048,
        num_draft=8, page_size=16, vocab=32000, match_prob=0.75),
    "gqa8b_ragged_bf16": WorkloadSpec(
        "gqa8b_ragged_bf16", batch=32, num_q_heads=32, num_kv_heads=8, head_dim=128,
        ctx=(1024, 8192), num_draft=4, page_size=16, vocab=128256, match_prob=0.7),
    "long_step_k16_bf16": WorkloadSpec(
        "long_step_k16_bf16", batch=4, num_q_heads=28, num_kv_heads=4, head_dim=128,
        ctx=32768, num_draft=16, page_size=32, vocab=152064, match_prob=0.85,
        draft_mode="geometric_break"),
    "int8kv_70b_layer": WorkloadSpec(
        "int8kv_70b_layer", batch=32, num_q_heads=64, num_kv_heads=8, head_dim=128, ctx=2048,
        num_draft=8, page_size=16, vocab=32000, q_dtype="bf16", kv_dtype="i8",
        match_prob=0.75),
}
WORKLOAD_ORDER = ["tiny_fp32", "mha7b_bf16", "gqa8b_ragged_bf16", "long_step_k16_bf16",
                  "int8kv_70b_layer"]


@dataclasses.dataclass
class VerifyInputs:
    spec: WorkloadSpec
    seed: int
    q: np.ndarray            # [B, k, Hq, D]    float32 or uint16 (bf16 bits)
    k_cache: np.ndarray      # [NP, Hkv, P, D]  float32, uint16 (bf16 bits) or int8
    v_cache: np.ndarray
    k_scale: Optional[np.ndarray]  # [NP, Hkv, P] uint16 (fp16 bits) for int8 caches
    v_scale: Optional[np.ndarray]
    block_table: np.ndarray  # [B, max_pages] int32
    ctx_lens: np.ndarray     # [B] int32
    logits: np.ndarray       # [B, k+1, V] float32 or uint16 (bf16 bits)
    draft_tokens: np.ndarray  # [B, k] int32
    scale: float             # softmax scale, float32-representable

    @property
    def num_pages(self) -> int:
        return self.k_cache.shape[0]

    @property
    def max_pages(self) -> int:
        return self.block_table.shape[1]


# ---------------------------------------------------------------- dtype helpers

def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (nearest, ties to even); finite inputs."""
    u = np.ascontiguousarray(x, np.float32).view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


BF16_NAN = np.uint16(0x7FC0)
F16_NAN = np.uint16(0x7E00)


def _round_to(x32: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "f32":
        return x32.astype(np.float32)
    if dtype == "bf16":
        return f32_to_bf16_bits(x32)
    raise ValueError(dtype)


def _as_f32(stored: np.ndarray, dtype: str) -> np.ndarray:
    return stored if dtype == "f32" else bf16_bits_to_f32(stored)


def quantize_int8_rows(x_bf16_bits: np.ndarray) -> Tuple[np.ndarray, np.ndarray]:
    """Per-row symmetric INT8 quantisation of bf16 rows (last axis).

    Returns (codes int8 [..., D], scale fp16 bits [...]).  Input preparation
    for the INT8 cache format; the product path only ever dequantises.
    """
    x = bf16_bits_to_f32(x_bf16_bits)
    amax = np.max(np.abs(x), axis=-1)
    s16 = (amax / np.float32(127.0)).astype(np.float16)
    s32 = s16.astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        c = np.rint(x / s32[..., None])
    c = np.where(s32[..., None] > 0, c, 0.0)
    c = np.clip(c, -127, 127).astype(np.int8)
    return c, s16.view(np.uint16)


# ---------------------------------------------------------------- generator

def _ctx_lens(spec: WorkloadSpec, rng: np.random.Generator) -> np.ndarray:
    c = spec.ctx
    if isinstance(c, int):
        return np.full(spec.batch, c, np.int32)
    if isinstance(c, tuple) and len(c) == 2:
        return rng.integers(c[0], c[1] + 1, size=spec.batch).astype(np.int32)
    arr = np.asarray(c, np.int32)
    assert arr.shape == (spec.batch,)
    return arr


def _normal_cache(rng, shape, dtype, chunk_pages=512):
    """N(0,1) cache of `shape` rounded to dtype, generated in page chunks."""
    out = np.empty(shape, np.float32 if dtype == "f32" else np.uint16)
    n = shape[0]
    per_page = int(np.prod(shape[1:]))
    for p0 in range(0, n, chunk_pages):
        p1 = min(n, p0 + chunk_pages)
        x = rng.standard_normal((p1 - p0) * per_page, dtype=np.float32)
        out[p0:p1] = _round_to(x, dtype).reshape((p1 - p0,) + tuple(shape[1:]))
    return out


def make_inputs(spec: Union[WorkloadSpec, str], seed: int = 0, canary: bool = True) -> VerifyInputs:
    if isinstance(spec, str):
        spec = WORKLOADS[spec]
    B, Hq, Hkv, D = spec.batch, spec.num_q_heads, spec.num_kv_heads, spec.head_dim
    k, P, V = spec.num_draft, spec.page_size, spec.vocab
    assert Hq % Hkv == 0 and k >= 1 and P >= 1
    streams = [np.random.default_rng(s) for s in np.random.SeedSequence(seed).spawn(9)]
    r_ctx, r_pages, r_q, r_k, r_v, r_logits, r_match, r_tok, r_break = streams

    ctx_lens = _ctx_lens(spec, r_ctx)
    n_pages = (ctx_lens.astype(np.int64) + k + P - 1) // P
    NP = int(n_pages.sum())
    max_pages = int(n_pages.max()) if B else 1
    perm = r_pages.permutation(NP).astype(np.int32)
    block_table = np.zeros((B, max_pages), np.int32)
    off = 0
    for b in range(B):
        block_table[b, : n_pages[b]] = perm[off: off + n_pages[b]]
        off += n_pages[b]

    q = _round_to(r_q.standard_normal((B, k, Hq, D), dtype=np.float32), spec.q_dtype)

    k_scale = v_scale = None
    if spec.kv_dtype == "i8":
        kb = _normal_cache(r_k, (NP, Hkv, P, D), "bf16")
        vb = _normal_cache(r_v, (NP, Hkv, P, D), "bf16")
        k_cache, k_scale = quantize_int8_rows(kb)
        v_cache, v_scale = quantize_int8_rows(vb)
        del kb, vb
    else:
        k_cache = _normal_cache(r_k, (NP, Hkv, P, D), spec.kv_dtype)
        v_cache = _normal_cache(r_v, (NP, Hkv, P, D), spec.kv_dtype)

    # Slots past the last key of each sequence: canaries (or zeros).
    for b in range(B):
        used = int(ctx_lens[b]) + k
        last_page = block_table[b, n_pages[b] - 1]
        first_free = used - (int(n_pages[b]) - 1) * P
        if first_free >= P:
            continue
        if spec.kv_dtype == "i8":
            k_cache[last_page, :, first_free:, :] = 0
            v_cache[last_page, :, first_free:, :] = 0
            fill = F16_NAN if canary else np.uint16(0)
            k_scale[last_page, :, first_free:] = fill
            v_scale[last_page, :, first_free:] = fill
        else:
            if spec.kv_dtype == "f32":
                fill = np.float32(np.nan) if canary else np.float32(0)
            else:
                fill = BF16_NAN if canary else np.uint16(0)
            k_cache[last_page, :, first_free:, :] = fill
            v_cache[last_page, :, first_free:, :] = fill

    logits = _round_to(
        r_logits.standard_normal((B, k + 1, V), dtype=np.float32) * np.float32(spec.logit_sigma),
        spec.logits_dtype)
    target = np.argmax(_as_f32(logits[:, :k, :], spec.logits_dtype), axis=-1).astype(np.int64)

    u = r_match.random((B, k))
    match = u < spec.match_prob
    if spec.draft_mode == "geometric_break":
        # positions agree until the first miss; every later one is a miss
        match = np.cumprod(match, axis=1).astype(bool)
    if spec.draft_mode == "uniform" or V == 1:
        other = r_tok.integers(0, V, size=(B, k))
    else:
        # uniform over the V-1 tokens that differ from the target's argmax
        other = r_tok.integers(0, V - 1, size=(B, k))
        other = other + (other >= target)
    draft = np.where(match, target, other).astype(np.int32)

    scale = float(np.float32(1.0 / math.sqrt(D)))
    return VerifyInputs(spec=spec, seed=seed, q=q, k_cache=k_cache, v_cache=v_cache,
                        k_scale=k_scale, v_scale=v_scale, block_table=block_table,
                        ctx_lens=ctx_lens, logits=logits, draft_tokens=draft, scale=scale)


def small_spec(name="small", **kw) -> WorkloadSpec:
    """A small workload for parity tests; keyword arguments override fields."""
    base = dict(batch=3, num_q_heads=8, num_kv_heads=2, head_dim=128, ctx=(40, 300),
                num_draft=4, page_size=16, vocab=1000)
    base.update(kw)
    return WorkloadSpec(name, **base)


def algorithmic_bytes(inp: VerifyInputs) -> dict:
    """Bytes the verification step must move at least once (per call).

    KV: every sequence's ctx_b + k keys, read once per (sequence, kv-head)
    (plus the fp16 scales for an INT8 cache); Q read, out written (q's
    dtype), lse written (fp32), block-table entries and ctx_lens read; all
    k+1 logits rows read; drafts read; accepted_len and next_token written.
    """
    s = inp.spec
    B, k, Hq, Hkv, D = s.batch, s.num_draft, s.num_q_heads, s.num_kv_heads, s.head_dim
    keys = int((inp.ctx_lens.astype(np.int64) + k).sum())
    kv_elem = {"f32": 4, "bf16": 2, "i8": 1}[s.kv_dtype]
    kv = 2 * keys * Hkv * D * kv_elem
    if s.kv_dtype == "i8":
        kv += 2 * keys * Hkv * 2
    q_elem = 4 if s.q_dtype == "f32" else 2
    pages_used = int(((inp.ctx_lens.astype(np.int64) + k + s.page_size - 1) // s.page_size).sum())
    attn = kv + 2 * B * k * Hq * D * q_elem + B * k * Hq * 4 + pages_used * 4 + B * 4
    lg_elem = 4 if s.logits_dtype == "f32" else 2
    accept = B * (k + 1) * s.vocab * lg_elem + B * k * 4 + 2 * B * 4
    return {"attn": attn, "accept": accept, "total": attn + accept, "kv": kv}


# ---------------------------------------------------------------- rejection-sampling inputs

@dataclasses.dataclass
class RejectionInputs:
    """Seeded inputs of rejection-sampling acceptance (stored dtype bits as
    in VerifyInputs: float32 arrays, or uint16 bf16 bits)."""
    dtype: str
    target_logits: np.ndarray  # [B, k+1, V]
    draft_logits: np.ndarray   # [B, k, V]
    draft_tokens: np.ndarray   # [B, k] int32, drawn from the drafter's distribution
    temperature: float
    seed: int                  # key of the verification draws


def make_rejection_inputs(batch: int, num_draft: int, vocab: int, dtype: str = "bf16",
                          seed: int = 0, sigma: float = math.sqrt(2.0), agreement: float = 0.8,
                          temperature: float = 1.0) -> RejectionInputs:
    """Target logits N(0, sigma^2); the drafter's logits are agreement * target
    + sqrt(1 - agreement^2) * fresh noise (a drafter that mostly agrees); each
    draft token is drawn from the drafter's softmax(logits / T) with numpy's
    generator (input construction only)."""
    rng = np.random.default_rng(np.random.SeedSequence([seed, 0x5EC]))
    B, k, V = batch, num_draft, vocab
    tl = rng.standard_normal((B, k + 1, V), dtype=np.float32) * np.float32(sigma)
    noise = rng.standard_normal((B, k, V), dtype=np.float32) * np.float32(sigma)
    a = np.float32(agreement)
    dl = a * tl[:, :k] + np.float32(math.sqrt(max(0.0, 1.0 - agreement ** 2))) * noise
    tl_s, dl_s = _round_to(tl, dtype), _round_to(dl.astype(np.float32), dtype)
    # draft tokens ~ softmax(stored draft logits / T), by inverse CDF on float64
    dq = _as_f32(dl_s, dtype).astype(np.float64) / temperature
    dq -= dq.max(axis=-1, keepdims=True)
    cdf = np.cumsum(np.exp(dq), axis=-1)
    u = rng.random((B, k, 1)) * cdf[..., -1:]
    drafts = np.minimum((cdf < u).sum(axis=-1), V - 1).astype(np.int32)
    return RejectionInputs(dtype=dtype, target_logits=tl_s, draft_logits=dl_s,
                           draft_tokens=np.ascontiguousarray(drafts), temperature=temperature,
                           seed=int(rng.integers(0, 2**63)))


# ---------------------------------------------------------------- draft trees

def tree_masks(parents: np.ndarray) -> np.ndarray:
    """Ancestor masks of draft trees: bit t of mask[b, i] is set when node t is
    node i or one of its ancestors.  parents [B, k] int32, parent < index,
    -1 for children of the last committed token."""
    B, k = parents.shape
    masks = np.zeros((B, k), np.uint64)
    for b in range(B):
        for i in range(k):
            p = int(parents[b, i])
            assert -1 <= p < i
            masks[b, i] = (masks[b, p] if p >= 0 else np.uint64(0)) | np.uint64(1 << i)
    return masks


def random_trees(batch: int, num_draft: int, seed: int = 0, width: float = 0.5) -> np.ndarray:
    """Seeded draft trees: node i's parent is -1 or an earlier node, nearer
    nodes likelier (width 0: a chain, larger: bushier)."""
    rng = np.random.default_rng(np.random.SeedSequence([seed, 0x7EE]))
    parents = np.zeros((batch, num_draft), np.int32)
    for b in range(batch):
        for i in range(num_draft):
            if i == 0 or rng.random() >= width:
                parents[b, i] = i - 1
            else:
                parents[b, i] = int(rng.integers(-1, i))
    return parents


def plant_tree_tokens(logits_f32: np.ndarray, parents: np.ndarray, match: float,
                      seed: int = 0) -> np.ndarray:
    """Draft tokens of a tree: node i copies the target's argmax at its parent
    with probability `match`, else a different random token (input
    construction; numpy.argmax on the stored logits)."""
    rng = np.random.default_rng(np.random.SeedSequence([seed, 0x70C]))
    B, k = parents.shape
    V = logits_f32.shape[-1]
    am = np.argmax(logits_f32, axis=-1)  # [B, k+1]
    tokens = np.zeros((B, k), np.int32)
    for b in range(B):
        for i in range(k):
            target = am[b, parents[b, i] + 1]
            if rng.random() < match:
                tokens[b, i] = target
            else:
                o = int(rng.integers(0, V - 1))
                tokens[b, i] = o + (o >= target)
    return tokens

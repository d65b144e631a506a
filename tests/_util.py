"""Shared test helpers: call the oracle on generator output, compare results."""
from __future__ import annotations

import numpy as np

from speculative_decoding_verification_attn_gb300.workload import VerifyInputs, bf16_bits_to_f32


def oracle_attn(oracle, inp: VerifyInputs):
    s = inp.spec
    return oracle.verify_attn(inp.q, s.q_dtype, inp.k_cache, inp.v_cache, s.kv_dtype,
                              inp.k_scale, inp.v_scale, inp.block_table, inp.ctx_lens, inp.scale)


def oracle_rows(oracle, inp: VerifyInputs, rows):
    s = inp.spec
    return oracle.attn_rows(inp.q, s.q_dtype, inp.k_cache, inp.v_cache, s.kv_dtype,
                            inp.k_scale, inp.v_scale, inp.block_table, inp.ctx_lens, inp.scale,
                            rows)


def oracle_accept(oracle, inp: VerifyInputs):
    return oracle.accept_greedy(inp.logits, inp.spec.logits_dtype, inp.draft_tokens)


def stored_to_f64(arr: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "f32":
        return arr.astype(np.float64)
    if dtype == "bf16":
        return bf16_bits_to_f32(arr).astype(np.float64)
    if dtype == "f16":
        return arr.view(np.float16).astype(np.float64)
    if dtype == "i8":
        return arr.astype(np.float64)
    raise ValueError(dtype)


def rel_l2(a, b) -> float:
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    den = np.linalg.norm(b.ravel())
    return float(np.linalg.norm((a - b).ravel()) / (den if den > 0 else 1.0))


def host_threads() -> int:
    """Host cores this process may run on."""
    import os
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:
        return max(1, os.cpu_count() or 1)


def all_rows(inp: VerifyInputs) -> np.ndarray:
    """Every (b, i, h) output row of a call, row-major like out[B, k, Hq]."""
    s = inp.spec
    grid = np.meshgrid(np.arange(s.batch), np.arange(s.num_draft), np.arange(s.num_q_heads),
                       indexing="ij")
    return np.stack(grid, -1).reshape(-1, 3).astype(np.int32)


def oracle_rows_parallel(oracle, inp: VerifyInputs, rows, threads=None):
    """oracle_rows over chunks of rows on every host core.  The oracle is a C
    library called through ctypes, which releases the GIL for the call, so
    threads run it in parallel on the same (shared, read-only) inputs."""
    from concurrent.futures import ThreadPoolExecutor
    rows = np.ascontiguousarray(np.asarray(rows, np.int32).reshape(-1, 3))
    threads = threads or host_threads()
    n = rows.shape[0]
    if n == 0:
        return np.zeros((0, inp.spec.head_dim)), np.zeros((0,))
    chunks = [c for c in np.array_split(rows, min(n, 8 * threads)) if len(c)]
    with ThreadPoolExecutor(max_workers=threads) as ex:
        parts = list(ex.map(lambda c: oracle_rows(oracle, inp, np.ascontiguousarray(c)), chunks))
    return (np.concatenate([p[0] for p in parts]), np.concatenate([p[1] for p in parts]))

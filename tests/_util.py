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

"""The seeded input generator: reproducibility, layout and the stated recipe."""
from __future__ import annotations

import numpy as np
import pytest

from speculative_decoding_verification_attn_gb300.workload import (
    WORKLOADS, bf16_bits_to_f32, f32_to_bf16_bits, make_inputs, quantize_int8_rows, small_spec)


def test_deterministic_per_seed():
    a = make_inputs(small_spec(kv_dtype="i8"), seed=4)
    b = make_inputs(small_spec(kv_dtype="i8"), seed=4)
    c = make_inputs(small_spec(kv_dtype="i8"), seed=5)
    for f in ("q", "k_cache", "v_cache", "k_scale", "block_table", "ctx_lens", "logits",
              "draft_tokens"):
        np.testing.assert_array_equal(getattr(a, f), getattr(b, f))
    assert not np.array_equal(a.k_cache, c.k_cache)


def test_block_table_is_a_page_permutation():
    inp = make_inputs(small_spec(batch=5, ctx=(0, 200), page_size=8), seed=1)
    P, k = 8, inp.spec.num_draft
    n = (inp.ctx_lens + k + P - 1) // P
    used = np.concatenate([inp.block_table[b, : n[b]] for b in range(5)])
    assert sorted(used.tolist()) == list(range(inp.num_pages))


def test_canaries_fill_only_unused_slots():
    inp = make_inputs(small_spec(batch=4, ctx=[3, 16, 29, 0], page_size=16), seed=2)
    P, k = 16, inp.spec.num_draft
    kf = bf16_bits_to_f32(inp.k_cache)
    for b in range(4):
        L = int(inp.ctx_lens[b]) + k
        n = (L + P - 1) // P
        for j in range(n * P):
            page, slot = inp.block_table[b, j // P], j % P
            assert np.isnan(kf[page, :, slot]).all() == (j >= L)


def test_int8_quantisation_round_trip():
    rng = np.random.default_rng(0)
    x = f32_to_bf16_bits(rng.standard_normal((64, 4, 128)).astype(np.float32))
    c, s = quantize_int8_rows(x)
    xf = bf16_bits_to_f32(x)
    sf = s.view(np.float16).astype(np.float32)
    amax = np.abs(xf).max(-1)
    err = np.abs(xf - c.astype(np.float32) * sf[..., None])
    # |x - c s| <= s/2, plus what the fp16 rounding of s costs at |x| = max|x|
    bound = sf / 2 + 127 * np.abs(sf - amax / 127) + 1e-7
    assert (err <= bound[..., None]).all()
    assert np.abs(c).max() <= 127


@pytest.mark.parametrize("mode,p", [("mismatch", 0.7), ("uniform", 0.8)])
def test_draft_match_rate(mode, p):
    inp = make_inputs(small_spec(batch=64, num_draft=16, vocab=300, logits_dtype="f32",
                                 draft_mode=mode, match_prob=p), seed=3)
    am = np.argmax(inp.logits[:, :16], axis=-1)
    rate = (inp.draft_tokens == am).mean()
    assert abs(rate - p) < 0.05


def test_geometric_break_never_recovers():
    inp = make_inputs(small_spec(batch=64, num_draft=16, vocab=300, logits_dtype="f32",
                                 draft_mode="geometric_break", match_prob=0.85), seed=3)
    am = np.argmax(inp.logits[:, :16], axis=-1)
    m = inp.draft_tokens == am
    for b in range(64):
        first = np.argmin(m[b]) if not m[b].all() else 16
        assert m[b, :first].all() and not m[b, first:].any()


def test_named_workloads_shapes():
    s = WORKLOADS["long_step_k16_bf16"]
    assert (s.batch, s.num_q_heads, s.num_kv_heads, s.num_draft, s.page_size) == (4, 28, 4, 16, 32)
    assert WORKLOADS["int8kv_70b_layer"].kv_dtype == "i8"
    assert WORKLOADS["tiny_fp32"].q_dtype == "f32"

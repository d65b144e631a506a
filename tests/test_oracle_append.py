"""Pins for the oracle's cache append, INT8 quantiser and commit (CPU only).

The quantiser restates CXL-SpecKV's "Algorithm 2 KV-Cache Compression"
(s = max|X|/127, c = round(X/s)) per (token, kv-head) row with an fp16 scale.
Pins: the round-trip error bound |x - c s| <= s/2 + max|x| 2^-11 (the second
term covers the fp16 rounding of s), the row maximum mapping to +-127, zero
rows, round-half-to-even on planted halves, the binary16 encoder against
numpy's float16 on every representable range, and the generator's
independent numpy quantiser.  The append is pinned by reading every written
row back through the page table and by leaving every other slot untouched;
the commit by the KVMU rule (validated length += accepted drafts + 1).
"""
from __future__ import annotations

import numpy as np
import pytest

from speculative_decoding_verification_attn_gb300.workload import (
    bf16_bits_to_f32, f32_to_bf16_bits, make_inputs, quantize_int8_rows, small_spec)


def test_quantizer_bounds_and_extremes(oracle_mod):
    rng = np.random.default_rng(0)
    x = rng.standard_normal((500, 128)).astype(np.float32) * rng.uniform(0.01, 50, (500, 1)).astype(np.float32)
    codes, sb = oracle_mod.quantize_rows(x, "f32")
    s = sb.view(np.float16).astype(np.float64)
    err = np.abs(x - codes.astype(np.float64) * s[:, None])
    amax = np.abs(x).max(axis=1)
    assert np.all(err <= s[:, None] / 2 + amax[:, None] * 2.0 ** -11 + 1e-12)
    # the largest magnitude of each row lands on +-127
    idx = np.abs(x).argmax(axis=1)
    assert np.all(np.abs(codes[np.arange(500), idx]) == 127)
    assert np.all(np.abs(codes) <= 127)


def test_quantizer_zero_row_and_halves(oracle_mod):
    x = np.zeros((2, 8), np.float32)
    # row 1: max 127 -> s = 1 exactly; 0.5 and 2.5 and -1.5 are exact halves
    x[1] = [127.0, 0.5, 2.5, -1.5, 1.5, -0.5, 3.49, -127.0]
    codes, sb = oracle_mod.quantize_rows(x, "f32")
    assert np.all(codes[0] == 0) and sb[0] == 0
    assert sb[1] == np.float16(1.0).view(np.uint16)
    assert list(codes[1]) == [127, 0, 2, -2, 2, 0, 3, -127]  # ties to even


def test_f16_encoder_matches_numpy(oracle_mod):
    # scales cover subnormal, normal and overflow ranges of binary16
    vals = np.concatenate([np.float32(2.0) ** np.arange(-30, 17, 0.37).astype(np.float32),
                           np.array([6.1e-5, 6.0e-8, 65504, 65519, 65520, 1e5], np.float32)])
    x = np.zeros((len(vals), 4), np.float32)
    x[:, 0] = vals * 127.0  # amax / 127 == vals up to the fp32 division
    _, sb = oracle_mod.quantize_rows(x, "f32")
    with np.errstate(over="ignore"):
        want = (np.abs(x[:, 0]) / np.float32(127.0)).astype(np.float16).view(np.uint16)
    assert np.array_equal(sb, want)


def test_quantizer_agrees_with_generator(oracle_mod):
    rng = np.random.default_rng(1)
    bits = f32_to_bf16_bits(rng.standard_normal((300, 128)).astype(np.float32) * 3)
    c1, s1 = oracle_mod.quantize_rows(bits, "bf16")
    c2, s2 = quantize_int8_rows(bits)
    assert np.array_equal(c1, c2) and np.array_equal(s1, s2)


@pytest.mark.parametrize("cache", ["bf16", "f32", "i8"])
def test_append_writes_through_page_table(oracle_mod, cache):
    inp = make_inputs(small_spec(kv_dtype=cache, q_dtype="bf16", ctx=(0, 100), page_size=16,
                                 num_draft=5), seed=3)
    s = inp.spec
    B, n, Hkv, D = s.batch, s.num_draft, s.num_kv_heads, s.head_dim
    rng = np.random.default_rng(2)
    kn = f32_to_bf16_bits(rng.standard_normal((B, n, Hkv, D)).astype(np.float32))
    vn = f32_to_bf16_bits(rng.standard_normal((B, n, Hkv, D)).astype(np.float32))
    kc, vc, ks, vs = oracle_mod.kv_append(kn, vn, "bf16", inp.k_cache, inp.v_cache, inp.k_scale,
                                          inp.v_scale, cache, inp.block_table, inp.ctx_lens)
    touched = np.zeros(inp.k_cache.shape[:3], bool)
    for b in range(B):
        for t in range(n):
            pos = int(inp.ctx_lens[b]) + t
            page = inp.block_table[b, pos // s.page_size]
            slot = pos % s.page_size
            touched[page, :, slot] = True
            for src, dst, sc in ((kn, kc, ks), (vn, vc, vs)):
                x = bf16_bits_to_f32(src[b, t])  # [Hkv, D]
                got = dst[page, :, slot]
                if cache == "bf16":
                    assert np.array_equal(got, src[b, t])
                elif cache == "f32":
                    assert np.array_equal(got, x)
                else:
                    c, sbits = quantize_int8_rows(src[b, t])
                    assert np.array_equal(got, c) and np.array_equal(sc[page, :, slot], sbits)
    # every other slot keeps its bytes (NaN canaries included)
    assert np.array_equal(kc[~touched].view(np.uint8), inp.k_cache[~touched].view(np.uint8))
    assert np.array_equal(vc[~touched].view(np.uint8), inp.v_cache[~touched].view(np.uint8))


def test_append_rejects_rows_outside_the_table(oracle_mod):
    inp = make_inputs(small_spec(), seed=4)
    s = inp.spec
    kn = np.zeros((s.batch, 1, s.num_kv_heads, s.head_dim), np.uint16)
    ctx = inp.ctx_lens.copy()
    ctx[0] = inp.max_pages * s.page_size  # first new row past the last page
    with pytest.raises(ValueError):
        oracle_mod.kv_append(kn, kn, "bf16", inp.k_cache, inp.v_cache, None, None, "bf16",
                             inp.block_table, ctx)


def test_commit_is_the_accept_pointer_move(oracle_mod):
    ctx = np.array([10, 0, 77], np.int32)
    acc = np.array([3, 0, 8], np.int32)
    assert list(oracle_mod.commit(ctx, acc, extra=1)) == [14, 1, 86]
    assert list(oracle_mod.commit(ctx, acc, extra=0)) == [13, 0, 85]

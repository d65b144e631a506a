"""Pins for the oracle's verification attention (CPU only).

Each test checks the oracle against something other than itself: a closed
form, an invariant the definition implies, or a library routine
(``torch.nn.functional.scaled_dot_product_attention`` / ``torch.logsumexp``)
on a dense re-layout of the same data.  A plausible slip in the oracle -- a
wrong GQA head map, an off-by-one causal boundary, a log2 lse, a mis-indexed
page or scale -- fails at least one of them.
"""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

from speculative_decoding_verification_attn_gb300.workload import (
    bf16_bits_to_f32, f32_to_bf16_bits, make_inputs, small_spec)

from _util import oracle_attn, oracle_rows, stored_to_f64


def n_pages_of(inp):
    P, k = inp.spec.page_size, inp.spec.num_draft
    return (inp.ctx_lens.astype(np.int64) + k + P - 1) // P


def contiguous_layout(inp):
    """Same logical cache, physical pages laid out sequence by sequence."""
    n_pages = n_pages_of(inp)
    order = np.concatenate([inp.block_table[b, : n_pages[b]] for b in range(len(n_pages))])
    bt = np.zeros_like(inp.block_table)
    off = 0
    for b, n in enumerate(n_pages):
        bt[b, :n] = np.arange(off, off + n)
        off += n
    new = dict(inp.__dict__)
    new.update(k_cache=np.ascontiguousarray(inp.k_cache[order]),
               v_cache=np.ascontiguousarray(inp.v_cache[order]), block_table=bt)
    if inp.k_scale is not None:
        new.update(k_scale=np.ascontiguousarray(inp.k_scale[order]),
                   v_scale=np.ascontiguousarray(inp.v_scale[order]))
    return type(inp)(**new), n_pages


def dense_kv(inp, n_pages, b):
    """[Hkv, L_b, D] float64 K and V of sequence b from a contiguous layout."""
    s = inp.spec
    off = int(n_pages[:b].sum())
    L = int(inp.ctx_lens[b]) + s.num_draft
    out = []
    for cache, sc in ((inp.k_cache, inp.k_scale), (inp.v_cache, inp.v_scale)):
        pages = stored_to_f64(cache[off: off + n_pages[b]], s.kv_dtype)  # [n, Hkv, P, D]
        if sc is not None:
            pages = pages * sc[off: off + n_pages[b]].view(np.float16).astype(np.float64)[..., None]
        x = pages.transpose(1, 0, 2, 3).reshape(s.num_kv_heads, -1, s.head_dim)[:, :L]
        out.append(x)
    return out


def sdpa_reference(inp):
    """Library attention on the dense layout: (out[B,k,Hq,D], lse[B,k,Hq])."""
    s = inp.spec
    cont, n_pages = contiguous_layout(inp)
    G = s.num_q_heads // s.num_kv_heads
    q = torch.from_numpy(stored_to_f64(inp.q, s.q_dtype))  # [B,k,Hq,D]
    outs, lses = [], []
    for b in range(s.batch):
        K, V = (torch.from_numpy(np.ascontiguousarray(x)) for x in dense_kv(cont, n_pages, b))
        K = K.repeat_interleave(G, dim=0)  # [Hq, L, D]
        V = V.repeat_interleave(G, dim=0)
        L = K.shape[1]
        ctx = int(inp.ctx_lens[b])
        pos = torch.arange(L)[None, :]
        qpos = ctx + torch.arange(s.num_draft)[:, None]
        mask = pos <= qpos  # [k, L]
        qb = q[b].permute(1, 0, 2)  # [Hq, k, D]
        o = torch.nn.functional.scaled_dot_product_attention(qb, K, V, attn_mask=mask,
                                                             scale=inp.scale)
        sc = inp.scale * torch.matmul(qb, K.transpose(1, 2))
        sc = sc.masked_fill(~mask, float("-inf"))
        outs.append(o.permute(1, 0, 2).numpy())
        lses.append(torch.logsumexp(sc, dim=-1).permute(1, 0).numpy())
    return np.stack(outs), np.stack(lses)


@pytest.mark.parametrize("spec_kw", [
    dict(),
    dict(num_q_heads=4, num_kv_heads=4, num_draft=1),
    dict(num_q_heads=7, num_kv_heads=1, num_draft=3, page_size=8, head_dim=64),
    dict(kv_dtype="i8", num_q_heads=8, num_kv_heads=2),
    dict(q_dtype="f32", kv_dtype="f32", head_dim=64, ctx=[0, 5, 33]),
])
def test_matches_library_attention(oracle_mod, spec_kw):
    inp = make_inputs(small_spec(**spec_kw), seed=11)
    out, lse = oracle_attn(oracle_mod, inp)
    ref_out, ref_lse = sdpa_reference(inp)
    np.testing.assert_allclose(out, ref_out, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(lse, ref_lse, rtol=1e-12, atol=1e-12)
    assert np.isfinite(out).all(), "canary slots leaked into the output"


def test_page_permutation_invariance(oracle_mod):
    inp = make_inputs(small_spec(kv_dtype="i8"), seed=3)
    cont, _ = contiguous_layout(inp)
    a = oracle_attn(oracle_mod, inp)
    b = oracle_attn(oracle_mod, cont)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


def test_single_key_closed_form(oracle_mod):
    # ctx = 0 and k = 1: the only visible key is the draft's own.
    inp = make_inputs(small_spec(batch=2, ctx=[0, 0], num_draft=1, num_q_heads=4,
                                 num_kv_heads=2), seed=5)
    out, lse = oracle_attn(oracle_mod, inp)
    s = inp.spec
    for b in range(2):
        page = inp.block_table[b, 0]
        for h in range(4):
            g = h // 2
            k0 = stored_to_f64(inp.k_cache[page, g, 0], "bf16")
            v0 = stored_to_f64(inp.v_cache[page, g, 0], "bf16")
            q = stored_to_f64(inp.q[b, 0, h], "bf16")
            np.testing.assert_array_equal(out[b, 0, h], v0)
            assert lse[b, 0, h] == pytest.approx(inp.scale * float(q @ k0), rel=1e-13)


def test_two_key_closed_form(oracle_mod):
    # ctx = 1, k = 1: out = sigmoid(s0 - s1) v0 + sigmoid(s1 - s0) v1.
    inp = make_inputs(small_spec(batch=1, ctx=[1], num_draft=1, num_q_heads=2,
                                 num_kv_heads=1), seed=6)
    out, lse = oracle_attn(oracle_mod, inp)
    page = inp.block_table[0, 0]
    K = stored_to_f64(inp.k_cache[page, 0, :2], "bf16")
    V = stored_to_f64(inp.v_cache[page, 0, :2], "bf16")
    for h in range(2):
        q = stored_to_f64(inp.q[0, 0, h], "bf16")
        s0, s1 = inp.scale * (K @ q)
        w0 = 1.0 / (1.0 + math.exp(s1 - s0))
        np.testing.assert_allclose(out[0, 0, h], w0 * V[0] + (1 - w0) * V[1], rtol=1e-12,
                                   atol=1e-14)
        assert lse[0, 0, h] == pytest.approx(np.logaddexp(s0, s1), rel=1e-13)


def test_uniform_values(oracle_mod):
    # Every V row of kv-head g equal to u_g  =>  out = u_g whatever the scores.
    inp = make_inputs(small_spec(), seed=7)
    rng = np.random.default_rng(0)
    u = f32_to_bf16_bits(rng.standard_normal((2, 128)).astype(np.float32))
    inp.v_cache[:] = u[None, :, None, :]
    out, _ = oracle_attn(oracle_mod, inp)
    want = bf16_bits_to_f32(u).astype(np.float64)
    for h in range(8):
        np.testing.assert_allclose(out[:, :, h], np.broadcast_to(want[h // 4], out[:, :, h].shape),
                                   rtol=1e-13, atol=1e-14)


def test_zero_query_mean_and_count(oracle_mod):
    # q = 0: uniform weights over the visible keys, lse = ln(#visible keys).
    inp = make_inputs(small_spec(batch=2, ctx=[17, 40], num_draft=5, page_size=8), seed=8)
    inp.q[:] = 0
    out, lse = oracle_attn(oracle_mod, inp)
    cont, n_pages = contiguous_layout(inp)
    for b in range(2):
        _, V = dense_kv(cont, n_pages, b)
        for i in range(5):
            n = int(inp.ctx_lens[b]) + i + 1
            np.testing.assert_allclose(lse[b, i], math.log(n), rtol=1e-14)
            for h in range(8):
                np.testing.assert_allclose(out[b, i, h], V[h // 4, :n].mean(axis=0), rtol=1e-12,
                                           atol=1e-14)


def test_causal_boundary(oracle_mod):
    # Changing key/value ctx+i+1 leaves row i unchanged; changing ctx+i does not.
    inp = make_inputs(small_spec(batch=1, ctx=[21], num_draft=4, page_size=4), seed=9)
    base_out, _ = oracle_attn(oracle_mod, inp)
    P = inp.spec.page_size
    for i in range(3):
        for j, changes in ((21 + i + 1, False), (21 + i, True)):
            pert = make_inputs(inp.spec, seed=9)
            page, slot = pert.block_table[0, j // P], j % P
            pert.k_cache[page, :, slot] = f32_to_bf16_bits(np.full((2, 128), 3.0, np.float32))
            pert.v_cache[page, :, slot] = f32_to_bf16_bits(np.full((2, 128), -5.0, np.float32))
            o, _ = oracle_attn(oracle_mod, pert)
            same = np.array_equal(o[0, i], base_out[0, i])
            assert same != changes, (i, j)


def test_gqa_equals_replicated_mha(oracle_mod):
    # Hq=8 over Hkv=2 equals MHA whose kv-heads repeat each group's head 4 times.
    inp = make_inputs(small_spec(num_q_heads=8, num_kv_heads=2), seed=10)
    out, lse = oracle_attn(oracle_mod, inp)
    mha = dict(inp.__dict__)
    mha["spec"] = small_spec(num_q_heads=8, num_kv_heads=8)
    mha["k_cache"] = np.ascontiguousarray(np.repeat(inp.k_cache, 4, axis=1))
    mha["v_cache"] = np.ascontiguousarray(np.repeat(inp.v_cache, 4, axis=1))
    out2, lse2 = oracle_attn(oracle_mod, type(inp)(**mha))
    np.testing.assert_array_equal(out, out2)
    np.testing.assert_array_equal(lse, lse2)


def test_int8_dequant_identity(oracle_mod):
    # INT8 codes with per-(token, head) fp16 scales equal an f32 cache holding c*s
    # (c*s is exact in float32: 8-bit code times 11-bit significand).
    inp = make_inputs(small_spec(kv_dtype="i8"), seed=12)
    f32 = dict(inp.__dict__)
    f32["spec"] = small_spec(kv_dtype="f32")
    for name, sname in (("k_cache", "k_scale"), ("v_cache", "v_scale")):
        sc = inp.__dict__[sname].view(np.float16).astype(np.float32)
        f32[name] = (inp.__dict__[name].astype(np.float32) * sc[..., None]).astype(np.float32)
    f32["k_scale"] = f32["v_scale"] = None
    a_out, a_lse = oracle_attn(oracle_mod, inp)
    b_out, b_lse = oracle_attn(oracle_mod, type(inp)(**f32))
    # canary rows hold NaN scales in both; they are never visible
    np.testing.assert_allclose(a_out, b_out, rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(a_lse, b_lse, rtol=1e-14)
    assert np.isfinite(a_out).all()


def test_k1_is_decode_attention(oracle_mod):
    # k = 1 is ordinary decode: one query over ctx+1 keys, checked against SDPA
    # with no mask at all.
    inp = make_inputs(small_spec(num_draft=1, ctx=[5, 64, 100]), seed=13)
    out, _ = oracle_attn(oracle_mod, inp)
    cont, n_pages = contiguous_layout(inp)
    for b in range(3):
        K, V = dense_kv(cont, n_pages, b)
        for h in range(8):
            q = torch.from_numpy(stored_to_f64(inp.q[b, 0, h], "bf16"))[None, None]
            o = torch.nn.functional.scaled_dot_product_attention(
                q, torch.from_numpy(K[h // 4])[None], torch.from_numpy(V[h // 4])[None],
                scale=inp.scale)
            np.testing.assert_allclose(out[b, 0, h], o[0, 0].numpy(), rtol=1e-10, atol=1e-12)


def test_rows_api_matches_full(oracle_mod):
    inp = make_inputs(small_spec(), seed=14)
    out, lse = oracle_attn(oracle_mod, inp)
    rows = np.array([[0, 0, 0], [2, 3, 7], [1, 2, 5]], np.int32)
    o, l = oracle_rows(oracle_mod, inp, rows)
    for n, (b, i, h) in enumerate(rows):
        np.testing.assert_array_equal(o[n], out[b, i, h])
        assert l[n] == lse[b, i, h]


def test_bad_page_reference_is_an_error(oracle_mod):
    inp = make_inputs(small_spec(), seed=15)
    inp.block_table[0, 0] = inp.num_pages  # out of range
    with pytest.raises(ValueError):
        oracle_attn(oracle_mod, inp)


def test_float_decoders_match_numpy(oracle_mod):
    bits = np.arange(0, 65536, 97, dtype=np.uint32).astype(np.uint16)
    f16 = bits.view(np.float16).astype(np.float64)
    b16 = bf16_bits_to_f32(bits).astype(np.float64)
    for n, x in enumerate(bits):
        a = oracle_mod.f16_bits_to_f64(int(x))
        b = oracle_mod.bf16_bits_to_f64(int(x))
        assert (a == f16[n]) or (math.isnan(a) and math.isnan(f16[n]))
        assert (b == b16[n]) or (math.isnan(b) and math.isnan(b16[n]))

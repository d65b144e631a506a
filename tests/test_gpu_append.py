"""GPU parity of spec_kv_append / spec_commit against the float64 oracle.

The append is compared byte for byte over the whole cache (and scale)
arrays: written rows bit-exact (INT8 codes and fp16 scales included, which
both sides decide in fp32), every other slot -- NaN canaries included --
untouched.  A full step then appends INT8 draft rows and verifies over them
on the tensor-core kernel, against the oracle on its own appended cache.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from speculative_decoding_verification_attn_gb300 import binding
from speculative_decoding_verification_attn_gb300.workload import (
    f32_to_bf16_bits, make_inputs, small_spec)

from gpu_util import assert_attn_close, gpu_attn, tol_for
from _util import oracle_attn

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _lib():
    from speculative_decoding_verification_attn_gb300 import build
    build.build()
    binding.load()
    for opt in range(binding.NUM_OPTIONS):
        binding.spec_set_option(opt, 0)


def new_rows(inp, src, seed, scale_spread=False):
    s = inp.spec
    rng = np.random.default_rng(seed)
    shape = (s.batch, s.num_draft, s.num_kv_heads, s.head_dim)
    k = rng.standard_normal(shape).astype(np.float32)
    v = rng.standard_normal(shape).astype(np.float32)
    if scale_spread:
        # row magnitudes from 1e-7 (subnormal fp16 scales) to 1e3
        k *= (10.0 ** rng.uniform(-7, 3, shape[:3] + (1,))).astype(np.float32)
        v *= (10.0 ** rng.uniform(-7, 3, shape[:3] + (1,))).astype(np.float32)
    if src == "bf16":
        return f32_to_bf16_bits(k), f32_to_bf16_bits(v)
    return k, v


def dev(a, kind):
    if kind == "bf16":
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def run_append(inp, kn, vn, src):
    t = binding.inputs_to_torch(inp)
    binding.spec_kv_append(dev(kn, src), dev(vn, src), t["k_cache"], t["v_cache"],
                           t["block_table"], t["ctx_lens"], t.get("k_scale"), t.get("v_scale"))
    torch.cuda.synchronize()
    as_bytes = lambda x: x.cpu().contiguous().view(torch.uint8).numpy() if x is not None else None
    return t, as_bytes(t["k_cache"]), as_bytes(t["v_cache"]), as_bytes(t.get("k_scale")), \
        as_bytes(t.get("v_scale"))


@pytest.mark.parametrize("cache,src", [("bf16", "bf16"), ("bf16", "f32"), ("f32", "bf16"),
                                       ("i8", "bf16"), ("i8", "f32")])
@pytest.mark.parametrize("kw", [
    dict(),
    dict(ctx=[0, 15, 16, 31], batch=4, num_draft=3),   # page boundaries
    dict(head_dim=64, page_size=32, num_draft=9),
    dict(head_dim=256, num_kv_heads=1, num_q_heads=1),
])
def test_append_bit_exact(oracle_mod, cache, src, kw):
    spec = small_spec(kv_dtype=cache, q_dtype="bf16", **kw)
    inp = make_inputs(spec, seed=51)
    kn, vn = new_rows(inp, src, 52, scale_spread=cache == "i8")
    _, kc, vc, ks, vs = run_append(inp, kn, vn, src)
    ok, ov, oks, ovs = oracle_mod.kv_append(kn, vn, src, inp.k_cache, inp.v_cache, inp.k_scale,
                                            inp.v_scale, cache, inp.block_table, inp.ctx_lens)
    assert np.array_equal(kc, ok.view(np.uint8).reshape(kc.shape))
    assert np.array_equal(vc, ov.view(np.uint8).reshape(vc.shape))
    if cache == "i8":
        assert np.array_equal(ks, oks.view(np.uint8).reshape(ks.shape))
        assert np.array_equal(vs, ovs.view(np.uint8).reshape(vs.shape))
    assert binding.spec_device_error() == 0


def test_bad_page_is_skipped_and_flagged(oracle_mod):
    inp = make_inputs(small_spec(ctx=[20, 40, 60], batch=3), seed=53)
    kn, vn = new_rows(inp, "bf16", 54)
    bad = inp.block_table.copy()
    bad[1, 40 // 16] = inp.num_pages + 3   # the page of sequence 1's first new row
    good_inp = make_inputs(small_spec(ctx=[20, 40, 60], batch=3), seed=53)
    inp.block_table = bad
    _, kc, _, _, _ = run_append(inp, kn, vn, "bf16")
    assert binding.spec_device_error() == binding.SPEC_DEVERR_PAGE
    # sequences 0 and 2 were written exactly as the oracle writes them
    ok, _, _, _ = oracle_mod.kv_append(kn[[0, 2]], vn[[0, 2]], "bf16", good_inp.k_cache,
                                       good_inp.v_cache, None, None, "bf16",
                                       np.ascontiguousarray(good_inp.block_table[[0, 2]]),
                                       np.ascontiguousarray(good_inp.ctx_lens[[0, 2]]))
    kc16 = kc.view(np.uint16).reshape(ok.shape)
    for b in (0, 2):
        for t in range(inp.spec.num_draft):
            pos = int(good_inp.ctx_lens[b]) + t
            page, slot = good_inp.block_table[b, pos // 16], pos % 16
            assert np.array_equal(kc16[page, :, slot], ok[page, :, slot])


def test_commit_matches_oracle(oracle_mod):
    rng = np.random.default_rng(55)
    ctx = rng.integers(0, 5000, 300).astype(np.int32)
    acc = rng.integers(0, 9, 300).astype(np.int32)
    for extra in (0, 1):
        c = torch.from_numpy(ctx.copy()).cuda()
        binding.spec_commit(c, torch.from_numpy(acc).cuda(), extra)
        torch.cuda.synchronize()
        assert np.array_equal(c.cpu().numpy(), oracle_mod.commit(ctx, acc, extra))


@pytest.mark.parametrize("kw", [dict(num_q_heads=16, num_kv_heads=2, num_draft=8),
                                dict(num_q_heads=8, num_kv_heads=2, num_draft=4)])
def test_append_then_verify_int8(oracle_mod, kw):
    # one step of the INT8 path: the drafts' rows are quantised into the
    # cache by the GPU, then the tensor-core kernel verifies over them
    spec = small_spec(kv_dtype="i8", q_dtype="bf16", ctx=(1, 300), **kw)
    inp = make_inputs(spec, seed=56)
    kn, vn = new_rows(inp, "bf16", 57)
    t, *_ = run_append(inp, kn, vn, "bf16")
    binding.spec_set_option(binding.SPEC_OPT_ATTN_PATH, 2)
    out, lse = gpu_attn(inp, t)
    ok, ov, oks, ovs = oracle_mod.kv_append(kn, vn, "bf16", inp.k_cache, inp.v_cache, inp.k_scale,
                                            inp.v_scale, "i8", inp.block_table, inp.ctx_lens)
    inp.k_cache, inp.v_cache, inp.k_scale, inp.v_scale = ok, ov, oks, ovs
    ref_out, ref_lse = oracle_attn(oracle_mod, inp)
    assert_attn_close(out, lse, ref_out, ref_lse, tol_for(inp), "append+verify")

"""GPU parity of the 128-key-tile tcgen05 kernel (attention path 5) with the oracle.

The kernel takes bf16 queries over a bf16 or INT8 cache (fp16 scales per
key), head_dim 128 and up to 128 query rows per kv-head.  Cases span 128-key
tile edges, ragged tails, contexts of zero,
every page size it takes, one long segment, forced stream-K splits of every
size (the combine in both its forms), charged splits, tree masks, and the
shapes it must refuse.  NaN canaries fill every unused cache slot.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from speculative_decoding_verification_attn_gb300 import binding
from speculative_decoding_verification_attn_gb300.workload import (
    make_inputs, random_trees, small_spec, tree_masks)

from gpu_util import assert_attn_close, check_attn_full, gpu_attn, tol_for

pytestmark = pytest.mark.gpu

PATH = 5


@pytest.fixture(autouse=True)
def _defaults():
    from speculative_decoding_verification_attn_gb300 import build
    build.build()
    binding.load()
    for opt in range(binding.NUM_OPTIONS):
        binding.spec_set_option(opt, 0)
    yield
    for opt in range(binding.NUM_OPTIONS):
        binding.spec_set_option(opt, 0)


CASES = [
    dict(num_q_heads=28, num_kv_heads=4, num_draft=16, page_size=32),       # 112 rows
    dict(num_q_heads=4, num_kv_heads=2, num_draft=64),                      # 128 rows, G = 2
    dict(num_q_heads=13, num_kv_heads=1, num_draft=5),                      # 65 rows
    dict(num_q_heads=16, num_kv_heads=2, num_draft=12, ctx=[0, 1, 127, 128, 129], batch=5),
    dict(num_q_heads=32, num_kv_heads=4, num_draft=9, ctx=(0, 40)),         # 72 rows, one tile
    dict(num_q_heads=16, num_kv_heads=2, num_draft=16, page_size=64, ctx=(1, 700)),
    dict(num_q_heads=16, num_kv_heads=2, num_draft=16, page_size=128, ctx=(100, 900)),
    dict(num_q_heads=16, num_kv_heads=2, num_draft=16, page_size=256, ctx=(250, 1200), batch=2),
    dict(batch=1, num_q_heads=28, num_kv_heads=4, num_draft=16, ctx=[5000]),  # one long segment
    dict(num_q_heads=96, num_kv_heads=1, num_draft=1, ctx=(0, 300)),        # k = 1, G = 96
    dict(batch=200, num_q_heads=28, num_kv_heads=4, num_draft=16, ctx=(0, 100)),  # many pieces
    dict(num_q_heads=16, num_kv_heads=2, num_draft=8),                      # 64 rows
    dict(num_q_heads=12, num_kv_heads=2, num_draft=4, ctx=(0, 700)),        # 24 rows
    dict(num_q_heads=8, num_kv_heads=2, num_draft=4),                       # 16 rows
    dict(num_q_heads=4, num_kv_heads=4, num_draft=1, ctx=[0, 1, 127, 128, 129], batch=5),  # 1 row
    dict(num_q_heads=32, num_kv_heads=32, num_draft=8, batch=2, ctx=(200, 900)),  # MHA, 8 rows
]


@pytest.mark.parametrize("kw", CASES, ids=[str(i) for i in range(len(CASES))])
def test_tc128_small(oracle_mod, kw):
    inp = make_inputs(small_spec(**kw), seed=81)
    binding.spec_set_option(binding.SPEC_OPT_ATTN_PATH, PATH)
    check_attn_full(oracle_mod, inp, str(kw))


# every size of split: one CTA (no combine), fewer CTAs than segments (the
# combine by boundary), more (by segment), and CTAs left without tiles
@pytest.mark.parametrize("heads", [(28, 4, 12), (16, 2, 16), (8, 4, 40), (8, 2, 4)],
                         ids=["84rows", "128rows", "80rows_G2", "16rows"])
@pytest.mark.parametrize("ctas", [1, 2, 5, 37, 152, 400])
def test_tc128_stream_k_splits(oracle_mod, ctas, heads):
    hq, hkv, k = heads
    inp = make_inputs(small_spec(batch=4, num_q_heads=hq, num_kv_heads=hkv, num_draft=k,
                                 ctx=(0, 1800)), seed=82)
    binding.spec_set_option(binding.SPEC_OPT_ATTN_PATH, PATH)
    binding.spec_set_option(binding.SPEC_OPT_NUM_CTAS, ctas)
    check_attn_full(oracle_mod, inp, "ctas=%d heads=%s" % (ctas, heads))


@pytest.mark.parametrize("weight", [1, 2, 5, 65])
@pytest.mark.parametrize("ctas", [5, 37, 152])
def test_tc128_split_weights(oracle_mod, weight, ctas):
    inp = make_inputs(small_spec(batch=6, num_q_heads=28, num_kv_heads=4, num_draft=12,
                                 ctx=(0, 3000)), seed=83)
    binding.spec_set_option(binding.SPEC_OPT_ATTN_PATH, PATH)
    binding.spec_set_option(binding.SPEC_OPT_NUM_CTAS, ctas)
    binding.spec_set_option(binding.SPEC_OPT_SPLIT_WEIGHT, weight)
    check_attn_full(oracle_mod, inp, "weight %d ctas %d" % (weight, ctas))


def test_tc128_long_step_shape_sampled(oracle_mod):
    # the long-context shape (28 q-heads over 4 kv-heads, 16 drafts, pages of
    # 32) at a shorter context, every output against the oracle
    inp = make_inputs(small_spec(batch=4, num_q_heads=28, num_kv_heads=4, num_draft=16,
                                 page_size=32, ctx=(3000, 6000)), seed=84)
    binding.spec_set_option(binding.SPEC_OPT_ATTN_PATH, PATH)
    check_attn_full(oracle_mod, inp, "long-step shape")


@pytest.mark.parametrize("width", [0.0, 0.5, 1.0])
@pytest.mark.parametrize("kw", [
    dict(num_q_heads=28, num_kv_heads=4, num_draft=16, page_size=32),
    dict(num_q_heads=2, num_kv_heads=1, num_draft=64, ctx=(0, 300)),       # 64-bit masks
    dict(num_q_heads=8, num_kv_heads=2, num_draft=4),                       # 16 rows
], ids=["112rows", "k64", "16rows"])
def test_tc128_tree_masks(oracle_mod, kw, width):
    spec = small_spec(**kw)
    inp = make_inputs(spec, seed=85)
    masks = tree_masks(random_trees(spec.batch, spec.num_draft, seed=86, width=width))
    binding.spec_set_option(binding.SPEC_OPT_ATTN_PATH, PATH)
    t = binding.inputs_to_torch(inp)
    o = binding.alloc_outputs(inp)
    o["out"].fill_(float("nan"))
    o["lse"].fill_(float("nan"))
    tm = torch.from_numpy(masks.view(np.int64)).cuda()
    binding.spec_verify_attn_tree(t["q"], t["k_cache"], t["v_cache"], t["block_table"],
                                  t["ctx_lens"], tm, spec.num_draft, inp.scale, o["out"],
                                  o["lse"])
    torch.cuda.synchronize()
    ref_out, ref_lse = oracle_mod.verify_attn_tree(
        inp.q, spec.q_dtype, inp.k_cache, inp.v_cache, spec.kv_dtype, inp.k_scale, inp.v_scale,
        inp.block_table, inp.ctx_lens, inp.scale, masks)
    assert_attn_close(o["out"].double().cpu().numpy(), o["lse"].double().cpu().numpy(), ref_out,
                      ref_lse, tol_for(inp), "tree %s width %s" % (kw, width))
    assert binding.spec_device_error() == 0


def test_tc128_close_to_tc64():
    # the two tcgen05 kernels differ only in tiling and rounding order
    inp = make_inputs(small_spec(batch=6, num_q_heads=28, num_kv_heads=4, num_draft=16,
                                 page_size=32, ctx=(0, 2500)), seed=87)
    t = binding.inputs_to_torch(inp)
    binding.spec_set_option(binding.SPEC_OPT_ATTN_PATH, PATH)
    a_out, a_lse = gpu_attn(inp, t)
    binding.spec_set_option(binding.SPEC_OPT_ATTN_PATH, 2)
    b_out, b_lse = gpu_attn(inp, t)
    assert np.isfinite(a_out).all() and np.isfinite(a_lse).all()
    assert np.abs(a_out - b_out).max() < 2e-2
    assert np.abs(a_lse - b_lse).max() < 1e-3


@pytest.mark.parametrize("kw", [
    dict(num_q_heads=32, num_kv_heads=2, num_draft=9),                     # 144 rows
    dict(num_q_heads=28, num_kv_heads=4, num_draft=16, head_dim=64),       # head_dim 64
    dict(num_q_heads=28, num_kv_heads=4, num_draft=16, q_dtype="f32", kv_dtype="f32"),
    dict(num_q_heads=28, num_kv_heads=4, num_draft=16, page_size=8),       # pages of 8
], ids=["144rows", "d64", "f32", "page8"])
def test_tc128_refuses_other_shapes(kw):
    inp = make_inputs(small_spec(**kw), seed=88)
    t = binding.inputs_to_torch(inp)
    o = binding.alloc_outputs(inp)
    binding.spec_set_option(binding.SPEC_OPT_ATTN_PATH, PATH)
    with pytest.raises(RuntimeError):
        binding.spec_verify_attn(t["q"], t["k_cache"], t["v_cache"], t["block_table"],
                                 t["ctx_lens"], inp.spec.num_draft, inp.scale, o["out"], o["lse"],
                                 t.get("k_scale"), t.get("v_scale"))


I8_CASES = [
    dict(num_q_heads=64, num_kv_heads=8, num_draft=8),                      # 64 rows
    dict(num_q_heads=28, num_kv_heads=4, num_draft=16, page_size=32),       # 112 rows
    dict(num_q_heads=8, num_kv_heads=2, num_draft=4),                       # 16 rows
    dict(num_q_heads=4, num_kv_heads=2, num_draft=64),                      # 128 rows
    dict(num_q_heads=16, num_kv_heads=2, num_draft=8, ctx=[0, 1, 127, 128, 129], batch=5),
    dict(num_q_heads=16, num_kv_heads=2, num_draft=8, page_size=64, ctx=(1, 700)),
    dict(num_q_heads=16, num_kv_heads=2, num_draft=8, page_size=256, ctx=(250, 1200), batch=2),
    dict(batch=1, num_q_heads=64, num_kv_heads=8, num_draft=8, ctx=[5000]),  # one long segment
    dict(batch=200, num_q_heads=28, num_kv_heads=4, num_draft=16, ctx=(0, 100)),  # many pieces
]


@pytest.mark.parametrize("kw", I8_CASES, ids=[str(i) for i in range(len(I8_CASES))])
def test_tc128_int8(oracle_mod, kw):
    inp = make_inputs(small_spec(kv_dtype="i8", **kw), seed=89)
    binding.spec_set_option(binding.SPEC_OPT_ATTN_PATH, PATH)
    check_attn_full(oracle_mod, inp, "i8 %s" % kw)


@pytest.mark.parametrize("ctas", [1, 2, 5, 37, 152, 400])
def test_tc128_int8_stream_k_splits(oracle_mod, ctas):
    inp = make_inputs(small_spec(batch=4, num_q_heads=64, num_kv_heads=8, num_draft=8,
                                 kv_dtype="i8", ctx=(0, 1800)), seed=90)
    binding.spec_set_option(binding.SPEC_OPT_ATTN_PATH, PATH)
    binding.spec_set_option(binding.SPEC_OPT_NUM_CTAS, ctas)
    check_attn_full(oracle_mod, inp, "i8 ctas=%d" % ctas)


def test_tc128_int8_close_to_tc64():
    # dequantization to fp16 before the MMAs (128-key kernel) against the
    # scales kept in fp32 (64-key kernel)
    inp = make_inputs(small_spec(batch=6, num_q_heads=64, num_kv_heads=8, num_draft=8,
                                 kv_dtype="i8", ctx=(0, 2500)), seed=91)
    t = binding.inputs_to_torch(inp)
    binding.spec_set_option(binding.SPEC_OPT_ATTN_PATH, PATH)
    a_out, a_lse = gpu_attn(inp, t)
    binding.spec_set_option(binding.SPEC_OPT_ATTN_PATH, 2)
    b_out, b_lse = gpu_attn(inp, t)
    assert np.isfinite(a_out).all() and np.isfinite(a_lse).all()
    assert np.abs(a_out - b_out).max() < 2e-2
    assert np.abs(a_lse - b_lse).max() < 1e-3


@pytest.mark.parametrize("width", [0.0, 0.5, 1.0])
def test_tc128_int8_tree_masks(oracle_mod, width):
    spec = small_spec(num_q_heads=28, num_kv_heads=4, num_draft=16, kv_dtype="i8")
    inp = make_inputs(spec, seed=92)
    masks = tree_masks(random_trees(spec.batch, spec.num_draft, seed=93, width=width))
    binding.spec_set_option(binding.SPEC_OPT_ATTN_PATH, PATH)
    t = binding.inputs_to_torch(inp)
    o = binding.alloc_outputs(inp)
    o["out"].fill_(float("nan"))
    o["lse"].fill_(float("nan"))
    tm = torch.from_numpy(masks.view(np.int64)).cuda()
    binding.spec_verify_attn_tree(t["q"], t["k_cache"], t["v_cache"], t["block_table"],
                                  t["ctx_lens"], tm, spec.num_draft, inp.scale, o["out"],
                                  o["lse"], t["k_scale"], t["v_scale"])
    torch.cuda.synchronize()
    ref_out, ref_lse = oracle_mod.verify_attn_tree(
        inp.q, spec.q_dtype, inp.k_cache, inp.v_cache, spec.kv_dtype, inp.k_scale, inp.v_scale,
        inp.block_table, inp.ctx_lens, inp.scale, masks)
    assert_attn_close(o["out"].double().cpu().numpy(), o["lse"].double().cpu().numpy(), ref_out,
                      ref_lse, tol_for(inp), "i8 tree width %s" % width)
    assert binding.spec_device_error() == 0


# more (sequence, kv-head) segments than CTAs, ragged lengths and one long
# sequence among short ones (a segment over many CTAs): the combine in its
# by-boundary form; two calls in a row give the same bits
@pytest.mark.parametrize("ctx", [(0, 4000), [9000] + [50] * 47], ids=["ragged", "one_long"])
@pytest.mark.parametrize("ctas", [37, 100, 152])
def test_tc128_many_segments(oracle_mod, ctx, ctas):
    inp = make_inputs(small_spec(batch=48, num_q_heads=28, num_kv_heads=4, num_draft=12,
                                 ctx=ctx), seed=94)
    binding.spec_set_option(binding.SPEC_OPT_ATTN_PATH, PATH)
    binding.spec_set_option(binding.SPEC_OPT_NUM_CTAS, ctas)
    t = binding.inputs_to_torch(inp)
    first, _ = gpu_attn(inp, t)
    check_attn_full(oracle_mod, inp, "many segments ctas=%d" % ctas)
    again, _ = gpu_attn(inp, t)
    assert np.array_equal(first, again)

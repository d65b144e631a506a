"""GPU parity of tree verification (attention and acceptance) with the oracle.

Every attention kernel is forced in turn over seeded random draft trees
(chains, bushy trees, stars) and compared with the float64 oracle at the
usual tolerances; a chain mask through spec_verify_attn_tree must reproduce
spec_verify_attn bit for bit.  Tree acceptance (both kernel forms) is
compared exactly, accepted paths included, and a chain must reproduce
greedy acceptance.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from speculative_decoding_verification_attn_gb300 import binding
from speculative_decoding_verification_attn_gb300.workload import (
    bf16_bits_to_f32, make_inputs, plant_tree_tokens, random_trees, small_spec, tree_masks)

from gpu_util import assert_attn_close, gpu_attn, tol_for

pytestmark = pytest.mark.gpu


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


def tree_oracle(oracle_mod, inp, masks):
    s = inp.spec
    return oracle_mod.verify_attn_tree(inp.q, s.q_dtype, inp.k_cache, inp.v_cache, s.kv_dtype,
                                       inp.k_scale, inp.v_scale, inp.block_table, inp.ctx_lens,
                                       inp.scale, masks)


def gpu_tree_attn(inp, masks, t=None):
    t = t or binding.inputs_to_torch(inp)
    o = binding.alloc_outputs(inp)
    o["out"].fill_(float("nan"))
    o["lse"].fill_(float("nan"))
    tm = torch.from_numpy(masks.view(np.int64)).cuda()
    binding.spec_verify_attn_tree(t["q"], t["k_cache"], t["v_cache"], t["block_table"],
                                  t["ctx_lens"], tm, inp.spec.num_draft, inp.scale, o["out"],
                                  o["lse"], t.get("k_scale"), t.get("v_scale"))
    torch.cuda.synchronize()
    return o["out"].double().cpu().numpy(), o["lse"].double().cpu().numpy()


CASES = [  # (attention path, spec)
    (3, dict(num_q_heads=8, num_kv_heads=2, num_draft=4)),                      # 16 rows: warp MMA
    (3, dict(num_q_heads=4, num_kv_heads=4, num_draft=16, ctx=(0, 200))),      # 16 rows, k = 16
    (2, dict(num_q_heads=28, num_kv_heads=4, num_draft=16, page_size=32)),     # 112 rows: tcgen05
    (2, dict(num_q_heads=16, num_kv_heads=2, num_draft=8, ctx=[0, 60, 130])), # 64 rows
    (2, dict(num_q_heads=2, num_kv_heads=2, num_draft=64, ctx=(0, 100))),     # k = 64, 64-bit masks
    (2, dict(num_q_heads=16, num_kv_heads=2, num_draft=8, kv_dtype="i8")),    # INT8 tcgen05
    (1, dict(num_q_heads=8, num_kv_heads=2, num_draft=6)),                     # SIMT
    (1, dict(q_dtype="f32", kv_dtype="f32", head_dim=64, num_draft=5)),        # SIMT fp32
    (4, dict(q_dtype="f32", kv_dtype="f32", head_dim=64, num_draft=5)),        # single pass
    (4, dict(num_q_heads=2, num_kv_heads=2, num_draft=64, ctx=(0, 40))),      # single pass, k = 64
    (5, dict(num_q_heads=28, num_kv_heads=4, num_draft=16, page_size=32)),     # 128-key tiles
    (5, dict(num_q_heads=8, num_kv_heads=2, num_draft=4)),                     # 128-key, 16 rows
]


@pytest.mark.parametrize("width", [0.0, 0.5, 1.0])
@pytest.mark.parametrize("path,kw", CASES, ids=[str(i) for i in range(len(CASES))])
def test_tree_attention_matches_oracle(oracle_mod, path, kw, width):
    spec = small_spec(**kw)
    inp = make_inputs(spec, seed=71)
    masks = tree_masks(random_trees(spec.batch, spec.num_draft, seed=72, width=width))
    binding.spec_set_option(binding.SPEC_OPT_ATTN_PATH, path)
    out, lse = gpu_tree_attn(inp, masks)
    ref_out, ref_lse = tree_oracle(oracle_mod, inp, masks)
    assert_attn_close(out, lse, ref_out, ref_lse, tol_for(inp), "tree path %d %s" % (path, kw))
    assert binding.spec_device_error() == 0


@pytest.mark.parametrize("path", [0, 1, 2, 3, 4, 5])
def test_chain_mask_reproduces_causal(path):
    # (the single-pass kernel holds whole sequences: shorter contexts there)
    ctx = (0, 100) if path == 4 else (0, 300)
    inp = make_inputs(small_spec(num_q_heads=8, num_kv_heads=2, num_draft=4, ctx=ctx), seed=73)
    chain = np.tile(np.arange(-1, 3, dtype=np.int32), (inp.spec.batch, 1))
    binding.spec_set_option(binding.SPEC_OPT_ATTN_PATH, path)
    t = binding.inputs_to_torch(inp)
    a_out, a_lse = gpu_attn(inp, t)
    b_out, b_lse = gpu_tree_attn(inp, tree_masks(chain), t)
    assert np.array_equal(a_out, b_out) and np.array_equal(a_lse, b_lse)


def tree_accept_inputs(B, k, V, seed, width, match):
    inp = make_inputs(small_spec(batch=B, num_draft=k, vocab=V), seed=seed)
    logits_f = bf16_bits_to_f32(inp.logits) if inp.spec.logits_dtype == "bf16" else inp.logits
    parents = random_trees(B, k, seed=seed + 1, width=width)
    tokens = plant_tree_tokens(logits_f, parents, match, seed=seed + 2)
    return inp, parents, tokens


@pytest.mark.parametrize("B,k,V,width,match", [
    (8, 6, 1000, 0.5, 0.8),       # cluster form
    (40, 20, 3000, 0.6, 0.85),    # k + 1 > 16: ticket form
    (300, 4, 32000, 1.0, 0.9),    # more sequences than SMs: ticket form
    (3, 64, 500, 0.4, 0.9),       # 64 nodes
])
def test_tree_acceptance_matches_oracle(oracle_mod, B, k, V, width, match):
    inp, parents, tokens = tree_accept_inputs(B, k, V, 74, width, match)
    t = binding.inputs_to_torch(inp)
    acc = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    nxt = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    path = torch.full((B, k), -7, dtype=torch.int32, device="cuda")
    binding.spec_accept_tree(t["logits"], torch.from_numpy(tokens).cuda(),
                             torch.from_numpy(parents).cuda(), k, acc, nxt, path)
    torch.cuda.synchronize()
    o_acc, o_nxt, o_path = oracle_mod.accept_tree(inp.logits, inp.spec.logits_dtype, tokens, parents)
    assert np.array_equal(acc.cpu().numpy(), o_acc)
    assert np.array_equal(nxt.cpu().numpy(), o_nxt)
    assert np.array_equal(path.cpu().numpy(), o_path)
    assert o_acc.max() >= 2  # the planted matches make some paths long
    assert binding.spec_device_error() == 0


def test_chain_tree_acceptance_equals_greedy():
    inp = make_inputs(small_spec(batch=50, num_draft=8, vocab=2000), seed=75)
    t = binding.inputs_to_torch(inp)
    chain = torch.from_numpy(np.tile(np.arange(-1, 7, dtype=np.int32), (50, 1))).cuda()
    o = [torch.empty(50, dtype=torch.int32, device="cuda") for _ in range(4)]
    binding.spec_accept_tree(t["logits"], t["draft_tokens"], chain, 8, o[0], o[1])
    binding.spec_accept_greedy(t["logits"], t["draft_tokens"], 8, o[2], o[3])
    torch.cuda.synchronize()
    assert torch.equal(o[0], o[2]) and torch.equal(o[1], o[3])


def test_bad_parent_is_flagged():
    inp, parents, tokens = tree_accept_inputs(4, 5, 1000, 76, 0.5, 0.9)
    parents[2, 3] = 3  # a node claiming itself as parent
    t = binding.inputs_to_torch(inp)
    acc = torch.empty(4, dtype=torch.int32, device="cuda")
    nxt = torch.empty(4, dtype=torch.int32, device="cuda")
    binding.spec_accept_tree(t["logits"], torch.from_numpy(tokens).cuda(),
                             torch.from_numpy(parents).cuda(), 5, acc, nxt)
    torch.cuda.synchronize()
    assert binding.spec_device_error() == binding.SPEC_DEVERR_TREE
    assert int(acc[2]) <= 3

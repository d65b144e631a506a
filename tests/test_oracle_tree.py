"""Pins for the oracle's tree verification (CPU only).

Token trees ("Decoding Speculative Decoding from First Principles", section
"Advances in speculators": SpecInfer / EAGLE-style trees verified in one
pass): draft node i attends to the context, its ancestors and itself, and
the accepted path follows the target's argmax from the root.  Pins: a chain
tree reproduces the causal oracle exactly; any tree against the library's
scaled_dot_product_attention with the ancestor mask on a dense layout;
relabelling the nodes (a topological renumbering of the tree, applied to
queries, K/V rows, masks and logits) permutes the outputs; tree acceptance
of a chain equals greedy acceptance; on random trees the accepted path is a
root path of matching nodes, each the lowest-index matching child of its
parent, ending where no child matches.  Each pin was checked to catch a
planted slip in the oracle (a query not seeing its own draft key, choosing
the highest-index matching child, stopping one node early).
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from speculative_decoding_verification_attn_gb300.workload import (
    bf16_bits_to_f32, make_inputs, plant_tree_tokens, random_trees, small_spec, tree_masks)

from _util import oracle_attn, stored_to_f64
from test_oracle_attn import contiguous_layout, dense_kv


def tree_oracle(oracle_mod, inp, masks):
    s = inp.spec
    return oracle_mod.verify_attn_tree(inp.q, s.q_dtype, inp.k_cache, inp.v_cache, s.kv_dtype,
                                       inp.k_scale, inp.v_scale, inp.block_table, inp.ctx_lens,
                                       inp.scale, masks)


def chain(B, k):
    return np.tile(np.arange(-1, k - 1, dtype=np.int32), (B, 1))


def test_chain_tree_is_causal(oracle_mod):
    inp = make_inputs(small_spec(num_draft=6, ctx=(0, 120)), seed=61)
    s = inp.spec
    out, lse = tree_oracle(oracle_mod, inp, tree_masks(chain(s.batch, s.num_draft)))
    ref_out, ref_lse = oracle_attn(oracle_mod, inp)
    assert np.array_equal(out, ref_out) and np.array_equal(lse, ref_lse)


@pytest.mark.parametrize("width", [0.0, 0.5, 1.0])
def test_tree_matches_library_attention(oracle_mod, width):
    inp = make_inputs(small_spec(num_draft=7, ctx=(0, 90), num_q_heads=4, num_kv_heads=2),
                      seed=62)
    s = inp.spec
    parents = random_trees(s.batch, s.num_draft, seed=3, width=width)
    masks = tree_masks(parents)
    out, lse = tree_oracle(oracle_mod, inp, masks)
    cont, n_pages = contiguous_layout(inp)
    G = s.num_q_heads // s.num_kv_heads
    q = torch.from_numpy(stored_to_f64(inp.q, s.q_dtype))
    for b in range(s.batch):
        K, V = (torch.from_numpy(np.ascontiguousarray(x)).repeat_interleave(G, dim=0)
                for x in dense_kv(cont, n_pages, b))
        ctx, L = int(inp.ctx_lens[b]), K.shape[1]
        vis = np.zeros((s.num_draft, L), bool)
        vis[:, :ctx] = True
        for i in range(s.num_draft):
            for t in range(s.num_draft):
                vis[i, ctx + t] = bool((int(masks[b, i]) >> t) & 1)
        mask = torch.from_numpy(vis)
        qb = q[b].permute(1, 0, 2)
        o = torch.nn.functional.scaled_dot_product_attention(qb, K, V, attn_mask=mask,
                                                             scale=inp.scale)
        sc = (inp.scale * torch.matmul(qb, K.transpose(1, 2))).masked_fill(~mask, float("-inf"))
        assert np.allclose(out[b], o.permute(1, 0, 2).numpy(), atol=1e-12, rtol=1e-12)
        assert np.allclose(lse[b], torch.logsumexp(sc, -1).permute(1, 0).numpy(), atol=1e-12)


def test_node_relabelling_permutes_outputs(oracle_mod):
    # a tree 0 -> {1, 2}, 1 -> 3 numbered in a second topological order
    inp = make_inputs(small_spec(num_draft=4, batch=2, ctx=[30, 47], page_size=16), seed=63)
    s = inp.spec
    parents = np.array([[-1, 0, 0, 1]] * 2, np.int32)
    perm = np.array([0, 2, 1, 3])          # new label -> old node
    inv = np.argsort(perm)
    new_parents = np.array([[-1 if parents[0, o] < 0 else inv[parents[0, o]] for o in perm]] * 2,
                           np.int32)
    out, lse = tree_oracle(oracle_mod, inp, tree_masks(parents))
    # move the draft rows: queries and the K/V slots of positions ctx + t
    inp2 = make_inputs(small_spec(num_draft=4, batch=2, ctx=[30, 47], page_size=16), seed=63)
    inp2.q = np.ascontiguousarray(inp.q[:, perm])
    P = s.page_size
    for b in range(s.batch):
        ctx = int(inp.ctx_lens[b])
        for new, old in enumerate(perm):
            pn, po = ctx + new, ctx + old
            for c_new, c_old in ((inp2.k_cache, inp.k_cache), (inp2.v_cache, inp.v_cache)):
                c_new[inp.block_table[b, pn // P], :, pn % P] = \
                    c_old[inp.block_table[b, po // P], :, po % P]
    out2, lse2 = tree_oracle(oracle_mod, inp2, tree_masks(new_parents))
    assert np.allclose(out2, out[:, perm], atol=1e-12) and np.allclose(lse2, lse[:, perm], atol=1e-12)


def test_chain_acceptance_is_greedy(oracle_mod):
    inp = make_inputs(small_spec(num_draft=6, batch=40, vocab=50), seed=64)
    parents = chain(40, 6)
    acc, nxt, path = oracle_mod.accept_tree(inp.logits, inp.spec.logits_dtype, inp.draft_tokens,
                                            parents)
    g_acc, g_nxt, _ = oracle_mod.accept_greedy(inp.logits, inp.spec.logits_dtype, inp.draft_tokens)
    assert np.array_equal(acc, g_acc) and np.array_equal(nxt, g_nxt)
    for b in range(40):
        assert list(path[b, :acc[b]]) == list(range(acc[b]))
        assert np.all(path[b, acc[b]:] == -1)


@pytest.mark.parametrize("width,match", [(0.5, 0.7), (1.0, 0.9), (0.3, 0.95)])
def test_tree_acceptance_properties(oracle_mod, width, match):
    rng = np.random.default_rng(65)
    B, k, V = 60, 10, 12
    logits = rng.standard_normal((B, k + 1, V)).astype(np.float32)
    parents = random_trees(B, k, seed=5, width=width)
    draft = plant_tree_tokens(logits, parents, match, seed=6)
    acc, nxt, path = oracle_mod.accept_tree(logits, "f32", draft, parents)
    am = np.argmax(logits.astype(np.float64), axis=-1)
    for b in range(B):
        def matching_children(p):
            return [c for c in range(k) if parents[b, c] == p and draft[b, c] == am[b, p + 1]]
        cur = -1
        for step in range(acc[b]):
            c = path[b, step]
            assert parents[b, c] == cur and c == min(matching_children(cur))
            cur = c
        assert matching_children(cur) == []
        assert nxt[b] == am[b, cur + 1]
        assert np.all(path[b, acc[b]:] == -1)


def test_bad_parent_is_an_error(oracle_mod):
    logits = np.zeros((1, 4, 5), np.float32)
    with pytest.raises(ValueError):
        oracle_mod.accept_tree(logits, "f32", np.zeros((1, 3), np.int32),
                               np.array([[-1, 1, 0]], np.int32))

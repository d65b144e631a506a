"""GPU parity of spec_accept_greedy against the oracle: bit-exact
accepted_len and next_token on every named workload and on edge cases
(vocabulary sizes that are not multiples of the 16-byte vector, slice
boundaries, planted ties, all / none accepted)."""
from __future__ import annotations

import dataclasses

import numpy as np
import pytest
import torch

from speculative_decoding_verification_attn_gb300 import binding
from speculative_decoding_verification_attn_gb300.workload import (
    WORKLOAD_ORDER, WORKLOADS, f32_to_bf16_bits, make_inputs, small_spec)

from gpu_util import check_accept, gpu_accept
from _util import oracle_accept

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from speculative_decoding_verification_attn_gb300 import build
    build.build()
    binding.load()


@pytest.mark.parametrize("name", WORKLOAD_ORDER)
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_named_workloads(oracle_mod, name, seed):
    # logits and drafts come from their own random streams; a full-size cache
    # is not needed for acceptance, so shrink the context to keep this quick
    small_ctx = dataclasses.replace(WORKLOADS[name], ctx=16)
    inp = make_inputs(small_ctx, seed=seed)
    check_accept(oracle_mod, inp)


@pytest.mark.parametrize("vocab", [1, 7, 8, 9, 1001, 8191, 8192, 8193, 40000])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("k", [1, 3, 64])
def test_vocab_and_draft_edges(oracle_mod, vocab, dtype, k):
    inp = make_inputs(small_spec(batch=5, num_draft=k, vocab=vocab, ctx=8, logits_dtype=dtype,
                                 match_prob=0.9, num_q_heads=2, num_kv_heads=1, head_dim=32),
                      seed=vocab + k)
    check_accept(oracle_mod, inp)


def test_planted_ties_across_slices(oracle_mod):
    inp = make_inputs(small_spec(batch=3, num_draft=2, vocab=20000, ctx=8, logits_dtype="f32",
                                 num_q_heads=2, num_kv_heads=1, head_dim=32), seed=4)
    lg = inp.logits
    lg[0, 0, [8191, 8192]] = 50.0         # tie across the slice boundary
    lg[0, 1, [19999, 100]] = 60.0         # tie between first and last slice
    lg[1, :, :] = 0.0                     # whole row tied: index 0 wins
    lg[1, :, 3] = -0.0
    lg[2, 2, [16383, 16384, 5]] = 9.0
    inp.draft_tokens[0] = [8191, 100]
    inp.draft_tokens[1] = [0, 1]
    check_accept(oracle_mod, inp)
    acc, nxt = gpu_accept(inp)
    assert acc[0] == 2 and nxt[0] == int(np.argmax(lg[0, 2]))
    assert acc[1] == 1 and nxt[1] == 0
    bf = dict(inp.__dict__)
    bf["logits"] = f32_to_bf16_bits(lg)
    bf["spec"] = small_spec(batch=3, num_draft=2, vocab=20000, ctx=8, logits_dtype="bf16",
                            num_q_heads=2, num_kv_heads=1, head_dim=32)
    check_accept(oracle_mod, type(inp)(**bf))


def test_all_and_none_accepted(oracle_mod):
    inp = make_inputs(small_spec(batch=4, num_draft=6, vocab=3000, ctx=8, logits_dtype="bf16",
                                 num_q_heads=2, num_kv_heads=1, head_dim=32), seed=5)
    _, _, am = oracle_accept(oracle_mod, inp)
    inp.draft_tokens[0] = am[0, :6]
    inp.draft_tokens[1] = (am[1, :6] + 1) % 3000
    inp.draft_tokens[2, :] = am[2, :6]
    inp.draft_tokens[2, 5] = (am[2, 5] + 1) % 3000
    acc, nxt = gpu_accept(inp)
    assert acc.tolist()[:3] == [6, 0, 5]
    assert nxt[0] == am[0, 6]  # bonus token
    check_accept(oracle_mod, inp)


def test_repeated_calls_are_stable(oracle_mod):
    inp = make_inputs(small_spec(batch=7, num_draft=4, vocab=70000, ctx=8,
                                 num_q_heads=2, num_kv_heads=1, head_dim=32), seed=6)
    t = binding.inputs_to_torch(inp)
    for _ in range(3):
        check_accept(oracle_mod, inp, t)


def test_misaligned_logits_rejected():
    lg = torch.zeros(2 * 5 * 100 + 1, dtype=torch.bfloat16, device="cuda")[1:].view(2, 5, 100)
    dr = torch.zeros(2, 4, dtype=torch.int32, device="cuda")
    acc = torch.zeros(2, dtype=torch.int32, device="cuda")
    with pytest.raises(binding.SpecError):
        binding.spec_accept_greedy(lg, dr, 4, acc, acc.clone())

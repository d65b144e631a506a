"""The allocation-free acceptance entry point (spec_accept_greedy_noalloc).

It exists for callers that cannot allocate device memory, such as a serving
loop whose GPU memory is reserved up front by its own allocator, or a host
that loads the library as a plugin without the right to allocate.  Its
scratch is a fixed array inside the library, shared by every call, so these
tests call it twice in a row (and on a second, different batch) and check
each result against the allocating entry point, spec_accept_greedy, and
against the float64 oracle, bit for bit.  This file is collected last so that
a run stopping at its first failure has already run every other test; it
also passes on its own in a fresh process.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from speculative_decoding_verification_attn_gb300 import binding
from speculative_decoding_verification_attn_gb300.workload import make_inputs, small_spec

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from speculative_decoding_verification_attn_gb300 import build
    build.build()
    binding.load()


def _spec(batch, num_draft, vocab, dtype):
    return small_spec(batch=batch, num_draft=num_draft, vocab=vocab, ctx=8, logits_dtype=dtype,
                      num_q_heads=2, num_kv_heads=1, head_dim=32, match_prob=0.8)


def _run(fn, t, k):
    B = t["logits"].shape[0]
    acc = torch.full((B,), -5, dtype=torch.int32, device="cuda")
    nxt = torch.full((B,), -5, dtype=torch.int32, device="cuda")
    fn(t["logits"], t["draft_tokens"], k, acc, nxt)
    torch.cuda.synchronize()
    return acc.cpu().numpy(), nxt.cpu().numpy()


@pytest.mark.parametrize("batch,num_draft,vocab,dtype", [
    (16, 6, 40000, "bf16"),
    (3, 1, 1001, "f32"),
    (64, 8, 128256, "bf16"),
])
def test_noalloc_matches_allocating_entry_point(oracle_mod, batch, num_draft, vocab, dtype):
    first = make_inputs(_spec(batch, num_draft, vocab, dtype), seed=batch + vocab)
    second = make_inputs(_spec(batch, num_draft, vocab, dtype), seed=batch + vocab + 1)
    for inp in (first, second):
        t = binding.inputs_to_torch(inp)
        want = _run(binding.spec_accept_greedy, t, num_draft)
        o_acc, o_nxt, _ = oracle_mod.accept_greedy(inp.logits, dtype, inp.draft_tokens)
        np.testing.assert_array_equal(want[0], o_acc)
        np.testing.assert_array_equal(want[1], o_nxt)
        for _ in range(2):  # two calls in a row share the fixed scratch
            got = _run(binding.spec_accept_greedy_noalloc, t, num_draft)
            np.testing.assert_array_equal(got[0], want[0])
            np.testing.assert_array_equal(got[1], want[1])
            np.testing.assert_array_equal(got[0], o_acc)
            np.testing.assert_array_equal(got[1], o_nxt)


def test_noalloc_rejects_sizes_beyond_its_scratch():
    B, k, V = 64, 64, 152064  # 64 * 65 * 19 partials > SPEC_NOALLOC_MAX_PARTIALS
    logits = torch.zeros((B, k + 1, V), dtype=torch.bfloat16, device="cuda")
    drafts = torch.zeros((B, k), dtype=torch.int32, device="cuda")
    acc = torch.zeros((B,), dtype=torch.int32, device="cuda")
    with pytest.raises(binding.SpecError, match="no-allocation scratch"):
        binding.spec_accept_greedy_noalloc(logits, drafts, k, acc, acc.clone())

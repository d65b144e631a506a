"""Pins for the oracle's greedy acceptance (CPU only).

The blog "Decoding Speculative Decoding from First Principles" (section
"Speculating to get sequence parallelism during decode") fixes the rule: the
target keeps drafts up to the first disagreement, emits its own token there,
and emits a bonus token when every draft agrees, so one pass yields between 1
and k+1 tokens.  The tests check the oracle against that statement written
as a set property (longest agreeing prefix = the largest n whose prefix
agrees), against ``numpy.argmax`` for per-row maxima, and on planted ties.
"""
from __future__ import annotations

import itertools

import numpy as np
import pytest

from speculative_decoding_verification_attn_gb300.workload import (
    bf16_bits_to_f32, f32_to_bf16_bits, make_inputs, small_spec)

from _util import oracle_accept


def expected_by_prefix_set(logits_f, drafts):
    """accepted = max{n : drafts[:n] == argmax[:n]}; next = argmax[accepted]."""
    am = np.argmax(logits_f, axis=-1)
    B, k = drafts.shape
    acc = np.array([max(n for n in range(k + 1) if np.array_equal(drafts[b, :n], am[b, :n]))
                    for b in range(B)])
    nxt = am[np.arange(B), acc]
    return acc, nxt, am


def test_brute_force_tiny_vocab(oracle_mod):
    # V = 3, k = 2: every draft vector against random and tied logit tables.
    rng = np.random.default_rng(0)
    tables = [rng.standard_normal((3, 3)).astype(np.float32) for _ in range(6)]
    tables.append(np.array([[1, 1, 0], [0, 2, 2], [5, 5, 5]], np.float32))
    tables.append(np.array([[-0.0, 0.0, -1], [0.0, -0.0, 0.0], [-3, -2, -2]], np.float32))
    drafts = np.array(list(itertools.product(range(3), repeat=2)), np.int32)
    for t in tables:
        logits = np.ascontiguousarray(np.broadcast_to(t, (len(drafts), 3, 3)))
        acc, nxt, am = oracle_mod.accept_greedy(logits, "f32", drafts)
        e_acc, e_nxt, e_am = expected_by_prefix_set(logits, drafts)
        np.testing.assert_array_equal(am, e_am)
        np.testing.assert_array_equal(acc, e_acc)
        np.testing.assert_array_equal(nxt, e_nxt)


@pytest.mark.parametrize("name_kw", [
    dict(logits_dtype="f32", vocab=1000),
    dict(logits_dtype="bf16", vocab=5003, num_draft=7),
    dict(logits_dtype="bf16", vocab=32000, draft_mode="geometric_break", match_prob=0.85),
])
def test_random_against_numpy_argmax(oracle_mod, name_kw):
    inp = make_inputs(small_spec(batch=16, **name_kw), seed=1)
    acc, nxt, am = oracle_accept(oracle_mod, inp)
    lf = inp.logits if inp.spec.logits_dtype == "f32" else bf16_bits_to_f32(inp.logits)
    e_acc, e_nxt, e_am = expected_by_prefix_set(lf, inp.draft_tokens)
    np.testing.assert_array_equal(am, e_am)
    np.testing.assert_array_equal(acc, e_acc)
    np.testing.assert_array_equal(nxt, e_nxt)
    k = inp.spec.num_draft
    assert ((acc >= 0) & (acc <= k)).all()
    tokens_out = acc + 1  # accepted drafts plus the target's own token
    assert ((tokens_out >= 1) & (tokens_out <= k + 1)).all()


def test_planted_ties_take_lowest_index(oracle_mod):
    V = 4096
    logits = np.zeros((1, 3, V), np.float32)
    logits[0, 0, [900, 17, 4000]] = 7.0   # tie between three indices
    logits[0, 1, [5, 6]] = 2.5
    logits[0, 2, V - 1] = 1.0
    bits = f32_to_bf16_bits(logits)
    for arr, dt in ((logits, "f32"), (bits, "bf16")):
        acc, nxt, am = oracle_mod.accept_greedy(arr, dt, np.array([[17, 5]], np.int32))
        assert am.tolist() == [[17, 5, V - 1]]
        assert acc.tolist() == [2] and nxt.tolist() == [V - 1]  # full accept -> bonus


def test_bf16_rounding_creates_ties(oracle_mod):
    # 8.03 and 8.0 differ in f32 but are the same bf16 value (ulp 2^-4 at 8).
    row = np.zeros((1, 2, 64), np.float32)
    row[0, 0, 40] = 8.03
    row[0, 0, 12] = 8.0
    f_acc, f_nxt, f_am = oracle_mod.accept_greedy(row, "f32", np.array([[12]], np.int32))
    b_acc, b_nxt, b_am = oracle_mod.accept_greedy(f32_to_bf16_bits(row), "bf16",
                                                  np.array([[12]], np.int32))
    assert f_am[0, 0] == 40 and f_acc[0] == 0 and f_nxt[0] == 40
    assert b_am[0, 0] == 12 and b_acc[0] == 1


def test_first_position_reject_and_full_accept(oracle_mod):
    inp = make_inputs(small_spec(batch=4, num_draft=5, vocab=777, logits_dtype="f32"), seed=2)
    _, _, am = oracle_accept(oracle_mod, inp)
    drafts = np.array([
        am[0, :5],                       # all agree -> bonus token from row k
        (am[1, :5] + 1) % 777,           # first position disagrees
        np.r_[am[2, :3], (am[2, 3] + 1) % 777, am[2, 4]],  # later agreement ignored
        np.r_[am[3, :4], (am[3, 4] + 5) % 777],
    ], np.int32)
    acc, nxt, _ = oracle_mod.accept_greedy(inp.logits, "f32", drafts)
    assert acc.tolist() == [5, 0, 3, 4]
    assert nxt.tolist() == [am[0, 5], am[1, 0], am[2, 3], am[3, 4]]

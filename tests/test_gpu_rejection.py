"""GPU parity of spec_accept_rejection against the float64 oracle.

Both sides draw from the same SplitMix64 stream, so the accepted length and
the next token are compared exactly.  The kernel decides in fp32: a test
whose uniform lies within 1e-4 of p/q, or a Gumbel-max whose two best keys
lie within 1e-3, may legitimately go the other way; such sequences are
checked for validity instead (and must be rare): the kept drafts passed and
the rejected one failed their tests with the same draws, and the emitted
token lies in the support of the residual (or of p after k acceptances)
with a Gumbel key within the tolerance of the best.  An independent
distribution check confirms that the GPU's first emitted token follows p.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from speculative_decoding_verification_attn_gb300 import binding
from speculative_decoding_verification_attn_gb300.workload import make_rejection_inputs

from _util import stored_to_f64

pytestmark = pytest.mark.gpu

U_AMBIG = 1e-4
KEY_AMBIG = 1e-3


@pytest.fixture(autouse=True)
def _lib():
    from speculative_decoding_verification_attn_gb300 import build
    build.build()
    binding.load()


def to_torch(r):
    kind = r.dtype
    def t(a):
        if kind == "bf16":
            return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).cuda()
        return torch.from_numpy(a).cuda()
    return t(r.target_logits), t(r.draft_logits), torch.from_numpy(r.draft_tokens).cuda()


def gpu_reject(r, seed=None, tl=None, dl=None, dr=None):
    if tl is None:
        tl, dl, dr = to_torch(r)
    B, k = r.draft_tokens.shape
    acc = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    nxt = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    binding.spec_accept_rejection(tl, dl, dr, k, r.temperature, r.seed if seed is None else seed,
                                  acc, nxt)
    torch.cuda.synchronize()
    return acc.cpu().numpy(), nxt.cpu().numpy()


def _probs(logits, dtype, temperature):
    """softmax(logits / T) per row in float64 (stored values widened)."""
    x = stored_to_f64(logits, dtype) / temperature
    x = x - x.max(axis=-1, keepdims=True)
    e = np.exp(x)
    return e / e.sum(axis=-1, keepdims=True)


def check_valid(oracle_mod, r, b, acc_b, nxt_b, p, q):
    """A result the fp32 kernel may legitimately reach on a near-tie: every
    kept draft passed its test u < p/q and the first rejected one failed it
    (each up to U_AMBIG, with the same SplitMix64 uniforms), the emitted token
    lies in the support of the residual max(p - q, 0) at the rejection (or of
    p after k acceptances), and its Gumbel key ln w + g is within KEY_AMBIG of
    the best key over that support."""
    k = r.draft_tokens.shape[1]
    x = r.draft_tokens[b]
    for i in range(min(acc_b + 1, k)):
        ratio = p[b, i, x[i]] / q[b, i, x[i]]
        u = oracle_mod.accept_uniform(r.seed, b, i)
        if i < acc_b:
            assert u < ratio + U_AMBIG, "sequence %d kept draft %d with u %.6g >= p/q %.6g" % (
                b, i, u, ratio)
        else:
            assert u >= ratio - U_AMBIG, "sequence %d rejected draft %d with u %.6g < p/q %.6g" % (
                b, i, u, ratio)
    if acc_b < k:
        w = np.maximum(p[b, acc_b] - q[b, acc_b], 0.0)
        # p and q are fp32 in the kernel: a token with p ~ q may sit on either side
        assert p[b, acc_b, nxt_b] >= q[b, acc_b, nxt_b] * (1 - 1e-4), (
            "sequence %d: token %d outside the residual's support" % (b, nxt_b))
    else:
        w = p[b, k]
    support = np.nonzero(w > 0)[0]
    keys = np.array([np.log(w[v]) + oracle_mod.gumbel(r.seed, b, int(v)) for v in support])
    got = (np.log(w[nxt_b]) if w[nxt_b] > 0 else -np.inf) + oracle_mod.gumbel(r.seed, b, nxt_b)
    assert got >= keys.max() - KEY_AMBIG, "sequence %d: token %d key %.6g, best %.6g" % (
        b, nxt_b, got, keys.max())


def check_against_oracle(oracle_mod, r, min_exact=0.9):
    acc, nxt = gpu_reject(r)
    o_acc, o_nxt, ratio, unif, gap = oracle_mod.accept_rejection(
        r.target_logits, r.draft_logits, r.dtype, r.draft_tokens, r.temperature, r.seed)
    B, k = r.draft_tokens.shape
    V = r.target_logits.shape[-1]
    assert np.all((acc >= 0) & (acc <= k)) and np.all((nxt >= 0) & (nxt < V))
    p = q = None
    exact = 0
    for b in range(B):
        n = o_acc[b]
        tested = min(n + 1, k)  # positions whose test the oracle ran
        ambiguous = bool(np.any(np.abs(unif[b, :tested] - ratio[b, :tested]) < U_AMBIG))
        if ambiguous or gap[b] < KEY_AMBIG:
            # near a tie the fp32 kernel may go the other way: check that its
            # result is one the rule allows
            if p is None:
                p = _probs(r.target_logits, r.dtype, r.temperature)
                q = _probs(r.draft_logits, r.dtype, r.temperature)
            check_valid(oracle_mod, r, b, int(acc[b]), int(nxt[b]), p, q)
            if ambiguous:
                continue
        assert acc[b] == n, "sequence %d: accepted %d, oracle %d" % (b, acc[b], n)
        if gap[b] < KEY_AMBIG:
            continue
        assert nxt[b] == o_nxt[b], "sequence %d: next %d, oracle %d" % (b, nxt[b], o_nxt[b])
        exact += 1
    assert exact >= min_exact * B, "only %d of %d sequences compared exactly" % (exact, B)
    assert binding.spec_device_error() == 0
    return acc, nxt


@pytest.mark.parametrize("dtype,B,k,V", [
    ("f32", 16, 4, 1000),
    ("bf16", 8, 8, 32000),
    ("bf16", 32, 1, 8192),       # exactly one slice
    ("bf16", 4, 16, 152064),     # long reasoning-step shape: 19 slices, 33 rows
    ("bf16", 6, 5, 1001),        # rows not on 16-byte boundaries
    ("f32", 5, 3, 777),
])
@pytest.mark.parametrize("seed", [0, 1])
def test_rejection_matches_oracle(oracle_mod, dtype, B, k, V, seed):
    r = make_rejection_inputs(B, k, V, dtype, seed=seed)
    check_against_oracle(oracle_mod, r)


def test_rejection_temperature(oracle_mod):
    r = make_rejection_inputs(12, 6, 4000, "bf16", seed=3, temperature=0.7)
    check_against_oracle(oracle_mod, r)


def test_all_drafts_kept_when_draft_equals_target(oracle_mod):
    r = make_rejection_inputs(16, 6, 5000, "f32", seed=4)
    r.draft_logits = np.ascontiguousarray(r.target_logits[:, :6])
    acc, nxt = check_against_oracle(oracle_mod, r)
    assert np.all(acc == 6)


def test_same_seed_same_tokens_new_seed_new_draws():
    r = make_rejection_inputs(64, 4, 3000, "bf16", seed=5, agreement=0.3)
    t = to_torch(r)
    a1 = gpu_reject(r, None, *t)
    a2 = gpu_reject(r, None, *t)
    a3 = gpu_reject(r, r.seed + 1, *t)
    assert np.array_equal(a1[0], a2[0]) and np.array_equal(a1[1], a2[1])
    assert not (np.array_equal(a1[0], a3[0]) and np.array_equal(a1[1], a3[1]))


def test_out_of_range_draft_is_rejected_and_flagged(oracle_mod):
    r = make_rejection_inputs(4, 3, 2000, "bf16", seed=6)
    r.draft_tokens[1, 0] = 2000
    acc, nxt = gpu_reject(r)
    assert acc[1] == 0 and 0 <= nxt[1] < 2000
    assert binding.spec_device_error() == binding.SPEC_DEVERR_TOKEN


def test_gpu_first_token_follows_target():
    # k = 1, drafts drawn from q: the first emitted token follows p
    B, V = 16000, 6
    rng = np.random.default_rng(11)
    lp = (rng.standard_normal(V) * 1.5).astype(np.float32)
    lq = (rng.standard_normal(V) * 1.5).astype(np.float32)
    q = np.exp(lq.astype(np.float64) - lq.max()); q /= q.sum()
    p = np.exp(lp.astype(np.float64) - lp.max()); p /= p.sum()
    tl = torch.from_numpy(np.tile(np.stack([lp, lp])[None], (B, 1, 1))).cuda()
    dl = torch.from_numpy(np.tile(lq[None, None], (B, 1, 1))).cuda()
    drafts = rng.choice(V, size=(B, 1), p=q).astype(np.int32)
    dr = torch.from_numpy(drafts).cuda()
    acc = torch.empty(B, dtype=torch.int32, device="cuda")
    nxt = torch.empty(B, dtype=torch.int32, device="cuda")
    binding.spec_accept_rejection(tl, dl, dr, 1, 1.0, 2024, acc, nxt)
    torch.cuda.synchronize()
    a, n = acc.cpu().numpy(), nxt.cpu().numpy()
    first = np.where(a == 1, drafts[:, 0], n)
    counts = np.bincount(first, minlength=V)
    sd = np.sqrt(B * p * (1 - p))
    assert np.all(np.abs(counts - B * p) <= 5 * sd)

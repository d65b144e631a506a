"""Helpers for the GPU parity tests: run the CUDA path, compare with the oracle."""
from __future__ import annotations

import numpy as np
import torch

from speculative_decoding_verification_attn_gb300 import binding
from speculative_decoding_verification_attn_gb300.workload import VerifyInputs

from _util import all_rows, oracle_accept, oracle_attn, oracle_rows, oracle_rows_parallel, rel_l2

# Tolerances for the attention output against the float64 oracle: fp32
# inputs keep fp32 arithmetic end to end (max-abs 1e-5); bf16 / INT8 caches
# round P to bf16 for the tensor cores and store a bf16 output (max-abs 2e-2
# and relative L2 3e-3).  lse (fp32 in both) gets 1e-5 / 2e-3 absolute.
TOL = {
    "f32": dict(max_abs=1e-5, rel_l2=None, lse=1e-5),
    "bf16": dict(max_abs=2e-2, rel_l2=3e-3, lse=2e-3),
}


def tol_for(inp: VerifyInputs):
    return TOL["f32"] if inp.spec.q_dtype == "f32" and inp.spec.kv_dtype == "f32" else TOL["bf16"]


def gpu_attn(inp: VerifyInputs, t=None):
    """Run spec_verify_attn; return (out float64 numpy, lse numpy)."""
    t = t or binding.inputs_to_torch(inp)
    o = binding.alloc_outputs(inp)
    o["out"].fill_(float("nan"))
    o["lse"].fill_(float("nan"))
    binding.spec_verify_attn(t["q"], t["k_cache"], t["v_cache"], t["block_table"], t["ctx_lens"],
                             inp.spec.num_draft, inp.scale, o["out"], o["lse"], t.get("k_scale"),
                             t.get("v_scale"))
    torch.cuda.synchronize()
    return o["out"].double().cpu().numpy(), o["lse"].double().cpu().numpy()


def gpu_accept(inp: VerifyInputs, t=None):
    t = t or binding.inputs_to_torch(inp)
    o = binding.alloc_outputs(inp)
    o["accepted_len"].fill_(-7)
    o["next_token"].fill_(-7)
    binding.spec_accept_greedy(t["logits"], t["draft_tokens"], inp.spec.num_draft,
                               o["accepted_len"], o["next_token"])
    torch.cuda.synchronize()
    return o["accepted_len"].cpu().numpy(), o["next_token"].cpu().numpy()


def assert_attn_close(out, lse, ref_out, ref_lse, tol, what=""):
    assert np.isfinite(out).all(), "non-finite output %s" % what
    err = np.abs(out - ref_out).max() if out.size else 0.0
    assert err <= tol["max_abs"], "%s max-abs %.3g > %.3g" % (what, err, tol["max_abs"])
    if tol["rel_l2"] is not None and out.size:
        r = rel_l2(out, ref_out)
        assert r <= tol["rel_l2"], "%s rel-L2 %.3g > %.3g" % (what, r, tol["rel_l2"])
    lerr = np.abs(lse - ref_lse).max() if lse.size else 0.0
    assert lerr <= tol["lse"], "%s lse max-abs %.3g > %.3g" % (what, lerr, tol["lse"])


def check_attn_full(oracle, inp: VerifyInputs, what=""):
    out, lse = gpu_attn(inp)
    ref_out, ref_lse = oracle_attn(oracle, inp)
    assert_attn_close(out, lse, ref_out, ref_lse, tol_for(inp), what)
    assert binding.spec_device_error() == 0


def check_attn_every_row(oracle, inp: VerifyInputs, t=None, what=""):
    """Every output row of a (full-size) call against the oracle, which runs
    on every host core."""
    out, lse = gpu_attn(inp, t)
    s = inp.spec
    ref_o, ref_l = oracle_rows_parallel(oracle, inp, all_rows(inp))
    ref_o = ref_o.reshape(s.batch, s.num_draft, s.num_q_heads, s.head_dim)
    ref_l = ref_l.reshape(s.batch, s.num_draft, s.num_q_heads)
    assert_attn_close(out, lse, ref_o, ref_l, tol_for(inp), what)
    assert binding.spec_device_error() == 0
    return out, lse


def check_accept(oracle, inp: VerifyInputs, t=None):
    acc, nxt = gpu_accept(inp, t)
    e_acc, e_nxt, _ = oracle_accept(oracle, inp)
    np.testing.assert_array_equal(acc, e_acc)
    np.testing.assert_array_equal(nxt, e_nxt)


_FULL = {}


def full_inputs(name: str, seed: int = 0):
    """Full-size named workload (cached for the session)."""
    from speculative_decoding_verification_attn_gb300.workload import make_inputs
    key = (name, seed)
    if key not in _FULL:
        _FULL.clear()  # keep at most one full-size workload in host memory
        _FULL[key] = make_inputs(name, seed=seed)
    return _FULL[key]

"""GPU parity of spec_verify_attn against the float64 oracle.

Small cases (the oracle computes every output) span several 64-key tiles,
ragged tails, contexts of zero, every supported page size, GQA groups of 1 to
8 and 1 to 128 query rows per kv-head, forced stream-K splits of every size,
every kernel; the named full-size workloads are checked on every output row,
for three seeds, at the launch configuration the benchmark times (the oracle
runs on every host core).  NaN canaries fill every
unused cache slot: a kernel that reads past a sequence shows non-finite
output.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from speculative_decoding_verification_attn_gb300 import binding
from speculative_decoding_verification_attn_gb300.workload import (
    WORKLOADS, make_inputs, small_spec)

from gpu_util import (assert_attn_close, check_attn_every_row, check_attn_full, full_inputs,
                      gpu_attn, tol_for)
from _util import oracle_attn

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


SMALL_BF16 = [
    dict(),
    dict(num_q_heads=4, num_kv_heads=4, num_draft=1),                    # 1 row per kv-head
    dict(num_q_heads=28, num_kv_heads=4, num_draft=16, page_size=32),     # 112 rows
    dict(num_q_heads=16, num_kv_heads=2, num_draft=8),                    # 64 rows
    dict(num_q_heads=4, num_kv_heads=2, num_draft=64),                    # 128 rows
    dict(ctx=[0, 1, 63, 64, 65], batch=5, num_draft=3),                   # tile edges
    dict(page_size=32, ctx=(1, 200), num_draft=2),
    dict(page_size=64, ctx=(1, 400)),
    dict(page_size=128, ctx=(100, 600)),
    dict(page_size=256, ctx=(250, 700), batch=2),
    dict(batch=1, num_q_heads=8, num_kv_heads=1, ctx=[3000]),              # one long segment
    dict(num_q_heads=7, num_kv_heads=7, num_draft=5, ctx=(0, 130)),
    dict(batch=1024, num_q_heads=4, num_kv_heads=2, num_draft=2, ctx=(0, 40)),  # most sequences
]


@pytest.mark.parametrize("kw", SMALL_BF16, ids=[str(i) for i in range(len(SMALL_BF16))])
def test_tensor_core_small(oracle_mod, kw):
    inp = make_inputs(small_spec(**kw), seed=21)
    binding.spec_set_option(binding.SPEC_OPT_ATTN_PATH, 2)
    check_attn_full(oracle_mod, inp, str(kw))


# query rows per kv-head 24 (four copies), 48 (two copies), 84 (one copy):
# each with both softmax sets, the merge of their states and of the copies,
# and the combine in its by-boundary (few CTAs) and by-segment forms
@pytest.mark.parametrize("heads", [(16, 4, 6), (16, 2, 6), (28, 4, 12)],
                         ids=["24rows", "48rows", "84rows"])
@pytest.mark.parametrize("ctas", [1, 2, 5, 37, 152, 400])
def test_tensor_core_stream_k_splits(oracle_mod, ctas, heads):
    hq, hkv, k = heads
    inp = make_inputs(small_spec(batch=4, num_q_heads=hq, num_kv_heads=hkv, num_draft=k,
                                 ctx=(0, 900)), seed=22)
    binding.spec_set_option(binding.SPEC_OPT_ATTN_PATH, 2)
    binding.spec_set_option(binding.SPEC_OPT_NUM_CTAS, ctas)
    check_attn_full(oracle_mod, inp, "ctas=%d heads=%s" % (ctas, heads))


# the split of the tile list over the persistent CTAs charges every segment a
# number of tiles for its fixed work (option value = tiles + 1; 1: the equal
# split): ranges then start and end at other places, with more or fewer
# pieces per segment and empty ranges when the charge dominates
@pytest.mark.parametrize("weight", [1, 2, 14, 65])
@pytest.mark.parametrize("path,kw", [
    (2, dict(num_q_heads=28, num_kv_heads=4, num_draft=12)),            # tcgen05, 84 rows
    (2, dict(num_q_heads=16, num_kv_heads=2, num_draft=6)),             # tcgen05, copies
    (2, dict(num_q_heads=32, num_kv_heads=4, num_draft=8, kv_dtype="i8")),
    (3, dict(num_q_heads=16, num_kv_heads=4, num_draft=4)),             # warp-MMA
], ids=["tc84", "tc48", "tc_i8", "mma16"])
@pytest.mark.parametrize("ctas", [5, 37, 152])
def test_split_weights(oracle_mod, weight, path, kw, ctas):
    inp = make_inputs(small_spec(batch=6, ctx=(0, 1500), **kw), seed=34)
    binding.spec_set_option(binding.SPEC_OPT_ATTN_PATH, path)
    binding.spec_set_option(binding.SPEC_OPT_NUM_CTAS, ctas)
    binding.spec_set_option(binding.SPEC_OPT_SPLIT_WEIGHT, weight)
    check_attn_full(oracle_mod, inp, "path %d weight %d ctas %d" % (path, weight, ctas))


SMALL_I8 = [
    dict(kv_dtype="i8"),                                                  # 16 rows
    dict(kv_dtype="i8", num_q_heads=4, num_kv_heads=4, num_draft=1),      # 1 row per kv-head
    dict(kv_dtype="i8", num_q_heads=16, num_kv_heads=2, num_draft=8),     # 64 rows
    dict(kv_dtype="i8", num_q_heads=28, num_kv_heads=4, num_draft=16, page_size=32),  # 112
    dict(kv_dtype="i8", num_q_heads=4, num_kv_heads=2, num_draft=64),     # 128 rows
    dict(kv_dtype="i8", ctx=[0, 1, 63, 64, 65], batch=5, num_draft=3),    # tile edges
    dict(kv_dtype="i8", page_size=64, ctx=(1, 400)),
    dict(kv_dtype="i8", page_size=256, ctx=(250, 700), batch=2),
    dict(kv_dtype="i8", batch=1, num_q_heads=8, num_kv_heads=1, ctx=[3000]),
]


@pytest.mark.parametrize("kw", SMALL_I8, ids=[str(i) for i in range(len(SMALL_I8))])
def test_tensor_core_int8_small(oracle_mod, kw):
    # INT8 cache widened to fp16 on chip; scales folded into scores and P
    inp = make_inputs(small_spec(**kw), seed=41)
    binding.spec_set_option(binding.SPEC_OPT_ATTN_PATH, 2)
    check_attn_full(oracle_mod, inp, "i8 %s" % kw)


@pytest.mark.parametrize("ctas", [1, 3, 37, 152, 400])
def test_tensor_core_int8_stream_k_splits(oracle_mod, ctas):
    inp = make_inputs(small_spec(batch=4, num_q_heads=32, num_kv_heads=4, num_draft=8,
                                 kv_dtype="i8", ctx=(0, 900)), seed=42)
    binding.spec_set_option(binding.SPEC_OPT_ATTN_PATH, 2)
    binding.spec_set_option(binding.SPEC_OPT_NUM_CTAS, ctas)
    check_attn_full(oracle_mod, inp, "i8 ctas=%d" % ctas)


def test_tensor_core_int8_matches_simt():
    inp = make_inputs(small_spec(batch=5, num_q_heads=24, num_kv_heads=4, num_draft=6,
                                 kv_dtype="i8", ctx=(0, 700)), seed=43)
    t = binding.inputs_to_torch(inp)
    binding.spec_set_option(binding.SPEC_OPT_ATTN_PATH, 2)
    a_out, a_lse = gpu_attn(inp, t)
    binding.spec_set_option(binding.SPEC_OPT_ATTN_PATH, 1)
    b_out, b_lse = gpu_attn(inp, t)
    assert np.abs(a_out - b_out).max() < 2e-2
    assert np.abs(a_lse - b_lse).max() < 2e-3


def test_int8_unaligned_scales_use_simt(oracle_mod):
    # scale arrays that are not 16-byte aligned cannot feed the bulk copies of
    # the tensor-core kernel: the automatic path runs the SIMT kernel, a
    # forced tensor-core path is refused
    inp = make_inputs(small_spec(kv_dtype="i8", num_q_heads=16, num_kv_heads=2, num_draft=8),
                      seed=44)
    t = binding.inputs_to_torch(inp)
    for key in ("k_scale", "v_scale"):
        flat = torch.empty(t[key].numel() + 8, dtype=t[key].dtype, device="cuda")
        shifted = flat[1:1 + t[key].numel()].view(t[key].shape)
        shifted.copy_(t[key])
        t[key] = shifted
    out, lse = gpu_attn(inp, t)
    ref_out, ref_lse = oracle_attn(oracle_mod, inp)
    assert_attn_close(out, lse, ref_out, ref_lse, tol_for(inp), "unaligned scales")
    binding.spec_set_option(binding.SPEC_OPT_ATTN_PATH, 2)
    with pytest.raises(binding.SpecError, match="does not support"):
        gpu_attn(inp, t)


@pytest.mark.parametrize("kw", [
    dict(),
    dict(kv_dtype="i8"),
    dict(kv_dtype="i8", num_q_heads=16, num_kv_heads=2, num_draft=8),
    dict(q_dtype="f32", kv_dtype="f32", head_dim=64),
    dict(q_dtype="f32", kv_dtype="i8", head_dim=256, num_draft=2),
    dict(q_dtype="bf16", kv_dtype="f32", head_dim=32, page_size=5, ctx=(0, 77)),
    dict(head_dim=96, page_size=3, ctx=[0, 10, 31]),
])
@pytest.mark.parametrize("chunk", [0, 16, 48])
def test_simt_small(oracle_mod, kw, chunk):
    inp = make_inputs(small_spec(**kw), seed=23)
    binding.spec_set_option(binding.SPEC_OPT_ATTN_PATH, 1)
    binding.spec_set_option(binding.SPEC_OPT_SIMT_CHUNK, chunk)
    check_attn_full(oracle_mod, inp, "%s chunk=%d" % (kw, chunk))


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_tiny_fp32_workload(oracle_mod, seed):
    check_attn_full(oracle_mod, make_inputs("tiny_fp32", seed=seed), "tiny_fp32")


# single-pass SIMT kernel: whole sequences in shared memory, one launch
SINGLE_PASS = [
    dict(q_dtype="f32", kv_dtype="f32", head_dim=64),
    dict(q_dtype="f32", kv_dtype="f32", head_dim=64, batch=1, num_q_heads=2, num_kv_heads=2,
         ctx=[128], num_draft=4),
    dict(ctx=(0, 150)),                                                       # bf16
    dict(kv_dtype="i8", num_q_heads=16, num_kv_heads=2, num_draft=8, ctx=(0, 110)),  # 64 rows
    dict(q_dtype="f32", kv_dtype="i8", head_dim=256, num_draft=2, ctx=(0, 60)),
    dict(q_dtype="bf16", kv_dtype="f32", head_dim=32, page_size=5, ctx=(0, 77)),
    dict(head_dim=96, page_size=3, ctx=[0, 10, 31]),
    dict(num_q_heads=4, num_kv_heads=2, num_draft=64, ctx=(0, 60)),          # 128 rows: 2 groups
    dict(batch=300, num_q_heads=4, num_kv_heads=4, num_draft=3, ctx=(0, 40)),
]


@pytest.mark.parametrize("kw", SINGLE_PASS, ids=[str(i) for i in range(len(SINGLE_PASS))])
def test_single_pass_simt(oracle_mod, kw):
    inp = make_inputs(small_spec(**kw), seed=35)
    binding.spec_set_option(binding.SPEC_OPT_ATTN_PATH, 4)
    check_attn_full(oracle_mod, inp, "single pass %s" % kw)


# the same kernel with each unit's keys split over a thread-block cluster
# (forced sizes, 5 not a power of two; ctx 0 leaves CTAs without keys)
CLUSTER_CASES = [
    dict(q_dtype="f32", kv_dtype="f32", head_dim=64, batch=1, num_q_heads=2, num_kv_heads=2,
         ctx=[128], num_draft=4),
    dict(q_dtype="f32", kv_dtype="f32", head_dim=64, batch=4, ctx=[0, 1, 7, 200]),
    dict(ctx=(0, 150)),                                                       # bf16
    dict(kv_dtype="i8", num_q_heads=16, num_kv_heads=2, num_draft=8, ctx=(0, 100)),  # 64 rows
    dict(q_dtype="f32", kv_dtype="i8", head_dim=256, num_draft=2, ctx=(0, 60)),
    dict(q_dtype="bf16", kv_dtype="f32", head_dim=32, page_size=5, ctx=(0, 77)),
    dict(num_q_heads=4, num_kv_heads=2, num_draft=64, ctx=(0, 40)),          # 128 rows: 2 groups
    dict(q_dtype="f32", kv_dtype="f32", head_dim=64, batch=2, ctx=[200, 250], num_draft=6),
]


@pytest.mark.parametrize("cluster", [2, 5, 8])
@pytest.mark.parametrize("kw", CLUSTER_CASES, ids=[str(i) for i in range(len(CLUSTER_CASES))])
def test_single_pass_cluster(oracle_mod, kw, cluster):
    inp = make_inputs(small_spec(**kw), seed=37)
    binding.spec_set_option(binding.SPEC_OPT_ATTN_PATH, 4)
    binding.spec_set_option(binding.SPEC_OPT_SMALL_CLUSTER, cluster)
    check_attn_full(oracle_mod, inp, "single pass, cluster %d, %s" % (cluster, kw))


def test_single_pass_cluster_matches_one_cta():
    # automatic (a cluster of 8 on this few units) against one CTA per unit
    inp = make_inputs("tiny_fp32", seed=3)
    t = binding.inputs_to_torch(inp)
    binding.spec_set_option(binding.SPEC_OPT_ATTN_PATH, 4)
    a_out, a_lse = gpu_attn(inp, t)
    binding.spec_set_option(binding.SPEC_OPT_SMALL_CLUSTER, 1)
    b_out, b_lse = gpu_attn(inp, t)
    assert np.abs(a_out - b_out).max() < 1e-5
    assert np.abs(a_lse - b_lse).max() < 1e-5


def test_single_pass_refuses_long_tables():
    # a block table longer than the kernel's shared memory holds: forced
    # single pass is refused, the automatic choice runs the chunked kernel
    inp = make_inputs(small_spec(q_dtype="f32", kv_dtype="f32", batch=1, ctx=[5000]), seed=36)
    binding.spec_set_option(binding.SPEC_OPT_ATTN_PATH, 4)
    with pytest.raises(binding.SpecError, match="does not support"):
        gpu_attn(inp)


def test_page_size_8_runs_on_simt(oracle_mod):
    # the tensor-core kernel loads one TMA box per page and needs >= 16 keys
    # per box; smaller pages go to the SIMT kernel under the automatic path
    inp = make_inputs(small_spec(page_size=8, ctx=(1, 200)), seed=29)
    check_attn_full(oracle_mod, inp, "page_size=8")
    for path in (2, 3):
        binding.spec_set_option(binding.SPEC_OPT_ATTN_PATH, path)
        with pytest.raises(binding.SpecError, match="does not support"):
            gpu_attn(inp)


def test_tensor_core_matches_simt():
    inp = make_inputs(small_spec(batch=6, num_q_heads=12, num_kv_heads=3, num_draft=5,
                                 ctx=(0, 700)), seed=24)
    t = binding.inputs_to_torch(inp)
    binding.spec_set_option(binding.SPEC_OPT_ATTN_PATH, 2)
    a_out, a_lse = gpu_attn(inp, t)
    binding.spec_set_option(binding.SPEC_OPT_ATTN_PATH, 1)
    b_out, b_lse = gpu_attn(inp, t)
    assert np.abs(a_out - b_out).max() < 2e-2
    assert np.abs(a_lse - b_lse).max() < 2e-3


FULL_SIZE = [(name, seed) for name in ("mha7b_bf16", "gqa8b_ragged_bf16", "long_step_k16_bf16",
                                        "int8kv_70b_layer") for seed in (0, 1, 2)]


@pytest.mark.parametrize("name,seed", FULL_SIZE, ids=["%s-%d" % c for c in FULL_SIZE])
def test_named_workload_every_row(oracle_mod, name, seed):
    # the full-size workloads at the launch configuration the benchmark times
    # (automatic kernel choice, one CTA per SM): every (b, i, h) output row
    # against the oracle, so every stream-K range boundary and piece merge of
    # the full-size split is checked
    inp = full_inputs(name, seed)
    check_attn_every_row(oracle_mod, inp, what="%s seed %d" % (name, seed))


def test_lse_optional(oracle_mod):
    inp = make_inputs(small_spec(), seed=25)
    t = binding.inputs_to_torch(inp)
    o = binding.alloc_outputs(inp)
    binding.spec_verify_attn(t["q"], t["k_cache"], t["v_cache"], t["block_table"], t["ctx_lens"],
                             inp.spec.num_draft, inp.scale, o["out"], None)
    torch.cuda.synchronize()
    ref, _ = oracle_attn(oracle_mod, inp)
    assert np.abs(o["out"].double().cpu().numpy() - ref).max() < 2e-2


@pytest.mark.parametrize("path", [1, 2])
def test_bad_page_id_is_clamped_and_flagged(path):
    inp = make_inputs(small_spec(), seed=26)
    inp.block_table[0, 0] = inp.num_pages + 5
    binding.spec_set_option(binding.SPEC_OPT_ATTN_PATH, path)
    assert binding.spec_device_error() == 0
    out, _ = gpu_attn(inp)
    assert binding.spec_device_error() == binding.SPEC_DEVERR_PAGE
    assert np.isfinite(out[1:]).all()


def test_validate_option_rejects_bad_tables():
    inp = make_inputs(small_spec(), seed=27)
    inp.block_table[1, 0] = -1
    binding.spec_set_option(binding.SPEC_OPT_VALIDATE, 1)
    with pytest.raises(binding.SpecError, match="block_table"):
        gpu_attn(inp)
    inp2 = make_inputs(small_spec(), seed=27)
    inp2.ctx_lens[0] = inp2.max_pages * inp2.spec.page_size
    with pytest.raises(binding.SpecError, match="ctx_lens"):
        gpu_attn(inp2)


def test_misaligned_pointer_rejected():
    inp = make_inputs(small_spec(), seed=28)
    t = binding.inputs_to_torch(inp)
    o = binding.alloc_outputs(inp)
    flat = torch.empty(t["q"].numel() + 8, dtype=torch.bfloat16, device="cuda")
    q_bad = flat[1:1 + t["q"].numel()].view(t["q"].shape)
    with pytest.raises(binding.SpecError, match="aligned"):
        binding.spec_verify_attn(q_bad, t["k_cache"], t["v_cache"], t["block_table"],
                                 t["ctx_lens"], inp.spec.num_draft, inp.scale, o["out"], o["lse"])


MMA_CASES = [k for k in SMALL_BF16
             if k.get("num_draft", 4) * (k.get("num_q_heads", 8) // k.get("num_kv_heads", 2)) <= 16]


@pytest.mark.parametrize("kw", MMA_CASES, ids=[str(i) for i in range(len(MMA_CASES))])
def test_warp_mma_small(oracle_mod, kw):
    inp = make_inputs(small_spec(**kw), seed=31)
    binding.spec_set_option(binding.SPEC_OPT_ATTN_PATH, 3)
    check_attn_full(oracle_mod, inp, "mma %s" % kw)


@pytest.mark.parametrize("ctas", [1, 3, 37, 152, 400])
def test_warp_mma_stream_k_splits(oracle_mod, ctas):
    inp = make_inputs(small_spec(batch=5, num_q_heads=16, num_kv_heads=4, num_draft=4,
                                 ctx=(0, 900)), seed=32)
    binding.spec_set_option(binding.SPEC_OPT_ATTN_PATH, 3)
    binding.spec_set_option(binding.SPEC_OPT_NUM_CTAS, ctas)
    check_attn_full(oracle_mod, inp, "mma ctas=%d" % ctas)


def test_warp_mma_matches_tcgen05():
    inp = make_inputs(small_spec(batch=6, num_q_heads=12, num_kv_heads=3, num_draft=4,
                                 ctx=(0, 700)), seed=33)
    t = binding.inputs_to_torch(inp)
    binding.spec_set_option(binding.SPEC_OPT_ATTN_PATH, 3)
    a_out, a_lse = gpu_attn(inp, t)
    binding.spec_set_option(binding.SPEC_OPT_ATTN_PATH, 2)
    b_out, b_lse = gpu_attn(inp, t)
    assert np.abs(a_out - b_out).max() < 2e-2
    assert np.abs(a_lse - b_lse).max() < 2e-3


def test_batch_beyond_tensor_core_limit(oracle_mod):
    # 1025 sequences: the tcgen05 kernel refuses a forced call; the automatic
    # choice still runs (another kernel) and matches the oracle
    inp = make_inputs(small_spec(batch=1025, num_q_heads=4, num_kv_heads=1, num_draft=8,
                                 ctx=(0, 20)), seed=23)
    binding.spec_set_option(binding.SPEC_OPT_ATTN_PATH, 2)
    t = binding.inputs_to_torch(inp)
    o = binding.alloc_outputs(inp)
    with pytest.raises(binding.SpecError):
        binding.run_verify(t, o, inp.spec.num_draft, inp.scale)
    binding.spec_set_option(binding.SPEC_OPT_ATTN_PATH, 0)
    out, lse = gpu_attn(inp, t)
    ref_out, ref_lse = oracle_attn(oracle_mod, inp)
    assert_attn_close(out, lse, ref_out, ref_lse, tol_for(inp), "batch 1025")


def test_descriptor_form_matches_flat_calls():
    # spec_verify_attn_tensors / spec_accept_greedy_tensors: same kernels, same
    # results as the flat calls, bit for bit (bf16 and INT8 caches)
    for kw in (dict(), dict(kv_dtype="i8", num_q_heads=16, num_kv_heads=2, num_draft=8)):
        inp = make_inputs(small_spec(**kw), seed=37)
        t = binding.inputs_to_torch(inp)
        a = binding.alloc_outputs(inp)
        b = binding.alloc_outputs(inp)
        s = inp.spec
        binding.spec_verify_attn(t["q"], t["k_cache"], t["v_cache"], t["block_table"],
                                 t["ctx_lens"], s.num_draft, inp.scale, a["out"], a["lse"],
                                 t.get("k_scale"), t.get("v_scale"))
        binding.spec_verify_attn_tensors(t["q"], t["k_cache"], t["v_cache"], t["block_table"],
                                         t["ctx_lens"], s.num_draft, inp.scale, b["out"], b["lse"],
                                         t.get("k_scale"), t.get("v_scale"))
        binding.spec_accept_greedy(t["logits"], t["draft_tokens"], s.num_draft, a["accepted_len"],
                                   a["next_token"])
        binding.spec_accept_greedy_tensors(t["logits"], t["draft_tokens"], s.num_draft,
                                           b["accepted_len"], b["next_token"])
        torch.cuda.synchronize()
        for n in ("out", "lse", "accepted_len", "next_token"):
            assert torch.equal(a[n], b[n]), n
    # a strided (non-dense) q is refused before anything runs
    wide = torch.empty(inp.q.shape[:-1] + (2 * s.head_dim,), dtype=t["q"].dtype, device="cuda")
    with pytest.raises(binding.SpecError, match="dense row-major"):
        binding.spec_verify_attn_tensors(wide[..., :s.head_dim], t["k_cache"], t["v_cache"],
                                         t["block_table"], t["ctx_lens"], s.num_draft, inp.scale,
                                         b["out"], b["lse"], t.get("k_scale"), t.get("v_scale"))

"""The C-ABI library: it builds for sm_103a, loads, exports every symbol the
public header declares, and rejects bad arguments before touching the GPU.
Runs without a GPU (argument validation precedes every CUDA call)."""
from __future__ import annotations

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "spec_verify.h")


@pytest.fixture(scope="module")
def lib():
    from speculative_decoding_verification_attn_gb300 import binding, build
    build.build()
    return binding.load()


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*SPEC_API\s+(?:int|const char \*)\s*(spec_\w+)\s*\(", text, re.M)))


def test_header_declares_the_calls():
    syms = declared_symbols()
    assert "spec_verify_attn" in syms and "spec_accept_greedy" in syms
    from speculative_decoding_verification_attn_gb300 import binding
    assert sorted(binding.EXPORTED) == syms


def test_every_declared_symbol_is_exported(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name
    assert lib.spec_version() >= 100


def test_internal_symbols_are_hidden(lib):
    with pytest.raises(AttributeError):
        getattr(lib, "_ZN5specv9simt_planERKNS_8AttnArgsEii")


def _attn(lib, **kw):
    args = dict(q=16, kc=16, vc=16, ks=None, vs=None, bt=16, ctx=16, B=1, k=4, Hq=8, Hkv=2, D=128,
                P=16, NP=8, MP=4, qdt=1, kvdt=1, scale=0.088, out=16, lse=None, stream=None)
    args.update(kw)
    vp = lambda x: None if x is None else ctypes.c_void_p(x)
    return lib.spec_verify_attn(vp(args["q"]), vp(args["kc"]), vp(args["vc"]), vp(args["ks"]),
                                vp(args["vs"]), vp(args["bt"]), vp(args["ctx"]), args["B"],
                                args["k"], args["Hq"], args["Hkv"], args["D"], args["P"],
                                args["NP"], args["MP"], args["qdt"], args["kvdt"], args["scale"],
                                vp(args["out"]), vp(args["lse"]), vp(args["stream"]))


@pytest.mark.parametrize("bad,needle", [
    (dict(k=0), "num_draft"),
    (dict(k=65), "num_draft"),
    (dict(Hq=6, Hkv=4), "multiple"),
    (dict(D=100), "head_dim"),
    (dict(P=0), "page_size"),
    (dict(qdt=3), "q_dtype"),
    (dict(kvdt=2), "kv_dtype"),
    (dict(q=0), "null"),
    (dict(kvdt=3), "I8"),
    (dict(q=24), "aligned"),
    (dict(scale=float("nan")), "NaN"),
])
def test_attn_rejects_bad_arguments(lib, bad, needle):
    rc = _attn(lib, **bad)
    assert rc == -1
    assert needle in lib.spec_last_error().decode()


def test_empty_batch_is_a_no_op(lib):
    assert _attn(lib, B=0, q=None, kc=None, vc=None, out=None) == 0
    assert lib.spec_last_error().decode() == ""


@pytest.mark.parametrize("bad,needle", [
    (dict(k=0), "num_draft"),
    (dict(V=0), "vocab"),
    (dict(dt=3), "logits_dtype"),
    (dict(logits=0), "null"),
    (dict(logits=18), "aligned"),
])
def test_accept_rejects_bad_arguments(lib, bad, needle):
    a = dict(logits=16, dt=1, draft=16, B=2, k=4, V=1000, acc=16, nxt=16)
    a.update(bad)
    vp = lambda x: ctypes.c_void_p(x) if x else None
    rc = lib.spec_accept_greedy(vp(a["logits"]), a["dt"], vp(a["draft"]), a["B"], a["k"], a["V"],
                                vp(a["acc"]), vp(a["nxt"]), None)
    assert rc == -1
    assert needle in lib.spec_last_error().decode()


@pytest.mark.parametrize("bad,needle", [
    (dict(k=0), "num_draft"),
    (dict(V=0), "vocab"),
    (dict(dt=2), "logits_dtype"),
    (dict(T=0.0), "temperature"),
    (dict(T=float("nan")), "temperature"),
    (dict(T=float("inf")), "temperature"),
    (dict(dl=0), "null"),
    (dict(tl=24), "aligned"),
    (dict(dl=40), "aligned"),
])
def test_rejection_rejects_bad_arguments(lib, bad, needle):
    a = dict(tl=16, dl=32, dt=1, draft=16, B=2, k=4, V=1000, T=1.0, acc=16, nxt=16)
    a.update(bad)
    vp = lambda x: ctypes.c_void_p(x) if x else None
    rc = lib.spec_accept_rejection(vp(a["tl"]), vp(a["dl"]), a["dt"], vp(a["draft"]), a["B"],
                                   a["k"], a["V"], a["T"], 7, vp(a["acc"]), vp(a["nxt"]), None)
    assert rc == -1
    assert needle in lib.spec_last_error().decode()


@pytest.mark.parametrize("bad,needle", [
    (dict(n=0), "num_new"),
    (dict(D=48), "head_dim"),
    (dict(src=3), "src_dtype"),
    (dict(cdt=2), "cache_dtype"),
    (dict(kc=0), "null"),
    (dict(cdt=3), "I8"),
])
def test_kv_append_rejects_bad_arguments(lib, bad, needle):
    a = dict(kn=16, vn=16, src=1, kc=16, vc=16, ks=None, vs=None, cdt=1, bt=16, ctx=16, B=2, n=4,
             Hkv=2, D=128, P=16, NP=8, MP=4)
    a.update(bad)
    vp = lambda x: ctypes.c_void_p(x) if x else None
    rc = lib.spec_kv_append(vp(a["kn"]), vp(a["vn"]), a["src"], vp(a["kc"]), vp(a["vc"]),
                            vp(a["ks"]), vp(a["vs"]), a["cdt"], vp(a["bt"]), vp(a["ctx"]), a["B"],
                            a["n"], a["Hkv"], a["D"], a["P"], a["NP"], a["MP"], None)
    assert rc == -1
    assert needle in lib.spec_last_error().decode()


@pytest.mark.parametrize("bad,needle", [
    (dict(nblk=-1), "num_blocks"),
    (dict(D=48), "head_dim"),
    (dict(D=288), "head_dim"),
    (dict(P=0), "page_size"),
    (dict(P=129), "page_size"),
    (dict(codes=0), "null"),
    (dict(np_=0), "null"),
])
def test_codec_rejects_bad_arguments(lib, bad, needle):
    a = dict(codes=64, pairs=64, np_=64, nblk=4, P=16, D=128)
    a.update(bad)
    vp = lambda x: ctypes.c_void_p(x) if x else None
    for rc in (lib.spec_codec_encode(vp(a["codes"]), a["nblk"], a["P"], a["D"], vp(a["pairs"]),
                                     vp(a["np_"]), None),
               lib.spec_codec_decode(vp(a["pairs"]), vp(a["np_"]), a["nblk"], a["P"], a["D"],
                                     vp(a["codes"]), None)):
        assert rc == -1
        assert needle in lib.spec_last_error().decode()


def test_codec_decode_rejects_unaligned(lib):
    rc = lib.spec_codec_decode(ctypes.c_void_p(66), ctypes.c_void_p(64), 4, 16, 128,
                               ctypes.c_void_p(64), None)
    assert rc == -1 and "aligned" in lib.spec_last_error().decode()


def test_options(lib):
    assert lib.spec_set_option(0, 6) == -1
    assert lib.spec_set_option(0, 5) == 0
    assert lib.spec_set_option(0, 4) == 0
    assert lib.spec_set_option(0, 3) == 0
    assert lib.spec_set_option(99, 0) == -1
    assert lib.spec_set_option(0, 0) == 0
    assert lib.spec_set_option(1, 0) == 0
    # split weight: 0 = each kernel's default, 1..257 = that many tiles + 1
    assert lib.spec_set_option(4, 258) == -1
    assert lib.spec_set_option(4, -1) == -1
    assert lib.spec_set_option(4, 7) == 0
    assert lib.spec_set_option(4, 0) == 0
    # single-pass cluster size: 0 = automatic, 1..8 forced
    assert lib.spec_set_option(5, 9) == -1
    assert lib.spec_set_option(5, -1) == -1
    assert lib.spec_set_option(5, 8) == 0
    assert lib.spec_set_option(5, 0) == 0
    assert lib.spec_set_option(6, 0) == -1


def test_binding_fails_loudly_without_library(tmp_path):
    from speculative_decoding_verification_attn_gb300 import binding
    with pytest.raises(RuntimeError):
        binding._open(str(tmp_path / "missing.so"))


# ---- descriptor form (spec_tensor_t): argument checks precede every CUDA call

def _desc(shape, dtype, data=4096, strides=None):
    from speculative_decoding_verification_attn_gb300 import binding
    d = binding.SpecTensor()
    d.data = data
    d.dtype = dtype
    d.ndim = len(shape)
    st = strides
    if st is None:
        st, acc = [], 1
        for n in reversed(shape):
            st.insert(0, acc)
            acc *= n
    for i, (n, s) in enumerate(zip(shape, st)):
        d.shape[i] = n
        d.stride[i] = s
    return d


def _attn_descs(**over):
    B, k, Hq, Hkv, D, NP, P, MP = 2, 4, 8, 2, 128, 16, 16, 8
    d = dict(q=_desc([B, k, Hq, D], 1), kc=_desc([NP, Hkv, P, D], 1), vc=_desc([NP, Hkv, P, D], 1),
             ks=None, vs=None, bt=_desc([B, MP], 4), ctx=_desc([B], 4),
             out=_desc([B, k, Hq, D], 1), lse=_desc([B, k, Hq], 0), k=k)
    d.update(over)
    return d


def _call_attn(lib, d):
    r = lambda x: None if x is None else ctypes.byref(x)
    return lib.spec_verify_attn_tensors(r(d["q"]), r(d["kc"]), r(d["vc"]), r(d["ks"]), r(d["vs"]),
                                        r(d["bt"]), r(d["ctx"]), d["k"], 0.088, r(d["out"]),
                                        r(d["lse"]), None)


@pytest.mark.parametrize("over,code,needle", [
    (dict(q=_desc([2, 4, 8], 1)), -1, "q: rank"),
    (dict(q=_desc([2, 4, 8, 128], 3)), -1, "q: unsupported element type"),
    (dict(k=5), -1, "q: dimension 1"),
    (dict(kc=_desc([16, 2, 16, 64], 1)), -1, "k_cache: dimension 3"),
    (dict(vc=_desc([16, 2, 16, 128], 0)), -1, "v_cache: unsupported element type"),
    (dict(kc=_desc([16, 2, 16, 128], 3), vc=_desc([16, 2, 16, 128], 3)), -1, "k_scale: null"),
    (dict(bt=_desc([3, 8], 4)), -1, "block_table: dimension 0"),
    (dict(ctx=_desc([2], 0)), -1, "ctx_lens: unsupported element type"),
    (dict(out=_desc([2, 4, 8, 128], 0)), -1, "out: unsupported element type"),
    (dict(lse=_desc([2, 4, 7], 0)), -1, "lse: dimension 2"),
    (dict(q=_desc([2, 4, 8, 128], 1, data=4098)), -1, "q: data must be 16-byte aligned"),
    (dict(q=_desc([2, 4, 8, 128], 1, strides=[4096, 1024, 256, 1])), -2, "dense row-major"),
    (dict(kc=_desc([16, 2, 16, 128], 1, strides=[2, 1, 32, 256])), -2, "dense row-major"),
])
def test_attn_descriptors_rejected(lib, over, code, needle):
    assert _call_attn(lib, _attn_descs(**over)) == code
    assert needle in lib.spec_last_error().decode()


@pytest.mark.parametrize("over,code,needle", [
    (dict(logits=_desc([2, 4, 1000], 1)), -1, "logits: dimension 1"),
    (dict(logits=_desc([2, 5, 1000], 3)), -1, "logits: unsupported element type"),
    (dict(drafts=_desc([2, 3], 4)), -1, "draft_tokens: dimension 1"),
    (dict(acc=_desc([2], 0)), -1, "accepted_len: unsupported element type"),
    (dict(nxt=_desc([3], 4)), -1, "next_token: dimension 0"),
    (dict(logits=_desc([2, 5, 1000], 1, strides=[5000, 1000, 2])), -2, "dense row-major"),
])
def test_accept_descriptors_rejected(lib, over, code, needle):
    d = dict(logits=_desc([2, 5, 1000], 1), drafts=_desc([2, 4], 4), acc=_desc([2], 4),
             nxt=_desc([2], 4))
    d.update(over)
    r = ctypes.byref
    rc = lib.spec_accept_greedy_tensors(r(d["logits"]), r(d["drafts"]), 4, r(d["acc"]),
                                        r(d["nxt"]), None)
    assert rc == code
    assert needle in lib.spec_last_error().decode()


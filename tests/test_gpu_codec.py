"""GPU parity of spec_codec_encode / spec_codec_decode against the oracle.

Encode: the pair count and every defined pair byte equal the oracle's, bit
for bit.  Decode: the oracle's streams decode to the original codes, and a
malformed block decodes as zeros with SPEC_DEVERR_CODEC set while its
neighbours decode correctly.  Shapes cover runs of one (full-range codes),
long runs split at 255 (zeros, tiny spreads, constant rows), head dims 32 to
256 and blocks up to the 16384-byte limit, and an INT8 cache made by the
workload generator.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from speculative_decoding_verification_attn_gb300 import binding
from speculative_decoding_verification_attn_gb300.workload import make_inputs, small_spec

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _lib():
    from speculative_decoding_verification_attn_gb300 import build
    build.build()
    binding.load()
    binding.spec_device_error()  # start from a clear error word


def gpu_encode(codes):
    nblk, P, D = codes.shape
    c = torch.from_numpy(np.ascontiguousarray(codes)).cuda()
    pairs = torch.full((nblk, 2 * P * D), 0xA5, dtype=torch.uint8, device="cuda")
    npairs = torch.full((nblk,), -7, dtype=torch.int32, device="cuda")
    binding.spec_codec_encode(c, pairs, npairs)
    torch.cuda.synchronize()
    return pairs.cpu().numpy(), npairs.cpu().numpy()


def gpu_decode(pairs, npairs, P, D):
    nblk = npairs.shape[0]
    out = torch.full((nblk, P, D), 99, dtype=torch.int8, device="cuda")
    binding.spec_codec_decode(torch.from_numpy(np.ascontiguousarray(pairs)).cuda(),
                              torch.from_numpy(np.ascontiguousarray(npairs)).cuda(), out)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def cases():
    rng = np.random.default_rng(81)
    out = []
    for P, D, spread in [(16, 128, 127), (16, 128, 2), (16, 128, 0), (1, 32, 127), (3, 64, 1),
                         (8, 256, 127), (64, 256, 0), (128, 128, 3), (32, 32, 127)]:
        c = rng.integers(-spread, spread + 1, (11, P, D)).astype(np.int8)
        c[2] = 0
        c[4] = c[4, :, :1]                       # constant rows
        c[6, :, :] = 127
        c[7] = (np.arange(P * D) // 300 % 3).reshape(P, D).astype(np.int8)  # long runs over rows
        out.append(c)
    return out


@pytest.mark.parametrize("idx", range(9))
def test_encode_bit_exact(oracle_mod, idx):
    codes = cases()[idx]
    pairs, npairs = gpu_encode(codes)
    ref_pairs, ref_np = oracle_mod.codec_encode(codes)
    assert np.array_equal(npairs, ref_np)
    for b in range(codes.shape[0]):
        n = 2 * int(ref_np[b])
        assert np.array_equal(pairs[b, :n], ref_pairs[b, :n]), "block %d" % b
    assert binding.spec_device_error() == 0


@pytest.mark.parametrize("idx", range(9))
def test_decode_and_round_trip(oracle_mod, idx):
    codes = cases()[idx]
    _, P, D = codes.shape
    ref_pairs, ref_np = oracle_mod.codec_encode(codes)
    assert np.array_equal(gpu_decode(ref_pairs, ref_np, P, D), codes)
    pairs, npairs = gpu_encode(codes)
    assert np.array_equal(gpu_decode(pairs, npairs, P, D), codes)
    assert binding.spec_device_error() == 0


def test_int8_cache_from_generator(oracle_mod):
    inp = make_inputs(small_spec(kv_dtype="i8", ctx=(1, 300), batch=3, num_q_heads=8,
                                 num_kv_heads=2), seed=82)
    kc = np.ascontiguousarray(inp.k_cache)            # [NP, Hkv, P, D] int8
    codes = kc.reshape(-1, kc.shape[2], kc.shape[3])
    pairs, npairs = gpu_encode(codes)
    ref_pairs, ref_np = oracle_mod.codec_encode(codes)
    assert np.array_equal(npairs, ref_np)
    assert np.array_equal(gpu_decode(pairs, npairs, *codes.shape[1:]), codes)


def test_malformed_block_flagged_and_zeroed(oracle_mod):
    codes = cases()[0][:6]
    _, P, D = codes.shape
    pairs, npairs = oracle_mod.codec_encode(codes)
    pairs = pairs.copy()
    npairs = npairs.copy()
    pairs[1, 0] = 0                     # block 1: a zero length
    npairs[3] = P * D + 5               # block 3: count beyond the block
    pairs[4, 2 * (int(npairs[4]) - 1)] += 1   # block 4: lengths sum past P*D
    out = gpu_decode(pairs, npairs, P, D)
    assert binding.spec_device_error() == binding.SPEC_DEVERR_CODEC
    for b in (1, 3, 4):
        assert np.all(out[b] == 0)
    for b in (0, 2, 5):
        assert np.array_equal(out[b], codes[b])

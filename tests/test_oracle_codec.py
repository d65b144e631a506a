"""Pins for the oracle's delta + run-length page codec (CPU only).

CXL-SpecKV ("Algorithm 2 KV-Cache Compression", output (s, D_RLE(c)); key
observation (5): neighbouring elements of a head vector are correlated, so
delta coding x_i - x_(i-1) compresses further) names the two steps without a
byte format.  The oracle's format: per (page, kv-head) block of P x D INT8
codes, deltas along the head dimension modulo 256 (restarting at each row),
then maximal runs of equal bytes as (length 1..255, value) byte pairs.

Pins: a worked example derived by hand; closed forms for constant, all-zero
and arithmetic-progression rows; the 255 split; format invariants on random
blocks (lengths sum to P*D, runs maximal, round trip exact); malformed
streams rejected.  Each pin was checked to catch a planted slip in the oracle
(delta not restarting at a row, a run cap of 256, a dropped last run,
decoding with a running sum over the whole block).
"""
from __future__ import annotations

import numpy as np
import pytest


def pairs_of(pairs, npairs, blk=0):
    n = int(npairs[blk])
    return [(int(pairs[blk, 2 * j]), int(pairs[blk, 2 * j + 1])) for j in range(n)]


def test_worked_example(oracle_mod):
    # rows [1 1 1 1] and [5 3 3 3]: deltas [1 0 0 0] and [5 -2 0 0]; -2 is byte
    # 254; the stream 1 0 0 0 5 254 0 0 has the runs 1, 0x3, 5, 254, 0x2
    codes = np.array([[[1, 1, 1, 1], [5, 3, 3, 3]]], np.int8)
    pairs, npairs = oracle_mod.codec_encode(codes)
    assert pairs_of(pairs, npairs) == [(1, 1), (3, 0), (1, 5), (1, 254), (2, 0)]
    assert np.array_equal(oracle_mod.codec_decode(pairs, npairs, 2, 4), codes)


@pytest.mark.parametrize("c", [7, -100, 127, -127])
def test_constant_block(oracle_mod, c):
    # every row is [c, 0, ..., 0] after the delta: two pairs per row
    P, D = 16, 128
    codes = np.full((1, P, D), c, np.int8)
    pairs, npairs = oracle_mod.codec_encode(codes)
    assert pairs_of(pairs, npairs) == [(1, c & 255), (D - 1, 0)] * P


def test_zero_block_splits_runs_at_255(oracle_mod):
    P, D = 4, 128   # 512 zero bytes: 255 + 255 + 2
    codes = np.zeros((1, P, D), np.int8)
    pairs, npairs = oracle_mod.codec_encode(codes)
    assert pairs_of(pairs, npairs) == [(255, 0), (255, 0), (2, 0)]
    assert np.array_equal(oracle_mod.codec_decode(pairs, npairs, P, D), codes)


def test_arithmetic_rows(oracle_mod):
    # row r = a_r + d * s_r (mod 256): deltas [a_r, s_r, ..., s_r]
    P, D = 3, 64
    a = [10, 200, 0]
    s = [3, 253, 0]
    codes = np.array([[(a[r] + d * s[r]) % 256 for d in range(D)] for r in range(P)],
                     np.uint8).view(np.int8)[None]
    pairs, npairs = oracle_mod.codec_encode(codes)
    # row 1 ends in 253, so row 2's zeros start a new run
    assert pairs_of(pairs, npairs) == [(1, 10), (63, 3), (1, 200), (63, 253), (64, 0)]


@pytest.mark.parametrize("seed,P,D,spread", [(1, 16, 128, 127), (2, 32, 128, 3), (3, 16, 64, 0),
                                             (4, 8, 256, 1)])
def test_invariants_random(oracle_mod, seed, P, D, spread):
    rng = np.random.default_rng(seed)
    nblk = 12
    # small spreads give long runs (including 255 splits), 127 gives runs of 1
    codes = rng.integers(-spread, spread + 1, (nblk, P, D)).astype(np.int8)
    codes[3] = 0
    codes[5, :, :] = codes[5, :, :1]      # rows constant
    pairs, npairs = oracle_mod.codec_encode(codes)
    n = P * D
    for blk in range(nblk):
        pr = pairs_of(pairs, npairs, blk)
        lens = [l for l, _ in pr]
        assert sum(lens) == n and all(1 <= l <= 255 for l in lens)
        # maximal runs: equal neighbours only after a full 255 run
        for (l0, v0), (_, v1) in zip(pr, pr[1:]):
            assert v0 != v1 or l0 == 255
        assert len(pr) <= n
    assert np.array_equal(oracle_mod.codec_decode(pairs, npairs, P, D), codes)


def test_malformed_streams_rejected(oracle_mod):
    P, D = 2, 4
    codes = np.array([[[1, 1, 1, 1], [5, 3, 3, 3]]], np.int8)
    pairs, npairs = oracle_mod.codec_encode(codes)
    short = pairs.copy()
    short[0, 2] = 2                       # lengths sum to 7
    with pytest.raises(ValueError):
        oracle_mod.codec_decode(short, npairs, P, D)
    zero = pairs.copy()
    zero[0, 0] = 0
    with pytest.raises(ValueError):
        oracle_mod.codec_decode(zero, npairs, P, D)
    with pytest.raises(ValueError):
        oracle_mod.codec_decode(pairs, np.array([P * D + 1], np.int32), P, D)

// Delta + run-length coding of INT8 KV pages.
//
// CXL-SpecKV compresses the cache in two lossless steps after INT8
// quantisation: delta coding of neighbouring elements of a head vector (key
// observation (5), delta_i = x_i - x_(i-1)) and run-length coding ("Algorithm
// 2 KV-Cache Compression", output (s, D_RLE(c))).  The page fixes no byte
// format; this one: a block is the P x D codes of one (page, kv-head),
// row-major; e[r][0] = c[r][0], e[r][d] = c[r][d] - c[r][d-1] (mod 256); the
// block's stream e becomes maximal runs of equal bytes, each stored as the
// byte pair (length 1..255, value), a longer run continuing in the next pair.
// Pairs of block i start at byte 2*P*D*i (the worst case, runs of one), and
// num_pairs[i] counts them.  The fp16 scales are not coded.
//
// Encode: one warp per block, 32 consecutive bytes per step.  A byte starts
// a run where it differs from the previous one; the run's start is a warp
// max-scan; a pair starts at a run start and every 255 bytes after it.  Each
// pair start writes its value and the previous pair's length (its distance
// from the previous start), the last length is written after the block.
//
// Decode: one warp per block.  128 pairs per step, four per lane (one
// 8-byte load): the exclusive warp scan of the lanes' length sums gives each
// run's offset, and each lane writes its runs into the block's staging
// buffer in shared memory; then each row's deltas are summed
// modulo 256 (a warp scan over D/32-byte lane slices) and the codes stored
// with coalesced 4-byte writes.  A malformed block (pair count outside
// [0, P*D], a zero length, lengths not summing to P*D) is written as zeros and
// sets the device error word; nothing outside the block is touched.
#include "common.cuh"

namespace specv {
namespace {

constexpr int kEncWarps = 8;
constexpr int kDecWarps = 4;

__device__ __forceinline__ unsigned lanemask_lt() {
    unsigned m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

__global__ void __launch_bounds__(kEncWarps * 32)
codec_encode_kernel(const uint8_t* __restrict__ codes, int64_t nblk, int P, int D,
                    uint8_t* __restrict__ pairs, int32_t* __restrict__ npairs) {
    const int lane = threadIdx.x & 31;
    const int64_t blk = (int64_t)blockIdx.x * kEncWarps + (threadIdx.x >> 5);
    if (blk >= nblk) return;
    const int n = P * D;  // a multiple of 32 (D is)
    const uint8_t* c = codes + blk * n;
    uint8_t* out = pairs + blk * 2 * (int64_t)n;
    // carries from the previous step: last code, last delta, start of the
    // run in progress, start of the pair in progress, pairs so far
    uint32_t c_prev = 0, e_prev = 0;
    int run_start = 0, pair_start = 0, np = 0;
    for (int i0 = 0; i0 < n; i0 += 32) {
        const int i = i0 + lane;
        const uint32_t ci = c[i];
        uint32_t cl = __shfl_up_sync(0xffffffffu, ci, 1);
        if (lane == 0) cl = c_prev;
        const uint32_t ei = (i % D) ? (ci - cl) & 255u : ci;
        uint32_t el = __shfl_up_sync(0xffffffffu, ei, 1);
        if (lane == 0) el = e_prev;
        const bool new_run = i == 0 || ei != el;
        // start of the run holding byte i: the last run start at or before i
        int rs = new_run ? i : run_start;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, rs, o);
            if (lane >= o) rs = max(rs, v);
        }
        const bool starts = new_run || ((i - rs) % 255 == 0);
        const unsigned sb = __ballot_sync(0xffffffffu, starts);
        if (starts) {
            const int p = np + __popc(sb & lanemask_lt());
            out[2 * p + 1] = (uint8_t)ei;
            // the previous pair ends here: in this step, or the carried one
            const unsigned below = sb & lanemask_lt();
            const int prev_start = below ? i0 + 31 - __clz(below) : pair_start;
            if (p > 0) out[2 * (p - 1)] = (uint8_t)(i - prev_start);
        }
        np += __popc(sb);
        if (sb) pair_start = i0 + 31 - __clz(sb);
        run_start = __shfl_sync(0xffffffffu, rs, 31);
        c_prev = __shfl_sync(0xffffffffu, ci, 31);
        e_prev = __shfl_sync(0xffffffffu, ei, 31);
    }
    if (lane == 0) {
        out[2 * (np - 1)] = (uint8_t)(n - pair_start);
        npairs[blk] = np;
    }
}

__global__ void __launch_bounds__(kDecWarps * 32)
codec_decode_kernel(const uint8_t* __restrict__ pairs, const int32_t* __restrict__ npairs,
                    int64_t nblk, int P, int D, uint8_t* __restrict__ codes, int* dev_err) {
    extern __shared__ uint8_t stage_all[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t blk = (int64_t)blockIdx.x * kDecWarps + warp;
    if (blk >= nblk) return;
    const int n = P * D;
    uint8_t* stage = stage_all + warp * n;
    const uint8_t* in = pairs + blk * 2 * (int64_t)n;
    uint8_t* c = codes + blk * n;
    const int np = __ldg(npairs + blk);
    bool bad = np < 0 || np > n;
    int pos = 0;  // bytes expanded so far
    // four pairs per lane and step (one 8-byte load), 128 pairs per step
    for (int j0 = 0; j0 < (bad ? 0 : np); j0 += 128) {
        const int j = j0 + lane * 4;
        uint32_t len[4] = {0, 0, 0, 0}, val[4] = {0, 0, 0, 0};
        if (j + 4 <= np) {
            const uint2 w = *reinterpret_cast<const uint2*>(in + 2 * j);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const uint32_t pr = (q < 2 ? w.x : w.y) >> (16 * (q & 1));
                len[q] = pr & 255u;
                val[q] = (pr >> 8) & 255u;
            }
        } else {
#pragma unroll
            for (int q = 0; q < 4; ++q)
                if (j + q < np) {
                    len[q] = in[2 * (j + q)];
                    val[q] = in[2 * (j + q) + 1];
                }
        }
        bool zero = false;
#pragma unroll
        for (int q = 0; q < 4; ++q) zero |= j + q < np && len[q] == 0;
        if (__any_sync(0xffffffffu, zero)) bad = true;
        const int tot = (int)(len[0] + len[1] + len[2] + len[3]);
        // exclusive scan of the lanes' totals: this lane's first run offset
        int incl = tot;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += v;
        }
        int start = pos + incl - tot;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            for (int t = 0; t < (int)len[q]; ++t)
                if (start + t < n) stage[start + t] = (uint8_t)val[q];
            start += (int)len[q];
        }
        pos += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (pos != n) bad = true;
    __syncwarp();
    if (bad) {
        for (int i = lane; i < n; i += 32) c[i] = 0;
        if (lane == 0) raise_device_error(dev_err, SPEC_DEVERR_CODEC);
        return;
    }
    // each row: sum of deltas mod 256, lane slices of W = D/32 bytes
    const int W = D / 32;
    for (int r = 0; r < P; ++r) {
        const uint8_t* er = stage + r * D + lane * W;
        uint32_t run = 0, v[8];
#pragma unroll
        for (int t = 0; t < 8; ++t)
            if (t < W) v[t] = (run += er[t]);  // inclusive within the slice
        uint32_t excl = run;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t x = __shfl_up_sync(0xffffffffu, excl, o);
            if (lane >= o) excl += x;
        }
        excl -= run;
        uint8_t* cr = c + r * D + lane * W;
        if (W == 4) {
            uint32_t w = 0;
#pragma unroll
            for (int t = 0; t < 4; ++t) w |= ((v[t] + excl) & 255u) << (8 * t);
            *reinterpret_cast<uint32_t*>(cr) = w;
        } else {
#pragma unroll
            for (int t = 0; t < 8; ++t)
                if (t < W) cr[t] = (uint8_t)(v[t] + excl);
        }
    }
}

}  // namespace

size_t codec_decode_smem(int P, int D) { return (size_t)kDecWarps * P * D; }

cudaError_t launch_codec_encode(const void* codes, int64_t nblk, int P, int D, void* pairs,
                                int32_t* npairs, cudaStream_t stream) {
    if (nblk == 0) return cudaSuccess;
    const int64_t grid = (nblk + kEncWarps - 1) / kEncWarps;
    codec_encode_kernel<<<(unsigned)grid, kEncWarps * 32, 0, stream>>>(
        static_cast<const uint8_t*>(codes), nblk, P, D, static_cast<uint8_t*>(pairs), npairs);
    return cudaGetLastError();
}

cudaError_t launch_codec_decode(const void* pairs, const int32_t* npairs, int64_t nblk, int P,
                                int D, void* codes, int* dev_err, cudaStream_t stream) {
    if (nblk == 0) return cudaSuccess;
    const size_t smem = codec_decode_smem(P, D);
    cudaError_t e = cudaFuncSetAttribute(codec_decode_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const int64_t grid = (nblk + kDecWarps - 1) / kDecWarps;
    codec_decode_kernel<<<(unsigned)grid, kDecWarps * 32, smem, stream>>>(
        static_cast<const uint8_t*>(pairs), npairs, nblk, P, D, static_cast<uint8_t*>(codes),
        dev_err);
    return cudaGetLastError();
}

}  // namespace specv

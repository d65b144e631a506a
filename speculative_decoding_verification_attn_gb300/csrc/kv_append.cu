// Writing the drafts' K/V rows into the paged cache, and the commit.
//
// Append: positions ctx_b .. ctx_b + n - 1 of sequence b receive the rows
// k_new / v_new [B, n, Hkv, D] at page block_table[b][pos / P], slot pos % P.
// An f32 or bf16 cache stores the value (bf16 rounded to nearest even); an
// INT8 cache stores CXL-SpecKV's "Algorithm 2 KV-Cache Compression" per
// (token, kv-head) row: s = fp16(max_d |x_d| / 127), c_d = clamp(rint(x_d /
// s), -127, 127), c = 0 when s = 0 -- each step in fp32 with IEEE division
// and round-half-to-even, so the codes are exactly those of any other
// correct fp32 evaluation.  One warp per (sequence, position, kv-head,
// tensor) row, lanes strided over the head dimension (coalesced); the row
// maximum is a warp reduction.  A position past the block table, or a page
// id outside [0, num_pages), writes nothing and sets the device error word.
//
// Commit: HeteroReason's KV Cache Management Unit advances the validated
// pointer over the accepted drafts ("Accept" mode) and leaves rejected ones
// behind, to be overwritten by the next append ("Rollback"):
// ctx_b += accepted_len_b + extra.
#include "common.cuh"

namespace specv {
namespace {

constexpr int kAppendWarps = 8;

struct AppendArgs {
    const void* k_new;
    const void* v_new;
    int32_t src_dtype;
    void* k_cache;
    void* v_cache;
    uint16_t* k_scale;
    uint16_t* v_scale;
    int32_t cache_dtype;
    const int32_t* block_table;
    const int32_t* ctx_lens;
    int32_t B, n, Hkv, D, P, num_pages, max_pages;
    int* dev_err;
};

__device__ __forceinline__ float load_src(const void* p, int dtype, int64_t i) {
    return dtype == SPEC_DTYPE_F32 ? static_cast<const float*>(p)[i]
                                   : __bfloat162float(static_cast<const __nv_bfloat16*>(p)[i]);
}

__global__ void __launch_bounds__(kAppendWarps * 32) kv_append_kernel(AppendArgs a) {
    const int lane = threadIdx.x & 31;
    const int64_t row = (int64_t)blockIdx.x * kAppendWarps + (threadIdx.x >> 5);
    const int64_t rows = (int64_t)a.B * a.n * a.Hkv * 2;
    if (row >= rows) return;
    const int tensor = (int)(row & 1);
    const int64_t r = row >> 1;  // (b, t, g)
    const int g = (int)(r % a.Hkv);
    const int t = (int)((r / a.Hkv) % a.n);
    const int b = (int)(r / a.Hkv / a.n);
    const int64_t pos = (int64_t)__ldg(a.ctx_lens + b) + t;
    if (pos < 0 || pos / a.P >= a.max_pages) {
        if (lane == 0) raise_device_error(a.dev_err, SPEC_DEVERR_CTX);
        return;
    }
    const int32_t page = __ldg(a.block_table + (int64_t)b * a.max_pages + pos / a.P);
    if (page < 0 || page >= a.num_pages) {
        if (lane == 0) raise_device_error(a.dev_err, SPEC_DEVERR_PAGE);
        return;
    }
    const int64_t src = r * a.D;
    const int64_t dst = (((int64_t)page * a.Hkv + g) * a.P + pos % a.P);
    const void* s_ptr = tensor ? a.v_new : a.k_new;
    void* c_ptr = tensor ? a.v_cache : a.k_cache;
    const int per = a.D / 32;  // head_dim is a multiple of 32, at most 256
    float x[8];
#pragma unroll
    for (int j = 0; j < 8; ++j)
        x[j] = j < per ? load_src(s_ptr, a.src_dtype, src + lane + 32 * j) : 0.f;
    if (a.cache_dtype == SPEC_DTYPE_F32) {
        float* c = static_cast<float*>(c_ptr) + dst * a.D;
#pragma unroll
        for (int j = 0; j < 8; ++j)
            if (j < per) c[lane + 32 * j] = x[j];
    } else if (a.cache_dtype == SPEC_DTYPE_BF16) {
        __nv_bfloat16* c = static_cast<__nv_bfloat16*>(c_ptr) + dst * a.D;
#pragma unroll
        for (int j = 0; j < 8; ++j)
            if (j < per) c[lane + 32 * j] = __float2bfloat16_rn(x[j]);
    } else {
        float amax = 0.f;
#pragma unroll
        for (int j = 0; j < 8; ++j)
            if (j < per) amax = fmaxf(amax, fabsf(x[j]));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        const __half s16 = __float2half_rn(__fdiv_rn(amax, 127.0f));
        const float s = __half2float(s16);
        int8_t* c = static_cast<int8_t*>(c_ptr) + dst * a.D;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            if (j >= per) continue;
            float q = 0.f;
            if (s > 0.f) q = fminf(fmaxf(rintf(__fdiv_rn(x[j], s)), -127.f), 127.f);
            c[lane + 32 * j] = (int8_t)q;
        }
        if (lane == 0) (tensor ? a.v_scale : a.k_scale)[dst] = __half_as_ushort(s16);
    }
}

__global__ void commit_kernel(int32_t* ctx_lens, const int32_t* accepted_len, int B, int extra) {
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b < B) ctx_lens[b] += accepted_len[b] + extra;
}

}  // namespace

cudaError_t launch_kv_append(const void* k_new, const void* v_new, int32_t src_dtype,
                             void* k_cache, void* v_cache, uint16_t* k_scale, uint16_t* v_scale,
                             int32_t cache_dtype, const int32_t* block_table,
                             const int32_t* ctx_lens, int B, int n, int Hkv, int D, int P,
                             int num_pages, int max_pages, int* dev_err, cudaStream_t stream) {
    const int64_t rows = (int64_t)B * n * Hkv * 2;
    if (rows == 0) return cudaSuccess;
    AppendArgs a{k_new, v_new, src_dtype, k_cache, v_cache, k_scale, v_scale, cache_dtype,
                 block_table, ctx_lens, B, n, Hkv, D, P, num_pages, max_pages, dev_err};
    const int64_t blocks = (rows + kAppendWarps - 1) / kAppendWarps;
    kv_append_kernel<<<(unsigned)blocks, kAppendWarps * 32, 0, stream>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_commit(int32_t* ctx_lens, const int32_t* accepted_len, int B, int extra,
                          cudaStream_t stream) {
    if (B == 0) return cudaSuccess;
    commit_kernel<<<(B + 255) / 256, 256, 0, stream>>>(ctx_lens, accepted_len, B, extra);
    return cudaGetLastError();
}

}  // namespace specv

// Verification attention for short contexts in one launch (CUDA cores).
//
// What it computes is the multi-query causal attention of the k draft
// queries over the paged cache ("Decoding Speculative Decoding from First
// Principles", "Parallelizing method 2: sequence parallel"): query i of
// sequence b sees keys 0 .. ctx_b + i (or the drafts its tree row names).
//
// When every sequence's keys fit in shared memory, a call is latency-bound:
// the chunked SIMT kernel walks 16-key tiles with a dependent page lookup per
// tile and merges its chunks in a second launch.  Here one CTA takes a whole
// (sequence, kv-head, query-row group): one round trip loads the block-table
// entries of the segment, its query rows and its context length; the next
// loads every K and V row of the segment (all loads issued before any is
// used), widened to fp32 in shared memory; then the scores of all rows and
// keys, an exact two-pass softmax per row (max, then the sum of
// exponentials) and P V, and the output and lse are written directly.
#include <math.h>

#include "common.cuh"

namespace specv {
namespace {

constexpr int kThreads = 512;
constexpr int kPad = 4;  // fp32 row padding of K: row stride = D + 4 floats
constexpr size_t kSmallAttnSmem = 200 * 1024;

__host__ __device__ inline int small_rows_per_group(int R) { return R < 64 ? R : 64; }
__host__ __device__ inline size_t round4(size_t n) { return (n + 3) & ~size_t(3); }

// Partial sums of P V when the key range is split over several parts: at
// most 4 rows x kThreads columns (see the P V loop).
constexpr int kRedFloats = 4 * kThreads;

// Shared memory of one CTA, in floats: K [Lcap][D + 4], V [Lcap][D],
// S [RG][Lcap] (rounded up to 4 floats), Q [RG][D], the P V partial sums,
// 1/l [RG]; then the Lcap/P page ids (ints).  Every float4-read array
// starts on 16 bytes.
__host__ __device__ inline size_t small_smem_bytes(int Lcap, int D, int RG, int P) {
    const size_t floats = (size_t)Lcap * (D + kPad) + (size_t)Lcap * D +
                          round4((size_t)RG * Lcap) + (size_t)RG * D + kRedFloats + RG;
    return floats * 4 + ((size_t)Lcap / P + 2) * 4;  // Lcap / P = max_pages
}

template <typename TKV>
__device__ __forceinline__ void widen16(const uint4 raw, float* dst, float s) {
    if constexpr (sizeof(TKV) == 4) {
        const float* f = reinterpret_cast<const float*>(&raw);
        reinterpret_cast<float4*>(dst)[0] = make_float4(f[0], f[1], f[2], f[3]);
    } else if constexpr (sizeof(TKV) == 2) {
        const __nv_bfloat16* h = reinterpret_cast<const __nv_bfloat16*>(&raw);
#pragma unroll
        for (int u = 0; u < 8; u += 4)
            reinterpret_cast<float4*>(dst)[u / 4] =
                make_float4(__bfloat162float(h[u]), __bfloat162float(h[u + 1]),
                            __bfloat162float(h[u + 2]), __bfloat162float(h[u + 3]));
    } else {
        const int8_t* c = reinterpret_cast<const int8_t*>(&raw);
#pragma unroll
        for (int u = 0; u < 16; u += 4)
            reinterpret_cast<float4*>(dst)[u / 4] =
                make_float4((float)c[u] * s, (float)c[u + 1] * s, (float)c[u + 2] * s,
                            (float)c[u + 3] * s);
    }
}

template <typename TQ, typename TKV>
__global__ void __launch_bounds__(kThreads)
attn_small_kernel(AttnArgs a, int Lcap, int RG, int row_groups) {
    extern __shared__ float4 smem4[];
    float* sm = reinterpret_cast<float*>(smem4);
    grid_dep_launch_dependents();
    grid_dep_wait();
    const int D = a.D, G = a.Hq / a.Hkv, R = a.k * G, P = a.P;
    const int rg = blockIdx.x % row_groups, seg = blockIdx.x / row_groups;
    const int kvh = seg % a.Hkv, b = seg / a.Hkv;
    const int r0 = rg * RG, nr = min(RG, R - r0);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int KS = D + kPad;
    float* Ks = sm;                          // [Lcap][D + 4]
    float* Vs = Ks + (size_t)Lcap * KS;      // [Lcap][D]
    float* S = Vs + (size_t)Lcap * D;        // [RG][Lcap]
    float* Qs = S + round4((size_t)RG * Lcap);  // [RG][D]
    float* red = Qs + (size_t)RG * D;        // [kRedFloats]
    float* inv_l = red + kRedFloats;         // [RG]
    int* pages = reinterpret_cast<int*>(inv_l + RG);

    // ---- round trip 1, all loads independent: the context length, every
    // block-table entry of the sequence (the used ones are checked below), the
    // query rows.  Lcap = max_pages * P keys: a context past Lcap - k is
    // clamped and flagged.
    int ctx = __ldg(a.ctx_lens + b);
    for (int p = tid; p < a.max_pages; p += kThreads)
        pages[p] = __ldg(a.block_table + (int64_t)b * a.max_pages + p);
    const TQ* q = static_cast<const TQ*>(a.q);
    for (int e = tid; e < nr * D; e += kThreads) {
        const int r = e / D, d = e % D, row = r0 + r;
        Qs[r * D + d] =
            Elem<TQ>::to_f32(q[(((int64_t)b * a.k + row / G) * a.Hq + kvh * G + row % G) * D + d]);
    }
    const int cap = Lcap - a.k;
    if (ctx < 0 || ctx > cap) {
        if (tid == 0) raise_device_error(a.dev_err, SPEC_DEVERR_CTX);
        ctx = ctx < 0 ? 0 : (cap < 0 ? 0 : cap);
    }
    const int L = ctx + a.k;
    __syncthreads();
    for (int p = tid; p < (L + P - 1) / P; p += kThreads) {
        const int id = pages[p];
        if (id < 0 || id >= a.num_pages) {
            raise_device_error(a.dev_err, SPEC_DEVERR_PAGE);
            pages[p] = 0;
        }
    }
    __syncthreads();

    // ---- round trip 2: every K and V row of the segment, 16 bytes per load,
    // all of a thread's loads issued before any is widened
    constexpr int E = 16 / (int)sizeof(TKV);  // elements per 16-byte chunk
    const int cpr = D / E;                     // chunks per row
    const int nch = L * cpr;
    constexpr int U = 8;  // 8 x 512 chunks: the tiny workloads' K and V in one round
    if constexpr (sizeof(TKV) == 4) {
        // fp32 cache: asynchronous copies straight into place, all in flight at once
        for (int c = tid; c < nch; c += kThreads) {
            const int j = c / cpr, ch = c % cpr;
            const int64_t row = ((int64_t)pages[j / P] * a.Hkv + kvh) * P + j % P;
            cp_async_16_cg(Ks + (size_t)j * KS + ch * E,
                           static_cast<const float*>(a.k_cache) + row * D + ch * E);
            cp_async_16_cg(Vs + (size_t)j * D + ch * E,
                           static_cast<const float*>(a.v_cache) + row * D + ch * E);
        }
        cp_async_commit();
        cp_async_wait<0>();
    } else
    for (int c0 = tid; c0 < nch; c0 += U * kThreads) {
        uint4 kr[U], vr[U];
        float ks[U], vs[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int c = c0 + u * kThreads;
            kr[u] = vr[u] = make_uint4(0, 0, 0, 0);
            ks[u] = vs[u] = 1.f;
            if (c < nch) {
                const int j = c / cpr, ch = c % cpr;
                const int64_t row = ((int64_t)pages[j / P] * a.Hkv + kvh) * P + j % P;
                kr[u] = __ldg(reinterpret_cast<const uint4*>(
                    static_cast<const TKV*>(a.k_cache) + row * D) + ch);
                vr[u] = __ldg(reinterpret_cast<const uint4*>(
                    static_cast<const TKV*>(a.v_cache) + row * D) + ch);
                if constexpr (sizeof(TKV) == 1) {
                    ks[u] = __half2float(__ushort_as_half(__ldg(a.k_scale + row)));
                    vs[u] = __half2float(__ushort_as_half(__ldg(a.v_scale + row)));
                }
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int c = c0 + u * kThreads;
            if (c < nch) {
                const int j = c / cpr, ch = c % cpr;
                widen16<TKV>(kr[u], Ks + (size_t)j * KS + ch * E, ks[u]);
                widen16<TKV>(vr[u], Vs + (size_t)j * D + ch * E, vs[u]);
            }
        }
    }
    __syncthreads();

    // ---- scores of every (row, key); -inf where the key is invisible.  A
    // thread takes one key and up to RB query rows, so each K row is read
    // from shared memory once per RB rows (the query rows are broadcasts:
    // the lanes of a warp share them)
    constexpr int RB = 4;
    const int nrb = (nr + RB - 1) / RB;
    for (int e = tid; e < nrb * L; e += kThreads) {
        const int rb = e / L, j = e % L;
        const float4* kv = reinterpret_cast<const float4*>(Ks + (size_t)j * KS);
        float acc[RB] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
        for (int d4 = 0; d4 < D / 4; ++d4) {
            const float4 y = kv[d4];
#pragma unroll
            for (int u = 0; u < RB; ++u) {
                const int r = min(rb * RB + u, nr - 1);
                const float4 x = reinterpret_cast<const float4*>(Qs + r * D)[d4];
                acc[u] = fmaf(x.x, y.x, acc[u]);
                acc[u] = fmaf(x.y, y.y, acc[u]);
                acc[u] = fmaf(x.z, y.z, acc[u]);
                acc[u] = fmaf(x.w, y.w, acc[u]);
            }
        }
#pragma unroll
        for (int u = 0; u < RB; ++u) {
            const int r = rb * RB + u;
            if (r < nr) {
                const int i = (r0 + r) / G;
                const bool vis = j < ctx || ((draft_bits(a, b, i) >> (j - ctx)) & 1ull);
                S[(size_t)r * Lcap + j] = vis ? acc[u] * a.scale : -INFINITY;
            }
        }
    }
    __syncthreads();

    // ---- exact softmax per row (a warp per row): max, then sum of exp
    float* lse_out = a.lse;
    for (int r = warp; r < nr; r += kThreads / 32) {
        float* sr = S + (size_t)r * Lcap;
        float m = -INFINITY;
        for (int j = lane; j < L; j += 32) m = fmaxf(m, sr[j]);
        m = warp_max(m);
        float sum = 0.f;
        for (int j = lane; j < L; j += 32) {
            const float p = sr[j] == -INFINITY ? 0.f : expf(sr[j] - m);
            sr[j] = p;
            sum += p;
        }
        sum = warp_sum(sum);
        if (lane == 0) {
            inv_l[r] = sum > 0.f ? 1.f / sum : 0.f;
            if (lse_out) {
                const int row = r0 + r;
                lse_out[((int64_t)b * a.k + row / G) * a.Hq + kvh * G + row % G] =
                    sum > 0.f ? m + logf(sum) : -INFINITY;
            }
        }
    }
    __syncthreads();

    // ---- out = P V / l.  A thread takes one head-dim column, RB query rows
    // and the keys of one of SF parts (SF > 1 when there are too few columns
    // to fill the CTA); the lanes of a warp hold consecutive columns of one
    // part, so V reads are conflict-free and P reads are broadcasts.  Split
    // parts meet in shared memory (SF * ncol <= kThreads columns of RB rows).
    TQ* out = static_cast<TQ*>(a.out);
    const int ncol = nrb * D;  // (row block, column) pairs
    int SF = 1;
    while (SF < 16 && ncol * SF * 2 <= kThreads) SF *= 2;
    const int klen = (L + SF - 1) / SF;
    for (int e0 = 0; e0 < ncol * SF; e0 += kThreads) {
        const int e = e0 + tid;
        if (e >= ncol * SF) continue;
        const int part = e / ncol, o = e % ncol, rb = o / D, d = o % D;
        const int k0 = part * klen, k1 = min(L, k0 + klen);
        float acc[RB] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
        for (int j = k0; j < k1; ++j) {
            const float v = Vs[(size_t)j * D + d];
#pragma unroll
            for (int u = 0; u < RB; ++u)
                acc[u] = fmaf(S[(size_t)min(rb * RB + u, nr - 1) * Lcap + j], v, acc[u]);
        }
#pragma unroll
        for (int u = 0; u < RB; ++u) {
            const int r = rb * RB + u;
            if (SF > 1) {
                red[(size_t)(part * ncol + o) * RB + u] = acc[u];
            } else if (r < nr) {
                const int row = r0 + r;
                out[(((int64_t)b * a.k + row / G) * a.Hq + kvh * G + row % G) * D + d] =
                    Elem<TQ>::from_f32(acc[u] * inv_l[r]);
            }
        }
    }
    if (SF > 1) {
        __syncthreads();
        for (int e = tid; e < nr * D; e += kThreads) {
            const int r = e / D, d = e % D, row = r0 + r;
            const int o = (r / RB) * D + d;
            float acc = 0.f;
            for (int part = 0; part < SF; ++part) acc += red[(size_t)(part * ncol + o) * RB + r % RB];
            out[(((int64_t)b * a.k + row / G) * a.Hq + kvh * G + row % G) * D + d] =
                Elem<TQ>::from_f32(acc * inv_l[r]);
        }
    }
}

template <typename TQ, typename TKV>
cudaError_t launch_typed(const AttnArgs& a, int Lcap, cudaStream_t stream) {
    const int R = a.k * (a.Hq / a.Hkv), RG = small_rows_per_group(R);
    const int row_groups = (R + RG - 1) / RG;
    const size_t smem = small_smem_bytes(Lcap, a.D, RG, a.P);
    auto kern = attn_small_kernel<TQ, TKV>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    const int64_t blocks = (int64_t)a.B * a.Hkv * row_groups;
    return launch_dependent(kern, dim3((unsigned)blocks), dim3(kThreads), smem, stream, a, Lcap, RG,
                            row_groups);
}

}  // namespace

// The longest context (keys, drafts included) the single-pass kernel holds,
// or 0 when it does not apply: every key a sequence can have -- the whole
// block table -- must fit the shared-memory plan.
int small_attn_max_keys(const AttnArgs& a) {
    const int R = a.k * (a.Hq / a.Hkv), RG = small_rows_per_group(R);
    const int64_t Lcap = (int64_t)a.max_pages * a.P;
    if (Lcap < 1 || Lcap > 4096) return 0;
    if ((int64_t)a.B * a.Hkv * ((R + RG - 1) / RG) >= (1LL << 31)) return 0;
    if (small_smem_bytes((int)Lcap, a.D, RG, a.P) > kSmallAttnSmem) return 0;
    return (int)Lcap;
}

cudaError_t launch_attn_small(const AttnArgs& a, cudaStream_t stream) {
    const int Lcap = small_attn_max_keys(a);
    if (Lcap == 0) return cudaErrorInvalidValue;
    const bool q32 = a.q_dtype == SPEC_DTYPE_F32;
    switch (a.kv_dtype) {
    case SPEC_DTYPE_F32:
        return q32 ? launch_typed<float, float>(a, Lcap, stream)
                   : launch_typed<__nv_bfloat16, float>(a, Lcap, stream);
    case SPEC_DTYPE_BF16:
        return q32 ? launch_typed<float, __nv_bfloat16>(a, Lcap, stream)
                   : launch_typed<__nv_bfloat16, __nv_bfloat16>(a, Lcap, stream);
    case SPEC_DTYPE_I8:
        return q32 ? launch_typed<float, int8_t>(a, Lcap, stream)
                   : launch_typed<__nv_bfloat16, int8_t>(a, Lcap, stream);
    default:
        return cudaErrorInvalidValue;
    }
}

}  // namespace specv

// Verification attention on the CUDA cores (SIMT): every dtype and shape the
// ABI accepts.  It runs the fp32 workload (where 1e-5 accuracy rules out
// reduced-precision tensor-core inputs) and every shape the tensor-core
// kernel does not cover, and serves as an independent GPU cross-check of it.
//
// What it computes is multi-query causal attention of the k draft queries
// over the paged cache ("Decoding Speculative Decoding from First
// Principles", "Parallelizing method 2: sequence parallel"): query i of
// sequence b sees keys 0 .. ctx_b + i.  Work split: one CTA per (sequence,
// kv-head, query-row group, key chunk).  All k*G query rows of a kv-head
// share every K/V row the CTA stages in shared memory, so the cache is read
// once per (sequence, kv-head).  Chunks produce (O/l, lse) partials that the
// combine kernel merges with log-sum-exp weights (split-KV).
#include <math.h>

#include "common.cuh"

namespace specv {
namespace {

constexpr int kThreads = 128;
constexpr int kKeyTile = 16;           // keys staged per iteration
constexpr int kRowElems = 2048;        // query rows x head_dim per CTA
constexpr int kMaxPerThread = kRowElems / kThreads;

struct SeqGeom {
    int ctx, L;  // cached context (clamped) and total keys
};

__device__ __forceinline__ SeqGeom seq_geom(const AttnArgs& a, int b) {
    int ctx = a.ctx_lens[b];
    const int64_t cap = (int64_t)a.max_pages * a.P - a.k;
    if (ctx < 0 || (int64_t)ctx > cap) {
        raise_device_error(a.dev_err, SPEC_DEVERR_CTX);
        ctx = ctx < 0 ? 0 : (int)(cap < 0 ? 0 : cap);
    }
    return {ctx, ctx + a.k};
}

__device__ __forceinline__ int64_t cache_row(const AttnArgs& a, int b, int kvh, int j) {
    int page = a.block_table[(int64_t)b * a.max_pages + j / a.P];
    if (page < 0 || page >= a.num_pages) {
        raise_device_error(a.dev_err, SPEC_DEVERR_PAGE);
        page = 0;
    }
    return ((int64_t)page * a.Hkv + kvh) * a.P + (j % a.P);
}

template <typename TKV>
__device__ __forceinline__ float load_kv(const AttnArgs& a, const void* cache, const uint16_t* sc,
                                         int64_t row, int d) {
    float x = Elem<TKV>::to_f32(static_cast<const TKV*>(cache)[row * a.D + d]);
    if constexpr (sizeof(TKV) == 1) x *= __half2float(__ushort_as_half(sc[row]));
    return x;
}

template <typename TQ, typename TKV>
__global__ void __launch_bounds__(kThreads)
attn_simt_kernel(AttnArgs a, SimtPlan p, float* __restrict__ part_o, float* __restrict__ part_lse) {
    extern __shared__ float sm[];
    grid_dep_launch_dependents();
    grid_dep_wait();
    const int D = a.D, G = a.Hq / a.Hkv, R = a.k * G, RG = p.rows_per_group;
    const int chunk_id = blockIdx.x;
    const int rg = blockIdx.y % p.row_groups;
    const int seg = blockIdx.y / p.row_groups;
    const int kvh = seg % a.Hkv, b = seg / a.Hkv;
    const SeqGeom sg = seq_geom(a, b);
    const int n_chunks = (sg.L + p.chunk - 1) / p.chunk;
    if (chunk_id >= n_chunks) return;
    const int j0 = chunk_id * p.chunk, j1 = min(sg.L, j0 + p.chunk);
    const int r0 = rg * RG, nr = min(RG, R - r0);
    if (nr <= 0) return;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    float* Qs = sm;                       // [RG][D]
    float* Ks = Qs + RG * D;              // [kKeyTile][D+1]
    float* Vs = Ks + kKeyTile * (D + 1);  // [kKeyTile][D]
    float* Ps = Vs + kKeyTile * D;        // [RG][kKeyTile]
    float* m_s = Ps + RG * kKeyTile;      // [RG] running max
    float* l_s = m_s + RG;                // [RG] running sum
    float* al_s = l_s + RG;               // [RG] rescale factor of this step

    const TQ* q = static_cast<const TQ*>(a.q);
    for (int e = tid; e < nr * D; e += kThreads) {
        const int r = e / D, d = e % D, row = r0 + r, i = row / G, g = row % G;
        Qs[r * D + d] = Elem<TQ>::to_f32(q[(((int64_t)b * a.k + i) * a.Hq + kvh * G + g) * D + d]);
    }
    for (int r = tid; r < nr; r += kThreads) {
        m_s[r] = -INFINITY;
        l_s[r] = 0.f;
    }
    float o[kMaxPerThread];
#pragma unroll
    for (int u = 0; u < kMaxPerThread; ++u) o[u] = 0.f;
    __syncthreads();

    for (int jt = j0; jt < j1; jt += kKeyTile) {
        for (int e = tid; e < kKeyTile * D; e += kThreads) {
            const int jj = e / D, d = e % D, j = jt + jj;
            float kx = 0.f, vx = 0.f;
            if (j < j1) {
                const int64_t row = cache_row(a, b, kvh, j);
                kx = load_kv<TKV>(a, a.k_cache, a.k_scale, row, d);
                vx = load_kv<TKV>(a, a.v_cache, a.v_scale, row, d);
            }
            Ks[jj * (D + 1) + d] = kx;
            Vs[jj * D + d] = vx;
        }
        __syncthreads();
        for (int e = tid; e < nr * kKeyTile; e += kThreads) {
            const int r = e / kKeyTile, jj = e % kKeyTile, j = jt + jj;
            const int i = (r0 + r) / G;
            float s = -INFINITY;
            // query i sees the context and the drafts of its row's bits
            // (causal chain: keys <= ctx + i)
            if (j < j1 && (j < sg.ctx || ((draft_bits(a, b, i) >> (j - sg.ctx)) & 1ull))) {
                float dot = 0.f;
                for (int d = 0; d < D; ++d) dot = fmaf(Qs[r * D + d], Ks[jj * (D + 1) + d], dot);
                s = dot * a.scale;
            }
            Ps[r * kKeyTile + jj] = s;
        }
        __syncthreads();
        for (int r = warp; r < nr; r += kThreads / 32) {
            const float s = lane < kKeyTile ? Ps[r * kKeyTile + lane] : -INFINITY;
            const float m_old = m_s[r];
            const float m_new = fmaxf(m_old, warp_max(s));
            const float pr = (m_new == -INFINITY) ? 0.f : expf(s - m_new);
            const float alpha = (m_new == -INFINITY) ? 1.f : expf(m_old - m_new);
            const float psum = warp_sum(pr);
            if (lane < kKeyTile) Ps[r * kKeyTile + lane] = pr;
            if (lane == 0) {
                m_s[r] = m_new;
                l_s[r] = l_s[r] * alpha + psum;
                al_s[r] = alpha;
            }
        }
        __syncthreads();
#pragma unroll
        for (int u = 0; u < kMaxPerThread; ++u) {
            const int e = tid + u * kThreads;
            if (e < nr * D) {
                const int r = e / D, d = e % D;
                float acc = o[u] * al_s[r];
#pragma unroll
                for (int jj = 0; jj < kKeyTile; ++jj)
                    acc = fmaf(Ps[r * kKeyTile + jj], Vs[jj * D + d], acc);
                o[u] = acc;
            }
        }
        __syncthreads();
    }

    TQ* out = static_cast<TQ*>(a.out);
#pragma unroll
    for (int u = 0; u < kMaxPerThread; ++u) {
        const int e = tid + u * kThreads;
        if (e >= nr * D) continue;
        const int r = e / D, d = e % D, row = r0 + r;
        const float l = l_s[r];
        const float val = l > 0.f ? o[u] / l : 0.f;
        const float lse = l > 0.f ? m_s[r] + logf(l) : -INFINITY;
        if (n_chunks == 1) {
            const int i = row / G, h = kvh * G + row % G;
            const int64_t orow = ((int64_t)b * a.k + i) * a.Hq + h;
            out[orow * D + d] = Elem<TQ>::from_f32(val);
            if (d == 0 && a.lse) a.lse[orow] = lse;
        } else {
            const int64_t pi = ((int64_t)seg * p.max_chunks + chunk_id) * R + row;
            part_o[pi * D + d] = val;
            if (d == 0) part_lse[pi] = lse;
        }
    }
}

// Merge the chunk partials of every split (sequence, kv-head): one warp per
// query row, lse_tot = ln sum_c exp(lse_c), out = sum_c exp(lse_c - lse_tot) O_c.
template <typename TQ>
__global__ void __launch_bounds__(256)
combine_simt_kernel(AttnArgs a, SimtPlan p, const float* __restrict__ part_o,
                    const float* __restrict__ part_lse) {
    grid_dep_launch_dependents();
    grid_dep_wait();
    const int seg = blockIdx.x, kvh = seg % a.Hkv, b = seg / a.Hkv;
    const int G = a.Hq / a.Hkv, R = a.k * G, D = a.D;
    const int row = blockIdx.y * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    if (row >= R) return;
    const SeqGeom sg = seq_geom(a, b);
    const int n = (sg.L + p.chunk - 1) / p.chunk;
    if (n <= 1) return;
    const int64_t base = (int64_t)seg * p.max_chunks * R + row;
    float m = -INFINITY;
    for (int c = lane; c < n; c += 32) m = fmaxf(m, part_lse[base + (int64_t)c * R]);
    m = warp_max(m);
    float tot = 0.f;
    for (int c = lane; c < n; c += 32) tot += expf(part_lse[base + (int64_t)c * R] - m);
    tot = warp_sum(tot);
    const float lse_tot = m + logf(tot);
    const int i = row / G, h = kvh * G + row % G;
    const int64_t orow = ((int64_t)b * a.k + i) * a.Hq + h;
    TQ* out = static_cast<TQ*>(a.out);
    for (int d = lane; d < D; d += 32) {
        float acc = 0.f;
        for (int c = 0; c < n; ++c) {
            const int64_t pi = base + (int64_t)c * R;
            const float w = expf(part_lse[pi] - lse_tot);
            acc = fmaf(w, part_o[pi * D + d], acc);
        }
        out[orow * D + d] = Elem<TQ>::from_f32(acc);
    }
    if (lane == 0 && a.lse) a.lse[orow] = lse_tot;
}

size_t smem_bytes(const AttnArgs& a, const SimtPlan& p) {
    const int RG = p.rows_per_group, D = a.D;
    return sizeof(float) *
           ((size_t)RG * D + kKeyTile * (D + 1) + kKeyTile * D + RG * kKeyTile + 3 * RG);
}

template <typename TQ, typename TKV>
cudaError_t launch_typed(const AttnArgs& a, const SimtPlan& p, float* part_o, float* part_lse,
                         cudaStream_t stream) {
    const size_t smem = smem_bytes(a, p);
    auto kern = attn_simt_kernel<TQ, TKV>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid(p.max_chunks, a.B * a.Hkv * p.row_groups);
    e = launch_dependent(kern, grid, dim3(kThreads), smem, stream, a, p, part_o, part_lse);
    if (e != cudaSuccess || p.max_chunks <= 1) return e;
    const int R = a.k * (a.Hq / a.Hkv);
    dim3 cgrid(a.B * a.Hkv, (R + 7) / 8);
    return launch_dependent(combine_simt_kernel<TQ>, cgrid, dim3(256), 0, stream, a, p,
                            static_cast<const float*>(part_o), static_cast<const float*>(part_lse));
}

}  // namespace

SimtPlan simt_plan(const AttnArgs& a, int num_sms, int forced_chunk) {
    SimtPlan p;
    const int R = a.k * (a.Hq / a.Hkv);
    p.rows_per_group = kRowElems / a.D;
    if (p.rows_per_group > R) p.rows_per_group = R;
    p.row_groups = (R + p.rows_per_group - 1) / p.rows_per_group;
    const int64_t max_L = (int64_t)a.max_pages * a.P;
    int64_t chunk;
    if (forced_chunk > 0) {
        chunk = forced_chunk;
    } else {
        const int64_t groups = (int64_t)a.B * a.Hkv * p.row_groups;
        int64_t want = (4LL * num_sms + groups - 1) / (groups > 0 ? groups : 1);
        if (want < 1) want = 1;
        chunk = (max_L + want - 1) / want;
    }
    chunk = ((chunk + kKeyTile - 1) / kKeyTile) * kKeyTile;
    if (chunk < kKeyTile) chunk = kKeyTile;
    if (chunk > max_L) chunk = ((max_L + kKeyTile - 1) / kKeyTile) * kKeyTile;
    if (chunk < kKeyTile) chunk = kKeyTile;
    p.chunk = (int32_t)chunk;
    p.max_chunks = (int32_t)((max_L + chunk - 1) / chunk);
    if (p.max_chunks < 1) p.max_chunks = 1;
    return p;
}

size_t simt_workspace_bytes(const AttnArgs& a, const SimtPlan& p) {
    if (p.max_chunks <= 1) return 0;
    const int64_t R = (int64_t)a.k * (a.Hq / a.Hkv);
    const int64_t rows = (int64_t)a.B * a.Hkv * p.max_chunks * R;
    return (size_t)rows * (a.D + 1) * sizeof(float) + 256;
}

cudaError_t launch_attn_simt(const AttnArgs& a, const SimtPlan& p, void* workspace,
                             cudaStream_t stream) {
    const int64_t R = (int64_t)a.k * (a.Hq / a.Hkv);
    const int64_t rows = (int64_t)a.B * a.Hkv * p.max_chunks * R;
    float* part_o = static_cast<float*>(workspace);
    float* part_lse = part_o ? part_o + rows * a.D : nullptr;
    const bool q32 = a.q_dtype == SPEC_DTYPE_F32;
    switch (a.kv_dtype) {
    case SPEC_DTYPE_F32:
        return q32 ? launch_typed<float, float>(a, p, part_o, part_lse, stream)
                   : launch_typed<__nv_bfloat16, float>(a, p, part_o, part_lse, stream);
    case SPEC_DTYPE_BF16:
        return q32 ? launch_typed<float, __nv_bfloat16>(a, p, part_o, part_lse, stream)
                   : launch_typed<__nv_bfloat16, __nv_bfloat16>(a, p, part_o, part_lse, stream);
    case SPEC_DTYPE_I8:
        return q32 ? launch_typed<float, int8_t>(a, p, part_o, part_lse, stream)
                   : launch_typed<__nv_bfloat16, int8_t>(a, p, part_o, part_lse, stream);
    default:
        return cudaErrorInvalidValue;
    }
}

}  // namespace specv

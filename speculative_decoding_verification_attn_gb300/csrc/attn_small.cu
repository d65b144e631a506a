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
//
// When the call has few such units and the GPU many SMs, a unit's keys are
// split over the CTAs of a thread-block cluster: each CTA runs the same steps
// on its share of the keys and keeps its rows' (max, sum, unnormalised P V)
// in shared memory; after a cluster barrier the CTAs merge the shares through
// distributed shared memory (the usual rescaling by exp(m_c - max m)), so the
// call still takes one launch and no global scratch.
#include <math.h>

#include "common.cuh"

namespace specv {
namespace {

constexpr int kThreads = 512;
constexpr int kPad = 4;  // fp32 row padding of K: row stride = D + 4 floats
constexpr size_t kSmallAttnSmem = 200 * 1024;
constexpr int kMaxSmallCluster = 8;  // portable cluster size

__host__ __device__ inline int small_rows_per_group(int R) { return R < 64 ? R : 64; }
__host__ __device__ inline size_t round4(size_t n) { return (n + 3) & ~size_t(3); }

// Partial sums of P V when the key range is split over several parts: at
// most 4 rows x kThreads columns (see the P V loop).
constexpr int kRedFloats = 4 * kThreads;

// Shared memory of one CTA, in floats: K [Lc][D + 4], V [Lc][D], S [RG][Lc]
// (rounded up to 4 floats), Q [RG][D] (later the CTA's unnormalised P V in
// the cluster form), the P V partial sums, per-row l (or 1/l) and max [RG];
// then the sequence's max_pages page ids (ints).  Lc = the keys one CTA
// holds.  Every float4-read array starts on 16 bytes.
__host__ __device__ inline size_t small_smem_bytes(int Lc, int D, int RG, int max_pages) {
    const size_t floats = (size_t)Lc * (D + kPad) + (size_t)Lc * D + round4((size_t)RG * Lc) +
                          (size_t)RG * D + kRedFloats + 2 * (size_t)RG;
    return floats * 4 + ((size_t)max_pages + 2) * 4;
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
attn_small_kernel(AttnArgs a, int Lcap, int RG, int row_groups, int csize) {
    extern __shared__ float4 smem4[];
    float* sm = reinterpret_cast<float*>(smem4);
    grid_dep_launch_dependents();
    grid_dep_wait();
    const int D = a.D, G = a.Hq / a.Hkv, R = a.k * G, P = a.P;
    // csize CTAs (a cluster of that size, or 1) per (sequence, kv-head, row group)
    const int crank = csize > 1 ? (int)cluster_ctarank() : 0;
    const int unit = blockIdx.x / csize;
    const int rg = unit % row_groups, seg = unit / row_groups;
    const int kvh = seg % a.Hkv, b = seg / a.Hkv;
    const int r0 = rg * RG, nr = min(RG, R - r0);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int KS = D + kPad;
    const int Lc = (Lcap + csize - 1) / csize;  // key rows this CTA holds
    float* Ks = sm;                          // [Lc][D + 4]
    float* Vs = Ks + (size_t)Lc * KS;        // [Lc][D]
    float* S = Vs + (size_t)Lc * D;          // [RG][Lc]
    float* Qs = S + round4((size_t)RG * Lc); // [RG][D]; the CTA's P V share in the cluster form
    float* red = Qs + (size_t)RG * D;        // [kRedFloats]
    float* rl = red + kRedFloats;            // [RG] 1/l (one CTA) or l (cluster)
    float* rm = rl + RG;                     // [RG] row max (cluster)
    int* pages = reinterpret_cast<int*>(rm + RG);

    // ---- round trip 1, all loads independent: the context length, every
    // block-table entry of the sequence (those of this CTA's keys are checked below), the
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
    // this CTA's keys [kb, kb + nk): an even share of the segment's L
    const int Ls = (L + csize - 1) / csize;
    const int kb = min(L, crank * Ls), nk = min(L, kb + Ls) - kb;
    __syncthreads();
    for (int p = kb / P + tid; p < (kb + nk + P - 1) / P; p += kThreads) {
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
    const int nch = nk * cpr;
    constexpr int U = 8;  // 8 x 512 chunks: the tiny workloads' K and V in one round
    if constexpr (sizeof(TKV) == 4) {
        // fp32 cache: asynchronous copies straight into place, all in flight at once
        for (int c = tid; c < nch; c += kThreads) {
            const int jl = c / cpr, ch = c % cpr, j = kb + jl;
            const int64_t row = ((int64_t)pages[j / P] * a.Hkv + kvh) * P + j % P;
            cp_async_16_cg(Ks + (size_t)jl * KS + ch * E,
                           static_cast<const float*>(a.k_cache) + row * D + ch * E);
            cp_async_16_cg(Vs + (size_t)jl * D + ch * E,
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
                const int j = kb + c / cpr, ch = c % cpr;
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
                const int jl = c / cpr, ch = c % cpr;
                widen16<TKV>(kr[u], Ks + (size_t)jl * KS + ch * E, ks[u]);
                widen16<TKV>(vr[u], Vs + (size_t)jl * D + ch * E, vs[u]);
            }
        }
    }
    __syncthreads();

    // ---- scores of every (row, key); -inf where the key is invisible.  A
    // group of T lanes takes one key and up to RB query rows, so each K row is
    // read from shared memory once per RB rows (the query rows are broadcasts:
    // the groups of a warp share them).  T > 1 (the head dim split over the
    // group's lanes, partial dots summed by shuffles) when there are too few
    // (row block, key) tasks to fill the CTA.
    constexpr int RB = 4;
    const int nrb = (nr + RB - 1) / RB;
    const int ntask = nrb * nk;
    int T = 1;
    while (T < 32 && T * 2 <= D / 4 && ntask * T * 2 <= kThreads) T *= 2;
    const int sub = tid & (T - 1);
    for (int e0 = 0; e0 < ntask; e0 += kThreads / T) {  // uniform over the CTA
        const int e = e0 + tid / T;
        const bool act = e < ntask;
        const int rb = act ? e / nk : 0, jl = act ? e % nk : 0;
        const float4* kv = reinterpret_cast<const float4*>(Ks + (size_t)jl * KS);
        float acc[RB] = {0.f, 0.f, 0.f, 0.f};
        if (act) {
#pragma unroll 4
            for (int d4 = sub; d4 < D / 4; d4 += T) {
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
        }
        for (int o = T / 2; o >= 1; o >>= 1)
#pragma unroll
            for (int u = 0; u < RB; ++u) acc[u] += __shfl_xor_sync(0xffffffffu, acc[u], o);
        if (act && sub == 0) {
            const int j = kb + jl;
#pragma unroll
            for (int u = 0; u < RB; ++u) {
                const int r = rb * RB + u;
                if (r < nr) {
                    const int i = (r0 + r) / G;
                    const bool vis = j < ctx || ((draft_bits(a, b, i) >> (j - ctx)) & 1ull);
                    S[(size_t)r * Lc + jl] = vis ? acc[u] * a.scale : -INFINITY;
                }
            }
        }
    }
    __syncthreads();

    // ---- exact softmax per row (a warp per row) over this CTA's keys: max,
    // then sum of exp.  The cluster form keeps (max, sum) for the merge.
    float* lse_out = a.lse;
    for (int r = warp; r < nr; r += kThreads / 32) {
        float* sr = S + (size_t)r * Lc;
        float m = -INFINITY;
        for (int j = lane; j < nk; j += 32) m = fmaxf(m, sr[j]);
        m = warp_max(m);
        float sum = 0.f;
        for (int j = lane; j < nk; j += 32) {
            const float p = sr[j] == -INFINITY ? 0.f : expf(sr[j] - m);
            sr[j] = p;
            sum += p;
        }
        sum = warp_sum(sum);
        if (lane == 0 && csize > 1) {
            rm[r] = m;
            rl[r] = sum;
        } else if (lane == 0) {
            rl[r] = sum > 0.f ? 1.f / sum : 0.f;
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
    // The cluster form keeps its unnormalised share in Qs (no longer read).
    TQ* out = static_cast<TQ*>(a.out);
    float* Os = Qs;
    auto put = [&](int r, int d, float v) {
        if (csize > 1) {
            Os[r * D + d] = v;
        } else {
            const int row = r0 + r;
            out[(((int64_t)b * a.k + row / G) * a.Hq + kvh * G + row % G) * D + d] =
                Elem<TQ>::from_f32(v * rl[r]);
        }
    };
    const int ncol = nrb * D;  // (row block, column) pairs
    int SF = 1;
    while (SF < 16 && ncol * SF * 2 <= kThreads) SF *= 2;
    const int klen = (nk + SF - 1) / SF;
    for (int e0 = 0; e0 < ncol * SF; e0 += kThreads) {
        const int e = e0 + tid;
        if (e >= ncol * SF) continue;
        const int part = e / ncol, o = e % ncol, rb = o / D, d = o % D;
        const int k0 = part * klen, k1 = min(nk, k0 + klen);
        float acc[RB] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
        for (int j = k0; j < k1; ++j) {
            const float v = Vs[(size_t)j * D + d];
#pragma unroll
            for (int u = 0; u < RB; ++u)
                acc[u] = fmaf(S[(size_t)min(rb * RB + u, nr - 1) * Lc + j], v, acc[u]);
        }
#pragma unroll
        for (int u = 0; u < RB; ++u) {
            const int r = rb * RB + u;
            if (SF > 1) red[(size_t)(part * ncol + o) * RB + u] = acc[u];
            else if (r < nr) put(r, d, acc[u]);
        }
    }
    if (SF > 1) {
        __syncthreads();
        for (int e = tid; e < nr * D; e += kThreads) {
            const int r = e / D, d = e % D;
            const int o = (r / RB) * D + d;
            float acc = 0.f;
            for (int part = 0; part < SF; ++part) acc += red[(size_t)(part * ncol + o) * RB + r % RB];
            put(r, d, acc);
        }
    }
    if (csize == 1) return;

    // ---- cluster merge: CTA c of the cluster finalises an even share of the
    // nr x D outputs from every CTA's (max m, sum l, P V share O) of the row:
    // M = max m_c, out = sum_c e^(m_c - M) O_c / sum_c e^(m_c - M) l_c and
    // lse = M + ln sum_c e^(m_c - M) l_c (CTAs with no visible key of the row
    // have m_c = -inf and drop out).
    cluster_arrive_release();
    cluster_wait_acquire();  // every CTA's shares are written
    const int tot = nr * D, per = (tot + csize - 1) / csize;
    const int e_end = min(tot, (crank + 1) * per);
    for (int e = crank * per + tid; e < e_end; e += kThreads) {
        const int r = e / D, d = e % D;
        float mc[kMaxSmallCluster], lc[kMaxSmallCluster], oc[kMaxSmallCluster];
#pragma unroll
        for (int c = 0; c < kMaxSmallCluster; ++c) {
            if (c < csize) {
                mc[c] = ld_cluster_f32(cluster_map(rm + r, (uint32_t)c));
                lc[c] = ld_cluster_f32(cluster_map(rl + r, (uint32_t)c));
                oc[c] = ld_cluster_f32(cluster_map(Os + r * D + d, (uint32_t)c));
            }
        }
        float M = -INFINITY;
#pragma unroll
        for (int c = 0; c < kMaxSmallCluster; ++c)
            if (c < csize) M = fmaxf(M, mc[c]);
        float lsum = 0.f, o = 0.f;
#pragma unroll
        for (int c = 0; c < kMaxSmallCluster; ++c) {
            if (c < csize && mc[c] != -INFINITY) {
                const float w = expf(mc[c] - M);
                lsum = fmaf(w, lc[c], lsum);
                o = fmaf(w, oc[c], o);
            }
        }
        const int row = r0 + r;
        const int64_t oi = ((int64_t)b * a.k + row / G) * a.Hq + kvh * G + row % G;
        out[oi * D + d] = Elem<TQ>::from_f32(M == -INFINITY ? 0.f : o / lsum);
        if (d == 0 && lse_out) lse_out[oi] = M == -INFINITY ? -INFINITY : M + logf(lsum);
    }
    cluster_arrive_relaxed();
    cluster_wait_acquire();  // no CTA leaves while its shares may still be read
}

template <typename TQ, typename TKV>
cudaError_t launch_typed(const AttnArgs& a, int Lcap, int csize, cudaStream_t stream) {
    const int R = a.k * (a.Hq / a.Hkv), RG = small_rows_per_group(R);
    const int row_groups = (R + RG - 1) / RG;
    const int Lc = (Lcap + csize - 1) / csize;
    const size_t smem = small_smem_bytes(Lc, a.D, RG, a.max_pages);
    auto kern = attn_small_kernel<TQ, TKV>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    const int64_t blocks = (int64_t)a.B * a.Hkv * row_groups * csize;
    if (csize == 1)
        return launch_dependent(kern, dim3((unsigned)blocks), dim3(kThreads), smem, stream, a, Lcap,
                                RG, row_groups, 1);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)csize;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kern, a, Lcap, RG, row_groups, csize);
}

template <typename TQ, typename TKV>
cudaError_t launch_sized(const AttnArgs& a, int Lcap, int csize, bool forced,
                         cudaStream_t stream) {
    if (csize > 1) {
        const cudaError_t e = launch_typed<TQ, TKV>(a, Lcap, csize, stream);
        if (e == cudaSuccess || forced) return e;
        (void)cudaGetLastError();  // a cluster the device cannot place: one CTA per unit
    }
    return launch_typed<TQ, TKV>(a, Lcap, 1, stream);
}

}  // namespace

// The longest context (keys, drafts included) the single-pass kernel holds,
// or 0 when it does not apply: every key a sequence can have -- the whole
// block table -- must fit the shared-memory plan.
int small_attn_max_keys(const AttnArgs& a) {
    const int R = a.k * (a.Hq / a.Hkv), RG = small_rows_per_group(R);
    const int64_t Lcap = (int64_t)a.max_pages * a.P;
    if (Lcap < 1 || Lcap > 4096) return 0;
    if ((int64_t)a.B * a.Hkv * ((R + RG - 1) / RG) * kMaxSmallCluster >= (1LL << 31)) return 0;
    if (small_smem_bytes((int)Lcap, a.D, RG, a.max_pages) > kSmallAttnSmem) return 0;
    return (int)Lcap;
}

// CTAs per (sequence, kv-head, row group): a cluster while the units times
// twice the size still fit the SMs once and each CTA keeps >= 16 keys of the
// block table, else 1.
int small_attn_cluster_size(const AttnArgs& a, int num_sms) {
    const int R = a.k * (a.Hq / a.Hkv), RG = small_rows_per_group(R);
    const int64_t units = (int64_t)a.B * a.Hkv * ((R + RG - 1) / RG);
    const int64_t Lcap = (int64_t)a.max_pages * a.P;
    int c = 1;
    while (c < kMaxSmallCluster && units * c * 2 <= num_sms && Lcap >= 32LL * c) c *= 2;
    return c;
}

cudaError_t launch_attn_small(const AttnArgs& a, int num_sms, int cluster, cudaStream_t stream) {
    const int Lcap = small_attn_max_keys(a);
    if (Lcap == 0 || cluster < 0 || cluster > kMaxSmallCluster) return cudaErrorInvalidValue;
    const bool forced = cluster > 0;
    const int cs = forced ? cluster : small_attn_cluster_size(a, num_sms);
    const bool q32 = a.q_dtype == SPEC_DTYPE_F32;
    switch (a.kv_dtype) {
    case SPEC_DTYPE_F32:
        return q32 ? launch_sized<float, float>(a, Lcap, cs, forced, stream)
                   : launch_sized<__nv_bfloat16, float>(a, Lcap, cs, forced, stream);
    case SPEC_DTYPE_BF16:
        return q32 ? launch_sized<float, __nv_bfloat16>(a, Lcap, cs, forced, stream)
                   : launch_sized<__nv_bfloat16, __nv_bfloat16>(a, Lcap, cs, forced, stream);
    case SPEC_DTYPE_I8:
        return q32 ? launch_sized<float, int8_t>(a, Lcap, cs, forced, stream)
                   : launch_sized<__nv_bfloat16, int8_t>(a, Lcap, cs, forced, stream);
    default:
        return cudaErrorInvalidValue;
    }
}

}  // namespace specv

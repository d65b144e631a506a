// Rejection-sampling acceptance ("Decoding Speculative Decoding from First
// Principles", section "How does this drafter maintain the same distribution
// of the target?").  p is the target's next-token distribution and q the
// drafter's, each softmax(logits / T).  Draft x at position i is kept while
// u_i < p_i(x)/q_i(x); at the first rejection n a token is drawn from the
// residual max(p_n - q_n, 0); after k acceptances the bonus token is drawn
// from p_k.  The emitted tokens then follow p exactly.
//
// Draws: the counter-based generator SplitMix64 (Steele, Lea and Flood,
// "Fast splittable pseudorandom number generators", 2014): draw number
// ((2b + kind) << 32) | j of seed s is the SplitMix64 mix of
// s + (draw + 1) * 0x9E3779B97F4A7C15; kind 0 gives the acceptance uniform of
// position j (24 bits in [0, 1)), kind 1 the Gumbel noise -ln(-ln u) of token
// j (u in (0, 1)).  A draw from weights w is the Gumbel-max choice
// argmax_x ln w(x) + g(x), lowest index on ties.
//
// Two launches, both HBM-bound:
//  1. rows: one CTA per (row, 2048-entry slice) of the k+1 target and k
//     draft rows of every sequence: online (max, sum of exp) of logits / T,
//     and on the target's bonus row the Gumbel-max partial.  The CTA taking
//     the last ticket of a sequence turns the partials into log-sum-exps,
//     runs the k acceptance tests (one thread each), and either emits the
//     bonus draw or records the rejected position for launch 2.
//  2. residual: one CTA per (sequence, slice) of the rejected position's two
//     rows (sequences that kept every draft exit at once); the last ticket
//     merges the Gumbel-max partials into the next token.
#include <limits.h>

#include <algorithm>
#include <type_traits>

#include "common.cuh"

namespace specv {
namespace {

constexpr int kRThreads = 256;
constexpr int kRSlice = 2048;  // vocabulary entries per CTA (many small CTAs balance the
                               // Gumbel-heavy rows against the plain ones)

__device__ __forceinline__ uint64_t sm64_at(uint64_t seed, uint64_t n) {
    uint64_t z = seed + (n + 1) * 0x9E3779B97F4A7C15ull;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}
__device__ __forceinline__ uint64_t draw_index(int b, int kind, int64_t j) {
    return ((uint64_t)(2 * (uint64_t)b + (uint64_t)kind) << 32) | (uint64_t)j;
}
// 24-bit uniforms, exact in fp32: [0, 1) and (0, 1)
__device__ __forceinline__ float unif_co(uint64_t z) { return (float)(z >> 40) * 0x1p-24f; }
__device__ __forceinline__ float unif_oo(uint64_t z) {
    return (float)((z >> 41) * 2 + 1) * 0x1p-24f;
}
// -ln(-ln u): the inner logarithm is accurate (the largest keys come from u
// near 1, where -ln u is small); the outer one is the fast hardware form,
// whose absolute error (~1e-6 on keys of ~10) is far below key gaps that
// decide a draw
__device__ __forceinline__ float gumbel(uint64_t seed, int b, int64_t x) {
    return -__logf(-logf(unif_oo(sm64_at(seed, draw_index(b, 1, x)))));
}
// (key, index) beats (bk, bi): larger key, or equal key and lower index
__device__ __forceinline__ bool better(float v, int i, float bv, int bi) {
    return v > bv || (v == bv && i < bi);
}

// running (max m, sum s of exp(l - m)) of a row in natural-log units
struct Lse {
    float m, s;
};
__device__ __forceinline__ Lse lse_merge(Lse a, Lse b) {
    const float m = fmaxf(a.m, b.m);
    if (m == -INFINITY) return {m, 0.f};
    return {m, a.s * __expf(a.m - m) + b.s * __expf(b.m - m)};
}

template <typename T> __device__ __forceinline__ float to_f(T x) { return Elem<T>::to_f32(x); }

struct RejArgs {
    const void* target;  // [B, k+1, V]
    const void* draft;   // [B, k, V]
    const int32_t* draft_tokens;
    int32_t B, k;
    int64_t V;
    float inv_t;
    uint64_t seed;
    int32_t* accepted_len;
    int32_t* next_token;
    int* dev_err;
};

// A slice is C chunks of kRSlice entries; the host takes C = 4 for large
// vocabularies (fewer, longer CTAs) and C = 1 otherwise (enough CTAs for the
// Gumbel-heavy rows to spread).  Vector path: the slice starts on a 16-byte
// boundary and holds whole 16-byte vectors; otherwise one entry at a time.
template <typename T, int C>
struct Slice {
    static constexpr int VEC = 16 / sizeof(T);
    static constexpr int PER = C * kRSlice / VEC / kRThreads;  // 16-byte loads per thread
    static __device__ __forceinline__ bool vector_path(const T* x, int64_t e0, int64_t e1) {
        return (reinterpret_cast<uintptr_t>(x + e0) & 15) == 0 && (e1 - e0) % VEC == 0;
    }
};

// (max, sum of exp) of logits / T over a slice: every load first, then the
// max, then the sum (no per-element branch)
template <typename T, int C>
__device__ __forceinline__ Lse slice_lse(const T* x, int64_t e0, int64_t e1, float inv_t) {
    using S = Slice<T, C>;
    const int tid = threadIdx.x;
    if (S::vector_path(x, e0, e1)) {
        const int nvec = (int)((e1 - e0) / S::VEC);
        const uint4* xv = reinterpret_cast<const uint4*>(x + e0);
        uint4 raw[S::PER];
#pragma unroll
        for (int u = 0; u < S::PER; ++u) {
            const int vi = tid + u * kRThreads;
            raw[u] = vi < nvec ? __ldcs(xv + vi) : make_uint4(0, 0, 0, 0);
        }
        float m = -INFINITY;
#pragma unroll
        for (int u = 0; u < S::PER; ++u) {
            if (tid + u * kRThreads >= nvec) continue;
            const T* el = reinterpret_cast<const T*>(&raw[u]);
#pragma unroll
            for (int q = 0; q < S::VEC; ++q) m = fmaxf(m, to_f(el[q]) * inv_t);
        }
        float sum = 0.f;
#pragma unroll
        for (int u = 0; u < S::PER; ++u) {
            if (tid + u * kRThreads >= nvec) continue;
            const T* el = reinterpret_cast<const T*>(&raw[u]);
#pragma unroll
            for (int q = 0; q < S::VEC; ++q) sum += __expf(to_f(el[q]) * inv_t - m);
        }
        return {m, sum};
    }
    Lse acc = {-INFINITY, 0.f};
    for (int64_t e = e0 + tid; e < e1; e += kRThreads) {
        const float l = to_f(x[e]) * inv_t;
        if (l > acc.m) {
            acc.s = acc.s * __expf(acc.m - l) + 1.f;  // exp(-inf) = 0 on the first element
            acc.m = l;
        } else {
            acc.s += __expf(l - acc.m);
        }
    }
    return acc;
}

// Visits the entries [e0, e1) of row xp and the same entries of row xq (if
// given), each thread in increasing index order: f(e, p, q).  For the
// Gumbel-heavy passes: one 16-byte vector per step, the next one in flight
// while the current one is processed (no unrolling across vectors).
template <typename T, int C, typename F>
__device__ __forceinline__ void walk_slice(const T* xp, const T* xq, int64_t e0, int64_t e1, F&& f) {
    using S = Slice<T, C>;
    const int tid = threadIdx.x;
    if (S::vector_path(xp, e0, e1) && (!xq || S::vector_path(xq, e0, e1))) {
        const int nvec = (int)((e1 - e0) / S::VEC);
        const uint4* pv = reinterpret_cast<const uint4*>(xp + e0);
        const uint4* qv = xq ? reinterpret_cast<const uint4*>(xq + e0) : nullptr;
        const uint4 z = make_uint4(0, 0, 0, 0);
        int vi = tid;
        uint4 cp = vi < nvec ? __ldcs(pv + vi) : z;
        uint4 cq = (qv && vi < nvec) ? __ldcs(qv + vi) : z;
#pragma unroll 1
        for (; vi < nvec; vi += kRThreads) {
            const int vn = vi + kRThreads;
            const uint4 np = vn < nvec ? __ldcs(pv + vn) : z;
            const uint4 nq = (qv && vn < nvec) ? __ldcs(qv + vn) : z;
            const T* ep = reinterpret_cast<const T*>(&cp);
            const T* eq = reinterpret_cast<const T*>(&cq);
#pragma unroll
            for (int q = 0; q < S::VEC; ++q) f(e0 + (int64_t)vi * S::VEC + q, to_f(ep[q]), to_f(eq[q]));
            cp = np;
            cq = nq;
        }
        return;
    }
    for (int64_t e = e0 + tid; e < e1; e += kRThreads)
        f(e, to_f(xp[e]), xq ? to_f(xq[e]) : 0.f);
}

// CTA-wide reductions; results valid in every thread
template <typename R, typename M>
__device__ __forceinline__ R block_reduce(R v, R* s_red, M&& merge) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        R w;
        w.a = __shfl_xor_sync(0xffffffffu, v.a, o);
        w.b = __shfl_xor_sync(0xffffffffu, v.b, o);
        v = merge(v, w);
    }
    if (lane == 0) s_red[warp] = v;
    __syncthreads();
    R r = s_red[0];
    for (int w = 1; w < kRThreads / 32; ++w) r = merge(r, s_red[w]);
    __syncthreads();
    return r;
}
struct LsePair {
    float a, b;  // (m, s)
};
struct KeyPair {
    float a;  // key
    int b;    // index
};
__device__ __forceinline__ LsePair merge_lse(LsePair x, LsePair y) {
    const Lse r = lse_merge({x.a, x.b}, {y.a, y.b});
    return {r.m, r.s};
}
__device__ __forceinline__ KeyPair merge_key(KeyPair x, KeyPair y) {
    return better(y.a, y.b, x.a, x.b) ? y : x;
}

// grid (slices, 2k+1 rows, B): row r <= k is target row r, r > k draft row r-k-1
template <typename T, int C>
__global__ void __launch_bounds__(kRThreads)
rej_rows_kernel(RejArgs a, float2* __restrict__ part_ms, float* __restrict__ part_gk,
                int* __restrict__ part_gi, int4* __restrict__ state, int32_t* __restrict__ tickets) {
    __shared__ LsePair s_lse[kRThreads / 32];
    __shared__ KeyPair s_key[kRThreads / 32];
    __shared__ float s_row_lse[129];  // 2k + 1 <= 129 rows
    __shared__ int s_last, s_first_fail;

    const int ns = gridDim.x, rows = gridDim.y;
    const int slice = blockIdx.x, r = blockIdx.y, b = blockIdx.z;
    const bool is_target = r <= a.k, bonus = r == a.k;
    const T* x = is_target
                     ? static_cast<const T*>(a.target) + ((int64_t)b * (a.k + 1) + r) * a.V
                     : static_cast<const T*>(a.draft) + ((int64_t)b * a.k + (r - a.k - 1)) * a.V;
    const int64_t sl = (int64_t)C * kRSlice;
    const int64_t e0 = (int64_t)slice * sl, e1 = min(a.V, e0 + sl);

    Lse acc = {-INFINITY, 0.f};
    float bk = -INFINITY;
    int bi = INT_MAX;
    if (!bonus) {
        acc = slice_lse<T, C>(x, e0, e1, a.inv_t);
    } else {
        walk_slice<T, C>(x, (const T*)nullptr, e0, e1, [&](int64_t e, float v, float) {
            const float l = v * a.inv_t;
            if (l > acc.m) {
                acc.s = acc.s * __expf(acc.m - l) + 1.f;
                acc.m = l;
            } else {
                acc.s += __expf(l - acc.m);
            }
            const float key = l + gumbel(a.seed, b, e);
            if (better(key, (int)e, bk, bi)) { bk = key; bi = (int)e; }
        });
    }
    const LsePair tot = block_reduce(LsePair{acc.m, acc.s}, s_lse, merge_lse);
    KeyPair best = {bk, bi};
    if (bonus) best = block_reduce(best, s_key, merge_key);
    if (threadIdx.x == 0) {
        part_ms[((int64_t)b * rows + r) * ns + slice] = make_float2(tot.a, tot.b);
        if (bonus) {
            part_gk[(int64_t)b * ns + slice] = best.a;
            part_gi[(int64_t)b * ns + slice] = best.b;
        }
        __threadfence();
        const int t = atomicAdd(&tickets[b], 1);
        s_last = t == rows * ns - 1;
        if (s_last) __threadfence();
    }
    __syncthreads();
    if (!s_last) return;
    // ---- last CTA of sequence b: log-sum-exp of every row, then the tests
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int rr = warp; rr < rows; rr += kRThreads / 32) {
        LsePair v = {-INFINITY, 0.f};
        for (int sl = lane; sl < ns; sl += 32) {
            const float2 p = __ldcg(part_ms + ((int64_t)b * rows + rr) * ns + sl);
            v = merge_lse(v, {p.x, p.y});
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            LsePair w;
            w.a = __shfl_xor_sync(0xffffffffu, v.a, o);
            w.b = __shfl_xor_sync(0xffffffffu, v.b, o);
            v = merge_lse(v, w);
        }
        if (lane == 0) s_row_lse[rr] = v.a + logf(v.b);
    }
    if (tid == 0) s_first_fail = a.k;
    __syncthreads();
    if (tid < a.k) {
        const int32_t xt = __ldg(a.draft_tokens + (int64_t)b * a.k + tid);
        bool fail;
        if (xt < 0 || xt >= a.V) {
            raise_device_error(a.dev_err, SPEC_DEVERR_TOKEN);
            fail = true;
        } else {
            const float lp = to_f(static_cast<const T*>(a.target)[((int64_t)b * (a.k + 1) + tid) * a.V + xt]) *
                                 a.inv_t - s_row_lse[tid];
            const float lq = to_f(static_cast<const T*>(a.draft)[((int64_t)b * a.k + tid) * a.V + xt]) *
                                 a.inv_t - s_row_lse[a.k + 1 + tid];
            const float ratio = expf(lp - lq);  // p(x) / q(x)
            const float u = unif_co(sm64_at(a.seed, draw_index(b, 0, tid)));
            fail = !(u < ratio);
        }
        if (fail) atomicMin(&s_first_fail, tid);
    }
    __syncthreads();
    const int n = s_first_fail;
    if (n == a.k) {
        // every draft kept: the bonus draw from p_k
        if (warp == 0) {
            KeyPair v = {-INFINITY, INT_MAX};
            for (int sl = lane; sl < ns; sl += 32)
                v = merge_key(v, {__ldcg(part_gk + (int64_t)b * ns + sl),
                                  __ldcg(part_gi + (int64_t)b * ns + sl)});
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                KeyPair w;
                w.a = __shfl_xor_sync(0xffffffffu, v.a, o);
                w.b = __shfl_xor_sync(0xffffffffu, v.b, o);
                v = merge_key(v, w);
            }
            if (lane == 0) {
                a.accepted_len[b] = a.k;
                a.next_token[b] = v.b;
                state[b] = make_int4(a.k, 0, 0, 0);
            }
        }
    } else if (tid == 0) {
        a.accepted_len[b] = n;
        state[b] = make_int4(n, __float_as_int(s_row_lse[n]), __float_as_int(s_row_lse[a.k + 1 + n]), 0);
    }
    if (tid == 0) tickets[b] = 0;  // ready for the residual launch / the next call
}

// grid (slices, B)
template <typename T, int C>
__global__ void __launch_bounds__(kRThreads)
rej_residual_kernel(RejArgs a, const int4* __restrict__ state, float* __restrict__ part_k,
                    int* __restrict__ part_i, int32_t* __restrict__ tickets) {
    __shared__ KeyPair s_key[kRThreads / 32];
    __shared__ int s_last;
    const int ns = gridDim.x;
    const int slice = blockIdx.x, b = blockIdx.y;
    const int4 st = __ldcg(state + b);
    const int n = st.x;
    if (n >= a.k) return;  // every draft kept: nothing to draw here
    const float lse_p = __int_as_float(st.y), lse_q = __int_as_float(st.z);
    const T* xp = static_cast<const T*>(a.target) + ((int64_t)b * (a.k + 1) + n) * a.V;
    const T* xq = static_cast<const T*>(a.draft) + ((int64_t)b * a.k + n) * a.V;
    const int64_t sl = (int64_t)C * kRSlice;
    const int64_t e0 = (int64_t)slice * sl, e1 = min(a.V, e0 + sl);
    float bk = -INFINITY;
    int bi = INT_MAX;
    walk_slice<T, C>(xp, xq, e0, e1, [&](int64_t e, float v, float vq) {
        // ln(p - q) + g where p > q
        const float w = __expf(v * a.inv_t - lse_p) - __expf(vq * a.inv_t - lse_q);
        if (w > 0.f) {
            const float key = logf(w) + gumbel(a.seed, b, e);
            if (better(key, (int)e, bk, bi)) { bk = key; bi = (int)e; }
        }
    });
    const KeyPair best = block_reduce(KeyPair{bk, bi}, s_key, merge_key);
    if (threadIdx.x == 0) {
        part_k[(int64_t)b * ns + slice] = best.a;
        part_i[(int64_t)b * ns + slice] = best.b;
        __threadfence();
        const int t = atomicAdd(&tickets[b], 1);
        s_last = t == ns - 1;
        if (s_last) __threadfence();
    }
    __syncthreads();
    if (!s_last) return;
    const int lane = threadIdx.x & 31;
    if (threadIdx.x < 32) {
        KeyPair v = {-INFINITY, INT_MAX};
        for (int q = lane; q < ns; q += 32)
            v = merge_key(v, {__ldcg(part_k + (int64_t)b * ns + q), __ldcg(part_i + (int64_t)b * ns + q)});
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            KeyPair w;
            w.a = __shfl_xor_sync(0xffffffffu, v.a, o);
            w.b = __shfl_xor_sync(0xffffffffu, v.b, o);
            v = merge_key(v, w);
        }
        if (lane == 0) {
            a.next_token[b] = v.b;
            tickets[b] = 0;  // ready for the next call
        }
    }
}

// chunks per slice: long CTAs for large vocabularies, short ones otherwise
int rej_chunks(int64_t V) { return V >= 65536 ? 4 : 1; }
int rej_slices(int64_t V) {
    const int64_t sl = (int64_t)rej_chunks(V) * kRSlice;
    return (int)((V + sl - 1) / sl);
}



}  // namespace

size_t rejection_workspace_bytes(int B, int k, int64_t V) {
    const int64_t ns = rej_slices(V);
    const int64_t units = (int64_t)B * (2 * k + 1) * ns;
    return (size_t)units * sizeof(float2) + (size_t)B * ns * (sizeof(float) + sizeof(int)) +
           (size_t)B * sizeof(int4) + 1024;
}

cudaError_t launch_accept_rejection(const void* target, const void* draft, int32_t dtype,
                                    const int32_t* draft_tokens, int B, int k, int64_t V,
                                    float temperature, uint64_t seed, int32_t* accepted_len,
                                    int32_t* next_token, void* workspace, int32_t* tickets,
                                    int* dev_err, cudaStream_t stream) {
    if (B == 0) return cudaSuccess;
    RejArgs a;
    a.target = target;
    a.draft = draft;
    a.draft_tokens = draft_tokens;
    a.B = B;
    a.k = k;
    a.V = V;
    a.inv_t = 1.0f / temperature;
    a.seed = seed;
    a.accepted_len = accepted_len;
    a.next_token = next_token;
    a.dev_err = dev_err;
    const int ns = rej_slices(V);
    const int64_t units = (int64_t)B * (2 * k + 1) * ns;
    // workspace: [units] float2 | [B*ns] float | [B*ns] int | [B] int4 (16-byte aligned)
    char* w = static_cast<char*>(workspace);
    float2* part_ms = reinterpret_cast<float2*>(w);
    w += (size_t)units * sizeof(float2);
    float* part_k = reinterpret_cast<float*>(w);
    w += (size_t)B * ns * sizeof(float);
    int* part_i = reinterpret_cast<int*>(w);
    w += (size_t)B * ns * sizeof(int);
    w = reinterpret_cast<char*>((reinterpret_cast<uintptr_t>(w) + 15) & ~uintptr_t(15));
    int4* state = reinterpret_cast<int4*>(w);
    const int rows = 2 * k + 1;
    auto go = [&](auto tag, auto ctag) {
        using T = decltype(tag);
        constexpr int C = decltype(ctag)::value;
        rej_rows_kernel<T, C><<<dim3(ns, rows, B), kRThreads, 0, stream>>>(a, part_ms, part_k,
                                                                          part_i, state, tickets);
        rej_residual_kernel<T, C><<<dim3(ns, B), kRThreads, 0, stream>>>(a, state, part_k, part_i,
                                                                       tickets);
    };
    using C1 = std::integral_constant<int, 1>;
    using C4 = std::integral_constant<int, 4>;
    const bool big = rej_chunks(V) == 4;
    if (dtype == SPEC_DTYPE_F32) {
        if (big) go(float(), C4()); else go(float(), C1());
    } else {
        if (big) go(__nv_bfloat16(), C4()); else go(__nv_bfloat16(), C1());
    }
    return cudaGetLastError();
}

}  // namespace specv

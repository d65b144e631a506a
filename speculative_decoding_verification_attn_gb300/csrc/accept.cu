// Greedy longest-prefix acceptance ("Decoding Speculative Decoding from First
// Principles", "Speculating to get sequence parallelism during decode"): the
// target's prediction at each of the k+1 positions is the argmax of its
// logits row; drafts are kept up to the first disagreement and the target's
// own token there (or the bonus token after k agreements) is emitted.
//
// One launch, in one of two forms.
//
//  * Cluster form (k + 1 <= 16 rows per sequence, rows starting on 16-byte
//    boundaries): one thread-block cluster per sequence, one CTA per
//    (row, vocabulary part).  Each CTA reduces its part with all of its
//    16-byte loads issued together, then writes its (max, lowest index) into
//    shared memory of the cluster's first CTA; after a cluster barrier that
//    CTA reduces each row's parts and runs the prefix match.  No global
//    workspace, fence or atomic lies on the path.
//  * Ticket form (everything else): each CTA reduces one 8192-entry slice of
//    one row, writes its pair to the workspace and takes a ticket of its
//    sequence; the CTA that takes the last ticket merges the sequence's
//    slices, runs the prefix match and resets the ticket, so no CTA ever
//    waits on another.
#include <limits.h>

#include <algorithm>
#include <mutex>

#include "common.cuh"

namespace specv {
namespace {

constexpr int kThreads = 256;   // ticket form
constexpr int kSlice = 8192;    // vocabulary entries per CTA (ticket form)
constexpr int kCThreads = 512;  // cluster form
constexpr int kMaxCluster = 16;
constexpr int kLoads = 8;       // 16-byte loads per thread per round (cluster form)

// (v, i) beats (bv, bi): larger value, or equal value and lower index.
__device__ __forceinline__ bool better(float v, int i, float bv, int bi) {
    return v > bv || (v == bv && i < bi);
}

__device__ __forceinline__ void warp_argmax(float& v, int& i) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, v, o);
        const int oi = __shfl_xor_sync(0xffffffffu, i, o);
        if (better(ov, oi, v, i)) {
            v = ov;
            i = oi;
        }
    }
}

template <typename T> __device__ __forceinline__ float to_f(T x) { return Elem<T>::to_f32(x); }

// Folds the 16-byte vector of elements base, base+1, ... into the running
// (max, lowest index) of a thread that visits its vectors in increasing
// index order: the vector's maximum is found with packed max instructions
// (which skip NaN, as the comparisons below do), and only a vector that
// raises the running maximum -- or the first one that is not all NaN -- is
// searched for the lowest index holding it.
__device__ __forceinline__ void fold_vec(const uint4& raw, int base, float& bv, int& bi,
                                         __nv_bfloat16) {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&raw);
    const __nv_bfloat162 m2 = __hmax2(__hmax2(h[0], h[1]), __hmax2(h[2], h[3]));
    const float vm = fmaxf(__low2float(m2), __high2float(m2));
    if (vm > bv || (bi == INT_MAX && vm == vm)) {
        const __nv_bfloat16* el = reinterpret_cast<const __nv_bfloat16*>(&raw);
#pragma unroll
        for (int q = 7; q >= 0; --q)
            if (__bfloat162float(el[q]) == vm) bi = base + q;
        bv = vm;
    }
}
__device__ __forceinline__ void fold_vec(const uint4& raw, int base, float& bv, int& bi, float) {
    const float* f = reinterpret_cast<const float*>(&raw);
    const float vm = fmaxf(fmaxf(f[0], f[1]), fmaxf(f[2], f[3]));
    if (vm > bv || (bi == INT_MAX && vm == vm)) {
#pragma unroll
        for (int q = 3; q >= 0; --q)
            if (f[q] == vm) bi = base + q;
        bv = vm;
    }
}

// CTA-wide (max, lowest index); the result is valid in thread 0.
template <int NT>
__device__ __forceinline__ void block_argmax(float& bv, int& bi, float* s_v, int* s_i) {
    const int tid = threadIdx.x;
    warp_argmax(bv, bi);
    if ((tid & 31) == 0) { s_v[tid >> 5] = bv; s_i[tid >> 5] = bi; }
    __syncthreads();
    if (tid < 32) {
        bv = tid < NT / 32 ? s_v[tid] : -INFINITY;
        bi = tid < NT / 32 ? s_i[tid] : INT_MAX;
        warp_argmax(bv, bi);
    }
}

// Prefix match of sequence b given the k+1 argmaxes in s_am; `my_draft` is
// draft tid of the sequence (threads < k).  Ends with a CTA barrier.
__device__ __forceinline__ void prefix_match(const AcceptArgs& a, int b, int my_draft,
                                             const int* s_am, int* s_first_miss) {
    const int tid = threadIdx.x;
    // accepted length = first position whose draft differs from the argmax
    if (tid < a.k && my_draft != s_am[tid]) atomicMin(s_first_miss, tid);
    __syncthreads();
    if (tid == 0) {
        const int n = *s_first_miss;
        a.accepted_len[b] = n;
        a.next_token[b] = s_am[n];
    }
}

// Greedy acceptance over a tree of drafts (SpecInfer / EAGLE-style token
// trees, "Decoding Speculative Decoding from First Principles", "Advances in
// speculators"): node i carries draft_tokens[b, i] and parent[b, i] in
// [-1, i); s_am[0] is the target's argmax at the root, s_am[i+1] after node
// i.  From the root, keep the lowest-index child whose token is the argmax
// at the current node; stop when none is.  Warp 0 only: each lane holds
// nodes lane and lane + 32, a step is one ballot.  Only children with a
// higher index than the current node are taken, so the walk ends within k
// steps even with corrupt parents (which are also flagged).
__device__ __forceinline__ void tree_walk(const AcceptArgs& a, int b, const int* s_am) {
    const int lane = threadIdx.x & 31;
    int par[2], tok[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int c = lane + 32 * h;
        par[h] = c < a.k ? __ldg(a.parent + (int64_t)b * a.k + c) : -2;
        tok[h] = c < a.k ? __ldg(a.draft + (int64_t)b * a.k + c) : -1;
        if (c < a.k && (par[h] < -1 || par[h] >= c)) raise_device_error(a.dev_err, SPEC_DEVERR_TREE);
    }
    int cur = -1, n = 0;
    for (int step = 0; step < a.k; ++step) {
        const int am = s_am[cur + 1];
        const unsigned b0 = __ballot_sync(0xffffffffu, par[0] == cur && lane > cur && tok[0] == am);
        const unsigned b1 =
            __ballot_sync(0xffffffffu, par[1] == cur && lane + 32 > cur && tok[1] == am);
        const int next = b0 ? __ffs(b0) - 1 : b1 ? 32 + __ffs(b1) - 1 : -1;
        if (next < 0) break;
        if (a.path && lane == 0) a.path[(int64_t)b * a.k + n] = next;
        ++n;
        cur = next;
    }
    if (a.path)
        for (int i = n + lane; i < a.k; i += 32) a.path[(int64_t)b * a.k + i] = -1;
    if (lane == 0) {
        a.accepted_len[b] = n;
        a.next_token[b] = s_am[cur + 1];
    }
}

// ---------------------------------------------------------------- cluster form

template <typename T>
__global__ void __launch_bounds__(kCThreads)
accept_cluster_kernel(AcceptArgs a, int parts, int64_t part_len) {
    constexpr int E = 16 / sizeof(T);  // elements per 16-byte load
    constexpr int ROUND = kCThreads * kLoads * E;
    __shared__ float c_v[kMaxCluster];  // first CTA: one entry per CTA of the cluster
    __shared__ int c_i[kMaxCluster];
    __shared__ float s_v[kCThreads / 32];
    __shared__ int s_i[kCThreads / 32];
    __shared__ int s_am[65];
    __shared__ int s_first_miss;

    grid_dep_launch_dependents();
    grid_dep_wait();
    const int tid = threadIdx.x;
    const int S = (a.k + 1) * parts;  // cluster size
    const uint32_t rank = cluster_ctarank();
    const int b = (int)(blockIdx.x / S);
    const int row = (int)rank / parts, part = (int)rank % parts;
    // phase 0 completes once every CTA of the cluster has started
    cluster_arrive_relaxed();
    const int my_draft = (rank == 0 && tid < a.k) ? __ldg(a.draft + (int64_t)b * a.k + tid) : 0;
    if (rank == 0 && tid == 0) s_first_miss = a.k;

    const T* x = static_cast<const T*>(a.logits) + ((int64_t)b * (a.k + 1) + row) * a.V;
    const int64_t e0 = (int64_t)part * part_len;
    const int64_t e1 = min(a.V, e0 + part_len);
    float bv = -INFINITY;
    int bi = INT_MAX;
    for (int64_t r0 = e0; r0 < e1; r0 += ROUND) {
        const int nvec = (int)((min(e1, r0 + ROUND) - r0) / E);
        const uint4* xv = reinterpret_cast<const uint4*>(x + r0);
        uint4 raw[kLoads];
#pragma unroll
        for (int u = 0; u < kLoads; ++u) {
            const int vi = tid + u * kCThreads;
            raw[u] = vi < nvec ? __ldcs(xv + vi) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < kLoads; ++u) {
            const int vi = tid + u * kCThreads;
            if (vi < nvec) fold_vec(raw[u], (int)(r0 + (int64_t)vi * E), bv, bi, T());
        }
    }
    block_argmax<kCThreads>(bv, bi, s_v, s_i);
    cluster_wait_acquire();  // phase 0: the first CTA's shared memory exists
    if (tid == 0) {
        st_cluster_f32(cluster_map(&c_v[rank], 0), bv);
        st_cluster_s32(cluster_map(&c_i[rank], 0), bi);
    }
    cluster_arrive_release();
    cluster_wait_acquire();  // phase 1: every CTA's pair is in the first CTA
    if (rank != 0) return;
    if (tid <= a.k) {
        float v = -INFINITY;
        int idx = INT_MAX;
        for (int p = 0; p < parts; ++p) {
            const int r = tid * parts + p;
            if (better(c_v[r], c_i[r], v, idx)) { v = c_v[r]; idx = c_i[r]; }
        }
        s_am[tid] = idx;
    }
    __syncthreads();
    if (a.parent) {
        if (tid < 32) tree_walk(a, b, s_am);
    } else {
        prefix_match(a, b, my_draft, s_am, &s_first_miss);
    }
}

// ---------------------------------------------------------------- ticket form

template <typename T>
__global__ void __launch_bounds__(kThreads)
accept_greedy_kernel(AcceptArgs a, int n_slices, float* __restrict__ part_v,
                     int* __restrict__ part_i, int32_t* __restrict__ tickets) {
    constexpr int VEC = 16 / sizeof(T);
    constexpr int PER = kSlice / VEC / kThreads;  // 16-byte loads per thread in a full slice
    __shared__ float s_v[kThreads / 32];
    __shared__ int s_i[kThreads / 32];
    __shared__ int s_last;
    __shared__ int s_am[65];
    __shared__ int s_first_miss;

    grid_dep_launch_dependents();
    grid_dep_wait();
    const int row = blockIdx.x / n_slices;  // row of [B, k+1]
    const int slice = blockIdx.x % n_slices;
    const int b = row / (a.k + 1);
    const int tid = threadIdx.x;
    // this sequence's drafts, read now so that the prefix match (done by the
    // CTA that merges the sequence) costs no extra memory round trip
    const int my_draft = tid < a.k ? __ldg(a.draft + (int64_t)b * a.k + tid) : 0;
    const T* x = static_cast<const T*>(a.logits) + (int64_t)row * a.V;
    const int64_t e0 = (int64_t)slice * kSlice;
    const int64_t e1 = min(a.V, e0 + (int64_t)kSlice);

    float bv = -INFINITY;
    int bi = INT_MAX;
    const uintptr_t addr = reinterpret_cast<uintptr_t>(x + e0);
    if ((addr & 15) == 0 && e1 - e0 == kSlice) {
        // full aligned slice: every load issued before any is used
        const uint4* xv = reinterpret_cast<const uint4*>(x + e0);
        uint4 raw[PER];
#pragma unroll
        for (int u = 0; u < PER; ++u) raw[u] = __ldcs(xv + tid + u * kThreads);
#pragma unroll
        for (int u = 0; u < PER; ++u)
            fold_vec(raw[u], (int)(e0 + (int64_t)(tid + u * kThreads) * VEC), bv, bi, T());
    } else {
        // unaligned head, 16-byte body, tail: each thread visits its elements
        // in increasing index order
        int64_t head = (int64_t)(((16 - (addr & 15)) & 15) / sizeof(T));
        if (head > e1 - e0) head = e1 - e0;
        if (tid < head) {
            const float v = to_f(x[e0 + tid]);
            if (better(v, (int)(e0 + tid), bv, bi)) { bv = v; bi = (int)(e0 + tid); }
        }
        const int64_t eb = e0 + head;
        const int64_t nvec = (e1 - eb) / VEC;
        const uint4* xv = reinterpret_cast<const uint4*>(x + eb);
        for (int64_t vi = tid; vi < nvec; vi += kThreads) {
            const uint4 raw = __ldcs(xv + vi);
            const T* el = reinterpret_cast<const T*>(&raw);
#pragma unroll
            for (int u = 0; u < VEC; ++u) {
                const float v = to_f(el[u]);
                const int idx = (int)(eb + vi * VEC + u);
                if (better(v, idx, bv, bi)) { bv = v; bi = idx; }
            }
        }
        const int64_t et = eb + nvec * VEC;
        if (et + tid < e1) {
            const float v = to_f(x[et + tid]);
            if (better(v, (int)(et + tid), bv, bi)) { bv = v; bi = (int)(et + tid); }
        }
    }

    block_argmax<kThreads>(bv, bi, s_v, s_i);
    if (tid == 0) {
        part_v[blockIdx.x] = bv;
        part_i[blockIdx.x] = bi;
        __threadfence();
        const int t = atomicAdd(&tickets[b], 1);
        s_last = (t == (a.k + 1) * n_slices - 1);
        if (s_last) __threadfence();
    }
    __syncthreads();
    if (!s_last) return;

    // Last CTA of sequence b: reduce each row's slices, then the prefix match.
    const int warp = tid >> 5, lane = tid & 31;
    for (int i = warp; i <= a.k; i += kThreads / 32) {
        const int64_t base = ((int64_t)b * (a.k + 1) + i) * n_slices;
        float v = -INFINITY;
        int idx = INT_MAX;
        for (int s = lane; s < n_slices; s += 32) {
            const float sv = __ldcg(part_v + base + s);
            const int si = __ldcg(part_i + base + s);
            if (better(sv, si, v, idx)) { v = sv; idx = si; }
        }
        warp_argmax(v, idx);
        if (lane == 0) s_am[i] = idx;
    }
    if (tid == 0) s_first_miss = a.k;
    __syncthreads();
    if (a.parent) {
        if (tid < 32) tree_walk(a, b, s_am);
    } else {
        prefix_match(a, b, my_draft, s_am, &s_first_miss);
    }
    if (tid == 0) tickets[b] = 0;  // ready for the next call
}

int num_slices(int64_t V) { return (int)((V + kSlice - 1) / kSlice); }

// Vocabulary parts per row of the cluster form, or 0 when it does not apply:
// more than 16 rows per sequence, rows not on 16-byte boundaries, or more
// CTAs than SMs (the form is for calls whose clusters all run at once).
int cluster_parts(const AcceptArgs& a, int sms) {
    const int E = a.dtype == SPEC_DTYPE_F32 ? 4 : 8;
    if (a.k + 1 > kMaxCluster || a.V % E != 0) return 0;
    const int64_t round = (int64_t)kCThreads * kLoads * E;
    const int64_t rows = (int64_t)a.B * (a.k + 1);
    int64_t parts = std::min<int64_t>(kMaxCluster / (a.k + 1), (a.V + round - 1) / round);
    parts = std::min<int64_t>(parts, sms / rows);
    return parts >= 1 ? (int)parts : 0;
}

template <typename T>
cudaError_t launch_cluster(const AcceptArgs& a, int parts, cudaStream_t stream) {
    const int E = 16 / (int)sizeof(T);
    int64_t part_len = (a.V + parts - 1) / parts;
    part_len = (part_len + E - 1) / E * E;  // parts start on 16-byte boundaries
    const int S = (a.k + 1) * parts;
    if (S > 8) {  // above the portable cluster size
        const cudaError_t e = cudaFuncSetAttribute(accept_cluster_kernel<T>,
                                                   cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((int64_t)a.B * S));
    cfg.blockDim = dim3(kCThreads);
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)S;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, accept_cluster_kernel<T>, a, parts, part_len);
}

}  // namespace

size_t accept_workspace_bytes(const AcceptArgs& a) {
    const int64_t parts = (int64_t)a.B * (a.k + 1) * num_slices(a.V);
    return (size_t)parts * (sizeof(float) + sizeof(int)) + 256;
}

cudaError_t launch_accept(const AcceptArgs& a, void* workspace, int32_t* tickets,
                          cudaStream_t stream) {
    if (a.B == 0) return cudaSuccess;
    int dev = 0, sms = 0;
    cudaError_t e0 = cudaGetDevice(&dev);
    if (e0 == cudaSuccess) e0 = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e0 != cudaSuccess) return e0;
    const int parts = cluster_parts(a, sms);
    if (parts > 0 && (int64_t)a.B * (a.k + 1) * parts < (1LL << 31)) {
        const cudaError_t e = a.dtype == SPEC_DTYPE_F32 ? launch_cluster<float>(a, parts, stream)
                                                        : launch_cluster<__nv_bfloat16>(a, parts, stream);
        if (e == cudaSuccess) return cudaSuccess;
        (void)cudaGetLastError();  // a cluster shape the device cannot place: ticket form
    }
    const int ns = num_slices(a.V);
    const int64_t total = (int64_t)a.B * (a.k + 1) * ns;
    float* pv = static_cast<float*>(workspace);
    int* pi = reinterpret_cast<int*>(pv + total);
    if (a.dtype == SPEC_DTYPE_F32)
        return launch_dependent(accept_greedy_kernel<float>, dim3((unsigned)total), dim3(kThreads), 0,
                                stream, a, ns, pv, pi, tickets);
    return launch_dependent(accept_greedy_kernel<__nv_bfloat16>, dim3((unsigned)total),
                            dim3(kThreads), 0, stream, a, ns, pv, pi, tickets);
}

}  // namespace specv

// ---------------------------------------------------------------- no-allocation variant
//
// Greedy acceptance for callers that cannot allocate device memory: serving
// loops whose device memory is reserved up front by their own allocator,
// where an extra cudaMalloc may fail or stall the step, and hosts that load
// the library as a plugin without the right to allocate.  The reduction
// partials and completion tickets live in one fixed array of this file;
// every call on a device shares it.

namespace specv {
namespace {

// (row, vocabulary slice) partials and sequences the fixed scratch holds
constexpr int64_t kNoAllocMaxPartials = SPEC_NOALLOC_MAX_PARTIALS;
constexpr int kNoAllocMaxBatch = SPEC_NOALLOC_MAX_BATCH;
constexpr size_t kNoAllocPartialBytes =
    (size_t)kNoAllocMaxPartials * (sizeof(float) + sizeof(int));

std::mutex g_noalloc_mu;
void* g_noalloc_addr[256] = {};  // device address of the scratch, per device

}  // namespace
}  // namespace specv

static __device__ __align__(256) unsigned char
    g_noalloc_scratch[specv::kNoAllocPartialBytes + specv::kNoAllocMaxBatch * sizeof(int32_t)];

namespace specv {
namespace {

// Device address of the fixed scratch on the current device.  The first call
// on a device looks it up with cudaGetSymbolAddress (which may load this
// library's device code); later calls reuse the cached address, which stays
// valid for the life of the device's primary context (a cudaDeviceReset would
// leave it stale; the header rules such calls out).
int noalloc_scratch(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return set_error(SPEC_ERR_CUDA, "cudaGetDevice failed");
    if (dev < 0 || dev >= 256) return set_error(SPEC_ERR_UNSUPPORTED, "device index >= 256");
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (!g_noalloc_addr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || !p)
            return set_error(SPEC_ERR_CUDA, "cudaGetSymbolAddress of the fixed scratch failed");
        g_noalloc_addr[dev] = p;
    }
    *out = g_noalloc_addr[dev];
    return SPEC_OK;
}

}  // namespace
}  // namespace specv

extern "C" int spec_accept_greedy_noalloc(const void* logits, int32_t logits_dtype,
                                          const int32_t* draft_tokens, int32_t batch,
                                          int32_t num_draft, int64_t vocab, int32_t* accepted_len,
                                          int32_t* next_token, void* stream) {
    using specv::set_error;
    set_error(SPEC_OK, "");
    if (batch < 0) return set_error(SPEC_ERR_INVALID, "batch < 0");
    if (num_draft < 1 || num_draft > 64)
        return set_error(SPEC_ERR_INVALID, "num_draft must be in [1, 64]");
    if (vocab < 1 || vocab >= (1LL << 31))
        return set_error(SPEC_ERR_INVALID, "vocab must be in [1, 2^31)");
    if (logits_dtype != SPEC_DTYPE_F32 && logits_dtype != SPEC_DTYPE_BF16)
        return set_error(SPEC_ERR_INVALID, "logits_dtype must be F32 or BF16");
    if (batch == 0) return SPEC_OK;
    if (!logits || !draft_tokens || !accepted_len || !next_token)
        return set_error(SPEC_ERR_INVALID, "null tensor pointer");
    if (reinterpret_cast<uintptr_t>(logits) & 15)
        return set_error(SPEC_ERR_INVALID, "logits must be 16-byte aligned");
    const int64_t parts = (int64_t)batch * (num_draft + 1) * specv::num_slices(vocab);
    if (batch > specv::kNoAllocMaxBatch || parts > specv::kNoAllocMaxPartials)
        return set_error(SPEC_ERR_UNSUPPORTED,
                         "too large for the fixed no-allocation scratch: needs batch <= "
                         "SPEC_NOALLOC_MAX_BATCH and batch * (num_draft + 1) * ceil(vocab / 8192) "
                         "<= SPEC_NOALLOC_MAX_PARTIALS");
    void* scratch = nullptr;
    const int rc = specv::noalloc_scratch(&scratch);
    if (rc) return rc;
    specv::AcceptArgs a;
    a.logits = logits;
    a.dtype = logits_dtype;
    a.draft = draft_tokens;
    a.B = batch;
    a.k = num_draft;
    a.V = vocab;
    a.accepted_len = accepted_len;
    a.next_token = next_token;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int32_t* tickets = reinterpret_cast<int32_t*>(static_cast<unsigned char*>(scratch) +
                                                  specv::kNoAllocPartialBytes);
    // the tickets must start at zero; the array keeps whatever the last call left
    cudaError_t e = cudaMemsetAsync(tickets, 0, sizeof(int32_t) * (size_t)batch, st);
    if (e == cudaSuccess) e = specv::launch_accept(a, scratch, tickets, st);
    if (e != cudaSuccess) return set_error(SPEC_ERR_CUDA, cudaGetErrorString(e));
    return SPEC_OK;
}

// Greedy longest-prefix acceptance ("Decoding Speculative Decoding from First
// Principles", "Speculating to get sequence parallelism during decode"): the
// target's prediction at each of the k+1 positions is the argmax of its
// logits row; drafts are kept up to the first disagreement and the target's
// own token there (or the bonus token after k agreements) is emitted.
//
// One launch.  Each CTA reduces one vocabulary slice of one logits row to a
// (max, lowest index) pair with 16-byte loads and warp shuffles, writes it to
// the workspace and takes a ticket of its sequence.  The CTA that takes the
// last ticket of a sequence merges that sequence's slices, runs the prefix
// match and resets the ticket, so no CTA ever waits on another.
#include <limits.h>

#include <mutex>

#include "common.cuh"

namespace specv {
namespace {

constexpr int kThreads = 256;
constexpr int kSlice = 8192;  // vocabulary entries per CTA

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

template <typename T>
__global__ void __launch_bounds__(kThreads)
accept_greedy_kernel(AcceptArgs a, int n_slices, float* __restrict__ part_v,
                     int* __restrict__ part_i, int32_t* __restrict__ tickets) {
    constexpr int VEC = 16 / sizeof(T);
    __shared__ float s_v[kThreads / 32];
    __shared__ int s_i[kThreads / 32];
    __shared__ int s_last;
    __shared__ int s_am[65];

    const int row = blockIdx.x / n_slices;  // row of [B, k+1]
    const int slice = blockIdx.x % n_slices;
    const int b = row / (a.k + 1);
    const int tid = threadIdx.x;
    const T* x = static_cast<const T*>(a.logits) + (int64_t)row * a.V;
    const int64_t e0 = (int64_t)slice * kSlice;
    const int64_t e1 = min(a.V, e0 + (int64_t)kSlice);

    float bv = -INFINITY;
    int bi = INT_MAX;
    // unaligned head, 16-byte body, tail: each thread visits its elements in
    // increasing index order
    const uintptr_t addr = reinterpret_cast<uintptr_t>(x + e0);
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

    warp_argmax(bv, bi);
    if ((tid & 31) == 0) { s_v[tid >> 5] = bv; s_i[tid >> 5] = bi; }
    __syncthreads();
    if (tid < 32) {
        bv = tid < kThreads / 32 ? s_v[tid] : -INFINITY;
        bi = tid < kThreads / 32 ? s_i[tid] : INT_MAX;
        warp_argmax(bv, bi);
        if (tid == 0) {
            part_v[blockIdx.x] = bv;
            part_i[blockIdx.x] = bi;
            __threadfence();
            const int t = atomicAdd(&tickets[b], 1);
            s_last = (t == (a.k + 1) * n_slices - 1);
        }
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();

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
    __syncthreads();
    if (tid == 0) {
        int n = 0;
        while (n < a.k && a.draft[(int64_t)b * a.k + n] == s_am[n]) ++n;
        a.accepted_len[b] = n;
        a.next_token[b] = s_am[n];
        tickets[b] = 0;  // ready for the next call
    }
}

int num_slices(int64_t V) { return (int)((V + kSlice - 1) / kSlice); }

}  // namespace

size_t accept_workspace_bytes(const AcceptArgs& a) {
    const int64_t parts = (int64_t)a.B * (a.k + 1) * num_slices(a.V);
    return (size_t)parts * (sizeof(float) + sizeof(int)) + 256;
}

cudaError_t launch_accept(const AcceptArgs& a, void* workspace, int32_t* tickets,
                          cudaStream_t stream) {
    if (a.B == 0) return cudaSuccess;
    const int ns = num_slices(a.V);
    const int64_t parts = (int64_t)a.B * (a.k + 1) * ns;
    float* pv = static_cast<float*>(workspace);
    int* pi = reinterpret_cast<int*>(pv + parts);
    if (a.dtype == SPEC_DTYPE_F32)
        accept_greedy_kernel<float><<<(unsigned)parts, kThreads, 0, stream>>>(a, ns, pv, pi, tickets);
    else
        accept_greedy_kernel<__nv_bfloat16>
            <<<(unsigned)parts, kThreads, 0, stream>>>(a, ns, pv, pi, tickets);
    return cudaGetLastError();
}

}  // namespace specv

// ---------------------------------------------------------------- no-allocation variant
//
// Greedy acceptance for callers that cannot allocate device memory: code that
// records the verification step into a CUDA graph (an allocation cannot be
// captured, and growing the library workspace synchronises the device), and
// serving loops whose device memory is reserved up front by their own
// allocator, where an extra cudaMalloc may fail or stall the step.  The
// reduction partials and completion tickets live in one fixed array of this
// file; every call on a device shares it.

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
// library's device code); later calls reuse the cached address.
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

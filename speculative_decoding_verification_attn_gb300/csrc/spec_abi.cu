// C ABI of the verification hot path: argument validation, the per-device
// workspace, path selection and launches on the caller's stream.  Every
// entry point returns a status code; on an error nothing is enqueued and the
// thread-local message says why.
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <atomic>
#include <initializer_list>
#include <mutex>
#include <string>
#include <vector>

#include "kernels.h"

namespace {

thread_local std::string g_err;

int fail(int code, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_err = buf;
    return code;
}

int cuda_fail(cudaError_t e, const char* what) {
    return fail(SPEC_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

std::atomic<int64_t> g_opt_path{0}, g_opt_ctas{0}, g_opt_validate{0}, g_opt_simt_chunk{0},
    g_opt_split{0}, g_opt_small_cluster{0};

// Per-device workspace: [error word | acceptance tickets | segment counters |
// scratch].  The header is zeroed at allocation; tickets and counters are
// reset by the kernels that use them.
constexpr size_t kHeader = 128 * 1024;
constexpr size_t kTicketsOff = 256, kCountersOff = 64 * 1024;
constexpr int kMaxTickets = (int)((kCountersOff - kTicketsOff) / 4);
constexpr int kMaxCounters = (int)((kHeader - kCountersOff) / 4);
struct Workspace {
    void* base = nullptr;
    size_t bytes = 0;
    int sms = 0;
};
std::mutex g_ws_mu;
std::vector<Workspace> g_ws;

// Returns the current device's workspace with at least `scratch` bytes of
// scratch space (allocating or growing it), or sets an error.
int get_workspace(size_t scratch, Workspace** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    std::lock_guard<std::mutex> lk(g_ws_mu);
    if ((int)g_ws.size() <= dev) g_ws.resize(dev + 1);
    Workspace& w = g_ws[dev];
    if (w.sms == 0) {
        e = cudaDeviceGetAttribute(&w.sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
    }
    const size_t need = kHeader + ((scratch + 255) & ~size_t(255));
    if (w.bytes < need) {
        if (w.base) {
            e = cudaDeviceSynchronize();  // earlier calls may still use the old buffer
            if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
            cudaFree(w.base);
            w.base = nullptr;
            w.bytes = 0;
        }
        size_t grow = need < (size_t)64 << 20 ? (size_t)64 << 20 : need;
        e = cudaMalloc(&w.base, grow);
        if (e != cudaSuccess) return cuda_fail(e, "cudaMalloc(workspace)");
        e = cudaMemset(w.base, 0, kHeader);
        if (e != cudaSuccess) return cuda_fail(e, "cudaMemset(workspace)");
        e = cudaDeviceSynchronize();
        if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
        w.bytes = grow;
    }
    *out = &w;
    return SPEC_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

int dtype_size(int32_t dt) {
    switch (dt) {
    case SPEC_DTYPE_F32: return 4;
    case SPEC_DTYPE_BF16: return 2;
    case SPEC_DTYPE_F16: return 2;
    case SPEC_DTYPE_I8: return 1;
    default: return 0;
    }
}

// Host-side check of block_table / ctx_lens (SPEC_OPT_VALIDATE).
int validate_tables(const specv::AttnArgs& a, cudaStream_t stream) {
    std::vector<int32_t> ctx(a.B), bt((size_t)a.B * a.max_pages);
    cudaError_t e = cudaMemcpyAsync(ctx.data(), a.ctx_lens, sizeof(int32_t) * a.B,
                                    cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(bt.data(), a.block_table, sizeof(int32_t) * bt.size(),
                            cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return cuda_fail(e, "validate: copy tables");
    for (int b = 0; b < a.B; ++b) {
        const int64_t L = (int64_t)ctx[b] + a.k;
        if (ctx[b] < 0 || L > (int64_t)a.max_pages * a.P)
            return fail(SPEC_ERR_INVALID, "ctx_lens[%d]=%d: ctx + num_draft exceeds the %d pages "
                        "of the block table", b, ctx[b], a.max_pages);
        const int64_t n = (L + a.P - 1) / a.P;
        for (int64_t p = 0; p < n; ++p) {
            const int32_t id = bt[(size_t)b * a.max_pages + p];
            if (id < 0 || id >= a.num_pages)
                return fail(SPEC_ERR_INVALID, "block_table[%d][%lld]=%d outside [0, %d)", b,
                            (long long)p, id, a.num_pages);
        }
    }
    return SPEC_OK;
}

}  // namespace

namespace specv {
// Records `msg` as this thread's last error and returns `code` (for entry
// points defined in other translation units).
int set_error(int code, const char* msg) { return fail(code, "%s", msg); }
}  // namespace specv

extern "C" {

int spec_version(void) { return 100; }

const char* spec_last_error(void) { return g_err.c_str(); }

int spec_set_option(int32_t option, int64_t value) {
    switch (option) {
    case SPEC_OPT_ATTN_PATH:
        if (value < 0 || value > 5)
            return fail(SPEC_ERR_INVALID, "attn path must be 0, 1, 2, 3, 4 or 5");
        g_opt_path = value;
        return SPEC_OK;
    case SPEC_OPT_NUM_CTAS:
        if (value < 0 || value > 65535) return fail(SPEC_ERR_INVALID, "num_ctas out of range");
        g_opt_ctas = value;
        return SPEC_OK;
    case SPEC_OPT_VALIDATE:
        g_opt_validate = value ? 1 : 0;
        return SPEC_OK;
    case SPEC_OPT_SIMT_CHUNK:
        if (value < 0 || value > (1 << 30)) return fail(SPEC_ERR_INVALID, "chunk out of range");
        g_opt_simt_chunk = value;
        return SPEC_OK;
    case SPEC_OPT_SPLIT_WEIGHT:
        if (value < 0 || value > 257) return fail(SPEC_ERR_INVALID, "split weight out of range");
        g_opt_split = value;
        return SPEC_OK;
    case SPEC_OPT_SMALL_CLUSTER:
        if (value < 0 || value > 8) return fail(SPEC_ERR_INVALID, "small cluster must be 0..8");
        g_opt_small_cluster = value;
        return SPEC_OK;
    default:
        return fail(SPEC_ERR_INVALID, "unknown option %d", option);
    }
}

}  // extern "C"

namespace {

int verify_attn_impl(const void* q, const void* k_cache, const void* v_cache, const void* k_scale,
                     const void* v_scale, const int32_t* block_table, const int32_t* ctx_lens,
                     const uint64_t* tree_mask, int32_t batch, int32_t num_draft,
                     int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                     int32_t page_size, int32_t num_pages, int32_t max_pages_per_seq,
                     int32_t q_dtype, int32_t kv_dtype, float scale, void* out, float* lse,
                     void* stream) {
    g_err.clear();
    if (batch < 0) return fail(SPEC_ERR_INVALID, "batch < 0");
    if (num_draft < 1 || num_draft > 64) return fail(SPEC_ERR_INVALID, "num_draft must be in [1, 64]");
    if (num_q_heads < 1 || num_kv_heads < 1 || num_q_heads % num_kv_heads)
        return fail(SPEC_ERR_INVALID, "num_q_heads must be a positive multiple of num_kv_heads");
    if (head_dim < 32 || head_dim > 256 || head_dim % 32)
        return fail(SPEC_ERR_INVALID, "head_dim must be a multiple of 32 in [32, 256]");
    if (page_size < 1) return fail(SPEC_ERR_INVALID, "page_size < 1");
    if (num_pages < 1 || max_pages_per_seq < 1)
        return fail(SPEC_ERR_INVALID, "num_pages and max_pages_per_seq must be >= 1");
    if (q_dtype != SPEC_DTYPE_F32 && q_dtype != SPEC_DTYPE_BF16)
        return fail(SPEC_ERR_INVALID, "q_dtype must be F32 or BF16");
    if (kv_dtype != SPEC_DTYPE_F32 && kv_dtype != SPEC_DTYPE_BF16 && kv_dtype != SPEC_DTYPE_I8)
        return fail(SPEC_ERR_INVALID, "kv_dtype must be F32, BF16 or I8");
    if (!(scale == scale)) return fail(SPEC_ERR_INVALID, "scale is NaN");
    if (batch == 0) return SPEC_OK;
    if (!q || !k_cache || !v_cache || !block_table || !ctx_lens || !out)
        return fail(SPEC_ERR_INVALID, "null tensor pointer");
    if (kv_dtype == SPEC_DTYPE_I8 && (!k_scale || !v_scale))
        return fail(SPEC_ERR_INVALID, "an I8 cache needs k_scale and v_scale");
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out))
        return fail(SPEC_ERR_INVALID, "q, caches and out must be 16-byte aligned");
    if ((int64_t)num_pages * num_kv_heads * page_size * head_dim >= (1LL << 40))
        return fail(SPEC_ERR_INVALID, "cache too large");
    const int64_t R = (int64_t)num_draft * (num_q_heads / num_kv_heads);
    (void)dtype_size;

    specv::AttnArgs a;
    a.q = q; a.k_cache = k_cache; a.v_cache = v_cache;
    a.k_scale = static_cast<const uint16_t*>(k_scale);
    a.v_scale = static_cast<const uint16_t*>(v_scale);
    a.block_table = block_table; a.ctx_lens = ctx_lens;
    a.B = batch; a.k = num_draft; a.Hq = num_q_heads; a.Hkv = num_kv_heads; a.D = head_dim;
    a.P = page_size; a.num_pages = num_pages; a.max_pages = max_pages_per_seq;
    a.q_dtype = q_dtype; a.kv_dtype = kv_dtype; a.scale = scale;
    a.out = out; a.lse = lse;
    a.dev_err = nullptr; a.seg_counters = nullptr;
    a.tree_mask = tree_mask;
    const int64_t split_opt = g_opt_split.load();
    a.split_alpha = split_opt > 0 ? (int32_t)(split_opt - 1) : -1;
    cudaStream_t st = static_cast<cudaStream_t>(stream);

    Workspace* ws = nullptr;
    int rc = get_workspace(0, &ws);
    if (rc) return rc;

    // kernels: 1 SIMT (chunked), 2 tcgen05 (64-key tiles), 3 warp MMA,
    // 4 single-pass SIMT, 5 tcgen05 (128-key tiles).  Automatic: a bf16
    // cache with head_dim 128 takes the 128-key tcgen05 kernel, except that
    // with <= 16 query rows per kv-head the warp-MMA kernel (whose pieces of
    // a split segment cost less) keeps the calls with more segments than SMs
    // and tables shorter than 3072 keys (about 24 tiles per segment, the
    // point where the two cross over when measured); the INT8 cache takes
    // the 64-key tcgen05 kernel; every other shape the single-pass SIMT
    // kernel when a whole sequence fits its shared memory, else the chunked one
    const int64_t path = g_opt_path.load();
    const bool tc_ok = specv::tc_supported(a), mma_ok = specv::mma_supported(a);
    const bool tc2_ok = specv::tc2_supported(a);
    const bool small_ok = specv::small_attn_max_keys(a) > 0;
    int kernel;
    if (path == 1) kernel = 1;
    else if (path >= 2) {
        if ((path == 2 && !tc_ok) || (path == 3 && !mma_ok) || (path == 4 && !small_ok) ||
            (path == 5 && !tc2_ok))
            return fail(SPEC_ERR_UNSUPPORTED, "forced attention kernel %d does not support this "
                        "shape/dtype", (int)path);
        kernel = (int)path;
    } else {
        const bool many_short = (int64_t)batch * num_kv_heads > ws->sms &&
                                (int64_t)max_pages_per_seq * page_size < 3072;
        const bool tc2_auto = tc2_ok && kv_dtype == SPEC_DTYPE_BF16;
        kernel = mma_ok && (many_short || !tc2_auto) ? 3 : tc2_auto ? 5 : tc_ok ? 2 : small_ok ? 4 : 1;
    }
    if (kernel == 3 && (int64_t)batch * num_kv_heads > kMaxCounters)
        return fail(SPEC_ERR_UNSUPPORTED, "batch * num_kv_heads > %d for the warp-MMA kernel",
                    kMaxCounters);
    const bool use_tc = kernel == 2 || kernel == 3 || kernel == 5;
    if (g_opt_validate.load()) {
        rc = validate_tables(a, st);
        if (rc) return rc;
    }
    cudaError_t e;
    if (use_tc) {
        int ctas = (int)g_opt_ctas.load();
        if (ctas <= 0) ctas = ws->sms;
        rc = get_workspace(specv::tc_workspace_bytes(a, ctas), &ws);
        if (rc) return rc;
        a.dev_err = static_cast<int*>(ws->base);
        a.seg_counters = reinterpret_cast<int*>(static_cast<char*>(ws->base) + kCountersOff);
        void* wsp = static_cast<char*>(ws->base) + kHeader;
        e = kernel == 3   ? specv::launch_attn_mma(a, ctas, wsp, st)
            : kernel == 5 ? specv::launch_attn_tc2(a, ctas, wsp, st)
                          : specv::launch_attn_tc(a, ctas, wsp, st);
        if (e != cudaSuccess) return cuda_fail(e, "verify_attn (tensor-core) launch");
    } else if (kernel == 4) {
        a.dev_err = static_cast<int*>(ws->base);
        e = specv::launch_attn_small(a, ws->sms, (int)g_opt_small_cluster.load(), st);
        if (e != cudaSuccess) return cuda_fail(e, "verify_attn (single-pass SIMT) launch");
    } else {
        const specv::SimtPlan p = specv::simt_plan(a, ws->sms, (int)g_opt_simt_chunk.load());
        const int64_t gy = (int64_t)batch * num_kv_heads * p.row_groups;
        if (gy > 65535 || R > (1 << 20))
            return fail(SPEC_ERR_UNSUPPORTED, "batch * num_kv_heads too large for the SIMT path");
        rc = get_workspace(specv::simt_workspace_bytes(a, p), &ws);
        if (rc) return rc;
        a.dev_err = static_cast<int*>(ws->base);
        e = specv::launch_attn_simt(a, p, static_cast<char*>(ws->base) + kHeader, st);
        if (e != cudaSuccess) return cuda_fail(e, "verify_attn (SIMT) launch");
    }
    return SPEC_OK;
}

}  // namespace

extern "C" {

int spec_verify_attn(const void* q, const void* k_cache, const void* v_cache, const void* k_scale,
                     const void* v_scale, const int32_t* block_table, const int32_t* ctx_lens,
                     int32_t batch, int32_t num_draft, int32_t num_q_heads, int32_t num_kv_heads,
                     int32_t head_dim, int32_t page_size, int32_t num_pages,
                     int32_t max_pages_per_seq, int32_t q_dtype, int32_t kv_dtype, float scale,
                     void* out, float* lse, void* stream) {
    return verify_attn_impl(q, k_cache, v_cache, k_scale, v_scale, block_table, ctx_lens, nullptr,
                            batch, num_draft, num_q_heads, num_kv_heads, head_dim, page_size,
                            num_pages, max_pages_per_seq, q_dtype, kv_dtype, scale, out, lse,
                            stream);
}

int spec_verify_attn_tree(const void* q, const void* k_cache, const void* v_cache,
                          const void* k_scale, const void* v_scale, const int32_t* block_table,
                          const int32_t* ctx_lens, const uint64_t* tree_mask, int32_t batch,
                          int32_t num_draft, int32_t num_q_heads, int32_t num_kv_heads,
                          int32_t head_dim, int32_t page_size, int32_t num_pages,
                          int32_t max_pages_per_seq, int32_t q_dtype, int32_t kv_dtype,
                          float scale, void* out, float* lse, void* stream) {
    if (batch > 0 && !tree_mask) return fail(SPEC_ERR_INVALID, "tree_mask is NULL");
    return verify_attn_impl(q, k_cache, v_cache, k_scale, v_scale, block_table, ctx_lens,
                            tree_mask, batch, num_draft, num_q_heads, num_kv_heads, head_dim,
                            page_size, num_pages, max_pages_per_seq, q_dtype, kv_dtype, scale,
                            out, lse, stream);
}

}  // extern "C"

namespace {

int accept_greedy_impl(const void* logits, int32_t logits_dtype, const int32_t* draft_tokens,
                       const int32_t* parents, int32_t batch, int32_t num_draft, int64_t vocab,
                       int32_t* accepted_len, int32_t* next_token, int32_t* path, void* stream) {
    g_err.clear();
    if (batch < 0) return fail(SPEC_ERR_INVALID, "batch < 0");
    if (num_draft < 1 || num_draft > 64) return fail(SPEC_ERR_INVALID, "num_draft must be in [1, 64]");
    if (vocab < 1 || vocab >= (1LL << 31)) return fail(SPEC_ERR_INVALID, "vocab must be in [1, 2^31)");
    if (logits_dtype != SPEC_DTYPE_F32 && logits_dtype != SPEC_DTYPE_BF16)
        return fail(SPEC_ERR_INVALID, "logits_dtype must be F32 or BF16");
    if (batch == 0) return SPEC_OK;
    if (batch > kMaxTickets) return fail(SPEC_ERR_UNSUPPORTED, "batch > %d", kMaxTickets);
    if (!logits || !draft_tokens || !accepted_len || !next_token)
        return fail(SPEC_ERR_INVALID, "null tensor pointer");
    if (!aligned16(logits)) return fail(SPEC_ERR_INVALID, "logits must be 16-byte aligned");
    specv::AcceptArgs a;
    a.logits = logits; a.dtype = logits_dtype; a.draft = draft_tokens; a.B = batch;
    a.k = num_draft; a.V = vocab; a.accepted_len = accepted_len; a.next_token = next_token;
    a.parent = parents; a.path = path;
    const int64_t blocks = (int64_t)batch * (num_draft + 1) * ((vocab + 8191) / 8192);
    if (blocks >= (1LL << 31)) return fail(SPEC_ERR_UNSUPPORTED, "logits too large");
    Workspace* ws = nullptr;
    int rc = get_workspace(specv::accept_workspace_bytes(a), &ws);
    if (rc) return rc;
    a.dev_err = static_cast<int*>(ws->base);
    int32_t* tickets = reinterpret_cast<int32_t*>(static_cast<char*>(ws->base) + kTicketsOff);
    cudaError_t e = specv::launch_accept(a, static_cast<char*>(ws->base) + kHeader, tickets,
                                         static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "accept_greedy launch");
    return SPEC_OK;
}

}  // namespace

extern "C" {

int spec_accept_greedy(const void* logits, int32_t logits_dtype, const int32_t* draft_tokens,
                       int32_t batch, int32_t num_draft, int64_t vocab, int32_t* accepted_len,
                       int32_t* next_token, void* stream) {
    return accept_greedy_impl(logits, logits_dtype, draft_tokens, nullptr, batch, num_draft, vocab,
                              accepted_len, next_token, nullptr, stream);
}

int spec_accept_tree(const void* logits, int32_t logits_dtype, const int32_t* draft_tokens,
                     const int32_t* parents, int32_t batch, int32_t num_draft, int64_t vocab,
                     int32_t* accepted_len, int32_t* next_token, int32_t* path, void* stream) {
    if (batch > 0 && !parents) return fail(SPEC_ERR_INVALID, "parents is NULL");
    return accept_greedy_impl(logits, logits_dtype, draft_tokens, parents, batch, num_draft,
                              vocab, accepted_len, next_token, path, stream);
}

int spec_accept_rejection(const void* target_logits, const void* draft_logits,
                          int32_t logits_dtype, const int32_t* draft_tokens, int32_t batch,
                          int32_t num_draft, int64_t vocab, float temperature, uint64_t seed,
                          int32_t* accepted_len, int32_t* next_token, void* stream) {
    g_err.clear();
    if (batch < 0) return fail(SPEC_ERR_INVALID, "batch < 0");
    if (num_draft < 1 || num_draft > 64) return fail(SPEC_ERR_INVALID, "num_draft must be in [1, 64]");
    if (vocab < 1 || vocab >= (1LL << 31)) return fail(SPEC_ERR_INVALID, "vocab must be in [1, 2^31)");
    if (logits_dtype != SPEC_DTYPE_F32 && logits_dtype != SPEC_DTYPE_BF16)
        return fail(SPEC_ERR_INVALID, "logits_dtype must be F32 or BF16");
    if (!(temperature > 0.f) || !(temperature < INFINITY))
        return fail(SPEC_ERR_INVALID, "temperature must be positive and finite");
    if (batch == 0) return SPEC_OK;
    if (batch > kMaxTickets) return fail(SPEC_ERR_UNSUPPORTED, "batch > %d", kMaxTickets);
    if (!target_logits || !draft_logits || !draft_tokens || !accepted_len || !next_token)
        return fail(SPEC_ERR_INVALID, "null tensor pointer");
    if (!aligned16(target_logits) || !aligned16(draft_logits))
        return fail(SPEC_ERR_INVALID, "logits must be 16-byte aligned");
    const int64_t units = (int64_t)batch * (2 * num_draft + 1) * ((vocab + 2047) / 2048);
    if (units >= (1LL << 31)) return fail(SPEC_ERR_UNSUPPORTED, "logits too large");
    Workspace* ws = nullptr;
    int rc = get_workspace(specv::rejection_workspace_bytes(batch, num_draft, vocab), &ws);
    if (rc) return rc;
    int32_t* tickets = reinterpret_cast<int32_t*>(static_cast<char*>(ws->base) + kTicketsOff);
    cudaError_t e = specv::launch_accept_rejection(
        target_logits, draft_logits, logits_dtype, draft_tokens, batch, num_draft, vocab,
        temperature, seed, accepted_len, next_token, static_cast<char*>(ws->base) + kHeader,
        tickets, static_cast<int*>(ws->base), static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "accept_rejection launch");
    return SPEC_OK;
}

int spec_kv_append(const void* k_new, const void* v_new, int32_t src_dtype, void* k_cache,
                   void* v_cache, void* k_scale, void* v_scale, int32_t cache_dtype,
                   const int32_t* block_table, const int32_t* ctx_lens, int32_t batch,
                   int32_t num_new, int32_t num_kv_heads, int32_t head_dim, int32_t page_size,
                   int32_t num_pages, int32_t max_pages_per_seq, void* stream) {
    g_err.clear();
    if (batch < 0) return fail(SPEC_ERR_INVALID, "batch < 0");
    if (num_new < 1) return fail(SPEC_ERR_INVALID, "num_new must be >= 1");
    if (num_kv_heads < 1) return fail(SPEC_ERR_INVALID, "num_kv_heads must be >= 1");
    if (head_dim < 32 || head_dim > 256 || head_dim % 32)
        return fail(SPEC_ERR_INVALID, "head_dim must be a multiple of 32 in [32, 256]");
    if (page_size < 1) return fail(SPEC_ERR_INVALID, "page_size < 1");
    if (num_pages < 1 || max_pages_per_seq < 1)
        return fail(SPEC_ERR_INVALID, "num_pages and max_pages_per_seq must be >= 1");
    if (src_dtype != SPEC_DTYPE_F32 && src_dtype != SPEC_DTYPE_BF16)
        return fail(SPEC_ERR_INVALID, "src_dtype must be F32 or BF16");
    if (cache_dtype != SPEC_DTYPE_F32 && cache_dtype != SPEC_DTYPE_BF16 &&
        cache_dtype != SPEC_DTYPE_I8)
        return fail(SPEC_ERR_INVALID, "cache_dtype must be F32, BF16 or I8");
    if (batch == 0) return SPEC_OK;
    if (!k_new || !v_new || !k_cache || !v_cache || !block_table || !ctx_lens)
        return fail(SPEC_ERR_INVALID, "null tensor pointer");
    if (cache_dtype == SPEC_DTYPE_I8 && (!k_scale || !v_scale))
        return fail(SPEC_ERR_INVALID, "an I8 cache needs k_scale and v_scale");
    if ((int64_t)batch * num_new * num_kv_heads * 2 / 8 >= (1LL << 31))
        return fail(SPEC_ERR_UNSUPPORTED, "too many rows");
    Workspace* ws = nullptr;
    int rc = get_workspace(0, &ws);
    if (rc) return rc;
    cudaError_t e = specv::launch_kv_append(
        k_new, v_new, src_dtype, k_cache, v_cache, static_cast<uint16_t*>(k_scale),
        static_cast<uint16_t*>(v_scale), cache_dtype, block_table, ctx_lens, batch, num_new,
        num_kv_heads, head_dim, page_size, num_pages, max_pages_per_seq,
        static_cast<int*>(ws->base), static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "kv_append launch");
    return SPEC_OK;
}

static int codec_args(int64_t num_blocks, int32_t page_size, int32_t head_dim) {
    if (num_blocks < 0) return fail(SPEC_ERR_INVALID, "num_blocks < 0");
    if (head_dim < 32 || head_dim > 256 || head_dim % 32)
        return fail(SPEC_ERR_INVALID, "head_dim must be a multiple of 32 in [32, 256]");
    if (page_size < 1 || (int64_t)page_size * head_dim > 16384)
        return fail(SPEC_ERR_INVALID, "page_size must be >= 1 with page_size * head_dim <= 16384");
    if (num_blocks / 8 >= (1LL << 31)) return fail(SPEC_ERR_UNSUPPORTED, "too many blocks");
    return SPEC_OK;
}

int spec_codec_encode(const void* codes, int64_t num_blocks, int32_t page_size, int32_t head_dim,
                      void* pairs, int32_t* num_pairs, void* stream) {
    g_err.clear();
    int rc = codec_args(num_blocks, page_size, head_dim);
    if (rc) return rc;
    if (num_blocks == 0) return SPEC_OK;
    if (!codes || !pairs || !num_pairs) return fail(SPEC_ERR_INVALID, "null tensor pointer");
    cudaError_t e = specv::launch_codec_encode(codes, num_blocks, page_size, head_dim, pairs,
                                               num_pairs, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "codec_encode launch");
    return SPEC_OK;
}

int spec_codec_decode(const void* pairs, const int32_t* num_pairs, int64_t num_blocks,
                      int32_t page_size, int32_t head_dim, void* codes, void* stream) {
    g_err.clear();
    int rc = codec_args(num_blocks, page_size, head_dim);
    if (rc) return rc;
    if (num_blocks == 0) return SPEC_OK;
    if (!codes || !pairs || !num_pairs) return fail(SPEC_ERR_INVALID, "null tensor pointer");
    if ((reinterpret_cast<uintptr_t>(pairs) & 15) || (reinterpret_cast<uintptr_t>(codes) & 15))
        return fail(SPEC_ERR_INVALID, "pairs and codes must be 16-byte aligned");
    Workspace* ws = nullptr;
    rc = get_workspace(0, &ws);
    if (rc) return rc;
    cudaError_t e = specv::launch_codec_decode(pairs, num_pairs, num_blocks, page_size, head_dim,
                                               codes, static_cast<int*>(ws->base),
                                               static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "codec_decode launch");
    return SPEC_OK;
}

int spec_commit(int32_t* ctx_lens, const int32_t* accepted_len, int32_t batch, int32_t extra,
                void* stream) {
    g_err.clear();
    if (batch < 0) return fail(SPEC_ERR_INVALID, "batch < 0");
    if (batch == 0) return SPEC_OK;
    if (!ctx_lens || !accepted_len) return fail(SPEC_ERR_INVALID, "null tensor pointer");
    cudaError_t e = specv::launch_commit(ctx_lens, accepted_len, batch, extra,
                                         static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "commit launch");
    return SPEC_OK;
}

int spec_device_error(int32_t* flags) {
    g_err.clear();
    if (!flags) return fail(SPEC_ERR_INVALID, "flags is NULL");
    Workspace* ws = nullptr;
    int rc = get_workspace(0, &ws);
    if (rc) return rc;
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
    int v = 0;
    e = cudaMemcpy(&v, ws->base, sizeof(int), cudaMemcpyDeviceToHost);
    if (e == cudaSuccess) e = cudaMemset(ws->base, 0, sizeof(int));
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e, "read device error word");
    *flags = v;
    return SPEC_OK;
}

int spec_release(void) {
    g_err.clear();
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    std::lock_guard<std::mutex> lk(g_ws_mu);
    if ((int)g_ws.size() > dev && g_ws[dev].base) {
        e = cudaDeviceSynchronize();
        if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
        cudaFree(g_ws[dev].base);
        g_ws[dev].base = nullptr;
        g_ws[dev].bytes = 0;
    }
    return SPEC_OK;
}

}  // extern "C"

// ---------------------------------------------------------------- tensor-descriptor form
//
// The same two calls taking self-describing tensors (pointer, element type,
// rank, shape, strides in elements): the descriptors are checked against
// one another and forwarded to the flat entry points above.  The kernels
// read dense row-major tensors, so any other stride is refused (-2).

namespace {

// Dense row-major strides of `t` (in elements) match the given ones?
bool dense(const spec_tensor_t& t) {
    int64_t s = 1;
    for (int d = t.ndim - 1; d >= 0; --d) {
        if (t.shape[d] != 1 && t.stride[d] != s) return false;
        s *= t.shape[d];
    }
    return true;
}

// Checks rank, element type, shape (-1 = any), alignment and density of a
// descriptor; returns 0 or sets the error.
int check_tensor(const spec_tensor_t* t, const char* name, int ndim, std::initializer_list<int32_t> dtypes,
                 std::initializer_list<int64_t> shape, bool need16 = false) {
    if (!t) return fail(SPEC_ERR_INVALID, "%s: null descriptor", name);
    if (t->ndim != ndim) return fail(SPEC_ERR_INVALID, "%s: rank %d, expected %d", name, t->ndim, ndim);
    bool ok = false;
    for (int32_t dt : dtypes) ok = ok || t->dtype == dt;
    if (!ok) return fail(SPEC_ERR_INVALID, "%s: unsupported element type %d", name, t->dtype);
    int d = 0;
    for (int64_t want : shape) {
        if (t->shape[d] < 0 || (want >= 0 && t->shape[d] != want))
            return fail(SPEC_ERR_INVALID, "%s: dimension %d is %lld, expected %lld", name, d,
                        (long long)t->shape[d], (long long)want);
        ++d;
    }
    if (need16 && (reinterpret_cast<uintptr_t>(t->data) & 15))
        return fail(SPEC_ERR_INVALID, "%s: data must be 16-byte aligned", name);
    if (!dense(*t))
        return fail(SPEC_ERR_UNSUPPORTED, "%s: only dense row-major strides are supported", name);
    return SPEC_OK;
}

bool fits_i32(int64_t v) { return v >= 0 && v < (1LL << 31); }

}  // namespace

extern "C" {

int spec_verify_attn_tensors(const spec_tensor_t* q, const spec_tensor_t* k_cache,
                             const spec_tensor_t* v_cache, const spec_tensor_t* k_scale,
                             const spec_tensor_t* v_scale, const spec_tensor_t* block_table,
                             const spec_tensor_t* ctx_lens, int32_t num_draft, float scale,
                             spec_tensor_t* out, spec_tensor_t* lse, void* stream) {
    g_err.clear();
    int rc = check_tensor(q, "q", 4, {SPEC_DTYPE_F32, SPEC_DTYPE_BF16}, {-1, num_draft, -1, -1}, true);
    if (rc) return rc;
    const int64_t B = q->shape[0], Hq = q->shape[2], D = q->shape[3];
    rc = check_tensor(k_cache, "k_cache", 4, {SPEC_DTYPE_F32, SPEC_DTYPE_BF16, SPEC_DTYPE_I8},
                      {-1, -1, -1, D}, true);
    if (rc) return rc;
    const int64_t NP = k_cache->shape[0], Hkv = k_cache->shape[1], P = k_cache->shape[2];
    rc = check_tensor(v_cache, "v_cache", 4, {k_cache->dtype}, {NP, Hkv, P, D}, true);
    if (rc) return rc;
    const bool i8 = k_cache->dtype == SPEC_DTYPE_I8;
    if (i8) {
        rc = check_tensor(k_scale, "k_scale", 3, {SPEC_DTYPE_F16}, {NP, Hkv, P});
        if (!rc) rc = check_tensor(v_scale, "v_scale", 3, {SPEC_DTYPE_F16}, {NP, Hkv, P});
        if (rc) return rc;
    }
    rc = check_tensor(block_table, "block_table", 2, {SPEC_DTYPE_I32}, {B, -1});
    if (!rc) rc = check_tensor(ctx_lens, "ctx_lens", 1, {SPEC_DTYPE_I32}, {B});
    if (!rc) rc = check_tensor(out, "out", 4, {q->dtype}, {B, num_draft, Hq, D}, true);
    if (!rc && lse) rc = check_tensor(lse, "lse", 3, {SPEC_DTYPE_F32}, {B, num_draft, Hq});
    if (rc) return rc;
    const int64_t MP = block_table->shape[1];
    if (!fits_i32(B) || !fits_i32(Hq) || !fits_i32(D) || !fits_i32(NP) || !fits_i32(Hkv) ||
        !fits_i32(P) || !fits_i32(MP))
        return fail(SPEC_ERR_INVALID, "a dimension does not fit int32");
    return spec_verify_attn(q->data, k_cache->data, v_cache->data, i8 ? k_scale->data : nullptr,
                            i8 ? v_scale->data : nullptr,
                            static_cast<const int32_t*>(block_table->data),
                            static_cast<const int32_t*>(ctx_lens->data), (int32_t)B, num_draft,
                            (int32_t)Hq, (int32_t)Hkv, (int32_t)D, (int32_t)P, (int32_t)NP,
                            (int32_t)MP, q->dtype, k_cache->dtype, scale, out->data,
                            lse ? static_cast<float*>(lse->data) : nullptr, stream);
}

int spec_accept_greedy_tensors(const spec_tensor_t* logits, const spec_tensor_t* draft_tokens,
                               int32_t num_draft, spec_tensor_t* accepted_len,
                               spec_tensor_t* next_token, void* stream) {
    g_err.clear();
    int rc = check_tensor(logits, "logits", 3, {SPEC_DTYPE_F32, SPEC_DTYPE_BF16},
                          {-1, (int64_t)num_draft + 1, -1}, true);
    if (rc) return rc;
    const int64_t B = logits->shape[0];
    rc = check_tensor(draft_tokens, "draft_tokens", 2, {SPEC_DTYPE_I32}, {B, num_draft});
    if (!rc) rc = check_tensor(accepted_len, "accepted_len", 1, {SPEC_DTYPE_I32}, {B});
    if (!rc) rc = check_tensor(next_token, "next_token", 1, {SPEC_DTYPE_I32}, {B});
    if (rc) return rc;
    if (!fits_i32(B)) return fail(SPEC_ERR_INVALID, "batch does not fit int32");
    return spec_accept_greedy(logits->data, logits->dtype,
                              static_cast<const int32_t*>(draft_tokens->data), (int32_t)B,
                              num_draft, logits->shape[2],
                              static_cast<int32_t*>(accepted_len->data),
                              static_cast<int32_t*>(next_token->data), stream);
}

}  // extern "C"

/*
 * spec_verify.h -- C ABI of the GB300 (sm_103a) verification hot path of
 * speculative decoding.
 *
 * The target model verifies k drafted tokens in one prefill-style pass
 * ("Decoding Speculative Decoding from First Principles", sections
 * "Parallelizing method 2: sequence parallel" and "Speculating to get
 * sequence parallelism during decode"; HeteroReason, "Phase 2: Speculating
 * and Verification", single-step parallel verification).  Two operations
 * make up that pass's data-parallel core:
 *
 *   spec_verify_attn    multi-query causal attention of each sequence's k
 *                       draft queries over its paged KV cache (GQA, optional
 *                       INT8 cache with per-(token, kv-head) fp16 scales as
 *                       produced by CXL-SpecKV's "Algorithm 2 KV-Cache
 *                       Compression");
 *   spec_accept_greedy  greedy longest-prefix acceptance: the accepted length
 *                       and the next (correction or bonus) token.
 *
 * Conventions shared by every call
 *   - All tensor pointers are DEVICE pointers (cudaMalloc'd, managed or
 *     otherwise device-accessible), dense row-major with the shapes given.
 *     The caller owns every tensor; the library never frees them.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Calls are
 *     asynchronous: they enqueue kernels and return without synchronising.
 *   - Return value: SPEC_OK (0) or a negative SPEC_ERR_* code.  On an error
 *     nothing is enqueued and spec_last_error() (thread-local) describes it.
 *   - The library owns a per-device workspace (split-KV partials, reduction
 *     partials, completion tickets, an error word), grown on demand with
 *     cudaMalloc on the first call that needs more (so a call that grows it
 *     synchronises the device) and kept until spec_release() or exit.
 *     Calls that overlap on the GPU (different streams without ordering)
 *     share it and race: order them on one stream, or serialise them.
 *   - Device-side input faults (a block_table entry outside [0, num_pages),
 *     a context longer than the block table covers) never fault the GPU:
 *     the kernels clamp the reference, set the device error word and carry
 *     on; spec_device_error() reads (and clears) that word.
 */
#ifndef SPEC_VERIFY_H
#define SPEC_VERIFY_H

#include <stdint.h>

#if defined(__GNUC__)
#define SPEC_API __attribute__((visibility("default")))
#else
#define SPEC_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Element types. */
enum {
    SPEC_DTYPE_F32 = 0,
    SPEC_DTYPE_BF16 = 1,
    SPEC_DTYPE_F16 = 2, /* scales only */
    SPEC_DTYPE_I8 = 3,
    SPEC_DTYPE_I32 = 4  /* tables, lengths and token ids (descriptor form) */
};

/* A tensor described by itself (the descriptor form of the two hot-path
 * calls): device pointer, element type, rank (<= 4), shape and strides, both
 * in elements, row-major order of dimensions.  The caller owns `data`. */
typedef struct {
    void *data;
    int32_t dtype;
    int32_t ndim;
    int64_t shape[4];
    int64_t stride[4];
} spec_tensor_t;

/* Status codes. */
enum {
    SPEC_OK = 0,
    SPEC_ERR_INVALID = -1,     /* bad pointer, shape, dtype or alignment */
    SPEC_ERR_UNSUPPORTED = -2, /* valid but not implemented (e.g. forced path) */
    SPEC_ERR_CUDA = -3         /* a CUDA call failed; message has the CUDA error */
};

/* Options for spec_set_option (process-wide; default 0 = automatic). */
enum {
    /* 0 auto, 1 SIMT (CUDA cores) kernel with split-KV chunks, 2 tcgen05
     * kernel (64-key tiles), 3 warp-MMA (mma.sync) kernel for <= 16 query
     * rows per kv-head, 4 single-pass SIMT kernel (whole sequences in shared
     * memory), 5 tcgen05 kernel with 128-key tiles (bf16 query and cache,
     * head_dim 128, up to 128 query rows per kv-head, power-of-two pages of
     * 16..256 keys) */
    SPEC_OPT_ATTN_PATH = 0,
    /* persistent CTAs of the tensor-core kernel; 0 = number of SMs */
    SPEC_OPT_NUM_CTAS = 1,
    /* 1: copy block_table and ctx_lens to the host and check them before
     * launching (synchronises the stream); 0: no host check */
    SPEC_OPT_VALIDATE = 2,
    /* key chunk of the SIMT kernel's split-KV; 0 = automatic */
    SPEC_OPT_SIMT_CHUNK = 3,
    /* tensor-core kernels: tiles charged per (sequence, kv-head) segment when
     * the tile list is split over the persistent CTAs (a segment piece's
     * fixed work); 0 = each kernel's default, v in [1, 257] = v - 1 tiles */
    SPEC_OPT_SPLIT_WEIGHT = 4,
    /* single-pass SIMT kernel: CTAs (one thread-block cluster) that share each
     * (sequence, kv-head, query-row group), merging their softmax states
     * through distributed shared memory; 0 = automatic (a cluster of up to 8
     * while the clusters fit the SMs and every CTA keeps >= 16 keys of the
     * block table; one CTA when the device cannot place it), 1..8 = forced
     * (a cluster the device cannot place fails the call with SPEC_ERR_CUDA) */
    SPEC_OPT_SMALL_CLUSTER = 5
};

/* Library version, major*10000 + minor*100 + patch. */
SPEC_API int spec_version(void);

/* Message of the last failed call on this thread ("" if none). */
SPEC_API const char *spec_last_error(void);

/* Set a process-wide option (see SPEC_OPT_*).  Returns SPEC_OK or
 * SPEC_ERR_INVALID for an unknown option or value. */
SPEC_API int spec_set_option(int32_t option, int64_t value);

/*
 * Verification attention.
 *
 * For sequence b, draft position i (query at absolute position ctx_b + i)
 * and query head h served by kv-head g = h / (num_q_heads / num_kv_heads):
 *   s_j  = scale * <q[b,i,h,:], K_j>        for keys j = 0 .. ctx_b + i
 *   lse  = ln sum_j exp(s_j)
 *   out  = sum_j exp(s_j - lse) * V_j
 * where key j lives in physical page block_table[b, j / page_size], slot
 * j % page_size.  The k draft keys (positions ctx_b .. ctx_b + k - 1) must
 * already be in the cache; this call only reads it.
 *
 *   q            [batch, num_draft, num_q_heads, head_dim]   q_dtype (F32|BF16)
 *   k_cache,
 *   v_cache      [num_pages, num_kv_heads, page_size, head_dim]  kv_dtype
 *                (F32 | BF16 | I8).  With I8 the element is c * s.
 *   k_scale,
 *   v_scale      [num_pages, num_kv_heads, page_size] fp16; required with
 *                I8, ignored (may be NULL) otherwise
 *   block_table  [batch, max_pages_per_seq] int32 physical page ids
 *   ctx_lens     [batch] int32 cached context per sequence, EXCLUDING the
 *                drafts; ctx_b + num_draft <= max_pages_per_seq * page_size
 *   scale        softmax scale (typically 1/sqrt(head_dim))
 *   out          [batch, num_draft, num_q_heads, head_dim] in q_dtype
 *   lse          [batch, num_draft, num_q_heads] fp32 natural log, or NULL
 *
 * Limits: 1 <= num_draft <= 64; num_q_heads % num_kv_heads == 0;
 * head_dim % 32 == 0 and head_dim <= 256; page_size >= 1; q, caches and out
 * 16-byte aligned.  A bf16 query over a bf16 cache with head_dim 128, a
 * power-of-two page_size in [16, 256] and batch <= 1024 runs on a
 * tensor-core kernel: the warp-MMA kernel when num_draft * (num_q_heads /
 * num_kv_heads) <= 16, the tcgen05 kernel up to 128.  Every other accepted
 * shape runs on the CUDA cores: in one launch when every sequence's keys
 * (max_pages_per_seq * page_size of them) fit the single-pass kernel's
 * shared memory, else on the chunked split-KV kernel and its combine.
 */
SPEC_API int spec_verify_attn(const void *q, const void *k_cache, const void *v_cache,
                     const void *k_scale, const void *v_scale,
                     const int32_t *block_table, const int32_t *ctx_lens,
                     int32_t batch, int32_t num_draft, int32_t num_q_heads,
                     int32_t num_kv_heads, int32_t head_dim, int32_t page_size,
                     int32_t num_pages, int32_t max_pages_per_seq,
                     int32_t q_dtype, int32_t kv_dtype, float scale,
                     void *out, float *lse, void *stream);

/*
 * Greedy acceptance.
 *
 * For sequence b let a_i = argmax_v logits[b, i, v] (lowest index on ties;
 * values compare as stored, so -0 == +0), i = 0 .. num_draft.  Then
 *   accepted_len[b] = the largest n <= num_draft with
 *                     draft_tokens[b, 0..n-1] == a_0..a_{n-1}
 *   next_token[b]   = a_{accepted_len[b]}  (the target's own token at the
 *                     first disagreement, or the bonus token after k
 *                     agreements)
 * so each sequence gains accepted_len[b] + 1 tokens ("Decoding Speculative
 * Decoding from First Principles", "Speculating to get sequence parallelism
 * during decode").  The caller commits by ctx_b += accepted_len[b] + 1.
 *
 *   logits        [batch, num_draft + 1, vocab]  logits_dtype (F32|BF16),
 *                 finite values (a NaN row has no defined argmax)
 *   draft_tokens  [batch, num_draft] int32
 *   accepted_len  [batch] int32, written
 *   next_token    [batch] int32, written
 *
 * Limits: 1 <= num_draft <= 64; 1 <= vocab < 2^31; logits 16-byte aligned.
 */
SPEC_API int spec_accept_greedy(const void *logits, int32_t logits_dtype, const int32_t *draft_tokens,
                       int32_t batch, int32_t num_draft, int64_t vocab,
                       int32_t *accepted_len, int32_t *next_token, void *stream);

/*
 * Descriptor form of spec_verify_attn and spec_accept_greedy.  Same
 * operations, results, limits and stream behaviour; every tensor comes as a
 * spec_tensor_t and the sizes are read from the descriptors:
 *   q [B, num_draft, Hq, D] (F32 | BF16), k_cache / v_cache [NP, Hkv, P, D]
 *   (F32 | BF16 | I8, same type), k_scale / v_scale [NP, Hkv, P] F16 (I8
 *   cache only, else ignored), block_table [B, max_pages] I32, ctx_lens [B]
 *   I32, out [B, num_draft, Hq, D] in q's type, lse [B, num_draft, Hq] F32
 *   or NULL;
 *   logits [B, num_draft + 1, V] (F32 | BF16), draft_tokens [B, num_draft]
 *   I32, accepted_len / next_token [B] I32.
 * Errors: SPEC_ERR_INVALID for a null descriptor, a wrong rank, element
 * type or size, or a q / cache / out / logits pointer not 16-byte aligned;
 * SPEC_ERR_UNSUPPORTED for strides other than dense row-major (the kernels
 * read dense tensors); then whatever the flat call returns.  Nothing is
 * enqueued on an error.
 */
SPEC_API int spec_verify_attn_tensors(const spec_tensor_t *q, const spec_tensor_t *k_cache,
                                      const spec_tensor_t *v_cache, const spec_tensor_t *k_scale,
                                      const spec_tensor_t *v_scale,
                                      const spec_tensor_t *block_table,
                                      const spec_tensor_t *ctx_lens, int32_t num_draft,
                                      float scale, spec_tensor_t *out, spec_tensor_t *lse,
                                      void *stream);
SPEC_API int spec_accept_greedy_tensors(const spec_tensor_t *logits,
                                        const spec_tensor_t *draft_tokens, int32_t num_draft,
                                        spec_tensor_t *accepted_len, spec_tensor_t *next_token,
                                        void *stream);

/*
 * Verification attention over a tree of drafts (token trees verified in one
 * pass: "Decoding Speculative Decoding from First Principles", section
 * "Advances in speculators").  Same arguments and results as
 * spec_verify_attn, except that draft query i of sequence b sees the whole
 * cached context and the draft keys t (position ctx_b + t) whose bit t is
 * set in tree_mask[b, i] (uint64 [batch, num_draft], device memory) -- for a
 * tree, node i's ancestors and itself.  The causal chain is the mask with
 * bits 0..i.  Runs on the same kernels as spec_verify_attn.
 */
SPEC_API int spec_verify_attn_tree(const void *q, const void *k_cache, const void *v_cache,
                                   const void *k_scale, const void *v_scale,
                                   const int32_t *block_table, const int32_t *ctx_lens,
                                   const uint64_t *tree_mask, int32_t batch, int32_t num_draft,
                                   int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                   int32_t page_size, int32_t num_pages,
                                   int32_t max_pages_per_seq, int32_t q_dtype, int32_t kv_dtype,
                                   float scale, void *out, float *lse, void *stream);

/*
 * Greedy acceptance over a tree of drafts.  Node i of sequence b carries
 * draft_tokens[b, i] and parents[b, i] in [-1, i) (-1: a child of the last
 * committed token); logits row 0 is the target's prediction at the root and
 * row i + 1 its prediction after node i ([batch, num_draft + 1, vocab]).
 * From the root, the walk keeps the lowest-index child whose token equals
 * the target's argmax at the current node (lowest vocabulary index on
 * ties), and stops when no child does:
 *   accepted_len[b] = number of kept nodes,
 *   next_token[b]   = the target's argmax after the last kept node,
 *   path[b, :]      = the kept nodes in order, -1 after them (path may be
 *                     NULL).
 * A chain (parents[b, i] = i - 1) gives spec_accept_greedy's results.  A
 * parent outside [-1, i) makes its node unreachable and sets
 * SPEC_DEVERR_TREE.  Limits as spec_accept_greedy.
 */
SPEC_API int spec_accept_tree(const void *logits, int32_t logits_dtype,
                              const int32_t *draft_tokens, const int32_t *parents, int32_t batch,
                              int32_t num_draft, int64_t vocab, int32_t *accepted_len,
                              int32_t *next_token, int32_t *path, void *stream);

/*
 * Delta + run-length coding of INT8 KV pages (CXL-SpecKV: key observation
 * (5), delta coding delta_i = x_i - x_(i-1) of neighbouring elements of a
 * head vector, and "Algorithm 2 KV-Cache Compression", whose output is
 * (s, D_RLE(c))).  Lossless; the fp16 scales are not coded.
 *
 *   codes      [num_blocks, page_size, head_dim] int8: one block per
 *              (page, kv-head), i.e. an INT8 cache [num_pages, Hkv, P, D]
 *              with num_blocks = num_pages * Hkv
 *   pairs      [num_blocks, 2 * page_size * head_dim] uint8: block i's
 *              (length, value) byte pairs from byte 2*P*D*i (room for the
 *              worst case, every run of length one); 16-byte aligned
 *   num_pairs  [num_blocks] int32: pairs of each block
 *
 * Format: in each row of a block, e[0] = c[0] and e[d] = c[d] - c[d-1]
 * modulo 256; the block's row-major stream e becomes maximal runs of equal
 * bytes, each the pair (length 1..255, value), a longer run continuing in the
 * next pair.  Encode writes pairs and num_pairs; decode writes codes.  A
 * malformed block (pair count outside [0, P*D], a zero length, lengths not
 * summing to P*D) decodes as zeros and sets SPEC_DEVERR_CODEC.
 * Limits: head_dim a multiple of 32 in [32, 256]; 1 <= page_size and
 * page_size * head_dim <= 16384; num_blocks >= 0.
 */
SPEC_API int spec_codec_encode(const void *codes, int64_t num_blocks, int32_t page_size,
                               int32_t head_dim, void *pairs, int32_t *num_pairs, void *stream);
SPEC_API int spec_codec_decode(const void *pairs, const int32_t *num_pairs, int64_t num_blocks,
                               int32_t page_size, int32_t head_dim, void *codes, void *stream);

/*
 * Greedy acceptance that allocates nothing.  (The pages have no counterpart:
 * this is an interface convenience of this library.)
 *
 * Same operation, arguments and results as spec_accept_greedy, for callers
 * that cannot allocate device memory: a serving process whose GPU memory is
 * reserved up front by its own caching allocator (a cudaMalloc outside that
 * pool can fail once the pool holds the device, and growing this library's
 * workspace synchronises the device in the middle of a step), or a host that
 * loads the library as a plugin without the right to allocate.  Its scratch
 * (reduction partials and completion tickets) is a fixed array of this
 * library's device code, present on every GPU that loads the library until
 * exit:
 *   - limits: batch <= SPEC_NOALLOC_MAX_BATCH and
 *     batch * (num_draft + 1) * ceil(vocab / 8192) <= SPEC_NOALLOC_MAX_PARTIALS
 *     (512 KiB of partials); larger calls return SPEC_ERR_UNSUPPORTED and
 *     enqueue nothing;
 *   - the first call on a device looks up the array's device address (and may
 *     load the library's device code): make it before any stream capture;
 *   - that address is kept for the life of the process: calls after
 *     cudaDeviceReset (or after the device's primary context was destroyed
 *     and re-created) are not supported;
 *   - every call shares the array and it keeps the last call's contents; the
 *     call clears the tickets itself (an async memset on `stream`), but calls
 *     that overlap on the GPU race: order them on one stream.
 * Calls no cudaMalloc, cudaFree or other allocating routine.
 */
enum { SPEC_NOALLOC_MAX_PARTIALS = 65536, SPEC_NOALLOC_MAX_BATCH = 4096 };
SPEC_API int spec_accept_greedy_noalloc(const void *logits, int32_t logits_dtype,
                                        const int32_t *draft_tokens, int32_t batch,
                                        int32_t num_draft, int64_t vocab, int32_t *accepted_len,
                                        int32_t *next_token, void *stream);

/*
 * Rejection-sampling acceptance ("Decoding Speculative Decoding from First
 * Principles", section "How does this drafter maintain the same
 * distribution of the target?").
 *
 * With p_i = softmax(target_logits[b, i, :] / temperature) and
 * q_i = softmax(draft_logits[b, i, :] / temperature), draft x_i =
 * draft_tokens[b, i] is kept while u_i < p_i(x_i) / q_i(x_i); at the first
 * rejection n a token is drawn from max(p_n - q_n, 0) (renormalised); after
 * k acceptances the bonus token is drawn from p_k.  The emitted tokens then
 * follow the target distribution exactly.
 *   accepted_len[b] = n (number of drafts kept), next_token[b] = the draw,
 *   so each sequence gains n + 1 tokens and commits by ctx_b += n + 1.
 *
 * Draws come from the counter-based generator SplitMix64 keyed by `seed`:
 * draw number ((2b + kind) << 32) | j is the SplitMix64 mix of
 * seed + (draw + 1) * 0x9E3779B97F4A7C15; kind 0 gives u_j = top 24 bits /
 * 2^24, kind 1 the Gumbel noise g_j = -ln(-ln u') (u' = (2 * top 23 bits +
 * 1) / 2^24) of token j, and a draw from weights w is argmax_x ln w(x) +
 * g_x (lowest index on ties).  The same seed gives the same tokens; use a
 * fresh seed per step.  Arithmetic is fp32, so a test u_i within ~1e-6 of
 * p/q, or two Gumbel keys within ~1e-6, may decide differently from an
 * exact evaluation.
 *
 *   target_logits  [batch, num_draft + 1, vocab]  logits_dtype (F32|BF16), finite
 *   draft_logits   [batch, num_draft, vocab]      same dtype, finite
 *   draft_tokens   [batch, num_draft] int32 in [0, vocab) (others are
 *                  rejected and flagged with SPEC_DEVERR_TOKEN)
 *   temperature    > 0 and finite
 *   accepted_len, next_token  [batch] int32, written
 *
 * Limits: 1 <= num_draft <= 64; 1 <= vocab < 2^31; both logits arrays
 * 16-byte aligned.  Uses the library workspace (grown on demand, like the
 * other calls).
 */
SPEC_API int spec_accept_rejection(const void *target_logits, const void *draft_logits,
                                   int32_t logits_dtype, const int32_t *draft_tokens,
                                   int32_t batch, int32_t num_draft, int64_t vocab,
                                   float temperature, uint64_t seed, int32_t *accepted_len,
                                   int32_t *next_token, void *stream);

/*
 * Write the drafts' K/V rows into the paged cache (the step before
 * verification: the target's projections of the k drafted tokens).
 *
 * Positions ctx_b .. ctx_b + num_new - 1 of sequence b receive rows
 * k_new / v_new [batch, num_new, num_kv_heads, head_dim] (src_dtype F32 |
 * BF16) at page block_table[b, pos / page_size], slot pos % page_size.
 *   - F32 / BF16 cache: the value (bf16 rounded to nearest even);
 *   - I8 cache: CXL-SpecKV's "Algorithm 2 KV-Cache Compression" per
 *     (token, kv-head) row: s = fp16(max_d |x_d| / 127) into k_scale /
 *     v_scale [num_pages, num_kv_heads, page_size], c_d = clamp(rint(x_d / s),
 *     -127, 127) (c = 0 when s = 0), every step in fp32 (IEEE division,
 *     round half to even), fp16 by round-to-nearest-even.
 * Caches, scales and tables as in spec_verify_attn; ctx_lens is not changed
 * (spec_commit moves it).  A position past the block table or a page id
 * outside [0, num_pages) writes nothing and sets SPEC_DEVERR_CTX /
 * SPEC_DEVERR_PAGE.  Limits: head_dim % 32 == 0 and <= 256; num_new >= 1.
 */
SPEC_API int spec_kv_append(const void *k_new, const void *v_new, int32_t src_dtype,
                            void *k_cache, void *v_cache, void *k_scale, void *v_scale,
                            int32_t cache_dtype, const int32_t *block_table,
                            const int32_t *ctx_lens, int32_t batch, int32_t num_new,
                            int32_t num_kv_heads, int32_t head_dim, int32_t page_size,
                            int32_t num_pages, int32_t max_pages_per_seq, void *stream);

/*
 * Commit a verification step on the device: ctx_lens[b] += accepted_len[b]
 * + extra (HeteroReason's KV Cache Management Unit, "Accept" mode: the
 * validated pointer moves over the accepted drafts; pass extra = 1 to count
 * the emitted correction / bonus token as well, once its row is appended).
 * Rejected drafts are left behind and the next spec_kv_append overwrites
 * them ("Rollback").  ctx_lens and accepted_len are device int32 [batch].
 */
SPEC_API int spec_commit(int32_t *ctx_lens, const int32_t *accepted_len, int32_t batch,
                         int32_t extra, void *stream);

/* Read and clear the device error word of the current device (synchronises
 * the device).  0 = no fault seen; otherwise a bitwise OR of SPEC_DEVERR_*. */
SPEC_API int spec_device_error(int32_t *flags);

enum {
    SPEC_DEVERR_PAGE = 1,    /* block_table entry outside [0, num_pages) (clamped) */
    SPEC_DEVERR_CTX = 2,     /* ctx_b + k beyond the block table (clamped) */
    SPEC_DEVERR_TIMEOUT = 4, /* a bounded on-chip wait gave up; results invalid */
    SPEC_DEVERR_TOKEN = 8,   /* a draft token outside [0, vocab) (treated as rejected) */
    SPEC_DEVERR_TREE = 16,   /* a tree parent outside [-1, i) (the node is never taken) */
    SPEC_DEVERR_CODEC = 32   /* a malformed coded block (decoded as zeros) */
};

/* Free the current device's workspace (synchronises the device). */
SPEC_API int spec_release(void);

#ifdef __cplusplus
}
#endif

#endif /* SPEC_VERIFY_H */

// Internal launch interface between the C-ABI shim (spec_abi.cu) and the
// kernel translation units.  Host-visible only; no torch types anywhere.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "spec_verify.h"

namespace specv {

// Geometry and pointers of one verification-attention call.
struct AttnArgs {
    const void* q;
    const void* k_cache;
    const void* v_cache;
    const uint16_t* k_scale;  // fp16 bits, INT8 caches only
    const uint16_t* v_scale;
    const int32_t* block_table;
    const int32_t* ctx_lens;
    int32_t B, k, Hq, Hkv, D, P, num_pages, max_pages;
    int32_t q_dtype, kv_dtype;
    float scale;
    void* out;
    float* lse;
    int* dev_err;       // device error word
    int* seg_counters;  // [B*Hkv] zeroed arrival counters (fused split-KV merge)
    // [B, k] draft-visibility bits (bit t of row i: query i sees draft t), or
    // null for the causal chain (bits 0..i)
    const uint64_t* tree_mask;
    // tensor-core kernels: tiles charged per segment when the tile list is
    // split over the persistent CTAs (TileSplit); < 0 = the kernel's default
    int32_t split_alpha = -1;
};

// Draft bits visible to query i of sequence b: the tree row, or the causal chain.
__host__ __device__ inline uint64_t draft_bits(const AttnArgs& a, int b, int i) {
#ifdef __CUDA_ARCH__
    if (a.tree_mask) return __ldg(a.tree_mask + (int64_t)b * a.k + i);
#else
    if (a.tree_mask) return a.tree_mask[(int64_t)b * a.k + i];
#endif
    return i >= 63 ? ~0ull : ((1ull << (i + 1)) - 1);
}

// ---- SIMT kernel (CUDA cores; any supported dtype / shape) ----
struct SimtPlan {
    int32_t chunk;       // keys per split chunk (multiple of 16)
    int32_t max_chunks;  // chunks per sequence at the longest possible context
    int32_t row_groups;  // query-row groups per (sequence, kv-head)
    int32_t rows_per_group;
};
SimtPlan simt_plan(const AttnArgs& a, int num_sms, int forced_chunk);
size_t simt_workspace_bytes(const AttnArgs& a, const SimtPlan& p);
cudaError_t launch_attn_simt(const AttnArgs& a, const SimtPlan& p, void* workspace,
                             cudaStream_t stream);

// ---- single-pass SIMT kernel for short contexts (one launch, no split) ----
// Longest context it holds (the whole block table of a sequence), or 0 when
// the call does not fit its shared-memory plan.
int small_attn_max_keys(const AttnArgs& a);
// CTAs (one cluster) per (sequence, kv-head, row group) the automatic choice takes.
int small_attn_cluster_size(const AttnArgs& a, int num_sms);
// `cluster` = CTAs per unit, 1..8, or 0 for the automatic choice (which falls
// back to one CTA when the device cannot place the cluster; a forced size
// returns the launch error instead).
cudaError_t launch_attn_small(const AttnArgs& a, int num_sms, int cluster, cudaStream_t stream);

// ---- tensor-core kernel (tcgen05 + TMA, persistent, split-KV stream-K) ----
bool tc_supported(const AttnArgs& a);
size_t tc_workspace_bytes(const AttnArgs& a, int num_ctas);
cudaError_t launch_attn_tc(const AttnArgs& a, int num_ctas, void* workspace, cudaStream_t stream);

// Merge of the split-KV partials written by a tensor-core kernel (its tiles
// over `num_ctas` persistent CTAs, split by TileSplit with `alpha` tiles
// charged per segment; partial slots [2*C][128][D]; per CTA boundary the
// segment record {b, kv-head, tile-in-segment, tiles} and the CTA's first
// tile; per sequence the tile prefix, in the kernel's tile units).
cudaError_t launch_combine_stream_k(const AttnArgs& a, int num_ctas, int alpha,
                                    const float* part_o, const float* part_lse,
                                    const int4* seg_rec, const int* seg_pre, cudaStream_t stream);

// ---- tensor-core kernel with 128-key tiles: bf16, head_dim 128, up to 128
// query rows per kv-head (two softmax sets); workspace as tc_workspace_bytes ----
bool tc2_supported(const AttnArgs& a);
cudaError_t launch_attn_tc2(const AttnArgs& a, int num_ctas, void* workspace, cudaStream_t stream);

// ---- warp-MMA kernel for k*G <= 16 query rows (mma.sync m16n8k16, TMA pages) ----
bool mma_supported(const AttnArgs& a);
cudaError_t launch_attn_mma(const AttnArgs& a, int num_ctas, void* workspace, cudaStream_t stream);

// ---- greedy acceptance ----
struct AcceptArgs {
    const void* logits;
    int32_t dtype;
    const int32_t* draft;
    int32_t B, k;
    int64_t V;
    int32_t* accepted_len;
    int32_t* next_token;
    // tree acceptance (null for the chain rule): parent [B, k] in [-1, i),
    // accepted node path [B, k] (-1 padded; may be null), device error word
    const int32_t* parent = nullptr;
    int32_t* path = nullptr;
    int* dev_err = nullptr;
};
size_t accept_workspace_bytes(const AcceptArgs& a);
// `tickets` must hold B zeroed int32 (self-resetting across calls).
cudaError_t launch_accept(const AcceptArgs& a, void* workspace, int32_t* tickets,
                          cudaStream_t stream);

// ---- rejection-sampling acceptance (two launches; see accept_rejection.cu) ----
size_t rejection_workspace_bytes(int B, int k, int64_t V);
// `tickets` must hold B zeroed int32 (self-resetting across calls).
cudaError_t launch_accept_rejection(const void* target, const void* draft, int32_t dtype,
                                    const int32_t* draft_tokens, int B, int k, int64_t V,
                                    float temperature, uint64_t seed, int32_t* accepted_len,
                                    int32_t* next_token, void* workspace, int32_t* tickets,
                                    int* dev_err, cudaStream_t stream);

// ---- drafts' K/V append (INT8 quantisation) and the commit ----
cudaError_t launch_kv_append(const void* k_new, const void* v_new, int32_t src_dtype,
                             void* k_cache, void* v_cache, uint16_t* k_scale, uint16_t* v_scale,
                             int32_t cache_dtype, const int32_t* block_table,
                             const int32_t* ctx_lens, int B, int n, int Hkv, int D, int P,
                             int num_pages, int max_pages, int* dev_err, cudaStream_t stream);
// ---- delta + run-length page codec (codec.cu) ----
size_t codec_decode_smem(int P, int D);
cudaError_t launch_codec_encode(const void* codes, int64_t nblk, int P, int D, void* pairs,
                                int32_t* npairs, cudaStream_t stream);
cudaError_t launch_codec_decode(const void* pairs, const int32_t* npairs, int64_t nblk, int P,
                                int D, void* codes, int* dev_err, cudaStream_t stream);

cudaError_t launch_commit(int32_t* ctx_lens, const int32_t* accepted_len, int B, int extra,
                          cudaStream_t stream);

// Sets the thread-local error message of the C ABI; returns `code`.
int set_error(int code, const char* msg);

}  // namespace specv

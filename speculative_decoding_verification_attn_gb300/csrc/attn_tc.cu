// Verification attention on the 5th-generation tensor cores (tcgen05 + TMEM),
// bf16 queries over a bf16 or INT8 paged KV cache, head_dim 128.
//
// What it computes: multi-query causal attention of each sequence's k draft
// queries over its paged cache ("Decoding Speculative Decoding from First
// Principles", "Parallelizing method 2: sequence parallel" and "Speculating
// to get sequence parallelism during decode"): query i of sequence b sees
// keys 0 .. ctx_b + i; kv-head g serves q-heads g*G .. g*G+G-1.
//
// Design (GB300 / sm_103a):
//  * All R = k*G query rows of one (sequence, kv-head) sit on the M side of
//    one 128-row MMA, so every K/V byte is read from HBM exactly once and
//    reused R times (the sequence-parallel amortisation the blog describes).
//    When R <= 64 the rows are replicated REP = 128 / roundup32(R) times
//    (4 copies for R <= 32, 2 for R <= 64), one copy per group of TMEM lane
//    quadrants, and copy c only keeps the keys of column slice c of every
//    64-key tile: the softmax work of a tile is spread over all four warps
//    instead of the one warp that owns lanes 0..R-1, and the copies' partial
//    (max, sum, O) are merged once per segment.
//  * Work is the list of 64-key tiles of every (sequence, kv-head) segment,
//    split evenly over a persistent grid of one CTA per SM (stream-K).  A CTA
//    walks a contiguous tile range that may cross segment boundaries; a
//    segment cut by a range boundary leaves (O/l, lse) partials that the
//    combine kernel merges with log-sum-exp weights (split-KV).
//  * Warp roles: 0-3 softmax / rescale / epilogue / P V issue (one (copy,
//    query row) per thread); 4 Q K^T issue and Q loads; TMA producers 5-7
//    (bf16 cache: tile it by warp 5 + it % 3) or 5 (INT8 cache); 8-11 a
//    second set of softmax warps taking every other tile with an O of its
//    own (bf16 cache) or the INT8 widening warps.
//  * S = Q K^T lands in one of two TMEM buffers (freed as soon as the
//    softmax has loaded it), the softmax warps write bf16 P to TMEM, and
//    O += P V takes P from there.  The running
//    max only moves when it grows by more than 2^8, so O is rarely rescaled
//    (exact in real arithmetic: O and l share the reference max), and a tile's
//    P is released without waiting for the previous tile's P V.
//  * Every mbarrier wait is bounded (1 s); a timeout sets the device error
//    word and an abort flag after which every role skips its remaining work
//    (still passing every CTA barrier) and returns.
#include <cuda.h>
#include <math.h>

#include "common.cuh"

namespace specv {
namespace {

constexpr int D = 128;
constexpr int TN = 64;           // keys per tile
constexpr int NK = 3;            // bf16 cache: K slots (freed when Q K^T has read them)
constexpr int NV = 6;            // bf16 cache: V slots (freed when P V has read them)
constexpr int ROWS = 128;        // MMA M: query rows (padded / replicated)
constexpr int Q_HALF = ROWS * 128;        // 16 KB: 64 head-dim columns of Q
constexpr int Q_BYTES = 2 * Q_HALF;       // 32 KB
constexpr int KV_BYTES = TN * D * 2;      // 16 KB per tensor per stage
constexpr int STAGE_BYTES = 2 * KV_BYTES; // K then V
constexpr int LOOKAHEAD_TILES = 6;        // block-table prefetch distance (all producers)
constexpr int BOX_ROWS = 16;              // keys per TMA box: 16 rows x 256 B = 4 KB
constexpr int MAX_BOX = TN / BOX_ROWS;    // boxes per tile
// TMEM columns: S buffers [0,128) (2 x 64 fp32); O [128,256) and, for the
// second softmax set, [256,384); P0 [384,416) P1 [416,448) (bf16 pairs); Q
// [448,512) (bf16 pairs)
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t TM_S = 0, TM_O = 128, TM_P = 384, TM_Q = 448;
constexpr int NSB = 2;  // S buffers (ping-pong: one per softmax warp set)
constexpr int MAX_BATCH = 1024;
constexpr int SCRATCH_BYTES = 16 * 1024;  // copy-merge buffer of the epilogue
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

// INT8 cache: raw boxes (16 keys x 128 int8 = 2 KB per tensor) and their
// fp16 scales land in NSR stages; four converter warps widen each tile into
// one of NCV fp16 operand stages.
constexpr int NSR = 4;
constexpr int NCV = 3;
constexpr int RAW8_KV = TN * D;                       // 8 KB of int8 per tensor per tile
constexpr int RAW8_STAGE = 2 * RAW8_KV + 2 * TN * 2;  // K, V, then k / v scales (fp16)

// A / B operand formats of tcgen05.mma kind::f16 (bf16 cache: bf16; INT8
// cache widened to fp16, so q and P are fp16 there too)
template <bool KV8>
__host__ __device__ constexpr uint32_t idesc_qk() {
    return KV8 ? umma_idesc_f16(ROWS, TN, 0, 0) : umma_idesc_bf16(ROWS, TN, 0, 0);
}
template <bool KV8>
__host__ __device__ constexpr uint32_t idesc_pv() {  // B (V) MN-major
    return KV8 ? umma_idesc_f16(ROWS, D, 0, 1) : umma_idesc_bf16(ROWS, D, 0, 1);
}
using Cursor = CursorT<TN>;

// Tiles charged per segment in the split over the CTAs: a piece boundary
// drains the tensor-core pipeline (the next piece's queries, the merge of the
// softmax states) for about six 64-key tiles of the bf16 cache's work, five
// of the INT8 cache's slower ones.
__host__ __device__ inline int split_alpha(const AttnArgs& a) {
    return a.split_alpha >= 0 ? a.split_alpha : a.kv_dtype == SPEC_DTYPE_I8 ? 5 : 6;
}

// Shared-memory plan (offsets from the 1024-aligned base).  INT8 cache:
// boxes land in NSR raw stages, converted tiles go to NCV operand stages,
// with one fp32 row of per-key k / v scales per operand stage.
//
// bf16 cache: TMA boxes land where the MMAs read them, and K and V have rings
// of their own -- a K slot is held only from
// its load until Q K^T has read it, a V slot until P V has -- so that the
// bytes in flight are not tied up behind the softmax.  K slot s at
// STAGES + s*16 KB, V slot s at VRING + s*16 KB (TMA lands there, the MMAs
// read it).
// INT8 cache: raw stages [K | V | scales] and operand stages [K | V].
template <bool KV8>
struct SmemT {
    static constexpr int NL = KV8 ? NSR : NK;  // stages the (K) producer fills
    static constexpr int NM = KV8 ? NCV : NK;  // stages Q K^T reads
    static constexpr int Q = 0;                // one Q staging buffer
    static constexpr int STAGES = Q + Q_BYTES;
    static constexpr int VRING = STAGES + (KV8 ? 0 : NK * KV_BYTES);  // bf16: V slots
    static constexpr int RAW = KV8 ? STAGES + NM * STAGE_BYTES : STAGES;
    static constexpr int RAW_STAGE = KV8 ? RAW8_STAGE : KV_BYTES;
    static constexpr int SCRATCH = KV8 ? RAW + NL * RAW_STAGE : VRING + NV * KV_BYTES;
    static constexpr int SCALES = SCRATCH + SCRATCH_BYTES;  // [NM][k, v][TN] float
    static constexpr int BARS = SCALES + (KV8 ? NM * 2 * TN * 4 : 0);
    // barriers (uint64 each): landed (TMA), operands ready (INT8 widening),
    // operand stage free (INT8: P V done; bf16: Q K^T done), raw stage free
    // (INT8), V landed / V slot free (bf16)
    static constexpr int B_KVFULL = 0, B_KREADY = NL, B_KVEMPTY = NL + NM,
                         B_RAWFREE = KV8 ? NL + 2 * NM : B_KVEMPTY,
                         B_VFULL = KV8 ? 0 : NL + 2 * NM, B_VEMPTY = B_VFULL + (KV8 ? 0 : NV),
                         B_QFULL = KV8 ? 2 * NL + 2 * NM : NL + 2 * NM + 2 * NV,
                         B_QFREE = B_QFULL + 1,
                         B_SFULL = B_QFULL + 2, B_SFREE = B_SFULL + NSB, B_ODONE = B_SFREE + NSB,
                         B_DRAIN = B_ODONE + 2, B_QCP = B_DRAIN + 3,
                         NUM_BARS = B_QCP + 1;
    // tmem base, abort flag, then (at +16) the CTA's tile range
    static constexpr int MISC = BARS + NUM_BARS * 8;
    // (m, l) of [set x copy][row]: bf16 two sets x up to 4 copies, INT8 one set
    static constexpr int NSTAT = KV8 ? 4 : 8;
    static constexpr int STAT = MISC + 32;
    // TMA producer warps (5, 6, ...): tile it is issued by warp 5 + it % NPROD.
    // bf16: three, since one issuing thread caps the bytes a CTA keeps in
    // flight; INT8: one (its raw boxes are small and the widening warps set
    // the pace, and idle producers' polling takes issue slots from them)
    static constexpr int NPROD = KV8 ? 1 : 3;
    static constexpr int LOOKAHEAD = LOOKAHEAD_TILES / NPROD;  // own tiles ahead
    static constexpr int PIDS = STAT + 2 * NSTAT * ROWS * 4;  // [NPROD][LOOKAHEAD+1][MAX_BOX] int
    static constexpr int CTX = PIDS + NPROD * (LOOKAHEAD + 1) * MAX_BOX * 4;  // [MAX_BATCH] int
    static constexpr int PRE = CTX + MAX_BATCH * 4;           // [MAX_BATCH+1] int
    static constexpr int END = PRE + (MAX_BATCH + 1) * 4;
};
template <bool KV8>
constexpr size_t smem_bytes() { return SmemT<KV8>::END + 1024; }  // + alignment slack
static_assert(smem_bytes<false>() <= 227 * 1024, "shared memory budget (bf16)");
static_assert(smem_bytes<true>() <= 227 * 1024, "shared memory budget (INT8)");
static_assert(SmemT<true>::RAW % 128 == 0 && RAW8_STAGE % 128 == 0, "TMA destination alignment");
// every ring slot is filled by one producer warp only, so that a warp's
// parity waits on a slot are in the slot's phase order
static_assert(NK % SmemT<false>::NPROD == 0 && NV % SmemT<false>::NPROD == 0 &&
                  NSR % SmemT<true>::NPROD == 0,
              "slot ownership");
static_assert(SmemT<false>::NPROD <= 3 && SmemT<true>::NPROD <= 3, "producers are warps 5-7");
// warps: softmax and P V issue 0-3, Q K^T and Q loads 4, TMA producers 5-7
// (INT8: 5; 6-7 idle), then a second set of softmax warps 8-11 (bf16) or the
// INT8 widening warps 8-11
template <bool KV8>
__host__ __device__ constexpr int threads() { return 12 * 32; }


struct TcParams {
    AttnArgs a;
    float* part_o;    // [2*C][ROWS][D]
    float* part_lse;  // [2*C][ROWS]
    int4* seg_rec;    // [C][2]: per CTA boundary, the segment of its first tile
    int* seg_pre;     // [B+1]: tiles of sequences before b (per kv-head)
};

// Row replication: RQ rows per copy (R rounded up to 32), REP copies.
__host__ __device__ constexpr int rows_per_copy(int R) { return ((R + 31) / 32) * 32; }
__host__ __device__ constexpr int num_copies(int R) {
    return (ROWS % rows_per_copy(R) == 0) ? ROWS / rows_per_copy(R) : 1;
}
// Row `row` of the 128-row Q tile holds real query data.
__device__ __forceinline__ bool q_row_used(int row, int R, int RQ, int REP) {
    return row / RQ < REP && row % RQ < R;
}

// What every role of a CTA shares.
struct Cta {
    const AttnArgs* a;
    const TcParams* prm;
    uint8_t* sm;
    uint64_t* bars;
    volatile int* abort_flag;
    const int* s_ctx;
    const int* s_pre;
    uint32_t tmem;
    const int64_t* rng;  // shared memory: the CTA's tile range [rng[0], rng[1])
    int n_tiles, R, G, BH;
};

// Load CW consecutive fp32 TMEM columns of this thread's lane.
template <int CW>
__device__ __forceinline__ void load_cols(uint32_t taddr, uint32_t (&v)[CW]) {
    if constexpr (CW == 16) {
        tmem_ld16(taddr, v);
    } else if constexpr (CW == 32) {
        tmem_ld32(taddr, v);
    } else {
        uint32_t (&lo)[32] = *reinterpret_cast<uint32_t(*)[32]>(&v[0]);
        uint32_t (&hi)[32] = *reinterpret_cast<uint32_t(*)[32]>(&v[32]);
        tmem_ld32(taddr, lo);
        tmem_ld32(taddr + 32, hi);
    }
}

template <int N>
__device__ __forceinline__ void store_cols(uint32_t taddr, const uint32_t* v) {
    if constexpr (N == 8) {
        tmem_st8(taddr, v);
    } else if constexpr (N == 16) {
        tmem_st16(taddr, v);
    } else {
        tmem_st32(taddr, *reinterpret_cast<const uint32_t(*)[32]>(v));
    }
}

// ================= softmax / rescale / epilogue / P V issue =================
// INT8 cache: S holds q . c_j (c_j the stored integers, exact in fp16); the
// key's scale turns it into the score (s_j = scale * s_k,j * S_j, s_k,j
// pre-multiplied by scale*log2(e) in the operand stage), and P V takes
// p_j * s_v,j, so that O = sum_j p_j s_v,j c_j = sum_j p_j v_j while the row
// sum keeps the plain p_j.
//
// PP (bf16 cache, one copy): two sets of softmax warps, 0-3 and 8-11, take
// alternate tiles ("ping-pong"), each with its own running max, row sum and
// O accumulator in TMEM, so that one set's barrier, TMEM and MUFU latencies
// hide behind the other's work.  The two states of a row are merged by
// log-sum-exp weights once per piece; each set writes half of the columns.
template <int REP, bool KV8, bool PP>
__device__ void softmax_role(const Cta& x) {
    using Smem = SmemT<KV8>;
    constexpr int RQ = REP == 4 ? 32 : REP == 2 ? 64 : ROWS;
    constexpr int CW = TN / REP;  // key columns of a tile owned by one thread
    const AttnArgs& a = *x.a;
    const int tid = threadIdx.x, lane = tid & 31;
    const int warp = (tid >> 5) & 3;                // TMEM lane quadrant
    const int set = PP && tid >= 8 * 32 ? 1 : 0;    // PP: this set takes tiles of parity `set`
    const int ltid = tid - set * 8 * 32;            // 0..127 inside the set
    const int R = x.R, G = x.G, k = a.k, BH = x.BH;
    const int c = (warp * 32) / RQ;                 // copy of this thread
    const int r = warp * 32 + lane - c * RQ;        // query row inside the copy
    const bool warp_active = c < REP && warp * 32 - c * RQ < R;
    const bool row_valid = warp_active && r < R;
    const int i_row = row_valid ? r / G : k - 1;
    const int cbase = c * CW;
    const float sl2 = a.scale * kLog2e;
    const uint32_t lane_base = x.tmem + ((uint32_t)(warp * 32) << 16);
    const uint32_t o_mine = TM_O + set * D;         // this set's O columns
    float* s_stat_m = reinterpret_cast<float*>(x.sm + Smem::STAT);
    float* s_stat_l = s_stat_m + Smem::NSTAT * ROWS;
    uint64_t* bars = x.bars;
    const uint64_t vdesc0 = umma_sdesc_sw128(
        smem_u32(x.sm + (KV8 ? Smem::STAGES + KV_BYTES : Smem::VRING)), BOX_ROWS * 128, 1024);

    if (REP > 1) {
        // P buffers start at zero: a lane only ever rewrites its copy's slice
        // (PP: each set its own buffer)
        const uint32_t zero[32] = {};
        if (!PP || set == 0) tmem_st32(lane_base + TM_P, zero);
        if (!PP || set == 1) tmem_st32(lane_base + TM_P + TN / 2, zero);
        tmem_wait_st();
    }
    float m_ref = -INFINITY, l = 0.f;
    bool has = false;  // this set has taken a tile of the current piece
    uint64_t mrow = 0;  // draft bits of this thread's query row, per piece
    Cursor cur;
    if (x.n_tiles > 0) cur.init(ld_shared_s64(x.rng), x.s_pre, x.s_ctx, a.B, a.Hkv, k);
    bool ok = true;
    for (int it = 0; it < x.n_tiles; ++it) {
        const bool first = (it == 0) || (cur.lt == 0);
        const bool last = (it == x.n_tiles - 1) || (cur.lt == cur.nb - 1);
        const int sb = it & 1, sq = it % NSB;  // P buffer / P V barrier, S buffer
        const bool mine = !PP || sb == set;
        const int ctx = x.s_ctx[cur.b], L = ctx + k, key0 = cur.lt * TN;
        const int nvalid = min(TN, L - key0);
        if (first) {
            m_ref = -INFINITY;
            l = 0.f;
            has = false;
            mrow = draft_bits(a, cur.b, i_row);
        }
        if (mine) {
            if (ok)
                ok = warp_wait(&bars[Smem::B_SFULL + sq], (it / NSB) & 1, x.abort_flag, a.dev_err);
            uint32_t sr[CW];
            if (ok && warp_active) {
                tc_fence_after();
                load_cols<CW>(lane_base + TM_S + sq * TN + cbase, sr);
                tmem_wait_ld();
            }
            // S buffer sq may take tile it + NSB once every warp of the set has loaded it
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[Smem::B_SFREE + sq]);
            if (ok && warp_active) {
                // visible columns of this slice as one bit word: the context
                // keys at its front, then the drafts of the row's bits (causal
                // chain: keys <= ctx + i), limited to the keys the tile holds
                uint32_t vlo, vhi;
                {
                    const int kc0 = key0 + cbase, nv = nvalid - cbase, nctx = ctx - kc0;
                    const uint64_t valid = nv >= 64 ? ~0ull : nv <= 0 ? 0ull : (1ull << nv) - 1;
                    const uint64_t cbits =
                        nctx >= 64 ? ~0ull : nctx <= 0 ? 0ull : (1ull << nctx) - 1;
                    const uint64_t dbits = nctx >= 64   ? 0ull
                                           : nctx >= 0  ? mrow << nctx
                                           : nctx > -64 ? mrow >> -nctx
                                                        : 0ull;
                    const uint64_t vis = (cbits | dbits) & valid;
                    vlo = (uint32_t)vis;
                    vhi = (uint32_t)(vis >> 32);
                }
                // INT8: per-key fp32 scales of this operand stage (k row, then v row)
                const float* sc_k = reinterpret_cast<const float*>(
                    x.sm + Smem::SCALES + (it % Smem::NM) * 2 * TN * 4) + cbase;
                const float* sc_v = sc_k + TN;
                // scores in log2 units, two columns per packed multiply
                // (bf16: scale*log2(e); INT8: the key's folded scale)
                float v[CW];
#pragma unroll
                for (int c4 = 0; c4 < CW / 4; ++c4) {
                    float4 f4 = make_float4(sl2, sl2, sl2, sl2);
                    if constexpr (KV8) f4 = reinterpret_cast<const float4*>(sc_k)[c4];
                    const int c = 4 * c4;
                    f2_split(f2_mul(f2(__uint_as_float(sr[c]), __uint_as_float(sr[c + 1])),
                                    f2(f4.x, f4.y)),
                             v[c], v[c + 1]);
                    f2_split(f2_mul(f2(__uint_as_float(sr[c + 2]), __uint_as_float(sr[c + 3])),
                                    f2(f4.z, f4.w)),
                             v[c + 2], v[c + 3]);
                }
                // masked scores become -inf (exp2 -> 0); a slice inside the
                // context -- nearly every tile -- skips the pass
                const bool full = CW == 64   ? (vlo & vhi) == ~0u
                                  : CW == 32 ? vlo == ~0u
                                             : (vlo | ~((1u << (CW & 31)) - 1u)) == ~0u;
                if (!full) {
#pragma unroll
                    for (int cc = 0; cc < CW; ++cc) {
                        const bool vis = ((cc < 32 ? vlo >> cc : vhi >> (cc - 32)) & 1u) != 0;
                        v[cc] = vis ? v[cc] : -INFINITY;
                    }
                }
                // four running maxima of three-input max for ILP
                float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                for (int c2 = 0; c2 < CW / 2; ++c2)
                    mx[c2 & 3] = fmax3(mx[c2 & 3], v[2 * c2], v[2 * c2 + 1]);
                const float mt = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
                const float m_new = fmaxf(m_ref, mt);
                float alpha = 1.f;
                const bool move = m_new > m_ref + kRescaleThreshold;  // also -inf -> finite
                if (move) {
                    alpha = (m_ref == -INFINITY) ? 0.f : fast_exp2(m_ref - m_new);
                    m_ref = m_new;
                    l *= alpha;
                }
                const float m_use = m_ref == -INFINITY ? 0.f : m_ref;  // keeps -inf - m finite
                const uint64_t neg_m = f2(-m_use, -m_use);
                uint32_t pk[CW / 2];
                uint64_t ps[2] = {f2(0.f, 0.f), f2(0.f, 0.f)};
#pragma unroll
                for (int c4 = 0; c4 < CW / 4; ++c4) {
                    float4 g4 = make_float4(1.f, 1.f, 1.f, 1.f);
                    if constexpr (KV8) g4 = reinterpret_cast<const float4*>(sc_v)[c4];
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int c = 4 * c4 + 2 * h;
                        float e0, e1;
                        f2_split(f2_add(f2(v[c], v[c + 1]), neg_m), e0, e1);
                        e0 = fast_exp2(e0);
                        e1 = fast_exp2(e1);
                        const uint64_t pe = f2(e0, e1);
                        ps[h] = f2_add(ps[h], pe);
                        if constexpr (KV8) {
                            // P V takes p_j * s_v,j
                            f2_split(f2_mul(pe, h ? f2(g4.z, g4.w) : f2(g4.x, g4.y)), e0, e1);
                            pk[2 * c4 + h] = pack_f16x2(e0, e1);
                        } else {
                            pk[2 * c4 + h] = pack_bf16x2(e0, e1);
                        }
                    }
                }
                {
                    float a0, a1, b0, b1;
                    f2_split(ps[0], a0, a1);
                    f2_split(ps[1], b0, b1);
                    l += (a0 + b0) + (a1 + b1);
                }
                // P buffer sb is free once P V(it-2) has finished (PP: this
                // set's previous P V).  P V of tile j completes a phase of
                // o_done[j & 1]; the next phase of that barrier needs this
                // tile's P, so the parity wait is unambiguous
                if (it >= 2) {
                    ok = warp_wait(&bars[Smem::B_ODONE + sb], ((it - 2) >> 1) & 1, x.abort_flag,
                                   a.dev_err);
                    tc_fence_after();
                }
                // this copy's slice of P; the other slices of this lane stay zero
                store_cols<CW / 2>(lane_base + TM_P + sb * (TN / 2) + cbase / 2, pk);
                tmem_wait_st();
                if (has && __any_sync(0xffffffffu, move)) {
                    // O must hold every earlier P V before it is rescaled (PP:
                    // the set's previous P V, tile it-2, was observed above)
                    if (!PP)
                        ok = warp_wait(&bars[Smem::B_ODONE + ((it - 1) & 1)],
                                       ((it - 1) >> 1) & 1, x.abort_flag, a.dev_err);
                    if (ok) {
                        tc_fence_after();
#pragma unroll
                        for (int c4 = 0; c4 < D / 32; ++c4) {
                            uint32_t ov[32];
                            tmem_ld32(lane_base + o_mine + c4 * 32, ov);
                            tmem_wait_ld();
#pragma unroll
                            for (int e = 0; e < 32; ++e)
                                ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
                            tmem_st32(lane_base + o_mine + c4 * 32, ov);
                        }
                        tmem_wait_st();
                    }
                }
            }
            if (!KV8 && ok && nvalid % BH != 0 && ltid < 32) {
                // keys past the sequence end inside its last page: zero their V
                // rows so that 0 * (stale or canary) never reaches O
                ok = warp_wait(&bars[Smem::B_VFULL + it % NV], (it / NV) & 1, x.abort_flag,
                               a.dev_err);
                if (ok) {
                    uint8_t* vst = x.sm + Smem::VRING + (it % NV) * KV_BYTES;
                    const int bx = nvalid / BH, r_end = BH;
                    for (int e = (nvalid % BH) * 16 + lane; e < r_end * 16; e += 32) {
                        const int rr = e / 16, h = (e / 8) & 1, ch = e % 8;
                        *reinterpret_cast<uint4*>(vst + bx * BH * 256 + h * BH * 128 + rr * 128 +
                                                  ch * 16) = make_uint4(0, 0, 0, 0);
                    }
                    fence_proxy_async_smem();
                }
            }
            // O += P V of tile it, issued from here: once every warp of the set
            // has stored its slice of P (and its warp 0 zeroed the V tail),
            // the set's thread 0 issues the MMAs -- not a warp of its own,
            // which the softmax warps would starve of issue slots
            tc_fence_before();
            named_bar_sync(6 + set, 128);
            if (ltid < 32) {
                // the set's warp 0 issues, converged, one elected lane
                __syncwarp();
                tc_fence_after();
                // INT8: the operand stage of tile it, widened; bf16: V slot it % NV
                const int s = KV8 ? it % Smem::NM : it % NV;
                const int nuse = KV8 ? it / Smem::NM : it / NV;
                if (ok)
                    ok = warp_wait(&bars[KV8 ? Smem::B_KREADY + s : Smem::B_VFULL + s], nuse & 1,
                                   x.abort_flag, a.dev_err);
                if (ok) {
                    // V box bx: MN-major, halves 2 KB apart (LBO), 8-key groups 1 KB (SBO)
                    const int nbox = (nvalid + BOX_ROWS - 1) / BOX_ROWS;
                    const uint64_t vd =
                        vdesc0 + ((uint32_t)(s * (KV8 ? STAGE_BYTES : KV_BYTES)) >> 4);
                    const uint32_t pcol = x.tmem + TM_P + sb * (TN / 2);
                    umma_ts_w(x.tmem + o_mine, pcol, vd, idesc_pv<KV8>(), has ? 1u : 0u);
#pragma unroll
                    for (int bx = 1; bx < MAX_BOX; ++bx)
                        if (bx < nbox)
                            umma_ts_w(x.tmem + o_mine, pcol + bx * (BOX_ROWS / 2),
                                      vd + ((bx * BOX_ROWS * 256) >> 4), idesc_pv<KV8>(), 1u);
                    // INT8: the operand stage is free; bf16: the V slot is
                    umma_commit_w(&bars[KV8 ? Smem::B_KVEMPTY + s : Smem::B_VEMPTY + s]);
                    umma_commit_w(&bars[Smem::B_ODONE + sb]);
                }
            }
            has = true;
        }

        if (last) {
            // ---- epilogue of the piece that ends at this tile
            if (ok && warp_active && has) {
                if (PP) {
                    // this set's latest P V (tile it or it-1); its previous one
                    // was observed before that tile's P was stored
                    const int itm = mine ? it : it - 1;
                    ok = warp_wait(&bars[Smem::B_ODONE + (itm & 1)], (itm >> 1) & 1,
                                   x.abort_flag, a.dev_err);
                } else {
                    // observe P V(it-1) before P V(it) so the parity wait is unambiguous
                    if (!first)
                        ok = warp_wait(&bars[Smem::B_ODONE + ((it - 1) & 1)],
                                       ((it - 1) >> 1) & 1, x.abort_flag, a.dev_err);
                    if (ok)
                        ok = warp_wait(&bars[Smem::B_ODONE + (it & 1)], (it >> 1) & 1,
                                       x.abort_flag, a.dev_err);
                }
                tc_fence_after();
            }
            const int64_t t_begin = ld_shared_s64(x.rng), t_end = ld_shared_s64(x.rng + 1);
            const bool complete = cur.seg_start >= t_begin && cur.seg_start + cur.nb <= t_end;
            const int slot = 2 * blockIdx.x + (cur.seg_start < t_begin ? 0 : 1);
            auto out_row = [&](int rr) {
                return ((int64_t)cur.b * k + rr / G) * a.Hq + cur.kvh * G + rr % G;
            };
            if constexpr (REP == 1) {
                // weights of the two sets' O (PP) or of the single O
                float w_mine = 1.f, w_other = 0.f, lt = l, mt = m_ref;
                if constexpr (PP) {
                    if (warp_active) {  // both sets' warps of a quadrant, every piece
                        s_stat_m[set * ROWS + warp * 32 + lane] = has ? m_ref : -INFINITY;
                        s_stat_l[set * ROWS + warp * 32 + lane] = has ? l : 0.f;
                        tc_fence_before();
                        named_bar_sync(2 + warp, 64);
                        tc_fence_after();
                        const float mo = s_stat_m[(1 - set) * ROWS + warp * 32 + lane];
                        const float lo = s_stat_l[(1 - set) * ROWS + warp * 32 + lane];
                        const float mm = has ? m_ref : -INFINITY;
                        mt = fmaxf(mm, mo);
                        w_mine = mm == -INFINITY ? 0.f : fast_exp2(mm - mt);
                        w_other = mo == -INFINITY ? 0.f : fast_exp2(mo - mt);
                        lt = w_mine * (has ? l : 0.f) + w_other * lo;
                    }
                }
                if (ok && warp_active) {
                    const float inv_l = lt > 0.f ? 1.f / lt : 0.f;
                    const float lse = lt > 0.f ? (mt + log2f(lt)) * kLn2 : -INFINITY;
                    const float wm = w_mine * inv_l, wo = w_other * inv_l;
                    const uint32_t o_other = TM_O + (1 - set) * D;
                    // PP: set s writes output columns [64 s, 64 s + 64) from both O
#pragma unroll
                    for (int c4 = (PP ? set * 2 : 0); c4 < (PP ? set * 2 + 2 : D / 32); ++c4) {
                        uint32_t ov[32], ow[32];
                        tmem_ld32(lane_base + o_mine + c4 * 32, ov);
                        if (PP) tmem_ld32(lane_base + o_other + c4 * 32, ow);
                        tmem_wait_ld();
                        float o[32];
#pragma unroll
                        for (int e = 0; e < 32; ++e) {
                            // a set without a tile of this piece holds stale O: weight 0, never read
                            const float a0 = wm > 0.f ? __uint_as_float(ov[e]) * wm : 0.f;
                            const float a1 = PP && wo > 0.f ? __uint_as_float(ow[e]) * wo : 0.f;
                            o[e] = a0 + a1;
                        }
                        if (!row_valid) continue;
                        if (complete) {
                            uint4* dst = reinterpret_cast<uint4*>(
                                static_cast<__nv_bfloat16*>(a.out) + out_row(r) * D + c4 * 32);
#pragma unroll
                            for (int v = 0; v < 4; ++v) {
                                uint4 w;
                                w.x = pack_bf16x2(o[8 * v + 0], o[8 * v + 1]);
                                w.y = pack_bf16x2(o[8 * v + 2], o[8 * v + 3]);
                                w.z = pack_bf16x2(o[8 * v + 4], o[8 * v + 5]);
                                w.w = pack_bf16x2(o[8 * v + 6], o[8 * v + 7]);
                                dst[v] = w;
                            }
                        } else {
                            float4* dst = reinterpret_cast<float4*>(
                                x.prm->part_o + ((int64_t)slot * ROWS + r) * D + c4 * 32);
#pragma unroll
                            for (int v = 0; v < 8; ++v)
                                dst[v] = make_float4(o[4 * v + 0], o[4 * v + 1], o[4 * v + 2],
                                                     o[4 * v + 3]);
                        }
                    }
                    if (row_valid && set == 0) {
                        if (complete) {
                            if (a.lse) a.lse[out_row(r)] = lse;
                        } else {
                            x.prm->part_lse[(int64_t)slot * ROWS + r] = lse;
                        }
                    }
                }
                if constexpr (PP) {
                    // the other set reads this set's O: neither starts the next
                    // piece's P V (which overwrites O) before both are done
                    if (warp_active) {
                        tc_fence_before();
                        named_bar_sync(2 + warp, 64);
                        tc_fence_after();
                    }
                }
            } else {
                // merge the states of every row -- REP copies, times two sets
                // with PP -- with weights from (m, l): the weighted O rows
                // are summed in fp32 in the scratch buffer (rows swizzled by
                // 16-byte chunk), one or two column passes
                constexpr int NSET = PP ? 2 : 1;
                constexpr int NTH = 128 * NSET;  // threads of the merge
                const int st_mine = set * REP + c;
                if (row_valid) {
                    // a set without a tile of this piece: m = -inf, l = 0
                    s_stat_m[st_mine * ROWS + r] = m_ref;
                    s_stat_l[st_mine * ROWS + r] = l;
                }
                named_bar_sync(1, NTH);
                float w = 0.f, lse = -INFINITY;
                if (row_valid) {
                    float mt = -INFINITY;
#pragma unroll
                    for (int sc = 0; sc < NSET * REP; ++sc) mt = fmaxf(mt, s_stat_m[sc * ROWS + r]);
                    float Lsum = 0.f;
#pragma unroll
                    for (int sc = 0; sc < NSET * REP; ++sc) {
                        const float mc = s_stat_m[sc * ROWS + r];
                        if (mc != -INFINITY) Lsum += s_stat_l[sc * ROWS + r] * fast_exp2(mc - mt);
                    }
                    w = (Lsum > 0.f && m_ref != -INFINITY) ? fast_exp2(m_ref - mt) / Lsum : 0.f;
                    lse = Lsum > 0.f ? (mt + log2f(Lsum)) * kLn2 : -INFINITY;
                }
                // columns per pass so that R x CPP floats fit the 16 KB scratch
                constexpr int CPP = REP == 4 ? D : D / 2;
                constexpr int NCH = CPP / 4;  // 16-byte chunks of a scratch row
                float* scratch = reinterpret_cast<float*>(x.sm + Smem::SCRATCH);
#pragma unroll
                for (int pass = 0; pass < D / CPP; ++pass) {
#pragma unroll 1
                    for (int sc = 0; sc < NSET * REP; ++sc) {
                        if (ok && warp_active && st_mine == sc) {
#pragma unroll
                            for (int c4 = 0; c4 < CPP / 32; ++c4) {
                                uint32_t ov[32];
                                tmem_ld32(lane_base + o_mine + pass * CPP + c4 * 32, ov);
                                tmem_wait_ld();
                                if (!row_valid) continue;
#pragma unroll
                                for (int v = 0; v < 8; ++v) {
                                    const int chunk = c4 * 8 + v;
                                    float4* dst = reinterpret_cast<float4*>(
                                        scratch + r * CPP + ((chunk ^ (r & (NCH - 1))) * 4));
                                    // weight 0: a state without keys (its O is
                                    // stale or never written) adds nothing
                                    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
                                    if (w > 0.f)
                                        o = make_float4(__uint_as_float(ov[4 * v + 0]) * w,
                                                        __uint_as_float(ov[4 * v + 1]) * w,
                                                        __uint_as_float(ov[4 * v + 2]) * w,
                                                        __uint_as_float(ov[4 * v + 3]) * w);
                                    if (sc > 0) {
                                        const float4 prev = *dst;
                                        o.x += prev.x;
                                        o.y += prev.y;
                                        o.z += prev.z;
                                        o.w += prev.w;
                                    }
                                    *dst = o;
                                }
                            }
                        }
                        named_bar_sync(1, NTH);
                    }
                    if (ok) {
                        for (int idx = ltid + set * 128; idx < R * NCH; idx += NTH) {
                            const int rr = idx / NCH, chunk = idx % NCH;
                            const float4 o = *reinterpret_cast<const float4*>(
                                scratch + rr * CPP + ((chunk ^ (rr & (NCH - 1))) * 4));
                            const int col = pass * CPP + chunk * 4;
                            if (complete) {
                                uint2 w2;
                                w2.x = pack_bf16x2(o.x, o.y);
                                w2.y = pack_bf16x2(o.z, o.w);
                                *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(a.out) +
                                                          out_row(rr) * D + col) = w2;
                            } else {
                                *reinterpret_cast<float4*>(
                                    x.prm->part_o + ((int64_t)slot * ROWS + rr) * D + col) = o;
                            }
                        }
                    }
                    named_bar_sync(1, NTH);  // scratch reused by the next pass / piece
                }
                if (ok && row_valid && st_mine == 0) {
                    if (complete) {
                        if (a.lse) a.lse[out_row(r)] = lse;
                    } else {
                        x.prm->part_lse[(int64_t)slot * ROWS + r] = lse;
                    }
                }
            }
        }
        if (it + 1 < x.n_tiles) cur.next(x.s_ctx, a.Hkv, k);
    }
    // every P V issued from here must finish before TMEM is released
    if (ltid < 32 && x.n_tiles > 0) {
        __syncwarp();
        umma_commit_w(&bars[Smem::B_DRAIN + 1 + set]);
        if (lane == 0) mbar_drain(&bars[Smem::B_DRAIN + 1 + set], 0);
    }
    __syncwarp();
}

template <bool KV8>
__global__ void __launch_bounds__(threads<KV8>(), 1)
attn_tc_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
               const __grid_constant__ CUtensorMap vmap, const TcParams prm) {
    using Smem = SmemT<KV8>;
    constexpr int NL = Smem::NL, NM = Smem::NM;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const AttnArgs& a = prm.a;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + Smem::BARS);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + Smem::MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + Smem::MISC + 4);
    int* pid_ring = reinterpret_cast<int*>(sm + Smem::PIDS);
    int* s_ctx = reinterpret_cast<int*>(sm + Smem::CTX);
    int* s_pre = reinterpret_cast<int*>(sm + Smem::PRE);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int B = a.B, k = a.k, Hkv = a.Hkv, G = a.Hq / a.Hkv, R = k * G, P = a.P;
    const int RQ = rows_per_copy(R), REP = num_copies(R);
    const int BH = BOX_ROWS;  // keys per TMA box (a 16-row slice of one page)

    // ---- setup: barriers, TMEM, zero Q pad rows, per-sequence tile prefix
    if (tid == 0) {
        for (int s = 0; s < NL; ++s) {
            mbar_init(&bars[Smem::B_KVFULL + s], 1);
            if (KV8) mbar_init(&bars[Smem::B_RAWFREE + s], 4);  // one per converter warp
        }
        for (int s = 0; s < NM; ++s) {
            mbar_init(&bars[Smem::B_KREADY + s], KV8 ? 4 : 1);
            mbar_init(&bars[Smem::B_KVEMPTY + s], 1);
        }
        if (!KV8)
            for (int s = 0; s < NV; ++s) {
                mbar_init(&bars[Smem::B_VFULL + s], 1);
                mbar_init(&bars[Smem::B_VEMPTY + s], 1);
            }
        mbar_init(&bars[Smem::B_QFULL], 1);
        mbar_init(&bars[Smem::B_QFREE], 1);
        mbar_init(&bars[Smem::B_QCP], 1);
        for (int q = 0; q < NSB; ++q) {
            mbar_init(&bars[Smem::B_SFULL + q], 1);
            mbar_init(&bars[Smem::B_SFREE + q], 4);  // the 4 warps of the set that took the tile
        }
        for (int q = 0; q < 2; ++q) mbar_init(&bars[Smem::B_ODONE + q], 1);  // even / odd tiles
        for (int q = 0; q < 3; ++q) mbar_init(&bars[Smem::B_DRAIN + q], 1);  // Q K^T, P V x2
        *abort_flag = 0;
        fence_mbar_init();
    }
    // the grids before this one have finished with every buffer this call touches
    // (and with the tensor memory of this SM)
    grid_dep_launch_dependents();
    grid_dep_wait();
    if (warp == 4) {
        tmem_alloc(tmem_slot, TMEM_COLS);
        tmem_relinquish();
    }
    {
        // rows that hold no query stay zero in both Q buffers
        uint4* q4 = reinterpret_cast<uint4*>(sm + Smem::Q);
        for (int e = tid; e < Q_BYTES / 16; e += threads<KV8>()) {
            const int row = (e % (Q_HALF / 16)) / 8;
            if (!q_row_used(row, R, RQ, REP)) q4[e] = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
    }
    if (warp == 4) {
        const int per = (B + 31) / 32, lo = lane * per, hi = min(B, lo + per);
        int sum = 0;
        for (int b = lo; b < hi; ++b) {
            int c = a.ctx_lens[b];
            const int64_t cap = (int64_t)a.max_pages * P - k;
            if (c < 0 || (int64_t)c > cap) {
                raise_device_error(a.dev_err, SPEC_DEVERR_CTX);
                c = c < 0 ? 0 : (int)(cap < 0 ? 0 : cap);
            }
            s_ctx[b] = c;
            sum += (c + k + TN - 1) / TN;
        }
        int incl = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += v;
        }
        int run = incl - sum;
        for (int b = lo; b < hi; ++b) {
            s_pre[b] = run;
            run += (s_ctx[b] + k + TN - 1) / TN;
        }
        if (lane == 31) s_pre[B] = incl;
        // the CTA's tile range [t_begin, t_end), kept in shared memory so that
        // it occupies no register through the role loops
        __syncwarp();  // the prefix above, written by this warp's lanes
        if (lane < 2) {
            TileSplit split;
            split.init(s_pre, B, Hkv, split_alpha(a), gridDim.x);
            reinterpret_cast<int64_t*>(sm + Smem::MISC + 16)[lane] = split.begin(blockIdx.x + lane);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    const int64_t T = (int64_t)s_pre[B] * Hkv;
    const int64_t* s_rng = reinterpret_cast<const int64_t*>(sm + Smem::MISC + 16);
    const int64_t t_begin = ld_shared_s64(s_rng);
    const int n_tiles = (int)(ld_shared_s64(s_rng + 1) - t_begin);
    if (tid == 0) {
        // the segment holding tile t_begin (b, kv-head, its tile index lt,
        // its length) and t_begin itself, for the combine; lt = -1: no tile
        // there
        int4 r0 = make_int4(0, 0, -1, 0);
        if (t_begin < T) {
            Cursor c0;
            c0.init(t_begin, s_pre, s_ctx, B, Hkv, k);
            r0 = make_int4(c0.b, c0.kvh, c0.lt, c0.nb);
        }
        prm.seg_rec[2 * blockIdx.x] = r0;
        prm.seg_rec[2 * blockIdx.x + 1] =
            make_int4((int)(t_begin & 0xffffffff), (int)(t_begin >> 32), 0, 0);
    }
    if (blockIdx.x == 0)
        for (int b = tid; b <= B; b += threads<KV8>()) prm.seg_pre[b] = s_pre[b];

    if (warp >= 5 && warp < 5 + Smem::NPROD) {
        // ================= TMA producers (warps 5 .. 4 + NPROD) =================
        // Tile it is issued by warp 5 + it % NPROD: one issuing thread caps
        // what a CTA can have in flight, several keep HBM busy.  A warp owns
        // its ring slots (slot counts are multiples of NPROD).  Boxes cover
        // both 64-column halves of their keys of one kv-head, landing as
        // [half][key][128 B] with the 128-byte swizzle the MMAs read; the
        // boxes of a tile are issued by parallel lanes, block-table entries
        // prefetched LOOKAHEAD own tiles ahead with cp.async.
        const int pw = warp - 5;
        int* pids = pid_ring + pw * (Smem::LOOKAHEAD + 1) * MAX_BOX;
        const int n_own = n_tiles > pw ? (n_tiles - 1 - pw) / Smem::NPROD + 1 : 0;
        Cursor cur, ahead;
        if (n_own > 0) {
            cur.init(t_begin + pw, s_pre, s_ctx, B, Hkv, k);
            ahead = cur;
        }
        // from tile `from` to this warp's next one
        auto advance = [&](Cursor& c, int from) {
            for (int j = 1; j <= Smem::NPROD; ++j)
                if (from + j < n_tiles) c.next(s_ctx, Hkv, k);
        };
        const uint64_t pol = l2_policy_evict_first();
        if (lane == 0 && pw == 0) {
            prefetch_tmap(&kmap);
            prefetch_tmap(&vmap);
        }
        auto fetch_pids = [&](int slot, const Cursor& c) {
            const int key0 = c.lt * TN;
            const int nvalid = min(TN, s_ctx[c.b] + k - key0);
            if (lane * BH < nvalid)
                cp_async_4(&pids[slot * MAX_BOX + lane],
                           &a.block_table[(int64_t)c.b * a.max_pages + (key0 + lane * BH) / P]);
        };
        for (int la = 0; la < Smem::LOOKAHEAD; ++la) {
            if (la < n_own) {
                fetch_pids(la % (Smem::LOOKAHEAD + 1), ahead);
                advance(ahead, pw + la * Smem::NPROD);
            }
            cp_async_commit();
        }
        int nk_issued = 0, nv_issued = 0;  // own tiles whose K (raw stage) / V went out
        bool ok = true;
        for (int q = 0; q < n_own && ok; ++q) {
            const int it = pw + q * Smem::NPROD;
            if (q + Smem::LOOKAHEAD < n_own) {
                fetch_pids((q + Smem::LOOKAHEAD) % (Smem::LOOKAHEAD + 1), ahead);
                advance(ahead, pw + (q + Smem::LOOKAHEAD) * Smem::NPROD);
            }
            cp_async_commit();
            cp_async_wait<Smem::LOOKAHEAD>();  // entries of tile `it`
            __syncwarp();
            const int* pid = pids + (q % (Smem::LOOKAHEAD + 1)) * MAX_BOX;
            const int key0 = cur.lt * TN;
            const int nvalid = min(TN, s_ctx[cur.b] + k - key0);
            const int nbox = (nvalid + BH - 1) / BH;
            auto page_of = [&](int bx) {
                int page = pid[bx];
                if (page < 0 || page >= a.num_pages) {
                    raise_device_error(a.dev_err, SPEC_DEVERR_PAGE);
                    page = 0;
                }
                return page;
            };
            {
                // K (bf16) / raw stage (INT8): free once Q K^T read it / the
                // converter warps widened it
                const int s = it % NL, use = it / NL;
                if (use >= 1)
                    ok = warp_wait(&bars[Smem::B_RAWFREE + s], (use - 1) & 1, abort_flag,
                                   a.dev_err);
                if (ok && lane == 0)
                    mbar_arrive_expect_tx(&bars[Smem::B_KVFULL + s],
                                          KV8 ? nbox * (2u * BH * D + 2u * BH * 2)
                                              : (nvalid + 7) / 8 * 2048u);
                __syncwarp();
                if (!ok) break;
                uint8_t* st = sm + Smem::RAW + s * Smem::RAW_STAGE;
                if constexpr (KV8) {
                    if (lane < 4 * nbox) {
                        const int bx = lane >> 2;
                        const int row = (page_of(bx) * Hkv + cur.kvh) * P + (key0 + bx * BH) % P;
                        // lane & 3: K box, V box (16 rows x 128 int8), k / v scales (16 fp16)
                        const int what = lane & 3;
                        if (what < 2)
                            tma_load_2d(st + what * RAW8_KV + bx * BH * D,
                                        what ? (const void*)&vmap : (const void*)&kmap,
                                        &bars[Smem::B_KVFULL + s], 0, row, pol);
                        else
                            bulk_load(st + 2 * RAW8_KV + (what - 2) * TN * 2 + bx * BH * 2,
                                      (what == 2 ? a.k_scale : a.v_scale) + row, BH * 2,
                                      &bars[Smem::B_KVFULL + s]);
                    }
                } else {
                    // 8-key boxes (lane j, 2 KB: both head-dim halves of 8 full
                    // rows) landing as [half 0 | half 1], so 8-key group g of
                    // half h sits at g*2 KB + h*1 KB -- the uniform stride an
                    // N = 64 Q K^T reads, with no relayout
                    if (lane * 8 < nvalid) {
                        const int row = (page_of(lane >> 1) * Hkv + cur.kvh) * P +
                                        (key0 + lane * 8) % P;
                        tma_load_3d_hint(st + lane * 2048, &kmap, &bars[Smem::B_KVFULL + s], 0,
                                         row, 0, pol);
                    }
                }
                nk_issued = q + 1;
            }
            if constexpr (!KV8) {
                // V: 16-key boxes (4 KB) in the layout P V reads, into slot
                // it % NV, free once P V of tile it - NV has read it
                const int s = it % NV, use = it / NV;
                if (use >= 1)
                    ok = warp_wait(&bars[Smem::B_VEMPTY + s], (use - 1) & 1, abort_flag,
                                   a.dev_err);
                if (ok && lane == 0) mbar_arrive_expect_tx(&bars[Smem::B_VFULL + s], nbox * 4096u);
                __syncwarp();
                if (!ok) break;
                if (lane < nbox) {
                    const int row = (page_of(lane) * Hkv + cur.kvh) * P + (key0 + lane * BH) % P;
                    tma_load_3d_hint(sm + Smem::VRING + s * KV_BYTES + lane * 4096, &vmap,
                                     &bars[Smem::B_VFULL + s], 0, row, 0, pol);
                }
                nv_issued = q + 1;
            }
            __syncwarp();
            advance(cur, it);
        }
        cp_async_wait<0>();
        if (!ok && lane == 0) {
            // drain: wait (bounded) for the latest copy into each slot this
            // warp filled (a slot's earlier phases completed before it was refilled)
            for (int q = max(0, nk_issued - 2); q < nk_issued; ++q) {
                const int it = pw + q * Smem::NPROD;
                const int last = pw + (nk_issued - 1) * Smem::NPROD;
                if (q == nk_issued - 1 || it % NL != last % NL)
                    mbar_drain(&bars[Smem::B_KVFULL + it % NL], (it / NL) & 1);
            }
            for (int q = max(0, nv_issued - 2); q < nv_issued; ++q) {
                const int it = pw + q * Smem::NPROD;
                const int last = pw + (nv_issued - 1) * Smem::NPROD;
                if (q == nv_issued - 1 || it % NV != last % NV)
                    mbar_drain(&bars[Smem::B_VFULL + it % NV], (it / NV) & 1);
            }
        }
    } else if (KV8 && warp >= 8) {
        // ================= INT8 widening (warps 8-11) =================
        // Raw stage -> operand stage: K lands in the order the N = 64
        // Q K^T reads (8-key groups 2 KB apart), V in the box order of P V
        // (16-key boxes 4 KB apart), both as fp16 with the 128-byte swizzle;
        // the per-key scales become fp32 rows (k pre-multiplied by
        // scale*log2(e)), zero past the sequence end.  Whole 16-key boxes are
        // widened; keys past the end hold finite values that P = 0 cancels.
        const int ct = tid - 8 * 32;  // 0..127
        const float sl2 = a.scale * kLog2e;
        Cursor cur;
        if (n_tiles > 0) cur.init(t_begin, s_pre, s_ctx, B, Hkv, k);
        bool ok = true;
        for (int it = 0; it < n_tiles && ok; ++it) {
            const int s = it % NL, m = it % NM;
            const int nvalid = min(TN, s_ctx[cur.b] + k - cur.lt * TN);
            const int nbox = (nvalid + BOX_ROWS - 1) / BOX_ROWS;
            ok = warp_wait(&bars[Smem::B_KVFULL + s], (it / NL) & 1, abort_flag, a.dev_err);
            // the operand stage is free once P V of tile it - NM has finished
            if (ok && it >= NM)
                ok = warp_wait(&bars[Smem::B_KVEMPTY + m], ((it / NM) - 1) & 1, abort_flag,
                               a.dev_err);
            if (!ok) break;
            const uint8_t* raw = sm + Smem::RAW + s * Smem::RAW_STAGE;
            uint8_t* kc = sm + Smem::STAGES + m * STAGE_BYTES;
            uint8_t* vc = kc + KV_BYTES;
            // all of a thread's raw chunks are loaded before any is widened,
            // so that the shared-memory loads overlap
            constexpr int PER = TN * 8 / 128;  // 16-byte chunks per thread and tensor
            const int nch = nbox * BOX_ROWS * 8;
            uint4 rks[PER], rvs[PER];
#pragma unroll
            for (int u = 0; u < PER; ++u) {
                const int id = ct + 128 * u;
                if (id < nch) {
                    rks[u] = *reinterpret_cast<const uint4*>(raw + id * 16);
                    rvs[u] = *reinterpret_cast<const uint4*>(raw + RAW8_KV + id * 16);
                }
            }
#pragma unroll
            for (int u = 0; u < PER; ++u) {
                const int id = ct + 128 * u;
                if (id >= nch) continue;
                // 16-byte chunk c16 (head-dim 16*c16 .. +15) of key j
                const int j = id >> 3, c16 = id & 7, h = c16 >> 2, sw = j & 7;
                uint4 k0, k1, v0, v1;
                i8x16_to_f16(rks[u], k0, k1);
                i8x16_to_f16(rvs[u], v0, v1);
                // fp16 chunks cc, cc+1 of half h; lanes of half 1 store their
                // odd chunk first so that 8 consecutive lanes hit 8 bank groups
                const int cc = (c16 & 3) * 2;
                const int o0 = ((cc + h) ^ sw) << 4, o1 = ((cc + 1 - h) ^ sw) << 4;
                uint8_t* kr = kc + (j >> 3) * 2048 + h * 1024 + (j & 7) * 128;
                uint8_t* vr = vc + (j >> 4) * 4096 + h * 2048 + (j & 15) * 128;
                *reinterpret_cast<uint4*>(kr + o0) = h ? k1 : k0;
                *reinterpret_cast<uint4*>(kr + o1) = h ? k0 : k1;
                *reinterpret_cast<uint4*>(vr + o0) = h ? v1 : v0;
                *reinterpret_cast<uint4*>(vr + o1) = h ? v0 : v1;
            }
            {
                const int j = ct & (TN - 1), which = ct >> 6;  // 0: k scales, 1: v scales
                const __half hs =
                    reinterpret_cast<const __half*>(raw + 2 * RAW8_KV + which * TN * 2)[j];
                const float f = j < nvalid ? __half2float(hs) * (which ? 1.f : sl2) : 0.f;
                reinterpret_cast<float*>(sm + Smem::SCALES + m * 2 * TN * 4)[which * TN + j] = f;
            }
            fence_proxy_async_smem();  // generic-proxy writes -> tensor-core reads
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&bars[Smem::B_RAWFREE + s]);
                mbar_arrive(&bars[Smem::B_KREADY + m]);
            }
            if (it + 1 < n_tiles) cur.next(s_ctx, Hkv, k);
        }
    } else if (warp == 4) {
        // ================= Q K^T issue (warp 4) =================
        // K arrives (bf16: as 8-key TMA boxes; INT8: widened by warps 8-11)
        // with 8-key groups 2 KB apart, one uniform stride for an N = 64 MMA.
        // P V is issued by the softmax warps.  This warp also loads Q: a
        // piece's Q goes to the staging buffer as soon as the previous
        // piece's Q has been copied out of it into TMEM.
        if (n_tiles > 0) {
            Cursor cur;
            cur.init(t_begin, s_pre, s_ctx, B, Hkv, k);
            int pc = -1;
            int q_issued = 0;  // pieces whose Q load has gone out
            bool ok = true;
            auto issue_q = [&](const Cursor& c) {  // lane 0
                mbar_arrive_expect_tx(&bars[Smem::B_QFULL], REP * 2 * R * 128);
                for (int cp = 0; cp < REP; ++cp)
                    for (int h = 0; h < 2; ++h)
                        tma_load_3d(sm + Smem::Q + h * Q_HALF + cp * RQ * 128, &qmap,
                                    &bars[Smem::B_QFULL], h * 64, c.kvh * G, c.b * k);
            };
            if (lane == 0) {
                prefetch_tmap(&qmap);
                issue_q(cur);
            }
            q_issued = 1;
            constexpr uint32_t kIdescQK = idesc_qk<KV8>();
            // smem descriptors are built once; an operand's start address
            // lives in the low 14 bits (in 16-byte units), so stepping to
            // another k-slice, box or stage is one 64-bit add
            const uint64_t qdesc0 = umma_sdesc_sw128(smem_u32(sm + Smem::Q), 16, 1024);
            const uint64_t kdesc0 = umma_sdesc_sw128(smem_u32(sm + Smem::STAGES), 16, 2048);
            for (int it = 0; it < n_tiles && ok; ++it) {
                const bool first = (it == 0) || (cur.lt == 0);
                if (first) ++pc;
                const int s = it % NM, sq = it % NSB;
                {
                    if (first && q_issued == pc) {
                        // the previous piece had a single tile: its copy to
                        // TMEM was not yet seen done when its MMAs went out
                        ok = warp_wait(&bars[Smem::B_QFREE], (pc - 1) & 1, abort_flag, a.dev_err);
                        if (ok && lane == 0) issue_q(cur);
                        __syncwarp();
                        q_issued = pc + 1;
                        if (!ok) break;
                    }
                    if (first) {
                        ok = warp_wait(&bars[Smem::B_QFULL], pc & 1, abort_flag, a.dev_err);
                        if (ok && pc >= 1) {
                            // the previous piece's MMAs still read TMEM Q: wait
                            // for them before overwriting it
                            __syncwarp();
                            umma_commit_w(&bars[Smem::B_QCP]);
                            ok = warp_wait(&bars[Smem::B_QCP], (pc - 1) & 1, abort_flag, a.dev_err);
                        }
                    }
                    if (KV8 && first && ok) {
                        // the piece's Q to fp16, in place (the MMAs read fp16
                        // operands when the cache is INT8)
                        uint4* q4 = reinterpret_cast<uint4*>(sm + Smem::Q);
#pragma unroll 4
                        for (int e = lane; e < Q_BYTES / 16; e += 32) q4[e] = bf16x8_to_f16(q4[e]);
                        fence_proxy_async_smem();
                    }
                    // K of tile it landed (bf16) / was widened (INT8)
                    if (ok)
                        ok = warp_wait(&bars[KV8 ? Smem::B_KREADY + s : Smem::B_KVFULL + s],
                                       (it / NM) & 1, abort_flag, a.dev_err);
                    // S buffer sq is free once every softmax warp has loaded tile it - NSB
                    if (ok && it >= NSB)
                        ok = warp_wait(&bars[Smem::B_SFREE + sq], ((it / NSB) - 1) & 1,
                                       abort_flag, a.dev_err);
                    if (!ok) break;
                    __syncwarp();
                    tc_fence_after();
                    // issued by the whole warp, one elected lane (operands are
                    // warp-uniform)
                    if (first) {
                        // the piece's Q: smem (TMA, 128-byte swizzle) -> TMEM;
                        // k-slice kk = half kk/4, 32-byte step kk%4
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk)
                            tmem_cp_128x256b_w(tmem + TM_Q + kk * 8,
                                               qdesc0 + (kk >> 2) * (Q_HALF >> 4) + (kk & 3) * 2);
                        // the staging buffer may take the next piece's Q once
                        // the copies are done
                        umma_commit_w(&bars[Smem::B_QFREE]);
                    }
                    {
                        // S = Q K^T: K half h of 8-key group g at g*2 KB + h*1 KB
                        const uint64_t kd =
                            kdesc0 + ((uint32_t)(s * (KV8 ? STAGE_BYTES : KV_BYTES)) >> 4);
                        const uint32_t dcol = tmem + TM_S + sq * TN;
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk)
                            umma_ts_w(dcol, tmem + TM_Q + kk * 8,
                                      kd + (kk >> 2) * (1024 >> 4) + (kk & 3) * 2, kIdescQK,
                                      kk ? 1u : 0u);
                        umma_commit_w(&bars[Smem::B_SFULL + sq]);
                        // bf16: the K slot is free as soon as Q K^T has read it
                        if (!KV8) umma_commit_w(&bars[Smem::B_KVEMPTY + s]);
                    }
                    // the next piece's Q, once this piece's copy to TMEM is done
                    // (not waited for: a later tile of the piece tries again)
                    const int next_it = it + (cur.nb - cur.lt);
                    if (q_issued == pc + 1 && next_it < n_tiles) {
                        bool go = false;
                        if (lane == 0 && mbar_try_wait(&bars[Smem::B_QFREE], pc & 1)) {
                            Cursor nx = cur;
                            nx.lt = nx.nb - 1;
                            nx.next(s_ctx, Hkv, k);
                            issue_q(nx);
                            go = true;
                        }
                        if (__shfl_sync(0xffffffffu, go, 0)) q_issued = pc + 2;
                    }
                    __syncwarp();
                }
                if (it + 1 < n_tiles) cur.next(s_ctx, Hkv, k);
            }
            // an abort leaves no Q copy in flight (Q loads complete in order,
            // each issued after the previous one was waited for)
            if (!ok && lane == 0) mbar_drain(&bars[Smem::B_QFULL], (q_issued - 1) & 1);
            // every tensor-core op of this warp must finish before TMEM is released
            __syncwarp();
            umma_commit_w(&bars[Smem::B_DRAIN]);
            if (lane == 0) mbar_drain(&bars[Smem::B_DRAIN], 0);
            __syncwarp();
        }
    } else if (warp < 4 || (!KV8 && warp >= 8)) {
        Cta x;
        x.a = &a;
        x.prm = &prm;
        x.sm = sm;
        x.bars = bars;
        x.abort_flag = abort_flag;
        x.s_ctx = s_ctx;
        x.s_pre = s_pre;
        x.tmem = tmem;
        x.rng = s_rng;
        x.n_tiles = n_tiles;
        x.R = R;
        x.G = G;
        x.BH = BH;
        // bf16 cache, one copy: warps 0-3 and 8-11 take alternate tiles;
        // with copies the second set has no work
        const bool second = warp >= 8;
        if (REP == 4) {
            if (KV8) {
                if (!second) softmax_role<4, true, false>(x);
            } else {
                softmax_role<4, false, true>(x);
            }
        } else if (REP == 2) {
            if (KV8) {
                if (!second) softmax_role<2, true, false>(x);
            } else {
                softmax_role<2, false, true>(x);
            }
        } else if (KV8) {
            softmax_role<1, true, false>(x);
        } else {
            softmax_role<1, false, true>(x);
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 4) tmem_dealloc(tmem, TMEM_COLS);
}

// Merge the partials of every segment cut by a CTA-range boundary.
// grid (B*Hkv segments or C-1 boundaries, ceil(R/8)), 8 warps, one query row
// per warp.
template <bool BY_SEG>
__global__ void __launch_bounds__(256)
combine_tc_kernel(AttnArgs a, int num_ctas, int alpha, const float* __restrict__ part_o,
                  const float* __restrict__ part_lse, const int4* __restrict__ seg_rec,
                  const int* __restrict__ seg_pre) {
    // BY_SEG: block x handles segment x (sequence x / Hkv, kv-head x % Hkv);
    // else the boundary between CTAs x and x + 1 -- the segment holding CTA
    // x+1's first tile, when that is not the segment's first tile and this
    // is the first boundary inside it.  The launch takes the form with fewer
    // blocks.
    grid_dep_launch_dependents();
    grid_dep_wait();
    const int G = a.Hq / a.Hkv, R = a.k * G;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t C = num_ctas;
    // the attention kernel's split of the tile list over its CTAs
    TileSplit split;
    split.init(seg_pre, a.B, a.Hkv, alpha, C);
    int b, kvh, nb;
    int64_t s0;
    if constexpr (BY_SEG) {
        b = blockIdx.x / a.Hkv;
        kvh = blockIdx.x % a.Hkv;
        const int p0 = __ldg(seg_pre + b);
        nb = __ldg(seg_pre + b + 1) - p0;
        s0 = (int64_t)p0 * a.Hkv + (int64_t)kvh * nb;
    } else {
        const int x = blockIdx.x + 1;
        const int4 r0 = __ldg(seg_rec + 2 * x), r1 = __ldg(seg_rec + 2 * x + 1);
        if (r0.z <= 0) return;  // the boundary is a segment start (or past the end)
        b = r0.x;
        kvh = r0.y;
        nb = r0.w;
        s0 = ((int64_t)(uint32_t)r1.x | ((int64_t)r1.y << 32)) - r0.z;
    }
    const int c_first = split.cta_of_cost(split.cost_of(b, kvh, 0, nb));
    const int c_last = split.cta_of_cost(split.cost_of(b, kvh, nb - 1, nb));
    if (BY_SEG ? c_first == c_last : c_first + 1 != (int)blockIdx.x + 1)
        return;  // written directly by its CTA / handled at an earlier boundary
    const int row = blockIdx.y * 8 + warp;
    if (row >= R) return;

    // CTA c's first tile, from its record (CTA C: the end of the list); a
    // CTA with an empty range wrote nothing and is skipped
    const int64_t T = (int64_t)__ldg(seg_pre + a.B) * a.Hkv;
    auto begin = [&](int c) -> int64_t {
        if (c >= C) return T;
        const int4 r = __ldg(seg_rec + 2 * c + 1);
        return (int64_t)(uint32_t)r.x | ((int64_t)r.y << 32);
    };
    auto empty = [&](int c) { return begin(c) == begin(c + 1); };
    auto slot_of = [&](int c) { return 2 * c + (s0 < begin(c) ? 0 : 1); };
    constexpr uint32_t kAll = 0xffffffffu;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float lse_tot;
    auto add = [&](float w, float4 v) {
        // a piece of weight 0 (an empty CTA range) wrote nothing: its value is
        // dropped, not multiplied
        if (w > 0.f) {
            acc.x = fmaf(w, v.x, acc.x);
            acc.y = fmaf(w, v.y, acc.y);
            acc.z = fmaf(w, v.z, acc.z);
            acc.w = fmaf(w, v.w, acc.w);
        }
    };
    const int npc = c_last - c_first + 1;
    if (npc <= 32) {
        // one piece per lane: its lse and the first 8 pieces' O rows (lane ->
        // 4 columns) are loaded together, before any of them is needed
        const int c = c_first + lane;
        const bool use = lane < npc && !empty(c);
        const float lw = use ? __ldg(part_lse + (int64_t)slot_of(c) * ROWS + row) : -INFINITY;
        const int64_t off = use ? ((int64_t)slot_of(c) * ROWS + row) * D : 0;
        float4 v[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int64_t oj = __shfl_sync(kAll, off, j);
            v[j] = j < npc ? __ldg(reinterpret_cast<const float4*>(part_o + oj) + lane)
                           : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        float m = lw;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(kAll, m, o));
        float t = lw == -INFINITY ? 0.f : expf(lw - m);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(kAll, t, o);
        lse_tot = m + logf(t);
        const float wl = lw == -INFINITY ? 0.f : expf(lw - lse_tot);
#pragma unroll
        for (int j = 0; j < 8; ++j) add(__shfl_sync(kAll, wl, j), v[j]);
#pragma unroll 8
        for (int j = 8; j < npc; ++j) {
            const float w = __shfl_sync(kAll, wl, j);
            const int64_t oj = __shfl_sync(kAll, off, j);
            add(w, __ldg(reinterpret_cast<const float4*>(part_o + oj) + lane));
        }
    } else {
        // more pieces than lanes: lse max, sum, then the weighted rows
        float m = -INFINITY;
        for (int c0 = c_first; c0 <= c_last; c0 += 32) {
            const int c = c0 + lane;
            const bool use = c <= c_last && !empty(c);
            m = fmaxf(m, use ? __ldg(part_lse + (int64_t)slot_of(c) * ROWS + row) : -INFINITY);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(kAll, m, o));
        float tsum = 0.f;
        for (int c0 = c_first; c0 <= c_last; c0 += 32) {
            const int c = c0 + lane;
            const bool use = c <= c_last && !empty(c);
            const float lw = use ? __ldg(part_lse + (int64_t)slot_of(c) * ROWS + row) : -INFINITY;
            if (lw != -INFINITY) tsum += expf(lw - m);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) tsum += __shfl_xor_sync(kAll, tsum, o);
        lse_tot = m + logf(tsum);
        for (int c0 = c_first; c0 <= c_last; c0 += 32) {
            const int c = c0 + lane;
            const bool use = c <= c_last && !empty(c);
            const float lw = use ? __ldg(part_lse + (int64_t)slot_of(c) * ROWS + row) : -INFINITY;
            const float wl = lw == -INFINITY ? 0.f : expf(lw - lse_tot);
            const int64_t off = use ? ((int64_t)slot_of(c) * ROWS + row) * D : 0;
            const int n = min(32, c_last - c0 + 1);
#pragma unroll 8
            for (int j = 0; j < n; ++j) {
                const float w = __shfl_sync(kAll, wl, j);
                const int64_t oj = __shfl_sync(kAll, off, j);
                add(w, __ldg(reinterpret_cast<const float4*>(part_o + oj) + lane));
            }
        }
    }
    const int i = row / G, h = kvh * G + row % G;
    const int64_t orow = ((int64_t)b * a.k + i) * a.Hq + h;
    uint2 o;
    o.x = pack_bf16x2(acc.x, acc.y);
    o.y = pack_bf16x2(acc.z, acc.w);
    reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(a.out) + orow * D)[lane] = o;
    if (lane == 0 && a.lse) a.lse[orow] = lse_tot;
}

// ---------------------------------------------------------------- host side

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

}  // namespace

bool tc_supported(const AttnArgs& a) {
    const int G = a.Hq / a.Hkv;
    const bool pow2 = (a.P & (a.P - 1)) == 0;
    // INT8 cache: the scales are fetched 16 keys (32 bytes) at a time with
    // bulk copies, which need 16-byte aligned sources
    const bool kv_ok =
        a.kv_dtype == SPEC_DTYPE_BF16 ||
        (a.kv_dtype == SPEC_DTYPE_I8 && a.k_scale && a.v_scale &&
         (reinterpret_cast<uintptr_t>(a.k_scale) & 15) == 0 &&
         (reinterpret_cast<uintptr_t>(a.v_scale) & 15) == 0);
    return a.q_dtype == SPEC_DTYPE_BF16 && kv_ok && a.D == D &&
           a.k * G <= ROWS && G <= 256 && pow2 && a.P >= 16 && a.P <= 256 && a.B <= MAX_BATCH &&
           (int64_t)a.num_pages * a.Hkv * a.P < (1LL << 31) && (int64_t)a.B * a.k < (1LL << 31);
}

size_t tc_workspace_bytes(const AttnArgs&, int num_ctas) {
    return (size_t)2 * num_ctas * ROWS * (D + 1) * sizeof(float) + (size_t)num_ctas * 32 +
           (size_t)(MAX_BATCH + 1) * 4 + 256;
}

cudaError_t launch_attn_tc(const AttnArgs& a, int num_ctas, void* workspace, cudaStream_t stream) {
    if (a.B == 0) return cudaSuccess;
    EncodeTiledFn encode = get_encode_fn();
    if (!encode) return cudaErrorNotSupported;
    const int G = a.Hq / a.Hkv;
    CUtensorMap qmap, kmap, vmap;
    {
        cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)a.Hq, (cuuint64_t)a.B * a.k};
        cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)a.Hq * D * 2};
        cuuint32_t box[3] = {64, (cuuint32_t)G, (cuuint32_t)a.k};
        cuuint32_t es[3] = {1, 1, 1};
        if (encode(&qmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(a.q), dims,
                   strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    // K/V: [rows = num_pages*Hkv*P] x [2 halves] x [64 columns]; one box =
    // BH consecutive rows of one page, both halves.  INT8: [rows] x [128
    // bytes], one unswizzled box of BH rows (the converter warps swizzle)
    const int BH = BOX_ROWS;
    const cuuint64_t rows = (cuuint64_t)a.num_pages * a.Hkv * a.P;
    const bool kv8 = a.kv_dtype == SPEC_DTYPE_I8;
    for (int t = 0; t < 2 && kv8; ++t) {
        cuuint64_t dims[2] = {(cuuint64_t)D, rows};
        cuuint64_t strides[1] = {(cuuint64_t)D};
        cuuint32_t box[2] = {(cuuint32_t)D, (cuuint32_t)BH};
        cuuint32_t es[2] = {1, 1};
        if (encode(t == 0 ? &kmap : &vmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2,
                   const_cast<void*>(t == 0 ? a.k_cache : a.v_cache), dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    for (int t = 0; t < 2 && !kv8; ++t) {
        cuuint64_t dims[3] = {64, rows, 2};
        cuuint64_t strides[2] = {(cuuint64_t)D * 2, 128};
        cuuint32_t box[3] = {64, (cuuint32_t)(t == 0 ? BH / 2 : BH), 2};  // K: 8-key boxes
        cuuint32_t es[3] = {1, 1, 1};
        if (encode(t == 0 ? &kmap : &vmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                   const_cast<void*>(t == 0 ? a.k_cache : a.v_cache), dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    TcParams prm;
    prm.a = a;
    prm.part_o = static_cast<float*>(workspace);
    prm.part_lse = prm.part_o + (size_t)2 * num_ctas * ROWS * D;
    prm.seg_rec = reinterpret_cast<int4*>(prm.part_lse + (size_t)2 * num_ctas * ROWS);
    prm.seg_pre = reinterpret_cast<int*>(prm.seg_rec + 2 * (size_t)num_ctas);
    cudaError_t e;
    if (kv8) {
        e = cudaFuncSetAttribute(attn_tc_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem_bytes<true>());
        if (e != cudaSuccess) return e;
        e = launch_dependent(attn_tc_kernel<true>, dim3(num_ctas), dim3(threads<true>()),
                             smem_bytes<true>(), stream, qmap, kmap, vmap, prm);
    } else {
        e = cudaFuncSetAttribute(attn_tc_kernel<false>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem_bytes<false>());
        if (e != cudaSuccess) return e;
        e = launch_dependent(attn_tc_kernel<false>, dim3(num_ctas), dim3(threads<false>()),
                             smem_bytes<false>(), stream, qmap, kmap, vmap, prm);
    }
    if (e != cudaSuccess) return e;
    return launch_combine_stream_k(a, num_ctas, split_alpha(a), prm.part_o, prm.part_lse,
                                   prm.seg_rec, prm.seg_pre, stream);
}

cudaError_t launch_combine_stream_k(const AttnArgs& a, int num_ctas, int alpha,
                                    const float* part_o, const float* part_lse,
                                    const int4* seg_rec, const int* seg_pre, cudaStream_t stream) {
    if (num_ctas < 2) return cudaSuccess;  // one CTA splits nothing
    const int R = a.k * (a.Hq / a.Hkv);
    const int64_t segs = (int64_t)a.B * a.Hkv;
    if (segs <= num_ctas - 1) {
        dim3 cgrid((unsigned)segs, (R + 7) / 8);
        return launch_dependent(combine_tc_kernel<true>, cgrid, dim3(256), 0, stream, a, num_ctas,
                                alpha, part_o, part_lse, seg_rec, seg_pre);
    } else {
        dim3 cgrid(num_ctas - 1, (R + 7) / 8);
        return launch_dependent(combine_tc_kernel<false>, cgrid, dim3(256), 0, stream, a, num_ctas,
                                alpha, part_o, part_lse, seg_rec, seg_pre);
    }
    return cudaGetLastError();
}

}  // namespace specv

// Verification attention for small query-row sets: k * G <= 16 rows per
// (sequence, kv-head), bf16 queries over a bf16 paged KV cache, head_dim 128.
//
// What it computes: multi-query causal attention of each sequence's k draft
// queries over its paged cache ("Decoding Speculative Decoding from First
// Principles", "Parallelizing method 2: sequence parallel" and "Speculating
// to get sequence parallelism during decode"): query i of sequence b sees
// keys 0 .. ctx_b + i; kv-head g serves q-heads g*G .. g*G+G-1.
//
// Design: the R <= 16 query rows of a (sequence, kv-head) form exactly one
// 16-row tile of the warp-level tensor-core MMA (m16n8k16, bf16 in, fp32
// accumulate), so every K/V byte is read from HBM once and used for all rows.
// Unlike a 128-row tcgen05 tile (mostly padding at 8-16 rows), the softmax
// lives in registers: no TMEM round trips and no per-tile hand-off between
// warps.
//
//  * Work: a stream-K list of 128-key tiles of every (sequence, kv-head)
//    segment over a persistent grid; a segment cut by a CTA-range boundary
//    leaves (O/l, lse) partials, and the last of its pieces to finish merges
//    them (atomic arrival count per segment, no waiting), so one launch does
//    the whole call.
//  * Warps: eight, two per SM sub-partition so that one hides the other's
//    MMA and shared-memory latency.  Warp w owns keys [16w, 16w+16) of every
//    tile -- one 4 KB TMA page box of K and one of V -- and keeps a private
//    ring of NS such box pairs: it refills a stage with its box NS tiles
//    ahead as soon as it has used it, so there is no producer warp, no
//    "stage empty" barrier and no serial TMA issue loop (each warp issues two
//    boxes per tile).  The block-table entry of that box is read at the start
//    of the tile and used after it, hiding its latency behind the MMAs.
//    Warp 0 also loads each piece's query rows, one piece ahead, into two
//    staging buffers.
//  * Per warp and tile: S = Q K^T (16 MMAs, K via ldmatrix), masked online
//    softmax in registers with a lazily moved reference max, P V (16 MMAs,
//    V via ldmatrix.trans, P straight from the S accumulators).  The eight
//    warps' (max, sum, O) are merged once per segment piece in shared memory.
//  * Every mbarrier wait is bounded (1 s); a timeout sets the device error
//    word and an abort flag after which every warp skips its remaining work,
//    still passing every CTA barrier, and waits (bounded) for its own loads
//    in flight before the CTA exits.
#include <cuda.h>
#include <math.h>

#include "common.cuh"

namespace specv {
namespace {

constexpr int D = 128;
constexpr int NW = 8;                // compute warps
constexpr int BOX_ROWS = 16;         // keys per TMA box = keys of one warp in a tile
constexpr int TN = NW * BOX_ROWS;    // 128 keys per tile
constexpr int NS = 3;                // stages of each warp's private K/V ring
constexpr int BOX_BYTES = BOX_ROWS * D * 2;  // 4 KB
constexpr int WSTAGE_BYTES = 2 * BOX_BYTES;  // one warp's K box + V box
constexpr int QROWS = 16;
constexpr int Q_HALF = QROWS * 128;  // 2 KB: 64 head-dim columns of 16 rows
constexpr int Q_BUF = 2 * Q_HALF;
constexpr int THREADS = NW * 32;
constexpr int MAX_BATCH = 1024;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;
// tiles charged per segment in the split over the CTAs: none -- measured on
// the 7B and 8B shapes, any charge made the slowest CTA later (this
// kernel's per-piece work is small next to its 128-key tiles)
constexpr int kSplitAlpha = 0;

using Cursor = CursorT<TN>;

struct Smem {
    static constexpr int RING = 0;                              // [NS][NW][K box, V box]
    static constexpr int Q = RING + NS * NW * WSTAGE_BYTES;     // 2 buffers x 2 halves x 2 KB
    static constexpr int PREF = Q + 2 * Q_BUF;                   // [16][D] float: other piece's O
    static constexpr int PREF_LSE = PREF + QROWS * D * 4;       // [128] float: its lse slot
    static constexpr int BARS = PREF_LSE + 128 * 4;
    static constexpr int B_KVFULL = 0, B_QFULL = NS * NW, NUM_BARS = NS * NW + 2;
    // abort flag, prefetch state / slot, then (at +16) the CTA's tile range
    static constexpr int MISC = BARS + NUM_BARS * 8;
    static constexpr int STAT = MISC + 32;                      // [NW][16] (m, l)
    static constexpr int CTX = STAT + 2 * NW * QROWS * 4;
    static constexpr int PRE = CTX + MAX_BATCH * 4;
    static constexpr int END = PRE + (MAX_BATCH + 1) * 4;
};
constexpr size_t SMEM_BYTES = Smem::END + 1024;
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
static_assert(NS <= 32, "stage bit masks");

struct MmaParams {
    AttnArgs a;
    float* part_o;    // [2*C][128][D]
    float* part_lse;  // [2*C][128]
};

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
// D += A(16x16 bf16, row) * B(16x8 bf16, col), fp32 accumulate
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
        "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Byte offset of (row, 16-byte chunk c of the 256-byte row) in a block laid
// out as [2 halves][rows][128 B] with the 128-byte swizzle (chunk ^ row%8).
__device__ __forceinline__ uint32_t sw_off(int row, int c, int half_bytes) {
    return (c >> 3) * half_bytes + row * 128 + (((c & 7) ^ (row & 7)) << 4);
}

__global__ void __launch_bounds__(THREADS, 1)
attn_mma_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
                const __grid_constant__ CUtensorMap vmap, const MmaParams prm) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const AttnArgs& a = prm.a;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + Smem::BARS);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + Smem::MISC);
    volatile int* s_pf = reinterpret_cast<volatile int*>(sm + Smem::MISC + 4);
    volatile int* s_pf_slot = reinterpret_cast<volatile int*>(sm + Smem::MISC + 8);
    int* s_ctx = reinterpret_cast<int*>(sm + Smem::CTX);
    int* s_pre = reinterpret_cast<int*>(sm + Smem::PRE);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int B = a.B, k = a.k, Hkv = a.Hkv, G = a.Hq / a.Hkv, R = k * G, P = a.P;

    if (tid == 0) {
        for (int i = 0; i < NS * NW; ++i) mbar_init(&bars[Smem::B_KVFULL + i], 1);
        mbar_init(&bars[Smem::B_QFULL], 1);
        mbar_init(&bars[Smem::B_QFULL + 1], 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    {
        // Q rows R..15 stay zero (the TMA writes rows 0..R-1 only)
        uint4* q4 = reinterpret_cast<uint4*>(sm + Smem::Q);
        for (int e = tid; e < 2 * Q_BUF / 16; e += THREADS) q4[e] = make_uint4(0, 0, 0, 0);
        fence_proxy_async_smem();
    }
    // the grids before this one have finished with every buffer this call touches
    grid_dep_launch_dependents();
    grid_dep_wait();
    if (warp == 0) {
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
    }

    // the CTA's tile range [t_begin, t_end), kept in shared memory; the split
    // is rebuilt where the merge needs it rather than held in registers
    int64_t* s_rng = reinterpret_cast<int64_t*>(sm + Smem::MISC + 16);
    auto make_split = [&]() {
        TileSplit sp;
        sp.init(s_pre, B, Hkv, a.split_alpha < 0 ? kSplitAlpha : a.split_alpha, gridDim.x);
        return sp;
    };
    if (warp == 0) {
        __syncwarp();  // the prefix above, written by this warp's lanes
        if (lane < 2) s_rng[lane] = make_split().begin(blockIdx.x + lane);
    }
    __syncthreads();
    auto t_begin = [&]() { return ld_shared_s64(s_rng); };
    auto t_end = [&]() { return ld_shared_s64(s_rng + 1); };
    const int n_tiles = (int)(t_end() - t_begin());

    {
        // ===== warp w owns keys [16w, 16w+16) of every tile and keeps its own
        // ring of NS K/V boxes, refilling a stage as soon as it is done with
        // it (no other warp reads this warp's boxes); warp 0 also loads the
        // query rows of each segment piece, one piece ahead, into two buffers
        const int g = lane >> 2, t4 = lane & 3;  // MMA fragment group / thread in group
        const float sl2 = a.scale * kLog2e;
        const uint32_t q_base = smem_u32(sm + Smem::Q);
        float* s_m = reinterpret_cast<float*>(sm + Smem::STAT);
        float* s_l = s_m + NW * QROWS;
        // the two rows this thread holds in every fragment: g and g + 8
        int irow[2];
        irow[0] = g < R ? g / G : k - 1;
        irow[1] = g + 8 < R ? (g + 8) / G : k - 1;
        uint64_t mrow[2] = {0, 0};  // draft bits of the two rows, per piece
        const int kv0 = warp * BOX_ROWS;  // this warp's first key in every tile
        uint8_t* ring = sm + Smem::RING + warp * WSTAGE_BYTES;  // stage s at + s * NW * WSTAGE_BYTES
        uint64_t* full = &bars[Smem::B_KVFULL + warp];           // stage s at full[s * NW]
        const uint64_t pol = l2_policy_evict_first();
        if (lane == 0) {
            prefetch_tmap(&kmap);
            prefetch_tmap(&vmap);
            if (warp == 0) prefetch_tmap(&qmap);
        }
        // does this warp's box of tile c hold any key of the sequence (warp-uniform)
        auto box_valid = [&](const Cursor& c) { return c.lt * TN + kv0 < s_ctx[c.b] + k; };
        auto table_entry = [&](const Cursor& c) {
            return a.block_table + (int64_t)c.b * a.max_pages + (c.lt * TN + kv0) / P;
        };
        // lane 0: load this warp's K and V boxes of tile c into stage st
        auto issue = [&](int st, const Cursor& c, int page) {
            if (page < 0 || page >= a.num_pages) {
                raise_device_error(a.dev_err, SPEC_DEVERR_PAGE);
                page = 0;
            }
            const int row = (page * Hkv + c.kvh) * P + (c.lt * TN + kv0) % P;
            uint8_t* dst = ring + st * NW * WSTAGE_BYTES;
            mbar_arrive_expect_tx(&full[st * NW], 2u * BOX_BYTES);
            tma_load_3d_hint(dst, &kmap, &full[st * NW], 0, row, 0, pol);
            tma_load_3d_hint(dst + BOX_BYTES, &vmap, &full[st * NW], 0, row, 0, pol);
        };

        // warp 0, lane 0: query rows of piece j (sequence b, kv-head kvh) into buffer j % 2
        auto issue_q = [&](int j, int b, int kvh) {
            uint64_t* bar = &bars[Smem::B_QFULL + (j & 1)];
            mbar_arrive_expect_tx(bar, 2 * R * 128);
            for (int h = 0; h < 2; ++h)
                tma_load_3d(sm + Smem::Q + (j & 1) * Q_BUF + h * Q_HALF, &qmap, bar, h * 64,
                            kvh * G, b * k);
        };
        // does a piece follow the one of cursor c in this CTA's range
        auto has_next_piece = [&](const Cursor& c) { return c.seg_start + c.nb < t_end(); };

        Cursor cur, ahead;  // ahead: the tile NS past cur, the next one to load
        uint32_t pending = 0, phase = 0;  // per stage: a load in flight / the parity it completes
        int q_issued = 0;                 // warp 0: pieces whose query rows were loaded
        if (n_tiles > 0) {
            cur.init(t_begin(), s_pre, s_ctx, B, Hkv, k);
            ahead = cur;
            if (warp == 0) {
                q_issued = has_next_piece(cur) ? 2 : 1;
                if (lane == 0) {
                    issue_q(0, cur.b, cur.kvh);
                    if (q_issued == 2)
                        issue_q(1, cur.kvh + 1 < Hkv ? cur.b : cur.b + 1,
                                cur.kvh + 1 < Hkv ? cur.kvh + 1 : 0);
                }
            }
            // prologue: block-table entries of tiles 0..NS-1 first, then their loads
            int pg[NS];
            {
                Cursor c = cur;
#pragma unroll
                for (int j = 0; j < NS; ++j) {
                    pg[j] = -1;
                    if (j < n_tiles) {
                        if (lane == 0 && box_valid(c)) pg[j] = __ldg(table_entry(c));
                        if (j + 1 < n_tiles) c.next(s_ctx, Hkv, k);
                    }
                }
            }
#pragma unroll
            for (int j = 0; j < NS; ++j) {
                if (j < n_tiles) {
                    if (box_valid(ahead)) {
                        if (lane == 0) issue(j, ahead, pg[j]);
                        pending |= 1u << j;
                    }
                    if (j + 1 < n_tiles) ahead.next(s_ctx, Hkv, k);
                }
            }
        }

        // pieces of a segment split over CTA ranges: CTA of tile t, empty
        // ranges, partial slot of CTA c's piece of the segment starting at s0
        // (the pieces of the segment under cursor c span CTAs first_cta(c) .. last_cta(c))
        auto first_cta = [&](const Cursor& c) {
            const TileSplit sp = make_split();
            return sp.cta_of_cost(sp.cost_of(c.b, c.kvh, 0, c.nb));
        };
        auto last_cta = [&](const Cursor& c) {
            const TileSplit sp = make_split();
            return sp.cta_of_cost(sp.cost_of(c.b, c.kvh, c.nb - 1, c.nb));
        };
        auto empty_cta = [&](int c) { return make_split().empty(c); };
        auto slot_of = [&](int c, int64_t s0) {
            return 2 * c + (s0 < make_split().begin(c) ? 0 : 1);
        };
        // End-of-range prefetch (warp 0).  The piece that ends this CTA's range
        // in a segment that continues in the next CTA is normally the last of
        // the segment's two pieces to finish (the other one ran at the start of
        // that CTA).  At its first tile warp 0 reads the segment's arrival
        // count; one tile later, if the other piece has arrived, it copies that
        // piece's partial into shared memory, and the merge then needs neither
        // this piece's partial in global memory nor another round trip.
        int pf_state = 0;  // 0 none, 1 count read issued, 2 partial copy issued, 3 unavailable,
                           // 4 other piece arrived (read its partial from global memory)
        int pf_cnt = 0, pf_slot = 0;
        float* pref = reinterpret_cast<float*>(sm + Smem::PREF);
        float* pref_lse = reinterpret_cast<float*>(sm + Smem::PREF_LSE);
        auto pf_ready = [&]() {  // warp 0, warp-uniform; acquires the other piece's partial
            const int ready = __shfl_sync(0xffffffffu, pf_cnt == 1 ? 1 : 0, 0);
            if (ready && lane == 0) __threadfence();
            __syncwarp();
            return ready != 0;
        };

        uint32_t qf[D / 16][4];
        float o[D / 8][4];
        float m_ref[2], lsum[2];
        bool ok = true;
        int pc = -1;
        for (int it = 0; it < n_tiles; ++it) {
            const bool first = (it == 0) || (cur.lt == 0);
            const bool last = (it == n_tiles - 1) || (cur.lt == cur.nb - 1);
            const int s = it % NS;
            const int ctx = s_ctx[cur.b], L = ctx + k, key0 = cur.lt * TN;
            const int nvalid = min(TN, L - key0);
            if (first) {
                mrow[0] = draft_bits(a, cur.b, irow[0]);
                mrow[1] = draft_bits(a, cur.b, irow[1]);
            }
            // block-table entry of the box NS tiles ahead: read now, used after this tile
            const bool refill = it + NS < n_tiles && box_valid(ahead);
            int pg_next = -1;
            if (refill && lane == 0) pg_next = __ldg(table_entry(ahead));
            if (first) {
                ++pc;
                // the next piece's rows go to the buffer of piece pc - 1, which
                // every warp read before the barriers that closed piece pc - 1
                if (warp == 0 && ok && pc >= 1 && has_next_piece(cur)) {
                    if (lane == 0)
                        issue_q(pc + 1, cur.kvh + 1 < Hkv ? cur.b : cur.b + 1,
                                cur.kvh + 1 < Hkv ? cur.kvh + 1 : 0);
                    q_issued = pc + 2;
                }
                if (ok)
                    ok = warp_wait(&bars[Smem::B_QFULL + (pc & 1)], (pc >> 1) & 1, abort_flag,
                                   a.dev_err);
                if (ok) {
                    // Q fragments: 16 rows x 16 columns per k-slice, from the
                    // 128-byte-swizzled staging buffer
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const int row = (lane & 7) + ((lane >> 3) & 1) * 8;
                        const int chunk = kk * 2 + (lane >> 4);
                        ldsm_x4(q_base + (pc & 1) * Q_BUF + sw_off(row, chunk, Q_HALF), qf[kk][0],
                                qf[kk][1], qf[kk][2], qf[kk][3]);
                    }
                }
#pragma unroll
                for (int j = 0; j < D / 8; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
                m_ref[0] = m_ref[1] = -INFINITY;
                lsum[0] = lsum[1] = 0.f;
                if (warp == 0 && ok && !has_next_piece(cur) && cur.seg_start + cur.nb > t_end()) {
                    const int64_t s0 = cur.seg_start;
                    int npieces = 0, other = -1;
                    for (int c = first_cta(cur); c <= last_cta(cur); ++c)
                        if (!empty_cta(c)) {
                            ++npieces;
                            if (c != (int)blockIdx.x) other = c;
                        }
                    if (npieces == 2) {
                        pf_slot = slot_of(other, s0);
                        if (lane == 0) pf_cnt = ld_acquire_gpu(&a.seg_counters[cur.b * Hkv + cur.kvh]);
                        pf_state = 1;
                    }
                }
            } else if (warp == 0 && pf_state == 1) {
                if (pf_ready()) {
                    const float* so = prm.part_o + (int64_t)pf_slot * 128 * D;
                    for (int c = lane; c < R * D / 4; c += 32) cp_async_16_cg(pref + c * 4, so + c * 4);
                    cp_async_16_cg(pref_lse + lane * 4, prm.part_lse + (int64_t)pf_slot * 128 + lane * 4);
                    cp_async_commit();
                    pf_state = 2;
                } else {
                    pf_state = 3;
                }
            }
            if (kv0 < nvalid) {
                if (ok) ok = warp_wait(&full[s * NW], (phase >> s) & 1, abort_flag, a.dev_err);
                if (ok) {
                    pending &= ~(1u << s);
                    phase ^= 1u << s;
                }
            }
            if (ok && kv0 < nvalid) {
                const uint32_t kb = smem_u32(ring + s * NW * WSTAGE_BYTES);
                const uint32_t vb = kb + BOX_BYTES;
                if (nvalid - kv0 < BOX_ROWS) {
                    // keys past the sequence end in this box: zero their V rows
                    // so that 0 * (stale or canary) never reaches O
                    uint8_t* vrow = ring + s * NW * WSTAGE_BYTES + BOX_BYTES;
                    for (int e = (nvalid - kv0) * 16 + lane; e < BOX_ROWS * 16; e += 32) {
                        const int r = e >> 4, c = e & 15;
                        *reinterpret_cast<uint4*>(vrow + sw_off(r, c, BOX_BYTES / 2)) =
                            make_uint4(0, 0, 0, 0);
                    }
                    fence_proxy_async_smem();  // before the next TMA write of this stage
                    __syncwarp();
                }
                // S = Q K^T over this warp's 16 keys: n-tile 0 = keys 0-7, 1 = keys 8-15;
                // even and odd k-steps accumulate separately (four dependent
                // MMA chains of four instead of two of eight), summed after
                float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
                float sd[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    uint32_t b00, b01, b10, b11;
                    const int key = (lane & 7) + (lane >> 4) * 8;
                    const int chunk = kk * 2 + ((lane >> 3) & 1);
                    ldsm_x4(kb + sw_off(key, chunk, BOX_BYTES / 2), b00, b01, b10, b11);
                    mma16816((kk & 1) ? sd[0] : sc[0], qf[kk], b00, b01);
                    mma16816((kk & 1) ? sd[1] : sc[1], qf[kk], b10, b11);
                }
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int e = 0; e < 4; ++e) sc[nt][e] += sd[nt][e];
                // masked scores (log2 units); -inf where the key is invisible
                float v[2][4];
                float mt[2] = {-INFINITY, -INFINITY};
                if (key0 + kv0 + BOX_ROWS <= ctx) {
                    // every key of this warp's slice is context: all visible
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            v[nt][e] = sc[nt][e] * sl2;
                            mt[e >> 1] = fmaxf(mt[e >> 1], v[nt][e]);
                        }
                } else {
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int hr = e >> 1;  // 0: row g, 1: row g + 8
                            const int kr = kv0 + nt * 8 + t4 * 2 + (e & 1);
                            // the context, then the drafts of the row's bits
                            // (causal chain: keys <= ctx + i)
                            const int key = key0 + kr;
                            const bool vis =
                                kr < nvalid &&
                                (key < ctx || ((mrow[hr] >> (key < ctx ? 0 : key - ctx)) & 1ull));
                            v[nt][e] = vis ? sc[nt][e] * sl2 : -INFINITY;
                            mt[hr] = fmaxf(mt[hr], v[nt][e]);
                        }
                }
                float alpha[2];
                bool moved = false;
#pragma unroll
                for (int hr = 0; hr < 2; ++hr) {
                    mt[hr] = fmaxf(mt[hr], __shfl_xor_sync(0xffffffffu, mt[hr], 1));
                    mt[hr] = fmaxf(mt[hr], __shfl_xor_sync(0xffffffffu, mt[hr], 2));
                    const float m_new = fmaxf(m_ref[hr], mt[hr]);
                    alpha[hr] = 1.f;
                    if (m_new > m_ref[hr] + kRescaleThreshold) {
                        alpha[hr] = m_ref[hr] == -INFINITY ? 0.f : fast_exp2(m_ref[hr] - m_new);
                        m_ref[hr] = m_new;
                        lsum[hr] *= alpha[hr];
                        moved = true;
                    }
                }
                if (__any_sync(0xffffffffu, moved)) {
#pragma unroll
                    for (int j = 0; j < D / 8; ++j) {
                        o[j][0] *= alpha[0];
                        o[j][1] *= alpha[0];
                        o[j][2] *= alpha[1];
                        o[j][3] *= alpha[1];
                    }
                }
                const float mu0 = m_ref[0] == -INFINITY ? 0.f : m_ref[0];
                const float mu1 = m_ref[1] == -INFINITY ? 0.f : m_ref[1];
                float p[2][4];
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                    p[nt][0] = fast_exp2(v[nt][0] - mu0);
                    p[nt][1] = fast_exp2(v[nt][1] - mu0);
                    p[nt][2] = fast_exp2(v[nt][2] - mu1);
                    p[nt][3] = fast_exp2(v[nt][3] - mu1);
                    lsum[0] += p[nt][0] + p[nt][1];
                    lsum[1] += p[nt][2] + p[nt][3];
                }
                // P as the A operand of P V: the two 8-key accumulator tiles
                // are exactly the two 8-column halves of a 16x16 A fragment
                uint32_t pa[4];
                pa[0] = pack_bf16x2(p[0][0], p[0][1]);
                pa[1] = pack_bf16x2(p[0][2], p[0][3]);
                pa[2] = pack_bf16x2(p[1][0], p[1][1]);
                pa[3] = pack_bf16x2(p[1][2], p[1][3]);
                // O += P V: 16 output n-tiles of 8 head-dim columns
#pragma unroll
                for (int j = 0; j < D / 8; j += 2) {
                    uint32_t b00, b01, b10, b11;
                    const int key = (lane & 7) + ((lane >> 3) & 1) * 8;
                    const int chunk = j + (lane >> 4);
                    ldsm_x4_t(vb + sw_off(key, chunk, BOX_BYTES / 2), b00, b01, b10, b11);
                    mma16816(o[j], pa, b00, b01);
                    mma16816(o[j + 1], pa, b10, b11);
                }
            }
            __syncwarp();
            // every read of stage s is done (its values fed the MMAs): refill it
            // with this warp's box NS tiles ahead -- after the merge when this
            // tile ends a segment piece, since the merge stages O in it
            if (refill && ok && !last) {
                if (lane == 0) issue(s, ahead, pg_next);
                pending |= 1u << s;
            }

            if (last) {
                // ---- merge the warps' (max, sum, O) of this segment piece
                if (warp == 0) {
                    if (pf_state == 1) pf_state = pf_ready() ? 4 : 3;
                    if (pf_state == 2) cp_async_wait<0>();
                    if (lane == 0) {
                        *s_pf = pf_state;
                        *s_pf_slot = pf_slot;
                    }
                }
                float lrow[2];
#pragma unroll
                for (int hr = 0; hr < 2; ++hr) {
                    lrow[hr] = lsum[hr];
                    lrow[hr] += __shfl_xor_sync(0xffffffffu, lrow[hr], 1);
                    lrow[hr] += __shfl_xor_sync(0xffffffffu, lrow[hr], 2);
                }
                if (t4 == 0) {
                    s_m[warp * QROWS + g] = m_ref[0];
                    s_m[warp * QROWS + g + 8] = m_ref[1];
                    s_l[warp * QROWS + g] = lrow[0];
                    s_l[warp * QROWS + g + 8] = lrow[1];
                }
                named_bar_sync(1, NW * 32);
                const int pf = *s_pf;
                float wgt[2], lse[2];
#pragma unroll
                for (int hr = 0; hr < 2; ++hr) {
                    const int row = g + 8 * hr;
                    float mt = -INFINITY;
#pragma unroll
                    for (int w = 0; w < NW; ++w) mt = fmaxf(mt, s_m[w * QROWS + row]);
                    float Ls = 0.f;
#pragma unroll
                    for (int w = 0; w < NW; ++w) {
                        const float mw = s_m[w * QROWS + row];
                        if (mw != -INFINITY) Ls += s_l[w * QROWS + row] * fast_exp2(mw - mt);
                    }
                    wgt[hr] = (Ls > 0.f && m_ref[hr] != -INFINITY) ? fast_exp2(m_ref[hr] - mt) / Ls
                                                                   : 0.f;
                    lse[hr] = Ls > 0.f ? (mt + log2f(Ls)) * kLn2 : -INFINITY;
                }
                // every warp stages its weighted O (fp32 [16][128], 8-column
                // blocks XOR-swizzled by row) in its own stage s, free until the
                // deferred refill below
                {
                    float* ob = reinterpret_cast<float*>(ring + s * NW * WSTAGE_BYTES);
#pragma unroll
                    for (int j = 0; j < D / 8; ++j) {
                        const int col = ((j ^ g) << 3) + t4 * 2;
                        *reinterpret_cast<float2*>(ob + g * D + col) =
                            make_float2(o[j][0] * wgt[0], o[j][1] * wgt[0]);
                        *reinterpret_cast<float2*>(ob + (g + 8) * D + col) =
                            make_float2(o[j][2] * wgt[1], o[j][3] * wgt[1]);
                    }
                    fence_proxy_async_smem();  // before the refill TMA writes this stage
                }
                named_bar_sync(1, NW * 32);
                // warp w sums the eight staged blocks of output columns
                // [16w, 16w+16): lane -> row lane/2, 8 columns as two 16-byte
                // halves, odd rows reading the upper half first so that each
                // quarter-warp touches eight distinct bank groups
                const int rr = lane >> 1, jb = 2 * warp + (lane & 1), hf = rr & 1;
                float acc[8];
                {
                    float4 sa = make_float4(0.f, 0.f, 0.f, 0.f), sb = sa;
#pragma unroll
                    for (int w = 0; w < NW; ++w) {
                        const float4* src = reinterpret_cast<const float4*>(
                            sm + Smem::RING + (s * NW + w) * WSTAGE_BYTES +
                            (rr * D + ((jb ^ (rr & 7)) << 3)) * 4);
                        const float4 x = src[hf], y = src[hf ^ 1];
                        sa.x += x.x; sa.y += x.y; sa.z += x.z; sa.w += x.w;
                        sb.x += y.x; sb.y += y.y; sb.z += y.z; sb.w += y.w;
                    }
                    const float4 lo4 = hf ? sb : sa, hi4 = hf ? sa : sb;
                    acc[0] = lo4.x; acc[1] = lo4.y; acc[2] = lo4.z; acc[3] = lo4.w;
                    acc[4] = hi4.x; acc[5] = hi4.y; acc[6] = hi4.z; acc[7] = hi4.w;
                }
                const bool complete = cur.seg_start >= t_begin() && cur.seg_start + cur.nb <= t_end();
                const int seg = cur.b * Hkv + cur.kvh;
                const int64_t orow_rr =
                    ((int64_t)cur.b * k + rr / G) * a.Hq + cur.kvh * G + rr % G;
                auto store_out = [&](int64_t orow, int c8, const float* v, float scale_) {
                    uint4 w4;
                    w4.x = pack_bf16x2(v[0] * scale_, v[1] * scale_);
                    w4.y = pack_bf16x2(v[2] * scale_, v[3] * scale_);
                    w4.z = pack_bf16x2(v[4] * scale_, v[5] * scale_);
                    w4.w = pack_bf16x2(v[6] * scale_, v[7] * scale_);
                    *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.out) + orow * D + c8 * 8) = w4;
                };
                bool count_arrival = false;
                if (complete) {
                    if (ok) {
                        if (rr < R) store_out(orow_rr, jb, acc, 1.f);
                        if (warp == 0 && t4 == 0 && a.lse) {
#pragma unroll
                            for (int hr = 0; hr < 2; ++hr) {
                                const int r2 = g + 8 * hr;
                                if (r2 < R)
                                    a.lse[((int64_t)cur.b * k + r2 / G) * a.Hq + cur.kvh * G + r2 % G] =
                                        lse[hr];
                            }
                        }
                    }
                } else if (pf == 2 || pf == 4) {
                    // every other piece of the segment has arrived: merge with
                    // its partial here, without publishing this one
                    if (ok && rr < R) {
                        float mt = -INFINITY;
#pragma unroll
                        for (int w = 0; w < NW; ++w) mt = fmaxf(mt, s_m[w * QROWS + rr]);
                        float Ls = 0.f;
#pragma unroll
                        for (int w = 0; w < NW; ++w) {
                            const float mw = s_m[w * QROWS + rr];
                            if (mw != -INFINITY) Ls += s_l[w * QROWS + rr] * fast_exp2(mw - mt);
                        }
                        const float l_own = Ls > 0.f ? (mt + log2f(Ls)) * kLn2 : -INFINITY;
                        const int oslot = *s_pf_slot;
                        float l_oth;
                        float4 y0, y1;
                        if (pf == 2) {
                            l_oth = pref_lse[rr];
                            y0 = *reinterpret_cast<const float4*>(pref + rr * D + jb * 8);
                            y1 = *reinterpret_cast<const float4*>(pref + rr * D + jb * 8 + 4);
                        } else {
                            l_oth = __ldcg(prm.part_lse + (int64_t)oslot * 128 + rr);
                            const float4* src = reinterpret_cast<const float4*>(
                                prm.part_o + ((int64_t)oslot * 128 + rr) * D + jb * 8);
                            y0 = __ldcg(src);
                            y1 = __ldcg(src + 1);
                        }
                        const float mx = fmaxf(l_own, l_oth);
                        const float w1 = l_own == -INFINITY ? 0.f : __expf(l_own - mx);
                        const float w2 = l_oth == -INFINITY ? 0.f : __expf(l_oth - mx);
                        const float tot = w1 + w2, inv = tot > 0.f ? 1.f / tot : 0.f;
                        float v8[8] = {w1 * acc[0] + w2 * y0.x, w1 * acc[1] + w2 * y0.y,
                                       w1 * acc[2] + w2 * y0.z, w1 * acc[3] + w2 * y0.w,
                                       w1 * acc[4] + w2 * y1.x, w1 * acc[5] + w2 * y1.y,
                                       w1 * acc[6] + w2 * y1.z, w1 * acc[7] + w2 * y1.w};
                        store_out(orow_rr, jb, v8, inv);
                        if (jb == 0 && a.lse) a.lse[orow_rr] = tot > 0.f ? mx + logf(tot) : -INFINITY;
                    }
                    if (tid == 0) a.seg_counters[seg] = 0;  // ready for the next call
                } else {
                    // publish this piece's partial; warp 0 then counts the
                    // arrival, and the last piece of the segment merges them all
                    const int slot = 2 * blockIdx.x + (cur.seg_start < t_begin() ? 0 : 1);
                    if (ok) {
                        if (rr < R) {
                            float4* dst = reinterpret_cast<float4*>(
                                prm.part_o + ((int64_t)slot * 128 + rr) * D + jb * 8);
                            dst[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
                            dst[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
                        }
                        if (warp == 0 && t4 == 0) {
#pragma unroll
                            for (int hr = 0; hr < 2; ++hr)
                                if (g + 8 * hr < R) prm.part_lse[(int64_t)slot * 128 + g + 8 * hr] = lse[hr];
                        }
                    }
                    count_arrival = true;
                }
                named_bar_sync(1, NW * 32);  // staged O read, partials written
                if (refill && ok) {
                    if (lane == 0) issue(s, ahead, pg_next);
                    pending |= 1u << s;
                }
                if (count_arrival && warp == 0) {
                    const int64_t s0 = cur.seg_start;
                    const int c_first = first_cta(cur), c_last = last_cta(cur);
                    const int ncta = c_last - c_first + 1;
                    // lane j: the partial slot of CTA c_first + j's piece, -1 for an
                    // empty range (computed once here when the segment spans at most
                    // 32 CTAs; per use beyond that)
                    int my_slot = -1;
                    if (lane < ncta) {
                        const TileSplit sp = make_split();
                        const int c = c_first + lane;
                        const int64_t b0 = sp.begin(c), b1 = sp.begin(c + 1);
                        if (b0 != b1) my_slot = 2 * c + (s0 < b0 ? 0 : 1);
                    }
                    const unsigned pieces = __ballot_sync(0xffffffffu, my_slot >= 0);
                    int npieces = __popc(pieces);
                    for (int j0 = 32; j0 < ncta; j0 += 32) {
                        const bool ne = j0 + lane < ncta && !empty_cta(c_first + j0 + lane);
                        npieces += __popc(__ballot_sync(0xffffffffu, ne));
                    }
                    int merger = 0;
                    if (lane == 0) {
                        __threadfence();  // release the partials (ordered by the barrier)
                        merger = atomicAdd(&a.seg_counters[seg], 1) == npieces - 1;
                        if (merger) __threadfence();  // acquire the other pieces' partials
                    }
                    merger = __shfl_sync(0xffffffffu, merger, 0);
                    if (merger) {
                        // warp 0 merges every piece's partial; the other warps go on.
                        // Every lane runs every round (the shuffles need the whole warp)
                        for (int base = 0; base < R * (D / 8); base += 32) {
                            const int idx = base + lane;
                            const bool act = idx < R * (D / 8);
                            const int r2 = act ? idx / (D / 8) : 0, c8 = idx % (D / 8);
                            float mx = -INFINITY, tot = 0.f;
                            float m8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
                            auto fold = [&](int sl) {
                                const float lw = __ldcg(prm.part_lse + (int64_t)sl * 128 + r2);
                                const float4* src = reinterpret_cast<const float4*>(
                                    prm.part_o + ((int64_t)sl * 128 + r2) * D + c8 * 8);
                                const float4 x0 = __ldcg(src), x1 = __ldcg(src + 1);
                                if (lw == -INFINITY) return;
                                const float mn = fmaxf(mx, lw);
                                const float sa = mx == -INFINITY ? 0.f : __expf(mx - mn);
                                const float sb = __expf(lw - mn);
                                mx = mn;
                                tot = tot * sa + sb;
                                m8[0] = m8[0] * sa + sb * x0.x; m8[1] = m8[1] * sa + sb * x0.y;
                                m8[2] = m8[2] * sa + sb * x0.z; m8[3] = m8[3] * sa + sb * x0.w;
                                m8[4] = m8[4] * sa + sb * x1.x; m8[5] = m8[5] * sa + sb * x1.y;
                                m8[6] = m8[6] * sa + sb * x1.z; m8[7] = m8[7] * sa + sb * x1.w;
                            };
                            if (ncta <= 32) {
                                for (unsigned m = pieces; m; m &= m - 1) {
                                    const int sl = __shfl_sync(0xffffffffu, my_slot, __ffs(m) - 1);
                                    if (act) fold(sl);
                                }
                            } else if (act) {
                                for (int c = c_first; c <= c_last; ++c)
                                    if (!empty_cta(c)) fold(slot_of(c, s0));
                            }
                            if (act) {
                                const int64_t orow =
                                    ((int64_t)cur.b * k + r2 / G) * a.Hq + cur.kvh * G + r2 % G;
                                store_out(orow, c8, m8, tot > 0.f ? 1.f / tot : 0.f);
                                if (c8 == 0 && a.lse) a.lse[orow] = tot > 0.f ? mx + logf(tot) : -INFINITY;
                            }
                        }
                        if (lane == 0) a.seg_counters[seg] = 0;  // ready for the next call
                    }
                }
            }
            if (it + NS + 1 < n_tiles) ahead.next(s_ctx, Hkv, k);
            if (it + 1 < n_tiles) cur.next(s_ctx, Hkv, k);
        }
        // loads still in flight (only after an abort) land before the CTA exits
        if (lane == 0) {
            for (int st = 0; st < NS; ++st)
                if ((pending >> st) & 1) mbar_drain(&full[st * NW], (phase >> st) & 1);
            // warp 0 issued piece j only after waiting for piece j - 2 of the
            // same buffer, so at most the last load of each buffer is in flight
            for (int j = q_issued - 2; j < q_issued; ++j)
                if (j >= 0) mbar_drain(&bars[Smem::B_QFULL + (j & 1)], (j >> 1) & 1);
        }
        cp_async_wait<0>();  // a prefetch an abort left unconsumed
    }
    __syncthreads();
}

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

bool mma_supported(const AttnArgs& a) {
    const int G = a.Hq / a.Hkv;
    const bool pow2 = (a.P & (a.P - 1)) == 0;
    return a.q_dtype == SPEC_DTYPE_BF16 && a.kv_dtype == SPEC_DTYPE_BF16 && a.D == D &&
           a.k * G <= QROWS && pow2 && a.P >= 16 && a.P <= 256 && a.B <= MAX_BATCH &&
           (int64_t)a.num_pages * a.Hkv * a.P < (1LL << 31) && (int64_t)a.B * a.k < (1LL << 31);
}

cudaError_t launch_attn_mma(const AttnArgs& a, int num_ctas, void* workspace, cudaStream_t stream) {
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
    const cuuint64_t rows = (cuuint64_t)a.num_pages * a.Hkv * a.P;
    for (int t = 0; t < 2; ++t) {
        cuuint64_t dims[3] = {64, rows, 2};
        cuuint64_t strides[2] = {(cuuint64_t)D * 2, 128};
        cuuint32_t box[3] = {64, (cuuint32_t)BOX_ROWS, 2};
        cuuint32_t es[3] = {1, 1, 1};
        if (encode(t == 0 ? &kmap : &vmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                   const_cast<void*>(t == 0 ? a.k_cache : a.v_cache), dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    MmaParams prm;
    prm.a = a;
    prm.part_o = static_cast<float*>(workspace);
    prm.part_lse = prm.part_o + (size_t)2 * num_ctas * 128 * D;
    cudaError_t e = cudaFuncSetAttribute(attn_mma_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)SMEM_BYTES);
    if (e != cudaSuccess) return e;
    e = launch_dependent(attn_mma_kernel, dim3(num_ctas), dim3(THREADS), SMEM_BYTES, stream, qmap,
                         kmap, vmap, prm);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace specv

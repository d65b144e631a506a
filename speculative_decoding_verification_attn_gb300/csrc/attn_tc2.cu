// Verification attention on the tcgen05 tensor cores with 128-key tiles, for
// up to 128 query rows per kv-head over a bf16 or INT8 paged cache, head_dim
// 128.
//
// What it computes: multi-query causal attention of each sequence's k draft
// queries over its paged cache ("Decoding Speculative Decoding from First
// Principles", "Parallelizing method 2: sequence parallel" and "Speculating
// to get sequence parallelism during decode"): query i of sequence b sees
// keys 0 .. ctx_b + i (or the drafts of its tree row); kv-head g serves
// q-heads g*G .. g*G+G-1.  All R = k*G query rows of a (sequence, kv-head)
// are the M side of one 128-row MMA, so every K/V byte is read once.
//
// Design.  The 64-key-tile kernel is paced by its hand-offs (each tile: 8
// Q K^T and 4 P V MMAs, two commits, a softmax set barrier and a P V issue
// from a softmax warp).  Here a tile is 128 keys: Q K^T is 8 MMAs of N = 128
// (A = Q from shared memory, B = K in 8-key groups, one TMA copy per page
// chunk), and the hand-offs per key halve.
//  * TMEM (512 columns): S of set 0 [0,128), S of set 1 [128,256), O of set 0
//    [256,384), O of set 1 [384,512).  P (bf16) is written over the S columns
//    it came from: keys 0..63 to columns [0,32), keys 64..127 to [64,96) of
//    the set's S buffer, which therefore stays busy until P V has read it.
//  * Warps: 0-3 and 8-11 two softmax sets taking alternate tiles, each with
//    its own S buffer, running max, row sum and O; 4 Q loads and Q K^T
//    issue; 5 and 6 TMA producers of K and of V (tile it into slot it % 2
//    of each ring); 7 P V issue.
//  * The softmax of a tile reads S in two 64-column halves: the row maximum
//    of both first, then p = 2^(s - m) of each half, packed to bf16 into
//    TMEM.  The running maximum moves only when it grows by more than 2^8
//    (O and the row sum share it, so the result is exact in real arithmetic).
//  * Work split: stream-K over the 128-key tiles with the per-segment charge
//    of TileSplit; partials of segments cut by a CTA range are merged by the
//    combine kernel of the 64-key kernel (same records, this kernel's tiles).
//  * INT8 cache (per-key fp16 scales): the producers land the raw int8 tile
//    in the upper half of its operand slot and its scales in a small stage;
//    four more warps (12-13 K, 14-15 V) dequantize it in place to fp16
//    (int8 * scale, one rounding) in the layout the MMAs read.  q is turned
//    to fp16 in place once per piece and P is packed as fp16, so A and B
//    share a type.
//    The 16 warps share the 64K registers of the block unevenly
//    (setmaxnreg): softmax 160 each, issue / copy 80, dequantization 112.
//  * Every mbarrier wait is bounded (1 s); a timeout sets the device error
//    word and an abort flag, after which every role skips its remaining work
//    (the softmax sets still pass their pairwise barriers), drains its copies
//    and tensor-core operations, and returns.
#include <cuda.h>
#include <math.h>

#include "common.cuh"

namespace specv {
namespace {

constexpr int D = 128;
constexpr int TN = 128;                 // keys per tile
constexpr int ROWS = 128;               // MMA M
constexpr int NVB = TN / 16;            // P V MMAs per tile (16 keys each)
constexpr int Q_HALF = ROWS * 128;      // 16 KB: 64 head-dim columns of Q
constexpr int Q_BYTES = 2 * Q_HALF;     // 32 KB
constexpr int SLOT_BYTES = TN * D * 2;  // 32 KB: one tile of K or of V
constexpr int LOOKAHEAD = 6;            // tiles of block-table entries prefetched
constexpr int MAX_BATCH = 1024;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t TM_S = 0, TM_O = 256;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units
// tiles charged per segment in the split over the CTAs (a piece boundary
// drains the pipeline: the next piece's Q, the merge of the two sets)
constexpr int kSplitAlpha = 3;

// A / B operand formats of tcgen05.mma kind::f16: bf16 cache: bf16; INT8
// cache widened to fp16, so q and P are fp16 there too
template <bool KV8>
constexpr uint32_t idesc_qk() {
    return KV8 ? umma_idesc_f16(ROWS, TN, 0, 0) : umma_idesc_bf16(ROWS, TN, 0, 0);
}
template <bool KV8>
constexpr uint32_t idesc_pv() {  // B (V) MN-major
    return KV8 ? umma_idesc_f16(ROWS, D, 0, 1) : umma_idesc_bf16(ROWS, D, 0, 1);
}
template <bool KV8>
constexpr int threads() { return KV8 ? 16 * 32 : 12 * 32; }

using Cursor = CursorT<TN>;

// INT8: the raw int8 tile (128 keys x 128 B = 16 KB) lands in the upper half
// of its 32 KB operand slot and is dequantized in place
constexpr int RAW_OFF = SLOT_BYTES / 2;

struct Smem {
    static constexpr int Q = 0;                         // 2 buffers (piece parity)
    static constexpr int KS = Q + 2 * Q_BYTES;          // 2 K slots
    static constexpr int VS = KS + 2 * SLOT_BYTES;      // 2 V slots
    static constexpr int BARS = VS + 2 * SLOT_BYTES;
    static constexpr int B_KFULL = 0, B_KEMPTY = 2, B_VFULL = 4, B_VEMPTY = 6, B_QFULL = 8,
                         B_QFREE = 10, B_SFULL = 12, B_PREADY = 14, B_SFREE = 16,
                         B_EPI = 18, B_DRAIN = 19, B_KREADY = 21, B_VREADY = 23, NUM_BARS = 25;
    static constexpr int MISC = BARS + NUM_BARS * 8;    // tmem base, abort flag, range at +16
    static constexpr int STAT = MISC + 32;              // (m, l) of [set][row]
    static constexpr int PIDS = STAT + 2 * 2 * ROWS * 4;  // [2 producers][LOOKAHEAD+1][8] int
    static constexpr int CTX = PIDS + 2 * (LOOKAHEAD + 1) * NVB * 4;
    static constexpr int PRE = CTX + MAX_BATCH * 4;
    // INT8: fp16 scales of tile it at stage it % 2, k then v
    static constexpr int SCRAW = (PRE + (MAX_BATCH + 1) * 4 + 127) / 128 * 128;
    static constexpr int END = SCRAW + 2 * 2 * TN * 2;
};
constexpr size_t SMEM_BYTES = Smem::END + 1024;  // + alignment slack
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");

struct Tc2Params {
    AttnArgs a;
    float* part_o;    // [2*C][ROWS][D]
    float* part_lse;  // [2*C][ROWS]
    int4* seg_rec;    // [C][2]
    int* seg_pre;     // [B+1]
};

// 64 consecutive fp32 TMEM columns of this thread's lane.
__device__ __forceinline__ void load64(uint32_t taddr, uint32_t (&v)[64]) {
    uint32_t (&lo)[32] = *reinterpret_cast<uint32_t(*)[32]>(&v[0]);
    uint32_t (&hi)[32] = *reinterpret_cast<uint32_t(*)[32]>(&v[32]);
    tmem_ld32(taddr, lo);
    tmem_ld32(taddr + 32, hi);
    tmem_wait_ld();
}

// Scores of 64 columns (raw fp32 bits from TMEM, rewritten in place) in log2
// units with the invisible ones at -inf; returns their maximum.  vis: bit c
// set when column c is visible.
__device__ __forceinline__ float scale_mask64(uint32_t (&r)[64], float sl2, uint64_t vis) {
#pragma unroll
    for (int c = 0; c < 64; c += 2) {
        float v0, v1;
        f2_split(f2_mul(f2(__uint_as_float(r[c]), __uint_as_float(r[c + 1])), f2(sl2, sl2)),
                 v0, v1);
        r[c] = __float_as_uint(v0);
        r[c + 1] = __float_as_uint(v1);
    }
    if (vis != ~0ull) {
#pragma unroll
        for (int c = 0; c < 64; ++c)
            r[c] = ((vis >> c) & 1ull) ? r[c] : __float_as_uint(-INFINITY);
    }
    float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
    for (int c2 = 0; c2 < 32; ++c2)
        mx[c2 & 3] =
            fmax3(mx[c2 & 3], __uint_as_float(r[2 * c2]), __uint_as_float(r[2 * c2 + 1]));
    return fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
}

// p = 2^(v - m) of 64 columns (fp32 bits), packed to bf16 (F16: fp16) pairs;
// returns their sum.
template <bool F16>
__device__ __forceinline__ float exp_pack64(const uint32_t (&v)[64], float m, uint32_t (&pk)[32]) {
    const uint64_t neg_m = f2(-m, -m);
    uint64_t ps[2] = {f2(0.f, 0.f), f2(0.f, 0.f)};
#pragma unroll
    for (int c = 0; c < 64; c += 2) {
        float e0, e1;
        f2_split(f2_add(f2(__uint_as_float(v[c]), __uint_as_float(v[c + 1])), neg_m), e0, e1);
        e0 = fast_exp2(e0);
        e1 = fast_exp2(e1);
        ps[(c >> 1) & 1] = f2_add(ps[(c >> 1) & 1], f2(e0, e1));
        pk[c >> 1] = F16 ? pack_f16x2(e0, e1) : pack_bf16x2(e0, e1);
    }
    float a0, a1, b0, b1;
    f2_split(ps[0], a0, a1);
    f2_split(ps[1], b0, b1);
    return (a0 + b0) + (a1 + b1);
}

// Visible columns [c0, c0 + 64) of a 128-key tile for a query row: the
// context keys, then the drafts of the row's bits, limited to the tile's keys.
__device__ __forceinline__ uint64_t visible64(int key0, int c0, int nvalid, int ctx,
                                              uint64_t mrow) {
    const int kc0 = key0 + c0, nv = nvalid - c0, nctx = ctx - kc0;
    const uint64_t valid = nv >= 64 ? ~0ull : nv <= 0 ? 0ull : (1ull << nv) - 1;
    const uint64_t cbits = nctx >= 64 ? ~0ull : nctx <= 0 ? 0ull : (1ull << nctx) - 1;
    const uint64_t dbits = nctx >= 64    ? 0ull
                           : nctx >= 0   ? mrow << nctx
                           : nctx > -64  ? mrow >> -nctx
                                         : 0ull;
    return (cbits | dbits) & valid;
}

template <bool KV8>
__global__ void __launch_bounds__(threads<KV8>(), 1)
attn_tc2_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
                const __grid_constant__ CUtensorMap vmap, const Tc2Params prm) {
    constexpr int NT = threads<KV8>();
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const AttnArgs& a = prm.a;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + Smem::BARS);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + Smem::MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + Smem::MISC + 4);
    int64_t* s_rng = reinterpret_cast<int64_t*>(sm + Smem::MISC + 16);
    int* s_ctx = reinterpret_cast<int*>(sm + Smem::CTX);
    int* s_pre = reinterpret_cast<int*>(sm + Smem::PRE);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int B = a.B, k = a.k, Hkv = a.Hkv, G = a.Hq / a.Hkv, R = k * G, P = a.P;
    const int CH = P < TN ? P : TN, NCH = TN / CH;  // keys per page chunk, chunks per tile

    if (tid == 0) {
        for (int s = 0; s < 2; ++s) {
            mbar_init(&bars[Smem::B_KFULL + s], 1);
            mbar_init(&bars[Smem::B_KEMPTY + s], 1);
            mbar_init(&bars[Smem::B_VFULL + s], 1);
            mbar_init(&bars[Smem::B_VEMPTY + s], 1);
            mbar_init(&bars[Smem::B_QFULL + s], 1);
            mbar_init(&bars[Smem::B_QFREE + s], 1);
            mbar_init(&bars[Smem::B_SFULL + s], 1);
            mbar_init(&bars[Smem::B_PREADY + s], 4);  // the 4 warps of the set
            mbar_init(&bars[Smem::B_SFREE + s], 1);
            mbar_init(&bars[Smem::B_KREADY + s], 2);  // INT8: the 2 warps converting K / V
            mbar_init(&bars[Smem::B_VREADY + s], 2);
        }
        mbar_init(&bars[Smem::B_EPI], 8);  // every softmax warp, once per piece
        mbar_init(&bars[Smem::B_DRAIN], 1);
        mbar_init(&bars[Smem::B_DRAIN + 1], 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    // the grids before this one have finished with every buffer this call
    // touches (and with the tensor memory of this SM)
    grid_dep_launch_dependents();
    grid_dep_wait();
    if (warp == 4) {
        tmem_alloc(tmem_slot, TMEM_COLS);
        tmem_relinquish();
    }
    {
        // Q rows R..127 stay zero in both buffers (the TMA writes rows < R)
        uint4* q4 = reinterpret_cast<uint4*>(sm + Smem::Q);
        for (int e = tid; e < 2 * Q_BYTES / 16; e += NT) {
            const int row = (e % (Q_HALF / 16)) / 8;
            if (row >= R) q4[e] = make_uint4(0, 0, 0, 0);
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
        __syncwarp();  // the prefix above, written by this warp's lanes
        if (lane < 2) {
            TileSplit split;
            split.init(s_pre, B, Hkv, a.split_alpha >= 0 ? a.split_alpha : kSplitAlpha, gridDim.x);
            s_rng[lane] = split.begin(blockIdx.x + lane);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const int64_t T = (int64_t)s_pre[B] * Hkv;
    const int64_t t_begin = ld_shared_s64(s_rng);
    const int n_tiles = (int)(ld_shared_s64(s_rng + 1) - t_begin);
    if (tid == 0) {
        // the segment holding tile t_begin and t_begin itself, for the combine
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
        for (int b = tid; b <= B; b += NT) prm.seg_pre[b] = s_pre[b];

    // does a piece follow the one of cursor c in this CTA's range
    auto has_next_piece = [&](const Cursor& c) {
        return c.seg_start + c.nb < ld_shared_s64(s_rng + 1);
    };
    // INT8 (16 warps on 64K registers): the softmax warpgroups take 160 each,
    // the issue / copy warpgroup gives its registers down to 80 and the
    // dequantizing one to 112 (2 x 160 + 80 + 112 = 4 x 128, the launch
    // allocation), each warpgroup as the first step of its branch
    if (warp >= 4 && warp < 8) {
    if constexpr (KV8) regs_dec<80>();
    if (warp == 5 || warp == 6) {
        // ================= TMA producers: warp 5 K, warp 6 V, every tile =================
        // Tile it goes to slot it % 2 of each ring: its K slot is free once
        // Q K^T of tile it - 2 read it, its V slot once P V of tile it - 2
        // did, so a K copy never waits on a P V.  A tile is NCH chunks of CH
        // = min(P, 128) keys, each inside one page (CH * 256 contiguous bytes
        // of the cache), and each chunk is one copy: K as 8-key groups, each
        // [half][8 rows][128 B] (2 KB), the layout an N = 128 Q K^T reads; V
        // as 16-key groups, each [half][16 rows][128 B] (4 KB), the layout a
        // P V of 16 keys reads.  Block-table entries (one per chunk) are
        // prefetched LOOKAHEAD tiles ahead with cp.async.
        // INT8: each chunk is CH * 128 raw bytes into the upper half of the
        // slot, and its CH fp16 scales into scale stage it % 2.
        const bool is_v = warp == 6;
        int* pids = reinterpret_cast<int*>(sm + Smem::PIDS) + (is_v ? 1 : 0) * (LOOKAHEAD + 1) * NVB;
        uint64_t* full = &bars[is_v ? Smem::B_VFULL : Smem::B_KFULL];
        uint64_t* empty = &bars[is_v ? Smem::B_VEMPTY : Smem::B_KEMPTY];
        uint8_t* ring = sm + (is_v ? Smem::VS : Smem::KS);
        const CUtensorMap* map = is_v ? &vmap : &kmap;
        const int gshift = is_v ? 4 : 3;  // log2 of the rows of a group
        Cursor cur, ahead;
        if (n_tiles > 0) {
            cur.init(t_begin, s_pre, s_ctx, B, Hkv, k);
            ahead = cur;
        }
        const uint64_t pol = l2_policy_evict_first();
        if (lane == 0) prefetch_tmap(map);
        auto fetch_pids = [&](int slot, const Cursor& c) {
            const int key0 = c.lt * TN;
            const int nvalid = min(TN, s_ctx[c.b] + k - key0);
            if (lane < NCH && lane * CH < nvalid)
                cp_async_4(&pids[slot * NVB + lane],
                           &a.block_table[(int64_t)c.b * a.max_pages + (key0 + lane * CH) / P]);
        };
        for (int la = 0; la < LOOKAHEAD; ++la) {
            if (la < n_tiles) {
                fetch_pids(la % (LOOKAHEAD + 1), ahead);
                if (la + 1 < n_tiles) ahead.next(s_ctx, Hkv, k);
            }
            cp_async_commit();
        }
        int n_issued = 0;
        bool ok = true;
        for (int it = 0; it < n_tiles && ok; ++it) {
            if (it + LOOKAHEAD < n_tiles) {
                fetch_pids((it + LOOKAHEAD) % (LOOKAHEAD + 1), ahead);
                if (it + LOOKAHEAD + 1 < n_tiles) ahead.next(s_ctx, Hkv, k);
            }
            cp_async_commit();
            cp_async_wait<LOOKAHEAD>();  // entries of tile `it`
            __syncwarp();
            const int* pid = pids + (it % (LOOKAHEAD + 1)) * NVB;
            const int key0 = cur.lt * TN;
            const int nvalid = min(TN, s_ctx[cur.b] + k - key0);
            const int nck = (nvalid + CH - 1) / CH;  // chunks holding keys of the tile
            const int s = it & 1;
            if (it >= 2) ok = warp_wait(&empty[s], ((it >> 1) - 1) & 1, abort_flag, a.dev_err);
            const uint32_t bytes = (uint32_t)(nck * CH) * (KV8 ? 128u + 2u : 256u);
            if (ok && lane == 0) mbar_arrive_expect_tx(&full[s], bytes);
            __syncwarp();
            if (!ok) break;
            if (lane < nck) {
                int page = pid[lane];
                if (page < 0 || page >= a.num_pages) {
                    raise_device_error(a.dev_err, SPEC_DEVERR_PAGE);
                    page = 0;
                }
                const int row = (page * Hkv + cur.kvh) * P + (key0 + lane * CH) % P;
                if constexpr (KV8) {
                    tma_load_2d(ring + s * SLOT_BYTES + RAW_OFF + lane * CH * 128, map, &full[s], 0,
                                row, pol);
                    bulk_load(sm + Smem::SCRAW + (s * 2 + (is_v ? 1 : 0)) * TN * 2 + lane * CH * 2,
                              (is_v ? a.v_scale : a.k_scale) + row, CH * 2, &full[s]);
                } else {
                    tma_load_4d_hint(ring + s * SLOT_BYTES + lane * CH * 256, map, &full[s], 0, 0,
                                     0, row >> gshift, pol);
                }
            }
            n_issued = it + 1;
            __syncwarp();
            if (it + 1 < n_tiles) cur.next(s_ctx, Hkv, k);
        }
        cp_async_wait<0>();
        if (!ok && lane == 0) {
            // the latest copy into each slot lands before the CTA exits
            for (int sl = 0; sl < 2; ++sl) {
                const int last = (n_issued - 1) - (((n_issued - 1) - sl) & 1);
                if (last >= 0) mbar_drain(&full[sl], (last >> 1) & 1);
            }
        }
    } else if (warp == 4) {
        // ================= Q loads and Q K^T issue =================
        if (n_tiles > 0) {
            Cursor cur;
            cur.init(t_begin, s_pre, s_ctx, B, Hkv, k);
            int pc = -1;                  // piece of the current tile
            int q_issued = 0;             // pieces whose Q load went out
            bool ok = true;
            auto issue_q = [&](int j, int b, int kvh) {  // lane 0: piece j into buffer j & 1
                uint64_t* bar = &bars[Smem::B_QFULL + (j & 1)];
                mbar_arrive_expect_tx(bar, 2 * R * 128);
                for (int h = 0; h < 2; ++h)
                    tma_load_3d(sm + Smem::Q + (j & 1) * Q_BYTES + h * Q_HALF, &qmap, bar, h * 64,
                                kvh * G, b * k);
            };
            if (lane == 0) {
                prefetch_tmap(&qmap);
                issue_q(0, cur.b, cur.kvh);
                if (has_next_piece(cur))
                    issue_q(1, cur.kvh + 1 < Hkv ? cur.b : cur.b + 1,
                            cur.kvh + 1 < Hkv ? cur.kvh + 1 : 0);
            }
            q_issued = has_next_piece(cur) ? 2 : 1;
            const uint64_t qdesc0 = umma_sdesc_sw128(smem_u32(sm + Smem::Q), 16, 1024);
            const uint64_t kdesc0 = umma_sdesc_sw128(smem_u32(sm + Smem::KS), 16, 2048);
            for (int it = 0; it < n_tiles && ok; ++it) {
                const bool first = (it == 0) || (cur.lt == 0);
                const bool last = (it == n_tiles - 1) || (cur.lt == cur.nb - 1);
                const int s = it & 1;
                if (first) {
                    ++pc;
                    // the piece after the next reuses the buffer of piece
                    // pc - 1, whose last Q K^T was committed to QFREE
                    if (pc >= 1 && q_issued == pc + 1 && has_next_piece(cur)) {
                        ok = warp_wait(&bars[Smem::B_QFREE + ((pc - 1) & 1)], ((pc - 1) >> 1) & 1,
                                       abort_flag, a.dev_err);
                        if (ok && lane == 0)
                            issue_q(pc + 1, cur.kvh + 1 < Hkv ? cur.b : cur.b + 1,
                                    cur.kvh + 1 < Hkv ? cur.kvh + 1 : 0);
                        __syncwarp();
                        q_issued = pc + 2;
                        if (!ok) break;
                    }
                    ok = warp_wait(&bars[Smem::B_QFULL + (pc & 1)], (pc >> 1) & 1, abort_flag,
                                   a.dev_err);
                    if (!ok) break;
                    if constexpr (KV8) {
                        // the piece's q to fp16, in place (rows < R; the rest are zero)
                        uint4* q4 = reinterpret_cast<uint4*>(sm + Smem::Q + (pc & 1) * Q_BYTES);
                        for (int e = lane; e < Q_BYTES / 16; e += 32)
                            if ((e % (Q_HALF / 16)) / 8 < R) q4[e] = bf16x8_to_f16(q4[e]);
                        fence_proxy_async_smem();
                        __syncwarp();
                    }
                }
                // K of tile it landed (INT8: widened); S buffer s free (P V of
                // tile it - 2 done)
                ok = warp_wait(&bars[(KV8 ? Smem::B_KREADY : Smem::B_KFULL) + s], (it >> 1) & 1,
                               abort_flag, a.dev_err);
                if (ok && it >= 2)
                    ok = warp_wait(&bars[Smem::B_SFREE + s], ((it >> 1) - 1) & 1, abort_flag,
                                   a.dev_err);
                if (!ok) break;
                __syncwarp();
                tc_fence_after();
                {
                    // S = Q K^T: k-slice kk at half kk/4 (Q: 16 KB on, K: 1 KB on
                    // in every 8-key group), 32-byte step kk%4
                    const uint64_t qd = qdesc0 + ((uint32_t)((pc & 1) * Q_BYTES) >> 4);
                    const uint64_t kd = kdesc0 + ((uint32_t)(s * SLOT_BYTES) >> 4);
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        umma_ss_w(tmem + TM_S + s * TN,
                                  qd + (kk >> 2) * (Q_HALF >> 4) + (kk & 3) * 2,
                                  kd + (kk >> 2) * (1024 >> 4) + (kk & 3) * 2, idesc_qk<KV8>(),
                                  kk ? 1u : 0u);
                    umma_commit_w(&bars[Smem::B_SFULL + s]);
                    umma_commit_w(&bars[Smem::B_KEMPTY + s]);
                    if (last) umma_commit_w(&bars[Smem::B_QFREE + (pc & 1)]);
                }
                if (it + 1 < n_tiles) cur.next(s_ctx, Hkv, k);
            }
            // Q loads in flight land before the CTA exits (loads of one buffer
            // complete in order)
            if (!ok && lane == 0)
                for (int j = max(0, q_issued - 2); j < q_issued; ++j)
                    mbar_drain(&bars[Smem::B_QFULL + (j & 1)], (j >> 1) & 1);
            // every tensor-core op of this warp finishes before TMEM is released
            __syncwarp();
            umma_commit_w(&bars[Smem::B_DRAIN]);
            if (lane == 0) mbar_drain(&bars[Smem::B_DRAIN], 0);
            __syncwarp();
        }
    } else if (warp == 7) {
        // ================= P V issue =================
        if (n_tiles > 0) {
            Cursor cur;
            cur.init(t_begin, s_pre, s_ctx, B, Hkv, k);
            int pc = -1;
            bool ok = true;
            bool has0 = false, has1 = false;  // set 0 / 1 issued a P V in this piece
            // V of 16 keys: MN-major, head-dim halves 2 KB apart (LBO), 8-key
            // groups 1 KB (SBO)
            const uint64_t vdesc0 = umma_sdesc_sw128(smem_u32(sm + Smem::VS), 2048, 1024);
            for (int it = 0; it < n_tiles && ok; ++it) {
                const bool first = (it == 0) || (cur.lt == 0);
                const int s = it & 1;
                const int nvalid = min(TN, s_ctx[cur.b] + k - cur.lt * TN);
                if (first) {
                    ++pc;
                    has0 = has1 = false;
                    // the previous piece's epilogue has read both O before the
                    // first P V of this piece overwrites them
                    if (pc >= 1)
                        ok = warp_wait(&bars[Smem::B_EPI], (pc - 1) & 1, abort_flag, a.dev_err);
                    if (!ok) break;
                }
                // this set's P of tile it stored; V of tile it landed (INT8:
                // widened)
                ok = warp_wait(&bars[Smem::B_PREADY + s], (it >> 1) & 1, abort_flag, a.dev_err);
                if (ok)
                    ok = warp_wait(&bars[(KV8 ? Smem::B_VREADY : Smem::B_VFULL) + s],
                                   (it >> 1) & 1, abort_flag, a.dev_err);
                if (!ok) break;
                const int nvb = (nvalid + 15) / 16;
                // (INT8: the widened rows past the sequence end are finite)
                if (!KV8 && nvalid % 16 != 0) {
                    // keys past the sequence end that the last P V reads: zero
                    // their V rows so that 0 * (stale or canary) never reaches O
                    uint8_t* vst = sm + Smem::VS + s * SLOT_BYTES;
                    for (int e = lane; e < (nvb * 16 - nvalid) * 16; e += 32) {
                        const int t = nvalid + e / 16, h = (e / 8) & 1, c16 = e % 8;
                        *reinterpret_cast<uint4*>(vst + (t / 16) * 4096 + h * 2048 +
                                                  (t % 16) * 128 + c16 * 16) =
                            make_uint4(0, 0, 0, 0);
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                }
                tc_fence_after();
                {
                    // O_s += P V: MMA j takes keys [16j, 16j + 16) (4 KB group j),
                    // their P at the S columns [8j, 8j + 8) (j < 4) or
                    // [64 + 8(j-4), ...)
                    const uint64_t vd = vdesc0 + ((uint32_t)(s * SLOT_BYTES) >> 4);
                    const bool hs = s ? has1 : has0;
                    const uint32_t sbuf = tmem + TM_S + s * TN;
                    const uint32_t od = tmem + TM_O + s * D;
#pragma unroll
                    for (int j = 0; j < NVB; ++j)
                        if (j < nvb)
                            umma_ts_w(od, sbuf + (j < 4 ? 8 * j : 64 + 8 * (j - 4)),
                                      vd + ((uint32_t)(j * 4096) >> 4), idesc_pv<KV8>(),
                                      (hs || j > 0) ? 1u : 0u);
                    umma_commit_w(&bars[Smem::B_VEMPTY + s]);
                    umma_commit_w(&bars[Smem::B_SFREE + s]);
                }
                if (s) has1 = true;
                else has0 = true;
                if (it + 1 < n_tiles) cur.next(s_ctx, Hkv, k);
            }
            __syncwarp();
            umma_commit_w(&bars[Smem::B_DRAIN + 1]);
            if (lane == 0) mbar_drain(&bars[Smem::B_DRAIN + 1], 0);
            __syncwarp();
        }
    }
    } else if (KV8 && warp >= 12) {
        if constexpr (KV8) regs_dec<112>();
        // ================= INT8 dequantization (warps 12-13 K, 14-15 V) =================
        // Every tile in order: each int8 widened exactly to fp16 and
        // multiplied by its key's fp16 scale (one rounding to fp16), written
        // in place over the slot in the layout the MMAs read.  The raw tile
        // sits in the upper half: rows 0..63 are written to the lower half
        // straight away; rows 64..127 land over the raw bytes, so the pair of
        // warps first reads all of them and meets at a barrier.  Whole page
        // chunks are converted; keys past the sequence end become zero rows
        // (their stored scale may be anything, NaN included).  Every warp
        // runs every tile and every barrier, also after an abort (then
        // without waiting or work).
        const bool is_v = warp >= 14;
        const int ct = tid - (is_v ? 14 : 12) * 32;  // 0..63
        Cursor c;
        if (n_tiles > 0) c.init(t_begin, s_pre, s_ctx, B, Hkv, k);
        bool ok = true;
        for (int it = 0; it < n_tiles; ++it) {
            const int s = it & 1;
            const int nvalid = min(TN, s_ctx[c.b] + k - c.lt * TN);
            const int nch = (nvalid + CH - 1) / CH * CH * 8;  // raw 16-byte chunks loaded
            if (ok)
                ok = warp_wait(&bars[(is_v ? Smem::B_VFULL : Smem::B_KFULL) + s], (it >> 1) & 1,
                               abort_flag, a.dev_err);
            uint8_t* slot = sm + (is_v ? Smem::VS : Smem::KS) + s * SLOT_BYTES;
            const __half* scl =
                reinterpret_cast<const __half*>(sm + Smem::SCRAW + (s * 2 + (is_v ? 1 : 0)) * TN * 2);
            // chunk id (key id / 8, 16 head dims id % 8): widen, scale, store
            auto put = [&](int id, uint4 raw) {
                const int j = id >> 3, c16 = id & 7, h = c16 >> 2, sw = j & 7;
                const __half2 sc2 = __half2half2(j < nvalid ? scl[j] : __float2half(0.f));
                uint4 lo, hi;
                i8x16_to_f16(raw, lo, hi);
                __half2* l2 = reinterpret_cast<__half2*>(&lo);
                __half2* h2 = reinterpret_cast<__half2*>(&hi);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    l2[e] = __hmul2(l2[e], sc2);
                    h2[e] = __hmul2(h2[e], sc2);
                }
                // fp16 chunks cc, cc+1 of half h (swizzled by the row); lanes
                // of half 1 store their odd chunk first so that 8 consecutive
                // lanes hit 8 bank groups
                const int cc = (c16 & 3) * 2;
                const int o0 = ((cc + h) ^ sw) << 4, o1 = ((cc + 1 - h) ^ sw) << 4;
                uint8_t* row = is_v ? slot + (j >> 4) * 4096 + h * 2048 + (j & 15) * 128
                                    : slot + (j >> 3) * 2048 + h * 1024 + (j & 7) * 128;
                *reinterpret_cast<uint4*>(row + o0) = h ? hi : lo;
                *reinterpret_cast<uint4*>(row + o1) = h ? lo : hi;
            };
            // rows 0..63: raw in [16, 24) KB, output in [0, 16) KB
#pragma unroll 4
            for (int u = 0; u < 8; ++u) {
                const int id = ct + 64 * u;
                if (ok && id < nch) put(id, *reinterpret_cast<const uint4*>(slot + RAW_OFF + id * 16));
            }
            // rows 64..127: read all raw first, their output overlaps it
            uint4 raw[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int id = 512 + ct + 64 * u;
                if (ok && id < nch) raw[u] = *reinterpret_cast<const uint4*>(slot + RAW_OFF + id * 16);
            }
            named_bar_sync(is_v ? 7 : 6, 64);
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int id = 512 + ct + 64 * u;
                if (ok && id < nch) put(id, raw[u]);
            }
            fence_proxy_async_smem();  // generic-proxy writes -> tensor-core reads
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[(is_v ? Smem::B_VREADY : Smem::B_KREADY) + s]);
            if (it + 1 < n_tiles) c.next(s_ctx, Hkv, k);
        }
    } else {
        if constexpr (KV8) regs_inc<160>();
        // ================= softmax sets (0: warps 0-3, even tiles; 1: 8-11, odd) =================
        const int set = warp >= 8 ? 1 : 0;
        const int quad = warp & 3;                 // TMEM lane quadrant
        const int r = quad * 32 + lane;            // query row of this thread
        const bool row_valid = r < R;
        const bool quad_active = quad * 32 < R;
        const int i_row = row_valid ? r / G : k - 1;
        const float sl2 = a.scale * kLog2e;
        const uint32_t lane_base = tmem + ((uint32_t)(quad * 32) << 16);
        const uint32_t s_mine = lane_base + TM_S + set * TN;
        const uint32_t o_mine = TM_O + set * D, o_other = TM_O + (1 - set) * D;
        float* s_stat_m = reinterpret_cast<float*>(sm + Smem::STAT);
        float* s_stat_l = s_stat_m + 2 * ROWS;
        float m_ref = -INFINITY, l = 0.f;
        bool has = false;       // this set took a tile of the current piece
        int own = 0;            // tiles this set has taken (its S / P V phase count)
        uint64_t mrow = 0;
        Cursor cur;
        if (n_tiles > 0) cur.init(t_begin, s_pre, s_ctx, B, Hkv, k);
        bool ok = true;
        int pc = -1;
        for (int it = 0; it < n_tiles; ++it) {
            const bool first = (it == 0) || (cur.lt == 0);
            const bool last = (it == n_tiles - 1) || (cur.lt == cur.nb - 1);
            const bool mine = (it & 1) == set;
            const int ctx = s_ctx[cur.b], key0 = cur.lt * TN;
            const int nvalid = min(TN, ctx + k - key0);
            if (first) {
                ++pc;
                m_ref = -INFINITY;
                l = 0.f;
                has = false;
                mrow = draft_bits(a, cur.b, i_row);
            }
            if (mine) {
                if (ok)
                    ok = warp_wait(&bars[Smem::B_SFULL + set], own & 1, abort_flag, a.dev_err);
                if (ok && quad_active) {
                    tc_fence_after();
                    uint32_t v[64];
                    const uint64_t vis0 = visible64(key0, 0, nvalid, ctx, mrow);
                    // row maximum over both halves; the second half stays in v
                    load64(s_mine, v);
                    const float mx0 = scale_mask64(v, sl2, vis0);
                    load64(s_mine + 64, v);
                    const float mx1 = scale_mask64(v, sl2, visible64(key0, 64, nvalid, ctx, mrow));
                    const float m_new = fmaxf(m_ref, fmaxf(mx0, mx1));
                    float alpha = 1.f;
                    const bool move = m_new > m_ref + kRescaleThreshold;  // also -inf -> finite
                    if (move) {
                        alpha = (m_ref == -INFINITY) ? 0.f : fast_exp2(m_ref - m_new);
                        m_ref = m_new;
                        l *= alpha;
                    }
                    const float m_use = m_ref == -INFINITY ? 0.f : m_ref;  // keeps -inf - m finite
                    uint32_t pk[32];
                    // P of keys 64..127 over S columns [64, 96), then keys 0..63
                    // (reloaded) over [0, 32)
                    l += exp_pack64<KV8>(v, m_use, pk);
                    tmem_st32(s_mine + 64, pk);
                    load64(s_mine, v);
                    scale_mask64(v, sl2, vis0);
                    l += exp_pack64<KV8>(v, m_use, pk);
                    tmem_st32(s_mine, pk);
                    tmem_wait_st();
                    if (has && __any_sync(0xffffffffu, move)) {
                        // O holds every earlier P V of this set (the S buffer of
                        // this tile was free only after the previous one read it)
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
                // P of this tile stored (every warp of the set arrives, active or not)
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars[Smem::B_PREADY + set]);
                has = true;
                ++own;
            }
            if (last) {
                // ---- epilogue of the piece that ends at this tile: merge the two
                // sets' (max, sum, O); each set writes half of the output columns
                if (ok && has)  // this set's last P V (tile own - 1) is done
                    ok = warp_wait(&bars[Smem::B_SFREE + set], (own - 1) & 1, abort_flag,
                                   a.dev_err);
                tc_fence_after();
                const int64_t tb = ld_shared_s64(s_rng), te = ld_shared_s64(s_rng + 1);
                const bool complete = cur.seg_start >= tb && cur.seg_start + cur.nb <= te;
                const int slot = 2 * blockIdx.x + (cur.seg_start < tb ? 0 : 1);
                s_stat_m[set * ROWS + r] = has ? m_ref : -INFINITY;
                s_stat_l[set * ROWS + r] = has ? l : 0.f;
                tc_fence_before();
                named_bar_sync(2 + quad, 64);  // the two sets' warps of this quadrant
                tc_fence_after();
                const float mo = s_stat_m[(1 - set) * ROWS + r];
                const float lo = s_stat_l[(1 - set) * ROWS + r];
                const float mm = has ? m_ref : -INFINITY;
                const float mt = fmaxf(mm, mo);
                const float w_mine = mm == -INFINITY ? 0.f : fast_exp2(mm - mt);
                const float w_other = mo == -INFINITY ? 0.f : fast_exp2(mo - mt);
                const float lt = w_mine * (has ? l : 0.f) + w_other * lo;
                if (ok && quad_active) {
                    const float inv_l = lt > 0.f ? 1.f / lt : 0.f;
                    const float lse = lt > 0.f ? (mt + log2f(lt)) * kLn2 : -INFINITY;
                    const float wm = w_mine * inv_l, wo = w_other * inv_l;
                    const int64_t orow = ((int64_t)cur.b * k + r / G) * a.Hq + cur.kvh * G + r % G;
#pragma unroll
                    for (int c4 = set * 2; c4 < set * 2 + 2; ++c4) {
                        uint32_t ov[32], ow[32];
                        tmem_ld32(lane_base + o_mine + c4 * 32, ov);
                        tmem_ld32(lane_base + o_other + c4 * 32, ow);
                        tmem_wait_ld();
                        float o[32];
#pragma unroll
                        for (int e = 0; e < 32; ++e) {
                            // a set without a tile of this piece holds stale O: weight 0
                            const float a0 = wm > 0.f ? __uint_as_float(ov[e]) * wm : 0.f;
                            const float a1 = wo > 0.f ? __uint_as_float(ow[e]) * wo : 0.f;
                            o[e] = a0 + a1;
                        }
                        if (!row_valid) continue;
                        if (complete) {
                            uint4* dst = reinterpret_cast<uint4*>(
                                static_cast<__nv_bfloat16*>(a.out) + orow * D + c4 * 32);
#pragma unroll
                            for (int v4 = 0; v4 < 4; ++v4) {
                                uint4 w;
                                w.x = pack_bf16x2(o[8 * v4 + 0], o[8 * v4 + 1]);
                                w.y = pack_bf16x2(o[8 * v4 + 2], o[8 * v4 + 3]);
                                w.z = pack_bf16x2(o[8 * v4 + 4], o[8 * v4 + 5]);
                                w.w = pack_bf16x2(o[8 * v4 + 6], o[8 * v4 + 7]);
                                dst[v4] = w;
                            }
                        } else {
                            float4* dst = reinterpret_cast<float4*>(
                                prm.part_o + ((int64_t)slot * ROWS + r) * D + c4 * 32);
#pragma unroll
                            for (int v4 = 0; v4 < 8; ++v4)
                                dst[v4] = make_float4(o[4 * v4 + 0], o[4 * v4 + 1], o[4 * v4 + 2],
                                                      o[4 * v4 + 3]);
                        }
                    }
                    if (row_valid && set == 0) {
                        if (complete) {
                            if (a.lse) a.lse[orow] = lse;
                        } else {
                            prm.part_lse[(int64_t)slot * ROWS + r] = lse;
                        }
                    }
                }
                // both sets have read both O: the next piece's P V may overwrite them
                tc_fence_before();
                named_bar_sync(2 + quad, 64);
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars[Smem::B_EPI]);
            }
            if (it + 1 < n_tiles) cur.next(s_ctx, Hkv, k);
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 4) tmem_dealloc(tmem, TMEM_COLS);
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

bool tc2_supported(const AttnArgs& a) {
    const int G = a.Hq / a.Hkv, R = a.k * G;
    const bool pow2 = (a.P & (a.P - 1)) == 0;
    // INT8 cache: the scales are fetched a page chunk (>= 32 bytes) at a time
    // with bulk copies, which need 16-byte aligned sources
    const bool kv_ok =
        a.kv_dtype == SPEC_DTYPE_BF16 ||
        (a.kv_dtype == SPEC_DTYPE_I8 && a.k_scale && a.v_scale &&
         (reinterpret_cast<uintptr_t>(a.k_scale) & 15) == 0 &&
         (reinterpret_cast<uintptr_t>(a.v_scale) & 15) == 0);
    return a.q_dtype == SPEC_DTYPE_BF16 && kv_ok && a.D == D &&
           R <= ROWS && G <= 256 && pow2 && a.P >= 16 && a.P <= 256 &&
           a.B <= MAX_BATCH && (int64_t)a.num_pages * a.Hkv * a.P < (1LL << 31) &&
           (int64_t)a.B * a.k < (1LL << 31);
}

int tc2_split_alpha(const AttnArgs& a) { return a.split_alpha >= 0 ? a.split_alpha : kSplitAlpha; }

cudaError_t launch_attn_tc2(const AttnArgs& a, int num_ctas, void* workspace, cudaStream_t stream) {
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
    // K / V rows (num_pages*Hkv*P of 256 B) seen as [groups of g rows] x
    // [2 halves] x [g rows] x [64 columns], g = 8 (K) or 16 (V); a box is CH =
    // min(P, 128) consecutive rows of one page, landing group by group.
    // INT8: rows of 128 bytes, a box CH rows as they are (the widening warps
    // swizzle)
    const cuuint64_t rows = (cuuint64_t)a.num_pages * a.Hkv * a.P;
    const cuuint32_t ch = (cuuint32_t)(a.P < TN ? a.P : TN);
    const bool kv8 = a.kv_dtype == SPEC_DTYPE_I8;
    for (int t = 0; t < 2 && kv8; ++t) {
        cuuint64_t dims[2] = {(cuuint64_t)D, rows};
        cuuint64_t strides[1] = {(cuuint64_t)D};
        cuuint32_t box[2] = {(cuuint32_t)D, ch};
        cuuint32_t es[2] = {1, 1};
        if (encode(t == 0 ? &kmap : &vmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2,
                   const_cast<void*>(t == 0 ? a.k_cache : a.v_cache), dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    for (int t = 0; t < 2 && !kv8; ++t) {
        const cuuint32_t g = t == 0 ? 8 : 16;
        cuuint64_t dims[4] = {64, g, 2, rows / g};
        cuuint64_t strides[3] = {(cuuint64_t)D * 2, 128, (cuuint64_t)g * D * 2};
        cuuint32_t box[4] = {64, g, 2, ch / g};
        cuuint32_t es[4] = {1, 1, 1, 1};
        if (encode(t == 0 ? &kmap : &vmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
                   const_cast<void*>(t == 0 ? a.k_cache : a.v_cache), dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    Tc2Params prm;
    prm.a = a;
    prm.part_o = static_cast<float*>(workspace);
    prm.part_lse = prm.part_o + (size_t)2 * num_ctas * ROWS * D;
    prm.seg_rec = reinterpret_cast<int4*>(prm.part_lse + (size_t)2 * num_ctas * ROWS);
    prm.seg_pre = reinterpret_cast<int*>(prm.seg_rec + 2 * (size_t)num_ctas);
    cudaError_t e;
    if (kv8) {
        e = cudaFuncSetAttribute(attn_tc2_kernel<true>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
        if (e != cudaSuccess) return e;
        e = launch_dependent(attn_tc2_kernel<true>, dim3(num_ctas), dim3(threads<true>()),
                             SMEM_BYTES, stream, qmap, kmap, vmap, prm);
    } else {
        e = cudaFuncSetAttribute(attn_tc2_kernel<false>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
        if (e != cudaSuccess) return e;
        e = launch_dependent(attn_tc2_kernel<false>, dim3(num_ctas), dim3(threads<false>()),
                             SMEM_BYTES, stream, qmap, kmap, vmap, prm);
    }
    if (e != cudaSuccess) return e;
    return launch_combine_stream_k(a, num_ctas, tc2_split_alpha(a), prm.part_o, prm.part_lse,
                                   prm.seg_rec, prm.seg_pre, stream);
}

}  // namespace specv

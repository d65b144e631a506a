// Device helpers shared by the verification kernels: element conversion,
// reductions, mbarrier / TMA / tcgen05 wrappers (inline PTX for sm_103a) and
// the bounded waits every on-chip spin uses.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kernels.h"

namespace specv {

// ------------------------------------------------------------------ elements

template <typename T> struct Elem;
template <> struct Elem<float> {
    static __device__ __forceinline__ float to_f32(float x) { return x; }
    static __device__ __forceinline__ float from_f32(float x) { return x; }
};
template <> struct Elem<__nv_bfloat16> {
    static __device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
    static __device__ __forceinline__ __nv_bfloat16 from_f32(float x) { return __float2bfloat16_rn(x); }
};
template <> struct Elem<int8_t> {
    static __device__ __forceinline__ float to_f32(int8_t x) { return (float)x; }
};

// Device error word (one per device, in the library workspace).
__device__ __forceinline__ void raise_device_error(int* err, int flag) {
    if (err) atomicOr(err, flag);
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Wall-clock bound of every on-chip wait; well above any legitimate wait.
constexpr uint64_t kWaitLimitNs = 1000ull * 1000ull * 1000ull;  // 1 s

// ------------------------------------------------------------------ smem / mbarrier

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(
                     smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ------------------------------------------------------------------ TMA

__device__ __forceinline__ void tma_load_2d(void* smem_dst, const void* tmap, uint64_t* bar,
                                            int32_t c0, int32_t c1, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_u32(smem_dst)),
        "l"(tmap), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void tma_load_3d(void* smem_dst, const void* tmap, uint64_t* bar,
                                            int32_t c0, int32_t c1, int32_t c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(smem_dst)),
        "l"(tmap), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}

__device__ __forceinline__ void tma_load_3d_hint(void* smem_dst, const void* tmap, uint64_t* bar,
                                                 int32_t c0, int32_t c1, int32_t c2,
                                                 uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%3, %4, %5}], [%2], %6;" ::"r"(smem_u32(smem_dst)),
        "l"(tmap), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void tma_load_4d_hint(void* smem_dst, const void* tmap, uint64_t* bar,
                                                 int32_t c0, int32_t c1, int32_t c2, int32_t c3,
                                                 uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%3, %4, %5, %6}], [%2], %7;" ::"r"(smem_u32(smem_dst)),
        "l"(tmap), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "l"(policy)
        : "memory");
}

// Plain bulk copy global -> shared (16-byte aligned address and size).
__device__ __forceinline__ void bulk_load(void* smem_dst, const void* gsrc, uint32_t bytes,
                                          uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(smem_u32(smem_dst)),
        "l"(gsrc), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ void prefetch_tmap(const void* tmap) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(tmap) : "memory");
}

// ------------------------------------------------------------------ tcgen05

__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// The tcgen05 issue instructions, run by a whole converged warp with
// warp-uniform operands; elect.sync picks the one lane (the lowest) that
// issues.  Issued that way the operands stay in the uniform datapath; from a
// one-lane branch with operands computed at run time each instruction costs
// several times more issue cycles.  ts: A from TMEM; ss: A from shared
// memory; commit: arrive on `bar` once every tcgen05 op this thread issued
// is done (it must come from the warp that issued them); cp: a 128-row x
// 256-bit matrix (a shared-memory descriptor) into TMEM lanes 0..127.
__device__ __forceinline__ void umma_ts_w(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred e, p;\n\telect.sync _|e, 0xffffffff;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void umma_ss_w(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred e, p;\n\telect.sync _|e, 0xffffffff;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void umma_commit_w(uint64_t* bar) {
    asm volatile(
        "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(
            smem_u32(bar))
        : "memory");
}
__device__ __forceinline__ void tmem_cp_128x256b_w(uint32_t taddr, uint64_t sdesc) {
    asm volatile(
        "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.cp.cta_group::1.128x256b [%0], %1;\n\t}" ::"r"(taddr), "l"(sdesc)
        : "memory");
}

// 32 lanes x 32 consecutive 32-bit columns (one row per thread of the warp).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
        "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
        "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t* r) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
        : "memory");
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t* r) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15])
        : "memory");
}

// 2^x on the MUFU unit (hardware approximation; -inf -> +0).
__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Barrier over `count` threads on hardware barrier `id` (1..15).
__device__ __forceinline__ void named_bar_sync(int id, int count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

__device__ __forceinline__ void tmem_wait_ld() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Instruction descriptor of tcgen05.mma kind::f16: bf16 A and B, fp32 D,
// M x N tile, A/B major-ness (0 = K-major, 1 = MN-major).
__host__ __device__ constexpr uint32_t umma_idesc_bf16(int M, int N, int a_mn_major,
                                                       int b_mn_major) {
    return (1u << 4)                          // D format: f32
           | (1u << 7)                        // A format: bf16
           | (1u << 10)                       // B format: bf16
           | ((uint32_t)a_mn_major << 15)     // A major
           | ((uint32_t)b_mn_major << 16)     // B major
           | ((uint32_t)(N >> 3) << 17)       // N / 8
           | ((uint32_t)(M >> 4) << 24);      // M / 16
}

// Same for fp16 A and B (format code 0).
__host__ __device__ constexpr uint32_t umma_idesc_f16(int M, int N, int a_mn_major,
                                                      int b_mn_major) {
    return (1u << 4)                          // D format: f32
           | ((uint32_t)a_mn_major << 15)     // A major
           | ((uint32_t)b_mn_major << 16)     // B major
           | ((uint32_t)(N >> 3) << 17)       // N / 8
           | ((uint32_t)(M >> 4) << 24);      // M / 16
}

// Shared-memory matrix descriptor (tcgen05 format), 128-byte swizzle.
//   start: smem byte address; lbo / sbo: leading / stride byte offsets.
__device__ __forceinline__ uint64_t umma_sdesc_sw128(uint32_t start, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= (uint64_t)((start >> 4) & 0x3FFF);
    d |= (uint64_t)((lbo >> 4) & 0x3FFF) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFF) << 32;
    d |= (uint64_t)1 << 46;   // descriptor version (sm_100 family)
    d |= (uint64_t)2 << 61;   // layout: 128-byte swizzle
    return d;
}

// Register budget of the calling warpgroup (all four warps execute it): the
// count moves between warpgroups inside the block's launch allocation.
template <uint32_t N> __device__ __forceinline__ void regs_dec() {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}
template <uint32_t N> __device__ __forceinline__ void regs_inc() {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}

// ------------------------------------------------------------------ persistent tile walk

// Split of the tile list over the C CTAs of a persistent grid.  Every piece
// of a segment a CTA processes costs fixed work besides its tiles (loading
// the piece's query rows, draining and merging its partial results), so an
// equal number of tiles per CTA leaves the CTAs whose ranges hold more
// segment starts finishing last.  The split therefore runs over a cost
// coordinate in which each segment (sequence b, kv-head h; sequences in
// order, kv-heads inside a sequence) is preceded by `alpha` units for that
// fixed work and then holds its nb(b) = pre[b+1] - pre[b] tiles; CTA c takes
// the tiles of costs [c W / C, (c+1) W / C).  alpha = 0 is the equal split.
// `pre` is the per-sequence tile prefix (per kv-head), in shared or global
// memory.
struct TileSplit {
    const int* pre;
    int B, Hkv, alpha;
    int64_t C, W;

    __device__ void init(const int* pre_, int B_, int Hkv_, int alpha_, int64_t C_) {
        pre = pre_;
        B = B_;
        Hkv = Hkv_;
        alpha = alpha_;
        C = C_;
        W = cost_pre(B);
    }
    // cost at the start of sequence b
    __device__ int64_t cost_pre(int b) const {
        return ((int64_t)pre[b] + (int64_t)alpha * b) * Hkv;
    }
    // the first tile at or after cost x (32-bit arithmetic when the list is
    // shorter than 2^31 cost units, as every realistic call is)
    __device__ int64_t tile_at(int64_t x) const {
        if (x >= W) return (int64_t)pre[B] * Hkv;
        if (alpha == 0) return x;  // the cost of a tile is its index
        int lo = 0, hi = B - 1;  // largest b with cost_pre(b) <= x
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (cost_pre(mid) <= x) lo = mid; else hi = mid - 1;
        }
        const int nb = pre[lo + 1] - pre[lo];
        const int64_t off = x - cost_pre(lo);
        int64_t h, r;
        if (W < (1LL << 31)) {
            const uint32_t o32 = (uint32_t)off, seg = (uint32_t)(nb + alpha);
            h = o32 / seg;
            r = o32 - (uint32_t)h * seg;
        } else {
            h = off / (nb + alpha);
            r = off % (nb + alpha);
        }
        return (int64_t)pre[lo] * Hkv + h * nb + (r > alpha ? r - alpha : 0);
    }
    // first tile of CTA c (c = C: the end of the list)
    __device__ int64_t begin(int64_t c) const {
        const int64_t x = W < (1LL << 31) && c < 65536
                              ? (int64_t)((uint64_t)c * (uint64_t)W / (uint64_t)C)
                              : c * W / C;
        return tile_at(x);
    }
    __device__ bool empty(int64_t c) const { return begin(c) == begin(c + 1); }
    // cost of tile lt of segment (b, kvh) with nb tiles
    __device__ int64_t cost_of(int b, int kvh, int lt, int nb) const {
        return cost_pre(b) + (int64_t)kvh * (nb + alpha) + alpha + lt;
    }
    // CTA whose range holds the tile of cost x
    __device__ int cta_of_cost(int64_t x) const { return (int)(((x + 1) * C - 1) / W); }
};

// A 64-bit value in shared memory, read afresh at every use: the persistent
// kernels keep their CTA range there so that it occupies no register through
// their main loops.
__device__ __forceinline__ int64_t ld_shared_s64(const int64_t* p) {
    int64_t v;
    asm volatile("ld.shared.s64 %0, [%1];" : "=l"(v) : "r"(smem_u32(p)) : "memory");
    return v;
}

// Verification work is the list of TILE_KEYS-key tiles of every (sequence,
// kv-head) segment, sequences in order, kv-heads inside a sequence.  pre[b]
// = tiles of sequences 0..b-1 (per kv-head), ctx[b] = clamped context.
// Walks a CTA's tile range: tile -> (sequence b, kv-head, tile-in-segment).
template <int TILE_KEYS>
struct CursorT {
    int b, kvh, lt, nb;
    int64_t seg_start;  // global index of the segment's first tile
    __device__ void init(int64_t t, const int* pre, const int* ctx, int B, int Hkv, int k) {
        int lo = 0, hi = B - 1;  // largest b with pre[b]*Hkv <= t
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if ((int64_t)pre[mid] * Hkv <= t) lo = mid; else hi = mid - 1;
        }
        b = lo;
        nb = (ctx[b] + k + TILE_KEYS - 1) / TILE_KEYS;
        const int64_t off = t - (int64_t)pre[b] * Hkv;
        kvh = (int)(off / nb);
        lt = (int)(off % nb);
        seg_start = (int64_t)pre[b] * Hkv + (int64_t)kvh * nb;
    }
    __device__ void next(const int* ctx, int Hkv, int k) {
        if (++lt == nb) {
            lt = 0;
            seg_start += nb;
            if (++kvh == Hkv) {
                kvh = 0;
                ++b;
                nb = (ctx[b] + k + TILE_KEYS - 1) / TILE_KEYS;
            }
        }
    }
};

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

// Packed fp32 pairs (sm_100+ f32x2 arithmetic, round-to-nearest-even per
// lane, as the scalar forms) and the three-input max.
__device__ __forceinline__ uint64_t f2(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void f2_split(uint64_t v, float& lo, float& hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// Widens 16 int8 (one 16-byte chunk) to 16 fp16 (two chunks), exactly: the
// byte u = c + 128 placed under the fp16 exponent of 1024 reads as 1024 + u,
// and subtracting 1152 leaves c (every step exact in fp16).
__device__ __forceinline__ void i8x16_to_f16(const uint4 r, uint4& lo, uint4& hi) {
    const uint32_t w[4] = {r.x ^ 0x80808080u, r.y ^ 0x80808080u, r.z ^ 0x80808080u,
                           r.w ^ 0x80808080u};
    uint32_t o[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t e01 = __byte_perm(w[i], 0x64646464u, 0x4140);
        const uint32_t e23 = __byte_perm(w[i], 0x64646464u, 0x4342);
        asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(o[2 * i]) : "r"(e01), "r"(0x64806480u));
        asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(o[2 * i + 1]) : "r"(e23), "r"(0x64806480u));
    }
    lo = make_uint4(o[0], o[1], o[2], o[3]);
    hi = make_uint4(o[4], o[5], o[6], o[7]);
}

// bf16 -> fp16 in place (8 values per 16-byte chunk), round to nearest even.
__device__ __forceinline__ uint4 bf16x8_to_f16(const uint4 r) {
    const uint32_t w[4] = {r.x, r.y, r.z, r.w};
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
        o[i] = pack_f16x2(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xffff0000u));
    return make_uint4(o[0], o[1], o[2], o[3]);
}

__device__ __forceinline__ void cp_async_4(void* smem_dst, const void* gsrc) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(smem_dst)), "l"(gsrc)
                 : "memory");
}
// ------------------------------------------------------------------ clusters
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_arrive_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_arrive_release() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_acquire() {
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// shared::cluster address of `p` (this CTA's shared memory) in CTA `rank`
__device__ __forceinline__ uint32_t cluster_map(const void* p, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
    return r;
}
__device__ __forceinline__ void st_cluster_f32(uint32_t addr, float v) {
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}
__device__ __forceinline__ void st_cluster_s32(uint32_t addr, int v) {
    asm volatile("st.shared::cluster.s32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ float ld_cluster_f32(uint32_t addr) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}

// 16-byte global -> shared copy that bypasses L1 (reads the L2 copy)
__device__ __forceinline__ void cp_async_16_cg(void* smem_dst, const void* gsrc) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(smem_dst)), "l"(gsrc)
                 : "memory");
}
// 32-bit load with acquire semantics at GPU scope
__device__ __forceinline__ int ld_acquire_gpu(const int* p) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N> __device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Warp-uniform bounded wait (the whole warp calls it): every lane polls in
// step and every decision is a warp vote, so the warp leaves converged.  A
// wait spun by one lane while the others park leaves the warp split, and the
// tcgen05.mma issued right after it (elect.sync) then issues several times
// slower for the rest of the batch.  Gives up when the CTA-wide abort flag
// is raised by another role, or after kWaitLimitNs, when it raises the abort
// flag and the device timeout error.  Returns true when the phase completed.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                          int* dev_err) {
    constexpr uint32_t kAll = 0xffffffffu;
    if (__all_sync(kAll, mbar_try_wait(bar, parity))) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        if (__all_sync(kAll, mbar_try_wait(bar, parity))) return true;
        if (__any_sync(kAll, *abort_flag != 0)) return false;
        if (__any_sync(kAll, globaltimer_ns() - t0 > kWaitLimitNs)) {
            if ((threadIdx.x & 31) == 0) {
                *abort_flag = 1;
                raise_device_error(dev_err, SPEC_DEVERR_TIMEOUT);
            }
            __syncwarp();
            return false;
        }
    }
}

// Bounded wait used only while draining after an abort (ignores the flag).
__device__ __forceinline__ void mbar_drain(uint64_t* bar, uint32_t parity) {
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity))
        if (globaltimer_ns() - t0 > kWaitLimitNs) return;
}


// ------------------------------------------------------------------ reductions

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}



// ------------------------------------------------------------------ dependent launch
//
// The step's kernels are launched with programmatic stream serialization: the
// next kernel on the stream may be scheduled while this one is still running,
// which hides the launch latency between the two calls of a step (and between
// steps).  Stream order is kept by the waits: every kernel waits for the
// grids before it to complete, and their writes to be visible, before its
// first global-memory access (read or write); until then it only sets up
// on-chip state.  A kernel launched without the attribute, or with nothing
// before it, passes the wait at once.
__device__ __forceinline__ void grid_dep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Launch `kernel` on `stream` with programmatic stream serialization.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                    cudaStream_t stream, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}
}  // namespace specv

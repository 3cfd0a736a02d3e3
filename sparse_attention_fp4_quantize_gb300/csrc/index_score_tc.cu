// Indexer scoring of many query tokens (prefill-shaped Full mode, FP8) on
// the 5th-generation tensor cores.
// Sources: "DeepSeek-V4.1-Flash：把 KV Cache 压缩到极限的百万上下文 MoE", section
// "Hierarchical Sparse Indexer——索引成本变常数" (Full layers score every entry);
// the score sum_h w_h * ReLU(q_h . k) is not on the pages.
//
// With thousands of query tokens per sequence the scores are a dense
// contraction: [T x 4 heads, 64] x [64, N keys].  Work item = (sequence b,
// 64-query tile, range of 128-key tiles), taken by a persistent CTA per SM in
// a static order.  The CTA is warp-specialised:
//  - warp 16 (producer) streams the operand tiles with TMA tensor copies into
//    shared memory, 64-byte swizzled (the layout tcgen05 reads directly): the
//    item's query tile (256 query-head rows x 64 B, FP8) into one of two Q
//    buffers, then its key tiles (128 keys x 64 B) through an 8-stage ring;
//    full / empty mbarriers per buffer;
//  - warp 17 (MMA) issues S^T [128 keys x 256 query-heads] = K . Q^T as two
//    tcgen05.mma kind::f8f6f4 (E4M3 x E4M3, K = 32 each) into one of two TMEM
//    accumulators and commits the key stage (empty) and the accumulator
//    (full) to mbarriers;
//  - warps 0..15 (epilogue) drain an accumulator while the next one fills:
//    TMEM lane = key, 4 consecutive columns = the 4 heads of one query, so
//    score = sum_h w_h * max(x_h, 0) stays inside a thread; keys at or beyond
//    the query's kv_len become -inf.  Each warp owns a TMEM lane quarter and
//    16 queries, read 8 queries (32 columns) at a time.
// Key tiles at or beyond every query's kv_len are neither loaded nor
// multiplied (-inf is written there).  The epilogue writes fp32 [B, T, N];
// each warp store covers 32 consecutive keys of one query (128 B).
//
// The first pass of the fused dense indexer (csa2_index_topk_dense, which
// never writes the score matrix) keeps only the order-preserving key of each
// 8-key block's maximum score; its kernel (index_blockmax_tc_kernel, below)
// uses the same pipeline with the MMA transposed, queries on the TMEM lanes.
// Every mbarrier wait is bounded; a thread that gives up raises a shared
// abort word that every other wait polls, so all roles leave their loops,
// the producer waits (bounded) for the copies it issued, and the CTA frees
// its TMEM and returns with CSA2_FLAG_TIMEOUT set.
#include <cuda.h>

#include "common.cuh"
#include "tc.cuh"

namespace csa2 {
namespace {

constexpr int QT = 64;                 // queries per tile
constexpr int QR = QT * 4;             // query-head rows (MMA N)
constexpr int KT = 128;                // keys per tile (MMA M)
constexpr int KTILES_PER_ITEM = 16;    // key tiles per work item
constexpr int STAGES = 8;              // key-tile ring
constexpr int EPI_WARPS = 16;          // 4 per TMEM lane quarter
constexpr int PRODUCER_WARP = EPI_WARPS, MMA_WARP = EPI_WARPS + 1;
constexpr int THREADS = (EPI_WARPS + 2) * 32;
constexpr uint32_t Q_BYTES = QR * 64;           // 16 KB
constexpr uint32_t K_BYTES = KT * 64;           // 8 KB per stage
constexpr uint32_t SW_SBO = 8 * 64;             // 64-byte swizzle: 8-row atoms of 512 bytes
// shared memory, from a 1024-byte aligned base
constexpr uint32_t OFF_K = 0;
constexpr uint32_t OFF_Q = OFF_K + STAGES * K_BYTES;     // 2 query tiles
constexpr uint32_t OFF_W = OFF_Q + 2 * Q_BYTES;          // float[QT][4]
constexpr uint32_t OFF_LT = OFF_W + QT * 16;             // int2[QT]: (kv_len clamped to N, 0)
constexpr uint32_t OFF_BAR = OFF_LT + QT * 8;            // mbarriers, see below
constexpr int NBARS = 2 * STAGES + 8;
constexpr uint32_t OFF_TMEM = OFF_BAR + NBARS * 8;
constexpr uint32_t OFF_ABORT = OFF_TMEM + 4;
constexpr uint32_t SMEM_USED = OFF_ABORT + 4;
// Ask for more than half of the SM's shared memory: one CTA per SM, so the
// CTA's 512 TMEM columns are never contended.  +1024 for the base alignment.
constexpr uint32_t SMEM = (SMEM_USED + 1024) > 120 * 1024 ? (SMEM_USED + 1024) : 120 * 1024;
constexpr uint32_t TMEM_COLS = 512;                   // 2 accumulators x 256 columns
constexpr uint32_t MAX_POLLS = 1u << 22;
static_assert(OFF_Q % 1024 == 0 && K_BYTES % 1024 == 0 && Q_BYTES % 1024 == 0, "swizzled tiles are 1024-aligned");

struct PrefillArgs {
    int B, T;
    int64_t N;
    const float *w;
    const int32_t *kv_len;
    float *scores;
    uint32_t *err_flag;
    int qtiles, ktiles, kranges;
    int64_t items;
    // block maxima (index_blockmax_tc_kernel): keys of the 8-key block maxima, [B*T, nblk]
    uint32_t *bmax;
    int64_t nblk;
};

// Twice sum_h w_h * max(x_h, 0), rounding step by step in the order
// w_0 m_0, + w_1 m_1, + w_2 m_2, + w_3 m_3.  x + |x| is exactly 2 max(x, 0)
// (one add with an absolute-value operand, off the integer/compare pipe), and
// scaling every operand of a rounding by 2 scales its result by 2 exactly
// (short of overflow or subnormal results), so half of this is that sum.
__device__ __forceinline__ float head_sum2(const float4 wq, const uint32_t *r) {
    auto relu2 = [](uint32_t v) { const float x = __uint_as_float(v); return __fadd_rn(x, fabsf(x)); };
    float s = __fmul_rn(wq.x, relu2(r[0]));
    s = __fmaf_rn(wq.y, relu2(r[1]), s);
    s = __fmaf_rn(wq.z, relu2(r[2]), s);
    return __fmaf_rn(wq.w, relu2(r[3]), s);
}

// Packed pairs of fp32 (sm_100 family): each lane of an f32x2 multiply or
// fused multiply-add rounds as its scalar instruction would, so two keys'
// head sums in one register pair equal two head_sum2 results bit for bit.
__device__ __forceinline__ float relu2f(uint32_t v) {   // 2 max(x, 0), as in head_sum2
    const float x = __uint_as_float(v);
    return __fadd_rn(x, fabsf(x));
}
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
    uint64_t d;
    asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(lo), "f"(hi));
    return d;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float &lo, float &hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ float max3f(float a, float b, float c) {   // the three-input form of fmaxf
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// K-major operand tile in the 64-byte swizzled canonical layout (rows of 64
// bytes, 8-row atoms of 512 bytes, as the TMA writes it with SWIZZLE_64B).
__device__ __forceinline__ uint64_t desc_sw64(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFF);
    d |= (uint64_t)1 << 16;                        // leading byte offset: unused for swizzled K-major
    d |= (uint64_t)((SW_SBO >> 4) & 0x3FFF) << 32;  // stride byte offset: one 8-row atom
    d |= (uint64_t)1 << 46;                        // descriptor version for sm_100-family
    d |= (uint64_t)4 << 61;                        // swizzle mode: 64-byte
    return d;
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int x, int y, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            dst),
        "l"((uint64_t)map), "r"(x), "r"(y), "r"(bar)
        : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
// Named barrier over the 16 epilogue warps only.
__device__ __forceinline__ void epi_sync() { asm volatile("bar.sync 1, %0;" ::"n"(EPI_WARPS * 32) : "memory"); }

// Bounded wait that also gives up once another thread has raised the abort word.
// sleep_ns > 0 backs off between polls, so that a waiting producer or MMA warp
// leaves the issue slots of its scheduler to the epilogue warps that share it.
__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity, volatile int *abort_word,
                                              uint32_t sleep_ns = 0) {
    for (uint32_t i = 0; i < MAX_POLLS; ++i) {
        uint32_t ok;
        asm volatile(
            "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(ok)
            : "r"(bar), "r"(parity)
            : "memory");
        if (ok) return true;
        if (sleep_ns) __nanosleep(sleep_ns);
        if ((i & 63) == 63 && *abort_word) return false;
    }
    *abort_word = 1;
    return false;
}

// Work item -> (sequence, query tile, key-tile range) and the longest visible
// prefix among the tile's queries (one warp; every lane gets the result).
struct Item {
    int64_t b;
    int t0, kt0, kt1, ntiles;   // ntiles: key tiles [kt0, kt0 + ntiles) hold a visible key
    int minlen;                 // shortest visible prefix (0 if the tile has fewer than 64 queries)
};
__device__ __forceinline__ Item item_of(const PrefillArgs &a, int64_t item, int lane) {
    Item it;
    const int kr = (int)(item % a.kranges);
    const int64_t rest = item / a.kranges;
    const int qt = (int)(rest % a.qtiles);
    it.b = rest / a.qtiles;
    it.t0 = qt * QT;
    it.kt0 = kr * KTILES_PER_ITEM;
    it.kt1 = min(a.ktiles, it.kt0 + KTILES_PER_ITEM);
    int m = 0, mn = 0x7FFFFFFF;
#pragma unroll
    for (int u = 0; u < QT / 32; ++u) {
        const int tq = it.t0 + lane + 32 * u;
        int l = 0;
        if (tq < a.T) {
            const int64_t len = (int64_t)a.kv_len[it.b * a.T + tq];
            l = (int)(len < 0 ? 0 : (len < a.N ? len : a.N));
        }
        m = max(m, l);
        mn = min(mn, l);
    }
    m = __reduce_max_sync(0xFFFFFFFFu, m);
    it.minlen = __reduce_min_sync(0xFFFFFFFFu, mn);
    const int vis = (m + KT - 1) / KT;   // key tiles with a visible key
    it.ntiles = max(0, min(it.kt1, vis) - it.kt0);
    return it;
}

__global__ void __launch_bounds__(THREADS, 1)
    index_score_prefill_tc_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
                                  PrefillArgs a) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const float4 *sW4 = reinterpret_cast<const float4 *>(smem + OFF_W);
    float *sW = reinterpret_cast<float *>(smem + OFF_W);
    int2 *sLT = reinterpret_cast<int2 *>(smem + OFF_LT);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + OFF_TMEM);
    volatile int *abort_word = reinterpret_cast<volatile int *>(smem + OFF_ABORT);
    const uint32_t sbase = tc::smem_u32(smem);
    const uint32_t bar0 = sbase + OFF_BAR;
    auto full = [&](int s) { return bar0 + 8u * s; };
    auto empty = [&](int s) { return bar0 + 8u * (STAGES + s); };
    auto tfull = [&](int j) { return bar0 + 8u * (2 * STAGES + j); };
    auto tempty = [&](int j) { return bar0 + 8u * (2 * STAGES + 2 + j); };
    auto qfull = [&](int j) { return bar0 + 8u * (2 * STAGES + 4 + j); };
    auto qempty = [&](int j) { return bar0 + 8u * (2 * STAGES + 6 + j); };
    const float NEG_INF = __int_as_float(0xff800000);

    if (tid == 0) {
        for (int s = 0; s < STAGES; ++s) {
            tc::mbar_init(full(s), 1);
            tc::mbar_init(empty(s), 1);
        }
        for (int j = 0; j < 2; ++j) {
            tc::mbar_init(tfull(j), 1);
            tc::mbar_init(tempty(j), EPI_WARPS);
            tc::mbar_init(qfull(j), 1);
            tc::mbar_init(qempty(j), 1);
        }
        *abort_word = 0;
        tc::mbar_init_fence();
    }
    if (warp == 0) tc::tmem_alloc(tmem_slot, TMEM_COLS);
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tmem = *tmem_slot;
    pdl_wait();
    pdl_launch_dependents();

    if (warp == PRODUCER_WARP) {
        // ---- TMA: the item's query tile, then its visible key tiles through the ring
        uint32_t kcount = 0, qcount = 0;
        bool run = true;
        for (int64_t item = blockIdx.x; run && item < a.items; item += gridDim.x) {
            const Item it = item_of(a, item, lane);
            const int qb = qcount & 1;
            if (!wait_or_abort(qempty(qb), ((qcount >> 1) & 1) ^ 1, abort_word, 256)) break;
            if (lane == 0) {
                mbar_expect_tx(qfull(qb), Q_BYTES);
                tma_load_2d(sbase + OFF_Q + qb * Q_BYTES, &qmap, 0, (int)((it.b * a.T + it.t0) * 4), qfull(qb));
            }
            ++qcount;
            for (int i = 0; i < it.ntiles; ++i) {
                const int s = kcount % STAGES;
                if (!wait_or_abort(empty(s), ((kcount / STAGES) & 1) ^ 1, abort_word, 256)) {
                    run = false;
                    break;
                }
                if (lane == 0) {
                    mbar_expect_tx(full(s), K_BYTES);
                    tma_load_2d(sbase + OFF_K + s * K_BYTES, &kmap, 0, (int)(it.b * a.N + (int64_t)(it.kt0 + i) * KT),
                                full(s));
                }
                ++kcount;
            }
        }
        if (*abort_word) {
            // copies still in flight land before the CTA leaves (bounded)
            for (uint32_t c = kcount > STAGES ? kcount - STAGES : 0; c < kcount; ++c)
                tc::mbar_wait(full(c % STAGES), (c / STAGES) & 1, MAX_POLLS);
            for (uint32_t c = qcount > 2 ? qcount - 2 : 0; c < qcount; ++c)
                tc::mbar_wait(qfull(c & 1), (c >> 1) & 1, MAX_POLLS);
        }
    } else if (warp == MMA_WARP) {
        // ---- tcgen05: two K = 32 MMAs per key tile into alternating accumulators
        constexpr uint32_t idesc = tc::idesc_e4m3_f32(KT, QR, false, false);
        uint32_t kcount = 0, qcount = 0, acount = 0;
        bool run = true;
        for (int64_t item = blockIdx.x; run && item < a.items; item += gridDim.x) {
            const Item it = item_of(a, item, lane);
            const int qb = qcount & 1;
            if (!wait_or_abort(qfull(qb), (qcount >> 1) & 1, abort_word, 64)) break;
            tc::fence_after();
            const uint32_t qaddr = sbase + OFF_Q + qb * Q_BYTES;
            for (int i = 0; i < it.ntiles; ++i) {
                const int s = kcount % STAGES, buf = acount & 1;
                if (!wait_or_abort(full(s), (kcount / STAGES) & 1, abort_word, 64) ||
                    !wait_or_abort(tempty(buf), ((acount >> 1) & 1) ^ 1, abort_word, 64)) {
                    run = false;
                    break;
                }
                tc::fence_after();
                if (lane == 0) {
                    const uint32_t kaddr = sbase + OFF_K + s * K_BYTES;
#pragma unroll
                    for (int ks = 0; ks < 2; ++ks)
                        tc::mma_f8(tmem + buf * 256, desc_sw64(kaddr + ks * 32), desc_sw64(qaddr + ks * 32), idesc,
                                   ks > 0);
                    tc::commit(empty(s));
                    tc::commit(tfull(buf));
                }
                __syncwarp();
                ++kcount;
                ++acount;
            }
            if (lane == 0) tc::commit(qempty(qb));   // the query tile is free once these MMAs are done
            __syncwarp();
            ++qcount;
        }
    } else {
        // ---- epilogue: warp w reads TMEM lane quarter w & 3 (32 keys, lane =
        // key) and the columns of queries 16 (w >> 2) .. +15, eight at a time
        const int lq = warp & 3, qg = warp >> 2;
        uint32_t acount = 0;
        bool run = true;
        for (int64_t item = blockIdx.x; run && item < a.items; item += gridDim.x) {
            const Item it = item_of(a, item, lane);
            epi_sync();   // the previous item's reads of sW / sLT are done
            if (tid < QT) {
                const int tq = it.t0 + tid;
                const bool v = tq < a.T;
                const int64_t row = it.b * a.T + (v ? tq : 0);
                for (int h = 0; h < 4; ++h) sW[tid * 4 + h] = v ? a.w[row * 4 + h] : 0.f;
                const int64_t len = v ? (int64_t)a.kv_len[row] : 0;
                sLT[tid] = make_int2((int)(len < 0 ? 0 : (len < a.N ? len : a.N)), 0);
            }
            epi_sync();
            const int64_t row0 = it.b * a.T + it.t0 + 16 * qg;
            for (int kt = it.kt0; kt < it.kt1; ++kt) {
                const bool did = kt - it.kt0 < it.ntiles;
                const int buf = acount & 1;
                if (did) {
                    if (!wait_or_abort(tfull(buf), (acount >> 1) & 1, abort_word)) {
                        run = false;
                        break;
                    }
                    tc::fence_after();
                }
                const int64_t key = (int64_t)kt * KT + 32 * lq + lane;
                // every key of the tile is below every query's kv_len (<= N): no mask
                const bool whole = did && (int64_t)(kt + 1) * KT <= it.minlen;
                const uint32_t ta = tmem + ((uint32_t)(32 * lq) << 16) + buf * 256 + 64 * qg;
#pragma unroll 1
                for (int h = 0; h < 2; ++h) {
                    uint32_t r[32];
                    if (did) {
                        tc::tmem_ld32(ta + 32 * h, r);
                        tc::tmem_ld_wait();
                        if (h == 1) {   // both halves are in registers: the accumulator is free
                            tc::fence_before();
                            __syncwarp();
                            if (lane == 0) mbar_arrive(tempty(buf));
                        }
                    }
                    const int q0 = 16 * qg + 8 * h;
                    float s[8];   // twice the scores (halved below: at the store, or once per block maximum)
#pragma unroll
                    for (int qq = 0; qq < 8; ++qq) {
                        float v = head_sum2(sW4[q0 + qq], r + 4 * qq);
                        if (!whole && !(did && key < sLT[q0 + qq].x)) v = NEG_INF;
                        s[qq] = v;
                    }
                    const int64_t rowh = row0 + 8 * h;
                    const int nq = a.T - (it.t0 + q0);   // queries of these eight that exist
                    if (key < a.N) {
#pragma unroll
                        for (int qq = 0; qq < 8; ++qq)
                            if (qq < nq) a.scores[(rowh + qq) * a.N + key] = 0.5f * s[qq];
                    }
                }
                if (did) ++acount;
            }
        }
    }
    if (*abort_word && tid == 0) flag_error(a.err_flag, CSA2_FLAG_TIMEOUT);
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    if (warp == 0) tc::tmem_dealloc(tmem, TMEM_COLS);
}

// ---------------------------------------------------------------------------
// BLOCKMAX with the queries on the TMEM lanes.  The same pipeline (a producer
// warp, an MMA warp and 16 epilogue warps over two accumulators) with the MMA
// transposed: per tile of 64 keys and per head h, D_h [128 queries x 64 keys]
// = Q_h . K^T (two kind::f8f6f4 MMAs, M128 N64 K32) into TMEM columns
// [256 buf + 64 h, +64).  An epilogue thread owns one query (its TMEM lane) and
// 16 keys of every tile: the head sum of a (query, key) pair reads the four
// heads' columns of its own lane and the maximum over a block of 8 keys stays
// in the thread, so neither needs a shuffle, and the query's weights and row
// length stay in registers for the whole work item.  The query tile arrives
// as one 3D tensor copy per head (the heads of a row are 64 bytes apart).
constexpr int BQ = 128;                          // queries per tile (MMA M: one TMEM lane each)
constexpr int BK = 64;                           // keys per tile (MMA N)
constexpr int BKTILES_PER_ITEM = 32;             // key tiles per work item (2048 keys)
constexpr uint32_t BQ_HEAD_BYTES = BQ * 64;      // 8 KB: one head of the query tile
constexpr uint32_t BQ_BYTES = 4 * BQ_HEAD_BYTES;
constexpr uint32_t BK_BYTES = BK * 64;           // 4 KB per stage
constexpr uint32_t BOFF_K = 0;
constexpr uint32_t BOFF_Q = BOFF_K + STAGES * BK_BYTES;   // 2 query tiles
constexpr uint32_t BOFF_BAR = BOFF_Q + 2 * BQ_BYTES;
constexpr uint32_t BOFF_TMEM = BOFF_BAR + NBARS * 8;
constexpr uint32_t BOFF_ABORT = BOFF_TMEM + 4;
constexpr uint32_t BSMEM_USED = BOFF_ABORT + 4;
constexpr uint32_t BSMEM = (BSMEM_USED + 1024) > 120 * 1024 ? (BSMEM_USED + 1024) : 120 * 1024;
static_assert(BOFF_Q % 1024 == 0 && BK_BYTES % 1024 == 0 && BQ_HEAD_BYTES % 1024 == 0, "swizzled tiles are 1024-aligned");
static_assert(4 * BK * 2 <= (int)TMEM_COLS, "two accumulators of four heads");

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *map, int x, int y, int z, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];" ::
            "r"(dst),
        "l"((uint64_t)map), "r"(x), "r"(y), "r"(z), "r"(bar)
        : "memory");
}

// Work item -> (sequence, 128-query tile, key-tile range) and the key tiles that
// hold a key visible to one of its queries (one warp; every lane gets the result).
struct BItem {
    int64_t b;
    int t0, kt0, ntiles;
};
__device__ __forceinline__ BItem bitem_of(const PrefillArgs &a, int64_t item, int lane) {
    BItem it;
    const int kr = (int)(item % a.kranges);
    const int64_t rest = item / a.kranges;
    const int qt = (int)(rest % a.qtiles);
    it.b = rest / a.qtiles;
    it.t0 = qt * BQ;
    it.kt0 = kr * BKTILES_PER_ITEM;
    const int kt1 = min(a.ktiles, it.kt0 + BKTILES_PER_ITEM);
    int m = 0;
#pragma unroll
    for (int u = 0; u < BQ / 32; ++u) {
        const int tq = it.t0 + lane + 32 * u;
        if (tq < a.T) {
            const int64_t len = (int64_t)a.kv_len[it.b * a.T + tq];
            m = max(m, (int)(len < 0 ? 0 : (len < a.N ? len : a.N)));
        }
    }
    m = __reduce_max_sync(0xFFFFFFFFu, m);
    it.ntiles = max(0, min(kt1, (m + BK - 1) / BK) - it.kt0);
    return it;
}

__global__ void __launch_bounds__(THREADS, 1)
    index_blockmax_tc_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
                             PrefillArgs a) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + BOFF_TMEM);
    volatile int *abort_word = reinterpret_cast<volatile int *>(smem + BOFF_ABORT);
    const uint32_t sbase = tc::smem_u32(smem);
    const uint32_t bar0 = sbase + BOFF_BAR;
    auto full = [&](int s) { return bar0 + 8u * s; };
    auto empty = [&](int s) { return bar0 + 8u * (STAGES + s); };
    auto tfull = [&](int j) { return bar0 + 8u * (2 * STAGES + j); };
    auto tempty = [&](int j) { return bar0 + 8u * (2 * STAGES + 2 + j); };
    auto qfull = [&](int j) { return bar0 + 8u * (2 * STAGES + 4 + j); };
    auto qempty = [&](int j) { return bar0 + 8u * (2 * STAGES + 6 + j); };
    const float NEG_INF = __int_as_float(0xff800000);

    if (tid == 0) {
        for (int s = 0; s < STAGES; ++s) {
            tc::mbar_init(full(s), 1);
            tc::mbar_init(empty(s), 1);
        }
        for (int j = 0; j < 2; ++j) {
            tc::mbar_init(tfull(j), 1);
            tc::mbar_init(tempty(j), EPI_WARPS);
            tc::mbar_init(qfull(j), 1);
            tc::mbar_init(qempty(j), 1);
        }
        *abort_word = 0;
        tc::mbar_init_fence();
    }
    if (warp == 0) tc::tmem_alloc(tmem_slot, TMEM_COLS);
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tmem = *tmem_slot;
    pdl_wait();
    pdl_launch_dependents();

    if (warp == PRODUCER_WARP) {
        // ---- TMA: the item's query tile (four heads), then its visible key tiles through the ring
        uint32_t kcount = 0, qcount = 0;
        bool run = true;
        for (int64_t item = blockIdx.x; run && item < a.items; item += gridDim.x) {
            const BItem it = bitem_of(a, item, lane);
            const int qb = qcount & 1;
            if (!wait_or_abort(qempty(qb), ((qcount >> 1) & 1) ^ 1, abort_word, 256)) break;
            if (lane == 0) {
                mbar_expect_tx(qfull(qb), BQ_BYTES);
#pragma unroll
                for (int h = 0; h < 4; ++h)
                    tma_load_3d(sbase + BOFF_Q + qb * BQ_BYTES + h * BQ_HEAD_BYTES, &qmap, 0, h,
                                (int)(it.b * a.T + it.t0), qfull(qb));
            }
            ++qcount;
            for (int i = 0; i < it.ntiles; ++i) {
                const int s = kcount % STAGES;
                if (!wait_or_abort(empty(s), ((kcount / STAGES) & 1) ^ 1, abort_word, 256)) {
                    run = false;
                    break;
                }
                if (lane == 0) {
                    mbar_expect_tx(full(s), BK_BYTES);
                    tma_load_2d(sbase + BOFF_K + s * BK_BYTES, &kmap, 0, (int)(it.b * a.N + (int64_t)(it.kt0 + i) * BK),
                                full(s));
                }
                ++kcount;
            }
        }
        if (*abort_word) {
            // copies still in flight land before the CTA leaves (bounded)
            for (uint32_t c = kcount > STAGES ? kcount - STAGES : 0; c < kcount; ++c)
                tc::mbar_wait(full(c % STAGES), (c / STAGES) & 1, MAX_POLLS);
            for (uint32_t c = qcount > 2 ? qcount - 2 : 0; c < qcount; ++c)
                tc::mbar_wait(qfull(c & 1), (c >> 1) & 1, MAX_POLLS);
        }
    } else if (warp == MMA_WARP) {
        // ---- tcgen05: per key tile and head, two K = 32 MMAs into the head's accumulator
        constexpr uint32_t idesc = tc::idesc_e4m3_f32(BQ, BK, false, false);
        uint32_t kcount = 0, qcount = 0, acount = 0;
        bool run = true;
        for (int64_t item = blockIdx.x; run && item < a.items; item += gridDim.x) {
            const BItem it = bitem_of(a, item, lane);
            const int qb = qcount & 1;
            if (!wait_or_abort(qfull(qb), (qcount >> 1) & 1, abort_word, 64)) break;
            tc::fence_after();
            const uint32_t qaddr = sbase + BOFF_Q + qb * BQ_BYTES;
            for (int i = 0; i < it.ntiles; ++i) {
                const int s = kcount % STAGES, buf = acount & 1;
                if (!wait_or_abort(full(s), (kcount / STAGES) & 1, abort_word, 64) ||
                    !wait_or_abort(tempty(buf), ((acount >> 1) & 1) ^ 1, abort_word, 64)) {
                    run = false;
                    break;
                }
                tc::fence_after();
                if (lane == 0) {
                    const uint32_t kaddr = sbase + BOFF_K + s * BK_BYTES;
#pragma unroll
                    for (int h = 0; h < 4; ++h)
#pragma unroll
                        for (int ks = 0; ks < 2; ++ks)
                            tc::mma_f8(tmem + buf * 256 + h * BK, desc_sw64(qaddr + h * BQ_HEAD_BYTES + ks * 32),
                                       desc_sw64(kaddr + ks * 32), idesc, ks > 0);
                    tc::commit(empty(s));
                    tc::commit(tfull(buf));
                }
                __syncwarp();
                ++kcount;
                ++acount;
            }
            if (lane == 0) tc::commit(qempty(qb));   // the query tile is free once these MMAs are done
            __syncwarp();
            ++qcount;
        }
    } else {
        // ---- epilogue: warp w reads TMEM lane quarter w & 3 (32 queries, lane = query) and
        // the 16 keys 16 (w >> 2) .. +15 of every tile, four heads of each
        const int lq = warp & 3, kg = warp >> 2;
        uint32_t acount = 0;
        bool run = true;
        for (int64_t item = blockIdx.x; run && item < a.items; item += gridDim.x) {
            const BItem it = bitem_of(a, item, lane);
            const int tq = it.t0 + 32 * lq + lane;   // this thread's query
            const bool qv = tq < a.T;
            const int64_t row = it.b * a.T + (qv ? tq : 0);
            float4 wq = make_float4(0.f, 0.f, 0.f, 0.f);
            int len = 0;   // N <= 2^18
            if (qv) {
                wq = make_float4(a.w[row * 4], a.w[row * 4 + 1], a.w[row * 4 + 2], a.w[row * 4 + 3]);
                const int64_t l = (int64_t)a.kv_len[row];
                len = (int)(l < 0 ? 0 : (l < a.N ? l : a.N));
            }
            const uint64_t w2[4] = {f2_pack(wq.x, wq.x), f2_pack(wq.y, wq.y), f2_pack(wq.z, wq.z), f2_pack(wq.w, wq.w)};
            uint32_t *brow = a.bmax + row * a.nblk;
            for (int i = 0; i < it.ntiles; ++i) {
                const int buf = acount & 1;
                if (!wait_or_abort(tfull(buf), (acount >> 1) & 1, abort_word)) {
                    run = false;
                    break;
                }
                tc::fence_after();
                uint32_t r[4][16];
                const uint32_t ta = tmem + ((uint32_t)(32 * lq) << 16) + buf * 256 + 16 * kg;
#pragma unroll
                for (int h = 0; h < 4; ++h) tc::tmem_ld16(ta + h * BK, r[h]);
                tc::tmem_ld_wait();
                tc::fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(tempty(buf));   // the accumulator is free
                const int key0 = (it.kt0 + i) * BK + 16 * kg;
                float m[2] = {NEG_INF, NEG_INF};
                if (key0 + 16 <= len) {   // all of this thread's keys are visible to its query
#pragma unroll
                    for (int j = 0; j < 16; j += 2) {   // keys j, j + 1 as one packed pair: head_sum2 of each
                        uint64_t s2 = f2_mul(f2_pack(relu2f(r[0][j]), relu2f(r[0][j + 1])), w2[0]);
                        s2 = f2_fma(f2_pack(relu2f(r[1][j]), relu2f(r[1][j + 1])), w2[1], s2);
                        s2 = f2_fma(f2_pack(relu2f(r[2][j]), relu2f(r[2][j + 1])), w2[2], s2);
                        s2 = f2_fma(f2_pack(relu2f(r[3][j]), relu2f(r[3][j + 1])), w2[3], s2);
                        float lo, hi;
                        f2_unpack(s2, lo, hi);
                        m[j >> 3] = max3f(m[j >> 3], lo, hi);   // twice the scores
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const uint32_t hv[4] = {r[0][j], r[1][j], r[2][j], r[3][j]};
                        const float v = key0 + j < len ? head_sum2(wq, hv) : NEG_INF;
                        m[j >> 3] = fmaxf(m[j >> 3], v);
                    }
                }
                if (qv) {
                    const int blk = key0 >> 3;   // this thread's first block
#pragma unroll
                    for (int u = 0; u < 2; ++u)
                        if (8 * (int64_t)(blk + u) < a.N) brow[blk + u] = score_key(0.5f * m[u]);
                }
                ++acount;
            }
        }
    }
    if (*abort_word && tid == 0) flag_error(a.err_flag, CSA2_FLAG_TIMEOUT);
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    if (warp == 0) tc::tmem_dealloc(tmem, TMEM_COLS);
}

}  // namespace

bool index_score_prefill_tc_supported(int T, csa2_dtype dt) { return dt == CSA2_FP8_E4M3 && T >= 64; }

// cuTensorMapEncodeTiled from the driver, looked up once through the runtime.
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
static EncodeTiledFn encode_tiled() {
    static const EncodeTiledFn fn = []() -> EncodeTiledFn {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        return reinterpret_cast<EncodeTiledFn>(p);
    }();
    return fn;
}

// A tensor map over `rows` rows of 64 bytes (FP8 vectors of the indexer) with
// boxes of box_rows rows, 64-byte swizzled in shared memory; rows past the end
// read as zero.
static csa2_status rows64_map(CUtensorMap *m, const void *base, uint64_t rows, uint32_t box_rows, const char *what) {
    const EncodeTiledFn f = encode_tiled();
    if (!f) {
        set_error("%s: cuTensorMapEncodeTiled is not available from the driver", what);
        return CSA2_ERR_CUDA;
    }
    const cuuint64_t dims[2] = {64, rows};
    const cuuint64_t strides[1] = {64};
    const cuuint32_t box[2] = {64, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = f(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        set_error("%s: cuTensorMapEncodeTiled failed (%d)", what, (int)r);
        return CSA2_ERR_CUDA;
    }
    return CSA2_OK;
}

// A tensor map over the query rows [rows][4 heads][64 bytes] as (64 bytes, head,
// row), boxes of one head of box_rows rows, 64-byte swizzled in shared memory;
// rows past the end read as zero.
static csa2_status heads64_map(CUtensorMap *m, const void *base, uint64_t rows, uint32_t box_rows, const char *what) {
    const EncodeTiledFn f = encode_tiled();
    if (!f) {
        set_error("%s: cuTensorMapEncodeTiled is not available from the driver", what);
        return CSA2_ERR_CUDA;
    }
    const cuuint64_t dims[3] = {64, 4, rows};
    const cuuint64_t strides[2] = {64, 256};
    const cuuint32_t box[3] = {64, 1, box_rows};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = f(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(base), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        set_error("%s: cuTensorMapEncodeTiled failed (%d)", what, (int)r);
        return CSA2_ERR_CUDA;
    }
    return CSA2_OK;
}

static PrefillArgs prefill_args(int B, int T, int64_t N, const float *w, const int32_t *kv_len, uint32_t *err_flag) {
    PrefillArgs a = {};
    a.B = B; a.T = T; a.N = N;
    a.w = w; a.kv_len = kv_len;
    a.err_flag = err_flag;
    a.qtiles = (T + QT - 1) / QT;
    a.ktiles = (int)((N + KT - 1) / KT);
    a.kranges = (a.ktiles + KTILES_PER_ITEM - 1) / KTILES_PER_ITEM;
    a.items = (int64_t)B * a.qtiles * a.kranges;
    return a;
}

static csa2_status launch_prefill(const PrefillArgs &a, const void *q, const void *k, cudaStream_t stream) {
    if (a.items == 0) return CSA2_OK;
    // TMA row coordinates are 32-bit
    if ((int64_t)a.B * a.T * 4 + QR > 0x7FFFFFFF || (int64_t)a.B * a.N + KT > 0x7FFFFFFF) {
        set_error("index_score_prefill_tc: B*T*4 or B*N beyond 2^31 rows");
        return CSA2_ERR_UNSUPPORTED;
    }
    CUtensorMap qm, km;
    csa2_status st = rows64_map(&qm, q, (uint64_t)a.B * a.T * 4, QR, "index_score_prefill_tc (q)");
    if (st != CSA2_OK) return st;
    st = rows64_map(&km, k, (uint64_t)a.B * a.N, KT, "index_score_prefill_tc (k)");
    if (st != CSA2_OK) return st;
    static bool smem_set[64];
    CSA2_CUDA_CALL(ensure_smem_limit((const void *)index_score_prefill_tc_kernel, (int)SMEM, smem_set),
                   "index_score_prefill_tc: smem attribute");
    const int64_t grid = a.items < num_sms() ? a.items : num_sms();
    CSA2_CUDA_CALL(launch_pdl(index_score_prefill_tc_kernel, dim3((unsigned)grid), dim3(THREADS), SMEM, stream,
                              qm, km, a),
                   "index_score_prefill_tc_kernel launch");
    CSA2_LAUNCH_CHECK("index_score_prefill_tc_kernel");
    return CSA2_OK;
}

csa2_status launch_index_score_prefill_tc(int B, int T, int64_t N, const void *q, const float *w, const void *k,
                                          const int32_t *kv_len, float *scores, uint32_t *err_flag,
                                          cudaStream_t stream) {
    PrefillArgs a = prefill_args(B, T, N, w, kv_len, err_flag);
    a.scores = scores;
    return launch_prefill(a, q, k, stream);
}

csa2_status launch_prefill_block_max(int B, int T, int64_t N, const void *q, const float *w, const void *k,
                                     const int32_t *kv_len, uint32_t *bmax, int64_t nblk, uint32_t *err_flag,
                                     cudaStream_t stream) {
    PrefillArgs a = prefill_args(B, T, N, w, kv_len, err_flag);
    a.bmax = bmax;
    a.nblk = nblk;
    a.qtiles = (T + BQ - 1) / BQ;
    a.ktiles = (int)((N + BK - 1) / BK);
    a.kranges = (a.ktiles + BKTILES_PER_ITEM - 1) / BKTILES_PER_ITEM;
    a.items = (int64_t)B * a.qtiles * a.kranges;
    if (a.items == 0) return CSA2_OK;
    // TMA row coordinates are 32-bit
    if ((int64_t)B * T + BQ > 0x7FFFFFFF || (int64_t)B * N + BK > 0x7FFFFFFF) {
        set_error("index_blockmax_tc: B*T or B*N beyond 2^31 rows");
        return CSA2_ERR_UNSUPPORTED;
    }
    CUtensorMap qm, km;
    csa2_status st = heads64_map(&qm, q, (uint64_t)B * T, BQ, "index_blockmax_tc (q)");
    if (st != CSA2_OK) return st;
    st = rows64_map(&km, k, (uint64_t)B * N, BK, "index_blockmax_tc (k)");
    if (st != CSA2_OK) return st;
    static bool smem_set[64];
    CSA2_CUDA_CALL(ensure_smem_limit((const void *)index_blockmax_tc_kernel, (int)BSMEM, smem_set),
                   "index_blockmax_tc: smem attribute");
    const int64_t grid = a.items < num_sms() ? a.items : num_sms();
    CSA2_CUDA_CALL(launch_pdl(index_blockmax_tc_kernel, dim3((unsigned)grid), dim3(THREADS), BSMEM, stream, qm, km, a),
                   "index_blockmax_tc_kernel launch");
    CSA2_LAUNCH_CHECK("index_blockmax_tc_kernel");
    return CSA2_OK;
}

}  // namespace csa2

// Indexer scoring of many query tokens (prefill-shaped Full mode, FP8) on
// the 5th-generation tensor cores.
// Sources: "DeepSeek-V4.1-Flash：把 KV Cache 压缩到极限的百万上下文 MoE", section
// "Hierarchical Sparse Indexer——索引成本变常数" (Full layers score every entry);
// the score sum_h w_h * ReLU(q_h . k) is not on the pages.
//
// With thousands of query tokens per sequence the scores are a dense
// contraction: [T x 4 heads, 64] x [64, N keys].  Work item = (sequence b,
// 64-query tile, range of 128-key tiles).  A persistent CTA per SM:
//  - keeps the query tile (256 query-head rows x 64 B, FP8) in shared memory
//    as the MMA B operand (K-major, no-swizzle core matrices);
//  - streams key tiles (128 keys x 64 B) through an 8-stage cp.async ring,
//    remapping each 16-byte chunk into the core-matrix layout;
//  - issues S^T [128 keys x 256 query-heads] = K . Q^T as two tcgen05.mma
//    kind::f8f6f4 (E4M3 x E4M3, K = 32 each) into one of two TMEM
//    accumulators, so the MMA of tile i+1 overlaps the epilogue of tile i;
//  - epilogue (16 warps): TMEM lane = key, 4 consecutive columns = the 4
//    heads of one query, so score = sum_h w_h * max(x_h, 0) stays inside a
//    thread;
//    keys at or beyond the query's kv_len become -inf; each warp store writes
//    32 consecutive keys of one query (128 B).
// Key tiles beyond every query's kv_len skip the MMA and store -inf.  The
// scores are fp32 [B, T, N]: this kernel is bound by writing them.
//
// The same main loop has a second epilogue, the first pass of the fused dense
// indexer (csa2_index_topk_dense) that never writes the score matrix:
// BLOCKMAX keeps the order-preserving key of each 8-key block's maximum
// score.  Three xor-shuffle steps reduce over the 8 lanes (= keys) of a block
// and transpose at the same time (each step keeps half of the queries), so
// one 32-lane store writes the 8 queries x 4 blocks of a warp.
#include "common.cuh"
#include "tc.cuh"

namespace csa2 {
namespace {

enum { EPI_SCORES = 0, EPI_BLOCKMAX = 1 };

constexpr int QT = 64;                 // queries per tile
constexpr int QR = QT * 4;             // query-head rows (MMA N)
constexpr int KT = 128;                // keys per tile (MMA M)
constexpr int KTILES_PER_ITEM = 16;    // key tiles per work item
constexpr int STAGES = 8;
constexpr int THREADS = 512;             // 16 warps: 4 per TMEM lane quarter
constexpr uint32_t Q_BYTES = QR * 64;           // 16 KB
constexpr uint32_t K_BYTES = KT * 64;           // 8 KB per stage
constexpr uint32_t SBO = 4 * 128;               // 8-row group stride (64 B rows = 4 core matrices)
constexpr uint32_t OFF_Q = 0;
constexpr uint32_t OFF_K = OFF_Q + Q_BYTES;
constexpr uint32_t OFF_W = OFF_K + STAGES * K_BYTES;  // float[QT][4]
constexpr uint32_t OFF_LT = OFF_W + QT * 16;          // int2[QT]: (kv_len clamped to N, 0)
constexpr uint32_t OFF_BAR = OFF_LT + QT * 8;         // 2 mbarriers
constexpr uint32_t OFF_TMEM = OFF_BAR + 16;
constexpr uint32_t OFF_SMAX = OFF_TMEM + 8;              // int[2]: longest kv_len of the tile's queries
constexpr uint32_t SMEM_USED = OFF_SMAX + 8;
// request more than half of the SM's shared memory: one CTA per SM, so the
// CTA's 512 TMEM columns are never contended
constexpr uint32_t SMEM = SMEM_USED > 120 * 1024 ? SMEM_USED : 120 * 1024;
constexpr uint32_t TMEM_COLS = 512;                   // 2 accumulators x 256 columns
constexpr uint32_t MAX_POLLS = 1u << 22;

struct PrefillArgs {
    int B, T;
    int64_t N;
    const uint8_t *q;
    const float *w;
    const uint8_t *k;
    const int32_t *kv_len;
    float *scores;
    uint32_t *err_flag;
    int qtiles, ktiles, kranges;
    int64_t items;
    // BLOCKMAX: keys of the 8-key block maxima, [B*T, nblk]
    uint32_t *bmax;
    int64_t nblk;
};

// sum_h w_h * max(x_h, 0) with every rounding spelled out, so that each pass
// computes the same fp32 value.
__device__ __forceinline__ float head_sum(const float4 wq, const uint32_t *r) {
    float s = __fmul_rn(wq.x, fmaxf(__uint_as_float(r[0]), 0.f));
    s = __fmaf_rn(wq.y, fmaxf(__uint_as_float(r[1]), 0.f), s);
    s = __fmaf_rn(wq.z, fmaxf(__uint_as_float(r[2]), 0.f), s);
    return __fmaf_rn(wq.w, fmaxf(__uint_as_float(r[3]), 0.f), s);
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, bool valid) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(valid ? 16 : 0));
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;"); }
template <int N>
__device__ __forceinline__ void cp_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

template <int EPI>
__global__ void __launch_bounds__(THREADS, 1) index_score_prefill_tc_kernel(PrefillArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    float *sW = reinterpret_cast<float *>(smem + OFF_W);
    const float4 *sW4 = reinterpret_cast<const float4 *>(smem + OFF_W);
    int2 *sLT = reinterpret_cast<int2 *>(smem + OFF_LT);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + OFF_TMEM);
    int *sMax = reinterpret_cast<int *>(smem + OFF_SMAX);
    const uint32_t bar0 = tc::smem_u32(smem + OFF_BAR);
    const uint32_t sq = tc::smem_u32(smem + OFF_Q), sk = tc::smem_u32(smem + OFF_K);
    const float NEG_INF = __int_as_float(0xff800000);

    if (tid == 0) {
        tc::mbar_init(bar0, 1);
        tc::mbar_init(bar0 + 8, 1);
        tc::mbar_init_fence();
    }
    if (warp == 0) tc::tmem_alloc(tmem_slot, TMEM_COLS);
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tmem = *tmem_slot;
    pdl_wait();
    pdl_launch_dependents();
    uint32_t uses0 = 0, uses1 = 0;   // completed phases of the two accumulator barriers
    bool ok = true;

    for (int64_t item = blockIdx.x; item < a.items; item += gridDim.x) {
        const int kr = (int)(item % a.kranges);
        const int64_t rest = item / a.kranges;
        const int qt = (int)(rest % a.qtiles);
        const int64_t b = rest / a.qtiles;
        const int t0 = qt * QT;
        const int kt0 = kr * KTILES_PER_ITEM;
        const int kt1 = min(a.ktiles, kt0 + KTILES_PER_ITEM);

        // ---- query tile (rows r = 4*query + head) and its w / kv_len
        __syncthreads();   // the previous item's epilogue reads of sW / sLT are done
        for (int c = tid; c < QR * 4; c += THREADS) {
            const int r = c >> 2, ch = c & 3, tq = t0 + (r >> 2);
            const bool v = tq < a.T;
            const uint8_t *src = a.q + ((b * a.T + (v ? tq : 0)) * 4 + (r & 3)) * 64 + ch * 16;
            cp_async16(sq + (r >> 3) * SBO + ch * 128 + (r & 7) * 16, src, v);
        }
        if (tid < QT) {   // warps 0 and 1
            const int tq = t0 + tid;
            const bool v = tq < a.T;
            const int64_t row = b * a.T + (v ? tq : 0);
            for (int h = 0; h < 4; ++h) sW[tid * 4 + h] = v ? a.w[row * 4 + h] : 0.f;
            int64_t len = v ? (int64_t)a.kv_len[row] : 0;
            const int lc = (int)(len < 0 ? 0 : (len < a.N ? len : a.N));
            sLT[tid] = make_int2(lc, 0);
            const int m = __reduce_max_sync(0xFFFFFFFFu, lc);
            if (lane == 0) sMax[warp] = m;
        }
        cp_commit();
        int maxlen = 0;   // longest visible prefix among the tile's queries, read after the first barrier

        auto load_ktile = [&](int kt, int stage) {
            for (int c = tid; c < KT * 4; c += THREADS) {
                const int r = c >> 2, ch = c & 3;
                const int64_t key = (int64_t)kt * KT + r;
                const bool v = key < a.N;
                const uint8_t *src = a.k + ((b * a.N + (v ? key : 0)) * 64) + ch * 16;
                cp_async16(sk + stage * K_BYTES + (r >> 3) * SBO + ch * 128 + (r & 7) * 16, src, v);
            }
            cp_commit();
        };
        // prologue: STAGES-1 key tiles in flight
        for (int i = 0; i < STAGES - 1; ++i) {
            if (kt0 + i < kt1) load_ktile(kt0 + i, i);
            else cp_commit();
        }

        int prev_tile = -1, prev_buf = 0;
        bool prev_mma = false;
        // Epilogue of one key tile: warp w reads TMEM lane quarter w & 3 (32
        // keys, lane = key) and the columns of queries 16 (w >> 2) .. +15.
        auto epilogue = [&](int tile, int buf, bool did_mma) {
            const int lq = warp & 3, qg = warp >> 2;
            const int64_t key = (int64_t)tile * KT + 32 * lq + lane;
            const int64_t row0 = b * a.T + t0 + 16 * qg;
            if (did_mma) {
                const uint32_t u = buf ? uses1 : uses0;
                ok = tc::mbar_wait(bar0 + 8 * buf, u & 1, MAX_POLLS) && ok;
                if (buf) ++uses1; else ++uses0;
                tc::fence_after();
            }
            // A skipped tile has no visible key for any query of the tile:
            // nothing to write for the block maxima.
            if (EPI != EPI_SCORES && !did_mma) return;
            const uint32_t ta = tmem + ((uint32_t)(32 * lq) << 16) + buf * 256 + 64 * qg;
            // eight queries of this warp's sixteen, from 32 TMEM columns.
            // Straight-line over the eight (queries past T have kv_len 0 in
            // sLT, so they are invalid without a branch): the independent
            // chains interleave.
            auto eight = [&](const uint32_t (&r)[32], int h) {
                const int q0 = 16 * qg + 8 * h;
                float s[8];
#pragma unroll
                for (int qq = 0; qq < 8; ++qq) {
                    const float4 wq = sW4[q0 + qq];
                    const int2 lt = sLT[q0 + qq];
                    s[qq] = (did_mma && key < lt.x) ? head_sum(wq, r + 4 * qq) : NEG_INF;
                }
                const int64_t rowh = row0 + 8 * h;
                const int nq = a.T - (t0 + q0);   // queries of these eight that exist
                if constexpr (EPI == EPI_SCORES) {
                    if (key < a.N) {
#pragma unroll
                        for (int qq = 0; qq < 8; ++qq)
                            if (qq < nq) a.scores[(rowh + qq) * a.N + key] = s[qq];
                    }
                } else if constexpr (EPI == EPI_BLOCKMAX) {
                    // Max over the 8 keys of each block, transposed on the way:
                    // at each xor step a lane keeps half of its queries and
                    // takes the partner's values for them.  Lane l ends with
                    // the block max of query 4 b0 + 2 b1 + b2 (b = bits of l)
                    // over keys 8 (l >> 3) .. +7 of its 32: one store for all.
                    const bool b0 = lane & 1, b1 = (lane >> 1) & 1, b2 = (lane >> 2) & 1;
                    float x[4], y[2];
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const float send = b0 ? s[j] : s[4 + j], keep = b0 ? s[4 + j] : s[j];
                        x[j] = fmaxf(keep, __shfl_xor_sync(0xFFFFFFFFu, send, 1));
                    }
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        const float send = b1 ? x[j] : x[2 + j], keep = b1 ? x[2 + j] : x[j];
                        y[j] = fmaxf(keep, __shfl_xor_sync(0xFFFFFFFFu, send, 2));
                    }
                    const float send = b2 ? y[0] : y[1], keep = b2 ? y[1] : y[0];
                    const float m = fmaxf(keep, __shfl_xor_sync(0xFFFFFFFFu, send, 4));
                    const int qs = 4 * b0 + 2 * b1 + b2;
                    const int64_t blk = (key - lane + 8 * (lane >> 3)) >> 3;   // this lane's block
                    if (qs < nq && 8 * blk < a.N) a.bmax[(rowh + qs) * a.nblk + blk] = score_key(m);
                }
            };
            if constexpr (EPI == EPI_SCORES) {
                // one half at a time: the store addresses need the registers
#pragma unroll 1
                for (int h = 0; h < 2; ++h) {
                    uint32_t r[32];
                    if (did_mma) {
                        tc::tmem_ld32(ta + 32 * h, r);
                        tc::tmem_ld_wait();
                    }
                    eight(r, h);
                }
            } else {
                uint32_t r0[32], r1[32];
                tc::tmem_ld32(ta, r0);
                tc::tmem_ld32(ta + 32, r1);
                tc::tmem_ld_wait();
                eight(r0, 0);
                eight(r1, 1);
            }
        };

        for (int kt = kt0; kt < kt1; ++kt) {
            const int i = kt - kt0;
            cp_wait<STAGES - 2>();      // tile kt (and the query tile) have landed
            tc::fence_async_smem();
            tc::fence_before();
            __syncthreads();
            tc::fence_after();
            const int buf = i & 1;
            if (i == 0) maxlen = max(sMax[0], sMax[1]);
            const bool do_mma = (int64_t)kt * KT < maxlen;
            if (tid == 0 && do_mma) {
                constexpr uint32_t idesc = tc::idesc_e4m3_f32(KT, QR, false, false);
                const uint32_t ka = sk + (i % STAGES) * K_BYTES;
#pragma unroll
                for (int ks = 0; ks < 2; ++ks)
                    tc::mma_f8(tmem + buf * 256, tc::desc_noswizzle(ka + ks * 256, 128, SBO),
                               tc::desc_noswizzle(sq + ks * 256, 128, SBO), idesc, ks > 0);
                tc::commit(bar0 + 8 * buf);
            }
            if (prev_tile >= 0) epilogue(prev_tile, prev_buf, prev_mma);   // also frees stage (i-1)%STAGES
            __syncthreads();
            if (kt + STAGES - 1 < kt1) load_ktile(kt + STAGES - 1, (i + STAGES - 1) % STAGES);
            else cp_commit();
            prev_tile = kt;
            prev_buf = buf;
            prev_mma = do_mma;
        }
        if (prev_tile >= 0) epilogue(prev_tile, prev_buf, prev_mma);
        cp_wait<0>();
    }
    if (!ok && tid == 0) flag_error(a.err_flag, CSA2_FLAG_TIMEOUT);
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    if (warp == 0) tc::tmem_dealloc(tmem, TMEM_COLS);
}

}  // namespace

bool index_score_prefill_tc_supported(int T, csa2_dtype dt) { return dt == CSA2_FP8_E4M3 && T >= 64; }

static PrefillArgs prefill_args(int B, int T, int64_t N, const void *q, const float *w, const void *k,
                                const int32_t *kv_len, uint32_t *err_flag) {
    PrefillArgs a = {};
    a.B = B; a.T = T; a.N = N;
    a.q = (const uint8_t *)q; a.w = w; a.k = (const uint8_t *)k; a.kv_len = kv_len;
    a.err_flag = err_flag;
    a.qtiles = (T + QT - 1) / QT;
    a.ktiles = (int)((N + KT - 1) / KT);
    a.kranges = (a.ktiles + KTILES_PER_ITEM - 1) / KTILES_PER_ITEM;
    a.items = (int64_t)B * a.qtiles * a.kranges;
    return a;
}

template <int EPI>
static csa2_status launch_prefill(const PrefillArgs &a, cudaStream_t stream) {
    static bool smem_set[64];
    CSA2_CUDA_CALL(ensure_smem_limit((const void *)index_score_prefill_tc_kernel<EPI>, (int)SMEM, smem_set),
                   "index_score_prefill_tc: smem attribute");
    int64_t grid = a.items < num_sms() ? a.items : num_sms();
    CSA2_CUDA_CALL(launch_pdl(index_score_prefill_tc_kernel<EPI>, dim3((unsigned)grid), dim3(THREADS), SMEM, stream,
                              a),
                   "index_score_prefill_tc_kernel launch");
    CSA2_LAUNCH_CHECK("index_score_prefill_tc_kernel");
    return CSA2_OK;
}

csa2_status launch_index_score_prefill_tc(int B, int T, int64_t N, const void *q, const float *w, const void *k,
                                          const int32_t *kv_len, float *scores, uint32_t *err_flag,
                                          cudaStream_t stream) {
    PrefillArgs a = prefill_args(B, T, N, q, w, k, kv_len, err_flag);
    a.scores = scores;
    return launch_prefill<EPI_SCORES>(a, stream);
}

csa2_status launch_prefill_block_max(int B, int T, int64_t N, const void *q, const float *w, const void *k,
                                     const int32_t *kv_len, uint32_t *bmax, int64_t nblk, uint32_t *err_flag,
                                     cudaStream_t stream) {
    PrefillArgs a = prefill_args(B, T, N, q, w, k, kv_len, err_flag);
    a.bmax = bmax;
    a.nblk = nblk;
    return launch_prefill<EPI_BLOCKMAX>(a, stream);
}


}  // namespace csa2

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
//  - streams key tiles (128 keys x 64 B) through a 4-stage cp.async ring,
//    remapping each 16-byte chunk into the core-matrix layout;
//  - issues S^T [128 keys x 256 query-heads] = K . Q^T as two tcgen05.mma
//    kind::f8f6f4 (E4M3 x E4M3, K = 32 each) into one of two TMEM
//    accumulators, so the MMA of tile i+1 overlaps the epilogue of tile i;
//  - epilogue (8 warps): TMEM lane = key, 4 consecutive columns = the 4 heads
//    of one query, so score = sum_h w_h * max(x_h, 0) stays inside a thread;
//    keys at or beyond the query's kv_len become -inf; each warp store writes
//    32 consecutive keys of one query (128 B).
// Key tiles beyond every query's kv_len skip the MMA and store -inf.  The
// scores are fp32 [B, T, N]: this kernel is bound by writing them.
#include "common.cuh"
#include "tc.cuh"

namespace csa2 {
namespace {

constexpr int QT = 64;                 // queries per tile
constexpr int QR = QT * 4;             // query-head rows (MMA N)
constexpr int KT = 128;                // keys per tile (MMA M)
constexpr int KTILES_PER_ITEM = 16;    // key tiles per work item
constexpr int STAGES = 4;
constexpr int THREADS = 256;
constexpr uint32_t Q_BYTES = QR * 64;           // 16 KB
constexpr uint32_t K_BYTES = KT * 64;           // 8 KB per stage
constexpr uint32_t SBO = 4 * 128;               // 8-row group stride (64 B rows = 4 core matrices)
constexpr uint32_t OFF_Q = 0;
constexpr uint32_t OFF_K = OFF_Q + Q_BYTES;
constexpr uint32_t OFF_W = OFF_K + STAGES * K_BYTES;  // float[QT][4]
constexpr uint32_t OFF_LEN = OFF_W + QT * 16;         // int[QT]
constexpr uint32_t OFF_BAR = OFF_LEN + QT * 4;        // 2 mbarriers
constexpr uint32_t OFF_TMEM = OFF_BAR + 16;
constexpr uint32_t SMEM_USED = OFF_TMEM + 16;
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
};

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, bool valid) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(valid ? 16 : 0));
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;"); }
template <int N>
__device__ __forceinline__ void cp_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

__global__ void __launch_bounds__(THREADS, 1) index_score_prefill_tc_kernel(PrefillArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    float *sW = reinterpret_cast<float *>(smem + OFF_W);
    int *sLen = reinterpret_cast<int *>(smem + OFF_LEN);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + OFF_TMEM);
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
        __syncthreads();   // the previous item's epilogue reads of sW / sLen are done
        for (int c = tid; c < QR * 4; c += THREADS) {
            const int r = c >> 2, ch = c & 3, tq = t0 + (r >> 2);
            const bool v = tq < a.T;
            const uint8_t *src = a.q + ((b * a.T + (v ? tq : 0)) * 4 + (r & 3)) * 64 + ch * 16;
            cp_async16(sq + (r >> 3) * SBO + ch * 128 + (r & 7) * 16, src, v);
        }
        if (tid < QT) {
            const int tq = t0 + tid;
            const bool v = tq < a.T;
            const int64_t row = b * a.T + (v ? tq : 0);
            for (int h = 0; h < 4; ++h) sW[tid * 4 + h] = v ? a.w[row * 4 + h] : 0.f;
            int64_t len = v ? (int64_t)a.kv_len[row] : 0;
            sLen[tid] = (int)(len < a.N ? len : a.N);
        }
        cp_commit();
        int maxlen = 0;
        {
            // longest visible prefix among the tile's queries (uniform across the CTA)
            int64_t m = 0;
            for (int i = 0; i < QT; ++i) {
                const int tq = t0 + i;
                if (tq < a.T) {
                    int64_t len = a.kv_len[b * a.T + tq];
                    m = len > m ? len : m;
                }
            }
            maxlen = (int)(m < a.N ? m : a.N);
        }

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
        auto epilogue = [&](int tile, int buf, bool did_mma) {
            const int64_t key = (int64_t)tile * KT + 32 * (warp & 3) + lane;
            const int qbase = 32 * (warp >> 2);    // warps 0-3: queries 0-31, warps 4-7: 32-63
            if (did_mma) {
                const uint32_t u = buf ? uses1 : uses0;
                ok = tc::mbar_wait(bar0 + 8 * buf, u & 1, MAX_POLLS) && ok;
                if (buf) ++uses1; else ++uses0;
                tc::fence_after();
            }
#pragma unroll 1
            for (int cblk = 0; cblk < 4; ++cblk) {   // 8 queries (32 columns) per TMEM load
                uint32_t r[32];
                if (did_mma) {
                    tc::tmem_ld32(tmem + ((uint32_t)(32 * (warp & 3)) << 16) + buf * 256 + 128 * (warp >> 2) + 32 * cblk, r);
                    tc::tmem_ld_wait();
                }
#pragma unroll
                for (int qq = 0; qq < 8; ++qq) {
                    const int ql = qbase + 8 * cblk + qq;
                    const int tq = t0 + ql;
                    if (tq >= a.T || key >= a.N) continue;
                    float s = NEG_INF;
                    if (did_mma && key < sLen[ql]) {
                        const float *wq = sW + ql * 4;
                        s = wq[0] * fmaxf(__uint_as_float(r[4 * qq]), 0.f) + wq[1] * fmaxf(__uint_as_float(r[4 * qq + 1]), 0.f) +
                            wq[2] * fmaxf(__uint_as_float(r[4 * qq + 2]), 0.f) + wq[3] * fmaxf(__uint_as_float(r[4 * qq + 3]), 0.f);
                    }
                    a.scores[(b * a.T + tq) * a.N + key] = s;
                }
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

csa2_status launch_index_score_prefill_tc(int B, int T, int64_t N, const void *q, const float *w, const void *k,
                                          const int32_t *kv_len, float *scores, uint32_t *err_flag,
                                          cudaStream_t stream) {
    static bool smem_set[64];
    CSA2_CUDA_CALL(ensure_smem_limit((const void *)index_score_prefill_tc_kernel, (int)SMEM, smem_set),
                   "index_score_prefill_tc: smem attribute");
    PrefillArgs a;
    a.B = B; a.T = T; a.N = N;
    a.q = (const uint8_t *)q; a.w = w; a.k = (const uint8_t *)k; a.kv_len = kv_len; a.scores = scores;
    a.err_flag = err_flag;
    a.qtiles = (T + QT - 1) / QT;
    a.ktiles = (int)((N + KT - 1) / KT);
    a.kranges = (a.ktiles + KTILES_PER_ITEM - 1) / KTILES_PER_ITEM;
    a.items = (int64_t)B * a.qtiles * a.kranges;
    int64_t grid = a.items < num_sms() ? a.items : num_sms();
    CSA2_CUDA_CALL(launch_pdl(index_score_prefill_tc_kernel, dim3((unsigned)grid), dim3(THREADS), SMEM, stream, a),
                   "index_score_prefill_tc_kernel launch");
    CSA2_LAUNCH_CHECK("index_score_prefill_tc_kernel");
    return CSA2_OK;
}

}  // namespace csa2

// csa2_topk and csa2_build_pool: per-row Top-K by radix select.
// Sources: "DeepSeek-V4.1-Flash：把 KV Cache 压缩到极限的百万上下文 MoE", CSA2
// section (Top-512 in every layer) and "Hierarchical Sparse Indexer" (a pool
// of at most 2048 blocks x 8 positions built from block scores);
// "552B参数干掉1.6T：DeepSeek V4.1 Flash技术深度解析", DeepSelect paragraph (the
// Top-K kernel of the sparse attention).
//
// Design.  Decode rows are few and long (32 x 16384 scores, 8 x 32768 block
// maxima), so one row is split over a thread-block cluster of C CTAs.  Each
// CTA loads its slice of the row ONCE from HBM into shared memory as
// order-preserving uint32 keys, then the cluster runs four 8-bit radix passes
// (most significant digit first).  Per pass every CTA builds a 256-bin
// histogram of the keys that still match the chosen prefix (warp-aggregated
// shared atomics), the cluster barrier publishes it, and every CTA sums the C
// histograms through distributed shared memory and picks the same digit.
// After the passes the K-th largest key T and the number of T-valued keys to
// take are known; CTAs then write the keys > T and the first ties (lowest
// positions first) with offsets derived from per-CTA counts exchanged the
// same way.  Only hardware cluster barriers are used: no flag spinning.
#include <cooperative_groups.h>

#include "common.cuh"

namespace cg = cooperative_groups;

namespace csa2 {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxCluster = 8;
constexpr int kMaxKeysPerCta = 32768;  // 128 KB of keys

enum Loader { LOAD_SCORES = 0, LOAD_REINDEX = 1, LOAD_BLOCKMAX = 2 };

struct TopkArgs {
    int loader;
    int64_t rows;
    int64_t M;               // scores row length
    const float *scores;
    const int32_t *kv_len;   // nullable (LOAD_SCORES)
    const int32_t *pool;     // LOAD_REINDEX
    int P;
    int K;
    int32_t *out;            // [rows, K]
    int chunk;               // keys per CTA
    int csize;               // CTAs per row (cluster size)
};

__device__ __forceinline__ int64_t row_len(const TopkArgs &a, int64_t row) {
    if (a.loader == LOAD_REINDEX) return a.M;
    int64_t len = a.kv_len ? (int64_t)a.kv_len[row] : a.M;
    len = len < a.M ? len : a.M;
    len = len > 0 ? len : 0;
    if (a.loader == LOAD_BLOCKMAX) return (len + 7) / 8;
    return len;
}

__global__ void __launch_bounds__(kThreads) topk_radix_kernel(TopkArgs a) {
    extern __shared__ uint32_t keys[];
    __shared__ uint32_t hist[2][256];
    __shared__ uint32_t wsum[8];
    __shared__ uint32_t sel_digit, sel_above, few_keys;
    __shared__ uint32_t cnt[2];               // this CTA's (#gt, #eq)
    __shared__ uint32_t wcnt[2][kWarps];

    cg::cluster_group cluster = cg::this_cluster();
    const int cta = (int)cluster.block_rank();
    const int64_t row = blockIdx.x / a.csize;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    const int64_t L = row_len(a, row);
    const int64_t beg = (int64_t)cta * a.chunk;
    int n = 0;
    if (beg < L) n = (int)((L - beg) < a.chunk ? (L - beg) : a.chunk);

    // ---------------------------------------------------------------- load
    const float *srow = a.scores + row * a.M;
    if (a.loader == LOAD_BLOCKMAX) {
        const int64_t len = a.kv_len ? min((int64_t)a.kv_len[row], a.M) : a.M;
        const bool vec = ((a.M & 3) == 0) && ((reinterpret_cast<uintptr_t>(a.scores) & 15) == 0);
        for (int i = tid; i < n; i += kThreads) {
            const int64_t j0 = (beg + i) * 8;
            float m = __int_as_float(0xff800000);
            if (vec && j0 + 8 <= len) {
                float4 x = __ldg(reinterpret_cast<const float4 *>(srow + j0));
                float4 y = __ldg(reinterpret_cast<const float4 *>(srow + j0) + 1);
                m = fmaxf(fmaxf(fmaxf(x.x, x.y), fmaxf(x.z, x.w)), fmaxf(fmaxf(y.x, y.y), fmaxf(y.z, y.w)));
            } else {
                for (int64_t j = j0; j < j0 + 8 && j < len; ++j) m = fmaxf(m, __ldg(srow + j));
            }
            keys[i] = score_key(m);
        }
    } else if (a.loader == LOAD_REINDEX) {
        const int32_t *prow = a.pool + row * a.P;
        for (int i = tid; i < n; i += kThreads) {
            const int64_t l = beg + i;
            uint32_t k = score_key(__ldg(srow + l));
            if (__ldg(prow + l / 8) < 0) k = 0;
            keys[i] = k;
        }
    } else {
        for (int i = tid; i < n; i += kThreads) keys[i] = score_key(__ldg(srow + beg + i));
    }

    // ---------------------------------------------------------------- radix select
    uint32_t prefix = 0, pmask = 0;
    uint32_t kk = (uint32_t)a.K;      // rank still to find among prefix-matching keys
    bool few = false;
    for (int pass = 0; pass < 4; ++pass) {
        const int shift = 24 - 8 * pass;
        uint32_t *h = hist[pass & 1];
        if (tid < 256) h[tid] = 0;
        __syncthreads();  // also orders the key loads before the first pass
        for (int base = 0; base < n; base += kThreads) {
            const int i = base + tid;
            uint32_t d = 0x100;  // "not participating"
            if (i < n) {
                const uint32_t k = keys[i];
                if ((k & pmask) == prefix) d = (k >> shift) & 0xFF;
            }
            const uint32_t peers = __match_any_sync(0xFFFFFFFFu, d);
            if (d != 0x100 && lane == __ffs(peers) - 1) atomicAdd(&h[d], __popc(peers));
        }
        cluster.sync();  // every CTA's histogram for this pass is complete
        uint32_t tot = 0;
        if (tid < 256) {
            for (int c = 0; c < a.csize; ++c) tot += cluster.map_shared_rank(h, c)[tid];
            // inclusive suffix sum over bins: S[b] = sum_{b' >= b} tot[b']
            uint32_t s = tot;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                uint32_t t = __shfl_down_sync(0xFFFFFFFFu, s, off);
                if (lane + off < 32) s += t;
            }
            if (lane == 0) wsum[warp] = s;  // warps 0..7 cover bins 32w..32w+31
            tot = s;
        }
        __syncthreads();
        if (tid < 256) {
            uint32_t s = tot;
            for (int w2 = warp + 1; w2 < 8; ++w2) s += wsum[w2];
            uint32_t s_next = __shfl_down_sync(0xFFFFFFFFu, s, 1);
            if (lane == 31) {
                s_next = 0;
                for (int w2 = warp + 1; w2 < 8; ++w2) s_next += wsum[w2];
            }
            if (tid == 0 && s < kk) few_keys = 1;
            if (tid == 0 && s >= kk) few_keys = 0;
            if (s >= kk && s_next < kk) {
                sel_digit = (uint32_t)tid;
                sel_above = s_next;
            }
        }
        __syncthreads();
        if (few_keys) {  // fewer candidate keys in the row than K (only at pass 0)
            few = true;
            break;
        }
        kk -= sel_above;
        prefix |= sel_digit << shift;
        pmask |= 0xFFu << shift;
        // The next pass writes the other histogram buffer; remote reads of this
        // one finish before any CTA passes the next cluster barrier.
    }
    // T: the K-th largest key; ties at T beyond kk are dropped.  T == 0 (an
    // invalid key) or "few" means: take every valid key, pad with -1.
    uint32_t T = few ? 0u : prefix;
    if (T == 0) kk = 0;

    // ---------------------------------------------------------------- counts
    uint32_t my_gt = 0, my_eq = 0;
    for (int i = tid; i < n; i += kThreads) {
        const uint32_t k = keys[i];
        my_gt += (k > T);
        my_eq += (T != 0 && k == T);
    }
    for (int off = 16; off > 0; off >>= 1) {
        my_gt += __shfl_xor_sync(0xFFFFFFFFu, my_gt, off);
        my_eq += __shfl_xor_sync(0xFFFFFFFFu, my_eq, off);
    }
    if (lane == 0) { wcnt[0][warp] = my_gt; wcnt[1][warp] = my_eq; }
    __syncthreads();
    if (tid == 0) {
        uint32_t g = 0, e = 0;
        for (int w2 = 0; w2 < kWarps; ++w2) { g += wcnt[0][w2]; e += wcnt[1][w2]; }
        cnt[0] = g; cnt[1] = e;
    }
    cluster.sync();
    uint32_t total_gt = 0, gt_before = 0, eq_before = 0, eq_total = 0;
    for (int c = 0; c < a.csize; ++c) {
        const uint32_t *rc = cluster.map_shared_rank(cnt, c);
        const uint32_t g = rc[0], e = rc[1];
        total_gt += g;
        eq_total += e;
        if (c < cta) { gt_before += g; eq_before += e; }
    }
    const uint32_t my_eq_all = cnt[1];
    const uint32_t take_before = eq_before < kk ? eq_before : kk;
    uint32_t take_me = kk > eq_before ? kk - eq_before : 0u;
    take_me = take_me < my_eq_all ? take_me : my_eq_all;
    const uint32_t eq_off = total_gt + take_before;
    const uint32_t total_sel = total_gt + (eq_total < kk ? eq_total : kk);
    cluster.sync();  // all remote reads of cnt done before any CTA may exit

    // ---------------------------------------------------------------- ordered write
    int32_t *orow = a.out + row * a.K;
    uint32_t run_gt = 0, run_eq = 0;
    for (int base = 0; base < n; base += kThreads) {
        const int i = base + tid;
        uint32_t k = (i < n) ? keys[i] : 0u;
        const bool is_gt = (i < n) && k > T;
        const bool is_eq = (i < n) && T != 0 && k == T;
        const uint32_t bg = __ballot_sync(0xFFFFFFFFu, is_gt);
        const uint32_t be = __ballot_sync(0xFFFFFFFFu, is_eq);
        const uint32_t lt_mask = (1u << lane) - 1u;
        __syncthreads();  // previous round's wcnt reads are done
        if (lane == 0) { wcnt[0][warp] = __popc(bg); wcnt[1][warp] = __popc(be); }
        __syncthreads();
        uint32_t og = 0, oe = 0, rg = 0, re = 0;
        for (int w2 = 0; w2 < kWarps; ++w2) {
            const uint32_t cg_ = wcnt[0][w2], ce = wcnt[1][w2];
            if (w2 < warp) { og += cg_; oe += ce; }
            rg += cg_; re += ce;
        }
        if (is_gt || is_eq) {
            const int64_t li = beg + i;
            int32_t id;
            if (a.loader == LOAD_REINDEX) {
                id = (int32_t)((int64_t)__ldg(a.pool + row * a.P + li / 8) * 8 + (li & 7));
            } else {
                id = (int32_t)li;
            }
            if (is_gt) {
                orow[gt_before + run_gt + og + __popc(bg & lt_mask)] = id;
            } else {
                const uint32_t r = run_eq + oe + __popc(be & lt_mask);
                if (r < take_me) orow[eq_off + r] = id;
            }
        }
        run_gt += rg;
        run_eq += re;
    }
    if (cta == 0)
        for (int s = (int)total_sel + tid; s < a.K; s += kThreads) orow[s] = -1;
}

csa2_status launch_topk(const TopkArgs &in, int64_t Lmax, cudaStream_t stream) {
    TopkArgs a = in;
    if (a.rows == 0) return CSA2_OK;
    int C = 1;
    const int sms = num_sms();
    while (C < kMaxCluster && a.rows * C * 2 <= sms) C *= 2;
    auto chunk_for = [&](int c) { int64_t ch = (Lmax + c - 1) / c; return (ch + 3) & ~int64_t(3); };
    while (C > 1 && chunk_for(C) < 1024) C /= 2;
    while (C < kMaxCluster && chunk_for(C) > kMaxKeysPerCta) C *= 2;
    int64_t chunk = chunk_for(C);
    if (chunk > kMaxKeysPerCta) {
        set_error("topk: row of %lld candidates exceeds %d per row", (long long)Lmax, kMaxCluster * kMaxKeysPerCta);
        return CSA2_ERR_UNSUPPORTED;
    }
    if (chunk < 4) chunk = 4;
    a.chunk = (int)chunk;
    a.csize = C;
    const size_t smem = (size_t)chunk * sizeof(uint32_t);
    static bool smem_set[64];
    CSA2_CUDA_CALL(ensure_smem_limit((const void *)topk_radix_kernel, kMaxKeysPerCta * (int)sizeof(uint32_t), smem_set),
                   "topk: smem attribute");
    const int64_t grid = a.rows * C;
    if (grid > 0x7FFFFFFF) {
        set_error("topk: too many rows");
        return CSA2_ERR_UNSUPPORTED;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    CSA2_CUDA_CALL(cudaLaunchKernelEx(&cfg, topk_radix_kernel, a), "topk_radix_kernel launch");
    CSA2_LAUNCH_CHECK("topk_radix_kernel");
    return CSA2_OK;
}

}  // namespace
}  // namespace csa2

using namespace csa2;

extern "C" size_t csa2_topk_workspace_bytes(int, int, int64_t, int) { return 0; }
extern "C" size_t csa2_build_pool_workspace_bytes(int, int, int64_t, int) { return 0; }

extern "C" csa2_status csa2_topk(csa2_mode mode, int B, int T, int64_t M, const float *scores,
                                 const int32_t *kv_len, const int32_t *pool_blocks, int P, int K,
                                 int32_t *idx, void *workspace, size_t ws_bytes, csa2_stream_t stream) {
    (void)workspace;
    (void)ws_bytes;
    clear_error();
    CSA2_REQUIRE(mode == CSA2_MODE_FULL || mode == CSA2_MODE_REINDEX || mode == CSA2_MODE_REUSE,
                 "topk: bad mode %d", (int)mode);
    if (mode == CSA2_MODE_REUSE) return CSA2_OK;
    CSA2_REQUIRE(B >= 0 && T >= 0 && M >= 0, "topk: negative shape");
    CSA2_REQUIRE(K >= 1 && K <= CSA2_MAX_K, "topk: K=%d not in [1,2048]", K);
    if (mode == CSA2_MODE_REINDEX) {
        CSA2_REQUIRE(pool_blocks != nullptr, "topk: REINDEX needs pool_blocks");
        CSA2_REQUIRE(P >= 1 && P <= CSA2_MAX_POOL && M == (int64_t)P * 8, "topk: REINDEX needs M == 8P, P in [1,2048]");
    } else {
        CSA2_REQUIRE(pool_blocks == nullptr, "topk: FULL takes no pool_blocks");
    }
    if ((int64_t)B * T == 0) return CSA2_OK;
    CSA2_REQUIRE(scores && idx, "topk: null pointer");
    CSA2_REQUIRE(aligned(scores, 4) && aligned(idx, 4), "topk: misaligned scores/idx");
    TopkArgs a = {};
    a.loader = (mode == CSA2_MODE_REINDEX) ? LOAD_REINDEX : LOAD_SCORES;
    a.rows = (int64_t)B * T;
    a.M = M;
    a.scores = scores;
    a.kv_len = (mode == CSA2_MODE_FULL) ? kv_len : nullptr;
    a.pool = pool_blocks;
    a.P = P;
    a.K = K;
    a.out = idx;
    return launch_topk(a, M, stream_of(stream));
}

extern "C" csa2_status csa2_build_pool(int B, int T, int64_t N, const float *scores,
                                       const int32_t *kv_len, int P, int G, int32_t *pool_blocks,
                                       void *workspace, size_t ws_bytes, csa2_stream_t stream) {
    (void)workspace;
    (void)ws_bytes;
    clear_error();
    CSA2_REQUIRE(B >= 0 && T >= 0 && N >= 0, "build_pool: negative shape");
    CSA2_REQUIRE(G == CSA2_POOL_BLOCK, "build_pool: G must be 8");
    CSA2_REQUIRE(P >= 1 && P <= CSA2_MAX_POOL, "build_pool: P=%d not in [1,2048]", P);
    if ((int64_t)B * T == 0) return CSA2_OK;
    CSA2_REQUIRE(scores && kv_len && pool_blocks, "build_pool: null pointer");
    CSA2_REQUIRE(aligned(scores, 4) && aligned(pool_blocks, 4), "build_pool: misaligned pointer");
    TopkArgs a = {};
    a.loader = LOAD_BLOCKMAX;
    a.rows = (int64_t)B * T;
    a.M = N;
    a.scores = scores;
    a.kv_len = kv_len;
    a.K = P;
    a.out = pool_blocks;
    return launch_topk(a, (N + 7) / 8, stream_of(stream));
}

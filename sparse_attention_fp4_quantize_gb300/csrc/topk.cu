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
// order-preserving uint32 keys and selects the slice's own Top-K with four
// 8-bit radix passes that need only CTA barriers.  Ranked by (score desc,
// position asc), every member of the row's Top-K is in its slice's Top-K, so
// CTA 0 then gathers the C candidate lists through distributed shared memory
// (one cluster exchange) and runs the same selection on them.  Ties at the
// K-th value go to the lowest positions.  Only hardware barriers are used:
// no flag spinning.
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
    int region;              // words of the key region (>= chunk, >= 2*C*K when C > 1)
};

__device__ __forceinline__ int64_t row_len(const TopkArgs &a, int64_t row) {
    if (a.loader == LOAD_REINDEX) return a.M;
    int64_t len = a.kv_len ? (int64_t)a.kv_len[row] : a.M;
    len = len < a.M ? len : a.M;
    len = len > 0 ? len : 0;
    if (a.loader == LOAD_BLOCKMAX) return (len + 7) / 8;
    return len;
}

// Radix select over keys[0, n) in shared memory: T = the K-th largest key and
// kk = how many keys equal to T are taken (every key > T is taken).  With
// fewer than K keys, or when the K-th largest is the invalid key 0, the result
// is T = 0, kk = 0: take every valid key.
__device__ void block_select(const uint32_t *keys, int n, int K, uint32_t *hist, uint32_t *wsum, uint32_t *bc,
                             uint32_t &T_out, uint32_t &kk_out) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (n < K) {
        T_out = 0;
        kk_out = 0;
        return;
    }
    uint32_t prefix = 0, pmask = 0, kk = (uint32_t)K;
    for (int pass = 0; pass < 4; ++pass) {
        const int shift = 24 - 8 * pass;
        if (tid < 256) hist[tid] = 0;
        __syncthreads();
        for (int base = 0; base < n; base += kThreads) {
            const int i = base + tid;
            uint32_t d = 0x100;  // not participating
            if (i < n) {
                const uint32_t k = keys[i];
                if ((k & pmask) == prefix) d = (k >> shift) & 0xFF;
            }
            const uint32_t peers = __match_any_sync(0xFFFFFFFFu, d);
            if (d != 0x100 && lane == __ffs(peers) - 1) atomicAdd(&hist[d], __popc(peers));
        }
        __syncthreads();
        if (tid < 256) {
            // inclusive suffix sums S[b] = sum_{b' >= b} hist[b'] (warps 0..7 cover 32 bins each)
            uint32_t sfx = hist[tid];
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const uint32_t y = __shfl_down_sync(0xFFFFFFFFu, sfx, off);
                if (lane + off < 32) sfx += y;
            }
            if (lane == 0) wsum[warp] = sfx;
        }
        __syncthreads();
        if (tid < 256) {
            uint32_t hi = 0;
            for (int w2 = warp + 1; w2 < 8; ++w2) hi += wsum[w2];
            uint32_t sfx = hist[tid];
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const uint32_t y = __shfl_down_sync(0xFFFFFFFFu, sfx, off);
                if (lane + off < 32) sfx += y;
            }
            sfx += hi;
            uint32_t nxt = __shfl_down_sync(0xFFFFFFFFu, sfx, 1);
            if (lane == 31) nxt = hi;
            if (sfx >= kk && nxt < kk) {
                bc[0] = (uint32_t)tid;
                bc[1] = nxt;
            }
        }
        __syncthreads();
        const uint32_t d = bc[0];
        kk -= bc[1];
        prefix |= d << shift;
        pmask |= 0xFFu << shift;
        __syncthreads();   // bc and hist are rewritten in the next pass
    }
    T_out = prefix;
    kk_out = prefix == 0 ? 0u : kk;
}

// Sum over the warps before this one of a per-warp value (lane 0 of each warp
// provides it); also returns the total.  `scratch` holds kWarps words.
__device__ __forceinline__ uint32_t warp_prefix(uint32_t v, uint32_t *scratch, uint32_t *total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) scratch[warp] = v;
    __syncthreads();
    uint32_t before = 0, all = 0;
#pragma unroll
    for (int w2 = 0; w2 < kWarps; ++w2) {
        const uint32_t x = scratch[w2];
        before += (w2 < warp) ? x : 0u;
        all += x;
    }
    *total = all;
    __syncthreads();  // scratch may be reused right after
    return before;
}

// Position-ordered compaction of the selected keys of keys[0, n): a key is
// selected if it is > T, or == T (T != 0) and among the first kk such keys.
// Warp w owns a contiguous run of positions and its lanes read consecutive
// words; ballots give the order inside a warp.  emit(i, slot) is called for
// every selected position i with its output slot; returns the number selected.
template <typename Emit>
__device__ int block_compact(const uint32_t *keys, int n, uint32_t T, uint32_t kk, uint32_t *scratch, Emit emit) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint32_t lt = (1u << lane) - 1u;
    int R = (n + kWarps - 1) / kWarps;
    R = (R + 31) & ~31;
    const int w0 = min(n, warp * R), w1 = min(n, w0 + R);
    uint32_t eq = 0;
    if (T != 0)
        for (int base = w0; base < w1; base += 32) {
            const int i = base + lane;
            eq += __popc(__ballot_sync(0xFFFFFFFFu, i < w1 && keys[i] == T));
        }
    uint32_t eq_total;
    const uint32_t eq_before = warp_prefix(eq, scratch, &eq_total);
    uint32_t sel = 0, tie = eq_before;
    for (int base = w0; base < w1; base += 32) {
        const int i = base + lane;
        const uint32_t k = i < w1 ? keys[i] : 0u;
        const bool is_eq = i < w1 && T != 0 && k == T;
        const uint32_t be = __ballot_sync(0xFFFFFFFFu, is_eq);
        const bool take = (i < w1 && k > T) || (is_eq && tie + __popc(be & lt) < kk);
        sel += __popc(__ballot_sync(0xFFFFFFFFu, take));
        tie += __popc(be);
    }
    uint32_t sel_total;
    uint32_t slot = warp_prefix(sel, scratch, &sel_total);
    tie = eq_before;
    for (int base = w0; base < w1; base += 32) {
        const int i = base + lane;
        const uint32_t k = i < w1 ? keys[i] : 0u;
        const bool is_eq = i < w1 && T != 0 && k == T;
        const uint32_t be = __ballot_sync(0xFFFFFFFFu, is_eq);
        const bool take = (i < w1 && k > T) || (is_eq && tie + __popc(be & lt) < kk);
        const uint32_t bs = __ballot_sync(0xFFFFFFFFu, take);
        if (take) emit(i, slot + __popc(bs & lt));
        slot += __popc(bs);
        tie += __popc(be);
    }
    return (int)sel_total;
}

__device__ __forceinline__ int32_t out_id(const TopkArgs &a, int64_t row, int64_t li) {
    if (a.loader == LOAD_REINDEX) return (int32_t)((int64_t)__ldg(a.pool + row * a.P + li / 8) * 8 + (li & 7));
    return (int32_t)li;
}

__global__ void __launch_bounds__(kThreads) topk_radix_kernel(TopkArgs a) {
    extern __shared__ uint32_t dyn[];
    __shared__ uint32_t hist[256];
    __shared__ uint32_t wsum[8];
    __shared__ uint32_t bc[4];
    __shared__ uint32_t scan[kWarps + 1];
    __shared__ int lcount;

    cg::cluster_group cluster = cg::this_cluster();
    const int cta = (int)cluster.block_rank();
    const int C = a.csize;
    const int64_t row = blockIdx.x / C;
    const int tid = threadIdx.x;
    const int K = a.K;

    // shared memory: [0, region) keys of this slice (later CTA 0's gathered
    // candidates), then K local candidate keys and K local ids
    uint32_t *keys = dyn;
    uint32_t *lkey = dyn + a.region;
    int32_t *lid = reinterpret_cast<int32_t *>(lkey + K);

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
                const float4 x = __ldg(reinterpret_cast<const float4 *>(srow + j0));
                const float4 y = __ldg(reinterpret_cast<const float4 *>(srow + j0) + 1);
                m = fmaxf(fmaxf(fmaxf(x.x, x.y), fmaxf(x.z, x.w)), fmaxf(fmaxf(y.x, y.y), fmaxf(y.z, y.w)));
            } else {
                for (int64_t j = j0; j < j0 + 8 && j < len; ++j) m = fmaxf(m, __ldg(srow + j));
            }
            keys[i] = score_key(m);
        }
    } else {
        const bool vec = ((a.M & 3) == 0) && ((reinterpret_cast<uintptr_t>(a.scores) & 15) == 0);
        const int n4 = vec ? (n & ~3) : 0;
        for (int i = 4 * tid; i < n4; i += 4 * kThreads) {
            const float4 x = __ldg(reinterpret_cast<const float4 *>(srow + beg + i));
            keys[i] = score_key(x.x);
            keys[i + 1] = score_key(x.y);
            keys[i + 2] = score_key(x.z);
            keys[i + 3] = score_key(x.w);
        }
        for (int i = n4 + tid; i < n; i += kThreads) keys[i] = score_key(__ldg(srow + beg + i));
        if (a.loader == LOAD_REINDEX) {
            __syncthreads();
            const int32_t *prow = a.pool + row * a.P;
            for (int i = tid; i < n; i += kThreads)
                if (__ldg(prow + (beg + i) / 8) < 0) keys[i] = 0;
        }
    }
    __syncthreads();

    // ---------------------------------------------------------------- this slice's Top-K
    uint32_t T, kk;
    block_select(keys, n, K, hist, wsum, bc, T, kk);
    int32_t *orow = a.out + row * (int64_t)K;
    if (C == 1) {
        const int total = block_compact(keys, n, T, kk, scan, [&](int i, uint32_t slot) {
            orow[slot] = out_id(a, row, beg + i);
        });
        for (int s2 = total + tid; s2 < K; s2 += kThreads) orow[s2] = -1;
        return;
    }
    const int total = block_compact(keys, n, T, kk, scan, [&](int i, uint32_t slot) {
        lkey[slot] = keys[i];
        lid[slot] = (int32_t)(beg + i);
    });
    if (tid == 0) lcount = total;
    cluster.sync();   // every CTA's candidate list is complete

    // ---------------------------------------------------------------- CTA 0 merges the lists
    int ncand = 0;
    if (cta == 0) {
        int off = 0;
        for (int c = 0; c < C; ++c) {
            const int cnt = *cluster.map_shared_rank(&lcount, c);
            const uint32_t *rk = cluster.map_shared_rank(lkey, c);
            const int32_t *ri = cluster.map_shared_rank(lid, c);
            for (int i = tid; i < cnt; i += kThreads) {
                keys[off + i] = rk[i];                                   // gathered keys
                reinterpret_cast<int32_t *>(keys + a.region / 2)[off + i] = ri[i];  // gathered ids
            }
            off += cnt;
        }
        ncand = off;
    }
    cluster.sync();   // remote lists read; the other CTAs may leave
    if (cta != 0) return;
    __syncthreads();
    uint32_t T2, kk2;
    block_select(keys, ncand, K, hist, wsum, bc, T2, kk2);
    const int32_t *gid = reinterpret_cast<const int32_t *>(keys + a.region / 2);
    const int total2 = block_compact(keys, ncand, T2, kk2, scan, [&](int i, uint32_t slot) {
        orow[slot] = out_id(a, row, gid[i]);
    });
    for (int s2 = total2 + tid; s2 < K; s2 += kThreads) orow[s2] = -1;
}

csa2_status launch_topk(const TopkArgs &in, int64_t Lmax, cudaStream_t stream) {
    TopkArgs a = in;
    if (a.rows == 0) return CSA2_OK;
    const int sms = num_sms();
    const size_t smem_cap = 220 * 1024;
    auto chunk_for = [&](int c) { int64_t ch = (Lmax + c - 1) / c; return (ch + 3) & ~int64_t(3); };
    auto smem_for = [&](int c) {
        int64_t region = chunk_for(c);
        if (c > 1 && region < 2 * (int64_t)c * a.K) region = 2 * (int64_t)c * a.K;
        return (size_t)(region + 2 * (int64_t)a.K) * sizeof(uint32_t);
    };
    int C = 1;
    while (C < kMaxCluster && a.rows * C * 2 <= sms) C *= 2;
    while (C > 1 && chunk_for(C) < 1024) C /= 2;
    while (C < kMaxCluster && (chunk_for(C) > kMaxKeysPerCta || smem_for(C) > smem_cap)) C *= 2;
    if (chunk_for(C) > kMaxKeysPerCta || smem_for(C) > smem_cap) {
        set_error("topk: a row of %lld candidates with K=%d does not fit %d CTAs", (long long)Lmax, a.K, kMaxCluster);
        return CSA2_ERR_UNSUPPORTED;
    }
    int64_t chunk = chunk_for(C);
    if (chunk < 4) chunk = 4;
    a.chunk = (int)chunk;
    a.csize = C;
    int64_t region = chunk;
    if (C > 1 && region < 2 * (int64_t)C * a.K) region = 2 * (int64_t)C * a.K;
    a.region = (int)((region + 1) & ~int64_t(1));
    const size_t smem = (size_t)(a.region + 2 * (int64_t)a.K) * sizeof(uint32_t);
    static bool smem_set[64];
    CSA2_CUDA_CALL(ensure_smem_limit((const void *)topk_radix_kernel, (int)smem_cap, smem_set), "topk: smem attribute");
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

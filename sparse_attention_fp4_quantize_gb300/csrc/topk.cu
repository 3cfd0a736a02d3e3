// csa2_topk, csa2_build_pool and the fused decode indexer csa2_index_topk:
// per-row Top-K by radix select.
// Sources: "DeepSeek-V4.1-Flash：把 KV Cache 压缩到极限的百万上下文 MoE", CSA2
// section (Top-512 in every layer) and "Hierarchical Sparse Indexer" (a pool
// of at most 2048 blocks x 8 positions built from block scores);
// "552B参数干掉1.6T：DeepSeek V4.1 Flash技术深度解析", DeepSelect paragraph (the
// Top-K kernel of the sparse attention).
//
// Design.  A row is split over a thread-block cluster of C CTAs (C = 1, 2, 4
// or 8).  Each CTA reads its slice of the row from HBM once and keeps it in
// shared memory as order-preserving uint32 keys.  The K-th largest key of the
// row is then found by a radix select over the whole cluster: for each digit
// (bits 31..21, 20..10, 9..0) every CTA histograms its slice into 2048 fine
// and 64 coarse bins and pushes its coarse bins into every CTA; after one
// cluster barrier every warp of every CTA locates the boundary bin itself
// from the coarse bins and the 32 fine bins of the boundary coarse bin, read
// from each CTA through distributed shared memory, so nothing waits for
// another CTA's answer.  A digit ends the search early when the boundary bin
// is taken whole (random float scores need two digits).  The selection is
// then compacted in position order across the cluster: every warp pushes its
// counts above and at the threshold into every CTA, one more barrier lets
// each warp sum the counts before it, and each CTA writes its own ids straight
// to the output.  Ties at the K-th value go to the lowest positions.  Only
// hardware barriers are used: no flag spinning.
//
// The fused indexer scores its slice of candidates (FP8 keys, the decode
// scorer's MMA tiling) straight into the same shared-memory keys, so the
// scores of a decode row never reach HBM.
#include <cooperative_groups.h>

#include "common.cuh"

namespace cg = cooperative_groups;

namespace csa2 {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kBins = 2048;    // widest digit: 11 bits
constexpr int kCoarse = 64;    // coarse bin = 32 fine bins
constexpr int kDigits = 3;     // bits 31..21, 20..10, 9..0
constexpr int kMaxCluster = 8;
constexpr int kMaxKeysPerCta = 49152;  // 192 KB of keys
constexpr int kSmemCap = 192 * 1024;   // dynamic shared memory ceiling (static use is ~33 KB)
static_assert(kBins == 4 * kThreads, "each thread owns one uint4 of fine bins");
static_assert(kCoarse == kThreads / 8, "eight threads make one coarse bin");
static_assert(kWarps <= 32, "one lane per warp in the count exchange");

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
    int chunk;               // keys per CTA (multiple of 4)
};

__device__ __forceinline__ int32_t out_id(const TopkArgs &a, int64_t row, int64_t li) {
    if (a.loader == LOAD_REINDEX) return (int32_t)((int64_t)__ldg(a.pool + row * a.P + li / 8) * 8 + (li & 7));
    return (int32_t)li;
}

__device__ __forceinline__ uint32_t warp_suffix_sum(uint32_t v) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const uint32_t y = __shfl_down_sync(0xFFFFFFFFu, v, off);
        if (lane + off < 32) v += y;
    }
    return v;
}

struct Boundary {
    uint32_t bin, above, inbin;
};

// The bin b of the cluster-wide histogram with S(b) >= kk > S(b+1), where S(b)
// counts the keys in bins >= b; computed by one warp on its own.
// `coarse` holds every CTA's coarse bins ([C][64], pushed here before the
// cluster barrier); the fine bins are read from each CTA.
template <int C>
__device__ __forceinline__ Boundary find_boundary(cg::cluster_group &cluster, const uint32_t *fine,
                                                  const uint32_t (*coarse)[kCoarse], uint32_t kk) {
    const int lane = threadIdx.x & 31;
    uint2 cs = make_uint2(0u, 0u);
#pragma unroll
    for (int c = 0; c < C; ++c) {
        const uint2 v = reinterpret_cast<const uint2 *>(coarse[c])[lane];
        cs.x += v.x;
        cs.y += v.y;
    }
    const uint32_t c0 = warp_suffix_sum(cs.x + cs.y);  // S over coarse bins >= 2 lane
    const uint32_t c1 = c0 - cs.x, c2 = c1 - cs.y;
    int sub = -1;
    uint32_t cabove = 0u;
    if (c1 >= kk && c2 < kk) { sub = 1; cabove = c2; }
    else if (c0 >= kk && c1 < kk) { sub = 0; cabove = c1; }
    const int cl = __ffs(__ballot_sync(0xFFFFFFFFu, sub >= 0)) - 1;
    const uint32_t cb = 2u * cl + (uint32_t)__shfl_sync(0xFFFFFFFFu, sub, cl);
    cabove = __shfl_sync(0xFFFFFFFFu, cabove, cl);
    uint32_t f = 0u;
#pragma unroll
    for (int c = 0; c < C; ++c) {
        const uint32_t *rf = C > 1 ? cluster.map_shared_rank(fine, c) : fine;
        f += rf[cb * 32u + lane];
    }
    const uint32_t f0 = warp_suffix_sum(f) + cabove;  // S(32 cb + lane)
    const uint32_t f1 = f0 - f;
    const int fl = __ffs(__ballot_sync(0xFFFFFFFFu, f0 >= kk && f1 < kk)) - 1;
    Boundary r;
    r.bin = cb * 32u + (uint32_t)fl;
    r.above = __shfl_sync(0xFFFFFFFFu, f1, fl);
    r.inbin = __shfl_sync(0xFFFFFFFFu, f, fl);
    return r;
}

// Shared memory of the cluster-wide selection.
template <int C>
struct SelSmem {
    uint32_t (*fine)[kBins];            // [kDigits][kBins] this CTA's histogram of each digit
    uint32_t (*coarse)[C][kCoarse];     // [kDigits][C][kCoarse] every CTA's coarse bins, pushed
    uint32_t (*wcnt)[2][kWarps];        // [C][2][kWarps] every CTA's per-warp (greater, equal) counts
};

// Cluster-wide radix select over every CTA's keys[0, 4 nm4) (zero-padded).  L
// is the row's candidate count: with at most K of them every valid key is
// taken.  Result: every key > T is selected, plus the first kk keys equal to
// T (T != 0).  The fine histograms must be zero on entry; they are left
// dirty (reset_fine before another selection).  Contains cluster barriers:
// every thread of every CTA of the cluster calls it.
template <int C>
__device__ void cluster_select(cg::cluster_group &cluster, int cta, const SelSmem<C> &sm, const uint32_t *keys,
                               int nm4, int64_t L, int K, uint32_t &T_out, uint32_t &kk_out) {
    const int tid = threadIdx.x, lane = tid & 31;
    uint32_t T = 0u, kk = 0u;
    if (L > K) {
        const uint4 *k4 = reinterpret_cast<const uint4 *>(keys);
        uint32_t prefix = 0u, pmask = 0u;
        kk = (uint32_t)K;
#pragma unroll 1
        for (int d = 0; d < kDigits; ++d) {
            const int shift = d == 0 ? 21 : (d == 1 ? 10 : 0);
            const uint32_t dmask = d == 2 ? 0x3FFu : 0x7FFu;
            uint32_t *h = sm.fine[d];
#pragma unroll 4
            for (int j = tid; j < nm4; j += kThreads) {
                const uint4 v = k4[j];
                if (v.x != 0u && (v.x & pmask) == prefix) atomicAdd(&h[(v.x >> shift) & dmask], 1u);
                if (v.y != 0u && (v.y & pmask) == prefix) atomicAdd(&h[(v.y >> shift) & dmask], 1u);
                if (v.z != 0u && (v.z & pmask) == prefix) atomicAdd(&h[(v.z >> shift) & dmask], 1u);
                if (v.w != 0u && (v.w & pmask) == prefix) atomicAdd(&h[(v.w >> shift) & dmask], 1u);
            }
            __syncthreads();
            {   // coarse bins (eight threads' fine bins each), pushed into every CTA
                const uint4 q = reinterpret_cast<const uint4 *>(h)[tid];
                uint32_t s = q.x + q.y + q.z + q.w;
                s += __shfl_xor_sync(0xFFFFFFFFu, s, 1);
                s += __shfl_xor_sync(0xFFFFFFFFu, s, 2);
                s += __shfl_xor_sync(0xFFFFFFFFu, s, 4);
                if ((tid & 7) == 0) {
#pragma unroll
                    for (int c = 0; c < C; ++c)
                        *(C > 1 ? cluster.map_shared_rank(&sm.coarse[d][cta][tid >> 3], c) : &sm.coarse[d][cta][tid >> 3]) = s;
                }
            }
            if (C > 1) cluster.sync(); else __syncthreads();  // every slice's histograms are complete
            if (d == 0) {  // at most K valid keys: take them all
                uint32_t tot = 0u;
#pragma unroll
                for (int c = 0; c < C; ++c) {
                    const uint2 v = reinterpret_cast<const uint2 *>(sm.coarse[0][c])[lane];
                    tot += v.x + v.y;
                }
                if (__reduce_add_sync(0xFFFFFFFFu, tot) <= (uint32_t)K) {
                    kk = 0u;
                    break;
                }
            }
            const Boundary bd = find_boundary<C>(cluster, h, sm.coarse[d], kk);
            kk -= bd.above;
            prefix |= bd.bin << shift;
            pmask |= dmask << shift;
            if (bd.inbin == kk) {  // the boundary bin is taken whole: every key >= prefix
                T = prefix - 1u;   // prefix >= 2^21 here: a bin that holds valid keys is never 0
                kk = 0u;
                break;
            }
            if (d == kDigits - 1) T = prefix;
        }
    }
    T_out = T;
    kk_out = kk;
}

// Zero the fine histograms for another selection (after a cluster barrier
// that follows every CTA's last read of them); the caller syncs the CTA.
template <int C>
__device__ __forceinline__ void reset_fine(const SelSmem<C> &sm) {
#pragma unroll
    for (int d = 0; d < kDigits; ++d) reinterpret_cast<uint4 *>(sm.fine[d])[threadIdx.x] = make_uint4(0u, 0u, 0u, 0u);
}

// Position-ordered compaction of the selection (T, kk) across the cluster:
// orow[slot] = id(i) for every selected slice position i, slots in row
// position order; the last CTA pads the row to K with -1.  Warp w owns a
// contiguous run of the slice; ballots order its lanes.  One cluster barrier
// (after it no CTA reads another's shared memory).
template <int C, typename IdFn>
__device__ void cluster_compact(cg::cluster_group &cluster, int cta, const SelSmem<C> &sm, const uint32_t *keys,
                                int nm, uint32_t T, uint32_t kk, int K, int32_t *orow, IdFn id) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    int R = (nm + kWarps - 1) / kWarps;
    R = (R + 31) & ~31;
    const int w0 = min(nm, warp * R), w1 = min(nm, w0 + R);
    uint32_t gt = 0, eq = 0;
    for (int base = w0; base < w1; base += 32) {
        const int i = base + lane;
        const uint32_t k = i < w1 ? keys[i] : 0u;
        gt += __popc(__ballot_sync(0xFFFFFFFFu, k > T));
        eq += __popc(__ballot_sync(0xFFFFFFFFu, T != 0u && k == T));
    }
    if (lane == 0) {   // publish this warp's counts in every CTA
#pragma unroll
        for (int c = 0; c < C; ++c) {
            uint32_t *dst = C > 1 ? cluster.map_shared_rank(&sm.wcnt[cta][0][warp], c) : &sm.wcnt[cta][0][warp];
            dst[0] = gt;
            dst[kWarps] = eq;
        }
    }
    if (C > 1) cluster.sync(); else __syncthreads();
    uint32_t bg = 0u, be_ = 0u, tg = 0u, te = 0u;     // (before this warp, in the row) counts
#pragma unroll
    for (int c = 0; c < C; ++c) {
        const uint32_t vg = lane < kWarps ? sm.wcnt[c][0][lane] : 0u, ve = lane < kWarps ? sm.wcnt[c][1][lane] : 0u;
        const bool before = c < cta || (c == cta && lane < warp);
        bg += before ? vg : 0u;
        be_ += before ? ve : 0u;
        tg += vg;
        te += ve;
    }
    const uint32_t gt_before = __reduce_add_sync(0xFFFFFFFFu, bg), eq_before = __reduce_add_sync(0xFFFFFFFFu, be_);
    const uint32_t lt = (1u << lane) - 1u;
    uint32_t tie = eq_before;
    uint32_t slot = gt_before + min(kk, tie);
    for (int base = w0; base < w1; base += 32) {
        const int i = base + lane;
        const uint32_t k = i < w1 ? keys[i] : 0u;
        const bool is_eq = T != 0u && k == T;
        const uint32_t bq = __ballot_sync(0xFFFFFFFFu, is_eq);
        const bool take = k > T || (is_eq && tie + __popc(bq & lt) < kk);
        const uint32_t bs = __ballot_sync(0xFFFFFFFFu, take);
        if (take) orow[slot + __popc(bs & lt)] = id(i);
        slot += __popc(bs);
        tie += __popc(bq);
    }
    if (cta == C - 1) {
        const uint32_t gt_total = __reduce_add_sync(0xFFFFFFFFu, tg), eq_total = __reduce_add_sync(0xFFFFFFFFu, te);
        const int total = (int)(gt_total + min(kk, eq_total));
        for (int s2 = total + tid; s2 < K; s2 += kThreads) orow[s2] = -1;
    }
}

template <int C>
__global__ void __launch_bounds__(kThreads) topk_radix_kernel(TopkArgs a) {
    extern __shared__ __align__(16) uint32_t keys[];          // this CTA's slice (+ zero padding to 4)
    __shared__ __align__(16) uint32_t fine[kDigits][kBins];
    __shared__ __align__(16) uint32_t coarse[kDigits][C][kCoarse];
    __shared__ uint32_t wcnt[C][2][kWarps];
    const SelSmem<C> sm = {fine, coarse, wcnt};

    cg::cluster_group cluster = cg::this_cluster();
    const int cta = C > 1 ? (int)cluster.block_rank() : 0;
    const int64_t row = blockIdx.x / C;
    const int tid = threadIdx.x;
    const int K = a.K;
    const int64_t beg = (int64_t)cta * a.chunk;

    // Issue the score loads before the row length is known: the slice is
    // clipped to the row's M entries, positions at or past the length masked.
    int64_t Mrow = a.M;
    if (a.loader == LOAD_BLOCKMAX) Mrow = (a.M + 7) / 8;
    int nm = 0;
    if (beg < Mrow) nm = (int)((Mrow - beg) < a.chunk ? (Mrow - beg) : a.chunk);
    const int nm4 = (nm + 3) >> 2;
    reset_fine(sm);
    // cluster barrier, first half: this CTA runs (its shared memory may be written once
    // every CTA has arrived: the wait follows the load)
    if (C > 1) asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
    pdl_wait();   // the set-up above overlaps the previous kernel's tail

    // ---------------------------------------------------------------- load
    int64_t L;
    const float *srow = a.scores + row * a.M;
    if (a.loader == LOAD_BLOCKMAX) {
        const int64_t len = a.kv_len ? max((int64_t)0, min((int64_t)a.kv_len[row], a.M)) : a.M;
        L = (len + 7) / 8;
        const bool vec = ((a.M & 3) == 0) && ((reinterpret_cast<uintptr_t>(a.scores) & 15) == 0);
#pragma unroll 4
        for (int i = tid; i < nm; i += kThreads) {
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
        const int32_t *prow = a.pool + row * a.P;
        const int q4 = vec ? (nm >> 2) : 0;
        const int64_t len = (a.loader == LOAD_SCORES && a.kv_len) ? (int64_t)a.kv_len[row] : a.M;
        L = len < a.M ? (len > 0 ? len : 0) : a.M;
        const int nv = (int)(L - beg < 0 ? 0 : (L - beg < nm ? L - beg : nm));  // valid positions of this slice
#pragma unroll 4
        for (int j = tid; j < q4; j += kThreads) {
            const float4 x = __ldg(reinterpret_cast<const float4 *>(srow + beg) + j);
            uint4 k = make_uint4(score_key(x.x), score_key(x.y), score_key(x.z), score_key(x.w));
            // the four positions share one pool block (beg and 4j are multiples of 4)
            if (a.loader == LOAD_REINDEX && __ldg(prow + (beg + 4 * j) / 8) < 0) k = make_uint4(0u, 0u, 0u, 0u);
            if (4 * j + 3 >= nv) {
                if (4 * j >= nv) k.x = 0u;
                if (4 * j + 1 >= nv) k.y = 0u;
                if (4 * j + 2 >= nv) k.z = 0u;
                k.w = 0u;
            }
            reinterpret_cast<uint4 *>(keys)[j] = k;
        }
        for (int i = 4 * q4 + tid; i < nm; i += kThreads) {
            uint32_t k = i < nv ? score_key(__ldg(srow + beg + i)) : 0u;
            if (a.loader == LOAD_REINDEX && __ldg(prow + (beg + i) / 8) < 0) k = 0u;
            keys[i] = k;
        }
    }
    if (tid < 4 * nm4 - nm) keys[nm + tid] = 0u;  // pad to a multiple of 4 with the invalid key
    __syncthreads();
    if (C > 1) asm volatile("barrier.cluster.wait.aligned;" ::: "memory");

    uint32_t T, kk;
    cluster_select<C>(cluster, cta, sm, keys, nm4, L, K, T, kk);
    pdl_launch_dependents();   // the next kernel may launch during the compaction
    cluster_compact<C>(cluster, cta, sm, keys, nm, T, kk, K, a.out + row * (int64_t)K,
                       [&](int i) { return out_id(a, row, beg + i); });
}

// ---------------------------------------------------------------------------
// Fused decode indexer: scores (FP8 keys and query, the same MMA tiling as the
// decode scorer of csa2_index_score) go straight into the cluster's shared
// memory as order-preserving keys, and the same cluster selection picks the
// Top-K -- and for a Full layer optionally the pool of Top-P_out 8-position
// blocks from the block maxima -- without writing the scores to HBM.
struct FusedArgs {
    int mode;
    int64_t rows;             // B * T query rows
    int T;
    int64_t N;                // entries per sequence
    int64_t M;                // candidates per row: N (Full) or 8 P (Reindex)
    const uint8_t *q;         // FP8 [rows, 4, 64]
    const float *w;           // [rows, 4]
    const uint8_t *k;         // FP8 [B, N, 64]
    const int32_t *kv_len;    // [rows]
    const int32_t *pool_in;   // Reindex [rows, P]
    int P;
    int K;
    int32_t *idx;             // [rows, K]
    int32_t *pool_out;        // Full, optional [rows, P_out]
    int P_out;
    uint32_t *err_flag;
    int chunk;                // candidates per CTA (multiple of 128)
};

template <int C>
__global__ void __launch_bounds__(kThreads) index_topk_kernel(FusedArgs a) {
    extern __shared__ __align__(16) uint32_t keys[];          // [chunk] scores as keys, then [chunk/8] block keys
    __shared__ __align__(16) uint32_t fine[kDigits][kBins];
    __shared__ __align__(16) uint32_t coarse[kDigits][C][kCoarse];
    __shared__ uint32_t wcnt[C][2][kWarps];
    const SelSmem<C> sm = {fine, coarse, wcnt};
    uint32_t *bkeys = keys + a.chunk;

    cg::cluster_group cluster = cg::this_cluster();
    const int cta = C > 1 ? (int)cluster.block_rank() : 0;
    const int64_t row = blockIdx.x / C;
    const int64_t b = row / a.T;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, t4 = lane & 3;
    const bool full = a.mode == CSA2_MODE_FULL;
    reset_fine(sm);
    if (C > 1) asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
    pdl_wait();

    // ---------------------------------------------------------------- score this slice
    int64_t len = a.kv_len[row];
    len = len < a.N ? (len > 0 ? len : 0) : a.N;
    // Full: the row's len valid positions are shared evenly by the cluster (slices of a
    // multiple of 128, in position order); Reindex: the 8P pool candidates, chunk by chunk
    int64_t beg, share;
    if (full) {
        share = (((len + C - 1) / C) + 127) & ~int64_t(127);
        if (share > a.chunk) share = a.chunk;   // cannot happen: len <= M
    } else {
        share = a.chunk;
    }
    beg = (int64_t)cta * share;
    const int64_t lim = full ? len : a.M;
    int nm = 0;
    if (beg < lim) nm = (int)((lim - beg) < share ? (lim - beg) : share);
    const int64_t nblocks_n = (a.N + 7) / 8;
    const uint4 q8 = (g < 4) ? __ldg(reinterpret_cast<const uint4 *>(a.q + (row * 4 + g) * 64 + 16 * t4))
                             : make_uint4(0, 0, 0, 0);
    const float w0 = (t4 < 2) ? a.w[row * 4 + 2 * t4] : 0.f;
    const float w1 = (t4 < 2) ? a.w[row * 4 + 2 * t4 + 1] : 0.f;
    const int nchunks = (nm + 127) / 128;
    // Reindex: a chunk's 16 pool block ids, checked (lanes 0-15 hold them)
    auto pool_ids = [&](int cb, int l) -> int32_t {
        const int64_t pidx = (beg + (int64_t)cb * 128) / 8 + l;
        if (cb >= nchunks || pidx >= a.P) return -1;
        int64_t blk = a.pool_in[row * a.P + pidx];
        if (blk < -1 || blk >= nblocks_n) {
            flag_error(a.err_flag, CSA2_FLAG_BAD_POOL);
            blk = -1;
        }
        return (int32_t)blk;
    };
    // Reindex: the ids of this warp's first two chunks are loaded together (lanes
    // 0-15: chunk warp, lanes 16-31: chunk warp + kWarps), off the chain of
    // dependent loads of each chunk.  The load is only issued here: the first
    // key loads go out at the positions an identity pool gives (pool slot p
    // holding block p, as a Full layer writes it when every block of the row
    // fits), and the ids are checked once those loads are in flight.
    const int pre_cb = warp + (lane >= 16 ? kWarps : 0);
    const int64_t pre_pidx = (beg + (int64_t)pre_cb * 128) / 8 + (lane & 15);
    const bool pre_in = !full && pre_cb < nchunks && pre_pidx < a.P;
    const int64_t pre_raw = pre_in ? (int64_t)a.pool_in[row * a.P + pre_pidx] : -1;
    int32_t pre_blk = -1;
    bool spec_ok = false;   // the warp's two chunks see an identity pool: the identity loads stand
    // Reindex: the slice's checked pool block ids are kept in shared memory (the
    // block-key area, unused without a pool to build), for the output ids
    int32_t *sBlk = reinterpret_cast<int32_t *>(bkeys);
    auto check_pre = [&]() {   // every lane of the warp
        int64_t blk = pre_raw;
        if (blk < -1 || blk >= nblocks_n) {
            flag_error(a.err_flag, CSA2_FLAG_BAD_POOL);
            blk = -1;
        }
        pre_blk = (int32_t)blk;
        if (pre_in) sBlk[pre_cb * 16 + (lane & 15)] = pre_blk;
        // the identity's positions are this slot's: block p, or no block past the row
        const bool same = !pre_in || blk == pre_pidx || (blk == -1 && pre_pidx * 8 >= len);
        spec_ok = __all_sync(0xFFFFFFFFu, same);
    };
    // A warp scores its chunks (cb = warp, warp + kWarps, ...) in halves of 4
    // groups (64 candidates), software-pipelined over two register buffers:
    // the loads of half k + 1 are in flight while half k is scored.
    const int nhalf = warp < nchunks ? 2 * ((nchunks - warp + kWarps - 1) / kWarps) : 0;
    int32_t chunk_blk = -1;   // Reindex, chunks past the first two: ids reloaded per chunk
    auto load_half = [&](int k, uint4 (&raw)[4][2], bool (&v)[4][2], bool ident) {
        const int it = k >> 1, cb = warp + kWarps * it, i0 = cb * 128 + 64 * (k & 1);
        if (!full && it >= 2 && (k & 1) == 0) {
            chunk_blk = lane < 16 ? pool_ids(cb, lane) : -1;
            if (lane < 16 && cb < nchunks) sBlk[cb * 16 + lane] = chunk_blk;
        }
        const int32_t ids = it < 2 ? pre_blk : chunk_blk;
        const int base_lane = (it < 2 ? 16 * (it & 1) : 0) + 8 * (k & 1);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                const int i = i0 + 16 * c + g + 8 * r;
                int64_t j;
                if (full || ident) {   // Reindex with an identity pool: candidate beg + i is position beg + i
                    j = beg + i;
                } else {
                    const int32_t blk = __shfl_sync(0xFFFFFFFFu, ids, base_lane + 2 * c + r);
                    j = blk >= 0 ? (int64_t)blk * 8 + g : -1;
                }
                v[c][r] = i < nm && j >= 0 && j < len;
                raw[c][r] = v[c][r] ? __ldg(reinterpret_cast<const uint4 *>(a.k + (b * a.N + j) * 64 + 16 * t4))
                                    : make_uint4(0, 0, 0, 0);
            }
        }
    };
    auto score_half = [&](int k, const uint4 (&raw)[4][2], const bool (&v)[4][2]) {
        const int i0 = (warp + kWarps * (k >> 1)) * 128 + 64 * (k & 1);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
            mma_e4m3_16832(acc, raw[c][0].x, raw[c][1].x, raw[c][0].y, raw[c][1].y, q8.x, q8.y);
            mma_e4m3_16832(acc, raw[c][0].z, raw[c][1].z, raw[c][0].w, raw[c][1].w, q8.z, q8.w);
            float s0 = w0 * fmaxf(acc[0], 0.f) + w1 * fmaxf(acc[1], 0.f);
            float s1 = w0 * fmaxf(acc[2], 0.f) + w1 * fmaxf(acc[3], 0.f);
            s0 += __shfl_xor_sync(0xFFFFFFFFu, s0, 1);
            s1 += __shfl_xor_sync(0xFFFFFFFFu, s1, 1);
            if (t4 == 0) {
                keys[i0 + 16 * c + g] = v[c][0] ? score_key(s0) : 0u;
                keys[i0 + 16 * c + g + 8] = v[c][1] ? score_key(s1) : 0u;
            }
        }
    };
    {
        uint4 ra[4][2], rb[4][2];
        bool va[4][2], vb[4][2];
        if (nhalf > 0) load_half(0, ra, va, !full);
        if (!full) {
            check_pre();
            if (!spec_ok && nhalf > 0) load_half(0, ra, va, false);   // not an identity pool: the real ids
        }
        const bool ident = !full && spec_ok;   // for the warp's first two chunks (k < 4)
        for (int k = 0; k < nhalf; k += 2) {   // nhalf is even
            load_half(k + 1, rb, vb, ident && k + 1 < 4);
            score_half(k, ra, va);
            if (k + 2 < nhalf) load_half(k + 2, ra, va, ident && k + 2 < 4);
            score_half(k + 1, rb, vb);
        }
    }
    __syncthreads();   // keys [0, 128 nchunks) written; the rest of [0, 4 nm4) is never read
    if (C > 1) asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
    const int nm4 = (nm + 3) >> 2;

    // ---------------------------------------------------------------- pool (Full, optional)
    if (a.pool_out && (len + 7) / 8 <= a.P_out) {
        // every block with a valid position is in the pool: this CTA's blocks [beg/8, beg/8 + nb)
        // go to the same slots (the slices are contiguous and 8-aligned), the last CTA pads
        const int nb = (nm + 7) / 8;
        const int64_t b0 = beg / 8, nbt = (len + 7) / 8;
        int32_t *prow = a.pool_out + row * (int64_t)a.P_out;
        for (int ib = tid; ib < nb; ib += kThreads) prow[b0 + ib] = (int32_t)(b0 + ib);
        if (cta == C - 1)
            for (int64_t s2 = nbt + tid; s2 < a.P_out; s2 += kThreads) prow[s2] = -1;
    } else if (a.pool_out) {
        const int nb = (nm + 7) / 8, nb4 = (nb + 3) >> 2;
        for (int ib = tid; ib < 4 * nb4; ib += kThreads) {
            uint32_t m = 0u;
            if (ib < nb) {
#pragma unroll
                for (int u = 0; u < 8; ++u) m = max(m, keys[8 * ib + u]);   // order-preserving keys
            }
            bkeys[ib] = m;
        }
        __syncthreads();
        uint32_t T, kk;
        cluster_select<C>(cluster, cta, sm, bkeys, nb4, (len + 7) / 8, a.P_out, T, kk);
        const int64_t b0 = beg / 8;
        cluster_compact<C>(cluster, cta, sm, bkeys, nb, T, kk, a.P_out, a.pool_out + row * (int64_t)a.P_out,
                           [&](int ib) { return (int32_t)(b0 + ib); });
        reset_fine(sm);
        // no CTA starts the next selection (its pushes) before every CTA is done with this one
        if (C > 1) cluster.sync(); else __syncthreads();
    }

    // ---------------------------------------------------------------- Top-K
    auto global_id = [&](int i) -> int32_t {   // candidate beg + i of the row -> entry position
        if (full) return (int32_t)(beg + i);
        return sBlk[i >> 3] * 8 + (i & 7);      // beg is a multiple of 128
    };
    uint32_t T, kk;
    cluster_select<C>(cluster, cta, sm, keys, nm4, full ? len : a.M, a.K, T, kk);
    pdl_launch_dependents();
    cluster_compact<C>(cluster, cta, sm, keys, nm, T, kk, a.K, a.idx + row * (int64_t)a.K,
                       [&](int i) { return global_id(i); });
}

// Keys per CTA and dynamic shared memory for a split of the rows over C CTAs.
struct TopkPlan {
    int64_t chunk;
    size_t smem;
};

TopkPlan plan_for(int64_t Lmax, int C) {
    TopkPlan p;
    p.chunk = ((Lmax + C - 1) / C + 3) & ~int64_t(3);
    if (p.chunk < 4) p.chunk = 4;
    p.smem = (size_t)p.chunk * sizeof(uint32_t);
    return p;
}

// CTAs per row: enough that a slice fits shared memory, and for rows of more
// than 4096 candidates up to 4 while the grid stays within one CTA per SM
// (wider clusters than 4 measured slower on 152-SM parts).
int cluster_for(int64_t rows, int64_t Lmax, int sms) {
    int C = 1;
    while (C < kMaxCluster && plan_for(Lmax, C).chunk > kMaxKeysPerCta) C *= 2;
    while (C < 4 && plan_for(Lmax, C).chunk > 4096 && rows * C * 2 <= (int64_t)sms) C *= 2;
    return C;
}

csa2_status launch_topk(const TopkArgs &in, int64_t Lmax, cudaStream_t stream) {
    TopkArgs a = in;
    if (a.rows == 0) return CSA2_OK;
    const int C = cluster_for(a.rows, Lmax, num_sms());
    const TopkPlan pl = plan_for(Lmax, C);
    if (pl.chunk > kMaxKeysPerCta || pl.smem > (size_t)kSmemCap) {
        set_error("topk: a row of %lld candidates does not fit %d CTAs", (long long)Lmax, kMaxCluster);
        return CSA2_ERR_UNSUPPORTED;
    }
    a.chunk = (int)pl.chunk;
    const int64_t grid = a.rows * C;
    if (grid > 0x7FFFFFFF) {
        set_error("topk: too many rows");
        return CSA2_ERR_UNSUPPORTED;
    }
    const void *fn = C == 1 ? (const void *)topk_radix_kernel<1>
                   : C == 2 ? (const void *)topk_radix_kernel<2>
                   : C == 4 ? (const void *)topk_radix_kernel<4>
                            : (const void *)topk_radix_kernel<8>;
    static bool smem_set[4][64];
    const int ci = C == 1 ? 0 : (C == 2 ? 1 : (C == 4 ? 2 : 3));
    CSA2_CUDA_CALL(ensure_smem_limit(fn, kSmemCap, smem_set[ci]), "topk: smem attribute");
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = pl.smem;
    cfg.stream = stream;
    // Launched without programmatic serialization: started early behind the
    // indexer, its waiting clusters slowed a decode step by ~8% on GB300.
    // It still lets the next kernel launch early (pdl_launch_dependents).
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    void *args[] = {&a};
    CSA2_CUDA_CALL(cudaLaunchKernelExC(&cfg, fn, args), "topk_radix_kernel launch");
    CSA2_LAUNCH_CHECK("topk_radix_kernel");
    return CSA2_OK;
}

csa2_status launch_index_topk(const FusedArgs &in, cudaStream_t stream) {
    FusedArgs a = in;
    if (a.rows == 0) return CSA2_OK;
    // keys and block keys of a slice: (chunk + chunk/8 + 4) words, chunk a multiple of 128
    auto chunk_for = [&](int c) {
        int64_t ch = ((a.M + c - 1) / c + 127) & ~int64_t(127);
        return ch < 128 ? (int64_t)128 : ch;
    };
    auto smem_for = [&](int c) { return (size_t)(chunk_for(c) + chunk_for(c) / 8 + 4) * sizeof(uint32_t); };
    int C = 1;
    while (C < kMaxCluster && smem_for(C) > (size_t)kSmemCap) C *= 2;
    while (C < kMaxCluster && chunk_for(C) > 2048 && a.rows * C * 2 <= (int64_t)num_sms()) C *= 2;
    const int64_t chunk = chunk_for(C);
    const size_t smem = smem_for(C);
    if (smem > (size_t)kSmemCap) {
        set_error("index_topk: a row of %lld candidates does not fit %d CTAs", (long long)a.M, kMaxCluster);
        return CSA2_ERR_UNSUPPORTED;
    }
    a.chunk = (int)chunk;
    const int64_t grid = a.rows * C;
    if (grid > 0x7FFFFFFF) {
        set_error("index_topk: too many rows");
        return CSA2_ERR_UNSUPPORTED;
    }
    const void *fn = C == 1 ? (const void *)index_topk_kernel<1>
                   : C == 2 ? (const void *)index_topk_kernel<2>
                   : C == 4 ? (const void *)index_topk_kernel<4>
                            : (const void *)index_topk_kernel<8>;
    static bool smem_set[4][64];
    const int ci = C == 1 ? 0 : (C == 2 ? 1 : (C == 4 ? 2 : 3));
    CSA2_CUDA_CALL(ensure_smem_limit(fn, kSmemCap, smem_set[ci]), "index_topk: smem attribute");
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    // programmatic serialization on (measured 1% faster decode steps; unlike the
    // standalone Top-K this kernel follows the attention, whose CTAs it cannot share SMs with)
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1] = pdl_attribute();
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    void *args[] = {&a};
    CSA2_CUDA_CALL(cudaLaunchKernelExC(&cfg, fn, args), "index_topk_kernel launch");
    CSA2_LAUNCH_CHECK("index_topk_kernel");
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

extern "C" csa2_status csa2_index_topk(csa2_mode mode, int B, int T, int64_t N, const void *q_idx, csa2_dtype q_dt,
                                       const float *w, const void *k_idx, csa2_dtype k_dt, const int32_t *kv_len,
                                       const int32_t *pool_blocks, int P, int K, int32_t *idx, int32_t *pool_out,
                                       int P_out, uint32_t *err_flag, csa2_stream_t stream) {
    clear_error();
    CSA2_REQUIRE(mode == CSA2_MODE_FULL || mode == CSA2_MODE_REINDEX || mode == CSA2_MODE_REUSE,
                 "index_topk: bad mode %d", (int)mode);
    if (mode == CSA2_MODE_REUSE) return CSA2_OK;
    CSA2_REQUIRE(B >= 0 && T >= 0 && N >= 0, "index_topk: negative shape");
    CSA2_REQUIRE(q_dt == CSA2_FP8_E4M3 && k_dt == CSA2_FP8_E4M3,
                 "index_topk: FP8 E4M3 indexer only (use csa2_index_score + csa2_topk for bf16)");
    CSA2_REQUIRE(K >= 1 && K <= CSA2_MAX_K, "index_topk: K=%d not in [1,2048]", K);
    if (mode == CSA2_MODE_REINDEX) {
        CSA2_REQUIRE(pool_blocks != nullptr, "index_topk: REINDEX needs pool_blocks");
        CSA2_REQUIRE(P >= 1 && P <= CSA2_MAX_POOL, "index_topk: P=%d not in [1,2048]", P);
        CSA2_REQUIRE(pool_out == nullptr, "index_topk: pool_out is for FULL only");
    } else {
        CSA2_REQUIRE(pool_blocks == nullptr, "index_topk: FULL takes no pool_blocks");
        if (pool_out) CSA2_REQUIRE(P_out >= 1 && P_out <= CSA2_MAX_POOL, "index_topk: P_out=%d not in [1,2048]", P_out);
    }
    if ((int64_t)B * T == 0) return CSA2_OK;
    CSA2_REQUIRE(q_idx && w && k_idx && kv_len && idx, "index_topk: null pointer");
    CSA2_REQUIRE(aligned(q_idx, 16) && aligned(k_idx, 16), "index_topk: q_idx/k_idx must be 16-byte aligned");
    CSA2_REQUIRE(aligned(w, 4) && aligned(kv_len, 4) && aligned(idx, 4) && aligned(pool_out, 4) &&
                     aligned(pool_blocks, 4),
                 "index_topk: misaligned pointer");
    FusedArgs a = {};
    a.mode = (int)mode;
    a.rows = (int64_t)B * T;
    a.T = T;
    a.N = N;
    a.M = (mode == CSA2_MODE_FULL) ? N : (int64_t)P * 8;
    a.q = (const uint8_t *)q_idx;
    a.w = w;
    a.k = (const uint8_t *)k_idx;
    a.kv_len = kv_len;
    a.pool_in = pool_blocks;
    a.P = P;
    a.K = K;
    a.idx = idx;
    a.pool_out = pool_out;
    a.P_out = pool_out ? P_out : 0;
    a.err_flag = err_flag;
    return launch_index_topk(a, stream_of(stream));
}

// csa2_index_topk_dense: Full-mode indexer scoring and Top-K for many query
// tokens per sequence (a prefill chunk) without the [B, T, N] score matrix.
// Sources: "DeepSeek-V4.1-Flash：把 KV Cache 压缩到极限的百万上下文 MoE", section
// "Hierarchical Sparse Indexer——索引成本变常数" (Full layers score every entry;
// Top-512 per query).  The passes below are this library's; the pages only
// state what is selected.
//
// Why it is exact.  Split each query's visible positions into aligned blocks
// of 8 and let tau be the K-th largest block maximum.  K blocks have a
// maximum >= tau, so at least K scores are >= tau: the K-th largest score is
// >= tau.  At most K-1 blocks have a maximum > tau, so at most 8(K-1) scores
// are > tau.  The Top-K is therefore every score > tau plus (K minus their
// count) of the scores equal to tau, and both sets fit in bounded lists.
//
// Kernels, in stream order:
//  1. index_score_prefill_tc_kernel<BLOCKMAX>: keys of the block maxima;
//  2. dense_threshold_kernel: one warp per query, tau by a three-pass 11-bit
//     radix select over the row's block maxima (staged in shared memory);
//     also clears the query's candidate counters;
//  3. index_score_prefill_tc_kernel<FILTER>: the same scores, appended to the
//     "above" list (key > tau) or the "tie" list (key == tau, first K kept);
//  4. dense_select_kernel: one warp per query, Top-K of the candidates (a
//     four-pass 8-bit radix select when K or more lie above tau, else all of
//     them, then ties, then -1).
#include "common.cuh"

namespace csa2 {
namespace {

constexpr int SEL_WARPS = 8;               // one warp per query row
constexpr int SEL_THREADS = 32 * SEL_WARPS;
constexpr int64_t MAX_N = 262144;

// The K-th largest of n >= K >= 1 keys key_at(0 .. n-1), by one warp, in
// radix passes of BITS-bit digits from the top (11: digits [31:21], [20:10],
// [9:0]; 8: four bytes).  Each pass counts the digits of the keys that share
// the prefix found so far in the warp's 2^BITS-bin shared histogram (plain
// shared atomics: lanes that hit the same bin are serialised by the
// hardware), then picks the bin where the count from the top reaches K.
template <int BITS>
__device__ __forceinline__ uint32_t warp_pick_bin(const uint32_t *hist, uint32_t k, uint32_t &before) {
    constexpr int PER = (1 << BITS) / 32;   // bins per lane: lane l holds bins PER l .. PER l + PER - 1
    const int lane = threadIdx.x & 31;
    uint32_t own = 0;
    const uint4 *h4 = reinterpret_cast<const uint4 *>(hist + PER * lane);
#pragma unroll
    for (int j = 0; j < PER / 4; ++j) {
        const uint4 v = h4[j];
        own += v.x + v.y + v.z + v.w;
    }
    uint32_t incl = own;   // inclusive suffix sum over lanes >= lane
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t v = __shfl_down_sync(0xFFFFFFFFu, incl, o);
        if (lane + o < 32) incl += v;
    }
    const uint32_t above = incl - own;   // keys in the bins of the lanes above
    const int L = __ffs(__ballot_sync(0xFFFFFFFFu, above < k && k <= above + own)) - 1;
    const uint32_t aboveL = __shfl_sync(0xFFFFFFFFu, above, L);
    // the warp scans lane L's PER bins together: lane j takes bins j*PER/32 ..
    constexpr int SUB = PER >= 32 ? PER / 32 : 1;   // bins per lane in this scan
    uint32_t cnt = 0;
    if (SUB * lane < PER) {
#pragma unroll
        for (int j = 0; j < SUB; ++j) cnt += hist[PER * L + SUB * lane + j];
    }
    uint32_t inc2 = cnt;   // inclusive suffix sum over the bins of lanes >= lane
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t v = __shfl_down_sync(0xFFFFFFFFu, inc2, o);
        if (lane + o < 32) inc2 += v;
    }
    const uint32_t ab2 = aboveL + inc2 - cnt;
    const bool hit = SUB * lane < PER && ab2 < k && k <= ab2 + cnt;
    const int M = __ffs(__ballot_sync(0xFFFFFFFFu, hit)) - 1;
    uint32_t d = 0, b = 0;
    if (lane == M) {
        uint32_t c = ab2;
#pragma unroll
        for (int j = SUB - 1; j >= 0; --j) {
            const uint32_t h = hist[PER * L + SUB * lane + j];
            if (c + h >= k) {
                d = (uint32_t)(PER * L + SUB * lane + j);
                b = c;
                break;
            }
            c += h;
        }
    }
    before = __shfl_sync(0xFFFFFFFFu, b, M);
    return __shfl_sync(0xFFFFFFFFu, d, M);
}

template <int BITS, typename KeyAt>
__device__ uint32_t warp_kth_largest(KeyAt key_at, int n, int K, uint32_t *hist) {
    constexpr int NB = 1 << BITS;
    const int lane = threadIdx.x & 31;
    uint32_t prefix = 0u, mask = 0u, k = (uint32_t)K;
#pragma unroll 1
    for (int shift = 32 - BITS; shift > -BITS; shift -= BITS) {
        const int sh = shift < 0 ? 0 : shift;
        const uint32_t dmask = (uint32_t)(NB - 1) >> (sh - shift);   // the last digit may be narrower
        uint4 *h4 = reinterpret_cast<uint4 *>(hist);
#pragma unroll
        for (int j = 0; j < NB / 128; ++j) h4[32 * j + lane] = make_uint4(0u, 0u, 0u, 0u);
        __syncwarp();
        for (int base = 0; base < n; base += 128) {
            uint32_t kk[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int i = base + 32 * j + lane;
                kk[j] = i < n ? key_at(i) : 0u;
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int i = base + 32 * j + lane;
                if (i < n && (kk[j] & mask) == prefix) atomicAdd(&hist[(kk[j] >> sh) & dmask], 1u);
            }
        }
        __syncwarp();
        uint32_t before;
        const uint32_t d = warp_pick_bin<BITS>(hist, k, before);
        prefix |= d << sh;
        mask |= dmask << sh;
        k -= before;
        __syncwarp();
    }
    return prefix;
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src));
}

// One warp per query row (blockDim.x / 32 rows per CTA).  The row's block
// maxima (nblk words, nblk a multiple of 4: rows are 16-byte aligned) are
// copied to the warp's slice of dynamic shared memory first, so the four
// radix passes read shared memory.
__global__ void __launch_bounds__(SEL_THREADS) dense_threshold_kernel(const uint32_t *__restrict__ bmax, int64_t nblk,
                                                                      const int32_t *__restrict__ kv_len, int64_t N,
                                                                      int rows, int K, uint32_t *__restrict__ tau,
                                                                      uint32_t *__restrict__ cnt) {
    extern __shared__ __align__(16) uint32_t dyn[];
    pdl_wait();
    pdl_launch_dependents();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nw = blockDim.x >> 5;
    uint32_t *hist = dyn + (int64_t)nw * nblk + 2048 * warp;   // after the staged maxima
    const int64_t r = (int64_t)blockIdx.x * nw + warp;
    if (r >= rows) return;
    int64_t len = kv_len[r];
    len = len < 0 ? 0 : (len > N ? N : len);
    const int nb = (int)((len + 7) / 8);
    if (lane == 0) {
        cnt[2 * r] = 0u;
        cnt[2 * r + 1] = 0u;
    }
    uint32_t t = 0u;   // fewer than K blocks: every visible position is a candidate
    if (nb >= K) {
        uint32_t *sk = dyn + (int64_t)warp * nblk;
        const uint32_t *row = bmax + r * nblk;
        for (int i = lane; 4 * i < nb; i += 32) cp_async16((uint32_t)__cvta_generic_to_shared(sk + 4 * i), row + 4 * i);
        asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
        __syncwarp();
        t = warp_kth_largest<11>([&](int i) { return sk[i]; }, nb, K, hist);
    }
    if (lane == 0) tau[r] = t;
}

__global__ void __launch_bounds__(SEL_THREADS) dense_select_kernel(const uint32_t *__restrict__ cnt,
                                                                   const uint2 *__restrict__ cand, int cap_gt,
                                                                   int cap_eq, int rows, int K,
                                                                   int32_t *__restrict__ idx) {
    __shared__ __align__(16) uint32_t hist[SEL_WARPS][256];
    pdl_wait();
    pdl_launch_dependents();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t r = (int64_t)blockIdx.x * SEL_WARPS + warp;
    if (r >= rows) return;
    const uint2 *c = cand + r * (int64_t)(cap_gt + cap_eq);
    int32_t *out = idx + r * K;
    const uint32_t c_gt = cnt[2 * r], c_eq = cnt[2 * r + 1];
    const int n_gt = (int)(c_gt < (uint32_t)cap_gt ? c_gt : (uint32_t)cap_gt);
    const int n_eq = (int)(c_eq < (uint32_t)cap_eq ? c_eq : (uint32_t)cap_eq);
    if (n_gt < K) {
        // all candidates above tau, then ties at tau, then padding
        for (int i = lane; i < n_gt; i += 32) out[i] = (int32_t)c[i].y;
        const int ne = n_eq < K - n_gt ? n_eq : K - n_gt;
        for (int i = lane; i < ne; i += 32) out[n_gt + i] = (int32_t)c[cap_gt + i].y;
        for (int i = n_gt + ne + lane; i < K; i += 32) out[i] = -1;
        return;
    }
    const uint32_t t = warp_kth_largest<8>([&](int i) { return c[i].x; }, n_gt, K, hist[warp]);
    // keys above t (fewer than K) first, then ties at t up to K, in list order
    uint32_t n_above = 0;
    for (int base = 0; base < n_gt; base += 32) {
        const int i = base + lane;
        const bool p = i < n_gt && c[i].x > t;
        n_above += (uint32_t)__popc(__ballot_sync(0xFFFFFFFFu, p));
    }
    uint32_t o_above = 0, o_tie = n_above;
    for (int base = 0; base < n_gt; base += 32) {
        const int i = base + lane;
        const uint32_t k = i < n_gt ? c[i].x : 0u;
        const uint32_t ba = __ballot_sync(0xFFFFFFFFu, i < n_gt && k > t);
        const uint32_t be = __ballot_sync(0xFFFFFFFFu, i < n_gt && k == t);
        const uint32_t below = (1u << lane) - 1u;
        if ((ba >> lane) & 1u) out[o_above + __popc(ba & below)] = (int32_t)c[i].y;
        if ((be >> lane) & 1u) {
            const uint32_t j = o_tie + (uint32_t)__popc(be & below);
            if (j < (uint32_t)K) out[j] = (int32_t)c[i].y;
        }
        o_above += (uint32_t)__popc(ba);
        o_tie += (uint32_t)__popc(be);
    }
}

}  // namespace
}  // namespace csa2

using namespace csa2;

static size_t align256(size_t b) { return (b + 255) & ~(size_t)255; }

struct DenseLayout {
    size_t bmax, tau, cnt, cand, total;
    int64_t nblk;
    int cap_gt, cap_eq;
};

static DenseLayout dense_layout(int B, int T, int64_t N, int K) {
    DenseLayout L;
    const size_t R = (size_t)B * (size_t)T;
    L.nblk = ((N + 7) / 8 + 3) / 4 * 4;   // block-maximum rows padded to 16 bytes
    L.cap_gt = 8 * (K - 1);
    L.cap_eq = K;
    L.bmax = 0;
    L.tau = L.bmax + align256(R * (size_t)L.nblk * 4);
    L.cnt = L.tau + align256(R * 4);
    L.cand = L.cnt + align256(R * 8);
    L.total = L.cand + align256(R * (size_t)(L.cap_gt + L.cap_eq) * 8);
    return L;
}

extern "C" size_t csa2_index_topk_dense_workspace_bytes(int B, int T, int64_t N, int K) {
    if (B < 0 || T < 0 || N < 0 || K < 1 || K > CSA2_MAX_K) return 0;
    return dense_layout(B, T, N, K).total;
}

extern "C" csa2_status csa2_index_topk_dense(int B, int T, int64_t N, const void *q_idx, csa2_dtype q_dt,
                                             const float *w, const void *k_idx, csa2_dtype k_dt,
                                             const int32_t *kv_len, int K, int32_t *idx, uint32_t *err_flag,
                                             void *workspace, size_t ws_bytes, csa2_stream_t stream) {
    clear_error();
    CSA2_REQUIRE(B >= 0 && T >= 0 && N >= 0, "index_topk_dense: negative shape");
    CSA2_REQUIRE(q_dt == CSA2_FP8_E4M3 && k_dt == CSA2_FP8_E4M3, "index_topk_dense: q_idx and k_idx must be FP8_E4M3");
    CSA2_REQUIRE(K >= 1 && K <= CSA2_MAX_K, "index_topk_dense: K=%d not in [1,2048]", K);
    if (N > MAX_N) {
        set_error("index_topk_dense: N=%lld > %lld", (long long)N, (long long)MAX_N);
        return CSA2_ERR_UNSUPPORTED;
    }
    if ((int64_t)B * T == 0) return CSA2_OK;
    CSA2_REQUIRE(idx && kv_len, "index_topk_dense: null idx / kv_len");
    CSA2_REQUIRE(N == 0 || (q_idx && w && k_idx), "index_topk_dense: null pointer");
    CSA2_REQUIRE(N == 0 || (aligned(q_idx, 16) && aligned(k_idx, 16)),
                 "index_topk_dense: q_idx/k_idx must be 16-byte aligned");
    CSA2_REQUIRE(aligned(w, 4) && aligned(kv_len, 4) && aligned(idx, 4), "index_topk_dense: misaligned w/kv_len/idx");
    const DenseLayout L = dense_layout(B, T, N, K);
    if (!workspace || ws_bytes < L.total || !aligned(workspace, 16)) {
        set_error("index_topk_dense: workspace needs %zu bytes, 16-byte aligned (got %zu)", L.total, ws_bytes);
        return CSA2_ERR_WORKSPACE;
    }
    uint8_t *ws = (uint8_t *)workspace;
    uint32_t *bmax = (uint32_t *)(ws + L.bmax);
    uint32_t *tau = (uint32_t *)(ws + L.tau);
    uint32_t *cnt = (uint32_t *)(ws + L.cnt);
    uint2 *cand = (uint2 *)(ws + L.cand);
    const unsigned rows = (unsigned)((int64_t)B * T);
    cudaStream_t s = stream_of(stream);
    csa2_status st;
    if (N > 0) {
        st = launch_prefill_block_max(B, T, N, q_idx, w, k_idx, kv_len, bmax, L.nblk, err_flag, s);
        if (st != CSA2_OK) return st;
    }
    // rows per threshold CTA: as many as fit in 64 KB of staged maxima (1 to 8)
    int64_t tw = 65536 / (L.nblk * 4 > 0 ? L.nblk * 4 : 1);
    tw = tw < 1 ? 1 : (tw > SEL_WARPS ? SEL_WARPS : tw);
    static bool thr_smem[64];
    CSA2_CUDA_CALL(ensure_smem_limit((const void *)dense_threshold_kernel, (int)(MAX_N / 8 * 4 + 8192), thr_smem),
                   "dense_threshold_kernel: smem attribute");
    CSA2_CUDA_CALL(launch_pdl(dense_threshold_kernel, dim3((unsigned)((rows + tw - 1) / tw)), dim3((unsigned)(32 * tw)),
                              (size_t)(tw * (L.nblk + 2048) * 4), s, (const uint32_t *)bmax, L.nblk, kv_len, N, (int)rows, K,
                              tau, cnt),
                   "dense_threshold_kernel launch");
    CSA2_LAUNCH_CHECK("dense_threshold_kernel");
    if (N > 0) {
        st = launch_prefill_filter(B, T, N, q_idx, w, k_idx, kv_len, bmax, L.nblk, tau, cnt, cand, L.cap_gt, L.cap_eq,
                                   err_flag, s);
        if (st != CSA2_OK) return st;
    }
    const unsigned sel_grid = (rows + SEL_WARPS - 1) / SEL_WARPS;
    CSA2_CUDA_CALL(launch_pdl(dense_select_kernel, dim3(sel_grid), dim3(SEL_THREADS), 0, s,
                              (const uint32_t *)cnt, (const uint2 *)cand, L.cap_gt, L.cap_eq, (int)rows, K, idx),
                   "dense_select_kernel launch");
    CSA2_LAUNCH_CHECK("dense_select_kernel");
    return CSA2_OK;
}

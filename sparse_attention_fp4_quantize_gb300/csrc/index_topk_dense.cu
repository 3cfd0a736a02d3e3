// csa2_index_topk_dense: Full-mode indexer scoring and Top-K for many query
// tokens per sequence (a prefill chunk) without the [B, T, N] score matrix.
// Sources: "DeepSeek-V4.1-Flash：把 KV Cache 压缩到极限的百万上下文 MoE", section
// "Hierarchical Sparse Indexer——索引成本变常数" (Full layers score every entry;
// Top-512 per query).  The passes below are this library's; the pages only
// state what is selected.
//
// Why it is exact.  Split each query's visible positions into aligned blocks
// of 8 and let tau be the K-th largest block maximum.  K blocks reach tau, so
// the K-th largest score is >= tau; a score outside the K blocks whose
// maximum is largest (ties at tau broken arbitrarily) is <= tau.  So the
// Top-K of the scores inside those K blocks (8K candidates) is a Top-K of the
// row, the same argument as the hierarchical pool's.  The rescoring below
// uses warp MMAs on keys converted to f16 while the block maxima come from
// the tensor-core pass, so the two may sum a score in a different order and
// differ in the last bits of fp32: a difference only at the K-th value,
// inside the selection's tie band.
//
// Kernels, in stream order:
//  1. index_blockmax_tc_kernel: keys of the 8-position block maxima,
//     [B*T, nblk] (the dense tcgen05 pass over every (query, key));
//  2. dense_rescore_kernel: one CTA per query.  The row's block maxima are
//     staged in shared memory; tau and the K blocks by a block-wide radix
//     select; the 8K candidates gathered (blocks are 512 contiguous bytes of
//     keys) and rescored with f16 mma.sync (FP8 -> f16 in registers, exact);
//     the Top-K of their scores by the same radix select, written in
//     position order of the candidates, -1 padded.
#include "common.cuh"

namespace csa2 {
namespace {

constexpr int RS_THREADS = 256;
constexpr int RS_WARPS = RS_THREADS / 32;
constexpr int64_t MAX_N = 262144;

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src));
}

// Sum of one value per thread over the CTA (scratch: RS_WARPS words; the
// caller's next barrier separates two uses).
__device__ __forceinline__ uint32_t block_sum(uint32_t v, uint32_t *scratch) {
    v = __reduce_add_sync(0xFFFFFFFFu, v);
    if ((threadIdx.x & 31) == 0) scratch[threadIdx.x >> 5] = v;
    __syncthreads();
    uint32_t s = 0;
#pragma unroll
    for (int i = 0; i < RS_WARPS; ++i) s += scratch[i];
    __syncthreads();
    return s;
}

__device__ __forceinline__ uint32_t warp_suffix(uint32_t v) {   // sum over lanes >= lane
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_down_sync(0xFFFFFFFFu, v, o);
        if (lane + o < 32) v += y;
    }
    return v;
}

// The K-th largest of n >= K >= 1 keys in shared memory (16-byte aligned, zero
// from n up to a multiple of 4), by the whole CTA:
// three radix passes over the digits [31:21], [20:10], [9:0].  Each pass
// histograms the keys that share the prefix found so far (2048 shared bins,
// shared atomics), then the thread whose 8 bins hold the K-th key from the
// top publishes the bin.  scratch: at least RS_WARPS + 2 words.  n_greater:
// the number of keys > the result (K less the keys equal to it that are needed).
__device__ uint32_t block_kth_largest(const uint32_t *keys, int n, int K, uint32_t *hist, uint32_t *scratch,
                                      uint32_t &n_greater) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    uint32_t prefix = 0u, mask = 0u, k = (uint32_t)K;
#pragma unroll 1
    for (int pass = 0; pass < 3; ++pass) {
        const int sh = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
        const uint32_t dmask = pass == 2 ? 1023u : 2047u;
        reinterpret_cast<uint4 *>(hist)[tid] = make_uint4(0u, 0u, 0u, 0u);
        reinterpret_cast<uint4 *>(hist)[tid + RS_THREADS] = make_uint4(0u, 0u, 0u, 0u);
        __syncthreads();
        for (int i = tid; 4 * i < n; i += RS_THREADS) {   // keys [n, 4 ceil(n / 4)) are zero
            const uint4 v = reinterpret_cast<const uint4 *>(keys)[i];
            if ((v.x & mask) == prefix) atomicAdd(&hist[(v.x >> sh) & dmask], 1u);
            if ((v.y & mask) == prefix) atomicAdd(&hist[(v.y >> sh) & dmask], 1u);
            if ((v.z & mask) == prefix) atomicAdd(&hist[(v.z >> sh) & dmask], 1u);
            if ((v.w & mask) == prefix) atomicAdd(&hist[(v.w >> sh) & dmask], 1u);
        }
        __syncthreads();
        // this thread's bins 8 tid .. 8 tid + 7, as two 16-byte reads (eight word
        // reads at a stride of eight words would meet each bank eight times)
        const uint4 ha = reinterpret_cast<const uint4 *>(hist)[2 * tid], hb = reinterpret_cast<const uint4 *>(hist)[2 * tid + 1];
        const uint32_t h[8] = {ha.x, ha.y, ha.z, ha.w, hb.x, hb.y, hb.z, hb.w};
        uint32_t own = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) own += h[j];
        const uint32_t incl = warp_suffix(own);
        if (lane == 0) scratch[warp] = incl;   // warp totals
        __syncthreads();
        uint32_t above = incl - own;
        for (int w2 = warp + 1; w2 < RS_WARPS; ++w2) above += scratch[w2];
        if (above < k && k <= above + own) {   // exactly one thread
            uint32_t c = above;
            for (int j = 7; j >= 0; --j) {
                if (c + h[j] >= k) {
                    scratch[RS_WARPS] = 8u * (uint32_t)tid + (uint32_t)j;
                    scratch[RS_WARPS + 1] = c;
                    break;
                }
                c += h[j];
            }
        }
        __syncthreads();
        const uint32_t bin = scratch[RS_WARPS], before = scratch[RS_WARPS + 1];
        const uint32_t inbin = hist[bin];
        prefix |= bin << sh;
        mask |= dmask << sh;
        k -= before;
        __syncthreads();   // scratch and the histogram are reused
        // the boundary bin is taken whole: exactly K keys are >= its lower
        // edge, so every key above edge - 1 is selected (prefix >= 2^21 here)
        if (inbin == k) {
            n_greater = (uint32_t)K;
            return prefix - 1u;
        }
    }
    n_greater = (uint32_t)K - k;   // k keys equal to the result complete the K
    return prefix;
}

// Writes to out[0, K): every i < n with keys[i] > T, then keys[i] == T until K
// are taken, lowest i first (T = 0: every nonzero key), then -1; pos(i) gives
// the output id.  above = the number of keys > T (known to the caller from the
// selection).  Warp w owns a contiguous run of the keys: a first pass counts
// its keys above and at T, the warps' counts give each warp its first slots,
// and a second pass writes the ids in position order (ballot prefixes, no
// atomics).  scratch: at least 2 RS_WARPS words; the caller's next barrier
// separates this from another use of it.
template <typename PosFn>
__device__ void block_emit(const uint32_t *keys, int n, uint32_t T, uint32_t above, int K, int32_t *out, PosFn pos,
                           uint32_t *scratch) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t room = above < (uint32_t)K ? (uint32_t)K - above : 0u;
    const bool ties = T != 0u && room != 0u;
    int R = (n + RS_WARPS - 1) / RS_WARPS;
    R = (R + 31) & ~31;
    const int w0 = min(n, warp * R), w1 = min(n, w0 + R);
    uint32_t cg = 0u, ce = 0u;
    for (int base = w0; base < w1; base += 32) {
        const int i = base + lane;
        const uint32_t k = i < w1 ? keys[i] : 0u;
        cg += __popc(__ballot_sync(0xFFFFFFFFu, k > T));
        if (ties) ce += __popc(__ballot_sync(0xFFFFFFFFu, k == T));
    }
    if (lane == 0) {
        scratch[warp] = cg;
        scratch[RS_WARPS + warp] = ce;
    }
    __syncthreads();
    uint32_t slot = 0u, tie = 0u, te = 0u;
#pragma unroll
    for (int w2 = 0; w2 < RS_WARPS; ++w2) {
        const uint32_t e2 = scratch[RS_WARPS + w2];
        if (w2 < warp) {
            slot += scratch[w2];
            tie += e2;
        }
        te += e2;
    }
    const uint32_t lt = (1u << lane) - 1u;
    for (int base = w0; base < w1; base += 32) {
        const int i = base + lane;
        const uint32_t k = i < w1 ? keys[i] : 0u;
        const uint32_t bg = __ballot_sync(0xFFFFFFFFu, k > T);
        if ((bg >> lane) & 1u) {
            const uint32_t s2 = slot + __popc(bg & lt);
            if (s2 < (uint32_t)K) out[s2] = pos(i);
        }
        slot += __popc(bg);
        if (ties) {
            const uint32_t be = __ballot_sync(0xFFFFFFFFu, k == T);
            if ((be >> lane) & 1u) {
                const uint32_t t2 = tie + __popc(be & lt);
                if (t2 < room) out[above + t2] = pos(i);
            }
            tie += __popc(be);
        }
    }
    const uint32_t taken = min((uint32_t)K, above) + min(room, te);
    for (int i = (int)taken + tid; i < K; i += RS_THREADS) out[i] = -1;
}

struct RescoreArgs {
    int T;
    int64_t N;
    int K;
    const uint32_t *bmax;   // [B*T, nblk] block-maximum keys
    int64_t nblk;           // multiple of 4
    const uint8_t *q;       // FP8 [B*T, 4, 64]
    const float *w;         // [B*T, 4]
    const uint8_t *k;       // FP8 [B, N, 64]
    const int32_t *kv_len;  // [B*T]
    int32_t *idx;           // [B*T, K]
};

__global__ void __launch_bounds__(RS_THREADS, 4) dense_rescore_kernel(RescoreArgs a) {
    extern __shared__ __align__(16) uint32_t dyn[];   // [nblk] maxima | [16 ceil(K/2)] candidate keys | [2 ceil(K/2)] blocks
    __shared__ __align__(16) uint32_t hist[2048];
    __shared__ uint32_t scratch[2 * RS_WARPS + 2];
    pdl_wait();
    pdl_launch_dependents();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, t4 = lane & 3;
    const int64_t r = blockIdx.x, b = r / a.T;
    int64_t len = a.kv_len[r];
    len = len < 0 ? 0 : (len > a.N ? a.N : len);
    const int nb = (int)((len + 7) / 8);
    uint32_t *sBm = dyn;
    uint32_t *sSc = dyn + a.nblk;   // 16 ceil(K / 2) slots: whole two-block tiles
    int32_t *sBlk = reinterpret_cast<int32_t *>(sSc + 16 * ((a.K + 1) / 2));
    int32_t *out = a.idx + r * a.K;

    // ---- the K blocks with the largest maxima (all of them when nb <= K)
    int nsel;
    if (nb <= a.K) {
        for (int i = tid; i < nb; i += RS_THREADS) sBlk[i] = i;
        nsel = nb;
    } else {
        const uint32_t *row = a.bmax + r * a.nblk;
        for (int i = tid; 4 * i < nb; i += RS_THREADS) cp_async16((uint32_t)__cvta_generic_to_shared(sBm + 4 * i), row + 4 * i);
        asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
        if (tid == ((nb - 1) >> 2) % RS_THREADS)   // the thread that copied the last group zeroes its tail
            for (int j = nb; j < ((nb + 3) & ~3); ++j) sBm[j] = 0u;
        __syncthreads();
        uint32_t above;
        const uint32_t tau = block_kth_largest(sBm, nb, a.K, hist, scratch, above);
        block_emit(sBm, nb, tau, above, a.K, sBlk, [](int i) { return (int32_t)i; }, scratch);
        nsel = a.K;
    }
    if (tid == 0 && (nsel & 1)) sBlk[nsel] = -1;   // the odd tile's second block: no position
    __syncthreads();

    // ---- rescore the 8 nsel candidates: a tile is two blocks (16 keys); lane
    // (g, t4) loads the 16 bytes of channels 16 t4 .. 16 t4 + 15 of key g of
    // each block (MMA rows g and g + 8; the 4 heads are columns 0-3 of n8) and
    // converts them to f16 (exact) for four m16n8k16 MMAs: MMA j takes the
    // lane's channels 16 t4 + 4 j .. + 3 as its k = 2 t4, 2 t4 + 1, 2 t4 + 8,
    // 2 t4 + 9, the query the same way (the FP8 warp MMA costs several times
    // the f16 one's instructions here, and the query is converted once).
    // Positions are below 2^18, so a block's position test and its byte offset
    // are 32-bit arithmetic (block -1 wraps to a position past every row length).
    const uint4 q8 = (g < 4) ? __ldg(reinterpret_cast<const uint4 *>(a.q + (r * 4 + g) * 64 + 16 * t4))
                             : make_uint4(0u, 0u, 0u, 0u);
    uint32_t qlo[4], qhi[4];
    e4m3x4_to_f16x2x2(q8.x, qlo[0], qhi[0]);
    e4m3x4_to_f16x2x2(q8.y, qlo[1], qhi[1]);
    e4m3x4_to_f16x2x2(q8.z, qlo[2], qhi[2]);
    e4m3x4_to_f16x2x2(q8.w, qlo[3], qhi[3]);
    const float w0 = (t4 < 2) ? a.w[r * 4 + 2 * t4] : 0.f;
    const float w1 = (t4 < 2) ? a.w[r * 4 + 2 * t4 + 1] : 0.f;
    const int ntile = (nsel + 1) / 2;
    const uint8_t *kq = a.k + b * a.N * 64 + 16 * t4;   // this lane's 16 bytes of the sequence's first key
    const uint32_t ulen = (uint32_t)len;
    const int2 *sBlk2 = reinterpret_cast<const int2 *>(sBlk);
    for (int t0 = warp; t0 < ntile; t0 += 4 * RS_WARPS) {
        uint4 raw[4][2];
        bool v[4][2];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int tl = t0 + u * RS_WARPS;
            const int2 bb = tl < ntile ? sBlk2[tl] : make_int2(-1, -1);
            const uint32_t blk[2] = {(uint32_t)bb.x, (uint32_t)bb.y};
#pragma unroll
            for (int rr = 0; rr < 2; ++rr) {   // a slot past the row reads the first key (its score is dropped)
                const uint32_t p = blk[rr] * 8u + (uint32_t)g;
                v[u][rr] = p < ulen;
                raw[u][rr] = __ldg(reinterpret_cast<const uint4 *>(kq + (v[u][rr] ? p * 64u : 0u)));
            }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int tl = t0 + u * RS_WARPS;
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
            const uint32_t w0r[4] = {raw[u][0].x, raw[u][0].y, raw[u][0].z, raw[u][0].w};
            const uint32_t w1r[4] = {raw[u][1].x, raw[u][1].y, raw[u][1].z, raw[u][1].w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                uint32_t a0, a2, a1, a3;
                e4m3x4_to_f16x2x2(w0r[j], a0, a2);   // row g: channels +0,+1 | +2,+3
                e4m3x4_to_f16x2x2(w1r[j], a1, a3);   // row g + 8
                mma_f16_16816(acc, a0, a1, a2, a3, qlo[j], qhi[j]);
            }
            float s0 = w0 * fmaxf(acc[0], 0.f) + w1 * fmaxf(acc[1], 0.f);
            float s1 = w0 * fmaxf(acc[2], 0.f) + w1 * fmaxf(acc[3], 0.f);
            s0 += __shfl_xor_sync(0xFFFFFFFFu, s0, 1);
            s1 += __shfl_xor_sync(0xFFFFFFFFu, s1, 1);
            if (t4 == 0 && tl < ntile) {
                sSc[16 * tl + g] = v[u][0] ? score_key(s0) : 0u;
                sSc[16 * tl + 8 + g] = v[u][1] ? score_key(s1) : 0u;
            }
        }
    }
    __syncthreads();

    // ---- Top-K of the candidates (every valid one when at most K)
    const int m = 16 * ntile;   // candidate slots (an odd block count leaves 8 empty)
    uint32_t nv = 0;
    for (int i = tid; i < m; i += RS_THREADS) nv += sSc[i] != 0u ? 1u : 0u;
    nv = block_sum(nv, scratch);
    uint32_t above = nv;   // at most K candidates: every nonzero key
    const uint32_t T = nv <= (uint32_t)a.K ? 0u : block_kth_largest(sSc, m, a.K, hist, scratch, above);
    block_emit(sSc, m, T, above, a.K, out, [&](int i) { return sBlk[i >> 3] * 8 + (i & 7); }, scratch);
}

}  // namespace
}  // namespace csa2

using namespace csa2;

static size_t align256(size_t b) { return (b + 255) & ~(size_t)255; }

static int64_t nblk_for(int64_t N) { return ((N + 7) / 8 + 3) / 4 * 4; }   // block-maximum rows padded to 16 bytes

extern "C" size_t csa2_index_topk_dense_workspace_bytes(int B, int T, int64_t N, int K) {
    if (B < 0 || T < 0 || N < 0 || K < 1 || K > CSA2_MAX_K) return 0;
    return align256((size_t)B * (size_t)T * (size_t)nblk_for(N) * 4);
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
    const int64_t nblk = nblk_for(N);
    const size_t need = csa2_index_topk_dense_workspace_bytes(B, T, N, K);
    if (!workspace || ws_bytes < need || !aligned(workspace, 16)) {
        set_error("index_topk_dense: workspace needs %zu bytes, 16-byte aligned (got %zu)", need, ws_bytes);
        return CSA2_ERR_WORKSPACE;
    }
    uint32_t *bmax = (uint32_t *)workspace;
    cudaStream_t s = stream_of(stream);
    if (N > 0) {
        const csa2_status st = launch_prefill_block_max(B, T, N, q_idx, w, k_idx, kv_len, bmax, nblk, err_flag, s);
        if (st != CSA2_OK) return st;
    }
    RescoreArgs ra;
    ra.T = T; ra.N = N; ra.K = K; ra.bmax = bmax; ra.nblk = nblk;
    ra.q = (const uint8_t *)q_idx; ra.w = w; ra.k = (const uint8_t *)k_idx; ra.kv_len = kv_len; ra.idx = idx;
    const size_t smem = (size_t)(nblk + 18 * (int64_t)((K + 1) / 2)) * 4;
    static bool smem_set[64];
    CSA2_CUDA_CALL(ensure_smem_limit((const void *)dense_rescore_kernel,
                                     (int)((nblk_for(MAX_N) + 18 * ((CSA2_MAX_K + 1) / 2)) * 4), smem_set),
                   "dense_rescore_kernel: smem attribute");
    CSA2_CUDA_CALL(launch_pdl(dense_rescore_kernel, dim3((unsigned)((int64_t)B * T)), dim3(RS_THREADS), smem, s, ra),
                   "dense_rescore_kernel launch");
    CSA2_LAUNCH_CHECK("dense_rescore_kernel");
    return CSA2_OK;
}

// Sparse FP4 attention on the 5th-generation tensor cores (tcgen05, TMEM),
// for 576-channel entries (512 latent + 64 RoPE), dv = 512, 64-head blocks,
// up to 512 selected entries.
// Sources: "DeepSeek-V4.1-Flash：把 KV Cache 压缩到极限的百万上下文 MoE", section
// "效率组件四件" item 4 (FP4 main KV) and the inference bullet of
// "优化器与训练基础设施" (Reuse layers run a fused attention kernel; prior art);
// "DeepSeek-V4.1-Flash: Pushing the Limits of KV Cache Compression", CSA2
// paragraph.  The attention itself is the MLA-style reading (K = all 576
// channels, V = the first 512).
//
// Layout of the work.  A thread-block cluster of S in {1, 2, 4} CTAs serves
// one query token and 64 heads; CTA c owns selected entries [128c, 128c+128).
// 512 threads: four per entry (144 channels each) and eight per head.
//  1. The TMA engine gathers the operands: one bulk copy per Q head row
//     (1152 B, on its own mbarrier) and one per selected entry's code row
//     (288 B); the 36-byte scale rows (not 16-byte sized) are plain loads.
//  2. Q (bf16) is scaled per head by a power of two into f16 (exact down to
//     2^-31 of the head's largest |q|, which must stay below 2^76; the scale
//     is folded into the logit factor) while the code rows are in flight; the
//     entries are dequantised once (E2M1 x E4M3 -> exact f16) into a no-swizzle core-matrix tile.
//  3. S^T [128 entries x 64 heads] = Khat . Q^T  (36 tcgen05.mma, M128 N64 K16)
//  4. softmax on a transposed copy of S^T in shared memory; P -> f16.
//  5. O^T [512 ch x 64 heads] = Vhat^T . P^T  (4 x 8 MMAs; the same Khat bytes
//     read MN-major), fp32 accumulators in TMEM.
//  6. Merge across the cluster: every CTA pushes its per-head (max, sum) into
//     every CTA's shared memory, normalises its partial O by the sum and
//     stages each other CTA's 128-channel slice as f16 below the P tile; after
//     one cluster barrier the TMA engine copies the slices into the owners'
//     shared memory (bulk shared -> remote shared copies completing on the
//     owner's mbarrier).  Each owner combines its slice with the weights
//     L_c 2^(m_c - M) / sum_c' L_c' 2^(m_c' - M) and writes it out, its own
//     part read straight from TMEM in fp32 (a single-CTA cluster writes all
//     of O / L that way, with no staging).
// Waits on the mbarriers are bounded; on timeout the kernel sets
// CSA2_FLAG_TIMEOUT and still runs every cluster barrier, so it always ends.
#include <cooperative_groups.h>
#include <type_traits>

#include "common.cuh"
#include "tc.cuh"

namespace cg = cooperative_groups;

namespace csa2 {
namespace {

constexpr int TM = 128;                    // entries per CTA (MMA M)
constexpr int D = 576, DV = 512, HB = 64;  // channels, value channels, heads per cluster
constexpr int THREADS = 512;               // 4 threads per entry, 8 per head
constexpr int MAX_S = 4;                   // CTAs per cluster
constexpr uint32_t KT_SBO = (D / 8) * 128;        // 9216: bytes per 8-entry group of the Khat tile
constexpr uint32_t KT_BYTES = (TM / 8) * KT_SBO;  // 147456
constexpr uint32_t Q_SBO = (D / 8) * 128;         // 9216: bytes per 8-head group of the Q tile
constexpr uint32_t Q_BYTES = (HB / 8) * Q_SBO;    // 73728
constexpr uint32_t QRAW_STRIDE = D * 2 + 16;      // 1168: staged bf16 Q rows (padded: conflict-free reads)
constexpr uint32_t CRAW_STRIDE = D / 2 + 16;      // 304: staged code rows (padded)
constexpr uint32_t OFF_QRAW = 0;                  // staging lives in the Khat region before dequant
constexpr uint32_t OFF_CRAW = HB * QRAW_STRIDE;   // 74752
constexpr int ST_STRIDE = TM + 8;                 // fp32 row stride of the transposed S (136)
constexpr uint32_t ST_BYTES = HB * ST_STRIDE * 4; // 34816
constexpr uint32_t P_SBO = (TM / 8) * 128;        // 2048: bytes per 8-head group of the P tile
constexpr uint32_t OFF_K = 0;
constexpr uint32_t OFF_Q = OFF_K + KT_BYTES;
constexpr uint32_t OFF_ST = OFF_Q;                // reuses the Q tile after S is computed
constexpr uint32_t OFF_P = OFF_Q + Q_BYTES - (HB / 8) * P_SBO;   // P at the end: staging fits below it
constexpr uint32_t OFF_MISC = OFF_Q + Q_BYTES;
constexpr uint32_t OFF_BAR = OFF_MISC;            // 5 mbarriers: Q, codes, S, O, received (64 bytes reserved)
constexpr uint32_t OFF_TMEM = OFF_BAR + 64;
constexpr uint32_t OFF_VALID = OFF_TMEM + 16;     // int[128]
constexpr uint32_t OFF_CS = OFF_VALID + TM * 4;   // float[64] logit factor per head
constexpr uint32_t OFF_M = OFF_CS + HB * 4;       // float[64] row max (log2 domain)
constexpr uint32_t OFF_L = OFF_M + HB * 4;        // float[64] row sum
constexpr uint32_t OFF_W = OFF_L + HB * 4;        // float[MAX_S][64] merge weights
constexpr uint32_t OFF_LSE = OFF_W + MAX_S * HB * 4;      // float[64]
constexpr uint32_t OFF_IL = OFF_LSE + HB * 4;             // float[64] 1 / row sum
constexpr uint32_t OFF_STATS = OFF_IL + HB * 4;           // float[MAX_S][2][64] every CTA's (max, sum)
constexpr uint32_t OFF_BETA = OFF_STATS + MAX_S * 2 * HB * 4;   // float[64] sparse-branch weight (FP8W merge)
constexpr uint32_t SMEM = OFF_BETA + HB * 4;
// Merge payload: the normalised partial O (O / L) of W channels as f16 rows of
// RSH halves (136 bytes: 8-byte accesses by consecutive channels are
// conflict-free).
constexpr int RSH = HB + 4;
__host__ __device__ constexpr uint32_t slice_bytes_for(int W) { return (uint32_t)W * RSH * 2; }
constexpr uint32_t TMEM_COLS = 512;               // S^T: 64 cols, O^T: 4 x 64 cols
constexpr uint32_t S_COL = 0, O_COL = 64;
constexpr uint32_t MAX_POLLS = 1u << 22;          // about a second of polling at most
static_assert(OFF_CRAW + TM * CRAW_STRIDE <= KT_BYTES, "staging must fit in the Khat region");
static_assert(MAX_S * slice_bytes_for(DV / MAX_S) <= KT_BYTES && 2 * slice_bytes_for(DV / 2) <= KT_BYTES,
              "received partials must fit in the Khat region");
static_assert(slice_bytes_for(DV / MAX_S) % 16 == 0 && slice_bytes_for(DV / 2) % 16 == 0, "bulk copy sizes");
static_assert(ST_BYTES + (HB / 8) * P_SBO <= Q_BYTES, "S^T copy and P must fit in the Q region");
static_assert((MAX_S - 1) * slice_bytes_for(DV / MAX_S) <= OFF_P - OFF_Q && slice_bytes_for(DV / 2) <= OFF_P - OFF_Q,
              "the slices owed to other CTAs are staged below P while P V runs");
static_assert(SMEM <= 227 * 1024, "shared memory");

struct TcArgs {
    int T, H, K, csize, hblocks;
    int64_t N;
    const uint16_t *q;
    const uint8_t *codes;
    const uint8_t *scales;
    const int32_t *idx;
    const int32_t *kv_len;
    float sm_scale;
    float *out;
    float *lse;
    uint32_t *err_flag;
    // sliding-window branch (FP8W): E4M3 rows [B, W, D], the first swa_len[bt]
    // of them attended; merged with the sparse branch's (o_sparse, lse_sparse)
    const uint8_t *kv8;
    int W;
    const int32_t *swa_len;
    const float *o_sparse;
    const float *lse_sparse;
    // optional L2 prefetch: the same selected rows of another pair of FP4 planes
    const uint8_t *pf_codes;
    const uint8_t *pf_scales;
    int64_t items;   // token kernel: (token, 64-head block) items, taken in turn by persistent CTAs
};

// 16 E4M3 bytes -> 16 f16 (exact), as 8 f16x2 words.
__device__ __forceinline__ void e4m3x16_to_f16(const uint4 v, uint32_t (&r)[8]) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r[2 * k]) : "h"((uint16_t)(w[k] & 0xFFFFu)));
        asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r[2 * k + 1]) : "h"((uint16_t)(w[k] >> 16)));
    }
}

__device__ __forceinline__ uint32_t e4m3_to_f16x2_bcast(uint32_t byte) {
    uint32_t r;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"((uint16_t)(byte | (byte << 8))));
    return r;
}

__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// Eight E2M1 codes (one word; byte i holds codes 2i (low nibble) and 2i + 1)
// -> four f16x2 words times the f16x2 scale sc (exact: at most 6 significant
// bits).  The word is split into its bytes by a vector move, not by shifts.
__device__ __forceinline__ void e2m1x8_scaled(uint32_t w, uint32_t sc, uint32_t *r) {
    uint32_t h0, h1, h2, h3;
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
        "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
        "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
        : "=r"(h0), "=r"(h1), "=r"(h2), "=r"(h3)
        : "r"(w));
    r[0] = hmul2(h0, sc);
    r[1] = hmul2(h1, sc);
    r[2] = hmul2(h2, sc);
    r[3] = hmul2(h3, sc);
}

__device__ __forceinline__ float max3f(float a, float b, float c) {   // the three-input form of fmaxf
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}
__device__ __forceinline__ float ex2(float x) {
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}

// Bulk global -> shared copy (TMA engine) completing on an mbarrier.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}


__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

// Bulk copy from this CTA's shared memory to another CTA's (TMA engine),
// completing on the destination CTA's mbarrier.
__device__ __forceinline__ void bulk_s2s(uint32_t dst_remote, uint32_t src_local, uint32_t bytes, uint32_t bar_remote) {
    asm volatile("cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     dst_remote),
                 "r"(src_local), "r"(bytes), "r"(bar_remote)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// L2 prefetch hints (no data is returned; nothing waits on them).
__device__ __forceinline__ void bulk_prefetch_l2(const void *src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}
__device__ __forceinline__ void prefetch_l2(const void *p) { asm volatile("prefetch.global.L2 [%0];" ::"l"(p)); }
__device__ __forceinline__ void bulk_wait_read0() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }

// FP8W = false: the sparse branch (FP4 entries gathered by idx).  FP8W = true:
// the sliding-window branch (the first swa_len E4M3 rows of the window,
// contiguous, no scales) merged at the end with the sparse branch's output.
// 32 lanes x N consecutive fp32 TMEM columns (N = 4 or 16).
template <int N>
__device__ __forceinline__ void tmem_ld_n(uint32_t taddr, uint32_t (&r)[N]) {
    static_assert(N == 4 || N == 16, "column counts");
    if constexpr (N == 16) {
        tc::tmem_ld16(taddr, r);
    } else {
        asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%4];"
                     : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                     : "r"(taddr));
    }
}

template <bool FP8W, int NH>
__global__ void __launch_bounds__(THREADS, 1) sparse_attn_tc_kernel(TcArgs a) {
    static_assert(NH == HB || (NH == HB / 4 && !FP8W), "64 heads per CTA, or 16 for few-token launches");
    constexpr int HPT = NH / 4;                 // heads per thread where a warp pair of lane quarter x head group works
    constexpr int RSHN = NH + 4;                // halves per channel row of an exchanged slice
    extern __shared__ __align__(128) uint8_t smem[];
    cg::cluster_group cluster = cg::this_cluster();
    const int rank = (int)cluster.block_rank();
    const int S = a.csize;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    const int64_t group = blockIdx.x / S;
    const int64_t bt = group / a.hblocks;
    const int hblk = (int)(group - bt * a.hblocks);
    const int64_t b = bt / a.T;
    const int h0 = hblk * NH;

    uint8_t *sK = smem + OFF_K;
    uint8_t *sQ = smem + OFF_Q;
    float *sT = reinterpret_cast<float *>(smem + OFF_ST);
    uint8_t *sP = smem + OFF_P;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + OFF_TMEM);
    int *sValid = reinterpret_cast<int *>(smem + OFF_VALID);
    float *sCs = reinterpret_cast<float *>(smem + OFF_CS);
    float *sM = reinterpret_cast<float *>(smem + OFF_M);
    float *sL = reinterpret_cast<float *>(smem + OFF_L);
    float *sW = reinterpret_cast<float *>(smem + OFF_W);
    float *sLse = reinterpret_cast<float *>(smem + OFF_LSE);
    float *sIL = reinterpret_cast<float *>(smem + OFF_IL);
    float *sStats = reinterpret_cast<float *>(smem + OFF_STATS);
    float *sBeta = reinterpret_cast<float *>(smem + OFF_BETA);
    const uint32_t bar_q = tc::smem_u32(smem + OFF_BAR);   // Q rows landed
    const uint32_t bar_ld = bar_q + 8;                       // code rows landed
    const uint32_t bar_s = bar_q + 16;                       // S MMA done
    const uint32_t bar_o = bar_q + 24;                       // P V done
    const uint32_t bar_rx = bar_q + 32;                      // other CTAs' slices landed

    const int e = tid & (TM - 1);   // entry of this thread in the tile
    const int qt = tid >> 7;        // which 144 channels of the entry (0..3)
    const int sel = rank * TM + e;

    if (tid == 0) {
        tc::mbar_init(bar_q, NH);    // one arrival per head row
        tc::mbar_init(bar_ld, TM);   // one arrival per entry
        tc::mbar_init(bar_s, 1);
        tc::mbar_init(bar_o, 1);
        tc::mbar_init(bar_rx, 1);
        tc::mbar_init_fence();
    }
    if (warp == 0) tc::tmem_alloc(tmem_slot, TMEM_COLS);
    if (tid < NH) reinterpret_cast<uint32_t *>(sM)[tid] = 0u;   // per-head max |q| (bits), used by 2a
    __syncthreads();
    // cluster barrier, first half: this CTA runs; the wait comes before the first remote store
    if (S > 1) asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
    pdl_wait();   // the set-up above overlaps the previous kernel's tail
    int64_t j, len;
    if constexpr (FP8W) {   // window row sel of the first swa_len
        len = a.swa_len[bt];
        len = len < a.W ? (len > 0 ? len : 0) : a.W;
        j = sel < len ? sel : -1;
    } else {
        j = (sel < a.K) ? (int64_t)__ldg(a.idx + bt * a.K + sel) : -1;   // this thread's entry
        len = a.kv_len ? (int64_t)a.kv_len[bt] : a.N;
        len = len < a.N ? len : a.N;
    }

    // ---- 1. gather: TMA bulk copies of Q rows and the selected code rows.
    // The copies of entry / head e are issued by the thread (e, qt) with
    // qt = (e / 8) mod 4, which spreads them over all 16 warps (8 or 16 each):
    // a warp issues its lanes' bulk copies one after another.
    const bool issuer = qt == ((e >> 3) & 3);
    if (issuer && e < NH) {        // Q rows do not depend on the indices: first
        const uint16_t *qrow = a.q + ((bt * a.H) + h0 + e) * (int64_t)D;
        mbar_arrive_expect_tx(bar_q, D * 2);
        bulk_g2s(tc::smem_u32(smem + OFF_QRAW + e * QRAW_STRIDE), qrow, D * 2, bar_q);
    }
    const bool valid = j >= 0 && j < len;
    if (issuer) {
        if (!valid && j != -1) flag_error(a.err_flag, CSA2_FLAG_BAD_INDEX);
        sValid[e] = valid ? 1 : 0;
        mbar_arrive_expect_tx(bar_ld, (valid && !FP8W) ? D / 2 : 0);
        if (valid && !FP8W)
            bulk_g2s(tc::smem_u32(smem + OFF_CRAW + e * CRAW_STRIDE), a.codes + (b * a.N + j) * (D / 2), D / 2, bar_ld);
    }
    // FP8W: this thread's nine 16-byte groups of its window row, loaded now (their
    // latency overlaps the Q conversion); the same group split as below
    uint4 w8[2][5];
    if constexpr (FP8W) {
        const uint8_t *row = a.kv8 + (b * a.W + (valid ? j : 0)) * (int64_t)D;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int qh = (qt + 2 * h) & 3, nh = qh < 2 ? 5 : 4;
#pragma unroll
            for (int i = 0; i < 5; ++i)
                w8[h][i] = (valid && i < nh) ? __ldg(reinterpret_cast<const uint4 *>(row + 16 * (18 * h + qh + 4 * i)))
                                              : make_uint4(0, 0, 0, 0);
        }
    }
    // the entry's 36 scale bytes as 9 words (consumed only by the dequantiser, so
    // their latency overlaps the Q conversion)
    uint32_t sw[9];
#pragma unroll
    for (int i = 0; i < 9; ++i) sw[i] = 0u;
    if (valid && !FP8W) {
        const uint32_t *srow = reinterpret_cast<const uint32_t *>(a.scales + (b * a.N + j) * (D / 16));
#pragma unroll
        for (int i = 0; i < 9; ++i) sw[i] = __ldg(srow + i);
    }
    bool ok = tc::mbar_wait(bar_q, 0, MAX_POLLS);   // Q first: its conversion overlaps the code copies

    // ---- 2a. staged Q -> registers, per-head power-of-two scale, f16 core-matrix tile [head][channel]
    {
        if constexpr (NH == HB) {
            // lanes: 8 heads x 4 chunk positions, so both the staged-row reads and the
            // tile stores touch every bank once per 128 bytes; a warp pair covers the
            // 72 chunks of its 8 heads (36 each, 9 per thread)
            const int hq = 8 * (warp & 7) + (lane & 7), cpos = lane >> 3, c0 = 36 * (warp >> 3);
            uint32_t *hmax = reinterpret_cast<uint32_t *>(sM);
            uint4 qv[9];
            {
                const uint8_t *qraw = smem + OFF_QRAW + hq * QRAW_STRIDE + (c0 + cpos) * 16;
#pragma unroll
                for (int i = 0; i < 9; ++i) qv[i] = *reinterpret_cast<const uint4 *>(qraw + i * 64);
                float mx = 0.f;
#pragma unroll
                for (int i = 0; i < 9; ++i) {
                    const uint32_t w4[4] = {qv[i].x, qv[i].y, qv[i].z, qv[i].w};
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        mx = fmaxf(mx, fmaxf(fabsf(__uint_as_float(w4[k] << 16)), fabsf(__uint_as_float(w4[k] & 0xFFFF0000u))));
                }
                mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 8));
                mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 16));
                if (cpos == 0) atomicMax(hmax + hq, __float_as_uint(mx));   // |q| >= 0: bit order = value order
            }
            __syncthreads();
            {
                const float mx = __uint_as_float(hmax[hq]);
                int e2 = (mx > 0.f) ? ((int)((__float_as_uint(mx) >> 23) & 0xFF) - 127) : 0;
                int sh = 14 - e2;  // max |q| * 2^sh in [2^14, 2^15)
                sh = sh < -60 ? -60 : (sh > 60 ? 60 : sh);
                const float up = ldexpf(1.0f, sh);
                uint8_t *qdst = sQ + (hq >> 3) * Q_SBO + (hq & 7) * 16 + (c0 + cpos) * 128;
#pragma unroll
                for (int i = 0; i < 9; ++i) {
                    const uint32_t w4[4] = {qv[i].x, qv[i].y, qv[i].z, qv[i].w};
                    uint32_t o[4];
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        o[k] = pack_f16x2(__uint_as_float(w4[k] << 16) * up, __uint_as_float(w4[k] & 0xFFFF0000u) * up);
                    *reinterpret_cast<uint4 *>(qdst + i * 512) = make_uint4(o[0], o[1], o[2], o[3]);
                }
                if (cpos == 0 && c0 == 0) sCs[hq] = a.sm_scale * ldexpf(1.0f, -sh) * 1.4426950408889634f;  // x log2(e)
            }
        } else {
            // 16 rows: 24 threads per row take three chunks each (warps 0..11); the eight
            // lanes of a quarter-warp take eight rows and chunks (2 j + s) mod 24 + 24 m,
            // so both the staged-row reads and the tile stores meet every bank once
            const int G = tid >> 3, jq = tid & 7;
            const bool act = tid < 3 * THREADS / 4;   // warp-uniform
            const int row = 8 * (G & 1) + jq, sg = G >> 1, cb = (2 * jq + sg) % 24;
            uint32_t *hmax = reinterpret_cast<uint32_t *>(sM);
            uint4 qv[3];
            if (act) {
                const uint8_t *qraw = smem + OFF_QRAW + row * QRAW_STRIDE;
#pragma unroll
                for (int m = 0; m < 3; ++m) qv[m] = *reinterpret_cast<const uint4 *>(qraw + (cb + 24 * m) * 16);
                float mx = 0.f;
#pragma unroll
                for (int m = 0; m < 3; ++m) {
                    const uint32_t w4[4] = {qv[m].x, qv[m].y, qv[m].z, qv[m].w};
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        mx = fmaxf(mx, fmaxf(fabsf(__uint_as_float(w4[k] << 16)), fabsf(__uint_as_float(w4[k] & 0xFFFF0000u))));
                }
                atomicMax(hmax + row, __float_as_uint(mx));   // |q| >= 0: bit order = value order
            }
            __syncthreads();
            if (act) {
                const float mx = __uint_as_float(hmax[row]);
                int e2 = (mx > 0.f) ? ((int)((__float_as_uint(mx) >> 23) & 0xFF) - 127) : 0;
                int sh = 14 - e2;  // max |q| * 2^sh in [2^14, 2^15)
                sh = sh < -60 ? -60 : (sh > 60 ? 60 : sh);
                const float up = ldexpf(1.0f, sh);
                uint8_t *qdst = sQ + (row >> 3) * Q_SBO + (row & 7) * 16;
#pragma unroll
                for (int m = 0; m < 3; ++m) {
                    const uint32_t w4[4] = {qv[m].x, qv[m].y, qv[m].z, qv[m].w};
                    uint32_t o[4];
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        o[k] = pack_f16x2(__uint_as_float(w4[k] << 16) * up, __uint_as_float(w4[k] & 0xFFFF0000u) * up);
                    *reinterpret_cast<uint4 *>(qdst + (cb + 24 * m) * 128) = make_uint4(o[0], o[1], o[2], o[3]);
                }
                if (sg == 0) sCs[row] = a.sm_scale * ldexpf(1.0f, -sh) * 1.4426950408889634f;  // x log2(e)
            }
        }
    }
    // ---- 2b. staged codes -> registers (the Khat tile overwrites the staging area)
    // The 36 16-channel groups of an entry are dequantised in two halves (groups
    // 0-17, then 18-35) so that the S MMAs of the first half run while the
    // second half is dequantised.  In half h the thread takes local groups
    // qh, qh + 4, ... (< 18) with qh = (qt + 2h) mod 4: nine groups in all.
    ok = tc::mbar_wait(bar_ld, 0, MAX_POLLS) && ok;
    uint2 cw[2][5] = {};   // per half: up to five groups, 8 code bytes (16 channels) each
    if constexpr (!FP8W) {
        const uint8_t *craw = smem + OFF_CRAW + e * CRAW_STRIDE;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int qh = (qt + 2 * h) & 3, nh = qh < 2 ? 5 : 4;
#pragma unroll
            for (int i = 0; i < 5; ++i)
                cw[h][i] = (valid && i < nh) ? *reinterpret_cast<const uint2 *>(craw + 8 * (18 * h + qh + 4 * i))
                                              : make_uint2(0, 0);
        }
    }
    __syncthreads();
    // ---- 2c. dequantise one half of this thread's groups into the Khat tile
    auto dequant_half = [&](const int h, auto &&before_group) {
        const int qh = (qt + 2 * h) & 3, nh = qh < 2 ? 5 : 4;
        uint8_t *kbase = sK + (e >> 3) * KT_SBO + (e & 7) * 16;
#pragma unroll
        for (int i = 0; i < 5; ++i) {
            before_group(i);
            if (i < nh) {
                const int g = 18 * h + qh + 4 * i;   // group of the entry
                // scale byte g: word g / 4, byte g % 4 (compile-time word choice by a select)
                const uint32_t word = h == 0 ? sw[i] : ((qh >> 1) ? sw[i < 4 ? 5 + i : 8] : sw[4 + i]);
                const int byte = h == 0 ? qh : ((2 + qh) & 3);
                uint32_t r[8] = {0, 0, 0, 0, 0, 0, 0, 0};
                if (FP8W) {
                    e4m3x16_to_f16(w8[h][i], r);   // zero bytes for an invalid entry
                } else if (valid) {
                    const uint32_t sc = e4m3_to_f16x2_bcast((word >> (8 * byte)) & 0xFFu);
                    e2m1x8_scaled(cw[h][i].x, sc, r);
                    e2m1x8_scaled(cw[h][i].y, sc, r + 4);
                }
                *reinterpret_cast<uint4 *>(kbase + (2 * g) * 128) = make_uint4(r[0], r[1], r[2], r[3]);
                *reinterpret_cast<uint4 *>(kbase + (2 * g + 1) * 128) = make_uint4(r[4], r[5], r[6], r[7]);
            }
        }
    };
    // ---- 3. S^T = Khat . Q^T  (M = 128 entries, N = 64 heads, K = 576): 18 k-steps per half
    const uint32_t a0s = tc::smem_u32(sK), b0s = tc::smem_u32(sQ);
    constexpr uint32_t idesc_s = tc::idesc_f16_f32(TM, NH, false, false);
    dequant_half(0, [](int) {});
    tc::fence_async_smem();
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint64_t da_s = tc::desc_noswizzle(a0s, 128, KT_SBO), db_s = tc::desc_noswizzle(b0s, 128, Q_SBO);
    // the first half's 18 MMAs, issued by thread 0 a few at a time between its
    // own second-half groups (four of them), so that the issue does not hold
    // its warp back while the tensor pipe drains
    dequant_half(1, [&](int i) {
        if (tid == 0 && i < 4)
#pragma unroll
            for (int ks = (D / 32) * i / 4; ks < (D / 32) * (i + 1) / 4; ++ks)
                tc::mma_f16(tmem + S_COL, tc::desc_at(da_s, ks * 256), tc::desc_at(db_s, ks * 256), idesc_s, ks > 0);
    });
    tc::fence_async_smem();
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    if (tid == 0) {
#pragma unroll
        for (int ks = D / 32; ks < D / 16; ++ks)
            tc::mma_f16(tmem + S_COL, tc::desc_at(da_s, ks * 256), tc::desc_at(db_s, ks * 256), idesc_s, true);
        tc::commit(bar_s);
    }
    ok = tc::mbar_wait(bar_s, 0, MAX_POLLS) && ok;
    tc::fence_after();
    // This CTA's own rows have landed and HBM is idle for the rest of the launch:
    // hint the same selected rows of the next planes (the layer that attends next
    // with these indices) into L2, so that its launch gathers them from L2.
    if constexpr (!FP8W) {
        if (a.pf_codes && issuer && valid) {
            const int64_t row = b * a.N + j;
            bulk_prefetch_l2(a.pf_codes + row * (D / 2), D / 2);
            const uint8_t *srow = a.pf_scales + row * (D / 16);
            prefetch_l2(srow);
            prefetch_l2(srow + D / 16 - 1);   // the 36 bytes may straddle two lines
        }
    }

    // ---- 4a. S^T -> shared memory, transposed to [head][entry] (the Q tile is free now)
    const int quarter = warp & 3, hh = warp >> 2;   // TMEM lane quarter, group of HPT columns (heads)
    {
        uint32_t r[HPT];
        tmem_ld_n(tmem + ((uint32_t)(32 * quarter) << 16) + S_COL + HPT * hh, r);
        tc::tmem_ld_wait();
        const int ee = 32 * quarter + lane;
        const bool v = ok && sValid[ee];
#pragma unroll
        for (int j4 = 0; j4 < HPT; j4 += 4) {   // four heads' logit factors per 16-byte load
            const float4 cs4 = *reinterpret_cast<const float4 *>(sCs + HPT * hh + j4);
            const float cs[4] = {cs4.x, cs4.y, cs4.z, cs4.w};
#pragma unroll
            for (int u = 0; u < 4; ++u)
                sT[(HPT * hh + j4 + u) * ST_STRIDE + ee] = v ? __uint_as_float(r[j4 + u]) * cs[u] : -INFINITY;
        }
    }
    __syncthreads();

    // ---- 4b. softmax per head over this CTA's entries; P -> f16 core-matrix tile [head][entry]
    {
        constexpr int TPH = THREADS / NH, EPT = TM / TPH;   // threads per head, entries per thread
        const int h = tid / TPH, part = tid % TPH;           // entries TPH i + part
        float z[EPT];
        float mx = -INFINITY;
#pragma unroll
        for (int i = 0; i < EPT; ++i) z[i] = sT[h * ST_STRIDE + TPH * i + part];
#pragma unroll
        for (int i = 0; i < EPT; i += 2) mx = max3f(mx, z[i], z[i + 1]);
#pragma unroll
        for (int o = 1; o < TPH; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
        // an entry at -inf gives ex2(-inf) = 0; a head with no entry (mx = -inf) subtracts 0
        const float mxs = mx == -INFINITY ? 0.f : mx;
        float sum = 0.f;
        uint8_t *pdst = sP + (h >> 3) * P_SBO + (h & 7) * 16;
#pragma unroll
        for (int i = 0; i < EPT; ++i) {
            const float p = ex2(z[i] - mxs);
            const __half ph = __float2half_rn(p);
            sum += __half2float(ph);
            const int en = TPH * i + part;   // entry
            *reinterpret_cast<__half *>(pdst + (en >> 3) * 128 + (en & 7) * 2) = ph;
        }
#pragma unroll
        for (int o = 1; o < TPH; o <<= 1) sum += __shfl_xor_sync(0xFFFFFFFFu, sum, o);
        if (part == 0) {
            sM[h] = mx;
            sL[h] = sum;
            sIL[h] = sum > 0.f ? 1.f / sum : 0.f;
        }
    }
    tc::fence_async_smem();
    tc::fence_before();
    __syncthreads();
    tc::fence_after();

    // ---- 5. O^T = Vhat^T . P^T  (4 blocks of M = 128 channels, N = 64 heads, K = 128 entries),
    // one commit for all (a commit per block measured slower: it held back the next block)
    const int W = DV / S;                      // channels per owner
    const int bpo = W / 128;                   // blocks per owner
    if (tid == 0) {
        const uint64_t da = tc::desc_noswizzle(tc::smem_u32(sK), KT_SBO, 128),
                       db = tc::desc_noswizzle(tc::smem_u32(sP), 128, P_SBO);
        constexpr uint32_t idesc = tc::idesc_f16_f32(TM, NH, true, false);
#pragma unroll
        for (int mb = 0; mb < DV / 128; ++mb)
#pragma unroll
            for (int ks = 0; ks < TM / 16; ++ks)
                tc::mma_f16(tmem + O_COL + mb * NH, tc::desc_at(da, ks * 2 * KT_SBO + mb * 16 * 128),
                            tc::desc_at(db, ks * 256), idesc, ks > 0);
        tc::commit(bar_o);
    }
    if (S > 1) {   // every CTA runs: publish this CTA's (max, sum) per head in every CTA of the cluster
        asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
        if (tid < NH)
            for (int c = 0; c < S; ++c) {
                float *st = cluster.map_shared_rank(sStats, c) + rank * 2 * NH;
                st[tid] = sM[tid];
                st[NH + tid] = sL[tid];
            }
    } else if (tid < NH) {
        sStats[tid] = sM[tid];
        sStats[NH + tid] = sL[tid];
    }
    ok = tc::mbar_wait(bar_o, 0, MAX_POLLS) && ok;
    pdl_launch_dependents();   // the next kernel may launch during the exchange
    tc::fence_after();

    // ---- 6. stage normalised O slices (f16) and (max, sum) for the owners of the channel slices
    // Payload for owner o: [W channels][RSH halves: 64 heads + pad] of O / L, then
    // 64 max + 64 sum (fp32).  A slice owed to another CTA is staged in the Q
    // region below P before the cluster barrier (overlapping the wait for the
    // slowest CTA); after it the TMA engine copies the slices into the owners'
    // shared memory (bulk shared -> remote shared, completing on the owner's
    // mbarrier).  The own slice is written in place (the Khat tile is free).
    const uint32_t slice_bytes = (uint32_t)W * RSHN * 2;
    uint8_t *stage = smem + OFF_Q;             // sT is dead; P stays above the staging
    uint8_t *recv = smem + OFF_K;              // received slices, by source rank
    if (tid == 0) asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar_rx),
                               "r"((uint32_t)(S - 1) * slice_bytes) : "memory");
    float il[HPT];                              // 1 / L of this thread's HPT heads
#pragma unroll
    for (int jj = 0; jj < HPT; ++jj) il[jj] = sIL[HPT * hh + jj];
    // slice o of the sending order (own slice last): stage it, and for another
    // CTA's slice copy it once the cluster barrier has passed
    auto stage_slice = [&](int o) {
        const int oo = (rank + 1 + o) % S;
        uint8_t *dst = (oo == rank) ? recv + (size_t)rank * slice_bytes : stage + (size_t)o * slice_bytes;
        for (int bi = 0; bi < bpo; ++bi) {
            const int mb = oo * bpo + bi;
            uint32_t r[HPT];
            tmem_ld_n(tmem + ((uint32_t)(32 * quarter) << 16) + O_COL + mb * NH + HPT * hh, r);
            tc::tmem_ld_wait();
            uint8_t *row = dst + (size_t)(bi * 128 + 32 * quarter + lane) * (RSHN * 2) + 2 * HPT * hh;
#pragma unroll
            for (int q4 = 0; q4 < HPT / 4; ++q4)
                *reinterpret_cast<uint2 *>(row + 8 * q4) =
                    make_uint2(pack_f16x2(__uint_as_float(r[4 * q4]) * il[4 * q4], __uint_as_float(r[4 * q4 + 1]) * il[4 * q4 + 1]),
                               pack_f16x2(__uint_as_float(r[4 * q4 + 2]) * il[4 * q4 + 2], __uint_as_float(r[4 * q4 + 3]) * il[4 * q4 + 3]));
        }
    };
    auto send_slice = [&](int o) {   // one thread; the slice's staging writes are fenced and synced
        const int oo = (rank + 1 + o) % S;
        uint32_t rdst, rbar;
        const uint32_t ldst = tc::smem_u32(recv + (size_t)rank * slice_bytes);
        asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(rdst) : "r"(ldst), "r"((uint32_t)oo));
        asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(rbar) : "r"(bar_rx), "r"((uint32_t)oo));
        bulk_s2s(rdst, tc::smem_u32(stage + (size_t)o * slice_bytes), slice_bytes, rbar);
        bulk_commit();
    };
    if (S > 1) stage_slice(0);                 // overlaps the wait for the slowest CTA
    if (!ok) flag_error(a.err_flag, CSA2_FLAG_TIMEOUT);   // any thread whose wait gave up
    tc::fence_async_smem();
    tc::fence_before();
    cluster.sync();                            // every CTA's P V is done: its Khat region may be written
    if (S > 1 && tid == 0) send_slice(0);
    // combine weights L_c 2^(m_c - M) / sum_c' L_c' 2^(m_c' - M) from every CTA's (max, sum)
    if (tid < NH) {
        float mc[MAX_S], lc[MAX_S];
        float M = -INFINITY;
#pragma unroll
        for (int c = 0; c < MAX_S; ++c) {
            if (c < S) {
                mc[c] = sStats[c * 2 * NH + tid];
                lc[c] = sStats[c * 2 * NH + NH + tid];
                M = fmaxf(M, mc[c]);
            }
        }
        float L = 0.f;
#pragma unroll
        for (int c = 0; c < MAX_S; ++c) {
            if (c < S) {
                const float wc = (M == -INFINITY || mc[c] == -INFINITY) ? 0.f : lc[c] * ex2(mc[c] - M);
                sW[c * NH + tid] = wc;
                L += wc;
            }
        }
        const float inv = L > 0.f ? 1.f / L : 0.f;
#pragma unroll
        for (int c = 0; c < MAX_S; ++c)
            if (c < S) sW[c * NH + tid] *= inv;
        sLse[tid] = (L > 0.f) ? (M + log2f(L)) * 0.6931471805599453f : -INFINITY;
        if constexpr (FP8W) {
            // merge with the sparse branch: the softmax over both branches' entries
            float beta = 0.f;
            if (a.o_sparse) {
                const float lw = sLse[tid], ls = a.lse_sparse[(bt * a.H) + h0 + tid];
                const float mx = fmaxf(lw, ls);
                float alpha = 0.f, lo = -INFINITY;
                if (mx != -INFINITY) {
                    const float ea = expf(lw - mx), eb = expf(ls - mx);
                    alpha = ea / (ea + eb);
                    beta = eb / (ea + eb);
                    lo = mx + logf(ea + eb);
                }
#pragma unroll
                for (int c = 0; c < MAX_S; ++c)
                    if (c < S) sW[c * NH + tid] *= alpha;
                sLse[tid] = lo;
            }
            sBeta[tid] = beta;
        }
    }
    if (S == 1) {
        // ---- 7'. one CTA holds every entry: O / L straight from TMEM to the
        // output in fp32 (lanes = 32 consecutive channels of one head per
        // store), times the merge weight (1, or the window's share) plus the
        // sparse branch's share
        ok = tc::mbar_wait(bar_rx, 0, MAX_POLLS) && ok;   // (no bytes expected: completes the phase)
        __syncthreads();                                   // the weights of the block above
        if (!ok) flag_error(a.err_flag, CSA2_FLAG_TIMEOUT);   // any thread whose wait gave up
        const int64_t hbase = (bt * a.H) + h0 + HPT * hh;
        // two 128-channel blocks at a time: their sparse-branch values are
        // loaded together, after the TMEM loads' wait
#pragma unroll 1
        for (int mb = 0; mb < DV / 128; mb += 2) {
            uint32_t r[2][HPT];
            tmem_ld_n(tmem + ((uint32_t)(32 * quarter) << 16) + O_COL + mb * NH + HPT * hh, r[0]);
            tmem_ld_n(tmem + ((uint32_t)(32 * quarter) << 16) + O_COL + (mb + 1) * NH + HPT * hh, r[1]);
            tc::tmem_ld_wait();
            float os[2][HPT];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int c = (mb + u) * 128 + 32 * quarter + lane;
#pragma unroll
                for (int jj = 0; jj < HPT; ++jj)
                    os[u][jj] = (FP8W && a.o_sparse) ? a.o_sparse[(hbase + jj) * (int64_t)DV + c] : 0.f;   // may alias out
            }
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int c = (mb + u) * 128 + 32 * quarter + lane;
#pragma unroll
                for (int jj = 0; jj < HPT; ++jj) {
                    const int h = HPT * hh + jj;
                    float v = __uint_as_float(r[u][jj]) * il[jj] * sW[h];
                    if (FP8W) v += sBeta[h] * os[u][jj];
                    a.out[(hbase + jj) * (int64_t)DV + c] = v;
                }
            }
        }
        if (a.lse && tid < NH) a.lse[(bt * a.H) + h0 + tid] = sLse[tid];
        tc::fence_before();
        __syncthreads();
        tc::fence_after();
        if (warp == 0) tc::tmem_dealloc(tmem, TMEM_COLS);
        return;
    }
    for (int o = 1; o + 1 < S; ++o) {   // the other CTAs' slices; the own one stays in TMEM
        stage_slice(o);
        tc::fence_async_smem();
        __syncthreads();
        if (tid == 0) send_slice(o);
    }
    __syncthreads();                           // the combine weights above

    // ---- 7. combine this CTA's channel slice with the weights: its own part
    // straight from TMEM in fp32 (the TMEM lane mapping: lane = channel, 16
    // heads per thread, every store of a warp covers 32 consecutive channels
    // of one head), the other CTAs' parts from their f16 slices
    {
        const int c_lo = rank * W;
        for (int bi = 0; bi < bpo; ++bi) {
            uint32_t r[HPT];
            tmem_ld_n(tmem + ((uint32_t)(32 * quarter) << 16) + O_COL + (rank * bpo + bi) * NH + HPT * hh, r);
            tc::tmem_ld_wait();
            if (bi == 0) ok = tc::mbar_wait(bar_rx, 0, MAX_POLLS) && ok;   // the other CTAs' slices (the own load overlaps)
            const int cl = bi * 128 + 32 * quarter + lane;   // channel within the slice
            const int64_t orow = (bt * a.H) + h0 + HPT * hh;
            constexpr int GH = HPT < 8 ? HPT : 8;            // heads per combine group (four per 8-byte read)
#pragma unroll
            for (int half = 0; half < HPT / GH; ++half) {
                float acc[GH];
#pragma unroll
                for (int i = 0; i < GH; ++i) {
                    const int jj = GH * half + i;
                    acc[i] = __uint_as_float(r[jj]) * il[jj] * sW[rank * NH + HPT * hh + jj];
                }
#pragma unroll
                for (int src = 0; src < MAX_S; ++src) {
                    if (src < S && src != rank) {
                        const uint8_t *rp =
                            recv + (size_t)src * slice_bytes + (size_t)cl * (RSHN * 2) + 2 * HPT * hh + 2 * GH * half;
                        const float *wsrc = sW + src * NH + HPT * hh + GH * half;
#pragma unroll
                        for (int g4 = 0; g4 < GH / 4; ++g4) {
                            const uint2 v = *reinterpret_cast<const uint2 *>(rp + 8 * g4);
                            const float2 a01 = __half22float2(*reinterpret_cast<const __half2 *>(&v.x));
                            const float2 a23 = __half22float2(*reinterpret_cast<const __half2 *>(&v.y));
                            acc[4 * g4] += wsrc[4 * g4] * a01.x;
                            acc[4 * g4 + 1] += wsrc[4 * g4 + 1] * a01.y;
                            acc[4 * g4 + 2] += wsrc[4 * g4 + 2] * a23.x;
                            acc[4 * g4 + 3] += wsrc[4 * g4 + 3] * a23.y;
                        }
                    }
                }
#pragma unroll
                for (int i = 0; i < GH; ++i) {
                    const int64_t oi = (orow + GH * half + i) * (int64_t)DV + c_lo + cl;
                    float v = acc[i];
                    if (FP8W && a.o_sparse) v += sBeta[HPT * hh + GH * half + i] * a.o_sparse[oi];   // may alias out
                    a.out[oi] = v;
                }
            }
        }
        if (rank == 0 && a.lse && tid < NH) a.lse[(bt * a.H) + h0 + tid] = sLse[tid];
    }
    if (!ok) flag_error(a.err_flag, CSA2_FLAG_TIMEOUT);   // any thread whose wait gave up
    if (tid == 0) bulk_wait_read0();           // staging reads done before this CTA may exit
    tc::fence_before();   // every warp's TMEM loads are done before the columns are freed
    __syncthreads();
    tc::fence_after();
    if (warp == 0) tc::tmem_dealloc(tmem, TMEM_COLS);
}


// ---------------------------------------------------------------------------
// Many query tokens: one CTA per (token, 64 heads) over all of its K <= 512
// selected entries in one pass with an online softmax, no cluster merge (used
// when a launch has enough (token, head-block) items to fill the GPU on its
// own, e.g. a prefill chunk).  Persistent: at most one CTA per SM, taking the
// items blockIdx.x, + gridDim.x, ...  512 threads; the same 128-entry tile
// and MMA shapes as above.  Per 128-entry tile t:
//  - the entry's 288 code bytes were loaded into registers while tile t-1
//    was computed (the first tile of an item: during the previous item's last
//    tile), 8 bytes per thread and load, four lanes per entry (lanes e,
//    e + 8, e + 16, e + 24), so one warp load touches 8 rows with one 32-byte
//    sector each and a quarter-warp's 16-byte tile stores cover 8 entries;
//    each lane loads three of the entry's nine scale words, shared by shuffles;
//  - the 576 channels are dequantised into the Khat tile in two parts:
//    channels 0..255 once P V of tile t-1 has read its first two channel
//    blocks (its last two still running), the rest once it is done, the first
//    part's S MMAs running meanwhile: S^T_t = Khat . Q^T into TMEM columns
//    [0, 64);
//  - z = S * c per head; the running maximum M moves only when a tile's
//    maximum exceeds it by more than 8 (log2 units), and then O^T and the
//    running sum are scaled by 2^(M_old - M_new), so P = 2^(z - M) <= 256;
//  - P_t in f16, laid out MN-major in the Khat tile's rotary channels (dead
//    once S_t is done); O^T += Vhat_t^T . P_t^T into TMEM columns [64, 320)
//    is issued at the start of tile t+1, ahead of its dequantisation.
// Once an item's last S is done the Q tile is free: the next item's Q rows
// (bf16) are copied into it and, after the item's last P V, converted there
// in place.  Finally out = O / L and lse = (M + log2 L) ln 2 per head, L
// summed over the f16-rounded P as the MMAs consumed it; O stays in TMEM and
// is stored during the next item's first tile.
constexpr uint32_t TK_OFF_K = 0;
constexpr uint32_t TK_OFF_Q = KT_BYTES;                        // Q tile
constexpr uint32_t TK_P_IN_GROUP = (DV / 8) * 128;             // P: the rotary core matrices of each 8-entry group
constexpr uint32_t TK_OFF_BAR = TK_OFF_Q + Q_BYTES;            // mbarriers: Q rows, S, P V
constexpr uint32_t TK_OFF_TMEM = TK_OFF_BAR + 32;
constexpr uint32_t TK_OFF_ROW = TK_OFF_TMEM + 16;              // int64[512] KV row of each selected entry, -1 if none
constexpr uint32_t TK_OFF_QMAX = TK_OFF_ROW + MAX_S * TM * 8;  // uint[64] per-head max |q| (bits)
constexpr uint32_t TK_OFF_CS = TK_OFF_QMAX + HB * 4;           // float[64] logit factor per head
constexpr uint32_t TK_OFF_PART = TK_OFF_CS + HB * 4;           // float[4][64] per lane quarter
constexpr uint32_t TK_OFF_M = TK_OFF_PART + 4 * HB * 4;        // float[64] running max (log2 domain)
constexpr uint32_t TK_OFF_L = TK_OFF_M + HB * 4;               // float[64] running sum
constexpr uint32_t TK_OFF_ALPHA = TK_OFF_L + HB * 4;           // float[64] rescale factor of this tile
constexpr uint32_t TK_OFF_ILP = TK_OFF_ALPHA + HB * 4;         // float[64] 1 / L of the previous item
constexpr uint32_t TK_SMEM = TK_OFF_ILP + HB * 4;
constexpr uint32_t TK_S_COL = 0, TK_O_COL = HB;                // S^T: 64 columns; O^T: 4 x 64
constexpr float TK_MAX_SLACK = 8.f;                            // P <= 2^8 between rescales
static_assert((HB / 8) * 128 == KT_SBO - TK_P_IN_GROUP, "P fills the rotary channels of an 8-entry group");
static_assert(TK_O_COL + (DV / 128) * HB <= TMEM_COLS, "TMEM columns");
static_assert(TK_SMEM <= 227 * 1024, "shared memory");

// Reduce-scatter of 16 values over the 32 lanes of a warp: afterwards lanes l
// and l ^ 1 both hold the reduction over all lanes of value (l >> 1) & 15.
template <bool MAX>
__device__ __forceinline__ float lane_reduce16(float (&v)[16], int lane) {
    auto op = [](float x, float y) { return MAX ? fmaxf(x, y) : x + y; };
    auto step = [&](auto half_c, int d) {
        constexpr int half = decltype(half_c)::value;
        const bool up = (lane & d) != 0;
#pragma unroll
        for (int j = 0; j < half; ++j) {
            const float send = up ? v[j] : v[j + half];
            const float keep = up ? v[j + half] : v[j];
            v[j] = op(keep, __shfl_xor_sync(0xFFFFFFFFu, send, d));
        }
    };
    step(std::integral_constant<int, 8>{}, 16);
    step(std::integral_constant<int, 4>{}, 8);
    step(std::integral_constant<int, 2>{}, 4);
    step(std::integral_constant<int, 1>{}, 2);
    return op(v[0], __shfl_xor_sync(0xFFFFFFFFu, v[0], 1));
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
            taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
        "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__global__ void __launch_bounds__(THREADS, 1) sparse_attn_tc_tokens_kernel(TcArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int ntiles = (a.K + TM - 1) / TM;

    uint8_t *sK = smem + TK_OFF_K;
    uint8_t *sQ = smem + TK_OFF_Q;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + TK_OFF_TMEM);
    int64_t *sRow = reinterpret_cast<int64_t *>(smem + TK_OFF_ROW);
    uint32_t *sQmax = reinterpret_cast<uint32_t *>(smem + TK_OFF_QMAX);
    float *sCs = reinterpret_cast<float *>(smem + TK_OFF_CS);
    float *sPart = reinterpret_cast<float *>(smem + TK_OFF_PART);
    float *sM = reinterpret_cast<float *>(smem + TK_OFF_M);
    float *sL = reinterpret_cast<float *>(smem + TK_OFF_L);
    float *sAlpha = reinterpret_cast<float *>(smem + TK_OFF_ALPHA);
    float *sILp = reinterpret_cast<float *>(smem + TK_OFF_ILP);
    const uint32_t bar_q = tc::smem_u32(smem + TK_OFF_BAR);   // Q rows landed
    const uint32_t bar_s = bar_q + 8;                           // S MMAs of a tile done
    const uint32_t bar_o = bar_q + 16;                          // P V MMAs of a tile done
    const uint32_t bar_o1 = bar_q + 24;                         // its first two channel blocks done

    // dequantisation: entry de of a tile, lane dq of its four (lanes e, e + 8, e + 16, e + 24:
    // a quarter-warp holds eight entries, so its 16-byte tile stores meet every bank once);
    // channel groups dq + 4 j
    const int de = 8 * warp + (lane & 7), dq = lane >> 3;
    const int quarter = warp & 3, hh = warp >> 2;    // TMEM lane quarter, 16-head group

    if (tid == 0) {
        tc::mbar_init(bar_q, HB);    // one arrival per head row
        tc::mbar_init(bar_s, 1);
        tc::mbar_init(bar_o, 1);
        tc::mbar_init(bar_o1, 1);
        tc::mbar_init_fence();
    }
    if (warp == 0) tc::tmem_alloc(tmem_slot, TMEM_COLS);
    if (tid < HB) {
        sQmax[tid] = 0u;
        sM[tid] = -INFINITY;
        sL[tid] = 0.f;
    }
    __syncthreads();
    pdl_wait();   // the set-up above overlaps the previous kernel's tail

    // item -> (token bt, sequence b, first head h0)
    int64_t item = blockIdx.x, bt, b;
    int h0;
    auto coords = [&](int64_t it, int64_t &bt_, int64_t &b_, int &h0_) {
        bt_ = it / a.hblocks;
        h0_ = (int)(it - bt_ * a.hblocks) * HB;
        b_ = bt_ / a.T;
    };
    // the Q rows of an item: one bulk copy per head row into the Q tile (bf16 rows of
    // 1152 bytes, converted there in place), issuers spread over the warps
    auto issue_q = [&](int64_t bt_, int h0_) {
        if ((tid & 7) == 0) {
            const int hr = tid >> 3;
            mbar_arrive_expect_tx(bar_q, D * 2);
            bulk_g2s(tc::smem_u32(sQ + hr * (D * 2)), a.q + ((bt_ * a.H) + h0_ + hr) * (int64_t)D, D * 2, bar_q);
        }
    };
    // the KV row of selected entry e of token bt_, -1 if none; bad indices flagged if asked
    auto row_at = [&](int64_t bt_, int64_t b_, int e, bool flag) -> int64_t {
        int64_t len = a.kv_len ? (int64_t)a.kv_len[bt_] : a.N;
        len = len < a.N ? len : a.N;
        const int64_t j = (e < a.K) ? (int64_t)__ldg(a.idx + bt_ * a.K + e) : -1;
        const bool v = j >= 0 && j < len;
        if (flag && !v && j != -1) flag_error(a.err_flag, CSA2_FLAG_BAD_INDEX);
        return v ? b_ * a.N + j : -1;
    };
    // the KV row of this thread's selected entry (entry tid < ntiles * TM <= THREADS)
    auto row_of = [&](int64_t bt_, int64_t b_) -> int64_t { return row_at(bt_, b_, tid, true); };
    coords(item, bt, b, h0);
    issue_q(bt, h0);
    if (tid < ntiles * TM) sRow[tid] = row_of(bt, b);
    __syncthreads();

    // this thread's code bytes of one tile, straight into registers, and three of
    // the entry's nine scale words (dq, dq + 4 and, for dq = 0, 8): the four lanes
    // of an entry share them by shuffles, so a warp load touches 8 rows once
    uint2 cw[9];
    uint32_t sw3[3], sw[9];
    auto load_row = [&](int64_t r) {
        if (r >= 0) {
            const uint2 *crow = reinterpret_cast<const uint2 *>(a.codes + r * (D / 2));
            const uint32_t *srow = reinterpret_cast<const uint32_t *>(a.scales + r * (D / 16));
#pragma unroll
            for (int j = 0; j < 9; ++j) cw[j] = __ldg(crow + dq + 4 * j);
            sw3[0] = __ldg(srow + dq);
            sw3[1] = __ldg(srow + 4 + dq);
            sw3[2] = __ldg(srow + 8 - 8 * (dq != 0));   // word 8 for lane 0 (the others reload word 0, unused)
        } else {
#pragma unroll
            for (int j = 0; j < 9; ++j) cw[j] = make_uint2(0u, 0u);
            sw3[0] = sw3[1] = sw3[2] = 0u;
        }
    };
    auto load_tile = [&](int t) { load_row(sRow[t * TM + de]); };
    // the entry's nine scale words in every lane of the entry (word j from its lane with dq = j mod 4)
    auto share_scales = [&]() {
#pragma unroll
        for (int j = 0; j < 9; ++j)
            sw[j] = __shfl_sync(0xFFFFFFFFu, j < 4 ? sw3[0] : (j < 8 ? sw3[1] : sw3[2]), (lane & 7) | ((j & 3) << 3));
    };
    // dequantise channel groups dq + 4 j, j in [j0, j1), of entry de into the Khat tile
    uint8_t *kbase = sK + warp * KT_SBO + (lane & 7) * 16;   // (de >> 3) == warp
    auto dequant = [&](auto j0_c, auto j1_c, bool valid, auto &&before_group) {
        constexpr int j0 = decltype(j0_c)::value, j1 = decltype(j1_c)::value;
#pragma unroll
        for (int j = j0; j < j1; ++j) {
            before_group(j - j0);
            const int g = dq + 4 * j;
            uint32_t r[8] = {0, 0, 0, 0, 0, 0, 0, 0};
            if (valid) {
                const uint32_t sc = e4m3_to_f16x2_bcast((sw[j] >> (8 * dq)) & 0xFFu);
                e2m1x8_scaled(cw[j].x, sc, r);
                e2m1x8_scaled(cw[j].y, sc, r + 4);
            }
            *reinterpret_cast<uint4 *>(kbase + (2 * g) * 128) = make_uint4(r[0], r[1], r[2], r[3]);
            *reinterpret_cast<uint4 *>(kbase + (2 * g + 1) * 128) = make_uint4(r[4], r[5], r[6], r[7]);
        }
    };
    const uint32_t tmem = *tmem_slot;
    const uint32_t a0s = tc::smem_u32(sK), b0s = tc::smem_u32(sQ);
    constexpr uint32_t idesc_s = tc::idesc_f16_f32(TM, HB, false, false);
    constexpr uint32_t idesc_o = tc::idesc_f16_f32(TM, HB, true, true);
    constexpr int KS_A = 16;   // groups 0..15 (channels 0..255: the value blocks P V reads first) go first
    const uint32_t s_lane = tmem + ((uint32_t)(32 * quarter) << 16);

    // operand descriptors: one base each, advanced by constant offsets per MMA
    const uint64_t da_s = tc::desc_noswizzle(a0s, 128, KT_SBO), db_s = tc::desc_noswizzle(b0s, 128, Q_SBO);
    const uint64_t da_o = tc::desc_noswizzle(a0s, KT_SBO, 128), db_o = tc::desc_noswizzle(a0s + TK_P_IN_GROUP, KT_SBO, 128);
    // P V of tile tp, value channel block mb, entry steps [ks0, ks1): O^T += Vhat^T . P^T
    auto pv_mmas = [&](int tp, int mb, int ks0, int ks1) {
#pragma unroll
        for (int ks = ks0; ks < ks1; ++ks)
            tc::mma_f16(tmem + TK_O_COL + mb * HB, tc::desc_at(da_o, ks * 2 * KT_SBO + mb * 16 * 128),
                        tc::desc_at(db_o, ks * 2 * KT_SBO), idesc_o, tp > 0 || ks > 0);
    };

    uint32_t cnt_q = 0, cnt_s = 0, cnt_o = 0, cnt_o1 = 0;   // completed phases waited on, per barrier
    bool ok = true;
    // out = O / L of the previous item, channel blocks [mb0, mb1) (lanes = 32
    // consecutive channels of one head per store).  O stays in TMEM until the
    // next item's first P V, so the stores of one item are spread over the
    // next item's first tile.
    int64_t prev_hbase = -1;   // first (token, head) row of the previous item, -1 if none
    auto emit_out = [&](int mb0, int mb1) {
        for (int mb = mb0; mb < mb1; ++mb) {
            uint32_t r[16];
            tc::tmem_ld16(s_lane + TK_O_COL + mb * HB + 16 * hh, r);
            tc::tmem_ld_wait();
            const int c = mb * 128 + 32 * quarter + lane;
#pragma unroll
            for (int jj = 0; jj < 16; ++jj)
                a.out[(prev_hbase + 16 * hh + jj) * (int64_t)DV + c] = __uint_as_float(r[jj]) * sILp[16 * hh + jj];
        }
    };
    // ---- Q (bf16 rows in the Q tile) -> registers -> per-head power-of-two scale -> the
    // f16 core-matrix tile in place.  Thread (G = tid / 8, j = tid mod 8) takes row
    // 8 (G mod 8) + j, chunks (j + G / 8) mod 8 + 8 k: the eight lanes of a quarter-warp
    // read eight rows at eight chunk residues and write eight rows of one core matrix,
    // so neither side meets a bank twice.  Every raw row is read before the barrier
    // that publishes the maxima, and written over only after it.
    auto convert_q = [&]() {
        ok = tc::mbar_wait(bar_q, cnt_q & 1, MAX_POLLS) && ok;
        ++cnt_q;
        const int qG = tid >> 3, qj = tid & 7;
        const int qh = 8 * (qG & 7) + qj, qc0 = (qj + (qG >> 3)) & 7;
        uint4 qv[9];
#pragma unroll
        for (int k = 0; k < 9; ++k) qv[k] = *reinterpret_cast<const uint4 *>(sQ + qh * (D * 2) + (qc0 + 8 * k) * 16);
        // max |q| on the bf16 bit patterns: a finite magnitude orders as its 15 low bits
        // (two per word, compared as unsigned 16-bit halves); four independent chains
        uint32_t m4[4] = {0u, 0u, 0u, 0u};
#pragma unroll
        for (int k = 0; k < 9; ++k) {
            const uint32_t w4[4] = {qv[k].x, qv[k].y, qv[k].z, qv[k].w};
#pragma unroll
            for (int u = 0; u < 4; ++u) m4[u] = __vmaxu2(m4[u], w4[u] & 0x7FFF7FFFu);
        }
        uint32_t mb2 = __vmaxu2(__vmaxu2(m4[0], m4[1]), __vmaxu2(m4[2], m4[3]));
        mb2 = max(mb2 & 0xFFFFu, mb2 >> 16);
        atomicMax(sQmax + qh, mb2 << 16);   // the float bits of |q|: bit order = value order
        __syncthreads();
        const float mx = __uint_as_float(sQmax[qh]);
        const int e2 = (mx > 0.f) ? ((int)((__float_as_uint(mx) >> 23) & 0xFF) - 127) : 0;
        int sh = 14 - e2;   // max |q| * 2^sh in [2^14, 2^15)
        sh = sh < -60 ? -60 : (sh > 60 ? 60 : sh);
        const float up = ldexpf(1.0f, sh);
        uint8_t *qdst = sQ + (qh >> 3) * Q_SBO + (qh & 7) * 16;
#pragma unroll
        for (int k = 0; k < 9; ++k) {
            const uint32_t w4[4] = {qv[k].x, qv[k].y, qv[k].z, qv[k].w};
            uint32_t o[4];
#pragma unroll
            for (int u = 0; u < 4; ++u)
                o[u] = pack_f16x2(__uint_as_float(w4[u] << 16) * up, __uint_as_float(w4[u] & 0xFFFF0000u) * up);
            *reinterpret_cast<uint4 *>(qdst + (qc0 + 8 * k) * 128) = make_uint4(o[0], o[1], o[2], o[3]);
        }
        if (qG < 8) sCs[qh] = a.sm_scale * ldexpf(1.0f, -sh) * 1.4426950408889634f;   // x log2(e)
    };
    bool tile0_loaded = false;
    for (;;) {   // the items of this CTA: blockIdx.x, + gridDim.x, ...
        // the next item of this CTA, if any: the code rows of its first tile and its Q
        // rows are fetched during this item's last tile
        const int64_t nitem = item + gridDim.x;
        const bool has_next = nitem < a.items;
        int64_t nbt = 0, nb = 0;
        int nh0 = 0;
        if (has_next) coords(nitem, nbt, nb, nh0);
        if (!tile0_loaded) load_tile(0);
        convert_q();
        for (int t = 0; t < ntiles; ++t) {
            // P V of tile t-1 is issued here: its first two channel blocks, then the
            // other two a few MMAs at a time between thread 0's first groups (the issue
            // waits on the tensor pipe).  Channels 0..255 are dequantised once the
            // first two blocks have read them, the rest once all of it is done.
            if (t > 0) {
                if (tid == 0) {
                    pv_mmas(t - 1, 0, 0, TM / 16);
                    pv_mmas(t - 1, 1, 0, TM / 16);
                    tc::commit(bar_o1);
                }
                ok = tc::mbar_wait(bar_o1, cnt_o1 & 1, MAX_POLLS) && ok;
                ++cnt_o1;
            }
            tc::fence_after();
            const bool valid = sRow[t * TM + de] >= 0;
            if (t == 0 && prev_hbase >= 0) emit_out(0, 2);
            share_scales();
            dequant(std::integral_constant<int, 0>{}, std::integral_constant<int, 4>{}, valid, [&](int i) {
                if (t > 0 && tid == 0) pv_mmas(t - 1, 2 + (i >> 1), (i & 1) * (TM / 32), ((i & 1) + 1) * (TM / 32));
            });
            if (t > 0 && tid == 0) tc::commit(bar_o);
            tc::fence_async_smem();
            tc::fence_before();
            __syncthreads();
            tc::fence_after();
            if (t > 0) {
                ok = tc::mbar_wait(bar_o, cnt_o & 1, MAX_POLLS) && ok;
                ++cnt_o;
            }
            tc::fence_after();
            if (t == 0 && prev_hbase >= 0) emit_out(2, 4);
            // the first part's 16 MMAs, four before each of thread 0's first four later groups
            dequant(std::integral_constant<int, 4>{}, std::integral_constant<int, 9>{}, valid, [&](int i) {
                if (tid == 0 && i < 4)
#pragma unroll
                    for (int ks = KS_A * i / 4; ks < KS_A * (i + 1) / 4; ++ks)
                        tc::mma_f16(tmem + TK_S_COL, tc::desc_at(da_s, ks * 256), tc::desc_at(db_s, ks * 256), idesc_s,
                                    ks > 0);
            });
            tc::fence_async_smem();
            tc::fence_before();
            __syncthreads();
            tc::fence_after();
            if (tid == 0) {
#pragma unroll
                for (int ks = KS_A; ks < D / 16; ++ks)
                    tc::mma_f16(tmem + TK_S_COL, tc::desc_at(da_s, ks * 256), tc::desc_at(db_s, ks * 256), idesc_s, true);
                tc::commit(bar_s);
            }
            if (t + 1 < ntiles)
                load_tile(t + 1);   // lands while this tile is finished
            else if (has_next)
                load_row(row_at(nbt, nb, de, false));   // the next item's first tile
            ok = tc::mbar_wait(bar_s, cnt_s & 1, MAX_POLLS) && ok;
            ++cnt_s;
            tc::fence_after();
            if (t + 1 == ntiles && has_next) issue_q(nbt, nh0);   // the Q tile is free once the last S is done


            // logits of this warp's 32 entries x 16 heads; the tile's per-head maximum
            uint32_t r[16];
            tc::tmem_ld16(s_lane + TK_S_COL + 16 * hh, r);
            tc::tmem_ld_wait();
            const int ee = 32 * quarter + lane;
            const bool v = ok && sRow[t * TM + ee] >= 0;
            // The running maxima move only when some logit of the tile exceeds
            // them by more than the slack (also the first finite one: M = -inf).
            // Each thread tests its own 16 values; when no thread finds one, the
            // tile's per-head maxima are not needed and M, L and O stay as they are.
            bool any_ex;
            {
                float z[16];
                bool exceed = false;
#pragma unroll
                for (int j4 = 0; j4 < 16; j4 += 4) {   // four heads' logit factors and maxima per 16-byte load
                    const float4 cs4 = *reinterpret_cast<const float4 *>(sCs + 16 * hh + j4);
                    const float4 mx4 = *reinterpret_cast<const float4 *>(sM + 16 * hh + j4);
                    const float cs[4] = {cs4.x, cs4.y, cs4.z, cs4.w}, mo[4] = {mx4.x, mx4.y, mx4.z, mx4.w};
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        z[j4 + u] = v ? __uint_as_float(r[j4 + u]) * cs[u] : -INFINITY;
                        exceed |= z[j4 + u] > mo[u] + TK_MAX_SLACK;
                    }
                }
                any_ex = __syncthreads_or(exceed) != 0;
                if (any_ex) {
                    const float m = lane_reduce16<true>(z, lane);
                    if ((lane & 1) == 0) sPart[quarter * HB + 16 * hh + (lane >> 1)] = m;
                }
            }
            bool any_resc = false;
            if (any_ex) {
                __syncthreads();
                bool resc = false;
                if (tid < HB) {
                    const float mt = fmaxf(fmaxf(sPart[tid], sPart[HB + tid]), fmaxf(sPart[2 * HB + tid], sPart[3 * HB + tid]));
                    const float mo = sM[tid];
                    float al = 1.f;
                    if (mt > mo + TK_MAX_SLACK) {   // also the first finite maximum (mo = -inf)
                        resc = mo != -INFINITY;
                        al = resc ? ex2(mo - mt) : 0.f;
                        sM[tid] = mt;
                        sL[tid] *= al;
                    }
                    sAlpha[tid] = al;
                }
                tc::fence_before();
                any_resc = __syncthreads_or(resc) != 0;
                tc::fence_after();
            }
            if (any_resc) {   // O^T *= alpha per head column (P V of t-1 is complete)
#pragma unroll 1
                for (int mb = 0; mb < DV / 128; ++mb) {
                    uint32_t o[16];
                    const uint32_t ta = s_lane + TK_O_COL + mb * HB + 16 * hh;
                    tc::tmem_ld16(ta, o);
                    tc::tmem_ld_wait();
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj) o[jj] = __float_as_uint(__uint_as_float(o[jj]) * sAlpha[16 * hh + jj]);
                    tmem_st16(ta, o);
                }
                tmem_st_wait();
            }
            // P_t = 2^(z - M) in f16 into the rotary channels of the Khat tile (MN-major: 8 heads per 16 bytes); row sums
            {
                float pf[16];
                uint32_t pk[8];
                if (v) {   // a valid entry reached its heads' running maxima: they are finite
#pragma unroll
                    for (int j4 = 0; j4 < 16; j4 += 4) {   // four heads' maxima and logit factors per 16-byte load
                        const float4 mx4 = *reinterpret_cast<const float4 *>(sM + 16 * hh + j4);
                        const float4 cs4 = *reinterpret_cast<const float4 *>(sCs + 16 * hh + j4);
                        const float mx[4] = {mx4.x, mx4.y, mx4.z, mx4.w}, cs[4] = {cs4.x, cs4.y, cs4.z, cs4.w};
#pragma unroll
                        for (int u = 0; u < 4; u += 2) {
                            const float z0 = __uint_as_float(r[j4 + u]) * cs[u];
                            const float z1 = __uint_as_float(r[j4 + u + 1]) * cs[u + 1];
                            const __half2 hp = __floats2half2_rn(ex2(z0 - mx[u]), ex2(z1 - mx[u + 1]));
                            pk[(j4 + u) / 2] = *reinterpret_cast<const uint32_t *>(&hp);
                            const float2 back = __half22float2(hp);
                            pf[j4 + u] = back.x;
                            pf[j4 + u + 1] = back.y;
                        }
                    }
                } else {
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj) pf[jj] = 0.f;
#pragma unroll
                    for (int jj = 0; jj < 8; ++jj) pk[jj] = 0u;
                }
                uint8_t *pdst = sK + (ee >> 3) * KT_SBO + TK_P_IN_GROUP + (ee & 7) * 16;
                *reinterpret_cast<uint4 *>(pdst + (2 * hh) * 128) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                *reinterpret_cast<uint4 *>(pdst + (2 * hh + 1) * 128) = make_uint4(pk[4], pk[5], pk[6], pk[7]);
                const float sum = lane_reduce16<false>(pf, lane);
                if ((lane & 1) == 0) sPart[quarter * HB + 16 * hh + (lane >> 1)] = sum;
            }
            tc::fence_async_smem();
            tc::fence_before();
            __syncthreads();
            tc::fence_after();
            if (tid < HB) sL[tid] += (sPart[tid] + sPart[HB + tid]) + (sPart[2 * HB + tid] + sPart[3 * HB + tid]);
        }
        if (tid == 0) {   // P V of the last tile
            for (int mb = 0; mb < DV / 128; ++mb) pv_mmas(ntiles - 1, mb, 0, TM / 16);
            tc::commit(bar_o);
        }
        ok = tc::mbar_wait(bar_o, cnt_o & 1, MAX_POLLS) && ok;
        ++cnt_o;
        tc::fence_after();
        // 1 / L and lse of this item; its O is stored during the next item's first tile
        if (tid < HB) {
            const float l = sL[tid], mx = sM[tid];
            sILp[tid] = l > 0.f ? 1.f / l : 0.f;
            if (a.lse)
                a.lse[(bt * a.H) + h0 + tid] = (l > 0.f && mx != -INFINITY) ? (mx + log2f(l)) * 0.6931471805599453f : -INFINITY;
        }
        prev_hbase = (bt * a.H) + h0;
        int64_t nrow = -1;
        if (has_next && tid < ntiles * TM) nrow = row_of(nbt, nb);
        // one decision for the whole CTA (a timeout in any thread ends its work); the
        // barrier also completes sILp and every read of this item's sL and sM
        tc::fence_before();
        const bool stop = __syncthreads_or(!ok) != 0 || !has_next;
        tc::fence_after();
        if (stop) {
            // (after a timeout the next item's Q copy is still waited for: no copy
            // into this CTA's shared memory may be in flight when it exits)
            if (has_next) (void)tc::mbar_wait(bar_q, cnt_q & 1, MAX_POLLS);
            emit_out(0, DV / 128);
            break;
        }
        if (tid < ntiles * TM) sRow[tid] = nrow;
        if (tid < HB) {
            sQmax[tid] = 0u;
            sM[tid] = -INFINITY;
            sL[tid] = 0.f;
        }
        __syncthreads();
        item = nitem;
        bt = nbt;
        b = nb;
        h0 = nh0;
        tile0_loaded = true;
    }
    if (!ok) flag_error(a.err_flag, CSA2_FLAG_TIMEOUT);   // any thread whose wait gave up
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    if (warp == 0) tc::tmem_dealloc(tmem, TMEM_COLS);
}
}  // namespace

bool sparse_attn_tc_supported(int D_, int dv, int H, int K) {
    return D_ == D && dv == DV && H % HB == 0 && K >= 1 && K <= MAX_S * TM;
}

// Entries split over a cluster of 1, 2 or 4 CTAs (the channel slices divide 512).
static int cluster_size_for(int entries) {
    const int tiles = (entries + TM - 1) / TM;
    return tiles <= 1 ? 1 : (tiles <= 2 ? 2 : 4);
}

template <bool FP8W, int NH>
static csa2_status launch_tc(TcArgs &a, int B, int entries, cudaStream_t stream) {
    static bool smem_set[64];
    CSA2_CUDA_CALL(ensure_smem_limit((const void *)sparse_attn_tc_kernel<FP8W, NH>, (int)SMEM, smem_set),
                   "sparse_attn_tc: smem attribute");
    a.csize = cluster_size_for(entries);
    a.hblocks = a.H / NH;
    const int64_t grid = (int64_t)B * a.T * a.hblocks * a.csize;
    if (grid > 0x7FFFFFFF) {
        set_error("sparse_attn_tc: grid too large");
        return CSA2_ERR_UNSUPPORTED;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3(THREADS, 1, 1);
    cfg.dynamicSmemBytes = SMEM;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = a.csize;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1] = pdl_attribute();
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    CSA2_CUDA_CALL(cudaLaunchKernelEx(&cfg, sparse_attn_tc_kernel<FP8W, NH>, a), "sparse_attn_tc_kernel launch");
    CSA2_LAUNCH_CHECK("sparse_attn_tc_kernel");
    return CSA2_OK;
}

static csa2_status launch_tc_tokens(TcArgs &a, int B, cudaStream_t stream) {
    static bool smem_set[64];
    CSA2_CUDA_CALL(ensure_smem_limit((const void *)sparse_attn_tc_tokens_kernel, (int)TK_SMEM, smem_set),
                   "sparse_attn_tc_tokens: smem attribute");
    a.hblocks = a.H / HB;
    a.csize = 1;
    a.items = (int64_t)B * a.T * a.hblocks;
    const int64_t grid = a.items < num_sms() ? a.items : num_sms();   // persistent: one CTA per SM at most
    CSA2_CUDA_CALL(launch_pdl(sparse_attn_tc_tokens_kernel, dim3((unsigned)grid), dim3(THREADS), TK_SMEM, stream, a),
                   "sparse_attn_tc_tokens_kernel launch");
    CSA2_LAUNCH_CHECK("sparse_attn_tc_tokens_kernel");
    return CSA2_OK;
}

// Many (token, 64-head) items: more than a quarter of the SMs, i.e. the cluster
// kernel's grid (up to four CTAs per item) would exceed one wave.
bool use_token_kernel(int64_t items) { return items * 4 > (int64_t)num_sms(); }

csa2_status launch_sparse_attn_tc(int B, int T, int H, int K, int64_t N, const void *q, const uint8_t *codes,
                                  const uint8_t *scales, const int32_t *idx, const int32_t *kv_len, float sm_scale,
                                  float *out, float *lse, uint32_t *err_flag, const uint8_t *pf_codes,
                                  const uint8_t *pf_scales, cudaStream_t stream) {
    TcArgs a = {};
    a.pf_codes = pf_codes; a.pf_scales = pf_scales;
    a.T = T; a.H = H; a.K = K; a.N = N;
    a.q = (const uint16_t *)q; a.codes = codes; a.scales = scales; a.idx = idx; a.kv_len = kv_len;
    a.sm_scale = sm_scale; a.out = out; a.lse = lse; a.err_flag = err_flag;
    const int64_t items = (int64_t)B * T * (H / HB);
    if (use_token_kernel(items)) return launch_tc_tokens(a, B, stream);
    // few tokens: each token's heads split over four CTA groups of 16 while that grid
    // still fits one wave of SMs (every per-head phase of a CTA shrinks fourfold)
    if (items * 4 * cluster_size_for(K) <= (int64_t)num_sms()) return launch_tc<false, HB / 4>(a, B, K, stream);
    return launch_tc<false, HB>(a, B, K, stream);
}

csa2_status launch_swa_attn_tc(int B, int T, int H, const void *q, const uint8_t *kv8, int W, const int32_t *swa_len,
                               float sm_scale, const float *o_sparse, const float *lse_sparse, float *out, float *lse,
                               uint32_t *err_flag, cudaStream_t stream) {
    TcArgs a = {};
    a.T = T; a.H = H; a.K = W; a.N = W;
    a.q = (const uint16_t *)q; a.sm_scale = sm_scale; a.out = out; a.lse = lse; a.err_flag = err_flag;
    a.kv8 = kv8; a.W = W; a.swa_len = swa_len; a.o_sparse = o_sparse; a.lse_sparse = lse_sparse;
    return launch_tc<true, HB>(a, B, W, stream);
}

}  // namespace csa2

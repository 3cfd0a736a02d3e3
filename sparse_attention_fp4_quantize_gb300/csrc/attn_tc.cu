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
//  1. The TMA engine gathers the operands: one bulk copy per Q head row
//     (1152 B) and one per selected entry's code row (288 B), completing on
//     one mbarrier; the 36-byte scale rows (not 16-byte sized) are plain loads.
//  2. Q (bf16) is scaled per head by a power of two into f16 (exact; the scale
//     is folded into the logit factor); the entries are dequantised once
//     (E2M1 x E4M3 -> exact f16) into a no-swizzle core-matrix tile.
//  3. S^T [128 entries x 64 heads] = Khat . Q^T  (36 tcgen05.mma, M128 N64 K16)
//  4. softmax on a transposed copy of S^T in shared memory; P -> f16.
//  5. O^T [512 ch x 64 heads] = Vhat^T . P^T  (4 x 8 MMAs; the same Khat bytes
//     read MN-major), fp32 accumulators in TMEM.
//  6. Merge across the cluster: every CTA stages the raw O slice and the
//     per-head (max, sum) owed to each other CTA in its own shared memory and
//     the TMA engine copies it into the owner's shared memory (bulk
//     shared -> remote shared copies completing on the owner's mbarrier; this
//     measured ~2x faster than per-thread remote stores and than a merge
//     through L2); each owner then combines its channel slice with weights
//     2^(m_c - M) / L and writes it out.
// Waits on the mbarriers are bounded; on timeout the kernel sets
// CSA2_FLAG_TIMEOUT and still runs every cluster barrier, so it always ends.
#include <cooperative_groups.h>

#include "common.cuh"
#include "tc.cuh"

namespace cg = cooperative_groups;

namespace csa2 {
namespace {

constexpr int TM = 128;                    // entries per CTA (MMA M)
constexpr int D = 576, DV = 512, HB = 64;  // channels, value channels, heads per cluster
constexpr int THREADS = 256;
constexpr int MAX_S = 4;                   // CTAs per cluster
constexpr uint32_t KT_SBO = (D / 8) * 128;        // 9216: bytes per 8-entry group of the Khat tile
constexpr uint32_t KT_BYTES = (TM / 8) * KT_SBO;  // 147456
constexpr uint32_t Q_SBO = (D / 8) * 128;         // 9216: bytes per 8-head group of the Q tile
constexpr uint32_t Q_BYTES = (HB / 8) * Q_SBO;    // 73728
constexpr uint32_t QRAW_STRIDE = D * 2 + 16;      // 1168: staged bf16 Q rows (padded: conflict-free reads)
constexpr uint32_t CRAW_STRIDE = D / 2 + 16;      // 304: staged code rows (padded)
constexpr uint32_t OFF_QRAW = 0;                  // staging lives in the Khat region before dequant
constexpr uint32_t OFF_CRAW = HB * QRAW_STRIDE;   // 74752
constexpr int ST_STRIDE = TM + 4;                 // fp32 row stride of the transposed S (132)
constexpr uint32_t ST_BYTES = HB * ST_STRIDE * 4; // 33792
constexpr uint32_t P_SBO = (TM / 8) * 128;        // 2048: bytes per 8-head group of the P tile
constexpr uint32_t OFF_K = 0;
constexpr uint32_t OFF_Q = OFF_K + KT_BYTES;
constexpr uint32_t OFF_ST = OFF_Q;                // reuses the Q tile after S is computed
constexpr uint32_t OFF_P = OFF_Q + ST_BYTES;
constexpr uint32_t OFF_MISC = OFF_Q + Q_BYTES;
constexpr uint32_t OFF_BAR = OFF_MISC;            // 4 mbarriers
constexpr uint32_t OFF_TMEM = OFF_BAR + 32;
constexpr uint32_t OFF_VALID = OFF_TMEM + 16;     // int[128]
constexpr uint32_t OFF_CS = OFF_VALID + TM * 4;   // float[64] logit factor per head
constexpr uint32_t OFF_M = OFF_CS + HB * 4;       // float[64] row max (log2 domain)
constexpr uint32_t OFF_L = OFF_M + HB * 4;        // float[64] row sum
constexpr uint32_t OFF_W = OFF_L + HB * 4;        // float[MAX_S][64] merge weights
constexpr uint32_t OFF_LSE = OFF_W + MAX_S * HB * 4;      // float[64]
constexpr uint32_t SMEM = OFF_LSE + HB * 4;
constexpr uint32_t TMEM_COLS = 512;               // S^T: 64 cols, O^T: 4 x 64 cols
constexpr uint32_t S_COL = 0, O_COL = 64;
constexpr uint32_t MAX_POLLS = 1u << 22;          // about a second of polling at most
static_assert(OFF_CRAW + TM * CRAW_STRIDE <= KT_BYTES, "staging must fit in the Khat region");
static_assert((DV * (HB + 4) + MAX_S * 2 * HB) * 4 <= KT_BYTES, "received partials must fit in the Khat region");
static_assert(((DV / 2) * (HB + 4) + 2 * HB) * 4 <= Q_BYTES, "a staged slice must fit in the Q region");
static_assert(ST_BYTES + (HB / 8) * P_SBO <= Q_BYTES, "S^T copy and P must fit in the Q region");
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
};

__device__ __forceinline__ uint32_t e2m1x2_to_f16x2(uint32_t byte) {
    uint32_t r;
    asm("{\n\t.reg .b8 t;\n\tcvt.u8.u32 t, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}" : "=r"(r) : "r"(byte));
    return r;
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

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
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
__device__ __forceinline__ void bulk_wait_read0() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read1() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }

__global__ void __launch_bounds__(THREADS, 1) sparse_attn_tc_kernel(TcArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    cg::cluster_group cluster = cg::this_cluster();
    const int rank = (int)cluster.block_rank();
    const int S = a.csize;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    const int64_t group = blockIdx.x / S;
    const int64_t bt = group / a.hblocks;
    const int hblk = (int)(group - bt * a.hblocks);
    const int64_t b = bt / a.T;
    const int h0 = hblk * HB;

    uint8_t *sK = smem + OFF_K;
    uint8_t *sQ = smem + OFF_Q;
    float *sT = reinterpret_cast<float *>(smem + OFF_ST);
    uint8_t *sP = smem + OFF_P;
    float *sRecv = reinterpret_cast<float *>(smem + OFF_K);  // received partial O after P V
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + OFF_TMEM);
    int *sValid = reinterpret_cast<int *>(smem + OFF_VALID);
    float *sCs = reinterpret_cast<float *>(smem + OFF_CS);
    float *sM = reinterpret_cast<float *>(smem + OFF_M);
    float *sL = reinterpret_cast<float *>(smem + OFF_L);
    float *sW = reinterpret_cast<float *>(smem + OFF_W);
    float *sLse = reinterpret_cast<float *>(smem + OFF_LSE);
    const uint32_t bar_ld = tc::smem_u32(smem + OFF_BAR);
    const uint32_t bar_s = bar_ld + 8;
    const uint32_t bar_o = bar_ld + 16;
    const uint32_t bar_rx = bar_ld + 24;

    const int e = tid & (TM - 1);   // entry of this thread in the tile
    const int half = tid >> 7;      // which 288 channels of the entry
    const int sel = rank * TM + e;

    if (tid == 0) {
        tc::mbar_init(bar_ld, TM);   // one arrival per entry thread
        tc::mbar_init(bar_s, 1);
        tc::mbar_init(bar_o, 1);
        tc::mbar_init(bar_rx, 1);
        tc::mbar_init_fence();
    }
    if (warp == 0) tc::tmem_alloc(tmem_slot, TMEM_COLS);
    __syncthreads();
    pdl_wait();   // the set-up above overlaps the previous kernel's tail
    const int64_t j = (sel < a.K) ? (int64_t)__ldg(a.idx + bt * a.K + sel) : -1;   // this thread's entry
    int64_t len = a.kv_len ? (int64_t)a.kv_len[bt] : a.N;
    len = len < a.N ? len : a.N;

    // ---- 1. gather: TMA bulk copies of Q rows and the selected code rows
    if (half == 0 && e < HB) {      // Q rows do not depend on the indices: first
        const uint16_t *qrow = a.q + ((bt * a.H) + h0 + e) * (int64_t)D;
        mbar_expect_tx(bar_ld, D * 2);
        bulk_g2s(tc::smem_u32(smem + OFF_QRAW + e * QRAW_STRIDE), qrow, D * 2, bar_ld);
    }
    const bool valid = j >= 0 && j < len;
    if (half == 0) {
        if (!valid && j != -1) flag_error(a.err_flag, CSA2_FLAG_BAD_INDEX);
        sValid[e] = valid ? 1 : 0;
        mbar_arrive_expect_tx(bar_ld, valid ? D / 2 : 0);
        if (valid)
            bulk_g2s(tc::smem_u32(smem + OFF_CRAW + e * CRAW_STRIDE), a.codes + (b * a.N + j) * (D / 2), D / 2, bar_ld);
    }
    uint32_t sw[5];                 // scale words: plain loads, consumed by the dequantiser
    if (valid) {
        const uint32_t *srow = reinterpret_cast<const uint32_t *>(a.scales + (b * a.N + j) * (D / 16)) + 4 * half;
#pragma unroll
        for (int i = 0; i < 5; ++i) sw[i] = __ldg(srow + i);
    }
    bool ok = tc::mbar_wait(bar_ld, 0, MAX_POLLS);

    // ---- 2a. staged Q -> registers, per-head power-of-two scale, f16 core-matrix tile [head][channel]
    {
        const int hq = warp * 8 + (lane & 7);
        const uint8_t *qraw = smem + OFF_QRAW + hq * QRAW_STRIDE;
        uint4 qv[18];
#pragma unroll
        for (int i = 0; i < 18; ++i) qv[i] = *reinterpret_cast<const uint4 *>(qraw + ((lane >> 3) + 4 * i) * 16);
        float mx = 0.f;
#pragma unroll
        for (int i = 0; i < 18; ++i) {
            const uint32_t w4[4] = {qv[i].x, qv[i].y, qv[i].z, qv[i].w};
#pragma unroll
            for (int k = 0; k < 4; ++k)
                mx = fmaxf(mx, fmaxf(fabsf(__uint_as_float(w4[k] << 16)), fabsf(__uint_as_float(w4[k] & 0xFFFF0000u))));
        }
        mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 8));
        mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 16));
        int e2 = (mx > 0.f) ? ((int)((__float_as_uint(mx) >> 23) & 0xFF) - 127) : 0;
        int sh = 14 - e2;  // max |q| * 2^sh in [2^14, 2^15)
        sh = sh < -60 ? -60 : (sh > 60 ? 60 : sh);
        const float up = ldexpf(1.0f, sh);
        uint8_t *qdst = sQ + warp * Q_SBO + (lane & 7) * 16;
#pragma unroll
        for (int i = 0; i < 18; ++i) {
            const uint32_t w4[4] = {qv[i].x, qv[i].y, qv[i].z, qv[i].w};
            uint32_t o[4];
#pragma unroll
            for (int k = 0; k < 4; ++k)
                o[k] = pack_f16x2(__uint_as_float(w4[k] << 16) * up, __uint_as_float(w4[k] & 0xFFFF0000u) * up);
            *reinterpret_cast<uint4 *>(qdst + ((lane >> 3) + 4 * i) * 128) = make_uint4(o[0], o[1], o[2], o[3]);
        }
        if ((lane >> 3) == 0) sCs[hq] = a.sm_scale * ldexpf(1.0f, -sh) * 1.4426950408889634f;  // x log2(e)
    }
    // ---- 2b. staged codes -> registers (the Khat tile overwrites the staging area)
    uint4 cw[9];
    {
        const uint8_t *craw = smem + OFF_CRAW + e * CRAW_STRIDE + half * 144;
#pragma unroll
        for (int i = 0; i < 9; ++i) cw[i] = valid ? *reinterpret_cast<const uint4 *>(craw + 16 * i) : make_uint4(0, 0, 0, 0);
    }
    __syncthreads();
    // ---- 2c. dequantise this thread's 288 channels of its entry into the Khat tile
    {
        uint8_t *kdst = sK + (e >> 3) * KT_SBO + (e & 7) * 16;
#pragma unroll
        for (int i = 0; i < 9; ++i) {
            const uint32_t w4[4] = {cw[i].x, cw[i].y, cw[i].z, cw[i].w};
#pragma unroll
            for (int gg = 0; gg < 2; ++gg) {           // the two 16-channel groups of this chunk
                const int lb = 2 * i + gg;            // group index within this half (0..17)
                uint32_t r[8] = {0, 0, 0, 0, 0, 0, 0, 0};
                if (valid) {
                    // scale byte lb + 2*half of the loaded words, compile-time indices only
                    const uint32_t s_lo = (sw[lb >> 2] >> (8 * (lb & 3))) & 0xFFu;
                    const uint32_t s_hi = (sw[(lb + 2) >> 2] >> (8 * ((lb + 2) & 3))) & 0xFFu;
                    const uint32_t sc = e4m3_to_f16x2_bcast(half ? s_hi : s_lo);
#pragma unroll
                    for (int k = 0; k < 2; ++k) {
                        const uint32_t wd = w4[2 * gg + k];
#pragma unroll
                        for (int bb = 0; bb < 4; ++bb) r[4 * k + bb] = hmul2(e2m1x2_to_f16x2((wd >> (8 * bb)) & 0xFF), sc);
                    }
                }
                const int c8 = half * 36 + 4 * i + 2 * gg;
                *reinterpret_cast<uint4 *>(kdst + c8 * 128) = make_uint4(r[0], r[1], r[2], r[3]);
                *reinterpret_cast<uint4 *>(kdst + (c8 + 1) * 128) = make_uint4(r[4], r[5], r[6], r[7]);
            }
        }
    }
    tc::fence_async_smem();
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tmem = *tmem_slot;

    // ---- 3. S^T = Khat . Q^T  (M = 128 entries, N = 64 heads, K = 576)
    if (tid == 0) {
        const uint32_t a0 = tc::smem_u32(sK), b0 = tc::smem_u32(sQ);
        constexpr uint32_t idesc = tc::idesc_f16_f32(TM, HB, false, false);
#pragma unroll 4
        for (int ks = 0; ks < D / 16; ++ks)
            tc::mma_f16(tmem + S_COL, tc::desc_noswizzle(a0 + ks * 256, 128, KT_SBO),
                        tc::desc_noswizzle(b0 + ks * 256, 128, Q_SBO), idesc, ks > 0);
        tc::commit(bar_s);
    }
    ok = tc::mbar_wait(bar_s, 0, MAX_POLLS) && ok;
    tc::fence_after();

    // ---- 4a. S^T -> shared memory, transposed to [head][entry] (the Q tile is free now)
    const int quarter = warp & 3, hh = warp >> 2;
    {
        uint32_t r[32];
        tc::tmem_ld32(tmem + ((uint32_t)(32 * quarter) << 16) + S_COL + 32 * hh, r);
        tc::tmem_ld_wait();
        const int ee = 32 * quarter + lane;
        const bool v = ok && sValid[ee];
#pragma unroll
        for (int jj = 0; jj < 32; ++jj) {
            const int h = 32 * hh + jj;
            sT[h * ST_STRIDE + ee] = v ? __uint_as_float(r[jj]) * sCs[h] : -INFINITY;
        }
    }
    __syncthreads();

    // ---- 4b. softmax per head over this CTA's entries; P -> f16 core-matrix tile [head][entry]
    {
        const int h = tid >> 2, part = tid & 3;
        float z[32];
        float mx = -INFINITY;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            z[i] = sT[h * ST_STRIDE + 4 * i + part];
            mx = fmaxf(mx, z[i]);
        }
        mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 2));
        float sum = 0.f;
        uint8_t *pdst = sP + (h >> 3) * P_SBO + (h & 7) * 16;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            const int ee = 4 * i + part;
            const float p = (mx == -INFINITY || z[i] == -INFINITY) ? 0.f : ex2(z[i] - mx);
            const __half ph = __float2half_rn(p);
            sum += __half2float(ph);
            *reinterpret_cast<__half *>(pdst + (ee >> 3) * 128 + (ee & 7) * 2) = ph;
        }
        sum += __shfl_xor_sync(0xFFFFFFFFu, sum, 1);
        sum += __shfl_xor_sync(0xFFFFFFFFu, sum, 2);
        if (part == 0) {
            sM[h] = mx;
            sL[h] = sum;
        }
    }
    tc::fence_async_smem();
    tc::fence_before();
    __syncthreads();
    tc::fence_after();

    // ---- 5. O^T = Vhat^T . P^T  (4 blocks of M = 128 channels, N = 64 heads, K = 128 entries)
    if (tid == 0) {
        const uint32_t a0 = tc::smem_u32(sK), b0 = tc::smem_u32(sP);
        constexpr uint32_t idesc = tc::idesc_f16_f32(TM, HB, true, false);
        for (int mb = 0; mb < DV / 128; ++mb)
#pragma unroll
            for (int ks = 0; ks < TM / 16; ++ks)
                tc::mma_f16(tmem + O_COL + mb * HB, tc::desc_noswizzle(a0 + ks * 2 * KT_SBO + mb * 16 * 128, KT_SBO, 128),
                            tc::desc_noswizzle(b0 + ks * 256, 128, P_SBO), idesc, ks > 0);
        tc::commit(bar_o);
    }
    ok = tc::mbar_wait(bar_o, 0, MAX_POLLS) && ok;
    pdl_launch_dependents();   // the next kernel may launch during the merge
    tc::fence_after();
    if (!ok && tid == 0) flag_error(a.err_flag, CSA2_FLAG_TIMEOUT);

    // ---- 6. send raw O slices and (max, sum) to the owners of the channel slices
    // Payload for owner o: [W channels][RS floats: 64 heads + pad] then 64 max + 64 sum.
    // Slices for other CTAs are staged in this CTA's Q region and moved by the
    // TMA engine (bulk shared -> remote shared copies completing on the owner's
    // mbarrier); the own slice is written in place.
    const int W = DV / S;                      // channels per owner
    constexpr int RS = HB + 4;                 // floats per received channel row
    const uint32_t slice_floats = (uint32_t)W * RS + 2 * HB;
    const uint32_t slice_bytes = slice_floats * 4;
    float *stage = reinterpret_cast<float *>(smem + OFF_Q);   // free after P V
    const int nbuf = (2 * slice_bytes <= Q_BYTES) ? 2 : 1;    // staging buffers (2 when S = 4)
    int sent = 0;
    if (tid == 0) asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar_rx),
                               "r"((uint32_t)(S - 1) * slice_bytes) : "memory");
    tc::fence_before();
    cluster.sync();                            // every CTA finished with its Khat tile
    for (int o = 0; o < S; ++o) {
        const int oo = (rank + 1 + o) % S;     // own slice last
        float *dst = (oo == rank) ? sRecv + (size_t)rank * slice_floats : stage + (size_t)(sent % nbuf) * slice_floats;
        if (oo != rank && sent >= nbuf) {
            if (tid == 0) {                    // this staging buffer's previous copy has read it
                if (nbuf == 2) bulk_wait_read1();
                else bulk_wait_read0();
            }
            __syncthreads();
        }
        for (int mb = oo * W / 128; mb < (oo + 1) * W / 128; ++mb) {
            uint32_t r[32];
            tc::tmem_ld32(tmem + ((uint32_t)(32 * quarter) << 16) + O_COL + mb * HB + 32 * hh, r);
            tc::tmem_ld_wait();
            float *row = dst + (size_t)(mb * 128 - oo * W + 32 * quarter + lane) * RS + 32 * hh;
#pragma unroll
            for (int q4 = 0; q4 < 8; ++q4)
                *reinterpret_cast<uint4 *>(row + 4 * q4) = make_uint4(r[4 * q4], r[4 * q4 + 1], r[4 * q4 + 2], r[4 * q4 + 3]);
        }
        if (tid < HB) {
            dst[(size_t)W * RS + tid] = sM[tid];
            dst[(size_t)W * RS + HB + tid] = sL[tid];
        }
        if (oo != rank) {
            tc::fence_async_smem();
            __syncthreads();
            if (tid == 0) {
                uint32_t rdst, rbar;
                const uint32_t ldst = tc::smem_u32(sRecv + (size_t)rank * slice_floats);
                asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(rdst) : "r"(ldst), "r"((uint32_t)oo));
                asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(rbar) : "r"(bar_rx), "r"((uint32_t)oo));
                bulk_s2s(rdst, tc::smem_u32(dst), slice_bytes, rbar);
                bulk_commit();
            }
            ++sent;
        }
    }
    if (tid == 0) bulk_wait_read0();           // staging reads done before this CTA may exit
    ok = tc::mbar_wait(bar_rx, 0, MAX_POLLS) && ok;   // the other CTAs' slices have landed
    __syncthreads();
    if (!ok && tid == 0) flag_error(a.err_flag, CSA2_FLAG_TIMEOUT);

    // ---- 7. combine this CTA's channel slice: weights 2^(m_c - M) / L per head
    if (tid < HB) {
        float M = -INFINITY;
        for (int c = 0; c < S; ++c) M = fmaxf(M, sRecv[(size_t)c * slice_floats + W * RS + tid]);
        float L = 0.f;
        for (int c = 0; c < S; ++c) {
            const float mc = sRecv[(size_t)c * slice_floats + W * RS + tid];
            const float wc = (M == -INFINITY || mc == -INFINITY) ? 0.f : ex2(mc - M);
            sW[c * HB + tid] = wc;
            L += wc * sRecv[(size_t)c * slice_floats + W * RS + HB + tid];
        }
        const float inv = L > 0.f ? 1.f / L : 0.f;
        for (int c = 0; c < S; ++c) sW[c * HB + tid] *= inv;
        sLse[tid] = (L > 0.f) ? (M + log2f(L)) * 0.6931471805599453f : -INFINITY;
    }
    __syncthreads();
    {
        // thread -> (4 heads, channel): lanes take consecutive channels, so each
        // output store of a warp covers 32 consecutive channels of one head
        const int c_lo = rank * W;
        for (int t = tid; t < (HB / 4) * W; t += THREADS) {
            const int h4 = t / W, c = t - h4 * W;
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int src = 0; src < S; ++src) {
                const float4 v = *reinterpret_cast<const float4 *>(sRecv + (size_t)src * slice_floats + (size_t)c * RS + 4 * h4);
                const float *w = sW + src * HB + 4 * h4;
                acc.x += w[0] * v.x; acc.y += w[1] * v.y; acc.z += w[2] * v.z; acc.w += w[3] * v.w;
            }
            float *o = a.out + ((bt * a.H) + h0 + 4 * h4) * (int64_t)DV + c_lo + c;
            o[0] = acc.x;
            o[DV] = acc.y;
            o[2 * DV] = acc.z;
            o[3 * DV] = acc.w;
        }
        if (rank == 0 && a.lse && tid < HB) a.lse[(bt * a.H) + h0 + tid] = sLse[tid];
    }
    tc::fence_after();
    if (warp == 0) tc::tmem_dealloc(tmem, TMEM_COLS);
}

}  // namespace

bool sparse_attn_tc_supported(int D_, int dv, int H, int K) {
    return D_ == D && dv == DV && H % HB == 0 && K >= 1 && K <= MAX_S * TM;
}

csa2_status launch_sparse_attn_tc(int B, int T, int H, int K, int64_t N, const void *q, const uint8_t *codes,
                                  const uint8_t *scales, const int32_t *idx, const int32_t *kv_len, float sm_scale,
                                  float *out, float *lse, uint32_t *err_flag, cudaStream_t stream) {
    static bool smem_set[64];
    CSA2_CUDA_CALL(ensure_smem_limit((const void *)sparse_attn_tc_kernel, (int)SMEM, smem_set),
                   "sparse_attn_tc: smem attribute");
    TcArgs a;
    a.T = T; a.H = H; a.K = K; a.N = N;
    const int tiles = (K + TM - 1) / TM;
    a.csize = tiles <= 1 ? 1 : (tiles <= 2 ? 2 : 4);   // 1, 2 or 4: the channel slices divide 512
    a.hblocks = H / HB;
    a.q = (const uint16_t *)q; a.codes = codes; a.scales = scales; a.idx = idx; a.kv_len = kv_len;
    a.sm_scale = sm_scale; a.out = out; a.lse = lse; a.err_flag = err_flag;
    const int64_t grid = (int64_t)B * T * a.hblocks * a.csize;
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
    CSA2_CUDA_CALL(cudaLaunchKernelEx(&cfg, sparse_attn_tc_kernel, a), "sparse_attn_tc_kernel launch");
    CSA2_LAUNCH_CHECK("sparse_attn_tc_kernel");
    return CSA2_OK;
}

}  // namespace csa2

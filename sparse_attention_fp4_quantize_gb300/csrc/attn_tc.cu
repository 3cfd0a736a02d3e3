// Sparse FP4 attention on the 5th-generation tensor cores (tcgen05, TMEM),
// for 576-channel entries (512 latent + 64 RoPE), dv = 512, 64-head blocks.
// Sources: "DeepSeek-V4.1-Flash：把 KV Cache 压缩到极限的百万上下文 MoE", section
// "效率组件四件" item 4 (FP4 main KV) and the inference bullet of
// "优化器与训练基础设施" (Reuse layers run a fused attention kernel; prior art);
// "DeepSeek-V4.1-Flash: Pushing the Limits of KV Cache Compression", CSA2
// paragraph.  The attention itself is the MLA-style reading (K = all 576
// channels, V = the first 512).
//
// Layout of the work.  A thread-block cluster of S = ceil(K/128) CTAs serves
// one query token and 64 heads; CTA c owns selected entries [128c, 128c+128).
// Every matrix product is a 128-row tcgen05.mma with fp32 accumulators in TMEM:
//   S^T [128 entries x 64 heads] = Khat [128 x 576] . Q^T      (36 MMAs, K=16)
//   O^T [512 ch x 64 heads]     += Vhat^T [512 x 128] . P^T    (4 x 8 MMAs)
// Khat is written ONCE to shared memory by the dequantiser (E2M1 x E4M3 ->
// exact f16) in the no-swizzle core-matrix layout; the S product reads it
// K-major and the P V product reads the same bytes MN-major as Vhat^T.
// Q (bf16) is scaled per head by a power of two into f16 (exact) and the
// scale is folded into the logit factor.  Softmax runs on a transposed copy
// of S^T in shared memory; P is rounded to f16 for the second product.
// The S CTAs then merge their partial outputs through distributed shared
// memory (no global scratch, no second kernel): each CTA scales its O by
// 2^(m_c - M) / L per head and CTA c sums channel slice c over the cluster.
// Waits on the MMA completion barrier are bounded; on timeout the kernel sets
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
constexpr uint32_t KT_SBO = (D / 8) * 128;      // 9216: bytes per 8-entry group of the Khat tile
constexpr uint32_t KT_BYTES = (TM / 8) * KT_SBO;  // 147456
constexpr uint32_t Q_SBO = (D / 8) * 128;        // 9216: bytes per 8-head group of the Q tile
constexpr uint32_t Q_BYTES = (HB / 8) * Q_SBO;   // 73728
constexpr int ST_STRIDE = TM + 4;               // fp32 row stride of the transposed S (132)
constexpr uint32_t ST_BYTES = HB * ST_STRIDE * 4;  // 33792
constexpr uint32_t P_SBO = (TM / 8) * 128;       // 2048: bytes per 8-head group of the P tile
constexpr int PO_STRIDE = DV + 4;               // fp32 row stride of the partial O (516)
constexpr uint32_t OFF_K = 0;
constexpr uint32_t OFF_Q = OFF_K + KT_BYTES;
constexpr uint32_t OFF_ST = OFF_Q;              // reuses the Q tile after S is computed
constexpr uint32_t OFF_P = OFF_Q + ST_BYTES;
constexpr uint32_t OFF_MISC = OFF_Q + Q_BYTES;
constexpr uint32_t OFF_BAR = OFF_MISC;          // 2 mbarriers
constexpr uint32_t OFF_TMEM = OFF_BAR + 16;
constexpr uint32_t OFF_VALID = OFF_TMEM + 16;   // int[128]
constexpr uint32_t OFF_CS = OFF_VALID + TM * 4;  // float[64] logit factor per head
constexpr uint32_t OFF_M = OFF_CS + HB * 4;      // float[64] row max (log2 domain)
constexpr uint32_t OFF_L = OFF_M + HB * 4;       // float[64] row sum
constexpr uint32_t OFF_W = OFF_L + HB * 4;       // float[64] merge weight
constexpr uint32_t OFF_LSE = OFF_W + HB * 4;     // float[64] final lse (natural log)
constexpr uint32_t SMEM = OFF_LSE + HB * 4;
constexpr uint32_t TMEM_COLS = 512;             // S^T: 64 cols, O^T: 4 x 64 cols
constexpr uint32_t S_COL = 0, O_COL = 64;
constexpr uint32_t MAX_POLLS = 1u << 22;  // about a second of polling at most
static_assert(HB * PO_STRIDE * 4 <= KT_BYTES, "partial O must fit in the Khat region");
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
    int64_t len = a.kv_len ? (int64_t)a.kv_len[bt] : a.N;
    len = len < a.N ? len : a.N;

    uint8_t *sK = smem + OFF_K;
    uint8_t *sQ = smem + OFF_Q;
    float *sT = reinterpret_cast<float *>(smem + OFF_ST);
    uint8_t *sP = smem + OFF_P;
    float *sPO = reinterpret_cast<float *>(smem + OFF_K);  // partial O after P V
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + OFF_TMEM);
    int *sValid = reinterpret_cast<int *>(smem + OFF_VALID);
    float *sCs = reinterpret_cast<float *>(smem + OFF_CS);
    float *sM = reinterpret_cast<float *>(smem + OFF_M);
    float *sL = reinterpret_cast<float *>(smem + OFF_L);
    float *sW = reinterpret_cast<float *>(smem + OFF_W);
    float *sLse = reinterpret_cast<float *>(smem + OFF_LSE);
    const uint32_t bar_s = tc::smem_u32(smem + OFF_BAR);
    const uint32_t bar_o = bar_s + 8;

    // ---- 1. issue every global load of this CTA first: the entry's codes/scales, Q
    const int e = tid & (TM - 1);   // entry of this thread in the tile
    const int half = tid >> 7;      // which 288 channels of the entry
    const int sel = rank * TM + e;
    int64_t j = (sel < a.K) ? (int64_t)__ldg(a.idx + bt * a.K + sel) : -1;
    const bool valid = j >= 0 && j < len;
    if (!valid && j != -1 && half == 0) flag_error(a.err_flag, CSA2_FLAG_BAD_INDEX);
    uint4 cw[9];
    uint32_t sw[5];
    if (valid) {
        const uint8_t *crow = a.codes + (b * a.N + j) * (D / 2) + half * 144;
        const uint32_t *srow = reinterpret_cast<const uint32_t *>(a.scales + (b * a.N + j) * (D / 16)) + 4 * half;
#pragma unroll
        for (int i = 0; i < 9; ++i) cw[i] = __ldg(reinterpret_cast<const uint4 *>(crow) + i);
#pragma unroll
        for (int i = 0; i < 5; ++i) sw[i] = __ldg(srow + i);
    }
    const int hq = warp * 8 + (lane & 7);   // head (within the block) whose Q this lane loads
    const uint16_t *qrow = a.q + ((bt * a.H) + h0 + hq) * (int64_t)D;
    uint4 qv[18];
#pragma unroll
    for (int i = 0; i < 18; ++i) qv[i] = __ldg(reinterpret_cast<const uint4 *>(qrow) + (lane >> 3) + 4 * i);

    if (warp == 0) tc::tmem_alloc(tmem_slot, TMEM_COLS);
    if (tid == 0) {
        tc::mbar_init(bar_s, 1);
        tc::mbar_init(bar_o, 1);
        tc::mbar_init_fence();
    }
    if (half == 0) sValid[e] = valid ? 1 : 0;

    // ---- 2. Q -> f16 with a per-head power-of-two scale, core-matrix layout [head][channel]
    {
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
            const int c8 = (lane >> 3) + 4 * i;
            *reinterpret_cast<uint4 *>(qdst + c8 * 128) = make_uint4(o[0], o[1], o[2], o[3]);
        }
        if ((lane >> 3) == 0) sCs[hq] = a.sm_scale * ldexpf(1.0f, -sh) * 1.4426950408889634f;  // x log2(e)
    }

    // ---- 3. dequantise this thread's 288 channels of its entry into the Khat tile
    {
        uint8_t *kdst = sK + (e >> 3) * KT_SBO + (e & 7) * 16;
#pragma unroll
        for (int i = 0; i < 9; ++i) {
            const uint32_t w4[4] = {cw[i].x, cw[i].y, cw[i].z, cw[i].w};
#pragma unroll
            for (int gg = 0; gg < 2; ++gg) {          // the two 16-channel groups of this chunk
                const int lb = 2 * i + gg;           // group index within this half (0..17)
                uint32_t r[8] = {0, 0, 0, 0, 0, 0, 0, 0};
                if (valid) {
                    // scale byte lb + 2*half of the loaded words: both candidates use
                    // compile-time indices (a runtime index would put sw in local memory)
                    constexpr int b0 = 0;
                    const uint32_t s_lo = (sw[(lb + b0) >> 2] >> (8 * ((lb + b0) & 3))) & 0xFFu;
                    const uint32_t s_hi = (sw[(lb + 2) >> 2] >> (8 * ((lb + 2) & 3))) & 0xFFu;
                    const uint32_t sb = half ? s_hi : s_lo;
                    const uint32_t sc = e4m3_to_f16x2_bcast(sb);
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

    // ---- 4. S^T = Khat . Q^T  (M = 128 entries, N = 64 heads, K = 576)
    if (tid == 0) {
        const uint32_t a0 = tc::smem_u32(sK), b0 = tc::smem_u32(sQ);
        constexpr uint32_t idesc = tc::idesc_f16_f32(TM, HB, false, false);
#pragma unroll 4
        for (int ks = 0; ks < D / 16; ++ks)
            tc::mma_f16(tmem + S_COL, tc::desc_noswizzle(a0 + ks * 256, 128, KT_SBO),
                        tc::desc_noswizzle(b0 + ks * 256, 128, Q_SBO), idesc, ks > 0);
        tc::commit(bar_s);
    }
    bool ok = tc::mbar_wait(bar_s, 0, MAX_POLLS);
    tc::fence_after();

    // ---- 5. S^T -> shared memory, transposed to [head][entry] (the Q tile is free now)
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

    // ---- 6. softmax per head over this CTA's entries; P -> f16 core-matrix layout [head][entry]
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

    // ---- 7. O^T = Vhat^T . P^T  (4 blocks of M = 128 channels, N = 64 heads, K = 128 entries)
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
    tc::fence_after();
    if (!ok && tid == 0) flag_error(a.err_flag, CSA2_FLAG_TIMEOUT);

    // ---- 8. merge weights across the cluster: M = max_c m_c, L = sum_c l_c 2^(m_c - M)
    cluster.sync();
    if (tid < HB) {
        float M = -INFINITY;
        for (int c = 0; c < S; ++c) M = fmaxf(M, cluster.map_shared_rank(sM, c)[tid]);
        float L = 0.f;
        if (M != -INFINITY)
            for (int c = 0; c < S; ++c) {
                const float mc = cluster.map_shared_rank(sM, c)[tid];
                if (mc != -INFINITY) L += cluster.map_shared_rank(sL, c)[tid] * ex2(mc - M);
            }
        const float mine = sM[tid];
        sW[tid] = (L > 0.f && mine != -INFINITY) ? ex2(mine - M) / L : 0.f;
        sLse[tid] = (L > 0.f) ? (M + log2f(L)) * 0.6931471805599453f : -INFINITY;
    }
    __syncthreads();

    // ---- 9. scaled partial O -> shared memory [head][channel] (the Khat tile is free now)
#pragma unroll 1
    for (int mb = 0; mb < DV / 128; ++mb) {
        uint32_t r[32];
        tc::tmem_ld32(tmem + ((uint32_t)(32 * quarter) << 16) + O_COL + mb * HB + 32 * hh, r);
        tc::tmem_ld_wait();
        const int ch = mb * 128 + 32 * quarter + lane;
#pragma unroll
        for (int jj = 0; jj < 32; ++jj) {
            const int h = 32 * hh + jj;
            sPO[h * PO_STRIDE + ch] = __uint_as_float(r[jj]) * sW[h];
        }
    }
    tc::fence_before();
    cluster.sync();  // every CTA's scaled partial is in its shared memory

    // ---- 10. CTA `rank` sums its channel slice over the cluster and writes out
    {
        int ch_per = (DV + S - 1) / S;
        ch_per = (ch_per + 3) & ~3;
        const int c_lo = rank * ch_per;
        const int c_hi = min(DV, c_lo + ch_per);
        const int n4 = (c_hi > c_lo) ? (c_hi - c_lo) / 4 : 0;
        const float *src[8];
#pragma unroll
        for (int r = 0; r < 8; ++r) src[r] = cluster.map_shared_rank(sPO, r < S ? r : 0);
        for (int t = tid; t < HB * n4; t += THREADS) {
            const int h = t / n4, c = c_lo + 4 * (t - h * n4);
            float4 v[8];
#pragma unroll
            for (int r = 0; r < 8; ++r)   // all remote loads first, then the sum
                if (r < S) v[r] = *reinterpret_cast<const float4 *>(src[r] + h * PO_STRIDE + c);
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int r = 0; r < 8; ++r)
                if (r < S) { acc.x += v[r].x; acc.y += v[r].y; acc.z += v[r].z; acc.w += v[r].w; }
            *reinterpret_cast<float4 *>(a.out + ((bt * a.H) + h0 + h) * (int64_t)DV + c) = acc;
        }
        if (rank == 0 && a.lse && tid < HB) a.lse[(bt * a.H) + h0 + tid] = sLse[tid];
    }
    cluster.sync();  // remote reads done before any CTA leaves
    tc::fence_after();
    if (warp == 0) tc::tmem_dealloc(tmem, TMEM_COLS);
}

}  // namespace

bool sparse_attn_tc_supported(int D_, int dv, int H, int K) {
    return D_ == D && dv == DV && H % HB == 0 && K >= 1 && K <= 8 * TM;
}

csa2_status launch_sparse_attn_tc(int B, int T, int H, int K, int64_t N, const void *q, const uint8_t *codes,
                                  const uint8_t *scales, const int32_t *idx, const int32_t *kv_len, float sm_scale,
                                  float *out, float *lse, uint32_t *err_flag, cudaStream_t stream) {
    static bool smem_set[64];
    CSA2_CUDA_CALL(ensure_smem_limit((const void *)sparse_attn_tc_kernel, (int)SMEM, smem_set),
                   "sparse_attn_tc: smem attribute");
    TcArgs a;
    a.T = T; a.H = H; a.K = K; a.N = N;
    a.csize = (K + TM - 1) / TM;
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
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = a.csize;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    CSA2_CUDA_CALL(cudaLaunchKernelEx(&cfg, sparse_attn_tc_kernel, a), "sparse_attn_tc_kernel launch");
    CSA2_LAUNCH_CHECK("sparse_attn_tc_kernel");
    return CSA2_OK;
}

}  // namespace csa2

// csa2_sparse_attn_fp4: attention of every query head over its Top-K selected
// FP4 entries, with the entries gathered from the FP4 planes and dequantised
// on chip.
// Sources: "DeepSeek-V4.1-Flash：把 KV Cache 压缩到极限的百万上下文 MoE", section
// "优化器与训练基础设施", inference bullet (Reuse layers run FlashMLA fused
// attention; prior art, not the blueprint) and section "效率组件四件" item 4
// (the FP4 main KV format); "DeepSeek-V4.1-Flash: Pushing the Limits of KV
// Cache Compression", CSA2 paragraph (Reuse layers reuse the Top-K).  The
// pages give no attention formula: MLA-style reading, K = all D channels,
// V = the first dv channels of the same entry.
//
// Design (per CTA: one query token, a block of heads, a slice of the K
// selected entries):
//  - Q is loaded once, scaled per head by a power of two into the f16 range
//    (exact for the bf16 inputs; the scale is folded into the logit factor)
//    and kept in shared memory.
//  - Entries are staged 32 at a time with cp.async (16-byte code chunks,
//    4-byte scale words) into a double buffer, then dequantised once into an
//    f16 tile: E2M1 x E4M3 products have <= 6 significant bits, so the f16
//    values are exact.  The same tile serves as K (all D channels) and V (the
//    first dv channels).
//  - S = Q K^T and O += P V run on the tensor cores (mma.m16n8k16, f16 in,
//    fp32 accumulate); P is rounded to f16 (11-bit mantissa) for P V.
//  - Online softmax in the log2 domain; split-KV partials (normalised O and
//    lse per split) are merged by a small combine kernel.
#include <mutex>

#include "common.cuh"

namespace csa2 {
namespace {

constexpr int TE = 32;  // entries per tile

__device__ __forceinline__ void mma_f16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], const void *p) {
    uint32_t a = (uint32_t)__cvta_generic_to_shared(p);
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(a));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], const void *p) {
    uint32_t a = (uint32_t)__cvta_generic_to_shared(p);
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(a));
}

__device__ __forceinline__ void cp_async16(void *smem, const void *gmem) {
    uint32_t s = (uint32_t)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(s), "l"(gmem));
}

__device__ __forceinline__ void cp_async4(void *smem, const void *gmem) {
    uint32_t s = (uint32_t)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(s), "l"(gmem));
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ float ex2(float x) {
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

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

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}

struct AttnArgs {
    int B, T, H, K;
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
    int splits;
    float *part_o;    // [splits, B*T, H, DV]
    float *part_lse;  // [splits, B*T, H]
};

template <int D, int DV, int NG>
struct AttnCfg {
    static constexpr int HB = 16 * NG;         // heads per CTA
    static constexpr int NWARP = 2 * NG;       // warp (hg, half)
    static constexpr int THREADS = 32 * NWARP;
    static constexpr int RS = D + 8;           // f16 row stride of Q and K tiles
    static constexpr int PS = TE + 8;          // f16 row stride of P
    static constexpr int CB = D / 2;           // code bytes per entry
    static constexpr int SB = D / 16;          // scale bytes per entry
    static constexpr int DVW = DV / 2;         // dv channels per warp
    static constexpr int NT_PV = DVW / 8;      // n8 tiles per warp in P V
    static constexpr size_t OFF_Q = 0;
    static constexpr size_t OFF_K = OFF_Q + (size_t)HB * RS * 2;
    static constexpr size_t OFF_C = OFF_K + (size_t)TE * RS * 2;
    static constexpr size_t OFF_S = OFF_C + 2 * (size_t)TE * CB;
    static constexpr size_t OFF_P = OFF_S + 2 * (size_t)TE * SB;
    static constexpr size_t OFF_MX = OFF_P + (size_t)HB * PS * 2;
    static constexpr size_t OFF_V = OFF_MX + 2 * (size_t)HB * 4;
    static constexpr size_t SMEM = OFF_V + 2 * TE * 4 + 2 * (size_t)HB * 4;
    static_assert(D % 16 == 0 && DV % 16 == 0 && DV <= D, "shape");
    static_assert(DVW % 16 == 0, "dv per warp must be a multiple of 16");
    static_assert((OFF_C % 16) == 0 && (OFF_S % 16) == 0 && (OFF_P % 16) == 0, "align");
};

template <int D, int DV, int NG>
__global__ void __launch_bounds__(AttnCfg<D, DV, NG>::THREADS, 1) sparse_attn_kernel(AttnArgs a) {
    using C = AttnCfg<D, DV, NG>;
    extern __shared__ __align__(16) uint8_t smem[];
    __half *sQ = reinterpret_cast<__half *>(smem + C::OFF_Q);
    __half *sK = reinterpret_cast<__half *>(smem + C::OFF_K);
    uint8_t *sC = smem + C::OFF_C;
    uint8_t *sS = smem + C::OFF_S;
    __half *sP = reinterpret_cast<__half *>(smem + C::OFF_P);
    float *sMax = reinterpret_cast<float *>(smem + C::OFF_MX);   // [2][HB]
    int32_t *sValid = reinterpret_cast<int32_t *>(smem + C::OFF_V);  // [2][TE]
    float *sL = reinterpret_cast<float *>(smem + C::OFF_V + 2 * TE * 4);  // [2][HB]

    pdl_wait();
    pdl_launch_dependents();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int hg = warp >> 1;    // head group of 16
    const int half = warp & 1;   // entry half in S, dv half in P V
    const int g = lane >> 2, t4 = lane & 3;
    const int64_t bt = blockIdx.x;
    const int split = blockIdx.y;
    const int hblk = blockIdx.z;
    const int64_t b = bt / a.T;
    const int h0 = hblk * C::HB;
    int64_t len = a.kv_len ? (int64_t)a.kv_len[bt] : a.N;
    len = len < a.N ? len : a.N;

    const int ntiles = (a.K + TE - 1) / TE;
    const int tbeg = (int)((int64_t)split * ntiles / a.splits);
    const int tend = (int)((int64_t)(split + 1) * ntiles / a.splits);
    const int32_t *idx_row = a.idx + bt * a.K;

    // ---- stage loader: cp.async of the codes/scales of tile `tile` into buffer `st`
    auto issue_tile = [&](int tile, int st) {
        uint8_t *dc = sC + st * TE * C::CB;
        uint8_t *ds = sS + st * TE * C::SB;
        constexpr int CCH = C::CB / 16;   // 16-byte code chunks per entry
        constexpr int SCH = C::SB / 4;    // 4-byte scale words per entry
        for (int task = tid; task < TE * (CCH + SCH); task += C::THREADS) {
            const int e = task / (CCH + SCH);
            const int c = task - e * (CCH + SCH);
            const int s = tile * TE + e;
            int64_t j = (s < a.K) ? (int64_t)__ldg(idx_row + s) : -1;
            if (j < 0 || j >= len) continue;
            const int64_t rowg = b * a.N + j;
            if (c < CCH)
                cp_async16(dc + e * C::CB + c * 16, a.codes + rowg * C::CB + c * 16);
            else
                cp_async4(ds + e * C::SB + (c - CCH) * 4, a.scales + rowg * C::SB + (c - CCH) * 4);
        }
        if (tid < TE) {
            const int s = tile * TE + tid;
            int64_t j = (s < a.K) ? (int64_t)__ldg(idx_row + s) : -1;
            int v = (j >= 0 && j < len) ? 1 : 0;
            if (!v && j != -1) flag_error(a.err_flag, CSA2_FLAG_BAD_INDEX);
            sValid[st * TE + tid] = v;
        }
        cp_async_commit();
    };

    if (tbeg < tend) issue_tile(tbeg, 0);

    // ---- Q: per-head power-of-two scale into f16, then to shared memory
    for (int hh = warp; hh < C::HB; hh += C::NWARP) {
        const uint16_t *qrow = a.q + ((bt * a.H) + h0 + hh) * (int64_t)D;
        float mx = 0.f;
        for (int c = lane; c < D / 8; c += 32) {
            uint4 v = __ldg(reinterpret_cast<const uint4 *>(qrow) + c);
            uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                mx = fmaxf(mx, fabsf(__uint_as_float(w[i] << 16)));
                mx = fmaxf(mx, fabsf(__uint_as_float(w[i] & 0xFFFF0000u)));
            }
        }
        for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, off));
        int e2 = (mx > 0.f) ? ((int)((__float_as_uint(mx) >> 23) & 0xFF) - 127) : 0;
        int sh = 14 - e2;                       // max |q| * 2^sh in [2^14, 2^15)
        sh = sh < -60 ? -60 : (sh > 60 ? 60 : sh);
        const float up = ldexpf(1.0f, sh);
        for (int c = lane; c < D / 8; c += 32) {
            uint4 v = __ldg(reinterpret_cast<const uint4 *>(qrow) + c);
            uint32_t w[4] = {v.x, v.y, v.z, v.w};
            uint32_t o[4];
#pragma unroll
            for (int i = 0; i < 4; ++i)
                o[i] = pack_f16x2(__uint_as_float(w[i] << 16) * up, __uint_as_float(w[i] & 0xFFFF0000u) * up);
            *reinterpret_cast<uint4 *>(sQ + hh * C::RS + c * 8) = make_uint4(o[0], o[1], o[2], o[3]);
        }
        if (lane == 0) sL[C::HB + hh] = a.sm_scale * ldexpf(1.0f, -sh) * 1.4426950408889634f;  // log2(e)
    }

    // ---- per-thread running state for rows (heads) hg*16+g and +8
    const int r0 = hg * 16 + g, r1 = r0 + 8;
    float m0 = -INFINITY, m1 = -INFINITY;   // running max (log2 domain)
    float l0 = 0.f, l1 = 0.f;               // partial sums over this warp's entries
    float o[C::NT_PV][4];
#pragma unroll
    for (int i = 0; i < C::NT_PV; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    __syncthreads();
    const float cs0 = sL[C::HB + r0], cs1 = sL[C::HB + r1];

    for (int tile = tbeg; tile < tend; ++tile) {
        const int st = (tile - tbeg) & 1;
        cp_async_wait_all();
        __syncthreads();  // stage `st` landed for every thread; previous P V done
        if (tile + 1 < tend) issue_tile(tile + 1, st ^ 1);

        // ---- dequantise the staged tile into sK (zeros for invalid entries)
        {
            const uint8_t *dc = sC + st * TE * C::CB;
            const uint8_t *ds = sS + st * TE * C::SB;
            for (int task = tid; task < TE * C::SB; task += C::THREADS) {
                const int e = task / C::SB, gi = task - e * C::SB;
                uint4 lo = make_uint4(0, 0, 0, 0), hi = make_uint4(0, 0, 0, 0);
                if (sValid[st * TE + e]) {
                    const uint2 cw = *reinterpret_cast<const uint2 *>(dc + e * C::CB + gi * 8);
                    const uint32_t sc = e4m3_to_f16x2_bcast(ds[e * C::SB + gi]);
                    uint32_t r[8];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        r[i] = hmul2(e2m1x2_to_f16x2((cw.x >> (8 * i)) & 0xFF), sc);
                        r[4 + i] = hmul2(e2m1x2_to_f16x2((cw.y >> (8 * i)) & 0xFF), sc);
                    }
                    lo = make_uint4(r[0], r[1], r[2], r[3]);
                    hi = make_uint4(r[4], r[5], r[6], r[7]);
                }
                uint4 *dst = reinterpret_cast<uint4 *>(sK + e * C::RS + gi * 16);
                dst[0] = lo;
                dst[1] = hi;
            }
        }
        __syncthreads();

        // ---- S = Q K^T for heads hg*16.., entries half*16..half*16+15
        float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        {
            const __half *qa = sQ + (hg * 16 + (lane & 15)) * C::RS + (lane >> 4) * 8;
            const __half *kb = sK + (half * 16 + (lane & 7) + ((lane >> 4) << 3)) * C::RS + ((lane >> 3) & 1) * 8;
#pragma unroll 4
            for (int ks = 0; ks < D / 16; ++ks) {
                uint32_t af[4], bfr[4];
                ldsm_x4(af, qa + ks * 16);
                ldsm_x4(bfr, kb + ks * 16);
                mma_f16(s[0], af[0], af[1], af[2], af[3], bfr[0], bfr[1]);
                mma_f16(s[1], af[0], af[1], af[2], af[3], bfr[2], bfr[3]);
            }
        }
        // ---- scale, mask, partial row max
        const int32_t *valid = sValid + st * TE + half * 16;
        float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                const bool ok = valid[nt * 8 + 2 * t4 + c] != 0;
                s[nt][c] = ok ? s[nt][c] * cs0 : -INFINITY;
                s[nt][2 + c] = ok ? s[nt][2 + c] * cs1 : -INFINITY;
                mx0 = fmaxf(mx0, s[nt][c]);
                mx1 = fmaxf(mx1, s[nt][2 + c]);
            }
        }
#pragma unroll
        for (int off = 1; off < 4; off <<= 1) {
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xFFFFFFFFu, mx0, off));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xFFFFFFFFu, mx1, off));
        }
        if (t4 == 0) {
            sMax[half * C::HB + r0] = mx0;
            sMax[half * C::HB + r1] = mx1;
        }
        __syncthreads();
        const float tm0 = fmaxf(sMax[r0], sMax[C::HB + r0]);
        const float tm1 = fmaxf(sMax[r1], sMax[C::HB + r1]);
        const float mn0 = fmaxf(m0, tm0), mn1 = fmaxf(m1, tm1);
        const float al0 = (mn0 == -INFINITY) ? 1.f : ex2(m0 - mn0);
        const float al1 = (mn1 == -INFINITY) ? 1.f : ex2(m1 - mn1);
        m0 = mn0;
        m1 = mn1;
        float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            float p[4];
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                p[c] = (s[nt][c] == -INFINITY) ? 0.f : ex2(s[nt][c] - mn0);
                p[2 + c] = (s[nt][2 + c] == -INFINITY) ? 0.f : ex2(s[nt][2 + c] - mn1);
            }
            const uint32_t lo = pack_f16x2(p[0], p[1]);
            const uint32_t hi = pack_f16x2(p[2], p[3]);
            // accumulate the f16-rounded probabilities so that l matches P V exactly
            const __half2 hl = *reinterpret_cast<const __half2 *>(&lo);
            const __half2 hh = *reinterpret_cast<const __half2 *>(&hi);
            ps0 += __low2float(hl) + __high2float(hl);
            ps1 += __low2float(hh) + __high2float(hh);
            const int col = half * 16 + nt * 8 + 2 * t4;
            *reinterpret_cast<uint32_t *>(sP + r0 * C::PS + col) = lo;
            *reinterpret_cast<uint32_t *>(sP + r1 * C::PS + col) = hi;
        }
        l0 = l0 * al0 + ps0;
        l1 = l1 * al1 + ps1;
#pragma unroll
        for (int i = 0; i < C::NT_PV; ++i) {
            o[i][0] *= al0; o[i][1] *= al0;
            o[i][2] *= al1; o[i][3] *= al1;
        }
        __syncthreads();  // sP complete

        // ---- O += P V : heads hg*16.., dv half*DVW .. +DVW, k = 32 entries
#pragma unroll
        for (int ks = 0; ks < TE / 16; ++ks) {
            uint32_t af[4];
            ldsm_x4(af, sP + (hg * 16 + (lane & 15)) * C::PS + ks * 16 + (lane >> 4) * 8);
            const __half *vb = sK + (ks * 16 + (lane & 7) + ((lane >> 3) & 1) * 8) * C::RS + half * C::DVW + (lane >> 4) * 8;
#pragma unroll
            for (int np = 0; np < C::NT_PV / 2; ++np) {
                uint32_t bfr[4];
                ldsm_x4_t(bfr, vb + np * 16);
                mma_f16(o[2 * np], af[0], af[1], af[2], af[3], bfr[0], bfr[1]);
                mma_f16(o[2 * np + 1], af[0], af[1], af[2], af[3], bfr[2], bfr[3]);
            }
        }
    }

    // ---- finalise: total l over the two entry halves, normalise, write
    for (int off = 1; off < 4; off <<= 1) {
        l0 += __shfl_xor_sync(0xFFFFFFFFu, l0, off);
        l1 += __shfl_xor_sync(0xFFFFFFFFu, l1, off);
    }
    __syncthreads();
    if (t4 == 0) {
        sMax[half * C::HB + r0] = l0;
        sMax[half * C::HB + r1] = l1;
    }
    __syncthreads();
    const float L0 = sMax[r0] + sMax[C::HB + r0];
    const float L1 = sMax[r1] + sMax[C::HB + r1];
    const float inv0 = L0 > 0.f ? 1.f / L0 : 0.f;
    const float inv1 = L1 > 0.f ? 1.f / L1 : 0.f;
    const float ln2 = 0.6931471805599453f;
    const float lse0 = L0 > 0.f ? (m0 + log2f(L0)) * ln2 : -INFINITY;
    const float lse1 = L1 > 0.f ? (m1 + log2f(L1)) * ln2 : -INFINITY;
    const int64_t hrow0 = bt * a.H + h0 + r0, hrow1 = bt * a.H + h0 + r1;
    float *dst0, *dst1;
    float *lse_dst;
    if (a.splits == 1) {
        dst0 = a.out + hrow0 * DV;
        dst1 = a.out + hrow1 * DV;
        lse_dst = a.lse;
    } else {
        const int64_t rows = (int64_t)a.B * a.T * a.H;
        dst0 = a.part_o + ((int64_t)split * rows + hrow0) * DV;
        dst1 = a.part_o + ((int64_t)split * rows + hrow1) * DV;
        lse_dst = a.part_lse + (int64_t)split * rows;
    }
#pragma unroll
    for (int i = 0; i < C::NT_PV; ++i) {
        const int col = half * C::DVW + i * 8 + 2 * t4;
        *reinterpret_cast<float2 *>(dst0 + col) = make_float2(o[i][0] * inv0, o[i][1] * inv0);
        *reinterpret_cast<float2 *>(dst1 + col) = make_float2(o[i][2] * inv1, o[i][3] * inv1);
    }
    if (lse_dst && half == 0 && t4 == 0) {
        lse_dst[hrow0] = lse0;
        lse_dst[hrow1] = lse1;
    }
}

// Merge split-KV partials: lse = log sum_s exp(lse_s), out = sum_s exp(lse_s - lse) O_s.
__global__ void __launch_bounds__(256) attn_combine_kernel(const float *__restrict__ part_o,
                                                           const float *__restrict__ part_lse, int splits,
                                                           int64_t rows, int dv, float *__restrict__ out,
                                                           float *__restrict__ lse) {
    pdl_wait();
    pdl_launch_dependents();
    const int64_t row = blockIdx.x;
    __shared__ float wts[64];
    __shared__ float s_lse;
    if (threadIdx.x == 0) {
        float m = -INFINITY;
        for (int s = 0; s < splits; ++s) m = fmaxf(m, part_lse[(int64_t)s * rows + row]);
        float tot = 0.f;
        for (int s = 0; s < splits; ++s) {
            const float l = part_lse[(int64_t)s * rows + row];
            const float w = (m == -INFINITY || l == -INFINITY) ? 0.f : expf(l - m);
            wts[s] = w;
            tot += w;
        }
        const float inv = tot > 0.f ? 1.f / tot : 0.f;
        for (int s = 0; s < splits; ++s) wts[s] *= inv;
        s_lse = tot > 0.f ? m + logf(tot) : -INFINITY;
    }
    __syncthreads();
    for (int c = threadIdx.x * 4; c < dv; c += blockDim.x * 4) {
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int s = 0; s < splits; ++s) {
            const float w = wts[s];
            if (w == 0.f) continue;
            const float4 v = *reinterpret_cast<const float4 *>(part_o + ((int64_t)s * rows + row) * dv + c);
            acc.x += w * v.x; acc.y += w * v.y; acc.z += w * v.z; acc.w += w * v.w;
        }
        *reinterpret_cast<float4 *>(out + row * dv + c) = acc;
    }
    if (lse && threadIdx.x == 0) lse[row] = s_lse;
}

int choose_splits(int64_t bt_hblocks, int K) {
    const int ntiles = (K + TE - 1) / TE;
    int64_t s = num_sms() / (bt_hblocks > 0 ? bt_hblocks : 1);
    if (s < 1) s = 1;
    if (s > ntiles) s = ntiles;
    if (s > 64) s = 64;
    return (int)s;
}

template <int D, int DV, int NG>
csa2_status launch_attn(AttnArgs a, cudaStream_t stream) {
    using C = AttnCfg<D, DV, NG>;
    auto kern = sparse_attn_kernel<D, DV, NG>;
    static bool smem_set[64];
    CSA2_CUDA_CALL(ensure_smem_limit((const void *)kern, (int)C::SMEM, smem_set), "sparse_attn: smem attribute");
    dim3 grid((unsigned)((int64_t)a.B * a.T), a.splits, a.H / C::HB);
    CSA2_CUDA_CALL(launch_pdl(kern, grid, dim3(C::THREADS), C::SMEM, stream, a), "sparse_attn_kernel launch");
    CSA2_LAUNCH_CHECK("sparse_attn_kernel");
    if (a.splits > 1) {
        const int64_t rows = (int64_t)a.B * a.T * a.H;
        CSA2_CUDA_CALL(launch_pdl(attn_combine_kernel, dim3((unsigned)rows), dim3(128), 0, stream,
                                  (const float *)a.part_o, (const float *)a.part_lse, a.splits, rows, DV, a.out,
                                  a.lse),
                       "attn_combine_kernel launch");
        CSA2_LAUNCH_CHECK("attn_combine_kernel");
    }
    return CSA2_OK;
}

int heads_per_cta(int D) { return D == 576 ? 64 : 16; }

bool supported(int D, int dv, int H) {
    if (D == 576 && dv == 512) return H % 64 == 0;
    if (D == 128 && dv == 64) return H % 16 == 0;
    return false;
}

}  // namespace
}  // namespace csa2

using namespace csa2;

extern "C" size_t csa2_sparse_attn_workspace_bytes(int B, int T, int H, int D, int dv, int K) {
    if (B <= 0 || T <= 0 || H <= 0 || K <= 0 || !supported(D, dv, H)) return 0;
    if (sparse_attn_tc_supported(D, dv, H, K)) return 0;  // cluster-merged, no scratch
    const int64_t bt = (int64_t)B * T;
    const int splits = choose_splits(bt * (H / heads_per_cta(D)), K);
    if (splits <= 1) return 0;
    const int64_t rows = bt * H;
    return (size_t)splits * rows * ((size_t)dv + 1) * sizeof(float) + 256;
}

// The attention of csa2_sparse_attn_fp4, with an optional L2 prefetch of the
// selected rows of a second pair of planes (pf_codes / pf_scales).
static csa2_status sparse_attn_impl(csa2_mode mode, int B, int T, int H, int D, int dv, const void *q,
                                    const uint8_t *codes, const uint8_t *scales, int64_t N, const int32_t *idx,
                                    int K, const int32_t *kv_len, float sm_scale, void *out, csa2_dtype out_dt,
                                    float *lse, uint32_t *err_flag, void *workspace, size_t ws_bytes,
                                    const uint8_t *pf_codes, const uint8_t *pf_scales, csa2_stream_t stream) {
    CSA2_REQUIRE(mode == CSA2_MODE_FULL || mode == CSA2_MODE_REINDEX || mode == CSA2_MODE_REUSE,
                 "sparse_attn: bad mode %d", (int)mode);
    CSA2_REQUIRE(B >= 0 && T >= 0 && H >= 0 && N >= 0, "sparse_attn: negative shape");
    CSA2_REQUIRE(K >= 1 && K <= CSA2_MAX_K, "sparse_attn: K=%d not in [1,2048]", K);
    CSA2_REQUIRE(out_dt == CSA2_FP32, "sparse_attn: only fp32 output is supported");
    if (!supported(D, dv, H)) {
        set_error("sparse_attn: unsupported (D=%d, dv=%d, H=%d)", D, dv, H);
        return CSA2_ERR_UNSUPPORTED;
    }
    if ((int64_t)B * T == 0 || H == 0) return CSA2_OK;
    CSA2_REQUIRE(q && codes && scales && idx && out, "sparse_attn: null pointer");
    CSA2_REQUIRE(aligned(q, 16) && aligned(codes, 16) && aligned(scales, 4), "sparse_attn: q/codes need 16-byte, scales 4-byte alignment");
    CSA2_REQUIRE(aligned(out, 16) && aligned(idx, 4), "sparse_attn: out needs 16-byte alignment");
    CSA2_REQUIRE((int64_t)B * T <= 0x7FFFFFFFLL && H / heads_per_cta(D) <= 65535, "sparse_attn: too many query tokens or heads");

    if (sparse_attn_tc_supported(D, dv, H, K))
        return launch_sparse_attn_tc(B, T, H, K, N, q, codes, scales, idx, kv_len, sm_scale, (float *)out, lse,
                                     err_flag, pf_codes, pf_scales, stream_of(stream));

    AttnArgs a = {};
    a.B = B; a.T = T; a.H = H; a.K = K; a.N = N;
    a.q = (const uint16_t *)q; a.codes = codes; a.scales = scales; a.idx = idx; a.kv_len = kv_len;
    a.sm_scale = sm_scale; a.out = (float *)out; a.lse = lse; a.err_flag = err_flag;
    const int64_t bt = (int64_t)B * T;
    a.splits = choose_splits(bt * (H / heads_per_cta(D)), K);
    if (a.splits > 1) {
        const size_t need = csa2_sparse_attn_workspace_bytes(B, T, H, D, dv, K);
        if (!workspace || ws_bytes < need) {
            set_error("sparse_attn: workspace of %zu bytes required, %zu given", need, workspace ? ws_bytes : 0);
            return CSA2_ERR_WORKSPACE;
        }
        CSA2_REQUIRE(aligned(workspace, 16), "sparse_attn: workspace must be 16-byte aligned");
        const int64_t rows = bt * H;
        a.part_o = (float *)workspace;
        a.part_lse = a.part_o + (size_t)a.splits * rows * dv;
    }
    if (D == 576) return launch_attn<576, 512, 4>(a, stream_of(stream));
    return launch_attn<128, 64, 1>(a, stream_of(stream));
}

extern "C" csa2_status csa2_sparse_attn_fp4(csa2_mode mode, int B, int T, int H, int D, int dv,
                                            const void *q, const uint8_t *codes, const uint8_t *scales,
                                            int64_t N, const int32_t *idx, int K, const int32_t *kv_len,
                                            float sm_scale, void *out, csa2_dtype out_dt, float *lse,
                                            uint32_t *err_flag, void *workspace, size_t ws_bytes,
                                            csa2_stream_t stream) {
    clear_error();
    return sparse_attn_impl(mode, B, T, H, D, dv, q, codes, scales, N, idx, K, kv_len, sm_scale, out, out_dt, lse,
                            err_flag, workspace, ws_bytes, nullptr, nullptr, stream);
}

extern "C" csa2_status csa2_sparse_attn_fp4_prefetch(csa2_mode mode, int B, int T, int H, int D, int dv,
                                                     const void *q, const uint8_t *codes, const uint8_t *scales,
                                                     int64_t N, const int32_t *idx, int K, const int32_t *kv_len,
                                                     float sm_scale, void *out, csa2_dtype out_dt, float *lse,
                                                     uint32_t *err_flag, void *workspace, size_t ws_bytes,
                                                     const uint8_t *next_codes, const uint8_t *next_scales,
                                                     csa2_stream_t stream) {
    clear_error();
    CSA2_REQUIRE((next_codes == nullptr) == (next_scales == nullptr),
                 "sparse_attn_prefetch: next_codes and next_scales go together");
    CSA2_REQUIRE(aligned(next_codes, 16) && aligned(next_scales, 4),
                 "sparse_attn_prefetch: next_codes needs 16-byte, next_scales 4-byte alignment");
    return sparse_attn_impl(mode, B, T, H, D, dv, q, codes, scales, N, idx, K, kv_len, sm_scale, out, out_dt, lse,
                            err_flag, workspace, ws_bytes, next_codes, next_scales, stream);
}

// ---------------------------------------------------------------------------
// No-allocation variant of csa2_sparse_attn_fp4.
//
// The split-KV attention needs scratch memory for its per-split partial
// outputs.  csa2_sparse_attn_fp4 takes that scratch from the caller; callers
// that may not allocate device memory at all (an engine that hands out every
// byte from a pool planned before serving starts, or code that must not call
// cudaMalloc/cudaFree because those calls can synchronise the device) use
// this entry point instead.  Its scratch is one file-scope device array of
// kNoAllocScratchBytes that is part of the library image: every GPU that
// loads the library holds it until the process exits.  The split policy keeps
// splits x query tokens x head blocks <= the SM count, so a shape needs at most
// SMs x 64 heads x (512 + 1) x 4 bytes (19.96 MB on a 152-SM GB300); larger
// GPUs may meet shapes that do not fit, which are rejected.
namespace csa2 {
namespace {
constexpr size_t kNoAllocScratchBytes = (size_t)20 << 20;  // 20 MiB
}
}  // namespace csa2

static __device__ __align__(256) unsigned char g_noalloc_attn_scratch[csa2::kNoAllocScratchBytes];

namespace csa2 {
namespace {
// Device address of the scratch array, looked up once per device with that
// device current (in host code the array's name is only a host-side stand-in).
std::mutex g_noalloc_mu;
void *g_noalloc_ptr[64];

cudaError_t noalloc_scratch(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_attn_scratch);
        if (e != cudaSuccess) return e;
        g_noalloc_ptr[dev] = p;
    }
    *out = g_noalloc_ptr[dev];
    return cudaSuccess;
}
}  // namespace
}  // namespace csa2

extern "C" size_t csa2_sparse_attn_noalloc_max_scratch_bytes(void) { return csa2::kNoAllocScratchBytes; }

extern "C" csa2_status csa2_sparse_attn_fp4_noalloc(csa2_mode mode, int B, int T, int H, int D, int dv,
                                                    const void *q, const uint8_t *codes, const uint8_t *scales,
                                                    int64_t N, const int32_t *idx, int K, const int32_t *kv_len,
                                                    float sm_scale, void *out, csa2_dtype out_dt, float *lse,
                                                    uint32_t *err_flag, csa2_stream_t stream) {
    clear_error();
    const size_t need = csa2_sparse_attn_workspace_bytes(B, T, H, D, dv, K);
    if (need > kNoAllocScratchBytes) {
        set_error("sparse_attn_noalloc: this shape needs %zu bytes of scratch, the built-in array holds %zu; "
                  "use csa2_sparse_attn_fp4 with a caller workspace",
                  need, kNoAllocScratchBytes);
        return CSA2_ERR_WORKSPACE;
    }
    void *scratch = nullptr;
    if (need > 0) {
        int dev = 0;
        CSA2_CUDA_CALL(cudaGetDevice(&dev), "sparse_attn_noalloc: current device");
        if (dev < 0 || dev >= 64) {
            set_error("sparse_attn_noalloc: device ordinal %d; the scratch address table covers devices 0-63", dev);
            return CSA2_ERR_UNSUPPORTED;
        }
        CSA2_CUDA_CALL(noalloc_scratch(&scratch), "sparse_attn_noalloc: scratch address");
    }
    // Every split rewrites all of its partial rows (empty splits write zeros
    // and lse = -inf), so nothing in the array needs clearing between calls.
    return csa2_sparse_attn_fp4(mode, B, T, H, D, dv, q, codes, scales, N, idx, K, kv_len, sm_scale, out, out_dt,
                                lse, err_flag, scratch, need > 0 ? kNoAllocScratchBytes : 0, stream);
}

extern "C" csa2_status csa2_swa_attn_fp8(int B, int T, int H, int D, int dv, const void *q, const uint8_t *swa_kv, int W,
                                         const int32_t *swa_len, float sm_scale, const float *o_sparse,
                                         const float *lse_sparse, float *out, float *lse, uint32_t *err_flag,
                                         csa2_stream_t stream) {
    clear_error();
    CSA2_REQUIRE(B >= 0 && T >= 0 && H >= 0, "swa_attn: negative shape");
    CSA2_REQUIRE(W >= 1 && W <= 512, "swa_attn: window capacity W=%d not in [1,512]", W);
    if (!(D == 576 && dv == 512 && H % 64 == 0)) {
        set_error("swa_attn: unsupported (D=%d, dv=%d, H=%d): D=576, dv=512, H a multiple of 64", D, dv, H);
        return CSA2_ERR_UNSUPPORTED;
    }
    CSA2_REQUIRE((o_sparse == nullptr) == (lse_sparse == nullptr), "swa_attn: o_sparse and lse_sparse go together");
    if ((int64_t)B * T == 0 || H == 0) return CSA2_OK;
    CSA2_REQUIRE(q && swa_kv && swa_len && out, "swa_attn: null pointer");
    CSA2_REQUIRE(aligned(q, 16) && aligned(swa_kv, 16) && aligned(out, 16) && aligned(swa_len, 4) &&
                     aligned(o_sparse, 16) && aligned(lse_sparse, 4) && aligned(lse, 4),
                 "swa_attn: q, swa_kv, out, o_sparse need 16-byte alignment");
    CSA2_REQUIRE((int64_t)B * T <= 0x7FFFFFFFLL, "swa_attn: too many query tokens");
    return launch_swa_attn_tc(B, T, H, q, swa_kv, W, swa_len, sm_scale, o_sparse, lse_sparse, out, lse, err_flag,
                              stream_of(stream));
}

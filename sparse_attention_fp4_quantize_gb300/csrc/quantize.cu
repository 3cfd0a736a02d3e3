// csa2_quantize_kv_fp4: post-RoPE bf16 KV rows -> FP4 E2M1 codes + one E4M3
// scale per 16 channels, no global scale.
// Source: "DeepSeek-V4.1-Flash：把 KV Cache 压缩到极限的百万上下文 MoE", section
// "效率组件四件", item 4 "FP4 主 KV Cache" (E2M1 + per-16-channel E4M3 scale,
// NVFP4-like without the second-level scale, quantised after RoPE).
//
// HBM-bound streaming kernel.  A thread takes 16-byte units (8 bf16 channels),
// UNR per pass; the two lanes of a pair own the two halves of a 16-channel
// group and exchange their half-amax with one shuffle.  Loads are 128-bit,
// read-only and L1-bypassing; each unit writes 4 code bytes and (even lane)
// 1 scale byte.
//
// Exact rounding without a divide.  Let s be the group scale (4 significant
// bits) and x a bf16 value (8 significant bits).  A tie of |x|/s on the E2M1
// grid (or of amax/6 on the E4M3 grid) happens only when the quotient is
// EXACTLY a midpoint, which has at most 5 significant bits; any other
// quotient lies at least 2^-8 (relative) away from every midpoint.  So the
// quotient is formed with a multiply by an approximate reciprocal (relative
// error < 2^-21), rounded to 12 significant bits -- which restores exact
// midpoints and cannot move any other value across one -- and then converted
// by the hardware's round-to-nearest-even, saturating cvt instruction.
#include "common.cuh"

namespace csa2 {
namespace {

// Division of a 32-bit unsigned by a runtime-invariant divisor with one
// multiply-high (Granlund & Montgomery, "Division by invariant integers using
// multiplication", PLDI 1994, round-up method with the n-bit fix-up).
struct FastDiv {
    uint32_t d, m, s;
    void init(uint32_t dd) {
        d = dd;
        if (dd == 1) { m = 0; s = 0; return; }
        uint32_t l = 32 - __builtin_clz(dd - 1);
        m = (uint32_t)((((1ull << 32) * ((1ull << l) - dd)) / dd) + 1);
        s = l;
    }
};

__device__ __forceinline__ uint32_t fdiv(uint32_t n, const FastDiv &f) {
    if (f.d == 1) return n;
    uint32_t t = __umulhi(n, f.m);
    return (t + ((n - t) >> 1)) >> (f.s - 1);
}

__device__ __forceinline__ uint4 ld_stream_v4(const void *p) {
    uint4 r;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

// Round a positive-or-negative fp32 to 12 significant bits (nearest).
__device__ __forceinline__ float round12(float v) {
    return __uint_as_float((__float_as_uint(v) + 0x800u) & 0xFFFFF000u);
}

// fp32 -> E4M3 byte, round to nearest even, saturating at +-448.
__device__ __forceinline__ uint32_t to_e4m3(float v) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(v));
    return r & 0xFFu;
}

// E4M3 byte -> fp32 (exact: via f16x2).
__device__ __forceinline__ float e4m3_to_f32(uint32_t b) {
    uint32_t h2;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"((uint16_t)b));
    return __half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFFu)));
}

// Two fp32 -> one byte of two E2M1 codes (hi -> upper nibble), RNE, satfinite.
__device__ __forceinline__ uint32_t to_e2m1x2(float hi, float lo) {
    uint32_t r;
    asm("{\n\t.reg .b8 t;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\t"
        "cvt.u32.u8 %0, t;\n\t}"
        : "=r"(r)
        : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ float rcp_approx(float x) {
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

// |bf16| max of the 8 values in a 16-byte unit, as fp32.
__device__ __forceinline__ float unit_amax(const uint4 &v) {
    const uint32_t m = 0x7FFF7FFFu;
    __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162 *>(&v.x);
    uint32_t w0 = v.x & m, w1 = v.y & m, w2 = v.z & m, w3 = v.w & m;
    a = __hmax2(*reinterpret_cast<__nv_bfloat162 *>(&w0), *reinterpret_cast<__nv_bfloat162 *>(&w1));
    __nv_bfloat162 c = __hmax2(*reinterpret_cast<__nv_bfloat162 *>(&w2), *reinterpret_cast<__nv_bfloat162 *>(&w3));
    a = __hmax2(a, c);
    return fmaxf(__low2float(a), __high2float(a));
}

__device__ __forceinline__ uint32_t encode_word(uint32_t w, float inv) {
    float lo = __uint_as_float(w << 16);
    float hi = __uint_as_float(w & 0xFFFF0000u);
    return to_e2m1x2(round12(hi * inv), round12(lo * inv));
}

constexpr int kThreads = 256;
// Units per thread per pass (UNR): 8 for large plain appends, 2 for small
// appends (a decode step's few hundred rows, which then spread over more
// SMs), 1 for the rotated units of the RoPE pass.

// RoPE of the append path, fused ahead of the quantiser: interleaved pairs
// (2i, 2i+1) of the last rope_dim channels rotated by a caller-supplied fp32
// table cos_sin[pos][i] = (cos, sin), in fp32 without fused multiply-add, then
// rounded to bf16 (nearest even) -- the rows the unfused path would store.
struct RopeArgs {
    const int32_t *pos;      // [rows] token position of each row
    const float2 *cos_sin;   // [n_pos, rope_dim / 2]
    int64_t n_pos;
    int rope_dim;
};

__device__ __forceinline__ uint32_t rope_word(uint32_t w, float2 cs) {
    const float a = __uint_as_float(w << 16), b = __uint_as_float(w & 0xFFFF0000u);
    const float ra = __fsub_rn(__fmul_rn(a, cs.x), __fmul_rn(b, cs.y));
    const float rb = __fadd_rn(__fmul_rn(a, cs.y), __fmul_rn(b, cs.x));
    return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(ra)) |
           ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(rb)) << 16);
}

template <bool ROPE, int UNR>
__global__ void __launch_bounds__(kThreads) quantize_fp4_kernel(
    const uint16_t *__restrict__ kv, uint32_t total_units, FastDiv upr_div, uint32_t first_unit, int D,
    int64_t stride, int64_t row0, const int64_t *__restrict__ dst_slot, int64_t n_slots,
    uint8_t *__restrict__ codes, uint8_t *__restrict__ scales, uint32_t *err_flag, RopeArgs rope) {
    pdl_wait();
    pdl_launch_dependents();
    const int lane = threadIdx.x & 31;
    const uint32_t nthreads = gridDim.x * kThreads;
    const uint32_t upr = upr_div.d;
    constexpr int kUnroll = UNR;
    // Warp-aligned base so that lane parity == unit parity (pairs share a group).
    for (uint32_t base = blockIdx.x * kThreads + (threadIdx.x & ~31u); base < total_units;
         base += nthreads * kUnroll) {
        uint4 v[kUnroll];
        uint32_t rr[kUnroll], ur[kUnroll];
        bool ok[kUnroll];
#pragma unroll
        for (int k = 0; k < kUnroll; ++k) {
            uint32_t u = base + lane + k * nthreads;
            ok[k] = u < total_units;
            uint32_t r = fdiv(ok[k] ? u : 0u, upr_div);
            rr[k] = r;
            ur[k] = first_unit + ((ok[k] ? u : 0u) - r * upr);
            v[k] = make_uint4(0, 0, 0, 0);
            if (ok[k]) v[k] = ld_stream_v4(kv + (row0 + r) * stride + (int64_t)ur[k] * 8);
        }
        if constexpr (ROPE) {
            const uint32_t u0 = (uint32_t)(D - rope.rope_dim) / 8;   // first unit of the rotated channels
#pragma unroll
            for (int k = 0; k < kUnroll; ++k) {
                if (!ok[k] || ur[k] < u0) continue;
                const int64_t p = rope.pos[row0 + rr[k]];
                if (p < 0 || p >= rope.n_pos) {   // both units of the group see the same row: skipped together
                    flag_error(err_flag, CSA2_FLAG_BAD_INDEX);
                    ok[k] = false;
                    continue;
                }
                const float2 *t = rope.cos_sin + p * (rope.rope_dim / 2) + (ur[k] - u0) * 4;
                v[k] = make_uint4(rope_word(v[k].x, t[0]), rope_word(v[k].y, t[1]), rope_word(v[k].z, t[2]),
                                  rope_word(v[k].w, t[3]));
            }
        }
#pragma unroll
        for (int k = 0; k < kUnroll; ++k) {
            // Warp-uniform: every lane of the warp takes part in the shuffle.
            float amax = unit_amax(v[k]);
            amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
            if (!ok[k]) continue;
            uint32_t sbyte = to_e4m3(round12(amax * (1.0f / 6.0f)));
            float inv = sbyte ? rcp_approx(e4m3_to_f32(sbyte)) : 0.0f;
            uint32_t c = encode_word(v[k].x, inv) | (encode_word(v[k].y, inv) << 8) |
                         (encode_word(v[k].z, inv) << 16) | (encode_word(v[k].w, inv) << 24);
            int64_t row = row0 + rr[k];
            int64_t slot = row;
            if (dst_slot) {
                slot = dst_slot[row];
                if (slot < 0 || slot >= n_slots) {
                    flag_error(err_flag, CSA2_FLAG_BAD_SLOT);
                    continue;
                }
            }
            *reinterpret_cast<uint32_t *>(codes + slot * (int64_t)(D / 2) + (int64_t)ur[k] * 4) = c;
            if ((ur[k] & 1) == 0) scales[slot * (int64_t)(D / 16) + ur[k] / 2] = (uint8_t)sbyte;
        }
    }
}

}  // namespace
}  // namespace csa2

using namespace csa2;

// Units (16-byte pieces of a row) [first_unit, first_unit + upr) of every row,
// in launches whose unit count fits comfortably in 32 bits.
template <bool ROPE>
static csa2_status launch_quantize_units(const void *kv, int64_t rows, int D, int64_t kv_row_stride, uint32_t first_unit,
                                         uint32_t upr, const int64_t *dst_slot, int64_t n_slots, uint8_t *codes,
                                         uint8_t *scales, uint32_t *err_flag, const RopeArgs &ra, csa2_stream_t stream) {
    FastDiv fd;
    fd.init(upr);
    const int64_t max_rows = (int64_t)(0x7FFFFFFFu / upr);
    const int max_blocks = num_sms() * 8;
    for (int64_t r0 = 0; r0 < rows; r0 += max_rows) {
        int64_t nr = rows - r0 < max_rows ? rows - r0 : max_rows;
        uint32_t units = (uint32_t)(nr * upr);
        // Plain units: the short unroll for small appends, the long one for
        // large ones (the grid then covers every SM several times over).
        // Rotated units: one per thread (the position -> table chain of each
        // unit is latency-bound: 2 or 4 per thread measured 346 / 364 us at
        // 1M rows against 345, 8 per thread 392).
        const bool small = (int64_t)units < (int64_t)num_sms() * kThreads * 16;
        const int unr = ROPE ? 1 : (small ? 2 : 8);
        const int64_t per_block = (int64_t)kThreads * unr;
        int64_t want = ((int64_t)units + per_block - 1) / per_block;
        int blocks = (int)(want < max_blocks ? want : max_blocks);
        if (blocks < 1) blocks = 1;
        void (*kern)(const uint16_t *, uint32_t, FastDiv, uint32_t, int, int64_t, int64_t, const int64_t *, int64_t,
                     uint8_t *, uint8_t *, uint32_t *, RopeArgs);
        if constexpr (ROPE) kern = quantize_fp4_kernel<true, 1>;
        else kern = small ? quantize_fp4_kernel<false, 2> : quantize_fp4_kernel<false, 8>;
        CSA2_CUDA_CALL(launch_pdl(kern, dim3(blocks), dim3(kThreads), 0, stream_of(stream), (const uint16_t *)kv,
                                  units, fd, first_unit, D, kv_row_stride, r0, dst_slot, n_slots, codes, scales,
                                  err_flag, ra),
                       "quantize_fp4_kernel launch");
        CSA2_LAUNCH_CHECK("quantize_fp4_kernel");
    }
    return CSA2_OK;
}

// Without RoPE: every unit of every row in one pass.  With RoPE: the latent
// units by the plain kernel (no rotation work, no divergence), then the
// rotated units by the RoPE kernel, whose warps all rotate.
static csa2_status launch_quantize(const void *kv, int64_t rows, int D, int64_t kv_row_stride,
                                   const int64_t *dst_slot, int64_t n_slots, uint8_t *codes, uint8_t *scales,
                                   uint32_t *err_flag, const RopeArgs *rope, csa2_stream_t stream) {
    const uint32_t upr = (uint32_t)(D / 8);
    const RopeArgs none = {nullptr, nullptr, 0, 0};
    if (!rope)
        return launch_quantize_units<false>(kv, rows, D, kv_row_stride, 0, upr, dst_slot, n_slots, codes, scales,
                                            err_flag, none, stream);
    const uint32_t u0 = (uint32_t)(D - rope->rope_dim) / 8;
    if (u0 > 0) {
        const csa2_status st = launch_quantize_units<false>(kv, rows, D, kv_row_stride, 0, u0, dst_slot, n_slots,
                                                            codes, scales, err_flag, none, stream);
        if (st != CSA2_OK) return st;
    }
    return launch_quantize_units<true>(kv, rows, D, kv_row_stride, u0, upr - u0, dst_slot, n_slots, codes, scales,
                                       err_flag, *rope, stream);
}

#define CSA2_QUANT_CHECKS()                                                                                    \
    CSA2_REQUIRE(rows >= 0, "quantize: rows < 0");                                                            \
    CSA2_REQUIRE(D >= 16 && D <= 4096 && D % 16 == 0, "quantize: D=%d must be a multiple of 16 in [16,4096]", \
                 D);                                                                                           \
    CSA2_REQUIRE(kv_row_stride >= D && kv_row_stride % 8 == 0,                                                 \
                 "quantize: kv_row_stride=%lld must be >= D and a multiple of 8", (long long)kv_row_stride);   \
    CSA2_REQUIRE(n_slots >= 0, "quantize: n_slots < 0");                                                      \
    CSA2_REQUIRE(dst_slot || rows <= n_slots, "quantize: rows > n_slots without dst_slot")

extern "C" csa2_status csa2_quantize_kv_fp4(const void *kv, int64_t rows, int D,
                                            int64_t kv_row_stride, const int64_t *dst_slot,
                                            int64_t n_slots, uint8_t *codes, uint8_t *scales,
                                            uint32_t *err_flag, csa2_stream_t stream) {
    clear_error();
    CSA2_QUANT_CHECKS();
    if (rows == 0) return CSA2_OK;
    CSA2_REQUIRE(kv && codes && scales, "quantize: null pointer");
    CSA2_REQUIRE(aligned(kv, 16), "quantize: kv must be 16-byte aligned");
    CSA2_REQUIRE(aligned(codes, 4), "quantize: codes must be 4-byte aligned");
    CSA2_REQUIRE(!dst_slot || aligned(dst_slot, 8), "quantize: dst_slot must be 8-byte aligned");
    return launch_quantize(kv, rows, D, kv_row_stride, dst_slot, n_slots, codes, scales, err_flag, nullptr, stream);
}

extern "C" csa2_status csa2_rope_quantize_kv_fp4(const void *kv, int64_t rows, int D, int64_t kv_row_stride,
                                                 const int32_t *pos, const float *cos_sin, int64_t n_pos,
                                                 int rope_dim, const int64_t *dst_slot, int64_t n_slots,
                                                 uint8_t *codes, uint8_t *scales, uint32_t *err_flag,
                                                 csa2_stream_t stream) {
    clear_error();
    CSA2_QUANT_CHECKS();
    CSA2_REQUIRE(rope_dim >= 16 && rope_dim <= D && rope_dim % 16 == 0,
                 "rope_quantize: rope_dim=%d must be a multiple of 16 in [16, D]", rope_dim);
    CSA2_REQUIRE(n_pos >= 1, "rope_quantize: n_pos < 1");
    if (rows == 0) return CSA2_OK;
    CSA2_REQUIRE(kv && codes && scales && pos && cos_sin, "rope_quantize: null pointer");
    CSA2_REQUIRE(aligned(kv, 16), "quantize: kv must be 16-byte aligned");
    CSA2_REQUIRE(aligned(codes, 4), "quantize: codes must be 4-byte aligned");
    CSA2_REQUIRE(!dst_slot || aligned(dst_slot, 8), "quantize: dst_slot must be 8-byte aligned");
    CSA2_REQUIRE(aligned(pos, 4) && aligned(cos_sin, 8), "rope_quantize: misaligned pos / cos_sin");
    const RopeArgs ra = {pos, reinterpret_cast<const float2 *>(cos_sin), n_pos, rope_dim};
    return launch_quantize(kv, rows, D, kv_row_stride, dst_slot, n_slots, codes, scales, err_flag, &ra, stream);
}

// Internal helpers shared by the libcsa2 translation units (host argument
// checks, thread-local error text, small device utilities).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>

#include "csa2.h"

namespace csa2 {

// ---------------------------------------------------------------- host side
void set_error(const char *fmt, ...);
void clear_error();
int num_sms();                 // SM count of the current device (cached per device)
int max_smem_optin();          // max dynamic shared memory per block (opt-in)

#define CSA2_REQUIRE(cond, ...)                 \
    do {                                        \
        if (!(cond)) {                          \
            ::csa2::set_error(__VA_ARGS__);     \
            return CSA2_ERR_INVALID_ARG;        \
        }                                       \
    } while (0)

#define CSA2_LAUNCH_CHECK(what)                                              \
    do {                                                                     \
        cudaError_t e_ = cudaGetLastError();                                 \
        if (e_ != cudaSuccess) {                                             \
            ::csa2::set_error("%s: %s", what, cudaGetErrorString(e_));      \
            return CSA2_ERR_CUDA;                                            \
        }                                                                    \
    } while (0)

#define CSA2_CUDA_CALL(call, what)                                           \
    do {                                                                     \
        cudaError_t e_ = (call);                                             \
        if (e_ != cudaSuccess) {                                             \
            ::csa2::set_error("%s: %s", what, cudaGetErrorString(e_));      \
            return CSA2_ERR_CUDA;                                            \
        }                                                                    \
    } while (0)

static inline bool aligned(const void *p, size_t a) { return ((uintptr_t)p % a) == 0; }

// Raise a kernel's dynamic shared-memory limit once per device (so that only
// kernel launches are issued while a caller captures a CUDA graph).
// `done` is per-kernel storage for up to 64 devices.
static inline cudaError_t ensure_smem_limit(const void *func, int bytes, bool *done) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64 && done[dev]) return cudaSuccess;
    e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess && dev >= 0 && dev < 64) done[dev] = true;
    return e;
}
static inline cudaStream_t stream_of(csa2_stream_t s) { return (cudaStream_t)s; }

// tcgen05 sparse attention (attn_tc.cu): D = 576, dv = 512, 64-head blocks, K <= 1024.
bool sparse_attn_tc_supported(int D, int dv, int H, int K);
// pf_codes / pf_scales: optional planes whose selected rows are prefetched into L2 (may be NULL).
csa2_status launch_sparse_attn_tc(int B, int T, int H, int K, int64_t N, const void *q, const uint8_t *codes,
                                  const uint8_t *scales, const int32_t *idx, const int32_t *kv_len, float sm_scale,
                                  float *out, float *lse, uint32_t *err_flag, const uint8_t *pf_codes,
                                  const uint8_t *pf_scales, cudaStream_t stream);
csa2_status launch_swa_attn_tc(int B, int T, int H, const void *q, const uint8_t *kv8, int W, const int32_t *swa_len,
                               float sm_scale, const float *o_sparse, const float *lse_sparse, float *out, float *lse,
                               uint32_t *err_flag, cudaStream_t stream);

// tcgen05 prefill scoring (index_score_tc.cu): FP8, Full mode, T >= 64.
bool index_score_prefill_tc_supported(int T, csa2_dtype dt);
csa2_status launch_index_score_prefill_tc(int B, int T, int64_t N, const void *q, const float *w, const void *k,
                                          const int32_t *kv_len, float *scores, uint32_t *err_flag,
                                          cudaStream_t stream);
// The first pass of the fused dense indexer (same tiles and MMAs as above):
// 8-key block-maximum keys [B*T, nblk].
csa2_status launch_prefill_block_max(int B, int T, int64_t N, const void *q, const float *w, const void *k,
                                     const int32_t *kv_len, uint32_t *bmax, int64_t nblk, uint32_t *err_flag,
                                     cudaStream_t stream);

// --------------------------------------------------------------- device side
// Order-preserving map of an fp32 score to uint32: larger score -> larger key.
// -inf (and NaN bit patterns that would sort below it) map to 0, the
// "not a candidate" key; every finite value maps to a key >= 0x00800000.
// -0 and +0 map to the same key.
__device__ __forceinline__ uint32_t score_key(float f) {
    uint32_t u = (f == 0.0f) ? 0u : __float_as_uint(f);
    uint32_t k = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    return (k <= 0x007FFFFFu) ? 0u : k;
}

// Programmatic dependent launch.  The library's kernels (all but the
// standalone Top-K) are launched with programmatic stream serialization allowed, so
// they may start while the previous kernel on the stream drains.  Before
// pdl_wait() a kernel touches only its own shared memory, TMEM and barriers;
// pdl_wait() returns once the previous grid has completed with its memory
// writes visible (without the launch attribute it returns at once).
// pdl_launch_dependents() lets the next kernel begin launching: at the start
// of short kernels, before the final phase of the attention and Top-K.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

static inline cudaLaunchAttribute pdl_attribute() {
    cudaLaunchAttribute at;
    at.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at.val.programmaticStreamSerializationAllowed = 1;
    return at;
}

// Plain (non-cluster) launch with the programmatic-serialization attribute.
template <typename... KArgs, typename... Args>
static inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                     cudaStream_t stream, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1] = {pdl_attribute()};
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// FP8 x FP8 -> fp32 tensor-core product, 16 keys x 8 columns x 32 d-values.
// A registers: {row g, k 4t..4t+3}, {row g+8, same k}, {row g, k 16+4t..}, {row g+8, ...};
// B registers: {k 4t..4t+3}, {k 16+4t..} of column g (g = lane / 4, t = lane % 4).
__device__ __forceinline__ void mma_e4m3_16832(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Four E4M3 bytes -> two f16x2 (bytes 0,1 -> lo; bytes 2,3 -> hi): exact, every
// E4M3 value is an f16 value.
__device__ __forceinline__ void e4m3x4_to_f16x2x2(uint32_t w, uint32_t &lo, uint32_t &hi) {
    asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\tcvt.rn.f16x2.e4m3x2 %0, l;\n\tcvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
        : "=r"(lo), "=r"(hi)
        : "r"(w));
}

// D += A . B, m16n8k16, f16 operands, fp32 accumulate (the legacy warp MMA).
__device__ __forceinline__ void mma_f16_16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                              uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void flag_error(uint32_t *err_flag, uint32_t bit) {
    if (err_flag) atomicOr(err_flag, bit);
}

}  // namespace csa2

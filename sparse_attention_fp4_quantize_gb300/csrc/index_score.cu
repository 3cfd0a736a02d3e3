// csa2_index_score: indexer scores sum_h w_h * ReLU(q_h . k) of query tokens
// against compressed index keys, over every entry (Full) or over the pool
// candidates (Reindex).
// Source: "DeepSeek-V4.1-Flash：把 KV Cache 压缩到极限的百万上下文 MoE", section
// "Hierarchical Sparse Indexer——索引成本变常数" (Full layers score all entries;
// Reindex layers only the <= 2048 x 8 pool); "DeepSeek-V4.1-Flash: Pushing the
// Limits of KV Cache Compression", CSA2 paragraph (Reindex reuses the KV and
// rescores with its own indexer Q).  The score formula is not on the pages.
//
// Decode-shaped (few query tokens per sequence): the work is a stream over
// the 64-byte keys, so one warp takes 16 keys at a time and puts them on the
// tensor cores as the A operand of an MMA with fp32 accumulation: FP8 keys
// and queries go straight into mma.m16n8k32 (e4m3 x e4m3; the products are
// exact), bf16 ones into mma.m16n8k16.  The B operand holds the 4 heads of up
// to two query tokens of the same sequence (8 columns).
//
// The dot product sums over d, so the k-order inside the MMA is free: lane
// (g, t) of the warp loads bytes [16t, 16t+16) of key rows g and g+8 with one
// 16-byte load each, and the query fragment uses the same d -> k assignment.
#include "common.cuh"

namespace csa2 {
namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two_bytes) {
    uint32_t r;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"((uint16_t)two_bytes));
    return r;
}

template <bool FP8>
__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
    if constexpr (FP8) {
        asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
            "{%0,%1,%2,%3};"
            : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
    } else {
        asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
            "{%0,%1,%2,%3};"
            : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
    }
}

// 16 consecutive d-values of one 64-wide row (FP8: 16 B; bf16: 32 B) ->
// 8 packed 2-element registers: reg 2s = d(4s, 4s+1), reg 2s+1 = d(4s+2, 4s+3).
template <bool FP8>
__device__ __forceinline__ void load_row16(const uint8_t *row, bool valid, uint32_t (&r)[8]) {
    if constexpr (FP8) {
        uint4 v = valid ? __ldg(reinterpret_cast<const uint4 *>(row)) : make_uint4(0, 0, 0, 0);
        uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int s = 0; s < 4; ++s) {
            r[2 * s] = e4m3x2_to_f16x2(w[s] & 0xFFFFu);
            r[2 * s + 1] = e4m3x2_to_f16x2(w[s] >> 16);
        }
    } else {
        uint4 v0 = valid ? __ldg(reinterpret_cast<const uint4 *>(row)) : make_uint4(0, 0, 0, 0);
        uint4 v1 = valid ? __ldg(reinterpret_cast<const uint4 *>(row) + 1) : make_uint4(0, 0, 0, 0);
        r[0] = v0.x; r[1] = v0.y; r[2] = v0.z; r[3] = v0.w;
        r[4] = v1.x; r[5] = v1.y; r[6] = v1.z; r[7] = v1.w;
    }
}

struct ScoreArgs {
    int mode, B, T;
    int64_t N;
    const uint8_t *q;
    const float *w;
    const uint8_t *k;
    const int32_t *kv_len;
    const int32_t *pool;
    int P;
    float *scores;
    uint32_t *err_flag;
    int64_t groups;  // key groups of 16 per task row
    int64_t tasks;
};

// One warp = one task (a group of 16 keys of one row) at a time.
//  FULL:    task = (b, group); the warp loops over the sequence's query tokens
//           two at a time (B columns 0-3 and 4-7).
//  REINDEX: task = (b*T+t, group of two pool blocks); one token.
template <bool FP8>
__global__ void __launch_bounds__(kThreads) index_score_kernel(ScoreArgs a) {
    constexpr int ES = FP8 ? 1 : 2;      // element size
    pdl_wait();
    pdl_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int g = lane >> 2, t4 = lane & 3;
    const int64_t warp = ((int64_t)blockIdx.x * kThreads + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * kThreads) >> 5;
    const float NEG_INF = __int_as_float(0xff800000);
    const int64_t nblocks_n = (a.N + 7) / 8;

    for (int64_t task = warp; task < a.tasks; task += nwarps) {
        const int64_t row = task / a.groups;      // b (FULL) or b*T+t (REINDEX)
        const int64_t grp = task - row * a.groups;
        const int64_t b = (a.mode == CSA2_MODE_FULL) ? row : row / a.T;

        // ---- the 16 keys of this group: rows g and g+8
        int64_t j0, j1;
        bool v0, v1;
        if (a.mode == CSA2_MODE_FULL) {
            j0 = grp * 16 + g;
            j1 = j0 + 8;
            // visible to at least one token of the sequence?
            v0 = j0 < a.N;
            v1 = j1 < a.N;
        } else {
            const int64_t p0 = grp * 2, p1 = p0 + 1;
            int64_t blk0 = a.pool[row * a.P + p0];
            int64_t blk1 = (p1 < a.P) ? (int64_t)a.pool[row * a.P + p1] : -1;
            if (blk0 < -1 || blk0 >= nblocks_n) { if (t4 == 0 && g == 0) flag_error(a.err_flag, CSA2_FLAG_BAD_POOL); blk0 = -1; }
            if (blk1 < -1 || blk1 >= nblocks_n) { if (t4 == 0 && g == 0) flag_error(a.err_flag, CSA2_FLAG_BAD_POOL); blk1 = -1; }
            int64_t len = a.kv_len[row];
            len = len < a.N ? len : a.N;
            j0 = blk0 * 8 + g;
            j1 = blk1 * 8 + g;
            v0 = blk0 >= 0 && j0 < len;
            v1 = blk1 >= 0 && j1 < len;
        }
        // Decode fast path: a FULL group beyond every token's kv_len is all -inf.
        if (a.mode == CSA2_MODE_FULL && a.T == 1) {
            int64_t len = a.kv_len[row];
            if (grp * 16 >= len) {
                if (lane < 16) {
                    int64_t j = grp * 16 + lane;
                    if (j < a.N) a.scores[row * a.N + j] = NEG_INF;
                }
                continue;
            }
        }
        uint32_t ka[8], kb[8];
        load_row16<FP8>(a.k + ((b * a.N + (v0 ? j0 : 0)) * 64 + 16 * t4) * ES, v0, ka);
        load_row16<FP8>(a.k + ((b * a.N + (v1 ? j1 : 0)) * 64 + 16 * t4) * ES, v1, kb);

        const int ntok = (a.mode == CSA2_MODE_FULL) ? a.T : 1;
        for (int tp = 0; tp < ntok; tp += 2) {
            // B fragment: column g = (token tp + g/4, head g%4)
            const int tok_b = tp + (g >> 2);
            const bool tb_ok = tok_b < ntok;
            const int64_t qrow = (a.mode == CSA2_MODE_FULL) ? (b * a.T + tok_b) : row;
            uint32_t qf[8];
            load_row16<FP8>(a.q + ((qrow * 4 + (g & 3)) * 64 + 16 * t4) * ES, tb_ok, qf);
            float c[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int s = 0; s < 4; ++s) {
                uint32_t af[4] = {ka[2 * s], kb[2 * s], ka[2 * s + 1], kb[2 * s + 1]};
                uint32_t bf[2] = {qf[2 * s], qf[2 * s + 1]};
                mma16816<FP8>(c, af, bf);
            }
            // Epilogue: lane holds columns 2*t4, 2*t4+1 = token tp + t4/2, heads
            // (2*t4)%4 and +1, for key rows g (c0,c1) and g+8 (c2,c3).
            const int tok_c = tp + (t4 >> 1);
            const int h0 = (2 * t4) & 3;
            const bool tc_ok = tok_c < ntok;
            const int64_t crow = (a.mode == CSA2_MODE_FULL) ? (b * a.T + tok_c) : row;
            float w0 = 0.f, w1 = 0.f;
            if (tc_ok) {
                w0 = a.w[crow * 4 + h0];
                w1 = a.w[crow * 4 + h0 + 1];
            }
            float s0 = w0 * fmaxf(c[0], 0.f) + w1 * fmaxf(c[1], 0.f);
            float s1 = w0 * fmaxf(c[2], 0.f) + w1 * fmaxf(c[3], 0.f);
            s0 += __shfl_xor_sync(0xFFFFFFFFu, s0, 1);
            s1 += __shfl_xor_sync(0xFFFFFFFFu, s1, 1);
            if ((t4 & 1) == 0 && tc_ok) {
                if (a.mode == CSA2_MODE_FULL) {
                    int64_t len = a.kv_len[crow];
                    len = len < a.N ? len : a.N;
                    float* out = a.scores + crow * a.N;
                    if (j0 < a.N) out[j0] = (j0 < len) ? s0 : NEG_INF;
                    if (j1 < a.N) out[j1] = (j1 < len) ? s1 : NEG_INF;
                } else {
                    const int64_t M = (int64_t)a.P * 8;
                    const int64_t l0 = grp * 16 + g, l1 = l0 + 8;
                    float *out = a.scores + row * M;
                    if (l0 < M) out[l0] = v0 ? s0 : NEG_INF;
                    if (l1 < M) out[l1] = v1 ? s1 : NEG_INF;
                }
            }
        }
    }
}

// Decode-shaped scoring (Full with one query token per sequence, or Reindex):
// one warp takes a chunk of CH consecutive 16-key groups of one row and
// issues every key load of the chunk (and, for Reindex, the chunk's pool ids
// in one lane-parallel load) before any arithmetic, so each warp keeps
// CH x 1 KB of keys in flight.
template <bool FP8>
__global__ void __launch_bounds__(kThreads, 2) index_score_decode_kernel(ScoreArgs a) {
    pdl_wait();
    pdl_launch_dependents();
    constexpr int ES = FP8 ? 1 : 2;
    constexpr int NV = FP8 ? 1 : 2;          // 16-byte loads per 16 d-values
    constexpr int CH = FP8 ? 8 : 4;          // groups per warp chunk
    const int lane = threadIdx.x & 31;
    const int g = lane >> 2, t4 = lane & 3;
    const int64_t warp = ((int64_t)blockIdx.x * kThreads + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * kThreads) >> 5;
    const float NEG_INF = __int_as_float(0xff800000);
    const int64_t nblocks_n = (a.N + 7) / 8;
    const bool full = a.mode == CSA2_MODE_FULL;
    const int64_t rows = full ? (int64_t)a.B : (int64_t)a.B * a.T;
    const int64_t cpr = (a.groups + CH - 1) / CH;   // chunks per row
    const int64_t M = full ? a.N : (int64_t)a.P * 8;

    for (int64_t ch = warp; ch < rows * cpr; ch += nwarps) {
        const int64_t row = ch / cpr;
        const int64_t g0 = (ch - row * cpr) * CH;
        const int64_t b = full ? row : row / a.T;
        int64_t len = a.kv_len[row];
        len = len < a.N ? len : a.N;
        int32_t myblk = -1;
        if (!full && lane < 2 * CH) {
            const int64_t pidx = 2 * g0 + lane;
            if (pidx < a.P) {
                int64_t blk = a.pool[row * a.P + pidx];
                if (blk < -1 || blk >= nblocks_n) {
                    flag_error(a.err_flag, CSA2_FLAG_BAD_POOL);
                    blk = -1;
                }
                myblk = (int32_t)blk;
            }
        }
        uint4 raw[CH][2][NV];
        bool v[CH][2];
#pragma unroll
        for (int c = 0; c < CH; ++c) {
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                int64_t j;
                if (full) {
                    j = (g0 + c) * 16 + g + 8 * r;
                } else {
                    const int32_t blk = __shfl_sync(0xFFFFFFFFu, myblk, 2 * c + r);
                    j = (blk >= 0) ? (int64_t)blk * 8 + g : -1;
                }
                v[c][r] = (g0 + c) < a.groups && j >= 0 && j < len;
                const uint4 *src = reinterpret_cast<const uint4 *>(a.k + ((b * a.N + (v[c][r] ? j : 0)) * 64 + 16 * t4) * ES);
#pragma unroll
                for (int u = 0; u < NV; ++u) raw[c][r][u] = v[c][r] ? __ldg(src + u) : make_uint4(0, 0, 0, 0);
            }
        }
        // FP8: the raw 16 bytes of d-values 16 t4 .. 16 t4 + 15 (head g < 4; columns 4-7 zero)
        // feed two k32 MMAs directly, the same d-permutation on keys and query;
        // bf16: converted fragments for four k16 MMAs
        uint32_t qf[8];
        uint4 q8 = make_uint4(0, 0, 0, 0);
        if constexpr (FP8) {
            if ((g >> 2) == 0) q8 = __ldg(reinterpret_cast<const uint4 *>(a.q + (row * 4 + g) * 64 + 16 * t4));
        } else {
            load_row16<FP8>(a.q + ((row * 4 + (g & 3)) * 64 + 16 * t4) * ES, (g >> 2) == 0, qf);
        }
        const float w0 = (t4 < 2) ? a.w[row * 4 + 2 * t4] : 0.f;
        const float w1 = (t4 < 2) ? a.w[row * 4 + 2 * t4 + 1] : 0.f;
        float *out = a.scores + row * M;
#pragma unroll
        for (int c = 0; c < CH; ++c) {
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
            if constexpr (FP8) {
                const uint4 ra = raw[c][0][0], rb = raw[c][1][0];   // keys g and g + 8
                mma_e4m3_16832(acc, ra.x, rb.x, ra.y, rb.y, q8.x, q8.y);
                mma_e4m3_16832(acc, ra.z, rb.z, ra.w, rb.w, q8.z, q8.w);
            } else {
                uint32_t ka[8], kb[8];
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    uint32_t *d = r ? kb : ka;
                    d[0] = raw[c][r][0].x; d[1] = raw[c][r][0].y; d[2] = raw[c][r][0].z; d[3] = raw[c][r][0].w;
                    d[4] = raw[c][r][NV - 1].x; d[5] = raw[c][r][NV - 1].y; d[6] = raw[c][r][NV - 1].z; d[7] = raw[c][r][NV - 1].w;
                }
#pragma unroll
                for (int s2 = 0; s2 < 4; ++s2) {
                    const uint32_t af[4] = {ka[2 * s2], kb[2 * s2], ka[2 * s2 + 1], kb[2 * s2 + 1]};
                    const uint32_t bf[2] = {qf[2 * s2], qf[2 * s2 + 1]};
                    mma16816<FP8>(acc, af, bf);
                }
            }
            float s0 = w0 * fmaxf(acc[0], 0.f) + w1 * fmaxf(acc[1], 0.f);
            float s1 = w0 * fmaxf(acc[2], 0.f) + w1 * fmaxf(acc[3], 0.f);
            s0 += __shfl_xor_sync(0xFFFFFFFFu, s0, 1);
            s1 += __shfl_xor_sync(0xFFFFFFFFu, s1, 1);
            if (t4 == 0) {
                const int64_t l0 = (g0 + c) * 16 + g, l1 = l0 + 8;
                if (l0 < M) out[l0] = v[c][0] ? s0 : NEG_INF;
                if (l1 < M) out[l1] = v[c][1] ? s1 : NEG_INF;
            }
        }
    }
}

}  // namespace
}  // namespace csa2

using namespace csa2;

extern "C" csa2_status csa2_index_score(csa2_mode mode, int B, int T, int64_t N, const void *q_idx,
                                        csa2_dtype q_dt, const float *w, const void *k_idx,
                                        csa2_dtype k_dt, const int32_t *kv_len,
                                        const int32_t *pool_blocks, int P, float *scores,
                                        uint32_t *err_flag, csa2_stream_t stream) {
    clear_error();
    CSA2_REQUIRE(mode == CSA2_MODE_FULL || mode == CSA2_MODE_REINDEX || mode == CSA2_MODE_REUSE,
                 "index_score: bad mode %d", (int)mode);
    if (mode == CSA2_MODE_REUSE) return CSA2_OK;
    CSA2_REQUIRE(B >= 0 && T >= 0 && N >= 0, "index_score: negative shape");
    CSA2_REQUIRE(q_dt == k_dt, "index_score: q_dt must equal k_dt");
    CSA2_REQUIRE(q_dt == CSA2_FP8_E4M3 || q_dt == CSA2_BF16, "index_score: dtype must be FP8_E4M3 or BF16");
    if (mode == CSA2_MODE_FULL) {
        CSA2_REQUIRE(pool_blocks == nullptr, "index_score: FULL takes no pool_blocks");
    } else {
        CSA2_REQUIRE(pool_blocks != nullptr, "index_score: REINDEX needs pool_blocks");
        CSA2_REQUIRE(P >= 1 && P <= CSA2_MAX_POOL, "index_score: P=%d not in [1,2048]", P);
    }
    if ((int64_t)B * T == 0 || N == 0) return CSA2_OK;
    CSA2_REQUIRE(q_idx && w && k_idx && kv_len && scores, "index_score: null pointer");
    CSA2_REQUIRE(aligned(q_idx, 16) && aligned(k_idx, 16), "index_score: q_idx/k_idx must be 16-byte aligned");
    CSA2_REQUIRE(aligned(w, 4) && aligned(scores, 4) && aligned(kv_len, 4), "index_score: misaligned w/scores/kv_len");

    ScoreArgs a;
    a.mode = (int)mode; a.B = B; a.T = T; a.N = N;
    a.q = (const uint8_t *)q_idx; a.w = w; a.k = (const uint8_t *)k_idx;
    a.kv_len = kv_len; a.pool = pool_blocks; a.P = P; a.scores = scores; a.err_flag = err_flag;
    if (mode == CSA2_MODE_FULL) {
        a.groups = (N + 15) / 16;
        a.tasks = (int64_t)B * a.groups;
    } else {
        a.groups = ((int64_t)P * 8 + 15) / 16;
        a.tasks = (int64_t)B * T * a.groups;
    }
    int64_t want = (a.tasks + (kThreads / 32) - 1) / (kThreads / 32);
    int64_t cap = (int64_t)num_sms() * 8;
    int blocks = (int)(want < cap ? want : cap);
    if (mode == CSA2_MODE_FULL && index_score_prefill_tc_supported(T, q_dt))
        return launch_index_score_prefill_tc(B, T, N, q_idx, w, k_idx, kv_len, scores, err_flag, stream_of(stream));
    const bool decode = (mode == CSA2_MODE_REINDEX) || T == 1;
    if (decode) {
        const int ch = (q_dt == CSA2_FP8_E4M3) ? 8 : 4;
        const int64_t rows = (mode == CSA2_MODE_FULL) ? (int64_t)B : (int64_t)B * T;
        const int64_t chunks = rows * ((a.groups + ch - 1) / ch);
        int64_t want_d = (chunks + (kThreads / 32) - 1) / (kThreads / 32);
        int64_t cap_d = (int64_t)num_sms() * 2;
        int blocks_d = (int)(want_d < cap_d ? want_d : cap_d);
        if (q_dt == CSA2_FP8_E4M3)
            CSA2_CUDA_CALL(launch_pdl(index_score_decode_kernel<true>, dim3(blocks_d), dim3(kThreads), 0,
                                      stream_of(stream), a),
                           "index_score_decode_kernel launch");
        else
            CSA2_CUDA_CALL(launch_pdl(index_score_decode_kernel<false>, dim3(blocks_d), dim3(kThreads), 0,
                                      stream_of(stream), a),
                           "index_score_decode_kernel launch");
    } else if (q_dt == CSA2_FP8_E4M3) {
        CSA2_CUDA_CALL(launch_pdl(index_score_kernel<true>, dim3(blocks), dim3(kThreads), 0, stream_of(stream), a),
                       "index_score_kernel launch");
    } else {
        CSA2_CUDA_CALL(launch_pdl(index_score_kernel<false>, dim3(blocks), dim3(kThreads), 0, stream_of(stream), a),
                       "index_score_kernel launch");
    }
    CSA2_LAUNCH_CHECK("index_score_kernel");
    return CSA2_OK;
}

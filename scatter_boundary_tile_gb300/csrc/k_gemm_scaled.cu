// Block-scaled GEMM  D = (A .* a_scale)(B .* b_scale) + acc.
//
// cuTile.jl "Operations", muladd_scaled: A (M,K) and B (K,N) in a
// low-precision float format (E4M3, E5M2 or E2M1), one scale per contiguous
// block of K / K_s elements along K (a_scale (M,K_s), b_scale (K_s,N), in
// E8M0 or E4M3), fp32 accumulator and acc.
//
// Path: the operand staging of the boundary-tile GEMM, with the scale folded
// in.  Each element is decoded from its format and multiplied by its block's
// scale in fp32, rounded to bf16 and written into the same padded K-major
// copies A' [Mp][Kp] and B'^T [Np][Kp] (zero past M, N, K) that the bf16
// GEMM stages; the tcgen05 kernel then runs unchanged and adds acc in its
// epilogue.  The scaled operand has at most 8 significant bits (a 4-bit E4M3
// significand times a power of two or times another 4-bit significand), so
// the bf16 copy is exact while it lies in bf16's normal range.
#include <cuda_bf16.h>

#include <algorithm>

#include "sbt_internal.cuh"

namespace {

constexpr int kFmtE4M3 = 0, kFmtE5M2 = 1, kFmtE8M0 = 2, kFmtE2M1 = 3;

// Value of one code, from the format definitions (OCP 8-bit floating point
// and microscaling formats).  Normal values are assembled as fp32 bit
// patterns; subnormal ones as (integer significand) * 2^-bias', both exact.
__device__ __forceinline__ float lowp_value(int fmt, uint32_t c) {
    if (fmt == kFmtE8M0) {
        if (c == 255u) return __uint_as_float(0x7FC00000u);
        return __uint_as_float(c ? c << 23 : 0x00400000u);  // 2^(c-127); c = 0 is the fp32 subnormal 2^-127
    }
    float v;
    uint32_t neg;
    if (fmt == kFmtE2M1) {
        neg = (c >> 3) & 1u;
        const uint32_t e = (c >> 1) & 3u, m = c & 1u;
        v = e ? __uint_as_float(((e + 126u) << 23) | (m << 22)) : 0.5f * (float)m;
    } else if (fmt == kFmtE4M3) {
        neg = c >> 7;
        const uint32_t e = (c >> 3) & 15u, m = c & 7u;
        if (e == 15u && m == 7u) return __uint_as_float(0x7FC00000u);
        v = e ? __uint_as_float(((e + 120u) << 23) | (m << 20)) : (float)m * 0x1p-9f;
    } else {  // E5M2
        neg = c >> 7;
        const uint32_t e = (c >> 2) & 31u, m = c & 3u;
        if (e == 31u) v = m ? __uint_as_float(0x7FC00000u) : __uint_as_float(0x7F800000u);
        else v = e ? __uint_as_float(((e + 112u) << 23) | (m << 21)) : (float)m * 0x1p-16f;
    }
    return neg ? -v : v;
}

// Code of element i (= row * ld + col) of a row-major operand; E2M1 packs two
// per byte, the even element in the low nibble.
__device__ __forceinline__ uint32_t lowp_code(int fmt, const uint8_t* __restrict__ p, int64_t i) {
    if (fmt == kFmtE2M1) return (uint32_t)(__ldg(p + (i >> 1)) >> (4 * (int)(i & 1))) & 15u;
    return __ldg(p + i);
}

__device__ __forceinline__ uint32_t bf16_bits(float x) {
    return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(x));
}

// A' [Mp][Kp] <- A .* a_scale, zero past M or K.  One 16-byte vector (8 k) of A' per task.
__global__ void __launch_bounds__(256) k_stage_scaled_a(int fmt, int sfmt, const uint8_t* __restrict__ A, int64_t lda,
                                                        const uint8_t* __restrict__ SA, int64_t ld_sa, int block,
                                                        int M, int K, uint16_t* __restrict__ Ap, int Kp,
                                                        int64_t total_vecs) {
    const int kv = Kp / 8;
    for (int64_t v = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; v < total_vecs;
         v += (int64_t)gridDim.x * blockDim.x) {
        const int64_t m = v / kv;
        const int k0 = (int)(v - m * kv) * 8;
        uint32_t w[4] = {0, 0, 0, 0};
        if (m < M && k0 < K) {
            int kb = k0 / block, kr = k0 - kb * block;
            float s = lowp_value(sfmt, __ldg(SA + m * ld_sa + kb));
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int k = k0 + e;
                if (k < K) {
                    if (kr == block) {  // next scale block
                        ++kb;
                        kr = 0;
                        s = lowp_value(sfmt, __ldg(SA + m * ld_sa + kb));
                    }
                    w[e >> 1] |= bf16_bits(lowp_value(fmt, lowp_code(fmt, A, m * lda + k)) * s) << (16 * (e & 1));
                    ++kr;
                }
            }
        }
        sbt_st_v4(Ap + m * Kp + k0, make_uint4(w[0], w[1], w[2], w[3]));
    }
}

// B'^T [Np][Kp] <- transpose of B .* b_scale, zero past K or N.  64 x 64 tiles
// through shared memory: reads along n, 16-byte writes along k.
__global__ void __launch_bounds__(256) k_stage_scaled_bt(int fmt, int sfmt, const uint8_t* __restrict__ B, int64_t ldb,
                                                         const uint8_t* __restrict__ SB, int64_t ld_sb, int block,
                                                         int K, int N, uint16_t* __restrict__ Bp, int Kp) {
    __shared__ uint16_t t[64][66];
    const int k0 = blockIdx.x * 64, n0 = blockIdx.y * 64;
#pragma unroll 4
    for (int i = 0; i < 16; ++i) {
        const int idx = i * 256 + threadIdx.x;
        const int kk = idx >> 6, nn = idx & 63;
        const int k = k0 + kk, n = n0 + nn;
        uint32_t x = 0;
        if (k < K && n < N) {
            const float s = lowp_value(sfmt, __ldg(SB + (int64_t)(k / block) * ld_sb + n));
            x = bf16_bits(lowp_value(fmt, lowp_code(fmt, B, (int64_t)k * ldb + n)) * s);
        }
        t[kk][nn] = (uint16_t)x;
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int task = i * 256 + threadIdx.x;  // 64 rows of B'^T x 8 vectors
        const int nn = task >> 3, kv = task & 7;
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e)
            w[e] = (uint32_t)t[kv * 8 + 2 * e][nn] | ((uint32_t)t[kv * 8 + 2 * e + 1][nn] << 16);
        sbt_st_v4(Bp + (int64_t)(n0 + nn) * Kp + k0 + kv * 8, make_uint4(w[0], w[1], w[2], w[3]));
    }
}

}  // namespace

sbt_status sbt_launch_gemm_block_scaled(sbt_context* ctx, int a_fmt, const void* A, int64_t lda, int b_fmt,
                                        const void* B, int64_t ldb, int s_fmt, const void* SA, int64_t ld_sa,
                                        const void* SB, int64_t ld_sb, int64_t Ks, const float* acc, int64_t ld_acc,
                                        float* D, int64_t ldd, int64_t M, int64_t N, int64_t K, void* workspace,
                                        cudaStream_t stream) {
    if (M > INT32_MAX / 2 || N > INT32_MAX / 2 || K > INT32_MAX / 2)
        return sbt_fail(SBT_ERR_INVALID_ARG, "gemm_block_scaled: extents must be below 2^30");
    if (K == 0) return sbt_launch_gemm_zero_k(ctx, D, ldd, true, acc, ld_acc, M, N, stream);
    const sbt_gemm_layout d = sbt_gemm_layout_of(M, N, K);
    if (d.Np / 64 > 65535) return sbt_fail(SBT_ERR_INVALID_ARG, "gemm_block_scaled: N too large for the staging grid");
    const int block = (int)(K / Ks);
    uint16_t* Ap = (uint16_t*)workspace;
    uint16_t* Bp = (uint16_t*)((char*)workspace + d.a_bytes);
    const int64_t vecs = d.Mp * (d.Kp / 8);
    const int grid = (int)std::min<int64_t>(sbt_cdiv(vecs, 256), (int64_t)ctx->sm_count * 8);
    k_stage_scaled_a<<<grid, 256, 0, stream>>>(a_fmt, s_fmt, (const uint8_t*)A, lda, (const uint8_t*)SA, ld_sa, block,
                                               (int)M, (int)K, Ap, (int)d.Kp, vecs);
    sbt_status st = sbt_after_launch(ctx, "gemm_block_scaled (stage A)");
    if (st) return st;
    dim3 g2((unsigned)(d.Kp / 64), (unsigned)(d.Np / 64));
    k_stage_scaled_bt<<<g2, 256, 0, stream>>>(b_fmt, s_fmt, (const uint8_t*)B, ldb, (const uint8_t*)SB, ld_sb, block,
                                              (int)K, (int)N, Bp, (int)d.Kp);
    if ((st = sbt_after_launch(ctx, "gemm_block_scaled (stage B)"))) return st;
    return sbt_launch_gemm_main(ctx, Ap, Bp, d, D, ldd, true, acc, ld_acc, M, N, K, stream);
}

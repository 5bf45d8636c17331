// Block-scaled GEMM  D = (A .* a_scale)(B .* b_scale) + acc.
//
// cuTile.jl "Operations", muladd_scaled: A (M,K) and B (K,N) in a
// low-precision float format (E4M3, E5M2 or E2M1), one scale per contiguous
// block of K / K_s elements along K (a_scale (M,K_s), b_scale (K_s,N), in
// E8M0 or E4M3), fp32 accumulator and acc.
//
// E4M3 / E5M2 / E2M1 operands with E8M0 scales over blocks of 32, and E2M1 x
// E2M1 with E4M3 scales over blocks of 16, run on the tensor cores' block
// scaling (k_gemm_mx.cu).  Every other combination takes this path: the operand staging of the boundary-tile GEMM, with the scale folded
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
// and microscaling formats).  The exponent and mantissa fields are placed at
// the top of an fp32 bit pattern and the result is rescaled by the power of
// two that turns the fp32 bias into the format's bias: the fields of a normal
// code become a normal fp32 number and those of a subnormal code an fp32
// subnormal with the same significand, so one exact multiply covers both.
template <int FMT>
__device__ __forceinline__ float lowp_value(uint32_t c) {
    if constexpr (FMT == kFmtE8M0) {
        return __uint_as_float(c == 255u ? 0x7FC00000u : c ? c << 23 : 0x00400000u);  // 2^(c-127)
    } else if constexpr (FMT == kFmtE2M1) {
        const float v = __uint_as_float((c & 7u) << 22) * 0x1p126f;  // bias 1
        return __uint_as_float(__float_as_uint(v) | ((c & 8u) << 28));
    } else if constexpr (FMT == kFmtE4M3) {
        const float v = __uint_as_float((c & 0x7Fu) << 20) * 0x1p120f;  // bias 7
        const uint32_t bits = (c & 0x7Fu) == 0x7Fu ? 0x7FC00000u : __float_as_uint(v);
        return __uint_as_float(bits | ((c & 0x80u) << 24));
    } else {  // E5M2
        const float v = __uint_as_float((c & 0x7Fu) << 21) * 0x1p112f;  // bias 15
        uint32_t bits = __float_as_uint(v);
        if ((c & 0x7Cu) == 0x7Cu) bits = (c & 3u) ? 0x7FC00000u : 0x7F800000u;
        return __uint_as_float(bits | ((c & 0x80u) << 24));
    }
}

// Code of element i (= row * ld + col) of a row-major operand; E2M1 packs two
// per byte, the even element in the low nibble.
template <int FMT>
__device__ __forceinline__ uint32_t lowp_code(const uint8_t* __restrict__ p, int64_t i) {
    if constexpr (FMT == kFmtE2M1) return (uint32_t)(__ldg(p + (i >> 1)) >> (4 * (int)(i & 1))) & 15u;
    else return __ldg(p + i);
}

// Four bytes p..p+3 (all inside the array) through aligned 4-byte loads, as
// sbt_load8_any does with eight.
__device__ __forceinline__ uint32_t load4_any(const uint8_t* p) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(p);
    const int sh = (int)(a & 3u) * 8;
    const uint32_t* w = reinterpret_cast<const uint32_t*>(a & ~(uintptr_t)3);
    const uint32_t lo = __ldg(w);
    if (sh == 0) return lo;
    return (lo >> sh) | (__ldg(w + 1) << (32 - sh));
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&v);
}

// A' [Mp][Kp] <- A .* a_scale, zero past M or K.  One 16-byte vector (8 k) of A' per task.
template <int FMT, int SFMT>
__global__ void __launch_bounds__(256) k_stage_scaled_a(const uint8_t* __restrict__ A, int64_t lda,
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
            float x[8];
            if (k0 + 8 <= K) {  // whole vector inside the row: word loads
                if constexpr (FMT == kFmtE2M1) {
                    const uint32_t c = load4_any(A + ((m * lda + k0) >> 1));
#pragma unroll
                    for (int e = 0; e < 8; ++e) x[e] = lowp_value<FMT>((c >> (4 * e)) & 15u);
                } else {
                    const uint64_t c = sbt_load8_any(A + m * lda + k0);
#pragma unroll
                    for (int e = 0; e < 8; ++e) x[e] = lowp_value<FMT>((uint32_t)(c >> (8 * e)) & 255u);
                }
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) x[e] = k0 + e < K ? lowp_value<FMT>(lowp_code<FMT>(A, m * lda + k0 + e)) : 0.f;
            }
            int kb = k0 / block, kr = k0 - kb * block;
            float s = lowp_value<SFMT>(__ldg(SA + m * ld_sa + kb));
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                if (kr == block) {  // next scale block (only read while k < K)
                    ++kb;
                    kr = 0;
                    if (k0 + e < K) s = lowp_value<SFMT>(__ldg(SA + m * ld_sa + kb));
                }
                x[e] *= s;
                ++kr;
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) w[e] = pack_bf16x2(x[2 * e], x[2 * e + 1]);
        }
        sbt_st_v4(Ap + m * Kp + k0, make_uint4(w[0], w[1], w[2], w[3]));
    }
}

// B'^T [Np][Kp] <- transpose of B .* b_scale, zero past K or N.  64 x 64 tiles
// through shared memory: reads along n, 16-byte writes along k.
template <int FMT, int SFMT>
__global__ void __launch_bounds__(256) k_stage_scaled_bt(const uint8_t* __restrict__ B, int64_t ldb,
                                                         const uint8_t* __restrict__ SB, int64_t ld_sb, int block,
                                                         int K, int N, uint16_t* __restrict__ Bp, int Kp) {
    __shared__ float t[64][65];
    __shared__ int s_kb[64];
    const int k0 = blockIdx.x * 64, n0 = blockIdx.y * 64;
    if (threadIdx.x < 64) s_kb[threadIdx.x] = (k0 + (int)threadIdx.x) / block;
    __syncthreads();
#pragma unroll 4
    for (int i = 0; i < 16; ++i) {
        const int idx = i * 256 + threadIdx.x;
        const int kk = idx >> 6, nn = idx & 63;
        const int k = k0 + kk, n = n0 + nn;
        float x = 0.f;
        if (k < K && n < N)
            x = lowp_value<FMT>(lowp_code<FMT>(B, (int64_t)k * ldb + n)) *
                lowp_value<SFMT>(__ldg(SB + (int64_t)s_kb[kk] * ld_sb + n));
        t[kk][nn] = x;
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int task = i * 256 + threadIdx.x;  // 64 rows of B'^T x 8 vectors
        const int nn = task >> 3, kv = task & 7;
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) w[e] = pack_bf16x2(t[kv * 8 + 2 * e][nn], t[kv * 8 + 2 * e + 1][nn]);
        sbt_st_v4(Bp + (int64_t)(n0 + nn) * Kp + k0 + kv * 8, make_uint4(w[0], w[1], w[2], w[3]));
    }
}

template <int FMT, int SFMT>
void launch_stage_a(dim3 g, cudaStream_t st, const uint8_t* A, int64_t lda, const uint8_t* SA, int64_t ld_sa,
                    int block, int M, int K, uint16_t* Ap, int Kp, int64_t vecs) {
    k_stage_scaled_a<FMT, SFMT><<<g, 256, 0, st>>>(A, lda, SA, ld_sa, block, M, K, Ap, Kp, vecs);
}

template <int FMT, int SFMT>
void launch_stage_bt(dim3 g, cudaStream_t st, const uint8_t* B, int64_t ldb, const uint8_t* SB, int64_t ld_sb,
                     int block, int K, int N, uint16_t* Bp, int Kp) {
    k_stage_scaled_bt<FMT, SFMT><<<g, 256, 0, st>>>(B, ldb, SB, ld_sb, block, K, N, Bp, Kp);
}

// One instantiation per (operand format, scale format) pair.
template <template <int, int> class F, typename... Args>
void dispatch_formats(int fmt, int sfmt, Args... args) {
    if (sfmt == kFmtE8M0) {
        if (fmt == kFmtE4M3) F<kFmtE4M3, kFmtE8M0>::run(args...);
        else if (fmt == kFmtE5M2) F<kFmtE5M2, kFmtE8M0>::run(args...);
        else F<kFmtE2M1, kFmtE8M0>::run(args...);
    } else {
        if (fmt == kFmtE4M3) F<kFmtE4M3, kFmtE4M3>::run(args...);
        else if (fmt == kFmtE5M2) F<kFmtE5M2, kFmtE4M3>::run(args...);
        else F<kFmtE2M1, kFmtE4M3>::run(args...);
    }
}

template <int FMT, int SFMT>
struct StageA {
    template <typename... Args>
    static void run(Args... args) { launch_stage_a<FMT, SFMT>(args...); }
};

template <int FMT, int SFMT>
struct StageBt {
    template <typename... Args>
    static void run(Args... args) { launch_stage_bt<FMT, SFMT>(args...); }
};

}  // namespace

sbt_status sbt_launch_gemm_block_scaled(sbt_context* ctx, int a_fmt, const void* A, int64_t lda, int b_fmt,
                                        const void* B, int64_t ldb, int s_fmt, const void* SA, int64_t ld_sa,
                                        const void* SB, int64_t ld_sb, int64_t Ks, const float* acc, int64_t ld_acc,
                                        float* D, int64_t ldd, int64_t M, int64_t N, int64_t K, void* workspace,
                                        cudaStream_t stream) {
    if (M > INT32_MAX / 2 || N > INT32_MAX / 2 || K > INT32_MAX / 2)
        return sbt_fail(SBT_ERR_INVALID_ARG, "gemm_block_scaled: extents must be below 2^30");
    if (K == 0) return sbt_launch_gemm_zero_k(ctx, D, ldd, true, acc, ld_acc, M, N, stream);
    // the tensor cores' block scaling: E8M0 scales over blocks of 32 with any of the operand
    // formats, and E4M3 scales over blocks of 16 with E2M1 x E2M1
    const bool mx = (s_fmt == kFmtE8M0 && K == 32 * Ks) ||
                    (s_fmt == kFmtE4M3 && K == 16 * Ks && a_fmt == kFmtE2M1 && b_fmt == kFmtE2M1);
    if (mx && (ctx->path == SBT_PATH_AUTO || ctx->path == SBT_PATH_TMA))
        return sbt_launch_gemm_mx(ctx, a_fmt, A, lda, b_fmt, B, ldb, s_fmt, SA, ld_sa, SB, ld_sb, acc, ld_acc, D, ldd,
                                  M, N, K, workspace, stream);
    const sbt_gemm_layout d = sbt_gemm_layout_of(M, N, K);
    if (d.Np / 64 > 65535) return sbt_fail(SBT_ERR_INVALID_ARG, "gemm_block_scaled: N too large for the staging grid");
    const int block = (int)(K / Ks);
    uint16_t* Ap = (uint16_t*)workspace;
    uint16_t* Bp = (uint16_t*)((char*)workspace + d.a_bytes);
    const int64_t vecs = d.Mp * (d.Kp / 8);
    const int grid = (int)std::min<int64_t>(sbt_cdiv(vecs, 256), (int64_t)ctx->sm_count * 8);
    dispatch_formats<StageA>(a_fmt, s_fmt, dim3((unsigned)grid), stream, (const uint8_t*)A, lda, (const uint8_t*)SA,
                             ld_sa, block, (int)M, (int)K, Ap, (int)d.Kp, vecs);
    sbt_status st = sbt_after_launch(ctx, "gemm_block_scaled (stage A)");
    if (st) return st;
    dim3 g2((unsigned)(d.Kp / 64), (unsigned)(d.Np / 64));
    dispatch_formats<StageBt>(b_fmt, s_fmt, g2, stream, (const uint8_t*)B, ldb, (const uint8_t*)SB, ld_sb, block,
                              (int)K, (int)N, Bp, (int)d.Kp);
    if ((st = sbt_after_launch(ctx, "gemm_block_scaled (stage B)"))) return st;
    return sbt_launch_gemm_main(ctx, Ap, Bp, d, D, ldd, true, acc, ld_acc, M, N, K, stream);
}

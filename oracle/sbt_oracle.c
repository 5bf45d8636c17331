/*
 * CPU oracle of bounds-checked tile movement and the boundary-tile GEMM.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, obviously correct
 * statement of what the CUDA path computes; only the test suite, the smoke
 * check and the benchmark's CPU baseline may load it.  It shares no code,
 * header, table or helper with the CUDA library and includes only the C
 * standard library.  Single-threaded, one element at a time.
 *
 * Conventions (each function names the passage it follows):
 *   - coordinates are zero-based and signed (Tylo.jl "Boundary tiles": the
 *     origin and all coordinates are zero-based; negative crop origins are
 *     supported);
 *   - arrays are row-major with explicit strides counted in elements;
 *   - movement copies raw element bits (es = element size in bytes, 2 or 4);
 *     no floating-point operation touches moved data, so NaN payloads and -0.0
 *     survive bit for bit;
 *   - `pad` points at one element's raw bits.
 *
 * Parity pins: every function is pinned by tests that do not call it again
 * (worked examples printed on the pages, numpy library special cases,
 * invariants); see tests/test_oracle_pins.py.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

static void put(void* base, int64_t off, int es, const void* v) { memcpy((char*)base + off * es, v, (size_t)es); }
static const void* at(const void* base, int64_t off, int es) { return (const char*)base + off * es; }

/* Padded tile load over a grid of tiles.
 * cuTile.jl "Memory", section "Bounds checking": a load that extends past the
 * array is padded; cuTile.jl "Memory", section "Tile windows": tile origins
 * advance by a per-dimension step.  Tile (ti, tj) starts at
 * (origin_r + ti*step_r, origin_c + tj*step_c); element (i, j) of it reads
 * src[r*stride_r + c*stride_c] when 0 <= r < rows and 0 <= c < cols, else pad.
 * dst holds the tiles contiguously as [grid_r][grid_c][tile_r][tile_c]. */
void oracle_tile_load_padded(int es, const void* src, int64_t rows, int64_t cols, int64_t stride_r,
                             int64_t stride_c, int64_t origin_r, int64_t origin_c, int64_t step_r, int64_t step_c,
                             int32_t grid_r, int32_t grid_c, int32_t tile_r, int32_t tile_c, void* dst,
                             const void* pad) {
    for (int32_t ti = 0; ti < grid_r; ++ti)
        for (int32_t tj = 0; tj < grid_c; ++tj)
            for (int32_t i = 0; i < tile_r; ++i)
                for (int32_t j = 0; j < tile_c; ++j) {
                    int64_t r = origin_r + (int64_t)ti * step_r + i;
                    int64_t c = origin_c + (int64_t)tj * step_c + j;
                    int64_t o = (((int64_t)ti * grid_c + tj) * tile_r + i) * tile_c + j;
                    if (r >= 0 && r < rows && c >= 0 && c < cols)
                        put(dst, o, es, at(src, r * stride_r + c * stride_c, es));
                    else
                        put(dst, o, es, pad);
                }
}

/* Clipped tile store, the inverse of the padded load.
 * cuTile.jl "Memory", section "Bounds checking": a store is clipped to the
 * array; Tylo.jl "Boundary tiles", section "Accumulator stores and GEMM": the
 * bounded store suppresses invalid coordinates and leaves the memory outside
 * the array unchanged.  Elements with an out-of-range coordinate are not
 * written; windows that overlap have no defined winner. */
void oracle_tile_store_clipped(int es, const void* src_tiles, int32_t grid_r, int32_t grid_c, int32_t tile_r,
                               int32_t tile_c, void* dst, int64_t rows, int64_t cols, int64_t stride_r,
                               int64_t stride_c, int64_t origin_r, int64_t origin_c, int64_t step_r, int64_t step_c) {
    for (int32_t ti = 0; ti < grid_r; ++ti)
        for (int32_t tj = 0; tj < grid_c; ++tj)
            for (int32_t i = 0; i < tile_r; ++i)
                for (int32_t j = 0; j < tile_c; ++j) {
                    int64_t r = origin_r + (int64_t)ti * step_r + i;
                    int64_t c = origin_c + (int64_t)tj * step_c + j;
                    int64_t o = (((int64_t)ti * grid_c + tj) * tile_r + i) * tile_c + j;
                    if (r >= 0 && r < rows && c >= 0 && c < cols)
                        put(dst, r * stride_r + c * stride_c, es, at(src_tiles, o, es));
                }
}

/* Row gather through an int32 index tile.
 * warp.tile_load_indexed, description: element (k, j) reads row
 * row_offset + idx[k] and column col_offset + j; every coordinate is checked
 * against both array bounds and an element outside reads the padding value, so
 * -1 serves as a sentinel.  The row offset is added to the index before the
 * check, in 64-bit.  cuTile.jl "Memory": gather takes a per-element mask and a
 * custom padding value for masked-out elements; mask == NULL means all true,
 * otherwise mask[k*ld_mask + j] != 0 is true.
 * Output element (k, j) is out[k*ld_out + j], k < n_idx, j < tile_c. */
void oracle_gather_rows(int es, const void* src, int64_t rows, int64_t cols, int64_t ld_src, const int32_t* idx,
                        int64_t n_idx, int64_t row_offset, int64_t col_offset, int32_t tile_c, const uint8_t* mask,
                        int64_t ld_mask, void* out, int64_t ld_out, const void* pad) {
    for (int64_t k = 0; k < n_idx; ++k) {
        int64_t r = (int64_t)idx[k] + row_offset;
        for (int32_t j = 0; j < tile_c; ++j) {
            int64_t c = col_offset + j;
            int m = mask ? (mask[k * ld_mask + j] != 0) : 1;
            if (m && r >= 0 && r < rows && c >= 0 && c < cols)
                put(out, k * ld_out + j, es, at(src, r * ld_src + c, es));
            else
                put(out, k * ld_out + j, es, pad);
        }
    }
}

/* Column gather (gather along axis 1).
 * warp.tile_load_indexed, description, with axis = 1: element (i, k) of the
 * tile reads row row_offset + i and column col_offset + idx[k] (the offset is
 * added before the check, in 64-bit); every coordinate is checked against both
 * bounds and an element outside reads the padding value.
 * Output element (i, k) is out[i*ld_out + k], i < tile_r, k < n_idx. */
void oracle_gather_cols(int es, const void* src, int64_t rows, int64_t cols, int64_t ld_src, const int32_t* idx,
                        int64_t n_idx, int64_t row_offset, int64_t col_offset, int32_t tile_r, void* out,
                        int64_t ld_out, const void* pad) {
    for (int32_t i = 0; i < tile_r; ++i) {
        int64_t r = row_offset + i;
        for (int64_t k = 0; k < n_idx; ++k) {
            int64_t c = (int64_t)idx[k] + col_offset;
            if (r >= 0 && r < rows && c >= 0 && c < cols)
                put(out, i * ld_out + k, es, at(src, r * ld_src + c, es));
            else
                put(out, i * ld_out + k, es, pad);
        }
    }
}

/* Masked row scatter.
 * cuTile.jl "Memory": scatter writes only where the mask is true and, like
 * every memory operation there, is bounds-checked (out-of-range elements are
 * clipped).  Source element (k, j) goes to dst row row_offset + idx[k],
 * column col_offset + j.  cuTile.jl "Memory", section "Sparse views": repeated
 * indices on a store conflict and are undefined; this loop lets the last one
 * win, which is one of the allowed outcomes. */
void oracle_scatter_rows_masked(int es, void* dst, int64_t rows, int64_t cols, int64_t ld_dst, const int32_t* idx,
                                int64_t n_idx, int64_t row_offset, int64_t col_offset, const void* src,
                                int64_t ld_src, int32_t tile_c, const uint8_t* mask, int64_t ld_mask) {
    for (int64_t k = 0; k < n_idx; ++k) {
        int64_t r = (int64_t)idx[k] + row_offset;
        for (int32_t j = 0; j < tile_c; ++j) {
            int64_t c = col_offset + j;
            int m = mask ? (mask[k * ld_mask + j] != 0) : 1;
            if (m && r >= 0 && r < rows && c >= 0 && c < cols)
                put(dst, r * ld_dst + c, es, at(src, k * ld_src + j, es));
        }
    }
}

/* Ragged 3D tile load.
 * Mojo "RaggedTMA3DTile", struct description: the source is a packed ragged
 * array (rows, middle_dim, depth) whose leading (row) dimension concatenates
 * sequences; tiles are taken per middle (head) index, and only `dynamic_dim`
 * rows of a tile are valid.  Read in the loading direction: sequence b owns
 * packed rows [cu[b], cu[b+1]); out[b][h][r][d] is x[(cu[b]+r)*ld_row +
 * h*ld_head + d] for r < cu[b+1]-cu[b] (and the packed row inside
 * [0, total_rows)), and zero for every other row up to t_pad.  The output is
 * dense [batch][heads][t_pad][depth]. */
void oracle_ragged_tile_load(int es, const void* x, int64_t total_rows, int32_t heads, int32_t depth, int64_t ld_row,
                             int64_t ld_head, const int32_t* cu_seqlens, int32_t batch, int32_t t_pad, void* out) {
    static const unsigned char zero[8] = {0};
    for (int32_t b = 0; b < batch; ++b) {
        int64_t off = cu_seqlens[b];
        int64_t len = (int64_t)cu_seqlens[b + 1] - cu_seqlens[b];
        for (int32_t h = 0; h < heads; ++h)
            for (int32_t r = 0; r < t_pad; ++r)
                for (int32_t d = 0; d < depth; ++d) {
                    int64_t row = off + r;
                    int64_t o = (((int64_t)b * heads + h) * t_pad + r) * depth + d;
                    if (r < len && row >= 0 && row < total_rows)
                        put(out, o, es, at(x, row * ld_row + (int64_t)h * ld_head + d, es));
                    else
                        put(out, o, es, zero);
                }
    }
}

static float f32_of(const void* p) { float f; memcpy(&f, p, 4); return f; }
static double bf16_bits_f64(uint16_t b) { uint32_t u = (uint32_t)b << 16; float f; memcpy(&f, &u, 4); return (double)f; }
static double f16_bits_f64(uint16_t h) {
    int e = (h >> 10) & 0x1F, m = h & 0x3FF;
    double v = e == 0 ? ldexp((double)m, -24) : (e == 31 ? (m ? NAN : INFINITY) : ldexp((double)(m | 0x400), e - 25));
    return (h & 0x8000) ? -v : v;
}
uint16_t oracle_bf16_rne(double x);
/* double -> binary16 bits, round to nearest even (spacing 2^(e-11) for normals, 2^-24 below 2^-14). */
static uint16_t f16_rne(double x) {
    if (isnan(x)) return 0x7E00;
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    double a = fabs(x);
    if (a == 0.0) return sign;
    int e;
    frexp(a, &e);
    int q_exp = e - 11 > -24 ? e - 11 : -24;
    double q = rint(ldexp(a, -q_exp));
    double y = ldexp(q, q_exp);
    if (y >= 65520.0 || isinf(a)) return sign | 0x7C00;
    if (y < 0x1p-14) return sign | (uint16_t)rint(ldexp(y, 24));
    frexp(y, &e);
    int m = (int)rint(ldexp(y, 11 - e)) - 0x400;
    return sign | (uint16_t)(((e + 14) << 10) | m);
}

/* Row scatter-add, the adjoint of the row gather.
 * warp.tile_load_indexed, description: in a backward pass the adjoint of the
 * gathered tile is accumulated atomically into the array's gradient at the
 * gathered locations.  Source element (k, j) is added to dst row
 * row_offset + idx[k], column col_offset + j, when that coordinate is inside
 * the array; elements that read padding in the forward pass have no location
 * and add nothing.  Each addition happens in the element type with one
 * rounding to nearest even (the exact sum of two values of the type is formed
 * in double first: double has more than 2p+2 significand bits for p = 24, 11
 * or 8, so rounding it again to the type is the correctly rounded sum).
 * es/kind: 4 = fp32, 2 = bf16, 3 = fp16 (2-byte storage). */
void oracle_scatter_add_rows(int kind, void* dst, int64_t rows, int64_t cols, int64_t ld_dst, const int32_t* idx,
                             int64_t n_idx, int64_t row_offset, int64_t col_offset, const void* src, int64_t ld_src,
                             int32_t tile_c) {
    int es = kind == 4 ? 4 : 2;
    for (int64_t k = 0; k < n_idx; ++k) {
        int64_t r = (int64_t)idx[k] + row_offset;
        if (r < 0 || r >= rows) continue;
        for (int32_t j = 0; j < tile_c; ++j) {
            int64_t c = col_offset + j;
            if (c < 0 || c >= cols) continue;
            char* d = (char*)dst + (r * ld_dst + c) * es;
            const char* s = (const char*)src + (k * ld_src + j) * es;
            if (kind == 4) {
                float v = (float)((double)f32_of(d) + (double)f32_of(s));
                memcpy(d, &v, 4);
            } else {
                uint16_t a, b, out;
                memcpy(&a, d, 2);
                memcpy(&b, s, 2);
                if (kind == 2)
                    out = oracle_bf16_rne(bf16_bits_f64(a) + bf16_bits_f64(b));
                else
                    out = f16_rne(f16_bits_f64(a) + f16_bits_f64(b));
                memcpy(d, &out, 2);
            }
        }
    }
}

/* Ragged 3D tile store, the inverse of the ragged load.
 * Mojo "RaggedTMA3DTile", async_copy_from_col / async_copy_batched: tiles
 * are copied from shared memory back to the packed ragged array, only the
 * first `dynamic_dim` rows (valid sequence positions) of a tile are written
 * and a box that overhangs the array is masked off.  Here: for b < batch,
 * h < heads, r < t_pad, d < depth, when r < cu[b+1]-cu[b] and the packed row
 * cu[b]+r lies in [0, total_rows):
 *   x[(cu[b]+r)*ld_row + h*ld_head + d] = tiles[((b*heads + h)*t_pad + r)*depth + d];
 * nothing else of x is written. */
void oracle_ragged_tile_store(int es, const void* tiles, int32_t batch, int32_t heads, int32_t depth, int32_t t_pad,
                              const int32_t* cu_seqlens, void* x, int64_t total_rows, int64_t ld_row,
                              int64_t ld_head) {
    for (int32_t b = 0; b < batch; ++b) {
        int64_t off = cu_seqlens[b];
        int64_t len = (int64_t)cu_seqlens[b + 1] - cu_seqlens[b];
        for (int32_t h = 0; h < heads; ++h)
            for (int32_t r = 0; r < t_pad; ++r)
                for (int32_t d = 0; d < depth; ++d) {
                    int64_t row = off + r;
                    if (r < len && row >= 0 && row < total_rows)
                        put(x, row * ld_row + (int64_t)h * ld_head + d, es,
                            at(tiles, (((int64_t)b * heads + h) * t_pad + r) * depth + d, es));
                }
    }
}

/* bf16 bits -> double (exact: bf16 is the top half of an IEEE binary32). */
static double bf16_to_f64(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

/* Low-precision formats, decoded from their definitions (OCP 8-bit floating
 * point and microscaling formats):
 *   fmt 0 = E4M3 (bias 7, subnormals, no infinities, S.1111.111 is NaN)
 *   fmt 1 = E5M2 (bias 15, IEEE-style infinities and NaNs)
 *   fmt 2 = E8M0 (unsigned exponent: 2^(e-127), 0xFF is NaN)
 *   fmt 3 = E2M1 (4-bit: bias 1, one subnormal 0.5, no infinities or NaNs;
 *           the code is the low 4 bits of b) */
double oracle_fp8_decode(int fmt, uint8_t b) {
    if (fmt == 2) return b == 0xFF ? NAN : ldexp(1.0, (int)b - 127);
    int sign, e, m;
    double v;
    if (fmt == 3) {
        sign = (b >> 3) & 1;
        e = (b >> 1) & 3;
        m = b & 1;
        v = e == 0 ? 0.5 * m : ldexp((double)(2 + m), e - 2);
        return sign ? -v : v;
    }
    sign = b >> 7;
    if (fmt == 0) {
        e = (b >> 3) & 15;
        m = b & 7;
        if (e == 15 && m == 7) return NAN;
        v = e == 0 ? ldexp((double)m, -9) : ldexp((double)(8 + m), e - 10);
    } else {
        e = (b >> 2) & 31;
        m = b & 3;
        if (e == 31) return m ? NAN : (sign ? -INFINITY : INFINITY);
        v = e == 0 ? ldexp((double)m, -16) : ldexp((double)(4 + m), e - 17);
    }
    return sign ? -v : v;
}

/* Element i (row * ld + col) of a row-major low-precision matrix.  E2M1
 * elements are packed two per byte, element i in byte i / 2, the even one in
 * the low nibble. */
static double lowp_at(int fmt, const uint8_t* p, int64_t i) {
    if (fmt == 3) return oracle_fp8_decode(3, (uint8_t)(p[i >> 1] >> (4 * (i & 1))));
    return oracle_fp8_decode(fmt, p[i]);
}

/* Block-scaled GEMM reference.
 * cuTile.jl "Operations", muladd_scaled: D = (a .* a_scale) * (b .* b_scale) + acc
 * where each scale element multiplies a contiguous block of `block` = K / K_s
 * elements along K; a_scale is (M, K_s), b_scale is (K_s, N).  Operands in
 * E4M3, E5M2 or E2M1 (afmt, bfmt), scales in E8M0 or E4M3 (sfmt), acc fp32
 * (NULL: zero).  Every scaled operand and every product is exact in double;
 * the sum runs in double over k = 0..K-1, then acc is added. */
void oracle_gemm_block_scaled_f64(int afmt, int bfmt, int sfmt, const uint8_t* A, int64_t lda, const uint8_t* SA,
                                  int64_t ldsa, const uint8_t* B, int64_t ldb, const uint8_t* SB, int64_t ldsb,
                                  const float* acc, int64_t ld_acc, int64_t M, int64_t N, int64_t K, int64_t block,
                                  double* D, int64_t ldd) {
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n) {
            double s = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                double a = lowp_at(afmt, A, m * lda + k) * oracle_fp8_decode(sfmt, SA[m * ldsa + k / block]);
                double b = lowp_at(bfmt, B, k * ldb + n) * oracle_fp8_decode(sfmt, SB[(k / block) * ldsb + n]);
                s += a * b;
            }
            D[m * ldd + n] = s + (acc ? (double)acc[m * ld_acc + n] : 0.0);
        }
}

/* GEMM reference, full matrix.
 * cuTile.jl "Operations", muladd: (M,K) x (K,N) -> (M,N), and bf16 inputs
 * accumulate in a wider type; Tylo.jl "Boundary tiles", section "Accumulator
 * stores and GEMM": the K loop and the output grid cover the logical extents
 * only.  Here every product of two bf16 values is exact in double and the sum
 * runs in double, k = 0..K-1:  C[m][n] = sum_k A[m][k] * B[k][n]. */
void oracle_gemm_f64(const uint16_t* A, int64_t lda, const uint16_t* B, int64_t ldb, int64_t M, int64_t N, int64_t K,
                     double* C, int64_t ldc) {
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n) {
            double s = 0.0;
            for (int64_t k = 0; k < K; ++k) s += bf16_to_f64(A[m * lda + k]) * bf16_to_f64(B[k * ldb + n]);
            C[m * ldc + n] = s;
        }
}

/* The same sum for a list of (m, n) positions, for spot checks of large shapes. */
void oracle_gemm_f64_at(const uint16_t* A, int64_t lda, const uint16_t* B, int64_t ldb, int64_t K, const int64_t* ms,
                        const int64_t* ns, int64_t count, double* out) {
    for (int64_t t = 0; t < count; ++t) {
        double s = 0.0;
        for (int64_t k = 0; k < K; ++k) s += bf16_to_f64(A[ms[t] * lda + k]) * bf16_to_f64(B[k * ldb + ns[t]]);
        out[t] = s;
    }
}

/* double -> bf16 bits, round to nearest, ties to even, in one step (no
 * intermediate binary32 rounding).  Tylo.jl "Boundary tiles", section
 * "Accumulator stores and GEMM": the accumulator is converted to the
 * destination type at the store; the mode is taken as IEEE's default.
 * x = f * 2^e with f in [0.5, 1): a bf16 normal keeps 8 significant bits, so
 * its spacing is 2^(e-8); below 2^-126 the spacing is fixed at 2^-133.
 * rint() rounds to nearest-even in the default floating-point environment. */
uint16_t oracle_bf16_rne(double x) {
    if (isnan(x)) return (uint16_t)0x7FC0;
    if (isinf(x)) return (uint16_t)(x > 0 ? 0x7F80 : 0xFF80);
    if (x == 0.0) return (uint16_t)(signbit(x) ? 0x8000 : 0x0000);
    int e;
    frexp(x, &e);
    int q_exp = e - 8 > -133 ? e - 8 : -133;
    double q = rint(ldexp(x, -q_exp));
    double y = ldexp(q, q_exp);
    if (fabs(y) >= 0x1p128) return (uint16_t)(y > 0 ? 0x7F80 : 0xFF80);
    float f = (float)y; /* exact: y has at most 8 significant bits and is in binary32 range */
    uint32_t u;
    memcpy(&u, &f, 4);
    return (uint16_t)(u >> 16);
}

void oracle_round_bf16(const double* in, int64_t n, uint16_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_bf16_rne(in[i]);
}

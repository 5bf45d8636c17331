"""Planted mistakes in the oracle fail its pins.

Each case copies the oracle, the input generators and the pin tests into a
scratch directory, plants one plausible mistake in the oracle's C source (a
dropped bound, swapped strides, a truncated offset, pad replaced by data, an
ignored mask, an off-by-one length, a transposed operand, a skipped term, the
wrong rounding, a wrong format field), rebuilds that copy and runs
tests/test_oracle_pins.py against it: every mutant must fail at least one pin.
This is what makes the pins evidence: they are not the oracle's formulas
typed twice.  Everything runs on the CPU; the repository's own oracle is not
touched.
"""
import concurrent.futures
import os
import shutil
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

MUTATIONS = {
    # gather (warp.tile_load_indexed, description)
    "gather_row_bound_dropped": (
        "if (m && r >= 0 && r < rows && c >= 0 && c < cols)\n                put(out, k * ld_out + j, es, at(src, r * ld_src + c, es));",
        "if (m && r >= 0 && c >= 0 && c < cols)\n                put(out, k * ld_out + j, es, at(src, r * ld_src + c, es));"),
    "gather_offset_in_32_bits": (
        "int64_t ld_out, const void* pad) {\n    for (int64_t k = 0; k < n_idx; ++k) {\n        int64_t r = (int64_t)idx[k] + row_offset;",
        "int64_t ld_out, const void* pad) {\n    for (int64_t k = 0; k < n_idx; ++k) {\n        int64_t r = (int32_t)((uint32_t)idx[k] + (uint32_t)row_offset);"),
    "gather_pad_replaced_by_data": (
        "                put(out, k * ld_out + j, es, pad);",
        "                put(out, k * ld_out + j, es, at(src, 0, es));"),
    "gather_mask_ignored": (
        "            int m = mask ? (mask[k * ld_mask + j] != 0) : 1;\n            if (m && r >= 0 && r < rows && c >= 0 && c < cols)\n                put(out",
        "            int m = 1;\n            if (m && r >= 0 && r < rows && c >= 0 && c < cols)\n                put(out"),
    "gather_cols_row_and_column_swapped": (
        "put(out, i * ld_out + k, es, at(src, r * ld_src + c, es));",
        "put(out, i * ld_out + k, es, at(src, c * ld_src + r, es));"),
    # padded load / clipped store (Tylo "Boundary tiles", cuTile "Memory")
    "tile_load_strides_swapped": (
        "put(dst, o, es, at(src, r * stride_r + c * stride_c, es));",
        "put(dst, o, es, at(src, r * stride_c + c * stride_r, es));"),
    "tile_load_column_bound_dropped": (
        "if (r >= 0 && r < rows && c >= 0 && c < cols)\n                        put(dst, o, es, at(src",
        "if (r >= 0 && r < rows && c >= 0)\n                        put(dst, o, es, at(src"),
    "tile_load_pad_written_as_zero": (
        "                        put(dst, o, es, pad);",
        "                        { static const unsigned char z[8] = {0}; put(dst, o, es, z); }"),
    "tile_load_row_step_read_as_tile_height": (
        "int64_t r = origin_r + (int64_t)ti * step_r + i;\n                    int64_t c = origin_c + (int64_t)tj * step_c + j;\n                    int64_t o = (((int64_t)ti * grid_c + tj) * tile_r + i) * tile_c + j;\n                    if (r >= 0 && r < rows && c >= 0 && c < cols)\n                        put(dst, o,",
        "int64_t r = origin_r + (int64_t)ti * tile_r + i;\n                    int64_t c = origin_c + (int64_t)tj * step_c + j;\n                    int64_t o = (((int64_t)ti * grid_c + tj) * tile_r + i) * tile_c + j;\n                    if (r >= 0 && r < rows && c >= 0 && c < cols)\n                        put(dst, o,"),
    "ragged_load_tail_not_zeroed": (
        "                        put(out, o, es, zero);",
        "                        put(out, o, es, at(x, 0, es));"),
    "tile_store_writes_one_column_past": (
        "if (r >= 0 && r < rows && c >= 0 && c < cols)\n                        put(dst, r * stride_r",
        "if (r >= 0 && r < rows && c >= 0 && c <= cols)\n                        put(dst, r * stride_r"),
    "tile_store_row_bound_dropped": (
        "if (r >= 0 && r < rows && c >= 0 && c < cols)\n                        put(dst, r * stride_r",
        "if (r >= 0 && c >= 0 && c < cols)\n                        put(dst, r * stride_r"),
    "tile_store_row_step_read_as_tile_height": (
        "int64_t r = origin_r + (int64_t)ti * step_r + i;\n                    int64_t c = origin_c + (int64_t)tj * step_c + j;\n                    int64_t o = (((int64_t)ti * grid_c + tj) * tile_r + i) * tile_c + j;\n                    if (r >= 0 && r < rows && c >= 0 && c < cols)\n                        put(dst, r * stride_r",
        "int64_t r = origin_r + (int64_t)ti * tile_r + i;\n                    int64_t c = origin_c + (int64_t)tj * step_c + j;\n                    int64_t o = (((int64_t)ti * grid_c + tj) * tile_r + i) * tile_c + j;\n                    if (r >= 0 && r < rows && c >= 0 && c < cols)\n                        put(dst, r * stride_r"),
    "gather_col_offset_ignored": (
        "            int64_t c = col_offset + j;\n            int m = mask ? (mask[k * ld_mask + j] != 0) : 1;\n            if (m && r >= 0 && r < rows && c >= 0 && c < cols)\n                put(out",
        "            int64_t c = j;\n            int m = mask ? (mask[k * ld_mask + j] != 0) : 1;\n            if (m && r >= 0 && r < rows && c >= 0 && c < cols)\n                put(out"),
    # masked scatter
    "scatter_row_offset_ignored": (
        "        int64_t r = (int64_t)idx[k] + row_offset;\n        for (int32_t j = 0; j < tile_c; ++j) {\n            int64_t c = col_offset + j;\n            int m = mask ? (mask[k * ld_mask + j] != 0) : 1;\n            if (m && r >= 0 && r < rows && c >= 0 && c < cols)\n                put(dst",
        "        int64_t r = (int64_t)idx[k];\n        for (int32_t j = 0; j < tile_c; ++j) {\n            int64_t c = col_offset + j;\n            int m = mask ? (mask[k * ld_mask + j] != 0) : 1;\n            if (m && r >= 0 && r < rows && c >= 0 && c < cols)\n                put(dst"),
    "scatter_add_row_offset_ignored": (
        "        int64_t r = (int64_t)idx[k] + row_offset;\n        if (r < 0 || r >= rows) continue;",
        "        int64_t r = (int64_t)idx[k];\n        if (r < 0 || r >= rows) continue;"),
    "ragged_store_head_and_row_strides_swapped": (
        "put(x, row * ld_row + (int64_t)h * ld_head + d, es,",
        "put(x, row * ld_head + (int64_t)h * ld_row + d, es,"),
    "block_scaled_acc_read_with_ldd": ("acc[m * ld_acc + n]", "acc[m * ldd + n]"),
    "bf16_rounded_to_nine_bits": (
        "int q_exp = e - 8 > -133 ? e - 8 : -133;",
        "int q_exp = e - 9 > -133 ? e - 9 : -133;"),
    "f16_overflow_tested_before_rounding": (
        "if (y >= 65520.0 || isinf(a)) return sign | 0x7C00;",
        "if (a > 65504.0 || isinf(a)) return sign | 0x7C00;"),
    "gather_output_leading_dimension_ignored": (
        "put(out, k * ld_out + j, es, at(src, r * ld_src + c, es));",
        "put(out, k * tile_c + j, es, at(src, r * ld_src + c, es));"),
    "gather_mask_leading_dimension_ignored": (
        "            int m = mask ? (mask[k * ld_mask + j] != 0) : 1;\n            if (m && r >= 0 && r < rows && c >= 0 && c < cols)\n                put(out",
        "            int m = mask ? (mask[k * tile_c + j] != 0) : 1;\n            if (m && r >= 0 && r < rows && c >= 0 && c < cols)\n                put(out"),
    "scatter_mask_leading_dimension_ignored": (
        "            int m = mask ? (mask[k * ld_mask + j] != 0) : 1;\n            if (m && r >= 0 && r < rows && c >= 0 && c < cols)\n                put(dst",
        "            int m = mask ? (mask[k * tile_c + j] != 0) : 1;\n            if (m && r >= 0 && r < rows && c >= 0 && c < cols)\n                put(dst"),
    "scatter_source_leading_dimension_ignored": (
        "put(dst, r * ld_dst + c, es, at(src, k * ld_src + j, es));",
        "put(dst, r * ld_dst + c, es, at(src, k * tile_c + j, es));"),
    "scatter_add_source_leading_dimension_ignored": (
        "const char* s = (const char*)src + (k * ld_src + j) * es;",
        "const char* s = (const char*)src + (k * tile_c + j) * es;"),
    "gather_cols_output_leading_dimension_ignored": (
        "put(out, i * ld_out + k, es, at(src, r * ld_src + c, es));",
        "put(out, i * n_idx + k, es, at(src, r * ld_src + c, es));"),
    "ragged_load_row_stride_read_as_dense": (
        "put(out, o, es, at(x, row * ld_row + (int64_t)h * ld_head + d, es));",
        "put(out, o, es, at(x, row * (int64_t)heads * depth + (int64_t)h * ld_head + d, es));"),
    "ragged_store_row_stride_read_as_dense": (
        "put(x, row * ld_row + (int64_t)h * ld_head + d, es,",
        "put(x, row * (int64_t)heads * depth + (int64_t)h * ld_head + d, es,"),
    "tile_load_row_stride_read_as_cols": (
        "put(dst, o, es, at(src, r * stride_r + c * stride_c, es));",
        "put(dst, o, es, at(src, r * cols + c * stride_c, es));"),
    "tile_store_row_stride_read_as_cols": (
        "put(dst, r * stride_r + c * stride_c, es, at(src_tiles, o, es));",
        "put(dst, r * cols + c * stride_c, es, at(src_tiles, o, es));"),
    "ragged_load_output_head_major": (
        "int64_t o = (((int64_t)b * heads + h) * t_pad + r) * depth + d;",
        "int64_t o = (((int64_t)h * batch + b) * t_pad + r) * depth + d;"),
    "tile_load_output_tile_column_major": (
        "int64_t o = (((int64_t)ti * grid_c + tj) * tile_r + i) * tile_c + j;\n                    if (r >= 0 && r < rows && c >= 0 && c < cols)\n                        put(dst, o, es, at(src",
        "int64_t o = (((int64_t)tj * grid_r + ti) * tile_r + i) * tile_c + j;\n                    if (r >= 0 && r < rows && c >= 0 && c < cols)\n                        put(dst, o, es, at(src"),
    "tile_store_input_tile_column_major": (
        "int64_t o = (((int64_t)ti * grid_c + tj) * tile_r + i) * tile_c + j;\n                    if (r >= 0 && r < rows && c >= 0 && c < cols)\n                        put(dst, r * stride_r",
        "int64_t o = (((int64_t)tj * grid_r + ti) * tile_r + i) * tile_c + j;\n                    if (r >= 0 && r < rows && c >= 0 && c < cols)\n                        put(dst, r * stride_r"),
    "ragged_store_packed_bound_dropped": (
        "if (r < len && row >= 0 && row < total_rows)\n                        put(x,",
        "if (r < len && row >= 0)\n                        put(x,"),
    "gather_cols_row_bound_dropped": (
        "if (r >= 0 && r < rows && c >= 0 && c < cols)\n                put(out, i * ld_out + k",
        "if (r >= 0 && c >= 0 && c < cols)\n                put(out, i * ld_out + k"),
    "scatter_column_bound_dropped": (
        "if (m && r >= 0 && r < rows && c >= 0 && c < cols)\n                put(dst",
        "if (m && r >= 0 && r < rows && c >= 0)\n                put(dst"),
    "scatter_mask_ignored": (
        "            int m = mask ? (mask[k * ld_mask + j] != 0) : 1;\n            if (m && r >= 0 && r < rows && c >= 0 && c < cols)\n                put(dst",
        "            int m = 1;\n            if (m && r >= 0 && r < rows && c >= 0 && c < cols)\n                put(dst"),
    # ragged load / store (Mojo "RaggedTMA3DTile")
    "ragged_load_length_off_by_one": (
        "if (r < len && row >= 0 && row < total_rows)\n                        put(out, o",
        "if (r <= len && row >= 0 && row < total_rows)\n                        put(out, o"),
    "ragged_load_head_and_row_strides_swapped": (
        "put(out, o, es, at(x, row * ld_row + (int64_t)h * ld_head + d, es));",
        "put(out, o, es, at(x, row * ld_head + (int64_t)h * ld_row + d, es));"),
    "ragged_store_length_off_by_one": (
        "if (r < len && row >= 0 && row < total_rows)\n                        put(x,",
        "if (r <= len && row >= 0 && row < total_rows)\n                        put(x,"),
    # gather backward
    "scatter_add_overwrites": (
        "float v = (float)((double)f32_of(d) + (double)f32_of(s));",
        "float v = f32_of(s);"),
    # GEMM and bf16 rounding
    "gemm_a_transposed": (
        "s += bf16_to_f64(A[m * lda + k]) * bf16_to_f64(B[k * ldb + n]);",
        "s += bf16_to_f64(A[k * lda + m]) * bf16_to_f64(B[k * ldb + n]);"),
    "gemm_skips_k0": (
        "for (int64_t k = 0; k < K; ++k) s += bf16_to_f64(A[m * lda + k])",
        "for (int64_t k = 1; k < K; ++k) s += bf16_to_f64(A[m * lda + k])"),
    "bf16_ties_away_from_zero": (
        "double q = rint(ldexp(x, -q_exp));",
        "double q = round(ldexp(x, -q_exp));"),
    "bf16_subnormal_clamp_dropped": (
        "int q_exp = e - 8 > -133 ? e - 8 : -133;",
        "int q_exp = e - 8;"),
    # block-scaled GEMM (cuTile "Operations", muladd_scaled) and the 8-bit / 4-bit formats
    "scale_indexed_by_k_mod_block": ("SA[m * ldsa + k / block]", "SA[m * ldsa + k % block]"),
    "b_scale_transposed": ("SB[(k / block) * ldsb + n]", "SB[n * ldsb + k / block]"),
    "e4m3_subnormal_exponent": (
        "v = e == 0 ? ldexp((double)m, -9) : ldexp((double)(8 + m), e - 10);",
        "v = e == 0 ? ldexp((double)m, -10) : ldexp((double)(8 + m), e - 10);"),
    "e4m3_bias": (
        "v = e == 0 ? ldexp((double)m, -9) : ldexp((double)(8 + m), e - 10);",
        "v = e == 0 ? ldexp((double)m, -9) : ldexp((double)(8 + m), e - 11);"),
    "e5m2_infinity_and_nan_swapped": (
        "if (e == 31) return m ? NAN : (sign ? -INFINITY : INFINITY);",
        "if (e == 31) return m ? (sign ? -INFINITY : INFINITY) : NAN;"),
    "e2m1_nibble_order": (
        "return oracle_fp8_decode(3, (uint8_t)(p[i >> 1] >> (4 * (i & 1))));",
        "return oracle_fp8_decode(3, (uint8_t)(p[i >> 1] >> (4 * (1 - (i & 1)))));"),
    "e8m0_bias": (
        "if (fmt == 2) return b == 0xFF ? NAN : ldexp(1.0, (int)b - 127);",
        "if (fmt == 2) return b == 0xFF ? NAN : ldexp(1.0, (int)b - 126);"),
    "block_scaled_acc_dropped": (
        "D[m * ldd + n] = s + (acc ? (double)acc[m * ld_acc + n] : 0.0);",
        "D[m * ldd + n] = s;"),
    "e4m3_nan_read_as_a_number": ("        if (e == 15 && m == 7) return NAN;\n", ""),
    "e2m1_sign_ignored": ("        sign = (b >> 3) & 1;", "        sign = 0;"),
    "e2m1_subnormal_value": (
        "v = e == 0 ? 0.5 * m : ldexp((double)(2 + m), e - 2);",
        "v = e == 0 ? 1.0 * m : ldexp((double)(2 + m), e - 2);"),
    "e5m2_subnormal_exponent": (
        "v = e == 0 ? ldexp((double)m, -16) : ldexp((double)(4 + m), e - 17);",
        "v = e == 0 ? ldexp((double)m, -17) : ldexp((double)(4 + m), e - 17);"),
    "a_scale_decoded_in_the_operand_format": (
        "oracle_fp8_decode(sfmt, SA[m * ldsa + k / block])",
        "oracle_fp8_decode(afmt, SA[m * ldsa + k / block])"),
    "b_scale_sign_ignored": (
        "oracle_fp8_decode(sfmt, SB[(k / block) * ldsb + n])",
        "fabs(oracle_fp8_decode(sfmt, SB[(k / block) * ldsb + n]))"),
    "a_scale_sign_ignored": (
        "oracle_fp8_decode(sfmt, SA[m * ldsa + k / block])",
        "fabs(oracle_fp8_decode(sfmt, SA[m * ldsa + k / block]))"),
    "b_scale_read_with_the_a_scale_stride": ("SB[(k / block) * ldsb + n]", "SB[(k / block) * ldsa + n]"),
    "scale_block_fixed_at_32": ("SA[m * ldsa + k / block]", "SA[m * ldsa + k / 32]"),
    # more movement mistakes
    "gather_cols_column_bound_dropped": (
        "if (r >= 0 && r < rows && c >= 0 && c < cols)\n                put(out, i * ld_out + k",
        "if (r >= 0 && r < rows && c >= 0)\n                put(out, i * ld_out + k"),
    "gather_cols_offset_ignored": (
        "int64_t c = (int64_t)idx[k] + col_offset;",
        "int64_t c = (int64_t)idx[k];"),
    "scatter_row_bound_dropped": (
        "if (m && r >= 0 && r < rows && c >= 0 && c < cols)\n                put(dst",
        "if (m && r >= 0 && c >= 0 && c < cols)\n                put(dst"),
    "scatter_source_transposed": (
        "put(dst, r * ld_dst + c, es, at(src, k * ld_src + j, es));",
        "put(dst, r * ld_dst + c, es, at(src, j * ld_src + k, es));"),
    "tile_store_strides_swapped": (
        "put(dst, r * stride_r + c * stride_c, es, at(src_tiles, o, es));",
        "put(dst, r * stride_c + c * stride_r, es, at(src_tiles, o, es));"),
    "ragged_load_packed_bound_dropped": (
        "if (r < len && row >= 0 && row < total_rows)\n                        put(out, o",
        "if (r < len && row >= 0)\n                        put(out, o"),
    "scatter_add_column_bound_dropped": ("if (c < 0 || c >= cols) continue;", "if (c < 0) continue;"),
    "scatter_add_f16_rounded_as_bf16": (
        "out = f16_rne(f16_bits_f64(a) + f16_bits_f64(b));",
        "out = oracle_bf16_rne(f16_bits_f64(a) + f16_bits_f64(b));"),
    "f16_decode_subnormal_exponent": (
        "double v = e == 0 ? ldexp((double)m, -24) : (e == 31",
        "double v = e == 0 ? ldexp((double)m, -25) : (e == 31"),
    "gemm_spot_check_indices_swapped": (
        "bf16_to_f64(A[ms[t] * lda + k]) * bf16_to_f64(B[k * ldb + ns[t]])",
        "bf16_to_f64(A[ns[t] * lda + k]) * bf16_to_f64(B[k * ldb + ms[t]])"),
    "bf16_nan_becomes_infinity": (
        "if (isnan(x)) return (uint16_t)0x7FC0;",
        "if (isnan(x)) return (uint16_t)0x7F80;"),
}

# Not in the list because no input can tell them from the oracle (equivalent mutants): rounding a
# scatter-add sum through binary32 before bf16 (binary32 carries more than 2p + 2 bits for p = 8, so
# the double rounding is innocuous), and dropping the subnormal clamp of the fp16 rounding (a sum of
# two binary16 values that lands below 2^-14 is a multiple of 2^-24 and needs no rounding), and testing the
# rounded fp16 sum for overflow with `> 65504` instead of `>= 65520` (the rounded value is on the fp16 grid,
# where the next value after 65504 is 65536, so the two tests agree).

IGNORE = shutil.ignore_patterns("__pycache__", "*.tmp*")


def run_mutant(base, name, old, new):
    d = os.path.join(base, name)
    shutil.copytree(os.path.join(ROOT, "oracle"), os.path.join(d, "oracle"),
                    ignore=shutil.ignore_patterns("__pycache__", "*.so", "*.tmp*"))
    shutil.copytree(os.path.join(ROOT, "synth"), os.path.join(d, "synth"), ignore=IGNORE)
    os.makedirs(os.path.join(d, "tests"))
    for f in ("conftest.py", "test_oracle_pins.py"):
        shutil.copy(os.path.join(ROOT, "tests", f), os.path.join(d, "tests", f))
    shutil.copytree(os.path.join(ROOT, "tests", "golden"), os.path.join(d, "tests", "golden"))
    src = os.path.join(d, "oracle", "sbt_oracle.c")
    s = open(src).read()
    if s.count(old) != 1:
        return "mutation site not found once"
    open(src, "w").write(s.replace(old, new))
    env = dict(os.environ, PYTHONPATH=d, CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, "-c", "import synth, oracle; synth.build(); oracle.build(force=True)"],
                       cwd=d, env=env, capture_output=True, text=True, timeout=300)
    if r.returncode:
        return "does not compile: " + r.stderr[-300:]
    r = subprocess.run([sys.executable, "-m", "pytest", "tests/test_oracle_pins.py", "-q", "-x", "-p",
                        "no:cacheprovider"], cwd=d, env=env, capture_output=True, text=True, timeout=600)
    return "caught" if r.returncode != 0 else "NOT CAUGHT"


def test_every_planted_mistake_fails_a_pin(tmp_path):
    with concurrent.futures.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
        futs = {name: ex.submit(run_mutant, str(tmp_path), name, old, new) for name, (old, new) in MUTATIONS.items()}
        results = {name: f.result() for name, f in futs.items()}
    bad = {name: r for name, r in results.items() if r != "caught"}
    assert not bad, bad

// Boundary-tile bf16 GEMM (placeholder until the tcgen05 kernel lands).
#include "sbt_internal.cuh"

size_t sbt_gemm_workspace_bytes(int64_t M, int64_t N, int64_t K) {
    (void)M; (void)N; (void)K;
    return 0;
}

sbt_status sbt_launch_gemm(sbt_context* ctx, const void* A, int64_t lda, const void* B, int64_t ldb, void* C,
                           int64_t ldc, sbt_dtype c_dtype, int64_t M, int64_t N, int64_t K, void* workspace,
                           size_t workspace_bytes, cudaStream_t stream) {
    (void)ctx; (void)A; (void)lda; (void)B; (void)ldb; (void)C; (void)ldc; (void)c_dtype; (void)M; (void)N; (void)K;
    (void)workspace; (void)workspace_bytes; (void)stream;
    return sbt_fail(SBT_ERR_UNSUPPORTED, "gemm_bounded: not built yet");
}

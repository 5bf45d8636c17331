// sbt_gemm_bounded_noalloc: the bounded GEMM with its operand-staging scratch
// in a fixed, library-owned device array instead of a caller workspace.
//
// Who needs this: callers that cannot allocate device memory at the point of
// the call -- plugins that live inside another framework's memory pool and
// are not allowed to call the CUDA allocator themselves, code running under a
// fixed device-memory budget that was committed up front, and latency-critical
// paths that cannot afford the implicit device synchronisation of
// cudaMalloc/cudaFree.  They still pass A, B and C.
//
// The scratch is one file-scope __device__ array per device, created when the
// library's module is loaded on that device and held until process exit.
// Host code may not use the array's name as a device address (on the host it
// is only a stand-in), so the device address is looked up with
// cudaGetSymbolAddress while that device is current, once per device, and
// cached.  The lookup runs on every call's first visit to a device, whatever
// the shape (also when nothing has to be staged), so the first call on a
// device is the only one that does it.  It leaves that device current on the
// calling thread, as every other call of the library does.
//
// Every call shares the array and it keeps the previous call's contents.  The
// GEMM's staging kernels write every byte of the scratch that the main kernel
// reads (the zero padding past M, N and K included), so nothing has to be
// cleared between calls.  Calls that can overlap on the GPU (different
// streams, or different host threads without ordering) race on the array.
#include <mutex>
#include <string>

#include "sbt_internal.cuh"

static __device__ __align__(256) unsigned char g_sbt_gemm_scratch[SBT_GEMM_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void* g_scratch_ptr[kMaxDevices] = {nullptr};

// Device address of this device's scratch array (looked up on first use).
sbt_status scratch_for_device(int device, void** out) {
    if (device < 0 || device >= kMaxDevices) return sbt_fail(SBT_ERR_INVALID_ARG, "gemm_bounded_noalloc: device index too large");
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (!g_scratch_ptr[device]) {
        sbt_status st = sbt_cuda_check(cudaSetDevice(device), "cudaSetDevice");
        if (st) return st;
        void* p = nullptr;
        st = sbt_cuda_check(cudaGetSymbolAddress(&p, g_sbt_gemm_scratch), "cudaGetSymbolAddress(gemm scratch)");
        if (st) return st;
        if (!p) return sbt_fail(SBT_ERR_CUDA, "cudaGetSymbolAddress returned NULL for the gemm scratch");
        g_scratch_ptr[device] = p;
    }
    *out = g_scratch_ptr[device];
    return SBT_OK;
}

}  // namespace

extern "C" SBT_API sbt_status sbt_gemm_bounded_noalloc(sbt_context* ctx, const void* A, int64_t lda, const void* B,
                                                       int64_t ldb, void* C, int64_t ldc, sbt_dtype c_dtype,
                                                       int64_t M, int64_t N, int64_t K, void* stream) {
    if (!ctx) return sbt_fail(SBT_ERR_INVALID_ARG, "ctx is NULL");
    size_t need = 0;
    sbt_status st = sbt_gemm_bounded_workspace_size(ctx, M, N, K, lda, ldb, &need);
    if (st) return st;
    if (need > SBT_GEMM_NOALLOC_SCRATCH_BYTES)
        return sbt_fail(SBT_ERR_INVALID_ARG,
                        "gemm_bounded_noalloc: this shape needs " + std::to_string(need) +
                            " bytes of staging scratch, more than the fixed " +
                            std::to_string((size_t)SBT_GEMM_NOALLOC_SCRATCH_BYTES) +
                            " bytes; use sbt_gemm_bounded with a caller workspace");
    void* scratch = nullptr;
    if ((st = scratch_for_device(ctx->device, &scratch))) return st;
    return sbt_gemm_bounded(ctx, A, lda, B, ldb, C, ldc, c_dtype, M, N, K, scratch, need > 0 ? SBT_GEMM_NOALLOC_SCRATCH_BYTES : 0,
                            stream);
}

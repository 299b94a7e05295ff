// Reconstruction GEMM of the feature-wise baseline ("Speedups are real, but memory
// is set by the ratio": the reconstruction-based variant materialises full-dimension
// keys and values before attention): K_b = C_K . U_K^T (and the same for values),
// written to HBM at full dimension. It is a plain GEMM, so it runs in cuBLAS
// (bf16 operands, float32 accumulation, bf16 result) rather than in a kernel of
// this library; the SlimKV path never calls it.
//
// Row-major out [rows, n] = C [rows, r] . U [n, r]^T is, in cuBLAS's column-major
// terms, out^T (n x rows) = op_T(U as r x n) . op_N(C^T as r x rows).
#include <cublas_v2.h>

#include <mutex>

#include "slimkv_internal.cuh"

namespace slimkv {

namespace {

// One handle per device, created on first use and kept until exit. No cuBLAS
// workspace is attached, so a call never allocates (and may be graph-captured
// once the handle exists).
cublasHandle_t handle_for_current_device(cudaError_t& err) {
    static std::mutex mu;
    static cublasHandle_t handles[64] = {};
    int dev = 0;
    err = cudaGetDevice(&dev);
    if (err != cudaSuccess || dev < 0 || dev >= 64) {
        if (err == cudaSuccess) err = cudaErrorInvalidDevice;
        return nullptr;
    }
    std::lock_guard<std::mutex> g(mu);
    if (handles[dev] == nullptr) {
        cublasHandle_t h = nullptr;
        if (cublasCreate(&h) != CUBLAS_STATUS_SUCCESS || cublasSetWorkspace(h, nullptr, 0) != CUBLAS_STATUS_SUCCESS) {
            if (h) cublasDestroy(h);
            err = cudaErrorUnknown;
            return nullptr;
        }
        handles[dev] = h;
    }
    return handles[dev];
}

}  // namespace

cudaError_t launch_reconstruct_gemm(const __nv_bfloat16* C, const __nv_bfloat16* U, __nv_bfloat16* out,
                                    int rows, int n, int r, cudaStream_t st) {
    cudaError_t err = cudaSuccess;
    cublasHandle_t h = handle_for_current_device(err);
    if (h == nullptr) return err;
    if (cublasSetStream(h, st) != CUBLAS_STATUS_SUCCESS) return cudaErrorUnknown;
    const float one = 1.f, zero = 0.f;
    const cublasStatus_t s = cublasGemmEx(h, CUBLAS_OP_T, CUBLAS_OP_N, n, rows, r, &one, U, CUDA_R_16BF, r, C,
                                          CUDA_R_16BF, r, &zero, out, CUDA_R_16BF, n, CUBLAS_COMPUTE_32F,
                                          CUBLAS_GEMM_DEFAULT);
    return s == CUBLAS_STATUS_SUCCESS ? cudaSuccess : cudaErrorUnknown;
}

}  // namespace slimkv

// Reconstruction GEMM of the feature-wise baseline: K_b = C_K . U_K^T (and the
// same for values), written to HBM at full dimension before attention.
#include "slimkv_internal.cuh"

namespace slimkv {

cudaError_t launch_reconstruct_gemm(const __nv_bfloat16* C, const __nv_bfloat16* U, __nv_bfloat16* out,
                                    int rows, int n, int r, cudaStream_t st) {
    return launch_simt_reconstruct<__nv_bfloat16>(C, U, out, rows, n, r, st);
}

}  // namespace slimkv

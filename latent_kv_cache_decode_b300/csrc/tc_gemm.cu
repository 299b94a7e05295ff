// Reconstruction GEMM of the feature-wise baseline, "Can SlimKV compress KV cache
// jointly across tokens and features", sections "Speedups are real, but memory is set
// by the ratio" and "Why feature compression stalls at key reconstruction": the
// reconstruction-based variant materialises full-dimension keys and values before
// attention, K_b = C_K . U_K^T and V_b = C_V . U_V^T, written to HBM at full width.
// The SlimKV path never calls it.
//
// out[rows, n] = C[rows, r] . U[n, r]^T, bf16 operands, float32 accumulation, bf16
// result, on the fifth-generation tensor cores (sm_103a):
//   * one CTA per 128 rows of C; its C tile (128 x r) is loaded once by TMA into shared
//     memory (128-byte swizzled, K-major) and serves every 128-column block of out;
//   * U streams through a ring of 128 x 64 chunks (TMA), one per 64 of r;
//   * warp 1 issues tcgen05.mma (M = 128, N = 128, K = 16) into one of two TMEM
//     accumulators, so the next column block's MMAs overlap the previous block's
//     write-out;
//   * warps 2-5 read the accumulator with tcgen05.ld (thread = output row), round to
//     bf16 and store 32 contiguous bytes per thread and step (whole 32-byte sectors).
// The write of `out` (rows x n bf16) dominates the traffic, so the kernel is bound by
// HBM bandwidth, not by the tensor cores.
#include <cuda.h>
#include <string.h>

#include <mutex>

#include "slimkv_internal.cuh"
#include "tc_ptx.cuh"

namespace slimkv {

namespace {

constexpr int kGM = 128;         // rows of C per CTA (MMA M)
constexpr int kGN = 128;         // columns of out per block (MMA N)
constexpr int kGK = 64;          // columns of r per chunk (one 128-byte swizzle span)
constexpr int kChunk = 16384;    // bytes of one 128 x 64 bf16 chunk
constexpr int kStages = 4;       // ring of U chunks
constexpr int kThreads = 192;    // warp 0 TMA, warp 1 MMA, warps 2-5 write-out
constexpr int kMaxR = 512;

struct GemmParams {
    CUtensorMap tmC;   // [rows, r] bf16, boxes of 128 rows x 64 columns
    CUtensorMap tmU;   // [n, r] bf16, boxes of 128 rows x 64 columns
    __nv_bfloat16* out;
    int rows, n, r;
};

__global__ void __launch_bounds__(kThreads, 1) recon_gemm_kernel(const __grid_constant__ GemmParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int nkc = (p.r + kGK - 1) / kGK;   // chunks of r
    const int ksteps = p.r / 16;              // 16-wide MMA k-steps
    const int nblk = p.n / kGN;               // column blocks of out
    uint8_t* a_s = smem;                      // nkc chunks of the C tile
    uint8_t* b_s = smem + nkc * kChunk;       // kStages chunks of U
    uint64_t* bars = reinterpret_cast<uint64_t*>(b_s + kStages * kChunk);
    uint64_t* a_full = bars;                  // the C tile landed            [TMA tx]
    uint64_t* full = bars + 1;                // ring slot s holds its chunk  [TMA tx]
    uint64_t* empty = full + kStages;         // ring slot s consumed         [commit]
    uint64_t* acc_full = empty + kStages;     // accumulator b complete       [commit]
    uint64_t* acc_empty = acc_full + 2;       // accumulator b read out       [128 arrivals]
    uint64_t* drain = acc_empty + 2;          // every MMA of the CTA done    [commit]
    volatile int* abort_flag = reinterpret_cast<volatile int*>(drain + 1);
    uint32_t* tmem_base_s = reinterpret_cast<uint32_t*>(drain + 2);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row0 = blockIdx.x * kGM;
    if (threadIdx.x == 0) {
        ptx::mbar_init(a_full, 1);
        for (int s = 0; s < kStages; ++s) {
            ptx::mbar_init(&full[s], 1);
            ptx::mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(&acc_full[b], 1);
            ptx::mbar_init(&acc_empty[b], 128);
        }
        ptx::mbar_init(drain, 1);
        *abort_flag = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 1) ptx::tmem_alloc(tmem_base_s, 2 * kGN);
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_base_s;
    // C and U are inputs of this call: the preceding kernels on the stream must be
    // complete before they are read
    pdl_wait();

    if (warp == 0) {
        // ------------------------------------------------------------------ TMA
        if (lane == 0) {
            ptx::tma_prefetch_desc(&p.tmC);
            ptx::tma_prefetch_desc(&p.tmU);
            ptx::mbar_expect_tx(a_full, nkc * kChunk);
            for (int c = 0; c < nkc; ++c) ptx::tma_load_2d(a_s + c * kChunk, &p.tmC, c * kGK, row0, a_full);
            int it = 0;
            for (int nb = 0; nb < nblk && !*abort_flag; ++nb)
                for (int c = 0; c < nkc; ++c, ++it) {
                    const int s = it % kStages;
                    if (it >= kStages) ptx::mbar_wait(&empty[s], (uint32_t)((it / kStages) - 1) & 1u, abort_flag);
                    ptx::mbar_expect_tx(&full[s], kChunk);
                    ptx::tma_load_2d(b_s + s * kChunk, &p.tmU, c * kGK, nb * kGN, &full[s]);
                }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------------ MMA
        if (lane == 0) {
            const uint32_t idesc = ptx::idesc_bf16(kGM, kGN, false, false);
            const uint64_t dA = ptx::sdesc_sw128(ptx::smem_u32(a_s), 16, 1024);
            const uint64_t dB = ptx::sdesc_sw128(ptx::smem_u32(b_s), 16, 1024);
            ptx::mbar_wait(a_full, 0, abort_flag);
            int it = 0;
            for (int nb = 0; nb < nblk && !*abort_flag; ++nb) {
                const int buf = nb & 1;
                if (nb >= 2) ptx::mbar_wait(&acc_empty[buf], (uint32_t)((nb >> 1) - 1) & 1u, abort_flag);
                ptx::tc_fence_after();
                const uint32_t d = tmem + (uint32_t)(buf * kGN);
                for (int c = 0; c < nkc; ++c, ++it) {
                    const int s = it % kStages;
                    ptx::mbar_wait(&full[s], (uint32_t)(it / kStages) & 1u, abort_flag);
                    ptx::tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < kGK / 16; ++kk) {
                        if (c * (kGK / 16) + kk >= ksteps) break;
                        const uint64_t a = dA + (uint64_t)((c * kChunk + kk * 32) >> 4);
                        const uint64_t b = dB + (uint64_t)((s * kChunk + kk * 32) >> 4);
                        ptx::mma_bf16(d, a, b, idesc, (c | kk) != 0 ? 1u : 0u);
                    }
                    ptx::mma_commit(&empty[s]);
                }
                ptx::mma_commit(&acc_full[buf]);
            }
            ptx::mma_commit(drain);
        }
    } else {
        // ------------------------------------------------------------- write-out
        const int q4 = warp & 3;
        const int row = q4 * 32 + lane;
        const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
        const bool row_ok = row0 + row < p.rows;
        __nv_bfloat16* orow = p.out + (size_t)(row0 + row) * p.n;
        for (int nb = 0; nb < nblk; ++nb) {
            const int buf = nb & 1;
            const bool ok = ptx::mbar_wait(&acc_full[buf], (uint32_t)(nb >> 1) & 1u, abort_flag);
            ptx::tc_fence_after();
#pragma unroll 1
            for (int c0 = 0; c0 < kGN; c0 += 16) {
                float v[16];
                ptx::tmem_ld16(tmem + lane_off + (uint32_t)(buf * kGN + c0), v);
                uint32_t pk[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const __nv_bfloat162 h2 = ok ? __floats2bfloat162_rn(v[2 * i], v[2 * i + 1])
                                                 : __floats2bfloat162_rn(__int_as_float(0x7fc00000),
                                                                         __int_as_float(0x7fc00000));
                    pk[i] = *reinterpret_cast<const uint32_t*>(&h2);
                }
                if (row_ok) {
                    uint4* dst = reinterpret_cast<uint4*>(orow + nb * kGN + c0);
                    dst[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                    dst[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
                }
            }
            ptx::tc_fence_before();
            ptx::mbar_arrive(&acc_empty[buf]);
        }
    }

    // ----------------------------------------------------------------- teardown
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        if (lane == 0) {
            volatile int never = 0;
            ptx::mbar_wait(drain, 0, &never);   // every MMA of this CTA has completed
        }
        __syncwarp();
        ptx::tmem_dealloc(tmem, 2 * kGN);
    }
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    });
    return fn;
}

// A row-major bf16 matrix [rows, cols] read in boxes of 128 rows x 64 columns with the
// 128-byte swizzle (rows past the end read as zero).
bool make_map_2d(CUtensorMap* tm, const void* base, int cols, int64_t rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    cuuint32_t box[2] = {(cuuint32_t)kGK, (cuuint32_t)kGM};
    cuuint32_t es[2] = {1, 1};
    return fn(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_reconstruct_gemm(const __nv_bfloat16* C, const __nv_bfloat16* U, __nv_bfloat16* out,
                                    int rows, int n, int r, cudaStream_t st) {
    if (rows <= 0 || n <= 0 || n % kGN != 0 || r < 16 || r % 16 != 0 || r > kMaxR) return cudaErrorInvalidValue;
    GemmParams p;
    memset(&p, 0, sizeof(p));
    if (!make_map_2d(&p.tmC, C, r, rows) || !make_map_2d(&p.tmU, U, r, n)) return cudaErrorInvalidValue;
    p.out = out;
    p.rows = rows;
    p.n = n;
    p.r = r;
    const int nkc = (r + kGK - 1) / kGK;
    const size_t smem = 1024 + (size_t)(nkc + kStages) * kChunk + 256;
    static std::atomic<unsigned long long> attr_done{0};
    const cudaError_t e = set_max_smem_once((const void*)recon_gemm_kernel,
                                            (int)(1024 + (size_t)(kMaxR / kGK + kStages) * kChunk + 256), attr_done);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((rows + kGM - 1) / kGM);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, recon_gemm_kernel, p);
}

}  // namespace slimkv

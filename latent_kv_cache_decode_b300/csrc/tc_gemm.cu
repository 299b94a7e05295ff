// Reconstruction GEMM of the feature-wise baseline, "Can SlimKV compress KV cache
// jointly across tokens and features", sections "Speedups are real, but memory is set
// by the ratio" and "Why feature compression stalls at key reconstruction": the
// reconstruction-based variant materialises full-dimension keys and values before
// attention, K_b = C_K . U_K^T and V_b = C_V . U_V^T, written to HBM at full width.
// The SlimKV path never calls it.
//
// out[rows, n] = C[rows, r] . U[n, r]^T, bf16 operands, float32 accumulation, bf16
// result, on the fifth-generation tensor cores (sm_103a):
//   * one CTA per 256 rows of C (two 128-row tiles; 128 rows for ranks above 384),
//     loaded once by TMA into shared memory (128-byte swizzled, K-major); the tiles
//     serve every 128-column block of out, and each U chunk serves both tiles, so that
//     U (re-read from L2 by every CTA) costs half the traffic;
//   * U streams through a ring of 128 x 64 chunks (TMA), one per 64 of r;
//   * warp 1 issues tcgen05.mma (M = 128, N = 128, K = 16, one per C tile) into one of
//     two TMEM accumulators, so the next column block's MMAs overlap the previous
//     block's write-out;
//   * warps 2-9 read the accumulator with tcgen05.ld (thread = output row, two warps
//     per row quarter, 32 columns per load), round to bf16 and store 64 contiguous
//     bytes of the row per load (whole 32-byte sectors);
//   * for the baseline that keeps beacon-key RoPE the write-out also rotates each
//     128-column block (one KV head) of a key row at its beacon's position, in float32
//     before the rounding.
// The write of `out` (rows x n bf16) dominates the traffic, so the kernel is bound by
// HBM bandwidth, not by the tensor cores.
#include <cuda.h>
#include <string.h>

#include <algorithm>
#include <mutex>

#include "slimkv_internal.cuh"
#include "tc_ptx.cuh"

namespace slimkv {

namespace {

constexpr int kGM = 128;         // rows of one C tile (MMA M); a CTA holds msub of them
constexpr int kGN = 128;         // columns of out per block (MMA N)
constexpr int kGK = 64;          // columns of r per chunk (one 128-byte swizzle span)
constexpr int kChunk = 16384;    // bytes of one 128 x 64 bf16 chunk
constexpr int kMaxStages = 8;    // ring of U chunks (fewer when the C tile is large)
constexpr int kSmemMax = 227 * 1024;
constexpr int kThreads = 320;    // warp 0 TMA, warp 1 MMA, warps 2-9 write-out
constexpr int kMaxR = 512;

struct GemmParams {
    CUtensorMap tmC;   // [rows, r] bf16, boxes of 128 rows x 64 columns
    CUtensorMap tmU;   // [n, r] bf16, boxes of 128 rows x 64 columns
    __nv_bfloat16* out;
    int rows, n, r;
    int stages;        // ring slots of U (2..kMaxStages)
    int msub;          // C tiles per CTA (1 or 2): every U chunk serves all of them
    // beacon-key RoPE (ratio > 0): row R is beacon j = R % rows_per_b, rotated at position
    // j * ratio + ratio - 1; turn[i] = theta_i / (2 pi) as a 64-bit fraction of a turn
    int ratio, rows_per_b;
    unsigned long long turn[64];
    unsigned long long* aborts;   // device counter of CTAs that gave up on a wait
};

__global__ void __launch_bounds__(kThreads, 1) recon_gemm_kernel(const __grid_constant__ GemmParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int nkc = (p.r + kGK - 1) / kGK;   // chunks of r
    const int ksteps = p.r / 16;              // 16-wide MMA k-steps
    const int nblk = p.n / kGN;               // column blocks of out
    const int msub = p.msub;
    uint8_t* a_s = smem;                      // msub x nkc chunks of the C tiles
    const int kStages = p.stages;
    uint8_t* b_s = smem + msub * nkc * kChunk;   // kStages chunks of U
    uint64_t* bars = reinterpret_cast<uint64_t*>(b_s + kStages * kChunk);
    uint64_t* a_full = bars;                  // the C tile landed            [TMA tx]
    uint64_t* full = bars + 1;                // ring slot s holds its chunk  [TMA tx]
    uint64_t* empty = full + kMaxStages;      // ring slot s consumed         [commit]
    uint64_t* acc_full = empty + kMaxStages;  // accumulator b complete       [commit]
    uint64_t* acc_empty = acc_full + 2;       // accumulator b read out       [256 arrivals]
    uint64_t* drain = acc_empty + 2;          // every MMA of the CTA done    [commit]
    volatile int* abort_flag = reinterpret_cast<volatile int*>(drain + 1);
    uint32_t* tmem_base_s = reinterpret_cast<uint32_t*>(drain + 2);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row0 = blockIdx.x * kGM * msub;
    // the CTAs take the column blocks in rotated orders, so that they do not all read the
    // same rows of U (held by the same few L2 slices) at the same time
    auto col_block = [&](int nb) { return (nb + blockIdx.x) % nblk; };
    if (threadIdx.x == 0) {
        ptx::mbar_init(a_full, 1);
        for (int s = 0; s < kStages; ++s) {
            ptx::mbar_init(&full[s], 1);
            ptx::mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(&acc_full[b], 1);
            ptx::mbar_init(&acc_empty[b], 256);
        }
        ptx::mbar_init(drain, 1);
        *abort_flag = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 1) ptx::tmem_alloc(tmem_base_s, 4 * kGN);
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
            ptx::mbar_expect_tx(a_full, msub * nkc * kChunk);
            for (int m = 0; m < msub; ++m)
                for (int c = 0; c < nkc; ++c)
                    ptx::tma_load_2d(a_s + (m * nkc + c) * kChunk, &p.tmC, c * kGK, row0 + m * kGM, a_full);
            int it = 0;
            for (int nb = 0; nb < nblk && !*abort_flag; ++nb)
                for (int c = 0; c < nkc; ++c, ++it) {
                    const int s = it % kStages;
                    if (it >= kStages) ptx::mbar_wait(&empty[s], (uint32_t)((it / kStages) - 1) & 1u, abort_flag);
                    ptx::mbar_expect_tx(&full[s], kChunk);
                    ptx::tma_load_2d(b_s + s * kChunk, &p.tmU, c * kGK, col_block(nb) * kGN, &full[s]);
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
                // accumulator buf: msub blocks of kGN columns, one per C tile
                const uint32_t d = tmem + (uint32_t)(buf * 2 * kGN);
                for (int c = 0; c < nkc; ++c, ++it) {
                    const int s = it % kStages;
                    ptx::mbar_wait(&full[s], (uint32_t)(it / kStages) & 1u, abort_flag);
                    ptx::tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < kGK / 16; ++kk) {
                        if (c * (kGK / 16) + kk >= ksteps) break;
                        const uint64_t b = dB + (uint64_t)((s * kChunk + kk * 32) >> 4);
                        for (int m = 0; m < msub; ++m) {
                            const uint64_t a = dA + (uint64_t)((((m * nkc + c) * kChunk) + kk * 32) >> 4);
                            ptx::mma_bf16(d + (uint32_t)(m * kGN), a, b, idesc, (c | kk) != 0 ? 1u : 0u);
                        }
                    }
                    ptx::mma_commit(&empty[s]);
                }
                ptx::mma_commit(&acc_full[buf]);
            }
            ptx::mma_commit(drain);
        }
    } else {
        // ------------------------------------------------------------- write-out
        // warps 2-9: two warps per TMEM lane quadrant. A thread stores 64 contiguous bytes
        // of its row per load (whole 32-byte sectors).
        const int q4 = warp & 3;
        const int w2 = (warp - 2) >> 2;          // 0 or 1
        const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
        if (p.ratio > 0) {
            // beacon-key RoPE (one C tile): a column block is one KV head (d = 128); warp
            // half w2 rotates the pairs (i, i + 64) for i in [32 w2, 32 w2 + 32), holding the
            // row's cos / sin for them across all blocks
            const int row = q4 * 32 + lane;
            const bool row_ok = row0 + row < p.rows;
            __nv_bfloat16* orow = p.out + (size_t)(row0 + row) * p.n;
            const unsigned long long j = (unsigned long long)((row0 + row) % p.rows_per_b);
            const unsigned long long pos = j * (unsigned long long)p.ratio + (unsigned long long)(p.ratio - 1);
            float cs[32], sn[32];
#pragma unroll
            for (int k = 0; k < 32; ++k) {
                // the angle reduced to a signed fraction of a turn (exact 64-bit wrap-around)
                const long long frac = (long long)(pos * p.turn[w2 * 32 + k]);
                sincospif((float)frac * 1.0842021724855044e-19f, &sn[k], &cs[k]);   // x 2^-63: half-turns
            }
            for (int nb = 0; nb < nblk; ++nb) {
                const int buf = nb & 1;
                const bool ok = ptx::mbar_wait(&acc_full[buf], (uint32_t)(nb >> 1) & 1u, abort_flag);
                ptx::tc_fence_after();
                float x1[32], x2[32];
                ptx::tmem_ld32(tmem + lane_off + (uint32_t)(buf * 2 * kGN + w2 * 32), x1);
                ptx::tmem_ld32(tmem + lane_off + (uint32_t)(buf * 2 * kGN + 64 + w2 * 32), x2);
                ptx::tc_fence_before();
                ptx::mbar_arrive(&acc_empty[buf]);   // the accumulator may take the next block
                uint32_t pk1[16], pk2[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const float a0 = x1[2 * i] * cs[2 * i] - x2[2 * i] * sn[2 * i];
                    const float a1 = x1[2 * i + 1] * cs[2 * i + 1] - x2[2 * i + 1] * sn[2 * i + 1];
                    const float b0 = x2[2 * i] * cs[2 * i] + x1[2 * i] * sn[2 * i];
                    const float b1 = x2[2 * i + 1] * cs[2 * i + 1] + x1[2 * i + 1] * sn[2 * i + 1];
                    const float nan = __int_as_float(0x7fc00000);
                    const __nv_bfloat162 h1 = __floats2bfloat162_rn(ok ? a0 : nan, ok ? a1 : nan);
                    const __nv_bfloat162 h2 = __floats2bfloat162_rn(ok ? b0 : nan, ok ? b1 : nan);
                    pk1[i] = *reinterpret_cast<const uint32_t*>(&h1);
                    pk2[i] = *reinterpret_cast<const uint32_t*>(&h2);
                }
                if (row_ok) {
                    uint4* d1 = reinterpret_cast<uint4*>(orow + col_block(nb) * kGN + w2 * 32);
                    uint4* d2 = reinterpret_cast<uint4*>(orow + col_block(nb) * kGN + 64 + w2 * 32);
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        d1[k] = make_uint4(pk1[4 * k], pk1[4 * k + 1], pk1[4 * k + 2], pk1[4 * k + 3]);
                        d2[k] = make_uint4(pk2[4 * k], pk2[4 * k + 1], pk2[4 * k + 2], pk2[4 * k + 3]);
                    }
                }
            }
        } else {
            // with two C tiles each warp takes one tile's 32 rows, else one 64-column half
            const int m = msub == 2 ? w2 : 0;        // C tile
            const int c_lo = msub == 2 ? 0 : w2 * 64, c_n = msub == 2 ? kGN : 64;
            const int row = m * kGM + q4 * 32 + lane;
            const bool row_ok = row0 + row < p.rows;
            __nv_bfloat16* orow = p.out + (size_t)(row0 + row) * p.n;
            for (int nb = 0; nb < nblk; ++nb) {
                const int buf = nb & 1;
                const bool ok = ptx::mbar_wait(&acc_full[buf], (uint32_t)(nb >> 1) & 1u, abort_flag);
                ptx::tc_fence_after();
#pragma unroll 1
                for (int c32 = c_lo; c32 < c_lo + c_n; c32 += 32) {
                    float v[32];
                    ptx::tmem_ld32(tmem + lane_off + (uint32_t)(buf * 2 * kGN + m * kGN + c32), v);
                    uint32_t pk[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const __nv_bfloat162 h2 = ok ? __floats2bfloat162_rn(v[2 * i], v[2 * i + 1])
                                                     : __floats2bfloat162_rn(__int_as_float(0x7fc00000),
                                                                             __int_as_float(0x7fc00000));
                        pk[i] = *reinterpret_cast<const uint32_t*>(&h2);
                    }
                    if (row_ok) {
                        uint4* dst = reinterpret_cast<uint4*>(orow + col_block(nb) * kGN + c32);
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            dst[k] = make_uint4(pk[4 * k], pk[4 * k + 1], pk[4 * k + 2], pk[4 * k + 3]);
                    }
                }
                ptx::tc_fence_before();
                ptx::mbar_arrive(&acc_empty[buf]);   // the accumulator may take the next block
            }
        }
    }

    // ----------------------------------------------------------------- teardown
    ptx::tc_fence_before();
    __syncthreads();
    if (threadIdx.x == 0 && *abort_flag && p.aborts != nullptr) atomicAdd(p.aborts, 1ull);
    if (warp == 1) {
        ptx::tc_fence_after();
        if (lane == 0) {
            volatile int never = 0;
            ptx::mbar_wait(drain, 0, &never);   // every MMA of this CTA has completed
        }
        __syncwarp();
        ptx::tmem_dealloc(tmem, 4 * kGN);
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
                                    int rows, int n, int r, cudaStream_t st, int beacon_ratio, int rows_per_b,
                                    double rope_base) {
    if (rows <= 0 || n <= 0 || n % kGN != 0 || r < 16 || r % 16 != 0 || r > kMaxR) return cudaErrorInvalidValue;
    if (beacon_ratio > 0 && rows_per_b <= 0) return cudaErrorInvalidValue;
    GemmParams p;
    memset(&p, 0, sizeof(p));
    if (!make_map_2d(&p.tmC, C, r, rows) || !make_map_2d(&p.tmU, U, r, n)) return cudaErrorInvalidValue;
    p.out = out;
    p.aborts = abort_counter();
    p.rows = rows;
    p.n = n;
    p.r = r;
    p.ratio = beacon_ratio > 0 ? beacon_ratio : 0;
    p.rows_per_b = rows_per_b;
    if (p.ratio > 0) rope_turns(rope_base, kGN, p.turn);
    // shared memory: the C tiles, then ring slots of U. Two C tiles per CTA when they
    // leave the ring at least four slots (each U chunk then serves 256 rows, halving
    // the re-reads of U from L2), else one.
    const int nkc = (r + kGK - 1) / kGK;
    p.msub = p.ratio == 0 && 1024 + 2 * nkc * kChunk + 256 + 4 * kChunk <= kSmemMax ? 2 : 1;
    const int fixed = 1024 + p.msub * nkc * kChunk + 256;
    p.stages = std::min(kMaxStages, (kSmemMax - fixed) / kChunk);
    if (p.stages < 2) return cudaErrorInvalidValue;
    const size_t smem = (size_t)fixed + (size_t)p.stages * kChunk;
    static std::atomic<unsigned long long> attr_done{0};
    const cudaError_t e = set_max_smem_once((const void*)recon_gemm_kernel, kSmemMax, attr_done);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((rows + kGM * p.msub - 1) / (kGM * p.msub));
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

// SIMT float32 kernels of libslimkv: query RoPE + latent projection, split
// combine with the value up-projection (both also used by the tensor-core path),
// and a plain split-context decode plus reconstruction GEMM used for float32
// storage, d = 64, and as an independent GPU cross-check of the tensor-core path.
//
// Source of the arithmetic: "Can SlimKV compress KV cache jointly across tokens
// and features", section "Latent-space attention removes the rebuild step"
// ((Q' U_K) C_K^T scores, (A C_V) U_V^T values, query projection after GQA
// grouping, RoPE on all queries and on raw keys only).
#include <math.h>

#include "slimkv_internal.cuh"

namespace slimkv {

namespace {

template <typename Kern, typename... Args>
cudaError_t launch_ex(Kern kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t st, bool pdl,
                      Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// ---------------------------------------------------------------------------
// Query RoPE and latent projection. One CTA per (KV group g, batch element b):
// q_rot[b,h] = RoPE(q[b,h], q_pos[b]) for the heads of group g, and, when q_lat
// is given, q_lat[b,h,:] = q_rot[b,h,:] . U_K^(g) (the projection is taken after
// grouping, so U_K^(g) is read once for the G heads that share it).
// The RoPE angle q_pos * base^(-2i/d) is formed and rotated in double precision.
// ---------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(256) qproj_kernel(const T* __restrict__ q,
                                                     const T* __restrict__ U_K,
                                                     const int32_t* __restrict__ q_pos,
                                                     float* __restrict__ q_rot,
                                                     float* __restrict__ q_lat, int Hq, int Hkv,
                                                     int d, int r_k, double base) {
    extern __shared__ float qr_s[];  // [G][d]
    pdl_trigger();
    const int g = blockIdx.x, b = blockIdx.y;
    const int G = Hq / Hkv;
    const int half = d >> 1;
    const double pos = (double)q_pos[b];
    for (int idx = threadIdx.x; idx < G * half; idx += blockDim.x) {
        const int hl = idx / half, i = idx - hl * half;
        const int h = g * G + hl;
        const double theta = pow(base, -2.0 * (double)i / (double)d);
        double sn, cs;
        sincos(pos * theta, &sn, &cs);
        const T* qh = q + ((size_t)b * Hq + h) * d;
        const double x1 = (double)to_f(qh[i]), x2 = (double)to_f(qh[i + half]);
        qr_s[hl * d + i] = (float)(x1 * cs - x2 * sn);
        qr_s[hl * d + i + half] = (float)(x2 * cs + x1 * sn);
    }
    __syncthreads();
    // the previous call's kernels may still read q_rot / q_lat of this workspace
    pdl_wait();
    for (int idx = threadIdx.x; idx < G * d; idx += blockDim.x) {
        const int hl = idx / d, i = idx - hl * d;
        q_rot[((size_t)b * Hq + g * G + hl) * d + i] = qr_s[idx];
    }
    if (q_lat == nullptr) return;
    for (int h0 = 0; h0 < G; h0 += 8) {
        const int nh = min(8, G - h0);
        for (int j = threadIdx.x; j < r_k; j += blockDim.x) {
            float acc[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) acc[k] = 0.f;
            const T* u = U_K + (size_t)g * d * r_k + j;
            for (int i = 0; i < d; ++i) {
                const float uv = to_f(u[(size_t)i * r_k]);
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    if (k < nh) acc[k] = fmaf(qr_s[(h0 + k) * d + i], uv, acc[k]);
            }
#pragma unroll
            for (int k = 0; k < 8; ++k)
                if (k < nh) q_lat[((size_t)b * Hq + g * G + h0 + k) * r_k + j] = acc[k];
        }
    }
}

// ---------------------------------------------------------------------------
// SIMT split decode. One CTA per (item, head). An item is a run of at most
// rpi rows of one segment. For each row j the CTA forms the log2-domain score
// s_j = scale*log2e * (query . key_j), keeps a running max m and sum l, and
// accumulates acc = sum_j exp2(s_j - m) value_j. Latent rows: key C_K[b,j],
// value C_V[b,j], query q_lat[b,h]. Raw rows: key K[b,t,g], value V[b,t,g],
// query q_rot[b,h].
// ---------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(128) simt_decode_kernel(SimtDecodeArgs a) {
    __shared__ float q_s[kMaxRank];
    __shared__ float p_s[128];
    __shared__ float red[4];
    const int item = blockIdx.x, h = blockIdx.y, tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    const int per_b = a.nit_L + a.nit_R0 + a.nit_R1;
    const int b = item / per_b;
    int k = item - b * per_b;
    const int G = a.Hq / a.Hkv, g = h / G;
    const T* Kp;
    const T* Vp;
    const float* qv;
    size_t ks, vs;
    int Dk, Dv, n_rows, rpi, kind;
    if (k < a.nit_L) {
        kind = 0;
        Kp = (const T*)a.C_K + (size_t)b * a.N_b * a.r_k;
        Vp = (const T*)a.C_V + (size_t)b * a.N_b * a.r_v;
        ks = a.r_k;
        vs = a.r_v;
        Dk = a.r_k;
        Dv = a.r_v;
        n_rows = a.N_b;
        rpi = a.rpi_L;
        qv = a.q_lat + ((size_t)b * a.Hq + h) * a.r_k;
    } else {
        k -= a.nit_L;
        int W = a.W0;
        const T* K = (const T*)a.K0;
        const T* V = (const T*)a.V0;
        if (k >= a.nit_R0) {
            k -= a.nit_R0;
            W = a.W1;
            K = (const T*)a.K1;
            V = (const T*)a.V1;
        }
        kind = 1;
        Kp = K + ((size_t)b * W * a.Hkv + g) * a.d;
        Vp = V + ((size_t)b * W * a.Hkv + g) * a.d;
        ks = vs = (size_t)a.Hkv * a.d;
        Dk = Dv = a.d;
        n_rows = W;
        rpi = a.rpi_R;
        qv = a.q_rot + ((size_t)b * a.Hq + h) * a.d;
    }
    const int row0 = k * rpi, row1 = min(n_rows, row0 + rpi);
    for (int i = tid; i < Dk; i += 128) q_s[i] = qv[i];
    __syncthreads();

    float m = -INFINITY, l = 0.f;
    float acc[kMaxRank / 128];
#pragma unroll
    for (int e = 0; e < kMaxRank / 128; ++e) acc[e] = 0.f;

    for (int c0 = row0; c0 < row1; c0 += 128) {
        const int j = c0 + tid;
        float s = -INFINITY;
        if (j < row1) {
            const T* kr = Kp + (size_t)j * ks;
            float dot = 0.f;
            for (int i = 0; i < Dk; ++i) dot = fmaf(q_s[i], to_f(kr[i]), dot);
            s = dot * a.scale_log2;
        }
        float cm = warp_max(s);
        if (lane == 0) red[warp] = cm;
        __syncthreads();
        cm = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
        __syncthreads();
        const float m_new = fmaxf(m, cm);  // finite: row c0 is valid
        const float alpha = exp2f(m - m_new);
        const float p = (j < row1) ? exp2f(s - m_new) : 0.f;
        p_s[tid] = p;
        float ps = warp_sum(p);
        if (lane == 0) red[warp] = ps;
        __syncthreads();
        ps = red[0] + red[1] + red[2] + red[3];
        l = l * alpha + ps;
        const int nv = min(128, row1 - c0);
#pragma unroll
        for (int e = 0; e < kMaxRank / 128; ++e) {
            const int col = tid + e * 128;
            if (col < Dv) {
                float v = acc[e] * alpha;
                const T* vp = Vp + (size_t)c0 * vs + col;
                for (int t = 0; t < nv; ++t) v = fmaf(p_s[t], to_f(vp[(size_t)t * vs]), v);
                acc[e] = v;
            }
        }
        m = m_new;
        __syncthreads();
    }
    const int slot = item;
    if (tid == 0) {
        a.ml[((size_t)slot * 2 + 0) * a.Hq + h] = m;
        a.ml[((size_t)slot * 2 + 1) * a.Hq + h] = l;
        if (h == 0) a.kind[slot] = kind;
    }
#pragma unroll
    for (int e = 0; e < kMaxRank / 128; ++e) {
        const int col = tid + e * 128;
        if (col < Dv) a.acc[((size_t)slot * a.Hq + h) * a.Dmax + col] = acc[e];
    }
}

// ---------------------------------------------------------------------------
// Split combine fused with the value up-projection. One CTA per (KV group g,
// batch element b), 128 threads. For each head h of the group it merges the
// partials of batch b by their log2-domain maxima:
//   M = max_s m_s, w_s = exp2(m_s - M), L = sum_s w_s l_s,
//   z = sum_{latent s} w_s acc_s (latent, r_v wide), y = sum_{raw s} w_s acc_s,
//   out[b,h,:] = (z . U_V^(g)T + y) / L.
// ---------------------------------------------------------------------------
constexpr int kCombHeads = 8;

template <typename T>
__global__ void __launch_bounds__(128) combine_kernel(CombineArgs a) {
    __shared__ float z_s[kCombHeads][kMaxRank];
    __shared__ float y_s[kCombHeads][128];
    __shared__ float M_s[kCombHeads], L_s[kCombHeads];
    pdl_trigger();
    const int g = blockIdx.x, b = blockIdx.y;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int G = a.Hq / a.Hkv;
    const bool latent = a.U_V != nullptr;
    pdl_wait();
    const int s0 = a.slot_begin[b], s1 = a.slot_begin[b + 1];
    for (int h0 = 0; h0 < G; h0 += kCombHeads) {
        const int nh = min(kCombHeads, G - h0);
        // per-head max and weighted sum, one warp per head
        for (int k = warp; k < nh; k += 4) {
            const int h = g * G + h0 + k;
            float M = -INFINITY;
            for (int s = s0 + lane; s < s1; s += 32) M = fmaxf(M, a.ml[((size_t)s * 2) * a.Hq + h]);
            M = warp_max(M);
            float L = 0.f;
            for (int s = s0 + lane; s < s1; s += 32) {
                const float ms = a.ml[((size_t)s * 2) * a.Hq + h];
                const float ls = a.ml[((size_t)s * 2 + 1) * a.Hq + h];
                L += (ls != 0.f) ? exp2f(ms - M) * ls : 0.f;   // a NaN partial poisons L
            }
            L = warp_sum(L);
            if (lane == 0) {
                M_s[k] = M;
                L_s[k] = L;
            }
        }
        __syncthreads();
        // weighted sums of the accumulators
        for (int k = 0; k < nh; ++k) {
            const int h = g * G + h0 + k;
            const float M = M_s[k];
            if (latent) {
                for (int j = tid; j < a.r_v; j += 128) {
                    float z = 0.f;
                    for (int s = s0; s < s1; ++s) {
                        if (a.kind[s] != 0) continue;
                        const float ls = a.ml[((size_t)s * 2 + 1) * a.Hq + h];
                        if (ls == 0.f) continue;
                        const float w = exp2f(a.ml[((size_t)s * 2) * a.Hq + h] - M);
                        z = fmaf(w, a.acc[((size_t)s * a.Hq + h) * a.Dmax + j], z);
                    }
                    z_s[k][j] = z;
                }
            }
            for (int i = tid; i < a.d; i += 128) {
                float y = 0.f;
                for (int s = s0; s < s1; ++s) {
                    if (a.kind[s] != 1) continue;
                    const float ls = a.ml[((size_t)s * 2 + 1) * a.Hq + h];
                    if (ls == 0.f) continue;
                    const float w = exp2f(a.ml[((size_t)s * 2) * a.Hq + h] - M);
                    y = fmaf(w, a.acc[((size_t)s * a.Hq + h) * a.Dmax + i], y);
                }
                y_s[k][i] = y;
            }
        }
        __syncthreads();
        // out row i of head k: (z_k . U_V^(g)[i,:] + y_k[i]) / L_k; one warp per row
        for (int i = warp; i < a.d; i += 4) {
            float part[kCombHeads];
#pragma unroll
            for (int k = 0; k < kCombHeads; ++k) part[k] = 0.f;
            if (latent) {
                const T* u = (const T*)a.U_V + ((size_t)g * a.d + i) * a.r_v;
                for (int j = lane; j < a.r_v; j += 32) {
                    const float uv = to_f(u[j]);
#pragma unroll
                    for (int k = 0; k < kCombHeads; ++k)
                        if (k < nh) part[k] = fmaf(z_s[k][j], uv, part[k]);
                }
            }
#pragma unroll
            for (int k = 0; k < kCombHeads; ++k) {
                if (k < nh) {
                    const float v = warp_sum(part[k]);
                    if (lane == 0) {
                        const int h = g * G + h0 + k;
                        a.out[((size_t)b * a.Hq + h) * a.d + i] = (v + y_s[k][i]) / L_s[k];
                    }
                }
            }
        }
        __syncthreads();
    }
}

// ---------------------------------------------------------------------------
// SIMT reconstruction GEMM: out[i, n] = sum_k C[i, k] U[n, k] (row-major,
// out [rows, n_cols] in the storage type). 32x32 output tile per CTA.
// ---------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(256) simt_reconstruct_kernel(const T* __restrict__ C,
                                                                const T* __restrict__ U,
                                                                T* __restrict__ out, int rows,
                                                                int n_cols, int r) {
    __shared__ float cs[32][33];
    __shared__ float us[32][33];
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;  // 32 x 8
    const int i0 = blockIdx.y * 32, n0 = blockIdx.x * 32;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    for (int k0 = 0; k0 < r; k0 += 32) {
        for (int rr = ty; rr < 32; rr += 8) {
            const int i = i0 + rr, n = n0 + rr, kk = k0 + tx;
            cs[rr][tx] = (i < rows && kk < r) ? to_f(C[(size_t)i * r + kk]) : 0.f;
            us[rr][tx] = (n < n_cols && kk < r) ? to_f(U[(size_t)n * r + kk]) : 0.f;
        }
        __syncthreads();
#pragma unroll 8
        for (int kk = 0; kk < 32; ++kk) {
            const float u = us[tx][kk];
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[e] = fmaf(cs[ty + 8 * e][kk], u, acc[e]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const int i = i0 + ty + 8 * e, n = n0 + tx;
        if (i < rows && n < n_cols) out[(size_t)i * n_cols + n] = from_f<T>(acc[e]);
    }
}

}  // namespace

template <typename T>
cudaError_t launch_qproj(const T* q, const T* U_K, const int32_t* q_pos, float* q_rot,
                         float* q_lat, int B, int Hq, int Hkv, int d, int r_k, double base,
                         cudaStream_t st, bool pdl) {
    const int G = Hq / Hkv;
    const size_t smem = (size_t)G * d * sizeof(float);
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(qproj_kernel<T>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    return launch_ex(qproj_kernel<T>, dim3(Hkv, B), dim3(256), smem, st, pdl, q, U_K, q_pos, q_rot,
                     q_lat, Hq, Hkv, d, r_k, base);
}

template <typename T>
cudaError_t launch_simt_decode(const SimtDecodeArgs& a, cudaStream_t st) {
    const int items = a.B * (a.nit_L + a.nit_R0 + a.nit_R1);
    simt_decode_kernel<T><<<dim3(items, a.Hq), 128, 0, st>>>(a);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_combine(const CombineArgs& a, cudaStream_t st, bool pdl) {
    return launch_ex(combine_kernel<T>, dim3(a.Hkv, a.B), dim3(128), 0, st, pdl, a);
}

template <typename T>
cudaError_t launch_simt_reconstruct(const T* C, const T* U, T* out, int rows, int n, int r,
                                    cudaStream_t st) {
    dim3 grid((n + 31) / 32, (rows + 31) / 32);
    simt_reconstruct_kernel<T><<<grid, 256, 0, st>>>(C, U, out, rows, n, r);
    return cudaGetLastError();
}

#define SLIMKV_INST(T)                                                                           \
    template cudaError_t launch_qproj<T>(const T*, const T*, const int32_t*, float*, float*, int, \
                                         int, int, int, int, double, cudaStream_t, bool);         \
    template cudaError_t launch_simt_decode<T>(const SimtDecodeArgs&, cudaStream_t);              \
    template cudaError_t launch_combine<T>(const CombineArgs&, cudaStream_t, bool);               \
    template cudaError_t launch_simt_reconstruct<T>(const T*, const T*, T*, int, int, int,        \
                                                    cudaStream_t);
SLIMKV_INST(float)
SLIMKV_INST(__nv_bfloat16)
#undef SLIMKV_INST

}  // namespace slimkv

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

#include <algorithm>

#include "slimkv_internal.cuh"
#include "tc_ptx.cuh"

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

// 16-byte asynchronous global -> shared copy (completion via cp_async_wait_all).
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(ptx::smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }
// Pull `bytes` (a multiple of 16, 16-byte aligned) of global memory into L2.
__device__ __forceinline__ void prefetch_l2(const void* src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// 16-byte vector of storage elements: 8 bf16 or 4 float32.
template <typename T> struct Vec16;
template <> struct Vec16<__nv_bfloat16> {
    static constexpr int N = 8;
    static __device__ __forceinline__ void to_f(const uint4& v, float* out) {
        const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 f = __bfloat1622float2(p[i]);
            out[2 * i] = f.x;
            out[2 * i + 1] = f.y;
        }
    }
};
template <> struct Vec16<float> {
    static constexpr int N = 4;
    static __device__ __forceinline__ void to_f(const uint4& v, float* out) {
        out[0] = __uint_as_float(v.x);
        out[1] = __uint_as_float(v.y);
        out[2] = __uint_as_float(v.z);
        out[3] = __uint_as_float(v.w);
    }
};

// ---------------------------------------------------------------------------
// Query RoPE and latent projection, "Latent-space attention removes the rebuild
// step": RoPE stays on every query, and the beacon query is projected into the
// latent space per GQA group, q_lat[b,h,:] = RoPE(q[b,h]) . U_K^(g) (the
// projection is taken after grouping, so U_K^(g) serves the G heads of group g).
//
// Grid (Hkv, blocks of 32 latent columns, row blocks). A row is one (batch
// element, head of group g) pair; a CTA holds at most 16 rows. The rotation angle
// p * theta_i is reduced modulo one turn exactly with 64-bit fixed-point arithmetic
// (turn[i] = theta_i / 2pi), then sin/cos of the reduced angle are taken in float32;
// every output is scaled by scale * log2(e).
//
// The kernel is small (128 threads, at most 25 KB of shared memory for float32
// storage, 16 KB for bf16) so that its CTAs fit on an SM next to a decode CTA.
//
// Ordering with neighbouring kernels: only the U_K block (a weight) is read before
// the grid-dependency wait; q and q_pos, which the preceding kernel may write, are
// read after it. Dependents are released at once: the decode kernel reads only its
// cache operands before its own wait (and a call's cache operands are never written
// by the kernels of the call before it).
// ---------------------------------------------------------------------------
constexpr int kQpRows = 16;
constexpr int kQpCols = 32;
constexpr int kQpThreads = 128;

template <typename T>
__global__ void __launch_bounds__(kQpThreads) qproj_kernel(const __grid_constant__ QprojArgs a) {
    // query rows, rotated and scaled (row stride padded by 4 floats)
    __shared__ __align__(16) float qr_s[kQpRows][128 + 4];
    __shared__ __align__(16) T u_s[128][kQpCols];   // U_K^(g) column block
    constexpr int VN = Vec16<T>::N;
    const int g = blockIdx.x, cb = blockIdx.y, rb = blockIdx.z;
    const int tid = threadIdx.x;
    const int G = a.Hq / a.Hkv, d = a.d, half = d >> 1;
    // rows of this block: r = r0 + rl (rl < nr), batch element r / G, head g * G + r % G
    const int r0 = rb * kQpRows, nr = min(kQpRows, a.B * G - r0);
    const bool proj = a.U_K != nullptr;

    // the U_K column block: a weight, copied before the dependency wait
    if (proj) {
        constexpr int cpr = kQpCols / VN;   // 16-byte chunks per row of the block
        for (int idx = tid; idx < d * cpr; idx += kQpThreads) {
            const int i = idx / cpr, e = (idx - i * cpr) * VN;
            cp_async16(&u_s[i][e], (const T*)a.U_K + ((size_t)g * d + i) * a.r_k + cb * kQpCols + e);
        }
        cp_async_commit();
    }
    pdl_trigger();
    pdl_wait();       // q, q_pos and this workspace are free to read / write from here

    // load, rotate and scale the query rows: item = (row, VN-wide chunk of the first
    // half); the thread loads both halves of the chunk and rotates them in registers
    const int cph = half / VN;   // chunks per half row
    for (int idx = tid; idx < nr * cph; idx += kQpThreads) {
        const int rl = idx / cph, e = (idx - rl * cph) * VN;
        const int r = r0 + rl, b = r / G, h = g * G + (r - b * G);
        const T* src = (const T*)a.q + ((size_t)b * a.Hq + h) * d;
        const uint4 v1 = *reinterpret_cast<const uint4*>(src + e);
        const uint4 v2 = *reinterpret_cast<const uint4*>(src + half + e);
        const unsigned long long pos = (unsigned long long)(long long)a.q_pos[b];
        float x1[VN], x2[VN];
        Vec16<T>::to_f(v1, x1);
        Vec16<T>::to_f(v2, x2);
#pragma unroll
        for (int k = 0; k < VN; ++k) {
            // cos / sin of p * theta_i: the angle reduced to a signed fraction of a turn
            // (exact 64-bit wrap-around), then sin / cos in float32
            const long long frac = (long long)(pos * a.turn[e + k]);
            float sn, cs;
            sincospif((float)frac * 1.0842021724855044e-19f, &sn, &cs);   // x 2^-63: half-turns
            qr_s[rl][e + k] = (x1[k] * cs - x2[k] * sn) * a.scale_log2;
            qr_s[rl][half + e + k] = (x2[k] * cs + x1[k] * sn) * a.scale_log2;
        }
    }
    if (proj) cp_async_wait_all();
    __syncthreads();

    // batch elements whose head 0 is a row of this block write the zero rows of the
    // absent heads (Hq <= h < NP) of their images (raw image: by the first column block)
    const int b_first = (r0 + G - 1) / G, b_end = (r0 + nr + G - 1) / G;
    const int npad = a.NP - a.Hq;
    if (cb == 0) {
        if (a.q_rot != nullptr) {
            for (int idx = tid; idx < nr * (d / 4); idx += kQpThreads) {
                const int rl = idx / (d / 4), e = (idx - rl * (d / 4)) * 4;
                const int r = r0 + rl, b = r / G, h = g * G + (r - b * G);
                *reinterpret_cast<float4*>(a.q_rot + ((size_t)b * a.Hq + h) * d + e) =
                    *reinterpret_cast<const float4*>(&qr_s[rl][e]);
            }
        }
        if (a.raw_img != nullptr) {
            // raw image of b: rows [0, NP) high, [NP, 2 NP) low parts of every head
            const size_t ib = raw_img_bytes(a.NP, d);
            const int units = d / 8;
            for (int idx = tid; idx < nr * units; idx += kQpThreads) {
                const int rl = idx / units, u = idx - rl * units;
                const int r = r0 + rl, b = r / G, h = g * G + (r - b * G);
                uint8_t* img = a.raw_img + (size_t)b * ib;
                const float* src = &qr_s[rl][u * 8];
                uint32_t hi[4], lo[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const __nv_bfloat162 h2 = __floats2bfloat162_rn(src[2 * k], src[2 * k + 1]);
                    const float2 hf = __bfloat1622float2(h2);
                    const __nv_bfloat162 l2 = __floats2bfloat162_rn(src[2 * k] - hf.x, src[2 * k + 1] - hf.y);
                    hi[k] = *reinterpret_cast<const uint32_t*>(&h2);
                    lo[k] = *reinterpret_cast<const uint32_t*>(&l2);
                }
                *reinterpret_cast<uint4*>(img + ptx::sw128_offset(h, u * 8, 2 * a.NP)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                *reinterpret_cast<uint4*>(img + ptx::sw128_offset(a.NP + h, u * 8, 2 * a.NP)) =
                    make_uint4(lo[0], lo[1], lo[2], lo[3]);
            }
            if (g == 0 && npad > 0) {
                const int n = (b_end - b_first) * 2 * npad * units;
                for (int idx = tid; idx < n; idx += kQpThreads) {
                    const int bl = idx / (2 * npad * units), rem = idx - bl * 2 * npad * units;
                    const int pr = rem / units, u = rem - pr * units;
                    const int row = pr < npad ? a.Hq + pr : a.NP + a.Hq + (pr - npad);
                    uint8_t* img = a.raw_img + (size_t)(b_first + bl) * ib;
                    *reinterpret_cast<uint4*>(img + ptx::sw128_offset(row, u * 8, 2 * a.NP)) = make_uint4(0u, 0u, 0u, 0u);
                }
            }
        }
    }
    if (!proj) return;
    if (a.lat_img != nullptr && g == 0 && npad > 0) {
        const int n = (b_end - b_first) * npad * kQpCols;
        for (int idx = tid; idx < n; idx += kQpThreads) {
            const int bl = idx / (npad * kQpCols), rem = idx - bl * npad * kQpCols;
            const int h = a.Hq + rem / kQpCols, col = cb * kQpCols + rem % kQpCols;
            uint8_t* img = a.lat_img + (size_t)(b_first + bl) * lat_img_bytes(a.NP, a.r_k);
            *reinterpret_cast<__nv_bfloat16*>(img + ptx::sw128_offset(h, col, a.NP)) = __float2bfloat16_rn(0.f);
        }
    }
    // q_lat block: 16 rows x 32 columns; thread = (column c, rows 4 rg .. 4 rg + 3)
    const int c = tid & (kQpCols - 1), rg = tid / kQpCols;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
    for (int i = 0; i < d; i += 4) {
        const float u0 = to_f(u_s[i][c]), u1 = to_f(u_s[i + 1][c]), u2 = to_f(u_s[i + 2][c]),
                    u3 = to_f(u_s[i + 3][c]);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float4 qv = *reinterpret_cast<const float4*>(&qr_s[rg * 4 + k][i]);
            acc[k] = fmaf(qv.x, u0, fmaf(qv.y, u1, fmaf(qv.z, u2, fmaf(qv.w, u3, acc[k]))));
        }
    }
    const int col = cb * kQpCols + c;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int rl = rg * 4 + k;
        if (rl < nr) {
            const int r = r0 + rl, b = r / G, h = g * G + (r - b * G);
            if (a.q_lat != nullptr) a.q_lat[((size_t)b * a.Hq + h) * a.r_k + col] = acc[k];
            if (a.lat_img != nullptr) {
                uint8_t* img = a.lat_img + (size_t)b * lat_img_bytes(a.NP, a.r_k);
                *reinterpret_cast<__nv_bfloat16*>(img + ptx::sw128_offset(h, col, a.NP)) = __float2bfloat16_rn(acc[k]);
            }
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
    int Dk, Dv, n_rows, rpi;
    if (k < a.nit_L) {
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
            s = dot;   // the query carries scale * log2(e)
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
    }
#pragma unroll
    for (int e = 0; e < kMaxRank / 128; ++e) {
        const int col = tid + e * 128;
        if (col < Dv) a.acc[((size_t)slot * a.Hq + h) * a.Dmax + col] = acc[e];
    }
}

// ---------------------------------------------------------------------------
// Split combine fused with the value up-projection ("(A C_V) U_V^T": the latent
// aggregate is up-projected once, after all beacon splits are merged). One CTA per
// (batch element b, KV group g and chunk of at most 4 of its heads). The partials of
// b cover every head; latent ones (r_v wide) occupy slots [slot_begin[b],
// slot_mid[b]), raw ones (d wide) [slot_mid[b], slot_begin[b+1]). They are merged by
// their log2-domain maxima:
//   M = max_s m_s, w_s = exp2(m_s - M), L = sum_s w_s l_s,
//   z = sum_{latent s} w_s acc_s (r_v wide), y = sum_{raw s} w_s acc_s (d wide),
//   out[b,h,i] = (z . U_V^(g)[i, :] + y[i]) / L.
// A partial with l = 0 covered no key of that head and is skipped; a NaN l (a decode
// CTA that gave up on a wait) propagates into the output.
//
// The kernel is latency-bound: it is laid out as three rounds of independent loads
// (the (m, l) pairs, then every partial value the merge needs, then U_V^(g), whose
// rows are pulled into L2 before the dependency wait), so that each round costs one
// memory round trip. It is small (256 threads, a few KB of shared memory) so that
// its CTAs fit on an SM next to a decode CTA.
// ---------------------------------------------------------------------------
constexpr int kCombThreads = 256;
constexpr int kCombHeads = 4;    // heads per CTA
constexpr int kCombBatch = 8;    // slots whose loads are in flight together
constexpr int kCombWeightRegs = 2;   // slots per lane whose (m, l) stay in registers

template <typename T>
__global__ void __launch_bounds__(kCombThreads) combine_kernel(const __grid_constant__ CombineArgs a) {
    extern __shared__ __align__(16) float dyn[];
    __shared__ float L_s[kCombHeads];
    const int b = blockIdx.x;
    const int G = a.Hq / a.Hkv, nhc = (G + kCombHeads - 1) / kCombHeads;
    const int g = blockIdx.y / nhc, hc = blockIdx.y - g * nhc;
    const int h0 = g * G + hc * kCombHeads, nh = min(kCombHeads, G - hc * kCombHeads);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int d = a.d;
    const int s0 = a.slot_begin[b], sm = a.slot_mid[b], s1 = a.slot_begin[b + 1];
    const int ns = s1 - s0, nl = sm - s0, nr = s1 - sm;
    const bool latent = a.U_V != nullptr;
    float* w_s = dyn;                                          // [ns][4] merge weights
    float* z_s = dyn + a.ns_max * kCombHeads;                  // [r_v][4] latent aggregate
    float* y_s = z_s + (latent ? a.r_v * kCombHeads : 0);      // [d][4] raw aggregate
    if (latent && tid < 2) {
        // U_V^(g): a weight, pulled into L2 before the dependency wait (two halves)
        const size_t half = (size_t)d * a.r_v * sizeof(T) / 2;
        prefetch_l2(reinterpret_cast<const char*>(a.U_V) + (size_t)g * d * a.r_v * sizeof(T) + tid * half,
                    (uint32_t)half);
    }
    pdl_trigger();
    pdl_wait();   // partials come from the decode kernel

    // round 1: merge weights of head h0 + warp over the slots of b; every lane loads its
    // (m, l) pairs once (up to kCombWeightRegs slots per lane stay in registers)
    if (warp < nh) {
        const int h = h0 + warp;
        constexpr int R = kCombWeightRegs;
        float mr[R], lr[R];
#pragma unroll
        for (int k = 0; k < R; ++k) {
            const int s = lane + 32 * k;
            mr[k] = s < ns ? a.ml[((size_t)(s0 + s) * 2) * a.Hq + h] : -INFINITY;
            lr[k] = s < ns ? a.ml[((size_t)(s0 + s) * 2 + 1) * a.Hq + h] : 0.f;
        }
        float M = -INFINITY;
#pragma unroll
        for (int k = 0; k < R; ++k)
            if (lr[k] != 0.f) M = fmaxf(M, mr[k]);   // a NaN (poisoned) l is kept
        for (int s = lane + 32 * R; s < ns; s += 32) {
            const float l = a.ml[((size_t)(s0 + s) * 2 + 1) * a.Hq + h];
            if (l != 0.f) M = fmaxf(M, a.ml[((size_t)(s0 + s) * 2) * a.Hq + h]);
        }
        M = warp_max(M);
        float L = 0.f;
#pragma unroll
        for (int k = 0; k < R; ++k) {
            const int s = lane + 32 * k;
            if (s < ns) {
                const float w = (lr[k] != 0.f) ? exp2f(mr[k] - M) : 0.f;
                w_s[s * kCombHeads + warp] = w;
                L = fmaf(w, lr[k], L);
            }
        }
        for (int s = lane + 32 * R; s < ns; s += 32) {
            const float m = a.ml[((size_t)(s0 + s) * 2) * a.Hq + h];
            const float l = a.ml[((size_t)(s0 + s) * 2 + 1) * a.Hq + h];
            const float w = (l != 0.f) ? exp2f(m - M) : 0.f;
            w_s[s * kCombHeads + warp] = w;
            L = fmaf(w, l, L);
        }
        L = warp_sum(L);
        if (lane == 0) L_s[warp] = L;
    }
    __syncthreads();
    // round 2: z (items of 4 latent columns x one head) and y (4 rows x one head);
    // every thread takes at most one item of each, loads batched over kCombBatch slots
    const size_t sstride = (size_t)a.Hq * a.Dmax;   // floats between consecutive slots
    auto merge = [&](int item, int first_slot, int nslot, int wbase) {
        const int col = (item >> 2) * 4, hh = item & 3;
        float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
        if (hh < nh) {
            const float* src = a.acc + ((size_t)first_slot * a.Hq + h0 + hh) * a.Dmax + col;
            for (int s = 0; s < nslot; s += kCombBatch) {
                float4 v[kCombBatch];
#pragma unroll
                for (int k = 0; k < kCombBatch; ++k)
                    v[k] = s + k < nslot ? *reinterpret_cast<const float4*>(src + (s + k) * sstride)
                                         : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int k = 0; k < kCombBatch; ++k) {
                    const float w = s + k < nslot ? w_s[(wbase + s + k) * kCombHeads + hh] : 0.f;
                    z.x = fmaf(w, v[k].x, z.x);
                    z.y = fmaf(w, v[k].y, z.y);
                    z.z = fmaf(w, v[k].z, z.z);
                    z.w = fmaf(w, v[k].w, z.w);
                }
            }
        }
        return z;
    };
    const int nz = latent ? a.r_v : 0;    // (r_v / 4) column quads x 4 heads
    const int ny = d;                     // (d / 4) row quads x 4 heads
    for (int it = tid; it < nz + ny; it += kCombThreads) {
        const bool zi = it < nz;
        const int item = zi ? it : it - nz;
        const float4 v = zi ? merge(item, s0, nl, 0) : merge(item, sm, nr, nl);
        float* dst = zi ? z_s : y_s;
        const int col = (item >> 2) * 4, hh = item & 3;
        dst[(col + 0) * kCombHeads + hh] = v.x;
        dst[(col + 1) * kCombHeads + hh] = v.y;
        dst[(col + 2) * kCombHeads + hh] = v.z;
        dst[(col + 3) * kCombHeads + hh] = v.w;
    }
    __syncthreads();
    // round 3: out[i] = (z . U_V^(g)[i, :] + y[i]) / L; thread = (row i, half jh of the
    // latent columns), the half row's U_V loads issued together
    for (int i2 = tid; i2 < 2 * d; i2 += kCombThreads) {
        const int i = i2 >> 1, jh = i2 & 1;
        float part[kCombHeads] = {0.f, 0.f, 0.f, 0.f};
        if (latent) {
            const int jn = a.r_v >> 1, j0 = jh * jn;
            const T* u = (const T*)a.U_V + ((size_t)g * d + i) * a.r_v + j0;
            const float4* z4 = reinterpret_cast<const float4*>(z_s) + j0;
            for (int jj = 0; jj < jn; jj += 64) {
                constexpr int VN = Vec16<T>::N;
                uint4 uv[64 / VN];
#pragma unroll
                for (int q = 0; q < 64 / VN; ++q)
                    uv[q] = jj + q * VN < jn ? *reinterpret_cast<const uint4*>(u + jj + q * VN) : make_uint4(0, 0, 0, 0);
#pragma unroll
                for (int q = 0; q < 64 / VN; ++q) {
                    float f[VN];
                    Vec16<T>::to_f(uv[q], f);
#pragma unroll
                    for (int e = 0; e < VN; ++e) {
                        if (jj + q * VN + e < jn) {
                            const float4 zz = z4[jj + q * VN + e];
                            part[0] = fmaf(zz.x, f[e], part[0]);
                            part[1] = fmaf(zz.y, f[e], part[1]);
                            part[2] = fmaf(zz.z, f[e], part[2]);
                            part[3] = fmaf(zz.w, f[e], part[3]);
                        }
                    }
                }
            }
        }
#pragma unroll
        for (int hh = 0; hh < kCombHeads; ++hh) part[hh] += __shfl_xor_sync(0xffffffffu, part[hh], 1);
        // the two threads of a row write two heads each
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const int hh = 2 * jh + k;
            if (hh < nh)
                a.out[((size_t)b * a.Hq + h0 + hh) * d + i] = (part[hh] + y_s[i * kCombHeads + hh]) / L_s[hh];
        }
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

void rope_turns(double base, int d, unsigned long long (&turn)[64]) {
    const long double two_pi = 6.283185307179586476925286766559L;
    for (int i = 0; i < 64; ++i) {
        turn[i] = 0;
        if (i < d / 2) {
            long double t = powl((long double)base, -2.0L * i / d) / two_pi;
            t -= floorl(t);
            turn[i] = (unsigned long long)(t * 18446744073709551616.0L + 0.5L);
        }
    }
}

template <typename T>
cudaError_t launch_qproj(const T* q, const T* U_K, const int32_t* q_pos, float* q_rot,
                         float* q_lat, int B, int Hq, int Hkv, int d, int r_k, double base,
                         float scale_log2, cudaStream_t st, bool pdl, uint8_t* lat_img,
                         uint8_t* raw_img, int NP) {
    QprojArgs a;
    a.lat_img = lat_img;
    a.raw_img = raw_img;
    a.NP = NP;
    a.q = q;
    a.U_K = U_K;
    a.q_pos = q_pos;
    a.q_rot = q_rot;
    a.q_lat = q_lat;
    a.B = B;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.d = d;
    a.r_k = r_k;
    a.rows = kQpRows;
    a.scale_log2 = scale_log2;
    rope_turns(base, d, a.turn);
    const int G = Hq / Hkv;
    const int row_blocks = (B * G + kQpRows - 1) / kQpRows;
    const int col_blocks = U_K ? r_k / kQpCols : 1;
    static std::atomic<unsigned long long> attr_done{0};
    const cudaError_t e = set_max_smem_once((const void*)qproj_kernel<T>, 0, attr_done);
    if (e != cudaSuccess) return e;
    return launch_ex(qproj_kernel<T>, dim3(Hkv, col_blocks, row_blocks), dim3(kQpThreads), 0, st, pdl, a);
}

template <typename T>
cudaError_t launch_simt_decode(const SimtDecodeArgs& a, cudaStream_t st) {
    const int items = a.B * (a.nit_L + a.nit_R0 + a.nit_R1);
    simt_decode_kernel<T><<<dim3(items, a.Hq), 128, 0, st>>>(a);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_combine(const CombineArgs& a, cudaStream_t st, bool pdl) {
    int ns_max = 0;
    for (int b = 0; b < a.B; ++b) ns_max = std::max(ns_max, a.slot_begin[b + 1] - a.slot_begin[b]);
    if (ns_max > kMaxSlotsPerB) return cudaErrorInvalidValue;
    CombineArgs b = a;
    b.ns_max = ns_max;
    const size_t smem = sizeof(float) * kCombHeads * ((size_t)ns_max + (a.U_V ? a.r_v : 0) + a.d);
    static std::atomic<unsigned long long> attr_done{0};
    const cudaError_t e = set_max_smem_once(
        (const void*)combine_kernel<T>, (int)(sizeof(float) * kCombHeads * (kMaxSlotsPerB + kMaxRank + 128)),
        attr_done);
    if (e != cudaSuccess) return e;
    const int G = a.Hq / a.Hkv, nhc = (G + kCombHeads - 1) / kCombHeads;
    return launch_ex(combine_kernel<T>, dim3(a.B, a.Hkv * nhc), dim3(kCombThreads), smem, st, pdl, b);
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
                                         int, int, int, int, double, float, cudaStream_t, bool,   \
                                         uint8_t*, uint8_t*, int);                                \
    template cudaError_t launch_simt_decode<T>(const SimtDecodeArgs&, cudaStream_t);              \
    template cudaError_t launch_combine<T>(const CombineArgs&, cudaStream_t, bool);               \
    template cudaError_t launch_simt_reconstruct<T>(const T*, const T*, T*, int, int, int,        \
                                                    cudaStream_t);
SLIMKV_INST(float)
SLIMKV_INST(__nv_bfloat16)
#undef SLIMKV_INST

}  // namespace slimkv

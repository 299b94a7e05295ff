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

// ---------------------------------------------------------------------------
// Query RoPE and latent projection, "Latent-space attention removes the rebuild
// step": RoPE stays on every query, and the beacon query is projected into the
// latent space per GQA group, q_lat[b,h,:] = RoPE(q[b,h]) . U_K^(g) (the
// projection is taken after grouping, so U_K^(g) serves the G heads of group g).
//
// Grid (Hkv, column blocks of 16 latent columns, row blocks). A row is one
// (batch element, head of group g) pair; a CTA holds at most 32 rows: `nbb`
// whole batch elements when G <= 32, else one 32-head chunk of one element.
// The rotation angle p * theta_i is reduced modulo one turn exactly with 64-bit
// fixed-point arithmetic (turn[i] = theta_i / 2pi), then sin/cos of the reduced
// angle are taken in float32; both outputs are scaled by scale * log2(e).
//
// Ordering with neighbouring kernels: only the U_K block (a weight) is read before
// the grid-dependency wait; q and q_pos, which the preceding kernel may write, are
// read after it, and dependents are released only after it, so a dependent kernel
// may read anything the preceding kernels wrote (the caches) without a wait of its own.
// ---------------------------------------------------------------------------
constexpr int kQpRows = 32;
constexpr int kQpCols = 32;
constexpr int kQpThreads = 256;
// Dynamic shared memory of the query projection when it is launched early behind a
// combine (it holds the U_K block; the rest is reserved, unused). Its CTAs are placed
// while the combine's CTAs still occupy the SMs, and by registers alone three of them
// would fit beside one combine CTA, so the block scheduler would stack them on a few
// SMs and the grid would end with those (measured: 1.6 us alone, up to 8 us stacked).
// With this reservation (plus the static rows) no SM takes two of them.
constexpr int kQpSpreadSmem = 112 * 1024;
constexpr int kQpUBytes = 128 * kQpCols * 4;   // the U_K column block (dynamic shared memory)

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

template <typename T>
__global__ void __launch_bounds__(kQpThreads) qproj_kernel(const __grid_constant__ QprojArgs a) {
    // query rows, rotated and scaled (row stride padded by 4 floats: the projection
    // reads two rows per warp, which then fall in different banks)
    __shared__ __align__(16) float qr_s[kQpRows][128 + 4];
    extern __shared__ __align__(16) float u_dyn[];
    float (*u_s)[kQpCols] = reinterpret_cast<float (*)[kQpCols]>(u_dyn);   // U_K^(g) column block [d][kQpCols]
    constexpr int VN = Vec16<T>::N;
    const int g = blockIdx.x, cb = blockIdx.y, rb = blockIdx.z;
    const int tid = threadIdx.x;
    const int G = a.Hq / a.Hkv, d = a.d, half = d >> 1;
    // rows of this block: batch elements [b0, b0 + nb) x heads-in-group [i0, i1)
    int b0, nb, i0, i1;
    if (a.hcn == 1) {
        b0 = rb * a.nbb;
        nb = min(a.nbb, a.B - b0);
        i0 = 0;
        i1 = G;
    } else {
        b0 = rb / a.hcn;
        nb = 1;
        i0 = (rb % a.hcn) * 32;
        i1 = min(G, i0 + 32);
    }
    const int ni = i1 - i0, rows = nb * ni;

    // the U_K column block: a weight, read before the dependency wait
    if (a.U_K != nullptr) {
        constexpr int upr = kQpCols / VN;   // vectors per row of the block
        for (int idx = tid; idx < d * upr; idx += kQpThreads) {
            const int i = idx / upr, e = (idx - i * upr) * VN;
            // columns past r_k (a last, partial block) read as zero
            const uint4 v = cb * kQpCols + e < a.r_k
                                ? *reinterpret_cast<const uint4*>((const T*)a.U_K + ((size_t)g * d + i) * a.r_k +
                                                                  cb * kQpCols + e)
                                : make_uint4(0u, 0u, 0u, 0u);
            float f[VN];
            Vec16<T>::to_f(v, f);
#pragma unroll
            for (int k = 0; k < VN; ++k) u_s[i][e + k] = f[k];
        }
    }
    pdl_wait();       // q, q_pos and this workspace are free to read / write from here
    pdl_trigger();

    // load, rotate and scale the query rows: item = (row, VN-wide chunk of the first
    // half); the thread loads both halves of the chunk and rotates them in registers
    const int cph = half / VN;   // chunks per half row
    for (int idx = tid; idx < rows * cph; idx += kQpThreads) {
        const int r = idx / cph, e = (idx - r * cph) * VN;
        const int bl = r / ni, h = g * G + i0 + (r - bl * ni);
        const T* src = (const T*)a.q + ((size_t)(b0 + bl) * a.Hq + h) * d;
        const uint4 v1 = *reinterpret_cast<const uint4*>(src + e);
        const uint4 v2 = *reinterpret_cast<const uint4*>(src + half + e);
        const unsigned long long pos = (unsigned long long)(long long)a.q_pos[b0 + bl];
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
            qr_s[r][e + k] = (x1[k] * cs - x2[k] * sn) * a.scale_log2;
            qr_s[r][half + e + k] = (x2[k] * cs + x1[k] * sn) * a.scale_log2;
        }
    }
    __syncthreads();
    if (cb == 0 && a.q_rot != nullptr) {
        for (int idx = tid; idx < rows * (d / 4); idx += kQpThreads) {
            const int r = idx / (d / 4), e = (idx - r * (d / 4)) * 4;
            const int bl = r / ni, h = g * G + i0 + (r - bl * ni);
            *reinterpret_cast<float4*>(a.q_rot + ((size_t)(b0 + bl) * a.Hq + h) * d + e) =
                *reinterpret_cast<const float4*>(&qr_s[r][e]);
        }
    }
    if (cb == 0 && a.raw_img != nullptr) {
        // raw image of (b, g): 32 rows x d, rows [0,16) high, [16,32) low parts of the
        // group's G (<= 16) heads; rows of absent heads are zero
        // rows of 128 columns: with d = 64 the columns past d are zero
        const size_t ib = raw_img_bytes(128);
        const int units = 128 / 8;
        for (int idx = tid; idx < nb * 16 * units; idx += kQpThreads) {
            const int bl = idx / (16 * units), rem = idx - bl * 16 * units;
            const int i = rem / units, u = rem - i * units;
            uint8_t* img = a.raw_img + ((size_t)(b0 + bl) * a.Hkv + g) * ib;
            uint32_t hi[4] = {0u, 0u, 0u, 0u}, lo[4] = {0u, 0u, 0u, 0u};
            if (i < G && u * 8 < d) {
                const float* src = &qr_s[bl * ni + i][u * 8];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const __nv_bfloat162 h2 = __floats2bfloat162_rn(src[2 * k], src[2 * k + 1]);
                    const float2 hf = __bfloat1622float2(h2);
                    const __nv_bfloat162 l2 = __floats2bfloat162_rn(src[2 * k] - hf.x, src[2 * k + 1] - hf.y);
                    hi[k] = *reinterpret_cast<const uint32_t*>(&h2);
                    lo[k] = *reinterpret_cast<const uint32_t*>(&l2);
                }
            }
            *reinterpret_cast<uint4*>(img + ptx::sw128_offset(i, u * 8, 32)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
            *reinterpret_cast<uint4*>(img + ptx::sw128_offset(16 + i, u * 8, 32)) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
        }
    }
    if (a.lat_img != nullptr && g == 0 && (a.hcn == 1 || rb % a.hcn == 0) && a.NP > a.Hq) {
        // rows of absent heads (Hq <= h < NP) of the latent image are zero, so that the
        // tensor-core path may treat every head column alike
        const int npad = a.NP - a.Hq;
        for (int idx = tid; idx < nb * npad * kQpCols; idx += kQpThreads) {
            const int bl = idx / (npad * kQpCols), rem = idx - bl * npad * kQpCols;
            const int h = a.Hq + rem / kQpCols, col = cb * kQpCols + rem % kQpCols;
            if (col >= a.r_k) continue;
            uint8_t* img = a.lat_img + (size_t)(b0 + bl) * lat_img_bytes(a.NP, a.r_k);
            *reinterpret_cast<__nv_bfloat16*>(img + ptx::sw128_offset(h, col, a.NP)) = __float2bfloat16_rn(0.f);
        }
    }
    if (a.U_K == nullptr) return;
    // q_lat block: 32 rows x kQpCols columns; thread = (column c, rows rg, rg + RG, ...)
    constexpr int RG = kQpThreads / kQpCols;     // row groups
    constexpr int RPT = kQpRows / RG;            // rows per thread
    const int c = tid & (kQpCols - 1), rg = tid / kQpCols;
    float acc[RPT];
#pragma unroll
    for (int k = 0; k < RPT; ++k) acc[k] = 0.f;
#pragma unroll 2
    for (int i = 0; i < d; i += 4) {
        const float u0 = u_s[i][c], u1 = u_s[i + 1][c], u2 = u_s[i + 2][c], u3 = u_s[i + 3][c];
#pragma unroll
        for (int k = 0; k < RPT; ++k) {
            const float4 q4 = *reinterpret_cast<const float4*>(&qr_s[rg + k * RG][i]);
            acc[k] = fmaf(q4.x, u0, fmaf(q4.y, u1, fmaf(q4.z, u2, fmaf(q4.w, u3, acc[k]))));
        }
    }
    const int col = cb * kQpCols + c;
#pragma unroll
    for (int k = 0; k < RPT; ++k) {
        const int r = rg + k * RG;
        const float v = acc[k];
        if (r < rows && col < a.r_k) {
            const int bl = r / ni, h = g * G + i0 + (r - bl * ni);
            if (a.q_lat != nullptr) a.q_lat[((size_t)(b0 + bl) * a.Hq + h) * a.r_k + col] = v;
            if (a.lat_img != nullptr) {
                uint8_t* img = a.lat_img + (size_t)(b0 + bl) * lat_img_bytes(a.NP, a.r_k);
                *reinterpret_cast<__nv_bfloat16*>(img + ptx::sw128_offset(h, col, a.NP)) = __float2bfloat16_rn(v);
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
            s = dot;   // the query carries scale * log2(e)
            if (a.alibi) {
                const long long qp = a.q_pos[b];
                const long long dk = kind == 0 ? (long long)j * a.ratio + a.ratio - 1 - qp
                                               : -((((qp - j) % n_rows) + n_rows) % n_rows);
                s = fmaf(a.slope_l2[h], (float)dk, s);
            }
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
// Split combine fused with the value up-projection ("(A C_V) U_V^T": the latent
// aggregate is up-projected once, after all beacon splits are merged). One CTA
// per (query head h, batch element b), g its KV group. The partials of batch b
// that cover head h (SlotKind) are merged by their log2-domain maxima:
//   M = max_s m_s, w_s = exp2(m_s - M), L = sum_s w_s l_s,
//   z = sum_{latent s} w_s acc_s (r_v wide), y = sum_{raw s} w_s acc_s (d wide),
//   out[b,h,:] = (z . U_V^(g)T + y) / L.
// Global loads are issued in independent batches so that the kernel costs a few
// memory round trips, not one per partial.
// ---------------------------------------------------------------------------
constexpr int kCombThreads = 256;
constexpr int kCombBatch = 16;
constexpr int kCombPrefetchCols = 256;   // latent columns of U_V staged before the wait (bf16)

// 16-byte asynchronous global -> shared copy (completion via cp_async_wait_all).
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(ptx::smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }
constexpr int kCombRowsPerWarp = 128 / (kCombThreads / 32);   // 16 output rows per warp (d <= 128)

template <typename T>
__global__ void __launch_bounds__(kCombThreads) combine_kernel(const __grid_constant__ CombineArgs a) {
    // per covering partial: slot, m, l (later the weight); latent and raw lists; then,
    // for bf16 storage, U_V^(g)[:, 0:256) staged by asynchronous copies
    extern __shared__ __align__(16) float dyn[];
    __shared__ __align__(16) float z_s[kMaxRank];
    __shared__ float y_s[128];
    __shared__ int n_lat_s, n_raw_s;
    __shared__ float L_s;
    const int h = blockIdx.x, b = blockIdx.y;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int G = a.Hq / a.Hkv, g = h / G;
    const bool latent = a.U_V != nullptr;
    constexpr int VN = Vec16<T>::N;
    const int nrow = (a.d + (kCombThreads / 32) - 1) / (kCombThreads / 32);

    const int s0 = a.slot_begin[b], ns = a.slot_begin[b + 1] - s0;
    // U_V^(g)[:, 0:256): a weight, copied before the dependency wait
    const bool prefetch = latent && VN == 8;
    T* u_stage = reinterpret_cast<T*>(dyn + ((6 * a.ns_max + 3) & ~3));
    if (prefetch) {
        const int cpr = min(a.r_v, kCombPrefetchCols) / 8;   // 16-byte chunks per row
        for (int idx = tid; idx < a.d * cpr; idx += kCombThreads) {
            const int i = idx / cpr, e = (idx - i * cpr) * 8;
            cp_async16(u_stage + i * kCombPrefetchCols + e, (const T*)a.U_V + ((size_t)g * a.d + i) * a.r_v + e);
        }
        cp_async_commit();
    }
    pdl_trigger();
    pdl_wait();   // partials come from the decode kernel

    int* lat_slot = reinterpret_cast<int*>(dyn);
    float* lat_m = dyn + ns;
    float* lat_l = dyn + 2 * ns;
    int* raw_slot = reinterpret_cast<int*>(dyn + 3 * ns);
    float* raw_m = dyn + 4 * ns;
    float* raw_l = dyn + 5 * ns;
    if (warp == 0) {
        // compact the partials that cover head h with their (m, l), one load each
        int nl = 0, nr = 0;
        float M = -INFINITY;
        for (int base = 0; base < ns; base += 32) {
            const int s = base + lane;
            int kd = -1;
            float m = -INFINITY, l = 0.f;
            if (s < ns) {
                kd = a.kind[s0 + s];
                m = a.ml[((size_t)(s0 + s) * 2) * a.Hq + h];
                l = a.ml[((size_t)(s0 + s) * 2 + 1) * a.Hq + h];
            }
            const bool is_lat = latent && kd == kSlotLatent;
            const bool is_raw = kd == kSlotRawAll || kd == kSlotRawGroup + g;
            const bool use = (is_lat || is_raw) && l != 0.f;   // a NaN (poisoned) l is kept
            if (use) M = fmaxf(M, m);
            const unsigned bl = __ballot_sync(0xffffffffu, use && is_lat);
            const unsigned br = __ballot_sync(0xffffffffu, use && is_raw);
            const unsigned below = (1u << lane) - 1u;
            if (use && is_lat) {
                const int o = nl + __popc(bl & below);
                lat_slot[o] = s0 + s;
                lat_m[o] = m;
                lat_l[o] = l;
            }
            if (use && is_raw) {
                const int o = nr + __popc(br & below);
                raw_slot[o] = s0 + s;
                raw_m[o] = m;
                raw_l[o] = l;
            }
            nl += __popc(bl);
            nr += __popc(br);
        }
        M = warp_max(M);
        __syncwarp();
        // weights w = exp2(m - M) (stored over m) and L = sum w l
        float L = 0.f;
        for (int i = lane; i < nl; i += 32) {
            const float w = exp2f(lat_m[i] - M);
            L = fmaf(w, lat_l[i], L);
            lat_m[i] = w;
        }
        for (int i = lane; i < nr; i += 32) {
            const float w = exp2f(raw_m[i] - M);
            L = fmaf(w, raw_l[i], L);
            raw_m[i] = w;
        }
        L = warp_sum(L);
        if (lane == 0) {
            n_lat_s = nl;
            n_raw_s = nr;
            L_s = L;
        }
    }
    __syncthreads();
    const int nl = n_lat_s, nr = n_raw_s;
    // z[j] and y[i]: batches of independent loads over the covering partials
    auto accumulate = [&](const int* slot, const float* w, int n, int col) {
        float acc = 0.f;
        for (int i0 = 0; i0 < n; i0 += kCombBatch) {
            float v[kCombBatch];
#pragma unroll
            for (int k = 0; k < kCombBatch; ++k)
                v[k] = (i0 + k < n) ? a.acc[((size_t)slot[i0 + k] * a.Hq + h) * a.Dmax + col] : 0.f;
#pragma unroll
            for (int k = 0; k < kCombBatch; ++k)
                if (i0 + k < n) acc = fmaf(w[i0 + k], v[k], acc);
        }
        return acc;
    };
    if (latent)
        for (int j = tid; j < a.r_v; j += kCombThreads) z_s[j] = accumulate(lat_slot, lat_m, nl, j);
    for (int i = tid; i < a.d; i += kCombThreads) y_s[i] = accumulate(raw_slot, raw_m, nr, i);
    if (prefetch) cp_async_wait_all();
    __syncthreads();
    const float invL = 1.f / L_s;
    if (!latent) {
        for (int i = tid; i < a.d; i += kCombThreads) a.out[((size_t)b * a.Hq + h) * a.d + i] = y_s[i] * invL;
        return;
    }
    // out[i] = (z . U_V^(g)[i, :] + y[i]) / L; a warp covers rows i = warp, warp + 8, ...
    // with lane l owning latent columns [8l, 8l + 8) of each 256-column chunk
    for (int c0 = 0; c0 < a.r_v; c0 += 256) {
        const int j = c0 + lane * 8;
        float zl[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) zl[e] = (j + e < a.r_v) ? z_s[j + e] : 0.f;
        float part[kCombRowsPerWarp];
#pragma unroll
        for (int r = 0; r < kCombRowsPerWarp; ++r) {
            part[r] = 0.f;
            const int i = warp + r * (kCombThreads / 32);
            if (r < nrow && i < a.d && j < a.r_v) {
                float f[8];
                if (prefetch && c0 == 0) {
                    Vec16<T>::to_f(*reinterpret_cast<const uint4*>(u_stage + i * kCombPrefetchCols + j), f);
                } else {
                    const T* u = (const T*)a.U_V + ((size_t)g * a.d + i) * a.r_v + j;
#pragma unroll
                    for (int q = 0; q < 8 / VN; ++q)
                        Vec16<T>::to_f(*reinterpret_cast<const uint4*>(u + q * VN), f + q * VN);
                }
#pragma unroll
                for (int e = 0; e < 8; ++e) part[r] = fmaf(zl[e], f[e], part[r]);
            }
        }
#pragma unroll
        for (int r = 0; r < kCombRowsPerWarp; ++r) {
            const float v = warp_sum(part[r]);
            const int i = warp + r * (kCombThreads / 32);
            if (lane == 0 && r < nrow && i < a.d) y_s[i] += v;
        }
    }
    __syncwarp();
    for (int r = 0; r < kCombRowsPerWarp; ++r) {
        const int i = warp + r * (kCombThreads / 32);
        if (lane == 0 && r < nrow && i < a.d) a.out[((size_t)b * a.Hq + h) * a.d + i] = y_s[i] * invL;
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
    a.scale_log2 = scale_log2;
    const int G = Hq / Hkv;
    if (G <= kQpRows) {
        a.nbb = kQpRows / G;
        a.hcn = 1;
    } else {
        a.nbb = 1;
        a.hcn = (G + kQpRows - 1) / kQpRows;
    }
    rope_turns(base, d, a.turn);
    const int row_blocks = (G <= kQpRows) ? (B + a.nbb - 1) / a.nbb : B * a.hcn;
    const int col_blocks = U_K ? (r_k + kQpCols - 1) / kQpCols : 1;
    static std::atomic<unsigned long long> attr_done{0};
    const cudaError_t e =
        set_max_smem_once((const void*)qproj_kernel<T>, std::max(kQpSpreadSmem, kQpUBytes), attr_done);
    if (e != cudaSuccess) return e;
    return launch_ex(qproj_kernel<T>, dim3(Hkv, col_blocks, row_blocks), dim3(kQpThreads),
                     (size_t)(pdl ? std::max(kQpSpreadSmem, kQpUBytes) : kQpUBytes), st, pdl, a);
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
    size_t smem = (size_t)((6 * ns_max + 3) & ~3) * sizeof(float);
    if (a.U_V != nullptr && sizeof(T) == 2) smem += (size_t)a.d * kCombPrefetchCols * sizeof(T);
    static std::atomic<unsigned long long> attr_done{0};
    const cudaError_t e = set_max_smem_once(
        (const void*)combine_kernel<T>,
        (int)(((6 * kMaxSlotsPerB + 3) & ~3) * sizeof(float) + 128 * kCombPrefetchCols * sizeof(T)), attr_done);
    if (e != cudaSuccess) return e;
    return launch_ex(combine_kernel<T>, dim3(a.Hq, a.B), dim3(kCombThreads), smem, st, pdl, b);
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

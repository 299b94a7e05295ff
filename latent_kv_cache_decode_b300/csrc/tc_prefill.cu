// Prefill-side attention of SlimKV: a chunk of new tokens attends to the latent beacon
// memory and, causally, to itself, in one softmax.
//
// "Can SlimKV compress KV cache jointly across tokens and features", section "Speedups
// are real, but memory is set by the ratio": time-to-first-token gains over the
// reconstruction variant come from skipping key-side RoPE and full-key materialisation
// for beacon states, i.e. the prompt is processed against the latent beacon memory by
// the rule of section "Latent-space attention removes the rebuild step". For query token
// t of the chunk (position p0 + t), head h of KV group g:
//   qr = RoPE(q[t,h], p0 + t),  q~ = qr . U_K^(g)
//   s  = [scale q~ . C_K^T ; scale qr . K_chunk[0..t, g]^T],  A = softmax(s)
//   out[t,h] = (A_beacon C_V) . U_V^(g)T + A_chunk V_chunk[0..t, g]
// (the chunk's keys are stored after RoPE at p0 + s).
//
// Two kernels:
//   * prefill_qrot_kernel stages the rotated, scaled queries of every (b, g) as rows
//     (t, head of g) of bf16 high and low parts, [hi (d) | lo (d)], for TMA;
//   * tc_prefill_kernel: one CTA per (block of 128 such rows, g, b), 192 threads. Warp 0
//     issues TMA loads, warp 1 the tcgen05 MMAs, warps 2-5 run the softmax with one
//     thread per query row (its TMEM lane). The CTA
//       1. streams the causal chunk tiles (64 tokens of KV head g): S = Q_hi K^T +
//          Q_lo K^T (the high / low split keeps raw scores, whose keys can be large,
//          at float32 accuracy), y += P V;
//       2. projects its queries into latent space on the tensor cores,
//          q~ = Q_hi U_K^(g) + Q_lo U_K^(g) (float32 in TMEM), and rounds q~ to bf16
//          into shared memory over the staged queries;
//       3. streams the beacon tiles (64 beacons): S = q~ C_K^T, z += P C_V (r_v wide);
//       4. adds the up-projection on the tensor cores, y += z_hi U_V^(g)T + z_lo
//          U_V^(g)T, and writes out = y / l.
//     One online softmax spans both phases (log2 domain, reference maximum moved only
//     when a tile's maximum exceeds it by more than kLazy; a move rescales the row's
//     accumulators in TMEM). TMEM: z in columns [0, 256), y in [256, 384), two score
//     buffers of 64 columns in [384, 512). Shared memory: a 64 KB query region, a ring
//     of four 32 KB slots, two 16 KB probability buffers.
// Supported here: bf16 storage, d = 128, ranks r_k, r_v in {64, 128, 192, 256}.
#include <cuda.h>
#include <string.h>

#include <algorithm>
#include <mutex>

#include "slimkv_internal.cuh"
#include "tc_ptx.cuh"

namespace slimkv {

namespace {

constexpr int kPThreads = 192;   // warp 0 TMA, warp 1 MMA, warps 2-5 softmax
constexpr int kPRows = 128;      // query rows per CTA (MMA M)
constexpr int kPKeys = 64;       // keys per tile (score MMA N)
constexpr int kPD = 128;         // head dimension
constexpr int kRing = 4;
constexpr int kSlotB = 32768;    // ring slot
constexpr int kQRegion = 65536;  // 128 rows x 256 bf16
constexpr int kPBuf = 16384;     // 128 rows x 64 bf16
constexpr int kBox8 = 8192;      // TMA box of 64 rows x 64 bf16 (128-byte swizzled)
constexpr int kBox16 = 16384;    // TMA box of 128 rows x 64 bf16
constexpr int kNumBars = 24;
constexpr int kSmemP = 1024 + kQRegion + kRing * kSlotB + 2 * kPBuf + kNumBars * 8 + 64;
constexpr uint32_t kTz = 0, kTy = 256, kTs = 384, kTCols = 512;
constexpr float kLazy = 8.f;     // log2 units a tile maximum may exceed the reference by

struct PrefillParams {
    CUtensorMap tmQ;    // staged queries [B * Hkv * rows_pad, 2 d] bf16, boxes 64 x 128
    CUtensorMap tmCK;   // C_K [B, N_b, r_k], boxes 64 x 64 x 1
    CUtensorMap tmCV;   // C_V [B, N_b, r_v]
    CUtensorMap tmK;    // K_chunk [B, T, Hkv, d], boxes 64 x 1 x 64 x 1
    CUtensorMap tmV;    // V_chunk
    CUtensorMap tmUK;   // U_K [Hkv d, r_k], boxes 64 x 128
    CUtensorMap tmUV;   // U_V [Hkv d, r_v]
    float* out;         // [B, T, Hq, d]
    unsigned long long* aborts;   // device counter of CTAs that gave up on a wait
    int T, Hq, Hkv, G, N_b, r_k, r_v, rows_pad;
};

struct QrotArgs {
    const __nv_bfloat16* q;   // [B, T, Hq, d]
    const int32_t* p0;        // [B]
    __nv_bfloat16* stage;     // [B, Hkv, rows_pad, 2 d]
    int B, T, Hq, Hkv, G, rows_pad;
    float scale_log2;
    unsigned long long turn[64];
};

// Staged query rows: row R of (b, g) is token R / G, head g G + R % G; rows past the
// chunk are zero. Block = 4 rows x 64 rotation pairs.
__global__ void __launch_bounds__(256) prefill_qrot_kernel(const __grid_constant__ QrotArgs a) {
    pdl_wait();
    pdl_trigger();
    const int i = threadIdx.x & 63;                      // pair (i, i + d/2)
    const long long row = (long long)blockIdx.x * 4 + (threadIdx.x >> 6);
    const long long per_bg = a.rows_pad;
    if (row >= (long long)a.B * a.Hkv * per_bg) return;
    const int bg = (int)(row / per_bg), R = (int)(row - (long long)bg * per_bg);
    const int b = bg / a.Hkv, g = bg - b * a.Hkv;
    const int t = R / a.G, hl = R - t * a.G;
    __nv_bfloat16* dst = a.stage + row * (2 * kPD);
    float x1r = 0.f, x2r = 0.f;
    if (t < a.T) {
        const __nv_bfloat16* src = a.q + (((size_t)b * a.T + t) * a.Hq + g * a.G + hl) * kPD;
        const float x1 = __bfloat162float(src[i]), x2 = __bfloat162float(src[i + kPD / 2]);
        const unsigned long long pos = (unsigned long long)((long long)a.p0[b] + t);
        // cos / sin of p theta_i from the angle reduced exactly to a signed fraction of
        // a turn (64-bit wrap-around), then sin / cos in float32
        const long long frac = (long long)(pos * a.turn[i]);
        float sn, cs;
        sincospif((float)frac * 1.0842021724855044e-19f, &sn, &cs);   // x 2^-63: half-turns
        x1r = (x1 * cs - x2 * sn) * a.scale_log2;
        x2r = (x2 * cs + x1 * sn) * a.scale_log2;
    }
    const __nv_bfloat16 h1 = __float2bfloat16_rn(x1r), h2 = __float2bfloat16_rn(x2r);
    dst[i] = h1;
    dst[i + kPD / 2] = h2;
    dst[kPD + i] = __float2bfloat16_rn(x1r - __bfloat162float(h1));
    dst[kPD + i + kPD / 2] = __float2bfloat16_rn(x2r - __bfloat162float(h2));
}

// Ring fill sequence of one CTA: raw K(j), V(j) for j < nraw; two fills of U_K^(g);
// latent K(j), V(j); two fills of U_V^(g).
struct Fills {
    int nraw, ntiles;
    __device__ int K(int j) const { return j < nraw ? 2 * j : 2 * j + 2; }
    __device__ int V(int j) const { return K(j) + 1; }
    __device__ int UK() const { return 2 * nraw; }
    __device__ int UV() const { return 2 * ntiles + 2; }
};
__device__ __forceinline__ uint32_t fslot(int f) { return (uint32_t)(f % kRing); }
__device__ __forceinline__ uint32_t fphase(int f) { return (uint32_t)((f / kRing) & 1); }

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&v);
}

// Write 32 consecutive columns [c0, c0 + 32) of row `row` of a K-major 128-byte swizzled
// operand with `rows` rows (chunks of 64 columns) as bf16. Returns nothing; `lo` (if not
// null) receives the low parts x - bf16(x) in a second operand of the same layout.
__device__ __forceinline__ void put_row32(uint8_t* hi_base, uint8_t* lo_base0, uint8_t* lo_base1, int row,
                                          int c0, const float (&v)[32]) {
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        uint32_t h[4], l[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float a = v[8 * u + 2 * k], b = v[8 * u + 2 * k + 1];
            h[k] = pack_bf16(a, b);
            if (lo_base0 != nullptr) {
                const float ah = __uint_as_float(h[k] << 16), bh = __uint_as_float(h[k] & 0xffff0000u);
                l[k] = pack_bf16(a - ah, b - bh);
            }
        }
        const int col = c0 + 8 * u;
        const uint32_t off = ptx::sw128_offset(row, col, kPRows);
        *reinterpret_cast<uint4*>(hi_base + off) = make_uint4(h[0], h[1], h[2], h[3]);
        if (lo_base0 != nullptr) {
            // the low parts' 64-column chunks c live in two ring slots: chunk c in slot
            // c / 2 at (c % 2) * 16 KB
            const int chunk = col >> 6;
            uint8_t* lb = (chunk >> 1) ? lo_base1 : lo_base0;
            const uint32_t loff = ptx::sw128_offset(row, col & 63, kPRows) + (uint32_t)((chunk & 1) * kBox16);
            *reinterpret_cast<uint4*>(lb + loff) = make_uint4(l[0], l[1], l[2], l[3]);
        }
    }
}

__global__ void __launch_bounds__(kPThreads, 1) tc_prefill_kernel(const __grid_constant__ PrefillParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* qreg = smem;
    uint8_t* ring = smem + kQRegion;
    uint8_t* pbuf = ring + kRing * kSlotB;
    uint64_t* bars = reinterpret_cast<uint64_t*>(pbuf + 2 * kPBuf);
    uint64_t* full = bars;              // [kRing] ring slot loaded            (TMA tx)
    uint64_t* empty = bars + 4;         // [kRing] ring slot consumed          (MMA commit)
    uint64_t* s_full = bars + 8;        // [2] scores of tile j in buffer j&1  (MMA commit)
    uint64_t* p_full = bars + 10;       // [2] P of tile j written             (128 arrivals)
    uint64_t* v_done = bars + 12;       // [2] value MMAs of tile j done       (MMA commit)
    uint64_t* q_full = bars + 14;       // staged queries loaded               (TMA tx)
    uint64_t* proj_done = bars + 15;    // latent query projection in TMEM     (MMA commit)
    uint64_t* qt_ready = bars + 16;     // latent query operand in smem        (128 arrivals)
    uint64_t* z_ready = bars + 17;      // z high / low operands in smem       (128 arrivals)
    uint64_t* y_done = bars + 18;       // up-projection added into y          (MMA commit)
    uint64_t* drain = bars + 19;        // every MMA of the CTA done           (MMA commit)
    uint32_t* tmem_s = reinterpret_cast<uint32_t*>(bars + kNumBars);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + kNumBars) + 1;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int c = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
    const int G = p.G, T = p.T;
    const int R0 = c * kPRows;
    const int t_hi = min(T - 1, (R0 + kPRows - 1) / G);
    Fills F;
    F.nraw = t_hi / kPKeys + 1;
    const int nlat = (p.N_b + kPKeys - 1) / kPKeys;
    F.ntiles = F.nraw + nlat;
    const bool has_lat = nlat > 0;

    if (threadIdx.x == 0) {
#pragma unroll 1
        for (int i = 0; i < kRing; ++i) {
            ptx::mbar_init(&full[i], 1);
            ptx::mbar_init(&empty[i], 1);
        }
#pragma unroll 1
        for (int i = 0; i < 2; ++i) {
            ptx::mbar_init(&s_full[i], 1);
            ptx::mbar_init(&p_full[i], 128);
            ptx::mbar_init(&v_done[i], 1);
        }
        ptx::mbar_init(q_full, 1);
        ptx::mbar_init(proj_done, 1);
        ptx::mbar_init(qt_ready, 128);
        ptx::mbar_init(z_ready, 128);
        ptx::mbar_init(y_done, 1);
        ptx::mbar_init(drain, 1);
        *abort_flag = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 1) ptx::tmem_alloc(tmem_s, kTCols);
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_s;
    pdl_wait();   // the staged queries come from the preceding kernel
    pdl_trigger();

    if (warp == 0) {
        // ---------------------------------------------------------------- producer
        if (lane == 0) {
            // beacon and chunk tiles keep the default L2 policy: every CTA of a batch element
            // (all its KV groups and row blocks) reads the same beacon tiles, so they
            // should stay in L2 rather than be streamed
            const int qrow = (b * p.Hkv + g) * p.rows_pad + R0;
            ptx::mbar_expect_tx(q_full, kQRegion);
#pragma unroll 1
            for (int i = 0; i < 4; ++i) ptx::tma_load_2d(qreg + i * kBox16, &p.tmQ, 64 * i, qrow, q_full);
            auto acquire = [&](int f) -> uint8_t* {
                if (f >= kRing) ptx::mbar_wait(&empty[fslot(f)], fphase(f) ^ 1u, abort_flag);
                return ring + fslot(f) * kSlotB;
            };
            const int nkc = p.r_k / 64, nvc = p.r_v / 64;
            auto load_u = [&](int f0, const CUtensorMap* tm, int nch) {
                for (int h = 0; h < 2; ++h) {
                    const int f = f0 + h;
                    uint8_t* dst = acquire(f);
                    const int n = max(0, min(2, nch - 2 * h));
                    ptx::mbar_expect_tx(&full[fslot(f)], (uint32_t)(n * kBox16));
                    for (int k = 0; k < n; ++k)
                        ptx::tma_load_2d(dst + k * kBox16, tm, 64 * (2 * h + k), g * kPD, &full[fslot(f)]);
                }
            };
#pragma unroll 1
            for (int j = 0; j < F.ntiles && !*abort_flag; ++j) {
                if (j == F.nraw) load_u(F.UK(), &p.tmUK, nkc);
                const bool lat = j >= F.nraw;
                for (int part = 0; part < 2; ++part) {
                    const int f = part ? F.V(j) : F.K(j);
                    uint8_t* dst = acquire(f);
                    uint64_t* fb = &full[fslot(f)];
                    if (lat) {
                        const int jl = j - F.nraw, n = part ? nvc : nkc;
                        const CUtensorMap* tm = part ? &p.tmCV : &p.tmCK;
                        ptx::mbar_expect_tx(fb, (uint32_t)(n * kBox8));
                        for (int k = 0; k < n; ++k)
                            ptx::tma_load_3d(dst + k * kBox8, tm, 64 * k, jl * kPKeys, b, fb);
                    } else {
                        const CUtensorMap* tm = part ? &p.tmV : &p.tmK;
                        ptx::mbar_expect_tx(fb, 2 * kBox8);
                        for (int k = 0; k < 2; ++k)
                            ptx::tma_load_4d(dst + k * kBox8, tm, 64 * k, g, j * kPKeys, b, fb);
                    }
                }
            }
            if (has_lat && !*abort_flag) load_u(F.UV(), &p.tmUV, nvc);
            if (*abort_flag) {
                // let copies still in flight land before the CTA winds down (bounded
                // waits; a fill that was never issued just times out)
                volatile int never = 0;
                ptx::mbar_wait(q_full, 0, &never);
                const int nf = has_lat ? F.UV() + 2 : 2 * F.ntiles;
#pragma unroll 1
                for (int f = max(0, nf - kRing); f < nf; ++f) ptx::mbar_wait(&full[fslot(f)], fphase(f), &never);
            }
        }
    } else if (warp == 1) {
        // --------------------------------------------------------------------- MMA
        if (lane == 0) {
            const uint32_t idS = ptx::idesc_bf16(kPRows, kPKeys, false, false);
            const uint32_t idVr = ptx::idesc_bf16(kPRows, kPD, false, true);
            const uint32_t idVl = ptx::idesc_bf16(kPRows, p.r_v, false, true);
            const uint32_t idP = ptx::idesc_bf16(kPRows, 64, false, true);
            const uint32_t idU = ptx::idesc_bf16(kPRows, kPD, false, false);
            const uint32_t q_addr = ptx::smem_u32(qreg), ring_addr = ptx::smem_u32(ring);
            const uint32_t p_addr = ptx::smem_u32(pbuf);
            auto kdesc = [](uint32_t a) { return ptx::sdesc_sw128(a, 16, 1024); };           // K-major
            auto mdesc = [](uint32_t a, uint32_t lbo) { return ptx::sdesc_sw128(a, lbo, 1024); };   // MN-major
            auto slot_addr = [&](int f) { return ring_addr + fslot(f) * kSlotB; };
            auto wait_full = [&](int f) {
                ptx::mbar_wait(&full[fslot(f)], fphase(f), abort_flag);
                ptx::tc_fence_after();
            };
            ptx::mbar_wait(q_full, 0, abort_flag);
            ptx::tc_fence_after();
            const int ksl = p.r_k / 16;
#pragma unroll 1
            for (int j = 0; j <= F.ntiles; ++j) {
                if (j < F.ntiles) {
                    const bool lat = j >= F.nraw;
                    if (j == F.nraw) {
                        // latent query projection: q~ = Q_hi U_K^(g) + Q_lo U_K^(g), one
                        // 64-column block of q~ per MMA (U_K^(g) is MN-major: d rows)
                        wait_full(F.UK());
                        wait_full(F.UK() + 1);
#pragma unroll 1
                        for (int nc = 0; nc < p.r_k / 64; ++nc) {
                            const uint32_t ub = slot_addr(F.UK() + nc / 2) + (nc & 1) * kBox16;
#pragma unroll 1
                            for (int kk = 0; kk < 16; ++kk) {
                                // k-steps 0-7: high part (chunks 0, 1), 8-15: low part (2, 3)
                                const int kd = kk & 7;
                                const uint32_t a = q_addr + (uint32_t)((kk >> 2) * kBox16 + (kk & 3) * 32);
                                const uint32_t bb = ub + (uint32_t)(kd * 2048);
                                ptx::mma_bf16(tmem + kTz + 64 * nc, kdesc(a), mdesc(bb, kBox16), idP, kk ? 1u : 0u);
                            }
                        }
                        ptx::mma_commit(proj_done);
                        ptx::mma_commit(&empty[fslot(F.UK())]);
                        ptx::mma_commit(&empty[fslot(F.UK() + 1)]);
                        ptx::mbar_wait(qt_ready, 0, abort_flag);   // q~ rounded into the query region
                        ptx::tc_fence_after();
                    }
                    // scores S(j) into buffer j & 1 (free once P(j - 2) was written)
                    if (j >= 2) {
                        ptx::mbar_wait(&p_full[j & 1], (uint32_t)((j - 2) >> 1) & 1u, abort_flag);
                        ptx::tc_fence_after();
                    }
                    wait_full(F.K(j));
                    const uint32_t kb = slot_addr(F.K(j));
                    const uint32_t dS = tmem + kTs + (uint32_t)((j & 1) * kPKeys);
                    if (lat) {
#pragma unroll 1
                        for (int kk = 0; kk < ksl; ++kk) {
                            const uint32_t a = q_addr + (uint32_t)((kk >> 2) * kBox16 + (kk & 3) * 32);
                            const uint32_t bb = kb + (uint32_t)((kk >> 2) * kBox8 + (kk & 3) * 32);
                            ptx::mma_bf16(dS, kdesc(a), kdesc(bb), idS, kk ? 1u : 0u);
                        }
                    } else {
#pragma unroll 1
                        for (int kk = 0; kk < 16; ++kk) {
                            const int kd = kk & 7;   // 0-7 high part, 8-15 low part of the query
                            const uint32_t a = q_addr + (uint32_t)((kk >> 2) * kBox16 + (kk & 3) * 32);
                            const uint32_t bb = kb + (uint32_t)((kd >> 2) * kBox8 + (kd & 3) * 32);
                            ptx::mma_bf16(dS, kdesc(a), kdesc(bb), idS, kk ? 1u : 0u);
                        }
                    }
                    ptx::mma_commit(&s_full[j & 1]);
                    ptx::mma_commit(&empty[fslot(F.K(j))]);
                }
                if (j >= 1) {
                    // values of tile jj = j - 1: y (raw) or z (latent) += P(jj) . V(jj)
                    const int jj = j - 1;
                    const bool lat = jj >= F.nraw;
                    ptx::mbar_wait(&p_full[jj & 1], (uint32_t)(jj >> 1) & 1u, abort_flag);
                    ptx::tc_fence_after();
                    wait_full(F.V(jj));
                    const uint32_t vb = slot_addr(F.V(jj));
                    const uint32_t pa = p_addr + (uint32_t)((jj & 1) * kPBuf);
                    const uint32_t acc0 = (jj == 0 || jj == F.nraw) ? 0u : 1u;
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        ptx::mma_bf16(tmem + (lat ? kTz : kTy), kdesc(pa + (uint32_t)(kk * 32)),
                                      mdesc(vb + (uint32_t)(kk * 2048), kBox8), lat ? idVl : idVr,
                                      kk ? 1u : acc0);
                    }
                    ptx::mma_commit(&v_done[jj & 1]);
                    ptx::mma_commit(&empty[fslot(F.V(jj))]);
                }
            }
            if (has_lat) {
                // up-projection: y += z_hi U_V^(g)T + z_lo U_V^(g)T (U_V^(g) rows = output
                // dimensions, K-major over r_v)
                ptx::mbar_wait(z_ready, 0, abort_flag);
                ptx::tc_fence_after();
                wait_full(F.UV());
                wait_full(F.UV() + 1);
                const int ksv = p.r_v / 16;
#pragma unroll 1
                for (int part = 0; part < 2; ++part) {
#pragma unroll 1
                    for (int kk = 0; kk < ksv; ++kk) {
                        const int ch = kk >> 2;
                        const uint32_t in = (uint32_t)((kk & 3) * 32);
                        const uint32_t a = part == 0
                                               ? q_addr + (uint32_t)(ch * kBox16) + in
                                               : slot_addr(F.UV() + 2 + ch / 2) + (uint32_t)((ch & 1) * kBox16) + in;
                        const uint32_t bb = slot_addr(F.UV() + ch / 2) + (uint32_t)((ch & 1) * kBox16) + in;
                        ptx::mma_bf16(tmem + kTy, kdesc(a), kdesc(bb), idU, 1u);
                    }
                }
            }
            ptx::mma_commit(y_done);
            ptx::mma_commit(drain);
        }
    } else {
        // ----------------------------------------------------------------- softmax
        const int q4 = warp & 3;
        const int row = q4 * 32 + lane;                // query row = TMEM lane
        const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
        const int R = R0 + row;
        const int t = R / G, hl = R - t * G;
        float m = -INFINITY, l = 0.f;
        float s[kPKeys];
#pragma unroll 1
        for (int j = 0; j < F.ntiles; ++j) {
            const bool lat = j >= F.nraw;
            if (j == F.nraw) {
                // the projected queries, rounded to bf16 over the staged queries (every
                // MMA that read those has completed with the projection)
                ptx::mbar_wait(proj_done, 0, abort_flag);
                ptx::tc_fence_after();
#pragma unroll 1
                for (int c0 = 0; c0 < p.r_k; c0 += 32) {
                    float v[32];
                    ptx::tmem_ld32(tmem + lane_off + kTz + (uint32_t)c0, v);
                    put_row32(qreg, nullptr, nullptr, row, c0, v);
                }
                ptx::fence_proxy_async_smem();
                ptx::tc_fence_before();
                ptx::mbar_arrive(qt_ready);
            }
            ptx::mbar_wait(&s_full[j & 1], (uint32_t)(j >> 1) & 1u, abort_flag);
            ptx::tc_fence_after();
            {
                float a[32], bq[32];
                const uint32_t sa = tmem + lane_off + kTs + (uint32_t)((j & 1) * kPKeys);
                ptx::tmem_ld32(sa, a);
                ptx::tmem_ld32(sa + 32, bq);
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    s[i] = a[i];
                    s[32 + i] = bq[i];
                }
            }
            // masks: raw keys after the row's token, beacons past N_b
            const int key0 = lat ? (j - F.nraw) * kPKeys : j * kPKeys;
            const int lim = lat ? p.N_b - 1 : t;
            float mt = -INFINITY;
#pragma unroll
            for (int i = 0; i < kPKeys; ++i) {
                if (key0 + i > lim) s[i] = -INFINITY;
                mt = fmaxf(mt, s[i]);
            }
            // a row whose tile maximum passes its reference by more than kLazy moves the
            // reference and rescales its accumulators; TMEM access is warp-wide, so the
            // warp rescales together, every other row by 1
            const bool need = mt > m + kLazy;
            const float alpha = need ? exp2f(m - mt) : 1.f;   // 0 for the first tile
            l *= alpha;
            if (need) m = mt;
            if (__any_sync(0xffffffffu, need)) {
                if (j >= 1) {
                    // rescale the accumulators once the previous tile's value MMAs are done
                    ptx::mbar_wait(&v_done[(j - 1) & 1], (uint32_t)((j - 1) >> 1) & 1u, abort_flag);
                    ptx::tc_fence_after();
#pragma unroll 1
                    for (int c0 = 0; c0 < kPD; c0 += 16) {
                        float v[16];
                        ptx::tmem_ld16(tmem + lane_off + kTy + (uint32_t)c0, v);
#pragma unroll
                        for (int i = 0; i < 16; ++i) v[i] *= alpha;
                        ptx::tmem_st16(tmem + lane_off + kTy + (uint32_t)c0, v);
                    }
                    if (j - 1 >= F.nraw) {
#pragma unroll 1
                        for (int c0 = 0; c0 < p.r_v; c0 += 16) {
                            float v[16];
                            ptx::tmem_ld16(tmem + lane_off + kTz + (uint32_t)c0, v);
#pragma unroll
                            for (int i = 0; i < 16; ++i) v[i] *= alpha;
                            ptx::tmem_st16(tmem + lane_off + kTz + (uint32_t)c0, v);
                        }
                    }
                }
            }
            // probabilities of this tile into P buffer j & 1 (free once V(j - 2) is done)
            if (j >= 2) ptx::mbar_wait(&v_done[j & 1], (uint32_t)((j - 2) >> 1) & 1u, abort_flag);
            uint8_t* pb = pbuf + (j & 1) * kPBuf;
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                uint32_t w[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const float e0 = exp2f(s[8 * u + 2 * k] - m), e1 = exp2f(s[8 * u + 2 * k + 1] - m);
                    l += e0 + e1;
                    w[k] = pack_bf16(e0, e1);
                }
                *reinterpret_cast<uint4*>(pb + ptx::sw128_offset(row, 8 * u, kPRows)) =
                    make_uint4(w[0], w[1], w[2], w[3]);
            }
            ptx::fence_proxy_async_smem();
            ptx::tc_fence_before();
            ptx::mbar_arrive(&p_full[j & 1]);
        }
        const int jl = F.ntiles - 1;
        ptx::mbar_wait(&v_done[jl & 1], (uint32_t)(jl >> 1) & 1u, abort_flag);
        ptx::tc_fence_after();
        if (has_lat) {
            // z as high and low bf16 parts: high over the latent queries (every score MMA
            // is done), low in the two ring slots after U_V^(g)'s
            uint8_t* lo0 = ring + fslot(F.UV() + 2) * kSlotB;
            uint8_t* lo1 = ring + fslot(F.UV() + 3) * kSlotB;
#pragma unroll 1
            for (int c0 = 0; c0 < p.r_v; c0 += 32) {
                float v[32];
                ptx::tmem_ld32(tmem + lane_off + kTz + (uint32_t)c0, v);
                put_row32(qreg, lo0, lo1, row, c0, v);
            }
            ptx::fence_proxy_async_smem();
            ptx::tc_fence_before();
            ptx::mbar_arrive(z_ready);
            ptx::mbar_wait(y_done, 0, abort_flag);
            ptx::tc_fence_after();
        }
        const float inv = 1.f / l;
        const bool bad = *abort_flag != 0;
        float* dst = p.out + (((size_t)b * T + t) * p.Hq + g * G + hl) * kPD;
#pragma unroll 1
        for (int c0 = 0; c0 < kPD; c0 += 32) {
            float v[32];
            ptx::tmem_ld32(tmem + lane_off + kTy + (uint32_t)c0, v);
            if (t < T) {
#pragma unroll
                for (int i = 0; i < 32; i += 4) {
                    float4 o = bad ? make_float4(NAN, NAN, NAN, NAN)
                                   : make_float4(v[i] * inv, v[i + 1] * inv, v[i + 2] * inv, v[i + 3] * inv);
                    *reinterpret_cast<float4*>(dst + c0 + i) = o;
                }
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
        ptx::tmem_dealloc(tmem, kTCols);
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

// A bf16 tensor of `rank` dimensions (innermost first), 128-byte swizzled boxes.
bool make_map(CUtensorMap* tm, const void* base, int rank, const cuuint64_t* dims, const cuuint32_t* box) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t strides[3];
    cuuint64_t s = 2;
    for (int i = 0; i + 1 < rank; ++i) {
        s *= dims[i];
        strides[i] = s;
    }
    cuuint32_t es[4] = {1, 1, 1, 1};
    return fn(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (cuuint32_t)rank, const_cast<void*>(base), dims, strides, box,
              es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool prefill_supported(int d, int N_b, int r_k, int r_v) {
    if (d != kPD) return false;
    if (N_b == 0) return true;
    return r_k >= 64 && r_k <= 256 && r_k % 64 == 0 && r_v >= 64 && r_v <= 256 && r_v % 64 == 0;
}

size_t prefill_stage_bytes(int B, int T, int Hq, int Hkv) {
    const int G = Hq / Hkv;
    const size_t rows_pad = ((size_t)T * G + kPRows - 1) / kPRows * kPRows;
    return (size_t)B * Hkv * rows_pad * 2 * kPD * sizeof(__nv_bfloat16);
}

cudaError_t launch_prefill(const PrefillCall& c, cudaStream_t st) {
    const int G = c.Hq / c.Hkv;
    const int rows_pad = (int)(((int64_t)c.T * G + kPRows - 1) / kPRows * kPRows);
    // 1. staged, rotated, scaled queries
    QrotArgs qa;
    memset(&qa, 0, sizeof(qa));
    qa.q = static_cast<const __nv_bfloat16*>(c.q);
    qa.p0 = c.p0;
    qa.stage = static_cast<__nv_bfloat16*>(c.stage);
    qa.B = c.B;
    qa.T = c.T;
    qa.Hq = c.Hq;
    qa.Hkv = c.Hkv;
    qa.G = G;
    qa.rows_pad = rows_pad;
    qa.scale_log2 = c.scale * kLog2e;
    rope_turns(c.rope_base, kPD, qa.turn);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    {
        const long long rows = (long long)c.B * c.Hkv * rows_pad;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)((rows + 3) / 4));
        cfg.blockDim = dim3(256);
        cfg.stream = st;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        const cudaError_t e = cudaLaunchKernelEx(&cfg, prefill_qrot_kernel, qa);
        if (e != cudaSuccess) return e;
    }
    // 2. the attention
    PrefillParams p;
    memset(&p, 0, sizeof(p));
    {
        const cuuint64_t dq[2] = {(cuuint64_t)2 * kPD, (cuuint64_t)c.B * c.Hkv * rows_pad};
        const cuuint32_t bq[2] = {64, kPRows};
        if (!make_map(&p.tmQ, c.stage, 2, dq, bq)) return cudaErrorInvalidValue;
        const cuuint64_t dk[4] = {(cuuint64_t)kPD, (cuuint64_t)c.Hkv, (cuuint64_t)c.T, (cuuint64_t)c.B};
        const cuuint32_t bk[4] = {64, 1, kPKeys, 1};
        if (!make_map(&p.tmK, c.K_chunk, 4, dk, bk) || !make_map(&p.tmV, c.V_chunk, 4, dk, bk))
            return cudaErrorInvalidValue;
        if (c.N_b > 0) {
            const cuuint64_t dck[3] = {(cuuint64_t)c.r_k, (cuuint64_t)c.N_b, (cuuint64_t)c.B};
            const cuuint64_t dcv[3] = {(cuuint64_t)c.r_v, (cuuint64_t)c.N_b, (cuuint64_t)c.B};
            const cuuint32_t bc[3] = {64, kPKeys, 1};
            const cuuint64_t duk[2] = {(cuuint64_t)c.r_k, (cuuint64_t)c.Hkv * kPD};
            const cuuint64_t duv[2] = {(cuuint64_t)c.r_v, (cuuint64_t)c.Hkv * kPD};
            const cuuint32_t bu[2] = {64, kPRows};
            if (!make_map(&p.tmCK, c.C_K, 3, dck, bc) || !make_map(&p.tmCV, c.C_V, 3, dcv, bc) ||
                !make_map(&p.tmUK, c.U_K, 2, duk, bu) || !make_map(&p.tmUV, c.U_V, 2, duv, bu))
                return cudaErrorInvalidValue;
        }
    }
    p.out = c.out;
    p.aborts = abort_counter();
    p.T = c.T;
    p.Hq = c.Hq;
    p.Hkv = c.Hkv;
    p.G = G;
    p.N_b = c.N_b;
    p.r_k = c.N_b > 0 ? c.r_k : 0;
    p.r_v = c.N_b > 0 ? c.r_v : 0;
    p.rows_pad = rows_pad;
    static std::atomic<unsigned long long> attr_done{0};
    const cudaError_t e = set_max_smem_once((const void*)tc_prefill_kernel, kSmemP, attr_done);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(rows_pad / kPRows, c.Hkv, c.B);
    cfg.blockDim = dim3(kPThreads);
    cfg.dynamicSmemBytes = kSmemP;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    timer_before(st);
    const cudaError_t e2 = cudaLaunchKernelEx(&cfg, tc_prefill_kernel, p);
    timer_after(st);
    return e2;
}

}  // namespace slimkv

// Tensor-core split-context decode for SlimKV on sm_103a (tcgen05 + TMA).
//
// "Can SlimKV compress KV cache jointly across tokens and features", section
// "Latent-space attention removes the rebuild step": per query head the scores
// are (RoPE(q) U_K^(g)) C_K^T against the RoPE-free latent beacon keys and
// RoPE(q) K_raw^T against the raw window, in one softmax; values aggregate as
// (A C_V) U_V^(g)T + A V_raw, the latent aggregate taken before the up-projection.
//
// Layout of the work. A "tile" is 128 key rows of one segment; a segment is all
// rows of one kind for one batch element:
//   latent: rows are beacons j of C_K[b] / C_V[b] (widths r_k / r_v);
//   raw:    rows are the flattened (token, KV head) pairs t*Hkv + g of K[b] / V[b]
//           (width d), so a 128-row tile is one contiguous 32 KB block of the cache.
// Every query head of batch element b shares a latent tile, so one tcgen05.mma
// with M = 128 tile rows and N = all heads (a bf16 high and low part of the query,
// N = 2*NP) gives the tile's scores S^T in TMEM. Raw tiles use the same MMA; a
// row of KV head g only counts for the heads of group g (block-diagonal mask,
// applied to the scores). The softmax warps turn S^T into P (bf16 high + low
// parts, zero outside the group) in shared memory, and a second MMA with M = 128
// rows of the value width accumulates acc^T[value dim, head] += V_tile^T P^T in
// TMEM, i.e. the latent aggregate A.C_V (or A.V_raw) per head.
//
// Roles (192 threads): warp 0 issues TMA loads into a ring of 32 KB slots, warp 1
// issues the MMAs and owns TMEM, warps 2-5 run the online softmax (running max in
// the log2 domain, rescaling the TMEM accumulator only when a head's max grows by
// more than 2^8) and write one partial (m, l, acc) per (CTA, segment) to the
// workspace. A separate kernel merges the partials and applies U_V^(g)T.
#include <cuda.h>
#include <string.h>

#include <algorithm>
#include <map>
#include <mutex>
#include <tuple>
#include <vector>

#include "../../include/slimkv.h"
#include "slimkv_internal.cuh"
#include "tc_decode.cuh"
#include "tc_ptx.cuh"

namespace slimkv {

namespace {

constexpr int kTile = 128;            // rows per tile (MMA M)
constexpr int kBox = 16384;           // one TMA box: 128 rows x 64 bf16 columns, 128B-swizzled
constexpr int kSlot = 2 * kBox;       // ring slot: 128 rows x 128 columns
constexpr int kThreads = 192;
constexpr int kSmemMax = 227 * 1024;  // dynamic shared memory we may use per CTA
constexpr int kNumKinds = 3;          // latent, raw source 0, raw source 1

struct TcParams {
    CUtensorMap tm[2 * kNumKinds];    // per kind: keys, values
    int B, Hq, Hkv, G;
    int rows[kNumKinds];              // key rows per batch element (0 = kind absent)
    int tiles[kNumKinds];             // tiles per batch element
    int dk[kNumKinds], dv[kNumKinds]; // key / value width
    int tiles_per_b;
    float scale_log2;
    const float* q_lat;               // [B, Hq, r_k]
    const float* q_rot;               // [B, Hq, d]
    float* acc;                       // [slots, Hq, Dmax]
    float* ml;                        // [slots, 2, Hq]
    int* kind;                        // [slots]
    int Dmax;
    int nslot, npbuf, lookahead;
    int q_cols;                       // columns of the query operand buffer (multiple of 64)
    uint32_t off_q, off_p, off_bar, off_red;
    uint32_t tmem_cols;
    int u_begin[kMaxCtas + 1];        // CTA i owns units (tiles) [u_begin[i], u_begin[i+1])
    int slot_base[kMaxCtas];          // first partial slot of CTA i
};

// Position of unit u: batch element, kind and tile index inside its segment.
struct UnitPos {
    int b, k, t;
};
__device__ __forceinline__ UnitPos unit_pos(const TcParams& p, int u) {
    UnitPos r;
    r.b = u / p.tiles_per_b;
    int t = u - r.b * p.tiles_per_b;
    r.k = 0;
    while (r.k < kNumKinds - 1 && t >= p.tiles[r.k]) {
        t -= p.tiles[r.k];
        ++r.k;
    }
    r.t = t;
    return r;
}

// The run of this CTA's units that starts at u and stays inside one segment.
struct Piece {
    int b, k, t0, n;
};
__device__ __forceinline__ Piece piece_at(const TcParams& p, int u, int u1) {
    const UnitPos q = unit_pos(p, u);
    Piece r;
    r.b = q.b;
    r.k = q.k;
    r.t0 = q.t;
    r.n = min(u1 - u, p.tiles[q.k] - q.t);
    return r;
}

struct TileInfo {
    int k, nK, nV;
    uint32_t ld0;   // index of the tile's first ring load
    bool first, last;
    int seg;
};

template <int NP>
__global__ void __launch_bounds__(kThreads, 1) tc_decode_kernel(const __grid_constant__ TcParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    constexpr int NQ = 2 * NP;
    uint8_t* ring = smem;
    uint8_t* qbuf = smem + p.off_q;          // [NQ rows x q_cols] query operand (hi rows, lo rows)
    uint8_t* pbuf = smem + p.off_p;          // [npbuf][hi, lo][NP x 128] probabilities
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + p.off_bar);
    float* red = reinterpret_cast<float*>(smem + p.off_red);   // [4][NP]
    float* m_run = red + 4 * NP;                               // [NP] running max (log2 domain)
    float* alpha_s = m_run + NP;                               // [NP] rescale factors
    // [0] abort; [1], [2] "some head rescales" for even / odd tiles (double-buffered
    // so a slow warp still reading one tile's flag never sees the next tile's reset)
    volatile int* flag = reinterpret_cast<volatile int*>(alpha_s + NP);
    uint32_t* tmem_base_s = reinterpret_cast<uint32_t*>(alpha_s + NP) + 4;

    uint64_t* full = bars;
    uint64_t* empty = bars + p.nslot;
    uint64_t* s_full = bars + 2 * p.nslot;
    uint64_t* s_empty = s_full + 2;
    uint64_t* p_full = s_empty + 2;
    uint64_t* p_empty = p_full + 2;
    uint64_t* q_full = p_empty + 2;
    uint64_t* q_empty = q_full + 1;
    uint64_t* acc_full = q_empty + 1;
    uint64_t* acc_empty = acc_full + 1;
    uint64_t* drain = acc_empty + 1;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int cta = blockIdx.x;
    const int u0 = p.u_begin[cta], u1 = p.u_begin[cta + 1];

    if (threadIdx.x == 0) {
        for (int i = 0; i < p.nslot; ++i) {
            ptx::mbar_init(&full[i], 1);
            ptx::mbar_init(&empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            ptx::mbar_init(&s_full[i], 1);
            ptx::mbar_init(&s_empty[i], 128);
            ptx::mbar_init(&p_full[i], 128);
            ptx::mbar_init(&p_empty[i], 1);
        }
        ptx::mbar_init(q_full, 1);
        ptx::mbar_init(q_empty, 1);
        ptx::mbar_init(acc_full, 1);
        ptx::mbar_init(acc_empty, 128);
        ptx::mbar_init(drain, 1);
        flag[0] = 0;
        flag[1] = 0;
        flag[2] = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 1) ptx::tmem_alloc(tmem_base_s, p.tmem_cols);
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_base_s;
    const uint32_t t_S = tmem;             // 2 score buffers, NQ columns each
    const uint32_t t_acc = tmem + 2 * NQ;  // value accumulators, NP columns per 128 value rows
    volatile int* abort_flag = &flag[0];
    pdl_trigger();

    if (warp == 0) {
        // ---------------------------------------------------------------- producer
        if (lane == 0) {
            for (int i = 0; i < 2 * kNumKinds; ++i)
                if (p.rows[i >> 1] > 0) ptx::tma_prefetch_desc(&p.tm[i]);
            uint32_t ld = 0;
            bool ok = true;
            for (int u = u0; ok && u < u1;) {
                const Piece pc = piece_at(p, u, u1);
                const int nK = (p.dk[pc.k] + 127) >> 7, nV = (p.dv[pc.k] + 127) >> 7;
                for (int t = pc.t0; ok && t < pc.t0 + pc.n; ++t) {
                    for (int part = 0; ok && part < 2; ++part) {
                        const CUtensorMap* tm = &p.tm[2 * pc.k + part];
                        const int nc = part ? nV : nK;
                        for (int c = 0; c < nc; ++c) {
                            const int slot = ld % p.nslot;
                            if (!ptx::mbar_wait(&empty[slot], ((ld / p.nslot) & 1) ^ 1, abort_flag)) {
                                ok = false;
                                break;
                            }
                            uint8_t* dst = ring + (size_t)slot * kSlot;
                            ptx::mbar_expect_tx(&full[slot], kSlot);
                            ptx::tma_load_3d(dst, tm, c * 128, t * kTile, pc.b, &full[slot]);
                            ptx::tma_load_3d(dst + kBox, tm, c * 128 + 64, t * kTile, pc.b, &full[slot]);
                            ++ld;
                        }
                    }
                }
                u += pc.n;
            }
            if (!ok) {
                // let the copies already in flight land before the CTA winds down
                const uint32_t first = ld > (uint32_t)p.nslot ? ld - p.nslot : 0u;
                for (uint32_t i = first; i < ld; ++i) {
                    volatile int never = 0;
                    ptx::mbar_wait(&full[i % p.nslot], (i / p.nslot) & 1, &never);
                }
            }
        }
    } else if (warp == 1) {
        // --------------------------------------------------------------------- MMA
        if (lane == 0) {
            const uint32_t idS = ptx::idesc_bf16(128, NQ, false, false);
            const uint32_t idV = ptx::idesc_bf16(128, NP, true, false);
            const uint32_t ring_a = ptx::smem_u32(ring);
            const uint32_t q_a = ptx::smem_u32(qbuf);
            const uint32_t p_a = ptx::smem_u32(pbuf);

            // scores: S^T[tile row, n] = sum_k K_tile[row, k] * Q[n, k]
            auto issue_S = [&](const TileInfo& ti, int jj) -> bool {
                if (ti.first && !ptx::mbar_wait(q_full, ti.seg & 1, abort_flag)) return false;
                const int sb = jj & 1;
                if (!ptx::mbar_wait(&s_empty[sb], ((jj >> 1) & 1) ^ 1, abort_flag)) return false;
                ptx::tc_fence_after();
                const int ksteps = p.dk[ti.k] >> 4;
                for (int c = 0; c < ti.nK; ++c) {
                    const uint32_t li = ti.ld0 + c;
                    const int slot = li % p.nslot;
                    if (!ptx::mbar_wait(&full[slot], (li / p.nslot) & 1, abort_flag)) return false;
                    ptx::tc_fence_after();
                    const int kn = min(8, ksteps - c * 8);
                    for (int kk = 0; kk < kn; ++kk) {
                        const uint32_t a = ring_a + slot * kSlot + (kk >> 2) * kBox + (kk & 3) * 32;
                        const int kg = c * 8 + kk;
                        const uint32_t bq = q_a + (kg >> 2) * (NQ * 128) + (kg & 3) * 32;
                        ptx::mma_bf16(t_S + sb * NQ, ptx::sdesc_sw128(a, 16, 1024),
                                      ptx::sdesc_sw128(bq, 16, 1024), idS, (c | kk) != 0 ? 1u : 0u);
                    }
                    ptx::mma_commit(&empty[slot]);
                }
                ptx::mma_commit(&s_full[sb]);
                if (ti.last) ptx::mma_commit(q_empty);
                return true;
            };
            // values: acc^T[value row, n] += V_tile[:, value row]^T . P^T  (hi and lo parts of P)
            auto issue_V = [&](const TileInfo& ti, int jj) -> bool {
                const int pb = jj % p.npbuf;
                if (!ptx::mbar_wait(&p_full[pb], (jj / p.npbuf) & 1, abort_flag)) return false;
                if (ti.first && ti.seg > 0 && !ptx::mbar_wait(acc_empty, (ti.seg - 1) & 1, abort_flag))
                    return false;
                ptx::tc_fence_after();
                const uint32_t phi = p_a + pb * (2 * NP * 256);
                const uint32_t plo = phi + NP * 256;
                for (int c = 0; c < ti.nV; ++c) {
                    const uint32_t li = ti.ld0 + ti.nK + c;
                    const int slot = li % p.nslot;
                    if (!ptx::mbar_wait(&full[slot], (li / p.nslot) & 1, abort_flag)) return false;
                    ptx::tc_fence_after();
                    for (int kk = 0; kk < 8; ++kk) {
                        const uint64_t ad = ptx::sdesc_sw128(ring_a + slot * kSlot + kk * 2048, kBox, 1024);
                        const uint32_t boff = (kk >> 2) * (NP * 128) + (kk & 3) * 32;
                        const uint32_t accum = (ti.first && kk == 0) ? 0u : 1u;
                        ptx::mma_bf16(t_acc + c * NP, ad, ptx::sdesc_sw128(phi + boff, 16, 1024), idV, accum);
                        ptx::mma_bf16(t_acc + c * NP, ad, ptx::sdesc_sw128(plo + boff, 16, 1024), idV, 1u);
                    }
                    ptx::mma_commit(&empty[slot]);
                }
                ptx::mma_commit(&p_empty[pb]);
                if (ti.last) ptx::mma_commit(acc_full);
                return true;
            };

            bool ok = true;
            int jS = 0, jV = 0, seg = 0;
            uint32_t ld = 0;
            TileInfo pend;
            bool has_pend = false;
            for (int u = u0; ok && u < u1; ++seg) {
                const Piece pc = piece_at(p, u, u1);
                for (int t = pc.t0; ok && t < pc.t0 + pc.n; ++t) {
                    TileInfo ti;
                    ti.k = pc.k;
                    ti.nK = (p.dk[pc.k] + 127) >> 7;
                    ti.nV = (p.dv[pc.k] + 127) >> 7;
                    ti.ld0 = ld;
                    ti.first = (t == pc.t0);
                    ti.last = (t == pc.t0 + pc.n - 1);
                    ti.seg = seg;
                    ld += ti.nK + ti.nV;
                    ok = issue_S(ti, jS++);
                    if (ok && has_pend) {
                        ok = issue_V(pend, jV++);
                        has_pend = false;
                    }
                    if (ok) {
                        if (p.lookahead) {
                            pend = ti;
                            has_pend = true;
                        } else {
                            ok = issue_V(ti, jV++);
                        }
                    }
                }
                u += pc.n;
            }
            if (ok && has_pend) ok = issue_V(pend, jV++);
            ptx::mma_commit(drain);   // arrives once every MMA issued above has completed
        }
    } else {
        // ----------------------------------------------------------------- softmax
        const int tid = threadIdx.x - 64;   // 0..127
        const int q4 = warp & 3;            // TMEM lane quadrant this warp may access
        const int myrow = q4 * 32 + lane;   // tile row (S) / value row (acc) of this thread
        const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
        const int G = p.G;
        float l_part[NP];

        pdl_wait();   // q_lat / q_rot are written by the preceding kernel

        // bf16 high / low parts of the query operand of segment (b, k)
        auto write_q = [&](int b, int k) {
            const int dk = p.dk[k];
            const float* src = (k == 0 ? p.q_lat : p.q_rot) + (size_t)b * p.Hq * dk;
            const int units = dk >> 3;
            for (int task = tid; task < NP * units; task += 128) {
                const int h = task / units, u = task - h * units;
                float v[8];
                if (h < p.Hq) {
                    const float4* s4 = reinterpret_cast<const float4*>(src + (size_t)h * dk + u * 8);
                    const float4 a = s4[0], c = s4[1];
                    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
                    v[4] = c.x; v[5] = c.y; v[6] = c.z; v[7] = c.w;
                } else {
#pragma unroll
                    for (int i = 0; i < 8; ++i) v[i] = 0.f;
                }
                uint32_t hi[4], lo[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const __nv_bfloat16 h0 = __float2bfloat16_rn(v[2 * i]);
                    const __nv_bfloat16 h1 = __float2bfloat16_rn(v[2 * i + 1]);
                    const __nv_bfloat16 l0 = __float2bfloat16_rn(v[2 * i] - __bfloat162float(h0));
                    const __nv_bfloat16 l1 = __float2bfloat16_rn(v[2 * i + 1] - __bfloat162float(h1));
                    hi[i] = (uint32_t)__bfloat16_as_ushort(h0) | ((uint32_t)__bfloat16_as_ushort(h1) << 16);
                    lo[i] = (uint32_t)__bfloat16_as_ushort(l0) | ((uint32_t)__bfloat16_as_ushort(l1) << 16);
                }
                *reinterpret_cast<uint4*>(qbuf + ptx::sw128_offset(h, u * 8, NQ)) =
                    make_uint4(hi[0], hi[1], hi[2], hi[3]);
                *reinterpret_cast<uint4*>(qbuf + ptx::sw128_offset(NP + h, u * 8, NQ)) =
                    make_uint4(lo[0], lo[1], lo[2], lo[3]);
            }
            ptx::fence_proxy_async_smem();
            ptx::named_bar(1, 128);
            if (tid == 0) ptx::mbar_arrive(q_full);
        };

        // A failed wait (abort) does not leave the loop: every softmax thread keeps
        // the same control flow so the named barriers stay matched; results are
        // poisoned at the end instead.
        if (u0 < u1) {
            const Piece p0 = piece_at(p, u0, u1);
            write_q(p0.b, p0.k);
        }
        int j = 0, seg = 0;
        for (int u = u0; u < u1; ++seg) {
            const Piece pc = piece_at(p, u, u1);
            const int k = pc.k;
            const int nMB = (p.dv[k] + 127) >> 7;
            if (tid < NP) m_run[tid] = -INFINITY;
#pragma unroll
            for (int h = 0; h < NP; ++h) l_part[h] = 0.f;
            ptx::named_bar(1, 128);
            for (int t = pc.t0; t < pc.t0 + pc.n; ++t, ++j) {
                const int sb = j & 1;
                ptx::mbar_wait(&s_full[sb], (j >> 1) & 1, abort_flag);
                ptx::tc_fence_after();
                float s[NP];
#pragma unroll
                for (int hc = 0; hc < NP / 16; ++hc) {
                    float hi[16], lo[16];
                    ptx::tmem_ld16x2(t_S + lane_off + sb * NQ + hc * 16,
                                     t_S + lane_off + sb * NQ + NP + hc * 16, hi, lo);
#pragma unroll
                    for (int i = 0; i < 16; ++i) s[hc * 16 + i] = (hi[i] + lo[i]) * p.scale_log2;
                }
                ptx::tc_fence_before();
                ptx::mbar_arrive(&s_empty[sb]);
                // mask rows past the segment end, padding heads and, for raw rows,
                // the heads of other KV groups
                const int row = t * kTile + myrow;
                const bool valid = row < p.rows[k];
                const int g = (k == 0) ? -1 : row % p.Hkv;
#pragma unroll
                for (int h = 0; h < NP; ++h) {
                    const bool keep = valid && h < p.Hq && (g < 0 || h / G == g);
                    if (!keep) s[h] = -INFINITY;
                }
                // per-head maximum over the tile's 128 rows
#pragma unroll
                for (int h = 0; h < NP; ++h) {
                    float v = s[h];
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
                    if (lane == 0) red[q4 * NP + h] = v;
                }
                volatile int* resc = &flag[1 + (j & 1)];
                if (tid == 0) *resc = 0;
                ptx::named_bar(1, 128);
                if (tid < NP) {
                    const float M = fmaxf(fmaxf(red[tid], red[NP + tid]), fmaxf(red[2 * NP + tid], red[3 * NP + tid]));
                    const float mo = m_run[tid];
                    float a = 1.f;
                    // lazy rescale: keep the reference max unless it grew by more than 8 (x256)
                    if (M > mo + 8.f) {
                        a = (mo == -INFINITY) ? 0.f : exp2f(mo - M);
                        m_run[tid] = M;
                        *resc = 1;
                    }
                    alpha_s[tid] = a;
                }
                ptx::named_bar(1, 128);
                if (*resc) {
#pragma unroll
                    for (int h = 0; h < NP; ++h) l_part[h] *= alpha_s[h];
                    if (t > pc.t0) {
                        // the accumulator holds earlier tiles of this piece: wait for
                        // their value MMAs, then scale each head's column
                        const int jp = j - 1;
                        ptx::mbar_wait(&p_empty[jp % p.npbuf], (jp / p.npbuf) & 1, abort_flag);
                        ptx::tc_fence_after();
                        for (int c = 0; c < nMB; ++c) {
#pragma unroll
                            for (int hc = 0; hc < NP / 16; ++hc) {
                                float v[16];
                                const uint32_t ta = t_acc + lane_off + c * NP + hc * 16;
                                ptx::tmem_ld16(ta, v);
#pragma unroll
                                for (int i = 0; i < 16; ++i) v[i] *= alpha_s[hc * 16 + i];
                                ptx::tmem_st16(ta, v);
                            }
                        }
                        ptx::tc_fence_before();
                    }
                }
                // probabilities against the reference max, as bf16 high + low parts
                const int pb = j % p.npbuf;
                if (j >= p.npbuf) ptx::mbar_wait(&p_empty[pb], ((j / p.npbuf) - 1) & 1, abort_flag);
                uint8_t* phi = pbuf + pb * (2 * NP * 256);
                uint8_t* plo = phi + NP * 256;
#pragma unroll
                for (int h = 0; h < NP; ++h) {
                    const float pr = (s[h] == -INFINITY) ? 0.f : exp2f(s[h] - m_run[h]);
                    l_part[h] += pr;
                    const __nv_bfloat16 ph = __float2bfloat16_rn(pr);
                    const __nv_bfloat16 pl = __float2bfloat16_rn(pr - __bfloat162float(ph));
                    const uint32_t off = ptx::sw128_offset(h, myrow, NP);
                    *reinterpret_cast<__nv_bfloat16*>(phi + off) = ph;
                    *reinterpret_cast<__nv_bfloat16*>(plo + off) = pl;
                }
                ptx::fence_proxy_async_smem();
                ptx::tc_fence_before();
                ptx::mbar_arrive(&p_full[pb]);
            }
            // the next piece's query operand goes in before this piece's partial is
            // written, so its score MMAs overlap the write-out
            if (u + pc.n < u1) {
                ptx::mbar_wait(q_empty, seg & 1, abort_flag);
                const Piece nx = piece_at(p, u + pc.n, u1);
                write_q(nx.b, nx.k);
            }
            // ---- partial of (CTA, piece): running max, sum and accumulator
            ptx::mbar_wait(acc_full, seg & 1, abort_flag);
            ptx::tc_fence_after();
#pragma unroll
            for (int h = 0; h < NP; ++h) {
                float v = l_part[h];
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
                if (lane == 0) red[q4 * NP + h] = v;
            }
            ptx::named_bar(1, 128);
            const int slot = p.slot_base[cta] + seg;
            if (tid < p.Hq) {
                const float L = red[tid] + red[NP + tid] + red[2 * NP + tid] + red[3 * NP + tid];
                p.ml[((size_t)slot * 2) * p.Hq + tid] = m_run[tid];
                p.ml[((size_t)slot * 2 + 1) * p.Hq + tid] = L;
            }
            if (tid == 0) p.kind[slot] = (k == 0) ? 0 : 1;
            const int dv = p.dv[k];
            for (int c = 0; c < nMB; ++c) {
                const int r = c * 128 + myrow;
#pragma unroll
                for (int hc = 0; hc < NP / 16; ++hc) {
                    float v[16];
                    ptx::tmem_ld16(t_acc + lane_off + c * NP + hc * 16, v);
                    if (r < dv) {
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            const int h = hc * 16 + i;
                            if (h < p.Hq) p.acc[((size_t)slot * p.Hq + h) * p.Dmax + r] = v[i];
                        }
                    }
                }
            }
            ptx::tc_fence_before();
            ptx::mbar_arrive(acc_empty);
            ptx::named_bar(1, 128);
            u += pc.n;
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
        ptx::tmem_dealloc(tmem, p.tmem_cols);
    }
    if (*abort_flag && warp >= 2) {
        // a wait ran out: poison this CTA's partials so the result is NaN, not stale
        const int tid = threadIdx.x - 64;
        int npieces = 0;
        for (int u = u0; u < u1;) {
            const Piece pc = piece_at(p, u, u1);
            u += pc.n;
            ++npieces;
        }
        for (int i = tid; i < npieces * p.Hq; i += 128) {
            const int slot = p.slot_base[cta] + i / p.Hq;
            p.ml[((size_t)slot * 2 + 1) * p.Hq + (i % p.Hq)] = __int_as_float(0x7fc00000);
        }
    }
}

// ------------------------------------------------------------------------ host

// Shared-memory plan of one launch.
struct SmemPlan {
    int NP, nslot, npbuf, lookahead, q_cols;
    uint32_t off_q, off_p, off_bar, off_red, total, tmem_cols;
    bool ok;
};

int round_up(int x, int m) { return (x + m - 1) / m * m; }

SmemPlan plan_smem(int Hq, const int dk[kNumKinds], const int dv[kNumKinds], const int rows[kNumKinds]) {
    SmemPlan s{};
    s.NP = round_up(Hq, 16);
    const int NQ = 2 * s.NP;
    int qc = 0, nmb = 0, need = 0;
    for (int k = 0; k < kNumKinds; ++k) {
        if (rows[k] <= 0) continue;
        qc = std::max(qc, dk[k]);
        nmb = std::max(nmb, (dv[k] + 127) / 128);
        need = std::max(need, (dk[k] + 127) / 128 + (dv[k] + 127) / 128);
    }
    s.q_cols = round_up(qc, 64);
    const int q_bytes = NQ * s.q_cols * 2;
    const int tmem = 2 * NQ + nmb * s.NP;
    s.tmem_cols = 32;
    while ((int)s.tmem_cols < tmem) s.tmem_cols *= 2;
    s.ok = false;
    if (s.NP > 64 || s.tmem_cols > 512) return s;
    for (s.npbuf = 2; s.npbuf >= 1; --s.npbuf) {
        const int p_bytes = s.npbuf * 2 * s.NP * 256;
        const int nbars = 2 * 16 + 13;   // up to 16 ring slots
        const int misc = nbars * 8 + (6 * s.NP + 16) * 4 + 1024;   // + alignment slack
        const int avail = kSmemMax - q_bytes - p_bytes - misc;
        s.nslot = std::min(16, avail / kSlot);
        if (s.nslot >= 2) break;
    }
    if (s.nslot < 2) return s;
    s.lookahead = (s.nslot >= need) ? 1 : 0;
    s.off_q = s.nslot * kSlot;
    s.off_p = s.off_q + q_bytes;
    s.off_bar = s.off_p + s.npbuf * 2 * s.NP * 256;
    s.off_red = s.off_bar + round_up((2 * s.nslot + 13) * 8, 16);
    s.total = s.off_red + (6 * s.NP + 16) * 4 + 1024;
    s.ok = s.total <= (uint32_t)kSmemMax;
    return s;
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

// 3-D bf16 tensor [B][rows][cols] (cols contiguous) read in boxes of 128 rows x 64
// columns with the 128-byte swizzle; rows/columns past the end read as zero.
bool make_map(CUtensorMap* tm, const void* base, int cols, int rows, int B) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)rows, (cuuint64_t)B};
    cuuint64_t strides[2] = {(cuuint64_t)cols * 2, (cuuint64_t)cols * 2 * (cuuint64_t)rows};
    cuuint32_t box[3] = {64, (cuuint32_t)kTile, 1};
    cuuint32_t es[3] = {1, 1, 1};
    return fn(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int sm_count() {
    int dev = 0, n = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    return n > 0 ? n : 148;
}

// Work plan: contiguous unit ranges per CTA with balanced bytes, partial slots per
// (CTA, segment piece) and per batch element.
struct WorkPlan {
    int n_ctas = 0;
    std::vector<int> u_begin, slot_base, batch_slot;
    int slots = 0;
};

WorkPlan make_plan(int B, const int tiles[kNumKinds], const int cost[kNumKinds], int max_ctas) {
    // runs of equal-cost units in unit order (batch-major, then kind)
    std::vector<std::pair<int, int>> runs;   // (count, cost)
    int64_t total = 0;
    int cmax = 1;
    for (int b = 0; b < B; ++b)
        for (int k = 0; k < kNumKinds; ++k)
            if (tiles[k] > 0) {
                runs.push_back({tiles[k], cost[k]});
                total += (int64_t)tiles[k] * cost[k];
                cmax = std::max(cmax, cost[k]);
            }
    int64_t units = 0;
    for (auto& r : runs) units += r.first;
    const int G = (int)std::max<int64_t>(1, std::min<int64_t>(max_ctas, units));
    // number of CTAs greedy packing needs with per-CTA budget T
    auto count = [&](int64_t T) {
        int ctas = 1;
        int64_t cur = 0;
        for (auto& r : runs) {
            int n = r.first;
            while (n > 0) {
                int64_t room = (T - cur) / r.second;
                if (room == 0) {
                    ++ctas;
                    cur = 0;
                    room = T / r.second;
                }
                const int take = (int)std::min<int64_t>(n, room);
                cur += (int64_t)take * r.second;
                n -= take;
            }
        }
        return ctas;
    };
    int64_t lo = std::max<int64_t>(cmax, (total + G - 1) / G), hi = std::max<int64_t>(lo, total);
    while (lo < hi) {
        const int64_t mid = (lo + hi) / 2;
        if (count(mid) <= G) hi = mid;
        else lo = mid + 1;
    }
    const int64_t T = lo;
    WorkPlan w;
    w.u_begin.push_back(0);
    int64_t cur = 0, u = 0;
    for (auto& r : runs) {
        int n = r.first;
        while (n > 0) {
            int64_t room = (T - cur) / r.second;
            if (room == 0) {
                w.u_begin.push_back((int)u);
                cur = 0;
                room = T / r.second;
            }
            const int take = (int)std::min<int64_t>(n, room);
            cur += (int64_t)take * r.second;
            u += take;
            n -= take;
        }
    }
    w.u_begin.push_back((int)u);
    w.n_ctas = (int)w.u_begin.size() - 1;
    // partial slots: one per (CTA, segment piece), consecutive; batch b owns a
    // contiguous slot range because units are batch-major
    int tiles_per_b = 0;
    for (int k = 0; k < kNumKinds; ++k) tiles_per_b += tiles[k];
    w.batch_slot.assign(B + 1, -1);
    int slot = 0;
    for (int i = 0; i < w.n_ctas; ++i) {
        w.slot_base.push_back(slot);
        int uu = w.u_begin[i];
        while (uu < w.u_begin[i + 1]) {
            const int b = uu / tiles_per_b;
            int t = uu - b * tiles_per_b, k = 0;
            while (k < kNumKinds - 1 && t >= tiles[k]) {
                t -= tiles[k];
                ++k;
            }
            const int n = std::min(w.u_begin[i + 1] - uu, tiles[k] - t);
            if (w.batch_slot[b] < 0) w.batch_slot[b] = slot;
            ++slot;
            uu += n;
        }
    }
    w.batch_slot[B] = slot;
    w.slots = slot;
    return w;
}

struct PlanKey {
    int B, tiles[kNumKinds], cost[kNumKinds], max_ctas;
    bool operator<(const PlanKey& o) const {
        return std::tie(B, tiles[0], tiles[1], tiles[2], cost[0], cost[1], cost[2], max_ctas) <
               std::tie(o.B, o.tiles[0], o.tiles[1], o.tiles[2], o.cost[0], o.cost[1], o.cost[2], o.max_ctas);
    }
};

const WorkPlan& cached_plan(int B, const int tiles[kNumKinds], const int cost[kNumKinds], int max_ctas) {
    static std::mutex mu;
    static std::map<PlanKey, WorkPlan> cache;
    PlanKey key{B, {tiles[0], tiles[1], tiles[2]}, {cost[0], cost[1], cost[2]}, max_ctas};
    std::lock_guard<std::mutex> g(mu);
    auto it = cache.find(key);
    if (it != cache.end()) return it->second;
    if (cache.size() > 256) cache.clear();
    return cache.emplace(key, make_plan(B, tiles, cost, max_ctas)).first->second;
}

template <int NP>
cudaError_t launch_decode(const TcParams& prm, int grid, uint32_t smem, cudaStream_t st) {
    static bool attr_done = false;
    if (!attr_done) {
        cudaError_t e = cudaFuncSetAttribute(tc_decode_kernel<NP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             kSmemMax);
        if (e != cudaSuccess) return e;
        attr_done = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, tc_decode_kernel<NP>, prm);
}

// Kinds of key rows of one call: rows / widths per batch element and operands.
struct Kinds {
    int rows[kNumKinds] = {0, 0, 0};
    int dk[kNumKinds] = {0, 0, 0};
    int dv[kNumKinds] = {0, 0, 0};
    const void* K[kNumKinds] = {nullptr, nullptr, nullptr};
    const void* V[kNumKinds] = {nullptr, nullptr, nullptr};
};

Kinds kinds_of(const TcCall& c) {
    Kinds s;
    if (c.which == SLIMKV_LATENT) {
        if (c.N_b > 0) {
            s.rows[0] = c.N_b;
            s.dk[0] = c.r_k;
            s.dv[0] = c.r_v;
            s.K[0] = c.C_K;
            s.V[0] = c.C_V;
        }
        if (c.W > 0) {
            s.rows[1] = c.W * c.Hkv;
            s.K[1] = c.K_raw;
            s.V[1] = c.V_raw;
        }
    } else if (c.which == SLIMKV_RECONSTRUCT) {
        s.rows[1] = c.N_b * c.Hkv;
        s.K[1] = c.kb;
        s.V[1] = c.vb;
        if (c.W > 0) {
            s.rows[2] = c.W * c.Hkv;
            s.K[2] = c.K_raw;
            s.V[2] = c.V_raw;
        }
    } else {
        s.rows[1] = c.W * c.Hkv;
        s.K[1] = c.K_raw;
        s.V[1] = c.V_raw;
    }
    for (int k = 1; k < kNumKinds; ++k)
        if (s.rows[k] > 0) s.dk[k] = s.dv[k] = c.d;
    return s;
}

}  // namespace

bool tc_supported(int Hq, int Hkv, int d, int N_b, int r_k, int r_v) {
    if (d != 128 || Hq > 64 || Hkv > 128) return false;
    int rows[kNumKinds] = {N_b, 1, 1}, dk[kNumKinds] = {r_k, d, d}, dv[kNumKinds] = {r_v, d, d};
    if (N_b <= 0) rows[0] = 0;
    return plan_smem(Hq, dk, dv, rows).ok;
}

cudaError_t tc_run(const TcCall& c, cudaStream_t st) {
    typedef __nv_bfloat16 bf16;
    const bool lat = c.which == SLIMKV_LATENT && c.N_b > 0;
    cudaError_t e = launch_qproj<bf16>((const bf16*)c.q, lat ? (const bf16*)c.U_K : nullptr, c.q_pos, c.q_rot,
                                       lat ? c.q_lat : nullptr, c.B, c.Hq, c.Hkv, c.d, c.r_k, c.rope_base, st,
                                       true);
    if (e != cudaSuccess) return e;
    if (c.which == SLIMKV_RECONSTRUCT) {
        // plain launches (no early trigger): the decode below reads K_b / V_b
        // before its own dependency wait, so they must be complete when it starts
        const int rows = c.B * c.N_b, n = c.Hkv * c.d;
        e = launch_reconstruct_gemm((const bf16*)c.C_K, (const bf16*)c.U_K, (bf16*)c.kb, rows, n, c.r_k, st);
        if (e != cudaSuccess) return e;
        e = launch_reconstruct_gemm((const bf16*)c.C_V, (const bf16*)c.U_V, (bf16*)c.vb, rows, n, c.r_v, st);
        if (e != cudaSuccess) return e;
    }
    const Kinds s = kinds_of(c);
    const SmemPlan sp = plan_smem(c.Hq, s.dk, s.dv, s.rows);
    if (!sp.ok) return cudaErrorInvalidValue;

    TcParams prm;   // copied into the launch's parameter space
    memset(&prm, 0, sizeof(prm));
    int tiles[kNumKinds], cost[kNumKinds];
    prm.tiles_per_b = 0;
    for (int k = 0; k < kNumKinds; ++k) {
        prm.rows[k] = s.rows[k];
        prm.dk[k] = s.dk[k];
        prm.dv[k] = s.dv[k];
        tiles[k] = s.rows[k] > 0 ? (s.rows[k] + kTile - 1) / kTile : 0;
        prm.tiles[k] = tiles[k];
        prm.tiles_per_b += tiles[k];
        // cost of a tile: the 32 KB slots it streams (+1 for its fixed per-tile work)
        cost[k] = (s.dk[k] + 127) / 128 + (s.dv[k] + 127) / 128 + 1;
        if (s.rows[k] > 0) {
            if (!make_map(&prm.tm[2 * k], s.K[k], s.dk[k], s.rows[k], c.B)) return cudaErrorInvalidValue;
            if (!make_map(&prm.tm[2 * k + 1], s.V[k], s.dv[k], s.rows[k], c.B)) return cudaErrorInvalidValue;
        }
    }
    const WorkPlan& w = cached_plan(c.B, tiles, cost, std::min(kMaxCtas, sm_count()));
    if (w.slots > c.slots) return cudaErrorInvalidValue;
    prm.B = c.B;
    prm.Hq = c.Hq;
    prm.Hkv = c.Hkv;
    prm.G = c.Hq / c.Hkv;
    prm.scale_log2 = c.scale_log2;
    prm.q_lat = c.q_lat;
    prm.q_rot = c.q_rot;
    prm.acc = c.acc;
    prm.ml = c.ml;
    prm.kind = c.kind;
    prm.Dmax = c.Dmax;
    prm.nslot = sp.nslot;
    prm.npbuf = sp.npbuf;
    prm.lookahead = sp.lookahead;
    prm.q_cols = sp.q_cols;
    prm.off_q = sp.off_q;
    prm.off_p = sp.off_p;
    prm.off_bar = sp.off_bar;
    prm.off_red = sp.off_red;
    prm.tmem_cols = sp.tmem_cols;
    for (int i = 0; i <= w.n_ctas; ++i) prm.u_begin[i] = w.u_begin[i];
    for (int i = 0; i < w.n_ctas; ++i) prm.slot_base[i] = w.slot_base[i];

    timer_before(st);
    switch (sp.NP) {
        case 16: e = launch_decode<16>(prm, w.n_ctas, sp.total, st); break;
        case 32: e = launch_decode<32>(prm, w.n_ctas, sp.total, st); break;
        case 48: e = launch_decode<48>(prm, w.n_ctas, sp.total, st); break;
        case 64: e = launch_decode<64>(prm, w.n_ctas, sp.total, st); break;
        default: e = cudaErrorInvalidValue;
    }
    timer_after(st);
    if (e != cudaSuccess) return e;

    CombineArgs cb;
    cb.B = c.B;
    cb.Hq = c.Hq;
    cb.Hkv = c.Hkv;
    cb.d = c.d;
    cb.r_v = c.r_v;
    cb.Dmax = c.Dmax;
    cb.U_V = lat ? c.U_V : nullptr;
    cb.acc = c.acc;
    cb.ml = c.ml;
    cb.kind = c.kind;
    cb.out = c.out;
    for (int b = 0; b <= c.B; ++b) cb.slot_begin[b] = w.batch_slot[b];
    return launch_combine<bf16>(cb, st, true);
}

}  // namespace slimkv

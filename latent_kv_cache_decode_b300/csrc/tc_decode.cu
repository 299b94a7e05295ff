// Tensor-core split-context decode for SlimKV on sm_103a (tcgen05 + TMA).
//
// "Can SlimKV compress KV cache jointly across tokens and features", section
// "Latent-space attention removes the rebuild step": per query head the scores
// are (RoPE(q) U_K^(g)) C_K^T against the RoPE-free latent beacon keys and
// RoPE(q) K_raw^T against the raw window, in one softmax; values aggregate as
// (A C_V) U_V^(g)T + A V_raw, the latent aggregate taken before the up-projection.
//
// Work layout. A "segment" is all key rows of one kind for one batch element:
//   latent: the N_b beacons of C_K[b] / C_V[b] (widths r_k / r_v), shared by
//           every query head (one latent cache per layer for all KV heads);
//   raw:    the tokens of KV head g in K[b] / V[b] (width d), read by the G
//           query heads of group g only; there is one raw segment per group.
// A "tile" (unit of work) is 128 rows of a segment. A host planner gives every
// CTA a contiguous, byte-balanced run of tiles (flash-decoding split of the
// context); a run's part inside one segment is a "piece", which produces one
// partial (m, l, acc) in the workspace, merged later by the combine kernel.
//
// Per tile, with the query operand Q = [q_hi ; q_lo] (bf16 high and low parts of
// the float32 query, which already carries scale * log2(e)), stacked along N:
//   scores  S^T[row, (part, head)] = tile[row, :] . Q[(part, head), :]
//           (one tcgen05.mma per 16-wide k-step, M = 128 rows, N = 2 x heads); the
//           softmax adds the two parts. The latent query is rounded to bf16 in one
//           part: latent scores are not peaked, so its rounding stays far inside the
//           error bar, while the raw window (whose keys can be large) keeps both;
//   softmax P[row, head] = exp2(S^T - m_ref[head]), rounded to bf16 (the rounding
//           of P, unlike that of the query, stays far inside the error bar: the
//           relative error of a weight is at most 2^-9 and averages out);
//   values  acc^T[value dim, head] += tile_V[:, value dim]^T . P (M = 128 value dims).
// Issuing few, wide MMAs matters: the issuing thread, not the tensor core, is the
// limit for narrow ones.
// m_ref is a lazy running maximum: it moves (and the TMEM accumulator is rescaled)
// only when some score exceeds it by more than kLazy (log2 units), which one warp
// vote per tile detects; so most tiles need no cross-row reduction at all.
//
// Roles (224 threads): warp 0 issues TMA loads into a ring of 32 KB slots, warp 1
// issues the score MMAs and owns TMEM, warp 6 issues the value MMAs, warps 2-5 (one
// per TMEM lane quadrant; thread = tile row) run the softmax and write the partials.
// The hot loops are kept small: with four roles running different code on one SM,
// the instruction cache, not the arithmetic, limits a kernel whose loops the
// compiler unrolls freely, so runtime-trip loops stay rolled and rare paths are
// out of line.
#include <cuda.h>
#include <string.h>

#include <algorithm>
#include <map>
#include <memory>
#include <mutex>
#include <tuple>
#include <vector>

#include "../../include/slimkv.h"
#include "slimkv_internal.cuh"
#include "tc_decode.cuh"
#include "tc_ptx.cuh"
#include "work_plan.h"

namespace slimkv {

namespace {

constexpr int kTile = 128;            // rows per tile (MMA M)
constexpr int kBox = 16384;           // one TMA box: 128 rows x 64 bf16 columns, 128B-swizzled
constexpr int kSlot = 2 * kBox;       // ring slot: 128 rows x 128 columns
constexpr int kThreads = 224;
constexpr int kSmemMax = 227 * 1024;  // dynamic shared memory one CTA may use
constexpr int kNumKinds = 3;          // latent, raw source 0, raw source 1
constexpr int kNG = 16;               // heads of a raw tile's query operand (the group's heads, padded)
// m_ref moves only when a score exceeds it by more than this (log2 units). P values up
// to 2^20 keep bf16's relative precision and stay far from fp32 overflow in the
// accumulator and row sums, so a generous margin keeps the rescale path (which waits
// for the previous value MMAs) off the common path even for peaked score distributions.
constexpr float kLazy = 20.f;
constexpr int kPAtom = 128 * 32;      // bytes of one 16-head column block of P per 128 rows (x 32 B)
constexpr int kRawCols = 128;         // columns of a raw tile row (d = 64 rows are zero-padded)
constexpr int kRBRaw = 2;             // 128-row blocks per raw tile: a raw tile is 256 tokens of one KV head
constexpr int kR = 16;                // depth of the per-tile barrier rings
constexpr int kMaxSlots = 16;

struct TcParams {
    CUtensorMap tm[2 * kNumKinds];    // per kind: keys, values (latent 3-D, raw 4-D)
    int B, Hq, Hkv, G;
    int rows[kNumKinds];              // rows of one segment (0 = kind absent)
    int tiles[kNumKinds];             // tiles of one segment
    int ngroups[kNumKinds];           // segments of this kind per batch element
    int dk[kNumKinds], dv[kNumKinds]; // key / value width
    int rb[kNumKinds];                // 128-row blocks per tile (1 latent, kRBRaw raw)
    int tiles_per_b;
    const uint8_t* lat_img;           // query images (operand layout: latent bf16, raw bf16 hi / lo)
    const uint8_t* raw_img;
    uint32_t lat_img_bytes, raw_img_bytes;
    float* acc;                       // [slots, Hq, Dmax]
    float* ml;                        // [slots, 2, Hq]
    int* kind;                        // [slots]
    int Dmax;
    int nslot;                        // ring slots of 32 KB
    int npbuf;                        // P buffers: 2, or 1 when the ring needs their room
    int accbuf;                       // TMEM accumulator buffers (1 or 2)
    int accstride;                    // TMEM columns of one accumulator buffer
    uint32_t off_q, off_p, off_bar, off_red;
    uint32_t tmem_cols;
    // ALiBi (alibi != 0): head h adds slope_l2[h] * (key position - q_pos[b]) to its scores
    // (log2 units); beacon j sits at j * ratio + ratio - 1, window slot s at the latest
    // position = s mod W not above q_pos[b]
    int alibi, ratio;
    const int32_t* q_pos;
    float slope_l2[64];
    unsigned long long* aborts;       // device counter of CTAs that gave up on a wait
    int d_raw;                        // head dimension of the raw rows (64 or 128; tiles are 128 wide)
    int withhold_cta;                 // test hook: this CTA skips its first key load (-1: none)
    int u_begin[kMaxCtas + 1];        // CTA i owns units (tiles) [u_begin[i], u_begin[i+1])
    int slot_base[kMaxCtas];          // first partial slot of CTA i
};

// The run of a CTA's units that starts at u and stays inside one segment.
struct Piece {
    int b, k, g, t0, n;
};
__device__ __forceinline__ Piece piece_at(const TcParams& p, int u, int u1) {
    Piece r;
    r.b = u / p.tiles_per_b;
    int t = u - r.b * p.tiles_per_b;
    int k = 0;
    for (; k < kNumKinds - 1; ++k) {
        const int span = p.ngroups[k] * p.tiles[k];
        if (t < span) break;
        t -= span;
    }
    r.k = k;
    r.g = t / p.tiles[k];
    r.t0 = t - r.g * p.tiles[k];
    r.n = min(u1 - u, p.tiles[k] - r.t0);
    return r;
}

// Walks a CTA's tiles in order: tile j (0-based), its piece index and position.
struct TileIter {
    const TcParams* p;
    int u, u1;
    Piece pc;
    int t, j, piece;
    __device__ __forceinline__ void init(const TcParams& prm, int u0, int u1_) {
        p = &prm;
        u = u0;
        u1 = u1_;
        j = 0;
        piece = 0;
        if (u < u1) {
            pc = piece_at(prm, u, u1);
            t = pc.t0;
        }
    }
    __device__ __forceinline__ bool valid() const { return u < u1; }
    __device__ __forceinline__ bool first() const { return t == pc.t0; }
    __device__ __forceinline__ void next() {
        ++j;
        ++t;
        if (t == pc.t0 + pc.n) {
            u += pc.n;
            ++piece;
            if (u < u1) {
                pc = piece_at(*p, u, u1);
                t = pc.t0;
            }
        }
    }
};

// Ring position s (< 2 n) modulo n.
__device__ __forceinline__ int ring_wrap(int s, int n) { return s >= n ? s - n : s; }

// Query operand image of a piece: the latent image of its batch element, or the raw
// image of its (batch element, KV group).
__device__ __forceinline__ void query_image(const TcParams& p, const Piece& pc, const uint8_t*& src,
                                            uint32_t& bytes) {
    if (pc.k == 0) {
        src = p.lat_img + (size_t)pc.b * p.lat_img_bytes;
        bytes = p.lat_img_bytes;
    } else {
        src = p.raw_img + ((size_t)pc.b * p.Hkv + pc.g) * p.raw_img_bytes;
        bytes = p.raw_img_bytes;
    }
}

// Barriers (all in shared memory), per tile j of the CTA, ring index j % kR:
//   kready  K tile (and, for a piece's first tile, its query image) landed   [TMA tx]
//   vready  V tile landed and P(j) written by the softmax warps             [TMA tx + 128 arrivals]
//   kfree   score MMAs of tile j complete: K slots reusable, S(j) readable  [commit]
//   vfree   value MMAs of tile j complete: V slots and P buffer reusable     [commit]
//   accfree[2] the softmax warps have read a piece's accumulator             [128 arrivals]
struct Bars {
    uint64_t* kready;
    uint64_t* vready;
    uint64_t* kfree;
    uint64_t* vfree;
    uint64_t* accfree;
    uint64_t* drain;
    uint64_t* qready;   // the CTA's first query image landed                       [TMA tx]
};
__device__ __forceinline__ uint32_t ph_of(int j) { return ((uint32_t)j / kR) & 1u; }

// Shared state of the softmax warps.
struct SoftCtx {
    Bars bar;
    uint8_t* pbuf;
    float* red;           // [4][NP] per-warp reductions
    float* m_ref_s;       // [NP] reference max (log2 domain) of the current piece
    float* alpha_s;       // [NP] rescale factors
    volatile int* flags;  // [2][4] per-tile "needs a new reference max" votes
    volatile int* abort;
    uint32_t t_S, t_accp, lane_off;   // t_accp: accumulator of the current piece
    int tid, wq, lane, myrow, nMB;
    int aw;               // TMEM columns per 128 value rows of the accumulator
    int npbuf;            // P buffers (1 or 2)
    const float* slope_s; // [NS] ALiBi slopes of the piece's score columns (log2 units)
};

// ALiBi offsets of this thread's rows in a tile (key position - query position, one per
// 128-row block); zero when ALiBi is off.
struct RowBias {
    float d[2];
};
// Add the ALiBi bias of 16 score columns (slopes at `sl`) for key offset `dk`.
__device__ __forceinline__ void add_bias(float (&x)[16], const float* sl, float dk) {
#pragma unroll
    for (int i = 0; i < 16; ++i) x[i] = fmaf(sl[i], dk, x[i]);
}


// TMEM columns of one score buffer: hi and lo scores (2 x NS columns) for each of
// the tile's row blocks; at least 64.
template <int NP> struct SBuf {
    // latent tiles: NP score columns; raw tiles: hi and lo columns of kNG heads per row block
    static constexpr int W = NP > 2 * kNG * kRBRaw ? NP : 2 * kNG * kRBRaw;
    // bytes of one P buffer: NP heads x 128 rows (latent) or kNG heads x 256 rows (raw), bf16
    static constexpr int PB = (NP > kNG * kRBRaw ? NP : kNG * kRBRaw) * 256;
};

// Scores of 16 heads of this thread's row: hi + lo parts (raw tiles) or one part.
template <bool LO, int NS>
__device__ __forceinline__ void load_scores(uint32_t tS, float (&x)[16]) {
    if (LO) {
        float lo[16];
        ptx::tmem_ld16x2(tS, tS + NS, x, lo);
#pragma unroll
        for (int i = 0; i < 16; ++i) x[i] += lo[i];
    } else {
        ptx::tmem_ld16(tS, x);
    }
}

// Reduction across the 32 lanes of 16 values per lane, one result per value:
// afterwards lane l holds the reduction of value l % 16 over all lanes. Butterfly that
// halves the values per lane at each step (15 shuffles down to one value, then one
// plain step across the two half-warps).
template <bool MAX>
__device__ __forceinline__ float warp_reduce16(float* v, int lane) {
    constexpr int N = 16;
#pragma unroll
    for (int w = N / 2; w >= 1; w /= 2) {
        const bool upper = (lane & w) != 0;
#pragma unroll
        for (int i = 0; i < w; ++i) {
            const float send = upper ? v[i] : v[i + w];
            const float keep = upper ? v[i + w] : v[i];
            const float got = __shfl_xor_sync(0xffffffffu, send, w);
            v[i] = MAX ? fmaxf(keep, got) : keep + got;
        }
    }
    float r = v[0];
#pragma unroll
    for (int w = N; w < 32; w *= 2) {
        const float got = __shfl_xor_sync(0xffffffffu, r, w);
        r = MAX ? fmaxf(r, got) : r + got;
    }
    return r;
}

// The rare path of the softmax, kept out of line so that the hot loop stays small in
// the instruction cache: a new reference maximum per head from this tile's scores,
// the rescale factors alpha = exp2(m_old - m_new), and, when the accumulator already
// holds earlier tiles of the piece (nMB > 0), the rescale of its columns once the
// previous value MMAs are done. All 128 softmax threads call it together.
template <int NS, int NP, int RB, bool LO, bool AL>
__device__ __noinline__ void softmax_new_ref(float* red, float* m_ref_s, float* alpha_s, uint64_t* vfree,
                                             volatile int* abort, uint32_t tS0, uint32_t t_acc_lane, int row0,
                                             int rows, int j, int nMB, int aw, int tid, int lane, int wq,
                                             const float* slope_s, float dk0, float dk1) {
    // per-head maximum over this warp's valid rows, then over the four warps
    float x[NS];
#pragma unroll
    for (int h = 0; h < NS; ++h) x[h] = -INFINITY;
    // (the TMEM loads are warp-collective: every lane loads, invalid rows are masked after)
#pragma unroll 1
    for (int rb = 0; rb < RB; ++rb) {
        const bool valid = row0 + rb * 128 < rows;
        const uint32_t tS = tS0 + rb * (LO ? 2 : 1) * NS;
#pragma unroll
        for (int hc = 0; hc < NS / 16; ++hc) {
            float sc[16];
            load_scores<LO, NS>(tS + hc * 16, sc);
            if (AL) add_bias(sc, slope_s + hc * 16, rb == 0 ? dk0 : dk1);
#pragma unroll
            for (int i = 0; i < 16; ++i) x[hc * 16 + i] = valid ? fmaxf(x[hc * 16 + i], sc[i]) : x[hc * 16 + i];
        }
    }
#pragma unroll
    for (int hc = 0; hc < NS / 16; ++hc) {
        const float wmax = warp_reduce16<true>(x + hc * 16, lane);
        if (lane < 16) red[wq * NP + hc * 16 + lane] = wmax;
    }
    ptx::named_bar(1, 128);
    if (tid < NS) {
        const float M = fmaxf(fmaxf(red[tid], red[NP + tid]), fmaxf(red[2 * NP + tid], red[3 * NP + tid]));
        const float mo = m_ref_s[tid];
        float a = 1.f;
        if (M > mo) {
            a = (mo == -INFINITY) ? 0.f : exp2f(mo - M);
            m_ref_s[tid] = M;
        }
        alpha_s[tid] = a;
    }
    ptx::named_bar(1, 128);
    if (nMB > 0) {
        ptx::mbar_wait(&vfree[(j - 1) % kR], ph_of(j - 1), abort);
        ptx::tc_fence_after();
#pragma unroll 1
        for (int cc = 0; cc < nMB; ++cc) {
#pragma unroll 1
            for (int hc = 0; hc < NS / 16; ++hc) {
                float v[16];
                const uint32_t ta = t_acc_lane + cc * aw + hc * 16;
                ptx::tmem_ld16(ta, v);
#pragma unroll
                for (int i = 0; i < 16; ++i) v[i] *= alpha_s[hc * 16 + i];
                ptx::tmem_st16(ta, v);
            }
        }
    }
}

// Softmax of tile j of the current piece: RB row blocks of 128 rows, NS heads wide;
// row0 is this thread's row index (segment-wide) in block 0. Reads S^T from TMEM
// (block rb at +rb*NS, or hi at +rb*2NS and lo at +rb*2NS+NS for raw tiles), writes P
// as the MN-major B operand of the value MMA (16-head column blocks of 128*RB rows x
// 32 bytes, 32-byte swizzle), then signals vready[j]. Every head column is processed
// alike: the query rows of absent heads are zero, so their scores are finite and
// their columns, which are never written out, cost no branches.
template <int NS, int NP, int RB, bool LO, bool AL>
__device__ __forceinline__ void softmax_tile(const SoftCtx& c, int j, int row0, int rows, bool has_prev,
                                             float (&l_part)[NP], float (&mref)[NP], const RowBias& rbias) {
    constexpr int SW = SBuf<NP>::W;
    const int jr = j % kR;
    ptx::mbar_wait(&c.bar.kfree[jr], ph_of(j), c.abort);   // S(j) complete
    ptx::tc_fence_after();
    const uint32_t tS0 = c.t_S + c.lane_off + (j & 1) * SW;

    // pass 1: does a score of this thread's rows exceed its head's reference by more
    // than kLazy? (The first tile of a piece has no reference yet: it always takes
    // the rare path, without the vote.)
    bool slow = !has_prev;
    if (has_prev) {
        float dmax = -INFINITY;
#pragma unroll
        for (int rb = 0; rb < RB; ++rb) {
            const uint32_t tS = tS0 + rb * (LO ? 2 : 1) * NS;
            float dm = -INFINITY;
#pragma unroll
            for (int hc = 0; hc < NS / 16; ++hc) {
                float sc[16];
                load_scores<LO, NS>(tS + hc * 16, sc);
                if (AL) add_bias(sc, c.slope_s + hc * 16, rbias.d[rb]);
#pragma unroll
                for (int i = 0; i < 16; ++i) dm = fmaxf(dm, sc[i] - mref[hc * 16 + i]);
            }
            dmax = (row0 + rb * 128 < rows) ? fmaxf(dmax, dm) : dmax;
        }
        const bool any = __any_sync(0xffffffffu, dmax > kLazy);
        volatile int* fl = c.flags + (j & 1) * 4;
        if (c.lane == 0) fl[c.wq] = any ? 1 : 0;
        ptx::named_bar(1, 128);
        slow = (fl[0] | fl[1] | fl[2] | fl[3]) != 0;
    }
    if (slow) {
        softmax_new_ref<NS, NP, RB, LO, AL>(c.red, c.m_ref_s, c.alpha_s, c.bar.vfree, c.abort, tS0,
                                            c.t_accp + c.lane_off, row0, rows, j, has_prev ? c.nMB : 0, c.aw, c.tid,
                                            c.lane, c.wq, c.slope_s, rbias.d[0], rbias.d[RB - 1]);
#pragma unroll
        for (int h = 0; h < NS; ++h) {
            mref[h] = c.m_ref_s[h];
            l_part[h] *= c.alpha_s[h];
        }
    }

    // pass 2: probabilities against the reference, rounded to bf16; the P buffer
    // (j mod npbuf) is free once the value MMAs of tile j - npbuf are done
    if (j >= c.npbuf) ptx::mbar_wait(&c.bar.vfree[(j - c.npbuf) % kR], ph_of(j - c.npbuf), c.abort);
    uint8_t* phi = c.pbuf + (j & (c.npbuf - 1)) * SBuf<NP>::PB;
#pragma unroll
    for (int rb = 0; rb < RB; ++rb) {
        const uint32_t tS = tS0 + rb * (LO ? 2 : 1) * NS;
        const bool valid = row0 + rb * 128 < rows;
        const int row = rb * 128 + c.myrow;
        const uint32_t row_off = row * 32;
        const uint32_t sw = ((row >> 2) & 1) << 4;
#pragma unroll
        for (int hc = 0; hc < NS / 16; ++hc) {
            float sc[16];
            load_scores<LO, NS>(tS + hc * 16, sc);
            if (AL) add_bias(sc, c.slope_s + hc * 16, rbias.d[rb]);
            uint32_t pk[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int h = hc * 16 + 2 * i;
                const float p0 = valid ? exp2f(sc[2 * i] - mref[h]) : 0.f;
                const float p1 = valid ? exp2f(sc[2 * i + 1] - mref[h + 1]) : 0.f;
                l_part[h] += p0;
                l_part[h + 1] += p1;
                const __nv_bfloat162 h2 = __floats2bfloat162_rn(p0, p1);
                pk[i] = *reinterpret_cast<const uint32_t*>(&h2);
            }
            const uint32_t o0 = hc * (kPAtom * RB) + row_off + (0u ^ sw);
            const uint32_t o1 = hc * (kPAtom * RB) + row_off + (16u ^ sw);
            *reinterpret_cast<uint4*>(phi + o0) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
            *reinterpret_cast<uint4*>(phi + o1) = make_uint4(pk[4], pk[5], pk[6], pk[7]);
        }
    }
    ptx::tc_fence_before();          // TMEM reads / writes of this tile before the signal
    ptx::fence_proxy_async_smem();   // P stores visible to the tensor core
    ptx::mbar_arrive(&c.bar.vready[jr]);
}

// Partial write-out of a piece, out of line (once per piece): (m, l) of the piece's
// real heads from the per-warp row sums in `red` (reduce_row_sums), and the
// accumulator columns read from TMEM, up to 32 columns per load and its wait.
template <int NS, int NP>
__device__ __noinline__ void write_partial_acc(float* ml, float* acc, int* kindp, const float* red,
                                               const float* m_ref_s, int Hq, int Dmax, int slot, int kind, int h0,
                                               int nvalid, int dv, int nMB, int aw, uint32_t t_acc_lane,
                                               int tid, int myrow) {
    if (tid < nvalid) {
        const float L = red[tid] + red[NP + tid] + red[2 * NP + tid] + red[3 * NP + tid];
        ml[((size_t)slot * 2) * Hq + h0 + tid] = m_ref_s[tid];
        ml[((size_t)slot * 2 + 1) * Hq + h0 + tid] = L;
    }
    if (tid == 0) kindp[slot] = kind;
#pragma unroll 1
    for (int cc = 0; cc < nMB; ++cc) {
        const int r = cc * 128 + myrow;
        const uint32_t ta = t_acc_lane + cc * aw;
        float v[NS];
        if constexpr (NS % 32 == 0) {
#pragma unroll
            for (int hc = 0; hc < NS / 32; ++hc) {
                float w[32];
                ptx::tmem_ld32(ta + hc * 32, w);
#pragma unroll
                for (int i = 0; i < 32; ++i) v[hc * 32 + i] = w[i];
            }
        } else {
#pragma unroll
            for (int hc = 0; hc < NS / 16; ++hc) {
                float w[16];
                ptx::tmem_ld16(ta + hc * 16, w);
#pragma unroll
                for (int i = 0; i < 16; ++i) v[hc * 16 + i] = w[i];
            }
        }
        if (r < dv) {
#pragma unroll
            for (int h = 0; h < NS; ++h)
                if (h < nvalid) acc[((size_t)slot * Hq + h0 + h) * Dmax + r] = v[h];
        }
    }
}

// End of a piece, first part: the per-warp row sums of every head into `red`. The
// sums are final once the piece's last softmax tile is done, so this runs while its
// last value MMAs are still in flight.
template <int NS, int NP>
__device__ __forceinline__ void reduce_row_sums(const SoftCtx& c, float (&l_part)[NP]) {
    float v[NS];
#pragma unroll
    for (int h = 0; h < NS; ++h) v[h] = l_part[h];
#pragma unroll
    for (int hc = 0; hc < NS / 16; ++hc) {
        const float wsum = warp_reduce16<false>(v + hc * 16, c.lane);
        if (c.lane < 16) c.red[c.wq * NP + hc * 16 + c.lane] = wsum;
    }
    ptx::named_bar(1, 128);
}

// End of a piece, second part (after its last value MMAs): write (m, l) and the
// accumulator columns of the piece's real heads to partial slot `slot`.
template <int NS, int NP>
__device__ __forceinline__ void write_partial(const TcParams& p, const SoftCtx& c, int slot, int kind,
                                              int h0, int nvalid, int dv) {
    write_partial_acc<NS, NP>(p.ml, p.acc, p.kind, c.red, c.m_ref_s, p.Hq, p.Dmax, slot, kind, h0, nvalid, dv, c.nMB,
                              c.aw, c.t_accp + c.lane_off, c.tid, c.myrow);
}

// NP: query heads rounded up to 16 (a template parameter, so the MMA issue sequences
// are straight-line code: a conditional branch between two tcgen05.mma instructions
// costs the issuing thread tens of cycles per MMA).
template <int NP, bool AL>
__global__ void __launch_bounds__(kThreads, 1) tc_decode_kernel(const __grid_constant__ TcParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* ring = smem;
    uint8_t* qbuf = smem + p.off_q;          // query operand of the current piece (image copy)
    uint8_t* pbuf = smem + p.off_p;          // [npbuf][NP/16 blocks][128 * RB rows x 32 B] bf16
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + p.off_bar);
    float* red = reinterpret_cast<float*>(smem + p.off_red);   // [4][NP]
    float* m_ref_s = red + 4 * NP;                             // [NP]
    float* alpha_s = m_ref_s + NP;                             // [NP]
    // [0] abort; [1..8] per-tile votes, two tiles deep (a slow warp still reading
    // one tile's votes never sees the next tile's)
    volatile int* flag = reinterpret_cast<volatile int*>(alpha_s + NP);
    uint32_t* tmem_base_s = reinterpret_cast<uint32_t*>(alpha_s + NP) + 12;
    int* owner = reinterpret_cast<int*>(alpha_s + NP) + 16;    // [kMaxSlots] producer's slot owners
    float* slope_s = reinterpret_cast<float*>(alpha_s + NP) + 32;   // [NP] ALiBi slopes of the piece's columns

    Bars bar;
    bar.kready = bars;
    bar.vready = bars + kR;
    bar.kfree = bars + 2 * kR;
    bar.vfree = bars + 3 * kR;
    bar.accfree = bars + 4 * kR;
    bar.drain = bars + 4 * kR + 2;      // [0] score issuer, [1] value issuer
    bar.qready = bars + 4 * kR + 4;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int cta = blockIdx.x;
    const int u0 = p.u_begin[cta], u1 = p.u_begin[cta + 1];

    if (threadIdx.x == 0) {
        #pragma unroll 1
        for (int i = 0; i < kR; ++i) {
            ptx::mbar_init(&bar.kready[i], 1);
            ptx::mbar_init(&bar.vready[i], 1 + 128);
            ptx::mbar_init(&bar.kfree[i], 1);
            ptx::mbar_init(&bar.vfree[i], 1);
        }
        ptx::mbar_init(&bar.accfree[0], 128);
        ptx::mbar_init(&bar.accfree[1], 128);
        ptx::mbar_init(&bar.drain[0], 1);
        ptx::mbar_init(&bar.drain[1], 1);
        ptx::mbar_init(bar.qready, 1);
        #pragma unroll 1
        for (int i = 0; i < 9; ++i) flag[i] = 0;
        #pragma unroll 1
        for (int i = 0; i < kMaxSlots; ++i) owner[i] = -1;
        ptx::fence_mbar_init();
    }
    if (warp == 1) ptx::tmem_alloc(tmem_base_s, p.tmem_cols);
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_base_s;
    constexpr int SW = SBuf<NP>::W;
    const uint32_t t_S = tmem;             // 2 score buffers of SW columns
    const uint32_t t_acc = tmem + 2 * SW;  // accumulator buffers
    const int aw = NP;   // TMEM columns per 128 value rows of the accumulator
    volatile int* abort_flag = &flag[0];
    pdl_trigger();

    if (warp == 0) {
        // ---------------------------------------------------------------- producer
        // Ring loads in the order the MMAs consume them: K(0), K(1), V(0), K(2), V(1),
        // ..., V(n-1) (keys run at most two tiles ahead of values). A piece's query
        // image is copied into the single query buffer once the score MMAs of the
        // previous piece are done (the CTA's first image is copied by the score
        // issuer, so that the key and value loads need not wait for the preceding
        // kernel); its bytes are part of the kready phase of the piece's first tile.
        if (lane == 0) {
#pragma unroll 1
            for (int i = 0; i < 2 * kNumKinds; ++i)
                if (p.rows[i >> 1] > 0) ptx::tma_prefetch_desc(&p.tm[i]);
            int pos = 0;                     // ring position of the next slot
            const uint64_t pol = ptx::policy_evict_first();   // the cache is streamed once
            bool pdl_done = false;
            // pending query-image copy (pieces after the first)
            bool q_pend = false;
            int q_tile = 0, q_after = 0;     // kready tile; tile whose score MMAs must finish first
            const uint8_t* q_src = nullptr;
            uint32_t q_bytes = 0;
            auto try_q = [&](bool block) {
                if (!q_pend) return;
                if (block) {
                    ptx::mbar_wait(&bar.kfree[q_after % kR], ph_of(q_after), abort_flag);
                } else if (!ptx::mbar_test(&bar.kfree[q_after % kR], ph_of(q_after))) {
                    return;
                }
                if (!pdl_done) {
                    pdl_wait();              // the images come from the preceding kernel
                    pdl_done = true;
                }
                ptx::bulk_load(qbuf, q_src, q_bytes, &bar.kready[q_tile % kR]);
                q_pend = false;
            };
            // wait until ring slot s is free (its previous tile part is consumed)
            auto slot_free = [&](int s) {
                const int o = owner[s];
                if (o < 0) return;
                const int oj = o >> 1;
                uint64_t* fb = (o & 1) ? &bar.vfree[oj % kR] : &bar.kfree[oj % kR];
                const uint32_t par = ph_of(oj);
                if (ptx::mbar_test(fb, par)) return;
                const uint64_t t0 = ptx::globaltimer();
#pragma unroll 1
                for (uint32_t spins = 1; !ptx::mbar_test(fb, par); ++spins) {
                    try_q(false);
                    if ((spins & 63u) == 0) {
                        if (*abort_flag) return;
                        if (ptx::globaltimer() - t0 > ptx::kWaitLimitNs) {
                            *abort_flag = 1;
                            return;
                        }
                    }
                }
            };
            TileIter kit, vit;
            kit.init(p, u0, u1);
            vit.init(p, u0, u1);
            int kiss = 0, viss = 0;   // tiles whose K / V loads were issued
#pragma unroll 1
            while (vit.valid() && !*abort_flag) {
                const bool isK = kit.valid() && kit.j <= vit.j + 1;
                TileIter ti = isK ? kit : vit;
                const int part = isK ? 0 : 1;
                const int k = ti.pc.k;
                const CUtensorMap* tm = &p.tm[2 * k + part];
                const int ncols = ((part ? p.dv[k] : p.dk[k]) + 127) >> 7;
                const int RBk = p.rb[k];
                const int nc = ncols * RBk;   // slots: column chunks x row blocks
#pragma unroll 1
                for (int c = 0; c < nc; ++c) slot_free(ring_wrap(pos + c, p.nslot));
                const int jr = ti.j % kR;
                // test hook: the first key tile of this CTA is never loaded, so the wait
                // for it runs out and the CTA takes the abort path
                const bool withheld = p.withhold_cta == cta && ti.j == 0 && part == 0;
                if (part == 0) {
                    if (ti.first() && ti.j > 0) {
                        if (q_pend) try_q(true);   // the previous piece's image goes first
                        query_image(p, ti.pc, q_src, q_bytes);
                        ptx::mbar_expect_tx_only(&bar.kready[jr], q_bytes);
                        q_pend = true;
                        q_tile = ti.j;
                        q_after = ti.j - 1;
                    }
                    if (!withheld) ptx::mbar_expect_tx(&bar.kready[jr], nc * kSlot);
                } else {
                    ptx::mbar_expect_tx(&bar.vready[jr], nc * kSlot);
                }
                uint64_t* rb = part ? &bar.vready[jr] : &bar.kready[jr];
#pragma unroll 1
                for (int c = 0; c < nc && !withheld; ++c) {
                    const int s = ring_wrap(pos + c, p.nslot);
                    uint8_t* dst = ring + (size_t)s * kSlot;
                    const int col = (c % ncols) * 128;
                    const int row = (ti.t * RBk + c / ncols) * kTile;
                    if (k == 0) {
                        ptx::tma_load_3d_hint(dst, tm, col, row, ti.pc.b, rb, pol);
                        ptx::tma_load_3d_hint(dst + kBox, tm, col + 64, row, ti.pc.b, rb, pol);
                    } else {
                        ptx::tma_load_4d_hint(dst, tm, col, ti.pc.g, row, ti.pc.b, rb, pol);
                        ptx::tma_load_4d_hint(dst + kBox, tm, col + 64, ti.pc.g, row, ti.pc.b, rb, pol);
                    }
                    owner[s] = (ti.j << 1) | part;
                }
                if (withheld)
                    for (int c = 0; c < nc; ++c) owner[ring_wrap(pos + c, p.nslot)] = (ti.j << 1) | part;
                pos = ring_wrap(pos + nc, p.nslot);
                try_q(false);
                if (isK) kiss = ti.j + 1;
                else viss = ti.j + 1;
                ti.next();
                if (isK) kit = ti;
                else vit = ti;
            }
            try_q(true);
            if (*abort_flag) {
                // let copies still in flight land before the CTA winds down (bounded waits;
                // a phase whose other arrivals never come just times out)
                volatile int never = 0;
#pragma unroll 1
                for (int j = max(0, kiss - kR / 2); j < kiss; ++j) ptx::mbar_wait(&bar.kready[j % kR], ph_of(j), &never);
#pragma unroll 1
                for (int j = max(0, viss - kR / 2); j < viss; ++j) ptx::mbar_wait(&bar.vready[j % kR], ph_of(j), &never);
            }
        }
    } else if (warp == 1 || warp == 6) {
        // --------------------------------------------------------------------- MMA
        // Two issuing threads: warp 1 issues the score MMAs, warp 6 the value MMAs, so
        // the two streams do not wait for each other. Per tile each issues after one
        // wait and ends with one commit; waits and commits stall an issuing thread
        // behind the tensor core's in-flight operand reads, so they are kept few. Both
        // walk the producer's sequence of tile parts to track ring positions.
        const bool s_issuer = warp == 1;
        if (lane == 0) {
            const uint32_t idS_lat = ptx::idesc_bf16(128, NP, false, false);
            const uint32_t idS_raw = ptx::idesc_bf16(128, 2 * kNG, false, false);
            const uint32_t idV_lat = ptx::idesc_bf16(128, NP, true, true);
            const uint32_t idV_raw = ptx::idesc_bf16(128, kNG, true, true);
            // base descriptors; a k-step or ring slot only adds (byte offset >> 4) to
            // the start-address field, which stays below 2^14 for shared memory
            const uint64_t dA_S = ptx::sdesc_sw128(ptx::smem_u32(ring), 16, 1024);      // K tile, K-major
            const uint64_t dA_V = ptx::sdesc_sw128(ptx::smem_u32(ring), kBox, 1024);    // V tile, MN-major
            const uint64_t dB_Q = ptx::sdesc_sw128(ptx::smem_u32(qbuf), 16, 1024);      // Q, K-major
            const uint64_t dB_P = ptx::sdesc_sw32(ptx::smem_u32(pbuf), kPAtom, 256);    // P (latent), MN-major
            const uint64_t dB_Pr = ptx::sdesc_sw32(ptx::smem_u32(pbuf), kPAtom * kRBRaw, 256);  // P (raw)
            int pos = 0;   // ring position, same sequence as the producer

            auto issue_S = [&](const TileIter& ti) {
                const int jr = ti.j % kR;
                if (ti.j >= 2) {
                    // score buffer (j & 1) is free once the softmax warps have read S(j - 2)
                    ptx::mbar_wait(&bar.vready[(ti.j - 2) % kR], ph_of(ti.j - 2), abort_flag);
                    ptx::tc_fence_after();
                }
                ptx::mbar_wait(&bar.kready[jr], ph_of(ti.j), abort_flag);
                const uint32_t dS = t_S + (ti.j & 1) * SW;
                if (ti.pc.k == 0) {
                    // latent tile: 128 beacons, key width r_k in 128-column chunks
                    const uint32_t qstride = NP * 128 >> 4;   // 64-column chunk of Q
                    const int ksteps = p.dk[0] >> 4;
                    const int nK = (p.dk[0] + 127) >> 7;
                    const int nfull = ksteps >> 3;   // whole 128-column chunks
#pragma unroll 1
                    for (int c = 0; c < nfull; ++c) {
                        const int s = ring_wrap(pos + c, p.nslot);
                        const uint64_t a0 = dA_S + (uint64_t)((s * kSlot) >> 4);
                        const uint64_t b0 = dB_Q + (uint64_t)(2 * c * qstride);
                        const uint32_t acc0 = c != 0 ? 1u : 0u;
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk)
                            ptx::mma_bf16(dS, a0 + (uint64_t)((kk >> 2) * (kBox >> 4) + (kk & 3) * 2),
                                          b0 + (uint64_t)((kk >> 2) * qstride + (kk & 3) * 2), idS_lat,
                                          kk == 0 ? acc0 : 1u);
                    }
                    if (nfull < nK) {
                        // a last, partial chunk (key width not a multiple of 128)
                        const int c = nfull;
                        const int s = ring_wrap(pos + c, p.nslot);
                        const uint64_t a0 = dA_S + (uint64_t)((s * kSlot) >> 4);
                        const uint64_t b0 = dB_Q + (uint64_t)(2 * c * qstride);
#pragma unroll 1
                        for (int kk = 0; kk < ksteps - 8 * c; ++kk)
                            ptx::mma_bf16(dS, a0 + (uint64_t)((kk >> 2) * (kBox >> 4) + (kk & 3) * 2),
                                          b0 + (uint64_t)((kk >> 2) * qstride + (kk & 3) * 2), idS_lat,
                                          (c | kk) != 0 ? 1u : 0u);
                    }
                    pos = ring_wrap(pos + nK, p.nslot);
                } else {
                    // raw tile: kRBRaw blocks of 128 tokens of one KV head, key width d = 128
                    const uint32_t qstride = 2 * kNG * 128 >> 4;
#pragma unroll
                    for (int rb = 0; rb < kRBRaw; ++rb) {
                        const int s = ring_wrap(pos + rb, p.nslot);
                        const uint64_t a0 = dA_S + (uint64_t)((s * kSlot) >> 4);
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk)
                            ptx::mma_bf16(dS + rb * 2 * kNG, a0 + (uint64_t)((kk >> 2) * (kBox >> 4) + (kk & 3) * 2),
                                          dB_Q + (uint64_t)((kk >> 2) * qstride + (kk & 3) * 2), idS_raw,
                                          kk == 0 ? 0u : 1u);
                    }
                    pos = ring_wrap(pos + kRBRaw, p.nslot);
                }
                ptx::mma_commit(&bar.kfree[jr]);
            };
            auto issue_V = [&](const TileIter& ti) {
                const int jr = ti.j % kR;
                ptx::mbar_wait(&bar.vready[jr], ph_of(ti.j), abort_flag);
                const int pc = ti.piece;
                if (ti.first()) {
                    // the accumulator buffer of this piece must have been read out
                    if (p.accbuf == 2) {
                        if (pc >= 2) ptx::mbar_wait(&bar.accfree[pc & 1], (uint32_t)((pc >> 1) - 1) & 1u, abort_flag);
                    } else if (pc >= 1) {
                        ptx::mbar_wait(&bar.accfree[0], (uint32_t)(pc - 1) & 1u, abort_flag);
                    }
                }
                ptx::tc_fence_after();
                const uint32_t abase = t_acc + (uint32_t)((p.accbuf == 2 ? (pc & 1) : 0) * p.accstride);
                const uint32_t acc0 = ti.first() ? 0u : 1u;
                const uint32_t pboff = (uint32_t)(((ti.j & (p.npbuf - 1)) * SBuf<NP>::PB) >> 4);
                if (ti.pc.k == 0) {
                    const uint64_t pd = dB_P + (uint64_t)pboff;
                    const int nV = (p.dv[0] + 127) >> 7;
#pragma unroll 1
                    for (int c = 0; c < nV; ++c) {
                        const int s = ring_wrap(pos + c, p.nslot);
                        const uint64_t vd = dA_V + (uint64_t)((s * kSlot) >> 4);
                        const uint32_t d0 = abase + c * aw;
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk) {
                            const uint64_t a = vd + (uint64_t)(kk * (2048 >> 4));
                            const uint64_t b = pd + (uint64_t)(kk * (512 >> 4));
                            ptx::mma_bf16(d0, a, b, idV_lat, kk == 0 ? acc0 : 1u);
                        }
                    }
                    pos = ring_wrap(pos + nV, p.nslot);
                } else {
                    // 256 tokens: k-steps 0-7 from block 0's slot, 8-15 from block 1's
                    const uint64_t pd = dB_Pr + (uint64_t)pboff;
#pragma unroll
                    for (int rb = 0; rb < kRBRaw; ++rb) {
                        const int s = ring_wrap(pos + rb, p.nslot);
                        const uint64_t vd = dA_V + (uint64_t)((s * kSlot) >> 4);
                        const uint32_t accr = rb == 0 ? acc0 : 1u;
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk) {
                            const uint64_t a = vd + (uint64_t)(kk * (2048 >> 4));
                            const uint64_t b = pd + (uint64_t)((rb * 8 + kk) * (512 >> 4));
                            ptx::mma_bf16(abase, a, b, idV_raw, kk == 0 ? accr : 1u);
                        }
                    }
                    pos = ring_wrap(pos + kRBRaw, p.nslot);
                }
                ptx::mma_commit(&bar.vfree[jr]);
            };

            TileIter kit, vit;
            kit.init(p, u0, u1);
            vit.init(p, u0, u1);
            if (s_issuer && kit.valid()) {
                // the CTA's first query image, once the preceding kernel has written it
                // (its own barrier: the key and value loads never wait for it)
                const uint8_t* q_src;
                uint32_t q_bytes;
                query_image(p, kit.pc, q_src, q_bytes);
                pdl_wait();
                ptx::mbar_expect_tx(bar.qready, q_bytes);
                ptx::bulk_load(qbuf, q_src, q_bytes, bar.qready);
                ptx::mbar_wait(bar.qready, 0, abort_flag);
            }
#pragma unroll 1
            while (vit.valid()) {
                const bool isK = kit.valid() && kit.j <= vit.j + 1;
                TileIter ti = isK ? kit : vit;
                if (isK == s_issuer) {
                    if (isK) issue_S(ti);
                    else issue_V(ti);
                } else {
                    const int k = ti.pc.k;
                    pos = ring_wrap(pos + (((isK ? p.dk[k] : p.dv[k]) + 127) >> 7) * p.rb[k], p.nslot);
                }
                ti.next();
                if (isK) kit = ti;
                else vit = ti;
            }
            ptx::mma_commit(&bar.drain[s_issuer ? 0 : 1]);   // arrives once this thread's MMAs completed
        }
    } else {
        // ----------------------------------------------------------------- softmax
        SoftCtx c;
        c.bar = bar;
        c.pbuf = pbuf;
        c.npbuf = p.npbuf;
        c.red = red;
        c.m_ref_s = m_ref_s;
        c.alpha_s = alpha_s;
        c.flags = flag + 1;
        c.slope_s = slope_s;
        c.abort = abort_flag;
        c.tid = threadIdx.x - 64;            // 0..127
        c.wq = c.tid >> 5;                   // softmax warp 0..3
        c.lane = lane;
        const int q4 = warp & 3;             // TMEM lane quadrant this warp may access
        c.myrow = q4 * 32 + lane;            // tile row (S) / value row (acc) of this thread
        c.lane_off = (uint32_t)(q4 * 32) << 16;
        c.t_S = t_S;
        c.aw = aw;
        const int G = p.G;
        float l_part[NP], mref[NP];

        pdl_wait();   // the workspace partials may still be read by the preceding calls' kernels

        TileIter it;
        it.init(p, u0, u1);
        while (it.valid()) {
            const Piece pc = it.pc;
            const int piece = it.piece;
            const int k = pc.k;
            const bool lat = (k == 0);
            const int nvalid = lat ? p.Hq : G;
            c.nMB = (p.dv[k] + 127) >> 7;
            c.t_accp = t_acc + (uint32_t)((p.accbuf == 2 ? (piece & 1) : 0) * p.accstride);
            if (c.tid < NP) {
                m_ref_s[c.tid] = -INFINITY;
                // ALiBi slopes of the piece's score columns: every head (latent), or the
                // heads of the piece's KV group (raw; padded columns get 0)
                if (AL)
                    slope_s[c.tid] = lat ? (c.tid < p.Hq ? p.slope_l2[c.tid] : 0.f)
                                         : (c.tid < G ? p.slope_l2[pc.g * G + c.tid] : 0.f);
            }
#pragma unroll
            for (int h = 0; h < NP; ++h) {
                l_part[h] = 0.f;
                mref[h] = -INFINITY;
            }
            const long long qp = AL ? (long long)p.q_pos[pc.b] : 0;
            ptx::named_bar(1, 128);
            int jl = it.j;
            #pragma unroll 1
            for (int n = 0; n < pc.n; ++n) {
                const int t = it.t;
                const int row0 = t * kTile * p.rb[k] + c.myrow;
                // key position - query position of this thread's rows (beacon j at
                // j * ratio + ratio - 1; window slot s at qp - ((qp - s) mod W))
                RowBias rbias = {{0.f, 0.f}};
                if (AL) {
#pragma unroll
                    for (int rb = 0; rb < 2; ++rb) {
                        const long long row = row0 + rb * 128;
                        const long long W = p.rows[k];
                        rbias.d[rb] = lat ? (float)(row * p.ratio + p.ratio - 1 - qp)
                                          : -(float)((((qp - row) % W) + W) % W);
                    }
                }
                jl = it.j;
                if (lat) softmax_tile<NP, NP, 1, false, AL>(c, it.j, row0, p.rows[k], t > pc.t0, l_part, mref, rbias);
                else softmax_tile<kNG, NP, kRBRaw, true, AL>(c, it.j, row0, p.rows[k], t > pc.t0, l_part, mref, rbias);
                it.next();
            }
            // ---- partial of (CTA, piece): reference max, row sum and accumulator
            if (lat) reduce_row_sums<NP, NP>(c, l_part);
            else reduce_row_sums<kNG, NP>(c, l_part);
            ptx::mbar_wait(&bar.vfree[jl % kR], ph_of(jl), abort_flag);   // V(jl) complete
            ptx::tc_fence_after();
            const int slot = p.slot_base[cta] + piece;
            if (lat) write_partial<NP, NP>(p, c, slot, kSlotLatent, 0, nvalid, p.dv[k]);
            else write_partial<kNG, NP>(p, c, slot, kSlotRawGroup + pc.g, pc.g * G, nvalid, p.d_raw);
            ptx::tc_fence_before();
            ptx::mbar_arrive(&bar.accfree[p.accbuf == 2 ? (piece & 1) : 0]);
            ptx::named_bar(1, 128);
        }
    }

    // ----------------------------------------------------------------- teardown
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        if (lane == 0) {
            volatile int never = 0;
            ptx::mbar_wait(&bar.drain[0], 0, &never);   // every MMA of this CTA has completed
            ptx::mbar_wait(&bar.drain[1], 0, &never);
            if (u0 < u1) ptx::mbar_wait(bar.qready, 0, &never);   // the first query copy has landed
        }
        __syncwarp();
        ptx::tmem_dealloc(tmem, p.tmem_cols);
    }
    if (*abort_flag && warp >= 2 && warp <= 5) {
        // a wait ran out: poison this CTA's partials so the result is NaN, not stale, and
        // count the CTA where the host can read it
        const int tid = threadIdx.x - 64;
        if (tid == 0 && p.aborts != nullptr) atomicAdd(p.aborts, 1ull);
        int npieces = 0;
        #pragma unroll 1
        for (int u = u0; u < u1;) {
            const Piece pc = piece_at(p, u, u1);
            u += pc.n;
            ++npieces;
        }
        #pragma unroll 1
        for (int i = tid; i < npieces * p.Hq; i += 128) {
            const int slot = p.slot_base[cta] + i / p.Hq;
            p.ml[((size_t)slot * 2 + 1) * p.Hq + (i % p.Hq)] = __int_as_float(0x7fc00000);
        }
    }
}

// ------------------------------------------------------------------------ host

// Shared-memory plan of one launch.
struct SmemPlan {
    int NP, nslot, q_cols, accbuf, accstride, npbuf;
    uint32_t off_q, off_p, off_bar, off_red, total, tmem_cols;
    bool ok;
};

int round_up(int x, int m) { return (x + m - 1) / m * m; }

// TMEM columns of one score buffer (host copy of SBuf<NP>::W).
int sbuf_w(int NP) { return std::max(NP, 2 * kNG * kRBRaw); }

SmemPlan plan_smem(int Hq, const int dk[kNumKinds], const int dv[kNumKinds], const int rows[kNumKinds]) {
    const int budget = kSmemMax;
    SmemPlan s{};
    s.NP = round_up(Hq, 16);
    int qc = 0, nmb = 0, maxK = 0, maxV = 0;
    for (int k = 0; k < kNumKinds; ++k) {
        if (rows[k] <= 0) continue;
        const int rbk = k == 0 ? 1 : kRBRaw;
        qc = std::max(qc, dk[k]);
        nmb = std::max(nmb, (dv[k] + 127) / 128);
        maxK = std::max(maxK, (dk[k] + 127) / 128 * rbk);   // ring slots of a tile's keys
        maxV = std::max(maxV, (dv[k] + 127) / 128 * rbk);
    }
    s.q_cols = round_up(qc, 64);
    s.ok = false;
    if (s.NP > 64) return s;
    // TMEM: two score buffers of sbuf_w(NP) columns, then one or two accumulator
    // buffers (two when they fit, so a piece's write-out overlaps the next piece)
    s.accstride = nmb * s.NP;
    int tmem = 0;
    for (s.accbuf = 2; s.accbuf >= 1; --s.accbuf) {
        tmem = 2 * sbuf_w(s.NP) + s.accbuf * s.accstride;
        if (tmem <= 512) break;
    }
    if (tmem > 512) return s;
    s.tmem_cols = 32;
    while ((int)s.tmem_cols < tmem) s.tmem_cols *= 2;
    // query buffer: the latent image (NP rows, bf16) or a raw image (hi and lo parts of kNG heads)
    const int q_bytes = std::max(rows[0] > 0 ? s.NP * round_up(dk[0], 64) * 2 : 0, 2 * kNG * 128 * 2);
    const int nbars = 4 * kR + 5;
    const int misc_bytes = (7 * s.NP + 32) * 4;
    // One tile part (keys or values) must fit the ring. The loads run in consumption
    // order and each waits only for earlier parts to be consumed, so a ring smaller
    // than a key plus a value tile (latent ranks above 256) still drains: it only
    // serialises those tiles' loads behind their consumers. Two P buffers let the
    // softmax of a tile run while the value MMAs of the previous one read theirs; when
    // the ring would not hold a tile part otherwise (64 heads at rank 512), one buffer
    // serialises the two instead.
    int p_bytes = 0;
    for (s.npbuf = 2; s.npbuf >= 1; --s.npbuf) {
        p_bytes = s.npbuf * std::max(s.NP, kNG * kRBRaw) * 256;   // bf16
        const int avail = budget - q_bytes - p_bytes - round_up(nbars * 8, 16) - misc_bytes - 1024;
        s.nslot = std::min(kMaxSlots, avail / kSlot);
        if (s.nslot >= std::max(maxK, maxV)) break;
    }
    if (s.npbuf < 1) return s;
    s.off_q = s.nslot * kSlot;
    s.off_p = s.off_q + q_bytes;
    s.off_bar = s.off_p + p_bytes;
    s.off_red = s.off_bar + round_up(nbars * 8, 16);
    s.total = s.off_red + misc_bytes + 1024;
    s.ok = s.total <= (uint32_t)budget;
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

// Latent operand: 3-D bf16 tensor [B][rows][cols] (cols contiguous) read in boxes of
// 128 rows x 64 columns with the 128-byte swizzle; rows/columns past the end read as zero.
bool make_map_latent(CUtensorMap* tm, const void* base, int cols, int rows, int B) {
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

// Raw operand: 4-D bf16 tensor [B][T][Hkv][d] read per KV head in boxes of 128
// tokens x 64 columns (one head), 128-byte swizzle; tokens past the end read as zero.
bool make_map_raw(CUtensorMap* tm, const void* base, int d, int Hkv, int T, int B) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[4] = {(cuuint64_t)d, (cuuint64_t)Hkv, (cuuint64_t)T, (cuuint64_t)B};
    cuuint64_t strides[3] = {(cuuint64_t)d * 2, (cuuint64_t)Hkv * d * 2, (cuuint64_t)T * Hkv * d * 2};
    cuuint32_t box[4] = {64, 1, (cuuint32_t)kTile, 1};
    cuuint32_t es[4] = {1, 1, 1, 1};
    return fn(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Encoded tensor maps are reused by later calls on the same buffers and sizes
// (encoding is a driver call; a decode step makes four per layer). Direct-mapped.
bool cached_map(CUtensorMap* tm, bool latent, const void* base, int a, int b, int c, int d) {
    struct Entry {
        bool valid = false;
        bool latent = false;
        const void* base = nullptr;
        int dims[4] = {0, 0, 0, 0};
        CUtensorMap tm;
    };
    static std::mutex mu;
    static Entry cache[512];
    const uint64_t h = ((uint64_t)(uintptr_t)base >> 8) * 0x9E3779B97F4A7C15ull ^
                       ((uint64_t)a * 31 + b) * 0xBF58476D1CE4E5B9ull ^ ((uint64_t)c * 131 + d + latent);
    Entry& e = cache[(h >> 40) % 512];
    {
        std::lock_guard<std::mutex> g(mu);
        if (e.valid && e.latent == latent && e.base == base && e.dims[0] == a && e.dims[1] == b &&
            e.dims[2] == c && e.dims[3] == d) {
            *tm = e.tm;
            return true;
        }
    }
    const bool ok = latent ? make_map_latent(tm, base, a, b, c) : make_map_raw(tm, base, a, b, c, d);
    if (ok) {
        std::lock_guard<std::mutex> g(mu);
        e.valid = true;
        e.latent = latent;
        e.base = base;
        e.dims[0] = a;
        e.dims[1] = b;
        e.dims[2] = c;
        e.dims[3] = d;
        e.tm = *tm;
    }
    return ok;
}

int sm_count() {
    static std::atomic<int> cached[64];
    int dev = 0, n = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && (n = cached[dev].load()) > 0) return n;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 148;
    if (dev >= 0 && dev < 64) cached[dev].store(n);
    return n;
}

using plan::WorkPlan;
using plan::SegList;
using plan::make_plan;

struct PlanKey {
    int B, max_ctas, lat_segs;
    std::vector<std::pair<int, int>> segs;
    bool operator<(const PlanKey& o) const {
        return std::tie(B, max_ctas, lat_segs, segs) < std::tie(o.B, o.max_ctas, o.lat_segs, o.segs);
    }
};

// A work plan and, per batch element, its first raw partial slot (the latent slots of b
// come first: units are ordered by segment, latent before raw).
struct CtaPlan {
    WorkPlan w;
    std::vector<int> batch_mid;
};

// Plans are built once per (batch, segment list, grid limit) and shared: the cache hands
// out shared ownership, so a plan stays valid for a caller while another thread clears
// the cache. lat_segs: segments of a batch element before the first raw one.
std::shared_ptr<const CtaPlan> cached_plan(int B, const SegList& sl, int lat_segs, int max_ctas) {
    static std::mutex mu;
    static std::map<PlanKey, std::shared_ptr<const CtaPlan>> cache;
    PlanKey key{B, max_ctas, lat_segs, sl.segs};
    std::lock_guard<std::mutex> g(mu);
    auto it = cache.find(key);
    if (it != cache.end()) return it->second;
    if (cache.size() > 256) cache.clear();
    auto cp = std::make_shared<CtaPlan>();
    cp->w = make_plan(B, sl, max_ctas);
    cp->batch_mid.resize(B);
    for (int b = 0; b < B; ++b) cp->batch_mid[b] = plan::first_slot_from_seg(cp->w, b, lat_segs);
    std::shared_ptr<const CtaPlan> r = cp;
    cache.emplace(std::move(key), r);
    return r;
}

template <int NP, bool AL>
cudaError_t launch_decode_t(const TcParams& prm, int grid, uint32_t smem, cudaStream_t st) {
    static std::atomic<unsigned long long> attr_done{0};
    const cudaError_t ea = set_max_smem_once((const void*)tc_decode_kernel<NP, AL>, kSmemMax, attr_done);
    if (ea != cudaSuccess) return ea;
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
    return cudaLaunchKernelEx(&cfg, tc_decode_kernel<NP, AL>, prm);
}
// The ALiBi bias is a separate instantiation: the plain decode keeps none of its code
// (the kernel's speed depends on its instruction-cache footprint).
template <int NP>
cudaError_t launch_decode(const TcParams& prm, int grid, uint32_t smem, cudaStream_t st) {
    return prm.alibi ? launch_decode_t<NP, true>(prm, grid, smem, st) : launch_decode_t<NP, false>(prm, grid, smem, st);
}

// Kinds of key rows of one call: rows / widths per segment and operands.
struct Kinds {
    int rows[kNumKinds] = {0, 0, 0};
    int ngroups[kNumKinds] = {0, 0, 0};
    int dk[kNumKinds] = {0, 0, 0};
    int dv[kNumKinds] = {0, 0, 0};
    const void* K[kNumKinds] = {nullptr, nullptr, nullptr};
    const void* V[kNumKinds] = {nullptr, nullptr, nullptr};
};

Kinds kinds_of(const TcCall& c) {
    Kinds s;
    auto raw = [&](int k, int T, const void* K, const void* V) {
        if (T <= 0) return;
        s.rows[k] = T;
        s.ngroups[k] = c.Hkv;
        // raw tiles are 128 columns wide; with d = 64 the second 64-column box of every
        // row lies past the tensor and is filled with zeros by the copy (no memory
        // traffic), so scores and value rows are those of d = 64
        s.dk[k] = s.dv[k] = kRawCols;
        s.K[k] = K;
        s.V[k] = V;
    };
    if (c.which == SLIMKV_LATENT) {
        if (c.N_b > 0) {
            s.rows[0] = c.N_b;
            s.ngroups[0] = 1;
            s.dk[0] = c.r_k;
            s.dv[0] = c.r_v;
            s.K[0] = c.C_K;
            s.V[0] = c.C_V;
        }
        raw(1, c.W, c.K_raw, c.V_raw);
    } else if (c.which == SLIMKV_RECONSTRUCT) {
        raw(1, c.N_b, c.kb, c.vb);
        raw(2, c.W, c.K_raw, c.V_raw);
    } else {
        raw(1, c.W, c.K_raw, c.V_raw);
    }
    return s;
}

}  // namespace

bool tc_supported(int Hq, int Hkv, int d, int N_b, int r_k, int r_v) {
    if ((d != 128 && d != 64) || Hq > 64 || Hkv > 128 || Hq / Hkv > kNG) return false;
    int rows[kNumKinds] = {N_b, 1, 1}, dk[kNumKinds] = {r_k, kRawCols, kRawCols},
        dv[kNumKinds] = {r_v, kRawCols, kRawCols};
    if (N_b <= 0) rows[0] = 0;
    return plan_smem(Hq, dk, dv, rows).ok;
}

cudaError_t tc_run(const TcCall& c, cudaStream_t st) {
    typedef __nv_bfloat16 bf16;
    const bool lat = c.which == SLIMKV_LATENT && c.N_b > 0;
    const int NPq = (c.Hq + 15) / 16 * 16;
    cudaError_t e = launch_qproj<bf16>((const bf16*)c.q, lat ? (const bf16*)c.U_K : nullptr, c.q_pos, nullptr,
                                       nullptr, c.B, c.Hq, c.Hkv, c.d, c.r_k, c.rope_base, c.scale_log2, st, true,
                                       lat ? c.lat_img : nullptr, c.raw_img, NPq);
    if (e != cudaSuccess) return e;
    if (c.which == SLIMKV_RECONSTRUCT) {
        // the reconstruction GEMMs (tc_gemm.cu) never release their dependents early: the
        // decode below reads K_b / V_b before its own dependency wait, so they must be
        // complete when it starts
        const int rows = c.B * c.N_b, n = c.Hkv * c.d;
        e = launch_reconstruct_gemm((const bf16*)c.C_K, (const bf16*)c.U_K, (bf16*)c.kb, rows, n, c.r_k, st,
                                    c.beacon_ratio, c.N_b, c.rope_base);
        if (e != cudaSuccess) return e;
        e = launch_reconstruct_gemm((const bf16*)c.C_V, (const bf16*)c.U_V, (bf16*)c.vb, rows, n, c.r_v, st);
        if (e != cudaSuccess) return e;
    }
    const Kinds s = kinds_of(c);
    const SmemPlan sp = plan_smem(c.Hq, s.dk, s.dv, s.rows);
    if (!sp.ok) return cudaErrorInvalidValue;

    TcParams prm;   // copied into the launch's parameter space
    memset(&prm, 0, sizeof(prm));
    SegList sl;
    prm.tiles_per_b = 0;
    for (int k = 0; k < kNumKinds; ++k) {
        prm.rows[k] = s.rows[k];
        prm.ngroups[k] = s.ngroups[k];
        prm.dk[k] = s.dk[k];
        prm.dv[k] = s.dv[k];
        prm.rb[k] = k == 0 ? 1 : kRBRaw;
        const int tile_rows = kTile * prm.rb[k];
        const int tiles = s.rows[k] > 0 ? (s.rows[k] + tile_rows - 1) / tile_rows : 0;
        prm.tiles[k] = tiles;
        prm.tiles_per_b += tiles * s.ngroups[k];
        // cost of a tile: the 32 KB slots it streams (+1 for its fixed per-tile work)
        const int cost = ((s.dk[k] + 127) / 128 + (s.dv[k] + 127) / 128) * prm.rb[k] + 1;
        for (int g = 0; g < s.ngroups[k]; ++g) sl.segs.push_back({tiles, cost});
        if (s.rows[k] > 0) {
            const bool ok = k == 0
                                ? cached_map(&prm.tm[0], true, s.K[0], s.dk[0], s.rows[0], c.B, 0) &&
                                      cached_map(&prm.tm[1], true, s.V[0], s.dv[0], s.rows[0], c.B, 0)
                                : cached_map(&prm.tm[2 * k], false, s.K[k], c.d, c.Hkv, s.rows[k], c.B) &&
                                      cached_map(&prm.tm[2 * k + 1], false, s.V[k], c.d, c.Hkv, s.rows[k], c.B);
            if (!ok) return cudaErrorInvalidValue;
        }
    }
    const int lat_segs = s.rows[0] > 0 ? s.ngroups[0] : 0;   // latent segments come first
    const std::shared_ptr<const CtaPlan> plan = cached_plan(c.B, sl, lat_segs, std::min(kMaxCtas, sm_count()));
    const WorkPlan& w = plan->w;
    if (w.slots > c.slots) return cudaErrorInvalidValue;
    prm.B = c.B;
    prm.Hq = c.Hq;
    prm.Hkv = c.Hkv;
    prm.G = c.Hq / c.Hkv;
    prm.lat_img = c.lat_img;
    prm.raw_img = c.raw_img;
    prm.lat_img_bytes = (uint32_t)lat_img_bytes(sp.NP, c.r_k);
    prm.raw_img_bytes = (uint32_t)raw_img_bytes(kRawCols);
    prm.d_raw = c.d;
    prm.acc = c.acc;
    prm.ml = c.ml;
    prm.kind = c.kind;
    prm.Dmax = c.Dmax;
    prm.nslot = sp.nslot;
    prm.npbuf = sp.npbuf;
    prm.accbuf = sp.accbuf;
    prm.accstride = sp.accstride;
    prm.off_q = sp.off_q;
    prm.off_p = sp.off_p;
    prm.off_bar = sp.off_bar;
    prm.off_red = sp.off_red;
    prm.tmem_cols = sp.tmem_cols;
    if (c.alibi_slopes != nullptr) {
        // ALiBi biases enter in the kernel's log2 units
        prm.alibi = 1;
        prm.ratio = c.beacon_ratio;
        prm.q_pos = c.q_pos;
        for (int h = 0; h < c.Hq; ++h) prm.slope_l2[h] = c.alibi_slopes[h] * kLog2e;
    }
    prm.aborts = abort_counter();
    prm.withhold_cta = take_withheld_cta();
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
    for (int b = 0; b < c.B; ++b) cb.slot_mid[b] = plan->batch_mid[b];
    return launch_tc_combine(cb, st);
}

}  // namespace slimkv

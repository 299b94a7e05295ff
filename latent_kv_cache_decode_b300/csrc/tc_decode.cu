// Tensor-core split-context decode for SlimKV on sm_103a (tcgen05 + TMA).
//
// "Can SlimKV compress KV cache jointly across tokens and features", section
// "Latent-space attention removes the rebuild step": per query head the scores
// are (RoPE(q) U_K^(g)) C_K^T against the RoPE-free latent beacon keys and
// RoPE(q) K_raw^T against the raw window, in one softmax; values aggregate as
// (A C_V) U_V^(g)T + A V_raw, the latent aggregate taken before the up-projection.
//
// Work layout. A "segment" is all key rows of one kind for one batch element,
// read as a 2-D [rows, width] bf16 matrix:
//   latent: the N_b beacons of C_K[b] / C_V[b] (widths r_k / r_v), shared by
//           every query head (one latent cache per layer for all KV heads);
//   raw:    the W x Hkv rows of K[b] / V[b] (row = token * Hkv + KV head, width d).
//           A raw row is scored by every head, and the softmax keeps only the
//           heads of the row's own KV group, so one query image serves the whole
//           window and raw tiles need no per-group split.
// A "tile" (unit of work) is 128 rows of a segment. A host planner gives every
// CTA a contiguous, byte-balanced run of tiles (flash-decoding split of the
// context); a run's part inside one segment is a "piece", which produces one
// partial (m, l, acc) in the workspace, merged later by the combine kernel.
//
// Per tile, with the query operand Q (float32 query carrying scale * log2(e)):
//   scores  S^T[row, col] = tile[row, :] . Q[col, :]   (M = 128 rows; one
//           tcgen05.mma per 16-wide k-step). Latent tiles: Q = bf16 of the latent
//           query, N = heads (latent scores are not peaked, so one bf16 part stays
//           far inside the error bar). Raw tiles: Q = [q_hi ; q_lo], the bf16 high
//           and low parts of the rotated query (raw keys can be large), N = 2 x
//           heads, and the softmax adds the two parts;
//   softmax P[row, head] = exp2(S^T - m_ref[head]) for the heads the row belongs
//           to (all heads for a latent row, the row's KV group for a raw row),
//           else 0; rounded to bf16 (relative error at most 2^-9 per weight,
//           averaging out in the sums);
//   values  acc^T[value dim, head] += tile_V[:, value dim]^T . P (M = 128 value dims).
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
//
// Query images. The kernel makes its own query operands ("RoPE ... on all queries";
// the projection is taken after GQA grouping): the rotated query of every head as bf16
// high and low parts (raw image) and its projection q . U_K^(g) (latent image), one
// pair of images per batch element in the workspace. The CTAs that work on a batch
// element share the work: units of (KV group, 64 latent columns) and (KV group, raw
// rows) are dealt out round-robin; each CTA publishes its units with a release flag,
// and a CTA copies an image into shared memory once every CTA of that batch element
// has flagged. The flags carry a token unique to the launch: a per-channel epoch in
// library-owned device memory (zero when the library loads) that the launch's CTAs
// read after the grid-dependency wait, the last of them advancing it; the host gives
// every workspace its own channel. So no workspace word needs a known initial value.
// While the first images are made, the producer already streams key and value tiles.
//
// Shared memory is kept below what one SM holds by about 30 KB whenever the shape
// allows, so that a combine CTA can sit on the same SM: with programmatic dependent
// launch, the next layer's decode CTAs take over an SM as soon as this layer's CTA
// leaves it and stream their first tiles while the combine runs.
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
// Preferred budget: leaves room on the SM for one query-projection and one combine CTA.
constexpr int kSmemShared = 196 * 1024;
constexpr int kNumKinds = 3;          // latent, raw source 0, raw source 1
// m_ref moves only when a score exceeds it by more than this (log2 units). P values up
// to 2^20 keep bf16's relative precision and stay far from fp32 overflow in the
// accumulator and row sums, so a generous margin keeps the rescale path (which waits
// for the previous value MMAs) off the common path even for peaked score distributions.
constexpr float kLazy = 20.f;
constexpr int kPAtom = 128 * 32;      // bytes of one 16-head column block of P per 128 rows (x 32 B)
constexpr int kR = 16;                // depth of the per-tile barrier rings
constexpr int kMaxSlots = 16;
constexpr int kChannels = 1024;       // launch-token channels (one per workspace in use)
// Bytes each CTA pulls into L2 beyond its first two tiles when it starts (see the producer).
constexpr int kPrefetchBytes = 384 * 1024;

// Per-channel launch epochs and check-in counts (zero when the module loads).
__device__ unsigned int g_chan_epoch[kChannels];
__device__ unsigned int g_chan_count[kChannels];

struct TcParams {
    CUtensorMap tm[2 * kNumKinds];    // per kind: keys, values (3-D [B][rows][width])
    int B, Hq, Hkv, G;
    int rows[kNumKinds];              // rows of one segment (0 = kind absent)
    int tiles[kNumKinds];             // tiles of one segment
    int dk[kNumKinds], dv[kNumKinds]; // key / value width
    int tiles_per_b;
    uint8_t* lat_img;                 // query images (operand layout: latent bf16, raw bf16 hi / lo)
    uint8_t* raw_img;
    uint32_t lat_img_bytes, raw_img_bytes;
    float* acc;                       // [slots, Hq, Dmax]
    float* ml;                        // [slots, 2, Hq]
    int Dmax;
    int nslot;                        // ring slots of 32 KB
    int accbuf;                       // TMEM accumulator buffers (1 or 2)
    int accstride;                    // TMEM columns of one accumulator buffer
    uint32_t off_q, off_p, off_bar, off_red;
    uint32_t tmem_cols;
    // query images, made by the kernel
    const __nv_bfloat16* q;           // [B, Hq, d] queries before RoPE
    const __nv_bfloat16* U_K;         // [Hkv * d, r_k] (latent images only)
    const int32_t* q_pos;             // [B]
    unsigned long long* flags;        // [gridDim.x] per-CTA "images published" flags (workspace)
    int ch;                           // launch-token channel
    int r_k;
    int ncb;                          // latent image units per KV group (64 columns each; 0: no latent image)
    int pf_tiles;                     // tiles after the first two whose boxes are pulled into L2 at the start
    int img_raw;                      // 1: raw images are needed
    float scale_log2;                 // score scale * log2(e), folded into both images
    unsigned long long turn[64];      // RoPE angles per pair as 64-bit fractions of a turn
    short cta_first[kMaxB], cta_last[kMaxB];   // CTAs whose runs touch batch element b
    int u_begin[kMaxCtas + 1];        // CTA i owns units (tiles) [u_begin[i], u_begin[i+1])
    int slot_base[kMaxCtas];          // first partial slot of CTA i
};

// The run of a CTA's units that starts at u and stays inside one segment.
struct Piece {
    int b, k, t0, n;
};
__device__ __forceinline__ Piece piece_at(const TcParams& p, int u, int u1) {
    Piece r;
    r.b = u / p.tiles_per_b;
    int t = u - r.b * p.tiles_per_b;
    int k = 0;
    for (; k < kNumKinds - 1; ++k) {
        if (t < p.tiles[k]) break;
        t -= p.tiles[k];
    }
    r.k = k;
    r.t0 = t;
    r.n = min(u1 - u, p.tiles[k] - t);
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

// Query operand image of a piece: the latent or the raw image of its batch element.
__device__ __forceinline__ void query_image(const TcParams& p, const Piece& pc, const uint8_t*& src,
                                            uint32_t& bytes) {
    if (pc.k == 0) {
        src = p.lat_img + (size_t)pc.b * p.lat_img_bytes;
        bytes = p.lat_img_bytes;
    } else {
        src = p.raw_img + (size_t)pc.b * p.raw_img_bytes;
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
    uint64_t* tok;      // the launch token is in shared memory                     [1 arrival]
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
};

// TMEM columns of one score buffer (hi and lo columns of every head for raw tiles)
// and bytes of one P buffer (NP heads x 128 rows, bf16).
template <int NP> struct SBuf {
    static constexpr int W = 2 * NP;
    static constexpr int PB = NP * 256;
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

// Whether head h is scored by this thread's row: every head for a latent row, the
// heads [hlo, hlo + hn) of the row's KV group for a raw row (LO).
template <bool LO>
__device__ __forceinline__ bool head_on(int h, int hlo, int hn) {
    return !LO || (unsigned)(h - hlo) < (unsigned)hn;
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
template <int NP, bool LO>
__device__ __noinline__ void softmax_new_ref(float* red, float* m_ref_s, float* alpha_s, uint64_t* vfree,
                                             volatile int* abort, uint32_t tS, uint32_t t_acc_lane, bool row_ok,
                                             int hlo, int hn, int j, int nMB, int aw, int tid, int lane, int wq) {
    // per-head maximum over this warp's scored rows, then over the four warps
    // (the TMEM loads are warp-collective: every lane loads, unscored entries are masked after)
    float x[NP];
#pragma unroll
    for (int hc = 0; hc < NP / 16; ++hc) {
        float sc[16];
        load_scores<LO, NP>(tS + hc * 16, sc);
#pragma unroll
        for (int i = 0; i < 16; ++i)
            x[hc * 16 + i] = (row_ok && head_on<LO>(hc * 16 + i, hlo, hn)) ? sc[i] : -INFINITY;
    }
#pragma unroll
    for (int hc = 0; hc < NP / 16; ++hc) {
        const float wmax = warp_reduce16<true>(x + hc * 16, lane);
        if (lane < 16) red[wq * NP + hc * 16 + lane] = wmax;
    }
    ptx::named_bar(1, 128);
    if (tid < NP) {
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
            for (int hc = 0; hc < NP / 16; ++hc) {
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

// Softmax of tile j of the current piece (128 rows, NP heads). row_ok: this thread's
// row lies inside the segment; [hlo, hlo + hn): the heads a raw row belongs to. Reads
// S^T from TMEM (hi at +0 and lo at +NP for raw tiles), writes P as the MN-major B
// operand of the value MMA (16-head column blocks of 128 rows x 32 bytes, 32-byte
// swizzle), then signals vready[j]. Every head column is processed alike, without
// per-head branches: the query rows of absent heads are zero, so their scores are
// finite, and their columns are never written out.
template <int NP, bool LO>
__device__ __forceinline__ void softmax_tile(const SoftCtx& c, int j, bool row_ok, int hlo, int hn, bool has_prev,
                                             float (&l_part)[NP]) {
    const float* mref = c.m_ref_s;   // reference maxima (shared; every thread reads the same words)
    constexpr int SW = SBuf<NP>::W;
    const int jr = j % kR;
    ptx::mbar_wait(&c.bar.kfree[jr], ph_of(j), c.abort);   // S(j) complete
    ptx::tc_fence_after();
    const uint32_t tS = c.t_S + c.lane_off + (j & 1) * SW;

    // pass 1: does a score of this thread's row exceed its head's reference by more
    // than kLazy? (The first tile of a piece has no reference yet: it always takes
    // the rare path, without the vote.)
    bool slow = !has_prev;
    if (has_prev) {
        float dm = -INFINITY;
#pragma unroll
        for (int hc = 0; hc < NP / 16; ++hc) {
            float sc[16];
            load_scores<LO, NP>(tS + hc * 16, sc);
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const float dd = sc[i] - mref[hc * 16 + i];
                dm = head_on<LO>(hc * 16 + i, hlo, hn) ? fmaxf(dm, dd) : dm;
            }
        }
        const bool any = __any_sync(0xffffffffu, row_ok && dm > kLazy);
        volatile int* fl = c.flags + (j & 1) * 4;
        if (c.lane == 0) fl[c.wq] = any ? 1 : 0;
        ptx::named_bar(1, 128);
        slow = (fl[0] | fl[1] | fl[2] | fl[3]) != 0;
    }
    if (slow) {
        softmax_new_ref<NP, LO>(c.red, c.m_ref_s, c.alpha_s, c.bar.vfree, c.abort, tS, c.t_accp + c.lane_off,
                                row_ok, hlo, hn, j, has_prev ? c.nMB : 0, c.aw, c.tid, c.lane, c.wq);
#pragma unroll
        for (int h = 0; h < NP; ++h) l_part[h] *= c.alpha_s[h];
    }

    // pass 2: probabilities against the reference, rounded to bf16; the P buffer
    // (j & 1) is free once the value MMAs of tile j - 2 are done
    if (j >= 2) ptx::mbar_wait(&c.bar.vfree[(j - 2) % kR], ph_of(j - 2), c.abort);
    uint8_t* phi = c.pbuf + (j & 1) * SBuf<NP>::PB;
    const int row = c.myrow;
    const uint32_t row_off = row * 32;
    const uint32_t sw = ((row >> 2) & 1) << 4;
#pragma unroll
    for (int hc = 0; hc < NP / 16; ++hc) {
        float sc[16];
        load_scores<LO, NP>(tS + hc * 16, sc);
        uint32_t pk[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int h = hc * 16 + 2 * i;
            const float e0 = exp2f(sc[2 * i] - mref[h]);
            const float e1 = exp2f(sc[2 * i + 1] - mref[h + 1]);
            const float p0 = (row_ok && head_on<LO>(h, hlo, hn)) ? e0 : 0.f;
            const float p1 = (row_ok && head_on<LO>(h + 1, hlo, hn)) ? e1 : 0.f;
            l_part[h] += p0;
            l_part[h + 1] += p1;
            const __nv_bfloat162 h2 = __floats2bfloat162_rn(p0, p1);
            pk[i] = *reinterpret_cast<const uint32_t*>(&h2);
        }
        const uint32_t o0 = hc * kPAtom + row_off + (0u ^ sw);
        const uint32_t o1 = hc * kPAtom + row_off + (16u ^ sw);
        *reinterpret_cast<uint4*>(phi + o0) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        *reinterpret_cast<uint4*>(phi + o1) = make_uint4(pk[4], pk[5], pk[6], pk[7]);
    }
    ptx::tc_fence_before();          // TMEM reads / writes of this tile before the signal
    ptx::fence_proxy_async_smem();   // P stores visible to the tensor core
    ptx::mbar_arrive(&c.bar.vready[jr]);
}

// Partial write-out of a piece, out of line (once per piece): (m, l) of the real
// heads from the per-warp row-sum reductions in `red`, and the accumulator columns
// read from TMEM.
template <int NP>
__device__ __noinline__ void write_partial_acc(float* ml, float* acc, const float* red, const float* m_ref_s,
                                               int Hq, int Dmax, int slot, int dv, int nMB, int aw,
                                               uint32_t t_acc_lane, int tid, int myrow) {
    if (tid < Hq) {
        const float L = red[tid] + red[NP + tid] + red[2 * NP + tid] + red[3 * NP + tid];
        ml[((size_t)slot * 2) * Hq + tid] = m_ref_s[tid];
        ml[((size_t)slot * 2 + 1) * Hq + tid] = L;
    }
#pragma unroll 1
    for (int cc = 0; cc < nMB; ++cc) {
        const int r = cc * 128 + myrow;
#pragma unroll 1
        for (int hc = 0; hc < NP / 16; ++hc) {
            float v[16];
            const uint32_t ta = t_acc_lane + cc * aw + hc * 16;
            ptx::tmem_ld16(ta, v);
            if (r < dv) {
                float* dst = acc + ((size_t)slot * Hq + hc * 16) * Dmax + r;
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    if (hc * 16 + i < Hq) dst[(size_t)i * Dmax] = v[i];
            }
        }
    }
}

// End of a piece: reduce the row sums, write (m, l) and the accumulator columns of
// the real heads to partial slot `slot`.
template <int NP>
__device__ __forceinline__ void write_partial(const TcParams& p, const SoftCtx& c, int slot, int dv,
                                              float (&l_part)[NP]) {
    float v[NP];
#pragma unroll
    for (int h = 0; h < NP; ++h) v[h] = l_part[h];
#pragma unroll
    for (int hc = 0; hc < NP / 16; ++hc) {
        const float wsum = warp_reduce16<false>(v + hc * 16, c.lane);
        if (c.lane < 16) c.red[c.wq * NP + hc * 16 + c.lane] = wsum;
    }
    ptx::named_bar(1, 128);
    write_partial_acc<NP>(p.ml, p.acc, c.red, c.m_ref_s, p.Hq, p.Dmax, slot, dv, c.nMB, c.aw,
                          c.t_accp + c.lane_off, c.tid, c.myrow);
}


// ------------------------------------------------------------------ query images

// splitmix64 finaliser: spreads (channel, epoch) over 64 bits.
__device__ __forceinline__ unsigned long long mix64(unsigned long long x) {
    x += 0x9E3779B97F4A7C15ull;
    x = (x ^ (x >> 30)) * 0xBF58476D1CE4E5B9ull;
    x = (x ^ (x >> 27)) * 0x94D049BB133111EBull;
    return x ^ (x >> 31);
}

// The launch's token (one thread per CTA, after the grid-dependency wait, when the
// previous launch on this channel has completed): every CTA reads the channel's epoch
// and then checks in; the last to check in resets the count and advances the epoch for
// the next launch. The check-in is acquire-release, so no CTA can read an epoch that
// the last one already advanced. The token is never 0.
__device__ __forceinline__ unsigned long long launch_token(int ch) {
    const unsigned int e = *reinterpret_cast<volatile unsigned int*>(&g_chan_epoch[ch]);
    unsigned int old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(old) : "l"(&g_chan_count[ch]) : "memory");
    if (old == gridDim.x - 1) {
        *reinterpret_cast<volatile unsigned int*>(&g_chan_count[ch]) = 0u;
        *reinterpret_cast<volatile unsigned int*>(&g_chan_epoch[ch]) = e + 1u;
    }
    return mix64(((unsigned long long)(unsigned)ch << 32) | e) | 1ull;
}

__device__ __forceinline__ unsigned long long ld_acquire(const unsigned long long* p) {
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_release(unsigned long long* p, unsigned long long v) {
    asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
// Order this thread's generic-proxy global writes (or reads' visibility) with later
// async-proxy (bulk copy) accesses.
__device__ __forceinline__ void fence_proxy_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Whole warp: wait until the flags of CTAs [lo, hi] all hold `tok` (bounded; false
// and *abort raised if the wait runs out or *abort is raised elsewhere).
__device__ __noinline__ bool poll_flags_warp(const unsigned long long* flags, int lo, int hi, unsigned long long tok,
                                             volatile int* abort) {
    const int lane = threadIdx.x & 31;
    const uint64_t t0 = ptx::globaltimer();
    for (uint32_t it = 0;; ++it) {
        bool ok = true;
        for (int c = lo + lane; c <= hi; c += 32) ok = ok && ld_acquire(flags + c) == tok;
        if (__all_sync(0xffffffffu, ok)) return true;
        __nanosleep(64);   // leave issue slots and memory bandwidth to the working warps
        if (*abort) return false;
        if (ptx::globaltimer() - t0 > ptx::kWaitLimitNs) {
            *abort = 1;
            return false;
        }
    }
}
// One thread: the same wait, eight flags at a time.
__device__ __noinline__ bool poll_flags_thread(const unsigned long long* flags, int lo, int hi, unsigned long long tok,
                                               volatile int* abort) {
    const uint64_t t0 = ptx::globaltimer();
    int c = lo;
    while (c <= hi) {
        unsigned long long v[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) v[k] = c + k <= hi ? ld_acquire(flags + c + k) : tok;
        int k = 0;
        while (k < 8 && v[k] == tok) ++k;
        c += k;
        if (k < 8 && c <= hi) {
            __nanosleep(64);
            if (*abort) return false;
            if (ptx::globaltimer() - t0 > ptx::kWaitLimitNs) {
                *abort = 1;
                return false;
            }
        }
    }
    return true;
}

// 16-byte asynchronous global -> shared copy (completion via cp_async_wait_all).
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(ptx::smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

// Stage the 64-latent-column block cb of U_K^(g) (rows k < 128, 128 bytes each; columns
// past r_k are left alone) into `dst`, by the 128 softmax threads (tid).
__device__ __forceinline__ void stage_ublock(const TcParams& p, int g, int cb, uint8_t* dst, int tid) {
    const __nv_bfloat16* base = p.U_K + (size_t)g * 128 * p.r_k + cb * 64;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int ch = tid + i * 128, row = ch >> 3, part = ch & 7;
        if (cb * 64 + part * 8 < p.r_k) cp_async16(dst + row * 128 + part * 16, base + (size_t)row * p.r_k + part * 8);
    }
    cp_async_commit();
}

// Image units of batch element b, round-robin over the CTAs that work on b: per KV
// group g, ncb latent units (64 columns of q . U_K^(g) for the group's heads) and, if
// raw images are needed, one raw unit (the group's rows of the hi / lo image). Run by
// the 128 softmax threads (tid); qr is shared scratch for G x d floats, ub for one
// 64-column block of U_K^(g) (128 rows x 128 bytes). `staged` (g * ncb + cb, or -1)
// names a block already being copied into ub.
__device__ __noinline__ void make_image_units(const TcParams& p, int cta, int b, float* qr, uint8_t* ub, int& staged,
                                              int tid) {
    const int G = p.G, NP = (p.Hq + 15) / 16 * 16;
    const int per_g = p.ncb + p.img_raw;
    const int nunits = p.Hkv * per_g;
    const int n_b = p.cta_last[b] - p.cta_first[b] + 1;
    const unsigned long long pos = (unsigned long long)(long long)p.q_pos[b];
#pragma unroll 1
    for (int u = cta - p.cta_first[b]; u < nunits; u += n_b) {
        const int g = u / per_g, kind = u - g * per_g;
        ptx::named_bar(1, 128);   // the previous unit is done with qr and ub
        if (kind < p.ncb) {
            if (staged != g * p.ncb + kind) stage_ublock(p, g, kind, ub, tid);
            staged = -1;
        }
        // rotated, scaled query rows of the group's heads (pair i = item % 64)
#pragma unroll 1
        for (int it = tid; it < G * 64; it += 128) {
            const int hh = it >> 6, i = it & 63;
            const __nv_bfloat16* src = p.q + ((size_t)b * p.Hq + g * G + hh) * 128;
            const float x1 = __bfloat162float(src[i]), x2 = __bfloat162float(src[i + 64]);
            // the angle reduced to a signed fraction of a turn (exact 64-bit wrap-around)
            const long long frac = (long long)(pos * p.turn[i]);
            float sn, cs;
            sincospif((float)frac * 1.0842021724855044e-19f, &sn, &cs);   // x 2^-63: half-turns
            qr[hh * 128 + i] = (x1 * cs - x2 * sn) * p.scale_log2;
            qr[hh * 128 + i + 64] = (x2 * cs + x1 * sn) * p.scale_log2;
        }
        cp_async_wait_all();
        ptx::named_bar(1, 128);
        if (kind < p.ncb) {
            // latent unit: column kind * 64 + (tid % 64) of q . U_K^(g), heads tid / 64, + 2, ...
            const int cl = tid & 63, col = kind * 64 + cl;
            uint8_t* img = p.lat_img + (size_t)b * p.lat_img_bytes;
            if (col < p.r_k) {
                const __nv_bfloat16* uc = reinterpret_cast<const __nv_bfloat16*>(ub) + cl;
#pragma unroll 1
                for (int hh = tid >> 6; hh < G; hh += 2) {
                    const float4* q4 = reinterpret_cast<const float4*>(qr + hh * 128);
                    float acc = 0.f;
#pragma unroll 8
                    for (int k4 = 0; k4 < 32; ++k4) {
                        const float4 qv = q4[k4];
                        acc = fmaf(qv.x, __bfloat162float(uc[(4 * k4 + 0) * 64]), acc);
                        acc = fmaf(qv.y, __bfloat162float(uc[(4 * k4 + 1) * 64]), acc);
                        acc = fmaf(qv.z, __bfloat162float(uc[(4 * k4 + 2) * 64]), acc);
                        acc = fmaf(qv.w, __bfloat162float(uc[(4 * k4 + 3) * 64]), acc);
                    }
                    *reinterpret_cast<__nv_bfloat16*>(img + ptx::sw128_offset(g * G + hh, col, NP)) =
                        __float2bfloat16_rn(acc);
                }
                if (g == 0)   // rows of absent heads are zero
                    for (int h = p.Hq + (tid >> 6); h < NP; h += 2)
                        *reinterpret_cast<__nv_bfloat16*>(img + ptx::sw128_offset(h, col, NP)) = __float2bfloat16_rn(0.f);
            }
        } else {
            // raw unit: the group's rows of the raw image, bf16 high part and the bf16 of the rest
            uint8_t* img = p.raw_img + (size_t)b * p.raw_img_bytes;
#pragma unroll 1
            for (int it = tid; it < G * 16; it += 128) {
                const int hh = it >> 4, un = it & 15;
                const float* src = qr + hh * 128 + un * 8;
                uint32_t hi[4], lo[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const __nv_bfloat162 h2 = __floats2bfloat162_rn(src[2 * k], src[2 * k + 1]);
                    const float2 hf = __bfloat1622float2(h2);
                    const __nv_bfloat162 l2 = __floats2bfloat162_rn(src[2 * k] - hf.x, src[2 * k + 1] - hf.y);
                    hi[k] = *reinterpret_cast<const uint32_t*>(&h2);
                    lo[k] = *reinterpret_cast<const uint32_t*>(&l2);
                }
                const int h = g * G + hh;
                *reinterpret_cast<uint4*>(img + ptx::sw128_offset(h, un * 8, 2 * NP)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                *reinterpret_cast<uint4*>(img + ptx::sw128_offset(NP + h, un * 8, 2 * NP)) =
                    make_uint4(lo[0], lo[1], lo[2], lo[3]);
            }
            if (g == 0) {
                const int npad = NP - p.Hq;
#pragma unroll 1
                for (int it = tid; it < 2 * npad * 16; it += 128) {
                    const int pr = it >> 4, un = it & 15;
                    const int row = pr < npad ? p.Hq + pr : NP + p.Hq + (pr - npad);
                    *reinterpret_cast<uint4*>(img + ptx::sw128_offset(row, un * 8, 2 * NP)) = make_uint4(0u, 0u, 0u, 0u);
                }
            }
        }
    }
}

// The first latent unit this CTA makes (batch element and unit), or false if none.
__device__ __forceinline__ bool first_latent_unit(const TcParams& p, int cta, int b_lo, int b_hi, int& g, int& cb) {
    const int per_g = p.ncb + p.img_raw;
    if (p.ncb == 0) return false;
    for (int b = b_lo; b <= b_hi; ++b) {
        const int n_b = p.cta_last[b] - p.cta_first[b] + 1;
        for (int u = cta - p.cta_first[b]; u < p.Hkv * per_g; u += n_b) {
            const int kind = u % per_g;
            if (kind < p.ncb) {
                g = u / per_g;
                cb = kind;
                return true;
            }
        }
    }
    return false;
}

// NP: query heads rounded up to 16 (a template parameter, so the MMA issue sequences
// are straight-line code: a conditional branch between two tcgen05.mma instructions
// costs the issuing thread tens of cycles per MMA).
// At most 200 registers per thread: registers are allocated to warps in groups of four,
// so the 7 warps of a CTA hold 8 warps' worth, and a combine CTA (8 warps of 48) must
// still fit beside it on the SM.
template <int NP>
__global__ void __maxnreg__(200) tc_decode_kernel(const __grid_constant__ TcParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* ring = smem;
    uint8_t* qbuf = smem + p.off_q;          // query operand of the current piece (image copy)
    uint8_t* pbuf = smem + p.off_p;          // [2][NP/16 blocks][128 rows x 32 B] bf16
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + p.off_bar);
    float* red = reinterpret_cast<float*>(smem + p.off_red);   // [4][NP]
    float* m_ref_s = red + 4 * NP;                             // [NP]
    float* alpha_s = m_ref_s + NP;                             // [NP]
    // [0] abort; [1..8] per-tile votes, two tiles deep (a slow warp still reading
    // one tile's votes never sees the next tile's)
    volatile int* flag = reinterpret_cast<volatile int*>(alpha_s + NP);
    uint32_t* tmem_base_s = reinterpret_cast<uint32_t*>(alpha_s + NP) + 12;
    int* owner = reinterpret_cast<int*>(alpha_s + NP) + 16;    // [kMaxSlots] producer's slot owners
    volatile unsigned long long* tok_s = reinterpret_cast<volatile unsigned long long*>(alpha_s + NP) + 16;

    Bars bar;
    bar.kready = bars;
    bar.vready = bars + kR;
    bar.kfree = bars + 2 * kR;
    bar.vfree = bars + 3 * kR;
    bar.accfree = bars + 4 * kR;
    bar.drain = bars + 4 * kR + 2;      // [0] score issuer, [1] value issuer
    bar.qready = bars + 4 * kR + 4;
    bar.tok = bars + 4 * kR + 5;

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
        ptx::mbar_init(bar.tok, 1);
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
            // the first piece's images were checked by the score issuer before its first MMA
            int flags_b = u0 < u1 ? u0 / p.tiles_per_b : -1;
            unsigned long long tok = 0;
            // pending query-image copy (pieces after the first)
            bool q_pend = false;
            int q_tile = 0, q_after = 0;     // kready tile; tile whose score MMAs must finish first
            int q_b = 0;                     // batch element of the pending image
            const uint8_t* q_src = nullptr;
            uint32_t q_bytes = 0;
            auto try_q = [&](bool block) {
                if (!q_pend) return;
                if (block) {
                    ptx::mbar_wait(&bar.kfree[q_after % kR], ph_of(q_after), abort_flag);
                } else if (!ptx::mbar_test(&bar.kfree[q_after % kR], ph_of(q_after))) {
                    return;
                }
                if (q_b != flags_b) {
                    // another batch element: wait until its images are published
                    if (tok == 0) {
                        ptx::mbar_wait(bar.tok, 0, abort_flag);
                        tok = *tok_s;
                    }
                    poll_flags_thread(p.flags, p.cta_first[q_b], p.cta_last[q_b], tok, abort_flag);
                    flags_b = q_b;
                }
                fence_proxy_async_global();
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
            // Once the first two key tiles are on their way, pull the next pf_tiles tiles into
            // L2: they stream from HBM while the query images are made (the ring alone
            // would fill and stall), and their ring loads later hit L2.
            bool pf_done = p.pf_tiles == 0;
            auto prefetch_l2 = [&]() {
                TileIter pf;
                pf.init(p, u0, u1);
                if (pf.valid()) pf.next();
                if (pf.valid()) pf.next();
#pragma unroll 1
                for (int n = 0; n < p.pf_tiles && pf.valid(); ++n, pf.next()) {
                    const int k = pf.pc.k;
#pragma unroll 1
                    for (int part = 0; part < 2; ++part) {
                        const int w = part ? p.dv[k] : p.dk[k];
#pragma unroll 1
                        for (int col = 0; col < w; col += 64)
                            ptx::tma_prefetch_3d(&p.tm[2 * k + part], col, pf.t * kTile, pf.pc.b);
                    }
                }
                pf_done = true;
            };
#pragma unroll 1
            while (vit.valid() && !*abort_flag) {
                if (!pf_done && kiss >= 2) prefetch_l2();
                const bool isK = kit.valid() && kit.j <= vit.j + 1;
                TileIter ti = isK ? kit : vit;
                const int part = isK ? 0 : 1;
                const int k = ti.pc.k;
                const CUtensorMap* tm = &p.tm[2 * k + part];
                const int nc = ((part ? p.dv[k] : p.dk[k]) + 127) >> 7;   // slots: 128-column chunks
#pragma unroll 1
                for (int c = 0; c < nc; ++c) slot_free(ring_wrap(pos + c, p.nslot));
                const int jr = ti.j % kR;
                if (part == 0) {
                    if (ti.first() && ti.j > 0) {
                        if (q_pend) try_q(true);   // the previous piece's image goes first
                        query_image(p, ti.pc, q_src, q_bytes);
                        ptx::mbar_expect_tx_only(&bar.kready[jr], q_bytes);
                        q_b = ti.pc.b;
                        q_pend = true;
                        q_tile = ti.j;
                        q_after = ti.j - 1;
                    }
                    ptx::mbar_expect_tx(&bar.kready[jr], nc * kSlot);
                } else {
                    ptx::mbar_expect_tx(&bar.vready[jr], nc * kSlot);
                }
                uint64_t* rb = part ? &bar.vready[jr] : &bar.kready[jr];
                const int row = ti.t * kTile;
#pragma unroll 1
                for (int c = 0; c < nc; ++c) {
                    const int s = ring_wrap(pos + c, p.nslot);
                    uint8_t* dst = ring + (size_t)s * kSlot;
                    ptx::tma_load_3d_hint(dst, tm, c * 128, row, ti.pc.b, rb, pol);
                    ptx::tma_load_3d_hint(dst + kBox, tm, c * 128 + 64, row, ti.pc.b, rb, pol);
                    owner[s] = (ti.j << 1) | part;
                }
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
        bool first_ok = true;
        if (s_issuer && u0 < u1) {
            // the CTA's first query image: published by the CTAs of its batch element in
            // this launch (the whole warp polls their flags)
            const int b = u0 / p.tiles_per_b;
            ptx::mbar_wait(bar.tok, 0, abort_flag);
            first_ok = poll_flags_warp(p.flags, p.cta_first[b], p.cta_last[b], *tok_s, abort_flag);
        }
        if (lane == 0) {
            const uint32_t idS_lat = ptx::idesc_bf16(128, NP, false, false);
            const uint32_t idS_raw = ptx::idesc_bf16(128, 2 * NP, false, false);
            const uint32_t idV = ptx::idesc_bf16(128, NP, true, true);
            // base descriptors; a k-step or ring slot only adds (byte offset >> 4) to
            // the start-address field, which stays below 2^14 for shared memory
            const uint64_t dA_S = ptx::sdesc_sw128(ptx::smem_u32(ring), 16, 1024);      // K tile, K-major
            const uint64_t dA_V = ptx::sdesc_sw128(ptx::smem_u32(ring), kBox, 1024);    // V tile, MN-major
            const uint64_t dB_Q = ptx::sdesc_sw128(ptx::smem_u32(qbuf), 16, 1024);      // Q, K-major
            const uint64_t dB_P = ptx::sdesc_sw32(ptx::smem_u32(pbuf), kPAtom, 256);    // P, MN-major
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
                // latent tiles: N = heads (one bf16 part of the latent query); raw tiles:
                // N = 2 x heads (hi and lo parts). Q is stored in 64-column chunks of N rows.
                const bool lat = ti.pc.k == 0;
                const uint32_t idS = lat ? idS_lat : idS_raw;
                const uint32_t qstride = (lat ? NP : 2 * NP) * 128 >> 4;
                const int ksteps = p.dk[ti.pc.k] >> 4;
                const int nK = (p.dk[ti.pc.k] + 127) >> 7;
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
                                      b0 + (uint64_t)((kk >> 2) * qstride + (kk & 3) * 2), idS, kk == 0 ? acc0 : 1u);
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
                                      b0 + (uint64_t)((kk >> 2) * qstride + (kk & 3) * 2), idS, (c | kk) != 0 ? 1u : 0u);
                }
                pos = ring_wrap(pos + nK, p.nslot);
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
                const uint64_t pd = dB_P + (uint64_t)(((ti.j & 1) * SBuf<NP>::PB) >> 4);
                const int nV = (p.dv[ti.pc.k] + 127) >> 7;
#pragma unroll 1
                for (int c = 0; c < nV; ++c) {
                    const int s = ring_wrap(pos + c, p.nslot);
                    const uint64_t vd = dA_V + (uint64_t)((s * kSlot) >> 4);
                    const uint32_t d0 = abase + c * aw;
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const uint64_t a = vd + (uint64_t)(kk * (2048 >> 4));
                        const uint64_t b = pd + (uint64_t)(kk * (512 >> 4));
                        ptx::mma_bf16(d0, a, b, idV, kk == 0 ? acc0 : 1u);
                    }
                }
                pos = ring_wrap(pos + nV, p.nslot);
                ptx::mma_commit(&bar.vfree[jr]);
            };

            TileIter kit, vit;
            kit.init(p, u0, u1);
            vit.init(p, u0, u1);
            if (s_issuer && kit.valid()) {
                // the CTA's first query image (its own barrier: the key and value loads
                // never wait for it)
                const uint8_t* q_src;
                uint32_t q_bytes;
                query_image(p, kit.pc, q_src, q_bytes);
                if (first_ok) {
                    fence_proxy_async_global();
                    ptx::mbar_expect_tx(bar.qready, q_bytes);
                    ptx::bulk_load(qbuf, q_src, q_bytes, bar.qready);
                    ptx::mbar_wait(bar.qready, 0, abort_flag);
                } else {
                    ptx::mbar_arrive(bar.qready);   // nothing to copy: the kernel is winding down
                }
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
                    pos = ring_wrap(pos + (((isK ? p.dk[k] : p.dv[k]) + 127) >> 7), p.nslot);
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
        c.red = red;
        c.m_ref_s = m_ref_s;
        c.alpha_s = alpha_s;
        c.flags = flag + 1;
        c.abort = abort_flag;
        c.tid = threadIdx.x - 64;            // 0..127
        c.wq = c.tid >> 5;                   // softmax warp 0..3
        c.lane = lane;
        const int q4 = warp & 3;             // TMEM lane quadrant this warp may access
        c.myrow = q4 * 32 + lane;            // tile row (S) / value row (acc) of this thread
        c.lane_off = (uint32_t)(q4 * 32) << 16;
        c.t_S = t_S;
        c.aw = aw;
        float l_part[NP];

        // ---- query images: this CTA's units of the batch elements its run touches
        const int b_lo = u0 / p.tiles_per_b, b_hi = (u1 - 1) / p.tiles_per_b;
        // U_K blocks of this CTA's latent units (weights, read before the wait): the first
        // is copied into the query buffer (free until the first image is copied, which
        // waits for this CTA's flag), the others are pulled into L2
        int staged = -1;
        {
            int g0, cb0;
            if (first_latent_unit(p, cta, b_lo, b_hi, g0, cb0)) {
                stage_ublock(p, g0, cb0, qbuf, c.tid);
                staged = g0 * p.ncb + cb0;
            }
            const int per_g = p.ncb + p.img_raw;
#pragma unroll 1
            for (int b = b_lo; b <= b_hi && p.ncb > 0; ++b) {
                const int n_b = p.cta_last[b] - p.cta_first[b] + 1;
#pragma unroll 1
                for (int u = cta - p.cta_first[b]; u < p.Hkv * per_g; u += n_b) {
                    const int g = u / per_g, cb = u - g * per_g;
                    if (cb < p.ncb && g * p.ncb + cb != staged) {
                        const char* row = reinterpret_cast<const char*>(p.U_K + ((size_t)g * 128 + c.tid) * p.r_k + cb * 64);
                        asm volatile("prefetch.global.L2 [%0];" ::"l"(row));
                    }
                }
            }
        }
        // the workspace partials and images may still be read by the preceding calls'
        // kernels, and q / q_pos may be written by the preceding kernel
        pdl_wait();
        unsigned long long tok = 0;
        if (c.tid == 0) {
            tok = launch_token(p.ch);
            *tok_s = tok;
            ptx::mbar_arrive(bar.tok);
        }
        float* qr = reinterpret_cast<float*>(pbuf);   // scratch until the first P is written
#pragma unroll 1
        for (int b = b_lo; b <= b_hi; ++b) make_image_units(p, cta, b, qr, qbuf, staged, c.tid);
        fence_proxy_async_global();
        __threadfence();
        ptx::named_bar(1, 128);
        if (c.tid == 0) st_release(p.flags + cta, tok);

        TileIter it;
        it.init(p, u0, u1);
        while (it.valid()) {
            const Piece pc = it.pc;
            const int piece = it.piece;
            const int k = pc.k;
            const bool lat = (k == 0);
            c.nMB = (p.dv[k] + 127) >> 7;
            c.t_accp = t_acc + (uint32_t)((p.accbuf == 2 ? (piece & 1) : 0) * p.accstride);
            if (c.tid < NP) m_ref_s[c.tid] = -INFINITY;
#pragma unroll
            for (int h = 0; h < NP; ++h) l_part[h] = 0.f;
            ptx::named_bar(1, 128);
            int jl = it.j;
            #pragma unroll 1
            for (int n = 0; n < pc.n; ++n) {
                const int row = it.t * kTile + c.myrow;   // row of this thread inside the segment
                const bool row_ok = row < p.rows[k];
                jl = it.j;
                if (lat) {
                    softmax_tile<NP, false>(c, it.j, row_ok, 0, NP, it.t > pc.t0, l_part);
                } else {
                    // raw row = token * Hkv + KV group: the row is scored by its group's heads
                    const int hlo = (row % p.Hkv) * p.G;
                    softmax_tile<NP, true>(c, it.j, row_ok, hlo, p.G, it.t > pc.t0, l_part);
                }
                it.next();
            }
            // ---- partial of (CTA, piece): reference max, row sum and accumulator
            ptx::mbar_wait(&bar.vfree[jl % kR], ph_of(jl), abort_flag);   // V(jl) complete
            ptx::tc_fence_after();
            write_partial<NP>(p, c, p.slot_base[cta] + piece, p.dv[k], l_part);
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
        // a wait ran out: poison this CTA's partials so the result is NaN, not stale
        const int tid = threadIdx.x - 64;
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
    int NP, nslot, accbuf, accstride;
    uint32_t off_q, off_p, off_bar, off_red, total, tmem_cols;
    bool ok;
};

int round_up(int x, int m) { return (x + m - 1) / m * m; }

// Plan within `budget` bytes of dynamic shared memory.
SmemPlan plan_smem_within(int Hq, const int dk[kNumKinds], const int dv[kNumKinds], const int rows[kNumKinds],
                          int budget) {
    SmemPlan s{};
    s.NP = round_up(Hq, 16);
    int nmb = 0, maxK = 0, maxV = 0;
    bool raw = false;
    for (int k = 0; k < kNumKinds; ++k) {
        if (rows[k] <= 0) continue;
        raw = raw || k > 0;
        nmb = std::max(nmb, (dv[k] + 127) / 128);
        maxK = std::max(maxK, (dk[k] + 127) / 128);   // ring slots of a tile's keys
        maxV = std::max(maxV, (dv[k] + 127) / 128);
    }
    s.ok = false;
    if (s.NP > 64) return s;
    // TMEM: two score buffers of 2 NP columns, then one or two accumulator buffers
    // (two when they fit, so a piece's write-out overlaps the next piece)
    const int sw = 2 * s.NP;
    s.accstride = nmb * s.NP;
    int tmem = 0;
    for (s.accbuf = 2; s.accbuf >= 1; --s.accbuf) {
        tmem = 2 * sw + s.accbuf * s.accstride;
        if (tmem <= 512) break;
    }
    if (tmem > 512) return s;
    s.tmem_cols = 32;
    while ((int)s.tmem_cols < tmem) s.tmem_cols *= 2;
    // query buffer: the latent image (NP rows, bf16) or the raw image (hi and lo parts);
    // before the first image it stages a 128 x 64 block of U_K (16 KB) for the latent image
    const int q_bytes = std::max({rows[0] > 0 ? s.NP * round_up(dk[0], 64) * 2 : 0, rows[0] > 0 ? 128 * 128 : 0,
                                  raw ? 2 * s.NP * 128 * 2 : 0});
    const int p_bytes = 2 * s.NP * 256;   // two P buffers (bf16)
    const int nbars = 4 * kR + 6;
    // red, m_ref, alpha (6 NP floats), then flags, TMEM base, slot owners and the token
    const int misc_bytes = (6 * s.NP + 40) * 4;
    const int avail = budget - q_bytes - p_bytes - round_up(nbars * 8, 16) - misc_bytes - 1024;
    s.nslot = std::min(kMaxSlots, avail / kSlot);
    // One tile part (keys or values) must fit the ring. The loads run in consumption
    // order and each waits only for earlier parts to be consumed, so a ring smaller
    // than a key plus a value tile (latent ranks above 256) still drains: it only
    // serialises those tiles' loads behind their consumers.
    if (s.nslot < std::max(maxK, maxV)) return s;
    s.off_q = s.nslot * kSlot;
    s.off_p = s.off_q + q_bytes;
    s.off_bar = s.off_p + p_bytes;
    s.off_red = s.off_bar + round_up(nbars * 8, 16);
    s.total = s.off_red + misc_bytes + 1024;
    s.ok = s.total <= (uint32_t)budget;
    return s;
}

// The shared budget when the ring still holds a key and a value tile part, else the
// whole of what a CTA may use.
SmemPlan plan_smem(int Hq, const int dk[kNumKinds], const int dv[kNumKinds], const int rows[kNumKinds]) {
    int maxKV = 0;
    for (int k = 0; k < kNumKinds; ++k)
        if (rows[k] > 0) maxKV = std::max(maxKV, (dk[k] + 127) / 128 + (dv[k] + 127) / 128);
    const SmemPlan s = plan_smem_within(Hq, dk, dv, rows, kSmemShared);
    if (s.ok && s.nslot > maxKV) return s;
    return plan_smem_within(Hq, dk, dv, rows, kSmemMax);
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

// A segment operand: 3-D bf16 tensor [B][rows][cols] (cols contiguous) read in boxes of
// 128 rows x 64 columns with the 128-byte swizzle; rows / columns past the end read as zero.
bool make_map(CUtensorMap* tm, const void* base, int cols, int64_t rows, int B) {
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

// Encoded tensor maps are reused by later calls on the same buffers and sizes
// (encoding is a driver call; a decode step makes four per layer). Direct-mapped.
bool cached_map(CUtensorMap* tm, const void* base, int cols, int64_t rows, int B) {
    struct Entry {
        bool valid = false;
        const void* base = nullptr;
        int cols = 0, B = 0;
        int64_t rows = 0;
        CUtensorMap tm;
    };
    static std::mutex mu;
    static Entry cache[512];
    const uint64_t h = ((uint64_t)(uintptr_t)base >> 8) * 0x9E3779B97F4A7C15ull ^
                       ((uint64_t)cols * 31 + (uint64_t)rows) * 0xBF58476D1CE4E5B9ull ^ (uint64_t)B;
    Entry& e = cache[(h >> 40) % 512];
    {
        std::lock_guard<std::mutex> g(mu);
        if (e.valid && e.base == base && e.cols == cols && e.rows == rows && e.B == B) {
            *tm = e.tm;
            return true;
        }
    }
    if (!make_map(tm, base, cols, rows, B)) return false;
    std::lock_guard<std::mutex> g(mu);
    e.valid = true;
    e.base = base;
    e.cols = cols;
    e.rows = rows;
    e.B = B;
    e.tm = *tm;
    return true;
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

// Launch-token channel of a workspace on the current device: each workspace in use
// keeps its own channel, so that launches on different workspaces (which may run
// concurrently on different streams) never share an epoch. When more than kChannels
// workspaces are in use, the least recently used one gives up its channel.
int channel_for(const void* ws) {
    struct Dev {
        std::map<const void*, int> of;
        const void* owner[kChannels] = {};
        uint64_t last[kChannels] = {};
        uint64_t tick = 0;
    };
    static std::mutex mu;
    static Dev devs[64];
    int dev = 0;
    cudaGetDevice(&dev);
    Dev& d = devs[dev & 63];
    std::lock_guard<std::mutex> g(mu);
    ++d.tick;
    auto it = d.of.find(ws);
    if (it != d.of.end()) {
        d.last[it->second] = d.tick;
        return it->second;
    }
    int ch = 0;
    for (int i = 1; i < kChannels; ++i)
        if (d.last[i] < d.last[ch]) ch = i;
    if (d.owner[ch] != nullptr) d.of.erase(d.owner[ch]);
    d.owner[ch] = ws;
    d.last[ch] = d.tick;
    d.of[ws] = ch;
    return ch;
}

struct PlanKey {
    int B, max_ctas;
    std::vector<std::pair<int, int>> segs;
    bool operator<(const PlanKey& o) const { return std::tie(B, max_ctas, segs) < std::tie(o.B, o.max_ctas, o.segs); }
};

// Plans are built once per (batch, segment list, grid limit) and shared: the cache
// hands out shared ownership, so a plan stays valid for a caller even when another
// thread clears the cache.
std::shared_ptr<const WorkPlan> cached_plan(int B, const SegList& sl, int max_ctas) {
    static std::mutex mu;
    static std::map<PlanKey, std::shared_ptr<const WorkPlan>> cache;
    PlanKey key{B, max_ctas, sl.segs};
    std::lock_guard<std::mutex> g(mu);
    auto it = cache.find(key);
    if (it != cache.end()) return it->second;
    if (cache.size() > 256) cache.clear();
    auto w = std::make_shared<const WorkPlan>(make_plan(B, sl, max_ctas));
    cache.emplace(std::move(key), w);
    return w;
}

template <int NP>
cudaError_t launch_decode(const TcParams& prm, int grid, uint32_t smem, cudaStream_t st) {
    static std::atomic<unsigned long long> attr_done{0};
    const cudaError_t ea = set_max_smem_once((const void*)tc_decode_kernel<NP>, kSmemMax, attr_done);
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
    return cudaLaunchKernelEx(&cfg, tc_decode_kernel<NP>, prm);
}

// Kinds of key rows of one call: rows / widths per segment and operands.
struct Kinds {
    int64_t rows[kNumKinds] = {0, 0, 0};
    int dk[kNumKinds] = {0, 0, 0};
    int dv[kNumKinds] = {0, 0, 0};
    const void* K[kNumKinds] = {nullptr, nullptr, nullptr};
    const void* V[kNumKinds] = {nullptr, nullptr, nullptr};
};

Kinds kinds_of(const TcCall& c) {
    Kinds s;
    // a raw source [B, T, Hkv, d] is read as [B, T * Hkv, d]
    auto raw = [&](int k, int T, const void* K, const void* V) {
        if (T <= 0) return;
        s.rows[k] = (int64_t)T * c.Hkv;
        s.dk[k] = s.dv[k] = c.d;
        s.K[k] = K;
        s.V[k] = V;
    };
    if (c.which == SLIMKV_LATENT) {
        if (c.N_b > 0) {
            s.rows[0] = c.N_b;
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
    if (d != 128 || Hq > 64 || Hkv > Hq) return false;
    int rows[kNumKinds] = {N_b, 1, 1}, dk[kNumKinds] = {r_k, d, d}, dv[kNumKinds] = {r_v, d, d};
    if (N_b <= 0) rows[0] = 0;
    return plan_smem(Hq, dk, dv, rows).ok;
}

cudaError_t tc_run(const TcCall& c, cudaStream_t st) {
    typedef __nv_bfloat16 bf16;
    const bool lat = c.which == SLIMKV_LATENT && c.N_b > 0;
    const bool has_raw = c.which != SLIMKV_LATENT || c.W > 0;
    cudaError_t e = cudaSuccess;
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
    int rows_i[kNumKinds];
    for (int k = 0; k < kNumKinds; ++k) rows_i[k] = s.rows[k] > 0 ? 1 : 0;
    const SmemPlan sp = plan_smem(c.Hq, s.dk, s.dv, rows_i);
    if (!sp.ok) return cudaErrorInvalidValue;

    TcParams prm;   // copied into the launch's parameter space
    memset(&prm, 0, sizeof(prm));
    SegList sl;
    int lat_segs = 0;   // segments of a batch element before the first raw one
    prm.tiles_per_b = 0;
    for (int k = 0; k < kNumKinds; ++k) {
        prm.rows[k] = (int)s.rows[k];
        prm.dk[k] = s.dk[k];
        prm.dv[k] = s.dv[k];
        const int tiles = s.rows[k] > 0 ? (int)((s.rows[k] + kTile - 1) / kTile) : 0;
        prm.tiles[k] = tiles;
        prm.tiles_per_b += tiles;
        if (tiles == 0) continue;
        // cost of a tile: the 32 KB slots it streams (+1 for its fixed per-tile work)
        const int cost = (s.dk[k] + 127) / 128 + (s.dv[k] + 127) / 128 + 1;
        sl.segs.push_back({tiles, cost});
        if (k == 0) lat_segs = 1;
        if (!cached_map(&prm.tm[2 * k], s.K[k], s.dk[k], s.rows[k], c.B) ||
            !cached_map(&prm.tm[2 * k + 1], s.V[k], s.dv[k], s.rows[k], c.B))
            return cudaErrorInvalidValue;
    }
    const std::shared_ptr<const WorkPlan> wp = cached_plan(c.B, sl, std::min(kMaxCtas, sm_count()));
    const WorkPlan& w = *wp;
    if (w.slots > c.slots) return cudaErrorInvalidValue;
    prm.B = c.B;
    prm.Hq = c.Hq;
    prm.Hkv = c.Hkv;
    prm.G = c.Hq / c.Hkv;
    prm.lat_img = c.lat_img;
    prm.raw_img = c.raw_img;
    prm.lat_img_bytes = (uint32_t)lat_img_bytes(sp.NP, c.r_k);
    prm.raw_img_bytes = (uint32_t)raw_img_bytes(sp.NP, c.d);
    prm.acc = c.acc;
    prm.ml = c.ml;
    prm.Dmax = c.Dmax;
    prm.nslot = sp.nslot;
    prm.accbuf = sp.accbuf;
    prm.accstride = sp.accstride;
    prm.off_q = sp.off_q;
    prm.off_p = sp.off_p;
    prm.off_bar = sp.off_bar;
    prm.off_red = sp.off_red;
    prm.tmem_cols = sp.tmem_cols;
    for (int i = 0; i <= w.n_ctas; ++i) prm.u_begin[i] = w.u_begin[i];
    for (int i = 0; i < w.n_ctas; ++i) prm.slot_base[i] = w.slot_base[i];
    // query images: the CTAs whose runs touch batch element b make b's images
    prm.q = (const bf16*)c.q;
    prm.U_K = lat ? (const bf16*)c.U_K : nullptr;
    prm.q_pos = c.q_pos;
    prm.flags = c.flags;
    prm.ch = channel_for(c.flags);
    prm.r_k = c.r_k;
    prm.ncb = lat ? (c.r_k + 63) / 64 : 0;
    {
        // about kPrefetchBytes per CTA, in tiles of the largest kind
        int tile_bytes = 0;
        for (int k = 0; k < kNumKinds; ++k)
            if (s.rows[k] > 0) tile_bytes = std::max(tile_bytes, kTile * (s.dk[k] + s.dv[k]) * 2);
        prm.pf_tiles = tile_bytes > 0 ? kPrefetchBytes / tile_bytes : 0;
    }
    prm.img_raw = has_raw ? 1 : 0;
    prm.scale_log2 = c.scale_log2;
    rope_turns(c.rope_base, c.d, prm.turn);
    for (int b = 0; b < c.B; ++b) prm.cta_first[b] = -1;
    for (int i = 0; i < w.n_ctas; ++i) {
        const int b0 = w.u_begin[i] / prm.tiles_per_b, b1 = (w.u_begin[i + 1] - 1) / prm.tiles_per_b;
        for (int b = b0; b <= b1; ++b) {
            if (prm.cta_first[b] < 0) prm.cta_first[b] = (short)i;
            prm.cta_last[b] = (short)i;
        }
    }

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
    cb.out = c.out;
    for (int b = 0; b <= c.B; ++b) cb.slot_begin[b] = w.batch_slot[b];
    for (int b = 0; b < c.B; ++b) cb.slot_mid[b] = plan::first_slot_from_seg(w, b, lat_segs);
    return launch_combine<bf16>(cb, st, true);
}

}  // namespace slimkv

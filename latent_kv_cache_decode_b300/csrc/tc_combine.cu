// Split combine of the tensor-core path, fused with the value up-projection.
//
// "Can SlimKV compress KV cache jointly across tokens and features", section
// "Latent-space attention removes the rebuild step": the latent aggregate A C_V is
// up-projected once by U_V^(g) after every beacon split has been merged, and the raw
// window's aggregate A V_raw is added in full dimension. The partials of one batch
// element b (m, l, acc per head, written by the decode kernel) are merged by their
// log2-domain maxima:
//   M = max_s m_s, w_s = exp2(m_s - M), L = sum_s w_s l_s,
//   z = sum_{latent s} w_s acc_s (r_v wide), y = sum_{raw s} w_s acc_s (d wide),
//   out[b, h, :] = (z . U_V^(g)T + y) / L.
// A partial with l = 0 covered no key of that head and is skipped; a NaN l (a decode
// CTA that gave up on a wait) propagates into the output.
//
// One CTA per (KV group g, chunk of <= 4 of its heads, batch element b, block of 32
// output rows), 256 threads. The kernel sits on the critical path between two layers,
// so it is built for latency: the CTA's 32 rows of U_V^(g) are copied into shared
// memory before the grid-dependency wait (they are weights); after the wait every
// thread issues the loads of its partial values (the slots of b are laid out latent
// first, then raw, so the host knows where each list starts) while one warp reads every
// partial's (kind, m, l) and forms the merge weights: one memory round in all. The
// up-projection runs from shared memory with every thread busy: thread (row, column
// block) sums 32 latent columns of each 256-column chunk, and the 8 blocks of a row are
// added across lanes.
#include "slimkv_internal.cuh"
#include "tc_ptx.cuh"

namespace slimkv {

namespace {

constexpr int kThreads = 256;
constexpr int kHeads = 4;    // heads per CTA
constexpr int kRows = 32;    // output rows per CTA
constexpr int kUCols = 256;  // latent columns of U_V^(g) staged in shared memory before the wait
constexpr int kBatch = 8;    // partial values of each item loaded before their sum

// 16-byte asynchronous global -> shared copy (completion via cp_async_wait_all).
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(ptx::smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ float bf16lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

__global__ void __maxnreg__(96) tc_combine_kernel(const __grid_constant__ CombineArgs a) {
    extern __shared__ __align__(16) float dyn[];
    __shared__ float L_s[kHeads];
    const int d = a.d;
    const int G = a.Hq / a.Hkv, nhc = (G + kHeads - 1) / kHeads;
    const int g = blockIdx.x / nhc, hc = blockIdx.x - g * nhc, b = blockIdx.y, i0 = blockIdx.z * kRows;
    const int h0 = g * G + hc * kHeads, nh = min(kHeads, G - hc * kHeads);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const bool latent = a.U_V != nullptr;
    const int r_v = latent ? a.r_v : 0;

    // U_V^(g)[i0 : i0 + 32, 0:256): a weight, copied into shared memory before the
    // dependency wait (rows ustride bytes apart: the 16-byte padding spreads a warp's rows
    // over the banks)
    const int ucols = min(r_v, kUCols), ustride = ucols * 2 + 16;
    uint8_t* u_s = reinterpret_cast<uint8_t*>(dyn);
    const __nv_bfloat16* ug =
        latent ? reinterpret_cast<const __nv_bfloat16*>(a.U_V) + ((size_t)g * d + i0) * r_v : nullptr;
    if (latent) {
        const int cpr = ucols / 8;   // 16-byte chunks per row
#pragma unroll 1
        for (int i = tid; i < kRows * cpr; i += kThreads) {
            const int row = i / cpr, c = i - row * cpr;
            cp_async16(u_s + row * ustride + c * 16, ug + (size_t)row * r_v + c * 8);
        }
        cp_async_commit();
    }
    pdl_trigger();
    pdl_wait();   // the partials come from the decode kernel

    // slots of b: latent partials [s0, sm), raw partials [sm, s1) (the raw ones of other
    // KV groups do not cover this CTA's heads and get weight 0)
    const int s0 = a.slot_begin[b], sm = a.slot_mid[b], s1 = a.slot_begin[b + 1];
    const int ns = s1 - s0, nsp = a.ns_max;
    float* w_s = dyn + (latent ? kRows * ustride / 4 : 0);   // [nsp][4] m, then the weight
    float* l_s = w_s + nsp * kHeads;                         // [nsp][4]
    // z: [chunk][4 heads][8 column blocks][32 + 4] (the padding spreads the blocks over
    // the banks); y: [4][32]
    float* z_s = l_s + nsp * kHeads;
    const int zchunks = (r_v + 255) / 256;
    float* y_s = z_s + zchunks * kHeads * 8 * 36;
    const size_t sstride = (size_t)a.Hq * a.Dmax;
    const int zq = r_v / 4, nz = kHeads * zq, nitems = nz + kHeads * (kRows / 4);

    // value loads of this thread's first two items, issued before the merge weights are known
    // (one memory round for the loads and the weights' (kind, m, l), which warp 0 reads)
    int it_ih[2], it_first[2], it_n[2];
    size_t it_off[2];
    float* it_dst[2];
    float4 v[2][kBatch];
    // warps 1..7 take the items (warp 0 forms the weights meanwhile)
    constexpr int kIt = kThreads - 32;
    const int it_tid = tid - 32;
    auto setup = [&](int round) {
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            const int item = warp == 0 ? nitems : round * 2 * kIt + q * kIt + it_tid;
            const bool zi = item < nz;
            const int j = zi ? item : item - nz;
            const int per = zi ? zq : kRows / 4;
            const int ih = j / per, c4 = (j - ih * per) * 4;
            const bool on = item < nitems && ih < nh;
            it_ih[q] = ih;
            it_first[q] = zi ? s0 : sm;
            it_n[q] = on ? (zi ? sm - s0 : s1 - sm) : 0;
            it_off[q] = (size_t)(h0 + ih) * a.Dmax + (zi ? c4 : i0 + c4);
            it_dst[q] = item >= nitems ? nullptr
                        : zi ? z_s + (((c4 >> 8) * kHeads + ih) * 8 + ((c4 & 255) >> 5)) * 36 + (c4 & 31)
                             : y_s + ih * kRows + c4;
        }
    };
    auto load = [&](int k0) {
#pragma unroll
        for (int q = 0; q < 2; ++q)
#pragma unroll
            for (int k = 0; k < kBatch; ++k)
                v[q][k] = k0 + k < it_n[q] ? *reinterpret_cast<const float4*>(
                                                  a.acc + (size_t)(it_first[q] + k0 + k) * sstride + it_off[q])
                                           : make_float4(0.f, 0.f, 0.f, 0.f);
    };
    if (warp > 0) {
        setup(0);
        load(0);
    } else {
        // merge weights of the chunk's heads: lane = slot, 32 slots at a time
        float mx[kHeads] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll 1
        for (int base = 0; base < ns; base += 32) {
            const int s = base + lane;
            if (s >= ns) continue;
            // kind, m and l in one memory round (the (m, l) of a slot that does not cover
            // this CTA's heads are read and dropped)
            const int kd = a.kind[s0 + s];
            float mm[kHeads], ll[kHeads];
#pragma unroll
            for (int k = 0; k < kHeads; ++k) {
                const int hk = h0 + min(k, nh - 1);
                mm[k] = a.ml[((size_t)(s0 + s) * 2) * a.Hq + hk];
                ll[k] = a.ml[((size_t)(s0 + s) * 2 + 1) * a.Hq + hk];
            }
            const bool cover = s0 + s < sm ? (latent && kd == kSlotLatent) : (kd == kSlotRawAll || kd == kSlotRawGroup + g);
            float m[kHeads], l[kHeads];
#pragma unroll
            for (int k = 0; k < kHeads; ++k) {
                m[k] = -INFINITY;
                l[k] = 0.f;
                if (k < nh && cover && ll[k] != 0.f) {   // a NaN (poisoned) l is kept
                    m[k] = mm[k];
                    l[k] = ll[k];
                }
                mx[k] = fmaxf(mx[k], m[k]);
            }
            *reinterpret_cast<float4*>(w_s + s * kHeads) = make_float4(m[0], m[1], m[2], m[3]);
            *reinterpret_cast<float4*>(l_s + s * kHeads) = make_float4(l[0], l[1], l[2], l[3]);
        }
#pragma unroll
        for (int k = 0; k < kHeads; ++k)
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) mx[k] = fmaxf(mx[k], __shfl_xor_sync(0xffffffffu, mx[k], o));
        float lsum[kHeads] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
        for (int s = lane; s < ns; s += 32) {
            const float4 m4 = *reinterpret_cast<const float4*>(w_s + s * kHeads);
            const float4 l4 = *reinterpret_cast<const float4*>(l_s + s * kHeads);
            const float mm[kHeads] = {m4.x, m4.y, m4.z, m4.w}, ll[kHeads] = {l4.x, l4.y, l4.z, l4.w};
            float w[kHeads];
#pragma unroll
            for (int k = 0; k < kHeads; ++k) {
                w[k] = mm[k] == -INFINITY ? 0.f : exp2f(mm[k] - mx[k]);
                lsum[k] = fmaf(w[k], ll[k], lsum[k]);
            }
            *reinterpret_cast<float4*>(w_s + s * kHeads) = make_float4(w[0], w[1], w[2], w[3]);
        }
#pragma unroll
        for (int k = 0; k < kHeads; ++k)
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) lsum[k] += __shfl_xor_sync(0xffffffffu, lsum[k], o);
        if (lane < kHeads) L_s[lane] = lane == 0 ? lsum[0] : lane == 1 ? lsum[1] : lane == 2 ? lsum[2] : lsum[3];
    }
    __syncthreads();

    // z[hh, :] and y[hh, i0 : i0 + 32): weighted sums of the loaded values (a slot of weight 0
    // is skipped, not multiplied: the raw partials of other groups hold no values for these heads)
#pragma unroll 1
    for (int round = 0; warp > 0 && round * 2 * kIt < nitems; ++round) {
        if (round > 0) {
            setup(round);
            load(0);
        }
        float4 r[2] = {make_float4(0.f, 0.f, 0.f, 0.f), make_float4(0.f, 0.f, 0.f, 0.f)};
        const int nmax = max(it_n[0], it_n[1]);
#pragma unroll 1
        for (int k0 = 0; k0 < nmax; k0 += kBatch) {
            if (k0 > 0) load(k0);
#pragma unroll
            for (int q = 0; q < 2; ++q)
#pragma unroll
                for (int k = 0; k < kBatch; ++k) {
                    const int s = it_first[q] - s0 + k0 + k;
                    const float w = k0 + k < it_n[q] ? w_s[s * kHeads + it_ih[q]] : 0.f;
                    if (w != 0.f) {
                        r[q].x = fmaf(w, v[q][k].x, r[q].x);
                        r[q].y = fmaf(w, v[q][k].y, r[q].y);
                        r[q].z = fmaf(w, v[q][k].z, r[q].z);
                        r[q].w = fmaf(w, v[q][k].w, r[q].w);
                    }
                }
        }
#pragma unroll
        for (int q = 0; q < 2; ++q)
            if (it_dst[q] != nullptr) *reinterpret_cast<float4*>(it_dst[q]) = r[q];
    }
    if (latent) cp_async_wait_all();
    __syncthreads();

    // out rows: thread (row il = tid / 8, column block jq = tid % 8) sums z . U_V^(g)[i0 + il,
    // 32 columns of each 256-column chunk] for the chunk's heads; the 8 blocks of a row are
    // then added across lanes
    const int il = tid >> 3, jq = tid & 7;
    float part[kHeads] = {0.f, 0.f, 0.f, 0.f};
    if (latent) {
#pragma unroll 1
        for (int ch = 0; ch < zchunks; ++ch) {
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int col = ch * 256 + jq * 32 + c * 8;
                if (col < r_v) {
                    const uint4 u = col < ucols
                                        ? *reinterpret_cast<const uint4*>(u_s + il * ustride + col * 2)
                                        : *reinterpret_cast<const uint4*>(ug + (size_t)il * r_v + col);
                    const float uf[8] = {bf16lo(u.x), bf16hi(u.x), bf16lo(u.y), bf16hi(u.y),
                                         bf16lo(u.z), bf16hi(u.z), bf16lo(u.w), bf16hi(u.w)};
#pragma unroll
                    for (int k = 0; k < kHeads; ++k) {
                        const float* zp = z_s + ((ch * kHeads + k) * 8 + jq) * 36 + c * 8;
                        const float4 za = *reinterpret_cast<const float4*>(zp);
                        const float4 zb = *reinterpret_cast<const float4*>(zp + 4);
                        part[k] = fmaf(za.x, uf[0], fmaf(za.y, uf[1], fmaf(za.z, uf[2], fmaf(za.w, uf[3], part[k]))));
                        part[k] = fmaf(zb.x, uf[4], fmaf(zb.y, uf[5], fmaf(zb.z, uf[6], fmaf(zb.w, uf[7], part[k]))));
                    }
                }
            }
        }
#pragma unroll
        for (int k = 0; k < kHeads; ++k)
#pragma unroll
            for (int o = 1; o < 8; o <<= 1) part[k] += __shfl_xor_sync(0xffffffffu, part[k], o);
    }
    // lane jq < 4 writes head jq of row il
    if (jq < nh) {
        const float pv = jq == 0 ? part[0] : jq == 1 ? part[1] : jq == 2 ? part[2] : part[3];
        a.out[((size_t)b * a.Hq + h0 + jq) * d + i0 + il] = (pv + y_s[jq * kRows + il]) / L_s[jq];
    }
}

}  // namespace

cudaError_t launch_tc_combine(const CombineArgs& a, cudaStream_t st) {
    int ns_max = 0;
    for (int b = 0; b < a.B; ++b) ns_max = std::max(ns_max, a.slot_begin[b + 1] - a.slot_begin[b]);
    if (ns_max > kMaxSlotsPerB || a.d % kRows != 0 || a.d > 128) return cudaErrorInvalidValue;
    CombineArgs c = a;
    c.ns_max = (ns_max + 3) & ~3;
    const int r_v = a.U_V != nullptr ? a.r_v : 0;
    auto bytes = [&](int rv, int nsp) {
        const size_t ub = rv > 0 ? (size_t)kRows * (std::min(rv, kUCols) * 2 + 16) : 0;
        return ub + (size_t)nsp * 2 * kHeads * sizeof(float) +
               ((size_t)(rv + 255) / 256 * kHeads * 8 * 36 + kHeads * kRows) * sizeof(float);
    };
    const size_t smem = bytes(r_v, c.ns_max);
    static std::atomic<unsigned long long> attr_done{0};
    const cudaError_t e =
        set_max_smem_once((const void*)tc_combine_kernel, (int)bytes(kMaxRank, kMaxSlotsPerB), attr_done);
    if (e != cudaSuccess) return e;
    const int G = a.Hq / a.Hkv, nhc = (G + kHeads - 1) / kHeads;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.Hkv * nhc, a.B, a.d / kRows);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, tc_combine_kernel, c);
}

}  // namespace slimkv

// C-ABI layer of libslimkv: argument checks, workspace partition, the host-side
// work planner, and kernel dispatch (tensor-core path or SIMT path).
#include <math.h>
#include <string.h>

#include <algorithm>

#include "slimkv_internal.cuh"
#include "tc_decode.cuh"

using namespace slimkv;

// CTAs of the tensor-core kernels that gave up on a bounded wait (one counter per
// device: every device that loads the library has its own copy of this variable).
__device__ unsigned long long g_slimkv_aborts;

namespace slimkv {
DecodeTimer& decode_timer() {
    static thread_local DecodeTimer t;
    return t;
}

// Looked up on every call (not cached): after a device reset the module is loaded
// again and the variable may live at another address.
unsigned long long* abort_counter() {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_slimkv_aborts) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    return static_cast<unsigned long long*>(p);
}

static thread_local int g_withhold_cta = -1;
int take_withheld_cta() {
    const int c = g_withhold_cta;
    g_withhold_cta = -1;
    return c;
}
}  // namespace slimkv

namespace {

int g_force_simt = 0;

constexpr size_t kAlign = 256;
size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

size_t elem_size(slimkv_dtype t) { return t == SLIMKV_F32 ? 4 : 2; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

slimkv_status check_shape(const slimkv_shape* s, int which) {
    if (s == nullptr) return SLIMKV_ERR_NULL;
    if (s->dtype != SLIMKV_F32 && s->dtype != SLIMKV_BF16) return SLIMKV_ERR_DTYPE;
    if (which < SLIMKV_LATENT || which > SLIMKV_PREFILL) return SLIMKV_ERR_SHAPE;
    if (s->B < 1 || s->B > kMaxB) return SLIMKV_ERR_SHAPE;
    if (s->Hq < 1 || s->Hq > kMaxHq || s->Hkv < 1 || s->Hq % s->Hkv != 0) return SLIMKV_ERR_SHAPE;
    if (s->d != 64 && s->d != 128) return SLIMKV_ERR_SHAPE;
    if (s->N_b < 0 || s->W < 0 || s->N_b > (1 << 24) || s->W > (1 << 24)) return SLIMKV_ERR_SHAPE;
    if ((int64_t)s->W * s->Hkv > (int64_t(1) << 28)) return SLIMKV_ERR_SHAPE;
    if ((int64_t)s->N_b * s->Hkv > (int64_t(1) << 28)) return SLIMKV_ERR_SHAPE;
    if (s->N_b + s->W < 1) return SLIMKV_ERR_SHAPE;
    if (s->N_b > 0) {
        if (s->r_k < 32 || s->r_k > kMaxRank || s->r_k % 32) return SLIMKV_ERR_SHAPE;
        if (s->r_v < 32 || s->r_v > kMaxRank || s->r_v % 32) return SLIMKV_ERR_SHAPE;
    }
    if (!isfinite(s->scale)) return SLIMKV_ERR_SHAPE;
    if (!(s->rope_base > 0.0) || !isfinite(s->rope_base)) return SLIMKV_ERR_SHAPE;
    if (which == SLIMKV_FULL_KV && (s->N_b != 0 || s->W < 1)) return SLIMKV_ERR_SHAPE;
    if (which == SLIMKV_RECONSTRUCT && s->N_b < 1) return SLIMKV_ERR_SHAPE;
    if (which == SLIMKV_PREFILL) {
        // the chunk (W tokens) is always present; the tensor-core prefill kernel covers
        // bf16, d = 128 and ranks that are multiples of 64 up to 256
        if (s->W < 1 || s->dtype != SLIMKV_BF16) return SLIMKV_ERR_SHAPE;
        // staged query rows per (batch element, KV group): T * G, indexed in int
        if ((int64_t)s->W * (s->Hq / s->Hkv) > (int64_t(1) << 26)) return SLIMKV_ERR_SHAPE;
        if (!prefill_supported(s->d, s->N_b, s->r_k, s->r_v)) return SLIMKV_ERR_SHAPE;
    }
    return SLIMKV_OK;
}

// Number of segments (runs of rows of one kind for one batch element): the latent
// beacons form one segment, raw rows one per KV head (the tensor-core path's split),
// so one partial slot per segment plus kSlotCap covers every plan.
int n_segments(const slimkv_shape* s, int which) {
    const int raw = s->W > 0 ? s->Hkv : 0;
    int per_b = 0;
    if (which == SLIMKV_LATENT) per_b = (s->N_b > 0) + raw;
    if (which == SLIMKV_RECONSTRUCT) per_b = s->Hkv + raw;   // materialised beacons are raw rows too
    if (which == SLIMKV_FULL_KV) per_b = raw;
    return per_b * s->B;
}

WsLayout layout(const slimkv_shape* s, int which) {
    WsLayout L;
    if (which == SLIMKV_PREFILL) {
        L.total = align_up(prefill_stage_bytes(s->B, s->W, s->Hq, s->Hkv));
        return L;
    }
    const bool lat = which == SLIMKV_LATENT && s->N_b > 0;
    L.Dmax = std::max(lat ? s->r_v : 0, s->d);
    L.slots = kSlotCap + n_segments(s, which);
    size_t off = 0;
    L.q_rot = off;
    off = align_up(off + sizeof(float) * s->B * s->Hq * s->d);
    L.q_lat = off;
    if (lat) off = align_up(off + sizeof(float) * s->B * s->Hq * s->r_k);
    const int NP = (s->Hq + 15) / 16 * 16;
    L.lat_img = off;
    if (lat) off = align_up(off + (size_t)s->B * lat_img_bytes(NP, s->r_k));
    L.raw_img = off;
    off = align_up(off + (size_t)s->B * s->Hkv * raw_img_bytes(128));   // 128 columns (d = 64 zero-padded)
    L.acc = off;
    off = align_up(off + sizeof(float) * (size_t)L.slots * s->Hq * L.Dmax);
    L.ml = off;
    off = align_up(off + sizeof(float) * (size_t)L.slots * 2 * s->Hq);
    L.kind = off;
    off = align_up(off + sizeof(int) * (size_t)L.slots);
    if (which == SLIMKV_RECONSTRUCT) {
        const size_t kv = (size_t)s->B * s->N_b * s->Hkv * s->d * elem_size(s->dtype);
        L.kb = off;
        off = align_up(off + kv);
        L.vb = off;
        off = align_up(off + kv);
    }
    L.total = off;
    return L;
}

int device_cc_major() {
    int dev = 0, major = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess) return 0;
    return major;
}

int select_path(const slimkv_shape* s, int which) {
    if (check_shape(s, which) != SLIMKV_OK) return -1;
    if (which == SLIMKV_PREFILL) return 1;   // tensor-core kernel only
    if (g_force_simt) return 0;
    if (s->dtype != SLIMKV_BF16) return 0;
    // d = 64 runs on the tensor cores with zero-padded raw tiles, except the
    // reconstruction baselines (their GEMM writes 128-column blocks per KV head)
    if (s->d != 128 && (s->d != 64 || which == SLIMKV_RECONSTRUCT)) return 0;
    if (!tc_supported(s->Hq, s->Hkv, s->d, which == SLIMKV_LATENT ? s->N_b : 0, s->r_k, s->r_v))
        return 0;
    return device_cc_major() == 10 ? 1 : 0;
}

struct Ptrs {
    const void* q;
    const void* C_K;
    const void* C_V;
    const void* K_raw;
    const void* V_raw;
    const void* U_K;
    const void* U_V;
    const int32_t* q_pos;
    float* out;
    void* ws;
    size_t ws_bytes;
    int beacon_ratio;   // reconstruction baseline with beacon-key RoPE (0: without); ALiBi beacon spacing
    const float* alibi_slopes = nullptr;   // host [Hq]: ALiBi slopes of slimkv_decode_attn_alibi (NULL: none)
};

slimkv_status check_ptrs(const slimkv_shape* s, int which, const Ptrs& p) {
    const bool beacons = s->N_b > 0 && which != SLIMKV_FULL_KV;
    if (!p.q || !p.q_pos || !p.out || !p.ws) return SLIMKV_ERR_NULL;
    if (beacons && (!p.C_K || !p.C_V || !p.U_K || !p.U_V)) return SLIMKV_ERR_NULL;
    if (s->W > 0 && (!p.K_raw || !p.V_raw)) return SLIMKV_ERR_NULL;
    if (!aligned16(p.q) || !aligned16(p.out)) return SLIMKV_ERR_ALIGN;
    if ((reinterpret_cast<uintptr_t>(p.q_pos) & 3u) != 0) return SLIMKV_ERR_ALIGN;
    if ((reinterpret_cast<uintptr_t>(p.ws) & (kAlign - 1)) != 0) return SLIMKV_ERR_ALIGN;
    if (beacons && (!aligned16(p.C_K) || !aligned16(p.C_V) || !aligned16(p.U_K) || !aligned16(p.U_V)))
        return SLIMKV_ERR_ALIGN;
    if (s->W > 0 && (!aligned16(p.K_raw) || !aligned16(p.V_raw))) return SLIMKV_ERR_ALIGN;
    if (p.ws_bytes < layout(s, which).total) return SLIMKV_ERR_WORKSPACE;
    return SLIMKV_OK;
}

inline int cdiv(int a, int b) { return (a + b - 1) / b; }

// SIMT path: qproj -> split decode (one CTA per item and head) -> combine.
template <typename T>
slimkv_status run_simt(const slimkv_shape* s, int which, const Ptrs& p, cudaStream_t st) {
    const WsLayout L = layout(s, which);
    char* ws = static_cast<char*>(p.ws);
    float* q_rot = reinterpret_cast<float*>(ws + L.q_rot);
    float* q_lat = reinterpret_cast<float*>(ws + L.q_lat);
    const bool lat = which == SLIMKV_LATENT && s->N_b > 0;
    cudaError_t e = launch_qproj<T>((const T*)p.q, lat ? (const T*)p.U_K : nullptr, p.q_pos, q_rot,
                                    lat ? q_lat : nullptr, s->B, s->Hq, s->Hkv, s->d, s->r_k,
                                    s->rope_base, s->scale * kLog2e, st, false);
    if (e != cudaSuccess) return SLIMKV_ERR_CUDA;

    SimtDecodeArgs a = {};
    a.B = s->B;
    a.Hq = s->Hq;
    a.Hkv = s->Hkv;
    a.d = s->d;
    a.N_b = lat ? s->N_b : 0;
    a.r_k = s->r_k;
    a.r_v = s->r_v;
    a.C_K = p.C_K;
    a.C_V = p.C_V;
    a.q_rot = q_rot;
    a.q_lat = q_lat;
    a.acc = reinterpret_cast<float*>(ws + L.acc);
    a.ml = reinterpret_cast<float*>(ws + L.ml);
    a.kind = reinterpret_cast<int*>(ws + L.kind);
    a.Dmax = L.Dmax;
    if (p.alibi_slopes != nullptr) {
        a.alibi = 1;
        a.ratio = p.beacon_ratio;
        a.q_pos = p.q_pos;
        for (int h = 0; h < s->Hq; ++h) a.slope_l2[h] = p.alibi_slopes[h] * kLog2e;
    }
    if (which == SLIMKV_RECONSTRUCT) {
        T* kb = reinterpret_cast<T*>(ws + L.kb);
        T* vb = reinterpret_cast<T*>(ws + L.vb);
        const int rows = s->B * s->N_b, n = s->Hkv * s->d;
        if (launch_simt_reconstruct<T>((const T*)p.C_K, (const T*)p.U_K, kb, rows, n, s->r_k, st) !=
            cudaSuccess)
            return SLIMKV_ERR_CUDA;
        if (p.beacon_ratio > 0 &&
            launch_beacon_rope<T>(kb, s->B, s->N_b, s->Hkv, s->d, p.beacon_ratio, s->rope_base, st) != cudaSuccess)
            return SLIMKV_ERR_CUDA;
        if (launch_simt_reconstruct<T>((const T*)p.C_V, (const T*)p.U_V, vb, rows, n, s->r_v, st) !=
            cudaSuccess)
            return SLIMKV_ERR_CUDA;
        a.K0 = kb;
        a.V0 = vb;
        a.W0 = s->N_b;
        a.K1 = p.K_raw;
        a.V1 = p.V_raw;
        a.W1 = s->W;
    } else {
        a.K0 = p.K_raw;
        a.V0 = p.V_raw;
        a.W0 = s->W;
        a.W1 = 0;
    }
    // rows per item: grow until the item count fits the slot capacity
    int rpi = 256;
    for (;;) {
        const int per_b = (a.N_b ? cdiv(a.N_b, rpi) : 0) + (a.W0 ? cdiv(a.W0, rpi) : 0) +
                          (a.W1 ? cdiv(a.W1, rpi) : 0);
        if ((int64_t)per_b * s->B <= L.slots) break;
        rpi *= 2;
    }
    a.rpi_L = a.rpi_R = rpi;
    a.nit_L = a.N_b ? cdiv(a.N_b, rpi) : 0;
    a.nit_R0 = a.W0 ? cdiv(a.W0, rpi) : 0;
    a.nit_R1 = a.W1 ? cdiv(a.W1, rpi) : 0;
    timer_before(st);
    const cudaError_t de = launch_simt_decode<T>(a, st);
    timer_after(st);
    if (de != cudaSuccess) return SLIMKV_ERR_CUDA;

    CombineArgs c;
    c.B = s->B;
    c.Hq = s->Hq;
    c.Hkv = s->Hkv;
    c.d = s->d;
    c.r_v = s->r_v;
    c.Dmax = L.Dmax;
    c.U_V = lat ? p.U_V : nullptr;
    c.acc = a.acc;
    c.ml = a.ml;
    c.kind = a.kind;
    c.out = p.out;
    const int per_b = a.nit_L + a.nit_R0 + a.nit_R1;
    for (int b = 0; b <= s->B; ++b) c.slot_begin[b] = b * per_b;
    if (launch_combine<T>(c, st, false) != cudaSuccess) return SLIMKV_ERR_CUDA;
    return SLIMKV_OK;
}

slimkv_status run(const slimkv_shape* s, int which, const Ptrs& p, void* stream) {
    slimkv_status st = check_shape(s, which);
    if (st != SLIMKV_OK) return st;
    st = check_ptrs(s, which, p);
    if (st != SLIMKV_OK) return st;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    if (select_path(s, which) == 1) {
        TcCall c;
        c.which = which;
        c.B = s->B;
        c.Hq = s->Hq;
        c.Hkv = s->Hkv;
        c.d = s->d;
        c.N_b = s->N_b;
        c.r_k = s->r_k;
        c.r_v = s->r_v;
        c.W = s->W;
        c.scale_log2 = s->scale * kLog2e;
        c.rope_base = s->rope_base;
        c.q = p.q;
        c.C_K = p.C_K;
        c.C_V = p.C_V;
        c.K_raw = p.K_raw;
        c.V_raw = p.V_raw;
        c.U_K = p.U_K;
        c.U_V = p.U_V;
        c.q_pos = p.q_pos;
        c.out = p.out;
        const WsLayout L = layout(s, which);
        char* ws = static_cast<char*>(p.ws);
        c.q_rot = reinterpret_cast<float*>(ws + L.q_rot);
        c.q_lat = reinterpret_cast<float*>(ws + L.q_lat);
        c.lat_img = reinterpret_cast<uint8_t*>(ws + L.lat_img);
        c.raw_img = reinterpret_cast<uint8_t*>(ws + L.raw_img);
        c.acc = reinterpret_cast<float*>(ws + L.acc);
        c.ml = reinterpret_cast<float*>(ws + L.ml);
        c.kind = reinterpret_cast<int*>(ws + L.kind);
        c.kb = ws + L.kb;
        c.vb = ws + L.vb;
        c.slots = L.slots;
        c.Dmax = L.Dmax;
        c.beacon_ratio = p.beacon_ratio;
        c.alibi_slopes = p.alibi_slopes;
        return tc_run(c, cs) == cudaSuccess ? SLIMKV_OK : SLIMKV_ERR_CUDA;
    }
    if (s->dtype == SLIMKV_F32) return run_simt<float>(s, which, p, cs);
    return run_simt<__nv_bfloat16>(s, which, p, cs);
}

}  // namespace

extern "C" {

size_t slimkv_workspace_bytes(const slimkv_shape* shape, int which) {
    if (check_shape(shape, which) != SLIMKV_OK) return 0;
    return layout(shape, which).total;
}

slimkv_status slimkv_decode_attn(const slimkv_shape* shape, const void* q, const void* C_K,
                                 const void* C_V, const void* K_raw, const void* V_raw,
                                 const void* U_K, const void* U_V, const int32_t* q_pos,
                                 float* out, void* workspace, size_t ws_bytes, void* stream) {
    Ptrs p{q, C_K, C_V, K_raw, V_raw, U_K, U_V, q_pos, out, workspace, ws_bytes, 0};
    return run(shape, SLIMKV_LATENT, p, stream);
}

slimkv_status slimkv_decode_attn_reconstruct(const slimkv_shape* shape, const void* q,
                                             const void* C_K, const void* C_V,
                                             const void* K_raw, const void* V_raw,
                                             const void* U_K, const void* U_V,
                                             const int32_t* q_pos, float* out,
                                             void* workspace, size_t ws_bytes, void* stream) {
    Ptrs p{q, C_K, C_V, K_raw, V_raw, U_K, U_V, q_pos, out, workspace, ws_bytes, 0};
    return run(shape, SLIMKV_RECONSTRUCT, p, stream);
}

slimkv_status slimkv_decode_attn_reconstruct_rope(const slimkv_shape* shape, const void* q,
                                                  const void* C_K, const void* C_V,
                                                  const void* K_raw, const void* V_raw,
                                                  const void* U_K, const void* U_V,
                                                  const int32_t* q_pos, int beacon_ratio, float* out,
                                                  void* workspace, size_t ws_bytes, void* stream) {
    if (beacon_ratio < 1) return SLIMKV_ERR_SHAPE;
    Ptrs p{q, C_K, C_V, K_raw, V_raw, U_K, U_V, q_pos, out, workspace, ws_bytes, beacon_ratio};
    return run(shape, SLIMKV_RECONSTRUCT, p, stream);
}

slimkv_status slimkv_decode_attn_alibi(const slimkv_shape* shape, const void* q, const void* C_K,
                                       const void* C_V, const void* K_raw, const void* V_raw,
                                       const void* U_K, const void* U_V, const int32_t* q_pos,
                                       const float* alibi_slopes, int beacon_ratio, float* out,
                                       void* workspace, size_t ws_bytes, void* stream) {
    if (alibi_slopes == nullptr) return SLIMKV_ERR_NULL;
    if (beacon_ratio < 1) return SLIMKV_ERR_SHAPE;
    if (shape != nullptr && shape->Hq >= 1 && shape->Hq <= kMaxHq)
        for (int h = 0; h < shape->Hq; ++h)
            if (!isfinite(alibi_slopes[h])) return SLIMKV_ERR_SHAPE;
    Ptrs p{q, C_K, C_V, K_raw, V_raw, U_K, U_V, q_pos, out, workspace, ws_bytes, beacon_ratio, alibi_slopes};
    return run(shape, SLIMKV_LATENT, p, stream);
}

slimkv_status slimkv_decode_attn_full_kv(const slimkv_shape* shape, const void* q, const void* K,
                                         const void* V, const int32_t* q_pos, float* out,
                                         void* workspace, size_t ws_bytes, void* stream) {
    Ptrs p{q, nullptr, nullptr, K, V, nullptr, nullptr, q_pos, out, workspace, ws_bytes, 0};
    return run(shape, SLIMKV_FULL_KV, p, stream);
}

slimkv_status slimkv_prefill_attn(const slimkv_shape* shape, const void* q, const void* C_K, const void* C_V,
                                  const void* K_chunk, const void* V_chunk, const void* U_K, const void* U_V,
                                  const int32_t* p0, float* out, void* workspace, size_t ws_bytes, void* stream) {
    slimkv_status st = check_shape(shape, SLIMKV_PREFILL);
    if (st != SLIMKV_OK) return st;
    Ptrs p{q, C_K, C_V, K_chunk, V_chunk, U_K, U_V, p0, out, workspace, ws_bytes, 0};
    st = check_ptrs(shape, SLIMKV_PREFILL, p);
    if (st != SLIMKV_OK) return st;
    PrefillCall c;
    c.B = shape->B;
    c.T = shape->W;
    c.Hq = shape->Hq;
    c.Hkv = shape->Hkv;
    c.N_b = shape->N_b;
    c.r_k = shape->r_k;
    c.r_v = shape->r_v;
    c.scale = shape->scale;
    c.rope_base = shape->rope_base;
    c.q = q;
    c.C_K = C_K;
    c.C_V = C_V;
    c.K_chunk = K_chunk;
    c.V_chunk = V_chunk;
    c.U_K = U_K;
    c.U_V = U_V;
    c.p0 = p0;
    c.out = out;
    c.stage = workspace;
    return launch_prefill(c, static_cast<cudaStream_t>(stream)) == cudaSuccess ? SLIMKV_OK : SLIMKV_ERR_CUDA;
}

const char* slimkv_status_str(slimkv_status status) {
    switch (status) {
        case SLIMKV_OK: return "ok";
        case SLIMKV_ERR_NULL: return "required pointer is NULL";
        case SLIMKV_ERR_SHAPE: return "invalid or unsupported shape";
        case SLIMKV_ERR_DTYPE: return "unknown dtype";
        case SLIMKV_ERR_ALIGN: return "pointer breaks the alignment rule";
        case SLIMKV_ERR_WORKSPACE: return "workspace too small";
        case SLIMKV_ERR_CUDA: return "CUDA launch or driver call failed";
        case SLIMKV_ERR_TOO_LARGE: return "shape needs more scratch than the no-allocation entry point holds";
    }
    return "unknown status";
}

slimkv_status slimkv_append_kv(const slimkv_shape* s, const void* k_new, const void* v_new, void* K_raw,
                               void* V_raw, const int32_t* pos, void* stream) {
    if (s == nullptr || k_new == nullptr || v_new == nullptr || K_raw == nullptr || V_raw == nullptr ||
        pos == nullptr)
        return SLIMKV_ERR_NULL;
    if (s->dtype != SLIMKV_F32 && s->dtype != SLIMKV_BF16) return SLIMKV_ERR_DTYPE;
    if (s->B < 1 || s->B > kMaxB || s->Hkv < 1 || s->Hkv > kMaxHq) return SLIMKV_ERR_SHAPE;
    if (s->d != 64 && s->d != 128) return SLIMKV_ERR_SHAPE;
    if (s->W < 1 || s->W > (1 << 24) || (int64_t)s->W * s->Hkv > (int64_t(1) << 28)) return SLIMKV_ERR_SHAPE;
    if (!(s->rope_base > 0.0) || !isfinite(s->rope_base)) return SLIMKV_ERR_SHAPE;
    if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(K_raw) || !aligned16(V_raw)) return SLIMKV_ERR_ALIGN;
    if ((reinterpret_cast<uintptr_t>(pos) & 3u) != 0) return SLIMKV_ERR_ALIGN;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (s->dtype == SLIMKV_F32)
        e = launch_append_kv<float>((const float*)k_new, (const float*)v_new, (float*)K_raw, (float*)V_raw, pos,
                                    s->B, s->Hkv, s->d, s->W, s->rope_base, st);
    else
        e = launch_append_kv<__nv_bfloat16>((const __nv_bfloat16*)k_new, (const __nv_bfloat16*)v_new,
                                            (__nv_bfloat16*)K_raw, (__nv_bfloat16*)V_raw, pos, s->B, s->Hkv,
                                            s->d, s->W, s->rope_base, st);
    return e == cudaSuccess ? SLIMKV_OK : SLIMKV_ERR_CUDA;
}

int slimkv_abi_version(void) { return SLIMKV_ABI_VERSION; }

int slimkv_kernel_path(const slimkv_shape* shape, int which) { return select_path(shape, which); }

void slimkv_time_next_decode(void* start_event, void* stop_event) {
    DecodeTimer& t = decode_timer();
    t.start = static_cast<cudaEvent_t>(start_event);
    t.stop = static_cast<cudaEvent_t>(stop_event);
    if (!t.start || !t.stop) t.start = t.stop = nullptr;
}

long long slimkv_abort_count(int reset) {
    unsigned long long* p = abort_counter();
    if (p == nullptr || cudaDeviceSynchronize() != cudaSuccess) return -1;
    unsigned long long n = 0;
    if (cudaMemcpy(&n, p, sizeof(n), cudaMemcpyDeviceToHost) != cudaSuccess) return -1;
    if (reset && cudaMemset(p, 0, sizeof(n)) != cudaSuccess) return -1;
    return (long long)n;
}

void slimkv_test_withhold_first_load(int cta) { g_withhold_cta = cta < 0 ? -1 : cta; }

int slimkv_force_simt(int on) {
    const int prev = g_force_simt;
    g_force_simt = on ? 1 : 0;
    return prev;
}

}  // extern "C"

// Raw-window append for multi-step decoding.
//
// "Can SlimKV compress KV cache jointly across tokens and features", section
// "Latent-space attention removes the rebuild step": RoPE applies to all queries
// and to the raw-window keys only, and the window keeps its keys after RoPE. In a
// generation loop each new key is therefore rotated once, at its own absolute
// position, as it enters the window. The window is used as a ring of W slots
// (token p in slot p mod W); attention does not depend on the order of the
// window's rows.
//
// One CTA per (batch element, KV head); thread i rotates the pair (i, i + d/2)
// (rotate-half) with the same fixed-point angle reduction as the query kernel,
// so a query and a key at equal positions are rotated by bit-identical angles.
#include <math.h>

#include "slimkv_internal.cuh"

namespace slimkv {

namespace {

struct AppendArgs {
    const void* k_new;      // [B, Hkv, d]
    const void* v_new;      // [B, Hkv, d]
    void* K;                // [B, W, Hkv, d] keys after RoPE
    void* V;                // [B, W, Hkv, d]
    const int32_t* pos;     // [B]
    int Hkv, d, W;
    unsigned long long turn[64];
};

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
template <typename T> __device__ __forceinline__ T from_f(float x);
template <> __device__ __forceinline__ float from_f<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

template <typename T>
__global__ void __launch_bounds__(64) append_kv_kernel(const __grid_constant__ AppendArgs a) {
    const int b = blockIdx.x, g = blockIdx.y, i = threadIdx.x, half = a.d >> 1;
    if (i >= half) return;
    const int p = a.pos[b];
    const int slot = ((p % a.W) + a.W) % a.W;
    const size_t src = ((size_t)b * a.Hkv + g) * a.d;
    const size_t dst = (((size_t)b * a.W + slot) * a.Hkv + g) * a.d;
    const T* kn = static_cast<const T*>(a.k_new);
    const T* vn = static_cast<const T*>(a.v_new);
    T* K = static_cast<T*>(a.K);
    T* V = static_cast<T*>(a.V);
    const float x1 = to_f(kn[src + i]), x2 = to_f(kn[src + half + i]);
    // p * theta_i reduced to a signed fraction of a turn (exact 64-bit wrap-around)
    const long long frac = (long long)((unsigned long long)(long long)p * a.turn[i]);
    float sn, cs;
    sincospif((float)frac * 1.0842021724855044e-19f, &sn, &cs);   // x 2^-63: half-turns
    K[dst + i] = from_f<T>(x1 * cs - x2 * sn);
    K[dst + half + i] = from_f<T>(x2 * cs + x1 * sn);
    V[dst + i] = vn[src + i];
    V[dst + half + i] = vn[src + half + i];
}

// Beacon-key RoPE of the reconstruction baseline that keeps it: row R = b * N_b + j of
// K_b [B * N_b, Hkv * d] is rotated in place at position j * ratio + ratio - 1 (the last
// token of the block beacon j condenses). One CTA per (row, KV head); thread i rotates
// the pair (i, i + d/2) with the same fixed-point angle reduction as the query kernel.
struct BeaconRopeArgs {
    void* K;                // [B * N_b, Hkv, d]
    int N_b, Hkv, d, ratio;
    unsigned long long turn[64];
};

template <typename T>
__global__ void __launch_bounds__(64) beacon_rope_kernel(const __grid_constant__ BeaconRopeArgs a) {
    const int row = blockIdx.x, g = blockIdx.y, i = threadIdx.x, half = a.d >> 1;
    if (i >= half) return;
    const unsigned long long j = (unsigned long long)(row % a.N_b);
    const unsigned long long p = j * (unsigned long long)a.ratio + (unsigned long long)(a.ratio - 1);
    T* K = static_cast<T*>(a.K) + ((size_t)row * a.Hkv + g) * a.d;
    const float x1 = to_f(K[i]), x2 = to_f(K[half + i]);
    const long long frac = (long long)(p * a.turn[i]);
    float sn, cs;
    sincospif((float)frac * 1.0842021724855044e-19f, &sn, &cs);   // x 2^-63: half-turns
    K[i] = from_f<T>(x1 * cs - x2 * sn);
    K[half + i] = from_f<T>(x2 * cs + x1 * sn);
}

}  // namespace

template <typename T>
cudaError_t launch_beacon_rope(T* K_b, int B, int N_b, int Hkv, int d, int ratio, double base, cudaStream_t st) {
    BeaconRopeArgs a;
    a.K = K_b;
    a.N_b = N_b;
    a.Hkv = Hkv;
    a.d = d;
    a.ratio = ratio;
    rope_turns(base, d, a.turn);
    beacon_rope_kernel<T><<<dim3(B * N_b, Hkv), dim3(64), 0, st>>>(a);
    return cudaGetLastError();
}

template cudaError_t launch_beacon_rope<float>(float*, int, int, int, int, int, double, cudaStream_t);
template cudaError_t launch_beacon_rope<__nv_bfloat16>(__nv_bfloat16*, int, int, int, int, int, double, cudaStream_t);

template <typename T>
cudaError_t launch_append_kv(const T* k_new, const T* v_new, T* K, T* V, const int32_t* pos, int B, int Hkv,
                             int d, int W, double base, cudaStream_t st) {
    AppendArgs a;
    a.k_new = k_new;
    a.v_new = v_new;
    a.K = K;
    a.V = V;
    a.pos = pos;
    a.Hkv = Hkv;
    a.d = d;
    a.W = W;
    rope_turns(base, d, a.turn);
    append_kv_kernel<T><<<dim3(B, Hkv), dim3(64), 0, st>>>(a);
    return cudaGetLastError();
}

template cudaError_t launch_append_kv<float>(const float*, const float*, float*, float*, const int32_t*, int, int,
                                             int, int, double, cudaStream_t);
template cudaError_t launch_append_kv<__nv_bfloat16>(const __nv_bfloat16*, const __nv_bfloat16*, __nv_bfloat16*,
                                                     __nv_bfloat16*, const int32_t*, int, int, int, int, double,
                                                     cudaStream_t);

}  // namespace slimkv

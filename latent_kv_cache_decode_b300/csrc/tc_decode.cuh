// Tensor-core (tcgen05 + TMA) path of libslimkv: entry points used by the C-ABI layer.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace slimkv {

// Everything one call of the tensor-core path needs (pointers are device memory).
struct TcCall {
    int which;                 // SLIMKV_LATENT / SLIMKV_RECONSTRUCT / SLIMKV_FULL_KV
    int B, Hq, Hkv, d, N_b, r_k, r_v, W;
    float scale_log2;
    double rope_base;
    const void* q;
    const void* C_K;
    const void* C_V;
    const void* K_raw;
    const void* V_raw;
    const void* U_K;
    const void* U_V;
    const int32_t* q_pos;
    float* out;
    float* q_rot;
    float* q_lat;
    uint8_t* lat_img;          // query images written by the query kernel
    uint8_t* raw_img;
    float* acc;
    float* ml;
    int* kind;
    void* kb;
    void* vb;
    int slots;
    int Dmax;
    int beacon_ratio;          // SLIMKV_RECONSTRUCT: > 0 rotates the beacon keys (RoPE at j*ratio + ratio - 1)
    const float* alibi_slopes; // SLIMKV_LATENT: host array [Hq] of ALiBi slopes (NULL: no bias)
};

// Whether the tensor-core path handles these sizes (bf16 storage assumed).
bool tc_supported(int Hq, int Hkv, int d, int N_b, int r_k, int r_v);

// Enqueue the whole call on `st`.
cudaError_t tc_run(const TcCall& c, cudaStream_t st);

}  // namespace slimkv

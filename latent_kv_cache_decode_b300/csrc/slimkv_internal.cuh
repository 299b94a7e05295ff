// Internal declarations shared by the kernels and the C-ABI layer of libslimkv.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <stdint.h>

#include "../../include/slimkv.h"

namespace slimkv {

constexpr int kMaxB = 256;      // batch elements per call
constexpr int kMaxHq = 128;     // query heads
constexpr int kMaxCtas = 296;   // CTAs of one tensor-core decode launch (2 per SM on 148 SMs)
constexpr int kSlotCap = 512;   // partial slots beyond one per segment
constexpr int kMaxRank = 512;
constexpr int kMaxSlotsPerB = 1024;   // partial slots of one batch element (combine limit)

// Scores are kept in the log2 domain: s2 = scale * log2(e) * (q . k).
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
template <typename T> __device__ __forceinline__ T from_f(float v);
template <> __device__ __forceinline__ float from_f<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float v) {
    return __float2bfloat16_rn(v);
}

// Programmatic dependent launch: wait for the preceding grid (and everything it
// waited on) to finish and flush, and allow the next grid to be scheduled.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;"); }

// Workspace partition (byte offsets from the workspace base, 256-byte aligned).
struct WsLayout {
    size_t q_rot = 0;    // float [B, Hq, d]          rotated queries
    size_t q_lat = 0;    // float [B, Hq, r_k]        latent queries q . U_K^(g)
    size_t acc = 0;      // float [slots, Hq, Dmax]   per-split value accumulators
    size_t ml = 0;       // float [slots, 2, Hq]      per-split running max (log2) and sum
    size_t kind = 0;     // int   [slots]             what a partial covers (SlotKind)
    size_t lat_img = 0;  // bf16  [B][NP x r_k]       latent query image (tensor-core path)
    size_t raw_img = 0;  // bf16  [B][Hkv][32 x d]    raw query images (tensor-core path)
    size_t kb = 0;       // T     [B, N_b, Hkv, d]    materialised beacon keys (reconstruct)
    size_t vb = 0;       // T     [B, N_b, Hkv, d]    materialised beacon values (reconstruct)
    size_t total = 0;
    int slots = 0;       // capacity in slots
    int Dmax = 0;        // accumulator width
};

// One "segment" is a run of key rows of one kind for one batch element. Rows of
// a latent segment are beacons; rows of a raw segment are (token, KV head) pairs
// flattened as token * Hkv + g, so one row is one d-vector of the cache.
enum SegKind { kSegLatent = 0, kSegRaw0 = 1, kSegRaw1 = 2 };

// What one partial slot holds: a latent accumulator (r_v wide) for every head, a
// raw accumulator (d wide) for every head, or a raw accumulator for the heads of
// one KV group g only (kSlotRawGroup + g; the other heads' rows are not written).
enum SlotKind { kSlotLatent = 0, kSlotRawAll = 1, kSlotRawGroup = 2 };
// Arguments of the SIMT split-decode kernel.
struct SimtDecodeArgs {
    int B, Hq, Hkv, d, N_b, r_k, r_v;
    int W0, W1;                 // tokens of raw sources 0 and 1 (0 = absent)
    const void* C_K;
    const void* C_V;
    const void* K0;
    const void* V0;
    const void* K1;
    const void* V1;
    const float* q_rot;
    const float* q_lat;
    float* acc;
    float* ml;
    int* kind;
    int Dmax;
    int rpi_L, rpi_R;            // rows (beacons / tokens) per item
    int nit_L, nit_R0, nit_R1;   // items per batch element
    // ALiBi (alibi != 0): head h adds slope_l2[h] * (key position - q_pos[b]) to its scores
    // (log2 units); beacon j sits at j * ratio + ratio - 1, window slot s (source 0) at the
    // latest position = s mod W0 not above q_pos[b]
    int alibi, ratio;
    const int32_t* q_pos;
    float slope_l2[kMaxHq];
};

// Arguments of the split-combine kernel (merges partials, applies U_V^(g)T).
struct CombineArgs {
    int B, Hq, Hkv, d, r_v, Dmax;
    int ns_max;                  // most partial slots of one batch element (set by the launcher)
    const void* U_V;             // NULL when no latent partials exist
    const float* acc;
    const float* ml;
    const int* kind;
    float* out;
    int slot_begin[kMaxB + 1];   // partial slots of batch element b: [slot_begin[b], slot_begin[b+1])
    int slot_mid[kMaxB];         // tensor-core path: b's latent slots [slot_begin, slot_mid), raw after
};

// Arguments of the query kernel (RoPE + latent projection). The RoPE angle of pair
// i at integer position p is p * theta_i; turn[i] holds theta_i / (2 pi) as a
// 64-bit fixed-point fraction of a turn, so p * turn[i] (mod 2^64) is the angle's
// fraction of a full turn, exact up to the rounding of turn[i].
struct QprojArgs {
    const void* q;
    const void* U_K;             // NULL: rotate only
    const int32_t* q_pos;
    float* q_rot;                // [B, Hq, d]   RoPE(q) * scale_log2 (NULL: not written)
    float* q_lat;                // [B, Hq, r_k] RoPE(q) . U_K^(g) * scale_log2 (NULL: not written)
    // Query operands of the tensor-core decode kernel, as bf16 high / low parts laid
    // out exactly as that kernel's shared-memory operand (128-byte swizzled rows of
    // 64 columns, for a 1024-byte aligned destination), so it can copy them in bulk:
    uint8_t* lat_img;            // per b: NP rows, bf16 of q_lat[b] (heads past Hq unused)
    uint8_t* raw_img;            // per (b, g): rows [0, 16) high, [16, 32) low parts of q_rot of group g
    int NP;                      // heads of the latent image, rounded up to 16
    int B, Hq, Hkv, d, r_k;
    int nbb, hcn;                // batch elements and 32-head chunks per CTA row block
    float scale_log2;            // score scale * log2(e), folded into both outputs
    unsigned long long turn[64];
};

// Raise a kernel's dynamic shared-memory limit to `bytes` (0: leave it) on the current
// device, once per device (`done` is the caller's bit mask of devices already set).
inline cudaError_t set_max_smem_once(const void* func, int bytes, std::atomic<unsigned long long>& done) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = 1ull << (dev & 63);
    if (done.load() & bit) return cudaSuccess;
    if (bytes > 0) e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    // every kernel of a call prefers the largest shared-memory carveout, so an SM
    // need not change its L1 / shared split between the call's kernels
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(func, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
    if (e == cudaSuccess) done.fetch_or(bit);
    return e;
}

// theta_i / (2 pi) for i < d / 2 as a 64-bit fixed-point fraction of a turn
// (theta_i = base^(-2i/d)); entries past d / 2 are zero.
void rope_turns(double base, int d, unsigned long long (&turn)[64]);

// Append the current token to the raw window ring (slot pos[b] mod W), key rotated at pos[b].
template <typename T>
cudaError_t launch_append_kv(const T* k_new, const T* v_new, T* K, T* V, const int32_t* pos, int B, int Hkv,
                             int d, int W, double base, cudaStream_t st);

// Prefill over the beacon memory and a causal chunk (tensor-core path).
struct PrefillCall {
    int B, T, Hq, Hkv, N_b, r_k, r_v;
    float scale;
    double rope_base;
    const void* q;         // [B, T, Hq, d] bf16
    const void* C_K;       // [B, N_b, r_k]
    const void* C_V;       // [B, N_b, r_v]
    const void* K_chunk;   // [B, T, Hkv, d] (stored after RoPE)
    const void* V_chunk;
    const void* U_K;       // [Hkv d, r_k]
    const void* U_V;
    const int32_t* p0;     // [B] position of chunk token 0
    float* out;            // [B, T, Hq, d]
    void* stage;           // prefill_stage_bytes of scratch
};
bool prefill_supported(int d, int N_b, int r_k, int r_v);
size_t prefill_stage_bytes(int B, int T, int Hq, int Hkv);
cudaError_t launch_prefill(const PrefillCall& c, cudaStream_t st);

// Device address of the current device's abort counter (CTAs of the tensor-core
// kernels that gave up on a bounded wait), or NULL if it cannot be had.
unsigned long long* abort_counter();
// The CTA that the next tensor-core decode launch of this host thread withholds its
// first key load from (slimkv_test_withhold_first_load), then -1 again.
int take_withheld_cta();

// Events requested by slimkv_time_next_decode for the next call of this thread.
struct DecodeTimer {
    cudaEvent_t start = nullptr, stop = nullptr;
};
DecodeTimer& decode_timer();
// Record the pending start event on `st` (before the decode launch).
// (recorded as external events, so that under stream capture they become event-record
// nodes of the graph that can be timed, rather than capture-internal dependencies)
inline void timer_before(cudaStream_t st) {
    if (decode_timer().start) cudaEventRecordWithFlags(decode_timer().start, st, cudaEventRecordExternal);
}
// Record the pending stop event on `st` (after the decode launch) and clear the request.
inline void timer_after(cudaStream_t st) {
    DecodeTimer& t = decode_timer();
    if (t.stop) cudaEventRecordWithFlags(t.stop, st, cudaEventRecordExternal);
    t.start = t.stop = nullptr;
}

// ---- kernels (simt_kernels.cu) ----
// Query RoPE and latent projection; outputs carry the factor scale*log2(e) so the
// decode kernels read scores directly in the log2 domain.
template <typename T>
cudaError_t launch_qproj(const T* q, const T* U_K, const int32_t* q_pos, float* q_rot,
                         float* q_lat, int B, int Hq, int Hkv, int d, int r_k, double base,
                         float scale_log2, cudaStream_t st, bool pdl, uint8_t* lat_img = nullptr,
                         uint8_t* raw_img = nullptr, int NP = 0);

// Bytes of the query images (latent: per batch element; raw: per (batch element, KV group)).
__host__ __device__ inline size_t lat_img_bytes(int NP, int r_k) { return (size_t)NP * ((r_k + 63) / 64 * 64) * 2; }
__host__ __device__ inline size_t raw_img_bytes(int d) { return (size_t)2 * 16 * d * 2; }
template <typename T>
cudaError_t launch_simt_decode(const SimtDecodeArgs& a, cudaStream_t st);
template <typename T>
cudaError_t launch_combine(const CombineArgs& a, cudaStream_t st, bool pdl);
// The tensor-core path's combine (bf16 U_V, d = 128; tc_combine.cu), launched with
// programmatic dependent launch.
cudaError_t launch_tc_combine(const CombineArgs& a, cudaStream_t st);
template <typename T>
cudaError_t launch_simt_reconstruct(const T* C, const T* U, T* out, int rows, int n, int r,
                                    cudaStream_t st);

// Materialise out[rows, n] = C[rows, r] . U[n, r]^T in bf16 on the tensor cores (reconstruction
// baseline, tc_gemm.cu; n a multiple of 128, r a multiple of 16 up to 512). With beacon_ratio > 0
// every 128-column block of a row (one KV head, d = 128) is also rotated (rotate-half RoPE) at
// position j * beacon_ratio + beacon_ratio - 1, j = row % rows_per_b (the beacon index).
cudaError_t launch_reconstruct_gemm(const __nv_bfloat16* C, const __nv_bfloat16* U, __nv_bfloat16* out,
                                    int rows, int n, int r, cudaStream_t st, int beacon_ratio = 0,
                                    int rows_per_b = 0, double rope_base = 10000.0);
// Rotate the rows of materialised beacon keys K_b [B * N_b, Hkv, d] in place at their beacon
// positions j * ratio + ratio - 1 (append_kv.cu; the SIMT path of the same baseline).
template <typename T>
cudaError_t launch_beacon_rope(T* K_b, int B, int N_b, int Hkv, int d, int ratio, double base, cudaStream_t st);

}  // namespace slimkv

// slimkv_decode_attn_noalloc: the SlimKV decode call for callers that cannot
// allocate device memory.
//
// Some host programs cannot hand this library a workspace: an inference engine
// that reserves nearly all of HBM in its own pool up front and forbids any other
// allocation, a plain C caller that links no device allocator, or a
// latency-critical decode loop where a cudaMalloc (which may synchronise the
// device and can fail once memory is fragmented) is not allowed. For them the
// scratch memory lives in one file-scope device array of fixed size, reserved
// when the library's device code is loaded and kept until the process exits.
#include <mutex>

#include "slimkv_internal.cuh"

namespace {

// Largest workspace the no-allocation entry point can serve, per device.
constexpr size_t kNoAllocScratchBytes = SLIMKV_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

// The scratch array. In host code `g_noalloc_scratch` names a host-side stand-in,
// not device memory: only the address returned by cudaGetSymbolAddress (taken
// with the target device current) may be handed to kernels.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up once per
// device. Returns nullptr if the lookup fails.
void* scratch_on_current_device() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_scratch_ptr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return nullptr;
        g_scratch_ptr[dev] = p;
    }
    return g_scratch_ptr[dev];
}

}  // namespace

extern "C" {

slimkv_status slimkv_decode_attn_noalloc(const slimkv_shape* shape, const void* q, const void* C_K,
                                         const void* C_V, const void* K_raw, const void* V_raw,
                                         const void* U_K, const void* U_V, const int32_t* q_pos,
                                         float* out, void* stream) {
    if (shape == nullptr) return SLIMKV_ERR_NULL;
    const size_t need = slimkv_workspace_bytes(shape, SLIMKV_LATENT);
    if (need == 0) {
        // invalid shape: let the regular entry point report which check failed
        // (it validates everything before touching the device)
        return slimkv_decode_attn(shape, q, C_K, C_V, K_raw, V_raw, U_K, U_V, q_pos, out,
                                  nullptr, 0, stream);
    }
    if (need > kNoAllocScratchBytes) return SLIMKV_ERR_TOO_LARGE;
    void* scratch = scratch_on_current_device();
    if (scratch == nullptr) return SLIMKV_ERR_CUDA;
    // Nothing in the workspace needs to start at zero: every call writes each
    // scratch word (rotated and latent queries, per-split partials) before it
    // reads it, so the previous call's leftovers are harmless.
    return slimkv_decode_attn(shape, q, C_K, C_V, K_raw, V_raw, U_K, U_V, q_pos, out, scratch,
                              kNoAllocScratchBytes, stream);
}

}  // extern "C"

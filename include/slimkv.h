/*
 * slimkv.h - C ABI of libslimkv: SlimKV reconstruction-free decode attention
 * for one transformer layer and one decode step (and its prefill-side and
 * comparison variants), on an NVIDIA B300 (sm_103a).
 *
 * The method. "Can SlimKV compress KV cache jointly across tokens and features"
 * (wispaper.ai), section "Latent-space attention removes the rebuild step": the
 * history of a sequence is folded into beacon states whose keys and values are
 * cached only as low-rank latent rows C_K, C_V, with no key-side RoPE; recent
 * raw tokens keep full-dimension keys with RoPE. RoPE is applied to every query.
 * A query head h of KV group g is scored against the beacons in latent space,
 * (RoPE(q_h) . U_K^(g)) . C_K^T, and against the raw window as
 * RoPE(q_h) . K_raw[:, g]^T; one softmax spans both score sets, and the values
 * are aggregated as (A_beacon . C_V) . U_V^(g)T + A_window . V_raw[:, g]. Beacon
 * keys are never materialised at full dimension. The SlimKV abstract
 * (omanscience.com citation record) states the same K-RoPE-free latent decode.
 *
 * Conventions used by every call:
 *  - Query head h belongs to KV group g = h / (Hq / Hkv) (contiguous groups).
 *  - U_K, U_V are row-major [Hkv*d, r]; U^(g) is the row block g*d .. g*d+d-1,
 *    the part of the up-projection that yields KV head g.
 *  - RoPE pairs element i with element i + d/2 ("rotate-half") at angle
 *    q_pos[b] * rope_base^(-2i/d); the angle is formed in double precision.
 *  - Raw-window keys (and full-KV keys) are stored after RoPE.
 *  - The same scale multiplies beacon and window scores (typically 1/sqrt(d)).
 *  - No masking: the decode query attends to every beacon and window row.
 *
 * Memory and ordering:
 *  - Every pointer is device memory owned by the caller; the library allocates
 *    and frees nothing. Each call only enqueues kernels on `stream` (a
 *    cudaStream_t passed as void*; NULL is the legacy default stream) and
 *    returns; buffers must stay valid until the stream has passed the call.
 *  - Every tensor pointer must be 16-byte aligned, and the workspace 256-byte
 *    aligned.
 *  - Kernels of a call may be launched before the previous call on the same
 *    stream has finished (programmatic dependent launch); each kernel waits for
 *    its predecessor before it reads the workspace or writes anything, but may
 *    read its cache operands (C_K, C_V, K_raw, V_raw, K, V, U_K, U_V) early.
 *    So the cache operands of a call must not alias the `out` or `workspace`
 *    of the slimkv call issued just before it on the same stream.
 *  - One workspace may be reused by consecutive calls on one stream; calls on
 *    different streams that may overlap need separate workspaces.
 *
 * Errors: every argument is checked on the host before any launch; a failed
 * check returns a status and launches nothing. SLIMKV_ERR_CUDA means a launch
 * or a driver call failed (the CUDA error is left for cudaGetLastError).
 */
#ifndef SLIMKV_H
#define SLIMKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* 2: adds slimkv_append_kv; 3: adds slimkv_decode_attn_reconstruct_rope and
 * slimkv_decode_attn_alibi; 4: adds slimkv_prefill_attn (SLIMKV_PREFILL),
 * slimkv_abort_count and slimkv_test_withhold_first_load. Earlier calls are
 * unchanged. */
#define SLIMKV_ABI_VERSION 4

typedef enum {
    SLIMKV_OK = 0,
    SLIMKV_ERR_NULL = 1,      /* a required pointer is NULL                       */
    SLIMKV_ERR_SHAPE = 2,     /* a size is out of range or inconsistent           */
    SLIMKV_ERR_DTYPE = 3,     /* unknown storage dtype                            */
    SLIMKV_ERR_ALIGN = 4,     /* a pointer breaks the alignment rule              */
    SLIMKV_ERR_WORKSPACE = 5, /* workspace missing or smaller than required       */
    SLIMKV_ERR_CUDA = 6,      /* a CUDA launch or driver call failed              */
    SLIMKV_ERR_TOO_LARGE = 7  /* the shape needs more scratch than the fixed array
                                 of slimkv_decode_attn_noalloc holds              */
} slimkv_status;

/* Storage type of q, C_K, C_V, K_raw, V_raw, K, V, U_K and U_V. Arithmetic is
 * float32 (tensor-core products take bf16 operands with float32 accumulation;
 * the query operand is split into a bf16 high and low part). `out` is float32. */
typedef enum { SLIMKV_F32 = 0, SLIMKV_BF16 = 1 } slimkv_dtype;

/* Problem sizes of one layer.
 *  B      batch elements (1..256)            Hq, Hkv  query / KV heads, Hq % Hkv == 0, Hq <= 128
 *  d      head dimension (64 or 128)          N_b      beacon states per batch element (>= 0)
 *  r_k    latent key rank, r_v latent value rank: multiples of 32 in [32, 512] when N_b > 0
 *  W      raw-window tokens per element (>= 0); N_b + W >= 1
 *  scale  score scale (finite)                rope_base RoPE base (> 0)
 *  N_b <= 2^24 and W <= 2^24. For slimkv_decode_attn_full_kv, N_b must be 0 and W is the
 *  cache length T. */
typedef struct {
    int B, Hq, Hkv, d, N_b, r_k, r_v, W;
    float scale;
    double rope_base;
    slimkv_dtype dtype;
} slimkv_shape;

/* which: SLIMKV_LATENT for slimkv_decode_attn, SLIMKV_RECONSTRUCT for
 * slimkv_decode_attn_reconstruct, SLIMKV_FULL_KV for slimkv_decode_attn_full_kv,
 * SLIMKV_PREFILL for slimkv_prefill_attn. */
enum { SLIMKV_LATENT = 0, SLIMKV_RECONSTRUCT = 1, SLIMKV_FULL_KV = 2, SLIMKV_PREFILL = 3 };

/* Bytes of device workspace the call `which` needs for `shape` (0 if the shape
 * is invalid). The workspace holds the rotated and latent queries, per-split
 * softmax partials and, for SLIMKV_RECONSTRUCT, the materialised K_b and V_b. */
size_t slimkv_workspace_bytes(const slimkv_shape* shape, int which);

/* SlimKV decode attention, "Latent-space attention removes the rebuild step":
 * out[b,h,:] = ( (A_b . C_V[b]) . U_V^(g)T + A_w . V_raw[b,:,g,:] ) / l, where the
 * scores are scale*(RoPE(q[b,h]) . U_K^(g)) . C_K[b]^T over the beacons and
 * scale*RoPE(q[b,h]) . K_raw[b,:,g,:]^T over the window, A = exp(s - max s) over
 * both sets and l = sum(A).
 *   q      [B, Hq, d]        queries before RoPE, position q_pos[b]
 *   C_K    [B, N_b, r_k]     latent beacon keys (no RoPE)           (unused if N_b == 0)
 *   C_V    [B, N_b, r_v]     latent beacon values                   (unused if N_b == 0)
 *   K_raw  [B, W, Hkv, d]    raw-window keys, RoPE already applied  (unused if W == 0)
 *   V_raw  [B, W, Hkv, d]    raw-window values                      (unused if W == 0)
 *   U_K    [Hkv*d, r_k]      key up-projection                      (unused if N_b == 0)
 *   U_V    [Hkv*d, r_v]      value up-projection                    (unused if N_b == 0)
 *   q_pos  [B] int32         query positions (device)
 *   out    [B, Hq, d] f32    result
 *   workspace, ws_bytes      device scratch, >= slimkv_workspace_bytes(shape, SLIMKV_LATENT)
 * Beacon keys and values are never expanded to full dimension. */
slimkv_status slimkv_decode_attn(const slimkv_shape* shape, const void* q, const void* C_K,
                                 const void* C_V, const void* K_raw, const void* V_raw,
                                 const void* U_K, const void* U_V, const int32_t* q_pos,
                                 float* out, void* workspace, size_t ws_bytes, void* stream);

/* The feature-wise baseline the SlimKV pages compare against ("Speedups are
 * real, but memory is set by the ratio": a reconstruction-based variant that
 * materialises full-dimensional K/V before attention): K_b = C_K . U_K^T and
 * V_b = C_V . U_V^T are written to the workspace as [B, N_b, Hkv, d] in the
 * storage dtype, then standard GQA attention runs over [K_b ; K_raw] with RoPE on
 * the query only (beacon keys get none, so the result equals slimkv_decode_attn
 * up to rounding). Same arguments as slimkv_decode_attn; workspace >=
 * slimkv_workspace_bytes(shape, SLIMKV_RECONSTRUCT). Requires N_b > 0. With bf16
 * storage and d = 128 the materialisation is the library's tensor-core GEMM (bf16 in,
 * float32 accumulate, bf16 out); otherwise a float32-accumulate SIMT GEMM. */
slimkv_status slimkv_decode_attn_reconstruct(const slimkv_shape* shape, const void* q,
                                             const void* C_K, const void* C_V,
                                             const void* K_raw, const void* V_raw,
                                             const void* U_K, const void* U_V,
                                             const int32_t* q_pos, float* out,
                                             void* workspace, size_t ws_bytes, void* stream);

/* slimkv_decode_attn with an ALiBi bias ("Latent-space attention removes the rebuild
 * step" and "Where SlimKV fits and where it does not": the bias is added after the QK
 * product, so the latent beacon scores take it unchanged). Every score of head h,
 * beacon or window, gains slopes[h] * (key position - q_pos[b]) before the softmax.
 * The pages give no key positions for beacons or the window; the positions taken are:
 *   beacon j      j * beacon_ratio + beacon_ratio - 1 (the last token of its block)
 *   window slot s q_pos[b] - ((q_pos[b] - s) mod W), the latest position congruent to s
 *                 modulo W that does not exceed q_pos[b] (the ring of slimkv_append_kv,
 *                 with the current token appended before the decode)
 *   alibi_slopes  host array of Hq finite slopes (natural-log units of the scores),
 *                 read during the call (NULL: SLIMKV_ERR_NULL)
 *   beacon_ratio  tokens per beacon (the compression ratio), >= 1
 * RoPE is applied as in slimkv_decode_attn. Other arguments, workspace size
 * (SLIMKV_LATENT) and requirements as slimkv_decode_attn. */
slimkv_status slimkv_decode_attn_alibi(const slimkv_shape* shape, const void* q, const void* C_K,
                                       const void* C_V, const void* K_raw, const void* V_raw,
                                       const void* U_K, const void* U_V, const int32_t* q_pos,
                                       const float* alibi_slopes, int beacon_ratio, float* out,
                                       void* workspace, size_t ws_bytes, void* stream);

/* The reconstruction baseline as the SlimKV pages run it ("Speedups are real, but
 * memory is set by the ratio": the baseline keeps beacon key RoPE). As
 * slimkv_decode_attn_reconstruct, except that every materialised beacon key of every
 * KV head is rotated (rotate-half RoPE, base shape->rope_base) at its beacon's
 * position before the attention. The pages do not say where a beacon sits; the
 * position taken is that of the last token of the block the beacon condenses,
 * j * beacon_ratio + beacon_ratio - 1 for beacon j. The result is therefore not
 * equal to slimkv_decode_attn (a rotated key has no latent form); the call exists to
 * time the pages' own baseline.
 *   beacon_ratio   tokens per beacon (the compression ratio), >= 1
 * Same other arguments, workspace size (SLIMKV_RECONSTRUCT) and requirements as
 * slimkv_decode_attn_reconstruct. With bf16 storage and d = 128 the rotation is part
 * of the tensor-core GEMM's write-out (float32, then rounded); otherwise a separate
 * pass rotates K_b in place. */
slimkv_status slimkv_decode_attn_reconstruct_rope(const slimkv_shape* shape, const void* q,
                                                  const void* C_K, const void* C_V,
                                                  const void* K_raw, const void* V_raw,
                                                  const void* U_K, const void* U_V,
                                                  const int32_t* q_pos, int beacon_ratio, float* out,
                                                  void* workspace, size_t ws_bytes, void* stream);

/* Uncompressed GQA decode attention ("Full KV" in the same section):
 * out[b,h,:] = softmax(scale * RoPE(q[b,h]) . K[b,:,g,:]^T) . V[b,:,g,:].
 *   K, V [B, T, Hkv, d] with T = shape->W (keys stored after RoPE); shape->N_b == 0.
 * workspace >= slimkv_workspace_bytes(shape, SLIMKV_FULL_KV). */
slimkv_status slimkv_decode_attn_full_kv(const slimkv_shape* shape, const void* q,
                                         const void* K, const void* V,
                                         const int32_t* q_pos, float* out,
                                         void* workspace, size_t ws_bytes, void* stream);

/* Prefill-side attention of one chunk of new tokens over the beacon memory and the
 * chunk itself ("Can SlimKV compress KV cache jointly across tokens and features",
 * section "Speedups are real, but memory is set by the ratio": time-to-first-token
 * gains come from skipping key-side RoPE and full-key materialisation for beacon
 * states). Query token t of the chunk sits at position p0[b] + t and sees every beacon
 * (latent scores, as in slimkv_decode_attn) and the chunk's tokens 0..t, in one softmax:
 *   s   = [scale*(RoPE(q[b,t,h]) . U_K^(g)) . C_K[b]^T ; scale*RoPE(q[b,t,h]) . K_chunk[b,0..t,g,:]^T]
 *   out[b,t,h,:] = ( (A_b . C_V[b]) . U_V^(g)T + A_c . V_chunk[b,0..t,g,:] ) / l
 *   q        [B, T, Hq, d]    chunk queries before RoPE, T = shape->W
 *   C_K, C_V [B, N_b, r_k / r_v] latent beacons (N_b may be 0)
 *   K_chunk  [B, T, Hkv, d]   the chunk's keys, stored after RoPE at p0[b] + s
 *   V_chunk  [B, T, Hkv, d]   the chunk's values
 *   U_K, U_V [Hkv*d, r_k / r_v]
 *   p0       [B] int32        position of chunk token 0 (device)
 *   out      [B, T, Hq, d] f32
 *   workspace >= slimkv_workspace_bytes(shape, SLIMKV_PREFILL) (the staged queries)
 * Runs on the tensor cores only: bf16 storage, d = 128 and, with beacons, r_k and r_v
 * multiples of 64 up to 256, and T * (Hq / Hkv) <= 2^26; other shapes return
 * SLIMKV_ERR_SHAPE. Same pointer rules
 * and errors as slimkv_decode_attn. */
slimkv_status slimkv_prefill_attn(const slimkv_shape* shape, const void* q, const void* C_K,
                                  const void* C_V, const void* K_chunk, const void* V_chunk,
                                  const void* U_K, const void* U_V, const int32_t* p0, float* out,
                                  void* workspace, size_t ws_bytes, void* stream);

/* Size of the fixed device scratch array behind slimkv_decode_attn_noalloc. */
#define SLIMKV_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)

/* slimkv_decode_attn for callers that cannot allocate device memory. The SlimKV
 * pages have no counterpart to this call; it exists for host programs that have no
 * way to hand the library a workspace: an inference engine that reserves nearly all
 * of HBM in its own pool and forbids other allocations, a plain C caller that links
 * no device allocator, or a latency-critical decode loop in which a cudaMalloc
 * (which may synchronise the device and can fail once memory is fragmented) is not
 * allowed.
 *
 * Arguments and result are those of slimkv_decode_attn without the workspace. The
 * scratch is one file-scope device array of SLIMKV_NOALLOC_SCRATCH_BYTES (64 MiB)
 * that every GPU which loads the library's device code holds until the process
 * exits; this call itself allocates and frees nothing.
 *  - A shape whose workspace (slimkv_workspace_bytes(shape, SLIMKV_LATENT)) exceeds
 *    SLIMKV_NOALLOC_SCRATCH_BYTES is rejected with SLIMKV_ERR_TOO_LARGE before any
 *    launch; other argument errors are reported as by slimkv_decode_attn.
 *  - The first call on a device looks up the array's device address on that device
 *    (cudaGetSymbolAddress, with that device current); make that first call before
 *    any stream capture. A failed lookup returns SLIMKV_ERR_CUDA. The address is kept
 *    for the life of the process: it does not survive cudaDeviceReset (or any other
 *    teardown of the device's primary context), after which this call must not be
 *    used again in the same process.
 *  - All calls on a device share the one array, and it keeps the previous call's
 *    contents; no call depends on them (each writes every scratch word before
 *    reading it). Calls that may overlap on the GPU (different streams, or
 *    different host threads without ordering) race on the array: serialise them,
 *    e.g. on one stream. */
slimkv_status slimkv_decode_attn_noalloc(const slimkv_shape* shape, const void* q,
                                         const void* C_K, const void* C_V,
                                         const void* K_raw, const void* V_raw,
                                         const void* U_K, const void* U_V,
                                         const int32_t* q_pos, float* out, void* stream);

/* Multi-step decode: append the current token to the raw window before the
 * layer's decode call. The decode rule keeps raw-window keys after RoPE ("RoPE ...
 * on raw keys only", section "Latent-space attention removes the rebuild step"),
 * so each new key is rotated once, here, at its own absolute position. The window
 * is a ring of W slots: the token at position pos[b] goes to slot pos[b] mod W,
 * replacing token pos[b] - W (the pages condense old raw tokens into beacons with
 * trained projections; that step is outside this library). Attention does not
 * depend on the order of window rows, so a later slimkv_decode_attn with
 * q_pos = pos sees the last W tokens including the new one.
 *   k_new, v_new  [B, Hkv, d]      the new token's key (before RoPE) and value
 *   K_raw, V_raw  [B, W, Hkv, d]   the window (keys after RoPE), updated in place
 *   pos           [B] int32        absolute positions, >= 0 (device)
 * Uses shape->B, Hkv, d, W (>= 1), rope_base and dtype; the other fields are
 * ignored. Pointers 16-byte aligned (pos 4-byte). Asynchronous on `stream`. */
slimkv_status slimkv_append_kv(const slimkv_shape* shape, const void* k_new, const void* v_new,
                               void* K_raw, void* V_raw, const int32_t* pos, void* stream);

/* Human-readable name of a status. Never NULL. */
const char* slimkv_status_str(slimkv_status status);

/* Failure detection. Every wait inside the tensor-core kernels is bounded (about 2 s);
 * a thread block whose wait runs out stops waiting, lets its copies in flight land,
 * frees its tensor memory, writes NaN into its part of the result and adds one to a
 * per-device counter, instead of hanging the GPU. slimkv_abort_count synchronises the
 * current device and returns that counter (thread blocks that gave up since the library
 * was loaded or last reset; with reset != 0 it is set back to 0), or -1 on a CUDA error.
 * A status of SLIMKV_OK from a call only means that its launches were accepted. */
long long slimkv_abort_count(int reset);

/* Test hook for the failure path above: in the next tensor-core decode launch made by
 * this host thread, thread block `cta` of the split-decode kernel does not load its
 * first key tile, so that its wait for it runs out (about 2 s later) and the abort path
 * runs. Nothing faults: the block returns, its result is NaN and the counter rises.
 * A negative `cta` clears a pending request. Not for production use. */
void slimkv_test_withhold_first_load(int cta);

/* SLIMKV_ABI_VERSION of the loaded library. */
int slimkv_abi_version(void);

/* Kernel path a call `which` with `shape` takes on the current device:
 * 1 = tcgen05/TMA path (bf16 storage, d == 128, sm_100-family device),
 * 0 = SIMT float32 path (float32 storage, shapes the tensor-core kernels do not take,
 * or forced), -1 = invalid shape. */
int slimkv_kernel_path(const slimkv_shape* shape, int which);

/* Process-wide switch: force the SIMT path for every later call (on != 0), or
 * restore automatic selection (on == 0). Returns the previous setting. Meant for
 * cross-checking the two paths; not thread-safe against concurrent calls. */
int slimkv_force_simt(int on);

/* Measurement hook: the next call made by this host thread records `start_event`
 * on its stream right before launching its split-decode kernel (for
 * slimkv_prefill_attn: its prefill kernel) and `stop_event` right after it (both cudaEvent_t passed as void*, created by the caller), so
 * cudaEventElapsedTime gives that kernel's duration. One-shot; NULL events
 * cancel a pending request. The events also stop the decode kernel from
 * overlapping the kernel before it, so the time measured is the kernel alone.
 * They are recorded as external events (cudaEventRecordExternal), so a call made
 * under stream capture puts timeable event-record nodes into the graph. */
void slimkv_time_next_decode(void* start_event, void* stop_event);

#ifdef __cplusplus
}
#endif

#endif /* SLIMKV_H */

"""Oracle for SlimKV decode-step attention: plain, slow, float64, CPU.

TEST INFRASTRUCTURE. Only the tests, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may import this module. The library's CUDA path
never calls it and shares no code with it.

Source: "Can SlimKV compress KV cache jointly across tokens and features"
(wispaper.ai), section "Latent-space attention removes the rebuild step", which
states the decode rule: RoPE stays on all queries and on raw-window keys; beacon
keys carry no key-side RoPE and are cached only as latent rows C_K, C_V; scores
against beacons are (Q' U_K) C_K^T with the query projection taken after
grouped-query grouping; values aggregate as (A C_V) U_V^T, i.e. in latent form
before the up-projection. The SlimKV abstract (omanscience.com citation record)
restates the same: a K-RoPE-free constraint enables latent-space attention in
decoding without full-dimensional reconstruction.

Readings where the pages are silent (each also listed in the design notes):
* RoPE pairs element i with element i + d/2 ("rotate-half"), with
  theta_i = base^(-2i/d); no frequency remapping.
* One softmax spans the beacon scores and the window scores of a query head.
* The score scale is the same for both sets (1/sqrt(d) in every workload).
* Query head h belongs to KV group g = h // (Hq / Hkv); U^(g) is the block of
  rows g*d .. (g+1)*d of U, i.e. the part of the up-projection that produces
  KV head g.
* No masking: a decode query sees every beacon and every window token.

Every function takes and returns float64 numpy arrays.
"""
from __future__ import annotations

import numpy as np


def rope_angles(d: int, pos: float, base: float) -> np.ndarray:
    """Angles p * theta_i for i < d/2, theta_i = base^(-2i/d) (float64)."""
    i = np.arange(d // 2, dtype=np.float64)
    theta = np.power(float(base), -2.0 * i / d)
    return float(pos) * theta


def rope(x: np.ndarray, pos: float, base: float) -> np.ndarray:
    """Rotate-half RoPE of the last axis of ``x`` at position ``pos``.

    For i < d/2: x'_i = x_i cos(p th_i) - x_{i+d/2} sin(p th_i) and
    x'_{i+d/2} = x_{i+d/2} cos(p th_i) + x_i sin(p th_i).
    """
    d = x.shape[-1]
    h = d // 2
    ang = rope_angles(d, pos, base)
    c, s = np.cos(ang), np.sin(ang)
    x1, x2 = x[..., :h], x[..., h:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def softmax_weights(scores: np.ndarray):
    """Unnormalised weights w = exp(s - max s), their sum l and the max m."""
    m = np.max(scores)
    w = np.exp(scores - m)
    return w, np.sum(w), m


def _groups(Hq: int, Hkv: int) -> int:
    if Hq % Hkv:
        raise ValueError("Hq must be a multiple of Hkv")
    return Hq // Hkv


def _pairs(B, Hq, pairs):
    return [(b, h) for b in range(B) for h in range(Hq)] if pairs is None else list(pairs)


def decode_attn(q, C_K, C_V, K_raw, V_raw, U_K, U_V, q_pos, scale, rope_base,
                pairs=None, return_weights=False):
    """Reconstruction-free decode attention for one layer.

    q [B,Hq,d]; C_K [B,N_b,r_k]; C_V [B,N_b,r_v]; K_raw, V_raw [B,W,Hkv,d]
    (keys stored after RoPE); U_K [Hkv*d,r_k]; U_V [Hkv*d,r_v]; q_pos [B].
    Returns out [B,Hq,d] (rows not in ``pairs`` stay zero) and, with
    ``return_weights``, the normalised weights of each computed (b, h).
    For every (b, h), with g its KV group and p its position:
      qr = RoPE(q[b,h], p)                 (query RoPE)
      qt = qr . U_K^(g)                    (query projected into latent space)
      s  = [scale * C_K[b] qt ; scale * K_raw[b,:,g] qr]   (one score vector)
      A  = softmax(s)
      out = (A_beacon . C_V[b]) . U_V^(g)T + A_window . V_raw[b,:,g]
    """
    B, Hq, d = q.shape
    Hkv = U_K.shape[0] // d if U_K is not None else K_raw.shape[2]
    G = _groups(Hq, Hkv)
    N_b = 0 if C_K is None else C_K.shape[1]
    out = np.zeros((B, Hq, d))
    weights = {}
    for b, h in _pairs(B, Hq, pairs):
        g = h // G
        qr = rope(q[b, h], q_pos[b], rope_base)
        parts = []
        if N_b:
            UKg = U_K[g * d:(g + 1) * d, :]          # [d, r_k]
            qt = qr @ UKg                            # (Q' U_K)
            parts.append(scale * (C_K[b] @ qt))      # (Q' U_K) C_K^T
        if K_raw is not None and K_raw.shape[1]:
            parts.append(scale * (K_raw[b, :, g, :] @ qr))
        s = np.concatenate(parts)
        w, l, _ = softmax_weights(s)
        o = np.zeros(d)
        if N_b:
            UVg = U_V[g * d:(g + 1) * d, :]          # [d, r_v]
            z = w[:N_b] @ C_V[b]                     # (A C_V): latent aggregate
            o = o + z @ UVg.T                        # ... then (.) U_V^T
        if K_raw is not None and K_raw.shape[1]:
            o = o + w[N_b:] @ V_raw[b, :, g, :]
        out[b, h] = o / l
        if return_weights:
            weights[(b, h)] = w / l
    return (out, weights) if return_weights else out


def window_positions(W: int, q_pos: int) -> np.ndarray:
    """Absolute positions of the W raw-window slots for a query at q_pos. The window is
    the ring of the decode loop (token p in slot p mod W, the current token appended
    before the decode), so slot s holds the latest position congruent to s mod W that
    does not exceed q_pos: q_pos - ((q_pos - s) mod W)."""
    s = np.arange(W)
    return (q_pos - np.mod(q_pos - s, W)).astype(np.float64)


def decode_attn_alibi(q, C_K, C_V, K_raw, V_raw, U_K, U_V, q_pos, scale, rope_base, slopes, ratio,
                      pairs=None):
    """The reconstruction-free decode with an ALiBi bias added after the QK product
    ("Latent-space attention removes the rebuild step" claims the latent scores stay
    compatible with ALiBi because the bias enters after QK). Head h adds
    slopes[h] * (key position - q_pos) to every score: beacon j sits at
    ``beacon_positions(N_b, ratio)[j]``, window slot s at ``window_positions``. The
    rest is ``decode_attn``: RoPE on the query and the raw keys, latent beacon scores
    (RoPE(q) U_K^(g)) C_K^T, one softmax, (A C_V) U_V^(g)T + A V_raw."""
    B, Hq, d = q.shape
    Hkv = U_K.shape[0] // d if U_K is not None else K_raw.shape[2]
    G = _groups(Hq, Hkv)
    N_b = 0 if C_K is None else C_K.shape[1]
    W = 0 if K_raw is None else K_raw.shape[1]
    out = np.zeros((B, Hq, d))
    for b, h in _pairs(B, Hq, pairs):
        g = h // G
        p = float(q_pos[b])
        qr = rope(q[b, h], p, rope_base)
        parts = []
        if N_b:
            qt = qr @ U_K[g * d:(g + 1) * d, :]
            parts.append(scale * (C_K[b] @ qt) + slopes[h] * (beacon_positions(N_b, ratio) - p))
        if W:
            parts.append(scale * (K_raw[b, :, g, :] @ qr) + slopes[h] * (window_positions(W, int(q_pos[b])) - p))
        s = np.concatenate(parts)
        w, l, _ = softmax_weights(s)
        o = np.zeros(d)
        if N_b:
            o = o + (w[:N_b] @ C_V[b]) @ U_V[g * d:(g + 1) * d, :].T
        if W:
            o = o + w[N_b:] @ V_raw[b, :, g, :]
        out[b, h] = o / l
    return out


def reconstruct_kv(C, U, Hkv: int, d: int):
    """Explicit reconstruction C . U^T reshaped to [B, N_b, Hkv, d] (no RoPE)."""
    B, N_b, _ = C.shape
    return (C @ U.T).reshape(B, N_b, Hkv, d)


def gqa_attn(q, K, V, q_pos, scale, rope_base, pairs=None):
    """Standard RoPE GQA decode attention over a cache of RoPE'd keys.

    q [B,Hq,d]; K, V [B,T,Hkv,d]. out[b,h] = softmax(scale * K[b,:,g] qr) V[b,:,g].
    """
    B, Hq, d = q.shape
    Hkv = K.shape[2]
    G = _groups(Hq, Hkv)
    out = np.zeros((B, Hq, d))
    for b, h in _pairs(B, Hq, pairs):
        g = h // G
        qr = rope(q[b, h], q_pos[b], rope_base)
        s = scale * (K[b, :, g, :] @ qr)
        w, l, _ = softmax_weights(s)
        out[b, h] = (w @ V[b, :, g, :]) / l
    return out


def decode_attn_reconstruct(q, C_K, C_V, K_raw, V_raw, U_K, U_V, q_pos, scale,
                            rope_base, pairs=None):
    """The feature-wise baseline: materialise K_b = C_K U_K^T and V_b = C_V U_V^T
    at full dimension (beacon keys get no RoPE), then attend over beacons and the
    raw window with standard GQA attention."""
    d = q.shape[2]
    Hkv = U_K.shape[0] // d
    K_b = reconstruct_kv(C_K, U_K, Hkv, d)
    V_b = reconstruct_kv(C_V, U_V, Hkv, d)
    K = np.concatenate([K_b, K_raw], axis=1)
    V = np.concatenate([V_b, V_raw], axis=1)
    return gqa_attn(q, K, V, q_pos, scale, rope_base, pairs=pairs)


def beacon_positions(N_b: int, ratio: int) -> np.ndarray:
    """Positions given to the beacon keys by the reconstruction baseline that keeps
    beacon-key RoPE. Reading taken (the pages say the baseline keeps beacon key RoPE
    but not where a beacon sits): beacon j condenses tokens j*ratio .. j*ratio +
    ratio - 1 and takes the position of the last of them, j*ratio + ratio - 1."""
    return np.arange(N_b, dtype=np.float64) * ratio + (ratio - 1)


def decode_attn_reconstruct_rope(q, C_K, C_V, K_raw, V_raw, U_K, U_V, q_pos, scale,
                                 rope_base, ratio, pairs=None):
    """The paper's reconstruction baseline ("Speedups are real, but memory is set by
    the ratio": it keeps beacon key RoPE): materialise K_b = C_K U_K^T and V_b =
    C_V U_V^T at full dimension, rotate every reconstructed beacon key of every KV
    head at its beacon position (``beacon_positions``), then attend over beacons and
    the raw window with standard GQA attention. Unlike ``decode_attn_reconstruct``
    this is not equal to the latent path: a rotated key has no latent form."""
    d = q.shape[2]
    Hkv = U_K.shape[0] // d
    K_b = reconstruct_kv(C_K, U_K, Hkv, d)
    V_b = reconstruct_kv(C_V, U_V, Hkv, d)
    for j, p in enumerate(beacon_positions(K_b.shape[1], ratio)):
        K_b[:, j] = rope(K_b[:, j], p, rope_base)
    K = np.concatenate([K_b, K_raw], axis=1)
    V = np.concatenate([V_b, V_raw], axis=1)
    return gqa_attn(q, K, V, q_pos, scale, rope_base, pairs=pairs)


def decode_attn_full_kv(q, K, V, q_pos, scale, rope_base, pairs=None):
    """Uncompressed GQA decode over a full RoPE'd cache (the speed baseline)."""
    return gqa_attn(q, K, V, q_pos, scale, rope_base, pairs=pairs)


# ---------------------------------------------------------------------------
# Multi-step decode: appending the current token to the raw window.
#
# The decode rule above keeps raw-window keys after RoPE. A generation loop
# therefore rotates each new key once, at its own absolute position, when it is
# appended. Reading taken here (the pages condense old raw tokens into beacons,
# which needs trained projections and is out of scope): the window is a ring of W
# slots, the token at absolute position p lives in slot p mod W, so appending
# token p replaces token p - W. Attention is invariant to the order of the window
# rows, so the ring order needs no bookkeeping.
# ---------------------------------------------------------------------------

def round_bf16(x: np.ndarray) -> np.ndarray:
    """Round float64 values to the nearest bfloat16 value, ties to even (the
    storage rounding of a bf16 cache), returned as float64. bfloat16 keeps 8
    significant bits: x = m 2^e with 0.5 <= |m| < 1 is rounded to a multiple of
    2^(e-8); numpy's round is round-half-to-even."""
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)
    return np.ldexp(np.round(m * 256.0), e - 8)


def append_kv(K_raw, V_raw, k_new, v_new, pos, rope_base, storage: str = "bf16"):
    """Append the current token of every batch element to the raw window.

    K_raw, V_raw [B, W, Hkv, d] (keys after RoPE); k_new, v_new [B, Hkv, d];
    pos [B] absolute positions. Slot pos[b] mod W of batch element b receives
    RoPE(k_new[b], pos[b]) and v_new[b], both rounded to the storage type
    ("bf16" or "f32"). Returns new arrays; the inputs are not modified."""
    K = np.array(K_raw, dtype=np.float64, copy=True)
    V = np.array(V_raw, dtype=np.float64, copy=True)
    W = K.shape[1]
    rnd = round_bf16 if storage == "bf16" else (lambda a: np.asarray(a, np.float32).astype(np.float64))
    for b in range(K.shape[0]):
        slot = int(pos[b]) % W
        K[b, slot] = rnd(rope(np.asarray(k_new[b], np.float64), float(pos[b]), rope_base))
        V[b, slot] = rnd(np.asarray(v_new[b], np.float64))
    return K, V


# ---------------------------------------------------------------------------
# Prefill: a chunk of new tokens attending to the beacons and, causally, to itself.
#
# "Speedups are real, but memory is set by the ratio" reports time-to-first-token
# gains over the reconstruction variant from skipping key-side RoPE and full-key
# materialisation for beacon states, i.e. the prompt's chunks are processed against
# the latent beacon memory by the same rule as a decode query. Reading taken here
# (the pages give no chunked-prefill formula): every query token t of a chunk of T
# tokens, at position p0 + t, sees every beacon of the memory (latent scores, no
# key-side RoPE) and the chunk's own tokens s <= t (keys stored after RoPE at
# p0 + s), all in one softmax. This is the decode rule with the raw window replaced
# by the causal prefix of the chunk.
# ---------------------------------------------------------------------------

def _triples(B, T, Hq, triples):
    if triples is None:
        return [(b, t, h) for b in range(B) for t in range(T) for h in range(Hq)]
    return list(triples)


def prefill_attn(q, C_K, C_V, K_chunk, V_chunk, U_K, U_V, p0, scale, rope_base, triples=None):
    """Chunked-prefill attention of one layer over the beacon memory and the chunk.

    q [B,T,Hq,d] (the chunk's queries, before RoPE); C_K [B,N_b,r_k]; C_V [B,N_b,r_v];
    K_chunk, V_chunk [B,T,Hkv,d] (the chunk's keys stored after RoPE at p0 + s, and its
    values); U_K [Hkv*d,r_k]; U_V [Hkv*d,r_v]; p0 [B] the position of chunk token 0.
    Returns out [B,T,Hq,d] (entries not in ``triples`` stay zero). For every (b, t, h),
    with g the KV group of h and p = p0[b] + t:
      qr = RoPE(q[b,t,h], p);  qt = qr . U_K^(g)
      s  = [scale * C_K[b] qt ; scale * K_chunk[b, 0..t, g] qr]
      A  = softmax(s)
      out = (A_beacon . C_V[b]) . U_V^(g)T + A_chunk . V_chunk[b, 0..t, g]
    """
    B, T, Hq, d = q.shape
    Hkv = U_K.shape[0] // d if U_K is not None else K_chunk.shape[2]
    G = _groups(Hq, Hkv)
    N_b = 0 if C_K is None else C_K.shape[1]
    out = np.zeros((B, T, Hq, d))
    for b, t, h in _triples(B, T, Hq, triples):
        g = h // G
        qr = rope(q[b, t, h], float(p0[b]) + t, rope_base)
        parts = []
        if N_b:
            qt = qr @ U_K[g * d:(g + 1) * d, :]
            parts.append(scale * (C_K[b] @ qt))
        parts.append(scale * (K_chunk[b, :t + 1, g, :] @ qr))   # causal: s <= t
        s = np.concatenate(parts)
        w, l, _ = softmax_weights(s)
        o = np.zeros(d)
        if N_b:
            o = o + (w[:N_b] @ C_V[b]) @ U_V[g * d:(g + 1) * d, :].T
        o = o + w[N_b:] @ V_chunk[b, :t + 1, g, :]
        out[b, t, h] = o / l
    return out

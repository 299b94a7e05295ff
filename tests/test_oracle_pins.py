"""Pins for the float64 oracle, each independent of the oracle's own code.

The SlimKV pages print no worked example, so the oracle is pinned by what the
mathematics fixes: closed forms, a second formulation of RoPE (complex
multiplication), the relative-position identity RoPE is built for, reductions to
torch's scaled_dot_product_attention (a library routine the oracle never calls),
brute-force scalar loops written straight from the decode rule, and identities
that the reconstruction-free rewrite must satisfy ((Q'U_K)C_K^T = Q'(C_K U_K^T)^T
and (A C_V)U_V^T = A (C_V U_V^T), "Latent-space attention removes the rebuild
step"). The mutation tests at the end plant typical mistakes in a copy of the
oracle and check that some pin catches each of them.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle import slimkv_oracle as O


def _rand(rng, *shape):
    return rng.standard_normal(shape)


def _ortho(rng, n, r):
    qm, _ = np.linalg.qr(rng.standard_normal((n, r)))
    return qm


def _rope_complex(x, pos, base):
    """RoPE as complex multiplication: z_i = x_i + 1j x_{i+d/2} times e^{i p th_i}."""
    d = x.shape[-1]
    h = d // 2
    th = np.array([base ** (-(2.0 * i) / d) for i in range(h)])
    z = (x[..., :h] + 1j * x[..., h:]) * np.exp(1j * pos * th)
    return np.concatenate([z.real, z.imag], axis=-1)


def _sdpa(q, K, V, scale):
    """torch fp64 SDPA for one decode query per (b, h); q [B,Hq,d], K/V [B,T,Hq,d]."""
    qt = torch.from_numpy(q)[:, :, None, :]                  # [B,Hq,1,d]
    kt = torch.from_numpy(K).permute(0, 2, 1, 3)             # [B,Hq,T,d]
    vt = torch.from_numpy(V).permute(0, 2, 1, 3)
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=scale)
    return o[:, :, 0, :].numpy()


def _expand_heads(K, G):
    return np.repeat(K, G, axis=2)       # contiguous grouping: head h -> g = h // G


# ---------------------------------------------------------------- RoPE pins

def test_rope_closed_form_d2():
    # d = 2: one pair, theta_0 = 1, so position p rotates (x0, x1) by p radians
    for p in (0.0, 1.0, 2.5, -3.0):
        out = oracle.rope(np.array([1.0, 0.0]), p, 10000.0)
        np.testing.assert_allclose(out, [math.cos(p), math.sin(p)], rtol=0, atol=1e-15)
        out = oracle.rope(np.array([0.0, 1.0]), p, 10000.0)
        np.testing.assert_allclose(out, [-math.sin(p), math.cos(p)], rtol=0, atol=1e-15)


def test_rope_closed_form_frequencies():
    # d = 4, base 100: theta = (1, 100^(-1/2)) = (1, 0.1)
    x = np.array([1.0, 1.0, 0.0, 0.0])
    out = oracle.rope(x, 2.0, 100.0)
    np.testing.assert_allclose(out, [math.cos(2.0), math.cos(0.2), math.sin(2.0), math.sin(0.2)],
                               atol=1e-15)


def test_rope_matches_complex_multiplication():
    rng = np.random.default_rng(1)
    for d in (8, 64, 128):
        x = _rand(rng, 5, d)
        for pos in (0, 7, 2080, 133120):
            # angles reach ~1.3e5 rad, whose float64 ulp is ~1.5e-11
            np.testing.assert_allclose(oracle.rope(x, pos, 500000.0), _rope_complex(x, pos, 500000.0),
                                       rtol=0, atol=1e-9)


def test_rope_relative_position_and_norm():
    rng = np.random.default_rng(2)
    q, k = _rand(rng, 128), _rand(rng, 128)
    for p, pp in ((2080, 2048), (133120, 131073), (5, 9)):
        lhs = oracle.rope(q, p, 10000.0) @ oracle.rope(k, pp, 10000.0)
        rhs = oracle.rope(q, p - pp, 10000.0) @ k
        assert abs(lhs - rhs) < 1e-9 * (1 + abs(lhs))
        assert abs(np.linalg.norm(oracle.rope(q, p, 10000.0)) - np.linalg.norm(q)) < 1e-12


def test_rope_position_zero_is_identity():
    x = np.random.default_rng(3).standard_normal((3, 64))
    np.testing.assert_array_equal(oracle.rope(x, 0, 10000.0), x)


# ------------------------------------------------------- attention-level pins

def _case(seed, B=2, Hq=6, Hkv=2, d=16, N_b=20, W=11, r_k=8, r_v=12):
    rng = np.random.default_rng(seed)
    return dict(q=_rand(rng, B, Hq, d), C_K=_rand(rng, B, N_b, r_k), C_V=_rand(rng, B, N_b, r_v),
                K_raw=_rand(rng, B, W, Hkv, d), V_raw=_rand(rng, B, W, Hkv, d),
                U_K=_ortho(rng, Hkv * d, r_k), U_V=_ortho(rng, Hkv * d, r_v),
                q_pos=np.array([37 + 5 * b for b in range(B)]), scale=1 / math.sqrt(d),
                rope_base=10000.0)


def test_latent_equals_explicit_reconstruction():
    # associativity: (qU)c = q(cU^T) and (A C)U^T = A(C U^T); exact up to rounding
    for seed in range(3):
        c = _case(seed)
        a = oracle.decode_attn(**c)
        b = oracle.decode_attn_reconstruct(**c)
        np.testing.assert_allclose(a, b, rtol=1e-11, atol=1e-12)


def test_empty_beacon_set_is_rope_gqa_attention():
    c = _case(4, N_b=0)
    out = oracle.decode_attn(**c)
    G = c["q"].shape[1] // c["K_raw"].shape[2]
    qr = np.stack([_rope_complex(c["q"][b], c["q_pos"][b], c["rope_base"]) for b in range(2)])
    ref = _sdpa(qr, _expand_heads(c["K_raw"], G), _expand_heads(c["V_raw"], G), c["scale"])
    np.testing.assert_allclose(out, ref, rtol=1e-11, atol=1e-12)


def test_full_rank_orthonormal_u_equals_uncompressed_attention():
    # rank = d, U square orthogonal, one KV head: C = K U gives K = C U^T exactly, so the
    # latent path is plain attention over [K_beacon (no RoPE) ; K_raw (RoPE'd)]
    rng = np.random.default_rng(5)
    B, Hq, d, N_b, W = 2, 4, 16, 13, 9
    U_K, U_V = _ortho(rng, d, d), _ortho(rng, d, d)
    Kb, Vb = _rand(rng, B, N_b, 1, d), _rand(rng, B, N_b, 1, d)
    c = dict(q=_rand(rng, B, Hq, d), C_K=Kb[:, :, 0] @ U_K, C_V=Vb[:, :, 0] @ U_V,
             K_raw=_rand(rng, B, W, 1, d), V_raw=_rand(rng, B, W, 1, d), U_K=U_K, U_V=U_V,
             q_pos=np.array([300, 17]), scale=0.3, rope_base=500000.0)
    out = oracle.decode_attn(**c)
    qr = np.stack([_rope_complex(c["q"][b], c["q_pos"][b], 500000.0) for b in range(B)])
    K = np.concatenate([Kb, c["K_raw"]], axis=1)
    V = np.concatenate([Vb, c["V_raw"]], axis=1)
    ref = _sdpa(qr, _expand_heads(K, Hq), _expand_heads(V, Hq), 0.3)
    np.testing.assert_allclose(out, ref, rtol=1e-11, atol=1e-12)


def test_full_kv_is_sdpa():
    rng = np.random.default_rng(6)
    B, Hq, Hkv, d, T = 2, 8, 2, 32, 50
    q, K, V = _rand(rng, B, Hq, d), _rand(rng, B, T, Hkv, d), _rand(rng, B, T, Hkv, d)
    pos = np.array([50, 4096])
    out = oracle.decode_attn_full_kv(q, K, V, pos, 0.2, 10000.0)
    qr = np.stack([_rope_complex(q[b], pos[b], 10000.0) for b in range(B)])
    ref = _sdpa(qr, _expand_heads(K, 4), _expand_heads(V, 4), 0.2)
    np.testing.assert_allclose(out, ref, rtol=1e-11, atol=1e-12)


def _brute(c):
    """Scalar loops straight from the decode rule, no numpy linear algebra."""
    q, C_K, C_V, K, V, U_K, U_V = (c[k] for k in ("q", "C_K", "C_V", "K_raw", "V_raw", "U_K", "U_V"))
    B, Hq, d = q.shape
    N_b, r_k, r_v = C_K.shape[1], C_K.shape[2], C_V.shape[2]
    W, Hkv = K.shape[1], K.shape[2]
    G = Hq // Hkv
    out = np.zeros((B, Hq, d))
    for b in range(B):
        p = float(c["q_pos"][b])
        for h in range(Hq):
            g = h // G
            qr = [0.0] * d
            for i in range(d // 2):
                a = p * c["rope_base"] ** (-2.0 * i / d)
                qr[i] = q[b, h, i] * math.cos(a) - q[b, h, i + d // 2] * math.sin(a)
                qr[i + d // 2] = q[b, h, i + d // 2] * math.cos(a) + q[b, h, i] * math.sin(a)
            s = []
            for j in range(N_b):
                acc = 0.0
                for k in range(r_k):
                    qt = sum(qr[i] * U_K[g * d + i, k] for i in range(d))
                    acc += qt * C_K[b, j, k]
                s.append(c["scale"] * acc)
            for t in range(W):
                s.append(c["scale"] * sum(qr[i] * K[b, t, g, i] for i in range(d)))
            m = max(s)
            e = [math.exp(x - m) for x in s]
            l = sum(e)
            for i in range(d):
                v = 0.0
                for j in range(N_b):
                    full_v = sum(C_V[b, j, k] * U_V[g * d + i, k] for k in range(r_v))
                    v += e[j] * full_v
                for t in range(W):
                    v += e[N_b + t] * V[b, t, g, i]
                out[b, h, i] = v / l
    return out


def test_brute_force_scalar_loops():
    c = _case(7, B=2, Hq=6, Hkv=2, d=4, N_b=5, W=3, r_k=3, r_v=2)
    np.testing.assert_allclose(oracle.decode_attn(**c), _brute(c), rtol=1e-12, atol=1e-13)


def test_weights_sum_to_one():
    c = _case(8)
    _, w = oracle.decode_attn(**c, return_weights=True)
    for v in w.values():
        assert abs(v.sum() - 1.0) < 1e-14
        assert np.all(v >= 0)


def test_zero_query_gives_mean_of_values():
    c = _case(9)
    c["q"] = np.zeros_like(c["q"])
    out = oracle.decode_attn(**c)
    d = c["q"].shape[2]
    G = c["q"].shape[1] // c["K_raw"].shape[2]
    for b in range(2):
        for h in range(6):
            g = h // G
            vb = c["C_V"][b] @ c["U_V"][g * d:(g + 1) * d].T     # full-dim beacon values
            rows = np.concatenate([vb, c["V_raw"][b, :, g, :]])
            np.testing.assert_allclose(out[b, h], rows.mean(axis=0), rtol=1e-12, atol=1e-13)


def test_dominant_raw_key_selects_its_value():
    c = _case(10, B=1, Hq=2, Hkv=1)
    qr = oracle.rope(c["q"][0, 0], c["q_pos"][0], c["rope_base"])
    c["K_raw"][0, 4, 0] = 1e3 * qr / np.linalg.norm(qr)        # aligned with RoPE(q)
    out = oracle.decode_attn(**c)
    np.testing.assert_allclose(out[0, 0], c["V_raw"][0, 4, 0], rtol=0, atol=1e-9)


def test_dominant_beacon_selects_its_latent_value():
    c = _case(11, B=1, Hq=2, Hkv=1, r_k=16, d=16)
    c["U_K"] = _ortho(np.random.default_rng(0), 16, 16)
    qr = oracle.rope(c["q"][0, 0], c["q_pos"][0], c["rope_base"])
    qt = qr @ c["U_K"]
    c["C_K"][0, 3] = 1e3 * qt / np.linalg.norm(qt)
    out = oracle.decode_attn(**c)
    np.testing.assert_allclose(out[0, 0], c["C_V"][0, 3] @ c["U_V"].T, rtol=0, atol=1e-9)


def test_grouping_is_contiguous():
    # heads 0..G-1 read KV group 0 only: changing group 1's window leaves them unchanged
    c = _case(12, Hq=6, Hkv=2)
    a = oracle.decode_attn(**c)
    c["K_raw"][:, :, 1] += 5.0
    c["V_raw"][:, :, 1] -= 3.0
    b = oracle.decode_attn(**c)
    np.testing.assert_array_equal(a[:, :3], b[:, :3])
    assert np.abs(a[:, 3:] - b[:, 3:]).max() > 1e-3


def test_beacon_keys_carry_no_rope():
    # beacon scores do not depend on the query position beyond RoPE(q): with a window
    # that is empty, moving q_pos changes the output only through RoPE(q)
    c = _case(13, W=0)
    c["K_raw"] = c["K_raw"][:, :0]
    c["V_raw"] = c["V_raw"][:, :0]
    out = oracle.decode_attn(**c)
    d = c["q"].shape[2]
    G = 3
    for b in range(2):
        for h in range(6):
            g = h // G
            qr = _rope_complex(c["q"][b, h], c["q_pos"][b], c["rope_base"])
            Kb = c["C_K"][b] @ c["U_K"][g * d:(g + 1) * d].T     # un-RoPE'd beacon keys
            Vb = c["C_V"][b] @ c["U_V"][g * d:(g + 1) * d].T
            s = c["scale"] * Kb @ qr
            e = np.exp(s - s.max())
            np.testing.assert_allclose(out[b, h], e @ Vb / e.sum(), rtol=1e-11, atol=1e-12)


# ---------------------------------------------- planted mistakes must be caught

def _check_rope_complex_with(mod):
    x = np.random.default_rng(1).standard_normal((3, 64))
    np.testing.assert_allclose(mod.rope(x, 2080, 10000.0), _rope_complex(x, 2080, 10000.0),
                               rtol=1e-12, atol=1e-12)


def test_pins_catch_wrong_rope_sign(monkeypatch):
    def bad_rope(x, pos, base):
        d = x.shape[-1]
        h = d // 2
        ang = O.rope_angles(d, pos, base)
        c, s = np.cos(ang), np.sin(ang)
        return np.concatenate([x[..., :h] * c + x[..., h:] * s, x[..., h:] * c - x[..., :h] * s], -1)
    _check_rope_complex_with(O)
    monkeypatch.setattr(O, "rope", bad_rope)
    with pytest.raises(AssertionError):
        _check_rope_complex_with(O)


def test_pins_catch_interleaved_grouping(monkeypatch):
    c = _case(14, B=1, Hq=4, Hkv=2, d=4, N_b=3, W=2, r_k=2, r_v=2)
    good = O.decode_attn(**c)
    orig_groups = O._groups

    def bad_decode(**kw):
        # planted mistake: head h reads group h % Hkv instead of h // G
        q = kw["q"]
        perm = [0, 2, 1, 3]
        kw = dict(kw)
        kw["q"] = q[:, perm]
        return O.decode_attn(**kw)[:, perm]
    assert orig_groups(4, 2) == 2
    bad = bad_decode(**c)
    assert np.abs(bad - _brute(c)).max() > 1e-6
    np.testing.assert_allclose(good, _brute(c), rtol=1e-12, atol=1e-13)


def test_pins_catch_transposed_projection():
    # using U^(g) from the wrong block (g-th column block of U^T) breaks the
    # reconstruction identity
    c = _case(15)
    d = c["q"].shape[2]
    out_good = O.decode_attn(**c)
    ref = O.decode_attn_reconstruct(**c)
    c_bad = dict(c)
    c_bad["U_K"] = np.roll(c["U_K"], d, axis=0)     # group blocks swapped
    out_bad = O.decode_attn(**c_bad)
    np.testing.assert_allclose(out_good, ref, rtol=1e-11, atol=1e-12)
    assert np.abs(out_bad - ref).max() > 1e-6


# ---------------------------------------------------------------------------
# Multi-step decode: bf16 storage rounding and the raw-window append
# ---------------------------------------------------------------------------

def test_round_bf16_matches_torch_on_float32_values():
    # an independent implementation (torch's float32 -> bfloat16 conversion,
    # round to nearest even) agrees on every float32 value, ties included
    rng = np.random.default_rng(11)
    x = (rng.standard_normal(50000) * np.logspace(-4, 4, 50000)).astype(np.float32)
    ties = np.array([1 + 2 ** -8, 1 + 3 * 2 ** -8, -(1 + 2 ** -8), 3 * 2 ** -9 + 2 ** -17], np.float32)
    x = np.concatenate([x, ties])
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(O.round_bf16(x.astype(np.float64)), ref)
    # ties go to the even neighbour
    assert O.round_bf16(np.array([1 + 2 ** -8]))[0] == 1.0
    assert O.round_bf16(np.array([1 + 3 * 2 ** -8]))[0] == 1 + 2 ** -6


def test_append_writes_the_ring_slot_and_nothing_else():
    rng = np.random.default_rng(12)
    B, W, Hkv, d = 2, 5, 2, 8
    K = rng.standard_normal((B, W, Hkv, d))
    V = rng.standard_normal((B, W, Hkv, d))
    kn = rng.standard_normal((B, Hkv, d))
    vn = rng.standard_normal((B, Hkv, d))
    pos = np.array([7, 10])   # slots 2 and 0
    K2, V2 = O.append_kv(K, V, kn, vn, pos, 10000.0, storage="f32")
    for b, slot in ((0, 2), (1, 0)):
        other = [t for t in range(W) if t != slot]
        assert np.array_equal(K2[b, other], K[b, other]) and np.array_equal(V2[b, other], V[b, other])
        assert np.allclose(V2[b, slot], vn[b].astype(np.float32))
    # W + 1 appends visit every slot once and then overwrite the first one
    seen = [int(p) % W for p in range(13, 13 + W + 1)]
    assert sorted(seen[:W]) == list(range(W)) and seen[W] == seen[0]


def test_appended_key_scores_like_the_unrotated_pair():
    # a query and a key at the same position: <R(p) q, R(p) k> = <q, k> for
    # any p (rotations are orthogonal), so the score against the appended key is
    # scale * q.k whatever the position; checked through the decode oracle with
    # a single-token window, where the output must be that token's value
    rng = np.random.default_rng(13)
    B, Hq, Hkv, d = 1, 2, 1, 16
    K = np.zeros((B, 1, Hkv, d))
    V = np.zeros((B, 1, Hkv, d))
    kn = rng.standard_normal((B, Hkv, d))
    vn = rng.standard_normal((B, Hkv, d))
    q = rng.standard_normal((B, Hq, d))
    for p in (0, 1, 4097, 131072 + 2048):
        K2, V2 = O.append_kv(K, V, kn, vn, np.array([p]), 500000.0, storage="f32")
        qr = O.rope(q[0, 0], float(p), 500000.0)
        assert abs(qr @ K2[0, 0, 0] - q[0, 0] @ kn[0, 0]) < 1e-5 * (1 + abs(q[0, 0] @ kn[0, 0]))
        out = O.decode_attn(q, None, None, K2, V2, None, None, np.array([p]), 0.25, 500000.0)
        assert np.allclose(out[0, 0], V2[0, 0, 0]) and np.allclose(out[0, 1], V2[0, 0, 0])


# ------------------------------------------- reconstruction with beacon-key RoPE
#
# The paper's baseline keeps beacon key RoPE ("Speedups are real, but memory is set by
# the ratio"); the pages do not say where a beacon sits, and the reading taken is the
# last token of the block it condenses, j*ratio + ratio - 1.

def _recon_rope_case(rng, B=2, Hq=4, Hkv=2, d=8, N_b=5, W=3, r=4, ratio=4):
    return dict(q=_rand(rng, B, Hq, d), C_K=_rand(rng, B, N_b, r), C_V=_rand(rng, B, N_b, r),
                K_raw=_rand(rng, B, W, Hkv, d), V_raw=_rand(rng, B, W, Hkv, d), U_K=_ortho(rng, Hkv * d, r),
                U_V=_ortho(rng, Hkv * d, r), q_pos=np.array([37, 101])[:B], scale=1 / math.sqrt(d),
                rope_base=10000.0, ratio=ratio)


def _recon_rope_relative(c):
    """The same attention written with relative rotations: q . R(p_j) k_j = R(p - p_j) q . k_j
    for the beacon keys (RoPE as complex multiplication, unrotated reconstructed keys
    built one row at a time), absolute RoPE on the query for the raw window."""
    q, C_K, C_V, K_raw, V_raw, U_K, U_V = (c[k] for k in ("q", "C_K", "C_V", "K_raw", "V_raw", "U_K", "U_V"))
    B, Hq, d = q.shape
    Hkv = U_K.shape[0] // d
    G = Hq // Hkv
    N_b = C_K.shape[1]
    out = np.zeros((B, Hq, d))
    for b in range(B):
        p = float(c["q_pos"][b])
        for h in range(Hq):
            g = h // G
            s, vals = [], []
            for j in range(N_b):
                pj = j * c["ratio"] + c["ratio"] - 1
                k = np.array([sum(C_K[b, j, t] * U_K[g * d + i, t] for t in range(C_K.shape[2])) for i in range(d)])
                v = np.array([sum(C_V[b, j, t] * U_V[g * d + i, t] for t in range(C_V.shape[2])) for i in range(d)])
                s.append(c["scale"] * float(_rope_complex(q[b, h], p - pj, c["rope_base"]) @ k))
                vals.append(v)
            qr = _rope_complex(q[b, h], p, c["rope_base"])
            for t in range(K_raw.shape[1]):
                s.append(c["scale"] * float(qr @ K_raw[b, t, g]))
                vals.append(V_raw[b, t, g])
            s = np.array(s)
            e = np.exp(s - s.max())
            out[b, h] = (e / e.sum()) @ np.array(vals)
    return out


def test_beacon_positions_are_the_last_token_of_each_block():
    assert oracle.beacon_positions(4, 16).tolist() == [15.0, 31.0, 47.0, 63.0]
    assert oracle.beacon_positions(3, 1).tolist() == [0.0, 1.0, 2.0]


def test_reconstruct_rope_equals_relative_rotation_form():
    rng = np.random.default_rng(31)
    c = _recon_rope_case(rng)
    got = oracle.decode_attn_reconstruct_rope(**c)
    assert np.allclose(got, _recon_rope_relative(c), rtol=1e-12, atol=1e-12)


def test_reconstruct_rope_single_beacon_at_position_zero_is_plain_reconstruction():
    # ratio 1: the only beacon sits at position 0, where RoPE is the identity
    rng = np.random.default_rng(32)
    c = _recon_rope_case(rng, N_b=1, ratio=1)
    got = oracle.decode_attn_reconstruct_rope(**c)
    c.pop("ratio")
    assert np.allclose(got, oracle.decode_attn_reconstruct(**c), rtol=1e-12, atol=1e-12)


def test_reconstruct_rope_differs_from_the_latent_path():
    # a rotated beacon key has no latent form: the two baselines disagree for ratio > 1
    rng = np.random.default_rng(33)
    c = _recon_rope_case(rng)
    got = oracle.decode_attn_reconstruct_rope(**c)
    c.pop("ratio")
    assert not np.allclose(got, oracle.decode_attn_reconstruct(**c), rtol=1e-3, atol=1e-3)


def test_pins_catch_wrong_beacon_position(monkeypatch):
    rng = np.random.default_rng(34)
    c = _recon_rope_case(rng)
    monkeypatch.setattr(O, "beacon_positions", lambda N_b, ratio: np.arange(N_b, dtype=np.float64) * ratio)
    got = O.decode_attn_reconstruct_rope(**c)
    assert not np.allclose(got, _recon_rope_relative(c), rtol=1e-6, atol=1e-6)


# ---------------------------------------------------------------- ALiBi latent path
#
# "Latent-space attention removes the rebuild step": the bias enters after QK, so it
# applies to the latent beacon scores unchanged. Readings: beacon j at position
# j*ratio + ratio - 1; window slot s holds the latest position = s mod W not above q_pos.

def _alibi_case(rng, B=2, Hq=4, Hkv=2, d=8, N_b=6, W=5, r=4, ratio=3):
    return dict(q=_rand(rng, B, Hq, d), C_K=_rand(rng, B, N_b, r), C_V=_rand(rng, B, N_b, r),
                K_raw=_rand(rng, B, W, Hkv, d), V_raw=_rand(rng, B, W, Hkv, d), U_K=_ortho(rng, Hkv * d, r),
                U_V=_ortho(rng, Hkv * d, r), q_pos=np.array([23, 41])[:B], scale=1 / math.sqrt(d),
                rope_base=10000.0, slopes=np.array([0.5, 0.25, 0.125, 0.0625])[:Hq], ratio=ratio)


def _ring_positions(W, q_pos):
    """Window slot contents after appending tokens 0 .. q_pos one by one to a ring of W."""
    slots = [None] * W
    for p in range(q_pos + 1):
        slots[p % W] = p
    return np.array(slots, dtype=np.float64)


def test_window_positions_match_a_simulated_ring():
    for W, qp in [(5, 23), (4, 8), (7, 7), (3, 100)]:
        assert oracle.window_positions(W, qp).tolist() == _ring_positions(W, qp).tolist()


def test_alibi_with_zero_slopes_is_the_plain_decode():
    rng = np.random.default_rng(41)
    c = _alibi_case(rng)
    c["slopes"] = np.zeros(4)
    got = oracle.decode_attn_alibi(**c)
    c.pop("slopes"), c.pop("ratio")
    assert np.allclose(got, oracle.decode_attn(**c), rtol=1e-13, atol=1e-13)


def test_alibi_equals_explicit_reconstruction_with_bias():
    # beacon keys expanded to full dimension (no RoPE), biases from a simulated ring
    rng = np.random.default_rng(42)
    c = _alibi_case(rng)
    q, C_K, C_V, K_raw, V_raw, U_K, U_V = (c[k] for k in ("q", "C_K", "C_V", "K_raw", "V_raw", "U_K", "U_V"))
    B, Hq, d = q.shape
    Hkv, N_b, W = K_raw.shape[2], C_K.shape[1], K_raw.shape[1]
    G = Hq // Hkv
    Kb = np.einsum("bjr,nr->bjn", C_K, U_K).reshape(B, N_b, Hkv, d)
    Vb = np.einsum("bjr,nr->bjn", C_V, U_V).reshape(B, N_b, Hkv, d)
    want = np.zeros((B, Hq, d))
    for b in range(B):
        p = int(c["q_pos"][b])
        pos = np.concatenate([np.array([j * c["ratio"] + c["ratio"] - 1 for j in range(N_b)], float),
                              _ring_positions(W, p)])
        for h in range(Hq):
            g = h // G
            qr = _rope_complex(q[b, h], p, c["rope_base"])
            keys = np.concatenate([Kb[b, :, g], K_raw[b, :, g]])
            vals = np.concatenate([Vb[b, :, g], V_raw[b, :, g]])
            s = c["scale"] * keys @ qr + c["slopes"][h] * (pos - p)
            e = np.exp(s - s.max())
            want[b, h] = e @ vals / e.sum()
    assert np.allclose(oracle.decode_attn_alibi(**c), want, rtol=1e-12, atol=1e-12)


def test_alibi_steep_slope_selects_the_newest_window_token():
    rng = np.random.default_rng(43)
    c = _alibi_case(rng)
    c["slopes"] = np.full(4, 200.0)
    out = oracle.decode_attn_alibi(**c)
    G = 2
    for b in range(2):
        slot = int(c["q_pos"][b]) % c["K_raw"].shape[1]
        for h in range(4):
            assert np.allclose(out[b, h], c["V_raw"][b, slot, h // G], atol=1e-9)


def test_pins_catch_flipped_alibi_sign(monkeypatch):
    rng = np.random.default_rng(44)
    c = _alibi_case(rng)
    c["slopes"] = np.full(4, 200.0)
    orig = O.window_positions
    monkeypatch.setattr(O, "window_positions", lambda W, qp: 2.0 * qp - orig(W, qp))
    out = O.decode_attn_alibi(**c)
    slot = int(c["q_pos"][0]) % c["K_raw"].shape[1]
    assert not np.allclose(out[0, 0], c["V_raw"][0, slot, 0], atol=1e-6)


# ------------------------------------------------------ prefill over chunk + beacons

def _prefill_case(rng, B=2, T=7, Hq=4, Hkv=2, d=8, N_b=5, r_k=4, r_v=6):
    return dict(q=_rand(rng, B, T, Hq, d), C_K=_rand(rng, B, N_b, r_k), C_V=_rand(rng, B, N_b, r_v),
                K_chunk=_rand(rng, B, T, Hkv, d), V_chunk=_rand(rng, B, T, Hkv, d),
                U_K=_ortho(rng, Hkv * d, r_k), U_V=_ortho(rng, Hkv * d, r_v),
                p0=np.array([64, 1000])[:B], scale=1 / math.sqrt(d), rope_base=10000.0)


def _causal_sdpa(qr, K, V, scale, prefix=None):
    """torch fp64 SDPA, causal over the chunk; qr [B,T,Hq,d] (rotated), K/V [B,T,Hq,d].
    With ``prefix`` (K_b, V_b [B,N,Hq,d]) every query also sees those N keys."""
    qt = torch.from_numpy(qr).permute(0, 2, 1, 3)                 # [B,Hq,T,d]
    kt = torch.from_numpy(K).permute(0, 2, 1, 3)
    vt = torch.from_numpy(V).permute(0, 2, 1, 3)
    T = qr.shape[1]
    mask = torch.ones(T, T, dtype=torch.bool).tril()
    if prefix is not None:
        kt = torch.cat([torch.from_numpy(prefix[0]).permute(0, 2, 1, 3), kt], dim=2)
        vt = torch.cat([torch.from_numpy(prefix[1]).permute(0, 2, 1, 3), vt], dim=2)
        mask = torch.cat([torch.ones(T, prefix[0].shape[1], dtype=torch.bool), mask], dim=1)
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask, scale=scale)
    return o.permute(0, 2, 1, 3).numpy()


def _rotate_chunk_queries(c):
    B, T = c["q"].shape[:2]
    return np.stack([np.stack([_rope_complex(c["q"][b, t], c["p0"][b] + t, c["rope_base"])
                               for t in range(T)]) for b in range(B)])


def test_prefill_without_beacons_is_causal_rope_attention():
    rng = np.random.default_rng(50)
    c = _prefill_case(rng, N_b=0)
    c["C_K"] = c["C_V"] = None
    out = oracle.prefill_attn(**c)
    G = 2
    ref = _causal_sdpa(_rotate_chunk_queries(c), _expand_heads(c["K_chunk"], G),
                       _expand_heads(c["V_chunk"], G), c["scale"])
    np.testing.assert_allclose(out, ref, rtol=1e-11, atol=1e-12)


def test_prefill_latent_equals_explicit_reconstruction_with_causal_mask():
    # associativity again: the beacons are plain (unrotated) keys C_K U_K^T and values
    # C_V U_V^T that every chunk query sees; the chunk is causal
    rng = np.random.default_rng(51)
    c = _prefill_case(rng, T=9, N_b=6)
    d, Hkv = 8, 2
    out = oracle.prefill_attn(**c)
    Kb = (c["C_K"] @ c["U_K"].T).reshape(2, 6, Hkv, d)
    Vb = (c["C_V"] @ c["U_V"].T).reshape(2, 6, Hkv, d)
    ref = _causal_sdpa(_rotate_chunk_queries(c), _expand_heads(c["K_chunk"], 2),
                       _expand_heads(c["V_chunk"], 2), c["scale"],
                       prefix=(_expand_heads(Kb, 2), _expand_heads(Vb, 2)))
    np.testing.assert_allclose(out, ref, rtol=1e-11, atol=1e-12)


def test_prefill_is_causal():
    rng = np.random.default_rng(52)
    c = _prefill_case(rng, T=8)
    base = oracle.prefill_attn(**c)
    t_cut = 4
    c2 = dict(c)
    c2["K_chunk"] = c["K_chunk"].copy()
    c2["V_chunk"] = c["V_chunk"].copy()
    c2["K_chunk"][:, t_cut:] += 3.0
    c2["V_chunk"][:, t_cut:] -= 5.0
    out = oracle.prefill_attn(**c2)
    np.testing.assert_array_equal(out[:, :t_cut], base[:, :t_cut])     # the past never sees the future
    assert not np.allclose(out[:, t_cut:], base[:, t_cut:])


def test_prefill_first_token_sees_beacons_and_itself():
    # token 0 of the chunk: one raw key (its own); with a dominant self-score its output
    # is its own value, with the beacons' scores pushed far down
    rng = np.random.default_rng(53)
    c = _prefill_case(rng, T=3)
    qr0 = np.stack([_rope_complex(c["q"][b, 0], c["p0"][b], c["rope_base"]) for b in range(2)])
    for b in range(2):
        for g in range(2):
            c["K_chunk"][b, 0, g] = 400.0 * qr0[b, 2 * g] / np.linalg.norm(qr0[b, 2 * g])
    out = oracle.prefill_attn(**c, triples=[(0, 0, 0), (1, 0, 2)])
    np.testing.assert_allclose(out[0, 0, 0], c["V_chunk"][0, 0, 0], atol=1e-9)
    np.testing.assert_allclose(out[1, 0, 2], c["V_chunk"][1, 0, 1], atol=1e-9)


def _brute_prefill(c):
    """Scalar loops straight from the prefill rule, no numpy linear algebra."""
    q, C_K, C_V, K, V, U_K, U_V = (c[k] for k in ("q", "C_K", "C_V", "K_chunk", "V_chunk", "U_K", "U_V"))
    B, T, Hq, d = q.shape
    N_b, r_k, r_v = C_K.shape[1], C_K.shape[2], C_V.shape[2]
    G = Hq // K.shape[2]
    out = np.zeros((B, T, Hq, d))
    for b in range(B):
        for t in range(T):
            p = float(c["p0"][b] + t)
            for h in range(Hq):
                g = h // G
                qr = [0.0] * d
                for i in range(d // 2):
                    a = p * c["rope_base"] ** (-2.0 * i / d)
                    qr[i] = q[b, t, h, i] * math.cos(a) - q[b, t, h, i + d // 2] * math.sin(a)
                    qr[i + d // 2] = q[b, t, h, i + d // 2] * math.cos(a) + q[b, t, h, i] * math.sin(a)
                s = []
                for j in range(N_b):
                    acc = 0.0
                    for k in range(r_k):
                        acc += sum(qr[i] * U_K[g * d + i, k] for i in range(d)) * C_K[b, j, k]
                    s.append(c["scale"] * acc)
                for u in range(t + 1):
                    s.append(c["scale"] * sum(qr[i] * K[b, u, g, i] for i in range(d)))
                m = max(s)
                e = [math.exp(x - m) for x in s]
                l = sum(e)
                for i in range(d):
                    v = 0.0
                    for j in range(N_b):
                        v += e[j] * sum(C_V[b, j, k] * U_V[g * d + i, k] for k in range(r_v))
                    for u in range(t + 1):
                        v += e[N_b + u] * V[b, u, g, i]
                    out[b, t, h, i] = v / l
    return out


def test_prefill_brute_force_scalar_loops():
    rng = np.random.default_rng(54)
    c = _prefill_case(rng, B=2, T=4, Hq=4, Hkv=2, d=4, N_b=3, r_k=3, r_v=2)
    np.testing.assert_allclose(oracle.prefill_attn(**c), _brute_prefill(c), rtol=1e-12, atol=1e-13)


def _mutated_prefill(old, new):
    """A copy of the oracle's prefill with one planted change in its source."""
    import inspect
    import textwrap
    src = textwrap.dedent(inspect.getsource(O.prefill_attn))
    assert src.count(old) >= 1
    ns = dict(vars(O))
    exec(compile(src.replace(old, new), "<mutated prefill>", "exec"), ns)
    return ns["prefill_attn"]


@pytest.mark.parametrize("old,new", [
    (":t + 1, g, :]", ":t, g, :]"),                         # token t does not see itself
    (":t + 1, g, :]", ":t + 2, g, :]"),                     # one token of the future leaks in
    ("float(p0[b]) + t", "float(p0[b])"),                   # every token rotated at p0
])
def test_pins_catch_prefill_mistakes(old, new):
    rng = np.random.default_rng(55)
    c = _prefill_case(rng, N_b=0, T=6)
    c["C_K"] = c["C_V"] = None
    ref = _causal_sdpa(_rotate_chunk_queries(c), _expand_heads(c["K_chunk"], 2),
                       _expand_heads(c["V_chunk"], 2), c["scale"])
    np.testing.assert_allclose(O.prefill_attn(**c), ref, rtol=1e-11, atol=1e-12)
    bad = _mutated_prefill(old, new)
    try:
        out = bad(**c)
    except ValueError:      # an empty score vector for t = 0 is caught too
        return
    assert not np.allclose(out, ref, atol=1e-6)

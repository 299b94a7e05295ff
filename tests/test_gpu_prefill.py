"""GPU parity of the prefill-side attention (a chunk over the beacon memory and,
causally, itself) against the float64 oracle's ``prefill_attn``.

Source: "Can SlimKV compress KV cache jointly across tokens and features", section
"Speedups are real, but memory is set by the ratio" (time-to-first-token gains from
skipping key-side RoPE and full-key materialisation for beacon states) and section
"Latent-space attention removes the rebuild step" (the latent scoring rule)."""
import numpy as np
import pytest
import torch

import oracle
from latent_kv_cache_decode_b300 import binding as bd
from latent_kv_cache_decode_b300 import workloads as wl
from tests.parity_util import assert_close, errors, row_errors, BF16_REL_L2, BF16_ROW_REL_L2, BF16_MAX_ABS

pytestmark = pytest.mark.gpu


def _inputs(w, T, layer=0, batch=None):
    t = wl.layer_tensors(w, layer, batch=batch)
    t.update(wl.prefill_chunk(w, layer, T, batch=batch))
    return t


def _gpu(w, t):
    d = {k: v.cuda() for k, v in t.items()}
    lat = w.N_b > 0
    o = bd.prefill_attn(d["q"], d["C_K"] if lat else None, d["C_V"] if lat else None, d["K_chunk"],
                        d["V_chunk"], d["U_K"] if lat else None, d["U_V"] if lat else None, d["p0"],
                        scale=w.scale, rope_base=w.rope_base)
    torch.cuda.synchronize()
    return o.cpu().double().numpy()


def _oracle(w, t, triples=None):
    f = {k: (wl.as_f64(v) if k != "p0" else v.numpy()) for k, v in t.items()}
    lat = w.N_b > 0
    return oracle.prefill_attn(f["q"], f["C_K"] if lat else None, f["C_V"] if lat else None, f["K_chunk"],
                               f["V_chunk"], f["U_K"], f["U_V"], f["p0"], w.scale, w.rope_base,
                               triples=triples)


CASES = {
    # ragged chunk (150 tokens: 600 query rows per KV group = 4 CTAs + a partial one),
    # ragged beacon count (200 = 3 tiles + 8 rows)
    "ragged": (dict(B=2, Hq=8, Hkv=2, N_b=200, rank=64, W=1, ratio=4), 150),
    "no-beacons": (dict(B=2, Hq=8, Hkv=2, N_b=0, rank=64, W=1, ratio=4), 100),
    "rank256-G8": (dict(B=1, Hq=16, Hkv=2, N_b=130, rank=256, W=1, ratio=8), 70),
    # G = 5: a CTA's 128 rows straddle token boundaries
    "G5-rank128": (dict(B=1, Hq=10, Hkv=2, N_b=64, rank=128, W=1, ratio=16), 77),
    "one-token": (dict(B=3, Hq=4, Hkv=2, N_b=96, rank=192, W=1, ratio=2), 1),
    # peaked chunk keys (1% of tokens x8), 2 chunk tiles per row block, many beacon tiles
    "peaked": (dict(B=1, Hq=8, Hkv=2, N_b=1024, rank=128, W=1, ratio=16, peak_frac=0.01,
                    peak_scale=8.0), 256),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_prefill_matches_oracle(name):
    kw, T = CASES[name]
    w = wl.custom(rope_base=500000.0, **kw)
    t = _inputs(w, T)
    assert_close(_gpu(w, t), _oracle(w, t), w.dtype, f"prefill {name}")


def test_prefill_is_causal_on_the_gpu():
    # changing the chunk's last tokens leaves every earlier query's output bit-identical
    w = wl.custom(B=1, Hq=8, Hkv=2, N_b=128, rank=64, W=1, ratio=4)
    t = _inputs(w, 130)
    a = _gpu(w, t)
    t2 = dict(t)
    t2["K_chunk"] = t["K_chunk"].clone()
    t2["V_chunk"] = t["V_chunk"].clone()
    t2["K_chunk"][:, 100:] *= 3
    t2["V_chunk"][:, 100:] += 1
    b = _gpu(w, t2)
    assert np.array_equal(a[:, :100], b[:, :100])
    assert not np.allclose(a[:, 100:], b[:, 100:])


def test_prefill_headline_chunk_sampled():
    # the benchmark's launch: a 1024-token chunk of every batch element of the
    # llama3.1-8b 128K / 16x layer (8192 beacons, rank 256, peaked chunk keys), checked
    # on sampled (b, t, h) against the oracle computed one by one
    w = wl.config(2)
    T = 1024
    t = _inputs(w, T)
    got = _gpu(w, t)
    assert np.all(np.isfinite(got))
    rng = np.random.default_rng(11)
    triples = [(int(b), int(tt), int(h)) for b, tt, h in
               zip(rng.integers(0, w.B, 48), rng.integers(0, T, 48), rng.integers(0, w.Hq, 48))]
    triples += [(0, 0, 0), (w.B - 1, T - 1, w.Hq - 1), (3, 511, 17), (5, 64, 31)]
    ref = _oracle(w, t, triples=triples)
    g = np.stack([got[b, tt, h] for b, tt, h in triples])
    r = np.stack([ref[b, tt, h] for b, tt, h in triples])
    rel, mx = errors(g, r)
    rows, worst = row_errors(g, r)
    assert rel <= BF16_REL_L2 and mx <= BF16_MAX_ABS, (rel, mx)
    assert rows[worst] <= BF16_ROW_REL_L2, (triples[worst], rows[worst])


def test_prefill_rejects_unsupported_shapes():
    dev = "cuda"
    q = torch.zeros(1, 4, 4, 128, dtype=torch.bfloat16, device=dev)
    kc = torch.zeros(1, 4, 1, 128, dtype=torch.bfloat16, device=dev)
    p0 = torch.zeros(1, dtype=torch.int32, device=dev)
    ck = torch.zeros(1, 64, 96, dtype=torch.bfloat16, device=dev)     # rank 96: not a multiple of 64
    u = torch.zeros(128, 96, dtype=torch.bfloat16, device=dev)
    with pytest.raises(bd.SlimkvError):
        bd.prefill_attn(q, ck, ck, kc, kc, u, u, p0)
    with pytest.raises(bd.SlimkvError):
        bd.prefill_attn(q.float(), None, None, kc.float(), kc.float(), None, None, p0)

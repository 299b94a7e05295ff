"""Multi-step decode on the GPU against the oracle: every step appends the new
token to the raw-window ring (slimkv_append_kv) and runs the layer's decode
(slimkv_decode_attn) at that token's position; the oracle does the same with
its own append. The loops run past the window length so that the ring wraps."""
import numpy as np
import pytest
import torch

import oracle
from latent_kv_cache_decode_b300 import binding as bd
from latent_kv_cache_decode_b300 import workloads as wl
from tests.parity_util import assert_close, f64, to_dev

pytestmark = pytest.mark.gpu

CASES = {
    # tensor-core path: bf16, d = 128; prompt positions 1024..1087 fill the 64 slots
    "bf16-tc": dict(B=2, Hq=8, Hkv=2, d=128, N_b=256, W=64, rank=64, ratio=4),
    # SIMT path: float32 storage, d = 64 (the tiny workload's shape)
    "f32-simt": dict(dtype="f32", B=1, Hq=4, Hkv=1, d=64, N_b=64, W=32, rank=32, ratio=32),
    # raw window only (no beacons), tensor-core path
    "bf16-window-only": dict(B=1, Hq=8, Hkv=2, d=128, N_b=0, W=32, rank=64, ratio=4),
    # the headline shape per batch element (32 / 8 heads, rank 256, 16x) with its peaked
    # raw keys (1% of the window's tokens scaled x8 before RoPE), two batch elements
    "bf16-headline-peaked": dict(B=2, Hq=32, Hkv=8, d=128, N_b=512, W=256, rank=256, ratio=16,
                                 peak_frac=0.01, peak_scale=8.0),
    # ALiBi through the ring wrap: the window positions follow the appends
    "bf16-tc-alibi": dict(B=2, Hq=8, Hkv=2, d=128, N_b=256, W=64, rank=64, ratio=4),
    "f32-simt-alibi": dict(dtype="f32", B=1, Hq=4, Hkv=1, d=64, N_b=64, W=32, rank=32, ratio=32),
}


@pytest.mark.parametrize("case", list(CASES))
def test_decode_loop_matches_oracle(case):
    bd.load()
    w = wl.custom(**CASES[case])
    steps = w.W + 5
    t = wl.layer_tensors(w, 0)
    st = wl.decode_steps(w, 0, steps)
    dev = to_dev(t)
    K, V = dev["K_raw"].clone(), dev["V_raw"].clone()
    f = f64(t)
    Ko, Vo = f["K_raw"], f["V_raw"]
    lat = w.N_b > 0
    alibi = case.endswith("-alibi")
    slopes = bd.alibi_slopes(w.Hq)
    for s in range(steps):
        pos = st["pos"][s]
        pd = pos.cuda()
        bd.append_kv(st["k_new"][s].cuda(), st["v_new"][s].cuda(), K, V, pd, rope_base=w.rope_base)
        if alibi:
            got = bd.decode_attn_alibi(st["q"][s].cuda(), dev["C_K"], dev["C_V"], K, V, dev["U_K"], dev["U_V"], pd,
                                       slopes, w.ratio, scale=w.scale, rope_base=w.rope_base)
        else:
            got = bd.decode_attn(st["q"][s].cuda(), dev["C_K"] if lat else None, dev["C_V"] if lat else None,
                                 K, V, dev["U_K"] if lat else None, dev["U_V"] if lat else None, pd,
                                 scale=w.scale, rope_base=w.rope_base)
        torch.cuda.synchronize()
        Ko, Vo = oracle.append_kv(Ko, Vo, wl.as_f64(st["k_new"][s]), wl.as_f64(st["v_new"][s]), pos.numpy(),
                                  w.rope_base, storage=w.dtype)
        if alibi:
            ref = oracle.decode_attn_alibi(wl.as_f64(st["q"][s]), f["C_K"], f["C_V"], Ko, Vo, f["U_K"], f["U_V"],
                                           pos.numpy(), w.scale, w.rope_base, np.array(slopes), w.ratio)
        else:
            ref = oracle.decode_attn(wl.as_f64(st["q"][s]), f["C_K"] if lat else None, f["C_V"] if lat else None,
                                     Ko, Vo, f["U_K"], f["U_V"], pos.numpy(), w.scale, w.rope_base)
        assert_close(got.cpu().double().numpy(), ref, w.dtype, f"{case} step {s}")
    # the window after the loop: values copied exactly, keys rotated in float32
    # then rounded to the storage type (the oracle rotates in float64)
    assert torch.equal(V.cpu().to(torch.float64), torch.from_numpy(Vo))
    Kg = K.cpu().double().numpy()
    tol = 2.0 ** -7 if w.dtype == "bf16" else 1e-6
    assert np.allclose(Kg, Ko, rtol=tol, atol=1e-6), np.abs(Kg - Ko).max()
    if w.dtype == "bf16":
        # nearly every key element rounds to the same bf16 value on both sides
        assert np.mean(Kg == Ko) > 0.999


def test_append_rejects_bad_arguments():
    bd.load()
    w = wl.custom(B=1, Hq=8, Hkv=2, d=128, N_b=0, W=16, rank=64, ratio=4)
    t = to_dev(wl.layer_tensors(w, 0))
    kn = torch.zeros((1, 2, 128), dtype=torch.bfloat16, device="cuda")
    pos = torch.zeros((1,), dtype=torch.int32, device="cuda")
    with pytest.raises(bd.SlimkvError) as e:
        bd.append_kv(kn, kn, t["K_raw"][:, :0].contiguous(), t["V_raw"][:, :0].contiguous(), pos)
    assert e.value.status in (1, 2)   # an empty window: no pointer / W = 0

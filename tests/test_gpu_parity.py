"""GPU vs float64 oracle on the same seeded inputs, through the C ABI.

Small cases are compared element by element; the full-size workloads are
compared on whole layers (the oracle handles one 128K/16x layer in seconds) and,
for the 128K full-KV cache, on sampled batch elements.
"""
import numpy as np
import pytest
import torch

from latent_kv_cache_decode_b300 import binding as bd
from latent_kv_cache_decode_b300 import workloads as wl
from tests.parity_util import assert_close, run_gpu, run_oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    bd.load()
    prev = bd.force_simt(False)
    yield
    bd.force_simt(prev)


@pytest.mark.parametrize("which", ["latent", "reconstruct"])
def test_config0_fp32(which):
    w = wl.config(0)
    t = wl.layer_tensors(w, 0)
    got = run_gpu(which, w, t)
    ref = run_oracle(which, w, t)
    assert_close(got, ref, "f32", f"config0 {which}")


def test_config0_fp32_full_kv():
    # the config-0 window as a full cache of RoPE'd keys
    w = wl.config(0)
    t = wl.layer_tensors(w, 0)
    t["K_full"], t["V_full"] = t["K_raw"], t["V_raw"]
    assert_close(run_gpu("full", w, t), run_oracle("full", w, t), "f32", "config0 full-kv")


def test_config0_against_stored_golden():
    import os
    w = wl.config(0)
    got = run_gpu("latent", w, wl.layer_tensors(w, 0))
    gold = np.loadtxt(os.path.join(os.path.dirname(__file__), "golden", "config0_latent_out.txt"))
    assert np.abs(got.reshape(gold.shape) - gold).max() <= 1e-5


def test_config1_one_layer():
    w = wl.config(1)
    t = wl.layer_tensors(w, 3)
    assert_close(run_gpu("latent", w, t), run_oracle("latent", w, t), "bf16", "config1 layer3")


def test_config2_full_layer():
    # 128K context, 16x, batch 8: the bench's headline workload, one whole layer
    w = wl.config(2)
    t = wl.layer_tensors(w, 0)
    assert_close(run_gpu("latent", w, t), run_oracle("latent", w, t), "bf16", "config2 layer0")


@pytest.mark.parametrize("layer", [0, 1, 2])
def test_config3_variable_rank_layers(layer):
    w = wl.config(3)
    # pick the layers with the smallest, largest and a middle rank
    order = sorted(range(w.layers), key=lambda i: w.ranks[i])
    L = [order[0], order[-1], order[len(order) // 2]][layer]
    t = wl.layer_tensors(w, L)
    assert_close(run_gpu("latent", w, t), run_oracle("latent", w, t), "bf16",
                 f"config3 layer{L} rank{w.ranks[L]}")


def test_config4_reconstruct_equals_oracle_and_latent():
    w = wl.config(4)
    t = wl.layer_tensors(w, 0)
    rec = run_gpu("reconstruct", w, t)
    lat = run_gpu("latent", w, t)
    ref = run_oracle("latent", w, t)
    assert_close(rec, ref, "bf16", "config4 reconstruct")
    assert_close(lat, ref, "bf16", "config4 latent")


def test_config4_full_kv_sampled():
    # [8, 131072, 8, 128] bf16 cache; the oracle checks batch elements 0 and 7, each
    # regenerated alone (the generator gives every batch element its own stream)
    w = wl.config(4)
    t = wl.layer_tensors(w, 0, with_full=True)
    got = run_gpu("full", w, t)
    del t
    for b in (0, 7):
        tb = wl.layer_tensors(w, 0, batch=[b], with_full=True)
        ref = run_oracle("full", w, tb)
        assert_close(got[b:b + 1], ref, "bf16", f"config4 full-kv b{b}")


EDGE = [
    dict(name="window-only", N_b=0, W=300),
    dict(name="beacons-only", N_b=300, W=0),
    dict(name="one-window-token", N_b=128, W=1),
    dict(name="ragged", N_b=333, W=77, B=3),
    dict(name="rank32", N_b=256, W=64, rank=32),
    dict(name="rank512", Hq=16, Hkv=4, N_b=200, W=50, rank=512),
    dict(name="mha", Hq=8, Hkv=8, N_b=150, W=40),
    dict(name="group5", Hq=40, Hkv=8, N_b=256, W=128),
    dict(name="mqa", Hq=16, Hkv=1, N_b=256, W=128),
    dict(name="d64-bf16", d=64, Hq=8, Hkv=2, N_b=130, W=70, rank=64),
    dict(name="big-heads", Hq=64, Hkv=8, N_b=200, W=100),
    # latent ranks above 256: a key or value tile part fills the whole ring
    dict(name="rank320", Hq=32, Hkv=8, N_b=300, W=90, rank=320),
    dict(name="rank512-g5", Hq=40, Hkv=8, N_b=300, W=100, rank=512),
    dict(name="rank512-64heads", Hq=64, Hkv=8, N_b=200, W=60, rank=512),
]


@pytest.mark.parametrize("Hq,rank", [(32, 320), (40, 384), (40, 512), (48, 512), (64, 512)])
def test_large_ranks_take_the_tensor_core_path(Hq, rank):
    # (64 heads at rank 512: a 64 KB query image, so the kernel runs with one P buffer
    # to keep four ring slots)
    w = wl.custom(Hq=Hq, Hkv=8, N_b=256, W=128, rank=rank)
    sh = bd.make_shape(w.B, w.Hq, w.Hkv, w.d, w.N_b, rank, rank, w.W, torch.bfloat16)
    assert bd.kernel_path(sh, bd.SLIMKV_LATENT) == 1


@pytest.mark.parametrize("which,path", [("latent", 1), ("full", 1), ("reconstruct", 0)])
def test_d64_paths(which, path):
    # bf16 with d = 64: the decode and full-KV attention run on the tensor cores with
    # zero-padded 128-column raw tiles; the reconstruction baselines stay on the SIMT path
    sh = bd.make_shape(2, 8, 2, 64, 0 if which == "full" else 128, 64, 64, 96, torch.bfloat16)
    code = {"latent": bd.SLIMKV_LATENT, "full": bd.SLIMKV_FULL_KV, "reconstruct": bd.SLIMKV_RECONSTRUCT}[which]
    assert bd.kernel_path(sh, code) == path


@pytest.mark.parametrize("case", [
    dict(B=3, Hq=8, Hkv=2, N_b=300, W=200, rank=128),        # several tiles and ragged ends
    dict(B=1, Hq=40, Hkv=8, N_b=256, W=129, rank=256),       # G = 5, rank 256
    dict(B=2, Hq=16, Hkv=2, N_b=0, W=600, rank=64),          # window only (3 raw tiles per head)
])
def test_d64_tensor_core_decode_matches_oracle(case):
    w = wl.custom(d=64, **case)
    t = wl.layer_tensors(w, 0)
    assert_close(run_gpu("latent", w, t), run_oracle("latent", w, t), w.dtype, f"d64 {case}")


@pytest.mark.parametrize("case", EDGE, ids=[c["name"] for c in EDGE])
@pytest.mark.parametrize("which", ["latent", "reconstruct", "full"])
def test_edge_cases(case, which):
    kw = {k: v for k, v in case.items() if k != "name"}
    w = wl.custom(**kw)
    if which == "reconstruct" and w.N_b == 0:
        pytest.skip("reconstruction needs beacons")
    t = wl.layer_tensors(w, 0)
    if which == "full":
        if w.W == 0:
            pytest.skip("full-KV needs a cache")
        t["K_full"], t["V_full"] = t["K_raw"], t["V_raw"]
    assert_close(run_gpu(which, w, t), run_oracle(which, w, t), w.dtype, f"{case['name']} {which}")


@pytest.mark.parametrize("case", [dict(N_b=333, W=77, B=2), dict(N_b=1024, W=256, B=2, Hq=40),
                                  dict(N_b=4096, W=1024, Hq=32, rank=256)])
def test_simt_and_tensor_core_paths_agree(case):
    w = wl.custom(**case)
    t = wl.layer_tensors(w, 0)
    a = run_gpu("latent", w, t)
    prev = bd.force_simt(True)
    try:
        b = run_gpu("latent", w, t)
    finally:
        bd.force_simt(prev)
    ref = run_oracle("latent", w, t)
    assert_close(a, ref, "bf16", "auto path")
    assert_close(b, ref, "bf16", "simt path")


def test_repeated_calls_reuse_workspace():
    w = wl.custom(B=2, N_b=500, W=200)
    t = wl.layer_tensors(w, 0)
    d = {k: v.cuda() for k, v in t.items()}
    ws = bd.Workspace()
    outs = []
    for _ in range(3):
        outs.append(bd.decode_attn(d["q"], d["C_K"], d["C_V"], d["K_raw"], d["V_raw"], d["U_K"],
                                   d["U_V"], d["q_pos"], scale=w.scale, rope_base=w.rope_base,
                                   workspace=ws).cpu())
    torch.cuda.synchronize()
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[1], outs[2])


# The reconstruction baseline that keeps beacon-key RoPE: tensor-core path (the rotation
# in the GEMM's write-out), and the SIMT path (float32 storage, or d = 64).
@pytest.mark.parametrize("case", [
    ("config0-f32", None),
    ("bf16-tc", dict(B=2, Hq=8, Hkv=2, d=128, N_b=256, W=64, rank=64, ratio=4)),
    ("bf16-tc-rank320", dict(B=1, Hq=8, Hkv=4, d=128, N_b=300, W=40, rank=320, ratio=16)),
    ("bf16-simt-d64", dict(B=2, Hq=4, Hkv=1, d=64, N_b=96, W=32, rank=64, ratio=8)),
])
def test_reconstruct_rope_matches_oracle(case):
    name, kw = case
    w = wl.config(0) if kw is None else wl.custom(**kw)
    t = wl.layer_tensors(w, 0)
    got = run_gpu("reconstruct_rope", w, t)
    ref = run_oracle("reconstruct_rope", w, t)
    assert_close(got, ref, w.dtype, f"reconstruct-rope {name}")


def test_config1_reconstruct_rope_one_layer():
    # beacon positions up to 4095 * 8 + 7 at the 32K context of config 1
    w = wl.config(1)
    t = wl.layer_tensors(w, 1)
    assert_close(run_gpu("reconstruct_rope", w, t), run_oracle("reconstruct_rope", w, t), "bf16",
                 "config1 reconstruct-rope")


# ALiBi on the reconstruction-free decode (tensor-core path for bf16, d = 128 or 64; SIMT
# path for float32 storage), with the slopes of bd.alibi_slopes.
@pytest.mark.parametrize("case", [
    ("config0-f32", None),
    ("bf16-tc", dict(B=2, Hq=8, Hkv=2, d=128, N_b=256, W=64, rank=64, ratio=4)),
    ("bf16-headline-shape", dict(B=2, Hq=32, Hkv=8, d=128, N_b=512, W=256, rank=256, ratio=16)),
    ("bf16-window-only", dict(B=1, Hq=8, Hkv=2, d=128, N_b=0, W=300, rank=64, ratio=4)),
    ("bf16-beacons-only", dict(B=1, Hq=8, Hkv=2, d=128, N_b=300, W=0, rank=64, ratio=8)),
    ("bf16-d64", dict(B=2, Hq=4, Hkv=1, d=64, N_b=96, W=32, rank=64, ratio=8)),
    ("bf16-d64-window-only", dict(B=1, Hq=8, Hkv=2, d=64, N_b=0, W=300, rank=64, ratio=4)),
])
def test_alibi_matches_oracle(case):
    name, kw = case
    w = wl.config(0) if kw is None else wl.custom(**kw)
    t = wl.layer_tensors(w, 0)
    assert_close(run_gpu("alibi", w, t), run_oracle("alibi", w, t), w.dtype, f"alibi {name}")

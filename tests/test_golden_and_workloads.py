"""Stored oracle outputs and the seeded workload recipes (CPU only)."""
import os

import numpy as np
import torch

from latent_kv_cache_decode_b300 import workloads as wl

HERE = os.path.dirname(os.path.abspath(__file__))


def test_golden_config0_matches_oracle():
    from tests.golden.make_golden import config0_arrays
    lat, rec = config0_arrays()
    g_lat = np.loadtxt(os.path.join(HERE, "golden", "config0_latent_out.txt"))
    g_rec = np.loadtxt(os.path.join(HERE, "golden", "config0_reconstruct_out.txt"))
    np.testing.assert_allclose(lat.reshape(g_lat.shape), g_lat, rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(rec.reshape(g_rec.shape), g_rec, rtol=1e-14, atol=1e-15)
    # the two formulations agree to float64 rounding
    np.testing.assert_allclose(lat, rec, rtol=1e-11, atol=1e-12)


def test_golden_prefill_matches_oracle():
    from tests.golden.make_golden import prefill_arrays
    pre = prefill_arrays()
    g = np.loadtxt(os.path.join(HERE, "golden", "config0_prefill_out.txt"))
    np.testing.assert_allclose(pre.reshape(g.shape), g, rtol=1e-14, atol=1e-15)


def test_config_shapes_and_positions():
    c1, c2, c3 = wl.config(1), wl.config(2), wl.config(3)
    assert (c1.B, c1.Hq, c1.Hkv, c1.d, c1.N_b, c1.rank, c1.W, c1.layers) == (1, 32, 8, 128, 4096, 256, 1024, 32)
    assert (c2.B, c2.N_b, c2.W, c2.q_pos) == (8, 8192, 2048, 8192 * 16 + 2048)
    assert wl.config(0).q_pos == 2080
    # 4 GiB of cache per 32-layer step at 128K / 16x
    assert sum(wl.cache_bytes(c2, l) for l in range(c2.layers)) == 4 << 30
    assert (c3.Hq, c3.Hkv, c3.layers) == (40, 8, 48)


def test_qwen_ranks_recipe():
    r = wl.config(3).ranks
    assert len(r) == 48
    assert all(x % 32 == 0 and 128 <= x <= 512 for x in r)
    assert sum(r) == 48 * 256
    assert r == wl._qwen_ranks(3, 48)          # deterministic


def test_layer_tensors_deterministic_and_sliceable():
    w = wl.custom(B=3, N_b=40, W=24, rank=32, Hq=4, Hkv=2, d=64)
    a = wl.layer_tensors(w, 0)
    b = wl.layer_tensors(w, 0, batch=[2])
    for k in ("C_K", "C_V", "K_raw", "V_raw", "q"):
        assert a[k].shape[0] == 3
        assert bool((a[k][2:3] == b[k]).all())
    assert bool((a["U_K"] == b["U_K"]).all())
    u = wl.as_f64(a["U_K"])
    # bf16-rounded orthonormal columns stay orthonormal to bf16 accuracy
    assert np.abs(u.T @ u - np.eye(u.shape[1])).max() < 2e-2


def test_peaked_keys_fraction():
    w = wl.custom(B=1, W=2000, N_b=0, rank=32, peak_frac=0.01, peak_scale=8.0, dtype="f32")
    k = wl.as_f64(wl.layer_tensors(w, 0)["K_raw"])[0]
    norms = np.linalg.norm(k.reshape(2000, -1), axis=1)
    big = norms > 4 * np.median(norms)
    assert big.sum() == 20


def test_decode_steps_are_seeded_per_batch_element():
    w = wl.custom(B=3, Hq=8, Hkv=2, d=128, N_b=64, W=32, rank=64, ratio=4)
    a = wl.decode_steps(w, 1, 4)
    b = wl.decode_steps(w, 1, 4)
    assert a["k_new"].shape == (4, 3, 2, 128) and a["q"].shape == (4, 3, 8, 128)
    assert all(torch.equal(a[k], b[k]) for k in a)                   # deterministic
    sub = wl.decode_steps(w, 1, 4, batch=[2])                         # a batch element alone
    assert torch.equal(sub["k_new"][:, 0], a["k_new"][:, 2]) and torch.equal(sub["q"][:, 0], a["q"][:, 2])
    assert not torch.equal(wl.decode_steps(w, 2, 4)["k_new"], a["k_new"])   # layers differ
    assert a["pos"].dtype == torch.int32
    assert a["pos"][:, 0].tolist() == [w.q_pos + s for s in range(4)]


def test_bench_traffic_guard(tmp_path, monkeypatch):
    # the recorded DRAM traffic is used only for its workload and while the kernel
    # sources hash as recorded (checked on a record written here, so that the test
    # does not depend on the committed capture being current)
    import hashlib
    import json
    import shutil
    import bench
    rels = ["latent_kv_cache_decode_b300/csrc/tc_decode.cu", "latent_kv_cache_decode_b300/csrc/tc_ptx.cuh"]
    for rel in rels:
        os.makedirs(os.path.dirname(tmp_path / rel), exist_ok=True)
        shutil.copy(os.path.join(bench.ROOT, rel), tmp_path / rel)
    w = wl.config(2)
    rec = {"workload": w.name + ", one layer", "dram_bytes_read_per_launch": 100,
           "dram_bytes_write_per_launch": 20,
           "source_sha256": {rel: hashlib.sha256(open(tmp_path / rel, "rb").read()).hexdigest() for rel in rels}}
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "tc_decode_traffic.json").write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench._measured_traffic(w, "latent") == 120
    assert bench._measured_traffic(w, "full") is None
    assert bench._measured_traffic(wl.config(1), "latent") is None
    (tmp_path / rels[0]).write_bytes(open(tmp_path / rels[0], "rb").read() + b"// changed\n")
    assert bench._measured_traffic(w, "latent") is None


def _bench_reference(env_extra):
    import json
    import subprocess
    import sys
    root = os.path.dirname(HERE)
    env = dict(os.environ, **env_extra)
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference", "--config", "0",
                        "--steps", "1", "--warmup", "3"], cwd=root, env=env, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    return [json.loads(l) for l in lines]


def test_bench_reference_arm_line():
    # the reference arm times the float64 oracle on the host and prints one JSON line
    # with the contract's keys, its own metric and an end-to-end record without copies
    (line,) = _bench_reference({})
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "impl", "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference" and line["higher_is_better"] is False
    assert line["value"] > 0 and line["warmup"] >= 3 and line["dtype"] == "f64"
    assert line["config"]["workload"] == wl.config(0).name
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == line["value"] and cb["sample"]
    e2e = line["e2e"]
    assert e2e["value"] == line["value"] and e2e["unit"] == line["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_bench_reference_arm_other_ranks_print_nothing():
    assert _bench_reference({"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"}) == []

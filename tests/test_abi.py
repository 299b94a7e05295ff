"""C-ABI checks that need no GPU: the library loads, exports every symbol the
header declares, sizes workspaces, and rejects bad arguments before any launch."""
import ctypes
import os
import re

import pytest

from latent_kv_cache_decode_b300 import binding as bd

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _header_functions():
    names = []
    for fn in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names += re.findall(r"\b(slimkv_[a-z0-9_]+)\s*\(", src)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    from latent_kv_cache_decode_b300 import build
    build.build()
    return bd.load()


def test_exports_every_declared_symbol(lib):
    declared = _header_functions()
    assert set(bd.EXPORTS) == set(declared), declared
    for name in declared:
        assert hasattr(lib, name), name


def test_abi_version_and_status_strings(lib):
    assert lib.slimkv_abi_version() == 4
    for code, name in bd.STATUS.items():
        s = lib.slimkv_status_str(code)
        assert isinstance(s, bytes) and len(s) > 0
    assert lib.slimkv_status_str(99) == b"unknown status"


def _shape(**kw):
    base = dict(B=8, Hq=32, Hkv=8, d=128, N_b=8192, r_k=256, r_v=256, W=2048, dtype=bd.SLIMKV_BF16,
                scale=0.08838834764831845, rope_base=500000.0)
    base.update(kw)
    return bd.make_shape(**base)


def test_workspace_sizes(lib):
    s = _shape()
    lat = bd.workspace_bytes(s, bd.SLIMKV_LATENT)
    rec = bd.workspace_bytes(s, bd.SLIMKV_RECONSTRUCT)
    assert lat > 0 and lat % 256 == 0
    # reconstruct also holds K_b and V_b: 2 * B * N_b * Hkv * d bf16
    assert rec >= 2 * 8 * 8192 * 8 * 128 * 2
    full = bd.workspace_bytes(_shape(N_b=0, W=131072), bd.SLIMKV_FULL_KV)
    assert full > 0
    assert bd.workspace_bytes(_shape(N_b=5), bd.SLIMKV_FULL_KV) == 0       # full-KV needs N_b == 0


@pytest.mark.parametrize("bad", [dict(Hq=30), dict(d=96), dict(r_k=48), dict(r_v=544), dict(B=0),
                                 dict(B=257), dict(N_b=0, W=0), dict(N_b=-1), dict(Hq=256, Hkv=8),
                                 dict(scale=float("inf")), dict(rope_base=0.0), dict(r_k=0)])
def test_invalid_shapes_rejected(lib, bad):
    s = _shape(**bad)
    assert bd.workspace_bytes(s, bd.SLIMKV_LATENT) == 0
    assert bd.kernel_path(s, bd.SLIMKV_LATENT) == -1
    st = lib.slimkv_decode_attn(ctypes.byref(s), *([256] * 7), 256, 256, 256, 1 << 40, None)
    assert st == 2


def test_bad_dtype(lib):
    s = _shape(dtype=7)
    st = lib.slimkv_decode_attn(ctypes.byref(s), *([256] * 7), 256, 256, 256, 1 << 40, None)
    assert st == 3


def _call(lib, s, ptrs, ws_bytes, fn="slimkv_decode_attn"):
    return getattr(lib, fn)(ctypes.byref(s), *ptrs, ws_bytes, None)


def test_null_misaligned_and_small_workspace_rejected(lib):
    s = _shape()
    good = [256 * (i + 1) for i in range(7)] + [4096, 8192, 1 << 20]   # 7 tensors, q_pos, out, ws
    need = bd.workspace_bytes(s, bd.SLIMKV_LATENT)
    for i in range(10):                                   # each required pointer NULL in turn
        p = list(good)
        p[i] = None
        assert _call(lib, s, p, need) == 1
    for i in range(7):                                    # each tensor 8-byte aligned only
        p = list(good)
        p[i] += 8
        assert _call(lib, s, p, need) == 4
    p = list(good)
    p[9] += 16                                            # workspace not 256-byte aligned
    assert _call(lib, s, p, need) == 4
    assert _call(lib, s, good, need - 1) == 5             # workspace one byte short
    # full-KV: 7 pointer arguments (q, K, V, q_pos, out, ws)
    sf = _shape(N_b=0, W=4096)
    needf = bd.workspace_bytes(sf, bd.SLIMKV_FULL_KV)
    st = lib.slimkv_decode_attn_full_kv(ctypes.byref(sf), 256, 512, None, 4096, 8192, 1 << 20,
                                        needf, None)
    assert st == 1
    st = lib.slimkv_decode_attn_full_kv(ctypes.byref(sf), 256, 512, 768, 4096, 8192, 1 << 20,
                                        needf - 256, None)
    assert st == 5
    # reconstruct requires beacons
    sr = _shape(N_b=0)
    assert _call(lib, sr, good, 1 << 40, "slimkv_decode_attn_reconstruct") == 2


def test_noalloc_host_checks(lib):
    # oversized shapes and bad shapes are rejected before any device work
    big = _shape(B=256, Hq=128, r_k=512, r_v=512)
    assert bd.workspace_bytes(big, bd.SLIMKV_LATENT) > bd.NOALLOC_SCRATCH_BYTES
    p = [256 * (i + 1) for i in range(7)] + [4096, 8192]
    assert lib.slimkv_decode_attn_noalloc(ctypes.byref(big), *p, None) == 7
    assert lib.slimkv_decode_attn_noalloc(ctypes.byref(_shape(Hq=30)), *p, None) == 2
    assert lib.slimkv_decode_attn_noalloc(None, *p, None) == 1
    assert lib.slimkv_status_str(7) != b"unknown status"


def test_unused_operands_may_be_null(lib):
    # W == 0: K_raw/V_raw may be NULL; N_b == 0: C_K, C_V, U_K, U_V may be NULL.
    # A too-small workspace is then the first error reported (nothing launches).
    s = _shape(W=0)
    p = [256, 512, 768, None, None, 1024, 1280, 4096, 8192, 1 << 20]
    assert _call(lib, s, p, 256) == 5
    s = _shape(N_b=0)
    p = [256, None, None, 768, 1024, None, None, 4096, 8192, 1 << 20]
    assert _call(lib, s, p, 256) == 5


def test_append_kv_host_checks(lib):
    # slimkv_append_kv rejects NULL, bad shapes and misaligned pointers before any launch
    s = _shape(W=64)
    good = [256, 512, 1024, 2048, 4096]                   # k_new, v_new, K_raw, V_raw, pos
    for i in range(5):
        p = list(good)
        p[i] = None
        assert lib.slimkv_append_kv(ctypes.byref(s), *p, None) == 1
    assert lib.slimkv_append_kv(None, *good, None) == 1
    for bad in (dict(W=0), dict(d=96), dict(B=0), dict(Hkv=0), dict(rope_base=-1.0), dict(W=1 << 25)):
        assert lib.slimkv_append_kv(ctypes.byref(_shape(**bad)), *good, None) == 2, bad
    assert lib.slimkv_append_kv(ctypes.byref(_shape(dtype=5)), *good, None) == 3
    for i in range(4):                                    # tensors 8-byte aligned only
        p = list(good)
        p[i] += 8
        assert lib.slimkv_append_kv(ctypes.byref(s), *p, None) == 4
    p = list(good)
    p[4] += 2                                             # positions not 4-byte aligned
    assert lib.slimkv_append_kv(ctypes.byref(s), *p, None) == 4


def test_plain_c_consumer(lib, tmp_path):
    # the header is plain C: a C99 program compiles against it, links the library and
    # runs the host-side checks
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc not available")
    so_dir = os.path.join(ROOT, "latent_kv_cache_decode_b300")
    exe = tmp_path / "abi_c_check"
    subprocess.run([gcc, "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                    os.path.join(ROOT, "tests", "native", "abi_c_check.c"), "-L", so_dir, "-lslimkv",
                    "-Wl,-rpath," + so_dir, "-o", str(exe)], check=True, capture_output=True, text=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "c abi ok" in r.stdout


def test_reconstruct_rope_host_checks(lib):
    # a beacon ratio below 1 is rejected before any launch; otherwise the checks of the
    # plain reconstruction apply (here: a workspace one byte short, a NULL pointer)
    s = _shape()
    good = [256 * (i + 1) for i in range(7)] + [4096]
    need = bd.workspace_bytes(s, bd.SLIMKV_RECONSTRUCT)
    fn = lib.slimkv_decode_attn_reconstruct_rope
    for bad_ratio in (0, -3):
        assert fn(ctypes.byref(s), *good, bad_ratio, 8192, 1 << 20, need, None) == 2
    assert fn(ctypes.byref(s), *good, 16, 8192, 1 << 20, need - 1, None) == 5
    nul = list(good)
    nul[1] = None
    assert fn(ctypes.byref(s), *nul, 16, 8192, 1 << 20, need, None) == 1
    assert fn(ctypes.byref(_shape(N_b=0)), *good, 16, 8192, 1 << 20, 1 << 40, None) == 2


def test_alibi_host_checks(lib):
    # slopes are required and finite, the beacon ratio >= 1; nothing launches
    s = _shape()
    good = [256 * (i + 1) for i in range(7)] + [4096]
    need = bd.workspace_bytes(s, bd.SLIMKV_LATENT)
    fn = lib.slimkv_decode_attn_alibi
    sl = (ctypes.c_float * s.Hq)(*([0.25] * s.Hq))
    slp = ctypes.cast(sl, ctypes.c_void_p)
    assert fn(ctypes.byref(s), *good, None, 16, 8192, 1 << 20, need, None) == 1
    assert fn(ctypes.byref(s), *good, slp, 0, 8192, 1 << 20, need, None) == 2
    bad = (ctypes.c_float * s.Hq)(*([0.25] * (s.Hq - 1) + [float("inf")]))
    assert fn(ctypes.byref(s), *good, ctypes.cast(bad, ctypes.c_void_p), 16, 8192, 1 << 20, need, None) == 2
    assert fn(ctypes.byref(s), *good, slp, 16, 8192, 1 << 20, need - 1, None) == 5


def test_alibi_slopes_follow_the_geometric_rule():
    assert bd.alibi_slopes(8) == [2.0 ** (-i) for i in range(1, 9)]
    s12 = bd.alibi_slopes(12)
    assert s12[:8] == bd.alibi_slopes(8) and s12[8:] == bd.alibi_slopes(16)[0::2][:4]


# ---------------------------------------------------------------- prefill (no launch)

def test_prefill_workspace_is_the_staged_queries(lib):
    # [B, Hkv, rows_pad, 2 d] bf16 with rows_pad = T * G rounded up to 128
    s = _shape(W=1024)
    assert bd.workspace_bytes(s, bd.SLIMKV_PREFILL) == 8 * 8 * 4096 * 256 * 2
    s = _shape(B=1, Hq=10, Hkv=2, N_b=64, r_k=128, r_v=128, W=77)      # 385 rows -> 512
    assert bd.workspace_bytes(s, bd.SLIMKV_PREFILL) == 1 * 2 * 512 * 256 * 2
    assert bd.workspace_bytes(_shape(N_b=0, W=100), bd.SLIMKV_PREFILL) > 0     # no beacons


@pytest.mark.parametrize("bad", [dict(dtype=bd.SLIMKV_F32), dict(d=64), dict(r_k=96), dict(r_v=320),
                                 dict(W=0), dict(Hq=30), dict(W=1 << 24, Hq=64)])
def test_prefill_rejects_unsupported_shapes(lib, bad):
    s = _shape(**bad)
    assert bd.workspace_bytes(s, bd.SLIMKV_PREFILL) == 0
    st = lib.slimkv_prefill_attn(ctypes.byref(s), *([256] * 7), 256, 256, 256, 1 << 40, None)
    assert st == 2


def test_prefill_rejects_null_and_misaligned_pointers(lib):
    s = _shape(W=64)
    ok = [256] * 7
    assert lib.slimkv_prefill_attn(ctypes.byref(s), *ok, None, 256, 256, 1 << 40, None) == 1     # p0
    assert lib.slimkv_prefill_attn(ctypes.byref(s), None, *ok[1:], 256, 256, 256, 1 << 40, None) == 1
    bad = list(ok)
    bad[3] = 264                                                                                 # K_chunk
    assert lib.slimkv_prefill_attn(ctypes.byref(s), *bad, 256, 256, 256, 1 << 40, None) == 4
    assert lib.slimkv_prefill_attn(ctypes.byref(s), *ok, 256, 256, 256, 16, None) == 5           # workspace


def test_abort_count_without_a_device_reports_an_error(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("needs a host without a GPU")
    assert lib.slimkv_abort_count(0) == -1

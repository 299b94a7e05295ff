"""slimkv_decode_attn_noalloc: the decode call for callers that cannot allocate
device memory (an engine that owns all of HBM through its own pool, a plain C caller
with no device allocator, a decode loop where cudaMalloc is not allowed). Its scratch
is a fixed device array inside the library, so the call takes no workspace.

Checked through the C ABI against slimkv_decode_attn (same inputs, caller-allocated
workspace) on two calls in a row with different inputs: the second call must not be
affected by what the first left in the shared array. Both entry points run the same
kernels with the same plan, so their outputs are compared bit for bit, and both are
compared with the float64 oracle. A large call followed by a small one checks that the
small call reads nothing the large one left behind: its reference runs on a fresh
workspace filled with NaN bytes. Collected last on purpose.
"""
import ctypes
import dataclasses

import pytest
import torch

from latent_kv_cache_decode_b300 import binding as bd
from latent_kv_cache_decode_b300 import workloads as wl
from tests.parity_util import assert_close, run_oracle, to_dev

pytestmark = pytest.mark.gpu


def _shape(w, layer=0):
    r = w.r(layer)
    return bd.make_shape(w.B, w.Hq, w.Hkv, w.d, w.N_b, r, r, w.W,
                         bd.SLIMKV_F32 if w.dtype == "f32" else bd.SLIMKV_BF16,
                         w.scale, w.rope_base)


def _noalloc_call(lib, sh, t, out):
    stream = torch.cuda.current_stream().cuda_stream
    return lib.slimkv_decode_attn_noalloc(
        ctypes.byref(sh), t["q"].data_ptr(), t["C_K"].data_ptr(), t["C_V"].data_ptr(),
        t["K_raw"].data_ptr(), t["V_raw"].data_ptr(), t["U_K"].data_ptr(), t["U_V"].data_ptr(),
        t["q_pos"].data_ptr(), out.data_ptr(), stream)


def _with_workspace(w, t, nan_fill=False):
    ws = bd.Workspace(torch.device("cuda", 0))
    if nan_fill:
        nb = bd.workspace_bytes(_shape(w), bd.SLIMKV_LATENT)
        ws.get(nb).fill_(0xFF)                   # every float32 word reads as NaN
    return bd.decode_attn(t["q"], t["C_K"], t["C_V"], t["K_raw"], t["V_raw"], t["U_K"],
                          t["U_V"], t["q_pos"], scale=w.scale, rope_base=w.rope_base, workspace=ws)


@pytest.mark.parametrize("w", [
    wl.config(0),
    wl.custom(B=2, Hq=32, Hkv=8, N_b=1000, W=300, rank=256, rope_base=500000.0),
], ids=["tiny-f32", "bf16-ragged"])
def test_noalloc_matches_workspace_entry_on_two_calls(w):
    lib = bd.load()
    torch.cuda.set_device(0)
    sh = _shape(w)
    assert bd.workspace_bytes(sh, bd.SLIMKV_LATENT) <= bd.NOALLOC_SCRATCH_BYTES
    for layer in range(2):                       # two calls in a row, different inputs
        w_l = w if layer == 0 else dataclasses.replace(w, seed=w.seed + 100)
        t = to_dev(wl.layer_tensors(w_l, 0))
        want = _with_workspace(w_l, t)
        got = torch.full((w.B, w.Hq, w.d), float("nan"), dtype=torch.float32, device="cuda")
        assert _noalloc_call(lib, sh, t, got) == 0
        torch.cuda.synchronize()
        assert torch.equal(got, want), f"noalloc call {layer + 1} differs from slimkv_decode_attn"
        ref = run_oracle("latent", w_l, wl.layer_tensors(w_l, 0))
        assert_close(got.double().cpu().numpy(), ref, w.dtype, f"noalloc call {layer + 1} vs oracle")


def test_noalloc_small_call_after_large_call_reads_nothing_stale():
    lib = bd.load()
    torch.cuda.set_device(0)
    big = wl.custom(B=8, Hq=32, Hkv=8, N_b=4000, W=700, rank=256, seed=11)
    small = wl.custom(B=1, Hq=8, Hkv=2, N_b=130, W=20, rank=64, seed=12)
    assert bd.workspace_bytes(_shape(big), bd.SLIMKV_LATENT) <= bd.NOALLOC_SCRATCH_BYTES
    tb = to_dev(wl.layer_tensors(big, 0))
    ob = torch.empty((big.B, big.Hq, big.d), dtype=torch.float32, device="cuda")
    assert _noalloc_call(lib, _shape(big), tb, ob) == 0
    ts = to_dev(wl.layer_tensors(small, 0))
    got = torch.full((small.B, small.Hq, small.d), float("nan"), dtype=torch.float32, device="cuda")
    assert _noalloc_call(lib, _shape(small), ts, got) == 0
    want = _with_workspace(small, ts, nan_fill=True)
    torch.cuda.synchronize()
    assert torch.equal(got, want)
    assert_close(got.double().cpu().numpy(), run_oracle("latent", small, wl.layer_tensors(small, 0)), "bf16",
                 "small noalloc call after a large one vs oracle")


def test_noalloc_rejects_oversized_shape_without_launch():
    lib = bd.load()
    # B=256 at rank 512 with 128 heads needs far more than the fixed scratch array
    sh = bd.make_shape(256, 128, 8, 128, 8192, 512, 512, 2048, bd.SLIMKV_BF16)
    assert bd.workspace_bytes(sh, bd.SLIMKV_LATENT) > bd.NOALLOC_SCRATCH_BYTES
    z = torch.zeros(16, dtype=torch.uint8, device="cuda")
    p = z.data_ptr()
    st = lib.slimkv_decode_attn_noalloc(ctypes.byref(sh), p, p, p, p, p, p, p, p, p, None)
    assert st == 7
    assert lib.slimkv_status_str(st) != b"unknown status"

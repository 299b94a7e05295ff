"""Failure detection on the GPU without a fault: every wait in the tensor-core kernels
is bounded, and a thread block whose wait runs out writes NaN into its share of the
result, counts itself in a device counter the host can read (slimkv_abort_count) and
returns, leaving the context usable. The test makes one wait run out by withholding a
single tile load (a barrier nothing completes), through the library's test hook."""
import numpy as np
import pytest
import torch

from latent_kv_cache_decode_b300 import binding as bd
from latent_kv_cache_decode_b300 import workloads as wl
from tests.parity_util import run_gpu

pytestmark = pytest.mark.gpu


def test_withheld_load_aborts_reports_and_leaves_the_context_usable():
    w = wl.custom(B=2, Hq=8, Hkv=2, N_b=256, rank=64, W=128)
    sh = bd.make_shape(w.B, w.Hq, w.Hkv, w.d, w.N_b, w.rank, w.rank, w.W, torch.bfloat16)
    if bd.kernel_path(sh, bd.SLIMKV_LATENT) != 1:
        pytest.skip("the bounded waits live in the tensor-core path (sm_103a)")
    t = wl.layer_tensors(w, 0)
    ref = run_gpu("latent", w, t)
    assert np.all(np.isfinite(ref))
    bd.abort_count(reset=True)
    assert bd.abort_count() == 0

    bd.withhold_first_load_for_test(0)          # CTA 0 of the next decode launch
    out = run_gpu("latent", w, t)               # returns after the ~2 s wait limit
    assert bd.abort_count(reset=True) >= 1
    bad = ~np.isfinite(out)
    assert bad.any(), "the aborted block's share of the result must be NaN"
    # what the aborted block did not cover is untouched by it
    clean = [b for b in range(w.B) if not bad[b].any()]
    assert clean, "only part of the batch depends on CTA 0"
    for b in clean:
        assert np.array_equal(out[b], ref[b])

    # the context still works, and the hook was one-shot
    again = run_gpu("latent", w, t)
    assert np.array_equal(again, ref)
    assert bd.abort_count() == 0

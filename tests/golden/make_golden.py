"""Writes the stored expected values under tests/golden/ from the float64 oracle.

Only the seeded input generator and ``oracle/`` run here. The SlimKV pages print
no worked example, so these files pin the oracle and the generator against
silent drift; they are not values taken from the pages.

Usage: python tests/golden/make_golden.py
"""
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402
from latent_kv_cache_decode_b300 import workloads as wl  # noqa: E402


def config0_arrays():
    w = wl.config(0)
    t = wl.layer_tensors(w, 0)
    f = {k: wl.as_f64(v) for k, v in t.items() if k != "q_pos"}
    pos = t["q_pos"].numpy()
    lat = oracle.decode_attn(f["q"], f["C_K"], f["C_V"], f["K_raw"], f["V_raw"], f["U_K"],
                             f["U_V"], pos, w.scale, w.rope_base)
    rec = oracle.decode_attn_reconstruct(f["q"], f["C_K"], f["C_V"], f["K_raw"], f["V_raw"],
                                         f["U_K"], f["U_V"], pos, w.scale, w.rope_base)
    return lat, rec


def prefill_arrays():
    """A 40-token chunk over the tiny workload's 64 beacons (ALiBi-free prefill rule)."""
    w = wl.config(0)
    t = wl.layer_tensors(w, 0)
    t.update(wl.prefill_chunk(w, 0, 40))
    f = {k: wl.as_f64(v) for k, v in t.items() if k not in ("q_pos", "p0")}
    return oracle.prefill_attn(f["q"], f["C_K"], f["C_V"], f["K_chunk"], f["V_chunk"], f["U_K"], f["U_V"],
                               t["p0"].numpy(), w.scale, w.rope_base)


def main():
    pre = prefill_arrays()
    np.savetxt(os.path.join(HERE, "config0_prefill_out.txt"), pre.reshape(-1, pre.shape[-1]), fmt="%.17e",
               header=("tiny fp32 workload (seed 0: B=1, Hq=4, Hkv=1, d=64, N_b=64, r=32), a 40-token chunk "
                       "at positions 2048..2087 (keys after RoPE, seeded draws); oracle output out[b,t,h,:] "
                       "one (token, head) per line; written by tests/golden/make_golden.py (prefill_attn)"))
    lat, rec = config0_arrays()
    hdr = ("tiny fp32 workload (seed 0: B=1, Hq=4, Hkv=1, d=64, N_b=64, r=32, W=32, "
           "q at position 2080, RoPE base 10000, scale 1/8); oracle output out[b,h,:] "
           "one head per line; written by tests/golden/make_golden.py")
    np.savetxt(os.path.join(HERE, "config0_latent_out.txt"), lat.reshape(-1, lat.shape[-1]),
               fmt="%.17e", header=hdr + " (decode_attn)")
    np.savetxt(os.path.join(HERE, "config0_reconstruct_out.txt"), rec.reshape(-1, rec.shape[-1]),
               fmt="%.17e", header=hdr + " (decode_attn_reconstruct)")


if __name__ == "__main__":
    main()

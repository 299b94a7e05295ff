"""Shared helpers of the GPU parity tests: run the library and the oracle on the
same seeded inputs and compare."""
import numpy as np
import torch

import oracle
from latent_kv_cache_decode_b300 import binding as bd
from latent_kv_cache_decode_b300 import workloads as wl

# tolerances: float32 storage -> max-abs 1e-5; bf16 storage (float32 accumulate)
# -> relative L2 <= 3e-3 over the whole output, <= 1.2e-2 for every single (b, h) row
# (a row is one head's weighted average: the rounding of its bf16 inputs and weights
# does not average out over other heads, so its bar is 4x the global one), and
# max-abs <= 2e-2
F32_MAX_ABS = 1e-5
BF16_REL_L2 = 3e-3
BF16_ROW_REL_L2 = 1.2e-2
BF16_MAX_ABS = 2e-2


def to_dev(t):
    return {k: v.cuda() for k, v in t.items()}


def f64(t):
    return {k: (wl.as_f64(v) if k != "q_pos" else v.numpy()) for k, v in t.items()}


def run_gpu(which, w, t, out=None):
    d = to_dev(t)
    kw = dict(scale=w.scale, rope_base=w.rope_base)
    if which == "latent":
        o = bd.decode_attn(d["q"], d["C_K"] if w.N_b else None, d["C_V"] if w.N_b else None,
                           d["K_raw"] if w.W else None, d["V_raw"] if w.W else None,
                           d["U_K"] if w.N_b else None, d["U_V"] if w.N_b else None,
                           d["q_pos"], **kw)
    elif which == "reconstruct":
        o = bd.decode_attn_reconstruct(d["q"], d["C_K"], d["C_V"], d["K_raw"] if w.W else None,
                                       d["V_raw"] if w.W else None, d["U_K"], d["U_V"],
                                       d["q_pos"], **kw)
    elif which == "alibi":
        o = bd.decode_attn_alibi(d["q"], d["C_K"] if w.N_b else None, d["C_V"] if w.N_b else None,
                                 d["K_raw"] if w.W else None, d["V_raw"] if w.W else None,
                                 d["U_K"] if w.N_b else None, d["U_V"] if w.N_b else None,
                                 d["q_pos"], bd.alibi_slopes(w.Hq), w.ratio, **kw)
    elif which == "reconstruct_rope":
        o = bd.decode_attn_reconstruct_rope(d["q"], d["C_K"], d["C_V"], d["K_raw"] if w.W else None,
                                            d["V_raw"] if w.W else None, d["U_K"], d["U_V"],
                                            d["q_pos"], w.ratio, **kw)
    else:
        o = bd.decode_attn_full_kv(d["q"], d["K_full"], d["V_full"], d["q_pos"], **kw)
    torch.cuda.synchronize()
    return o.cpu().double().numpy()


def run_oracle(which, w, t, pairs=None):
    f = f64(t)
    if which == "latent":
        return oracle.decode_attn(f["q"], f["C_K"] if w.N_b else None, f["C_V"] if w.N_b else None,
                                  f["K_raw"] if w.W else None, f["V_raw"] if w.W else None,
                                  f["U_K"], f["U_V"], f["q_pos"], w.scale, w.rope_base, pairs=pairs)
    if which == "reconstruct":
        return oracle.decode_attn_reconstruct(f["q"], f["C_K"], f["C_V"], f["K_raw"], f["V_raw"],
                                              f["U_K"], f["U_V"], f["q_pos"], w.scale, w.rope_base,
                                              pairs=pairs)
    if which == "alibi":
        return oracle.decode_attn_alibi(f["q"], f["C_K"] if w.N_b else None, f["C_V"] if w.N_b else None,
                                        f["K_raw"] if w.W else None, f["V_raw"] if w.W else None,
                                        f["U_K"], f["U_V"], f["q_pos"], w.scale, w.rope_base,
                                        np.array(bd.alibi_slopes(w.Hq)), w.ratio, pairs=pairs)
    if which == "reconstruct_rope":
        return oracle.decode_attn_reconstruct_rope(f["q"], f["C_K"], f["C_V"], f["K_raw"], f["V_raw"],
                                                   f["U_K"], f["U_V"], f["q_pos"], w.scale, w.rope_base,
                                                   w.ratio, pairs=pairs)
    return oracle.decode_attn_full_kv(f["q"], f["K_full"], f["V_full"], f["q_pos"], w.scale,
                                      w.rope_base, pairs=pairs)


def errors(got, ref):
    diff = got - ref
    rel = float(np.linalg.norm(diff) / max(np.linalg.norm(ref), 1e-30))
    return rel, float(np.abs(diff).max())


def row_errors(got, ref):
    """Relative L2 error of every (b, h) output row (last axis), and the worst row."""
    g = got.reshape(-1, got.shape[-1])
    r = ref.reshape(-1, ref.shape[-1])
    rel = np.linalg.norm(g - r, axis=1) / np.maximum(np.linalg.norm(r, axis=1), 1e-30)
    return rel, int(np.argmax(rel))


def assert_close(got, ref, dtype, what=""):
    rel, mx = errors(got, ref)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    if dtype == "f32":
        assert mx <= F32_MAX_ABS, f"{what}: max-abs {mx:.3e} > {F32_MAX_ABS} (rel-L2 {rel:.3e})"
    else:
        assert rel <= BF16_REL_L2 and mx <= BF16_MAX_ABS, \
            f"{what}: rel-L2 {rel:.3e} (bar {BF16_REL_L2}), max-abs {mx:.3e} (bar {BF16_MAX_ABS})"
        rows, worst = row_errors(got, ref)
        assert rows[worst] <= BF16_ROW_REL_L2, \
            f"{what}: row {worst} (b, h) = {divmod(worst, got.shape[-2])} rel-L2 {rows[worst]:.3e} " \
            f"(bar {BF16_ROW_REL_L2}; whole-output rel-L2 {rel:.3e})"
    return rel, mx

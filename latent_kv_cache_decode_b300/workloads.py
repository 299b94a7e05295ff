"""Seeded synthetic inputs for SlimKV decode-step attention.

This module only draws random numbers and shapes tensors. It holds none of the
attention arithmetic: it is shared by the tests, the benchmark and the oracle
comparisons, and nothing in it computes a score, a softmax or a projection.

Workloads follow the long-context decode settings the SlimKV pages measure
(Llama-3.1-8B and Qwen2.5-14B attention shapes, "Speedups are real, but memory
is set by the ratio" on "Can SlimKV compress KV cache jointly across tokens and
features"). No trained weights or datasets are involved: every tensor is drawn
from a seeded normal distribution, and the up-projections are random matrices
with orthonormal columns.

Readings fixed here:
* The raw window stores keys after RoPE. A RoPE rotation maps an i.i.d. N(0,1)
  pair to an i.i.d. N(0,1) pair, so a stored (rotated) key is drawn directly
  from N(0,1); the window positions therefore never enter the computation, only
  the query position does.
* Every (seed, layer, batch element, tensor) gets its own generator
  (``numpy.random.default_rng([seed, layer, b, tensor_id])``), so any single
  layer or batch element can be regenerated alone.
* bf16 storage rounds the float32 draw to nearest-even bf16; the oracle reads
  those exact bf16 values widened to float64.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, List, Optional

import numpy as np
import torch

# tensor ids used as part of the per-tensor seed
_TID = {"U_K": 0, "U_V": 1, "C_K": 2, "C_V": 3, "K_raw": 4, "V_raw": 5, "q": 6,
        "peaks": 7, "ranks": 8, "K_full": 9, "V_full": 10, "k_new": 11, "v_new": 12,
        "q_step": 13, "q_chunk": 14, "K_chunk": 15, "V_chunk": 16, "chunk_peaks": 17}


@dataclasses.dataclass(frozen=True)
class Workload:
    """One decode-step workload: per-layer attention shapes plus data recipe."""
    name: str
    seed: int
    dtype: str                 # "f32" or "bf16" (storage of q, C, K, V, U)
    B: int
    Hq: int
    Hkv: int
    d: int
    N_b: int                   # beacon states per batch element
    W: int                     # raw-window tokens per batch element
    layers: int
    rope_base: float
    ranks: Optional[List[int]] = None   # per-layer latent rank (r_k = r_v)
    rank: int = 0                        # uniform rank when ranks is None
    ratio: int = 1                       # token compression ratio (positions only)
    peak_frac: float = 0.0               # fraction of raw keys scaled by peak_scale
    peak_scale: float = 1.0
    T_full: int = 0                      # full-KV cache length (comparison workload)

    def r(self, layer: int) -> int:
        return self.ranks[layer] if self.ranks is not None else self.rank

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def q_pos(self) -> int:
        # beacons fold N_b * ratio tokens, the window follows them, and the
        # query sits right after the window
        return self.N_b * self.ratio + self.W

    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16


def _qwen_ranks(seed: int, layers: int, lo_units: int = 4, hi_units: int = 16,
                mean_units: int = 8) -> List[int]:
    """Per-layer ranks in multiples of 32 in [32*lo, 32*hi] with an exact mean.

    Stand-in for the layer-adaptive rank allocation the pages describe (a
    floor-constrained equal-energy rule whose details they do not give): every
    layer starts at the floor, and the remaining budget is handed out one unit
    of 32 at a time to a uniformly drawn layer that is still below the cap.
    """
    rng = np.random.default_rng([seed, _TID["ranks"]])
    units = [lo_units] * layers
    spare = layers * mean_units - layers * lo_units
    while spare > 0:
        open_layers = [i for i in range(layers) if units[i] < hi_units]
        i = open_layers[int(rng.integers(len(open_layers)))]
        units[i] += 1
        spare -= 1
    return [32 * u for u in units]


def config(idx: int) -> Workload:
    """The five decode workloads (0: tiny fp32, 1-3: model shapes, 4: comparison)."""
    if idx == 0:
        return Workload("tiny-f32", 0, "f32", B=1, Hq=4, Hkv=1, d=64, N_b=64, W=32,
                        layers=1, rope_base=10000.0, rank=32, ratio=32)
    if idx == 1:
        return Workload("llama3.1-8b-32k-8x", 1, "bf16", B=1, Hq=32, Hkv=8, d=128,
                        N_b=4096, W=1024, layers=32, rope_base=500000.0, rank=256,
                        ratio=8)
    if idx == 2:
        return Workload("llama3.1-8b-128k-16x", 2, "bf16", B=8, Hq=32, Hkv=8, d=128,
                        N_b=8192, W=2048, layers=32, rope_base=500000.0, rank=256,
                        ratio=16, peak_frac=0.01, peak_scale=8.0)
    if idx == 3:
        return Workload("qwen2.5-14b-64k-32x", 3, "bf16", B=4, Hq=40, Hkv=8, d=128,
                        N_b=2048, W=1024, layers=48, rope_base=1000000.0,
                        ranks=_qwen_ranks(3, 48), ratio=32)
    if idx == 4:
        return Workload("llama3.1-8b-128k-16x-compare", 4, "bf16", B=8, Hq=32, Hkv=8,
                        d=128, N_b=8192, W=2048, layers=32, rope_base=500000.0,
                        rank=256, ratio=16, peak_frac=0.01, peak_scale=8.0,
                        T_full=131072)
    raise ValueError(f"no workload {idx}")


def custom(**kw) -> Workload:
    """A workload with explicit shapes (edge cases, small parity cases)."""
    base = dict(name="custom", seed=7, dtype="bf16", B=1, Hq=8, Hkv=2, d=128, N_b=256,
                W=128, layers=1, rope_base=10000.0, rank=64, ratio=4)
    base.update(kw)
    return Workload(**base)


def _rng(seed: int, *key: int) -> np.random.Generator:
    return np.random.default_rng([seed, *key])


def _normal(rng: np.random.Generator, shape) -> np.ndarray:
    return rng.standard_normal(shape, dtype=np.float32)


def orthonormal_columns(rng: np.random.Generator, rows: int, cols: int) -> np.ndarray:
    """rows x cols matrix with orthonormal columns (QR of a float64 Gaussian,
    column signs fixed so that diag(R) > 0)."""
    if cols > rows:
        raise ValueError(f"{rows}x{cols} cannot have orthonormal columns")
    a = rng.standard_normal((rows, cols))
    qm, rm = np.linalg.qr(a)
    sgn = np.sign(np.diag(rm))
    sgn[sgn == 0] = 1.0
    return qm * sgn[None, :]


def _store(x: np.ndarray, w: Workload) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(w.torch_dtype())


def layer_tensors(w: Workload, layer: int, batch: Optional[List[int]] = None,
                  with_full: bool = False) -> Dict[str, torch.Tensor]:
    """CPU tensors (storage dtype) for one layer of workload ``w``.

    Keys: q [B,Hq,d], C_K [B,N_b,r], C_V [B,N_b,r], K_raw [B,W,Hkv,d],
    V_raw [B,W,Hkv,d], U_K [Hkv*d,r], U_V [Hkv*d,r], q_pos [B] int32 and, with
    ``with_full``, K_full/V_full [B,T_full,Hkv,d]. ``batch`` selects a subset of
    batch elements (their data is identical to the full draw).
    """
    bs = list(range(w.B)) if batch is None else list(batch)
    r = w.r(layer)
    s = w.seed
    out: Dict[str, torch.Tensor] = {}
    out["U_K"] = _store(orthonormal_columns(_rng(s, layer, _TID["U_K"]), w.Hkv * w.d, r), w)
    out["U_V"] = _store(orthonormal_columns(_rng(s, layer, _TID["U_V"]), w.Hkv * w.d, r), w)
    ck, cv, kr, vr, qq, kf, vf = [], [], [], [], [], [], []
    for b in bs:
        ck.append(_normal(_rng(s, layer, b, _TID["C_K"]), (w.N_b, r)))
        cv.append(_normal(_rng(s, layer, b, _TID["C_V"]), (w.N_b, r)))
        k = _normal(_rng(s, layer, b, _TID["K_raw"]), (w.W, w.Hkv, w.d))
        if w.peak_frac > 0 and w.W > 0:
            n_peak = int(round(w.peak_frac * w.W))
            idx = _rng(s, layer, b, _TID["peaks"]).choice(w.W, size=n_peak, replace=False)
            k[idx] *= np.float32(w.peak_scale)
        kr.append(k)
        vr.append(_normal(_rng(s, layer, b, _TID["V_raw"]), (w.W, w.Hkv, w.d)))
        qq.append(_normal(_rng(s, layer, b, _TID["q"]), (w.Hq, w.d)))
        if with_full:
            kf.append(_normal(_rng(s, layer, b, _TID["K_full"]), (w.T_full, w.Hkv, w.d)))
            vf.append(_normal(_rng(s, layer, b, _TID["V_full"]), (w.T_full, w.Hkv, w.d)))
    out["C_K"] = _store(np.stack(ck), w)
    out["C_V"] = _store(np.stack(cv), w)
    out["K_raw"] = _store(np.stack(kr), w)
    out["V_raw"] = _store(np.stack(vr), w)
    out["q"] = _store(np.stack(qq), w)
    out["q_pos"] = torch.full((len(bs),), w.q_pos, dtype=torch.int32)
    if with_full:
        out["K_full"] = _store(np.stack(kf), w)
        out["V_full"] = _store(np.stack(vf), w)
    return out


def decode_steps(w: Workload, layer: int, steps: int,
                 batch: Optional[List[int]] = None) -> Dict[str, torch.Tensor]:
    """CPU tensors (storage dtype) for ``steps`` generated tokens of one layer.

    Keys: k_new, v_new [S,B,Hkv,d] (the new tokens' keys before RoPE and values),
    q [S,B,Hq,d] and pos [S,B] int32. Token s sits at position q_pos + s, right
    after the prompt window, whose tokens q_pos - W .. q_pos - 1 are taken to be
    stored in slots (position mod W)."""
    bs = list(range(w.B)) if batch is None else list(batch)
    s = w.seed
    kn = np.stack([_normal(_rng(s, layer, b, _TID["k_new"]), (steps, w.Hkv, w.d)) for b in bs], axis=1)
    vn = np.stack([_normal(_rng(s, layer, b, _TID["v_new"]), (steps, w.Hkv, w.d)) for b in bs], axis=1)
    qq = np.stack([_normal(_rng(s, layer, b, _TID["q_step"]), (steps, w.Hq, w.d)) for b in bs], axis=1)
    pos = w.q_pos + np.arange(steps, dtype=np.int64)[:, None] + np.zeros((1, len(bs)), dtype=np.int64)
    return {"k_new": _store(kn, w), "v_new": _store(vn, w), "q": _store(qq, w),
            "pos": torch.from_numpy(pos.astype(np.int32))}


def prefill_chunk(w: Workload, layer: int, T: int,
                  batch: Optional[List[int]] = None) -> Dict[str, torch.Tensor]:
    """CPU tensors (storage dtype) for one prefill chunk of T tokens of one layer.

    Keys: q [B,T,Hq,d] (before RoPE), K_chunk, V_chunk [B,T,Hkv,d] (keys stored after
    RoPE, drawn directly as N(0,1) like the window keys) and p0 [B] int32, the position
    of chunk token 0. The chunk follows the tokens the beacons fold: p0 = N_b * ratio.
    With ``peak_frac`` set, that fraction of the chunk's tokens have their keys scaled
    by ``peak_scale`` on every KV head, as in the raw window."""
    bs = list(range(w.B)) if batch is None else list(batch)
    s = w.seed
    qq, kc, vc = [], [], []
    for b in bs:
        qq.append(_normal(_rng(s, layer, b, _TID["q_chunk"]), (T, w.Hq, w.d)))
        k = _normal(_rng(s, layer, b, _TID["K_chunk"]), (T, w.Hkv, w.d))
        if w.peak_frac > 0 and T > 0:
            n_peak = int(round(w.peak_frac * T))
            idx = _rng(s, layer, b, _TID["chunk_peaks"]).choice(T, size=n_peak, replace=False)
            k[idx] *= np.float32(w.peak_scale)
        kc.append(k)
        vc.append(_normal(_rng(s, layer, b, _TID["V_chunk"]), (T, w.Hkv, w.d)))
    return {"q": _store(np.stack(qq), w), "K_chunk": _store(np.stack(kc), w),
            "V_chunk": _store(np.stack(vc), w),
            "p0": torch.full((len(bs),), w.N_b * w.ratio, dtype=torch.int32)}


def as_f64(t: torch.Tensor) -> np.ndarray:
    """Exact widening of a stored tensor to a float64 numpy array."""
    return t.to(torch.float64).numpy()


def cache_bytes(w: Workload, layer: int) -> int:
    """Bytes of cache one layer reads per decode step (latent C_K, C_V and the raw
    window K, V), all batch elements."""
    es = 4 if w.dtype == "f32" else 2
    r = w.r(layer)
    return w.B * (w.N_b * 2 * r + 2 * w.W * w.Hkv * w.d) * es


def u_bytes(w: Workload, layer: int) -> int:
    es = 4 if w.dtype == "f32" else 2
    return 2 * w.Hkv * w.d * w.r(layer) * es

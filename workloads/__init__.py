"""Seeded synthetic inputs for the Mixtral-style MoE feed-forward layer.

This module is shared by the fp64 oracle (``oracle/``) and by the CUDA path
(``sparse_mixture_experts_56_b300``).  It holds no arithmetic of the layer
itself: it only names the workload shapes, draws seeded Gaussian tensors and
stores them as bf16 bit patterns (round-to-nearest-even) or fp32.

Shapes follow the Mixtral 8x7B description: d_model = 4096, d_ff = 14336,
n = 8 experts, top-K = 2 ("Mixtral of Experts", xyznot.com summary, section
"Método (con las ecuaciones clave)").  The pages measure the model only on
public suites (MMLU, GSM8K, ...) and the Pile; none of that is used here.  The
synthetic tensors below stand in for real activations and trained weights.

Distributions (standard-deviation reading of N(0, s)):
  x ~ N(0, 1); W_g ~ N(0, 0.02); w1, w3 ~ N(0, 1/sqrt(d)); w2 ~ N(0, 1/sqrt(f)).
Every tensor is drawn in fp32 from its own ``numpy.random.SeedSequence``
``[seed, workload, layer, tensor, chunk]`` (chunks of 2**24 values, so that
large tensors are drawn by several threads and still reproduce exactly), then
rounded to bf16 for the bf16 workloads.
"""
from __future__ import annotations

import dataclasses
import os
from concurrent.futures import ThreadPoolExecutor
from typing import Dict, Optional

import numpy as np

__all__ = [
    "Workload", "WORKLOADS", "workload", "custom", "make_inputs", "bf16_round_bits",
    "bf16_bits_to_f32", "logit_bias_vector", "TENSOR_IDS", "active_flops", "expert_weight_bytes",
]

_CHUNK = 1 << 24

# tensor ids used in the seed sequence (stable: changing them changes every input)
TENSOR_IDS = {"x": 0, "wg": 1, "w1": 2, "w3": 3, "w2": 4, "dy": 5}


@dataclasses.dataclass(frozen=True)
class Workload:
    """One MoE-layer workload: shapes, storage dtype and routing extras."""
    wid: int            # workload id used in the seed sequence
    name: str
    T: int              # tokens
    d: int              # d_model
    f: int              # d_ff (expert intermediate size)
    n: int              # experts
    k: int              # experts kept per token
    dtype: str          # "f32" or "bf16": storage type of x, W_g, w1, w3, w2, y
    skew_bias: bool = False     # per-expert logit bias 1.5*(e==0) + 0.75*(e==1)
    layers: int = 1             # stacked layers (h <- h + MoE_l(RMSNorm(h)))
    residual: bool = False
    rms_eps: float = 1e-5

    @property
    def assignments(self) -> int:
        return self.T * self.k


WORKLOADS: Dict[int, Workload] = {
    1: Workload(1, "tiny-fp32-t64", T=64, d=128, f=256, n=8, k=2, dtype="f32"),
    2: Workload(2, "mixtral-decode-t32", T=32, d=4096, f=14336, n=8, k=2, dtype="bf16"),
    3: Workload(3, "mixtral-prefill-t4096", T=4096, d=4096, f=14336, n=8, k=2, dtype="bf16"),
    4: Workload(4, "mixtral-skewed-t16384", T=16384, d=4096, f=14336, n=8, k=2, dtype="bf16",
                skew_bias=True),
    5: Workload(5, "mixtral-stack4-t8192", T=8192, d=4096, f=14336, n=8, k=2, dtype="bf16",
                layers=4, residual=True),
}


def workload(i: int) -> Workload:
    return WORKLOADS[i]


def custom(T: int, d: int, f: int, n: int, k: int, dtype: str = "bf16", *, wid: int = 100,
           skew_bias: bool = False, name: Optional[str] = None) -> Workload:
    """A test-sized workload with the same distributions (distinct seed stream via ``wid``)."""
    return Workload(wid, name or f"custom-t{T}-d{d}-f{f}-n{n}-k{k}-{dtype}", T=T, d=d, f=f, n=n,
                    k=k, dtype=dtype, skew_bias=skew_bias)


def logit_bias_vector(n: int) -> np.ndarray:
    """Per-expert logit bias of the skewed workload: b_e = 1.5*(e==0) + 0.75*(e==1)."""
    b = np.zeros(n, dtype=np.float32)
    if n > 0:
        b[0] = 1.5
    if n > 1:
        b[1] = 0.75
    return b


def active_flops(w: Workload) -> float:
    """Active FLOPs of one layer pass: 2 * T * K * 3 * d * f (three expert matmuls)."""
    return 2.0 * w.T * w.k * 3.0 * w.d * w.f


def expert_weight_bytes(w: Workload) -> int:
    """Bytes of all experts' w1, w3, w2 of one layer in the storage dtype."""
    esz = 2 if w.dtype == "bf16" else 4
    return 3 * w.n * w.d * w.f * esz


# ----------------------------------------------------------------------------------------
# bf16 storage helpers (data format only)
# ----------------------------------------------------------------------------------------
def bf16_round_bits(a: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit pattern (uint16), round to nearest, ties to even.  Inputs are finite."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    r = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """bf16 bit pattern (uint16) -> the exact fp32 value it encodes."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _threads() -> int:
    env = os.environ.get("MOE_GEN_THREADS")
    if env:
        return max(1, int(env))
    try:
        return max(1, min(32, len(os.sched_getaffinity(0))))
    except AttributeError:  # pragma: no cover
        return max(1, min(32, os.cpu_count() or 1))


def _draw(shape, std: float, seed: int, w: Workload, layer: int, tensor: str, as_bf16: bool):
    """Draw N(0, std) of ``shape`` chunk by chunk, each chunk from its own seed sequence."""
    total = int(np.prod(shape)) if len(shape) else 1
    out = np.empty(total, dtype=np.uint16 if as_bf16 else np.float32)
    tid = TENSOR_IDS[tensor]
    nchunks = max(1, (total + _CHUNK - 1) // _CHUNK)

    def work(c: int) -> None:
        lo = c * _CHUNK
        hi = min(total, lo + _CHUNK)
        if hi <= lo:
            return
        ss = np.random.SeedSequence([seed, w.wid, layer, tid, c])
        rng = np.random.Generator(np.random.PCG64(ss))
        v = rng.standard_normal(hi - lo, dtype=np.float32)
        v *= np.float32(std)
        out[lo:hi] = bf16_round_bits(v) if as_bf16 else v

    nt = min(_threads(), nchunks)
    if nt <= 1:
        for c in range(nchunks):
            work(c)
    else:
        with ThreadPoolExecutor(max_workers=nt) as ex:
            list(ex.map(work, range(nchunks)))
    return out.reshape(shape)


def make_inputs(w: Workload, seed: int = 0, layer: int = 0,
                tensors=("x", "wg", "w1", "w3", "w2")) -> Dict[str, np.ndarray]:
    """Seeded inputs of one layer.

    Returns a dict with (bf16 workloads: uint16 bit patterns; f32 workloads: float32):
      x  [T, d]      token activations (for stacked workloads: the input of layer 0)
      wg [d, n]      router weight W_g (row-major d x n, so logits = x @ W_g)
      w1 [n, f, d]   per-expert gate projection, out x in (K-major rows)
      w3 [n, f, d]   per-expert up projection, out x in
      w2 [n, d, f]   per-expert down projection, out x in
      dy [T, d]      (only when asked for) gradient of the layer output, N(0, 1), for the
                     backward
      bias [n] fp32  logit bias, or None
    ``x`` depends only on (seed, workload); weights also on ``layer``.
    """
    bf = w.dtype == "bf16"
    out: Dict[str, np.ndarray] = {}
    if "x" in tensors:
        out["x"] = _draw((w.T, w.d), 1.0, seed, w, 0, "x", bf)
    if "wg" in tensors:
        out["wg"] = _draw((w.d, w.n), 0.02, seed, w, layer, "wg", bf)
    if "w1" in tensors:
        out["w1"] = _draw((w.n, w.f, w.d), 1.0 / np.sqrt(w.d), seed, w, layer, "w1", bf)
    if "w3" in tensors:
        out["w3"] = _draw((w.n, w.f, w.d), 1.0 / np.sqrt(w.d), seed, w, layer, "w3", bf)
    if "w2" in tensors:
        out["w2"] = _draw((w.n, w.d, w.f), 1.0 / np.sqrt(w.f), seed, w, layer, "w2", bf)
    if "dy" in tensors:
        out["dy"] = _draw((w.T, w.d), 1.0, seed, w, layer, "dy", bf)
    out["bias"] = logit_bias_vector(w.n) if w.skew_bias else None
    return out


def as_f32(a: np.ndarray, w: Workload) -> np.ndarray:
    """The fp32 values of a stored tensor (bf16 bits are expanded exactly)."""
    return bf16_bits_to_f32(a) if w.dtype == "bf16" else np.asarray(a, dtype=np.float32)

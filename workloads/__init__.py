"""Seeded synthetic inputs for the MoE finalize + residual + RMSNorm path.

This module only *draws* inputs: router choices, router weights, the
expert-grouped GEMM2 output, the residual stream and gamma.  It holds none of
the finalize arithmetic (no weighted sum, no residual add, no normalisation,
no output rounding), so the CUDA path and the CPU oracle can both be fed from
it without sharing any of the method's code.

Every workload follows the same draw order:
routing -> router weights -> expert_out -> outlier rows -> residual -> gamma
(the host stream draws routing, weights, the outlier-row choice and gamma in
that order; expert_out and residual come from two torch streams of their own).

* Small draws (routing, weights, outlier-row choice, gamma) use NumPy's PCG64
  ``default_rng(seed)`` on the host.
* The two large tensors (``expert_out`` [R, H] and ``residual`` [T, H]) are
  drawn with a ``torch.Generator`` seeded from the same seed, on the device
  where they will live, in fixed-size chunks.  CPU and CUDA generators give
  different streams, so a test that compares the two paths always hands
  *copies of the same tensors* to both sides.

Normal laws are written N(mean, variance), as in the workload table of the
design notes: N(0, 4) has standard deviation 2, N(1, 0.1) has standard
deviation sqrt(0.1).

The expert-grouped layout is the one a grouped GEMM2 writes: the flat
(token, slot) pairs ``s = t*k + j`` are stably sorted by their expert id; row
``p`` of ``expert_out`` holds the data of the pair at position ``p``; and
``permuted_row_of[t, j]`` is that position.
"""
from __future__ import annotations

import dataclasses
import math
from dataclasses import dataclass
from typing import Dict, Optional

import numpy as np
import torch

__all__ = [
    "Workload", "TINY_REF", "PREFILL", "STRESS", "decode", "wide",
    "DECODE_TOKENS", "WIDE_TOKENS", "all_named", "by_name",
    "draw_routing", "grouped_index_map", "make_inputs", "algorithmic_bytes",
]

_CHUNK = 1 << 24  # elements per torch draw; fixed so streams are reproducible


@dataclass(frozen=True)
class Workload:
    """One synthetic configuration.

    routing: ``"logits"`` (top-k of N(0,1) logits per token over E experts),
    ``"uniform"`` (k distinct experts uniformly at random) or ``"zipf"``
    (k distinct experts by Gumbel-top-k on log p_e, p_e ~ (e+1)^-zipf_s).
    weights: ``"softmax_logits"`` (softmax over the k selected logits),
    ``"softmax"`` (softmax of k fresh N(0,1) draws, sorted descending) or
    ``"uniform"`` (k Uniform(0,1) draws, sorted descending, unnormalised).
    """

    name: str
    T: int
    H: int
    k: int = 8
    E: int = 128
    routing: str = "uniform"
    zipf_s: float = 0.0
    weights: str = "softmax"
    expert_dist: str = "normal"      # or "student_t3"
    expert_var: float = 1.0          # variance of the normal law (or scale^2 for t)
    outlier_frac: float = 0.0        # fraction of expert_out rows scaled
    outlier_scale: float = 1.0
    residual_var: float = 1.0
    gamma_mean: float = 1.0
    gamma_var: float = 0.1
    eps: float = 1e-6
    seed: int = 0
    extra_rows: int = 0              # rows of expert_out beyond T*k (unused)

    @property
    def R(self) -> int:
        return self.T * self.k + self.extra_rows

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# --- the named configurations ------------------------------------------------

TINY_REF = Workload("tiny_ref", T=16, H=4096, k=8, E=64, routing="logits",
                    weights="softmax_logits", eps=1e-6)

DECODE_TOKENS = (1, 2, 4, 8, 16, 32, 64, 128)


def decode(T: int) -> Workload:
    return Workload(f"decode_T{T}", T=T, H=4096, k=8, E=128, routing="uniform",
                    weights="softmax", eps=1e-6)


PREFILL = Workload("prefill", T=16384, H=4096, k=8, E=128, routing="zipf",
                   zipf_s=1.2, weights="softmax", eps=1e-6)

WIDE_TOKENS = (1, 8, 64, 512, 4096, 8192)


def wide(T: int) -> Workload:
    return Workload(f"wide_T{T}", T=T, H=8192, k=8, E=256, routing="uniform",
                    weights="softmax", expert_var=0.5, residual_var=4.0,
                    eps=1e-5)


STRESS = Workload("stress", T=32768, H=8192, k=8, E=256, routing="zipf",
                  zipf_s=1.5, weights="uniform", expert_dist="student_t3",
                  expert_var=0.25, outlier_frac=0.01, outlier_scale=100.0,
                  eps=1e-6)


def all_named() -> Dict[str, Workload]:
    out = {TINY_REF.name: TINY_REF, PREFILL.name: PREFILL, STRESS.name: STRESS}
    for t in DECODE_TOKENS:
        out[decode(t).name] = decode(t)
    for t in WIDE_TOKENS:
        out[wide(t).name] = wide(t)
    return out


def by_name(name: str) -> Workload:
    return all_named()[name]


def algorithmic_bytes(T: int, H: int, k: int) -> int:
    """Bytes one call must move: k gathered bf16 rows, the fp32 residual read
    and written, the bf16 output, and the int32 index + fp32 weight of every
    slot.  Gamma (2*H bytes, read once per call) is left out."""
    return T * k * H * 2 + T * H * (4 + 4 + 2) + T * k * (4 + 4)


# --- routing -------------------------------------------------------------------

def draw_routing(wl: Workload, rng: np.random.Generator):
    """Returns (expert_of[T,k] int64, weights[T,k] float32); slot j holds the
    j-th highest routing score."""
    T, k, E = wl.T, wl.k, wl.E
    if k > E:
        raise ValueError("k distinct experts need E >= k")
    if wl.routing == "logits":
        logits = rng.standard_normal((T, E))
        order = np.argsort(-logits, axis=1, kind="stable")[:, :k]
        chosen = np.take_along_axis(logits, order, axis=1)
    elif wl.routing in ("uniform", "zipf"):
        if wl.routing == "zipf":
            logp = -wl.zipf_s * np.log(np.arange(1, E + 1, dtype=np.float64))
        else:
            logp = np.zeros(E)
        scores = logp[None, :] + rng.gumbel(size=(T, E))
        order = np.argsort(-scores, axis=1, kind="stable")[:, :k]
        chosen = None
    else:
        raise ValueError(f"unknown routing {wl.routing!r}")

    if wl.weights == "softmax_logits":
        z = chosen - chosen.max(axis=1, keepdims=True)
        p = np.exp(z)
        w = p / p.sum(axis=1, keepdims=True)
    elif wl.weights == "softmax":
        g = rng.standard_normal((T, k))
        z = g - g.max(axis=1, keepdims=True)
        p = np.exp(z)
        w = -np.sort(-(p / p.sum(axis=1, keepdims=True)), axis=1)
    elif wl.weights == "uniform":
        w = -np.sort(-rng.random((T, k)), axis=1)
    else:
        raise ValueError(f"unknown weights {wl.weights!r}")
    return order.astype(np.int64), w.astype(np.float32)


def grouped_index_map(expert_of: np.ndarray) -> np.ndarray:
    """permuted_row_of[t, j] = position of pair (t, j) after a stable sort of
    the flat pairs by expert id (the row a grouped GEMM2 writes it to)."""
    T, k = expert_of.shape
    order = np.argsort(expert_of.reshape(-1), kind="stable")
    pos = np.empty(T * k, dtype=np.int64)
    pos[order] = np.arange(T * k)
    return pos.reshape(T, k).astype(np.int32)


# --- dense tensors -------------------------------------------------------------

def _torch_gen(seed: int, device: torch.device, stream: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed((seed * 1_000_003 + stream * 7919) & 0x7FFF_FFFF_FFFF_FFFF)
    return g


def _fill_rows(out: torch.Tensor, dist: str, scale: float, gen: torch.Generator,
               row_scale: Optional[torch.Tensor] = None) -> None:
    """Fills a contiguous 2-D tensor block of rows by block of rows.

    Values are drawn in fp32, multiplied by ``scale`` (and by ``row_scale[r]``
    for row r when given) and then rounded to ``out.dtype`` by torch's copy.
    ``dist`` is ``"normal"`` (N(0,1)) or ``"student_t3"`` (Z / sqrt(V/3), V the
    sum of three squared standard normals, i.e. chi-square with 3 degrees of
    freedom).  The block size is fixed, so the stream is reproducible."""
    rows, cols = out.shape
    if rows == 0 or cols == 0:
        return
    rb = max(1, _CHUNK // cols)
    for r0 in range(0, rows, rb):
        r1 = min(rows, r0 + rb)
        m = (r1 - r0) * cols
        x = torch.randn(m, generator=gen, device=out.device, dtype=torch.float32)
        if dist == "student_t3":
            v = torch.randn(3, m, generator=gen, device=out.device, dtype=torch.float32)
            v = v.square_().sum(dim=0).div_(3.0)
            x.mul_(torch.rsqrt(v))
        elif dist != "normal":
            raise ValueError(f"unknown distribution {dist!r}")
        x = x.view(r1 - r0, cols)
        if scale != 1.0:
            x.mul_(scale)
        if row_scale is not None:
            x.mul_(row_scale[r0:r1, None])
        out[r0:r1].copy_(x)


def make_inputs(wl: Workload, device="cpu", *, T: Optional[int] = None) -> dict:
    """Draws every input of one call of the path for workload ``wl``.

    Returns a dict with torch tensors on ``device``:
    ``expert_out`` bf16 [R, H], ``permuted_row_of`` int32 [T, k],
    ``topk_weights`` fp32 [T, k], ``residual`` fp32 [T, H], ``gamma`` bf16 [H],
    the float ``eps``, and host-side ``expert_of`` (int64 [T, k]) and
    ``outlier_rows`` for reference.

    The outlier rows of expert_out (a fraction of all rows, chosen without
    replacement) are multiplied in fp32 before the single rounding to bf16.
    Their choice is the NumPy draw that follows the router weights; the torch
    streams for expert_out and residual are separate, so the order of the
    NumPy draws stays routing -> weights -> outlier rows -> gamma.
    """
    if T is not None:
        wl = wl.with_(T=T)
    device = torch.device(device)
    rng = np.random.default_rng(wl.seed)
    expert_of, w = draw_routing(wl, rng)
    idx = grouped_index_map(expert_of)

    R, H = wl.R, wl.H
    n_out = int(round(wl.outlier_frac * wl.T * wl.k))
    outlier_rows = (np.sort(rng.choice(R, size=n_out, replace=False)) if n_out
                    else np.zeros(0, dtype=np.int64))
    row_scale = None
    if n_out:
        rs = np.ones(R, dtype=np.float32)
        rs[outlier_rows] = wl.outlier_scale
        row_scale = torch.from_numpy(rs).to(device)

    expert_out = torch.empty((R, H), dtype=torch.bfloat16, device=device)
    _fill_rows(expert_out, wl.expert_dist, math.sqrt(wl.expert_var),
               _torch_gen(wl.seed, device, 1), row_scale)

    residual = torch.empty((wl.T, H), dtype=torch.float32, device=device)
    _fill_rows(residual, "normal", math.sqrt(wl.residual_var),
               _torch_gen(wl.seed, device, 2))

    gamma_np = rng.normal(wl.gamma_mean, math.sqrt(wl.gamma_var), size=H)
    gamma = torch.from_numpy(gamma_np.astype(np.float32)).to(torch.bfloat16).to(device)

    return {
        "workload": wl,
        "expert_out": expert_out,
        "permuted_row_of": torch.from_numpy(idx).to(device),
        "topk_weights": torch.from_numpy(w).to(device),
        "residual": residual,
        "gamma": gamma,
        "eps": float(wl.eps),
        "expert_of": expert_of,
        "outlier_rows": outlier_rows,
    }

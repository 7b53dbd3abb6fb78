"""Seeded synthetic workloads for speculative-sampling verification.

This module only draws random inputs: logits, uniforms and per-row draft
lengths.  It holds none of the verification arithmetic (no softmax, no
filtering, no sampling from p or q); draft tokens, which must be drawn from
the filtered draft law q, are produced by the caller with a sampler.

Every row has its own Philox stream (``SeedSequence(seed).spawn``), so any
subset of rows of a batch can be regenerated exactly without drawing the
rest.  Logits are float32 arrays, or uint16 arrays holding bfloat16 bit
patterns (round-to-nearest-even from float32).

Workloads (the pages' Pythia-2.8b / Pythia-70m decode on WikiText-2 is
stood in for by these seeded shapes and value distributions):

  0 "pr1"       B=1,    gamma=4, V=50304,  fp32, draft ~ N(0, 3^2),
                target = 0.9 draft + 0.436 N(0, 3^2); run greedy and at T=1.
  1 "mixed"     B=64,   gamma=4, V=50304,  fp32, T=1, top-k 50 then top-p 0.9;
                target = a draft + sqrt(1 - a^2) N(0, 3^2), a ~ U(0.6, 0.95) per row.
  2 "zipf"      B=256,  gamma=8, V=128256, bf16, T=0.8, top-p 0.95;
                draft = Zipf(1.1) log-frequency (fixed seeded rank permutation)
                + Gumbel(0, 1) + N(0, 1); target = draft + N(0, 1.5^2).
  3 "dirichlet" B=4096, gamma=4, V=1024,   fp32, T=1; p, q ~ Dirichlet(0.3)
                stored as log-probabilities (log 0 = -inf).
  4 "ragged"    B=512,  gamma_b ~ U{1..8} (gamma_max=8), V=152064, bf16,
                T=0.7, top-k 100 then top-p 0.9, logits as in 2, position
                stride padded to V + 64 elements.

Draft cascades (``cascade_levels``): between a batch's target t (level 0)
and draft d (level L), level l = 1 .. L-1 holds (1 - c) t + c d at the
drafted positions and t + c N(0, 3^2) at the last one, c = l / L, so each
level is closer to the target than the one below it; every stage after the
first gets fresh uniforms.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    gamma_max: int
    V: int
    dtype: str            # "f32" or "bf16"
    temperature: float
    top_k: int
    top_p: float
    kind: str             # logits recipe
    ragged: bool = False
    pos_pad: int = 0      # extra elements per position (padded stride)
    steps: int = 1        # verify steps the pages' workload runs
    extra: dict = field(default_factory=dict)


WORKLOADS = {
    0: Workload("pr1-B1-g4-V50304-f32", 1, 4, 50304, "f32", 1.0, 0, 1.0, "gauss09",
                steps=200),
    1: Workload("mixed-B64-g4-V50304-f32-k50-p0.9", 64, 4, 50304, "f32", 1.0, 50, 0.9,
                "gauss_alpha", steps=1000),
    2: Workload("zipf-B256-g8-V128256-bf16-T0.8-p0.95", 256, 8, 128256, "bf16", 0.8, 0, 0.95,
                "zipf"),
    3: Workload("dirichlet-B4096-g4-V1024-f32", 4096, 4, 1024, "f32", 1.0, 0, 1.0,
                "dirichlet", steps=245),
    4: Workload("ragged-B512-g1..8-V152064-bf16-T0.7-k100-p0.9", 512, 8, 152064, "bf16",
                0.7, 100, 0.9, "zipf", ragged=True, pos_pad=64),
}


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (nearest, ties to even); returns uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (u >> 16) & 1
    r = (u + np.uint32(0x7FFF) + lsb) >> 16
    nan = np.isnan(x)
    out = r.astype(np.uint16)
    if nan.any():
        out[nan] = 0x7FC0
    return out


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << 16).view(np.float32)


def _row_rngs(seed: int, B: int):
    return [np.random.Generator(np.random.Philox(s)) for s in np.random.SeedSequence(seed).spawn(B)]


def _zipf_logfreq(seed: int, V: int, s: float = 1.1) -> np.ndarray:
    """log of Zipf(s) frequency of each token id, ranks via a seeded permutation."""
    perm = np.random.Generator(np.random.Philox(np.random.SeedSequence([seed, 0x5A1F]))).permutation(V)
    lf = np.empty(V, np.float32)
    lf[perm] = (-s * np.log(np.arange(1, V + 1, dtype=np.float64))).astype(np.float32)
    return lf


def _gen_row(w: Workload, rng: np.random.Generator, logfreq, gm_b: int):
    """Target [gamma_max+1, V] and draft [gamma_max, V] float32 logits of one row."""
    G, V = w.gamma_max, w.V
    if w.kind == "gauss09":
        d = rng.standard_normal((G + 1, V), dtype=np.float32) * 3.0
        n = rng.standard_normal((G + 1, V), dtype=np.float32) * 3.0
        t = 0.9 * d + 0.436 * n
        return t, d[:G]
    if w.kind == "gauss_alpha":
        a = np.float32(rng.uniform(0.6, 0.95))
        d = rng.standard_normal((G + 1, V), dtype=np.float32) * 3.0
        n = rng.standard_normal((G + 1, V), dtype=np.float32) * 3.0
        t = a * d + np.float32(np.sqrt(1.0 - a * a)) * n
        return t, d[:G]
    if w.kind == "zipf":
        g = (-np.log(-np.log(rng.random((G + 1, V), dtype=np.float64)))).astype(np.float32)
        d = logfreq[None, :] + g + rng.standard_normal((G + 1, V), dtype=np.float32)
        t = d + 1.5 * rng.standard_normal((G + 1, V), dtype=np.float32)
        return t, d[:G]
    if w.kind == "dirichlet":
        alpha = np.full(V, 0.3)
        with np.errstate(divide="ignore"):
            t = np.log(rng.dirichlet(alpha, size=G + 1)).astype(np.float32)
            d = np.log(rng.dirichlet(alpha, size=G)).astype(np.float32)
        return t, d
    raise ValueError(w.kind)


def make_batch(w: Workload | int, seed: int, rows=None, threads: int | None = None) -> dict:
    """Generate a batch (or the given subset of its rows, in that order).

    Returns dict with: target [n, G+1, S] and draft [n, G, S] (float32 or
    uint16 bf16 bits; S = V + pos_pad, only the first V of each position are
    logits), uniforms [n, G+1, 2] float32 in [0, 1), draft_uniforms [n, G]
    float32 (for sampling draft tokens), gamma_per_row [n] int32 or None,
    plus the workload parameters.
    """
    if isinstance(w, int):
        w = WORKLOADS[w]
    rows = np.arange(w.B) if rows is None else np.asarray(rows)
    n, G, V, S = len(rows), w.gamma_max, w.V, w.V + w.pos_pad
    rngs = _row_rngs(seed, w.B)
    logfreq = _zipf_logfreq(seed, V) if w.kind == "zipf" else None
    bf = w.dtype == "bf16"
    target = np.zeros((n, G + 1, S), np.uint16 if bf else np.float32)
    draft = np.zeros((n, G, S), np.uint16 if bf else np.float32)
    uni = np.empty((n, G + 1, 2), np.float32)
    du = np.empty((n, G), np.float32)
    gam = np.empty(n, np.int32) if w.ragged else None

    def one(j):
        rng = rngs[int(rows[j])]
        # The order of draws is fixed: gamma, uniforms, draft uniforms, logits.
        gb = int(rng.integers(1, G + 1)) if w.ragged else G
        uni[j] = rng.random((G + 1, 2), dtype=np.float32)
        du[j] = rng.random(G, dtype=np.float32)
        t, d = _gen_row(w, rng, logfreq, gb)
        if bf:
            target[j, :, :V] = f32_to_bf16_bits(t)
            draft[j, :, :V] = f32_to_bf16_bits(d)
        else:
            target[j, :, :V] = t
            draft[j, :, :V] = d
        if gam is not None:
            gam[j] = gb

    nt = threads or min(16, os.cpu_count() or 1)
    if nt > 1 and n > 1:
        with ThreadPoolExecutor(nt) as ex:
            list(ex.map(one, range(n)))
    else:
        for j in range(n):
            one(j)
    return {"workload": w, "target": target, "draft": draft, "uniforms": uni,
            "draft_uniforms": du, "gamma_per_row": gam, "rows": rows}


def cascade_levels(batch: dict, n_levels: int, seed: int) -> dict:
    """Logits of the levels of a draft cascade built on a batch (see the
    module docstring): returns levels [target, level 1, ..., draft] (arrays
    in the batch's storage, intermediate levels shaped like the target) and
    uniforms [L, n, G+1, 2] (stage 0: the batch's own)."""
    w = batch["workload"]
    L = n_levels - 1
    if L < 1:
        raise ValueError("a cascade has at least two levels")
    bf = w.dtype == "bf16"
    tgt, drf = batch["target"], batch["draft"]
    n, G1, S = tgt.shape
    G, V = G1 - 1, w.V
    levels = [tgt] + [np.zeros_like(tgt) for _ in range(L - 1)] + [drf]
    uni = np.empty((L, n) + batch["uniforms"].shape[1:], np.float32)
    uni[0] = batch["uniforms"]
    dec = (lambda x: bf16_bits_to_f32(x)) if bf else (lambda x: x)
    enc = f32_to_bf16_bits if bf else (lambda x: x)
    for j, r in enumerate(batch["rows"]):
        rng = np.random.Generator(np.random.Philox(np.random.SeedSequence([seed, 0xCA5C, int(r)])))
        if L > 1:
            uni[1:, j] = rng.random((L - 1,) + batch["uniforms"].shape[1:], dtype=np.float32)
        t = dec(tgt[j, :, :V]).astype(np.float32)
        d = dec(drf[j, :, :V]).astype(np.float32)
        noise = rng.standard_normal(V, dtype=np.float32) * np.float32(3.0)
        for l in range(1, L):
            c = np.float32(l / L)
            m = np.empty((G1, V), np.float32)
            with np.errstate(invalid="ignore"):
                m[:G] = (np.float32(1) - c) * t[:G] + c * d
            m[G] = t[G] + c * noise
            levels[l][j, :, :V] = enc(m)
    return {"levels": levels, "uniforms": uni}

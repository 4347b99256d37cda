"""Seeded synthetic workloads shaped like the pages' verify / training batches.

This module only draws random inputs: logits, drafted tokens and uniforms.  It
holds none of the verify arithmetic (no softmax, overlap, acceptance or
residual), so the CUDA path and the fp64 oracle can both be fed from it without
sharing any of the method's code.

Drafted tokens are drawn from q = softmax(z_d / T) with the Gumbel-max trick
(argmax of z_d / T plus Gumbel noise), which samples q exactly without forming
it; at T == 0 the drafter is greedy (argmax z_d, first index on ties).

Recipes (vocabulary sizes are those of the Qwen and DeepSeek tokenizers the
pages discuss; K up to 7 drafted positions, batch 1..256):

* ``small``:    B=1, K=4, V=1024 fp32; z_t ~ N(0, 2^2); z_d = z_t + N(0, 0.5^2).
* ``entropy``:  B=32, K=4, V=151936 bf16; per row sigma in {1, 2, 4};
                z_t ~ N(0, sigma^2); z_d = z_t + N(0, 0.7^2).
* ``zipf``:     B=128, K=7, V=129280 bf16; z_t[v] = -1.1 ln(rank_v) + N(0, 0.3^2)
                with a random rank permutation per row; z_d = z_t except in
                20% of batch rows, where z_d is z_t permuted across v.
* ``e2e``:      B=256, K=7, V=151936 bf16; z_t ~ N(0, 2^2); z_d = z_t + N(0, 0.5^2).
* ``sweep``:    any B, K at V=151936 bf16; z_t ~ N(0, 2^2); z_d = z_t + N(0, 0.5^2).
"""

from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch


@dataclass
class Workload:
    """One batch of verify inputs (CPU tensors)."""

    name: str
    target: torch.Tensor        # [B, K+1, V] (verify) or [B, K, V] (overlap / E2E-TV)
    draft: torch.Tensor         # [B, K, V]
    draft_tokens: torch.Tensor  # int32 [B, K]
    u_accept: torch.Tensor      # float32 [B, K], in [0, 1)
    u_final: torch.Tensor       # float32 [B], in [0, 1)
    temperature: float          # exactly representable in float32

    @property
    def shape(self):
        B, K, V = self.draft.shape
        return B, K, V

    def nbytes(self):
        return self.target.numel() * self.target.element_size() + \
            self.draft.numel() * self.draft.element_size()


def f64(t: torch.Tensor) -> np.ndarray:
    """Exact float64 widening of a bf16 / fp32 tensor (for the oracle)."""
    return t.detach().to("cpu", torch.float64).numpy()


def fp32_temperature(t: float) -> float:
    """The temperature as the float32 value both implementations receive."""
    return float(np.float32(t))


def _round(x: np.ndarray, dtype: torch.dtype) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(dtype)


def _gumbel_draft(rng, zd: torch.Tensor, temperature: float) -> torch.Tensor:
    """Drafted tokens y ~ softmax(z_d / T) by Gumbel-max, row by row."""
    B, K, V = zd.shape
    out = np.empty((B, K), dtype=np.int32)
    z = zd.reshape(B * K, V)
    step = max(1, (1 << 22) // max(V, 1))
    for r0 in range(0, B * K, step):
        r1 = min(B * K, r0 + step)
        x = z[r0:r1].to(torch.float64).numpy()
        if temperature > 0:
            u = rng.random((r1 - r0, V))
            u = np.maximum(u, np.finfo(np.float64).tiny)
            x = x / temperature - np.log(-np.log(u))
        out.reshape(-1)[r0:r1] = np.argmax(x, axis=1)
    return torch.from_numpy(out)


def _uniforms(rng, B, K):
    ua = torch.from_numpy(rng.random((B, K), dtype=np.float32))
    uf = torch.from_numpy(rng.random((B,), dtype=np.float32))
    return ua, uf


def gaussian(B, K, V, *, sigma=2.0, noise=0.5, dtype=torch.bfloat16,
             temperature=1.0, seed=0, bonus=True, name="gaussian", draft_tokens=True):
    """z_t ~ N(0, sigma^2) (sigma a scalar or one value per batch row),
    z_d = z_t + N(0, noise^2); both rounded to ``dtype``.  With
    ``draft_tokens=False`` no tokens are drafted (all zero), as for the
    E2E-TV loss, which consumes logits only."""
    rng = np.random.Generator(np.random.PCG64(seed))
    KT = K + 1 if bonus else K
    sig = np.broadcast_to(np.asarray(sigma, dtype=np.float32).reshape(-1, 1, 1)
                          if np.ndim(sigma) else np.float32(sigma), (B, 1, 1))
    zt32 = rng.standard_normal((B, KT, V), dtype=np.float32) * sig
    zd32 = zt32[:, :K] + rng.standard_normal((B, K, V), dtype=np.float32) * np.float32(noise)
    target = _round(zt32, dtype)
    draft = _round(zd32, dtype)
    del zt32, zd32
    t = fp32_temperature(temperature)
    y = _gumbel_draft(rng, draft, t) if draft_tokens else torch.zeros((B, K), dtype=torch.int32)
    ua, uf = _uniforms(rng, B, K)
    return Workload(name, target, draft, y, ua, uf, t)


def small(seed=0, temperature=1.0):
    """B=1, K=4, V=1024 fp32 logits (one call of the latency-bound case)."""
    return gaussian(1, 4, 1024, sigma=2.0, noise=0.5, dtype=torch.float32,
                    temperature=temperature, seed=seed, name="small")


def entropy_mix(seed=0, temperature=1.0, B=32, K=4, V=151936):
    """Per-row sigma drawn from {1, 2, 4} to vary the target entropy;
    draft noise N(0, 0.7^2)."""
    rng = np.random.Generator(np.random.PCG64(seed + 7919))
    sig = rng.choice(np.array([1.0, 2.0, 4.0], dtype=np.float32), size=B)
    return gaussian(B, K, V, sigma=sig, noise=0.7, dtype=torch.bfloat16,
                    temperature=temperature, seed=seed, name="entropy")


def zipf(seed=0, B=128, K=7, V=129280, temperature=1.0, low_frac=0.2, bonus=True):
    """Zipf-shaped target logits -1.1 ln(rank) + N(0, 0.3^2) with a random
    rank permutation per row; the draft equals the target except in a
    ``low_frac`` share of batch rows, whose draft rows are the target rows
    permuted across the vocabulary (low overlap)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    KT = K + 1 if bonus else K
    base = (-1.1 * np.log(np.arange(1, V + 1, dtype=np.float64))).astype(np.float32)
    zt32 = np.empty((B, KT, V), dtype=np.float32)
    for b in range(B):
        for k in range(KT):
            zt32[b, k] = base[rng.permutation(V)]
    zt32 += rng.standard_normal((B, KT, V), dtype=np.float32) * np.float32(0.3)
    target = _round(zt32, torch.bfloat16)
    del zt32
    draft = target[:, :K].clone()
    n_low = int(round(low_frac * B))
    low_rows = rng.choice(B, size=n_low, replace=False) if n_low else np.array([], dtype=np.int64)
    for b in low_rows:
        for k in range(K):
            draft[b, k] = draft[b, k][torch.from_numpy(rng.permutation(V))]
    t = fp32_temperature(temperature)
    y = _gumbel_draft(rng, draft, t)
    ua, uf = _uniforms(rng, B, K)
    w = Workload("zipf", target, draft, y, ua, uf, t)
    w.low_rows = np.sort(low_rows)
    return w


def greedy_tokens(draft: torch.Tensor) -> torch.Tensor:
    """The tokens a greedy (T == 0) drafter proposes: argmax z_d per position,
    first index on ties."""
    return _gumbel_draft(None, draft, 0.0)


def e2e(seed=0, B=256, K=7, V=151936):
    """E2E-TV training batch: target and draft logits [B, K, V] (no bonus row)."""
    return gaussian(B, K, V, sigma=2.0, noise=0.5, dtype=torch.bfloat16,
                    temperature=1.0, seed=seed, bonus=False, name="e2e", draft_tokens=False)


def sweep(B, K, seed=0, V=151936):
    """One point of the batch x K sweep."""
    return gaussian(B, K, V, sigma=2.0, noise=0.5, dtype=torch.bfloat16,
                    temperature=1.0, seed=seed, name=f"sweep_B{B}_K{K}")

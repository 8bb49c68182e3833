"""Seeded synthetic KV-cache workloads.

This module only draws random numbers: it holds none of the codec's
arithmetic and is shared by the tests (which feed its tensors to both the
CUDA library and the CPU oracle) and by ``bench.py``.

Every tensor is ``x = mu + z diag(sqrt(lam)) Qb^T`` with ``z ~ N(0, I)``,
``Qb`` a random orthogonal basis (QR of a Gaussian, columns signed by the
diagonal of R) and ``lam_j = decay^j`` -- the Llama-3.1-8B / Qwen-2.5-7B
attention shapes of the workloads this library targets, with synthetic
statistics in place of real model caches (no weights or datasets are used).
``mu``, ``Qb`` and the outlier channels are fixed per (workload, layer,
tensor, head) and shared by the calibration rows, the cache rows and the
decode queries; ``z`` is drawn independently for each role.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import torch

BASE_SEED = 20261202
TENSOR = {"k": 0, "v": 1, "q": 2}
ROLE = {"calib": 0, "cache": 1, "query": 2, "params": 3}


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    index: int                 # workload number, part of every seed
    n_q_heads: int
    n_kv_heads: int
    batch: int
    seq_len: int               # cached tokens per batch row
    n_calib: int               # calibration tokens per head
    decay: float               # lam_j = decay ** j
    bits: float                # average bits per element
    dtype: torch.dtype
    mu_std: tuple = (1.0, 1.0, 1.0)    # std of the per-channel mean for (k, v, q)
    k_scaled_outliers: int = 0         # channels of K multiplied by 10
    k_heavy_outliers: int = 0          # channels of K replaced by 10 * Student-t(3)
    layers: int = 1
    head_dim: int = 128

    @property
    def group(self) -> int:
        return self.n_q_heads // self.n_kv_heads


WORKLOADS = {
    # one head, fp32: small enough for the oracle to finish in seconds
    "tiny": Workload("tiny", 1, n_q_heads=16, n_kv_heads=1, batch=1, seq_len=1024, n_calib=512,
                     decay=0.9, bits=2.75, dtype=torch.float32, k_scaled_outliers=4),
    # Llama-3.1-8B-shaped layer, batch 1 at 32k context
    "llama_32k": Workload("llama_32k", 2, n_q_heads=32, n_kv_heads=8, batch=1, seq_len=32768,
                          n_calib=4096, decay=0.95, bits=2.75, dtype=torch.bfloat16),
    # Llama-3.1-8B-shaped layer, batch 16 x 8k, heavy-tailed K outlier channels
    "llama_b16_8k": Workload("llama_b16_8k", 3, n_q_heads=32, n_kv_heads=8, batch=16, seq_len=8192,
                             n_calib=4096, decay=0.95, bits=2.75, dtype=torch.bfloat16,
                             mu_std=(0.0, 0.0, 0.0), k_heavy_outliers=3),
    # Qwen-2.5-7B-shaped layer, batch 4 x 128k, nonzero key mean with variance 4
    "qwen_128k": Workload("qwen_128k", 4, n_q_heads=28, n_kv_heads=4, batch=4, seq_len=131072,
                          n_calib=4096, decay=0.93, bits=2.75, dtype=torch.bfloat16,
                          mu_std=(2.0, 0.0, 0.0)),
    # 32-layer Llama-3.1-8B-shaped stack; bits and seq_len are swept
    "llama_stack": Workload("llama_stack", 5, n_q_heads=32, n_kv_heads=8, batch=1, seq_len=32768,
                            n_calib=4096, decay=0.95, bits=2.75, dtype=torch.bfloat16,
                            mu_std=(0.0, 0.0, 0.0), layers=32),
}


def seed_of(wl: Workload, layer: int, tensor: str, head: int, role: str, batch: int = 0) -> int:
    s = wl.index
    for v, m in ((layer, 64), (head, 128), (TENSOR[tensor], 4), (ROLE[role], 4), (batch, 64)):
        s = s * m + v
    return BASE_SEED + s


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


@dataclasses.dataclass
class HeadParams:
    mu: torch.Tensor        # [d] float32
    basis: torch.Tensor     # [d][d] float32, orthogonal
    scale: torch.Tensor     # [d] float32 = sqrt(lam)
    outliers: torch.Tensor  # int64 channel indices (may be empty)


def head_params(wl: Workload, layer: int, tensor: str, head: int) -> HeadParams:
    """Distribution parameters of one head, drawn on the CPU in float64."""
    d = wl.head_dim
    g = _gen(seed_of(wl, layer, tensor, head, "params"), "cpu")
    mu = torch.randn(d, generator=g, dtype=torch.float64) * wl.mu_std[TENSOR[tensor]]
    A = torch.randn(d, d, generator=g, dtype=torch.float64)
    Qm, Rm = torch.linalg.qr(A)
    Qm = Qm * torch.sign(torch.diagonal(Rm)).unsqueeze(0)
    scale = torch.tensor([wl.decay ** j for j in range(d)], dtype=torch.float64).sqrt()
    n_out = wl.k_scaled_outliers + wl.k_heavy_outliers if tensor == "k" else 0
    outl = torch.randperm(d, generator=g)[:n_out].sort().values
    return HeadParams(mu.float(), Qm.float(), scale.float(), outl)


def _draw(wl: Workload, p: HeadParams, n: int, seed: int, device) -> torch.Tensor:
    g = _gen(seed, device)
    z = torch.randn(n, wl.head_dim, generator=g, device=device, dtype=torch.float32)
    x = (z * p.scale.to(device)) @ p.basis.to(device).T + p.mu.to(device)
    if p.outliers.numel():
        idx = p.outliers.to(device)
        if wl.k_scaled_outliers:
            x[:, idx] *= 10.0
        if wl.k_heavy_outliers:
            zz = torch.randn(n, idx.numel(), generator=g, device=device)
            chi = torch.randn(n, idx.numel(), 3, generator=g, device=device).pow(2).sum(-1) / 3.0
            x[:, idx] = 10.0 * zz / chi.sqrt()
    return x.to(wl.dtype)


def calib_inputs(wl: Workload, layer: int = 0, device="cpu", n_calib: Optional[int] = None):
    """(k_cal, v_cal [H_kv][N][d], q_cal [H_q][N][d]) in the workload dtype."""
    N = n_calib or wl.n_calib
    out = []
    for t, H in (("k", wl.n_kv_heads), ("v", wl.n_kv_heads), ("q", wl.n_q_heads)):
        out.append(torch.stack([_draw(wl, head_params(wl, layer, t, h), N,
                                      seed_of(wl, layer, t, h, "calib"), device)
                                for h in range(H)]))
    return tuple(out)


def cache_inputs(wl: Workload, layer: int = 0, device="cpu", seq_len: Optional[int] = None,
                 batch: Optional[int] = None, tensors=("k", "v")):
    """Cache rows [B][H_kv][L][d] for each requested tensor ('k', 'v')."""
    L = seq_len if seq_len is not None else wl.seq_len
    Bsz = batch if batch is not None else wl.batch
    res = []
    for t in tensors:
        x = torch.empty(Bsz, wl.n_kv_heads, L, wl.head_dim, dtype=wl.dtype, device=device)
        for h in range(wl.n_kv_heads):
            p = head_params(wl, layer, t, h)
            for b in range(Bsz):
                x[b, h] = _draw(wl, p, L, seed_of(wl, layer, t, h, "cache", b), device)
        res.append(x)
    return tuple(res)


def query_inputs(wl: Workload, layer: int = 0, device="cpu", batch: Optional[int] = None,
                 step: int = 0):
    """Decode queries [B][H_q][d]; `step` selects an independent draw."""
    Bsz = batch if batch is not None else wl.batch
    q = torch.empty(Bsz, wl.n_q_heads, wl.head_dim, dtype=wl.dtype, device=device)
    for h in range(wl.n_q_heads):
        p = head_params(wl, layer, "q", h)
        for b in range(Bsz):
            q[b, h] = _draw(wl, p, 1, seed_of(wl, layer, "q", h, "query", b) + 7919 * step,
                            device)[0]
    return q

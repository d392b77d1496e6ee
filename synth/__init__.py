"""Seeded synthetic Q, K, V for the attention configurations.

This module draws inputs only; it holds none of the attention method's arithmetic, so both the
CUDA path and the CPU oracle can be fed from it.

Recipe (one batch, bf16 [B, H, S, D], token index t-major over a T x Hg x Wg space-time grid):
  * field F[t, c], c < 128: a sum of 8 low-frequency 3-D cosine modes per channel,
    sum_m A_m cos(2 pi (k_tau tau/T + k_y y/Hg + k_x x/Wg) + phi_m), k_* in {0,1,2} not all zero,
    A_m ~ N(0, 1), phi_m ~ U[0, 2 pi), plus N(0, 0.5^2) noise (0.5 read as the standard deviation);
  * per head independent Gaussian projections W ~ N(0, 1/128) of shape 128 x D; Q = F W_Q, etc.;
  * locality (video-like configs): W_K = (W_Q + 0.5 G)/sqrt(1.25), so keys near a query's own
    space-time position tend to score highest;
  * Q and K are scaled by sqrt(target/sigma) each, sigma the std of q.k/sqrt(D) over 4096 random
    pairs, so the pre-softmax scores have std ~target (3; 0.5 for the "near-uniform" heads);
  * V outliers: round(frac*S) tokens without replacement per head, each with a fresh random
    8-channel subset multiplied by `mult`;
  * finally every tensor is rounded to bf16.
These stand in for the captured post-RoPE activations of the video models the pages measure on,
which are not available here.
"""
from __future__ import annotations

import math

import numpy as np
import torch

CONFIGS: dict[str, dict] = {
    "tiny": dict(B=1, H=1, S=1024, D=128, grid=(4, 16, 16), k=8, iters=3, locality=False,
                 outlier_frac=0.005, outlier_mult=30.0, uniform_heads=0.0),
    "small": dict(B=1, H=8, S=8192, D=128, grid=(8, 32, 32), k=64, iters=4, locality=False,
                  outlier_frac=0.005, outlier_mult=30.0, uniform_heads=0.0),
    "wan": dict(B=1, H=40, S=75600, D=128, grid=(21, 45, 80), k=591, iters=4, locality=True,
                outlier_frac=0.005, outlier_mult=30.0, uniform_heads=0.0),
    "l1344": dict(B=1, H=48, S=64512, D=128, grid=(16, 48, 84), k=504, iters=4, locality=True,
                  outlier_frac=0.01, outlier_mult=50.0, uniform_heads=0.1),
}
SWEEP_S = (4096, 16384, 32768, 65536, 131072)
SWEEP_D = (64, 128)
for _d in SWEEP_D:
    for _s in SWEEP_S:
        CONFIGS[f"sweep_d{_d}_s{_s}"] = dict(B=1, H=16, S=_s, D=_d, grid=(_s // 1024, 32, 32), k=_s // 128, iters=4,
                                             locality=False, outlier_frac=0.005, outlier_mult=30.0,
                                             uniform_heads=0.0)


def config(name: str, **override) -> dict:
    cfg = dict(CONFIGS[name])
    cfg.update(override)
    cfg["name"] = name
    return cfg


def custom(S: int, D: int = 128, H: int = 1, B: int = 1, k: int | None = None, iters: int = 3,
           locality: bool = False, outlier_frac: float = 0.005, outlier_mult: float = 30.0,
           uniform_heads: float = 0.0) -> dict:
    """A config of arbitrary length (ragged tails, edge cases); the grid is 1 x 1 x S."""
    return dict(name=f"custom_s{S}_d{D}", B=B, H=H, S=S, D=D, grid=(1, 1, S), k=k or max(1, S // 128), iters=iters,
                locality=locality, outlier_frac=outlier_frac, outlier_mult=outlier_mult,
                uniform_heads=uniform_heads)


def _field(rng: np.random.Generator, grid, C: int = 128, n_modes: int = 8) -> np.ndarray:
    T, Hg, Wg = grid
    S = T * Hg * Wg
    idx = np.arange(S)
    tau = (idx // (Hg * Wg)) / T
    yy = ((idx // Wg) % Hg) / Hg
    xx = (idx % Wg) / Wg
    kk = rng.integers(0, 3, size=(C, n_modes, 3))
    zero = kk.sum(axis=2) == 0
    kk[zero, rng.integers(0, 3, size=int(zero.sum()))] = 1
    amp = rng.normal(size=(C, n_modes))
    phi = rng.uniform(0.0, 2.0 * math.pi, size=(C, n_modes))
    F = np.zeros((S, C), dtype=np.float32)
    for c in range(C):
        ph = 2.0 * math.pi * (np.outer(tau, kk[c, :, 0]) + np.outer(yy, kk[c, :, 1]) + np.outer(xx, kk[c, :, 2]))
        F[:, c] = (amp[c] * np.cos(ph + phi[c])).sum(axis=1).astype(np.float32)
    F += rng.normal(0.0, 0.5, size=(S, C)).astype(np.float32)
    return F


def make_inputs(cfg: dict, seed: int = 0, device="cpu"):
    """Return (Q, K, V) bf16 tensors [B, H, S, D] on `device`, fully determined by (cfg, seed)."""
    rng = np.random.default_rng(seed)
    B, H, S, D = cfg["B"], cfg["H"], cfg["S"], cfg["D"]
    T, Hg, Wg = cfg["grid"]
    assert T * Hg * Wg == S, "grid must cover the sequence"
    dev = torch.device(device)
    Q = torch.empty((B, H, S, D), dtype=torch.bfloat16, device=dev)
    K = torch.empty_like(Q)
    V = torch.empty_like(Q)
    n_uniform = int(round(cfg["uniform_heads"] * H))
    for b in range(B):
        F = torch.from_numpy(_field(rng, cfg["grid"])).to(dev)
        uniform = set(rng.choice(H, size=n_uniform, replace=False).tolist()) if n_uniform else set()
        for h in range(H):
            wq = rng.normal(0.0, 1.0 / math.sqrt(128.0), size=(128, D)).astype(np.float32)
            if cfg["locality"]:
                g = rng.normal(0.0, 1.0 / math.sqrt(128.0), size=(128, D)).astype(np.float32)
                wk = ((wq + 0.5 * g) / math.sqrt(1.25)).astype(np.float32)
            else:
                wk = rng.normal(0.0, 1.0 / math.sqrt(128.0), size=(128, D)).astype(np.float32)
            wv = rng.normal(0.0, 1.0 / math.sqrt(128.0), size=(128, D)).astype(np.float32)
            q = F @ torch.from_numpy(wq).to(dev)
            k = F @ torch.from_numpy(wk).to(dev)
            v = F @ torch.from_numpy(wv).to(dev)
            ia = torch.from_numpy(rng.integers(0, S, size=4096)).to(dev)
            ib = torch.from_numpy(rng.integers(0, S, size=4096)).to(dev)
            sig = float(((q[ia] * k[ib]).sum(dim=1) / math.sqrt(D)).std().item())
            target = 0.5 if h in uniform else 3.0
            # a one-token sequence has no score spread to normalise: leave the projections as drawn
            f = math.sqrt(target / sig) if sig > 1e-6 else 1.0
            q = q * f
            k = k * f
            n_out = int(round(cfg["outlier_frac"] * S))
            if n_out:
                toks = rng.choice(S, size=n_out, replace=False)
                chans = np.stack([rng.choice(D, size=min(8, D), replace=False) for _ in range(n_out)])
                t_idx = torch.from_numpy(np.repeat(toks, chans.shape[1])).to(dev)
                c_idx = torch.from_numpy(chans.reshape(-1)).to(dev)
                v[t_idx, c_idx] = v[t_idx, c_idx] * cfg["outlier_mult"]
            Q[b, h] = q.to(torch.bfloat16)
            K[b, h] = k.to(torch.bfloat16)
            V[b, h] = v.to(torch.bfloat16)
    return Q, K, V


def flops(cfg: dict) -> float:
    """Attention FLOPs of one forward, 4 B H S^2 D (the QK^T and PV products)."""
    return 4.0 * cfg["B"] * cfg["H"] * float(cfg["S"]) ** 2 * cfg["D"]

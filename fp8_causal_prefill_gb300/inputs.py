"""Seeded synthetic inputs for causal prefill attention (shared by the tests, the bench and the smoke run).

This module holds no arithmetic of the attention method: it draws Q/K/V, applies the per-tensor FP8
quantisation that precedes the kernel (descale = amax/448, round-to-nearest-even into e4m3 by the
PyTorch cast), rounds to bfloat16 for the BF16 twin, and reports one statistic of the drawn scores.

Workloads (stand-ins for the pages' Gaussian kernel benchmarks and captured model activations, which
need trained weights and are not available here):

* ``gaussian``: Q, K, V ~ N(0, 1), drawn in that order from ``numpy.random.default_rng(seed)``.
* ``mistral``: Q, K ~ N(0, 1), then per KV head 4 outlier channels (``rng.choice(D, 4)``) scaled by 12
  in K and in every query head of its group, then a rotary rotation of channel pairs (2i, 2i+1) by
  ``pos * 10000^(-2i/D)``, then quantisation.  V ~ N(0, 1).  This reproduces the property the pages
  report for Mistral-7B layer 20: most (row, 64-key block) pairs sit more than 8 binades below the
  row maximum (captivela ZYFA article, "Tiga Trik": 91%).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

E4M3_MAX = 448.0


@dataclass(frozen=True)
class Shape:
    B: int
    S: int
    H: int
    H_kv: int
    D_qk: int
    D_v: int
    kind: str = "gaussian"

    @property
    def causal_flops(self) -> float:
        """Algorithmic causal FLOPs, B*H*S^2*(D_qk+D_v): half the dense count."""
        return float(self.B) * self.H * self.S * self.S * (self.D_qk + self.D_v)


CONFIGS = {
    "tiny": Shape(1, 256, 2, 2, 64, 64),
    "gqa4k": Shape(1, 4096, 32, 8, 128, 128),
    "mistral16k": Shape(1, 16384, 32, 8, 128, 128, "mistral"),
    "bench32k": Shape(1, 32768, 32, 8, 128, 128),
    "mla32k": Shape(1, 32768, 16, 16, 192, 128),
}


@dataclass
class Problem:
    shape: Shape
    seed: int
    q: np.ndarray = field(repr=False)          # fp32 draws [B,S,H,Dqk]
    k: np.ndarray = field(repr=False)
    v: np.ndarray = field(repr=False)
    q8: torch.Tensor = field(repr=False)       # uint8 e4m3 codes, CPU
    k8: torch.Tensor = field(repr=False)
    v8: torch.Tensor = field(repr=False)
    dq: float = 1.0
    dk: float = 1.0
    dv: float = 1.0
    qb: torch.Tensor | None = field(default=None, repr=False)   # bfloat16, CPU
    kb: torch.Tensor | None = field(default=None, repr=False)
    vb: torch.Tensor | None = field(default=None, repr=False)


def quantize_e4m3(x: np.ndarray):
    """Per-tensor FP8 quantisation: descale = amax/448 (fp32), codes = e4m3_rn(x / descale)."""
    amax = np.float32(np.max(np.abs(x))) if x.size else np.float32(0)
    descale = np.float32(amax / np.float32(E4M3_MAX)) if amax > 0 else np.float32(1.0)
    scaled = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)) / torch.tensor(descale)
    codes = scaled.to(torch.float8_e4m3fn).view(torch.uint8).contiguous()
    return codes, float(descale)


def _rotary(x: np.ndarray) -> np.ndarray:
    """Rotate channel pairs (2i, 2i+1) of x [B,S,H,D] by pos * 10000^(-2i/D)."""
    b_, s_, h_, d_ = x.shape
    pos = np.arange(s_, dtype=np.float64)[:, None]
    inv = 10000.0 ** (-np.arange(0, d_, 2, dtype=np.float64) / d_)
    ang = pos * inv[None, :]                                        # [S, D/2]
    c = np.cos(ang).astype(np.float32)[None, :, None, :]
    s = np.sin(ang).astype(np.float32)[None, :, None, :]
    xe, xo = x[..., 0::2], x[..., 1::2]
    out = np.empty_like(x)
    out[..., 0::2] = xe * c - xo * s
    out[..., 1::2] = xe * s + xo * c
    return out


def make_problem(shape: Shape, seed: int = 0, bf16: bool = True, fp8: bool = True) -> Problem:
    rng = np.random.default_rng(seed)
    sh = shape
    q = rng.standard_normal((sh.B, sh.S, sh.H, sh.D_qk), dtype=np.float32)
    k = rng.standard_normal((sh.B, sh.S, sh.H_kv, sh.D_qk), dtype=np.float32)
    v = rng.standard_normal((sh.B, sh.S, sh.H_kv, sh.D_v), dtype=np.float32)
    if sh.kind == "mistral":
        group = sh.H // sh.H_kv
        for hk in range(sh.H_kv):
            ch = rng.choice(sh.D_qk, 4, replace=False)
            k[:, :, hk, ch] *= 12.0
            for g in range(group):
                q[:, :, hk * group + g, ch] *= 12.0
        q = _rotary(q)
        k = _rotary(k)
    elif sh.kind != "gaussian":
        raise ValueError(f"unknown workload kind {sh.kind!r}")
    empty = torch.empty(0, dtype=torch.uint8)
    q8, dq = quantize_e4m3(q) if fp8 else (empty, 1.0)
    k8, dk = quantize_e4m3(k) if fp8 else (empty, 1.0)
    v8, dv = quantize_e4m3(v) if fp8 else (empty, 1.0)
    p = Problem(sh, seed, q, k, v, q8, k8, v8, dq, dk, dv)
    if bf16:
        p.qb = torch.from_numpy(q).to(torch.bfloat16)
        p.kb = torch.from_numpy(k).to(torch.bfloat16)
        p.vb = torch.from_numpy(v).to(torch.bfloat16)
    return p


def sample_rows(S: int, n_random: int = 512, edge: int = 128, seed: int = 1) -> np.ndarray:
    """Rows checked at long sequence lengths: the first and last ``edge`` rows plus seeded random rows."""
    rng = np.random.default_rng(seed)
    rows = set(range(min(edge, S))) | set(range(max(0, S - edge), S))
    if S > 2 * edge:
        rows |= set(rng.choice(np.arange(edge, S - edge), size=min(n_random, S - 2 * edge),
                               replace=False).tolist())
    return np.array(sorted(rows), dtype=np.int64)


def far_block_fraction(p: Problem, rows: np.ndarray, head: int = 0, binades: float = 8.0,
                       block: int = 64) -> float:
    """Fraction of (row, 64-key block) pairs whose largest probability lies more than ``binades``
    binades below the row's largest probability, from float64 scores of the fp32 draws."""
    sh = p.shape
    scale = 1.0 / math.sqrt(sh.D_qk)
    kh = head // (sh.H // sh.H_kv)
    far = total = 0
    for i in rows:
        n = int(i) + 1
        s = (p.q[0, i, head, :].astype(np.float64) @ p.k[0, :n, kh, :].astype(np.float64).T) * scale
        y = s * math.log2(math.e)
        nb = -(-n // block)
        padded = np.full(nb * block, -np.inf)
        padded[:n] = y
        bmax = padded.reshape(nb, block).max(axis=1)
        far += int(np.sum(bmax < y.max() - binades))
        total += nb
    return far / max(total, 1)

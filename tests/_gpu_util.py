"""Helpers shared by the GPU tests: run the CUDA path through the public binding and evaluate the oracle
on the same seeded inputs."""
from __future__ import annotations

import numpy as np
import torch

import oracle as O
from fp8_causal_prefill_gb300 import flash_attn_func
from fp8_causal_prefill_gb300.inputs import Problem

FP8_TOL = 1e-2     # relative L2 against the Lean-P emulation (O2)
BF16_TOL = 4e-3    # relative L2 against the BF16 emulation (O4)


def to_device(p: Problem, dtype: str, device="cuda"):
    if dtype == "fp8":
        q, k, v = (t.to(device).view(torch.float8_e4m3fn) for t in (p.q8, p.k8, p.v8))
        ds = [torch.tensor([d], dtype=torch.float32, device=device) for d in (p.dq, p.dk, p.dv)]
        return q, k, v, ds
    return p.qb.to(device), p.kb.to(device), p.vb.to(device), [None, None, None]


def run_gpu(p: Problem, dtype: str, scale=None) -> torch.Tensor:
    q, k, v, ds = to_device(p, dtype)
    out = flash_attn_func(q, k, v, softmax_scale=scale, q_descale=ds[0], k_descale=ds[1], v_descale=ds[2])
    torch.cuda.synchronize()
    return out


def scale_of(p: Problem, scale=None) -> float:
    return O.default_softmax_scale(p.shape.D_qk) if not scale else float(np.float32(scale))


def oracle_out(p: Problem, dtype: str, rows=None, heads=None, scale=None) -> np.ndarray:
    sc = scale_of(p, scale)
    if dtype == "fp8":
        return O.leanp_causal_attention(p.q8.numpy(), p.k8.numpy(), p.v8.numpy(), p.dq, p.dk, p.dv, sc,
                                        rows=rows, heads=heads)
    f = lambda t: t.float().numpy().astype(np.float64)  # noqa: E731
    return O.bf16_causal_attention(f(p.qb), f(p.kb), f(p.vb), sc, rows=rows, heads=heads)


def select(out: torch.Tensor, rows=None, heads=None) -> np.ndarray:
    x = out.float().cpu().numpy().astype(np.float64)
    if rows is not None:
        x = x[:, rows]
    if heads is not None:
        x = x[:, :, heads]
    return x


def per_row_rel(x: np.ndarray, ref: np.ndarray) -> np.ndarray:
    num = np.linalg.norm((x - ref).reshape(-1, x.shape[-1]), axis=1)
    den = np.linalg.norm(ref.reshape(-1, ref.shape[-1]), axis=1)
    return num / np.maximum(den, 1e-30)

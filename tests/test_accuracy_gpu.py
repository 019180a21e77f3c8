"""Accuracy against float64 attention, reported per workload beside the plain FP8 comparator.

For every workload the CUDA output is compared with exact float64 attention on the same dequantised
inputs (O1), next to the error of the Lean-P emulation itself (O2, the FP8 parity target) and of a
plain exact-exponential FP8 path that divides by the unrounded sum (O3).  The pages report lower
error for their method on captured activations against another library; on synthetic inputs the
numbers are reported, and the gate is only that the CUDA path's error is the emulation's error (the
kernel adds no error of its own beyond the parity tolerance).  Run with ``-s`` to see the table.
"""
import numpy as np
import pytest

import oracle as O
from _gpu_util import run_gpu, scale_of, select
from fp8_causal_prefill_gb300.inputs import CONFIGS, make_problem, sample_rows

pytestmark = pytest.mark.gpu

CASES = [("tiny", None), ("gqa4k", [0, 17]), ("mistral16k", [0, 31]), ("bench32k", [0, 31]), ("mla32k", [0, 15])]


def _per_head(p, h, rows, dtype):
    """O1 / O2 / O3 (FP8) or O1 / O4 (BF16) for one query head on the given rows."""
    sh = p.shape
    hk = h // (sh.H // sh.H_kv)
    sc = scale_of(p)
    if dtype == "fp8":
        q8, k8, v8 = (t.numpy()[:, :, [hh]] for t, hh in ((p.q8, h), (p.k8, hk), (p.v8, hk)))
        o1 = O.exact_causal_attention(O.dequant_e4m3(q8, p.dq), O.dequant_e4m3(k8, p.dk), O.dequant_e4m3(v8, p.dv),
                                      sc, rows=rows)
        o2 = O.leanp_causal_attention(q8, k8, v8, p.dq, p.dk, p.dv, sc, rows=rows)
        o3 = O.plain_fp8_causal_attention(q8, k8, v8, p.dq, p.dk, p.dv, sc, rows=rows)
        return o1, o2, o3
    f = lambda t, hh: t.float().numpy().astype(np.float64)[:, :, [hh]]  # noqa: E731
    qb, kb, vb = f(p.qb, h), f(p.kb, hk), f(p.vb, hk)
    return O.exact_causal_attention(qb, kb, vb, sc, rows=rows), O.bf16_causal_attention(qb, kb, vb, sc, rows=rows)


@pytest.mark.parametrize("dtype", ["fp8", "bf16"])
@pytest.mark.parametrize("name,heads", CASES, ids=[c[0] for c in CASES])
def test_error_vs_float64_beside_plain_fp8(name, heads, dtype):
    if name == "mistral16k" and dtype == "bf16":
        pytest.skip("the captured-activation stand-in is an FP8 workload")
    p = make_problem(CONFIGS[name], seed=0, bf16=(dtype == "bf16"), fp8=(dtype == "fp8"))
    out = run_gpu(p, dtype)
    sh = p.shape
    rows = sample_rows(sh.S) if sh.S > 4096 else np.arange(sh.S)
    heads = heads if heads is not None else list(range(sh.H))
    gpu = select(out, rows=rows, heads=heads)
    parts = [_per_head(p, h, rows, dtype) for h in heads]
    o1 = np.concatenate([x[0] for x in parts], axis=2)
    if dtype == "fp8":
        o2 = np.concatenate([x[1] for x in parts], axis=2)
        o3 = np.concatenate([x[2] for x in parts], axis=2)
        e_gpu, e_o2, e_o3 = O.rel_l2(gpu, o1), O.rel_l2(o2, o1), O.rel_l2(o3, o1)
        print(f"\n[accuracy] {name} fp8: rel-L2 vs float64  cuda {e_gpu:.4e}  lean-P emulation {e_o2:.4e}  "
              f"plain fp8 {e_o3:.4e}  cuda-vs-emulation {O.rel_l2(gpu, o2):.4e}")
        assert abs(e_gpu - e_o2) <= 0.1 * e_o2 + 1e-3
        assert e_gpu < 0.06 and e_o3 < 0.06
    else:
        o4 = np.concatenate([x[1] for x in parts], axis=2)
        e_gpu, e_o4 = O.rel_l2(gpu, o1), O.rel_l2(o4, o1)
        print(f"\n[accuracy] {name} bf16: rel-L2 vs float64  cuda {e_gpu:.4e}  bf16 emulation {e_o4:.4e}")
        assert abs(e_gpu - e_o4) <= 0.2 * e_o4 + 1e-3
        assert e_gpu < 1e-2

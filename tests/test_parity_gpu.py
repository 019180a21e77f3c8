"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle, element by element.

FP8 is compared with the Lean-P emulation (O2), BF16 with the BF16 emulation (O4), by relative L2 over
all compared outputs (1e-2 and 4e-3), plus a per-row bound that catches localised faults.  Small shapes
are compared in full; the full-size workloads are compared on a seeded sample of rows (the first and
last 128 rows plus 512 random rows) in two heads, in the same launch configuration the bench times.
"""
import numpy as np
import pytest
import torch

import oracle as O
from _gpu_util import BF16_TOL, FP8_TOL, oracle_out, per_row_rel, run_gpu, scale_of, select, to_device
from fp8_causal_prefill_gb300 import flash_attn_func, zyfa_check_errors
from fp8_causal_prefill_gb300.inputs import CONFIGS, Shape, make_problem, sample_rows

pytestmark = pytest.mark.gpu

TOL = {"fp8": FP8_TOL, "bf16": BF16_TOL}
ROW_TOL = {"fp8": 5e-2, "bf16": 2e-2}

SMALL = [
    Shape(1, 1, 1, 1, 128, 128),
    Shape(1, 2, 2, 1, 128, 128),
    Shape(1, 63, 2, 2, 128, 128),
    Shape(1, 64, 2, 1, 128, 128),
    Shape(1, 65, 3, 1, 128, 128),
    Shape(1, 127, 2, 2, 128, 128),
    Shape(1, 128, 2, 2, 128, 128),
    Shape(1, 129, 2, 1, 128, 128),
    Shape(1, 255, 2, 2, 128, 128),
    Shape(1, 256, 2, 2, 128, 128),
    Shape(1, 257, 4, 2, 128, 128),
    Shape(1, 385, 2, 1, 128, 128),
    Shape(2, 520, 2, 2, 128, 128),
    Shape(2, 383, 4, 1, 128, 128),
    Shape(1, 1000, 4, 4, 128, 128),
    Shape(1, 256, 2, 2, 64, 64),
    Shape(2, 333, 3, 1, 64, 64),
    Shape(1, 1, 2, 2, 192, 128),
    Shape(1, 130, 2, 2, 192, 128),
    Shape(1, 513, 2, 1, 192, 128),
    Shape(1, 300, 4, 4, 192, 128),
    Shape(1, 2048, 4, 1, 128, 128, "mistral"),
]


def _id(s):
    return f"B{s.B}S{s.S}H{s.H}kv{s.H_kv}D{s.D_qk}-{s.D_v}{'-m' if s.kind != 'gaussian' else ''}"


@pytest.mark.parametrize("dtype", ["fp8", "bf16"])
@pytest.mark.parametrize("shape", SMALL, ids=_id)
def test_small_shapes_full_compare(shape, dtype):
    p = make_problem(shape, seed=shape.S + 17 * shape.H)
    out = run_gpu(p, dtype)
    assert zyfa_check_errors() == 0
    got = select(out)
    ref = oracle_out(p, dtype)
    assert np.all(np.isfinite(got))
    err = O.rel_l2(got, ref)
    assert err <= TOL[dtype], err
    assert per_row_rel(got, ref).max() <= ROW_TOL[dtype]


@pytest.mark.parametrize("dtype", ["fp8", "bf16"])
def test_tiny_config_and_explicit_scale(dtype):
    p = make_problem(CONFIGS["tiny"], seed=0)
    got = select(run_gpu(p, dtype, scale=0.125))
    ref = oracle_out(p, dtype, scale=0.125)
    assert O.rel_l2(got, ref) <= TOL[dtype]
    got2 = select(run_gpu(p, dtype, scale=0.3))
    ref2 = oracle_out(p, dtype, scale=0.3)
    assert O.rel_l2(got2, ref2) <= TOL[dtype]


@pytest.mark.parametrize("dtype", ["fp8", "bf16"])
def test_gqa4k_all_rows_four_heads(dtype):
    p = make_problem(CONFIGS["gqa4k"], seed=0)
    out = run_gpu(p, dtype)
    heads = [0, 5, 18, 31]
    got = select(out, heads=heads)
    ref = oracle_out(p, dtype, heads=heads)
    assert O.rel_l2(got, ref) <= TOL[dtype]
    assert per_row_rel(got, ref).max() <= ROW_TOL[dtype]
    assert torch.isfinite(out.float()).all()


@pytest.mark.parametrize("name,dtype", [("mistral16k", "fp8"), ("mistral16k", "bf16"), ("bench32k", "fp8"),
                                        ("bench32k", "bf16"), ("mla32k", "fp8"), ("mla32k", "bf16")])
def test_full_size_sampled_rows(name, dtype):
    p = make_problem(CONFIGS[name], seed=0, bf16=(dtype == "bf16"), fp8=(dtype == "fp8"))
    out = run_gpu(p, dtype)
    rows = sample_rows(p.shape.S)
    heads = [0, p.shape.H - 1]
    got = select(out, rows=rows, heads=heads)
    ref = oracle_out(p, dtype, rows=rows, heads=heads)
    assert O.rel_l2(got, ref) <= TOL[dtype]
    assert per_row_rel(got, ref).max() <= ROW_TOL[dtype]
    assert torch.isfinite(out.float()).all()


def test_output_canaries_untouched():
    # out is a view into a larger buffer: the bytes before and after it keep their sentinel value
    p = make_problem(Shape(1, 300, 2, 1, 128, 128), seed=3)
    q, k, v, ds = to_device(p, "fp8")
    n = 300 * 2 * 128
    buf = torch.full((n + 4096,), 7.0, dtype=torch.bfloat16, device="cuda")
    out = buf[2048:2048 + n].view(1, 300, 2, 128)
    flash_attn_func(q, k, v, q_descale=ds[0], k_descale=ds[1], v_descale=ds[2], out=out)
    torch.cuda.synchronize()
    assert torch.all(buf[:2048] == 7.0) and torch.all(buf[2048 + n:] == 7.0)
    assert O.rel_l2(select(out), oracle_out(p, "fp8")) <= FP8_TOL


def test_no_descale_means_one():
    p = make_problem(Shape(1, 200, 2, 2, 128, 128), seed=4)
    q, k, v, _ = to_device(p, "fp8")
    got = select(flash_attn_func(q, k, v))
    ref = O.leanp_causal_attention(p.q8.numpy(), p.k8.numpy(), p.v8.numpy(), 1.0, 1.0, 1.0,
                                   scale_of(p))
    assert O.rel_l2(got, ref) <= FP8_TOL


def test_uint8_codes_accepted_and_equal_to_fp8_dtype():
    p = make_problem(Shape(1, 150, 2, 1, 128, 128), seed=5)
    q, k, v, ds = to_device(p, "fp8")
    a = flash_attn_func(q, k, v, q_descale=ds[0], k_descale=ds[1], v_descale=ds[2])
    b = flash_attn_func(q.view(torch.uint8), k.view(torch.uint8), v.view(torch.uint8), q_descale=ds[0],
                        k_descale=ds[1], v_descale=ds[2])
    assert torch.equal(a, b)


def test_zero_queries_give_prefix_mean():
    # closed form on the device: Q = 0 -> every output row is the running mean of V
    p = make_problem(Shape(1, 500, 2, 1, 128, 128), seed=6)
    p.q8.zero_()
    out = select(run_gpu(p, "fp8"))
    vv = O.e4m3_decode(p.v8.numpy())[0, :, 0, :] * p.dv
    mean = np.cumsum(vv, axis=0) / np.arange(1, 501)[:, None]
    for h in range(2):
        np.testing.assert_allclose(out[0, :, h, :], mean, rtol=1e-2, atol=2e-3 * np.abs(mean).max())


def test_misaligned_pointer_rejected_on_device():
    p = make_problem(Shape(1, 64, 1, 1, 128, 128), seed=7)
    q, k, v, _ = to_device(p, "fp8")
    raw = torch.empty(64 * 128 + 16, dtype=torch.uint8, device="cuda")
    qm = raw[1:1 + 64 * 128].view(1, 64, 1, 128)
    with pytest.raises(Exception):
        flash_attn_func(qm.view(torch.float8_e4m3fn), k, v)

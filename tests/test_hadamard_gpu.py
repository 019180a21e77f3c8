"""GPU parity of the Hadamard pre-pass (zyfa_hadamard_quantize_e4m3) with its oracle: codes and
descale bit for bit (both sides rotate in float32 in the same stage order, multiply every rotated
value by the same fp32 scale fl32(448/amax) and round to e4m3), and attention on rotated inputs."""
import math

import numpy as np
import pytest
import torch

import oracle as O
from _gpu_util import FP8_TOL, select
from fp8_causal_prefill_gb300 import api, flash_attn_func, hadamard_quantize_e4m3, hadamard_quantize_qk_e4m3
from fp8_causal_prefill_gb300.inputs import CONFIGS, Shape, make_problem, quantize_e4m3

pytestmark = pytest.mark.gpu


def _bf16(x):
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)


def _oracle(xb):
    return O.hadamard_quantize_e4m3(xb.float().numpy())


@pytest.mark.parametrize("D", [64, 128, 192])
@pytest.mark.parametrize("rows", [1, 37, 256, 257, 1000, 4109])
def test_codes_and_descale_bit_exact(rows, D):
    rng = np.random.default_rng(rows * 7 + D)
    x = rng.standard_normal((rows, D)).astype(np.float32)
    x[:, rng.choice(D, 3, replace=False)] *= 20.0          # outlier channels
    xb = _bf16(x)
    codes, ds = hadamard_quantize_e4m3(xb.cuda())
    torch.cuda.synchronize()
    ref_codes, ref_ds = _oracle(xb)
    assert float(ds.item()) == ref_ds
    np.testing.assert_array_equal(codes.view(torch.uint8).cpu().numpy(), ref_codes)


def test_zero_input_gives_descale_one():
    codes, ds = hadamard_quantize_e4m3(torch.zeros((300, 128), dtype=torch.bfloat16, device="cuda"))
    torch.cuda.synchronize()
    assert ds.item() == 1.0 and int(codes.view(torch.uint8).max()) == 0


def test_full_size_q_sampled_rows():
    sh = CONFIGS["bench32k"]
    p = make_problem(sh, seed=0, fp8=False)
    xb = p.qb.reshape(-1, sh.D_qk)
    codes, ds = hadamard_quantize_e4m3(xb.cuda())
    torch.cuda.synchronize()
    # descale: the oracle's per-tensor maximum over the whole rotated tensor (chunked: max is exact)
    amax = np.float32(0.0)
    for c in range(0, xb.shape[0], 1 << 16):
        y = O.fwht_f32(xb[c:c + (1 << 16)].float().numpy(), 128)
        amax = max(amax, np.float32(np.abs(y).max()))
    ref_ds = float(np.float32(amax / np.float32(448.0)))
    assert float(ds.item()) == ref_ds
    rng = np.random.default_rng(5)
    rows = np.sort(rng.choice(xb.shape[0], 2000, replace=False))
    y = O.fwht_f32(xb[rows].float().numpy(), 128)
    ref = O.e4m3_encode_rne_satfinite((y * np.float32(np.float32(448.0) / amax)).astype(np.float32).astype(np.float64))
    np.testing.assert_array_equal(codes.view(torch.uint8).cpu().numpy()[rows], ref)


def test_attention_on_rotated_inputs():
    # Rotated Q/K codes go straight into the attention kernel; it matches the Lean-P oracle on those
    # codes, and against float64 attention on the unquantised inputs its error is lower than without
    # the rotation on the outlier (captured-activation stand-in) workload.
    sh = Shape(1, 2048, 4, 1, 128, 128, "mistral")
    p = make_problem(sh, seed=0)
    q8r, dqr = hadamard_quantize_e4m3(p.qb.cuda())
    k8r, dkr = hadamard_quantize_e4m3(p.kb.cuda())
    v8 = p.v8.cuda().view(torch.float8_e4m3fn)
    dv = torch.tensor([p.dv], dtype=torch.float32, device="cuda")
    out = flash_attn_func(q8r, k8r, v8, q_descale=dqr, k_descale=dkr, v_descale=dv)
    torch.cuda.synchronize()
    sc = O.default_softmax_scale(128)
    q8n, k8n = q8r.view(torch.uint8).cpu().numpy(), k8r.view(torch.uint8).cpu().numpy()
    ref = O.leanp_causal_attention(q8n, k8n, p.v8.numpy(), dqr.item(), dkr.item(), p.dv, sc)
    got = select(out)
    assert O.rel_l2(got, ref) <= FP8_TOL
    # error against float64 attention on the unquantised (bf16) inputs, with and without the rotation
    rows = np.arange(0, 2048, 9)
    f = lambda t: t.float().numpy().astype(np.float64)  # noqa: E731
    exact = O.exact_causal_attention(f(p.qb), f(p.kb), f(p.vb), sc, rows=rows)
    plain_q8, dq = quantize_e4m3(f(p.qb).astype(np.float32))
    plain_k8, dk = quantize_e4m3(f(p.kb).astype(np.float32))
    plain = flash_attn_func(plain_q8.cuda().view(torch.float8_e4m3fn), plain_k8.cuda().view(torch.float8_e4m3fn), v8,
                            q_descale=torch.tensor([dq], device="cuda"), k_descale=torch.tensor([dk], device="cuda"),
                            v_descale=dv)
    torch.cuda.synchronize()
    e_rot = O.rel_l2(got[:, rows], exact)
    e_plain = O.rel_l2(select(plain)[:, rows], exact)
    print(f"\n[hadamard] attention error vs float64: rotated {e_rot:.4e}  plain {e_plain:.4e}")
    assert e_rot < 0.8 * e_plain


def test_workspace_checks():
    x = torch.zeros((600, 128), dtype=torch.bfloat16, device="cuda")
    c = torch.empty((600, 128), dtype=torch.uint8, device="cuda")
    d = torch.empty(1, dtype=torch.float32, device="cuda")
    ws = torch.empty(4, dtype=torch.float32, device="cuda")     # needs 5 floats for 600 rows
    assert api.zyfa_hadamard_workspace_bytes(600) == 20
    st = api.zyfa_hadamard_quantize_e4m3(x.data_ptr(), c.data_ptr(), d.data_ptr(), 600, 128, ws.data_ptr(), 16)
    assert st == 1
    assert api.zyfa_hadamard_quantize_e4m3(x.data_ptr(), c.data_ptr(), d.data_ptr(), 0, 128, 0, 0) == 0
    assert api.zyfa_hadamard_quantize_e4m3(x.data_ptr(), c.data_ptr(), d.data_ptr(), 600, 96, ws.data_ptr(), 8) == 2


@pytest.mark.parametrize("D", [64, 128, 192])
@pytest.mark.parametrize("q_rows,k_rows", [(1, 1), (4109, 257), (256, 1000), (70001, 13)])
def test_q_and_k_in_one_launch_equal_the_oracle(q_rows, k_rows, D):
    # Q and K share a launch per pass but keep their own maxima: codes and descales equal the
    # oracle's for each tensor on its own, bit for bit (the K maximum differs from Q's on purpose)
    rng = np.random.default_rng(q_rows + 3 * k_rows + D)
    xq = _bf16(rng.standard_normal((q_rows, D)) * 3.0)
    xk = _bf16(rng.standard_normal((k_rows, D)))
    q8, dq, k8, dk = hadamard_quantize_qk_e4m3(xq.cuda(), xk.cuda())
    torch.cuda.synchronize()
    for codes, ds, xb in ((q8, dq, xq), (k8, dk, xk)):
        ref_codes, ref_ds = _oracle(xb)
        assert float(ds.item()) == float(ref_ds)
        assert np.array_equal(codes.view(torch.uint8).cpu().numpy(), ref_codes)


def test_q_and_k_in_one_launch_at_the_bench_size_equal_separate_calls():
    # the bench workload's Q (1,048,576 rows) and K (262,144 rows): the joint call reproduces two
    # separate calls bit for bit
    g = torch.Generator(device="cuda").manual_seed(11)
    xq = torch.randn((1 << 20, 128), generator=g, device="cuda").to(torch.bfloat16)
    xk = torch.randn((1 << 18, 128), generator=g, device="cuda").to(torch.bfloat16)
    q8, dq, k8, dk = hadamard_quantize_qk_e4m3(xq, xk)
    q8s, dqs = hadamard_quantize_e4m3(xq)
    k8s, dks = hadamard_quantize_e4m3(xk)
    torch.cuda.synchronize()
    assert torch.equal(dq, dqs) and torch.equal(dk, dks)
    assert torch.equal(q8.view(torch.uint8), q8s.view(torch.uint8))
    assert torch.equal(k8.view(torch.uint8), k8s.view(torch.uint8))


def test_q_and_k_workspace_and_empty_tensor_checks():
    x = torch.zeros((600, 128), dtype=torch.bfloat16, device="cuda")
    c = torch.empty((600, 128), dtype=torch.uint8, device="cuda")
    d = torch.empty(2, dtype=torch.float32, device="cuda")
    one = api.zyfa_hadamard_workspace_bytes(600)
    ws = torch.empty(2 * one // 4, dtype=torch.float32, device="cuda")
    args = (x.data_ptr(), c.data_ptr(), d.data_ptr(), 600, x.data_ptr(), c.data_ptr(), d.data_ptr() + 4)
    assert api.zyfa_hadamard_quantize_qk_e4m3(*args, 600, 128, ws.data_ptr(), 2 * one - 4) == 1  # short workspace
    assert api.zyfa_hadamard_quantize_qk_e4m3(*args, 600, 96, ws.data_ptr(), 2 * one) == 2       # head dim
    assert api.zyfa_hadamard_quantize_qk_e4m3(*args, 0, 128, ws.data_ptr(), one) == 0            # K empty
    torch.cuda.synchronize()
    assert float(d[0].item()) == 1.0                    # all-zero Q: descale 1

"""Edge cases at the extremes: a sequence four times the bench length; score ranges so wide that
whole 64-key blocks fall more than 127 binades below the row's reference (their E8M0 scale leaves the
representable range; the method's weights there are below 2^-127 of the row's largest and vanish); and
scores that climb ~90 binades along a row, which the block-scaled paths absorb without moving the
row's reference."""
import numpy as np
import pytest
import torch

import oracle as O
from _gpu_util import BF16_TOL, FP8_TOL, oracle_out, per_row_rel, run_gpu, select, to_device
from fp8_causal_prefill_gb300 import flash_attn_func, zyfa_check_errors
from fp8_causal_prefill_gb300.inputs import Shape, make_problem, sample_rows

pytestmark = pytest.mark.gpu


def test_sequence_of_128k_tokens_sampled_rows():
    sh = Shape(1, 131072, 2, 1, 128, 128)
    p = make_problem(sh, seed=31, bf16=False)
    q, k, v, ds = to_device(p, "fp8")
    out = flash_attn_func(q, k, v, q_descale=ds[0], k_descale=ds[1], v_descale=ds[2])
    torch.cuda.synchronize()
    assert zyfa_check_errors() == 0
    rows = sample_rows(sh.S, n_random=96, edge=32, seed=4)
    got = select(out, rows=rows)
    ref = oracle_out(p, "fp8", rows=rows)
    assert O.rel_l2(got, ref) <= FP8_TOL
    assert per_row_rel(got, ref).max() <= 5e-2
    assert torch.isfinite(out.float()).all()


@pytest.mark.parametrize("p_mode", ["lean", "exact", "exact-noblock"])
def test_extreme_score_range(p_mode):
    # the same codes with q/k descales 10x larger: score spreads of ~800 binades per row (up to ~700
    # binades from zero), so many blocks sit more than 127 binades below the row maximum (weight 0 in
    # the oracle, at most 2^-127 of it on the device) while the top blocks decide the output.  (The
    # block exponents stay far inside the range where 55.625 - 8e is exact in fp32.)
    sh = Shape(1, 700, 2, 1, 128, 128)
    p = make_problem(sh, seed=32, bf16=False)
    p.dq, p.dk = p.dq * 10.0, p.dk * 10.0
    q, k, v, ds = to_device(p, "fp8")
    out = flash_attn_func(q, k, v, q_descale=ds[0], k_descale=ds[1], v_descale=ds[2], p_mode=p_mode)
    torch.cuda.synchronize()
    assert zyfa_check_errors() == 0
    f = {"exact": O.exactp_causal_attention, "exact-noblock": O.exactp_noblock_causal_attention}.get(
        p_mode, O.leanp_causal_attention)
    ref = f(p.q8.numpy(), p.k8.numpy(), p.v8.numpy(), p.dq, p.dk, p.dv, O.default_softmax_scale(128))
    got = select(out)
    assert np.all(np.isfinite(got))
    assert O.rel_l2(got, ref) <= FP8_TOL


def test_extreme_score_range_bf16():
    # q scaled by 40 (re-rounded to bf16): scores spread over hundreds of binades per row, so the row
    # reference rises many times (conditional rescales of O and l) and most probabilities underflow;
    # the device flushes results below 2^-126 to zero, the oracle keeps bf16 subnormals down to 2^-133,
    # a difference of at most 2^-126 of the row's largest weight
    sh = Shape(1, 700, 2, 1, 128, 128)
    p = make_problem(sh, seed=33)
    p.qb = (p.qb.float() * 40.0).to(torch.bfloat16)
    out = run_gpu(p, "bf16")
    assert zyfa_check_errors() == 0
    got = select(out)
    assert np.all(np.isfinite(got))
    assert O.rel_l2(got, oracle_out(p, "bf16")) <= BF16_TOL


@pytest.mark.parametrize("p_mode", ["lean", "exact"])
def test_row_reference_lagging_by_up_to_ninety_binades(p_mode):
    # Scores that rise along the keys: q = e_0 (and 0.5 e_0 for the second head), k_j = r_j e_0 with
    # r_j climbing to 448, scaled so that a row's last keys sit ~90 binades above its first tile.  The
    # block-scaled paths let the row reference lag that far without a rescale (the scale factors carry
    # 2^(e - M) up to 2^90 and O grows accordingly in fp32), so the output must still match the
    # emulation, which normalises against the row's true maximum, and stay finite.
    S, D = 1500, 64
    q8 = np.zeros((1, S, 2, D), dtype=np.uint8)
    q8[:, :, 0, 0] = 0x38          # 1.0
    q8[:, :, 1, 0] = 0x30          # 0.5
    k8 = np.zeros((1, S, 1, D), dtype=np.uint8)
    k8[0, :, 0, 0] = O.e4m3_encode_rne_satfinite(448.0 * np.arange(S) / (S - 1))
    rng = np.random.default_rng(5)
    v8 = O.e4m3_encode_rne_satfinite(rng.standard_normal((1, S, 1, D)))
    scale, dq, dk, dv = 0.125, 1.0, 1.114, 1.0
    a = O.fp8_score_scale(scale, dq, dk)
    assert 700 < 448 * a < 740            # the ramp spans about 90 binades at its end
    q, k, v = (torch.from_numpy(x).cuda().view(torch.float8_e4m3fn) for x in (q8, k8, v8))
    ds = [torch.tensor([x], dtype=torch.float32, device="cuda") for x in (dq, dk, dv)]
    out = flash_attn_func(q, k, v, softmax_scale=scale, q_descale=ds[0], k_descale=ds[1], v_descale=ds[2],
                          p_mode=p_mode)
    torch.cuda.synchronize()
    assert zyfa_check_errors() == 0
    f = O.exactp_causal_attention if p_mode == "exact" else O.leanp_causal_attention
    ref = f(q8, k8, v8, dq, dk, dv, scale)
    got = select(out)
    assert np.all(np.isfinite(got))
    assert O.rel_l2(got, ref) <= FP8_TOL
    assert per_row_rel(got, ref).max() <= 5e-2

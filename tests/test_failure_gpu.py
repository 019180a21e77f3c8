"""Failure detection on the GPU without a fault: every pipeline wait in the kernel is bounded, so a
pipeline that never receives its data ends with a timeout status that the host reads, and the CUDA
context stays usable for the next call."""
import pytest
import torch

import oracle as O
from _gpu_util import FP8_TOL, oracle_out, select, to_device
from fp8_causal_prefill_gb300 import api, flash_attn_func, zyfa_check_errors
from fp8_causal_prefill_gb300.inputs import Shape, make_problem

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype", ["fp8", "bf16"])
def test_stalled_pipeline_times_out_and_context_survives(dtype):
    sh = Shape(1, 700, 2, 1, 128, 128)
    p = make_problem(sh, seed=21)
    q, k, v, ds = to_device(p, dtype)
    assert zyfa_check_errors() == 0
    out = torch.full((1, 700, 2, 128), 3.0, dtype=torch.bfloat16, device="cuda")
    code = api.ZYFA_DTYPE_E4M3 if dtype == "fp8" else api.ZYFA_DTYPE_BF16
    stream = torch.cuda.current_stream().cuda_stream
    st = api.zyfa_selftest_stalled_pipeline(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), sh.B, sh.S,
                                            sh.H, sh.H_kv, sh.D_qk, sh.D_v, code, stream)
    assert st == 0
    assert zyfa_check_errors(stream) == 5          # ZYFA_ERR_TIMEOUT, read and cleared
    assert zyfa_check_errors(stream) == 0
    assert torch.all(out == 3.0)                   # nothing was written
    # the context is intact: a normal call right after still matches the oracle
    if dtype == "fp8":
        got = flash_attn_func(q, k, v, q_descale=ds[0], k_descale=ds[1], v_descale=ds[2])
        torch.cuda.synchronize()
        assert zyfa_check_errors() == 0
        assert O.rel_l2(select(got), oracle_out(p, "fp8")) <= FP8_TOL
    else:
        got = flash_attn_func(q, k, v)
        torch.cuda.synchronize()
        assert zyfa_check_errors() == 0
        assert torch.isfinite(got.float()).all()


def test_selftest_validates_arguments_like_the_main_entry():
    st = api.zyfa_selftest_stalled_pipeline(0, 0, 0, 0, 1, 16, 3, 2, 128, 128, api.ZYFA_DTYPE_E4M3, 0)
    assert st == 1                                 # H % H_kv != 0

"""GPU determinism: repeated launches on the same inputs produce bitwise-identical outputs (the pages
report bitwise-identical outputs over 7,200 launches; spbcomputers.ru ZYFA article, section "Точность").
The kernel has no atomics on data and a static work schedule, so every launch performs the same
arithmetic in the same order."""
import pytest
import torch

from _gpu_util import to_device
from fp8_causal_prefill_gb300 import flash_attn_func, zyfa_check_errors
from fp8_causal_prefill_gb300.inputs import CONFIGS, make_problem

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name,dtype,launches", [("bench32k", "fp8", 1000), ("gqa4k", "bf16", 1000),
                                                 ("mla32k", "fp8", 200)])
def test_bitwise_identical_over_repeated_launches(name, dtype, launches):
    p = make_problem(CONFIGS[name], seed=0, bf16=(dtype == "bf16"), fp8=(dtype == "fp8"))
    q, k, v, ds = to_device(p, dtype)
    ref = flash_attn_func(q, k, v, q_descale=ds[0], k_descale=ds[1], v_descale=ds[2])
    out = torch.empty_like(ref)
    mismatches = torch.zeros((), dtype=torch.int64, device=ref.device)
    for _ in range(launches):
        flash_attn_func(q, k, v, q_descale=ds[0], k_descale=ds[1], v_descale=ds[2], out=out)
        mismatches += (out.view(torch.int16) != ref.view(torch.int16)).any().to(torch.int64)
    torch.cuda.synchronize()
    assert zyfa_check_errors() == 0
    assert int(mismatches) == 0

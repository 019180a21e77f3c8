"""The tensor-core rate probe (zyfa_probe_mma_rate) through the C ABI: it runs, reports no timeout, and
measures the dense per-SM rates its FLOP count implies for the tcgen05 MMA forms the attention kernel
uses (FP8 e4m3 twice BF16 per cycle; the pages quote FP8 throughput as a share of the FP8 peak,
captivela ZYFA article, "Angka Nyata")."""
import pytest
import torch

from fp8_causal_prefill_gb300 import api

pytestmark = pytest.mark.gpu


def _rate(fp8):
    lib = api.load_library()
    nsm = torch.cuda.get_device_properties(0).multi_processor_count
    cycles = torch.zeros(nsm, dtype=torch.int64, device="cuda")
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    iters = 2000
    assert lib.zyfa_probe_mma_rate(fp8, iters, nsm, cycles.data_ptr(), flag.data_ptr(), None) == 0
    torch.cuda.synchronize()
    assert int(flag.item()) == 0
    c = cycles.cpu()
    assert bool((c > 0).all())
    return lib.zyfa_probe_mma_flops_per_iter(fp8) * iters / float(c.max())


def test_fp8_rate_is_twice_bf16_per_cycle():
    fp8, bf16 = _rate(1), _rate(0)
    # a CTA's span includes its last MMAs' drain, so the measured rate sits a little under the steady one
    assert 0.9 * 16384 < fp8 <= 16384 * 1.01
    assert 0.9 * 8192 < bf16 <= 8192 * 1.01
    assert 1.9 < fp8 / bf16 < 2.1


def _form_rate(form):
    lib = api.load_library()
    nsm = torch.cuda.get_device_properties(0).multi_processor_count
    cycles = torch.zeros(nsm, dtype=torch.int64, device="cuda")
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    iters = 2000
    assert lib.zyfa_probe_mma_form_rate(form, iters, nsm, cycles.data_ptr(), flag.data_ptr(), None) == 0
    torch.cuda.synchronize()
    assert int(flag.item()) == 0
    c = cycles.cpu()
    assert bool((c > 0).all())
    return lib.zyfa_probe_mma_form_flops_per_iter(form) * iters / float(c.max())


def test_the_kernels_fp8_mma_forms_run_at_the_dense_rate():
    # the score tile (N=128 from shared memory), the block-scaled PV (N=144, P in tensor memory) and
    # the two in sequence each reach the FP8 rate when issued back to back
    for form in (0, 1, 2):
        assert 0.9 * 16384 < _form_rate(form) <= 16384 * 1.01, form


def test_n64_score_halves_are_slower_than_one_n128_tile():
    # an N=64 score MMA reads all of Q from shared memory for half the keys: the two halves of a tile
    # take longer than the single N=128 MMA
    assert _form_rate(3) < 0.85 * _form_rate(0)


def test_probe_rejects_bad_arguments():
    lib = api.load_library()
    assert lib.zyfa_probe_mma_rate(2, 10, 1, 16, 16, None) == 1
    assert lib.zyfa_probe_mma_rate(1, 0, 1, 16, 16, None) == 1
    assert lib.zyfa_probe_mma_rate(1, 10, 1, 0, 16, None) == 1
    assert lib.zyfa_probe_mma_form_rate(6, 10, 1, 16, 16, None) == 1
    assert lib.zyfa_probe_mma_form_rate(-1, 10, 1, 16, 16, None) == 1
    assert lib.zyfa_probe_mma_form_rate(0, 0, 1, 16, 16, None) == 1
    assert lib.zyfa_probe_mma_form_flops_per_iter(6) == -1

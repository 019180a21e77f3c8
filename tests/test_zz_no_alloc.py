"""The allocation-free Hadamard pre-pass (zyfa_hadamard_quantize_e4m3_noalloc), through the C ABI.

It serves callers that cannot allocate device memory on their call path (a serving runtime with a
fixed memory plan, a C host program without a device allocator); its scratch is a fixed array inside
the library.  Its output must equal the workspace entry point's, bit for bit, on two calls in a row
(the second call reuses the scratch the first one left behind).  This file is collected last."""
import numpy as np
import pytest
import torch

from fp8_causal_prefill_gb300 import api

pytestmark = pytest.mark.gpu


def _input(rows, d, seed):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((rows, d)).astype(np.float32)
    x[:, rng.choice(d, 3, replace=False)] *= 16.0
    return torch.from_numpy(x).to(torch.bfloat16).cuda()


def _with_workspace(x):
    rows, d = x.shape
    c = torch.empty((rows, d), dtype=torch.uint8, device="cuda")
    ds = torch.empty(1, dtype=torch.float32, device="cuda")
    ws = torch.empty(max(1, api.zyfa_hadamard_workspace_bytes(rows) // 4), dtype=torch.float32, device="cuda")
    assert api.zyfa_hadamard_quantize_e4m3(x.data_ptr(), c.data_ptr(), ds.data_ptr(), rows, d, ws.data_ptr(),
                                           ws.numel() * 4) == 0
    torch.cuda.synchronize()
    return c, ds


def _no_alloc(x):
    rows, d = x.shape
    c = torch.full((rows, d), 0xAB, dtype=torch.uint8, device="cuda")
    ds = torch.full((1,), -1.0, dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()
    assert api.zyfa_hadamard_quantize_e4m3_noalloc(x.data_ptr(), c.data_ptr(), ds.data_ptr(), rows, d) == 0
    torch.cuda.synchronize()
    assert api.zyfa_check_errors() == 0
    return c, ds


@pytest.mark.parametrize("d", [64, 128, 192])
def test_no_alloc_equals_workspace_entry_on_two_calls_in_a_row(d):
    # two allocation-free calls back to back: a large input, then a smaller one with a different
    # maximum, which must not see the partial maxima the first call left in the shared scratch
    xs = [_input(70001, d, 1 + d), _input(3000, d, 2 + d)]
    refs = [_with_workspace(x) for x in xs]
    gots = [_no_alloc(x) for x in xs]
    for (ref_c, ref_ds), (got_c, got_ds) in zip(refs, gots):
        assert torch.equal(got_ds, ref_ds)
        assert torch.equal(got_c, ref_c)


def test_no_alloc_at_its_largest_accepted_size():
    # 4,194,304 rows fill the library's scratch to its last slot (32,768 partial maxima)
    rows = 4_194_304
    g = torch.Generator(device="cuda").manual_seed(5)
    x = torch.randn((rows, 64), generator=g, device="cuda").to(torch.bfloat16)
    x[rows - 7, 3] = 300.0               # the tensor's maximum sits in the last 128-row block
    ref_c, ref_ds = _with_workspace(x)
    got_c, got_ds = _no_alloc(x)
    assert torch.equal(got_ds, ref_ds)
    assert torch.equal(got_c, ref_c)


def test_no_alloc_rejects_rows_beyond_its_scratch():
    x = torch.zeros((128, 128), dtype=torch.bfloat16, device="cuda")
    c = torch.empty((128, 128), dtype=torch.uint8, device="cuda")
    ds = torch.empty(1, dtype=torch.float32, device="cuda")
    too_many = 4_194_304 + 1
    assert api.zyfa_hadamard_quantize_e4m3_noalloc(x.data_ptr(), c.data_ptr(), ds.data_ptr(), too_many, 128) == 2
    assert api.zyfa_hadamard_quantize_e4m3_noalloc(x.data_ptr(), c.data_ptr(), ds.data_ptr(), 0, 128) == 0

"""The host-buffer entry point (zyfa_attn_fwd_causal_host): uploads, chunked kernels and downloads
overlapped; its output must equal the device-buffer call's bit for bit (every query row is computed by
the same kernel arithmetic whichever chunk it falls in)."""
import numpy as np
import pytest
import torch

from _gpu_util import to_device
from fp8_causal_prefill_gb300 import api, flash_attn_func, zyfa_check_errors
from fp8_causal_prefill_gb300.inputs import Shape, make_problem

pytestmark = pytest.mark.gpu


def _run_host(p, dtype, chunks, pinned=True):
    sh = p.shape
    host = [t.contiguous() for t in ((p.q8, p.k8, p.v8) if dtype == "fp8" else (p.qb, p.kb, p.vb))]
    if pinned:
        host = [h.pin_memory() for h in host]
    out_h = torch.empty((sh.B, sh.S, sh.H, sh.D_v), dtype=torch.bfloat16)
    if pinned:
        out_h = out_h.pin_memory()
    dev = [torch.empty(h.shape, dtype=h.dtype, device="cuda") for h in host]
    out_d = torch.empty(out_h.shape, dtype=torch.bfloat16, device="cuda")
    desc = torch.tensor([p.dq, p.dk, p.dv], dtype=torch.float32, device="cuda")
    code = api.ZYFA_DTYPE_E4M3 if dtype == "fp8" else api.ZYFA_DTYPE_BF16
    d = desc.data_ptr() if dtype == "fp8" else 0
    stream = torch.cuda.current_stream().cuda_stream
    st = api.zyfa_attn_fwd_causal_host(host[0].data_ptr(), host[1].data_ptr(), host[2].data_ptr(), out_h.data_ptr(),
                                       dev[0].data_ptr(), dev[1].data_ptr(), dev[2].data_ptr(), out_d.data_ptr(),
                                       sh.B, sh.S, sh.H, sh.H_kv, sh.D_qk, sh.D_v, 0.0, code, d, d + 4 if d else 0,
                                       d + 8 if d else 0, chunks, stream)
    assert st == 0
    torch.cuda.current_stream().synchronize()
    assert zyfa_check_errors() == 0
    return out_h, out_d


def _reference(p, dtype):
    q, k, v, ds = to_device(p, dtype)
    out = flash_attn_func(q, k, v, q_descale=ds[0], k_descale=ds[1], v_descale=ds[2])
    torch.cuda.synchronize()
    return out.cpu()


@pytest.mark.parametrize("dtype", ["fp8", "bf16"])
@pytest.mark.parametrize("shape,chunks", [(Shape(1, 1000, 4, 2, 128, 128), 1), (Shape(1, 1000, 4, 2, 128, 128), 3),
                                          (Shape(2, 520, 2, 2, 128, 128), 0), (Shape(1, 8192, 8, 2, 128, 128), 0),
                                          (Shape(1, 700, 2, 2, 192, 128), 64), (Shape(3, 600, 8, 4, 64, 64), 2),
                                          (Shape(3, 300, 6, 3, 64, 64), 2), (Shape(2, 10000, 4, 2, 128, 128), 0)],
                         ids=["S1000c1", "S1000c3", "B2S520", "S8192", "mla-S700-c64", "B3-D64-halves", "B3-D64-oddkv",
                              "B2S10000-tail-plan"])
def test_host_pipeline_equals_device_call(shape, chunks, dtype):
    p = make_problem(shape, seed=shape.S + chunks)
    out_h, out_d = _run_host(p, dtype, chunks)
    ref = _reference(p, dtype)
    assert torch.equal(out_h, ref)
    assert torch.equal(out_d.cpu(), ref)


def test_pageable_host_memory_still_correct():
    p = make_problem(Shape(1, 900, 2, 1, 128, 128), seed=9)
    out_h, _ = _run_host(p, "fp8", 4, pinned=False)
    assert torch.equal(out_h, _reference(p, "fp8"))


def test_host_entry_rejects_bad_arguments():
    assert api.zyfa_attn_fwd_causal_host(16, 16, 16, 16, 16, 16, 16, 16, 1, 64, 2, 2, 128, 128, 0.0, 0, 0, 0, 0, -1) == 1
    assert api.zyfa_attn_fwd_causal_host(0, 16, 16, 16, 16, 16, 16, 16, 1, 64, 2, 2, 128, 128, 0.0, 0, 0, 0, 0, 2) == 1
    assert api.zyfa_attn_fwd_causal_host(16, 16, 16, 16, 16, 16, 16, 16, 1, 64, 2, 2, 96, 96, 0.0, 0, 0, 0, 0, 2) == 2


def test_host_entry_checks_device_buffers_before_any_copy():
    # a misaligned or missing device buffer is reported before anything is enqueued: the device
    # buffers and the host output keep their contents
    p = make_problem(Shape(1, 300, 2, 1, 128, 128), seed=4, bf16=False)
    host = [t.contiguous().pin_memory() for t in (p.q8, p.k8, p.v8)]
    out_h = torch.full((1, 300, 2, 128), 7.0, dtype=torch.bfloat16).pin_memory()
    dev = [torch.zeros(h.numel() + 16, dtype=torch.uint8, device="cuda") for h in host]
    out_d = torch.zeros(300 * 2 * 128 + 8, dtype=torch.bfloat16, device="cuda")
    hp = [h.data_ptr() for h in host] + [out_h.data_ptr()]

    def call(qd, kd, vd, od, scale=0.0):
        return api.zyfa_attn_fwd_causal_host(*hp, qd, kd, vd, od, 1, 300, 2, 1, 128, 128, scale, api.ZYFA_DTYPE_E4M3,
                                             0, 0, 0, 4, torch.cuda.current_stream().cuda_stream)
    ok = [d.data_ptr() for d in dev] + [out_d.data_ptr()]
    assert call(ok[0] + 8, ok[1], ok[2], ok[3]) == 3          # misaligned q_dev
    assert call(ok[0], ok[1], ok[2], ok[3] + 2) == 3          # misaligned out_dev
    assert call(ok[0], 0, ok[2], ok[3]) == 1                  # missing k_dev
    assert call(ok[0], ok[1], ok[2], ok[3], scale=-1.0) == 1  # bad scale
    torch.cuda.synchronize()
    assert all(int(d.count_nonzero()) == 0 for d in dev) and int(out_d.count_nonzero()) == 0
    assert bool((out_h == 7.0).all())

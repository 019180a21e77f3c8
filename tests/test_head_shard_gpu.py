"""Sharding by heads or by batch reproduces the unsharded call bit for bit (GPU).

A caller that spreads attention over several GPUs gives each one a contiguous group of KV heads
(with their query heads) or a slice of the batch, as per-shard tensors, and calls the same entry
point; the outputs stay sharded and nothing is exchanged.  That is correct only if a head's output
does not depend on which other heads or batches share the launch.  Here the shards run one after
the other on one GPU and their outputs are compared with the whole call's, bitwise.
"""
import pytest
import torch

from _gpu_util import to_device
from fp8_causal_prefill_gb300 import flash_attn_func, zyfa_check_errors
from fp8_causal_prefill_gb300.inputs import CONFIGS, Shape, make_problem

pytestmark = pytest.mark.gpu


def _call(q, k, v, ds):
    return flash_attn_func(q.contiguous(), k.contiguous(), v.contiguous(), q_descale=ds[0], k_descale=ds[1],
                           v_descale=ds[2])


@pytest.mark.parametrize("dtype", ["fp8", "bf16"])
@pytest.mark.parametrize("shape", [CONFIGS["gqa4k"], Shape(2, 1500, 8, 4, 192, 128)],
                         ids=["gqa4k", "B2S1500H8kv4D192"])
def test_kv_head_groups_and_batch_shards_reproduce_the_whole_call(shape, dtype):
    p = make_problem(shape, seed=3, bf16=(dtype == "bf16"), fp8=(dtype == "fp8"))
    q, k, v, ds = to_device(p, dtype)
    whole = _call(q, k, v, ds)
    g = shape.H // shape.H_kv                 # query heads per KV head
    # two contiguous KV-head groups of unequal size, each with its query heads
    cut = shape.H_kv // 2 + (shape.H_kv % 2)
    parts = []
    for hk0, hk1 in ((0, cut), (cut, shape.H_kv)):
        parts.append(_call(q[:, :, hk0 * g:hk1 * g], k[:, :, hk0:hk1], v[:, :, hk0:hk1], ds))
    heads = torch.cat(parts, dim=2)
    torch.cuda.synchronize()
    assert zyfa_check_errors() == 0
    assert torch.equal(heads.view(torch.int16), whole.view(torch.int16))
    if shape.B > 1:
        rows = torch.cat([_call(q[b:b + 1], k[b:b + 1], v[b:b + 1], ds) for b in range(shape.B)], dim=0)
        torch.cuda.synchronize()
        assert torch.equal(rows.view(torch.int16), whole.view(torch.int16))

"""The allocation-free entry point, for callers that cannot allocate device memory.

tllm_decode_attn_splitkv_noalloc keeps its split records in the library's own device
array instead of a caller workspace. Callers that cannot allocate are, for example, engines
that reserve all of device memory for their own pools, and plugin hosts that pass only
tensors.

The test calls it through the C ABI twice in a row, on two different workloads. Before the
second call the array is filled with stale records (NaN outputs, other log-sum-exps) by a
call on altered inputs. Each result must
  - equal the regular entry point's (tllm_decode_attn_splitkv with a caller-owned workspace)
    bit for bit: the same kernels on the same inputs and plan;
  - match the CPU fp64 oracle within the parity tolerance;
  - leave the array's status word without TLLM_FLAG_TIMEOUT.
It also checks that a plan needing more than the array is refused. The file name makes
pytest collect it last.
"""
import dataclasses

import pytest
import torch

from split_kv_paged_gb300 import binding as B
from split_kv_paged_gb300 import workloads as W
from tests.gpu_helpers import assert_close, new_out, oracle_out, plan_for, poisoned_workspace

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from split_kv_paged_gb300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    B.lib()


def _noalloc(inp, plan, S):
    wl = inp.wl
    got = new_out(wl)
    B.tllm_decode_attn_splitkv_noalloc(inp.q, inp.k_cache, inp.v_cache, inp.block_table, inp.context_lens, wl.Lq,
                                       inp.kv_scales, inp.sinks, wl.window, S, plan, got)
    torch.cuda.synchronize()
    flags = B.tllm_decode_attn_noalloc_read_status()
    assert not (flags & B.TLLM_FLAG_TIMEOUT), f"no-alloc call on {wl.name}: a pipeline wait timed out"
    return got


def _regular(inp, plan, S):
    wl = inp.wl
    ws = poisoned_workspace(plan)
    ref = new_out(wl)
    B.tllm_decode_attn_splitkv(inp.q, inp.k_cache, inp.v_cache, inp.block_table, inp.context_lens, wl.Lq,
                               inp.kv_scales, inp.sinks, wl.window, S, ws, ref)
    torch.cuda.synchronize()
    assert not (B.tllm_decode_attn_read_status(ws) & B.TLLM_FLAG_TIMEOUT)
    return ref


def _stale_records(inp, plan, S):
    """One no-alloc call on the same shape with doubled keys and NaN values: the array then
    holds NaN partial outputs and log-sum-exps that differ from the real call's."""
    stale = dataclasses.replace(inp, k_cache=inp.k_cache.clone(), v_cache=inp.v_cache.clone())
    if inp.wl.kv_dtype == "e4m3":
        stale.v_cache.view(torch.uint8).fill_(0x7F)
        scales = inp.kv_scales.clone()
        scales[0].mul_(2.0)
        stale.kv_scales = scales
    else:
        stale.v_cache.fill_(float("nan"))
        stale.k_cache.mul_(2.0)
    out = new_out(inp.wl)
    B.tllm_decode_attn_splitkv_noalloc(stale.q, stale.k_cache, stale.v_cache, stale.block_table, stale.context_lens,
                                       inp.wl.Lq, stale.kv_scales, stale.sinks, inp.wl.window, S, plan, out)
    torch.cuda.synchronize()


def test_noalloc_matches_regular_entry_point_and_oracle_twice():
    first = W.mtp4_fp8_long(batch=4, ctx=1).replace(ctx=[9000, 130, 4100, 1])
    second = W.window_sink_bf16(batch=5, max_ctx=7000).replace(ctx=[7000, 5000, 64, 4097, 2])
    for k, (wl, seed, S) in enumerate(((first, 31, 4), (second, 32, 3))):
        inp = W.make_inputs(wl, seed, device="cuda")
        plan = plan_for(wl, splits=S, num_pages=inp.num_pages)
        assert plan.workspace_bytes <= B.tllm_decode_attn_noalloc_scratch_bytes()
        if k > 0:
            _stale_records(inp, plan, S)
        got = _noalloc(inp, plan, S)
        ref = _regular(inp, plan, S)
        assert torch.equal(got, ref), f"no-alloc and regular entry points differ on {wl.name}"
        want, _ = oracle_out(inp)
        assert_close(got, want, wl.kv_dtype, f"no-alloc vs oracle on {wl.name}")


def test_noalloc_rejects_plans_beyond_the_array():
    wl = W.mtp4_fp8_long(batch=200, ctx=200_000)
    plan = plan_for(wl, splits=64, num_pages=wl.pages_needed())
    assert plan.workspace_bytes > B.tllm_decode_attn_noalloc_scratch_bytes()
    x = torch.zeros(16, device="cuda")
    with pytest.raises(B.TllmError) as e:
        B.tllm_decode_attn_splitkv_noalloc(x, x, x, x, x, wl.Lq, x, None, 0, 64, plan, x)
    assert e.value.status == B.TLLM_ERR_WORKSPACE_TOO_SMALL

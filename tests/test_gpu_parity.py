"""GPU parity: the CUDA path (through the C ABI) against the CPU fp64 oracle on the same
seeded inputs, element by element, for the five measured workloads, their edge cases
and a fuzz grid of small shapes.

Tolerance (written in tests/gpu_helpers.py): |gpu - ref| <= tol + tol*|ref| per
element, relative L2 <= tol, per-row cosine >= 0.9999, with tol = 2e-3 for fp16/bf16 KV
and 5e-3 for FP8/INT8 KV. Rows that see no key must be exactly zero.
"""
import itertools
import random

import numpy as np
import pytest
import torch

from split_kv_paged_gb300 import binding as B
from split_kv_paged_gb300 import workloads as W
from tests.gpu_helpers import (abs_value_inputs, assert_close, assert_close_conditioned, new_out, oracle_out,
                               plan_for, poison_cache, poisoned_workspace, run_gpu)

pytestmark = pytest.mark.gpu

KERNELS = [B.TLLM_KERNEL_AUTO, B.TLLM_KERNEL_GENERIC]


@pytest.fixture(scope="module", autouse=True)
def built():
    from split_kv_paged_gb300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    B.lib()


def _inputs(wl, seed, poison=True):
    inp = W.make_inputs(wl, seed, device="cuda")
    if poison:
        poison_cache(inp)
    return inp


# --- the five measured workloads ---------------------------------------------

@pytest.mark.parametrize("kernel", KERNELS)
def test_single_decode_fp16(kernel):
    wl = W.single_decode().replace(extra_pages=8)
    inp = _inputs(wl, 1001)
    ref, _ = oracle_out(inp)
    for S in (1, 4):
        out, plan, _ = run_gpu(inp, kernel, splits=S)
        assert plan.num_splits == S
        assert_close(out, ref, wl.kv_dtype, f"single_decode S={S}")


@pytest.mark.parametrize("kernel", KERNELS)
def test_verify16_int8(kernel):
    wl = W.verify16_int8().replace(extra_pages=16)
    inp = _inputs(wl, 1002)
    ref, _ = oracle_out(inp)
    for S in (2, 4, 8):
        out, plan, _ = run_gpu(inp, kernel, splits=S)
        assert_close(out, ref, wl.kv_dtype, f"verify16 S={S}")


@pytest.mark.parametrize("kernel", KERNELS)
def test_mtp4_fp8_reduced(kernel):
    """The batch-200 x 200k workload's shape at sizes the oracle checks whole: several
    tiles per split and ragged tails."""
    wl = W.mtp4_fp8_long(batch=6, ctx=1).replace(ctx=[20000, 12345, 777, 4, 3, 40001], extra_pages=10)
    inp = _inputs(wl, 1003)
    ref, _ = oracle_out(inp)
    for S in (0, 1, 3, 16):
        out, plan, _ = run_gpu(inp, kernel, splits=S)
        assert_close(out, ref, wl.kv_dtype, f"mtp4 reduced S={plan.num_splits}")


@pytest.mark.parametrize("bs", [128, 16])
@pytest.mark.parametrize("kernel", KERNELS)
def test_ragged_fp8(bs, kernel):
    wl = W.ragged_fp8(bs=bs).replace(extra_pages=4)
    inp = _inputs(wl, 1004)
    ref, _ = oracle_out(inp)
    out, plan, _ = run_gpu(inp, kernel)
    assert_close(out, ref, wl.kv_dtype, f"ragged bs={bs} S={plan.num_splits}")


def test_window_sink_graph_replay():
    """Captured once as a CUDA graph, replayed 10 times with freshly drawn lengths,
    block tables and sink logits (aiter PR #5628, Validation: graph replay after
    changing lengths and sink logits). Pages before each window map to a NaN page."""
    wl = W.window_sink_bf16()
    inp = W.make_window_pool_inputs(wl, 1005, device="cuda")
    W.redraw_window_lengths(inp)
    plan = plan_for(wl, host_ctx=None, num_pages=inp.num_pages, max_ctx_hint=32768)
    ws = poisoned_workspace(plan)
    out = new_out(wl)
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        B.run(inp, ws, out)          # warm-up outside capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        B.run(inp, ws, out)
    for rep in range(10):
        ctx = W.redraw_window_lengths(inp)
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        ref, _ = oracle_out(inp)
        assert_close(out, ref, wl.kv_dtype, f"replay {rep} ctx[:4]={ctx[:4]}")


def persistent_pass_requests(plan, n_sm: int):
    """Requests whose split items open and close each pass of the persistent grid: the
    kernels give CTA c the items c, c + grid, c + 2 grid, ... of the (request x kv head,
    split) list, so pass k covers items [k grid, (k + 1) grid)."""
    S, Hkv = plan.num_splits, plan.desc.num_kv_heads
    n_items = plan.batch * Hkv * S
    grid = min(n_items, n_sm)
    idx = set()
    for first in range(0, n_items, grid):
        last = min(n_items, first + grid) - 1
        idx.add(first // S // Hkv)
        idx.add(last // S // Hkv)
        idx.add((first + last) // 2 // S // Hkv)
    return sorted(idx)


def test_mtp4_fp8_full_size_sampled():
    """The full batch-200 x 200,000 workload in the launch configuration the benchmark
    times; the oracle checks whole requests from every pass of the persistent grid (the
    first, middle and last request of each pass)."""
    wl = W.mtp4_fp8_long()
    inp = W.make_inputs(wl, 1003, device="cuda")
    out, plan, _ = run_gpu(inp)
    assert plan.num_splits > 1
    idx = persistent_pass_requests(plan, torch.cuda.get_device_properties(0).multi_processor_count)
    assert 8 <= len(idx) <= 16, idx
    sub = W.gather_requests(inp, idx)
    ref, _ = oracle_out(sub)
    assert_close(out[idx], ref, wl.kv_dtype, "full-size sampled")
    assert torch.isfinite(out.float()).all()
    del inp
    torch.cuda.empty_cache()


# --- edge cases and invariants -----------------------------------------------

@pytest.mark.parametrize("kernel", KERNELS)
def test_empty_and_short_contexts(kernel):
    wl = W.mtp4_fp8_long(batch=5, ctx=1).replace(ctx=[0, 1, 2, 3, 5])
    inp = _inputs(wl, 7)
    ref, _ = oracle_out(inp)
    for S in (1, 2):
        out, _, _ = run_gpu(inp, kernel, splits=S)
        assert_close(out, ref, wl.kv_dtype, f"short S={S}")
        assert out[0].float().abs().max() == 0


@pytest.mark.parametrize("kernel", KERNELS)
def test_split_count_does_not_change_the_result(kernel):
    wl = W.verify16_int8().replace(ctx=[5000])
    inp = _inputs(wl, 8)
    ref, _ = oracle_out(inp)
    outs = []
    for S in (1, 2, 3, 5, 7, 16):
        out, _, _ = run_gpu(inp, kernel, splits=S)
        assert_close(out, ref, wl.kv_dtype, f"S={S}")
        outs.append(out.float())
    for o in outs[1:]:
        assert (o - outs[0]).abs().max() <= 2 * 5e-3


@pytest.mark.parametrize("kernel", KERNELS)
def test_page_permutation_invariance(kernel):
    wl = W.window_sink_bf16(batch=3, max_ctx=3000).replace(ctx=[3000, 1000, 17], window=0, sinks=True)
    inp = _inputs(wl, 9, poison=False)
    out1, _, _ = run_gpu(inp, kernel, splits=3)
    perm = torch.randperm(inp.num_pages, generator=torch.Generator().manual_seed(3)).cuda()
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(inp.num_pages, device="cuda")
    inp.k_cache = inp.k_cache[perm].contiguous()
    inp.v_cache = inp.v_cache[perm].contiguous()
    inp.block_table = inv[inp.block_table.long()].to(torch.int32)
    out2, _, _ = run_gpu(inp, kernel, splits=3)
    assert torch.equal(out1, out2)


@pytest.mark.parametrize("kernel", KERNELS)
def test_determinism(kernel):
    """num_splits = 1 is bit-identical run to run; so is every S (fixed merge order, no
    atomics)."""
    wl = W.mtp4_fp8_long(batch=3, ctx=9000)
    inp = _inputs(wl, 10)
    for S in (1, 4):
        a, plan, ws = run_gpu(inp, kernel, splits=S)
        for _ in range(2):
            b, _, _ = run_gpu(inp, kernel, splits=S, plan=plan, ws=ws)
            assert torch.equal(a, b)


@pytest.mark.parametrize("kernel", KERNELS)
def test_stage_entry_points_compose(kernel):
    wl = W.mtp4_fp8_long(batch=2, ctx=3000)
    inp = _inputs(wl, 11)
    ref_out, plan, ws = run_gpu(inp, kernel, splits=4)
    out = new_out(wl)
    args = (inp.q, inp.k_cache, inp.v_cache, inp.block_table, inp.context_lens, wl.Lq, inp.kv_scales, inp.sinks,
            wl.window, 4, ws, out)
    B.tllm_decode_attn_partial(*args)
    B.tllm_decode_attn_combine(*args)
    torch.cuda.synchronize()
    assert torch.equal(out, ref_out)


REC_TORCH = {B.TLLM_RECORD_F32: torch.float32, B.TLLM_RECORD_BF16: torch.bfloat16, B.TLLM_RECORD_F16: torch.float16}


@pytest.mark.parametrize("rec", [B.TLLM_RECORD_F32, B.TLLM_RECORD_BF16, B.TLLM_RECORD_F16])
@pytest.mark.parametrize("kernel", KERNELS)
def test_partial_records_match_oracle_partials(kernel, rec):
    """The split records themselves: O_s and LSE_s of every split equal the oracle's
    attention restricted to that split's key range, in each record type."""
    wl = W.mtp4_fp8_long(batch=2, ctx=1).replace(ctx=[3001, 1500], window=700, sinks=True)
    inp = _inputs(wl, 12)
    S = 3
    desc = B.desc_for(wl, kernel, num_pages=inp.num_pages, record_type=rec)
    plan = B.tllm_decode_attn_plan(desc, wl.B, wl.Lq, wl.window, host_ctx_lens=wl.ctx, splits_override=S)
    ws = poisoned_workspace(plan)
    out = new_out(wl)
    B.tllm_decode_attn_partial(inp.q, inp.k_cache, inp.v_cache, inp.block_table, inp.context_lens, wl.Lq,
                               inp.kv_scales, inp.sinks, wl.window, S, ws, out)
    torch.cuda.synchronize()
    so, lo, oo = B.tllm_decode_attn_workspace_layout(plan)
    R, D, Smax = plan.rows, wl.D, plan.max_splits
    lse = ws.buffer[lo:lo + wl.B * wl.Hkv * Smax * R * 4].view(torch.float32).view(wl.B, wl.Hkv, Smax, R).cpu()
    esz = torch.finfo(REC_TORCH[rec]).bits // 8
    orec = ws.buffer[oo:oo + wl.B * wl.Hkv * Smax * R * D * esz].view(REC_TORCH[rec]).view(
        wl.B, wl.Hkv, Smax, R, D).float().cpu()
    G = wl.G
    for b, ctx in enumerate(wl.ctx):
        t0, t1, n = B.tllm_decode_attn_split_range(plan, ctx, wl.Lq, wl.window, S, 0)
        assert n > 1
        for s in range(n):
            t0, t1, _ = B.tllm_decode_attn_split_range(plan, ctx, wl.Lq, wl.window, S, s)
            o_ref, l_ref = oracle_out(inp, sinks=None, key_range=(t0, t1))
            for r in range(R):
                i, h = r // G, (r % G)
                lr = l_ref[b, i, h]
                lg = float(lse[b, 0, s, r]) * np.log(2.0)
                if np.isneginf(lr):
                    assert lg == float("-inf")
                    assert torch.all(orec[b, 0, s, r] == 0)
                else:
                    assert abs(lg - lr) <= 1e-3 * max(1.0, abs(lr)), (b, s, r, lg, lr)
                    np.testing.assert_allclose(orec[b, 0, s, r].double().numpy(), o_ref[b, i, h], rtol=5e-3,
                                               atol=5e-3)


@pytest.mark.parametrize("kernel", KERNELS)
def test_device_data_faults_set_status_and_stay_finite(kernel):
    _check_device_data_faults(W.mtp4_fp8_long(batch=3, ctx=1000), kernel)


@pytest.mark.parametrize("wl,kernel", [
    (W.verify16_int8().replace(ctx=[1000, 1000, 1000]), B.TLLM_KERNEL_TC_I8),
    (W.window_sink_bf16(batch=3).replace(ctx=[1000] * 3, Hq=32, Hkv=4, Lq=4, window=0, sinks=False),
     B.TLLM_KERNEL_TC_I8),
    (W.window_sink_bf16(batch=3).replace(ctx=[1000] * 3, Hq=32, Hkv=2, Lq=1, D=256, window=0, sinks=False),
     B.TLLM_KERNEL_SIMT),
    (W.window_sink_bf16(batch=3).replace(ctx=[1000] * 3, Hq=32, Hkv=2, Lq=1, D=256, window=0, sinks=False),
     B.TLLM_KERNEL_TC_I8),
    (W.single_decode().replace(ctx=[1000] * 3), B.TLLM_KERNEL_SIMT),
    (W.window_sink_bf16(batch=3).replace(ctx=[1000] * 3, window=0, sinks=False), B.TLLM_KERNEL_TC_B16),
])
def test_device_data_faults_in_every_kernel(wl, kernel):
    """A clamped context length and out-of-range page ids (too large, negative) in the widening,
    CUDA-core (one and several row blocks) and 16-bit kernels: flagged, masked, finite."""
    _check_device_data_faults(wl, kernel)


def _check_device_data_faults(wl, kernel):
    inp = _inputs(wl, 13, poison=False)
    plan = plan_for(wl, kernel, 2, num_pages=inp.num_pages)
    ws = poisoned_workspace(plan)
    # a context length beyond the block table: clamped to max_blocks * bs
    inp.context_lens[1] = 10 ** 6
    out, _, _ = run_gpu(inp, kernel, plan=plan, ws=ws)
    flags = B.tllm_decode_attn_read_status(ws, reset=True)
    assert flags & B.TLLM_FLAG_CTX_CLAMPED
    inp.context_lens[1] = wl.max_blocks * wl.bs
    ref, _ = oracle_out(inp)
    assert_close(out, ref, wl.kv_dtype, "clamped ctx")
    # a page id outside the cache: masked, flagged, finite
    inp.block_table[2, 3] = inp.num_pages + 5
    out, _, _ = run_gpu(inp, kernel, plan=plan, ws=ws)
    flags = B.tllm_decode_attn_read_status(ws, reset=True)
    assert flags & B.TLLM_FLAG_BAD_PAGE
    assert torch.isfinite(out.float()).all()
    inp.block_table[2, 3] = -7
    out, _, _ = run_gpu(inp, kernel, plan=plan, ws=ws)
    assert B.tllm_decode_attn_read_status(ws, reset=True) & B.TLLM_FLAG_BAD_PAGE
    assert torch.isfinite(out.float()).all()


# --- fuzz grid ---------------------------------------------------------------------

def _fuzz_cases(n=40, seed=123):
    rng = random.Random(seed)
    kvs = ["f16", "bf16", "e4m3", "i8"]
    for k in range(n):
        kv = kvs[k % 4]
        q = "f16" if kv == "f16" else rng.choice(["bf16", "f32"])
        Hkv = rng.choice([1, 2, 4])
        G = rng.choice([1, 2, 3, 4, 7, 8])
        D = rng.choice([64, 128, 256])
        bs = rng.choice([1, 8, 16, 32, 64, 128])
        Lq = rng.choice([1, 1, 2, 4, 16])
        B_ = rng.choice([1, 2, 3, 5])
        ctx = [rng.choice([0, 1, 15, 16, 17, 100, 1000, 3333, rng.randint(1, 6000)]) for _ in range(B_)]
        window = rng.choice([0, 0, 1, 7, 64, 500])
        sinks = rng.random() < 0.4
        S = rng.choice([1, 2, 3, 5, 8, 16])
        out = rng.choice(["f32", "bf16", "f16"])
        yield pytest.param(dict(ctx=ctx, Lq=Lq, Hq=Hkv * G, Hkv=Hkv, D=D, bs=bs, q_dtype=q, kv_dtype=kv,
                                out_dtype=out, window=window, sinks=sinks, extra_pages=3,
                                kv_std=0.5 if kv == "e4m3" else 1.0, scale_range=(0.005, 0.02) if kv == "i8"
                                else (0.5, 2.0)), S, id=f"f{k}")


@pytest.mark.parametrize("spec,S", list(_fuzz_cases()))
@pytest.mark.parametrize("kernel", KERNELS)
def test_fuzz(spec, S, kernel):
    wl = W.Workload("fuzz", **spec)
    inp = _inputs(wl, 2000 + S)
    ref, _ = oracle_out(inp)
    out, _, _ = run_gpu(inp, kernel, splits=S)
    assert_close(out, ref, wl.kv_dtype, f"fuzz {spec} S={S}")


# --- FP8 tensor-core kernel specifics -------------------------------------------

TC = B.TLLM_KERNEL_TC_FP8


@pytest.mark.parametrize("Hq,Hkv,Lq", [(16, 1, 4), (8, 1, 8), (4, 1, 16), (1, 1, 1), (32, 2, 2), (64, 1, 1),
                                       (16, 2, 3), (2, 2, 1)])
@pytest.mark.parametrize("bs", [8, 16, 64, 128])
def test_tc_fp8_row_shapes(Hq, Hkv, Lq, bs):
    wl = W.mtp4_fp8_long(batch=3, ctx=1).replace(ctx=[5000, 777, 129], Hq=Hq, Hkv=Hkv, Lq=Lq, bs=bs, extra_pages=3)
    inp = _inputs(wl, 40 + bs)
    plan = plan_for(wl, TC, 2, num_pages=inp.num_pages)
    assert plan.kernel == TC
    ref, _ = oracle_out(inp)
    for S in (1, 2):
        out, _, _ = run_gpu(inp, TC, splits=S)
        assert_close(out, ref, wl.kv_dtype, f"tc rows Hq{Hq} Hkv{Hkv} Lq{Lq} bs{bs} S{S}")


@pytest.mark.parametrize("window", [1, 100, 128, 300, 4096])
def test_tc_fp8_window_and_sinks(window):
    wl = W.mtp4_fp8_long(batch=4, ctx=1).replace(ctx=[9000, 4100, 250, 5], window=window, sinks=True,
                                                 extra_pages=2)
    inp = _inputs(wl, 50 + window)
    ref, _ = oracle_out(inp)
    for S in (1, 3):
        out, _, _ = run_gpu(inp, TC, splits=S)
        assert_close(out, ref, wl.kv_dtype, f"tc window {window} S{S}")


def test_tc_fp8_scale_edge_cases():
    """V scales that grow along the context (the P scale shrinks: O is rescaled by powers
    of two), zero V scales (keys still count in the denominator) and negative scales."""
    wl = W.mtp4_fp8_long(batch=3, ctx=1).replace(ctx=[6000, 3000, 700])
    inp = _inputs(wl, 60, poison=False)
    sc = inp.kv_scales
    for b in range(wl.B):
        n = (wl.ctx[b] + wl.bs - 1) // wl.bs
        pages = inp.block_table[b, :n].long()
        ramp = torch.logspace(-3, 3, n, device="cuda")
        sc[1][pages] = ramp[:, None, None].expand(n, wl.Hkv, wl.bs)
    sc[1].view(-1)[::7] = 0.0
    sc[0].view(-1)[::11] *= -1.0
    sc[1].view(-1)[::13] *= -1.0
    ref, _ = oracle_out(inp)
    cond, _ = oracle_out(abs_value_inputs(inp))
    for S in (1, 2):
        out, _, _ = run_gpu(inp, TC, splits=S)
        assert_close_conditioned(out, ref, cond, wl.kv_dtype, f"tc scales S{S}")
        g, _, _ = run_gpu(inp, B.TLLM_KERNEL_GENERIC, splits=S)
        assert_close_conditioned(g, ref, cond, wl.kv_dtype, f"generic scales S{S}")


def test_tc_fp8_matches_generic_kernel():
    wl = W.mtp4_fp8_long(batch=4, ctx=1).replace(ctx=[30000, 12000, 129, 1])
    inp = _inputs(wl, 70)
    a, _, _ = run_gpu(inp, TC, splits=3)
    g, _, _ = run_gpu(inp, B.TLLM_KERNEL_GENERIC, splits=3)
    ref, _ = oracle_out(inp)
    assert_close(a, ref, wl.kv_dtype, "tc")
    assert_close(g, ref, wl.kv_dtype, "generic")


@pytest.mark.parametrize("splits", [0, 16, 45])
def test_tc_fp8_repeatable(splits):
    """Every warp of the tensor-core kernel reads shared state only after the barrier that
    publishes it: repeated runs give bit-identical outputs, for any split count (the combine
    visits splits in a fixed order)."""
    wl = W.mtp4_fp8_long(batch=6, ctx=1).replace(ctx=[20000, 12345, 777, 4, 3, 40001], extra_pages=10)
    inp = _inputs(wl, 1003)
    first, plan, _ = run_gpu(inp, TC, splits=splits)
    for _ in range(6):
        again, _, _ = run_gpu(inp, TC, splits=splits)
        assert torch.equal(first, again), f"S={plan.num_splits}: outputs differ between runs"


# --- the pipelined CUDA-core kernel for few packed rows -------------------------

SIMT = B.TLLM_KERNEL_SIMT
SIMT_DTYPES = [("f16", "f16", "f32"), ("bf16", "bf16", "bf16"), ("bf16", "e4m3", "bf16"), ("bf16", "i8", "bf16")]


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("q_kv_out", SIMT_DTYPES)
def test_simt_dtypes_and_head_dims(D, q_kv_out):
    """Every KV type the kernel reads, at every head_dim it supports, with ragged lengths
    (shorter than a tile, not a multiple of the page, several tiles) and 1..4 splits."""
    qd, kvd, od = q_kv_out
    wl = W.single_decode().replace(ctx=[3001, 100, 17, 1], D=D, Hq=8, Hkv=2, q_dtype=qd, kv_dtype=kvd,
                                   out_dtype=od, scale=0.0, extra_pages=4)
    inp = _inputs(wl, 80 + D)
    plan = plan_for(wl, SIMT, 2, num_pages=inp.num_pages)
    assert plan.kernel == SIMT
    ref, _ = oracle_out(inp)
    for S in (1, 2, 4):
        out, _, _ = run_gpu(inp, SIMT, splits=S)
        assert_close(out, ref, wl.kv_dtype, f"simt {kvd} D{D} S{S}")


@pytest.mark.parametrize("bs", [8, 16, 64, 128])
@pytest.mark.parametrize("Hq,Hkv,Lq", [(7, 1, 1), (8, 2, 1), (4, 2, 4), (16, 4, 2), (2, 2, 1)])
def test_simt_rows_and_block_sizes(Hq, Hkv, Lq, bs):
    """Packed rows 1..8 (GQA groups times query rows, causal among the query rows) at every
    block size, including pages larger than a tile."""
    wl = W.single_decode().replace(ctx=[2500, 333, 64], Hq=Hq, Hkv=Hkv, Lq=Lq, D=128, bs=bs, q_dtype="bf16",
                                   kv_dtype="bf16", out_dtype="bf16", scale=0.0, extra_pages=3)
    inp = _inputs(wl, 90 + bs + Hq)
    ref, _ = oracle_out(inp)
    for S in (1, 3):
        out, plan, _ = run_gpu(inp, SIMT, splits=S)
        assert plan.kernel == SIMT
        assert_close(out, ref, wl.kv_dtype, f"simt rows Hq{Hq} Hkv{Hkv} Lq{Lq} bs{bs} S{S}")


@pytest.mark.parametrize("window", [1, 37, 64, 4096])
def test_simt_window_and_sinks(window):
    wl = W.window_sink_bf16(batch=5).replace(ctx=[9000, 4097, 300, 2, 1], window=window, extra_pages=2)
    inp = _inputs(wl, 100 + window)
    ref, _ = oracle_out(inp)
    for S in (1, 4):
        out, _, _ = run_gpu(inp, SIMT, splits=S)
        assert_close(out, ref, wl.kv_dtype, f"simt window {window} S{S}")


def test_simt_bad_pages_are_masked_and_flagged():
    """A page id outside the pool: its tokens are skipped (never read) and the status word
    says so. The request is then the same masked problem the generic kernel solves; the
    other request is untouched and matches the oracle."""
    wl = W.single_decode().replace(ctx=[700, 500], Hq=4, Hkv=1, D=128, q_dtype="bf16", kv_dtype="bf16",
                                   out_dtype="bf16", scale=0.0, extra_pages=2)
    inp = _inputs(wl, 110, poison=False)
    ref, _ = oracle_out(inp)
    inp.block_table[0, 3] = inp.num_pages + 5          # page 3 of request 0: tokens 48..63
    out, plan, ws = run_gpu(inp, SIMT, splits=2)
    assert_close(out[1:], ref[1:], wl.kv_dtype, "simt: request without a bad page")
    assert B.tllm_decode_attn_read_status(ws) & B.TLLM_FLAG_BAD_PAGE
    g, _, gws = run_gpu(inp, B.TLLM_KERNEL_GENERIC, splits=2)
    assert B.tllm_decode_attn_read_status(gws) & B.TLLM_FLAG_BAD_PAGE
    assert_close(out, g.double().cpu().numpy(), wl.kv_dtype, "simt vs generic with a bad page")


def test_simt_repeatable():
    wl = W.window_sink_bf16(batch=6).replace(ctx=[20000, 5000, 4096, 777, 3, 1], extra_pages=2)
    inp = _inputs(wl, 120)
    for S in (0, 5):
        first, plan, _ = run_gpu(inp, SIMT, splits=S)
        for _ in range(4):
            again, _, _ = run_gpu(inp, SIMT, splits=S)
            assert torch.equal(first, again), f"S={plan.num_splits}: outputs differ between runs"


# --- the 16-bit tensor-core kernel for few rows (tcgen05, tokens on the MMA's M) ------

TCB16 = B.TLLM_KERNEL_TC_B16
B16_DTYPES = [("f16", "f16", "f32"), ("bf16", "bf16", "bf16"), ("f16", "f16", "f16"), ("bf16", "bf16", "f32")]


@pytest.mark.parametrize("q_kv_out", B16_DTYPES)
def test_tc_b16_dtypes(q_kv_out):
    """f16 and bf16 caches (the query in the same type) into every output type, with ragged
    lengths (shorter than a tile, not a multiple of the page, several tiles) and 1..4 splits."""
    qd, kvd, od = q_kv_out
    wl = W.single_decode().replace(ctx=[3001, 100, 17, 1], D=128, Hq=8, Hkv=2, q_dtype=qd, kv_dtype=kvd,
                                   out_dtype=od, scale=0.0, extra_pages=4)
    inp = _inputs(wl, 130 + len(qd))
    ref, _ = oracle_out(inp)
    for S in (1, 2, 4):
        out, plan, _ = run_gpu(inp, TCB16, splits=S)
        assert plan.kernel == TCB16
        assert_close(out, ref, wl.kv_dtype, f"tc_b16 {kvd}->{od} S{S}")


@pytest.mark.parametrize("bs", [8, 16, 64, 128])
@pytest.mark.parametrize("Hq,Hkv,Lq", [(7, 1, 1), (8, 2, 1), (4, 2, 4), (2, 2, 1), (16, 1, 1), (4, 1, 3), (8, 1, 2)])
def test_tc_b16_rows_and_block_sizes(Hq, Hkv, Lq, bs):
    """Packed rows 1..16 (GQA groups times query rows, causal among the query rows; 4, 8 and
    16 are the padded row counts of the kernel's variants) at every block size."""
    wl = W.single_decode().replace(ctx=[2500, 333, 64], Hq=Hq, Hkv=Hkv, Lq=Lq, D=128, bs=bs, q_dtype="bf16",
                                   kv_dtype="bf16", out_dtype="bf16", scale=0.0, extra_pages=3)
    inp = _inputs(wl, 140 + bs + Hq + Lq)
    ref, _ = oracle_out(inp)
    for S in (1, 3):
        out, plan, _ = run_gpu(inp, TCB16, splits=S)
        assert plan.kernel == TCB16
        assert_close(out, ref, wl.kv_dtype, f"tc_b16 rows Hq{Hq} Hkv{Hkv} Lq{Lq} bs{bs} S{S}")


@pytest.mark.parametrize("window", [1, 37, 128, 4096])
def test_tc_b16_window_and_sinks(window):
    wl = W.window_sink_bf16(batch=5).replace(ctx=[9000, 4097, 300, 2, 1], window=window, extra_pages=2)
    inp = _inputs(wl, 150 + window)
    ref, _ = oracle_out(inp)
    for S in (1, 4):
        out, plan, _ = run_gpu(inp, TCB16, splits=S)
        assert plan.kernel == TCB16
        assert_close(out, ref, wl.kv_dtype, f"tc_b16 window {window} S{S}")


def test_tc_b16_large_scores_and_peaked_rows():
    """Scores of magnitude up to ~60 in log2 units: a few dominant keys per row, rows whose
    maximum jumps late in the context (the O rescale), and near-cancelling value rows."""
    wl = W.single_decode().replace(ctx=[5000, 700], Hq=8, Hkv=1, D=128, q_dtype="bf16", kv_dtype="bf16",
                                   out_dtype="f32", scale=0.0, extra_pages=2)
    inp = _inputs(wl, 160)
    inp.q.mul_(4.0)
    flat = inp.k_cache.view(-1, wl.D)
    flat[::97].mul_(6.0)                     # a sparse set of large keys
    ref, _ = oracle_out(inp)
    for S in (1, 2, 5):
        out, _, _ = run_gpu(inp, TCB16, splits=S)
        assert_close(out, ref, wl.kv_dtype, f"tc_b16 large scores S{S}")


def test_tc_b16_bad_pages_are_masked_and_flagged():
    wl = W.single_decode().replace(ctx=[700, 500], Hq=4, Hkv=1, D=128, q_dtype="bf16", kv_dtype="bf16",
                                   out_dtype="bf16", scale=0.0, extra_pages=2)
    inp = _inputs(wl, 170, poison=False)
    ref, _ = oracle_out(inp)
    inp.block_table[0, 3] = inp.num_pages + 5          # page 3 of request 0: tokens 48..63
    out, plan, ws = run_gpu(inp, TCB16, splits=2)
    assert_close(out[1:], ref[1:], wl.kv_dtype, "tc_b16: request without a bad page")
    assert B.tllm_decode_attn_read_status(ws) & B.TLLM_FLAG_BAD_PAGE
    g, _, _ = run_gpu(inp, B.TLLM_KERNEL_GENERIC, splits=2)
    assert_close(out, g.double().cpu().numpy(), wl.kv_dtype, "tc_b16 vs generic with a bad page")


def test_tc_b16_repeatable():
    wl = W.window_sink_bf16(batch=6).replace(ctx=[20000, 5000, 4096, 777, 3, 1], extra_pages=2)
    inp = _inputs(wl, 180)
    for S in (0, 5):
        first, plan, _ = run_gpu(inp, TCB16, splits=S)
        for _ in range(4):
            again, _, _ = run_gpu(inp, TCB16, splits=S)
            assert torch.equal(first, again), f"S={plan.num_splits}: outputs differ between runs"


# --- the INT8 tensor-core kernel (tcgen05, int8 widened to f16) ---------------------

TCI8 = B.TLLM_KERNEL_TC_I8


@pytest.mark.parametrize("D", [128, 256])
@pytest.mark.parametrize("Hq,Hkv,Lq", [(24, 4, 16), (8, 1, 16), (4, 4, 4), (16, 2, 1), (32, 1, 4)])
def test_tc_i8_rows_and_head_dims(Hq, Hkv, Lq, D):
    """Packed rows 4..128 (the verify shape is 6 x 16 = 96), head_dim 128 and 256, ragged
    lengths (several tiles, a tail, shorter than a tile) and 1..3 splits."""
    wl = W.verify16_int8().replace(ctx=[3000, 700, 65, 17], Hq=Hq, Hkv=Hkv, Lq=Lq, D=D, extra_pages=4)
    inp = _inputs(wl, 130 + D + Hq)
    plan = plan_for(wl, TCI8, 2, num_pages=inp.num_pages)
    assert plan.kernel == TCI8
    ref, _ = oracle_out(inp)
    for S in (1, 3):
        out, _, _ = run_gpu(inp, TCI8, splits=S)
        assert_close(out, ref, wl.kv_dtype, f"tc_i8 Hq{Hq} Hkv{Hkv} Lq{Lq} D{D} S{S}")


@pytest.mark.parametrize("bs", [8, 16, 64, 128])
def test_tc_i8_block_sizes(bs):
    wl = W.verify16_int8().replace(ctx=[2500, 333, 129], bs=bs, extra_pages=3)
    inp = _inputs(wl, 140 + bs)
    ref, _ = oracle_out(inp)
    for S in (1, 4):
        out, plan, _ = run_gpu(inp, TCI8, splits=S)
        assert plan.kernel == TCI8
        assert_close(out, ref, wl.kv_dtype, f"tc_i8 bs{bs} S{S}")


@pytest.mark.parametrize("window", [1, 100, 4096])
def test_tc_i8_window_and_sinks(window):
    wl = W.verify16_int8().replace(ctx=[9000, 4100, 250, 5], window=window, sinks=True, extra_pages=2)
    inp = _inputs(wl, 150 + window)
    ref, _ = oracle_out(inp)
    for S in (1, 3):
        out, _, _ = run_gpu(inp, TCI8, splits=S)
        assert_close(out, ref, wl.kv_dtype, f"tc_i8 window {window} S{S}")


def test_tc_i8_scale_edge_cases():
    """V scales growing over six decades, zero and negative scales (the conditioned bound:
    outputs that are small differences of large terms)."""
    wl = W.verify16_int8().replace(ctx=[6000, 3000, 700])
    inp = _inputs(wl, 160, poison=False)
    sc = inp.kv_scales
    for b in range(wl.B):
        n = (wl.ctx[b] + wl.bs - 1) // wl.bs
        pages = inp.block_table[b, :n].long()
        ramp = torch.logspace(-3, 3, n, device="cuda")
        sc[1][pages] = ramp[:, None, None].expand(n, wl.Hkv, wl.bs)
    sc[1].view(-1)[::7] = 0.0
    sc[0].view(-1)[::11] *= -1.0
    sc[1].view(-1)[::13] *= -1.0
    ref, _ = oracle_out(inp)
    cond, _ = oracle_out(abs_value_inputs(inp))
    for S in (1, 2):
        out, _, _ = run_gpu(inp, TCI8, splits=S)
        assert_close_conditioned(out, ref, cond, wl.kv_dtype, f"tc_i8 scales S{S}")


@pytest.mark.parametrize("q_dtype,out_dtype", [("f16", "f16"), ("f16", "f32"), ("bf16", "f32")])
def test_tc_i8_query_and_output_types(q_dtype, out_dtype):
    wl = W.verify16_int8().replace(ctx=[2100, 640, 33], q_dtype=q_dtype, out_dtype=out_dtype, extra_pages=2)
    inp = _inputs(wl, 175)
    ref, _ = oracle_out(inp)
    for S in (1, 3):
        out, plan, _ = run_gpu(inp, TCI8, splits=S)
        assert plan.kernel == TCI8
        assert_close(out, ref, wl.kv_dtype, f"tc_i8 q {q_dtype} out {out_dtype} S{S}")


def test_tc_i8_query_magnitudes():
    """A bf16 query row enters the f16 contraction after a power-of-two scale: rows spread over
    the bf16 range (2^-100 .. 2^60), rows holding elements 2^-30 of their largest, and an all-zero
    row all match the oracle."""
    wl = W.verify16_int8().replace(ctx=[3000, 900], extra_pages=2)
    inp = _inputs(wl, 180)
    q = inp.q.float()
    exps = [-100, -40, -8, 0, 6, 20, 60]
    for b in range(wl.B):
        for i in range(wl.Lq):
            for h in range(wl.Hq):
                q[b, i, h] *= 2.0 ** exps[(b * 7 + i * 3 + h) % len(exps)]
    q[:, 1, :, ::3] *= 2.0 ** -30                 # elements far below the row's largest
    q[0, 2, 5] = 0.0                              # a zero row: uniform weights
    inp.q.copy_(q.to(inp.q.dtype))
    ref, _ = oracle_out(inp)
    for S in (1, 2):
        out, _, _ = run_gpu(inp, TCI8, splits=S)
        assert_close(out, ref, wl.kv_dtype, f"tc_i8 query magnitudes S{S}")


def test_tc_i8_repeatable():
    wl = W.verify16_int8().replace(ctx=[20676, 5000, 777, 3], extra_pages=2)
    inp = _inputs(wl, 170)
    for S in (0, 7):
        first, plan, _ = run_gpu(inp, TCI8, splits=S)
        for _ in range(4):
            again, _, _ = run_gpu(inp, TCI8, splits=S)
            assert torch.equal(first, again), f"S={plan.num_splits}: outputs differ between runs"


# --- contiguous cache (no block table) ----------------------------------------------

def _contiguous(inp):
    """The same problem in a contiguous cache: block i of request b moved to page
    b * max_blocks + i; unused pages poisoned. Returns the new caches and scales."""
    wl = inp.wl
    n_pages = wl.B * wl.max_blocks
    shape = (n_pages,) + tuple(inp.k_cache.shape[1:])
    k = torch.empty(shape, dtype=inp.k_cache.dtype, device="cuda")
    v = torch.empty_like(k)
    if wl.kv_dtype == "e4m3":
        k.view(torch.uint8).fill_(0x7F)
        v.view(torch.uint8).fill_(0x7F)
    elif wl.kv_dtype == "i8":
        k.zero_()
        v.zero_()
    else:
        k.fill_(float("nan"))
        v.fill_(float("nan"))
    sc = None
    if inp.kv_scales is not None:
        sc = torch.full((2, n_pages) + tuple(inp.kv_scales.shape[2:]), float("nan"), dtype=torch.float32,
                        device="cuda")
    for b in range(wl.B):
        n = (int(inp.context_lens[b]) + wl.bs - 1) // wl.bs
        src = inp.block_table[b, :n].long()
        dst = torch.arange(b * wl.max_blocks, b * wl.max_blocks + n, device="cuda")
        k[dst] = inp.k_cache[src]
        v[dst] = inp.v_cache[src]
        if sc is not None:
            sc[:, dst] = inp.kv_scales[:, src]
    return k, v, sc, n_pages


@pytest.mark.parametrize("wl,kernel", [
    (W.mtp4_fp8_long(batch=3, ctx=1).replace(ctx=[5000, 777, 3]), B.TLLM_KERNEL_TC_FP8),
    (W.verify16_int8().replace(ctx=[3000, 700]), B.TLLM_KERNEL_TC_I8),
    (W.window_sink_bf16(batch=3).replace(ctx=[6000, 4097, 17]), B.TLLM_KERNEL_TC_B16),
    (W.single_decode().replace(ctx=[2048, 300]), B.TLLM_KERNEL_SIMT),
    (W.single_decode().replace(ctx=[2048, 300]), B.TLLM_KERNEL_GENERIC),
    (W.window_sink_bf16(batch=2).replace(ctx=[3000, 650], Hq=32, Hkv=4, Lq=4), B.TLLM_KERNEL_TC_I8),
    (W.window_sink_bf16(batch=2).replace(ctx=[3000, 650], Hq=32, Hkv=4, Lq=4, D=64, kv_dtype="f16"),
     B.TLLM_KERNEL_TC_I8),
    (W.window_sink_bf16(batch=2).replace(ctx=[3000, 650], Hq=32, Hkv=2, Lq=2, D=256), B.TLLM_KERNEL_SIMT),
])
def test_contiguous_cache_without_block_table(wl, kernel):
    """block_table = NULL: request b's block i is page b * max_blocks + i. The result equals
    the oracle on the paged layout of the same data."""
    inp = _inputs(wl, 190, poison=False)
    ref, _ = oracle_out(inp)
    k, v, sc, n_pages = _contiguous(inp)
    for S in (1, 3):
        plan = plan_for(wl, kernel, S, num_pages=n_pages)
        assert plan.kernel == kernel
        ws = poisoned_workspace(plan)
        out = new_out(wl)
        B.tllm_decode_attn_splitkv(inp.q, k, v, None, inp.context_lens, wl.Lq, sc, inp.sinks, wl.window, S, ws,
                                   out)
        torch.cuda.synchronize()
        assert not (B.tllm_decode_attn_read_status(ws) & (B.TLLM_FLAG_TIMEOUT | B.TLLM_FLAG_BAD_PAGE))
        assert_close(out, ref, wl.kv_dtype, f"contiguous {wl.name} kernel {kernel} S{S}")


# --- dimension-major ("transposed") V cache ----------------------------------------------

@pytest.mark.parametrize("bs", [16, 32, 128])
@pytest.mark.parametrize("kernel", [B.TLLM_KERNEL_TC_FP8, B.TLLM_KERNEL_GENERIC])
def test_dim_major_v_cache(bs, kernel):
    """V stored [num_pages, Hkv, D, bs] (aiter PR #5628, Performance table: the transposed V
    layout): the same problem as the token-major cache, checked against the oracle on the
    token-major data. Partial tiles (window, short requests) zero the unread tokens' columns."""
    wl = W.mtp4_fp8_long(batch=4, ctx=1).replace(ctx=[7000, 1500, 130, 5], bs=bs, window=700, sinks=True,
                                                 extra_pages=3)
    inp = _inputs(wl, 200 + bs)
    ref, _ = oracle_out(inp)
    v_dm = inp.v_cache.transpose(-1, -2).contiguous()
    for S in (1, 3):
        desc = B.desc_for(wl, kernel, num_pages=inp.num_pages, v_layout=B.TLLM_V_DIM_MAJOR)
        plan = B.tllm_decode_attn_plan(desc, wl.B, wl.Lq, wl.window, host_ctx_lens=wl.ctx, splits_override=S)
        assert plan.kernel == kernel
        ws = poisoned_workspace(plan)
        out = new_out(wl)
        B.tllm_decode_attn_splitkv(inp.q, inp.k_cache, v_dm, inp.block_table, inp.context_lens, wl.Lq,
                                   inp.kv_scales, inp.sinks, wl.window, S, ws, out)
        torch.cuda.synchronize()
        assert not (B.tllm_decode_attn_read_status(ws) & B.TLLM_FLAG_TIMEOUT)
        assert_close(out, ref, wl.kv_dtype, f"dim-major V bs{bs} kernel {kernel} S{S}")



@pytest.mark.parametrize("kv_dtype,q_dtype,D,bs,Hq,Hkv,Lq", [
    ("f16", "f16", 64, 8, 14, 2, 1), ("bf16", "bf16", 128, 16, 32, 8, 1), ("bf16", "bf16", 256, 32, 32, 2, 1),
    ("i8", "bf16", 256, 16, 24, 4, 16), ("e4m3", "bf16", 64, 64, 16, 1, 4), ("i8", "f16", 128, 128, 8, 2, 2),
    ("f16", "bf16", 128, 16, 12, 4, 3), ("i8", "bf16", 128, 8, 8, 2, 1), ("e4m3", "f16", 256, 8, 16, 2, 2),
])
def test_dim_major_v_cuda_core_kernel(kv_dtype, q_dtype, D, bs, Hq, Hkv, Lq):
    """The pipelined CUDA-core kernel on a transposed V cache (AUTO's choice for 8 rows or fewer
    where the FP8 tensor-core kernel does not apply, pinned here for more): every cache type and
    head_dim, pages of 8 to 128 tokens, one row block and several, with a window, sinks, ragged
    lengths and poisoned tails and pages."""
    wl = W.verify16_int8().replace(ctx=[3000, 700, 65, 9], Hq=Hq, Hkv=Hkv, Lq=Lq, D=D, bs=bs, kv_dtype=kv_dtype,
                                   q_dtype=q_dtype, window=900, sinks=True, extra_pages=4,
                                   kv_std=0.5 if kv_dtype == "e4m3" else 1.0)
    inp = _inputs(wl, 300 + D + bs + Hq)
    ref, _ = oracle_out(inp)
    v_dm = inp.v_cache.transpose(-1, -2).contiguous()
    for S in (1, 3):
        desc = B.desc_for(wl, B.TLLM_KERNEL_SIMT, num_pages=inp.num_pages, v_layout=B.TLLM_V_DIM_MAJOR)
        plan = B.tllm_decode_attn_plan(desc, wl.B, wl.Lq, wl.window, host_ctx_lens=wl.ctx, splits_override=S)
        assert plan.kernel == B.TLLM_KERNEL_SIMT
        ws = poisoned_workspace(plan)
        out = new_out(wl)
        B.tllm_decode_attn_splitkv(inp.q, inp.k_cache, v_dm, inp.block_table, inp.context_lens, wl.Lq,
                                   inp.kv_scales, inp.sinks, wl.window, S, ws, out)
        torch.cuda.synchronize()
        assert not (B.tllm_decode_attn_read_status(ws) & B.TLLM_FLAG_TIMEOUT)
        assert_close(out, ref, wl.kv_dtype, f"dim-major V simt {kv_dtype} D{D} bs{bs} S{S}")


@pytest.mark.parametrize("kv_dtype,q_dtype,D,bs,Hq,Hkv,Lq", [
    ("i8", "bf16", 256, 16, 24, 4, 16), ("e4m3", "bf16", 64, 64, 16, 1, 4), ("i8", "f16", 128, 128, 8, 2, 4),
    ("f16", "f16", 64, 8, 14, 2, 2), ("bf16", "bf16", 128, 16, 32, 8, 4), ("bf16", "bf16", 64, 32, 32, 2, 2),
    ("f16", "f16", 128, 128, 12, 4, 3), ("e4m3", "f16", 128, 32, 16, 2, 8), ("i8", "bf16", 64, 16, 16, 1, 8),
    ("e4m3", "bf16", 256, 16, 8, 1, 1), ("i8", "bf16", 256, 8, 24, 4, 16), ("e4m3", "bf16", 128, 8, 16, 2, 4),
    ("i8", "f16", 64, 8, 8, 1, 2),
])
def test_dim_major_v_widening_kernel(kv_dtype, q_dtype, D, bs, Hq, Hkv, Lq):
    """The widening tensor-core kernel on a transposed V cache (AUTO's choice past 8 rows where
    the FP8 kernel does not apply): each page's [D, bs] block is staged as it lies and widened
    into the K-major f16 operand of the PV product. Every cache type, head_dim 64 to 256, pages
    of 8 to 128 tokens (8-bit 8-token pages copied whole, two dims per 16-byte chunk), 8 to 128
    rows, with a window, sinks, ragged lengths and poisoned tails
    and pages (whose NaN codes must not reach the product)."""
    wl = W.verify16_int8().replace(ctx=[3000, 700, 65, 9], Hq=Hq, Hkv=Hkv, Lq=Lq, D=D, bs=bs, kv_dtype=kv_dtype,
                                   q_dtype=q_dtype, window=900, sinks=True, extra_pages=4,
                                   kv_std=0.5 if kv_dtype == "e4m3" else 1.0)
    inp = _inputs(wl, 400 + D + bs + Hq)
    ref, _ = oracle_out(inp)
    v_dm = inp.v_cache.transpose(-1, -2).contiguous()
    for S in (1, 3):
        desc = B.desc_for(wl, B.TLLM_KERNEL_TC_I8, num_pages=inp.num_pages, v_layout=B.TLLM_V_DIM_MAJOR)
        plan = B.tllm_decode_attn_plan(desc, wl.B, wl.Lq, wl.window, host_ctx_lens=wl.ctx, splits_override=S)
        assert plan.kernel == B.TLLM_KERNEL_TC_I8
        ws = poisoned_workspace(plan)
        out = new_out(wl)
        B.tllm_decode_attn_splitkv(inp.q, inp.k_cache, v_dm, inp.block_table, inp.context_lens, wl.Lq,
                                   inp.kv_scales, inp.sinks, wl.window, S, ws, out)
        torch.cuda.synchronize()
        assert not (B.tllm_decode_attn_read_status(ws) & B.TLLM_FLAG_TIMEOUT)
        assert_close(out, ref, wl.kv_dtype, f"dim-major V widening {kv_dtype} D{D} bs{bs} S{S}")


# --- 16-bit split records -------------------------------------------------------------

@pytest.mark.parametrize("rec", [B.TLLM_RECORD_BF16, B.TLLM_RECORD_F16])
@pytest.mark.parametrize("wl,seed", [
    (W.mtp4_fp8_long(batch=6, ctx=1).replace(ctx=[20000, 12345, 777, 4, 3, 40001], extra_pages=10), 1003),
    (W.verify16_int8().replace(extra_pages=16), 1002),
    (W.ragged_fp8(bs=128).replace(extra_pages=4), 1004),
    (W.window_sink_bf16(batch=5).replace(ctx=[9000, 4097, 300, 2, 1]), 1005),
    (W.single_decode().replace(extra_pages=8), 1001),
])
def test_sixteen_bit_records(wl, seed, rec):
    """The whole call with bf16 or f16 split records (aiter PR #5628, Changes: a 16-bit partial
    output per row): the records' one extra rounding stays inside the parity tolerance, at the
    planner's split count and at a forced larger one."""
    inp = _inputs(wl, seed)
    ref, _ = oracle_out(inp)
    for S in (0, 5):
        desc = B.desc_for(wl, num_pages=inp.num_pages, record_type=rec)
        plan = B.tllm_decode_attn_plan(desc, wl.B, wl.Lq, wl.window, host_ctx_lens=wl.ctx, splits_override=S)
        out, _, _ = run_gpu(inp, plan=plan)
        assert_close(out, ref, wl.kv_dtype, f"{wl.name} records {rec} S={plan.num_splits}")


# --- fused combine (the last CTA of a request merges) -------------------------------------

def test_fused_combine_single_decode():
    """The single decode at S = 4 and 8 with the fused combine asked for: the CTA that writes a
    request's last split record merges them (tiny-llm PR #11, open question 1), no combine launch. The
    partial entry point alone then gives the final output, the counters are back at zero after
    every call, repeated calls are bit-identical, and the result matches the oracle."""
    wl = W.single_decode().replace(extra_pages=8)
    inp = _inputs(wl, 1001)
    ref, _ = oracle_out(inp)
    for S in (4, 8):
        desc = B.desc_for(wl, num_pages=inp.num_pages, combine_mode=B.TLLM_COMBINE_FUSED)
        plan = B.tllm_decode_attn_plan(desc, wl.B, wl.Lq, wl.window, host_ctx_lens=wl.ctx, splits_override=S)
        assert plan.kernel == B.TLLM_KERNEL_SIMT and plan.fused_combine == 1
        ws = poisoned_workspace(plan)
        outs = []
        for rep in range(3):
            out = new_out(wl)
            B.tllm_decode_attn_partial(inp.q, inp.k_cache, inp.v_cache, inp.block_table, inp.context_lens, wl.Lq,
                                       inp.kv_scales, inp.sinks, wl.window, S, ws, out)
            torch.cuda.synchronize()
            _, lo, _ = B.tllm_decode_attn_workspace_layout(plan)
            assert int(ws.buffer[256:lo].view(torch.int32).abs().sum()) == 0, "counters not back at zero"
            assert_close(out, ref, wl.kv_dtype, f"fused S{S} rep{rep}")
            outs.append(out)
        assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])


def test_fused_combine_with_window_sinks_and_empty_rows():
    wl = W.window_sink_bf16(batch=6).replace(ctx=[9000, 4097, 300, 2, 1, 0], Hq=8, Hkv=2, window=333,
                                             extra_pages=2)
    inp = _inputs(wl, 211)
    ref, _ = oracle_out(inp)
    desc = B.desc_for(wl, B.TLLM_KERNEL_SIMT, num_pages=inp.num_pages, combine_mode=B.TLLM_COMBINE_FUSED)
    plan = B.tllm_decode_attn_plan(desc, wl.B, wl.Lq, wl.window, host_ctx_lens=wl.ctx, splits_override=5)
    assert plan.fused_combine == 1
    out, _, _ = run_gpu(inp, plan=plan)
    assert_close(out, ref, wl.kv_dtype, "fused window + sinks")
    assert out[5].float().abs().max() == 0



# --- the widening kernel on FP8 e4m3 caches and head_dim 64 ------------------------------

@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("Hq,Hkv,Lq", [(24, 4, 16), (8, 1, 16), (16, 1, 8)])
def test_widening_kernel_fp8_cache(Hq, Hkv, Lq, D):
    """FP8 e4m3 caches widened to f16 (exact) by the same kernel that widens int8, at every
    head_dim: the shapes the FP8 tensor-core kernel does not take (head_dim 64 / 256, or more
    than 64 packed rows), with a window, sinks and ragged lengths."""
    wl = W.mtp4_fp8_long(batch=3, ctx=1).replace(ctx=[3000, 700, 17], Hq=Hq, Hkv=Hkv, Lq=Lq, D=D, window=900,
                                                 sinks=True, extra_pages=4)
    inp = _inputs(wl, 220 + D + Hq)
    ref, _ = oracle_out(inp)
    for S in (1, 3):
        out, plan, _ = run_gpu(inp, TCI8, splits=S)
        assert plan.kernel == TCI8
        assert_close(out, ref, wl.kv_dtype, f"widening e4m3 Hq{Hq} Hkv{Hkv} Lq{Lq} D{D} S{S}")


@pytest.mark.parametrize("Hq,Hkv,Lq", [(24, 4, 16), (4, 4, 4), (32, 1, 4)])
def test_widening_kernel_int8_head_dim_64(Hq, Hkv, Lq):
    wl = W.verify16_int8().replace(ctx=[3000, 700, 65, 17], Hq=Hq, Hkv=Hkv, Lq=Lq, D=64, extra_pages=4)
    inp = _inputs(wl, 230 + Hq)
    ref, _ = oracle_out(inp)
    for S in (1, 3):
        out, plan, _ = run_gpu(inp, TCI8, splits=S)
        assert plan.kernel == TCI8
        assert_close(out, ref, wl.kv_dtype, f"widening int8 D64 Hq{Hq} Hkv{Hkv} Lq{Lq} S{S}")


# --- the widening kernel on 16-bit caches ----------------------------------------------

@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("q_dtype,kv_dtype", [("bf16", "bf16"), ("f16", "f16"), ("bf16", "f16"), ("f16", "bf16")])
@pytest.mark.parametrize("Hq,Hkv,Lq", [(24, 4, 16), (8, 1, 16), (32, 4, 2)])
def test_widening_kernel_16bit_cache(Hq, Hkv, Lq, q_dtype, kv_dtype, D):
    """f16 caches copied and bf16 caches scaled into f16 by a power of two per tile: the shapes
    the 16-bit tensor-core kernel does not take (more than 16 packed rows, head_dim 64 or 256,
    query and cache of different types), with a window, sinks, ragged lengths and poisoned
    tails. Head_dim 256 runs the instance with one-deep staging rings (and one f16 K buffer
    for bf16)."""
    wl = W.window_sink_bf16(batch=4).replace(ctx=[3000, 700, 65, 17], Hq=Hq, Hkv=Hkv, Lq=Lq, D=D, q_dtype=q_dtype,
                                             kv_dtype=kv_dtype, window=900, bs=16, extra_pages=4)
    inp = _inputs(wl, 240 + D + Hq + len(q_dtype + kv_dtype))
    ref, _ = oracle_out(inp)
    for S in (1, 3):
        out, plan, _ = run_gpu(inp, TCI8, splits=S)
        assert plan.kernel == TCI8
        assert_close(out, ref, wl.kv_dtype, f"widening {kv_dtype} q {q_dtype} Hq{Hq} Hkv{Hkv} Lq{Lq} D{D} S{S}")


@pytest.mark.parametrize("bs", [8, 64, 128])
def test_widening_kernel_16bit_block_sizes(bs):
    wl = W.window_sink_bf16(batch=3).replace(ctx=[2500, 333, 129], Hq=32, Hkv=4, Lq=4, bs=bs, window=0, sinks=False,
                                             extra_pages=3)
    inp = _inputs(wl, 250 + bs)
    ref, _ = oracle_out(inp)
    for S in (1, 4):
        out, plan, _ = run_gpu(inp, TCI8, splits=S)
        assert plan.kernel == TCI8
        assert_close(out, ref, wl.kv_dtype, f"widening bf16 bs{bs} S{S}")


@pytest.mark.parametrize("kv_dtype", ["bf16", "f16"])
@pytest.mark.parametrize("bs", [8, 64, 128])
def test_widening_kernel_16bit_head_dim_256_block_sizes(bs, kv_dtype):
    """Head_dim 256 with a 16-bit cache over many tiles per split (the one-deep rings' phases
    cycle many times), pages of 8 to 128 tokens, a window and sinks."""
    wl = W.window_sink_bf16(batch=3).replace(ctx=[6000, 333, 129], Hq=16, Hkv=1, Lq=2, D=256, bs=bs,
                                             kv_dtype=kv_dtype, window=2500, extra_pages=3)
    inp = _inputs(wl, 260 + bs + len(kv_dtype))
    ref, _ = oracle_out(inp)
    for S in (1, 5):
        out, plan, _ = run_gpu(inp, B.TLLM_KERNEL_AUTO, splits=S)
        assert plan.kernel == TCI8
        assert_close(out, ref, wl.kv_dtype, f"widening {kv_dtype} D256 bs{bs} S{S}")


def test_widening_kernel_bf16_tile_magnitudes():
    """The per-tile power of two of a bf16 cache: pages whose K and V values sit anywhere from
    2^-60 to 2^60 (tiles of very different size in one split), and pages holding elements 2^-30 of
    their largest, all match the oracle (the conditioned bound: outputs that are small
    differences of large terms)."""
    wl = W.window_sink_bf16(batch=2).replace(ctx=[3000, 900], Hq=32, Hkv=4, Lq=4, window=0, sinks=False,
                                             extra_pages=2)
    inp = _inputs(wl, 260, poison=False)
    exps_v = [-60, -20, -3, 0, 5, 17, 60]
    exps_k = [-12, -4, 0, 2, 3]
    for b in range(wl.B):
        n = (wl.ctx[b] + wl.bs - 1) // wl.bs
        pages = inp.block_table[b, :n].long()
        for i, pg in enumerate(pages.tolist()):
            inp.v_cache[pg] *= 2.0 ** exps_v[(i + b) % len(exps_v)]
            inp.k_cache[pg] *= 2.0 ** exps_k[(3 * i + b) % len(exps_k)]
    inp.v_cache[..., ::5] *= 2.0 ** -30
    ref, _ = oracle_out(inp)
    cond, _ = oracle_out(abs_value_inputs(inp))
    for S in (1, 3):
        out, plan, _ = run_gpu(inp, TCI8, splits=S)
        assert plan.kernel == TCI8
        assert_close_conditioned(out, ref, cond, wl.kv_dtype, f"widening bf16 magnitudes S{S}")


@pytest.mark.parametrize("kv_dtype,D,Lq", [("bf16", 128, 4), ("f16", 64, 16), ("bf16", 64, 2)])
def test_auto_takes_the_widening_kernel_for_16bit_caches(kv_dtype, D, Lq):
    """AUTO sends 16-bit caches the 16-bit tensor-core kernel does not take to the widening
    kernel (not the generic one), and the result matches the oracle."""
    wl = W.window_sink_bf16(batch=3).replace(ctx=[2000, 300, 40], Hq=32, Hkv=4, Lq=Lq, D=D, q_dtype="bf16",
                                             kv_dtype=kv_dtype, extra_pages=2)
    inp = _inputs(wl, 270 + D + Lq)
    ref, _ = oracle_out(inp)
    out, plan, _ = run_gpu(inp, B.TLLM_KERNEL_AUTO)
    assert plan.kernel == TCI8
    assert_close(out, ref, wl.kv_dtype, f"auto {kv_dtype} D{D} Lq{Lq}")


# --- the CUDA-core kernel in row blocks (more than 8 packed rows) -------------------------------

@pytest.mark.parametrize("q_dtype,kv_dtype", [("bf16", "bf16"), ("f16", "f16"), ("bf16", "f16")])
@pytest.mark.parametrize("Hq,Hkv,Lq", [(32, 4, 2), (16, 1, 4), (12, 4, 3)])
def test_simt_row_blocks_head_dim_256_16bit(Hq, Hkv, Lq, q_dtype, kv_dtype):
    """16-bit caches at head_dim 256 with 9..64 packed rows on the CUDA-core kernel (pinned; AUTO
    takes the widening kernel there), in blocks of 8 rows, the last one ragged, with a window,
    sinks, ragged lengths and poisoned tails."""
    wl = W.window_sink_bf16(batch=4).replace(ctx=[2600, 700, 65, 17], Hq=Hq, Hkv=Hkv, Lq=Lq, D=256, q_dtype=q_dtype,
                                             kv_dtype=kv_dtype, window=900, bs=16, extra_pages=4)
    inp = _inputs(wl, 280 + Hq + Lq + len(q_dtype + kv_dtype))
    ref, _ = oracle_out(inp)
    for S in (1, 3):
        out, plan, _ = run_gpu(inp, B.TLLM_KERNEL_SIMT, splits=S)
        assert plan.kernel == B.TLLM_KERNEL_SIMT
        assert_close(out, ref, wl.kv_dtype, f"simt rows {Hq // Hkv * Lq} {kv_dtype} q {q_dtype} S{S}")


@pytest.mark.parametrize("kv_dtype,D,Hq,Hkv,Lq", [("f16", 128, 24, 1, 1), ("i8", 64, 12, 2, 2), ("e4m3", 128, 20, 1, 2)])
def test_simt_row_blocks_pinned(kv_dtype, D, Hq, Hkv, Lq):
    """The CUDA-core kernel pinned on shapes with more than 8 rows (3 to 5 row blocks) for the
    other cache types and head_dims."""
    wl = W.verify16_int8().replace(ctx=[1900, 300, 40], Hq=Hq, Hkv=Hkv, Lq=Lq, D=D, kv_dtype=kv_dtype, q_dtype="bf16",
                                   extra_pages=2)
    inp = _inputs(wl, 290 + D + Hq)
    ref, _ = oracle_out(inp)
    for S in (1, 4):
        out, plan, _ = run_gpu(inp, B.TLLM_KERNEL_SIMT, splits=S)
        assert plan.kernel == B.TLLM_KERNEL_SIMT
        assert_close(out, ref, wl.kv_dtype, f"simt pinned {kv_dtype} D{D} rows {Hq // Hkv * Lq} S{S}")


# --- failure detection: a bounded wait that runs out ------------------------------------

def test_pipeline_wait_timeout_is_reported_and_the_context_recovers():
    """Failure detection without a GPU fault: with the test stall the widening kernel's QK^T
    issuer issues nothing, so the waits on S run out after their 2 s bound. The kernel sets
    TLLM_FLAG_TIMEOUT, skips its output stores (one split: the output keeps its NaN fill) and
    frees its tensor memory; the next calls on the same context run normally and match the
    oracle."""
    import time
    wl = W.verify16_int8().replace(ctx=[700, 300], extra_pages=2)
    inp = _inputs(wl, 310)
    ref, _ = oracle_out(inp)
    for S in (1, 2):
        desc = B.desc_for(wl, TCI8, num_pages=inp.num_pages)
        desc.test_stall = 1
        plan = B.tllm_decode_attn_plan(desc, wl.B, wl.Lq, wl.window, host_ctx_lens=wl.ctx, splits_override=S)
        ws = B.Workspace(plan)
        out = new_out(wl).fill_(float("nan"))
        t = time.time()
        B.run(inp, ws, out)
        torch.cuda.synchronize()
        assert time.time() - t < 60
        assert B.tllm_decode_attn_read_status(ws, reset=True) & B.TLLM_FLAG_TIMEOUT
        if S == 1:
            assert torch.isnan(out.float()).all(), "a timed-out call stored output"
        good, _, ws2 = run_gpu(inp, TCI8, splits=S)
        assert not (B.tllm_decode_attn_read_status(ws2) & B.TLLM_FLAG_TIMEOUT)
        assert_close(good, ref, wl.kv_dtype, f"after a timed-out call S{S}")

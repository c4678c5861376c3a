"""The C-ABI library on the host (no GPU): symbols, planner, split rule, argument checks.

Nothing here launches a kernel: every call either is host-only (plan, layout, split
range, status strings) or fails its argument checks before any launch.
"""
import ctypes
import glob
import math
import os
import re

import pytest

from split_kv_paged_gb300 import binding as B
from split_kv_paged_gb300 import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from split_kv_paged_gb300 import build
    build.build()
    return B.lib()


def declared_functions():
    names = []
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(tllm_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert "tllm_decode_attn_plan" in names and "tllm_decode_attn_splitkv" in names
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(lib):
    assert B.tllm_status_string(0) == "ok"
    assert "workspace" in B.tllm_status_string(3)


def _plan(wl, **kw):
    return B.tllm_decode_attn_plan(B.desc_for(wl), wl.B, wl.Lq, wl.window, **kw)


def test_plan_basic_fields(lib):
    wl = W.verify16_int8()
    p = _plan(wl, splits_override=8)
    assert p.num_splits == 8 and p.max_splits == 8
    assert p.rows == 6 * 16
    assert p.min_chunk % p.split_align == 0
    so, lo, oo = B.tllm_decode_attn_workspace_layout(p)
    assert so == 0 and lo >= 4 and oo > lo and p.workspace_bytes >= oo


def test_record_bytes_match_printed_verify_scratch(lib):
    """hipfire PR #760, Memory: about 3 MiB of split records at S8 / 16 rows / H24 / D256.
    The O records of that plan are exactly 8 x 16 x 24 x 256 x 4 bytes."""
    p = _plan(W.verify16_int8(), splits_override=8)
    so, lo, oo = B.tllm_decode_attn_workspace_layout(p)
    o_bytes = p.batch * p.desc.num_kv_heads * p.max_splits * p.rows * p.desc.head_dim * 4
    assert o_bytes == 3 * 2 ** 20
    assert p.workspace_bytes - oo >= o_bytes


@pytest.mark.parametrize("wl", [W.single_decode(), W.verify16_int8(), W.mtp4_fp8_long(), W.ragged_fp8(bs=128),
                                W.ragged_fp8(bs=16), W.window_sink_bf16()])
def test_auto_plan_is_sane(lib, wl):
    p = _plan(wl, host_ctx_lens=wl.ctx)
    assert 1 <= p.num_splits <= 256
    longest = max(wl.ctx)
    # a split is never shorter than min_chunk, so S never exceeds what the longest request can use
    assert p.num_splits <= max(1, math.ceil(longest / p.min_chunk))


def test_long_batch_fills_the_gpu(lib):
    """Batch 200 x 200k with one KV head: the plan must give more than one split per
    request (200 CTAs would leave most of 152 SMs idle in the second wave)."""
    wl = W.mtp4_fp8_long()
    p = _plan(wl, host_ctx_lens=wl.ctx)
    assert p.num_splits > 1


@pytest.mark.parametrize("ctx,lq,window,S", [(0, 1, 0, 4), (1, 1, 0, 4), (2048, 1, 0, 4), (20676, 16, 0, 8),
                                             (20676, 16, 0, 3), (200000, 4, 0, 16), (31000, 1, 4096, 3),
                                             (3, 4, 0, 2), (4100, 1, 4096, 5), (129, 4, 128, 7)])
def test_split_ranges_tile_the_visible_union(lib, ctx, lq, window, S):
    wl = W.window_sink_bf16().replace(ctx=[max(ctx, 1)], Lq=lq, window=window)
    p = _plan(wl, splits_override=S)
    lo_vis = max(0, ctx - lq + 1 - window) if window else 0
    ranges = [B.tllm_decode_attn_split_range(p, ctx, lq, window, S, s) for s in range(S)]
    n = ranges[0][2]
    assert 1 <= n <= S
    used = [(a, b) for a, b, _ in ranges[:n]]
    for a, b, _ in ranges[n:]:
        assert a == b                                            # unused splits are empty
    assert used[0][0] <= lo_vis and used[0][0] % p.split_align == 0
    assert used[-1][1] == ctx
    for (a0, b0), (a1, b1) in zip(used, used[1:]):
        assert b0 == a1 and a1 % p.split_align == 0             # contiguous, aligned
    for a, b in used[:-1]:
        assert b - a >= p.min_chunk or ctx == b


def _fake_call(name, plan, ws_bytes=None, **over):
    ws = B.tllm_workspace(ctypes.pointer(plan), 256, plan.workspace_bytes if ws_bytes is None else ws_bytes)
    args = dict(q=256, k=256, v=256, bt=256, ctx=256, lq=plan.query_len, scales=256, sinks=None,
                window=plan.window, S=plan.num_splits, out=256)
    args.update(over)
    f = getattr(B.lib(), name)
    return f(args["q"], args["k"], args["v"], args["bt"], args["ctx"], args["lq"], args["scales"], args["sinks"],
             args["window"], args["S"], ctypes.byref(ws), args["out"], None)


@pytest.mark.parametrize("name", ["tllm_decode_attn_splitkv", "tllm_decode_attn_partial", "tllm_decode_attn_combine"])
@pytest.mark.parametrize("over,status", [
    (dict(q=None), B.TLLM_ERR_INVALID_ARG),
    (dict(k=None), B.TLLM_ERR_INVALID_ARG),
    (dict(ctx=None), B.TLLM_ERR_INVALID_ARG),
    (dict(out=None), B.TLLM_ERR_INVALID_ARG),
    (dict(scales=None), B.TLLM_ERR_INVALID_ARG),        # FP8 KV needs scales
    (dict(S=0), B.TLLM_ERR_INVALID_ARG),
    (dict(S=9), B.TLLM_ERR_INVALID_ARG),                # beyond plan capacity
    (dict(lq=5), B.TLLM_ERR_INVALID_ARG),               # more rows than planned
    (dict(lq=0), B.TLLM_ERR_INVALID_ARG),
    (dict(window=-1), B.TLLM_ERR_INVALID_ARG),
    (dict(ws_bytes=1024), B.TLLM_ERR_WORKSPACE_TOO_SMALL),
])
def test_host_fault_injection(lib, name, over, status):
    wl = W.mtp4_fp8_long(batch=2, ctx=5000)
    plan = _plan(wl, splits_override=8)
    over = dict(over)
    ws_bytes = over.pop("ws_bytes", None)
    assert _fake_call(name, plan, ws_bytes=ws_bytes, **over) == status


def test_misaligned_workspace_is_rejected(lib):
    wl = W.mtp4_fp8_long(batch=2, ctx=5000)
    plan = _plan(wl, splits_override=2)
    ws = B.tllm_workspace(ctypes.pointer(plan), 256 + 16, plan.workspace_bytes)
    st = B.lib().tllm_decode_attn_splitkv(256, 256, 256, 256, 256, 4, 256, None, 0, 2, ctypes.byref(ws), 256, None)
    assert st == B.TLLM_ERR_INVALID_ARG


@pytest.mark.parametrize("field,value,status", [
    ("num_q_heads", 15, B.TLLM_ERR_INVALID_ARG),       # not a multiple of Hkv=2
    ("head_dim", 96, B.TLLM_ERR_UNSUPPORTED),
    ("kv_dtype", B.TLLM_F32, B.TLLM_ERR_UNSUPPORTED),
    ("q_dtype", B.TLLM_INT8, B.TLLM_ERR_UNSUPPORTED),
    ("block_size", 0, B.TLLM_ERR_INVALID_ARG),
    ("block_size", 512, B.TLLM_ERR_UNSUPPORTED),
    ("num_pages", 0, B.TLLM_ERR_INVALID_ARG),
    ("softmax_scale", -1.0, B.TLLM_ERR_INVALID_ARG),
    ("test_stall", 2, B.TLLM_ERR_INVALID_ARG),
])
def test_plan_rejects_bad_desc(lib, field, value, status):
    d = B.desc_for(W.single_decode())
    setattr(d, field, value)
    plan = B.tllm_decode_attn_plan_t()
    st = B.lib().tllm_decode_attn_plan(ctypes.byref(d), 1, 1, 0, None, 0, 0, 0, 0, ctypes.byref(plan))
    assert st == status


def test_plan_rejects_bad_call_shape(lib):
    d = B.desc_for(W.single_decode())
    plan = B.tllm_decode_attn_plan_t()
    for batch, lq, window, so in [(0, 1, 0, 0), (1, 0, 0, 0), (1, 1, -1, 0), (1, 1, 0, -2)]:
        st = B.lib().tllm_decode_attn_plan(ctypes.byref(d), batch, lq, window, None, 0, 0, 0, so, ctypes.byref(plan))
        assert st == B.TLLM_ERR_INVALID_ARG


@pytest.mark.parametrize("wl,kernel", [
    (W.mtp4_fp8_long(), B.TLLM_KERNEL_TC_FP8),
    (W.ragged_fp8(bs=128), B.TLLM_KERNEL_TC_FP8),
    (W.verify16_int8(), B.TLLM_KERNEL_TC_I8),
    (W.window_sink_bf16(), B.TLLM_KERNEL_TC_B16),
    (W.single_decode(), B.TLLM_KERNEL_SIMT),                                             # D 64
    (W.window_sink_bf16().replace(Hq=16, Hkv=1), B.TLLM_KERNEL_TC_B16),                   # 16 rows
    (W.window_sink_bf16().replace(Hq=4, Hkv=1, Lq=4), B.TLLM_KERNEL_TC_B16),              # 16 rows
    (W.window_sink_bf16().replace(Hq=32, Hkv=1), B.TLLM_KERNEL_TC_I8),                    # 32 rows
    (W.window_sink_bf16().replace(Hq=32, Hkv=1, D=256), B.TLLM_KERNEL_TC_I8),             # 32 rows, D 256
    (W.window_sink_bf16().replace(kv_dtype="f16"), B.TLLM_KERNEL_SIMT),                   # bf16 Q, f16 KV
    (W.window_sink_bf16().replace(q_dtype="f16", kv_dtype="f16", out_dtype="f16"), B.TLLM_KERNEL_TC_B16),
    (W.window_sink_bf16().replace(D=256), B.TLLM_KERNEL_SIMT),
])
def test_auto_kernel_choice(lib, wl, kernel):
    """AUTO takes the FP8 tensor-core kernel for e4m3 KV at head_dim 128, the 16-bit one for
    f16/bf16 KV with a query of the same type, head_dim 128 and at most 16 packed rows, the
    widening one for int8 KV, and for other 16-bit shapes with more than 8 rows, then the
    CUDA-core kernels."""
    p = _plan(wl, host_ctx_lens=wl.ctx)
    assert p.kernel == kernel


@pytest.mark.parametrize("change", [dict(D=64), dict(kv_dtype="f16"), dict(Hq=32, Hkv=1), dict(bs=256)])
def test_pinned_tc_b16_rejects_shapes_it_does_not_cover(lib, change):
    wl = W.window_sink_bf16().replace(**change)
    d = B.desc_for(wl, B.TLLM_KERNEL_TC_B16)
    plan = B.tllm_decode_attn_plan_t()
    st = B.lib().tllm_decode_attn_plan(ctypes.byref(d), wl.B, wl.Lq, wl.window, None, 0, 0, 0, 0, ctypes.byref(plan))
    assert st == B.TLLM_ERR_UNSUPPORTED


@pytest.mark.parametrize("wl,field", [
    (W.mtp4_fp8_long(batch=2, ctx=5000), "out"),
    (W.mtp4_fp8_long(batch=2, ctx=5000), "q"),
    (W.verify16_int8(), "out"),
    (W.window_sink_bf16(batch=4, max_ctx=5000), "q"),
    (W.window_sink_bf16(batch=4, max_ctx=5000), "k"),
])
def test_tensor_core_kernels_reject_misaligned_pointers(lib, wl, field):
    """TMA boxes, 16-byte query loads and (FP8, INT8) 16-byte row stores need 16-byte aligned
    buffers: the call returns TLLM_ERR_INVALID_ARG before any launch."""
    plan = _plan(wl, host_ctx_lens=wl.ctx, splits_override=2)
    assert plan.kernel in (B.TLLM_KERNEL_TC_FP8, B.TLLM_KERNEL_TC_I8, B.TLLM_KERNEL_TC_B16)
    over = {field: 256 + 2, "S": plan.num_splits, "lq": wl.Lq, "window": wl.window}
    for name in ("tllm_decode_attn_splitkv", "tllm_decode_attn_partial"):
        assert _fake_call(name, plan, **over) == B.TLLM_ERR_INVALID_ARG


@pytest.mark.parametrize("wl,S", [
    (W.mtp4_fp8_long(), 3),            # 600 items on 152 SMs: four even waves
    (W.ragged_fp8(bs=128), 131),       # 12-tile splits: 131 of the 200k request + 15 short, one wave
    (W.verify16_int8(), 36),
    (W.single_decode(), 32),           # one 64-token tile per split: 64 CTAs, all in one wave
    (W.window_sink_bf16(), 1),         # HBM-bound 16-bit kernel: no split, no combine
])
def test_planner_choices_on_the_measured_workloads(lib, wl, S):
    """The split counts the planner picks for the five measured workloads; each matches the
    fastest count of the bench's split sweeps on a GB300 (the HBM-bound model of the 16-bit
    kernel picks S = 1 for the window workload, measured faster than S = 2 and S = 3)."""
    assert _plan(wl, host_ctx_lens=wl.ctx).num_splits == S


def test_planner_splits_a_small_batch_for_the_16_bit_kernel(lib):
    """Four requests x 8 KV heads leave most SMs idle without splits: the HBM-bound model
    still splits them."""
    wl = W.window_sink_bf16(batch=4)
    p = _plan(wl, host_ctx_lens=wl.ctx)
    assert p.kernel == B.TLLM_KERNEL_TC_B16 and p.num_splits > 1


def test_noalloc_refuses_plans_beyond_its_array(lib):
    """The allocation-free entry point checks the plan against its fixed array before any
    CUDA call."""
    wl = W.mtp4_fp8_long()
    plan = _plan(wl, host_ctx_lens=wl.ctx, splits_override=16)     # 105 MB of split records
    assert plan.workspace_bytes > B.tllm_decode_attn_noalloc_scratch_bytes()
    st = B.lib().tllm_decode_attn_splitkv_noalloc(256, 256, 256, 256, 256, wl.Lq, 256, None, 0, plan.num_splits,
                                                  ctypes.byref(plan), 256, None)
    assert st == B.TLLM_ERR_WORKSPACE_TOO_SMALL


def test_noalloc_array_size_matches_the_header(lib):
    """The size the library reports for its record area is the header's macro."""
    text = open(os.path.join(ROOT, "include", "tllm_decode_attn.h")).read()
    m = re.search(r"#define\s+TLLM_NOALLOC_SCRATCH_BYTES\s+\((\d+)u\s*<<\s*(\d+)\)", text)
    assert m, "macro not found"
    assert B.tllm_decode_attn_noalloc_scratch_bytes() == int(m.group(1)) << int(m.group(2))


def test_noalloc_checks_arguments_before_queueing_anything(lib):
    """A bad argument to the no-alloc entry point returns its status before any work is queued:
    the status word of the record area (zeroed at each call start) is not touched, so the call
    needs no GPU to fail."""
    wl = W.mtp4_fp8_long(batch=2, ctx=3000)
    plan = _plan(wl, host_ctx_lens=wl.ctx, splits_override=2)
    # a null query pointer, then a misaligned one (the FP8 tensor-core kernel needs 16 bytes)
    for q in (None, 258):
        st = B.lib().tllm_decode_attn_splitkv_noalloc(q, 256, 256, 256, 256, wl.Lq, 256, None, 0, 2,
                                                      ctypes.byref(plan), 256, None)
        assert st == B.TLLM_ERR_INVALID_ARG


@pytest.mark.parametrize("bs", [128, 16])
def test_planner_fits_the_ragged_batch_in_one_item_wave(lib, bs):
    """The 200k + 15 x 1k batch: the work-based split size gives the long request as many
    equal splits as leave one work-list item per SM, and each short request one split."""
    wl = W.ragged_fp8(bs=bs)
    plan = _plan(wl, host_ctx_lens=wl.ctx, num_sms=152)
    counts = [B.tllm_decode_attn_split_range(plan, c, wl.Lq, 0, plan.num_splits, 0)[2] for c in wl.ctx]
    assert sum(counts) * wl.Hkv <= 152
    assert counts[1:] == [1] * 15
    assert counts[0] == plan.num_splits > 92
    sizes = [B.tllm_decode_attn_split_range(plan, wl.ctx[0], wl.Lq, 0, plan.num_splits, s) for s in range(counts[0])]
    assert max(t1 - t0 for t0, t1, _ in sizes) == plan.min_chunk


def test_contiguous_cache_needs_every_request_block(lib):
    """Without a block table the cache must hold batch x max_blocks_per_seq pages; a smaller
    one is refused before any launch."""
    wl = W.mtp4_fp8_long(batch=4, ctx=1000)
    desc = B.desc_for(wl, num_pages=4 * wl.max_blocks - 1)
    plan = B.tllm_decode_attn_plan(desc, wl.B, wl.Lq, wl.window, host_ctx_lens=wl.ctx, splits_override=2)
    ws = B.tllm_workspace(ctypes.pointer(plan), 256, plan.workspace_bytes)
    st = B.lib().tllm_decode_attn_splitkv(256, 256, 256, None, 256, wl.Lq, 256, None, 0, 2, ctypes.byref(ws), 256,
                                          None)
    assert st == B.TLLM_ERR_INVALID_ARG


def test_dim_major_v_routes_to_kernels_that_read_it(lib):
    """AUTO with a transposed V cache: the FP8 tensor-core kernel for FP8 KV (head_dim 128, pages
    of 16 or more tokens, at most 64 rows); the widening tensor-core kernel for more than 8 rows
    of the other quantised shapes (8-token pages included) and of 16-bit caches up to head_dim
    128; the pipelined CUDA-core kernel for the rest."""
    def plan(wl):
        return B.tllm_decode_attn_plan(B.desc_for(wl, v_layout=B.TLLM_V_DIM_MAJOR), wl.B, wl.Lq, 0,
                                       host_ctx_lens=wl.ctx)
    assert plan(W.mtp4_fp8_long(batch=2, ctx=4000)).kernel == B.TLLM_KERNEL_TC_FP8
    assert plan(W.mtp4_fp8_long(batch=2, ctx=4000, bs=8)).kernel == B.TLLM_KERNEL_TC_I8
    assert plan(W.window_sink_bf16(batch=2)).kernel == B.TLLM_KERNEL_SIMT
    assert plan(W.window_sink_bf16(batch=2).replace(bs=8, D=256, Hq=32, Hkv=2)).kernel == B.TLLM_KERNEL_SIMT
    assert plan(W.verify16_int8()).kernel == B.TLLM_KERNEL_TC_I8
    assert plan(W.mtp4_fp8_long(batch=2, ctx=4000).replace(D=64)).kernel == B.TLLM_KERNEL_TC_I8
    assert plan(W.window_sink_bf16(batch=2).replace(bs=8, D=128, Hq=32, Hkv=2)).kernel == B.TLLM_KERNEL_TC_I8
    assert plan(W.verify16_int8().replace(Lq=1)).kernel == B.TLLM_KERNEL_SIMT        # 6 rows
    assert plan(W.verify16_int8().replace(bs=8)).kernel == B.TLLM_KERNEL_TC_I8
    assert plan(W.verify16_int8().replace(bs=8, Lq=1)).kernel == B.TLLM_KERNEL_SIMT


def test_sixteen_bit_records_halve_the_record_area(lib):
    """A 16-bit record plan needs half the partial-output bytes of an fp32 one; the LSE area is
    unchanged."""
    wl = W.ragged_fp8(bs=128)
    plans = [B.tllm_decode_attn_plan(B.desc_for(wl, record_type=r), wl.B, wl.Lq, 0, host_ctx_lens=wl.ctx)
             for r in (B.TLLM_RECORD_F32, B.TLLM_RECORD_BF16, B.TLLM_RECORD_F16)]
    f32, bf16, f16 = plans
    assert bf16.num_splits == f32.num_splits and bf16.workspace_bytes == f16.workspace_bytes
    _, lo, oo = B.tllm_decode_attn_workspace_layout(f32)
    o32 = f32.workspace_bytes - oo
    _, lo16, oo16 = B.tllm_decode_attn_workspace_layout(bf16)
    assert (lo16, oo16) == (lo, oo)
    assert abs((bf16.workspace_bytes - oo16) * 2 - o32) <= 512


def test_fused_combine_only_when_asked_and_for_small_records(lib):
    """The fused merge is taken only when the desc asks for it, by the few-row CUDA-core kernel
    when a request's records are small (the single decode); not for one split, not for the
    tensor-core kernels' large records, and never by default."""
    wl = W.single_decode()
    def plan(w, S=0, mode=B.TLLM_COMBINE_FUSED):
        return B.tllm_decode_attn_plan(B.desc_for(w, combine_mode=mode), w.B, w.Lq, w.window, host_ctx_lens=w.ctx,
                                       splits_override=S)
    assert plan(wl, 4).fused_combine == 1
    assert plan(wl, 4, B.TLLM_COMBINE_KERNEL).fused_combine == 0
    assert plan(wl, 1).fused_combine == 0
    for wl2 in (W.verify16_int8(), W.ragged_fp8(bs=128), W.mtp4_fp8_long()):
        assert plan(wl2).fused_combine == 0
        assert _plan(wl2, host_ctx_lens=wl2.ctx).fused_combine == 0


def test_workspace_header_holds_one_counter_per_request_and_kv_head(lib):
    wl = W.window_sink_bf16(batch=64)
    p = _plan(wl, host_ctx_lens=wl.ctx, splits_override=2)
    so, lo, oo = B.tllm_decode_attn_workspace_layout(p)
    assert so == 0 and lo >= 256 + 4 * wl.B * wl.Hkv and lo % 256 == 0



@pytest.mark.parametrize("kv", ["e4m3", "i8"])
@pytest.mark.parametrize("D", [64, 128, 256])
def test_auto_never_falls_back_for_quantised_caches(lib, kv, D):
    """FP8 and INT8 caches with a 16-bit query: for every head_dim and up to 128 packed rows,
    AUTO picks a tensor-core kernel (or the pipelined CUDA-core kernel for at most 8 rows),
    never the generic kernel."""
    for G, Lq in ((1, 1), (7, 1), (4, 4), (8, 4), (16, 4), (24, 4), (6, 16), (8, 16)):
        wl = W.mtp4_fp8_long(batch=2, ctx=1000).replace(Hq=G, Hkv=1, Lq=Lq, D=D, kv_dtype=kv, q_dtype="bf16")
        k = _plan(wl, host_ctx_lens=wl.ctx).kernel
        assert k != B.TLLM_KERNEL_GENERIC, (kv, D, G * Lq)
        if G * Lq > 8:
            assert k in (B.TLLM_KERNEL_TC_FP8, B.TLLM_KERNEL_TC_I8), (kv, D, G * Lq, k)


@pytest.mark.parametrize("v_layout", [B.TLLM_V_TOKEN_MAJOR, B.TLLM_V_DIM_MAJOR])
@pytest.mark.parametrize("kv", ["e4m3", "i8", "f16", "bf16"])
def test_auto_never_falls_back_for_any_page_size_or_v_layout(lib, kv, v_layout):
    """Every cache type, head_dim, page size (8 to 128 tokens) and V layout, with 1 to 128
    packed rows and either 16-bit query: AUTO never picks the generic kernel."""
    for D in (64, 128, 256):
        for bs in (8, 16, 32, 64, 128):
            for q in ("bf16", "f16"):
                for G, Lq in ((1, 1), (7, 1), (8, 1), (4, 4), (16, 4), (6, 16), (8, 16)):
                    wl = W.mtp4_fp8_long(batch=2, ctx=1000).replace(Hq=G, Hkv=1, Lq=Lq, D=D, bs=bs, kv_dtype=kv,
                                                                    q_dtype=q)
                    desc = B.desc_for(wl, v_layout=v_layout)
                    k = B.tllm_decode_attn_plan(desc, wl.B, wl.Lq, 0, host_ctx_lens=wl.ctx).kernel
                    assert k != B.TLLM_KERNEL_GENERIC, (kv, q, D, bs, G * Lq, v_layout)


@pytest.mark.parametrize("kv,q", [("bf16", "bf16"), ("f16", "f16"), ("f16", "bf16"), ("bf16", "f16")])
@pytest.mark.parametrize("D", [64, 128, 256])
def test_auto_never_falls_back_for_16bit_caches(lib, kv, q, D):
    """f16 and bf16 caches at every head_dim, up to 128 packed rows, with the query of either
    16-bit type: AUTO picks a tensor-core kernel for more than 8 rows (the widening kernel,
    head_dim 256 included) and the pipelined CUDA-core kernel for at most 8, never the generic
    kernel; the 16-bit tensor-core kernel keeps the shapes it takes (same query and cache type,
    head_dim 128, at most 16 rows)."""
    for G, Lq in ((1, 1), (7, 1), (4, 4), (8, 2), (8, 4), (24, 4), (6, 16), (8, 16)):
        wl = W.window_sink_bf16(batch=2).replace(Hq=G, Hkv=1, Lq=Lq, D=D, kv_dtype=kv, q_dtype=q)
        k = _plan(wl, host_ctx_lens=wl.ctx).kernel
        rows = G * Lq
        assert k != B.TLLM_KERNEL_GENERIC, (kv, q, D, rows)
        if q == kv and D == 128 and rows <= 16:
            assert k == B.TLLM_KERNEL_TC_B16, (kv, q, D, rows, k)
        elif rows > 8:
            assert k == B.TLLM_KERNEL_TC_I8, (kv, q, D, rows, k)
        else:
            assert k == B.TLLM_KERNEL_SIMT, (kv, q, D, rows, k)


def test_fused_combine_needs_one_row_block(lib):
    """The fused merge counts one arrival per split; with more than 8 rows the CUDA-core kernel
    runs several row blocks per split, so the plan keeps the combine kernel."""
    wl = W.window_sink_bf16(batch=2).replace(ctx=[2000, 900], Hq=32, Hkv=2, Lq=1, D=256)
    d = B.desc_for(wl, B.TLLM_KERNEL_SIMT, combine_mode=B.TLLM_COMBINE_FUSED)
    p = B.tllm_decode_attn_plan(d, wl.B, wl.Lq, wl.window, host_ctx_lens=wl.ctx, splits_override=4)
    assert p.kernel == B.TLLM_KERNEL_SIMT and p.fused_combine == 0
    wl8 = wl.replace(Hq=16)
    p8 = B.tllm_decode_attn_plan(B.desc_for(wl8, B.TLLM_KERNEL_SIMT, combine_mode=B.TLLM_COMBINE_FUSED), wl8.B,
                                 wl8.Lq, wl8.window,
                                 host_ctx_lens=wl8.ctx, splits_override=4)
    assert p8.kernel == B.TLLM_KERNEL_SIMT and p8.fused_combine == 1

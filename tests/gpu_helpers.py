"""Shared helpers of the GPU parity tests: run the CUDA path through the C ABI, run
the oracle on host copies of the same seeded inputs, and compare."""
import numpy as np
import torch

import oracle
from split_kv_paged_gb300 import binding as B
from split_kv_paged_gb300 import workloads as W

NAN_BYTE = 0xFF      # an all-ones fp32 is a NaN


def tol_for(kv_dtype: str) -> float:
    """Tolerance of the computation on this KV precision: 5e-3 for FP8 / INT8 KV, 2e-3
    for 16-bit KV, as max abs/rel error (|gpu - ref| <= tol + tol*|ref|), and also as the
    bound on the relative L2 error of the whole output."""
    return 5e-3 if kv_dtype in W.QUANTISED else 2e-3


# Unit roundoff of the output type: storing the result rounds it to nearest, which by
# itself moves a value by up to this fraction of its magnitude (2^-8 for bf16: 8 bits
# of precision). The bound adds it on top of the computation's tolerance.
OUT_ROUNDOFF = {"f32": 2.0 ** -24, "f16": 2.0 ** -11, "bf16": 2.0 ** -8}


def plan_for(wl, kernel=B.TLLM_KERNEL_AUTO, splits=0, host_ctx=None, num_pages=None, **kw):
    desc = B.desc_for(wl, kernel, num_pages=num_pages)
    return B.tllm_decode_attn_plan(desc, wl.B, wl.Lq, wl.window,
                                   host_ctx_lens=wl.ctx if host_ctx is None else host_ctx,
                                   splits_override=splits, **kw)


def poisoned_workspace(plan) -> B.Workspace:
    """A workspace whose split-record areas hold NaN bytes; its header (status word and the
    fused combine's arrival counters) is zero, as the C ABI asks before a first call."""
    ws = B.Workspace(plan)
    ws.buffer.fill_(NAN_BYTE)
    _, lo, _ = B.tllm_decode_attn_workspace_layout(plan)
    ws.buffer[:lo].zero_()
    return ws


def new_out(wl, fill=float("nan")) -> torch.Tensor:
    return torch.full((wl.B, wl.Lq, wl.Hq, wl.D), fill, dtype=W.DTYPES[wl.out_dtype], device="cuda")


def run_gpu(inp, kernel=B.TLLM_KERNEL_AUTO, splits=0, plan=None, ws=None, out=None, num_splits=None):
    wl = inp.wl
    if plan is None:
        plan = plan_for(wl, kernel, splits, num_pages=inp.num_pages)
    if ws is None:
        ws = poisoned_workspace(plan)
    if out is None:
        out = new_out(wl)
    B.run(inp, ws, out, num_splits=plan.num_splits if num_splits is None else num_splits)
    torch.cuda.synchronize()
    assert not (B.tllm_decode_attn_read_status(ws) & B.TLLM_FLAG_TIMEOUT), "a pipeline wait timed out"
    return out, plan, ws


def oracle_out(inp, window=None, sinks="inp", key_range=None):
    h = inp.to("cpu")
    wl = inp.wl
    return oracle.attention(h.q, h.k_cache, h.v_cache, h.kv_scales, h.block_table, h.context_lens,
                            h.sinks if sinks == "inp" else sinks, q_dtype=wl.q_dtype, kv_dtype=wl.kv_dtype,
                            window=wl.window if window is None else window, scale=wl.scale or None,
                            key_range=key_range)


def out_name(t: torch.Tensor) -> str:
    return {torch.float32: "f32", torch.float16: "f16", torch.bfloat16: "bf16"}[t.dtype]


def assert_close(got: torch.Tensor, ref: np.ndarray, kv_dtype: str, what: str = ""):
    g = got.detach().double().cpu().numpy()
    tol = tol_for(kv_dtype)
    u = OUT_ROUNDOFF[out_name(got)]
    assert g.shape == ref.shape, (g.shape, ref.shape)
    assert np.isfinite(g).all(), f"{what}: non-finite outputs at {np.argwhere(~np.isfinite(g))[:5].tolist()}"
    err = np.abs(g - ref)
    bound = tol + (tol + u) * np.abs(ref)
    bad = err > bound
    if bad.any():
        idx = np.argwhere(bad)[:5].tolist()
        raise AssertionError(f"{what}: {bad.sum()} elements outside tolerance {tol}; worst err "
                             f"{err.max():.3e}; first {idx}; got {g[tuple(idx[0])]:.6f} ref {ref[tuple(idx[0])]:.6f}")
    nref = np.linalg.norm(ref)
    if nref > 0:
        rel = np.linalg.norm(g - ref) / nref
        assert rel <= tol + u, f"{what}: relative L2 error {rel:.3e} > {tol + u}"
    # per-row cosine on rows that see keys; rows that see none must be exactly zero
    gr = g.reshape(-1, g.shape[-1])
    rr = ref.reshape(-1, ref.shape[-1])
    nr = np.linalg.norm(rr, axis=1)
    zero = nr == 0
    assert np.all(gr[zero] == 0), f"{what}: rows with no visible key must be zero"
    live = ~zero
    if live.any():
        cos = (gr[live] * rr[live]).sum(1) / (np.linalg.norm(gr[live], axis=1) * nr[live])
        assert cos.min() >= 0.9999, f"{what}: min row cosine {cos.min():.6f}"


def referenced_pages(inp) -> torch.Tensor:
    wl = inp.wl
    used = torch.zeros(inp.num_pages, dtype=torch.bool, device=inp.block_table.device)
    for b in range(wl.B):
        c = int(inp.context_lens[b])
        n = (c + wl.bs - 1) // wl.bs
        used[inp.block_table[b, :n].long()] = True
    return used


def poison_cache(inp):
    """NaN (or NaN scales for INT8) in every unreferenced page and in the slots past
    each request's last token; none of it may reach the output."""
    wl = inp.wl
    unused = ~referenced_pages(inp)
    def poison(cache, which):
        if wl.kv_dtype == "i8":
            inp.kv_scales[which][unused] = float("nan")
        elif wl.kv_dtype == "e4m3":
            cache.view(torch.uint8)[unused] = 0x7F
        else:
            cache[unused] = float("nan")
    poison(inp.k_cache, 0)
    poison(inp.v_cache, 1)
    for b in range(wl.B):
        c = int(inp.context_lens[b])
        if c % wl.bs == 0 or c == 0:
            continue
        page = int(inp.block_table[b, c // wl.bs])
        for which, cache in ((0, inp.k_cache), (1, inp.v_cache)):
            if wl.kv_dtype == "i8":
                inp.kv_scales[which][page, :, c % wl.bs:] = float("nan")
            elif wl.kv_dtype == "e4m3":
                cache.view(torch.uint8)[page, :, c % wl.bs:] = 0x7F
            else:
                cache[page, :, c % wl.bs:] = float("nan")


def abs_value_inputs(inp):
    """The same attention problem with every V element and V scale replaced by its
    absolute value: the oracle on it gives sum_t w_t |v_t|, the scale of the terms whose
    sum is the output (the condition of the weighted sum)."""
    a = inp.to("cpu")
    wl = inp.wl
    v = a.v_cache.clone()
    if wl.kv_dtype == "e4m3":
        v.view(torch.uint8).bitwise_and_(0x7F)
    else:
        v = v.abs()
    a.v_cache = v
    if a.kv_scales is not None:
        sc = a.kv_scales.clone()
        sc[1] = sc[1].abs()
        a.kv_scales = sc
    return a


def assert_close_conditioned(got: torch.Tensor, ref: np.ndarray, cond: np.ndarray, kv_dtype: str, what: str = ""):
    """The tolerance for outputs that are small differences of large terms.

    cond = sum_t w_t |v_t| (the oracle on |V|) is the magnitude of the terms whose weighted
    sum is the output. Elements without cancellation (cond <= 4 |ref|) must meet the plain
    bound of assert_close, |gpu - ref| <= tol + (tol + u) |ref|. Every element must meet
    |gpu - ref| <= tol * cond + u * |ref|: the forward error bound of a weighted sum
    computed with relative precision tol per term, plus the output's own rounding. Returns
    the worst ratio of error to the plain bound on the cancelling elements, for the report."""
    g = got.detach().double().cpu().numpy()
    tol = tol_for(kv_dtype)
    u = OUT_ROUNDOFF[out_name(got)]
    assert np.isfinite(g).all(), f"{what}: non-finite outputs"
    err = np.abs(g - ref)
    plain = tol + (tol + u) * np.abs(ref)
    calm = cond <= 4.0 * np.abs(ref)
    bad_plain = calm & (err > plain)
    assert not bad_plain.any(), (f"{what}: {bad_plain.sum()} of {calm.sum()} non-cancelling elements outside the "
                                 f"plain bound; worst ratio {(err / plain)[calm].max():.3f}")
    bound = tol * cond + u * np.abs(ref) + 1e-30
    bad = err > bound
    assert not bad.any(), f"{what}: {bad.sum()} elements outside the conditioned bound; worst ratio {(err / bound).max():.3f}"
    worst = float((err / plain)[~calm].max()) if (~calm).any() else 0.0
    print(f"{what}: {calm.sum()} non-cancelling elements within the plain bound (worst "
          f"{(err / plain)[calm].max() if calm.any() else 0.0:.3f}); on the {(~calm).sum()} cancelling elements "
          f"the worst error / plain bound is {worst:.3f}, conditioned bound worst {(err / bound).max():.3f}")
    return worst

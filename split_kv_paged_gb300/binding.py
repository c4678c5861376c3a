"""Thin ctypes binding over ``libtllm_decode_attn.so`` (argument marshalling only).

Every entry point has the name of the C function it wraps. Tensors are passed as raw
device pointers; torch is used only to own device memory and streams. Loading fails
loudly if the CUDA library has not been built: there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libtllm_decode_attn.so")

# tllm_status
TLLM_OK, TLLM_ERR_INVALID_ARG, TLLM_ERR_UNSUPPORTED, TLLM_ERR_WORKSPACE_TOO_SMALL, TLLM_ERR_CUDA = range(5)
# tllm_dtype
TLLM_F16, TLLM_BF16, TLLM_F32, TLLM_FP8_E4M3, TLLM_INT8 = range(5)
# tllm_kernel
TLLM_KERNEL_AUTO, TLLM_KERNEL_GENERIC, TLLM_KERNEL_SIMT, TLLM_KERNEL_TC_FP8, TLLM_KERNEL_TC_I8, TLLM_KERNEL_TC_B16 = range(6)
# tllm_v_layout
TLLM_V_TOKEN_MAJOR, TLLM_V_DIM_MAJOR = range(2)
# tllm_record_type
TLLM_RECORD_F32, TLLM_RECORD_BF16, TLLM_RECORD_F16 = range(3)
# tllm_combine_mode
TLLM_COMBINE_KERNEL, TLLM_COMBINE_FUSED = range(2)
TLLM_FLAG_CTX_CLAMPED = 0x1
TLLM_FLAG_BAD_PAGE = 0x2
TLLM_FLAG_TIMEOUT = 0x4

DTYPE_OF_NAME = {"f16": TLLM_F16, "bf16": TLLM_BF16, "f32": TLLM_F32, "e4m3": TLLM_FP8_E4M3, "i8": TLLM_INT8}
DTYPE_OF_TORCH = {torch.float16: TLLM_F16, torch.bfloat16: TLLM_BF16, torch.float32: TLLM_F32,
                  torch.float8_e4m3fn: TLLM_FP8_E4M3, torch.int8: TLLM_INT8}


class TllmError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {tllm_status_string(status)} ({status})")


class tllm_decode_attn_desc(ctypes.Structure):
    _fields_ = [("num_q_heads", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("block_size", ctypes.c_int32),
                ("max_blocks_per_seq", ctypes.c_int32), ("num_pages", ctypes.c_int32),
                ("q_dtype", ctypes.c_int), ("kv_dtype", ctypes.c_int), ("out_dtype", ctypes.c_int),
                ("softmax_scale", ctypes.c_float), ("kernel", ctypes.c_int), ("v_layout", ctypes.c_int),
                ("record_type", ctypes.c_int), ("combine_mode", ctypes.c_int), ("test_stall", ctypes.c_int32)]


class tllm_decode_attn_plan_t(ctypes.Structure):
    _fields_ = [("desc", tllm_decode_attn_desc), ("batch", ctypes.c_int32), ("query_len", ctypes.c_int32),
                ("window", ctypes.c_int32), ("num_splits", ctypes.c_int32), ("max_splits", ctypes.c_int32),
                ("min_chunk", ctypes.c_int32), ("split_align", ctypes.c_int32), ("kernel", ctypes.c_int32),
                ("rows", ctypes.c_int32), ("fused_combine", ctypes.c_int32), ("reserved", ctypes.c_int32 * 6),
                ("workspace_bytes", ctypes.c_size_t)]


class tllm_workspace(ctypes.Structure):
    _fields_ = [("plan", ctypes.POINTER(tllm_decode_attn_plan_t)), ("ptr", ctypes.c_void_p),
                ("bytes", ctypes.c_size_t)]


_lock = threading.Lock()
_lib = None

_CALL_ARGS = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32,
              ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32, ctypes.POINTER(tllm_workspace),
              ctypes.c_void_p, ctypes.c_void_p]


def lib() -> ctypes.CDLL:
    """The loaded C library. Raises if it was not built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"{LIB_PATH} is missing: build it with split_kv_paged_gb300.build.build()")
            L = ctypes.CDLL(LIB_PATH)
            L.tllm_status_string.restype = ctypes.c_char_p
            L.tllm_status_string.argtypes = [ctypes.c_int]
            L.tllm_decode_attn_plan.restype = ctypes.c_int
            L.tllm_decode_attn_plan.argtypes = [ctypes.POINTER(tllm_decode_attn_desc), ctypes.c_int32, ctypes.c_int32,
                                                ctypes.c_int32, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64,
                                                ctypes.c_int32, ctypes.c_int32, ctypes.POINTER(tllm_decode_attn_plan_t)]
            for name in ("tllm_decode_attn_splitkv", "tllm_decode_attn_partial", "tllm_decode_attn_combine"):
                f = getattr(L, name)
                f.restype = ctypes.c_int
                f.argtypes = _CALL_ARGS
            L.tllm_decode_attn_workspace_layout.restype = ctypes.c_int
            L.tllm_decode_attn_workspace_layout.argtypes = [ctypes.POINTER(tllm_decode_attn_plan_t)] + \
                [ctypes.POINTER(ctypes.c_size_t)] * 3
            L.tllm_decode_attn_split_range.restype = ctypes.c_int
            L.tllm_decode_attn_split_range.argtypes = [ctypes.POINTER(tllm_decode_attn_plan_t)] + \
                [ctypes.c_int32] * 5 + [ctypes.POINTER(ctypes.c_int32)] * 3
            L.tllm_decode_attn_splitkv_noalloc.restype = ctypes.c_int
            L.tllm_decode_attn_splitkv_noalloc.argtypes = _CALL_ARGS[:10] + [
                ctypes.POINTER(tllm_decode_attn_plan_t), ctypes.c_void_p, ctypes.c_void_p]
            L.tllm_decode_attn_noalloc_read_status.restype = ctypes.c_int
            L.tllm_decode_attn_noalloc_read_status.argtypes = [ctypes.POINTER(ctypes.c_uint32), ctypes.c_int32,
                                                               ctypes.c_void_p]
            L.tllm_decode_attn_noalloc_scratch_bytes.restype = ctypes.c_size_t
            L.tllm_decode_attn_noalloc_scratch_bytes.argtypes = []
            L.tllm_decode_attn_read_status.restype = ctypes.c_int
            L.tllm_decode_attn_read_status.argtypes = [ctypes.POINTER(tllm_workspace), ctypes.POINTER(ctypes.c_uint32),
                                                       ctypes.c_int32, ctypes.c_void_p]
            _lib = L
    return _lib


def tllm_status_string(status: int) -> str:
    return lib().tllm_status_string(int(status)).decode()


def _check(status: int, where: str) -> None:
    if status != TLLM_OK:
        raise TllmError(status, where)


def make_desc(num_q_heads, num_kv_heads, head_dim, block_size, max_blocks_per_seq, num_pages, q_dtype, kv_dtype,
              out_dtype, softmax_scale=0.0, kernel=TLLM_KERNEL_AUTO,
              v_layout=TLLM_V_TOKEN_MAJOR, record_type=TLLM_RECORD_F32,
              combine_mode=TLLM_COMBINE_KERNEL) -> tllm_decode_attn_desc:
    def code(x):
        if isinstance(x, str):
            return DTYPE_OF_NAME[x]
        if isinstance(x, torch.dtype):
            return DTYPE_OF_TORCH[x]
        return int(x)
    return tllm_decode_attn_desc(int(num_q_heads), int(num_kv_heads), int(head_dim), int(block_size),
                                 int(max_blocks_per_seq), int(num_pages), code(q_dtype), code(kv_dtype),
                                 code(out_dtype), float(softmax_scale), int(kernel), int(v_layout),
                                 int(record_type), int(combine_mode))


def tllm_decode_attn_plan(desc: tllm_decode_attn_desc, batch: int, query_len: int, window: int = 0,
                          host_ctx_lens=None, max_ctx_hint: int = 0, total_ctx_hint: int = 0, num_sms: int = 0,
                          splits_override: int = 0) -> tllm_decode_attn_plan_t:
    plan = tllm_decode_attn_plan_t()
    arr = None
    if host_ctx_lens is not None:
        vals = [int(x) for x in (host_ctx_lens.tolist() if hasattr(host_ctx_lens, "tolist") else host_ctx_lens)]
        arr = (ctypes.c_int32 * len(vals))(*vals)
    st = lib().tllm_decode_attn_plan(ctypes.byref(desc), int(batch), int(query_len), int(window),
                                     ctypes.cast(arr, ctypes.c_void_p) if arr is not None else None,
                                     int(max_ctx_hint), int(total_ctx_hint), int(num_sms), int(splits_override),
                                     ctypes.byref(plan))
    _check(st, "tllm_decode_attn_plan")
    return plan


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else t.data_ptr()


class Workspace:
    """A plan plus a caller-owned device buffer of plan.workspace_bytes (torch-allocated)."""

    def __init__(self, plan: tllm_decode_attn_plan_t, device="cuda", buffer: Optional[torch.Tensor] = None):
        self.plan = plan
        if buffer is None:
            buffer = torch.zeros(int(plan.workspace_bytes), dtype=torch.uint8, device=device)
        self.buffer = buffer
        self.c = tllm_workspace(ctypes.pointer(self.plan), buffer.data_ptr(), buffer.numel())

    def layout(self):
        return tllm_decode_attn_workspace_layout(self.plan)


def _stream_handle(stream) -> Optional[int]:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _call(name, q, k_cache, v_cache, block_table, context_lens, query_len, kv_scales, sinks, window, num_splits,
          workspace: Workspace, out, stream=None):
    f = getattr(lib(), name)
    st = f(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), _ptr(context_lens), int(query_len),
           _ptr(kv_scales), _ptr(sinks), int(window), int(num_splits), ctypes.byref(workspace.c), _ptr(out),
           _stream_handle(stream))
    _check(st, name)


def tllm_decode_attn_splitkv(q, k_cache, v_cache, block_table, context_lens, query_len, kv_scales, sinks, window,
                             num_splits, workspace: Workspace, out, stream=None) -> None:
    _call("tllm_decode_attn_splitkv", q, k_cache, v_cache, block_table, context_lens, query_len, kv_scales, sinks,
          window, num_splits, workspace, out, stream)


def tllm_decode_attn_partial(q, k_cache, v_cache, block_table, context_lens, query_len, kv_scales, sinks, window,
                             num_splits, workspace: Workspace, out, stream=None) -> None:
    _call("tllm_decode_attn_partial", q, k_cache, v_cache, block_table, context_lens, query_len, kv_scales, sinks,
          window, num_splits, workspace, out, stream)


def tllm_decode_attn_combine(q, k_cache, v_cache, block_table, context_lens, query_len, kv_scales, sinks, window,
                             num_splits, workspace: Workspace, out, stream=None) -> None:
    _call("tllm_decode_attn_combine", q, k_cache, v_cache, block_table, context_lens, query_len, kv_scales, sinks,
          window, num_splits, workspace, out, stream)


def tllm_decode_attn_noalloc_scratch_bytes() -> int:
    """Size of the library-owned record area of the no-alloc entry point (read from the library)."""
    return int(lib().tllm_decode_attn_noalloc_scratch_bytes())


def tllm_decode_attn_noalloc_read_status(reset: bool = False, stream=None) -> int:
    """Status word (TLLM_FLAG_*) of the no-alloc entry point's record area."""
    flags = ctypes.c_uint32()
    _check(lib().tllm_decode_attn_noalloc_read_status(ctypes.byref(flags), int(bool(reset)), _stream_handle(stream)),
           "tllm_decode_attn_noalloc_read_status")
    return flags.value


def tllm_decode_attn_splitkv_noalloc(q, k_cache, v_cache, block_table, context_lens, query_len, kv_scales, sinks,
                                     window, num_splits, plan: tllm_decode_attn_plan_t, out, stream=None) -> None:
    """The split-KV call with the records in the library's own device array, for callers
    that cannot allocate device memory (no workspace argument)."""
    st = lib().tllm_decode_attn_splitkv_noalloc(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table),
                                                _ptr(context_lens), int(query_len), _ptr(kv_scales), _ptr(sinks),
                                                int(window), int(num_splits), ctypes.byref(plan), _ptr(out),
                                                _stream_handle(stream))
    _check(st, "tllm_decode_attn_splitkv_noalloc")


def tllm_decode_attn_workspace_layout(plan: tllm_decode_attn_plan_t):
    so, lo, oo = ctypes.c_size_t(), ctypes.c_size_t(), ctypes.c_size_t()
    _check(lib().tllm_decode_attn_workspace_layout(ctypes.byref(plan), ctypes.byref(so), ctypes.byref(lo),
                                                   ctypes.byref(oo)), "tllm_decode_attn_workspace_layout")
    return so.value, lo.value, oo.value


def tllm_decode_attn_split_range(plan: tllm_decode_attn_plan_t, ctx: int, query_len: int, window: int,
                                 num_splits: int, split: int):
    t0, t1, n = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
    _check(lib().tllm_decode_attn_split_range(ctypes.byref(plan), int(ctx), int(query_len), int(window),
                                              int(num_splits), int(split), ctypes.byref(t0), ctypes.byref(t1),
                                              ctypes.byref(n)), "tllm_decode_attn_split_range")
    return t0.value, t1.value, n.value


def tllm_decode_attn_read_status(workspace: Workspace, reset: bool = False, stream=None) -> int:
    flags = ctypes.c_uint32()
    _check(lib().tllm_decode_attn_read_status(ctypes.byref(workspace.c), ctypes.byref(flags), int(bool(reset)),
                                              _stream_handle(stream)), "tllm_decode_attn_read_status")
    return flags.value


# --- convenience over the paged-cache inputs drawn by ``workloads`` -------------------

def desc_for(wl, kernel=TLLM_KERNEL_AUTO, num_pages: Optional[int] = None,
             v_layout=TLLM_V_TOKEN_MAJOR, record_type=TLLM_RECORD_F32,
             combine_mode=TLLM_COMBINE_KERNEL) -> tllm_decode_attn_desc:
    return make_desc(wl.Hq, wl.Hkv, wl.D, wl.bs, wl.max_blocks, num_pages if num_pages is not None else
                     wl.pages_needed() + wl.extra_pages, wl.q_dtype, wl.kv_dtype, wl.out_dtype, wl.scale, kernel,
                     v_layout, record_type, combine_mode)


def run(inp, workspace: Workspace, out: torch.Tensor, num_splits: Optional[int] = None, stream=None,
        window: Optional[int] = None) -> torch.Tensor:
    """One call of tllm_decode_attn_splitkv over an ``Inputs`` bundle already on the device."""
    wl = inp.wl
    tllm_decode_attn_splitkv(inp.q, inp.k_cache, inp.v_cache, inp.block_table, inp.context_lens, wl.Lq,
                             inp.kv_scales, inp.sinks, wl.window if window is None else window,
                             workspace.plan.num_splits if num_splits is None else num_splits, workspace, out, stream)
    return out

"""Paged grouped-query decode attention for GB300 (sm_103a).

Thin binding over the C ABI in ``include/decode_attn.h`` (the shared library
``_build/libpaged_gqa_decode.so``, built by ``build.build()``).  This module
only marshals arguments: torch tensors become raw device pointers, the
current CUDA stream becomes the ``stream`` argument, and the workspace is a
torch allocation cached per device and stream.  Every step of the computation runs in
the library's CUDA kernels; there is no other code path, and calling any
entry point without the built library raises.

Entry points (same names as the C ABI):
  decode_attn, decode_attn_split, decode_attn_combine, decode_attn_host,
  decode_attn_workspace_size, decode_attn_make_plan, decode_attn_strerror
"""
from __future__ import annotations

import ctypes
import functools
import os
import threading
from typing import Optional

__all__ = [
    "DecodeAttnParams", "DecodeAttnPlan", "DecodeAttnError", "load_library", "library_path",
    "make_params", "decode_attn", "decode_attn_split", "decode_attn_combine",
    "decode_attn_host", "decode_attn_workspace_size", "decode_attn_make_plan",
    "decode_attn_strerror", "VARIANT_AUTO", "VARIANT_SIMT", "VARIANT_MMA",
    "DEV_BAD_LEN", "DEV_BAD_PAGE", "DEV_OVER_HINT", "DEV_TIMEOUT", "DEV_CHECK",
    "decode_attn_static_scratch", "decode_attn_workspace_clear", "DEV_WORKSPACE",
    "decode_kv_append", "decode_attn_append", "DTYPE_FP16", "DTYPE_BF16",
    "SCHEDULE_AUTO", "SCHEDULE_GRID", "SCHEDULE_CLUSTER",
]

VARIANT_AUTO, VARIANT_SIMT, VARIANT_MMA = 0, 1, 2
SCHEDULE_AUTO, SCHEDULE_GRID, SCHEDULE_CLUSTER = 0, 1, 2
DTYPE_FP16, DTYPE_BF16 = 0, 1
DEV_BAD_LEN, DEV_BAD_PAGE, DEV_OVER_HINT, DEV_TIMEOUT, DEV_WORKSPACE = 1, 2, 4, 8, 16
DEV_CHECK = 32  # the checked build only: an index outside its buffer

_HERE = os.path.dirname(os.path.abspath(__file__))


def library_path() -> str:
    """The library this process loads: the checked build (bounds-checked
    kernels) when DECODE_ATTN_CHECKED=1, else the release build."""
    if os.environ.get("DECODE_ATTN_CHECKED") == "1":
        return os.path.join(_HERE, "_build_checked", "libpaged_gqa_decode_checked.so")
    return os.path.join(_HERE, "_build", "libpaged_gqa_decode.so")


class DecodeAttnParams(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "batch", "num_q_heads", "num_kv_heads", "head_dim", "page_size",
        "max_pages_per_seq", "num_pages", "max_seq_len")] + [
        ("scale", ctypes.c_float), ("window", ctypes.c_int32), ("variant", ctypes.c_int32),
        ("split_min", ctypes.c_int32), ("force_chunk", ctypes.c_int32),
        ("num_queries", ctypes.c_int32), ("dtype", ctypes.c_int32),
        ("schedule", ctypes.c_int32)]


class DecodeAttnPlan(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "split", "variant", "group_pad", "tile_tokens", "chunk_tokens", "max_shards",
        "grid_x", "grid_y", "grid_z", "ctas_per_sm", "head_fastest", "ring_stages",
        "cluster", "balanced")] + [
        ("workspace_bytes", ctypes.c_size_t)]

    def as_dict(self):
        return {n: getattr(self, n) for n, _ in self._fields_}


class DecodeAttnError(RuntimeError):
    def __init__(self, code: int, where: str):
        super().__init__(f"{where}: {decode_attn_strerror(code)} (status {code})")
        self.code = code


_lib = None
_lock = threading.Lock()


def load_library():
    """The CUDA library, loaded once.  Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            path = library_path()
            if not os.path.exists(path):
                raise RuntimeError(
                    f"CUDA library not built ({path} missing); run "
                    "paged_gqa_decode_06_gb300.build.build()")
            lib = ctypes.CDLL(path)
            P, i32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
            PP = ctypes.POINTER(DecodeAttnParams)
            lib.decode_attn_make_plan.argtypes = [PP, i32, ctypes.POINTER(DecodeAttnPlan)]
            lib.decode_attn_make_plan.restype = ctypes.c_int
            lib.decode_attn_workspace_size.argtypes = [PP, ctypes.c_int]
            lib.decode_attn_workspace_size.restype = sz
            for name in ("decode_attn", "decode_attn_split"):
                f = getattr(lib, name)
                f.argtypes = [PP, P, P, P, P, P, P, P, sz, P, P]
                f.restype = ctypes.c_int
            lib.decode_attn_combine.argtypes = [PP, P, P, P, sz, P, P]
            lib.decode_attn_combine.restype = ctypes.c_int
            lib.decode_attn_host.argtypes = [PP] + [P] * 12 + [sz, P, sz, P, P]
            lib.decode_attn_host.restype = ctypes.c_int
            lib.decode_kv_append.argtypes = [PP, P, P, P, P, P, P, P, P]
            lib.decode_kv_append.restype = ctypes.c_int
            lib.decode_attn_append.argtypes = [PP, P, P, P, P, P, P, P, P, P, sz, P, P]
            lib.decode_attn_append.restype = ctypes.c_int
            lib.decode_attn_workspace_clear.argtypes = [PP, P, sz, P]
            lib.decode_attn_workspace_clear.restype = ctypes.c_int
            lib.decode_attn_strerror.argtypes = [ctypes.c_int]
            lib.decode_attn_strerror.restype = ctypes.c_char_p
            _lib = lib
    return _lib


def _on_device_of(name: str, index: int):
    """Runs the wrapped call with the CUDA device of its tensor argument
    `name` (positional `index`) current: the library launches on the current
    device, and the default stream is that device's current stream, so
    tensors on another GPU than the current one still get their own device."""
    def deco(fn):
        @functools.wraps(fn)
        def wrapper(*args, **kwargs):
            import torch
            t = kwargs.get(name, args[index] if len(args) > index else None)
            if isinstance(t, torch.Tensor) and t.is_cuda and \
                    t.device.index not in (None, torch.cuda.current_device()):
                with torch.cuda.device(t.device):
                    return fn(*args, **kwargs)
            return fn(*args, **kwargs)
        return wrapper
    return deco


def decode_attn_strerror(code: int) -> str:
    return load_library().decode_attn_strerror(int(code)).decode()


def make_params(q, k_pages, page_table, scale: float, window: int = 0,
                max_seq_len: Optional[int] = None, variant: int = VARIANT_AUTO,
                split_min: int = 0, force_chunk: int = 0,
                schedule: int = SCHEDULE_AUTO) -> DecodeAttnParams:
    """Parameters from tensor shapes: q [B,Hq,D] (or [B,T,Hq,D] for T query
    positions per sequence), k_pages [P,PS,Hkv,D], page_table [B,maxPages].
    ``max_seq_len`` is a host-side bound on seq_lens (it sizes the grid;
    None = the page table's capacity).  ``schedule``: SCHEDULE_AUTO (the
    planner's grid or cluster plan), SCHEDULE_GRID or SCHEDULE_CLUSTER (a
    schedule the shape cannot take raises DecodeAttnError at planning)."""
    if len(q.shape) == 4:
        B, T, Hq, D = q.shape
    else:
        (B, Hq, D), T = q.shape, 1
    P, PS, Hkv, D2 = k_pages.shape
    if D2 != D:
        raise ValueError("q and k_pages head_dim differ")
    return DecodeAttnParams(
        batch=B, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D, page_size=PS,
        max_pages_per_seq=page_table.shape[1], num_pages=P,
        max_seq_len=int(max_seq_len) if max_seq_len else 0, scale=float(scale),
        window=int(window), variant=int(variant), split_min=int(split_min),
        force_chunk=int(force_chunk), num_queries=int(T), dtype=_dtype_code(q),
        schedule=int(schedule))


def _dtype_code(t) -> int:
    """DTYPE_BF16 for torch.bfloat16 tensors, else DTYPE_FP16."""
    return DTYPE_BF16 if str(getattr(t, "dtype", "")) == "torch.bfloat16" else DTYPE_FP16


def _elem_dtype(t):
    import torch
    if t.dtype not in (torch.float16, torch.bfloat16):
        raise TypeError(f"expected float16 or bfloat16 tensors, got {t.dtype}")
    return t.dtype


def decode_attn_make_plan(params: DecodeAttnParams, num_sms: int) -> DecodeAttnPlan:
    plan = DecodeAttnPlan()
    st = load_library().decode_attn_make_plan(ctypes.byref(params), int(num_sms),
                                              ctypes.byref(plan))
    if st:
        raise DecodeAttnError(st, "decode_attn_make_plan")
    return plan


def decode_attn_workspace_size(params: DecodeAttnParams, device: int) -> int:
    return int(load_library().decode_attn_workspace_size(ctypes.byref(params), int(device)))


@_on_device_of("workspace", 1)
def decode_attn_workspace_clear(params: DecodeAttnParams, workspace, stream=None) -> None:
    """Zeroes the workspace's shard tickets (needed once for a workspace that
    was not allocated zero-filled, or after a DEV_TIMEOUT / DEV_WORKSPACE)."""
    nbytes = workspace.numel() * workspace.element_size()
    st = load_library().decode_attn_workspace_clear(ctypes.byref(params), _ptr(workspace),
                                                    nbytes, _stream_handle(stream))
    if st:
        raise DecodeAttnError(st, "decode_attn_workspace_clear")


# ------------------------------------------------------------ torch glue

_ws_cache: dict = {}


def _workspace(device, nbytes: int, stream=None):
    """The cached workspace of (device, stream): calls on different streams
    may run at the same time, so each stream has its own tickets and
    partials.  A buffer is allocated zero-filled on the stream it serves, so
    the fill is ordered before that stream's kernels (and a replaced buffer
    is only reused by later work of the same stream)."""
    import torch
    if nbytes == 0:
        return None
    index = device.index if device.index is not None else torch.cuda.current_device()
    s = stream if stream is not None else torch.cuda.current_stream(index)
    key = (index, s.cuda_stream)
    buf = _ws_cache.get(key)
    if buf is None or buf.numel() < nbytes:
        # zero-filled: its shard tickets must start at zero (the kernels leave
        # them zero after every completed call)
        with torch.cuda.stream(s):
            buf = torch.zeros(max(nbytes, 1 << 20), dtype=torch.uint8, device=device)
        _ws_cache[key] = buf
    return buf


def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _check(t, dtype, name, device=None):
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")


def _stream_handle(stream) -> int:
    """The raw handle of `stream`, by default the current device's current
    stream; a stream of another device than the current one is refused."""
    import torch
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if stream.device.index != torch.cuda.current_device():
        raise ValueError(f"stream is on {stream.device}, the tensors on "
                         f"cuda:{torch.cuda.current_device()}")
    return stream.cuda_stream


def _prepare(q, k_pages, v_pages, page_table, seq_lens, out, scale, window, max_seq_len,
             variant, split_min, force_chunk, workspace, schedule=SCHEDULE_AUTO, stream=None):
    import torch
    dev = q.device
    if dev.type != "cuda":
        raise ValueError("decode_attn runs on CUDA tensors (use decode_attn_host for host "
                         "buffers)")
    et = _elem_dtype(q)
    _check(q, et, "q", dev)
    _check(k_pages, et, "k_pages", dev)
    _check(v_pages, et, "v_pages", dev)
    _check(page_table, torch.int32, "page_table", dev)
    _check(seq_lens, torch.int32, "seq_lens", dev)
    if v_pages.shape != k_pages.shape:
        raise ValueError("k_pages and v_pages shapes differ")
    p = make_params(q, k_pages, page_table, scale, window, max_seq_len, variant, split_min,
                    force_chunk, schedule)
    if out is None:
        out = torch.empty_like(q)
    _check(out, et, "out", dev)
    need = decode_attn_workspace_size(p, dev.index if dev.index is not None else
                                      torch.cuda.current_device())
    if workspace is None:
        workspace = _workspace(dev, need, stream)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    return p, out, workspace, ws_bytes


@_on_device_of("q", 0)
def decode_attn(q, k_pages, v_pages, page_table, seq_lens, scale: float, window: int = 0,
                out=None, max_seq_len: Optional[int] = None, workspace=None, err_flag=None,
                variant: int = VARIANT_AUTO, split_min: int = 0, force_chunk: int = 0,
                stream=None, schedule: int = SCHEDULE_AUTO):
    """One decode step of paged GQA attention; returns ``out`` [B,Hq,D] fp16.

    q [B,Hq,D] fp16, k_pages/v_pages [P,PS,Hkv,D] fp16, page_table [B,maxPages]
    int32, seq_lens [B] int32, all on one CUDA device.  ``window`` > 0 attends
    the last min(L, window) positions.  ``err_flag``: optional int32 device
    tensor of one element that receives DEV_* bits.  Enqueued on ``stream``
    (default: torch's current stream); does not synchronise.  ``workspace``:
    by default a zero-filled buffer cached per (device, stream); pass one to
    keep its fill out of a captured graph."""
    p, out, ws, ws_bytes = _prepare(q, k_pages, v_pages, page_table, seq_lens, out, scale,
                                    window, max_seq_len, variant, split_min, force_chunk,
                                    workspace, schedule, stream)
    st = load_library().decode_attn(ctypes.byref(p), _ptr(q), _ptr(k_pages), _ptr(v_pages),
                                    _ptr(page_table), _ptr(seq_lens), _ptr(out), _ptr(ws),
                                    ws_bytes, _ptr(err_flag), _stream_handle(stream))
    if st:
        raise DecodeAttnError(st, "decode_attn")
    return out


@_on_device_of("k_pages", 3)
def decode_kv_append(k_new, v_new, positions, k_pages, v_pages, page_table, err_flag=None,
                     stream=None):
    """Writes the step's new rows k_new/v_new [B,Hkv,D] at positions[b]
    (int32, -1 = none) into the paged pools, bit for bit."""
    import torch
    dev = k_pages.device
    et = _elem_dtype(k_pages)
    _check(k_new, et, "k_new", dev)
    _check(v_new, et, "v_new", dev)
    _check(positions, torch.int32, "positions", dev)
    _check(k_pages, et, "k_pages", dev)
    _check(v_pages, et, "v_pages", dev)
    _check(page_table, torch.int32, "page_table", dev)
    P, PS, Hkv, D = k_pages.shape
    if tuple(k_new.shape) != (page_table.shape[0], Hkv, D) or v_new.shape != k_new.shape:
        raise ValueError("k_new / v_new must be [B, Hkv, D]")
    p = DecodeAttnParams(batch=page_table.shape[0], num_q_heads=Hkv, num_kv_heads=Hkv,
                         head_dim=D, page_size=PS, max_pages_per_seq=page_table.shape[1],
                         num_pages=P, max_seq_len=0, scale=1.0, window=0, variant=0,
                         split_min=0, force_chunk=0, num_queries=1, dtype=_dtype_code(k_pages),
                         schedule=0)
    st = load_library().decode_kv_append(ctypes.byref(p), _ptr(k_new), _ptr(v_new),
                                         _ptr(positions), _ptr(k_pages), _ptr(v_pages),
                                         _ptr(page_table), _ptr(err_flag),
                                         _stream_handle(stream))
    if st:
        raise DecodeAttnError(st, "decode_kv_append")


@_on_device_of("q", 0)
def decode_attn_append(q, k_new, v_new, k_pages, v_pages, page_table, seq_lens, scale: float,
                       window: int = 0, out=None, max_seq_len: Optional[int] = None,
                       workspace=None, err_flag=None, variant: int = VARIANT_AUTO,
                       split_min: int = 0, force_chunk: int = 0, stream=None,
                       schedule: int = SCHEDULE_AUTO):
    """Append + attention in one launch: writes k_new/v_new [B,Hkv,D] (or
    [B,T,Hkv,D] with q [B,T,Hq,D]) at the last T positions of each sequence
    (seq_lens counts them), then attends as decode_attn."""
    import torch
    p, out, ws, ws_bytes = _prepare(q, k_pages, v_pages, page_table, seq_lens, out, scale,
                                    window, max_seq_len, variant, split_min, force_chunk,
                                    workspace, schedule, stream)
    _check(k_new, q.dtype, "k_new", q.device)
    _check(v_new, q.dtype, "v_new", q.device)
    st = load_library().decode_attn_append(ctypes.byref(p), _ptr(q), _ptr(k_new), _ptr(v_new),
                                           _ptr(k_pages), _ptr(v_pages), _ptr(page_table),
                                           _ptr(seq_lens), _ptr(out), _ptr(ws), ws_bytes,
                                           _ptr(err_flag), _stream_handle(stream))
    if st:
        raise DecodeAttnError(st, "decode_attn_append")
    return out


@_on_device_of("q", 0)
def decode_attn_split(q, k_pages, v_pages, page_table, seq_lens, scale: float, window: int = 0,
                      out=None, max_seq_len=None, workspace=None, err_flag=None,
                      variant: int = VARIANT_AUTO, split_min: int = 0, force_chunk: int = 0,
                      stream=None, schedule: int = SCHEDULE_AUTO):
    """The shard kernel alone (writes ``out`` directly for a single-pass plan,
    partials into ``workspace`` otherwise).  Returns (out, workspace)."""
    p, out, ws, ws_bytes = _prepare(q, k_pages, v_pages, page_table, seq_lens, out, scale,
                                    window, max_seq_len, variant, split_min, force_chunk,
                                    workspace, schedule, stream)
    st = load_library().decode_attn_split(ctypes.byref(p), _ptr(q), _ptr(k_pages),
                                          _ptr(v_pages), _ptr(page_table), _ptr(seq_lens),
                                          _ptr(out), _ptr(ws), ws_bytes, _ptr(err_flag),
                                          _stream_handle(stream))
    if st:
        raise DecodeAttnError(st, "decode_attn_split")
    return out, ws


@_on_device_of("out", 2)
def decode_attn_combine(params: DecodeAttnParams, seq_lens, out, workspace, err_flag=None,
                        stream=None):
    """The ordered combine alone, for ``params`` as used by decode_attn_split."""
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = load_library().decode_attn_combine(ctypes.byref(params), _ptr(seq_lens), _ptr(out),
                                            _ptr(workspace), ws_bytes, _ptr(err_flag),
                                            _stream_handle(stream))
    if st:
        raise DecodeAttnError(st, "decode_attn_combine")
    return out


@_on_device_of("d_q", 7)
def decode_attn_host(params: DecodeAttnParams, q_host, k_host, v_host, table_host, lens_host,
                     out_host, d_q, d_k, d_v, d_table, d_lens, d_out, workspace,
                     kv_bytes_to_copy: int = 0, err_flag=None, stream=None):
    """End-to-end step from host buffers (pinned CPU tensors): copies in,
    decode_attn, copies ``out`` back; enqueued on ``stream``, not awaited."""
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = load_library().decode_attn_host(
        ctypes.byref(params), _ptr(q_host), _ptr(k_host), _ptr(v_host), _ptr(table_host),
        _ptr(lens_host), _ptr(out_host), _ptr(d_q), _ptr(d_k), _ptr(d_v), _ptr(d_table),
        _ptr(d_lens), _ptr(d_out), int(kv_bytes_to_copy), _ptr(workspace), ws_bytes,
        _ptr(err_flag), _stream_handle(stream))
    if st:
        raise DecodeAttnError(st, "decode_attn_host")
    return out_host


# ------------------------------------------- no-allocation variant

def _static_scratch_fn():
    f = load_library().decode_attn_static_scratch
    if f.argtypes is None:
        P = ctypes.c_void_p
        f.argtypes = [ctypes.POINTER(DecodeAttnParams), P, P, P, P, P, P, P, P]
        f.restype = ctypes.c_int
    return f


@_on_device_of("q", 0)
def decode_attn_static_scratch(q, k_pages, v_pages, page_table, seq_lens, scale: float,
                               window: int = 0, out=None, max_seq_len: Optional[int] = None,
                               err_flag=None, variant: int = VARIANT_AUTO, split_min: int = 0,
                               force_chunk: int = 0, stream=None,
                               schedule: int = SCHEDULE_AUTO):
    """decode_attn for callers that cannot allocate device memory: the shard
    partials use the library's fixed 8 MiB device array instead of a
    workspace (shared by all calls on a device; overlapping calls race).
    Only ``out`` is created here when not given; pass it to allocate nothing."""
    import torch
    dev = q.device
    et = _elem_dtype(q)
    for t, dt, n in ((q, et, "q"), (k_pages, et, "k_pages"), (v_pages, et, "v_pages"),
                     (page_table, torch.int32, "page_table"), (seq_lens, torch.int32, "seq_lens")):
        _check(t, dt, n, dev)
    if out is None:
        out = torch.empty_like(q)
    _check(out, et, "out", dev)
    p = make_params(q, k_pages, page_table, scale, window, max_seq_len, variant, split_min,
                    force_chunk, schedule)
    st = _static_scratch_fn()(ctypes.byref(p), _ptr(q), _ptr(k_pages), _ptr(v_pages),
                              _ptr(page_table), _ptr(seq_lens), _ptr(out), _ptr(err_flag),
                              _stream_handle(stream))
    if st:
        raise DecodeAttnError(st, "decode_attn_static_scratch")
    return out

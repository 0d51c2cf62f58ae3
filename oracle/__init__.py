"""f64 CPU oracle for paged grouped-query decode attention.

TEST INFRASTRUCTURE ONLY.  The tests, the smoke check in ``__graft_entry__``
and the CPU-baseline leg of ``bench.py`` are the only callers allowed; the
library in ``paged_gqa_decode_06_gb300`` never imports this package.  The
arithmetic lives in ``decode_attn_oracle.c`` (plain C, IEEE double); this
module compiles it with gcc and marshals numpy arrays to it through ctypes.

What it computes, and the readings taken where the pages are silent, is
stated at the top of the C file.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "decode_attn_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "libdecode_attn_oracle.so")
_lock = threading.Lock()
_lib = None


class OracleShape(ctypes.Structure):
    _fields_ = [
        ("batch", ctypes.c_int32),
        ("num_q_heads", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("page_size", ctypes.c_int32),
        ("max_pages", ctypes.c_int32),
        ("num_pages", ctypes.c_int32),
        ("dtype", ctypes.c_int32),
    ]


def build(force: bool = False) -> str:
    """Compile the C oracle into ``oracle/_build`` (no-op when up to date)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
           "-pthread", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _bind(lib):
    P = ctypes.c_void_p
    i32, i64, f64 = ctypes.c_int32, ctypes.c_int64, ctypes.c_double
    lib.oracle_half_to_double.argtypes = [ctypes.c_uint16]
    lib.oracle_half_to_double.restype = f64
    lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
    lib.oracle_bf16_to_double.restype = f64
    lib.oracle_decode_attn_f64.argtypes = [
        ctypes.POINTER(OracleShape), P, P, P, P, P, f64, i32, P, i32, i32, P, P]
    lib.oracle_decode_attn_f64.restype = ctypes.c_int
    lib.oracle_partial_f64.argtypes = [
        ctypes.POINTER(OracleShape), P, P, P, P, i32, i32, f64, i64, i64, P, P, P]
    lib.oracle_partial_f64.restype = ctypes.c_int
    lib.oracle_merge_f64.argtypes = [i32, i32, P, P, P, P]
    lib.oracle_merge_f64.restype = None
    lib.oracle_decode_attn_multi_f64.argtypes = [
        ctypes.POINTER(OracleShape), i32, P, P, P, P, P, f64, i32, P, P]
    lib.oracle_decode_attn_multi_f64.restype = ctypes.c_int
    lib.oracle_kv_append_u16.argtypes = [ctypes.POINTER(OracleShape), P, P, P, P, P, P, P]
    lib.oracle_kv_append_u16.restype = ctypes.c_int
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
    return _lib


def compile_variant(src_text: str, out_dir: str) -> "Oracle":
    """Compile a modified copy of the oracle source (used only by the test
    that plants mistakes in the oracle to show its pins catch them)."""
    src = os.path.join(out_dir, "variant.c")
    lib = os.path.join(out_dir, "libvariant.so")
    with open(src, "w") as f:
        f.write(src_text)
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
                    "-pthread", src, "-o", lib, "-lm"], check=True)
    return Oracle(_bind(ctypes.CDLL(lib)))


def source_text() -> str:
    with open(_SRC) as f:
        return f.read()


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


class Bf16(np.ndarray):
    """uint16 array marked as holding bfloat16 bit patterns."""


def as_bf16_bits(a) -> "Bf16":
    return np.ascontiguousarray(a, dtype=np.uint16).view(Bf16)


def dtype_code(x) -> int:
    """0 for fp16 data, 1 for bfloat16 (torch.bfloat16 tensors or Bf16 arrays)."""
    if isinstance(x, Bf16):
        return 1
    if hasattr(x, "dtype") and str(x.dtype) == "torch.bfloat16":
        return 1
    return 0


def _as_u16(x) -> np.ndarray:
    """16-bit float data (numpy float16/uint16, or a CPU torch.float16 /
    torch.bfloat16 tensor) as its uint16 bit patterns."""
    if hasattr(x, "detach"):  # torch tensor
        import torch
        x = x.detach().to("cpu").contiguous().view(torch.int16).numpy()
    a = np.ascontiguousarray(x)
    if isinstance(a, Bf16):
        a = a.view(np.ndarray)
    if a.dtype == np.float16 or a.dtype == np.int16:
        a = a.view(np.uint16)
    assert a.dtype == np.uint16, a.dtype
    return a


def _as_i32(x) -> np.ndarray:
    if hasattr(x, "detach"):
        x = x.detach().to("cpu").numpy()
    return np.ascontiguousarray(x, dtype=np.int32)


def shape_of(q, k_pages, page_table) -> OracleShape:
    B, Hq, D = q.shape
    P, PS, Hkv, D2 = k_pages.shape
    assert D == D2
    return OracleShape(B, Hq, Hkv, D, PS, page_table.shape[1], P, dtype_code(k_pages))


def _half_to_double(lib, bits: int) -> float:
    return lib.oracle_half_to_double(bits)


def _bf16_to_double(lib, bits: int) -> float:
    return lib.oracle_bf16_to_double(bits)


def default_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def _decode_attn(lib, q, k_pages, v_pages, page_table, seq_lens, scale, window=0, rows=None,
                threads=None, return_errors=False):
    """f64 decode attention.  Shapes: q [B,Hq,D], k/v_pages [P,PS,Hkv,D] (fp16),
    page_table [B,maxPages] i32, seq_lens [B] i32.  Returns [B,Hq,D] f64, or
    [len(rows),D] when ``rows`` (flat b*Hq+hq indices) is given."""
    sh = shape_of(q, k_pages, page_table)
    qa, ka, va = _as_u16(q), _as_u16(k_pages), _as_u16(v_pages)
    pt, sl = _as_i32(page_table), _as_i32(seq_lens)
    if rows is None:
        n, rows_arr, rp = sh.batch * sh.num_q_heads, None, None
    else:
        rows_arr = np.ascontiguousarray(rows, dtype=np.int32)
        n, rp = rows_arr.size, _ptr(rows_arr)
    out = np.zeros((max(n, 1), sh.head_dim), dtype=np.float64)
    err = np.zeros(max(n, 1), dtype=np.int32)
    nt = threads or default_threads()
    st = lib.oracle_decode_attn_f64(ctypes.byref(sh), _ptr(qa), _ptr(ka), _ptr(va), _ptr(pt),
                                    _ptr(sl), float(scale), int(window), rp, n, nt, _ptr(out),
                                    _ptr(err))
    if st < 0:
        raise ValueError("oracle: bad shape")
    out = out[:n]
    if rows is None:
        out = out.reshape(sh.batch, sh.num_q_heads, sh.head_dim)
    if return_errors:
        return out, err[:n]
    return out


def _partial(lib, q, k_pages, v_pages, page_table, b, hq, scale, lo, hi):
    """(m, l, acc[D]) of row (b, hq) over logical positions [lo, hi)."""
    sh = shape_of(q, k_pages, page_table)
    qa, ka, va, pt = _as_u16(q), _as_u16(k_pages), _as_u16(v_pages), _as_i32(page_table)
    m, l = ctypes.c_double(), ctypes.c_double()
    acc = np.zeros(sh.head_dim, dtype=np.float64)
    st = lib.oracle_partial_f64(ctypes.byref(sh), _ptr(qa), _ptr(ka), _ptr(va), _ptr(pt),
                                int(b), int(hq), float(scale), int(lo), int(hi),
                                ctypes.byref(m), ctypes.byref(l), _ptr(acc))
    if st != 0:
        raise ValueError("oracle: bad page id in range")
    return m.value, l.value, acc


def _merge(lib, ms, ls, accs):
    """Ordered merge of partials (ascending index) into one output row."""
    m = np.ascontiguousarray(ms, dtype=np.float64)
    l = np.ascontiguousarray(ls, dtype=np.float64)
    acc = np.ascontiguousarray(accs, dtype=np.float64)
    n, D = acc.shape
    out = np.zeros(D, dtype=np.float64)
    lib.oracle_merge_f64(n, D, _ptr(m), _ptr(l), _ptr(acc), _ptr(out))
    return out


def _kv_append(lib, k_new, v_new, positions, page_table, k_pages, v_pages):
    """Returns new (k_pages, v_pages) uint16 arrays with the step's rows
    k_new/v_new [B,Hkv,D] written at positions[b] (inputs untouched), and the
    per-sequence error flags."""
    ka = _as_u16(k_pages).copy()
    va = _as_u16(v_pages).copy()
    kn, vn = _as_u16(k_new), _as_u16(v_new)
    pos, pt = _as_i32(positions), _as_i32(page_table)
    P_, PS, Hkv, D = ka.shape
    B = pt.shape[0]
    assert kn.shape == (B, Hkv, D) and vn.shape == (B, Hkv, D)
    sh = OracleShape(B, Hkv, Hkv, D, PS, pt.shape[1], P_)
    err = np.zeros(max(B, 1), dtype=np.int32)
    st = lib.oracle_kv_append_u16(ctypes.byref(sh), _ptr(kn), _ptr(vn), _ptr(pos), _ptr(pt),
                                  _ptr(ka), _ptr(va), _ptr(err))
    if st < 0:
        raise ValueError("oracle: bad shape")
    return ka, va, err[:B]


def _decode_attn_multi(lib, q, k_pages, v_pages, page_table, seq_lens, scale, window=0,
                       return_errors=False):
    """Several query positions per sequence: q [B,T,Hq,D] -> out [B,T,Hq,D]
    f64; query t of sequence b sits at position seq_lens[b] - T + t."""
    qa = _as_u16(q)
    B, T, Hq, D = qa.shape
    ka, va = _as_u16(k_pages), _as_u16(v_pages)
    pt, sl = _as_i32(page_table), _as_i32(seq_lens)
    P_, PS, Hkv, _ = ka.shape
    sh = OracleShape(B, Hq, Hkv, D, PS, pt.shape[1], P_, dtype_code(k_pages))
    out = np.zeros((max(B * T * Hq, 1), D), dtype=np.float64)
    err = np.zeros(max(B * T * Hq, 1), dtype=np.int32)
    st = lib.oracle_decode_attn_multi_f64(ctypes.byref(sh), T, _ptr(qa), _ptr(ka), _ptr(va),
                                          _ptr(pt), _ptr(sl), float(scale), int(window),
                                          _ptr(out), _ptr(err))
    if st < 0:
        raise ValueError("oracle: bad shape")
    out = out[:B * T * Hq].reshape(B, T, Hq, D)
    if return_errors:
        return out, err[:B * T * Hq].reshape(B, T, Hq)
    return out


class Oracle:
    """The oracle's entry points bound to one compiled library."""

    def __init__(self, lib):
        self.lib = lib

    def half_to_double(self, bits):
        return _half_to_double(self.lib, bits)

    def bf16_to_double(self, bits):
        return _bf16_to_double(self.lib, bits)

    def decode_attn(self, *a, **k):
        return _decode_attn(self.lib, *a, **k)

    def partial(self, *a, **k):
        return _partial(self.lib, *a, **k)

    def merge(self, *a, **k):
        return _merge(self.lib, *a, **k)

    def kv_append(self, *a, **k):
        return _kv_append(self.lib, *a, **k)

    def decode_attn_multi(self, *a, **k):
        return _decode_attn_multi(self.lib, *a, **k)


def default() -> Oracle:
    return Oracle(_load())


def half_to_double(bits: int) -> float:
    return _half_to_double(_load(), bits)


def decode_attn(*a, **k):
    """See ``_decode_attn``."""
    return _decode_attn(_load(), *a, **k)


def partial(*a, **k):
    return _partial(_load(), *a, **k)


def merge(*a, **k):
    return _merge(_load(), *a, **k)


def kv_append(*a, **k):
    """See ``_kv_append``."""
    return _kv_append(_load(), *a, **k)


def decode_attn_multi(*a, **k):
    """See ``_decode_attn_multi``."""
    return _decode_attn_multi(_load(), *a, **k)

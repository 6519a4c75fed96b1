"""Float64 CPU oracle for paged decode attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
legs of ``bench.py`` may import this package.  The product path (the CUDA
library and its binding in ``paged_kv_attention_attn_gb300``) never imports,
links or runs anything here, and this package imports nothing from it.

The arithmetic lives in ``pa_oracle.c`` (plain C, float64, loops over the
definition); this module compiles it with gcc and exposes it through ctypes
with numpy arrays.  ``pool_model`` and ``plan_model`` restate the allocator
policy and the partition-planner rule as plain Python.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "pa_oracle.c")
BUILD_DIR = os.path.join(HERE, "_build")
LIB_PATH = os.path.join(BUILD_DIR, "liboracle.so")

F16, Q8_0, Q4_0 = 0, 1, 2
TYPE_NAMES = {"f16": F16, "q8_0": Q8_0, "q4_0": Q4_0}

OR_OK, OR_ERR_INVALID, OR_ERR_NOMEM, OR_ERR_CORRUPT = 0, -1, -2, -5

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile pa_oracle.c into _build/liboracle.so with gcc (no fast-math,
    no FMA contraction, so float32 steps round exactly as written)."""
    os.makedirs(BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(LIB_PATH)
            and os.path.getmtime(LIB_PATH) >= os.path.getmtime(SRC)):
        return LIB_PATH
    tmp = LIB_PATH + f".{os.getpid()}.tmp"
    cmd = ["gcc", "-O2", "-std=c11", "-D_GNU_SOURCE", "-ffp-contract=off",
           "-fno-fast-math", "-fPIC", "-shared", "-pthread", SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


class OrArgs(ctypes.Structure):
    _fields_ = [
        ("k_pool", ctypes.c_void_p), ("v_pool", ctypes.c_void_p),
        ("n_pool_blocks", ctypes.c_uint64),
        ("block_table", ctypes.c_void_p), ("table_stride", ctypes.c_uint32),
        ("seq_lens", ctypes.c_void_p), ("q", ctypes.c_void_p),
        ("scale", ctypes.c_double),
        ("n_seqs", ctypes.c_uint32), ("hq", ctypes.c_uint32), ("hkv", ctypes.c_uint32),
        ("d", ctypes.c_uint32), ("block_size", ctypes.c_uint32),
        ("k_type", ctypes.c_int32), ("v_type", ctypes.c_int32),
        ("q_tokens", ctypes.c_uint32),
    ]


def lib():
    global _lib
    with _lock:
        if _lib is None:
            path = build()
            L = ctypes.CDLL(path)
            L.or_half_to_double.argtypes = [ctypes.c_uint16]
            L.or_half_to_double.restype = ctypes.c_double
            L.or_float_to_half_rn.argtypes = [ctypes.c_float]
            L.or_float_to_half_rn.restype = ctypes.c_uint16
            L.or_row_bytes.argtypes = [ctypes.c_int, ctypes.c_uint32]
            L.or_row_bytes.restype = ctypes.c_uint64
            L.or_dequant_row.argtypes = [ctypes.c_int, ctypes.c_void_p, ctypes.c_uint32,
                                         ctypes.c_void_p]
            L.or_dequant_row.restype = None
            L.or_quantize_q8_1.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64,
                                           ctypes.c_uint32]
            L.or_quantize_q8_1.restype = ctypes.c_int
            L.or_dequant_q8_1_row.argtypes = [ctypes.c_void_p, ctypes.c_uint32, ctypes.c_void_p]
            L.or_dequant_q8_1_row.restype = None
            L.or_quantize_row.argtypes = [ctypes.c_int, ctypes.c_void_p, ctypes.c_uint32,
                                          ctypes.c_void_p]
            L.or_quantize_row.restype = ctypes.c_int
            L.or_row_offset.argtypes = [ctypes.c_int64, ctypes.c_uint32, ctypes.c_uint32,
                                        ctypes.c_uint32, ctypes.c_uint32, ctypes.c_uint64]
            L.or_row_offset.restype = ctypes.c_uint64
            L.or_decode_units.argtypes = [ctypes.POINTER(OrArgs), ctypes.c_void_p, ctypes.c_int64,
                                          ctypes.c_uint32, ctypes.c_void_p, ctypes.c_int]
            L.or_decode_units.restype = ctypes.c_int
            L.or_merge.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                   ctypes.c_int64, ctypes.c_uint32, ctypes.c_uint32,
                                   ctypes.c_void_p]
            L.or_merge.restype = ctypes.c_int
            L.or_vmax_units.argtypes = [ctypes.POINTER(OrArgs), ctypes.c_void_p, ctypes.c_int64,
                                        ctypes.POINTER(ctypes.c_double)]
            L.or_vmax_units.restype = ctypes.c_int
            _lib = L
    return _lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


# ------------------------------------------------------------------ formats

def half_to_double(bits: int) -> float:
    return lib().or_half_to_double(int(bits))


def float_to_half_rn(x: float) -> int:
    return int(lib().or_float_to_half_rn(float(np.float32(x))))


def row_bytes(type_: int, d: int) -> int:
    return int(lib().or_row_bytes(int(type_), int(d)))


def dequant_row(type_: int, row: np.ndarray, d: int) -> np.ndarray:
    row = np.ascontiguousarray(row, dtype=np.uint8)
    assert row.size >= row_bytes(type_, d)
    out = np.empty(d, dtype=np.float64)
    lib().or_dequant_row(int(type_), _ptr(row), int(d), _ptr(out))
    return out


def quantize_q8_1(x: np.ndarray) -> np.ndarray:
    """x: float32 [..., D] -> uint8 [..., D/32*36] q8_1 blocks."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    d = x.shape[-1]
    n_rows = x.size // d
    out = np.empty(x.shape[:-1] + (d // 32 * 36,), dtype=np.uint8)
    rc = lib().or_quantize_q8_1(_ptr(x), _ptr(out), n_rows, d)
    if rc != OR_OK:
        raise ValueError(f"or_quantize_q8_1 rc={rc}")
    return out


def quantize_row(type_: int, x: np.ndarray) -> np.ndarray:
    """One float32 row of D values -> its pool-row bytes (F16 / Q8_0 / Q4_0),
    the append step's quantiser."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    d = x.shape[-1]
    out = np.empty(row_bytes(type_, d), dtype=np.uint8)
    rc = lib().or_quantize_row(int(type_), _ptr(x), int(d), _ptr(out))
    if rc != OR_OK:
        raise ValueError(f"or_quantize_row rc={rc}")
    return out


def dequant_q8_1_row(blocks: np.ndarray, d: int) -> np.ndarray:
    blocks = np.ascontiguousarray(blocks, dtype=np.uint8)
    out = np.empty(d, dtype=np.float64)
    lib().or_dequant_q8_1_row(_ptr(blocks), int(d), _ptr(out))
    return out


def row_offset(block: int, slot: int, kv_head: int, block_size: int, hkv: int,
               row_bytes_: int) -> int:
    return int(lib().or_row_offset(block, slot, kv_head, block_size, hkv, row_bytes_))


# ---------------------------------------------------------------- attention

class OracleError(RuntimeError):
    def __init__(self, rc: int):
        super().__init__(f"oracle refused: rc={rc}")
        self.rc = rc


def _args(k_pool, v_pool, block_table, seq_lens, q, hkv, block_size, k_type, v_type, scale):
    """q: float32 [S][hq][d], or [S][T][hq][d] for T query tokens per
    sequence (query row u = s * T + i)."""
    q = np.ascontiguousarray(q, dtype=np.float32)
    T = q.shape[1] if q.ndim == 4 else 1
    q = q.reshape(-1, q.shape[-2], q.shape[-1])
    S = q.shape[0] // T
    _, hq, d = q.shape
    k_pool = np.ascontiguousarray(k_pool).view(np.uint8)
    v_pool = np.ascontiguousarray(v_pool).view(np.uint8)
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    krb, vrb = row_bytes(k_type, d), row_bytes(v_type, d)
    n_blocks = k_pool.size // (block_size * hkv * krb)
    assert v_pool.size // (block_size * hkv * vrb) == n_blocks
    a = OrArgs(k_pool=_ptr(k_pool), v_pool=_ptr(v_pool), n_pool_blocks=n_blocks,
               block_table=_ptr(bt), table_stride=bt.shape[1] if bt.ndim == 2 else bt.size,
               seq_lens=_ptr(sl), q=_ptr(q),
               scale=float(1.0 / np.sqrt(d)) if scale is None else float(scale),
               n_seqs=S, hq=hq, hkv=hkv, d=d, block_size=block_size,
               k_type=int(k_type), v_type=int(v_type), q_tokens=T)
    keep = (q, k_pool, v_pool, bt, sl)  # arrays the struct points into
    return a, keep


def vmax(k_pool, v_pool, block_table, seq_lens, q, *, hkv, block_size, k_type, v_type,
         units=None) -> float:
    """max |Vhat| over the live rows that the listed units (default: every
    sequence and K/V head) read."""
    a, keep = _args(k_pool, v_pool, block_table, seq_lens, q, hkv, block_size, k_type, v_type,
                    None)
    S, hq, _ = keep[0].shape
    if units is None:
        units = [(s, h) for s in range(S) for h in range(0, hq, hq // hkv)]
    u = np.ascontiguousarray(np.asarray(units, dtype=np.int32).reshape(-1, 2))
    out = ctypes.c_double(0.0)
    rc = lib().or_vmax_units(ctypes.byref(a), _ptr(u), u.shape[0], ctypes.byref(out))
    if rc != OR_OK:
        raise OracleError(rc)
    return float(out.value)


def decode(k_pool, v_pool, block_table, seq_lens, q, *, hkv: int, block_size: int,
           k_type: int, v_type: int, scale: float | None = None, units=None,
           part_tokens: int = 0, n_threads: int | None = None) -> np.ndarray:
    """Float64 decode attention.

    k_pool / v_pool: uint8 arrays whose bytes are the token-major pools
    [n_blocks][block_size][hkv][row_bytes].  block_table int32 [S][stride],
    seq_lens int32 [S], q float32 [S][Hq][D], or [S][T][Hq][D] for T query
    tokens per sequence (token i at position L - T + i attends causally to
    keys 0 .. L - T + i).  units: optional list of (query row, head) pairs,
    query row u = s * T + i; default every pair.  Returns float64
    [n_units][D] (or q's shape when units is None).  part_tokens > 0 selects
    the partitioned-with-merge form of the same definition."""
    a, keep = _args(k_pool, v_pool, block_table, seq_lens, q, hkv, block_size, k_type, v_type,
                    scale)
    S, hq, d = keep[0].shape
    full = units is None
    if full:
        units = [(s, h) for s in range(S) for h in range(hq)]
    u = np.ascontiguousarray(np.asarray(units, dtype=np.int32).reshape(-1, 2))
    out = np.zeros((u.shape[0], d), dtype=np.float64)
    if n_threads is None:
        n_threads = max(1, len(os.sched_getaffinity(0)))
    rc = lib().or_decode_units(ctypes.byref(a), _ptr(u), u.shape[0], int(part_tokens),
                               _ptr(out), int(n_threads))
    if rc != OR_OK:
        raise OracleError(rc)
    return out.reshape(np.shape(q)) if full else out


def merge(o_bits: np.ndarray, ml: np.ndarray, n_live: np.ndarray) -> np.ndarray:
    """Float64 merge of f16 partials.  o_bits uint16 [U][P][D] (f16 bit
    patterns of o_p), ml float32 [U][P][2] (m_p in log2 domain, l_p),
    n_live int32 [U].  Returns float64 [U][D]."""
    o_bits = np.ascontiguousarray(o_bits, dtype=np.uint16)
    ml = np.ascontiguousarray(ml, dtype=np.float32)
    nl = np.ascontiguousarray(n_live, dtype=np.int32)
    U, P, D = o_bits.shape
    out = np.zeros((U, D), dtype=np.float64)
    rc = lib().or_merge(_ptr(o_bits), _ptr(ml), _ptr(nl), U, P, D, _ptr(out))
    if rc != OR_OK:
        raise OracleError(rc)
    return out

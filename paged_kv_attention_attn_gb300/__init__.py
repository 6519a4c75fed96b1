"""Python binding of libpa.so, the paged decode-attention library for GB300.

Argument marshalling only: every step of the decode path runs in the
library's CUDA kernels.  PyTorch provides device memory and streams.  The
binding fails loudly (ImportError at first use) when the library has not been
built; there is no CPU fallback.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading
from dataclasses import dataclass

import torch

F16, Q8_0, Q4_0 = 0, 1, 2
TYPES = {"f16": F16, "q8_0": Q8_0, "q4_0": Q4_0}

PA_OK, PA_ERR_INVALID, PA_ERR_NOMEM, PA_ERR_STALE = 0, -1, -2, -3
PA_ERR_CUDA, PA_ERR_CORRUPT_TABLE, PA_ERR_RANGE, PA_ERR_TIMEOUT = -4, -5, -6, -7
PA_STATUS_CORRUPT_TABLE, PA_STATUS_TIMEOUT, PA_STATUS_LEN_OVER_PLAN = 1, 2, 4
PA_STATUS_APPEND_RANGE = 8
PA_FLAG_PLAIN = 1
PA_FLAG_MERGE_NO_WAIT = 2
PA_PLAN_STREAM_OK = 1
PA_PLAN_MULTI_TOKEN = 2

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_build", "libpa.so")


class PAError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{msg} [{code}]")
        self.code = code


class PlanIn(ctypes.Structure):
    _fields_ = [("n_seqs", ctypes.c_uint32), ("max_len", ctypes.c_uint32),
                ("total_len", ctypes.c_uint64), ("block_size", ctypes.c_uint32),
                ("hq", ctypes.c_uint32), ("hkv", ctypes.c_uint32), ("d", ctypes.c_uint32),
                ("k_type", ctypes.c_int), ("v_type", ctypes.c_int),
                ("sm_count", ctypes.c_int32), ("ctas_per_sm", ctypes.c_int32),
                ("force_parts", ctypes.c_int32), ("q_tokens", ctypes.c_uint32),
                ("flags", ctypes.c_uint32)]


class Plan(ctypes.Structure):
    _fields_ = [("part_tokens", ctypes.c_uint32), ("n_parts", ctypes.c_uint32),
                ("direct", ctypes.c_uint32), ("n_ctas", ctypes.c_uint32),
                ("part_o_bytes", ctypes.c_uint64), ("part_ml_bytes", ctypes.c_uint64),
                ("counter_bytes", ctypes.c_uint64), ("q_tokens", ctypes.c_uint32),
                ("n_direct", ctypes.c_uint32), ("stream", ctypes.c_uint32),
                ("multi", ctypes.c_uint32)]

    def as_dict(self):
        return {k: int(getattr(self, k)) for k, _ in self._fields_}


class DecodeArgs(ctypes.Structure):
    _fields_ = [("k_pool", ctypes.c_void_p), ("v_pool", ctypes.c_void_p),
                ("n_pool_blocks", ctypes.c_uint64),
                ("block_table", ctypes.c_void_p), ("table_stride", ctypes.c_uint32),
                ("seq_lens", ctypes.c_void_p), ("q", ctypes.c_void_p),
                ("scale", ctypes.c_float),
                ("part_o", ctypes.c_void_p), ("part_ml", ctypes.c_void_p),
                ("out", ctypes.c_void_p), ("status", ctypes.c_void_p),
                ("n_seqs", ctypes.c_uint32), ("hq", ctypes.c_uint32), ("hkv", ctypes.c_uint32),
                ("d", ctypes.c_uint32), ("block_size", ctypes.c_uint32),
                ("k_type", ctypes.c_int), ("v_type", ctypes.c_int),
                ("flags", ctypes.c_uint32)]


_lib = None
_lock = threading.Lock()
_vp, _u32, _u64, _i32 = ctypes.c_void_p, ctypes.c_uint32, ctypes.c_uint64, ctypes.c_int32

class AppendArgs(ctypes.Structure):
    _fields_ = [("k_pool", ctypes.c_void_p), ("v_pool", ctypes.c_void_p),
                ("n_pool_blocks", ctypes.c_uint64),
                ("block_table", ctypes.c_void_p), ("table_stride", ctypes.c_uint32),
                ("seq_lens", ctypes.c_void_p), ("k_new", ctypes.c_void_p),
                ("v_new", ctypes.c_void_p), ("fresh_blocks", ctypes.c_void_p),
                ("status", ctypes.c_void_p),
                ("n_seqs", ctypes.c_uint32), ("hkv", ctypes.c_uint32), ("d", ctypes.c_uint32),
                ("block_size", ctypes.c_uint32), ("k_type", ctypes.c_int),
                ("v_type", ctypes.c_int)]


_SIGNATURES = {
    "pa_strerror": ([ctypes.c_int], ctypes.c_char_p),
    "pa_last_error": ([], ctypes.c_char_p),
    "pa_row_bytes": ([ctypes.c_int, _u32], _u64),
    "pa_pool_create": ([_u32, ctypes.POINTER(_vp)], ctypes.c_int),
    "pa_pool_destroy": ([_vp], None),
    "pa_pool_alloc": ([_vp, _u32, _vp], ctypes.c_int),
    "pa_pool_free": ([_vp, _u32, _vp], ctypes.c_int),
    "pa_handle_block": ([_u64], _i32),
    "pa_pool_free_count": ([_vp], _u32),
    "pa_pool_capacity": ([_vp], _u32),
    "pa_quantize_q": ([_vp, _vp, _u32, _u32, _vp], ctypes.c_int),
    "pa_plan": ([ctypes.POINTER(PlanIn), ctypes.POINTER(Plan)], ctypes.c_int),
    "pa_query_occupancy": ([ctypes.POINTER(PlanIn), ctypes.POINTER(_i32),
                            ctypes.POINTER(_i32)], ctypes.c_int),
    "pa_decode_partial": ([ctypes.POINTER(DecodeArgs), ctypes.POINTER(Plan), _vp],
                          ctypes.c_int),
    "pa_decode_kernel_name": ([ctypes.c_int, ctypes.c_int, _u32, _u32, _u32, _u32, _u32],
                              ctypes.c_char_p),
    "pa_decode_fused": ([ctypes.POINTER(DecodeArgs), ctypes.POINTER(Plan), _vp, _vp],
                        ctypes.c_int),
    "pa_decode_step_fused": ([ctypes.POINTER(DecodeArgs), ctypes.POINTER(Plan), _vp, _vp, _vp],
                             ctypes.c_int),
    "pa_merge": ([_vp, _vp, _vp, _vp, _u32, _u32, _u32, ctypes.POINTER(Plan), _vp],
                 ctypes.c_int),
    "pa_decode_step": ([ctypes.POINTER(DecodeArgs), ctypes.POINTER(Plan), _vp, _vp],
                       ctypes.c_int),
    "pa_decode_step_host": ([_vp, _vp, ctypes.POINTER(DecodeArgs), ctypes.POINTER(Plan),
                             _vp, _vp], ctypes.c_int),
    "pa_decode_step_noalloc": ([ctypes.POINTER(DecodeArgs), ctypes.POINTER(Plan), _vp],
                               ctypes.c_int),
    "pa_decode_step_fused_host": ([_vp, _vp, ctypes.POINTER(DecodeArgs), ctypes.POINTER(Plan),
                                   _vp, _vp, _vp], ctypes.c_int),
    "pa_append_kv": ([ctypes.POINTER(AppendArgs), _vp], ctypes.c_int),
    "pa_status_read": ([_vp, _vp, ctypes.POINTER(_i32), ctypes.c_int], ctypes.c_int),
    "pa_debug_row_offsets": ([_vp, _u32, _vp, _u32, _u32, _u32, _u32, _u64, _u64, _vp,
                              _vp, _vp], ctypes.c_int),
}
EXPORTS = list(_SIGNATURES)


def lib(path: str | None = None):
    """Loads libpa.so (built in-tree by ``build.py``); raises if it is missing."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise ImportError(f"libpa.so not built at {p}: run "
                              "python -m paged_kv_attention_attn_gb300.build")
        L = ctypes.CDLL(p)
        for name, (argt, rest) in _SIGNATURES.items():
            fn = getattr(L, name)
            fn.argtypes = argt
            fn.restype = rest
        _lib = L
        return _lib


def _check(rc: int):
    if rc != PA_OK:
        L = lib()
        raise PAError(rc, f"{L.pa_strerror(rc).decode()}: {L.pa_last_error().decode()}")


def _ptr(t: torch.Tensor | None) -> int | None:
    return None if t is None else t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        if torch.cuda.is_available() and torch.cuda.is_initialized():
            return torch.cuda.current_stream().cuda_stream
        return None
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def row_bytes(type_: int, d: int) -> int:
    return int(lib().pa_row_bytes(int(type_), int(d)))


# ------------------------------------------------------------------ allocator

class Pool:
    """Fixed-block allocator (host object owned by the library)."""

    def __init__(self, n_blocks: int):
        h = _vp()
        _check(lib().pa_pool_create(int(n_blocks), ctypes.byref(h)))
        self._h = h

    def close(self):
        if getattr(self, "_h", None):
            lib().pa_pool_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def alloc(self, n: int) -> list[int]:
        arr = (ctypes.c_uint64 * max(1, n))()
        _check(lib().pa_pool_alloc(self._h, int(n), arr))
        return [int(arr[i]) for i in range(n)]

    def free(self, handles) -> None:
        handles = list(handles)
        arr = (ctypes.c_uint64 * max(1, len(handles)))(*handles)
        _check(lib().pa_pool_free(self._h, len(handles), arr))

    def free_count(self) -> int:
        return int(lib().pa_pool_free_count(self._h))

    def capacity(self) -> int:
        return int(lib().pa_pool_capacity(self._h))

    @staticmethod
    def block_of(h: int) -> int:
        return int(lib().pa_handle_block(ctypes.c_uint64(h)))


# -------------------------------------------------------------------- planner

def _plan_in(n_seqs, max_len, total_len, block_size, hq, hkv, d, k_type, v_type,
             sm_count, ctas_per_sm, force_parts):
    return PlanIn(n_seqs=n_seqs, max_len=max_len, total_len=total_len, block_size=block_size,
                  hq=hq, hkv=hkv, d=d, k_type=k_type, v_type=v_type, sm_count=sm_count,
                  ctas_per_sm=ctas_per_sm, force_parts=force_parts)


def query_occupancy(*, hq, hkv, d, block_size, k_type, v_type) -> tuple[int, int]:
    pin = _plan_in(1, 0, 0, block_size, hq, hkv, d, k_type, v_type, 1, 1, 0)
    sm, cps = _i32(), _i32()
    _check(lib().pa_query_occupancy(ctypes.byref(pin), ctypes.byref(sm), ctypes.byref(cps)))
    return int(sm.value), int(cps.value)


def plan(*, seq_lens, block_size, hq, hkv, d, k_type, v_type, sm_count=None,
         ctas_per_sm=None, force_parts=0, q_tokens=1, stream_ok=False, multi=False) -> Plan:
    """pa_plan for these lengths; q_tokens query tokens per sequence;
    stream_ok lets the planner return a stream plan (fused calls only);
    multi asks for a multi-token plan (the tokens of a sequence together)."""
    lens = [int(x) for x in seq_lens]
    if sm_count is None or ctas_per_sm is None:
        sm, cps = query_occupancy(hq=hq, hkv=hkv, d=d, block_size=block_size, k_type=k_type,
                                  v_type=v_type)
        sm_count = sm if sm_count is None else sm_count
        ctas_per_sm = cps if ctas_per_sm is None else ctas_per_sm
    pin = _plan_in(len(lens), max(lens) if lens else 0, sum(lens), block_size, hq, hkv, d,
                   k_type, v_type, sm_count, ctas_per_sm, force_parts)
    pin.q_tokens = int(q_tokens)
    pin.flags = (PA_PLAN_STREAM_OK if stream_ok else 0) | (PA_PLAN_MULTI_TOKEN if multi else 0)
    out = Plan()
    _check(lib().pa_plan(ctypes.byref(pin), ctypes.byref(out)))
    return out


# ---------------------------------------------------------------- device ops

def quantize_q(q: torch.Tensor, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """float32 [..., D] (CUDA) -> uint8 [..., D/32*36] q8_1 blocks."""
    assert q.is_cuda and q.dtype == torch.float32 and q.is_contiguous()
    d = q.shape[-1]
    n_rows = q.numel() // d if d else 0
    if out is None:
        out = torch.empty(q.shape[:-1] + (d // 32 * 36,), dtype=torch.uint8, device=q.device)
    _check(lib().pa_quantize_q(_ptr(q), _ptr(out), n_rows, d, _stream(stream)))
    return out


@dataclass
class Workspace:
    """Caller-owned device buffers of one decode step."""
    plan: Plan
    out: torch.Tensor       # float32 [S, hq, d]
    part_o: torch.Tensor    # float16 [S, hq, n_parts, d] (empty if direct)
    part_ml: torch.Tensor   # float32 [S, hq, n_parts, 2]
    status: torch.Tensor    # int32 [1]
    q8_1: torch.Tensor      # uint8 [S, hq, d/32*36]
    counters: torch.Tensor  # int32 [S], zero: fused-merge completion counters


def workspace(pl: Plan, *, n_seqs, hq, d, device) -> Workspace:
    """Buffers of one step: out float32 [S, hq, d], or [S, T, hq, d] for a
    plan with T > 1 query tokens per sequence; partials per partitioned query
    row (the rows after the plan's n_direct leading direct ones)."""
    P = 0 if pl.direct else int(pl.n_parts)
    T = max(1, int(pl.q_tokens))
    rows = n_seqs * T - (0 if pl.direct else int(pl.n_direct))
    lead = (n_seqs,) if T == 1 else (n_seqs, T)
    return Workspace(
        plan=pl,
        out=torch.zeros(lead + (hq, d), dtype=torch.float32, device=device),
        part_o=torch.empty((rows, hq, P, d), dtype=torch.float16, device=device),
        part_ml=torch.empty((rows, hq, P, 2), dtype=torch.float32, device=device),
        status=torch.zeros(1, dtype=torch.int32, device=device),
        q8_1=torch.empty(lead + (hq, d // 32 * 36), dtype=torch.uint8, device=device),
        counters=torch.zeros(max(1, int(pl.counter_bytes) // 4), dtype=torch.int32,
                             device=device))


def make_args(*, k_pool, v_pool, block_table, seq_lens, q, ws: Workspace, hkv, block_size,
              k_type, v_type, scale=None, flags=0) -> DecodeArgs:
    S, hq, d = ws.out.shape[0], ws.out.shape[-2], ws.out.shape[-1]
    return DecodeArgs(k_pool=_ptr(k_pool), v_pool=_ptr(v_pool), n_pool_blocks=k_pool.shape[0],
                      block_table=_ptr(block_table), table_stride=block_table.shape[1],
                      seq_lens=_ptr(seq_lens), q=_ptr(q),
                      scale=float(1.0 / math.sqrt(d)) if scale is None else float(scale),
                      part_o=_ptr(ws.part_o) if ws.part_o.numel() else None,
                      part_ml=_ptr(ws.part_ml) if ws.part_ml.numel() else None,
                      out=_ptr(ws.out), status=_ptr(ws.status), n_seqs=S, hq=hq, hkv=hkv, d=d,
                      block_size=block_size, k_type=k_type, v_type=v_type, flags=flags)


def decode_partial(args: DecodeArgs, pl: Plan, stream=None) -> None:
    _check(lib().pa_decode_partial(ctypes.byref(args), ctypes.byref(pl), _stream(stream)))


def decode_kernel_name(*, k_type, v_type, d, hq, hkv, block_size, flags=0) -> str | None:
    """Which decode kernel pa_decode_partial would launch for these shapes."""
    r = lib().pa_decode_kernel_name(k_type, v_type, d, hq, hkv, block_size, flags)
    return r.decode() if r else None


def decode_fused(args: DecodeArgs, ws: Workspace, stream=None) -> None:
    """pa_decode_fused: decode with the merge inside the same launch."""
    _check(lib().pa_decode_fused(ctypes.byref(args), ctypes.byref(ws.plan), _ptr(ws.counters),
                                 _stream(stream)))


def decode_step_fused(args: DecodeArgs, ws: Workspace, stream=None) -> None:
    """pa_decode_step_fused: the step with the in-launch merge (args.q is the
    float32 query).  On the fast kernel one launch that also quantises the
    query; otherwise the q8_1 pre-pass first."""
    _check(lib().pa_decode_step_fused(ctypes.byref(args), ctypes.byref(ws.plan), _ptr(ws.q8_1),
                                      _ptr(ws.counters), _stream(stream)))


def append_kv(*, k_pool, v_pool, block_table, seq_lens, k_new, v_new, fresh_blocks, status,
              hkv, block_size, k_type, v_type, stream=None) -> None:
    """pa_append_kv: quantise each sequence's new K/V rows (float32
    [S, hkv, d]) into the pool at its resident length; fresh_blocks[s] is
    taken when the token starts a block."""
    S, _, d = k_new.shape
    a = AppendArgs(k_pool=_ptr(k_pool), v_pool=_ptr(v_pool), n_pool_blocks=k_pool.shape[0],
                   block_table=_ptr(block_table), table_stride=block_table.shape[1],
                   seq_lens=_ptr(seq_lens), k_new=_ptr(k_new), v_new=_ptr(v_new),
                   fresh_blocks=_ptr(fresh_blocks), status=_ptr(status), n_seqs=S, hkv=hkv,
                   d=d, block_size=block_size, k_type=k_type, v_type=v_type)
    _check(lib().pa_append_kv(ctypes.byref(a), _stream(stream)))


def merge(ws: Workspace, seq_lens: torch.Tensor, stream=None) -> None:
    S, hq, d = ws.out.shape
    _check(lib().pa_merge(_ptr(ws.part_o), _ptr(ws.part_ml), _ptr(seq_lens), _ptr(ws.out), S, hq,
                          d, ctypes.byref(ws.plan), _stream(stream)))


def decode_step(args: DecodeArgs, ws: Workspace, stream=None) -> None:
    """pa_decode_step: quantise Q (quantised K), decode, merge (unless direct).
    args.q must point at the float32 query."""
    _check(lib().pa_decode_step(ctypes.byref(args), ctypes.byref(ws.plan), _ptr(ws.q8_1),
                                _stream(stream)))


def decode_step_host(q_host: torch.Tensor, out_host: torch.Tensor, args: DecodeArgs,
                     ws: Workspace, stream=None) -> None:
    """pa_decode_step_host: q from and out to host (page-locked) memory."""
    assert not q_host.is_cuda and not out_host.is_cuda
    _check(lib().pa_decode_step_host(_ptr(q_host), _ptr(out_host), ctypes.byref(args),
                                     ctypes.byref(ws.plan), _ptr(ws.q8_1), _stream(stream)))


NOALLOC_SCRATCH_BYTES = 16 << 20


def decode_step_noalloc(args: DecodeArgs, pl: Plan, stream=None) -> None:
    """pa_decode_step_noalloc: the decode step with the library's static
    scratch instead of caller buffers, for callers that cannot allocate
    device memory.  args.q must point at the float32 query; args.part_o and
    args.part_ml are ignored."""
    _check(lib().pa_decode_step_noalloc(ctypes.byref(args), ctypes.byref(pl), _stream(stream)))


def decode_step_fused_host(q_host: torch.Tensor, out_host: torch.Tensor, args: DecodeArgs,
                           ws: Workspace, stream=None) -> None:
    """pa_decode_step_fused_host: host q in, fused decode, host out back."""
    assert not q_host.is_cuda and not out_host.is_cuda
    _check(lib().pa_decode_step_fused_host(_ptr(q_host), _ptr(out_host), ctypes.byref(args),
                                           ctypes.byref(ws.plan), _ptr(ws.q8_1),
                                           _ptr(ws.counters), _stream(stream)))


def status_read(status: torch.Tensor, reset: bool = True, stream=None) -> int:
    """Returns the status word bits (synchronises the stream)."""
    v = _i32()
    rc = lib().pa_status_read(_ptr(status), _stream(stream), ctypes.byref(v), int(reset))
    if rc not in (PA_OK, PA_ERR_CORRUPT_TABLE, PA_ERR_TIMEOUT, PA_ERR_RANGE):
        _check(rc)
    return int(v.value)


def debug_row_offsets(block_table, seq_lens, *, max_tokens, block_size, hkv, row_bytes_,
                      n_pool_blocks, status, stream=None) -> torch.Tensor:
    S = seq_lens.shape[0]
    out = torch.empty((S, max_tokens, hkv), dtype=torch.int64, device=block_table.device)
    _check(lib().pa_debug_row_offsets(_ptr(block_table), block_table.shape[1], _ptr(seq_lens), S,
                                      max_tokens, block_size, hkv, row_bytes_, n_pool_blocks,
                                      _ptr(out), _ptr(status), _stream(stream)))
    return out

"""Benchmark of one paged decode-attention step on GB300.

Workload (default): the uniform batch at Qwen attention dims -- 8 sequences
of 131,072 tokens, D=256, Hq=24, Hkv=4, 16-token blocks, Q4_0 K/V from
N(0,1), fp32 Q from N(0,1) quantised to q8_1, block tables randomly
interleaved in one pool ("feat: add paged-attention monolithic decode-only AR
foundation", lucebox pull 555, Benchmark results).  A step is the whole hot
path through the public call pa_decode_step_fused: q8_1 quantisation of the
query, the decode and the merge.  With the fast kernel that is one launch
(the kernel quantises the query itself and merges in-launch); otherwise the
q8_1 pre-pass and the decode launch (--unfused: pre-pass, decode, merge).

Prints ONE JSON line (rank 0).  `value` is achieved algorithmic HBM
bandwidth in GB/s over all ranks (bytes every rank's steps must move / the
slowest rank's time); `us_per_step` is the step time.  The roofline object
reports the decode kernel alone, timed with CUDA events around its launch
inside the timed loop.  `--impl reference` times the float64 CPU oracle on
a bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = ("paged decode-attn µs/step and achieved HBM GB/s vs GB300 peak "
          "(Q4_0 K/V, 1 GPU)")
WORKLOADS = {
    # uniform batches 1/2/4/8 x 4K/32K/128K, Q4_0
    **{f"uniform-q4_0-b{b}x{c}": (lambda b=b, c=c: synth.uniform_spec(b, c, synth.Q4_0))
       for b in (1, 2, 4, 8) for c in (4096, 32768, 131072)},
    "ragged-q4_0-128k+7x8k": lambda: synth.ragged_spec(synth.Q4_0),
    # the same rows in the padded contiguous layout (identity tables)
    "ragged-q4_0-128k+7x8k-contiguous": lambda: synth.ragged_spec(synth.Q4_0),
    **{f"sweep-{n}-{tag}": (lambda t=t, sh=sh: synth.dtype_sweep_spec(t, short=sh))
       for n, t in (("f16", synth.F16), ("q8_0", synth.Q8_0), ("q4_0", synth.Q4_0))
       for tag, sh in (("b4x32768", False), ("short", True))},
    # the six mixed K x V pairs of the dtype sweep (4 x 32768)
    **{f"sweep-{kn}-{vn}-b4x32768": (lambda kt=kt, vt=vt: synth.dtype_sweep_spec(kt, v_type=vt))
       for kn, kt in (("f16", synth.F16), ("q8_0", synth.Q8_0), ("q4_0", synth.Q4_0))
       for vn, vt in (("f16", synth.F16), ("q8_0", synth.Q8_0), ("q4_0", synth.Q4_0))
       if kt != vt},
    "verify-q4_0-b8x32768-T4": synth.verify_spec,
    # batches wider than the machine (152 SMs): a short last wave filled by
    # splitting its sequences, and whole waves
    **{f"wide-q4_0-b{b}x{c}": (lambda b=b, c=c: synth.uniform_spec(b, c, synth.Q4_0))
       for b, c in ((160, 6912), (512, 4096), (304, 4096), (1024, 1024))},
    "tiny-f16-L200": synth.tiny_spec,
    "largepool-f16-b16x300000": synth.large_pool_spec,
}
DEFAULT_WORKLOAD = "uniform-q4_0-b8x131072"
L2_BYTES = 129 * 2**20        # GB300 L2
FLUSH_BYTES = 512 * 2**20     # the write that evicts it between timed steps (--flush on)
MAX_LAYERS = 1024             # pool copies cycled through when K/V is under twice the L2


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def algorithmic_bytes(spec, plan, fused: bool = True, in_kernel_q: bool = False) -> dict:
    """Bytes the method must move in one step, by class.  With the fused
    merge the decode launch also reads the partials back and writes out;
    with in-kernel quantisation it reads the float32 query and there is no
    pre-pass."""
    S, hq, d = spec.n_seqs, spec.hq, spec.d
    T = int(spec.extra.get("q_tokens", 1))
    krb, vrb = synth.row_bytes(spec.k_type, d), synth.row_bytes(spec.v_type, d)
    lens = spec.seq_lens
    kv = sum(lens) * spec.hkv * (krb + vrb)   # once: a sequence's query rows share them
    table = sum(math.ceil(L / spec.block_size) for L in lens) * 4
    rows = [max(0, L - (T - 1 - i)) for L in lens for i in range(T)]
    q_f32 = S * T * hq * d * 4
    q81 = S * T * hq * d // 32 * 36
    quantised = spec.k_type != synth.F16
    prepass = (q_f32 + q81) if quantised and not in_kernel_q else 0
    q_read = q81 if quantised and not in_kernel_q else q_f32
    out = S * T * hq * d * 4
    if plan.direct:
        part_w = part_r = 0
        dec_out = out
    elif getattr(plan, "stream", 0):
        # a stream plan: rows cut by the CTAs' tile ranges get one partial per
        # CTA that covers them; the others are written directly
        chunk = plan.part_tokens // 16
        pre, live, out_direct = 0, 0, 0
        for L in rows:
            tiles = -(-L // 16)
            if tiles:
                nr = (pre + tiles - 1) // chunk - pre // chunk + 1
                if nr > 1:
                    live += nr
                else:
                    out_direct += hq * d * 4
            pre += tiles
        part_w = part_r = live * hq * (2 * d + 8)
        dec_out = part_w + out_direct
        out -= out_direct  # what the merges write
    else:
        # the leading n_direct rows of a wave-filling plan write out directly
        nd = int(plan.n_direct)
        live = sum(math.ceil(L / plan.part_tokens) for L in rows[nd:])
        part_w = part_r = live * hq * (2 * d + 8)
        out_direct = nd * hq * d * 4
        dec_out = part_w + out_direct
        out -= out_direct  # what the merge writes
    merge = 0 if plan.direct else part_r + out + S * 4
    decode = kv + table + q_read + dec_out + S * 4
    if fused and not plan.direct:
        decode += merge
        merge = 0
    return dict(kv=kv, table=table, prepass=prepass, decode=decode, merge=merge,
                step=prepass + decode + merge)


class ClockSampler:
    """nvidia-smi clock / throttle samples while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4)
                          if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
    return world, rank, local


def reduce_max(x: float, world: int, device) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def aggregate(bytes_per_step_per_rank: float, steps: int, world: int, max_seconds: float):
    """Whole-job GB/s: bytes all ranks moved over the slowest rank's time."""
    return bytes_per_step_per_rank * steps * world / max_seconds / 1e9


def traffic_from_profiles(kernel_name: str, workload: str, plan: dict):
    """dram bytes per launch from a committed ncu summary, if it was taken on
    the current kernel source, for this workload and plan; else None."""
    p = os.path.join(ROOT, "profiles", "decode_traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p))
    if (d.get("kernel") != kernel_name or d.get("source_sha") != kernel_source_sha()
            or d.get("workload_name") != workload or d.get("plan") != plan):
        return None
    return d.get("dram_bytes_per_launch")


# the sources the fast decode kernel is compiled from (the planner, the API
# and the other kernels do not change its launches' traffic for a given plan);
# of fast_kernel.cuh only the device part, above its host section
KERNEL_SOURCES = ("fast_kernel.cuh", "pa_device.cuh", "pa_internal.h", "k_fast.cu")
HOST_SECTION = b"\n// ------------------------------------------------------------------- host\n"


def kernel_source_sha() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "paged_kv_attention_attn_gb300", "csrc")
    for f in KERNEL_SOURCES:
        text = open(os.path.join(csrc, f), "rb").read()
        if f == "fast_kernel.cuh" and HOST_SECTION in text:
            text = text[:text.index(HOST_SECTION)]
        h.update(text)
    return h.hexdigest()[:16]


# ------------------------------------------------------------------ oracle

def oracle_sample(case_host, spec, seqs, threads, group=None):
    """Times the float64 oracle on sequences `seqs` (full context; all query
    heads, or only those of K/V head `group`) of the workload; returns
    (seconds, algorithmic bytes: the K/V rows those heads need, once, and
    their outputs)."""
    import oracle
    k, v, bt, sl, q = case_host
    G = spec.hq // spec.hkv
    T = int(spec.extra.get("q_tokens", 1))
    heads = range(spec.hq) if group is None else range(group * G, (group + 1) * G)
    units = [(s * T + i, h) for s in seqs for i in range(T) for h in heads]
    t0 = time.perf_counter()
    oracle.decode(k, v, bt, sl, q, hkv=spec.hkv, block_size=spec.block_size,
                  k_type=spec.k_type, v_type=spec.v_type, units=units, n_threads=threads)
    dt = time.perf_counter() - t0
    krb, vrb = synth.row_bytes(spec.k_type, spec.d), synth.row_bytes(spec.v_type, spec.d)
    kv_heads = spec.hkv if group is None else 1
    nbytes = sum(spec.seq_lens[s] * kv_heads * (krb + vrb) for s in seqs)
    nbytes += len(units) * spec.d * 8
    return dt, nbytes


def host_copy(case):
    return [case.k_pool.cpu().numpy(), case.v_pool.cpu().numpy(),
            case.block_table.cpu().numpy(), case.seq_lens.cpu().numpy(), case.q.cpu().numpy()]


def run_reference(a, world, rank):
    """The reference arm: the oracle as it stands, on the host cores."""
    if rank != 0:
        return
    import oracle
    oracle.build()
    spec = WORKLOADS[a.workload]()
    dev = "cuda:0" if torch.cuda.is_available() else "cpu"
    case = synth.build_case(spec, seed=a.seed, device=dev)
    host = host_copy(case)
    del case
    threads = len(os.sched_getaffinity(0))
    # each step a bounded sample: the query heads of one K/V head of one
    # sequence, full context, taking the sequences and heads in turn
    def unit(i):
        return [i % spec.n_seqs], (i // spec.n_seqs) % spec.hkv
    for i in range(a.warmup):
        seqs, g = unit(i)
        oracle_sample(host, spec, seqs, threads, group=g)
    tot_t, tot_b = 0.0, 0
    for i in range(a.steps):
        seqs, g = unit(i)
        dt, nb = oracle_sample(host, spec, seqs, threads, group=g)
        tot_t += dt
        tot_b += nb
    gbs = tot_b / tot_t / 1e9
    G = spec.hq // spec.hkv
    sample = (f"per step the {G} query heads of one K/V head of one sequence, full context "
              f"({max(spec.seq_lens)} tokens at most), sequences and heads in turn")
    line = {"impl": "reference", "metric": METRIC, "value": gbs, "unit": "GB/s",
            "n_gpus": world, "steps": a.steps, "warmup": a.warmup,
            "ms_per_step": tot_t / a.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": a.workload, "sample": sample},
            "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------- ours

def time_append(spec, dev, stream, K, warmup):
    """The step before the decode: pa_append_kv of one new token per
    sequence of the workload (its types, heads and head size), K calls back
    to back between two events.  Separate one-block-per-sequence buffers;
    every call starts from its own copy of the lengths (mid-block, so no
    fresh block), so that each writes the same slot and the workload's own
    pools are left alone."""
    import ctypes
    import paged_kv_attention_attn_gb300 as pa
    S, B, hkv, d = spec.n_seqs, spec.block_size, spec.hkv, spec.d
    krb, vrb = synth.row_bytes(spec.k_type, d), synth.row_bytes(spec.v_type, d)
    kp = torch.zeros((S, B, hkv, krb), dtype=torch.uint8, device=dev)
    vp = torch.zeros((S, B, hkv, vrb), dtype=torch.uint8, device=dev)
    table = torch.arange(S, dtype=torch.int32, device=dev).view(S, 1)
    lens = torch.full((warmup + K, S), B // 2, dtype=torch.int32, device=dev)
    g = torch.Generator(device=dev).manual_seed(7)
    k_new = torch.randn((S, hkv, d), generator=g, device=dev)
    v_new = torch.randn((S, hkv, d), generator=g, device=dev)
    fresh = torch.zeros(S, dtype=torch.int32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    calls = [pa.AppendArgs(k_pool=kp.data_ptr(), v_pool=vp.data_ptr(), n_pool_blocks=S,
                           block_table=table.data_ptr(), table_stride=1,
                           seq_lens=lens[i].data_ptr(), k_new=k_new.data_ptr(),
                           v_new=v_new.data_ptr(), fresh_blocks=fresh.data_ptr(),
                           status=status.data_ptr(), n_seqs=S, hkv=hkv, d=d, block_size=B,
                           k_type=spec.k_type, v_type=spec.v_type) for i in range(warmup + K)]
    refs = [ctypes.byref(c) for c in calls]
    L, sh = pa.lib(), stream.cuda_stream
    for i in range(warmup):
        if L.pa_append_kv(refs[i], sh) != 0:
            raise RuntimeError(L.pa_last_error().decode())
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(warmup, warmup + K):
        L.pa_append_kv(refs[i], sh)
    e1.record(stream)
    torch.cuda.synchronize()
    assert pa.status_read(status) == 0
    us = e0.elapsed_time(e1) * 1e3 / K
    nbytes = S * hkv * d * 4 * 2 + S * hkv * (krb + vrb) + S * 4 * 3
    return {"us_per_call": us, "GB/s": nbytes / us / 1e3, "bytes_per_call": nbytes,
            "n_seqs": S, "calls": K,
            "how": "pa_append_kv of one token per sequence, back to back between two events"}


def check_status(pa, status, what: str):
    """The kernels' status word must still be clear after `what`: a corrupt
    table, a length past the plan or an abandoned pipeline wait during the
    timed steps makes the whole line invalid."""
    bits = pa.status_read(status)
    if bits:
        raise RuntimeError(f"status word 0x{bits:x} raised during {what}")


def run_ours(a, world, rank, local):
    import paged_kv_attention_attn_gb300 as pa
    from paged_kv_attention_attn_gb300 import build as pa_build
    pa_build.build()
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    spec = WORKLOADS[a.workload]()
    case = synth.build_case(spec, seed=a.seed + 1000 * rank, device=dev, chunk_blocks=1024)
    if a.workload.endswith("-contiguous"):
        case = synth.contiguous_twin(case)
    flags = pa.PA_FLAG_PLAIN if a.plain else 0
    pl = pa.plan(q_tokens=int(spec.extra.get("q_tokens", 1)),
                 seq_lens=spec.seq_lens, block_size=spec.block_size, hq=spec.hq, hkv=spec.hkv,
                 d=spec.d, k_type=spec.k_type, v_type=spec.v_type,
                 stream_ok=not a.unfused and not a.plain and a.stream == "on",
                 multi=not a.plain and a.multi == "on", force_parts=a.force_parts)
    ws = pa.workspace(pl, n_seqs=spec.n_seqs, hq=spec.hq, d=spec.d, device=dev)
    quantised = spec.k_type != synth.F16
    kv_bytes = (case.k_pool.numel() + case.v_pool.numel())
    # K/V under twice the L2: the steps take copies of the pools in turn, like
    # the layers of a model that share one block table and one query buffer,
    # so every step reads K/V that the L2 no longer holds (unless --flush on)
    n_layers = 1
    if a.flush == "auto" and kv_bytes < 2 * L2_BYTES:
        n_layers = min(MAX_LAYERS, -(-2 * L2_BYTES // kv_bytes) + 1)
    pools = [(case.k_pool, case.v_pool)] + [(case.k_pool.clone(), case.v_pool.clone())
                                            for _ in range(n_layers - 1)]

    def args_for(kp, vp, q):
        return pa.make_args(k_pool=kp, v_pool=vp, block_table=case.block_table,
                            seq_lens=case.seq_lens, q=q, ws=ws, hkv=spec.hkv,
                            block_size=spec.block_size, k_type=spec.k_type,
                            v_type=spec.v_type, flags=flags)
    layer_args = [args_for(kp, vp, case.q) for kp, vp in pools]
    layer_dec_args = [args_for(kp, vp, ws.q8_1 if quantised else case.q) for kp, vp in pools]
    args, dec_args = layer_args[0], layer_dec_args[0]
    kname = pa.decode_kernel_name(k_type=spec.k_type, v_type=spec.v_type, d=spec.d,
                                  hq=spec.hq, hkv=spec.hkv, block_size=spec.block_size,
                                  flags=flags)
    # the fused step of the fast kernel quantises the query itself: one launch
    in_kernel_q = (not a.unfused and quantised and kname == "fast_decode_kernel"
                   and not pl.stream)
    nb = algorithmic_bytes(spec, pl, fused=not a.unfused, in_kernel_q=in_kernel_q)
    stream = torch.cuda.current_stream()
    L = pa.lib()
    import ctypes
    p_plan = ctypes.byref(pl)
    sh = stream.cuda_stream

    fused = not a.unfused
    counters = ws.counters.data_ptr()
    p_layer_args = [ctypes.byref(x) for x in layer_args]
    p_layer_dec_args = [ctypes.byref(x) for x in layer_dec_args]
    layer = [0]  # the pool copy of the next step

    def step(ev0=None, ev1=None):
        p_step_args = p_layer_args[layer[0]]
        p_args = p_layer_dec_args[layer[0]]
        layer[0] = (layer[0] + 1) % n_layers
        if in_kernel_q or (pl.stream and fused):  # the public fused step
            if ev0 is not None:
                ev0.record(stream)
            rc = L.pa_decode_step_fused(p_step_args, p_plan, ws.q8_1.data_ptr(), counters, sh)
            if ev1 is not None:
                ev1.record(stream)
            return rc
        if quantised:
            L.pa_quantize_q(case.q.data_ptr(), ws.q8_1.data_ptr(), case.q.numel() // spec.d,
                            spec.d, sh)
        if ev0 is not None:
            ev0.record(stream)
        if fused:  # merge inside the decode launch
            rc = L.pa_decode_fused(p_args, p_plan, counters, sh)
        else:
            rc = L.pa_decode_partial(p_args, p_plan, sh)
        if ev1 is not None:
            ev1.record(stream)
        if not fused and not pl.direct:
            L.pa_merge(ws.part_o.data_ptr(), ws.part_ml.data_ptr(), case.seq_lens.data_ptr(),
                       ws.out.data_ptr(), spec.n_seqs, spec.hq, spec.d, p_plan, sh)
        return rc

    # correctness of the configuration before timing, then one step on every
    # pool copy (each copy's tensor maps are encoded once, as a model's layers
    # would have them after its first token), then the warm-up
    if step() != 0:
        raise RuntimeError(L.pa_last_error().decode())
    torch.cuda.synchronize()
    assert pa.status_read(ws.status) == 0
    for _ in range(n_layers - 1):
        step()
    for _ in range(a.warmup):
        step()
    torch.cuda.synchronize()

    K = a.steps
    # K/V smaller than twice the L2: a write of FLUSH_BYTES between steps
    # evicts it, and a read of the same buffer then writes the dirty lines
    # back, so that the step starts on a clean L2 holding none of its inputs;
    # only the steps themselves are timed (events around each)
    flush = a.flush == "on"
    flush_buf = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev) if flush else None

    def flush_l2(k):
        flush_buf.fill_(k & 0xFF)
        flush_buf.view(torch.int32).sum()
    # one launch per step and nothing between steps: the launches run back to
    # back and the decode time is the timed region over K; otherwise events
    # bracket the decode launch of every step
    per_launch = flush or not in_kernel_q
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(K)] if per_launch else None
    sevs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            for _ in range(K)] if flush else None
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    start.record(stream)
    for k in range(K):
        if flush:
            flush_l2(k)
            sevs[k][0].record(stream)
        if per_launch:
            step(*evs[k])
        else:
            step()
        if flush:
            sevs[k][1].record(stream)
    end.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    check_status(pa, ws.status, "the timed steps")
    total_ms = start.elapsed_time(end)
    step_ms = sum(e0.elapsed_time(e1) for e0, e1 in sevs) if flush else total_ms
    max_s = reduce_max(step_ms / 1e3, world, dev)
    value = aggregate(nb["step"], K, world, max_s)
    ms_per_step = max_s * 1e3 / K
    dec_avg_ms = (sum(e0.elapsed_time(e1) for e0, e1 in evs) / K if per_launch
                  else total_ms / K)
    peak, peak_kind = load_peaks()
    dec_achieved = nb["decode"] / (dec_avg_ms / 1e3) / 1e9

    # the spread of single steps: after the timed region, up to 200 more steps
    # each between two events (this pass feeds no other figure)
    n_dist = min(K, 200)
    dist_evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                for _ in range(n_dist)]
    for k in range(n_dist):
        if flush:
            flush_l2(k)
        dist_evs[k][0].record(stream)
        step()
        dist_evs[k][1].record(stream)
    torch.cuda.synchronize()
    check_status(pa, ws.status, "the single-step timing pass")
    dist = sorted(e0.elapsed_time(e1) * 1e3 for e0, e1 in dist_evs)
    step_dist = {"p10": dist[n_dist // 10], "median": dist[n_dist // 2],
                 "p90": dist[(9 * n_dist) // 10], "n": n_dist,
                 "how": "events around each step, after the timed region"}

    # end to end through the public C call with host buffers
    q_host = case.q.cpu().pin_memory()
    out_host = torch.empty(ws.out.shape, dtype=torch.float32).pin_memory()
    qdev = torch.empty_like(case.q)
    e2e_call = pa.decode_step_host if a.unfused else pa.decode_step_fused_host
    e2e_layer_args = [args_for(kp, vp, qdev) for kp, vp in pools]
    for k in range(a.warmup):
        e2e_call(q_host, out_host, e2e_layer_args[k % n_layers], ws)
    torch.cuda.synchronize()
    barrier(world)
    e2e_evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(K if flush else 1)]
    if flush:  # every call timed alone, after the L2 flush
        for k in range(K):
            flush_l2(k)
            e2e_evs[k][0].record(stream)
            e2e_call(q_host, out_host, e2e_layer_args[0], ws)
            e2e_evs[k][1].record(stream)
    else:
        e2e_evs[0][0].record(stream)
        for k in range(K):
            e2e_call(q_host, out_host, e2e_layer_args[k % n_layers], ws)
        e2e_evs[0][1].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    check_status(pa, ws.status, "the end-to-end steps")
    e2e_s = reduce_max(sum(e0.elapsed_time(e1) for e0, e1 in e2e_evs) / 1e3, world, dev)
    h2d = q_host.numel() * 4
    d2h = out_host.numel() * 4
    e2e = {"value": aggregate(nb["step"], K, world, e2e_s), "unit": "GB/s",
           "us_per_step": e2e_s * 1e6 / K, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}

    append = time_append(spec, dev, stream, min(K, 500), a.warmup)

    cpu = None
    if world == 1 and not a.no_cpu_baseline:
        host = host_copy(case)
        threads = len(os.sched_getaffinity(0))
        # a bounded sample of about CPU_SECONDS of oracle work: whole sequences,
        # every query head, full context, in turn until the time is spent
        dt = cb = 0.0
        done = []
        while dt < a.cpu_seconds and len(done) < 64 * spec.n_seqs:
            s = len(done) % spec.n_seqs
            t, b = oracle_sample(host, spec, [s], threads)
            dt, cb = dt + t, cb + b
            done.append(s)
        cpu = {"value": cb / dt / 1e9, "unit": "GB/s", "cores": threads, "kind": "oracle",
               "sample": f"{len(done)} whole sequences of the workload in turn (every query "
                         f"head, full context, {sum(spec.seq_lens[s] for s in done)} tokens), "
                         f"{dt:.1f} s wall"}

    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": K,
        "warmup": a.warmup, "ms_per_step": ms_per_step, "us_per_step": ms_per_step * 1e3,
        "step_us_dist": step_dist,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded N(0,1), see synth/)",
        "config": {"workload": a.workload, "batch": spec.n_seqs,
                   "context": max(spec.seq_lens), "d": spec.d, "hq": spec.hq,
                   "hkv": spec.hkv, "block_size": spec.block_size,
                   "kv_type": synth.TYPE_LABEL[spec.k_type],
                   "l2": (f"L2 flushed between steps by a {FLUSH_BYTES >> 20} MiB write and read; "
                          f"{nb['kv'] / 1e9:.3f} GB of K/V per step" if flush else
                          f"inputs larger than L2: {n_layers} copies of the K/V pools "
                          f"({n_layers * kv_bytes / 1e6:.0f} MB), one per step in turn, like the "
                          f"layers of a model sharing one block table; {nb['kv'] / 1e9:.4f} GB of "
                          f"K/V read per step" if n_layers > 1 else
                          f"inputs larger than L2: {nb['kv'] / 1e9:.3f} GB of K/V per step"
                          if kv_bytes >= L2_BYTES else
                          f"L2 not flushed: {nb['kv'] / 1e9:.3f} GB of K/V per step"),
                   "timing": ("events around each step" if per_launch else
                              "back-to-back launches, events around the timed region"),
                   "kernel": kname, "plan": pl.as_dict(),
                   "step": ("one launch: in-kernel q8_1 quantisation, decode, in-launch merge"
                            if in_kernel_q else
                            "stream plan: q8_1 pre-pass + stream-K decode with in-launch merges"
                            if pl.stream else
                            "multi-token plan: q8_1 pre-pass + decode of each sequence's tokens "
                            "together + merge kernel" if pl.multi else
                            "q8_1 pre-pass + decode with in-launch merge" if fused else
                            "q8_1 pre-pass + decode + merge kernel"),
                   "bytes_per_step": nb},
        "roofline": {"bound": "hbm", "achieved": dec_achieved, "peak": peak, "unit": "GB/s",
                     "frac": dec_achieved / peak, "peak_kind": peak_kind,
                     "kernel": kname, "kernel_us": dec_avg_ms * 1e3,
                     "bytes_per_launch": nb["decode"],
                     "traffic": traffic_from_profiles(kname, a.workload, pl.as_dict())},
        "cpu_baseline": cpu,
        "append": append,
        "e2e": e2e,
        "gpu_launches": K * (1 if in_kernel_q else
                             (2 if quantised else 1) +
                             (0 if (pl.direct or ((fused or pl.stream) and not pl.multi))
                              else 1)),
        "clocks": clk,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default=DEFAULT_WORKLOAD)
    ap.add_argument("--seed", type=int, default=2001)
    ap.add_argument("--plain", action="store_true", help="force the plain decode kernel")
    ap.add_argument("--unfused", action="store_true",
                    help="time the three-launch step (separate merge) instead of the fused one")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--flush", choices=["auto", "on", "off"], default="auto",
                    help="auto: K/V under 2 x L2 cycles through pool copies (one per step); "
                         "on: flush the L2 before every step instead; off: neither")
    ap.add_argument("--multi", choices=["on", "off"], default="on",
                    help="several query tokens per sequence: decode a sequence's tokens together")
    ap.add_argument("--stream", choices=["on", "off"], default="off",
                    help="let the planner return stream plans (batches wider than the grid)")
    ap.add_argument("--force-parts", type=int, default=0,
                    help="partitions per sequence instead of the planner's choice (profiling "
                         "cases: the benchmark's partition length on a smaller batch)")
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="oracle work timed for cpu_baseline (whole sequences in turn)")
    a = ap.parse_args()
    a.warmup = max(a.warmup, 3)
    world, rank, local = dist_setup()
    if a.impl == "reference":
        run_reference(a, world, rank)
    else:
        run_ours(a, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()

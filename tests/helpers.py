"""Shared helpers of the GPU tests: run the CUDA path through the C ABI and
evaluate the oracle on the same inputs (copied back to the host)."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import paged_kv_attention_attn_gb300 as pa
import synth

CANARY = 0x5A


def tol_for(spec) -> float:
    """The accuracy gate: max|err| <= tol * max|V| over the live rows."""
    return 2e-3 if spec.k_type == synth.F16 and spec.v_type == synth.F16 else 5e-3


def host_inputs(case):
    return [case.k_pool.cpu().numpy(), case.v_pool.cpu().numpy(),
            case.block_table.cpu().numpy(), case.seq_lens.cpu().numpy(), case.q.cpu().numpy()]


def oracle_kw(spec):
    return dict(hkv=spec.hkv, block_size=spec.block_size, k_type=spec.k_type,
                v_type=spec.v_type)


def oracle_out(case, units=None, **kw):
    return oracle.decode(*host_inputs(case), **oracle_kw(case.spec), units=units, **kw)


def oracle_vmax(case, units=None):
    return oracle.vmax(*host_inputs(case), **oracle_kw(case.spec), units=units)


def with_canary(t: torch.Tensor, extra_bytes: int = 4096):
    """A view of a larger uint8 buffer whose tail is a canary pattern; returns
    (view shaped like t, tail) so that a test can check nothing overran."""
    nbytes = t.numel() * t.element_size()
    buf = torch.full((nbytes + extra_bytes,), CANARY, dtype=torch.uint8, device=t.device)
    view = buf[:nbytes].view(t.dtype).view(t.shape)
    view.copy_(t)
    return view, buf[nbytes:]


def run(case, *, force_parts=0, flags=0, plan=None, canary=False, step=True, stream=None,
        fused=False, out_fill=None, q=None):
    """One decode step of `case` through the C ABI.  Returns (out float32
    tensor, workspace, plan, canary tails).  out_fill pre-fills the output
    buffer; q replaces the case's query."""
    sp = case.spec
    dev = case.k_pool.device
    pl = plan or pa.plan(seq_lens=sp.seq_lens, block_size=sp.block_size, hq=sp.hq, hkv=sp.hkv,
                         d=sp.d, k_type=sp.k_type, v_type=sp.v_type, force_parts=force_parts)
    ws = pa.workspace(pl, n_seqs=sp.n_seqs, hq=sp.hq, d=sp.d, device=dev)
    tails = []
    if out_fill is not None:
        ws.out.fill_(out_fill)
    if canary:
        ws.out, t1 = with_canary(ws.out)
        ws.part_o, t2 = with_canary(ws.part_o)
        ws.part_ml, t3 = with_canary(ws.part_ml)
        tails = [t1, t2, t3]
    args = pa.make_args(k_pool=case.k_pool, v_pool=case.v_pool, block_table=case.block_table,
                        seq_lens=case.seq_lens, q=case.q if q is None else q, ws=ws,
                        hkv=sp.hkv, block_size=sp.block_size, k_type=sp.k_type,
                        v_type=sp.v_type, flags=flags)
    if fused:
        pa.decode_step_fused(args, ws, stream=stream)
    elif step:
        pa.decode_step(args, ws, stream=stream)
    else:
        if sp.k_type != synth.F16:
            pa.quantize_q(case.q if q is None else q, out=ws.q8_1, stream=stream)
            args.q = ws.q8_1.data_ptr()
        pa.decode_partial(args, pl, stream=stream)
        if not pl.direct:
            pa.merge(ws, case.seq_lens, stream=stream)
    torch.cuda.synchronize()
    return ws.out, ws, pl, tails


def check_canaries(tails):
    for t in tails:
        assert bool((t == CANARY).all()), "a kernel wrote past the end of a buffer"


# worst max|err| / max|V| seen per workload label, printed at the end of the
# run (the margin of each gate: the gate is tol_for(spec))
MARGINS: dict = {}


def record_margin(label: str, err: float, vmax: float, tol: float):
    r = err / vmax if vmax > 0 else 0.0
    if r >= MARGINS.get(label, (-1.0, tol))[0]:
        MARGINS[label] = (r, tol)


def assert_close(case, got: torch.Tensor, ref: np.ndarray, vmax: float, units=None,
                 label: str | None = None):
    g = got.cpu().double().numpy()
    if units is not None:
        g = np.stack([g[s, h] for s, h in units])
    assert np.isfinite(g).all(), "non-finite output"
    err = float(np.abs(g - ref).max()) if g.size else 0.0
    bound = tol_for(case.spec) * vmax
    if label is not None:
        record_margin(label, err, vmax, tol_for(case.spec))
    assert err <= bound, f"{case.spec.name}: max|err| {err:.3e} > {bound:.3e}"
    return err

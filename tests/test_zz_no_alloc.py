"""The decode step for callers that cannot allocate device memory.

pa_decode_step_noalloc serves code that may not call cudaMalloc while it
decodes (a host callback, an engine whose device memory belongs to another
allocator or to a fixed budget): it keeps the q8_1 and partial buffers in
the library's own static device array instead of taking them from the
caller.  These tests call it through the C ABI and check that two calls in
a row -- the second on a different workload, so it reuses the array the
first one left dirty -- give the output of pa_decode_step within the
accuracy gate the other GPU tests use, and that a step too large for the
array is refused before anything runs.

This file is collected last on purpose."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import paged_kv_attention_attn_gb300 as pa
import synth
from tests import helpers as H

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def built():
    from paged_kv_attention_attn_gb300 import build
    build.build()
    oracle.build()


def _args(case, ws):
    sp = case.spec
    return pa.make_args(k_pool=case.k_pool, v_pool=case.v_pool, block_table=case.block_table,
                        seq_lens=case.seq_lens, q=case.q, ws=ws, hkv=sp.hkv,
                        block_size=sp.block_size, k_type=sp.k_type, v_type=sp.v_type)


def test_noalloc_step_matches_the_buffered_step_twice_in_a_row():
    specs = [synth.CaseSpec(seq_lens=[3000, 700, 0, 129], k_type=synth.Q4_0,
                            v_type=synth.Q4_0, junk=9, name="noalloc-q4_0"),
             synth.CaseSpec(seq_lens=[1500, 33], k_type=synth.F16, v_type=synth.Q8_0, d=128,
                            hq=32, hkv=8, block_size=32, junk=4, name="noalloc-f16-q8_0")]
    for i, spec in enumerate(specs):
        case = synth.build_case(spec, seed=2500 + i, device=DEV)
        ref_out, _, pl, _ = H.run(case, force_parts=6)
        assert not pl.direct
        ws = pa.workspace(pl, n_seqs=spec.n_seqs, hq=spec.hq, d=spec.d, device=DEV)
        ws.out.fill_(float("nan"))
        args = _args(case, ws)
        args.part_o = None   # not used by this entry point
        args.part_ml = None
        rc = pa.lib().pa_decode_step_noalloc(ctypes.byref(args), ctypes.byref(pl),
                                              torch.cuda.current_stream().cuda_stream)
        assert rc == pa.PA_OK, pa.lib().pa_last_error()
        torch.cuda.synchronize()
        assert pa.status_read(ws.status) == 0
        got = ws.out.cpu().double().numpy()
        ref = ref_out.cpu().double().numpy()
        assert np.isfinite(got).all()
        vmax = H.oracle_vmax(case)
        assert np.abs(got - ref).max() <= H.tol_for(spec) * vmax
        # and both stay within the gate against the oracle itself
        H.assert_close(case, ws.out, H.oracle_out(case), vmax)


def _noalloc_step(case, pl):
    """One pa_decode_step_noalloc call on a NaN-filled output; returns it."""
    sp = case.spec
    ws = pa.workspace(pl, n_seqs=sp.n_seqs, hq=sp.hq, d=sp.d, device=DEV)
    ws.out.fill_(float("nan"))
    args = _args(case, ws)
    args.part_o = None
    args.part_ml = None
    rc = pa.lib().pa_decode_step_noalloc(ctypes.byref(args), ctypes.byref(pl),
                                          torch.cuda.current_stream().cuda_stream)
    assert rc == pa.PA_OK, pa.lib().pa_last_error()
    torch.cuda.synchronize()
    assert pa.status_read(ws.status) == 0
    return ws.out


@pytest.mark.parametrize("what", ["wave-filling", "direct", "two-query-tokens"])
def test_noalloc_step_on_other_plans(what):
    """The plans the first test does not reach: a wave-filling plan (its
    leading rows direct, partials only for the split rows after them), a
    direct plan (no partials at all) and two query tokens per sequence.
    Each against pa_decode_step on the same plan, and against the oracle."""
    if what == "wave-filling":
        lens = [700, 650, 0, 700, 16, 690, 700, 680, 0, 700]
        spec = synth.CaseSpec(seq_lens=lens, k_type=synth.Q4_0, v_type=synth.Q4_0, junk=5,
                              name="noalloc-wavefill")
        pl = pa.plan(seq_lens=lens, block_size=16, hq=24, hkv=4, d=256, k_type=2, v_type=2,
                     sm_count=4, ctas_per_sm=1)
        assert pl.n_direct == 8 and not pl.direct
    elif what == "direct":
        lens = [300, 0, 1, 47]
        spec = synth.CaseSpec(seq_lens=lens, k_type=synth.Q8_0, v_type=synth.Q8_0, junk=2,
                              name="noalloc-direct")
        pl = pa.plan(seq_lens=lens, block_size=16, hq=24, hkv=4, d=256, k_type=1, v_type=1,
                     force_parts=1)
        assert pl.direct
    else:
        lens = [300, 41, 0, 520]
        spec = synth.CaseSpec(seq_lens=lens, k_type=synth.Q4_0, v_type=synth.Q4_0, junk=3,
                              extra={"q_tokens": 2}, name="noalloc-T2")
        pl = pa.plan(seq_lens=lens, block_size=16, hq=24, hkv=4, d=256, k_type=2, v_type=2,
                     force_parts=3, q_tokens=2)
        assert pl.q_tokens == 2 and not pl.direct
    case = synth.build_case(spec, seed=2600 + len(what), device=DEV)
    ref_out, _, _, _ = H.run(case, plan=pl)
    got = _noalloc_step(case, pl)
    vmax = H.oracle_vmax(case)
    g, r = got.cpu().double().numpy(), ref_out.cpu().double().numpy()
    assert np.isfinite(g).all()
    assert np.abs(g - r).max() <= H.tol_for(spec) * vmax
    H.assert_close(case, got, H.oracle_out(case), vmax)


def test_noalloc_refuses_bad_arguments_before_any_launch():
    """A call that the decode's own checks refuse (a misaligned pool) is
    refused before the query pre-pass runs: the output is left as it was
    and nothing was launched into the stream."""
    spec = synth.CaseSpec(seq_lens=[100, 37], k_type=synth.Q4_0, v_type=synth.Q4_0, junk=2,
                          name="noalloc-refused")
    case = synth.build_case(spec, seed=2700, device=DEV)
    pl = pa.plan(seq_lens=spec.seq_lens, block_size=16, hq=24, hkv=4, d=256, k_type=2,
                 v_type=2, force_parts=2)
    ws = pa.workspace(pl, n_seqs=spec.n_seqs, hq=spec.hq, d=spec.d, device=DEV)
    ws.out.fill_(3.0)
    args = _args(case, ws)
    args.k_pool = args.k_pool + 8  # not 16-byte aligned
    rc = pa.lib().pa_decode_step_noalloc(ctypes.byref(args), ctypes.byref(pl),
                                          torch.cuda.current_stream().cuda_stream)
    assert rc == pa.PA_ERR_INVALID
    assert b"pa_decode_step_noalloc" in pa.lib().pa_last_error()
    torch.cuda.synchronize()
    assert bool((ws.out == 3.0).all())


def test_noalloc_refuses_a_step_larger_than_its_scratch():
    # 64 sequences x 24 heads x 64 partitions x 256 dims of f16 partials is
    # about 50 MB, beyond the static array; nothing may be launched.
    S, hq, d = 64, 24, 256
    pl = pa.Plan(part_tokens=128, n_parts=64, direct=0, n_ctas=S * 64)
    out = torch.full((S, hq, d), 7.0, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    dummy = torch.zeros(1024, dtype=torch.uint8, device=DEV)
    args = pa.DecodeArgs(k_pool=dummy.data_ptr(), v_pool=dummy.data_ptr(), n_pool_blocks=1,
                         block_table=dummy.data_ptr(), table_stride=1,
                         seq_lens=dummy.data_ptr(), q=dummy.data_ptr(), scale=0.0625,
                         out=out.data_ptr(), status=status.data_ptr(), n_seqs=S, hq=hq,
                         hkv=4, d=d, block_size=16, k_type=pa.Q4_0, v_type=pa.Q4_0)
    rc = pa.lib().pa_decode_step_noalloc(ctypes.byref(args), ctypes.byref(pl), None)
    assert rc == pa.PA_ERR_RANGE
    assert b"pa_decode_step_noalloc" in pa.lib().pa_last_error()
    torch.cuda.synchronize()
    assert bool((out == 7.0).all())

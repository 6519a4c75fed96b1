"""Stream plans on the GPU: each CTA of the grid takes an equal range of the
rows' 16-token tiles, across row boundaries ("feat: add paged-attention
monolithic decode-only AR foundation", lucebox pull 555, Roadmap: the
stream-K decode kernel for ragged batches).  Small machines (a forced
sm_count) make batches wider than the grid at test sizes, so that rows are
cut by range boundaries (one partial per CTA, merged by the CTA that
completes the count), fall whole inside a range (output written directly),
or hold no token.  Every output against the oracle within the gate; the
paged layout equals its contiguous twin bit for bit; the counters return to
zero; repeated calls reuse them."""
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


def stream_plan(spec, sm_count, q_tokens=1):
    pl = pa.plan(seq_lens=spec.seq_lens, block_size=spec.block_size, hq=spec.hq, hkv=spec.hkv,
                 d=spec.d, k_type=spec.k_type, v_type=spec.v_type, sm_count=sm_count,
                 ctas_per_sm=1, q_tokens=q_tokens, stream_ok=True)
    assert pl.stream == 1 and not pl.direct and pl.n_direct == 0
    return pl


LENS = [700, 1500, 0, 33, 16, 2900, 1, 0, 480, 1200, 64, 999]


@pytest.mark.parametrize("t,d,hq,hkv,B", [
    (synth.Q4_0, 256, 24, 4, 16),
    (synth.Q8_0, 256, 24, 4, 32),
    (synth.F16, 256, 24, 4, 16),
    (synth.F16, 128, 32, 8, 32),
])
def test_stream_plan_matches_the_oracle(t, d, hq, hkv, B):
    spec = synth.CaseSpec(seq_lens=LENS, k_type=t, v_type=t, d=d, hq=hq, hkv=hkv, block_size=B,
                          junk=5, outliers=True, name=f"stream-{t}-{d}")
    case = synth.build_case(spec, seed=6100 + t + d, device=DEV)
    pl = stream_plan(spec, sm_count=5)
    out, ws, _, tails = H.run(case, plan=pl, fused=True, canary=True, out_fill=float("nan"))
    H.check_canaries(tails)
    assert pa.status_read(ws.status) == 0
    assert int(ws.counters.abs().sum()) == 0
    H.assert_close(case, out, H.oracle_out(case), H.oracle_vmax(case), label=spec.name)
    g = out.cpu()
    for s_, L in enumerate(LENS):
        if L == 0:
            assert bool((g[s_] == 0).all())


@pytest.mark.parametrize("sm_count", [3, 7, 11])
def test_stream_paged_equals_contiguous_and_calls_repeat(sm_count):
    """Different grids cut the rows at different places; for each, the paged
    pools and their contiguous twin give the same bits, and three calls in a
    row on one workspace give the same bits with the counters back at zero."""
    spec = synth.CaseSpec(seq_lens=LENS, k_type=synth.Q4_0, v_type=synth.Q4_0, junk=9,
                          name="stream-paged")
    case = synth.build_case(spec, seed=6200 + sm_count, device=DEV)
    pl = stream_plan(spec, sm_count)
    ref, ws, _, _ = H.run(case, plan=pl, fused=True)
    twin = synth.contiguous_twin(case)
    out2, _, _, _ = H.run(twin, plan=pl, fused=True)
    assert torch.equal(ref.view(torch.int32), out2.view(torch.int32))
    args = pa.make_args(k_pool=case.k_pool, v_pool=case.v_pool, block_table=case.block_table,
                        seq_lens=case.seq_lens, q=case.q, ws=ws, hkv=4, block_size=16,
                        k_type=spec.k_type, v_type=spec.v_type)
    for _ in range(3):
        ws.out.fill_(float("nan"))
        pa.decode_step_fused(args, ws)
        torch.cuda.synchronize()
        assert torch.equal(ws.out.view(torch.int32), ref.view(torch.int32))
        assert int(ws.counters.abs().sum()) == 0
    assert pa.status_read(ws.status) == 0
    H.assert_close(case, ref, H.oracle_out(case), H.oracle_vmax(case), label="stream-paged")


def test_stream_plan_with_two_query_tokens():
    lens = [300, 41, 0, 520, 777, 64, 1000]
    spec = synth.CaseSpec(seq_lens=lens, k_type=synth.Q4_0, v_type=synth.Q4_0, junk=3,
                          extra={"q_tokens": 2}, name="stream-T2")
    case = synth.build_case(spec, seed=6300, device=DEV)
    pl = stream_plan(spec, sm_count=4, q_tokens=2)
    out, ws, _, _ = H.run(case, plan=pl, fused=True)
    assert pa.status_read(ws.status) == 0
    H.assert_close(case, out, H.oracle_out(case), H.oracle_vmax(case), label="stream-T2")


def test_stream_plans_run_only_through_the_fused_calls():
    spec = synth.CaseSpec(seq_lens=[200, 300, 100], k_type=synth.Q4_0, v_type=synth.Q4_0,
                          name="stream-refused")
    case = synth.build_case(spec, seed=6400, device=DEV)
    pl = stream_plan(spec, sm_count=2)
    ws = pa.workspace(pl, n_seqs=3, hq=24, d=256, device=DEV)
    ws.out.fill_(5.0)
    L = pa.lib()
    sh = torch.cuda.current_stream().cuda_stream
    for flags in (0, pa.PA_FLAG_PLAIN):
        args = pa.make_args(k_pool=case.k_pool, v_pool=case.v_pool,
                            block_table=case.block_table, seq_lens=case.seq_lens, q=case.q,
                            ws=ws, hkv=4, block_size=16, k_type=2, v_type=2, flags=flags)
        assert L.pa_decode_partial(ctypes.byref(args), ctypes.byref(pl), sh) == pa.PA_ERR_INVALID
        assert L.pa_decode_step(ctypes.byref(args), ctypes.byref(pl), ws.q8_1.data_ptr(),
                                sh) == pa.PA_ERR_INVALID
    args.flags = pa.PA_FLAG_PLAIN
    assert L.pa_decode_fused(ctypes.byref(args), ctypes.byref(pl), ws.counters.data_ptr(),
                             sh) == pa.PA_ERR_INVALID
    assert L.pa_merge(ws.part_o.data_ptr(), ws.part_ml.data_ptr(), case.seq_lens.data_ptr(),
                      ws.out.data_ptr(), 3, 24, 256, ctypes.byref(pl), sh) == pa.PA_ERR_INVALID
    torch.cuda.synchronize()
    assert bool((ws.out == 5.0).all())

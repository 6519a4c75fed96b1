"""Several query tokens per sequence (a verify window or prompt chunk over the
paged cache, TensorFold pull 1418, What): token i of sequence s sits at
position L - T + i and attends causally to the keys 0 .. L - T + i.  The CUDA
path is checked against the oracle's causal form for both kernels, every
mode, plain and mixed K/V types, and the paged layout against a contiguous
layout of the same cache bit for bit."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_attention_attn_gb300 as pa
import synth
from tests import helpers as H

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
KERNELS = {"fast": 0, "plain": pa.PA_FLAG_PLAIN}


@pytest.fixture(scope="module", autouse=True)
def built():
    from paged_kv_attention_attn_gb300 import build
    build.build()
    oracle.build()


def _q4(spec, T, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(spec.n_seqs, T, spec.hq, spec.d, generator=g).to(DEV)


def _plan(spec, T, force):
    return pa.plan(seq_lens=spec.seq_lens, block_size=spec.block_size, hq=spec.hq,
                   hkv=spec.hkv, d=spec.d, k_type=spec.k_type, v_type=spec.v_type,
                   force_parts=force, q_tokens=T)


def _oracle(case, q4):
    k, v, bt, sl, _ = H.host_inputs(case)
    return oracle.decode(k, v, bt, sl, q4.cpu().numpy(), **H.oracle_kw(case.spec))


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("kt,vt", [(synth.F16, synth.F16), (synth.Q4_0, synth.Q4_0),
                                   (synth.Q8_0, synth.Q4_0)])
@pytest.mark.parametrize("T", [2, 5])
def test_several_query_tokens_match_the_oracle(kernel, kt, vt, T):
    spec = synth.CaseSpec(seq_lens=[700, 3, 0, 130, 16], k_type=kt, v_type=vt, junk=3)
    case = synth.build_case(spec, seed=3300 + 10 * kt + vt, device=DEV)
    q4 = _q4(spec, T, 3400 + T)
    ref = _oracle(case, q4)
    vmax = H.oracle_vmax(case)
    outs = []
    for force in (0, 1, 4):
        pl = _plan(spec, T, force)
        assert pl.q_tokens == T
        for fused in (False, True):
            out, ws, _, _ = H.run(case, plan=pl, q=q4, flags=KERNELS[kernel], fused=fused,
                                  out_fill=float("nan"))
            assert pa.status_read(ws.status) == 0
            assert tuple(out.shape) == (spec.n_seqs, T, spec.hq, spec.d)
            H.assert_close(case, out, ref, vmax)
            outs.append(out.clone())
            assert int(ws.counters.abs().sum()) == 0
    # the fused and separate merges agree bit for bit in each plan
    for a, b in zip(outs[0::2], outs[1::2]):
        assert torch.equal(a.view(torch.int32), b.view(torch.int32))


@pytest.mark.parametrize("kernel", KERNELS)
def test_several_query_tokens_paged_equals_contiguous(kernel):
    spec = synth.CaseSpec(seq_lens=[1000, 257, 64], k_type=synth.Q4_0, v_type=synth.Q4_0,
                          junk=6)
    case = synth.build_case(spec, seed=3500, device=DEV)
    twin = synth.contiguous_twin(case)
    q4 = _q4(spec, 4, 3501)
    pl = _plan(spec, 4, 3)
    a, _, _, _ = H.run(case, plan=pl, q=q4, flags=KERNELS[kernel], fused=True)
    b, _, _, _ = H.run(twin, plan=pl, q=q4, flags=KERNELS[kernel], fused=True)
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))


# ---------------------------------------------------- multi-token plans
#
# The T tokens of a sequence decoded together (T * G query columns of each
# K/V head per tile, a warp pair per head splitting the head dimension).

def _mt_plan(spec, T, force=0, sm_count=None):
    kw = dict(seq_lens=spec.seq_lens, block_size=spec.block_size, hq=spec.hq, hkv=spec.hkv,
              d=spec.d, k_type=spec.k_type, v_type=spec.v_type, force_parts=force, q_tokens=T,
              multi=True)
    if sm_count is not None:
        kw.update(sm_count=sm_count, ctas_per_sm=1)
    pl = pa.plan(**kw)
    assert pl.multi == 1 and pl.q_tokens == T
    return pl


@pytest.mark.parametrize("T,hq,hkv,B", [(2, 24, 4, 16), (4, 24, 4, 16), (3, 24, 4, 32),
                                        (6, 8, 2, 16), (3, 8, 1, 16)])
@pytest.mark.parametrize("force", [0, 1, 5])
def test_multi_token_plan_matches_the_oracle(T, hq, hkv, B, force):
    """Every mode (auto, direct, partitioned), every entry point (three
    launches, fused), lengths shorter than the window and empty sequences:
    against the oracle's causal form, and the fused step equal to the
    three-launch step bit for bit."""
    lens = [700, 3, 0, 130, 16, 2, 1999]
    spec = synth.CaseSpec(seq_lens=lens, k_type=synth.Q4_0, v_type=synth.Q4_0, hq=hq, hkv=hkv,
                          block_size=B, junk=4, outliers=True)
    case = synth.build_case(spec, seed=3600 + T + hkv, device=DEV)
    q4 = _q4(spec, T, 3700 + T)
    ref, vmax = _oracle(case, q4), H.oracle_vmax(case)
    pl = _mt_plan(spec, T, force)
    assert pl.direct == (force == 1)
    a, ws_a, _, tails = H.run(case, plan=pl, q=q4, canary=True, out_fill=float("nan"))
    b, ws_b, _, _ = H.run(case, plan=pl, q=q4, fused=True, out_fill=float("nan"))
    H.check_canaries(tails)
    assert pa.status_read(ws_a.status) == 0 and pa.status_read(ws_b.status) == 0
    H.assert_close(case, a, ref, vmax, label=f"multi-token T{T} G{hq // hkv}")
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))


def test_multi_token_plan_against_the_row_plan_and_contiguous():
    """The multi-token plan and the per-row plan of the same window agree
    within the gate; the paged layout equals its contiguous twin bit for
    bit; a small machine gives many partitions per sequence."""
    spec = synth.CaseSpec(seq_lens=[3000, 1025, 64, 4100], k_type=synth.Q4_0, v_type=synth.Q4_0,
                          junk=6)
    case = synth.build_case(spec, seed=3800, device=DEV)
    q4 = _q4(spec, 4, 3801)
    pl = _mt_plan(spec, 4, sm_count=20)
    assert not pl.direct and pl.n_parts >= 4
    a, _, _, _ = H.run(case, plan=pl, q=q4, fused=True)
    twin = synth.contiguous_twin(case)
    b, _, _, _ = H.run(twin, plan=pl, q=q4, fused=True)
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))
    row, _, _, _ = H.run(case, plan=_plan(spec, 4, 0), q=q4, fused=True)
    vmax = H.oracle_vmax(case)
    assert float((a - row).abs().max()) <= H.tol_for(spec) * vmax
    H.assert_close(case, a, _oracle(case, q4), vmax, label="multi-token 4 x ragged")


def test_multi_token_plans_need_the_fast_kernel():
    spec = synth.CaseSpec(seq_lens=[200, 300], k_type=synth.Q4_0, v_type=synth.Q4_0)
    case = synth.build_case(spec, seed=3900, device=DEV)
    q4 = _q4(spec, 2, 3901)
    pl = _mt_plan(spec, 2)
    with pytest.raises(pa.PAError) as e:
        H.run(case, plan=pl, q=q4, flags=pa.PA_FLAG_PLAIN)
    assert e.value.code == pa.PA_ERR_INVALID

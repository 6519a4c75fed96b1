"""GPU parity at the workloads' full sizes, in the launch configuration the
benchmark times (planner defaults): every (sequence, head) output against the
oracle (for the 10 GiB pool, every head of four sequences), element by
element within the gate, plus layout invariants that hold at any size.

Workloads ("feat: add paged-attention monolithic decode-only AR foundation",
lucebox pull 555, Benchmark results; "fix(paged-attention): use 64-bit pool
offsets in the fused decode kernels", mlxcel issue 2153, Acceptance
Criteria): uniform Q4_0 batches up to 8 x 131072; the ragged 128K + 7 x 8K
batch against its padded contiguous layout; the dtype sweep with outliers and
its short ragged batch; the 163,840-block f16 pool past 2^32 elements; and a
131,073-block pool whose only non-zero data sits past the 2^32-element
offset."""
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


def oracle_for(case, seqs=None, units=None):
    """The oracle on a compact host copy of `seqs` (default: every sequence)
    of the case: (reference rows, their max|V|, the units in the case's
    numbering).  units: (sequence, head) pairs of the listed sequences,
    default every head of each."""
    seqs = list(range(case.spec.n_seqs)) if seqs is None else sorted(seqs)
    small = synth.gather_sequences(case, seqs)
    remap = {s: i for i, s in enumerate(seqs)}
    if units is None:
        units = [(s, h) for s in seqs for h in range(case.spec.hq)]
    su = [(remap[s], h) for s, h in units]
    return H.oracle_out(small, units=su), H.oracle_vmax(small, units=su), units


def check_against(case, out, ref, label):
    """Every listed output element against the oracle, within the gate."""
    r, vmax, units = ref
    return H.assert_close(case, out, r, vmax, units=units, label=label)


@pytest.mark.parametrize("batch,ctx", [(1, 4096), (2, 32768), (8, 131072)])
def test_uniform_q4_0(batch, ctx):
    """Every (sequence, head) output of both kernels against the oracle, and
    the one-launch fused step equal to the three-launch step bit for bit."""
    case = synth.build_case(synth.uniform_spec(batch, ctx), seed=2000 + batch, device=DEV)
    ref = oracle_for(case)
    for kernel, flags in KERNELS.items():
        out, ws, pl, _ = H.run(case, flags=flags)
        assert pa.status_read(ws.status) == 0
        check_against(case, out, ref, f"{case.spec.name} {kernel}")
        fused, ws2, _, _ = H.run(case, flags=flags, fused=True)
        assert torch.equal(fused.view(torch.int32), out.view(torch.int32))
        assert int(ws2.counters.abs().sum()) == 0


def test_ragged_paged_equals_padded_contiguous():
    case = synth.build_case(synth.ragged_spec(), seed=3000, device=DEV)
    ref = oracle_for(case)
    # the padded 8 x 131072 contiguous layout of the same rows
    twin = synth.contiguous_twin(case)
    assert twin.k_pool.shape[0] == 8 * 8192
    for kernel, flags in KERNELS.items():
        out, ws, pl, _ = H.run(case, flags=flags)
        assert pa.status_read(ws.status) == 0
        out2, _, pl2, _ = H.run(twin, flags=flags)
        assert pl.as_dict() == pl2.as_dict()
        assert torch.equal(out.view(torch.int32), out2.view(torch.int32))
        check_against(case, out, ref, f"{case.spec.name} {kernel}")


@pytest.mark.parametrize("t", [synth.F16, synth.Q8_0, synth.Q4_0])
@pytest.mark.parametrize("short", [False, True])
def test_dtype_sweep(t, short):
    case = synth.build_case(synth.dtype_sweep_spec(t, short=short), seed=4000 + t, device=DEV)
    ref = oracle_for(case)
    for kernel, flags in KERNELS.items():
        out, ws, pl, tails = H.run(case, flags=flags, canary=True)
        assert pa.status_read(ws.status) == 0
        H.check_canaries(tails)
        check_against(case, out, ref, f"{case.spec.name} {kernel}")


def test_large_pool_past_2_to_the_32():
    """Every head of the four sequences holding the most blocks at ids >=
    131,072 (past 2^32 elements of the slab), one of them the sequence that
    holds the pool's final block, on both kernels."""
    spec = synth.large_pool_spec()
    assert spec.n_pool_blocks * spec.block_size * spec.hkv * spec.d > 2**32
    case = synth.build_case(spec, seed=5000, device=DEV, chunk_blocks=1024)
    bt = case.block_table.cpu()
    high = (bt >= 131072).sum(dim=1)
    assert int(high.sum()) > 0 and bool((bt == spec.n_pool_blocks - 1).any())
    s_last = int(((bt == spec.n_pool_blocks - 1).any(dim=1)).nonzero()[0])
    order = [int(s) for s in torch.argsort(high, descending=True)]
    seqs = [s_last] + [s for s in order if s != s_last][:3]
    ref = oracle_for(case, seqs=seqs)
    for kernel, flags in KERNELS.items():
        out, ws, pl, _ = H.run(case, flags=flags)
        assert pa.status_read(ws.status) == 0
        check_against(case, out, ref, f"{spec.name} {kernel} (4 sequences)")
    del case
    torch.cuda.empty_cache()


@pytest.mark.parametrize("kernel", KERNELS)
def test_data_only_past_the_wrap_point(kernel):
    """131,073 blocks of [32, 8, 128] f16; every block is zero except the
    last, which starts at element 2^32.  A sequence of 40 tokens reads the
    last block then block 0; an offset wrapped to 32 bits would read block 0
    for the first 32 tokens and give a different output."""
    B, hkv, d, hq = 32, 8, 128, 32
    n = 131_073
    k_pool = torch.zeros((n, B, hkv, 2 * d), dtype=torch.uint8, device=DEV)
    v_pool = torch.zeros_like(k_pool)
    g = torch.Generator(device=DEV).manual_seed(77)
    x = torch.randn((B, hkv, d), generator=g, device=DEV)
    k_pool[n - 1] = synth.encode(x, synth.F16)
    v_pool[n - 1] = synth.encode(torch.randn((B, hkv, d), generator=g, device=DEV), synth.F16)
    table = torch.tensor([[n - 1, 0]], dtype=torch.int32, device=DEV)
    lens = torch.tensor([40], dtype=torch.int32, device=DEV)
    q = torch.randn((1, hq, d), generator=g, device=DEV)
    spec = synth.CaseSpec(seq_lens=[40], d=d, hq=hq, hkv=hkv, block_size=B, k_type=synth.F16,
                          v_type=synth.F16, n_pool_blocks=n)
    case = synth.Case(spec=spec, k_pool=k_pool, v_pool=v_pool, block_table=table,
                      seq_lens=lens, q=q, seed=77)
    for force in (0, 2):
        out, ws, _, _ = H.run(case, force_parts=force, flags=KERNELS[kernel])
        assert pa.status_read(ws.status) == 0
        small = synth.gather_sequences(case, [0])
        ref = H.oracle_out(small)
        H.assert_close(case, out, ref, H.oracle_vmax(small))
        # the wrapped reading differs from it by far more than the gate
        wrapped = small.k_pool.clone()
        wrapped[0] = 0
        wv = small.v_pool.clone()
        wv[0] = 0
        bad = oracle.decode(wrapped.numpy(), wv.numpy(), small.block_table.numpy(),
                            small.seq_lens.numpy(), small.q.numpy(), hkv=hkv, block_size=B,
                            k_type=0, v_type=0)
        assert np.abs(bad - ref).max() > 0.05
    del k_pool, v_pool, case
    torch.cuda.empty_cache()

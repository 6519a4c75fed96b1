"""GPU parity tests at oracle-sized inputs: the CUDA path through the C ABI
against the float64 oracle, element by element.

Covered: the q8_1 pre-pass bit for bit; the tiny F16 workload; every K/V
type pair in direct, forced-single, planner and forced-many modes, on both
kernels; block-boundary lengths including empty sequences; paged ==
contiguous bit for bit under a shuffled table with poisoned junk blocks;
run-to-run determinism; the corrupt-table guard; a red control; the 64-bit
row offsets bit for bit; the merge kernel alone; the host-buffer step."""
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
TYPES = [synth.F16, synth.Q8_0, synth.Q4_0]


@pytest.fixture(scope="module", autouse=True)
def built():
    from paged_kv_attention_attn_gb300 import build
    build.build()
    oracle.build()


def test_quantize_q_bit_exact():
    g = torch.Generator().manual_seed(3)
    x = torch.randn(37, 256, generator=g) * torch.rand(37, 1, generator=g) * 50
    x[0, :32] = 0.0                                 # zero block
    x[1, :32] = torch.arange(32) - 15.5             # ties after scaling
    x[2, 0], x[2, 1:32] = 127.0, 2.5                # d = 1: x/d ties round away
    x[3, 32:64] = 1e-30                             # tiny values
    got = pa.quantize_q(x.to(DEV)).cpu().numpy()
    ref = oracle.quantize_q8_1(x.numpy())
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("force", [0, 1, 7])
def test_tiny_f16(kernel, force):
    case = synth.build_case(synth.tiny_spec(), seed=1000, device=DEV)
    out, ws, pl, tails = H.run(case, force_parts=force, flags=KERNELS[kernel], canary=True)
    assert pa.status_read(ws.status) == 0
    H.check_canaries(tails)
    H.assert_close(case, out, H.oracle_out(case), H.oracle_vmax(case))


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("kt", TYPES)
@pytest.mark.parametrize("vt", TYPES)
@pytest.mark.parametrize("force", [0, 1, 5])
def test_type_pairs_and_modes(kernel, kt, vt, force):
    spec = synth.CaseSpec(seq_lens=[600, 37, 0, 257], k_type=kt, v_type=vt, junk=11,
                          outliers=True, name=f"pair-{kt}{vt}")
    case = synth.build_case(spec, seed=1100 + 3 * kt + vt, device=DEV)
    out, ws, pl, tails = H.run(case, force_parts=force, flags=KERNELS[kernel], canary=True)
    assert pa.status_read(ws.status) == 0
    H.check_canaries(tails)
    H.assert_close(case, out, H.oracle_out(case), H.oracle_vmax(case))


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("shape", [dict(d=128, hq=32, hkv=8, block_size=32),
                                   dict(d=256, hq=8, hkv=8, block_size=16),
                                   dict(d=128, hq=8, hkv=1, block_size=16)])
def test_other_head_shapes(kernel, shape):
    spec = synth.CaseSpec(seq_lens=[333, 64, 1], k_type=synth.F16, v_type=synth.F16, junk=5,
                          **shape)
    case = synth.build_case(spec, seed=1200, device=DEV)
    for force in (0, 3):
        out, ws, _, _ = H.run(case, force_parts=force, flags=KERNELS[kernel])
        H.assert_close(case, out, H.oracle_out(case), H.oracle_vmax(case))


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("hq,hkv", [(8, 8), (8, 2), (32, 4), (64, 8)])
def test_q4_0_other_head_shapes(kernel, hq, hkv):
    """Q4_0 (D = 256) beyond the 24 / 4 heads of the benchmark: one query head
    per K/V head, groups narrower than the tensor-core tile (dead query
    columns), and rows whose query items outnumber the CTA's threads (hq * 16
    > warps * 32: the CTA-wide query quantisation of the 32-token path takes
    several rounds).  Against the oracle, and the one-launch step (query
    quantised in the kernel) equal to the three-launch step (q8_1 pre-pass)
    bit for bit."""
    spec = synth.CaseSpec(seq_lens=[700, 33, 0, 2000], k_type=synth.Q4_0, v_type=synth.Q4_0,
                          hq=hq, hkv=hkv, junk=5, outliers=True)
    case = synth.build_case(spec, seed=1250 + hq + hkv, device=DEV)
    ref, vmax = H.oracle_out(case), H.oracle_vmax(case)
    for force in (0, 3):
        a, ws, _, tails = H.run(case, force_parts=force, flags=KERNELS[kernel], canary=True)
        H.check_canaries(tails)
        assert pa.status_read(ws.status) == 0
        H.assert_close(case, a, ref, vmax, label=f"Q4_0 hq{hq} hkv{hkv} force{force}")
        b, ws_b, _, _ = H.run(case, force_parts=force, flags=KERNELS[kernel], fused=True)
        assert pa.status_read(ws_b.status) == 0
        assert torch.equal(a.view(torch.int32), b.view(torch.int32))


@pytest.mark.parametrize("kernel", KERNELS)
def test_q4_0_32_token_blocks(kernel):
    """Q4_0 with 32-token blocks: the two 16-token halves of a 32-token tile
    come from one block (partitions start on block boundaries).  Against the
    oracle in every mode, and the one-launch step equal to the three-launch
    step bit for bit."""
    spec = synth.CaseSpec(seq_lens=[1000, 17, 0, 64, 333], k_type=synth.Q4_0,
                          v_type=synth.Q4_0, block_size=32, junk=7, outliers=True)
    case = synth.build_case(spec, seed=1280, device=DEV)
    ref, vmax = H.oracle_out(case), H.oracle_vmax(case)
    for force in (0, 1, 5):
        a, ws, _, tails = H.run(case, force_parts=force, flags=KERNELS[kernel], canary=True)
        H.check_canaries(tails)
        assert pa.status_read(ws.status) == 0
        H.assert_close(case, a, ref, vmax, label=f"Q4_0 B32 force{force}")
        b, _, _, _ = H.run(case, force_parts=force, flags=KERNELS[kernel], fused=True)
        assert torch.equal(a.view(torch.int32), b.view(torch.int32))


@pytest.mark.parametrize("kernel", KERNELS)
def test_block_boundary_lengths(kernel):
    lens = [0, 1, 15, 16, 17, 31, 32, 33, 200, 127, 128, 129, 255, 256, 257]
    spec = synth.CaseSpec(seq_lens=lens, k_type=synth.Q4_0, v_type=synth.Q4_0, junk=13)
    case = synth.build_case(spec, seed=1300, device=DEV)
    for force in (0, 2):
        out, ws, _, tails = H.run(case, force_parts=force, flags=KERNELS[kernel], canary=True)
        H.check_canaries(tails)
        got = out.cpu().numpy()
        assert np.all(got[0] == 0.0)  # empty sequence
        H.assert_close(case, out, H.oracle_out(case), H.oracle_vmax(case))


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("t", TYPES)
def test_paged_equals_contiguous_bit_for_bit(kernel, t):
    spec = synth.CaseSpec(seq_lens=[1000, 77, 300, 16], k_type=t, v_type=t, junk=40)
    case = synth.build_case(spec, seed=1400 + t, device=DEV)
    twin = synth.contiguous_twin(case)
    for force in (0, 1, 4):
        a, _, pa_, _ = H.run(case, force_parts=force, flags=KERNELS[kernel])
        b, _, pb_, _ = H.run(twin, force_parts=force, flags=KERNELS[kernel])
        assert pa_.as_dict() == pb_.as_dict()
        assert torch.equal(a.view(torch.int32), b.view(torch.int32))


@pytest.mark.parametrize("kernel", KERNELS)
def test_run_to_run_deterministic(kernel):
    spec = synth.CaseSpec(seq_lens=[2000, 500], k_type=synth.Q4_0, v_type=synth.Q4_0, junk=3)
    case = synth.build_case(spec, seed=1500, device=DEV)
    a, _, _, _ = H.run(case, flags=KERNELS[kernel])
    b, _, _, _ = H.run(case, flags=KERNELS[kernel])
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))


@pytest.mark.parametrize("kernel", KERNELS)
def test_corrupt_table_is_guarded(kernel):
    spec = synth.CaseSpec(seq_lens=[100, 50], k_type=synth.Q4_0, v_type=synth.Q4_0, junk=2)
    case = synth.build_case(spec, seed=1600, device=DEV)
    case.block_table[0, 3] = case.n_blocks + 1000   # past the pool
    case.block_table[1, 0] = -7
    out, ws, _, _ = H.run(case, flags=KERNELS[kernel])
    assert pa.status_read(ws.status) & pa.PA_STATUS_CORRUPT_TABLE
    assert pa.status_read(ws.status) == 0  # the read above reset it
    assert torch.isfinite(out).all()


@pytest.mark.parametrize("kernel", KERNELS)
def test_red_control_wrong_in_range_table_fails_parity(kernel):
    """A table whose first entry names a later block of the sequence: the
    kernel reads valid data and sets no status bit, but the comparison with
    the oracle (given the true table) must fail."""
    spec = synth.CaseSpec(seq_lens=[160], k_type=synth.F16, v_type=synth.F16, junk=4)
    case = synth.build_case(spec, seed=1700, device=DEV)
    ref, vmax = H.oracle_out(case), H.oracle_vmax(case)
    case.block_table[0, 0] = case.block_table[0, 5]
    out, ws, _, _ = H.run(case, flags=KERNELS[kernel])
    assert pa.status_read(ws.status) == 0
    with pytest.raises(AssertionError):
        H.assert_close(case, out, ref, vmax)


def test_row_offsets_bit_exact():
    spec = synth.CaseSpec(seq_lens=[70, 0, 33, 16], k_type=synth.Q4_0, v_type=synth.Q4_0,
                          junk=6, block_size=32)
    case = synth.build_case(spec, seed=1800, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    rb = pa.row_bytes(synth.Q4_0, spec.d)
    maxt = 80
    got = pa.debug_row_offsets(case.block_table, case.seq_lens, max_tokens=maxt,
                               block_size=32, hkv=spec.hkv, row_bytes_=rb,
                               n_pool_blocks=case.n_blocks, status=status).cpu().numpy()
    bt = case.block_table.cpu().numpy()
    for s, L in enumerate(spec.seq_lens):
        for t in range(maxt):
            for g in range(spec.hkv):
                v = int(got[s, t, g]) & 0xFFFFFFFFFFFFFFFF
                if t < L:
                    assert v == oracle.row_offset(int(bt[s, t // 32]), t % 32, g, 32, spec.hkv, rb)
                else:
                    assert v == 0xFFFFFFFFFFFFFFFF


def test_row_offsets_past_2_to_the_32():
    """Offsets of blocks around the 2^32-element wrap point of a [32, 8, 128]
    f16 pool, computed by the kernels' device routine, equal the oracle's; no
    pool memory is needed for this."""
    B, hkv, d = 32, 8, 128
    rb = 2 * d
    ids = torch.tensor([[0, 131071, 131072, 131073, 163839, 2**31 - 1]], dtype=torch.int32)
    lens = torch.tensor([6 * B], dtype=torch.int32)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    got = pa.debug_row_offsets(ids.to(DEV), lens.to(DEV), max_tokens=6 * B, block_size=B,
                               hkv=hkv, row_bytes_=rb, n_pool_blocks=2**31,
                               status=status).cpu().numpy()
    for t in range(6 * B):
        for g in range(hkv):
            want = oracle.row_offset(int(ids[0, t // B]), t % B, g, B, hkv, rb)
            assert int(got[0, t, g]) == want
    assert int(got[0, 2 * B, 0]) == 2**32 * 2  # element offset exactly 2^32


def test_merge_kernel_against_oracle_merge():
    rng = np.random.default_rng(5)
    S, hq, d, P, part = 3, 4, 128, 6, 64
    lens = [P * part, 2 * part + 5, 0]
    o = rng.standard_normal((S, hq, P, d)).astype(np.float16)
    ml = np.zeros((S, hq, P, 2), dtype=np.float32)
    ml[..., 0] = rng.uniform(-20, 20, (S, hq, P))
    ml[..., 1] = rng.uniform(0.5, 40, (S, hq, P))
    ml[0, 1, 2, 1] = 0.0               # a dead partition inside a live sequence
    o[0, 1, 2] = np.float16(np.nan)    # whose o must not be read
    pl = pa.Plan(part_tokens=part, n_parts=P, direct=0, n_ctas=S * P)
    ws = pa.workspace(pl, n_seqs=S, hq=hq, d=d, device=DEV)
    ws.part_o.copy_(torch.from_numpy(o))
    ws.part_ml.copy_(torch.from_numpy(ml))
    seq_lens = torch.tensor(lens, dtype=torch.int32, device=DEV)
    pa.merge(ws, seq_lens)
    torch.cuda.synchronize()
    got = ws.out.cpu().double().numpy().reshape(S * hq, d)
    n_live = np.repeat([-(-L // part) for L in lens], hq).astype(np.int32)
    ref = oracle.merge(o.view(np.uint16).reshape(S * hq, P, d), ml.reshape(S * hq, P, 2), n_live)
    assert np.isfinite(got).all()
    np.testing.assert_allclose(got, ref, rtol=0, atol=2e-5 * np.abs(o.astype(np.float64)[
        np.isfinite(o.astype(np.float64))]).max())


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("q_pinned", [True, False])
def test_host_buffer_step_equals_device_step(kernel, q_pinned):
    """The host-buffer steps give the device step's bits, for a partitioned
    and a direct plan.  Page-locked q_host is staged by a kernel, pageable
    q_host copied.  Page-locked out_host: the kernels store into it and the
    device out buffer is left as it was; pageable out_host: the device out
    buffer is copied back."""
    spec = synth.CaseSpec(seq_lens=[700, 90], k_type=synth.Q4_0, v_type=synth.Q4_0, junk=3)
    case = synth.build_case(spec, seed=1900, device=DEV)
    q_host = case.q.cpu().pin_memory() if q_pinned else case.q.cpu().clone()
    for force in (0, 1):
        dev_out, _, _, _ = H.run(case, force_parts=force, flags=KERNELS[kernel])
        pl = pa.plan(seq_lens=spec.seq_lens, block_size=16, hq=24, hkv=4, d=256,
                     k_type=spec.k_type, v_type=spec.v_type, force_parts=force)
        ws = pa.workspace(pl, n_seqs=2, hq=24, d=256, device=DEV)
        qdev = torch.empty_like(case.q)
        args = pa.make_args(k_pool=case.k_pool, v_pool=case.v_pool,
                            block_table=case.block_table, seq_lens=case.seq_lens, q=qdev,
                            ws=ws, hkv=4, block_size=16, k_type=spec.k_type,
                            v_type=spec.v_type, flags=KERNELS[kernel])
        for out_host, direct_store in ((torch.empty(2, 24, 256).pin_memory(), True),
                                       (torch.empty(2, 24, 256), False)):
            for call in (pa.decode_step_host, pa.decode_step_fused_host):
                out_host.fill_(float("nan"))
                ws.out.fill_(float("nan"))
                call(q_host, out_host, args, ws)
                torch.cuda.synchronize()
                assert torch.equal(out_host.view(torch.int32), dev_out.cpu().view(torch.int32))
                assert bool(ws.out.isnan().all()) == direct_store
                assert torch.equal(qdev.view(torch.int32), case.q.view(torch.int32))


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("t", [synth.Q4_0, synth.F16])
def test_host_buffer_steps_back_to_back(kernel, t):
    """Host-buffer steps queued back to back, each with its own query in
    page-locked memory and the same device query buffer: a step's query is
    staged while the previous step's kernels finish, so each step must still
    see its own query.  Each output equals the device step of its query bit
    for bit."""
    spec = synth.CaseSpec(seq_lens=[3000, 700, 90, 5000], k_type=t, v_type=t, junk=3)
    case = synth.build_case(spec, seed=1950 + t, device=DEV)
    g = torch.Generator().manual_seed(1951)
    qs = [torch.randn(tuple(case.q.shape), generator=g) for _ in range(6)]
    refs = [H.run(case, q=q.to(DEV), flags=KERNELS[kernel], fused=True)[0].cpu() for q in qs]
    pl = pa.plan(seq_lens=spec.seq_lens, block_size=16, hq=24, hkv=4, d=256, k_type=t, v_type=t)
    ws = pa.workspace(pl, n_seqs=spec.n_seqs, hq=24, d=256, device=DEV)
    qdev = torch.empty_like(case.q)
    args = pa.make_args(k_pool=case.k_pool, v_pool=case.v_pool, block_table=case.block_table,
                        seq_lens=case.seq_lens, q=qdev, ws=ws, hkv=4, block_size=16, k_type=t,
                        v_type=t, flags=KERNELS[kernel])
    q_hosts = [q.pin_memory() for q in qs]
    outs = [torch.full(tuple(case.q.shape), float("nan")).pin_memory() for _ in qs]
    for rep in range(3):
        for q_host, out_host in zip(q_hosts, outs):
            pa.decode_step_fused_host(q_host, out_host, args, ws)
        torch.cuda.synchronize()
        assert pa.status_read(ws.status) == 0
        for out_host, ref in zip(outs, refs):
            assert torch.equal(out_host.view(torch.int32), ref.view(torch.int32))


# ------------------------------------------------------------- fused merge

@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("t", TYPES)
@pytest.mark.parametrize("force", [0, 1, 6, 60])
def test_fused_merge_equals_separate_merge(kernel, t, force):
    """The in-launch merge runs the same merge arithmetic as pa_merge, so the
    two paths give the same bits; the counters are left at zero.  force=60
    makes 47 partitions of the longest sequence: a two-pass plan, which on the
    fast kernel stages its merge rows in shared memory (the short sequences
    of the same plan merge in one pass)."""
    spec = synth.CaseSpec(seq_lens=[1500, 33, 0, 700, 16], k_type=t, v_type=t, junk=7,
                          outliers=True)
    case = synth.build_case(spec, seed=2600 + t, device=DEV)
    a, _, pl, _ = H.run(case, force_parts=force, flags=KERNELS[kernel])
    b, ws, pl2, tails = H.run(case, force_parts=force, flags=KERNELS[kernel], fused=True,
                              canary=True)
    H.check_canaries(tails)
    assert pl.as_dict() == pl2.as_dict()
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))
    assert int(ws.counters.abs().sum()) == 0
    assert pa.status_read(ws.status) == 0
    H.assert_close(case, b, H.oracle_out(case), H.oracle_vmax(case))


@pytest.mark.parametrize("kernel", KERNELS)
def test_fused_merge_repeated_calls_reuse_counters(kernel):
    spec = synth.CaseSpec(seq_lens=[2000, 300], k_type=synth.Q4_0, v_type=synth.Q4_0, junk=3)
    case = synth.build_case(spec, seed=2700, device=DEV)
    ref, _, pl, _ = H.run(case, force_parts=5, flags=KERNELS[kernel])
    ws = pa.workspace(pl, n_seqs=2, hq=24, d=256, device=DEV)
    args = pa.make_args(k_pool=case.k_pool, v_pool=case.v_pool, block_table=case.block_table,
                        seq_lens=case.seq_lens, q=case.q, ws=ws, hkv=4, block_size=16,
                        k_type=spec.k_type, v_type=spec.v_type, flags=KERNELS[kernel])
    for _ in range(3):
        ws.out.fill_(float("nan"))
        pa.decode_step_fused(args, ws)
        torch.cuda.synchronize()
        assert torch.equal(ws.out.view(torch.int32), ref.view(torch.int32))
        assert int(ws.counters.abs().sum()) == 0


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("t", [synth.F16, synth.Q4_0])
def test_every_output_row_is_written(kernel, t):
    """Every mode of the step writes every output row: the rows of empty
    sequences are zero whatever the buffer held before (NaN here)."""
    spec = synth.CaseSpec(seq_lens=[0, 900, 0, 0, 40, 0], k_type=t, v_type=t, junk=3)
    case = synth.build_case(spec, seed=2800 + t, device=DEV)
    ref, vmax = H.oracle_out(case), H.oracle_vmax(case)
    for force in (0, 1, 5):
        for fused in (False, True):
            out, ws, pl, _ = H.run(case, force_parts=force, flags=KERNELS[kernel], fused=fused,
                                   out_fill=float("nan"))
            assert pa.status_read(ws.status) == 0
            g = out.cpu()
            for s_, L in enumerate(spec.seq_lens):
                if L == 0:
                    assert bool((g[s_] == 0).all()), (force, fused, s_)
            H.assert_close(case, out, ref, vmax)
            assert int(ws.counters.abs().sum()) == 0


def _adversarial_query(q):
    """Blocks that exercise the q8_1 rounding: all zero, exact ties (the
    scale is a power of two so x / d is k + 1/2 exactly), a signed zero, tiny
    and large magnitudes, and values at the clamp."""
    q = q.clone()
    q[0, 0, :32] = 0.0
    ties = torch.tensor([15.875] + [(k + 0.5) * 0.125 for k in range(-15, 15)] + [-15.875])
    q[0, 1, 32:64] = ties
    q[0, 2, 64:96] = ties.flip(0) * -4.0
    q[0, 3, :32] = -0.0
    q[0, 3, 5] = 2.0 ** -20
    q[1, 4, :] = q[1, 4, :] * 1e-4
    q[1, 5, :] = q[1, 5, :] * 40.0
    return q


def test_in_kernel_query_quantisation_matches_the_pre_pass():
    """The fused step of the fast kernel quantises the query itself with the
    pre-pass's arithmetic; its output equals the three-launch step's bit for
    bit, also on blocks built to expose rounding differences."""
    spec = synth.CaseSpec(seq_lens=[700, 333], k_type=synth.Q4_0, v_type=synth.Q4_0, junk=2)
    case = synth.build_case(spec, seed=2900, device=DEV)
    q = _adversarial_query(case.q)
    for force in (0, 1, 4):
        a, _, _, _ = H.run(case, force_parts=force, q=q)
        b, ws, _, _ = H.run(case, force_parts=force, q=q, fused=True, out_fill=float("nan"))
        assert pa.status_read(ws.status) == 0
        assert torch.equal(a.view(torch.int32), b.view(torch.int32)), force
    # and the pre-pass itself codes these blocks as the oracle does
    got = pa.quantize_q(q).cpu().numpy().reshape(-1, 8 * 36)
    ref = oracle.quantize_q8_1(q.cpu().numpy().reshape(-1, 256))
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("fused", [False, True])
def test_lengths_past_the_plan_are_flagged_and_stay_in_bounds(kernel, fused):
    """Device lengths that the plan does not cover (a sequence longer than
    n_parts * part_tokens; more partitions than the grid has CTAs) set
    PA_STATUS_LEN_OVER_PLAN, and nothing is written past the buffers."""
    spec = synth.CaseSpec(seq_lens=[3000, 1000], k_type=synth.Q4_0, v_type=synth.Q4_0, junk=2)
    case = synth.build_case(spec, seed=3100, device=DEV)
    for planned in ([1000, 1000], [1000, 100]):
        pl = pa.plan(seq_lens=planned, block_size=16, hq=24, hkv=4, d=256, k_type=synth.Q4_0,
                     v_type=synth.Q4_0, force_parts=4)
        assert not pl.direct
        out, ws, _, tails = H.run(case, plan=pl, flags=KERNELS[kernel], fused=fused,
                                  canary=True)
        H.check_canaries(tails)
        assert pa.status_read(ws.status) & pa.PA_STATUS_LEN_OVER_PLAN, planned
    # lengths inside the plan raise nothing
    out, ws, _, _ = H.run(case, force_parts=4, flags=KERNELS[kernel], fused=fused)
    assert pa.status_read(ws.status) == 0


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("force", [6, 8, 24, 60])
@pytest.mark.parametrize("no_wait", [False, True])
def test_fused_merge_waits_for_every_partition(kernel, force, no_wait):
    """The in-launch merge of a sequence must start only after its last
    partition (one pass) or last group (two passes) is written.  Many
    sequences with many partitions each, several launches in a row: any
    early merge shows up as a difference from the separate merge.  On the
    fast kernel the one-pass plans whose grid is resident at once merge
    cooperatively (every CTA of a sequence waits for the others and merges
    its share of the rows); no_wait makes every such wait give up at once, so
    the CTA that completes each count merges the rows of the others."""
    spec = synth.CaseSpec(seq_lens=[4000 - 37 * i for i in range(24)], k_type=synth.Q4_0,
                          v_type=synth.Q4_0, junk=5)
    case = synth.build_case(spec, seed=3200 + force, device=DEV)
    ref, _, pl, _ = H.run(case, force_parts=force, flags=KERNELS[kernel])
    ws = pa.workspace(pl, n_seqs=spec.n_seqs, hq=24, d=256, device=DEV)
    flags = KERNELS[kernel] | (pa.PA_FLAG_MERGE_NO_WAIT if no_wait else 0)
    args = pa.make_args(k_pool=case.k_pool, v_pool=case.v_pool, block_table=case.block_table,
                        seq_lens=case.seq_lens, q=case.q, ws=ws, hkv=4, block_size=16,
                        k_type=spec.k_type, v_type=spec.v_type, flags=flags)
    for _ in range(6):
        ws.out.fill_(float("nan"))
        pa.decode_step_fused(args, ws)
        torch.cuda.synchronize()
        assert torch.equal(ws.out.view(torch.int32), ref.view(torch.int32))
        assert int(ws.counters.abs().sum()) == 0


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("t", TYPES)
def test_sharp_softmax(kernel, t):
    """Query norms six times the unit draws: scores spread over tens of log2
    units, so nearly every probability, and its product with a V block scale,
    lies deep below the maximum, many in the f16 subnormal range."""
    spec = synth.CaseSpec(seq_lens=[3000, 517, 16], k_type=t, v_type=t, outliers=True,
                          name=f"sharp-{t}")
    case = synth.build_case(spec, seed=1400 + t, device=DEV)
    case.q.mul_(6.0)
    out, ws, pl, _ = H.run(case, flags=KERNELS[kernel])
    assert pa.status_read(ws.status) == 0
    H.assert_close(case, out, H.oracle_out(case), H.oracle_vmax(case))


@pytest.mark.parametrize("t", TYPES)
def test_long_single_partition(t):
    """One partition of 40000 tokens: every warp of the fast kernel folds
    more than 800 tiles into one accumulator."""
    spec = synth.CaseSpec(seq_lens=[40000], k_type=t, v_type=t, outliers=True,
                          name=f"long-{t}")
    case = synth.build_case(spec, seed=1500 + t, device=DEV)
    out, ws, pl, _ = H.run(case, force_parts=1)
    assert pa.status_read(ws.status) == 0
    H.assert_close(case, out, H.oracle_out(case), H.oracle_vmax(case))


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("t", TYPES)
def test_wave_filling_plan(kernel, t):
    """A batch wider than the machine (here 4 slots, so that a few rows make
    it wide) and about even, so that it would run direct: 10 rows = 2 waves +
    2, so the first 8 rows run direct and the last 2 are split in halves to
    fill the third wave.  Empty rows sit on both sides of the cut.  Fused and
    separate merges, against the oracle; the fused merge gives the separate
    merge's bits and leaves the counters at zero."""
    lens = [700, 650, 0, 700, 16, 690, 700, 680, 0, 700]
    spec = synth.CaseSpec(seq_lens=lens, k_type=t, v_type=t, junk=5, outliers=True,
                          name=f"wavefill-{t}")
    case = synth.build_case(spec, seed=3400 + t, device=DEV)
    pl = pa.plan(seq_lens=lens, block_size=16, hq=24, hkv=4, d=256, k_type=t, v_type=t,
                 sm_count=4, ctas_per_sm=1)
    assert pl.n_direct == 8 and not pl.direct and pl.n_parts >= 2
    ref, vmax = H.oracle_out(case), H.oracle_vmax(case)
    a, ws_a, _, _ = H.run(case, plan=pl, flags=KERNELS[kernel], canary=True)
    b, ws_b, _, tails = H.run(case, plan=pl, flags=KERNELS[kernel], fused=True, canary=True)
    H.check_canaries(tails)
    assert pa.status_read(ws_a.status) == 0 and pa.status_read(ws_b.status) == 0
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))
    assert int(ws_b.counters.abs().sum()) == 0
    H.assert_close(case, b, ref, vmax)


@pytest.mark.parametrize("kernel", KERNELS)
def test_wave_filling_plan_two_pass(kernel):
    """41 rows of 5000 tokens on 40 slots: 40 direct rows, and the last row in
    40 partitions of 128 tokens, merged in two passes (the staged merge on
    the fast kernel)."""
    lens = [5000] * 41
    spec = synth.CaseSpec(seq_lens=lens, k_type=synth.Q4_0, v_type=synth.Q4_0, junk=3,
                          name="wavefill-2pass")
    case = synth.build_case(spec, seed=3450, device=DEV)
    pl = pa.plan(seq_lens=lens, block_size=16, hq=24, hkv=4, d=256, k_type=2, v_type=2,
                 sm_count=40, ctas_per_sm=1)
    assert (pl.n_direct, pl.n_parts, pl.part_tokens) == (40, 40, 128)
    a, _, _, _ = H.run(case, plan=pl, flags=KERNELS[kernel])
    b, ws, _, _ = H.run(case, plan=pl, flags=KERNELS[kernel], fused=True)
    assert pa.status_read(ws.status) == 0
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))
    assert int(ws.counters.abs().sum()) == 0
    units = [(s, h) for s in (0, 17, 39, 40) for h in (0, 5, 23)]
    H.assert_close(case, b, H.oracle_out(case, units=units), H.oracle_vmax(case, units=units),
                   units=units)


@pytest.mark.parametrize("kernel", KERNELS)
def test_wave_filling_plan_multitoken(kernel):
    """The same cut over query rows: 5 sequences x 2 query tokens = 10 rows on
    4 slots, 8 direct rows and 2 split ones (the last sequence's tokens)."""
    lens = [300, 41, 0, 520, 777]
    spec = synth.CaseSpec(seq_lens=lens, k_type=synth.Q4_0, v_type=synth.Q4_0, junk=3,
                          extra={"q_tokens": 2}, name="wavefill-T2")
    case = synth.build_case(spec, seed=3500, device=DEV)
    pl = pa.plan(seq_lens=lens, block_size=16, hq=24, hkv=4, d=256, k_type=2, v_type=2,
                 sm_count=4, ctas_per_sm=1, q_tokens=2)
    assert pl.n_direct == 8 and not pl.direct
    out, ws, _, _ = H.run(case, plan=pl, flags=KERNELS[kernel], fused=True)
    assert pa.status_read(ws.status) == 0
    H.assert_close(case, out, H.oracle_out(case), H.oracle_vmax(case))

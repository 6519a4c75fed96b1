"""Pins for the oracle's pool-row quantisers and its model of the K/V append
step.  The quantisers are checked against synth's encoders (separate code,
torch) byte for byte, and against closed forms of the ggml convention; the
append model against the allocator model and a direct encode."""
import numpy as np
import pytest
import torch

import oracle
import synth
from oracle import append_model, pool_model


def _synth_bytes(x: np.ndarray, type_: int) -> np.ndarray:
    return synth.encode(torch.from_numpy(x), type_).numpy()


@pytest.mark.parametrize("type_", [synth.F16, synth.Q8_0, synth.Q4_0])
def test_quantize_row_equals_the_independent_encoder(type_):
    g = torch.Generator().manual_seed(11)
    x = synth.source_values(g, (400, 256), "cpu", outliers=True).numpy() * 3
    x[0, :32] = 0.0                                   # zero block
    x[0, 32:64] = 0.0
    x[0, 32] = -0.0                                   # zero block led by -0
    x[1, :32] = np.round(x[1, :32])                   # integer values: exact ties
    x[2, 5], x[2, 9] = 4.0, -4.0                      # equal magnitudes
    x[3, :] *= 1e-3
    ref = _synth_bytes(x, type_)
    got = np.stack([oracle.quantize_row(type_, r) for r in x])
    assert np.array_equal(got, ref)


def test_q4_0_closed_form_grid():
    # x_j = (j - 8) / 2 for j < 16: m = -4 (first largest), d = 0.5, nib_j = j
    x = np.concatenate([(np.arange(16) - 8) * 0.5, (np.arange(16) - 8) * 0.25]).astype(np.float32)
    row = oracle.quantize_row(oracle.Q4_0, x)
    assert np.frombuffer(row[:2].tobytes(), np.float16)[0] == 0.5
    lo = row[2:18] & 0xF
    hi = row[2:18] >> 4
    assert list(lo) == list(range(16))
    assert list(hi) == [int(np.floor(v * 2 + 8.5)) for v in x[16:]]
    assert np.array_equal(oracle.dequant_row(oracle.Q4_0, row, 32)[:16], x[:16])


def test_q4_0_first_of_equal_magnitudes_sets_the_sign():
    x = np.zeros(32, dtype=np.float32)
    x[2], x[5] = 3.0, -3.0
    row = oracle.quantize_row(oracle.Q4_0, x)
    d = float(np.frombuffer(row[:2].tobytes(), np.float16)[0])
    assert d == -0.375                                # m = +3 (index 2), d = m / -8
    nib = [(row[2 + j % 16] >> (4 * (j // 16))) & 0xF for j in range(32)]
    assert nib[2] == 0 and nib[5] == 15 and nib[0] == 8   # +3 -> 0, -3 -> 16 clamped, 0 -> 8


def test_q8_0_ties_round_away_and_zero_block():
    x = np.zeros(32, dtype=np.float32)
    x[0] = 127.0                                      # d = 1, id = 1
    x[1:5] = [2.5, -2.5, 0.5, -126.5]
    row = oracle.quantize_row(oracle.Q8_0, x)
    q = row[2:].view(np.int8)
    assert list(q[:5]) == [127, 3, -3, 1, -127]
    z = oracle.quantize_row(oracle.Q8_0, np.zeros(32, np.float32))
    assert not z.any()


def _state(S, stride, n_blocks, B, hkv, d, kt, vt):
    rk, rv = oracle.row_bytes(kt, d), oracle.row_bytes(vt, d)
    pool_k = np.full((n_blocks, B, hkv, rk), 0xFF, np.uint8)
    pool_v = np.full((n_blocks, B, hkv, rv), 0xFF, np.uint8)
    table = np.full((S, stride), -1, np.int32)
    lens = np.zeros(S, np.int32)
    return pool_k, pool_v, table, lens


@pytest.mark.parametrize("B", [16, 32])
def test_append_model_builds_what_a_direct_encode_gives(B):
    """Appending tokens one step at a time, with fresh blocks from the
    allocator model at every block boundary, leaves every token's rows where
    the table says and equal to a direct encode of that token."""
    S, hkv, d, kt, vt, steps = 3, 2, 64, synth.Q4_0, synth.Q8_0, 70
    n_blocks = S * (steps // B + 2)
    pool_k, pool_v, table, lens = _state(S, steps // B + 1, n_blocks, B, hkv, d, kt, vt)
    alloc = pool_model.PoolModel(n_blocks)
    rng = np.random.default_rng(5)
    hist_k = rng.standard_normal((steps, S, hkv, d)).astype(np.float32)
    hist_v = rng.standard_normal((steps, S, hkv, d)).astype(np.float32)
    starts = [0, 5, 17]                               # sequences join at different steps
    for t in range(steps):
        fresh = np.full(S, -1, np.int32)
        snapshot = lens.copy()
        for s in range(S):
            if t >= starts[s] and lens[s] % B == 0:
                rc, hs = alloc.alloc(1)
                assert rc == pool_model.OK
                fresh[s] = pool_model.PoolModel.block_of(hs[0])
        act = [s for s in range(S) if t >= starts[s]]
        sub = np.array(act)
        t_sub, l_sub = table[sub], lens[sub]
        st = append_model.append(pool_k, pool_v, t_sub, l_sub, hist_k[t, sub], hist_v[t, sub],
                                 fresh[sub], block_size=B, k_type=kt, v_type=vt)
        table[sub], lens[sub] = t_sub, l_sub
        assert st == 0
        assert np.array_equal(lens[sub], snapshot[sub] + 1)
    for s in range(S):
        for pos in range(int(lens[s])):
            blk, slot = table[s, pos // B], pos % B
            t = starts[s] + pos
            for g in range(hkv):
                assert np.array_equal(pool_k[blk, slot, g], oracle.quantize_row(kt, hist_k[t, s, g]))
                assert np.array_equal(pool_v[blk, slot, g], oracle.quantize_row(vt, hist_v[t, s, g]))
    used = table[table >= 0]
    assert len(set(used.tolist())) == used.size       # no block shared


def test_append_model_flags_a_full_table_and_a_bad_block():
    pool_k, pool_v, table, lens = _state(2, 1, 4, 16, 1, 32, synth.F16, synth.F16)
    lens[:] = [16, 0]                                 # sequence 0 has no table entry left
    kv = np.ones((2, 1, 32), np.float32)
    st = append_model.append(pool_k, pool_v, table, lens, kv, kv, np.array([0, 9], np.int32),
                             block_size=16, k_type=synth.F16, v_type=synth.F16)
    assert st == append_model.STATUS_APPEND_RANGE | append_model.STATUS_CORRUPT_TABLE
    assert list(lens) == [16, 0] and (table == -1).all() and (pool_k == 0xFF).all()

"""Pins for the oracle's attention, partition/merge and table walk.

The oracle is compared with torch's scaled_dot_product_attention in float64
(a library routine) on rows the oracle itself dequantised, with closed-form
special cases, with invariants (any block-table permutation with poisoned
junk blocks; one partition vs many) and with red controls that a correct
checker must flag."""
import numpy as np
import pytest
import scipy.special
import torch

import oracle
import synth


def _np(case):
    return (case.k_pool.numpy(), case.v_pool.numpy(), case.block_table.numpy(),
            case.seq_lens.numpy(), case.q.numpy())


def oracle_decode(case, **kw):
    k, v, bt, sl, q = _np(case)
    sp = case.spec
    return oracle.decode(k, v, bt, sl, q, hkv=sp.hkv, block_size=sp.block_size,
                         k_type=sp.k_type, v_type=sp.v_type, **kw)


def dequant_seq(case, s, side):
    """float64 [L, hkv, D] rows of sequence s, read through its table."""
    sp = case.spec
    pool = (case.k_pool if side == "k" else case.v_pool).numpy()
    t_ = sp.k_type if side == "k" else sp.v_type
    L = sp.seq_lens[s]
    out = np.zeros((L, sp.hkv, sp.d))
    for t in range(L):
        blk = int(case.block_table[s, t // sp.block_size])
        for g in range(sp.hkv):
            out[t, g] = oracle.dequant_row(t_, pool[blk, t % sp.block_size, g], sp.d)
    return out


def query_rows(case, s):
    sp = case.spec
    q = case.q[s].numpy()
    if sp.k_type == synth.F16:
        return q.astype(np.float64)
    blocks = oracle.quantize_q8_1(q)
    return np.stack([oracle.dequant_q8_1_row(blocks[h], sp.d) for h in range(sp.hq)])


def sdpa_reference(case):
    """torch SDPA in float64; GQA by repeating each K/V head G times."""
    sp = case.spec
    G = sp.hq // sp.hkv
    out = np.zeros((sp.n_seqs, sp.hq, sp.d))
    for s in range(sp.n_seqs):
        if sp.seq_lens[s] == 0:
            continue
        k = torch.from_numpy(dequant_seq(case, s, "k")).permute(1, 0, 2)  # [hkv, L, D]
        v = torch.from_numpy(dequant_seq(case, s, "v")).permute(1, 0, 2)
        k = k.repeat_interleave(G, dim=0)
        v = v.repeat_interleave(G, dim=0)
        q = torch.from_numpy(query_rows(case, s)).unsqueeze(1)  # [hq, 1, D]
        o = torch.nn.functional.scaled_dot_product_attention(
            q.unsqueeze(0), k.unsqueeze(0), v.unsqueeze(0), scale=1.0 / np.sqrt(sp.d))
        out[s] = o[0, :, 0, :].numpy()
    return out


SMALL = [
    dict(seq_lens=[200], k_type=synth.F16, v_type=synth.F16, n_pool_blocks=32),
    dict(seq_lens=[37, 1, 0, 64], k_type=synth.Q4_0, v_type=synth.Q4_0, junk=5, d=128,
         hq=8, hkv=2),
    dict(seq_lens=[50, 17], k_type=synth.Q8_0, v_type=synth.Q4_0, junk=3, d=64, hq=6, hkv=3,
         block_size=32),
    dict(seq_lens=[33, 16], k_type=synth.F16, v_type=synth.Q8_0, junk=2, d=32, hq=4, hkv=1,
         outliers=True),
]


@pytest.mark.parametrize("kw", SMALL)
def test_oracle_matches_torch_sdpa(kw):
    case = synth.build_case(synth.CaseSpec(**kw), seed=11)
    got = oracle_decode(case)
    ref = sdpa_reference(case)
    assert np.all(np.isfinite(got))
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


def test_oracle_red_control_wrong_table_is_detected():
    """A table whose first entry names a later block of the same sequence
    (an in-range but wrong table) must not agree with the reference."""
    case = synth.build_case(synth.CaseSpec(seq_lens=[64], k_type=synth.F16, v_type=synth.F16,
                                           junk=4, d=64, hq=4, hkv=2), seed=5)
    ref = sdpa_reference(case)
    bad = case.block_table.clone()
    bad[0, 0] = bad[0, 2]
    k, v, _, sl, q = _np(case)
    got = oracle.decode(k, v, bad.numpy(), sl, q, hkv=2, block_size=16, k_type=0, v_type=0)
    assert np.abs(got - ref).max() > 1e-3


def test_oracle_corrupt_table_refused():
    case = synth.build_case(synth.CaseSpec(seq_lens=[40], k_type=synth.Q4_0, v_type=synth.Q4_0,
                                           junk=1, d=64, hq=2, hkv=1), seed=6)
    k, v, bt, sl, q = _np(case)
    bt = bt.copy()
    bt[0, 1] = case.n_blocks  # one past the pool
    with pytest.raises(oracle.OracleError) as e:
        oracle.decode(k, v, bt, sl, q, hkv=1, block_size=16, k_type=2, v_type=2)
    assert e.value.rc == oracle.OR_ERR_CORRUPT
    bt[0, 1] = -3
    with pytest.raises(oracle.OracleError):
        oracle.decode(k, v, bt, sl, q, hkv=1, block_size=16, k_type=2, v_type=2)


def test_paged_equals_contiguous_under_permutation_with_junk():
    spec = synth.CaseSpec(seq_lens=[100, 45, 16, 3], k_type=synth.Q4_0, v_type=synth.Q8_0,
                          junk=9, d=64, hq=8, hkv=2)
    case = synth.build_case(spec, seed=21)
    twin = synth.contiguous_twin(case)
    a = oracle_decode(case)
    b = oracle_decode(twin)
    assert np.array_equal(a, b)  # same arithmetic in the same order: identical
    assert np.all(np.isfinite(a))  # no poisoned byte was read


@pytest.mark.parametrize("part", [32, 64, 96])
def test_partitioned_equals_single_pass(part):
    spec = synth.CaseSpec(seq_lens=[257, 31, 0, 128], k_type=synth.Q4_0, v_type=synth.Q4_0,
                          junk=3, d=64, hq=4, hkv=1, outliers=True)
    case = synth.build_case(spec, seed=4)
    a = oracle_decode(case)
    b = oracle_decode(case, part_tokens=part)
    np.testing.assert_allclose(b, a, rtol=1e-12, atol=1e-13)


def _f16_rows(x):
    return synth.encode(torch.from_numpy(np.asarray(x, dtype=np.float32)), synth.F16)


def test_closed_form_length_one_returns_the_v_row():
    case = synth.build_case(synth.CaseSpec(seq_lens=[1], k_type=synth.Q4_0, v_type=synth.Q4_0,
                                           junk=2, d=64, hq=4, hkv=2), seed=8)
    got = oracle_decode(case)
    v = dequant_seq(case, 0, "v")
    for h in range(4):
        assert np.array_equal(got[0, h], v[0, h // 2])


def test_closed_form_equal_keys_give_the_mean_of_v():
    spec = synth.CaseSpec(seq_lens=[40], k_type=synth.F16, v_type=synth.F16, junk=1, d=32,
                          hq=2, hkv=1)
    case = synth.build_case(spec, seed=9)
    row = case.k_pool[int(case.block_table[0, 0]), 0, 0].clone()
    for t in range(40):
        case.k_pool[int(case.block_table[0, t // 16]), t % 16, 0] = row
    got = oracle_decode(case)
    v = dequant_seq(case, 0, "v")
    np.testing.assert_allclose(got[0, 0], v[:, 0].mean(axis=0), rtol=0, atol=1e-14)


def test_closed_form_zero_query_gives_the_mean_of_v():
    spec = synth.CaseSpec(seq_lens=[23], k_type=synth.Q8_0, v_type=synth.Q4_0, junk=0, d=64,
                          hq=3, hkv=1)
    case = synth.build_case(spec, seed=10)
    case.q.zero_()
    got = oracle_decode(case)
    v = dequant_seq(case, 0, "v")
    for h in range(3):
        np.testing.assert_allclose(got[0, h], v[:, 0].mean(axis=0), rtol=0, atol=1e-14)


def test_closed_form_one_dominant_score_selects_its_row():
    spec = synth.CaseSpec(seq_lens=[30], k_type=synth.F16, v_type=synth.F16, junk=0, d=32,
                          hq=1, hkv=1)
    case = synth.build_case(spec, seed=12)
    qv = np.zeros(32, dtype=np.float32)
    qv[0] = 1.0
    case.q[0, 0] = torch.from_numpy(qv)
    # key 17 has component 0 = 100 * sqrt(D), every other key 0 there: its
    # score is 100 above the rest, so its weight is within e^-100 * 29 of 1
    for t in range(30):
        blk, sl = int(case.block_table[0, t // 16]), t % 16
        kr = np.zeros(32, dtype=np.float32)
        kr[0] = 100 * np.sqrt(32) if t == 17 else 0.0
        case.k_pool[blk, sl, 0] = _f16_rows(kr)
    got = oracle_decode(case)
    v = dequant_seq(case, 0, "v")
    np.testing.assert_allclose(got[0, 0], v[17, 0], rtol=0, atol=1e-30 + 1e-40)


def test_empty_sequence_gives_zero():
    spec = synth.CaseSpec(seq_lens=[0, 5], k_type=synth.Q4_0, v_type=synth.Q4_0, junk=1,
                          d=32, hq=2, hkv=1)
    case = synth.build_case(spec, seed=13)
    got = oracle_decode(case)
    assert np.all(got[0] == 0.0)
    assert np.all(np.isfinite(got[1]))


def test_units_subset_matches_full():
    spec = synth.CaseSpec(seq_lens=[70, 20], k_type=synth.Q4_0, v_type=synth.Q4_0, junk=2,
                          d=64, hq=4, hkv=2)
    case = synth.build_case(spec, seed=14)
    full = oracle_decode(case)
    sub = oracle_decode(case, units=[(1, 3), (0, 0)])
    assert np.array_equal(sub[0], full[1, 3]) and np.array_equal(sub[1], full[0, 0])


# -------------------------------------------------------------------- merge

def test_merge_against_full_softmax():
    """Partials built in float64 from random scores, o_p rounded to f16; the
    merge must equal scipy's softmax-weighted sum up to that f16 rounding."""
    rng = np.random.default_rng(2)
    U, P, D, T = 6, 5, 16, 40
    log2e = 1.0 / np.log(2.0)
    obits = np.zeros((U, P, D), dtype=np.uint16)
    ml = np.zeros((U, P, 2), dtype=np.float32)
    n_live = rng.integers(1, P + 1, size=U).astype(np.int32)
    ref = np.zeros((U, D))
    bound = np.zeros(U)
    for u in range(U):
        nl = n_live[u]
        s = rng.standard_normal((nl, T)) * 3  # natural-log scores
        v = rng.standard_normal((nl, T, D))
        w = scipy.special.softmax(s.reshape(-1))
        ref[u] = w @ v.reshape(-1, D)
        for p in range(nl):
            m2 = (s[p] * log2e).max()
            e = np.exp2(s[p] * log2e - m2)
            ml[u, p] = [np.float32(m2), np.float32(e.sum())]
            o = (e @ v[p]) / e.sum()
            obits[u, p] = o.astype(np.float16).view(np.uint16)
        bound[u] = 2.0**-10 * np.abs(v).max() + 1e-5
    got = oracle.merge(obits, ml, n_live)
    for u in range(U):
        assert np.abs(got[u] - ref[u]).max() <= bound[u]


def test_merge_dead_and_single_partials():
    D = 8
    o = np.zeros((3, 3, D), dtype=np.uint16)
    ml = np.zeros((3, 3, 2), dtype=np.float32)
    row = np.arange(D, dtype=np.float16)
    o[0, 1] = row.view(np.uint16)
    ml[0, 1] = [5.0, 3.0]           # the only live partial
    ml[0, 0] = [100.0, 0.0]         # dead (l = 0) even though m is large
    o[0, 0] = np.float16(np.nan).view(np.uint16)  # and its o is never read
    ml[1, :] = [[1.0, 0.0]] * 3     # all dead -> 0
    o[2, 0] = np.full(D, 1.0, dtype=np.float16).view(np.uint16)
    o[2, 1] = np.full(D, 3.0, dtype=np.float16).view(np.uint16)
    ml[2, 0] = [2.0, 1.0]
    ml[2, 1] = [1.0, 2.0]           # weights 1 * 2^0 and 2 * 2^-1: equal
    got = oracle.merge(o, ml, np.array([3, 3, 2], dtype=np.int32))
    assert np.array_equal(got[0], row.astype(np.float64))
    assert np.all(got[1] == 0.0)
    assert np.all(got[2] == 2.0)


# ------------------------------------------------- several query tokens

def _query_rows_of(case, q_hd):
    """float64 [hq, D] query rows as the oracle uses them (q8_1 for a
    quantised K)."""
    sp = case.spec
    if sp.k_type == synth.F16:
        return q_hd.astype(np.float64)
    blocks = oracle.quantize_q8_1(q_hd)
    return np.stack([oracle.dequant_q8_1_row(blocks[h], sp.d) for h in range(sp.hq)])


def causal_sdpa_reference(case, q4):
    """torch SDPA in float64 for T query tokens per sequence: token i sits at
    position L - T + i and sees the keys 0 .. L - T + i (a boolean mask); a
    token with no key gives 0."""
    sp = case.spec
    G, T = sp.hq // sp.hkv, q4.shape[1]
    out = np.zeros((sp.n_seqs, T, sp.hq, sp.d))
    for s in range(sp.n_seqs):
        L = sp.seq_lens[s]
        if L == 0:
            continue
        k = torch.from_numpy(dequant_seq(case, s, "k")).permute(1, 0, 2).repeat_interleave(G, 0)
        v = torch.from_numpy(dequant_seq(case, s, "v")).permute(1, 0, 2).repeat_interleave(G, 0)
        q = torch.from_numpy(np.stack([_query_rows_of(case, q4[s, i]) for i in range(T)], 1))
        mask = torch.tensor([[t <= L - T + i for t in range(L)] for i in range(T)])
        o = torch.nn.functional.scaled_dot_product_attention(
            q.unsqueeze(0), k.unsqueeze(0), v.unsqueeze(0), attn_mask=mask,
            scale=1.0 / np.sqrt(sp.d))[0].permute(1, 0, 2).numpy()   # [T, hq, D]
        for i in range(T):
            if L - T + i >= 0:
                out[s, i] = o[i]
    return out


MULTI = [
    (dict(seq_lens=[40, 2, 0, 17], k_type=synth.F16, v_type=synth.F16, junk=3, d=64, hq=4,
          hkv=2), 3),
    (dict(seq_lens=[50, 5], k_type=synth.Q8_0, v_type=synth.Q4_0, junk=2, d=64, hq=6, hkv=3,
          block_size=32), 4),
    (dict(seq_lens=[33], k_type=synth.Q4_0, v_type=synth.F16, d=32, hq=2, hkv=1), 7),
]


@pytest.mark.parametrize("kw,T", MULTI)
def test_oracle_several_query_tokens_match_causal_sdpa(kw, T):
    case = synth.build_case(synth.CaseSpec(**kw), seed=21)
    q4 = np.random.default_rng(4).standard_normal((case.spec.n_seqs, T, case.spec.hq,
                                                   case.spec.d)).astype(np.float32)
    k, v, bt, sl, _ = _np(case)
    sp = case.spec
    got = oracle.decode(k, v, bt, sl, q4, hkv=sp.hkv, block_size=sp.block_size,
                        k_type=sp.k_type, v_type=sp.v_type)
    assert got.shape == q4.shape
    np.testing.assert_allclose(got, causal_sdpa_reference(case, q4), rtol=1e-12, atol=1e-12)
    # partitioned form of the same rows
    got_p = oracle.decode(k, v, bt, sl, q4, hkv=sp.hkv, block_size=sp.block_size,
                          k_type=sp.k_type, v_type=sp.v_type, part_tokens=16)
    np.testing.assert_allclose(got_p, got, rtol=1e-12, atol=1e-12)


def test_query_token_i_is_the_one_token_step_on_the_prefix():
    kw, T = MULTI[0]
    case = synth.build_case(synth.CaseSpec(**kw), seed=22)
    sp = case.spec
    q4 = np.random.default_rng(5).standard_normal((sp.n_seqs, T, sp.hq, sp.d)).astype(np.float32)
    k, v, bt, sl, _ = _np(case)
    got = oracle.decode(k, v, bt, sl, q4, hkv=sp.hkv, block_size=sp.block_size,
                        k_type=sp.k_type, v_type=sp.v_type)
    for i in range(T):
        li = np.maximum(sl - (T - 1 - i), 0).astype(np.int32)
        one = oracle.decode(k, v, bt, li, q4[:, i], hkv=sp.hkv, block_size=sp.block_size,
                            k_type=sp.k_type, v_type=sp.v_type)
        assert np.array_equal(got[:, i], one)
    # one token in the 4-D form is the plain step
    one = oracle.decode(k, v, bt, sl, q4[:, :1], hkv=sp.hkv, block_size=sp.block_size,
                        k_type=sp.k_type, v_type=sp.v_type)
    ref = oracle.decode(k, v, bt, sl, q4[:, 0], hkv=sp.hkv, block_size=sp.block_size,
                        k_type=sp.k_type, v_type=sp.v_type)
    assert np.array_equal(one[:, 0], ref)


# ------------------------------------------------------- the gate's scale

def _vmax_case():
    """A case built by hand for the pin of oracle.vmax: K rows Q8_0, V rows
    F16 (so the expected value comes from numpy's own half decoding), D=32,
    Hq=4, Hkv=2 (heads 0, 1 read K/V head 0; heads 2, 3 head 1), 16-token
    blocks.  Sequences of 20, 0 and 33 tokens.  The live V rows of head 0
    stay below 1 except two planted values (2.5 at token 19 of sequence 0,
    3.5 at token 32 of sequence 2); every row that a plausible mistake would
    read instead holds a larger magnitude: K (100), the other K/V head's V
    (40), junk blocks (70), slots past L in a last block (60) and the block
    that the empty sequence's table row names (80)."""
    d, hq, hkv, B = 32, 4, 2, 16
    lens = [20, 0, 33]
    table = np.array([[5, 2, -1], [7, -1, -1], [0, 3, 6]], dtype=np.int32)
    n_blocks = 8                      # 1 and 4 are junk; 7 is named only by the empty row
    rng = np.random.default_rng(31)
    v = np.clip(rng.standard_normal((n_blocks, B, hkv, d)), -0.99, 0.99).astype(np.float16)
    v[:, :, 1, :] = 40.0              # K/V head 1 everywhere
    v[[1, 4]] = 70.0                  # junk blocks
    v[7] = 80.0                       # the block of the empty sequence's table row
    v[2, 4:] = 60.0                   # sequence 0: slots 4..15 of its last block (L = 20)
    v[6, 1:] = 60.0                   # sequence 2: slots 1..15 of its last block (L = 33)
    v[2, 3, 0, 5] = -2.5              # sequence 0, token 19, head 0
    v[6, 0, 0, 7] = 3.5               # sequence 2, token 32, head 0
    v_pool = v.view(np.uint8).reshape(n_blocks, B, hkv, 2 * d)
    # Q8_0 K rows: scale 100 (f16) and every code 1, so |K| = 100 everywhere
    k_row = np.zeros(34, dtype=np.uint8)
    k_row[0:2] = np.array([100.0], dtype=np.float16).view(np.uint8)
    k_row[2:] = 1
    k_pool = np.broadcast_to(k_row, (n_blocks, B, hkv, 34)).copy()
    q = rng.standard_normal((3, hq, d)).astype(np.float32)
    return dict(k_pool=k_pool, v_pool=v_pool, table=table, lens=np.array(lens, np.int32), q=q,
                hkv=hkv, B=B)


def _numpy_vmax(c, units, T=1):
    """max |V| over the rows the units read, walked in numpy from the
    definition (row u of a T-token plan is token u % T of sequence u // T
    and sees L - T + 1 + u % T keys)."""
    G = c["q"].shape[-2] // c["hkv"]
    v = c["v_pool"].view(np.float16).reshape(c["v_pool"].shape[:3] + (-1,))
    m = 0.0
    for u, h in units:
        s, i = divmod(u, T)
        L = max(int(c["lens"][s]) - (T - 1 - i), 0)
        for t in range(L):
            blk = int(c["table"][s, t // c["B"]])
            m = max(m, float(np.abs(v[blk, t % c["B"], h // G].astype(np.float64)).max()))
    return m


@pytest.mark.parametrize("units,expect", [
    ([(0, 0), (2, 1)], 3.5),   # both planted values of head 0; 3.5 is the larger
    ([(0, 1)], 2.5),           # sequence 0 alone: its planted value
    ([(1, 0)], 0.0),           # the empty sequence reads no row
    ([(1, 0), (0, 2)], 40.0),  # K/V head 1 of sequence 0
])
def test_oracle_vmax_reads_exactly_the_units_live_v_rows(units, expect):
    c = _vmax_case()
    got = oracle.vmax(c["k_pool"], c["v_pool"], c["table"], c["lens"], c["q"], hkv=c["hkv"],
                      block_size=c["B"], k_type=synth.Q8_0, v_type=synth.F16, units=units)
    assert got == expect
    assert got == _numpy_vmax(c, units)


def test_oracle_vmax_of_query_rows_sees_only_their_causal_prefix():
    """With two query tokens per sequence, row 0 (token 0 of sequence 0)
    sees 19 keys and misses the planted 2.5 at token 19; row 1 sees it."""
    c = _vmax_case()
    q2 = np.stack([c["q"], c["q"]], axis=1)  # [S, T=2, hq, d]
    kw = dict(hkv=c["hkv"], block_size=c["B"], k_type=synth.Q8_0, v_type=synth.F16)
    first = oracle.vmax(c["k_pool"], c["v_pool"], c["table"], c["lens"], q2, units=[(0, 0)],
                        **kw)
    second = oracle.vmax(c["k_pool"], c["v_pool"], c["table"], c["lens"], q2, units=[(1, 0)],
                         **kw)
    assert 0.0 < first < 1.0 and first == _numpy_vmax(c, [(0, 0)], T=2)
    assert second == 2.5

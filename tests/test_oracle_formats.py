"""Pins for the oracle's format code: f16 conversions, Q4_0 / Q8_0 / q8_1,
row sizes and 64-bit row offsets.  Each check ties the oracle to something
other than itself: numpy's IEEE half conversions, closed forms of the block
formats, numbers printed on the pages, or the independent encoders in
``synth`` (round-trip bounds)."""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_half_to_double_all_patterns_match_numpy():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.half_to_double(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_float_to_half_rn_matches_numpy():
    rng = np.random.default_rng(1)
    bits = rng.integers(0, 2**32, size=200_000, dtype=np.uint64).astype(np.uint32)
    xs = bits.view(np.float32)
    edge = np.array([0.0, -0.0, 1.0, 65504.0, 65519.99, 65520.0, 1e-8, 2.0**-24, 2.0**-25,
                     3 * 2.0**-26, 2.0**-14, 2.0**-14 * (1 - 2.0**-11), 1 + 2.0**-11,
                     1 + 3 * 2.0**-11, np.inf, -np.inf], dtype=np.float32)
    xs = np.concatenate([xs, edge, -edge])
    # half-way points between neighbouring halves (ties to even)
    hb = np.arange(0, 0x7bff, 7, dtype=np.uint16)
    lo = hb.view(np.float16).astype(np.float64)
    hi = (hb + 1).view(np.float16).astype(np.float64)
    xs = np.concatenate([xs, ((lo + hi) / 2).astype(np.float32)])
    with np.errstate(over="ignore"):  # values beyond the half range overflow to inf on purpose
        ref = xs.astype(np.float16).view(np.uint16)
    got = np.array([oracle.float_to_half_rn(float(x)) for x in xs], dtype=np.uint16)
    isnan = np.isnan(xs)
    assert np.all((got[isnan] & 0x7c00) == 0x7c00) and np.all((got[isnan] & 0x3ff) != 0)
    assert np.array_equal(got[~isnan], ref[~isnan])


def _half_bits(x):
    return int(np.float16(x).view(np.uint16))


def test_q4_0_closed_forms():
    # block: d = 0.5; byte j holds low nibble lo_j, high nibble hi_j
    d = 0.5
    lo = [8, 0, 15, 1, 2, 3, 4, 5, 6, 7, 9, 10, 11, 12, 13, 14]
    hi = [0, 15, 8, 14, 13, 12, 11, 10, 9, 7, 6, 5, 4, 3, 2, 1]
    blk = bytearray(_half_bits(d).to_bytes(2, "little"))
    blk += bytes((h << 4) | l for l, h in zip(lo, hi))
    row = np.frombuffer(bytes(blk), dtype=np.uint8)
    x = oracle.dequant_row(oracle.Q4_0, row, 32)
    assert x[0] == 0.0          # nibble 8 -> 0
    assert x[1] == -8 * d       # nibble 0 -> -8 d
    assert x[2] == 7 * d        # nibble 15 -> +7 d
    assert x[16] == -8 * d      # high nibble of byte 0 is value 16
    assert x[17] == 7 * d
    assert x[18] == 0.0
    assert x[31] == (1 - 8) * d


def test_q8_0_closed_forms():
    d = 0.25
    q = np.array([-127, -1, 0, 1, 127] + [3] * 27, dtype=np.int8)
    row = np.frombuffer(_half_bits(d).to_bytes(2, "little") + q.tobytes(), dtype=np.uint8)
    x = oracle.dequant_row(oracle.Q8_0, row, 32)
    assert list(x[:5]) == [-127 * d, -d, 0.0, d, 127 * d]
    assert np.all(x[5:] == 3 * d)


@pytest.mark.parametrize("type_", [synth.F16, synth.Q8_0, synth.Q4_0])
def test_round_trip_against_independent_encoder(type_):
    """synth's encoder (input generation) and the oracle's decoder are
    separate code; a swapped nibble half, a wrong scale offset or a sign
    slip in either breaks this bound."""
    g = torch.Generator().manual_seed(7)
    x = torch.randn(64, 256, generator=g) * 3
    enc = synth.encode(x, type_).numpy()
    for r in range(x.shape[0]):
        xh = oracle.dequant_row(type_, enc[r], 256)
        xr = x[r].double().numpy()
        if type_ == synth.F16:
            assert np.all(np.abs(xh - xr) <= np.abs(xr) * 2.0**-11 + 2.0**-25)
            continue
        for b in range(8):
            blk = xr[32 * b:32 * b + 32]
            amax = np.abs(blk).max()
            step = amax / 127 if type_ == synth.Q8_0 else amax / 8
            err = np.abs(xh[32 * b:32 * b + 32] - blk).max()
            # half a quantisation step, plus the f16 rounding of the scale
            bound = step / 2 + amax * 2.0**-10
            if type_ == synth.Q4_0:
                bound = step + amax * 2.0**-10  # 16 levels, the top one clipped
            assert err <= bound, (r, b, err, bound)


def test_row_bytes_pinned_by_the_pages_capacity_numbers():
    g = json.load(open(os.path.join(GOLDEN, "capacity_q4_0.json")))
    d, hkv = g["d"], g["hkv"]
    per_token = 2 * hkv * oracle.row_bytes(oracle.Q4_0, d)  # K and V
    assert per_token == 1152
    lens = g["seq_lens"]
    live = sum(math.ceil(L / g["block_size"]) * g["block_size"] for L in lens)
    assert live == g["live_block_rounded_tokens"]
    padded = len(lens) * max(lens)
    assert padded == g["padded_slots"]
    MiB, GiB = 2.0**20, 2.0**30
    assert padded * per_token / MiB == g["one_layer_padded_MiB"]
    assert round(live * per_token / MiB) == g["one_layer_paged_MiB"]
    assert f"{g['layers'] * padded * per_token / GiB:.3f}" == g["sixteen_layer_padded_GiB"]
    assert f"{g['layers'] * live * per_token / GiB:.3f}" == g["sixteen_layer_paged_GiB"]
    assert f"{padded / live:.2f}" == g["reduction"]
    assert f"{100 * (1 - live / padded):.2f}" == g["saving_percent"]
    # the other two formats by their block sizes (2 + 32 bytes, 2 bytes per value)
    assert oracle.row_bytes(oracle.Q8_0, 256) == 8 * 34
    assert oracle.row_bytes(oracle.F16, 256) == 512


def test_row_offset_64bit_pinned_by_the_pages_wrap_point():
    g = json.load(open(os.path.join(GOLDEN, "offset64_llama.json")))
    B, hkv, d, es = g["block_size"], g["hkv"], g["d"], g["bytes_per_element"]
    rb = d * es
    assert g["wrap_blocks"] * B == g["wrap_token_slots"]
    assert g["wrap_token_slots"] * hkv * d == 2**32
    assert g["wrap_token_slots"] * hkv * d * es == g["wrap_GiB_per_side"] * 2**30
    # first row past the wrap point: element offset exactly 2^32
    off = oracle.row_offset(g["wrap_blocks"], 0, 0, B, hkv, rb)
    assert off == 2**32 * es
    assert (off // es) & 0xFFFFFFFF == 0  # a 32-bit offset would wrap to row 0
    # a pool of exactly 2^32 elements addresses its last element
    last = oracle.row_offset(g["wrap_blocks"] - 1, B - 1, hkv - 1, B, hkv, rb) // es + d - 1
    assert last == 2**32 - 1
    # the last block of the page's 131,073-block test pool
    off_last = oracle.row_offset(g["test_pool_blocks"] - 1, B - 1, hkv - 1, B, hkv, rb)
    assert off_last + rb == g["test_pool_blocks"] * B * hkv * rb


def test_row_offset_is_a_bijection_on_a_small_pool():
    n, B, hkv, rb = 5, 16, 3, 144
    offs = sorted(oracle.row_offset(b, s, h, B, hkv, rb)
                  for b in range(n) for s in range(B) for h in range(hkv))
    assert offs == [i * rb for i in range(n * B * hkv)]


# --------------------------------------------------------------- q8_1

def _q8_1_fields(blk):
    d = np.frombuffer(blk[0:2].tobytes(), dtype=np.float16)[0]
    s = np.frombuffer(blk[2:4].tobytes(), dtype=np.float16)[0]
    q = blk[4:36].view(np.int8)
    return float(d), float(s), q


def test_q8_1_properties_random():
    rng = np.random.default_rng(3)
    x = (rng.standard_normal((50, 256)) * rng.uniform(0.01, 100, (50, 1))).astype(np.float32)
    out = oracle.quantize_q8_1(x)
    assert out.shape == (50, 8 * 36)
    for r in range(50):
        for b in range(8):
            blk = out[r, 36 * b:36 * b + 36]
            d16, s16, q = _q8_1_fields(blk)
            xb = x[r, 32 * b:32 * b + 32]
            amax = float(np.abs(xb).max())
            d32 = np.float32(amax) / np.float32(127)
            assert d16 == float(np.float16(d32))
            assert np.abs(q).max() == 127
            assert q[np.argmax(np.abs(xb))] == np.sign(xb[np.argmax(np.abs(xb))]) * 127
            # within half a step of the float32 scale
            assert np.all(np.abs(q.astype(np.float64) * float(d32) - xb) <= float(d32) * 0.5001)
            assert s16 == float(np.float16(np.float32(d32) * np.float32(q.astype(np.int64).sum())))


def test_q8_1_ties_round_half_away_from_zero_and_zero_block():
    xb = np.zeros(32, dtype=np.float32)
    xb[0] = 127.0                     # d = 1 exactly, so x / d = x
    xb[1:5] = [2.5, -2.5, 0.5, -0.5]  # ties: away from zero
    xb[5:7] = [1.4999999, -126.5]
    out = oracle.quantize_q8_1(xb.reshape(1, 32))
    d16, s16, q = _q8_1_fields(out[0])
    assert d16 == 1.0
    assert list(q[:7]) == [127, 3, -3, 1, -1, 1, -127]
    z = oracle.quantize_q8_1(np.zeros((1, 32), dtype=np.float32))
    assert not z.any()


def test_q8_1_dequant_definition():
    x = np.linspace(-3, 3, 64, dtype=np.float32).reshape(1, 64)
    blocks = oracle.quantize_q8_1(x)[0]
    xh = oracle.dequant_q8_1_row(blocks, 64)
    for b in range(2):
        d16, _, q = _q8_1_fields(blocks[36 * b:36 * b + 36])
        assert np.array_equal(xh[32 * b:32 * b + 32], q.astype(np.float64) * d16)

"""CPU tests of the C ABI: the library loads and exports every declared
symbol; the allocator and the planner match their plain-Python models bit for
bit; refusals happen before any device work (no GPU is touched here)."""
import ctypes
import os
import random
import re
import subprocess
import sys

import pytest

import paged_kv_attention_attn_gb300 as pa
from oracle import plan_model, pool_model

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def built():
    from paged_kv_attention_attn_gb300 import build
    build.build()
    pa.lib()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "pa.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pa_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported():
    names = declared_functions()
    assert len(names) >= 19
    L = pa.lib()
    for n in names:
        assert hasattr(L, n), n
    assert sorted(pa.EXPORTS) == names


def test_strerror_and_row_bytes():
    L = pa.lib()
    assert L.pa_strerror(pa.PA_ERR_CORRUPT_TABLE) == b"PA_ERR_CORRUPT_TABLE"
    assert L.pa_strerror(12345) == b"PA_ERR_UNKNOWN"
    assert pa.row_bytes(pa.Q4_0, 256) == 144 and pa.row_bytes(pa.Q8_0, 256) == 272
    assert pa.row_bytes(pa.F16, 128) == 256 and pa.row_bytes(pa.F16, 100) == 0


def test_pool_matches_model_on_random_traces():
    rng = random.Random(0)
    for trial in range(20):
        n = rng.randint(1, 64)
        cpool, mpool = pa.Pool(n), pool_model.PoolModel(n)
        live = []
        for _ in range(400):
            r = rng.random()
            if r < 0.5:
                k = rng.randint(0, n // 2 + 2)
                mrc, mh = mpool.alloc(k)
                try:
                    ch = cpool.alloc(k)
                    crc = pa.PA_OK
                except pa.PAError as e:
                    ch, crc = [], e.code
                assert crc == mrc and ch == mh
                live += ch
            else:
                pick = rng.sample(live, min(len(live), rng.randint(0, 4))) if live else []
                if rng.random() < 0.25 and live:
                    # a stale, repeated or out-of-range handle somewhere in the list
                    bad = rng.choice([pick + pick[:1] if pick else [live[0], live[0]],
                                      pick + [(99 << 32) | (live[0] & 0xFFFFFFFF)],
                                      pick + [(1 << 32) | (n + 5)]])
                    pick = bad
                mrc = mpool.free(pick)
                try:
                    cpool.free(pick)
                    crc = pa.PA_OK
                except pa.PAError as e:
                    crc = e.code
                assert crc == mrc
                if mrc == pool_model.OK:
                    for h in pick:
                        live.remove(h)
            assert cpool.free_count() == mpool.free_count()
        assert cpool.capacity() == n
        cpool.close()


def test_pool_refusals():
    with pytest.raises(pa.PAError) as e:
        pa.Pool(0)
    assert e.value.code == pa.PA_ERR_INVALID
    p = pa.Pool(3)
    with pytest.raises(pa.PAError) as e:
        p.alloc(4)
    assert e.value.code == pa.PA_ERR_NOMEM and "pa_pool_alloc" in str(e.value)
    assert p.free_count() == 3
    hs = p.alloc(2)
    assert [pa.Pool.block_of(h) for h in hs] == [0, 1]


def test_plan_matches_model():
    rng = random.Random(2)
    for _ in range(4000):
        S = rng.choice([rng.randint(1, 64), rng.randint(100, 2000)])
        lens = [rng.choice([0, 1, 16, 33, rng.randint(0, 400000)]) for _ in range(S)]
        kw = dict(n_seqs=S, max_len=max(lens), total_len=sum(lens),
                  block_size=rng.choice([16, 32, 8]), hq=rng.choice([24, 32, 12, 7]),
                  hkv=rng.choice([4, 8, 1]), d=rng.choice([128, 256, 64]),
                  k_type=rng.choice([0, 1, 2]), v_type=rng.choice([0, 1, 2]),
                  sm_count=rng.choice([152, 148, 1]), ctas_per_sm=rng.choice([1, 2]),
                  force_parts=rng.choice([0, 0, 3, 64]), q_tokens=rng.choice([1, 1, 2, 5]),
                  flags=rng.choice([0, 1, 2, 3]))
        mrc, mp = plan_model.plan(**kw)
        pin = pa.PlanIn(**kw)
        out = pa.Plan()
        crc = pa.lib().pa_plan(ctypes.byref(pin), ctypes.byref(out))
        assert crc == mrc, kw
        if crc == 0:
            assert out.as_dict() == mp, kw


def _dummy_args(**over):
    base = dict(k_pool=16, v_pool=16, n_pool_blocks=4, block_table=16, table_stride=1,
                seq_lens=16, q=16, scale=0.0625, part_o=16, part_ml=16, out=16, status=16,
                n_seqs=1, hq=24, hkv=4, d=256, block_size=16, k_type=2, v_type=2, flags=0)
    base.update(over)
    return pa.DecodeArgs(**base)


@pytest.mark.parametrize("over,code", [
    (dict(hq=25), pa.PA_ERR_INVALID),
    (dict(d=192), pa.PA_ERR_INVALID),
    (dict(block_size=8), pa.PA_ERR_INVALID),
    (dict(k_type=7), pa.PA_ERR_INVALID),
    (dict(status=None), pa.PA_ERR_INVALID),
    (dict(k_pool=8), pa.PA_ERR_INVALID),          # misaligned pool
    (dict(n_pool_blocks=0), pa.PA_ERR_RANGE),
    (dict(n_pool_blocks=(1 << 31) + 1), pa.PA_ERR_RANGE),
    (dict(scale=float("nan")), pa.PA_ERR_INVALID),
])
def test_decode_refusals_happen_before_any_launch(over, code):
    pl = pa.Plan(part_tokens=128, n_parts=2, direct=0, n_ctas=2, part_o_bytes=0, part_ml_bytes=0)
    a = _dummy_args(**over)
    rc = pa.lib().pa_decode_partial(ctypes.byref(a), ctypes.byref(pl), None)
    assert rc == code
    assert pa.lib().pa_last_error().startswith(b"pa_decode_partial: ")


def test_merge_and_plan_refusals():
    L = pa.lib()
    direct = pa.Plan(part_tokens=32, n_parts=1, direct=1, n_ctas=1)
    assert L.pa_merge(16, 16, 16, 16, 1, 24, 256, ctypes.byref(direct), None) == pa.PA_ERR_INVALID
    bad = pa.Plan(part_tokens=33, n_parts=2, direct=0, n_ctas=1)
    assert L.pa_merge(16, 16, 16, 16, 1, 24, 256, ctypes.byref(bad), None) == pa.PA_ERR_INVALID
    big = pa.Plan(part_tokens=32, n_parts=1 << 20, direct=0, n_ctas=1)
    assert L.pa_merge(16, 16, 16, 16, 1 << 12, 64, 256, ctypes.byref(big), None) == \
        pa.PA_ERR_RANGE
    assert b"pa_merge" in L.pa_last_error()
    assert L.pa_quantize_q(16, 16, 1, 48, None) == pa.PA_ERR_INVALID


def test_fused_refuses_missing_counters():
    pl = pa.Plan(part_tokens=128, n_parts=2, direct=0, n_ctas=2, part_o_bytes=0, part_ml_bytes=0)
    a = _dummy_args()
    assert pa.lib().pa_decode_fused(ctypes.byref(a), ctypes.byref(pl), None, None) == \
        pa.PA_ERR_INVALID
    assert pa.lib().pa_last_error().startswith(b"pa_decode_fused: ")
    assert pa.lib().pa_decode_step_fused(ctypes.byref(a), ctypes.byref(pl), 16, 2, None) == \
        pa.PA_ERR_INVALID


def test_append_refuses_bad_arguments_before_any_launch():
    L = pa.lib()
    good = dict(k_pool=16, v_pool=16, n_pool_blocks=4, block_table=16, table_stride=2,
                seq_lens=16, k_new=16, v_new=16, fresh_blocks=16, status=16, n_seqs=2, hkv=4,
                d=256, block_size=16, k_type=pa.Q4_0, v_type=pa.Q4_0)
    assert L.pa_append_kv(None, None) == pa.PA_ERR_INVALID
    for key, bad, rc in [("d", 96, pa.PA_ERR_INVALID), ("block_size", 8, pa.PA_ERR_INVALID),
                         ("hkv", 0, pa.PA_ERR_INVALID), ("k_type", 7, pa.PA_ERR_INVALID),
                         ("status", None, pa.PA_ERR_INVALID), ("k_new", 20, pa.PA_ERR_INVALID),
                         ("table_stride", 0, pa.PA_ERR_INVALID),
                         ("n_pool_blocks", 2 ** 31 + 1, pa.PA_ERR_RANGE)]:
        a = pa.AppendArgs(**dict(good, **{key: bad}))
        assert L.pa_append_kv(ctypes.byref(a), None) == rc, key
        assert L.pa_last_error().startswith(b"pa_append_kv: ")
    # an empty batch is a no-op that touches nothing
    a = pa.AppendArgs(**dict(good, n_seqs=0))
    assert L.pa_append_kv(ctypes.byref(a), None) == pa.PA_OK


def test_plan_log_line_when_asked():
    """PA_LOG_PLAN=1 makes pa_plan write one line with its inputs and the plan
    to stderr; without it nothing is written."""
    code = ("import paged_kv_attention_attn_gb300 as pa; "
            "pa.plan(seq_lens=[131072] * 8, block_size=16, hq=24, hkv=4, d=256, k_type=2, "
            "v_type=2, sm_count=152, ctas_per_sm=1)")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    for value, expect in (("1", True), ("0", False), (None, False)):
        env = dict(os.environ)
        env.pop("PA_LOG_PLAN", None)
        if value is not None:
            env["PA_LOG_PLAN"] = value
        r = subprocess.run([sys.executable, "-c", code], cwd=root, env=env, capture_output=True,
                           text=True, timeout=300)
        assert r.returncode == 0, r.stderr[-2000:]
        lines = [l for l in r.stderr.splitlines() if l.startswith("pa_plan:")]
        if expect:
            assert lines == ["pa_plan: n_seqs=8 q_tokens=1 max_len=131072 total_len=1048576 "
                             "slots=152 force_parts=0 flags=0 -> part_tokens=6912 n_parts=19 "
                             "direct=0 n_direct=0 n_ctas=152 stream=0 multi=0"]
        else:
            assert lines == []

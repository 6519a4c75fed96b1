"""Pins for the plain-Python allocator and planner models: the properties
the pages state (all-or-nothing allocation, stale-handle detection,
immediate release; partitions cover every token, direct mode has one) and
the build's frozen reading of the order."""
import math
import random

from oracle import plan_model, pool_model


def test_pool_fresh_order_and_handles():
    p = pool_model.PoolModel(5)
    rc, hs = p.alloc(3)
    assert rc == pool_model.OK
    assert [pool_model.PoolModel.block_of(h) for h in hs] == [0, 1, 2]
    assert all(h >> 32 == 1 for h in hs) and 0 not in hs
    assert p.free_count() == 2


def test_pool_all_or_nothing():
    p = pool_model.PoolModel(4)
    p.alloc(3)
    before = (list(p.stack), list(p.gen), list(p.live))
    rc, hs = p.alloc(2)
    assert rc == pool_model.NOMEM and hs == []
    assert (list(p.stack), list(p.gen), list(p.live)) == before


def test_pool_stale_double_and_duplicate_free_release_nothing():
    p = pool_model.PoolModel(4)
    _, hs = p.alloc(3)
    assert p.free([hs[1]]) == pool_model.OK
    snap = (list(p.stack), list(p.gen), list(p.live))
    assert p.free([hs[0], hs[1]]) == pool_model.STALE      # hs[1] already freed
    assert p.free([hs[0], hs[0]]) == pool_model.STALE      # listed twice
    assert p.free([(7 << 32) | 2]) == pool_model.STALE     # wrong generation
    assert p.free([(1 << 32) | 9]) == pool_model.STALE     # id out of range
    assert (list(p.stack), list(p.gen), list(p.live)) == snap
    # the stale handle stays stale after its block is reused
    _, again = p.alloc(1)
    assert pool_model.PoolModel.block_of(again[0]) == 1 and again[0] != hs[1]
    assert p.free([hs[1]]) == pool_model.STALE


def test_pool_release_is_immediate_and_lifo():
    p = pool_model.PoolModel(6)
    _, hs = p.alloc(6)
    assert p.free_count() == 0
    assert p.free([hs[4], hs[2]]) == pool_model.OK
    assert p.free_count() == 2
    _, hs2 = p.alloc(2)
    assert [pool_model.PoolModel.block_of(h) for h in hs2] == [2, 4]


def test_pool_generation_skips_zero_on_wrap():
    p = pool_model.PoolModel(1)
    p.gen[0] = 0xFFFFFFFF
    _, hs = p.alloc(1)
    assert hs[0] >> 32 == 0xFFFFFFFF
    p.free(hs)
    _, hs = p.alloc(1)
    assert hs[0] >> 32 == 1


def test_pool_random_trace_invariants():
    rng = random.Random(0)
    p = pool_model.PoolModel(50)
    live = set()
    for _ in range(2000):
        if rng.random() < 0.55:
            rc, hs = p.alloc(rng.randint(0, 12))
            if rc == pool_model.OK:
                assert not (set(hs) & live)
                live |= set(hs)
        elif live:
            k = rng.randint(1, min(5, len(live)))
            hs = rng.sample(sorted(live), k)
            assert p.free(hs) == pool_model.OK
            live -= set(hs)
        assert p.free_count() + len(live) == 50
        ids = [pool_model.PoolModel.block_of(h) for h in live]
        assert len(set(ids)) == len(ids)


def _plan(**kw):
    base = dict(n_seqs=1, max_len=0, total_len=0, block_size=16, hq=24, hkv=4, d=256,
                k_type=2, v_type=2, sm_count=152, ctas_per_sm=1, force_parts=0)
    base.update(kw)
    return plan_model.plan(**base)


def test_plan_covers_every_token_and_bounds_the_grid():
    rng = random.Random(1)
    for _ in range(3000):
        S = rng.randint(1, 40)
        lens = [rng.choice([0, 1, 15, 16, 17, 200, rng.randint(0, 300000)]) for _ in range(S)]
        mx, tot = max(lens), sum(lens)
        force = rng.choice([0, 0, 1, 2, 7, 1000])
        T = rng.choice([1, 1, 2, 6])
        sm, cps = rng.choice([1, 152, 160]), rng.choice([1, 2, 3])
        rc, p = _plan(n_seqs=S, max_len=mx, total_len=tot, force_parts=force,
                      block_size=rng.choice([16, 32]), sm_count=sm, ctas_per_sm=cps,
                      q_tokens=T)
        assert rc == plan_model.OK
        P, n = p["part_tokens"], p["n_parts"]
        assert P % 32 == 0 and P > 0
        assert n * P >= mx and (n - 1) * P < max(mx, 1)
        assert p["direct"] == (n == 1)
        # the grid has a CTA for every live partition of every query row and
        # one for every empty row (which writes its zero output); the leading
        # n_direct rows of a wave-filling plan have one CTA each
        rows = [max(0, L - (T - 1 - i)) for L in lens for i in range(T)]
        nd = p["n_direct"]
        live = nd + sum(max(1, math.ceil(L / P)) for L in rows[nd:])
        assert p["n_ctas"] >= (S * T if p["direct"] else live)
        assert p["n_ctas"] <= S * T * n
        if nd:
            # only a direct-sized batch wider than the machine fills its last wave
            slots = sm * cps
            assert not force and not p["direct"] and n >= 2 and S * T > slots
            assert nd == S * T - (S * T) % slots and p["n_ctas"] == nd + (S * T - nd) * n
        if force:
            assert n <= force
        elif not p["direct"] and S * T < sm * cps:
            # fewer query rows than slots: the grid fits one wave
            assert p["n_ctas"] <= sm * cps
        if not p["direct"]:
            assert p["part_o_bytes"] == (S * T - nd) * 24 * n * 256 * 2
            assert p["part_ml_bytes"] == (S * T - nd) * 24 * n * 8


def test_plan_worked_examples():
    # uniform 8 x 128K on 152 SMs: the live work spread over one wave
    rc, p = _plan(n_seqs=8, max_len=131072, total_len=8 * 131072)
    assert (p["part_tokens"], p["n_parts"], p["n_ctas"]) == (6912, 19, 152)
    # ragged 128K + 7 x 8K: partitions sized by total work, not by the longest
    # sequence; 1248 tokens (the work over 152 slots) would bound the grid at
    # 151 + 8 = 159 CTAs, a second wave, so they grow to ceil(188416 / 144)
    # rounded to 1312: at most 144 + 8 = 152 CTAs (149 live)
    rc, p = _plan(n_seqs=8, max_len=131072, total_len=131072 + 7 * 8192)
    assert p["part_tokens"] == 1312 and p["n_parts"] == 100
    assert sum(math.ceil(L / 1312) for L in [131072] + [8192] * 7) == 149 <= p["n_ctas"] == 152
    # a nearly uniform batch that would spill past one wave fits it instead:
    # 3 x 100000 rounds to 51 partitions each (153 CTAs), one wave takes 50
    rc, p = _plan(n_seqs=3, max_len=100000, total_len=300000)
    assert (p["part_tokens"], p["n_parts"], p["n_ctas"]) == (2016, 50, 150)
    # a verify window of 4 tokens on 8 x 32768: 32 query rows in one wave
    rc, p = _plan(n_seqs=8, max_len=32768, total_len=8 * 32768, q_tokens=4)
    assert (p["part_tokens"], p["n_parts"], p["n_ctas"]) == (8192, 4, 128)
    # a batch of whole waves runs direct
    rc, p = _plan(n_seqs=304, max_len=4096, total_len=304 * 4096)
    assert p["direct"] == 1 and p["n_ctas"] == 304 and p["n_direct"] == 0
    # wider batches fill their last wave: 160 x 6912 keeps 152 direct rows and
    # splits the other 8 into ceil(6912 / 19) -> 384-token partitions (18 each),
    # 152 + 144 CTAs instead of a second wave of 8 full-length ones
    rc, p = _plan(n_seqs=160, max_len=6912, total_len=160 * 6912)
    assert (p["part_tokens"], p["n_parts"], p["n_direct"], p["n_ctas"]) == (384, 18, 152, 296)
    assert p["part_o_bytes"] == 8 * 24 * 18 * 256 * 2 and p["direct"] == 0
    # 512 x 4096: three direct waves (456 rows) and 56 rows in halves
    rc, p = _plan(n_seqs=512, max_len=4096, total_len=512 * 4096)
    assert (p["part_tokens"], p["n_parts"], p["n_direct"], p["n_ctas"]) == (2048, 2, 456, 568)
    # 230 x 4096: a last wave of 78 rows in thirds, two waves of 1376-token
    # partitions (2 x (1376 + 512) < 4096 + 512 in the planner's estimate)
    rc, p = _plan(n_seqs=230, max_len=4096, total_len=230 * 4096)
    assert (p["part_tokens"], p["n_parts"], p["n_direct"], p["n_ctas"]) == (1376, 3, 152, 386)
    # 256 x 4096: no split of the last 104 rows beats leaving them whole
    rc, p = _plan(n_seqs=256, max_len=4096, total_len=256 * 4096)
    assert p["direct"] == 1 and p["n_ctas"] == 256
    # forcing one partition is direct; empty batch is direct
    assert _plan(n_seqs=4, max_len=32768, total_len=4 * 32768, force_parts=1)[1]["direct"] == 1
    assert _plan(n_seqs=3, max_len=0, total_len=0)[1]["direct"] == 1


def test_plan_rejects_bad_input():
    assert _plan(hq=25)[0] == plan_model.INVALID
    assert _plan(block_size=8)[0] == plan_model.INVALID
    assert _plan(d=96)[0] == plan_model.INVALID
    assert _plan(n_seqs=2, max_len=10, total_len=30)[0] == plan_model.INVALID
    assert _plan(hq=48, hkv=4)[0] == plan_model.INVALID  # group of 12 > 8

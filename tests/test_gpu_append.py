"""The K/V append step on the GPU against the oracle's append model.

Sequences join at different steps and grow through many block boundaries;
every fresh block comes from the allocator model and only its id is
uploaded.  After every step the device pools, table and lengths equal the
model's bit for bit (whole pools compared, so nothing was written anywhere
else), and the decode over the appended cache matches the oracle."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_attention_attn_gb300 as pa
import synth
from oracle import append_model, pool_model
from tests import helpers as H

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def built():
    from paged_kv_attention_attn_gb300 import build
    build.build()
    oracle.build()


def _rows(rng, shape, step):
    x = rng.standard_normal(shape).astype(np.float32) * (1 + step % 3)
    x[..., :32] = np.where(rng.random(x[..., :32].shape) < 0.05, 0.0, x[..., :32])
    if step % 7 == 0:
        x[0, 0, :32] = 0.0
        x[0, 0, 0] = -0.0               # zero block led by -0
        x[-1, -1, 32:64] = np.round(x[-1, -1, 32:64])   # ties
    return x


@pytest.mark.parametrize("kt,vt,d,hkv,B", [
    (synth.Q4_0, synth.Q4_0, 256, 4, 16),
    (synth.Q8_0, synth.Q4_0, 256, 4, 32),
    (synth.F16, synth.Q8_0, 128, 8, 16),
    (synth.Q4_0, synth.F16, 128, 2, 32),
])
def test_append_steps_equal_the_model_and_decode_matches(kt, vt, d, hkv, B):
    S, steps = 5, 75
    joins = [0, 3, 16, 17, 40]           # sequence s appends from step joins[s] on
    stride = steps // B + 2
    n_blocks = S * stride + 7
    rk, rv = oracle.row_bytes(kt, d), oracle.row_bytes(vt, d)
    pk = np.full((n_blocks, B, hkv, rk), 0xFF, np.uint8)
    pv = np.full((n_blocks, B, hkv, rv), 0xFF, np.uint8)
    table = np.full((S, stride), -1, np.int32)
    lens = np.zeros(S, np.int32)
    dk, dv = torch.from_numpy(pk).to(DEV), torch.from_numpy(pv).to(DEV)
    dt, dl = torch.from_numpy(table).to(DEV), torch.from_numpy(lens).to(DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    alloc = pool_model.PoolModel(n_blocks)
    # shuffle the free stack so that neighbouring sequences get scattered blocks
    rng = np.random.default_rng(kt * 10 + vt)
    rng.shuffle(alloc.stack)
    for t in range(steps):
        n = sum(1 for j in joins if j <= t)       # the first n sequences take part
        fresh = np.full(S, -1, np.int32)
        for s in range(n):
            if lens[s] % B == 0:
                rc, hs = alloc.alloc(1)
                assert rc == pool_model.OK
                fresh[s] = pool_model.PoolModel.block_of(hs[0])
        kn, vn = _rows(rng, (n, hkv, d), t), _rows(rng, (n, hkv, d), t + 1)
        t_sub, l_sub = table[:n].copy(), lens[:n].copy()
        st = append_model.append(pk, pv, t_sub, l_sub, kn, vn, fresh[:n], block_size=B,
                                 k_type=kt, v_type=vt)
        table[:n], lens[:n] = t_sub, l_sub
        assert st == 0
        pa.append_kv(k_pool=dk, v_pool=dv, block_table=dt[:n], seq_lens=dl[:n],
                     k_new=torch.from_numpy(kn).to(DEV), v_new=torch.from_numpy(vn).to(DEV),
                     fresh_blocks=torch.from_numpy(fresh[:n]).to(DEV), status=status, hkv=hkv,
                     block_size=B, k_type=kt, v_type=vt)
        if t % 15 == 0 or t == steps - 1:
            torch.cuda.synchronize()
            assert pa.status_read(status) == 0
            assert np.array_equal(dl.cpu().numpy(), lens)
            assert np.array_equal(dt.cpu().numpy(), table)
            assert np.array_equal(dk.cpu().numpy(), pk)
            assert np.array_equal(dv.cpu().numpy(), pv)
    # decode over what was appended
    hq = hkv * 3
    spec = synth.CaseSpec(seq_lens=[int(x) for x in lens], k_type=kt, v_type=vt, d=d, hq=hq,
                          hkv=hkv, block_size=B, name="appended")
    q = torch.from_numpy(rng.standard_normal((S, hq, d)).astype(np.float32)).to(DEV)
    case = synth.Case(spec=spec, k_pool=dk, v_pool=dv, block_table=dt, seq_lens=dl, q=q,
                      seed=0)
    for fused in (False, True):
        out, ws, _, _ = H.run(case, fused=fused, force_parts=3)
        assert pa.status_read(ws.status) == 0
        H.assert_close(case, out, H.oracle_out(case), H.oracle_vmax(case))


def test_append_flags_a_full_table_and_an_out_of_pool_block():
    B, d, hkv = 16, 128, 2
    pk = np.full((4, B, hkv, 2 * d), 0xAB, np.uint8)
    table = np.array([[0], [-1]], np.int32)
    lens = np.array([16, 0], np.int32)                 # sequence 0: no entry left
    dk, dv = torch.from_numpy(pk).to(DEV), torch.from_numpy(pk.copy()).to(DEV)
    dt, dl = torch.from_numpy(table).to(DEV), torch.from_numpy(lens).to(DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    rows = torch.ones(2, hkv, d, device=DEV)
    pa.append_kv(k_pool=dk, v_pool=dv, block_table=dt, seq_lens=dl, k_new=rows, v_new=rows,
                 fresh_blocks=torch.tensor([0, 4], dtype=torch.int32, device=DEV),
                 status=status, hkv=hkv, block_size=B, k_type=synth.F16, v_type=synth.F16)
    torch.cuda.synchronize()
    st = pa.status_read(status)
    assert st == pa.PA_STATUS_APPEND_RANGE | pa.PA_STATUS_CORRUPT_TABLE
    assert np.array_equal(dl.cpu().numpy(), lens) and np.array_equal(dt.cpu().numpy(), table)
    assert np.array_equal(dk.cpu().numpy(), pk) and np.array_equal(dv.cpu().numpy(), pk)

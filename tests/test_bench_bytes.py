"""The numerator of the roofline: bench.algorithmic_bytes against closed
forms written out here for the headline plan, a direct plan and a
wave-filling plan (CPU)."""
import os
import sys

import paged_kv_attention_attn_gb300 as pa
import synth

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402


def _plan(spec):
    return pa.plan(seq_lens=spec.seq_lens, block_size=16, hq=24, hkv=4, d=256,
                   k_type=spec.k_type, v_type=spec.v_type, sm_count=152, ctas_per_sm=1)


def test_headline_bytes():
    spec = synth.uniform_spec(8, 131072)
    pl = _plan(spec)
    nb = bench.algorithmic_bytes(spec, pl, fused=True, in_kernel_q=True)
    kv = 8 * 131072 * 4 * 2 * 144                 # tokens x heads x (K, V) x row bytes
    table = 8 * 131072 // 16 * 4                  # one int32 per block
    q = 8 * 24 * 256 * 4                          # the float32 query, read in the kernel
    parts = 8 * 19 * 24 * (2 * 256 + 8)           # f16 partials + (m, l), written and read
    out = 8 * 24 * 256 * 4
    lens = 8 * 4                                  # read by the decode and by the merge
    assert nb["kv"] == kv and nb["table"] == table and nb["prepass"] == 0
    assert nb["decode"] == kv + table + q + 2 * parts + out + 2 * lens
    assert nb["step"] == nb["decode"] == 1212408896


def test_direct_plan_bytes():
    spec = synth.uniform_spec(304, 4096)
    pl = _plan(spec)
    assert pl.direct
    nb = bench.algorithmic_bytes(spec, pl, fused=True, in_kernel_q=True)
    kv = 304 * 4096 * 4 * 2 * 144
    assert nb["decode"] == kv + 304 * 256 * 4 + 304 * 24 * 256 * 4 * 2 + 304 * 4


def test_wave_filling_plan_bytes():
    spec = synth.uniform_spec(160, 6912)
    pl = _plan(spec)
    assert (pl.n_direct, pl.n_parts, pl.part_tokens) == (152, 18, 384)
    nb = bench.algorithmic_bytes(spec, pl, fused=True, in_kernel_q=True)
    kv = 160 * 6912 * 4 * 2 * 144
    table = 160 * 6912 // 16 * 4
    q = 160 * 24 * 256 * 4
    parts = 8 * 18 * 24 * (2 * 256 + 8)           # only the 8 split rows have partials
    out = 160 * 24 * 256 * 4                      # 152 rows by the decode, 8 by the merge
    assert nb["decode"] == kv + table + q + 2 * parts + out + 2 * 160 * 4


def test_dram_record_is_consistent_with_its_workload():
    """The committed ncu DRAM record that bench.py reports as roofline.traffic:
    its plan is the planner's plan for the workload it names (152 SMs), and
    its bytes are the algorithmic bytes of that launch to ncu's three
    significant figures (every K/V byte read once).  bench.py reports it only
    while its source hash matches the kernel sources."""
    import json
    rec = json.load(open(os.path.join(bench.ROOT, "profiles", "decode_traffic.json")))
    assert rec["workload_name"] == "uniform-q4_0-b8x131072"
    spec = synth.uniform_spec(8, 131072)
    pl = _plan(spec)
    assert rec["plan"] == pl.as_dict()
    nb = bench.algorithmic_bytes(spec, pl, fused=True, in_kernel_q=True)["step"]
    assert abs(rec["dram_bytes_per_launch"] - nb) <= 0.005 * nb
    assert rec["dram_bytes_per_launch"] == rec["dram_bytes_read"] + rec["dram_bytes_write"]
    assert len(rec["source_sha"]) == 16

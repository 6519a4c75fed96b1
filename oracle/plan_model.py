"""Plain-Python model of the partition planner (test oracle).

"feat: add paged-attention monolithic decode-only AR foundation" (lucebox
pull 555), Summary, says only that context partitioning is occupancy-aware
and that the partials are merged by a stable split-softmax merge; Benchmark
results notes that short sequences in a ragged batch carry dead partitions
sized by the longest sequence.  The exact rule is this build's reading,
frozen here so that the C++ planner can be compared with it exactly:

- partitions are whole multiples of TILE = 32 tokens (so they start on a
  block boundary for block sizes 16 and 32);
- forced: part_tokens = roundup(ceil(max_len / force_parts), 32);
- otherwise the total live work is spread over the resident CTA slots:
  part_tokens = roundup(ceil(total_len / (sm_count * ctas_per_sm)), 32),
  at least MIN_PART = 128 tokens and at most roundup(max_len, 32); when the
  batch is nearly uniform (10 * total_len >= 9 * S * max_len), S <= slots,
  and S * ceil(max_len / part_tokens) would exceed the slots, it is instead
  roundup(ceil(max_len / floor(slots / S)), 32) within the same bounds, so
  that the CTAs fit one wave;
- then, if the partitions are still more than one per sequence, S < slots,
  and the grid bound min(S * n_parts, ceil(total_len / part_tokens) + S)
  (below) would exceed the slots, part_tokens grows to
  roundup(ceil(total_len / (slots - S)), 32) (at most roundup(max_len, 32)),
  so that the bound, and so the grid, fits one wave;
- n_parts = ceil(max_len / part_tokens) (partition slots per sequence, the
  partial buffers' second dimension); a sequence of length L has
  ceil(L / part_tokens) live partitions;
- a batch wider than the machine (S > slots) left direct by the above, with
  S = k * slots + r and r > 0, may split the r rows of its last wave: for
  np = 2 .. 64 (stopping where fewer than 2 partitions remain), part =
  max(128, roundup(ceil(max_len / np), 32)), nparts = ceil(max_len / part),
  the estimated time ceil(r * nparts / slots) * (part + CTA_COST) with
  CTA_COST = 512 tokens; the first strict minimum below max_len + CTA_COST
  (the time of leaving them whole) wins, and then the first n_direct =
  k * slots sequences stay direct (one CTA each) and the last r take
  part_tokens = part, n_parts = nparts; otherwise the plan stays direct.
  Every other plan has n_direct = 0;
- n_parts == 1 selects direct mode: no partials, the decode kernel writes
  the output itself;
- the decode grid has n_ctas = S in direct mode, otherwise n_direct +
  min(m * n_parts, ceil(total_len / part_tokens) + m) CTAs with m = S -
  n_direct (n_direct + m * n_parts for a wave-filling plan), an upper bound
  on the live (sequence, partition) pairs;
- an empty batch (max_len == 0) is direct with part_tokens = 32;
- partial buffers and counters cover the m partitioned sequences only:
  part_o_bytes = m * hq * n_parts * d * 2, part_ml_bytes = m * hq * n_parts
  * 8, and the fused merge keeps 1 + ceil(sqrt(n_parts)) int32 completion
  counters per such sequence (one for the last pass, one per group of the
  two-pass merge): counter_bytes = 4 * m * (1 + ceil(sqrt(n_parts))); all 0
  when direct;
- a stream plan (flags & STREAM_OK, no force_parts, max_len > 0, rows >
  sm_count * ctas_per_sm = slots, rows <= 16384, k_type == v_type, hkv in
  {1, 2, 4, 8}, d = 256 or F16): B = ceil((T * total_len + 15 * rows) / 16)
  tiles at most, chunk = roundup(ceil(B / slots), 2), part_tokens = 16 *
  chunk, n_parts = ceil(ceil(max_len / 16) / chunk) + 1 when that is <= 32
  (else the rules above), n_ctas = min(slots, ceil(B / chunk)), direct = 0,
  n_direct = 0, stream = 1, partials and counters for every row;
- a multi-token plan (flags & MULTI_TOKEN, T >= 2, Q4_0 K and V, d = 256,
  hkv in {1, 2, 4}, T * hq / hkv <= 24): the one-token plan of the
  sequences (a plan with direct rows becomes direct: part_tokens =
  roundup(max_len, 32), n_parts = 1, n_ctas = n_seqs) with multi = 1,
  q_tokens = T and partial buffers and counters for the n_seqs * T rows;
- with q_tokens = T > 1 (several query tokens per sequence, each a query
  row of its own that attends causally) the rule runs over the S * T query
  rows with T * total_len tokens of work: every S above reads S * T and
  total_len reads T * total_len.
"""
import math

TILE = 32
MIN_PART = 128
CTA_COST = 512  # a CTA's fixed work in tokens of streaming (wave-filling plans)
STREAM_OK = 1   # flags: the plan may be a stream plan
MULTI_TOKEN = 2  # flags: decode the T query tokens of a sequence together

OK, INVALID = 0, -1


def _cdiv(a: int, b: int) -> int:
    return -(-a // b)


def _roundup(a: int, b: int) -> int:
    return _cdiv(a, b) * b


def plan(*, n_seqs, max_len, total_len, block_size, hq, hkv, d, k_type, v_type,
         sm_count, ctas_per_sm, force_parts=0, q_tokens=1, flags=0):
    """Returns (rc, dict).  dict keys: part_tokens, n_parts, direct, n_ctas,
    part_o_bytes, part_ml_bytes, counter_bytes, q_tokens, n_direct, stream,
    multi."""
    if (n_seqs < 1 or block_size not in (16, 32) or hkv < 1 or hq < hkv or hq % hkv
            or hq // hkv > 8 or d not in (128, 256) or k_type not in (0, 1, 2)
            or v_type not in (0, 1, 2) or sm_count < 1 or ctas_per_sm < 1
            or force_parts < 0 or max_len < 0 or total_len < max_len
            or total_len > n_seqs * max_len):
        return INVALID, None
    T = max(1, q_tokens)
    if T > 4096:
        return INVALID, None
    if ((flags & MULTI_TOKEN) and T >= 2 and k_type == 2 and v_type == 2 and d == 256
            and hkv in (1, 2, 4) and T * (hq // hkv) <= 24):
        rc, b = plan(n_seqs=n_seqs, max_len=max_len, total_len=total_len,
                     block_size=block_size, hq=hq, hkv=hkv, d=d, k_type=k_type, v_type=v_type,
                     sm_count=sm_count, ctas_per_sm=ctas_per_sm, force_parts=force_parts)
        if rc != OK:
            return rc, None
        if b["n_direct"]:
            b.update(part_tokens=_roundup(max_len, TILE), n_parts=1, direct=1, n_direct=0,
                     n_ctas=n_seqs)
        rows, P = n_seqs * T, b["n_parts"]
        direct = b["direct"]
        b.update(q_tokens=T, multi=1,
                 part_o_bytes=0 if direct else rows * hq * P * d * 2,
                 part_ml_bytes=0 if direct else rows * hq * P * 8,
                 counter_bytes=0 if direct else 4 * rows * (1 + math.isqrt(P - 1) + 1))
        return OK, b
    rows, work = n_seqs * T, T * total_len   # query rows and their work at most
    n_direct = 0
    if max_len == 0:
        part, n_parts = TILE, 1
    elif force_parts > 0:
        part = _roundup(_cdiv(max_len, force_parts), TILE)
        n_parts = _cdiv(max_len, part)
    else:
        slots = sm_count * ctas_per_sm
        part = max(MIN_PART, _roundup(_cdiv(work, slots), TILE))
        part = min(part, _roundup(max_len, TILE))
        if (rows * _cdiv(max_len, part) > slots and rows <= slots
                and 10 * work >= 9 * rows * max_len):
            part = max(MIN_PART, _roundup(_cdiv(max_len, slots // rows), TILE))
            part = min(part, _roundup(max_len, TILE))
        np_ = _cdiv(max_len, part)
        if np_ > 1 and min(rows * np_, _cdiv(work, part) + rows) > slots and rows < slots:
            part = max(part, min(_roundup(_cdiv(work, slots - rows), TILE),
                                 _roundup(max_len, TILE)))
        n_parts = _cdiv(max_len, part)
        r = rows % slots
        if n_parts == 1 and rows > slots and r > 0:
            best_t, best_part = max_len + CTA_COST, 0
            for np_ in range(2, 65):
                pr = max(MIN_PART, _roundup(_cdiv(max_len, np_), TILE))
                nparts = _cdiv(max_len, pr)
                if nparts < 2:
                    break
                t = _cdiv(r * nparts, slots) * (pr + CTA_COST)
                if t < best_t:
                    best_t, best_part = t, pr
            if best_part:
                part, n_parts, n_direct = best_part, _cdiv(max_len, best_part), rows - r
    # a stream plan: equal ranges of the rows' 16-token tiles per CTA
    slots = sm_count * ctas_per_sm
    shapes = k_type == v_type and hkv in (1, 2, 4, 8) and (d == 256 or k_type == 0)
    if ((flags & STREAM_OK) and force_parts == 0 and max_len > 0 and rows > slots
            and rows <= 16384 and shapes):
        bound = _cdiv(work + 15 * rows, 16)
        chunk = _roundup(_cdiv(bound, slots), 2)
        np_ = _cdiv(_cdiv(max_len, 16), chunk) + 1
        if np_ <= 32:
            return OK, dict(part_tokens=16 * chunk, n_parts=np_, direct=0,
                            n_ctas=min(slots, _cdiv(bound, chunk)),
                            part_o_bytes=rows * hq * np_ * d * 2,
                            part_ml_bytes=rows * hq * np_ * 8,
                            counter_bytes=4 * rows * (1 + math.isqrt(np_ - 1) + 1),
                            q_tokens=T, n_direct=0, stream=1, multi=0)
    direct = 1 if n_parts == 1 else 0
    if direct:
        n_ctas = rows
        po = pm = cb = 0
    else:
        m = rows - n_direct
        n_ctas = n_direct + (m * n_parts if n_direct else
                             min(m * n_parts, _cdiv(work, part) + m))
        po = m * hq * n_parts * d * 2
        pm = m * hq * n_parts * 8
        cb = 4 * m * (1 + math.isqrt(n_parts - 1) + 1)
    return OK, dict(part_tokens=part, n_parts=n_parts, direct=direct, n_ctas=n_ctas,
                    part_o_bytes=po, part_ml_bytes=pm, counter_bytes=cb, q_tokens=T,
                    n_direct=n_direct, stream=0, multi=0)

"""Seeded synthetic inputs for paged decode attention.

This module is shared by the oracle side and the CUDA side of the tests and
of the benchmark; it holds none of the attention arithmetic.  It draws
source values, encodes them into the pool formats the method reads (the
encoders are input generation: the decode step only ever decodes), places
the blocks of each sequence in one pool through a shuffled block table, and
poisons every byte the decode step must never read.

Workload shapes follow the pages' measurements ("feat: add paged-attention
monolithic decode-only AR foundation", lucebox pull 555, Benchmark results:
Qwen attention dims D=256, Hq=24, Hkv=4, 16-token blocks, Q4_0 K/V, uniform
batches 1/2/4/8 x 4K/32K/128K and a ragged 128K + 7 x 8K batch;
"fix(paged-attention): use 64-bit pool offsets in the fused decode kernels",
mlxcel issue 2153, Acceptance Criteria: an f16 pool of [32, 8, 128] blocks
past 2^32 elements).  All values are N(0, 1) draws from torch generators
seeded per case; nothing is read from any dataset.

Formats (block = 32 values along the head dimension):
  F16   2 bytes per value, IEEE binary16;
  Q8_0  34 bytes: f16 scale d, 32 int8 q;            value q * d;
  Q4_0  18 bytes: f16 scale d, 16 bytes of nibbles;  value (nib - 8) * d,
        value j < 16 in the low nibble of byte j, value j + 16 in its high
        nibble (the ggml layout).
Pools are token-major: [n_blocks][block_size][hkv][row_bytes] bytes.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

F16, Q8_0, Q4_0 = 0, 1, 2
TYPE_NAMES = {"f16": F16, "q8_0": Q8_0, "q4_0": Q4_0}
TYPE_LABEL = {F16: "f16", Q8_0: "q8_0", Q4_0: "q4_0"}
POISON = 0xFF  # every byte 0xFF: an f16 NaN, and a NaN scale for Q8_0 / Q4_0


def row_bytes(type_: int, d: int) -> int:
    if d % 32:
        raise ValueError("d must be a multiple of 32")
    return {F16: 2 * d, Q8_0: d // 32 * 34, Q4_0: d // 32 * 18}[type_]


# -------------------------------------------------------------- encoders

def _f16_bytes(x: torch.Tensor) -> torch.Tensor:
    """float tensor [..., n] -> uint8 [..., 2n] little-endian f16 bytes."""
    return x.to(torch.float16).contiguous().view(torch.uint8)


def _round_half_away(x: torch.Tensor) -> torch.Tensor:
    return torch.sign(x) * torch.floor(torch.abs(x) + 0.5)


def encode_q8_0(x: torch.Tensor) -> torch.Tensor:
    """float32 [..., D] -> uint8 [..., D/32*34]: d = amax/127, q = round(x/d)."""
    shp = x.shape
    xb = x.reshape(-1, 32).to(torch.float32)
    amax = xb.abs().amax(dim=1, keepdim=True)
    d = amax / 127.0
    inv = torch.where(d > 0, 1.0 / d, torch.zeros_like(d))
    q = _round_half_away(xb * inv).clamp(-127, 127).to(torch.int8)
    out = torch.cat([_f16_bytes(d), q.view(torch.uint8)], dim=1)
    return out.reshape(*shp[:-1], shp[-1] // 32 * 34)


def encode_q4_0(x: torch.Tensor) -> torch.Tensor:
    """float32 [..., D] -> uint8 [..., D/32*18] in the ggml Q4_0 convention:
    m = the value of largest magnitude (with its sign), d = m / -8,
    nib = min(15, floor(x / d + 8.5)); low nibbles hold values 0..15 of the
    block, high nibbles values 16..31."""
    shp = x.shape
    xb = x.reshape(-1, 32).to(torch.float32)
    idx = xb.abs().argmax(dim=1, keepdim=True)
    m = torch.gather(xb, 1, idx)
    d = m / -8.0
    inv = torch.where(d != 0, 1.0 / d, torch.zeros_like(d))
    nib = torch.clamp(torch.floor(xb * inv + 8.5), 0, 15).to(torch.uint8)
    packed = nib[:, :16] | (nib[:, 16:] << 4)
    out = torch.cat([_f16_bytes(d), packed], dim=1)
    return out.reshape(*shp[:-1], shp[-1] // 32 * 18)


def encode(x: torch.Tensor, type_: int) -> torch.Tensor:
    if type_ == F16:
        return _f16_bytes(x)
    if type_ == Q8_0:
        return encode_q8_0(x)
    if type_ == Q4_0:
        return encode_q4_0(x)
    raise ValueError(type_)


def source_values(gen: torch.Generator, shape, device, outliers: bool) -> torch.Tensor:
    """N(0,1) float32; with outliers, each value independently x8 with p=0.01."""
    x = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    if outliers:
        mask = torch.rand(shape, generator=gen, device=device) < 0.01
        x = torch.where(mask, x * 8.0, x)
    return x


# ------------------------------------------------------------------ cases

@dataclass
class CaseSpec:
    """One synthetic decode-step workload."""
    seq_lens: list
    d: int = 256
    hq: int = 24
    hkv: int = 4
    block_size: int = 16
    k_type: int = Q4_0
    v_type: int = Q4_0
    n_pool_blocks: int | None = None  # None: the used blocks plus `junk` spare ones
    junk: int = 0
    layout: str = "shuffled"          # "shuffled" | "identity"
    outliers: bool = False
    force_last_block: bool = False    # make the pool's final block one of the used ones
    name: str = ""
    extra: dict = field(default_factory=dict)

    @property
    def n_seqs(self) -> int:
        return len(self.seq_lens)

    def blocks_per_seq(self):
        return [math.ceil(L / self.block_size) for L in self.seq_lens]


@dataclass
class Case:
    spec: CaseSpec
    k_pool: torch.Tensor       # uint8 [n_blocks, B, hkv, krb]
    v_pool: torch.Tensor       # uint8 [n_blocks, B, hkv, vrb]
    block_table: torch.Tensor  # int32 [S, stride]; unused entries are -1
    seq_lens: torch.Tensor     # int32 [S]
    q: torch.Tensor            # float32 [S, hq, d]
    seed: int

    @property
    def n_blocks(self) -> int:
        return self.k_pool.shape[0]


def _fill_rows(pool, ids, spec, type_, gen, device, chunk):
    """Encode fresh source rows into pool blocks `ids` (a 1-D long tensor)."""
    B, hkv, d = spec.block_size, spec.hkv, spec.d
    for i in range(0, ids.numel(), chunk):
        sel = ids[i:i + chunk]
        x = source_values(gen, (sel.numel(), B, hkv, d), device, spec.outliers)
        pool[sel] = encode(x, type_).reshape(sel.numel(), B, hkv, -1)


def build_case(spec: CaseSpec, seed: int, device="cpu", chunk_blocks: int = 2048) -> Case:
    """Generate pools, block table, lengths and Q for `spec` on `device`.

    Used blocks get fresh encoded N(0,1) rows; spare (junk) blocks and the
    slots past each sequence's length in its last block are poisoned with
    0xFF bytes (NaN), so that any read the decode step must not make shows
    up as NaN in its output.  Table entries past a sequence's last block are
    -1 (outside the pool)."""
    device = torch.device(device)
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    S, B = spec.n_seqs, spec.block_size
    nbs = spec.blocks_per_seq()
    used = sum(nbs)
    n_blocks = spec.n_pool_blocks if spec.n_pool_blocks is not None else used + spec.junk
    if n_blocks < used:
        raise ValueError("pool too small")
    stride = max(1, max(nbs) if nbs else 1)
    krb, vrb = row_bytes(spec.k_type, spec.d), row_bytes(spec.v_type, spec.d)
    k_pool = torch.full((n_blocks, B, spec.hkv, krb), POISON, dtype=torch.uint8, device=device)
    v_pool = torch.full((n_blocks, B, spec.hkv, vrb), POISON, dtype=torch.uint8, device=device)

    if spec.layout == "identity":
        # sequence s owns blocks s*stride .. s*stride + nbs[s] - 1
        ids = torch.cat([torch.arange(s * stride, s * stride + nbs[s], dtype=torch.long)
                         for s in range(S)]) if used else torch.zeros(0, dtype=torch.long)
        if n_blocks < S * stride:
            raise ValueError("identity layout needs S * stride blocks")
    else:
        perm = torch.randperm(n_blocks, generator=torch.Generator().manual_seed(seed ^ 0x5EED))
        ids = perm[:used].clone()
        if spec.force_last_block and used and not bool((ids == n_blocks - 1).any()):
            ids[-1] = n_blocks - 1
    table = torch.full((S, stride), -1, dtype=torch.int32)
    off = 0
    for s in range(S):
        table[s, :nbs[s]] = ids[off:off + nbs[s]].to(torch.int32)
        off += nbs[s]
    ids_dev = ids.to(device)
    _fill_rows(k_pool, ids_dev, spec, spec.k_type, gen, device, chunk_blocks)
    _fill_rows(v_pool, ids_dev, spec, spec.v_type, gen, device, chunk_blocks)
    # poison the tail slots of each sequence's last block
    for s in range(S):
        L = spec.seq_lens[s]
        if L % B:
            last = int(table[s, nbs[s] - 1])
            k_pool[last, L % B:] = POISON
            v_pool[last, L % B:] = POISON
    # T query tokens per sequence (spec.extra["q_tokens"]): q is [S, T, hq, d]
    T = int(spec.extra.get("q_tokens", 1))
    q = source_values(gen, (S, spec.hq, spec.d) if T == 1 else (S, T, spec.hq, spec.d), device,
                      False)
    lens = torch.tensor(spec.seq_lens, dtype=torch.int32)
    return Case(spec=spec, k_pool=k_pool, v_pool=v_pool, block_table=table.to(device),
                seq_lens=lens.to(device), q=q, seed=seed)


def contiguous_twin(case: Case) -> Case:
    """The same workload in the contiguous layout: sequence s occupies pool
    blocks s*stride .. s*stride+stride-1 in order (identity table), with the
    same bytes in every used slot; blocks past a sequence's end are poison."""
    spec = case.spec
    S, stride = case.block_table.shape
    dev = case.k_pool.device
    kc = torch.full((S * stride,) + tuple(case.k_pool.shape[1:]), POISON, dtype=torch.uint8,
                    device=dev)
    vc = torch.full((S * stride,) + tuple(case.v_pool.shape[1:]), POISON, dtype=torch.uint8,
                    device=dev)
    bt = case.block_table.to("cpu")
    table = torch.full((S, stride), -1, dtype=torch.int32)
    for s, nb in enumerate(spec.blocks_per_seq()):
        if nb:
            src = bt[s, :nb].to(torch.long).to(dev)
            dst = torch.arange(s * stride, s * stride + nb, dtype=torch.long, device=dev)
            kc[dst] = case.k_pool[src]
            vc[dst] = case.v_pool[src]
            table[s, :nb] = torch.arange(s * stride, s * stride + nb, dtype=torch.int32)
    spec2 = CaseSpec(**{**spec.__dict__, "layout": "identity", "n_pool_blocks": S * stride,
                        "junk": 0})
    return Case(spec=spec2, k_pool=kc, v_pool=vc, block_table=table.to(dev),
                seq_lens=case.seq_lens.clone(), q=case.q.clone(), seed=case.seed)


def gather_sequences(case: Case, seqs) -> Case:
    """A compact copy holding only the blocks of the listed sequences, in
    table order, for evaluating sampled outputs of a large case on the host.
    Returns a CPU Case whose sequence i is case's sequence seqs[i]."""
    spec = case.spec
    bt = case.block_table.to("cpu")
    nbs = spec.blocks_per_seq()
    parts_k, parts_v, lens = [], [], []
    stride = max(1, max(nbs[s] for s in seqs))
    table = torch.full((len(seqs), stride), -1, dtype=torch.int32)
    base = 0
    for i, s in enumerate(seqs):
        nb = nbs[s]
        src = bt[s, :nb].to(torch.long).to(case.k_pool.device)
        parts_k.append(case.k_pool.index_select(0, src).cpu())
        parts_v.append(case.v_pool.index_select(0, src).cpu())
        table[i, :nb] = torch.arange(base, base + nb, dtype=torch.int32)
        base += nb
        lens.append(spec.seq_lens[s])
    spec2 = CaseSpec(**{**spec.__dict__, "seq_lens": lens, "layout": "identity",
                        "n_pool_blocks": base, "junk": 0})
    return Case(spec=spec2, k_pool=torch.cat(parts_k), v_pool=torch.cat(parts_v),
                block_table=table, seq_lens=torch.tensor(lens, dtype=torch.int32),
                q=case.q[list(seqs)].cpu(), seed=case.seed)


# ----------------------------------------------------- the pages' workloads

def tiny_spec() -> CaseSpec:
    """1 sequence of 200 tokens (12 full blocks + 8 slots), F16 K/V, D=256,
    Hq=24, Hkv=4, 16-token blocks, the 13 used blocks shuffled among 19
    poisoned junk blocks in a 32-block pool."""
    return CaseSpec(seq_lens=[200], k_type=F16, v_type=F16, n_pool_blocks=32,
                    name="tiny-f16-L200")


def uniform_spec(batch: int, ctx: int, type_: int = Q4_0) -> CaseSpec:
    """Uniform batch at Qwen attention dims: every sequence `ctx` tokens; the
    pool holds exactly the used blocks, interleaved by a random permutation."""
    return CaseSpec(seq_lens=[ctx] * batch, k_type=type_, v_type=type_,
                    name=f"uniform-{TYPE_LABEL[type_]}-b{batch}x{ctx}")


def ragged_spec(type_: int = Q4_0) -> CaseSpec:
    """One 131072-token and seven 8192-token sequences, one shuffled pool."""
    return CaseSpec(seq_lens=[131072] + [8192] * 7, k_type=type_, v_type=type_,
                    name=f"ragged-{TYPE_LABEL[type_]}-128k+7x8k")


def dtype_sweep_spec(type_: int, short: bool = False, v_type: int | None = None) -> CaseSpec:
    """Batch 4 x 32768 (or the short ragged 4096 + 7 x 256), N(0,1) values
    with 1% outliers at x8; V of type v_type when given (a mixed pair)."""
    lens = [4096] + [256] * 7 if short else [32768] * 4
    tag = "short" if short else "b4x32k"
    vt = type_ if v_type is None else v_type
    pair = TYPE_LABEL[type_] if vt == type_ else f"{TYPE_LABEL[type_]}-{TYPE_LABEL[vt]}"
    return CaseSpec(seq_lens=lens, k_type=type_, v_type=vt, outliers=True,
                    name=f"sweep-{pair}-{tag}")


def verify_spec(n_seqs: int = 8, ctx: int = 32768, T: int = 4, type_: int = Q4_0) -> CaseSpec:
    """A verify window: T query tokens per sequence (token i at position
    ctx - T + i attends to the keys up to its own position) over uniform
    contexts, Q4_0 K/V at the Qwen attention dims."""
    return CaseSpec(seq_lens=[ctx] * n_seqs, k_type=type_, v_type=type_,
                    name=f"verify-{TYPE_LABEL[type_]}-b{n_seqs}x{ctx}-T{T}", extra={"q_tokens": T})


def large_pool_spec(n_seqs: int = 16, ctx: int = 300_000) -> CaseSpec:
    """Llama-style D=128, Hq=32, Hkv=8, 32-token blocks, F16: a slab of
    163,840 blocks per side (5,368,709,120 elements, past 2^32), 16 x 300,000
    tokens drawn from a random permutation, the final block forced in use."""
    return CaseSpec(seq_lens=[ctx] * n_seqs, d=128, hq=32, hkv=8, block_size=32,
                    k_type=F16, v_type=F16, n_pool_blocks=163_840, force_last_block=True,
                    name=f"largepool-f16-b{n_seqs}x{ctx}")

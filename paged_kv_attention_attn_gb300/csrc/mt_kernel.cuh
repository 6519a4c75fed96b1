// mt_kernel.cuh -- the query tokens of a sequence decoded together (Q4_0 K/V,
// D = 256): a verify window or a prompt chunk of T tokens over one paged
// cache ("TensorFold pull 1418", What: several query rows per sequence over
// one paged cache).
//
// The one-token kernel runs such a plan as T independent query rows, so
// every K/V row is dequantised and multiplied T times.  Here the T * G query
// columns of a K/V head (token i, head j as column i * G + j, at most 24:
// three n-tiles of the MMA) share one pass: each 16-token tile's nibbles are
// expanded once and feed all columns.  The accumulator of 24 columns does not
// fit one warp, so a pair of warps serves each K/V head and splits the head
// dimension: warp half h takes the 32-value blocks 4h .. 4h+3 (dims 128h ..
// 128h + 127) for both products.  Per tile the pair adds its two partial
// scores through shared memory (each warp then holds the full scores and
// runs the same softmax), and each warp keeps O for its own dims, so at the
// end each writes its half of every column's row directly: no combine.
// Query token i (row seq * T + i) sees keys < L - T + 1 + i (causal).  The
// pair shares one TMA ring; the slot of tile k - 1 is refilled once both
// warps have passed tile k's score exchange.  Partials go through pa_merge's
// kernel.
#pragma once

#include "fast_kernel.cuh"

namespace pa {
namespace {

constexpr uint32_t kMtMaxCols = 24;  // T * G at most: three n-tiles
constexpr int kMtNT = 3;
constexpr int kMtHalfBlocks = 4;     // 32-value blocks per warp half (D = 256)

// Shared-memory layout after the 1024-byte aligned base (hkv pairs, nsw
// slots per pair).
struct MtLayout {
    uint32_t nsw, rings, qb, qc, xch, scr, ok, bars, total;
};

__host__ __device__ inline MtLayout mt_layout(uint32_t hkv, uint32_t nsw)
{
    MtLayout l;
    l.nsw = nsw;
    l.rings = 0;                                               // [hkv][nsw] Q40 slots
    l.qb = hkv * nsw * Q40::kSlot;                             // [hkv][3][8][32] uint4
    l.qc = l.qb + hkv * kMtNT * 8 * 32 * 16;                   // [hkv][3][8][32] float2
    l.xch = l.qc + hkv * kMtNT * 8 * 32 * 8;                   // [2][2 hkv][32][12] float
    l.scr = l.xch + 2 * (2 * hkv) * 32 * 12 * 4;               // [2 hkv] dk f32, dv f16
    l.ok = l.scr + (2 * hkv) * kMtHalfBlocks * kTile * 6;      // [hkv][nsw] int
    l.bars = (l.ok + hkv * nsw * 4 + 7) & ~7u;                 // [hkv][nsw] mbarriers
    l.total = l.bars + hkv * nsw * 8;
    return l;
}

// The slots per pair that fit kSmemBudget (at most 8), 0 if fewer than 2.
__host__ inline uint32_t mt_slots(uint32_t hkv)
{
    for (uint32_t nsw = 8; nsw >= 2; --nsw)
        if (1024 + mt_layout(hkv, nsw).total <= kSmemBudget)
            return nsw;
    return 0;
}

__device__ __forceinline__ void pair_sync(uint32_t id)
{
    asm volatile("bar.sync %0, 64;" ::"r"(id) : "memory");
}

__global__ void __launch_bounds__(256, 1) mt_decode_kernel(const __grid_constant__ FastArgs a)
{
    const DecodeParams &p = a.p;
    extern __shared__ __align__(16) uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t hkv = p.hkv, G = p.hq / hkv, T = p.q_tokens, NC = T * G;
    const uint32_t NSW = a.n_slots, SLOT = Q40::kSlot, VOFF = Q40::kSideK;
    const MtLayout lay = mt_layout(hkv, NSW);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, gid = lane >> 2, tig = lane & 3;
    const uint32_t g = (uint32_t)warp >> 1, half = (uint32_t)warp & 1;
    const uint32_t base_u = smem_u32(smem);
    uint8_t *ring = smem + lay.rings + (size_t)g * NSW * SLOT;
    const uint32_t ring_u = smem_u32(ring);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + lay.bars) + g * NSW;
    int *slot_ok = reinterpret_cast<int *>(smem + lay.ok) + g * NSW;
    const uint32_t qb_u = base_u + lay.qb + (g * kMtNT * 8 * 32) * 16;
    const uint32_t qc_u = base_u + lay.qc + (g * kMtNT * 8 * 32) * 8;
    float *xch = reinterpret_cast<float *>(smem + lay.xch);
    const uint32_t scr_u = base_u + lay.scr + (uint32_t)warp * kMtHalfBlocks * kTile * 6;
    constexpr uint32_t DK = 0, DV = kMtHalfBlocks * kTile * 4;  // dk f32 [4][16], dv f16 [4][16]

    __shared__ bool s_bad[2][8];  // per tile parity and warp: a wait that ran out
    if (half == 0 && lane == 0) {
        for (uint32_t s = 0; s < NSW; ++s)
            mbar_init(&full[s], 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    grid_dependency_wait();

    // this CTA's (sequence, partition): the last query token's length L
    // decides the partitions (its keys include every other token's)
    const uint32_t S = p.n_seqs / T;
    uint32_t seq, part;
    if (!p.direct && blockIdx.x == gridDim.x - 1 && warp == 0)
        check_grid_vs_plan(p.seq_lens, 1, S, p.part_tokens, p.n_parts, 0, p.status);
    if (p.direct) {
        seq = blockIdx.x;
        part = 0;
    } else if (!cta_work(p.seq_lens, 1, S, p.part_tokens, p.n_parts, 0, blockIdx.x, &seq,
                         &part)) {
        return;
    }
    const int32_t Ls = p.seq_lens[seq];
    const uint32_t L = Ls > 0 ? (uint32_t)Ls : 0u;
    if (!p.direct && part == 0 && tid == 0)
        check_len_vs_plan(Ls, p.n_parts, p.part_tokens, p.status);
    const uint32_t t0 = p.direct ? 0u : part * p.part_tokens;
    const uint32_t t1 = p.direct ? L : min(L, t0 + p.part_tokens);
    const uint32_t n_tiles = t1 > t0 ? (t1 - t0 + kTile - 1) / kTile : 0u;
    const int32_t *bt = p.block_table + (uint64_t)seq * p.table_stride;
    const CUtensorMap *tmk = &a.tm[0][g], *tmv = &a.tm[1][g];
    const uint32_t bshift = p.block_size == 32 ? 5 : 4, bmask = p.block_size - 1;

    // half 0, lane 0: start the copy of tile k (block id blk) into slot s
    auto issue = [&](uint32_t k, uint32_t s, int32_t blk) {
        const uint32_t tok = t0 + kTile * k;
        const bool ok = block_in_pool(blk, p.n_pool_blocks);
        slot_ok[s] = ok;
        if (ok) {
            uint8_t *dst = ring + (size_t)s * SLOT;
            const int y = (blk << bshift) + (int)(tok & bmask);
            fence_proxy_async();
            const uint64_t pol = l2_evict_first_policy();
            mbar_arrive_expect_tx(&full[s], SLOT);
            tma_load_2d_hint(dst, tmk, 0, y, &full[s], pol);
            tma_load_2d_hint(dst + VOFF, tmv, 0, y, &full[s], pol);
        } else {
            atomicOr(p.status, PA_STATUS_CORRUPT_TABLE);
            mbar_arrive(&full[s]);
        }
    };
    auto tile_block = [&](uint32_t k) -> int32_t {
        return k < n_tiles ? bt[(t0 + kTile * k) >> bshift] : 0;
    };
    const uint32_t pro = n_tiles < NSW ? n_tiles : NSW;
    if (half == 0) {
        const int32_t b = tile_block(lane);  // tiles 0 .. 31 (pro <= 8)
        for (uint32_t k = 0; k < pro; ++k) {
            const int32_t bk = __shfl_sync(0xffffffffu, b, k);
            if (lane == 0)
                issue(k, k, bk);
        }
        __syncwarp();
    }

    // query fragments of my blocks for all three n-tiles: column c = nt * 8 +
    // gid is token c / G, head c % G of the group (q8_1 from the pre-pass)
    for (int nt = 0; nt < kMtNT; ++nt) {
        const uint32_t c = nt * 8 + gid;
        const bool live = c < NC;
        const uint32_t i = live ? c / G : 0u, j = live ? c % G : 0u;
        const uint8_t *qrow = static_cast<const uint8_t *>(p.q) +
                              (((uint64_t)seq * T + i) * p.hq + g * G + j) * (8 * 36);
#pragma unroll
        for (int bb = 0; bb < kMtHalfBlocks; ++bb) {
            const int b = (int)half * kMtHalfBlocks + bb;
            const uint8_t *blk = qrow + 36 * b;
            const uint32_t w0 = *reinterpret_cast<const uint32_t *>(blk + 4 + 4 * tig);
            const uint32_t w1 = *reinterpret_cast<const uint32_t *>(blk + 20 + 4 * tig);
            const float d = live ? half_bits_to_float(load_u16(blk)) * p.scale_log2 : 0.0f;
            __half qh[8];
            float corr = 0.0f;
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int code = (int)(int8_t)(uint8_t)((e < 4 ? w0 : w1) >> (8 * (e & 3)));
                qh[e] = __float2half_rn((float)code * d);
                // low nibbles read as 1024 + n, high as 64 + n; the value is n - 8
                corr += __half2float(qh[e]) * (e < 4 ? 1032.0f : 72.0f);
            }
            corr += __shfl_xor_sync(0xffffffffu, corr, 1);
            corr += __shfl_xor_sync(0xffffffffu, corr, 2);
            const float n0 = -__shfl_sync(0xffffffffu, corr, 8 * tig);
            const float n1 = -__shfl_sync(0xffffffffu, corr, 8 * tig + 4);
            const uint32_t rec = (uint32_t)((nt * 8 + b) * 32 + lane);
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(qb_u + rec * 16),
                         "r"(h2_bits(__halves2half2(qh[0], qh[2]))),
                         "r"(h2_bits(__halves2half2(qh[1], qh[3]))),
                         "r"(h2_bits(__halves2half2(qh[4], qh[6]))),
                         "r"(h2_bits(__halves2half2(qh[5], qh[7]))));
            asm volatile("st.shared.v2.f32 [%0], {%1, %2};" ::"r"(qc_u + rec * 8), "f"(n0),
                         "f"(n1));
        }
    }
    __syncwarp();  // each warp reads only the records it wrote

    // per column of mine (n-tile nt, column 2 tig + e): the causal limit
    uint32_t lim[kMtNT][2];
#pragma unroll
    for (int nt = 0; nt < kMtNT; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const uint32_t c = nt * 8 + 2 * tig + e;
            const int64_t li = c < NC ? (int64_t)L - T + 1 + c / G : 0;
            lim[nt][e] = li > 0 ? (uint32_t)li : 0u;
        }

    NibbleConsts K;
    K.init();
    float o[2 * kMtHalfBlocks][kMtNT][4];
#pragma unroll
    for (int mt = 0; mt < 2 * kMtHalfBlocks; ++mt)
#pragma unroll
        for (int nt = 0; nt < kMtNT; ++nt)
            o[mt][nt][0] = o[mt][nt][1] = o[mt][nt][2] = o[mt][nt][3] = 0.0f;
    float mref[kMtNT][2], lsum[kMtNT][2];
#pragma unroll
    for (int nt = 0; nt < kMtNT; ++nt)
        mref[nt][0] = mref[nt][1] = -INFINITY, lsum[nt][0] = lsum[nt][1] = 0.0f;
    bool aborted = false;
    uint32_t issued = pro;
    int32_t ids = half == 0 ? tile_block(NSW + lane) : 0;  // tiles NSW .. NSW + 31
    uint32_t ids_base = NSW;

    for (uint32_t k = 0; k < n_tiles; ++k) {
        const uint32_t s = k % NSW, phase = (k / NSW) & 1u;
        bool done = mbar_try_wait(&full[s], phase);
        if (!done) {
            const uint64_t tw = global_ns();
            while (!(done = mbar_try_wait(&full[s], phase)) && global_ns() - tw < kWaitNs) {
            }
        }
        // a pair abandons its tiles together, after this tile's exchange
        // (the partner must not wait on an exchange that will not come)
        bool bad = !__all_sync(0xffffffffu, done);
        if (bad && lane == 0)
            atomicOr(p.status, PA_STATUS_TIMEOUT);
        const uint32_t ks = t0 + kTile * k;
        const int nvalid = slot_ok[s] ? (int)min(16u, t1 - ks) : 0;
        const uint32_t kh = ring_u + s * SLOT, vh = kh + VOFF;
        // block scales of my blocks: dk as float (pair t, t+8 adjacent), dv as half
        {
            const int t = lane & 15, b0 = lane >> 4;
            const bool v = t < nvalid && !bad;
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                const int bb = b0 + 2 * r, b = (int)half * kMtHalfBlocks + bb;
                const uint32_t kd = lds_u16(kh + t * Q40::RB + 18 * b);
                const uint32_t vd = lds_u16(vh + t * Q40::RB + 18 * b);
                sts_f32(scr_u + DK + 4 * (bb * kTile + 2 * (t & 7) + (t >> 3)),
                        v ? half_bits_to_float((uint16_t)kd) : 0.0f);
                sts_u16(scr_u + DV + 2 * (bb * kTile + t), v ? vd : 0u);
            }
        }
        __syncwarp();
        // partial scores over my blocks, all three n-tiles
        float sc[kMtNT][4];
#pragma unroll
        for (int nt = 0; nt < kMtNT; ++nt)
            sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.0f;
        {
            uint32_t r0 = kh + gid * Q40::RB + 4 * tig + 36 * (2 * half);
#pragma unroll
            for (int pb = 0; pb < 2; ++pb) {
                const uint32_t a0 = lds_u32(r0), a1 = lds_u32(r0 + 4), a2 = lds_u32(r0 + 20);
                const uint32_t b0 = lds_u32(r0 + 8 * Q40::RB), b1 = lds_u32(r0 + 8 * Q40::RB + 4);
                const uint32_t b2 = lds_u32(r0 + 8 * Q40::RB + 20);
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    const int bb = 2 * pb + q, b = (int)half * kMtHalfBlocks + bb;
                    const uint32_t x0 = q ? a2 : __funnelshift_r(a0, a1, 16);
                    const uint32_t x1 = q ? b2 : __funnelshift_r(b0, b1, 16);
                    const uint32_t y0 = x0 >> 8, y1 = x1 >> 8;
                    const uint32_t lo0 = and_or(x0, K.mlo, K.blo), lo1 = and_or(x1, K.mlo, K.blo);
                    const uint32_t lo2 = and_or(y0, K.mlo, K.blo), lo3 = and_or(y1, K.mlo, K.blo);
                    const uint32_t hi0 = and_or(x0, K.mhi, K.bhi), hi1 = and_or(x1, K.mhi, K.bhi);
                    const uint32_t hi2 = and_or(y0, K.mhi, K.bhi), hi3 = and_or(y1, K.mhi, K.bhi);
                    const float2 dk = lds_f2(scr_u + DK + 4 * (bb * kTile + 2 * gid));
#pragma unroll
                    for (int nt = 0; nt < kMtNT; ++nt) {
                        const uint32_t rec = (uint32_t)((nt * 8 + b) * 32 + lane);
                        uint32_t qb0, qb1, qb2, qb3;
                        asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                                     : "=r"(qb0), "=r"(qb1), "=r"(qb2), "=r"(qb3)
                                     : "r"(qb_u + rec * 16));
                        const float2 cc = lds_f2(qc_u + rec * 8);
                        float c[4] = {cc.x, cc.y, cc.x, cc.y};
                        mma16816(c, lo0, lo1, lo2, lo3, qb0, qb1);
                        mma16816(c, hi0, hi1, hi2, hi3, qb2, qb3);
                        sc[nt][0] = fmaf(c[0], dk.x, sc[nt][0]);
                        sc[nt][1] = fmaf(c[1], dk.x, sc[nt][1]);
                        sc[nt][2] = fmaf(c[2], dk.y, sc[nt][2]);
                        sc[nt][3] = fmaf(c[3], dk.y, sc[nt][3]);
                    }
                }
                r0 += 36;
            }
        }
        // the pair adds its two halves (a + b == b + a: both warps hold the
        // same full scores)
        {
            float *mine = xch + (((k & 1u) * (2 * hkv) + (uint32_t)warp) * 32 + lane) * 12;
            const float *other = xch + (((k & 1u) * (2 * hkv) + ((uint32_t)warp ^ 1u)) * 32 + lane) * 12;
#pragma unroll
            for (int nt = 0; nt < kMtNT; ++nt)
                *reinterpret_cast<float4 *>(mine + 4 * nt) =
                    make_float4(sc[nt][0], sc[nt][1], sc[nt][2], sc[nt][3]);
            if (lane == 0)
                s_bad[k & 1u][warp] = bad;
            pair_sync(1 + g);
#pragma unroll
            for (int nt = 0; nt < kMtNT; ++nt) {
                const float4 v = *reinterpret_cast<const float4 *>(other + 4 * nt);
                sc[nt][0] += v.x;
                sc[nt][1] += v.y;
                sc[nt][2] += v.z;
                sc[nt][3] += v.w;
            }
            bad = s_bad[k & 1u][warp] || s_bad[k & 1u][warp ^ 1];
        }
        // both warps are past tile k - 1: refill its slot
        if (half == 0 && k >= 1 && k - 1 + NSW < n_tiles && !bad) {
            const uint32_t kn = k - 1 + NSW;
            if (kn - ids_base >= 32) {
                ids_base += 32;
                ids = tile_block(ids_base + lane);
            }
            const int32_t b = __shfl_sync(0xffffffffu, ids, kn - ids_base);
            if (lane == 0)
                issue(kn, (k - 1) % NSW, b);
            issued = kn + 1;
        }
        if (bad) {
            aborted = true;
            break;
        }
        // causal and length masks per column
#pragma unroll
        for (int nt = 0; nt < kMtNT; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const uint32_t t = ks + gid + 8 * (e >> 1);
                const bool ok = (int)(gid + 8 * (e >> 1)) < nvalid && t < lim[nt][e & 1];
                if (!ok)
                    sc[nt][e] = -INFINITY;
            }
        // online softmax per column (log2 domain, reference maximum)
        bool over = false;
#pragma unroll
        for (int nt = 0; nt < kMtNT; ++nt)
            over = over || fmaxf(sc[nt][0], sc[nt][2]) > mref[nt][0] ||
                   fmaxf(sc[nt][1], sc[nt][3]) > mref[nt][1];
        if (__builtin_expect(__any_sync(0xffffffffu, over), 0)) {
#pragma unroll
            for (int nt = 0; nt < kMtNT; ++nt) {
                float m0 = fmaxf(sc[nt][0], sc[nt][2]), m1 = fmaxf(sc[nt][1], sc[nt][3]);
#pragma unroll
                for (int off = 4; off < 32; off <<= 1) {
                    m0 = fmaxf(m0, __shfl_xor_sync(0xffffffffu, m0, off));
                    m1 = fmaxf(m1, __shfl_xor_sync(0xffffffffu, m1, off));
                }
                const float n0 = m0 > mref[nt][0] ? m0 + kHeadroom : mref[nt][0];
                const float n1 = m1 > mref[nt][1] ? m1 + kHeadroom : mref[nt][1];
                const float a0 = mref[nt][0] == -INFINITY ? 0.0f : exp2f(mref[nt][0] - n0);
                const float a1 = mref[nt][1] == -INFINITY ? 0.0f : exp2f(mref[nt][1] - n1);
#pragma unroll
                for (int mt = 0; mt < 2 * kMtHalfBlocks; ++mt) {
                    o[mt][nt][0] *= a0;
                    o[mt][nt][1] *= a1;
                    o[mt][nt][2] *= a0;
                    o[mt][nt][3] *= a1;
                }
                lsum[nt][0] *= a0;
                lsum[nt][1] *= a1;
                mref[nt][0] = n0;
                mref[nt][1] = n1;
            }
        }
        uint32_t pp[kMtNT][2];
#pragma unroll
        for (int nt = 0; nt < kMtNT; ++nt) {
            const float ms0 = mref[nt][0] == -INFINITY ? 0.0f : mref[nt][0];
            const float ms1 = mref[nt][1] == -INFINITY ? 0.0f : mref[nt][1];
            const float q00 = exp2f(sc[nt][0] - ms0), q01 = exp2f(sc[nt][1] - ms1);
            const float q10 = exp2f(sc[nt][2] - ms0), q11 = exp2f(sc[nt][3] - ms1);
            lsum[nt][0] += q00 + q10;
            lsum[nt][1] += q01 + q11;
            pp[nt][0] = movmatrix_t(h2_bits(__floats2half2_rn(q00, q01)));
            pp[nt][1] = movmatrix_t(h2_bits(__floats2half2_rn(q10, q11)));
        }
        // PV over my blocks: the V operand (n - 8, exact) is expanded once for
        // all three n-tiles; d_v is folded into P per block
        {
            const uint32_t ra = vh + (2 * tig) * Q40::RB + 2 + 2 * gid;
            const uint32_t rc = ra + 8 * Q40::RB;
#pragma unroll
            for (int bb = 0; bb < kMtHalfBlocks; ++bb) {
                const int b = (int)half * kMtHalfBlocks + bb;
                const uint32_t ua = lds_u16(ra + 18 * b), ub = lds_u16(ra + Q40::RB + 18 * b);
                const uint32_t uc = lds_u16(rc + 18 * b), ud = lds_u16(rc + Q40::RB + 18 * b);
                const uint32_t xab = __byte_perm(ua, ub, 0x5410), yab = xab >> 8;
                const uint32_t xcd = __byte_perm(uc, ud, 0x5410), ycd = xcd >> 8;
                const uint32_t dva = lds_u32(scr_u + DV + 2 * (bb * kTile + 2 * tig));
                const uint32_t dvb = lds_u32(scr_u + DV + 2 * (bb * kTile + 8 + 2 * tig));
                const uint32_t l0 = hadd2_bits(and_or(xab, K.mlo, K.blo), K.nlo[0]);
                const uint32_t l1 = hadd2_bits(and_or(yab, K.mlo, K.blo), K.nlo[1]);
                const uint32_t l2 = hadd2_bits(and_or(xcd, K.mlo, K.blo), K.nlo[2]);
                const uint32_t l3 = hadd2_bits(and_or(ycd, K.mlo, K.blo), K.nlo[3]);
                const uint32_t h0 = hadd2_bits(and_or(xab, K.mhi, K.bhi), K.nhi[0]);
                const uint32_t h1 = hadd2_bits(and_or(yab, K.mhi, K.bhi), K.nhi[1]);
                const uint32_t h2 = hadd2_bits(and_or(xcd, K.mhi, K.bhi), K.nhi[2]);
                const uint32_t h3 = hadd2_bits(and_or(ycd, K.mhi, K.bhi), K.nhi[3]);
#pragma unroll
                for (int nt = 0; nt < kMtNT; ++nt) {
                    const uint32_t b0 = hmul2_bits(pp[nt][0], dva), b1 = hmul2_bits(pp[nt][1], dvb);
                    mma16816(o[2 * bb][nt], l0, l1, l2, l3, b0, b1);
                    mma16816(o[2 * bb + 1][nt], h0, h1, h2, h3, b0, b1);
                }
            }
        }
        __syncwarp();
    }
    launch_dependents();
    if (aborted && half == 0 && lane == 0) {
        // let the pair's copies still in flight land (bounded)
        for (uint32_t k = issued > NSW ? issued - NSW : 0; k < issued; ++k) {
            const uint64_t tw = global_ns();
            while (!mbar_try_wait(&full[k % NSW], (k / NSW) & 1) && global_ns() - tw < kWaitNs) {
            }
        }
    }
    // the sums of each column over the warp's 32 lanes (tokens gid, gid + 8)
#pragma unroll
    for (int nt = 0; nt < kMtNT; ++nt)
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            lsum[nt][0] += __shfl_xor_sync(0xffffffffu, lsum[nt][0], off);
            lsum[nt][1] += __shfl_xor_sync(0xffffffffu, lsum[nt][1], off);
        }
    // my half of every column's row: O / l as the f16 partial (or the f32
    // output of a direct plan); a row with no key in this partition is left
    // to the merge (it counts only partitions below the row's length) or, for
    // a direct plan, written as zeros
    __half *po = static_cast<__half *>(p.part_o);
    float2 *pml = reinterpret_cast<float2 *>(p.part_ml);
#pragma unroll
    for (int nt = 0; nt < kMtNT; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const uint32_t c = nt * 8 + 2 * tig + e;
            if (c >= NC)
                continue;
            const uint32_t i = c / G, j = c % G;
            const uint64_t row = ((uint64_t)seq * T + i) * p.hq + g * G + j;
            const bool has = t0 < lim[nt][e];
            const float l = lsum[nt][e];
            const float inv = has && l > 0.0f ? 1.0f / l : 0.0f;
            if (p.direct) {
                float *dst = p.out + row * 256 + 128 * half;
#pragma unroll
                for (int mt = 0; mt < 2 * kMtHalfBlocks; ++mt)
                    *reinterpret_cast<float2 *>(dst + Q40::dim_of(mt, gid, 0)) =
                        make_float2(o[mt][nt][e] * inv, o[mt][nt][e + 2] * inv);
            } else if (has) {
                __half *dst = po + (row * p.n_parts + part) * 256 + 128 * half;
#pragma unroll
                for (int mt = 0; mt < 2 * kMtHalfBlocks; ++mt)
                    *reinterpret_cast<__half2 *>(dst + Q40::dim_of(mt, gid, 0)) =
                        __floats2half2_rn(o[mt][nt][e] * inv, o[mt][nt][e + 2] * inv);
                if (half == 0 && gid == 0)
                    pml[row * p.n_parts + part] =
                        make_float2(l > 0.0f ? mref[nt][e] : -INFINITY, l);
            }
        }
}

// Whether the multi-token kernel serves these shapes: Q4_0 K and V, D = 256,
// at most 4 K/V heads, 2 <= T and T * G <= 24.
__host__ inline bool mt_supported(pa_type kt, pa_type vt, uint32_t d, uint32_t hq, uint32_t hkv,
                                  uint32_t T)
{
    return kt == PA_Q4_0 && vt == PA_Q4_0 && d == 256 && (hkv == 1 || hkv == 2 || hkv == 4) &&
           hq % hkv == 0 && T >= 2 && T * (hq / hkv) <= kMtMaxCols && mt_slots(hkv) >= 2;
}

int launch_mt(const DecodeParams &p, cudaStream_t st, const char *entry)
{
    if (!mt_supported(PA_Q4_0, PA_Q4_0, p.d, p.hq, p.hkv, p.q_tokens))
        return fail(PA_ERR_INVALID, entry, "multi-token plan: shapes unsupported");
    const uint32_t nsw = mt_slots(p.hkv);
    const MtLayout lay = mt_layout(p.hkv, nsw);
    FastArgs a;
    memset(&a, 0, sizeof a);
    int rc = cached_maps<Q40>(p, a, entry);
    if (rc)
        return rc;
    a.p = p;
    a.n_slots = nsw;
    a.slot_bytes = Q40::kSlot;
    a.region_bytes = lay.total;
    static std::once_flag once;
    static cudaError_t attr = cudaSuccess;
    std::call_once(once, [] {
        attr = cudaFuncSetAttribute(mt_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)(kSmemBudget + 4096));
    });
    rc = cuda_check(attr, entry, "cudaFuncSetAttribute");
    if (rc)
        return rc;
    static const bool pdl_on = env_on("PA_PDL");
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.n_ctas);
    cfg.blockDim = dim3(64 * p.hkv);
    cfg.dynamicSmemBytes = 1024 + lay.total;
    cfg.stream = st;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = pdl_on ? 1 : 0;
    cudaError_t e = cudaLaunchKernelEx(&cfg, mt_decode_kernel, a);
    if (e != cudaSuccess)
        return cuda_check(e, entry, "mt_decode_kernel launch");
    return cuda_check(cudaGetLastError(), entry, "mt_decode_kernel launch");
}

}  // namespace
}  // namespace pa

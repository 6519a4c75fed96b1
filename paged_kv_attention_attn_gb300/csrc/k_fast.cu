// k_fast.cu -- the fast sm_103a paged decode kernel.
//
// One CTA per live (sequence, partition) covers every K/V head.  A producer
// warp walks the partition's block-table entries and stages each 16-token
// tile of K and V into a ring of shared-memory stages with TMA tensor copies
// (cp.async.bulk.tensor, one tensor map per side and K/V head, so that the
// rows of one head land contiguously in shared memory), completing on
// mbarriers.  Eight consumer warps share the K/V heads (8 / Hkv warps per
// head, taking alternate tiles): each computes the scores of all query heads
// of its group with tensor-core MMAs (m16n8k16, f16 operands, f32
// accumulators; query heads on M, padded to 16), an online softmax in the
// log2 domain that rescales only when a running maximum changes, and PV with
// the head dimension on M.  At the end the warps of one head combine their
// (m, l, O) and write the normalised f16 partial with (m, l), or the output
// itself for a direct plan.
//
// Q4_0 K/V stay 4-bit in HBM and in shared memory; nibbles become f16 in
// registers with one LOP3 per two values (the nibble is OR-ed into the
// mantissa of 1024 or 64, so the f16 value is bias + nibble exactly).  The
// QK dot of each 32-value block is an exact integer: the q8_1 query is the A
// operand as exact f16 integers, the biases are removed by starting the
// accumulator at minus their (exact) contribution, and the block's scales
// d_k * d_q multiply the result.  For PV the V nibble minus 8 is an exact f16
// operand and the block scale d_v is folded into the probabilities.
//
// Sources: "feat: add paged-attention monolithic decode-only AR foundation"
// (lucebox pull 555), Summary -- one pass over each K/V row serves all query
// heads of its group, 32-token-class tiles, skip-if-unchanged rescale,
// exp2 softmax, f16 normalised partials, occupancy-aware partitions;
// "fix(paged-attention): use 64-bit pool offsets in the fused decode
// kernels" (mlxcel issue 2153) -- pool rows are addressed by TMA from 32-bit
// slot coordinates and 64-bit strides, never by a 32-bit product.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cudaTypedefs.h>
#include <math.h>

#include <cstring>
#include <mutex>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

constexpr int kTile = 16;  // tokens per stage
constexpr int kMaxHkv = 8;
constexpr size_t kSmemBudget = 220 * 1024;
constexpr uint64_t kWaitNs = 2000000000ull;  // bound of every mbarrier wait (2 s)

struct FastArgs {
    CUtensorMap tm[2][kMaxHkv];  // [K, V][head]
    DecodeParams p;
    uint32_t n_slots;            // ring slots per warp
    uint32_t slot_bytes;         // K then V rows of one head for one tile
    uint32_t region_bytes;       // all rings; reused at the end to park (m, l, O)
};

// ------------------------------------------------------------------- PTX

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ uint64_t global_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred P;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 P, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, P;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int x, int y,
                                            uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void fence_proxy_async()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t (&r)[4], uint32_t addr)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

__device__ __forceinline__ uint32_t h2_bits(__half2 h) { return *reinterpret_cast<uint32_t *>(&h); }
__device__ __forceinline__ __half2 bits_h2(uint32_t u) { return *reinterpret_cast<__half2 *>(&u); }

__device__ __forceinline__ uint32_t hsub2_bits(uint32_t x, uint32_t y)
{
    return h2_bits(__hsub2(bits_h2(x), bits_h2(y)));
}

__device__ __forceinline__ uint32_t hmul2_bits(uint32_t x, uint32_t y)
{
    return h2_bits(__hmul2(bits_h2(x), bits_h2(y)));
}

// ------------------------------------------------------------ per-type code
//
// Each type provides the shared-memory layout of one stage and, for one
// consumer warp, the query fragments, the scores of one tile and the PV update
// of one tile.  Thread roles follow the m16n8k16 fragment layout: gid = lane/4,
// tig = lane%4.  QK: A = query heads (row gid; rows >= G and gid+8 are zero),
// B = keys (column gid = token).  PV: A = values (rows = dimensions), B =
// probabilities (column gid = query head), C = O[dimension][head].

// --- Q4_0, D = 256 --------------------------------------------------------
struct Q40 {
    static constexpr int D = 256;
    static constexpr int NB = D / 32;       // 32-value blocks per row
    static constexpr int RB = NB * 18;      // row bytes
    static constexpr int MT = D / 16;       // PV m-tiles
    static constexpr int SCRATCH = NB * kTile * 4 + NB * kTile * 2;  // dk f32, dv f16
    static constexpr bool kZeroInvalidV = false;
    static constexpr uint32_t kTmaX = 1;    // TMA boxes per (side, head)

    static __host__ __device__ constexpr uint32_t side_bytes(uint32_t hkv)
    {
        return hkv * kTile * RB;
    }

    struct Frag {
        uint32_t qa[NB][4];  // per block: low-dims a0, a2; high-dims a0, a2
        float ncorr[NB];     // minus the bias contribution of the block (exact)
        float dqs[NB];       // d_q * scale * log2(e)
    };

    // Query head row gid of group g: q8_1 bytes -> exact f16 integers in the
    // dimension order the nibble expansion produces (see qk_block).
    __device__ static void load_q(const DecodeParams &p, uint32_t s, uint32_t h0, uint32_t G,
                                  int gid, int tig, Frag &f)
    {
        const bool live = (uint32_t)gid < G;
        const uint8_t *row = static_cast<const uint8_t *>(p.q) +
                             ((uint64_t)s * p.hq + h0 + (live ? gid : 0)) * NB * 36;
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            const uint8_t *blk = row + 36 * b;
            int q[8];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                q[j] = live ? (int)(int8_t)blk[4 + 4 * tig + j] : 0;       // dims 4tig+j
                q[4 + j] = live ? (int)(int8_t)blk[20 + 4 * tig + j] : 0;  // dims 16+4tig+j
            }
            f.qa[b][0] = h2_bits(__halves2half2(__int2half_rn(q[0]), __int2half_rn(q[2])));
            f.qa[b][1] = h2_bits(__halves2half2(__int2half_rn(q[1]), __int2half_rn(q[3])));
            f.qa[b][2] = h2_bits(__halves2half2(__int2half_rn(q[4]), __int2half_rn(q[6])));
            f.qa[b][3] = h2_bits(__halves2half2(__int2half_rn(q[5]), __int2half_rn(q[7])));
            int lo = q[0] + q[1] + q[2] + q[3], hi = q[4] + q[5] + q[6] + q[7];
            lo += __shfl_xor_sync(0xffffffffu, lo, 1);
            lo += __shfl_xor_sync(0xffffffffu, lo, 2);
            hi += __shfl_xor_sync(0xffffffffu, hi, 1);
            hi += __shfl_xor_sync(0xffffffffu, hi, 2);
            // low nibbles read as 1024 + n, high nibbles as 64 + n; the value is n - 8
            f.ncorr[b] = -(float)(1032 * lo + 72 * hi);
            f.dqs[b] = live ? half_bits_to_float(load_u16(blk)) * p.scale_log2 : 0.0f;
        }
    }

    // Copies the tile's block scales of head g into the warp's scratch:
    // dk float [NB][16] and dv half [NB][16], zero for invalid tokens.
    __device__ static void extract(const uint8_t *kh, const uint8_t *vh, uint8_t *scr,
                                   int nvalid, int lane)
    {
        float *dk = reinterpret_cast<float *>(scr);
        uint16_t *dv = reinterpret_cast<uint16_t *>(scr + NB * kTile * 4);
#pragma unroll
        for (int k = 0; k < NB * kTile / 32; ++k) {
            const int e = lane + 32 * k, t = e & 15, b = e >> 4;
            const bool v = t < nvalid;
            const uint16_t kd = load_u16(kh + t * RB + 18 * b);
            const uint16_t vd = load_u16(vh + t * RB + 18 * b);
            dk[e] = v ? half_bits_to_float(kd) : 0.0f;
            dv[e] = v ? vd : (uint16_t)0;
        }
    }

    // QK of one 32-value block for the 8 tokens of this n-tile; w holds the
    // 8 nibbles of dims 4tig..4tig+3 (low) and 16+4tig..19+4tig (high).
    __device__ static __forceinline__ void qk_block(const Frag &f, int b, uint32_t w, float dk0,
                                                    float dk1, float &s0, float &s1)
    {
        const uint32_t x = w >> 8;
        const uint32_t blo0 = (w & 0x000F000Fu) | 0x64006400u;  // dims 4tig, 4tig+2
        const uint32_t blo1 = (x & 0x000F000Fu) | 0x64006400u;  // dims 4tig+1, 4tig+3
        const uint32_t bhi0 = (w & 0x00F000F0u) | 0x54005400u;
        const uint32_t bhi1 = (x & 0x00F000F0u) | 0x54005400u;
        float c[4] = {f.ncorr[b], f.ncorr[b], 0.0f, 0.0f};
        mma16816(c, f.qa[b][0], 0u, f.qa[b][1], 0u, blo0, blo1);
        mma16816(c, f.qa[b][2], 0u, f.qa[b][3], 0u, bhi0, bhi1);
        s0 = fmaf(c[0] * dk0, f.dqs[b], s0);
        s1 = fmaf(c[1] * dk1, f.dqs[b], s1);
    }

    // Scores (log2 units, unmasked) of tokens nt*8 + 2tig + {0, 1}.
    __device__ static void scores(const Frag &f, const uint8_t *kh, const uint8_t *scr, int gid,
                                  int tig, float (&sc)[2][2])
    {
        const float *dk = reinterpret_cast<const float *>(scr);
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            const uint32_t *wr = reinterpret_cast<const uint32_t *>(kh + (nt * 8 + gid) * RB);
            float s0 = 0.0f, s1 = 0.0f;
#pragma unroll
            for (int pb = 0; pb < NB / 2; ++pb) {
                // blocks 2pb and 2pb+1 share 36 bytes = 9 aligned words
                const uint32_t w0 = wr[9 * pb + tig], w1 = wr[9 * pb + tig + 1];
                const uint32_t w2 = wr[9 * pb + 5 + tig];
                const uint32_t wa = __funnelshift_r(w0, w1, 16);
                const float2 k0 = *reinterpret_cast<const float2 *>(dk + (2 * pb) * kTile + nt * 8 + 2 * tig);
                const float2 k1 = *reinterpret_cast<const float2 *>(dk + (2 * pb + 1) * kTile + nt * 8 + 2 * tig);
                qk_block(f, 2 * pb, wa, k0.x, k0.y, s0, s1);
                qk_block(f, 2 * pb + 1, w2, k1.x, k1.y, s0, s1);
            }
            sc[nt][0] = s0;
            sc[nt][1] = s1;
        }
    }

    // O += V^T P' over the tile; P' = P * d_v per block.
    __device__ static void pv(float (&o)[MT][4], const uint8_t *vh, const uint8_t *scr, uint32_t p0,
                              uint32_t p1, int gid, int tig)
    {
        const uint16_t *dv = reinterpret_cast<const uint16_t *>(scr + NB * kTile * 4);
        const uint8_t *ra = vh + (2 * tig) * RB + 2 + 2 * gid;
        const uint8_t *rc = vh + (2 * tig + 8) * RB + 2 + 2 * gid;
        const uint32_t kLo = 0x64086408u;  // 1032
        const uint32_t kHi = 0x54805480u;  // 72
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            const uint32_t ua = load_u16(ra + 18 * b), ub = load_u16(ra + RB + 18 * b);
            const uint32_t uc = load_u16(rc + 18 * b), ud = load_u16(rc + RB + 18 * b);
            const uint32_t xab = __byte_perm(ua, ub, 0x5410), yab = xab >> 8;
            const uint32_t xcd = __byte_perm(uc, ud, 0x5410), ycd = xcd >> 8;
            const uint32_t b0 = hmul2_bits(p0, *reinterpret_cast<const uint32_t *>(dv + b * kTile + 2 * tig));
            const uint32_t b1 = hmul2_bits(p1, *reinterpret_cast<const uint32_t *>(dv + b * kTile + 8 + 2 * tig));
            mma16816(o[2 * b], hsub2_bits((xab & 0x000F000Fu) | 0x64006400u, kLo),
                     hsub2_bits((yab & 0x000F000Fu) | 0x64006400u, kLo),
                     hsub2_bits((xcd & 0x000F000Fu) | 0x64006400u, kLo),
                     hsub2_bits((ycd & 0x000F000Fu) | 0x64006400u, kLo), b0, b1);
            mma16816(o[2 * b + 1], hsub2_bits((xab & 0x00F000F0u) | 0x54005400u, kHi),
                     hsub2_bits((yab & 0x00F000F0u) | 0x54005400u, kHi),
                     hsub2_bits((xcd & 0x00F000F0u) | 0x54005400u, kHi),
                     hsub2_bits((ycd & 0x00F000F0u) | 0x54005400u, kHi), b0, b1);
        }
    }

    // Output dimension of PV C-fragment row (gid or gid+8) of m-tile mt.
    __device__ static __forceinline__ int dim_of(int mt, int gid, int upper)
    {
        return 32 * (mt >> 1) + 16 * (mt & 1) + 2 * gid + upper;
    }
};

// --- F16, D = 128 or 256 ----------------------------------------------------
// Stage layout per side: [head][64-dim chunk][16 tokens][128 B], written by
// TMA with the 128-byte swizzle (16-byte chunk c of row t stored at c ^ (t&7)),
// read with ldmatrix without bank conflicts.
template <int D_>
struct F16T {
    static constexpr int D = D_;
    static constexpr int NC = D / 64;   // 64-dim chunks
    static constexpr int KS = D / 16;   // k-steps
    static constexpr int MT = D / 16;
    static constexpr int SCRATCH = 0;
    static constexpr bool kZeroInvalidV = true;
    static constexpr uint32_t kTmaX = NC;

    static __host__ __device__ constexpr uint32_t side_bytes(uint32_t hkv)
    {
        return hkv * kTile * D * 2;
    }

    struct Frag {
        uint32_t qa[KS][2];  // a0, a2 of each k-step
        float scale;
    };

    __device__ static void load_q(const DecodeParams &p, uint32_t s, uint32_t h0, uint32_t G,
                                  int gid, int tig, Frag &f)
    {
        const bool live = (uint32_t)gid < G;
        const float *row = static_cast<const float *>(p.q) +
                           ((uint64_t)s * p.hq + h0 + (live ? gid : 0)) * D;
#pragma unroll
        for (int j = 0; j < KS; ++j) {
            const float2 x = live ? *reinterpret_cast<const float2 *>(row + 16 * j + 2 * tig)
                                  : make_float2(0.f, 0.f);
            const float2 y = live ? *reinterpret_cast<const float2 *>(row + 16 * j + 8 + 2 * tig)
                                  : make_float2(0.f, 0.f);
            f.qa[j][0] = h2_bits(__floats2half2_rn(x.x, x.y));
            f.qa[j][1] = h2_bits(__floats2half2_rn(y.x, y.y));
        }
        f.scale = p.scale_log2;
    }

    __device__ static __forceinline__ uint32_t chunk_addr(const uint8_t *sub, int token, int c16)
    {
        return smem_u32(sub + token * 128 + ((c16 ^ (token & 7)) << 4));
    }

    // Zero V rows of tokens >= nvalid (their bytes may be anything).
    __device__ static void zero_invalid_v(uint8_t *vh, int nvalid, int lane)
    {
        const int rows = (kTile - nvalid) * NC;
        for (int i = lane; i < rows * 8; i += 32) {
            const int r = i >> 3, part = i & 7;
            const int c = r / (kTile - nvalid), t = nvalid + r % (kTile - nvalid);
            reinterpret_cast<uint4 *>(vh + (c * kTile + t) * 128)[part] = make_uint4(0, 0, 0, 0);
        }
    }

    __device__ static void scores(const Frag &f, const uint8_t *kh, const uint8_t *, int gid,
                                  int tig, float (&sc)[2][2])
    {
        const int lane = gid * 4 + tig;
        const int mi = lane >> 3, r = lane & 7;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            float c[4] = {0.f, 0.f, 0.f, 0.f};
            const int token = nt * 8 + r;
#pragma unroll
            for (int j2 = 0; j2 < KS / 2; ++j2) {
                uint32_t bq[4];
                const uint8_t *sub = kh + (j2 >> 1) * kTile * 128;
                ldsm_x4(bq, chunk_addr(sub, token, (j2 & 1) * 4 + mi));
                mma16816(c, f.qa[2 * j2][0], 0u, f.qa[2 * j2][1], 0u, bq[0], bq[1]);
                mma16816(c, f.qa[2 * j2 + 1][0], 0u, f.qa[2 * j2 + 1][1], 0u, bq[2], bq[3]);
            }
            sc[nt][0] = c[0] * f.scale;
            sc[nt][1] = c[1] * f.scale;
        }
    }

    __device__ static void pv(float (&o)[MT][4], const uint8_t *vh, const uint8_t *, uint32_t p0,
                              uint32_t p1, int gid, int tig)
    {
        const int lane = gid * 4 + tig;
        const int mi = lane >> 3, r = lane & 7;
        const int token = (mi >> 1) * 8 + r;
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
            uint32_t a[4];
            const uint8_t *sub = vh + (mt >> 2) * kTile * 128;
            ldsm_x4_trans(a, chunk_addr(sub, token, (mt & 3) * 2 + (mi & 1)));
            mma16816(o[mt], a[0], a[1], a[2], a[3], p0, p1);
        }
    }

    __device__ static __forceinline__ int dim_of(int mt, int gid, int upper)
    {
        return 16 * mt + gid + 8 * upper;
    }
};

// ------------------------------------------------------------------ kernel
//
// Warp w serves K/V head g = w % hkv and the tiles i = sub, sub + wph, ... of
// the partition (sub = w / hkv, wph = warps / hkv).  It owns a private ring of
// n_slots stages, each holding the K and V rows of its head for one tile, and
// it alone issues their TMA copies and waits on their mbarriers, so the main
// loop needs no synchronisation between warps.  Rows of a tile for the other
// heads are fetched by the other warps at about the same time; the whole
// 16-token block is one contiguous range of the pool.

template <class T>
__global__ void __launch_bounds__(256, 1) fast_decode_kernel(const __grid_constant__ FastArgs a)
{
    const DecodeParams &p = a.p;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~uintptr_t(1023));
    const uint32_t NSW = a.n_slots, SLOT = a.slot_bytes, nwarps = blockDim.x >> 5;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t hkv = p.hkv, G = p.hq / p.hkv, wph = nwarps / hkv;
    uint8_t *ring = smem + (size_t)warp * NSW * SLOT;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + a.region_bytes) + warp * NSW;
    int *slot_ok = reinterpret_cast<int *>(reinterpret_cast<uint64_t *>(smem + a.region_bytes) +
                                           nwarps * NSW) + warp * NSW;
    uint8_t *scr = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(slot_ok + (nwarps - warp) * NSW) + 15) & ~uintptr_t(15)) +
        warp * T::SCRATCH;

    if (lane == 0) {
        for (uint32_t s = 0; s < NSW; ++s)
            mbar_init(&full[s], 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    uint32_t seq, part;
    if (p.direct) {
        seq = blockIdx.x;
        part = 0;
    } else if (!cta_work(p.seq_lens, p.n_seqs, p.part_tokens, blockIdx.x, &seq, &part)) {
        return;  // past the last live partition: nothing was issued
    }
    const int32_t L = p.seq_lens[seq] > 0 ? p.seq_lens[seq] : 0;
    const uint32_t t0 = p.direct ? 0u : part * p.part_tokens;
    const uint32_t t1 = p.direct ? (uint32_t)L : min((uint32_t)L, t0 + p.part_tokens);
    const uint32_t n_tiles = (t1 - t0 + kTile - 1) / kTile;
    const int gid = lane >> 2, tig = lane & 3;
    const uint32_t g = warp % hkv, sub = warp / hkv;
    const uint32_t n_my = n_tiles > sub ? (n_tiles - sub + wph - 1) / wph : 0;
    const int32_t *bt = p.block_table + (uint64_t)seq * p.table_stride;
    const CUtensorMap *tmk = &a.tm[0][g], *tmv = &a.tm[1][g];
    const uint32_t side = SLOT / 2;

    // block ids of my tiles k0 .. k0+31, one per lane
    auto fetch_ids = [&](uint32_t k0) -> int32_t {
        const uint32_t k = k0 + lane;
        return k < n_my ? bt[(t0 + kTile * (sub + k * wph)) / p.block_size] : 0;
    };
    // lane 0: start the copy of my tile k (block id blk) into its slot
    auto issue = [&](uint32_t k, int32_t blk) {
        const uint32_t s = k % NSW;
        const uint32_t tok = t0 + kTile * (sub + k * wph);
        const bool ok = block_in_pool(blk, p.n_pool_blocks);
        slot_ok[s] = ok;
        if (ok) {
            uint8_t *dst = ring + (size_t)s * SLOT;
            const int y = blk * (int)p.block_size + (int)(tok % p.block_size);
            fence_proxy_async();  // earlier generic reads of this slot come first
            mbar_arrive_expect_tx(&full[s], SLOT);
#pragma unroll
            for (uint32_t c = 0; c < T::kTmaX; ++c) {
                tma_load_2d(dst + c * (side / T::kTmaX), tmk, 64 * c, y, &full[s]);
                tma_load_2d(dst + side + c * (side / T::kTmaX), tmv, 64 * c, y, &full[s]);
            }
        } else {
            atomicOr(p.status, PA_STATUS_CORRUPT_TABLE);
            mbar_arrive(&full[s]);
        }
    };

    int32_t ids = fetch_ids(0), ids_next = fetch_ids(32);
    const uint32_t pro = n_my < NSW ? n_my : NSW;
    for (uint32_t k = 0; k < pro; ++k) {
        const int32_t b = __shfl_sync(0xffffffffu, ids, k);
        if (lane == 0)
            issue(k, b);
    }
    __syncwarp();

    typename T::Frag f;
    T::load_q(p, seq, g * G, G, gid, tig, f);
    float o[T::MT][4];
#pragma unroll
    for (int mt = 0; mt < T::MT; ++mt)
        o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.0f;
    float m_run = -INFINITY, l_run = 0.0f;
    bool aborted = false;
    uint32_t issued = pro;

    for (uint32_t k = 0; k < n_my; ++k) {
        const uint32_t s = k % NSW;
        // every lane waits (bounded) and so acquires the slot's TMA writes itself
        bool done = mbar_try_wait(&full[s], (k / NSW) & 1);
        if (!done) {
            const uint64_t tw = global_ns();
            while (!(done = mbar_try_wait(&full[s], (k / NSW) & 1)) && global_ns() - tw < kWaitNs) {
            }
        }
        if (!__all_sync(0xffffffffu, done)) {
            if (lane == 0)
                atomicOr(p.status, PA_STATUS_TIMEOUT);
            aborted = true;
            break;
        }
        const uint32_t i = sub + k * wph;
        const int nvalid = slot_ok[s] ? (int)min(16u, t1 - (t0 + kTile * i)) : 0;
        uint8_t *kh = ring + (size_t)s * SLOT;
        uint8_t *vh = kh + side;
        if constexpr (T::kZeroInvalidV) {
            if (nvalid < kTile) {
                T::zero_invalid_v(vh, nvalid, lane);
                __syncwarp();
            }
        } else {
            T::extract(kh, vh, scr, nvalid, lane);
            __syncwarp();
        }
        float sc[2][2];
        T::scores(f, kh, scr, gid, tig, sc);
        // online softmax over the tile, log2 domain; rescale only on a new max
        float tmax = -INFINITY;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                if (nt * 8 + 2 * tig + j >= nvalid)
                    sc[nt][j] = -INFINITY;
                tmax = fmaxf(tmax, sc[nt][j]);
            }
        tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 1));
        tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 2));
        if (__any_sync(0xffffffffu, tmax > m_run)) {
            const float m_new = fmaxf(m_run, tmax);
            const float alpha = m_run == -INFINITY ? 0.0f : exp2f(m_run - m_new);
            const float a0 = __shfl_sync(0xffffffffu, alpha, 8 * tig);
            const float a1 = __shfl_sync(0xffffffffu, alpha, 8 * tig + 4);
#pragma unroll
            for (int mt = 0; mt < T::MT; ++mt) {
                o[mt][0] *= a0;
                o[mt][1] *= a1;
                o[mt][2] *= a0;
                o[mt][3] *= a1;
            }
            l_run *= alpha;
            m_run = m_new;
        }
        const float ms = m_run == -INFINITY ? 0.0f : m_run;
        float pr[2][2];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                pr[nt][j] = exp2f(sc[nt][j] - ms);
                l_run += pr[nt][j];
            }
        const uint32_t p0 = h2_bits(__floats2half2_rn(pr[0][0], pr[0][1]));
        const uint32_t p1 = h2_bits(__floats2half2_rn(pr[1][0], pr[1][1]));
        T::pv(o, vh, scr, p0, p1, gid, tig);
        __syncwarp();  // all reads of this slot are done
        // refill the slot with my tile k + NSW
        const uint32_t kn = k + NSW;
        if (kn < n_my) {
            if ((kn & 31) == 0) {
                ids = ids_next;
                ids_next = fetch_ids(kn + 32);
            }
            const int32_t b = __shfl_sync(0xffffffffu, ids, kn & 31);
            if (lane == 0)
                issue(kn, b);
            issued = kn + 1;
        }
        __syncwarp();
    }
    if (aborted && lane == 0) {
        // let my copies still in flight land (bounded) before the CTA moves on
        for (uint32_t k = issued > NSW ? issued - NSW : 0; k < issued; ++k) {
            const uint64_t tw = global_ns();
            while (!mbar_try_wait(&full[k % NSW], (k / NSW) & 1) && global_ns() - tw < kWaitNs) {
            }
        }
    }
    l_run += __shfl_xor_sync(0xffffffffu, l_run, 1);
    l_run += __shfl_xor_sync(0xffffffffu, l_run, 2);

    // park (m, l, O) of every warp in the now idle rings, then the first warp
    // of each head combines them
    __syncthreads();
    float *park = reinterpret_cast<float *>(smem);
    const int per_warp = 16 + 32 * 4 * T::MT;
    float *mine = park + warp * per_warp;
    if (tig == 0) {
        mine[gid] = m_run;
        mine[8 + gid] = l_run;
    }
#pragma unroll
    for (int mt = 0; mt < T::MT; ++mt)
#pragma unroll
        for (int e = 0; e < 4; ++e)
            mine[16 + (mt * 4 + e) * 32 + lane] = o[mt][e];
    __syncthreads();
    if (sub != 0)
        return;
    float M[2], l[2], fk[8][2];
#pragma unroll
    for (int c = 0; c < 2; ++c) {
        const int h = 2 * tig + c;
        M[c] = -INFINITY;
        for (uint32_t k = 0; k < wph; ++k)
            M[c] = fmaxf(M[c], park[(g + k * hkv) * per_warp + h]);
        l[c] = 0.0f;
        for (uint32_t k = 0; k < wph; ++k) {
            const float mk = park[(g + k * hkv) * per_warp + h];
            const float f2 = M[c] == -INFINITY ? 0.0f : exp2f(mk - M[c]);
            fk[k][c] = f2;
            l[c] += park[(g + k * hkv) * per_warp + 8 + h] * f2;
        }
    }
    float inv[2];
#pragma unroll
    for (int c = 0; c < 2; ++c)
        inv[c] = l[c] > 0.0f ? 1.0f / l[c] : 0.0f;
    const uint64_t sh0 = (uint64_t)seq * p.hq + g * G;
#pragma unroll
    for (int mt = 0; mt < T::MT; ++mt) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int c = e & 1, upper = e >> 1;
            float v = 0.0f;
            for (uint32_t k = 0; k < wph; ++k)
                v += park[(g + k * hkv) * per_warp + 16 + (mt * 4 + e) * 32 + lane] * fk[k][c];
            const uint32_t h = 2 * tig + c;
            if (h >= G)
                continue;
            const int dim = T::dim_of(mt, gid, upper);
            if (p.direct) {
                p.out[(sh0 + h) * T::D + dim] = v * inv[c];
            } else {
                __half *po = static_cast<__half *>(p.part_o);
                po[((sh0 + h) * p.n_parts + part) * T::D + dim] = __float2half_rn(v * inv[c]);
            }
        }
    }
    if (!p.direct && gid == 0) {
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            const uint32_t h = 2 * tig + c;
            if (h < G)
                reinterpret_cast<float2 *>(p.part_ml)[(sh0 + h) * p.n_parts + part] =
                    make_float2(l[c] > 0.0f ? M[c] : -INFINITY, l[c]);
        }
    }
}

// ------------------------------------------------------------------- host

PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

// Launch geometry of one kernel instance: warps per head and ring slots.
struct Geometry {
    uint32_t wph = 0, warps = 0, n_slots = 0, slot_bytes = 0, region = 0;
    size_t smem = 0;
};

template <class T>
Geometry geometry(uint32_t hkv)
{
    Geometry gm;
    const size_t slot = 2 * (size_t)T::side_bytes(1);
    const size_t park_per_warp = (16 + 32 * 4 * T::MT) * 4;
    for (uint32_t wph = 8 / hkv; wph >= 1; wph /= 2) {
        const uint32_t warps = wph * hkv;
        const size_t fixed = 1024 + warps * (size_t)T::SCRATCH + warps * 16 * 12 + 64;
        if (fixed >= kSmemBudget)
            continue;
        size_t ns = (kSmemBudget - fixed) / (warps * slot);
        if (ns > 8)
            ns = 8;
        if (ns >= 2) {
            gm.wph = wph;
            gm.warps = warps;
            gm.n_slots = (uint32_t)ns;
            gm.slot_bytes = (uint32_t)slot;
            size_t ring = warps * ns * slot, park = warps * park_per_warp;
            gm.region = (uint32_t)(ring > park ? ring : park);
            gm.smem = 1024 + gm.region + warps * ns * (8 + 4) + 16 + warps * (size_t)T::SCRATCH;
            return gm;
        }
        if (wph == 1)
            break;
    }
    return gm;
}

template <class T>
int encode_maps(const DecodeParams &p, FastArgs &a, const char *entry)
{
    auto enc = encode_fn();
    if (!enc)
        return fail(PA_ERR_CUDA, entry, "cuTensorMapEncodeTiled unavailable");
    const uint64_t rb = T::side_bytes(1) / kTile;  // bytes of one row
    const uint64_t n_slots = p.n_pool_blocks * p.block_size;
    for (int side = 0; side < 2; ++side) {
        const uint8_t *pool = side ? p.v_pool : p.k_pool;
        for (uint32_t g = 0; g < p.hkv; ++g) {
            cuuint64_t dims[2] = {rb / 2, n_slots}, strides[1] = {(cuuint64_t)p.hkv * rb};
            cuuint32_t box[2] = {T::kTmaX > 1 ? 64u : (cuuint32_t)(rb / 2), (cuuint32_t)kTile};
            cuuint32_t estr[2] = {1, 1};
            // f16 rows: 64-value chunks with the 128-byte swizzle; Q4_0 rows whole
            const CUtensorMapSwizzle sw =
                T::kTmaX > 1 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE;
            CUresult r = enc(&a.tm[side][g], CU_TENSOR_MAP_DATA_TYPE_UINT16, 2,
                             const_cast<uint8_t *>(pool) + g * rb, dims, strides, box, estr,
                             CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
            if (r != CUDA_SUCCESS)
                return fail(PA_ERR_CUDA, entry, "cuTensorMapEncodeTiled failed (%d)", (int)r);
        }
    }
    return PA_OK;
}

// Raises the kernel's dynamic shared-memory limit once per device.
template <class T>
cudaError_t allow_smem()
{
    static std::mutex mu;
    static bool done[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= 64)
        return e != cudaSuccess ? e : cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (!done[dev]) {
        e = cudaFuncSetAttribute(fast_decode_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)(kSmemBudget + 4096));
        if (e != cudaSuccess)
            return e;
        done[dev] = true;
    }
    return cudaSuccess;
}

template <class T>
int launch_t(const DecodeParams &p, cudaStream_t st, const char *entry)
{
    const Geometry gm = geometry<T>(p.hkv);
    if (!gm.warps)
        return fail(PA_ERR_INVALID, entry, "fast kernel: a tile does not fit shared memory");
    FastArgs a;
    memset(&a, 0, sizeof a);
    int rc = encode_maps<T>(p, a, entry);
    if (rc)
        return rc;
    a.p = p;
    a.n_slots = gm.n_slots;
    a.slot_bytes = gm.slot_bytes;
    a.region_bytes = gm.region;
    rc = cuda_check(allow_smem<T>(), entry, "cudaFuncSetAttribute");
    if (rc)
        return rc;
    fast_decode_kernel<T><<<p.n_ctas, gm.warps * 32, gm.smem, st>>>(a);
    return cuda_check(cudaGetLastError(), entry, "fast_decode_kernel launch");
}

template <class T>
int occupancy_t(uint32_t hkv, int *cps)
{
    const Geometry gm = geometry<T>(hkv);
    if (!gm.warps)
        return PA_ERR_INVALID;
    cudaError_t e = allow_smem<T>();
    if (e == cudaSuccess)
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(cps, fast_decode_kernel<T>,
                                                          gm.warps * 32, gm.smem);
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

bool hkv_ok(uint32_t hkv) { return hkv == 1 || hkv == 2 || hkv == 4 || hkv == 8; }

}  // namespace

bool fast_decode_supported(pa_type kt, pa_type vt, uint32_t d, uint32_t hq, uint32_t hkv,
                           uint32_t block_size)
{
    if (kt != vt || !hkv_ok(hkv) || hq % hkv || hq / hkv > 8 ||
        (block_size != 16 && block_size != 32))
        return false;
    if (kt == PA_Q4_0)
        return d == 256 && geometry<Q40>(hkv).warps > 0;
    if (kt == PA_F16)
        return d == 256 ? geometry<F16T<256>>(hkv).warps > 0
                        : d == 128 && geometry<F16T<128>>(hkv).warps > 0;
    return false;
}

int fast_decode_occupancy(pa_type kt, pa_type, uint32_t d, uint32_t, uint32_t hkv, uint32_t,
                          int *ctas_per_sm)
{
    if (kt == PA_Q4_0)
        return occupancy_t<Q40>(hkv, ctas_per_sm);
    return d == 256 ? occupancy_t<F16T<256>>(hkv, ctas_per_sm)
                    : occupancy_t<F16T<128>>(hkv, ctas_per_sm);
}

int launch_fast_decode(const DecodeParams &p, pa_type kt, pa_type vt, cudaStream_t st,
                       const char *entry)
{
    // TMA slot coordinates are int32: larger pools take the plain kernel
    if (p.n_pool_blocks * p.block_size >= (1ull << 31))
        return launch_plain_decode(p, kt, vt, st, entry);
    if (kt == PA_Q4_0)
        return launch_t<Q40>(p, st, entry);
    if (p.d == 256)
        return launch_t<F16T<256>>(p, st, entry);
    return launch_t<F16T<128>>(p, st, entry);
}

}  // namespace pa

// fast_kernel.cuh -- the fast sm_103a paged decode kernel, shared by the
// translation units that instantiate it (same K/V type; mixed K x V types).
//
// One CTA per live (sequence, partition) covers every K/V head, so one walk of
// the block table serves all of them and every K/V row is read from HBM once
// for all query heads of its group.  Warp w serves K/V head g = w % Hkv and the
// tiles sub, sub + wph, ... of the partition (16 tokens each; sub = w / Hkv,
// wph warps per head).  It owns a private ring of shared-memory slots that it
// fills itself with TMA tensor copies (cp.async.bulk.tensor, one tensor map per
// side and K/V head, completing on the slot's mbarrier), so the main loop has no
// producer warp and no synchronisation between warps.  Per tile the warp
// computes the scores of its group's query heads on the tensor cores
// (mma.sync with the tokens on M), an online softmax in the log2 domain with a
// reference maximum that moves only when a score passes it, and PV with the
// head dimension on M.  At the end the warps park (m, l, O) in the idle rings,
// the CTA combines them and writes the f16 partial (or the output of a direct
// plan), and the in-launch merge runs in the CTA that completes a count.
//
// Quantised rows stay quantised in HBM and in shared memory and are expanded
// in registers: Q4_0 nibbles with one LOP3 per two values (OR-ed into the
// mantissa of 1024 or 64: bias + nibble exactly), Q8_0 codes straight into
// the integer tensor path for scores and into biased f16 for PV.  The biases
// are removed by the accumulator's start value (scores), by an exact f16
// subtraction from the operands (Q4_0 PV) or by a constant-A MMA (Q8_0 PV),
// and block scales multiply the block dots (K) or the probabilities (V).
//
// Sources: "feat: add paged-attention monolithic decode-only AR foundation"
// (lucebox pull 555), Summary -- one pass over each K/V row serves all query
// heads of its group, skip-if-unchanged rescale, exp2 softmax, f16 normalised
// partials, q8_1 query, occupancy-aware partitions; "fix(paged-attention): use
// 64-bit pool offsets in the fused decode kernels" (mlxcel issue 2153) -- pool
// rows are addressed by TMA from 32-bit slot coordinates and 64-bit strides,
// never by a 32-bit product.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cudaTypedefs.h>
#include <math.h>

#include <cstdlib>
#include <cstring>
#include <mutex>
#include <unordered_map>

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
    uint32_t coop;               // in-launch merge shared by the CTAs of a sequence
    uint32_t coop_wait_ns;       // bound of a CTA's wait for the others of its sequence
    uint32_t n_slots32;          // 32-token slots per K/V head (types with kTile32)
    uint32_t bar_slots;          // mbarriers and flag words per warp (>= n_slots)
};

// Bound of the wait of the cooperative merge: far above the spread of the
// finishing times of one sequence's CTAs in a grid that is resident at once.
constexpr uint32_t kCoopWaitNs = 100000;

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

// A 2-D tensor copy of box (x, y) into shared memory, completing on the
// mbarrier, with an L2 eviction-priority hint (a createpolicy value).
__device__ __forceinline__ void tma_load_2d_hint(void *dst, const CUtensorMap *map, int x, int y,
                                                 uint64_t *bar, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// L2 policy for data read once: evicted before anything else, so that a
// stream of K/V rows does not push the kernel's code, the block table, the
// lengths and the partials out of the L2.
__device__ __forceinline__ uint64_t l2_evict_first_policy()
{
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// One contiguous global range into shared memory (both 16-byte aligned, bytes
// a multiple of 16), completing on the mbarrier.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes,
                                          uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// Generic-proxy writes to global memory (other CTAs' partials, seen through
// an acquire) before this thread's later bulk copies read them.
__device__ __forceinline__ void fence_proxy_async_global()
{
    asm volatile("fence.proxy.async.global;" ::: "memory");
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

// D = A B + C with C separate from D (C may be a constant quad).
__device__ __forceinline__ void mma16816_c(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                           uint32_t a3, uint32_t b0, uint32_t b1, const float (&c)[4])
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%10,%11,%12,%13};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]), "f"(c[2]),
          "f"(c[3]));
}

// D = A B + C, m16n8k8 in tf32 with f32 accumulation.
__device__ __forceinline__ void mma1688_tf32(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                             uint32_t a3, uint32_t b0, uint32_t b1,
                                             const float (&c)[4])
{
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%10,%11,%12,%13};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]), "f"(c[2]),
          "f"(c[3]));
}

// 2^x by the hardware's approximation (relative error about 2^-22), results
// below 2^-126 flushed to zero: the probabilities of the online softmax,
// whose arguments are at most -4 there.
__device__ __forceinline__ float ex2_ftz(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// f32 to tf32, rounded to nearest (ties away), as the f32 bit pattern.
__device__ __forceinline__ uint32_t to_tf32(float x)
{
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return r;
}

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
        : "r"(addr)
        : "memory");
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t (&r)[4], uint32_t addr)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
        : "r"(addr)
        : "memory");
}

__device__ __forceinline__ uint32_t h2_bits(__half2 h) { return *reinterpret_cast<uint32_t *>(&h); }
__device__ __forceinline__ __half2 bits_h2(uint32_t u) { return *reinterpret_cast<__half2 *>(&u); }

__device__ __forceinline__ uint32_t hadd2_bits(uint32_t x, uint32_t y)
{
    return h2_bits(__hadd2(bits_h2(x), bits_h2(y)));
}

__device__ __forceinline__ uint32_t hmul2_bits(uint32_t x, uint32_t y)
{
    return h2_bits(__hmul2(bits_h2(x), bits_h2(y)));
}

// Shared-memory accesses by 32-bit shared-window address.
__device__ __forceinline__ uint32_t lds_u32(uint32_t a)
{
    uint32_t v;
    asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(a) : "memory");
    return v;
}

__device__ __forceinline__ float lds_f32(uint32_t a)
{
    float v;
    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(a) : "memory");
    return v;
}

__device__ __forceinline__ uint32_t lds_u16(uint32_t a)
{
    uint32_t v;  // zero-extended into a 32-bit register
    asm volatile("ld.shared.u16 %0, [%1];" : "=r"(v) : "r"(a) : "memory");
    return v;
}

__device__ __forceinline__ float2 lds_f2(uint32_t a)
{
    float2 v;
    asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(a) : "memory");
    return v;
}

__device__ __forceinline__ void sts_f32(uint32_t a, float v)
{
    asm volatile("st.shared.f32 [%0], %1;" ::"r"(a), "f"(v));
}

__device__ __forceinline__ void sts_u16(uint32_t a, uint32_t v)
{
    asm volatile("st.shared.u16 [%0], %1;" ::"r"(a), "r"(v));  // low 16 bits stored
}

// A 32-bit constant the compiler cannot fold back into immediates, so it is
// materialised once and kept in a register.
__device__ __forceinline__ uint32_t opaque(uint32_t v)
{
    uint32_t r;
    asm volatile("mov.b32 %0, %1;" : "=r"(r) : "r"(v));
    return r;
}

__device__ __forceinline__ uint32_t ld_acquire_u32(const int32_t *p)
{
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Atomic add at GPU scope with acquire and release semantics; returns the
// old value.
__device__ __forceinline__ uint32_t atom_add_acq_rel(int32_t *p, uint32_t v)
{
    uint32_t old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;"
                 : "=r"(old)
                 : "l"(p), "r"(v)
                 : "memory");
    return old;
}

// Programmatic dependent launch: the wait for the grids this one depends on
// (their writes visible), and the signal that the grids depending on this
// one may be scheduled.
__device__ __forceinline__ void grid_dependency_wait()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// (x & m) | c in one LOP3.
__device__ __forceinline__ uint32_t and_or(uint32_t x, uint32_t m, uint32_t c)
{
    uint32_t r;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(x), "r"(m), "r"(c));
    return r;
}

// Register constants of the Q4_0 nibble expansion: masks and f16 biases.
struct NibbleConsts {
    uint32_t mlo, mhi, blo, bhi;  // 0x000F000F, 0x00F000F0, f16 1024 | 1024, f16 64 | 64
    uint32_t nlo[4], nhi[4];      // -1032 and -72 (f16 pairs): 1024 + n or 64 + n to n - 8
    __device__ __forceinline__ void init()
    {
        mlo = opaque(0x000F000Fu);
        mhi = opaque(0x00F000F0u);
        blo = opaque(0x64006400u);
        bhi = opaque(0x54005400u);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            nlo[i] = opaque(0xE408E408u);
            nhi[i] = opaque(0xD480D480u);
        }
    }
};

// Transposes an 8x8 matrix of 16-bit values held in mma fragment layout.
__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x)
{
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

// ------------------------------------------------------------ per-type code
//
// Each type provides the layout of one ring slot and, for one warp, the
// query fragments, the scores of one 16-token tile and the PV update of one
// tile.  Thread roles follow the m16n8k16 fragment layout: gid = lane/4,
// tig = lane%4.
//  QK: A = keys (row = token of the tile), B = queries (column gid = query
//      head of the group; columns >= G are zero), C = S[token][head].  Each
//      thread ends with the scores of tokens gid, gid+8 for heads 2tig, 2tig+1
//      in log2 units.
//  PV: A = values (row = head dimension), B = probabilities (column gid =
//      query head), C = O[dimension][head]: columns 2tig, 2tig+1 are again this
//      thread's heads.

// --- the q8_1 query, shared by the quantised-K types ------------------------
//
// Lane (gid, tig) holds, for query head gid of its group, the eight values of
// each 32-value block at dims 4tig..4tig+3 and 16+4tig..19+4tig: float32 when
// the kernel quantises the query itself, else the q8_1 codes and scale.  They
// are fetched before the first K/V copies are issued, so that these loads do
// not queue behind them.
template <int NB>
struct Q81Query {
    struct Raw {
        float4 x[NB][2];
        uint32_t w[NB][2];
        uint32_t d[NB];
    };

    // Blocks b with b % nw == w only: the nw warps of a K/V head share the work.
    __device__ static void fetch(const DecodeParams &p, uint32_t s, uint32_t h0, uint32_t G,
                                 int gid, int tig, uint32_t w, uint32_t nw, Raw &r)
    {
        const uint64_t row = (uint64_t)s * p.hq + h0 + ((uint32_t)gid < G ? gid : 0);
        if (p.q_f32) {
            const float *x = static_cast<const float *>(p.q) + row * NB * 32;
#pragma unroll
            for (int b = 0; b < NB; ++b) {
                if ((uint32_t)b % nw != w)
                    continue;
                r.x[b][0] = *reinterpret_cast<const float4 *>(x + 32 * b + 4 * tig);
                r.x[b][1] = *reinterpret_cast<const float4 *>(x + 32 * b + 16 + 4 * tig);
            }
        } else {
            const uint8_t *blk = static_cast<const uint8_t *>(p.q) + row * NB * 36;
#pragma unroll
            for (int b = 0; b < NB; ++b) {
                if ((uint32_t)b % nw != w)
                    continue;
                r.d[b] = load_u16(blk + 36 * b);
                r.w[b][0] = *reinterpret_cast<const uint32_t *>(blk + 36 * b + 4 + 4 * tig);
                r.w[b][1] = *reinterpret_cast<const uint32_t *>(blk + 36 * b + 20 + 4 * tig);
            }
        }
    }

    // The q8_1 codes of this lane's eight values of block b and the block's
    // f16-rounded scale.  A float32 query is quantised with the pre-pass's
    // arithmetic (q8_1_code); the four lanes of a quad hold one block, so its
    // maximum magnitude is two shuffles away.
    __device__ static __forceinline__ void codes(const DecodeParams &p, const Raw &r, int b,
                                                 int (&code)[8], float &d16)
    {
        if (p.q_f32) {
            const float v[8] = {r.x[b][0].x, r.x[b][0].y, r.x[b][0].z, r.x[b][0].w,
                                r.x[b][1].x, r.x[b][1].y, r.x[b][1].z, r.x[b][1].w};
            float amax = 0.0f;
#pragma unroll
            for (int j = 0; j < 8; ++j)
                amax = fmaxf(amax, fabsf(v[j]));
            amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
            amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
            const float d = amax / 127.0f, inv_d = 1.0f / d;
            // q8_1_code without its division: the product by 1 / d rounds
            // to the quotient's code unless it lies within 3e-5 of a
            // half-integer (or is not finite) in some lane; then the warp
            // takes q8_1_code itself for the block
            bool near = false;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const float rj = v[j] * inv_d, a = fabsf(rj);
                near |= !(fabsf(a - truncf(a) - 0.5f) > 3.0e-5f);
                code[j] = (int)fminf(fmaxf(roundf(rj), -127.0f), 127.0f);
            }
            if (__any_sync(0xffffffffu, near)) {
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    code[j] = q8_1_code(v[j], amax, d, inv_d);
            }
            d16 = __half2float(__float2half_rn(amax == 0.0f ? 0.0f : d));
        } else {
#pragma unroll
            for (int j = 0; j < 8; ++j)
                code[j] = (int)(int8_t)(uint8_t)(r.w[b][j >> 2] >> (8 * (j & 3)));
            d16 = half_bits_to_float((uint16_t)r.d[b]);
        }
    }
};

// --- Q4_0, D = 256 --------------------------------------------------------
template <uint32_t KMAXW>
struct Q40T {
    static constexpr int D = 256;
    static constexpr int NB = D / 32;       // 32-value blocks per row
    static constexpr int RB = NB * 18;      // row bytes
    static constexpr int MT = D / 16;       // PV m-tiles
    static constexpr int DK = 0, DV = NB * kTile * 4;  // scratch: dk f32, dv f16
    static constexpr int SCRATCH = NB * kTile * 4 + NB * kTile * 2;
    static constexpr bool kZeroInvalidV = false;
    static constexpr uint32_t kTmaX = 1;    // TMA boxes per (side, head)
    static constexpr uint32_t kMaxWarps = KMAXW;
    static constexpr int kMergeBatch = 8;
    static constexpr bool kStagedMerge = true;
    // the one-launch instance takes 32-token tiles from rings shared by the
    // warps of a K/V head (range_body32); its scratch holds two 16-token halves
    static constexpr bool kTile32 = true;
    static constexpr int SCRATCH2 = 2 * SCRATCH;
    static constexpr bool kStream = true;

    static __host__ __device__ constexpr uint32_t side_bytes(uint32_t hkv)
    {
        return hkv * kTile * RB;
    }

    // Slot layout and tensor maps: both sides alike.
    static constexpr uint32_t kSideK = side_bytes(1), kSideV = side_bytes(1);
    static constexpr uint32_t kVOff = kSideK, kSlot = kSideK + kSideV;
    static constexpr uint32_t kTmaXK = kTmaX, kTmaXV = kTmaX;
    static constexpr uint32_t kRowK = kSideK / kTile, kRowV = kSideV / kTile;
    static constexpr bool kExtract = !kZeroInvalidV;
    static constexpr uint32_t kTypeKey = PA_Q4_0 * 3 + PA_Q4_0;

    // Query fragments live in shared memory, one 16-byte record per (block,
    // lane) of each K/V head (the four B registers), then the bias term of
    // each (query head, block): minus the sum of the block's qhat times 1032
    // (low nibbles, read as 1024 + n) or 72 (high nibbles, read as 64 + n).
    static constexpr int QREC = 16;                      // one uint4 per (block, lane)
    static constexpr int QCORR = NB * 32 * QREC;         // offset of the bias terms
    static constexpr int QBYTES = QCORR + 8 * NB * 4;    // per K/V head
    struct Frag {
        uint32_t q;                 // shared address of this lane's records (block 0)
        uint32_t ch0, ch1, cl0, cl1;  // bias of head gid, blocks tig, tig+4: tf32 high, low parts
    };

    using Consts = NibbleConsts;
    using QRaw = typename Q81Query<NB>::Raw;
    __device__ static void fetch_q(const DecodeParams &p, uint32_t s, uint32_t h0, uint32_t G,
                                   int gid, int tig, uint32_t w, uint32_t nw, QRaw &r)
    {
        Q81Query<NB>::fetch(p, s, h0, G, gid, tig, w, nw, r);
    }

    // Writes the fragments of query head gid of the group: qhat = f16(q * d_q
    // * scale * log2 e), in the dimension order the nibble expansion produces
    // (see block()).  One warp per K/V head calls this.
    __device__ static void store_q(const DecodeParams &p, const QRaw &r, uint32_t G, int gid,
                                   int tig, uint32_t w, uint32_t nw, uint32_t qsm)
    {
        const int lane = gid * 4 + tig;
        const bool live = (uint32_t)gid < G;
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            if ((uint32_t)b % nw != w)
                continue;
            int code[8];
            float d16;
            Q81Query<NB>::codes(p, r, b, code, d16);
            const float d = live ? d16 * p.scale_log2 : 0.0f;
            __half qh[8];
            float corr = 0.0f;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                qh[j] = __float2half_rn((float)code[j] * d);
                // low nibbles read as 1024 + n, high as 64 + n; the value is n - 8
                corr += __half2float(qh[j]) * (j < 4 ? 1032.0f : 72.0f);
            }
            corr += __shfl_xor_sync(0xffffffffu, corr, 1);
            corr += __shfl_xor_sync(0xffffffffu, corr, 2);
            const uint32_t rr = qsm + (b * 32 + lane) * QREC;
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(rr),
                         "r"(h2_bits(__halves2half2(qh[0], qh[2]))),
                         "r"(h2_bits(__halves2half2(qh[1], qh[3]))),
                         "r"(h2_bits(__halves2half2(qh[4], qh[6]))),
                         "r"(h2_bits(__halves2half2(qh[5], qh[7]))));
            if (tig == 0)
                sts_f32(qsm + QCORR + 4 * (gid * NB + b), -corr);
        }
    }

    // The query records of every K/V head of query row s (what store_q
    // writes, bit for bit), by all threads of the CTA at once: thread item
    // i = (head h, block b, half c) holds the 16 values of lanes tig = 2c,
    // 2c+1 of the block's quad -- dims 8c..8c+7 and 16+8c..16+8c+7.  One
    // item per thread instead of NB / wph blocks per warp in turn; the
    // codes, scales and bias sums are formed in the same order as there.
    struct QItems {
        float4 x[4];      // f32 query: dims 8c..8c+3, 8c+4.., 16+8c.., 20+8c..
        uint32_t w[4];    // q8_1 query: the codes of the same dims
        uint32_t d;       // q8_1 query: the block's f16 scale
    };
    __device__ static void fetch_q_cta(const DecodeParams &p, uint32_t s, uint32_t i, QItems &r)
    {
        if (i >= p.hq * 16)
            return;
        const uint32_t h = i >> 4, b = (i >> 1) & 7, c = i & 1;
        const uint64_t row = (uint64_t)s * p.hq + h;
        if (p.q_f32) {
            const float *x = static_cast<const float *>(p.q) + row * D + 32 * b + 8 * c;
#pragma unroll
            for (int k = 0; k < 4; ++k)
                r.x[k] = *reinterpret_cast<const float4 *>(x + 16 * (k >> 1) + 4 * (k & 1));
        } else {
            const uint8_t *blk = static_cast<const uint8_t *>(p.q) + row * NB * 36 + 36 * b;
            r.d = load_u16(blk);
#pragma unroll
            for (int k = 0; k < 4; ++k)
                r.w[k] = *reinterpret_cast<const uint32_t *>(blk + 4 + 8 * c + 16 * (k >> 1) +
                                                             4 * (k & 1));
        }
    }
    // Every thread of the CTA, after fetch_q_cta of item threadIdx.x: the
    // records of the live heads (items past the CTA's threads in further
    // rounds), zero records and bias terms for the columns past each group.
    __device__ static void store_q_cta(const DecodeParams &p, uint32_t s, QItems &r,
                                       uint32_t qsm_base)
    {
        const uint32_t hq = p.hq, G = hq / p.hkv, n = hq * 16, nt = blockDim.x;
        for (uint32_t k = threadIdx.x; k < p.hkv * (8 - G) * NB * 4; k += nt) {
            const uint32_t tig = k & 3, b = (k >> 2) % NB, rr = (k >> 2) / NB;
            const uint32_t g = rr / (8 - G), gid = G + rr % (8 - G);
            const uint32_t base = qsm_base + g * QBYTES;
            asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(
                             base + (b * 32 + gid * 4 + tig) * QREC),
                         "r"(0u));
            if (tig == 0)
                sts_f32(base + QCORR + 4 * (gid * NB + b), 0.0f);
        }
        // a warp's items: all of it or none live but at the end (n is a
        // multiple of 16, nt of 32)
        for (uint32_t i = threadIdx.x; i - (i & 31) < n; i += nt) {
            if (i >= nt)
                fetch_q_cta(p, s, i, r);
            item_q_cta(p, r, i, qsm_base);
        }
    }
    __device__ static __forceinline__ void item_q_cta(const DecodeParams &p, const QItems &r,
                                                      uint32_t i, uint32_t qsm_base)
    {
        const uint32_t hq = p.hq, G = hq / p.hkv, n = hq * 16;
        const bool live = i < n;
        const uint32_t h = i >> 4, b = (i >> 1) & 7, c = i & 1;
        int code[16];  // dims 8c+k (k < 8), 16+8c+k-8 (k >= 8)
        float d16;
        if (p.q_f32) {
            float v[16];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                v[4 * k] = live ? r.x[k].x : 0.0f;
                v[4 * k + 1] = live ? r.x[k].y : 0.0f;
                v[4 * k + 2] = live ? r.x[k].z : 0.0f;
                v[4 * k + 3] = live ? r.x[k].w : 0.0f;
            }
            float amax = 0.0f;
#pragma unroll
            for (int k = 0; k < 16; ++k)
                amax = fmaxf(amax, fabsf(v[k]));
            amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
            const float d = amax / 127.0f, inv_d = 1.0f / d;
            bool near = false;
#pragma unroll
            for (int k = 0; k < 16; ++k) {
                const float rk = v[k] * inv_d, a = fabsf(rk);
                near |= !(fabsf(a - truncf(a) - 0.5f) > 3.0e-5f);
                code[k] = (int)fminf(fmaxf(roundf(rk), -127.0f), 127.0f);
            }
            if (__any_sync(0xffffffffu, near)) {
#pragma unroll
                for (int k = 0; k < 16; ++k)
                    code[k] = q8_1_code(v[k], amax, d, inv_d);
            }
            d16 = __half2float(__float2half_rn(amax == 0.0f ? 0.0f : d));
        } else {
#pragma unroll
            for (int k = 0; k < 16; ++k)
                code[k] = (int)(int8_t)(uint8_t)(r.w[k >> 2] >> (8 * (k & 3)));
            d16 = half_bits_to_float((uint16_t)r.d);
        }
        const float d = d16 * p.scale_log2;
        const uint32_t g = h / G, gid = h % G;
        const uint32_t base = qsm_base + g * QBYTES;
        float cc = 0.0f;
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            // lane tig = 2c + e: j = 0..3 dims 4tig.., j = 4..7 dims 16+4tig..
            __half qh[8];
            float corr = 0.0f;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                qh[j] = __float2half_rn((float)code[(j < 4 ? 0 : 8) + 4 * e + (j & 3)] * d);
                corr += __half2float(qh[j]) * (j < 4 ? 1032.0f : 72.0f);
            }
            cc = e == 0 ? corr : cc + corr;
            if (live)
                asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(
                                 base + (b * 32 + gid * 4 + 2 * c + e) * QREC),
                             "r"(h2_bits(__halves2half2(qh[0], qh[2]))),
                             "r"(h2_bits(__halves2half2(qh[1], qh[3]))),
                             "r"(h2_bits(__halves2half2(qh[4], qh[6]))),
                             "r"(h2_bits(__halves2half2(qh[5], qh[7]))));
        }
        cc += __shfl_xor_sync(0xffffffffu, cc, 1);
        if (live && c == 0)
            sts_f32(base + QCORR + 4 * (gid * NB + b), -cc);
    }

    // The B fragments of the bias product (see scores()): blocks tig and
    // tig+4 of head gid, as a tf32 high part and the tf32 remainder, so the
    // pair holds the f32 term to about 21 bits.
    __device__ static void load_q(uint32_t qsm, int lane, Frag &f)
    {
        f.q = qsm + lane * QREC;
        const uint32_t c = qsm + QCORR + 4 * ((lane >> 2) * NB + (lane & 3));
        const float c0 = lds_f32(c), c1 = lds_f32(c + 16);
        f.ch0 = to_tf32(c0);
        f.ch1 = to_tf32(c1);
        f.cl0 = to_tf32(c0 - __uint_as_float(f.ch0));
        f.cl1 = to_tf32(c1 - __uint_as_float(f.ch1));
    }

    // Block scales of the tile into the warp's scratch: dk as float with the
    // pair (t, t+8) adjacent, dv as half in token order; zero for invalid tokens.
    __device__ static void extract(uint32_t kh, uint32_t vh, uint32_t scr, int nvalid, int lane)
    {
        // lane covers token t = lane % 16 of blocks lane / 16 + 2k, k = 0..3
        const int t = lane & 15, b0 = lane >> 4;
        const bool v = t < nvalid;
        const uint32_t ka = kh + t * RB + 18 * b0, va = vh + t * RB + 18 * b0;
        const uint32_t sk = scr + DK + 4 * (b0 * kTile + 2 * (t & 7) + (t >> 3));
        const uint32_t sv = scr + DV + 2 * (b0 * kTile + t);
#pragma unroll
        for (int k = 0; k < NB / 2; ++k) {
            const uint32_t kd = lds_u16(ka + 36 * k);
            const uint32_t vd = lds_u16(va + 36 * k);
            sts_f32(sk + 128 * k, v ? half_bits_to_float((uint16_t)kd) : 0.0f);
            sts_u16(sv + 64 * k, v ? vd : 0u);
        }
    }

    // The K and V halves of extract, for rows of this type beside the other
    // side's rows of another type.
    __device__ static void extract_k(uint32_t kh, uint32_t scr, int nvalid, int lane)
    {
        const int t = lane & 15, b0 = lane >> 4;
        const bool v = t < nvalid;
        const uint32_t ka = kh + t * RB + 18 * b0;
        const uint32_t sk = scr + DK + 4 * (b0 * kTile + 2 * (t & 7) + (t >> 3));
#pragma unroll
        for (int k = 0; k < NB / 2; ++k)
            sts_f32(sk + 128 * k, v ? half_bits_to_float((uint16_t)lds_u16(ka + 36 * k)) : 0.0f);
    }
    __device__ static void extract_v(uint32_t vh, uint32_t scr, int nvalid, int lane)
    {
        const int t = lane & 15, b0 = lane >> 4;
        const bool v = t < nvalid;
        const uint32_t va = vh + t * RB + 18 * b0;
        const uint32_t sv = scr + DV + 2 * (b0 * kTile + t);
#pragma unroll
        for (int k = 0; k < NB / 2; ++k)
            sts_u16(sv + 64 * k, v ? lds_u16(va + 36 * k) : 0u);
    }

    // One 32-value block: x0 / x1 are the nibble words of tokens gid / gid+8
    // holding dims 4tig..4tig+3 (low nibbles) and 16+4tig..19+4tig (high).
    // The block's dot of the biased nibbles, times d_k, adds to s.
    __device__ static __forceinline__ void block(const NibbleConsts &K, uint32_t qrec, uint32_t x0,
                                                 uint32_t x1, float2 dk, float (&s)[4])
    {
        uint32_t qb0, qb1, qb2, qb3;
        float c[4];
        const float zero[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
            : "=r"(qb0), "=r"(qb1), "=r"(qb2), "=r"(qb3)
            : "r"(qrec)
            : "memory");
        const uint32_t y0 = x0 >> 8, y1 = x1 >> 8;
        mma16816_c(c, and_or(x0, K.mlo, K.blo), and_or(x1, K.mlo, K.blo), and_or(y0, K.mlo, K.blo),
                   and_or(y1, K.mlo, K.blo), qb0, qb1, zero);
        mma16816(c, and_or(x0, K.mhi, K.bhi), and_or(x1, K.mhi, K.bhi), and_or(y0, K.mhi, K.bhi),
                 and_or(y1, K.mhi, K.bhi), qb2, qb3);
        s[0] = fmaf(c[0], dk.x, s[0]);
        s[1] = fmaf(c[1], dk.x, s[1]);
        s[2] = fmaf(c[2], dk.y, s[2]);
        s[3] = fmaf(c[3], dk.y, s[3]);
    }

    // Scores of the tile: s starts at the bias term sum_b d_k[t][b] *
    // bias[head][b], two tf32 MMAs over the 8 blocks (A: the d_k of tokens
    // gid, gid+8, blocks tig, tig+4, exact in tf32 as f16 values; B: the
    // bias's high part, then its remainder); then each block adds d_k times
    // the dot of its biased nibbles.
    // block() for the two 16-token halves of a 32-token tile: one load of
    // the query record serves both (x: rows gid, gid+8; z: rows 16+gid, 24+gid).
    __device__ static __forceinline__ void block2(const NibbleConsts &K, uint32_t qrec, uint32_t x0,
                                                  uint32_t x1, uint32_t z0, uint32_t z1, float2 dkx,
                                                  float2 dkz, float (&sx)[4], float (&sz)[4])
    {
        uint32_t qb0, qb1, qb2, qb3;
        const float zero[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
            : "=r"(qb0), "=r"(qb1), "=r"(qb2), "=r"(qb3)
            : "r"(qrec)
            : "memory");
        {
            float c[4];
            const uint32_t y0 = x0 >> 8, y1 = x1 >> 8;
            mma16816_c(c, and_or(x0, K.mlo, K.blo), and_or(x1, K.mlo, K.blo),
                       and_or(y0, K.mlo, K.blo), and_or(y1, K.mlo, K.blo), qb0, qb1, zero);
            mma16816(c, and_or(x0, K.mhi, K.bhi), and_or(x1, K.mhi, K.bhi),
                     and_or(y0, K.mhi, K.bhi), and_or(y1, K.mhi, K.bhi), qb2, qb3);
            sx[0] = fmaf(c[0], dkx.x, sx[0]);
            sx[1] = fmaf(c[1], dkx.x, sx[1]);
            sx[2] = fmaf(c[2], dkx.y, sx[2]);
            sx[3] = fmaf(c[3], dkx.y, sx[3]);
        }
        {
            float c[4];
            const uint32_t y0 = z0 >> 8, y1 = z1 >> 8;
            mma16816_c(c, and_or(z0, K.mlo, K.blo), and_or(z1, K.mlo, K.blo),
                       and_or(y0, K.mlo, K.blo), and_or(y1, K.mlo, K.blo), qb0, qb1, zero);
            mma16816(c, and_or(z0, K.mhi, K.bhi), and_or(z1, K.mhi, K.bhi),
                     and_or(y0, K.mhi, K.bhi), and_or(y1, K.mhi, K.bhi), qb2, qb3);
            sz[0] = fmaf(c[0], dkz.x, sz[0]);
            sz[1] = fmaf(c[1], dkz.x, sz[1]);
            sz[2] = fmaf(c[2], dkz.y, sz[2]);
            sz[3] = fmaf(c[3], dkz.y, sz[3]);
        }
    }

    // The bias product of scores() for one 16-token half (scratch scr).
    __device__ static __forceinline__ void bias16(const Frag &f, uint32_t scr, int gid, int tig,
                                                  float (&s)[4])
    {
        const uint32_t dk = scr + DK + 8 * gid;
        const float2 d0 = lds_f2(dk + 4 * kTile * tig), d1 = lds_f2(dk + 4 * kTile * (tig + 4));
        const uint32_t a0 = __float_as_uint(d0.x), a1 = __float_as_uint(d0.y);
        const uint32_t a2 = __float_as_uint(d1.x), a3 = __float_as_uint(d1.y);
        const float zero[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        mma1688_tf32(s, a0, a1, a2, a3, f.ch0, f.ch1, zero);
        mma1688_tf32(s, a0, a1, a2, a3, f.cl0, f.cl1, s);
    }

    // scores() of a 32-token tile: K rows 0..31 at kh (pitch RB), the two
    // halves' scales at scr and scr + SCRATCH; sx: tokens 0..15, sz: 16..31.
    __device__ static void scores2(const NibbleConsts &K, const Frag &f, uint32_t kh, uint32_t scr,
                                   int gid, int tig, float (&sx)[4], float (&sz)[4])
    {
        uint32_t r0 = kh + gid * RB + 4 * tig;
        uint32_t dk = scr + DK + 8 * gid;
        uint32_t qr = f.q;
        bias16(f, scr, gid, tig, sx);
        bias16(f, scr + SCRATCH, gid, tig, sz);
#pragma unroll
        for (int pb = 0; pb < NB / 2; ++pb) {
            const uint32_t a0 = lds_u32(r0), a1 = lds_u32(r0 + 4), a2 = lds_u32(r0 + 20);
            const uint32_t b0 = lds_u32(r0 + 8 * RB), b1 = lds_u32(r0 + 8 * RB + 4);
            const uint32_t b2 = lds_u32(r0 + 8 * RB + 20);
            const uint32_t c0 = lds_u32(r0 + 16 * RB), c1 = lds_u32(r0 + 16 * RB + 4);
            const uint32_t c2 = lds_u32(r0 + 16 * RB + 20);
            const uint32_t d0 = lds_u32(r0 + 24 * RB), d1 = lds_u32(r0 + 24 * RB + 4);
            const uint32_t d2 = lds_u32(r0 + 24 * RB + 20);
            const float2 kx0 = lds_f2(dk), kx1 = lds_f2(dk + 4 * kTile);
            const float2 kz0 = lds_f2(dk + SCRATCH), kz1 = lds_f2(dk + SCRATCH + 4 * kTile);
            block2(K, qr, __funnelshift_r(a0, a1, 16), __funnelshift_r(b0, b1, 16),
                   __funnelshift_r(c0, c1, 16), __funnelshift_r(d0, d1, 16), kx0, kz0, sx, sz);
            block2(K, qr + 32 * QREC, a2, b2, c2, d2, kx1, kz1, sx, sz);
            r0 += 36;
            dk += 2 * 4 * kTile;
            qr += 2 * 32 * QREC;
        }
    }

    __device__ static void scores(const NibbleConsts &K, const Frag &f, uint32_t kh, uint32_t scr,
                                  int gid, int tig, float (&s)[4])
    {
        uint32_t r0 = kh + gid * RB + 4 * tig;
        uint32_t dk = scr + DK + 8 * gid;
        uint32_t qr = f.q;
        {
            const float2 d0 = lds_f2(dk + 4 * kTile * tig), d1 = lds_f2(dk + 4 * kTile * (tig + 4));
            const uint32_t a0 = __float_as_uint(d0.x), a1 = __float_as_uint(d0.y);
            const uint32_t a2 = __float_as_uint(d1.x), a3 = __float_as_uint(d1.y);
            const float zero[4] = {0.0f, 0.0f, 0.0f, 0.0f};
            mma1688_tf32(s, a0, a1, a2, a3, f.ch0, f.ch1, zero);
            mma1688_tf32(s, a0, a1, a2, a3, f.cl0, f.cl1, s);
        }
#pragma unroll
        for (int pb = 0; pb < NB / 2; ++pb) {
            // blocks 2pb and 2pb+1 share 36 bytes = 9 aligned words
            const uint32_t a0 = lds_u32(r0), a1 = lds_u32(r0 + 4), a2 = lds_u32(r0 + 20);
            const uint32_t b0 = lds_u32(r0 + 8 * RB), b1 = lds_u32(r0 + 8 * RB + 4);
            const uint32_t b2 = lds_u32(r0 + 8 * RB + 20);
            const float2 k0 = lds_f2(dk);
            const float2 k1 = lds_f2(dk + 4 * kTile);
            block(K, qr, __funnelshift_r(a0, a1, 16), __funnelshift_r(b0, b1, 16), k0, s);
            block(K, qr + 32 * QREC, a2, b2, k1, s);
            r0 += 36;
            dk += 2 * 4 * kTile;
            qr += 2 * 32 * QREC;
        }
    }

    // O += V^T P' over the tile, P' = P * d_v per block.  The V operand is the
    // nibble read as 1024 + n (low nibbles) or 64 + n (high nibbles) minus
    // 1032 (or 72): n - 8 exactly, one HADD2 per two values.
    __device__ static void pv(const NibbleConsts &K, float (&o)[MT][4], uint32_t vh, uint32_t scr,
                              uint32_t p0, uint32_t p1, int gid, int tig)
    {
        const uint32_t ra = vh + (2 * tig) * RB + 2 + 2 * gid;
        const uint32_t rc = ra + 8 * RB;
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            const uint32_t ua = lds_u16(ra + 18 * b), ub = lds_u16(ra + RB + 18 * b);
            const uint32_t uc = lds_u16(rc + 18 * b), ud = lds_u16(rc + RB + 18 * b);
            const uint32_t xab = __byte_perm(ua, ub, 0x5410), yab = xab >> 8;
            const uint32_t xcd = __byte_perm(uc, ud, 0x5410), ycd = xcd >> 8;
            const uint32_t b0 = hmul2_bits(p0, lds_u32(scr + DV + 2 * (b * kTile + 2 * tig)));
            const uint32_t b1 = hmul2_bits(p1, lds_u32(scr + DV + 2 * (b * kTile + 8 + 2 * tig)));
            // (1024 + n) - 1032 and (64 + n) - 72 are n - 8 exactly
            mma16816(o[2 * b], hadd2_bits(and_or(xab, K.mlo, K.blo), K.nlo[0]),
                     hadd2_bits(and_or(yab, K.mlo, K.blo), K.nlo[1]),
                     hadd2_bits(and_or(xcd, K.mlo, K.blo), K.nlo[2]),
                     hadd2_bits(and_or(ycd, K.mlo, K.blo), K.nlo[3]), b0, b1);
            mma16816(o[2 * b + 1], hadd2_bits(and_or(xab, K.mhi, K.bhi), K.nhi[0]),
                     hadd2_bits(and_or(yab, K.mhi, K.bhi), K.nhi[1]),
                     hadd2_bits(and_or(xcd, K.mhi, K.bhi), K.nhi[2]),
                     hadd2_bits(and_or(ycd, K.mhi, K.bhi), K.nhi[3]), b0, b1);
        }
    }

    // Output dimension of PV C-fragment row (gid or gid+8) of m-tile mt.
    __device__ static __forceinline__ int dim_of(int mt, int gid, int upper)
    {
        return 32 * (mt >> 1) + 16 * (mt & 1) + 2 * gid + upper;
    }
    static constexpr bool kDimPairs = true;  // dim_of(mt, gid, 1) == dim_of(mt, gid, 0) + 1
};

using Q40 = Q40T<12>;

// --- Q8_0, D = 256 --------------------------------------------------------
// Slot layout per side: 16 rows of 272 bytes (eight 34-byte blocks: f16 d,
// then 32 int8 codes), written by TMA without swizzle; the 272-byte pitch puts
// the rows of a warp's loads in different banks.
//  QK runs on the integer tensor path: mma m16n8k32 s8 x s8 -> s32 takes the
//  Q8_0 codes of 16 tokens x 32 dims as A and the q8_1 codes of the query as
//  B, so each block's dot is an exact integer (the pages' q8_1 dot), scaled by
//  d_k * d_q * scale * log2 e in f32.
//  PV: the code c becomes the exact f16 1024 + (c ^ 0x80) with one byte
//  permute per two values; one extra MMA with every A entry -1152 removes the
//  bias, and d_v is folded into P as for Q4_0.
template <uint32_t KMAXW>
struct Q80T {
    static constexpr int D = 256;
    static constexpr int NB = D / 32;
    static constexpr int BB = 34;           // block bytes
    static constexpr int RB = NB * BB;      // row bytes (272)
    static constexpr int MT = D / 16;
    static constexpr int DK = 0, DV = NB * kTile * 4;
    static constexpr int SCRATCH = NB * kTile * 4 + NB * kTile * 2;
    static constexpr bool kZeroInvalidV = false;
    static constexpr uint32_t kTmaX = 1;
    static constexpr uint32_t kMaxWarps = KMAXW;
    static constexpr int kMergeBatch = 12;
    static constexpr bool kStagedMerge = true;
    static constexpr bool kStream = true;
    static constexpr bool kTile32 = false;

    static __host__ __device__ constexpr uint32_t side_bytes(uint32_t hkv)
    {
        return hkv * kTile * RB;
    }

    // Slot layout and tensor maps: both sides alike.
    static constexpr uint32_t kSideK = side_bytes(1), kSideV = side_bytes(1);
    static constexpr uint32_t kVOff = kSideK, kSlot = kSideK + kSideV;
    static constexpr uint32_t kTmaXK = kTmaX, kTmaXV = kTmaX;
    static constexpr uint32_t kRowK = kSideK / kTile, kRowV = kSideV / kTile;
    static constexpr bool kExtract = !kZeroInvalidV;
    static constexpr uint32_t kTypeKey = PA_Q8_0 * 3 + PA_Q8_0;

    struct Consts {
        uint32_t flip, f16hi;  // 0x80808080; bytes 0x64 (the high byte of f16 1024)
        uint32_t nb[4];        // A quad of -1152 (f16 pairs)
        __device__ __forceinline__ void init()
        {
            flip = opaque(0x80808080u);
            f16hi = opaque(0x64646464u);
#pragma unroll
            for (int i = 0; i < 4; ++i)
                nb[i] = opaque(0xE480E480u);
        }
    };

    // Query fragments in shared memory, one 16-byte record per (block, lane)
    // of each K/V head: the two B registers (the q8_1 codes of query head gid
    // at dims 4tig.. and 16+4tig..), then d_q * scale * log2 e of the heads
    // 2tig and 2tig+1 (this thread's C columns).
    static constexpr int QREC = 16;
    static constexpr int QBYTES = NB * 32 * QREC;
    struct Frag {
        uint32_t q;
    };
    using QRaw = typename Q81Query<NB>::Raw;

    __device__ static void fetch_q(const DecodeParams &p, uint32_t s, uint32_t h0, uint32_t G,
                                   int gid, int tig, uint32_t w, uint32_t nw, QRaw &r)
    {
        Q81Query<NB>::fetch(p, s, h0, G, gid, tig, w, nw, r);
    }

    __device__ static void store_q(const DecodeParams &p, const QRaw &r, uint32_t G, int gid,
                                   int tig, uint32_t w, uint32_t nw, uint32_t qsm)
    {
        const int lane = gid * 4 + tig;
        const bool live = (uint32_t)gid < G;
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            if ((uint32_t)b % nw != w)
                continue;
            int code[8];
            float d16;
            Q81Query<NB>::codes(p, r, b, code, d16);
            const float dq = live ? d16 * p.scale_log2 : 0.0f;
            uint32_t w[2];
#pragma unroll
            for (int h = 0; h < 2; ++h)
                w[h] = (uint32_t)(code[4 * h] & 0xFF) | (uint32_t)(code[4 * h + 1] & 0xFF) << 8 |
                       (uint32_t)(code[4 * h + 2] & 0xFF) << 16 |
                       (uint32_t)(code[4 * h + 3] & 0xFF) << 24;
            // the scales of heads 2tig and 2tig+1 live in lanes 8tig and 8tig+4
            const float q0 = __shfl_sync(0xffffffffu, dq, 8 * tig);
            const float q1 = __shfl_sync(0xffffffffu, dq, 8 * tig + 4);
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(
                             qsm + (b * 32 + lane) * QREC),
                         "r"(w[0]), "r"(w[1]), "r"(__float_as_uint(q0)), "r"(__float_as_uint(q1)));
        }
    }

    __device__ static void load_q(uint32_t qsm, int lane, Frag &f) { f.q = qsm + lane * QREC; }

    // Block scales into the warp's scratch, as for Q4_0: dk as float with the
    // pair (t, t+8) adjacent, dv as half in token order; zero for invalid tokens.
    __device__ static void extract(uint32_t kh, uint32_t vh, uint32_t scr, int nvalid, int lane)
    {
        const int t = lane & 15, b0 = lane >> 4;
        const bool v = t < nvalid;
        const uint32_t ka = kh + t * RB + BB * b0, va = vh + t * RB + BB * b0;
        const uint32_t sk = scr + DK + 4 * (b0 * kTile + 2 * (t & 7) + (t >> 3));
        const uint32_t sv = scr + DV + 2 * (b0 * kTile + t);
#pragma unroll
        for (int k = 0; k < NB / 2; ++k) {
            const uint32_t kd = lds_u16(ka + 2 * BB * k);
            const uint32_t vd = lds_u16(va + 2 * BB * k);
            sts_f32(sk + 128 * k, v ? half_bits_to_float((uint16_t)kd) : 0.0f);
            sts_u16(sv + 64 * k, v ? vd : 0u);
        }
    }

    __device__ static void extract_k(uint32_t kh, uint32_t scr, int nvalid, int lane)
    {
        const int t = lane & 15, b0 = lane >> 4;
        const bool v = t < nvalid;
        const uint32_t ka = kh + t * RB + BB * b0;
        const uint32_t sk = scr + DK + 4 * (b0 * kTile + 2 * (t & 7) + (t >> 3));
#pragma unroll
        for (int k = 0; k < NB / 2; ++k)
            sts_f32(sk + 128 * k,
                    v ? half_bits_to_float((uint16_t)lds_u16(ka + 2 * BB * k)) : 0.0f);
    }
    __device__ static void extract_v(uint32_t vh, uint32_t scr, int nvalid, int lane)
    {
        const int t = lane & 15, b0 = lane >> 4;
        const bool v = t < nvalid;
        const uint32_t va = vh + t * RB + BB * b0;
        const uint32_t sv = scr + DV + 2 * (b0 * kTile + t);
#pragma unroll
        for (int k = 0; k < NB / 2; ++k)
            sts_u16(sv + 64 * k, v ? lds_u16(va + 2 * BB * k) : 0u);
    }

    __device__ static __forceinline__ void imma(int (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                                uint32_t a3, uint32_t b0, uint32_t b1)
    {
        asm volatile(
            "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
            "{%8,%9}, {%0,%1,%2,%3};"
            : "+r"(c[0]), "+r"(c[1]), "+r"(c[2]), "+r"(c[3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    }

    // One block: a0..a3 are the code words of tokens gid / gid+8 at dims
    // 4tig.. (a0, a1) and 16+4tig.. (a2, a3).
    __device__ static __forceinline__ void block(uint32_t qrec, uint32_t a0, uint32_t a1,
                                                 uint32_t a2, uint32_t a3, float2 dk,
                                                 float (&s)[4])
    {
        uint32_t b0, b1, q0, q1;
        asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
            : "=r"(b0), "=r"(b1), "=r"(q0), "=r"(q1)
            : "r"(qrec)
            : "memory");
        int c[4] = {0, 0, 0, 0};
        imma(c, a0, a1, a2, a3, b0, b1);
        const float dq0 = __uint_as_float(q0), dq1 = __uint_as_float(q1);
        s[0] = fmaf((float)c[0], dk.x * dq0, s[0]);
        s[1] = fmaf((float)c[1], dk.x * dq1, s[1]);
        s[2] = fmaf((float)c[2], dk.y * dq0, s[2]);
        s[3] = fmaf((float)c[3], dk.y * dq1, s[3]);
    }

    __device__ static void scores(const Consts &, const Frag &f, uint32_t kh, uint32_t scr,
                                  int gid, int tig, float (&s)[4])
    {
        // blocks 2pb (codes 2 bytes past a word boundary) and 2pb+1 (aligned)
        uint32_t r0 = kh + gid * RB + 4 * tig, r1 = r0 + 8 * RB;
        uint32_t dk = scr + DK + 8 * gid;
        uint32_t qr = f.q;
        s[0] = s[1] = s[2] = s[3] = 0.0f;
#pragma unroll
        for (int pb = 0; pb < NB / 2; ++pb) {
            const uint32_t x0 = lds_u32(r0), x1 = lds_u32(r0 + 4), x2 = lds_u32(r0 + 16),
                           x3 = lds_u32(r0 + 20);
            const uint32_t y0 = lds_u32(r1), y1 = lds_u32(r1 + 4), y2 = lds_u32(r1 + 16),
                           y3 = lds_u32(r1 + 20);
            const uint32_t u0 = lds_u32(r0 + 36), u2 = lds_u32(r0 + 52);
            const uint32_t v0 = lds_u32(r1 + 36), v2 = lds_u32(r1 + 52);
            const float2 k0 = lds_f2(dk), k1 = lds_f2(dk + 4 * kTile);
            block(qr, __funnelshift_r(x0, x1, 16), __funnelshift_r(y0, y1, 16),
                  __funnelshift_r(x2, x3, 16), __funnelshift_r(y2, y3, 16), k0, s);
            block(qr + 32 * QREC, u0, v0, u2, v2, k1, s);
            r0 += 2 * BB;
            r1 += 2 * BB;
            dk += 2 * 4 * kTile;
            qr += 2 * 32 * QREC;
        }
    }

    // O += V^T P' over the tile, P' = P * d_v per block.  m-tile 2b holds dims
    // 32b + 2gid (row gid) and 32b + 2gid + 1 (row gid + 8); m-tile 2b+1 the
    // same 16 dims higher.  A register pairs one dim of tokens (2tig, 2tig+1)
    // or (2tig+8, 2tig+9).
    __device__ static void pv(const Consts &K, float (&o)[MT][4], uint32_t vh, uint32_t scr,
                              uint32_t p0, uint32_t p1, int gid, int tig)
    {
        const uint32_t ra = vh + (2 * tig) * RB + 2 + 2 * gid;
        const uint32_t rc = ra + 8 * RB;
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            const uint32_t b0 = hmul2_bits(p0, lds_u32(scr + DV + 2 * (b * kTile + 2 * tig)));
            const uint32_t b1 =
                hmul2_bits(p1, lds_u32(scr + DV + 2 * (b * kTile + 8 + 2 * tig)));
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const uint32_t off = BB * b + 16 * hh;
                const uint32_t ua = lds_u16(ra + off), ub = lds_u16(ra + RB + off);
                const uint32_t uc = lds_u16(rc + off), ud = lds_u16(rc + RB + off);
                // [a.dim0, a.dim1, b.dim0, b.dim1], each code flipped to c + 128
                const uint32_t xab = __byte_perm(ua, ub, 0x5410) ^ K.flip;
                const uint32_t xcd = __byte_perm(uc, ud, 0x5410) ^ K.flip;
                // the bias 1152 comes off in a second MMA with a constant A
                // (for Q8_0 this keeps more time than the operand subtraction
                // that Q4_0 uses)
                float(&acc)[4] = o[2 * b + hh];
                mma16816(acc, __byte_perm(xab, K.f16hi, 0x4240), __byte_perm(xab, K.f16hi, 0x4341),
                         __byte_perm(xcd, K.f16hi, 0x4240), __byte_perm(xcd, K.f16hi, 0x4341),
                         b0, b1);
                mma16816(acc, K.nb[0], K.nb[1], K.nb[2], K.nb[3], b0, b1);
            }
        }
    }

    __device__ static __forceinline__ int dim_of(int mt, int gid, int upper)
    {
        return 16 * mt + 2 * gid + upper;
    }
    static constexpr bool kDimPairs = true;
};

using Q80 = Q80T<8>;

// --- F16, D = 128 or 256 ----------------------------------------------------
// Slot layout per side: [64-dim chunk][16 tokens][128 B], written by TMA with
// the 128-byte swizzle (16-byte chunk c of row t stored at c ^ (t & 7)), read
// with ldmatrix without bank conflicts.
template <int D_>
struct F16T {
    static constexpr int D = D_;
    static constexpr int NC = D / 64;   // 64-dim chunks
    static constexpr int KS = D / 16;   // k-steps
    static constexpr int MT = D / 16;
    static constexpr int SCRATCH = 0;
    static constexpr bool kZeroInvalidV = true;
    static constexpr uint32_t kTmaX = NC;
    static constexpr uint32_t kMaxWarps = 8;
    static constexpr int kMergeBatch = 12;
    static constexpr bool kStagedMerge = true;
    static constexpr bool kStream = true;
    static constexpr bool kTile32 = false;

    static __host__ __device__ constexpr uint32_t side_bytes(uint32_t hkv)
    {
        return hkv * kTile * D * 2;
    }

    // Slot layout and tensor maps: both sides alike.
    static constexpr uint32_t kSideK = side_bytes(1), kSideV = side_bytes(1);
    static constexpr uint32_t kVOff = kSideK, kSlot = kSideK + kSideV;
    static constexpr uint32_t kTmaXK = kTmaX, kTmaXV = kTmaX;
    static constexpr uint32_t kRowK = kSideK / kTile, kRowV = kSideV / kTile;
    static constexpr bool kExtract = !kZeroInvalidV;
    static constexpr uint32_t kTypeKey = (PA_F16 * 3 + PA_F16) + 9 * (D / 128);

    static constexpr int QBYTES = 0;
    struct Frag {
        uint32_t qb[KS][2];  // B fragments (query column gid) of each k-step
    };
    struct Consts {
        __device__ void init() {}
    };

    // This lane's query values (query head gid of the group), fetched before
    // the first K/V copies are issued so that the loads do not queue behind them.
    struct QRaw {
        float2 x[KS][2];
    };
    __device__ static void fetch_q(const DecodeParams &p, uint32_t s, uint32_t h0, uint32_t G,
                                   int gid, int tig, uint32_t, uint32_t, QRaw &r)
    {
        const float *row = static_cast<const float *>(p.q) +
                           ((uint64_t)s * p.hq + h0 + ((uint32_t)gid < G ? gid : 0)) * D;
#pragma unroll
        for (int j = 0; j < KS; ++j) {
            r.x[j][0] = *reinterpret_cast<const float2 *>(row + 16 * j + 2 * tig);
            r.x[j][1] = *reinterpret_cast<const float2 *>(row + 16 * j + 8 + 2 * tig);
        }
    }

    __device__ static void load_q(const DecodeParams &p, const QRaw &r, uint32_t G, int gid,
                                  Frag &f)
    {
        const float sc = (uint32_t)gid < G ? p.scale_log2 : 0.0f;
#pragma unroll
        for (int j = 0; j < KS; ++j) {
            f.qb[j][0] = h2_bits(__floats2half2_rn(r.x[j][0].x * sc, r.x[j][0].y * sc));
            f.qb[j][1] = h2_bits(__floats2half2_rn(r.x[j][1].x * sc, r.x[j][1].y * sc));
        }
    }

    __device__ static __forceinline__ uint32_t chunk_addr(uint32_t sub, int token, int c16)
    {
        return sub + token * 128 + ((c16 ^ (token & 7)) << 4);
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

    // Two accumulator chains (even and odd k-steps), added at the end: with
    // one warp per scheduler a single chain of KS dependent MMAs is latency.
    __device__ static void scores(const Consts &, const Frag &f, uint32_t kh, uint32_t,
                                  int gid, int tig, float (&s)[4])
    {
        const int lane = gid * 4 + tig;
        const int mi = lane >> 3, r = lane & 7;
        const int token = (mi & 1) * 8 + r;
        float c[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
        for (int j = 0; j < KS; ++j) {
            uint32_t a[4];
            ldsm_x4(a, chunk_addr(kh + (j >> 2) * kTile * 128, token, 2 * (j & 3) + (mi >> 1)));
            mma16816(c[j & 1], a[0], a[1], a[2], a[3], f.qb[j][0], f.qb[j][1]);
        }
        s[0] = c[0][0] + c[1][0];
        s[1] = c[0][1] + c[1][1];
        s[2] = c[0][2] + c[1][2];
        s[3] = c[0][3] + c[1][3];
    }

    __device__ static void pv(const Consts &, float (&o)[MT][4], uint32_t vh, uint32_t,
                              uint32_t p0, uint32_t p1, int gid, int tig)
    {
        const int lane = gid * 4 + tig;
        const int mi = lane >> 3, r = lane & 7;
        const int token = (mi >> 1) * 8 + r;
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
            uint32_t a[4];
            ldsm_x4_trans(a, chunk_addr(vh + (mt >> 2) * kTile * 128, token, (mt & 3) * 2 + (mi & 1)));
            mma16816(o[mt], a[0], a[1], a[2], a[3], p0, p1);
        }
    }

    __device__ static __forceinline__ int dim_of(int mt, int gid, int upper)
    {
        return 16 * mt + gid + 8 * upper;
    }
    static constexpr bool kDimPairs = false;
};

// --- mixed K x V types, D = 256 -------------------------------------------
// The K part of one type (query fragments, scores, K rows) and the V part of
// another (PV, V rows).  Each side keeps its own row layout and tensor maps;
// the V rows start on a 1024-byte boundary when either side uses the 128-byte
// swizzle (its pattern is taken from the address bits), else on 128 bytes.
template <class KT, class VT>
struct Mix {
    static_assert(KT::D == VT::D, "one head dimension");
    static constexpr int D = KT::D, MT = VT::MT;
    static constexpr int SCRATCH = KT::SCRATCH > VT::SCRATCH ? KT::SCRATCH : VT::SCRATCH;
    static constexpr bool kZeroInvalidV = VT::kZeroInvalidV;
    static constexpr bool kExtract = KT::kExtract || VT::kExtract;
    static constexpr uint32_t kMaxWarps =
        KT::kMaxWarps < VT::kMaxWarps ? KT::kMaxWarps : VT::kMaxWarps;
    static constexpr int kMergeBatch =
        KT::kMergeBatch < VT::kMergeBatch ? KT::kMergeBatch : VT::kMergeBatch;
    static constexpr bool kStagedMerge = false;  // one instance per mixed pair
    static constexpr bool kStream = false;       // stream plans take one K/V type
    static constexpr bool kTile32 = false;
    static constexpr uint32_t kSideK = KT::kSideK, kSideV = VT::kSideV;
    static constexpr uint32_t kTmaXK = KT::kTmaXK, kTmaXV = VT::kTmaXV;
    static constexpr uint32_t kRowK = KT::kRowK, kRowV = VT::kRowV;
    static constexpr uint32_t kAlign = (kTmaXK > 1 || kTmaXV > 1) ? 1024u : 128u;
    static constexpr uint32_t kVOff = (kSideK + kAlign - 1) / kAlign * kAlign;
    static constexpr uint32_t kSlot = (kVOff + kSideV + kAlign - 1) / kAlign * kAlign;
    static constexpr uint32_t kTypeKey = 100 + 32 * KT::kTypeKey + VT::kTypeKey;
    static constexpr int QBYTES = KT::QBYTES;
    using Frag = typename KT::Frag;
    using QRaw = typename KT::QRaw;
    struct Consts {
        typename KT::Consts k;
        typename VT::Consts v;
        __device__ __forceinline__ void init()
        {
            k.init();
            v.init();
        }
    };

    __device__ static void fetch_q(const DecodeParams &p, uint32_t s, uint32_t h0, uint32_t G,
                                   int gid, int tig, uint32_t w, uint32_t nw, QRaw &r)
    {
        KT::fetch_q(p, s, h0, G, gid, tig, w, nw, r);
    }
    __device__ static void store_q(const DecodeParams &p, const QRaw &r, uint32_t G, int gid,
                                   int tig, uint32_t w, uint32_t nw, uint32_t qsm)
    {
        KT::store_q(p, r, G, gid, tig, w, nw, qsm);
    }
    __device__ static void load_q(uint32_t qsm, int lane, Frag &f) { KT::load_q(qsm, lane, f); }
    __device__ static void load_q(const DecodeParams &p, const QRaw &r, uint32_t G, int gid,
                                  Frag &f)
    {
        KT::load_q(p, r, G, gid, f);
    }
    __device__ static void extract(uint32_t kh, uint32_t vh, uint32_t scr, int nvalid, int lane)
    {
        if constexpr (KT::kExtract)
            KT::extract_k(kh, scr, nvalid, lane);
        if constexpr (VT::kExtract)
            VT::extract_v(vh, scr, nvalid, lane);
    }
    __device__ static void zero_invalid_v(uint8_t *vh, int nvalid, int lane)
    {
        VT::zero_invalid_v(vh, nvalid, lane);
    }
    __device__ static void scores(const Consts &K, const Frag &f, uint32_t kh, uint32_t scr,
                                  int gid, int tig, float (&s)[4])
    {
        KT::scores(K.k, f, kh, scr, gid, tig, s);
    }
    __device__ static void pv(const Consts &K, float (&o)[MT][4], uint32_t vh, uint32_t scr,
                              uint32_t p0, uint32_t p1, int gid, int tig)
    {
        VT::pv(K.v, o, vh, scr, p0, p1, gid, tig);
    }
    __device__ static __forceinline__ int dim_of(int mt, int gid, int upper)
    {
        return VT::dim_of(mt, gid, upper);
    }
    static constexpr bool kDimPairs = VT::kDimPairs;
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

constexpr float kHeadroom = 4.0f;  // log2 units kept between the reference and the max

// Parked (m, l, O) of one warp: m of its 8 head columns, then l, then O as
// 8 rows of D floats (row stride D + 4, so that the fragment stores of the
// four tig lanes fall in different banks).
// After the warps' records: per query head, the combine's factors f_k of
// the head's warps, then 1 / l, M and l (kFac floats per head).
template <class T>
struct Park {
    static constexpr int kRow = T::D + 4;
    static constexpr int kWarp = 16 + 8 * kRow;
    static constexpr int kFac = T::kMaxWarps + 3;
    static constexpr int kFacBytes = 64 * kFac * 4;  // 64 query heads at most
};

template <class T>
__device__ __forceinline__ void combine_and_write(const DecodeParams &p, const float *park,
                                                  float *fac, uint32_t hkv, uint32_t wph,
                                                  uint32_t G, uint32_t seq, uint32_t part,
                                                  bool dir);

// One row of the in-launch merge by one warp from partials staged in shared
// memory: m partials of D halves at po (global; partial k at po + k * stride
// * D) and their (m, l) at pml (stride likewise).  Lane 0 copies the m rows
// into this warp's stage with bulk copies on the warp's mbarrier (parity
// `phase`, flipped here), the lanes fetch the (m, l) meanwhile, and then the
// weighted sum runs from shared memory.  The arithmetic is that of
// merge_rows_warp_v for m <= 32 (weight of partial k in lane k, warp sums,
// partials added in order), so the results are the same bits.  False if a
// copy did not land in time (status flagged; nothing written).
template <bool kPartial>
__device__ bool merge_row_staged(const DecodeParams &p, const __half *po, const float2 *pml,
                                 uint32_t m, uint32_t stride, uint32_t stage, uint64_t *bar,
                                 uint32_t &phase, float *out_f, __half *out_o, float2 *out_ml)
{
    const int lane = threadIdx.x & 31;
    const uint32_t D = p.d, rb = D * 2;
    if (lane == 0) {
        fence_proxy_async();  // this warp's earlier reads of the stage come first
        mbar_arrive_expect_tx(bar, m * rb);
        if (stride == 1)
            bulk_load(stage, po, m * rb, bar);
        else
            for (uint32_t k = 0; k < m; ++k)
                bulk_load(stage + k * rb, po + (uint64_t)k * stride * D, rb, bar);
    }
    float2 ml = make_float2(-INFINITY, 0.0f);
    if ((uint32_t)lane < m)
        ml = __ldcg(pml + (uint64_t)lane * stride);
    const float M = warp_max(ml.y > 0.0f ? ml.x : -INFINITY);
    const float w = ml.y > 0.0f ? ml.y * exp2f(ml.x - M) : 0.0f;
    const float s = warp_sum(w);
    bool done = mbar_try_wait(bar, phase);
    if (!done) {
        const uint64_t tw = global_ns();
        while (!(done = mbar_try_wait(bar, phase)) && global_ns() - tw < kWaitNs) {
        }
    }
    phase ^= 1;
    if (!__all_sync(0xffffffffu, done)) {
        if (lane == 0) {
            atomicOr(p.status, PA_STATUS_TIMEOUT);
            // let the copies land (bounded) before the stage is given up
            const uint64_t tw = global_ns();
            while (!mbar_try_wait(bar, phase ^ 1) && global_ns() - tw < kWaitNs) {
            }
        }
        __syncwarp();
        return false;
    }
    // lane l owns the dimension quads 4l.. and 128 + 4l.. (D = 256) or 4l.. (D = 128)
    float acc[8];
#pragma unroll
    for (int j = 0; j < 8; ++j)
        acc[j] = 0.0f;
    const uint32_t base = stage + 8 * lane;
    // every partial sits in the stage, so it is loaded whatever its weight
    // and added only for a positive weight: the sums of a skip, without a
    // branch between each weight and its loads
#pragma unroll 4
    for (uint32_t k = 0; k < m; ++k) {
        const float wk = __shfl_sync(0xffffffffu, w, k);
        const uint32_t a = base + k * rb;
        uint32_t h[4];
        asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(h[0]), "=r"(h[1]) : "r"(a) : "memory");
        if (D == 256)
            asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];"
                         : "=r"(h[2]), "=r"(h[3])
                         : "r"(a + 256)
                         : "memory");
        else
            h[2] = h[3] = 0u;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float2 f = __half22float2(bits_h2(h[j]));
            const float x = fmaf(wk, f.x, acc[2 * j]), y = fmaf(wk, f.y, acc[2 * j + 1]);
            acc[2 * j] = wk > 0.0f ? x : acc[2 * j];
            acc[2 * j + 1] = wk > 0.0f ? y : acc[2 * j + 1];
        }
    }
    __syncwarp();  // the stage is read before the next row lands
    const float inv = s > 0.0f ? 1.0f / s : 0.0f;
    for (int q = 0; q < (D == 256 ? 2 : 1); ++q) {
        if constexpr (kPartial) {
            *reinterpret_cast<uint2 *>(out_o + 128 * q + 4 * lane) =
                make_uint2(h2_bits(__floats2half2_rn(acc[4 * q] * inv, acc[4 * q + 1] * inv)),
                           h2_bits(__floats2half2_rn(acc[4 * q + 2] * inv, acc[4 * q + 3] * inv)));
        } else {
            *reinterpret_cast<float4 *>(out_f + 128 * q + 4 * lane) =
                make_float4(acc[4 * q] * inv, acc[4 * q + 1] * inv, acc[4 * q + 2] * inv,
                            acc[4 * q + 3] * inv);
        }
    }
    if (kPartial && lane == 0)
        *out_ml = make_float2(s > 0.0f ? M : -INFINITY, s);
    return true;
}

// The in-launch merge, out of line so that its registers do not add to the
// main loop's: fused_merge, with BATCH partials of each of two rows in flight
// per warp.
template <int BATCH>
__device__ __noinline__ void merge_tail(const DecodeParams &p, uint32_t seq, uint32_t part,
                                        uint32_t warp, uint32_t nwarps)
{
    fused_merge<BATCH>(p, seq, part, warp, nwarps);
}

// The in-launch merge of a plan of more than 32 partitions (two passes), out
// of line as above.  When the passes of this sequence merge at most
// min(32, cap) partials per row (cap: the rows a warp's share of the idle
// rings holds) and the partials are 16-byte aligned, each warp copies its
// rows into shared memory one at a time (merge_row_staged): one bulk copy per
// row instead of rounds of loads, with the same groups, order and arithmetic
// as fused_merge.  Otherwise fused_merge.
template <int BATCH>
__device__ __noinline__ void merge_tail_staged(const DecodeParams &p, uint32_t seq,
                                               uint32_t part, uint32_t warp, uint32_t nwarps,
                                               uint32_t stage, uint32_t cap, uint64_t *bar,
                                               uint32_t phase)
{
    const int32_t L = row_len(p.seq_lens, p.q_tokens, seq);
    uint32_t n = L > 0 ? ((uint32_t)L + p.part_tokens - 1) / p.part_tokens : 0;
    n = n < p.n_parts ? n : p.n_parts;
    const uint32_t gs = merge_group_size(n), ng = n > gs ? (n + gs - 1) / gs : 1;
    const uint32_t widest = gs > ng ? gs : ng;
    if (bar == nullptr || ng == 1 || widest > 32 || widest > cap ||
        (reinterpret_cast<uintptr_t>(p.part_o) & 15u) != 0) {
        fused_merge<BATCH>(p, seq, part, warp, nwarps);
        return;
    }
    fence_proxy_async();  // every thread's generic accesses to the rings come first
    const uint64_t pseq = seq - p.n_direct;  // index of the row's partials and counters
    int32_t *cnt = p.counters + pseq * merge_counters_per_seq(p.n_parts);
    const __half *po = static_cast<const __half *>(p.part_o);
    const float2 *pml = reinterpret_cast<const float2 *>(p.part_ml);
    const int lane = threadIdx.x & 31;
    bool ok = true;  // a copy that timed out ends this warp's merging, not its arrivals
    const uint32_t g = part / gs, p0 = g * gs, ng_g = min(gs, n - p0);
    if (!merge_arrive(cnt + 1 + g, ng_g))
        return;
    if (lane == 0)
        fence_proxy_async_global();
    __syncwarp();
    for (uint32_t h = warp; h < p.hq && ok; h += nwarps) {
        const uint64_t r = pseq * p.hq + h;
        // in place: the group's first slot, read before it is written
        __half *ro = const_cast<__half *>(po) + (r * p.n_parts + p0) * p.d;
        float2 *rm = const_cast<float2 *>(pml) + r * p.n_parts + p0;
        ok = merge_row_staged<true>(p, ro, rm, ng_g, 1, stage, bar, phase, nullptr, ro, rm);
    }
    if (!merge_arrive(cnt, ng))
        return;
    if (lane == 0)
        fence_proxy_async_global();
    __syncwarp();
    for (uint32_t h = warp; h < p.hq && ok; h += nwarps) {
        const uint64_t r = pseq * p.hq + h;
        ok = merge_row_staged<false>(p, po + r * p.n_parts * p.d, pml + r * p.n_parts, ng, gs,
                                     stage, bar, phase, p.out + ((uint64_t)seq * p.hq + h) * p.d,
                                     nullptr, nullptr);
    }
}

// The in-launch merge shared by the CTAs of a sequence, for one-pass plans
// whose grid is resident at once (every CTA of the launch holds an SM slot
// from the start, so the CTAs of a sequence finish within microseconds of one
// another).  Each CTA counts its partial (word 0 of the sequence's counters),
// waits until the count is complete, then merges the rows r with r % na ==
// its partition (na = the sequence's live partitions), each row with the same
// arithmetic, in the same order, as every other merge here.  The wait is
// bounded (wait_ns): a CTA whose wait runs out sets its bit in word 1 and
// merges nothing unless the count completed meanwhile; the CTA that completes
// the count merges the rows of every partition whose bit it sees.  The two
// sides order their write and read of words 0 and 1 with sequentially
// consistent fences, so at least one of them merges each such row (both may:
// they write the same bits).  Word 2 counts the CTAs that have read words 0
// and 1 (counted while the rows are merged); the last one resets the three
// words to 0.
// A row's partials are contiguous, so a merging warp copies them into its
// share of the idle rings with one bulk copy and sums them from shared
// memory (merge_row_staged): one round trip, and a short loop -- this code
// runs once per launch, when the instruction caches do not hold it.
template <class T>
__device__ __noinline__ void merge_coop(const DecodeParams &p, uint32_t seq, uint32_t part,
                                        int32_t L, uint32_t warp, uint32_t nwarps,
                                        uint32_t wait_ns, uint32_t region, uint32_t region_bytes)
{
    __shared__ uint32_t s_set;
    const int lane = threadIdx.x & 31;
    uint32_t n = L > 0 ? ((uint32_t)L + p.part_tokens - 1) / p.part_tokens : 0;
    n = n < p.n_parts ? n : p.n_parts;
    const uint32_t na = n > 0 ? n : 1u;  // arrivals: an empty sequence has one CTA
    const uint64_t pseq = seq - p.n_direct;
    int32_t *cnt = p.counters + pseq * merge_counters_per_seq(p.n_parts);
    __syncthreads();  // every thread's partial stores come before the count
    if (threadIdx.x == 0) {
        __threadfence();
        const uint32_t old = atomicAdd(reinterpret_cast<unsigned *>(cnt), 1u);
        uint32_t set = 0;
        if (old + 1 == na) {
            __threadfence();  // the count before the read of the stop bits
            set = (1u << part) | *reinterpret_cast<volatile uint32_t *>(cnt + 1);
        } else {
            const uint64_t t0 = global_ns();
            while (true) {
                if (ld_acquire_u32(cnt) >= na) {
                    set = 1u << part;
                    break;
                }
                if (global_ns() - t0 >= wait_ns) {
                    atomicOr(reinterpret_cast<unsigned *>(cnt + 1), 1u << part);
                    __threadfence();  // the stop bit before the read of the count
                    if (*reinterpret_cast<volatile uint32_t *>(cnt) >= na)
                        set = 1u << part;
                    break;
                }
                __nanosleep(128);
            }
        }
        __threadfence();  // the counted CTAs' partials before this CTA's reads
        s_set = set;
    }
    __syncthreads();
    const uint32_t set = s_set;
    // this CTA's reads of words 0 and 1 are done (thread 0, before the
    // barrier): the first thread of the last warp counts it on word 2 while
    // the rows are merged, and the CTA that completes that count resets the
    // three words for the next launch (the partials need no such order: a
    // later launch writes them only after this grid has completed)
    if (threadIdx.x == blockDim.x - 32) {
        if (atom_add_acq_rel(cnt + 2, 1u) + 1 == na) {
            cnt[0] = 0;
            cnt[1] = 0;
            cnt[2] = 0;
        }
    }
    if (set) {
        const __half *po = static_cast<const __half *>(p.part_o);
        const float2 *pml = reinterpret_cast<const float2 *>(p.part_ml);
        // k consecutive warp shares of the rings hold one row's n partials
        // and the worker's mbarrier (its last 16 bytes)
        const uint32_t share = (region_bytes / nwarps) & ~15u;
        const uint32_t need = n * p.d * 2 + 16;
        const uint32_t k = share ? (need + share - 1) / share : 0;
        const bool staged = n > 0 && k >= 1 && k <= nwarps &&
                            (reinterpret_cast<uintptr_t>(p.part_o) & 15u) == 0;
        const uint32_t workers = staged ? nwarps / k : nwarps;
        const bool worker = staged ? warp % k == 0 : true;
        const uint32_t wid = staged ? warp / k : warp;
        uint32_t stage = 0, phase = 0;
        uint64_t *bar = nullptr;
        if (staged && worker) {
            stage = region + warp * share;
            bar = reinterpret_cast<uint64_t *>(__cvta_shared_to_generic(stage + k * share - 16));
            if (lane == 0) {
                mbar_init(bar, 1);
                asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
            }
            __syncwarp();
        }
        // rows r = j, j + na, ... of each partition j in the set; the u-th
        // goes to worker u % workers
        uint32_t u = 0;
        for (uint32_t bits = set; bits; bits &= bits - 1) {
            for (uint32_t r = __ffs(bits) - 1; r < p.hq; r += na, ++u) {
                if (!(worker && wid < workers && u % workers == wid))
                    continue;
                const uint64_t row = pseq * p.hq + r;
                const __half *rpo = po + row * p.n_parts * p.d;
                const float2 *rml = pml + row * p.n_parts;
                float *rout = p.out + ((uint64_t)seq * p.hq + r) * p.d;
                if (staged)
                    merge_row_staged<false>(p, rpo, rml, n, 1, stage, bar, phase, rout, nullptr,
                                            nullptr);
                else if (p.d == 256)
                    merge_rows_warp_v<8, 1, false, 8>(&rpo, &rml, n, 1, p.d, 1, &rout, nullptr,
                                                      nullptr);
                else
                    merge_rows_warp_v<4, 1, false, 8>(&rpo, &rml, n, 1, p.d, 1, &rout, nullptr,
                                                      nullptr);
            }
        }
    }
}

// The end of a range: each warp parks (m, l, O) of its query heads in the
// idle rings, head-major (the lanes' sums l first added across the warp),
// then all warps of the CTA combine them into the partial or the output.
// Called by every thread after a barrier that follows the last ring read.
template <class T>
__device__ __forceinline__ void park_and_combine(const DecodeParams &p, uint8_t *smem,
                                                 const float (&o)[T::MT][4], float mref0,
                                                 float mref1, float l0, float l1, uint32_t nwarps,
                                                 uint32_t hkv, uint32_t G, uint32_t seq,
                                                 uint32_t part, bool dir)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int gid = lane >> 2, tig = lane & 3;
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
        l0 += __shfl_xor_sync(0xffffffffu, l0, off);
        l1 += __shfl_xor_sync(0xffffffffu, l1, off);
    }
    float *park = reinterpret_cast<float *>(smem);
    float *mine = park + warp * Park<T>::kWarp;
    if (gid == 0) {
        mine[2 * tig] = mref0;
        mine[2 * tig + 1] = mref1;
        mine[8 + 2 * tig] = l0;
        mine[8 + 2 * tig + 1] = l1;
    }
    // the columns of query heads past the group (2 tig + e % 2 >= G) are not read
    if (2u * tig < G) {
#pragma unroll
        for (int mt = 0; mt < T::MT; ++mt) {
            if constexpr (T::kDimPairs) {
                // the two rows of a column are adjacent dimensions: one 8-byte store
#pragma unroll
                for (int c = 0; c < 2; ++c)
                    if (c == 0 || 2u * tig + 1 < G)
                        *reinterpret_cast<float2 *>(
                            mine + 16 + (2 * tig + c) * Park<T>::kRow + T::dim_of(mt, gid, 0)) =
                            make_float2(o[mt][c], o[mt][c + 2]);
            } else {
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    if ((e & 1) == 0 || 2u * tig + 1 < G)
                        mine[16 + (2 * tig + (e & 1)) * Park<T>::kRow +
                             T::dim_of(mt, gid, e >> 1)] = o[mt][e];
            }
        }
    }
    __syncthreads();
    combine_and_write<T>(p, park, park + nwarps * Park<T>::kWarp, hkv, nwarps / hkv, G, seq, part,
                         dir);
}

// The decode of one token range [t0, t1) of one query row (`seq`), by the whole
// CTA: the table walk, the per-warp TMA rings, the tile loop, and the combine
// of the warps' results into the range's partial (index `part`), or into the
// output row when `dir`.  The rings continue from slot s / parity phase (the
// next use of each warp's ring: use u of a ring takes slot u % NSW with
// parity (u / NSW) % 2) and are left drained, at the slot and parity after
// the range's last tile.  any_abort: a bounded wait of some warp ran out
// (status flagged; the rings may then hold copies of this range), reported
// only by the kReportAbort instances.  kTrigger: the CTA allows the next
// grid on the stream to be scheduled once its tile loop ends (a caller that
// reads inputs after the range, as the stream kernel's next segment does,
// passes false and triggers after its last read).
template <class T, bool kReportAbort, bool kTrigger = true>
__device__ __forceinline__ void range_body(const FastArgs &a, uint8_t *smem, uint32_t seq,
                                           uint32_t part, int32_t Lrow, uint32_t t0in,
                                           bool dir, uint32_t t1in, uint32_t &s,
                                           uint32_t &phase, uint32_t &n_my_out,
                                           bool &any_abort)
{
    const DecodeParams &p = a.p;
    const uint32_t NSW = a.n_slots, SLOT = a.slot_bytes, nwarps = blockDim.x >> 5;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t hkv = p.hkv, G = p.hq / p.hkv, wph = nwarps / hkv;
    uint8_t *ring = smem + (size_t)warp * NSW * SLOT;
    const uint32_t ring_u = smem_u32(ring);
    // after the rings: mbarriers [nwarps][bar_slots], flag words likewise,
    // then the scratch; this body uses the first nwarps * NSW of each
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + a.region_bytes);
    uint64_t *full = bars + warp * NSW;
    int *ok_all = reinterpret_cast<int *>(bars + nwarps * a.bar_slots);
    int *slot_ok = ok_all + warp * NSW;
    const uint32_t scr_base = (smem_u32(ok_all + nwarps * a.bar_slots) + 15u) & ~15u;
    const uint32_t scr_u = scr_base + warp * T::SCRATCH;
    const uint32_t qsm_base = scr_base + nwarps * T::SCRATCH;  // per K/V head: T::QBYTES
    const uint32_t s0 = s, u0 = phase * NSW + s;  // this warp's ring use at the range start
    const int32_t L = Lrow > 0 ? Lrow : 0;
    const uint32_t t0 = t0in;
    const uint32_t t1 = min((uint32_t)L, t1in);
    const uint32_t n_tiles = (t1 - t0 + kTile - 1) / kTile;
    const int gid = lane >> 2, tig = lane & 3;
    const uint32_t g = warp % hkv, sub = warp / hkv;
    const uint32_t n_my = n_tiles > sub ? (n_tiles - sub + wph - 1) / wph : 0;
    const int32_t *bt = p.block_table + (uint64_t)table_row(p.q_tokens, seq) * p.table_stride;
    const CUtensorMap *tmk = &a.tm[0][g], *tmv = &a.tm[1][g];
    // V rows of a slot start here: the slot's middle for one type on both
    // sides, the padded K size for a mixed pair
    constexpr bool kSym = T::kSideK == T::kSideV && T::kTmaXK == T::kTmaXV;
    const uint32_t voff = kSym ? SLOT / 2 : T::kVOff;
    const uint32_t bshift = p.block_size == 32 ? 5 : 4, bmask = p.block_size - 1;

    // block ids of my tiles k0 .. k0+31, one per lane
    auto fetch_ids = [&](uint32_t k0) -> int32_t {
        const uint32_t k = k0 + lane;
        return k < n_my ? bt[(t0 + kTile * (sub + k * wph)) >> bshift] : 0;
    };
    // lane 0: start the copy of my tile k (block id blk) into slot s
    auto issue = [&](uint32_t k, uint32_t s, int32_t blk) {
        const uint32_t tok = t0 + kTile * (sub + k * wph);
        const bool ok = block_in_pool(blk, p.n_pool_blocks);
        slot_ok[s] = ok;
        if (ok) {
            uint8_t *dst = ring + (size_t)s * SLOT;
            const int y = (blk << bshift) + (int)(tok & bmask);
            fence_proxy_async();  // earlier generic reads of this slot come first
            // K/V rows are read once: evict-first in the L2
            const uint64_t pol = l2_evict_first_policy();
            if constexpr (kSym) {
                mbar_arrive_expect_tx(&full[s], SLOT);
#pragma unroll
                for (uint32_t c = 0; c < T::kTmaXK; ++c) {
                    tma_load_2d_hint(dst + c * (voff / T::kTmaXK), tmk, 64 * c, y, &full[s], pol);
                    tma_load_2d_hint(dst + voff + c * (voff / T::kTmaXK), tmv, 64 * c, y,
                                     &full[s], pol);
                }
            } else {
                mbar_arrive_expect_tx(&full[s], T::kSideK + T::kSideV);
#pragma unroll
                for (uint32_t c = 0; c < T::kTmaXK; ++c)
                    tma_load_2d_hint(dst + c * (T::kSideK / T::kTmaXK), tmk, 64 * c, y, &full[s],
                                     pol);
#pragma unroll
                for (uint32_t c = 0; c < T::kTmaXV; ++c)
                    tma_load_2d_hint(dst + voff + c * (T::kSideV / T::kTmaXV), tmv, 64 * c, y,
                                     &full[s], pol);
            }
        } else {
            atomicOr(p.status, PA_STATUS_CORRUPT_TABLE);
            mbar_arrive(&full[s]);
        }
    };

    int32_t ids = fetch_ids(0), ids_next = fetch_ids(32);
    // quantised K: the wph warps of a head split its query blocks
    typename T::QRaw qraw;
    T::fetch_q(p, seq, g * G, G, gid, tig, sub, wph, qraw);
    const uint32_t pro = n_my < NSW ? n_my : NSW;
    for (uint32_t k = 0; k < pro; ++k) {
        const int32_t b = __shfl_sync(0xffffffffu, ids, k);
        uint32_t sk = s0 + k;
        sk = sk >= NSW ? sk - NSW : sk;
        if (lane == 0)
            issue(k, sk, b);
    }
    __syncwarp();

    typename T::Consts K;
    K.init();
    typename T::Frag f;
    if constexpr (T::QBYTES > 0) {
        T::store_q(p, qraw, G, gid, tig, sub, wph, qsm_base + g * T::QBYTES);
        __syncthreads();
        T::load_q(qsm_base + g * T::QBYTES, lane, f);
    } else {
        T::load_q(p, qraw, G, gid, f);
    }
    float o[T::MT][4];
#pragma unroll
    for (int mt = 0; mt < T::MT; ++mt)
        o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.0f;
    // softmax state of this thread's heads 2tig and 2tig+1: reference max
    // (>= every score seen) and the partial sum over its tokens
    float mref0 = -INFINITY, mref1 = -INFINITY, l0 = 0.0f, l1 = 0.0f;
    bool aborted = false;
    uint32_t issued = pro;

    for (uint32_t k = 0; k < n_my; ++k) {
        // every lane waits (bounded) and so acquires the slot's TMA writes itself
        bool done = mbar_try_wait(&full[s], phase);
        if (!done) {
            const uint64_t tw = global_ns();
            while (!(done = mbar_try_wait(&full[s], phase)) && global_ns() - tw < kWaitNs) {
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
        const uint32_t kh = ring_u + s * SLOT, vh = kh + voff;
        if constexpr (T::kZeroInvalidV) {
            if (nvalid < kTile) {
                T::zero_invalid_v(ring + (size_t)s * SLOT + voff, nvalid, lane);
                __syncwarp();
            }
        }
        if constexpr (T::kExtract) {
            T::extract(kh, vh, scr_u, nvalid, lane);
            __syncwarp();
        }
        float sc[4];
        T::scores(K, f, kh, scr_u, gid, tig, sc);
        // online softmax over the tile (log2 domain); the reference max moves,
        // and the accumulators are rescaled, only when a score passes it
        if (gid >= nvalid)
            sc[0] = sc[1] = -INFINITY;
        if (gid + 8 >= nvalid)
            sc[2] = sc[3] = -INFINITY;
        // a score above its reference is rare: each lane checks its own four,
        // and only then does the warp form the tile maxima of its heads
        const bool over = fmaxf(sc[0], sc[2]) > mref0 || fmaxf(sc[1], sc[3]) > mref1;
        if (__builtin_expect(__any_sync(0xffffffffu, over), 0)) {
            float t0m = fmaxf(sc[0], sc[2]), t1m = fmaxf(sc[1], sc[3]);
#pragma unroll
            for (int off = 4; off < 32; off <<= 1) {
                t0m = fmaxf(t0m, __shfl_xor_sync(0xffffffffu, t0m, off));
                t1m = fmaxf(t1m, __shfl_xor_sync(0xffffffffu, t1m, off));
            }
            const float n0 = t0m > mref0 ? t0m + kHeadroom : mref0;
            const float n1 = t1m > mref1 ? t1m + kHeadroom : mref1;
            const float a0 = mref0 == -INFINITY ? 0.0f : exp2f(mref0 - n0);
            const float a1 = mref1 == -INFINITY ? 0.0f : exp2f(mref1 - n1);
#pragma unroll
            for (int mt = 0; mt < T::MT; ++mt) {
                o[mt][0] *= a0;
                o[mt][1] *= a1;
                o[mt][2] *= a0;
                o[mt][3] *= a1;
            }
            l0 *= a0;
            l1 *= a1;
            mref0 = n0;
            mref1 = n1;
        }
        const float ms0 = mref0 == -INFINITY ? 0.0f : mref0;
        const float ms1 = mref1 == -INFINITY ? 0.0f : mref1;
        const float q00 = ex2_ftz(sc[0] - ms0), q01 = ex2_ftz(sc[1] - ms1);
        const float q10 = ex2_ftz(sc[2] - ms0), q11 = ex2_ftz(sc[3] - ms1);
        l0 += q00 + q10;
        l1 += q01 + q11;
        // P[token][head] as two 8x8 blocks (tokens 0-7, 8-15) -> PV B operand
        const uint32_t p0 = movmatrix_t(h2_bits(__floats2half2_rn(q00, q01)));
        const uint32_t p1 = movmatrix_t(h2_bits(__floats2half2_rn(q10, q11)));
        T::pv(K, o, vh, scr_u, p0, p1, gid, tig);
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
                issue(kn, s, b);
            issued = kn + 1;
        }
        if (++s == NSW) {
            s = 0;
            phase ^= 1;
        }
    }
    // the next grid on this stream may be scheduled once every CTA is here
    // (its CTAs take the SMs that this grid's CTAs leave, and wait for this
    // grid's completion before they read anything); no input is read after
    if constexpr (kTrigger)
        launch_dependents();
    if (aborted && lane == 0) {
        // let my copies still in flight land (bounded) before the CTA moves on
        for (uint32_t k = issued > NSW ? issued - NSW : 0; k < issued; ++k) {
            const uint32_t u = u0 + k;
            const uint64_t tw = global_ns();
            while (!mbar_try_wait(&full[u % NSW], (u / NSW) & 1) && global_ns() - tw < kWaitNs) {
            }
        }
    }
    // every ring is drained: the rings are free
    if constexpr (kReportAbort)
        any_abort = __syncthreads_or(aborted);
    else
        __syncthreads();
    park_and_combine<T>(p, smem, o, mref0, mref1, l0, l1, nwarps, hkv, G, seq, part, dir);
    n_my_out = n_my;
}

// range_body for one-token rows of a type with kTile32 (Q4_0) in 32-token
// tiles, which halves the per-tile work that does not grow with the tokens:
// the wait, the copy issue, the softmax vote and the loop, and each query
// record load serves 32 tokens.  The warps of K/V head g share a ring of
// S = n_slots32 slots, each the K rows then the V rows of 32 tokens (one
// 16-row box per side and 16-token half); warp sub of the head takes tiles
// sub, sub + wph, ... of [t0, t1); tile t sits in slot t % S with parity
// (t / S) % 2, and the warp that has read tile t refills the slot with tile
// t + S.  Each slot has wph mbarriers used in turn: tile t completes barrier
// (t % S, (t / S) % wph), the (t / (S wph))-th time, so a barrier's tiles
// are t, t + wph S, ..., all of one warp.  Its waits therefore always come
// after its previous phase completed (a tile the same warp read), and the
// issuer of tile t, who read tile t - S, arrives on it after that phase too
// (t - wph S came through the ring before t - S did), so a parity names
// one phase.  (With one barrier per slot, the warp waiting for tile t could
// meet the barrier still in the phase of tile t - S, another warp's, and a
// parity would match that.)  A slot's flag word holds which halves were
// copied (bits 0, 1: a half with tokens whose block is in the pool) and,
// above them, t + 1 for the tile last issued into the slot (the drain after
// a timeout uses it).  The arithmetic per 16-token half is that of
// range_body; the online softmax moves its reference once per 32 tokens.
template <class T, bool kReportAbort>
__device__ __forceinline__ void range_body32(const FastArgs &a, uint8_t *smem, uint32_t seq,
                                             uint32_t part, int32_t Lrow, uint32_t t0in,
                                             bool dir, uint32_t t1in, bool &any_abort)
{
    const DecodeParams &p = a.p;
    const uint32_t BS = a.bar_slots, S = a.n_slots32, nwarps = blockDim.x >> 5;
    constexpr uint32_t HALF = T::kSideK;  // 16 rows of one side
    constexpr uint32_t SLOT = 4 * HALF;   // K rows 0..31, then V rows 0..31
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t hkv = p.hkv, G = p.hq / p.hkv, wph = nwarps / hkv;
    const int gid = lane >> 2, tig = lane & 3;
    const uint32_t g = warp % hkv, sub = warp / hkv;
    uint8_t *ring = smem + (size_t)g * S * SLOT;
    const uint32_t ring_u = smem_u32(ring);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + a.region_bytes);
    uint64_t *hbar = bars + g * wph * S;  // head g's barriers: slot s, turn e at s + S e
    int *ok_all = reinterpret_cast<int *>(bars + nwarps * BS);
    int *slot_ok = ok_all + g * S;
    const uint32_t scr_base = (smem_u32(ok_all + nwarps * BS) + 15u) & ~15u;
    const uint32_t scr_u = scr_base + warp * T::SCRATCH2;
    const uint32_t qsm_base = scr_base + nwarps * T::SCRATCH2;  // per K/V head: T::QBYTES
    const int32_t L = Lrow > 0 ? Lrow : 0;
    const uint32_t t0 = t0in, t1 = min((uint32_t)L, t1in);
    const uint32_t n_tiles = t1 > t0 ? (t1 - t0 + 31) / 32 : 0u;
    const uint32_t n_my = n_tiles > sub ? (n_tiles - sub + wph - 1) / wph : 0u;
    const int32_t *bt = p.block_table + (uint64_t)table_row(p.q_tokens, seq) * p.table_stride;
    const CUtensorMap *tmk = &a.tm[0][g], *tmv = &a.tm[1][g];
    const uint32_t bshift = p.block_size == 32 ? 5 : 4, bmask = p.block_size - 1;

    // the block ids of tile t's halves (0 past the range)
    auto ids_of = [&](uint32_t t, int32_t &b0, int32_t &b1) {
        const uint32_t tok = t0 + 32 * t;
        b0 = t < n_tiles && tok < t1 ? bt[tok >> bshift] : 0;
        b1 = t < n_tiles && tok + 16 < t1 ? bt[(tok + 16) >> bshift] : 0;
    };
    // lane 0: the copies of tile t (block ids b0, b1 of its halves) into slot
    // s = t % S at shared address dst, completing barrier fb.  A refill
    // follows this warp's reads of the slot without a proxy fence: each of
    // those loads has returned its value (consumed by the tensor-core
    // operations before the warp barrier that precedes the issue), so a copy
    // issued after them cannot change what they read -- the ordering the TMA
    // pipelines of CUTLASS rely on when a consumer releases a stage with a
    // bare mbarrier arrive.
    auto issue = [&](uint32_t t, uint32_t s, uint8_t *dst, uint64_t *fb, int32_t b0, int32_t b1) {
        const uint32_t tok = t0 + 32 * t;
        uint32_t bits = 0;
        if (tok < t1) {
            if (block_in_pool(b0, p.n_pool_blocks))
                bits |= 1u;
            else
                atomicOr(p.status, PA_STATUS_CORRUPT_TABLE);
        }
        if (tok + 16 < t1) {
            if (block_in_pool(b1, p.n_pool_blocks))
                bits |= 2u;
            else
                atomicOr(p.status, PA_STATUS_CORRUPT_TABLE);
        }
        slot_ok[s] = (int)((t + 1u) << 2 | bits);
        // K/V rows are read once: evict-first in the L2
        const uint64_t pol = l2_evict_first_policy();
        mbar_arrive_expect_tx(fb, (bits & 1u ? 2 * HALF : 0u) + (bits & 2u ? 2 * HALF : 0u));
        if (bits & 1u) {
            const int y = (b0 << bshift) + (int)(tok & bmask);
            tma_load_2d_hint(dst, tmk, 0, y, fb, pol);
            tma_load_2d_hint(dst + 2 * HALF, tmv, 0, y, fb, pol);
        }
        if (bits & 2u) {
            const int y = (b1 << bshift) + (int)((tok + 16) & bmask);
            tma_load_2d_hint(dst + HALF, tmk, 0, y, fb, pol);
            tma_load_2d_hint(dst + 3 * HALF, tmv, 0, y, fb, pol);
        }
    };
    // the block ids of my refills r0 .. r0+31, one refill per lane: refill r
    // follows my tile r and brings tile sub + S + r * wph
    auto fetch_refills = [&](uint32_t r0, int32_t &b0, int32_t &b1) {
        const uint32_t r = r0 + (uint32_t)lane;
        ids_of(r < n_my ? sub + S + r * wph : n_tiles, b0, b1);
    };

    int32_t rb0 = 0, rb1 = 0, nb0 = 0, nb1 = 0;
    fetch_refills(0, rb0, rb1);
    fetch_refills(32, nb0, nb1);
    // the query of the row: one (head, block, half) item per thread
    typename T::QItems qitems;
    T::fetch_q_cta(p, seq, threadIdx.x, qitems);
    // my tiles among the ring's first S: lane k loads the block ids of the
    // k-th, so that one round trip serves them all
    {
        const uint32_t tk = sub + (uint32_t)lane * wph;
        int32_t kb0 = 0, kb1 = 0;
        if (tk < S)
            ids_of(tk, kb0, kb1);
        uint32_t k = 0;
        for (uint32_t t = sub; t < S && t < n_tiles; t += wph, ++k) {
            const int32_t b0 = __shfl_sync(0xffffffffu, kb0, k);
            const int32_t b1 = __shfl_sync(0xffffffffu, kb1, k);
            if (lane == 0)
                issue(t, t, ring + (size_t)t * SLOT, hbar + t, b0, b1);
        }
    }
    __syncwarp();

    typename T::Consts K;
    K.init();
    typename T::Frag f;
    T::store_q_cta(p, seq, qitems, qsm_base);
    __syncthreads();
    T::load_q(qsm_base + g * T::QBYTES, lane, f);
    float o[T::MT][4];
#pragma unroll
    for (int mt = 0; mt < T::MT; ++mt)
        o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.0f;
    float mref0 = -INFINITY, mref1 = -INFINITY, l0 = 0.0f, l1 = 0.0f;
    bool aborted = false;

    // my tile t = sub + i * wph: slot s (shared address kh), barrier turn e,
    // parity par (wph < S: one wrap at most per step), first token t0 + 32 t
    uint32_t s = sub, e = 0, par = 0, t = sub, kh = ring_u + sub * SLOT, tok = t0 + 32 * sub;
    for (uint32_t i = 0; i < n_my; ++i, t += wph, tok += 32 * wph) {
        uint64_t *fb = hbar + s + S * e;
        // every lane waits (bounded) and so acquires the slot's TMA writes itself
        bool done = mbar_try_wait(fb, par);
        if (!done) {
            const uint64_t tw = global_ns();
            while (!(done = mbar_try_wait(fb, par)) && global_ns() - tw < kWaitNs) {
            }
        }
        if (!__all_sync(0xffffffffu, done)) {
            if (lane == 0)
                atomicOr(p.status, PA_STATUS_TIMEOUT);
            aborted = true;
            break;
        }
        const uint32_t okb = (uint32_t)slot_ok[s] & 3u;
        const uint32_t nv = t1 - tok;  // >= 1 tokens from the tile's start
        const int nva = okb & 1u ? (int)min(16u, nv) : 0;
        const int nvb = okb & 2u && nv > 16 ? (int)min(16u, nv - 16) : 0;
        const uint32_t vh = kh + 2 * HALF;
        T::extract(kh, vh, scr_u, nva, lane);
        T::extract(kh + HALF, vh + HALF, scr_u + T::SCRATCH, nvb, lane);
        __syncwarp();
        float sx[4], sz[4];
        T::scores2(K, f, kh, scr_u, gid, tig, sx, sz);
        if (gid >= nva)
            sx[0] = sx[1] = -INFINITY;
        if (gid + 8 >= nva)
            sx[2] = sx[3] = -INFINITY;
        if (gid >= nvb)
            sz[0] = sz[1] = -INFINITY;
        if (gid + 8 >= nvb)
            sz[2] = sz[3] = -INFINITY;
        const float m0 = fmaxf(fmaxf(sx[0], sx[2]), fmaxf(sz[0], sz[2]));
        const float m1 = fmaxf(fmaxf(sx[1], sx[3]), fmaxf(sz[1], sz[3]));
        if (__builtin_expect(__any_sync(0xffffffffu, m0 > mref0 || m1 > mref1), 0)) {
            float t0m = m0, t1m = m1;
#pragma unroll
            for (int off = 4; off < 32; off <<= 1) {
                t0m = fmaxf(t0m, __shfl_xor_sync(0xffffffffu, t0m, off));
                t1m = fmaxf(t1m, __shfl_xor_sync(0xffffffffu, t1m, off));
            }
            const float n0 = t0m > mref0 ? t0m + kHeadroom : mref0;
            const float n1 = t1m > mref1 ? t1m + kHeadroom : mref1;
            const float a0 = mref0 == -INFINITY ? 0.0f : exp2f(mref0 - n0);
            const float a1 = mref1 == -INFINITY ? 0.0f : exp2f(mref1 - n1);
#pragma unroll
            for (int mt = 0; mt < T::MT; ++mt) {
                o[mt][0] *= a0;
                o[mt][1] *= a1;
                o[mt][2] *= a0;
                o[mt][3] *= a1;
            }
            l0 *= a0;
            l1 *= a1;
            mref0 = n0;
            mref1 = n1;
        }
        const float ms0 = mref0 == -INFINITY ? 0.0f : mref0;
        const float ms1 = mref1 == -INFINITY ? 0.0f : mref1;
        const float x00 = ex2_ftz(sx[0] - ms0), x01 = ex2_ftz(sx[1] - ms1);
        const float x10 = ex2_ftz(sx[2] - ms0), x11 = ex2_ftz(sx[3] - ms1);
        const float z00 = ex2_ftz(sz[0] - ms0), z01 = ex2_ftz(sz[1] - ms1);
        const float z10 = ex2_ftz(sz[2] - ms0), z11 = ex2_ftz(sz[3] - ms1);
        l0 += (x00 + x10) + (z00 + z10);
        l1 += (x01 + x11) + (z01 + z11);
        // P[token][head] as 8x8 blocks (tokens 0-7, 8-15 of each half) -> PV B operands
        T::pv(K, o, vh, scr_u, movmatrix_t(h2_bits(__floats2half2_rn(x00, x01))),
              movmatrix_t(h2_bits(__floats2half2_rn(x10, x11))), gid, tig);
        T::pv(K, o, vh + HALF, scr_u + T::SCRATCH,
              movmatrix_t(h2_bits(__floats2half2_rn(z00, z01))),
              movmatrix_t(h2_bits(__floats2half2_rn(z10, z11))), gid, tig);
        __syncwarp();  // all reads of this slot are done
        // refill the slot with tile t + S (my refill i)
        if (t + S < n_tiles) {
            if ((i & 31u) == 0 && i > 0) {
                rb0 = nb0;
                rb1 = nb1;
                fetch_refills(i + 32, nb0, nb1);
            }
            const int32_t b0 = __shfl_sync(0xffffffffu, rb0, i & 31u);
            const int32_t b1 = __shfl_sync(0xffffffffu, rb1, i & 31u);
            // tile t + S: the same slot, the next barrier turn
            uint64_t *nb = hbar + s + S * (e + 1 == wph ? 0u : e + 1);
            if (lane == 0)
                issue(t + S, s, ring + (kh - ring_u), nb, b0, b1);
        }
        s += wph;
        kh += wph * SLOT;
        if (s >= S) {
            s -= S;
            kh -= S * SLOT;
            if (++e == wph) {
                e = 0;
                par ^= 1u;
            }
        }
    }
    // the next grid on this stream may be scheduled once every CTA is here
    // (no input is read after)
    launch_dependents();
    const bool cta_abort = __syncthreads_or(aborted);
    if constexpr (kReportAbort)
        any_abort = cta_abort;
    if (cta_abort) {
        // copies still in flight land (bounded) before the rings are reused:
        // the tile last issued into each slot of each ring (tl = word / 4 - 1)
        if (sub == 0 && lane == 0) {
            for (uint32_t k = 0; k < S; ++k) {
                const uint32_t n = (uint32_t)slot_ok[k] >> 2;
                if (n == 0)
                    continue;
                const uint32_t tl = n - 1;
                uint64_t *lb = hbar + k + S * ((tl / S) % wph);
                const uint64_t tw = global_ns();
                while (!mbar_try_wait(lb, (tl / (S * wph)) & 1u) && global_ns() - tw < kWaitNs) {
                }
            }
        }
        __syncthreads();
    }
    park_and_combine<T>(p, smem, o, mref0, mref1, l0, l1, nwarps, hkv, G, seq, part, dir);
}

// kStaged: the instance for plans of more than 32 partitions, whose merges
// run in two passes (merge_tail_staged); the other plans take the instance
// without it, whose code stays as it was tuned.
template <class T, bool kStaged = false>
__global__ void __launch_bounds__(T::kMaxWarps * 32, 1)
    fast_decode_kernel(const __grid_constant__ FastArgs a)
{
    const DecodeParams &p = a.p;
    extern __shared__ __align__(16) uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t NSW = a.n_slots, nwarps = blockDim.x >> 5;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + a.region_bytes) + warp * NSW;

    // a kTile32 type takes 32-token tiles (range_body32) in both instances,
    // so that a step gives the same bits through either
    constexpr bool k32 = T::kTile32;
    if (lane == 0) {
        // every mbarrier and flag word after the rings (bar_slots per warp)
        uint64_t *bars = reinterpret_cast<uint64_t *>(smem + a.region_bytes);
        int *flags = reinterpret_cast<int *>(bars + nwarps * a.bar_slots);
        for (uint32_t s = 0; s < a.bar_slots; ++s) {
            mbar_init(&bars[warp * a.bar_slots + s], 1);
            flags[warp * a.bar_slots + s] = 0;  // no tile issued
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    // everything below reads inputs that an earlier grid may have written
    grid_dependency_wait();

    uint32_t seq, part;
    if (!p.direct && blockIdx.x == gridDim.x - 1 && warp == 0)
        check_grid_vs_plan(p.seq_lens, p.q_tokens, p.n_seqs, p.part_tokens, p.n_parts,
                           p.n_direct, p.status);
    if (p.direct) {
        seq = blockIdx.x;
        part = 0;
    } else if (!cta_work(p.seq_lens, p.q_tokens, p.n_seqs, p.part_tokens, p.n_parts,
                         p.n_direct, blockIdx.x, &seq, &part)) {
        return;  // past the last live partition: nothing was issued
    } else if (seq >= p.n_direct && part == 0 && tid == 0) {
        check_len_vs_plan(row_len(p.seq_lens, p.q_tokens, seq), p.n_parts, p.part_tokens,
                          p.status);
    }
    // a direct CTA: the whole row, output written here (every CTA of a direct
    // plan, and the leading rows of a wave-filling plan)
    const bool dir = p.direct || seq < p.n_direct;
    const int32_t Lrow = row_len(p.seq_lens, p.q_tokens, seq);
    const uint32_t t0 = dir ? 0u : part * p.part_tokens;
    const uint32_t t1 = dir ? (uint32_t)max(Lrow, 0) : t0 + p.part_tokens;
    uint32_t s = 0, phase = 0, n_my = 0;  // fresh rings
    bool any_abort = false;
    if constexpr (k32)
        range_body32<T, kStaged>(a, smem, seq, part, Lrow, t0, dir, t1, any_abort);
    else
        range_body<T, kStaged>(a, smem, seq, part, Lrow, t0, dir, t1, s, phase, n_my, any_abort);
    if (p.counters && !dir) {
        if (a.coop) {
            merge_coop<T>(p, seq, part, Lrow, warp, nwarps, a.coop_wait_ns, smem_u32(smem),
                          a.region_bytes);
        } else if constexpr (kStaged) {
            // each warp stages its merge rows in its share of the idle rings
            // and waits on its slot-0 mbarrier, whose next parity follows the
            // loop's uses of slot 0 (all landed unless the loop aborted)
            const uint32_t share = (a.region_bytes / nwarps) & ~15u;
            uint32_t phase0 = ((n_my + NSW - 1) / NSW) & 1u;
            if constexpr (k32) {
                // the 32-token rings used these barriers head by head: the
                // warp's slot-0 barrier starts afresh for the merge (no copy
                // is pending on it: the rings were drained before the combine)
                if (lane == 0 && !any_abort) {
                    asm volatile("mbarrier.inval.shared::cta.b64 [%0];" ::"r"(smem_u32(full))
                                 : "memory");
                    mbar_init(full, 1);
                    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
                }
                __syncwarp();
                phase0 = 0;
            }
            merge_tail_staged<T::kMergeBatch>(p, seq, part, warp, nwarps,
                                              smem_u32(smem) + warp * share, share / (p.d * 2),
                                              any_abort ? nullptr : full, phase0);
        } else {
            merge_tail<T::kMergeBatch>(p, seq, part, warp, nwarps);
        }
    }
}

// range_body out of line, for the stream kernel: the segment walk's own
// values are saved around the call, not held through the tile loop.
// Returns the rings' next slot, with their parity in bit 8 and an abort in
// bit 9.
template <class T>
__device__ __noinline__ uint32_t stream_range(const FastArgs &a, uint8_t *smem, uint32_t seq,
                                              uint32_t part, int32_t L, uint32_t t0, bool dir,
                                              uint32_t t1, uint32_t ring)
{
    uint32_t s = ring & 0xffu, phase = (ring >> 8) & 1u, n_my = 0;
    bool any_abort = false;
    range_body<T, true, false>(a, smem, seq, part, L, t0, dir, t1, s, phase, n_my, any_abort);
    return s | phase << 8 | (any_abort ? 1u : 0u) << 9;
}

// Exclusive prefix of the query rows' tile counts (ceil(L / 16), 0 for an
// empty row) into pre[0 .. rows], pre[rows] = all tiles; every thread of the
// CTA takes part.  Each thread sums a run of consecutive rows, the run sums
// are scanned across the CTA, then each thread writes its run's prefixes.
__device__ __forceinline__ void block_tile_prefix(const DecodeParams &p, uint32_t *pre,
                                                  uint32_t rows)
{
    __shared__ uint32_t wsum[32];
    const uint32_t nt = blockDim.x, t = threadIdx.x, lane = t & 31, w = t >> 5;
    const uint32_t per = (rows + nt - 1) / nt;
    const uint32_t r0 = min(t * per, rows), r1 = min(r0 + per, rows);
    auto tiles = [&](uint32_t r) -> uint32_t {
        const int32_t L = row_len(p.seq_lens, p.q_tokens, r);
        return L > 0 ? ((uint32_t)L + kTile - 1) / kTile : 0u;
    };
    uint32_t sum = 0;
    for (uint32_t r = r0; r < r1; ++r)
        sum += tiles(r);
    uint32_t x = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
        if ((int)lane >= o)
            x += y;
    }
    if (lane == 31)
        wsum[w] = x;
    __syncthreads();
    if (w == 0) {
        uint32_t v = lane < (nt >> 5) ? wsum[lane] : 0u;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(0xffffffffu, v, o);
            if ((int)lane >= o)
                v += y;
        }
        __syncwarp();
        wsum[lane] = v;
    }
    __syncthreads();
    uint32_t base = (w > 0 ? wsum[w - 1] : 0u) + x - sum;
    for (uint32_t r = r0; r < r1; ++r) {
        pre[r] = base;
        base += tiles(r);
    }
    if (t == nt - 1)
        pre[rows] = base;
}

// Stream-K decode for batches wider than the machine (a stream plan): the
// tiles of all query rows, in row order, are cut into equal ranges of
// chunk = part_tokens / 16 tiles, one per CTA ("feat: add paged-attention
// monolithic decode-only AR foundation", lucebox pull 555, Roadmap: the
// stream-K decode kernel for ragged batches).  A CTA walks the segments of
// its range (a row's tiles inside it) in order on the same per-warp rings:
// a segment that is a whole row writes the row's output; a row cut by range
// boundaries gets one partial per CTA that covers it (index: the CTA minus
// the row's first CTA), counted on the row's completion counter, and the CTA
// that completes the count merges the row after its own segments, with the
// arithmetic of pa_merge.  Nothing waits.  Rows without tokens are written as
// zeros by CTA (row mod grid).
template <class T>
__global__ void __launch_bounds__(T::kMaxWarps * 32, 1)
    stream_decode_kernel(const __grid_constant__ FastArgs a)
{
    const DecodeParams &p = a.p;
    extern __shared__ __align__(16) uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t NSW = a.n_slots, nwarps = blockDim.x >> 5;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + a.region_bytes) + warp * NSW;
    __shared__ uint32_t s_row0, s_pre0, s_total;

    if (lane == 0) {
        for (uint32_t s = 0; s < NSW; ++s)
            mbar_init(&full[s], 1);  // range_body's: the first NSW of the warp's
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    // everything below reads inputs that an earlier grid may have written
    grid_dependency_wait();

    // the rows' tile prefix, in the ring region before any copy lands there
    const uint32_t rows = p.n_seqs, chunk = p.part_tokens / kTile;
    uint32_t *pre = reinterpret_cast<uint32_t *>(smem);
    block_tile_prefix(p, pre, rows);
    __syncthreads();
    const uint32_t c0 = blockIdx.x * chunk;
    if (tid == 0) {
        // the first row whose tiles reach past c0
        uint32_t lo = 0, hi = rows;
        while (lo < hi) {
            const uint32_t mid = (lo + hi) / 2;
            if (pre[mid + 1] > c0)
                hi = mid;
            else
                lo = mid + 1;
        }
        s_row0 = lo;
        s_pre0 = lo < rows ? pre[lo] : pre[rows];
        s_total = pre[rows];
        if (blockIdx.x == gridDim.x - 1 && (uint64_t)pre[rows] > (uint64_t)gridDim.x * chunk)
            atomicOr(p.status, PA_STATUS_LEN_OVER_PLAN);  // tiles past the last range
    }
    __syncthreads();  // the rings take the region back below
    // The segment walk keeps its CTA-wide state in shared memory (st_row:
    // the next row, st_pre: its first tile; st_m*: the rows this CTA merges),
    // so that only the rings' slot and parity stay in registers through the
    // tile loops.
    __shared__ uint32_t st_row, st_pre, st_nm, st_mrow[2], st_mn[2];
    if (tid == 0) {
        st_row = s_row0;
        st_pre = s_pre0;
        st_nm = 0;
    }
    __syncthreads();
    uint32_t s = 0, phase = 0;  // the rings' next use
    bool any_abort = false;
    // one segment of row r starting at tile pr of the concatenation: its
    // tile range [at, bt) in the row, whether it is the whole row, the CTA of
    // the row's first tile and the number of CTAs the row spans (nothing of
    // it stays live through a segment's tile loop: it is formed again after)
    struct Seg {
        int32_t L;
        uint32_t tiles, at, bt, cf, nr;
        bool dir;
    };
    auto segment = [&](uint32_t r, uint32_t pr) -> Seg {
        Seg g;
        g.L = row_len(p.seq_lens, p.q_tokens, r);
        g.tiles = g.L > 0 ? ((uint32_t)g.L + kTile - 1) / kTile : 0u;
        const uint32_t c1 = min(c0 + chunk, s_total);
        g.at = c0 > pr ? c0 - pr : 0u;
        g.bt = min(c1 - pr, g.tiles);
        g.dir = g.at == 0 && g.bt == g.tiles;
        g.cf = pr / chunk;
        g.nr = g.tiles ? (pr + g.tiles - 1) / chunk - g.cf + 1 : 0u;
        return g;
    };
    while (!any_abort) {
        if (st_row >= rows || st_pre >= min(c0 + chunk, s_total))
            break;
        {
            const Seg g = segment(st_row, st_pre);
            if (g.tiles > 0 && !g.dir && g.nr > p.n_parts) {
                // lengths past what the plan covers: the row is left out
                if (tid == 0)
                    atomicOr(p.status, PA_STATUS_LEN_OVER_PLAN);
            } else if (g.tiles > 0) {
                const uint32_t rs =
                    stream_range<T>(a, smem, st_row, blockIdx.x - g.cf, g.L, g.at * kTile, g.dir,
                                    g.bt * kTile, s | phase << 8);
                s = rs & 0xffu;
                phase = (rs >> 8) & 1u;
                any_abort = (rs >> 9) & 1u;
                const Seg h = segment(st_row, st_pre);
                const bool last =
                    !h.dir && merge_arrive(p.counters + (uint64_t)st_row *
                                                            merge_counters_per_seq(p.n_parts),
                                           h.nr);
                if (last && tid == 0 && st_nm < 2) {
                    st_mrow[st_nm] = st_row;
                    st_mn[st_nm] = h.nr;
                    ++st_nm;
                }
            }
        }
        __syncthreads();  // every thread is done with st_row / st_pre
        if (tid == 0) {
            const Seg g = segment(st_row, st_pre);
            st_pre += g.tiles;
            ++st_row;
        }
        __syncthreads();  // the combine's reads of the rings before the next copies
    }
    // every input read (the last segment's query included): the next grid on
    // the stream may be scheduled
    launch_dependents();
    // the rows whose count this CTA completed: all partials written and visible
    const __half *po = static_cast<const __half *>(p.part_o);
    const float2 *pml = reinterpret_cast<const float2 *>(p.part_ml);
    for (uint32_t i = 0; i < st_nm; ++i) {
        for (uint32_t h = warp; h < p.hq; h += nwarps) {
            const uint64_t row = (uint64_t)st_mrow[i] * p.hq + h;
            const __half *rpo = po + row * p.n_parts * p.d;
            const float2 *rml = pml + row * p.n_parts;
            float *rout = p.out + row * p.d;
            if (p.d == 256)
                merge_rows_warp_v<8, 1, false, 8>(&rpo, &rml, st_mn[i], 1, p.d, 1, &rout, nullptr,
                                                  nullptr);
            else
                merge_rows_warp_v<4, 1, false, 8>(&rpo, &rml, st_mn[i], 1, p.d, 1, &rout,
                                                  nullptr, nullptr);
        }
    }
    // rows without tokens: zero output
    for (uint32_t rz = blockIdx.x; rz < rows; rz += gridDim.x) {
        if (row_len(p.seq_lens, p.q_tokens, rz) > 0)
            continue;
        float4 *o4 = reinterpret_cast<float4 *>(p.out + (uint64_t)rz * p.hq * p.d);
        for (uint32_t i = tid; i < p.hq * p.d / 4; i += blockDim.x)
            o4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
}

// Combine of the parked (m, l, O) of the wph warps of every head group into
// the partition's result: for each query head, M = max of the warps'
// reference maxima, f_k = 2^(m_k - M), O = sum f_k O_k / sum f_k l_k.  First
// one thread per query head forms M, the f_k and 1 / sum f_k l_k into `fac`;
// then every thread of the CTA takes 8-dim chunks of the output rows, so the
// partial rows are written with coalesced 16-byte stores (f16 partials) or
// 32-byte stores (the f32 output of a direct CTA, `dir`).  The loops stay
// rolled: this runs once per launch, from cold instruction caches.
template <class T>
__device__ __forceinline__ void combine_and_write(const DecodeParams &p, const float *park,
                                                  float *fac, uint32_t hkv, uint32_t wph,
                                                  uint32_t G, uint32_t seq, uint32_t part,
                                                  bool dir)
{
    constexpr uint32_t NQ = T::D / 8;
    constexpr uint32_t FS = Park<T>::kFac;
    const uint32_t nh = hkv * G;
    for (uint32_t hg = threadIdx.x; hg < nh; hg += blockDim.x) {
        const uint32_t g = hg / G, h = hg - g * G;
        float M = -INFINITY;
#pragma unroll 1
        for (uint32_t k = 0; k < wph; ++k)
            M = fmaxf(M, park[(g + k * hkv) * Park<T>::kWarp + h]);
        float l = 0.0f;
#pragma unroll 1
        for (uint32_t k = 0; k < wph; ++k) {
            const float *w = park + (g + k * hkv) * Park<T>::kWarp;
            const float mk = w[h];
            const float f = mk == -INFINITY ? 0.0f : exp2f(mk - M);
            l = fmaf(w[8 + h], f, l);
            fac[hg * FS + k] = f;
        }
        fac[hg * FS + T::kMaxWarps] = l > 0.0f ? 1.0f / l : 0.0f;
        fac[hg * FS + T::kMaxWarps + 1] = l > 0.0f ? M : -INFINITY;
        fac[hg * FS + T::kMaxWarps + 2] = l;
    }
    __syncthreads();
    const uint32_t n_chunks = nh * NQ;
#pragma unroll 1
    for (uint32_t c = threadIdx.x; c < n_chunks; c += blockDim.x) {
        const uint32_t hg = c / NQ, q = c % NQ;
        const uint32_t g = hg / G, h = hg - g * G;
        float acc[8];
#pragma unroll
        for (int j = 0; j < 8; ++j)
            acc[j] = 0.0f;
#pragma unroll 4
        for (uint32_t k = 0; k < wph; ++k) {
            const float f = fac[hg * FS + k];
            const float4 *src = reinterpret_cast<const float4 *>(
                park + (g + k * hkv) * Park<T>::kWarp + 16 + h * Park<T>::kRow + 8 * q);
            const float4 a = src[0], b = src[1];
            acc[0] = fmaf(f, a.x, acc[0]);
            acc[1] = fmaf(f, a.y, acc[1]);
            acc[2] = fmaf(f, a.z, acc[2]);
            acc[3] = fmaf(f, a.w, acc[3]);
            acc[4] = fmaf(f, b.x, acc[4]);
            acc[5] = fmaf(f, b.y, acc[5]);
            acc[6] = fmaf(f, b.z, acc[6]);
            acc[7] = fmaf(f, b.w, acc[7]);
        }
        const float inv = fac[hg * FS + T::kMaxWarps];
        if (dir) {
            const uint64_t row = (uint64_t)seq * p.hq + hg;
            float4 *dst = reinterpret_cast<float4 *>(p.out + row * T::D + 8 * q);
            dst[0] = make_float4(acc[0] * inv, acc[1] * inv, acc[2] * inv, acc[3] * inv);
            dst[1] = make_float4(acc[4] * inv, acc[5] * inv, acc[6] * inv, acc[7] * inv);
        } else {
            uint4 v;
            v.x = h2_bits(__floats2half2_rn(acc[0] * inv, acc[1] * inv));
            v.y = h2_bits(__floats2half2_rn(acc[2] * inv, acc[3] * inv));
            v.z = h2_bits(__floats2half2_rn(acc[4] * inv, acc[5] * inv));
            v.w = h2_bits(__floats2half2_rn(acc[6] * inv, acc[7] * inv));
            // partials of partitioned row seq sit at index seq - n_direct
            const uint64_t row = (uint64_t)(seq - p.n_direct) * p.hq + hg;
            __half *po = static_cast<__half *>(p.part_o);
            *reinterpret_cast<uint4 *>(po + (row * p.n_parts + part) * T::D + 8 * q) = v;
            if (q == 0)
                reinterpret_cast<float2 *>(p.part_ml)[row * p.n_parts + part] = make_float2(
                    fac[hg * FS + T::kMaxWarps + 1], fac[hg * FS + T::kMaxWarps + 2]);
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
    uint32_t slots32 = 0;    // 32-token slots per K/V head (kTile32 types)
    uint32_t bar_slots = 0;  // mbarriers and flag words per warp
    size_t smem = 0;
};

template <class T>
Geometry geometry(uint32_t hkv)
{
    Geometry gm;
    const size_t slot = T::kSlot;
    const size_t park_per_warp = Park<T>::kWarp * 4, fac_bytes = Park<T>::kFacBytes;
    for (uint32_t wph = T::kMaxWarps / hkv; wph >= 1; --wph) {
        const uint32_t warps = wph * hkv;
        const size_t fixed = 1024 + warps * (size_t)T::SCRATCH + warps * 16 * 12 + 64 +
                             hkv * (size_t)T::QBYTES;
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
            size_t ring = warps * ns * slot, park = warps * park_per_warp + fac_bytes;
            gm.region = (uint32_t)(ring > park ? ring : park);
            gm.bar_slots = (uint32_t)ns;
            gm.smem = 1024 + gm.region + warps * ns * (8 + 4) + 16 + warps * (size_t)T::SCRATCH +
                      hkv * (size_t)T::QBYTES;
            if constexpr (T::kTile32) {
                // the 32-token rings of range_body32: S slots of 4 * kSideK per
                // head, at least one per warp of the head and one more; wph
                // barriers per slot (S per warp), flag words likewise; twice
                // the scratch per warp
                const size_t slot32 = 4 * (size_t)T::kSideK;
                size_t s32 = 32;
                for (; s32 > wph; --s32) {
                    const size_t bs = s32 > ns ? s32 : ns;
                    const size_t need = 1024 + warps * bs * (8 + 4) + 16 +
                                        warps * (size_t)T::SCRATCH2 + hkv * (size_t)T::QBYTES +
                                        (hkv * s32 * slot32 > gm.region ? hkv * s32 * slot32
                                                                        : gm.region);
                    if (need <= kSmemBudget)
                        break;
                }
                if (s32 < wph + 1)
                    return Geometry{};
                gm.slots32 = (uint32_t)s32;
                gm.bar_slots = (uint32_t)(s32 > ns ? s32 : ns);
                if (hkv * s32 * slot32 > gm.region)
                    gm.region = (uint32_t)(hkv * s32 * slot32);
                gm.smem = 1024 + warps * (size_t)gm.bar_slots * (8 + 4) + 16 +
                          warps * (size_t)T::SCRATCH2 + hkv * (size_t)T::QBYTES + gm.region;
            }
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
    const uint64_t n_slots = p.n_pool_blocks * p.block_size;
    for (int side = 0; side < 2; ++side) {
        const uint8_t *pool = side ? p.v_pool : p.k_pool;
        const uint64_t rb = side ? T::kRowV : T::kRowK;  // bytes of one row
        const uint32_t nx = side ? T::kTmaXV : T::kTmaXK;
        for (uint32_t g = 0; g < p.hkv; ++g) {
            cuuint64_t dims[2] = {rb / 2, n_slots}, strides[1] = {(cuuint64_t)p.hkv * rb};
            cuuint32_t box[2] = {nx > 1 ? 64u : (cuuint32_t)(rb / 2), (cuuint32_t)kTile};
            cuuint32_t estr[2] = {1, 1};
            // f16 rows: 64-value chunks with the 128-byte swizzle; quantised rows whole
            const CUtensorMapSwizzle sw =
                nx > 1 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE;
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
        e = cudaFuncSetAttribute(fast_decode_kernel<T, false>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)(kSmemBudget + 4096));
        if (e == cudaSuccess && T::kStagedMerge)
            e = cudaFuncSetAttribute(fast_decode_kernel<T, T::kStagedMerge>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)(kSmemBudget + 4096));
        if constexpr (T::kStream)
            if (e == cudaSuccess)
                e = cudaFuncSetAttribute(stream_decode_kernel<T>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)(kSmemBudget + 4096));
        if (e != cudaSuccess)
            return e;
        done[dev] = true;
    }
    return cudaSuccess;
}

// The tensor maps depend only on the pools, their size and the head layout.
// Encodings are kept per pool pair, so that the steps of every layer of a
// model (one pool pair each) skip the encoding; the table is emptied when it
// passes kMaxMaps entries.
struct MapKey {
    const void *k, *v;
    uint64_t n_blocks;
    uint32_t block_size, hkv, d, type;
    bool operator==(const MapKey &o) const
    {
        return k == o.k && v == o.v && n_blocks == o.n_blocks && block_size == o.block_size &&
               hkv == o.hkv && d == o.d && type == o.type;
    }
};

struct MapKeyHash {
    size_t operator()(const MapKey &m) const
    {
        uint64_t h = reinterpret_cast<uintptr_t>(m.k) * 0x9E3779B97F4A7C15ull;
        h ^= reinterpret_cast<uintptr_t>(m.v) + 0x632BE59BD9B4E019ull + (h << 6) + (h >> 2);
        h ^= m.n_blocks + ((uint64_t)m.block_size << 40) + ((uint64_t)m.hkv << 48) +
             ((uint64_t)m.d << 20) + m.type + (h << 6) + (h >> 2);
        return (size_t)h;
    }
};

struct Maps {
    CUtensorMap tm[2][kMaxHkv];
};

template <class T>
int cached_maps(const DecodeParams &p, FastArgs &a, const char *entry)
{
    constexpr size_t kMaxMaps = 4096;
    static std::mutex mu;
    static std::unordered_map<MapKey, Maps, MapKeyHash> table;
    const MapKey key{p.k_pool, p.v_pool, p.n_pool_blocks, p.block_size, p.hkv, (uint32_t)T::D,
                     T::kTypeKey};
    std::lock_guard<std::mutex> lock(mu);
    const auto it = table.find(key);
    if (it != table.end()) {
        memcpy(a.tm, it->second.tm, sizeof a.tm);
        return PA_OK;
    }
    int rc = encode_maps<T>(p, a, entry);
    if (rc)
        return rc;
    try {
        if (table.size() >= kMaxMaps)
            table.clear();
        Maps m;
        memcpy(m.tm, a.tm, sizeof a.tm);
        table.emplace(key, m);
    } catch (...) {
        // out of host memory: this launch still has its maps
    }
    return PA_OK;
}

// A boolean setting from the environment, read once: unset, "" or anything
// but "0" keeps the default `on`.
bool env_on(const char *name)
{
    const char *v = getenv(name);
    return !(v && v[0] == '0' && v[1] == '\0');
}

// CTA slots of the current device for this instance (SMs x CTAs per SM), once
// per device; 0 if unknown.
template <class T>
uint32_t resident_slots(const Geometry &gm)
{
    static std::mutex mu;
    static uint32_t slots[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return 0;
    std::lock_guard<std::mutex> lock(mu);
    if (!slots[dev]) {
        int sms = 0, cps = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&cps, fast_decode_kernel<T, false>,
                                                          gm.warps * 32, gm.smem) != cudaSuccess) {
            cudaGetLastError();
            return 0;
        }
        slots[dev] = (uint32_t)(sms * cps);
    }
    return slots[dev];
}

template <class T>
int launch_t(const DecodeParams &p, cudaStream_t st, const char *entry)
{
    const Geometry gm = geometry<T>(p.hkv);
    if (!gm.warps)
        return fail(PA_ERR_INVALID, entry, "fast kernel: a tile does not fit shared memory");
    FastArgs a;
    memset(&a, 0, sizeof a);
    int rc = cached_maps<T>(p, a, entry);
    if (rc)
        return rc;
    a.p = p;
    a.n_slots = gm.n_slots;
    a.slot_bytes = gm.slot_bytes;
    a.region_bytes = gm.region;
    a.n_slots32 = gm.slots32;
    a.bar_slots = gm.bar_slots;
    rc = cuda_check(allow_smem<T>(), entry, "cudaFuncSetAttribute");
    if (rc)
        return rc;
    // the cooperative in-launch merge: one-pass plans (at most 32 partitions)
    // without direct rows whose whole grid is resident at once
    static const bool coop_on = env_on("PA_COOP_MERGE");
    a.coop = coop_on && p.counters && !p.direct && p.n_direct == 0 &&
             merge_group_size(p.n_parts) >= p.n_parts && p.n_ctas <= resident_slots<T>(gm);
    a.coop_wait_ns = p.merge_no_wait ? 0u : kCoopWaitNs;
    // two-pass merges (more than 32 partitions) on CTAs of 8 warps or more
    // take the instance with the staged merge
    const bool staged = T::kStagedMerge && p.counters && !p.direct &&
                        merge_group_size(p.n_parts) < p.n_parts && gm.warps >= 8;
    // programmatic dependent launch: this grid may be scheduled while the
    // previous grid on the stream finishes; the kernel waits for that grid
    // (griddepcontrol.wait) before it reads any input
    static const bool pdl_on = env_on("PA_PDL");
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.n_ctas);
    cfg.blockDim = dim3(gm.warps * 32);
    cfg.dynamicSmemBytes = gm.smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_on ? 1 : 0;
    cudaError_t e;
    if (p.stream) {
        // stream plans: the rows' tile prefix is formed in the ring region
        if (!T::kStream || (uint64_t)(p.n_seqs + 1) * 4 > gm.region)
            return fail(PA_ERR_INVALID, entry, "stream plan: %u query rows unsupported here",
                        p.n_seqs);
        a.coop = 0;
        if constexpr (T::kStream)
            e = cudaLaunchKernelEx(&cfg, stream_decode_kernel<T>, a);
        else
            e = cudaErrorInvalidValue;
    } else if (staged) {
        e = cudaLaunchKernelEx(&cfg, fast_decode_kernel<T, T::kStagedMerge>, a);
    } else {
        e = cudaLaunchKernelEx(&cfg, fast_decode_kernel<T, false>, a);
    }
    if (e != cudaSuccess)
        return cuda_check(e, entry, "fast_decode_kernel launch");
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
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(cps, fast_decode_kernel<T, false>,
                                                          gm.warps * 32, gm.smem);
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

bool hkv_ok(uint32_t hkv) { return hkv == 1 || hkv == 2 || hkv == 4 || hkv == 8; }

}  // namespace
}  // namespace pa

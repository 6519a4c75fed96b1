// pa_device.cuh -- device helpers shared by the library's kernels.
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

namespace pa {

constexpr float kLog2e = 1.4426950408889634f;

// Byte offset of the pool row (block, slot, K/V head): widened to 64 bits
// before the first multiply ("fix(paged-attention): use 64-bit pool offsets
// in the fused decode kernels", mlxcel issue 2153, Proposed Solution).  The
// block id is validated by the caller (0 <= block < n_pool_blocks).
__device__ __forceinline__ uint64_t row_offset(int32_t block, uint32_t slot, uint32_t kv_head,
                                               uint32_t block_size, uint32_t hkv,
                                               uint64_t row_bytes)
{
    uint64_t token_slot = (uint64_t)(uint32_t)block * (uint64_t)block_size + slot;
    return (token_slot * (uint64_t)hkv + kv_head) * row_bytes;
}

__device__ __forceinline__ bool block_in_pool(int32_t block, uint64_t n_pool_blocks)
{
    return block >= 0 && (uint64_t)block < n_pool_blocks;
}

__device__ __forceinline__ float half_bits_to_float(uint16_t b)
{
    return __half2float(__ushort_as_half(b));
}

__device__ __forceinline__ uint16_t load_u16(const uint8_t *p)
{
    // pool scale fields sit at 2-byte aligned offsets
    return *reinterpret_cast<const uint16_t *>(p);
}

__device__ __forceinline__ float warp_max(float v)
{
#pragma unroll
    for (int o = 16; o; o >>= 1)
        v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o; o >>= 1)
        v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ int warp_sum_int(int v)
{
#pragma unroll
    for (int o = 16; o; o >>= 1)
        v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Maps a CTA of a partitioned decode grid to its (sequence, partition): CTAs
// enumerate the live (s, p) pairs in order of s, then p, where sequence s has
// ceil(L_s / part_tokens) live partitions.  Executed by one full warp; returns
// false when the CTA index is past the last live pair.
__device__ __forceinline__ bool cta_work(const int32_t *seq_lens, uint32_t n_seqs,
                                         uint32_t part_tokens, uint32_t cta, uint32_t *seq,
                                         uint32_t *part)
{
    const int lane = threadIdx.x & 31;
    uint32_t base = 0;
    for (uint32_t s0 = 0; s0 < n_seqs; s0 += 32) {
        uint32_t s = s0 + lane;
        int32_t L = s < n_seqs ? seq_lens[s] : 0;
        uint32_t n = L > 0 ? ((uint32_t)L + part_tokens - 1) / part_tokens : 0;
        uint32_t incl = n;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            uint32_t t = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o)
                incl += t;
        }
        unsigned hit = __ballot_sync(0xffffffffu, cta < base + incl);
        if (hit) {
            int l = __ffs(hit) - 1;
            uint32_t incl_l = __shfl_sync(0xffffffffu, incl, l);
            uint32_t n_l = __shfl_sync(0xffffffffu, n, l);
            *seq = s0 + l;
            *part = cta - (base + incl_l - n_l);
            return true;
        }
        base += __shfl_sync(0xffffffffu, incl, 31);
    }
    return false;
}

// Stable split-softmax merge of the stored partials of one (sequence, query
// head) row, NR rows at once by one warp ("feat: add paged-attention monolithic
// decode-only AR foundation", lucebox pull 555, Summary): M = max m_p over
// partials with l_p > 0, w_p = l_p 2^(m_p - M), out = sum_p w_p o_p / sum_p w_p;
// partials with l_p == 0 are skipped and none gives 0.  po[r] / pml[r] point
// at row r's partials (rows r >= nr are skipped); loads go through L2 (.cg) so
// that partials written by other CTAs of the same launch are seen.  D is a
// multiple of 32.
template <int VEC, int NR>
__device__ __forceinline__ void merge_rows_warp_v(const __half *const *po, const float2 *const *pml,
                                                  float *const *out, int nr, uint32_t n_live,
                                                  uint32_t D)
{
    const int lane = threadIdx.x & 31;
    // reference maximum over live partials, per row
    float M[NR];
#pragma unroll
    for (int r = 0; r < NR; ++r)
        M[r] = -INFINITY;
    for (uint32_t p = lane; p < n_live; p += 32) {
#pragma unroll
        for (int r = 0; r < NR; ++r) {
            if (r < nr) {
                const float2 ml = __ldcg(pml[r] + p);
                if (ml.y > 0.0f)
                    M[r] = fmaxf(M[r], ml.x);
            }
        }
    }
    float acc[NR][VEC], ws[NR];  // ws: lane-partial sum of the weights
#pragma unroll
    for (int r = 0; r < NR; ++r) {
        M[r] = warp_max(M[r]);
        ws[r] = 0.0f;
#pragma unroll
        for (int j = 0; j < VEC; ++j)
            acc[r][j] = 0.0f;
    }
    for (uint32_t c = 0; c < n_live; c += 32) {
        // lane p holds the weight of partial c + p (0 for dead or absent ones)
        float w[NR];
#pragma unroll
        for (int r = 0; r < NR; ++r) {
            w[r] = 0.0f;
            if (r < nr && c + lane < n_live) {
                const float2 ml = __ldcg(pml[r] + c + lane);
                if (ml.y > 0.0f)
                    w[r] = ml.y * exp2f(ml.x - M[r]);
            }
            ws[r] += w[r];
        }
        const uint32_t cnt = min(32u, n_live - c);
        for (uint32_t q0 = 0; q0 < cnt; q0 += 8) {
            // eight partial rows of every row in flight at once; VEC values each
            uint4 raw[NR][8];
#pragma unroll
            for (int r = 0; r < NR; ++r) {
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    if (r < nr && q0 + k < cnt) {
                        const __half *src = po[r] + (uint64_t)(c + q0 + k) * D + VEC * lane;
                        if constexpr (VEC == 8) {
                            raw[r][k] = __ldcg(reinterpret_cast<const uint4 *>(src));
                        } else {
                            const uint2 r2 = __ldcg(reinterpret_cast<const uint2 *>(src));
                            raw[r][k] = make_uint4(r2.x, r2.y, 0u, 0u);
                        }
                    }
                }
            }
#pragma unroll
            for (int r = 0; r < NR; ++r) {
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const float wk = __shfl_sync(0xffffffffu, w[r], (q0 + k) & 31);
                    if (r < nr && q0 + k < cnt && wk > 0.0f) {
                        const __half2 *h2 = reinterpret_cast<const __half2 *>(&raw[r][k]);
#pragma unroll
                        for (int j = 0; j < VEC / 2; ++j) {
                            const float2 f = __half22float2(h2[j]);
                            acc[r][2 * j] = fmaf(wk, f.x, acc[r][2 * j]);
                            acc[r][2 * j + 1] = fmaf(wk, f.y, acc[r][2 * j + 1]);
                        }
                    }
                }
            }
        }
    }
#pragma unroll
    for (int r = 0; r < NR; ++r) {
        const float s = warp_sum(ws[r]);
        const float inv = s > 0.0f ? 1.0f / s : 0.0f;
        if (r < nr) {
            float *o = out[r] + VEC * lane;
#pragma unroll
            for (int j = 0; j < VEC; ++j)
                o[j] = acc[r][j] * inv;
        }
    }
}

// Stable split-softmax merge of the stored partials of one (sequence, query
// head) row, NR rows at once by one warp ("feat: add paged-attention monolithic
// decode-only AR foundation", lucebox pull 555, Summary): M = max m_p over
// partials with l_p > 0, w_p = l_p 2^(m_p - M), out = sum_p w_p o_p / sum_p w_p;
// partials with l_p == 0 are skipped and none gives 0.  po[r] / pml[r] point
// at row r's partials (rows r >= nr are skipped); loads go through L2 (.cg) so
// that partials written by other CTAs of the same launch are seen.  D is a
// multiple of 32.
template <int VEC>
__device__ __forceinline__ void merge_row_warp_v(const __half *po, const float2 *pml, float *out,
                                                 uint32_t n_live, uint32_t D)
{
    const int lane = threadIdx.x & 31;
    // reference maximum over live partials
    float M = -INFINITY;
    for (uint32_t p = lane; p < n_live; p += 32) {
        const float2 ml = __ldcg(pml + p);
        if (ml.y > 0.0f)
            M = fmaxf(M, ml.x);
    }
    M = warp_max(M);
    float acc[VEC];
#pragma unroll
    for (int j = 0; j < VEC; ++j)
        acc[j] = 0.0f;
    float ws = 0.0f;  // lane-partial sum of the weights
    for (uint32_t c = 0; c < n_live; c += 32) {
        // lane p holds the weight of partial c + p (0 for dead or absent ones)
        float w = 0.0f;
        if (c + lane < n_live) {
            const float2 ml = __ldcg(pml + c + lane);
            if (ml.y > 0.0f)
                w = ml.y * exp2f(ml.x - M);
        }
        ws += w;
        const uint32_t cnt = min(32u, n_live - c);
        for (uint32_t q0 = 0; q0 < cnt; q0 += 8) {
            // eight partial rows in flight at once; this lane's VEC values each
            uint4 raw[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const uint32_t pk = c + q0 + k;
                if (q0 + k < cnt) {
                    const __half *src = po + (uint64_t)pk * D + VEC * lane;
                    if constexpr (VEC == 8) {
                        raw[k] = __ldcg(reinterpret_cast<const uint4 *>(src));
                    } else {
                        const uint2 r2 = __ldcg(reinterpret_cast<const uint2 *>(src));
                        raw[k] = make_uint4(r2.x, r2.y, 0u, 0u);
                    }
                }
            }
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const float wk = __shfl_sync(0xffffffffu, w, (q0 + k) & 31);
                if (q0 + k < cnt && wk > 0.0f) {
                    const __half2 *h2 = reinterpret_cast<const __half2 *>(&raw[k]);
#pragma unroll
                    for (int j = 0; j < VEC / 2; ++j) {
                        const float2 f = __half22float2(h2[j]);
                        acc[2 * j] = fmaf(wk, f.x, acc[2 * j]);
                        acc[2 * j + 1] = fmaf(wk, f.y, acc[2 * j + 1]);
                    }
                }
            }
        }
    }
    ws = warp_sum(ws);
    const float inv = ws > 0.0f ? 1.0f / ws : 0.0f;
    float *o = out + VEC * lane;
#pragma unroll
    for (int j = 0; j < VEC; ++j)
        o[j] = acc[j] * inv;
}

// Stable split-softmax merge of the stored partials of one (sequence, query
// head) row, NR rows at once by one warp ("feat: add paged-attention monolithic
// decode-only AR foundation", lucebox pull 555, Summary): M = max m_p over
// partials with l_p > 0, w_p = l_p 2^(m_p - M), out = sum_p w_p o_p / sum_p w_p
// (summed in partition order); partials with l_p == 0 are skipped and none
// gives 0.  po / pml point at the row's partials; loads go through L2 (.cg) so
// that partials written by other CTAs of the same launch are seen.  Lane i owns
// dims [D/32 * i, D/32 * (i+1)); D is 128 or 256.
__device__ __forceinline__ void merge_row_warp(const __half *po, const float2 *pml, float *out,
                                               uint32_t n_live, uint32_t D)
{
    if (D == 256)
        merge_rows_warp_v<8, 1>(&po, &pml, &out, 1, n_live, D);
    else
        merge_rows_warp_v<4, 1>(&po, &pml, &out, 1, n_live, D);
}

// Two rows at once, with the same arithmetic per row as merge_row_warp (the
// loads of both rows are in flight together); row 1 is skipped when nr == 1.
__device__ __forceinline__ void merge_row_pair_warp(const __half *const po[2],
                                                    const float2 *const pml[2],
                                                    float *const out[2], int nr,
                                                    uint32_t n_live, uint32_t D)
{
    if (D == 256)
        merge_rows_warp_v<8, 2>(po, pml, out, nr, n_live, D);
    else
        merge_rows_warp_v<4, 2>(po, pml, out, nr, n_live, D);
}

// In-launch merge ("HRX: multi-pass KV-block reduction for flash-attention
// decode-split", llama.cpp fork pull 13, Changes: the reduction runs in the
// same launch through an atomic completion counter, with no second dispatch and
// no waiting).  Called by every thread of a CTA after it has written the
// partials of (sequence seq, its partition): the CTA that completes the
// sequence's count merges all its rows into out and resets the counter to 0.
// Nothing ever waits on another CTA.
template <class P>
__device__ inline void fused_merge_tail(const P &p, uint32_t seq, uint32_t warp, uint32_t nwarps)
{
    __shared__ int last;
    __threadfence();  // this thread's partial writes before the count
    __syncthreads();
    const int32_t L = p.seq_lens[seq];
    const uint32_t n_live = L > 0 ? ((uint32_t)L + p.part_tokens - 1) / p.part_tokens : 0;
    if (threadIdx.x == 0) {
        const int old = atomicAdd(&p.counters[seq], 1);
        last = (uint32_t)(old + 1) == n_live;
        if (last)
            p.counters[seq] = 0;  // every partition of this launch has counted
    }
    __syncthreads();
    if (!last)
        return;
    __threadfence();  // the other CTAs' partials are visible past their counts
    const __half *po = static_cast<const __half *>(p.part_o);
    const float2 *pml = reinterpret_cast<const float2 *>(p.part_ml);
    // rows h and h + nwarps together, so that a warp has both rows' loads in flight
    for (uint32_t h = warp; h < p.hq; h += 2 * nwarps) {
        const uint64_t s0 = (uint64_t)seq * p.hq + h;
        const uint64_t s1 = h + nwarps < p.hq ? s0 + nwarps : s0;
        const __half *rpo[2] = {po + s0 * p.n_parts * p.d, po + s1 * p.n_parts * p.d};
        const float2 *rml[2] = {pml + s0 * p.n_parts, pml + s1 * p.n_parts};
        float *rout[2] = {p.out + s0 * p.d, p.out + s1 * p.d};
        merge_row_pair_warp(rpo, rml, rout, h + nwarps < p.hq ? 2 : 1, n_live, p.d);
    }
}

}  // namespace pa

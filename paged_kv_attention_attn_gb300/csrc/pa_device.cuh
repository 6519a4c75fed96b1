// pa_device.cuh -- device helpers shared by the library's kernels.
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

#include "pa_internal.h"

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

// q8_1 code of value v in a block of 32 whose largest magnitude is amax, with
// the block scale d = amax / 127 ("feat: add paged-attention monolithic
// decode-only AR foundation", lucebox pull 555, Summary: Q is quantised to
// q8_1 once per step).  float32 IEEE division, roundf (ties away from zero),
// clamped to [-127, 127]; an all-zero block codes as 0.  The q8_1 pre-pass
// kernel and the decode kernel that quantises its own query share this, so
// both give the same codes.
// The product v * inv_d (inv_d = 1 / d rounded) is within about 1.5e-5 of the
// exact quotient v / d, and so is the rounded quotient (|v / d| <= 127 + a
// rounding step); both round to the same integer unless a half-integer lies
// within that distance.  So the quotient is divided out exactly only when the
// product is within 3e-5 of a half-integer, and the codes are those of the
// IEEE division either way.
__device__ __forceinline__ int q8_1_code(float v, float amax, float d, float inv_d)
{
    if (amax == 0.0f)
        return 0;
    const float r = v * inv_d;
    const float a = fabsf(r);
    const float q = fabsf(a - truncf(a) - 0.5f) > 3.0e-5f ? roundf(r) : roundf(v / d);
    return (int)fminf(fmaxf(q, -127.0f), 127.0f);
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

// Query rows.  A plan with T query tokens per sequence decodes n_seqs * T
// rows; row v is token i = v % T of sequence v / T, at position L - T + i,
// and attends to the keys 0 .. L - T + i ("TensorFold pull 1418", What:
// several query rows of a sequence -- a prompt chunk or a verify window --
// over one paged cache).  With one token the row is the sequence.
__device__ __forceinline__ int32_t row_len(const int32_t *seq_lens, uint32_t T, uint32_t v)
{
    if (T <= 1)
        return seq_lens[v];
    const int32_t L = seq_lens[v / T] - (int32_t)(T - 1 - v % T);
    return L > 0 ? L : 0;
}
__device__ __forceinline__ uint32_t table_row(uint32_t T, uint32_t v)
{
    return T <= 1 ? v : v / T;
}

// Maps a CTA of a partitioned decode grid to its (sequence, partition): CTAs
// enumerate the (s, p) pairs in order of s, then p, where sequence s has
// min(ceil(L_s / part_tokens), n_parts) live partitions, and an empty
// sequence (L_s <= 0) one empty partition.  Executed by one full warp; returns false when the CTA
// index is past the last pair.
__device__ __forceinline__ bool cta_work(const int32_t *seq_lens, uint32_t T, uint32_t n_seqs,
                                         uint32_t part_tokens, uint32_t n_parts,
                                         uint32_t n_direct, uint32_t cta, uint32_t *seq,
                                         uint32_t *part)
{
    // the leading n_direct rows of a wave-filling plan: one CTA each, in order
    if (cta < n_direct) {
        *seq = cta;
        *part = 0;
        return true;
    }
    cta -= n_direct;
    const int lane = threadIdx.x & 31;
    uint32_t base = 0;
    for (uint32_t s0 = n_direct; s0 < n_seqs; s0 += 32) {
        uint32_t s = s0 + lane;
        // an empty sequence still gets one CTA, which writes its zero output
        // (or its empty partial, and its arrival at the completion count)
        const int32_t L = s < n_seqs ? row_len(seq_lens, T, s) : 0;
        uint32_t n = L > 0 ? ((uint32_t)L + part_tokens - 1) / part_tokens : (s < n_seqs ? 1u : 0u);
        n = n < n_parts ? n : n_parts;  // a sequence longer than the plan is cut
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

// ------------------------------------------------------------------ merge
//
// Stable split-softmax merge ("feat: add paged-attention monolithic
// decode-only AR foundation", lucebox pull 555, Summary): for one (sequence,
// query head) row with live partials p (normalised o_p, m_p, l_p): M = max m_p
// over partials with l_p > 0, w_p = l_p 2^(m_p - M), out = sum_p w_p o_p /
// sum_p w_p; partials with l_p == 0 are skipped and none gives 0.
//
// A row with more than 32 live partials is merged in two passes ("HRX:
// multi-pass KV-block reduction for flash-attention decode-split", llama.cpp
// fork pull 13, What: hierarchical KV-block reduction): the partials are cut
// into groups of gs = merge_group_size(n) consecutive ones, each group is
// merged into one partial of the same form (f16 o, (m, l)), then the group
// results are merged.  The merge is associative, so this is the flat merge up
// to rounding.  The in-launch merge and the separate merge kernel use the same
// groups and the same arithmetic, so they give the same bits.

// Merge of n partials of each of NR rows by one warp (rows r >= nr are
// skipped); partial p of row r is at po[r] + p * stride * D and pml[r] +
// p * stride.  kPartial: the result is written in partial form (f16 o to
// out_o[r], (M, or -inf when no weight, and sum w) to out_ml[r]); else as
// float32 to out_f[r].  Lane i owns the VEC/4 dimension quads
// [128 j + 4 i, 128 j + 4 i + 4), so that every load and store of the warp is
// one contiguous run.  The weight sum is lane-partial (lane i adds the
// weights of partials i, i + 32, ... in order) and then a butterfly; every
// dimension is summed in partial order.
// Loads go through L2 (.cg) so that partials written by other CTAs of the
// same launch are seen.
template <int VEC, int NR, bool kPartial, int BATCH = 8>
__device__ __forceinline__ void merge_rows_warp_v(const __half *const *po, const float2 *const *pml,
                                                  uint32_t n, uint32_t stride, uint32_t D,
                                                  int nr, float *const *out_f,
                                                  __half *const *out_o, float2 *const *out_ml)
{
    const int lane = threadIdx.x & 31;
    // BATCH partials of every row in flight at once (the batch size changes
    // only how many loads are in flight, not the order of the arithmetic)
    uint4 raw[NR][BATCH];
    auto load_batch = [&](uint32_t base, uint32_t cnt) {
#pragma unroll
        for (int r = 0; r < NR; ++r) {
#pragma unroll
            for (int k = 0; k < BATCH; ++k) {
                if (r < nr && (uint32_t)k < cnt) {
                    const __half *src = po[r] + (uint64_t)(base + k) * stride * D + 4 * lane;
                    const uint2 q0 = __ldcg(reinterpret_cast<const uint2 *>(src));
                    uint2 q1 = make_uint2(0u, 0u);
                    if constexpr (VEC == 8)
                        q1 = __ldcg(reinterpret_cast<const uint2 *>(src + 128));
                    raw[r][k] = make_uint4(q0.x, q0.y, q1.x, q1.y);
                }
            }
        }
    };
    // the first batch and the (m, l) of partial `lane` are loaded together:
    // neither depends on the reference maximum
    load_batch(0, n < BATCH ? n : BATCH);
    float2 ml0[NR];
    float M[NR];
#pragma unroll
    for (int r = 0; r < NR; ++r) {
        ml0[r] = make_float2(-INFINITY, 0.0f);
        if (r < nr && (uint32_t)lane < n)
            ml0[r] = __ldcg(pml[r] + (uint64_t)lane * stride);
        M[r] = ml0[r].y > 0.0f ? ml0[r].x : -INFINITY;
    }
    for (uint32_t p = lane + 32; p < n; p += 32) {
#pragma unroll
        for (int r = 0; r < NR; ++r) {
            if (r < nr) {
                const float2 ml = __ldcg(pml[r] + (uint64_t)p * stride);
                if (ml.y > 0.0f)
                    M[r] = fmaxf(M[r], ml.x);
            }
        }
    }
    float acc[NR][VEC], ws[NR];
#pragma unroll
    for (int r = 0; r < NR; ++r) {
        M[r] = warp_max(M[r]);
        ws[r] = 0.0f;
#pragma unroll
        for (int j = 0; j < VEC; ++j)
            acc[r][j] = 0.0f;
    }
    for (uint32_t c = 0; c < n; c += 32) {
        // lane i holds the weight of partial c + i (0 for dead or absent ones)
        float w[NR];
#pragma unroll
        for (int r = 0; r < NR; ++r) {
            w[r] = 0.0f;
            if (r < nr && c + lane < n) {
                const float2 ml = c == 0 ? ml0[r] : __ldcg(pml[r] + (uint64_t)(c + lane) * stride);
                if (ml.y > 0.0f)
                    w[r] = ml.y * exp2f(ml.x - M[r]);
            }
            ws[r] += w[r];
        }
        const uint32_t cnt = min(32u, n - c);
        for (uint32_t q0 = 0; q0 < cnt; q0 += BATCH) {
            if (c + q0 > 0)
                load_batch(c + q0, cnt - q0 < BATCH ? cnt - q0 : BATCH);
#pragma unroll
            for (int r = 0; r < NR; ++r) {
#pragma unroll
                for (int k = 0; k < BATCH; ++k) {
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
        if (r >= nr)
            continue;
        if constexpr (kPartial) {
            uint32_t h[VEC / 2];
#pragma unroll
            for (int j = 0; j < VEC / 2; ++j) {
                const __half2 v = __floats2half2_rn(acc[r][2 * j] * inv, acc[r][2 * j + 1] * inv);
                h[j] = *reinterpret_cast<const uint32_t *>(&v);
            }
#pragma unroll
            for (int i = 0; i < VEC / 4; ++i)
                *reinterpret_cast<uint2 *>(out_o[r] + 128 * i + 4 * lane) =
                    make_uint2(h[2 * i], h[2 * i + 1]);
            if (lane == 0)
                *out_ml[r] = make_float2(s > 0.0f ? M[r] : -INFINITY, s);
        } else {
#pragma unroll
            for (int i = 0; i < VEC / 4; ++i)
                *reinterpret_cast<float4 *>(out_f[r] + 128 * i + 4 * lane) =
                    make_float4(acc[r][4 * i] * inv, acc[r][4 * i + 1] * inv,
                                acc[r][4 * i + 2] * inv, acc[r][4 * i + 3] * inv);
        }
    }
}

// Records a sequence longer than the plan covers (its partitions past n_parts
// are left out).  Called by thread 0 of the CTA of partition 0.
__device__ __forceinline__ void check_len_vs_plan(int32_t L, uint32_t n_parts,
                                                  uint32_t part_tokens, int32_t *status)
{
    if (L > 0 && (uint64_t)L > (uint64_t)n_parts * part_tokens)
        atomicOr(status, PA_STATUS_LEN_OVER_PLAN);
}

// Records lengths that need more (sequence, partition) pairs than the grid has
// CTAs (the pairs past the grid are left out).  Called by one full warp of the
// grid's last CTA.
__device__ __forceinline__ void check_grid_vs_plan(const int32_t *seq_lens, uint32_t T,
                                                   uint32_t n_seqs, uint32_t part_tokens,
                                                   uint32_t n_parts, uint32_t n_direct,
                                                   int32_t *status)
{
    const int lane = threadIdx.x & 31;
    uint64_t pairs = lane == 0 ? n_direct : 0;  // the direct rows: one CTA each
    for (uint32_t s = n_direct + lane; s < n_seqs; s += 32) {
        const int32_t L = row_len(seq_lens, T, s);
        uint32_t n = L > 0 ? ((uint32_t)L + part_tokens - 1) / part_tokens : 1u;
        pairs += n < n_parts ? n : n_parts;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        pairs += __shfl_xor_sync(0xffffffffu, pairs, o);
    if (lane == 0 && pairs > gridDim.x)
        atomicOr(status, PA_STATUS_LEN_OVER_PLAN);
}

// One row merged by one warp, the flat merge or the two passes as above,
// float32 out.  The group results are staged in scr (this warp's D halves
// and one (m, l)) exactly as the in-launch merge stores them in part_o, so
// the second pass sees the same bits.
template <int VEC>
__device__ __forceinline__ void merge_row_two_pass_warp(const __half *po, const float2 *pml,
                                                        float *out, uint32_t n, uint32_t D,
                                                        __half *scr, float2 *scr_ml)
{
    const uint32_t gs = merge_group_size(n);
    if (gs >= n) {
        merge_rows_warp_v<VEC, 1, false>(&po, &pml, n, 1, D, 1, &out, nullptr, nullptr);
        return;
    }
    const int lane = threadIdx.x & 31;
    const uint32_t ng = (n + gs - 1) / gs;
    // the second pass's reference maximum: that of the groups is that of all
    float M = -INFINITY;
    for (uint32_t p = lane; p < n; p += 32) {
        const float2 ml = __ldcg(pml + p);
        if (ml.y > 0.0f)
            M = fmaxf(M, ml.x);
    }
    M = warp_max(M);
    float acc[VEC], ws = 0.0f;
#pragma unroll
    for (int j = 0; j < VEC; ++j)
        acc[j] = 0.0f;
    for (uint32_t g = 0; g < ng; ++g) {
        const uint32_t p0 = g * gs, ng_g = min(gs, n - p0);
        const __half *gpo = po + (uint64_t)p0 * D;
        const float2 *gml = pml + p0;
        merge_rows_warp_v<VEC, 1, true>(&gpo, &gml, ng_g, 1, D, 1, nullptr, &scr, &scr_ml);
        __syncwarp();
        const float2 ml = *scr_ml;
        const float w = ml.y > 0.0f ? ml.y * exp2f(ml.x - M) : 0.0f;
        if ((g & 31) == (uint32_t)lane)
            ws += w;
        if (w > 0.0f) {
#pragma unroll
            for (int j = 0; j < VEC / 2; ++j) {
                const __half2 *h2 =
                    reinterpret_cast<const __half2 *>(scr + 128 * (j / 2) + 4 * lane) + (j & 1);
                const float2 f = __half22float2(*h2);
                acc[2 * j] = fmaf(w, f.x, acc[2 * j]);
                acc[2 * j + 1] = fmaf(w, f.y, acc[2 * j + 1]);
            }
        }
        __syncwarp();  // the group result is read before the next one lands
    }
    ws = warp_sum(ws);
    const float inv = ws > 0.0f ? 1.0f / ws : 0.0f;
#pragma unroll
    for (int i = 0; i < VEC / 4; ++i)
        *reinterpret_cast<float4 *>(out + 128 * i + 4 * lane) =
            make_float4(acc[4 * i] * inv, acc[4 * i + 1] * inv, acc[4 * i + 2] * inv,
                        acc[4 * i + 3] * inv);
}

// Arrival of a CTA at a completion counter of the in-launch merge ("HRX:
// multi-pass KV-block reduction for flash-attention decode-split", llama.cpp
// fork pull 13, Changes: the reduction runs in the same launch through an
// atomic completion counter, no second dispatch, no waiting).  Called by every
// thread after the CTA's writes that the count covers; true in the CTA whose
// arrival is the target-th, which resets the counter to 0 for the next launch
// and may then read everything the counted CTAs wrote.  Nothing waits.
__device__ inline bool merge_arrive(int32_t *counter, uint32_t target)
{
    __shared__ int last;
    __threadfence();  // this thread's writes before the count
    __syncthreads();
    if (threadIdx.x == 0) {
        const int old = atomicAdd(counter, 1);
        last = (uint32_t)(old + 1) == target;
        if (last)
            *counter = 0;
    }
    __syncthreads();
    if (!last)
        return false;
    __threadfence();  // the counted CTAs' writes are visible past their counts
    return true;
}

// The in-launch merge, run by every thread of the CTA of (sequence seq,
// partition part) after it has written its partials.  One pass: the CTA that
// completes the sequence merges all its rows into out.  Two passes: the CTA
// that completes a group merges the group's partials of every row into the
// group's first partial slot, and the CTA that completes the last group merges
// the group results into out.  An empty sequence has one CTA and writes 0.
template <int BATCH = 8, class P>
__device__ inline void fused_merge(const P &p, uint32_t seq, uint32_t part, uint32_t warp,
                                   uint32_t nwarps)
{
    const int32_t L = row_len(p.seq_lens, p.q_tokens, seq);
    uint32_t n = L > 0 ? ((uint32_t)L + p.part_tokens - 1) / p.part_tokens : 0;
    n = n < p.n_parts ? n : p.n_parts;
    const uint32_t gs = merge_group_size(n), ng = n > gs ? (n + gs - 1) / gs : 1;
    // partials and counters of partitioned row seq sit at index seq - n_direct
    const uint64_t pseq = seq - p.n_direct;
    int32_t *cnt = p.counters + pseq * merge_counters_per_seq(p.n_parts);
    const __half *po = static_cast<const __half *>(p.part_o);
    const float2 *pml = reinterpret_cast<const float2 *>(p.part_ml);
    if (ng > 1) {
        const uint32_t g = part / gs, p0 = g * gs, ng_g = min(gs, n - p0);
        if (!merge_arrive(cnt + 1 + g, ng_g))
            return;
        for (uint32_t h = warp; h < p.hq; h += 2 * nwarps) {
            const uint64_t s0 = pseq * p.hq + h;
            const uint64_t s1 = h + nwarps < p.hq ? s0 + nwarps : s0;
            const __half *rpo[2] = {po + (s0 * p.n_parts + p0) * p.d,
                                    po + (s1 * p.n_parts + p0) * p.d};
            const float2 *rml[2] = {pml + s0 * p.n_parts + p0, pml + s1 * p.n_parts + p0};
            // in place: the group's first slot, read before it is written
            __half *ro[2] = {const_cast<__half *>(rpo[0]), const_cast<__half *>(rpo[1])};
            float2 *rm[2] = {const_cast<float2 *>(rml[0]), const_cast<float2 *>(rml[1])};
            const int nr = h + nwarps < p.hq ? 2 : 1;
            if (p.d == 256)
                merge_rows_warp_v<8, 2, true, BATCH>(rpo, rml, ng_g, 1, p.d, nr, nullptr, ro, rm);
            else
                merge_rows_warp_v<4, 2, true, BATCH>(rpo, rml, ng_g, 1, p.d, nr, nullptr, ro, rm);
        }
    }
    // the last pass counts the group mergers, or every partition of the
    // sequence (an empty sequence has one CTA)
    if (!merge_arrive(cnt, ng > 1 ? ng : (n > 0 ? n : 1u)))
        return;
    const uint32_t m = ng > 1 ? ng : n, stride = ng > 1 ? gs : 1;
    for (uint32_t h = warp; h < p.hq; h += 2 * nwarps) {
        const uint64_t s0 = pseq * p.hq + h;
        const uint64_t s1 = h + nwarps < p.hq ? s0 + nwarps : s0;
        const uint64_t o0 = (uint64_t)seq * p.hq + h;
        const uint64_t o1 = h + nwarps < p.hq ? o0 + nwarps : o0;
        const __half *rpo[2] = {po + s0 * p.n_parts * p.d, po + s1 * p.n_parts * p.d};
        const float2 *rml[2] = {pml + s0 * p.n_parts, pml + s1 * p.n_parts};
        float *rout[2] = {p.out + o0 * p.d, p.out + o1 * p.d};
        const int nr = h + nwarps < p.hq ? 2 : 1;
        if (p.d == 256)
            merge_rows_warp_v<8, 2, false, BATCH>(rpo, rml, m, stride, p.d, nr, rout, nullptr, nullptr);
        else
            merge_rows_warp_v<4, 2, false, BATCH>(rpo, rml, m, stride, p.d, nr, rout, nullptr, nullptr);
    }
}

}  // namespace pa

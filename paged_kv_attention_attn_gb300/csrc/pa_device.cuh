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

}  // namespace pa

// k_append.cu -- the K/V append step: each sequence's new token is quantised
// into the pool, at the position its resident length names, through its
// resident block table.
//
// "feat: add paged-attention monolithic decode-only AR foundation" (lucebox
// pull 555), Summary: the paging metadata (block table and sequence lengths)
// stays on the device next to the K/V pool, and a decode step uploads only
// the 4-byte id of each fresh 16-token block instead of the whole table;
// Validation: prefill through many block boundaries.  The row formats are the
// decode kernels' (F16, Q8_0, Q4_0); the quantisers follow the ggml reference
// convention in float32, with no contracted multiply-add, so that the bytes
// are the same on every machine.
#include <cuda_fp16.h>
#include <math.h>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

struct AppendParams {
    uint8_t *k_pool, *v_pool;
    uint64_t n_pool_blocks;
    int32_t *block_table;
    uint32_t table_stride;
    int32_t *seq_lens;
    const float *k_new, *v_new;
    const int32_t *fresh;
    int32_t *status;
    uint32_t n_seqs, hkv, d, block_size;
    uint32_t k_type, v_type;
    uint64_t k_row_bytes, v_row_bytes;
};

// One warp quantises one row of D values into its pool bytes; in a 32-value
// block lane i holds value i.
//  Q8_0: amax = max|x|, d = amax / 127, q = clamp(roundf(x * (1/d)), +-127).
//  Q4_0: m = the first value of largest magnitude, d = m / -8,
//        nib = min(15, floor(x * (1/d) + 8.5)); values j and j + 16 share
//        byte j (low, high nibble).
//  F16:  round to nearest even.
// A zero scale gives 1/d = 0.  The scale is stored as f16 (nearest even).
__device__ void quantize_row_warp(uint32_t type, const float *x, uint32_t D, uint8_t *dst)
{
    const int lane = threadIdx.x & 31;
    if (type == PA_F16) {
        for (uint32_t i = lane; i < D; i += 32)
            reinterpret_cast<uint16_t *>(dst)[i] = __half_as_ushort(__float2half_rn(x[i]));
        return;
    }
    for (uint32_t b = 0; b < D / 32; ++b) {
        const float v = x[32 * b + lane];
        if (type == PA_Q8_0) {
            const float amax = warp_max(fabsf(v));
            const float d = amax / 127.0f;
            const float id = d > 0.0f ? 1.0f / d : 0.0f;
            const float r = fminf(fmaxf(roundf(__fmul_rn(v, id)), -127.0f), 127.0f);
            dst[34 * b + 2 + lane] = (uint8_t)(int8_t)(int)r;
            if (lane == 0)
                *reinterpret_cast<uint16_t *>(dst + 34 * b) = __half_as_ushort(__float2half_rn(d));
        } else {
            // the lane of the largest magnitude, the lowest lane among equals
            float ba = fabsf(v);
            int bl = lane;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                const float oa = __shfl_xor_sync(0xffffffffu, ba, off);
                const int ol = __shfl_xor_sync(0xffffffffu, bl, off);
                if (oa > ba || (oa == ba && ol < bl)) {
                    ba = oa;
                    bl = ol;
                }
            }
            const float m = __shfl_sync(0xffffffffu, v, bl);
            const float d = m / -8.0f;
            const float id = d != 0.0f ? 1.0f / d : 0.0f;
            const float f = fminf(fmaxf(floorf(__fadd_rn(__fmul_rn(v, id), 8.5f)), 0.0f), 15.0f);
            const uint32_t nib = (uint32_t)(int)f;
            const uint32_t hi = __shfl_down_sync(0xffffffffu, nib, 16);
            if (lane < 16)
                dst[18 * b + 2 + lane] = (uint8_t)(nib | (hi << 4));
            if (lane == 0)
                *reinterpret_cast<uint16_t *>(dst + 18 * b) = __half_as_ushort(__float2half_rn(d));
        }
    }
}

// One CTA per sequence, 2 * hkv warps (K rows, then V rows).  Thread 0
// resolves the block: a token at slot 0 takes the fresh id and installs it in
// the table, any other slot uses the table's entry.  A table with no entry
// left, or an id outside the pool, leaves the sequence untouched and sets a
// status bit.  The length grows by one after the rows are written.
__global__ void __launch_bounds__(512) append_kernel(const AppendParams p)
{
    __shared__ int blk_sh, slot_sh;
    const uint32_t s = blockIdx.x;
    if (threadIdx.x == 0) {
        int blk = -1, slot = 0;
        const int32_t L = p.seq_lens[s];
        if (L >= 0 && (uint32_t)L / p.block_size < p.table_stride) {
            const uint32_t j = (uint32_t)L / p.block_size;
            slot = (int)((uint32_t)L % p.block_size);
            int32_t *te = p.block_table + (uint64_t)s * p.table_stride + j;
            const int32_t cand = slot == 0 ? p.fresh[s] : *te;
            if (block_in_pool(cand, p.n_pool_blocks)) {
                blk = cand;
                if (slot == 0)
                    *te = cand;
            } else {
                atomicOr(p.status, PA_STATUS_CORRUPT_TABLE);
            }
        } else {
            atomicOr(p.status, PA_STATUS_APPEND_RANGE);
        }
        blk_sh = blk;
        slot_sh = slot;
    }
    __syncthreads();
    const int blk = blk_sh;
    if (blk < 0)
        return;
    const uint32_t warp = threadIdx.x >> 5;
    const uint32_t side = warp / p.hkv, g = warp % p.hkv;
    const uint64_t rb = side ? p.v_row_bytes : p.k_row_bytes;
    uint8_t *dst = (side ? p.v_pool : p.k_pool) +
                   row_offset(blk, (uint32_t)slot_sh, g, p.block_size, p.hkv, rb);
    const float *x = (side ? p.v_new : p.k_new) + ((uint64_t)s * p.hkv + g) * p.d;
    quantize_row_warp(side ? p.v_type : p.k_type, x, p.d, dst);
    __syncthreads();
    if (threadIdx.x == 0)
        p.seq_lens[s] += 1;
}

int launch_append(const pa_append_args *a, cudaStream_t st, const char *entry)
{
    AppendParams p;
    p.k_pool = static_cast<uint8_t *>(a->k_pool);
    p.v_pool = static_cast<uint8_t *>(a->v_pool);
    p.n_pool_blocks = a->n_pool_blocks;
    p.block_table = a->block_table;
    p.table_stride = a->table_stride;
    p.seq_lens = a->seq_lens;
    p.k_new = a->k_new;
    p.v_new = a->v_new;
    p.fresh = a->fresh_blocks;
    p.status = a->status;
    p.n_seqs = a->n_seqs;
    p.hkv = a->hkv;
    p.d = a->d;
    p.block_size = a->block_size;
    p.k_type = a->k_type;
    p.v_type = a->v_type;
    p.k_row_bytes = pa_row_bytes(a->k_type, a->d);
    p.v_row_bytes = pa_row_bytes(a->v_type, a->d);
    if (a->n_seqs == 0)
        return PA_OK;
    append_kernel<<<a->n_seqs, 64 * a->hkv, 0, st>>>(p);
    return cuda_check(cudaGetLastError(), entry, "append_kernel launch");
}

}  // namespace pa

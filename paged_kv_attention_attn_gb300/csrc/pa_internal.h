// pa_internal.h -- declarations shared by the library's translation units.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "pa.h"

namespace pa {

// Records "<entry>: <reason>" as this thread's last error and returns code.
int fail(int code, const char *entry, const char *fmt, ...);
// Wraps a CUDA runtime result: PA_OK, or PA_ERR_CUDA with the runtime's text.
int cuda_check(cudaError_t e, const char *entry, const char *what);

inline cudaStream_t stream_of(pa_stream_t s) { return reinterpret_cast<cudaStream_t>(s); }

// Everything a decode kernel needs, resolved on the host.
#ifdef __CUDACC__
#define PA_HD __host__ __device__
#else
#define PA_HD
#endif

// Smallest g with g * g >= n.
inline PA_HD uint32_t ceil_sqrt_u32(uint32_t n)
{
    uint32_t lo = 0, hi = 65536;
    while (lo < hi) {
        const uint32_t mid = (lo + hi) / 2;
        if ((uint64_t)mid * mid >= n)
            hi = mid;
        else
            lo = mid + 1;
    }
    return lo;
}

// Group size of the merge of n live partials: all of them (one pass) up to 32,
// else ceil(sqrt(n)), so that both passes of the two-pass merge take about
// sqrt(n) partials.
inline PA_HD uint32_t merge_group_size(uint32_t n)
{
    return n <= 32 ? (n > 0 ? n : 1u) : ceil_sqrt_u32(n);
}

// Completion counters per sequence of the in-launch merge: one for the last
// pass and one per group (a sequence has at most ceil(sqrt(n_parts)) groups).
inline PA_HD uint32_t merge_counters_per_seq(uint32_t n_parts)
{
    return 1u + ceil_sqrt_u32(n_parts);
}

struct DecodeParams {
    const uint8_t *k_pool, *v_pool;
    uint64_t n_pool_blocks;
    const int32_t *block_table;
    uint32_t table_stride;
    const int32_t *seq_lens;
    const void *q;          // float32 [S][hq][d] (F16 K, or q_f32) or q8_1 blocks
    uint32_t q_f32;         // quantised K, fast kernel: q is float32 and each CTA
                            // quantises the rows it needs to q8_1 itself
    float scale_log2;       // scale * log2(e)
    void *part_o;           // f16 [S][hq][n_parts][d]
    float *part_ml;         // float2 [S][hq][n_parts]
    float *out;             // float32 [S][hq][d]
    int32_t *status;
    uint32_t n_seqs, hq, hkv, d, block_size;
    uint32_t part_tokens, n_parts, direct, n_ctas;
    uint64_t k_row_bytes, v_row_bytes;
    int32_t *counters;      // fused merge: per-sequence completion counters, or null
    uint32_t q_tokens;      // query tokens per sequence; n_seqs counts query rows
    uint32_t n_direct;      // leading rows decoded directly in a partitioned plan; the
                            // partials, counters and merges index row r at r - n_direct
    uint32_t merge_no_wait; // PA_FLAG_MERGE_NO_WAIT: cooperative merges give up waiting
    uint32_t stream;        // a stream plan: CTA c takes tiles [c, c + 1) * part_tokens / 16
    uint32_t multi;         // a multi-token plan: a CTA takes a sequence's T query rows
};

// The argument checks of pa_decode_partial alone: PA_OK, or the error
// already recorded for `entry`.  Launches nothing.
int check_decode(const pa_decode_args *a, const pa_plan_t *plan, const char *entry);

// Launchers (each returns PA_OK or an error already recorded for `entry`).
// Copies `bytes` (a multiple of 16) from src_dev, a device-mapped host
// buffer, to dst on the stream, as a grid that lets the next grid be
// scheduled at once and completes after the previous grid (k_plain.cu).
int launch_stage_q(const void *src_dev, void *dst, size_t bytes, cudaStream_t st,
                   const char *entry);
int launch_quantize_q(const float *q, void *q8_1, uint32_t n_rows, uint32_t d,
                      cudaStream_t st, const char *entry);
int launch_plain_decode(const DecodeParams &p, pa_type kt, pa_type vt, cudaStream_t st,
                        const char *entry);
int plain_decode_occupancy(pa_type kt, pa_type vt, uint32_t d, uint32_t hq, int *ctas_per_sm);
int launch_merge(const void *part_o, const float *part_ml, const int32_t *seq_lens, float *out,
                 uint32_t n_seqs, uint32_t q_tokens, uint32_t hq, uint32_t d, uint32_t n_parts,
                 uint32_t part_tokens, uint32_t n_direct, cudaStream_t st, const char *entry);
int launch_append(const pa_append_args *a, cudaStream_t st, const char *entry);
int launch_debug_offsets(const int32_t *block_table, uint32_t table_stride,
                         const int32_t *seq_lens, uint32_t n_seqs, uint32_t max_tokens,
                         uint32_t block_size, uint32_t hkv, uint64_t row_bytes,
                         uint64_t n_pool_blocks, uint64_t *offsets, int32_t *status,
                         cudaStream_t st, const char *entry);

// The fast sm_103a kernel: whether it handles these shapes, its occupancy,
// and its launcher.
bool fast_decode_supported(pa_type kt, pa_type vt, uint32_t d, uint32_t hq, uint32_t hkv,
                           uint32_t block_size);
int fast_decode_occupancy(pa_type kt, pa_type vt, uint32_t d, uint32_t hq, uint32_t hkv,
                          uint32_t block_size, int *ctas_per_sm);
int launch_fast_decode(const DecodeParams &p, pa_type kt, pa_type vt, cudaStream_t st,
                       const char *entry);
// Whether the multi-token kernel serves these shapes with T query tokens.
bool mt_decode_supported(pa_type kt, pa_type vt, uint32_t d, uint32_t hq, uint32_t hkv,
                         uint32_t T);
// The mixed K x V type instances of the fast kernel (D = 256).
bool fast_mixed_supported(pa_type kt, pa_type vt, uint32_t hkv);
int fast_mixed_occupancy(pa_type kt, pa_type vt, uint32_t hkv, int *ctas_per_sm);
int launch_fast_mixed(const DecodeParams &p, pa_type kt, pa_type vt, cudaStream_t st,
                      const char *entry);

}  // namespace pa

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
struct DecodeParams {
    const uint8_t *k_pool, *v_pool;
    uint64_t n_pool_blocks;
    const int32_t *block_table;
    uint32_t table_stride;
    const int32_t *seq_lens;
    const void *q;          // float32 [S][hq][d] (F16 K) or q8_1 blocks
    float scale_log2;       // scale * log2(e)
    void *part_o;           // f16 [S][hq][n_parts][d]
    float *part_ml;         // float2 [S][hq][n_parts]
    float *out;             // float32 [S][hq][d]
    int32_t *status;
    uint32_t n_seqs, hq, hkv, d, block_size;
    uint32_t part_tokens, n_parts, direct, n_ctas;
    uint64_t k_row_bytes, v_row_bytes;
    int32_t *counters;      // fused merge: per-sequence completion counters, or null
};

// Launchers (each returns PA_OK or an error already recorded for `entry`).
int launch_quantize_q(const float *q, void *q8_1, uint32_t n_rows, uint32_t d,
                      cudaStream_t st, const char *entry);
int launch_plain_decode(const DecodeParams &p, pa_type kt, pa_type vt, cudaStream_t st,
                        const char *entry);
int plain_decode_occupancy(pa_type kt, pa_type vt, uint32_t d, uint32_t hq, int *ctas_per_sm);
int launch_merge(const void *part_o, const float *part_ml, const int32_t *seq_lens, float *out,
                 uint32_t n_seqs, uint32_t hq, uint32_t d, uint32_t n_parts,
                 uint32_t part_tokens, cudaStream_t st, const char *entry);
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

}  // namespace pa

// k_plain.cu -- the q8_1 pre-pass, the plain decode kernel, the merge and the
// debug row-offset kernel.
//
// The plain decode kernel is the simple, general form of the method: one warp
// per query head, one token per lane for the scores of a 32-token tile, an
// online softmax in the log2 domain, and D/32 output dimensions per lane for
// the PV accumulation.  It serves every supported shape and type and is the
// second implementation that the fast kernel is checked against.
#include <cuda_fp16.h>
#include <math.h>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

// ------------------------------------------------------------ q8_1 pre-pass
// "feat: add paged-attention monolithic decode-only AR foundation" (lucebox
// pull 555), Summary: Q is quantised once per step by a pre-pass.  One warp
// per block of 32 values; every step in float32 with IEEE division and
// roundf (ties away from zero).
__global__ void __launch_bounds__(256) quantize_q8_1_kernel(const float *__restrict__ x,
                                                            uint8_t *__restrict__ out,
                                                            uint64_t n_blocks)
{
    const int lane = threadIdx.x & 31;
    const uint64_t warps = (uint64_t)gridDim.x * (blockDim.x >> 5);
    for (uint64_t b = (uint64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); b < n_blocks;
         b += warps) {
        const float v = x[b * 32 + lane];
        const float amax = warp_max(fabsf(v));
        float d = amax / 127.0f;
        const int q = q8_1_code(v, amax, d, 1.0f / d);
        const int sum = warp_sum_int(q);
        if (amax == 0.0f)
            d = 0.0f;
        uint8_t *blk = out + b * 36;
        blk[4 + lane] = (uint8_t)(int8_t)q;
        if (lane == 0) {
            reinterpret_cast<uint16_t *>(blk)[0] = __half_as_ushort(__float2half_rn(d));
            reinterpret_cast<uint16_t *>(blk)[1] =
                __half_as_ushort(__float2half_rn(d * (float)sum));
        }
    }
}

int launch_quantize_q(const float *q, void *q8_1, uint32_t n_rows, uint32_t d, cudaStream_t st,
                      const char *entry)
{
    uint64_t n_blocks = (uint64_t)n_rows * (d / 32);
    if (n_blocks == 0)
        return PA_OK;
    uint64_t want = (n_blocks + 7) / 8;
    unsigned grid = (unsigned)(want < 65535 * 16 ? want : 65535 * 16);
    quantize_q8_1_kernel<<<grid, 256, 0, st>>>(q, static_cast<uint8_t *>(q8_1), n_blocks);
    return cuda_check(cudaGetLastError(), entry, "quantize_q8_1_kernel launch");
}

// -------------------------------------------------------- query staging
//
// The query of a host-buffer step, read from page-locked host memory that the
// device maps and written to the device query buffer.  The grid lets the next
// grid on the stream (the decode) be scheduled at once, copies, and then waits
// for the previous grid on the stream before it completes, so the decode,
// which waits for this grid before it reads anything, comes after both.  It
// may run while the previous grid finishes, once that grid allows its
// dependents to be scheduled; this library's kernels do so only after their
// last read of the query.  One warp per CTA and few registers, so that its
// CTAs fit beside a decode CTA on an SM.
__global__ void __maxnreg__(32) stage_query_kernel(const uint4 *__restrict__ src,
                                                   uint4 *__restrict__ dst, uint32_t n16)
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const uint32_t stride = gridDim.x * 32u;
    uint32_t i = blockIdx.x * 32u + threadIdx.x;
    for (; i + 3 * stride < n16; i += 4 * stride) {
        const uint4 a = src[i], b = src[i + stride], c = src[i + 2 * stride],
                    e = src[i + 3 * stride];
        dst[i] = a;
        dst[i + stride] = b;
        dst[i + 2 * stride] = c;
        dst[i + 3 * stride] = e;
    }
    for (; i < n16; i += stride)
        dst[i] = src[i];
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

int launch_stage_q(const void *src_dev, void *dst, size_t bytes, cudaStream_t st,
                   const char *entry)
{
    if (bytes == 0)
        return PA_OK;
    if ((bytes & 15u) || bytes / 16 > 0xffffffffull ||
        (reinterpret_cast<uintptr_t>(src_dev) & 15u) || (reinterpret_cast<uintptr_t>(dst) & 15u))
        return fail(PA_ERR_INVALID, entry, "query staging needs 16-byte sizes and addresses");
    const uint32_t n16 = (uint32_t)(bytes / 16);
    const uint32_t want = (n16 + 127) / 128;  // four 16-byte loads per thread in flight
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(want < 1024 ? want : 1024);
    cfg.blockDim = dim3(32);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cuda_check(cudaLaunchKernelEx(&cfg, stage_query_kernel,
                                         static_cast<const uint4 *>(src_dev),
                                         static_cast<uint4 *>(dst), n16),
                      entry, "stage_query_kernel launch");
}

// ------------------------------------------------------------ plain decode

template <int T>
struct Row;

template <>
struct Row<PA_F16> {
    __host__ __device__ static constexpr int kQBytes(int D) { return D * 4; }
    __device__ static void stage_q(const DecodeParams &p, uint32_t s, uint32_t h, uint8_t *sm,
                                   int lane)
    {
        const float *q = static_cast<const float *>(p.q) + ((uint64_t)s * p.hq + h) * p.d;
        float *qs = reinterpret_cast<float *>(sm);
        for (uint32_t i = lane; i < p.d; i += 32)
            qs[i] = q[i];
    }
    // scale-free dot product of the staged query with one K row
    template <int D>
    __device__ static float dot(const uint8_t *sm, const uint8_t *row)
    {
        const float *qs = reinterpret_cast<const float *>(sm);
        const uint2 *r = reinterpret_cast<const uint2 *>(row);
        float acc = 0.0f;
#pragma unroll 4
        for (int i = 0; i < D / 4; ++i) {
            uint2 w = r[i];
            float2 a = __half22float2(*reinterpret_cast<__half2 *>(&w.x));
            float2 b = __half22float2(*reinterpret_cast<__half2 *>(&w.y));
            acc = fmaf(qs[4 * i + 0], a.x, acc);
            acc = fmaf(qs[4 * i + 1], a.y, acc);
            acc = fmaf(qs[4 * i + 2], b.x, acc);
            acc = fmaf(qs[4 * i + 3], b.y, acc);
        }
        return acc;
    }
    // this lane's D/32 consecutive values of one V row
    template <int D>
    __device__ static void value(const uint8_t *row, int lane, float *v)
    {
        constexpr int DPL = D / 32;
        const __half *r = reinterpret_cast<const __half *>(row) + lane * DPL;
#pragma unroll
        for (int k = 0; k < DPL; ++k)
            v[k] = __half2float(r[k]);
    }
};

// q8_1 staging shared by the quantised-K rows: int8 q[D] then float dq[D/32].
__device__ inline void stage_q8_1(const DecodeParams &p, uint32_t s, uint32_t h, uint8_t *sm,
                                  int lane)
{
    const uint32_t nb = p.d / 32;
    const uint8_t *src =
        static_cast<const uint8_t *>(p.q) + ((uint64_t)s * p.hq + h) * nb * 36;
    int8_t *qs = reinterpret_cast<int8_t *>(sm);
    float *dq = reinterpret_cast<float *>(sm + p.d);
    for (uint32_t i = lane; i < p.d; i += 32)
        qs[i] = (int8_t)src[(i / 32) * 36 + 4 + (i % 32)];
    for (uint32_t b = lane; b < nb; b += 32)
        dq[b] = half_bits_to_float(load_u16(src + b * 36));
}

template <>
struct Row<PA_Q8_0> {
    __host__ __device__ static constexpr int kQBytes(int D) { return D + D / 32 * 4; }
    __device__ static void stage_q(const DecodeParams &p, uint32_t s, uint32_t h, uint8_t *sm,
                                   int lane)
    {
        stage_q8_1(p, s, h, sm, lane);
    }
    template <int D>
    __device__ static float dot(const uint8_t *sm, const uint8_t *row)
    {
        const int8_t *qs = reinterpret_cast<const int8_t *>(sm);
        const float *dq = reinterpret_cast<const float *>(sm + D);
        float acc = 0.0f;
        for (int b = 0; b < D / 32; ++b) {
            const uint8_t *blk = row + 34 * b;
            const float dk = half_bits_to_float(load_u16(blk));
            int isum = 0;
#pragma unroll
            for (int j = 0; j < 32; ++j)
                isum += (int)qs[32 * b + j] * (int)(int8_t)blk[2 + j];
            acc = fmaf((float)isum, dk * dq[b], acc);
        }
        return acc;
    }
    template <int D>
    __device__ static void value(const uint8_t *row, int lane, float *v)
    {
        constexpr int DPL = D / 32;
        const int i0 = lane * DPL;
        const uint8_t *blk = row + 34 * (i0 / 32);
        const float d = half_bits_to_float(load_u16(blk));
#pragma unroll
        for (int k = 0; k < DPL; ++k)
            v[k] = (float)(int8_t)blk[2 + (i0 % 32) + k] * d;
    }
};

template <>
struct Row<PA_Q4_0> {
    __host__ __device__ static constexpr int kQBytes(int D) { return D + D / 32 * 4; }
    __device__ static void stage_q(const DecodeParams &p, uint32_t s, uint32_t h, uint8_t *sm,
                                   int lane)
    {
        stage_q8_1(p, s, h, sm, lane);
    }
    template <int D>
    __device__ static float dot(const uint8_t *sm, const uint8_t *row)
    {
        const int8_t *qs = reinterpret_cast<const int8_t *>(sm);
        const float *dq = reinterpret_cast<const float *>(sm + D);
        float acc = 0.0f;
        for (int b = 0; b < D / 32; ++b) {
            const uint8_t *blk = row + 18 * b;
            const float dk = half_bits_to_float(load_u16(blk));
            int isum = 0;
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const int byte = blk[2 + j];
                isum += (int)qs[32 * b + j] * ((byte & 15) - 8);
                isum += (int)qs[32 * b + 16 + j] * ((byte >> 4) - 8);
            }
            acc = fmaf((float)isum, dk * dq[b], acc);
        }
        return acc;
    }
    template <int D>
    __device__ static void value(const uint8_t *row, int lane, float *v)
    {
        constexpr int DPL = D / 32;
        const int i0 = lane * DPL;
        const uint8_t *blk = row + 18 * (i0 / 32);
        const float d = half_bits_to_float(load_u16(blk));
#pragma unroll
        for (int k = 0; k < DPL; ++k) {
            const int j = (i0 % 32) + k;
            const int nib = j < 16 ? (blk[2 + j] & 15) : (blk[2 + j - 16] >> 4);
            v[k] = (float)(nib - 8) * d;
        }
    }
};

constexpr int kPlainWarps = 16;

template <int KT, int VT, int D>
__global__ void __launch_bounds__(kPlainWarps * 32) plain_decode_kernel(const DecodeParams p)
{
    constexpr int DPL = D / 32;
    constexpr int QB = Row<KT>::kQBytes(D);
    extern __shared__ __align__(16) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nwarps = blockDim.x >> 5;
    uint8_t *qsm = smem + warp * ((QB + 15) / 16 * 16);

    uint32_t s, part;
    if (!p.direct && blockIdx.x == gridDim.x - 1 && warp == 0)
        check_grid_vs_plan(p.seq_lens, p.q_tokens, p.n_seqs, p.part_tokens, p.n_parts,
                           p.n_direct, p.status);
    if (p.direct) {
        s = blockIdx.x;
        part = 0;
        if (s >= p.n_seqs)
            return;
    } else if (!cta_work(p.seq_lens, p.q_tokens, p.n_seqs, p.part_tokens, p.n_parts,
                         p.n_direct, blockIdx.x, &s, &part)) {
        return;
    } else if (s >= p.n_direct && part == 0 && threadIdx.x == 0) {
        check_len_vs_plan(row_len(p.seq_lens, p.q_tokens, s), p.n_parts, p.part_tokens,
                          p.status);
    }
    // a direct CTA: the whole row, output written here
    const bool dir = p.direct || s < p.n_direct;
    const int32_t Lrow = row_len(p.seq_lens, p.q_tokens, s);
    const int32_t L = Lrow > 0 ? Lrow : 0;
    const uint32_t t0 = dir ? 0u : part * p.part_tokens;
    const uint32_t t1 = dir ? (uint32_t)L : min((uint32_t)L, t0 + p.part_tokens);
    const int32_t *bt = p.block_table + (uint64_t)table_row(p.q_tokens, s) * p.table_stride;
    const uint32_t G = p.hq / p.hkv;

    for (uint32_t h = warp; h < p.hq; h += nwarps) {
        const uint32_t g = h / G;
        Row<KT>::stage_q(p, s, h, qsm, lane);
        __syncwarp();
        float m = -INFINITY, l = 0.0f;
        float acc[DPL];
#pragma unroll
        for (int k = 0; k < DPL; ++k)
            acc[k] = 0.0f;
        for (uint32_t tile = t0; tile < t1; tile += 32) {
            const uint32_t t = tile + lane;
            bool valid = t < t1;
            int32_t blk = valid ? bt[t / p.block_size] : 0;
            if (valid && !block_in_pool(blk, p.n_pool_blocks)) {
                atomicOr(p.status, PA_STATUS_CORRUPT_TABLE);
                valid = false;
            }
            float s2 = -INFINITY;
            if (valid) {
                const uint8_t *row = p.k_pool + row_offset(blk, t % p.block_size, g, p.block_size,
                                                           p.hkv, p.k_row_bytes);
                s2 = Row<KT>::template dot<D>(qsm, row) * p.scale_log2;
            }
            const float mt = warp_max(s2);
            if (mt == -INFINITY)
                continue;
            const float mn = fmaxf(m, mt);
            const float alpha = exp2f(m - mn);
            const float pv = valid ? exp2f(s2 - mn) : 0.0f;
            l = l * alpha + warp_sum(pv);
#pragma unroll
            for (int k = 0; k < DPL; ++k)
                acc[k] *= alpha;
            m = mn;
            unsigned vm = __ballot_sync(0xffffffffu, valid);
            while (vm) {
                const int j = __ffs(vm) - 1;
                vm &= vm - 1;
                const float pj = __shfl_sync(0xffffffffu, pv, j);
                const int32_t bj = __shfl_sync(0xffffffffu, blk, j);
                const uint32_t tj = tile + j;
                const uint8_t *vrow = p.v_pool + row_offset(bj, tj % p.block_size, g,
                                                            p.block_size, p.hkv, p.v_row_bytes);
                float v[DPL];
                Row<VT>::template value<D>(vrow, lane, v);
#pragma unroll
                for (int k = 0; k < DPL; ++k)
                    acc[k] = fmaf(pj, v[k], acc[k]);
            }
        }
        const float inv = l > 0.0f ? 1.0f / l : 0.0f;
        const uint64_t sh = (uint64_t)s * p.hq + h;
        if (dir) {
            float *o = p.out + sh * D + lane * DPL;
#pragma unroll
            for (int k = 0; k < DPL; ++k)
                o[k] = acc[k] * inv;
        } else {
            // partials of partitioned row s sit at index s - n_direct
            const uint64_t slot = ((uint64_t)(s - p.n_direct) * p.hq + h) * p.n_parts + part;
            __half *o = static_cast<__half *>(p.part_o) + slot * D + lane * DPL;
#pragma unroll
            for (int k = 0; k < DPL; ++k)
                o[k] = __float2half_rn(acc[k] * inv);
            if (lane == 0)
                reinterpret_cast<float2 *>(p.part_ml)[slot] = make_float2(m, l);
        }
        __syncwarp();
    }
    if (p.counters && !dir)
        fused_merge(p, s, part, threadIdx.x >> 5, blockDim.x >> 5);
}

template <int KT, int VT, int D>
static void *plain_fn()
{
    return reinterpret_cast<void *>(&plain_decode_kernel<KT, VT, D>);
}

static void *plain_kernel_ptr(pa_type kt, pa_type vt, uint32_t d)
{
#define PA_PLAIN_CASE(K, V)                                                                   \
    if (kt == K && vt == V)                                                                   \
        return d == 128 ? plain_fn<K, V, 128>() : plain_fn<K, V, 256>();
    PA_PLAIN_CASE(PA_F16, PA_F16)
    PA_PLAIN_CASE(PA_F16, PA_Q8_0)
    PA_PLAIN_CASE(PA_F16, PA_Q4_0)
    PA_PLAIN_CASE(PA_Q8_0, PA_F16)
    PA_PLAIN_CASE(PA_Q8_0, PA_Q8_0)
    PA_PLAIN_CASE(PA_Q8_0, PA_Q4_0)
    PA_PLAIN_CASE(PA_Q4_0, PA_F16)
    PA_PLAIN_CASE(PA_Q4_0, PA_Q8_0)
    PA_PLAIN_CASE(PA_Q4_0, PA_Q4_0)
#undef PA_PLAIN_CASE
    return nullptr;
}

static size_t plain_smem(pa_type kt, uint32_t d, int warps)
{
    size_t qb = kt == PA_F16 ? (size_t)d * 4 : (size_t)d + d / 32 * 4;
    return (qb + 15) / 16 * 16 * warps;
}

static int plain_warps(uint32_t hq) { return hq < (uint32_t)kPlainWarps ? (int)hq : kPlainWarps; }

int plain_decode_occupancy(pa_type kt, pa_type vt, uint32_t d, uint32_t hq, int *ctas_per_sm)
{
    void *fn = plain_kernel_ptr(kt, vt, d);
    if (!fn)
        return PA_ERR_INVALID;
    int w = plain_warps(hq);
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas_per_sm, fn, w * 32,
                                                                  plain_smem(kt, d, w));
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

int launch_plain_decode(const DecodeParams &p, pa_type kt, pa_type vt, cudaStream_t st,
                        const char *entry)
{
    void *fn = plain_kernel_ptr(kt, vt, p.d);
    if (!fn)
        return fail(PA_ERR_INVALID, entry, "no plain kernel for these types / d");
    int w = plain_warps(p.hq);
    void *args[] = {const_cast<DecodeParams *>(&p)};
    cudaError_t e = cudaLaunchKernel(fn, dim3(p.n_ctas), dim3(w * 32), args,
                                     plain_smem(kt, p.d, w), st);
    return cuda_check(e, entry, "plain_decode_kernel launch");
}

// -------------------------------------------------------------------- merge
// Stable split-softmax merge of the stored f16 partials: one warp per
// (sequence, query head) row, the same routine the fused decode uses.
__global__ void __launch_bounds__(128) merge_kernel(const __half *__restrict__ po,
                                                    const float2 *__restrict__ pml,
                                                    const int32_t *__restrict__ seq_lens,
                                                    float *__restrict__ out, uint32_t T,
                                                    uint32_t hq, uint32_t D, uint32_t n_parts,
                                                    uint32_t part_tokens, uint32_t n_direct,
                                                    uint64_t units)
{
    // unit sh: (partitioned row, head) at partial index sh; its row is
    // n_direct + sh / hq (the leading direct rows have no partials)
    const uint64_t sh = (uint64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (sh >= units)
        return;
    const uint64_t osh = sh + (uint64_t)n_direct * hq;  // its output row
    const int32_t L = row_len(seq_lens, T, (uint32_t)(osh / hq));
    uint32_t n_live = L > 0 ? ((uint32_t)L + part_tokens - 1) / part_tokens : 0;
    if (n_live > n_parts)
        n_live = n_parts;
    // this warp's stage for the group results of a two-pass merge
    __shared__ __align__(16) __half scr[4][256];
    __shared__ float2 scr_ml[4];
    const int w = threadIdx.x >> 5;
    if (D == 256)
        merge_row_two_pass_warp<8>(po + sh * n_parts * D, pml + sh * n_parts, out + osh * D,
                                   n_live, D, scr[w], &scr_ml[w]);
    else
        merge_row_two_pass_warp<4>(po + sh * n_parts * D, pml + sh * n_parts, out + osh * D,
                                   n_live, D, scr[w], &scr_ml[w]);
}

int launch_merge(const void *part_o, const float *part_ml, const int32_t *seq_lens, float *out,
                 uint32_t n_seqs, uint32_t q_tokens, uint32_t hq, uint32_t d, uint32_t n_parts,
                 uint32_t part_tokens, uint32_t n_direct, cudaStream_t st, const char *entry)
{
    const uint32_t T = q_tokens > 1 ? q_tokens : 1;
    const uint64_t rows = (uint64_t)n_seqs * T;
    if (n_direct > rows)
        return fail(PA_ERR_INVALID, entry, "n_direct %u exceeds the %llu query rows", n_direct,
                    (unsigned long long)rows);
    uint64_t units = (rows - n_direct) * hq;
    if (units == 0)
        return PA_OK;
    if ((units + 3) / 4 > 0x7fffffffull)
        return fail(PA_ERR_RANGE, entry, "n_seqs * hq too large for the merge grid");
    if (d != 128 && d != 256)
        return fail(PA_ERR_INVALID, entry, "d %u unsupported by the merge (128 or 256)", d);
    merge_kernel<<<(unsigned)((units + 3) / 4), 128, 0, st>>>(
        static_cast<const __half *>(part_o), reinterpret_cast<const float2 *>(part_ml), seq_lens,
        out, T, hq, d, n_parts, part_tokens, n_direct, units);
    return cuda_check(cudaGetLastError(), entry, "merge_kernel launch");
}

// ----------------------------------------------------------- debug offsets

__global__ void debug_offsets_kernel(const int32_t *__restrict__ bt, uint32_t stride,
                                     const int32_t *__restrict__ lens, uint32_t n_seqs,
                                     uint32_t max_tokens, uint32_t B, uint32_t hkv,
                                     uint64_t row_bytes, uint64_t n_pool_blocks,
                                     uint64_t *__restrict__ offsets, int32_t *status)
{
    const uint64_t total = (uint64_t)n_seqs * max_tokens * hkv;
    for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (uint64_t)gridDim.x * blockDim.x) {
        const uint32_t g = (uint32_t)(i % hkv);
        const uint32_t t = (uint32_t)((i / hkv) % max_tokens);
        const uint32_t s = (uint32_t)(i / ((uint64_t)hkv * max_tokens));
        uint64_t off = ~0ull;
        if ((int32_t)t < lens[s]) {
            const int32_t blk = bt[(uint64_t)s * stride + t / B];
            if (block_in_pool(blk, n_pool_blocks))
                off = row_offset(blk, t % B, g, B, hkv, row_bytes);
            else
                atomicOr(status, PA_STATUS_CORRUPT_TABLE);
        }
        offsets[i] = off;
    }
}

int launch_debug_offsets(const int32_t *block_table, uint32_t table_stride,
                         const int32_t *seq_lens, uint32_t n_seqs, uint32_t max_tokens,
                         uint32_t block_size, uint32_t hkv, uint64_t row_bytes,
                         uint64_t n_pool_blocks, uint64_t *offsets, int32_t *status,
                         cudaStream_t st, const char *entry)
{
    uint64_t total = (uint64_t)n_seqs * max_tokens * hkv;
    if (total == 0)
        return PA_OK;
    uint64_t want = (total + 255) / 256;
    unsigned grid = (unsigned)(want < 1u << 20 ? want : 1u << 20);
    debug_offsets_kernel<<<grid, 256, 0, st>>>(block_table, table_stride, seq_lens, n_seqs,
                                               max_tokens, block_size, hkv, row_bytes,
                                               n_pool_blocks, offsets, status);
    return cuda_check(cudaGetLastError(), entry, "debug_offsets_kernel launch");
}

}  // namespace pa

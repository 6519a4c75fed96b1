/*
 * pa.h -- C ABI of the paged decode-attention library (libpa.so) for GB300.
 *
 * One decode step of attention over a paged K/V cache: for every sequence,
 * one query token per query head attends to that sequence's K/V rows, which
 * are gathered through a per-sequence block table of fixed-size blocks kept
 * in one pool.  Sources (page title + section):
 *
 *  [P1] "feat: add paged-attention monolithic decode-only AR foundation"
 *       (lucebox pull 555): Summary (allocator; the decode op for GQA with
 *       F16/Q4_0/Q8_0 K/V; Q quantised once per step; f16 partials; an
 *       occupancy-aware partition count with a stable split-softmax merge),
 *       Scope (unsupported combinations fail explicitly), Benchmark results
 *       (dead partitions of short sequences), Validation (empty sequences,
 *       page boundaries, shuffled blocks, corrupt block-table bounds guards).
 *  [P4] "fix(paged-attention): use 64-bit pool offsets in the fused decode
 *       kernels" (mlxcel issue 2153): Proposed Solution (the pool offset is
 *       widened to 64 bits before the multiply; tables stay int32; an
 *       oversize launch is refused by name instead of wrapping).
 *
 * Conventions for every call:
 *  - All device memory (pools, Q, q8_1, tables, lengths, partials, output,
 *    status word) is allocated and owned by the caller.  The library never
 *    allocates or frees device memory and never synchronises, except
 *    pa_status_read, which synchronises its stream by design.
 *  - Device pointers are plain pointers into the current device's memory;
 *    every kernel is launched asynchronously on the given stream.
 *  - Return value: PA_OK or a negative PA_ERR_* code.  On failure nothing is
 *    launched and no caller buffer is touched; pa_last_error() then names the
 *    entry point and the reason (thread-local text).  No C++ exception ever
 *    crosses this interface.
 *
 * Data layouts (block = 32 values along the head dimension d):
 *  - F16 row:  d IEEE binary16 values (2*d bytes).
 *  - Q8_0 row: d/32 blocks of 34 bytes: f16 scale, 32 int8; value = q*scale.
 *  - Q4_0 row: d/32 blocks of 18 bytes: f16 scale, 16 bytes of nibbles;
 *    value j < 16 is the low nibble of byte j, value j+16 its high nibble;
 *    value = (nibble - 8) * scale.
 *  - q8_1 row: d/32 blocks of 36 bytes: f16 d, f16 s, 32 int8 q;
 *    value = q * d, s = d * sum(q).
 *  - A pool is token-major bytes [n_blocks][block_size][hkv][row_bytes]; the
 *    row of (block b, slot j, K/V head g) starts at byte
 *    (((uint64_t)b * block_size + j) * hkv + g) * row_bytes.
 *  - Block table: int32 [n_seqs][table_stride]; token t of sequence s lives
 *    in block table[s][t / block_size], slot t % block_size.
 *  - Query head h reads K/V head h / (hq / hkv).
 */
#ifndef PA_H
#define PA_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* The CUDA runtime's stream handle (identical to cudaStream_t); NULL is the
 * legacy default stream. */
typedef struct CUstream_st *pa_stream_t;

/* ------------------------------------------------------------- codes */
#define PA_OK 0
#define PA_ERR_INVALID (-1)       /* bad or unsupported argument */
#define PA_ERR_NOMEM (-2)         /* allocator: request exceeds the free count */
#define PA_ERR_STALE (-3)         /* allocator: bad, stale or duplicate handle */
#define PA_ERR_CUDA (-4)          /* a CUDA runtime call or launch failed */
#define PA_ERR_CORRUPT_TABLE (-5) /* device guard saw a block id outside the pool */
#define PA_ERR_RANGE (-6)         /* a size beyond a documented limit */
#define PA_ERR_TIMEOUT (-7)       /* a kernel gave up a bounded wait (see pa_status_read) */

/* Device status word bits (written by the kernels with atomicOr). */
#define PA_STATUS_CORRUPT_TABLE 1 /* a block id outside [0, n_pool_blocks) */
#define PA_STATUS_TIMEOUT 2       /* a pipeline wait exceeded its bound (2 s); output invalid */
#define PA_STATUS_LEN_OVER_PLAN 4 /* lengths the plan does not cover: a sequence longer than
                                     n_parts * part_tokens, or more (sequence, partition) pairs
                                     than n_ctas; the work past the plan was left out and the
                                     output is invalid */
#define PA_STATUS_APPEND_RANGE 8  /* pa_append_kv: a sequence whose table has no entry left for
                                     its new token (or a negative length); it was left untouched */

typedef enum { PA_F16 = 0, PA_Q8_0 = 1, PA_Q4_0 = 2 } pa_type;

/* Name of a return code ("PA_OK", "PA_ERR_INVALID", ...); never NULL. */
const char *pa_strerror(int code);
/* Text of the last failure on this thread: "<entry point>: <reason>". */
const char *pa_last_error(void);
/* Bytes of one K or V row of d values of the given type; 0 if unsupported. */
uint64_t pa_row_bytes(pa_type type, uint32_t d);

/* ------------------------------------------------------- allocator
 * [P1] Summary: an exact pool of fixed-size blocks; allocation is
 * transactional, stale handles are detected, release is immediate.
 * Host-only; the object is owned by the library (create/destroy) and is not
 * thread-safe (one owner thread, or external locking).
 * Policy: ids 0..n-1 on a LIFO free stack (a fresh pool hands out 0, 1, 2,
 * ...).  A handle is (generation << 32) | block id; generations start at 1,
 * advance by one on release and skip 0 on wrap, so 0 is never a valid
 * handle. */
typedef uint64_t pa_handle;
typedef struct pa_pool pa_pool;

/* n_blocks in [1, 2^31 - 1].  *out receives the pool.  PA_ERR_INVALID on a
 * bad count or NULL out; PA_ERR_NOMEM if host memory runs out. */
int pa_pool_create(uint32_t n_blocks, pa_pool **out);
void pa_pool_destroy(pa_pool *pool);
/* All or nothing: n handles into out[0..n), or PA_ERR_NOMEM with the pool
 * and out untouched when n exceeds the free count.  n == 0 is a no-op. */
int pa_pool_alloc(pa_pool *pool, uint32_t n, pa_handle *out);
/* Validates every handle first (id in range, block live, generation current,
 * no handle listed twice); any failure returns PA_ERR_STALE and releases
 * nothing.  Otherwise releases them in order; each block is reusable at
 * once and the last one released is the next one handed out. */
int pa_pool_free(pa_pool *pool, uint32_t n, const pa_handle *handles);
/* The int32 block id to write into a block table. */
int32_t pa_handle_block(pa_handle h);
uint32_t pa_pool_free_count(const pa_pool *pool);
uint32_t pa_pool_capacity(const pa_pool *pool);

/* ------------------------------------------------------- Q pre-pass
 * [P1] Summary: Q is quantised once per step by a pre-pass, and the
 * quantised-K dot products use it.  q: float32 [n_rows][d] (device);
 * q8_1: n_rows * d/32 blocks of 36 bytes (device).  Per block of 32, in
 * float32: amax = max|x|, d = amax / 127, q = clamp(roundf(x / d), -127,
 * 127) (IEEE division, ties away from zero), d = q = 0 for an all-zero
 * block; stores f16_rn(d) and f16_rn(d * sum(q)).  Inputs must be finite.
 * d must be a multiple of 32; n_rows == 0 is a no-op.
 * PA_ERR_INVALID / PA_ERR_CUDA. */
int pa_quantize_q(const float *q, void *q8_1, uint32_t n_rows, uint32_t d, pa_stream_t stream);

/* ------------------------------------------------------- planner
 * [P1] Summary and Benchmark results: occupancy-aware context partitioning;
 * dead partitions of short sequences are sized by the longest one, so this
 * rule sizes partitions by the total live work instead.  The rule (pure
 * integer function, host only):
 *  - partitions are multiples of 32 tokens;
 *  - force_parts > 0: part_tokens = roundup(ceil(max_len / force_parts), 32);
 *  - else part_tokens = roundup(ceil(total_len / (sm_count * ctas_per_sm)),
 *    32), clamped to [128, roundup(max_len, 32)]; a nearly uniform batch
 *    (10 * total_len >= 9 * n_seqs * max_len) with n_seqs <= slots whose
 *    n_seqs * ceil(max_len / part_tokens) would exceed the slots takes
 *    roundup(ceil(max_len / floor(slots / n_seqs)), 32) instead, within the
 *    same bounds (one wave of CTAs); then any plan of more than one
 *    partition per sequence with n_seqs < slots whose grid bound (n_ctas
 *    below) would exceed the slots takes part_tokens =
 *    roundup(ceil(total_len / (slots - n_seqs)), 32) if that is larger (at
 *    most roundup(max_len, 32)), so that the grid fits one wave;
 *  - n_parts = ceil(max_len / part_tokens); direct = (n_parts == 1): no
 *    partials, the decode kernel writes the output;
 *  - a batch wider than the machine (n_seqs > slots) that this makes direct,
 *    with n_seqs = k * slots + r and 0 < r, may fill its last wave instead:
 *    the first n_direct = k * slots sequences stay direct (one CTA each,
 *    output written by the decode kernel) and the last r are split into
 *    n_parts >= 2 partitions of part_tokens = max(128, roundup(ceil(max_len
 *    / np), 32)), where np in 2..64 minimises ceil(r * n_parts / slots) *
 *    (part_tokens + 512), the estimated time of those waves (512 tokens
 *    stand for a CTA's fixed work), if that is below max_len + 512 (the
 *    first minimum wins); direct = 0.  Every other plan has n_direct = 0;
 *  - n_ctas = n_seqs when direct, else n_direct + min(m * n_parts,
 *    ceil(total_len / part_tokens) + m) with m = n_seqs - n_direct (>= the
 *    live partitions; a wave-filling plan counts m * n_parts);
 *  - partial buffers, for the m partitioned sequences only (sequence s at
 *    index s - n_direct): part_o f16 [m][hq][n_parts][d] and part_ml
 *    float32 [m][hq][n_parts][2] (0 bytes when direct);
 *  - counter_bytes = 4 * m * (1 + ceil(sqrt(n_parts))), the int32
 *    completion counters of the fused merge (0 when direct).
 * Several query tokens ([P2] What: a prompt chunk or a verify window of
 * several query rows per sequence over one paged cache): with q_tokens = T,
 * query token i of sequence s sits at position L_s - T + i and attends to the
 * keys 0 .. L_s - T + i.  The rule then runs over the n_seqs * T query rows
 * (row u = s * T + i, of length L_s - T + 1 + i) with T * total_len tokens of
 * work: every n_seqs above reads n_seqs * T and total_len reads T * total_len;
 * max_len and n_parts are per row.
 * Stream plans ("feat: add paged-attention monolithic decode-only AR
 * foundation", lucebox pull 555, Roadmap: stream-K decode): with
 * PA_PLAN_STREAM_OK in flags, force_parts = 0, more query rows than slots,
 * k_type == v_type, hkv in {1, 2, 4, 8} and d = 256 (or F16 K/V), the grid
 * takes equal ranges of the rows' 16-token tiles instead of whole rows or
 * partitions: with B = ceil((T * total_len + 15 * rows) / 16) (a bound on
 * the tiles), chunk = roundup(ceil(B / slots), 2) tiles, part_tokens =
 * 16 * chunk, n_ctas = min(slots, ceil(B / chunk)), n_parts = ceil(ceil(
 * max_len / 16) / chunk) + 1 (the most CTAs one row can span), stream = 1,
 * direct = 0, n_direct = 0, partial buffers and counters for every row
 * (m = rows below), if n_parts <= 32 and rows <= 16384; else the rules above.
 * Multi-token plans ([P2] What: a verify window or prompt chunk as several
 * query rows over one paged cache): with PA_PLAN_MULTI_TOKEN in flags,
 * q_tokens = T >= 2, Q4_0 K and V, d = 256, hkv in {1, 2, 4} and T * hq /
 * hkv <= 24, the plan is the one-token plan of the n_seqs sequences (the
 * rules above with q_tokens = 1; a plan that would keep direct rows becomes
 * direct), with multi = 1, q_tokens = T, and the partial buffers and
 * counters of the n_seqs * T query rows: one CTA takes one partition of a
 * sequence for all its T tokens, whose partials pa_merge merges per row.
 * Limits: block_size 16 or 32, d 128 or 256, hq a multiple of hkv with
 * hq / hkv <= 8, total_len <= n_seqs * max_len.  PA_ERR_INVALID otherwise. */
typedef struct {
    uint32_t n_seqs, max_len;
    uint64_t total_len;          /* sum of the sequence lengths */
    uint32_t block_size, hq, hkv, d;
    pa_type k_type, v_type;
    int32_t sm_count, ctas_per_sm;
    int32_t force_parts;         /* 0 = automatic */
    uint32_t q_tokens;           /* query tokens per sequence (0 or 1: one; see below) */
    uint32_t flags;              /* PA_PLAN_* */
} pa_plan_in;

/* pa_plan_in.flags: the plan may be a stream plan (see below); only
 * pa_decode_fused and pa_decode_step_fused on the fast kernel run those. */
#define PA_PLAN_STREAM_OK 1u
/* pa_plan_in.flags: with q_tokens = T >= 2, decode the T query tokens of a
 * sequence together (see below); the fast kernel runs those plans. */
#define PA_PLAN_MULTI_TOKEN 2u

typedef struct {
    uint32_t part_tokens, n_parts, direct, n_ctas;
    uint64_t part_o_bytes, part_ml_bytes;
    uint64_t counter_bytes;      /* completion counters of pa_decode_fused (0 when direct) */
    uint32_t q_tokens;           /* query tokens per sequence (>= 1) */
    uint32_t n_direct;           /* leading query rows decoded directly in a partitioned plan */
    uint32_t stream;             /* 1: a stream plan (equal tile ranges per CTA) */
    uint32_t multi;              /* 1: a multi-token plan (the T tokens of a sequence together) */
} pa_plan_t;

/* With the environment variable PA_LOG_PLAN set (to anything but "" or
 * "0"), every successful pa_plan also writes one line with its inputs and
 * the chosen plan to stderr. */
int pa_plan(const pa_plan_in *in, pa_plan_t *out);
/* Fills sm_count and ctas_per_sm of the current device for the decode
 * kernel that pa_decode_partial would choose for these shapes.
 * PA_ERR_INVALID / PA_ERR_CUDA. */
int pa_query_occupancy(const pa_plan_in *in, int32_t *sm_count, int32_t *ctas_per_sm);

/* ------------------------------------------------------- decode
 * [P1] Summary / [P4] Proposed Solution.  For sequence s of length L_s and
 * query head h (g = h / (hq/hkv)): scores s_t = scale * <Qhat_h, Khat_t,g>
 * over t < L_s, p = softmax(s), O[s][h] = sum_t p_t * Vhat_t,g.  Qhat is
 * the float32 query for F16 K and the q8_1 row otherwise; Khat / Vhat are
 * the dequantised rows.  L_s == 0 gives O = 0.  Only the first
 * ceil(L_s / block_size) table entries of a sequence and only slots < L_s
 * are read.
 * Partitioned plans write, for each live partition p of each (s, h),
 * part_o[s][h][p][:] = (sum over the partition of 2^(s2_t - m) V_t) / l in
 * f16 and part_ml[s][h][p] = (m, l), where s2_t = s_t * log2(e), m is the
 * partition maximum of s2_t and l = sum 2^(s2_t - m); pa_merge then forms
 * O.  Direct plans write out directly and touch no partial.  A wave-filling
 * plan (plan->n_direct > 0) writes out directly for its first n_direct
 * query rows and partials for the others, at row index s - n_direct.
 * Stream plans run only through pa_decode_fused and pa_decode_step_fused on
 * the fast kernel (PA_ERR_INVALID here and in pa_merge and pa_decode_step).
 * A block id outside [0, n_pool_blocks) is never dereferenced: the kernel
 * sets PA_STATUS_CORRUPT_TABLE in *status and treats that block's tokens as
 * absent (pa_status_read reports it).  Pool offsets are 64-bit throughout:
 * pools past 2^32 elements are supported.
 * With plan->q_tokens = T > 1 ([P2] What) every sequence has T query tokens:
 * q, out and the partials hold n_seqs * T query rows (row s * T + i, token i
 * of sequence s, at position L_s - T + i, attending to the keys 0 .. L_s - T
 * + i); the block table and lengths stay per sequence.  A row with no key
 * gives O = 0. */
typedef struct {
    const void *k_pool, *v_pool;     /* device, token-major pools, 16-byte aligned */
    uint64_t n_pool_blocks;          /* 1 .. 2^31 */
    const int32_t *block_table;      /* device int32 [n_seqs][table_stride] */
    uint32_t table_stride;
    const int32_t *seq_lens;         /* device int32 [n_seqs], 0 <= L <= table_stride*block_size */
    const void *q;                   /* device: float32 [n_seqs][T][hq][d] for F16 K,
                                        q8_1 [n_seqs][T][hq][d/32] otherwise (T = q_tokens) */
    float scale;                     /* softmax scale; callers pass 1/sqrt(d) */
    void *part_o;                    /* device f16 [n_seqs*T - n_direct][hq][n_parts][d]
                                        (unused if direct) */
    float *part_ml;                  /* device float32 [n_seqs*T - n_direct][hq][n_parts][2] */
    float *out;                      /* device float32 [n_seqs][T][hq][d], 16-byte aligned
                                        (written if direct or fused) */
    int32_t *status;                 /* device int32 status word (required) */
    uint32_t n_seqs, hq, hkv, d, block_size;
    pa_type k_type, v_type;
    uint32_t flags;                  /* PA_FLAG_* */
} pa_decode_args;

/* flags: choose the kernel.  0 = the fast sm_103a kernel where it supports
 * the shapes, else the plain kernel; PA_FLAG_PLAIN forces the plain kernel
 * (one warp per query head, CUDA cores), kept as a second implementation. */
#define PA_FLAG_PLAIN 1u
/* For tests: the cooperative in-launch merge (see pa_decode_fused) gives up
 * waiting at once, so the CTA that completes each count merges the rows of
 * every CTA that stopped waiting.  The output is the same bit for bit. */
#define PA_FLAG_MERGE_NO_WAIT 2u

int pa_decode_partial(const pa_decode_args *args, const pa_plan_t *plan, pa_stream_t stream);

/* Name of the decode kernel pa_decode_partial launches for these shapes and
 * flags ("fast_decode_kernel" or "plain_decode_kernel"); NULL for shapes no
 * kernel supports.  Host only, no device work. */
const char *pa_decode_kernel_name(pa_type k_type, pa_type v_type, uint32_t d, uint32_t hq,
                                  uint32_t hkv, uint32_t block_size, uint32_t flags);

/* Merge ([P1] Summary: stable split-softmax merge).  For each (s, h) with
 * n_live = min(ceil(L_s / part_tokens), n_parts) live partitions: M = max
 * m_p over partitions with l_p > 0, w_p = l_p 2^(m_p - M), out = sum w_p o_p
 * / sum w_p; partitions with l_p == 0 are skipped and no live partition gives
 * 0.  More than 32 live partitions are merged in two passes ([P3] What:
 * hierarchical reduction): groups of gs = ceil(sqrt(n_live)) consecutive
 * partitions are merged into f16 partials of the same form, then those; the
 * same as the flat merge up to rounding.  Reads the partials only.  Layouts
 * as in pa_decode_args; the first plan->n_direct query rows have no
 * partials and their out rows are left as they are.  PA_ERR_INVALID for a
 * direct plan (nothing to merge).  Indexing is 64-bit; PA_ERR_RANGE if the partial buffer exceeds
 * 2^40 elements. */
int pa_merge(const void *part_o, const float *part_ml, const int32_t *seq_lens, float *out,
             uint32_t n_seqs, uint32_t hq, uint32_t d, const pa_plan_t *plan,
             pa_stream_t stream);

/* pa_decode_partial with the merge done inside the same launch ("HRX:
 * multi-pass KV-block reduction for flash-attention decode-split", llama.cpp
 * fork pull 13, Changes: an atomic completion counter lets the reduction run
 * in the decode launch itself, with no second dispatch).  Every CTA writes its
 * partial as pa_decode_partial does and counts it; the CTA that completes a
 * count merges: for a one-pass sequence all its partials into out, for a
 * two-pass one (see pa_merge) its group's partials into the group's first
 * partial slot, and the CTA that completes the last group the group results
 * into out.  The result is pa_merge's bit for bit.  Every count is reset to 0
 * by the CTA that completes it, and no CTA waits for another -- except on the
 * fast kernel, for one-pass plans (n_parts <= 32, n_direct == 0) whose whole
 * grid fits the device at once: there the CTAs of a sequence wait for each
 * other (at most 100 us; an environment variable PA_COOP_MERGE=0 turns this
 * off) and each merges its share of the rows, same bits again; a CTA whose
 * wait runs out leaves its rows to the CTA that completes the count.  The
 * fast kernel is launched with programmatic stream serialisation (off with
 * PA_PDL=0): it may be scheduled while the previous kernel on the stream
 * finishes, and waits for that kernel's completion before it reads any
 * input.
 * counters: device int32 [plan->counter_bytes / 4], caller-owned, all zero
 * before the first call; every completed call leaves them zero.  After a call
 * that reported PA_STATUS_TIMEOUT or PA_STATUS_LEN_OVER_PLAN the caller
 * zeroes them again.  Calls that
 * share a counter array must not overlap on the GPU.  The partials are
 * overwritten by the group results.  Direct plans ignore counters (may be
 * NULL) and behave as pa_decode_partial.  part_o / part_ml / out are required
 * for partitioned plans. */
int pa_decode_fused(const pa_decode_args *args, const pa_plan_t *plan, int32_t *counters,
                    pa_stream_t stream);

/* pa_decode_step with the fused merge, args->q the float32 query.  Where the
 * fast kernel serves the shapes and K is quantised, it quantises the query
 * rows itself with pa_quantize_q's arithmetic (the same q8_1 codes) and the
 * step is one launch; otherwise pa_quantize_q (quantised K) into
 * q8_1_scratch, then pa_decode_fused.  q8_1_scratch (n_seqs*hq*d/32*36 bytes,
 * 16-byte aligned) is required for quantised K either way. */
int pa_decode_step_fused(const pa_decode_args *args, const pa_plan_t *plan, void *q8_1_scratch,
                         int32_t *counters, pa_stream_t stream);

/* One full decode step on the device: pa_quantize_q (quantised K only, into
 * q8_1_scratch of n_seqs*hq*d/32*36 bytes), pa_decode_partial, and pa_merge
 * unless the plan is direct.  args->q must point at the float32 query; the
 * call substitutes q8_1_scratch for the kernel.  Same errors as the parts. */
int pa_decode_step(const pa_decode_args *args, const pa_plan_t *plan, void *q8_1_scratch,
                   pa_stream_t stream);

/* The same step with the query taken from and the output returned to HOST
 * memory: copies q_host (float32 [n_seqs][hq][d]) into args->q (device),
 * runs pa_decode_step, and returns the output in out_host, all on `stream`.
 * When out_host is page-locked memory mapped into the device's address space
 * (cudaHostAlloc / cudaMallocHost under unified addressing, 16-byte aligned),
 * the kernels store the output into it directly and args->out is left
 * untouched; otherwise args->out is copied back into out_host.  Page-locked,
 * mapped q_host (16-byte aligned) is staged into args->q by a small kernel
 * launched with programmatic stream serialisation: it may run while the
 * previous kernel on the stream finishes, once that kernel has let its
 * dependents be scheduled, and it completes only after that kernel, so the
 * decode after it sees both.  A previous kernel that lets its dependents be
 * scheduled must then be done reading args->q (this library's kernels are).
 * Other q_host is copied with cudaMemcpyAsync.  The caller synchronises
 * before reading out_host. */
int pa_decode_step_host(const float *q_host, float *out_host, const pa_decode_args *args,
                        const pa_plan_t *plan, void *q8_1_scratch, pa_stream_t stream);

/* The same device step for callers that cannot allocate device memory.
 * The pages have no counterpart to this call; it exists for users of this
 * library whose code may not call cudaMalloc at decode time (for example a
 * component that runs inside a host callback, or a serving engine whose
 * memory is owned by another allocator or capped by a fixed budget) and so
 * cannot supply the q8_1 and partial buffers that pa_decode_step takes.
 * Here that scratch lives in one static device array of the library,
 * PA_NOALLOC_SCRATCH_BYTES long, which every GPU that loads the library
 * holds until the process exits.  The caller still passes every input and
 * output in *args (pools, table, lengths, the float32 query in args->q, out
 * and the status word); args->part_o and args->part_ml are ignored.
 *  - The first call on a device looks up the array's device address with
 *    that device current (cudaGetSymbolAddress); later calls reuse it while
 *    the device keeps the same context (a context made again, after
 *    cudaDeviceReset say, is looked up afresh).  Make the first call on a
 *    device before any stream capture.
 *  - Every argument is checked before anything is launched, as for
 *    pa_decode_step.
 *  - A step whose scratch (q8_1 rows plus partials, each rounded up to 256
 *    bytes) exceeds PA_NOALLOC_SCRATCH_BYTES is refused with PA_ERR_RANGE
 *    and the size it would need; nothing is launched.
 *  - No allocation happens: no cudaMalloc, cudaFree or allocating routine.
 *  - Every call shares the one array and finds the previous call's bytes in
 *    it; nothing in it needs to start at zero.  Calls whose kernels overlap
 *    on the GPU (different streams, or different host threads without
 *    ordering) race on the array: order them on one stream.
 * Errors as pa_decode_step. */
#define PA_NOALLOC_SCRATCH_BYTES (16ull << 20)
int pa_decode_step_noalloc(const pa_decode_args *args, const pa_plan_t *plan,
                           pa_stream_t stream);

/* pa_decode_step_host with the fused merge: host q in, host out back, with
 * pa_decode_step_fused in between, all on `stream`. */
int pa_decode_step_fused_host(const float *q_host, float *out_host, const pa_decode_args *args,
                              const pa_plan_t *plan, void *q8_1_scratch, int32_t *counters,
                              pa_stream_t stream);

/* ------------------------------------------------------- K/V append
 * The step before the decode ([P1] Summary: the paging metadata -- block
 * table and sequence lengths -- stays resident on the device next to the
 * pool, and a decode step uploads only the 4-byte id of each fresh 16-token
 * block; [P1] Validation: prefill through many block boundaries).  For each
 * sequence s, with L = seq_lens[s] read on the device: the new token's K and
 * V rows of every K/V head are quantised to the pool's row format and
 * written at slot L % B of block table[s][L / B], and seq_lens[s] becomes
 * L + 1.  When L % B == 0 the token starts a block: the call takes
 * fresh_blocks[s] (allocated by the caller, e.g. pa_pool_alloc) and writes it
 * into table[s][L / B]; fresh_blocks is read for no other sequence.
 * Quantisers (float32, no contracted multiply-add; the ggml convention):
 * Q8_0 d = amax/127, q = clamp(roundf(x * (1/d)), +-127); Q4_0 m = the first
 * value of largest magnitude, d = m / -8, nib = min(15, floor(x * (1/d) +
 * 8.5)); F16 round to nearest even; scales stored as f16 (nearest even).
 * A sequence whose table has no entry L / B (L / B >= table_stride) sets
 * PA_STATUS_APPEND_RANGE, one whose block id is outside [0, n_pool_blocks)
 * sets PA_STATUS_CORRUPT_TABLE; either is left untouched (rows, table,
 * length).  One launch; everything device memory on `stream`.
 * PA_ERR_INVALID for bad arguments (checked before any launch). */
typedef struct {
    void *k_pool, *v_pool;           /* device pools, as in pa_decode_args, 16-byte aligned */
    uint64_t n_pool_blocks;          /* 1 .. 2^31 */
    int32_t *block_table;            /* device int32 [n_seqs][table_stride], updated in place */
    uint32_t table_stride;
    int32_t *seq_lens;               /* device int32 [n_seqs], incremented in place */
    const float *k_new, *v_new;      /* device float32 [n_seqs][hkv][d], 16-byte aligned */
    const int32_t *fresh_blocks;     /* device int32 [n_seqs] (see above) */
    int32_t *status;                 /* device int32 status word (required) */
    uint32_t n_seqs, hkv, d, block_size;
    pa_type k_type, v_type;
} pa_append_args;

int pa_append_kv(const pa_append_args *args, pa_stream_t stream);

/* Reads the status word into *host_out (synchronising `stream`); reset != 0
 * clears it afterwards.  Returns PA_ERR_TIMEOUT if the timeout bit is set,
 * else PA_ERR_RANGE if the lengths-over-plan or the append-range bit is set,
 * else PA_ERR_CORRUPT_TABLE if the corrupt-table bit is set, PA_OK
 * otherwise, PA_ERR_CUDA on a runtime failure. */
int pa_status_read(int32_t *dev_status, pa_stream_t stream, int32_t *host_out, int reset);

/* Debug ([P4] Acceptance Criteria: the offsets must be 64-bit).  Writes the
 * byte offset of every row the decode step reads into offsets, a device
 * uint64 array [n_seqs][max_tokens][hkv]: entry (s, t, g) for t < L_s is the
 * offset of that row in a pool of row_bytes-sized rows, computed by the same
 * device routine the decode kernels use; other entries are UINT64_MAX.
 * Out-of-pool block ids also give UINT64_MAX and set PA_STATUS_CORRUPT_TABLE. */
int pa_debug_row_offsets(const int32_t *block_table, uint32_t table_stride,
                         const int32_t *seq_lens, uint32_t n_seqs, uint32_t max_tokens,
                         uint32_t block_size, uint32_t hkv, uint64_t row_bytes,
                         uint64_t n_pool_blocks, uint64_t *offsets, int32_t *status,
                         pa_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* PA_H */

// pa_api.cu -- device-side entry points of the C ABI: argument validation,
// kernel selection and launch glue.  Every check runs before anything is
// launched, so a refused call touches no caller buffer.
#include <math.h>

#include "pa_internal.h"

using pa::cuda_check;
using pa::fail;

namespace {

bool type_ok(pa_type t) { return (unsigned)t <= 2u; }

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_plan(const pa_plan_t *plan, const char *E)
{
    if (!plan)
        return fail(PA_ERR_INVALID, E, "plan is NULL");
    if (plan->part_tokens == 0 || plan->part_tokens % 32 || plan->n_parts == 0 ||
        plan->direct != (plan->n_parts == 1u) || plan->n_ctas == 0)
        return fail(PA_ERR_INVALID, E, "inconsistent plan (part_tokens %u, n_parts %u, direct %u)",
                    plan->part_tokens, plan->n_parts, plan->direct);
    return PA_OK;
}

int check_shapes(uint32_t n_seqs, uint32_t hq, uint32_t hkv, uint32_t d, uint32_t B,
                 pa_type kt, pa_type vt, const char *E)
{
    if (n_seqs == 0)
        return fail(PA_ERR_INVALID, E, "n_seqs is 0");
    if (hkv == 0 || hq < hkv || hq % hkv || hq / hkv > 8)
        return fail(PA_ERR_INVALID, E, "hq %u / hkv %u unsupported (group <= 8)", hq, hkv);
    if (d != 128 && d != 256)
        return fail(PA_ERR_INVALID, E, "d %u unsupported (128 or 256)", d);
    if (B != 16 && B != 32)
        return fail(PA_ERR_INVALID, E, "block_size %u unsupported (16 or 32)", B);
    if (!type_ok(kt) || !type_ok(vt))
        return fail(PA_ERR_INVALID, E, "unknown K/V type");
    return PA_OK;
}

bool use_fast(const pa_decode_args *a)
{
    return !(a->flags & PA_FLAG_PLAIN) &&
           pa::fast_decode_supported(a->k_type, a->v_type, a->d, a->hq, a->hkv, a->block_size);
}

// Validates a decode call and resolves it into kernel parameters.
int resolve(const pa_decode_args *a, const pa_plan_t *plan, const char *E, pa::DecodeParams *p)
{
    if (!a)
        return fail(PA_ERR_INVALID, E, "args is NULL");
    int rc = check_plan(plan, E);
    if (rc)
        return rc;
    rc = check_shapes(a->n_seqs, a->hq, a->hkv, a->d, a->block_size, a->k_type, a->v_type, E);
    if (rc)
        return rc;
    if (!a->k_pool || !a->v_pool || !a->block_table || !a->seq_lens || !a->q || !a->status)
        return fail(PA_ERR_INVALID, E, "NULL device pointer");
    if (!aligned16(a->k_pool) || !aligned16(a->v_pool) || !aligned16(a->q))
        return fail(PA_ERR_INVALID, E, "pools and q must be 16-byte aligned");
    if (plan->direct ? !a->out : (!a->part_o || !a->part_ml))
        return fail(PA_ERR_INVALID, E, plan->direct ? "direct plan needs out"
                                                    : "partitioned plan needs part_o and part_ml");
    if (!plan->direct && (!aligned16(a->part_o) || (reinterpret_cast<uintptr_t>(a->part_ml) & 7)))
        return fail(PA_ERR_INVALID, E, "part_o must be 16-byte and part_ml 8-byte aligned");
    if (a->out && (reinterpret_cast<uintptr_t>(a->out) & 15))
        return fail(PA_ERR_INVALID, E, "out must be 16-byte aligned");
    const uint32_t T = plan->q_tokens > 1 ? plan->q_tokens : 1;
    if ((uint64_t)a->n_seqs * T > 0x7fffffffull)
        return fail(PA_ERR_RANGE, E, "n_seqs * q_tokens exceeds 2^31 - 1");
    // a direct plan has one CTA per query row, or per sequence when the
    // sequence's T rows are decoded together (a multi-token plan)
    if (plan->direct && plan->n_ctas != (plan->multi ? a->n_seqs : a->n_seqs * T))
        return fail(PA_ERR_INVALID, E, "direct plan must have n_ctas == n_seqs%s",
                    plan->multi ? "" : " * q_tokens");
    if (plan->direct ? plan->n_direct != 0
                     : (plan->n_direct >= a->n_seqs * T || plan->n_ctas <= plan->n_direct))
        return fail(PA_ERR_INVALID, E, "inconsistent n_direct %u for %u query rows",
                    plan->n_direct, a->n_seqs * T);
    if (a->table_stride == 0)
        return fail(PA_ERR_INVALID, E, "table_stride is 0");
    if (a->n_pool_blocks == 0 || a->n_pool_blocks > 0x80000000ull)
        return fail(PA_ERR_RANGE, E, "n_pool_blocks must be in [1, 2^31] (int32 table ids)");
    if (!isfinite(a->scale))
        return fail(PA_ERR_INVALID, E, "scale is not finite");
    p->k_pool = static_cast<const uint8_t *>(a->k_pool);
    p->v_pool = static_cast<const uint8_t *>(a->v_pool);
    p->n_pool_blocks = a->n_pool_blocks;
    p->block_table = a->block_table;
    p->table_stride = a->table_stride;
    p->seq_lens = a->seq_lens;
    p->q = a->q;
    p->scale_log2 = a->scale * 1.4426950408889634f;
    p->part_o = a->part_o;
    p->part_ml = a->part_ml;
    p->out = a->out;
    p->status = a->status;
    p->n_seqs = a->n_seqs * T;  // query rows
    p->q_tokens = T;
    p->hq = a->hq;
    p->hkv = a->hkv;
    p->d = a->d;
    p->block_size = a->block_size;
    p->part_tokens = plan->part_tokens;
    p->n_parts = plan->n_parts;
    p->direct = plan->direct;
    p->n_ctas = plan->n_ctas;
    p->k_row_bytes = pa_row_bytes(a->k_type, a->d);
    p->v_row_bytes = pa_row_bytes(a->v_type, a->d);
    p->counters = nullptr;
    p->q_f32 = 0;
    p->n_direct = plan->direct ? 0 : plan->n_direct;
    p->merge_no_wait = (a->flags & PA_FLAG_MERGE_NO_WAIT) ? 1u : 0u;
    p->stream = plan->stream ? 1u : 0u;
    p->multi = plan->multi ? 1u : 0u;
    if (plan->multi) {
        if (plan->stream || plan->n_direct ||
            !pa::mt_decode_supported(a->k_type, a->v_type, a->d, a->hq, a->hkv, T) ||
            !use_fast(a))
            return fail(PA_ERR_INVALID, E, "multi-token plans need the fast kernel and its shapes");
    }
    if (plan->stream) {
        if (plan->direct || plan->n_direct || plan->n_parts > 32)
            return fail(PA_ERR_INVALID, E, "inconsistent stream plan");
        if (a->k_type != a->v_type || !use_fast(a))
            return fail(PA_ERR_INVALID, E, "stream plans need the fast kernel and one K/V type");
    }
    return PA_OK;
}

int launch_decode(const pa_decode_args *a, const pa::DecodeParams &p, cudaStream_t st,
                  const char *E)
{
    return use_fast(a) ? pa::launch_fast_decode(p, a->k_type, a->v_type, st, E)
                       : pa::launch_plain_decode(p, a->k_type, a->v_type, st, E);
}

}  // namespace

int pa::check_decode(const pa_decode_args *a, const pa_plan_t *plan, const char *entry)
{
    pa::DecodeParams p;
    return resolve(a, plan, entry, &p);
}

extern "C" int pa_quantize_q(const float *q, void *q8_1, uint32_t n_rows, uint32_t d,
                             pa_stream_t stream)
{
    static const char *E = "pa_quantize_q";
    if (d == 0 || d % 32)
        return fail(PA_ERR_INVALID, E, "d %u is not a positive multiple of 32", d);
    if (n_rows && (!q || !q8_1))
        return fail(PA_ERR_INVALID, E, "NULL device pointer");
    if (n_rows && (!aligned16(q) || (reinterpret_cast<uintptr_t>(q8_1) & 3)))
        return fail(PA_ERR_INVALID, E, "q must be 16-byte and q8_1 4-byte aligned");
    return pa::launch_quantize_q(q, q8_1, n_rows, d, pa::stream_of(stream), E);
}

extern "C" int pa_query_occupancy(const pa_plan_in *in, int32_t *sm_count, int32_t *ctas_per_sm)
{
    static const char *E = "pa_query_occupancy";
    if (!in || !sm_count || !ctas_per_sm)
        return fail(PA_ERR_INVALID, E, "NULL argument");
    int rc = check_shapes(in->n_seqs ? in->n_seqs : 1, in->hq, in->hkv, in->d, in->block_size,
                          in->k_type, in->v_type, E);
    if (rc)
        return rc;
    int dev = 0, sms = 0;
    rc = cuda_check(cudaGetDevice(&dev), E, "cudaGetDevice");
    if (rc)
        return rc;
    rc = cuda_check(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev), E,
                    "cudaDeviceGetAttribute");
    if (rc)
        return rc;
    int cps = 0;
    if (pa::fast_decode_supported(in->k_type, in->v_type, in->d, in->hq, in->hkv,
                                  in->block_size))
        rc = pa::fast_decode_occupancy(in->k_type, in->v_type, in->d, in->hq, in->hkv,
                                       in->block_size, &cps);
    else
        rc = pa::plain_decode_occupancy(in->k_type, in->v_type, in->d, in->hq, &cps);
    if (rc)
        return fail(PA_ERR_CUDA, E, "occupancy query failed: %s",
                    cudaGetErrorString(cudaGetLastError()));
    *sm_count = sms;
    *ctas_per_sm = cps > 0 ? cps : 1;
    return PA_OK;
}

extern "C" int pa_decode_partial(const pa_decode_args *args, const pa_plan_t *plan,
                                 pa_stream_t stream)
{
    static const char *E = "pa_decode_partial";
    pa::DecodeParams p;
    int rc = resolve(args, plan, E, &p);
    if (rc)
        return rc;
    if (plan->stream)
        return fail(PA_ERR_INVALID, E, "stream plans run only through the fused calls");
    return launch_decode(args, p, pa::stream_of(stream), E);
}

extern "C" const char *pa_decode_kernel_name(pa_type kt, pa_type vt, uint32_t d, uint32_t hq,
                                             uint32_t hkv, uint32_t block_size, uint32_t flags)
{
    if (check_shapes(1, hq, hkv, d, block_size, kt, vt, "pa_decode_kernel_name"))
        return nullptr;
    if (!(flags & PA_FLAG_PLAIN) && pa::fast_decode_supported(kt, vt, d, hq, hkv, block_size))
        return "fast_decode_kernel";
    return "plain_decode_kernel";
}

// The decode launch of a fused call, and for a partitioned multi-token plan
// (whose kernel writes partials only) the merge kernel after it.
static int decode_then_merge(const pa_decode_args *args, const pa_plan_t *plan,
                             const pa::DecodeParams &p, cudaStream_t st, const char *E)
{
    int rc = launch_decode(args, p, st, E);
    if (rc || !plan->multi || plan->direct)
        return rc;
    return pa::launch_merge(args->part_o, args->part_ml, args->seq_lens, p.out, args->n_seqs,
                            plan->q_tokens, args->hq, args->d, plan->n_parts, plan->part_tokens,
                            0, st, E);
}

extern "C" int pa_decode_fused(const pa_decode_args *args, const pa_plan_t *plan,
                               int32_t *counters, pa_stream_t stream)
{
    static const char *E = "pa_decode_fused";
    pa::DecodeParams p;
    int rc = resolve(args, plan, E, &p);
    if (rc)
        return rc;
    if (!plan->direct) {
        if (!counters || (reinterpret_cast<uintptr_t>(counters) & 3))
            return fail(PA_ERR_INVALID, E, "a partitioned plan needs 4-byte aligned counters");
        if (!args->out)
            return fail(PA_ERR_INVALID, E, "out is NULL");
        if (!plan->multi)
            p.counters = counters;
    }
    return decode_then_merge(args, plan, p, pa::stream_of(stream), E);
}

extern "C" int pa_decode_step_fused(const pa_decode_args *args, const pa_plan_t *plan,
                                    void *q8_1_scratch, int32_t *counters, pa_stream_t stream)
{
    static const char *E = "pa_decode_step_fused";
    pa::DecodeParams p;
    int rc = resolve(args, plan, E, &p);
    if (rc)
        return rc;
    if (!plan->direct) {
        if (!counters || (reinterpret_cast<uintptr_t>(counters) & 3))
            return fail(PA_ERR_INVALID, E, "a partitioned plan needs 4-byte aligned counters");
        if (!args->out)
            return fail(PA_ERR_INVALID, E, "out is NULL");
        if (!plan->multi)
            p.counters = counters;
    }
    cudaStream_t st = pa::stream_of(stream);
    if (args->k_type != PA_F16) {
        if (!q8_1_scratch || (reinterpret_cast<uintptr_t>(q8_1_scratch) & 15))
            return fail(PA_ERR_INVALID, E, "quantised K needs a 16-byte aligned q8_1_scratch");
        if (use_fast(args) && !plan->stream && !plan->multi) {
            // the fast kernel quantises the query rows itself: one launch per step
            p.q_f32 = 1;
            return launch_decode(args, p, st, E);
        }
        rc = pa::launch_quantize_q(static_cast<const float *>(args->q), q8_1_scratch,
                                   p.n_seqs * args->hq, args->d, st, E);
        if (rc)
            return rc;
        p.q = q8_1_scratch;
    }
    return decode_then_merge(args, plan, p, st, E);
}

extern "C" int pa_merge(const void *part_o, const float *part_ml, const int32_t *seq_lens,
                        float *out, uint32_t n_seqs, uint32_t hq, uint32_t d,
                        const pa_plan_t *plan, pa_stream_t stream)
{
    static const char *E = "pa_merge";
    int rc = check_plan(plan, E);
    if (rc)
        return rc;
    if (plan->stream)
        return fail(PA_ERR_INVALID, E, "stream plans merge inside the fused calls");
    if (plan->direct)
        return fail(PA_ERR_INVALID, E, "a direct plan has no partials to merge");
    if (!part_o || !part_ml || !seq_lens || !out)
        return fail(PA_ERR_INVALID, E, "NULL device pointer");
    if (!aligned16(part_o) || (reinterpret_cast<uintptr_t>(part_ml) & 7) ||
        (reinterpret_cast<uintptr_t>(out) & 15))
        return fail(PA_ERR_INVALID, E, "part_o and out must be 16-byte, part_ml 8-byte aligned");
    if (n_seqs == 0 || hq == 0 || (d != 128 && d != 256))
        return fail(PA_ERR_INVALID, E, "bad shape (n_seqs %u, hq %u, d %u)", n_seqs, hq, d);
    const uint64_t T = plan->q_tokens > 1 ? plan->q_tokens : 1;
    if (plan->n_direct >= (uint64_t)n_seqs * T)
        return fail(PA_ERR_INVALID, E, "n_direct %u leaves no partitioned row of %llu",
                    plan->n_direct, (unsigned long long)((uint64_t)n_seqs * T));
    const uint64_t elems = ((uint64_t)n_seqs * T - plan->n_direct) * hq * plan->n_parts * d;
    if (elems > (1ull << 40))
        return fail(PA_ERR_RANGE, E, "partial buffer of %llu elements exceeds 2^40",
                    (unsigned long long)elems);
    return pa::launch_merge(part_o, part_ml, seq_lens, out, n_seqs, plan->q_tokens, hq, d,
                            plan->n_parts, plan->part_tokens, plan->n_direct,
                            pa::stream_of(stream), E);
}

extern "C" int pa_decode_step(const pa_decode_args *args, const pa_plan_t *plan,
                              void *q8_1_scratch, pa_stream_t stream)
{
    static const char *E = "pa_decode_step";
    pa::DecodeParams p;
    int rc = resolve(args, plan, E, &p);
    if (rc)
        return rc;
    if (plan->stream)
        return fail(PA_ERR_INVALID, E, "stream plans run only through the fused calls");
    cudaStream_t st = pa::stream_of(stream);
    if (args->k_type != PA_F16) {
        if (!q8_1_scratch || (reinterpret_cast<uintptr_t>(q8_1_scratch) & 15))
            return fail(PA_ERR_INVALID, E, "quantised K needs a 16-byte aligned q8_1_scratch");
        rc = pa::launch_quantize_q(static_cast<const float *>(args->q), q8_1_scratch,
                                   p.n_seqs * args->hq, args->d, st, E);
        if (rc)
            return rc;
        p.q = q8_1_scratch;
    }
    rc = launch_decode(args, p, st, E);
    if (rc || plan->direct)
        return rc;
    return pa::launch_merge(args->part_o, args->part_ml, args->seq_lens, args->out,
                            args->n_seqs, plan->q_tokens, args->hq, args->d, plan->n_parts,
                            plan->part_tokens, plan->n_direct, st, E);
}

// The device address of page-locked host memory that the kernels may load
// from or store to directly (16-byte aligned for their vector accesses), or
// nullptr for any other pointer: pageable memory is never handed to a kernel.
static float *mapped_host(float *h)
{
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, h) != cudaSuccess) {
        cudaGetLastError();  // clear the (non-sticky) error of an unknown pointer
        return nullptr;
    }
    if (at.type != cudaMemoryTypeHost || at.devicePointer == nullptr ||
        (reinterpret_cast<uintptr_t>(at.devicePointer) & 15u) != 0)
        return nullptr;
    return static_cast<float *>(at.devicePointer);
}

// The query of a host-buffer step into args->q: page-locked host memory that
// the device maps is staged by a kernel that overlaps the previous kernel's
// end (launch_stage_q); anything else takes an asynchronous copy.
static int copy_q_in(const float *q_host, const void *q_dev, size_t bytes, cudaStream_t st,
                     const char *E)
{
    const float *mapped = mapped_host(const_cast<float *>(q_host));
    if (mapped && (bytes & 15u) == 0 && (reinterpret_cast<uintptr_t>(q_dev) & 15u) == 0)
        return pa::launch_stage_q(mapped, const_cast<void *>(q_dev), bytes, st, E);
    return cuda_check(cudaMemcpyAsync(const_cast<void *>(q_dev), q_host, bytes,
                                      cudaMemcpyHostToDevice, st),
                      E, "copy of q to the device");
}

extern "C" int pa_decode_step_host(const float *q_host, float *out_host,
                                   const pa_decode_args *args, const pa_plan_t *plan,
                                   void *q8_1_scratch, pa_stream_t stream)
{
    static const char *E = "pa_decode_step_host";
    if (!q_host || !out_host || !args || !args->q || !args->out)
        return fail(PA_ERR_INVALID, E, "NULL host or device pointer");
    pa::DecodeParams p;
    int rc = resolve(args, plan, E, &p);  // refuse before copying anything
    if (rc)
        return rc;
    const size_t bytes = (size_t)p.n_seqs * args->hq * args->d * sizeof(float);
    cudaStream_t st = pa::stream_of(stream);
    rc = copy_q_in(q_host, args->q, bytes, st, E);
    if (rc)
        return rc;
    // page-locked out_host: the kernels write it directly, no copy back
    pa_decode_args a = *args;
    float *out_mapped = mapped_host(out_host);
    if (out_mapped)
        a.out = out_mapped;
    rc = pa_decode_step(&a, plan, q8_1_scratch, stream);
    if (rc || out_mapped)
        return rc;
    return cuda_check(cudaMemcpyAsync(out_host, args->out, bytes, cudaMemcpyDeviceToHost, st), E,
                      "copy of out to the host");
}

extern "C" int pa_decode_step_fused_host(const float *q_host, float *out_host,
                                         const pa_decode_args *args, const pa_plan_t *plan,
                                         void *q8_1_scratch, int32_t *counters,
                                         pa_stream_t stream)
{
    static const char *E = "pa_decode_step_fused_host";
    if (!q_host || !out_host || !args || !args->q || !args->out)
        return fail(PA_ERR_INVALID, E, "NULL host or device pointer");
    pa::DecodeParams p;
    int rc = resolve(args, plan, E, &p);  // refuse before copying anything
    if (rc)
        return rc;
    if (!plan->direct && !counters)
        return fail(PA_ERR_INVALID, E, "a partitioned plan needs counters");
    const size_t bytes = (size_t)p.n_seqs * args->hq * args->d * sizeof(float);
    cudaStream_t st = pa::stream_of(stream);
    rc = copy_q_in(q_host, args->q, bytes, st, E);
    if (rc)
        return rc;
    // page-locked out_host: the kernels write it directly, no copy back
    pa_decode_args a = *args;
    float *out_mapped = mapped_host(out_host);
    if (out_mapped)
        a.out = out_mapped;
    rc = pa_decode_step_fused(&a, plan, q8_1_scratch, counters, stream);
    if (rc || out_mapped)
        return rc;
    return cuda_check(cudaMemcpyAsync(out_host, args->out, bytes, cudaMemcpyDeviceToHost, st), E,
                      "copy of out to the host");
}

extern "C" int pa_append_kv(const pa_append_args *a, pa_stream_t stream)
{
    static const char *E = "pa_append_kv";
    if (!a)
        return fail(PA_ERR_INVALID, E, "NULL args");
    if (a->n_seqs == 0)
        return PA_OK;
    if (!a->k_pool || !a->v_pool || !a->block_table || !a->seq_lens || !a->k_new ||
        !a->v_new || !a->fresh_blocks || !a->status)
        return fail(PA_ERR_INVALID, E, "NULL device pointer");
    if (a->k_type < PA_F16 || a->k_type > PA_Q4_0 || a->v_type < PA_F16 || a->v_type > PA_Q4_0)
        return fail(PA_ERR_INVALID, E, "unknown K/V type");
    if (a->d != 128 && a->d != 256)
        return fail(PA_ERR_INVALID, E, "d %u unsupported (128 or 256)", a->d);
    if (a->block_size != 16 && a->block_size != 32)
        return fail(PA_ERR_INVALID, E, "block_size %u unsupported (16 or 32)", a->block_size);
    if (a->hkv == 0 || a->hkv > 8)
        return fail(PA_ERR_INVALID, E, "hkv %u unsupported (1..8)", a->hkv);
    if (a->table_stride == 0)
        return fail(PA_ERR_INVALID, E, "table_stride is 0");
    if (a->n_pool_blocks == 0 || a->n_pool_blocks > 0x80000000ull)
        return fail(PA_ERR_RANGE, E, "n_pool_blocks must be in [1, 2^31] (int32 table ids)");
    if (a->n_seqs > 0x7fffffffu)
        return fail(PA_ERR_RANGE, E, "n_seqs exceeds the grid");
    if (!aligned16(a->k_pool) || !aligned16(a->v_pool) || !aligned16(a->k_new) ||
        !aligned16(a->v_new))
        return fail(PA_ERR_INVALID, E, "pools and new rows must be 16-byte aligned");
    return pa::launch_append(a, pa::stream_of(stream), E);
}

extern "C" int pa_status_read(int32_t *dev_status, pa_stream_t stream, int32_t *host_out,
                              int reset)
{
    static const char *E = "pa_status_read";
    if (!dev_status || !host_out)
        return fail(PA_ERR_INVALID, E, "NULL pointer");
    cudaStream_t st = pa::stream_of(stream);
    int32_t v = 0;
    int rc = cuda_check(cudaMemcpyAsync(&v, dev_status, sizeof v, cudaMemcpyDeviceToHost, st), E,
                        "status copy");
    if (!rc)
        rc = cuda_check(cudaStreamSynchronize(st), E, "stream synchronise");
    if (!rc && reset) {
        rc = cuda_check(cudaMemsetAsync(dev_status, 0, sizeof(int32_t), st), E, "status reset");
        if (!rc)
            rc = cuda_check(cudaStreamSynchronize(st), E, "stream synchronise");
    }
    if (rc)
        return rc;
    *host_out = v;
    if (v & PA_STATUS_TIMEOUT)
        return fail(PA_ERR_TIMEOUT, E, "a kernel abandoned a bounded pipeline wait");
    if (v & PA_STATUS_LEN_OVER_PLAN)
        return fail(PA_ERR_RANGE, E, "sequence lengths past what the plan covers were left out");
    if (v & PA_STATUS_APPEND_RANGE)
        return fail(PA_ERR_RANGE, E, "an append found no table entry left for a sequence");
    if (v & PA_STATUS_CORRUPT_TABLE)
        return fail(PA_ERR_CORRUPT_TABLE, E, "a block id outside the pool was skipped");
    return PA_OK;
}

extern "C" int pa_debug_row_offsets(const int32_t *block_table, uint32_t table_stride,
                                    const int32_t *seq_lens, uint32_t n_seqs,
                                    uint32_t max_tokens, uint32_t block_size, uint32_t hkv,
                                    uint64_t row_bytes, uint64_t n_pool_blocks,
                                    uint64_t *offsets, int32_t *status, pa_stream_t stream)
{
    static const char *E = "pa_debug_row_offsets";
    if (!block_table || !seq_lens || !offsets || !status)
        return fail(PA_ERR_INVALID, E, "NULL device pointer");
    if (block_size == 0 || hkv == 0 || row_bytes == 0 || table_stride == 0)
        return fail(PA_ERR_INVALID, E, "zero size");
    return pa::launch_debug_offsets(block_table, table_stride, seq_lens, n_seqs, max_tokens,
                                    block_size, hkv, row_bytes, n_pool_blocks, offsets, status,
                                    pa::stream_of(stream), E);
}

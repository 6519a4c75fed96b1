// pa_noalloc.cu -- a decode step for callers that cannot allocate device
// memory.
//
// pa_decode_step needs three scratch buffers besides its inputs and output:
// the q8_1 copy of the query and the per-partition partials.  Some callers
// cannot provide them: code that runs where cudaMalloc is off limits (inside
// a host callback, while another component owns every allocation through its
// own arena, or under a memory budget that forbids growing), or that must
// not block on the allocator at decode time.  pa_decode_step_noalloc keeps
// that scratch in one static device array of this file instead.  The array
// is part of the library image: every GPU that loads the library holds
// PA_NOALLOC_SCRATCH_BYTES of it until the process exits.
//
// The step itself is the existing one: this file calls pa_quantize_q,
// pa_decode_partial and pa_merge with pointers into the array and changes
// nothing in them.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "pa_internal.h"

namespace {

// The scratch.  In host code this name is only a stand-in for the symbol,
// not a device address; the address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[PA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
// Per device: the address looked up, and the unique id of the context it
// was looked up in.  A context that is destroyed and made again (after
// cudaDeviceReset, say) has a new id, so the look-up runs again there.
struct Entry {
    void *addr = nullptr;
    unsigned long long ctx_id = 0;
    bool valid = false;
};
Entry g_entry[kMaxDevices];

// The driver's cuCtxGetCurrent and cuCtxGetId, through the runtime's entry
// point query (the library links only the runtime).
struct CtxFns {
    PFN_cuCtxGetCurrent_v4000 current = nullptr;
    PFN_cuCtxGetId_v12000 id = nullptr;
};

const CtxFns &ctx_fns()
{
    static CtxFns f;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            f.current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            f.id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
    });
    return f;
}

// Device address of the scratch in the current device's context.  The
// look-up (cudaGetSymbolAddress, with that device current) runs on the first
// call on a device and again only when the device's context has changed
// since; it allocates nothing.
int scratch_address(void **out, const char *E)
{
    int dev = -1;
    int rc = pa::cuda_check(cudaGetDevice(&dev), E, "cudaGetDevice");
    if (rc)
        return rc;
    if (dev < 0 || dev >= kMaxDevices)
        return pa::fail(PA_ERR_RANGE, E, "device ordinal %d beyond %d", dev, kMaxDevices);
    // make the device's primary context current on this thread (the
    // runtime initialises it here if no earlier call did)
    rc = pa::cuda_check(cudaSetDevice(dev), E, "cudaSetDevice");
    if (rc)
        return rc;
    const CtxFns &f = ctx_fns();
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    // a context that cannot be identified is looked up afresh every call
    const bool known = f.current && f.id && f.current(&ctx) == CUDA_SUCCESS && ctx &&
                       f.id(ctx, &id) == CUDA_SUCCESS;
    std::lock_guard<std::mutex> lock(g_mu);
    Entry &e = g_entry[dev];
    if (!known || !e.valid || e.ctx_id != id) {
        void *p = nullptr;
        rc = pa::cuda_check(cudaGetSymbolAddress(&p, g_noalloc_scratch), E,
                            "cudaGetSymbolAddress of the static scratch");
        if (rc)
            return rc;
        e.addr = p;
        e.ctx_id = id;
        e.valid = known;
    }
    *out = e.addr;
    return PA_OK;
}

uint64_t round256(uint64_t x) { return (x + 255) & ~255ull; }

}  // namespace

extern "C" int pa_decode_step_noalloc(const pa_decode_args *args, const pa_plan_t *plan,
                                      pa_stream_t stream)
{
    static const char *E = "pa_decode_step_noalloc";
    if (!args || !plan)
        return pa::fail(PA_ERR_INVALID, E, "NULL args or plan");
    if (plan->n_parts == 0 || plan->direct != (plan->n_parts == 1u))
        return pa::fail(PA_ERR_INVALID, E, "inconsistent plan");
    if (plan->stream)
        return pa::fail(PA_ERR_INVALID, E, "stream plans run only through the fused calls");
    const bool quantised = args->k_type != PA_F16;
    const uint64_t rows = (uint64_t)args->n_seqs * (plan->q_tokens > 1 ? plan->q_tokens : 1) *
                          args->hq;
    const uint64_t q81_bytes = quantised ? round256(rows * (args->d / 32) * 36ull) : 0;
    // partials of the partitioned rows only (those after the n_direct leading ones)
    const uint64_t prows = plan->direct || plan->n_direct * (uint64_t)args->hq > rows
                               ? 0
                               : rows - (uint64_t)plan->n_direct * args->hq;
    const uint64_t po_bytes = plan->direct ? 0 : round256(prows * plan->n_parts * args->d * 2ull);
    const uint64_t pm_bytes = plan->direct ? 0 : round256(prows * plan->n_parts * 8ull);
    const uint64_t need = q81_bytes + po_bytes + pm_bytes;
    if (need > PA_NOALLOC_SCRATCH_BYTES)
        return pa::fail(PA_ERR_RANGE, E,
                        "this step needs %llu bytes of scratch; the library's static scratch "
                        "holds %llu (use pa_decode_step with caller buffers)",
                        (unsigned long long)need, (unsigned long long)PA_NOALLOC_SCRATCH_BYTES);
    void *base = nullptr;
    int rc = scratch_address(&base, E);
    if (rc)
        return rc;
    unsigned char *s = static_cast<unsigned char *>(base);
    pa_decode_args a = *args;
    if (!plan->direct) {
        a.part_o = s + q81_bytes;
        a.part_ml = reinterpret_cast<float *>(s + q81_bytes + po_bytes);
    }
    // every check of the decode call runs before the pre-pass is launched,
    // so a refused call launches nothing
    rc = pa::check_decode(&a, plan, E);
    if (rc)
        return rc;
    // Nothing in the scratch has to start at zero: the pre-pass writes every
    // q8_1 block, and the merge reads only partitions the decode kernel wrote
    // in this same step.
    if (quantised) {
        rc = pa_quantize_q(static_cast<const float *>(args->q), s, (uint32_t)rows, args->d,
                           stream);
        if (rc)
            return rc;
        a.q = s;
    }
    rc = pa_decode_partial(&a, plan, stream);
    if (rc || plan->direct)
        return rc;
    return pa_merge(a.part_o, a.part_ml, a.seq_lens, a.out, a.n_seqs, a.hq, a.d, plan, stream);
}

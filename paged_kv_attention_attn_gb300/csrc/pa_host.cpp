// pa_host.cpp -- host-only parts of the C ABI: error reporting, the fixed-block
// allocator and the partition planner.  No device code and no allocation of
// device memory here.
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <new>
#include <vector>

#include "pa_internal.h"

namespace pa {

static thread_local char g_last_error[512] = "";

int fail(int code, const char *entry, const char *fmt, ...)
{
    char msg[400];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(msg, sizeof msg, fmt, ap);
    va_end(ap);
    snprintf(g_last_error, sizeof g_last_error, "%s: %s", entry, msg);
    return code;
}

int cuda_check(cudaError_t e, const char *entry, const char *what)
{
    if (e == cudaSuccess)
        return PA_OK;
    return fail(PA_ERR_CUDA, entry, "%s: %s", what, cudaGetErrorString(e));
}

}  // namespace pa

using pa::fail;

extern "C" const char *pa_strerror(int code)
{
    switch (code) {
    case PA_OK: return "PA_OK";
    case PA_ERR_INVALID: return "PA_ERR_INVALID";
    case PA_ERR_NOMEM: return "PA_ERR_NOMEM";
    case PA_ERR_STALE: return "PA_ERR_STALE";
    case PA_ERR_CUDA: return "PA_ERR_CUDA";
    case PA_ERR_CORRUPT_TABLE: return "PA_ERR_CORRUPT_TABLE";
    case PA_ERR_RANGE: return "PA_ERR_RANGE";
    case PA_ERR_TIMEOUT: return "PA_ERR_TIMEOUT";
    default: return "PA_ERR_UNKNOWN";
    }
}

extern "C" const char *pa_last_error(void) { return pa::g_last_error; }

extern "C" uint64_t pa_row_bytes(pa_type type, uint32_t d)
{
    if (d == 0 || d % 32 != 0)
        return 0;
    switch (type) {
    case PA_F16: return 2ull * d;
    case PA_Q8_0: return (uint64_t)(d / 32) * 34ull;
    case PA_Q4_0: return (uint64_t)(d / 32) * 18ull;
    default: return 0;
    }
}

// ------------------------------------------------------------------ allocator
//
// Fixed-block pool with transactional allocation, stale-handle detection and
// immediate release ("feat: add paged-attention monolithic decode-only AR
// foundation", lucebox pull 555, Summary).  LIFO free stack; handle =
// (generation << 32) | id; generation starts at 1, advances on release and
// skips 0 on wrap.

struct pa_pool {
    uint32_t n;
    std::vector<uint32_t> gen;
    std::vector<uint8_t> live;
    std::vector<uint32_t> stack;  // back() is the next id handed out
    std::vector<uint8_t> mark;    // scratch for duplicate detection in free
};

extern "C" int pa_pool_create(uint32_t n_blocks, pa_pool **out)
{
    static const char *E = "pa_pool_create";
    if (!out)
        return fail(PA_ERR_INVALID, E, "out is NULL");
    *out = nullptr;
    if (n_blocks == 0 || n_blocks > 0x7fffffffu)
        return fail(PA_ERR_INVALID, E, "n_blocks %u outside [1, 2^31-1]", n_blocks);
    pa_pool *p = new (std::nothrow) pa_pool;
    if (!p)
        return fail(PA_ERR_NOMEM, E, "host allocation failed");
    try {
        p->n = n_blocks;
        p->gen.assign(n_blocks, 1u);
        p->live.assign(n_blocks, 0);
        p->mark.assign(n_blocks, 0);
        p->stack.resize(n_blocks);
        for (uint32_t i = 0; i < n_blocks; ++i)
            p->stack[i] = n_blocks - 1 - i;
    } catch (...) {
        delete p;
        return fail(PA_ERR_NOMEM, E, "host allocation failed");
    }
    *out = p;
    return PA_OK;
}

extern "C" void pa_pool_destroy(pa_pool *pool) { delete pool; }

extern "C" int pa_pool_alloc(pa_pool *pool, uint32_t n, pa_handle *out)
{
    static const char *E = "pa_pool_alloc";
    if (!pool || (n && !out))
        return fail(PA_ERR_INVALID, E, "NULL pool or out");
    if (n > pool->stack.size())
        return fail(PA_ERR_NOMEM, E, "%u blocks requested, %zu free", n, pool->stack.size());
    for (uint32_t i = 0; i < n; ++i) {
        uint32_t id = pool->stack.back();
        pool->stack.pop_back();
        pool->live[id] = 1;
        out[i] = ((uint64_t)pool->gen[id] << 32) | id;
    }
    return PA_OK;
}

extern "C" int pa_pool_free(pa_pool *pool, uint32_t n, const pa_handle *h)
{
    static const char *E = "pa_pool_free";
    if (!pool || (n && !h))
        return fail(PA_ERR_INVALID, E, "NULL pool or handles");
    // validate everything first; marks catch a handle listed twice
    uint32_t bad = n;
    for (uint32_t i = 0; i < n; ++i) {
        uint64_t id = h[i] & 0xffffffffull;
        uint32_t g = (uint32_t)(h[i] >> 32);
        if (id >= pool->n || !pool->live[id] || pool->gen[id] != g || pool->mark[id]) {
            bad = i;
            break;
        }
        pool->mark[id] = 1;
    }
    for (uint32_t i = 0; i < bad; ++i)
        pool->mark[h[i] & 0xffffffffull] = 0;
    if (bad < n)
        return fail(PA_ERR_STALE, E, "handle %u (0x%llx) is stale, out of range or repeated",
                    bad, (unsigned long long)h[bad]);
    for (uint32_t i = 0; i < n; ++i) {
        uint32_t id = (uint32_t)(h[i] & 0xffffffffull);
        pool->live[id] = 0;
        uint32_t g = pool->gen[id] + 1;
        pool->gen[id] = g ? g : 1;
        pool->stack.push_back(id);
    }
    return PA_OK;
}

extern "C" int32_t pa_handle_block(pa_handle h) { return (int32_t)(uint32_t)(h & 0xffffffffull); }

extern "C" uint32_t pa_pool_free_count(const pa_pool *pool)
{
    return pool ? (uint32_t)pool->stack.size() : 0;
}

extern "C" uint32_t pa_pool_capacity(const pa_pool *pool) { return pool ? pool->n : 0; }

// -------------------------------------------------------------------- planner

static uint64_t cdiv(uint64_t a, uint64_t b) { return (a + b - 1) / b; }
static uint64_t roundup(uint64_t a, uint64_t b) { return cdiv(a, b) * b; }

static int pa_plan_quiet(const pa_plan_in *in, pa_plan_t *out);

extern "C" int pa_plan(const pa_plan_in *in, pa_plan_t *out)
{
    const int rc = pa_plan_quiet(in, out);
    if (rc)
        return rc;
    // PA_LOG_PLAN (set, not "0"): one line per plan on stderr
    const char *log = getenv("PA_LOG_PLAN");
    if (log && *log && strcmp(log, "0") != 0)
        fprintf(stderr,
                "pa_plan: n_seqs=%u q_tokens=%u max_len=%u total_len=%llu slots=%lld "
                "force_parts=%d flags=%u -> part_tokens=%u n_parts=%u direct=%u n_direct=%u "
                "n_ctas=%u stream=%u multi=%u\n",
                in->n_seqs, out->q_tokens, in->max_len, (unsigned long long)in->total_len,
                (long long)in->sm_count * in->ctas_per_sm, in->force_parts, in->flags,
                out->part_tokens, out->n_parts, out->direct, out->n_direct, out->n_ctas,
                out->stream, out->multi);
    return PA_OK;
}

static int pa_plan_quiet(const pa_plan_in *in, pa_plan_t *out)
{
    static const char *E = "pa_plan";
    const uint64_t TILE = 32, MIN_PART = 128;
    if (!in || !out)
        return fail(PA_ERR_INVALID, E, "NULL argument");
    if (in->n_seqs < 1)
        return fail(PA_ERR_INVALID, E, "n_seqs must be >= 1");
    if (in->block_size != 16 && in->block_size != 32)
        return fail(PA_ERR_INVALID, E, "block_size %u unsupported (16 or 32)", in->block_size);
    if (in->hkv < 1 || in->hq < in->hkv || in->hq % in->hkv || in->hq / in->hkv > 8)
        return fail(PA_ERR_INVALID, E, "hq %u / hkv %u: need hq %% hkv == 0 and a group <= 8",
                    in->hq, in->hkv);
    if (in->d != 128 && in->d != 256)
        return fail(PA_ERR_INVALID, E, "d %u unsupported (128 or 256)", in->d);
    if ((unsigned)in->k_type > 2u || (unsigned)in->v_type > 2u)
        return fail(PA_ERR_INVALID, E, "unknown K/V type");
    if (in->sm_count < 1 || in->ctas_per_sm < 1 || in->force_parts < 0)
        return fail(PA_ERR_INVALID, E, "sm_count / ctas_per_sm / force_parts out of range");
    if (in->total_len < in->max_len || in->total_len > (uint64_t)in->n_seqs * in->max_len)
        return fail(PA_ERR_INVALID, E, "total_len inconsistent with max_len and n_seqs");
    // T query tokens per sequence: n_seqs * T query rows, each at most max_len
    // long, T * total_len tokens of work at most
    const uint64_t T = in->q_tokens > 1 ? in->q_tokens : 1;
    if (T > 4096)
        return fail(PA_ERR_INVALID, E, "q_tokens %u exceeds 4096", in->q_tokens);
    // a multi-token plan: the one-token plan of the sequences, for T rows each
    if ((in->flags & PA_PLAN_MULTI_TOKEN) && T >= 2 && in->k_type == PA_Q4_0 &&
        in->v_type == PA_Q4_0 && in->d == 256 &&
        (in->hkv == 1 || in->hkv == 2 || in->hkv == 4) && T * (in->hq / in->hkv) <= 24) {
        pa_plan_in one = *in;
        one.q_tokens = 1;
        one.flags = 0;
        pa_plan_t b;
        int rc = pa_plan_quiet(&one, &b);
        if (rc)
            return rc;
        if (b.n_direct) {  // no direct rows in a partitioned multi-token plan
            b.part_tokens = (uint32_t)roundup(in->max_len, TILE);
            b.n_parts = 1;
            b.direct = 1;
            b.n_direct = 0;
            b.n_ctas = in->n_seqs;
        }
        const uint64_t rows = (uint64_t)in->n_seqs * T;
        b.q_tokens = (uint32_t)T;
        b.multi = 1;
        b.part_o_bytes = b.direct ? 0 : rows * in->hq * b.n_parts * in->d * 2ull;
        b.part_ml_bytes = b.direct ? 0 : rows * in->hq * b.n_parts * 8ull;
        b.counter_bytes =
            b.direct ? 0 : rows * pa::merge_counters_per_seq(b.n_parts) * 4ull;
        *out = b;
        return PA_OK;
    }
    const uint64_t rows = (uint64_t)in->n_seqs * T, work = T * in->total_len;
    if (rows > 0x7fffffffull)
        return fail(PA_ERR_RANGE, E, "n_seqs * q_tokens exceeds 2^31 - 1");
    uint64_t part, n_parts, n_direct = 0;
    if (in->max_len == 0) {
        part = TILE;
        n_parts = 1;
    } else if (in->force_parts > 0) {
        part = roundup(cdiv(in->max_len, (uint64_t)in->force_parts), TILE);
        n_parts = cdiv(in->max_len, part);
    } else {
        uint64_t slots = (uint64_t)in->sm_count * (uint64_t)in->ctas_per_sm;
        part = roundup(cdiv(work, slots), TILE);
        if (part < MIN_PART) part = MIN_PART;
        uint64_t cap = roundup(in->max_len, TILE);
        if (part > cap) part = cap;
        // a nearly uniform batch whose rows would round up to more CTAs than
        // slots takes partitions that fit every row's share into one wave
        if (rows * cdiv(in->max_len, part) > slots && rows <= slots &&
            10 * work >= 9 * rows * (uint64_t)in->max_len) {
            part = roundup(cdiv(in->max_len, slots / rows), TILE);
            if (part < MIN_PART) part = MIN_PART;
            if (part > cap) part = cap;
        }
        // any other batch whose grid bound would pass the slots: partitions
        // long enough that ceil(work / part) + rows CTAs fit one wave
        const uint64_t np = cdiv(in->max_len, part);
        const uint64_t bound = rows * np < cdiv(work, part) + rows ? rows * np
                                                                   : cdiv(work, part) + rows;
        if (np > 1 && bound > slots && rows < slots) {
            const uint64_t wide = roundup(cdiv(work, slots - rows), TILE);
            if (wide > part) part = wide < cap ? wide : cap;
        }
        n_parts = cdiv(in->max_len, part);
        // a direct batch wider than the machine with a partial last wave:
        // the full waves stay direct, and the r rows of the last one are
        // split into the partition count np (2..64) that minimises the
        // estimated time of what follows the full waves,
        //   ceil(r * np / slots) waves * (partition tokens + CTA_COST),
        // against max_len + CTA_COST for leaving them whole.  CTA_COST is
        // the fixed work of a CTA (prologue, combine, merge arrival, about
        // 15 us) in tokens streamed at one SM's share of HBM (about 26 ns).
        const uint64_t CTA_COST = 512;
        const uint64_t r = rows % slots;
        if (n_parts == 1 && rows > slots && r > 0) {
            uint64_t best_t = in->max_len + CTA_COST, best_part = 0;
            for (uint64_t np = 2; np <= 64; ++np) {
                uint64_t pr = roundup(cdiv(in->max_len, np), TILE);
                if (pr < MIN_PART) pr = MIN_PART;
                const uint64_t nparts = cdiv(in->max_len, pr);
                if (nparts < 2)
                    break;
                const uint64_t t = cdiv(r * nparts, slots) * (pr + CTA_COST);
                if (t < best_t) {
                    best_t = t;
                    best_part = pr;
                }
            }
            if (best_part) {
                part = best_part;
                n_parts = cdiv(in->max_len, best_part);
                n_direct = rows - r;
            }
        }
    }
    // a stream plan for a batch wider than the machine (see pa.h): equal
    // ranges of the rows' tiles per CTA instead of whole rows in waves
    {
        const uint64_t slots = (uint64_t)in->sm_count * (uint64_t)in->ctas_per_sm;
        const bool shapes = in->k_type == in->v_type &&
                            (in->hkv == 1 || in->hkv == 2 || in->hkv == 4 || in->hkv == 8) &&
                            (in->d == 256 || in->k_type == PA_F16);
        if ((in->flags & PA_PLAN_STREAM_OK) && in->force_parts == 0 && in->max_len > 0 &&
            rows > slots && rows <= 16384 && shapes) {
            const uint64_t bound = cdiv(work + 15 * rows, 16);
            const uint64_t chunk = roundup(cdiv(bound, slots), 2);
            const uint64_t np = cdiv(cdiv(in->max_len, 16), chunk) + 1;
            if (np <= 32) {
                pa_plan_t p;
                memset(&p, 0, sizeof p);
                p.part_tokens = (uint32_t)(16 * chunk);
                p.n_parts = (uint32_t)np;
                p.n_ctas = (uint32_t)(cdiv(bound, chunk) < slots ? cdiv(bound, chunk) : slots);
                p.q_tokens = (uint32_t)T;
                p.stream = 1;
                p.part_o_bytes = rows * in->hq * np * in->d * 2ull;
                p.part_ml_bytes = rows * in->hq * np * 8ull;
                p.counter_bytes = rows * pa::merge_counters_per_seq((uint32_t)np) * 4ull;
                *out = p;
                return PA_OK;
            }
        }
    }
    {
    pa_plan_t p;
    memset(&p, 0, sizeof p);
    p.part_tokens = (uint32_t)part;
    p.n_parts = (uint32_t)n_parts;
    p.direct = n_parts == 1;
    p.q_tokens = (uint32_t)T;
    p.n_direct = (uint32_t)n_direct;
    if (p.direct) {
        p.n_ctas = (uint32_t)rows;
    } else {
        const uint64_t m = rows - n_direct;  // partitioned rows
        uint64_t a = m * n_parts;
        uint64_t b = cdiv(work, part) + m;
        uint64_t n = n_direct + (n_direct || a < b ? a : b);
        if (n > 0x7fffffffull)
            return fail(PA_ERR_RANGE, E, "grid of %llu CTAs exceeds 2^31-1", (unsigned long long)n);
        p.n_ctas = (uint32_t)n;
        p.part_o_bytes = m * in->hq * n_parts * in->d * 2ull;
        p.part_ml_bytes = m * in->hq * n_parts * 8ull;
        p.counter_bytes = m * pa::merge_counters_per_seq((uint32_t)n_parts) * 4ull;
    }
    *out = p;
    }
    return PA_OK;
}

// k_fast.cu -- the fast sm_103a decode kernel (not yet enabled: every shape
// falls back to the plain kernel).
#include "pa_internal.h"

namespace pa {

bool fast_decode_supported(pa_type, pa_type, uint32_t, uint32_t, uint32_t, uint32_t)
{
    return false;
}

int fast_decode_occupancy(pa_type, pa_type, uint32_t, uint32_t, uint32_t, uint32_t,
                          int *ctas_per_sm)
{
    *ctas_per_sm = 1;
    return PA_OK;
}

int launch_fast_decode(const DecodeParams &, pa_type, pa_type, cudaStream_t, const char *entry)
{
    return fail(PA_ERR_INVALID, entry, "fast kernel unavailable for these shapes");
}

}  // namespace pa

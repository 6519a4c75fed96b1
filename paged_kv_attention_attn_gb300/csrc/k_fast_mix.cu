// k_fast_mix.cu -- the fast sm_103a decode kernel for K and V of different
// types (F16, Q8_0, Q4_0; D = 256): the scores of the K type beside the PV of
// the V type in one kernel ("feat: add paged-attention monolithic decode-only
// AR foundation" (lucebox pull 555), Validation: all nine F16 / Q4_0 / Q8_0
// K/V combinations).  Same kernel as k_fast.cu, other instances.
#include "fast_kernel.cuh"

namespace pa {
namespace {

using F16D = F16T<256>;

// Calls f with a default-constructed Mix<K, V> for the pair, or returns
// fallback for a pair that is not mixed.
template <class Fn, class R>
R with_mix(pa_type kt, pa_type vt, R fallback, Fn &&f)
{
    if (kt == PA_F16 && vt == PA_Q8_0)
        return f(Mix<F16D, Q80>{});
    if (kt == PA_F16 && vt == PA_Q4_0)
        return f(Mix<F16D, Q40>{});
    if (kt == PA_Q8_0 && vt == PA_F16)
        return f(Mix<Q80, F16D>{});
    if (kt == PA_Q8_0 && vt == PA_Q4_0)
        return f(Mix<Q80, Q40>{});
    if (kt == PA_Q4_0 && vt == PA_F16)
        return f(Mix<Q40, F16D>{});
    if (kt == PA_Q4_0 && vt == PA_Q8_0)
        return f(Mix<Q40, Q80>{});
    return fallback;
}

}  // namespace

bool fast_mixed_supported(pa_type kt, pa_type vt, uint32_t hkv)
{
    return with_mix(kt, vt, false, [&](auto m) {
        return geometry<decltype(m)>(hkv).warps > 0;
    });
}

int fast_mixed_occupancy(pa_type kt, pa_type vt, uint32_t hkv, int *ctas_per_sm)
{
    return with_mix(kt, vt, (int)PA_ERR_INVALID, [&](auto m) {
        return occupancy_t<decltype(m)>(hkv, ctas_per_sm);
    });
}

int launch_fast_mixed(const DecodeParams &p, pa_type kt, pa_type vt, cudaStream_t st,
                      const char *entry)
{
    return with_mix(kt, vt, fail(PA_ERR_INVALID, entry, "not a mixed K/V type pair"),
                    [&](auto m) { return launch_t<decltype(m)>(p, st, entry); });
}

}  // namespace pa

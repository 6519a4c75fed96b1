// k_fast.cu -- the fast sm_103a decode kernel for K and V of one type (F16
// with D = 128 or 256, Q8_0 and Q4_0 with D = 256), and the dispatch between
// these, the mixed-type instances (k_fast_mix.cu) and the plain kernel.
#include "fast_kernel.cuh"
#include "mt_kernel.cuh"

namespace pa {

bool fast_decode_supported(pa_type kt, pa_type vt, uint32_t d, uint32_t hq, uint32_t hkv,
                           uint32_t block_size)
{
    if (!hkv_ok(hkv) || hq % hkv || hq / hkv > 8 || (block_size != 16 && block_size != 32))
        return false;
    if (kt != vt)
        return d == 256 && fast_mixed_supported(kt, vt, hkv);
    if (kt == PA_Q4_0)
        return d == 256 && geometry<Q40>(hkv).warps > 0;
    if (kt == PA_Q8_0)
        return d == 256 && geometry<Q80>(hkv).warps > 0;
    if (kt == PA_F16)
        return d == 256 ? geometry<F16T<256>>(hkv).warps > 0
                        : d == 128 && geometry<F16T<128>>(hkv).warps > 0;
    return false;
}

int fast_decode_occupancy(pa_type kt, pa_type vt, uint32_t d, uint32_t, uint32_t hkv, uint32_t,
                          int *ctas_per_sm)
{
    if (kt != vt)
        return fast_mixed_occupancy(kt, vt, hkv, ctas_per_sm);
    if (kt == PA_Q4_0)
        return occupancy_t<Q40>(hkv, ctas_per_sm);
    if (kt == PA_Q8_0)
        return occupancy_t<Q80>(hkv, ctas_per_sm);
    return d == 256 ? occupancy_t<F16T<256>>(hkv, ctas_per_sm)
                    : occupancy_t<F16T<128>>(hkv, ctas_per_sm);
}

bool mt_decode_supported(pa_type kt, pa_type vt, uint32_t d, uint32_t hq, uint32_t hkv,
                         uint32_t T)
{
    return mt_supported(kt, vt, d, hq, hkv, T);
}

int launch_fast_decode(const DecodeParams &p, pa_type kt, pa_type vt, cudaStream_t st,
                       const char *entry)
{
    if (p.multi)
        return launch_mt(p, st, entry);
    // TMA slot coordinates are int32: larger pools take the plain kernel
    if (p.n_pool_blocks * p.block_size >= (1ull << 31))
        return launch_plain_decode(p, kt, vt, st, entry);
    if (kt != vt)
        return launch_fast_mixed(p, kt, vt, st, entry);
    if (kt == PA_Q4_0)
        return launch_t<Q40>(p, st, entry);
    if (kt == PA_Q8_0)
        return launch_t<Q80>(p, st, entry);
    if (p.d == 256)
        return launch_t<F16T<256>>(p, st, entry);
    return launch_t<F16T<128>>(p, st, entry);
}

}  // namespace pa

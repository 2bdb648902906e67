// kernels_small.cu -- instantiations of the single-launch dynamic-scale
// kernel (NVFP4 or FP8) for a few decode tokens (nvfp4_small.cuh).
#include "dispatch.h"
#include "nvfp4_small.cuh"

namespace tpar {

namespace {
// One item per thread only: with more, the two-kernel path measured faster.
template <int NR, bool F16, bool FP8>
const void* pick_small(int ipt)
{
    return ipt == 1 ? reinterpret_cast<const void*>(&small_dynamic_kernel<NR, 1, F16, FP8>) : nullptr;
}

template <bool F16, bool FP8>
const void* pick_small_nr(int nr, int ipt)
{
    switch (nr) {
    case 1: return pick_small<1, F16, FP8>(ipt);
    case 2: return pick_small<2, F16, FP8>(ipt);
    case 4: return pick_small<4, F16, FP8>(ipt);
    case 8: return pick_small<8, F16, FP8>(ipt);
    case 16: return pick_small<16, F16, FP8>(ipt);
    default: return nullptr;
    }
}
}  // namespace

const void* small_kernel_for(int nr, int ipt, bool f16, bool fp8)
{
    if (fp8)
        return f16 ? pick_small_nr<true, true>(nr, ipt) : pick_small_nr<false, true>(nr, ipt);
    return f16 ? pick_small_nr<true, false>(nr, ipt) : pick_small_nr<false, false>(nr, ipt);
}

}  // namespace tpar

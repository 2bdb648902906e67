// kernels_small.cu -- instantiations of the single-launch dynamic-scale
// NVFP4 kernel for a few decode tokens (nvfp4_small.cuh).
#include "dispatch.h"
#include "nvfp4_small.cuh"

namespace tpar {

namespace {
template <int NR>
const void* pick_small(int ipt)
{
    switch (ipt) {
    case 1: return reinterpret_cast<const void*>(&nvfp4_small_kernel<NR, 1>);
    case 2: return reinterpret_cast<const void*>(&nvfp4_small_kernel<NR, 2>);
    case 4: return reinterpret_cast<const void*>(&nvfp4_small_kernel<NR, 4>);
    default: return nullptr;
    }
}
}  // namespace

const void* small_kernel_for(int nr, int ipt)
{
    switch (nr) {
    case 1: return pick_small<1>(ipt);
    case 2: return pick_small<2>(ipt);
    case 4: return pick_small<4>(ipt);
    case 8: return pick_small<8>(ipt);
    case 16: return pick_small<16>(ipt);
    default: return nullptr;
    }
}

}  // namespace tpar

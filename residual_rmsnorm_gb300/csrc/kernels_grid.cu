// kernels_grid.cu -- instantiations of the single-launch dynamic-scale NVFP4
// kernel that buffers its rows on chip across a cooperative grid
// (nvfp4_grid.cuh).
#include "dispatch.h"
#include "nvfp4_grid.cuh"

namespace tpar {

namespace {
template <int NR, bool F16>
const void* pick_grid(int vpt)
{
    switch (vpt) {
    case 1: return reinterpret_cast<const void*>(&nvfp4_grid_kernel<NR, 1, F16>);
    case 2: return reinterpret_cast<const void*>(&nvfp4_grid_kernel<NR, 2, F16>);
    default: return nullptr;
    }
}

template <bool F16>
const void* pick_grid_nr(int nr, int vpt)
{
    switch (nr) {
    case 1: return pick_grid<1, F16>(vpt);
    case 2: return pick_grid<2, F16>(vpt);
    case 4: return pick_grid<4, F16>(vpt);
    case 8: return pick_grid<8, F16>(vpt);
    case 16: return pick_grid<16, F16>(vpt);
    default: return nullptr;
    }
}
}  // namespace

const void* grid_kernel_for(int nr, int vpt, bool f16)
{
    return f16 ? pick_grid_nr<true>(nr, vpt) : pick_grid_nr<false>(nr, vpt);
}

}  // namespace tpar

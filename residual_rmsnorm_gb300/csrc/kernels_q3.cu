// kernels_q3.cu -- instantiations of the fused kernel for quantisation
// mode 3 (per-tensor FP8 with a given scale; modes 0-2 are
// in kernels_q0.cu .. kernels_q2.cu). One translation unit per mode so the build
// compiles them in parallel.
#include "dispatch.h"
#include "kernels.cuh"

namespace tpar {

namespace {
template <int NR>
const void* pick(int vpt, bool cluster)
{
    if (cluster) {
        switch (vpt) {
        case 1: return reinterpret_cast<const void*>(&fused_rmsnorm_kernel<NR, 1, true, 3>);
        case 2: return reinterpret_cast<const void*>(&fused_rmsnorm_kernel<NR, 2, true, 3>);
        default: return nullptr;
        }
    }
    switch (vpt) {
    case 1: return reinterpret_cast<const void*>(&fused_rmsnorm_kernel<NR, 1, false, 3>);
    case 2: return reinterpret_cast<const void*>(&fused_rmsnorm_kernel<NR, 2, false, 3>);
    case 4: return reinterpret_cast<const void*>(&fused_rmsnorm_kernel<NR, 4, false, 3>);
    case 8: return reinterpret_cast<const void*>(&fused_rmsnorm_kernel<NR, 8, false, 3>);
    default: return nullptr;
    }
}
}  // namespace

const void* fused_kernel_q3(int nr, int vpt, bool cluster)
{
    switch (nr) {
    case 1: return pick<1>(vpt, cluster);
    case 2: return pick<2>(vpt, cluster);
    case 4: return pick<4>(vpt, cluster);
    case 8: return pick<8>(vpt, cluster);
    case 16: return pick<16>(vpt, cluster);
    default: return nullptr;
    }
}

}  // namespace tpar

// kernels_stream_fp16.cu -- instantiations of the TMA-fed bandwidth kernel
// (stream.cuh) for fp16 tensors.
#include "dispatch.h"
#include "stream.cuh"

namespace tpar {

namespace {
template <int NR, int Q>
const void* pick_stream(int vpt)
{
    switch (vpt) {
    case 1: return reinterpret_cast<const void*>(&stream_rmsnorm_kernel<NR, 1, Q, true>);
    case 2: return reinterpret_cast<const void*>(&stream_rmsnorm_kernel<NR, 2, Q, true>);
    case 4: return reinterpret_cast<const void*>(&stream_rmsnorm_kernel<NR, 4, Q, true>);
    case 8: return reinterpret_cast<const void*>(&stream_rmsnorm_kernel<NR, 8, Q, true>);
    default: return nullptr;
    }
}

template <int Q>
const void* pick_stream_nr(int nr, int vpt)
{
    switch (nr) {
    case 1: return pick_stream<1, Q>(vpt);
    case 2: return pick_stream<2, Q>(vpt);
    case 4: return pick_stream<4, Q>(vpt);
    case 8: return pick_stream<8, Q>(vpt);
    case 16: return pick_stream<16, Q>(vpt);
    default: return nullptr;
    }
}
}  // namespace

const void* stream_kernel_fp16(int qmode, int nr, int vpt)
{
    switch (qmode) {
    case 0: return pick_stream_nr<0>(nr, vpt);
    case 1: return pick_stream_nr<1>(nr, vpt);
    case 2: return pick_stream_nr<2>(nr, vpt);
    default: return nullptr;  // FP8 output is not built into the stream kernel
    }
}

}  // namespace tpar

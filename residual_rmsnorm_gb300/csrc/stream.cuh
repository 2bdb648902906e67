// stream.cuh -- the bandwidth form of the fused epilogue: a persistent,
// warp-specialised kernel fed by TMA bulk copies.
//
// Same arithmetic as fused_rmsnorm_kernel ("Deep Dive: AllReduce and
// AllReduce Fusion in TensorRT-LLM", 6.3 Inside the Fused Kernel: rank sum,
// residual add, store residual_out, RMSNorm, store norm_out, quantise), but
// the inputs reach the SM through the tensor memory accelerator instead of
// per-thread loads:
//   * one CTA per SM strides over rows t = blockIdx.x, + gridDim.x, ...;
//   * warp 0 is the producer: one elected lane streams, in order, the row
//     of every partial and of the residual (d*2 contiguous bytes each) into
//     a ring of shared-memory stages with cp.async.bulk, each completing on
//     the stage's "full" mbarrier;
//   * the other warps consume the stages in the same order, accumulating
//     the row in fp32 registers, and release each stage on its "empty"
//     mbarrier; then they reduce the row's sum of squares (named barrier
//     among consumers only), normalise and store.
// While the consumers reduce and store row t, the producer is already
// filling the ring with row t + gridDim.x, so HBM sees no per-row bubble.
// Every wait is bounded (%globaltimer); an expired wait sets the device
// error word, stops the loops, and the producer drains its own copies.
#pragma once

#include "kernels.cuh"

namespace tpar {

struct StreamArgs {
    FusedArgs f;       // pointers, sizes, epilogue outputs (slice unused)
    int stages;        // ring depth; stage bytes = d * 2
    int consumers;     // consumer threads (multiple of 32), blockDim.x - 32
};

// Shared-memory ring layout: [stages][d] bf16 rows, then 2*stages mbarriers.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// Barrier among the consumer warps only (id 1; the producer never joins).
__device__ __forceinline__ void consumers_sync(int nthreads)
{
    asm volatile("bar.sync 1, %0;" ::"r"(nthreads) : "memory");
}

constexpr uint64_t kStreamWaitNs = 500ull * 1000 * 1000;

template <int NR, int VPT, int QMODE, bool F16>
__global__ void __launch_bounds__(544, 1) stream_rmsnorm_kernel(const __grid_constant__ StreamArgs sa)
{
    extern __shared__ __align__(128) unsigned char ring[];
    const FusedArgs& a = sa.f;
    pdl_wait();
    pdl_launch_dependents();

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int S = sa.stages;
    const int C = sa.consumers;
    const int nvec = a.nvec;
    const uint32_t row_bytes = static_cast<uint32_t>(nvec) * 16u;
    const int nsrc = a.n_ranks + (a.residual ? 1 : 0);  // rows streamed per token
    uint64_t* bars = reinterpret_cast<uint64_t*>(ring + static_cast<size_t>(S) * row_bytes);
    const uint32_t full0 = smem_addr(bars);
    const uint32_t empty0 = smem_addr(bars + S);
    const uint32_t ring0 = smem_addr(ring);

    __shared__ float wsh[2][kMaxRowWarps];  // per-32-vector partial sums of squares
    __shared__ float warp_mx[32];
    __shared__ int abort_flag;   // set by any thread whose bounded wait expired
    __shared__ int stop_sh[2];   // abort_flag as sampled once per row, for a uniform exit

    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full0 + 8u * s, 1);
            mbar_init(empty0 + 8u * s, static_cast<uint32_t>(C / 32));
        }
        abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    if (warp == 0) {
        // ------------------------------------------------ producer
        if (lane == 0) {
            int s = 0;
            uint32_t round = 0;
            int64_t issued = 0;
            bool ok = true;
            for (int64_t t = blockIdx.x; t < a.T && ok; t += gridDim.x) {
                for (int j = 0; j < nsrc && ok; ++j) {
                    const uint32_t full = full0 + 8u * s, empty = empty0 + 8u * s;
                    if (round > 0 && !mbar_wait_parity_bounded(empty, (round - 1) & 1u, kStreamWaitNs)) {
                        ok = false;
                        break;
                    }
                    const uint4* src = (j < a.n_ranks ? a.partials[j] : a.residual) + t * static_cast<int64_t>(nvec);
                    // debug builds check the row read and the stage written; a
                    // skipped copy completes its stage by a plain arrive
                    if (TPAR_IN_RANGE(a.err, t * static_cast<int64_t>(nvec) + nvec - 1, a.n_vec_total) &&
                        TPAR_IN_RANGE(a.err, s, S)) {
                        mbar_arrive_expect_tx(full, row_bytes);
                        bulk_g2s(ring0 + static_cast<uint32_t>(s) * row_bytes, src, row_bytes, full);
                    } else {
                        mbar_arrive(full);
                    }
                    ++issued;
                    if (++s == S) {
                        s = 0;
                        ++round;
                    }
                }
                if (*reinterpret_cast<volatile int*>(&abort_flag))
                    ok = false;
            }
            if (!ok) {
                if (a.err)
                    atomicOr(a.err, TPAR_DEVERR_STREAM_WAIT);
                *reinterpret_cast<volatile int*>(&abort_flag) = 1;
            }
            // Drain: no copy of ours may still be in flight when the CTA exits.
            // The last min(issued, S) stages hold the newest copies.
            const int64_t pending = issued < S ? issued : S;
            for (int64_t k = 0; k < pending; ++k) {
                const int64_t idx = issued - 1 - k;
                const int st = static_cast<int>(idx % S);
                const uint32_t rd = static_cast<uint32_t>(idx / S);
                mbar_wait_parity_bounded(full0 + 8u * st, rd & 1u, kStreamWaitNs);
            }
        }
        return;
    }

    // ---------------------------------------------------- consumers
    const int c = tid - 32;  // consumer index; vectors c + j*C of each row
    const int cwarp = warp - 1;
    const int nwarps = C / 32;
    float g_given = 0.0f;
    if constexpr (QMODE == kQuantGiven)
        g_given = *a.gscale;
    uint4 gam[VPT];
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
        const int v = c + j * C;
        gam[j] = v < nvec ? ld_reuse(a.gamma + v) : make_uint4(0u, 0u, 0u, 0u);
    }
    float amax_local = 0.0f;
    int s = 0;
    uint32_t round = 0;
    bool ok = true;
    int it = 0;
    for (int64_t t = blockIdx.x; t < a.T; t += gridDim.x, ++it) {
        const int64_t rowv = t * static_cast<int64_t>(nvec);
        float h[VPT][8];
#pragma unroll
        for (int j = 0; j < VPT; ++j)
#pragma unroll
            for (int e = 0; e < 8; ++e)
                h[j][e] = 0.0f;
        // rows in the producer's order: partials 0..N-1, then the residual
        for (int src = 0; src < nsrc; ++src) {
            const uint32_t full = full0 + 8u * s, empty = empty0 + 8u * s;
            if (ok && !mbar_wait_parity_bounded(full, round & 1u, kStreamWaitNs)) {
                ok = false;
                if (a.err && lane == 0)
                    atomicOr(a.err, TPAR_DEVERR_STREAM_WAIT);
                *reinterpret_cast<volatile int*>(&abort_flag) = 1;
            }
            const uint4* stage = reinterpret_cast<const uint4*>(ring + static_cast<size_t>(s) * row_bytes);
#pragma unroll
            for (int j = 0; j < VPT; ++j) {
                const int v = c + j * C;
                if (v < nvec) {
                    const uint4 x = stage[v];
                    if (src == 0)
                        unpack8_dt(x, h[j], F16);
                    else
                        add8_dt(x, h[j], F16);
                }
            }
            __syncwarp();
            if (lane == 0)
                mbar_arrive(empty);
            if (++s == S) {
                s = 0;
                ++round;
            }
        }
        const int buf = it & 1;
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            const int v = c + j * C;
            float ss = 0.0f;
            if (v < nvec) {
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    ss = fmaf(h[j][e], h[j][e], ss);
                if (a.out_residual && TPAR_IN_RANGE(a.err, rowv + v, a.n_vec_total))
                    st_v4(a.out_residual + rowv + v, pack8_dt(h[j], F16));
            }
            ss = warp_sum(ss);
            const int w = (j * C + 32 * cwarp) >> 5;
            if (lane == 0 && 32 * w < nvec && TPAR_IN_RANGE(a.err, w, kMaxRowWarps))
                wsh[buf][w] = ss;
        }
        if (c == 0)
            stop_sh[buf] = *reinterpret_cast<volatile int*>(&abort_flag);
        consumers_sync(C);
        const float tot = canonical_row_sum(wsh[buf], (nvec + 31) >> 5, lane);
        const float rinv = rsqrtf(fmaf(tot, a.inv_d, a.eps));
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            const int v = c + j * C;
            emit_vector<QMODE, F16>(a, v < nvec, rowv + v, t, v, h[j], gam[j], rinv, g_given, amax_local);
        }
        if (stop_sh[buf])
            break;  // the same sample for every consumer: all leave together
    }
    if constexpr (QMODE == kQuantAmax) {
        const float m = warp_max(amax_local);
        if (lane == 0)
            warp_mx[cwarp] = m;
        consumers_sync(C);
        if (cwarp == 0) {
            const float cm = warp_max(lane < nwarps ? warp_mx[lane] : 0.0f);
            if (lane == 0 && cm > 0.0f)
                atomicMax(a.amax_bits, __float_as_uint(cm));
        }
    }
}

}  // namespace tpar

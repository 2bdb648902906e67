// nvfp4_grid.cuh -- single-launch fused epilogue with a dynamic NVFP4 global
// scale for batches that fit on chip, across all SMs.
//
// The dynamic scale g = amax(|out_norm|) / (6 * 448) needs every element of
// the tensor before any block is quantised. With a cooperative launch (all
// CTAs resident at once, guaranteed by the launch) one kernel does both
// passes without writing and re-reading out_norm through HBM:
//   1. each CTA runs the fused epilogue ("Deep Dive: AllReduce and AllReduce
//      Fusion in TensorRT-LLM", 6.3: rank sum, residual add, store
//      residual_out, RMSNorm, store norm_out) on its rows t = blockIdx.x,
//      + gridDim.x, ..., keeping each row's emitted bf16 values in shared
//      memory and their absolute maximum in a register;
//   2. the CTA folds its maximum into the workspace amax (one atomic) and
//      arrives at a grid barrier (one counter), waiting for the others with
//      a %globaltimer bound;
//   3. every CTA reads g = amax / 2688 and quantises its rows from shared
//      memory (6.5): E4M3 block scales and E2M1 codes, exactly as the
//      two-kernel path does; the last CTA out zeroes the workspace.
// Rows, the sum-of-squares order and the quantiser arithmetic are those of
// the row kernel and of phase B, so the results are bit-identical to the
// two-kernel path.
#pragma once

#include "kernels.cuh"

namespace tpar {

struct GridArgs {
    FusedArgs f;   // inputs, outputs (out_norm may be null), codes, scales, T, nvec
    float* gscale; // output: g
    uint32_t* ws;  // workspace: [1] amax bits, [0] exit count, [3] barrier arrivals
    int rows;      // rows per CTA buffered in shared memory (ceil(T / gridDim.x))
};

constexpr int kGridSmemBudget = 200 * 1024;        // bytes of buffered rows per CTA
constexpr int kGridMaxVpt = 2;                     // vectors per thread: d <= 8192
constexpr uint64_t kGridWaitNs = 200ull * 1000 * 1000;

template <int NR, int VPT, bool F16>
__global__ void __launch_bounds__(fused_max_threads(NR, VPT, false))
    nvfp4_grid_kernel(const __grid_constant__ GridArgs ga)
{
    extern __shared__ __align__(16) uint4 ybuf[];  // [rows][nvec] emitted values
    const FusedArgs& a = ga.f;
    pdl_wait();
    pdl_launch_dependents();

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int nwarps = blockDim.x >> 5;
    const int B = static_cast<int>(blockDim.x);
    const int nvec = a.nvec;
    const int64_t G = gridDim.x;
    const int nW = (nvec + 31) >> 5;
    [[maybe_unused]] const int64_t buf_vecs = static_cast<int64_t>(ga.rows) * nvec;  // checked by debug builds
    __shared__ float wsh[2][kMaxRowWarps];
    __shared__ float red[32];
    __shared__ float g_sh;

    uint4 gam[VPT];
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
        const int v = tid + j * B;
        gam[j] = (v < nvec && TPAR_IN_RANGE(a.err, v, a.nvec)) ? ld_reuse(a.gamma + v) : make_uint4(0u, 0u, 0u, 0u);
    }
    float amax_local = 0.0f;

    // ---- 1. the fused epilogue of this CTA's rows (the row kernel's order)
    int k = 0;
    for (int64_t t = blockIdx.x; t < a.T; t += G, ++k) {
        const int64_t rowv = t * static_cast<int64_t>(nvec);
        float h[VPT][8];
        float ss[VPT];
        // loads in groups of G vectors, every load of a group issued first
        // (the row kernel's grouping: bounded registers for many ranks)
        constexpr int GRP = (NR >= 16 || VPT == 1) ? 1 : 2;
#pragma unroll
        for (int j0 = 0; j0 < VPT; j0 += GRP) {
            uint4 x[GRP][NR];
            uint4 rv[GRP];
#pragma unroll
            for (int jj = 0; jj < GRP; ++jj) {
                const int v = tid + (j0 + jj) * B;
                if (v < nvec) {
                    const bool in = TPAR_IN_RANGE(a.err, rowv + v, a.n_vec_total);
#pragma unroll
                    for (int r = 0; r < NR; ++r)
                        if (r < a.n_ranks)
                            x[jj][r] = in ? ld_stream(a.partials[r] + rowv + v) : make_uint4(0u, 0u, 0u, 0u);
                    rv[jj] = (a.residual && in) ? ld_coherent(a.residual + rowv + v) : make_uint4(0u, 0u, 0u, 0u);
                }
            }
#pragma unroll
            for (int jj = 0; jj < GRP; ++jj) {
                const int j = j0 + jj;
                const int v = tid + j * B;
                ss[j] = 0.0f;
                if (v < nvec) {
                    unpack8_dt(x[jj][0], h[j], F16);
#pragma unroll
                    for (int r = 1; r < NR; ++r)
                        if (r < a.n_ranks)
                            add8_dt(x[jj][r], h[j], F16);
                    if (a.residual)
                        add8_dt(rv[jj], h[j], F16);
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        ss[j] = fmaf(h[j][e], h[j][e], ss[j]);
                    if (a.out_residual && TPAR_IN_RANGE(a.err, rowv + v, a.n_vec_total))
                        st_v4(a.out_residual + rowv + v, pack8_dt(h[j], F16));
                } else {
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        h[j][e] = 0.0f;
                }
            }
        }
        const int buf = k & 1;
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            const float s = warp_sum(ss[j]);
            const int w = (j * B + 32 * warp) >> 5;
            if (lane == 0 && 32 * w < nvec && TPAR_IN_RANGE(a.err, w, kMaxRowWarps))
                wsh[buf][w] = s;
        }
        __syncthreads();
        const float tot = canonical_row_sum(wsh[buf], nW, lane);
        const float rinv = rsqrtf(fmaf(tot, a.inv_d, a.eps));
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            const int v = tid + j * B;
            if (v < nvec) {
                float gm[8], y[8];
                unpack8_dt(gam[j], gm, F16);
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    y[e] = h[j][e] * rinv * gm[e];
                const uint4 yb = pack8_dt(y, F16);
                if (a.out_norm && TPAR_IN_RANGE(a.err, rowv + v, a.n_vec_total))
                    st_v4(a.out_norm + rowv + v, yb);
                if (TPAR_IN_RANGE(a.err, static_cast<int64_t>(k) * nvec + v, buf_vecs))
                    ybuf[static_cast<int64_t>(k) * nvec + v] = yb;
                float yq[8];
                unpack8_dt(yb, yq, F16);
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    amax_local = fmaxf(amax_local, fabsf(yq[e]));
            }
        }
    }

    // ---- 2. grid-wide amax: one atomic per CTA, then a bounded grid barrier
    {
        const float m = warp_max(amax_local);
        if (lane == 0)
            red[warp] = m;
    }
    __syncthreads();
    if (tid == 0) {
        float c = 0.0f;
        for (int w = 0; w < nwarps; ++w)
            c = fmaxf(c, red[w]);
        if (c > 0.0f)
            atomicMax(ga.ws + 1, __float_as_uint(c));  // |y| >= 0 orders like its bits
        __threadfence();
        atomicAdd(ga.ws + 3, 1u);
        const uint64_t t0 = global_ns();
        const uint32_t arrivals = static_cast<uint32_t>(G + TPAR_EXTRA_WAIT(a));
        while (*reinterpret_cast<volatile uint32_t*>(ga.ws + 3) < arrivals) {
            if (global_ns() - t0 > kGridWaitNs) {
                if (a.err)
                    atomicOr(a.err, TPAR_DEVERR_GRID_WAIT);
                break;
            }
            __nanosleep(64);
        }
        __threadfence();
        const float g = __fdiv_rn(__uint_as_float(*reinterpret_cast<volatile uint32_t*>(ga.ws + 1)), 2688.0f);
        g_sh = g;
        if (blockIdx.x == 0)
            *ga.gscale = g;
    }
    __syncthreads();
    const float g = g_sh;

    // ---- 3. quantise the buffered rows (a 16-element block = the vectors of
    // a lane pair, as in the fused given-scale pass)
    k = 0;
    for (int64_t t = blockIdx.x; t < a.T; t += G, ++k) {
        const int64_t rowv = t * static_cast<int64_t>(nvec);
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            const int v = tid + j * B;
            const bool valid = v < nvec;
            float yq[8];
            if (valid && TPAR_IN_RANGE(a.err, static_cast<int64_t>(k) * nvec + v, buf_vecs)) {
                unpack8_dt(ybuf[static_cast<int64_t>(k) * nvec + v], yq, F16);
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    yq[e] = 0.0f;
            }
            float bmax = 0.0f;
#pragma unroll
            for (int e = 0; e < 8; ++e)
                bmax = fmaxf(bmax, fabsf(yq[e]));
            bmax = fmaxf(bmax, __shfl_xor_sync(0xffffffffu, bmax, 1));
            if (valid) {
                const int64_t gv = rowv + v;
                uint32_t sbyte;
                const float inv = nvfp4_block_scale(g, bmax, sbyte);
                float q[8];
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    q[e] = __fmul_rn(yq[e], inv);
                if (TPAR_IN_RANGE(a.err, gv, a.n_vec_total))
                    st_u32(a.codes + gv, e2m1x8_from_f32(q));
                const int64_t si = scale_index(a.sf_tiles, gv >> 1, t, v);
                if ((gv & 1) == 0 && TPAR_IN_RANGE(a.err, si, a.n_scales))
                    st_u8(a.scales + si, sbyte);
            }
        }
    }

    // ---- the last CTA to have read the amax zeroes the workspace
    if (tid == 0) {
        __threadfence();
        if (atomicAdd(ga.ws, 1u) == static_cast<uint32_t>(G) - 1) {
            ga.ws[0] = 0u;
            ga.ws[3] = 0u;
            ga.ws[1] = 0u;
        }
    }
}

}  // namespace tpar

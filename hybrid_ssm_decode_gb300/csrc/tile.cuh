// Tile split shared by the Mamba-2 and Gated DeltaNet kernels.
//
// One thread block per (sequence, head) tile of an FP32 state with P rows and
// N contiguous columns (Mamba-2: P x N; Gated DeltaNet: d_v x d_k). Each
// thread holds 8 float4: thread t owns columns 4*(t % (N/4)) .. +3 of rows
// t/(N/4) + j*(P/8), j = 0..7. A row's threads are adjacent lanes, so a
// row-dot is a segmented warp reduction.
#pragma once

#include "common.cuh"

namespace rssm {

template <int P_, int N_>
struct Tile {
    static constexpr int P = P_, N = N_;
    static constexpr int kThreads = P * N / 32;  // 8 float4 per thread
    static constexpr int TPR = N / 4;            // threads per state row
    static constexpr int RPP = kThreads / TPR;   // rows per pass
    static constexpr int J = 8;
    static constexpr int kWarps = kThreads / 32;
    static_assert(P == RPP * J, "tile split");
    static_assert(TPR >= 8 && TPR <= 32, "row split");
    static_assert(kThreads >= P && kThreads >= N, "one thread per row/column at least");
};

template <class L>
__device__ __forceinline__ void load_state(float4 (&hv)[8], const float* tile_base, int row0,
                                           int col4, uint64_t pol) {
    const float4* src = reinterpret_cast<const float4*>(tile_base);
#pragma unroll
    for (int j = 0; j < 8; ++j) hv[j] = ld_stream(src + (row0 + j * L::RPP) * L::TPR + col4, pol);
}

template <class L>
__device__ __forceinline__ void store_state(const float4 (&hv)[8], float* tile_base, int row0,
                                            int col4) {
    float4* dst = reinterpret_cast<float4*>(tile_base);
#pragma unroll
    for (int j = 0; j < 8; ++j) dst[(row0 + j * L::RPP) * L::TPR + col4] = hv[j];
}

__device__ __forceinline__ void store_out(void* y, size_t idx, float v, bool f32) {
    if (f32) reinterpret_cast<float*>(y)[idx] = v;
    else reinterpret_cast<__nv_bfloat16*>(y)[idx] = __float2bfloat16_rn(v);
}

// Row-dot of the thread's 8 float4 with cv, reduced over the row's lanes and
// written through `emit(row, value)` by one lane per row.
template <class L, class Emit>
__device__ __forceinline__ void row_dots(float (&part)[8], int lane, int row0, Emit emit) {
    float rs = group_reduce_multi<8, L::TPR>(part, lane);
    constexpr int kLanesPerValue = L::TPR / 8;
    if ((lane % kLanesPerValue) == 0) {
        const int jj = (lane % L::TPR) / kLanesPerValue;
        emit(row0 + jj * L::RPP, rs);
    }
}

// Fold m records into the thread's slice of the checkpoint:
//   h <- gamma h + sum_i cf_i x_i B_i^T,  cf_i = dt_i prod_{j>i} a_j
// sB [m][N] holds B_i, sX [m][P] holds cf_i x_i (both FP32, shared memory).
template <class L>
__device__ __forceinline__ void fold_records(float4 (&hv)[8], const float* sB, const float* sX,
                                             int m, float gamma, int row0, int col4) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        hv[j].x *= gamma; hv[j].y *= gamma; hv[j].z *= gamma; hv[j].w *= gamma;
    }
    for (int i = 0; i < m; ++i) {
        const float4 bv = *reinterpret_cast<const float4*>(sB + i * L::N + col4 * 4);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float xw = sX[i * L::P + row0 + j * L::RPP];
            hv[j].x = fmaf(xw, bv.x, hv[j].x);
            hv[j].y = fmaf(xw, bv.y, hv[j].y);
            hv[j].z = fmaf(xw, bv.z, hv[j].z);
            hv[j].w = fmaf(xw, bv.w, hv[j].w);
        }
    }
}

}  // namespace rssm

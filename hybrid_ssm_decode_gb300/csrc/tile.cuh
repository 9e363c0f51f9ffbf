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

// Suffix sums of dt over the records of a window, on one warp. Lane i < m
// holds dt_i (record i, oldest first). Returns the decay of record i,
// exp(A * sum_{i<j<m} dt_j) (the product of a_j over the later records), and
// sets gamma = exp(A * sum_{j<m} dt_j), the decay of the checkpoint.
__device__ __forceinline__ float window_decay(float dt_i, int lane, int m, float A, float& gamma) {
    float suf = (lane < m) ? dt_i : 0.f;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        float o = __shfl_down_sync(0xffffffffu, suf, off);
        if (lane + off < 32) suf += o;
    }
    float excl = __shfl_down_sync(0xffffffffu, suf, 1);
    if (lane == 31) excl = 0.f;
    gamma = expf(A * __shfl_sync(0xffffffffu, suf, 0));
    return expf(A * excl);
}

// ---------------------------------------------------------------------------
// Read copy writer (the Turkish page, section "Kuantizasyon hatasinin
// sinirlandirilmasi": a low-precision copy serves the reads). It quantises the
// thread-distributed tile `hv` (value j of a thread sits in row row_of(j)).
// `sync` is the barrier of the threads that share the tile (a block or a
// named group).
//   FP8:   s = amax/448, code = E4M3(h * (1/s))
//   NVFP4: s = amax/2688; per 16 consecutive columns, bs = E4M3(bmax * (1/(6 s))),
//          code = E2M1(h * (1/(bs s))), two codes per byte, even element low
//          nibble.
// Every step is IEEE round-to-nearest in float32, so the codes are
// reproducible bit for bit from the FP32 tile.
// ---------------------------------------------------------------------------
// With WB (write-back) the values in hv are replaced by the stored ones
// (codes decoded times their scales), for a copy made from a stored tile.
template <class L, int RF, bool WB = false, class Sync, class RowOf, class ChunkOf, int J>
__device__ __forceinline__ void write_read_copy(float4 (&hv)[J], uint8_t* codes_tile,
                                                uint8_t* bscale_tile, float* tscale_out,
                                                float* s_red, int t, int lane, int warp,
                                                RowOf row_of, ChunkOf chunk_of, Sync sync) {
    float mx = 0.f;
#pragma unroll
    for (int j = 0; j < J; ++j)
        mx = fmaxf(mx, fmaxf(fmaxf(fabsf(hv[j].x), fabsf(hv[j].y)),
                             fmaxf(fabsf(hv[j].z), fabsf(hv[j].w))));
    mx = warp_max(mx);
    sync();  // s_red may hold an earlier reduction
    if (lane == 0) s_red[warp] = mx;
    sync();
    float amax = 0.f;
#pragma unroll
    for (int w = 0; w < L::kWarps; ++w) amax = fmaxf(amax, s_red[w]);

    if (RF == RSSM_READ_FP8) {
        const float s = __fdiv_rn(amax, 448.f);
        const float r = (s != 0.f) ? __frcp_rn(s) : 0.f;
#pragma unroll
        for (int j = 0; j < J; ++j) {
            uint32_t w = 0;
            if (s != 0.f) {
                w = static_cast<uint32_t>(e4m3x2(__fmul_rn(hv[j].x, r), __fmul_rn(hv[j].y, r))) |
                    (static_cast<uint32_t>(e4m3x2(__fmul_rn(hv[j].z, r), __fmul_rn(hv[j].w, r))) << 16);
            }
            reinterpret_cast<uint32_t*>(codes_tile)[row_of(j) * (L::N / 4) + chunk_of(j)] = w;
            if (WB) {
                const float2 lo = e4m3x2_to_f2(static_cast<uint16_t>(w & 0xFFFFu));
                const float2 hi = e4m3x2_to_f2(static_cast<uint16_t>(w >> 16));
                hv[j] = make_float4(__fmul_rn(lo.x, s), __fmul_rn(lo.y, s), __fmul_rn(hi.x, s), __fmul_rn(hi.y, s));
            }
        }
        if (t == 0) *tscale_out = s;
    } else {
        const float st = __fdiv_rn(amax, 2688.f);
        const float st6 = __fmul_rn(6.f, st);
        const float r6 = (st6 != 0.f) ? __frcp_rn(st6) : 0.f;   // one reciprocal per tile
#pragma unroll
        for (int j = 0; j < J; ++j) {
            float bm = fmaxf(fmaxf(fabsf(hv[j].x), fabsf(hv[j].y)), fmaxf(fabsf(hv[j].z), fabsf(hv[j].w)));
            bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 1));
            bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 2));
            const uint32_t bs = (st6 == 0.f) ? 0u : (e4m3x2(__fmul_rn(bm, r6), 0.f) & 0xFFu);
            const float es = __fmul_rn(e4m3_to_f(bs), st);
            uint32_t code = 0;
            if (es != 0.f) {
                const float r = __frcp_rn(es);
                code = e2m1x2(__fmul_rn(hv[j].x, r), __fmul_rn(hv[j].y, r)) |
                       (e2m1x2(__fmul_rn(hv[j].z, r), __fmul_rn(hv[j].w, r)) << 8);
            }
            const int row = row_of(j);
            reinterpret_cast<uint16_t*>(codes_tile)[row * (L::N / 4) + chunk_of(j)] = static_cast<uint16_t>(code);
            if ((chunk_of(j) & 3) == 0) bscale_tile[row * (L::N / 16) + (chunk_of(j) >> 2)] = static_cast<uint8_t>(bs);
            if (WB) {
                const float2 lo = e2m1x2_to_f2(code & 0xFFu);
                const float2 hi = e2m1x2_to_f2((code >> 8) & 0xFFu);
                hv[j] = make_float4(__fmul_rn(lo.x, es), __fmul_rn(lo.y, es), __fmul_rn(hi.x, es), __fmul_rn(hi.y, es));
            }
        }
        if (t == 0) *tscale_out = st;
    }
}

// Suffix products of alpha over the records of a window, on one warp. Lane
// j < m holds alpha_j. Returns rho_j = prod_{j<l<m} alpha_l and sets
// gamma = prod_{l<m} alpha_l.
__device__ __forceinline__ float window_rho(float al, int lane, int m, float& gamma) {
    float suf = (lane < m) ? al : 1.f;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        float o = __shfl_down_sync(0xffffffffu, suf, off);
        if (lane + off < 32) suf *= o;
    }
    float excl = __shfl_down_sync(0xffffffffu, suf, 1);
    if (lane == 31) excl = 1.f;
    gamma = __shfl_sync(0xffffffffu, suf, 0);
    return excl;
}

}  // namespace rssm

// Mamba-2 decode kernels: the conventional step, the snapshot-rollback
// baseline and the read-copy quantiser. The replay kernels are in
// m2_replay_tma.cu (one token), m2_draft_tma.cu (drafts) and m2_commit_tma.cu
// (commit and flush).
//
// Method: "ReplaySSM beschleunigt das Decoding von Hybridmodellen durch
// Caching der Eingaben statt des Zustands", section "Wie es funktioniert";
// "NVIDIA ve Dao AI Lab, ... ReplaySSM'i sundu", sections "ReplaySSM nasil
// calisir?" and "Durum trafigini azaltma ve rollback'in basitlestirilmesi".
//
// One thread block per (sequence b, head h) tile. The FP32 state h[P][N]
// (N contiguous) is split so that each thread holds 8 float4: thread t owns
// columns 4*(t % (N/4)) .. +3 of rows t/(N/4) + j*(P/8), j = 0..7. A row's
// threads are adjacent lanes, so a row-dot is a segmented warp reduction.
#include <algorithm>

#include "tile.cuh"

namespace rssm {
namespace {

// ---------------------------------------------------------------------------
// Conventional decode step (the in-build baseline): load the state, decay and
// update it, compute the output, store the state ("Wie es funktioniert",
// first paragraph).
// ---------------------------------------------------------------------------
template <class L, typename TI>
__global__ void __launch_bounds__(L::kThreads) m2_conv_step_kernel(const M2Args a, const int out_f32) {
    constexpr int P = L::P, N = L::N;
    const int tile = blockIdx.x;
    const int b = tile / a.H, hh = tile - b * a.H;
    const int g = hh / (a.H / a.G);
    const int t = threadIdx.x, lane = t & 31;
    const int col4 = t % L::TPR, row0 = t / L::TPR;
    const uint64_t pol = l2_evict_first();
    const size_t tile_off = static_cast<size_t>(tile) * P * N;

    float4 hv[8];
    load_state<L>(hv, a.ckpt + tile_off, row0, col4, pol);

    const TI* xt = reinterpret_cast<const TI*>(a.x) + (static_cast<size_t>(b) * a.H + hh) * P;
    const TI* Bt = reinterpret_cast<const TI*>(a.Bm) + (static_cast<size_t>(b) * a.G + g) * N;
    const TI* Ct = reinterpret_cast<const TI*>(a.C) + (static_cast<size_t>(b) * a.G + g) * N;
    const float dtf = to_f(reinterpret_cast<const TI*>(a.dt)[static_cast<size_t>(b) * a.H + hh]);
    const float decay = expf(dtf * a.A[hh]);
    const float4 bv = load4(Bt + col4 * 4);
    const float4 cv = load4(Ct + col4 * 4);

    float part[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const float dx = dtf * to_f(xt[row0 + j * L::RPP]);
        hv[j].x = fmaf(decay, hv[j].x, dx * bv.x);
        hv[j].y = fmaf(decay, hv[j].y, dx * bv.y);
        hv[j].z = fmaf(decay, hv[j].z, dx * bv.z);
        hv[j].w = fmaf(decay, hv[j].w, dx * bv.w);
        part[j] = dot4(hv[j], cv);
    }
    store_state<L>(hv, a.ckpt + tile_off, row0, col4);
    const float Dh = a.D[hh];
    const size_t ybase = (static_cast<size_t>(b) * a.H + hh) * P;
    row_dots<L>(part, lane, row0, [&](int r, float v) {
        store_out(a.y, ybase + r, fmaf(Dh, to_f(xt[r]), v), out_f32 != 0);
    });
}

// ---------------------------------------------------------------------------
// Quantised-recurrence baseline ("NVIDIA ve Dao AI Lab, ... ReplaySSM'i
// sundu", section "Kuantizasyon hatasinin sinirlandirilmasi": a quantised
// state recurs, so its rounding error accumulates with the sequence length).
// The conventional step with the state itself stored as FP8 or NVFP4 tiles:
// dequantise, decay and update in FP32, output from the updated FP32 values,
// quantise (the read-copy writer's format and rounding) and store the codes.
// It is the comparison point for the read copy, whose recurrence stays on the
// FP32 checkpoint.
// ---------------------------------------------------------------------------
template <class L, typename TI, int RF>
__global__ void __launch_bounds__(L::kThreads) m2_qconv_step_kernel(const M2Args a, const int out_f32) {
    constexpr int P = L::P, N = L::N;
    __shared__ float s_red[L::kWarps];
    const int tile = blockIdx.x;
    const int b = tile / a.H, hh = tile - b * a.H;
    const int g = hh / (a.H / a.G);
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const int col4 = t % L::TPR, row0 = t / L::TPR;
    const size_t tile_off = static_cast<size_t>(tile) * P * N;
    uint8_t* codes = a.rc_codes + (RF == RSSM_READ_FP8 ? tile_off : tile_off / 2);
    uint8_t* bsc = (RF == RSSM_READ_NVFP4) ? a.rc_bscale + tile_off / 16 : nullptr;
    const float ts = a.rc_tscale[tile];

    // dequantise this thread's values: code x (block scale x) tile scale
    float4 hv[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const int row = row0 + j * L::RPP;
        const int idx = row * L::TPR + col4;
        if (RF == RSSM_READ_FP8) {
            const uint32_t u = reinterpret_cast<const uint32_t*>(codes)[idx];
            const float2 lo = e4m3x2_to_f2(static_cast<uint16_t>(u & 0xFFFFu));
            const float2 hi = e4m3x2_to_f2(static_cast<uint16_t>(u >> 16));
            hv[j] = make_float4(lo.x * ts, lo.y * ts, hi.x * ts, hi.y * ts);
        } else {
            const uint32_t u = reinterpret_cast<const uint16_t*>(codes)[idx];
            const float es = __fmul_rn(e4m3_to_f(bsc[row * (N / 16) + (col4 >> 2)]), ts);
            const float2 lo = e2m1x2_to_f2(u & 0xFFu);
            const float2 hi = e2m1x2_to_f2((u >> 8) & 0xFFu);
            hv[j] = make_float4(lo.x * es, lo.y * es, hi.x * es, hi.y * es);
        }
    }

    const TI* xt = reinterpret_cast<const TI*>(a.x) + (static_cast<size_t>(b) * a.H + hh) * P;
    const TI* Bt = reinterpret_cast<const TI*>(a.Bm) + (static_cast<size_t>(b) * a.G + g) * N;
    const TI* Ct = reinterpret_cast<const TI*>(a.C) + (static_cast<size_t>(b) * a.G + g) * N;
    const float dtf = to_f(reinterpret_cast<const TI*>(a.dt)[static_cast<size_t>(b) * a.H + hh]);
    const float decay = expf(dtf * a.A[hh]);
    const float4 bv = load4(Bt + col4 * 4);
    const float4 cv = load4(Ct + col4 * 4);

    float part[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const float dx = dtf * to_f(xt[row0 + j * L::RPP]);
        hv[j].x = fmaf(decay, hv[j].x, dx * bv.x);
        hv[j].y = fmaf(decay, hv[j].y, dx * bv.y);
        hv[j].z = fmaf(decay, hv[j].z, dx * bv.z);
        hv[j].w = fmaf(decay, hv[j].w, dx * bv.w);
        part[j] = dot4(hv[j], cv);
    }
    const float Dh = a.D[hh];
    const size_t ybase = (static_cast<size_t>(b) * a.H + hh) * P;
    row_dots<L>(part, lane, row0, [&](int r, float v) {
        store_out(a.y, ybase + r, fmaf(Dh, to_f(xt[r]), v), out_f32 != 0);
    });
    // every thread has read its codes and the scales before the writer's
    // first barrier, so the tile is rewritten in place
    write_read_copy<L, RF>(hv, codes, bsc, a.rc_tscale + tile, s_red, t, lane, warp,
                           [&](int j) { return row0 + j * L::RPP; }, [&](int) { return col4; },
                           [] { __syncthreads(); });
}

// Snapshot baseline for drafts: T conventional updates from the live state,
// a full-state snapshot after each; the live state is not written.
template <class L, typename TI>
__global__ void __launch_bounds__(L::kThreads) m2_snap_draft_kernel(const M2Args a, const int out_f32) {
    constexpr int P = L::P, N = L::N;
    const int tile = blockIdx.x;
    const int b = tile / a.H, hh = tile - b * a.H;
    const int g = hh / (a.H / a.G);
    const int t = threadIdx.x, lane = t & 31;
    const int col4 = t % L::TPR, row0 = t / L::TPR;
    const int T = a.T;
    const uint64_t pol = l2_evict_first();
    const size_t tile_off = static_cast<size_t>(tile) * P * N;
    const size_t state_elems = static_cast<size_t>(a.B) * a.H * P * N;

    float4 hv[8];
    load_state<L>(hv, a.ckpt + tile_off, row0, col4, pol);
    const float A = a.A[hh], Dh = a.D[hh];
    for (int tau = 0; tau < T; ++tau) {
        const TI* xt = reinterpret_cast<const TI*>(a.x) + ((static_cast<size_t>(b) * T + tau) * a.H + hh) * P;
        const TI* Bt = reinterpret_cast<const TI*>(a.Bm) + ((static_cast<size_t>(b) * T + tau) * a.G + g) * N;
        const TI* Ct = reinterpret_cast<const TI*>(a.C) + ((static_cast<size_t>(b) * T + tau) * a.G + g) * N;
        const float dtf = to_f(reinterpret_cast<const TI*>(a.dt)[(static_cast<size_t>(b) * T + tau) * a.H + hh]);
        const float decay = expf(dtf * A);
        const float4 bv = load4(Bt + col4 * 4);
        const float4 cv = load4(Ct + col4 * 4);
        float part[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float dx = dtf * to_f(xt[row0 + j * L::RPP]);
            hv[j].x = fmaf(decay, hv[j].x, dx * bv.x);
            hv[j].y = fmaf(decay, hv[j].y, dx * bv.y);
            hv[j].z = fmaf(decay, hv[j].z, dx * bv.z);
            hv[j].w = fmaf(decay, hv[j].w, dx * bv.w);
            part[j] = dot4(hv[j], cv);
        }
        store_state<L>(hv, a.snap + tau * state_elems + tile_off, row0, col4);
        const size_t ybase = ((static_cast<size_t>(b) * T + tau) * a.H + hh) * P;
        row_dots<L>(part, lane, row0, [&](int r, float v) {
            store_out(a.y, ybase + r, fmaf(Dh, to_f(xt[r]), v), out_f32 != 0);
        });
    }
}

// Snapshot restore: live state <- snapshot a_b (state after a_b drafts).
template <class L>
__global__ void __launch_bounds__(L::kThreads) m2_snap_restore_kernel(const M2Args a) {
    constexpr int P = L::P, N = L::N;
    const int tile = blockIdx.x;
    const int b = tile / a.H, hh = tile - b * a.H;
    const int t = threadIdx.x;
    int acc = a.accepted[b];
    if (acc < 0 || acc > a.T) {
        if (t == 0 && hh == 0) report_error(a.err, RSSM_DEV_ACCEPTED_RANGE, b, acc);
        return;
    }
    if (acc == 0) return;
    const size_t state_elems = static_cast<size_t>(a.B) * a.H * P * N;
    const size_t tile_off = static_cast<size_t>(tile) * P * N;
    const float4* src = reinterpret_cast<const float4*>(a.snap + (acc - 1) * state_elems + tile_off);
    float4* dst = reinterpret_cast<float4*>(a.ckpt + tile_off);
    const uint64_t pol = l2_evict_first();
#pragma unroll
    for (int j = 0; j < 8; ++j) dst[t + j * L::kThreads] = ld_stream(src + t + j * L::kThreads, pol);
}

// ---------------------------------------------------------------------------
// Standalone read-copy writer (create, and the bit-exactness check).
// ---------------------------------------------------------------------------
// One copy tile of the standalone writer, on one block.
template <class L, int RF, typename TS>
__device__ __forceinline__ void quantize_tile(const TS* src, uint8_t* codes, uint8_t* bscale, float* tscale,
                                              int64_t tile) {
    __shared__ float s_red[L::kWarps];
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const int col4 = t % L::TPR, row0 = t / L::TPR;
    const size_t n_el = static_cast<size_t>(L::P) * L::N;
    const size_t tile_off = static_cast<size_t>(tile) * n_el;
    float4 hv[8];
    if constexpr (sizeof(TS) == 4) {
        load_state<L>(hv, src + tile_off, row0, col4, l2_evict_first());
    } else {
        const uint2* s2 = reinterpret_cast<const uint2*>(src + tile_off);
#pragma unroll
        for (int j = 0; j < 8; ++j) hv[j] = f16x4_to_f32(s2[(row0 + j * L::RPP) * L::TPR + col4]);
    }
    uint8_t* ct = codes + (RF == RSSM_READ_FP8 ? tile_off : tile_off / 2);
    uint8_t* bt = (RF == RSSM_READ_NVFP4) ? bscale + tile * (n_el / 16) : nullptr;
    write_read_copy<L, RF>(hv, ct, bt, tscale + tile, s_red, t, lane, warp,
                           [&](int j) { return row0 + j * L::RPP; }, [&](int) { return col4; },
                           [] { __syncthreads(); });
}

// counts != nullptr: only the copy tiles whose (sequence, head) record count
// is `mark` (the tiles that a flush-only launch of this step folded) are
// written; `per` copy tiles share one count (the 64-row halves of a GDN tile).
// Block q takes tiles q, q + grid, ... A filtered launch has a few blocks
// per SM: each thread of a block reads the count of one of the block's next
// kThreads tiles, the selected ones are listed in shared memory, and the
// block quantises the list (so the skipped tiles cost no serial count read).
template <class L, int RF, typename TS>
__global__ void __launch_bounds__(L::kThreads)
quantize_kernel(const TS* src, uint8_t* codes, uint8_t* bscale, float* tscale, const int32_t* counts, int mark,
                int per, int64_t tiles) {
    __shared__ int s_list[L::kThreads];
    __shared__ int s_n;
    const int64_t stride = gridDim.x;
    for (int64_t base = blockIdx.x; base < tiles; base += stride * L::kThreads) {
        if (threadIdx.x == 0) s_n = 0;
        __syncthreads();
        const int64_t mine = base + threadIdx.x * stride;
        if (mine < tiles && (counts == nullptr || counts[mine / per] == mark))
            s_list[atomicAdd(&s_n, 1)] = threadIdx.x;
        __syncthreads();
        const int n = s_n;
        for (int i = 0; i < n; ++i) quantize_tile<L, RF, TS>(src, codes, bscale, tscale, base + s_list[i] * stride);
        __syncthreads();   // s_n and s_list are rewritten next
    }
}

// ---------------------------------------------------------------------------
// dispatch
// ---------------------------------------------------------------------------
template <template <class> class F, class... Args>
cudaError_t with_tile(int P, int N, bool* supported, Args&&... args) {
    *supported = true;
    if (P == 64 && N == 128) return F<Tile<64, 128>>::run(args...);
    if (P == 64 && N == 64) return F<Tile<64, 64>>::run(args...);
    if (P == 128 && N == 128) return F<Tile<128, 128>>::run(args...);
    if (P == 128 && N == 64) return F<Tile<128, 64>>::run(args...);
    *supported = false;
    return cudaSuccess;
}

template <class K>
cudaError_t launch(K kernel, int grid, int block, size_t smem, cudaStream_t s, const M2Args& a) {
    if (grid == 0) return cudaSuccess;
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
        if (e != cudaSuccess) return e;
    }
    kernel<<<grid, block, smem, s>>>(a);
    return cudaGetLastError();
}

template <class K>
cudaError_t launch_o(K kernel, int grid, int block, size_t smem, cudaStream_t s, const M2Args& a,
                     int out_f32) {
    if (grid == 0) return cudaSuccess;
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
        if (e != cudaSuccess) return e;
    }
    kernel<<<grid, block, smem, s>>>(a, out_f32);
    return cudaGetLastError();
}

template <class L> struct ConvF {
    static cudaError_t run(const M2Args& a, int in_dt, int out_dt, int rf, cudaStream_t s) {
        const int grid = a.B * a.H;
        const int of = (out_dt == RSSM_F32);
        if (in_dt == RSSM_F32) {
            if (rf == RSSM_READ_FP8) return launch_o(m2_qconv_step_kernel<L, float, RSSM_READ_FP8>, grid, L::kThreads, 0, s, a, of);
            if (rf == RSSM_READ_NVFP4) return launch_o(m2_qconv_step_kernel<L, float, RSSM_READ_NVFP4>, grid, L::kThreads, 0, s, a, of);
            return launch_o(m2_conv_step_kernel<L, float>, grid, L::kThreads, 0, s, a, of);
        }
        if (rf == RSSM_READ_FP8) return launch_o(m2_qconv_step_kernel<L, __nv_bfloat16, RSSM_READ_FP8>, grid, L::kThreads, 0, s, a, of);
        if (rf == RSSM_READ_NVFP4) return launch_o(m2_qconv_step_kernel<L, __nv_bfloat16, RSSM_READ_NVFP4>, grid, L::kThreads, 0, s, a, of);
        return launch_o(m2_conv_step_kernel<L, __nv_bfloat16>, grid, L::kThreads, 0, s, a, of);
    }
};

template <class L> struct SnapDraftF {
    static cudaError_t run(const M2Args& a, int in_dt, int out_dt, cudaStream_t s) {
        const int grid = a.B * a.H;
        const int of = (out_dt == RSSM_F32);
        if (in_dt == RSSM_F32) return launch_o(m2_snap_draft_kernel<L, float>, grid, L::kThreads, 0, s, a, of);
        return launch_o(m2_snap_draft_kernel<L, __nv_bfloat16>, grid, L::kThreads, 0, s, a, of);
    }
};

template <class L> struct SnapRestoreF {
    static cudaError_t run(const M2Args& a, cudaStream_t s) {
        return launch(m2_snap_restore_kernel<L>, a.B * a.H, L::kThreads, 0, s, a);
    }
};

template <class L> struct QuantF {
    template <typename TS>
    static cudaError_t run(int fmt, int64_t tiles, const TS* src, uint8_t* codes, uint8_t* bscale,
                           float* tscale, cudaStream_t s, const int32_t* counts = nullptr, int mark = 0,
                           int per = 1) {
        if (tiles == 0) return cudaSuccess;
        int64_t grid = tiles;
        if (counts != nullptr) {
            // a filtered launch: 8 blocks per SM stride over the tiles
            int num_sms = 0, smem_optin = 0;
            const cudaError_t e = device_limits(&num_sms, &smem_optin);
            if (e != cudaSuccess) return e;
            if (grid > 8LL * num_sms) grid = 8LL * num_sms;
        }
        if (grid > 0x7FFFFFFF) grid = 0x7FFFFFFF;
        const unsigned g = static_cast<unsigned>(grid);
        if (fmt == RSSM_READ_FP8)
            quantize_kernel<L, RSSM_READ_FP8, TS><<<g, L::kThreads, 0, s>>>(src, codes, bscale, tscale, counts, mark,
                                                                            per, tiles);
        else
            quantize_kernel<L, RSSM_READ_NVFP4, TS><<<g, L::kThreads, 0, s>>>(src, codes, bscale, tscale, counts,
                                                                              mark, per, tiles);
        return cudaGetLastError();
    }
};

// Quantise FP8 tiles (codes + one scale per tile), decoded, into format RF.
template <class L, int RF>
__global__ void __launch_bounds__(L::kThreads)
requantize_fp8_kernel(const uint8_t* src, const float* src_ts, uint8_t* codes, uint8_t* bscale, float* tscale) {
    __shared__ float s_red[L::kWarps];
    const int tile = blockIdx.x;
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const int col4 = t % L::TPR, row0 = t / L::TPR;
    const size_t n_el = static_cast<size_t>(L::P) * L::N;
    const size_t tile_off = static_cast<size_t>(tile) * n_el;
    const float ts = src_ts[tile];
    const uint32_t* s4 = reinterpret_cast<const uint32_t*>(src + tile_off);
    float4 hv[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const uint32_t u = s4[(row0 + j * L::RPP) * L::TPR + col4];
        const float2 lo = e4m3x2_to_f2(static_cast<uint16_t>(u & 0xFFFFu));
        const float2 hi = e4m3x2_to_f2(static_cast<uint16_t>(u >> 16));
        hv[j] = make_float4(__fmul_rn(lo.x, ts), __fmul_rn(lo.y, ts), __fmul_rn(hi.x, ts), __fmul_rn(hi.y, ts));
    }
    uint8_t* ct = codes + (RF == RSSM_READ_FP8 ? tile_off : tile_off / 2);
    uint8_t* bt = (RF == RSSM_READ_NVFP4) ? bscale + tile * (n_el / 16) : nullptr;
    write_read_copy<L, RF>(hv, ct, bt, tscale + tile, s_red, t, lane, warp,
                           [&](int j) { return row0 + j * L::RPP; }, [&](int) { return col4; },
                           [] { __syncthreads(); });
}

template <class L> struct RequantF {
    static cudaError_t run(int fmt, int64_t tiles, const uint8_t* src, const float* src_ts, uint8_t* codes,
                           uint8_t* bscale, float* tscale, cudaStream_t s) {
        if (tiles == 0) return cudaSuccess;
        if (fmt == RSSM_READ_FP8)
            requantize_fp8_kernel<L, RSSM_READ_FP8><<<static_cast<unsigned>(tiles), L::kThreads, 0, s>>>(
                src, src_ts, codes, bscale, tscale);
        else
            requantize_fp8_kernel<L, RSSM_READ_NVFP4><<<static_cast<unsigned>(tiles), L::kThreads, 0, s>>>(
                src, src_ts, codes, bscale, tscale);
        return cudaGetLastError();
    }
};

__global__ void f32_to_f16_kernel(const float4* src, uint2* dst, int64_t n4) {
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n4;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x)
        dst[i] = f32_to_f16x4(src[i]);
}

}  // namespace

cudaError_t m2_conv_step(const M2Args& a, int P, int N, int in_dt, int out_dt, int rf, cudaStream_t s,
                         bool* supported) {
    return with_tile<ConvF>(P, N, supported, a, in_dt, out_dt, rf, s);
}
cudaError_t m2_snap_draft(const M2Args& a, int P, int N, int in_dt, int out_dt, cudaStream_t s,
                          bool* supported) {
    return with_tile<SnapDraftF>(P, N, supported, a, in_dt, out_dt, s);
}
cudaError_t m2_snap_restore(const M2Args& a, int P, int N, cudaStream_t s, bool* supported) {
    return with_tile<SnapRestoreF>(P, N, supported, a, s);
}
cudaError_t quantize_tiles(int fmt, int64_t tiles, int rows, int cols, const float* src,
                           uint8_t* codes, uint8_t* bscale, float* tscale, cudaStream_t s,
                           bool* supported) {
    return with_tile<QuantF>(rows, cols, supported, fmt, tiles, src, codes, bscale, tscale, s);
}
cudaError_t quantize_tiles_from_fp8(int fmt, int64_t tiles, int rows, int cols, const uint8_t* src_codes,
                                    const float* src_tscale, uint8_t* codes, uint8_t* bscale, float* tscale,
                                    cudaStream_t s, bool* supported) {
    return with_tile<RequantF>(rows, cols, supported, fmt, tiles, src_codes, src_tscale, codes, bscale, tscale, s);
}
cudaError_t quantize_marked_tiles(int fmt, int64_t tiles, int rows, int cols, const float* src, const __half* src16,
                                  uint8_t* codes, uint8_t* bscale, float* tscale, const int32_t* counts, int mark,
                                  int per, cudaStream_t s, bool* supported) {
    if (src16 != nullptr)
        return with_tile<QuantF>(rows, cols, supported, fmt, tiles, src16, codes, bscale, tscale, s, counts, mark, per);
    return with_tile<QuantF>(rows, cols, supported, fmt, tiles, src, codes, bscale, tscale, s, counts, mark, per);
}
cudaError_t quantize_tiles_f16(int fmt, int64_t tiles, int rows, int cols, const __half* src,
                               uint8_t* codes, uint8_t* bscale, float* tscale, cudaStream_t s,
                               bool* supported) {
    return with_tile<QuantF>(rows, cols, supported, fmt, tiles, src, codes, bscale, tscale, s);
}
cudaError_t f32_to_f16_array(const float* src, __half* dst, int64_t n, cudaStream_t s) {
    if (n == 0) return cudaSuccess;
    const int64_t n4 = n / 4;
    const int grid = static_cast<int>(std::min<int64_t>((n4 + 255) / 256, 152 * 16));
    f32_to_f16_kernel<<<grid, 256, 0, s>>>(reinterpret_cast<const float4*>(src), reinterpret_cast<uint2*>(dst), n4);
    return cudaGetLastError();
}

}  // namespace rssm

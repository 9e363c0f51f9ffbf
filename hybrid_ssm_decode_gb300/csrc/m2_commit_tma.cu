// Mamba-2 commit after speculative drafts, and the explicit flush, persistent
// and pipelined for GB300.
//
// Method: "NVIDIA ve Dao AI Lab, ... ReplaySSM'i sundu", section "Durum
// trafigini azaltma ve rollback'in basitlestirilmesi": rejected drafts are
// dropped by moving the buffer pointer, with no state to restore; a sequence
// whose committed records fill the window folds them into the checkpoint,
// which is written once ("ReplaySSM beschleunigt ...", section "Wie es
// funktioniert", 2nd paragraph).
//
// Every tile: c <- c + a_b. A tile whose new count m reaches k (every tile
// with m > 0 when forced) folds all m records and resets c:
//   h_ckpt <- gamma h_ckpt + sum_{i<m} exp(A sum_{i<j<m} dt_j) dt_i x_i B_i^T,
//   gamma = exp(A sum_{j<m} dt_j),
// then rewrites its read copy (or leaves it to a quantiser launch that
// follows, over the tiles whose count is then 0). After a round of drafts only the sequences
// whose window filled fold (about one in nine at a mean of 1.8 accepted
// tokens and k = 16), and all heads of such a sequence fold together.
//
// Structure. Block q of the grid takes tiles q, q + grid, q + 2 grid, ...
// (strided, so one sequence's heads spread over all blocks and the folding
// work is balanced). Its setup warp applies every pointer move and lists the
// tiles that fold; a producer thread streams only those tiles' checkpoint,
// x, B and dt records through the stage ring; consumer groups fold in
// registers with the one-token step kernel's thread split (a warp covers 16
// rows, 8 lanes share 4 rows and split the columns). Waits are bounded as in
// the step kernels.
#include "m2_pipeline.cuh"

namespace rssm {
namespace {

struct CmGeom {
    int state, bsc, xrec, brec, dtrec, bytes;
};

// bsc: a block-scale region for an NVFP4 checkpoint
__host__ __device__ inline CmGeom commit_geom(int P, int N, int cap, int in_sz, bool bsc) {
    CmGeom g;
    int off = 0;
    g.state = off; off += align128(P * N * 4);
    g.bsc = off;   off += bsc ? align128(P * N / 16) : 0;
    g.xrec = off;  off += align128(cap * P * in_sz);
    g.brec = off;  off += align128(cap * N * in_sz);
    g.dtrec = off; off += align128(cap * in_sz);
    g.bytes = off;
    return g;
}

template <class L, typename TI, int RF, int NG, int CK>
__global__ void __launch_bounds__(32 + NG * L::kThreads, 1)
m2_commit_tma_kernel(const M2Args a, const int S, const int tiles_per_cta) {
    constexpr int P = L::P, N = L::N, GT = L::kThreads, GW = L::kWarps;
    constexpr int CPL = L::CPL, CH = N / 4, JJ = L::J;
    constexpr int in_sz = static_cast<int>(sizeof(TI));
    extern __shared__ __align__(128) unsigned char dsm[];
    __shared__ __align__(8) uint64_t full_bar[kMaxStages];
    __shared__ __align__(8) uint64_t empty_bar[kMaxStages];
    __shared__ __align__(8) uint64_t group_bar[NG];
    __shared__ int s_tile[kMaxTilesPerCta];   // tiles that fold, in order
    __shared__ int s_m[kMaxTilesPerCta];      // and their record counts
    __shared__ int s_nf;
    __shared__ float g_red[NG][GW];
    __shared__ volatile int s_abort;

    const int total = a.B * a.H;
    const int stride = gridDim.x;
    const int nt = (blockIdx.x < total) ? (total - 1 - blockIdx.x) / stride + 1 : 0;
    constexpr int CKF = ck_tile_fmt(CK);
    constexpr bool kAliased = (CKF != RSSM_READ_NONE && RF == CKF);   // the copy is the checkpoint
    const CmGeom geo = commit_geom(P, N, a.cap, in_sz, CK == kCkNVFP4);
    const int tid = threadIdx.x;
    const int hpg = a.H / a.G;

    if (tid < 32) {
        // --------------------------------- setup: pointer moves, fold list
        const int lane = tid;
        int nf = 0;
        for (int base = 0; base < nt; base += 32) {
            const int i = base + lane;
            bool fold = false;
            int m = 0, tile = 0;
            if (i < nt) {
                tile = blockIdx.x + i * stride;
                const int b = tile / a.H, hh = tile - b * a.H;
                const int c = a.counts[tile];
                if (c < 0 || c > a.cap) {
                    report_error(a.err, RSSM_DEV_COUNT_RANGE, tile, c);
                } else {
                    int acc = 0;
                    if (a.accepted != nullptr) {
                        acc = a.accepted[b];
                        if (acc < 0 || acc > a.T || c + acc > a.cap) {
                            if (hh == 0) report_error(a.err, RSSM_DEV_ACCEPTED_RANGE, b, acc);
                            acc = 0;
                        }
                    }
                    m = c + acc;
                    fold = a.force ? (m > 0) : (m >= a.k);
                    if (!fold && acc != 0) a.counts[tile] = m;
                }
            }
            const unsigned bal = __ballot_sync(0xffffffffu, fold);
            if (fold) {
                const int pos = nf + __popc(bal & ((1u << lane) - 1u));
                s_tile[pos] = tile;
                s_m[pos] = m;
            }
            nf += __popc(bal);
        }
        if (lane == 0) {
            s_nf = nf;
            for (int q = 0; q < S; ++q) {
                mbar_init(&full_bar[q], 1);
                mbar_init(&empty_bar[q], GW);
            }
            for (int q = 0; q < NG; ++q) mbar_init(&group_bar[q], GW);
            s_abort = 0;
            fence_mbar_init();
        }
    }
    __syncthreads();
    const int nf = s_nf;

    if (tid < 32) {
        // ------------------------------------------------------------- producer
        if (tid != 0) return;
        const uint64_t pol = l2_evict_first();
        uint32_t issued = 0, last_par = 0;
        int s = 0;
        uint32_t round = 0;
        for (int w = 0; w < nf; ++w) {
            if (s_abort) break;
            if (!mbar_wait_bounded(&empty_bar[s], (round & 1u) ^ 1u)) {
                report_error(a.err, kDevTimeout, s_tile[w], 40);
                s_abort = 1;
                break;
            }
            const int tile = s_tile[w], m = s_m[w];
            const int b = tile / a.H, hh = tile - b * a.H;
            const int grp = hh / hpg;
            unsigned char* st = dsm + static_cast<size_t>(s) * geo.bytes;
            const size_t toff = static_cast<size_t>(tile) * P * N;
            const uint32_t state_bytes = (CK == kCkFP8) ? P * N : (CK == kCkNVFP4) ? P * N / 2 : P * N * (CK == kCkF16 ? 2 : 4);
            const uint32_t bsc_bytes = (CK == kCkNVFP4) ? P * N / 16 : 0;
            const uint32_t xrec_bytes = m * P * in_sz, brec_bytes = m * N * in_sz;
            const uint32_t dtrec_bytes = a.cap * in_sz;
            mbar_arrive_expect_tx(&full_bar[s], state_bytes + bsc_bytes + xrec_bytes + brec_bytes + dtrec_bytes);
            const unsigned char* ckb = reinterpret_cast<const unsigned char*>(a.ckpt);
            const void* state_src = (CK == kCkF16) ? static_cast<const void*>(reinterpret_cast<const __half*>(a.ckpt) + toff)
                                    : (CK == kCkFP8) ? static_cast<const void*>(ckb + toff)
                                    : (CK == kCkNVFP4) ? static_cast<const void*>(ckb + toff / 2)
                                    : static_cast<const void*>(a.ckpt + toff);
            bulk_g2s_hint(st + geo.state, state_src, state_bytes, &full_bar[s], pol);
            if (bsc_bytes) bulk_g2s(st + geo.bsc, a.ck_bscale + toff / 16, bsc_bytes, &full_bar[s]);
            bulk_g2s(st + geo.xrec, reinterpret_cast<const TI*>(a.buf_x) + static_cast<size_t>(tile) * a.cap * P,
                     xrec_bytes, &full_bar[s]);
            bulk_g2s(st + geo.brec,
                     reinterpret_cast<const TI*>(a.buf_b) + (static_cast<size_t>(b) * a.G + grp) * a.cap * N,
                     brec_bytes, &full_bar[s]);
            bulk_g2s(st + geo.dtrec, reinterpret_cast<const TI*>(a.buf_dt) + static_cast<size_t>(tile) * a.cap,
                     dtrec_bytes, &full_bar[s]);
            issued |= 1u << s;
            last_par = (last_par & ~(1u << s)) | ((round & 1u) << s);
            if (++s == S) { s = 0; ++round; }
        }
        for (int q = 0; q < S; ++q)
            if ((issued >> q) & 1u)
                if (!mbar_wait_bounded(&full_bar[q], (last_par >> q) & 1u))
                    report_error(a.err, kDevTimeout, blockIdx.x, 41);
        return;
    }

    // --------------------------------------------------------------- consumers
    const int g = (tid - 32) / GT;
    const int gt = (tid - 32) - g * GT;
    const int lane = gt & 31, gw = gt >> 5;
    const int cl = lane & 7;
    const int rbase = gw * 16 + (lane >> 3) * 4;

    uint32_t gphase = 0;
    auto gsync = [&] {
        __syncwarp();
        int ok = 1;
        if (lane == 0) {
            mbar_arrive(&group_bar[g]);
            ok = mbar_wait_bounded(&group_bar[g], gphase) ? 1 : 0;
            if (!ok && !s_abort) {
                report_error(a.err, kDevTimeout, blockIdx.x, 42);
                s_abort = 1;
            }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (ok) mbar_try_wait(&group_bar[g], gphase);
        gphase ^= 1u;
        __syncwarp();
    };
    auto row_of = [&](int j) { return rbase + j / CPL; };
    auto chunk_of = [&](int j) { return cl + 8 * (j % CPL); };

    for (int w = g; w < nf; w += NG) {
        const int s = w % S;
        const uint32_t par = static_cast<uint32_t>(w / S) & 1u;
        int ok = 0;
        if (lane == 0) ok = (!s_abort && mbar_wait_bounded(&full_bar[s], par)) ? 1 : 0;
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) {
            if (lane == 0 && !s_abort) {
                report_error(a.err, kDevTimeout, s_tile[w], 43);
                s_abort = 1;
            }
            break;
        }
        mbar_try_wait(&full_bar[s], par);

        const int tile = s_tile[w], m = s_m[w];
        const int hh = tile % a.H;
        const unsigned char* st = dsm + static_cast<size_t>(s) * geo.bytes;
        const TI* sx = reinterpret_cast<const TI*>(st + geo.xrec);
        const TI* sb = reinterpret_cast<const TI*>(st + geo.brec);
        const TI* sdt = reinterpret_cast<const TI*>(st + geo.dtrec);

        // decays of the window (lane i holds record i)
        const float dti = (lane < m) ? to_f(sdt[lane]) : 0.f;
        float gamma;
        const float decay = window_decay(dti, lane, m, a.A[hh], gamma);
        const float cf = decay * dti;   // dt_i prod_{j>i} a_j

        // fold the m records into this thread's values, write them once
        float4 hv[JJ];
        const float cts = (CKF != RSSM_READ_NONE) ? a.ck_tscale[tile] : 1.f;
#pragma unroll
        for (int jj = 0; jj < JJ; ++jj) {
            const int idx = row_of(jj) * CH + chunk_of(jj);
            float4 v;
            if constexpr (CK == kCkF16) {
                v = f16x4_to_f32(reinterpret_cast<const uint2*>(st + geo.state)[idx]);
            } else if constexpr (CK == kCkFP8) {
                const uint32_t u = reinterpret_cast<const uint32_t*>(st + geo.state)[idx];
                const float2 lo = e4m3x2_to_f2(static_cast<uint16_t>(u & 0xFFFFu));
                const float2 hi = e4m3x2_to_f2(static_cast<uint16_t>(u >> 16));
                v = make_float4(__fmul_rn(lo.x, cts), __fmul_rn(lo.y, cts), __fmul_rn(hi.x, cts), __fmul_rn(hi.y, cts));
            } else if constexpr (CK == kCkNVFP4) {
                const uint32_t u = reinterpret_cast<const uint16_t*>(st + geo.state)[idx];
                const float es = __fmul_rn(e4m3_to_f((st + geo.bsc)[row_of(jj) * (N / 16) + (chunk_of(jj) >> 2)]), cts);
                const float2 lo = e2m1x2_to_f2(u & 0xFFu);
                const float2 hi = e2m1x2_to_f2((u >> 8) & 0xFFu);
                v = make_float4(__fmul_rn(lo.x, es), __fmul_rn(lo.y, es), __fmul_rn(hi.x, es), __fmul_rn(hi.y, es));
            } else {
                v = reinterpret_cast<const float4*>(st + geo.state)[idx];
            }
            hv[jj] = make_float4(v.x * gamma, v.y * gamma, v.z * gamma, v.w * gamma);
        }
        for (int i = 0; i < m; ++i) {
            const float cfi = __shfl_sync(0xffffffffu, cf, i);
            float xr[4];
            load_x4<TI>(sx + i * P + rbase, xr);
            const TI* Bi = sb + i * N;
#pragma unroll
            for (int q = 0; q < CPL; ++q) {
                const float4 bv = load4(Bi + (cl + 8 * q) * 4);
                const float2 b01 = make_float2(bv.x, bv.y), b23 = make_float2(bv.z, bv.w);
#pragma unroll
                for (int p = 0; p < 4; ++p) {
                    const float xp = cfi * xr[p];
                    const float2 x2 = make_float2(xp, xp);
                    float4& h = hv[p * CPL + q];
                    const float2 h01 = __ffma2_rn(x2, b01, make_float2(h.x, h.y));
                    const float2 h23 = __ffma2_rn(x2, b23, make_float2(h.z, h.w));
                    h = make_float4(h01.x, h01.y, h23.x, h23.y);
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty_bar[s]);   // the stage is no longer read

        const size_t tile_off = static_cast<size_t>(tile) * P * N;
        if constexpr (CKF != RSSM_READ_NONE) {
            // tile-format checkpoint: quantise, keep the stored values for the copy
            unsigned char* ckw = reinterpret_cast<unsigned char*>(a.ckpt);
            write_read_copy<L, CKF, true>(hv, ckw + (CKF == RSSM_READ_FP8 ? tile_off : tile_off / 2),
                                          CKF == RSSM_READ_NVFP4 ? a.ck_bscale + tile_off / 16 : nullptr,
                                          a.ck_tscale + tile, g_red[g], gt, lane, gw, row_of, chunk_of, gsync);
        } else if constexpr (CK == kCkF16) {
            // FP16 checkpoint: store rounded, make the read copy from the rounded values
            uint2* dst = reinterpret_cast<uint2*>(reinterpret_cast<__half*>(a.ckpt) + tile_off);
#pragma unroll
            for (int jj = 0; jj < JJ; ++jj) {
                const uint2 u = f32_to_f16x4(hv[jj]);
                dst[row_of(jj) * CH + chunk_of(jj)] = u;
                hv[jj] = f16x4_to_f32(u);
            }
        } else {
            float4* dst = reinterpret_cast<float4*>(a.ckpt + tile_off);
#pragma unroll
            for (int jj = 0; jj < JJ; ++jj) dst[row_of(jj) * CH + chunk_of(jj)] = hv[jj];
        }
        if (RF != RSSM_READ_NONE && !kAliased && !a.defer_copy) {
            uint8_t* codes = a.rc_codes + (RF == RSSM_READ_FP8 ? tile_off : tile_off / 2);
            uint8_t* bsc = (RF == RSSM_READ_NVFP4) ? a.rc_bscale + tile_off / 16 : nullptr;
            write_read_copy<L, RF>(hv, codes, bsc, a.rc_tscale + tile, g_red[g], gt, lane, gw, row_of, chunk_of,
                                   gsync);
        }
        if (gt == 0) a.counts[tile] = 0;
    }
}

template <class L, typename TI, int RF, int NG, int CK>
cudaError_t launch_commit_ng(const M2Args& a, int S, int grid, int per, size_t smem, cudaStream_t s) {
    auto kernel = m2_commit_tma_kernel<L, TI, RF, NG, CK>;
    static LaunchCache lc;
    cudaError_t e = cached_dyn_smem(lc, kernel, smem);
    if (e != cudaSuccess) return e;
    kernel<<<grid, 32 + NG * L::kThreads, smem, s>>>(a, S, per);
    return cudaGetLastError();
}

template <class L, typename TI, int RF, int CK = kCkF32>
cudaError_t launch_commit(const M2Args& a, cudaStream_t s) {
    const int total = a.B * a.H;
    if (total == 0) return cudaSuccess;
    int num_sms = 0, smem_optin = 0;
    cudaError_t e = device_limits(&num_sms, &smem_optin);
    if (e != cudaSuccess) return e;
    constexpr bool kTwo = L::kThreads <= 128;
    static LaunchCache lc;
    int static_smem = 0;
    e = cached_static_smem(lc, m2_commit_tma_kernel<L, TI, RF, kTwo ? 2 : 1, CK>, &static_smem);
    if (e != cudaSuccess) return e;
    const CmGeom geo = commit_geom(L::P, L::N, a.cap, static_cast<int>(sizeof(TI)), CK == kCkNVFP4);
    const int avail = smem_optin - static_smem - 1024;
    int smax = avail / geo.bytes;
    if (smax > kMaxStages) smax = kMaxStages;
    // every stage has one owner group: S is a multiple of the group count
    const int ng = (kTwo && smax >= 4) ? 2 : 1;
    const int S = (smax / ng) * ng;
    if (S < 2) return cudaErrorInvalidConfiguration;
    int grid = num_sms;
    if ((total + grid - 1) / grid > kMaxTilesPerCta) grid = (total + kMaxTilesPerCta - 1) / kMaxTilesPerCta;
    if (grid > total) grid = total;
    const size_t smem = static_cast<size_t>(S) * geo.bytes;
    if constexpr (kTwo) {
        if (ng == 2) return launch_commit_ng<L, TI, RF, 2, CK>(a, S, grid, 0, smem, s);
    }
    return launch_commit_ng<L, TI, RF, 1, CK>(a, S, grid, 0, smem, s);
}

template <class L>
cudaError_t run_commit(const M2Args& a, int in_dt, int rf, cudaStream_t s) {
    using BF = __nv_bfloat16;
    if (a.ck != kCkF32) {
        if (in_dt != RSSM_BF16) return cudaErrorInvalidValue;
        if (a.ck == kCkF16) {
            if (rf == RSSM_READ_FP8) return launch_commit<L, BF, RSSM_READ_FP8, kCkF16>(a, s);
            if (rf == RSSM_READ_NVFP4) return launch_commit<L, BF, RSSM_READ_NVFP4, kCkF16>(a, s);
            return launch_commit<L, BF, RSSM_READ_NONE, kCkF16>(a, s);
        }
        if (a.ck == kCkFP8) {
            if (rf == RSSM_READ_NVFP4) return launch_commit<L, BF, RSSM_READ_NVFP4, kCkFP8>(a, s);
            if (rf == RSSM_READ_FP8) return launch_commit<L, BF, RSSM_READ_FP8, kCkFP8>(a, s);
            return cudaErrorInvalidValue;
        }
        if (rf == RSSM_READ_NVFP4) return launch_commit<L, BF, RSSM_READ_NVFP4, kCkNVFP4>(a, s);
        return cudaErrorInvalidValue;
    }
    if (in_dt == RSSM_F32) {
        if (rf == RSSM_READ_FP8) return launch_commit<L, float, RSSM_READ_FP8>(a, s);
        if (rf == RSSM_READ_NVFP4) return launch_commit<L, float, RSSM_READ_NVFP4>(a, s);
        return launch_commit<L, float, RSSM_READ_NONE>(a, s);
    }
    if (rf == RSSM_READ_FP8) return launch_commit<L, __nv_bfloat16, RSSM_READ_FP8>(a, s);
    if (rf == RSSM_READ_NVFP4) return launch_commit<L, __nv_bfloat16, RSSM_READ_NVFP4>(a, s);
    return launch_commit<L, __nv_bfloat16, RSSM_READ_NONE>(a, s);
}

}  // namespace

cudaError_t m2_commit(const M2Args& a, int P, int N, int in_dt, int rf, cudaStream_t s, bool* supported) {
    *supported = true;
    if (P == 64 && N == 128) return run_commit<GTile<64, 128>>(a, in_dt, rf, s);
    if (P == 64 && N == 64) return run_commit<GTile<64, 64>>(a, in_dt, rf, s);
    if (P == 128 && N == 128) return run_commit<GTile<128, 128>>(a, in_dt, rf, s);
    if (P == 128 && N == 64) return run_commit<GTile<128, 64>>(a, in_dt, rf, s);
    *supported = false;
    return cudaSuccess;
}

}  // namespace rssm

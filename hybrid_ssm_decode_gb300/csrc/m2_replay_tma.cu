// Mamba-2 ReplaySSM decode step (one token per sequence), persistent and
// pipelined for GB300.
//
// Method: "ReplaySSM beschleunigt das Decoding von Hybridmodellen durch
// Caching der Eingaben statt des Zustands", section "Wie es funktioniert";
// "NVIDIA ve Dao AI Lab, ... ReplaySSM'i sundu", section "ReplaySSM nasil
// calisir?". A non-flush step reads the checkpoint and the buffered inputs
// and stores no state. The step that fills the buffer folds it into the
// checkpoint and writes the checkpoint once.
//
// Structure. One block per SM walks a contiguous range of (sequence, head)
// tiles.
//  * Producer (one thread). Before the loop it reads the whole range's record
//    counts and step sizes, so it never waits on a dependent load. For each
//    tile it then fills one stage of a shared-memory ring with bulk async
//    copies (cp.async.bulk, mbarrier transaction counts): the FP32 checkpoint
//    tile (or its low-precision read copy), the tile's buffered x and dt
//    records, its group's B records, and this token's x, B and C.
//  * Consumers (NG groups of P*N/32 threads). They take alternate tiles and
//    compute each output from shared memory. On a flush tile a group folds
//    the records in registers, then writes the checkpoint (and its read copy)
//    once.
// Every mbarrier wait is bounded (kWaitLimitNs). On expiry the kernel
// reports kDevTimeout in the error word, stops issuing, and waits (again
// bounded) for its own copies in flight before it returns.
#include "tile.cuh"

namespace rssm {
namespace {

constexpr int kMaxStages = 8;
constexpr int kMaxTilesPerCta = 512;

struct StageHdr {
    int c;            // records buffered before this token (-1: count out of range)
    uint32_t dt_raw;  // this token's dt, raw bits of the input dtype
    float tscale;     // read-copy tile scale (1 for the FP32 checkpoint)
    int pad;
};

struct StageGeom {
    int hdr, state, bsc, xrec, brec, dtrec, xt, bt, ct, bytes;
};

__host__ __device__ inline int align128(int v) { return (v + 127) & ~127; }

__host__ __device__ inline StageGeom stage_geom(int P, int N, int cap, int in_sz, int rf) {
    StageGeom g;
    int off = 0;
    g.hdr = off;   off += 128;
    g.state = off; off += align128(P * N * 4);
    g.bsc = off;   off += (rf == RSSM_READ_NVFP4) ? align128(P * N / 16) : 0;
    g.xrec = off;  off += align128(cap * P * in_sz);
    g.brec = off;  off += align128(cap * N * in_sz);
    g.dtrec = off; off += align128(cap * in_sz);
    g.xt = off;    off += align128(P * in_sz);
    g.bt = off;    off += align128(N * in_sz);
    g.ct = off;    off += align128(N * in_sz);
    g.bytes = off;
    return g;
}

__device__ __forceinline__ float raw_to_f(uint32_t raw, float*) { return __uint_as_float(raw); }
__device__ __forceinline__ float raw_to_f(uint32_t raw, __nv_bfloat16*) { return __uint_as_float(raw << 16); }

template <typename TI>
__device__ __forceinline__ uint32_t raw_of(const TI* p);
template <>
__device__ __forceinline__ uint32_t raw_of<float>(const float* p) { return __float_as_uint(*p); }
template <>
__device__ __forceinline__ uint32_t raw_of<__nv_bfloat16>(const __nv_bfloat16* p) {
    return *reinterpret_cast<const uint16_t*>(p);
}

template <typename TI>
__device__ __forceinline__ void store_raw(TI* p, uint32_t raw);
template <>
__device__ __forceinline__ void store_raw<float>(float* p, uint32_t raw) { *p = __uint_as_float(raw); }
template <>
__device__ __forceinline__ void store_raw<__nv_bfloat16>(__nv_bfloat16* p, uint32_t raw) {
    *reinterpret_cast<uint16_t*>(p) = static_cast<uint16_t>(raw);
}

template <class L, typename TI, int RF, int NG>
__global__ void __launch_bounds__(32 + NG * L::kThreads, 1)
m2_replay_step_tma_kernel(const M2Args a, const int out_f32, const int S, const int tiles_per_cta) {
    constexpr int P = L::P, N = L::N, GT = L::kThreads, GW = L::kWarps;
    constexpr int in_sz = static_cast<int>(sizeof(TI));
    extern __shared__ __align__(128) unsigned char dsm[];
    __shared__ __align__(8) uint64_t full_bar[kMaxStages];
    __shared__ __align__(8) uint64_t empty_bar[kMaxStages];
    __shared__ int s_cnt[kMaxTilesPerCta];
    __shared__ uint32_t s_dtv[kMaxTilesPerCta];
    __shared__ float s_ts[RF != RSSM_READ_NONE ? kMaxTilesPerCta : 1];
    __shared__ float g_w[NG][2][kMaxCap], g_cf[NG][2][kMaxCap];
    __shared__ float g_red[NG][GW];
    __shared__ volatile int s_abort;

    const int total = a.B * a.H;
    const int t0 = blockIdx.x * tiles_per_cta;
    const int nt = max(0, min(tiles_per_cta, total - t0));
    const StageGeom geo = stage_geom(P, N, a.cap, in_sz, RF);
    const int tid = threadIdx.x;

    if (tid < 32) {
        for (int i = tid; i < nt; i += 32) {
            s_cnt[i] = a.counts[t0 + i];
            s_dtv[i] = raw_of<TI>(reinterpret_cast<const TI*>(a.dt) + t0 + i);
            if (RF != RSSM_READ_NONE) s_ts[RF != RSSM_READ_NONE ? i : 0] = a.rc_tscale[t0 + i];
        }
        if (tid == 0) {
            for (int s = 0; s < S; ++s) {
                mbar_init(&full_bar[s], 1);
                mbar_init(&empty_bar[s], GW);
            }
            s_abort = 0;
            fence_mbar_init();
        }
    }
    __syncthreads();

    if (tid < 32) {
        // ------------------------------------------------------------- producer
        if (tid != 0) return;
        const uint64_t pol = l2_evict_first();
        uint32_t issued = 0, last_par = 0;
        for (int j = 0; j < nt; ++j) {
            if (s_abort) break;
            const int s = j % S;
            const uint32_t round = static_cast<uint32_t>(j / S);
            if (!mbar_wait_bounded(&empty_bar[s], (round & 1u) ^ 1u)) {
                report_error(a.err, kDevTimeout, t0 + j, 0);
                s_abort = 1;
                break;
            }
            const int tile = t0 + j;
            const int b = tile / a.H, hh = tile - b * a.H, g = hh / (a.H / a.G);
            const int c = s_cnt[j];
            const bool cok = (c >= 0 && c < a.k);
            const int nrec = cok ? c : 0;
            const bool flush = cok && (c + 1 == a.k);
            const bool use_rc = (RF != RSSM_READ_NONE) && !flush;
            unsigned char* st = dsm + static_cast<size_t>(s) * geo.bytes;
            StageHdr* hdr = reinterpret_cast<StageHdr*>(st + geo.hdr);
            hdr->c = cok ? c : -1;
            hdr->dt_raw = s_dtv[j];
            hdr->tscale = (RF != RSSM_READ_NONE && use_rc) ? s_ts[RF != RSSM_READ_NONE ? j : 0] : 1.f;

            const size_t tile_off = static_cast<size_t>(tile) * P * N;
            const uint32_t state_bytes =
                use_rc ? (RF == RSSM_READ_FP8 ? P * N : P * N / 2) : P * N * 4;
            const uint32_t bsc_bytes = (use_rc && RF == RSSM_READ_NVFP4) ? P * N / 16 : 0;
            const uint32_t xrec_bytes = nrec * P * in_sz, brec_bytes = nrec * N * in_sz;
            const uint32_t dtrec_bytes = a.cap * in_sz;
            const uint32_t tok_bytes = P * in_sz + 2 * N * in_sz;
            mbar_arrive_expect_tx(&full_bar[s], state_bytes + bsc_bytes + xrec_bytes + brec_bytes +
                                                    dtrec_bytes + tok_bytes);
            const void* state_src;
            if (!use_rc) state_src = a.ckpt + tile_off;
            else if (RF == RSSM_READ_FP8) state_src = a.rc_codes + tile_off;
            else state_src = a.rc_codes + tile_off / 2;
            bulk_g2s_hint(st + geo.state, state_src, state_bytes, &full_bar[s], pol);
            if (bsc_bytes) bulk_g2s(st + geo.bsc, a.rc_bscale + tile_off / 16, bsc_bytes, &full_bar[s]);
            const TI* bx = reinterpret_cast<const TI*>(a.buf_x) + static_cast<size_t>(tile) * a.cap * P;
            const TI* bb = reinterpret_cast<const TI*>(a.buf_b) + (static_cast<size_t>(b) * a.G + g) * a.cap * N;
            const TI* bdt = reinterpret_cast<const TI*>(a.buf_dt) + static_cast<size_t>(tile) * a.cap;
            if (xrec_bytes) bulk_g2s(st + geo.xrec, bx, xrec_bytes, &full_bar[s]);
            if (brec_bytes) bulk_g2s(st + geo.brec, bb, brec_bytes, &full_bar[s]);
            bulk_g2s(st + geo.dtrec, bdt, dtrec_bytes, &full_bar[s]);
            bulk_g2s(st + geo.xt, reinterpret_cast<const TI*>(a.x) + static_cast<size_t>(tile) * P,
                     P * in_sz, &full_bar[s]);
            bulk_g2s(st + geo.bt, reinterpret_cast<const TI*>(a.Bm) + (static_cast<size_t>(b) * a.G + g) * N,
                     N * in_sz, &full_bar[s]);
            bulk_g2s(st + geo.ct, reinterpret_cast<const TI*>(a.C) + (static_cast<size_t>(b) * a.G + g) * N,
                     N * in_sz, &full_bar[s]);
            issued |= 1u << s;
            last_par = (last_par & ~(1u << s)) | ((round & 1u) << s);
        }
        // our own copies in flight must land before the block may exit
        for (int s = 0; s < S; ++s)
            if ((issued >> s) & 1u)
                if (!mbar_wait_bounded(&full_bar[s], (last_par >> s) & 1u))
                    report_error(a.err, kDevTimeout, t0, 1);
        return;
    }

    // --------------------------------------------------------------- consumers
    // Thread gt of a group owns columns 4*col4..+3 of the 8 consecutive rows
    // rb..rb+7, so one 16-byte shared load brings a record's x values for all
    // of its rows. Per tile: every warp scans the window's dt (decays and
    // gamma, no cross-warp step), each warp forms B_i.C_t for its share of
    // the records, one group barrier, then each lane adds its own record's
    // x term to its slice of h_ckpt.C_t before the row reduction, so the
    // buffered-input term costs no extra pass. Warps release the stage one by
    // one (the empty barrier counts warps), and the per-group scratch is
    // double-buffered by tile parity.
    const int g = (tid - 32) / GT;
    const int gt = (tid - 32) - g * GT;
    const int lane = gt & 31, gw = gt >> 5;
    const int col4 = gt % L::TPR, rb = (gt / L::TPR) * 8;
    const int bar_id = 1 + g;
    auto gsync = [&] { named_sync(bar_id, GT); };
    constexpr int XV = 8 * in_sz / 16;  // 16-byte vectors per 8 x values

    for (int j = g, it = 0; j < nt; j += NG, ++it) {
        const int s = j % S;
        const uint32_t par = static_cast<uint32_t>(j / S) & 1u;
        const int pb = it & 1;   // scratch buffer of this tile
        int ok = 0;
        if (lane == 0) ok = (!s_abort && mbar_wait_bounded(&full_bar[s], par)) ? 1 : 0;
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (ok) mbar_try_wait(&full_bar[s], par);   // acquire the bulk-copied bytes in every lane
        else if (lane == 0 && !s_abort) {
            report_error(a.err, kDevTimeout, t0 + j, 2);
            s_abort = 1;
        }

        const int tile = t0 + j;
        const int b = tile / a.H, hh = tile - b * a.H, grp = hh / (a.H / a.G);
        const unsigned char* st = dsm + static_cast<size_t>(s) * geo.bytes;
        const StageHdr hdr = *reinterpret_cast<const StageHdr*>(st + geo.hdr);
        const int c = ok ? hdr.c : -1;
        const int m = c + 1;
        const bool flush = (m == a.k);
        const TI* sx = reinterpret_cast<const TI*>(st + geo.xrec);
        const TI* sb = reinterpret_cast<const TI*>(st + geo.brec);
        const TI* sdt = reinterpret_cast<const TI*>(st + geo.dtrec);
        const TI* sxt = reinterpret_cast<const TI*>(st + geo.xt);
        const TI* sbt = reinterpret_cast<const TI*>(st + geo.bt);
        const TI* sct = reinterpret_cast<const TI*>(st + geo.ct);
        float* w_s = g_w[g][pb];
        float* cf_s = g_cf[g][pb];

        // decays (every warp), and B_i . C_t -> w_i for this warp's records
        float gamma = 1.f;
        if (c >= 0) {
            const float dt_t = raw_to_f(hdr.dt_raw, static_cast<TI*>(nullptr));
            const float dti = (lane < c) ? to_f(sdt[lane]) : (lane == c ? dt_t : 0.f);
            const float decay = window_decay(dti, lane, m, a.A[hh], gamma);
            const float cf = decay * dti;
            for (int i = gw; i < m; i += GW) {
                const TI* Bi = (i < c) ? sb + i * N : sbt;
                float sacc = 0.f;
                for (int n = lane * 4; n < N; n += 128) sacc += dot4(load4(Bi + n), load4(sct + n));
                sacc = warp_sum(sacc);
                const float cfi = __shfl_sync(0xffffffffu, cf, i);
                if (lane == 0) {
                    w_s[i] = cfi * sacc;
                    cf_s[i] = cfi;
                }
            }
        }
        gsync();
        if (s_abort) break;

        if (c < 0) {
            if (gt == 0) report_error(a.err, RSSM_DEV_COUNT_RANGE, tile, s_cnt[j]);
        } else {
            // checkpoint (or read copy) times C_t, scaled by gamma, plus this
            // lane's records' x terms; then the row reduction
            const float4 cv = load4(sct + col4 * 4);
            const float gs = gamma * hdr.tscale;
            float part[8];
            if (RF == RSSM_READ_NONE || flush) {
                const float4* sh = reinterpret_cast<const float4*>(st + geo.state);
#pragma unroll
                for (int jj = 0; jj < 8; ++jj) part[jj] = gs * dot4(sh[(rb + jj) * L::TPR + col4], cv);
            } else if (RF == RSSM_READ_FP8) {
                const uint32_t* sc = reinterpret_cast<const uint32_t*>(st + geo.state);
#pragma unroll
                for (int jj = 0; jj < 8; ++jj) {
                    const uint32_t w = sc[(rb + jj) * L::TPR + col4];
                    const float2 lo = e4m3x2_to_f2(static_cast<uint16_t>(w & 0xFFFFu));
                    const float2 hi = e4m3x2_to_f2(static_cast<uint16_t>(w >> 16));
                    part[jj] = gs * dot4(make_float4(lo.x, lo.y, hi.x, hi.y), cv);
                }
            } else {
                const uint16_t* sc = reinterpret_cast<const uint16_t*>(st + geo.state);
                const uint8_t* sbs = st + geo.bsc;
#pragma unroll
                for (int jj = 0; jj < 8; ++jj) {
                    const int row = rb + jj;
                    const uint32_t w = sc[row * L::TPR + col4];
                    const float2 lo = e2m1x2_to_f2(w & 0xFFu);
                    const float2 hi = e2m1x2_to_f2(w >> 8);
                    part[jj] = gs * e4m3_to_f(sbs[row * (N / 16) + (col4 >> 2)]) *
                               dot4(make_float4(lo.x, lo.y, hi.x, hi.y), cv);
                }
            }
            for (int i = col4; i < m; i += L::TPR) {
                const TI* xi = (i < c) ? sx + i * P : sxt;
                const float wi = (i < c) ? w_s[i] : w_s[c] + a.D[hh];
                const uint4* xv = reinterpret_cast<const uint4*>(xi + rb);
#pragma unroll
                for (int q = 0; q < XV; ++q) {
                    const uint4 u = xv[q];
                    const uint32_t wd[4] = {u.x, u.y, u.z, u.w};
                    if (sizeof(TI) == 2) {
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            part[q * 8 + 2 * e] = fmaf(wi, __uint_as_float(wd[e] << 16), part[q * 8 + 2 * e]);
                            part[q * 8 + 2 * e + 1] =
                                fmaf(wi, __uint_as_float(wd[e] & 0xFFFF0000u), part[q * 8 + 2 * e + 1]);
                        }
                    } else {
#pragma unroll
                        for (int e = 0; e < 4; ++e) part[q * 4 + e] = fmaf(wi, __uint_as_float(wd[e]), part[q * 4 + e]);
                    }
                }
            }
            {
                const float rs = group_reduce_multi<8, L::TPR>(part, lane);
                constexpr int kLanesPerValue = L::TPR / 8;
                if ((lane % kLanesPerValue) == 0) {
                    const int r = rb + (lane % L::TPR) / kLanesPerValue;
                    store_out(a.y, static_cast<size_t>(tile) * P + r, rs, out_f32 != 0);
                }
            }

            if (!flush) {
                // append this token's record at slot c (16-byte vectors)
                uint4* bx = reinterpret_cast<uint4*>(reinterpret_cast<TI*>(a.buf_x) +
                                                     (static_cast<size_t>(tile) * a.cap + c) * P);
                const uint4* xs = reinterpret_cast<const uint4*>(sxt);
                for (int q = gt; q < P * in_sz / 16; q += GT) bx[q] = xs[q];
                if (gt == 0) {
                    store_raw<TI>(reinterpret_cast<TI*>(a.buf_dt) + static_cast<size_t>(tile) * a.cap + c,
                                  hdr.dt_raw);
                    a.counts[tile] = m;
                }
                if (hh % (a.H / a.G) == 0) {
                    uint4* bb = reinterpret_cast<uint4*>(reinterpret_cast<TI*>(a.buf_b) +
                                                         ((static_cast<size_t>(b) * a.G + grp) * a.cap + c) * N);
                    const uint4* bs = reinterpret_cast<const uint4*>(sbt);
                    for (int q = gt; q < N * in_sz / 16; q += GT) bb[q] = bs[q];
                }
            } else {
                // fold the k records into the checkpoint and write it once
                const float4* sh = reinterpret_cast<const float4*>(st + geo.state);
                float4 hv[8];
#pragma unroll
                for (int jj = 0; jj < 8; ++jj) {
                    const float4 v = sh[(rb + jj) * L::TPR + col4];
                    hv[jj] = make_float4(v.x * gamma, v.y * gamma, v.z * gamma, v.w * gamma);
                }
                for (int i = 0; i < m; ++i) {
                    const TI* Bi = (i < c) ? sb + i * N : sbt;
                    const TI* xi = (i < c) ? sx + i * P : sxt;
                    const float cfi = cf_s[i];
                    float4 bv = load4(Bi + col4 * 4);
                    bv = make_float4(cfi * bv.x, cfi * bv.y, cfi * bv.z, cfi * bv.w);
                    const uint4* xv = reinterpret_cast<const uint4*>(xi + rb);
                    float xr[8];
#pragma unroll
                    for (int q = 0; q < XV; ++q) {
                        const uint4 u = xv[q];
                        const uint32_t wd[4] = {u.x, u.y, u.z, u.w};
                        if (sizeof(TI) == 2) {
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                xr[q * 8 + 2 * e] = __uint_as_float(wd[e] << 16);
                                xr[q * 8 + 2 * e + 1] = __uint_as_float(wd[e] & 0xFFFF0000u);
                            }
                        } else {
#pragma unroll
                            for (int e = 0; e < 4; ++e) xr[q * 4 + e] = __uint_as_float(wd[e]);
                        }
                    }
#pragma unroll
                    for (int jj = 0; jj < 8; ++jj) {
                        hv[jj].x = fmaf(xr[jj], bv.x, hv[jj].x);
                        hv[jj].y = fmaf(xr[jj], bv.y, hv[jj].y);
                        hv[jj].z = fmaf(xr[jj], bv.z, hv[jj].z);
                        hv[jj].w = fmaf(xr[jj], bv.w, hv[jj].w);
                    }
                }
                const size_t tile_off = static_cast<size_t>(tile) * P * N;
                float4* dst = reinterpret_cast<float4*>(a.ckpt + tile_off);
#pragma unroll
                for (int jj = 0; jj < 8; ++jj) dst[(rb + jj) * L::TPR + col4] = hv[jj];
                if (RF != RSSM_READ_NONE) {
                    uint8_t* codes = a.rc_codes + (RF == RSSM_READ_FP8 ? tile_off : tile_off / 2);
                    uint8_t* bsc = (RF == RSSM_READ_NVFP4) ? a.rc_bscale + tile_off / 16 : nullptr;
                    write_read_copy<L, RF>(hv, codes, bsc, a.rc_tscale + tile, g_red[g], gt, lane, gw,
                                           [&](int jj) { return rb + jj; }, col4, gsync);
                }
                if (gt == 0) a.counts[tile] = 0;
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty_bar[s]);  // this warp is done with the stage
    }
}

int g_num_sms = 0;
int g_smem_optin = 0;

cudaError_t device_limits() {
    if (g_num_sms) return cudaSuccess;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&g_num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&g_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    return e;
}

template <class L, typename TI, int RF>
cudaError_t launch_tma(const M2Args& a, int out_f32, cudaStream_t s) {
    constexpr int NG = (32 + 2 * L::kThreads <= 1024) ? 2 : 1;
    const int total = a.B * a.H;
    if (total == 0) return cudaSuccess;
    cudaError_t e = device_limits();
    if (e != cudaSuccess) return e;
    auto kernel = m2_replay_step_tma_kernel<L, TI, RF, NG>;
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, kernel);
    if (e != cudaSuccess) return e;
    const StageGeom geo = stage_geom(L::P, L::N, a.cap, static_cast<int>(sizeof(TI)), RF);
    const int avail = g_smem_optin - static_cast<int>(fa.sharedSizeBytes) - 1024;
    int S = avail / geo.bytes;
    if (S > kMaxStages) S = kMaxStages;
    if (S < 2) return cudaErrorInvalidConfiguration;
    int grid = g_num_sms;
    if ((total + grid - 1) / grid > kMaxTilesPerCta) grid = (total + kMaxTilesPerCta - 1) / kMaxTilesPerCta;
    if (grid > total) grid = total;
    const int per = (total + grid - 1) / grid;
    grid = (total + per - 1) / per;
    const size_t smem = static_cast<size_t>(S) * geo.bytes;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    kernel<<<grid, 32 + NG * L::kThreads, smem, s>>>(a, out_f32, S, per);
    return cudaGetLastError();
}

template <class L>
cudaError_t run_tma(const M2Args& a, int in_dt, int out_dt, int rf, cudaStream_t s) {
    const int of = (out_dt == RSSM_F32);
    if (in_dt == RSSM_F32) {
        if (rf == RSSM_READ_FP8) return launch_tma<L, float, RSSM_READ_FP8>(a, of, s);
        if (rf == RSSM_READ_NVFP4) return launch_tma<L, float, RSSM_READ_NVFP4>(a, of, s);
        return launch_tma<L, float, RSSM_READ_NONE>(a, of, s);
    }
    if (rf == RSSM_READ_FP8) return launch_tma<L, __nv_bfloat16, RSSM_READ_FP8>(a, of, s);
    if (rf == RSSM_READ_NVFP4) return launch_tma<L, __nv_bfloat16, RSSM_READ_NVFP4>(a, of, s);
    return launch_tma<L, __nv_bfloat16, RSSM_READ_NONE>(a, of, s);
}

}  // namespace

cudaError_t m2_replay_step(const M2Args& a, int P, int N, int in_dt, int out_dt, int rf,
                           cudaStream_t s, bool* supported) {
    *supported = true;
    if (P == 64 && N == 128) return run_tma<Tile<64, 128>>(a, in_dt, out_dt, rf, s);
    if (P == 64 && N == 64) return run_tma<Tile<64, 64>>(a, in_dt, out_dt, rf, s);
    if (P == 128 && N == 128) return run_tma<Tile<128, 128>>(a, in_dt, out_dt, rf, s);
    if (P == 128 && N == 64) return run_tma<Tile<128, 64>>(a, in_dt, out_dt, rf, s);
    *supported = false;
    return cudaSuccess;
}

}  // namespace rssm

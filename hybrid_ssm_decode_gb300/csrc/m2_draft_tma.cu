// Mamba-2 ReplaySSM speculative draft step (T > 1 tokens per sequence),
// persistent and pipelined for GB300.
//
// Method: "NVIDIA ve Dao AI Lab, ... ReplaySSM'i sundu", section "Durum
// trafigini azaltma ve rollback'in basitlestirilmesi" (drafts are appended
// to the buffer; a rejected suffix is dropped by moving the buffer pointer,
// with no state to restore); "ReplaySSM beschleunigt ...", section "Wie es
// funktioniert".
#include "m2_pipeline.cuh"

namespace rssm {
namespace {

// ---------------------------------------------------------------------------
// Speculative draft step (T > 1 tokens per sequence; "NVIDIA ve Dao AI Lab,
// ... ReplaySSM'i sundu", section "Durum trafigini azaltma ve rollback'in
// basitlestirilmesi"): appends T uncommitted records at slots c..c+T-1 and
// writes, for each draft tau, the output from the FP32 checkpoint and records
// 0..c+tau. No state is written; the verify step moves the count.
// Same pipeline as the lean kernel. A stage holds the checkpoint tile (or its
// FP8 / NVFP4 read copy) and the T drafts' B and C vectors; each lane loads
// the x and dt values of the records and drafts it needs one tile ahead. A
// lane keeps its 4 state rows in registers for the T row-dots, and the
// drafts' records are appended from the stage (B) and from the registers that
// hold them (x, dt).
// With a read copy (RF = FP8 or NVFP4) the drafts' checkpoint term reads the
// copy, as the one-token non-flush step does ("... ReplaySSM'i sundu",
// section "Kuantizasyon hatasinin sinirlandirilmasi"); the records are exact.
// For bf16 inputs one m16n8k16 MMA per 16 columns dots a warp's 16 copy rows
// with all T drafts' C at once (draft n in MMA column n), so the copy is
// decoded once for every draft.
// ---------------------------------------------------------------------------
struct DrGeom {
    int bcv, state, bsc, bt, ct, bytes;
};

__host__ __device__ inline DrGeom draft_geom(int P, int N, int T, int in_sz, int rf) {
    DrGeom g;
    int off = 0;
    g.bcv = off;   off += (rf != RSSM_READ_NONE) ? T * 128 : 0;   // window dots: float [tau][i] = B_i . C_tau
    g.state = off; off += align128(rf == RSSM_READ_NONE ? P * N * 4 : (rf == RSSM_READ_FP8 ? P * N : P * N / 2));
    g.bsc = off;   off += (rf == RSSM_READ_NVFP4) ? align128(P * N / 16) : 0;
    g.bt = off;    off += align128(T * N * in_sz);
    g.ct = off;    off += align128(T * N * in_sz);
    g.bytes = off;
    return g;
}

// A read copy's stages are small, so the dots warp (below) runs far enough
// ahead; with the FP32 checkpoint's six stages the consumers form the dots
// themselves (measured: 664 us against 836 us with the dots warp at B512).
template <int RF>
__host__ __device__ constexpr int draft_lead() { return RF != RSSM_READ_NONE ? 64 : 32; }

template <class L, typename TI, int RF, int NG, int TMAX>
__global__ void __launch_bounds__(draft_lead<RF>() + NG * L::kThreads, 1)
m2_replay_draft_tma_kernel(const M2Args a, const int out_f32, const int S, const int tiles_per_cta) {
    constexpr int P = L::P, N = L::N, GT = L::kThreads, GW = L::kWarps, CPL = L::CPL, CH = N / 4;
    constexpr int in_sz = static_cast<int>(sizeof(TI));
    extern __shared__ __align__(128) unsigned char dsm[];
    __shared__ __align__(8) uint64_t full_bar[kMaxStages];
    __shared__ __align__(8) uint64_t empty_bar[kMaxStages];
    __shared__ int s_cnt[kMaxTilesPerCta];
    constexpr bool kCopy = (RF != RSSM_READ_NONE);
    constexpr bool kMma = kCopy && sizeof(TI) == 2;
    constexpr bool kDotsWarp = draft_lead<RF>() == 64;
    __shared__ float s_ts[kCopy ? kMaxTilesPerCta : 1];
    __shared__ __align__(8) uint64_t dots_bar;   // the dots warp's scratch copies
    __shared__ volatile int s_abort;

    const int T = a.T;
    const int total = a.B * a.H;
    const int t0 = blockIdx.x * tiles_per_cta;
    const int nt = max(0, min(tiles_per_cta, total - t0));
    const DrGeom geo = draft_geom(P, N, T, in_sz, RF);
    const int tid = threadIdx.x;
    const int hpg = a.H / a.G;

    if (tid < 32) {
        for (int i = tid; i < nt; i += 32) {
            int c = a.counts[t0 + i];
            if (c < 0 || c >= a.k || c + T > a.cap) {
                report_error(a.err, RSSM_DEV_COUNT_RANGE, t0 + i, c);
                c = -1;
            }
            s_cnt[i] = c;
            if (kCopy) s_ts[kCopy ? i : 0] = a.rc_tscale[t0 + i];
        }
        if (tid == 0) {
            for (int q = 0; q < S; ++q) {
                mbar_init(&full_bar[q], kDotsWarp ? 2 : 1);   // the producer (and the dots warp)
                mbar_init(&empty_bar[q], GW);
            }
            mbar_init(&dots_bar, 1);
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
        int s = 0;
        uint32_t round = 0;
        int b = t0 / a.H, hh = t0 - b * a.H;
        int g = hh / hpg, hin = hh - g * hpg;
        for (int j = 0; j < nt; ++j) {
            if (s_abort) break;
            if (!mbar_wait_bounded(&empty_bar[s], (round & 1u) ^ 1u)) {
                report_error(a.err, kDevTimeout, t0 + j, 30);
                s_abort = 1;
                break;
            }
            unsigned char* st = dsm + static_cast<size_t>(s) * geo.bytes;
            const size_t tile_off = static_cast<size_t>(t0 + j) * P * N;
            const uint32_t state_bytes = (RF == RSSM_READ_NONE) ? P * N * 4 : (RF == RSSM_READ_FP8 ? P * N : P * N / 2);
            const uint32_t bsc_bytes = (RF == RSSM_READ_NVFP4) ? P * N / 16 : 0;
            mbar_arrive_expect_tx(&full_bar[s], state_bytes + bsc_bytes + 2 * T * N * in_sz);
            const void* state_src;
            if (RF == RSSM_READ_NONE) state_src = a.ckpt + tile_off;
            else state_src = a.rc_codes + (RF == RSSM_READ_FP8 ? tile_off : tile_off / 2);
            bulk_g2s_hint(st + geo.state, state_src, state_bytes, &full_bar[s], pol);
            if (bsc_bytes) bulk_g2s(st + geo.bsc, a.rc_bscale + tile_off / 16, bsc_bytes, &full_bar[s]);
            for (int tau = 0; tau < T; ++tau) {
                const size_t row = (static_cast<size_t>(b) * T + tau) * a.G + g;
                bulk_g2s(st + geo.bt + tau * N * in_sz, reinterpret_cast<const TI*>(a.Bm) + row * N, N * in_sz,
                         &full_bar[s]);
                bulk_g2s(st + geo.ct + tau * N * in_sz, reinterpret_cast<const TI*>(a.C) + row * N, N * in_sz,
                         &full_bar[s]);
            }
            issued |= 1u << s;
            last_par = (last_par & ~(1u << s)) | ((round & 1u) << s);
            if (++s == S) { s = 0; ++round; }
            if (++hh == a.H) { hh = 0; ++b; g = 0; hin = 0; }
            else if (++hin == hpg) { hin = 0; ++g; }
        }
        for (int q = 0; q < S; ++q)
            if ((issued >> q) & 1u)
                if (!mbar_wait_bounded(&full_bar[q], (last_par >> q) & 1u))
                    report_error(a.err, kDevTimeout, t0, 31);
        return;
    }

    if (kDotsWarp && tid < 64) {
        // ------------------------------------------------------------ dots warp
        // The window dots B_i . C_tau depend only on the key (sequence, B/C
        // group, count). This warp forms every draft's dots with the
        // consumers' former arithmetic (the same quads and reductions, from
        // the same values, copied into its scratch in one round trip) when the
        // key changes. Every stage carries its key's dots and completes only
        // with this warp's arrive (the full barriers count the producer's
        // arrive and this one), so the copies are not held up meanwhile.
        const int lane = tid - 32, cl = lane & 7;
        const uint64_t keep = l2_evict_last();   // records are read again by later steps of the window
        unsigned char* scr = dsm + static_cast<size_t>(S) * geo.bytes;        // B rows: records, then drafts
        unsigned char* scr_c = scr + static_cast<size_t>(a.cap) * N * in_sz;  // C rows
        uint32_t dpar = 0;
        int s = 0;
        uint32_t round = 0;
        int b = t0 / a.H, hh = t0 - b * a.H;
        int g = hh / hpg, hin = hh - g * hpg;
        int key_b = -1, key_g = -1, key_c = -1;
        float bc[TMAX];   // lane i: B_i . C_tau of the current key
#pragma unroll
        for (int tau = 0; tau < TMAX; ++tau) bc[tau] = 0.f;
        for (int j = 0; j < nt; ++j) {
            int ok = 1;
            if (lane == 0) {
                if (s_abort) {
                    ok = 0;
                } else if (!mbar_wait_bounded(&empty_bar[s], (round & 1u) ^ 1u)) {
                    report_error(a.err, kDevTimeout, t0 + j, 33);
                    s_abort = 1;
                    ok = 0;
                }
            }
            if (!__shfl_sync(0xffffffffu, ok, 0)) break;
            const int c = s_cnt[j];
            if (c >= 0) {
                if (b != key_b || g != key_g || c != key_c) {
                    const int M = c + T;
                    const TI* gb = reinterpret_cast<const TI*>(a.buf_b) + (static_cast<size_t>(b) * a.G + g) * a.cap * N;
                    auto draft_row = [&](const void* base) {
                        return [=](int tau) {
                            return reinterpret_cast<const TI*>(base) + ((static_cast<size_t>(b) * T + tau) * a.G + g) * N;
                        };
                    };
                    if (!dots_fetch<TI>(scr, scr_c, gb, c, T, draft_row(a.Bm), draft_row(a.C), N, &dots_bar, dpar,
                                        keep, lane, a.err, t0 + j)) {
                        if (lane == 0) s_abort = 1;
                        break;
                    }
                    dpar ^= 1u;
                    const TI* sbs = reinterpret_cast<const TI*>(scr);
                    const TI* scs = reinterpret_cast<const TI*>(scr_c);
#pragma unroll
                    for (int tau = 0; tau < TMAX; ++tau) bc[tau] = 0.f;
                    for (int qd = 0; 16 * qd < M; ++qd) {
                        Chunk4<TI> bq[4][CPL];
                        load_bquad<TI, CPL>(bq, qd, M, lane, cl, [&](int i) { return sbs + i * N; });
#pragma unroll
                        for (int tau = 0; tau < TMAX; ++tau) {
                            if (tau < T) {
                                float4 cv[CPL];
#pragma unroll
                                for (int q = 0; q < CPL; ++q) cv[q] = load4(scs + tau * N + (cl + 8 * q) * 4);
                                quad_dots<TI, CPL>(bc[tau], bq, cv, qd, c + tau + 1, lane);
                            }
                        }
                    }
                    __syncwarp();   // the scratch is read before the next key's copies
                    key_b = b; key_g = g; key_c = c;
                }
                float* dst = reinterpret_cast<float*>(dsm + static_cast<size_t>(s) * geo.bytes + geo.bcv);
#pragma unroll
                for (int tau = 0; tau < TMAX; ++tau)
                    if (tau < T) dst[tau * 32 + lane] = bc[tau];
            }
            __syncwarp();   // the dots are written before lane 0's arrive releases them
            if (lane == 0) mbar_arrive(&full_bar[s]);
            if (++s == S) { s = 0; ++round; }
            if (++hh == a.H) { hh = 0; ++b; g = 0; hin = 0; }
            else if (++hin == hpg) { hin = 0; ++g; }
        }
        return;
    }

    // --------------------------------------------------------------- consumers
    const int g = (tid - draft_lead<RF>()) / GT;
    const int gt = (tid - draft_lead<RF>()) - g * GT;
    const int lane = gt & 31, gw = gt >> 5;
    const int cl = lane & 7;
    const int rbase = gw * 16 + (lane >> 3) * 4;

    // records and drafts of the group's next tile, loaded one tile ahead:
    // lane i holds dt_i; xr[k] holds x of record cl + 8k for the lane's rows
    XRaw<TI> xr[4];
    uint32_t dtr = 0;
    auto prefetch = [&](int j) {
        const int c = s_cnt[j];
        if (c < 0) return;
        const int tile = t0 + j;
        const int bj = tile / a.H, hj = tile - bj * a.H;
        const size_t base = static_cast<size_t>(tile) * a.cap;
        const int M = c + T;
        if (lane < c) dtr = raw_of<TI>(reinterpret_cast<const TI*>(a.buf_dt) + base + lane);
        else if (lane < M)
            dtr = raw_of<TI>(reinterpret_cast<const TI*>(a.dt) + (static_cast<size_t>(bj) * T + (lane - c)) * a.H + hj);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int i = cl + 8 * k;
            if (i < c) xr[k].load(reinterpret_cast<const TI*>(a.buf_x) + (base + i) * P + rbase);
            else if (i < M)
                xr[k].load(reinterpret_cast<const TI*>(a.x) +
                           ((static_cast<size_t>(bj) * T + (i - c)) * a.H + hj) * P + rbase);
        }
    };
    if (g < nt) prefetch(g);

    int s = g % S;
    uint32_t round = static_cast<uint32_t>(g / S);
    int b = (t0 + g) / a.H, hh = (t0 + g) - b * a.H;
    int grp = hh / hpg, hin = hh - grp * hpg;
    int key_b = -1, key_g = -1, key_c = -1;
    int cf_b = -1, cf_g = -1;
    CFragMulti<N> cf;   // the drafts' C as MMA B fragments (bf16 inputs with a read copy)
    float bc[TMAX];   // lane i: B_i . C_tau
#pragma unroll
    for (int tau = 0; tau < TMAX; ++tau) bc[tau] = 0.f;

    for (int j = g; j < nt; j += NG) {
        const uint32_t par = round & 1u;
        int ok = 0;
        if (lane == 0) ok = (!s_abort && mbar_wait_bounded(&full_bar[s], par)) ? 1 : 0;
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) {
            if (lane == 0 && !s_abort) {
                report_error(a.err, kDevTimeout, t0 + j, 32);
                s_abort = 1;
            }
            break;
        }
        mbar_try_wait(&full_bar[s], par);

        const int tile = t0 + j;
        const unsigned char* st = dsm + static_cast<size_t>(s) * geo.bytes;
        const int c = s_cnt[j];
        if (c < 0) {
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty_bar[s]);
            if (j + NG < nt) prefetch(j + NG);
        } else {
            const int M = c + T;
            const TI* sbt = reinterpret_cast<const TI*>(st + geo.bt);
            const TI* sct = reinterpret_cast<const TI*>(st + geo.ct);
            if constexpr (kDotsWarp) {
                // formed by the dots warp
#pragma unroll
                for (int tau = 0; tau < TMAX; ++tau)
                    bc[tau] = reinterpret_cast<const float*>(st + geo.bcv)[min(tau, T - 1) * 32 + lane];
            } else if (b != key_b || grp != key_g || c != key_c) {
                // B_i . C_tau for every draft: each quad of B records is loaded
                // once and dotted with every draft's C
                const TI* gb = reinterpret_cast<const TI*>(a.buf_b) + (static_cast<size_t>(b) * a.G + grp) * a.cap * N;
#pragma unroll
                for (int tau = 0; tau < TMAX; ++tau) bc[tau] = 0.f;
                for (int qd = 0; 16 * qd < M; ++qd) {
                    Chunk4<TI> bq[4][CPL];
                    load_bquad<TI, CPL>(bq, qd, M, lane, cl,
                                        [&](int i) { return (i < c) ? gb + i * N : sbt + (i - c) * N; });
#pragma unroll
                    for (int tau = 0; tau < TMAX; ++tau) {
                        if (tau < T) {
                            float4 cv[CPL];
#pragma unroll
                            for (int q = 0; q < CPL; ++q) cv[q] = load4(sct + tau * N + (cl + 8 * q) * 4);
                            quad_dots<TI, CPL>(bc[tau], bq, cv, qd, c + tau + 1, lane);
                        }
                    }
                }
                key_b = b; key_g = grp; key_c = c;
            }
            // row-dots of this lane's 4 state rows with every draft's C, and
            // each draft's scale of them. Drafts past T repeat the last one,
            // so the loops have no data-dependent branches; their results are
            // dropped.
            float part[TMAX][4];
            float tsc[TMAX];
            if constexpr (RF == RSSM_READ_NONE) {
                // each state chunk is read once and used for all drafts (the
                // per-row FMA order is the one-token kernels')
                const float4* sh = reinterpret_cast<const float4*>(st + geo.state);
                float2 acc2[TMAX][4];
#pragma unroll
                for (int tau = 0; tau < TMAX; ++tau)
#pragma unroll
                    for (int p = 0; p < 4; ++p) acc2[tau][p] = make_float2(0.f, 0.f);
#pragma unroll
                for (int q = 0; q < CPL; ++q) {
                    float4 h[4];
#pragma unroll
                    for (int p = 0; p < 4; ++p) h[p] = sh[(rbase + p) * CH + cl + 8 * q];
#pragma unroll
                    for (int tau = 0; tau < TMAX; ++tau) {
                        const float4 cq = load4(sct + min(tau, T - 1) * N + (cl + 8 * q) * 4);
#pragma unroll
                        for (int p = 0; p < 4; ++p) {
                            acc2[tau][p] = __ffma2_rn(make_float2(h[p].x, h[p].y), make_float2(cq.x, cq.y), acc2[tau][p]);
                            acc2[tau][p] = __ffma2_rn(make_float2(h[p].z, h[p].w), make_float2(cq.z, cq.w), acc2[tau][p]);
                        }
                    }
                }
#pragma unroll
                for (int tau = 0; tau < TMAX; ++tau) {
                    tsc[tau] = 1.f;
#pragma unroll
                    for (int p = 0; p < 4; ++p) part[tau][p] = 0.f + acc2[tau][p].x + acc2[tau][p].y;   // as stage_row_dots sums it
                }
            } else if constexpr (kMma) {
                if (b != cf_b || grp != cf_g) {
                    make_cfrag_multi<N>(cf, reinterpret_cast<const __nv_bfloat16*>(sct), T, lane);
                    cf_b = b; cf_g = grp;
                }
                float d[4];   // rows gw*16 + lane/4 (d[0], d[1]) and + 8 (d[2], d[3]), drafts 2(lane%4) and + 1
                rc_mma_rows<RF, N>(d, st + geo.state, st + geo.bsc, cf.b, gw * 16, lane);
                const float ts = s_ts[kCopy ? j : 0];
                // draft tau's dot of row w (of the warp's 16) is in lane
                // 4 (w % 8) + tau / 2, element 2 (w / 8) + tau % 2; hand it to
                // lane cl = 0 of the row's group, whose 8-lane reduction in
                // nonflush_finish then sums it with zeros
#pragma unroll
                for (int tau = 0; tau < TMAX; ++tau) {
                    const int tq = min(tau, T - 1);
                    const float lo = (tq & 1) ? d[1] : d[0];
                    const float hi = (tq & 1) ? d[3] : d[2];
#pragma unroll
                    for (int p = 0; p < 4; ++p) {
                        const int w = (lane >> 3) * 4 + p;
                        const int src = 4 * (w & 7) + (tq >> 1);
                        const float vlo = __shfl_sync(0xffffffffu, lo, src);
                        const float vhi = __shfl_sync(0xffffffffu, hi, src);
                        part[tau][p] = (cl == 0) ? (w < 8 ? vlo : vhi) : 0.f;
                    }
                    tsc[tau] = ts * __shfl_sync(0xffffffffu, cf.inv_scale, 4 * tq);
                }
            } else {
                // FP32 inputs: the one-token kernels' decode and FMA order,
                // once per draft
                const float ts = s_ts[kCopy ? j : 0];
#pragma unroll
                for (int tau = 0; tau < TMAX; ++tau) {
                    float4 cv[CPL];
#pragma unroll
                    for (int q = 0; q < CPL; ++q) cv[q] = load4(sct + min(tau, T - 1) * N + (cl + 8 * q) * 4);
                    stage_row_dots<RF, CPL, N>(part[tau], st + geo.state, st + geo.bsc, cv, rbase, cl);
                    tsc[tau] = ts;
                }
            }
            // append the drafts' B records (once per B/C group), from the stage
            if (gw == GW - 1 && hin == 0) {
                uint4* bbp = reinterpret_cast<uint4*>(reinterpret_cast<TI*>(a.buf_b) +
                                                      ((static_cast<size_t>(b) * a.G + grp) * a.cap + c) * N);
                const uint4* bs = reinterpret_cast<const uint4*>(sbt);
                for (int q = lane; q < T * N * in_sz / 16; q += 32) bbp[q] = bs[q];
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty_bar[s]);

            // x and dt of the records and drafts, from the prefetch registers;
            // the drafts' x and dt are appended from there too
            float xk[4][4];
            const size_t base = static_cast<size_t>(tile) * a.cap;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int i = cl + 8 * k;
                if (i < M) xr[k].to(xk[k]);
                if (i >= c && i < M) store_x4raw<TI>(reinterpret_cast<TI*>(a.buf_x) + (base + i) * P + rbase, xr[k]);
            }
            const float dt_all = (lane < M) ? raw_to_f(dtr, static_cast<TI*>(nullptr)) : 0.f;
            if (gw == 0 && lane >= c && lane < M)
                store_raw<TI>(reinterpret_cast<TI*>(a.buf_dt) + base + lane, dtr);
            if (j + NG < nt) prefetch(j + NG);

            const float Ah = a.A[hh], Dh = a.D[hh];
            float rs[TMAX];
#pragma unroll
            for (int tau = 0; tau < TMAX; ++tau) {
                const int tq = min(tau, T - 1);
                const int m = c + tq + 1;
                const float dti = (lane < m) ? dt_all : 0.f;
                rs[tau] = nonflush_finish(part[tau], xk, dti, bc[tau], c + tq, m, Ah, Dh, tsc[tau], lane, cl);
            }
            if ((lane & 1) == 0) {
#pragma unroll
                for (int tau = 0; tau < TMAX; ++tau)
                    if (tau < T)
                        store_out(a.y, ((static_cast<size_t>(b) * T + tau) * a.H + hh) * P + rbase + ((lane & 7) >> 1),
                                  rs[tau], out_f32 != 0);
            }
        }
        s += NG;
        while (s >= S) { s -= S; ++round; }
        hh += NG;
        hin += NG;
        if (hh >= a.H) {
            hh -= a.H;
            ++b;
            grp = hh / hpg;
            hin = hh - grp * hpg;
        } else {
            while (hin >= hpg) { hin -= hpg; ++grp; }
        }
    }
}

template <class L, typename TI, int RF, int NG, int TMAX>
cudaError_t launch_draft_ng(const M2Args& a, int out_f32, int S, int grid, int per, size_t smem,
                            cudaStream_t s) {
    auto kernel = m2_replay_draft_tma_kernel<L, TI, RF, NG, TMAX>;
    static LaunchCache lc;
    cudaError_t e = cached_dyn_smem(lc, kernel, smem);
    if (e != cudaSuccess) return e;
    kernel<<<grid, draft_lead<RF>() + NG * L::kThreads, smem, s>>>(a, out_f32, S, per);
    return cudaGetLastError();
}

template <class L, typename TI, int RF, int TMAX>
cudaError_t launch_draft(const M2Args& a, int out_f32, cudaStream_t s) {
    const int total = a.B * a.H;
    if (total == 0) return cudaSuccess;
    int num_sms = 0, smem_optin = 0;
    cudaError_t e = device_limits(&num_sms, &smem_optin);
    if (e != cudaSuccess) return e;
    constexpr bool kSmall = L::kThreads <= 128;
    static LaunchCache lc;
    int static_smem = 0;
    e = cached_static_smem(lc, m2_replay_draft_tma_kernel<L, TI, RF, kSmall ? 2 : 1, TMAX>, &static_smem);
    if (e != cudaSuccess) return e;
    const DrGeom geo = draft_geom(L::P, L::N, a.T, static_cast<int>(sizeof(TI)), RF);
    const int scratch = (RF != RSSM_READ_NONE) ? align128((a.cap + a.T) * L::N * static_cast<int>(sizeof(TI)))
                                               : 0;   // the dots warp's
    const int avail = smem_optin - static_smem - 1024 - scratch;
    int smax = avail / geo.bytes;
    if (smax > kMaxStages) smax = kMaxStages;
    // each stage has one owner group: S is a multiple of the group count.
    // Two groups (168 registers a thread) measured faster than three (128
    // registers, with spills).
    // A read copy's small stages leave room for three groups (128 registers
    // a thread) with bf16 inputs: the copy path is bound by instruction
    // latency, not by bytes.
    constexpr bool kThree = kSmall && RF != RSSM_READ_NONE && sizeof(TI) == 2;
    const int ng = (kThree && smax >= 6) ? 3 : (kSmall && smax >= 4) ? 2 : 1;
    const int S = (smax / ng) * ng;
    if (S < 2) return cudaErrorInvalidConfiguration;
    int grid = num_sms;
    if ((total + grid - 1) / grid > kMaxTilesPerCta) grid = (total + kMaxTilesPerCta - 1) / kMaxTilesPerCta;
    if (grid > total) grid = total;
    const int per = (total + grid - 1) / grid;
    grid = (total + per - 1) / per;
    const size_t smem = static_cast<size_t>(S) * geo.bytes + scratch;
    if constexpr (kThree) {
        if (ng == 3) return launch_draft_ng<L, TI, RF, 3, TMAX>(a, out_f32, S, grid, per, smem, s);
    }
    if constexpr (kSmall) {
        if (ng == 2) return launch_draft_ng<L, TI, RF, 2, TMAX>(a, out_f32, S, grid, per, smem, s);
    }
    return launch_draft_ng<L, TI, RF, 1, TMAX>(a, out_f32, S, grid, per, smem, s);
}

template <class L, typename TI, int RF>
cudaError_t launch_draft_t(const M2Args& a, int out_f32, cudaStream_t s) {
    if (a.T <= 2) return launch_draft<L, TI, RF, 2>(a, out_f32, s);
    if (a.T <= 4) return launch_draft<L, TI, RF, 4>(a, out_f32, s);
    return launch_draft<L, TI, RF, kMaxDraft>(a, out_f32, s);
}

template <class L, typename TI>
cudaError_t launch_draft_rf(const M2Args& a, int out_f32, int rf, cudaStream_t s) {
    if (rf == RSSM_READ_FP8) return launch_draft_t<L, TI, RSSM_READ_FP8>(a, out_f32, s);
    if (rf == RSSM_READ_NVFP4) return launch_draft_t<L, TI, RSSM_READ_NVFP4>(a, out_f32, s);
    return launch_draft_t<L, TI, RSSM_READ_NONE>(a, out_f32, s);
}

template <class L>
cudaError_t run_draft(const M2Args& a, int in_dt, int out_dt, int rf, cudaStream_t s) {
    const int of = (out_dt == RSSM_F32);
    if (in_dt == RSSM_F32) return launch_draft_rf<L, float>(a, of, rf, s);
    return launch_draft_rf<L, __nv_bfloat16>(a, of, rf, s);
}

}  // namespace

cudaError_t m2_replay_draft(const M2Args& a, int P, int N, int in_dt, int out_dt, int rf, cudaStream_t s,
                            bool* supported) {
    *supported = true;
    if (a.T < 2 || a.T > kMaxDraft) return cudaErrorInvalidValue;
    if (a.ck != kCkF32) {   // drafts read an FP32 checkpoint or its copy
        *supported = false;
        return cudaSuccess;
    }
    if (P == 64 && N == 128) return run_draft<GTile<64, 128>>(a, in_dt, out_dt, rf, s);
    if (P == 64 && N == 64) return run_draft<GTile<64, 64>>(a, in_dt, out_dt, rf, s);
    if (P == 128 && N == 128) return run_draft<GTile<128, 128>>(a, in_dt, out_dt, rf, s);
    if (P == 128 && N == 64) return run_draft<GTile<128, 64>>(a, in_dt, out_dt, rf, s);
    *supported = false;
    return cudaSuccess;
}

}  // namespace rssm

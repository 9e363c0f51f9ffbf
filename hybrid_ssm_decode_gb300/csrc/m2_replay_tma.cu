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
//   y_t = gamma (h_ckpt C_t) + sum_{i<=m} w_i x_i + D x_t,
//   gamma = exp(A sum_{j<=m} dt_j),
//   w_i = exp(A sum_{i<j<=m} dt_j) dt_i (B_i . C_t)
//   flush: h_ckpt <- gamma h_ckpt + sum_i exp(A sum_{j>i} dt_j) dt_i x_i B_i^T
//
// Structure. One block per SM walks a contiguous range of (sequence, head)
// tiles (P x N FP32 each).
//  * Producer (one thread). Before the loop it reads the whole range's
//    record counts and step sizes, so it never waits on a dependent load. For
//    each tile it then fills one stage of a shared-memory ring with bulk
//    async copies (cp.async.bulk completing mbarrier transaction counts): the
//    checkpoint tile (or its FP8/NVFP4 read copy), the tile's buffered x and
//    dt records, its B/C group's B records, and this token's x, B and C.
//  * Consumers (NG = 2 groups of P/16 warps for P = 64, else 1 group). A
//    group takes every NG-th tile; its warps work independently:
//      - a warp covers 16 rows; 8 lanes share 4 consecutive rows and split
//        the columns, so a row-dot is a sum over 8 lanes and a record's x
//        values for a lane's rows are one 8-byte shared load;
//      - every warp scans the window's dt itself (decays and gamma stay in
//        registers, lane i holding record i);
//      - B_i . C_t depends only on (sequence, B/C group, record count), and a
//        group's tiles are neighbouring heads, so each warp keeps the dots in
//        registers and recomputes them only when that key changes;
//      - on a non-flush tile the warp forms its row-dots of the state with
//        C_t and loads its records' x values, then releases the stage before
//        the rest (decays, weights, reduction), so the producer refills the
//        stage while the warp works;
//      - lane cl adds records cl, cl+8, ... to its partial row sums before the
//        row reduction, so the buffered-input term needs no extra pass.
//    On a flush tile each warp folds the records into its values in
//    registers and writes them to global memory; only the read-copy writer
//    needs the whole tile (its amax), through a bounded mbarrier barrier.
// Every mbarrier wait is bounded (kWaitLimitNs). On expiry the kernel
// reports kDevTimeout in the error word, stops issuing, and waits (again
// bounded) for its own copies in flight before it returns.
#include "m2_pipeline.cuh"

namespace rssm {
namespace {

struct StageHdr {
    int c;            // records buffered before this token (-1: count out of range)
    uint32_t dt_raw;  // this token's dt, raw bits of the input dtype
    float tscale;     // read-copy tile scale (1 for the FP32 checkpoint)
    int pad;
};

struct StageGeom {
    int hdr, state, bsc, xrec, brec, dtrec, xt, bt, ct, bytes;
};

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

// NG consumer groups; S stages, a multiple of NG. Tile j uses stage j % S and
// group j % NG, so every stage has one owner group that consumes its rounds
// in order. A group therefore never tests a stage's full barrier for round r
// while round r-1 is still incomplete, which a parity wait could not tell
// apart from round r being complete.
// The stage's block-scale region exists when the copy or the checkpoint is NVFP4.
__host__ __device__ constexpr int stage_rf(int rf, int ck) {
    return (ck == kCkNVFP4) ? RSSM_READ_NVFP4 : rf;
}

// CK: the checkpoint's storage (kCkF32 / kCkF16 / kCkFP8 / kCkNVFP4). With a
// tile-format checkpoint and no separate copy, RF is that format and the
// read-copy pointers address the checkpoint itself.
template <class L, typename TI, int RF, int NG, int CK>
__global__ void __launch_bounds__(32 + NG * L::kThreads, 1)
m2_replay_step_tma_kernel(const M2Args a, const int out_f32, const int S, const int tiles_per_cta,
                          const int only_flush) {
    constexpr int CKF = ck_tile_fmt(CK);                 // tile format of the checkpoint, if any
    constexpr bool kAliased = (CKF != RSSM_READ_NONE && RF == CKF);   // the copy is the checkpoint
    constexpr int P = L::P, N = L::N, GT = L::kThreads, GW = L::kWarps;
    constexpr int in_sz = static_cast<int>(sizeof(TI));
    extern __shared__ __align__(128) unsigned char dsm[];
    __shared__ __align__(8) uint64_t full_bar[kMaxStages];
    __shared__ __align__(8) uint64_t empty_bar[kMaxStages];
    __shared__ __align__(8) uint64_t group_bar[NG];
    __shared__ int s_cnt[kMaxTilesPerCta];
    __shared__ uint32_t s_dtv[kMaxTilesPerCta];
    __shared__ float s_ts[RF != RSSM_READ_NONE ? kMaxTilesPerCta : 1];
    __shared__ float s_cts[CKF != RSSM_READ_NONE ? kMaxTilesPerCta : 1];
    __shared__ float g_red[NG][GW];
    __shared__ int s_list[kMaxTilesPerCta];   // only_flush: the range's flush tiles, in order
    __shared__ int s_nitems;
    __shared__ volatile int s_abort;

    const int total = a.B * a.H;
    // A flush-only launch takes every grid-th tile (block q: q, q + grid, ...):
    // a sequence's heads flush together, so contiguous ranges would pile the
    // flushing tiles onto a few blocks. Otherwise each block takes a range.
    const int t0 = blockIdx.x * tiles_per_cta;
    const int nt = only_flush ? max(0, (total - static_cast<int>(blockIdx.x) + static_cast<int>(gridDim.x) - 1) /
                                           static_cast<int>(gridDim.x))
                              : max(0, min(tiles_per_cta, total - t0));
    auto tile_at = [&](int j) { return only_flush ? static_cast<int>(blockIdx.x + j * gridDim.x) : t0 + j; };
    const StageGeom geo = stage_geom(P, N, a.cap, in_sz, stage_rf(RF, CK));
    const int tid = threadIdx.x;
    const int hpg = a.H / a.G;

    if (tid < 32) {
        for (int i = tid; i < nt; i += 32) {
            const int ti = tile_at(i);
            s_cnt[i] = a.counts[ti];
            s_dtv[i] = raw_of<TI>(reinterpret_cast<const TI*>(a.dt) + ti);
            if (RF != RSSM_READ_NONE) s_ts[RF != RSSM_READ_NONE ? i : 0] = a.rc_tscale[ti];
            if (CKF != RSSM_READ_NONE) s_cts[CKF != RSSM_READ_NONE ? i : 0] = a.ck_tscale[ti];
        }
        if (only_flush) {
            // the work items are the tiles that complete their window
            // (c = k - 1); the lean kernel of the same step takes the others
            __syncwarp();
            int n = 0;
            for (int i0 = 0; i0 < nt; i0 += 32) {
                const int i = i0 + tid;
                const bool f = i < nt && s_cnt[i] == a.k - 1;
                const unsigned bal = __ballot_sync(0xffffffffu, f);
                if (f) s_list[n + __popc(bal & ((1u << tid) - 1u))] = i;
                n += __popc(bal);
            }
            if (tid == 0) s_nitems = n;
        } else if (tid == 0) {
            s_nitems = nt;
        }
        if (tid == 0) {
            for (int s = 0; s < S; ++s) {
                mbar_init(&full_bar[s], 1);
                mbar_init(&empty_bar[s], GW);
            }
            for (int g = 0; g < NG; ++g) mbar_init(&group_bar[g], GW);
            s_abort = 0;
            fence_mbar_init();
        }
    }
    __syncthreads();

    if (tid < 32) {
        // ------------------------------------------------------------- producer
        if (tid != 0) return;
        const uint64_t pol = l2_evict_first();
        const uint64_t keep = l2_evict_last();   // records: read again later in the window
        uint32_t issued = 0, last_par = 0;
        int s = 0;
        uint32_t round = 0;
        const int nitems = s_nitems;
        for (int u = 0; u < nitems; ++u) {
            const int j = only_flush ? s_list[u] : u;
            const int b = tile_at(j) / a.H, hh = tile_at(j) - b * a.H;
            const int g = hh / hpg;
            if (s_abort) break;
            if (!mbar_wait_bounded(&empty_bar[s], (round & 1u) ^ 1u)) {
                report_error(a.err, kDevTimeout, tile_at(j), 0);
                s_abort = 1;
                break;
            }
            const int tile = tile_at(j);
            const int c = s_cnt[j];
            const bool cok = (c >= 0 && c < a.k);
            const int nrec = cok ? c : 0;
            const bool flush = cok && (c + 1 == a.k);
            const bool use_rc = (RF != RSSM_READ_NONE) && !flush;
            unsigned char* st = dsm + static_cast<size_t>(s) * geo.bytes;
            StageHdr* hdr = reinterpret_cast<StageHdr*>(st + geo.hdr);
            hdr->c = cok ? c : -1;
            hdr->dt_raw = s_dtv[j];
            hdr->tscale = (RF != RSSM_READ_NONE && use_rc) ? s_ts[RF != RSSM_READ_NONE ? j : 0]
                          : (CKF != RSSM_READ_NONE) ? s_cts[CKF != RSSM_READ_NONE ? j : 0] : 1.f;

            const size_t tile_off = static_cast<size_t>(tile) * P * N;
            // bytes of the stored tile (checkpoint or copy) in format f
            auto tile_bytes = [&](int f) -> uint32_t {
                return f == RSSM_READ_FP8 ? P * N : f == RSSM_READ_NVFP4 ? P * N / 2 : P * N * (CK == kCkF16 ? 2 : 4);
            };
            const int fmt = use_rc ? RF : CKF;
            const uint32_t state_bytes = tile_bytes(fmt);
            const uint32_t bsc_bytes = (fmt == RSSM_READ_NVFP4) ? P * N / 16 : 0;
            const uint32_t xrec_bytes = nrec * P * in_sz, brec_bytes = nrec * N * in_sz;
            const uint32_t dtrec_bytes = a.cap * in_sz;
            const uint32_t tok_bytes = P * in_sz + 2 * N * in_sz;
            mbar_arrive_expect_tx(&full_bar[s], state_bytes + bsc_bytes + xrec_bytes + brec_bytes +
                                                    dtrec_bytes + tok_bytes);
            const void* state_src;
            const unsigned char* ckb = reinterpret_cast<const unsigned char*>(a.ckpt);
            if (use_rc) state_src = a.rc_codes + (RF == RSSM_READ_FP8 ? tile_off : tile_off / 2);
            else if (CK == kCkF16) state_src = reinterpret_cast<const __half*>(a.ckpt) + tile_off;
            else if (CK == kCkFP8) state_src = ckb + tile_off;
            else if (CK == kCkNVFP4) state_src = ckb + tile_off / 2;
            else state_src = a.ckpt + tile_off;
            bulk_g2s_hint(st + geo.state, state_src, state_bytes, &full_bar[s], pol);
            if (bsc_bytes)
                bulk_g2s(st + geo.bsc, (use_rc ? a.rc_bscale : a.ck_bscale) + tile_off / 16, bsc_bytes, &full_bar[s]);
            const size_t grp_row = static_cast<size_t>(b) * a.G + g;
            const TI* bx = reinterpret_cast<const TI*>(a.buf_x) + static_cast<size_t>(tile) * a.cap * P;
            const TI* bb = reinterpret_cast<const TI*>(a.buf_b) + grp_row * a.cap * N;
            const TI* bdt = reinterpret_cast<const TI*>(a.buf_dt) + static_cast<size_t>(tile) * a.cap;
            if (xrec_bytes) bulk_g2s_hint(st + geo.xrec, bx, xrec_bytes, &full_bar[s], keep);
            if (brec_bytes) bulk_g2s_hint(st + geo.brec, bb, brec_bytes, &full_bar[s], keep);
            bulk_g2s_hint(st + geo.dtrec, bdt, dtrec_bytes, &full_bar[s], keep);
            bulk_g2s(st + geo.xt, reinterpret_cast<const TI*>(a.x) + static_cast<size_t>(tile) * P,
                     P * in_sz, &full_bar[s]);
            bulk_g2s(st + geo.bt, reinterpret_cast<const TI*>(a.Bm) + grp_row * N, N * in_sz, &full_bar[s]);
            bulk_g2s(st + geo.ct, reinterpret_cast<const TI*>(a.C) + grp_row * N, N * in_sz, &full_bar[s]);
            issued |= 1u << s;
            last_par = (last_par & ~(1u << s)) | ((round & 1u) << s);
            if (++s == S) { s = 0; ++round; }
        }
        // our own copies in flight must land before the block may exit
        for (int q = 0; q < S; ++q)
            if ((issued >> q) & 1u)
                if (!mbar_wait_bounded(&full_bar[q], (last_par >> q) & 1u))
                    report_error(a.err, kDevTimeout, t0, 1);
        return;
    }

    // --------------------------------------------------------------- consumers
    constexpr int CPL = L::CPL, CH = N / 4, JJ = L::J;
    const int g = (tid - 32) / GT;
    const int gt = (tid - 32) - g * GT;
    const int lane = gt & 31, gw = gt >> 5;
    const int cl = lane & 7;                          // column lane in the row group
    const int rbase = gw * 16 + (lane >> 3) * 4;      // first of this lane's 4 rows
    const uint64_t keep = l2_evict_last();            // record appends stay in L2

    // Bounded barrier of the group's warps (read-copy writer only): an
    // mbarrier that counts warps; every wait gives up after kWaitLimitNs.
    uint32_t gphase = 0;
    auto gsync = [&] {
        __syncwarp();
        int ok = 1;
        if (lane == 0) {
            mbar_arrive(&group_bar[g]);
            ok = mbar_wait_bounded(&group_bar[g], gphase) ? 1 : 0;
            if (!ok && !s_abort) {
                report_error(a.err, kDevTimeout, t0, 3);
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

    int s = g % S;
    uint32_t round = static_cast<uint32_t>(g / S);
    int key_b = -1, key_g = -1, key_c = -1;   // key of the dots held in bc
    float bc = 0.f;                          // lane i: B_i . C_t
    const int nitems = s_nitems;

    for (int u = g; u < nitems; u += NG) {
        const int j = only_flush ? s_list[u] : u;
        const int b = tile_at(j) / a.H, hh = tile_at(j) - b * a.H;
        const int grp = hh / hpg, hin = hh - grp * hpg;
        const uint32_t par = round & 1u;
        int ok = 0;
        if (lane == 0) ok = (!s_abort && mbar_wait_bounded(&full_bar[s], par)) ? 1 : 0;
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) {
            if (lane == 0 && !s_abort) {
                report_error(a.err, kDevTimeout, tile_at(j), 2);
                s_abort = 1;
            }
            break;
        }
        mbar_try_wait(&full_bar[s], par);   // acquire the bulk-copied bytes in every lane

        const int tile = tile_at(j);
        const unsigned char* st = dsm + static_cast<size_t>(s) * geo.bytes;
        const StageHdr hdr = *reinterpret_cast<const StageHdr*>(st + geo.hdr);
        const int c = hdr.c;
        bool released = false;
        if (c < 0) {
            if (gt == 0) report_error(a.err, RSSM_DEV_COUNT_RANGE, tile, s_cnt[j]);
        } else {
            const int m = c + 1;
            const bool flush = (m == a.k);
            const TI* sx = reinterpret_cast<const TI*>(st + geo.xrec);
            const TI* sb = reinterpret_cast<const TI*>(st + geo.brec);
            const TI* sdt = reinterpret_cast<const TI*>(st + geo.dtrec);
            const TI* sxt = reinterpret_cast<const TI*>(st + geo.xt);
            const TI* sbt = reinterpret_cast<const TI*>(st + geo.bt);
            const TI* sct = reinterpret_cast<const TI*>(st + geo.ct);
            float4 cv[CPL];
#pragma unroll
            for (int q = 0; q < CPL; ++q) cv[q] = load4(sct + (cl + 8 * q) * 4);

            // B_i . C_t for the window when the (sequence, group, count) key changed
            if (b != key_b || grp != key_g || c != key_c) {
                window_dots<TI, CPL>(bc, cv, m, lane, cl, [&](int i) { return (i < c) ? sb + i * N : sbt; });
                key_b = b; key_g = grp; key_c = c;
            }
            const float dt_t = raw_to_f(hdr.dt_raw, static_cast<TI*>(nullptr));
            const float dti = (lane < c) ? to_f(sdt[lane]) : (lane == c ? dt_t : 0.f);
            const float Dh = a.D[hh];
            const float Ah = a.A[hh];

            if (!flush) {
                // ---- read this warp's share of the stage: the checkpoint (or
                //      read copy) row-dots with C_t and its records' x values;
                //      then release the stage so the producer can refill it
                float part[4];
                stage_row_dots<(RF == RSSM_READ_NONE && CK == kCkF16) ? kReadF16Ckpt : RF, CPL, N>(
                    part, st + geo.state, st + geo.bsc, cv, rbase, cl);
                // x of this lane's rows for records cl, cl+8, cl+16, cl+24
                float xk[4][4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int i = cl + 8 * k;
                    if (i < m) load_x4<TI>(((i < c) ? sx + i * P : sxt) + rbase, xk[k]);
                }
                // append this token's record at slot c (16-byte vectors, from the stage)
                if (gw == 0) {
                    uint4* bx = reinterpret_cast<uint4*>(reinterpret_cast<TI*>(a.buf_x) +
                                                         (static_cast<size_t>(tile) * a.cap + c) * P);
                    const uint4* xs = reinterpret_cast<const uint4*>(sxt);
                    for (int q = lane; q < P * in_sz / 16; q += 32) st_keep_v4(bx + q, xs[q], keep);
                }
                if (gw == GW - 1 && hin == 0) {
                    uint4* bbp = reinterpret_cast<uint4*>(reinterpret_cast<TI*>(a.buf_b) +
                                                          ((static_cast<size_t>(b) * a.G + grp) * a.cap + c) * N);
                    const uint4* bs = reinterpret_cast<const uint4*>(sbt);
                    for (int q = lane; q < N * in_sz / 16; q += 32) st_keep_v4(bbp + q, bs[q], keep);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty_bar[s]);
                released = true;

                // ---- the rest from registers
                const float rs = nonflush_finish(part, xk, dti, bc, c, m, Ah, Dh, hdr.tscale, lane, cl);
                if ((lane & 1) == 0)
                    store_out(a.y, static_cast<size_t>(tile) * P + rbase + ((lane & 7) >> 1), rs, out_f32 != 0);
                if (gw == 0 && lane == 0) {
                    store_raw_keep<TI>(reinterpret_cast<TI*>(a.buf_dt) + static_cast<size_t>(tile) * a.cap + c,
                                       hdr.dt_raw, keep);
                    a.counts[tile] = m;
                }
            } else {
                // ---- flush: output, then fold the k records into this thread's
                //      values and write them once (the stage is held until the end)
                float gamma;
                const float decay = window_decay(dti, lane, m, Ah, gamma);
                const float cf = decay * dti;                    // dt_i prod_{j>i} a_j
                const float w = (lane < m) ? cf * bc : 0.f;
                float wk[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int i = cl + 8 * k;
                    wk[k] = __shfl_sync(0xffffffffu, w, i) + (i == c ? Dh : 0.f);
                }
                // the checkpoint's value at float4 index idx (FP32, or FP16 widened)
                auto ckv = [&](int idx) -> float4 {
                    if constexpr (CK == kCkF16) {
                        return f16x4_to_f32(reinterpret_cast<const uint2*>(st + geo.state)[idx]);
                    } else if constexpr (CK == kCkFP8) {
                        const uint32_t u = reinterpret_cast<const uint32_t*>(st + geo.state)[idx];
                        const float2 lo = e4m3x2_to_f2(static_cast<uint16_t>(u & 0xFFFFu));
                        const float2 hi = e4m3x2_to_f2(static_cast<uint16_t>(u >> 16));
                        const float ts = hdr.tscale;
                        return make_float4(__fmul_rn(lo.x, ts), __fmul_rn(lo.y, ts), __fmul_rn(hi.x, ts),
                                           __fmul_rn(hi.y, ts));
                    } else if constexpr (CK == kCkNVFP4) {
                        const uint32_t u = reinterpret_cast<const uint16_t*>(st + geo.state)[idx];
                        const int row = idx / CH, chunk = idx - row * CH;
                        const float es = __fmul_rn(e4m3_to_f((st + geo.bsc)[row * (N / 16) + (chunk >> 2)]), hdr.tscale);
                        const float2 lo = e2m1x2_to_f2(u & 0xFFu);
                        const float2 hi = e2m1x2_to_f2((u >> 8) & 0xFFu);
                        return make_float4(__fmul_rn(lo.x, es), __fmul_rn(lo.y, es), __fmul_rn(hi.x, es),
                                           __fmul_rn(hi.y, es));
                    } else {
                        return reinterpret_cast<const float4*>(st + geo.state)[idx];
                    }
                };
                float part[4];
#pragma unroll
                for (int p = 0; p < 4; ++p) {
                    float acc = 0.f;
#pragma unroll
                    for (int q = 0; q < CPL; ++q) acc += dot4(ckv(row_of(p * CPL + q) * CH + chunk_of(p * CPL + q)), cv[q]);
                    part[p] = gamma * acc;
                }
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int i = cl + 8 * k;
                    if (i < m) {
                        float xr[4];
                        load_x4<TI>(((i < c) ? sx + i * P : sxt) + rbase, xr);
#pragma unroll
                        for (int p = 0; p < 4; ++p) part[p] = fmaf(wk[k], xr[p], part[p]);
                    }
                }
                {
                    const float rs = group_reduce_multi<4, 8>(part, lane);
                    if ((lane & 1) == 0)
                        store_out(a.y, static_cast<size_t>(tile) * P + rbase + ((lane & 7) >> 1), rs,
                                  out_f32 != 0);
                }
                const size_t tile_off = static_cast<size_t>(tile) * P * N;
                float4 hv[JJ];
#pragma unroll
                for (int jj = 0; jj < JJ; ++jj) {
                    const float4 v = ckv(row_of(jj) * CH + chunk_of(jj));
                    hv[jj] = make_float4(v.x * gamma, v.y * gamma, v.z * gamma, v.w * gamma);
                }
                for (int i = 0; i < m; ++i) {
                    const float cfi = __shfl_sync(0xffffffffu, cf, i);
                    const TI* Bi = (i < c) ? sb + i * N : sbt;
                    float xr[4];
                    load_x4<TI>(((i < c) ? sx + i * P : sxt) + rbase, xr);
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
                if constexpr (CK == kCkF16) {
                    // the new checkpoint is rounded to FP16; the read copy is
                    // made from the rounded values
                    uint2* dst = reinterpret_cast<uint2*>(reinterpret_cast<__half*>(a.ckpt) + tile_off);
#pragma unroll
                    for (int jj = 0; jj < JJ; ++jj) {
                        const uint2 u = f32_to_f16x4(hv[jj]);
                        dst[row_of(jj) * CH + chunk_of(jj)] = u;
                        hv[jj] = f16x4_to_f32(u);
                    }
                } else if constexpr (CKF != RSSM_READ_NONE) {
                    // tile-format checkpoint: quantise the fold and keep the
                    // stored values for the copy
                    unsigned char* ckw = reinterpret_cast<unsigned char*>(a.ckpt);
                    write_read_copy<L, CKF, true>(hv, ckw + (CKF == RSSM_READ_FP8 ? tile_off : tile_off / 2),
                                                  CKF == RSSM_READ_NVFP4 ? a.ck_bscale + tile_off / 16 : nullptr,
                                                  a.ck_tscale + tile, g_red[g], gt, lane, gw, row_of, chunk_of, gsync);
                } else {
                    float4* dst = reinterpret_cast<float4*>(a.ckpt + tile_off);
#pragma unroll
                    for (int jj = 0; jj < JJ; ++jj) dst[row_of(jj) * CH + chunk_of(jj)] = hv[jj];
                }
                if (RF != RSSM_READ_NONE && !kAliased && !a.defer_copy) {
                    uint8_t* codes = a.rc_codes + (RF == RSSM_READ_FP8 ? tile_off : tile_off / 2);
                    uint8_t* bsc = (RF == RSSM_READ_NVFP4) ? a.rc_bscale + tile_off / 16 : nullptr;
                    write_read_copy<L, RF>(hv, codes, bsc, a.rc_tscale + tile, g_red[g], gt, lane, gw, row_of,
                                           chunk_of, gsync);
                }
                // a flush-only launch marks the tile with k: the lean launch
                // that follows in the same step resets it to 0 and skips it
                if (gt == 0) a.counts[tile] = only_flush ? a.k : 0;
            }
        }
        if (!released) {
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty_bar[s]);  // this warp is done with the stage
        }
        // next item of this group: NG items on
        s += NG;
        while (s >= S) { s -= S; ++round; }
    }
}

// ---------------------------------------------------------------------------
// Lean non-flush kernel: for launches in which no tile completes its window
// (the host knows every tile's record count is below k - 1). A stage holds only
// the checkpoint (or its read copy) and this token's x, B and C, so more of
// them fit in shared memory. Each lane loads the x and dt values of its own
// buffered records from global memory (where they sit in L2) one tile ahead,
// into registers. The window dots B_i . C_t depend only on (sequence, B/C
// group, count): a dots warp (warp 1; warp 0 is the producer) forms them once
// per key and per block, instead of every consumer warp forming them, and
// every stage carries them (B256 lean launch, FP8 copy: 141 -> 117 us). The
// arithmetic is the fused kernel's (the shared functions above).
// A tile whose count is out of range for this kernel is reported
// (RSSM_DEV_COUNT_RANGE) and left unchanged.
// ---------------------------------------------------------------------------
struct NfGeom {
    int hdr, bcv, state, bsc, xt, bt, ct, bytes;
};

__host__ __device__ inline NfGeom nf_geom(int P, int N, int in_sz, int rf) {
    NfGeom g;
    int off = 0;
    g.hdr = off;   off += 128;
    g.bcv = off;   off += 128;   // the window dots B_i . C_t (float i = record i)
    g.state = off; off += align128(rf == RSSM_READ_NONE ? P * N * 4 : rf == kReadF16Ckpt ? P * N * 2
                                                                  : (rf == RSSM_READ_FP8 ? P * N : P * N / 2));
    g.bsc = off;   off += (rf == RSSM_READ_NVFP4) ? align128(P * N / 16) : 0;
    g.xt = off;    off += align128(P * in_sz);
    g.bt = off;    off += align128(N * in_sz);
    g.ct = off;    off += align128(N * in_sz);
    g.bytes = off;
    return g;
}

template <class L, typename TI, int RF, int NG>
__global__ void __launch_bounds__(64 + NG * L::kThreads, 1)
m2_replay_nf_kernel(const M2Args a, const int out_f32, const int S, const int tiles_per_cta,
                    const int skip_flush) {
    constexpr int P = L::P, N = L::N, GT = L::kThreads, GW = L::kWarps, CPL = L::CPL;
    constexpr int in_sz = static_cast<int>(sizeof(TI));
    extern __shared__ __align__(128) unsigned char dsm[];
    __shared__ __align__(8) uint64_t full_bar[kMaxStages];
    __shared__ __align__(8) uint64_t empty_bar[kMaxStages];
    __shared__ int s_cnt[kMaxTilesPerCta];
    __shared__ uint32_t s_dtv[kMaxTilesPerCta];
    constexpr bool kCopy = (RF == RSSM_READ_FP8 || RF == RSSM_READ_NVFP4);   // the stage holds a read copy
    __shared__ float s_ts[kCopy ? kMaxTilesPerCta : 1];
    __shared__ __align__(8) uint64_t dots_bar;   // the dots warp's scratch copies
    __shared__ volatile int s_abort;

    const int total = a.B * a.H;
    const int t0 = blockIdx.x * tiles_per_cta;
    const int nt = max(0, min(tiles_per_cta, total - t0));
    const NfGeom geo = nf_geom(P, N, in_sz, RF);
    const int tid = threadIdx.x;
    const int hpg = a.H / a.G;

    if (tid < 32) {
        for (int i = tid; i < nt; i += 32) {
            int c = a.counts[t0 + i];
            if (skip_flush && c == a.k) {
                // flushed by the flush-only launch that ran first in this step
                a.counts[t0 + i] = 0;
                c = -2;
            }
            s_cnt[i] = c;
            s_dtv[i] = raw_of<TI>(reinterpret_cast<const TI*>(a.dt) + t0 + i);
            if (kCopy) s_ts[kCopy ? i : 0] = a.rc_tscale[t0 + i];
        }
        if (tid == 0) {
            for (int q = 0; q < S; ++q) {
                mbar_init(&full_bar[q], 2);   // the producer and the dots warp
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
                report_error(a.err, kDevTimeout, t0 + j, 20);
                s_abort = 1;
                break;
            }
            const int tile = t0 + j;
            const int c = s_cnt[j];
            const bool cok = (c >= 0 && c + 1 < a.k);
            unsigned char* st = dsm + static_cast<size_t>(s) * geo.bytes;
            StageHdr* hdr = reinterpret_cast<StageHdr*>(st + geo.hdr);
            if (c == -2) {
                // flushed already in this step: nothing to copy
                hdr->c = -2;
                mbar_arrive_expect_tx(&full_bar[s], 0);
                issued |= 1u << s;
                last_par = (last_par & ~(1u << s)) | ((round & 1u) << s);
                if (++s == S) { s = 0; ++round; }
                if (++hh == a.H) { hh = 0; ++b; g = 0; hin = 0; }
                else if (++hin == hpg) { hin = 0; ++g; }
                continue;
            }
            hdr->c = cok ? c : -1;
            hdr->dt_raw = s_dtv[j];
            hdr->tscale = kCopy ? s_ts[kCopy ? j : 0] : 1.f;
            const size_t tile_off = static_cast<size_t>(tile) * P * N;
            const uint32_t state_bytes = (RF == RSSM_READ_NONE) ? P * N * 4
                                         : (RF == kReadF16Ckpt) ? P * N * 2
                                         : (RF == RSSM_READ_FP8 ? P * N : P * N / 2);
            const uint32_t bsc_bytes = (RF == RSSM_READ_NVFP4) ? P * N / 16 : 0;
            const uint32_t tok_bytes = P * in_sz + 2 * N * in_sz;
            mbar_arrive_expect_tx(&full_bar[s], state_bytes + bsc_bytes + tok_bytes);
            const void* state_src;
            if (RF == RSSM_READ_NONE) state_src = a.ckpt + tile_off;
            else if (RF == kReadF16Ckpt) state_src = reinterpret_cast<const __half*>(a.ckpt) + tile_off;
            else if (RF == RSSM_READ_FP8) state_src = a.rc_codes + tile_off;
            else state_src = a.rc_codes + tile_off / 2;
            bulk_g2s_hint(st + geo.state, state_src, state_bytes, &full_bar[s], pol);
            if (bsc_bytes) bulk_g2s(st + geo.bsc, a.rc_bscale + tile_off / 16, bsc_bytes, &full_bar[s]);
            const size_t grp_row = static_cast<size_t>(b) * a.G + g;
            bulk_g2s(st + geo.xt, reinterpret_cast<const TI*>(a.x) + static_cast<size_t>(tile) * P,
                     P * in_sz, &full_bar[s]);
            bulk_g2s(st + geo.bt, reinterpret_cast<const TI*>(a.Bm) + grp_row * N, N * in_sz, &full_bar[s]);
            bulk_g2s(st + geo.ct, reinterpret_cast<const TI*>(a.C) + grp_row * N, N * in_sz, &full_bar[s]);
            issued |= 1u << s;
            last_par = (last_par & ~(1u << s)) | ((round & 1u) << s);
            if (++s == S) { s = 0; ++round; }
            if (++hh == a.H) { hh = 0; ++b; g = 0; hin = 0; }
            else if (++hin == hpg) { hin = 0; ++g; }
        }
        for (int q = 0; q < S; ++q)
            if ((issued >> q) & 1u)
                if (!mbar_wait_bounded(&full_bar[q], (last_par >> q) & 1u))
                    report_error(a.err, kDevTimeout, t0, 21);
        return;
    }

    if (tid < 64) {
        // ------------------------------------------------------------ dots warp
        // The window dots B_i . C_t depend only on the key (sequence, B/C
        // group, count). This warp forms them with the consumers' former
        // arithmetic (window_dots, from the same values, copied into its
        // scratch in one round trip) when the key changes. Every stage
        // carries its key's dots and completes only with this warp's arrive
        // (the full barriers count the producer's arrive and this one), so the
        // copies are not held up meanwhile.
        const int lane = tid - 32, cl = lane & 7;
        const uint64_t keep = l2_evict_last();   // records are read again by later steps of the window
        unsigned char* scr = dsm + static_cast<size_t>(S) * geo.bytes;        // B rows: records, then the token
        unsigned char* scr_c = scr + static_cast<size_t>(a.cap) * N * in_sz;  // C row
        uint32_t dpar = 0;
        int s = 0;
        uint32_t round = 0;
        int b = t0 / a.H, hh = t0 - b * a.H;
        int g = hh / hpg, hin = hh - g * hpg;
        int key_b = -1, key_g = -1, key_c = -1;
        float bc = 0.f;   // lane i: B_i . C_t of the current key
        for (int j = 0; j < nt; ++j) {
            int ok = 1;
            if (lane == 0) {
                if (s_abort) {
                    ok = 0;
                } else if (!mbar_wait_bounded(&empty_bar[s], (round & 1u) ^ 1u)) {
                    report_error(a.err, kDevTimeout, t0 + j, 23);
                    s_abort = 1;
                    ok = 0;
                }
            }
            if (!__shfl_sync(0xffffffffu, ok, 0)) break;
            const int c = s_cnt[j];
            if (c >= 0 && c + 1 < a.k) {
                if (b != key_b || g != key_g || c != key_c) {
                    const size_t grp_row = static_cast<size_t>(b) * a.G + g;
                    const TI* gb = reinterpret_cast<const TI*>(a.buf_b) + grp_row * a.cap * N;
                    auto tok = [&](const void* base) {
                        return [=](int) { return reinterpret_cast<const TI*>(base) + grp_row * N; };
                    };
                    if (!dots_fetch<TI>(scr, scr_c, gb, c, 1, tok(a.Bm), tok(a.C), N, &dots_bar, dpar, keep, lane,
                                        a.err, t0 + j)) {
                        if (lane == 0) s_abort = 1;
                        break;
                    }
                    dpar ^= 1u;
                    const TI* sbs = reinterpret_cast<const TI*>(scr);
                    const TI* scs = reinterpret_cast<const TI*>(scr_c);
                    float4 cv[CPL];
#pragma unroll
                    for (int q = 0; q < CPL; ++q) cv[q] = load4(scs + (cl + 8 * q) * 4);
                    window_dots<TI, CPL>(bc, cv, c + 1, lane, cl, [&](int i) { return sbs + i * N; });
                    __syncwarp();   // the scratch is read before the next key's copies
                    key_b = b; key_g = g; key_c = c;
                }
                reinterpret_cast<float*>(dsm + static_cast<size_t>(s) * geo.bytes + geo.bcv)[lane] = bc;
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
    const int g = (tid - 64) / GT;
    const int gt = (tid - 64) - g * GT;
    const int lane = gt & 31, gw = gt >> 5;
    const int cl = lane & 7;
    const int rbase = gw * 16 + (lane >> 3) * 4;
    const uint64_t keep = l2_evict_last();   // records are read again by later steps of the window

    // records of the group's next tile, loaded one tile ahead
    XRaw<TI> xr[4];
    uint32_t dtr = 0;
    auto prefetch = [&](int j) {
        const int c = s_cnt[j];
        if (c < 0 || c + 1 >= a.k) return;
        const size_t base = static_cast<size_t>(t0 + j) * a.cap;
        if (lane < c) dtr = raw_keep<TI>(reinterpret_cast<const TI*>(a.buf_dt) + base + lane, keep);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int i = cl + 8 * k;
            if (i < c) xr[k].load_keep(reinterpret_cast<const TI*>(a.buf_x) + (base + i) * P + rbase, keep);
        }
    };
    if (g < nt) prefetch(g);

    int s = g % S;
    uint32_t round = static_cast<uint32_t>(g / S);
    int b = (t0 + g) / a.H, hh = (t0 + g) - b * a.H;
    int grp = hh / hpg, hin = hh - grp * hpg;
    // read-copy row-dots on the tensor cores (bf16 inputs): C_t's B fragments,
    // rebuilt when the (sequence, B/C group) changes. The FP16 checkpoint keeps
    // the FP32-pipe row-dots: its values need no decoding, and the MMA path's
    // fragment shuffles made it slower.
    constexpr bool kMma = kCopy && sizeof(TI) == 2;
    CFrag<N> cf;
    int cf_b = -1, cf_g = -1;

    for (int j = g; j < nt; j += NG) {
        const uint32_t par = round & 1u;
        int ok = 0;
        if (lane == 0) ok = (!s_abort && mbar_wait_bounded(&full_bar[s], par)) ? 1 : 0;
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) {
            if (lane == 0 && !s_abort) {
                report_error(a.err, kDevTimeout, t0 + j, 22);
                s_abort = 1;
            }
            break;
        }
        mbar_try_wait(&full_bar[s], par);

        const int tile = t0 + j;
        const unsigned char* st = dsm + static_cast<size_t>(s) * geo.bytes;
        const StageHdr hdr = *reinterpret_cast<const StageHdr*>(st + geo.hdr);
        const int c = hdr.c;
        if (c < 0) {
            if (c == -1 && gt == 0) report_error(a.err, RSSM_DEV_COUNT_RANGE, tile, s_cnt[j]);
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty_bar[s]);
            if (j + NG < nt) prefetch(j + NG);
        } else {
            const int m = c + 1;
            const TI* sxt = reinterpret_cast<const TI*>(st + geo.xt);
            const TI* sbt = reinterpret_cast<const TI*>(st + geo.bt);
            const TI* sct = reinterpret_cast<const TI*>(st + geo.ct);
            const float bc = reinterpret_cast<const float*>(st + geo.bcv)[lane];   // formed by the producer warp
            float part[4];
            float tscale = hdr.tscale;
            if constexpr (kMma) {
                if (b != cf_b || grp != cf_g) {
                    make_cfrag<N>(cf, reinterpret_cast<const __nv_bfloat16*>(sct), lane);
                    cf_b = b; cf_g = grp;
                }
                float dA, dB;   // rows gw*16 + lane/4 and + 8
                rc_row_dots_mma<RF, N>(dA, dB, st + geo.state, st + geo.bsc, cf, gw * 16, lane);
                // hand each row's dot to lane cl = 0 of its row group; the
                // 8-lane reduction in nonflush_finish then sums it with zeros
#pragma unroll
                for (int p = 0; p < 4; ++p) {
                    const int w = (lane >> 3) * 4 + p;          // row within the warp's 16
                    const float vA = __shfl_sync(0xffffffffu, dA, 4 * (w & 7));
                    const float vB = __shfl_sync(0xffffffffu, dB, 4 * (w & 7));
                    part[p] = (cl == 0) ? (w < 8 ? vA : vB) : 0.f;
                }
                tscale *= cf.inv_scale;
            } else {
                float4 cv[CPL];
#pragma unroll
                for (int q = 0; q < CPL; ++q) cv[q] = load4(sct + (cl + 8 * q) * 4);
                stage_row_dots<RF, CPL, N>(part, st + geo.state, st + geo.bsc, cv, rbase, cl);
            }
            float xk[4][4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int i = cl + 8 * k;
                if (i < c) xr[k].to(xk[k]);
                else if (i == c) load_x4<TI>(sxt + rbase, xk[k]);
            }
            const float dt_t = raw_to_f(hdr.dt_raw, static_cast<TI*>(nullptr));
            const float dti = (lane < c) ? raw_to_f(dtr, static_cast<TI*>(nullptr)) : (lane == c ? dt_t : 0.f);
            // append this token's record at slot c (16-byte vectors, from the stage)
            if (gw == 0) {
                uint4* bx = reinterpret_cast<uint4*>(reinterpret_cast<TI*>(a.buf_x) +
                                                     (static_cast<size_t>(tile) * a.cap + c) * P);
                const uint4* xs = reinterpret_cast<const uint4*>(sxt);
                for (int q = lane; q < P * in_sz / 16; q += 32) st_keep_v4(bx + q, xs[q], keep);
            }
            if (gw == GW - 1 && hin == 0) {
                uint4* bbp = reinterpret_cast<uint4*>(reinterpret_cast<TI*>(a.buf_b) +
                                                      ((static_cast<size_t>(b) * a.G + grp) * a.cap + c) * N);
                const uint4* bs = reinterpret_cast<const uint4*>(sbt);
                for (int q = lane; q < N * in_sz / 16; q += 32) st_keep_v4(bbp + q, bs[q], keep);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty_bar[s]);
            if (j + NG < nt) prefetch(j + NG);

            const float rs = nonflush_finish(part, xk, dti, bc, c, m, a.A[hh], a.D[hh], tscale, lane, cl);
            if ((lane & 1) == 0)
                store_out(a.y, static_cast<size_t>(tile) * P + rbase + ((lane & 7) >> 1), rs, out_f32 != 0);
            if (gw == 0 && lane == 0) {
                store_raw_keep<TI>(reinterpret_cast<TI*>(a.buf_dt) + static_cast<size_t>(tile) * a.cap + c, hdr.dt_raw, keep);
                a.counts[tile] = m;
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

// ---------------------------------------------------------------------------
// Direct non-flush kernel for small batches: one block per tile and no
// pipeline. With few tiles per SM the persistent kernel's ring has nothing to
// overlap, and its setup and bulk-copy round trips set the step time. Here
// every consumer lane loads its 4 rows of the FP32 checkpoint, this token's
// inputs and its records straight from global memory (the state at these
// batch sizes sits in L2) and runs the lean kernel's arithmetic (the shared
// functions above, in the same order), so the outputs and records are the
// same bits. skip_flush: as in the lean kernel.
// ---------------------------------------------------------------------------
template <class L, typename TI>
__global__ void __launch_bounds__(L::kThreads)
m2_replay_nf_direct_kernel(const M2Args a, const int out_f32, const int skip_flush) {
    constexpr int P = L::P, N = L::N, GW = L::kWarps, CPL = L::CPL;
    constexpr int in_sz = static_cast<int>(sizeof(TI));
    const int tile = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, gw = tid >> 5;
    const int cl = lane & 7;
    const int rbase = gw * 16 + (lane >> 3) * 4;
    const int hpg = a.H / a.G;
    const int b = tile / a.H, hh = tile - b * a.H;
    const int grp = hh / hpg, hin = hh - grp * hpg;
    const uint64_t keep = l2_evict_last();
    const size_t grp_row = static_cast<size_t>(b) * a.G + grp;
    const TI* xt = reinterpret_cast<const TI*>(a.x) + static_cast<size_t>(tile) * P;
    const TI* bt = reinterpret_cast<const TI*>(a.Bm) + grp_row * N;
    const TI* ct = reinterpret_cast<const TI*>(a.C) + grp_row * N;
    const TI* gb = reinterpret_cast<const TI*>(a.buf_b) + grp_row * a.cap * N;
    const size_t base = static_cast<size_t>(tile) * a.cap;

    // Every load that does not depend on the record count is issued with it:
    // the records of every slot a non-flush window can hold (c < k - 1), the
    // first quad of B records, this token's inputs and the state row-dots.
    const int c = a.counts[tile];
    const int kmax = a.k - 1;
    XRaw<TI> xr[4];
    uint32_t dtr = 0;
    if (lane < kmax) dtr = raw_keep<TI>(reinterpret_cast<const TI*>(a.buf_dt) + base + lane, keep);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int i = cl + 8 * k;
        if (i < kmax) xr[k].load_keep(reinterpret_cast<const TI*>(a.buf_x) + (base + i) * P + rbase, keep);
    }
    Chunk4<TI> bq[4][CPL], btq[CPL];
    load_bquad<TI, CPL>(bq, 0, kmax, lane, cl, [&](int i) { return gb + i * N; }, kmax, keep);
#pragma unroll
    for (int q = 0; q < CPL; ++q) btq[q].load(bt + (cl + 8 * q) * 4);
    float4 cv[CPL];
#pragma unroll
    for (int q = 0; q < CPL; ++q) cv[q] = load4(ct + (cl + 8 * q) * 4);
    float part[4];
    stage_row_dots<RSSM_READ_NONE, CPL, N>(part, reinterpret_cast<const unsigned char*>(a.ckpt + static_cast<size_t>(tile) * P * N),
                                          nullptr, cv, rbase, cl);
    const uint32_t dt_raw = raw_of<TI>(reinterpret_cast<const TI*>(a.dt) + tile);

    if (skip_flush && c == a.k) {   // flushed by the flush-only launch of this step
        __syncthreads();
        if (tid == 0) a.counts[tile] = 0;
        return;
    }
    if (c < 0 || c + 1 >= a.k) {
        if (tid == 0) report_error(a.err, RSSM_DEV_COUNT_RANGE, tile, c);
        return;
    }
    const int m = c + 1;
    // the window's B records as window_dots reads them: record c is this
    // token's B, records past it are zero
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
        const int i = (lane >> 3) + 4 * kk;
#pragma unroll
        for (int q = 0; q < CPL; ++q) {
            if (i == c) bq[kk][q] = btq[q];
            else if (i > c) bq[kk][q].zero();
        }
    }
    float bc = 0.f;
    quad_dots<TI, CPL>(bc, bq, cv, 0, m, lane);
    for (int qd = 1; 16 * qd < m; ++qd) {   // windows past 16 records
        Chunk4<TI> bq2[4][CPL];
        load_bquad<TI, CPL>(bq2, qd, m, lane, cl, [&](int i) { return (i < c) ? gb + i * N : bt; }, c, keep);
        quad_dots<TI, CPL>(bc, bq2, cv, qd, m, lane);
    }
    float xk[4][4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int i = cl + 8 * k;
        if (i < c) xr[k].to(xk[k]);
        else if (i == c) load_x4<TI>(xt + rbase, xk[k]);
    }
    const float dt_t = raw_to_f(dt_raw, static_cast<TI*>(nullptr));
    const float dti = (lane < c) ? raw_to_f(dtr, static_cast<TI*>(nullptr)) : (lane == c ? dt_t : 0.f);
    // append this token's record at slot c
    if (gw == 0) {
        uint4* bx = reinterpret_cast<uint4*>(reinterpret_cast<TI*>(a.buf_x) + (base + c) * P);
        const uint4* xs = reinterpret_cast<const uint4*>(xt);
        for (int q = lane; q < P * in_sz / 16; q += 32) st_keep_v4(bx + q, xs[q], keep);
    }
    if (gw == GW - 1 && hin == 0) {
        uint4* bbp = reinterpret_cast<uint4*>(reinterpret_cast<TI*>(a.buf_b) + (grp_row * a.cap + c) * N);
        const uint4* bs = reinterpret_cast<const uint4*>(bt);
        for (int q = lane; q < N * in_sz / 16; q += 32) st_keep_v4(bbp + q, bs[q], keep);
    }
    const float rs = nonflush_finish(part, xk, dti, bc, c, m, a.A[hh], a.D[hh], 1.f, lane, cl);
    if ((lane & 1) == 0) store_out(a.y, static_cast<size_t>(tile) * P + rbase + ((lane & 7) >> 1), rs, out_f32 != 0);
    // every warp has read the count and the records before they move
    __syncthreads();
    if (tid == 0) {
        store_raw_keep<TI>(reinterpret_cast<TI*>(a.buf_dt) + base + c, dt_raw, keep);
        a.counts[tile] = m;
    }
}

// Direct flush kernel for small batches (FP32 checkpoint, no read copy): one
// block per tile, no pipeline. Every load is issued with the count: the tile,
// this token's inputs and the window's records (B, x, dt), which the block
// then keeps in shared memory, so the launch waits on one round of loads.
// Then the step kernel's flush arithmetic, in the same order: the output of
// the token that completes the window, then the fold of its k records into
// the checkpoint, written once. A tile whose count is not k - 1 is left
// alone; in a step that runs only this kernel (every tile due) it is
// reported. only_flush: the flushed tile is marked with count k for the lean
// launch that follows in the same step.
template <class L, typename TI>
__global__ void __launch_bounds__(L::kThreads)
m2_replay_flush_direct_kernel(const M2Args a, const int out_f32, const int only_flush) {
    constexpr int P = L::P, N = L::N, CPL = L::CPL, CH = N / 4, JJ = L::J, NTHR = L::kThreads;
    constexpr int in_sz = static_cast<int>(sizeof(TI));
    constexpr int BCH = N * in_sz / 16, XCH = P * in_sz / 16;        // 16-byte chunks of a B / x record
    constexpr int BPT = (kMaxCap * BCH + NTHR - 1) / NTHR;         // of them per thread, at most
    constexpr int XPT = (kMaxCap * XCH + NTHR - 1) / NTHR;
    __shared__ __align__(16) unsigned char s_b[kMaxCap * N * in_sz];   // B records, slot c: this token's B
    __shared__ __align__(16) unsigned char s_x[kMaxCap * P * in_sz];   // x records, slot c: this token's x
    const int tile = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, gw = tid >> 5;
    const int cl = lane & 7;
    const int rbase = gw * 16 + (lane >> 3) * 4;
    const int hpg = a.H / a.G;
    const int b = tile / a.H, hh = tile - b * a.H;
    const int grp = hh / hpg;
    const size_t grp_row = static_cast<size_t>(b) * a.G + grp;
    const size_t tile_off = static_cast<size_t>(tile) * P * N;
    const TI* xt = reinterpret_cast<const TI*>(a.x) + static_cast<size_t>(tile) * P;
    const TI* bt = reinterpret_cast<const TI*>(a.Bm) + grp_row * N;
    const TI* ct = reinterpret_cast<const TI*>(a.C) + grp_row * N;
    const uint4* gx = reinterpret_cast<const uint4*>(reinterpret_cast<const TI*>(a.buf_x) +
                                                     static_cast<size_t>(tile) * a.cap * P);
    const uint4* gb = reinterpret_cast<const uint4*>(reinterpret_cast<const TI*>(a.buf_b) + grp_row * a.cap * N);
    const TI* gdt = reinterpret_cast<const TI*>(a.buf_dt) + static_cast<size_t>(tile) * a.cap;
    auto row_of = [&](int j) { return rbase + j / CPL; };
    auto chunk_of = [&](int j) { return cl + 8 * (j % CPL); };

    const int c = a.counts[tile];
    const int cm = a.k - 1;   // the count of a tile that flushes
    uint4 breg[BPT], xreg[XPT];
#pragma unroll
    for (int i = 0; i < BPT; ++i) {
        const int q = tid + i * NTHR, j = q / BCH;
        breg[i] = (j < cm) ? gb[q] : (j == cm) ? reinterpret_cast<const uint4*>(bt)[q - j * BCH]
                                               : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int i = 0; i < XPT; ++i) {
        const int q = tid + i * NTHR, j = q / XCH;
        xreg[i] = (j < cm) ? gx[q] : (j == cm) ? reinterpret_cast<const uint4*>(xt)[q - j * XCH]
                                               : make_uint4(0u, 0u, 0u, 0u);
    }
    const uint32_t dtr = (lane < cm) ? raw_of<TI>(gdt + lane) : 0u;
    const float4* ck = reinterpret_cast<const float4*>(a.ckpt + tile_off);
    float4 hv[JJ];
#pragma unroll
    for (int jj = 0; jj < JJ; ++jj) hv[jj] = ck[row_of(jj) * CH + chunk_of(jj)];
    float4 cv[CPL];
#pragma unroll
    for (int q = 0; q < CPL; ++q) cv[q] = load4(ct + (cl + 8 * q) * 4);
    const uint32_t dt_raw = raw_of<TI>(reinterpret_cast<const TI*>(a.dt) + tile);
    const float Dh = a.D[hh], Ah = a.A[hh];

    if (c != cm) {
        if (!only_flush && tid == 0) report_error(a.err, RSSM_DEV_COUNT_RANGE, tile, c);
        return;
    }
    const int m = c + 1;
#pragma unroll
    for (int i = 0; i < BPT; ++i) {
        const int q = tid + i * NTHR;
        if (q < m * BCH) reinterpret_cast<uint4*>(s_b)[q] = breg[i];
    }
#pragma unroll
    for (int i = 0; i < XPT; ++i) {
        const int q = tid + i * NTHR;
        if (q < m * XCH) reinterpret_cast<uint4*>(s_x)[q] = xreg[i];
    }
    __syncthreads();   // also: every thread has read the tile and the count
    const TI* sb = reinterpret_cast<const TI*>(s_b);
    const TI* sx = reinterpret_cast<const TI*>(s_x);

    float bc;
    window_dots<TI, CPL>(bc, cv, m, lane, cl, [&](int i) { return sb + i * N; });
    const float dt_t = raw_to_f(dt_raw, static_cast<TI*>(nullptr));
    const float dti = (lane < c) ? raw_to_f(dtr, static_cast<TI*>(nullptr)) : (lane == c ? dt_t : 0.f);
    float gamma;
    const float decay = window_decay(dti, lane, m, Ah, gamma);
    const float cf = decay * dti;                    // dt_i prod_{j>i} a_j
    const float w = (lane < m) ? cf * bc : 0.f;
    float wk[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int i = cl + 8 * k;
        wk[k] = __shfl_sync(0xffffffffu, w, i) + (i == c ? Dh : 0.f);
    }
    // output of the flushing token (the step kernel's order)
    float part[4];
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        float acc = 0.f;
#pragma unroll
        for (int q = 0; q < CPL; ++q) acc += dot4(hv[p * CPL + q], cv[q]);
        part[p] = gamma * acc;
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int i = cl + 8 * k;
        if (i < m) {
            float xr[4];
            load_x4<TI>(sx + i * P + rbase, xr);
#pragma unroll
            for (int p = 0; p < 4; ++p) part[p] = fmaf(wk[k], xr[p], part[p]);
        }
    }
    {
        const float rs = group_reduce_multi<4, 8>(part, lane);
        if ((lane & 1) == 0) store_out(a.y, static_cast<size_t>(tile) * P + rbase + ((lane & 7) >> 1), rs, out_f32 != 0);
    }
    // fold: h <- gamma h + sum_i cf_i x_i B_i^T
#pragma unroll
    for (int jj = 0; jj < JJ; ++jj) hv[jj] = make_float4(hv[jj].x * gamma, hv[jj].y * gamma, hv[jj].z * gamma, hv[jj].w * gamma);
    for (int i = 0; i < m; ++i) {
        const float cfi = __shfl_sync(0xffffffffu, cf, i);
        const TI* Bi = sb + i * N;
        float xr[4];
        load_x4<TI>(sx + i * P + rbase, xr);
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
    float4* dst = reinterpret_cast<float4*>(a.ckpt + tile_off);
#pragma unroll
    for (int jj = 0; jj < JJ; ++jj) dst[row_of(jj) * CH + chunk_of(jj)] = hv[jj];
    if (tid == 0) a.counts[tile] = only_flush ? a.k : 0;
}

// Tiles up to which a non-flush step of FP32-checkpoint replay runs the direct
// kernel instead of the persistent one.
constexpr int kDirectTilesPerSm = 16;


template <class L, typename TI, int RF, int NG, int CK>
cudaError_t launch_tma_ng(const M2Args& a, int out_f32, int S, int grid, int per, size_t smem, int only_flush,
                          cudaStream_t s) {
    auto kernel = m2_replay_step_tma_kernel<L, TI, RF, NG, CK>;
    static LaunchCache lc;
    cudaError_t e = cached_dyn_smem(lc, kernel, smem);
    if (e != cudaSuccess) return e;
    kernel<<<grid, 32 + NG * L::kThreads, smem, s>>>(a, out_f32, S, per, only_flush);
    return cudaGetLastError();
}

// only_flush: the launch takes only the tiles that complete their window and
// marks them with count k; the lean kernel, run next with skip_flush in the
// same step, takes the rest and resets the marks.
template <class L, typename TI, int RF, int CK>
cudaError_t launch_tma(const M2Args& a, int out_f32, int only_flush, cudaStream_t s) {
    const int total = a.B * a.H;
    if (total == 0) return cudaSuccess;
    int num_sms = 0, smem_optin = 0;
    cudaError_t e = device_limits(&num_sms, &smem_optin);
    if (e != cudaSuccess) return e;
    // two consumer groups for tiles of up to 64 rows (a 288-thread block
    // keeps the fold in registers), else one; size the ring for that kernel
    constexpr bool kTwo = L::kThreads <= 128;
    static LaunchCache lc;
    int static_smem = 0;
    e = cached_static_smem(lc, m2_replay_step_tma_kernel<L, TI, RF, kTwo ? 2 : 1, CK>, &static_smem);
    if (e != cudaSuccess) return e;
    const StageGeom geo = stage_geom(L::P, L::N, a.cap, static_cast<int>(sizeof(TI)), stage_rf(RF, CK));
    const int avail = smem_optin - static_smem - 1024;
    int smax = avail / geo.bytes;
    if (smax > kMaxStages) smax = kMaxStages;
    const int ng = (kTwo && smax >= 4) ? 2 : 1;
    const int S = (smax / ng) * ng;
    if (S < 2) return cudaErrorInvalidConfiguration;
    int grid = num_sms;
    if ((total + grid - 1) / grid > kMaxTilesPerCta) grid = (total + kMaxTilesPerCta - 1) / kMaxTilesPerCta;
    if (grid > total) grid = total;
    const int per = (total + grid - 1) / grid;
    grid = (total + per - 1) / per;
    const size_t smem = static_cast<size_t>(S) * geo.bytes;
    if constexpr (kTwo) {
        if (ng == 2) return launch_tma_ng<L, TI, RF, 2, CK>(a, out_f32, S, grid, per, smem, only_flush, s);
    }
    return launch_tma_ng<L, TI, RF, 1, CK>(a, out_f32, S, grid, per, smem, only_flush, s);
}

template <class L, typename TI, int RF, int NG>
cudaError_t launch_nf_ng(const M2Args& a, int out_f32, int S, int grid, int per, size_t smem, int skip_flush,
                         cudaStream_t s) {
    auto kernel = m2_replay_nf_kernel<L, TI, RF, NG>;
    static LaunchCache lc;
    cudaError_t e = cached_dyn_smem(lc, kernel, smem);
    if (e != cudaSuccess) return e;
    kernel<<<grid, 64 + NG * L::kThreads, smem, s>>>(a, out_f32, S, per, skip_flush);
    return cudaGetLastError();
}

// skip_flush: the flush-only launch of the same step ran first and marked the
// tiles it flushed with count k; this launch resets them to 0 and skips them.
template <class L, typename TI, int RF>
cudaError_t launch_nf(const M2Args& a, int out_f32, int skip_flush, cudaStream_t s) {
    const int total = a.B * a.H;
    if (total == 0) return cudaSuccess;
    int num_sms = 0, smem_optin = 0;
    cudaError_t e = device_limits(&num_sms, &smem_optin);
    if (e != cudaSuccess) return e;
    constexpr bool kSmall = L::kThreads <= 128;
    static LaunchCache lc;
    int static_smem = 0;
    e = cached_static_smem(lc, m2_replay_nf_kernel<L, TI, RF, kSmall ? 3 : 1>, &static_smem);
    if (e != cudaSuccess) return e;
    const NfGeom geo = nf_geom(L::P, L::N, static_cast<int>(sizeof(TI)), RF);
    const int scratch = align128((a.cap + 1) * L::N * static_cast<int>(sizeof(TI)));   // the dots warp's
    const int avail = smem_optin - static_smem - 1024 - scratch;
    int smax = avail / geo.bytes;
    if (smax > kMaxStages) smax = kMaxStages;
    // each stage has one owner group: S is a multiple of the group count
    int ng = 1;
    if (kSmall && smax >= 6) ng = 3;
    else if (kSmall && smax >= 4) ng = 2;
    const int S = (smax / ng) * ng;
    if (S < 2) return cudaErrorInvalidConfiguration;
    int grid = num_sms;
    if ((total + grid - 1) / grid > kMaxTilesPerCta) grid = (total + kMaxTilesPerCta - 1) / kMaxTilesPerCta;
    if (grid > total) grid = total;
    const int per = (total + grid - 1) / grid;
    grid = (total + per - 1) / per;
    const size_t smem = static_cast<size_t>(S) * geo.bytes + scratch;
    if constexpr (kSmall) {
        if (ng == 3) return launch_nf_ng<L, TI, RF, 3>(a, out_f32, S, grid, per, smem, skip_flush, s);
        if (ng == 2) return launch_nf_ng<L, TI, RF, 2>(a, out_f32, S, grid, per, smem, skip_flush, s);
    }
    return launch_nf_ng<L, TI, RF, 1>(a, out_f32, S, grid, per, smem, skip_flush, s);
}

template <class L, typename TI, int RF>
cudaError_t launch_path(const M2Args& a, int out_f32, int path, cudaStream_t s) {
    const bool lean = (path == kStepNonFlush || path == kStepSkipFlush);
    if constexpr (RF == RSSM_READ_NONE) {
        int num_sms = 0, smem_optin = 0;
        cudaError_t e = device_limits(&num_sms, &smem_optin);
        if (e != cudaSuccess) return e;
        const int total = a.B * a.H;
        if (total > 0 && total <= kDirectTilesPerSm * num_sms) {
            // a one-token step with every tile flushing, or the flush part of
            // a split step; kStepAny otherwise means mixed counts, which the
            // host sends to the split path
            if (lean) m2_replay_nf_direct_kernel<L, TI><<<total, L::kThreads, 0, s>>>(a, out_f32, path == kStepSkipFlush);
            else m2_replay_flush_direct_kernel<L, TI><<<total, L::kThreads, 0, s>>>(a, out_f32, path == kStepFlushOnly);
            return cudaGetLastError();
        }
    }
    if (lean) return launch_nf<L, TI, RF>(a, out_f32, path == kStepSkipFlush, s);
    return launch_tma<L, TI, RF, kCkF32>(a, out_f32, path == kStepFlushOnly, s);
}

// Low-precision checkpoints (bf16 inputs). FP16: the lean kernel reads the
// FP16 tile when there is no read copy; the fused kernel folds in FP32 and
// stores FP16. Tile formats: the lean kernel reads the copy, which is the
// checkpoint itself when no separate copy is configured; the fused kernel
// decodes, folds in FP32 and re-quantises.
template <class L, int RF, int CK>
cudaError_t launch_path_ck(const M2Args& a, int out_f32, int path, cudaStream_t s) {
    if (path == kStepNonFlush || path == kStepSkipFlush)
        return launch_nf<L, __nv_bfloat16, (RF == RSSM_READ_NONE && CK == kCkF16) ? kReadF16Ckpt : RF>(
            a, out_f32, path == kStepSkipFlush, s);
    return launch_tma<L, __nv_bfloat16, RF, CK>(a, out_f32, path == kStepFlushOnly, s);
}

template <class L>
cudaError_t run_tma(const M2Args& a, int in_dt, int out_dt, int rf, int path, cudaStream_t s) {
    const int of = (out_dt == RSSM_F32);
    if (a.ck != kCkF32) {
        if (in_dt != RSSM_BF16) return cudaErrorInvalidValue;
        if (a.ck == kCkF16) {
            if (rf == RSSM_READ_FP8) return launch_path_ck<L, RSSM_READ_FP8, kCkF16>(a, of, path, s);
            if (rf == RSSM_READ_NVFP4) return launch_path_ck<L, RSSM_READ_NVFP4, kCkF16>(a, of, path, s);
            return launch_path_ck<L, RSSM_READ_NONE, kCkF16>(a, of, path, s);
        }
        if (a.ck == kCkFP8) {
            if (rf == RSSM_READ_NVFP4) return launch_path_ck<L, RSSM_READ_NVFP4, kCkFP8>(a, of, path, s);
            if (rf == RSSM_READ_FP8) return launch_path_ck<L, RSSM_READ_FP8, kCkFP8>(a, of, path, s);
            return cudaErrorInvalidValue;
        }
        if (rf == RSSM_READ_NVFP4) return launch_path_ck<L, RSSM_READ_NVFP4, kCkNVFP4>(a, of, path, s);
        return cudaErrorInvalidValue;
    }
    if (in_dt == RSSM_F32) {
        if (rf == RSSM_READ_FP8) return launch_path<L, float, RSSM_READ_FP8>(a, of, path, s);
        if (rf == RSSM_READ_NVFP4) return launch_path<L, float, RSSM_READ_NVFP4>(a, of, path, s);
        return launch_path<L, float, RSSM_READ_NONE>(a, of, path, s);
    }
    if (rf == RSSM_READ_FP8) return launch_path<L, __nv_bfloat16, RSSM_READ_FP8>(a, of, path, s);
    if (rf == RSSM_READ_NVFP4) return launch_path<L, __nv_bfloat16, RSSM_READ_NVFP4>(a, of, path, s);
    return launch_path<L, __nv_bfloat16, RSSM_READ_NONE>(a, of, path, s);
}

}  // namespace

cudaError_t m2_replay_step(const M2Args& a, int P, int N, int in_dt, int out_dt, int rf, int path,
                           cudaStream_t s, bool* supported) {
    *supported = true;
    if (P == 64 && N == 128) return run_tma<GTile<64, 128>>(a, in_dt, out_dt, rf, path, s);
    if (P == 64 && N == 64) return run_tma<GTile<64, 64>>(a, in_dt, out_dt, rf, path, s);
    if (P == 128 && N == 128) return run_tma<GTile<128, 128>>(a, in_dt, out_dt, rf, path, s);
    if (P == 128 && N == 64) return run_tma<GTile<128, 64>>(a, in_dt, out_dt, rf, path, s);
    *supported = false;
    return cudaSuccess;
}

}  // namespace rssm

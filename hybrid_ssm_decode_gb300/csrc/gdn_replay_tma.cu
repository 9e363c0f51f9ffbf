// Gated DeltaNet ReplaySSM decode step (one token per sequence), persistent
// and pipelined for GB300.
//
// Method: "ReplaySSM beschleunigt ...", section "Wichtige Details" (Gated
// DeltaNet); "NVIDIA ve Dao AI Lab, ... ReplaySSM'i sundu", section "Durum
// trafigini azaltma ve rollback'in basitlestirilmesi" (output-only
// evaluation, the intermediate state formed by two small matrix products).
//
// Window algebra (records j = 0..c since the checkpoint S0, record c is this
// token; gamma = prod_{l<=c} alpha_l, rho_j = prod_{j<l<=c} alpha_l):
//   u_c = beta_c (v_c - gamma S0 k_c - sum_{j<c} rho_j (k_j . k_c) u_j)
//   o_c = gamma S0 (scale q) + sum_{j<c} rho_j (k_j . scale q) u_j + (k_c . scale q) u_c
//   flush: S0 <- gamma S0 + sum_{j<=c} rho_j u_j k_j^T
// u_j is row j of U = T (V - diag(gamma) K S0^T), T = (I + diag(beta) A)^-1
// diag(beta), solved by forward substitution when token j arrives and kept in
// the record. Each step evaluates the two products S0 [k_c ; q] and the masked
// (q K^T) U.
//
// Structure. One block per SM walks a contiguous range of (sequence, head)
// tiles. A work item is one 64-row half of a tile's d_v x d_k FP32 state, so a
// stage holds 32 KiB of state like the Mamba-2 kernel.
//  * Producer (one thread): reads the range's record counts and gates up
//    front, then fills the shared-memory ring with bulk async copies: the
//    half-tile of S0, the tile's k and alpha records, the half's u records,
//    and this token's q, k and half of v.
//  * Consumers (NG groups of 4 warps): a group takes every NG-th work item,
//    and each warp forms the item's key dots (k_j . k_c, k_j . q) itself,
//    four records per pass (no cross-warp step). A warp covers 16 rows; 8 lanes share 4 consecutive rows and split
//    the columns, so each row-dot is a sum over 8 lanes, and one 8-value
//    reduction gives both -gamma S0 k - sum rho kappa u and gamma S0 q +
//    sum rho lambda u for the lane's rows.
// Every wait is bounded (kWaitLimitNs); on expiry the kernel reports
// kDevTimeout and stops, after waiting (bounded) for its own copies.
#include "gdn_pipeline.cuh"

namespace rssm {
namespace {

struct GHdr {
    int c;        // records buffered before this token (-1: count out of range)
    float alpha;  // this token's gate
    float beta;
    int pad;
};

struct GGeom {
    int hdr, state, krec, urec, arec, qt, kt, vt, vrec, brec, bytes;
};

// Read-copy writer traits for one 64-row half (4 warps, DK columns).
template <int DK>
struct GdnHalfRC {
    static constexpr int kWarps = 4, N = DK;
};

// rf FP8 / NVFP4 (a read copy): the stage also holds the half's v records
// and the tile's beta records, from which a flush replays the window.
// rf kGdnF16: the checkpoint half is stored in FP16.
__host__ __device__ inline GGeom gstage_geom(int DK, int cap, int in_sz, int rf) {
    const bool copy = (rf == RSSM_READ_FP8 || rf == RSSM_READ_NVFP4);
    GGeom g;
    int off = 0;
    g.hdr = off;   off += 128;
    g.state = off; off += galign128(64 * DK * (rf == kGdnF16 ? 2 : 4));
    g.krec = off;  off += galign128(cap * DK * in_sz);
    g.urec = off;  off += galign128(cap * 64 * 4);
    g.arec = off;  off += galign128(cap * 4);
    g.qt = off;    off += galign128(DK * in_sz);
    g.kt = off;    off += galign128(DK * in_sz);
    g.vt = off;    off += galign128(64 * in_sz);
    g.vrec = off;  off += copy ? galign128(cap * 64 * in_sz) : 0;
    g.brec = off;  off += copy ? galign128(cap * 4) : 0;
    g.bytes = off;
    return g;
}

template <class L, typename TI, int NG, int RF>
__global__ void __launch_bounds__(32 + NG * L::kThreads, 1)
gdn_replay_step_tma_kernel(const GDNArgs a, const int out_f32, const int S, const int tiles_per_cta,
                           const int only_flush) {
    constexpr int DV = L::DV, DK = L::DK, HALVES = L::HALVES, GT = L::kThreads, GW = L::kWarps;
    constexpr int CPL = L::CPL, CH = DK / 4, JJ = L::J;
    constexpr int in_sz = static_cast<int>(sizeof(TI));
    extern __shared__ __align__(128) unsigned char dsm[];
    __shared__ __align__(8) uint64_t full_bar[kMaxStages];
    __shared__ __align__(8) uint64_t empty_bar[kMaxStages];
    __shared__ int s_cnt[kMaxTilesPerCta];
    __shared__ float s_al[kMaxTilesPerCta], s_be[kMaxTilesPerCta];
    __shared__ __align__(8) uint64_t group_bar[NG];   // read-copy writer only
    __shared__ float g_red[NG][GW];
    __shared__ int s_list[kMaxTilesPerCta];   // only_flush: the range's flush tiles, in order
    __shared__ int s_ntl;
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
    const GGeom geo = gstage_geom(DK, a.cap, in_sz, RF);
    constexpr bool kCopy = (RF == RSSM_READ_FP8 || RF == RSSM_READ_NVFP4);   // a read copy
    constexpr bool k16 = (RF == kGdnF16);                                    // an FP16 checkpoint
    const int tid = threadIdx.x;

    if (tid < 32) {
        for (int i = tid; i < nt; i += 32) {
            const int ti = tile_at(i);
            s_cnt[i] = a.counts[ti];
            s_al[i] = a.alpha[ti];
            s_be[i] = a.beta[ti];
        }
        if (only_flush) {
            // the work items are the halves of the tiles that complete their
            // window (c = k - 1); the lean kernel of the same step takes the others
            __syncwarp();
            int n = 0;
            for (int i0 = 0; i0 < nt; i0 += 32) {
                const int i = i0 + tid;
                const bool f = i < nt && s_cnt[i] == a.kflush - 1;
                const unsigned bal = __ballot_sync(0xffffffffu, f);
                if (f) s_list[n + __popc(bal & ((1u << tid) - 1u))] = i;
                n += __popc(bal);
            }
            if (tid == 0) s_ntl = n;
        } else if (tid == 0) {
            s_ntl = nt;
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
    const int ni = s_ntl * HALVES;
    auto tile_of_item = [&](int w) { return only_flush ? s_list[w / HALVES] : w / HALVES; };

    if (tid < 32) {
        // ------------------------------------------------------------- producer
        if (tid != 0) return;
        const uint64_t pol = l2_evict_first();
        uint32_t issued = 0, last_par = 0;
        int s = 0;
        uint32_t round = 0;
        for (int w = 0; w < ni; ++w) {
            if (s_abort) break;
            if (!mbar_wait_bounded(&empty_bar[s], (round & 1u) ^ 1u)) {
                report_error(a.err, kDevTimeout, t0, 10);
                s_abort = 1;
                break;
            }
            const int tl = tile_of_item(w), half = w % HALVES;
            const int tile = tile_at(tl);
            const int c = s_cnt[tl];
            const bool cok = (c >= 0 && c < a.kflush);
            const int nrec = cok ? c : 0;
            unsigned char* st = dsm + static_cast<size_t>(s) * geo.bytes;
            GHdr* hdr = reinterpret_cast<GHdr*>(st + geo.hdr);
            hdr->c = cok ? c : -1;
            hdr->alpha = s_al[tl];
            hdr->beta = s_be[tl];
            const uint32_t state_bytes = 64 * DK * (k16 ? 2 : 4);
            const uint32_t krec_bytes = nrec * DK * in_sz, urec_bytes = nrec * 64 * 4;
            const uint32_t arec_bytes = a.cap * 4;
            const uint32_t tok_bytes = 2 * DK * in_sz + 64 * in_sz;
            const uint32_t vrec_bytes = kCopy ? nrec * 64 * in_sz : 0;
            const uint32_t brec_bytes = kCopy ? a.cap * 4 : 0;
            mbar_arrive_expect_tx(&full_bar[s], state_bytes + krec_bytes + urec_bytes + arec_bytes + tok_bytes +
                                                    vrec_bytes + brec_bytes);
            const size_t bh = static_cast<size_t>(tile);
            if (k16)
                bulk_g2s_hint(st + geo.state, reinterpret_cast<const __half*>(a.ckpt) + (bh * DV + half * 64) * DK,
                              state_bytes, &full_bar[s], pol);
            else
                bulk_g2s_hint(st + geo.state, a.ckpt + (bh * DV + half * 64) * DK, state_bytes, &full_bar[s], pol);
            if (krec_bytes)
                bulk_g2s(st + geo.krec, reinterpret_cast<const TI*>(a.buf_k) + bh * a.cap * DK, krec_bytes,
                         &full_bar[s]);
            if (urec_bytes)
                bulk_g2s(st + geo.urec, a.buf_u + (bh * HALVES + half) * a.cap * 64, urec_bytes, &full_bar[s]);
            bulk_g2s(st + geo.arec, a.buf_a + bh * a.cap, arec_bytes, &full_bar[s]);
            bulk_g2s(st + geo.qt, reinterpret_cast<const TI*>(a.q) + bh * DK, DK * in_sz, &full_bar[s]);
            bulk_g2s(st + geo.kt, reinterpret_cast<const TI*>(a.k) + bh * DK, DK * in_sz, &full_bar[s]);
            bulk_g2s(st + geo.vt, reinterpret_cast<const TI*>(a.v) + bh * DV + half * 64, 64 * in_sz,
                     &full_bar[s]);
            if (vrec_bytes)
                bulk_g2s(st + geo.vrec, reinterpret_cast<const TI*>(a.buf_v) + (bh * HALVES + half) * a.cap * 64,
                         vrec_bytes, &full_bar[s]);
            if (brec_bytes) bulk_g2s(st + geo.brec, a.buf_beta + bh * a.cap, brec_bytes, &full_bar[s]);
            issued |= 1u << s;
            last_par = (last_par & ~(1u << s)) | ((round & 1u) << s);
            if (++s == S) { s = 0; ++round; }
        }
        for (int q = 0; q < S; ++q)
            if ((issued >> q) & 1u)
                if (!mbar_wait_bounded(&full_bar[q], (last_par >> q) & 1u))
                    report_error(a.err, kDevTimeout, t0, 11);
        return;
    }

    // --------------------------------------------------------------- consumers
    const int g = (tid - 32) / GT;
    const int gt = (tid - 32) - g * GT;
    const int lane = gt & 31, gw = gt >> 5;
    const int cl = lane & 7;
    const int rloc = gw * 16 + (lane >> 3) * 4;   // first of the lane's 4 rows in the half
    auto row_of = [&](int j) { return rloc + j / CPL; };
    auto chunk_of = [&](int j) { return cl + 8 * (j % CPL); };
    // bounded barrier of the group's warps (read-copy writer only)
    uint32_t gphase = 0;
    auto gsync = [&] {
        __syncwarp();
        int ok = 1;
        if (lane == 0) {
            mbar_arrive(&group_bar[g]);
            ok = mbar_wait_bounded(&group_bar[g], gphase) ? 1 : 0;
            if (!ok && !s_abort) {
                report_error(a.err, kDevTimeout, t0, 13);
                s_abort = 1;
            }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (ok) mbar_try_wait(&group_bar[g], gphase);
        gphase ^= 1u;
        __syncwarp();
    };

    for (int w = g; w < ni; w += NG) {
        {
            const int tl = tile_of_item(w), half = w % HALVES;
            const int tile = tile_at(tl);
            const int s = w % S;
            const uint32_t par = static_cast<uint32_t>(w / S) & 1u;
            int ok = 0;
            if (lane == 0) ok = (!s_abort && mbar_wait_bounded(&full_bar[s], par)) ? 1 : 0;
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) {
                if (lane == 0 && !s_abort) {
                    report_error(a.err, kDevTimeout, tile, 12);
                    s_abort = 1;
                }
                return;
            }
            mbar_try_wait(&full_bar[s], par);

            const unsigned char* st = dsm + static_cast<size_t>(s) * geo.bytes;
            const GHdr hdr = *reinterpret_cast<const GHdr*>(st + geo.hdr);
            const int c = hdr.c;
            const int m = c + 1;
            const TI* sk = reinterpret_cast<const TI*>(st + geo.krec);
            const float* su = reinterpret_cast<const float*>(st + geo.urec);
            const float* sa = reinterpret_cast<const float*>(st + geo.arec);
            const TI* sq = reinterpret_cast<const TI*>(st + geo.qt);
            const TI* skt = reinterpret_cast<const TI*>(st + geo.kt);
            const TI* sv = reinterpret_cast<const TI*>(st + geo.vt);

            float4 kv[CPL], qv[CPL];
#pragma unroll
            for (int q = 0; q < CPL; ++q) {
                kv[q] = load4(skt + (cl + 8 * q) * 4);
                const float4 t = load4(sq + (cl + 8 * q) * 4);
                qv[q] = make_float4(t.x * a.scale, t.y * a.scale, t.z * a.scale, t.w * a.scale);
            }

            // a read-copy flush replays the window from the FP32 half and needs
            // none of the window-form terms below
            const bool replay = kCopy && c >= 0 && (m == a.kflush);
            float kap = 0.f, lam = 0.f;   // lane j: k_j . k_c and k_j . (scale q)
            if (!replay)
                gdn_key_dots<CPL>(kap, lam, kv, qv, m, lane, [&](int qd, int kk, int q) {
                    const int j = 16 * qd + (lane >> 3) + 4 * kk;
                    return (j < c) ? load4(sk + j * DK + (cl + 8 * q) * 4) : (j == c ? kv[q] : zero4());
                });
            if (c < 0) {
                if (gt == 0 && half == 0) report_error(a.err, RSSM_DEV_COUNT_RANGE, tile, s_cnt[tl]);
            } else {
                const bool flush = (m == a.kflush);
                const HalfRef<k16> sh{st + geo.state};
                const int rr = rloc + (cl & 3);                           // this lane's row (cl < 4)
                float gamma = 1.f, rho = 1.f, uc = 0.f, o = 0.f;
                if (!replay) {
                    // decay products of the window (lane j holds record j)
                    const float al = (lane < c) ? sa[lane] : (lane == c ? hdr.alpha : 1.f);
                    rho = window_rho(al, lane, m, gamma);
                    const float wk = (lane < c) ? rho * kap : 0.f;   // weights of u_j in u_c
                    const float wq = (lane < c) ? rho * lam : 0.f;   // weights of u_j in o_c
                    const float lam_c = __shfl_sync(0xffffffffu, lam, c & 31);

                    // S0 [k ; q] for the lane's rows, unscaled; then u_c and o_c
                    float pk[4], pq[4];
                    gdn_state_dots<CPL, DK>(pk, pq, sh, kv, qv, rloc, cl);
                    float uk[4][4];
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const int j = cl + 8 * kk;
                        if (j < c) load_u4(su + j * 64 + rloc, uk[kk]);
                    }
                    gdn_finish(pk, pq, uk, gamma, wk, wq, c, lane, cl, to_f(sv[rr]), hdr.beta, lam_c, &uc, &o);
                    if (cl < 4) store_out(a.o, static_cast<size_t>(tile) * DV + half * 64 + rr, o, out_f32 != 0);
                }

                if (!flush) {
                    // append this token's record at slot c: u rows of this half; k, alpha once
                    // (with a read copy also v and beta, which a flush replays). With
                    // max_draft = 1 every count is known, so a read-copy layer only
                    // reaches this kernel on flush steps; this branch reads the FP32 half.
                    const size_t slot = ((static_cast<size_t>(tile) * HALVES + half) * a.cap + c) * 64 + rr;
                    if (cl < 4) a.buf_u[slot] = uc;
                    if (kCopy && cl < 4) reinterpret_cast<TI*>(a.buf_v)[slot] = sv[rr];
                    if (kCopy && half == 0 && gt == 0)
                        a.buf_beta[static_cast<size_t>(tile) * a.cap + c] = hdr.beta;
                    if (half == 0 && gw == 0) {
                        uint4* bk = reinterpret_cast<uint4*>(reinterpret_cast<TI*>(a.buf_k) +
                                                             (static_cast<size_t>(tile) * a.cap + c) * DK);
                        const uint4* ks = reinterpret_cast<const uint4*>(skt);
                        for (int q = lane; q < DK * in_sz / 16; q += 32) bk[q] = ks[q];
                        if (lane == 0) a.buf_a[static_cast<size_t>(tile) * a.cap + c] = hdr.alpha;
                    }
                    if (half == HALVES - 1 && gt == 0) a.counts[tile] = m;
                } else if constexpr (kCopy) {
                    // replay the window through the recurrence from the FP32 half
                    // (the stored u rows were formed from the copy), then write the
                    // half and its copy
                    float4 hv[JJ];
#pragma unroll
                    for (int jj = 0; jj < JJ; ++jj) hv[jj] = sh(row_of(jj) * CH + chunk_of(jj));
                    const TI* svr = reinterpret_cast<const TI*>(st + geo.vrec);
                    const float* sbr = reinterpret_cast<const float*>(st + geo.brec);
                    for (int j = 0; j < m; ++j) {
                        const TI* kj = (j < c) ? sk + j * DK : skt;
                        float4 kb[CPL];
#pragma unroll
                        for (int q = 0; q < CPL; ++q) kb[q] = load4(kj + (cl + 8 * q) * 4);
                        float vr4[4];
#pragma unroll
                        for (int p = 0; p < 4; ++p) vr4[p] = to_f((j < c) ? svr[j * 64 + rloc + p] : sv[rloc + p]);
                        gdn_token_update<CPL>(hv, kb, vr4, (j < c) ? sa[j] : hdr.alpha, (j < c) ? sbr[j] : hdr.beta);
                    }
                    float oq[4];
#pragma unroll
                    for (int p = 0; p < 4; ++p) {
                        float acc = 0.f;
#pragma unroll
                        for (int q = 0; q < CPL; ++q) acc += dot4(hv[p * CPL + q], qv[q]);
                        oq[p] = acc;
                    }
                    rowgroup_allsum4(oq);
                    if (cl < 4) {
                        const float ov = (cl == 0) ? oq[0] : (cl == 1) ? oq[1] : (cl == 2) ? oq[2] : oq[3];
                        store_out(a.o, static_cast<size_t>(tile) * DV + half * 64 + rr, ov, out_f32 != 0);
                    }
                    const size_t hrow = static_cast<size_t>(tile) * DV + half * 64;
                    float4* dst = reinterpret_cast<float4*>(a.ckpt + hrow * DK);
#pragma unroll
                    for (int jj = 0; jj < JJ; ++jj) dst[row_of(jj) * CH + chunk_of(jj)] = hv[jj];
                    if (!a.defer_copy) {
                        uint8_t* codes = a.rc_codes + (RF == RSSM_READ_FP8 ? hrow * DK : hrow * DK / 2);
                        uint8_t* bsc = (RF == RSSM_READ_NVFP4) ? a.rc_bscale + hrow * (DK / 16) : nullptr;
                        write_read_copy<GdnHalfRC<DK>, RF>(hv, codes, bsc,
                                                           a.rc_tscale + static_cast<size_t>(tile) * HALVES + half,
                                                           g_red[g], gt, lane, gw, row_of, chunk_of, gsync);
                    }
                    if (half == HALVES - 1 && gt == 0) a.counts[tile] = only_flush ? a.kflush : 0;
                } else {
                    // fold the window into this half: S0 <- gamma S0 + sum_j rho_j u_j k_j^T
                    float4 hv[JJ];
#pragma unroll
                    for (int jj = 0; jj < JJ; ++jj) {
                        const float4 v = sh(row_of(jj) * CH + chunk_of(jj));
                        hv[jj] = make_float4(v.x * gamma, v.y * gamma, v.z * gamma, v.w * gamma);
                    }
                    const int rg0 = lane & ~7;   // first lane of this row group
                    for (int j = 0; j < m; ++j) {
                        const float rj = __shfl_sync(0xffffffffu, rho, j);
                        float u[4];
                        if (j < c) {
                            load_u4(su + j * 64 + rloc, u);
                        } else {
#pragma unroll
                            for (int p = 0; p < 4; ++p) u[p] = __shfl_sync(0xffffffffu, uc, rg0 + p);
                        }
                        const TI* kj = (j < c) ? sk + j * DK : skt;
#pragma unroll
                        for (int q = 0; q < CPL; ++q) {
                            const float4 kb = load4(kj + (cl + 8 * q) * 4);
#pragma unroll
                            for (int p = 0; p < 4; ++p) {
                                const float x = rj * u[p];
                                const float2 x2 = make_float2(x, x);
                                float4& h = hv[p * CPL + q];
                                const float2 h01 = __ffma2_rn(x2, lo2(kb), lo2(h));
                                const float2 h23 = __ffma2_rn(x2, hi2(kb), hi2(h));
                                h = make_float4(h01.x, h01.y, h23.x, h23.y);
                            }
                        }
                    }
                    const size_t hoff = (static_cast<size_t>(tile) * DV + half * 64) * DK;
                    if constexpr (k16) {
                        // FP16 checkpoint: rounded once, on the store
                        uint2* dst = reinterpret_cast<uint2*>(reinterpret_cast<__half*>(a.ckpt) + hoff);
#pragma unroll
                        for (int jj = 0; jj < JJ; ++jj) dst[row_of(jj) * CH + chunk_of(jj)] = f32_to_f16x4(hv[jj]);
                    } else {
                        float4* dst = reinterpret_cast<float4*>(a.ckpt + hoff);
#pragma unroll
                        for (int jj = 0; jj < JJ; ++jj) dst[row_of(jj) * CH + chunk_of(jj)] = hv[jj];
                    }
                    if (half == HALVES - 1 && gt == 0) a.counts[tile] = only_flush ? a.kflush : 0;
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty_bar[s]);
        }
    }
}

// ---------------------------------------------------------------------------
// Lean non-flush step, for launches in which no tile completes its window
// (every record count c satisfies c + 1 < k; a tile outside that range is
// reported as RSSM_DEV_COUNT_RANGE and left untouched).
//  * Stages hold only the 64-row state half and this token's q, k and half
//    of v (about 33 KiB), so more of them fit and more consumer groups run.
//  * Each consumer lane loads the records it needs for its group's next item
//    into registers while it finishes the current one: the k columns of 4
//    records once the state row-dots are formed, the u rows of up to 4
//    records and one alpha once the output is.
//  * The stage goes back to the producer as soon as the state row-dots are
//    formed; the weights, output and appends follow from registers.
// The arithmetic is the fused kernel's (same helpers, same order), so both
// kernels give bit-identical outputs and records.
// ---------------------------------------------------------------------------
struct NGeom {
    int state, bsc, qt, kt, vt, bytes;
};

// rf: the stage holds the FP32 half (RSSM_READ_NONE), the FP16 one (kGdnF16)
// or its read copy
__host__ __device__ inline NGeom nstage_geom(int DK, int in_sz, int rf) {
    NGeom g;
    int off = 0;
    g.state = off; off += galign128(rf == RSSM_READ_NONE ? 64 * DK * 4 : rf == kGdnF16 ? 64 * DK * 2
                                                         : rf == RSSM_READ_FP8 ? 64 * DK : 64 * DK / 2);
    g.bsc = off;   off += (rf == RSSM_READ_NVFP4) ? galign128(64 * DK / 16) : 0;
    g.qt = off;    off += galign128(DK * in_sz);
    g.kt = off;    off += galign128(DK * in_sz);
    g.vt = off;    off += galign128(64 * in_sz);
    g.bytes = off;
    return g;
}

template <class L, typename TI, int NG, int NQ, int RF>
__global__ void __launch_bounds__(32 + NG * L::kThreads, 1)
gdn_replay_nf_kernel(const GDNArgs a, const int out_f32, const int S, const int tiles_per_cta,
                     const int skip_flush) {
    constexpr int DV = L::DV, DK = L::DK, HALVES = L::HALVES, GT = L::kThreads, GW = L::kWarps;
    constexpr int CPL = L::CPL;
    constexpr int in_sz = static_cast<int>(sizeof(TI));
    using R = Raw4<TI>;
    extern __shared__ __align__(128) unsigned char dsm[];
    __shared__ __align__(8) uint64_t full_bar[kMaxStages];
    __shared__ __align__(8) uint64_t empty_bar[kMaxStages];
    __shared__ int s_cnt[kMaxTilesPerCta];
    __shared__ float s_al[kMaxTilesPerCta], s_be[kMaxTilesPerCta];
    __shared__ volatile int s_abort;

    const int total = a.B * a.H;
    const int t0 = blockIdx.x * tiles_per_cta;
    const int nt = max(0, min(tiles_per_cta, total - t0));
    const int ni = nt * HALVES;
    const NGeom geo = nstage_geom(DK, in_sz, RF);
    constexpr bool kCopy = (RF == RSSM_READ_FP8 || RF == RSSM_READ_NVFP4);   // a read copy
    constexpr bool k16 = (RF == kGdnF16);                                    // an FP16 checkpoint
    const int tid = threadIdx.x;

    if (tid < 32) {
        for (int i = tid; i < nt; i += 32) {
            int c = a.counts[t0 + i];
            if (skip_flush && c == a.kflush) {
                // flushed by the flush-only launch that ran first in this step
                a.counts[t0 + i] = 0;
                c = -2;
            } else if (c < 0 || c + 1 >= a.kflush) {
                report_error(a.err, RSSM_DEV_COUNT_RANGE, t0 + i, c);
                c = -1;
            }
            s_cnt[i] = c;
            s_al[i] = a.alpha[t0 + i];
            s_be[i] = a.beta[t0 + i];
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
        int s = 0;
        uint32_t round = 0;
        for (int w = 0; w < ni; ++w) {
            if (s_abort) break;
            if (!mbar_wait_bounded(&empty_bar[s], (round & 1u) ^ 1u)) {
                report_error(a.err, kDevTimeout, t0, 20);
                s_abort = 1;
                break;
            }
            const int tl = w / HALVES, half = w - tl * HALVES;
            const size_t bh = static_cast<size_t>(t0 + tl);
            unsigned char* st = dsm + static_cast<size_t>(s) * geo.bytes;
            const size_t row0 = bh * DV + half * 64;
            if (s_cnt[tl] == -2) {   // skipped: nothing to copy
                mbar_arrive_expect_tx(&full_bar[s], 0);
                issued |= 1u << s;
                last_par = (last_par & ~(1u << s)) | ((round & 1u) << s);
                if (++s == S) { s = 0; ++round; }
                continue;
            }
            const uint32_t state_bytes = (RF == RSSM_READ_NONE) ? 64 * DK * 4 : k16 ? 64 * DK * 2
                                         : (RF == RSSM_READ_FP8) ? 64 * DK : 64 * DK / 2;
            const uint32_t bsc_bytes = (RF == RSSM_READ_NVFP4) ? 64 * DK / 16 : 0;
            mbar_arrive_expect_tx(&full_bar[s], state_bytes + bsc_bytes + 2 * DK * in_sz + 64 * in_sz);
            if (RF == RSSM_READ_NONE)
                bulk_g2s_hint(st + geo.state, a.ckpt + row0 * DK, state_bytes, &full_bar[s], pol);
            else if (k16)
                bulk_g2s_hint(st + geo.state, reinterpret_cast<const __half*>(a.ckpt) + row0 * DK, state_bytes,
                              &full_bar[s], pol);
            else
                bulk_g2s_hint(st + geo.state, a.rc_codes + row0 * DK / (RF == RSSM_READ_FP8 ? 1 : 2), state_bytes,
                              &full_bar[s], pol);
            if (bsc_bytes) bulk_g2s(st + geo.bsc, a.rc_bscale + row0 * (DK / 16), bsc_bytes, &full_bar[s]);
            bulk_g2s(st + geo.qt, reinterpret_cast<const TI*>(a.q) + bh * DK, DK * in_sz, &full_bar[s]);
            bulk_g2s(st + geo.kt, reinterpret_cast<const TI*>(a.k) + bh * DK, DK * in_sz, &full_bar[s]);
            bulk_g2s(st + geo.vt, reinterpret_cast<const TI*>(a.v) + bh * DV + half * 64, 64 * in_sz,
                     &full_bar[s]);
            issued |= 1u << s;
            last_par = (last_par & ~(1u << s)) | ((round & 1u) << s);
            if (++s == S) { s = 0; ++round; }
        }
        for (int q = 0; q < S; ++q)
            if ((issued >> q) & 1u)
                if (!mbar_wait_bounded(&full_bar[q], (last_par >> q) & 1u))
                    report_error(a.err, kDevTimeout, t0, 21);
        return;
    }

    // --------------------------------------------------------------- consumers
    const int g = (tid - 32) / GT;
    const int gt = (tid - 32) - g * GT;
    const int lane = gt & 31, gw = gt >> 5;
    const int cl = lane & 7, rg = lane >> 3;
    const int rloc = gw * 16 + rg * 4;   // first of the lane's 4 rows in the half

    // records of the group's next item, loaded ahead
    typename R::T kp[4][CPL];   // k_j columns cl + 8q, j = rg + 4kk
    float4 up[4];               // u_j rows rloc..rloc+3, j = cl + 8kk
    float ap;                   // alpha_lane
    auto prefetch_k = [&](int w) {
        if (w >= ni) return;
        const int tl = w / HALVES;
        const int c = s_cnt[tl];
        const TI* kb = reinterpret_cast<const TI*>(a.buf_k) + static_cast<size_t>(t0 + tl) * a.cap * DK;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            const int j = rg + 4 * kk;
#pragma unroll
            for (int q = 0; q < CPL; ++q) kp[kk][q] = (j < c) ? R::ld(kb + j * DK + (cl + 8 * q) * 4) : R::zero();
        }
    };
    auto prefetch_u = [&](int w) {
        if (w >= ni) return;
        const int tl = w / HALVES, half = w - tl * HALVES;
        const size_t tile = static_cast<size_t>(t0 + tl);
        const int c = s_cnt[tl];
        const float* ub = a.buf_u + (tile * HALVES + half) * a.cap * 64;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            const int j = cl + 8 * kk;
            up[kk] = (j < c) ? __ldg(reinterpret_cast<const float4*>(ub + j * 64 + rloc)) : zero4();
        }
        ap = (lane < c) ? __ldg(a.buf_a + tile * a.cap + lane) : 1.f;
    };
    // With a read copy the items are bound by instructions: a group then takes
    // every NG-th tile and both of its halves, one after the other, and half 0
    // forms the window's key dots for both (S is a multiple of NG * HALVES, so
    // every stage keeps one owner group). On the FP32 half, which is bound by
    // DRAM, the group takes every NG-th half and forms its own key dots: that
    // order measured faster there.
    constexpr bool kShare = kCopy && (HALVES > 1);
    const int first = kShare ? g * HALVES : g;
    prefetch_k(first);
    prefetch_u(first);
    float kap = 0.f, lam = 0.f;   // lane j: k_j . k_c and k_j . (scale q)

    for (int it = 0;; ++it) {
        int w, tl, half, w_next;
        if (kShare) {
            tl = g + (it / HALVES) * NG;
            half = it % HALVES;
            w = tl * HALVES + half;
            w_next = (half + 1 < HALVES) ? w + 1 : (tl + NG) * HALVES;
            if (tl >= nt) break;
        } else {
            w = g + it * NG;
            tl = w / HALVES;
            half = w - tl * HALVES;
            w_next = w + NG;
            if (w >= ni) break;
        }
        const int tile = t0 + tl;
        const int s = w % S;
        const uint32_t par = static_cast<uint32_t>(w / S) & 1u;
        int ok = 0;
        if (lane == 0) ok = (!s_abort && mbar_wait_bounded(&full_bar[s], par)) ? 1 : 0;
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) {
            if (lane == 0 && !s_abort) {
                report_error(a.err, kDevTimeout, tile, 22);
                s_abort = 1;
            }
            return;
        }
        mbar_try_wait(&full_bar[s], par);

        const unsigned char* st = dsm + static_cast<size_t>(s) * geo.bytes;
        const int c = s_cnt[tl];
        const int m = c + 1;
        const TI* sq = reinterpret_cast<const TI*>(st + geo.qt);
        const TI* skt = reinterpret_cast<const TI*>(st + geo.kt);
        const TI* sv = reinterpret_cast<const TI*>(st + geo.vt);

        float4 kv[CPL], qv[CPL];
#pragma unroll
        for (int q = 0; q < CPL; ++q) {
            kv[q] = load4(skt + (cl + 8 * q) * 4);
            const float4 t = load4(sq + (cl + 8 * q) * 4);
            qv[q] = make_float4(t.x * a.scale, t.y * a.scale, t.z * a.scale, t.w * a.scale);
        }
        // key dots (lane j: k_j . k_c and k_j . (scale q)); NQ = 2 when windows
        // reach past 16 records, whose second quad is read here directly
        if (!kShare || half == 0) {
            if (NQ == 1) {
                gdn_key_dots<CPL>(kap, lam, kv, qv, min(m, 16), lane, [&](int, int kk, int q) {
                    const int j = rg + 4 * kk;
                    return (j < c) ? R::f(kp[kk][q]) : (j == c ? kv[q] : zero4());
                });
            } else {
                const TI* kb = reinterpret_cast<const TI*>(a.buf_k) + static_cast<size_t>(tile) * a.cap * DK;
                gdn_key_dots<CPL>(kap, lam, kv, qv, m, lane, [&](int qd, int kk, int q) {
                    const int j = 16 * qd + rg + 4 * kk;
                    if (qd == 0) return (j < c) ? R::f(kp[kk][q]) : (j == c ? kv[q] : zero4());
                    return (j < c) ? load4(kb + j * DK + (cl + 8 * q) * 4) : (j == c ? kv[q] : zero4());
                });
            }
            if (kShare) prefetch_k((tl + NG) * HALVES);   // the next tile's record keys
        }

        const int rr = rloc + (cl & 3);   // this lane's row (cl < 4)
        float pk[4], pq[4], vr = 0.f;
        TI vraw{};
        // the copy's tile scale multiplies the state dots (1 for the FP32 half)
        const float ts = !kCopy ? 1.f : __ldg(a.rc_tscale + static_cast<size_t>(tile) * HALVES + half);
        if (c >= 0) {
            if constexpr (!kCopy)
                gdn_state_dots<CPL, DK>(pk, pq, HalfRef<k16>{st + geo.state}, kv, qv, rloc, cl);
            else
                gdn_copy_dots<RF, CPL, DK>(pk, pq, st + geo.state, st + geo.bsc, kv, qv, rloc, cl);
            vraw = sv[rr];
            vr = to_f(vraw);
            // append this token's k and alpha at slot c (once per tile, from the stage)
            if (half == 0 && gw == 0) {
                uint4* bk = reinterpret_cast<uint4*>(reinterpret_cast<TI*>(a.buf_k) +
                                                     (static_cast<size_t>(tile) * a.cap + c) * DK);
                const uint4* ks = reinterpret_cast<const uint4*>(skt);
                for (int q = lane; q < DK * in_sz / 16; q += 32) bk[q] = ks[q];
                if (lane == 0) a.buf_a[static_cast<size_t>(tile) * a.cap + c] = s_al[tl];
                if (kCopy && lane == 0) a.buf_beta[static_cast<size_t>(tile) * a.cap + c] = s_be[tl];
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty_bar[s]);
        if (!kShare) prefetch_k(w_next);
        if (c < 0) {
            prefetch_u(w_next);
            continue;
        }

        const float al = (lane < c) ? ap : (lane == c ? s_al[tl] : 1.f);
        float gamma;
        const float rho = window_rho(al, lane, m, gamma);
        const float wk = (lane < c) ? rho * kap : 0.f;
        const float wq = (lane < c) ? rho * lam : 0.f;
        const float lam_c = __shfl_sync(0xffffffffu, lam, c & 31);
        float uk[4][4];
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            uk[kk][0] = up[kk].x; uk[kk][1] = up[kk].y; uk[kk][2] = up[kk].z; uk[kk][3] = up[kk].w;
        }
        float uc, o;
        gdn_finish(pk, pq, uk, gamma * ts, wk, wq, c, lane, cl, vr, s_be[tl], lam_c, &uc, &o);
        prefetch_u(w_next);
        if (cl < 4) {
            store_out(a.o, static_cast<size_t>(tile) * DV + half * 64 + rr, o, out_f32 != 0);
            const size_t slot = ((static_cast<size_t>(tile) * HALVES + half) * a.cap + c) * 64 + rr;
            a.buf_u[slot] = uc;
            if (kCopy) reinterpret_cast<TI*>(a.buf_v)[slot] = vraw;
        }
        if (half == HALVES - 1 && gt == 0) a.counts[tile] = m;
    }
}

// ---------------------------------------------------------------------------
// Direct non-flush kernel for small batches (FP32 or FP16 checkpoint): one
// block per tile, one group of 4 warps per 64-row half, no pipeline. With few
// tiles per SM the persistent kernel's ring has nothing to overlap. Every load
// that does not depend on the record count is issued with the count, so the
// launch waits on one round of loads instead of one per dependent step (count,
// records, keys, state half, token): the records of every slot a non-flush
// window can hold are loaded and masked once the count is known. That takes
// the registers of one block per SM; above one tile per SM the launch runs in
// waves, which still measured faster than a lighter kernel waiting on five
// rounds. The lean kernel's arithmetic (the shared helpers, in the same
// order), so outputs and records are the same bits. skip_flush: as in the
// lean kernel.
// ---------------------------------------------------------------------------
template <class L, typename TI, bool F16>
__global__ void __launch_bounds__(L::HALVES * L::kThreads, 1)
gdn_replay_nf_direct_kernel(const GDNArgs a, const int out_f32, const int skip_flush) {
    constexpr int DV = L::DV, DK = L::DK, HALVES = L::HALVES, GT = L::kThreads, CPL = L::CPL;
    constexpr int in_sz = static_cast<int>(sizeof(TI));
    using R = Raw4<TI>;
    const int tile = blockIdx.x;
    const int tid = threadIdx.x;
    const int half = tid / GT, gt = tid - half * GT;
    const int lane = gt & 31, gw = gt >> 5;
    const int cl = lane & 7, rg = lane >> 3;
    const int rloc = gw * 16 + rg * 4;
    const int rr = rloc + (cl & 3);
    const size_t bh = static_cast<size_t>(tile);
    const TI* kt = reinterpret_cast<const TI*>(a.k) + bh * DK;
    const TI* qt = reinterpret_cast<const TI*>(a.q) + bh * DK;
    const TI* kb = reinterpret_cast<const TI*>(a.buf_k) + bh * a.cap * DK;
    const float* ub = a.buf_u + (bh * HALVES + half) * a.cap * 64;

    const int c = a.counts[tile];
    const int kmax = a.kflush - 1;   // records a non-flush window holds before its token
    float4 kv[CPL], qv[CPL];
#pragma unroll
    for (int q = 0; q < CPL; ++q) {
        kv[q] = load4(kt + (cl + 8 * q) * 4);
        const float4 t = load4(qt + (cl + 8 * q) * 4);
        qv[q] = make_float4(t.x * a.scale, t.y * a.scale, t.z * a.scale, t.w * a.scale);
    }
    float4 up[4];
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
        const int j = cl + 8 * kk;
        up[kk] = (j < kmax) ? __ldg(reinterpret_cast<const float4*>(ub + j * 64 + rloc)) : zero4();
    }
    float ap = (lane < kmax) ? __ldg(a.buf_a + bh * a.cap + lane) : 1.f;
    typename R::T kr[4][CPL];   // the first 16 records' k columns of this lane
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
        const int j = rg + 4 * kk;
#pragma unroll
        for (int q = 0; q < CPL; ++q) kr[kk][q] = (j < kmax) ? R::ld(kb + j * DK + (cl + 8 * q) * 4) : R::zero();
    }
    float pk[4], pq[4];
    const size_t hoff = (bh * DV + half * 64) * DK;
    gdn_state_dots<CPL, DK>(pk, pq,
                            HalfRef<F16>{F16 ? static_cast<const void*>(reinterpret_cast<const __half*>(a.ckpt) + hoff)
                                             : static_cast<const void*>(a.ckpt + hoff)},
                            kv, qv, rloc, cl);
    const TI vraw = reinterpret_cast<const TI*>(a.v)[bh * DV + half * 64 + rr];
    const float al_t = a.alpha[bh], be_t = a.beta[bh];

    if (skip_flush && c == a.kflush) {   // flushed by the flush-only launch of this step
        __syncthreads();
        if (tid == 0) a.counts[tile] = 0;
        return;
    }
    if (c < 0 || c + 1 >= a.kflush) {
        if (tid == 0) report_error(a.err, RSSM_DEV_COUNT_RANGE, tile, c);
        return;
    }
    const int m = c + 1;
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
        if (cl + 8 * kk >= c) up[kk] = zero4();
    if (lane >= c) ap = 1.f;
    const float vr = to_f(vraw);
    float kap = 0.f, lam = 0.f;   // lane j: k_j . k_c and k_j . (scale q)
    gdn_key_dots<CPL>(kap, lam, kv, qv, m, lane, [&](int qd, int kk, int q) {
        const int j = 16 * qd + rg + 4 * kk;
        if (qd == 0) return (j < c) ? R::f(kr[kk][q]) : (j == c ? kv[q] : zero4());
        return (j < c) ? R::f(R::ld(kb + j * DK + (cl + 8 * q) * 4)) : (j == c ? kv[q] : zero4());
    });
    // append this token's k and alpha at slot c (once per tile)
    if (half == 0 && gw == 0) {
        uint4* bk = reinterpret_cast<uint4*>(reinterpret_cast<TI*>(a.buf_k) + (bh * a.cap + c) * DK);
        const uint4* ks = reinterpret_cast<const uint4*>(kt);
        for (int q = lane; q < DK * in_sz / 16; q += 32) bk[q] = ks[q];
        if (lane == 0) a.buf_a[bh * a.cap + c] = al_t;
    }
    const float al = (lane < c) ? ap : (lane == c ? al_t : 1.f);
    float gamma;
    const float rho = window_rho(al, lane, m, gamma);
    const float wk = (lane < c) ? rho * kap : 0.f;
    const float wq = (lane < c) ? rho * lam : 0.f;
    const float lam_c = __shfl_sync(0xffffffffu, lam, c & 31);
    float uk[4][4];
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
        uk[kk][0] = up[kk].x; uk[kk][1] = up[kk].y; uk[kk][2] = up[kk].z; uk[kk][3] = up[kk].w;
    }
    float uc, o;
    gdn_finish(pk, pq, uk, gamma, wk, wq, c, lane, cl, vr, be_t, lam_c, &uc, &o);
    if (cl < 4) {
        store_out(a.o, bh * DV + half * 64 + rr, o, out_f32 != 0);
        a.buf_u[((bh * HALVES + half) * a.cap + c) * 64 + rr] = uc;
    }
    // every thread has read the count before it moves
    __syncthreads();
    if (tid == 0) a.counts[tile] = m;
}

// Direct flush kernel for small batches (FP32 or FP16 checkpoint, no read
// copy): one block per tile, one group of 4 warps per 64-row half, no
// pipeline. Every load is issued with the count: the half, this token's
// inputs, and the window's records (k, the half's u rows, alpha), which the
// block then keeps in shared memory. Then the fused kernel's flush
// arithmetic, in the same order: the output of the token that completes the
// window, and the fold S <- gamma S + sum_j rho_j u_j k_j^T, written once.
// In a step that runs only this kernel, a tile whose count is below k - 1
// (its pointer was moved back) takes the non-flush step instead, as in the
// fused kernel: the same output, then this token's record appended. In the
// flush part of a split step (only_flush) such a tile is left to the lean
// launch, and the flushed tile is marked with count k for it.
template <class L, typename TI, bool F16>
__global__ void __launch_bounds__(L::HALVES * L::kThreads, 1)
gdn_replay_flush_direct_kernel(const GDNArgs a, const int out_f32, const int only_flush) {
    constexpr int DV = L::DV, DK = L::DK, HALVES = L::HALVES, GT = L::kThreads, CPL = L::CPL;
    constexpr int CH = DK / 4, JJ = L::J, NTHR = HALVES * GT;
    constexpr int in_sz = static_cast<int>(sizeof(TI));
    constexpr int KCH = DK * in_sz / 16;                        // 16-byte chunks of a k record
    constexpr int KPT = (kMaxCap * KCH + NTHR - 1) / NTHR;      // of them per thread, at most
    constexpr int UPT = (kMaxCap * 16 + GT - 1) / GT;           // u float4 per thread of a group, at most
    __shared__ __align__(16) unsigned char s_kb[kMaxCap * DK * in_sz];   // k records, slot c: this token's k
    __shared__ __align__(16) float s_u[HALVES * kMaxCap * 64];           // [half][record][row]
    __shared__ float s_a[kMaxCap];
    const int tile = blockIdx.x;
    const int tid = threadIdx.x;
    const int half = tid / GT, gt = tid - half * GT;
    const int lane = gt & 31, gw = gt >> 5;
    const int cl = lane & 7;
    const int rloc = gw * 16 + (lane >> 3) * 4;   // first of the lane's 4 rows in the half
    const int rr = rloc + (cl & 3);
    auto row_of = [&](int j) { return rloc + j / CPL; };
    auto chunk_of = [&](int j) { return cl + 8 * (j % CPL); };
    const size_t bh = static_cast<size_t>(tile);
    const TI* kt = reinterpret_cast<const TI*>(a.k) + bh * DK;
    const TI* qt = reinterpret_cast<const TI*>(a.q) + bh * DK;
    const uint4* kbuf = reinterpret_cast<const uint4*>(reinterpret_cast<const TI*>(a.buf_k) + bh * a.cap * DK);
    const float4* ubuf = reinterpret_cast<const float4*>(a.buf_u + (bh * HALVES + half) * a.cap * 64);

    const int c = a.counts[tile];
    const int cm = a.kflush - 1;   // the count of a tile that flushes
    uint4 kreg[KPT];
#pragma unroll
    for (int i = 0; i < KPT; ++i) {
        const int q = tid + i * NTHR, j = q / KCH;
        kreg[i] = (j < cm) ? kbuf[q] : (j == cm) ? reinterpret_cast<const uint4*>(kt)[q - j * KCH]
                                                 : make_uint4(0u, 0u, 0u, 0u);
    }
    float4 ureg[UPT];
#pragma unroll
    for (int i = 0; i < UPT; ++i) {
        const int q = gt + i * GT;
        ureg[i] = (q < cm * 16) ? ubuf[q] : zero4();
    }
    const float arec = (tid < cm) ? a.buf_a[bh * a.cap + tid] : 1.f;
    float4 kv[CPL], qv[CPL];
#pragma unroll
    for (int q = 0; q < CPL; ++q) {
        kv[q] = load4(kt + (cl + 8 * q) * 4);
        const float4 t = load4(qt + (cl + 8 * q) * 4);
        qv[q] = make_float4(t.x * a.scale, t.y * a.scale, t.z * a.scale, t.w * a.scale);
    }
    const size_t hoff = (bh * DV + half * 64) * DK;
    const HalfRef<F16> sh{F16 ? static_cast<const void*>(reinterpret_cast<const __half*>(a.ckpt) + hoff)
                              : static_cast<const void*>(a.ckpt + hoff)};
    float4 hv[JJ];
#pragma unroll
    for (int jj = 0; jj < JJ; ++jj) hv[jj] = sh(row_of(jj) * CH + chunk_of(jj));
    const TI vraw = reinterpret_cast<const TI*>(a.v)[bh * DV + half * 64 + rr];
    const float al_t = a.alpha[bh], be_t = a.beta[bh];

    if (c < 0 || c > cm) {
        if (!only_flush && tid == 0) report_error(a.err, RSSM_DEV_COUNT_RANGE, tile, c);
        return;
    }
    if (only_flush && c != cm) return;
    const bool flush = (c == cm);
    const int m = c + 1;
#pragma unroll
    for (int i = 0; i < KPT; ++i) {
        const int q = tid + i * NTHR;
        if (q < m * KCH) reinterpret_cast<uint4*>(s_kb)[q] = kreg[i];
    }
    float* su = s_u + half * kMaxCap * 64;
#pragma unroll
    for (int i = 0; i < UPT; ++i) {
        const int q = gt + i * GT;
        if (q < c * 16) reinterpret_cast<float4*>(su)[q] = ureg[i];
    }
    if (tid < c) s_a[tid] = arec;
    __syncthreads();   // also: every thread has read the count

    const TI* sk = reinterpret_cast<const TI*>(s_kb);
    float kap = 0.f, lam = 0.f;   // lane j: k_j . k_c and k_j . (scale q)
    gdn_key_dots<CPL>(kap, lam, kv, qv, m, lane, [&](int qd, int kk, int q) {
        const int j = 16 * qd + (lane >> 3) + 4 * kk;
        return (j < c) ? load4(sk + j * DK + (cl + 8 * q) * 4) : (j == c ? kv[q] : zero4());
    });
    const float al = (lane < c) ? s_a[lane] : (lane == c ? al_t : 1.f);
    float gamma;
    const float rho = window_rho(al, lane, m, gamma);
    const float wk = (lane < c) ? rho * kap : 0.f;
    const float wq = (lane < c) ? rho * lam : 0.f;
    const float lam_c = __shfl_sync(0xffffffffu, lam, c & 31);
    float pk[4], pq[4];
    gdn_state_dots<CPL, DK>(pk, pq, sh, kv, qv, rloc, cl);
    float uk[4][4];
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
        const int j = cl + 8 * kk;
        if (j < c) load_u4(su + j * 64 + rloc, uk[kk]);
    }
    float uc, o;
    gdn_finish(pk, pq, uk, gamma, wk, wq, c, lane, cl, to_f(vraw), be_t, lam_c, &uc, &o);
    if (cl < 4) store_out(a.o, bh * DV + half * 64 + rr, o, out_f32 != 0);
    if (!flush) {
        // append this token's record at slot c: u rows of this half; k, alpha once
        if (cl < 4) a.buf_u[((bh * HALVES + half) * a.cap + c) * 64 + rr] = uc;
        if (half == 0 && gw == 0) {
            uint4* bk = reinterpret_cast<uint4*>(reinterpret_cast<TI*>(a.buf_k) + (bh * a.cap + c) * DK);
            for (int q = lane; q < KCH; q += 32) bk[q] = reinterpret_cast<const uint4*>(kt)[q];
            if (lane == 0) a.buf_a[bh * a.cap + c] = al_t;
        }
        if (tid == 0) a.counts[tile] = m;
        return;
    }

    // fold the window into this half: S0 <- gamma S0 + sum_j rho_j u_j k_j^T
#pragma unroll
    for (int jj = 0; jj < JJ; ++jj) hv[jj] = make_float4(hv[jj].x * gamma, hv[jj].y * gamma, hv[jj].z * gamma, hv[jj].w * gamma);
    const int rg0 = lane & ~7;   // first lane of this row group
    for (int j = 0; j < m; ++j) {
        const float rj = __shfl_sync(0xffffffffu, rho, j);
        float u[4];
        if (j < c) {
            load_u4(su + j * 64 + rloc, u);
        } else {
#pragma unroll
            for (int p = 0; p < 4; ++p) u[p] = __shfl_sync(0xffffffffu, uc, rg0 + p);
        }
        const TI* kj = sk + j * DK;
#pragma unroll
        for (int q = 0; q < CPL; ++q) {
            const float4 kb = load4(kj + (cl + 8 * q) * 4);
#pragma unroll
            for (int p = 0; p < 4; ++p) {
                const float x = rj * u[p];
                const float2 x2 = make_float2(x, x);
                float4& h = hv[p * CPL + q];
                const float2 h01 = __ffma2_rn(x2, lo2(kb), lo2(h));
                const float2 h23 = __ffma2_rn(x2, hi2(kb), hi2(h));
                h = make_float4(h01.x, h01.y, h23.x, h23.y);
            }
        }
    }
    if constexpr (F16) {
        uint2* dst = reinterpret_cast<uint2*>(reinterpret_cast<__half*>(a.ckpt) + hoff);
#pragma unroll
        for (int jj = 0; jj < JJ; ++jj) dst[row_of(jj) * CH + chunk_of(jj)] = f32_to_f16x4(hv[jj]);
    } else {
        float4* dst = reinterpret_cast<float4*>(a.ckpt + hoff);
#pragma unroll
        for (int jj = 0; jj < JJ; ++jj) dst[row_of(jj) * CH + chunk_of(jj)] = hv[jj];
    }
    if (tid == 0) a.counts[tile] = only_flush ? a.kflush : 0;
}

// Tiles up to which a step of an FP32 or FP16 half runs the direct kernels.
constexpr int kDirectTilesPerSm = 4;

// split (two launches of one step): the step kernel takes only the tiles that
// complete their window and marks them with count k; the lean kernel, launched
// next, resets the marks and takes the other tiles.
template <class L, typename TI, int NG, bool LEAN, int RF>
cudaError_t launch_ng(const GDNArgs& a, int out_f32, int S, int grid, int per, size_t smem, int split,
                      cudaStream_t s) {
    // a non-flush window holds at most k - 1 records
    const bool nq1 = a.kflush - 1 <= 16;
    auto kernel = !LEAN ? gdn_replay_step_tma_kernel<L, TI, NG, RF>
                        : nq1 ? gdn_replay_nf_kernel<L, TI, NG, 1, RF> : gdn_replay_nf_kernel<L, TI, NG, 2, RF>;
    static LaunchCache lc[2];   // one per kernel this launcher may choose
    cudaError_t e = cached_dyn_smem(lc[(!LEAN || nq1) ? 0 : 1], kernel, smem);
    if (e != cudaSuccess) return e;
    kernel<<<grid, 32 + NG * L::kThreads, smem, s>>>(a, out_f32, S, per, split);
    return cudaGetLastError();
}

template <class L, typename TI, bool LEAN, int RF>
cudaError_t launch(const GDNArgs& a, int out_f32, int split, cudaStream_t s) {
    const int total = a.B * a.H;
    if (total == 0) return cudaSuccess;
    int num_sms = 0, smem_optin = 0;
    cudaError_t e = device_limits(&num_sms, &smem_optin);
    if (e != cudaSuccess) return e;
    if constexpr (LEAN && (RF == RSSM_READ_NONE || RF == kGdnF16)) {
        if (total <= kDirectTilesPerSm * num_sms) {
            gdn_replay_nf_direct_kernel<L, TI, RF == kGdnF16><<<total, L::HALVES * L::kThreads, 0, s>>>(a, out_f32, split);
            return cudaGetLastError();
        }
    }
    if constexpr (!LEAN && (RF == RSSM_READ_NONE || RF == kGdnF16)) {
        // a step whose every tile flushes, or the flush part of a split step
        if (total <= kDirectTilesPerSm * num_sms) {
            gdn_replay_flush_direct_kernel<L, TI, RF == kGdnF16><<<total, L::HALVES * L::kThreads, 0, s>>>(a, out_f32, split);
            return cudaGetLastError();
        }
    }
    static LaunchCache lc;
    int static_smem = 0;
    e = cached_static_smem(lc, LEAN ? gdn_replay_nf_kernel<L, TI, 3, 2, RF> : gdn_replay_step_tma_kernel<L, TI, 2, RF>, &static_smem);
    if (e != cudaSuccess) return e;
    const int in_sz = static_cast<int>(sizeof(TI));
    const int stage = LEAN ? nstage_geom(L::DK, in_sz, RF).bytes : gstage_geom(L::DK, a.cap, in_sz, RF).bytes;
    const int avail = smem_optin - static_smem - 1024;
    int smax = avail / stage;
    if (smax > kMaxStages) smax = kMaxStages;
    // every stage must have one owner group: S is a multiple of NG. Three
    // lean groups fit 128 registers a thread except with FP32 inputs and
    // d_k = 128 (four columns of 4 records prefetched as float4).
    const bool three = LEAN && smax >= 6 && !(sizeof(TI) == 4 && L::DK == 128);
    const int ng = three ? 3 : (smax >= 4) ? 2 : 1;
    // one owner group per stage: with a read copy the lean kernel gives a group
    // both halves of a tile in a row, so its ring is a multiple of ng * HALVES
    const int unit = (LEAN && (RF == RSSM_READ_FP8 || RF == RSSM_READ_NVFP4)) ? ng * L::HALVES : ng;
    const int S = (smax / unit) * unit;
    if (S < 2) return cudaErrorInvalidConfiguration;
    int grid = num_sms;
    if ((total + grid - 1) / grid > kMaxTilesPerCta) grid = (total + kMaxTilesPerCta - 1) / kMaxTilesPerCta;
    if (grid > total) grid = total;
    const int per = (total + grid - 1) / grid;
    grid = (total + per - 1) / per;
    const size_t smem = static_cast<size_t>(S) * stage;
    if (ng == 3) return launch_ng<L, TI, 3, LEAN, RF>(a, out_f32, S, grid, per, smem, split, s);
    if (ng == 2) return launch_ng<L, TI, 2, LEAN, RF>(a, out_f32, S, grid, per, smem, split, s);
    return launch_ng<L, TI, 1, LEAN, RF>(a, out_f32, S, grid, per, smem, split, s);
}

template <class L>
cudaError_t run(const GDNArgs& a, int in_dt, int out_dt, int path, cudaStream_t s) {
    const int of = (out_dt == RSSM_F32);
    const bool lean = (path == kStepNonFlush || path == kStepSkipFlush);
    const int sp = (path == kStepSkipFlush || path == kStepFlushOnly);
    using BF = __nv_bfloat16;
    if (a.ck == kCkF16) {   // FP16 checkpoint: bf16 inputs, no read copy
        if (in_dt != RSSM_BF16 || a.rf != RSSM_READ_NONE) return cudaErrorInvalidValue;
        return lean ? launch<L, BF, true, kGdnF16>(a, of, sp, s) : launch<L, BF, false, kGdnF16>(a, of, sp, s);
    }
    if (a.rf != RSSM_READ_NONE) {   // read copies: bf16 inputs
        if (in_dt != RSSM_BF16) return cudaErrorInvalidValue;
        if (a.rf == RSSM_READ_FP8)
            return lean ? launch<L, BF, true, RSSM_READ_FP8>(a, of, sp, s) : launch<L, BF, false, RSSM_READ_FP8>(a, of, sp, s);
        return lean ? launch<L, BF, true, RSSM_READ_NVFP4>(a, of, sp, s)
                    : launch<L, BF, false, RSSM_READ_NVFP4>(a, of, sp, s);
    }
    if (in_dt == RSSM_F32)
        return lean ? launch<L, float, true, RSSM_READ_NONE>(a, of, sp, s)
                    : launch<L, float, false, RSSM_READ_NONE>(a, of, sp, s);
    return lean ? launch<L, BF, true, RSSM_READ_NONE>(a, of, sp, s) : launch<L, BF, false, RSSM_READ_NONE>(a, of, sp, s);
}

}  // namespace

cudaError_t gdn_replay_step(const GDNArgs& a, int DV, int DK, int in_dt, int out_dt, int path, cudaStream_t s,
                            bool* supported) {
    *supported = true;
    if (DV == 128 && DK == 128) return run<GdnTile<128, 128>>(a, in_dt, out_dt, path, s);
    if (DV == 64 && DK == 64) return run<GdnTile<64, 64>>(a, in_dt, out_dt, path, s);
    if (DV == 64 && DK == 128) return run<GdnTile<64, 128>>(a, in_dt, out_dt, path, s);
    if (DV == 128 && DK == 64) return run<GdnTile<128, 64>>(a, in_dt, out_dt, path, s);
    *supported = false;
    return cudaSuccess;
}

}  // namespace rssm


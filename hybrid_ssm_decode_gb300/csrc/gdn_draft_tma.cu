// Gated DeltaNet ReplaySSM speculative draft step (T > 1 tokens per sequence),
// persistent and pipelined for GB300.
//
// Method: "NVIDIA ve Dao AI Lab, ... ReplaySSM'i sundu", section "Durum
// trafigini azaltma ve rollback'in basitlestirilmesi": drafts are appended
// to the buffer unverified and a rejected suffix is dropped by moving the
// buffer pointer; "ReplaySSM beschleunigt ...", section "Wichtige Details"
// (Gated DeltaNet, the WY/UT window form).
//
// Draft tau of a (sequence, head) with c committed records is token c + tau of
// the window. Its record row u and output follow the one-token step with the
// window's records 0 .. c + tau - 1, which now include the earlier drafts:
//   u_{c+tau} = beta (v - gamma S0 k - sum_{j<c+tau} rho_j (k_j . k) u_j)
//   o_{c+tau} = gamma S0 (scale q) + sum_{j<c+tau} rho_j (k_j . scale q) u_j
//               + (k . scale q) u_{c+tau}
// The drafts' records (k, u, alpha) are appended at slots c .. c+T-1; no
// state is written and the count is left for the verify step to move.
//
// Structure: the one-token fused kernel's pipeline. A work item is one 64-row
// half of a tile; a stage holds the half of S0, the tile's buffered k, u and
// alpha records, and the drafts' q, k and half of v. A group takes both halves
// of a tile in a row.
//  * Phase A, from the stage: every draft's key dots with the window (half 0
//    only, kept per thread for half 1; on the tensor cores for bf16 inputs),
//    every draft's state row-dots from one pass over the half, the records'
//    u rows and the drafts' v values; then the stage is released.
//  * Phase B, from registers: each draft's reduction over the committed
//    records (independent across drafts), then, per row in the lane that
//    holds it, the drafts in order: the earlier drafts' u rows enter as a
//    T x T triangular solve.
// With FP32 inputs draft 0 is exactly the one-token step's arithmetic; with
// bf16 inputs it differs only in the order of the key dots' sums.
// With a read copy (RF = FP8 or NVFP4; "... ReplaySSM'i sundu", section
// "Kuantizasyon hatasinin sinirlandirilmasi") the stage holds the half's copy
// and the state row-dots decode it (the copy's half scale joins gamma), and
// the drafts' records also keep v and beta, from which a flush replays the
// window through the recurrence from the FP32 checkpoint.
#include "gdn_pipeline.cuh"

namespace rssm {
namespace {

struct DGeom {
    int state, bsc, krec, urec, arec, qd, kd, vd, bytes;
};

// rf: the stage holds the FP32 half (RSSM_READ_NONE) or its read copy
__host__ __device__ inline DGeom draft_geom(int DK, int cap, int T, int in_sz, int rf) {
    DGeom g;
    int off = 0;
    g.state = off; off += galign128(rf == RSSM_READ_NONE ? 64 * DK * 4 : rf == RSSM_READ_FP8 ? 64 * DK : 64 * DK / 2);
    g.bsc = off;   off += (rf == RSSM_READ_NVFP4) ? galign128(64 * DK / 16) : 0;
    g.krec = off;  off += galign128(cap * DK * in_sz);
    g.urec = off;  off += galign128(cap * 64 * 4);
    g.arec = off;  off += galign128(cap * 4);
    g.qd = off;    off += galign128(T * DK * in_sz);
    g.kd = off;    off += galign128(T * DK * in_sz);
    g.vd = off;    off += galign128(T * 64 * in_sz);
    g.bytes = off;
    return g;
}

// Every draft's key dots in one pass over the window (the records, then the
// drafts' own keys at positions c, c+1, ...): for draft t, lane j ends with
// kap[t] = k_j . k_t and lam[t] = k_j . (scale q_t) for j <= c + t (zero past
// it). Each record chunk is read once for all drafts, and the drafts' sums
// are independent. Per draft the chunks and the accumulation order are
// gdn_key_dots's, so draft 0's dots are the one-token step's bits.
template <int CPL, int DK, int TMAX, typename TI>
__device__ __forceinline__ void draft_key_dots(float (&kap)[TMAX], float (&lam)[TMAX], const TI* sk, const TI* skd,
                                               const TI* sqd, float scale, int c, int T, int lane) {
    constexpr int DB = 2;   // drafts per pass: a pass keeps 2 drafts' sums and key columns live
    const int rg = lane >> 3, cl = lane & 7;
#pragma unroll
    for (int t = 0; t < TMAX; ++t) kap[t] = lam[t] = 0.f;
    const int mmax = c + T;
    const int src = (lane & 3) * 8 + 2 * ((lane >> 2) & 3);
    for (int qd = 0; 16 * qd < mmax; ++qd) {
#pragma unroll
        for (int t0 = 0; t0 < TMAX; t0 += DB) {
            float dk[DB][4], dq[DB][4];
#pragma unroll
            for (int t = 0; t < DB; ++t)
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) dk[t][kk] = dq[t][kk] = 0.f;
#pragma unroll
            for (int q = 0; q < CPL; ++q) {
                float4 kv[DB], qv[DB];
#pragma unroll
                for (int t = 0; t < DB; ++t) {
                    const int tq = min(t0 + t, T - 1);
                    kv[t] = load4(skd + tq * DK + (cl + 8 * q) * 4);
                    const float4 u = load4(sqd + tq * DK + (cl + 8 * q) * 4);
                    qv[t] = make_float4(u.x * scale, u.y * scale, u.z * scale, u.w * scale);
                }
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const int j = 16 * qd + rg + 4 * kk;
                    float4 kb = zero4();
                    if (j < c) kb = load4(sk + j * DK + (cl + 8 * q) * 4);
                    else if (j < mmax) kb = load4(skd + (j - c) * DK + (cl + 8 * q) * 4);
#pragma unroll
                    for (int t = 0; t < DB; ++t) {
                        const float4 kt = (j <= c + t0 + t) ? kb : zero4();
                        dk[t][kk] += dot4(kt, kv[t]);
                        dq[t][kk] += dot4(kt, qv[t]);
                    }
                }
            }
#pragma unroll
            for (int t = 0; t < DB; ++t) {
                if (t0 + t >= TMAX) break;
                float v[8];
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    v[2 * kk] = dk[t][kk];
                    v[2 * kk + 1] = dq[t][kk];
                }
                const float red = group_reduce_multi<8, 8>(v, lane);
                const float k1 = __shfl_sync(0xffffffffu, red, src);
                const float l1 = __shfl_sync(0xffffffffu, red, src + 1);
                if ((lane >> 4) == qd) {
                    kap[t0 + t] = k1;
                    lam[t0 + t] = l1;
                }
            }
        }
    }
}

__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// draft_key_dots for bf16 inputs on the tensor cores: the window's keys (rows:
// records 0..c-1, then the drafts' keys) times the matrix whose columns are
// k_0..k_3 and q_0..q_3 (T <= 4), as m16n8k16 MMAs (bf16 products are exact,
// the sums FP32). A warp's 32 x 8 result goes through its 1 KiB scratch so
// that lane j ends with record j's row; lam is scaled after the product.
template <int DK, int TMAX>
__device__ __forceinline__ void draft_key_dots_mma(float (&kap)[TMAX], float (&lam)[TMAX], const __nv_bfloat16* sk,
                                                   const __nv_bfloat16* skd, const __nv_bfloat16* sqd, float scale,
                                                   int c, int T, int lane, float* scratch) {
    static_assert(TMAX <= 4, "columns: 4 keys, 4 queries");
    constexpr int KS = DK / 16;
    const int g = lane >> 2, t = lane & 3;
    const int mmax = c + T;
    // B: column n = g (key n, or query n - 4), rows 16 ks + 2t .. +1 and +8 .. +9
    const __nv_bfloat16* vec = (g < 4) ? ((g < T) ? skd + g * DK : nullptr) : ((g - 4 < T) ? sqd + (g - 4) * DK : nullptr);
    uint32_t bf[KS][2];
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
        bf[ks][0] = vec ? *reinterpret_cast<const uint32_t*>(vec + 16 * ks + 2 * t) : 0u;
        bf[ks][1] = vec ? *reinterpret_cast<const uint32_t*>(vec + 16 * ks + 2 * t + 8) : 0u;
    }
    auto rec = [&](int r) -> const __nv_bfloat16* {
        return (r < c) ? sk + r * DK : (r < mmax) ? skd + (r - c) * DK : nullptr;
    };
    for (int mt = 0; 16 * mt < mmax; ++mt) {
        const int r0 = 16 * mt + g, r1 = r0 + 8;
        const __nv_bfloat16* p0 = rec(r0);
        const __nv_bfloat16* p1 = rec(r1);
        float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
            const uint32_t a0 = p0 ? *reinterpret_cast<const uint32_t*>(p0 + 16 * ks + 2 * t) : 0u;
            const uint32_t a1 = p1 ? *reinterpret_cast<const uint32_t*>(p1 + 16 * ks + 2 * t) : 0u;
            const uint32_t a2 = p0 ? *reinterpret_cast<const uint32_t*>(p0 + 16 * ks + 2 * t + 8) : 0u;
            const uint32_t a3 = p1 ? *reinterpret_cast<const uint32_t*>(p1 + 16 * ks + 2 * t + 8) : 0u;
            mma_bf16_16816(d, a0, a1, a2, a3, bf[ks][0], bf[ks][1]);
        }
        *reinterpret_cast<float2*>(scratch + r0 * 8 + 2 * t) = make_float2(d[0], d[1]);
        *reinterpret_cast<float2*>(scratch + r1 * 8 + 2 * t) = make_float2(d[2], d[3]);
    }
    __syncwarp();
    float v[8];
    if (lane < mmax) {
        const float4 lo = *reinterpret_cast<const float4*>(scratch + lane * 8);
        const float4 hi = *reinterpret_cast<const float4*>(scratch + lane * 8 + 4);
        v[0] = lo.x; v[1] = lo.y; v[2] = lo.z; v[3] = lo.w;
        v[4] = hi.x; v[5] = hi.y; v[6] = hi.z; v[7] = hi.w;
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = 0.f;
    }
    __syncwarp();   // the scratch is rewritten by the next call
#pragma unroll
    for (int tau = 0; tau < TMAX; ++tau) {
        const bool in = lane <= c + tau;
        kap[tau] = in ? v[tau] : 0.f;
        lam[tau] = in ? scale * v[4 + tau] : 0.f;
    }
}

// TMAX: the draft count the kernel is built for (T = TMAX), or kMaxDraft for
// any T up to it.
template <class L, typename TI, int NG, int TMAX, int RF>
__global__ void __launch_bounds__(32 + NG * L::kThreads, 1)
gdn_replay_draft_kernel(const GDNArgs a, const int out_f32, const int S, const int tiles_per_cta) {
    constexpr int DV = L::DV, DK = L::DK, HALVES = L::HALVES, GT = L::kThreads, GW = L::kWarps;
    constexpr int CPL = L::CPL;
    constexpr int in_sz = static_cast<int>(sizeof(TI));
    extern __shared__ __align__(128) unsigned char dsm[];
    __shared__ __align__(8) uint64_t full_bar[kMaxStages];
    __shared__ __align__(8) uint64_t empty_bar[kMaxStages];
    __shared__ int s_cnt[kMaxTilesPerCta];
    // each lane's key dots of half 0, kept for half 1 (written and read by
    // the same thread); with bf16 inputs the tensor-core key dots' scratch
    constexpr bool kMmaKeys = sizeof(TI) == 2 && TMAX <= 4;
    __shared__ float s_kst[NG][4][TMAX][2][32];
    __shared__ __align__(16) float s_kscr[kMmaKeys ? NG * 4 : 1][32 * 8];
    __shared__ volatile int s_abort;

    const int T = (TMAX < kMaxDraft) ? TMAX : a.T;
    const int total = a.B * a.H;
    const int t0 = blockIdx.x * tiles_per_cta;
    const int nt = max(0, min(tiles_per_cta, total - t0));
    const int ni = nt * HALVES;
    const DGeom geo = draft_geom(DK, a.cap, T, in_sz, RF);
    constexpr bool kCopy = (RF != RSSM_READ_NONE);   // the drafts read the copy
    const int tid = threadIdx.x;

    if (tid < 32) {
        for (int i = tid; i < nt; i += 32) {
            int c = a.counts[t0 + i];
            if (c < 0 || c >= a.kflush || c + T > a.cap) {
                report_error(a.err, RSSM_DEV_COUNT_RANGE, t0 + i, c);
                c = -1;
            }
            s_cnt[i] = c;
        }
        if (tid == 0) {
            for (int q = 0; q < S; ++q) {
                mbar_init(&full_bar[q], 1);
                mbar_init(&empty_bar[q], GW);
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
                report_error(a.err, kDevTimeout, t0, 50);
                s_abort = 1;
                break;
            }
            const int tl = w / HALVES, half = w - tl * HALVES;
            const int tile = t0 + tl;
            const int b = tile / a.H, hh = tile - b * a.H;
            const int nrec = max(s_cnt[tl], 0);
            unsigned char* st = dsm + static_cast<size_t>(s) * geo.bytes;
            const uint32_t state_bytes = (RF == RSSM_READ_NONE) ? 64 * DK * 4 : (RF == RSSM_READ_FP8) ? 64 * DK : 64 * DK / 2;
            const uint32_t bsc_bytes = (RF == RSSM_READ_NVFP4) ? 64 * DK / 16 : 0;
            const uint32_t krec_bytes = nrec * DK * in_sz, urec_bytes = nrec * 64 * 4;
            const uint32_t arec_bytes = a.cap * 4;
            const uint32_t draft_bytes = T * (2 * DK * in_sz + 64 * in_sz);
            mbar_arrive_expect_tx(&full_bar[s], state_bytes + bsc_bytes + krec_bytes + urec_bytes + arec_bytes +
                                                    draft_bytes);
            const size_t bh = static_cast<size_t>(tile);
            const size_t row0 = bh * DV + half * 64;
            if (RF == RSSM_READ_NONE)
                bulk_g2s_hint(st + geo.state, a.ckpt + row0 * DK, state_bytes, &full_bar[s], pol);
            else
                bulk_g2s_hint(st + geo.state, a.rc_codes + row0 * DK / (RF == RSSM_READ_FP8 ? 1 : 2), state_bytes,
                              &full_bar[s], pol);
            if (bsc_bytes) bulk_g2s(st + geo.bsc, a.rc_bscale + row0 * (DK / 16), bsc_bytes, &full_bar[s]);
            if (krec_bytes)
                bulk_g2s(st + geo.krec, reinterpret_cast<const TI*>(a.buf_k) + bh * a.cap * DK, krec_bytes,
                         &full_bar[s]);
            if (urec_bytes)
                bulk_g2s(st + geo.urec, a.buf_u + (bh * HALVES + half) * a.cap * 64, urec_bytes, &full_bar[s]);
            bulk_g2s(st + geo.arec, a.buf_a + bh * a.cap, arec_bytes, &full_bar[s]);
            for (int tau = 0; tau < T; ++tau) {
                const size_t row = (static_cast<size_t>(b) * T + tau) * a.H + hh;
                bulk_g2s(st + geo.qd + tau * DK * in_sz, reinterpret_cast<const TI*>(a.q) + row * DK, DK * in_sz,
                         &full_bar[s]);
                bulk_g2s(st + geo.kd + tau * DK * in_sz, reinterpret_cast<const TI*>(a.k) + row * DK, DK * in_sz,
                         &full_bar[s]);
                bulk_g2s(st + geo.vd + tau * 64 * in_sz, reinterpret_cast<const TI*>(a.v) + row * DV + half * 64,
                         64 * in_sz, &full_bar[s]);
            }
            issued |= 1u << s;
            last_par = (last_par & ~(1u << s)) | ((round & 1u) << s);
            if (++s == S) { s = 0; ++round; }
        }
        for (int q = 0; q < S; ++q)
            if ((issued >> q) & 1u)
                if (!mbar_wait_bounded(&full_bar[q], (last_par >> q) & 1u))
                    report_error(a.err, kDevTimeout, t0, 51);
        return;
    }

    // --------------------------------------------------------------- consumers
    const int g = (tid - 32) / GT;
    const int gt = (tid - 32) - g * GT;
    const int lane = gt & 31, gw = gt >> 5;
    const int cl = lane & 7, rg = lane >> 3;
    const int rloc = gw * 16 + rg * 4;   // first of the lane's 4 rows in the half
    const int rr = rloc + (cl & 3);      // this lane's row (cl < 4)

    // A group takes every NG-th tile and both of its halves, one after the
    // other: every draft's key dots are the same for both halves, so half 0
    // forms them and half 1 reuses them. (S is a multiple of NG * HALVES, so
    // every stage keeps one owner group.)
    for (int it = 0;; ++it) {
        const int tl = g + (it / HALVES) * NG, half = it % HALVES;
        if (tl >= nt) break;
        const int w = tl * HALVES + half;
        const int tile = t0 + tl;
        const int b = tile / a.H, hh = tile - b * a.H;
        const int s = w % S;
        const uint32_t par = static_cast<uint32_t>(w / S) & 1u;
        int ok = 0;
        if (lane == 0) ok = (!s_abort && mbar_wait_bounded(&full_bar[s], par)) ? 1 : 0;
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) {
            if (lane == 0 && !s_abort) {
                report_error(a.err, kDevTimeout, tile, 52);
                s_abort = 1;
            }
            return;
        }
        mbar_try_wait(&full_bar[s], par);

        const unsigned char* st = dsm + static_cast<size_t>(s) * geo.bytes;
        const int c = s_cnt[tl];
        if (c < 0) {
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty_bar[s]);
            continue;
        }
        const TI* sk = reinterpret_cast<const TI*>(st + geo.krec);
        const float* su = reinterpret_cast<const float*>(st + geo.urec);
        const float* sa = reinterpret_cast<const float*>(st + geo.arec);
        const TI* sqd = reinterpret_cast<const TI*>(st + geo.qd);
        const TI* skd = reinterpret_cast<const TI*>(st + geo.kd);
        const TI* svd = reinterpret_cast<const TI*>(st + geo.vd);
        // the copy's half scale multiplies the state dots (1 for the FP32 half)
        const float ts = !kCopy ? 1.f : __ldg(a.rc_tscale + static_cast<size_t>(tile) * HALVES + half);
        // alpha of draft (lane - c) for lanes c .. c+T-1
        const int dl = lane - c;
        const float ad = (dl >= 0 && dl < T) ? __ldg(a.alpha + (static_cast<size_t>(b) * T + dl) * a.H + hh) : 1.f;
        const float arec = (lane < c) ? sa[lane] : 1.f;

        // ---- phase A, from the stage: every draft's key dots (half 0 only)
        //      and state row-dots (independent of the other drafts' u rows),
        //      the records' u rows, and the drafts' v values; then release
        //      the stage. Drafts past T repeat the last one and are dropped.
        if (half == 0) {
            float kap[TMAX], lam[TMAX];
            if constexpr (kMmaKeys)
                draft_key_dots_mma<DK, TMAX>(kap, lam, reinterpret_cast<const __nv_bfloat16*>(sk),
                                             reinterpret_cast<const __nv_bfloat16*>(skd),
                                             reinterpret_cast<const __nv_bfloat16*>(sqd), a.scale, c, T, lane,
                                             s_kscr[kMmaKeys ? g * 4 + gw : 0]);
            else
                draft_key_dots<CPL, DK, TMAX>(kap, lam, sk, skd, sqd, a.scale, c, T, lane);
#pragma unroll
            for (int tau = 0; tau < TMAX; ++tau) {
                s_kst[g][gw][tau][0][lane] = kap[tau];
                s_kst[g][gw][tau][1][lane] = lam[tau];
            }
        }
        float kapd[TMAX], lamd[TMAX], pkd[TMAX][4], pqd[TMAX][4], vrd[TMAX];
        // every draft's state row-dots from one pass over the half
        if constexpr (kCopy)
            gdn_state_dots_multi<CPL, DK, TMAX>(pkd, pqd, CopyRef<RF, DK>{st + geo.state, st + geo.bsc}, skd, sqd,
                                                a.scale, T, rloc, cl);
        else
            gdn_state_dots_multi<CPL, DK, TMAX>(pkd, pqd, reinterpret_cast<const float4*>(st + geo.state), skd,
                                                sqd, a.scale, T, rloc, cl);
#pragma unroll
        for (int tau = 0; tau < TMAX; ++tau) {
            const int tq = min(tau, T - 1);
            vrd[tau] = to_f(svd[tq * 64 + rr]);
            kapd[tau] = s_kst[g][gw][tq][0][lane];
            lamd[tau] = s_kst[g][gw][tq][1][lane];
        }
        float urec[4][4];   // u rows of the records in this lane's set (j < c)
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            const int j = cl + 8 * kk;
            float4 v = zero4();
            if (j < c) v = *reinterpret_cast<const float4*>(su + j * 64 + rloc);
            urec[kk][0] = v.x; urec[kk][1] = v.y; urec[kk][2] = v.z; urec[kk][3] = v.w;
        }
        // append the drafts' k and alpha (once per tile, from the stage)
        if (half == 0 && gw == 0) {
            uint4* bk = reinterpret_cast<uint4*>(reinterpret_cast<TI*>(a.buf_k) +
                                                 (static_cast<size_t>(tile) * a.cap + c) * DK);
            const uint4* ks = reinterpret_cast<const uint4*>(skd);
            for (int q = lane; q < T * DK * in_sz / 16; q += 32) bk[q] = ks[q];
            if (dl >= 0 && dl < T) {
                a.buf_a[static_cast<size_t>(tile) * a.cap + lane] = ad;
                // with a read copy a flush replays v and beta too
                if (kCopy)
                    a.buf_beta[static_cast<size_t>(tile) * a.cap + lane] =
                        __ldg(a.beta + (static_cast<size_t>(b) * T + dl) * a.H + hh);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty_bar[s]);

        // ---- phase B, from registers. Each draft's reduction covers the
        //      committed records only, so the T reductions are independent;
        //      the earlier drafts' u rows enter afterwards, per row, in the
        //      lane that holds the row (a T x T triangular solve). Draft 0 is
        //      the one-token step's arithmetic exactly.
        float ru[TMAX], ro[TMAX], lamc[TMAX], bet[TMAX];
        float wkd[TMAX][TMAX], wqd[TMAX][TMAX];   // [tau'][tau]: weight of draft tau''s u in draft tau
#pragma unroll
        for (int tau = 0; tau < TMAX; ++tau) {
            ru[tau] = ro[tau] = lamc[tau] = bet[tau] = 0.f;
#pragma unroll
            for (int tp = 0; tp < TMAX; ++tp) wkd[tp][tau] = wqd[tp][tau] = 0.f;
            if (tau < T) {
                const int cc = c + tau;
                const int m = cc + 1;
                const float al = (lane < c) ? arec : (lane <= cc ? ad : 1.f);
                float gamma;
                const float rho = window_rho(al, lane, m, gamma);
                const float wk = (lane < cc) ? rho * kapd[tau] : 0.f;
                const float wq = (lane < cc) ? rho * lamd[tau] : 0.f;
                lamc[tau] = __shfl_sync(0xffffffffu, lamd[tau], cc & 31);
                bet[tau] = __ldg(a.beta + (static_cast<size_t>(b) * T + tau) * a.H + hh);
                gdn_finish_parts(pkd[tau], pqd[tau], urec, gamma * ts, wk, wq, c, lane, cl, &ru[tau], &ro[tau]);
#pragma unroll
                for (int tp = 0; tp < TMAX; ++tp) {
                    if (tp < tau) {
                        wkd[tp][tau] = __shfl_sync(0xffffffffu, wk, (c + tp) & 31);
                        wqd[tp][tau] = __shfl_sync(0xffffffffu, wq, (c + tp) & 31);
                    }
                }
            }
        }
        float ud[TMAX];
#pragma unroll
        for (int tau = 0; tau < TMAX; ++tau) {
            if (tau < T) {
                const int cc = c + tau;
                float r = ru[tau], o = ro[tau];
#pragma unroll
                for (int tp = 0; tp < TMAX; ++tp) {
                    if (tp < tau) {
                        r = fmaf(-wkd[tp][tau], ud[tp], r);
                        o = fmaf(wqd[tp][tau], ud[tp], o);
                    }
                }
                const float uc = bet[tau] * (vrd[tau] + r);
                ud[tau] = uc;
                o = o + lamc[tau] * uc;
                if (cl < 4) {
                    store_out(a.o, ((static_cast<size_t>(b) * T + tau) * a.H + hh) * DV + half * 64 + rr, o,
                              out_f32 != 0);
                    const size_t slot = ((static_cast<size_t>(tile) * HALVES + half) * a.cap + cc) * 64 + rr;
                    a.buf_u[slot] = uc;
                    if (kCopy) reinterpret_cast<TI*>(a.buf_v)[slot] = svd[min(tau, T - 1) * 64 + rr];
                }
            }
        }
    }
}

template <class L, typename TI, int NG, int TMAX, int RF>
cudaError_t launch_draft_ng(const GDNArgs& a, int out_f32, int S, int grid, int per, size_t smem, cudaStream_t s) {
    auto kernel = gdn_replay_draft_kernel<L, TI, NG, TMAX, RF>;
    static LaunchCache lc;
    cudaError_t e = cached_dyn_smem(lc, kernel, smem);
    if (e != cudaSuccess) return e;
    kernel<<<grid, 32 + NG * L::kThreads, smem, s>>>(a, out_f32, S, per);
    return cudaGetLastError();
}

template <class L, typename TI, int TMAX, int RF>
cudaError_t launch_draft(const GDNArgs& a, int out_f32, cudaStream_t s) {
    const int total = a.B * a.H;
    if (total == 0) return cudaSuccess;
    int num_sms = 0, smem_optin = 0;
    cudaError_t e = device_limits(&num_sms, &smem_optin);
    if (e != cudaSuccess) return e;
    static LaunchCache lc;
    int static_smem = 0;
    constexpr bool kTwoFit = (sizeof(TI) == 2 && TMAX <= 4) || TMAX <= 2;
    // the static shared memory of the larger build that may be launched
    e = cached_static_smem(lc, gdn_replay_draft_kernel<L, TI, kTwoFit ? 2 : 1, TMAX, RF>, &static_smem);
    if (e != cudaSuccess) return e;
    const DGeom geo = draft_geom(L::DK, a.cap, a.T, static_cast<int>(sizeof(TI)), RF);
    const int avail = smem_optin - static_smem - 1024;
    int smax = avail / geo.bytes;
    if (smax > kMaxStages) smax = kMaxStages;
    // every stage has one owner group: a group takes both halves of a tile in
    // a row, so S is a multiple of the group count times the halves
    // two groups fit the 168 registers a thread that nine warps allow with the
    // tensor-core key dots (bf16, T <= 4) or with two drafts; otherwise one
    // group, without spills
    const int ng = (kTwoFit && smax >= 2 * L::HALVES) ? 2 : 1;
    const int S = (smax / (ng * L::HALVES)) * (ng * L::HALVES);
    if (S < 2) return cudaErrorInvalidConfiguration;
    int grid = num_sms;
    if ((total + grid - 1) / grid > kMaxTilesPerCta) grid = (total + kMaxTilesPerCta - 1) / kMaxTilesPerCta;
    if (grid > total) grid = total;
    const int per = (total + grid - 1) / grid;
    grid = (total + per - 1) / per;
    const size_t smem = static_cast<size_t>(S) * geo.bytes;
    if constexpr (kTwoFit) {   // (two groups are never chosen otherwise: not built)
        if (ng == 2) return launch_draft_ng<L, TI, 2, TMAX, RF>(a, out_f32, S, grid, per, smem, s);
    }
    return launch_draft_ng<L, TI, 1, TMAX, RF>(a, out_f32, S, grid, per, smem, s);
}

template <class L, typename TI, int RF>
cudaError_t launch_draft_t(const GDNArgs& a, int out_f32, cudaStream_t s) {
    if (a.T == 2) return launch_draft<L, TI, 2, RF>(a, out_f32, s);
    if (a.T == 3) return launch_draft<L, TI, 3, RF>(a, out_f32, s);
    if (a.T == 4) return launch_draft<L, TI, 4, RF>(a, out_f32, s);
    return launch_draft<L, TI, kMaxDraft, RF>(a, out_f32, s);
}

template <class L>
cudaError_t run_draft(const GDNArgs& a, int in_dt, int out_dt, cudaStream_t s) {
    const int of = (out_dt == RSSM_F32);
    using BF = __nv_bfloat16;
    if (a.rf != RSSM_READ_NONE) {   // drafts that read the copy: bf16 inputs
        if (in_dt != RSSM_BF16) return cudaErrorInvalidValue;
        if (a.rf == RSSM_READ_FP8) return launch_draft_t<L, BF, RSSM_READ_FP8>(a, of, s);
        return launch_draft_t<L, BF, RSSM_READ_NVFP4>(a, of, s);
    }
    if (in_dt == RSSM_F32) return launch_draft_t<L, float, RSSM_READ_NONE>(a, of, s);
    return launch_draft_t<L, BF, RSSM_READ_NONE>(a, of, s);
}

}  // namespace

cudaError_t gdn_replay_draft(const GDNArgs& a, int DV, int DK, int in_dt, int out_dt, cudaStream_t s,
                             bool* supported) {
    *supported = true;
    if (a.T < 2 || a.T > kMaxDraft) return cudaErrorInvalidValue;
    if (DV == 128 && DK == 128) return run_draft<GdnTile<128, 128>>(a, in_dt, out_dt, s);
    if (DV == 64 && DK == 64) return run_draft<GdnTile<64, 64>>(a, in_dt, out_dt, s);
    if (DV == 64 && DK == 128) return run_draft<GdnTile<64, 128>>(a, in_dt, out_dt, s);
    if (DV == 128 && DK == 64) return run_draft<GdnTile<128, 64>>(a, in_dt, out_dt, s);
    *supported = false;
    return cudaSuccess;
}

}  // namespace rssm

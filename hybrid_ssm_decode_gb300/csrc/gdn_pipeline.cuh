// Pieces shared by the Gated DeltaNet replay kernels: the one-token fused and
// lean kernels (gdn_replay_tma.cu) and the speculative draft kernel
// (gdn_draft_tma.cu). It holds the tile split, the key dots, the state
// row-dots and the WY/UT finish, which every kernel calls in the same order,
// so they give bit-identical outputs for the same window.
//
// Method: "ReplaySSM beschleunigt ...", section "Wichtige Details" (Gated
// DeltaNet); "NVIDIA ve Dao AI Lab, ... ReplaySSM'i sundu", section "Durum
// trafigini azaltma ve rollback'in basitlestirilmesi".
#pragma once

#include "tile.cuh"

namespace rssm {
namespace {

constexpr int kMaxStages = 24;   // up to 24 stages of small (read-copy) halves
constexpr int kMaxTilesPerCta = 512;

template <int DV_, int DK_>
struct GdnTile {
    static constexpr int DV = DV_, DK = DK_;
    static constexpr int HALVES = DV / 64;    // 64-row work items per tile
    static constexpr int kWarps = 4;          // 16 rows each
    static constexpr int kThreads = 128;
    static constexpr int CPL = DK / 32;       // float4 columns per lane and row
    static constexpr int J = 4 * CPL;
    static_assert(DV % 64 == 0 && DK % 32 == 0, "tile split");
};

__host__ __device__ inline int galign128(int v) { return (v + 127) & ~127; }

// 4 consecutive FP32 values (rows r..r+3) of one u record.
__device__ __forceinline__ void load_u4(const float* p, float (&u)[4]) {
    const float4 v = *reinterpret_cast<const float4*>(p);
    u[0] = v.x; u[1] = v.y; u[2] = v.z; u[3] = v.w;
}

__device__ __forceinline__ float4 zero4() { return make_float4(0.f, 0.f, 0.f, 0.f); }

__device__ __forceinline__ float2 lo2(float4 v) { return make_float2(v.x, v.y); }
__device__ __forceinline__ float2 hi2(float4 v) { return make_float2(v.z, v.w); }

// Key dots of up to 16 records of the window, per warp: kappa_j = k_j . k_c
// and lambda_j = k_j . (scale q). Row group rg (lanes 8rg..8rg+7) takes
// records rg, rg+4, rg+8, rg+12 of the quad and its lane cl the column
// blocks cl + 8q; one 8-value group reduction sums all of them. On return
// lane j (and lane j + 16) holds the pair of record j of the quad.
// chunk(kk, q) gives column block cl + 8q of record rg + 4kk (zero past the
// window).
template <int CPL, class Chunk>
__device__ __forceinline__ void gdn_key_dots16(float& kap, float& lam, const float4 (&kv)[CPL],
                                               const float4 (&qv)[CPL], int lane, Chunk chunk) {
    float v[8];
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
        float dk = 0.f, dq = 0.f;
#pragma unroll
        for (int q = 0; q < CPL; ++q) {
            const float4 kb = chunk(kk, q);
            dk += dot4(kb, kv[q]);
            dq += dot4(kb, qv[q]);
        }
        v[2 * kk] = dk;
        v[2 * kk + 1] = dq;
    }
    const float red = group_reduce_multi<8, 8>(v, lane);   // lane 8rg + cl: value cl of row group rg
    const int src = (lane & 3) * 8 + 2 * ((lane >> 2) & 3);
    kap = __shfl_sync(0xffffffffu, red, src);
    lam = __shfl_sync(0xffffffffu, red, src + 1);
}

// All key dots of a window of m <= 32 records: lane j ends with record j's
// pair (zero for j >= m). chunk(qd, kk, q) is column block cl + 8q of record
// 16qd + rg + 4kk.
template <int CPL, class Chunk>
__device__ __forceinline__ void gdn_key_dots(float& kap, float& lam, const float4 (&kv)[CPL],
                                             const float4 (&qv)[CPL], int m, int lane, Chunk chunk) {
    kap = 0.f;
    lam = 0.f;
    for (int qd = 0; 16 * qd < m; ++qd) {
        float k1, l1;
        gdn_key_dots16<CPL>(k1, l1, kv, qv, lane, [&](int kk, int q) { return chunk(qd, kk, q); });
        if ((lane >> 4) == qd) {
            kap = k1;
            lam = l1;
        }
    }
}

// The read code of an FP16 checkpoint in the GDN replay kernels (a stored
// format, not a read copy: RSSM_READ_NONE, FP8 and NVFP4 are 0 to 2).
constexpr int kGdnF16 = 3;

// A 64-row state half as stored: FP32, or FP16 widened to FP32 on load
// (exact). idx counts 4-element chunks.
template <bool F16>
struct HalfRef {
    const void* p;
    __device__ __forceinline__ float4 operator()(int idx) const {
        if constexpr (F16) return f16x4_to_f32(reinterpret_cast<const uint2*>(p)[idx]);
        else return reinterpret_cast<const float4*>(p)[idx];
    }
};

template <int CPL, int DK, bool F16>
__device__ __forceinline__ void gdn_state_dots(float (&pk)[4], float (&pq)[4], HalfRef<F16> sh,
                                               const float4 (&kv)[CPL], const float4 (&qv)[CPL], int rloc,
                                               int cl);

// Unscaled S0 k and S0 q row-dots of this lane's 4 rows, from a stage.
template <int CPL, int DK>
__device__ __forceinline__ void gdn_state_dots(float (&pk)[4], float (&pq)[4], const float4* sh,
                                               const float4 (&kv)[CPL], const float4 (&qv)[CPL], int rloc,
                                               int cl) {
    gdn_state_dots<CPL, DK>(pk, pq, HalfRef<false>{sh}, kv, qv, rloc, cl);
}

// The same from a state half read through `sh` (HalfRef: FP32 or FP16).
template <int CPL, int DK, bool F16>
__device__ __forceinline__ void gdn_state_dots(float (&pk)[4], float (&pq)[4], HalfRef<F16> sh,
                                               const float4 (&kv)[CPL], const float4 (&qv)[CPL], int rloc,
                                               int cl) {
    constexpr int CH = DK / 4;
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        float2 ak = make_float2(0.f, 0.f), aq = make_float2(0.f, 0.f);
#pragma unroll
        for (int q = 0; q < CPL; ++q) {
            const float4 h = sh((rloc + p) * CH + cl + 8 * q);
            ak = __ffma2_rn(lo2(h), lo2(kv[q]), ak);
            ak = __ffma2_rn(hi2(h), hi2(kv[q]), ak);
            aq = __ffma2_rn(lo2(h), lo2(qv[q]), aq);
            aq = __ffma2_rn(hi2(h), hi2(qv[q]), aq);
        }
        pk[p] = ak.x + ak.y;
        pq[p] = aq.x + aq.y;
    }
}

// gdn_state_dots for up to TMAX drafts, two drafts per pass over the stage's
// state: each state chunk read serves two drafts' k and q. The
// accumulation order of each draft's dots is gdn_state_dots's (columns in
// order, low pair then high pair), so draft tau's values are the same bits.
// Drafts at or past T repeat draft T - 1. kd, qd: the drafts' k and q rows
// ([T][DK], input dtype) in shared memory; q is multiplied by scale first.
// A read-copy half (FP8, or NVFP4 with its block scales) decoded on load to
// unscaled values (block scale applied, tile scale not), as gdn_copy_dots
// decodes it. idx counts 4-element chunks.
template <int RF, int DK>
struct CopyRef {
    const unsigned char* codes;
    const unsigned char* bsc;
    __device__ __forceinline__ float4 operator()(int idx) const {
        constexpr int CH = DK / 4;
        if constexpr (RF == RSSM_READ_FP8) {
            const uint32_t u = reinterpret_cast<const uint32_t*>(codes)[idx];
            const float2 lo = e4m3x2_to_f2(static_cast<uint16_t>(u & 0xFFFFu));
            const float2 hi = e4m3x2_to_f2(static_cast<uint16_t>(u >> 16));
            return make_float4(lo.x, lo.y, hi.x, hi.y);
        } else {
            const int row = idx / CH, chunk = idx - row * CH;
            const uint32_t u = reinterpret_cast<const uint16_t*>(codes)[idx];
            const float bs = e4m3_to_f(bsc[row * (DK / 16) + (chunk >> 2)]);
            const float2 lo = e2m1x2_to_f2(u & 0xFFu);
            const float2 hi = e2m1x2_to_f2((u >> 8) & 0xFFu);
            return make_float4(lo.x * bs, lo.y * bs, hi.x * bs, hi.y * bs);
        }
    }
};

template <int CPL, int DK, int TMAX, typename TI, class SL>
__device__ __forceinline__ void gdn_state_dots_multi(float (&pk)[TMAX][4], float (&pq)[TMAX][4], SL sh,
                                                     const TI* kd, const TI* qd, float scale, int T, int rloc,
                                                     int cl);

template <int CPL, int DK, int TMAX, typename TI>
__device__ __forceinline__ void gdn_state_dots_multi(float (&pk)[TMAX][4], float (&pq)[TMAX][4], const float4* sh,
                                                     const TI* kd, const TI* qd, float scale, int T, int rloc,
                                                     int cl) {
    gdn_state_dots_multi<CPL, DK, TMAX>(pk, pq, HalfRef<false>{sh}, kd, qd, scale, T, rloc, cl);
}

// The same from a state half read through `sh` (HalfRef or CopyRef).
template <int CPL, int DK, int TMAX, typename TI, class SL>
__device__ __forceinline__ void gdn_state_dots_multi(float (&pk)[TMAX][4], float (&pq)[TMAX][4], SL sh,
                                                     const TI* kd, const TI* qd, float scale, int T, int rloc,
                                                     int cl) {
    constexpr int CH = DK / 4;
    constexpr int DB = TMAX < 2 ? TMAX : 2;   // drafts per pass over the state (bounds the live sums)
#pragma unroll
    for (int t0 = 0; t0 < TMAX; t0 += DB) {
        float2 ak[DB][4], aq[DB][4];
#pragma unroll
        for (int t = 0; t < DB; ++t)
#pragma unroll
            for (int p = 0; p < 4; ++p) {
                ak[t][p] = make_float2(0.f, 0.f);
                aq[t][p] = make_float2(0.f, 0.f);
            }
#pragma unroll
        for (int q = 0; q < CPL; ++q) {
            float4 kv[DB], qv[DB];
#pragma unroll
            for (int t = 0; t < DB; ++t) {
                const int tq = min(t0 + t, T - 1);
                kv[t] = load4(kd + tq * DK + (cl + 8 * q) * 4);
                const float4 u = load4(qd + tq * DK + (cl + 8 * q) * 4);
                qv[t] = make_float4(u.x * scale, u.y * scale, u.z * scale, u.w * scale);
            }
#pragma unroll
            for (int p = 0; p < 4; ++p) {
                const float4 h = sh((rloc + p) * CH + cl + 8 * q);
#pragma unroll
                for (int t = 0; t < DB; ++t) {
                    ak[t][p] = __ffma2_rn(lo2(h), lo2(kv[t]), ak[t][p]);
                    ak[t][p] = __ffma2_rn(hi2(h), hi2(kv[t]), ak[t][p]);
                    aq[t][p] = __ffma2_rn(lo2(h), lo2(qv[t]), aq[t][p]);
                    aq[t][p] = __ffma2_rn(hi2(h), hi2(qv[t]), aq[t][p]);
                }
            }
        }
#pragma unroll
        for (int t = 0; t < DB; ++t) {
            if (t0 + t >= TMAX) break;
#pragma unroll
            for (int p = 0; p < 4; ++p) {
                pk[t0 + t][p] = ak[t][p].x + ak[t][p].y;
                pq[t0 + t][p] = aq[t][p].x + aq[t][p].y;
            }
        }
    }
}

// The same row-dots from a read copy of the half (FP8 codes, or NVFP4 codes
// with their E4M3 block scales), unscaled by the copy's tile scale.
template <int RF, int CPL, int DK>
__device__ __forceinline__ void gdn_copy_dots(float (&pk)[4], float (&pq)[4], const unsigned char* codes,
                                              const unsigned char* bsc, const float4 (&kv)[CPL],
                                              const float4 (&qv)[CPL], int rloc, int cl) {
    constexpr int CH = DK / 4;
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        float2 ak = make_float2(0.f, 0.f), aq = make_float2(0.f, 0.f);
#pragma unroll
        for (int q = 0; q < CPL; ++q) {
            const int row = rloc + p, chunk = cl + 8 * q;
            float2 lo, hi;
            if (RF == RSSM_READ_FP8) {
                const uint32_t u = reinterpret_cast<const uint32_t*>(codes)[row * CH + chunk];
                lo = e4m3x2_to_f2(static_cast<uint16_t>(u & 0xFFFFu));
                hi = e4m3x2_to_f2(static_cast<uint16_t>(u >> 16));
            } else {
                const uint32_t u = reinterpret_cast<const uint16_t*>(codes)[row * CH + chunk];
                const float bs = e4m3_to_f(bsc[row * (DK / 16) + (chunk >> 2)]);
                lo = e2m1x2_to_f2(u & 0xFFu);
                hi = e2m1x2_to_f2((u >> 8) & 0xFFu);
                lo = make_float2(lo.x * bs, lo.y * bs);
                hi = make_float2(hi.x * bs, hi.y * bs);
            }
            ak = __ffma2_rn(lo, lo2(kv[q]), ak);
            ak = __ffma2_rn(hi, hi2(kv[q]), ak);
            aq = __ffma2_rn(lo, lo2(qv[q]), aq);
            aq = __ffma2_rn(hi, hi2(qv[q]), aq);
        }
        pk[p] = ak.x + ak.y;
        pq[p] = aq.x + aq.y;
    }
}

// Sum of 4 row values over the 8 lanes of a row group, left in every lane.
__device__ __forceinline__ void rowgroup_allsum4(float (&v)[4]) {
#pragma unroll
    for (int off = 1; off < 8; off <<= 1) {
#pragma unroll
        for (int p = 0; p < 4; ++p) v[p] += __shfl_xor_sync(0xffffffffu, v[p], off);
    }
}

// One token of the recurrence on this lane's part of a half-state held in
// registers (hv[p * CPL + q]: row rloc + p, column block cl + 8q):
//   w = S k, S <- alpha S + beta (v - alpha w) k^T.
// kb: the token's key columns; vr: v at the lane's 4 rows.
template <int CPL>
__device__ __forceinline__ void gdn_token_update(float4 (&hv)[4 * CPL], const float4 (&kb)[CPL],
                                                 const float (&vr)[4], float alpha, float beta) {
    float w[4];
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        float2 acc = make_float2(0.f, 0.f);
#pragma unroll
        for (int q = 0; q < CPL; ++q) {
            acc = __ffma2_rn(lo2(hv[p * CPL + q]), lo2(kb[q]), acc);
            acc = __ffma2_rn(hi2(hv[p * CPL + q]), hi2(kb[q]), acc);
        }
        w[p] = acc.x + acc.y;
    }
    rowgroup_allsum4(w);
    const float2 a2 = make_float2(alpha, alpha);
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        const float d = beta * (vr[p] - alpha * w[p]);
        const float2 d2 = make_float2(d, d);
#pragma unroll
        for (int q = 0; q < CPL; ++q) {
            float4& h = hv[p * CPL + q];
            const float2 h01 = __ffma2_rn(d2, lo2(kb[q]), __fmul2_rn(a2, lo2(h)));
            const float2 h23 = __ffma2_rn(d2, hi2(kb[q]), __fmul2_rn(a2, hi2(h)));
            h = make_float4(h01.x, h01.y, h23.x, h23.y);
        }
    }
}

// u_c and o_c for this lane's row (lanes cl < 4) from the state dots, the
// lane's records' u rows (uk[kk] for record cl + 8kk < c) and the weights.
// Returns the lane's part of the 8-value reduction; *uc and *o are valid
// where cl < 4.
__device__ __forceinline__ void gdn_finish(const float (&pk)[4], const float (&pq)[4], const float (&uk)[4][4],
                                           float gamma, float wk, float wq, int c, int lane, int cl, float vr,
                                           float beta, float lam_c, float* uc, float* o) {
    float part[8];
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        part[p] = -gamma * pk[p];
        part[4 + p] = gamma * pq[p];
    }
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
        const int j = cl + 8 * kk;
        const float ak = __shfl_sync(0xffffffffu, wk, j);
        const float aq = __shfl_sync(0xffffffffu, wq, j);
        if (j < c) {
#pragma unroll
            for (int p = 0; p < 4; ++p) {
                part[p] = fmaf(-ak, uk[kk][p], part[p]);
                part[4 + p] = fmaf(aq, uk[kk][p], part[4 + p]);
            }
        }
    }
    const float red = group_reduce_multi<8, 8>(part, lane);   // lane cl: value cl
    const float t2 = __shfl_down_sync(0xffffffffu, red, 4);
    *uc = beta * (vr + red);
    *o = t2 + lam_c * (*uc);
}

// The reduced parts of gdn_finish before they are combined: ru = -(gamma S0 k
// + sum_{j<c} w_j u_j) and ro = gamma S0 q + sum_{j<c} wq_j u_j for this
// lane's row (lanes cl < 4), in gdn_finish's arithmetic and order; then
// u_c = beta (v + ru) and o_c = ro + lambda_c u_c reproduce gdn_finish.
__device__ __forceinline__ void gdn_finish_parts(const float (&pk)[4], const float (&pq)[4], const float (&uk)[4][4],
                                                 float gamma, float wk, float wq, int c, int lane, int cl,
                                                 float* ru, float* ro) {
    float part[8];
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        part[p] = -gamma * pk[p];
        part[4 + p] = gamma * pq[p];
    }
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
        const int j = cl + 8 * kk;
        const float ak = __shfl_sync(0xffffffffu, wk, j);
        const float aq = __shfl_sync(0xffffffffu, wq, j);
        if (j < c) {
#pragma unroll
            for (int p = 0; p < 4; ++p) {
                part[p] = fmaf(-ak, uk[kk][p], part[p]);
                part[4 + p] = fmaf(aq, uk[kk][p], part[4 + p]);
            }
        }
    }
    const float red = group_reduce_multi<8, 8>(part, lane);   // lane cl: value cl
    *ro = __shfl_down_sync(0xffffffffu, red, 4);
    *ru = red;
    (void)cl;
}

// Four input elements as loaded (raw) and as FP32.
template <typename TI>
struct Raw4;
template <>
struct Raw4<float> {
    using T = float4;
    static __device__ __forceinline__ T ld(const float* p) { return __ldg(reinterpret_cast<const float4*>(p)); }
    static __device__ __forceinline__ T zero() { return make_float4(0.f, 0.f, 0.f, 0.f); }
    static __device__ __forceinline__ float4 f(T v) { return v; }
};
template <>
struct Raw4<__nv_bfloat16> {
    using T = uint2;
    static __device__ __forceinline__ T ld(const __nv_bfloat16* p) {
        return __ldg(reinterpret_cast<const uint2*>(p));
    }
    static __device__ __forceinline__ T zero() { return make_uint2(0u, 0u); }
    static __device__ __forceinline__ float4 f(T u) {
        return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xFFFF0000u),
                           __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xFFFF0000u));
    }
};


}  // namespace
}  // namespace rssm

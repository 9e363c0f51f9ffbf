// Pieces shared by the Mamba-2 replay kernels: the one-token fused and lean
// kernels (m2_replay_tma.cu) and the speculative draft kernel
// (m2_draft_tma.cu). It holds the consumer thread split of a tile, the
// input-element helpers, and the arithmetic the kernels share, so that they
// give bit-identical outputs for the same window.
//
// Method: "ReplaySSM beschleunigt das Decoding von Hybridmodellen durch
// Caching der Eingaben statt des Zustands", section "Wie es funktioniert".
#pragma once

#include "tile.cuh"

namespace rssm {
namespace {

constexpr int kMaxStages = 24;   // up to 24 stages of small (read-copy) tiles
constexpr int kMaxTilesPerCta = 512;
// Stage format value beside RSSM_READ_NONE / FP8 / NVFP4: the stage holds the
// FP16 checkpoint itself.
constexpr int kReadF16Ckpt = 3;

// Thread split of one tile for a consumer group. A warp covers 16 rows; in a
// warp, lanes 8*rg .. 8*rg+7 share the 4 consecutive rows 4*rg .. 4*rg+3 and
// lane cl = lane % 8 of them holds float4 columns cl, cl+8, cl+16, ... (N/32
// of them). So a row-dot is a sum over 8 lanes, a record's x values for the
// lane's rows are one 8-byte load, and one warp-wide 16-byte load covers
// 4 rows x 128 contiguous bytes (no bank conflict beyond the 4 wavefronts).
template <int P_, int N_>
struct GTile {
    static constexpr int P = P_, N = N_;
    static constexpr int kWarps = P / 16;
    static constexpr int kThreads = kWarps * 32;
    static constexpr int CPL = N / 32;      // float4 columns per lane and row
    static constexpr int J = 4 * CPL;       // float4 per thread
    static_assert(P % 16 == 0 && N % 32 == 0, "tile split");
};

__host__ __device__ inline int align128(int v) { return (v + 127) & ~127; }

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

// The same for a record in global memory, kept in L2 (evict-last).
template <typename TI>
__device__ __forceinline__ uint32_t raw_keep(const TI* p, uint64_t pol) {
    return sizeof(TI) == 2 ? ld_keep_u16(p, pol) : ld_keep_u32(p, pol);
}
template <typename TI>
__device__ __forceinline__ void store_raw_keep(TI* p, uint32_t raw, uint64_t pol) {
    if (sizeof(TI) == 2) st_keep_u16(p, raw, pol);
    else st_keep_u32(p, raw, pol);
}

template <typename TI>
__device__ __forceinline__ void store_raw(TI* p, uint32_t raw);
template <>
__device__ __forceinline__ void store_raw<float>(float* p, uint32_t raw) { *p = __uint_as_float(raw); }
template <>
__device__ __forceinline__ void store_raw<__nv_bfloat16>(__nv_bfloat16* p, uint32_t raw) {
    *reinterpret_cast<uint16_t*>(p) = static_cast<uint16_t>(raw);
}

// 4 consecutive x values (rows r..r+3) of one record, from shared memory.
template <typename TI>
__device__ __forceinline__ void load_x4(const TI* p, float (&x)[4]) {
    if (sizeof(TI) == 2) {
        const uint2 u = *reinterpret_cast<const uint2*>(p);
        x[0] = __uint_as_float(u.x << 16);
        x[1] = __uint_as_float(u.x & 0xFFFF0000u);
        x[2] = __uint_as_float(u.y << 16);
        x[3] = __uint_as_float(u.y & 0xFFFF0000u);
    } else {
        const uint4 u = *reinterpret_cast<const uint4*>(p);
        x[0] = __uint_as_float(u.x);
        x[1] = __uint_as_float(u.y);
        x[2] = __uint_as_float(u.z);
        x[3] = __uint_as_float(u.w);
    }
}

// ---------------------------------------------------------------------------
// Arithmetic shared by the fused kernel and the lean non-flush kernel, so the
// two produce bit-identical outputs for the same tile.
// ---------------------------------------------------------------------------

// Four consecutive input elements as loaded (generic address: global or
// shared memory), converted to FP32 where used.
template <typename TI> struct Chunk4;
template <> struct Chunk4<__nv_bfloat16> {
    uint2 v;
    __device__ __forceinline__ void load(const __nv_bfloat16* p) { v = *reinterpret_cast<const uint2*>(p); }
    __device__ __forceinline__ void load_keep(const __nv_bfloat16* p, uint64_t pol) { v = ld_keep_u2(p, pol); }
    __device__ __forceinline__ void zero() { v = make_uint2(0u, 0u); }
    __device__ __forceinline__ float4 f() const {
        return make_float4(__uint_as_float(v.x << 16), __uint_as_float(v.x & 0xFFFF0000u),
                           __uint_as_float(v.y << 16), __uint_as_float(v.y & 0xFFFF0000u));
    }
};
template <> struct Chunk4<float> {
    float4 v;
    __device__ __forceinline__ void load(const float* p) { v = *reinterpret_cast<const float4*>(p); }
    __device__ __forceinline__ void load_keep(const float* p, uint64_t pol) { v = ld_keep_f4(p, pol); }
    __device__ __forceinline__ void zero() { v = make_float4(0.f, 0.f, 0.f, 0.f); }
    __device__ __forceinline__ float4 f() const { return v; }
};

// Loads of one quad of a window's B records: row group rg takes records
// 16qd + rg + 4kk (kk < 4), lane cl their column blocks cl + 8q; records at or
// past `lim` read as zero. All loads are issued before any is used. Records
// below `nkeep` are in global memory and are loaded with the L2 policy `pol`.
template <typename TI, int CPL, class BPtr>
__device__ __forceinline__ void load_bquad(Chunk4<TI> (&bq)[4][CPL], int qd, int lim, int lane, int cl, BPtr bptr,
                                           int nkeep = 0, uint64_t pol = 0) {
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
        const int i = 16 * qd + (lane >> 3) + 4 * kk;
#pragma unroll
        for (int q = 0; q < CPL; ++q) {
            if (i < nkeep) bq[kk][q].load_keep(bptr(i) + (cl + 8 * q) * 4, pol);
            else if (i < lim) bq[kk][q].load(bptr(i) + (cl + 8 * q) * 4);
            else bq[kk][q].zero();
        }
    }
}

// Dots of one loaded quad with one C vector, for a window of m records;
// lanes 16qd .. 16qd+15 receive record (lane - 16qd)'s dot in bc.
template <typename TI, int CPL>
__device__ __forceinline__ void quad_dots(float& bc, const Chunk4<TI> (&bq)[4][CPL], const float4 (&cv)[CPL],
                                          int qd, int m, int lane) {
    float v[4];
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
        float d = 0.f;
        if (16 * qd + (lane >> 3) + 4 * kk < m) {
#pragma unroll
            for (int q = 0; q < CPL; ++q) d += dot4(bq[kk][q].f(), cv[q]);
        }
        v[kk] = d;
    }
    const float r = group_reduce_multi<4, 8>(v, lane);   // lane 8rg + cl: pass cl / 2 of row group rg
    const float t = __shfl_sync(0xffffffffu, r, (lane & 3) * 8 + 2 * ((lane >> 2) & 3));
    if ((lane >> 4) == qd) bc = t;
}

// B_i . C_t for the m <= 32 records of a window: on return lane i holds
// record i's dot (zero for i >= m). bptr(i) gives record i's B vector (global
// or shared memory).
template <typename TI, int CPL, class BPtr>
__device__ __forceinline__ void window_dots(float& bc, const float4 (&cv)[CPL], int m, int lane, int cl,
                                            BPtr bptr, int nkeep = 0, uint64_t pol = 0) {
    bc = 0.f;
    for (int qd = 0; 16 * qd < m; ++qd) {
        Chunk4<TI> bq[4][CPL];
        load_bquad<TI, CPL>(bq, qd, m, lane, cl, bptr, nkeep, pol);
        quad_dots<TI, CPL>(bc, bq, cv, qd, m, lane);
    }
}

// The window-dot key's inputs, copied into the dots warp's scratch in one
// round trip: records 0..c-1 of the B/C group's B buffer (L2 evict-last, as
// they are read again later in the window), then the ntok token rows of B
// (brow(tau)) after them, and the ntok token rows of C (crow(tau)) at sc.
// Lane 0 issues the copies and waits (bounded) on `bar`, phase `par`.
// Returns false on a timeout, after reporting it and waiting once more
// (bounded) for the copies in flight.
template <typename TI, class BRow, class CRow>
__device__ __forceinline__ bool dots_fetch(unsigned char* sb, unsigned char* sc, const TI* gb, int c, int ntok,
                                           BRow brow, CRow crow, int N, uint64_t* bar, uint32_t par,
                                           uint64_t keep, int lane, int32_t* err, int where) {
    int ok = 1;
    if (lane == 0) {
        const uint32_t row = static_cast<uint32_t>(N * sizeof(TI));
        mbar_arrive_expect_tx(bar, (c + 2 * ntok) * row);
        if (c > 0) bulk_g2s_hint(sb, gb, c * row, bar, keep);
        for (int tau = 0; tau < ntok; ++tau) {
            bulk_g2s(sb + (c + tau) * row, brow(tau), row, bar);
            bulk_g2s(sc + tau * row, crow(tau), row, bar);
        }
        if (!mbar_wait_bounded(bar, par)) {
            report_error(err, kDevTimeout, where, 34);
            mbar_wait_bounded(bar, par);
            ok = 0;
        }
    }
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (ok) mbar_try_wait(bar, par);   // every lane observes the completed phase
    return ok != 0;
}

// Unscaled row-dots of this lane's 4 rows of the checkpoint (FP32 or FP16) or
// of its read copy, with its C_t columns, read from a stage.
template <int RF, int CPL, int N>
__device__ __forceinline__ void stage_row_dots(float (&part)[4], const unsigned char* state,
                                               const unsigned char* bsc, const float4 (&cv)[CPL], int rbase,
                                               int cl) {
    constexpr int CH = N / 4;
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        float acc = 0.f;
        float2 acc2 = make_float2(0.f, 0.f);
#pragma unroll
        for (int q = 0; q < CPL; ++q) {
            const int row = rbase + p, chunk = cl + 8 * q;
            const int idx = row * CH + chunk;
            if (RF == RSSM_READ_NONE || RF == kReadF16Ckpt) {
                const float4 h = (RF == RSSM_READ_NONE) ? reinterpret_cast<const float4*>(state)[idx]
                                                        : f16x4_to_f32(reinterpret_cast<const uint2*>(state)[idx]);
                acc2 = __ffma2_rn(make_float2(h.x, h.y), make_float2(cv[q].x, cv[q].y), acc2);
                acc2 = __ffma2_rn(make_float2(h.z, h.w), make_float2(cv[q].z, cv[q].w), acc2);
            } else if (RF == RSSM_READ_FP8) {
                const uint32_t u = reinterpret_cast<const uint32_t*>(state)[idx];
                const float2 lo = e4m3x2_to_f2(static_cast<uint16_t>(u & 0xFFFFu));
                const float2 hi = e4m3x2_to_f2(static_cast<uint16_t>(u >> 16));
                acc += dot4(make_float4(lo.x, lo.y, hi.x, hi.y), cv[q]);
            } else {
                const uint32_t u = reinterpret_cast<const uint16_t*>(state)[idx];
                const float bs = e4m3_to_f(bsc[row * (N / 16) + (chunk >> 2)]);
                const float2 lo = e2m1x2_to_f2(u & 0xFFu);
                const float2 hi = e2m1x2_to_f2((u >> 8) & 0xFFu);
                acc += bs * dot4(make_float4(lo.x, lo.y, hi.x, hi.y), cv[q]);
            }
        }
        part[p] = acc + acc2.x + acc2.y;
    }
}

// Non-flush output of this lane's 4 rows from the unscaled row-dots, the x
// values of the lane's records (cl, cl+8, ...: xk[k] valid where
// cl + 8k < m) and the window's dt (lane i: dt_i). Returns the reduced row
// value held by this lane (row rbase + (lane & 7)/2, even lanes).
__device__ __forceinline__ float nonflush_finish(float (&part)[4], const float (&xk)[4][4], float dti,
                                                 float bc, int c, int m, float Ah, float Dh, float tscale,
                                                 int lane, int cl) {
    float gamma;
    const float decay = window_decay(dti, lane, m, Ah, gamma);
    const float w = (lane < m) ? decay * dti * bc : 0.f;
    const float gs = gamma * tscale;
#pragma unroll
    for (int p = 0; p < 4; ++p) part[p] *= gs;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int i = cl + 8 * k;
        const float wk = __shfl_sync(0xffffffffu, w, i) + (i == c ? Dh : 0.f);
        if (i < m) {
#pragma unroll
            for (int p = 0; p < 4; ++p) part[p] = fmaf(wk, xk[k][p], part[p]);
        }
    }
    return group_reduce_multi<4, 8>(part, lane);
}

// ---------------------------------------------------------------------------
// Read-copy row-dots on the tensor cores (bf16 inputs). A warp's 16 rows of
// the FP8 / NVFP4 copy times C_t, as one m16n8k16 MMA (f16 in, FP32
// accumulate) per 16 columns. This replaces the per-element decode and FMAs
// of row_dot, which bound the copy paths by instruction issue.
//  * E4M3 and E2M1 codes convert exactly to f16, and so does an E2M1 code
//    times its E4M3 block scale (at most 6 significant bits, within range).
//  * C_t enters as f16 after an exact power-of-two scaling that puts its
//    largest element in [2^14, 2^15): a bf16 value is then an f16 value,
//    except elements below 2^-28 of the largest, which round to f16
//    subnormals. The products are exact; the sums are FP32.
//  * The MMA's column order is free (the same permutation on A's columns
//    and B's rows): lane (g, t) = (lane / 4, lane % 4) takes columns
//    (N/4) t .. (N/4) t + N/4 - 1 of rows g and g + 8, so its codes are
//    contiguous 16-byte loads; MMA j uses its columns 4j .. 4j + 3.
//  * Every lane gets the same B fragment (C in every MMA column), so every
//    lane ends with the dots of rows g (d[0]) and g + 8 (d[2]).
// ---------------------------------------------------------------------------
template <int N>
struct CFrag {
    uint32_t b[N / 16][2];   // B fragments of the N/16 column blocks
    float inv_scale;         // 1 / the power-of-two scale of C
};

__device__ __forceinline__ uint32_t f16x2_bits(float lo, float hi) {
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&h);
}

__device__ __forceinline__ uint32_t cvt_e4m3x2_f16x2(uint32_t two_codes) {
    uint32_t h2;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(static_cast<uint16_t>(two_codes)));
    return h2;
}

__device__ __forceinline__ uint32_t cvt_e2m1x2_f16x2(uint32_t byte) {
    uint32_t h2;
    asm("{\n\t.reg .b8 t;\n\tcvt.u8.u32 t, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}" : "=r"(h2) : "r"(byte));
    return h2;
}

__device__ __forceinline__ uint32_t hmul2_bits(uint32_t a, uint32_t b) {
    const __half2 r = __hmul2(*reinterpret_cast<const __half2*>(&a), *reinterpret_cast<const __half2*>(&b));
    return *reinterpret_cast<const uint32_t*>(&r);
}

__device__ __forceinline__ void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                              uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// B fragments of C_t (bf16, in shared memory) for the MMA row-dots.
template <int N>
__device__ __forceinline__ void make_cfrag(CFrag<N>& f, const __nv_bfloat16* ct, int lane) {
    constexpr int CPT = N / 4;               // columns per lane position t
    const int t = lane & 3;
    float v[CPT];
#pragma unroll
    for (int q = 0; q < CPT / 4; ++q) {
        const float4 c4 = load4(ct + CPT * t + 4 * q);
        v[4 * q] = c4.x; v[4 * q + 1] = c4.y; v[4 * q + 2] = c4.z; v[4 * q + 3] = c4.w;
    }
    float mx = 0.f;
#pragma unroll
    for (int i = 0; i < CPT; ++i) mx = fmaxf(mx, fabsf(v[i]));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    int e = 0;
    if (mx > 0.f) frexpf(mx, &e);
    int sh = 15 - e;                          // mx * 2^sh in [2^14, 2^15)
    if (sh > 126) sh = 126;
    if (mx == 0.f) sh = 0;
    const float sc = ldexpf(1.f, sh);
    f.inv_scale = ldexpf(1.f, -sh);
#pragma unroll
    for (int j = 0; j < N / 16; ++j) {
        f.b[j][0] = f16x2_bits(v[4 * j] * sc, v[4 * j + 1] * sc);
        f.b[j][1] = f16x2_bits(v[4 * j + 2] * sc, v[4 * j + 3] * sc);
    }
}

// The MMA fragment d of rows r0 + g and r0 + g + 8 of the copy times the B
// fragments in f: d[0], d[1] = row r0 + g, columns 2t, 2t + 1; d[2], d[3] =
// row r0 + g + 8. With one C vector in every column (CFrag), d[0] = d[1] and
// d[2] = d[3] are the two rows' dots; with one draft's C per column
// (CFragMulti), column n is draft n's dot.
template <int RF, int N>
__device__ __forceinline__ void rc_mma_rows(float (&d)[4], const unsigned char* state, const unsigned char* bsc,
                                            const uint32_t (&fb)[N / 16][2], int r0, int lane) {
    constexpr int NJ = N / 16;
    const int g = lane >> 2, t = lane & 3;
    const int rA = r0 + g, rB = r0 + g + 8;
    d[0] = d[1] = d[2] = d[3] = 0.f;
    if (RF == RSSM_READ_FP8) {
        // N/4 code bytes per lane and row
        uint32_t wa[NJ], wb[NJ];
        if (N == 128) {
            // two 16-byte halves; odd rows read the upper half first, so the
            // 8 lanes of a load phase (2 rows) hit 8 different bank groups
            const int hA = g & 1;
            const uint4* pa = reinterpret_cast<const uint4*>(state + rA * N + 32 * t);
            const uint4* pb = reinterpret_cast<const uint4*>(state + rB * N + 32 * t);
            const uint4 a_first = pa[hA], a_second = pa[hA ^ 1];
            const uint4 b_first = pb[hA], b_second = pb[hA ^ 1];
            const uint4 a_lo = hA ? a_second : a_first, a_hi = hA ? a_first : a_second;
            const uint4 b_lo = hA ? b_second : b_first, b_hi = hA ? b_first : b_second;
            wa[0] = a_lo.x; wa[1] = a_lo.y; wa[2] = a_lo.z; wa[3] = a_lo.w;
            wa[4] = a_hi.x; wa[5] = a_hi.y; wa[6] = a_hi.z; wa[7] = a_hi.w;
            wb[0] = b_lo.x; wb[1] = b_lo.y; wb[2] = b_lo.z; wb[3] = b_lo.w;
            wb[4] = b_hi.x; wb[5] = b_hi.y; wb[6] = b_hi.z; wb[7] = b_hi.w;
        } else {
            const uint4 a4 = *reinterpret_cast<const uint4*>(state + rA * N + 16 * t);
            const uint4 b4 = *reinterpret_cast<const uint4*>(state + rB * N + 16 * t);
            wa[0] = a4.x; wa[1] = a4.y; wa[2] = a4.z; wa[3] = a4.w;
            wb[0] = b4.x; wb[1] = b4.y; wb[2] = b4.z; wb[3] = b4.w;
        }
#pragma unroll
        for (int j = 0; j < NJ; ++j)
            mma_f16_16816(d, cvt_e4m3x2_f16x2(wa[j] & 0xFFFFu), cvt_e4m3x2_f16x2(wb[j] & 0xFFFFu),
                          cvt_e4m3x2_f16x2(wa[j] >> 16), cvt_e4m3x2_f16x2(wb[j] >> 16), fb[j][0], fb[j][1]);
    } else {
        // N/8 code bytes per lane and row; block scales of its N/64 blocks
        uint32_t wa[NJ / 2], wb[NJ / 2];
        if (N == 128) {
            const uint4 a4 = *reinterpret_cast<const uint4*>(state + rA * (N / 2) + 16 * t);
            const uint4 b4 = *reinterpret_cast<const uint4*>(state + rB * (N / 2) + 16 * t);
            wa[0] = a4.x; wa[1] = a4.y; wa[2] = a4.z; wa[3] = a4.w;
            wb[0] = b4.x; wb[1] = b4.y; wb[2] = b4.z; wb[3] = b4.w;
        } else {
            const uint2 a2 = *reinterpret_cast<const uint2*>(state + rA * (N / 2) + 8 * t);
            const uint2 b2 = *reinterpret_cast<const uint2*>(state + rB * (N / 2) + 8 * t);
            wa[0] = a2.x; wa[1] = a2.y;
            wb[0] = b2.x; wb[1] = b2.y;
        }
        uint32_t sA, sB;   // block scales as f16x2 (N = 128: blocks 2t, 2t + 1; N = 64: block t twice)
        if (N == 128) {
            sA = cvt_e4m3x2_f16x2(*reinterpret_cast<const uint16_t*>(bsc + rA * (N / 16) + 2 * t));
            sB = cvt_e4m3x2_f16x2(*reinterpret_cast<const uint16_t*>(bsc + rB * (N / 16) + 2 * t));
        } else {
            sA = cvt_e4m3x2_f16x2(bsc[rA * (N / 16) + t] * 0x101u);
            sB = cvt_e4m3x2_f16x2(bsc[rB * (N / 16) + t] * 0x101u);
        }
        const uint32_t sA0 = __byte_perm(sA, 0, 0x1010), sA1 = __byte_perm(sA, 0, 0x3232);
        const uint32_t sB0 = __byte_perm(sB, 0, 0x1010), sB1 = __byte_perm(sB, 0, 0x3232);
#pragma unroll
        for (int j = 0; j < NJ; ++j) {
            const uint32_t ba = (wa[j / 2] >> (16 * (j & 1))) & 0xFFFFu;   // codes of columns 4j .. 4j+3
            const uint32_t bb = (wb[j / 2] >> (16 * (j & 1))) & 0xFFFFu;
            const uint32_t xa = (j < 4) ? sA0 : sA1, xb = (j < 4) ? sB0 : sB1;
            mma_f16_16816(d, hmul2_bits(cvt_e2m1x2_f16x2(ba & 0xFFu), xa), hmul2_bits(cvt_e2m1x2_f16x2(bb & 0xFFu), xb),
                          hmul2_bits(cvt_e2m1x2_f16x2(ba >> 8), xa), hmul2_bits(cvt_e2m1x2_f16x2(bb >> 8), xb),
                          fb[j][0], fb[j][1]);
        }
    }
}

// Dots of rows r0 + g (dA) and r0 + g + 8 (dB) of the copy with C_t, times
// the C scale (the tile scale is applied by the caller).
template <int RF, int N>
__device__ __forceinline__ void rc_row_dots_mma(float& dA, float& dB, const unsigned char* state,
                                                const unsigned char* bsc, const CFrag<N>& f, int r0, int lane) {
    float d[4];
    rc_mma_rows<RF, N>(d, state, bsc, f.b, r0, lane);
    dA = d[0];
    dB = d[2];
}

// B fragments with one draft's C per MMA column: lane (g, t) holds column n =
// g, draft g's C (zero for g >= T), each draft scaled by its own power of two
// as in make_cfrag; lanes 4n .. 4n + 3 hold draft n's inverse scale.
template <int N>
struct CFragMulti {
    uint32_t b[N / 16][2];
    float inv_scale;
};

template <int N>
__device__ __forceinline__ void make_cfrag_multi(CFragMulti<N>& f, const __nv_bfloat16* ct, int T, int lane) {
    constexpr int CPT = N / 4;
    const int g = lane >> 2, t = lane & 3;
    const bool live = g < T;
    float v[CPT];
#pragma unroll
    for (int q = 0; q < CPT / 4; ++q) {
        const float4 c4 = live ? load4(ct + g * N + CPT * t + 4 * q) : make_float4(0.f, 0.f, 0.f, 0.f);
        v[4 * q] = c4.x; v[4 * q + 1] = c4.y; v[4 * q + 2] = c4.z; v[4 * q + 3] = c4.w;
    }
    float mx = 0.f;
#pragma unroll
    for (int i = 0; i < CPT; ++i) mx = fmaxf(mx, fabsf(v[i]));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    int e = 0;
    if (mx > 0.f) frexpf(mx, &e);
    int sh = 15 - e;                          // mx * 2^sh in [2^14, 2^15)
    if (sh > 126) sh = 126;
    if (mx == 0.f) sh = 0;
    const float sc = ldexpf(1.f, sh);
    f.inv_scale = ldexpf(1.f, -sh);
#pragma unroll
    for (int j = 0; j < N / 16; ++j) {
        f.b[j][0] = f16x2_bits(v[4 * j] * sc, v[4 * j + 1] * sc);
        f.b[j][1] = f16x2_bits(v[4 * j + 2] * sc, v[4 * j + 3] * sc);
    }
}

// Raw x values of 4 consecutive rows of one record, from global memory.
template <typename TI> struct XRaw;
template <> struct XRaw<__nv_bfloat16> {
    uint2 v;
    __device__ __forceinline__ void load(const __nv_bfloat16* p) { v = __ldg(reinterpret_cast<const uint2*>(p)); }
    __device__ __forceinline__ void load_keep(const __nv_bfloat16* p, uint64_t pol) { v = ld_keep_u2(p, pol); }
    __device__ __forceinline__ void to(float (&x)[4]) const {
        x[0] = __uint_as_float(v.x << 16);
        x[1] = __uint_as_float(v.x & 0xFFFF0000u);
        x[2] = __uint_as_float(v.y << 16);
        x[3] = __uint_as_float(v.y & 0xFFFF0000u);
    }
};
template <> struct XRaw<float> {
    float4 v;
    __device__ __forceinline__ void load(const float* p) { v = __ldg(reinterpret_cast<const float4*>(p)); }
    __device__ __forceinline__ void load_keep(const float* p, uint64_t pol) { v = ld_keep_f4(p, pol); }
    __device__ __forceinline__ void to(float (&x)[4]) const { x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w; }
};

template <typename TI>
__device__ __forceinline__ void store_x4raw(TI* p, const XRaw<TI>& r);
template <>
__device__ __forceinline__ void store_x4raw<float>(float* p, const XRaw<float>& r) {
    *reinterpret_cast<float4*>(p) = r.v;
}
template <>
__device__ __forceinline__ void store_x4raw<__nv_bfloat16>(__nv_bfloat16* p, const XRaw<__nv_bfloat16>& r) {
    *reinterpret_cast<uint2*>(p) = r.v;
}


}  // namespace
}  // namespace rssm

// Device helpers shared by the librssm kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "rssm.h"

namespace rssm {

constexpr int kMaxCap = 32;      // buffer records per (sequence, head), at most
constexpr int kMaxDraft = 8;     // drafted tokens per decode step, at most
constexpr int kDevTimeout = RSSM_DEV_TIMEOUT;   // device error code: a bounded wait ran out

// --------------------------------------------------------------------------
// Kernel arguments (one struct per SSM kind, passed by value)
// --------------------------------------------------------------------------
struct M2Args {
    float* ckpt;          // [B][H][P][N] FP32
    int32_t* counts;      // [B][H]
    int32_t* err;         // [4]
    void* buf_x;          // [B][H][cap][P]
    void* buf_b;          // [B][G][cap][N]
    void* buf_dt;         // [B][H][cap]
    uint8_t* rc_codes;    // read copy
    uint8_t* rc_bscale;
    float* rc_tscale;
    float* snap;          // [Tmax][B][H][P][N]
    const float* A;       // [H]
    const float* D;       // [H]
    const void* x;        // [B][T][H][P]
    const void* Bm;       // [B][T][G][N]
    const void* C;        // [B][T][G][N]
    const void* dt;       // [B][T][H]
    void* y;              // [B][T][H][P]
    const int32_t* accepted;  // [B]
    int B, H, G, k, cap, T;
    int force;            // commit kernel: fold every tile with c > 0
    int ck;               // checkpoint storage: kCkF32, kCkF16, kCkFP8, kCkNVFP4
    uint8_t* ck_bscale;   // tile-format checkpoint: NVFP4 block scales [B][H][P][N/16]
    float* ck_tscale;     // tile-format checkpoint: tile scales [B][H]
    int defer_copy;       // step / commit kernels: folded tiles leave the read copy to a quantiser launch
};

// Checkpoint storage kinds (replay, bf16 inputs for all but kCkF32). The tile
// formats are the read-copy formats; their codes sit in the ckpt region.
enum { kCkF32 = 0, kCkF16 = 1, kCkFP8 = 2, kCkNVFP4 = 3 };
__host__ __device__ constexpr int ck_tile_fmt(int ck) {
    return ck == kCkFP8 ? RSSM_READ_FP8 : ck == kCkNVFP4 ? RSSM_READ_NVFP4 : RSSM_READ_NONE;
}

struct GDNArgs {
    float* ckpt;          // [B][H][DV][DK]
    int32_t* counts;      // [B][H]
    int32_t* err;
    void* buf_k;          // [B][H][cap][DK] in_dtype
    float* buf_u;         // [B][H][DV/64][cap][64]
    float* buf_a;         // [B][H][cap]
    const void* q;        // [B][T][H][DK]
    const void* k;        // [B][T][H][DK]
    const void* v;        // [B][T][H][DV]
    const float* alpha;   // [B][T][H]
    const float* beta;    // [B][T][H]
    void* o;              // [B][T][H][DV]
    const int32_t* accepted;  // [B]
    // read copy (one copy tile per 64-row half) and the records a flush
    // replays from with a read copy
    uint8_t* rc_codes;    // FP8 [B][H][DV][DK]; NVFP4 [B][H][DV][DK/2]
    uint8_t* rc_bscale;   // NVFP4 [B][H][DV][DK/16]
    float* rc_tscale;     // [B][H][DV/64]
    void* buf_v;          // [B][H][DV/64][cap][64] in_dtype
    float* buf_beta;      // [B][H][cap]
    float* snap;          // conventional drafts: [Tmax][B][H][DV][DK]
    int B, H, kflush, cap, T;
    float scale;
    int force;
    int rf;               // RSSM_READ_*
    int defer_copy;       // step kernel: flush tiles leave the read copy to a quantiser launch
    int ck;               // checkpoint storage: kCkF32 or kCkF16
};

// Launchers (defined in m2_kernels.cu, m2_replay_tma.cu, m2_draft_tma.cu,
// m2_commit_tma.cu, gdn_kernels.cu, gdn_replay_tma.cu, gdn_draft_tma.cu). path:
//  kStepAny       the replay step kernel, every tile (flush or not);
//  kStepNonFlush  the lean kernel, for launches in which no tile completes its
//                 window (the caller knows every record count is below k - 1);
//  kStepFlushOnly the replay step kernel over only the tiles that complete
//                 their window (c = k - 1); it marks them with count k;
//  kStepSkipFlush launched next in the same step: the lean kernel over the
//                 other tiles, resetting the marked ones to 0.
enum { kStepAny = 0, kStepNonFlush = 1, kStepSkipFlush = 2, kStepFlushOnly = 3 };
cudaError_t m2_replay_step(const M2Args& a, int P, int N, int in_dt, int out_dt, int rf, int path,
                           cudaStream_t s, bool* supported);
cudaError_t m2_replay_draft(const M2Args& a, int P, int N, int in_dt, int out_dt, int rf,
                            cudaStream_t s, bool* supported);
cudaError_t m2_commit(const M2Args& a, int P, int N, int in_dt, int rf, cudaStream_t s,
                      bool* supported);
// rf != RSSM_READ_NONE: the quantised-recurrence baseline (state stored as
// FP8 / NVFP4 tiles in the read-copy regions, re-quantised every step).
cudaError_t m2_conv_step(const M2Args& a, int P, int N, int in_dt, int out_dt, int rf, cudaStream_t s,
                         bool* supported);
cudaError_t m2_snap_draft(const M2Args& a, int P, int N, int in_dt, int out_dt,
                          cudaStream_t s, bool* supported);
cudaError_t m2_snap_restore(const M2Args& a, int P, int N, cudaStream_t s, bool* supported);
cudaError_t gdn_replay_step(const GDNArgs& a, int DV, int DK, int in_dt, int out_dt, int path,
                            cudaStream_t s, bool* supported);
cudaError_t gdn_replay_draft(const GDNArgs& a, int DV, int DK, int in_dt, int out_dt, cudaStream_t s,
                             bool* supported);
cudaError_t gdn_commit(const GDNArgs& a, int DV, int DK, int in_dt, cudaStream_t s,
                       bool* supported);
cudaError_t gdn_conv_step(const GDNArgs& a, int DV, int DK, int in_dt, int out_dt,
                          cudaStream_t s, bool* supported);
cudaError_t gdn_snap_draft(const GDNArgs& a, int DV, int DK, int in_dt, int out_dt, cudaStream_t s,
                           bool* supported);
cudaError_t gdn_snap_restore(const GDNArgs& a, int DV, int DK, cudaStream_t s, bool* supported);
cudaError_t quantize_tiles(int fmt, int64_t tiles, int rows, int cols, const float* src,
                           uint8_t* codes, uint8_t* bscale, float* tscale, cudaStream_t s,
                           bool* supported);
// The same writer from an FP16 checkpoint.
// Quantise FP8 tiles (codes + tile scales, as stored), decoded, into `fmt`.
cudaError_t quantize_tiles_from_fp8(int fmt, int64_t tiles, int rows, int cols, const uint8_t* src_codes,
                                    const float* src_tscale, uint8_t* codes, uint8_t* bscale, float* tscale,
                                    cudaStream_t s, bool* supported);
cudaError_t quantize_tiles_f16(int fmt, int64_t tiles, int rows, int cols, const __half* src,
                               uint8_t* codes, uint8_t* bscale, float* tscale, cudaStream_t s,
                               bool* supported);
// The writer over FP32 (src) or FP16 (src16 != nullptr) tiles; with counts,
// only the tiles whose count is `mark` (the tiles a flush-only launch folded);
// `per` copy tiles share one count.
cudaError_t quantize_marked_tiles(int fmt, int64_t tiles, int rows, int cols, const float* src, const __half* src16,
                                  uint8_t* codes, uint8_t* bscale, float* tscale, const int32_t* counts, int mark,
                                  int per, cudaStream_t s, bool* supported);
// Multiprocessor count and opt-in shared memory per block of the current
// device (queried once per device ordinal).
cudaError_t device_limits(int* num_sms, int* smem_optin);

// Launch facts of one kernel, per device ordinal, so that a launch makes no
// attribute call after the first one on its device. A launcher keeps one in
// a function-local static (one per kernel instantiation, zero-initialised).
struct LaunchCache {
    static constexpr int kDevices = 64;
    int static_smem[kDevices];   // static shared memory + 1; 0: not queried yet
    int dyn_limit[kDevices];     // dynamic shared memory limit set so far
};

template <class K>
cudaError_t cached_static_smem(LaunchCache& lc, K kernel, int* bytes) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const bool slot = dev >= 0 && dev < LaunchCache::kDevices;
    if (slot && lc.static_smem[dev] > 0) {
        *bytes = lc.static_smem[dev] - 1;
        return cudaSuccess;
    }
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, kernel);
    if (e != cudaSuccess) return e;
    *bytes = static_cast<int>(fa.sharedSizeBytes);
    if (slot) lc.static_smem[dev] = *bytes + 1;
    return cudaSuccess;
}

template <class K>
cudaError_t cached_dyn_smem(LaunchCache& lc, K kernel, size_t smem) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const bool slot = dev >= 0 && dev < LaunchCache::kDevices;
    if (slot && lc.dyn_limit[dev] >= static_cast<int>(smem)) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e == cudaSuccess && slot) lc.dyn_limit[dev] = static_cast<int>(smem);
    return e;
}
// FP32 -> FP16 (round to nearest even), n a multiple of 4, 8-byte aligned.
cudaError_t f32_to_f16_array(const float* src, __half* dst, int64_t n, cudaStream_t s);

// --------------------------------------------------------------------------
// Memory access
// --------------------------------------------------------------------------
__device__ __forceinline__ uint64_t l2_evict_first() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

__device__ __forceinline__ uint64_t l2_evict_last() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// 16-byte read-only load that skips L1 and marks the line evict-first in L2:
// for data streamed once per step (the checkpoint).
__device__ __forceinline__ float4 ld_stream(const float4* p, uint64_t pol) {
    float4 v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.f32 {%0,%1,%2,%3}, [%4], %5;"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "l"(p), "l"(pol));
    return v;
}

__device__ __forceinline__ uint32_t ld_stream_u32(const uint32_t* p, uint64_t pol) {
    uint32_t v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.b32 %0, [%1], %2;"
                 : "=r"(v) : "l"(p), "l"(pol));
    return v;
}

__device__ __forceinline__ uint16_t ld_stream_u16(const uint16_t* p, uint64_t pol) {
    uint16_t v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.b16 %0, [%1], %2;"
                 : "=h"(v) : "l"(p), "l"(pol));
    return v;
}

// Loads and stores of the buffered records, marked evict-last in L2: the
// later steps of the window read them again, while the checkpoint stream
// (evict-first) passes through.
__device__ __forceinline__ uint2 ld_keep_u2(const void* p, uint64_t pol) {
    uint2 v;
    asm volatile("ld.global.nc.L2::cache_hint.v2.b32 {%0,%1}, [%2], %3;" : "=r"(v.x), "=r"(v.y) : "l"(p), "l"(pol));
    return v;
}
__device__ __forceinline__ float4 ld_keep_f4(const void* p, uint64_t pol) {
    float4 v;
    asm volatile("ld.global.nc.L2::cache_hint.v4.f32 {%0,%1,%2,%3}, [%4], %5;"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "l"(p), "l"(pol));
    return v;
}
__device__ __forceinline__ uint32_t ld_keep_u32(const void* p, uint64_t pol) {
    uint32_t v;
    asm volatile("ld.global.nc.L2::cache_hint.b32 %0, [%1], %2;" : "=r"(v) : "l"(p), "l"(pol));
    return v;
}
__device__ __forceinline__ uint32_t ld_keep_u16(const void* p, uint64_t pol) {
    uint16_t v;
    asm volatile("ld.global.nc.L2::cache_hint.b16 %0, [%1], %2;" : "=h"(v) : "l"(p), "l"(pol));
    return v;
}
__device__ __forceinline__ void st_keep_v4(void* p, uint4 v, uint64_t pol) {
    asm volatile("st.global.L2::cache_hint.v4.b32 [%0], {%1,%2,%3,%4}, %5;"
                 ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w), "l"(pol) : "memory");
}
__device__ __forceinline__ void st_keep_u32(void* p, uint32_t v, uint64_t pol) {
    asm volatile("st.global.L2::cache_hint.b32 [%0], %1, %2;" ::"l"(p), "r"(v), "l"(pol) : "memory");
}
__device__ __forceinline__ void st_keep_u16(void* p, uint32_t v, uint64_t pol) {
    asm volatile("st.global.L2::cache_hint.b16 [%0], %1, %2;" ::"l"(p), "h"(static_cast<uint16_t>(v)), "l"(pol)
                 : "memory");
}

__device__ __forceinline__ float to_f(float v) { return v; }
__device__ __forceinline__ float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }

template <typename T> __device__ __forceinline__ T from_f(float v);
template <> __device__ __forceinline__ float from_f<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float v) {
    return __float2bfloat16_rn(v);
}

// Four consecutive elements (16-byte aligned for float, 8-byte for bf16).
__device__ __forceinline__ float4 load4(const float* p) {
    return *reinterpret_cast<const float4*>(p);
}
__device__ __forceinline__ float4 load4(const __nv_bfloat16* p) {
    uint2 u = *reinterpret_cast<const uint2*>(p);
    float4 r;
    r.x = __uint_as_float(u.x << 16);
    r.y = __uint_as_float(u.x & 0xFFFF0000u);
    r.z = __uint_as_float(u.y << 16);
    r.w = __uint_as_float(u.y & 0xFFFF0000u);
    return r;
}

__device__ __forceinline__ float dot4(float4 a, float4 b) {
    return a.x * b.x + a.y * b.y + a.z * b.z + a.w * b.w;
}

// --------------------------------------------------------------------------
// Warp reductions
// --------------------------------------------------------------------------
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

template <int X> struct Log2 { static constexpr int value = 1 + Log2<X / 2>::value; };
template <> struct Log2<1> { static constexpr int value = 0; };

// Sum V per-lane values over groups of W adjacent lanes (V <= W <= 32, both
// powers of two) with V-1 + log2(W/V) shuffles instead of V*log2(W): each step
// halves the values a lane keeps and swaps the other half with its partner.
// On return, lane l holds the group-wide sum of value index
// (l % W) >> log2(W/V).
template <int V, int W>
__device__ __forceinline__ float group_reduce_multi(float (&v)[V], int lane) {
    static_assert(V >= 1 && V <= W && W <= 32, "bad reduction shape");
#pragma unroll
    for (int s = V / 2, off = W / 2; s >= 1; s >>= 1, off >>= 1) {
        const bool upper = (lane & off) != 0;
#pragma unroll
        for (int i = 0; i < s; ++i) {
            float send = upper ? v[i] : v[i + s];
            float keep = upper ? v[i + s] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
        }
    }
    float r = v[0];
#pragma unroll
    for (int off = W / (2 * V); off >= 1; off >>= 1) r += __shfl_xor_sync(0xffffffffu, r, off);
    return r;
}

// FP16 checkpoint values: 4 halves <-> float4 (exact widening; narrowing
// rounds to nearest even).
__device__ __forceinline__ float4 f16x4_to_f32(uint2 u) {
    const float2 lo = __half22float2(*reinterpret_cast<const __half2*>(&u.x));
    const float2 hi = __half22float2(*reinterpret_cast<const __half2*>(&u.y));
    return make_float4(lo.x, lo.y, hi.x, hi.y);
}
__device__ __forceinline__ uint2 f32_to_f16x4(float4 v) {
    const __half2 lo = __floats2half2_rn(v.x, v.y), hi = __floats2half2_rn(v.z, v.w);
    return make_uint2(*reinterpret_cast<const uint32_t*>(&lo), *reinterpret_cast<const uint32_t*>(&hi));
}

// --------------------------------------------------------------------------
// mbarrier + bulk async copy (TMA, non-tensor) and bounded waits
// --------------------------------------------------------------------------
constexpr uint64_t kWaitLimitNs = 1000000000ull;  // 1 s: far above any normal stage latency

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

// Make barrier initialisation visible to the async (bulk copy) proxy.
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
                 ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
    return ok != 0;
}

// Wait for the phase with the given parity to complete, for at most
// limit_ns (kWaitLimitNs in the kernels). Returns false on timeout; the caller
// reports it and stops.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  uint64_t limit_ns = kWaitLimitNs) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() - t0 > limit_ns) return false;
    }
    return true;
}

// Bulk copy global -> shared (16-byte aligned addresses, size a multiple of
// 16), completing `bytes` of the barrier's transaction count.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void bulk_g2s_hint(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                              uint64_t pol) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;"
        ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(pol) : "memory");
}

// Named barrier for a subset of the block's warps (ids 1..15).
__device__ __forceinline__ void named_sync(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// --------------------------------------------------------------------------
// Device error word: err[0] first code, err[1] count, err[2] tile, err[3] value
// --------------------------------------------------------------------------
__device__ __forceinline__ void report_error(int32_t* err, int code, int tile, int value) {
    if (atomicCAS(err, 0, code) == 0) {
        err[2] = tile;
        err[3] = value;
    }
    atomicAdd(err + 1, 1);
}

// --------------------------------------------------------------------------
// FP8 E4M3 / FP4 E2M1 codecs (hardware conversions: round to nearest even,
// saturate to the largest finite value)
// --------------------------------------------------------------------------
// Two floats -> two E4M3 codes, lo in bits 0..7 and hi in bits 8..15.
__device__ __forceinline__ uint16_t e4m3x2(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// Two floats -> two E2M1 codes, lo in bits 0..3 and hi in bits 4..7.
__device__ __forceinline__ uint32_t e2m1x2(float lo, float hi) {
    uint32_t r;
    asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u32.u8 %0, t;\n\t}"
        : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// Two E4M3 codes (bits 0..7, 8..15) -> two floats (exact).
__device__ __forceinline__ float2 e4m3x2_to_f2(uint16_t c) {
    uint32_t h2;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(c));
    __half2 h = *reinterpret_cast<__half2*>(&h2);
    return __half22float2(h);
}

// Two E2M1 codes (bits 0..3, 4..7 of the low byte) -> two floats (exact).
__device__ __forceinline__ float2 e2m1x2_to_f2(uint32_t c) {
    uint32_t h2;
    asm("{\n\t.reg .b8 t;\n\tcvt.u8.u32 t, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}"
        : "=r"(h2) : "r"(c));
    __half2 h = *reinterpret_cast<__half2*>(&h2);
    return __half22float2(h);
}

__device__ __forceinline__ float e4m3_to_f(uint32_t c) {
    return e4m3x2_to_f2(static_cast<uint16_t>(c & 0xFF)).x;
}

}  // namespace rssm

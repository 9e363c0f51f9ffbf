// Gated DeltaNet decode kernels: the fold kernel (explicit flush) and the
// conventional step. The one-token replay step is in gdn_replay_tma.cu.
//
// Recurrence per (sequence, head), S in R^{d_v x d_k}:
//   S_t = alpha_t S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,  o_t = S_t (scale q_t)
// ("ReplaySSM beschleunigt ...", section "Wichtige Details" names Gated
// DeltaNet; "NVIDIA ve Dao AI Lab, ... ReplaySSM'i sundu", section "Durum
// trafigini azaltma ve rollback'in basitlestirilmesi": output-only
// evaluation, the intermediate state formed by two small matrix products).
//
// Window algebra. Records i = 0..c since the checkpoint S0 (record c is the
// current token). With gamma_i = prod_{l<=i} alpha_l, the state after record i is
//   S_i = gamma_i S0 + sum_{j<=i} (gamma_i/gamma_j) u_j k_j^T,
// where the rows u_j of U = T (V - diag(gamma) K S0^T),
// T = (I + diag(beta) A)^{-1} diag(beta), A[i][j] = (gamma_i/gamma_j)(k_i.k_j) (j<i),
// follow by forward substitution:
//   u_c = beta_c (v_c - gamma_c S0 k_c - sum_{j<c} (gamma_c/gamma_j)(k_j.k_c) u_j).
// Row u_j depends only on S0 and records <= j, so it is solved once, when
// token j arrives, and kept in the record in place of (v_j, beta_j). Each step
// then needs the two products S0 [k_c ; q_c] and the masked (q K^T) U:
//   o_c = gamma_c S0 q + sum_{j<c} (gamma_c/gamma_j)(k_j.q) u_j + (k_c.q) u_c.
// The flush folds the window: S0 <- gamma_c S0 + sum_{j<=c} (gamma_c/gamma_j) u_j k_j^T.
#include "tile.cuh"

namespace rssm {
namespace {

__device__ __forceinline__ float4 scale4(float4 v, float s) {
    return make_float4(v.x * s, v.y * s, v.z * s, v.w * s);
}

// ---------------------------------------------------------------------------
// Commit after drafts, and the explicit flush: c <- c + a_b; a tile whose new
// count m reaches k (every tile with m > 0 when forced) folds its records,
// S0 <- gamma S0 + sum_{j<m} rho_j u_j k_j^T, and resets c.
// ---------------------------------------------------------------------------
// F16: the checkpoint is stored in FP16, widened on load and rounded once on
// the store.
template <class L, typename TI, bool F16>
__global__ void __launch_bounds__(L::kThreads) gdn_commit_kernel(const GDNArgs a) {
    constexpr int DV = L::P, DK = L::N, kThreads = L::kThreads;
    extern __shared__ float dsm[];
    __shared__ float s_rho[kMaxCap];
    __shared__ float s_gamma;

    const int tile = blockIdx.x;
    const int b = tile / a.H, hh = tile - b * a.H;
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const int col4 = t % L::TPR, row0 = t / L::TPR;
    const int c = a.counts[tile];
    if (c < 0 || c > a.cap) {
        if (t == 0) report_error(a.err, RSSM_DEV_COUNT_RANGE, tile, c);
        return;
    }
    // after drafts: the pointer moves past the accepted ones (rejected drafts
    // are dropped by that move alone)
    int acc = 0;
    if (a.accepted != nullptr) {
        acc = a.accepted[b];
        if (acc < 0 || acc > a.T || c + acc > a.cap) {
            if (t == 0 && hh == 0) report_error(a.err, RSSM_DEV_ACCEPTED_RANGE, b, acc);
            acc = 0;
        }
    }
    const int m = c + acc;
    const bool fold = a.force ? (m > 0) : (m >= a.kflush);
    if (!fold) {
        if (t == 0 && acc != 0) a.counts[tile] = m;
        return;
    }

    const size_t tile_off = static_cast<size_t>(tile) * DV * DK;
    uint2* ck16 = reinterpret_cast<uint2*>(reinterpret_cast<__half*>(a.ckpt) + tile_off);
    float4 hv[8];
    if constexpr (F16) {
#pragma unroll
        for (int j = 0; j < 8; ++j) hv[j] = f16x4_to_f32(ck16[(row0 + j * L::RPP) * L::TPR + col4]);
    } else {
        load_state<L>(hv, a.ckpt + tile_off, row0, col4, l2_evict_first());
    }
    auto store = [&]() {
        if constexpr (F16) {
#pragma unroll
            for (int j = 0; j < 8; ++j) ck16[(row0 + j * L::RPP) * L::TPR + col4] = f32_to_f16x4(hv[j]);
        } else {
            store_state<L>(hv, a.ckpt + tile_off, row0, col4);
        }
    };
    const TI* bk = reinterpret_cast<const TI*>(a.buf_k) + static_cast<size_t>(tile) * a.cap * DK;
    const float* bu = a.buf_u + static_cast<size_t>(tile) * a.cap * DV;
    const float* ba = a.buf_a + static_cast<size_t>(tile) * a.cap;
    if (a.rf != RSSM_READ_NONE) {
        // with a read copy the stored u rows were formed from the copy: replay
        // the records (k, v, alpha, beta) through the recurrence instead,
        //   S <- alpha S + beta (v - alpha S k) k^T
        float* s_u = dsm;   // [DV]
        const TI* bv = reinterpret_cast<const TI*>(a.buf_v) + static_cast<size_t>(tile) * (DV / 64) * a.cap * 64;
        const float* bb = a.buf_beta + static_cast<size_t>(tile) * a.cap;
        for (int j = 0; j < m; ++j) {
            const float al = ba[j], be = bb[j];
            const float4 kv = load4(bk + j * DK + col4 * 4);
            float part[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) part[i] = dot4(hv[i], kv);
            row_dots<L>(part, lane, row0, [&](int r, float sk) {
                s_u[r] = be * (to_f(bv[((r / 64) * a.cap + j) * 64 + (r % 64)]) - al * sk);
            });
            __syncthreads();
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float u = s_u[row0 + i * L::RPP];
                hv[i].x = fmaf(al, hv[i].x, u * kv.x);
                hv[i].y = fmaf(al, hv[i].y, u * kv.y);
                hv[i].z = fmaf(al, hv[i].z, u * kv.z);
                hv[i].w = fmaf(al, hv[i].w, u * kv.w);
            }
            __syncthreads();   // s_u is rewritten by the next record
        }
        store();
        if (t == 0) a.counts[tile] = 0;
        return;
    }
    if (warp == 0) {
        float gamma;
        const float rho = window_rho((lane < m) ? ba[lane] : 1.f, lane, m, gamma);
        if (lane < m) s_rho[lane] = rho;
        if (lane == 0) s_gamma = gamma;
    }
    __syncthreads();
    float* sK = dsm;
    float* sU = dsm + a.cap * DK;
    for (int idx = t; idx < m * DK; idx += kThreads) sK[idx] = to_f(bk[idx]);
    // u records are stored per 64-row half: [DV/64][cap][64]
    for (int idx = t; idx < m * DV; idx += kThreads) {
        const int j = idx / DV, r = idx - j * DV;
        sU[idx] = s_rho[j] * bu[(static_cast<size_t>(r / 64) * a.cap + j) * 64 + (r % 64)];
    }
    __syncthreads();
    fold_records<L>(hv, sK, sU, m, s_gamma, row0, col4);
    store();
    if (t == 0) a.counts[tile] = 0;
}

// ---------------------------------------------------------------------------
// Conventional step (the in-build baseline): read S, u = beta (v - alpha S k),
// S <- alpha S + u k^T, o = S (scale q), write S.
// ---------------------------------------------------------------------------
template <class L, typename TI>
__global__ void __launch_bounds__(L::kThreads)
gdn_conv_step_kernel(const GDNArgs a, const int out_f32) {
    constexpr int DV = L::P, DK = L::N, kThreads = L::kThreads;
    __shared__ float s_u[DV];
    const int tile = blockIdx.x;
    const int b = tile / a.H, hh = tile - b * a.H;
    const int t = threadIdx.x, lane = t & 31;
    const int col4 = t % L::TPR, row0 = t / L::TPR;
    const size_t tile_off = static_cast<size_t>(tile) * DV * DK;

    float4 hv[8];
    load_state<L>(hv, a.ckpt + tile_off, row0, col4, l2_evict_first());
    const size_t bh = static_cast<size_t>(b) * a.H + hh;
    const TI* qt = reinterpret_cast<const TI*>(a.q) + bh * DK;
    const TI* kt = reinterpret_cast<const TI*>(a.k) + bh * DK;
    const TI* vt = reinterpret_cast<const TI*>(a.v) + bh * DV;
    const float al = a.alpha[bh], be = a.beta[bh];
    const float4 kv = load4(kt + col4 * 4);
    const float4 qv = scale4(load4(qt + col4 * 4), a.scale);

    float part[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) part[j] = dot4(hv[j], kv);
    row_dots<L>(part, lane, row0, [&](int r, float sk) {
        s_u[r] = be * (to_f(vt[r]) - al * sk);
    });
    __syncthreads();
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const float u = s_u[row0 + j * L::RPP];
        hv[j].x = fmaf(al, hv[j].x, u * kv.x);
        hv[j].y = fmaf(al, hv[j].y, u * kv.y);
        hv[j].z = fmaf(al, hv[j].z, u * kv.z);
        hv[j].w = fmaf(al, hv[j].w, u * kv.w);
        part[j] = dot4(hv[j], qv);
    }
    store_state<L>(hv, a.ckpt + tile_off, row0, col4);
    row_dots<L>(part, lane, row0, [&](int r, float v) { store_out(a.o, bh * DV + r, v, out_f32 != 0); });
    (void)kThreads;
}

// ---------------------------------------------------------------------------
// Quantised-recurrence baseline ("NVIDIA ve Dao AI Lab, ... ReplaySSM'i sundu",
// section "Kuantizasyon hatasinin sinirlandirilmasi"): the state itself lives
// in the read-copy tile format, one copy tile per 64-row half. Each token
// dequantises it, runs the conventional step in FP32, writes the output and
// re-quantises the updated state in place (the read-copy writer's format and
// rounding). It is the comparison point for the read copy, whose recurrence
// stays on the FP32 checkpoint.
// ---------------------------------------------------------------------------
template <class L, typename TI, int RF>
__global__ void __launch_bounds__(L::kThreads)
gdn_qconv_step_kernel(const GDNArgs a, const int out_f32) {
    constexpr int DV = L::P, DK = L::N, J = 8;
    constexpr int HALVES = DV / 64, JH = J / HALVES;   // a thread's values per half (rows row0 + j RPP)
    static_assert(64 % L::RPP == 0 && L::RPP * JH == 64, "half split");
    __shared__ float s_u[DV];
    __shared__ float s_red[L::kWarps];
    const int tile = blockIdx.x;
    const int b = tile / a.H, hh = tile - b * a.H;
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const int col4 = t % L::TPR, row0 = t / L::TPR;
    const size_t half_elems = static_cast<size_t>(64) * DK;

    // dequantise this thread's values: code x (block scale x) half scale
    float4 hv[J];
#pragma unroll
    for (int hf = 0; hf < HALVES; ++hf) {
        const size_t ht = static_cast<size_t>(tile) * HALVES + hf;
        const uint8_t* codes = a.rc_codes + (RF == RSSM_READ_FP8 ? ht * half_elems : ht * half_elems / 2);
        const uint8_t* bsc = (RF == RSSM_READ_NVFP4) ? a.rc_bscale + ht * half_elems / 16 : nullptr;
        const float ts = a.rc_tscale[ht];
#pragma unroll
        for (int jj = 0; jj < JH; ++jj) {
            const int row = row0 + jj * L::RPP;   // within the half
            const int idx = row * L::TPR + col4;
            float4& h = hv[hf * JH + jj];
            if (RF == RSSM_READ_FP8) {
                const uint32_t u = reinterpret_cast<const uint32_t*>(codes)[idx];
                const float2 lo = e4m3x2_to_f2(static_cast<uint16_t>(u & 0xFFFFu));
                const float2 hi = e4m3x2_to_f2(static_cast<uint16_t>(u >> 16));
                h = make_float4(lo.x * ts, lo.y * ts, hi.x * ts, hi.y * ts);
            } else {
                const uint32_t u = reinterpret_cast<const uint16_t*>(codes)[idx];
                const float es = __fmul_rn(e4m3_to_f(bsc[row * (DK / 16) + (col4 >> 2)]), ts);
                const float2 lo = e2m1x2_to_f2(u & 0xFFu);
                const float2 hi = e2m1x2_to_f2((u >> 8) & 0xFFu);
                h = make_float4(lo.x * es, lo.y * es, hi.x * es, hi.y * es);
            }
        }
    }

    // the conventional step on the decoded values
    const size_t bh = static_cast<size_t>(b) * a.H + hh;
    const TI* qt = reinterpret_cast<const TI*>(a.q) + bh * DK;
    const TI* kt = reinterpret_cast<const TI*>(a.k) + bh * DK;
    const TI* vt = reinterpret_cast<const TI*>(a.v) + bh * DV;
    const float al = a.alpha[bh], be = a.beta[bh];
    const float4 kv = load4(kt + col4 * 4);
    const float4 qv = scale4(load4(qt + col4 * 4), a.scale);
    float part[J];
#pragma unroll
    for (int j = 0; j < J; ++j) part[j] = dot4(hv[j], kv);
    row_dots<L>(part, lane, row0, [&](int r, float sk) {
        s_u[r] = be * (to_f(vt[r]) - al * sk);
    });
    __syncthreads();
#pragma unroll
    for (int j = 0; j < J; ++j) {
        const float u = s_u[row0 + j * L::RPP];
        hv[j].x = fmaf(al, hv[j].x, u * kv.x);
        hv[j].y = fmaf(al, hv[j].y, u * kv.y);
        hv[j].z = fmaf(al, hv[j].z, u * kv.z);
        hv[j].w = fmaf(al, hv[j].w, u * kv.w);
        part[j] = dot4(hv[j], qv);
    }
    row_dots<L>(part, lane, row0, [&](int r, float v) { store_out(a.o, bh * DV + r, v, out_f32 != 0); });

    // re-quantise each half in place: every thread has read its codes and
    // scales before the writer's first barrier
#pragma unroll
    for (int hf = 0; hf < HALVES; ++hf) {
        const size_t ht = static_cast<size_t>(tile) * HALVES + hf;
        uint8_t* codes = a.rc_codes + (RF == RSSM_READ_FP8 ? ht * half_elems : ht * half_elems / 2);
        uint8_t* bsc = (RF == RSSM_READ_NVFP4) ? a.rc_bscale + ht * half_elems / 16 : nullptr;
        write_read_copy<L, RF>(reinterpret_cast<float4(&)[JH]>(hv[hf * JH]), codes, bsc, a.rc_tscale + ht, s_red,
                               t, lane, warp, [&](int jj) { return row0 + jj * L::RPP; }, [&](int) { return col4; },
                               [] { __syncthreads(); });
    }
}

// ---------------------------------------------------------------------------
// Snapshot baseline for drafts ("Wie es funktioniert", 2nd paragraph: the
// state snapshots per draft token that replay removes): T conventional steps
// from the live state, each writing a full-state snapshot and its output;
// the live state itself is not written.
// ---------------------------------------------------------------------------
template <class L, typename TI>
__global__ void __launch_bounds__(L::kThreads)
gdn_snap_draft_kernel(const GDNArgs a, const int out_f32) {
    constexpr int DV = L::P, DK = L::N;
    __shared__ float s_u[DV];
    const int tile = blockIdx.x;
    const int b = tile / a.H, hh = tile - b * a.H;
    const int t = threadIdx.x, lane = t & 31;
    const int col4 = t % L::TPR, row0 = t / L::TPR;
    const int T = a.T;
    const size_t tile_off = static_cast<size_t>(tile) * DV * DK;
    const size_t state_elems = static_cast<size_t>(a.B) * a.H * DV * DK;

    float4 hv[8];
    load_state<L>(hv, a.ckpt + tile_off, row0, col4, l2_evict_first());
    for (int tau = 0; tau < T; ++tau) {
        const size_t bth = (static_cast<size_t>(b) * T + tau) * a.H + hh;
        const TI* qt = reinterpret_cast<const TI*>(a.q) + bth * DK;
        const TI* kt = reinterpret_cast<const TI*>(a.k) + bth * DK;
        const TI* vt = reinterpret_cast<const TI*>(a.v) + bth * DV;
        const float al = a.alpha[bth], be = a.beta[bth];
        const float4 kv = load4(kt + col4 * 4);
        const float4 qv = scale4(load4(qt + col4 * 4), a.scale);
        float part[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) part[j] = dot4(hv[j], kv);
        __syncthreads();   // s_u of the previous draft has been read
        row_dots<L>(part, lane, row0, [&](int r, float sk) { s_u[r] = be * (to_f(vt[r]) - al * sk); });
        __syncthreads();
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float u = s_u[row0 + j * L::RPP];
            hv[j].x = fmaf(al, hv[j].x, u * kv.x);
            hv[j].y = fmaf(al, hv[j].y, u * kv.y);
            hv[j].z = fmaf(al, hv[j].z, u * kv.z);
            hv[j].w = fmaf(al, hv[j].w, u * kv.w);
            part[j] = dot4(hv[j], qv);
        }
        store_state<L>(hv, a.snap + tau * state_elems + tile_off, row0, col4);
        row_dots<L>(part, lane, row0, [&](int r, float v) { store_out(a.o, bth * DV + r, v, out_f32 != 0); });
    }
}

// Snapshot restore: live state <- snapshot a_b (the state after a_b drafts).
template <class L>
__global__ void __launch_bounds__(L::kThreads) gdn_snap_restore_kernel(const GDNArgs a) {
    constexpr int DV = L::P, DK = L::N;
    const int tile = blockIdx.x;
    const int b = tile / a.H, hh = tile - b * a.H;
    const int t = threadIdx.x;
    const int acc = a.accepted[b];
    if (acc < 0 || acc > a.T) {
        if (t == 0 && hh == 0) report_error(a.err, RSSM_DEV_ACCEPTED_RANGE, b, acc);
        return;
    }
    if (acc == 0) return;
    const size_t state_elems = static_cast<size_t>(a.B) * a.H * DV * DK;
    const size_t tile_off = static_cast<size_t>(tile) * DV * DK;
    const float4* src = reinterpret_cast<const float4*>(a.snap + (acc - 1) * state_elems + tile_off);
    float4* dst = reinterpret_cast<float4*>(a.ckpt + tile_off);
    const uint64_t pol = l2_evict_first();
#pragma unroll
    for (int j = 0; j < 8; ++j) dst[t + j * L::kThreads] = ld_stream(src + t + j * L::kThreads, pol);
}

template <class K, class... Args>
cudaError_t launch(K kernel, int grid, int block, size_t smem, cudaStream_t s, Args... args) {
    if (grid == 0) return cudaSuccess;
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
        if (e != cudaSuccess) return e;
    }
    kernel<<<grid, block, smem, s>>>(args...);
    return cudaGetLastError();
}

template <template <class> class F, class... Args>
cudaError_t with_tile(int DV, int DK, bool* supported, Args&&... args) {
    *supported = true;
    if (DV == 128 && DK == 128) return F<Tile<128, 128>>::run(args...);
    if (DV == 64 && DK == 64) return F<Tile<64, 64>>::run(args...);
    if (DV == 64 && DK == 128) return F<Tile<64, 128>>::run(args...);
    if (DV == 128 && DK == 64) return F<Tile<128, 64>>::run(args...);
    *supported = false;
    return cudaSuccess;
}

template <class L> struct CommitF {
    static cudaError_t run(const GDNArgs& a, int in_dt, cudaStream_t s) {
        const size_t smem = static_cast<size_t>(a.cap) * (L::P + L::N) * sizeof(float);   // >= P floats
        if (a.ck == kCkF16) {
            if (in_dt != RSSM_BF16) return cudaErrorInvalidValue;
            return launch(gdn_commit_kernel<L, __nv_bfloat16, true>, a.B * a.H, L::kThreads, smem, s, a);
        }
        if (in_dt == RSSM_F32) return launch(gdn_commit_kernel<L, float, false>, a.B * a.H, L::kThreads, smem, s, a);
        return launch(gdn_commit_kernel<L, __nv_bfloat16, false>, a.B * a.H, L::kThreads, smem, s, a);
    }
};

template <class L> struct ConvF {
    static cudaError_t run(const GDNArgs& a, int in_dt, int out_dt, cudaStream_t s) {
        const int of = (out_dt == RSSM_F32);
        const int grid = a.B * a.H;
        if (in_dt == RSSM_F32) {
            if (a.rf == RSSM_READ_FP8) return launch(gdn_qconv_step_kernel<L, float, RSSM_READ_FP8>, grid, L::kThreads, 0, s, a, of);
            if (a.rf == RSSM_READ_NVFP4) return launch(gdn_qconv_step_kernel<L, float, RSSM_READ_NVFP4>, grid, L::kThreads, 0, s, a, of);
            return launch(gdn_conv_step_kernel<L, float>, grid, L::kThreads, 0, s, a, of);
        }
        if (a.rf == RSSM_READ_FP8) return launch(gdn_qconv_step_kernel<L, __nv_bfloat16, RSSM_READ_FP8>, grid, L::kThreads, 0, s, a, of);
        if (a.rf == RSSM_READ_NVFP4) return launch(gdn_qconv_step_kernel<L, __nv_bfloat16, RSSM_READ_NVFP4>, grid, L::kThreads, 0, s, a, of);
        return launch(gdn_conv_step_kernel<L, __nv_bfloat16>, grid, L::kThreads, 0, s, a, of);
    }
};

template <class L> struct SnapDraftF {
    static cudaError_t run(const GDNArgs& a, int in_dt, int out_dt, cudaStream_t s) {
        const int of = (out_dt == RSSM_F32);
        if (in_dt == RSSM_F32) return launch(gdn_snap_draft_kernel<L, float>, a.B * a.H, L::kThreads, 0, s, a, of);
        return launch(gdn_snap_draft_kernel<L, __nv_bfloat16>, a.B * a.H, L::kThreads, 0, s, a, of);
    }
};

template <class L> struct SnapRestoreF {
    static cudaError_t run(const GDNArgs& a, cudaStream_t s) {
        return launch(gdn_snap_restore_kernel<L>, a.B * a.H, L::kThreads, 0, s, a);
    }
};

}  // namespace

cudaError_t gdn_snap_draft(const GDNArgs& a, int DV, int DK, int in_dt, int out_dt, cudaStream_t s,
                           bool* supported) {
    return with_tile<SnapDraftF>(DV, DK, supported, a, in_dt, out_dt, s);
}
cudaError_t gdn_snap_restore(const GDNArgs& a, int DV, int DK, cudaStream_t s, bool* supported) {
    return with_tile<SnapRestoreF>(DV, DK, supported, a, s);
}

cudaError_t gdn_commit(const GDNArgs& a, int DV, int DK, int in_dt, cudaStream_t s, bool* supported) {
    return with_tile<CommitF>(DV, DK, supported, a, in_dt, s);
}
cudaError_t gdn_conv_step(const GDNArgs& a, int DV, int DK, int in_dt, int out_dt, cudaStream_t s,
                          bool* supported) {
    return with_tile<ConvF>(DV, DK, supported, a, in_dt, out_dt, s);
}

}  // namespace rssm

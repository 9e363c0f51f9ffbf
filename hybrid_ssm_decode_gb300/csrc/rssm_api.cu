// C ABI of librssm (declared in include/rssm.h): argument validation,
// workspace layout, the host handle, and kernel dispatch. Every entry point
// returns a status and never throws; all device work goes to the caller's
// stream, on the caller's memory.
#include <cstdlib>
#include <cstring>
#include <new>

#include "common.cuh"

using namespace rssm;

namespace {

// One thread waits on an mbarrier that nothing arrives at, with the pipelined
// kernels' bounded wait, and records the timeout as they do.
__global__ void bounded_wait_check_kernel(uint64_t limit_ns, int32_t* err) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x != 0) return;
    mbar_init(&bar, 1);
    fence_mbar_init();
    const uint64_t t0 = globaltimer_ns();
    if (!mbar_wait_bounded(&bar, 0, limit_ns)) {
        const uint64_t waited = globaltimer_ns() - t0;
        report_error(err, kDevTimeout, -1, waited > 0x7FFFFFFFull ? 0x7FFFFFFF : static_cast<int>(waited));
    }
}

// Tiles per record count: entry c (0..kMaxCap) counts tiles holding c
// records, entry kMaxCap + 1 those outside that range. One block; lanes with
// the same count add once per warp.
__global__ void count_hist_kernel(const int32_t* __restrict__ counts, int n, int32_t* __restrict__ hist) {
    __shared__ int sh[kMaxCap + 2];
    for (int i = threadIdx.x; i < kMaxCap + 2; i += blockDim.x) sh[i] = 0;
    __syncthreads();
    const int lane = threadIdx.x & 31;
    for (int64_t base = 0; base < n; base += blockDim.x) {
        const int64_t i = base + threadIdx.x;
        const bool in = i < n;
        int c = in ? counts[i] : -2;
        const int bin = (c >= 0 && c <= kMaxCap) ? c : (c == -2 ? -1 : kMaxCap + 1);
        const unsigned same = __match_any_sync(0xffffffffu, bin);
        if (bin >= 0 && lane == __ffs(same) - 1) atomicAdd(&sh[bin], __popc(same));
    }
    __syncthreads();
    for (int i = threadIdx.x; i < kMaxCap + 2; i += blockDim.x) hist[i] = sh[i];
}

}  // namespace

struct rssm_handle {
    rssm_config cfg;
    rssm_layout lay;
    char* base;
    const float* A;
    const float* D;
    int pending_T;     // drafts appended by the last decode_step, awaiting verify
    // Tiles per record count (0..kMaxCap), while the host knows them: after
    // create, a flush, a count summary from the device, and plain steps since.
    bool counts_known;
    int64_t hist[kMaxCap + 1];
    unsigned char image_hdr[256];   // header of this handle's state image
};

namespace {

constexpr size_t kAlign = 256;

size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool dims_supported(int rows, int cols) {
    return (rows == 64 || rows == 128) && (cols == 64 || cols == 128);
}

rssm_status check_config(const rssm_config* c) {
    if (c == nullptr) return RSSM_ERR_INVALID_ARG;
    if (c->kind != RSSM_MAMBA2 && c->kind != RSSM_GDN) return RSSM_ERR_INVALID_ARG;
    if (c->mode != RSSM_REPLAY && c->mode != RSSM_CONVENTIONAL) return RSSM_ERR_INVALID_ARG;
    if (c->batch < 1 || c->heads < 1 || c->head_dim < 1 || c->state_dim < 1)
        return RSSM_ERR_INVALID_ARG;
    if (c->in_dtype != RSSM_F32 && c->in_dtype != RSSM_BF16) return RSSM_ERR_INVALID_ARG;
    if (c->out_dtype != 0 && c->out_dtype != RSSM_F32 && c->out_dtype != RSSM_BF16)
        return RSSM_ERR_INVALID_ARG;
    if (c->read_fmt < RSSM_READ_NONE || c->read_fmt > RSSM_READ_NVFP4) return RSSM_ERR_INVALID_ARG;
    if (c->k < 1 || c->k > kMaxCap) return RSSM_ERR_INVALID_ARG;
    if (c->max_draft < 1) return RSSM_ERR_INVALID_ARG;
    if (c->kind == RSSM_MAMBA2 && (c->groups < 1 || c->heads % c->groups != 0))
        return RSSM_ERR_INVALID_ARG;
    if (static_cast<int64_t>(c->batch) * c->heads > 0x7FFFFFFF) return RSSM_ERR_INVALID_ARG;
    if (!dims_supported(c->head_dim, c->state_dim)) return RSSM_ERR_UNSUPPORTED;
    if (c->max_draft > kMaxDraft) return RSSM_ERR_UNSUPPORTED;
    if (c->mode == RSSM_REPLAY && c->k - 1 + c->max_draft > kMaxCap) return RSSM_ERR_UNSUPPORTED;
    // replay drafts read the copy; the snapshot baseline reads the live state
    if (c->read_fmt != RSSM_READ_NONE && c->max_draft != 1 && c->mode != RSSM_REPLAY) return RSSM_ERR_UNSUPPORTED;
    // a GDN read copy (REPLAY) takes bf16 inputs; CONVENTIONAL with a read
    // format is the quantised-recurrence baseline, either input dtype
    if (c->read_fmt != RSSM_READ_NONE && c->kind == RSSM_GDN && c->mode == RSSM_REPLAY && c->in_dtype != RSSM_BF16)
        return RSSM_ERR_UNSUPPORTED;
    if (c->ckpt_dtype != 0 && c->ckpt_dtype != RSSM_F32 && c->ckpt_dtype != RSSM_F16 &&
        c->ckpt_dtype != RSSM_CKPT_FP8 && c->ckpt_dtype != RSSM_CKPT_NVFP4)
        return RSSM_ERR_INVALID_ARG;
    const bool lowp = (c->ckpt_dtype != 0 && c->ckpt_dtype != RSSM_F32);
    if (lowp && (c->mode != RSSM_REPLAY || c->in_dtype != RSSM_BF16 || c->max_draft != 1))
        return RSSM_ERR_UNSUPPORTED;
    // GDN: an FP16 checkpoint without a read copy
    if (lowp && c->kind == RSSM_GDN && (c->ckpt_dtype != RSSM_F16 || c->read_fmt != RSSM_READ_NONE))
        return RSSM_ERR_UNSUPPORTED;
    // a tile-format checkpoint is read itself, or through an NVFP4 copy of an FP8 one
    if (c->ckpt_dtype == RSSM_CKPT_FP8 && c->read_fmt == RSSM_READ_FP8) return RSSM_ERR_UNSUPPORTED;
    if (c->ckpt_dtype == RSSM_CKPT_NVFP4 && c->read_fmt != RSSM_READ_NONE) return RSSM_ERR_UNSUPPORTED;
    return RSSM_OK;
}

rssm_status make_layout(const rssm_config* c, rssm_layout* L) {
    rssm_status st = check_config(c);
    if (st != RSSM_OK) return st;
    std::memset(L, 0, sizeof(*L));
    const size_t B = c->batch, H = c->heads, R = c->head_dim, Cc = c->state_dim;
    const size_t tiles = B * H, elems = tiles * R * Cc;
    const size_t in_sz = (c->in_dtype == RSSM_F32) ? 4 : 2;
    const bool replay = (c->mode == RSSM_REPLAY);
    // records are bulk-copied per tile, so a tile's record arrays are whole
    // 16-byte units: the slot count is rounded up to a multiple of 8
    const size_t cap = replay ? round_up(static_cast<size_t>(c->k - 1 + c->max_draft), 8) : 0;
    size_t off = 0;
    auto take = [&](size_t bytes, size_t& o, size_t& sz) {
        o = bytes ? off : 0;
        sz = bytes;
        off += round_up(bytes, kAlign);
    };
    const size_t ck_bytes = (c->ckpt_dtype == RSSM_F16) ? elems * 2
                            : (c->ckpt_dtype == RSSM_CKPT_FP8) ? elems
                            : (c->ckpt_dtype == RSSM_CKPT_NVFP4) ? elems / 2 : elems * 4;
    take(ck_bytes, L->ckpt, L->ckpt_bytes);
    take(tiles * 4, L->counts, L->counts_bytes);
    take(16, L->err, L->err_bytes);
    if (replay && c->kind == RSSM_MAMBA2) {
        take(tiles * cap * R * in_sz, L->buf_x, L->buf_x_bytes);
        take(B * c->groups * cap * Cc * in_sz, L->buf_b, L->buf_b_bytes);
        take(tiles * cap * in_sz, L->buf_dt, L->buf_dt_bytes);
    }
    if (replay && c->kind == RSSM_GDN) {
        take(tiles * cap * Cc * in_sz, L->buf_k, L->buf_k_bytes);
        take(tiles * cap * R * 4, L->buf_u, L->buf_u_bytes);
        take(tiles * cap * 4, L->buf_a, L->buf_a_bytes);
    }
    // one copy tile per Mamba-2 tile, per 64-row half of a GDN tile
    const size_t ctiles = (c->kind == RSSM_GDN) ? tiles * (R / 64) : tiles;
    if (c->read_fmt == RSSM_READ_FP8) {
        take(elems, L->rc_codes, L->rc_codes_bytes);
        take(ctiles * 4, L->rc_tscale, L->rc_tscale_bytes);
    } else if (c->read_fmt == RSSM_READ_NVFP4) {
        take(elems / 2, L->rc_codes, L->rc_codes_bytes);
        take(elems / 16, L->rc_bscale, L->rc_bscale_bytes);
        take(ctiles * 4, L->rc_tscale, L->rc_tscale_bytes);
    }
    if (!replay && c->max_draft > 1) take(elems * 4 * c->max_draft, L->snap, L->snap_bytes);
    if (replay && c->kind == RSSM_GDN && c->read_fmt != RSSM_READ_NONE) {
        take(tiles * cap * R * in_sz, L->buf_v, L->buf_v_bytes);
        take(tiles * cap * 4, L->buf_beta, L->buf_beta_bytes);
    }
    if (c->ckpt_dtype == RSSM_CKPT_NVFP4) take(elems / 16, L->ckpt_bscale, L->ckpt_bscale_bytes);
    if (c->ckpt_dtype == RSSM_CKPT_FP8 || c->ckpt_dtype == RSSM_CKPT_NVFP4)
        take(tiles * 4, L->ckpt_tscale, L->ckpt_tscale_bytes);
    take((kMaxCap + 2) * 4, L->cnt_hist, L->cnt_hist_bytes);
    L->total_bytes = off;
    L->capacity = static_cast<int32_t>(cap);
    return RSSM_OK;
}

template <class T> T* region(const rssm_handle* h, size_t off, size_t bytes) {
    return bytes ? reinterpret_cast<T*>(h->base + off) : nullptr;
}

int out_dtype_of(const rssm_config& c) { return c.out_dtype ? c.out_dtype : c.in_dtype; }

M2Args m2_args(const rssm_handle* h) {
    M2Args a{};
    const rssm_layout& L = h->lay;
    a.ckpt = region<float>(h, L.ckpt, L.ckpt_bytes);
    a.counts = region<int32_t>(h, L.counts, L.counts_bytes);
    a.err = region<int32_t>(h, L.err, L.err_bytes);
    a.buf_x = region<void>(h, L.buf_x, L.buf_x_bytes);
    a.buf_b = region<void>(h, L.buf_b, L.buf_b_bytes);
    a.buf_dt = region<void>(h, L.buf_dt, L.buf_dt_bytes);
    a.rc_codes = region<uint8_t>(h, L.rc_codes, L.rc_codes_bytes);
    a.rc_bscale = region<uint8_t>(h, L.rc_bscale, L.rc_bscale_bytes);
    a.rc_tscale = region<float>(h, L.rc_tscale, L.rc_tscale_bytes);
    a.snap = region<float>(h, L.snap, L.snap_bytes);
    a.A = h->A;
    a.D = h->D;
    a.B = h->cfg.batch;
    a.H = h->cfg.heads;
    a.G = h->cfg.groups;
    a.k = h->cfg.k;
    a.cap = L.capacity;
    a.T = 1;
    const int cd = h->cfg.ckpt_dtype;
    a.ck = (cd == RSSM_F16) ? kCkF16 : (cd == RSSM_CKPT_FP8) ? kCkFP8 : (cd == RSSM_CKPT_NVFP4) ? kCkNVFP4 : kCkF32;
    a.ck_bscale = region<uint8_t>(h, L.ckpt_bscale, L.ckpt_bscale_bytes);
    a.ck_tscale = region<float>(h, L.ckpt_tscale, L.ckpt_tscale_bytes);
    if (ck_tile_fmt(a.ck) != RSSM_READ_NONE && h->cfg.read_fmt == RSSM_READ_NONE) {
        // the checkpoint is its own read copy
        a.rc_codes = reinterpret_cast<uint8_t*>(a.ckpt);
        a.rc_bscale = a.ck_bscale;
        a.rc_tscale = a.ck_tscale;
    }
    return a;
}

// The format the Mamba-2 non-flush reads use: the copy's, else that of a
// tile-format checkpoint, else none.
int m2_read_fmt(const rssm_config& c) {
    if (c.read_fmt != RSSM_READ_NONE) return c.read_fmt;
    if (c.ckpt_dtype == RSSM_CKPT_FP8) return RSSM_READ_FP8;
    if (c.ckpt_dtype == RSSM_CKPT_NVFP4) return RSSM_READ_NVFP4;
    return RSSM_READ_NONE;
}

GDNArgs gdn_args(const rssm_handle* h) {
    GDNArgs a{};
    const rssm_layout& L = h->lay;
    a.ckpt = region<float>(h, L.ckpt, L.ckpt_bytes);
    a.counts = region<int32_t>(h, L.counts, L.counts_bytes);
    a.err = region<int32_t>(h, L.err, L.err_bytes);
    a.buf_k = region<void>(h, L.buf_k, L.buf_k_bytes);
    a.buf_u = region<float>(h, L.buf_u, L.buf_u_bytes);
    a.buf_a = region<float>(h, L.buf_a, L.buf_a_bytes);
    a.rc_codes = region<uint8_t>(h, L.rc_codes, L.rc_codes_bytes);
    a.rc_bscale = region<uint8_t>(h, L.rc_bscale, L.rc_bscale_bytes);
    a.rc_tscale = region<float>(h, L.rc_tscale, L.rc_tscale_bytes);
    a.buf_v = region<void>(h, L.buf_v, L.buf_v_bytes);
    a.buf_beta = region<float>(h, L.buf_beta, L.buf_beta_bytes);
    a.snap = region<float>(h, L.snap, L.snap_bytes);
    a.rf = h->cfg.read_fmt;
    a.ck = (h->cfg.ckpt_dtype == RSSM_F16) ? kCkF16 : kCkF32;
    a.B = h->cfg.batch;
    a.H = h->cfg.heads;
    a.kflush = h->cfg.k;
    a.cap = L.capacity;
    a.T = 1;
    a.scale = (h->cfg.gdn_scale == 0.f) ? 1.f : h->cfg.gdn_scale;
    return a;
}

rssm_status cuda_status(cudaError_t e, bool supported) {
    if (!supported) return RSSM_ERR_UNSUPPORTED;
    return (e == cudaSuccess) ? RSSM_OK : RSSM_ERR_CUDA;
}

// ---- the host's knowledge of the record counts ----------------------------
void counts_all_zero(rssm_handle* h) {
    for (int c = 0; c <= kMaxCap; ++c) h->hist[c] = 0;
    h->hist[0] = static_cast<int64_t>(h->cfg.batch) * h->cfg.heads;
    h->counts_known = true;
}

int counts_max(const rssm_handle* h) {
    for (int c = kMaxCap; c >= 0; --c)
        if (h->hist[c]) return c;
    return 0;
}

int counts_min(const rssm_handle* h) {
    for (int c = 0; c <= kMaxCap; ++c)
        if (h->hist[c]) return c;
    return 0;
}

// How a one-token replay step runs, from what the host knows of the counts:
// the lean kernel alone when no tile completes its window; the step kernel
// alone when every tile does; otherwise (mixed or unknown counts) the lean
// kernel over the non-flush tiles and a second launch over the flush tiles.
enum StepPlan { kPlanLean, kPlanFused, kPlanSplit };

StepPlan step_plan(const rssm_handle* h) {
    if (!h->counts_known) return kPlanSplit;
    const int k = h->cfg.k;
    if (counts_max(h) + 1 < k) return kPlanLean;
    if (h->hist[k - 1] == static_cast<int64_t>(h->cfg.batch) * h->cfg.heads) return kPlanFused;
    return kPlanSplit;
}

// After a one-token step: every count grows by one, and the tiles that held
// k - 1 records flushed to 0.
void counts_after_step(rssm_handle* h) {
    if (!h->counts_known) return;
    const int k = h->cfg.k;
    const int64_t flushed = h->hist[k - 1];
    for (int c = k - 1; c >= 1; --c) h->hist[c] = h->hist[c - 1];
    h->hist[0] = flushed;
}

// Summary of the counts on the device -> the handle. Synchronises `s`.
cudaError_t counts_from_device(rssm_handle* h, cudaStream_t s) {
    int32_t* d_hist = reinterpret_cast<int32_t*>(h->base + h->lay.cnt_hist);
    const int n = h->cfg.batch * h->cfg.heads;
    count_hist_kernel<<<1, 1024, 0, s>>>(reinterpret_cast<const int32_t*>(h->base + h->lay.counts), n, d_hist);
    cudaError_t e = cudaGetLastError();
    int32_t hist[kMaxCap + 2];
    if (e == cudaSuccess) e = cudaMemcpyAsync(hist, d_hist, sizeof(hist), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) {
        h->counts_known = false;
        return e;
    }
    bool ok = hist[kMaxCap + 1] == 0;
    for (int c = h->cfg.k; c <= kMaxCap; ++c) ok = ok && hist[c] == 0;   // a count >= k is never kept
    for (int c = 0; c <= kMaxCap; ++c) h->hist[c] = hist[c];
    h->counts_known = ok;
    return cudaSuccess;
}

// ---- state image ------------------------------------------------------------
constexpr size_t kImageHdr = 256;
constexpr char kImageMagic[8] = {'R', 'S', 'S', 'M', 'S', 'T', 'A', 'T'};

struct ImageHdr {               // the first bytes of the 256-byte header
    char magic[8];
    int32_t abi_version;
    int32_t hdr_bytes;
    rssm_config cfg;
    uint64_t image_bytes;
};
static_assert(sizeof(ImageHdr) <= kImageHdr, "image header too large");

struct Region {
    size_t off, bytes;
};

// The state regions in image order (absent regions have 0 bytes).
int state_regions(const rssm_layout& L, Region* r) {
    const Region all[] = {{L.ckpt, L.ckpt_bytes},         {L.ckpt_bscale, L.ckpt_bscale_bytes},
                          {L.ckpt_tscale, L.ckpt_tscale_bytes}, {L.counts, L.counts_bytes},
                          {L.buf_x, L.buf_x_bytes},       {L.buf_b, L.buf_b_bytes},
                          {L.buf_dt, L.buf_dt_bytes},     {L.buf_k, L.buf_k_bytes},
                          {L.buf_u, L.buf_u_bytes},       {L.buf_a, L.buf_a_bytes},
                          {L.buf_v, L.buf_v_bytes},       {L.buf_beta, L.buf_beta_bytes},
                          {L.rc_codes, L.rc_codes_bytes}, {L.rc_bscale, L.rc_bscale_bytes},
                          {L.rc_tscale, L.rc_tscale_bytes}};
    int n = 0;
    for (const Region& x : all) r[n++] = x;
    return n;
}

size_t image_bytes(const rssm_layout& L) {
    Region r[16];
    const int n = state_regions(L, r);
    size_t total = kImageHdr;
    for (int i = 0; i < n; ++i) total += round_up(r[i].bytes, kAlign);
    return total;
}

void make_image_hdr(rssm_handle* h) {
    std::memset(h->image_hdr, 0, sizeof(h->image_hdr));
    ImageHdr hd;
    std::memset(&hd, 0, sizeof(hd));
    std::memcpy(hd.magic, kImageMagic, sizeof(hd.magic));
    hd.abi_version = RSSM_ABI_VERSION;
    hd.hdr_bytes = static_cast<int32_t>(kImageHdr);
    hd.cfg = h->cfg;
    hd.image_bytes = image_bytes(h->lay);
    std::memcpy(h->image_hdr, &hd, sizeof(hd));
}

// Copy every state region between the workspace and an image (to_image:
// workspace -> image).
cudaError_t copy_state(rssm_handle* h, char* image, bool to_image, cudaStream_t s) {
    Region r[16];
    const int n = state_regions(h->lay, r);
    size_t off = kImageHdr;
    cudaError_t e = cudaSuccess;
    for (int i = 0; i < n && e == cudaSuccess; ++i) {
        if (r[i].bytes == 0) continue;
        char* ws = h->base + r[i].off;
        e = to_image ? cudaMemcpyAsync(image + off, ws, r[i].bytes, cudaMemcpyDeviceToDevice, s)
                     : cudaMemcpyAsync(ws, image + off, r[i].bytes, cudaMemcpyDeviceToDevice, s);
        off += round_up(r[i].bytes, kAlign);
    }
    return e;
}

}  // namespace

namespace rssm {

// Per-device launch limits, queried once per device ordinal.
cudaError_t device_limits(int* num_sms, int* smem_optin) {
    constexpr int kMaxDevices = 64;
    static int sms[kMaxDevices], optin[kMaxDevices];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < kMaxDevices && sms[dev] > 0 && optin[dev] > 0) {
        *num_sms = sms[dev];
        *smem_optin = optin[dev];
        return cudaSuccess;
    }
    int a = 0, b = 0;
    e = cudaDeviceGetAttribute(&a, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&b, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < kMaxDevices) {
        optin[dev] = b;
        sms[dev] = a;
    }
    *num_sms = a;
    *smem_optin = b;
    return cudaSuccess;
}

}  // namespace rssm

extern "C" {

int32_t rssm_abi_version(void) { return RSSM_ABI_VERSION; }

const char* rssm_status_string(rssm_status s) {
    switch (s) {
        case RSSM_OK: return "ok";
        case RSSM_ERR_INVALID_ARG: return "invalid argument";
        case RSSM_ERR_UNSUPPORTED: return "unsupported configuration";
        case RSSM_ERR_CAPACITY: return "capacity exceeded";
        case RSSM_ERR_CUDA: return "CUDA error";
        case RSSM_ERR_STATE: return "call out of order";
    }
    return "unknown status";
}

rssm_status rssm_workspace_size(const rssm_config* cfg, size_t* bytes) {
    if (bytes == nullptr) return RSSM_ERR_INVALID_ARG;
    rssm_layout L;
    rssm_status st = make_layout(cfg, &L);
    if (st != RSSM_OK) return st;
    *bytes = L.total_bytes;
    return RSSM_OK;
}

rssm_status rssm_layout_for(const rssm_config* cfg, rssm_layout* out) {
    if (out == nullptr) return RSSM_ERR_INVALID_ARG;
    return make_layout(cfg, out);
}

rssm_status rssm_create(const rssm_config* cfg, void* d_workspace, size_t workspace_bytes,
                        const float* d_A, const float* d_D, const float* d_state0, void* stream,
                        rssm_handle** out) {
    if (out == nullptr) return RSSM_ERR_INVALID_ARG;
    *out = nullptr;
    rssm_layout L;
    rssm_status st = make_layout(cfg, &L);
    if (st != RSSM_OK) return st;
    if (d_workspace == nullptr || (reinterpret_cast<uintptr_t>(d_workspace) % kAlign) != 0)
        return RSSM_ERR_INVALID_ARG;
    if (workspace_bytes < L.total_bytes) return RSSM_ERR_CAPACITY;
    if (cfg->kind == RSSM_MAMBA2 && (d_A == nullptr || d_D == nullptr)) return RSSM_ERR_INVALID_ARG;
    if (d_state0 != nullptr && !aligned16(d_state0)) return RSSM_ERR_INVALID_ARG;

    rssm_handle* h = new (std::nothrow) rssm_handle;
    if (h == nullptr) return RSSM_ERR_CAPACITY;
    h->cfg = *cfg;
    h->lay = L;
    h->base = static_cast<char*>(d_workspace);
    h->A = d_A;
    h->D = d_D;
    h->pending_T = 0;
    counts_all_zero(h);
    make_image_hdr(h);

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaSuccess;
    const bool ck16 = (cfg->ckpt_dtype == RSSM_F16);
    const int ckf = (cfg->ckpt_dtype == RSSM_CKPT_FP8) ? RSSM_READ_FP8
                    : (cfg->ckpt_dtype == RSSM_CKPT_NVFP4) ? RSSM_READ_NVFP4 : RSSM_READ_NONE;
    const int64_t n_el = static_cast<int64_t>(cfg->batch) * cfg->heads * cfg->head_dim * cfg->state_dim;
    const int64_t n_tiles = static_cast<int64_t>(cfg->batch) * cfg->heads;
    if (d_state0 != nullptr && ck16) {
        e = f32_to_f16_array(d_state0, reinterpret_cast<__half*>(h->base + L.ckpt), n_el, s);
    } else if (d_state0 != nullptr && ckf != RSSM_READ_NONE) {
        bool sup = true;
        e = quantize_tiles(ckf, n_tiles, cfg->head_dim, cfg->state_dim, d_state0,
                           region<uint8_t>(h, L.ckpt, L.ckpt_bytes),
                           region<uint8_t>(h, L.ckpt_bscale, L.ckpt_bscale_bytes),
                           region<float>(h, L.ckpt_tscale, L.ckpt_tscale_bytes), s, &sup);
        if (!sup) {
            delete h;
            return RSSM_ERR_UNSUPPORTED;
        }
    } else if (d_state0 != nullptr) {
        e = cudaMemcpyAsync(h->base + L.ckpt, d_state0, L.ckpt_bytes, cudaMemcpyDeviceToDevice, s);
    } else {
        e = cudaMemsetAsync(h->base + L.ckpt, 0, L.ckpt_bytes, s);
        if (e == cudaSuccess && L.ckpt_bscale_bytes) e = cudaMemsetAsync(h->base + L.ckpt_bscale, 0, L.ckpt_bscale_bytes, s);
        if (e == cudaSuccess && L.ckpt_tscale_bytes) e = cudaMemsetAsync(h->base + L.ckpt_tscale, 0, L.ckpt_tscale_bytes, s);
    }
    if (e == cudaSuccess) e = cudaMemsetAsync(h->base + L.counts, 0, L.counts_bytes, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(h->base + L.err, 0, L.err_bytes, s);
    if (e == cudaSuccess && cfg->read_fmt != RSSM_READ_NONE) {
        bool sup = true;
        int64_t tiles = static_cast<int64_t>(cfg->batch) * cfg->heads;
        int32_t rows = cfg->head_dim;
        if (cfg->kind == RSSM_GDN) {   // one copy tile per 64-row half
            tiles *= cfg->head_dim / 64;
            rows = 64;
        }
        if (ckf == RSSM_READ_FP8)   // the copy of the stored FP8 values
            e = quantize_tiles_from_fp8(cfg->read_fmt, tiles, cfg->head_dim, cfg->state_dim,
                                        region<uint8_t>(h, L.ckpt, L.ckpt_bytes),
                                        region<float>(h, L.ckpt_tscale, L.ckpt_tscale_bytes),
                                        region<uint8_t>(h, L.rc_codes, L.rc_codes_bytes),
                                        region<uint8_t>(h, L.rc_bscale, L.rc_bscale_bytes),
                                        region<float>(h, L.rc_tscale, L.rc_tscale_bytes), s, &sup);
        else if (ck16)
            e = quantize_tiles_f16(cfg->read_fmt, tiles, cfg->head_dim, cfg->state_dim,
                                   region<__half>(h, L.ckpt, L.ckpt_bytes),
                                   region<uint8_t>(h, L.rc_codes, L.rc_codes_bytes),
                                   region<uint8_t>(h, L.rc_bscale, L.rc_bscale_bytes),
                                   region<float>(h, L.rc_tscale, L.rc_tscale_bytes), s, &sup);
        else
            e = quantize_tiles(cfg->read_fmt, tiles, rows, cfg->state_dim,
                               region<float>(h, L.ckpt, L.ckpt_bytes),
                               region<uint8_t>(h, L.rc_codes, L.rc_codes_bytes),
                               region<uint8_t>(h, L.rc_bscale, L.rc_bscale_bytes),
                               region<float>(h, L.rc_tscale, L.rc_tscale_bytes), s, &sup);
        if (!sup) {
            delete h;
            return RSSM_ERR_UNSUPPORTED;
        }
    }
    if (e != cudaSuccess) {
        delete h;
        return RSSM_ERR_CUDA;
    }
    *out = h;
    return RSSM_OK;
}

rssm_status rssm_get_layout(const rssm_handle* h, rssm_layout* out) {
    if (h == nullptr || out == nullptr) return RSSM_ERR_INVALID_ARG;
    *out = h->lay;
    return RSSM_OK;
}

// Mamba-2 replay commit (verify) or explicit flush (a.force). An NVFP4 copy
// of an FP32 or FP16 checkpoint comes from a quantiser launch after the
// commit, over the tiles whose count is then 0: those that folded, and those
// with no record since their last fold, whose checkpoint and so whose codes
// are unchanged. Its many blocks per SM hide the block scales' latency better
// than the commit kernel's consumer warps (B512 verify 299 -> see the bench
// record); the FP8 writer stays fused, as in the step.
cudaError_t m2_commit_copy(const rssm_handle* h, M2Args a, cudaStream_t s, bool* sup) {
    const rssm_config& c = h->cfg;
    const bool defer = c.read_fmt == RSSM_READ_NVFP4 && (a.ck == kCkF32 || a.ck == kCkF16);
    a.defer_copy = defer ? 1 : 0;
    cudaError_t e = m2_commit(a, c.head_dim, c.state_dim, c.in_dtype, m2_read_fmt(c), s, sup);
    if (defer && e == cudaSuccess && *sup)
        e = quantize_marked_tiles(c.read_fmt, static_cast<int64_t>(c.batch) * c.heads, c.head_dim, c.state_dim,
                                  a.ck == kCkF32 ? a.ckpt : nullptr,
                                  a.ck == kCkF16 ? reinterpret_cast<const __half*>(a.ckpt) : nullptr,
                                  a.rc_codes, a.rc_bscale, a.rc_tscale, a.counts, 0, 1, s, sup);
    return e;
}

rssm_status rssm_decode_step(rssm_handle* h, int32_t T, const rssm_inputs* in, void* d_y,
                             void* stream) {
    if (h == nullptr || in == nullptr || d_y == nullptr || T < 1) return RSSM_ERR_INVALID_ARG;
    if (!aligned16(d_y)) return RSSM_ERR_INVALID_ARG;
    if (T > h->cfg.max_draft) return RSSM_ERR_CAPACITY;
    if (h->pending_T != 0) return RSSM_ERR_STATE;
    const rssm_config& c = h->cfg;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int out_dt = out_dtype_of(c);
    bool sup = true;
    cudaError_t e = cudaSuccess;

    if (c.kind == RSSM_MAMBA2) {
        const void* req[4] = {in->x, in->Bm, in->C, in->dt};
        for (const void* p : req)
            if (p == nullptr || !aligned16(p)) return RSSM_ERR_INVALID_ARG;
        M2Args a = m2_args(h);
        a.x = in->x; a.Bm = in->Bm; a.C = in->C; a.dt = in->dt;
        a.y = d_y;
        a.T = T;
        if (c.mode == RSSM_REPLAY) {
            if (T == 1) {
                // While every tile holds the same record count (from create, a
                // flush, or plain decode since), the host knows whether this
                // token completes the window. Steps that do not use the lean
                // non-flush kernel; all others use the kernel that handles both.
                const StepPlan plan = step_plan(h);
                const int rf = m2_read_fmt(c);
                // An NVFP4 read copy of an FP32 or FP16 checkpoint is written
                // by the quantiser launch that follows the flush, over the
                // tiles that flushed: its many blocks per SM hide the block
                // scales' latency far better than the flush kernel's few
                // consumer warps (the same codes, from the same stored values;
                // B256 flush 1104 -> 603 us). The FP8 writer is cheap enough to
                // stay fused (525 us fused, 599 us with the extra launch).
                const bool defer = c.read_fmt == RSSM_READ_NVFP4 && (a.ck == kCkF32 || a.ck == kCkF16);
                a.defer_copy = defer ? 1 : 0;
                const int64_t n_tiles = static_cast<int64_t>(c.batch) * c.heads;
                auto copy_flushed = [&](bool marked) {
                    if (!defer || e != cudaSuccess || !sup) return;
                    e = quantize_marked_tiles(c.read_fmt, n_tiles, c.head_dim, c.state_dim,
                                              a.ck == kCkF32 ? a.ckpt : nullptr,
                                              a.ck == kCkF16 ? reinterpret_cast<const __half*>(a.ckpt) : nullptr,
                                              a.rc_codes, a.rc_bscale, a.rc_tscale, marked ? a.counts : nullptr,
                                              c.k, 1, s, &sup);
                };
                if (plan == kPlanLean) {
                    e = m2_replay_step(a, c.head_dim, c.state_dim, c.in_dtype, out_dt, rf, kStepNonFlush, s, &sup);
                } else if (plan == kPlanFused) {
                    e = m2_replay_step(a, c.head_dim, c.state_dim, c.in_dtype, out_dt, rf, kStepAny, s, &sup);
                    copy_flushed(false);
                } else {
                    // flush tiles first (marked with count k), their copies,
                    // then the others (the lean launch resets the marks)
                    e = m2_replay_step(a, c.head_dim, c.state_dim, c.in_dtype, out_dt, rf, kStepFlushOnly, s, &sup);
                    copy_flushed(true);
                    if (e == cudaSuccess && sup)
                        e = m2_replay_step(a, c.head_dim, c.state_dim, c.in_dtype, out_dt, rf, kStepSkipFlush, s,
                                           &sup);
                }
                if (e == cudaSuccess && sup) counts_after_step(h);
            } else {
                e = m2_replay_draft(a, c.head_dim, c.state_dim, c.in_dtype, out_dt, c.read_fmt, s, &sup);
            }
        } else {
            if (T == 1) e = m2_conv_step(a, c.head_dim, c.state_dim, c.in_dtype, out_dt, c.read_fmt, s, &sup);
            else e = m2_snap_draft(a, c.head_dim, c.state_dim, c.in_dtype, out_dt, s, &sup);
        }
    } else {
        const void* req[5] = {in->q, in->k, in->v, in->alpha, in->beta};
        for (const void* p : req)
            if (p == nullptr || !aligned16(p)) return RSSM_ERR_INVALID_ARG;
        GDNArgs a = gdn_args(h);
        a.q = in->q; a.k = in->k; a.v = in->v; a.alpha = in->alpha; a.beta = in->beta;
        a.o = d_y;
        a.T = T;
        if (c.mode == RSSM_REPLAY && T > 1) {
            e = gdn_replay_draft(a, c.head_dim, c.state_dim, c.in_dtype, out_dt, s, &sup);
        } else if (c.mode == RSSM_REPLAY) {
            // the same uniform-count fast path as for Mamba-2
            const StepPlan plan = step_plan(h);
            // an NVFP4 copy of the halves that flushed comes from a quantiser
            // launch after the flush, as for Mamba-2 (one copy tile per half;
            // B256 flush 913 -> 684 us; FP8 stays fused: 620 us against 795)
            const bool defer = c.read_fmt == RSSM_READ_NVFP4;
            a.defer_copy = defer ? 1 : 0;
            const int halves = c.head_dim / 64;
            auto copy_flushed = [&](bool marked) {
                if (!defer || e != cudaSuccess || !sup) return;
                e = quantize_marked_tiles(c.read_fmt, static_cast<int64_t>(c.batch) * c.heads * halves, 64,
                                          c.state_dim, a.ckpt, nullptr, a.rc_codes, a.rc_bscale, a.rc_tscale,
                                          marked ? a.counts : nullptr, c.k, halves, s, &sup);
            };
            if (plan == kPlanLean) {
                e = gdn_replay_step(a, c.head_dim, c.state_dim, c.in_dtype, out_dt, kStepNonFlush, s, &sup);
            } else if (plan == kPlanFused) {
                e = gdn_replay_step(a, c.head_dim, c.state_dim, c.in_dtype, out_dt, kStepAny, s, &sup);
                copy_flushed(false);
            } else {
                e = gdn_replay_step(a, c.head_dim, c.state_dim, c.in_dtype, out_dt, kStepFlushOnly, s, &sup);
                copy_flushed(true);
                if (e == cudaSuccess && sup)
                    e = gdn_replay_step(a, c.head_dim, c.state_dim, c.in_dtype, out_dt, kStepSkipFlush, s, &sup);
            }
            if (e == cudaSuccess && sup) counts_after_step(h);
        } else if (T > 1) {
            e = gdn_snap_draft(a, c.head_dim, c.state_dim, c.in_dtype, out_dt, s, &sup);
        } else {
            e = gdn_conv_step(a, c.head_dim, c.state_dim, c.in_dtype, out_dt, s, &sup);
        }
    }
    rssm_status st = cuda_status(e, sup);
    if (st == RSSM_OK && T > 1) h->pending_T = T;
    return st;
}

rssm_status rssm_verify_rollback(rssm_handle* h, const int32_t* d_accepted, void* stream) {
    if (h == nullptr || d_accepted == nullptr) return RSSM_ERR_INVALID_ARG;
    if (h->pending_T == 0) return RSSM_OK;
    const rssm_config& c = h->cfg;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    bool sup = true;
    cudaError_t e = cudaSuccess;
    if (c.kind == RSSM_GDN) {
        GDNArgs a = gdn_args(h);
        a.accepted = d_accepted;
        a.T = h->pending_T;
        if (c.mode == RSSM_REPLAY) {
            e = gdn_commit(a, c.head_dim, c.state_dim, c.in_dtype, s, &sup);
            // the commit kernel writes FP32 only: the halves whose count is
            // then 0 get their copy (those that folded, and those with no
            // record since their last fold, whose codes come out unchanged)
            if (e == cudaSuccess && sup && c.read_fmt != RSSM_READ_NONE) {
                const int halves = c.head_dim / 64;
                e = quantize_marked_tiles(c.read_fmt, static_cast<int64_t>(c.batch) * c.heads * halves, 64,
                                          c.state_dim, a.ckpt, nullptr, a.rc_codes, a.rc_bscale, a.rc_tscale,
                                          a.counts, 0, halves, s, &sup);
            }
        } else {
            e = gdn_snap_restore(a, c.head_dim, c.state_dim, s, &sup);
        }
    } else {
        M2Args a = m2_args(h);
        a.accepted = d_accepted;
        a.T = h->pending_T;
        if (c.mode == RSSM_REPLAY) e = m2_commit_copy(h, a, s, &sup);
        else e = m2_snap_restore(a, c.head_dim, c.state_dim, s, &sup);
    }
    rssm_status st = cuda_status(e, sup);
    if (st == RSSM_OK) {
        h->pending_T = 0;
        h->counts_known = false;   // the acceptance counts are on the device
    }
    return st;
}

rssm_status rssm_flush(rssm_handle* h, void* stream) {
    if (h == nullptr) return RSSM_ERR_INVALID_ARG;
    if (h->pending_T != 0) return RSSM_ERR_STATE;
    const rssm_config& c = h->cfg;
    if (c.mode != RSSM_REPLAY) return RSSM_OK;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    bool sup = true;
    cudaError_t e;
    if (c.kind == RSSM_MAMBA2) {
        M2Args a = m2_args(h);
        a.force = 1;
        e = m2_commit_copy(h, a, s, &sup);
        if (e == cudaSuccess && sup) counts_all_zero(h);
    } else {
        GDNArgs a = gdn_args(h);
        a.force = 1;
        e = gdn_commit(a, c.head_dim, c.state_dim, c.in_dtype, s, &sup);
        // the commit kernel writes FP32 only: refresh every half's copy (an
        // unchanged half quantises to the same codes)
        if (e == cudaSuccess && sup && c.read_fmt != RSSM_READ_NONE)
            e = quantize_tiles(c.read_fmt, static_cast<int64_t>(c.batch) * c.heads * (c.head_dim / 64), 64,
                               c.state_dim, a.ckpt, a.rc_codes, a.rc_bscale, a.rc_tscale, s, &sup);
        if (e == cudaSuccess && sup) counts_all_zero(h);
    }
    return cuda_status(e, sup);
}

rssm_status rssm_get_error(rssm_handle* h, int32_t* err4, void* stream) {
    if (h == nullptr || err4 == nullptr) return RSSM_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    void* dev = h->base + h->lay.err;
    cudaError_t e = cudaMemcpyAsync(err4, dev, 16, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e == cudaSuccess) e = cudaMemsetAsync(dev, 0, 16, s);
    // a tile that reported an error may not have advanced its count as the
    // host assumed
    if (e != cudaSuccess || err4[0] != RSSM_DEV_OK) h->counts_known = false;
    return (e == cudaSuccess) ? RSSM_OK : RSSM_ERR_CUDA;
}

rssm_status rssm_state_bytes(const rssm_handle* h, size_t* bytes) {
    if (h == nullptr || bytes == nullptr) return RSSM_ERR_INVALID_ARG;
    *bytes = image_bytes(h->lay);
    return RSSM_OK;
}

rssm_status rssm_export_state(rssm_handle* h, void* d_dst, size_t bytes, void* stream) {
    if (h == nullptr || d_dst == nullptr || !aligned16(d_dst)) return RSSM_ERR_INVALID_ARG;
    if (bytes < image_bytes(h->lay)) return RSSM_ERR_INVALID_ARG;
    if (h->pending_T != 0) return RSSM_ERR_STATE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemcpyAsync(d_dst, h->image_hdr, kImageHdr, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) e = copy_state(h, static_cast<char*>(d_dst), true, s);
    return (e == cudaSuccess) ? RSSM_OK : RSSM_ERR_CUDA;
}

rssm_status rssm_import_state(rssm_handle* h, const void* d_src, size_t bytes, void* stream) {
    if (h == nullptr || d_src == nullptr || !aligned16(d_src)) return RSSM_ERR_INVALID_ARG;
    const size_t need = image_bytes(h->lay);
    if (bytes < need) return RSSM_ERR_INVALID_ARG;
    if (h->pending_T != 0) return RSSM_ERR_STATE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    unsigned char hdr[kImageHdr];
    cudaError_t e = cudaMemcpyAsync(hdr, d_src, kImageHdr, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return RSSM_ERR_CUDA;
    // the whole header, padding included, must be this handle's
    if (std::memcmp(hdr, h->image_hdr, kImageHdr) != 0) return RSSM_ERR_INVALID_ARG;
    h->counts_known = false;
    e = copy_state(h, const_cast<char*>(static_cast<const char*>(d_src)), false, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(h->base + h->lay.err, 0, h->lay.err_bytes, s);
    if (e == cudaSuccess && h->cfg.mode == RSSM_REPLAY) e = counts_from_device(h, s);
    else if (e == cudaSuccess) {
        counts_all_zero(h);
        e = cudaStreamSynchronize(s);
    }
    return (e == cudaSuccess) ? RSSM_OK : RSSM_ERR_CUDA;
}

rssm_status rssm_sync_counts(rssm_handle* h, void* stream) {
    if (h == nullptr) return RSSM_ERR_INVALID_ARG;
    if (h->pending_T != 0) return RSSM_ERR_STATE;
    if (h->cfg.mode != RSSM_REPLAY) return RSSM_OK;
    return counts_from_device(h, static_cast<cudaStream_t>(stream)) == cudaSuccess ? RSSM_OK : RSSM_ERR_CUDA;
}

rssm_status rssm_count_summary(const rssm_handle* h, int32_t* known, int32_t* min_count, int32_t* max_count) {
    if (h == nullptr || known == nullptr || min_count == nullptr || max_count == nullptr)
        return RSSM_ERR_INVALID_ARG;
    *known = h->counts_known ? 1 : 0;
    *min_count = h->counts_known ? counts_min(h) : -1;
    *max_count = h->counts_known ? counts_max(h) : -1;
    return RSSM_OK;
}

rssm_status rssm_quantize(int32_t fmt, int64_t tiles, int32_t rows, int32_t cols, const float* d_src,
                          void* d_codes, void* d_bscale, float* d_tscale, void* stream) {
    if (fmt != RSSM_READ_FP8 && fmt != RSSM_READ_NVFP4) return RSSM_ERR_INVALID_ARG;
    if (tiles < 0 || tiles > 0x7FFFFFFF || rows < 1 || cols < 1) return RSSM_ERR_INVALID_ARG;
    if (!dims_supported(rows, cols)) return RSSM_ERR_UNSUPPORTED;
    if (tiles == 0) return RSSM_OK;
    if (d_src == nullptr || d_codes == nullptr || d_tscale == nullptr || !aligned16(d_src) ||
        !aligned16(d_codes))
        return RSSM_ERR_INVALID_ARG;
    if (fmt == RSSM_READ_NVFP4 && d_bscale == nullptr) return RSSM_ERR_INVALID_ARG;
    bool sup = true;
    cudaError_t e = quantize_tiles(fmt, tiles, rows, cols, d_src, static_cast<uint8_t*>(d_codes),
                                   static_cast<uint8_t*>(d_bscale), d_tscale,
                                   static_cast<cudaStream_t>(stream), &sup);
    return cuda_status(e, sup);
}

rssm_status rssm_destroy(rssm_handle* h) {
    if (h == nullptr) return RSSM_ERR_INVALID_ARG;
    delete h;
    return RSSM_OK;
}

rssm_status rssm_check_bounded_wait(int64_t limit_ns, int32_t* d_err4, void* stream) {
    if (d_err4 == nullptr || limit_ns < 1 || limit_ns > static_cast<int64_t>(kWaitLimitNs))
        return RSSM_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemsetAsync(d_err4, 0, 4 * sizeof(int32_t), s);
    if (e == cudaSuccess) {
        bounded_wait_check_kernel<<<1, 32, 0, s>>>(static_cast<uint64_t>(limit_ns), d_err4);
        e = cudaGetLastError();
    }
    return e == cudaSuccess ? RSSM_OK : RSSM_ERR_CUDA;
}

}  // extern "C"

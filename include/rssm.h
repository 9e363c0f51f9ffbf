/*
 * rssm.h -- C ABI of librssm, the ReplaySSM decode step for the SSM layers
 * of hybrid language models, on NVIDIA GB300 (sm_103a).
 *
 * Sources. Pages cited by title and section:
 *  [DE] "ReplaySSM beschleunigt das Decoding von Hybridmodellen durch Caching
 *       der Eingaben statt des Zustands", sections "Wie es funktioniert" and
 *       "Wichtige Details".
 *  [TR] "NVIDIA ve Dao AI Lab, hibrit model cozumlemesini hizlandirmak icin
 *       ReplaySSM'i sundu", sections "ReplaySSM nasil calisir?", "Durum
 *       trafigini azaltma ve rollback'in basitlestirilmesi", "Kuantizasyon
 *       hatasinin sinirlandirilmasi".
 *
 * The method. Each (sequence, head) SSM state is a high-precision checkpoint
 * plus a buffer of the inputs of the tokens seen since the checkpoint was
 * written ([DE] "Wie es funktioniert"; [TR] "ReplaySSM nasil calisir?"). A
 * non-flush decode step appends this token's inputs to the buffer and
 * computes the output from the checkpoint and the buffered inputs, without
 * storing state. The step that fills the buffer (k records) is the flush
 * step. It folds every buffered input into the checkpoint, writes the
 * checkpoint once and empties the buffer. Speculative drafts are appended to
 * the buffer unverified. Rejecting them only moves the buffer pointer, with
 * no state snapshot ([DE] "Wie es funktioniert", 2nd paragraph; [TR] "Durum
 * trafigini azaltma ..."). An optional low-precision read copy of the
 * checkpoint (FP8 E4M3 or NVFP4) serves the output reads. The recurrence
 * itself always runs on the FP32 checkpoint ([TR] "Kuantizasyon
 * hatasinin sinirlandirilmasi").
 *
 * Two SSM kinds:
 *  - Mamba-2: state h in R^{P x N} per head, inputs x_t[H][P], B_t,C_t[G][N]
 *    (heads h use group h / (H/G)), dt_t[H]; parameters A_h < 0, D_h.
 *      h_t = exp(dt_t A_h) h_{t-1} + dt_t x_t B_t^T ;  y_t = h_t C_t + D_h x_t
 *  - Gated DeltaNet: state S in R^{d_v x d_k} per head, inputs q_t,k_t[H][d_k],
 *    v_t[H][d_v], alpha_t, beta_t [H].
 *      S_t = alpha_t S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T ;
 *      o_t = S_t (scale q_t)
 * The outputs equal these recurrences up to floating-point rounding.
 *
 * Conventions (all functions):
 *  - Memory ownership: the CALLER owns every device buffer. That covers the
 *    workspace, the parameters, the inputs, the outputs and the acceptance
 *    counts. The library allocates only the small host handle. It never calls
 *    cudaMalloc.
 *  - Pointers named d_* are device pointers, all others host pointers.
 *    `stream` is a cudaStream_t passed as void* (NULL = legacy default).
 *  - Calls that launch work are asynchronous on `stream`. They return a
 *    status synchronously for every error the host can detect, and never throw
 *    or abort. Errors detected on the device (an acceptance count out of range,
 *    a corrupted record count, a bounded wait that ran out) set a device error
 *    word and leave that (sequence, head) unchanged. rssm_get_error reads the
 *    word.
 *  - All device buffers must be 16-byte aligned. Strides are dense (no padding).
 *  - A handle is not thread-safe. Work for one handle must be ordered on one
 *    stream, or by the caller.
 */
#ifndef RSSM_H
#define RSSM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define RSSM_ABI_VERSION 5

/* Most buffer records one (sequence, head) holds (k - 1 + max_draft <= 32). */
#define RSSM_MAX_RECORDS 32

typedef enum {
    RSSM_OK = 0,
    RSSM_ERR_INVALID_ARG = 1,  /* null pointer, bad size, misaligned buffer    */
    RSSM_ERR_UNSUPPORTED = 2,  /* valid but not built (shape, dtype, mode)     */
    RSSM_ERR_CAPACITY = 3,     /* workspace too small, T > max_draft           */
    RSSM_ERR_CUDA = 4,         /* a CUDA runtime call or launch failed         */
    RSSM_ERR_STATE = 5         /* call out of order (drafts pending, ...)      */
} rssm_status;

enum { RSSM_MAMBA2 = 1, RSSM_GDN = 2 };                  /* rssm_config.kind     */
enum { RSSM_REPLAY = 1, RSSM_CONVENTIONAL = 2 };         /* rssm_config.mode     */
enum { RSSM_F32 = 1, RSSM_BF16 = 2, RSSM_F16 = 3 };      /* in/out_dtype; ckpt_dtype */
enum { RSSM_CKPT_FP8 = 4, RSSM_CKPT_NVFP4 = 5 };        /* ckpt_dtype: tile formats */
enum { RSSM_READ_NONE = 0, RSSM_READ_FP8 = 1, RSSM_READ_NVFP4 = 2 }; /* read_fmt */

/* Device error codes reported through rssm_get_error (err[0]). RSSM_DEV_TIMEOUT:
 * a kernel's bounded wait on one of its pipeline barriers ran out (1 s); the
 * kernel stopped issuing, drained its own copies and returned. */
enum { RSSM_DEV_OK = 0, RSSM_DEV_ACCEPTED_RANGE = 1, RSSM_DEV_COUNT_RANGE = 2, RSSM_DEV_TIMEOUT = 3 };

/*
 * Layer configuration.
 *   kind       RSSM_MAMBA2 or RSSM_GDN.
 *   mode       RSSM_REPLAY (checkpoint + input buffer) or RSSM_CONVENTIONAL (the
 *              load/decay/update/store step, with snapshot rollback for drafts;
 *              kept as the comparison baseline).
 *   batch      B >= 1 sequences.  heads H >= 1.
 *   head_dim   Mamba-2 P, GDN d_v (rows of the state).  Supported: 64, 128.
 *   state_dim  Mamba-2 N, GDN d_k (columns, contiguous). Supported: 64, 128.
 *   groups     Mamba-2 G (H % G == 0); ignored (set 1) for GDN.
 *   k          flush threshold = buffer records per window, 1..32
 *              ([TR] "ReplaySSM nasil calisir?": a 16-record buffer). k = 1
 *              flushes on every token, which is the conventional step.
 *   max_draft  T_max >= 1, the most tokens one rssm_decode_step may draft.
 *              The buffer holds k - 1 + T_max records, at most 32. Drafts
 *              (T_max > 1) are built for REPLAY and for CONVENTIONAL (the
 *              snapshot baseline), for both kinds.
 *   in_dtype   RSSM_F32 or RSSM_BF16: dtype of x, B, C, dt (Mamba-2) and
 *              q, k, v (GDN). alpha, beta are always FP32.
 *   out_dtype  RSSM_F32 or RSSM_BF16 for y/o; 0 means "same as in_dtype".
 *   read_fmt   RSSM_READ_NONE, RSSM_READ_FP8 (E4M3 codes, one FP32 scale per
 *              tile) or RSSM_READ_NVFP4 (E2M1 codes, one E4M3 scale per 16
 *              consecutive state_dim elements, one FP32 scale per tile).
 *              REPLAY (Mamba-2 or GDN): a read copy of the checkpoint that
 *              the non-flush outputs read; the recurrence stays on the FP32
 *              checkpoint. Drafts (max_draft > 1) read the copy too;
 *              CONVENTIONAL takes max_draft = 1 with a read copy. A
 *              Mamba-2 tile is one copy tile; a GDN tile is two or one
 *              64-row halves, each a copy tile. A GDN read copy (REPLAY)
 *              takes bf16 inputs; its records then also keep v and beta, and
 *              a GDN flush replays the window's records through the
 *              recurrence from the FP32 checkpoint, so the copy's error never
 *              reaches it.
 *              CONVENTIONAL (Mamba-2 and GDN): the quantised-recurrence
 *              baseline ([TR] "Kuantizasyon hatasinin sinirlandirilmasi"):
 *              the state itself is kept in that format (the same copy
 *              tiles), dequantised, updated in FP32 and re-quantised at every
 *              step; the FP32 region then holds only the initial state.
 *   gdn_scale  GDN query scale (o = S (gdn_scale q)); 0 means 1.
 *   ckpt_dtype 0 or RSSM_F32: FP32 checkpoint. RSSM_F16: FP16 checkpoint
 *              ([TR] "Kuantizasyon hatasinin sinirlandirilmasi": an FP16
 *              recurrence checkpoint under low-precision reads). Every flush
 *              folds in FP32 and rounds the new checkpoint to FP16 (round to
 *              nearest even); the read copy, if any, is made from the rounded
 *              values. Mamba-2 REPLAY with bf16 inputs and max_draft = 1
 *              only. The ckpt region then holds FP16 [B][H][P][N]; the
 *              d_state0 argument of rssm_create stays FP32 and is rounded.
 *              RSSM_CKPT_FP8 / RSSM_CKPT_NVFP4: the checkpoint kept in a
 *              read-copy tile format (same sentence: FP8 recurrence, and the
 *              full NVFP4 checkpoint it compares against). Every flush decodes
 *              it, folds in FP32 and quantises the result; rssm_create
 *              quantises d_state0. Non-flush outputs read the checkpoint
 *              itself unless read_fmt names a copy; only an NVFP4 copy of an
 *              FP8 checkpoint is allowed, made from the stored values. Same
 *              restrictions as RSSM_F16. Codes in ckpt, scales in
 *              ckpt_bscale / ckpt_tscale.
 */
typedef struct {
    int32_t kind;
    int32_t mode;
    int32_t batch;
    int32_t heads;
    int32_t head_dim;
    int32_t state_dim;
    int32_t groups;
    int32_t k;
    int32_t max_draft;
    int32_t in_dtype;
    int32_t out_dtype;
    int32_t read_fmt;
    float gdn_scale;
    int32_t ckpt_dtype;
} rssm_config;

/*
 * Per-step inputs: device pointers, dense, sequence-major with the T drafted
 * tokens of a sequence adjacent ([B][T][...]; T = 1 for plain decode).
 *   Mamba-2: x [B][T][H][P], Bm and C [B][T][G][N], dt [B][T][H]  (in_dtype).
 *            dt is the positive step size after its activation.
 *   GDN:     q, k [B][T][H][d_k], v [B][T][H][d_v] (in_dtype);
 *            alpha, beta [B][T][H] (FP32).
 * Unused members may be NULL.
 */
typedef struct {
    const void* x;
    const void* Bm;
    const void* C;
    const void* dt;
    const void* q;
    const void* k;
    const void* v;
    const float* alpha;
    const float* beta;
} rssm_inputs;

/*
 * Byte offsets (from the workspace base) and sizes of the workspace regions.
 * Regions of size 0 are absent. Layouts (dense, row-major):
 *   ckpt       FP32 [B][H][head_dim][state_dim]  checkpoint (conventional: live state);
 *              FP16 when ckpt_dtype = RSSM_F16
 *   counts     int32 [B][H]   committed buffer records per (sequence, head)
 *   err        int32 [4]      device error word: code, count, tile, value
 *   buf_x      Mamba-2 x records   in_dtype [B][H][cap][P]
 *   buf_b      Mamba-2 B records   in_dtype [B][G][cap][N]
 *   buf_dt     Mamba-2 dt records  in_dtype [B][H][cap]
 *   buf_k      GDN k records       in_dtype [B][H][cap][d_k]
 *   buf_u      GDN u records       FP32 [B][H][d_v/64][cap][64] (see rssm_decode_step):
 *              record j's row r at [b][h][r/64][j][r%64], so each 64-row half
 *              of a tile's records is contiguous
 *   buf_a      GDN alpha records   FP32 [B][H][cap]
 *   rc_codes   read copy codes: FP8 uint8 [B][H][R][C]; NVFP4 uint8 [B][H][R][C/2]
 *              (element 2i in the low nibble); R, C = head_dim, state_dim
 *   rc_bscale  NVFP4 block scales (E4M3) uint8 [B][H][R][C/16]
 *   rc_tscale  read-copy tile scales FP32: Mamba-2 [B][H]; GDN [B][H][d_v/64]
 *              (one per 64-row half)
 *   snap       conventional drafts: FP32 [T_max][B][H][head_dim][state_dim]
 *   buf_v      GDN v records (read copies only) in_dtype [B][H][d_v/64][cap][64]
 *   buf_beta   GDN beta records (read copies only) FP32 [B][H][cap]
 *   ckpt_bscale  NVFP4 checkpoint block scales (E4M3) uint8 [B][H][P][N/16]
 *   ckpt_tscale  tile-format checkpoint tile scales FP32 [B][H]; the ckpt
 *              region then holds the codes (FP8 [B][H][P][N], NVFP4
 *              [B][H][P][N/2])
 *   cnt_hist   int32 [RSSM_MAX_RECORDS + 2]  record-count summary written by
 *              rssm_sync_counts and rssm_import_state: entry c (0..32) is the
 *              number of tiles holding c records, the last entry the number of
 *              tiles whose count is outside 0..32
 *   capacity   cap = k - 1 + max_draft rounded up to a multiple of 8 (record
 *              slots per buffer; the rounding keeps each tile's record arrays
 *              in whole 16-byte units)
 */
typedef struct {
    size_t ckpt, ckpt_bytes;
    size_t counts, counts_bytes;
    size_t err, err_bytes;
    size_t buf_x, buf_x_bytes;
    size_t buf_b, buf_b_bytes;
    size_t buf_dt, buf_dt_bytes;
    size_t buf_k, buf_k_bytes;
    size_t buf_u, buf_u_bytes;
    size_t buf_a, buf_a_bytes;
    size_t rc_codes, rc_codes_bytes;
    size_t rc_bscale, rc_bscale_bytes;
    size_t rc_tscale, rc_tscale_bytes;
    size_t snap, snap_bytes;
    size_t buf_v, buf_v_bytes;
    size_t buf_beta, buf_beta_bytes;
    size_t ckpt_bscale, ckpt_bscale_bytes;
    size_t ckpt_tscale, ckpt_tscale_bytes;
    size_t cnt_hist, cnt_hist_bytes;
    size_t total_bytes;
    int32_t capacity;
} rssm_layout;

typedef struct rssm_handle rssm_handle;

/* Library ABI version (RSSM_ABI_VERSION). */
int32_t rssm_abi_version(void);

/* Static string for a status code; never NULL. */
const char* rssm_status_string(rssm_status status);

/*
 * Workspace bytes that rssm_create needs for `cfg`. The value covers the
 * checkpoint, buffer, counts, read copy and snapshots, each region 256-byte
 * aligned. Host only; needs no GPU.
 * Errors: INVALID_ARG (null pointer, inconsistent sizes), UNSUPPORTED.
 */
rssm_status rssm_workspace_size(const rssm_config* cfg, size_t* bytes);

/*
 * Region offsets for `cfg`, the same as rssm_get_layout returns after create.
 * Host only; needs no GPU.
 */
rssm_status rssm_layout_for(const rssm_config* cfg, rssm_layout* out);

/*
 * Create a layer on the caller's workspace ([DE] "Wie es funktioniert": the
 * state is a checkpoint plus a buffer of recent inputs).
 *   d_workspace   device, >= rssm_workspace_size bytes, 256-byte aligned;
 *                 owned by the caller and must outlive the handle.
 *   d_A, d_D      Mamba-2 FP32 [H] (A_h < 0); kept by pointer, must outlive
 *                 the handle. NULL for GDN.
 *   d_state0      FP32 [B][H][head_dim][state_dim] initial state, copied into
 *                 the checkpoint; NULL = zeros.
 * Zeroes the counts and the error word. Writes the read copy of the initial
 * state when read_fmt != NONE. All of this is enqueued on `stream`.
 * Errors: INVALID_ARG, UNSUPPORTED, CAPACITY (workspace too small), CUDA.
 */
rssm_status rssm_create(const rssm_config* cfg, void* d_workspace, size_t workspace_bytes,
                        const float* d_A, const float* d_D, const float* d_state0, void* stream,
                        rssm_handle** out);

/* Region offsets of a created handle (see rssm_layout). */
rssm_status rssm_get_layout(const rssm_handle* h, rssm_layout* out);

/*
 * One decode step of T tokens per sequence.
 *  REPLAY, T == 1 ([DE] "Wie es funktioniert"; [TR] "ReplaySSM nasil calisir?"):
 *    appends the token's record at slot c (c = committed records). If c+1 < k,
 *    the output comes from the checkpoint and the buffered records, and no
 *    state is stored (non-flush step). If c+1 == k, it folds all k records
 *    into the checkpoint, writes it once (and its read copy), and resets c to 0
 *    (flush step).
 *    Mamba-2 output, with m = c+1 records i = 1..m (m = this token):
 *      y = exp(A sum_{j<=m} dt_j) h_ckpt C_m
 *          + sum_{i<=m} exp(A sum_{i<j<=m} dt_j) dt_i (B_i . C_m) x_i + D x_m
 *    GDN output: the WY/UT form of the window. Each record stores the row u_i
 *    of U = T (V - diag(gamma) K S_ckpt^T), T = (I + diag(beta) A)^-1 diag(beta).
 *    The row is solved by forward substitution when token i arrives, and U
 *    replaces v_i and beta_i in the record. Then
 *      o = gamma_m S_ckpt q + sum_{i<=m} (gamma_m/gamma_i)(k_i . q) u_i,
 *    evaluated as two small products: S_ckpt [k_m; q] and the masked
 *    (q K^T) U. With a read copy, S_ckpt in these products is the copy, the
 *    record also keeps v_i and beta_i, and the flush step replays the
 *    window's records through the recurrence from the FP32 checkpoint.
 *    With a low-precision checkpoint (ckpt_dtype) the fold reads the stored
 *    values and stores the new checkpoint in that format.
 *    The handle keeps on the host how many tiles hold each record count
 *    (known after create, rssm_flush, rssm_sync_counts, rssm_import_state
 *    and plain T == 1 steps since; unknown after rssm_verify_rollback and
 *    after rssm_get_error reported a device error). While it is known and
 *    every count c satisfies c+1 < k, the step runs a kernel that handles only
 *    non-flush tiles; otherwise a kernel that handles both kinds of tile. The
 *    outputs are the same bits either way. The workspace regions are written
 *    by the library alone: a tile whose count the caller changed so that it
 *    is due to flush in such a step is left unchanged and reported as
 *    RSSM_DEV_COUNT_RANGE. At small batches (up to 16 tiles per SM for
 *    Mamba-2, 4 for GDN) a step whose every tile is due runs one block per
 *    tile; there the Mamba-2 kernel likewise reports, and leaves unchanged, a
 *    tile whose count the caller moved below k - 1, while the GDN kernel
 *    takes its non-flush step.
 *  REPLAY, T > 1 (speculative drafts; [TR] "Durum trafigini azaltma ...",
 *    2nd paragraph): appends T uncommitted records at slots c..c+T-1 and
 *    writes, for each draft tau, the output from the checkpoint and records
 *    1..c+tau. With a read copy the checkpoint term reads the copy, as the
 *    one-token non-flush outputs do ([TR] "Kuantizasyon hatasinin
 *    sinirlandirilmasi"). No state is written. rssm_verify_rollback must follow before
 *    the next decode_step. GDN drafts solve each draft's record row u after
 *    the earlier drafts' rows, so draft tau's row and output are the
 *    one-token step's with the earlier drafts committed.
 *  CONVENTIONAL, T == 1: loads the state, decays and updates it, computes the
 *    output and stores the state ([DE] "Wie es funktioniert", 1st paragraph).
 *  CONVENTIONAL, T > 1: runs T conventional updates from the live state and
 *    writes a full-state snapshot after each ([DE] "Wie es funktioniert": the
 *    snapshot per draft token that ReplaySSM removes). The live state is
 *    unchanged. Both kinds.
 *  d_y: Mamba-2 [B][T][H][P], GDN [B][T][H][d_v], out_dtype.
 * Errors: INVALID_ARG (null or misaligned pointers, T < 1), CAPACITY
 * (T > max_draft), STATE (drafts pending), UNSUPPORTED, CUDA.
 */
rssm_status rssm_decode_step(rssm_handle* h, int32_t T, const rssm_inputs* in, void* d_y,
                             void* stream);

/*
 * Resolve the drafts of the last rssm_decode_step(T > 1).
 *  d_accepted: device int32 [B], accepted draft count a_b in 0..T per sequence.
 *  REPLAY (Mamba-2 and GDN): c_b += a_b. Records past c_b are discarded by
 *    that pointer move alone; no state is restored ([DE] "Wie es
 *    funktioniert", 2nd paragraph). Where c_b >= k, the committed records are
 *    folded into the checkpoint, which is written once (with its read copy),
 *    and c_b becomes 0.
 *  CONVENTIONAL: copies snapshot a_b into the live state where a_b >= 1.
 *  An a_b outside 0..T sets RSSM_DEV_ACCEPTED_RANGE and leaves sequence b as
 *  if a_b = 0. With no drafts pending, the call is a no-op returning RSSM_OK.
 *  The accepted counts stay on the device, so afterwards the handle no longer
 *  knows the record counts; rssm_sync_counts brings that knowledge back
 *  before a run of plain T == 1 steps.
 * Errors: INVALID_ARG, CUDA.
 */
rssm_status rssm_verify_rollback(rssm_handle* h, const int32_t* d_accepted, void* stream);

/*
 * Fold every committed record into the checkpoint now, and write it (and its
 * read copy), for tiles with c > 0 ([DE] "Wie es funktioniert", 2nd
 * paragraph: the flush folds the buffered inputs into the checkpoint and
 * writes it once; here the caller asks for it before the window is full).
 * Afterwards c = 0, and the checkpoint alone is the complete state, for
 * example to end a sequence. The fold rounds differently from the one the
 * k-th token would have made, so outputs after an early flush are equal to
 * an uninterrupted run only up to rounding; rssm_export_state keeps the exact
 * bits instead. CONVENTIONAL: no-op.
 * Errors: INVALID_ARG (null handle), STATE (drafts pending), CUDA.
 */
rssm_status rssm_flush(rssm_handle* h, void* stream);

/*
 * Copy the device error word to err4[0..3] (code, count, tile, value) and
 * clear it. Synchronises `stream`. Returns RSSM_OK when the copy worked;
 * err4[0] != 0 reports a device-detected error.
 */
rssm_status rssm_get_error(rssm_handle* h, int32_t* err4, void* stream);

/*
 * The read-copy writer on its own ([TR] "Kuantizasyon hatasinin
 * sinirlandirilmasi": a low-precision copy for reads). It is the same code
 * the flush step runs, fused. It quantises `tiles` FP32 tiles of rows x cols
 * (cols = 64 or 128, dense) from d_src:
 *   RSSM_READ_FP8:   s = amax/448 per tile, codes E4M3(x * (1/s)) -> d_codes
 *                    uint8 [tiles][rows][cols]; d_tscale FP32 [tiles].
 *   RSSM_READ_NVFP4: s = amax/(6*448) per tile; per 16 consecutive elements
 *                    of a row, block scale E4M3(amax_blk * (1/(6 s))) -> d_bscale
 *                    [tiles][rows][cols/16]; codes E2M1(x * (1/(bs*s))) packed two per
 *                    byte, element 2i in the low nibble -> d_codes [tiles][rows][cols/2].
 * Rounding is to nearest even, with saturation to the largest finite code.
 * Errors: INVALID_ARG, UNSUPPORTED, CUDA.
 */
rssm_status rssm_quantize(int32_t fmt, int64_t tiles, int32_t rows, int32_t cols,
                          const float* d_src, void* d_codes, void* d_bscale, float* d_tscale,
                          void* stream);

/*
 * Check of the bounded-wait path on the device, for failure-detection tests.
 * Launches one block whose thread waits on a shared-memory mbarrier that
 * nothing completes, with the bounded wait the pipelined kernels use but a
 * limit of limit_ns. When the limit runs out the kernel records the timeout
 * the way those kernels do: d_err4[0] = RSSM_DEV_TIMEOUT, d_err4[1] = 1,
 * d_err4[2] = -1 (no tile), d_err4[3] = the nanoseconds waited (saturated to
 * INT32_MAX). Then it returns, and the context stays usable.
 *   limit_ns  1 .. 1e9.
 *   d_err4    device int32 [4], caller-owned; zeroed by the call first.
 * Errors: INVALID_ARG (null pointer, limit out of range), CUDA.
 */
rssm_status rssm_check_bounded_wait(int64_t limit_ns, int32_t* d_err4, void* stream);

/*
 * The layer's state as a portable image, for checkpoint / resume of a serving
 * process. [TR] "ReplaySSM nasil calisir?", 2nd paragraph: a sequence's state
 * is its high-precision checkpoint, the buffer of inputs since that
 * checkpoint, and the buffer pointer. The image therefore holds all three
 * for every (sequence, head): the checkpoint (with its scales for the tile
 * formats), the record counts, every record region, and the read copy. A
 * handle created with the same rssm_config and given the image continues the
 * decode with outputs bit-identical to an uninterrupted run: nothing is
 * folded or rounded on the way.
 *
 * Image layout (device memory, caller-owned): a 256-byte header (the bytes
 * "RSSMSTAT", the ABI version, the header size, the rssm_config, the image
 * size), then the regions ckpt, ckpt_bscale, ckpt_tscale, counts, buf_x,
 * buf_b, buf_dt, buf_k, buf_u, buf_a, buf_v, buf_beta, rc_codes, rc_bscale,
 * rc_tscale of rssm_layout that are present, each at the next 256-byte
 * boundary, with their workspace bytes unchanged. Snapshots and the error
 * word are not part of the state.
 */

/* Bytes of the image of this handle's state. Host only. */
rssm_status rssm_state_bytes(const rssm_handle* h, size_t* bytes);

/*
 * Write the image to d_dst (device, 16-byte aligned, >= rssm_state_bytes).
 * Asynchronous on `stream`; the header comes from host memory owned by the
 * handle. The workspace is only read.
 * Errors: INVALID_ARG (null, misaligned, too small), STATE (drafts pending:
 * verify them first), CUDA.
 */
rssm_status rssm_export_state(rssm_handle* h, void* d_dst, size_t bytes, void* stream);

/*
 * Replace the handle's state with an image written by rssm_export_state for
 * the same rssm_config (the header is checked field by field). Copies the
 * regions into the workspace, then reads the record counts as
 * rssm_sync_counts does. Synchronises `stream`. The error word is cleared.
 * Errors: INVALID_ARG (null, misaligned, too small, not an image, another
 * configuration or ABI version), STATE (drafts pending), CUDA.
 */
rssm_status rssm_import_state(rssm_handle* h, const void* d_src, size_t bytes, void* stream);

/*
 * Count on the device how many tiles hold each record count (the cnt_hist
 * region), copy that summary to the handle and synchronise `stream`. After
 * rssm_verify_rollback the counts differ per sequence and live on the device
 * only; this call lets the following plain T == 1 steps run the non-flush
 * kernel again wherever no tile can complete its window ([TR] "Durum
 * trafigini azaltma ...", 2nd paragraph: the buffer pointer is the whole
 * rollback, so the counts are all the host needs to know). A count outside
 * 0..k-1 leaves the knowledge unknown (and is reported by the next step).
 * REPLAY only; CONVENTIONAL: no-op.
 * Errors: INVALID_ARG, STATE (drafts pending), CUDA.
 */
rssm_status rssm_sync_counts(rssm_handle* h, void* stream);

/*
 * What the handle knows about the record counts, without touching the
 * device: *known = 1 and the smallest and largest count over all tiles, or
 * *known = 0 (min and max then -1). Host only.
 */
rssm_status rssm_count_summary(const rssm_handle* h, int32_t* known, int32_t* min_count,
                               int32_t* max_count);

/*
 * Free the host handle. The workspace and all other device memory stay the
 * caller's ([DE] "Wie es funktioniert": the state is the checkpoint and the
 * buffer, which live in the caller's workspace, so dropping the handle loses
 * nothing; rssm_import_state resumes it in a new handle). In-flight work on
 * the stream is not waited for.
 * Errors: INVALID_ARG (null handle).
 */
rssm_status rssm_destroy(rssm_handle* h);

#ifdef __cplusplus
}
#endif

#endif /* RSSM_H */

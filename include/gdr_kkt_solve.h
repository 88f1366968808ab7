/*
 * gdr_kkt_solve.h - C ABI of the GB300 (sm_103a) chunk-forward kkt_solve step of
 * Gated DeltaNet.
 *
 * Operation (MindSpeed-Ops PR #135 page, "feat(triton): add
 * chunk_gated_delta_rule_fwd_kkt_solve", section "What this PR does" and its
 * API block): one call equals solve_tril(chunk_scaled_dot_kkt_fwd(k, g, beta)).
 * For every sequence, every chunk of at most 64 tokens counted from the
 * sequence start, and every head h:
 *     A[i][j] = beta_i * (k_i . k_j) * exp(g_i - g_j)   for j < i < L, else 0
 *     out[chunk row i][h][0..63] = row i of (I + A)^{-1}
 * with L <= 64 the chunk's length.  Columns >= L of a partial chunk are 0.  The
 * gate exponent is clamped to [-50, 50] as on the same page's bot summary; for
 * chunk-local log-decays (g non-increasing inside a chunk) the clamp never binds
 * on the lower triangle.
 *
 * Conventions for every entry point below:
 *   - All tensor pointers are DEVICE pointers owned by the caller (except for
 *     gdr_kkt_solve_host, which takes host pointers and a device workspace).
 *     No device memory is allocated or freed by the library, and no pointer is
 *     retained after return.
 *   - Work is enqueued on `stream` (a cudaStream_t passed as void*; NULL = the
 *     legacy default stream) and the call returns without synchronising.
 *   - Errors are returned as gdr_status codes; the library never aborts, traps
 *     or prints.  Argument errors are detected on the host before any launch,
 *     and then nothing is enqueued and `out` is untouched.
 *   - Calls are thread-safe: the only mutable host state (a driver entry point,
 *     per-device set-up, the host-buffer call's streams and events) is
 *     initialised once under a lock.
 *   - After one call on a device (which sets up the library's per-device state
 *     outside any capture), gdr_kkt_solve and gdr_kkt_solve_ex on that device
 *     can be captured into a CUDA graph by stream capture; a replay reads the
 *     input buffers as they are at replay time.
 */
#ifndef GDR_KKT_SOLVE_H
#define GDR_KKT_SOLVE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    GDR_OK = 0,
    GDR_ERR_NULL = -1,    /* a required pointer is NULL                        */
    GDR_ERR_SHAPE = -2,   /* negative size, K not in {64,128,192,256} (K <= 128 for
                             fp32 keys and for chunk 128), overflow           */
    GDR_ERR_CHUNK = -3,   /* chunk_size not 64 (or 128 for the fused call)      */
    GDR_ERR_DTYPE = -4,   /* a dtype argument outside the supported set (k: bf16
                             or fp16, or fp32 in the fused chunk-64 call)      */
    GDR_ERR_ALIGN = -5,   /* a pointer is not aligned as documented below      */
    GDR_ERR_DEVICE = -6,  /* no current CUDA device, or it is not sm_103       */
    GDR_ERR_CUDA = -7,    /* a CUDA runtime/driver call failed (launch, TMA map) */
    GDR_ERR_TIMEOUT = -8, /* a device-side bounded wait ran out (see gdr_kkt_solve_device_status) */
    GDR_ERR_SCRATCH = -9, /* too large for gdr_kkt_solve_unfused_noalloc's fixed scratch */
    GDR_ERR_CU_SEQLENS = -10 /* cu_seqlens breaks its contract (found by gdr_check_cu_seqlens) */
} gdr_status;

typedef enum {
    GDR_F32 = 0,          /* IEEE fp32                                         */
    GDR_BF16 = 1,         /* bfloat16 (outputs: round-to-nearest-even from fp32) */
    GDR_F16 = 2           /* IEEE fp16 (outputs: round-to-nearest-even from fp32) */
} gdr_dtype;

/*
 * gdr_kkt_solve - (I + A)^{-1} of every 64-token chunk and head.
 *
 *   k          bf16 [B, T, H, K] contiguous; with cu_seqlens: [1, T, H, K].
 *              16-byte aligned.  K is 64, 128, 192 or 256.
 *   g          fp32 [B, T, H] (same leading layout as k) chunk-local cumulative
 *              log-gate, or NULL (gate factor 1).  4-byte aligned.
 *   beta       bf16 [B, T, H], or NULL (beta = 1).  2-byte aligned.
 *   cu_seqlens int32 [B + 1] device array, or NULL.  When given, B is the number
 *              of packed sequences, T the total token count, and sequence n
 *              covers token rows [cu[n], cu[n+1]); chunks restart at every
 *              sequence start (same page, bot summary: the T_local fix).  The
 *              contents are the caller's contract: cu[0] = 0, non-decreasing,
 *              cu[B] <= T.  Token rows outside every sequence are not written.
 *   B, T, H, K sizes; B, T or H equal to 0 is an empty problem (returns GDR_OK,
 *              enqueues nothing).  B*T must be below 2^31.
 *   chunk_size 64 (or 128, see gdr_kkt_solve_ex); any other value returns
 *              GDR_ERR_CHUNK, as the page's API raises ValueError for chunk
 *              sizes it does not support.
 *   out_dtype  GDR_F32, GDR_BF16 or GDR_F16.
 *   out        [B, T, H, 64] of out_dtype, 16-byte aligned.  Every row of a
 *              real token is fully written (zeros included); no separate
 *              zero-fill is needed.  Must not overlap the inputs.
 *   stream     cudaStream_t as void*.
 * Returns GDR_OK when the kernel was enqueued, else an error code.
 */
int gdr_kkt_solve(const void *k, const float *g, const void *beta,
                  const int32_t *cu_seqlens, int64_t B, int64_t T, int64_t H,
                  int64_t K, int chunk_size, int out_dtype, void *out,
                  void *stream);

/*
 * gdr_kkt_solve_ex - the same operation for the other input types the page's
 * unit tests cover (same page, "How was this patch tested": fp32, bf16 and fp16
 * inputs; its API block takes k, g and beta of the caller's dtype).
 *
 *   k_dtype    GDR_BF16 or GDR_F16 (the Gram runs on the tensor cores in that
 *              type; products are exact in the fp32 accumulator), or GDR_F32
 *              with K = 64 or 128 and chunk_size 64.  With fp32 or fp16 output
 *              each key is split into a tf32 part and a remainder and the Gram
 *              is the tf32 product of the parts plus the two cross products
 *              of their bf16 roundings (at most about 2^-18 relative error per
 *              key product); with bf16 output the Gram is one tf32 product of the keys as
 *              given (each key element narrowed by at most 2^-10 of itself,
 *              below the output's own rounding).  fp32 keys with other K or
 *              chunk sizes return GDR_ERR_SHAPE or GDR_ERR_DTYPE.
 *   chunk_size 64, or 128 (K = 64 or 128; bf16 or fp16 keys): out is then
 *              [B, T, H, 128] and each 128-token chunk is one problem, as in
 *              the PyPTO page "GatedDeltaRule算子性能优化案例", section 3.2.
 *   beta_dtype GDR_F32 (4-byte aligned), GDR_BF16 or GDR_F16 (2-byte aligned);
 *              ignored when beta is NULL.
 *   out_dtype  GDR_F32, GDR_BF16 or GDR_F16.
 * Every other argument, the alignment rules, the return codes and the
 * ownership and stream conventions are those of gdr_kkt_solve, which equals
 * gdr_kkt_solve_ex(k, GDR_BF16, g, beta, GDR_BF16, ...).
 */
int gdr_kkt_solve_ex(const void *k, int k_dtype, const float *g, const void *beta,
                     int beta_dtype, const int32_t *cu_seqlens, int64_t B, int64_t T,
                     int64_t H, int64_t K, int chunk_size, int out_dtype, void *out,
                     void *stream);

/*
 * The unfused chain, in two calls, as on the same page ("What this PR does":
 * the fused call replaces chunk_scaled_dot_kkt_fwd followed by solve_tril, with
 * A passed between them through HBM as [B, T, H, 64]).  It is the baseline
 * that measures the fusion: A makes a round trip through HBM (256 bytes per
 * token-head written and read again).  Both calls run the fused kernel's own
 * arithmetic, so gdr_solve_tril(gdr_chunk_scaled_dot_kkt(...)) equals
 * gdr_kkt_solve_ex(...) bit for bit.
 *
 * gdr_chunk_scaled_dot_kkt - writes A [B, T, H, 64] fp32 (16-byte aligned):
 *   A[i][j] = beta_i (k_i . k_j) exp(g_i - g_j) for j < i < L, and exactly 0 on
 *   and above the diagonal and in columns >= L.  Rows of tokens outside every
 *   sequence are not written.  Other arguments as in gdr_kkt_solve_ex.
 */
int gdr_chunk_scaled_dot_kkt(const void *k, int k_dtype, const float *g, const void *beta,
                             int beta_dtype, const int32_t *cu_seqlens, int64_t B, int64_t T,
                             int64_t H, int64_t K, int chunk_size, float *A, void *stream);

/*
 * gdr_solve_tril - out = (I + A)^{-1} of every chunk and head from A [B, T, H,
 *   64] fp32 (16-byte aligned; only the strictly lower part of each chunk's
 *   L x L block is read).  cu_seqlens, B, T, H, chunk_size, out_dtype and out
 *   as in gdr_kkt_solve.
 */
int gdr_solve_tril(const float *A, const int32_t *cu_seqlens, int64_t B, int64_t T, int64_t H,
                   int chunk_size, int out_dtype, void *out, void *stream);

/*
 * gdr_kkt_solve_unfused_noalloc - the unfused chain above in one call that
 * allocates nothing.  The paper has no counterpart; this entry point exists for
 * callers that may not allocate device memory while they run: a serving
 * runtime whose device memory is planned up front with a fixed budget, or code
 * that cannot afford cudaMalloc's implicit device synchronisation.  They pass
 * inputs and outputs as for gdr_kkt_solve_ex; A goes through a scratch array
 * that is part of the library's device image (64 MiB on every GPU that loads
 * the library, held until the process exits).
 *
 *   Limit: at most 262144 token-heads per call (B*T*H, or T*H with
 *          cu_seqlens); larger problems return GDR_ERR_SCRATCH before anything
 *          is enqueued.
 *   Inputs: those of the unfused chain, a subset of gdr_kkt_solve_ex's: keys
 *          bf16 or fp16 only (fp32 keys return GDR_ERR_DTYPE) and chunk_size 64
 *          only (128 returns GDR_ERR_CHUNK); K, beta and output types, layouts
 *          and alignment as for gdr_kkt_solve_ex.  Where both accept the
 *          arguments, the result equals gdr_kkt_solve_ex's bit for bit.
 *   Set-up: the first call on a device, with that device current, looks up the
 *          scratch's device address (cudaGetSymbolAddress) and keeps it for
 *          later calls; make that first call before any stream capture.
 *   Races:  every call on a device shares the one scratch array.  Calls whose
 *          work overlaps on the GPU (different streams without ordering between
 *          them, or several host threads on different streams) race on it and
 *          give wrong results; order them, for example on one stream.  Nothing
 *          in the scratch needs to start at zero: each call writes every row of
 *          A that it later reads, and the array keeps the last call's contents.
 */
int gdr_kkt_solve_unfused_noalloc(const void *k, int k_dtype, const float *g, const void *beta,
                                  int beta_dtype, const int32_t *cu_seqlens, int64_t B, int64_t T,
                                  int64_t H, int64_t K, int chunk_size, int out_dtype, void *out,
                                  void *stream);

/*
 * gdr_kkt_solve_host - gdr_kkt_solve_ex on HOST buffers (no counterpart on the
 * pages; for callers whose inputs and output live in host memory).  k, g, beta,
 * cu_seqlens and out are host pointers with the layouts of gdr_kkt_solve_ex;
 * `workspace` is a device buffer of at least
 * gdr_kkt_solve_host_workspace_bytes(k_dtype, B, T, H, K, chunk_size,
 * out_dtype) bytes, 256-byte aligned, owned by the caller (the library still
 * allocates no device memory).  The call copies the inputs into the workspace,
 * runs the kernel and copies the output back, slice by slice (runs of whole
 * chunks of one sequence) over two internal streams, so that host-to-device
 * copies, kernels and device-to-host copies of different slices overlap;
 * packed sequences (cu_seqlens) go as one slice, and then only the rows of
 * real tokens are written to out.  The work is ordered after everything
 * enqueued on `stream` before the call, and everything enqueued on `stream`
 * afterwards waits for it (synchronise `stream` before reading out).  The
 * result equals gdr_kkt_solve_ex's, bit for bit whenever every chunk's
 * log-gate lies within 30 of the midpoint of its first and last value (the
 * kernel's factored gate), else to rounding.
 *   Host memory: page-locked buffers let the copies run asynchronously and
 *          overlap; pageable ones work, without the overlap.
 *   Streams: the two internal streams and three events per device are created
 *          on the first call on that device and kept until exit.  Calls on one
 *          device enqueue one at a time.  The call is not meant for stream
 *          capture.
 *   Errors: every check of gdr_kkt_solve_ex, plus GDR_ERR_NULL (workspace),
 *          GDR_ERR_SHAPE (workspace too small), GDR_ERR_ALIGN (workspace), all
 *          before anything is enqueued.
 */
int gdr_kkt_solve_host(const void *k, int k_dtype, const float *g, const void *beta, int beta_dtype,
                       const int32_t *cu_seqlens, int64_t B, int64_t T, int64_t H, int64_t K, int chunk_size,
                       int out_dtype, void *out, void *workspace, int64_t workspace_bytes, void *stream);

/* Device workspace bytes gdr_kkt_solve_host needs (for fixed-length and packed
 * inputs alike; room for beta in any type), or a negative gdr_status for
 * invalid types or sizes. */
int64_t gdr_kkt_solve_host_workspace_bytes(int k_dtype, int64_t B, int64_t T, int64_t H, int64_t K,
                                           int chunk_size, int out_dtype);

/*
 * gdr_check_cu_seqlens - device-side check of the packed-sequence contract that
 * gdr_kkt_solve and the other calls take on trust (no counterpart on the pages,
 * which only show that varlen bookkeeping is where mistakes hide: MindSpeed-Ops
 * PR #135 page, bot summary, the T_local fix).  The calls' tile schedule
 * assumes cu[0] = 0, cu[n] <= cu[n+1] for every n < B, and cu[B] <= T; a
 * broken array cannot make them write outside `out` or read outside the
 * inputs, but chunks of the misdescribed sequences are then silently skipped.
 * This call enqueues one small kernel on `stream` that reads cu_seqlens[0..B]
 * (device memory, 4-byte aligned) and, when any of the three conditions fails,
 * records GDR_ERR_CU_SEQLENS in the device status word (read and cleared by
 * gdr_kkt_solve_device_status; an earlier unread status is kept).  It never
 * traps and writes nothing else.  Opt-in: enqueue it before the call it guards,
 * on the same stream.  Returns GDR_OK when enqueued (also for B = 0, which
 * checks cu[0] only), GDR_ERR_NULL, GDR_ERR_ALIGN, GDR_ERR_SHAPE (B or T
 * negative or B >= 2^31), GDR_ERR_DEVICE or GDR_ERR_CUDA.
 */
int gdr_check_cu_seqlens(const int32_t *cu_seqlens, int64_t B, int64_t T, void *stream);

/* Human-readable text for a gdr_status value (static storage, never NULL). */
const char *gdr_status_string(int status);

/*
 * gdr_kkt_solve_device_status - reads the device-side status word of the
 * current device and resets it to GDR_OK.  Synchronises the current device.
 * The kernel's pipeline waits are bounded; if one ever runs out (a defect, not
 * an input error), the kernel stops early, leaves its outputs incomplete and
 * records GDR_ERR_TIMEOUT here.  Writes the recorded status to *status and
 * returns GDR_OK, or GDR_ERR_NULL / GDR_ERR_CUDA.
 */
int gdr_kkt_solve_device_status(int *status);

/*
 * gdr_selftest_bounded_wait - test hook for the failure path above (no
 * counterpart on the pages).  Enqueues a one-thread kernel on `stream` that
 * waits, through the kernels' own bounded wait but with a 20 ms limit, on a
 * barrier phase that nothing completes; the wait runs out and the kernel
 * records GDR_ERR_TIMEOUT in the device status word and returns normally, so
 * the context stays usable.  A following gdr_kkt_solve_device_status reports
 * GDR_ERR_TIMEOUT.  Returns GDR_OK when enqueued.
 */
int gdr_selftest_bounded_wait(void *stream);

/*
 * gdr_kkt_solve_num_sms - number of persistent CTAs one call launches at most
 * on the current device (one per SM).  Returns a negative gdr_status on error.
 */
int gdr_kkt_solve_num_sms(void);

#ifdef __cplusplus
}
#endif

#endif /* GDR_KKT_SOLVE_H */

/*
 * txl.h - C ABI of the GB300 (sm_103a) Transformer-XL relative-position
 * attention library.
 *
 * The operations follow "Transformer-XL: Attentive Language Models Beyond a
 * Fixed-Length Context" (Dai et al.):
 *   - §3.2, segment-level recurrence: the hidden states of earlier segments are
 *     cached (a memory of length M per layer) and prepended, without gradient,
 *     to the current segment as extended context for keys and values;
 *   - §3.3, the relative score
 *       A_ij = q_i.k_j + q_i.W_kR R_{i-j} + u.k_j + v.W_kR R_{i-j}
 *     with the sinusoid table R, then a masked softmax over the extended
 *     context and a product with the values (the N-layer summary);
 *   - Appendix B, the reversed table Q_k = W_kR R_{M+L-1-k} and the left shift
 *     that turns q Q^T into the position term, which the kernel realises by
 *     index arithmetic inside its tiles.
 *
 * Conventions for every entry point:
 *   - All pointers are device pointers unless stated otherwise.  The caller owns
 *     every buffer; the library keeps no reference after the call returns.
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL is the legacy default
 *     stream) and the call returns once it is launched.  Inputs must stay valid
 *     and unmodified until the stream reaches the work.
 *   - Arguments are validated on the host before anything is launched; a bad
 *     argument returns an error code and enqueues nothing.
 *   - Kernels that wait on on-chip barriers give up after a time limit and
 *     record TXL_ERR_TIMEOUT in a device status word; txl_device_status()
 *     reads and clears it.
 *   - Return values are txl_status codes (0 = success).
 */
#ifndef TXL_H
#define TXL_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    TXL_OK = 0,
    TXL_ERR_INVALID_ARG = -1, /* null pointer, negative size, bad dtype code */
    TXL_ERR_UNSUPPORTED = -2, /* a shape or dtype the library has no kernel for */
    TXL_ERR_MISALIGNED = -3,  /* a pointer breaks the stated alignment */
    TXL_ERR_SHAPE = -4,       /* sizes inconsistent with each other */
    TXL_ERR_CUDA = -5,        /* a CUDA runtime or driver call failed */
    TXL_ERR_TIMEOUT = -6,     /* a kernel gave up waiting on an on-chip barrier */
    TXL_ERR_WORKSPACE = -7,   /* workspace missing or too small for the request */
    TXL_ERR_INDEX = -8        /* a device-side index check failed (debug builds only) */
} txl_status;

typedef enum {
    TXL_F32 = 0, /* IEEE binary32 */
    TXL_BF16 = 1 /* bfloat16 */
} txl_dtype;

/* Human-readable name of a status code (static string, never NULL). */
const char *txl_status_string(int status);

/* Library version: major*10000 + minor*100 + patch. */
int txl_version(void);

/*
 * txl_rel_pos_emb - the sinusoid relative encoding table R of §3.3 ("R is a
 * sinusoid encoding matrix without learnable parameters"; row p stands for a
 * relative distance of p), written in Appendix B's reversed row order.
 *
 *   R     [K][d_model], dtype `dtype` (TXL_F32 or TXL_BF16), row-major.
 *         Row rho holds distance p = K-1-rho:
 *           R[rho][2k]   = sin(p * w_k),  R[rho][2k+1] = cos(p * w_k),
 *           w_k = 10000^(-2k/d_model).
 *         Multiplying by W_kR^T gives the per-head operand `r` of
 *         txl_relattn_fwd.
 *   K >= 1, d_model even and >= 2.  R must be 4-byte aligned.
 * Errors: TXL_ERR_INVALID_ARG (null R, K < 1, odd or non-positive d_model,
 * bad dtype), TXL_ERR_MISALIGNED, TXL_ERR_CUDA.
 */
int txl_rel_pos_emb(void *R, int K, int d_model, int dtype, void *stream);

/*
 * txl_relattn_workspace_size - bytes of device workspace txl_relattn_fwd needs
 * when it splits the key range of a head over `n_splits` thread blocks
 * (n_splits <= 1 needs none).  Pure host arithmetic.
 */
size_t txl_relattn_workspace_size(int B, int H, int L, int dh, int n_splits);

/* Kernels txl_relattn_fwd may run (reported by txl_relattn_plan). */
typedef enum {
    TXL_KERNEL_TC = 1,     /* bf16: tensor cores (tcgen05, TMEM, TMA), 128-row query tiles */
    TXL_KERNEL_DECODE = 2, /* bf16, L = 1: split-K decode kernel on the CUDA cores, fp32 */
    TXL_KERNEL_F32 = 3,    /* fp32: CUDA cores */
    TXL_KERNEL_DECODE_MMA = 4 /* bf16, 2 <= L <= 8: split-K decode kernel, warp-level tensor-core MMAs */
} txl_kernel;

/*
 * txl_relattn_plan - the kernel and the split txl_relattn_fwd would use for a
 * call with these arguments and a workspace of `workspace_bytes` bytes (0 = no
 * workspace; a non-zero size stands for a 256-byte aligned workspace).  Host
 * arithmetic plus cached device attributes of the current device; launches
 * nothing.
 *   *kernel  a txl_kernel value
 *   *splits  key ranges per query tile (TXL_KERNEL_TC) or per (b, h)
 *            (TXL_KERNEL_DECODE, TXL_KERNEL_DECODE_MMA); 1 for TXL_KERNEL_F32
 * Returns the status the call would return for its sizes (TXL_ERR_WORKSPACE
 * when the split needs more workspace than given), or TXL_ERR_INVALID_ARG for
 * NULL outputs.
 */
int txl_relattn_plan(int B, int H, int M, int L, int r_rows, int dh, int dtype, int n_splits,
                     size_t workspace_bytes, int *kernel, int *splits);

/*
 * txl_relattn_fwd - forward relative-position attention of one layer over the
 * extended context (§3.2 recurrence, §3.3 score and N-layer summary,
 * Appendix B shift).
 *
 * With K = M + L keys (memory rows first, then the segment), for every batch
 * b, head h, query i in [0,L) and key j in [0,K):
 *   delta  = M + i - j                        (relative distance)
 *   A_ij   = scale * ((q_i + u).k_j + (q_i + v_bias).r[row(delta)])  if delta >= 0
 *   A_ij   = -inf                                                     otherwise
 *   out_i  = sum_j softmax_j(A_i.) v_j,   lse_i = log sum_j exp(A_ij)
 * where r[row] = W_kR R_{distance} in Appendix B's reversed order: with
 * r_rows rows per head, row(delta) = r_rows - 1 - delta.  A table built for
 * exactly K keys has r_rows = K; a longer table (r_rows > K, e.g. cached for the
 * largest memory) is used as is.
 *
 * Layouts (dense, row-major, innermost dimension dh contiguous):
 *   q   [B][H][L][dh]        k, v [B][H][K][dh]
 *   r   [H][r_rows][dh]      u, v_bias [H][dh]
 *   out [B][H][L][dh]        lse [B][H][L] fp32, natural log (may be NULL)
 * dtype TXL_BF16: q, k, v, r, u, v_bias and out are bf16; scores, softmax and
 *   accumulation are fp32 on the tensor cores (tcgen05).  dh must be 64; q, k,
 *   v and r must be 16-byte aligned.  Segments of L <= 8 queries (decoding a
 *   few new tokens against a long memory) always take a split-K decode kernel
 *   instead: from L = 2 on the tensor cores' warp-level MMAs with q + u, q + v
 *   and P each carried as a bf16 pair (value and residual), for L = 1 the CUDA
 *   cores in fp32; either way the error before the output's bf16 rounding is
 *   far below that rounding (txl_relattn_plan tells which kernel).  For it n_splits
 *   counts key ranges per (b, h), each a whole number of 32-key chunks,
 *   at most one per 128 keys (larger requests are capped, ranges that would
 *   hold no key are dropped); up to 8 ranges of a head run as one thread-block
 *   cluster and merge in distributed shared memory, needing no workspace.
 * dtype TXL_F32: every tensor is fp32 and the arithmetic is fp32 on the CUDA
 *   cores (no TF32).  dh must be 64.
 * M >= 0, L >= 1, r_rows >= K, B >= 1, H >= 1.
 *
 * n_splits: 0 lets the library choose; 1 processes each head's keys in one
 * thread block; n > 1 splits the key range over n blocks and merges their
 * partial results (needs txl_relattn_workspace_size(B,H,L,dh,n) bytes of
 * workspace, 256-byte aligned, owned by the caller, contents undefined on
 * return).  A workspace that is NULL or too small limits the automatic choice
 * to 1 and makes an explicit n > 1 fail with TXL_ERR_WORKSPACE.
 *
 * Errors: TXL_ERR_INVALID_ARG, TXL_ERR_UNSUPPORTED (dh != 64, bad dtype),
 * TXL_ERR_MISALIGNED, TXL_ERR_SHAPE (r_rows < K), TXL_ERR_WORKSPACE,
 * TXL_ERR_CUDA.
 */
int txl_relattn_fwd(const void *q, const void *k, const void *v, const void *r, int r_rows,
                    const void *u, const void *v_bias, void *out, float *lse, int B, int H,
                    int M, int L, int dh, float scale, int dtype, int n_splits,
                    void *workspace, size_t workspace_bytes, void *stream);

/*
 * txl_relattn_fwd_strided - txl_relattn_fwd with the (b, h) planes of k and v
 * kv_stride elements apart instead of K * dh, so that the K = M + L keys of each
 * plane can be a window of a larger buffer (the memory of §3.2 kept in place,
 * the segment's rows written behind it; see txl_kv_window below) and nothing
 * has to be concatenated before the call.
 *
 *   k, v  plane p = b*H + h starts at k + p * kv_stride (elements); within a
 *         plane the K rows of dh elements are contiguous, memory rows first.
 *         Only those K rows of each plane are read.
 *   kv_stride >= K * dh and a multiple of 8 (16 bytes of bf16: every plane
 *         starts 16-byte aligned when k and v do).
 * Everything else (q, r, u, v_bias, out, lse, n_splits, workspace, the
 * kernels, results and errors) is as for txl_relattn_fwd, which is this call
 * with kv_stride = K * dh.
 * Errors: those of txl_relattn_fwd; TXL_ERR_INVALID_ARG for kv_stride < 1,
 * TXL_ERR_SHAPE for kv_stride < K * dh, TXL_ERR_MISALIGNED for a kv_stride not
 * a multiple of 8.
 */
int txl_relattn_fwd_strided(const void *q, const void *k, const void *v, long long kv_stride,
                            const void *r, int r_rows, const void *u, const void *v_bias,
                            void *out, float *lse, int B, int H, int M, int L, int dh,
                            float scale, int dtype, int n_splits, void *workspace,
                            size_t workspace_bytes, void *stream);

/*
 * TXL_NOALLOC_SCRATCH_BYTES - size of the scratch array built into the library
 * for txl_relattn_fwd_noalloc (32 MiB).
 */
#define TXL_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)

/*
 * txl_relattn_fwd_noalloc - txl_relattn_fwd for callers that cannot allocate
 * device memory when they run it (for example plugins of inference engines
 * whose execute step must not allocate, or runtimes whose device memory budget
 * is fixed at start-up).  The paper has no counterpart: this is a property of
 * the library, not of the method.
 *
 * Same arguments, layouts, results and errors as txl_relattn_fwd, without the
 * workspace.  When a head's key range is split over several blocks, the
 * partial results go to a scratch array that is part of the library: one
 * device array of TXL_NOALLOC_SCRATCH_BYTES that every GPU which loads the
 * library holds until the process exits.  The call itself allocates nothing
 * (no cudaMalloc, cudaFree or allocating library routine).
 *   - A split whose partial results need more than the scratch returns
 *     TXL_ERR_WORKSPACE and launches nothing.  What counts is the split the
 *     call runs, as txl_relattn_plan reports it for workspace_bytes =
 *     TXL_NOALLOC_SCRATCH_BYTES: requests above the key-tile count are capped
 *     first, and decode key ranges merged inside a thread-block cluster need
 *     no scratch; otherwise it needs txl_relattn_workspace_size(B, H, L, dh,
 *     splits) bytes.  n_splits = 0 chooses a split that fits (or none).
 *   - Every call shares the array and leaves its partial results in it; calls
 *     that may run at the same time on the GPU (other streams, or other host
 *     threads without ordering) race on it and must be serialised by the
 *     caller.
 *   - The first call on a device looks up the array's device address (a
 *     runtime query, done once per device with that device current); make that
 *     first call before any stream capture.
 */
int txl_relattn_fwd_noalloc(const void *q, const void *k, const void *v, const void *r,
                            int r_rows, const void *u, const void *v_bias, void *out, float *lse,
                            int B, int H, int M, int L, int dh, float scale, int dtype,
                            int n_splits, void *stream);

/*
 * Segment memory of one layer (§3.2: "cache a predefined length-M old hidden
 * states spanning (possibly) multiple segments"), kept as a ring buffer.
 *
 *   mem  [B][capacity][d] on the device, owned by the caller.
 *   txl_mem_state lives in HOST memory and is owned by the caller:
 *     head     slot that receives the next row
 *     fill     rows currently held (0..capacity)
 *     capacity M, the memory length
 * Logical row t (0 = oldest) of the fill rows sits in slot
 * (head - fill + t) mod capacity.  Initialise with {0, 0, M}.
 */
typedef struct {
    int head;
    int fill;
    int capacity;
} txl_mem_state;

/*
 * txl_mem_concat - the extended context h~ = [SG(m) o h] of §3.2 / §3.3 for
 * the current segment: ext[b] = the fill memory rows oldest-first, then the L
 * rows of h_new.  SG (stop-gradient) is the identity in a forward pass.
 *   ext   [B][fill + L][d]   h_new [B][L][d]   same dtype (TXL_F32 / TXL_BF16)
 * Rows are copied in 16-byte units: d * element size must be a multiple of 16
 * and every pointer 16-byte aligned.
 * Errors: TXL_ERR_INVALID_ARG, TXL_ERR_MISALIGNED, TXL_ERR_SHAPE, TXL_ERR_CUDA.
 */
int txl_mem_concat(void *ext, const void *mem, const txl_mem_state *st, const void *h_new,
                   int B, int L, int d, int dtype, void *stream);

/*
 * txl_mem_update - advance the memory with the current segment's states:
 * the memory becomes the newest `capacity` rows of [m o h_new] (§3.2, the
 * summary's m^n_tau).  Writes at most min(L, capacity) rows into the ring and
 * updates *st on the host (head advances by L mod capacity, fill saturates at
 * capacity).  Same layout and alignment rules as txl_mem_concat.
 * Errors: TXL_ERR_INVALID_ARG, TXL_ERR_MISALIGNED, TXL_ERR_SHAPE, TXL_ERR_CUDA;
 * *st is unchanged on error.
 */
int txl_mem_update(void *mem, txl_mem_state *st, const void *h_new, int B, int L, int d,
                   int dtype, void *stream);

/*
 * A memory of §3.2 ("a predefined length-M old hidden states spanning
 * (possibly) multiple segments") kept as a contiguous window of a larger
 * buffer, one window per plane (e.g. the projected keys or values of each
 * (batch, head)), so that [memory ; segment] is read in place by
 * txl_relattn_fwd_strided.
 *
 *   buf   [planes][capacity][d] on the device, owned by the caller.
 *   txl_kv_window lives in HOST memory and is owned by the caller:
 *     start     row of the oldest memory row in every plane
 *     fill      memory rows held (0..M)
 *     capacity  rows per plane of buf; at least 2 * M + L for segments of L rows
 *     M         memory length
 * Initialise with {0, 0, capacity, M}.  Per segment:
 *   txl_kv_window_append  puts the segment's L rows behind the memory rows;
 *                         afterwards rows [start, start + fill + L) of every
 *                         plane are [memory ; segment] (K = fill + L keys, at a
 *                         plane stride of capacity * d elements);
 *   (attention over that window)
 *   txl_kv_window_advance keeps the newest M rows as the memory (host only).
 */
typedef struct {
    int start;
    int fill;
    int capacity;
    int M;
} txl_kv_window;

/*
 * txl_kv_window_append - copy seg [planes][L][d] into rows start + fill ..
 * start + fill + L - 1 of every plane.  When those rows would run past the
 * buffer's end, the fill memory rows are first copied to rows 0 .. fill - 1 and
 * start becomes 0 (with capacity >= 2M + L the two ranges never overlap).
 * Same dtype and 16-byte rules as txl_mem_update.  Updates w->start on the host.
 * Errors: TXL_ERR_INVALID_ARG (bad state, sizes, pointers or dtype),
 * TXL_ERR_SHAPE (capacity < 2M + L), TXL_ERR_MISALIGNED, TXL_ERR_CUDA; *w is
 * unchanged on error.
 */
int txl_kv_window_append(void *buf, txl_kv_window *w, const void *seg, int planes, int L, int d,
                         int dtype, void *stream);

/*
 * txl_kv_window_advance - after attending to a segment of L rows appended by
 * txl_kv_window_append: the memory becomes the newest min(fill + L, M) rows of
 * [memory ; segment] (§3.2, the summary's m^n_tau).  Host arithmetic only.
 * Errors: TXL_ERR_INVALID_ARG (bad state, L < 0), TXL_ERR_SHAPE (the window
 * would run past the buffer: the segment was not appended).
 */
int txl_kv_window_advance(txl_kv_window *w, int L);

/*
 * txl_qkv_project - one layer's projections for a segment, written where the
 * attention reads them, with the memory update in the same launch ("Transformer-XL:
 * Attentive Language Models Beyond a Fixed-Length Context", §3.3 N-layer
 * summary: q = h W_q^T and k, v = h~ W_kE^T, h~ W_v^T, of which only the
 * segment's rows are new when the memory's k and v are kept in a window; §3.2:
 * the memory takes the newest states).  One GEMM, Y = h W^T over the stacked
 * weights, on the tensor cores (bf16 in, fp32 accumulate, bf16 out), whose
 * epilogue writes
 *   q      [B][H][L][dh]                               (when q != NULL)
 *   k, v   rows start + fill .. start + fill + L - 1 of the window planes of
 *          kv_buf: keys in planes 0 .. B*H-1, values in planes B*H .. 2*B*H-1
 *          ([2*B*H][capacity][dh], plane = b*H + h), exactly as
 *          txl_kv_window_append would place them (moving the memory rows to
 *          the buffer's front first when needed; updates kv_win->start)
 *   mem    the memory ring [B][capacity][d_model] advanced as txl_mem_update
 *          would (when mem != NULL; updates *mem_st)
 * h [B][L][d_model]; w [n_out * H * dh][d_model] with n_out = 3 (rows W_q,
 * W_kE, W_v, head-major inside each) when q != NULL, else 2 (W_kE, W_v).
 * All bf16, dense, 16-byte aligned; dh must be 64 and d_model a multiple of 8.
 * The caller owns every buffer and both states (host memory).  Asynchronous on
 * `stream`.  Errors: TXL_ERR_INVALID_ARG (NULL h, w, kv_buf or kv_win, bad
 * sizes or states, mem without mem_st), TXL_ERR_UNSUPPORTED (dh != 64),
 * TXL_ERR_SHAPE (window capacity < 2M + L, ring row width), TXL_ERR_MISALIGNED,
 * TXL_ERR_CUDA; the states are unchanged on error.
 */
int txl_qkv_project(const void *h, const void *w, int B, int L, int d_model, int H, int dh,
                    void *q, void *kv_buf, txl_kv_window *kv_win, void *mem,
                    txl_mem_state *mem_st, void *stream);

/*
 * txl_relattn_bwd - backward of txl_relattn_fwd for one segment (training
 * backpropagates within a segment, "Transformer-XL: Attentive Language Models
 * Beyond a Fixed-Length Context" §3.2; the memory is SG(m): no gradient leaves
 * through it, but its projected keys and values receive one like the
 * segment's).  With A_ij the §3.3 score times `scale`, P = softmax_j(A) over
 * the kept keys (j <= i + M), O = P v and dout = dL/dO:
 *   D_i   = sum_j P_ij (dout_i . v_j)
 *   g_ij  = scale P_ij (dout_i . v_j - D_i)
 *   dq_i  = sum_j g_ij (k_j + r(M+i-j))       dk_j = sum_i g_ij (q_i + u)
 *   dv_j  = sum_i P_ij dout_i                 du   = sum_{b,i,j} g_ij k_j
 *   dr(d) = sum_{b, i-j = d-M} g_ij (q_i + v) dv_bias = sum_{b,i,j} g_ij r(M+i-j)
 * where r(d) is the table row of distance d (row r_rows - 1 - d of r).  P is
 * recomputed; so are its log-sum-exp and D (exactly, in fp32): nothing from the
 * forward call is needed.
 * Inputs, bf16, dense and 16-byte aligned, layouts as txl_relattn_fwd:
 *   q, dout [B][H][L][dh]   k, v [B][H][M+L][dh]   r [H][r_rows][dh]
 *   u, v_bias [H][dh]
 * Outputs, fp32, dense, written (not accumulated), 16-byte aligned:
 *   dq [B][H][L][dh]   dk, dv [B][H][M+L][dh]   dr [H][r_rows][dh] (rows of
 *   distances >= M+L are zero)   du, dv_bias [H][dh]
 * workspace: txl_relattn_bwd_workspace_size(B, H, L, M) bytes of device
 * memory, 256-byte aligned (per-row statistics, per-block bias and dq
 * partials, and g of every query-key pair: B*H*L rows of M+L rounded up to 64
 * fp32, from which the table gradient is summed); 0 for sizes out of range.  The sums
 * over the batch and the key splits are ordered, so results repeat bit for
 * bit.  dh must be 64 and dtype
 * TXL_DTYPE_BF16.  Asynchronous on `stream`.  Errors: TXL_ERR_INVALID_ARG
 * (NULL pointer, bad sizes), TXL_ERR_UNSUPPORTED (dh, dtype, sizes past the
 * grid limits), TXL_ERR_SHAPE (r_rows < M+L), TXL_ERR_MISALIGNED,
 * TXL_ERR_WORKSPACE, TXL_ERR_CUDA.
 */
size_t txl_relattn_bwd_workspace_size(int B, int H, int L, int M);
int txl_relattn_bwd(const void *q, const void *k, const void *v, const void *r, int r_rows,
                    const void *u, const void *v_bias, const void *dout, float *dq, float *dk,
                    float *dv, float *dr, float *du, float *dv_bias, int B, int H, int M, int L,
                    int dh, float scale, int dtype, void *workspace, size_t workspace_bytes,
                    void *stream);

/*
 * txl_device_status - synchronise `stream`, then read and clear the device
 * status word in which kernels record barrier time-outs (and, in a debug
 * build, failed index checks).  Returns TXL_OK, TXL_ERR_TIMEOUT (a time-out was
 * recorded), TXL_ERR_INDEX (only failed index checks were) or TXL_ERR_CUDA.
 */
int txl_device_status(void *stream);

/*
 * txl_set_wait_limit_ns - time limit, in nanoseconds, after which a kernel's
 * on-chip barrier wait gives up (default 1e9).  Applies to later launches from
 * this process.  Returns the previous value.
 */
uint64_t txl_set_wait_limit_ns(uint64_t ns);

/*
 * txl_debug_wait_timeout - launch one small kernel that waits on a barrier no
 * one will complete, with the time limit `ns`; it must give up, record the
 * time-out and return.  Lets a test check the time-out path without hanging
 * anything.  Returns the status txl_device_status() reports afterwards
 * (TXL_ERR_TIMEOUT when the path works).
 */
int txl_debug_wait_timeout(uint64_t ns, void *stream);

/*
 * Debug build.  A library compiled with -DTXL_DEBUG checks, inside its kernels,
 * the index arithmetic of the hot path (work split of each block, every row of
 * the shared-memory ring that applies the Appendix B shift, TMEM columns of the
 * table chunks, output rows, decode key and table ranges, memory ring slots and
 * window rows).  A failed check records TXL_ERR_INDEX in the device status word
 * and the kernel goes on: nothing traps.  Release builds compile the checks
 * away.
 *
 * txl_debug_checks - 1 in a debug build, 0 otherwise.
 * txl_debug_index_probe - launch one small kernel that fails one check on
 *   purpose, then return txl_device_status(stream): TXL_ERR_INDEX in a debug
 *   build (the reporting path works), TXL_OK in a release build.
 */
int txl_debug_checks(void);
int txl_debug_index_probe(void *stream);

#ifdef __cplusplus
}
#endif

#endif /* TXL_H */

/*
 * fa.h -- C ABI of the GB300 (sm_103a) exact-attention library, libfa_gb300.so.
 *
 * What is computed (tensortonic.com "FlashAttention", sections 1, 4-7;
 * wiki.ai-engineering.at "Flash Attention", The Core Problem):
 *
 *     S = scale * Q K^T  (+ causal mask: key j allowed for query i iff j <= i)
 *     O = softmax_rows(S) V
 *     L_i = m_i + log(l_i)  = log sum_j exp(S_ij)        (natural log)
 *
 * computed tile by tile with a running (m, l, u) state per query row; the
 * n x n score matrix is never written to device memory.  The backward pass
 * rebuilds every weight as P_ij = exp(S_ij - L_i) (section 7) and forms
 *
 *     D_i = rowsum(dO o O),  dS = P o (dO V^T - D),
 *     dV = P^T dO,  dQ = scale * dS K,  dK = scale * dS^T Q.
 *
 * Layouts (all row-major, contiguous, element strides implied):
 *   dense  (cu_seqlens == NULL): Q, K, V, O, dO, dQ, dK, dV are [B, H, N, D];
 *          lse is [B, H, N] float32.
 *   packed (cu_seqlens != NULL): B sequences packed along one token axis of
 *          length total_tokens = cu_seqlens[B]; tensors are [H, total_tokens, D]
 *          and lse is [H, total_tokens].  Sequence s owns tokens
 *          cu_seqlens[s] .. cu_seqlens[s+1]-1 of every head and attends only
 *          within itself.  N is the maximum sequence length (grid sizing only).
 *   Causal alignment is square / top-left within each sequence.
 *
 * Types: FA_BF16 -- Q, K, V, O, dO, dQ, dK, dV are bfloat16; arithmetic is
 *          tcgen05 tensor-core bf16 x bf16 -> fp32 for the five contractions,
 *          fp32 for softmax; head width D must be 64 or 128.
 *        FA_F32  -- all of them float32; arithmetic is fp32 FMA (no TF32);
 *          D must be 32, 64 or 128.
 *        FA_F16  -- as FA_BF16 with IEEE half precision tensors (fp16 x fp16
 *          -> fp32 tensor-core products; P and dS are rounded to fp16 before
 *          their products); D must be 64 or 128.  (The 16-bit input type
 *          of nexusofnerds.com "FlashAttention"; the pages give no separate
 *          tolerance for it.)
 *        lse is always float32.
 *
 * Ownership and memory: every pointer argument is a DEVICE pointer owned by the
 * caller (except where stated); the library allocates no device memory and
 * keeps no state beyond cached per-device properties and a per-device status
 * word.  All pointers to tensors must be 16-byte aligned.
 *
 * Asynchrony: fa_fwd and fa_bwd validate their arguments on the host, enqueue
 * kernels on `stream` (a cudaStream_t; NULL = legacy default stream) and
 * return without waiting.  A return of FA_OK means "enqueued".  Faults the
 * kernels detect themselves (malformed cu_seqlens, a bounded wait that ran
 * out) are latched in a per-device status word read by
 * fa_get_last_device_error.
 *
 * CUDA graphs: fa_fwd, fa_bwd, fa_fwd_dropout, fa_bwd_dropout,
 * fa_bwd_deterministic and fa_decode enqueue no host synchronisation and no
 * allocation, and pass their work lists by value in the kernel parameters, so
 * a stream capture of them replays correctly on new contents of the same
 * buffers.  Make one eager call of each first: it performs the one-time
 * per-device look-ups (status word address, tensor-map encoder).  A captured
 * backward reuses its workspace on every replay (its tile counter is reset by
 * the replay itself); replays that overlap on the GPU need workspaces of their
 * own, as overlapping eager calls do.  Dropout replays the captured seed and
 * offset.
 *
 * Errors: invalid arguments return an error code before anything is launched;
 * nothing aborts the process.
 */
#ifndef FA_GB300_H
#define FA_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FA_OK = 0,
  FA_ERR_INVALID = -1,      /* NULL pointer, negative size, scale not finite and > 0, bad cu_seqlens */
  FA_ERR_UNSUPPORTED = -2,  /* head width or dtype this build has no kernel for */
  FA_ERR_ALIGN = -3,        /* a tensor pointer is not 16-byte aligned */
  FA_ERR_CUDA = -4,         /* a CUDA runtime/driver call failed (launch, tensor map) */
  FA_ERR_TIMEOUT = -5,      /* a kernel's bounded wait expired (reported by fa_get_last_device_error) */
  FA_ERR_WORKSPACE = -6     /* workspace NULL, misaligned or smaller than fa_bwd_workspace_size */
} fa_status;

typedef enum { FA_BF16 = 0, FA_F32 = 1, FA_F16 = 2 } fa_dtype;

/*
 * Forward pass.  tensortonic.com "FlashAttention" sections 5-7.
 *   q, k, v       in : [B,H,N,D] (dense) or [H,T,D] (packed), dtype
 *   o             out: same layout and dtype as q; O = u / l rounded to nearest
 *   lse           out: float32 [B,H,N] or [H,T]; natural-log L = m + log(l)
 *   B, H, N, D    batch (or number of packed sequences), heads, tokens (or max
 *                 sequence length when packed), head width; B, H, N >= 0
 *   scale         multiplies Q K^T before the mask and softmax (1/sqrt(D) is
 *                 the usual value); must be finite and > 0 (FA_ERR_INVALID
 *                 otherwise: the kernels take each row's maximum over the
 *                 unscaled scores, which is the maximum of the scaled ones only
 *                 for a positive scale)
 *   causal        0 = full attention, 1 = key j allowed for query i iff j <= i
 *   cu_seqlens    NULL for dense; else DEVICE int32[B+1], non-decreasing,
 *                 cu_seqlens[0] = 0, cu_seqlens[B] = total_tokens, every
 *                 length <= N.  A violation found on the device skips that
 *                 sequence and latches FA_ERR_INVALID.
 *   total_tokens  T for packed input (ignored when cu_seqlens == NULL)
 *   stream        cudaStream_t
 * Rows of a packed sequence of length 0 produce nothing.
 */
fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                 int B, int H, int N, int D, float scale, int causal,
                 const int32_t* cu_seqlens, int total_tokens,
                 fa_dtype dtype, void* stream);

/*
 * Bytes of device workspace fa_bwd needs: D_i (float32 per row) and, for the
 * tensor-core path, a float32 dQ accumulator of the shape of Q and a 256-byte
 * block holding the counter from which the backward's CTAs take key tiles
 * (each part rounded up to 256 bytes).  Pure host arithmetic; never fails
 * (returns 0 for invalid sizes).
 */
size_t fa_bwd_workspace_size(int B, int H, int N, int D, const int32_t* cu_seqlens,
                             int total_tokens, fa_dtype dtype);

/*
 * Backward pass.  tensortonic.com "FlashAttention" section 7 (weights rebuilt
 * as exp(s_ij - L_i)); gradient algebra in the file header.
 *   q, k, v, o    in : as passed to / produced by fa_fwd
 *   lse           in : float32 L from fa_fwd
 *   dout          in : upstream gradient dO, same layout and dtype as o
 *   dq, dk, dv    out: gradients, same layout and dtype as q (overwritten)
 *   workspace     DEVICE scratch of at least fa_bwd_workspace_size(...)
 *                 bytes, 256-byte aligned, owned by the caller; its contents
 *                 on entry do not matter; calls sharing a workspace must not
 *                 overlap on the device
 *   other arguments as for fa_fwd
 * dK and dV are written deterministically; dQ is accumulated in float32 with
 * atomic adds on the tensor-core path, so its last bits may vary run to run.
 */
fa_status fa_bwd(const void* q, const void* k, const void* v, const void* o,
                 const float* lse, const void* dout,
                 void* dq, void* dk, void* dv,
                 int B, int H, int N, int D, float scale, int causal,
                 const int32_t* cu_seqlens, int total_tokens, fa_dtype dtype,
                 void* workspace, size_t workspace_bytes, void* stream);

/*
 * Backward pass for callers that cannot allocate device memory.  The pages
 * have no counterpart: this is a deployment convenience, not a step of the
 * method.
 *
 * fa_bwd needs scratch (D_i per row and, for bf16, a float32 dQ accumulator)
 * that the caller allocates.  Some callers cannot: a plugin inside a host
 * application that owns all device memory through its own pool and forbids
 * direct cudaMalloc, or a latency-critical loop that must not pay for a
 * cudaMalloc (which may synchronise the device).  fa_bwd_static_ws takes the
 * same arguments as fa_bwd minus the workspace and uses instead a fixed
 * array of FA_BWD_STATIC_WS_BYTES that the library keeps in device memory on
 * every GPU that loads it, until the process exits.  It calls no allocator.
 *   - The first call on a device looks up that array's device address
 *     (cudaGetSymbolAddress, with that device current) and caches it for the
 *     device's current context; make that first call before any stream
 *     capture.  A device reset destroys the context and the array with it:
 *     the first call after one looks the address up again (again before any
 *     capture).
 *   - Problems whose fa_bwd_workspace_size exceeds FA_BWD_STATIC_WS_BYTES are
 *     rejected with FA_ERR_WORKSPACE before anything is launched
 *     (fa_last_error_detail says why).  The workspace takes 4 * (D + 1)
 *     bytes per row (rows = B*H*N dense, H*total_tokens packed; each of its
 *     two parts rounded up to 256 bytes) plus 256 bytes for bf16 / fp16 and 4
 *     bytes per row for float32, so 16 MiB holds at most 32,513 rows at
 *     D = 128, 64,526 rows at D = 64 and 4,194,304 rows in float32.
 *   - Every call on a device shares the one array.  Its previous contents do
 *     not matter (the backward rewrites D_i and zeroes the dQ accumulator
 *     before reading them), but calls that overlap on the GPU -- on different
 *     streams or from different host threads -- race on it and give wrong
 *     gradients.  Serialise them.
 * Results are those of fa_bwd with a caller workspace.
 */
#define FA_BWD_STATIC_WS_BYTES ((size_t)16 << 20)
fa_status fa_bwd_static_ws(const void* q, const void* k, const void* v, const void* o,
                           const float* lse, const void* dout,
                           void* dq, void* dk, void* dv,
                           int B, int H, int N, int D, float scale, int causal,
                           const int32_t* cu_seqlens, int total_tokens, fa_dtype dtype,
                           void* stream);

/* Static English text for a status code. */
const char* fa_strerror(fa_status status);

/*
 * Synchronises `stream`, then returns and clears the current device's latched
 * kernel status: FA_OK, FA_ERR_TIMEOUT (a bounded wait inside a kernel ran
 * out; the kernel stopped its work, released its tensor memory and returned)
 * or FA_ERR_INVALID (malformed cu_seqlens seen on the device).  Returns
 * FA_ERR_CUDA if the synchronisation itself fails, or if a kernel found its
 * launch environment unusable (it then skipped its work).
 */
fa_status fa_get_last_device_error(void* stream);

/*
 * Upper bound, in nanoseconds, on every bounded wait inside the kernels
 * (default 2e9 ns).  Applies to launches made after the call, on every device.
 * Values below 1000 are raised to 1000.
 */
void fa_set_wait_limit_ns(unsigned long long limit_ns);

/*
 * Failure-detection self-test: launches one CTA that waits, with the current
 * wait limit, on a shared-memory barrier nothing ever signals, then returns
 * fa_get_last_device_error(stream) -- FA_ERR_TIMEOUT when the bounded wait
 * works.  No fault, trap or hang is involved.
 */
fa_status fa_selftest_wait_timeout(void* stream);

/*
 * Unit check of the tensor-core building blocks on one tile, for tests: the
 * products the method is made of (tensortonic.com "FlashAttention", section
 * 5: scores S = Q K^T of a query tile against a key tile, then the weights of
 * that tile times its values) formed the way the kernels form them.  One CTA
 * loads a and b with TMA, forms S = a b^T in tensor memory, writes it to
 * s_out, rounds it to dtype and forms O = round(S) b with tensor-memory
 * operand A, writes O to o_out, and copies a back out of its swizzled
 * shared-memory tile into a_copy.
 *   a, b     in : DEVICE [128, D] row-major, dtype (FA_BF16 or FA_F16)
 *   s_out    out: DEVICE float32 [128, 128]
 *   o_out    out: DEVICE float32 [128, D]
 *   a_copy   out: DEVICE [128, D], dtype; equals a bit for bit when correct
 *   D        64 or 128 (FA_ERR_UNSUPPORTED otherwise, or for FA_F32)
 * Every pointer must be non-NULL (FA_ERR_INVALID) and 16-byte aligned
 * (FA_ERR_ALIGN).  Synchronises `stream` and returns
 * fa_get_last_device_error(stream); FA_ERR_CUDA if a launch fails.
 */
fa_status fa_selftest_tile(const void* a, const void* b, float* s_out, float* o_out, void* a_copy, int D,
                           fa_dtype dtype, void* stream);

/*
 * Name of the kernel family fa_fwd / fa_bwd launch for this dtype and head
 * width ("tcgen05" for bf16, "simt_f32" for float32), or NULL when
 * unsupported.  Host only.
 */
const char* fa_path_name(fa_dtype dtype, int D);

/*
 * Human-readable detail of the most recent FA_ERR_CUDA returned on the
 * calling host thread (which step failed and the CUDA error text); an empty
 * string when there is none.  The pointer stays valid until the next call on
 * this thread.
 */
const char* fa_last_error_detail(void);

/*
 * Instrumentation: the next fa_bwd call made on this host thread records
 * `start_event` (a cudaEvent_t) on its stream right before its main
 * gradient kernel and `stop_event` right after it, so a caller can time that
 * kernel alone (the preprocess and dQ conversion launches fall outside).
 * Either may be NULL.  The request is consumed by that call.
 */
void fa_bwd_time_main_kernel(void* start_event, void* stop_event);

/*
 * Instrumentation: measured throughput of the GPU's special-function units
 * for ex2.approx.f32, the instruction the kernels use for every attention
 * weight (tensortonic.com "FlashAttention", section 5: each weight is an
 * exponential of a shifted score).  Launches one CTA per SM in which every
 * thread runs 8 independent 2^(-x) recurrences for `iters` rounds (1 ..
 * 2^20) between two reads of the SM clock, waits for it, and writes the mean
 * over CTAs of exponentials per clock per SM to *ex2_per_clk_per_sm (host
 * pointer).  Synchronises `stream`.  FA_ERR_INVALID for a NULL pointer or
 * iters out of range, FA_ERR_CUDA if a CUDA call fails.
 */
fa_status fa_probe_ex2_rate(int iters, double* ex2_per_clk_per_sm, void* stream);

/*
 * Number of kernels this library has launched in this process (all devices,
 * all entry points, including failed launches it detected).  Host only.
 */
unsigned long long fa_launch_count(void);

/*
 * Host-only view of the work lists of the persistent tensor-core launches
 * (instrumentation and tests; no GPU needed).  kernel 0 = the forward, whose
 * items are pairs of 128-row query tiles; kernel 1 = the backward, whose
 * items are 128-key tiles.  D: the head width, 64 or 128.  cu_seqlens: NULL
 * for dense input, else a HOST copy of the packed offsets (int32[B+1]).  Two
 * forms (written to
 * *form): 0 = a table worked out on the host, for dense inputs of at most
 * 4096 items -- items in the order the one-CTA-per-item grid would hand them
 * out (heaviest first inside groups of heads -- one group of all heads when
 * the operands they re-read fit in L2 together, which depends on the head
 * width D), each to the CTA with the least work so far, at most
 * min(n_ctas, 160) CTAs; 1 = the forward's closed-form
 * list, for larger or packed inputs -- unit u = b * H + h, the units' items
 * rank-major (all units' heaviest first), CTA c of n = min(n_ctas,
 * B * H * ranks) taking virtual item k * n + c for even k and
 * k * n + n - 1 - c for odd k, skipping the ranks its sequence does not
 * have; 2 = the backward's queue, for larger or packed inputs -- one list,
 * in the order the CTAs take the tiles from a counter as they need them:
 * units in groups of about 4, each group's tiles rank-major (off[0] = 0,
 * off[i] = item count for i >= 1).
 * Item codes are u * R + pair (forward) or u * R + key tile (backward), with
 * R = ceil(ceil(N / 128) / 2) pairs or ceil(N / 128) key tiles.  Writes
 * off[0 .. c] (off must hold n_ctas + 1 entries; CTA i works on
 * items[off[i] .. off[i + 1]), in that order) and returns the number of
 * items; -1 for arguments out of range, -2 if `cap` is below the item count.
 */
int fa_schedule_preview(int kernel, const int32_t* cu_seqlens, int B, int H, int N, int D, int causal, int n_ctas,
                        int* off, unsigned int* items, int cap, int* form);

/* Attention dropout (tensortonic.com "FlashAttention" section 7: the backward
 * must reproduce the forward's dropout decisions from saved generator state).
 * Same arguments as fa_fwd / fa_bwd plus:
 *   p_drop  probability of dropping an attention weight, 0 <= p_drop < 1
 *           (FA_ERR_INVALID otherwise; 0 gives exactly fa_fwd / fa_bwd);
 *   seed, offset  select the decisions, which are regenerated, never stored:
 *           element (i, j) of head bh = b * H + h (i, j counted from the start
 *           of the element's own sequence) is kept iff word j mod 4 of the
 *           counter-based generator Philox4x32-10 (Salmon et al., SC 2011) on
 *           counter (j / 4, i, bh, offset) and key (seed mod 2^32, seed / 2^32),
 *           divided by 2^32, is >= p_drop.
 * Kept weights are scaled by 1 / (1 - p_drop): O = (P o Z) V / (1 - p_drop); lse
 * is that of the undropped softmax.  fa_bwd_dropout must get the same
 * p_drop, seed and offset as the forward that produced o.  Tensor-core path
 * only (bf16 / fp16, D 64 or 128): FA_ERR_UNSUPPORTED for float32 with
 * p_drop > 0. */
fa_status fa_fwd_dropout(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N,
                         int D, float scale, int causal, const int32_t* cu_seqlens, int total_tokens,
                         fa_dtype dtype, float p_drop, uint64_t seed, uint32_t offset, void* stream);
fa_status fa_bwd_dropout(const void* q, const void* k, const void* v, const void* o, const float* lse,
                         const void* dout, void* dq, void* dk, void* dv, int B, int H, int N, int D, float scale,
                         int causal, const int32_t* cu_seqlens, int total_tokens, fa_dtype dtype, float p_drop,
                         uint64_t seed, uint32_t offset, void* workspace, size_t workspace_bytes, void* stream);

/* Deterministic backward (not on the pages; a variant of the backward's dQ
 * step): the same gradients as fa_bwd / fa_bwd_dropout, but every sum is taken
 * in a fixed order, so repeated calls give bit-identical dq, dk, dv.  dK and
 * dV come from the key-stationary kernel without its dQ product; dQ from a
 * query-stationary kernel that accumulates each 128-query tile in tensor memory
 * over the key tiles (recomputing S and dP there) and writes it once, instead
 * of adding per-key-tile partials into a float32 accumulator.  Costs three more
 * tile products per (query tile, key tile) pair.
 * Arguments as fa_bwd_dropout (p_drop = 0: no dropout).  workspace needs only
 * ceil(rows * 4 / 256) * 256 bytes (rows = B*H*N dense, H*total_tokens packed)
 * plus 256 for bf16 / fp16; fa_bwd_workspace_size's larger value is accepted
 * too.  float32 inputs run
 * the float32 path, which is deterministic already (FA_ERR_UNSUPPORTED if
 * p_drop > 0 there). */
fa_status fa_bwd_deterministic(const void* q, const void* k, const void* v, const void* o, const float* lse,
                               const void* dout, void* dq, void* dk, void* dv, int B, int H, int N, int D,
                               float scale, int causal, const int32_t* cu_seqlens, int total_tokens, fa_dtype dtype,
                               float p_drop, uint64_t seed, uint32_t offset, void* workspace, size_t workspace_bytes,
                               void* stream);

/* Cached decoding step (tensortonic.com "FlashAttention" section 8: a
 * generation step has a few new queries and a long set of cached keys and
 * values; section 9: the newest query must be aligned with its actual position
 * in the key cache).
 *
 *   q    [B, H, nq, D]  the new queries            (dtype, device)
 *   k, v [B, H, nk, D]  the cache, including the entries of the new tokens
 *                       (may be NULL when nk == 0)
 *   o    [B, H, nq, D]  written (dtype);  lse [B, H, nq] float32, natural log
 *
 * Query row i sits at position nk - nq + i of the sequence, so causal allows
 * key j iff j <= i + (nk - nq) (the square top-left mask of fa_fwd is the
 * nq == nk case).  Rows with no allowed key (nq > nk, causal) get O = 0 and
 * lse = -inf.  Any nq >= 1 is accepted; the kernel is built for nq <= 8 (one
 * CTA serves up to 8 rows).  D must be 64 or 128; all three dtypes.  The work
 * streams K and V once (HBM-bound): keys are split across CTAs and the partial
 * states are merged by a second kernel (section 5's rescaling rule), in fp32.
 *
 * workspace: device scratch of fa_decode_workspace_size(...) bytes (0 when a
 * single split suffices; then workspace may be NULL), 256-byte aligned, owned
 * by the caller.  Errors: FA_ERR_INVALID / UNSUPPORTED / ALIGN / WORKSPACE
 * before any launch, FA_ERR_CUDA if a launch fails.  Asynchronous on stream. */
size_t fa_decode_workspace_size(int B, int H, int nq, int nk, int D, fa_dtype dtype);
fa_status fa_decode(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int nq, int nk,
                    int D, float scale, int causal, fa_dtype dtype, void* workspace, size_t workspace_bytes,
                    void* stream);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_H */

/*
 * fa.h -- C ABI of the GB300 (sm_103a) fused exact attention library (libfa.so).
 *
 * The operation (FlashAttention-4 blog, opening section and "Forward pass"
 * section; FlashAttention-4 paper summary, notation table):
 *
 *   S = alpha * Q K^T  (+ causal mask: key j visible to query i iff j <= i)
 *   P = softmax(S) row-wise,   O = P V,   LSE_i = ln sum_j exp(S_ij)
 *
 * and its gradients (FlashAttention-4 blog, "Backward pass" section: the five
 * products S, dP, dV, dK, dQ plus the elementwise work for P and dS):
 *
 *   dV = P^T dO,  dP = dO V^T,  D_i = sum_j P_ij dP_ij,  dS = P * (dP - D),
 *   dQ = alpha dS K,  dK = alpha dS^T Q.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Element types: q, k, v, o, do, dq, dk, dv are bfloat16 (raw 16-bit
 *   storage, passed as void*); lse is float32; cu_seqlens is int32.
 * - Head dimension d is 64, 128 or 256 (the pages' balance point moves with
 *   d: FlashAttention-4 paper summary, "Roofline" remarks).  Hq must be a multiple of Hkv; query head h reads
 *   key/value head h / (Hq / Hkv).
 * - Fixed-length layout (cu_seqlens == NULL): q, o, do, dq are [B, N, Hq, d]
 *   row-major, k, v, dk, dv are [B, N, Hkv, d]; lse is [B, Hq, N].
 * - Variable-length layout (cu_seqlens != NULL): B sequences packed along
 *   the token axis; N is then the TOTAL token count T; q, o are [T, Hq, d],
 *   k, v are [T, Hkv, d], lse is [Hq, T].  cu_seqlens is a DEVICE array of
 *   B+1 non-decreasing offsets with cu_seqlens[0] = 0 and cu_seqlens[B] = T;
 *   max_seqlen is an upper bound on every sequence length.  Malformed
 *   offsets are sanitised by one rule in every kernel: c'_0 = clamp(c_0, 0,
 *   T), c'_s = max(c'_{s-1}, clamp(c_s, 0, T)), and sequence s is rows
 *   [c'_s, c'_{s+1}).  Sequences thus never overlap and never leave the
 *   tensors; rows outside every sequence are not written (o, lse, dk, dv)
 *   or written as zero (dq).  A sanitised sequence longer than 131072
 *   tokens (possible only when max_seqlen understates the lengths) makes a
 *   d = 64/128 call compute nothing and report FA_ERR_INVALID through
 *   fa_get_device_status; the d = 256 forward has no such limit.
 * - Causal masks are top-left aligned within each sequence (query and key
 *   lengths are equal).
 * - Pointers are device pointers owned by the caller; the library allocates
 *   no device memory.  Every tensor must be 16-byte aligned and contiguous.
 * - Calls are asynchronous: they validate arguments on the host, enqueue
 *   kernels on `stream` and return.  They never synchronise (except
 *   fa_get_device_status).  No exception crosses the ABI.
 * - Return value: FA_OK, or a negative fa_status for invalid arguments
 *   (nothing is launched) or a launch error.  Device-side faults of the
 *   pipeline's own bounded waits are reported through fa_get_device_status.
 */
#ifndef FA_H_
#define FA_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    FA_OK = 0,
    FA_ERR_INVALID = -1,      /* null pointer, bad size, bad scale           */
    FA_ERR_UNSUPPORTED = -2,  /* legal but not built: d not 64/128/256, ... */
    FA_ERR_ALIGN = -3,        /* a tensor is not 16-byte aligned            */
    FA_ERR_LAUNCH = -4,       /* CUDA reported an error at launch           */
    FA_ERR_TIMEOUT = -5,      /* a device-side wait gave up (see status)    */
    FA_ERR_WORKSPACE = -6     /* backward workspace missing or too small    */
} fa_status;

/* Human-readable name of a status code (static string, never NULL). */
const char *fa_status_string(int status);

/* Number of streaming multiprocessors the kernels size their persistent
 * grids by on the current device (>0), or a negative fa_status. */
int fa_num_sms(void);

/*
 * Process-wide tuning of the forward kernel (affects later fa_fwd calls):
 *   exp2_emu_sixteenths: share of the softmax exponentials evaluated on the
 *     FMA pipe by the polynomial (fa_exp2_emu) instead of MUFU.EX2, in
 *     sixteenths (0 to 4, i.e. up to 25 %; FlashAttention-4 paper summary
 *     §3.1.3 uses 10-25 %).  Both d = 128 forward kernels and the d = 64 one
 *     apply it.
 *   tau: conditional-rescale threshold in log2 units, 0 <= tau <= 64
 *     (default log2(256) = 8; tau = 0 rescales whenever the max grows).
 * At d = 256 only tau applies: that forward evaluates every exponential on
 * MUFU (its exponentials are off the critical path; the products set the
 * pace).  Every setting gives the same attention up to rounding.  Not thread-safe
 * with concurrent fa_fwd calls.  Errors: FA_ERR_UNSUPPORTED, FA_ERR_INVALID.
 */
int fa_set_tuning(int exp2_emu_sixteenths, float tau);

/*
 * Process-wide choice of the forward kernel (affects later fa_fwd calls):
 *   0 -- two 128-row query tiles per CTA in ping-pong, 128-key tiles: the
 *        pipeline of the FlashAttention-4 blog, "Forward pass";
 *   2 -- (default) CTA pairs (clusters of two): 256 query rows per pair and
 *        256-key blocks, each product one M = 256 UMMA over both SMs, so each
 *        SM loads and reads only half of every K and V block.
 * Kernel 2 serves fixed-length and packed varlen inputs with d = 128; d = 64
 * calls use kernel 0.
 * Both compute the same attention up to rounding.
 * Errors: FA_ERR_INVALID (any other value).
 */
int fa_set_fwd_kernel(int kernel);

/*
 * Number of CTA pairs forward kernel 2 keeps resident (its persistent grid is
 * that many clusters of two; a cluster must fit inside one GPC, so this can be
 * below half the SM count).  0 until the kernel has been launched once in
 * this process.  Never fails.
 */
int fa_fwd_pairs_resident(void);

/*
 * Process-wide choice of the backward main kernel (affects later fa_bwd
 * calls; FlashAttention-4 blog, "2-CTA backward"):
 *   0 -- (default) one CTA per 128-key tile;
 *   1 -- CTA pairs per 256-key block: S^T, dP^T, dV and dK are
 *        M = 256 products over both SMs (each stages half of every B
 *        operand), dQ an M = 128 pair product after an exchange of half of
 *        dS through distributed shared memory; the dQ of a tile is computed
 *        during the next tile, in the S columns beside P^T ("2-CTA
 *        backward": the previous tile's dQ before the current dP).
 * Kernel 1 serves d = 128 inputs, fixed length or packed varlen, atomic or
 * deterministic; other head dims use kernel 0 (d = 256 its own kernel).
 * Both compute the same gradients up to the order of the fp32 dQ
 * additions; kernel 0 is the faster on GB300.  Errors: FA_ERR_INVALID.
 */
int fa_set_bwd_kernel(int kernel);

/*
 * Number of CTA pairs backward kernel 1 keeps resident; 0 until it has been
 * launched once in this process.  Never fails.
 */
int fa_bwd_pairs_resident(void);

/*
 * Process-wide order in which the kernels take their work units (affects
 * later fa_fwd and fa_bwd calls), for testing the scheduler:
 *   0 -- (default) the cost-ordered schedule (FlashAttention-4 blog,
 *        "Scheduling"): longest-processing-time first under a causal mask
 *        and for packed varlen batches (sequences sorted by length),
 *        L2-sized (batch, head) sections, zig-zag couples of query blocks;
 *   1 -- plain enumeration: (sequence, head) major, query tiles (forward)
 *        or key tiles (backward) ascending, sequences in index order.
 * Each work unit's arithmetic does not depend on the order, so the forward's
 * O and LSE and the deterministic backward's gradients are bitwise the same
 * under both; the atomic backward's dQ differs by the order of its fp32
 * additions only.  Order 1 is slower under a causal mask or with unequal
 * sequence lengths.  Not thread-safe with concurrent calls.
 * Errors: FA_ERR_INVALID (any other value).
 */
int fa_set_schedule_order(int order);

/*
 * Debug counters for the scheduler's exactly-once property (FlashAttention-4
 * blog, "Scheduling": every work tile is handed out once) and for the
 * conditional rescale (paper summary §3.1.4: how often tau = 8 skips).
 * Process-wide; affects later fa_fwd / fa_bwd calls; all NULL (the default)
 * turns counting off.  The caller owns and zeroes the device buffers; the
 * kernels only add to them (atomically), so calls accumulate.  With T the
 * token count (B * N fixed length, the packed total for varlen):
 *   visits (int [Hq * T] for fa_fwd, [Hkv * T] for fa_bwd; may be NULL):
 *     fa_fwd adds 1 at [h * T + r] when it finishes the 128-row query tile
 *     of head h starting at token row r; fa_bwd adds 1 at [hk * T + r] when
 *     it finishes the work unit of key/value head hk whose 128-key tile
 *     starts at row r (its dK, dV written; units split by query-head group
 *     count once per group);
 *   inner (int [Hq * T], fa_bwd; may be NULL): 1 at [h * T + r] each time a
 *     128-key tile's dQ contribution to the query tile of head h starting at
 *     row r has been added (so the count is the number of key tiles that see
 *     the query tile; at d = 256 the query tiles are the kernel's 64-row
 *     steps, counted by the first head-dim half's pass);
 *   rescales (unsigned long long [2], fa_fwd; may be NULL): [1] counts the
 *     per-warp rescale decisions after each row block's first key block,
 *     [0] those that took the rescale branch (tau exceeded).
 * Tile starts are the sequence start plus multiples of 128.  Counting costs
 * an atomic per tile (and per warp decision): a debugging aid, not for
 * timed runs.  While any counter is armed, the CTA-pair forward, the CTA-pair
 * backward and both d = 256 kernels run a separate build that counts; the
 * build without the counters has no trace of them.
 * Errors: FA_ERR_ALIGN (misaligned pointer).
 */
int fa_set_debug_counters(int *visits, int *inner, unsigned long long *rescales);

/*
 * Forward: O and LSE of exact attention (FlashAttention-4 blog, "Forward
 * pass: a new softmax pipeline with conditional rescaling").
 *
 * q [B,N,Hq,d], k/v [B,N,Hkv,d] bf16 in; o [B,N,Hq,d] bf16 out,
 * lse [B,Hq,N] float32 out (natural log, includes alpha).  Varlen: see
 * above.  alpha > 0 is the logit scale (normally 1/sqrt(d)).
 * causal: 0 or 1.  N == 0 (or T == 0) is a no-op returning FA_OK.
 * Errors: FA_ERR_INVALID (null pointer, B<1, N<0, Hq/Hkv<1, Hq % Hkv,
 * alpha not finite and > 0, varlen without max_seqlen>0),
 * FA_ERR_UNSUPPORTED (d not 64, 128 or 256; varlen with B > 1024 or
 * max_seqlen > 131072),
 * FA_ERR_ALIGN, FA_ERR_LAUNCH.  d = 256 runs on a kernel of its own (one
 * 128-row query tile per CTA, 64-key blocks) whatever fa_set_fwd_kernel says.
 */
int fa_fwd(const void *q, const void *k, const void *v, void *o, float *lse,
           int B, int Hq, int Hkv, int N, int d, float alpha, int causal,
           const int *cu_seqlens, int max_seqlen, cudaStream_t stream);

/*
 * Bytes of device workspace fa_bwd needs (the library allocates none):
 * D (rowsum(dO*O), fp32), the fp32 dQ accumulator, the deterministic-mode
 * semaphores, the varlen work list and, for varlen at d = 64 or 128, room
 * for fp32 dK and dV partial sums (Hq * T * d / 2 bytes; used when the work
 * is split by query-head group, see fa_bwd).  N is the sequence length
 * (fixed length) or the total token count T (varlen = 1).  Returns 0 for
 * invalid sizes (d not 64, 128 or 256 among them).  About (4 d + 4) * Hq * T
 * bytes (varlen at d = 64 / 128: (4.5 d + 4) * Hq * T).
 */
size_t fa_bwd_workspace_size(int B, int Hq, int N, int d, int deterministic, int varlen);

/*
 * Backward: dQ, dK, dV of exact attention (FlashAttention-4 blog, "Backward
 * pass", "Deterministic mode").  Inputs q, k, v, the forward's o and lse,
 * and the upstream gradient dout (layouts as in fa_fwd); outputs dq like q,
 * dk and dv like k (bf16; for Hkv < Hq, dk/dv sum over the query heads of
 * each group).  deterministic = 1 adds dQ contributions in a fixed order
 * (bit-identical across runs); 0 uses unordered fp32 reductions.
 * workspace: device memory of at least fa_bwd_workspace_size(...) bytes,
 * 256-byte aligned, owned by the caller; its contents need no
 * initialisation and are overwritten.  Calls that share a workspace must not
 * overlap on the GPU.
 * d = 256 runs on a kernel of its own: the dK / dV accumulators of a
 * 128-key tile would fill all of tensor memory, so each tile is processed
 * once per head-dim half of the gradients (recomputing S and dP for each),
 * with queries in 64-row steps (fa_set_bwd_kernel does not apply).
 * Packed varlen batches in atomic mode whose key/value heads each serve at
 * least 16 query heads (a multiple of 8; MQA-like) run, on the one-CTA
 * kernel at d = 64 or 128, as work units of 8 query heads each: the CTAs of
 * a wave then share one head group's rows of Q, dO and the dQ accumulator
 * in L2 (FlashAttention-4 blog, "Scheduling": L2-sized sections), and each
 * unit adds its group's share of dK and dV into fp32 sums in the workspace
 * that the last stage converts to bf16 (dK times alpha).
 * Errors: as fa_fwd, plus FA_ERR_WORKSPACE (NULL, misaligned or too small)
 * and FA_ERR_UNSUPPORTED (varlen with max_seqlen > 131072 or B > 1024).
 */
int fa_bwd(const void *q, const void *k, const void *v, const void *o, const float *lse,
           const void *dout, void *dq, void *dk, void *dv,
           int B, int Hq, int Hkv, int N, int d, float alpha, int causal,
           const int *cu_seqlens, int max_seqlen, int deterministic,
           void *workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * fa_bwd split into its three launches, for callers that time or schedule
 * them separately: stages is a bit mask, 1 = preprocess (D, zero the dQ
 * accumulator and semaphores, varlen work list), 2 = main kernel (dK, dV and
 * the dQ accumulator), 4 = dQ postprocess (dq = bf16(alpha * accumulator)).
 * Stages must run in this order on one workspace; fa_bwd == stages 7.  For
 * a packed varlen batch, stage 1 plans the work list for the backward kernel
 * selected at that time (fa_set_bwd_kernel) and for the call's mode (units
 * split by query-head group or not, see fa_bwd): a stage 2 run with the
 * other selection or the other mode computes nothing and reports
 * FA_ERR_INVALID through fa_get_device_status.  With split units, stage 4
 * also writes dk and dv.
 */
int fa_bwd_stages(int stages, const void *q, const void *k, const void *v, const void *o,
                  const float *lse, const void *dout, void *dq, void *dk, void *dv,
                  int B, int Hq, int Hkv, int N, int d, float alpha, int causal,
                  const int *cu_seqlens, int max_seqlen, int deterministic,
                  void *workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * fa_bwd without a workspace argument, for callers that cannot allocate
 * device memory when they need gradients (for example code running under a
 * framework that owns every device allocation, or a plugin whose host
 * application forbids allocation after start-up).  The FlashAttention-4 pages
 * have no counterpart: this is a library convenience.
 *
 * It computes exactly what fa_bwd computes (same arguments, minus the
 * workspace) and allocates nothing: its scratch is a 64 MiB array of static
 * device storage inside the library, reserved on every GPU that loads the
 * library until the process exits.  Sizes whose workspace
 * (fa_bwd_workspace_size) exceeds 64 MiB -- about Hq * T > 130000 -- are
 * rejected with FA_ERR_WORKSPACE before anything is launched; other errors
 * as fa_bwd.
 * - The first call on each device looks up the array's device address
 *   (cudaGetSymbolAddress) with that device current; make that first call
 *   before any stream capture.
 * - All calls on a device share the one scratch array, which keeps the last
 *   call's contents (each call re-zeroes what must start at zero).  Calls
 *   that overlap on the GPU (different streams, or concurrent host threads)
 *   race on it and produce wrong gradients: serialise them.
 * - A device-side wait timeout (or an offset table the plan stage rejects)
 *   is recorded in the scratch area's own status word;
 *   fa_get_device_status reports and clears it on this device, as it does
 *   for a workspace passed to it.
 * Argument errors are fa_bwd's, checked in fa_bwd's order (FA_ERR_UNSUPPORTED
 * for an unbuilt head dim, ...); a call with no tokens returns FA_OK.
 */
int fa_bwd_noalloc(const void *q, const void *k, const void *v, const void *o, const float *lse,
                   const void *dout, void *dq, void *dk, void *dv,
                   int B, int Hq, int Hkv, int N, int d, float alpha, int causal,
                   const int *cu_seqlens, int max_seqlen, int deterministic, cudaStream_t stream);

/*
 * Reads (and clears) the library's device status word on the current
 * device after synchronising `stream`: FA_OK, or FA_ERR_TIMEOUT when a
 * kernel's bounded wait gave up (the kernel then skipped its remaining work,
 * drained its own copies, freed its tensor memory and returned), or
 * FA_ERR_INVALID when a kernel rejected a device-side table (a varlen batch
 * whose sanitised offsets hold a sequence longer than the 131072-token
 * limit: nothing is computed for that call).
 * `workspace` may be NULL; when it is a backward workspace its status word
 * is read (and cleared) too, and after a reported failure the main stage's
 * unit claim counter in the workspace is rewound, so that a later
 * fa_bwd_stages call with stages == 2 alone starts from the first unit.
 * The status word of fa_bwd_noalloc's scratch area on this device is read,
 * cleared and rewound the same way once a no-allocation call has run here.
 * The first non-OK code found is returned (device word, then workspace,
 * then scratch area); all of them are cleared.
 */
int fa_get_device_status(const void *workspace, cudaStream_t stream);

/*
 * The forward kernel's FMA-pipe exponential, exposed for testing: y[i] =
 * 2^x[i] by Cody-Waite range reduction (n = floor(x), f = x - n) and a
 * degree-3 Horner polynomial in f with p0 = 1, scaled by adding n to the
 * exponent bits (FlashAttention-4 blog, "Faster exponential" section;
 * paper summary §3.1.3: max relative error 8.77e-5 on [0,1)).  Inputs below
 * -127 (and -inf) give 0 or a value below 2^-126.  Each element is
 * evaluated both in the scalar form (ping-pong forward) and in the packed
 * two-lane form (CTA-pair forward); where the two differ in any bit, y[i] is
 * NaN.  x, y: device float32 arrays of n elements.
 * Errors: FA_ERR_INVALID, FA_ERR_LAUNCH.
 */
int fa_exp2_emu(const float *x, float *y, int64_t n, cudaStream_t stream);

/*
 * Diagnostic for the failure-detection path, for tests: enqueues a one-block
 * kernel on `stream` whose warp waits, through the same bounded mbarrier
 * wait every kernel here uses, on a barrier nothing ever arrives at.  After
 * the wait limit (about 2 s) it records FA_ERR_TIMEOUT in the current
 * device's status word and returns; the context stays usable, and
 * fa_get_device_status(NULL, stream) then reports (and clears) the timeout.
 * Errors: FA_ERR_LAUNCH.
 */
int fa_selftest_timeout(cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* FA_H_ */

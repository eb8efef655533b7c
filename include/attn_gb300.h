/*
 * attn_gb300.h - C ABI of the fused exact-attention forward pass for GB300 (sm_103a).
 *
 * The operation ("FlashAttention (HI)" page, section "Problems of standard attention",
 * formula Attention(Q,K,V) = softmax(Q K^T / sqrt(d_k)) V; computed as the
 * pages' fused, tiled kernel with an online softmax, sections "Tiling and
 * block processing", "Online softmax computation" and "Combining operations
 * in one CUDA kernel"):
 *
 *   for every batch b, head h and query row i
 *     s_j    = scale * <q[b,i,h,:], k[b,j,h,:]>          for j in A(i)
 *     o[b,i,h,:] = sum_j softmax(s)_j * v[b,j,h,:]
 *     lse[b,h,i] = ln sum_j exp(s_j)                       (natural log, fp32)
 *
 *   A(i) = {0 .. N_k-1}; with causal != 0, A(i) = {j : j <= i + N_k - N_q}
 *   (bottom-right alignment; j <= i when N_q == N_k).  A row whose A(i) is
 *   empty gets o = 0 and lse = -inf.  The N_q x N_k score matrix is never
 *   written to memory.
 *
 * Layouts (all contiguous, row-major, device memory):
 *   q, o : [B, N_q, H, d]      k, v : [B, N_k, H, d]      lse : [B, H, N_q] fp32
 *   o is bf16 for bf16 and e4m3 inputs, fp16 for fp16 inputs.
 *   d (head dimension) must be 64, 128 or 256 (head size 256 is named among
 *   FlashAttention-2's extensions on the "FlashAttention (HI)" page, section
 *   "Development and further research").  d = 256 runs a kernel with one 128-row query tile per CTA
 *   (its 256-column fp32 output accumulator fills half of TMEM).
 *   q, k, v, o must be 16-byte aligned; lse 4-byte aligned.  lse may be NULL
 *   (then it is not written).
 *
 * FP8 ("FlashAttention-3 (BN)" page, section "Low precision (FP8) and reducing
 * quantisation error"): q, k, v hold
 *   float8 e4m3 codes; the real inputs are code * descale with one fp32
 *   descale per (batch, head): q_descale, k_descale, v_descale are device
 *   arrays of B*H floats indexed b*H + h.
 *
 * Ownership: the caller allocates and owns every buffer.  The library
 *   allocates no device memory; inputs are never modified.  (attn_fwd_host
 *   creates two streams and a few events per device on its first call and
 *   keeps them for the life of the process.)
 *
 * Asynchrony: calls are enqueued on `stream` (a cudaStream_t; NULL = legacy
 *   default stream) and return at once; results are valid once the stream has
 *   reached them.  Results are deterministic (a fixed reduction order per row).
 *
 * Errors: arguments are checked before anything is launched and give
 *   ATTN_ERR_INVALID_ARG (null pointer, negative size, misaligned pointer,
 *   non-finite or non-positive scale, bad dtype) or ATTN_ERR_UNSUPPORTED
 *   (d not 64, 128 or 256; N_q or N_k above ATTN_MAX_SEQ_LEN; a grid dimension
 *   out of range).  ATTN_ERR_CUDA reports a
 *   failed tensor-map encode or launch (cudaGetLastError is cleared).
 *   Kernels never trap: every wait inside them is bounded; a wait that runs
 *   out sets a device status word, the kernel returns, and attn_check_status
 *   reports ATTN_ERR_TIMEOUT.  Zero-sized problems (B, H or N_q == 0) launch
 *   nothing and return ATTN_OK; N_k == 0 writes o = 0 and lse = -inf.
 */
#ifndef ATTN_GB300_H
#define ATTN_GB300_H

#include <stddef.h>

#if defined(__GNUC__)
#define ATTN_API __attribute__((visibility("default")))
#else
#define ATTN_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    ATTN_OK = 0,
    ATTN_ERR_INVALID_ARG = 1,
    ATTN_ERR_UNSUPPORTED = 2,
    ATTN_ERR_CUDA = 3,
    ATTN_ERR_TIMEOUT = 4,
    ATTN_ERR_SCRATCH_LIMIT = 5
} attn_status_t;

typedef enum {
    ATTN_BF16 = 0,
    ATTN_FP16 = 1,
    ATTN_FP8_E4M3 = 2,
    ATTN_FP32 = 3  /* input of attn_quantize_e4m3 only */
} attn_dtype_t;

/* Fused forward pass on the tensor cores (tcgen05 MMAs, TMEM accumulators,
 * TMA-fed shared-memory ring).  dtype ATTN_FP8_E4M3 means unit descales. */
ATTN_API attn_status_t attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                       int B, int H, int N_q, int N_k, int d, float scale, int causal,
                       attn_dtype_t dtype, void* stream);

/* FP8 e4m3 forward pass with per-(batch, head) fp32 descales (device arrays of
 * B*H floats; none may be NULL).  o is bf16. */
ATTN_API attn_status_t attn_fwd_fp8(const void* q, const void* k, const void* v, void* o, float* lse,
                           const float* q_descale, const float* k_descale,
                           const float* v_descale,
                           int B, int H, int N_q, int N_k, int d, float scale, int causal,
                           void* stream);

/* attn_fwd_fp8 with a caller workspace, for d = 64 and 128: the P V product
 * runs on fp16 operands (fp16 P; see "FlashAttention-3 (BN)", section "Low
 * precision (FP8) and reducing quantisation error", on FP8's accuracy cost),
 * so every e4m3 V value must be widened to fp16 (exactly).  attn_fwd_fp8 does
 * that on chip in every CTA that reads a V tile; here one elementwise kernel
 * first writes the fp16 copy of v into the workspace and the attention kernel
 * then loads fp16 V tiles directly.  The result is bit for bit that of
 * attn_fwd_fp8 with the same arguments.
 * workspace: device memory of at least attn_fwd_fp8_workspace_bytes(B, H, N_k,
 * d) bytes (fp16 [B, N_k, H, d]), 16-byte aligned, overwritten; it must not
 * overlap any argument.  d = 256 runs attn_fwd_fp8's kernel and does not use
 * the workspace.  Errors as attn_fwd_fp8, plus ATTN_ERR_INVALID_ARG for a
 * missing, misaligned or too small workspace. */
ATTN_API attn_status_t attn_fwd_fp8_ws(const void* q, const void* k, const void* v, void* o,
                                       float* lse, const float* q_descale,
                                       const float* k_descale, const float* v_descale, int B,
                                       int H, int N_q, int N_k, int d, float scale, int causal,
                                       void* workspace, size_t workspace_bytes, void* stream);

/* Workspace bytes attn_fwd_fp8_ws needs: 2 * B * N_k * H * d for d = 64 or
 * 128, 0 for d = 256 or invalid arguments. */
ATTN_API size_t attn_fwd_fp8_workspace_bytes(int B, int H, int N_k, int d);

/* The same operation on the CUDA cores only (fp32 FMAs, no tensor cores): a
 * second, independent GPU implementation used to cross-check the tensor-core
 * path.  Descales may be NULL (unit) and are used only for ATTN_FP8_E4M3. */
ATTN_API attn_status_t attn_fwd_simt(const void* q, const void* k, const void* v, void* o, float* lse,
                            const float* q_descale, const float* k_descale,
                            const float* v_descale,
                            int B, int H, int N_q, int N_k, int d, float scale, int causal,
                            attn_dtype_t dtype, void* stream);

/* Incoherent processing + FP8 quantisation ("FlashAttention-3 (BN)" page,
 * section "Low precision (FP8) and reducing quantisation error"): each row of
 * x [B, N, H, d] (ATTN_BF16, ATTN_FP16 or ATTN_FP32) is multiplied by the
 * random orthogonal matrix M = diag(signs) H_d / sqrt(d), H_d the Sylvester
 * Hadamard matrix, then quantised to e4m3 codes [B, N, H, d] with one fp32
 * descale per (batch, head) written to descale [B*H]: descale = amax / 448
 * (1 when amax = 0), code = round-to-nearest-even(y / descale) saturated to
 * +-448.  signs: device array of d values +1 / -1; NULL quantises without the
 * rotation (use that for V).  Apply the same signs to q and k: Q M (K M)^T =
 * Q K^T, so attn_fwd_fp8 on the outputs computes the same attention with
 * outliers spread over all coordinates.  d must be 64, 128 or 256; codes 16-byte
 * aligned.  Enqueued on `stream`; allocates nothing (descale also serves as
 * the amax accumulator). */
ATTN_API attn_status_t attn_quantize_e4m3(const void* x, attn_dtype_t x_dtype, void* codes,
                                          float* descale, int B, int N, int H, int d,
                                          const float* signs, void* stream);

/* Grouped-query / multi-query attention: q, o are [B, N_q, H, d]; k, v are
 * [B, N_k, H_kv, d] with H % H_kv == 0, and query head h attends with K/V head
 * h / (H / H_kv) (H_kv == H: multi-head; H_kv == 1: multi-query).  These are
 * the Multi-Query Attention architectures "FlashAttention (HI)" lists under
 * FlashAttention-2.  Descales (e4m3 only, NULL = unit): q_descale [B*H],
 * k_descale and v_descale [B*H_kv], indexed b*H + h and b*H_kv + h_kv.
 * Everything else as attn_fwd; ATTN_ERR_INVALID_ARG if H_kv < 1 or H is not a
 * multiple of H_kv. */
ATTN_API attn_status_t attn_fwd_gqa(const void* q, const void* k, const void* v, void* o,
                                    float* lse, const float* q_descale, const float* k_descale,
                                    const float* v_descale, int B, int H, int H_kv, int N_q,
                                    int N_k, int d, float scale, int causal, attn_dtype_t dtype,
                                    void* stream);

/* Split-KV forward pass (the same operation as attn_fwd / attn_fwd_fp8).  Each
 * 256-row query-tile pair's K/V range is cut into num_splits contiguous parts
 * processed by separate CTAs, which adds parallelism when B*H*N_q is small and
 * N_k is long ("FlashAttention-2 (BN)" page, section "Improved parallelism":
 * spreading one head's work over more SMs).  Each part writes its partial
 * output, normalised by its own row sum, and its log-sum-exp to `workspace`;
 * a second kernel merges the parts exactly:
 *   lse = ln sum_s exp(lse_s),   o = sum_s exp(lse_s - lse) * o_s.
 * num_splits: 1..32 (1 = the plain tensor-core kernel, workspace unused).
 * workspace: caller-allocated device memory of at least
 *   attn_splitkv_workspace_bytes(B, H, N_q, d, num_splits) bytes, 16-byte
 *   aligned; it is overwritten (layout: fp32 partial outputs
 *   [num_splits][B*H][N_q][d], then fp32 partial lse [num_splits][B*H][N_q]).
 * Descales: as attn_fwd_simt (NULL = unit; used for ATTN_FP8_E4M3 only).
 * Errors as attn_fwd, plus ATTN_ERR_INVALID_ARG for num_splits out of range or
 * a missing, misaligned or too small workspace. */
ATTN_API attn_status_t attn_fwd_splitkv(const void* q, const void* k, const void* v, void* o,
                                        float* lse, const float* q_descale,
                                        const float* k_descale, const float* v_descale, int B,
                                        int H, int N_q, int N_k, int d, float scale, int causal,
                                        attn_dtype_t dtype, int num_splits, void* workspace,
                                        size_t workspace_bytes, void* stream);

/* Workspace bytes attn_fwd_splitkv needs (0 for num_splits == 1 or invalid
 * arguments). */
ATTN_API size_t attn_splitkv_workspace_bytes(int B, int H, int N_q, int d, int num_splits);

/* A num_splits for attn_fwd_splitkv on a GPU with num_sms SMs: the count (1 ..
 * 32) that minimises an estimate of the time in 128-key steps, waves of CTAs
 * x (key tiles per CTA + 3 steps of fixed cost per CTA) + the combine pass
 * (1 + splits / 8 steps).  1 when splitting does not pay (enough query tiles
 * to fill the GPU) or for invalid arguments.  Host arithmetic only: no CUDA
 * call. */
ATTN_API int attn_splitkv_num_splits(int B, int H, int N_q, int N_k, int d, int num_sms);

/* Backward pass: gradients of the forward's O with respect to q, k and v for an
 * upstream gradient dO (the pages name training speedups, "FlashAttention
 * (HI)" page, section "Empirical results", but do not write the backward pass
 * out; this is the derivative of the formula above).  With P the forward's row
 * softmax (P_ij = exp(scale q_i.k_j - lse_i), masked entries 0):
 *   D_i = sum_t dO_it o_it,  dS = P (dO v^T - D),
 *   dq = scale dS k,  dk = scale dS^T q,  dv = P^T dO.
 * Inputs: q, o, dO [B, N_q, H, d]; k, v [B, N_k, H, d]; lse [B, H, N_q] fp32 as
 * written by attn_fwd for the same q, k, v, scale and causal (o likewise).
 * Outputs dq [B, N_q, H, d], dk, dv [B, N_k, H, d], in dtype (bf16 or fp16;
 * ATTN_FP8_E4M3 gives ATTN_ERR_UNSUPPORTED), fp32 accumulation.  A key no
 * query row may attend gets dk = dv = 0; a query row with no allowed key gets
 * dq = 0.  d must be 64 or 128; k, v have H heads (attn_bwd_gqa for fewer).
 * workspace: caller-allocated device memory of at least
 * attn_bwd_workspace_bytes(B, H, N_q) bytes, 16-byte aligned, overwritten
 * (fp32 lse * log2(e) and D per row, each padded to a multiple of 128 rows).
 * Every output element is written by one CTA: the result is deterministic.
 * Errors as attn_fwd, plus ATTN_ERR_INVALID_ARG for a missing, misaligned or
 * too small workspace. */
ATTN_API attn_status_t attn_bwd(const void* q, const void* k, const void* v, const void* o,
                                const float* lse, const void* dO, void* dq, void* dk, void* dv,
                                int B, int H, int N_q, int N_k, int d, float scale, int causal,
                                attn_dtype_t dtype, void* workspace, size_t workspace_bytes,
                                void* stream);

/* attn_bwd for grouped-query / multi-query attention: k, v, dk, dv are
 * [B, N_k, H_kv, d] with H % H_kv == 0; query head h uses K/V head
 * h / (H / H_kv), and dk, dv of a K/V head sum the contributions of its
 * H / H_kv query heads (each summed in one CTA: still deterministic).
 * ATTN_ERR_INVALID_ARG if H_kv < 1 or H % H_kv != 0.  Otherwise as attn_bwd. */
ATTN_API attn_status_t attn_bwd_gqa(const void* q, const void* k, const void* v, const void* o,
                                    const float* lse, const void* dO, void* dq, void* dk,
                                    void* dv, int B, int H, int H_kv, int N_q, int N_k, int d,
                                    float scale, int causal, attn_dtype_t dtype, void* workspace,
                                    size_t workspace_bytes, void* stream);

/* Workspace bytes attn_bwd and attn_bwd_gqa need (0 for invalid arguments). */
ATTN_API size_t attn_bwd_workspace_bytes(int B, int H, int N_q);

/* Forward pass on HOST-resident tensors (the same operation and layouts as
 * attn_fwd / attn_fwd_fp8, with q, k, v, o, lse and, for ATTN_FP8_E4M3, the
 * three descale arrays of B*H floats in host memory; H_kv = H).  Host buffers
 * should be page-locked (cudaHostAlloc / pinned), or the copies cannot overlap.
 *
 * The (batch, head) pairs are cut into about four chunks of whole heads of
 * one batch row.  Over a ring of three device slots in `workspace`, the copy
 * of chunk c + 1 to the device (an internal stream), the kernel on chunk c
 * (on `stream`) and the copy of chunk c - 1 back to the host (a second
 * internal stream) run at the same time.  Every (batch, head) is computed as
 * attn_fwd computes it, so the results equal those of attn_fwd on device
 * copies of the inputs bit for bit.
 *
 * workspace: device memory of attn_fwd_host_workspace_bytes(...) bytes,
 *   256-byte aligned, owned by the caller, overwritten.  lse may be NULL.
 * Ordering: the copies start after the work already queued on `stream`; work
 *   queued on `stream` afterwards sees o and lse written in host memory (for
 *   example a cudaStreamSynchronize(stream) before the host reads them).
 * Threads: calls on one device from several host threads are enqueued one
 *   after the other (an internal lock per device).
 * Errors: as attn_fwd, plus ATTN_ERR_INVALID_ARG for a missing, misaligned or
 *   short workspace; ATTN_ERR_CUDA if a copy or an internal stream or event
 *   cannot be set up. */
ATTN_API attn_status_t attn_fwd_host(const void* q, const void* k, const void* v, void* o,
                                     float* lse, const float* q_descale, const float* k_descale,
                                     const float* v_descale, int B, int H, int N_q, int N_k, int d,
                                     float scale, int causal, attn_dtype_t dtype, void* workspace,
                                     size_t workspace_bytes, void* stream);

/* Workspace bytes attn_fwd_host needs (0 for invalid or empty arguments). */
ATTN_API size_t attn_fwd_host_workspace_bytes(int B, int H, int N_q, int N_k, int d,
                                              attn_dtype_t dtype);

/* Longest sequence (N_q, N_k; N of attn_quantize_e4m3) any entry point takes:
 * row and key indices, and TMA coordinates up to two query tiles past the
 * end, stay within int.  Longer sequences give ATTN_ERR_UNSUPPORTED. */
#define ATTN_MAX_SEQ_LEN (2147483647 - 256)

/* Size of the fixed scratch array attn_fwd_splitkv_static uses (bytes). */
#define ATTN_STATIC_SCRATCH_BYTES (32 * 1024 * 1024)

/* attn_fwd_splitkv without a caller workspace, for callers that cannot
 * allocate device memory (for example a plugin inside a host program that owns
 * all device memory through its own pool and forbids raw cudaMalloc, or a
 * latency-critical loop that cannot afford the device-wide synchronisation an
 * allocation can cause).  The pages have no counterpart: this is a deployment
 * interface, not part of the method.
 *
 * Scratch: a fixed array of ATTN_STATIC_SCRATCH_BYTES compiled into the
 * library, held by every GPU that loads it until the process exits.  The call
 * allocates nothing (no cudaMalloc, no allocating library routine).  The
 * problem must fit: attn_splitkv_workspace_bytes(B, H, N_q, d, num_splits) <=
 * ATTN_STATIC_SCRATCH_BYTES, else ATTN_ERR_SCRATCH_LIMIT and nothing runs.
 * num_splits: 2..32.  Other arguments, layouts and errors as attn_fwd_splitkv.
 * The first call on each device looks up the array's device address
 * (cudaGetSymbolAddress, with that device current); make that first call
 * before any stream capture.  With lazy module loading (CUDA's default,
 * CUDA_MODULE_LOADING=LAZY) the library's device code, and the array with it,
 * is loaded on a device by the first library call that needs it there: that
 * load reserves the array's memory and may synchronise.  Callers that cannot
 * afford either make their first call on each device outside the region where
 * allocation is not allowed (for example at start-up); later calls reserve
 * nothing.  The looked-up address is kept per device ordinal for the life of
 * the process: after cudaDeviceReset on a device, do not call this function
 * on that device again in the same process (the kept address would be
 * stale).  All calls share the one array, so calls whose
 * work overlaps on the GPU (other streams, other host threads) race: order
 * them on one stream or synchronise between them.  No state carries over from
 * one call to the next that the result depends on. */
ATTN_API attn_status_t attn_fwd_splitkv_static(const void* q, const void* k, const void* v,
                                               void* o, float* lse, const float* q_descale,
                                               const float* k_descale, const float* v_descale,
                                               int B, int H, int N_q, int N_k, int d, float scale,
                                               int causal, attn_dtype_t dtype, int num_splits,
                                               void* stream);

/* Health check of the kernels' bounded waits: launches a one-thread kernel
 * that waits, with the wait the attention kernel uses, on a barrier nothing
 * arrives at, so the wait runs out after timeout_us microseconds (1 .. 10^7)
 * and sets the device status word; the next attn_check_status then returns
 * ATTN_ERR_TIMEOUT and the context stays usable.  Nothing traps or hangs. */
ATTN_API attn_status_t attn_selftest_wait(unsigned timeout_us, void* stream);

/* Health check of the attention kernels' own abort path (the failure
 * detection of the tensor-core kernels: every wait bounded, then drain, free
 * TMEM, exit).  Runs the kernel attn_fwd / attn_fwd_fp8 would run for these
 * arguments (same layouts, dtypes, head dimensions 64 / 128 / 256), except that
 * the K/V loader stops after the first ring item and every bounded wait gives
 * up after timeout_us microseconds (1 .. 10^7; normal calls use 2 s).  The
 * waits for the withheld tiles run out, each role drains what it issued (those
 * drains keep the 2 s limit), TMEM is freed and the CTAs exit; the next
 * attn_check_status returns ATTN_ERR_TIMEOUT and clears the status, and the
 * context stays usable.  o and lse are left with undefined contents.  Needs
 * N_q > 0 and N_k > 0 (else ATTN_ERR_INVALID_ARG); other errors as attn_fwd.
 * workspace: NULL, or for ATTN_FP8_E4M3 at d = 64 / 128 a workspace as
 * attn_fwd_fp8_ws takes (then that function's kernels run: the V widening in
 * full, the attention kernel cut short); a workspace for any other dtype or d,
 * or one that is misaligned or too small, gives ATTN_ERR_INVALID_ARG.
 * Not part of the method: a diagnostic of the failure-detection path. */
ATTN_API attn_status_t attn_selftest_abort(const void* q, const void* k, const void* v, void* o,
                                           float* lse, const float* q_descale,
                                           const float* k_descale, const float* v_descale,
                                           int B, int H, int N_q, int N_k, int d, float scale,
                                           int causal, attn_dtype_t dtype, void* workspace,
                                           size_t workspace_bytes, unsigned timeout_us,
                                           void* stream);

/* Synchronises `stream`, then returns and clears the device status word:
 * ATTN_ERR_TIMEOUT if a bounded wait inside a kernel ran out since the last
 * call, ATTN_ERR_CUDA if the stream reports an error, else ATTN_OK. */
ATTN_API attn_status_t attn_check_status(void* stream);

/* Static, human-readable name of a status code. */
ATTN_API const char* attn_status_string(attn_status_t s);

/* Name of the CUDA error (cudaGetErrorName, e.g. "cudaErrorIllegalAddress")
 * behind the last ATTN_ERR_CUDA returned on the calling host thread, or
 * "none" if this thread has had none.  Static string; never fails.  After a
 * device-side fault the CUDA context is unusable and every later call of the
 * process returns ATTN_ERR_CUDA. */
ATTN_API const char* attn_last_cuda_error(void);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_GB300_H */

/*
 * Exact tiled attention on one GB300 (sm_103a): the C ABI of libfa.so.
 *
 * O = softmax(scale * Q K^T [+ causal mask]) V, computed tile by tile with an
 * online softmax so that the N x N score matrix never reaches HBM, plus the
 * recomputing backward that yields dQ, dK and dV.
 *
 * Sources for what is computed (pages on FlashAttention-2):
 *  - "flashattention-2" glossary: "How FlashAttention-2 Works (Tiled
 *    Algorithm)" table (Q tile loaded once, K/V tiles streamed, S = Q K^T,
 *    online softmax, O accumulated, written once) and the "Performance
 *    Comparison" table (the result is exact; memory O(N)).
 *  - "Flash Attention v2" notes: "Detailed Algorithm Comparison", forward
 *    pass (running max m, running sum l, rescale factor exp(m - m_new), the
 *    statistics kept for the backward) and "Backward Pass Computation"
 *    (recompute S and P per block, then dP, dQ, dK, dV).
 *  - "FlashAttention-2 paper" digest: "Three changes" (deferred rescaling,
 *    query blocks split across thread blocks even within one head).
 *
 * Conventions shared by every entry point
 *  - Tensors q, k, v, o, dO, dq, dk, dv are bf16, shape [B, H, N, d],
 *    contiguous, d innermost. lse is fp32 [B, H, N] (natural log).
 *  - All tensor pointers are DEVICE pointers owned by the caller, 16-byte
 *    aligned. The library keeps no reference to them after the call.
 *  - d must be 32, 64, 96 or 128; B, H, N >= 1; B*H < 2^31 (offsets are computed in
 *    64 bits, so a tensor may hold more than 2^31 elements). The dense
 *    entry points also take d = 256 ("Flash Attention v2" notes, "Detailed
 *    Differences", 3 "Head Dimension Support"): fa_fwd, fa_fwd_strided,
 *    fa_bwd, fa_bwd_strided, fa_bwd_workspace_size, the three backward
 *    stages and fa_bwd_noalloc, with B*H*ceil(N/64) < 2^31. The unequal-
 *    length, packed and decode entry points reject it (FA_ERR_UNSUPPORTED).
 *  - Causal masking is top-left aligned with equal query and key lengths:
 *    query i sees keys j <= i. scale must be finite and >= 0.
 *  - stream is a cudaStream_t (NULL = the legacy default stream). Every call
 *    only enqueues work and returns; outputs are valid once the stream has
 *    reached that point. No call synchronises the device.
 *  - So the attention calls (forward, backward and its stages, the packed-
 *    batch pair, decode) can be captured into a CUDA graph on a capturing
 *    stream. Each replay runs the same kernels on the buffers as they are
 *    at replay time; pointers, sizes and scale are fixed at capture. Make
 *    one ordinary call on the device before capturing, so that the
 *    per-device set-up below is not done inside the capture.
 *  - Argument errors are reported before anything is enqueued, and the
 *    outputs are then untouched. Launch failures return FA_ERR_CUDA.
 *  - A kernel that waits on an on-chip barrier for longer than 2 s gives up,
 *    leaves the GPU usable and records FA_ERR_TIMEOUT in a device status word
 *    shared by all calls of the process; fa_last_device_status() reads it.
 *  - Per-device set-up (SM count, device addresses of the status word and of
 *    fa_bwd_noalloc's array) is done at the first call on each device, and
 *    again when the current CUDA context is a new one (after cudaDeviceReset).
 */
#ifndef FA_H
#define FA_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum fa_status {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = 1, /* null or misaligned pointer, size < 1, bad scale */
  FA_ERR_UNSUPPORTED = 2, /* head dimension not supported by the call, or B*H too large */
  FA_ERR_CUDA = 3,        /* a CUDA runtime or driver call failed */
  FA_ERR_TIMEOUT = 4,     /* a device-side bounded wait expired */
  FA_ERR_WORKSPACE = 5,   /* backward workspace null or too small */
  FA_ERR_DEVICE_CHECK = 6 /* debug build only: a device-side index check failed */
} fa_status;

/* Version of this ABI; bumped on any incompatible change. 2: the packed
 * backward's workspace size also takes the longest key length
 * (fa_bwd_varlen_workspace_size). */
int fa_abi_version(void);

/*
 * Forward. Writes o = softmax(scale * q k^T [masked]) v in bf16 and
 * lse[b,h,i] = ln sum_j exp(scale * q_i . k_j) over the visible keys, in fp32.
 * ("flashattention-2" glossary, "How FlashAttention-2 Works (Tiled
 * Algorithm)", steps 1-7; "Flash Attention v2" notes, "Detailed Algorithm
 * Comparison", forward pass, with the final division by the row sum and the
 * statistics stored for the backward as one log-sum-exp per row.)
 * q, k, v: inputs; o, lse: outputs, fully overwritten (rows 0..N-1).
 */
fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                 int N, int d, int causal, float scale, void* stream);

/*
 * fa_fwd for tensors in any layout whose rows hold d contiguous values, such
 * as [B, N, H, d] or K and V packed in one [B, N, 2, H, d] buffer (the
 * "Flash Attention v2" notes, "Migration from v1 to v2": the packed-KV
 * variant of the API). strides: 12 element strides, (batch, head, row) for
 * q, k, v and o in that order; each a positive multiple of 8 (16 bytes).
 * lse stays a contiguous fp32 [B, H, N] array. Results are those of fa_fwd
 * on the same values.
 */
fa_status fa_fwd_strided(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                         int H, int N, int d, const long long* strides, int causal, float scale,
                         void* stream);

/*
 * Size in bytes of the device workspace fa_bwd needs for these sizes: an
 * fp32 [B,H,N] row term D and an fp32 [B,H,N,d] dQ accumulator. Returns 0
 * for arguments fa_bwd would reject.
 */
size_t fa_bwd_workspace_size(int B, int H, int N, int d);

/*
 * Backward of the loss sum(o * dO). Recomputes S and P per tile from q, k and
 * the forward's lse ("Flash Attention v2" notes, "Backward Pass
 * Computation": recompute S block by block, then dP, dQ, dK, dV) with the
 * full softmax Jacobian:
 *   D_i = sum_c dO_ic o_ic,  P_ij = exp(scale q_i.k_j - lse_i),
 *   dS_ij = P_ij (dO_i.v_j - D_i),
 *   dq = scale dS k,  dk = scale dS^T q,  dv = P^T dO.
 * q, k, v, o, lse, dO: inputs (o and lse as written by fa_fwd with the same
 * arguments). dq, dk, dv: outputs, fully overwritten. workspace: device
 * memory of at least fa_bwd_workspace_size() bytes, 16-byte aligned, owned by
 * the caller, clobbered by the call (its contents on entry do not matter).
 */
fa_status fa_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
                 const void* dO, void* dq, void* dk, void* dv, int B, int H, int N, int d,
                 int causal, float scale, void* workspace, size_t workspace_bytes, void* stream);

/*
 * fa_bwd with the path of dQ chosen by the caller. The pages leave open how
 * the dQ contributions of the key blocks are summed ("Flash Attention v2"
 * notes, "Backward Pass Computation"; "FlashAttention-2 paper" digest, "Three
 * changes": work split over query blocks):
 *  FA_DQ_ATOMIC: the dK/dV kernel adds each (key block, query block) tile's
 *    dS K to an fp32 accumulator in the workspace with atomic adds, and a
 *    last pass converts it to bf16 (5 tile products per tile pair). The
 *    summation order of the atomics varies, so dq may differ in its last
 *    bits between runs; dk and dv do not.
 *  FA_DQ_SEPARATE (d = 64 or 128): the dK/dV kernel skips dQ, and a second,
 *    query-stationary kernel recomputes S and dP for each (query block, key
 *    block) tile and sums dQ in tensor memory (7 products per tile pair, no
 *    atomics): dq is the same bits on every run. Other d: FA_ERR_UNSUPPORTED.
 *  FA_DQ_AUTO: the path fa_bwd takes, the one measured faster for the shape.
 * Arguments, workspace and errors otherwise as for fa_bwd; an unknown dq_path
 * returns FA_ERR_INVALID_ARG.
 */
enum { FA_DQ_AUTO = 0, FA_DQ_ATOMIC = 1, FA_DQ_SEPARATE = 2 };
fa_status fa_bwd_with_dq_path(const void* q, const void* k, const void* v, const void* o,
                              const float* lse, const void* dO, void* dq, void* dk, void* dv,
                              int B, int H, int N, int d, int causal, float scale, int dq_path,
                              void* workspace, size_t workspace_bytes, void* stream);

/*
 * fa_bwd for strided tensors (see fa_fwd_strided). strides: 24 element
 * strides, (batch, head, row) for q, k, v, o, dO, dq, dk, dv in that order;
 * each a positive multiple of 8. lse and the workspace are as for fa_bwd.
 */
fa_status fa_bwd_strided(const void* q, const void* k, const void* v, const void* o,
                         const float* lse, const void* dO, void* dq, void* dk, void* dv, int B,
                         int H, int N, int d, const long long* strides, int causal, float scale,
                         void* workspace, size_t workspace_bytes, void* stream);

/*
 * The three stages fa_bwd runs, in this order, for callers that schedule or
 * time them separately. Arguments as for fa_bwd; the same workspace must be
 * passed to all three, and the stages of one backward must not overlap with
 * another call that uses that workspace.
 *  1. fa_bwd_preprocess: D_i = sum_c dO_ic o_ic, the lse rows in log2 units,
 *     and zeroes the fp32 dQ accumulator (all in the workspace).
 *  2. fa_bwd_dkdv: for every key block, loops over the query blocks,
 *     recomputes S and P, writes dk and dv, and adds each block's
 *     contribution dS K to the dQ accumulator.
 *  3. fa_bwd_dq_finalize: dq = bf16(scale * dQ accumulator).
 */
fa_status fa_bwd_preprocess(const void* o, const float* lse, const void* dO, int B, int H, int N,
                            int d, void* workspace, size_t workspace_bytes, void* stream);
fa_status fa_bwd_dkdv(const void* q, const void* k, const void* v, const void* dO, void* dk,
                      void* dv, int B, int H, int N, int d, int causal, float scale,
                      void* workspace, size_t workspace_bytes, void* stream);
fa_status fa_bwd_dq_finalize(void* dq, int B, int H, int N, int d, float scale, void* workspace,
                             size_t workspace_bytes, void* stream);

/*
 * Sequences of unequal lengths. The pages state the method for one length N;
 * for serving batches of requests of different lengths ("Flash Attention v2"
 * notes, "Performance Comparison: v1 vs v2", continuous batching; "Detailed
 * Differences", 4 "Batch and Sequence Length Support") they fix no
 * convention. Here Nq query rows attend to Nk key rows and the causal mask
 * is aligned at the bottom right: query i sees key j when j <= i + Nk - Nq,
 * so the last query sees every key; with Nq = Nk this is the rule above. A
 * query row that sees no key (causal with Nq > Nk, or a sequence with no
 * keys) gets o = 0 and lse = -inf, and its gradients are zero.
 *
 * fa_fwd_nqnk / fa_bwd_nqnk: B dense sequences, q, o, dO, dq of shape
 * [B, H, Nq, d] and k, v, dk, dv of shape [B, H, Nk, d] (Nq, Nk >= 1); lse is
 * fp32 [B, H, Nq]. strides: as for fa_fwd_strided / fa_bwd_strided (12 or
 * 24), or NULL for contiguous tensors. fa_bwd_nqnk takes a workspace of
 * fa_bwd_workspace_size(B, H, Nq, d) bytes. Errors as for fa_fwd / fa_bwd.
 */
fa_status fa_fwd_nqnk(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                      int H, int Nq, int Nk, int d, const long long* strides, int causal,
                      float scale, void* stream);
fa_status fa_bwd_nqnk(const void* q, const void* k, const void* v, const void* o,
                      const float* lse, const void* dO, void* dq, void* dk, void* dv, int B,
                      int H, int Nq, int Nk, int d, const long long* strides, int causal,
                      float scale, void* workspace, size_t workspace_bytes, void* stream);

/*
 * fa_fwd_varlen / fa_bwd_varlen: a packed batch of B sequences along the
 * token axis. q, o, dO, dq hold total_q rows and k, v, dk, dv total_k rows,
 * each row H heads of d values: [total, H, d] when strides is NULL, else
 * strides gives (head, row) element strides per tensor (8 numbers for q, k,
 * v, o; 16 for q, k, v, o, dO, dq, dk, dv), positive multiples of 8.
 * cu_seqlens_q, cu_seqlens_k: DEVICE int32 arrays of B + 1 prefix offsets
 * (0 = cu[0] <= cu[1] <= ... <= cu[B] = total); sequence b owns query rows
 * cu_seqlens_q[b] .. cu_seqlens_q[b+1]-1 and key rows cu_seqlens_k[b] ..
 * cu_seqlens_k[b+1]-1, and may be empty. max_seqlen_q / max_seqlen_k (>= 1)
 * bound the lengths. lse is fp32 [H, total_q]. The offsets are read on the
 * device: offsets that break these rules give wrong results but no access
 * outside the buffers, and are reported as FA_ERR_INVALID_ARG by the next
 * fa_last_device_status(). fa_bwd_varlen takes a workspace of
 * fa_bwd_varlen_workspace_size(B, H, total_q, max_seqlen_k, d) bytes.
 */
fa_status fa_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse,
                        const int* cu_seqlens_q, const int* cu_seqlens_k, int B, int H,
                        int total_q, int total_k, int max_seqlen_q, int max_seqlen_k, int d,
                        const long long* strides, int causal, float scale, void* stream);
size_t fa_bwd_varlen_workspace_size(int B, int H, int total_q, int max_seqlen_k, int d);
fa_status fa_bwd_varlen(const void* q, const void* k, const void* v, const void* o,
                        const float* lse, const void* dO, void* dq, void* dk, void* dv,
                        const int* cu_seqlens_q, const int* cu_seqlens_k, int B, int H,
                        int total_q, int total_k, int max_seqlen_q, int max_seqlen_k, int d,
                        const long long* strides, int causal, float scale, void* workspace,
                        size_t workspace_bytes, void* stream);

/*
 * Decode: Nq new query rows (1 <= Nq <= 16) of each of B sequences and H
 * heads against a key/value cache, the serving use the pages name
 * ("flashattention-2" glossary, "Adoption": vLLM's attention backend;
 * "Flash Attention v2" notes, "Performance Comparison: v1 vs v2": 256-token
 * generation). Computes o and lse exactly as fa_fwd_nqnk would, with the
 * keys of each (batch, head) split over several thread blocks and the parts
 * merged by their log-sum-exp (the identity behind the online softmax,
 * "Flash Attention v2" notes, "Detailed Algorithm Comparison", forward pass).
 * With Nq >= 8 it runs the tensor-core forward instead: over whole caches
 * when the (batch, head) pairs are at least as many as the GPU's SMs (the
 * workspace is then unused), else, at d = 64 and 128, with each sequence's
 * visible keys divided evenly over a number of splits that fills the SMs,
 * each split's rows normalised in fp32 and merged by log-sum-exp.
 *  q, o: bf16 [B, H, Nq, d]; k_cache, v_cache: bf16 [B, H, Nk, d]; strides: 12
 *  element strides (batch, head, row) for q, k_cache, v_cache, o as in
 *  fa_fwd_strided (a [B, Nk, H, d] cache is a view), or NULL for contiguous
 *  tensors. lse: fp32 [B, H, Nq].
 *  cache_seqlens: NULL (every sequence has Nk keys) or a DEVICE int32 array
 *  of B valid key counts in 0..Nk; the causal mask is aligned at the bottom
 *  right of each sequence's keys (row r sees key j <= r + nk - Nq). Counts
 *  outside 0..Nk are clamped and reported as FA_ERR_INVALID_ARG by the next
 *  fa_last_device_status(). Rows that see no key get o = 0, lse = -inf.
 *  workspace: device memory of fa_decode_workspace_size() bytes, 16-byte
 *  aligned (NULL is accepted when that size is 16 or less and the call needs
 *  none). Nq > 16 returns FA_ERR_UNSUPPORTED (use fa_fwd_nqnk).
 */
size_t fa_decode_workspace_size(int B, int H, int Nq, int Nk, int d);
fa_status fa_decode(const void* q, const void* k_cache, const void* v_cache, void* o, float* lse,
                    const int* cache_seqlens, int B, int H, int Nq, int Nk, int d,
                    const long long* strides, int causal, float scale, void* workspace,
                    size_t workspace_bytes, void* stream);

/*
 * Microbenchmark of the arithmetic units the softmax runs on (no counterpart
 * in the method; it measures the secondary roofs next to the tensor pipe):
 * enqueues three kernels that run independent chains of ex2.approx.ftz.f32
 * (the MUFU exponential), fma.rn.f32 and the two-lane fma.rn.f32x2 on every SM,
 * 2 blocks x 1024 threads x 8 chains x iters instructions per SM each.
 * cycles: DEVICE array of 6 unsigned 64-bit values, 8-byte aligned; after the
 * stream reaches the call, cycles[0], [2] and [4] hold the ex2, FFMA and
 * FFMA2 kernel's longest SM span in clock64 cycles, from the earlier of the
 * SM's two blocks' starts to the later of their ends (cycles[1], [3], [5]
 * are scratch). Operations per clock per SM = 16384 x iters / cycles (twice
 * that for FFMA2, which does two FMAs per instruction). iters in 1..2^20.
 */
fa_status fa_measure_unit_rates(unsigned long long* cycles, int iters, void* stream);

/*
 * Self-test of the failure path (no counterpart in the method): enqueues a
 * one-thread kernel that waits on an on-chip barrier nothing ever arrives on,
 * with a limit of limit_ms milliseconds (1..2000) instead of the 2 s the
 * attention kernels use. The wait gives up and records FA_ERR_TIMEOUT, which
 * the next fa_last_device_status() returns; the GPU context stays usable.
 */
fa_status fa_selftest_wait_timeout(int limit_ms, void* stream);

/*
 * Backward without any allocation, for callers that cannot allocate device
 * memory: code whose device memory all belongs to its own pool, or code that
 * must not call cudaMalloc while running because cudaMalloc can synchronise
 * the device and take unbounded time. The paper has no counterpart; this is a
 * deployment variant of fa_bwd.
 *
 * Same arguments, results and errors as fa_bwd, minus the workspace: the
 * library uses a fixed device array of FA_NOALLOC_SCRATCH_BYTES instead. The
 * call is accepted when fa_bwd_workspace_size(B, H, N, d) is at most
 * FA_NOALLOC_SCRATCH_BYTES, that is when
 *   4 * (2 * B*H * roundup(N, 128) + B*H*N*d) <= 33554432 bytes
 * (e.g. B*H = 15 heads of N = 4096 at d = 128); larger sizes return
 * FA_ERR_WORKSPACE before anything is enqueued. The call allocates nothing
 * and calls no allocating routine.
 * When the array is mapped: CUDA loads the library's device code lazily, per
 * device, and the array's memory is reserved at that load. The library forces
 * the load at its first call of ANY entry point on a device (that call also
 * looks up the array's device address with cudaGetSymbolAddress), and keeps
 * the array until the process exits. So a caller that hands all remaining
 * device memory to its own pool, or that captures streams into graphs, makes
 * one library call on each device before doing so; fa_last_device_status(NULL)
 * is enough. After cudaDeviceReset the next call looks the address up again in
 * the new context, so the same rule applies after a reset.
 * All calls share the one array and it keeps the last call's contents; the
 * call itself rewrites every part it reads, so nothing needs clearing. Calls
 * that overlap on the GPU (different streams or host threads) race on the
 * array and give wrong results: run them one after another.
 */
#define FA_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)
fa_status fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o,
                         const float* lse, const void* dO, void* dq, void* dk, void* dv, int B,
                         int H, int N, int d, int causal, float scale, void* stream);

/*
 * The debug build. The same sources compiled with FA_DEBUG make
 * libfa_debug.so, with the same entry points. Its kernels (a) take the limit
 * of their bounded on-chip waits from a device variable that
 * fa_set_wait_limit_ns sets, and (b) check the indices of their global-memory
 * stores (row < rows, column < d, offset inside the tensor its strides span)
 * before each store: a failed check skips the store and records
 * FA_ERR_DEVICE_CHECK, which fa_last_device_status returns. The release
 * library (libfa.so) has neither; there these calls return
 * FA_ERR_UNSUPPORTED. (No counterpart in the method: failure detection.)
 *
 * fa_is_debug_build: 1 in libfa_debug.so, 0 in libfa.so.
 * fa_set_wait_limit_ns: the wall-clock limit, in ns, of every bounded wait of
 *   the kernels on the current device (default FA_WAIT_LIMIT_NS_DEFAULT, 2 s;
 *   at most that, else FA_ERR_INVALID_ARG). 0 makes every wait that does not
 *   complete at its first try give up at once, so the next attention call
 *   takes its abort path: its roles stop, let the copies in flight land,
 *   release tensor memory, and the kernel records FA_ERR_TIMEOUT; its outputs
 *   are then undefined. Synchronises the device; not for use while other
 *   work of this library runs.
 * fa_selftest_index_check: enqueues a kernel whose one index check fails (no
 *   memory is accessed); the next fa_last_device_status returns
 *   FA_ERR_DEVICE_CHECK.
 */
#define FA_WAIT_LIMIT_NS_DEFAULT 2000000000ull
int fa_is_debug_build(void);
fa_status fa_set_wait_limit_ns(unsigned long long limit_ns);
fa_status fa_selftest_index_check(void* stream);

/*
 * Self-test of the forward softmax's FMA-pipe exponential (no counterpart in
 * the method; a numerical building block): y[i] = 2^x[i] for n >= 1 device
 * floats, evaluated exactly as the forward kernel does for part of each row
 * (range reduction, degree-3 polynomial, exponent insertion; inputs clamped
 * at -125). Maximum relative error about 7.5e-5.
 */
fa_status fa_selftest_exp2(const float* x, float* y, int n, void* stream);

/* Static, human-readable name of a status code (never NULL). */
const char* fa_status_string(int status);

/*
 * Synchronises the stream, then returns FA_ERR_TIMEOUT if any kernel of this
 * process has recorded a bounded-wait timeout since the last call,
 * FA_ERR_INVALID_ARG if a packed batch's offsets broke the rules of
 * fa_fwd_varlen or a decode cache length was outside 0..Nk (the first such
 * record wins; the call clears it),
 * FA_ERR_DEVICE_CHECK if a debug-build index check failed,
 * FA_ERR_CUDA if the synchronisation failed, else FA_OK.
 */
fa_status fa_last_device_status(void* stream);

#ifdef __cplusplus
}
#endif

#endif /* FA_H */

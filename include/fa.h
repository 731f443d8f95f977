/*
 * fa.h — C ABI of libfa_gb300: exact IO-aware softmax attention on GB300
 * (sm_103a), forward and backward, dense batches and packed variable-length
 * batches.
 *
 * Operation (all entry points):
 *   S = scale · Q Kᵀ, P = softmax(S) row by row, O = P V
 *   ("08 · FlashAttention", section 一; "LLM Systems 22: Flash Attention",
 *   section 2.1).  The forward never forms S or P in device memory: it streams
 *   K/V tiles through shared memory and keeps a running row max m and row sum
 *   l, rescaling the partial O as m grows ("LLM Systems 22", section 3.1;
 *   "08 · FlashAttention", section 二), and writes O and the row log-sum-exp
 *   only.  The backward recomputes P tile by tile from Q, K and the saved LSE
 *   ("LLM Systems 22", section 3.2; "08 · FlashAttention", section 三) and
 *   forms dV = Pᵀ dO, dP = dO Vᵀ, dS = P ∘ (dP − D), dQ = scale · dS K,
 *   dK = scale · dSᵀ Q with D_i = Σ_k dO_ik O_ik.
 *
 * Conventions shared by every entry point:
 *   - Element type: bf16 for q, k, v, o, do, dq, dk, dv (raw 16-bit words),
 *     fp32 for lse and the workspace.
 *   - Dense layout [B, N, H, d], row-major: element (b, n, h, k) at
 *     ((b·N + n)·H + h)·d + k — the token-major layout of the ``mha_fwd``
 *     entry in "Flash Attention实现深度解析" (seekfood), section 3.1.
 *     Packed layout [T, H, d]: sequence s occupies rows
 *     cu_seqlens[s] .. cu_seqlens[s+1]−1.
 *   - LSE: fp32 [B, H, N] (packed: [nseq, H, max_seqlen]); natural log of the
 *     scaled scores, LSE_i = ln Σ_j exp(S_ij) over visible keys.  Entries
 *     past a packed sequence's length are not written.
 *   - causal != 0: key j is visible to query i iff j <= i (within a sequence);
 *     no other masks are supported ("08 · FlashAttention", section 四).
 *   - d must be 64 or 128.  Every pointer must be a device pointer, 16-byte
 *     aligned, all on one device; the call makes the device owning q current
 *     on the calling thread and launches there.  The caller owns every
 *     buffer; the library allocates nothing and never frees.  All work is
 *     enqueued on `stream` (a cudaStream_t of that device; NULL = legacy
 *     default stream) and returns without synchronising.
 *   - Errors: argument errors are detected on the host before any launch and
 *     returned as a non-zero fa_status; nothing is enqueued then.  There is
 *     no fallback path: an unsupported case is an error, never a slower
 *     route.  Device-side failures (a bounded wait that ran out) are reported
 *     by fa_get_device_error().
 *   - Device state: per device, the library caches the device addresses of
 *     its static device variables (the error word, the no-alloc scratch)
 *     and the kernels' shared-memory limits, on first use.  A
 *     cudaDeviceReset() invalidates them: do not use the library on a device
 *     after resetting it in the same process.
 */
#ifndef FA_GB300_H
#define FA_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define FA_API __attribute__((visibility("default")))
#else
#define FA_API
#endif

typedef int fa_status;

enum {
  FA_OK = 0,
  FA_ERR_NULL = 1,          /* a required pointer is NULL */
  FA_ERR_ALIGN = 2,         /* a pointer is not 16-byte aligned */
  FA_ERR_HEAD_DIM = 3,      /* d not in {64, 128} */
  FA_ERR_SHAPE = 4,         /* B, H, N, nseq, total or max_seqlen out of range (among them: more
                               than 2^31 - 1 (sequence, head, 128-row tile) triples) */
  FA_ERR_ARCH = 5,          /* current device is not compute capability 10.3 */
  FA_ERR_CUDA = 6,          /* a CUDA runtime/driver call or launch failed */
  FA_ERR_TIMEOUT = 7,       /* a kernel's bounded wait expired (device side) */
  FA_ERR_WORKSPACE = 8,     /* workspace missing or smaller than required */
  FA_ERR_SCALE = 9,         /* scale not finite */
  FA_ERR_NOT_DEVICE = 10,   /* q is not device memory (its device is the one launched on) */
  FA_ERR_SCRATCH_LIMIT = 11 /* fa_bwd_noalloc: problem needs more than FA_NOALLOC_SCRATCH_BYTES */
};

/* Human-readable name of a status code (static string, never NULL). */
FA_API const char* fa_status_string(fa_status status);

/*
 * Forward, dense batch.
 *   q, k, v  [in]  bf16 [B, N, H, d]
 *   o        [out] bf16 [B, N, H, d]
 *   lse      [out] fp32 [B, H, N]
 *   scale    softmax scale applied to Q Kᵀ (usually 1/sqrt(d))
 * Tiling with online softmax: "LLM Systems 22", section 3.1 and
 * "08 · FlashAttention", section 二 (query tile outer, key/value tiles inner,
 * O written once).
 */
FA_API fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
                 float scale, int causal, void* stream);

/* Bytes of fp32 workspace fa_bwd needs: D [B, H, N] (padded to 256 bytes)
 * followed by the dQ accumulator, H·d values for each of B·N rows rounded up
 * to a multiple of 128. */
FA_API size_t fa_bwd_workspace_bytes(int B, int H, int N, int d);

/*
 * Backward, dense batch.  Recomputes P from q, k and lse ("LLM Systems 22",
 * section 3.2: keep only the row statistics, reload Q, K, V tile by tile and
 * rebuild the attention tile on chip).
 *   q, k, v, o, dout [in]  bf16 [B, N, H, d] (o and lse from fa_fwd)
 *   lse              [in]  fp32 [B, H, N]
 *   dq, dk, dv       [out] bf16 [B, N, H, d]
 *   workspace        device scratch of at least fa_bwd_workspace_bytes(),
 *                    16-byte aligned; contents on entry are ignored.
 */
FA_API fa_status fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
                 void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes, int B, int H, int N, int d,
                 float scale, int causal, void* stream);

/*
 * Forward, packed variable-length batch ("08 · FlashAttention", section 四:
 * packing with cu_seqlens instead of a padding mask).
 *   q, k, v     [in]  bf16 [total, H, d]
 *   o           [out] bf16 [total, H, d]
 *   lse         [out] fp32 [nseq, H, max_seqlen]
 *   cu_seqlens  [in]  device int32 [nseq + 1], cu_seqlens[0] = 0, non-decreasing,
 *               cu_seqlens[nseq] = total, every length <= max_seqlen.  The
 *               library does not read it on the host; a violation is
 *               undefined behaviour (out-of-range rows are not touched, but
 *               results are meaningless).
 */
FA_API fa_status fa_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse, const int* cu_seqlens,
                        int nseq, int max_seqlen, int total, int H, int d, float scale, int causal, void* stream);

/* Workspace for fa_bwd_varlen: D [nseq, H, max_seqlen] (padded to 256 bytes)
 * and the fp32 dQ accumulator for `total` rows rounded up to a multiple of
 * 128, H·d values each. */
FA_API size_t fa_bwd_varlen_workspace_bytes(int total, int nseq, int max_seqlen, int H, int d);

/* Backward, packed variable-length batch; arguments as fa_bwd and
 * fa_fwd_varlen. */
FA_API fa_status fa_bwd_varlen(const void* q, const void* k, const void* v, const void* o, const void* dout,
                        const float* lse, void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes,
                        const int* cu_seqlens, int nseq, int max_seqlen, int total, int H, int d, float scale,
                        int causal, void* stream);

/*
 * Decode forward against a key/value cache, split along the cache ("LLM
 * Systems 22: Flash Attention", sections 5.1 and 5.2: Split-KV /
 * Flash-Decoding).  q, o: bf16 [B, Nq, H, d], the Nq (1 .. 8) newest tokens;
 * k, v: bf16 [B, Nk, H, d], the whole cache including those tokens.  lse:
 * fp32 [B, H, Nq].  causal != 0: the new tokens are the cache's last Nq
 * positions, so query i sees keys j <= Nk − Nq + i (lower-right alignment;
 * with Nq = 1 every key); causal == 0: every key.  The cache is split into
 * chunks of 128 to 1024 keys; each chunk's partial softmax statistics and
 * unnormalised output go to `workspace` (at least
 * fa_decode_workspace_bytes(B, H, Nq, Nk, d) bytes, 16-byte aligned, caller
 * owned) and a second kernel merges them.  Other conventions as fa_fwd.
 * Nq outside 1 .. 8 or Nk < 1 is FA_ERR_SHAPE; a short workspace is
 * FA_ERR_WORKSPACE.
 */
FA_API size_t fa_decode_workspace_bytes(int B, int H, int Nq, int Nk, int d);
FA_API fa_status fa_fwd_decode(const void* q, const void* k, const void* v, void* o, float* lse, void* workspace,
                               size_t workspace_bytes, int B, int H, int Nq, int Nk, int d, float scale, int causal,
                               void* stream);

/*
 * Synchronises `stream`, then reads and clears the error word of the device
 * the stream belongs to (NULL, the legacy default stream: the current
 * device); the calling thread's current device is left as it was.  Returns
 * FA_OK, FA_ERR_TIMEOUT (some kernel's bounded mbarrier wait ran out and the
 * kernel returned early: its outputs are invalid) or FA_ERR_CUDA (the
 * synchronisation or the read itself failed).
 */
FA_API fa_status fa_get_device_error(void* stream);

/* Text describing the most recent FA_ERR_CUDA returned on the calling host
 * thread (which call failed and the CUDA error string); "" if none.  The
 * string is owned by the library and valid until the next call on this
 * thread. */
FA_API const char* fa_last_error_detail(void);

/*
 * Self-test of the bounded-wait path (no counterpart on the pages): launches
 * one CTA that waits on an mbarrier nothing ever arrives on, with a limit of
 * `limit_ns` nanoseconds (clamped to [1e3, 2e9]).  The kernel gives up after
 * the limit, records FA_ERR_TIMEOUT in the error word and exits normally, so
 * fa_get_device_error() afterwards returns FA_ERR_TIMEOUT.
 */
FA_API fa_status fa_selftest_wait_timeout(uint64_t limit_ns, void* stream);

/*
 * Unit-rate microbenchmarks for the MUFU-vs-tensor argument ("LLM Systems
 * 22: Flash Attention", section 4.1.2: exponential cycles against GEMM
 * cycles; section 4.2: how the two rates scale on Blackwell).  Runs one CTA
 * per SM on the current device, synchronises `stream`, and writes to
 * *result the rate per SM per SM-clock (measured with the SM cycle counter):
 *   which = 0: ex2.approx.f32 results per SM-clock
 *           1: cvt.rn.bf16x2.f32 conversions per SM-clock
 *           2: fp32 FMAs per SM-clock
 *           3: tcgen05.mma bf16 FLOPs per SM-clock, M=128 N=256 K=16, SMEM operands
 *           4: the same with N=128
 *           5: the same with N=128 and the A operand read from TMEM
 *           6, 7: cases 3 and 5 with pseudo-random bf16 operands instead of
 *              zeros (the data a real GEMM switches, and the power it draws)
 *           8: bf16 FLOPs per SM-clock of the forward kernel's MMA stream
 *              alone (two query tiles: O_t += P_t V with P_t from TMEM,
 *              then S_t = Q K^T over P_t's columns; d = 128)
 *           9: the same with 64-column O tiles
 *          10: case 9 with P_t in TMEM columns that no MMA writes
 *          11: case 8 with both PV MMAs issued before both S MMAs
 *          38: exponentials per SM per clock in the softmax's per-pair step
 *              with its bf16 packing: two ex2 + one cvt.rn.bf16x2.f32
 *          40: the forward softmax's full per-pair step (paired FMA, two
 *              ex2, paired add into the row sum, cvt pack), in exponentials
 *          42: largest relative difference of the polynomial exp2 (FMA pipe)
 *              from ex2.approx over [-30, 8]; -1 if a clamped input gave a
 *              negative, NaN or non-tiny value
 *          43: step 40 with a quarter of the pairs through the polynomial exp2
 * `iters` (1 .. 2^20) sets the loop length.  Returns FA_ERR_SHAPE for an
 * unknown `which` or out-of-range `iters`.
 */
FA_API fa_status fa_microbench(int which, int iters, double* result, void* stream);

/*
 * Kernel timing hook (no counterpart on the pages; for measurement only).
 * Makes the next fa_bwd / fa_bwd_varlen call issued from this host thread
 * record `start_event` immediately before and `end_event` immediately after
 * its main kernel (the tile loop), on that call's stream, so the caller can
 * time that kernel alone with cudaEventElapsedTime.  Both are cudaEvent_t
 * handles created by the caller; the hook is consumed by that one call.
 * Passing NULL for both clears a pending hook.
 */
FA_API fa_status fa_set_kernel_events(void* start_event, void* end_event);

/*
 * Launch order of the attention kernels' CTAs (host only, needs no GPU; for
 * inspection and tests).  Both the forward and the backward launch one CTA
 * per (pair, tile) item, pair = sequence·H + head, tile = the kernel's tile
 * index in its heaviest-first order under a causal mask (forward: query-tile
 * groups from the last; backward: key tiles from the first), following the
 * longest-processing-time-first scheduling of causal attention ("LLM Systems
 * 22: Flash Attention", section 4.1.5).  CTAs start in launch order as SMs
 * free up.  The items go in groups of `group` consecutive pairs: every tile
 * of a group before the next group; within a group, tile by tile, pairs in
 * order.  `group` is the smallest divisor of npairs whose group·ntiles items
 * fill at least one wave of `slots` resident CTAs (searched up to four times
 * that size), else npairs.  Launch configurations: the forward takes
 * 256 query rows per tile at d = 128 (one CTA per SM) and 128 at d = 64 (two
 * per SM); the backward 128 keys per tile, one CTA per SM.
 *   npairs, ntiles, slots  positive; npairs·ntiles <= 2^31 − 1
 *   group                  [out] the group size (may be NULL)
 *   pair, tile             [out] host int arrays of `capacity` entries (may be
 *                          NULL): the item of launch index b for b < capacity
 * Returns FA_ERR_SHAPE for sizes out of range.
 */
FA_API fa_status fa_cta_order(int npairs, int ntiles, int slots, int* group, int* pair, int* tile,
                              long long capacity);

/*
 * Backward, dense batch, without a caller-supplied workspace.  (The pages
 * have no counterpart: this is a deployment convenience.)
 *
 * Some callers cannot allocate device memory at the point where they need
 * the backward: a plugin running inside a host framework that owns all
 * device memory and hands the plugin no workspace, or a latency-critical
 * path where allocating is forbidden because it can synchronise the device
 * or fail under fragmentation.  This entry point serves them: it takes the
 * same arguments as fa_bwd minus the workspace and allocates nothing (no
 * cudaMalloc, cudaFree or allocating library routine).  Its scratch — the D
 * row statistic and the fp32 dQ accumulator, exactly what
 * fa_bwd_workspace_bytes() sizes — lives in one file-scope static device
 * array of FA_NOALLOC_SCRATCH_BYTES bytes that every GPU which loads the
 * library holds until the process exits.
 *
 *   - Limit: problems whose fa_bwd_workspace_bytes(B, H, N, d) exceeds
 *     FA_NOALLOC_SCRATCH_BYTES are rejected with FA_ERR_SCRATCH_LIMIT before
 *     anything is enqueued (e.g. B=1, H=8, N=4096, d=128 needs 16.9 MB and
 *     fits; B=1, H=16, N=4096, d=128 needs 33.8 MB and does not).
 *   - Set-up: the first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current and caches it; make
 *     that first call before any stream capture.
 *   - Sharing: every call on a device uses the same array.  The kernels
 *     re-initialise the parts that must start at zero on every call, so stale
 *     contents from an earlier call do not leak in, but two calls that
 *     overlap on the GPU (different streams, or concurrent host threads)
 *     race on the array and produce wrong gradients: serialise them.
 * Other arguments, layouts and errors are those of fa_bwd.
 */
#define FA_NOALLOC_SCRATCH_BYTES (32u << 20)
FA_API fa_status fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const void* dout,
                                const float* lse, void* dq, void* dk, void* dv, int B, int H, int N, int d,
                                float scale, int causal, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_H */

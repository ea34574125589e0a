/*
 * attn.h -- C ABI of the GB300 (sm_103a) exact attention forward library
 * (libattn_sm103.so).
 *
 * What is computed.  For query row i of head hq in batch b:
 *     O[b,i,hq,:] = sum_j P_ij V[b,j,hkv,:],   P_ij = exp(s_ij - LSE_i),
 *     s_ij = scale * <Q[b,i,hq,:], K[b,j,hkv,:]>   (-inf where masked),
 *     LSE_i = ln sum_j exp(s_ij),
 * i.e. O = softmax(scale * Q K^T + mask) V plus the per-row natural-log
 * log-sum-exp ("FlashAttention: Part 2", chizkidd.github.io, section 2.1
 * for the function and section 1.3 for the one LSE per row).  The result is
 * reached by tiling over K/V blocks with a running max and sum (same page,
 * section 6.2); the N x N score matrix is never written to memory.
 *
 * Grouped heads: Hkv divides Hq and query head hq reads KV head
 * hq / (Hq / Hkv) (pyshine.com flash-attention tour, "Why You Need This":
 * K and V may carry fewer heads than Q when the counts divide).
 * Masks: causal aligned top-left (key j visible to row i iff j <= i) or
 * bottom-right, and a local window (attn_fwd_window, attn_fwd_kvcache).
 * A row that sees no key gets O = 0 and LSE = -inf.
 *
 * Layout: every tensor is dense and row-major, BSHD with d innermost:
 *     q, o : [B, Nq, Hq, d]  bf16
 *     k, v : [B, Nk, Hkv, d] bf16
 *     lse  : [B, Hq, Nq]     fp32
 * Supported head dims: d = 64 and d = 128.
 *
 * Ownership: every pointer is device memory owned by the caller.  The
 * library allocates nothing and keeps no pointer after a call returns.
 * Every call is asynchronous on the given stream (a cudaStream_t passed as
 * void*, NULL for the legacy default stream); nothing synchronises except
 * attn_get_device_status.
 *
 * Errors: arguments are checked on the host before anything is launched; a
 * failed check returns its code and launches nothing.  No exception crosses
 * this interface.  Problems only the device can see (a pipeline wait that
 * ran out of time, a cache length outside [0, max_seqlen]) are recorded in
 * a library-wide device status word that attn_get_device_status reports.
 * When it reports ATTN_ERR_TIMEOUT, the o and lse of the calls made since
 * the previous status read are undefined (they may hold finite values).
 */
#ifndef ATTN_SM103_H
#define ATTN_SM103_H

#include <stddef.h>

/* Exported symbols of the shared library (everything else is hidden). */
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
  ATTN_ERR_INVALID_ARG = 1,  /* a size, head count, scale or pointer is invalid */
  ATTN_ERR_UNSUPPORTED = 2,  /* valid but not built: d not in {64, 128}, ... */
  ATTN_ERR_MISALIGNED = 3,   /* a pointer is not 16-byte aligned */
  ATTN_ERR_LAUNCH = 4,       /* the CUDA runtime refused a launch or a query */
  ATTN_ERR_TIMEOUT = 5,      /* device: a pipeline wait gave up (reported later) */
  ATTN_ERR_DEVICE_ARG = 6,   /* device: a cache length or page index was out of range */
  ATTN_ERR_WORKSPACE = 7     /* workspace missing or smaller than required */
} attn_status;

#define ATTN_CAUSAL_NONE 0
#define ATTN_CAUSAL_TOP_LEFT 1
#define ATTN_CAUSAL_BOTTOM_RIGHT 2

/*
 * Prefill / training-shape forward.
 *   q [B,Nq,Hq,d], k and v [B,Nk,Hkv,d] bf16 in; o [B,Nq,Hq,d] bf16 and
 *   lse [B,Hq,Nq] fp32 out.
 *   causal: ATTN_CAUSAL_NONE (0); ATTN_CAUSAL_TOP_LEFT (1): key j is seen
 *            by row i iff j <= i; ATTN_CAUSAL_BOTTOM_RIGHT (2): iff
 *            j <= i + Nk - Nq, so the last query row sees every key (the
 *            alignment the pyshine.com flash-attention tour names; with
 *            Nq > Nk the first Nq - Nk rows see none: O = 0, LSE = -inf).
 *   scale: finite softmax scale applied to Q K^T (1/sqrt(d) usually).
 * Tiled over 128-row query tiles and 128-key K/V tiles: TMA loads into
 * shared memory, tcgen05 MMAs accumulate S = Q K^T and O += P V in Tensor
 * Memory, the softmax runs on CUDA cores with an online running max/sum
 * ("FlashAttention: Part 2", section 6.2), normalisation is deferred to the
 * end and the O rescale is skipped when a row's max did not move
 * ("Trace FlashAttention's evolution through plain PyTorch code", FA2 and
 * FA4 paragraphs); key tiles wholly above the causal diagonal are skipped.
 * Constraints: B, Hq, Hkv >= 1; Nq >= 0; Nk >= 0; Hq % Hkv == 0;
 * d in {64, 128}; all pointers 16-byte aligned (lse: 4-byte) and non-NULL
 * unless B*Nq == 0.  Nq + Nk must stay below 2^31 - 256.
 */
ATTN_API attn_status attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                     int B, int Hq, int Hkv, int Nq, int Nk, int d,
                     int causal, float scale, void* stream);

/*
 * Local (sliding-window) attention: attn_fwd with a window (window_left,
 * window_right).  Query row i sits at key position pos_i = i + Nk - Nq
 * (aligned bottom-right) and sees key j only if
 *     pos_i - window_left <= j <= pos_i + window_right
 * ("FlashAttention: Part 2", section 3.2: local attention keeps i -> j only
 * for |i - j| <= w; the pyshine.com tour, "From Install to Causal
 * Attention", passes the window as a (left, right) pair next to causal, as
 * in causal with (1023, 0)).  A negative side is unbounded; (-1, -1) is
 * attn_fwd.  The window intersects the causal mask chosen by `causal`;
 * with causal = 0, (w, 0) is bottom-right causal attention over the last
 * w + 1 keys.  Key tiles outside every row's window are never loaded.
 * Arguments, constraints and errors otherwise as for attn_fwd; the inputs
 * must be finite wherever a tile is loaded (keys of [0, Nk) in tiles that
 * some row's window touches).
 */
ATTN_API attn_status attn_fwd_window(const void* q, const void* k, const void* v, void* o, float* lse,
                     int B, int Hq, int Hkv, int Nq, int Nk, int d, int causal,
                     int window_left, int window_right, float scale, void* stream);

/*
 * The same forward against a KV cache with a length per sequence: a block
 * of Nq new query rows (a chunk of a prompt, or several decode tokens)
 * attends to the first seqlens[b] keys of sequence b (pyshine.com
 * flash-attention tour, "Why You Need This": prefill and decode against a
 * KV cache with per-sequence lengths).
 *   q [B,Nq,Hq,d] bf16; k_cache, v_cache [B,max_seqlen,Hkv,d] bf16;
 *   seqlens: device int32 [B], each in [0, max_seqlen]; keys at or past
 *            seqlens[b] are never read into the result, whatever they hold;
 *   o [B,Nq,Hq,d] bf16, lse [B,Hq,Nq] fp32 out;
 *   causal: as for attn_fwd, with Nk = seqlens[b]: ATTN_CAUSAL_BOTTOM_RIGHT
 *            puts query row i at cache position seqlens[b] - Nq + i (the
 *            new rows are the last Nq keys of the cache).
 *   window_left, window_right: a local window as for attn_fwd_window,
 *            positions taken with Nk = seqlens[b]; -1, -1 for none.
 * Constraints and errors are those of attn_fwd; a seqlens entry outside
 * [0, max_seqlen] is clamped and reported as ATTN_ERR_DEVICE_ARG by
 * attn_get_device_status.
 */
ATTN_API attn_status attn_fwd_kvcache(const void* q, const void* k_cache, const void* v_cache,
                             const int* seqlens, int max_seqlen, void* o, float* lse,
                             int B, int Hq, int Hkv, int Nq, int d, int causal,
                             int window_left, int window_right, float scale, void* stream);

/*
 * Bytes of workspace attn_fwd_splitkv needs: fp32 partial outputs and
 * partial LSEs for ceil(max_seqlen / chunk) splits of every (b, hq).
 * Returns 0 for invalid arguments.
 */
ATTN_API size_t attn_splitkv_workspace_size(int B, int Hq, int max_seqlen, int d, int chunk);

/*
 * Query-length-one decode against a KV cache, split over the key axis
 * (pyshine.com flash-attention tour, "Why You Need This": with one query
 * the cache is split across thread blocks and the partial results are
 * combined).
 *   q [B,1,Hq,d] bf16; k_cache, v_cache [B,max_seqlen,Hkv,d] bf16;
 *   seqlens: device int32 [B], valid cache length of each sequence
 *            (keys 0 .. seqlens[b]-1 are attended; nothing at or beyond
 *            seqlens[b] is read into the result, whatever it holds);
 *   o [B,1,Hq,d] bf16 and lse [B,Hq,1] fp32 out;
 *   chunk: keys per split, a positive multiple of 64 (1024 typical);
 *   workspace: device memory of at least
 *            attn_splitkv_workspace_size(B, Hq, max_seqlen, d, chunk) bytes,
 *            16-byte aligned, owned by the caller, contents ignored on entry.
 * Two launches on `stream`: the split kernel writes each split's
 * normalised partial output and LSE to the workspace, the combine kernel
 * merges them.  A seqlens entry outside [0, max_seqlen] is clamped and
 * reported as ATTN_ERR_DEVICE_ARG by attn_get_device_status.
 */
ATTN_API attn_status attn_fwd_splitkv(const void* q, const void* k_cache, const void* v_cache,
                             const int* seqlens, int max_seqlen,
                             void* o, float* lse,
                             int B, int Hq, int Hkv, int d, float scale, int chunk,
                             void* workspace, size_t workspace_bytes, void* stream);

/*
 * The same decode against a paged KV cache (pyshine.com flash-attention
 * tour, "Why You Need This": a paged KV cache for serving).  Key k of
 * sequence b lives in row k % page_size of page block_table[b][k / page_size]
 * of the page pools:
 *   k_pages, v_pages [num_pages, page_size, Hkv, d] bf16, 16-byte aligned;
 *   block_table: device int32 [B, max_blocks], row b lists the pages of
 *            sequence b in key order (entries past its length are not read);
 *   page_size: a positive multiple of 64 (the kernel's key tile), with
 *            chunk / page_size + 2 <= 128 (pages of one split);
 *   seqlens: device int32 [B], each in [0, max_blocks * page_size].
 * The other arguments, the workspace (sized for max_seqlen = max_blocks *
 * page_size) and the results are those of attn_fwd_splitkv.  A page index
 * outside [0, num_pages) is replaced by page 0 for the read and reported as
 * ATTN_ERR_DEVICE_ARG by attn_get_device_status.
 */
ATTN_API attn_status attn_fwd_splitkv_paged(const void* q, const void* k_pages, const void* v_pages,
                                            const int* block_table, int max_blocks, int page_size,
                                            int num_pages, const int* seqlens,
                                            void* o, float* lse,
                                            int B, int Hq, int Hkv, int d, float scale, int chunk,
                                            void* workspace, size_t workspace_bytes, void* stream);

/*
 * Split-KV decode that allocates nothing, for callers that cannot call
 * cudaMalloc or pass a workspace: code running inside a custom allocator or
 * memory-pool callback, under a strict no-allocation policy of an inference
 * server's hot loop, or behind a plain C interface with no device memory of
 * its own to spare.  The paper has no counterpart to this entry point.
 *
 * Same arguments and results as attn_fwd_splitkv, minus the workspace: the
 * partial results go to a fixed scratch array compiled into the library,
 * ATTN_SPLITKV_NOALLOC_MAX_BYTES (8 MiB) in size, which every GPU that loads
 * the library holds until the process exits.  That covers, for example,
 * B=16, Hq=32, d=128, max_seqlen=16384, chunk=1024 (about 4.2 MB).
 *   - Arguments are checked as attn_fwd_splitkv checks them, with the same
 *     codes, before the size check; then it returns ATTN_ERR_WORKSPACE,
 *     launching nothing and making no CUDA call, when
 *     attn_splitkv_workspace_size(B, Hq, max_seqlen, d, chunk) exceeds the
 *     scratch size.
 *   - Calls no cudaMalloc, cudaFree or other allocating routine.
 *   - The first call on a device (with that device current) looks up the
 *     scratch's device address once and keeps it until the process exits;
 *     make that first call before any stream capture.  A device reset
 *     (cudaDeviceReset) after that first call is not supported: the kept
 *     address would no longer be valid.  Returns ATTN_ERR_LAUNCH if the
 *     lookup fails.
 *   - If a split's pipeline wait times out, the combine still reads that
 *     split's scratch rows, which then hold an earlier call's values: o and
 *     lse are undefined whenever attn_get_device_status reports
 *     ATTN_ERR_TIMEOUT.
 *   - Every call on a device shares the one scratch array, which keeps the
 *     last call's contents (nothing needs clearing: each call writes every
 *     partial it reads).  Calls whose kernels may overlap on the GPU (on
 *     different streams with no ordering between them) race on it: order
 *     them on one stream or with events.
 */
#define ATTN_SPLITKV_NOALLOC_MAX_BYTES (8u << 20)
ATTN_API attn_status attn_fwd_splitkv_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                              const int* seqlens, int max_seqlen,
                                              void* o, float* lse,
                                              int B, int Hq, int Hkv, int d, float scale, int chunk,
                                              void* stream);

/*
 * Synchronises `stream`, then reads and clears the library's device status
 * word.  Returns ATTN_OK, ATTN_ERR_TIMEOUT, ATTN_ERR_DEVICE_ARG, or
 * ATTN_ERR_LAUNCH if the stream itself reports an error.
 */
ATTN_API attn_status attn_get_device_status(void* stream);

/*
 * Self-test of failure detection.  Every wait of the library's kernels on a
 * pipeline barrier is bounded: when it runs out (2 s) the kernel records
 * ATTN_ERR_TIMEOUT, lets its in-flight copies and tensor-core work finish,
 * frees its Tensor Memory and returns, instead of hanging.  This call
 * launches one small kernel on `stream` whose waits can never be satisfied
 * (barriers that nothing completes): one warp gives up after limit_ns
 * (clamped to [1 us, 2 s]) and the other, with the full limit, must give up
 * as soon as it sees the first one's abort.  Afterwards
 * attn_get_device_status returns ATTN_ERR_TIMEOUT once and the context is
 * usable.  Returns ATTN_OK when the kernel was launched.  The pages have no
 * counterpart to this call; it exists so that the timeout path can be
 * tested without a GPU fault.
 */
ATTN_API attn_status attn_selftest_wait_timeout(unsigned long long limit_ns, void* stream);

/*
 * Self-test of the software exponential: y[i] = 2^x[i] computed the way the
 * prefill kernel computes a fraction of the softmax's exponentials when the
 * library is built with ATTN_EXP2_POLY = K > 0 (every K-th pair of a row's
 * p values), which FA4 does on Blackwell to relieve the MUFU unit
 * ("FlashAttention: Part 2", sections 1.7 and 1.8).  Cody and Waite's range
 * reduction x = n + f, |f| <= 1/2, a degree-3 polynomial for 2^f (largest
 * relative error 1.01e-4 over [-1/2, 1/2]) and n added to the exponent; x is
 * clamped to [-125, 64] first.  Present in every build (the default build's
 * prefill uses the MUFU exponential for every p).
 *   x, y: device float32 arrays of n elements, 4-byte aligned.
 * Returns ATTN_OK once launched on `stream`; ATTN_ERR_INVALID_ARG for n < 0
 * or a NULL pointer (n > 0).
 */
ATTN_API attn_status attn_selftest_exp2_poly(const float* x, float* y, long long n, void* stream);

/*
 * Measurement helper: reads `bytes` of device memory at `buf` once, as a
 * plain stream of 16-byte loads with several in flight per thread over the
 * whole GPU, and XORs a fold of the data into *sink (device memory, 8-byte
 * aligned; its value is meaningless, it only keeps the loads).  Timed on a
 * buffer far larger than L2, it gives the HBM read rate a read-bound kernel
 * (the split-KV decode) is measured against, next to the copy rate.  The
 * pages have no counterpart to this call.
 *   buf: 16-byte aligned, bytes a multiple of 16.
 * Returns ATTN_OK once launched on `stream`.
 */
ATTN_API attn_status attn_probe_read_bandwidth(const void* buf, size_t bytes, unsigned long long* sink,
                                               void* stream);

/* Static, human-readable name of a status code. Never NULL. */
ATTN_API const char* attn_status_string(attn_status s);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_SM103_H */

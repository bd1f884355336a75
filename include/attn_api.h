/*
 * attn_api.h -- C ABI of the B300 (sm_103a) exact self-attention forward library
 * (libattn_fwd.so).
 *
 * The operation (every entry point below computes exactly this, up to rounding):
 *
 *   for every batch b, query head hq, query row i:
 *     kv    = hq / (Hq / Hkv)                               grouped-query head map
 *     L     = N, or key_len[b] for attn_fwd_padded         valid (unpadded) length
 *     J(i)  = { j : i < L && j < L && (!causal || j <= i)
 *                   && (window == 0 || i - j < window)
 *                   && (window == 0 || causal || j - i < window) }
 *     s_ij  = scale * q[b,hq,i,:] . k[b,kv,j,:]              for j in J(i)
 *     lse_i = ln( sum_{j in J(i)} exp(s_ij) )                natural log, scale included
 *     o[b,hq,i,:] = sum_{j in J(i)} exp(s_ij - lse_i) * v[b,kv,j,:]
 *
 * Sources, by page and section: the attention score QK^T/sqrt(D) and
 * Attention = Softmax(score) V ("Background - Attention Mechanism" on the SpAtten
 * review, coolstone2000.github.io); scaling by sqrt(d_k), the row softmax, the
 * weighted sum of V, independent heads and the look-ahead mask under which a token
 * attends to itself and earlier tokens (palettepath-it.com self-attention guide,
 * sections on scaled dot-product scores, softmax normalisation, parallel heads and
 * look-ahead masking); grouped-query and sliding-window attention as compared
 * variants ("Attentions Under the Microscope" summary, gist.science, section
 * "방법론"); the tensor layout [batch, heads, n, d] of the framework call
 * F.scaled_dot_product_attention(q, k, v) (devhandbook.co.kr, Example 2). The head
 * map kv = hq / G and the window rule i - j < window are readings of the pages,
 * which name both variants without fixing either; without the look-ahead mask the
 * window is read symmetrically, |i - j| < window (the sliding-window row of the
 * devhandbook.co.kr comparison table). Padding follows the guide's padding mask:
 * padded tokens neither give nor receive attention (section "패딩 마스킹 (Padding
 * Masking)"), with validity per token read as right padding, as in the
 * devhandbook.co.kr variable-length example ("Example 7"). A row with no visible key
 * (a padded row) gets o = 0 and lse = -inf.
 *
 * Conventions shared by every entry point:
 *   - Tensors are dense and contiguous, row-major, in the layouts stated per
 *     argument. bf16 means IEEE bfloat16 bit patterns (2 bytes).
 *   - The caller owns every buffer. The library allocates nothing per call and keeps
 *     only a per-device table of cached device attributes plus one device-side
 *     status word per device (see attn_device_error).
 *   - Calls are asynchronous with respect to the host on `stream` (a cudaStream_t
 *     passed as void*; NULL = the legacy default stream) and never synchronise,
 *     except attn_device_error and attn_selftest_wait_timeout, which say so.
 *   - Argument errors are detected on the host before anything is launched or any
 *     memory is touched; the call then returns a negative attn_status and has no
 *     other effect. No error is fatal.
 *   - Calls on different streams, from different host threads, are safe.
 *   - Stream order is kept. Each kernel is launched as a programmatic dependent of the
 *     kernel before it on the stream: its prologue (barriers, tensor-memory allocation,
 *     tensor-map prefetch) may run while that kernel finishes, but it touches no global
 *     memory before that kernel has completed and its writes are visible
 *     (griddepcontrol.wait). A kernel that follows one of these calls and was itself
 *     launched with programmatic stream serialisation must wait likewise. Inside a CUDA
 *     graph the same holds through programmatic dependency edges.
 */
#ifndef ATTN_API_H
#define ATTN_API_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    ATTN_OK = 0,
    ATTN_ERR_NULLPTR = -1,     /* a required pointer is NULL */
    ATTN_ERR_ALIGN = -2,       /* q, k, v, o not 16-byte aligned, or lse not 4-byte aligned */
    ATTN_ERR_SHAPE = -3,       /* B, Hq, Hkv or N < 1; Hq % Hkv != 0; window < 0;
                                  scale not finite and > 0; sizes beyond the index range */
    ATTN_ERR_UNSUPPORTED = -4, /* d not 64 or 128; the current device is not an sm_103
                                  (B300-class) GPU */
    ATTN_ERR_CUDA = -5,        /* a CUDA runtime call failed; see attn_last_cuda_error */
    ATTN_ERR_TIMEOUT = -6,     /* a kernel wait gave up (reported by attn_device_error) */
    ATTN_ERR_WORKSPACE = -7,   /* the caller's workspace is smaller than required */
    ATTN_ERR_SCRATCH_LIMIT = -8, /* attn_fwd_decode_noalloc: the split results would need more
                                   than its fixed scratch (ATTN_DECODE_NOALLOC_SCRATCH_BYTES) */
    ATTN_ERR_BOUNDS = -9        /* debug build only: an index check failed (attn_device_error) */
} attn_status;

/*
 * attn_fwd -- exact attention forward on device buffers.
 *
 *   q    device, bf16 [B, Hq,  N, d], 16-byte aligned (read)
 *   k    device, bf16 [B, Hkv, N, d], 16-byte aligned (read)
 *   v    device, bf16 [B, Hkv, N, d], 16-byte aligned (read)
 *   o    device, bf16 [B, Hq,  N, d], 16-byte aligned (written; fp32 accumulation,
 *        rounded to nearest even once at the end)
 *   lse  device, fp32 [B, Hq, N], 4-byte aligned (written; natural-log log-sum-exp
 *        of the scaled scores over J(i))
 *   B, Hq, Hkv, N, d   sizes; Hq must be a multiple of Hkv; d is 64 or 128
 *   causal  0 = bidirectional, 1 = look-ahead mask (j <= i)
 *   window  0 = none; W > 0 restricts keys to i-W+1 .. i with causal = 1, and to
 *           i-W+1 .. i+W-1 without it; W >= N excludes nothing
 *   scale   multiplier of q.k (callers pass 1/sqrt(d)); finite and > 0
 *   stream  cudaStream_t as void*
 *
 * o and lse must not overlap q, k or v. Returns ATTN_OK once the kernel is queued.
 */
int attn_fwd(const void *q, const void *k, const void *v, void *o, float *lse,
             int B, int Hq, int Hkv, int N, int d, int causal, int window, float scale,
             void *stream);

/*
 * attn_fwd_padded -- attn_fwd with per-batch padding.
 *
 *   key_len  device, int32 [B], 4-byte aligned (read): the first key_len[b] tokens of
 *            batch b are valid, the rest are padding (values are clamped to [0, N]).
 *            Padded keys are invisible to every query; padded query rows see no key
 *            and get o = 0, lse = -inf.
 * Every other argument is as for attn_fwd. Query tiles made only of padding load
 * nothing and write the zero output directly. ATTN_ERR_NULLPTR when key_len is NULL.
 */
int attn_fwd_padded(const void *q, const void *k, const void *v, void *o, float *lse,
                    const int *key_len, int B, int Hq, int Hkv, int N, int d, int causal,
                    int window, float scale, void *stream);

/*
 * attn_fwd_o32 -- attn_fwd (or, with key_len, attn_fwd_padded) writing O as fp32: the
 * same kernel and arithmetic, with the final O / (sum of rounded P) stored unrounded.
 * attn_fwd's bf16 O is exactly this value rounded to nearest even. It exists to measure
 * the kernel's own error apart from the bf16 output format: for |O| in [4, 8) half a
 * bf16 spacing (2^-6) already exceeds an absolute error bar of 1e-2.
 *
 *   o32      device, fp32 [B, Hq, N, d], 16-byte aligned (written)
 *   key_len  NULL, or as for attn_fwd_padded
 * Every other argument is as for attn_fwd. ATTN_ERR_NULLPTR when o32 is NULL.
 */
int attn_fwd_o32(const void *q, const void *k, const void *v, float *o32, float *lse,
                 const int *key_len, int B, int Hq, int Hkv, int N, int d, int causal,
                 int window, float scale, void *stream);

/*
 * attn_fwd_decode -- the decode shape: Nq query rows that are the LAST Nq positions of
 * a sequence of Nk >= Nq tokens whose keys and values are given (a key-value cache read
 * by the newest tokens: the generation stage in the SpAtten review's "Background"
 * section). Query row i stands at position i + Nk - Nq and the mask of attn_fwd applies
 * to that position. With Nq = Nk it computes what attn_fwd computes.
 *
 *   q    device, bf16 [B, Hq,  Nq, d], 16-byte aligned (read)
 *   k, v device, bf16 [B, Hkv, Nk, d], 16-byte aligned (read)
 *   o    device, bf16 [B, Hq,  Nq, d], 16-byte aligned (written)
 *   lse  device, fp32 [B, Hq,  Nq], 4-byte aligned (written; natural log)
 *   causal, window, scale   as for attn_fwd, on positions
 *   splits  number of parts the key sequence is divided into, each computed by its own
 *           CTA; 0 = the library's choice for the current device (see below); values
 *           above the number of 128-key tiles are reduced to it
 *   workspace, workspace_bytes  device scratch owned by the caller, 256-byte aligned,
 *           at least attn_fwd_decode_workspace_size(...) bytes; unused (may be NULL)
 *           when the split count is 1. It holds each split's fp32 partial O and LSE,
 *           which a second kernel merges by log-sum-exp into o and lse.
 *
 * The G = Hq / Hkv query heads that share a KV head are packed into one tile of
 * G * Nq <= 128 rows (ATTN_ERR_UNSUPPORTED otherwise), so every K/V tile is read once
 * per split for all of them. With G * Nq <= 32 rows and 16 or more key tiles per split,
 * both query tiles of a CTA work on one split, on alternate key tiles, and their results
 * are merged in the CTA.
 * ATTN_ERR_WORKSPACE when the workspace is too small.
 * Asynchronous on `stream`; calls that share a workspace must not overlap.
 */
size_t attn_fwd_decode_workspace_size(int B, int Hq, int Hkv, int Nq, int Nk, int d, int splits);
int attn_fwd_decode(const void *q, const void *k, const void *v, void *o, float *lse, int B, int Hq,
                    int Hkv, int Nq, int Nk, int d, int causal, int window, float scale, int splits,
                    void *workspace, size_t workspace_bytes, void *stream);

/*
 * attn_quantize_e4m3 -- FP8 block quantisation, as the FlashAttention-3 review's "Block
 * Quantization" describes it (deepmi.me): Q, K and V are split into blocks of B_r = 128
 * rows x d, each block gets its own scale from its largest magnitude, and the scaled
 * values are rounded to FP8 e4m3 (4-bit exponent, 3-bit mantissa; the variant with no
 * infinity, largest value 448).
 *
 *   x       device, bf16 [BH, N, d] (any leading shape flattened to BH heads), 16-byte
 *           aligned (read); d is 64 or 128
 *   codes   device, uint8 [BH, N, d], 8-byte aligned (written): e4m3(x * 448 / amax),
 *           round to nearest even, saturating at 448
 *   scales  device, fp32 [BH, ceil(N / 128)], 4-byte aligned (written): amax / 448 of
 *           each block (1 for an all-zero block); the value of a code is code x scale
 * The division 448 / amax and the products are IEEE fp32 operations. BH <= 65535.
 */
int attn_quantize_e4m3(const void *x, void *codes, float *scales, int BH, int N, int d, void *stream);

/*
 * attn_quantize_e4m3_hadamard -- incoherent processing then block quantisation, as the
 * FlashAttention-3 review's "Incoherent Processing" describes it for Q and K: each row x
 * is rotated by the random orthogonal matrix M = diag(s) H / sqrt(d), with s a random
 * +-1 per channel and H the Hadamard matrix (Sylvester construction, entry (i, j) =
 * (-1)^popcount(i & j)). The rotated values x M are then block quantised as by
 * attn_quantize_e4m3. Since M M^T = I, Q' K'^T = Q K^T: quantise Q and K with the same
 * signs, V with attn_quantize_e4m3, and call attn_fwd_fp8 with the usual scale.
 *
 *   x       device, bf16 [BH, N, d], 16-byte aligned (read); d = 128
 *   neg_lo, neg_hi  the signs: bit c of the 128-bit value (neg_hi:neg_lo) set means
 *           s_c = -1 (the caller draws them; the same signs for Q and K)
 *   codes   device, uint8 [BH, N, d], 16-byte aligned (written): e4m3(y * 448 / amax)
 *           with y = (x o s) H in fp32 and amax the block's largest |y|
 *   scales  device, fp32 [BH, ceil(N / 128)], 4-byte aligned (written):
 *           (amax / 448) / sqrt(128) (1 for an all-zero block); code x scale
 *           approximates the rotated value
 * y is formed in fp32 by the fast Walsh-Hadamard transform. Its rounding can move a
 * code that sits within a few fp32 ulps of a rounding boundary to the neighbouring
 * code. BH <= 65535. ATTN_ERR_UNSUPPORTED for d != 128.
 */
int attn_quantize_e4m3_hadamard(const void *x, uint64_t neg_lo, uint64_t neg_hi, void *codes,
                                float *scales, int BH, int N, int d, void *stream);

/*
 * attn_fwd_fp8 -- the attention forward of attn_fwd on e4m3 operands (the FP8 path of the
 * FlashAttention-3 review): Q, K, V given as codes and block scales from
 * attn_quantize_e4m3; the computed result is attention on the dequantised values.
 *
 *   q8       device, uint8 [B, Hq, N, d] e4m3 codes; k8, v8 [B, Hkv, N, d]; 16-byte aligned
 *   q_scale  device, fp32 [B * Hq, ceil(N / 128)]; k_scale, v_scale [B * Hkv, ceil(N / 128)]
 *   o, lse, B, Hq, Hkv, N, causal, window, scale, stream   as for attn_fwd
 *   d        128 (ATTN_ERR_UNSUPPORTED otherwise)
 *
 * S = q_scale x k_scale x (Q8 K8^T) exactly (fp32 accumulation); P is rounded to e4m3 for
 * the P.V product, with each V block's scale folded into P relative to the head's
 * largest V scale; O is normalised by the sum of the P values actually used, the LSE by
 * the unrounded sum.
 */
int attn_fwd_fp8(const void *q8, const void *k8, const void *v8, const float *q_scale,
                 const float *k_scale, const float *v_scale, void *o, float *lse, int B, int Hq,
                 int Hkv, int N, int d, int causal, int window, float scale, void *stream);

/*
 * attn_bwd -- gradients of attn_fwd's output with respect to Q, K and V. The FlashAttention-3
 * review (deepmi.me, "Results: Backward Pass" and "Computation and memory requirements")
 * names the backward pass and puts its cost at about 2.5 times the forward's; it gives no
 * formulas, so the gradients are those of the forward's definition by the chain rule,
 * with the forward's O and LSE taken as inputs:
 *
 *   P  = exp(scale S - lse)   the forward's softmax weights (0 where masked or padded)
 *   dP = dO V^T,  D_i = sum_c dO_ic O_ic,  dS = P o (dP - D)
 *   dQ = scale dS K,  dK = scale dS^T Q,  dV = P^T dO
 *
 * dK and dV of a key/value head sum over the Hq / Hkv query heads that read it.
 *
 *   q, k, v, B, Hq, Hkv, N, d, causal, window, scale, stream   as for attn_fwd (the same
 *            values the forward ran with)
 *   key_len  NULL, or the device int32 [B] valid lengths of attn_fwd_padded
 *   o, lse   device, the forward's outputs for these inputs (read): o bf16 [B, Hq, N, d],
 *            16-byte aligned; lse fp32 [B, Hq, N] (natural log, -inf on padded rows)
 *   dout     device, bf16 [B, Hq, N, d], 16-byte aligned (read): the gradient of o
 *   dq       device, bf16 [B, Hq, N, d], 16-byte aligned (written)
 *   dk, dv   device, bf16 [B, Hkv, N, d], 16-byte aligned (written); rows of keys that no
 *            query sees (padding) are written as zeros
 *   workspace  device, 256-byte aligned, at least attn_bwd_workspace_size(B, Hq, N, d)
 *            bytes, caller-owned (overwritten): lse log2(e), then D, of every query row,
 *            fp32 [B, Hq, ceil(N / 128) x 128] each (rows past N zero)
 *
 * Arithmetic: S and dP accumulate in fp32 on the tensor cores; P and dS are rounded to
 * bf16 as the operands of the dV, dK and dQ products, which accumulate in fp32 in a
 * fixed order (the result does not vary from run to run); the results are rounded to
 * bf16 once. Errors as for attn_fwd, and ATTN_ERR_WORKSPACE for a short workspace;
 * asynchronous on `stream`.
 */
size_t attn_bwd_workspace_size(int B, int Hq, int N, int d);
int attn_bwd(const void *q, const void *k, const void *v, const void *o, const float *lse,
             const void *dout, void *dq, void *dk, void *dv, const int *key_len, int B, int Hq,
             int Hkv, int N, int d, int causal, int window, float scale, void *workspace,
             size_t workspace_bytes, void *stream);

/*
 * attn_fwd_decode_noalloc -- attn_fwd_decode for callers that cannot allocate device
 * memory. The pages have no counterpart to this entry point; it exists for users of the
 * library.
 *
 * Who needs it: a caller whose device memory is fixed before it starts serving (a
 * serving loop that reserved its whole budget at start-up and may not grow it per
 * request), a caller running where the allocator must not be re-entered (for instance
 * from inside a memory-pool or allocator callback), or a plain C host that holds only
 * the tensors it passes and has no device allocator of its own. attn_fwd_decode needs
 * a workspace for the split results; this variant needs none.
 *
 * Arguments and results are those of attn_fwd_decode without the workspace: the split
 * results go to a fixed scratch array of ATTN_DECODE_NOALLOC_SCRATCH_BYTES (8 MiB) that
 * the library defines in device memory; every device holds it from the moment it loads
 * the library until the process exits. The split count (0 = the library's choice, the
 * same as attn_fwd_decode's) must leave splits x B x Hq x Nq x (d + 1) x 4 bytes (plus
 * alignment) within it, else ATTN_ERR_SCRATCH_LIMIT and nothing runs; with one split
 * the scratch is not touched.
 *
 * Nothing is allocated or freed: no cudaMalloc, cudaFree or allocating library call.
 * The first call on each device looks up the scratch array's device address
 * (cudaGetSymbolAddress, with that device current) and caches it; make that first call
 * before any stream capture. Every call on a device shares the one array and each split
 * overwrites all of its part before the merge reads it, so nothing needs clearing;
 * calls whose kernels overlap on the GPU (different streams, or different host threads)
 * race on it and must be serialised by the caller. The cached address stays valid for
 * the life of the device's primary context: after cudaDeviceReset on a device, this
 * entry point must not be called on that device again in the same process.
 */
#define ATTN_DECODE_NOALLOC_SCRATCH_BYTES (8u << 20)
int attn_fwd_decode_noalloc(const void *q, const void *k, const void *v, void *o, float *lse, int B,
                            int Hq, int Hkv, int Nq, int Nk, int d, int causal, int window, float scale,
                            int splits, void *stream);

/*
 * attn_fwd_host -- the same operation for callers whose tensors live in host memory.
 *
 * Copies q, k and v into the caller-owned device buffers dq, dk, dv, runs the forward
 * writing do_ and dlse, and copies do_ and dlse back into ho and hlse. Layouts, sizes
 * and alignment rules are those of attn_fwd, for both the host and the device buffers.
 *
 * The (batch, KV head) groups are independent, so the call is pipelined over up to 8
 * chunks of consecutive groups: host-to-device copies on a library-owned stream, the
 * kernel of each chunk on `stream`, device-to-host copies on a second library-owned
 * stream, ordered by events, so that the copies of one chunk overlap the kernel and the
 * copies of the others. The two streams and their events are created once per device,
 * on the first call there, and kept until the process exits; nothing is allocated per
 * call. Work queued on `stream` before the call is complete before the first copy, and
 * `stream` reaches the end of the call only after the last copy, so the results in ho
 * and hlse are valid once `stream` has been synchronised. Calls from several host
 * threads are safe; their copies share the library streams. Host buffers should be
 * page-locked (cudaHostAlloc / pinned) for the copies to be asynchronous; with pageable
 * memory CUDA stages them synchronously.
 */
int attn_fwd_host(const void *hq, const void *hk, const void *hv, void *ho, float *hlse,
                  void *dq, void *dk, void *dv, void *do_, float *dlse,
                  int B, int Hq, int Hkv, int N, int d, int causal, int window, float scale,
                  void *stream);

/* Human-readable name of an attn_status value (a static string; never NULL). */
const char *attn_status_str(int status);

/* cudaError_t of the most recent ATTN_ERR_CUDA returned on the calling host thread
 * (0 if none). */
int attn_last_cuda_error(void);

/*
 * attn_device_error -- synchronises the current device, then reports whether any
 * kernel of this library on it has given up a wait since the last clear: every
 * pipeline wait inside the kernels is bounded (2 s); a wait that runs out sets a
 * device-side status word, makes the kernel drain its own copies in flight, free
 * its tensor memory and return. Returns ATTN_OK, ATTN_ERR_TIMEOUT, ATTN_ERR_BOUNDS
 * (debug build: an index check failed; takes precedence), or ATTN_ERR_CUDA.
 * clear != 0 resets the word after reading it.
 */
int attn_device_error(int clear);

/*
 * The debug build (libattn_fwd_debug.so, compiled with ATTN_DEBUG defined) has the
 * same entry points and results. Its kernels check the indices that the scheduling
 * arithmetic produces before each access: shared-memory stages and buffers, tensor-
 * memory column ranges, tensor-map coordinates, global rows written and per-batch or
 * per-block values read. A failed check skips the access and records the failure
 * instead of faulting: attn_device_error then returns ATTN_ERR_BOUNDS. No page
 * describes this; it stands in for a memory checker, to run the test shapes under.
 *
 * attn_debug_build     1 in the debug build, 0 in the release build.
 * attn_debug_first_site  synchronises, returns the number of the first check that
 *                      failed since the last clear (0: none; always 0 in the release
 *                      build), or ATTN_ERR_CUDA; clear != 0 resets it.
 * attn_debug_selftest  debug build: queues one kernel whose only action is a failed
 *                      check at site 99 (nothing is accessed), to test the reporting;
 *                      ATTN_ERR_UNSUPPORTED in the release build.
 */
int attn_debug_build(void);
int attn_debug_first_site(int clear);
int attn_debug_selftest(void);

/*
 * attn_selftest_wait_timeout -- exercises the bounded-wait failure path without a
 * fault: launches one block that waits on a pipeline barrier that nothing will ever
 * complete, with a limit of limit_ns nanoseconds (1 .. 10^9), synchronises, and
 * returns what attn_device_error reports afterwards (expected: ATTN_ERR_TIMEOUT),
 * clearing the status word. ATTN_ERR_SHAPE for a limit outside the range.
 */
int attn_selftest_wait_timeout(int64_t limit_ns);

/* Library ABI version: major * 10000 + minor * 100 + patch. */
int attn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_API_H */

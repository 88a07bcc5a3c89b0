/*
 * ptq.h -- C ABI of the GB300 (sm_103a) PTQ1_0 ternary matmul library.
 *
 * PTQ1_0 ("A 27B model in 5.5 GB: Bonsai ternary on Ferrox, locally",
 * section "What Bonsai is"): every weight is -1, 0 or +1; five weights are
 * packed base-3 into one byte; each run of 128 weights along K (a "block")
 * has one 16-bit scale.  A block is 26 bytes of trits plus a 2-byte scale,
 * 1.75 bits per weight.  The stored weights have a 1024-wide signed
 * Walsh-Hadamard rotation folded in, so activations must be rotated the same
 * way before every matmul (same section; section "What Ferrox does with
 * it").
 *
 * Layouts (all row-major, all caller-owned):
 *   trits  int8   N x K, values in {-1, 0, +1}
 *   wq     uint8  N x (K/128) x 26: row n is (K/128)*26 bytes; inside a block
 *                 byte j holds weights 5j..5j+4 as base-3 digits (weight 5j
 *                 most significant, digit = trit + 1); byte 25 holds weights
 *                 125..127 and two pad digits equal to 1.
 *   scales uint16 N x (K/128) IEEE binary16 bit patterns (one per block);
 *                 subnormal scales are honoured exactly.
 *   signs  int8   K values, each +1 or -1; rotation block b uses
 *                 signs[1024 b .. 1024 b + 1023].
 *   x, y   activations: PTQ_F32 -> float, PTQ_BF16 -> bfloat16 bit patterns.
 *
 * Conventions:
 *   - Every call returns a ptq_status and never aborts.  A call refused by
 *     its argument checks (any status but PTQ_OK and PTQ_ERR_CUDA) has
 *     launched nothing.  PTQ_ERR_CUDA from a call that launches several
 *     kernels may follow launches already made.  ptq_last_error() returns a
 *     message for the calling thread's most recent failure.
 *   - Device pointers must be 16-byte aligned (signs: 4-byte aligned).
 *   - Device calls are asynchronous on `stream` (NULL = the legacy default
 *     stream); the library never synchronises inside a call and allocates no
 *     device memory.  Scratch memory, where a call needs it, is passed in.
 *   - Sizes are checked with overflow-safe arithmetic; unsupported
 *     combinations are refused by name (PTQ_ERR_UNSUPPORTED), never guessed.
 */
#ifndef PTQ_H
#define PTQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define PTQ_API __attribute__((visibility("default")))
#define PTQ_NODISCARD __attribute__((warn_unused_result))
#else
#define PTQ_API
#define PTQ_NODISCARD
#endif

/* Same type as cudaStream_t, declared without the CUDA headers. */
struct CUstream_st;
typedef struct CUstream_st* ptq_stream_t;

typedef enum ptq_status {
  PTQ_OK = 0,
  PTQ_ERR_NULL = 1,        /* a required pointer is NULL */
  PTQ_ERR_SHAPE = 2,       /* a size is negative, overflows, or breaks a
                              divisibility rule (K % 128, K % 1024) */
  PTQ_ERR_ALIGN = 3,       /* a pointer is not aligned as required */
  PTQ_ERR_VALUE = 4,       /* an input value is invalid (a trit not in
                              {-1,0,1}, an unknown dtype) */
  PTQ_ERR_UNSUPPORTED = 5, /* a valid but unsupported (M, dtype) combination */
  PTQ_ERR_WORKSPACE = 6,   /* workspace missing or too small */
  PTQ_ERR_CUDA = 7,        /* a CUDA runtime call or launch failed */
  PTQ_ERR_TIMEOUT = 8,     /* a bounded device-side wait ran out */
  PTQ_ERR_RANGE = 9        /* reported by ptq_device_check: a value the bf16
                              route keeps in fp16 (the rotated operands of
                              ptq_rotate_matmul, ptq_ffn, ptq_ffn_stack and
                              ptq_ffn_noalloc) exceeded the fp16 range
                              (|v| >= 65520) and was stored as infinity */
} ptq_status;

typedef enum ptq_dtype { PTQ_F32 = 0, PTQ_BF16 = 1 } ptq_dtype;

/* ptq1_pack -- host-side PTQ1_0 encoder (used to build test weights).
 * Encodes N x K trits into wq (host memory, (K/128)*26 bytes per row) with
 * digit = trit + 1, v = sum_i d_i 3^(4-i), byte = ceil(256 v / 243).  The
 * decode it must invert is the peel of "What Ferrox does with it": digit n
 * of byte is floor(3^(n+1) u) - 3 floor(3^n u), u = byte / 256.
 * Errors: PTQ_ERR_NULL, PTQ_ERR_SHAPE (N < 0, K <= 0, K % 128 != 0, size
 * overflow), PTQ_ERR_VALUE (a trit outside {-1,0,1}; wq is then untouched).
 * Synchronous; touches no GPU. */
PTQ_API PTQ_NODISCARD ptq_status ptq1_pack(const int8_t* trits, uint8_t* wq,
                                           int64_t N, int64_t K);

/* ptq1_unpack -- device-side decode of PTQ1_0 bytes into N x K int8 trits,
 * with the fp32 peel of "What Ferrox does with it".  Bit-exact; exists so
 * the codec of the matmul kernels can be tested on its own.
 * wq and trits are device pointers. */
PTQ_API PTQ_NODISCARD ptq_status ptq1_unpack(const uint8_t* wq, int8_t* trits,
                                             int64_t N, int64_t K,
                                             ptq_stream_t stream);

/* ptq_fwht -- signed Walsh-Hadamard rotation of activations
 * ("What Bonsai is": a 1024-wide butterfly with a sign pattern).  For every
 * row m and every 1024-block b:
 *     y[m, 1024b + j] = (1/32) sum_i (-1)^popcount(i & j) s[1024b + i] x[m, 1024b + i]
 * i.e. flip signs, apply the Sylvester-ordered Hadamard matrix, scale by
 * 1/32 (which makes the rotation orthogonal).  x, y: M x K of `dtype`
 * (device); y may equal x (in place); signs: K int8 (device).  Arithmetic is
 * fp32; a bf16 output is rounded to nearest-even once, at the end.
 * Errors: PTQ_ERR_NULL, PTQ_ERR_SHAPE (K % 1024 != 0), PTQ_ERR_ALIGN,
 * PTQ_ERR_VALUE (dtype), PTQ_ERR_CUDA. */
PTQ_API PTQ_NODISCARD ptq_status ptq_fwht(const void* x, void* y,
                                          const int8_t* signs, int64_t M,
                                          int64_t K, ptq_dtype dtype,
                                          ptq_stream_t stream);

/* ptq_matmul_workspace_bytes -- scratch size ptq_matmul needs for
 * (M, N, K, dtype); 0 when it needs none or the arguments are invalid.
 * fp32 decode (M <= 8, K/128 even): one fp32 partial row sum per (token,
 * K-chunk of at most 640 weights, output row); required.
 * bf16 GEMM: fp32 partial sums for shapes with too few output tiles to fill
 * the GPU, whose K is then split in up to 6 parts; optional (with less, the
 * product runs with fewer splits). */
PTQ_API size_t ptq_matmul_workspace_bytes(int64_t M, int64_t N, int64_t K,
                                          ptq_dtype dtype);

/* ptq_matmul -- y = x W^T for a PTQ1_0 weight W (N x K):
 *     y[m, n] = sum_b scale[n, b] * sum_{i<128} trit[n, 128b + i] * x[m, 128b + i]
 * x is M x K and must already be rotated (ptq_fwht) when W carries the fold.
 * Routing (one table, queryable with ptq_route):
 *   PTQ_F32,  1 <= M <= 8 : decode GEMV by per-position lookup tables of the
 *                           five-trit sums, the tokens one after the other in
 *                           one launch, fp32 throughout (K/128 odd: a GEMV
 *                           with the fp32 peel)
 *   PTQ_BF16, M >= 1      : prefill GEMM, bf16 in / fp32 accumulate / bf16 out
 *   PTQ_F32,  M > 8       : refused with PTQ_ERR_UNSUPPORTED
 * M == 0 or N == 0 is a no-op.  Requires K % 128 == 0 (fastest at
 * K % 1024 == 0).  All pointers are device pointers.
 * workspace: device scratch of ptq_matmul_workspace_bytes(...) bytes, 16-byte
 * aligned, caller-owned, any initial contents, unspecified contents on
 * return; may be NULL when that size is 0 or the route is the bf16 GEMM.  Calls whose kernels overlap
 * on the GPU need separate workspaces.  Results are bitwise reproducible:
 * the same inputs give the same bits on every run.
 * Errors: PTQ_ERR_NULL, PTQ_ERR_SHAPE, PTQ_ERR_ALIGN, PTQ_ERR_VALUE (dtype),
 * PTQ_ERR_UNSUPPORTED, PTQ_ERR_WORKSPACE, PTQ_ERR_CUDA. */
PTQ_API PTQ_NODISCARD ptq_status ptq_matmul(const uint8_t* wq,
                                            const uint16_t* scales,
                                            const void* x, void* y, int64_t M,
                                            int64_t N, int64_t K,
                                            ptq_dtype dtype, void* workspace,
                                            size_t workspace_bytes,
                                            ptq_stream_t stream);

/* ptq_rotate_matmul_workspace_bytes -- scratch size of ptq_rotate_matmul;
 * 0 when the arguments are invalid. */
PTQ_API size_t ptq_rotate_matmul_workspace_bytes(int64_t M, int64_t N,
                                                 int64_t K, ptq_dtype dtype);

/* ptq_rotate_matmul -- y = (R x) W^T: the signed rotation of ptq_fwht applied
 * to x (un-rotated, not modified), then ptq_matmul.  This is the order the
 * pages prescribe for a folded weight ("What Ferrox does with it": rotate
 * the activation before every matmul).  On the fp32 decode route (M <= 8) the
 * rotation runs inside the GEMV, on the activations each thread block reads;
 * otherwise it is a separate kernel writing R x into the workspace.
 * signs: K int8 (device, 4-byte aligned).  Requires K % 1024 == 0.
 * workspace: at least ptq_rotate_matmul_workspace_bytes(...) bytes, 16-byte
 * aligned, any initial contents.  Other arguments, routing and errors as
 * ptq_matmul.
 * fp16 operand range (PTQ_BF16): the rotated activation R x is held in
 * fp16 between the rotation and the tensor-core GEMM (11 significant bits,
 * so the block scale times a trit is exact), so |R x| must stay below 65520.
 * Beyond that the value is stored as infinity and the output is not finite;
 * the rotation then raises the device status word and the next
 * ptq_device_check returns PTQ_ERR_RANGE.  The fp32 route has no such
 * limit. */
PTQ_API PTQ_NODISCARD ptq_status ptq_rotate_matmul(
    const uint8_t* wq, const uint16_t* scales, const void* x,
    const int8_t* signs, void* y, int64_t M, int64_t N, int64_t K,
    ptq_dtype dtype, void* workspace, size_t workspace_bytes,
    ptq_stream_t stream);

/* ptq_rotate_matmul_host_workspace_bytes -- device scratch of
 * ptq_rotate_matmul_host: room for x and y, then ptq_rotate_matmul's own
 * workspace (each rounded up to 256 bytes); 0 when the arguments are
 * invalid. */
PTQ_API size_t ptq_rotate_matmul_host_workspace_bytes(int64_t M, int64_t N,
                                                      int64_t K, ptq_dtype dtype);

/* ptq_rotate_matmul_host -- ptq_rotate_matmul on host buffers, for callers
 * whose activations live on the host: copies x_host (M x K, host) into the
 * workspace, runs ptq_rotate_matmul there, and copies y (M x N) back to
 * y_host, all queued on `stream` (one cudaMemcpyAsync each way).  The call
 * returns once the work is queued: y_host is valid after the stream is
 * synchronised, and x_host must stay unchanged until then.  Page-locked host
 * memory gives asynchronous copies; other host memory works but the copies
 * then synchronise.  When the runtime maps both host buffers into the
 * device's address space (page-locked memory on a system with unified
 * addressing), the kernels read x and write y there directly instead, with
 * no copies.  wq, scales and signs are device pointers as in
 * ptq_rotate_matmul.  workspace: at least
 * ptq_rotate_matmul_host_workspace_bytes(...) bytes, 256-byte aligned.
 * Errors as ptq_rotate_matmul, plus PTQ_ERR_NULL for a NULL host buffer and
 * PTQ_ERR_CUDA if a copy cannot be queued. */
PTQ_API PTQ_NODISCARD ptq_status ptq_rotate_matmul_host(
    const uint8_t* wq, const uint16_t* scales, const void* x_host,
    const int8_t* signs, void* y_host, int64_t M, int64_t N, int64_t K,
    ptq_dtype dtype, void* workspace, size_t workspace_bytes,
    ptq_stream_t stream);

/* ptq_ffn_workspace_bytes -- scratch size ptq_ffn needs for (M, H, I, dtype);
 * 0 when the arguments are invalid. */
PTQ_API size_t ptq_ffn_workspace_bytes(int64_t M, int64_t H, int64_t I,
                                       ptq_dtype dtype);

/* ptq_ffn -- the feed-forward block of "Speed, and where it goes":
 *     xr = R_in x;  [g; u] = W_gu xr;  h = silu(g) * u;  hr = R_mid h;  y = W_d hr
 * with silu(a) = a / (1 + e^-a), R_* the signed rotations of ptq_fwht.
 * wgu_q/wgu_s: the fused gate+up weight, 2I x H, gate rows 0..I-1 then up
 * rows I..2I-1.  wd_q/wd_s: the down weight, H x I.  signs_in: H values,
 * signs_mid: I values.  x, y: M x H (x is not modified).  Requires
 * H % 1024 == 0 and I % 1024 == 0; dtype routing as in ptq_matmul.
 * workspace: device scratch of at least ptq_ffn_workspace_bytes(...) bytes,
 * 16-byte aligned, owned by the caller; its contents on return are
 * unspecified.  Errors as ptq_matmul, plus PTQ_ERR_WORKSPACE.
 * fp16 operand range (PTQ_BF16): the rotated operands xr = R_in x and
 * hr = R_mid h are held in fp16 (the block scale times a trit is exact in
 * fp16); gate/up and h stay fp32 and y is bf16.  |xr| and |hr| must stay
 * below 65520: beyond it the value is stored as infinity, y is not finite,
 * and the next ptq_device_check returns PTQ_ERR_RANGE.  The fp32 route has
 * no such limit. */
PTQ_API PTQ_NODISCARD ptq_status ptq_ffn(
    const uint8_t* wgu_q, const uint16_t* wgu_s, const uint8_t* wd_q,
    const uint16_t* wd_s, const int8_t* signs_in, const int8_t* signs_mid,
    const void* x, void* y, int64_t M, int64_t H, int64_t I, ptq_dtype dtype,
    void* workspace, size_t workspace_bytes, ptq_stream_t stream);

/* ---- the chained feed-forward stack ("A 27B model in 5.5 GB: Bonsai ternary
 * on Ferrox, locally", section "Speed, and where it goes", which names running
 * the whole layer on the device, norms and residual adds included, as the
 * next step).  The page gives no formula; this library reads it as the usual
 * pre-norm residual stack, for l = 0 .. L-1:
 *     xn = x / sqrt(mean_k x_k^2 + eps) * g_l;   x = x + FFN_l(xn)
 * with FFN_l the block of ptq_ffn and g_l a per-layer gain vector. */

/* One layer of the stack: ptq_ffn's weights and signs (same shapes and
 * formats) and the RMSNorm gains, H fp32 values, 16-byte aligned.  All
 * pointers are device pointers owned by the caller. */
typedef struct ptq_ffn_layer {
  const uint8_t* wgu_q;
  const uint16_t* wgu_s;
  const uint8_t* wd_q;
  const uint16_t* wd_s;
  const int8_t* signs_in;
  const int8_t* signs_mid;
  const float* norm_w;
} ptq_ffn_layer;

/* ptq_ffn_stack_workspace_bytes -- scratch ptq_ffn_stack needs; 0 when the
 * arguments are invalid. */
PTQ_API size_t ptq_ffn_stack_workspace_bytes(int64_t M, int64_t H, int64_t I,
                                             ptq_dtype dtype);

/* ptq_ffn_stack -- L chained pre-norm feed-forward blocks over the residual
 * stream x (M x H fp32, device, 16-byte aligned, updated in place).
 * layers: a HOST array of L entries, read during the call only.  eps: the
 * RMSNorm's epsilon, finite and >= 0.  dtype selects the blocks' routing and
 * activation type as in ptq_ffn: PTQ_F32 (M <= 8) keeps xn and the block
 * output in fp32; PTQ_BF16 stores them in bf16 (the residual stream stays
 * fp32 either way).  ptq_ffn_stack_route names the implementation: one
 * persistent launch per 24 layers for 1 to 8 fp32 tokens, else per layer an
 * add-and-norm kernel and the block's kernels, and a final add.  The
 * persistent path adds the row sums of its projections with atomics, so its
 * results may differ between runs by fp32 rounding; the per-layer path is
 * bitwise reproducible.  When the device cannot hold the persistent grid
 * (its SMs partly held elsewhere) the call takes the per-layer path.
 * workspace: device scratch of ptq_ffn_stack_workspace_bytes(...) bytes,
 * 16-byte aligned, caller-owned, contents unspecified on return.  Every
 * layer is validated before the first launch, so a refused call leaves x
 * unchanged.  L == 0 or M == 0 is a no-op.  Errors as ptq_ffn (the message
 * names the layer), plus PTQ_ERR_VALUE for a bad eps.  On PTQ_BF16 each
 * block has ptq_ffn's fp16 operand range (PTQ_ERR_RANGE from
 * ptq_device_check when it is exceeded). */
PTQ_API PTQ_NODISCARD ptq_status ptq_ffn_stack(
    const ptq_ffn_layer* layers, int64_t L, float* x, int64_t M, int64_t H,
    int64_t I, float eps, ptq_dtype dtype, void* workspace,
    size_t workspace_bytes, ptq_stream_t stream);

/* ptq_ffn_stack_ex -- ptq_ffn_stack with flags.  PTQ_STACK_DETERMINISTIC
 * takes the per-layer path for every M and dtype, whose results are bitwise
 * reproducible.  Other bits are refused with PTQ_ERR_VALUE.
 * ptq_ffn_stack(...) is ptq_ffn_stack_ex(..., 0, stream). */
#define PTQ_STACK_DETERMINISTIC 1u
PTQ_API PTQ_NODISCARD ptq_status ptq_ffn_stack_ex(
    const ptq_ffn_layer* layers, int64_t L, float* x, int64_t M, int64_t H,
    int64_t I, float eps, ptq_dtype dtype, void* workspace,
    size_t workspace_bytes, unsigned flags, ptq_stream_t stream);

/* ptq_ffn_stack_route -- which implementation ptq_ffn_stack (no flags) uses
 * for (M, H, I, dtype) on the current device: "stack_decode_persistent"
 * (M = 1 to 8, PTQ_F32: the whole stack in one cooperative launch per 24
 * layers, the tokens taken in turn inside each phase, one CTA per SM, the
 * layers separated by grid-wide barriers whose waits are bounded -- a wait
 * that runs out raises the status ptq_device_check reports) or
 * "stack_per_layer" (an add-and-norm kernel, then ptq_ffn's kernels, per
 * layer).  *name points to a static string.  Errors:
 * PTQ_ERR_NULL, PTQ_ERR_VALUE (dtype), PTQ_ERR_SHAPE, PTQ_ERR_UNSUPPORTED
 * (no kernel for M and dtype). */
PTQ_API PTQ_NODISCARD ptq_status ptq_ffn_stack_route(int64_t M, int64_t H,
                                                     int64_t I, ptq_dtype dtype,
                                                     const char** name);

/* ptq_ffn_noalloc -- ptq_ffn without a workspace argument; it allocates
 * nothing.  (The source pages have no counterpart: this exists for callers,
 * not for the method.)
 * Some callers cannot allocate device memory: real-time decode loops that
 * may not take the synchronisation and latency of cudaMalloc, plug-ins that
 * are handed a stream but no allocator, and hosts whose device memory is
 * held by another allocator that a C caller cannot reach.  This entry point
 * takes the block's scratch from one file-scope device array of
 * PTQ_FFN_NOALLOC_SCRATCH_BYTES bytes that every device loading the library
 * holds until the process exits; inputs and output are still the caller's.
 * Arguments, layouts, errors and the bf16 route's fp16 operand range are
 * those of ptq_ffn; a shape whose scratch
 * (ptq_ffn_workspace_bytes) exceeds the array is refused with
 * PTQ_ERR_WORKSPACE.  At the default shapes (H = 5120, I = 17408) that admits
 * the fp32 decode path up to M = 2 (1.48 MB of scratch a token, most of it
 * the decode GEMV's per-chunk row sums) and the bf16 path up to M = 16.
 * The first call on a device looks the array's device address up
 * (cudaGetSymbolAddress) and caches it; make that first call before any
 * stream capture.  All calls share the one array and it keeps the last
 * call's contents (none of which has to start at zero): calls whose kernels
 * overlap on the GPU race on it, so order them on one stream. */
#define PTQ_FFN_NOALLOC_SCRATCH_BYTES (4 * 1024 * 1024)
PTQ_API PTQ_NODISCARD ptq_status ptq_ffn_noalloc(
    const uint8_t* wgu_q, const uint16_t* wgu_s, const uint8_t* wd_q,
    const uint16_t* wd_s, const int8_t* signs_in, const int8_t* signs_mid,
    const void* x, void* y, int64_t M, int64_t H, int64_t I, ptq_dtype dtype,
    ptq_stream_t stream);

/* ---- PQ2_0 ("Why I Am Building Another Inference Engine", section
 * "Level 2: The short answer"): each ternary weight in 2 bits plus one
 * 16-bit scale per 128 weights, 2.125 bits per weight.  The page fixes only
 * that much; this library reads it as:
 *   wq     uint8  N x (K/128) x 32: weight 4j + i of a block is bits 2i and
 *                 2i + 1 of its byte j, code = trit + 1; the decode is
 *                 trit = code - 1 for all four codes (no encoder writes 3,
 *                 which therefore decodes to +2);
 *   scales uint16 N x (K/128) binary16 patterns, as for PTQ1_0.
 * The rotation, x and y are as for PTQ1_0. */

/* ptq2_pack -- host-side PQ2_0 encoder.  Errors as ptq1_pack. */
PTQ_API PTQ_NODISCARD ptq_status ptq2_pack(const int8_t* trits, uint8_t* wq,
                                           int64_t N, int64_t K);

/* ptq2_unpack -- device decode of PQ2_0 codes into N x K int8 trits
 * (bit-exact test export).  trits 4-byte aligned.  Errors as ptq1_unpack,
 * plus PTQ_ERR_ALIGN. */
PTQ_API PTQ_NODISCARD ptq_status ptq2_unpack(const uint8_t* wq, int8_t* trits,
                                             int64_t N, int64_t K,
                                             ptq_stream_t stream);

/* ptq_matmul_pq2_workspace_bytes -- scratch ptq_matmul_pq2 needs (or, for
 * the bf16 GEMM, can use for K splits); 0 for invalid arguments or none. */
PTQ_API size_t ptq_matmul_pq2_workspace_bytes(int64_t M, int64_t N,
                                              int64_t K, ptq_dtype dtype);

/* ptq_matmul_pq2 -- ptq_matmul over PQ2_0 weights: the same definition
 * (y = x W^T with W = trit x block scale), dtype routing and workspace rules.
 * Both routes use the TMA-fed kernels, so K % 1024 == 0 is required
 * (otherwise PTQ_ERR_UNSUPPORTED); every other error as ptq_matmul. */
PTQ_API PTQ_NODISCARD ptq_status ptq_matmul_pq2(
    const uint8_t* wq, const uint16_t* scales, const void* x, void* y,
    int64_t M, int64_t N, int64_t K, ptq_dtype dtype, void* workspace,
    size_t workspace_bytes, ptq_stream_t stream);

/* ptq_embed -- token-embedding lookup on a rotated table.
 * "What Bonsai is": the rotation folded into the weights is undone on the
 * embedding table after each lookup.  Row v of the table holds R e_v, with R
 * the signed rotation of ptq_fwht; this call gathers the rows ids[0..M-1] and
 * returns out[m] = R^T table[ids[m]] = D_s H table[ids[m]] / 32 per
 * 1024-block (the butterfly first, then the signs: R is orthonormal).
 *   table  V x H, dtype (PTQ_F32 float, PTQ_BF16 bfloat16), row-major
 *   ids    M int32 token ids (device)
 *   signs  H values, +1 or -1 (those of the rotation folded into the table)
 *   out    M x H, dtype; must not overlap the table
 * Arithmetic is fp32; a bf16 output is rounded to nearest-even once.  An id
 * outside [0, V) gives a row of quiet NaN (nothing is read for it): the
 * ids are on the device, so the call cannot refuse them.
 * Requires H % 1024 == 0, V >= 1; table and out 16-byte aligned, ids and
 * signs 4-byte aligned.  M = 0 is a no-op.
 * Errors: PTQ_ERR_NULL, PTQ_ERR_SHAPE, PTQ_ERR_ALIGN, PTQ_ERR_VALUE (dtype),
 * PTQ_ERR_CUDA. */
PTQ_API PTQ_NODISCARD ptq_status ptq_embed(const void* table,
                                           const int32_t* ids,
                                           const int8_t* signs, void* out,
                                           int64_t M, int64_t V, int64_t H,
                                           ptq_dtype dtype,
                                           ptq_stream_t stream);

/* ptq_embed_ptq1 -- ptq_embed for a PTQ1_0 table: wq V x (H/128) x 26
 * bytes and scales V x (H/128) binary16 patterns (the layouts above); row v
 * is trit x block scale, decoded exactly in fp32.  out (M x H) is
 * out_dtype.  wq and scales 16-byte aligned; everything else as ptq_embed. */
PTQ_API PTQ_NODISCARD ptq_status ptq_embed_ptq1(
    const uint8_t* wq, const uint16_t* scales, const int32_t* ids,
    const int8_t* signs, void* out, int64_t M, int64_t V, int64_t H,
    ptq_dtype out_dtype, ptq_stream_t stream);

/* ptq_route -- the kernel ptq_matmul would run for (M, dtype) when K/128 is
 * even: writes its name to *kernel_name (static storage) and returns PTQ_OK,
 * or returns PTQ_ERR_UNSUPPORTED / PTQ_ERR_VALUE.  Host only. */
PTQ_API PTQ_NODISCARD ptq_status ptq_route(int64_t M, ptq_dtype dtype,
                                           const char** kernel_name);

/* ptq_device_check -- synchronises `stream`, then reads and clears the
 * library's device status word.  Returns PTQ_ERR_TIMEOUT if a bounded
 * device-side wait in an earlier kernel ran out (that kernel's outputs are
 * then invalid), else PTQ_ERR_RANGE if a bf16-route call stored an operand
 * beyond the fp16 range as infinity (its outputs are then not finite),
 * PTQ_ERR_CUDA if the stream reports an error, else PTQ_OK. */
PTQ_API PTQ_NODISCARD ptq_status ptq_device_check(ptq_stream_t stream);

/* ptq_matmul_bf16_accumulator -- test export: ptq_matmul's bf16 route (the
 * prefill GEMM: same kernel, expanded t * bf16(s) weight tiles and split-K
 * choice) writing the fp32 accumulator y (M x N fp32, device, 16-byte
 * aligned) instead of rounding it to bf16.  It lets tests hold the route's
 * arithmetic to the bare 1e-2 rms(y) bound of the workload text, which the
 * bf16 output's own rounding (up to 2^-8 |y|) would otherwise hide.
 * workspace: as ptq_matmul with PTQ_BF16 (may be NULL: fewer K splits).
 * Errors as ptq_matmul. */
PTQ_API PTQ_NODISCARD ptq_status ptq_matmul_bf16_accumulator(
    const uint8_t* wq, const uint16_t* scales, const void* x, float* y,
    int64_t M, int64_t N, int64_t K, void* workspace, size_t workspace_bytes,
    ptq_stream_t stream);

/* ptq_matmul_f32_peel -- test export: ptq_matmul's fp32 route (1 <= M <= 8)
 * computed by its other kernel, the SIMT GEMV that peels the trits on the
 * float pipe with 16-byte loads (the route's kernel when K/128 is odd), on
 * any shape.  It lets the peel design of "What Ferrox does with it" be timed
 * against the table-lookup kernel on the same weights.  No workspace.
 * x must already be rotated.  Arguments and errors as ptq_matmul with
 * PTQ_F32. */
PTQ_API PTQ_NODISCARD ptq_status ptq_matmul_f32_peel(
    const uint8_t* wq, const uint16_t* scales, const float* x, float* y,
    int64_t M, int64_t N, int64_t K, ptq_stream_t stream);

/* ptq_gemv_plan -- introspection: the launch ptq_matmul's fp32 decode route
 * (pq2 != 0: ptq_matmul_pq2's) makes for (M, N, K) on the current device,
 * K % 1024 == 0, plain output (ptq_ffn's gate/up projection always adds the
 * reduction kernel).  plan (host, 4 int32): CTAs, thread-block cluster size
 * (0: no clusters), K-chunks a row is cut into, kernels launched.  At one
 * token, when the device holds enough clusters of one CTA per K-chunk, the
 * chunks of a row group form a cluster that adds its row sums in distributed
 * shared memory and writes y (one kernel); otherwise a second kernel adds the
 * chunk sums from the workspace.  Both give the same bits.  Host only (it
 * asks the current device).  Errors: PTQ_ERR_NULL, PTQ_ERR_UNSUPPORTED,
 * PTQ_ERR_CUDA. */
PTQ_API PTQ_NODISCARD ptq_status ptq_gemv_plan(int64_t M, int64_t N, int64_t K,
                                               int pq2, int32_t plan[4]);

/* ptq_selftest_timeout -- test export for the timeout path.  Launches one
 * CTA that waits, with the library's bounded mbarrier wait and a short poll
 * limit, on a barrier that nothing arrives on; the wait runs out and the
 * kernel raises the device status word and returns (no fault, no hang).  The
 * next ptq_device_check on the stream then returns PTQ_ERR_TIMEOUT and
 * clears the word.  Errors: PTQ_ERR_CUDA. */
PTQ_API PTQ_NODISCARD ptq_status ptq_selftest_timeout(ptq_stream_t stream);

/* ptq_selftest_grid_timeout -- test export for the grid barrier of the
 * persistent stack (ptq_ffn_stack_route "stack_decode_persistent").
 * Launches 8 CTAs of which one never arrives at the barrier; the other
 * seven poll, with the stack's bounded wait and a short poll limit, run
 * out, raise the device status word and return (no fault, no hang).  The
 * next ptq_device_check then returns PTQ_ERR_TIMEOUT.  Errors:
 * PTQ_ERR_CUDA. */
PTQ_API PTQ_NODISCARD ptq_status ptq_selftest_grid_timeout(ptq_stream_t stream);

/* ptq_status_str -- static name of a status code. */
PTQ_API const char* ptq_status_str(ptq_status status);

/* ptq_last_error -- message describing the calling thread's last failure
 * ("" if none).  Valid until the thread's next library call. */
PTQ_API const char* ptq_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* PTQ_H */

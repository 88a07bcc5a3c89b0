// ptq_internal.cuh -- declarations shared by the translation units of the
// CUDA library (launchers, geometry constants, the device status word).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/ptq.h"

namespace ptq {

// PTQ1_0 geometry ("What Bonsai is": 128 weights per 16-bit scale, five
// trits per byte).
constexpr int kBlockWeights = 128;
constexpr int kBlockBytes = 26;   // ceil(128 / 5)
constexpr int kRot = 1024;        // rotation width
constexpr int kGroupBlocks = kRot / kBlockWeights;     // 8 blocks per 1024
constexpr int kGroupBytes = kGroupBlocks * kBlockBytes;  // 208 = 13 * 16

// Activation storage types used inside the library.  F16 never crosses the
// C ABI: the feed-forward block keeps its rotated tensor-core operands in
// fp16 (11 significant bits; the block scale times a trit is exact in fp16).
enum class Act { F32, BF16, F16 };
inline Act act_of(ptq_dtype d) { return d == PTQ_BF16 ? Act::BF16 : Act::F32; }

// Device status word: bounded waits that run out OR in kDevTimeout; a
// finite value that overflows the fp16 range where the bf16 route stores its
// rotated tensor-core operands (|v| >= 65520 rounds to infinity) ORs in
// kDevRange.
constexpr int kDevTimeout = 1;
constexpr int kDevRange = 2;

// Launch with programmatic dependent launch allowed: the kernel may start
// while the previous kernel in the stream is still running, and must run
// `griddepcontrol.wait` before it touches anything that kernel writes.  Used
// for kernels whose prologue (weight prefetch) does not depend on it.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t st, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_release() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Records a failure message for ptq_last_error() and returns `s`.
ptq_status fail(ptq_status s, const char* fmt, ...);
// Maps a CUDA error to PTQ_ERR_CUDA with a message naming `what`.
ptq_status cuda_fail(cudaError_t e, const char* what);

// ---- launchers (arguments already validated) -------------------------------
cudaError_t launch_unpack(const uint8_t* wq, int8_t* trits, int64_t N,
                          int64_t K, cudaStream_t st);
cudaError_t launch_unpack_pq2(const uint8_t* wq, int8_t* trits, int64_t N, int64_t K,
                              cudaStream_t st);
// Supported (in, out): (F32, F32), (BF16, BF16), (BF16, F16), (F32, F16).
// An F16 output raises kDevRange in the device status word when a finite
// rotated value lies beyond the fp16 range (it is stored as infinity).
cudaError_t launch_fwht(const void* x, Act in, void* y, Act out,
                        const int8_t* signs, int64_t M, int64_t K, cudaStream_t st);
cudaError_t launch_gemv(const uint8_t* wq, const uint16_t* scales,
                        const float* x, float* y, int64_t M, int64_t N,
                        int64_t K, cudaStream_t st);
// Embedding lookup on a rotated table (k_embed.cu): out[m] = R^T table[ids[m]].
// Dense tables: (F32, F32) or (BF16, BF16).  PTQ1_0 tables: out F32 or BF16.
cudaError_t launch_embed(const void* table, Act table_t, const int32_t* ids, const int8_t* signs,
                         void* out, Act out_t, int64_t M, int64_t V, int64_t H, cudaStream_t st);
cudaError_t launch_embed_ptq1(const uint8_t* wq, const uint16_t* scales, const int32_t* ids,
                              const int8_t* signs, void* out, Act out_t, int64_t M, int64_t V,
                              int64_t H, cudaStream_t st);
// Decode by lookup tables (k_gemv_lut.cu) of M tokens: x is M x K, y M x N.
// part: scratch of gemv_lut_workspace_bytes(N, K, M) bytes (the row sums of
// every K-chunk of every token).  cudaErrorNotSupported when the shape does
// not fit it (K/128 odd, more K-chunks than SMs); the caller then runs
// launch_gemv.
// signs != NULL: x is not rotated yet and the kernel rotates it (K % 1024).
// SwiGLU (M = 1 only): the weight is the fused gate+up (N = 2I) and y
// receives h (I).
enum class LutEpilogue { Plain, SwiGLU };
cudaError_t launch_gemv_lut(const uint8_t* wq, const uint16_t* scales, const float* x,
                            const int8_t* signs, float* y, float* part, int64_t M, int64_t N,
                            int64_t K, LutEpilogue ep, cudaStream_t st);
size_t gemv_lut_workspace_bytes(int64_t N, int64_t K, int64_t M);
// K-chunks of a row (0 when the table-lookup GEMV does not serve K), and the
// CTAs that share one chunk's rows on a device of `sms` SMs.
int64_t gemv_lut_chunks(int64_t K);
int64_t gemv_lut_ctas_per_chunk(int64_t sms, int64_t nch, int64_t N);
// The same decode for PQ2_0 weights (k_gemv_lut.cu): K % 1024 == 0 only.
cudaError_t launch_gemv_lut_pq2(const uint8_t* wq, const uint16_t* scales, const float* x,
                                const int8_t* signs, float* y, float* part, int64_t M, int64_t N,
                                int64_t K, cudaStream_t st);
int64_t gemv_lut_pq2_chunks(int64_t K);
size_t gemv_lut_pq2_workspace_bytes(int64_t N, int64_t K, int64_t M);
// The launch launch_gemv_lut (pq2: launch_gemv_lut_pq2) makes for M tokens,
// plain epilogue, on the current device: CTAs, cluster size (0: none), K
// chunks and kernels (the GEMV and, unless its clusters write y or a row has
// one chunk, the chunk reduction).  cudaErrorNotSupported when the TMA-fed
// kernel does not serve the shape.
struct LutPlan {
  int ctas, cluster, chunks, kernels;
};
cudaError_t gemv_lut_plan(int64_t M, int64_t N, int64_t K, bool pq2, LutPlan* plan);
// Whether launch_gemv_lut serves (N, K) on the current device (with the
// rotation when `rotate`).
bool gemv_lut_supported(int64_t N, int64_t K, bool rotate);
// x is BF16 or F16; y is BF16 or F32.  ws: split-K scratch (may be NULL;
// then, or when it is smaller than gemm_tc_workspace_bytes, fewer splits).
cudaError_t launch_gemm(const uint8_t* wq, const uint16_t* scales, const void* x, Act x_t,
                        void* y, Act y_t, int64_t M, int64_t N, int64_t K, void* ws,
                        size_t ws_bytes, cudaStream_t st);
// gu: M x 2I fp32 (gate half first) -> h: M x I fp32.
cudaError_t launch_swiglu(const float* gu, float* h, int64_t M, int64_t I,
                          cudaStream_t st);

// Decode tokens (fp32) the persistent stack serves at once.
constexpr int kStackMaxTokens = 8;

// The chained feed-forward stack for M = 1..8 fp32 decode tokens, as one
// persistent launch per 24 layers (k_stack_decode.cu).  x: M x H fp32,
// updated in place.  gu0, gu1: M x 2I fp32 scratch each; ss: 2M fp32; bars:
// one unsigned per launch (all zeroed here).  Every layer's tensor maps are
// made before the first launch.  cudaErrorNotSupported when the shapes or
// the device do not fit it, or the device cannot hold the cooperative grid
// at launch time (nothing ran then).
cudaError_t launch_stack_decode(const ptq_ffn_layer* layers, int64_t L, float* x, int64_t M,
                                float* gu0, float* gu1, float* ss, unsigned* bars, int64_t H,
                                int64_t I, float eps, cudaStream_t st);
// A grid barrier of the persistent stack that one CTA never reaches: the
// others' bounded waits run out and raise the status word.
cudaError_t launch_selftest_grid_timeout(cudaStream_t st);
// Whether launch_stack_decode serves (H, I) on the current device.
bool stack_decode_supported(int64_t H, int64_t I);
// Workspace bytes launch_stack_decode needs in `ss` and `bars`.
size_t stack_decode_ss_bytes(int64_t M);
size_t stack_decode_bar_bytes(int64_t L);

// Residual add and RMSNorm between chained blocks (k_norm.cu): per row of
// x (M x H fp32, in place) x += y, then xn = x / sqrt(mean(x^2) + eps) * g.
// y and xn are F32 or BF16 (t); y == nullptr skips the add, xn == nullptr
// the norm.  H % 4 == 0; x, y, g, xn 16-byte aligned.
cudaError_t launch_add_rmsnorm(float* x, const void* y, const float* g, void* xn, Act t,
                               int64_t M, int64_t H, float eps, cudaStream_t st);

// Tensor-core GEMM (k_gemm_tc.cu); cudaErrorNotSupported when the shape does
// not fit it (the caller then uses the SIMT kernel).
cudaError_t launch_gemm_tc(const uint8_t* wq, const uint16_t* scales, const void* x, Act x_t,
                           void* y, Act y_t, int64_t M, int64_t N, int64_t K, void* ws,
                           size_t ws_bytes, cudaStream_t st);
// The tensor-core GEMM over PQ2_0 weights (bf16 x, bf16 y; K % 1024 == 0);
// ws as launch_gemm_tc.
cudaError_t launch_gemm_tc_pq2(const uint8_t* wq, const uint16_t* scales, const void* x, void* y,
                               int64_t M, int64_t N, int64_t K, void* ws, size_t ws_bytes,
                               cudaStream_t st);
// The gate+up GEMM of the feed-forward block with SwiGLU in its epilogue:
// wq/scales hold 2I rows (gate then up), h = silu(g) * u is M x I fp32.
// cudaErrorNotSupported when the shape would be split along K (the caller
// then runs the GEMM into fp32 and launch_swiglu).
cudaError_t launch_gemm_tc_swiglu(const uint8_t* wq, const uint16_t* scales, const void* x,
                                  Act x_t, float* h, int64_t M, int64_t I, int64_t K,
                                  cudaStream_t st);
// K splits of the tensor-core GEMM for a shape, and the fp32 partial-sum
// scratch they need (0 when the product runs unsplit).
int gemm_tc_splits(int64_t M, int64_t N, int64_t K);
size_t gemm_tc_workspace_bytes(int64_t M, int64_t N, int64_t K);

// 2-D TMA tensor map over a row-major array (tma_util.cu): `inner` elements
// per row, `rows` rows `row_bytes` apart, boxes of box_inner x box_rows.
cudaError_t encode_tma_2d(CUtensorMap* map, CUtensorMapDataType dt, const void* base,
                          uint64_t inner, uint64_t rows, uint64_t row_bytes, uint32_t box_inner,
                          uint32_t box_rows, CUtensorMapSwizzle swizzle);

// One CTA waits (bounded) on an mbarrier nothing arrives on and raises the
// device status word when the wait runs out (k_selftest.cu).
cudaError_t launch_selftest_timeout(cudaStream_t st);

// Device status word access (defined in api.cu).
cudaError_t read_and_clear_device_status(int* out, cudaStream_t st);
int* device_status_ptr();

}  // namespace ptq

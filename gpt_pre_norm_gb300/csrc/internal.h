// internal.h -- declarations shared by the host orchestrator (gpt2_api.cu)
// and the kernel launchers (gemm_tc.cu, attention.cu, rowwise.cu, simt_fp32.cu).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "gpt2.h"

namespace gpt2 {

typedef __nv_bfloat16 bf16;

// Profiled kernel kinds (names returned by gpt2_profile_read).
enum KernelKind : int {
  kKindEmbed = 0,
  kKindLayerNorm,
  kKindGemmQkv,
  kKindAttention,
  kKindGemmProj,
  kKindGemmFc,
  kKindGemmMlpProj,
  kKindGemmLogits,
  kKindGemmOther,
  kKindDecodeAttention,
  kKindDecodeCombine,
  kKindSimtFp32,
  kKindArgmax,
  kKindLossCombine,
  kKindCount
};

// Epilogues of the tensor-core GEMM.
enum EpiKind : int {
  kEpiBias = 0,       // out_16 = acc + bias                (bf16 or fp16)
  kEpiGelu,           // out_16 = gelu_tanh(acc + bias)     (bf16 or fp16)
  kEpiResidF32,       // out_f32  = resid_f32 + acc + bias
  kEpiResidBf16In,    // out_f32  = resid_bf16 + acc + bias
  kEpiResidBf16Out,   // out_bf16 = resid_f32 + acc + bias
  kEpiLogits,         // out_f32  = acc (no bias, N tail masked)
  kEpiQkv,            // acc + bias scattered to Q [B,h,T,64] and the K/V cache
  kEpiLogitsT,        // (internal) kEpiLogits computed as W A^T: TMEM lanes = vocabulary
  kEpiHeadLoss,       // the tied head (tokens on TMEM lanes) reduced to per-token partials
  kEpiHeadTopK,       // the tied head reduced to per-token top-k candidates and logsumexp partials
  kEpiCount
};

// Where c_attn's keys and values go: a cache laid out [.., 2, h, T_cap, 64]
// with the element strides below (token stride = d_h).
struct KvDst {
  void* base;
  long long s_batch;  // elements between sequences
  long long s_kv;     // elements between the K and V halves
  long long s_head;   // elements between heads (= T_cap * d_h)
  int t_past;         // first position written
};

// Vocabulary entries per partial of the head reduced to the loss (one
// 256-wide tile of the head per token).
constexpr int kHeadLossBlock = 256;
// Candidates the top-k head keeps per (token, vocabulary block): the largest k allowed.
constexpr int kTopKMax = 8;

struct EpiParams {
  const void* bias;         // [N], mode dtype
  const void* resid;        // [M, ldo] (fp32 or bf16 by kind)
  void* out;                // [M, ldo] (fp32 or bf16 by kind)
  int ldo;                  // row stride of resid and out, elements
  void* q;                  // Q destination [B, h, T, d_h] (kEpiQkv)
  KvDst kv;                 // K/V destination (kEpiQkv)
  int T;                    // tokens per sequence (kEpiQkv)
  int d;                    // model width (kEpiQkv)
  // kEpiHeadLoss: per token t and vocabulary block j of kHeadLossBlock entries, the
  // maximum logit part_m[j * n_tok + t], the sum over the block of
  // 2^((z - max) log2 e) part_s[..], the lowest index of the maximum part_i[..];
  // tgt_logit[t] = the logit of entry tgt[t] for 0 <= tgt[t] < V (a target
  // past V may leave -inf there, which the combine ignores: it reports the
  // target as bad).
  const int32_t* tgt;
  float* tgt_logit;
  float* part_m;
  float* part_s;
  int32_t* part_i;
  // kEpiHeadTopK: part_m, part_s as above, and the block's topk_k largest
  // logits in descending order (among equal values the lower index first; NaN
  // and -inf never taken) in the first topk_k of kTopKMax slots
  // topk_v[(j * n_tok + t) * kTopKMax + i], with their indices topk_i[..]
  // (-inf and 0x7fffffff where the block has fewer; the later slots hold
  // some of the next largest, and are not read).
  float* topk_v;
  int32_t* topk_i;
  int topk_k;
};

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// Per-device launch environment.
struct LaunchEnv {
  int num_sms;
  unsigned* err;          // device error word
  EncodeTiledFn encode;   // cuTensorMapEncodeTiled
  unsigned long long wait_ns;  // limit of every bounded wait in the kernels
};

// Tensor-core GEMM (16-bit operands, fp32 accumulate in TMEM): C = A[M,K]
// W[N,K]^T with epilogue `kind`.  A and W are both fp16 (operands_f16) or both
// bf16; out_f16 selects fp16 over bf16 for the kEpiBias / kEpiGelu outputs.
// Returns a gpt2_status.
int launch_gemm_tc(const LaunchEnv& env, int kind, const void* A, const void* W, int M, int N,
                   int K, const EpiParams& ep, cudaStream_t stream, double* flops, double* bytes,
                   bool operands_f16, bool out_f16);

// Weight-streaming GEMM for M <= 32 rows (cached decode): fp16 X [M, K] and
// W [N, K], fp32 accumulate, epilogues kEpiQkv / kEpiGelu / kEpiBias (fp16
// out) / kEpiResidF32 (K > 1024 only in place, out == resid).
bool smallm_supported(int kind, int M, int K);
// w_early: W was written before the current call's first launch, so its loads
// may start before the previous kernel completes.
int launch_gemm_smallm(const LaunchEnv& env, int kind, const __half* X, const __half* W, int M,
                       int N, int K, const EpiParams& ep, cudaStream_t stream, double* flops,
                       double* bytes, bool w_early = false);

// fp32 SIMT GEMM with the same epilogues (fp32 storage throughout).
int launch_gemm_fp32(const LaunchEnv& env, int kind, const float* A, const float* W, int M, int N,
                     int K, const EpiParams& ep, int d_h, cudaStream_t stream);

// Element-wise bf16 -> fp16 copies of up to kMaxConvSegs arrays (run by the
// extra blocks of a LayerNorm launch).
constexpr int kMaxConvSegs = 4;
struct ConvSegs {
  const bf16* src[kMaxConvSegs];
  __half* dst[kMaxConvSegs];
  long long n[kMaxConvSegs];
  int count;
};

// LayerNorm rows of d: x fp32 or bf16 -> y (mode BF16: bf16, or fp16 when
// y_f16; g, b bf16) or fp32 (mode FP32).  `side`, if given, is a weight
// conversion done by extra blocks of the same launch (both are memory-bound
// and too small to fill the GPU's memory pipeline alone).  With `err`, an fp16
// output or converted weight past the fp16 range (or not finite) raises the
// range bit.
int launch_layer_norm(int mode, const void* x, int x_dtype, const void* g, const void* b, int rows,
                      int d, void* y, cudaStream_t stream, bool y_f16 = false,
                      const ConvSegs* side = nullptr, unsigned* err = nullptr);


// Per token t < n_tok: merges the n_vblk partials of kEpiHeadLoss into
// logsumexp L and the argmax; loss[t] = L - tgt_logit[t] for 0 <= tgt[t] < V,
// 0 for tgt[t] < 0 (NaN and the bad-token error bit for tgt[t] >= V);
// next[t] = the argmax.  loss, next and tgt may be null.
// Top-k of every token from the top-k head's partials: top_v[t * k + i],
// top_i[..] for i < k (descending, lower index first among equal values; -1 where
// fewer than k finite logits exist), lse[t] = logsumexp (NULL to skip).
int launch_head_topk_combine(const float* part_m, const float* part_s, const float* topk_v,
                             const int32_t* topk_i, int n_vblk, int n_tok, int k, float* top_v,
                             int32_t* top_i, float* lse, cudaStream_t stream);
int launch_head_loss_combine(const float* part_m, const float* part_s, const int32_t* part_i,
                             int n_vblk, int n_tok, int V, const int32_t* tgt,
                             const float* tgt_logit, float* loss, int32_t* next, unsigned* err,
                             cudaStream_t stream);

// out[r * out_stride] = next[r] = argmax over the V values of row r (rows
// row_stride apart); the lowest index among equal maxima.
int launch_argmax_rows(const float* x, int rows, int V, long long row_stride, int32_t* out,
                       long long out_stride, int32_t* next, cudaStream_t stream);

// H[b,t,:] = wte[ids[b,t]] + wpe[t_past + t] -> fp32.
int launch_embed(int mode, const int32_t* ids, const void* wte, const void* wpe, int B, int T,
                 int t_past, int d, int n_vocab, float* H, unsigned* err, cudaStream_t stream);

// Causal prefill attention, bf16 Q/K/V, d_h = 64, on tcgen05 (TMEM
// accumulators, TMA); the output [B, T, h*64] is fp16 when out_f16, else bf16.
int launch_attention_tc(const LaunchEnv& env, const bf16* q, const bf16* kv, long long s_batch,
                        long long s_kv, long long s_head, int B, int h, int T, int t_past,
                        void* out, cudaStream_t stream, bool out_f16);


// Single-token decode attention, bf16 Q/K/V, d_h = 64: split over keys,
// partial results combined through `partials` (floats, see
// decode_partials_floats); output fp16 when out_f16, else bf16.
int launch_decode_attention_bf16(const bf16* q, const bf16* kv, long long kv_s_batch,
                                 long long kv_s_kv, long long kv_s_head, int B, int h, int t_len,
                                 void* out, float* partials, int splits, cudaStream_t stream,
                                 int* launches, bool out_f16 = false, unsigned* err = nullptr,
                                 unsigned long long wait_ns = 0);  // 0: the default limit
size_t decode_partials_floats(int B, int h, int splits);
int decode_splits(int B, int h, int t_len, int num_sms);

// fp32 attention (any d_h <= 256), with cache offset.
int launch_attention_fp32(const float* q, const float* kv, long long kv_s_batch, long long kv_s_kv,
                          long long kv_s_head, int B, int h, int T, int t_past, int d_h,
                          float* out, cudaStream_t stream);

// Raises the dynamic shared-memory limit of kernel `fn` to `bytes` on the
// current device, the first time it is asked for that (device, kernel, size):
// the attribute is per device, and later calls make no CUDA call at all (so
// they are safe inside a stream capture).  Thread-safe.  Returns false when
// the runtime refuses.
bool ensure_smem_limit(const void* fn, int bytes);

// Overlap with the previous kernel of the stream.  Every launch may overlap
// it unless the calling thread asked for one plain launch: an API call whose
// kernels read cached weights before waiting on their predecessor asks for it
// before its first launch, which then starts only once all earlier work in the
// stream has finished; every later launch of the call starts after that one,
// so weights written by earlier calls are complete when they are read.
void request_plain_launch();
bool take_pdl_permission();  // false once after request_plain_launch()

// Launches `kernel` on `stream` with programmatic stream serialisation (the
// kernel must call pdl_wait() before touching global memory).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = take_pdl_permission() ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

}  // namespace gpt2

// gemm_smallm.cu -- weight-streaming GEMM for a few rows: C[M,N] = X[M,K] W[N,K]^T
// with M <= 32 (one new token per sequence in cached decode), fp16 operands,
// fp32 accumulation, the epilogues of the decode block (bias + Q/K/V split,
// bias + GELU, bias + in-place fp32 residual).
//
// At M = 32 the products are bound by reading W from HBM (about 32 flops per
// byte), so the design maximises bytes in flight rather than MMA rate:
//   - one CTA per 16 output features (and per 1024-wide K chunk), 4 warps, each
//     warp a 256-wide K slice;
//   - one thread issues every TMA load of the CTA's W slice (16 x 1024 fp16)
//     and X chunk (32 x 1024 fp16) at kernel start, 64-wide boxes with the
//     128-byte swizzle, all completing on one mbarrier: one round trip;
//   - "swap AB" mma.sync m16n8k16: W rows are the 16-row A operand, the 32
//     tokens four 8-column B tiles; 16-byte shared loads feed both operands
//     through a consistent permutation of k (the sum over k is order-free);
//   - the four warps' partial tiles are summed in shared memory and the
//     epilogue (bias, GELU, residual, Q/K/V split) is applied once;
//     when K spans several chunks, the chunks add into the fp32 residual with
//     atomics (in-place residual epilogue only).
//
// Early weights: when W was written before the current call began, its loads
// are issued before the wait on the previous kernel, so the weight stream
// overlaps that kernel's tail.
#include "device.cuh"
#include "internal.h"

namespace gpt2 {
namespace {

constexpr int kFeat = 16;               // output features per CTA
constexpr int kKChunk = 1024;           // K per CTA
constexpr int kWarps = 4;               // K slices of 256
constexpr int kSlice = kKChunk / kWarps;
constexpr int kTok = 32;                // token rows (M <= 32)
constexpr int kBoxK = 64;               // k per TMA box: one 128-byte swizzle row
constexpr int kBoxes = kKChunk / kBoxK;
constexpr int kXBox = kTok * 128;       // bytes of one X box (32 rows x 64 k)
constexpr int kWBox = kFeat * 128;      // bytes of one W box (16 rows x 64 k)
constexpr size_t kSmem = 1024 /* alignment */ + static_cast<size_t>(kBoxes) * (kXBox + kWBox) +
                         static_cast<size_t>(kWarps) * kFeat * kTok * 4 + 16;

struct SmallArgs {
  int M, N, K;
  unsigned* err;
  EpiParams ep;
  int w_early;  // W may be read before the previous kernel completes
};

// 16-byte chunk c (0..7) of row r in a 128-byte-swizzled box row.
__device__ __forceinline__ const uint4* box_chunk(const uint8_t* box, int r, int c) {
  return reinterpret_cast<const uint4*>(box + r * 128 + ((c ^ (r & 7)) << 4));
}

__device__ __forceinline__ void mma_f16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                              uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
      "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

template <int KIND>
__global__ void __launch_bounds__(kWarps * 32)
    gemm_smallm(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                const SmallArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sX = smem;                                  // [kBoxes][32 rows x 128 B]
  uint8_t* sW = sX + kBoxes * kXBox;                   // [kBoxes][16 rows x 128 B]
  float* sP = reinterpret_cast<float*>(sW + kBoxes * kWBox);  // [warp][feature][token]
  uint64_t* bar = reinterpret_cast<uint64_t*>(sP + kWarps * kFeat * kTok);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int f0 = blockIdx.x * kFeat;
  const int k0 = blockIdx.y * kKChunk;
  const int M = a.M, N = a.N;

  if (threadIdx.x == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  pdl_trigger();
  // Every box of the CTA at once, on one barrier; boxes past M / N / K read
  // as zero.  W first, and before the wait on the previous kernel when W was
  // written before this call began (it is not produced by that kernel).
  if (threadIdx.x == 0) {
    tma_prefetch_desc(&tmX);
    tma_prefetch_desc(&tmW);
    mbar_arrive_expect_tx(bar, kBoxes * (kWBox + kXBox));
    if (a.w_early)
      for (int j = 0; j < kBoxes; ++j) tma_load_2d(sW + j * kWBox, &tmW, bar, k0 + j * kBoxK, f0);
  }
  pdl_wait();
  if (threadIdx.x == 0) {
    if (!a.w_early)
      for (int j = 0; j < kBoxes; ++j) tma_load_2d(sW + j * kWBox, &tmW, bar, k0 + j * kBoxK, f0);
    for (int j = 0; j < kBoxes; ++j) tma_load_2d(sX + j * kXBox, &tmX, bar, k0 + j * kBoxK, 0);
  }
  mbar_wait_bounded(bar, 0, nullptr, a.err);

  // Warp's K slice [warp*256, +256): 8 steps of 32 k.  Thread (g, t) takes
  // the 8 consecutive k at 8t of each 32-step for A rows g, g+8 and tokens
  // g, g+8, g+16, g+24; mma k-step 0 uses the first four, k-step 1 the rest.
  const int g = lane >> 2, t = lane & 3;
  float acc[4][4];
#pragma unroll
  for (int n = 0; n < 4; ++n)
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[n][e] = 0.f;
#pragma unroll 2
  for (int s = 0; s < kSlice / 32; ++s) {
    const int box = (warp * kSlice + s * 32) / kBoxK;  // 64-wide box of this 32-step
    const int c = (s & 1) * 4 + t;                     // 16-byte chunk within the box row
    const uint4 w0 = *box_chunk(sW + box * kWBox, g, c);
    const uint4 w1 = *box_chunk(sW + box * kWBox, g + 8, c);
    const uint32_t A0[4] = {w0.x, w1.x, w0.y, w1.y};  // k-step 0: a0 a1 a2 a3
    const uint32_t A1[4] = {w0.z, w1.z, w0.w, w1.w};  // k-step 1
#pragma unroll
    for (int n = 0; n < 4; ++n) {
      const uint4 x = *box_chunk(sX + box * kXBox, 8 * n + g, c);
      mma_f16_16816(acc[n], A0, x.x, x.y);
      mma_f16_16816(acc[n], A1, x.z, x.w);
    }
  }
  // acc[n][0..1]: feature g, tokens 8n + 2t, +1; acc[n][2..3]: feature g + 8.
  float* P = sP + warp * kFeat * kTok;
#pragma unroll
  for (int n = 0; n < 4; ++n) {
    P[g * kTok + 8 * n + 2 * t] = acc[n][0];
    P[g * kTok + 8 * n + 2 * t + 1] = acc[n][1];
    P[(g + 8) * kTok + 8 * n + 2 * t] = acc[n][2];
    P[(g + 8) * kTok + 8 * n + 2 * t + 1] = acc[n][3];
  }
  __syncthreads();

  // Epilogue: 512 outputs (16 features x 32 tokens), 4 per thread, the
  // feature index fastest so neighbouring threads write neighbouring columns.
  const EpiParams& ep = a.ep;
  uint32_t mag = 0u;  // kEpiGelu: largest fp16 output magnitude (bits)
  for (int o = threadIdx.x; o < kFeat * kTok; o += blockDim.x) {
    const int fl = o % kFeat, tok = o / kFeat;
    const int f = f0 + fl;
    if (tok >= M || f >= N) continue;
    float v = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) v += sP[w * kFeat * kTok + fl * kTok + tok];
    {
      const bool add_bias = blockIdx.y == 0;
      if (add_bias) v += __bfloat162float(static_cast<const bf16*>(ep.bias)[f]);
      if constexpr (KIND == kEpiResidF32) {
        float* o_ = static_cast<float*>(ep.out) + static_cast<size_t>(tok) * ep.ldo + f;
        if (gridDim.y == 1) {
          *o_ = static_cast<const float*>(ep.resid)[static_cast<size_t>(tok) * ep.ldo + f] + v;
        } else {
          atomicAdd(o_, v);  // in place: out == resid, chunks accumulate
        }
      } else if constexpr (KIND == kEpiGelu) {
        const __half h = __float2half_rn(gelu_tanh_approx(v));
        mag = fp16_max_mag(mag, static_cast<uint32_t>(__half_as_ushort(h)));
        static_cast<__half*>(ep.out)[static_cast<size_t>(tok) * ep.ldo + f] = h;
      } else if constexpr (KIND == kEpiBias) {
        static_cast<__half*>(ep.out)[static_cast<size_t>(tok) * ep.ldo + f] = __float2half_rn(v);
      } else if constexpr (KIND == kEpiQkv) {
        const int which = f / ep.d;
        const int within = f - which * ep.d;
        const int head = within >> 6, dim = within & 63;
        const int bi = tok / ep.T, tt = tok - bi * ep.T;
        bf16* dst;
        if (which == 0) {
          dst = static_cast<bf16*>(ep.q) +
                ((static_cast<size_t>(bi) * (ep.d >> 6) + head) * ep.T + tt) * 64 + dim;
        } else {
          dst = static_cast<bf16*>(ep.kv.base) + bi * ep.kv.s_batch + (which - 1) * ep.kv.s_kv +
                head * ep.kv.s_head + static_cast<long long>(ep.kv.t_past + tt) * 64 + dim;
        }
        *dst = __float2bfloat16_rn(v);
      }
    }
  }
  // An fp16 GELU output past 65504 (or not finite) would feed the next product.
  if (KIND == kEpiGelu && fp16_nonfinite(mag)) raise_error(a.err, kErrRange);
}

template <int KIND>
cudaError_t launch_kind(dim3 grid, cudaStream_t s, const CUtensorMap& tmX, const CUtensorMap& tmW,
                        const SmallArgs& a) {
  if (!ensure_smem_limit(reinterpret_cast<const void*>(&gemm_smallm<KIND>),
                         static_cast<int>(kSmem)))
    return cudaErrorInvalidValue;
  return launch_pdl(gemm_smallm<KIND>, grid, dim3(kWarps * 32), kSmem, s, tmX, tmW, a);
}

// fp16 [rows, K] K-major, boxes of 64 k x box_rows with the 128-byte swizzle.
bool encode_rows_f16(const LaunchEnv& env, CUtensorMap* map, const void* base, int rows, int K,
                     int box_rows) {
  if ((reinterpret_cast<uintptr_t>(base) & 15) != 0) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * 2};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(kBoxK), static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  return env.encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base), dims,
                    strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

}  // namespace

bool smallm_supported(int kind, int M, int K) {
  if (M <= 0 || M > kTok || K % 8 != 0) return false;
  switch (kind) {
    case kEpiQkv: case kEpiGelu: case kEpiBias: return K <= kKChunk;
    case kEpiResidF32: return true;  // K chunks add atomically into the residual
    default: return false;
  }
}

int launch_gemm_smallm(const LaunchEnv& env, int kind, const __half* X, const __half* W, int M,
                       int N, int K, const EpiParams& ep, cudaStream_t stream, double* flops,
                       double* bytes, bool w_early) {
  if (!smallm_supported(kind, M, K) || N <= 0) return GPT2_ERR_UNSUPPORTED;
  const int chunks = (K + kKChunk - 1) / kKChunk;
  if (chunks > 1 && (kind != kEpiResidF32 || ep.out != ep.resid)) return GPT2_ERR_UNSUPPORTED;
  CUtensorMap tmX, tmW;
  if (!encode_rows_f16(env, &tmX, X, M, K, kTok) || !encode_rows_f16(env, &tmW, W, N, K, kFeat))
    return GPT2_ERR_CUDA;
  SmallArgs a{M, N, K, env.err, ep, w_early ? 1 : 0};
  const dim3 grid((N + kFeat - 1) / kFeat, chunks);
  cudaError_t e;
  switch (kind) {
    case kEpiQkv: e = launch_kind<kEpiQkv>(grid, stream, tmX, tmW, a); break;
    case kEpiGelu: e = launch_kind<kEpiGelu>(grid, stream, tmX, tmW, a); break;
    case kEpiBias: e = launch_kind<kEpiBias>(grid, stream, tmX, tmW, a); break;
    case kEpiResidF32: e = launch_kind<kEpiResidF32>(grid, stream, tmX, tmW, a); break;
    default: return GPT2_ERR_UNSUPPORTED;
  }
  if (e != cudaSuccess) return GPT2_ERR_CUDA;
  if (flops) *flops = 2.0 * M * N * static_cast<double>(K);
  if (bytes) *bytes = 2.0 * (static_cast<double>(N) * K + static_cast<double>(M) * K) +
                      (kind == kEpiResidF32 ? 8.0 : 2.0) * M * N;
  return GPT2_OK;
}

}  // namespace gpt2

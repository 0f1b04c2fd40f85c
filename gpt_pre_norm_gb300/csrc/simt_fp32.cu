// simt_fp32.cu -- fp32 GEMM on the CUDA cores: C[M,N] = A[M,K] * W[N,K]^T
// with the same epilogues as the tensor-core GEMM (bias, GELU tanh form,
// residual add, logits, QKV split into heads and the KV cache).
//
// fp32 mode exists for exact-ish checking: TF32 tensor cores keep 10 mantissa
// bits, too few for a 1e-4 bound, so every product here is an fp32 FMA.
// Tiles of 64 x 64 outputs, 16 x 16 threads with 4 x 4 outputs each, K staged
// through shared memory 16 at a time.
#include <math.h>

#include "device.cuh"
#include "internal.h"

namespace gpt2 {

namespace {

constexpr int kT = 64;   // output tile
constexpr int kKt = 16;  // K step

struct Fp32Args {
  int M, N, K, d_h;
  EpiParams ep;
};

template <int KIND>
__device__ __forceinline__ void epi_store(const Fp32Args& a, int m, int n, float acc) {
  const EpiParams& ep = a.ep;
  if constexpr (KIND == kEpiLogits) {
    static_cast<float*>(ep.out)[static_cast<size_t>(m) * ep.ldo + n] = acc;
    return;
  } else {
    const float v = acc + static_cast<const float*>(ep.bias)[n];
    if constexpr (KIND == kEpiBias) {
      static_cast<float*>(ep.out)[static_cast<size_t>(m) * ep.ldo + n] = v;
    } else if constexpr (KIND == kEpiGelu) {
      static_cast<float*>(ep.out)[static_cast<size_t>(m) * ep.ldo + n] = gelu_tanh(v);
    } else if constexpr (KIND == kEpiResidF32) {
      const size_t off = static_cast<size_t>(m) * ep.ldo + n;
      static_cast<float*>(ep.out)[off] = static_cast<const float*>(ep.resid)[off] + v;
    } else if constexpr (KIND == kEpiQkv) {
      const int which = n / ep.d;
      const int within = n - which * ep.d;
      const int head = within / a.d_h, dim = within - head * a.d_h;
      const int h = ep.d / a.d_h;
      const int bi = m / ep.T, t = m - bi * ep.T;
      if (which == 0) {
        static_cast<float*>(ep.q)[((static_cast<size_t>(bi) * h + head) * ep.T + t) * a.d_h + dim] = v;
      } else {
        static_cast<float*>(ep.kv.base)[bi * ep.kv.s_batch + (which - 1) * ep.kv.s_kv +
                                        head * ep.kv.s_head +
                                        static_cast<long long>(ep.kv.t_past + t) * a.d_h + dim] = v;
      }
    }
  }
}

template <int KIND>
__global__ void __launch_bounds__(256)
    gemm_fp32_kernel(const float* __restrict__ A, const float* __restrict__ W, const Fp32Args a) {
  __shared__ float sA[kKt][kT + 1];
  __shared__ float sW[kKt][kT + 1];
  pdl_trigger();
  pdl_wait();
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const int m0 = blockIdx.y * kT, n0 = blockIdx.x * kT;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < a.K; k0 += kKt) {
    for (int i = threadIdx.x; i < kKt * kT; i += 256) {
      const int r = i / kKt, c = i % kKt;
      const int m = m0 + r, n = n0 + r, k = k0 + c;
      sA[c][r] = (m < a.M && k < a.K) ? A[static_cast<size_t>(m) * a.K + k] : 0.f;
      sW[c][r] = (n < a.N && k < a.K) ? W[static_cast<size_t>(n) * a.K + k] : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < kKt; ++kk) {
      float av[4], wv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        av[i] = sA[kk][ty + 16 * i];
        wv[i] = sW[kk][tx + 16 * i];
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], wv[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int m = m0 + ty + 16 * i;
    if (m >= a.M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = n0 + tx + 16 * j;
      if (n < a.N) epi_store<KIND>(a, m, n, acc[i][j]);
    }
  }
}

}  // namespace

int launch_gemm_fp32(const LaunchEnv& env, int kind, const float* A, const float* W, int M, int N,
                     int K, const EpiParams& ep, int d_h, cudaStream_t stream) {
  (void)env;
  if (M <= 0 || N <= 0 || K <= 0) return GPT2_ERR_INVALID_ARG;
  if (kind == kEpiQkv && (d_h <= 0 || ep.d % d_h != 0 || N != 3 * ep.d)) return GPT2_ERR_INVALID_ARG;
  Fp32Args a{M, N, K, d_h, ep};
  dim3 grid((N + kT - 1) / kT, (M + kT - 1) / kT);
  if (grid.y > 65535) return GPT2_ERR_UNSUPPORTED;
  cudaError_t e;
  const dim3 block(256);
  switch (kind) {
    case kEpiBias: e = launch_pdl(gemm_fp32_kernel<kEpiBias>, grid, block, 0, stream, A, W, a); break;
    case kEpiGelu: e = launch_pdl(gemm_fp32_kernel<kEpiGelu>, grid, block, 0, stream, A, W, a); break;
    case kEpiResidF32:
      e = launch_pdl(gemm_fp32_kernel<kEpiResidF32>, grid, block, 0, stream, A, W, a);
      break;
    case kEpiLogits: e = launch_pdl(gemm_fp32_kernel<kEpiLogits>, grid, block, 0, stream, A, W, a); break;
    case kEpiQkv: e = launch_pdl(gemm_fp32_kernel<kEpiQkv>, grid, block, 0, stream, A, W, a); break;
    default: return GPT2_ERR_INVALID_ARG;
  }
  return e == cudaSuccess ? GPT2_OK : GPT2_ERR_CUDA;
}

}  // namespace gpt2

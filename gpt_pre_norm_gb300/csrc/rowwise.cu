// rowwise.cu -- the memory-bound row kernels: LayerNorm (fused with the cast
// of its output, and carrying the bf16 -> fp16 weight conversion of the
// products that follow it as extra blocks of the same launch) and the
// embedding gather + position add.
//
// LayerNorm follows the openai/gpt-2 ``norm`` excerpt on the "GPT-2
// Transformer block" page: over the feature axis u = mean(x), s = mean((x -
// u)^2) (biased), y = (x - u) * rsqrt(s + eps) * g + b with eps = 1e-5 ("GPT-2
// Decoder Block", "How it works").  One warp owns one row, keeps it in
// registers, and reduces with shuffles: one read of x, one write of y.
//
// The embedding follows "GPT-2 Full Forward Pass", "How it works":
// H0[b, t] = wte[ids[b, t]] + wpe[T_past + t], written in fp32 (the residual
// stream).  One warp per token, 16-byte loads.
#include <type_traits>

#include "device.cuh"
#include "internal.h"

namespace gpt2 {

namespace {

constexpr float kLnEps = 1e-5f;
constexpr int kRowThreads = 256;
constexpr int kRowsPerBlock = kRowThreads / 32;

__device__ __forceinline__ void load2(const float* p, float& a, float& b) {
  const float2 v = *reinterpret_cast<const float2*>(p);
  a = v.x;
  b = v.y;
}
__device__ __forceinline__ void load2(const bf16* p, float& a, float& b) {
  const uint32_t v = *reinterpret_cast<const uint32_t*>(p);
  a = bf16_lo(v);
  b = bf16_hi(v);
}
__device__ __forceinline__ void store2(float* p, float a, float b) {
  *reinterpret_cast<float2*>(p) = make_float2(a, b);
}
__device__ __forceinline__ void store2(bf16* p, float a, float b) {
  *reinterpret_cast<uint32_t*>(p) = pack_bf16x2(a, b);
}
__device__ __forceinline__ void store2(__half* p, float a, float b) {
  *reinterpret_cast<uint32_t*>(p) = pack_f16x2(a, b);
}

// Stores that also keep the magnitude test of fp16 outputs (the bits of the
// packed halves, see fp16_max_mag); other output types store only.
template <typename TY>
__device__ __forceinline__ void store2c(TY* p, float a, float b, uint32_t&) {
  store2(p, a, b);
}
__device__ __forceinline__ void store2c(__half* p, float a, float b, uint32_t& mag) {
  const uint32_t w = pack_f16x2(a, b);
  mag = fp16_max_mag(mag, w);
  *reinterpret_cast<uint32_t*>(p) = w;
}
__device__ __forceinline__ void report_range(uint32_t mag, unsigned* err) {
  if (__any_sync(0xffffffffu, fp16_nonfinite(mag)) && (threadIdx.x & 31) == 0)
    raise_error(err, kErrRange);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  return v;
}

__device__ __forceinline__ uint4 bf16x8_to_f16x8(const uint4 v) {
  return make_uint4(pack_f16x2(bf16_lo(v.x), bf16_hi(v.x)), pack_f16x2(bf16_lo(v.y), bf16_hi(v.y)),
                    pack_f16x2(bf16_lo(v.z), bf16_hi(v.z)), pack_f16x2(bf16_lo(v.w), bf16_hi(v.w)));
}

// bf16 -> fp16 conversion of up to kMaxConvSegs arrays, cut into blocks of
// kRowThreads x kConvChunks 16-byte chunks; first[i] is array i's first block.
// A bf16 value converts exactly unless its magnitude is below 2^-14 (fp16
// subnormal range) or above 65504.
constexpr int kConvChunks = 8;
constexpr long long kConvBlockChunks = static_cast<long long>(kRowThreads) * kConvChunks;

struct ConvJob {
  const bf16* src[kMaxConvSegs];
  __half* dst[kMaxConvSegs];
  long long n[kMaxConvSegs];
  int first[kMaxConvSegs + 1];  // first[count] = blocks in all
  int count;
  unsigned* err;  // range bit: a value past the fp16 range (the LayerNorm's too)
};

ConvJob make_conv_job(const ConvSegs* segs, unsigned* err) {
  ConvJob j{};
  j.err = err;
  j.count = segs ? segs->count : 0;
  for (int i = 0; i < j.count; ++i) {
    j.src[i] = segs->src[i];
    j.dst[i] = segs->dst[i];
    j.n[i] = segs->n[i];
    const long long chunks = (segs->n[i] + 7) / 8;
    const long long blocks = (chunks + kConvBlockChunks - 1) / kConvBlockChunks;
    j.first[i + 1] = j.first[i] + static_cast<int>(blocks < 1 ? 1 : blocks);
  }
  return j;
}

// Block b of a conversion job: all of its loads are issued before any store.
// A bf16 value whose magnitude exceeds 65504 becomes an fp16 infinity: that
// raises the range bit (the products would use infinite weights).
__device__ __forceinline__ void convert_part(const ConvJob& job, int b) {
  int i = 0;
  while (i + 1 < job.count && b >= job.first[i + 1]) ++i;
  const uint4* __restrict__ src = reinterpret_cast<const uint4*>(job.src[i]);
  uint4* __restrict__ dst = reinterpret_cast<uint4*>(job.dst[i]);
  const long long n = job.n[i], n8 = n / 8;
  const long long c0 = static_cast<long long>(b - job.first[i]) * kConvBlockChunks + threadIdx.x;
  uint4 v[kConvChunks];
#pragma unroll
  for (int k = 0; k < kConvChunks; ++k) {
    const long long c = c0 + static_cast<long long>(k) * kRowThreads;
    if (c < n8) v[k] = src[c];
  }
  uint32_t mag = 0u;
#pragma unroll
  for (int k = 0; k < kConvChunks; ++k) {
    const long long c = c0 + static_cast<long long>(k) * kRowThreads;
    if (c < n8) {
      const uint4 h = bf16x8_to_f16x8(v[k]);
      mag = fp16_max_mag(fp16_max_mag(mag, h.x), h.y);
      mag = fp16_max_mag(fp16_max_mag(mag, h.z), h.w);
      dst[c] = h;
    }
  }
  if (b == job.first[i + 1] - 1) {  // the array's last block: its ragged tail
    const bf16* s1 = job.src[i];
    __half* d1 = job.dst[i];
    for (long long e = n8 * 8 + threadIdx.x; e < n; e += kRowThreads) {
      const __half h = __float2half_rn(__bfloat162float(s1[e]));
      mag = fp16_max_mag(mag, static_cast<uint32_t>(__half_as_ushort(h)));
      d1[e] = h;
    }
  }
  if (__any_sync(0xffffffffu, fp16_nonfinite(mag)) && (threadIdx.x & 31) == 0)
    raise_error(job.err, kErrRange);
}

// Row held in registers: NP pairs per lane, d <= 64 * NP, d even (the form
// used where the 16-byte one does not apply).  TX input, TP gain/bias, TY output.
template <typename TX, typename TP, typename TY, int NP>
__global__ void __launch_bounds__(kRowThreads)
    layer_norm_reg(const TX* __restrict__ x, const TP* __restrict__ g, const TP* __restrict__ b,
                   int rows, int d, TY* __restrict__ y, const __grid_constant__ ConvJob side) {
  pdl_trigger();
  pdl_wait();
  const int conv_blocks = side.first[side.count];
  if (static_cast<int>(blockIdx.x) < conv_blocks) {
    convert_part(side, blockIdx.x);
    return;
  }
  const int row = (blockIdx.x - conv_blocks) * kRowsPerBlock + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const TX* xr = x + static_cast<size_t>(row) * d;
  float v[2 * NP];
  float sum = 0.f;
#pragma unroll
  for (int i = 0; i < NP; ++i) {
    const int c = 2 * (lane + 32 * i);
    if (c < d) {
      load2(xr + c, v[2 * i], v[2 * i + 1]);
    } else {
      v[2 * i] = v[2 * i + 1] = 0.f;
    }
    sum += v[2 * i] + v[2 * i + 1];
  }
  const float inv_d = 1.0f / static_cast<float>(d);
  const float u = warp_sum(sum) * inv_d;
  float sq = 0.f;
#pragma unroll
  for (int i = 0; i < NP; ++i) {
    const int c = 2 * (lane + 32 * i);
    if (c < d) {
      const float a0 = v[2 * i] - u, a1 = v[2 * i + 1] - u;
      sq = fmaf(a0, a0, fmaf(a1, a1, sq));
    }
  }
  const float s = warp_sum(sq) * inv_d;
  const float rstd = rsqrtf(s + kLnEps);
  TY* yr = y + static_cast<size_t>(row) * d;
  uint32_t mag = 0u;
#pragma unroll
  for (int i = 0; i < NP; ++i) {
    const int c = 2 * (lane + 32 * i);
    if (c < d) {
      float g0, g1, b0, b1;
      load2(g + c, g0, g1);
      load2(b + c, b0, b1);
      store2c(yr + c, (v[2 * i] - u) * rstd * g0 + b0, (v[2 * i + 1] - u) * rstd * g1 + b1, mag);
    }
  }
  report_range(mag, side.err);
}

// Eight consecutive row values <-> registers with 16-byte accesses.
__device__ __forceinline__ void load8(const float* p, float* v) {
  const float4 a = reinterpret_cast<const float4*>(p)[0], c = reinterpret_cast<const float4*>(p)[1];
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = c.x; v[5] = c.y; v[6] = c.z; v[7] = c.w;
}
__device__ __forceinline__ void load8(const bf16* p, float* v) {
  const uint4 w = *reinterpret_cast<const uint4*>(p);
  const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = bf16_lo(u[i]);
    v[2 * i + 1] = bf16_hi(u[i]);
  }
}
__device__ __forceinline__ void store8(float* p, const float* v) {
  reinterpret_cast<float4*>(p)[0] = make_float4(v[0], v[1], v[2], v[3]);
  reinterpret_cast<float4*>(p)[1] = make_float4(v[4], v[5], v[6], v[7]);
}
__device__ __forceinline__ void store8(bf16* p, const float* v) {
  *reinterpret_cast<uint4*>(p) = make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]),
                                            pack_bf16x2(v[4], v[5]), pack_bf16x2(v[6], v[7]));
}
__device__ __forceinline__ void store8(__half* p, const float* v) {
  *reinterpret_cast<uint4*>(p) = make_uint4(pack_f16x2(v[0], v[1]), pack_f16x2(v[2], v[3]),
                                            pack_f16x2(v[4], v[5]), pack_f16x2(v[6], v[7]));
}
template <typename TY>
__device__ __forceinline__ void store8c(TY* p, const float* v, uint32_t&) {
  store8(p, v);
}
__device__ __forceinline__ void store8c(__half* p, const float* v, uint32_t& mag) {
  const uint4 w = make_uint4(pack_f16x2(v[0], v[1]), pack_f16x2(v[2], v[3]),
                             pack_f16x2(v[4], v[5]), pack_f16x2(v[6], v[7]));
  mag = fp16_max_mag(fp16_max_mag(mag, w.x), w.y);
  mag = fp16_max_mag(fp16_max_mag(mag, w.z), w.w);
  *reinterpret_cast<uint4*>(p) = w;
}

// Row held in registers as NC groups of eight values per lane (group
// lane + 32 i covers elements 8 (lane + 32 i) .. +7): 16-byte loads and
// stores, d % 8 == 0, d <= 256 NC; mean and variance in two passes over the
// registers.
template <typename TX, typename TP, typename TY, int NC>
__global__ void __launch_bounds__(kRowThreads, NC <= 3 ? 6 : (NC <= 4 ? 5 : 3))
    layer_norm_vec(const TX* __restrict__ x, const TP* __restrict__ g, const TP* __restrict__ b,
                   int rows, int d, TY* __restrict__ y, const __grid_constant__ ConvJob side) {
  pdl_trigger();
  pdl_wait();
  const int conv_blocks = side.first[side.count];
  if (static_cast<int>(blockIdx.x) < conv_blocks) {
    convert_part(side, blockIdx.x);
    return;
  }
  const int row = (blockIdx.x - conv_blocks) * kRowsPerBlock + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const int ng = d >> 3;
  const TX* xr = x + static_cast<size_t>(row) * d;
  float v[8 * NC];
  float sum = 0.f;
#pragma unroll
  for (int i = 0; i < NC; ++i) {
    const int gi = lane + 32 * i;
    if (gi < ng) {
      load8(xr + 8 * gi, v + 8 * i);
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) v[8 * i + e] = 0.f;
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) sum += v[8 * i + e];
  }
  const float inv_d = 1.0f / static_cast<float>(d);
  const float u = warp_sum(sum) * inv_d;
  float sq = 0.f;
#pragma unroll
  for (int i = 0; i < NC; ++i) {
    if (lane + 32 * i < ng) {
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float a = v[8 * i + e] - u;
        sq = fmaf(a, a, sq);
      }
    }
  }
  const float rstd = rsqrtf(warp_sum(sq) * inv_d + kLnEps);
  TY* yr = y + static_cast<size_t>(row) * d;
  uint32_t mag = 0u;
#pragma unroll
  for (int i = 0; i < NC; ++i) {
    const int gi = lane + 32 * i;
    if (gi < ng) {
      float gg[8], bb[8], o[8];
      load8(g + 8 * gi, gg);
      load8(b + 8 * gi, bb);
#pragma unroll
      for (int e = 0; e < 8; ++e) o[e] = (v[8 * i + e] - u) * rstd * gg[e] + bb[e];
      store8c(yr + 8 * gi, o, mag);
    }
  }
  report_range(mag, side.err);
}

__device__ __forceinline__ float ld1(const float* p) { return *p; }
__device__ __forceinline__ float ld1(const bf16* p) { return __bfloat162float(*p); }
__device__ __forceinline__ void st1(float* p, float v) { *p = v; }
__device__ __forceinline__ void st1(bf16* p, float v) { *p = __float2bfloat16_rn(v); }
__device__ __forceinline__ void st1(__half* p, float v) { *p = __float2half_rn(v); }

// Any d: three passes over the row in global memory.
template <typename TX, typename TP, typename TY>
__global__ void __launch_bounds__(kRowThreads)
    layer_norm_any(const TX* __restrict__ x, const TP* __restrict__ g, const TP* __restrict__ b,
                   int rows, int d, TY* __restrict__ y, const __grid_constant__ ConvJob side) {
  pdl_trigger();
  pdl_wait();
  const int conv_blocks = side.first[side.count];
  if (static_cast<int>(blockIdx.x) < conv_blocks) {
    convert_part(side, blockIdx.x);
    return;
  }
  const int row = (blockIdx.x - conv_blocks) * kRowsPerBlock + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const TX* xr = x + static_cast<size_t>(row) * d;
  float sum = 0.f;
  for (int c = lane; c < d; c += 32) sum += ld1(xr + c);
  const float u = warp_sum(sum) / static_cast<float>(d);
  float sq = 0.f;
  for (int c = lane; c < d; c += 32) {
    const float a = ld1(xr + c) - u;
    sq = fmaf(a, a, sq);
  }
  const float rstd = rsqrtf(warp_sum(sq) / static_cast<float>(d) + kLnEps);
  TY* yr = y + static_cast<size_t>(row) * d;
  uint32_t mag = 0u;
  for (int c = lane; c < d; c += 32) {
    const float o = (ld1(xr + c) - u) * rstd * ld1(g + c) + ld1(b + c);
    st1(yr + c, o);
    if constexpr (sizeof(TY) == 2 && !std::is_same<TY, bf16>::value)
      mag = fp16_max_mag(mag, static_cast<uint32_t>(__half_as_ushort(__float2half_rn(o))));
  }
  report_range(mag, side.err);
}

__host__ __device__ inline bool aligned16(const void* p) {
  return (reinterpret_cast<uintptr_t>(p) & 15) == 0;
}

// The conversion blocks come first in the grid, so they start in the first
// wave; the LayerNorm rows follow.
template <typename TX, typename TP, typename TY>
int ln_dispatch(const TX* x, const TP* g, const TP* b, int rows, int d, TY* y, cudaStream_t s,
                const ConvJob& side) {
  const unsigned blocks = static_cast<unsigned>((rows + kRowsPerBlock - 1) / kRowsPerBlock) +
                          static_cast<unsigned>(side.first[side.count]);
  const dim3 grid(blocks), block(kRowThreads);
  cudaError_t e;
  const bool vec = d % 8 == 0 && aligned16(x) && aligned16(g) && aligned16(b) && aligned16(y);
  if (vec && d <= 256 * 1) {
    e = launch_pdl(layer_norm_vec<TX, TP, TY, 1>, grid, block, 0, s, x, g, b, rows, d, y, side);
  } else if (vec && d <= 256 * 3) {
    e = launch_pdl(layer_norm_vec<TX, TP, TY, 3>, grid, block, 0, s, x, g, b, rows, d, y, side);
  } else if (vec && d <= 256 * 4) {
    e = launch_pdl(layer_norm_vec<TX, TP, TY, 4>, grid, block, 0, s, x, g, b, rows, d, y, side);
  } else if (vec && d <= 256 * 7) {
    e = launch_pdl(layer_norm_vec<TX, TP, TY, 7>, grid, block, 0, s, x, g, b, rows, d, y, side);
  } else if (d % 2 == 0 && d <= 64 * 4) {
    e = launch_pdl(layer_norm_reg<TX, TP, TY, 4>, grid, block, 0, s, x, g, b, rows, d, y, side);
  } else if (d % 2 == 0 && d <= 64 * 12) {
    e = launch_pdl(layer_norm_reg<TX, TP, TY, 12>, grid, block, 0, s, x, g, b, rows, d, y, side);
  } else if (d % 2 == 0 && d <= 64 * 16) {
    e = launch_pdl(layer_norm_reg<TX, TP, TY, 16>, grid, block, 0, s, x, g, b, rows, d, y, side);
  } else if (d % 2 == 0 && d <= 64 * 25) {
    e = launch_pdl(layer_norm_reg<TX, TP, TY, 25>, grid, block, 0, s, x, g, b, rows, d, y, side);
  } else {
    e = launch_pdl(layer_norm_any<TX, TP, TY>, grid, block, 0, s, x, g, b, rows, d, y, side);
  }
  return e == cudaSuccess ? GPT2_OK : GPT2_ERR_CUDA;
}

// ---------------------------------------------------------------- embed ----
__device__ __forceinline__ int checked_id(const int32_t* ids, size_t i, int n_vocab, unsigned* err) {
  int id = ids[i];
  if (id < 0 || id >= n_vocab) {
    raise_error(err, kErrBadToken);
    id = id < 0 ? 0 : n_vocab - 1;
  }
  return id;
}

__global__ void __launch_bounds__(kRowThreads)
    embed_bf16(const int32_t* __restrict__ ids, const bf16* __restrict__ wte,
               const bf16* __restrict__ wpe, int rows, int T, int t_past, int d, int n_vocab,
               float* __restrict__ H, unsigned* err) {
  pdl_trigger();
  pdl_wait();
  const int row = blockIdx.x * kRowsPerBlock + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const int id = checked_id(ids, row, n_vocab, err);
  const int pos = t_past + row % T;
  const bf16* e = wte + static_cast<size_t>(id) * d;
  const bf16* p = wpe + static_cast<size_t>(pos) * d;
  float* h = H + static_cast<size_t>(row) * d;
  for (int c = lane * 8; c < d; c += 32 * 8) {  // d % 8 == 0
    const uint4 ev = *reinterpret_cast<const uint4*>(e + c);
    const uint4 pv = *reinterpret_cast<const uint4*>(p + c);
    const uint32_t ew[4] = {ev.x, ev.y, ev.z, ev.w};
    const uint32_t pw[4] = {pv.x, pv.y, pv.z, pv.w};
    float4 lo, hi;
    lo.x = bf16_lo(ew[0]) + bf16_lo(pw[0]);
    lo.y = bf16_hi(ew[0]) + bf16_hi(pw[0]);
    lo.z = bf16_lo(ew[1]) + bf16_lo(pw[1]);
    lo.w = bf16_hi(ew[1]) + bf16_hi(pw[1]);
    hi.x = bf16_lo(ew[2]) + bf16_lo(pw[2]);
    hi.y = bf16_hi(ew[2]) + bf16_hi(pw[2]);
    hi.z = bf16_lo(ew[3]) + bf16_lo(pw[3]);
    hi.w = bf16_hi(ew[3]) + bf16_hi(pw[3]);
    *reinterpret_cast<float4*>(h + c) = lo;
    *reinterpret_cast<float4*>(h + c + 4) = hi;
  }
}

__global__ void __launch_bounds__(kRowThreads)
    embed_fp32(const int32_t* __restrict__ ids, const float* __restrict__ wte,
               const float* __restrict__ wpe, int rows, int T, int t_past, int d, int n_vocab,
               float* __restrict__ H, unsigned* err) {
  pdl_trigger();
  pdl_wait();
  const int row = blockIdx.x * kRowsPerBlock + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const int id = checked_id(ids, row, n_vocab, err);
  const int pos = t_past + row % T;
  const float* e = wte + static_cast<size_t>(id) * d;
  const float* p = wpe + static_cast<size_t>(pos) * d;
  float* h = H + static_cast<size_t>(row) * d;
  for (int c = lane; c < d; c += 32) h[c] = e[c] + p[c];
}

// Index of the largest value of each row (the lowest index among equal
// values; NaN never wins).  One block per row.
__global__ void __launch_bounds__(kRowThreads)
    argmax_rows(const float* __restrict__ x, int V, long long row_stride, int32_t* __restrict__ out,
                long long out_stride, int32_t* __restrict__ next) {
  pdl_trigger();
  pdl_wait();
  const float* r = x + blockIdx.x * row_stride;
  float best = -INFINITY;
  int idx = V;  // no value seen yet
  for (int v = threadIdx.x; v < V; v += kRowThreads) {
    const float f = r[v];
    if (f > best || (idx == V && !(f != f))) {
      best = f;
      idx = v;
    }
  }
  // Reduce (value, index): larger value, then lower index.
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float ob = __shfl_xor_sync(0xffffffffu, best, off);
    const int oi = __shfl_xor_sync(0xffffffffu, idx, off);
    if (ob > best || (ob == best && oi < idx)) {
      best = ob;
      idx = oi;
    }
  }
  __shared__ float sb[kRowsPerBlock];
  __shared__ int si[kRowsPerBlock];
  const int w = threadIdx.x >> 5;
  if ((threadIdx.x & 31) == 0) {
    sb[w] = best;
    si[w] = idx;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int i = 1; i < kRowsPerBlock; ++i)
      if (sb[i] > best || (sb[i] == best && si[i] < idx)) {
        best = sb[i];
        idx = si[i];
      }
    const int id = idx < V ? idx : 0;  // a row of NaN only: token 0
    out[blockIdx.x * out_stride] = id;
    next[blockIdx.x] = id;
  }
}

// Next-token loss from the fused head's partials: 32 tokens per block (one per
// lane), kLossSlices warps each merging every kLossSlices-th vocabulary block
// (reads of 32 consecutive tokens' partials), then their results in shared
// memory.
constexpr int kLossSlices = 16;

__device__ __forceinline__ void lse_merge_rw(float& m, float& s, int& i, float m2, float s2,
                                             int i2) {
  const bool take = m2 > m || (m2 == m && i2 < i);
  const float hi = take ? m2 : m, lo = take ? m : m2;
  const float s_hi = take ? s2 : s, s_lo = take ? s : s2;
  i = take ? i2 : i;
  m = hi;
  s = s_hi + (lo == -INFINITY ? 0.f : s_lo * exp2f((lo - hi) * 1.4426950408889634f));
}

__global__ void __launch_bounds__(32 * kLossSlices)
    head_loss_combine(const float* __restrict__ pm, const float* __restrict__ ps,
                      const int32_t* __restrict__ pi, int n_vblk, int n_tok, int V,
                      const int32_t* __restrict__ tgt, const float* __restrict__ tl,
                      float* __restrict__ loss, int32_t* __restrict__ next, unsigned* err) {
  pdl_trigger();
  pdl_wait();
  __shared__ float sm[kLossSlices][32], ss[kLossSlices][32];
  __shared__ int si[kLossSlices][32];
  const int lane = threadIdx.x & 31, slice = threadIdx.x >> 5;
  const int t = blockIdx.x * 32 + lane;
  float m = -INFINITY, sum = 0.f;
  int idx = 0x7fffffff;
  if (t < n_tok) {
    for (int j = slice; j < n_vblk; j += kLossSlices) {
      const size_t o = static_cast<size_t>(j) * n_tok + t;
      lse_merge_rw(m, sum, idx, pm[o], ps[o], pi[o]);
    }
  }
  sm[slice][lane] = m;
  ss[slice][lane] = sum;
  si[slice][lane] = idx;
  __syncthreads();
  if (slice != 0 || t >= n_tok) return;
  for (int k = 1; k < kLossSlices; ++k) lse_merge_rw(m, sum, idx, sm[k][lane], ss[k][lane], si[k][lane]);
  if (next) next[t] = idx < V ? idx : 0;  // all logits NaN: token 0
  if (loss) {
    const int y = tgt ? tgt[t] : -1;
    if (y < 0) {
      loss[t] = 0.f;
    } else if (y >= V) {
      loss[t] = __int_as_float(0x7fc00000);  // NaN
      raise_error(err, kErrBadToken);
    } else {
      loss[t] = m + logf(sum) - tl[t];
    }
  }
}

// (v1, i1) ranks before (v2, i2): larger value, or equal value and lower index.
__device__ __forceinline__ bool topk_before(float v1, int i1, float v2, int i2) {
  return v1 > v2 || (v1 == v2 && i1 < i2);
}

// Inserts (v, i) into the sorted list tv / ti (descending by topk_before)
// when it ranks before the last entry: a branch-free network (the entries
// ranking before (v, i) keep their places, the others move down one).
__device__ __forceinline__ void topk_insert(float (&tv)[kTopKMax], int (&ti)[kTopKMax], float v,
                                            int i) {
  bool gt[kTopKMax];
#pragma unroll
  for (int j = 0; j < kTopKMax; ++j) gt[j] = topk_before(v, i, tv[j], ti[j]);
#pragma unroll
  for (int j = kTopKMax - 1; j > 0; --j) {
    tv[j] = gt[j] ? (gt[j - 1] ? tv[j - 1] : v) : tv[j];
    ti[j] = gt[j] ? (gt[j - 1] ? ti[j - 1] : i) : ti[j];
  }
  tv[0] = gt[0] ? v : tv[0];
  ti[0] = gt[0] ? i : ti[0];
}

// Top-k from the top-k head's partials: 32 tokens per block (one per lane),
// kLossSlices warps each merging every kLossSlices-th vocabulary block (the
// 32 consecutive tokens' candidate lists: 1 KB runs of values and of ids),
// then the warps' lists and logsumexp partials in shared memory.  A block's candidates are sorted, so the scan of
// a block stops at the first one that does not enter the list.
__global__ void __launch_bounds__(32 * kLossSlices)
    head_topk_combine(const float* __restrict__ pm, const float* __restrict__ ps,
                      const float* __restrict__ cv, const int32_t* __restrict__ ci, int n_vblk,
                      int n_tok, int k, float* __restrict__ top_v, int32_t* __restrict__ top_i,
                      float* __restrict__ lse) {
  pdl_trigger();
  pdl_wait();
  __shared__ float sv[kLossSlices][kTopKMax][32];
  __shared__ int si[kLossSlices][kTopKMax][32];
  __shared__ float sm[kLossSlices][32], ss[kLossSlices][32];
  const int lane = threadIdx.x & 31, slice = threadIdx.x >> 5;
  const int t = blockIdx.x * 32 + lane;
  float tv[kTopKMax];
  int ti[kTopKMax];
#pragma unroll
  for (int j = 0; j < kTopKMax; ++j) {
    tv[j] = -INFINITY;
    ti[j] = 0x7fffffff;
  }
  float m = -INFINITY, sum = 0.f;
  int dummy = 0;
  if (t < n_tok) {
    for (int b = slice; b < n_vblk; b += kLossSlices) {
      // All of the block's loads first (one round trip), then the merge.
      const size_t o = static_cast<size_t>(b) * n_tok + t;
      const float bm = pm[o], bs = ps[o];
      // The token's candidates: 32 contiguous bytes of values and of ids.
      static_assert(kTopKMax == 8, "two 16-byte loads per list");
      const float4* sv4 = reinterpret_cast<const float4*>(cv + o * kTopKMax);
      const int4* si4 = reinterpret_cast<const int4*>(ci + o * kTopKMax);
      const float4 v0 = sv4[0], v1 = sv4[1];
      const int4 i0 = si4[0], i1 = si4[1];
      float cvv[kTopKMax] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
      int cii[kTopKMax] = {i0.x, i0.y, i0.z, i0.w, i1.x, i1.y, i1.z, i1.w};
#pragma unroll
      for (int j = 0; j < kTopKMax; ++j) {
        cvv[j] = j < k ? cvv[j] : -INFINITY;
        cii[j] = j < k ? cii[j] : 0x7fffffff;
      }
      lse_merge_rw(m, sum, dummy, bm, bs, 0);
#pragma unroll
      for (int j = 0; j < kTopKMax; ++j) {
        if (!topk_before(cvv[j], cii[j], tv[kTopKMax - 1], ti[kTopKMax - 1])) break;
        topk_insert(tv, ti, cvv[j], cii[j]);
      }
    }
  }
#pragma unroll
  for (int j = 0; j < kTopKMax; ++j) {
    sv[slice][j][lane] = tv[j];
    si[slice][j][lane] = ti[j];
  }
  sm[slice][lane] = m;
  ss[slice][lane] = sum;
  __syncthreads();
  if (slice != 0 || t >= n_tok) return;
  for (int w = 1; w < kLossSlices; ++w) {
    lse_merge_rw(m, sum, dummy, sm[w][lane], ss[w][lane], 0);
    for (int j = 0; j < k; ++j) {
      const float v = sv[w][j][lane];
      const int id = si[w][j][lane];
      if (!topk_before(v, id, tv[kTopKMax - 1], ti[kTopKMax - 1])) break;
      topk_insert(tv, ti, v, id);
    }
  }
#pragma unroll
  for (int j = 0; j < kTopKMax; ++j) {
    if (j < k) {
      top_v[static_cast<size_t>(t) * k + j] = tv[j];
      top_i[static_cast<size_t>(t) * k + j] = ti[j] == 0x7fffffff ? -1 : ti[j];
    }
  }
  if (lse) lse[t] = m + logf(sum);
}

}  // namespace

int launch_head_topk_combine(const float* part_m, const float* part_s, const float* topk_v,
                             const int32_t* topk_i, int n_vblk, int n_tok, int k, float* top_v,
                             int32_t* top_i, float* lse, cudaStream_t stream) {
  if (n_vblk <= 0 || n_tok <= 0 || k < 1 || k > kTopKMax || !part_m || !part_s || !topk_v ||
      !topk_i || !top_v || !top_i)
    return GPT2_ERR_INVALID_ARG;
  const cudaError_t e =
      launch_pdl(head_topk_combine, dim3((n_tok + 31) / 32), dim3(32 * kLossSlices), 0, stream,
                 part_m, part_s, topk_v, topk_i, n_vblk, n_tok, k, top_v, top_i, lse);
  return e == cudaSuccess ? GPT2_OK : GPT2_ERR_CUDA;
}

int launch_head_loss_combine(const float* part_m, const float* part_s, const int32_t* part_i,
                             int n_vblk, int n_tok, int V, const int32_t* tgt,
                             const float* tgt_logit, float* loss, int32_t* next, unsigned* err,
                             cudaStream_t stream) {
  if (n_vblk <= 0 || n_tok <= 0 || V <= 0 || !part_m || !part_s || !part_i)
    return GPT2_ERR_INVALID_ARG;
  const cudaError_t e =
      launch_pdl(head_loss_combine, dim3((n_tok + 31) / 32), dim3(32 * kLossSlices), 0, stream,
                 part_m, part_s, part_i, n_vblk, n_tok, V, tgt, tgt_logit, loss, next, err);
  return e == cudaSuccess ? GPT2_OK : GPT2_ERR_CUDA;
}

int launch_layer_norm(int mode, const void* x, int x_dtype, const void* g, const void* b, int rows,
                      int d, void* y, cudaStream_t stream, bool y_f16, const ConvSegs* side,
                      unsigned* err) {
  if (rows <= 0 || d <= 0) return GPT2_ERR_INVALID_ARG;
  if (side && (side->count < 0 || side->count > kMaxConvSegs)) return GPT2_ERR_INVALID_ARG;
  const ConvJob job = make_conv_job(side, err);
  if (mode == GPT2_BF16) {
    if (d % 2 != 0) return GPT2_ERR_UNSUPPORTED;
    const bf16* gg = static_cast<const bf16*>(g);
    const bf16* bb = static_cast<const bf16*>(b);
    if (x_dtype == GPT2_FP32) {
      const float* xx = static_cast<const float*>(x);
      return y_f16 ? ln_dispatch(xx, gg, bb, rows, d, static_cast<__half*>(y), stream, job)
                   : ln_dispatch(xx, gg, bb, rows, d, static_cast<bf16*>(y), stream, job);
    }
    if (x_dtype == GPT2_BF16) {
      const bf16* xx = static_cast<const bf16*>(x);
      return y_f16 ? ln_dispatch(xx, gg, bb, rows, d, static_cast<__half*>(y), stream, job)
                   : ln_dispatch(xx, gg, bb, rows, d, static_cast<bf16*>(y), stream, job);
    }
    return GPT2_ERR_INVALID_ARG;
  }
  if (mode == GPT2_FP32 && x_dtype == GPT2_FP32)
    return ln_dispatch(static_cast<const float*>(x), static_cast<const float*>(g),
                       static_cast<const float*>(b), rows, d, static_cast<float*>(y), stream, job);
  return GPT2_ERR_INVALID_ARG;
}

int launch_argmax_rows(const float* x, int rows, int V, long long row_stride, int32_t* out,
                       long long out_stride, int32_t* next, cudaStream_t stream) {
  if (rows <= 0 || V <= 0) return GPT2_ERR_INVALID_ARG;
  const cudaError_t e = launch_pdl(argmax_rows, dim3(rows), dim3(kRowThreads), 0, stream, x, V,
                                   row_stride, out, out_stride, next);
  return e == cudaSuccess ? GPT2_OK : GPT2_ERR_CUDA;
}

int launch_embed(int mode, const int32_t* ids, const void* wte, const void* wpe, int B, int T,
                 int t_past, int d, int n_vocab, float* H, unsigned* err, cudaStream_t stream) {
  if (B <= 0 || T <= 0 || d <= 0 || n_vocab <= 0) return GPT2_ERR_INVALID_ARG;
  const int rows = B * T;
  const unsigned blocks = static_cast<unsigned>((rows + kRowsPerBlock - 1) / kRowsPerBlock);
  if (mode == GPT2_BF16) {
    if (d % 8 != 0) return GPT2_ERR_UNSUPPORTED;
    if (launch_pdl(embed_bf16, dim3(blocks), dim3(kRowThreads), 0, stream, ids,
                   static_cast<const bf16*>(wte), static_cast<const bf16*>(wpe), rows, T, t_past,
                   d, n_vocab, H, err) != cudaSuccess)
      return GPT2_ERR_CUDA;
  } else {
    if (launch_pdl(embed_fp32, dim3(blocks), dim3(kRowThreads), 0, stream, ids,
                   static_cast<const float*>(wte), static_cast<const float*>(wpe), rows, T,
                   t_past, d, n_vocab, H, err) != cudaSuccess)
      return GPT2_ERR_CUDA;
  }
  return cudaGetLastError() == cudaSuccess ? GPT2_OK : GPT2_ERR_CUDA;
}

}  // namespace gpt2

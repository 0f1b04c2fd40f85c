// attention.cu -- causal multi-head attention kernels.
//
// Computes, per sequence b and head, o_i = sum_{j <= p_i} softmax_j(q_i . k_j /
// sqrt(d_h)) v_j with p_i = T_past + i the query's absolute position ("GPT-2
// Block - TorchCode", "Reference Solution": scores, upper-triangular -inf
// mask, softmax over keys, weights @ v; "GPT-2 Full Forward Pass", "How it
// works": cached keys/values come first on the sequence axis).  Keys and
// values are read from the KV cache the c_attn epilogue wrote; the output is
// written with heads merged, [B, T, h * d_h].
//
//   (causal prefill on the tcgen05 tensor cores is in attn_tc.cu)
//   attn_decode_bf16    one new token: split over keys (when there are few
//                       sequence x head pairs), one CTA per (pair, split); the
//                       split's key and value rows, contiguous in the cache,
//                       stream into a 3-stage shared-memory ring by 64-row bulk
//                       copies; 8 warps, each 8-lane group scoring one key at
//                       a time with online softmax; partial (max, sum, o)
//                       merged across groups by shuffles, across warps in
//                       shared memory, and across CTAs by attn_decode_combine.
//   attn_fp32           fp32 storage, any d_h <= 256, one warp per query.
#include <math.h>

#include <algorithm>

#include "device.cuh"
#include "internal.h"

namespace gpt2 {

namespace {

constexpr int kDh = 64;
constexpr float kLog2e = 1.4426950408889634f;

constexpr int kDecThreads = 256;
constexpr int kDecWarps = kDecThreads / 32;
constexpr int kPartialStride = kDh + 2;  // o[64], m, l

constexpr int kDecStageKeys = 64;                        // keys per stage
constexpr int kDecStages = 3;                           // four CTAs of 50 KB fit on an SM
constexpr uint32_t kDecRowBytes = kDh * 2;               // one key (or value) row: 128 B
constexpr size_t kDecSmem = 2 * kDecStages * kDecStageKeys * kDecRowBytes + 64;

__global__ void __launch_bounds__(kDecThreads)
    attn_decode_bf16(const bf16* __restrict__ q, const bf16* __restrict__ kv, long long s_batch,
                     long long s_kv, long long s_head, int h, int t_len, int chunk,
                     uint16_t* __restrict__ out, float* __restrict__ partials, int out_f16,
                     unsigned* err, unsigned long long wait_ns) {
  extern __shared__ __align__(128) uint8_t dsm[];
  uint8_t* sK = dsm;                                             // [stages][64 rows]
  uint8_t* sV = dsm + kDecStages * kDecStageKeys * kDecRowBytes;  // [stages][64 rows]
  uint64_t* full = reinterpret_cast<uint64_t*>(sV + kDecStages * kDecStageKeys * kDecRowBytes);
  __shared__ float s_m[kDecWarps], s_l[kDecWarps];
  __shared__ float s_o[kDecWarps][kDh];
  __shared__ int s_abort;

  const int split = blockIdx.x, splits = gridDim.x;
  const int bh = blockIdx.y;
  const int b = bh / h, head = bh - b * h;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int grp = lane >> 3, sub = lane & 7;  // 4 groups of 8 lanes; 8 dims per lane

  const int k_begin = split * chunk;
  const int k_end = min(t_len, k_begin + chunk);
  const int n_keys = max(0, k_end - k_begin);
  const int ns = (n_keys + kDecStageKeys - 1) / kDecStageKeys;

  if (tid == 0) {
    for (int i = 0; i < kDecStages; ++i) mbar_init(&full[i], 1);
    s_abort = 0;
    fence_mbar_init();
  }
  __syncthreads();
  pdl_trigger();
  pdl_wait();

  // The split's keys of this head are one contiguous run of 128-byte rows in
  // the cache (K, and V s_kv further on): each stage is one bulk copy of up
  // to 64 rows of each, issued by thread 0.
  const bf16* Kg = kv + b * s_batch + head * s_head + static_cast<size_t>(k_begin) * kDh;
  const bf16* Vg = Kg + s_kv;
  auto issue = [&](int j) {
    const int slot = j % kDecStages;
    const int nk = min(kDecStageKeys, n_keys - j * kDecStageKeys);
    const uint32_t bytes = static_cast<uint32_t>(nk) * kDecRowBytes;
    mbar_arrive_expect_tx(&full[slot], 2 * bytes);
    bulk_load(sK + slot * kDecStageKeys * kDecRowBytes,
              Kg + static_cast<size_t>(j) * kDecStageKeys * kDh, bytes, &full[slot]);
    bulk_load(sV + slot * kDecStageKeys * kDecRowBytes,
              Vg + static_cast<size_t>(j) * kDecStageKeys * kDh, bytes, &full[slot]);
  };
  int issued = 0;
  if (tid == 0)
    for (; issued < min(ns, kDecStages); ++issued) issue(issued);

  const float sl2 = 0.125f * kLog2e;
  float qv[8];
  {
    const uint4 qq = *reinterpret_cast<const uint4*>(q + static_cast<size_t>(bh) * kDh + sub * 8);
    const uint32_t w[4] = {qq.x, qq.y, qq.z, qq.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      qv[2 * i] = bf16_lo(w[i]) * sl2;
      qv[2 * i + 1] = bf16_hi(w[i]) * sl2;
    }
  }
  float m = -INFINITY, l = 0.f, o[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) o[i] = 0.f;

  // Stage j: warp w takes keys 8w .. 8w+7 of the stage, group g keys 8w+2g
  // and 8w+2g+1, each key read by its 8 lanes (16 bytes each).
  int j = 0;
  for (; j < ns; ++j) {
    const int slot = j % kDecStages;
    const bool got = mbar_wait_bounded(&full[slot], static_cast<uint32_t>(j / kDecStages) & 1u,
                                       &s_abort, err, wait_ns);
    if (got) {
      const int nk = min(kDecStageKeys, n_keys - j * kDecStageKeys);
      const uint8_t* kb = sK + slot * kDecStageKeys * kDecRowBytes;
      const uint8_t* vb = sV + slot * kDecStageKeys * kDecRowBytes;
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int key = warp * 8 + grp * 2 + u;
        const bool ok = key < nk;
        const int kr = ok ? key : 0;
        const uint4 kw4 = *reinterpret_cast<const uint4*>(kb + kr * kDecRowBytes + sub * 16);
        const uint32_t kw[4] = {kw4.x, kw4.y, kw4.z, kw4.w};
        float sc = 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          sc = fmaf(qv[2 * i], bf16_lo(kw[i]), sc);
          sc = fmaf(qv[2 * i + 1], bf16_hi(kw[i]), sc);
        }
        sc += __shfl_xor_sync(0xffffffffu, sc, 1);
        sc += __shfl_xor_sync(0xffffffffu, sc, 2);
        sc += __shfl_xor_sync(0xffffffffu, sc, 4);
        if (!ok) continue;
        const float mn = fmaxf(m, sc);
        const float alpha = ex2(m - mn);
        const float p = ex2(sc - mn);
        m = mn;
        l = l * alpha + p;
        const uint4 vw4 = *reinterpret_cast<const uint4*>(vb + kr * kDecRowBytes + sub * 16);
        const uint32_t vw[4] = {vw4.x, vw4.y, vw4.z, vw4.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          o[2 * i] = fmaf(p, bf16_lo(vw[i]), o[2 * i] * alpha);
          o[2 * i + 1] = fmaf(p, bf16_hi(vw[i]), o[2 * i + 1] * alpha);
        }
      }
    }
    // Every thread agrees on going on; then the stage's slot is refilled.
    if (!__syncthreads_and(got)) break;
    if (tid == 0 && issued < ns) issue(issued++);
  }
  if (j < ns) {
    // A wait ran out: the copies still in flight must land before the CTA
    // exits, and this (sequence, head)'s result becomes NaN (its output row,
    // or this split's partial, which makes the combined row NaN), so that a
    // caller without the error word cannot mistake stale memory for a result.
    if (tid == 0)
      for (int k = j; k < issued; ++k)
        mbar_wait_bounded(&full[k % kDecStages], static_cast<uint32_t>(k / kDecStages) & 1u,
                          nullptr, err);
    if (warp == 0) {
      const float nan = __int_as_float(0x7fc00000);
      if (splits == 1) {
        *reinterpret_cast<uint32_t*>(out + static_cast<size_t>(bh) * kDh + 2 * lane) =
            pack_16x2(nan, nan, out_f16 != 0);
      } else {
        float* pp = partials + (static_cast<size_t>(bh) * splits + split) * kPartialStride;
        pp[2 * lane] = nan;
        pp[2 * lane + 1] = nan;
        if (lane == 0) {
          pp[kDh] = nan;
          pp[kDh + 1] = nan;
        }
      }
    }
    return;
  }
  // Merge the four key groups of the warp (lanes sub, sub+8, sub+16, sub+24).
#pragma unroll
  for (int off = 8; off < 32; off <<= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, off);
    const float l2 = __shfl_xor_sync(0xffffffffu, l, off);
    const float mn = fmaxf(m, m2);
    const float a1 = (m == -INFINITY) ? 0.f : ex2(m - mn);
    const float a2 = (m2 == -INFINITY) ? 0.f : ex2(m2 - mn);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float o2 = __shfl_xor_sync(0xffffffffu, o[i], off);
      o[i] = o[i] * a1 + o2 * a2;
    }
    l = l * a1 + l2 * a2;
    m = mn;
  }
  if (grp == 0) {
#pragma unroll
    for (int i = 0; i < 8; ++i) s_o[warp][sub * 8 + i] = o[i];
    if (sub == 0) {
      s_m[warp] = m;
      s_l[warp] = l;
    }
  }
  __syncthreads();
  if (warp == 0) {
    // Lane t owns dims 2t, 2t+1.
    float mx = -INFINITY;
#pragma unroll
    for (int w = 0; w < kDecWarps; ++w) mx = fmaxf(mx, s_m[w]);
    float lsum = 0.f, o0 = 0.f, o1 = 0.f;
#pragma unroll
    for (int w = 0; w < kDecWarps; ++w) {
      const float a = (s_m[w] == -INFINITY) ? 0.f : ex2(s_m[w] - mx);
      lsum += s_l[w] * a;
      o0 += s_o[w][2 * lane] * a;
      o1 += s_o[w][2 * lane + 1] * a;
    }
    if (splits == 1) {
      const float inv = 1.f / lsum;
      *reinterpret_cast<uint32_t*>(out + static_cast<size_t>(bh) * kDh + 2 * lane) =
          pack_16x2(o0 * inv, o1 * inv, out_f16 != 0);
    } else {
      float* pp = partials + (static_cast<size_t>(bh) * splits + split) * kPartialStride;
      pp[2 * lane] = o0;
      pp[2 * lane + 1] = o1;
      if (lane == 0) {
        pp[kDh] = mx;
        pp[kDh + 1] = lsum;
      }
    }
  }
}

// One warp per (sequence, head): merges the splits' partial results.
__global__ void attn_decode_combine(const float* __restrict__ partials, int n_bh, int splits,
                                    uint16_t* __restrict__ out, int out_f16) {
  pdl_trigger();
  pdl_wait();
  const int bh = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (bh >= n_bh) return;
  const float* pp = partials + static_cast<size_t>(bh) * splits * kPartialStride;
  float mx = -INFINITY;
  for (int s = 0; s < splits; ++s) mx = fmaxf(mx, pp[s * kPartialStride + kDh]);
  float lsum = 0.f, o0 = 0.f, o1 = 0.f;
  for (int s = 0; s < splits; ++s) {
    const float ms = pp[s * kPartialStride + kDh];
    const float a = (ms == -INFINITY) ? 0.f : ex2(ms - mx);
    lsum += pp[s * kPartialStride + kDh + 1] * a;
    o0 += pp[s * kPartialStride + 2 * lane] * a;
    o1 += pp[s * kPartialStride + 2 * lane + 1] * a;
  }
  const float inv = 1.f / lsum;
  *reinterpret_cast<uint32_t*>(out + static_cast<size_t>(bh) * kDh + 2 * lane) =
      pack_16x2(o0 * inv, o1 * inv, out_f16 != 0);
}

// -------------------------------------------------------------------- fp32 --
constexpr int kF32MaxPerLane = 8;  // d_h <= 256

__global__ void attn_fp32(const float* __restrict__ q, const float* __restrict__ kv,
                          long long s_batch, long long s_kv, long long s_head, int B, int h,
                          int T, int t_past, int dh, float* __restrict__ out) {
  pdl_trigger();
  pdl_wait();
  const int row = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);  // (b, head, i)
  const int lane = threadIdx.x & 31;
  if (row >= B * h * T) return;
  const int i = row % T;
  const int bh = row / T;
  const int b = bh / h, head = bh - b * h;
  const float* qr = q + static_cast<size_t>(row) * dh;
  const float* Kg = kv + b * s_batch + head * s_head;
  const float* Vg = Kg + s_kv;
  const float scale = 1.0f / sqrtf(static_cast<float>(dh));
  float qv[kF32MaxPerLane], o[kF32MaxPerLane];
#pragma unroll
  for (int u = 0; u < kF32MaxPerLane; ++u) {
    const int c = lane + 32 * u;
    qv[u] = c < dh ? qr[c] : 0.f;
    o[u] = 0.f;
  }
  float m = -INFINITY, l = 0.f;
  const int p = t_past + i;
  for (int j = 0; j <= p; ++j) {
    float sc = 0.f;
#pragma unroll
    for (int u = 0; u < kF32MaxPerLane; ++u) {
      const int c = lane + 32 * u;
      if (c < dh) sc = fmaf(qv[u], Kg[static_cast<size_t>(j) * dh + c], sc);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) sc += __shfl_xor_sync(0xffffffffu, sc, off);
    sc *= scale;
    const float mn = fmaxf(m, sc);
    const float alpha = expf(m - mn);
    const float pj = expf(sc - mn);
    l = l * alpha + pj;
#pragma unroll
    for (int u = 0; u < kF32MaxPerLane; ++u) {
      const int c = lane + 32 * u;
      if (c < dh) o[u] = o[u] * alpha + pj * Vg[static_cast<size_t>(j) * dh + c];
    }
    m = mn;
  }
  const int d = h * dh;
  float* orow = out + (static_cast<size_t>(b) * T + i) * d + head * dh;
#pragma unroll
  for (int u = 0; u < kF32MaxPerLane; ++u) {
    const int c = lane + 32 * u;
    if (c < dh) orow[c] = o[u] / l;
  }
}

}  // namespace

size_t decode_partials_floats(int B, int h, int splits) {
  return static_cast<size_t>(B) * h * splits * kPartialStride;
}

int decode_splits(int B, int h, int t_len, int num_sms) {
  const int bh = B * h;
  int splits = (2 * num_sms + bh - 1) / bh;         // about two CTAs per SM
  splits = std::min(splits, (t_len + 255) / 256);   // at least 256 keys per split
  return std::max(1, std::min(splits, 64));
}

int launch_decode_attention_bf16(const bf16* q, const bf16* kv, long long s_batch, long long s_kv,
                                 long long s_head, int B, int h, int t_len, void* out,
                                 float* partials, int splits, cudaStream_t stream,
                                 int* launches, bool out_f16, unsigned* err,
                                 unsigned long long wait_ns) {
  if (B <= 0 || h <= 0 || t_len <= 0 || splits <= 0 || splits > 65535) return GPT2_ERR_INVALID_ARG;
  if (static_cast<long long>(B) * h > 65535) return GPT2_ERR_UNSUPPORTED;  // grid.y
  if (splits > 1 && partials == nullptr) return GPT2_ERR_INVALID_ARG;
  const int chunk = (t_len + splits - 1) / splits;
  dim3 grid(splits, B * h);
  if (!ensure_smem_limit(reinterpret_cast<const void*>(&attn_decode_bf16),
                         static_cast<int>(kDecSmem)))
    return GPT2_ERR_CUDA;
  cudaError_t e = launch_pdl(attn_decode_bf16, grid, dim3(kDecThreads), kDecSmem, stream, q, kv,
                             s_batch, s_kv, s_head, h, t_len, chunk, static_cast<uint16_t*>(out),
                             partials, out_f16 ? 1 : 0, err, wait_ns ? wait_ns : kWaitLimitNs);
  if (e != cudaSuccess) return GPT2_ERR_CUDA;
  int n = 1;
  if (splits > 1) {
    const int n_bh = B * h;
    e = launch_pdl(attn_decode_combine, dim3((n_bh + 7) / 8), dim3(256), 0, stream,
                   static_cast<const float*>(partials), n_bh, splits,
                   static_cast<uint16_t*>(out), out_f16 ? 1 : 0);
    if (e != cudaSuccess) return GPT2_ERR_CUDA;
    ++n;
  }
  if (launches) *launches = n;
  return cudaGetLastError() == cudaSuccess ? GPT2_OK : GPT2_ERR_CUDA;
}

int launch_attention_fp32(const float* q, const float* kv, long long s_batch, long long s_kv,
                          long long s_head, int B, int h, int T, int t_past, int d_h, float* out,
                          cudaStream_t stream) {
  if (B <= 0 || h <= 0 || T <= 0 || t_past < 0 || d_h <= 0 || d_h > 32 * kF32MaxPerLane)
    return GPT2_ERR_INVALID_ARG;
  const long long rows = static_cast<long long>(B) * h * T;
  const int warps_per_block = 8;
  const long long blocks = (rows + warps_per_block - 1) / warps_per_block;
  if (blocks > 0x7fffffffLL) return GPT2_ERR_UNSUPPORTED;
  const cudaError_t e = launch_pdl(attn_fp32, dim3(static_cast<unsigned>(blocks)),
                                   dim3(32 * warps_per_block), 0, stream, q, kv, s_batch, s_kv,
                                   s_head, B, h, T, t_past, d_h, out);
  return e == cudaSuccess ? GPT2_OK : GPT2_ERR_CUDA;
}

}  // namespace gpt2

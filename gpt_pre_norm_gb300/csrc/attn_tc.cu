// attn_tc.cu -- causal prefill attention on the tcgen05 tensor cores, d_h = 64.
//
// Per sequence b, head and query i (absolute position p_i = T_past + i):
// o_i = sum_{j <= p_i} softmax_j(q_i . k_j / sqrt(64)) v_j ("GPT-2 Block -
// TorchCode", "Reference Solution": scores, upper-triangular mask, softmax
// over keys, weights @ v; "GPT-2 Full Forward Pass", "How it works": cached
// keys and values come first on the sequence axis).  Q is [B, h, T, 64]; K and
// V are read from the KV cache ([.., T_cap, 64] rows per head) and the output
// goes to [B, T, h * 64] with the heads merged.
//
// One CTA per (sequence x head, 128-query tile), 6 warps, two CTAs per SM:
//   warp 0      TMA: the Q tile once, then the 64-key K and V tiles of each
//               step into separate rings (128-byte swizzle): a K stage is
//               free again once its scores are computed, a V stage only
//               after its P V product, so K runs further ahead.  One thread
//               polls both rings and issues whichever copy is possible.  The
//               rings are as deep as two CTAs per SM allow (P lives in TMEM,
//               not in shared memory): a copy takes microseconds when the
//               memory system is busy, and the steps in flight must cover it.
//   warp 1      allocates 256 TMEM columns; one thread issues
//                 S_j = Q K_j^T  (M=128, N=64, K=64; K-major operands)
//               into one of two TMEM score buffers, one step ahead, and
//                 O += P_j V_j  (M=128, N=64, K=64; P from TMEM,
//                                V used as stored, [key][dim]: MN-major B)
//               into one TMEM output accumulator.
//   warps 2-5   one query row per thread: S_j from TMEM, causal mask on the
//               steps that cross the diagonal, row maximum, P = 2^(s - m)
//               in bf16 to one of two TMEM buffers (the next product's A).
//               The reference maximum m of the online softmax moves only
//               when a row's maximum passes it by more than 2^8: P then
//               stays below 256 (no overflow in bf16 or in the fp32 sums),
//               and the rescale of O and l by 2^(m_old - m_new) is rare; when
//               a warp needs one, it waits for the last product and rescales
//               its rows of O in TMEM.  At the end o / l is written through
//               shared memory by a TMA store.
// Steps entirely above the diagonal are never loaded; the query tiles with
// the most keys start first.  Every wait on an mbarrier is bounded: one that
// runs out raises the error word, and the CTA drains its copies and MMAs,
// frees TMEM and returns.
#include <math.h>
#include <string.h>

#include <algorithm>

#include "device.cuh"
#include "internal.h"

namespace gpt2 {

namespace {

constexpr int kD = 64;
constexpr int kQT = 128;                        // queries per CTA
constexpr int kKT = 64;                         // keys per step
constexpr int kSK = 5;                          // K ring
constexpr int kSV = 6;                          // V ring
constexpr int kThreads = 192;
constexpr uint32_t kQBytes = kQT * kD * 2;      // 16 KB
constexpr uint32_t kKVBytes = kKT * kD * 2;     // 8 KB: one K or V tile
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kColS = 0;                   // two score buffers of 64 columns (fp32)
constexpr uint32_t kColP = 128;                 // two P buffers of 32 columns (bf16 pairs)
constexpr uint32_t kColO = 192;                 // the output accumulator, 64 columns
constexpr float kRescaleLog2 = 8.f;             // max. lag of the reference maximum (log2)
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kBars = 1 + 2 * kSK + 2 * kSV + 3 * 2 + 1;
constexpr size_t kSmemBytes =
    1024 + kQBytes + (kSK + kSV) * kKVBytes + kBars * 8 + 16;
static_assert(2 * (kSmemBytes + 1024) <= 233472, "two CTAs per SM");

struct AttnArgs {
  int T, t_past, h, n_qtiles;
  int out_f16;  // output fp16 (else bf16)
  unsigned* err;
};

__global__ void __launch_bounds__(kThreads, 2)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                   const AttnArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = sm;
  uint8_t* sK = sQ + kQBytes;                  // [kSK][8 KB]
  uint8_t* sV = sK + kSK * kKVBytes;           // [kSV][8 KB]
  uint64_t* q_full = reinterpret_cast<uint64_t*>(sV + kSV * kKVBytes);
  uint64_t* k_full = q_full + 1;               // [kSK] K landed
  uint64_t* k_empty = k_full + kSK;            // [kSK] its scores computed
  uint64_t* v_full = k_empty + kSK;            // [kSV] V landed
  uint64_t* v_empty = v_full + kSV;            // [kSV] its P V product done
  // A softmax warp reads S_j before it publishes P_j, so P_j published by
  // all four warps also means that S_j's buffer (next used by S_{j+2}) has
  // been read, and that any rescale of O for step j is done.
  uint64_t* s_full = v_empty + kSV;            // [2] scores ready
  uint64_t* p_full = s_full + 2;               // [2] P written, O rescaled (4 warps)
  uint64_t* pv_done = p_full + 2;              // [2] P_j V_j done (P_j's buffer read, O updated)
  uint64_t* mma_done = pv_done + 2;            // [1]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bh = blockIdx.x;
  const int qt = a.n_qtiles - 1 - static_cast<int>(blockIdx.y);  // most keys first
  const int b = bh / a.h, head = bh - b * a.h;
  const int q0 = qt * kQT;
  const int q_last = min(q0 + kQT, a.T) - 1;
  const int n_kt = (a.t_past + q_last + 1 + kKT - 1) / kKT;  // steps up to the last query

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < kSK; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
    }
    for (int s = 0; s < kSV; ++s) {
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], 4);
      mbar_init(&pv_done[i], 1);
    }
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_trigger();
  pdl_wait();

  if (warp == 0 && lane == 0) {
    // ---------------------------------------------------------- producer --
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    mbar_arrive_expect_tx(q_full, kQBytes);
    tma_load_3d(sQ, &tmQ, q_full, 0, q0, bh);
    // Next K and V steps to load; a stage is free once the product that read
    // its previous tile has completed (no wait for the first pass).
    int kj = 0, vj = 0;
    bool ok = true;
    unsigned long long t_idle = 0;
    while (kj < n_kt || vj < n_kt) {
      bool progress = false;
      if (kj < n_kt && (kj < kSK || mbar_test_wait(&k_empty[kj % kSK],
                                                   static_cast<uint32_t>(kj / kSK - 1) & 1u))) {
        const int s = kj % kSK;
        mbar_arrive_expect_tx(&k_full[s], kKVBytes);
        tma_load_4d(sK + s * kKVBytes, &tmK, &k_full[s], 0, kj * kKT, head, b);
        ++kj;
        progress = true;
      }
      if (vj < n_kt && (vj < kSV || mbar_test_wait(&v_empty[vj % kSV],
                                                   static_cast<uint32_t>(vj / kSV - 1) & 1u))) {
        const int s = vj % kSV;
        mbar_arrive_expect_tx(&v_full[s], kKVBytes);
        tma_load_4d(sV + s * kKVBytes, &tmV, &v_full[s], 0, vj * kKT, head, b);
        ++vj;
        progress = true;
      }
      if (progress) {
        t_idle = 0;
      } else {
        // Neither ring has a free stage: the same bounded wait as elsewhere.
        __nanosleep(32);
        const unsigned long long now = global_timer_ns();
        if (t_idle == 0) {
          t_idle = now;
        } else if (*abort_flag || now - t_idle > kWaitLimitNs) {
          if (!*abort_flag) raise_error(a.err, kErrTimeout);
          *abort_flag = 1;
          ok = false;
          break;
        }
      }
    }
    if (!ok) {
      // Drain: every copy already issued must land before the CTA exits.
      mbar_wait_bounded(q_full, 0, nullptr, a.err);
      for (int j = max(0, kj - kSK); j < kj; ++j)
        mbar_wait_bounded(&k_full[j % kSK], static_cast<uint32_t>(j / kSK) & 1u, nullptr, a.err);
      for (int j = max(0, vj - kSV); j < vj; ++j)
        mbar_wait_bounded(&v_full[j % kSV], static_cast<uint32_t>(j / kSV) & 1u, nullptr, a.err);
    }
  } else if (warp == 1 && lane == 0) {
    // ------------------------------------------------------- MMA issuer --
    const uint32_t id_s = umma_idesc_16(kQT, kKT, false, false);
    const uint32_t id_pv = umma_idesc_16(kQT, kD, false, true);
    const uint64_t q_desc = sdesc_k_sw128(smem_u32(sQ));
    bool ok = mbar_wait_bounded(q_full, 0, abort_flag, a.err);
    auto issue_s = [&](int j) -> bool {
      const int s = j % kSK, sb = j & 1;
      // S_{j-2}, the buffer's previous tile, was read before P_{j-2} was
      // published, which this thread has already waited for.
      if (!mbar_wait_bounded(&k_full[s], static_cast<uint32_t>(j / kSK) & 1u, abort_flag, a.err))
        return false;
      tc_fence_after();
      const uint64_t k_desc = sdesc_k_sw128(smem_u32(sK + s * kKVBytes));
      const uint32_t d = tmem + kColS + sb * 64;
#pragma unroll
      for (int k = 0; k < kD / 16; ++k)
        umma_f16kind(d, q_desc + 2 * k, k_desc + 2 * k, id_s, k != 0 ? 1u : 0u);
      umma_commit(&s_full[sb]);
      umma_commit(&k_empty[s]);
      return true;
    };
    if (ok) ok = issue_s(0);
    for (int j = 0; ok && j < n_kt; ++j) {
      if (j + 1 < n_kt && !(ok = issue_s(j + 1))) break;
      const int pb = j & 1, s = j % kSV;
      if (!mbar_wait_bounded(&v_full[s], static_cast<uint32_t>(j / kSV) & 1u, abort_flag, a.err) ||
          !mbar_wait_bounded(&p_full[pb], static_cast<uint32_t>(j >> 1) & 1u, abort_flag, a.err)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t p_tmem = tmem + kColP + pb * 32;
      const uint64_t v_desc = sdesc_mn_sw128(smem_u32(sV + s * kKVBytes));
      const uint32_t d = tmem + kColO;
#pragma unroll
      for (int k = 0; k < kKT / 16; ++k)  // 16 keys: +8 columns of P, +2048 B in V
        umma_f16kind_ts(d, p_tmem + 8 * k, v_desc + 128 * k, id_pv, (j | k) != 0 ? 1u : 0u);
      umma_commit(&pv_done[pb]);
      umma_commit(&v_empty[s]);
    }
    // Every MMA issued above must retire before TMEM is freed.
    umma_commit(mma_done);
    mbar_wait_bounded(mma_done, 0, nullptr, a.err);
  } else if (warp >= 2) {
    // ---------------------------------------------------------- softmax --
    const int quarter = warp & 3;                // TMEM lanes 32 * quarter ..
    const int r = quarter * 32 + lane;           // query row in the tile
    const int pos = a.t_past + q0 + r;           // its absolute position
    const uint32_t trow = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const float sl2 = 0.125f * kLog2e;           // 1/sqrt(64), in log2 units
    float m = -INFINITY, l = 0.f;                // reference maximum (log2 units), row sum
    bool ok = true;
    // The product P_t V_t has completed (pv_done of step t; never more than
    // one phase behind when waited for).
    auto wait_pv = [&](int t) -> bool {
      return mbar_wait_bounded(&pv_done[t & 1], static_cast<uint32_t>(t >> 1) & 1u, abort_flag,
                               a.err);
    };

    for (int j = 0; j < n_kt; ++j) {
      const int sb = j & 1;
      if (!mbar_wait_bounded(&s_full[sb], static_cast<uint32_t>(j >> 1) & 1u, abort_flag, a.err)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t sr[kKT];
      tmem_ld_32x32b_x32(trow + kColS + sb * 64, *reinterpret_cast<uint32_t(*)[32]>(sr));
      tmem_ld_32x32b_x32(trow + kColS + sb * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(sr + 32));
      tmem_ld_wait();

      // Raw scores; the 1/sqrt(64) scale (in log2 units) is applied to the
      // row maximum and inside the exponent's fused multiply-add.
      const int key0 = j * kKT;
      float mx = -INFINITY;
      if (key0 + kKT - 1 > pos) {                 // this step crosses the row's diagonal
#pragma unroll
        for (int c = 0; c < kKT; ++c) {
          const float x = key0 + c <= pos ? __uint_as_float(sr[c]) : -INFINITY;
          sr[c] = __float_as_uint(x);
          mx = fmaxf(mx, x);
        }
      } else {
#pragma unroll
        for (int c = 0; c < kKT; ++c) mx = fmaxf(mx, __uint_as_float(sr[c]));
      }
      // A new reference maximum only when this row's passed it by more than
      // kRescaleLog2 (always on the row's first key); O and l scale by
      // 2^(m_old - m_new) (0 while m_old = -inf).
      const float m_row = mx * sl2;
      const bool bump = m_row > m + kRescaleLog2;
      const float alpha = bump ? ex2(m - m_row) : 1.f;
      if (bump) m = m_row;
      l *= alpha;
      if (j > 0 && __any_sync(0xffffffffu, bump)) {
        // O holds P_0 V_0 + .. + P_{j-1} V_{j-1}: wait for the last product,
        // then rescale this warp's 32 rows in place (alpha = 1 elsewhere).
        if (!(ok = wait_pv(j - 1))) break;
        tc_fence_after();
        uint32_t ov[kD];
        tmem_ld_32x32b_x32(trow + kColO, *reinterpret_cast<uint32_t(*)[32]>(ov));
        tmem_ld_32x32b_x32(trow + kColO + 32, *reinterpret_cast<uint32_t(*)[32]>(ov + 32));
        tmem_ld_wait();
#pragma unroll
        for (int c = 0; c < kD; ++c) ov[c] = __float_as_uint(__uint_as_float(ov[c]) * alpha);
        tmem_st_32x32b_x32(trow + kColO, *reinterpret_cast<uint32_t(*)[32]>(ov));
        tmem_st_32x32b_x32(trow + kColO + 32, *reinterpret_cast<uint32_t(*)[32]>(ov + 32));
        tmem_st_wait();
      }
      const float m_use = m == -INFINITY ? 0.f : m;  // a row with no key yet
      float lj = 0.f;
      uint32_t pk[kKT / 2];
#pragma unroll
      for (int c = 0; c < kKT / 2; ++c) {
        const float p0 = ex2(fmaf(__uint_as_float(sr[2 * c]), sl2, -m_use));
        const float p1 = ex2(fmaf(__uint_as_float(sr[2 * c + 1]), sl2, -m_use));
        lj += p0 + p1;
        pk[c] = pack_bf16x2(p0, p1);
      }
      l += lj;
      // P_j: this row's 64 keys as 32 bf16 pairs in TMEM lane r, in the
      // buffer P_{j-2} V_{j-2} read last.
      if (j >= 2 && !(ok = wait_pv(j - 2))) break;
      tmem_st_32x32b_x32(trow + kColP + sb * 32, pk);
      tmem_st_wait();
      tc_fence_before();  // this warp's TMEM reads and writes come first
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[sb]);
    }
    float o[kD];
    if (ok && (ok = wait_pv(n_kt - 1))) {
      tc_fence_after();
      uint32_t ov[kD];
      tmem_ld_32x32b_x32(trow + kColO, *reinterpret_cast<uint32_t(*)[32]>(ov));
      tmem_ld_32x32b_x32(trow + kColO + 32, *reinterpret_cast<uint32_t(*)[32]>(ov + 32));
      tmem_ld_wait();
#pragma unroll
      for (int c = 0; c < kD; ++c) o[c] = __uint_as_float(ov[c]);
    }
    if (ok) {
      // o / l through shared memory (the Q tile's: every product is done)
      // and one TMA store of this warp's 32 rows; rows past T are not written.
      const float inv = 1.0f / l;
      uint8_t* orow = sQ + r * 128;
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e)
          w[e] = pack_16x2(o[8 * c + 2 * e] * inv, o[8 * c + 2 * e + 1] * inv, a.out_f16 != 0);
        *reinterpret_cast<uint4*>(orow + ((c ^ (r & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        tma_store_3d(&tmO, sQ + quarter * 32 * 128, head * kD, q0 + quarter * 32, b);
        bulk_commit_group();
        bulk_wait_group<0>();
      }
      __syncwarp();
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

bool encode(const LaunchEnv& env, CUtensorMap* map, const void* base, int rank,
            const cuuint64_t* dims, const cuuint64_t* strides, const cuuint32_t* box, bool f16) {
  if ((reinterpret_cast<uintptr_t>(base) & 15) != 0) return false;
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  return env.encode(map, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                    rank, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

}  // namespace

int launch_attention_tc(const LaunchEnv& env, const bf16* q, const bf16* kv, long long s_batch,
                        long long s_kv, long long s_head, int B, int h, int T, int t_past,
                        void* out, cudaStream_t stream, bool out_f16) {
  if (B <= 0 || h <= 0 || T <= 0 || t_past < 0) return GPT2_ERR_INVALID_ARG;
  const int n_qtiles = (T + kQT - 1) / kQT;
  if (n_qtiles > 65535 || B * h > 0x7fffffff) return GPT2_ERR_UNSUPPORTED;
  const long long t_all = static_cast<long long>(t_past) + T;
  CUtensorMap tmQ, tmK, tmV, tmO;
  // Q [B*h, T, 64]; K and V of the cache {64 dims, t_all positions, h heads,
  // B sequences}; the output {h*64, T, B}.
  const cuuint64_t qd[3] = {kD, static_cast<cuuint64_t>(T), static_cast<cuuint64_t>(B) * h};
  const cuuint64_t qs[2] = {kD * 2, static_cast<cuuint64_t>(T) * kD * 2};
  const cuuint32_t qb[3] = {kD, kQT, 1};
  const cuuint64_t kd[4] = {kD, static_cast<cuuint64_t>(t_all), static_cast<cuuint64_t>(h),
                            static_cast<cuuint64_t>(B)};
  const cuuint64_t ks[3] = {kD * 2, static_cast<cuuint64_t>(s_head) * 2,
                            static_cast<cuuint64_t>(s_batch) * 2};
  const cuuint32_t kb[4] = {kD, kKT, 1, 1};
  const cuuint64_t od[3] = {static_cast<cuuint64_t>(h) * kD, static_cast<cuuint64_t>(T),
                            static_cast<cuuint64_t>(B)};
  const cuuint64_t os[2] = {static_cast<cuuint64_t>(h) * kD * 2,
                            static_cast<cuuint64_t>(T) * h * kD * 2};
  const cuuint32_t ob[3] = {kD, 32, 1};
  if ((s_head * 2) % 16 != 0 || (s_batch * 2) % 16 != 0 || (s_kv * 2) % 16 != 0)
    return GPT2_ERR_ALIGNMENT;
  if (!encode(env, &tmQ, q, 3, qd, qs, qb, false) || !encode(env, &tmK, kv, 4, kd, ks, kb, false) ||
      !encode(env, &tmV, kv + s_kv, 4, kd, ks, kb, false) ||
      !encode(env, &tmO, out, 3, od, os, ob, out_f16))
    return GPT2_ERR_CUDA;
  static bool attr_set = false;
  if (!attr_set) {
    if (cudaFuncSetAttribute(attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kSmemBytes)) != cudaSuccess)
      return GPT2_ERR_CUDA;
    attr_set = true;
  }
  AttnArgs args{T, t_past, h, n_qtiles, out_f16 ? 1 : 0, env.err};
  const cudaError_t e = launch_pdl(attn_tc_kernel, dim3(B * h, n_qtiles), dim3(kThreads),
                                   kSmemBytes, stream, tmQ, tmK, tmV, tmO, args);
  return e == cudaSuccess ? GPT2_OK : GPT2_ERR_CUDA;
}

}  // namespace gpt2

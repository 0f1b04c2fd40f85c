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
// A persistent kernel: two resident CTAs per SM, each walking its share of
// the (sequence x head, 128-query tile) work items, dealt out longest first
// in rounds that alternate direction; every role runs on into the next tile, so one tile's Q and
// first K/V tiles load while the previous tile finishes.  6 warps:
//   warp 0      TMA: each tile's Q (two buffers), then the 64-key K and V
//               tiles of each step into separate rings (128-byte swizzle):
//               a K stage is free again once its scores are computed, a V
//               stage only after its P V product, so K runs further ahead.  One thread
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
//               its rows of O in TMEM.  At the tile's end each thread
//               writes its row of o / l (128 contiguous bytes).
// Steps entirely above the diagonal are never loaded.  Every wait on an
// mbarrier is bounded: one that runs out raises the error word, and the CTA
// drains its copies and MMAs, frees TMEM and returns.
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
constexpr int kSK = 4;                          // K ring
constexpr int kSV = 5;                          // V ring
constexpr int kThreads = 192;
constexpr uint32_t kQBytes = kQT * kD * 2;      // 16 KB
constexpr uint32_t kKVBytes = kKT * kD * 2;     // 8 KB: one K or V tile
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kColS = 0;                   // two score buffers of 64 columns (fp32)
constexpr uint32_t kColP = 128;                 // two P buffers of 32 columns (bf16 pairs)
constexpr uint32_t kColO = 192;                 // the output accumulator, 64 columns
constexpr float kRescaleLog2 = 8.f;             // max. lag of the reference maximum (log2)
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kBars = 5 * 2 + 2 * kSK + 2 * kSV + 1;
constexpr size_t kSmemBytes =
    1024 + 2 * kQBytes + (kSK + kSV) * kKVBytes + kBars * 8 + 16;
static_assert(2 * (kSmemBytes + 1024) <= 233472, "two CTAs per SM");

struct AttnArgs {
  int T, t_past, h, n_qtiles, n_bh;
  int n_work;   // n_bh * n_qtiles query tiles
  int out_f16;  // output fp16 (else bf16)
  void* out;    // [B, T, h * 64]
  unsigned* err;
  unsigned long long wait_ns;  // limit of each bounded wait
};

// Work item w: the query tiles with the most keys first, then sequence x head.
struct Tile {
  int bh, b, head, q0, n_kt;
};
__device__ __forceinline__ Tile tile_of(const AttnArgs& a, int w) {
  Tile t;
  const int qt = a.n_qtiles - 1 - w / a.n_bh;
  t.bh = w - (w / a.n_bh) * a.n_bh;
  t.b = t.bh / a.h;
  t.head = t.bh - t.b * a.h;
  t.q0 = qt * kQT;
  const int q_last = min(t.q0 + kQT, a.T) - 1;
  t.n_kt = (a.t_past + q_last + 1 + kKT - 1) / kKT;  // steps up to the last query
  return t;
}

__global__ void __launch_bounds__(kThreads, 2)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const AttnArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = sm;                            // [2][16 KB] by tile parity
  uint8_t* sK = sQ + 2 * kQBytes;              // [kSK][8 KB]
  uint8_t* sV = sK + kSK * kKVBytes;           // [kSV][8 KB]
  uint64_t* q_full = reinterpret_cast<uint64_t*>(sV + kSV * kKVBytes);  // [2]
  uint64_t* q_empty = q_full + 2;              // [2] the tile's last S product done
  uint64_t* k_full = q_empty + 2;              // [kSK] K landed
  uint64_t* k_empty = k_full + kSK;            // [kSK] its scores computed
  uint64_t* v_full = k_empty + kSK;            // [kSV] V landed
  uint64_t* v_empty = v_full + kSV;            // [kSV] its P V product done
  // A softmax warp reads S_g before it publishes P_g, and reads a tile's O
  // before it publishes P of the next tile's first step: so P_g published by
  // all four warps also means that S_g's buffer (next used by S_{g+2}) has
  // been read, that any rescale of O for step g is done, and, on a tile's
  // first step, that the previous tile's O has been read.  Steps g count on
  // across the CTA's tiles.
  uint64_t* s_full = v_empty + kSV;            // [2] scores ready
  uint64_t* p_full = s_full + 2;               // [2] P written, O rescaled / read (4 warps)
  uint64_t* pv_done = p_full + 2;              // [2] P_g V_g done (P_g's buffer read, O updated)
  uint64_t* mma_done = pv_done + 2;            // [1]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // This CTA's k-th work item: rounds of gridDim.x items, in reverse CTA
  // order on odd rounds, so that long and short tiles pair up.
  const int cta = static_cast<int>(blockIdx.x), n_cta = static_cast<int>(gridDim.x);
  auto work = [&](int k) { return k * n_cta + ((k & 1) ? n_cta - 1 - cta : cta); };
  const int w0 = cta;

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&q_full[i], 1);
      mbar_init(&q_empty[i], 1);
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], 4);
      mbar_init(&pv_done[i], 1);
    }
    for (int s = 0; s < kSK; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
    }
    for (int s = 0; s < kSV; ++s) {
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
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
    // Two streams over the CTA's tiles: K (with each tile's Q ahead of its
    // first K) and V.  A stage is free once the product that read its
    // previous tile has completed (no wait for the first pass).
    int kw = w0, kj = 0, kt = 0, kg = 0;       // K stream: work item, step, tile count, global step
    int vw = w0, vj = 0, vt = 0, vg = 0;       // V stream
    Tile tk = tile_of(a, w0 < a.n_work ? w0 : 0), tv = tk;
    bool ok = true;
    unsigned long long t_idle = 0;
    int q_issued = 0;                           // Q loads issued (= tiles whose Q is on its way)
    while (kw < a.n_work || vw < a.n_work) {
      bool progress = false;
      if (kw < a.n_work && kj == 0 && q_issued == kt) {
        // The tile's Q goes first, into the buffer of tile kt - 2.
        if (kt < 2 ||
            mbar_test_wait(&q_empty[kt & 1], static_cast<uint32_t>((kt >> 1) - 1) & 1u)) {
          mbar_arrive_expect_tx(&q_full[kt & 1], kQBytes);
          tma_load_3d(sQ + (kt & 1) * kQBytes, &tmQ, &q_full[kt & 1], 0, tk.q0, tk.bh);
          ++q_issued;
          progress = true;
        }
      } else if (kw < a.n_work) {
        if (kg < kSK ||
            mbar_test_wait(&k_empty[kg % kSK], static_cast<uint32_t>(kg / kSK - 1) & 1u)) {
          const int s = kg % kSK;
          mbar_arrive_expect_tx(&k_full[s], kKVBytes);
          tma_load_4d(sK + s * kKVBytes, &tmK, &k_full[s], 0, kj * kKT, tk.head, tk.b);
          ++kg;
          progress = true;
          if (++kj == tk.n_kt) {
            kj = 0;
            ++kt;
            kw = work(kt);
            if (kw < a.n_work) tk = tile_of(a, kw);
          }
        }
      }
      if (vw < a.n_work &&
          (vg < kSV || mbar_test_wait(&v_empty[vg % kSV], static_cast<uint32_t>(vg / kSV - 1) & 1u))) {
        const int s = vg % kSV;
        mbar_arrive_expect_tx(&v_full[s], kKVBytes);
        tma_load_4d(sV + s * kKVBytes, &tmV, &v_full[s], 0, vj * kKT, tv.head, tv.b);
        ++vg;
        progress = true;
        if (++vj == tv.n_kt) {
          vj = 0;
          vw = work(++vt);
          if (vw < a.n_work) tv = tile_of(a, vw);
        }
      }
      if (progress) {
        t_idle = 0;
      } else {
        // Nothing could be issued: the same bounded wait as elsewhere.
        __nanosleep(32);
        const unsigned long long now = global_timer_ns();
        if (t_idle == 0) {
          t_idle = now;
        } else if (*abort_flag || now - t_idle > a.wait_ns) {
          if (!*abort_flag) raise_error(a.err, kErrTimeout);
          *abort_flag = 1;
          ok = false;
          break;
        }
      }
    }
    if (!ok) {
      // Drain: every copy already issued must land before the CTA exits.
      for (int t = max(0, q_issued - 2); t < q_issued; ++t)
        mbar_wait_bounded(&q_full[t & 1], static_cast<uint32_t>(t >> 1) & 1u, nullptr, a.err);
      for (int g = max(0, kg - kSK); g < kg; ++g)
        mbar_wait_bounded(&k_full[g % kSK], static_cast<uint32_t>(g / kSK) & 1u, nullptr, a.err);
      for (int g = max(0, vg - kSV); g < vg; ++g)
        mbar_wait_bounded(&v_full[g % kSV], static_cast<uint32_t>(g / kSV) & 1u, nullptr, a.err);
    }
  } else if (warp == 1 && lane == 0) {
    // ------------------------------------------------------- MMA issuer --
    const uint32_t id_s = umma_idesc_16(kQT, kKT, false, false);
    const uint32_t id_pv = umma_idesc_16(kQT, kD, false, true);
    // S cursor (one step ahead of the P V cursor), over the CTA's tiles.
    int sw = w0, sj = 0, st = 0, sg = 0;       // work item, step, tile count, global step
    Tile ts = tile_of(a, w0 < a.n_work ? w0 : 0);
    auto issue_s = [&]() -> bool {
      const int s = sg % kSK, sb = sg & 1;
      if (sj == 0 && !mbar_wait_bounded(&q_full[st & 1], static_cast<uint32_t>(st >> 1) & 1u,
                                        abort_flag, a.err, a.wait_ns))
        return false;
      // S_{g-2}, the buffer's previous tile, was read before P_{g-2} was
      // published, which this thread has already waited for.
      if (!mbar_wait_bounded(&k_full[s], static_cast<uint32_t>(sg / kSK) & 1u, abort_flag, a.err,
                             a.wait_ns))
        return false;
      tc_fence_after();
      const uint64_t q_desc = sdesc_k_sw128(smem_u32(sQ + (st & 1) * kQBytes));
      const uint64_t k_desc = sdesc_k_sw128(smem_u32(sK + s * kKVBytes));
      const uint32_t d = tmem + kColS + sb * 64;
#pragma unroll
      for (int k = 0; k < kD / 16; ++k)
        umma_f16kind(d, q_desc + 2 * k, k_desc + 2 * k, id_s, k != 0 ? 1u : 0u);
      umma_commit(&s_full[sb]);
      umma_commit(&k_empty[s]);
      ++sg;
      if (++sj == ts.n_kt) {
        umma_commit(&q_empty[st & 1]);  // the tile's Q buffer is free once this product is done
        sj = 0;
        ++st;
        sw = work(st);
        if (sw < a.n_work) ts = tile_of(a, sw);
      }
      return true;
    };
    bool ok = w0 >= a.n_work || issue_s();
    int g = 0;
    for (int t = 0, w = w0; ok && w < a.n_work; w = work(++t)) {
      const int n_kt = tile_of(a, w).n_kt;
      for (int j = 0; j < n_kt; ++j, ++g) {
        if (sw < a.n_work && !(ok = issue_s())) break;
        const int pb = g & 1, s = g % kSV;
        if (!mbar_wait_bounded(&v_full[s], static_cast<uint32_t>(g / kSV) & 1u, abort_flag, a.err,
                               a.wait_ns) ||
            !mbar_wait_bounded(&p_full[pb], static_cast<uint32_t>(g >> 1) & 1u, abort_flag, a.err,
                               a.wait_ns)) {
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
    }
    // Every MMA issued above must retire before TMEM is freed.
    umma_commit(mma_done);
    mbar_wait_bounded(mma_done, 0, nullptr, a.err);
  } else if (warp >= 2) {
    // ---------------------------------------------------------- softmax --
    const int quarter = warp & 3;                // TMEM lanes 32 * quarter ..
    const int r = quarter * 32 + lane;           // query row in the tile
    const uint32_t trow = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const float sl2 = 0.125f * kLog2e;           // 1/sqrt(64), in log2 units
    bool ok = true;
    bool bad = false;                            // an output value out of range
    // The product P_t V_t has completed (pv_done of step t; never more than
    // one phase behind when waited for).
    auto wait_pv = [&](int t) -> bool {
      return mbar_wait_bounded(&pv_done[t & 1], static_cast<uint32_t>(t >> 1) & 1u, abort_flag,
                               a.err, a.wait_ns);
    };
    int g = 0;
    for (int t = 0, w = w0; ok && w < a.n_work; w = work(++t)) {
      const Tile tl = tile_of(a, w);
      const int pos = a.t_past + tl.q0 + r;      // this row's absolute position
      float m = -INFINITY, l = 0.f;              // reference maximum (log2 units), row sum
      for (int j = 0; j < tl.n_kt; ++j) {
        const int gj = g + j, sb = gj & 1;
        if (!mbar_wait_bounded(&s_full[sb], static_cast<uint32_t>(gj >> 1) & 1u, abort_flag,
                               a.err, a.wait_ns)) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t sr[kKT];
        tmem_ld_32x32b_x32(trow + kColS + sb * 64, *reinterpret_cast<uint32_t(*)[32]>(sr));
        tmem_ld_32x32b_x32(trow + kColS + sb * 64 + 32,
                           *reinterpret_cast<uint32_t(*)[32]>(sr + 32));
        tmem_ld_wait();

        // Raw scores; the 1/sqrt(64) scale (in log2 units) is applied to the
        // row maximum and inside the exponent's fused multiply-add.
        const int key0 = j * kKT;
        if (__any_sync(0xffffffffu, key0 + kKT - 1 > pos)) {  // a step crossing some row's diagonal
#pragma unroll
          for (int c = 0; c < kKT; ++c)
            if (key0 + c > pos) sr[c] = __float_as_uint(-INFINITY);
        }
        // Row maximum over eight independent chains (keys i, i + 8, ..., i + 56):
        // three-input maxima over keys 0..55, a two-input one for 56..63.
        float mx;
        {
          static_assert(kKT == 64, "the chains below cover 64 keys");
          float m8[8];
#pragma unroll
          for (int i = 0; i < 8; ++i)
            m8[i] = max3(__uint_as_float(sr[i]), __uint_as_float(sr[8 + i]),
                         __uint_as_float(sr[16 + i]));
#pragma unroll
          for (int c = 24; c < 56; c += 16)
#pragma unroll
            for (int i = 0; i < 8; ++i)
              m8[i] = max3(m8[i], __uint_as_float(sr[c + i]), __uint_as_float(sr[c + 8 + i]));
#pragma unroll
          for (int i = 0; i < 8; ++i) m8[i] = fmaxf(m8[i], __uint_as_float(sr[56 + i]));
          mx = max3(max3(m8[0], m8[1], m8[2]), max3(m8[3], m8[4], m8[5]), fmaxf(m8[6], m8[7]));
        }
        // A new reference maximum only when this row's passed it by more
        // than kRescaleLog2 (always on the row's first key); O and l scale
        // by 2^(m_old - m_new) (0 while m_old = -inf).
        const float m_row = mx * sl2;
        const bool bump = m_row > m + kRescaleLog2;
        const float alpha = bump ? ex2(m - m_row) : 1.f;
        if (bump) m = m_row;
        l *= alpha;
        if (j > 0 && __any_sync(0xffffffffu, bump)) {
          // O holds this tile's P V products so far: wait for the last one,
          // then rescale this warp's 32 rows in place (alpha = 1 elsewhere).
          if (!(ok = wait_pv(gj - 1))) break;
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
        // Packed pairs: x = s * scale - m for two keys per instruction, the
        // row sum in four packed accumulators.
        const uint64_t sl2_2 = f2(sl2, sl2), nm_2 = f2(-m_use, -m_use);
        uint64_t ls2[4] = {0ull, 0ull, 0ull, 0ull};
        uint32_t pk[kKT / 2];
#pragma unroll
        for (int c = 0; c < kKT / 2; ++c) {
          float x0, x1;
          f2_split(ffma2(f2(__uint_as_float(sr[2 * c]), __uint_as_float(sr[2 * c + 1])), sl2_2,
                         nm_2),
                   x0, x1);
          const float p0 = ex2(x0), p1 = ex2(x1);
          ls2[c & 3] = fadd2(ls2[c & 3], f2(p0, p1));
          pk[c] = pack_bf16x2(p0, p1);
        }
        {
          float a0, a1;
          f2_split(fadd2(fadd2(ls2[0], ls2[1]), fadd2(ls2[2], ls2[3])), a0, a1);
          l += a0 + a1;
        }
        // P_g: this row's 64 keys as 32 bf16 pairs in TMEM lane r, in the
        // buffer P_{g-2} V_{g-2} read last.
        if (gj >= 2 && !(ok = wait_pv(gj - 2))) break;
        tmem_st_32x32b_x32(trow + kColP + sb * 32, pk);
        tmem_st_wait();
        tc_fence_before();  // this warp's TMEM reads and writes come first
        __syncwarp();
        if (lane == 0) mbar_arrive(&p_full[sb]);
      }
      if (!ok) break;
      g += tl.n_kt;
      // o / l straight to the output: 128 contiguous bytes per row, rows
      // past T not written.  O is read before this warp publishes the next
      // tile's first P, which the next tile's first product waits for.
      if (!(ok = wait_pv(g - 1))) break;
      tc_fence_after();
      uint32_t ov[kD];
      tmem_ld_32x32b_x32(trow + kColO, *reinterpret_cast<uint32_t(*)[32]>(ov));
      tmem_ld_32x32b_x32(trow + kColO + 32, *reinterpret_cast<uint32_t(*)[32]>(ov + 32));
      tmem_ld_wait();
      const float inv = 1.0f / l;
      const int row = tl.q0 + r;
      if (row < a.T) {
        // fp16 output: values beyond 65504 would become inf; either kind:
        // nothing non-finite.
        const float lim = a.out_f16 ? 65504.f : 3.4028235e38f;
        uint4* dst = reinterpret_cast<uint4*>(
            static_cast<uint16_t*>(a.out) +
            (static_cast<size_t>(tl.b) * a.T + row) * (static_cast<size_t>(a.h) * kD) +
            tl.head * kD);
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          uint32_t wv[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float o0 = __uint_as_float(ov[8 * c + 2 * e]) * inv;
            const float o1 = __uint_as_float(ov[8 * c + 2 * e + 1]) * inv;
            bad |= !(fabsf(o0) <= lim) || !(fabsf(o1) <= lim);
            wv[e] = pack_16x2(o0, o1, a.out_f16 != 0);
          }
          dst[c] = make_uint4(wv[0], wv[1], wv[2], wv[3]);
        }
      }
    }
    if (__any_sync(0xffffffffu, bad) && lane == 0) raise_error(a.err, kErrRange);
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
  CUtensorMap tmQ, tmK, tmV;
  // Q [B*h, T, 64]; K and V of the cache {64 dims, t_all positions, h heads,
  // B sequences}.
  const cuuint64_t qd[3] = {kD, static_cast<cuuint64_t>(T), static_cast<cuuint64_t>(B) * h};
  const cuuint64_t qs[2] = {kD * 2, static_cast<cuuint64_t>(T) * kD * 2};
  const cuuint32_t qb[3] = {kD, kQT, 1};
  const cuuint64_t kd[4] = {kD, static_cast<cuuint64_t>(t_all), static_cast<cuuint64_t>(h),
                            static_cast<cuuint64_t>(B)};
  const cuuint64_t ks[3] = {kD * 2, static_cast<cuuint64_t>(s_head) * 2,
                            static_cast<cuuint64_t>(s_batch) * 2};
  const cuuint32_t kb[4] = {kD, kKT, 1, 1};
  if ((s_head * 2) % 16 != 0 || (s_batch * 2) % 16 != 0 || (s_kv * 2) % 16 != 0 ||
      (reinterpret_cast<uintptr_t>(out) & 15) != 0)
    return GPT2_ERR_ALIGNMENT;
  if (!encode(env, &tmQ, q, 3, qd, qs, qb, false) || !encode(env, &tmK, kv, 4, kd, ks, kb, false) ||
      !encode(env, &tmV, kv + s_kv, 4, kd, ks, kb, false))
    return GPT2_ERR_CUDA;
  if (!ensure_smem_limit(reinterpret_cast<const void*>(&attn_tc_kernel),
                         static_cast<int>(kSmemBytes)))
    return GPT2_ERR_CUDA;
  const long long n_work = static_cast<long long>(B) * h * n_qtiles;
  if (n_work > 0x7fffffff) return GPT2_ERR_UNSUPPORTED;
  AttnArgs args{T, t_past, h, n_qtiles, B * h, static_cast<int>(n_work), out_f16 ? 1 : 0, out,
                env.err, env.wait_ns};
  // Two resident CTAs per SM, each walking the tiles w = blockIdx.x, + grid, ...
  const int grid = static_cast<int>(std::min<long long>(n_work, 2LL * env.num_sms));
  const cudaError_t e = launch_pdl(attn_tc_kernel, dim3(grid), dim3(kThreads), kSmemBytes, stream,
                                   tmQ, tmK, tmV, args);
  return e == cudaSuccess ? GPT2_OK : GPT2_ERR_CUDA;
}

}  // namespace gpt2

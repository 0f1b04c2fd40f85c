// gemm_tc.cu -- tensor-core GEMM for sm_103a: C[M,N] = A[M,K] * W[N,K]^T,
// 16-bit operands (fp16 for the products of the bf16 forward, whose
// activations are written as fp16 and weights converted from bf16; bf16 when
// a caller passes bf16 operands), fp32 accumulation in tensor memory, fused
// epilogues.
//
// It computes the five Linear products of the GPT-2 forward ("GPT-2 Full
// Forward Pass", "How it works": fused c_attn d->3d, attention c_proj, c_fc
// d->4d, mlp c_proj, and the tied head LN_f(H) W_e^T), with the epilogues the
// block needs: bias; bias + GELU (tanh form); bias + residual add ("GPT-2
// Decoder Block", "How it works": x <- x + a, x <- x + m); the QKV split into
// heads with the keys/values written straight into the KV cache; and fp32
// logits with a ragged vocabulary tail.
//
// Design (one CTA per SM, persistent over output tiles of 128 x BN):
//   warp 0      TMA producer: 128x64 A and BNx64 W boxes, 128-byte swizzle,
//               into a ring of `stages` shared-memory slots (mbarrier pairs).
//   warp 1      MMA issuer: one thread issues tcgen05.mma (M=128, N=BN,
//               K=16) x4 per slot into one of two TMEM accumulators.
//   warp 2      allocates / frees 512 TMEM columns.
//   warps 4..   epilogue, two warps per TMEM lane quarter, each taking half
//               of the tile's columns (one warp, all of them, for the bf16
//               block output) in chunks of 32 x 32: tcgen05.ld, bias /
//               GELU / residual in registers, the chunk written to a swizzled
//               shared-memory box, and one TMA tensor store per chunk (the
//               fp32 residual arrives the same way, by a TMA load).  Q, K and
//               V chunks go to their head-major destinations by 3-D TMA
//               stores.  fp32 logits rows are only 4-byte aligned, so that
//               epilogue transposes through shared memory and each store
//               instruction writes one row's 32 consecutive columns.  The
//               head reduced to the next-token loss writes no logits: each
//               thread reduces its token's 256 entries of the tile.
// Two accumulators let the epilogue of tile i overlap the mainloop of i+1.
// Every mbarrier wait is bounded; a wait that runs out raises the context's
// error word and the CTA drains its copies, frees TMEM and returns.
#include <string.h>

#include <algorithm>

#include "device.cuh"
#include "internal.h"

namespace gpt2 {

namespace {

constexpr int kBM = 128;
constexpr int kBK = 64;                       // one 128-byte swizzle row of bf16
// Epilogue warps: two per TMEM lane quarter (each taking half of a tile's
// columns), or one for the bf16 block output made from the fp32 residual
// (measured on GB300 for the block's mlp c_proj: GPT-2-small 43.3 -> 41.2 us,
// GPT-2-XL shape 80 -> 70 us with four; the in-place fp32 residual epilogue
// is faster with eight).  The top-k head has eight in two groups of four, one
// group per accumulator: each warp reduces whole rows of 256 entries, and the
// two groups drain alternate tiles at the same time.
__host__ __device__ constexpr int epi_warps(int k) {
  return k == kEpiResidBf16Out || k == kEpiHeadLoss ? 4 : 8;
}
// Epilogue groups that each own one accumulator (else every epilogue warp
// takes part in every tile).
__host__ __device__ constexpr bool acc_groups(int k) { return k == kEpiHeadTopK; }
__host__ __device__ constexpr int epi_threads(int k) { return 128 + 32 * epi_warps(k); }
constexpr uint32_t kABytes = kBM * kBK * 2;   // 16 KB per A slot
constexpr int kMaxStages = 8;
constexpr uint32_t kTmemCols = 512;           // two accumulators of up to 256 columns
constexpr int kSmemLimit = 232448;            // 227 KB opt-in per CTA
constexpr int kRBuf = 32 * 32 * 4;            // fp32 32x32 box, rows of 128 B, 128-byte swizzle
constexpr int kOBuf = 32 * 32 * 2;            // bf16 32x32 box, rows of 64 B, 64-byte swizzle
constexpr int kBiasBufs = 3;                  // bias buffers per column segment, by tile index mod 3
constexpr int kBiasBytes = kBiasBufs * 256 * 2;  // bf16 bias of a tile's columns, per buffer
constexpr int kLogitsLd = 33;                 // logits transpose row stride (floats)

static_assert(kRBuf % 1024 == 0 && kOBuf % 1024 == 0, "staging boxes must stay 1 KB aligned");

__host__ __device__ constexpr bool uses_rbuf(int k) {
  return k == kEpiResidF32 || k == kEpiResidBf16In || k == kEpiResidBf16Out;
}
__host__ __device__ constexpr bool uses_obuf(int k) {
  return k == kEpiBias || k == kEpiGelu || k == kEpiQkv || k == kEpiResidBf16Out;
}
__host__ __device__ constexpr int slot_bytes(int k) {
  return (uses_rbuf(k) ? kRBuf : 0) + (uses_obuf(k) ? kOBuf : 0);
}
// Shared memory of one epilogue warp: two staging slots (multiples of 1 KB,
// so every swizzled box stays 1024-byte aligned), or (logits) one transposed
// 32 x 32 chunk.  The bias buffers follow all warps' slots:
// the four warps of a column half share one (each writes the same values),
// and three of them rotate by tile, so a warp that runs two tiles ahead of
// another (the most the two accumulators allow) never overwrites a buffer
// still being read.
__host__ __device__ constexpr int epi_warp_bytes(int k) {
  return k == kEpiLogits ? 32 * kLogitsLd * 4
         : k == kEpiLogitsT ? 0
         : k == kEpiHeadLoss ? 0
         : k == kEpiHeadTopK ? 32 * 33 * 4
                             : 2 * slot_bytes(k);
}
__host__ __device__ constexpr int epi_bias_bytes(int k) {
  return k == kEpiLogits || k == kEpiLogitsT || k == kEpiHeadLoss || k == kEpiHeadTopK
             ? 0
             : kBiasBytes;
}

struct GemmArgs {
  int M, N, K;
  int BN;
  int stages;
  int num_m_blocks;
  int num_n_blocks;
  int n_inner;       // tile index runs over N blocks first (else over M blocks)
  int num_tiles;
  int vec_ok;        // row stride allows 16-byte vector access of out / resid
  int tma_out;       // output written by TMA stores through tmO
  int tma_resid;     // fp32 residual read by TMA loads through tmR
  int tma_qkv;       // Q / K / V written by 3-D TMA stores through tmQ / tmKV
  int kv_z_per_seq;  // tmKV rows (heads) between sequences
  int out_f16;       // 16-bit outputs of kEpiBias / kEpiGelu are fp16 (else bf16)
  uint32_t idesc;    // tcgen05.mma instruction descriptor (operand kind, tile)
  unsigned* err;
  unsigned long long wait_ns;  // limit of each bounded wait (the drains keep 2 s)
  EpiParams ep;
};

// Dynamic shared memory of one CTA; cg = 2 holds half of the tile's B rows.
__device__ __forceinline__ void tile_coords(const GemmArgs& a, int tile, int& m_blk, int& n_blk) {
  if (a.n_inner) {
    m_blk = tile / a.num_n_blocks;
    n_blk = tile - m_blk * a.num_n_blocks;
  } else {
    n_blk = tile / a.num_m_blocks;
    m_blk = tile - n_blk * a.num_m_blocks;
  }
}

__host__ __device__ inline size_t smem_bytes_for(int kind, int BN, int stages, int cg) {
  return 1024 /* alignment slack */ +
         static_cast<size_t>(stages) * (kABytes + (BN / cg) * kBK * 2) +
         static_cast<size_t>(epi_warps(kind)) * epi_warp_bytes(kind) + epi_bias_bytes(kind) +
         (2 * stages + 5 + 2 * epi_warps(kind)) * sizeof(uint64_t) + 16;
}

__device__ __forceinline__ void unpack8(const uint4 v, float* f) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = bf16_lo(w[i]);
    f[2 * i + 1] = bf16_hi(w[i]);
  }
}

__device__ __forceinline__ uint4 pack8(const float* f, bool f16) {
  return make_uint4(pack_16x2(f[0], f[1], f16), pack_16x2(f[2], f[3], f16),
                    pack_16x2(f[4], f[5], f16), pack_16x2(f[6], f[7], f16));
}

__device__ __forceinline__ void store32_16(void* dst, const float (&v)[32], bool f16) {
  uint4* p = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int i = 0; i < 4; ++i) p[i] = pack8(v + 8 * i, f16);
}

// Row r of a 32x32 fp32 box with the 128-byte swizzle: 16-byte chunk c of
// the row sits at chunk position c ^ (r & 7).
__device__ __forceinline__ void box_write_f32(uint8_t* box, int r, const float (&v)[32]) {
#pragma unroll
  for (int c = 0; c < 8; ++c)
    *reinterpret_cast<float4*>(box + r * 128 + ((c ^ (r & 7)) << 4)) =
        make_float4(v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
}
__device__ __forceinline__ void box_read_f32(const uint8_t* box, int r, float (&v)[32]) {
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    const float4 x = *reinterpret_cast<const float4*>(box + r * 128 + ((c ^ (r & 7)) << 4));
    v[4 * c] = x.x; v[4 * c + 1] = x.y; v[4 * c + 2] = x.z; v[4 * c + 3] = x.w;
  }
}
// Row r of a 32x32 16-bit box with the 64-byte swizzle: chunk c at c ^ ((r >> 1) & 3).
__device__ __forceinline__ void box_write_16(uint8_t* box, int r, const float (&v)[32], bool f16) {
#pragma unroll
  for (int c = 0; c < 4; ++c)
    *reinterpret_cast<uint4*>(box + r * 64 + ((c ^ ((r >> 1) & 3)) << 4)) = pack8(v + 8 * c, f16);
}

// The same box row from 16 packed pairs.
__device__ __forceinline__ void box_write_packed(uint8_t* box, int r, const uint32_t (&w)[16]) {
#pragma unroll
  for (int c = 0; c < 4; ++c)
    *reinterpret_cast<uint4*>(box + r * 64 + ((c ^ ((r >> 1) & 3)) << 4)) =
        make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
}

// Per-warp epilogue state carried across chunks and tiles.
struct EpiState {
  int chunk;          // chunks processed so far (selects the staging slot)
  uint32_t rpar;      // bit s: parity of the next wait on residual barrier s
  uint32_t inflight;  // bit s: a residual load into slot s is in flight
  uint4 rnext[4];     // kEpiResidBf16In: next chunk's bf16 residual, one row of 32
};

// Issues the TMA load of the fp32 residual box of chunk column `col` into slot s.
__device__ __forceinline__ void resid_load(uint8_t* rb, uint64_t* bar, const CUtensorMap* tmR,
                                           int col, int row0) {
  fence_proxy_async_smem();  // earlier generic reads of the box come first
  mbar_arrive_expect_tx(bar, kRBuf);
  tma_load_2d(rb, tmR, bar, col, row0);
}

// Loads one row's 32 bf16 residual values (columns col .. col+31) into registers.
__device__ __forceinline__ void resid16_fetch(const GemmArgs& a, int row, int col, uint4 (&v)[4]) {
  const EpiParams& ep = a.ep;
  const bf16* rp = static_cast<const bf16*>(ep.resid) + static_cast<size_t>(row) * ep.ldo + col;
  if (row >= a.M) {
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] = make_uint4(0u, 0u, 0u, 0u);
  } else if (col + 32 <= a.N && a.vec_ok) {
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] = reinterpret_cast<const uint4*>(rp)[i];
  } else {
    uint32_t w[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const uint32_t lo = col + 2 * j < a.N ? reinterpret_cast<const uint16_t*>(rp)[2 * j] : 0u;
      const uint32_t hi = col + 2 * j + 1 < a.N ? reinterpret_cast<const uint16_t*>(rp)[2 * j + 1] : 0u;
      w[j] = lo | (hi << 16);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
  }
}

// Work a warp can do for its share of a tile before the accumulator is ready:
// the bias of its columns into shared memory, the fp32 residual boxes of its
// first two chunks by TMA, the bf16 residual of its first chunk into registers.
template <int KIND>
__device__ __forceinline__ void epilogue_prefetch(int row0, int ncol0, int ncols, int lane,
                                                  uint8_t* epi, uint16_t* bias_s, uint64_t* rbar,
                                                  EpiState& s, const GemmArgs& a,
                                                  const CUtensorMap* tmR) {
  if constexpr (KIND != kEpiLogits && KIND != kEpiLogitsT && KIND != kEpiHeadLoss &&
                KIND != kEpiHeadTopK) {
    const int N = a.N;
    for (int j = 4 * lane; j < ncols; j += 128) {
      const int col = ncol0 + j;
      const uint16_t* bp = static_cast<const uint16_t*>(a.ep.bias) + col;
      uint2 w;
      if (col + 4 <= N) {
        w = *reinterpret_cast<const uint2*>(bp);
      } else {
        const uint32_t b0 = col < N ? bp[0] : 0u, b1 = col + 1 < N ? bp[1] : 0u;
        const uint32_t b2 = col + 2 < N ? bp[2] : 0u;
        w = make_uint2(b0 | (b1 << 16), b2);
      }
      *reinterpret_cast<uint2*>(bias_s + j) = w;
    }
    if constexpr (KIND == kEpiResidF32 || KIND == kEpiResidBf16Out) {
      if (a.tma_resid && lane == 0) {
        // kEpiResidF32 stages its output in the residual box: the stores that
        // last read the slots must be done.
        if constexpr (KIND == kEpiResidF32) bulk_wait_group_read<0>();
        for (int c = 0; c < 2; ++c) {
          const int col = ncol0 + 32 * c;
          if (32 * c >= ncols || col >= N) break;
          const int slot = (s.chunk + c) & 1;
          resid_load(epi + slot * slot_bytes(KIND), &rbar[slot], tmR, col, row0);
          s.inflight |= 1u << slot;
        }
      }
    }
    if constexpr (KIND == kEpiResidBf16In) resid16_fetch(a, row0 + lane, ncol0, s.rnext);
    __syncwarp();
  }
}

// kEpiHeadLoss, one warp's share of a tile of the head: tokens on the TMEM
// lanes (this thread: token row0 + lane), vocabulary entries on the columns
// (this warp: the kHeadLossBlock entries from ncol0, the whole tile).  Each thread reduces its
// token's entries, 32 at a time, to the maximum, the lowest index of it and
// the sum of 2^((z - max) log2 e), rescaling the sum when a later chunk
// raises the maximum, and stores the block's partial; the thread whose
// entries hold its token's target stores the target logit.  No data leaves
// the thread: no shared memory, no shuffles.
__device__ __forceinline__ void head_loss_rows(uint32_t tbase, int row0, int ncol0, int lane,
                                               const GemmArgs& a) {
  constexpr float kL2e = 1.4426950408889634f;
  const EpiParams& ep = a.ep;
  const int n_tok = a.M, V = a.N;
  const int row = row0 + lane;
  const bool row_ok = row < n_tok;
  if (ncol0 >= V) return;  // a half tile past the vocabulary (warp-uniform)
  const int y = (ep.tgt && row_ok) ? ep.tgt[row] : -1;
  float m = -INFINITY, sum = 0.f;
  int idx = 0x7fffffff;
  for (int c = 0; c < kHeadLossBlock; c += 32) {
    const int col0 = ncol0 + c;
    if (col0 >= V) break;  // warp-uniform
    uint32_t r[32];
    tmem_ld_32x32b_x32(tbase + static_cast<uint32_t>(c), r);
    tmem_ld_wait();
    if (col0 + 32 > V) {  // the vocabulary's ragged end: entries past it do not count
#pragma unroll
      for (int i = 0; i < 32; ++i)
        if (col0 + i >= V) r[i] = __float_as_uint(-INFINITY);
    }
    if (y >= col0 && y < col0 + 32) {
      float t = 0.f;
#pragma unroll
      for (int i = 0; i < 32; ++i)
        if (i == y - col0) t = __uint_as_float(r[i]);
      ep.tgt_logit[row] = t;
    }
    // Chunk maximum and its first index: four interleaved running maxima
    // (strictly greater, so each keeps its first index), merged lowest index
    // first on ties.
    float cm[4];
    int ci[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      cm[k] = __uint_as_float(r[k]);
      ci[k] = k;
    }
#pragma unroll
    for (int i = 4; i < 32; ++i) {
      const float v = __uint_as_float(r[i]);
      if (v > cm[i & 3]) {
        cm[i & 3] = v;
        ci[i & 3] = i;
      }
    }
#pragma unroll
    for (int k = 1; k < 4; ++k)
      if (cm[k] > cm[0] || (cm[k] == cm[0] && ci[k] < ci[0])) {
        cm[0] = cm[k];
        ci[0] = ci[k];
      }
    if (cm[0] > m) {  // a new maximum (strictly: earlier chunks keep ties)
      sum = m == -INFINITY ? 0.f : sum * ex2((m - cm[0]) * kL2e);
      m = cm[0];
      idx = col0 + ci[0];
    }
    const float ml = m * kL2e;
    float s4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int i = 0; i < 32; ++i) s4[i & 3] += ex2(fmaf(__uint_as_float(r[i]), kL2e, -ml));
    sum += (s4[0] + s4[1]) + (s4[2] + s4[3]);
  }
  if (row_ok) {
    const size_t o = static_cast<size_t>(ncol0 / kHeadLossBlock) * n_tok + row;
    ep.part_m[o] = m;
    ep.part_s[o] = sum;
    ep.part_i[o] = idx;
  }
}

// min with NaN propagation (min.NaN): a NaN entry must not pass for a second
// largest value (fminf would return the other operand).
__device__ __forceinline__ float fmin_nan(float a, float b) {
  float r;
  asm("min.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}

// Sorts 16 values in descending order (bitonic network, fixed indices).
__device__ __forceinline__ void sort16_desc(float (&v)[16]) {
#pragma unroll
  for (int ks = 1; ks <= 4; ++ks) {
    const int k = 1 << ks;
#pragma unroll
    for (int js = ks - 1; js >= 0; --js) {
      const int j = 1 << js;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int l = i ^ j;
        if (l > i) {
          const float hi = fmaxf(v[i], v[l]), lo = fminf(v[i], v[l]);
          const bool desc = (i & k) == 0;
          v[i] = desc ? hi : lo;
          v[l] = desc ? lo : hi;
        }
      }
    }
  }
}

// kEpiHeadTopK, one warp's share of a tile of the head, laid out as for
// head_loss_rows: each thread owns token row0 + lane and the tile's
// kHeadLossBlock vocabulary entries from ncol0.  Every lane is another token,
// so inserting entries one by one into a sorted list would make the warp run
// the insertion at nearly every entry.  Instead, in two passes over TMEM:
//   1. each 32-entry chunk's largest and second largest entry (NaN and the
//      entries past V left out): the largest of all is the block's maximum
//      (the base of the logsumexp sum, so no rescaling is needed), and the
//      k-th largest of these 16 values is a floor under the block's top k
//      (they are k distinct entries at least that large);
//   2. the sum of 2^((z - max) log2 e), and the entries at or above the floor
//      as a bit mask (about one in nine on random logits); when any lane of
//      the warp has some, the chunk goes to shared memory (rows padded to 33
//      floats: conflict-free), and each lane inserts its candidates, in index
//      order, into its sorted list of kTopKMax with a branch-free network
//      (strict comparisons: among equal values the lower index stays first).
// The first k entries of the list are the block's top k; the floor is kept
// above -inf, so NaN and -inf entries are never candidates.
__device__ __forceinline__ void head_topk_rows(uint32_t tbase, int row0, int ncol0, int lane,
                                               const GemmArgs& a, float* stage) {
  constexpr float kL2e = 1.4426950408889634f;
  constexpr int kChunks = kHeadLossBlock / 32;
  static_assert(2 * kChunks == 16 && kTopKMax <= 16, "floor from 16 chunk values");
  const EpiParams& ep = a.ep;
  const int n_tok = a.M, V = a.N;
  const int row = row0 + lane;
  if (ncol0 >= V) return;  // a half tile past the vocabulary (warp-uniform)
  const int n_live = min(kHeadLossBlock, V - ncol0);  // entries below V
  const int n_chunks = (n_live + 31) / 32;
  float* srow = stage + lane * 33;
  // Pass 1: the chunks' two largest entries, shifted in at the front.
  float top[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) top[j] = -INFINITY;
  for (int c = 0; c < n_chunks; ++c) {
    uint32_t r[32];
    tmem_ld_32x32b_x32(tbase + static_cast<uint32_t>(32 * c), r);
    tmem_ld_wait();
    float m1 = -INFINITY, m2 = -INFINITY;
    if (32 * c + 32 <= n_live) {
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const float v = __uint_as_float(r[i]);
        m2 = fmaxf(m2, fmin_nan(m1, v));
        m1 = fmaxf(m1, v);
      }
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const float v = 32 * c + i < n_live ? __uint_as_float(r[i]) : -INFINITY;
        m2 = fmaxf(m2, fmin_nan(m1, v));
        m1 = fmaxf(m1, v);
      }
    }
#pragma unroll
    for (int j = 15; j >= 2; --j) top[j] = top[j - 2];
    top[0] = m1;
    top[1] = m2;
  }
  sort16_desc(top);
  const float m = top[0];
  float thr = top[0];  // top[k - 1], as the least of the first k (no indexed read)
#pragma unroll
  for (int j = 1; j < kTopKMax; ++j) thr = j < ep.topk_k ? fminf(thr, top[j]) : thr;
  thr = fmaxf(thr, -3.402823466e38f);  // never -inf: -inf entries are no candidates
  // Pass 2: the sum, and the candidates.
  float tv[kTopKMax];
  int ti[kTopKMax];
#pragma unroll
  for (int j = 0; j < kTopKMax; ++j) {
    tv[j] = -INFINITY;
    ti[j] = 0x7fffffff;
  }
  const float ml = m * kL2e;
  float s4[4] = {0.f, 0.f, 0.f, 0.f};
  for (int c = 0; c < n_chunks; ++c) {
    const int col0 = ncol0 + 32 * c;
    uint32_t r[32];
    tmem_ld_32x32b_x32(tbase + static_cast<uint32_t>(32 * c), r);
    tmem_ld_wait();
    uint32_t mask = 0u;
    if (32 * c + 32 <= n_live) {
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const float v = __uint_as_float(r[i]);
        s4[i & 3] += ex2(fmaf(v, kL2e, -ml));
        mask |= (v >= thr ? 1u : 0u) << i;
      }
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const float v = __uint_as_float(r[i]);
        const bool live = 32 * c + i < n_live;
        if (live) s4[i & 3] += ex2(fmaf(v, kL2e, -ml));
        mask |= (live && v >= thr ? 1u : 0u) << i;
      }
    }
    if (__any_sync(0xffffffffu, mask != 0u)) {
#pragma unroll
      for (int i = 0; i < 32; ++i) srow[i] = __uint_as_float(r[i]);
      __syncwarp();
      while (mask) {
        const int i = __ffs(mask) - 1;
        mask &= mask - 1u;
        const float v = srow[i];
        const int id = col0 + i;
        bool gt[kTopKMax];
#pragma unroll
        for (int j = 0; j < kTopKMax; ++j) gt[j] = v > tv[j];
#pragma unroll
        for (int j = kTopKMax - 1; j > 0; --j) {
          tv[j] = gt[j] ? (gt[j - 1] ? tv[j - 1] : v) : tv[j];
          ti[j] = gt[j] ? (gt[j - 1] ? ti[j - 1] : id) : ti[j];
        }
        tv[0] = gt[0] ? v : tv[0];
        ti[0] = gt[0] ? id : ti[0];
      }
      __syncwarp();  // the stage is read before the next chunk overwrites it
    }
  }
  if (row < n_tok) {
    const size_t vb = static_cast<size_t>(ncol0 / kHeadLossBlock);
    ep.part_m[vb * n_tok + row] = m;
    ep.part_s[vb * n_tok + row] = (s4[0] + s4[1]) + (s4[2] + s4[3]);
    // The token's kTopKMax candidates contiguous (32 bytes each for values and
    // ids): the warp's 32 tokens write 1 KB runs.
    static_assert(kTopKMax == 8, "two 16-byte stores per list");
    float4* dv = reinterpret_cast<float4*>(ep.topk_v + (vb * n_tok + row) * kTopKMax);
    int4* di = reinterpret_cast<int4*>(ep.topk_i + (vb * n_tok + row) * kTopKMax);
    dv[0] = make_float4(tv[0], tv[1], tv[2], tv[3]);
    dv[1] = make_float4(tv[4], tv[5], tv[6], tv[7]);
    di[0] = make_int4(ti[0], ti[1], ti[2], ti[3]);
    di[1] = make_int4(ti[4], ti[5], ti[6], ti[7]);
  }
}

// Epilogue of one warp's share of a tile: rows row0 .. row0+31 (this thread:
// row0 + lane), columns ncol0 .. ncol0+ncols-1, accumulator at TMEM tbase.
template <int KIND>
__device__ __forceinline__ void epilogue_tile(uint32_t tbase, int row0, int ncol0, int ncols,
                                              int lane, uint8_t* epi, const uint16_t* bias_s,
                                              uint64_t* rbar, EpiState& s, const GemmArgs& a,
                                              const CUtensorMap* tmO, const CUtensorMap* tmR,
                                              const CUtensorMap* tmQ, const CUtensorMap* tmKV,
                                              volatile int* abort_flag) {
  const EpiParams& ep = a.ep;
  const int M = a.M, N = a.N;
  const int row = row0 + lane;
  const bool row_ok = row < M;
  const int seg_end = min(ncols, N - ncol0);  // valid columns of this warp's segment
  int qkv_b = 0, qkv_t = 0;
  if constexpr (KIND == kEpiQkv) {
    qkv_b = row / ep.T;
    qkv_t = row - qkv_b * ep.T;
  }
  uint32_t mag = 0u;  // kEpiGelu, fp16 output: largest magnitude (fp16 bits) written
  for (int c = 0; c < seg_end; c += 32) {
    const int col = ncol0 + c;
    uint32_t r[32];
    const size_t off = static_cast<size_t>(row) * ep.ldo + col;

    if constexpr (KIND == kEpiLogitsT) {
      // Transposed accumulator (the head computed as W_e H^T): this thread's
      // TMEM lane is vocabulary entry `row`, the chunk's 32 columns are 32
      // consecutive tokens, so for each token the warp writes 32 consecutive
      // logits of one row with one store, straight from registers.
      tmem_ld_32x32b_x32(tbase + static_cast<uint32_t>(c), r);
      tmem_ld_wait();
      const int nt = min(32, N - col);  // tokens in this chunk
      if (row_ok) {
        float* o = static_cast<float*>(ep.out) + static_cast<size_t>(col) * ep.ldo + row;
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (j < nt) o[static_cast<size_t>(j) * ep.ldo] = __uint_as_float(r[j]);
      }
    } else if constexpr (KIND == kEpiLogits) {
      // fp32 logits rows are only 4-byte aligned: transpose the chunk through
      // shared memory so each store instruction writes 32 consecutive columns
      // of one row.
      tmem_ld_32x32b_x32(tbase + static_cast<uint32_t>(c), r);
      tmem_ld_wait();
      float* st = reinterpret_cast<float*>(epi);
#pragma unroll
      for (int j = 0; j < 32; ++j) st[lane * kLogitsLd + j] = __uint_as_float(r[j]);
      __syncwarp();
      float* out = static_cast<float*>(ep.out);
      const int ccol = col + lane;
      if (ccol < N) {
#pragma unroll 8
        for (int rr = 0; rr < 32; ++rr) {
          const int rrow = row0 + rr;
          if (rrow < M) out[static_cast<size_t>(rrow) * ep.ldo + ccol] = st[rr * kLogitsLd + lane];
        }
      }
      __syncwarp();
    } else {
      const int slot = s.chunk & 1;
      ++s.chunk;
      uint8_t* rb = epi + slot * slot_bytes(KIND);
      uint8_t* ob = rb + (uses_rbuf(KIND) ? kRBuf : 0);
      const bool tma_store_path = (KIND == kEpiQkv) ? a.tma_qkv != 0 : a.tma_out != 0;
      constexpr bool kFp32Resid = KIND == kEpiResidF32 || KIND == kEpiResidBf16Out;
      // bf16 for Q/K/V and the block output; the caller's choice for the others.
      const bool out16 = (KIND == kEpiBias || KIND == kEpiGelu) && a.out_f16 != 0;
      const bool tma_resid = kFp32Resid && a.tma_resid != 0;
      if (tma_store_path) {
        // The TMA store that last used this slot must be done reading it.
        if (lane == 0) bulk_wait_group_read<1>();
        __syncwarp();
      }
      if (KIND == kEpiResidF32 && tma_resid && c >= 64 && lane == 0) {
        resid_load(rb, &rbar[slot], tmR, col, row0);
        s.inflight |= 1u << slot;
      }
      tmem_ld_32x32b_x32(tbase + static_cast<uint32_t>(c), r);
      const bool full = (col + 32 <= N) && a.vec_ok;
      float rv[32];
      if constexpr (kFp32Resid) {
        if (!tma_resid) {
          const float* rp = static_cast<const float*>(ep.resid) + off;
          if (full && row_ok) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const float4 v = reinterpret_cast<const float4*>(rp)[i];
              rv[4 * i] = v.x; rv[4 * i + 1] = v.y; rv[4 * i + 2] = v.z; rv[4 * i + 3] = v.w;
            }
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) rv[j] = (row_ok && col + j < N) ? rp[j] : 0.f;
          }
        }
      } else if constexpr (KIND == kEpiResidBf16In) {
#pragma unroll
        for (int i = 0; i < 4; ++i) unpack8(s.rnext[i], rv + 8 * i);
        if (c + 32 < seg_end) resid16_fetch(a, row, col + 32, s.rnext);
      }
      float bv[32];
#pragma unroll
      for (int i = 0; i < 4; ++i) unpack8(*reinterpret_cast<const uint4*>(bias_s + c + 8 * i), bv + 8 * i);
      tmem_ld_wait();
      if (tma_resid) {
        // A wait that runs out ends this tile's epilogue: the load stays
        // marked in flight, and the CTA's final drain waits for it.
        if (!mbar_wait_bounded(&rbar[slot], (s.rpar >> slot) & 1u, abort_flag, a.err, a.wait_ns))
          return;
        s.rpar ^= 1u << slot;
        s.inflight &= ~(1u << slot);
        box_read_f32(rb, lane, rv);
        if constexpr (KIND == kEpiResidBf16Out) {
          // The box is free again: fetch the residual of chunk c+2 into it.
          __syncwarp();
          if (c + 64 < seg_end && lane == 0) {
            resid_load(rb, &rbar[slot], tmR, col + 64, row0);
            s.inflight |= 1u << slot;
          }
        }
      }
      float v[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]) + bv[j];
      if constexpr (KIND == kEpiGelu) {
        if (out16) {
          // fp16 output: GELU on packed pairs (half the instructions), the
          // result already in its stored form.
          uint32_t w[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            w[i] = gelu_tanh_f16x2(v[2 * i], v[2 * i + 1]);
            mag = fp16_max_mag(mag, w[i]);
          }
          if (tma_store_path) {
            box_write_packed(ob, lane, w);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_2d(tmO, ob, col, row0);
              bulk_commit_group();
            }
          } else if (row_ok) {
            uint16_t* o = static_cast<uint16_t*>(ep.out) + off;
            if (full) {
#pragma unroll
              for (int i = 0; i < 4; ++i)
                reinterpret_cast<uint4*>(o)[i] =
                    make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
            } else {
#pragma unroll
              for (int j = 0; j < 32; ++j)
                if (col + j < N) o[j] = static_cast<uint16_t>(w[j >> 1] >> (16 * (j & 1)));
            }
          }
          continue;
        }
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = gelu_tanh_approx(v[j]);
      }
      if constexpr (uses_rbuf(KIND)) {
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] += rv[j];
      }

      if (tma_store_path) {
        if constexpr (uses_obuf(KIND)) box_write_16(ob, lane, v, out16);
        else box_write_f32(rb, lane, v);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          if constexpr (KIND == kEpiQkv) {
            // 64-column chunks of c_attn's output are one of Q/K/V and one head;
            // the 32 rows are 32 consecutive tokens of one sequence.
            const int which = col / ep.d;
            const int head = (col - which * ep.d) >> 6;
            const int dim0 = col & 63;
            const int b0 = row0 / ep.T, t0 = row0 - b0 * ep.T;
            if (which == 0)
              tma_store_3d(tmQ, ob, dim0, t0, b0 * (ep.d >> 6) + head);
            else
              tma_store_3d(tmKV, ob, dim0, ep.kv.t_past + t0,
                           b0 * a.kv_z_per_seq + (which - 1) * (ep.d >> 6) + head);
          } else {
            tma_store_2d(tmO, uses_obuf(KIND) ? static_cast<const void*>(ob) : rb, col, row0);
          }
          bulk_commit_group();
        }
      } else if constexpr (KIND == kEpiQkv) {
        const int which = col / ep.d;
        const int head = (col - which * ep.d) >> 6;
        const int dim0 = col & 63;
        bf16* dst;
        if (which == 0) {
          dst = static_cast<bf16*>(ep.q) +
                ((static_cast<size_t>(qkv_b) * (ep.d >> 6) + head) * ep.T + qkv_t) * 64 + dim0;
        } else {
          dst = static_cast<bf16*>(ep.kv.base) + qkv_b * ep.kv.s_batch + (which - 1) * ep.kv.s_kv +
                head * ep.kv.s_head + static_cast<long long>(ep.kv.t_past + qkv_t) * 64 + dim0;
        }
        if (row_ok) store32_16(dst, v, false);
      } else if constexpr (uses_obuf(KIND)) {
        uint16_t* o = static_cast<uint16_t*>(ep.out) + off;
        if (full && row_ok) {
          store32_16(o, v, out16);
        } else if (row_ok) {
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (col + j < N) o[j] = static_cast<uint16_t>(pack_16x2(v[j], 0.f, out16) & 0xFFFFu);
        }
      } else {
        float* o = static_cast<float*>(ep.out) + off;
        if (full && row_ok) {
#pragma unroll
          for (int i = 0; i < 8; ++i)
            reinterpret_cast<float4*>(o)[i] =
                make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
        } else if (row_ok) {
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (col + j < N) o[j] = v[j];
        }
      }
    }
  }
  if constexpr (KIND == kEpiGelu) {
    // An fp16 GELU output past 65504 (or not finite) would feed the next
    // product: report it (the rows past M hold zeros).
    if (__any_sync(0xffffffffu, fp16_nonfinite(mag)) && lane == 0) raise_error(a.err, kErrRange);
  }
}

// CG = 1: one CTA per tile of 128 x BN.  CG = 2: a cluster of two CTAs per
// tile of 256 x BN; each CTA loads its 128 rows of A and half of the tile's B
// rows into its own shared memory, both CTAs' copies complete on the first
// CTA's stage barrier, the first CTA issues the pair MMA, and each CTA's
// epilogue drains its own 128 accumulator rows.
template <int KIND, int CG>
__global__ void __launch_bounds__(epi_threads(KIND), 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmO, const __grid_constant__ CUtensorMap tmR,
                   const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmKV,
                   const GemmArgs args) {
  constexpr int kEpiWarps = epi_warps(KIND);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const int BN = args.BN, S = args.stages;
  const uint32_t b_bytes = static_cast<uint32_t>(BN / CG) * kBK * 2;  // this CTA's B rows
  uint8_t* sA = smem;
  uint8_t* sB = smem + static_cast<size_t>(S) * kABytes;
  uint8_t* sEpi = sB + static_cast<size_t>(S) * b_bytes;
  uint64_t* bars =
      reinterpret_cast<uint64_t*>(sEpi + static_cast<size_t>(kEpiWarps) * epi_warp_bytes(KIND) +
                                  epi_bias_bytes(KIND));
  uint64_t* full = bars;                  // [S]   TMA landed (pair: both CTAs', first CTA's barrier)
  uint64_t* empty = bars + S;             // [S]   slot consumed by the MMAs
  uint64_t* tfull = bars + 2 * S;         // [2]   accumulator ready
  uint64_t* tempty = bars + 2 * S + 2;    // [2]   accumulator drained (pair: both CTAs)
  uint64_t* mma_done = bars + 2 * S + 4;  // [1]   every issued MMA retired
  uint64_t* rbars = bars + 2 * S + 5;     // [8][2] residual loads of the epilogue warps
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(rbars + 2 * kEpiWarps);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int KB = (args.K + kBK - 1) / kBK;
  const uint32_t rank = CG == 2 ? cluster_ctarank() : 0u;
  const int first_tile = CG == 2 ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
  const int tile_step = CG == 2 ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);
  const int tile_rows = kBM * CG;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&tfull[i], 1);
      mbar_init(&tempty[i], (acc_groups(KIND) ? 4 : kEpiWarps) * CG);
    }
    mbar_init(mma_done, 1);
    for (int i = 0; i < 2 * kEpiWarps; ++i) mbar_init(&rbars[i], 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 2) {
    if constexpr (CG == 2) {
      tmem_alloc_pair(tmem_slot, kTmemCols);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(tmem_slot, kTmemCols);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  __syncthreads();
  if constexpr (CG == 2) cluster_sync();  // both CTAs' barriers exist before any remote use
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // Set-up above touched only shared memory and TMEM: let the next kernel
  // launch, then wait for the previous one before any global access.
  pdl_trigger();
  pdl_wait();

  if (warp == 0 && lane == 0) {
    // ---------------------------------------------------------- producer --
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    uint32_t issued = 0u, issued_par = 0u;  // bit s: slot s has a load issued / its parity
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    const uint32_t full0 = CG == 2 ? mapa_shared(smem_u32(full), 0u) : 0u;  // first CTA's barriers
    for (int tile = first_tile; ok && tile < args.num_tiles; tile += tile_step) {
      int m_blk, n_blk;
      tile_coords(args, tile, m_blk, n_blk);
      const int a_row = m_blk * tile_rows + static_cast<int>(rank) * kBM;
      const int b_row = n_blk * BN + static_cast<int>(rank) * (BN / CG);
      for (int kb = 0; kb < KB; ++kb) {
        if (!mbar_wait_bounded(&empty[stage], phase ^ 1u, abort_flag, args.err, args.wait_ns)) {
          ok = false;
          break;
        }
        if constexpr (CG == 2) {
          // The first CTA's barrier counts both CTAs' bytes; only it arrives.
          const uint32_t bar = full0 + stage * static_cast<uint32_t>(sizeof(uint64_t));
          if (rank == 0) mbar_arrive_expect_tx(&full[stage], 2u * (kABytes + b_bytes));
          tma_load_2d_pair(sA + static_cast<size_t>(stage) * kABytes, &tmA, bar, kb * kBK, a_row);
          tma_load_2d_pair(sB + static_cast<size_t>(stage) * b_bytes, &tmB, bar, kb * kBK, b_row);
        } else {
          mbar_arrive_expect_tx(&full[stage], kABytes + b_bytes);
          tma_load_2d(sA + static_cast<size_t>(stage) * kABytes, &tmA, &full[stage], kb * kBK, a_row);
          tma_load_2d(sB + static_cast<size_t>(stage) * b_bytes, &tmB, &full[stage], kb * kBK, b_row);
        }
        issued |= 1u << stage;
        issued_par = (issued_par & ~(1u << stage)) | (phase << stage);
        if (++stage == S) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    if (!ok && rank == 0) {
      // Drain: every copy already issued must land before the CTA exits.
      for (int s = 0; s < S; ++s)
        if ((issued >> s) & 1u)
          mbar_wait_bounded(&full[s], (issued_par >> s) & 1u, nullptr, args.err);
    } else if (!ok) {
      // A pair's second CTA cannot wait on the first CTA's barriers, which
      // count its copies: it lets 50 us pass (a copy lands within
      // microseconds) before going on to the closing cluster barrier.
      const unsigned long long t0 = global_timer_ns();
      while (global_timer_ns() - t0 < 50000ull) __nanosleep(1000);
    }
  } else if (warp == 1 && lane == 0 && rank == 0) {
    // ------------------------------------------------------- MMA issuer --
    const uint32_t idesc = args.idesc;
    int stage = 0;
    uint32_t phase = 0;
    int it = 0;
    bool ok = true;
    for (int tile = first_tile; ok && tile < args.num_tiles; tile += tile_step, ++it) {
      const int acc = it & 1;
      const uint32_t acc_par = static_cast<uint32_t>((it >> 1) & 1);
      if (!mbar_wait_bounded(&tempty[acc], acc_par ^ 1u, abort_flag, args.err, args.wait_ns))
        break;
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * 256);
      for (int kb = 0; kb < KB; ++kb) {
        if (!mbar_wait_bounded(&full[stage], phase, abort_flag, args.err, args.wait_ns)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t a_desc = sdesc_k_sw128(smem_u32(sA + static_cast<size_t>(stage) * kABytes));
        const uint64_t b_desc = sdesc_k_sw128(smem_u32(sB + static_cast<size_t>(stage) * b_bytes));
#pragma unroll
        for (int k = 0; k < kBK / 16; ++k) {
          // +32 bytes per 16-element K slice: +2 in the descriptor's address field.
          if constexpr (CG == 2)
            umma_f16kind_pair(d_tmem, a_desc + 2 * k, b_desc + 2 * k, idesc, (kb | k) != 0 ? 1u : 0u);
          else
            umma_f16kind(d_tmem, a_desc + 2 * k, b_desc + 2 * k, idesc, (kb | k) != 0 ? 1u : 0u);
        }
        if constexpr (CG == 2) umma_commit_pair(&empty[stage], 3);
        else umma_commit(&empty[stage]);
        if (++stage == S) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (ok) {
        if constexpr (CG == 2) umma_commit_pair(&tfull[acc], 3);
        else umma_commit(&tfull[acc]);
      }
    }
    // Every MMA issued above must retire before TMEM is freed.
    if constexpr (CG == 2) umma_commit_pair(mma_done, 1);
    else umma_commit(mma_done);
    mbar_wait_bounded(mma_done, 0, nullptr, args.err);
  } else if (warp >= 4) {
    // --------------------------------------------------------- epilogue --
    // Warp w may read TMEM lanes 32*(w%4) .. +31; the two warps of a lane
    // quarter split the tile's columns in halves, or (accumulator groups)
    // each takes every other tile, all its columns.  What does not depend on
    // the accumulator is fetched before waiting for it.
    constexpr bool kGroups = acc_groups(KIND);
    const int e = warp - 4;
    const int quarter = warp & 3;
    const int half = kGroups ? 0 : e >> 2;     // column segment
    const int group = kGroups ? e >> 2 : 0;    // accumulator (tiles it, it % 2 == group)
    const int ncols = kGroups ? BN : BN / (kEpiWarps / 4);
    uint8_t* epi = sEpi + static_cast<size_t>(e) * epi_warp_bytes(KIND);
    uint16_t* bias_half = reinterpret_cast<uint16_t*>(sEpi + kEpiWarps * epi_warp_bytes(KIND)) +
                          half * kBiasBufs * (256 / (kEpiWarps / 4));
    uint64_t* rbar = rbars + 2 * e;
    EpiState st;
    st.chunk = 0;
    st.rpar = 0u;
    st.inflight = 0u;
    if (lane == 0) {
      if (args.tma_out) tma_prefetch_desc(&tmO);
      if (args.tma_resid) tma_prefetch_desc(&tmR);
    }
    // The accumulator-drained barrier lives in the pair's first CTA.
    const uint32_t tempty_addr = CG == 2 ? mapa_shared(smem_u32(tempty), 0u) : 0u;
    const int it_step = kGroups ? 2 : 1;
    int it = group;
    for (int tile = first_tile + group * tile_step; tile < args.num_tiles;
         tile += it_step * tile_step, it += it_step) {
      const int acc = it & 1;
      const uint32_t acc_par = static_cast<uint32_t>((it >> 1) & 1);
      int m_blk, n_blk;
      tile_coords(args, tile, m_blk, n_blk);
      const int row0 = m_blk * tile_rows + static_cast<int>(rank) * kBM + quarter * 32;
      const int ncol0 = n_blk * BN + half * ncols;
      uint16_t* bias_s = bias_half + (it % kBiasBufs) * (256 / (kEpiWarps / 4));
      if (*abort_flag) break;  // a wait of this CTA ran out: no new loads
      epilogue_prefetch<KIND>(row0, ncol0, ncols, lane, epi, bias_s, rbar, st, args, &tmR);
      if (!mbar_wait_bounded(&tfull[acc], acc_par, abort_flag, args.err, args.wait_ns)) break;
      tc_fence_after();
      const uint32_t tbase = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                             static_cast<uint32_t>(acc * 256 + half * ncols);
      if constexpr (KIND == kEpiHeadLoss) {
        head_loss_rows(tbase, row0, ncol0, lane, args);
      } else if constexpr (KIND == kEpiHeadTopK) {
        head_topk_rows(tbase, row0, ncol0, lane, args, reinterpret_cast<float*>(epi));
      } else {
        epilogue_tile<KIND>(tbase, row0, ncol0, ncols, lane, epi, bias_s, rbar, st, args, &tmO,
                            &tmR, &tmQ, &tmKV, abort_flag);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if constexpr (CG == 2)
          mbar_arrive_cluster(tempty_addr + acc * static_cast<uint32_t>(sizeof(uint64_t)));
        else
          mbar_arrive(&tempty[acc]);
      }
    }
    // Residual loads still in flight (after an abort) must land, and every TMA
    // store must be complete, before the CTA's shared memory goes.
    if (lane == 0) {
      for (int sl = 0; sl < 2; ++sl)
        if ((st.inflight >> sl) & 1u)
          mbar_wait_bounded(&rbar[sl], (st.rpar >> sl) & 1u, nullptr, args.err);
      bulk_wait_group<0>();
    }
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  // Pair: the partner's shared memory and TMEM stay in use (remote arrivals,
  // MMAs of the first CTA) until both CTAs get here.
  if constexpr (CG == 2) cluster_sync();
  tc_fence_after();
  if (warp == 2) {
    if constexpr (CG == 2) tmem_dealloc_pair(tmem_base, kTmemCols);
    else tmem_dealloc(tmem_base, kTmemCols);
  }
}

template <int KIND>
void* kernel_ptr(int cg) {
  return cg == 2 ? reinterpret_cast<void*>(&gemm_tc_kernel<KIND, 2>)
                 : reinterpret_cast<void*>(&gemm_tc_kernel<KIND, 1>);
}

void* kernel_for(int kind, int cg) {
  switch (kind) {
    case kEpiBias: return kernel_ptr<kEpiBias>(cg);
    case kEpiGelu: return kernel_ptr<kEpiGelu>(cg);
    case kEpiResidF32: return kernel_ptr<kEpiResidF32>(cg);
    case kEpiResidBf16In: return kernel_ptr<kEpiResidBf16In>(cg);
    case kEpiResidBf16Out: return kernel_ptr<kEpiResidBf16Out>(cg);
    case kEpiLogits: return kernel_ptr<kEpiLogits>(cg);
    case kEpiLogitsT: return kernel_ptr<kEpiLogitsT>(cg);
    case kEpiHeadLoss: return kernel_ptr<kEpiHeadLoss>(cg);
    case kEpiHeadTopK: return kernel_ptr<kEpiHeadTopK>(cg);
    case kEpiQkv: return kernel_ptr<kEpiQkv>(cg);
    default: return nullptr;
  }
}

bool encode_kmajor_16(const LaunchEnv& env, CUtensorMap* map, const void* base, int rows, int K,
                      int box_rows, bool f16) {
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * 2};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(kBK), static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = env.encode(map,
                                f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                    : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                                2, const_cast<void*>(base), dims, strides, box, estr,
                                CU_TENSOR_MAP_INTERLEAVE_NONE,
                                CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// A [rows, cols] row-major matrix with row stride ld elements, boxes of 32 x 32;
// fp32, or 16-bit (fp16 when f16, else bf16).
bool encode_box32(const LaunchEnv& env, CUtensorMap* map, const void* base, bool fp32, int rows,
                  int cols, int ld, bool f16 = false) {
  const size_t es = fp32 ? 4 : 2;
  if (!aligned16(base) || (static_cast<size_t>(ld) * es) % 16 != 0) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * es};
  const cuuint32_t box[2] = {32, 32};
  const cuuint32_t estr[2] = {1, 1};
  return env.encode(map,
                    fp32  ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                    : f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                          : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                    2, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE,
                    fp32 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                    CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

// Head-major bf16 rows of 64: dims {64, tokens, z}, token stride 128 B, z
// stride z_stride elements; boxes of 32 dims x 32 tokens x 1.
bool encode_heads(const LaunchEnv& env, CUtensorMap* map, const void* base, long long tokens,
                  long long z, long long z_stride) {
  if (!aligned16(base) || (z_stride * 2) % 16 != 0) return false;
  const cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(tokens), static_cast<cuuint64_t>(z)};
  const cuuint64_t strides[2] = {128, static_cast<cuuint64_t>(z_stride) * 2};
  const cuuint32_t box[3] = {32, 32, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return env.encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims,
                    strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                    CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

// Tile width: the candidate minimising waves x (width cost + 32): the busiest
// SM's (or CTA pair's) share of the work plus a per-tile cost (operand
// reloads, epilogue start), preferring wider tiles on ties.  Tiles have
// tile_rows rows and `units` of them run at once.  Narrow MMAs do less work
// per cycle, so a tile's width cost is its time relative to a 256-wide one,
// fitted to GB300 timings of the GPT-2-small products in 256-, 192- and
// 128-wide tiles (e.g. c_fc: 34.9, 37.0 and 50.1 us).
int choose_bn(int M, int N, int tile_rows, int units) {
  const int num_sms = units;
  const int m_blocks = (M + tile_rows - 1) / tile_rows;
  int best = 256;
  long long best_cost = -1;
  for (int bn : {256, 192, 128, 64}) {
    const long long tiles = static_cast<long long>(m_blocks) * ((N + bn - 1) / bn);
    const long long waves = (tiles + num_sms - 1) / num_sms;
    const int width_cost = bn == 256 ? 256 : bn == 192 ? 235 : bn == 128 ? 190 : 120;
    const long long cost = waves * (width_cost + 32);
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best = bn;
    }
  }
  return best;
}

}  // namespace

int launch_gemm_tc(const LaunchEnv& env, int kind_in, const void* A_in, const void* W_in,
                   int M_in, int N_in, int K, const EpiParams& ep, cudaStream_t stream,
                   double* flops, double* bytes, bool operands_f16, bool out_f16) {
  if (M_in <= 0 || N_in <= 0 || K <= 0 || kind_in < 0 || kind_in == kEpiLogitsT ||
      kind_in >= kEpiCount)
    return GPT2_ERR_INVALID_ARG;
  if (K % 8 != 0) return GPT2_ERR_UNSUPPORTED;
  const bool reduced_head = kind_in == kEpiHeadLoss || kind_in == kEpiHeadTopK;
  if (kind_in != kEpiLogits && !reduced_head && (N_in % 2 != 0))
    return GPT2_ERR_UNSUPPORTED;
  if (kind_in == kEpiQkv && (ep.d % 64 != 0 || N_in != 3 * ep.d)) return GPT2_ERR_UNSUPPORTED;
  // The tied head that writes logits runs transposed, logits^T = W_e H^T:
  // vocabulary entries on the TMEM lanes and tokens on the columns, so the
  // epilogue stores each token's logits row segment straight from registers;
  // the tile index runs over token blocks first, so each block of W_e is
  // streamed from HBM once.  The head reduced to the loss keeps tokens on the
  // lanes (each thread reduces its own token's entries); its tile index runs
  // over token blocks first by the default order, with the same effect.
  int kind = kind_in, M = M_in, N = N_in;
  const void* A = A_in;
  const void* W = W_in;
  const bool transposed = kind_in == kEpiLogits;
  const bool head = transposed || reduced_head;
  if (transposed) {
    if (kind_in == kEpiLogits) kind = kEpiLogitsT;
    std::swap(A, W);
    std::swap(M, N);
  }
  // CTA pairs (256-row tiles on two SMs, each holding half of B) where the
  // mainloop is long enough to gain from halving each SM's operand traffic
  // (measured on GB300: faster from K = 1600 up, no gain at K = 768), and for
  // the transposed head, whose 256-entry vocabulary tiles give each token row
  // 1 KB of contiguous logits per tile (GPT-2-small head 564 -> 542 us).
  const int cg =
      (M > kBM && (K >= 1024 || head) && env.num_sms >= 2) ? 2 : 1;
  void* fn = kernel_for(kind, cg);
  if (!fn) return GPT2_ERR_INVALID_ARG;

  const int units = cg == 2 ? env.num_sms / 2 : env.num_sms;
  // The loss epilogue's partials cover one whole tile's kHeadLossBlock entries.
  const int BN = reduced_head ? kHeadLossBlock : choose_bn(M, N, kBM * cg, units);
  int stages = kMaxStages;
  while (stages > 2 && smem_bytes_for(kind, BN, stages, cg) > static_cast<size_t>(kSmemLimit))
    --stages;
  const size_t smem = smem_bytes_for(kind, BN, stages, cg);

  CUtensorMap tmA, tmB, tmO, tmR, tmQ, tmKV;
  memset(&tmO, 0, sizeof(tmO));
  memset(&tmR, 0, sizeof(tmR));
  memset(&tmQ, 0, sizeof(tmQ));
  memset(&tmKV, 0, sizeof(tmKV));
  if (!encode_kmajor_16(env, &tmA, A, M, K, kBM, operands_f16)) return GPT2_ERR_CUDA;
  if (!encode_kmajor_16(env, &tmB, W, N, K, BN / cg, operands_f16)) return GPT2_ERR_CUDA;

  GemmArgs args;
  args.M = M;
  args.N = N;
  args.K = K;
  args.BN = BN;
  args.stages = stages;
  args.num_m_blocks = (M + kBM * cg - 1) / (kBM * cg);
  args.num_n_blocks = (N + BN - 1) / BN;
  args.n_inner = transposed ? 1 : 0;
  args.num_tiles = args.num_m_blocks * args.num_n_blocks;
  args.vec_ok = (kind == kEpiResidF32 || kind == kEpiResidBf16In) ? (ep.ldo % 4 == 0)
                                                                  : (ep.ldo % 8 == 0);
  args.tma_out = 0;
  args.tma_resid = 0;
  args.tma_qkv = 0;
  args.kv_z_per_seq = 0;
  args.out_f16 = out_f16 ? 1 : 0;
  args.idesc = umma_idesc_16(kBM * cg, BN, operands_f16);
  args.err = env.err;
  args.wait_ns = env.wait_ns;
  args.ep = ep;
  if (kind == kEpiBias || kind == kEpiGelu)
    args.tma_out = encode_box32(env, &tmO, ep.out, false, M, N, ep.ldo, out_f16);
  else if (kind == kEpiResidBf16Out)
    args.tma_out = encode_box32(env, &tmO, ep.out, false, M, N, ep.ldo);
  else if (kind == kEpiResidF32 || kind == kEpiResidBf16In)
    args.tma_out = encode_box32(env, &tmO, ep.out, true, M, N, ep.ldo);
  if (kind == kEpiResidF32 || kind == kEpiResidBf16Out)
    args.tma_resid = encode_box32(env, &tmR, ep.resid, true, M, N, ep.ldo);
  if (kind == kEpiQkv && ep.T % 32 == 0 && M % ep.T == 0) {
    // Q [B*h, T, 64]; the cache of this layer as rows of heads: z = b *
    // (heads per sequence in the cache layout) + kv * h + head.
    const int h = ep.d / 64;
    const long long B = M / ep.T;
    const long long z_per_seq = ep.kv.s_batch / ep.kv.s_head;
    const long long t_cap = ep.kv.s_head / 64;
    args.kv_z_per_seq = static_cast<int>(z_per_seq);
    args.tma_qkv = encode_heads(env, &tmQ, ep.q, ep.T, B * h, static_cast<long long>(ep.T) * 64) &&
                   encode_heads(env, &tmKV, ep.kv.base, t_cap, (B - 1) * z_per_seq + 2 * h,
                                ep.kv.s_head);
  }

  // The opt-in limit does not depend on the call: set once per device.
  if (!ensure_smem_limit(fn, kSmemLimit)) return GPT2_ERR_CUDA;
  const int grid = std::min(args.num_tiles, units) * cg;
  void* params[] = {&tmA, &tmB, &tmO, &tmR, &tmQ, &tmKV, &args};
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(static_cast<unsigned>(epi_threads(kind)));
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = take_pdl_permission() ? 1 : 0;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = static_cast<unsigned>(cg);
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  if (cudaLaunchKernelExC(&cfg, fn, params) != cudaSuccess) return GPT2_ERR_CUDA;

  if (flops) *flops = 2.0 * M_in * N_in * static_cast<double>(K);
  if (bytes) {
    double b = 2.0 * (static_cast<double>(M_in) * K + static_cast<double>(N_in) * K);
    const double mn = static_cast<double>(M_in) * N_in;
    switch (kind_in) {
      case kEpiBias: case kEpiGelu: case kEpiQkv: b += 2.0 * mn + 2.0 * N; break;
      case kEpiResidF32: b += 8.0 * mn + 2.0 * N; break;
      case kEpiResidBf16In: b += 6.0 * mn + 2.0 * N; break;
      case kEpiResidBf16Out: b += 6.0 * mn + 2.0 * N; break;
      case kEpiLogits: b += 4.0 * mn; break;
      case kEpiHeadLoss: b += 12.0 * mn / kHeadLossBlock; break;  // the per-block partials
      case kEpiHeadTopK: b += (8.0 + 8.0 * kTopKMax) * mn / kHeadLossBlock; break;
    }
    *bytes = b;
  }
  return GPT2_OK;
}

}  // namespace gpt2

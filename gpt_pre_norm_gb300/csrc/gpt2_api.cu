// gpt2_api.cu -- the C ABI: argument validation, workspace plan, and the
// launch sequence of the block, the full forward and cached decode.
//
// Block ("GPT-2 Decoder Block", "How it works"; openai/gpt-2 ``block`` on the
// "GPT-2 Transformer block" page):
//   LN1 -> c_attn [bias, split Q|K|V into heads, K/V into the cache]
//       -> causal attention (prefill) | split-KV attention (one new token)
//       -> c_proj [bias + residual]  -> LN2 -> c_fc [bias + GELU]
//       -> mlp c_proj [bias + residual]
// Full forward ("GPT-2 Full Forward Pass", "How it works"):
//   embed (wte[ids] + wpe[T_past + t]) -> L blocks on an fp32 residual stream
//       -> ln_f -> tied head (A = LN_f(H), W = wte, fp32 logits).
#include <string.h>

#include <algorithm>
#include <mutex>
#include <new>
#include <vector>

#include "device.cuh"
#include "internal.h"

using namespace gpt2;

namespace {

const char* kKindNames[kKindCount] = {
    "embed",          "layer_norm",        "gemm_c_attn",    "attention_prefill",
    "gemm_c_proj",    "gemm_c_fc",         "gemm_mlp_c_proj", "gemm_lm_head",
    "gemm_other",     "attention_decode",  "attention_decode_combine", "simt_fp32",
    "argmax",         "loss_combine"};

struct ProfRec {
  int kind;
  int kernels;  // kernel launches inside the bracket
  cudaEvent_t start, stop;
  double flops, bytes;
};

// Offsets (bytes) of the workspace regions.
struct WsPlan {
  size_t err, ln, q, kv, attn, resid, fc, partials, wconv, ids, hloss, htopk, total;
};

// Vocabulary blocks of the fused head's per-token partials (kHeadLossBlock
// entries each, one per tile of the head).
int loss_vblocks(const gpt2_hparams& hp) {
  return (hp.n_vocab + kHeadLossBlock - 1) / kHeadLossBlock;
}

// fp16 working copies of the weights (bf16 mode): per layer slot, c_attn
// [3d, d] at 0, c_proj [d, d] at 3d^2, c_fc [4d, d] at 4d^2, mlp c_proj
// [d, 4d] at 8d^2 (elements); wte after the n_layer slots.
size_t layer_slot_elems(const gpt2_hparams& hp) {
  return 12 * static_cast<size_t>(hp.n_embd) * hp.n_embd;
}

size_t align256(size_t v) { return (v + 255) & ~static_cast<size_t>(255); }

WsPlan plan_workspace(const gpt2_hparams& hp, int max_B, int max_T) {
  const size_t es = hp.dtype == GPT2_BF16 ? 2 : 4;
  const size_t M = static_cast<size_t>(max_B) * max_T;
  const size_t d = hp.n_embd;
  WsPlan p;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off += align256(bytes);
    return o;
  };
  p.err = take(256);
  p.ln = take(M * d * es);
  p.q = take(M * d * es);
  p.kv = take(2 * static_cast<size_t>(max_B) * hp.n_ctx * d * es);  // [B, 2, h, n_ctx, d_h]
  p.attn = take(M * d * es);
  p.resid = take(M * d * 4);
  p.fc = take(M * 4 * d * es);
  p.partials = take(decode_partials_floats(max_B, hp.n_head, 64) * 4);
  p.wconv = take(hp.dtype == GPT2_BF16 ? 2 * (hp.n_layer * layer_slot_elems(hp) +
                                              static_cast<size_t>(hp.n_vocab) * hp.n_embd)
                                       : 0);
  p.ids = take(static_cast<size_t>(max_B) * 4);  // greedy generation: the next token ids
  // fused head + loss (bf16 mode): target logits [M], then the partials'
  // maxima, sums and indices [vocab blocks][M]
  p.hloss = take(hp.dtype == GPT2_BF16
                     ? M * 4 * (1 + 3 * static_cast<size_t>(loss_vblocks(hp)))
                     : 0);
  // top-k head (bf16 mode): kTopKMax candidate logits and indices per (vocabulary
  // block, token); its maxima and sums share the loss partials' arrays
  p.htopk = take(hp.dtype == GPT2_BF16
                     ? M * 8 * static_cast<size_t>(kTopKMax) * loss_vblocks(hp)
                     : 0);
  p.total = off;
  return p;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

}  // namespace

struct gpt2_ctx {
  gpt2_hparams hp;
  int max_B, max_T;
  int device;
  uint8_t* ws;
  size_t ws_bytes;
  WsPlan plan;
  LaunchEnv env;
  bool prof;
  int extra_kernels;  // set by a launch function that launched more than one kernel
  bool cache_weights;  // keep fp16 weight copies across calls
  std::vector<const void*> conv_src;  // source of each converted weight (cache keys)
  std::vector<ProfRec> recs;
  std::vector<cudaEvent_t> free_events;
  long long launches[kKindCount];
  double total_ms[kKindCount], flops[kKindCount], bytes[kKindCount];

  template <typename T>
  T* at(size_t off) { return reinterpret_cast<T*>(ws + off); }

  cudaEvent_t take_event() {
    if (!free_events.empty()) {
      cudaEvent_t e = free_events.back();
      free_events.pop_back();
      return e;
    }
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    return e;
  }

  // Runs one launch function, bracketed by events when profiling.
  template <typename F>
  int run(int kind, cudaStream_t s, F&& f) {
    ProfRec r{kind, 1, nullptr, nullptr, 0.0, 0.0};
    extra_kernels = 0;
    if (prof) {
      r.start = take_event();
      r.stop = take_event();
      if (!r.start || !r.stop) return GPT2_ERR_CUDA;
      cudaEventRecord(r.start, s);
    }
    const int st = f(&r.flops, &r.bytes);
    r.kernels += extra_kernels;
    if (prof) {
      cudaEventRecord(r.stop, s);
      recs.push_back(r);
    }
    return st;
  }
};

namespace {

int validate_block_params(const gpt2_block_params* p) {
  if (!p) return GPT2_ERR_INVALID_ARG;
  const void* ptrs[12] = {p->ln1_g, p->ln1_b, p->attn_w, p->attn_b, p->proj_w, p->proj_b,
                          p->ln2_g, p->ln2_b, p->fc_w, p->fc_b, p->mlp_proj_w, p->mlp_proj_b};
  for (const void* q : ptrs) {
    if (!q) return GPT2_ERR_INVALID_ARG;
    if (!aligned16(q)) return GPT2_ERR_ALIGNMENT;
  }
  return GPT2_OK;
}

int validate_kv(const gpt2_kv* kv, bool is_present) {
  if (!kv) return GPT2_OK;
  if (!kv->data || kv->T_cap <= 0) return GPT2_ERR_INVALID_ARG;
  if (!aligned16(kv->data)) return GPT2_ERR_ALIGNMENT;
  if (!is_present && (kv->T_len < 0 || kv->T_len > kv->T_cap)) return GPT2_ERR_INVALID_ARG;
  return GPT2_OK;
}

// A cache view for one layer: strides in elements.
struct KvView {
  uint8_t* base;  // layer's base
  long long s_batch, s_kv, s_head;
  int t_cap;
};

KvView layer_view(void* data, int t_cap, int n_layers, int layer, int h, int dh, size_t es) {
  KvView v;
  const long long s_head = static_cast<long long>(t_cap) * dh;
  const long long s_kv = static_cast<long long>(h) * s_head;
  v.s_head = s_head;
  v.s_kv = s_kv;
  v.s_batch = static_cast<long long>(n_layers) * 2 * s_kv;
  v.base = static_cast<uint8_t*>(data) + static_cast<size_t>(layer) * 2 * s_kv * es;
  v.t_cap = t_cap;
  return v;
}

// Copies positions [0, t) of every (b, k/v, head) row from src to dst.
int copy_positions(const KvView& dst, const KvView& src, int B, int h, int t, int dh, size_t es,
                   cudaStream_t s) {
  if (t <= 0) return GPT2_OK;
  for (int b = 0; b < B; ++b) {
    // Rows (kv, head) of one sequence are uniformly strided by s_head.
    const uint8_t* sp = src.base + static_cast<size_t>(b) * src.s_batch * es;
    uint8_t* dp = dst.base + static_cast<size_t>(b) * dst.s_batch * es;
    if (cudaMemcpy2DAsync(dp, static_cast<size_t>(dst.s_head) * es, sp,
                          static_cast<size_t>(src.s_head) * es,
                          static_cast<size_t>(t) * dh * es, 2 * static_cast<size_t>(h),
                          cudaMemcpyDeviceToDevice, s) != cudaSuccess)
      return GPT2_ERR_CUDA;
  }
  return GPT2_OK;
}

// fp16 copies of one block's four weight matrices.
struct BlockW16 {
  const __half *attn_w, *proj_w, *fc_w, *mlp_proj_w;
};

// The fp16 copies of a block's weights in layer slot `slot`: fills `segs`
// with the conversions still to do (matrices the cache already holds are
// skipped); the LayerNorm launch in front of the block's first product runs
// them.
void block_weight_conversions(gpt2_ctx* c, int slot, const gpt2_block_params* p, BlockW16* w,
                              ConvSegs* segs) {
  const size_t d = c->hp.n_embd;
  __half* base = reinterpret_cast<__half*>(c->ws + c->plan.wconv) + slot * layer_slot_elems(c->hp);
  const void* srcs[4] = {p->attn_w, p->proj_w, p->fc_w, p->mlp_proj_w};
  const size_t offs[4] = {0, 3 * d * d, 4 * d * d, 8 * d * d};
  const size_t ns[4] = {3 * d * d, d * d, 4 * d * d, 4 * d * d};
  *segs = ConvSegs{};
  for (int i = 0; i < 4; ++i) {
    const size_t key = static_cast<size_t>(slot) * 4 + i;
    if (c->cache_weights && c->conv_src[key] == srcs[i]) continue;
    segs->src[segs->count] = static_cast<const bf16*>(srcs[i]);
    segs->dst[segs->count] = base + offs[i];
    segs->n[segs->count] = static_cast<long long>(ns[i]);
    ++segs->count;
    c->conv_src[key] = c->cache_weights ? srcs[i] : nullptr;
  }
  w->attn_w = base + offs[0];
  w->proj_w = base + offs[1];
  w->fc_w = base + offs[2];
  w->mlp_proj_w = base + offs[3];
}

// The tied embedding's fp16 copy (for the head); conversion as above.
void wte_conversion(gpt2_ctx* c, const void* wte, const __half** out, ConvSegs* segs) {
  const size_t key = static_cast<size_t>(c->hp.n_layer) * 4;
  __half* dst = reinterpret_cast<__half*>(c->ws + c->plan.wconv) +
                c->hp.n_layer * layer_slot_elems(c->hp);
  *out = dst;
  *segs = ConvSegs{};
  if (c->cache_weights && c->conv_src[key] == wte) return;
  c->conv_src[key] = c->cache_weights ? wte : nullptr;
  segs->src[0] = static_cast<const bf16*>(wte);
  segs->dst[0] = dst;
  segs->n[0] = static_cast<long long>(c->hp.n_vocab) * c->hp.n_embd;
  segs->count = 1;
}

double conversion_bytes(const ConvSegs& segs) {
  double n = 0;
  for (int i = 0; i < segs.count; ++i) n += static_cast<double>(segs.n[i]);
  return 4.0 * n;
}

// A bf16-mode product with fp16 operands: the weight-streaming kernel for a
// few rows when it implements the epilogue, else the tensor-core GEMM.
// w_early: W was made by an earlier call (see request_plain_launch).
int gemm16(gpt2_ctx* c, int kind, const void* A, const __half* W, int M, int N, int K,
           const EpiParams& e, bool out_f16, cudaStream_t s, double* fl, double* by,
           bool w_early = false) {
  const bool in_place_ok = kind != kEpiResidF32 || K <= 1024 || e.out == e.resid;
  if (smallm_supported(kind, M, K) && in_place_ok && (kind != kEpiBias || out_f16))
    return launch_gemm_smallm(c->env, kind, static_cast<const __half*>(A), W, M, N, K, e, s, fl,
                              by, w_early);
  return launch_gemm_tc(c->env, kind, A, W, M, N, K, e, s, fl, by, true, out_f16);
}

// One block on the context's workspace.  x_in: block input (mode dtype for
// the standalone block, fp32 residual stream for the full forward, in which
// case out == x_in and residual adds are in place).
int block_sequence(gpt2_ctx* c, const gpt2_block_params* p, int slot, int B, int T,
                   const void* x_in, bool x_is_stream, void* out, const KvView& kv, int t_past,
                   cudaStream_t s) {
  const gpt2_hparams& hp = c->hp;
  const int d = hp.n_embd, h = hp.n_head, dh = d / h;
  const int M = B * T;
  const bool bf = hp.dtype == GPT2_BF16;
  const int x_dtype = x_is_stream ? GPT2_FP32 : hp.dtype;
  void* ln = c->ws + c->plan.ln;
  void* q = c->ws + c->plan.q;
  void* attn = c->ws + c->plan.attn;
  float* resid = c->at<float>(c->plan.resid);
  void* fc = c->ws + c->plan.fc;
  int st = GPT2_OK;

  // bf16 mode: the GEMM operands are fp16 (activations written by the
  // producing kernels; weights converted from bf16 per call, or cached).
  BlockW16 w{};
  ConvSegs conv{};
  if (bf) block_weight_conversions(c, slot, p, &w, &conv);
  // Cached weights (every fp16 copy of this layer made by an earlier call):
  // the few-row products start their weight streams before waiting on the
  // previous kernel.  The call asked for a plain first launch (forward_trunk,
  // gpt2_block_forward), so those copies are complete.
  const bool w_early = bf && c->cache_weights && conv.count == 0;

  // LN1, with the block's weight conversion in the same launch
  st = c->run(kKindLayerNorm, s, [&](double* fl, double* by) {
    *fl = 0;
    *by = static_cast<double>(M) * d * ((x_dtype == GPT2_FP32 ? 4 : 2) + (bf ? 2 : 4)) +
          conversion_bytes(conv);
    return launch_layer_norm(hp.dtype, x_in, x_dtype, p->ln1_g, p->ln1_b, M, d, ln, s, bf,
                             conv.count ? &conv : nullptr, c->env.err);
  });
  if (st) return st;

  // c_attn -> Q and the K/V cache at positions [t_past, t_past + T)
  EpiParams e{};
  e.bias = p->attn_b;
  e.q = q;
  e.kv.base = kv.base;
  e.kv.s_batch = kv.s_batch;
  e.kv.s_kv = kv.s_kv;
  e.kv.s_head = kv.s_head;
  e.kv.t_past = t_past;
  e.T = T;
  e.d = d;
  e.ldo = 3 * d;
  st = c->run(bf ? kKindGemmQkv : kKindSimtFp32, s, [&](double* fl, double* by) {
    if (bf)
      return gemm16(c, kEpiQkv, ln, w.attn_w, M, 3 * d, d, e, false, s, fl, by, w_early);
    return launch_gemm_fp32(c->env, kEpiQkv, static_cast<const float*>(ln),
                            static_cast<const float*>(p->attn_w), M, 3 * d, d, e, dh, s);
  });
  if (st) return st;

  // Attention over the t_past + T cached positions.
  const int t_len = t_past + T;
  if (bf && T == 1 && t_past > 0) {
    const int splits = decode_splits(B, h, t_len, c->env.num_sms);
    int nl = 0;
    st = c->run(kKindDecodeAttention, s, [&](double* fl, double* by) {
      *fl = 4.0 * B * h * static_cast<double>(t_len) * dh;
      *by = static_cast<double>(B) * h * (2.0 * t_len * dh * 2 + 2.0 * dh * 2);
      const int r = launch_decode_attention_bf16(
          static_cast<const bf16*>(q), reinterpret_cast<const bf16*>(kv.base), kv.s_batch,
          kv.s_kv, kv.s_head, B, h, t_len, attn, c->at<float>(c->plan.partials), splits, s, &nl,
          true, c->env.err, c->env.wait_ns);
      c->extra_kernels = nl - 1;
      return r;
    });
  } else if (bf) {
    st = c->run(kKindAttention, s, [&](double* fl, double* by) {
      // Causal work: each query sees t_past + i + 1 keys.
      const double pairs = static_cast<double>(T) * t_past + 0.5 * T * (T + 1.0);
      *fl = 4.0 * B * h * pairs * dh;
      *by = static_cast<double>(B) * h * (2.0 * T * dh * 2 + 2.0 * t_len * dh * 2);
      return launch_attention_tc(c->env, static_cast<const bf16*>(q),
                                 reinterpret_cast<const bf16*>(kv.base), kv.s_batch, kv.s_kv,
                                 kv.s_head, B, h, T, t_past, attn, s, true);
    });
  } else {
    st = c->run(kKindSimtFp32, s, [&](double*, double*) {
      return launch_attention_fp32(static_cast<const float*>(q),
                                   reinterpret_cast<const float*>(kv.base), kv.s_batch, kv.s_kv,
                                   kv.s_head, B, h, T, t_past, dh, static_cast<float*>(attn), s);
    });
  }
  if (st) return st;

  // c_proj + bias + residual: x' = x + a (fp32)
  EpiParams e2{};
  e2.bias = p->proj_b;
  e2.ldo = d;
  float* xprime = x_is_stream ? static_cast<float*>(out) : resid;
  e2.resid = x_in;
  e2.out = xprime;
  st = c->run(bf ? kKindGemmProj : kKindSimtFp32, s, [&](double* fl, double* by) {
    if (bf) {
      const int kind = x_is_stream ? kEpiResidF32 : kEpiResidBf16In;
      return gemm16(c, kind, attn, w.proj_w, M, d, d, e2, false, s, fl, by, w_early);
    }
    return launch_gemm_fp32(c->env, kEpiResidF32, static_cast<const float*>(attn),
                            static_cast<const float*>(p->proj_w), M, d, d, e2, dh, s);
  });
  if (st) return st;

  // LN2
  st = c->run(kKindLayerNorm, s, [&](double* fl, double* by) {
    *fl = 0;
    *by = static_cast<double>(M) * d * (4 + (bf ? 2 : 4));
    return launch_layer_norm(hp.dtype, xprime, GPT2_FP32, p->ln2_g, p->ln2_b, M, d, ln, s, bf,
                             nullptr, c->env.err);
  });
  if (st) return st;

  // c_fc + bias + GELU
  EpiParams e3{};
  e3.bias = p->fc_b;
  e3.out = fc;
  e3.ldo = 4 * d;
  st = c->run(bf ? kKindGemmFc : kKindSimtFp32, s, [&](double* fl, double* by) {
    if (bf)
      return gemm16(c, kEpiGelu, ln, w.fc_w, M, 4 * d, d, e3, true, s, fl, by, w_early);
    return launch_gemm_fp32(c->env, kEpiGelu, static_cast<const float*>(ln),
                            static_cast<const float*>(p->fc_w), M, 4 * d, d, e3, dh, s);
  });
  if (st) return st;

  // mlp c_proj + bias + residual: out = x' + m
  EpiParams e4{};
  e4.bias = p->mlp_proj_b;
  e4.resid = xprime;
  e4.out = out;
  e4.ldo = d;
  st = c->run(bf ? kKindGemmMlpProj : kKindSimtFp32, s, [&](double* fl, double* by) {
    if (bf) {
      const int kind = x_is_stream ? kEpiResidF32 : kEpiResidBf16Out;
      return gemm16(c, kind, fc, w.mlp_proj_w, M, d, 4 * d, e4, false, s, fl, by, w_early);
    }
    return launch_gemm_fp32(c->env, kEpiResidF32, static_cast<const float*>(fc),
                            static_cast<const float*>(p->mlp_proj_w), M, d, 4 * d, e4, dh, s);
  });
  return st;
}

int check_ctx_shapes(const gpt2_ctx* c, int B, int T) {
  if (B <= 0 || T <= 0) return GPT2_ERR_INVALID_ARG;
  if (B > c->max_B || static_cast<long long>(B) * T > static_cast<long long>(c->max_B) * c->max_T)
    return GPT2_ERR_WORKSPACE;
  return GPT2_OK;
}

int check_mode_shape(const gpt2_hparams& hp) {
  if (hp.n_embd <= 0 || hp.n_head <= 0 || hp.n_ctx <= 0 || hp.n_layer <= 0 || hp.n_vocab <= 0)
    return GPT2_ERR_INVALID_ARG;
  if (hp.dtype != GPT2_BF16 && hp.dtype != GPT2_FP32) return GPT2_ERR_INVALID_ARG;
  if (hp.n_embd % hp.n_head != 0) return GPT2_ERR_UNSUPPORTED;
  const int dh = hp.n_embd / hp.n_head;
  if (hp.dtype == GPT2_BF16 && dh != 64) return GPT2_ERR_UNSUPPORTED;
  if (hp.dtype == GPT2_FP32 && dh > 256) return GPT2_ERR_UNSUPPORTED;
  return GPT2_OK;
}

std::mutex g_smem_attr_mutex;
struct SmemAttr {
  int device;
  const void* fn;
  int bytes;
};
std::vector<SmemAttr> g_smem_attrs;

std::once_flag g_encode_once;
EncodeTiledFn g_encode = nullptr;

EncodeTiledFn get_encode() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  });
  return g_encode;
}

}  // namespace

namespace gpt2 {

namespace {
thread_local bool t_plain_next = false;
}  // namespace

void request_plain_launch() { t_plain_next = true; }

bool take_pdl_permission() {
  const bool plain = t_plain_next;
  t_plain_next = false;
  return !plain;
}

bool ensure_smem_limit(const void* fn, int bytes) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  std::lock_guard<std::mutex> lock(g_smem_attr_mutex);
  for (const SmemAttr& a : g_smem_attrs)
    if (a.device == dev && a.fn == fn && a.bytes >= bytes) return true;
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess)
    return false;
  for (SmemAttr& a : g_smem_attrs)
    if (a.device == dev && a.fn == fn) {
      a.bytes = bytes;
      return true;
    }
  g_smem_attrs.push_back(SmemAttr{dev, fn, bytes});
  return true;
}

namespace {
// One thread waits on an mbarrier nothing completes, with the kernels' bounded
// wait and a short limit: the wait runs out and raises the timeout bit.
__global__ void wait_timeout_kernel(unsigned* err, unsigned long long limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait_bounded(&bar, 0, nullptr, err, limit_ns);
}
}  // namespace
}  // namespace gpt2

extern "C" {

const char* gpt2_status_string(int status) {
  switch (status) {
    case GPT2_OK: return "ok";
    case GPT2_ERR_INVALID_ARG: return "invalid argument";
    case GPT2_ERR_UNSUPPORTED: return "unsupported shape for this mode";
    case GPT2_ERR_CTX_OVERFLOW: return "positions beyond n_ctx or cache capacity";
    case GPT2_ERR_ALIGNMENT: return "device pointer not 16-byte aligned";
    case GPT2_ERR_CUDA: return "CUDA runtime error";
    case GPT2_ERR_DEVICE_TIMEOUT: return "a kernel wait timed out";
    case GPT2_ERR_WORKSPACE: return "workspace too small for the request";
    case GPT2_ERR_NO_DEVICE: return "no sm_100-family GPU is current";
    case GPT2_ERR_RANGE:
      return "a value outside the fp16 operand range (|v| > 65504) or not finite";
    default: return "unknown status";
  }
}

int gpt2_workspace_bytes(const gpt2_hparams* hp, int max_B, int max_T, size_t* bytes) {
  if (!hp || !bytes || max_B <= 0 || max_T <= 0) return GPT2_ERR_INVALID_ARG;
  const int st = check_mode_shape(*hp);
  if (st) return st;
  *bytes = plan_workspace(*hp, max_B, max_T).total;
  return GPT2_OK;
}

int gpt2_ctx_create(const gpt2_hparams* hp, int max_B, int max_T, void* workspace,
                    size_t workspace_bytes, gpt2_ctx** out) {
  if (!hp || !out || !workspace || max_B <= 0 || max_T <= 0) return GPT2_ERR_INVALID_ARG;
  *out = nullptr;
  int st = check_mode_shape(*hp);
  if (st) return st;
  if (reinterpret_cast<uintptr_t>(workspace) & 255) return GPT2_ERR_ALIGNMENT;
  const WsPlan plan = plan_workspace(*hp, max_B, max_T);
  if (workspace_bytes < plan.total) return GPT2_ERR_WORKSPACE;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return GPT2_ERR_NO_DEVICE;
  int major = 0, sms = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return GPT2_ERR_NO_DEVICE;
  if (major != 10) return GPT2_ERR_NO_DEVICE;
  EncodeTiledFn enc = get_encode();
  if (!enc) return GPT2_ERR_CUDA;
  gpt2_ctx* c = new (std::nothrow) gpt2_ctx();
  if (!c) return GPT2_ERR_INVALID_ARG;
  c->hp = *hp;
  c->max_B = max_B;
  c->max_T = max_T;
  c->device = dev;
  c->ws = static_cast<uint8_t*>(workspace);
  c->ws_bytes = workspace_bytes;
  c->plan = plan;
  c->env.num_sms = sms;
  c->env.err = c->at<unsigned>(plan.err);
  c->env.encode = enc;
  c->env.wait_ns = kWaitLimitNs;
  c->prof = false;
  c->extra_kernels = 0;
  c->cache_weights = false;
  c->conv_src.assign(static_cast<size_t>(hp->n_layer) * 4 + 1, nullptr);
  for (int k = 0; k < kKindCount; ++k) {
    c->launches[k] = 0;
    c->total_ms[k] = c->flops[k] = c->bytes[k] = 0.0;
  }
  if (cudaMemset(c->env.err, 0, sizeof(unsigned)) != cudaSuccess) {
    delete c;
    return GPT2_ERR_CUDA;
  }
  *out = c;
  return GPT2_OK;
}

void gpt2_ctx_destroy(gpt2_ctx* c) {
  if (!c) return;
  for (auto& r : c->recs) {
    cudaEventDestroy(r.start);
    cudaEventDestroy(r.stop);
  }
  for (auto e : c->free_events) cudaEventDestroy(e);
  delete c;
}

int gpt2_selftest_wait_timeout(gpt2_ctx* c, int limit_us, void* stream) {
  if (!c || limit_us < 1 || limit_us > 1000000) return GPT2_ERR_INVALID_ARG;
  gpt2::wait_timeout_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
      c->env.err, static_cast<unsigned long long>(limit_us) * 1000ull);
  return cudaGetLastError() == cudaSuccess ? GPT2_OK : GPT2_ERR_CUDA;
}

int gpt2_ctx_set_wait_limit(gpt2_ctx* c, long long limit_ns) {
  if (!c) return GPT2_ERR_INVALID_ARG;
  c->env.wait_ns = limit_ns > 0 ? static_cast<unsigned long long>(limit_ns) : kWaitLimitNs;
  return GPT2_OK;
}

int gpt2_sync_status(gpt2_ctx* c, void* stream) {
  if (!c) return GPT2_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return GPT2_ERR_CUDA;
  if (cudaGetLastError() != cudaSuccess) return GPT2_ERR_CUDA;
  unsigned word = 0;
  if (cudaMemcpy(&word, c->env.err, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess)
    return GPT2_ERR_CUDA;
  if (word != 0 && cudaMemset(c->env.err, 0, sizeof(unsigned)) != cudaSuccess) return GPT2_ERR_CUDA;
  if (word & kErrTimeout) return GPT2_ERR_DEVICE_TIMEOUT;
  if (word & kErrBadToken) return GPT2_ERR_INVALID_ARG;
  if (word & kErrRange) return GPT2_ERR_RANGE;
  return GPT2_OK;
}

int gpt2_block_forward(gpt2_ctx* c, const void* x, const gpt2_block_params* params, int B, int T,
                       int d, int n_head, const gpt2_kv* past, gpt2_kv* present, void* out,
                       void* stream) {
  if (!c || !x || !out) return GPT2_ERR_INVALID_ARG;
  if (d != c->hp.n_embd || n_head != c->hp.n_head) return GPT2_ERR_INVALID_ARG;
  int st = check_ctx_shapes(c, B, T);
  if (st) return st;
  if ((st = validate_block_params(params))) return st;
  if ((st = validate_kv(past, false)) || (st = validate_kv(present, true))) return st;
  if (!aligned16(x) || !aligned16(out)) return GPT2_ERR_ALIGNMENT;
  const int t_past = past ? past->T_len : 0;
  if (t_past + T > c->hp.n_ctx) return GPT2_ERR_CTX_OVERFLOW;
  if (present && t_past + T > present->T_cap) return GPT2_ERR_CTX_OVERFLOW;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int h = n_head, dh = d / h;
  const size_t es = c->hp.dtype == GPT2_BF16 ? 2 : 4;
  // Cached fp16 weights are read before waits on the previous kernel: the
  // call's first launch waits for all earlier work (request_plain_launch).
  if (c->hp.dtype == GPT2_BF16 && c->cache_weights) request_plain_launch();

  KvView dst;
  if (present) {
    dst = layer_view(present->data, present->T_cap, 1, 0, h, dh, es);
    if (past && past->data != present->data) {
      const KvView src = layer_view(past->data, past->T_cap, 1, 0, h, dh, es);
      if ((st = copy_positions(dst, src, B, h, t_past, dh, es, s))) return st;
    }
  } else {
    dst = layer_view(c->ws + c->plan.kv, c->hp.n_ctx, 1, 0, h, dh, es);
    if (past) {
      const KvView src = layer_view(past->data, past->T_cap, 1, 0, h, dh, es);
      if ((st = copy_positions(dst, src, B, h, t_past, dh, es, s))) return st;
    }
  }
  st = block_sequence(c, params, 0, B, T, x, false, out, dst, t_past, s);
  if (st) return st;
  if (present) present->T_len = t_past + T;
  return GPT2_OK;
}

int gpt2_block_forward_postnorm(gpt2_ctx* c, const void* x, const gpt2_block_params* p, int B,
                                int T, int d, int n_head, void* out, void* stream) {
  if (!c || !x || !out) return GPT2_ERR_INVALID_ARG;
  if (d != c->hp.n_embd || n_head != c->hp.n_head) return GPT2_ERR_INVALID_ARG;
  int st = check_ctx_shapes(c, B, T);
  if (st) return st;
  if ((st = validate_block_params(p))) return st;
  if (!aligned16(x) || !aligned16(out)) return GPT2_ERR_ALIGNMENT;
  if (T > c->hp.n_ctx) return GPT2_ERR_CTX_OVERFLOW;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const gpt2_hparams& hp = c->hp;
  const int h = n_head, dh = d / h, M = B * T;
  const bool bf = hp.dtype == GPT2_BF16;
  const size_t es = bf ? 2 : 4;
  const KvView kv = layer_view(c->ws + c->plan.kv, hp.n_ctx, 1, 0, h, dh, es);
  void* x1 = c->ws + c->plan.ln;      // LN1 output: the normalised stream
  void* q = c->ws + c->plan.q;
  void* attn = c->ws + c->plan.attn;
  float* pre = c->at<float>(c->plan.resid);  // x + a, then x1 + m (fp32)
  void* fc = c->ws + c->plan.fc;

  // c_attn on x itself -> Q and the block's K/V
  EpiParams e{};
  e.bias = p->attn_b;
  e.q = q;
  e.kv.base = kv.base;
  e.kv.s_batch = kv.s_batch;
  e.kv.s_kv = kv.s_kv;
  e.kv.s_head = kv.s_head;
  e.kv.t_past = 0;
  e.T = T;
  e.d = d;
  e.ldo = 3 * d;
  st = c->run(bf ? kKindGemmQkv : kKindSimtFp32, s, [&](double* fl, double* by) {
    if (bf)
      return launch_gemm_tc(c->env, kEpiQkv, x, p->attn_w, M, 3 * d, d, e, s, fl, by, false, false);
    return launch_gemm_fp32(c->env, kEpiQkv, static_cast<const float*>(x),
                            static_cast<const float*>(p->attn_w), M, 3 * d, d, e, dh, s);
  });
  if (st) return st;
  st = c->run(bf ? kKindAttention : kKindSimtFp32, s, [&](double* fl, double* by) {
    *fl = 4.0 * B * h * (0.5 * T * (T + 1.0)) * dh;
    *by = static_cast<double>(B) * h * (2.0 * T * dh * 2 + 2.0 * T * dh * 2);
    if (bf)
      return launch_attention_tc(c->env, static_cast<const bf16*>(q),
                                 reinterpret_cast<const bf16*>(kv.base), kv.s_batch, kv.s_kv,
                                 kv.s_head, B, h, T, 0, attn, s, false);
    return launch_attention_fp32(static_cast<const float*>(q),
                                 reinterpret_cast<const float*>(kv.base), kv.s_batch, kv.s_kv,
                                 kv.s_head, B, h, T, 0, dh, static_cast<float*>(attn), s);
  });
  if (st) return st;
  // pre = x + c_proj(attn) + b (fp32)
  EpiParams e2{};
  e2.bias = p->proj_b;
  e2.ldo = d;
  e2.resid = x;
  e2.out = pre;
  st = c->run(bf ? kKindGemmProj : kKindSimtFp32, s, [&](double* fl, double* by) {
    if (bf)
      return launch_gemm_tc(c->env, kEpiResidBf16In, attn, p->proj_w, M, d, d, e2, s, fl, by,
                            false, false);
    return launch_gemm_fp32(c->env, kEpiResidF32, static_cast<const float*>(attn),
                            static_cast<const float*>(p->proj_w), M, d, d, e2, dh, s);
  });
  if (st) return st;
  // x1 = LN1(pre)
  st = c->run(kKindLayerNorm, s, [&](double* fl, double* by) {
    *fl = 0;
    *by = static_cast<double>(M) * d * (4 + es);
    return launch_layer_norm(hp.dtype, pre, GPT2_FP32, p->ln1_g, p->ln1_b, M, d, x1, s, false);
  });
  if (st) return st;
  // fc = GELU(c_fc(x1))
  EpiParams e3{};
  e3.bias = p->fc_b;
  e3.out = fc;
  e3.ldo = 4 * d;
  st = c->run(bf ? kKindGemmFc : kKindSimtFp32, s, [&](double* fl, double* by) {
    if (bf)
      return launch_gemm_tc(c->env, kEpiGelu, x1, p->fc_w, M, 4 * d, d, e3, s, fl, by, false,
                            false);
    return launch_gemm_fp32(c->env, kEpiGelu, static_cast<const float*>(x1),
                            static_cast<const float*>(p->fc_w), M, 4 * d, d, e3, dh, s);
  });
  if (st) return st;
  // pre = x1 + mlp_proj(fc) + b (fp32)
  EpiParams e4{};
  e4.bias = p->mlp_proj_b;
  e4.ldo = d;
  e4.resid = x1;
  e4.out = pre;
  st = c->run(bf ? kKindGemmMlpProj : kKindSimtFp32, s, [&](double* fl, double* by) {
    if (bf)
      return launch_gemm_tc(c->env, kEpiResidBf16In, fc, p->mlp_proj_w, M, d, 4 * d, e4, s, fl,
                            by, false, false);
    return launch_gemm_fp32(c->env, kEpiResidF32, static_cast<const float*>(fc),
                            static_cast<const float*>(p->mlp_proj_w), M, d, 4 * d, e4, dh, s);
  });
  if (st) return st;
  // out = LN2(pre)
  return c->run(kKindLayerNorm, s, [&](double* fl, double* by) {
    *fl = 0;
    *by = static_cast<double>(M) * d * (4 + es);
    return launch_layer_norm(hp.dtype, pre, GPT2_FP32, p->ln2_g, p->ln2_b, M, d, out, s, false);
  });
}

namespace {

// Everything of the full forward before the head: validation, the embedding,
// the L blocks and LN_f into the workspace's `ln` rows (fp16 in bf16 mode);
// *wte16 receives the tied embedding's fp16 copy (bf16 mode).  *t_past_out is
// the position of the first new token.
int forward_trunk(gpt2_ctx* c, const int32_t* ids, int B, int T, const gpt2_params* params, int L,
                  const gpt2_kv* past, gpt2_kv* present, cudaStream_t s, const __half** wte16,
                  int* t_past_out) {
  if (!c || !ids || !params || !params->blocks) return GPT2_ERR_INVALID_ARG;
  if (L != c->hp.n_layer) return GPT2_ERR_INVALID_ARG;
  int st = check_ctx_shapes(c, B, T);
  if (st) return st;
  const void* mp[4] = {params->wte, params->wpe, params->lnf_g, params->lnf_b};
  for (const void* p : mp) {
    if (!p) return GPT2_ERR_INVALID_ARG;
    if (!aligned16(p)) return GPT2_ERR_ALIGNMENT;
  }
  for (int l = 0; l < L; ++l)
    if ((st = validate_block_params(&params->blocks[l]))) return st;
  if ((st = validate_kv(past, false)) || (st = validate_kv(present, true))) return st;
  if (!aligned16(ids)) return GPT2_ERR_ALIGNMENT;
  const int t_past = past ? past->T_len : 0;
  if (t_past + T > c->hp.n_ctx) return GPT2_ERR_CTX_OVERFLOW;
  if (present && t_past + T > present->T_cap) return GPT2_ERR_CTX_OVERFLOW;
  *t_past_out = t_past;

  const gpt2_hparams& hp = c->hp;
  const int d = hp.n_embd, h = hp.n_head, dh = d / h, V = hp.n_vocab;
  const int M = B * T;
  const bool bf = hp.dtype == GPT2_BF16;
  const size_t es = bf ? 2 : 4;
  float* H = c->at<float>(c->plan.resid);

  // Cached fp16 weights are read before waits on the previous kernel: the
  // call's first launch waits for all earlier work (request_plain_launch).
  if (bf && c->cache_weights) request_plain_launch();
  st = c->run(kKindEmbed, s, [&](double* fl, double* by) {
    *fl = 0;
    *by = static_cast<double>(M) * d * (2.0 * es + 4.0) + 4.0 * M;
    return launch_embed(hp.dtype, ids, params->wte, params->wpe, B, T, t_past, d, V, H,
                        c->env.err, s);
  });
  if (st) return st;

  for (int l = 0; l < L; ++l) {
    KvView dst;
    if (present) {
      dst = layer_view(present->data, present->T_cap, L, l, h, dh, es);
      if (past && past->data != present->data) {
        const KvView src = layer_view(past->data, past->T_cap, L, l, h, dh, es);
        if ((st = copy_positions(dst, src, B, h, t_past, dh, es, s))) return st;
      }
    } else {
      dst = layer_view(c->ws + c->plan.kv, hp.n_ctx, 1, 0, h, dh, es);
      if (past) {
        const KvView src = layer_view(past->data, past->T_cap, L, l, h, dh, es);
        if ((st = copy_positions(dst, src, B, h, t_past, dh, es, s))) return st;
      }
    }
    st = block_sequence(c, &params->blocks[l], l, B, T, H, true, H, dst, t_past, s);
    if (st) return st;
  }

  // LN_f, with the tied embedding's fp16 conversion in the same launch
  *wte16 = nullptr;
  ConvSegs conv{};
  if (bf) wte_conversion(c, params->wte, wte16, &conv);
  void* ln = c->ws + c->plan.ln;
  return c->run(kKindLayerNorm, s, [&](double* fl, double* by) {
    *fl = 0;
    *by = static_cast<double>(M) * d * (4 + es) + conversion_bytes(conv);
    return launch_layer_norm(hp.dtype, H, GPT2_FP32, params->lnf_g, params->lnf_b, M, d, ln, s,
                             bf, conv.count ? &conv : nullptr, c->env.err);
  });
}

}  // namespace

int gpt2_forward(gpt2_ctx* c, const int32_t* ids, int B, int T, const gpt2_params* params, int L,
                 const gpt2_kv* past, gpt2_kv* present, float* logits, void* stream) {
  if (!c || !logits) return GPT2_ERR_INVALID_ARG;
  if (!aligned16(logits)) return GPT2_ERR_ALIGNMENT;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const __half* wte16 = nullptr;
  int t_past = 0;
  int st = forward_trunk(c, ids, B, T, params, L, past, present, s, &wte16, &t_past);
  if (st) return st;
  const gpt2_hparams& hp = c->hp;
  const int d = hp.n_embd, dh = d / hp.n_head, V = hp.n_vocab, M = B * T;
  const bool bf = hp.dtype == GPT2_BF16;
  void* ln = c->ws + c->plan.ln;
  EpiParams e{};
  e.out = logits;
  e.ldo = V;
  st = c->run(bf ? kKindGemmLogits : kKindSimtFp32, s, [&](double* fl, double* by) {
    if (bf)
      return gemm16(c, kEpiLogits, ln, wte16, M, V, d, e, false, s, fl, by);
    return launch_gemm_fp32(c->env, kEpiLogits, static_cast<const float*>(ln),
                            static_cast<const float*>(params->wte), M, V, d, e, dh, s);
  });
  if (st) return st;
  if (present) present->T_len = t_past + T;
  return GPT2_OK;
}

int gpt2_forward_loss(gpt2_ctx* c, const int32_t* ids, const int32_t* targets, int B, int T,
                      const gpt2_params* params, int L, const gpt2_kv* past, gpt2_kv* present,
                      float* loss, int32_t* next_ids, void* stream) {
  if (!c || (!loss && !next_ids)) return GPT2_ERR_INVALID_ARG;
  if (loss && !targets) return GPT2_ERR_INVALID_ARG;
  if (c->hp.dtype != GPT2_BF16) return GPT2_ERR_UNSUPPORTED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const __half* wte16 = nullptr;
  int t_past = 0;
  int st = forward_trunk(c, ids, B, T, params, L, past, present, s, &wte16, &t_past);
  if (st) return st;
  const gpt2_hparams& hp = c->hp;
  const int d = hp.n_embd, V = hp.n_vocab, M = B * T;
  const int nvb = loss_vblocks(hp);
  float* tl = c->at<float>(c->plan.hloss);
  float* pm = tl + M;
  float* ps = pm + static_cast<size_t>(nvb) * M;
  int32_t* pi = reinterpret_cast<int32_t*>(ps + static_cast<size_t>(nvb) * M);
  EpiParams e{};
  e.tgt = loss ? targets : nullptr;
  e.tgt_logit = tl;
  e.part_m = pm;
  e.part_s = ps;
  e.part_i = pi;
  st = c->run(kKindGemmLogits, s, [&](double* fl, double* by) {
    return launch_gemm_tc(c->env, kEpiHeadLoss, c->ws + c->plan.ln, wte16, M, V, d, e, s, fl,
                          by, true, false);
  });
  if (st) return st;
  st = c->run(kKindLossCombine, s, [&](double* fl, double* by) {
    *fl = 0;
    *by = 12.0 * nvb * M + 12.0 * M;
    return launch_head_loss_combine(pm, ps, pi, nvb, M, V, loss ? targets : nullptr, tl, loss,
                                    next_ids, c->env.err, s);
  });
  if (st) return st;
  if (present) present->T_len = t_past + T;
  return GPT2_OK;
}

int gpt2_forward_topk(gpt2_ctx* c, const int32_t* ids, int B, int T, const gpt2_params* params,
                      int L, const gpt2_kv* past, gpt2_kv* present, int k, float* top_logits,
                      int32_t* top_ids, float* lse, void* stream) {
  if (!c || !top_logits || !top_ids) return GPT2_ERR_INVALID_ARG;
  if (k < 1 || k > kTopKMax || k > c->hp.n_vocab) return GPT2_ERR_INVALID_ARG;
  if (c->hp.dtype != GPT2_BF16) return GPT2_ERR_UNSUPPORTED;
  if (!aligned16(top_logits) || !aligned16(top_ids) || (lse && !aligned16(lse)))
    return GPT2_ERR_ALIGNMENT;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const __half* wte16 = nullptr;
  int t_past = 0;
  int st = forward_trunk(c, ids, B, T, params, L, past, present, s, &wte16, &t_past);
  if (st) return st;
  const gpt2_hparams& hp = c->hp;
  const int d = hp.n_embd, V = hp.n_vocab, M = B * T;
  const int nvb = loss_vblocks(hp);
  float* pm = c->at<float>(c->plan.hloss) + M;
  float* ps = pm + static_cast<size_t>(nvb) * M;
  float* tv = c->at<float>(c->plan.htopk);
  int32_t* ti = reinterpret_cast<int32_t*>(tv + static_cast<size_t>(nvb) * kTopKMax * M);
  EpiParams e{};
  e.part_m = pm;
  e.part_s = ps;
  e.topk_v = tv;
  e.topk_i = ti;
  e.topk_k = k;
  st = c->run(kKindGemmLogits, s, [&](double* fl, double* by) {
    return launch_gemm_tc(c->env, kEpiHeadTopK, c->ws + c->plan.ln, wte16, M, V, d, e, s, fl,
                          by, true, false);
  });
  if (st) return st;
  st = c->run(kKindLossCombine, s, [&](double* fl, double* by) {
    *fl = 0;
    *by = static_cast<double>(nvb) * M * (8.0 + 8.0 * k) + 8.0 * M * k + 4.0 * M;
    return launch_head_topk_combine(pm, ps, tv, ti, nvb, M, k, top_logits, top_ids, lse, s);
  });
  if (st) return st;
  if (present) present->T_len = t_past + T;
  return GPT2_OK;
}

int gpt2_generate_greedy(gpt2_ctx* c, const int32_t* ids, int B, int T_prompt,
                         const gpt2_params* params, int L, gpt2_kv* cache, int n_new, float* logits,
                         int32_t* out_ids, void* stream) {
  if (!c || !ids || !params || !cache || !logits || !out_ids || n_new <= 0)
    return GPT2_ERR_INVALID_ARG;
  if (T_prompt <= 0) return GPT2_ERR_INVALID_ARG;
  if (!aligned16(out_ids)) return GPT2_ERR_ALIGNMENT;
  const int t0 = cache->T_len;
  // The last generated token is not run through the model.
  const long long t_end = static_cast<long long>(t0) + T_prompt + n_new - 1;
  if (t_end > c->hp.n_ctx || t_end > cache->T_cap) return GPT2_ERR_CTX_OVERFLOW;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int V = c->hp.n_vocab;
  int32_t* next = c->at<int32_t>(c->plan.ids);
  // The prompt (after any cached prefix), then the argmax of its last position.
  int st = gpt2_forward(c, ids, B, T_prompt, params, L, t0 > 0 ? cache : nullptr, cache, logits,
                        stream);
  if (st) return st;
  for (int i = 0; i < n_new; ++i) {
    const int T = i == 0 ? T_prompt : 1;
    st = c->run(kKindArgmax, s, [&](double* fl, double* by) {
      *fl = 0;
      *by = 4.0 * B * V;
      return launch_argmax_rows(logits + static_cast<size_t>(T - 1) * V, B, V,
                                static_cast<long long>(T) * V, out_ids + i, n_new, next, s);
    });
    if (st) return st;
    if (i + 1 < n_new &&
        (st = gpt2_forward(c, next, B, 1, params, L, cache, cache, logits, stream)))
      return st;
  }
  return GPT2_OK;
}

int gpt2_layer_norm(int mode, const void* x, int x_dtype, const void* g, const void* b, int rows,
                    int d, void* y, void* stream) {
  if (!x || !g || !b || !y) return GPT2_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(g) || !aligned16(b) || !aligned16(y)) return GPT2_ERR_ALIGNMENT;
  return launch_layer_norm(mode, x, x_dtype, g, b, rows, d, y, static_cast<cudaStream_t>(stream));
}

int gpt2_linear(gpt2_ctx* c, int epilogue, const void* A, const void* W, const void* bias,
                const float* resid, void* out, int M, int N, int K, void* stream) {
  if (!c || !A || !W || !out || M <= 0 || N <= 0 || K <= 0) return GPT2_ERR_INVALID_ARG;
  if (!aligned16(A) || !aligned16(W) || !aligned16(out)) return GPT2_ERR_ALIGNMENT;
  int kind;
  switch (epilogue) {
    case GPT2_EPI_BIAS: kind = kEpiBias; break;
    case GPT2_EPI_BIAS_GELU: kind = kEpiGelu; break;
    case GPT2_EPI_BIAS_RESID: kind = kEpiResidF32; break;
    case GPT2_EPI_LOGITS: kind = kEpiLogits; break;
    default: return GPT2_ERR_INVALID_ARG;
  }
  if (kind != kEpiLogits && !bias) return GPT2_ERR_INVALID_ARG;
  if (kind == kEpiResidF32 && !resid) return GPT2_ERR_INVALID_ARG;
  if ((bias && !aligned16(bias)) || (resid && !aligned16(resid))) return GPT2_ERR_ALIGNMENT;
  EpiParams e{};
  e.bias = bias;
  e.resid = resid;
  e.out = out;
  e.ldo = N;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const bool bf = c->hp.dtype == GPT2_BF16;
  return c->run(bf ? kKindGemmOther : kKindSimtFp32, s, [&](double* fl, double* by) {
    if (bf)
      return launch_gemm_tc(c->env, kind, A, W, M, N, K, e, s, fl, by, false, false);
    return launch_gemm_fp32(c->env, kind, static_cast<const float*>(A),
                            static_cast<const float*>(W), M, N, K, e, 1, s);
  });
}

int gpt2_attention(gpt2_ctx* c, const void* q, const void* kv, int B, int n_head, int T,
                   int T_past, int T_cap, int d_h, void* out, void* stream) {
  if (!c || !q || !kv || !out) return GPT2_ERR_INVALID_ARG;
  if (B <= 0 || n_head <= 0 || T <= 0 || T_past < 0 || d_h <= 0) return GPT2_ERR_INVALID_ARG;
  if (T_past + T > T_cap) return GPT2_ERR_CTX_OVERFLOW;
  if (!aligned16(q) || !aligned16(kv) || !aligned16(out)) return GPT2_ERR_ALIGNMENT;
  const bool bf = c->hp.dtype == GPT2_BF16;
  if (bf && d_h != 64) return GPT2_ERR_UNSUPPORTED;
  if (B > c->max_B || n_head > c->hp.n_head) return GPT2_ERR_WORKSPACE;
  const size_t es = bf ? 2 : 4;
  const KvView v = layer_view(const_cast<void*>(kv), T_cap, 1, 0, n_head, d_h, es);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int t_len = T_past + T;
  if (bf && T == 1 && T_past > 0) {
    const int splits = decode_splits(B, n_head, t_len, c->env.num_sms);
    int nl = 0;
    return c->run(kKindDecodeAttention, s, [&](double*, double*) {
      const int r = launch_decode_attention_bf16(
          static_cast<const bf16*>(q), reinterpret_cast<const bf16*>(v.base), v.s_batch, v.s_kv,
          v.s_head, B, n_head, t_len, out, c->at<float>(c->plan.partials), splits, s, &nl, false,
          c->env.err, c->env.wait_ns);
      c->extra_kernels = nl - 1;
      return r;
    });
  }
  if (bf)
    return c->run(kKindAttention, s, [&](double*, double*) {
      return launch_attention_tc(c->env, static_cast<const bf16*>(q),
                                 reinterpret_cast<const bf16*>(v.base), v.s_batch, v.s_kv,
                                 v.s_head, B, n_head, T, T_past, out, s, false);
    });
  return c->run(kKindSimtFp32, s, [&](double*, double*) {
    return launch_attention_fp32(static_cast<const float*>(q),
                                 reinterpret_cast<const float*>(v.base), v.s_batch, v.s_kv,
                                 v.s_head, B, n_head, T, T_past, d_h, static_cast<float*>(out), s);
  });
}

int gpt2_embed(gpt2_ctx* c, const int32_t* ids, const void* wte, const void* wpe, int B, int T,
               int T_past, float* H, void* stream) {
  if (!c || !ids || !wte || !wpe || !H || B <= 0 || T <= 0 || T_past < 0)
    return GPT2_ERR_INVALID_ARG;
  if (T_past + T > c->hp.n_ctx) return GPT2_ERR_CTX_OVERFLOW;
  if (!aligned16(ids) || !aligned16(wte) || !aligned16(wpe) || !aligned16(H))
    return GPT2_ERR_ALIGNMENT;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return c->run(kKindEmbed, s, [&](double*, double*) {
    return launch_embed(c->hp.dtype, ids, wte, wpe, B, T, T_past, c->hp.n_embd, c->hp.n_vocab, H,
                        c->env.err, s);
  });
}

int gpt2_ctx_cache_weights(gpt2_ctx* c, int enable) {
  if (!c) return GPT2_ERR_INVALID_ARG;
  c->cache_weights = enable != 0;
  std::fill(c->conv_src.begin(), c->conv_src.end(), nullptr);
  return GPT2_OK;
}

int gpt2_profile_enable(gpt2_ctx* c, int enable) {
  if (!c) return GPT2_ERR_INVALID_ARG;
  c->prof = enable != 0;
  return GPT2_OK;
}

int gpt2_profile_kinds(void) { return kKindCount; }

int gpt2_profile_read(gpt2_ctx* c, int kind, const char** name, long long* launches,
                      double* total_ms, double* flops, double* bytes) {
  if (!c || kind < 0 || kind >= kKindCount) return GPT2_ERR_INVALID_ARG;
  for (auto& r : c->recs) {
    if (cudaEventSynchronize(r.stop) != cudaSuccess) return GPT2_ERR_CUDA;
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, r.start, r.stop) != cudaSuccess) return GPT2_ERR_CUDA;
    c->launches[r.kind] += r.kernels;
    c->total_ms[r.kind] += ms;
    c->flops[r.kind] += r.flops;
    c->bytes[r.kind] += r.bytes;
    c->free_events.push_back(r.start);
    c->free_events.push_back(r.stop);
  }
  c->recs.clear();
  if (name) *name = kKindNames[kind];
  if (launches) *launches = c->launches[kind];
  if (total_ms) *total_ms = c->total_ms[kind];
  if (flops) *flops = c->flops[kind];
  if (bytes) *bytes = c->bytes[kind];
  return GPT2_OK;
}

int gpt2_profile_reset(gpt2_ctx* c) {
  if (!c) return GPT2_ERR_INVALID_ARG;
  for (auto& r : c->recs) {
    cudaEventSynchronize(r.stop);
    c->free_events.push_back(r.start);
    c->free_events.push_back(r.stop);
  }
  c->recs.clear();
  for (int k = 0; k < kKindCount; ++k) {
    c->launches[k] = 0;
    c->total_ms[k] = c->flops[k] = c->bytes[k] = 0.0;
  }
  return GPT2_OK;
}

}  // extern "C"

// noalloc.cu -- single-token decode attention that allocates nothing.
//
// Some callers cannot allocate device memory: a plugin that is handed only
// input/output pointers and a stream by its host application, a process whose
// device memory is already reserved in full by another allocator, or a
// latency-critical path that must not take cudaMalloc's implicit
// synchronisation.  This entry point serves them: the split-KV partial
// results live in a fixed array compiled into the library instead of a
// caller-provided workspace.
//
// The array is a file-scope __device__ variable: every GPU that loads the
// library holds it (1 MiB) until the process exits.  In host code its name is
// only a host-side stand-in, so its device address is looked up once per
// device, with that device current, by cudaGetSymbolAddress.
#include <atomic>
#include <mutex>

#include "device.cuh"
#include "internal.h"

namespace gpt2 {
namespace {

constexpr size_t kScratchBytes = 1u << 20;  // 1 MiB
constexpr size_t kScratchFloats = kScratchBytes / sizeof(float);
constexpr int kMaxDevices = 64;

static __device__ __align__(256) float g_decode_scratch[kScratchFloats];
// The entry point's device error word (a bounded wait that ran out), read and
// cleared by gpt2_attention_decode_noalloc_status.
static __device__ unsigned g_decode_err;

struct DeviceSetup {
  bool done = false;
  float* scratch = nullptr;
  unsigned* err = nullptr;
  int num_sms = 0;
};

// Limit of the kernel's bounded waits, for every device (0: the default 2 s).
std::atomic<unsigned long long> g_wait_ns{0};

std::mutex g_setup_mutex;
DeviceSetup g_setup[kMaxDevices];

// Looks up the scratch array's device address and the SM count for the
// current device, once.  Returns a gpt2_status.
int setup_current_device(DeviceSetup** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return GPT2_ERR_NO_DEVICE;
  if (dev < 0 || dev >= kMaxDevices) return GPT2_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  DeviceSetup& s = g_setup[dev];
  if (!s.done) {
    void* p = nullptr;
    void* e = nullptr;
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess ||
        cudaGetSymbolAddress(&e, g_decode_err) != cudaSuccess)
      return GPT2_ERR_CUDA;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return GPT2_ERR_CUDA;
    s.scratch = static_cast<float*>(p);
    s.err = static_cast<unsigned*>(e);
    s.num_sms = sms;
    s.done = true;
  }
  *out = &s;
  return GPT2_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

}  // namespace
}  // namespace gpt2

using namespace gpt2;

extern "C" int gpt2_attention_decode_noalloc(const void* q, const void* kv, int B, int n_head,
                                             int T_past, int T_cap, int d_h, int splits,
                                             void* out, void* stream) {
  if (!q || !kv || !out) return GPT2_ERR_INVALID_ARG;
  if (B <= 0 || n_head <= 0 || T_past <= 0 || splits < 0) return GPT2_ERR_INVALID_ARG;
  if (d_h != 64) return GPT2_ERR_UNSUPPORTED;
  if (T_past + 1 > T_cap) return GPT2_ERR_CTX_OVERFLOW;
  if (!aligned16(q) || !aligned16(kv) || !aligned16(out)) return GPT2_ERR_ALIGNMENT;
  // One CTA row per (sequence, head) pair: the grid's y extent.
  if (static_cast<long long>(B) * n_head > 65535) return GPT2_ERR_UNSUPPORTED;
  DeviceSetup* dev = nullptr;
  int st = setup_current_device(&dev);
  if (st) return st;
  const int t_len = T_past + 1;
  if (splits == 0) splits = decode_splits(B, n_head, t_len, dev->num_sms);
  if (splits > t_len || splits > 65535) return GPT2_ERR_INVALID_ARG;
  if (splits > 1 && decode_partials_floats(B, n_head, splits) > kScratchFloats)
    return GPT2_ERR_WORKSPACE;
  const long long s_head = static_cast<long long>(T_cap) * d_h;
  const long long s_kv = static_cast<long long>(n_head) * s_head;
  return launch_decode_attention_bf16(static_cast<const bf16*>(q), static_cast<const bf16*>(kv),
                                      2 * s_kv, s_kv, s_head, B, n_head, t_len,
                                      static_cast<bf16*>(out), dev->scratch, splits,
                                      static_cast<cudaStream_t>(stream), nullptr, false, dev->err,
                                      g_wait_ns.load());
}

extern "C" int gpt2_attention_decode_noalloc_status(void* stream) {
  DeviceSetup* dev = nullptr;
  const int st = setup_current_device(&dev);
  if (st) return st;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return GPT2_ERR_CUDA;
  unsigned word = 0;
  if (cudaMemcpy(&word, dev->err, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess)
    return GPT2_ERR_CUDA;
  if (word != 0 && cudaMemset(dev->err, 0, sizeof(unsigned)) != cudaSuccess) return GPT2_ERR_CUDA;
  return (word & kErrTimeout) ? GPT2_ERR_DEVICE_TIMEOUT : GPT2_OK;
}

extern "C" int gpt2_attention_decode_noalloc_set_wait_limit(long long limit_ns) {
  g_wait_ns.store(limit_ns > 0 ? static_cast<unsigned long long>(limit_ns) : 0ull);
  return GPT2_OK;
}

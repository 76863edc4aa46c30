// Window attention for callers that cannot allocate device memory.
//
// Some callers of this library cannot call cudaMalloc: code running while a CUDA graph is
// being captured (allocation would break the capture), allocator-less embedded runtimes,
// and host code that must not take the driver's allocation lock on a latency-critical
// path.  mono_attention_noalloc runs the same split-window attention kernel as a layer
// step, but its scratch (per-split partial results, the combine counters and a status
// word) lives in one fixed array compiled into this library instead of in a handle's
// arena.  The array costs MONO_NOALLOC_SCRATCH_BYTES of device memory on every GPU that
// loads the library, for as long as the process lives.
#include <algorithm>
#include <mutex>

#include "../../include/mono_layer.h"
#include "kernels.h"

using namespace mono;

namespace {

// [0, 256) status word; [256, kPartOff) combine counters; [kPartOff, end) split partials.
static __device__ __align__(256) unsigned char g_scratch[MONO_NOALLOC_SCRATCH_BYTES];

constexpr size_t kCounterOff = 256;
constexpr size_t kPartOff = 8192;
constexpr int kMaxDevices = 64;

std::mutex g_mu;
void* g_base[kMaxDevices] = {};
int g_sms[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up once per device.
int scratch_for_current_device(void** base, int* sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    (void)cudaGetLastError();
    return MONO_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) return MONO_ERR_UNSUPPORTED_DEVICE;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_base[dev]) {
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) {
      (void)cudaGetLastError();
      return MONO_ERR_CUDA;
    }
    if (prop.major != 10 || prop.minor != 3) return MONO_ERR_UNSUPPORTED_DEVICE;
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || !p) {
      (void)cudaGetLastError();
      return MONO_ERR_CUDA;
    }
    if (attention_prepare(64) != cudaSuccess || attention_prepare(128) != cudaSuccess) {
      (void)cudaGetLastError();
      return MONO_ERR_CUDA;
    }
    g_sms[dev] = prop.multiProcessorCount;
    g_base[dev] = p;
  }
  *base = g_base[dev];
  *sms = g_sms[dev];
  return MONO_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

}  // namespace

extern "C" int mono_attention_noalloc(const mono_layer_spec* s, const void* q, void* o,
                                      const int32_t* positions, const int32_t* row_req,
                                      const int32_t* block_table, int32_t max_blocks,
                                      int32_t n_req, int32_t rows, const uint8_t* kv_cache,
                                      int64_t kv_stride_block, int64_t kv_stride_tok,
                                      int64_t kv_num_blocks, void* stream) {
  if (!s || !q || !o || !positions || !row_req || !block_table || !kv_cache)
    return MONO_ERR_INVALID_ARG;
  if (rows < 1 || max_blocks < 1 || n_req < 1 || kv_num_blocks < 1) return MONO_ERR_INVALID_ARG;
  if (rows > 48) return MONO_ERR_TOO_MANY_ROWS;
  if (s->head_dim != 64 && s->head_dim != 128) return MONO_ERR_UNSUPPORTED_DIMS;
  if (s->kv_dim <= 0 || s->kv_dim % s->head_dim || s->kv_dim > 1024 || s->n_q_heads <= 0)
    return MONO_ERR_UNSUPPORTED_DIMS;
  const int G = s->kv_dim / s->head_dim;
  if (s->n_q_heads % G || s->n_q_heads / G > 16) return MONO_ERR_UNSUPPORTED_DIMS;
  if (s->window < 1 || s->window > 1024 || s->swa_width < 1 || s->swa_width > 1024 ||
      s->block_size < 1 || s->kv_record_bytes < s->kv_dim + 4)
    return MONO_ERR_UNSUPPORTED_DIMS;
  // q is read and o written in 16-byte vectors: a misaligned caller pointer is refused here
  // instead of faulting in the kernel
  if (!aligned16(q) || !aligned16(o) || !aligned16(kv_cache) || kv_stride_tok % 16 ||
      kv_stride_block % 16)
    return MONO_ERR_BAD_ALIGNMENT;
  if (kv_stride_tok < s->kv_record_bytes || kv_stride_block < (int64_t)s->block_size * kv_stride_tok)
    return MONO_ERR_BAD_KV_VIEW;

  void* base = nullptr;
  int sms = 0;
  int rc = scratch_for_current_device(&base, &sms);
  if (rc != MONO_OK) return rc;

  // Same split choice as a layer step (one split per 128 window keys); a problem whose
  // partials do not fit the scratch array is refused.
  const int width = std::max(s->causal ? s->window : s->swa_width, s->window);
  const int splits = (width + 127) / 128;
  auto part_bytes = [&](int S) {
    return (size_t)rows * s->n_q_heads * S * (s->head_dim + ATTN_PART_HEAD) * sizeof(float);
  };
  const size_t cap = MONO_NOALLOC_SCRATCH_BYTES - kPartOff;
  if (splits > 1 && part_bytes(splits) > cap) return MONO_ERR_TOO_MANY_ROWS;

  const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  // The array keeps the previous call's contents: the status word and the combine
  // counters must start at zero.
  cudaError_t e = cudaMemsetAsync(base, 0, kPartOff, st);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    return MONO_ERR_CUDA;
  }
  unsigned char* b = static_cast<unsigned char*>(base);
  AttnArgs a = {};
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.o = static_cast<__half*>(o);
  a.positions = positions;
  a.row_req = row_req;
  a.block_table = block_table;
  a.rows = rows;
  a.max_blocks = max_blocks;
  a.n_req = n_req;
  a.block_size = s->block_size;
  a.n_q = s->n_q_heads;
  a.kv_dim = s->kv_dim;
  a.window = s->window;
  a.swa_width = s->swa_width;
  a.causal = s->causal;
  a.cache = kv_cache;
  a.stride_block = kv_stride_block;
  a.stride_tok = kv_stride_tok;
  a.num_blocks = kv_num_blocks;
  a.splits = splits;
  a.part = reinterpret_cast<float*>(b + kPartOff);
  a.counters = reinterpret_cast<int*>(b + kCounterOff);
  a.status = reinterpret_cast<int*>(b);
  e = launch_attention(Launch{st, false}, a, s->head_dim, G);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    return MONO_ERR_CUDA;
  }
  return MONO_OK;
}

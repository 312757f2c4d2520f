// attn_decode_static: attn_decode with a library-owned, fixed-size scratch
// buffer instead of a caller-provided workspace.
//
// Some callers cannot allocate device memory for scratch: plugin hosts that own
// every device allocation and hand the library only input and output buffers,
// and serving loops that must not call cudaMalloc while other streams are busy
// (it can synchronise the device).  For them this entry point keeps its
// scratch in a file-scope __device__ array of OSCAR_KV_STATIC_SCRATCH_BYTES.
// The array exists on every GPU that loads the library, for the life of the
// process.  All calls share it: calls whose work overlaps on the GPU (different
// streams, or different host threads without ordering) race on it.  Nothing in
// it has to start at zero: each call zeroes its split-completion counters in
// its first kernel and writes every partial result before reading it, so stale
// contents from an earlier call are never read.
#include <mutex>

#include "internal.h"

namespace {

static __device__ __align__(256) unsigned char g_decode_scratch[OSCAR_KV_STATIC_SCRATCH_BYTES];

std::mutex g_scratch_mu;
void* g_scratch_ptr[64] = {nullptr};

// Device address of the scratch array on the current device, looked up once per
// device (host code cannot use the array's name as a device address).
void* scratch_for_current_device(int* err) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    *err = OSCAR_ERR_LAUNCH;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || !p) {
      *err = OSCAR_ERR_LAUNCH;
      return nullptr;
    }
    g_scratch_ptr[dev] = p;
  }
  return g_scratch_ptr[dev];
}

}  // namespace

extern "C" int attn_decode_static(const oscar_kv_config* cfg, const void* cache, int32_t layer, const void* q,
                                  const int32_t* seq_lens, int32_t seq_len_hint, const float* R_K,
                                  const float* R_V, float sm_scale, int32_t num_splits, void* out, float* lse,
                                  int32_t* dev_status, void* stream) {
  if (!cfg) return OSCAR_ERR_INVALID;
  oscar_kv_layout lay;
  const int v = kv_layout_query(cfg, &lay);
  if (v != OSCAR_OK) return v;
  // the smallest decode (one split) must fit in the fixed array
  const uint64_t one_split = oscar::decode_workspace_bytes(oscar::geom_of(cfg), 1);
  if (one_split > OSCAR_KV_STATIC_SCRATCH_BYTES) return OSCAR_ERR_WORKSPACE;
  int err = OSCAR_OK;
  void* ws = scratch_for_current_device(&err);
  if (!ws) return err;
  return attn_decode(cfg, cache, layer, q, seq_lens, seq_len_hint, R_K, R_V, sm_scale, num_splits, out, lse, ws,
                     OSCAR_KV_STATIC_SCRATCH_BYTES, dev_status, stream);
}

// mla_verify_attn_noalloc: the verify call for callers that cannot allocate device
// memory. The split partials go to a scratch array the library holds itself.
#include <mutex>

#include "common.cuh"

namespace {

constexpr size_t kScratchBytes = MLA_VERIFY_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

// The scratch every call on a device shares. In host code `g_scratch` names a host-side
// stand-in, not device memory: kernels are only ever given the address looked up below.
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

void* g_scratch_addr[kMaxDevices];  // device address of g_scratch, per device, once looked up
std::mutex g_scratch_mutex;

// Device address of the scratch array on the current device (looked up once per device).
int scratch_on_current_device(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return MLA_ERR_NO_DEVICE;
  if (dev >= kMaxDevices) return MLA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || p == nullptr) return MLA_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return MLA_OK;
}

}  // namespace

extern "C" int mla_verify_attn_noalloc(const mla_verify_desc* desc, const void* q, const void* kv_pool,
                                       const int32_t* slot_table, const int32_t* seq_lens,
                                       const int32_t* tree_parent, void* out, float* lse, int32_t* dev_status,
                                       mla_stream_t stream) {
  size_t need = 0;
  int rc = mla_verify_workspace_size(desc, &need);
  if (rc != MLA_OK) return rc;
  if (need > kScratchBytes) return MLA_ERR_WORKSPACE_TOO_SMALL;
  void* scratch = nullptr;
  rc = scratch_on_current_device(&scratch);
  if (rc != MLA_OK) return rc;
  return mla_verify_attn(desc, q, kv_pool, slot_table, seq_lens, tree_parent, out, lse, scratch, kScratchBytes,
                         dev_status, stream);
}

// mla_no_alloc.cu -- mla_decode_no_alloc: the decode for callers that cannot allocate
// device memory.  Its scratch is the static device buffer below instead of a
// caller-provided workspace; everything else is mla_decode unchanged.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/mla_decode.h"

#define MLA_EXPORT extern "C" __attribute__((visibility("default")))

// The scratch every mla_decode_no_alloc call on a device uses (held until process exit).
static __device__ __align__(256) unsigned char g_mla_no_alloc_scratch[MLA_NO_ALLOC_SCRATCH_BYTES];

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch[kMaxDevices] = {nullptr};

// Device address of the static scratch on the current device.  In host code the array's
// name is only a host-side stand-in, so the address comes from cudaGetSymbolAddress,
// looked up once per device with that device current.
mla_status_t scratch_on_current_device(void** ptr) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MLA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return MLA_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_scratch[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_mla_no_alloc_scratch) != cudaSuccess || p == nullptr) return MLA_ERR_CUDA;
    g_scratch[dev] = p;
  }
  *ptr = g_scratch[dev];
  return MLA_OK;
}
}  // namespace

MLA_EXPORT mla_status_t mla_decode_no_alloc(const void* q_nope, const void* q_pe, const void* kv_cache,
                                            const int32_t* block_table, int max_pages, const int32_t* seq_lens,
                                            int B, int q_len, int H, int num_pages, int page_size,
                                            float sm_scale, int kv_dtype, float kv_scale, int num_splits,
                                            void* out, float* lse, mla_stream_t stream, void** scratch_used) {
  if (B == 0)  // an empty batch enqueues nothing and needs no scratch
    return mla_decode(q_nope, q_pe, kv_cache, block_table, max_pages, seq_lens, B, q_len, H, num_pages,
                      page_size, sm_scale, kv_dtype, kv_scale, num_splits, nullptr, 0, out, lse, stream);
  size_t need = 0;
  mla_status_t st = mla_decode_workspace_size(B, q_len, H, num_splits, &need);
  if (st != MLA_OK) return st;
  if (need > (size_t)MLA_NO_ALLOC_SCRATCH_BYTES) return MLA_ERR_WORKSPACE_TOO_SMALL;
  void* scratch = nullptr;
  st = scratch_on_current_device(&scratch);
  if (st != MLA_OK) return st;
  if (scratch_used) *scratch_used = scratch;
  // every word of the scratch a call reads (status words, plan, partials) is written
  // earlier in the same call: the buffer needs no initialisation
  return mla_decode(q_nope, q_pe, kv_cache, block_table, max_pages, seq_lens, B, q_len, H, num_pages, page_size,
                    sm_scale, kv_dtype, kv_scale, num_splits, scratch, (size_t)MLA_NO_ALLOC_SCRATCH_BYTES, out,
                    lse, stream);
}

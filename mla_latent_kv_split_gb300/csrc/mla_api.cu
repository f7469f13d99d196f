// mla_api.cu -- the C ABI (include/mla_decode.h): host-side validation, workspace sizing,
// the host copy of the schedule, and the launches.  Everything is enqueued on the
// caller's stream; nothing here allocates device memory or synchronises, except
// mla_decode_read_status.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <atomic>
#include <mutex>
#include <vector>

#include "mla_device.cuh"

#define MLA_EXPORT extern "C" __attribute__((visibility("default")))

namespace mla {
cudaError_t launch_decode_tc(const DecodeParams& p, cudaStream_t stream);
cudaError_t launch_decode_small(const DecodeParams& p, int parts_max, cudaStream_t stream);
int tc_max_clusters();
cudaError_t launch_splitk_reduce(uint8_t* ws, int U, int H, int slots_cap, int status_ctas, const float* sinks,
                                 uint16_t* out, float* lse, cudaStream_t stream, bool pdl);
cudaError_t launch_kv_append(const uint16_t* latent, long long latent_stride, const uint16_t* rope,
                             long long rope_stride, const int64_t* slots, int T, uint8_t* cache, long long num_slots,
                             int page_size, int kv_dtype, float kv_scale, uint32_t* status, cudaStream_t stream);
cudaError_t launch_batched_gemv(const uint16_t* x, long long x_token_stride, long long x_head_stride,
                                const uint16_t* w, uint16_t* out, long long out_token_stride,
                                long long out_head_stride, int T, int H, int N, int K, uint32_t* status,
                                cudaStream_t stream);
}  // namespace mla

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_mu;
int g_workers[kMaxDevices] = {0};

// Scheduling workers on the current device: one per co-resident 2-CTA cluster of the
// tensor-core kernel (at most one per pair of SMs).
cudaError_t current_workers(int* workers) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_workers[dev] == 0) {
    int sms = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    int w = sms >= 2 ? sms / 2 : 1;
    int clusters = mla::tc_max_clusters();
    if (clusters > 0 && clusters < w) w = clusters;
    if (w > mla::kMaxCtas / 2) w = mla::kMaxCtas / 2;  // one status word per CTA in the header
    g_workers[dev] = w;
  }
  *workers = g_workers[dev];
  return cudaSuccess;
}

bool aligned(const void* p, uintptr_t a) { return ((uintptr_t)p % a) == 0; }

mla_status_t check_shape(int B, int q_len, int H, int num_splits) {
  if (B < 0 || q_len < 1 || H < 1 || num_splits < 0) return MLA_ERR_INVALID_ARG;
  if (H % 16 != 0 || H > MLA_MAX_HEADS) return MLA_ERR_UNSUPPORTED;
  if (q_len > MLA_MAX_Q_LEN) return MLA_ERR_UNSUPPORTED;
  if ((long long)B * q_len > MLA_MAX_UNITS) return MLA_ERR_UNSUPPORTED;
  if (num_splits > 4096) return MLA_ERR_UNSUPPORTED;
  return MLA_OK;
}

mla_status_t check_geometry(int B, int q_len, int max_pages, int num_pages, int page_size) {
  if (max_pages < 1 || num_pages < 1) return MLA_ERR_INVALID_ARG;
  if (page_size != 32 && page_size != 64) return MLA_ERR_UNSUPPORTED;
  if ((long long)max_pages * page_size > 0x7fffffffLL) return MLA_ERR_UNSUPPORTED;
  if ((long long)B * q_len * max_pages > 0x7fffffffLL) return MLA_ERR_UNSUPPORTED;
  return MLA_OK;
}

size_t required_bytes(int units, int H, int num_splits, int workers) {
  return mla::workspace_bytes_for(mla::max_slots(units, num_splits, workers), H);
}

int slots_that_fit(size_t workspace_bytes, int H) {
  if (workspace_bytes < mla::kHeaderBytes) return 0;
  size_t per = (size_t)H * (mla::kLatent + 1) * 4;
  size_t n = (workspace_bytes - mla::kHeaderBytes) / per;
  return n > 0x7fffffff ? 0x7fffffff : (int)n;
}

// bf16 calls whose ranges span at most this many cache positions run on the CUDA-core
// kernel; see mla_decode_set_small_call_limit.
std::atomic<size_t> g_small_call_limit{MLA_SMALL_CALL_DEFAULT};

// CTAs of the CUDA-core kernel for this call, or 0 when it goes to the tensor-core kernel.
// A range's positions are bounded by the table's capacity (one range per (b, i)), or with
// forced splits by the span of one part: roundup(cdiv(capacity, num_splits), 64).  The
// kernel's CTAs (one per range and head, one resident per SM) must fit in one wave: a
// second wave costs more than the tensor-core kernel's set-up.
int small_call_ctas(int kv_dtype, int U, int H, int max_pages, int page_size, int num_splits, int workers) {
  if (kv_dtype != MLA_KV_BF16) return 0;
  const size_t cap = (size_t)max_pages * page_size;
  const size_t span = num_splits > 0 ? (cap + num_splits - 1) / num_splits : cap;
  if (((span + 63) & ~(size_t)63) > g_small_call_limit.load(std::memory_order_relaxed)) return 0;
  const size_t ctas = (size_t)U * (num_splits > 0 ? num_splits : 1) * H;
  return ctas <= (size_t)2 * workers && ctas <= (size_t)mla::kMaxCtas ? (int)ctas : 0;
}

}  // namespace

MLA_EXPORT size_t mla_decode_set_small_call_limit(size_t limit) {
  return g_small_call_limit.exchange(limit);
}

MLA_EXPORT int mla_decode_abi_version(void) { return 3; }

MLA_EXPORT const char* mla_status_string(mla_status_t s) {
  switch (s) {
    case MLA_OK: return "MLA_OK";
    case MLA_ERR_INVALID_ARG: return "MLA_ERR_INVALID_ARG";
    case MLA_ERR_UNSUPPORTED: return "MLA_ERR_UNSUPPORTED";
    case MLA_ERR_WORKSPACE_TOO_SMALL: return "MLA_ERR_WORKSPACE_TOO_SMALL";
    case MLA_ERR_CUDA: return "MLA_ERR_CUDA";
    case MLA_ERR_DEVICE_STATUS: return "MLA_ERR_DEVICE_STATUS";
  }
  return "MLA_ERR_UNKNOWN";
}

MLA_EXPORT mla_status_t mla_decode_num_workers(int* workers) {
  if (!workers) return MLA_ERR_INVALID_ARG;
  return current_workers(workers) == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

MLA_EXPORT mla_status_t mla_decode_workspace_size(int B, int q_len, int H, int num_splits,
                                                  size_t* bytes) {
  if (!bytes || B < 1) return MLA_ERR_INVALID_ARG;
  mla_status_t st = check_shape(B, q_len, H, num_splits);
  if (st != MLA_OK) return st;
  // forced splits bound the partials per (b, i) without reference to the device
  int C = 0;
  if (num_splits == 0 && current_workers(&C) != cudaSuccess) return MLA_ERR_CUDA;
  *bytes = required_bytes(B * q_len, H, num_splits, C);
  return MLA_OK;
}

MLA_EXPORT mla_status_t mla_decode_plan_host(const int32_t* seq_lens, int B, int q_len, int max_pages,
                                             int page_size, int num_splits, int window, int workers,
                                             int32_t* unit_tile_begin, int32_t* unit_tiles,
                                             int32_t* unit_parts, int32_t* unit_slot,
                                             int32_t* slots_used) {
  if (!seq_lens || !unit_tile_begin || !unit_tiles || !unit_parts || !unit_slot || !slots_used)
    return MLA_ERR_INVALID_ARG;
  if (B < 1 || window < 0) return MLA_ERR_INVALID_ARG;
  mla_status_t st = check_shape(B, q_len, 16, num_splits);
  if (st != MLA_OK) return st;
  st = check_geometry(B, q_len, max_pages, 1, page_size);
  if (st != MLA_OK) return st;
  int C = workers;
  if (C <= 0 && current_workers(&C) != cudaSuccess) return MLA_ERR_CUDA;
  std::vector<mla::UnitPlan> plan((size_t)B * q_len);
  int slots = mla::plan_host(seq_lens, B, q_len, max_pages, page_size, num_splits, C, plan.data(), window);
  for (int u = 0; u < B * q_len; ++u) {
    unit_tile_begin[u] = plan[u].tile_begin;
    unit_tiles[u] = plan[u].tiles;
    unit_parts[u] = plan[u].parts;
    unit_slot[u] = plan[u].slot;
  }
  *slots_used = slots;
  return MLA_OK;
}

MLA_EXPORT mla_status_t mla_decode_ex(const void* q_nope, const void* q_pe, const void* kv_cache,
                                      const int32_t* block_table, int max_pages, const int32_t* seq_lens,
                                      int B, int q_len, int H, int num_pages, int page_size, float sm_scale,
                                      int kv_dtype, float kv_scale, int num_splits, int window,
                                      const float* sinks, void* workspace, size_t workspace_bytes, void* out,
                                      float* lse, mla_stream_t stream) {
  if (window < 0) return MLA_ERR_INVALID_ARG;
  mla_status_t st = check_shape(B, q_len, H, num_splits);
  if (st != MLA_OK) return st;
  st = check_geometry(B, q_len, max_pages, num_pages, page_size);
  if (st != MLA_OK) return st;
  if (kv_dtype != MLA_KV_BF16 && kv_dtype != MLA_KV_FP8_E4M3 && kv_dtype != MLA_KV_NVFP4)
    return MLA_ERR_INVALID_ARG;
  if (!isfinite(sm_scale)) return MLA_ERR_INVALID_ARG;
  if (kv_dtype == MLA_KV_FP8_E4M3 && !(isfinite(kv_scale) && kv_scale > 0.f)) return MLA_ERR_INVALID_ARG;
  if (B == 0) return MLA_OK;
  if (!q_nope || !q_pe || !kv_cache || !block_table || !seq_lens || !workspace || !out)
    return MLA_ERR_INVALID_ARG;
  if (!aligned(q_nope, 16) || !aligned(q_pe, 16) || !aligned(kv_cache, 128) || !aligned(block_table, 16) ||
      !aligned(seq_lens, 4) || !aligned(workspace, 256) || !aligned(out, 16) || (lse && !aligned(lse, 4)) ||
      (sinks && !aligned(sinks, 4)))
    return MLA_ERR_INVALID_ARG;
  int C = 0;
  if (current_workers(&C) != cudaSuccess) return MLA_ERR_CUDA;
  const int U = B * q_len;
  if (workspace_bytes < required_bytes(U, H, num_splits, C)) return MLA_ERR_WORKSPACE_TOO_SMALL;

  mla::DecodeParams p;
  p.q_nope = static_cast<const uint16_t*>(q_nope);
  p.q_pe = static_cast<const uint16_t*>(q_pe);
  p.cache = static_cast<const uint8_t*>(kv_cache);
  p.block_table = block_table;
  p.seq_lens = seq_lens;
  p.max_pages = max_pages;
  p.B = B;
  p.q_len = q_len;
  p.H = H;
  p.num_pages = num_pages;
  p.page_size = page_size;
  p.sm_scale = sm_scale;
  p.kv_scale = kv_dtype == MLA_KV_FP8_E4M3 ? kv_scale : 1.f;
  p.kv_dtype = kv_dtype;
  p.num_splits = num_splits;
  p.workers = C;
  p.slots_cap = slots_that_fit(workspace_bytes, H);
  p.ws = static_cast<uint8_t*>(workspace);
  p.out = static_cast<uint16_t*>(out);
  p.lse = lse;
  p.window = window;
  p.sinks = sinks;

  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // No host-side reset: each decode CTA writes its status word at exit and the reduce (which
  // always runs, after the decode) folds them into the call's status word.
  const int small_ctas = small_call_ctas(kv_dtype, U, H, max_pages, page_size, num_splits, p.workers);
  cudaError_t le = small_ctas > 0 ? mla::launch_decode_small(p, num_splits > 0 ? num_splits : 1, s)
                                  : mla::launch_decode_tc(p, s);
  if (le != cudaSuccess) return MLA_ERR_CUDA;
  const int status_ctas = small_ctas > 0 ? small_ctas : 2 * p.workers;
  if (mla::launch_splitk_reduce(p.ws, U, H, p.slots_cap, status_ctas, sinks, p.out, lse, s, true) != cudaSuccess)
    return MLA_ERR_CUDA;
  return MLA_OK;
}

MLA_EXPORT mla_status_t mla_decode(const void* q_nope, const void* q_pe, const void* kv_cache,
                                   const int32_t* block_table, int max_pages, const int32_t* seq_lens,
                                   int B, int q_len, int H, int num_pages, int page_size, float sm_scale,
                                   int kv_dtype, float kv_scale, int num_splits, void* workspace,
                                   size_t workspace_bytes, void* out, float* lse, mla_stream_t stream) {
  return mla_decode_ex(q_nope, q_pe, kv_cache, block_table, max_pages, seq_lens, B, q_len, H, num_pages, page_size,
                       sm_scale, kv_dtype, kv_scale, num_splits, 0, nullptr, workspace, workspace_bytes, out, lse,
                       stream);
}

MLA_EXPORT mla_status_t mla_splitk_reduce(const void* workspace, size_t workspace_bytes, int B, int q_len,
                                          int H, const float* sinks, void* out, float* lse, mla_stream_t stream) {
  mla_status_t st = check_shape(B, q_len, H, 0);
  if (st != MLA_OK) return st;
  if (B == 0) return MLA_OK;
  if (!workspace || !out) return MLA_ERR_INVALID_ARG;
  if (!aligned(workspace, 256) || !aligned(out, 16) || (lse && !aligned(lse, 4)) || (sinks && !aligned(sinks, 4)))
    return MLA_ERR_INVALID_ARG;
  if (workspace_bytes < mla::kHeaderBytes) return MLA_ERR_WORKSPACE_TOO_SMALL;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (mla::launch_splitk_reduce(static_cast<uint8_t*>(const_cast<void*>(workspace)), B * q_len, H,
                                slots_that_fit(workspace_bytes, H), 0, sinks, static_cast<uint16_t*>(out), lse, s,
                                false) != cudaSuccess)
    return MLA_ERR_CUDA;
  return MLA_OK;
}

MLA_EXPORT mla_status_t mla_decode_read_status(const void* workspace, uint32_t* device_status,
                                               mla_stream_t stream) {
  if (!workspace || !device_status) return MLA_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  uint32_t v = 0;
  if (cudaMemcpyAsync(&v, workspace, 4, cudaMemcpyDeviceToHost, s) != cudaSuccess) return MLA_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return MLA_ERR_CUDA;
  *device_status = v;
  return v ? MLA_ERR_DEVICE_STATUS : MLA_OK;
}

MLA_EXPORT mla_status_t mla_kv_append(const void* latent, int64_t latent_stride, const void* rope, int64_t rope_stride,
                                      const int64_t* slots, int T, void* kv_cache, int num_pages, int page_size,
                                      int kv_dtype, float kv_scale, uint32_t* device_status, mla_stream_t stream) {
  if (T < 0 || num_pages < 1) return MLA_ERR_INVALID_ARG;
  if (page_size != 32 && page_size != 64) return MLA_ERR_UNSUPPORTED;
  if (kv_dtype != MLA_KV_BF16 && kv_dtype != MLA_KV_FP8_E4M3 && kv_dtype != MLA_KV_NVFP4) return MLA_ERR_INVALID_ARG;
  if (kv_dtype == MLA_KV_FP8_E4M3 && !(isfinite(kv_scale) && kv_scale > 0.f)) return MLA_ERR_INVALID_ARG;
  if (T == 0) return MLA_OK;
  if (!latent || !rope || !slots || !kv_cache) return MLA_ERR_INVALID_ARG;
  if (latent_stride < 512 || rope_stride < 64 || latent_stride % 8 || rope_stride % 8) return MLA_ERR_INVALID_ARG;
  if (!aligned(latent, 16) || !aligned(rope, 16) || !aligned(slots, 8) || !aligned(kv_cache, 128) ||
      (device_status && !aligned(device_status, 4)))
    return MLA_ERR_INVALID_ARG;
  if (mla::launch_kv_append(static_cast<const uint16_t*>(latent), latent_stride, static_cast<const uint16_t*>(rope),
                            rope_stride, slots, T, static_cast<uint8_t*>(kv_cache), (long long)num_pages * page_size,
                            page_size, kv_dtype, kv_dtype == MLA_KV_FP8_E4M3 ? kv_scale : 1.f, device_status,
                            reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return MLA_ERR_CUDA;
  return MLA_OK;
}

MLA_EXPORT mla_status_t mla_batched_gemv(const void* x, int64_t x_token_stride, int64_t x_head_stride,
                                         const void* weight, void* out, int64_t out_token_stride,
                                         int64_t out_head_stride, int T, int H, int N, int K,
                                         uint32_t* device_status, mla_stream_t stream) {
  if (T < 0 || H < 1 || N < 1 || K < 8 || K % 8) return MLA_ERR_INVALID_ARG;
  if ((long long)H * N > 0x7fffffffLL || T > 0xffffff || H > 65535) return MLA_ERR_UNSUPPORTED;
  if (T == 0) return MLA_OK;
  if (!x || !weight || !out) return MLA_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(weight, 16) || !aligned(out, 16) || (device_status && !aligned(device_status, 4)))
    return MLA_ERR_INVALID_ARG;
  if (x_head_stride < K || x_head_stride % 8 || x_token_stride % 8 || x_token_stride < (int64_t)H * x_head_stride)
    return MLA_ERR_INVALID_ARG;
  if (out_head_stride < N || out_token_stride < 0) return MLA_ERR_INVALID_ARG;
  cudaError_t e = mla::launch_batched_gemv(static_cast<const uint16_t*>(x), x_token_stride, x_head_stride,
                                           static_cast<const uint16_t*>(weight), static_cast<uint16_t*>(out),
                                           out_token_stride, out_head_stride, T, H, N, K, device_status,
                                           reinterpret_cast<cudaStream_t>(stream));
  if (e == cudaErrorInvalidValue) return MLA_ERR_INVALID_ARG;
  return e == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

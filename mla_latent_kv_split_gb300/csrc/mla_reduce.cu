// mla_reduce.cu -- LSE-weighted split-K combine (TileGym mla_decoding_split_kv.py calls
// splitk_reduce on the per-split outputs and log-sum-exps).
//
// For a (b, i) cut into S > 1 parts with partials (o_s [H,512], lse_s [H]):
//   M = max_s lse_s;  lse = M + log(sum_s exp(lse_s - M));  out = sum_s exp(lse_s - lse) o_s.
// A (b, i) with nothing visible gets out = 0 and lse = -inf; one with a single part was
// written by the decode kernel and is skipped.  One CTA of 128 threads per (unit, head):
// each thread owns 4 consecutive output columns (one float4 per partial).
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "mla_device.cuh"

namespace mla {

constexpr int kReduceThreads = 128;

__global__ void __launch_bounds__(kReduceThreads)
mla_splitk_reduce_kernel(const uint8_t* __restrict__ ws, int U, int H, int slots_cap,
                         uint16_t* __restrict__ out, float* __restrict__ lse) {
  // Programmatic dependent launch: everything before this point overlaps the decode
  // kernel's tail; the plan and partials are read only after the decode has completed.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int u = blockIdx.x, h = blockIdx.y, tid = threadIdx.x;
  const int2 pl = reinterpret_cast<const int2*>(ws + kPlanOffset)[u];
  const int parts = pl.x, slot = pl.y;
  const size_t row = (size_t)u * H + h;
  if (parts == 1) return;
  uint2 packed;
  float lse_v;
  if (parts <= 0 || slot < 0 || slot + parts > slots_cap) {
    packed = make_uint2(0u, 0u);
    lse_v = -INFINITY;
  } else {
    const float* pls = reinterpret_cast<const float*>(ws + partial_lse_offset(slots_cap, H));
    const float4* po = reinterpret_cast<const float4*>(ws + partial_o_offset());
    float M = -INFINITY;
    for (int s = 0; s < parts; ++s) M = fmaxf(M, pls[(size_t)(slot + s) * H + h]);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (M == -INFINITY) {
      lse_v = -INFINITY;
    } else {
      float tot = 0.f;
      for (int s = 0; s < parts; ++s) tot += expf(pls[(size_t)(slot + s) * H + h] - M);
      lse_v = M + logf(tot);
      for (int s = 0; s < parts; ++s) {
        float w = expf(pls[(size_t)(slot + s) * H + h] - lse_v);
        float4 v = po[((size_t)(slot + s) * H + h) * (kLatent / 4) + tid];
        acc.x = fmaf(w, v.x, acc.x);
        acc.y = fmaf(w, v.y, acc.y);
        acc.z = fmaf(w, v.z, acc.z);
        acc.w = fmaf(w, v.w, acc.w);
      }
    }
    packed.x = (unsigned)float_to_bf16_bits_rn(acc.x) | ((unsigned)float_to_bf16_bits_rn(acc.y) << 16);
    packed.y = (unsigned)float_to_bf16_bits_rn(acc.z) | ((unsigned)float_to_bf16_bits_rn(acc.w) << 16);
  }
  reinterpret_cast<uint2*>(out + row * kLatent)[tid] = packed;
  if (lse && tid == 0) lse[row] = lse_v;
}

cudaError_t launch_splitk_reduce(const uint8_t* ws, int U, int H, int slots_cap, uint16_t* out,
                                 float* lse, cudaStream_t stream, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(U, H);
  cfg.blockDim = dim3(kReduceThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, mla_splitk_reduce_kernel, ws, U, H, slots_cap, out, lse);
}

}  // namespace mla

// mla_reduce.cu -- LSE-weighted split-K combine (TileGym mla_decoding_split_kv.py calls
// splitk_reduce on the per-split outputs and log-sum-exps).
//
// For a (b, i) cut into S > 1 parts with partials (o_s [H,512], lse_s [H]):
//   lse = log sum_s exp(lse_s);  out = sum_s exp(lse_s - lse) o_s.
// evaluated in one pass with a running maximum (parts taken two at a time).  A (b, i) with
// nothing visible gets out = 0 and lse = -inf; one with a single part was written by the
// decode kernel and is skipped.  With per-head attention sinks (gpt-oss style: one extra
// logit per head that takes part in the normaliser but has no value row), the sink joins
// the combined normaliser here: lse' = log(exp(lse) + exp(sink_h)), out' = out *
// exp(lse - lse'); a (b, i) with nothing visible then gets lse = sink_h.  After a decode, the first CTA also folds the decode CTAs'
// status bits into the call's status word.
//
// One CTA of 256 threads per (unit, 32 heads, 128 columns): lane = head, warp = one 16-column
// group.  The partials are stored column-octet-major ([slot][64][H][8] bf16), so for one
// octet a warp's 32 heads are 512 contiguous bytes; each thread reads its 16 columns as two
// such coalesced loads per part and writes its 32 output bytes whole.  Every load of a
// group of parts is issued before any is used: a part group costs one memory round trip,
// and the whole grid (units x H/32 x 4 CTAs) is resident at once.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "mla_device.cuh"

namespace mla {

constexpr int kReduceThreads = 256;
constexpr int kReduceHeads = 32;                     // lanes
constexpr int kReduceColGroups = kReduceThreads / 32;  // warps: 16 columns each
constexpr int kPartGroup = 3;

__global__ void __launch_bounds__(kReduceThreads, 4)
mla_splitk_reduce_kernel(uint8_t* __restrict__ ws, int U, int H, int slots_cap, int status_ctas,
                         const float* __restrict__ sinks, uint16_t* __restrict__ out, float* __restrict__ lse) {
  // Programmatic dependent launch: everything before this point overlaps the decode
  // kernel's tail; the plan and partials are read only after the decode has completed.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (status_ctas > 0 && blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0 && threadIdx.x < 32) {
    // the call's status word: the OR of every decode CTA's status bits
    unsigned bits = 0;
    for (int c = threadIdx.x; c < status_ctas; c += 32) bits |= reinterpret_cast<const unsigned*>(ws + kCtaStatusOffset)[c];
    bits = __reduce_or_sync(0xffffffffu, bits);
    if (threadIdx.x == 0) *reinterpret_cast<unsigned*>(ws) = bits;
  }
  const int u = blockIdx.x, lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int h = blockIdx.y * kReduceHeads + lane;
  const int col0 = 16 * kReduceColGroups * blockIdx.z + 16 * warp;  // this thread's 16 output columns
  if (h >= H) return;
  const int2 pl = reinterpret_cast<const int2*>(ws + kPlanOffset)[u];
  const int parts = pl.x, slot = pl.y;
  if (parts == 1) return;
  const size_t row = (size_t)u * H + h;
  float acc[16];
#pragma unroll
  for (int k = 0; k < 16; ++k) acc[k] = 0.f;
  float m = -INFINITY, l = 0.f;
  if (parts > 1 && slot >= 0 && slot + parts <= slots_cap) {
    const float* pls = reinterpret_cast<const float*>(ws + partial_lse_offset(slots_cap, H));
    const uint4* po = reinterpret_cast<const uint4*>(ws + partial_o_offset());
    for (int s0 = 0; s0 < parts; s0 += kPartGroup) {
      float ls[kPartGroup];
      uint4 v[kPartGroup][2];
#pragma unroll
      for (int j = 0; j < kPartGroup; ++j) {
        const bool ok = s0 + j < parts;
        const size_t r = (size_t)(slot + s0 + j);
        ls[j] = ok ? pls[r * H + h] : -INFINITY;
#pragma unroll
        for (int k = 0; k < 2; ++k) v[j][k] = ok ? po[(r * 64 + (col0 >> 3) + k) * H + h] : make_uint4(0u, 0u, 0u, 0u);
      }
      float mn = m;
#pragma unroll
      for (int j = 0; j < kPartGroup; ++j) mn = fmaxf(mn, ls[j]);
      if (mn == -INFINITY) continue;
      const float sc = expf(m - mn);  // m = -inf -> 0
      l *= sc;
#pragma unroll
      for (int k = 0; k < 16; ++k) acc[k] *= sc;
#pragma unroll
      for (int j = 0; j < kPartGroup; ++j) {
        const float w = expf(ls[j] - mn);  // missing parts: -inf -> 0
        l += w;
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          const uint32_t e[4] = {v[j][k].x, v[j][k].y, v[j][k].z, v[j][k].w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            acc[8 * k + 2 * i] = fmaf(w, __uint_as_float(e[i] << 16), acc[8 * k + 2 * i]);
            acc[8 * k + 2 * i + 1] = fmaf(w, __uint_as_float(e[i] & 0xFFFF0000u), acc[8 * k + 2 * i + 1]);
          }
        }
      }
      m = mn;
    }
  }
  if (sinks != nullptr) {
    const float sk = __ldg(sinks + h);
    const float mn = fmaxf(m, sk);
    if (mn != -INFINITY) {
      const float sc = l > 0.f ? expf(m - mn) : 0.f;
      l = l * sc + expf(sk - mn);
#pragma unroll
      for (int k = 0; k < 16; ++k) acc[k] *= sc;
      m = mn;
    }
  }
  const float inv = l > 0.f ? 1.f / l : 0.f;
  uint32_t pk[8];
#pragma unroll
  for (int k = 0; k < 8; ++k)
    pk[k] = (uint32_t)float_to_bf16_bits_rn(acc[2 * k] * inv) | ((uint32_t)float_to_bf16_bits_rn(acc[2 * k + 1] * inv) << 16);
  uint4* dst = reinterpret_cast<uint4*>(out + row * kLatent + col0);
  dst[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
  dst[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
  if (lse && blockIdx.z == 0 && warp == 0) lse[row] = l > 0.f ? m + logf(l) : -INFINITY;
}

cudaError_t launch_splitk_reduce(uint8_t* ws, int U, int H, int slots_cap, int status_ctas, const float* sinks,
                                 uint16_t* out, float* lse, cudaStream_t stream, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(U, (H + kReduceHeads - 1) / kReduceHeads, kLatent / (16 * kReduceColGroups));
  cfg.blockDim = dim3(kReduceThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, mla_splitk_reduce_kernel, ws, U, H, slots_cap, status_ctas, sinks, out, lse);
}

}  // namespace mla

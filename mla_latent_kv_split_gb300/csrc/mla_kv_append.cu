// mla_kv_append.cu -- writes this step's new tokens into the paged latent cache, quantising
// on the way in (tokenspeed "tokenspeed_mla.py", CuteDSLMLABackend.forward_decode: the new
// tokens' latent and rope go to their cache locations before the decode reads them; metrale
// "kv_cache_mla.rs", mla_cache_assemble and the NVFP4 / FP8 page layouts).
//
// One thread per 16-value group of two tokens: a token is 36 groups (32 latent, 4 rope), a
// block of 288 threads takes 16 tokens (thread i: group i % 36 of tokens i / 36 and i / 36 + 8),
// so a warp reads 32 consecutive groups (1 KB) of one token.  Both tokens' loads are issued
// before either is converted: with the occupancy bound below (5 blocks per SM) more bytes are
// in flight than with one token per thread at 7 blocks per SM, which is what the quantising
// formats need (FP8 -5 %, NVFP4 -7 % at 65,536 tokens; bf16 equal).
//   bf16 : the group's 32 bytes copied.
//   FP8  : 16 E4M3 codes of x / kv_scale (fp32 quotient), one 16-byte store.
//   NVFP4: scale s = E4M3(amax / 6), 16 E2M1 codes of x / value(s) packed two per byte
//          (element 2j in the low nibble of byte j, one 8-byte store), the scale byte in the
//          page's scale section.  A group whose scale is 0 stores zero codes.
// Conversions use the hardware's round-to-nearest-even, saturating (satfinite) converts.
// Quotients are the correctly rounded fp32 x / d, computed as x * r with r the correctly
// rounded reciprocal of d and one correction step (Markstein's method): the remainder
// x - q*d is exact by FMA and q + remainder * r rounds to the nearest quotient.
// HBM-bound; at a decode step's few hundred tokens, launch-latency-bound.
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/mla_decode.h"

namespace mla {

namespace {

constexpr int kGroups = 36;                      // 16-value groups per 576-value token
constexpr int kAppendRows = 8;                   // token rows per block (36 threads each)
constexpr int kTokensPerThread = 2;              // tokens kAppendRows apart
constexpr int kAppendTokens = kAppendRows * kTokensPerThread;  // tokens per block
constexpr int kAppendThreads = kGroups * kAppendRows;

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

// Two values -> two E4M3 codes, `lo` in the low byte.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  uint16_t d;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(d) : "f"(hi), "f"(lo));
  return d;
}

// Eight values -> eight E2M1 codes in one word, element 2j in the low nibble of byte j.
__device__ __forceinline__ uint32_t e2m1x8(const float* x) {
  uint32_t d;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
      "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
      : "=r"(d)
      : "f"(x[0]), "f"(x[1]), "f"(x[2]), "f"(x[3]), "f"(x[4]), "f"(x[5]), "f"(x[6]), "f"(x[7]));
  return d;
}

// x / d rounded to nearest even, for d > 0 finite and r = RN(1 / d) (Markstein's final
// step).  An exact quotient (zero remainder: zeros keep their sign) and a non-finite first
// approximation (an infinite x) are returned as they are.
__device__ __forceinline__ float div_rn_by(float x, float d, float r) {
  const float q0 = x * r;
  const float e = fmaf(-q0, d, x);
  return (e == 0.f || !isfinite(q0)) ? q0 : fmaf(e, r, q0);
}
__device__ __forceinline__ float rcp_rn(float d) {
  float r;
  asm("rcp.rn.f32 %0, %1;" : "=f"(r) : "f"(d));
  return r;
}

// Value of one E4M3 code (exact: every E4M3 value is an f16 value).
__device__ __forceinline__ float e4m3_value(uint32_t code) {
  uint32_t h2;
  const uint16_t c = (uint16_t)(code & 0xFFu);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(c));
  return __half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFFu)));
}

}  // namespace

// Group g of one token (its 16 values: a, b) -> the token's cache location `slot`.
__device__ __forceinline__ void append_group(uint4 a, uint4 b, long long slot, int g, uint8_t* __restrict__ cache,
                                             int page_size, int kv_dtype, float kv_scale) {
  if (kv_dtype == MLA_KV_BF16) {
    uint4* dst = reinterpret_cast<uint4*>(cache + (size_t)slot * (MLA_CACHE_DIM * 2) + 32 * g);
    dst[0] = a;
    dst[1] = b;
    return;
  }
  float x[16];
  {
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      x[2 * k] = bf16_lo(w[k]);
      x[2 * k + 1] = bf16_hi(w[k]);
    }
  }
  if (kv_dtype == MLA_KV_FP8_E4M3) {
    const float r = rcp_rn(kv_scale);
    uint32_t w[4];
#pragma unroll
    for (int k = 0; k < 4; ++k)
      w[k] = e4m3x2(div_rn_by(x[4 * k], kv_scale, r), div_rn_by(x[4 * k + 1], kv_scale, r)) |
             (e4m3x2(div_rn_by(x[4 * k + 2], kv_scale, r), div_rn_by(x[4 * k + 3], kv_scale, r)) << 16);
    *reinterpret_cast<uint4*>(cache + (size_t)slot * MLA_CACHE_DIM + 16 * g) = make_uint4(w[0], w[1], w[2], w[3]);
    return;
  }
  float amax = 0.f;
#pragma unroll
  for (int k = 0; k < 16; ++k) amax = fmaxf(amax, fabsf(x[k]));
  const uint32_t s_code = e4m3x2(div_rn_by(amax, 6.f, rcp_rn(6.f)), 0.f) & 0xFFu;
  const float sv = e4m3_value(s_code);
  uint32_t d0 = 0u, d1 = 0u;
  if (sv > 0.f) {
    const float r = rcp_rn(sv);
#pragma unroll
    for (int k = 0; k < 16; ++k) x[k] = div_rn_by(x[k], sv, r);
    d0 = e2m1x8(x);
    d1 = e2m1x8(x + 8);
  }
  const long long page = slot / page_size, row = slot - page * page_size;
  uint8_t* base = cache + (size_t)page * ((size_t)page_size * (MLA_CACHE_DIM / 2 + MLA_CACHE_DIM / 16));
  *reinterpret_cast<uint2*>(base + row * (MLA_CACHE_DIM / 2) + 8 * g) = make_uint2(d0, d1);
  base[(size_t)page_size * (MLA_CACHE_DIM / 2) + row * (MLA_CACHE_DIM / 16) + g] = (uint8_t)s_code;
}


__global__ void __launch_bounds__(kAppendThreads, 5)
mla_kv_append_kernel(const uint16_t* __restrict__ latent, long long latent_stride, const uint16_t* __restrict__ rope,
                     long long rope_stride, const int64_t* __restrict__ slots, int T, uint8_t* __restrict__ cache,
                     long long num_slots, int page_size, int kv_dtype, float kv_scale, uint32_t* status) {
  const int row = threadIdx.x / kGroups;
  const int g = threadIdx.x % kGroups;
  uint4 a[kTokensPerThread], b[kTokensPerThread];
  long long slot[kTokensPerThread];
#pragma unroll
  for (int j = 0; j < kTokensPerThread; ++j) {
    const int t = blockIdx.x * kAppendTokens + j * kAppendRows + row;
    slot[j] = -1;  // past the end: nothing to write
    if (t < T) {
      slot[j] = __ldg(slots + t);
      const uint16_t* lat = latent + (size_t)t * latent_stride;
      const uint16_t* rp = rope + (size_t)t * rope_stride;
      const uint4* src = reinterpret_cast<const uint4*>(g < 32 ? lat + 16 * g : rp + 16 * (g - 32));
      a[j] = __ldg(src);
      b[j] = __ldg(src + 1);
    }
  }
#pragma unroll
  for (int j = 0; j < kTokensPerThread; ++j) {
    if (slot[j] < 0) continue;  // padding
    if (slot[j] >= num_slots) {
      if (g == 0 && status != nullptr) atomicOr(status, MLA_STATUS_SLOT_OUT_OF_RANGE);
      continue;
    }
    append_group(a[j], b[j], slot[j], g, cache, page_size, kv_dtype, kv_scale);
  }
}

cudaError_t launch_kv_append(const uint16_t* latent, long long latent_stride, const uint16_t* rope,
                             long long rope_stride, const int64_t* slots, int T, uint8_t* cache, long long num_slots,
                             int page_size, int kv_dtype, float kv_scale, uint32_t* status, cudaStream_t stream) {
  const int blocks = (T + kAppendTokens - 1) / kAppendTokens;
  mla_kv_append_kernel<<<blocks, kAppendThreads, 0, stream>>>(latent, latent_stride, rope, rope_stride, slots, T,
                                                              cache, num_slots, page_size, kv_dtype, kv_scale, status);
  return cudaGetLastError();
}

}  // namespace mla

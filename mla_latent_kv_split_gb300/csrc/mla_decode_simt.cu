// mla_decode_simt.cu -- straightforward CUDA-core split-KV MLA decode (fp32 FMA).
//
// Kept as the plain cross-check of the tensor-core kernel: one CTA per (scheduling
// worker, group of 16 heads) walks the worker's work items; per 32-token chunk it decodes
// the cache rows to fp32 in shared memory, scores them against the 16 absorbed queries
// ([q_nope | q_pe], 576 wide), runs the online softmax, and accumulates
// O[16 x 512] += P[16 x 32] . V[32 x 512] with V = the latent columns of the same rows
// (TileGym mla_decoding_split_kv.py: K = V = KV; tokenspeed forward_decode: paged cache).
// Finished (b, i) go straight to `out`/`lse`; split ones to the workspace partials.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "mla_device.cuh"

namespace mla {

constexpr int kSimtHeads = 16;
constexpr int kSimtChunk = 32;
constexpr int kSimtThreads = 256;
constexpr int kRowPad = kDim + 1;  // 577: conflict-free row stride in shared memory

struct SimtSmem {
  float q[kSimtHeads][kRowPad];
  float kv[kSimtChunk][kRowPad];
  float p[kSimtHeads][kSimtChunk];
  int valid[kSimtChunk];
  int scratch[33];
  PlanSmem plan;
};

__device__ __forceinline__ float load_cache_value(const DecodeParams& p, int page, int row, int col) {
  if (p.kv_dtype == MLA_KV_BF16) {
    const uint16_t* c = reinterpret_cast<const uint16_t*>(p.cache);
    return bf16_bits_to_float(c[((size_t)page * p.page_size + row) * kDim + col]);
  }
  if (p.kv_dtype == MLA_KV_FP8_E4M3) {
    return e4m3_to_float(p.cache[((size_t)page * p.page_size + row) * kDim + col]) * p.kv_scale;
  }
  const uint8_t* base = p.cache + (size_t)page * page_stride_bytes(MLA_KV_NVFP4, p.page_size);
  unsigned byte = base[row * (kDim / 2) + (col >> 1)];
  unsigned nib = (col & 1) ? (byte >> 4) : (byte & 0xFu);
  unsigned sc = base[(size_t)p.page_size * (kDim / 2) + row * (kDim / kNvfp4Group) + col / kNvfp4Group];
  return e2m1_to_float(nib) * e4m3_to_float(sc);
}

__global__ void __launch_bounds__(kSimtThreads)
mla_decode_simt_kernel(DecodeParams p) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  SimtSmem& S = *reinterpret_cast<SimtSmem*>(smem_raw);
  const int tid = threadIdx.x;
  const int worker = blockIdx.x;
  const int h0 = blockIdx.y * kSimtHeads;
  const bool leader = blockIdx.x == 0 && blockIdx.y == 0;

  compute_plan(p, S.plan, S.scratch, leader);

  const int hl = tid / 16;  // local head of this thread (scores, softmax, O rows)
  const int j = tid % 16;   // token pair (scores) / column phase (O)
  const int h = h0 + hl;

  for_each_item(p, S.plan, worker, [&](const WorkItem& it) {
    const int b = it.u / p.q_len, i = it.u % p.q_len;
    // load the 16 absorbed queries as fp32
    for (int k = tid; k < kSimtHeads * kDim; k += kSimtThreads) {
      int hh = k / kDim, c = k % kDim;
      size_t row = ((size_t)b * p.q_len + i) * p.H + h0 + hh;
      uint16_t bits = c < kLatent ? p.q_nope[row * kLatent + c] : p.q_pe[row * kRope + (c - kLatent)];
      S.q[hh][c] = bf16_bits_to_float(bits);
    }
    float m = -INFINITY, l = 0.f;
    float o[kLatent / 16];
#pragma unroll
    for (int k = 0; k < kLatent / 16; ++k) o[k] = 0.f;

    for (int t0 = it.tok_lo; t0 < it.tok_hi; t0 += kSimtChunk) {
      __syncthreads();  // previous chunk fully consumed (and q written)
      if (tid < kSimtChunk) {
        int t = t0 + tid;
        int ok = 0;
        if (t < it.tok_hi) {
          int page = __ldg(p.block_table + (size_t)b * p.max_pages + t / p.page_size);
          if (page >= 0 && page < p.num_pages) ok = 1;
          else set_status(p.ws, MLA_STATUS_PAGE_OUT_OF_RANGE);
        }
        S.valid[tid] = ok;
      }
      __syncthreads();
      for (int k = tid; k < kSimtChunk * kDim; k += kSimtThreads) {
        int r = k / kDim, c = k % kDim;
        float v = 0.f;
        if (S.valid[r]) {
          int t = t0 + r;
          int page = __ldg(p.block_table + (size_t)b * p.max_pages + t / p.page_size);
          v = load_cache_value(p, page, t % p.page_size, c);
        }
        S.kv[r][c] = v;
      }
      __syncthreads();
      // scores for tokens j and j+16 of this chunk
      float s0 = 0.f, s1 = 0.f;
#pragma unroll 8
      for (int c = 0; c < kDim; ++c) {
        float qv = S.q[hl][c];
        s0 = fmaf(qv, S.kv[j][c], s0);
        s1 = fmaf(qv, S.kv[j + 16][c], s1);
      }
      s0 = S.valid[j] ? s0 * p.sm_scale : -INFINITY;
      s1 = S.valid[j + 16] ? s1 * p.sm_scale : -INFINITY;
      float mx = fmaxf(s0, s1);
#pragma unroll
      for (int d = 8; d >= 1; d >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, d));
      float m_new = fmaxf(m, mx);
      float alpha = 1.f, p0 = 0.f, p1 = 0.f;
      if (m_new != -INFINITY) {
        alpha = expf(m - m_new);  // m = -inf -> 0
        p0 = expf(s0 - m_new);
        p1 = expf(s1 - m_new);
      }
      float ps = p0 + p1;
#pragma unroll
      for (int d = 8; d >= 1; d >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, d);
      l = l * alpha + ps;
      m = m_new;
      S.p[hl][j] = p0;
      S.p[hl][j + 16] = p1;
      __syncthreads();
#pragma unroll
      for (int k = 0; k < kLatent / 16; ++k) o[k] *= alpha;
      for (int r = 0; r < kSimtChunk; ++r) {
        float pr = S.p[hl][r];
#pragma unroll
        for (int k = 0; k < kLatent / 16; ++k) o[k] = fmaf(pr, S.kv[r][j + 16 * k], o[k]);
      }
    }
    // epilogue
    const size_t row = ((size_t)b * p.q_len + i) * p.H + h;
    float inv = l > 0.f ? 1.f / l : 0.f;
    float lse_v = l > 0.f ? m + logf(l) : -INFINITY;
    if (it.slot < 0) {
#pragma unroll
      for (int k = 0; k < kLatent / 16; ++k) p.out[row * kLatent + j + 16 * k] = float_to_bf16_bits_rn(o[k] * inv);
      if (p.lse && j == 0) p.lse[row] = lse_v;
    } else if (it.slot < p.slots_cap) {
      float* po = reinterpret_cast<float*>(p.ws + partial_o_offset()) + ((size_t)it.slot * p.H + h) * kLatent;
      float* pls = reinterpret_cast<float*>(p.ws + partial_lse_offset(p.slots_cap, p.H));
#pragma unroll
      for (int k = 0; k < kLatent / 16; ++k) po[j + 16 * k] = o[k] * inv;
      if (j == 0) pls[(size_t)it.slot * p.H + h] = lse_v;
    }
  });
}

size_t simt_smem_bytes() { return sizeof(SimtSmem); }

cudaError_t launch_decode_simt(const DecodeParams& p, cudaStream_t stream) {
  static_assert(sizeof(SimtSmem) < 227 * 1024, "shared memory budget");
  cudaError_t e = cudaFuncSetAttribute(mla_decode_simt_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)sizeof(SimtSmem));
  if (e != cudaSuccess) return e;
  dim3 grid(p.workers, p.H / kSimtHeads);
  mla_decode_simt_kernel<<<grid, kSimtThreads, sizeof(SimtSmem), stream>>>(p);
  return cudaGetLastError();
}

}  // namespace mla

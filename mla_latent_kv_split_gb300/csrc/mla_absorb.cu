// mla_absorb.cu -- the per-head projections on either side of the absorbed decode, one
// launch over all heads (metrale "kv_cache_mla.rs", mla_batched_gemv:
// output[head, n] = sum_k weight[head, n, k] * input[head, k], BF16):
//   Q absorption     q_lat[t, h, :512] = W_UK[h]^T q_nope[t, h, :128]   (weight [512, 128])
//   V up-projection  o[t, h, :128]     = W_UV[h] o_lat[t, h, :512]      (weight [128, 512])
// batched over the step's T tokens: out[t, h, n] = sum_k w[h, n, k] x[t, h, k], fp32
// accumulation, bf16 result.
//
// One CTA per (128 weight rows, head, token tile): the weight rows are the M side of a
// tcgen05 MMA (M = 128) and the tokens its N side (16..256), so a decode step's few tokens
// still fill the tensor core's M dimension and every weight byte is read once per token
// tile.  TMA brings 64-column (128-byte, 128-byte-swizzled) K chunks of both operands into
// a ring of up to eight stages (all of K at decode sizes); one thread issues the MMAs
// into TMEM; the four warps read the accumulator back (lane = weight row) and store bf16.  Bound by HBM for decode-sized T
// (the weights dominate), by the tensor pipe only for thousands of tokens.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "../../include/mla_decode.h"
#include "mla_ptx.cuh"
#include "mla_tmap.cuh"

namespace mla {
namespace gemv {

constexpr int kThreads = 128;
constexpr int kBlockM = 128;     // weight rows per CTA
constexpr int kBlockK = 64;      // bf16 columns per K chunk: one 128-byte swizzle row
constexpr int kMaxStages = 8;
constexpr uint32_t kStageBudget = 200 * 1024;  // shared memory for the stage ring
constexpr uint32_t kMaxSmem = kStageBudget + 8 * 1024;  // ring + control words + alignment, at most
constexpr int kMaxTokens = 256;  // tokens per CTA (MMA N)
constexpr uint32_t kABytes = kBlockM * kBlockK * 2;

struct Ctrl {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  uint64_t done;
  uint32_t tmem;
  int abort;
};

__host__ __device__ constexpr uint32_t stage_bytes(int tt) { return kABytes + (uint32_t)tt * kBlockK * 2; }
__host__ __device__ constexpr uint32_t tmem_cols(int tt) { return tt <= 32 ? 32 : tt <= 64 ? 64 : tt <= 128 ? 128 : 256; }

__global__ void __launch_bounds__(kThreads)
mla_batched_gemv_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_x,
                        uint16_t* __restrict__ out, long long out_token_stride, long long out_head_stride, int T,
                        int N, int K, int tt, int stages, uint32_t* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Ctrl& C = *reinterpret_cast<Ctrl*>(smem + stages * stage_bytes(tt));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * kBlockM, h = blockIdx.y, t0 = blockIdx.z * tt;
  const int nk = (K + kBlockK - 1) / kBlockK;
  const uint32_t ncols = tmem_cols(tt);
  volatile int* abort_flag = &C.abort;

  const uint32_t smem0 = ptx::smem_u32(smem);
  auto issue = [&](int kc) {  // K chunk kc of the weight rows and of the token rows
    const int st = kc % stages;
    const uint32_t a = smem0 + st * stage_bytes(tt), full = ptx::smem_u32(&C.full[st]);
    ptx::mbar_arrive_expect_tx(full, stage_bytes(tt));
    ptx::tma_load_2d(a, &tm_w, kc * kBlockK, h * N + n0, full);
    ptx::tma_load_3d(a + kABytes, &tm_x, kc * kBlockK, h, t0, full);
  };
  const int first = nk < stages ? nk : stages;
  // Programmatic dependent launch: the next kernel on the stream may start its own
  // set-up now; this one reads the activations (and writes its output) only after
  // griddepcontrol.wait, i.e. once the kernel before it has completed.  The weights are
  // not produced by that kernel, so the first ring's weight loads leave before the wait.
  asm volatile("griddepcontrol.launch_dependents;");
  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      ptx::mbar_init(ptx::smem_u32(&C.full[s]), 1);
      ptx::mbar_init(ptx::smem_u32(&C.empty[s]), 1);
    }
    ptx::mbar_init(ptx::smem_u32(&C.done), 1);
    C.abort = 0;
    ptx::fence_mbar_init_cluster();
    // the first ring's worth of loads leaves before the TMEM allocation and the block
    // barrier: its weight chunks at once, its token chunks once the previous kernel is done
    for (int kc = 0; kc < first; ++kc) {
      const uint32_t a = smem0 + (kc % stages) * stage_bytes(tt), full = ptx::smem_u32(&C.full[kc % stages]);
      ptx::mbar_arrive_expect_tx(full, stage_bytes(tt));
      ptx::tma_load_2d(a, &tm_w, kc * kBlockK, h * N + n0, full);
    }
  }
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (threadIdx.x == 0)
    for (int kc = 0; kc < first; ++kc)
      ptx::tma_load_3d(smem0 + (kc % stages) * stage_bytes(tt) + kABytes, &tm_x, kc * kBlockK, h, t0,
                       ptx::smem_u32(&C.full[kc % stages]));
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_u32(&C.tmem), ncols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = C.tmem;

  if (warp == 0 && lane == 0) {
    // ---- producer: the remaining K chunks, each into a stage its MMAs have released
    int kc = first;
    for (; kc < nk; ++kc) {
      const int st = kc % stages;
      if (!ptx::mbar_wait(ptx::smem_u32(&C.empty[st]), ((kc / stages) - 1) & 1, abort_flag)) break;
      issue(kc);
    }
    // loads still in flight after an abort land before the CTA exits
    for (int k = max(0, kc - stages); k < kc; ++k)
      ptx::mbar_drain(ptx::smem_u32(&C.full[k % stages]), (k / stages) & 1);
  } else if (warp == 1 && lane == 0) {
    // ---- MMA issuer: D[128 rows x tt tokens] += W[128 x 64] . X[tt x 64]^T per chunk
    const uint32_t idesc = ptx::idesc_f16(1, 0, kBlockM, (uint32_t)tt);
    bool ok = true;
    for (int kc = 0; kc < nk; ++kc) {
      const int st = kc % stages;
      if (!ptx::mbar_wait(ptx::smem_u32(&C.full[st]), (kc / stages) & 1, abort_flag)) {
        ok = false;
        break;
      }
      ptx::tc_fence_after();
      const uint32_t a = smem0 + st * stage_bytes(tt);
      const uint64_t adesc = ptx::umma_desc(a, 16, 1024, 2), bdesc = ptx::umma_desc(a + kABytes, 16, 1024, 2);
#pragma unroll
      for (int j = 0; j < kBlockK / 16; ++j)  // 16 columns (32 bytes) per MMA
        ptx::mma_ss(tmem, adesc + 2 * j, bdesc + 2 * j, idesc, (kc | j) ? 1u : 0u);
      ptx::mma_commit(ptx::smem_u32(&C.empty[st]));
    }
    if (ok) ptx::mma_commit(ptx::smem_u32(&C.done));
  }
  __syncwarp();
  // ---- epilogue: lane = weight row n, 16 tokens per TMEM load
  // (the warp's lanes take the same branch below: the TMEM loads are warp-collective)
  const bool done = __all_sync(0xffffffffu, ptx::mbar_wait(ptx::smem_u32(&C.done), 0, abort_flag));
  ptx::tc_fence_after();
  if (done) {
    const int n = n0 + 32 * warp + lane;
    uint16_t* o = out + (size_t)h * out_head_stride + n;
    const uint32_t taddr = tmem + ((uint32_t)(32 * warp) << 16);
    for (int c0 = 0; c0 < tt; c0 += 16) {
      uint32_t r[16];
      ptx::tmem_ld16(taddr + c0, r);
      ptx::tmem_ld_wait();
      if (n < N) {
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int t = t0 + c0 + j;
          if (t < T) o[(size_t)t * out_token_stride] = __bfloat16_as_ushort(__float2bfloat16_rn(__uint_as_float(r[j])));
        }
      }
    }
  } else if (threadIdx.x == 0 && status != nullptr) {
    atomicOr(status, MLA_STATUS_WAIT_TIMEOUT);
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) ptx::tmem_dealloc(tmem, ncols);
}

}  // namespace gemv

// Token tile: at most 256 tokens per CTA, tiles balanced, rounded up to 16 (MMA N).
int gemv_token_tile(int T) {
  const int tiles = (T + gemv::kMaxTokens - 1) / gemv::kMaxTokens;
  const int per = (T + tiles - 1) / tiles;
  return (per + 15) / 16 * 16;
}

cudaError_t launch_batched_gemv(const uint16_t* x, long long x_token_stride, long long x_head_stride,
                                const uint16_t* w, uint16_t* out, long long out_token_stride,
                                long long out_head_stride, int T, int H, int N, int K, uint32_t* status,
                                cudaStream_t stream) {
  EncodeTiledFn fn = tmap_encode_fn();
  if (!fn) return cudaErrorNotSupported;
  const int tt = gemv_token_tile(T);
  const int nk = (K + gemv::kBlockK - 1) / gemv::kBlockK;
  // as many K chunks in flight as fit: the whole K extent for the MLA shapes at decode sizes
  int stages = (int)(gemv::kStageBudget / gemv::stage_bytes(tt));
  if (stages > gemv::kMaxStages) stages = gemv::kMaxStages;
  if (stages > nk) stages = nk;
  CUtensorMap tm_w, tm_x;
  {
    cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)H * N};
    cuuint64_t strides[1] = {(cuuint64_t)K * 2};
    cuuint32_t box[2] = {gemv::kBlockK, gemv::kBlockM};
    cuuint32_t estr[2] = {1, 1};
    if (fn(&tm_w, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(w), dims, strides, box, estr,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  {
    cuuint64_t dims[3] = {(cuuint64_t)K, (cuuint64_t)H, (cuuint64_t)T};
    cuuint64_t strides[2] = {(cuuint64_t)x_head_stride * 2, (cuuint64_t)x_token_stride * 2};
    cuuint32_t box[3] = {gemv::kBlockK, 1, (cuuint32_t)tt};
    cuuint32_t estr[3] = {1, 1, 1};
    if (fn(&tm_x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<uint16_t*>(x), dims, strides, box, estr,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  // Shared memory: the stage ring, control words, 1 KB alignment slack; at least enough that
  // the CTAs resident on one SM never ask for more than its 512 TMEM columns.
  const uint32_t cols = gemv::tmem_cols(tt);
  size_t smem = (size_t)stages * gemv::stage_bytes(tt) + sizeof(gemv::Ctrl) + 1024;
  const size_t sm_smem = 233472;  // per-SM shared memory (228 KB)
  const size_t floor_smem = sm_smem / (512 / cols + 1) + 1;
  if (smem < floor_smem) smem = floor_smem;
  if (smem > gemv::kMaxSmem) return cudaErrorInvalidValue;  // cannot happen: the ring fits kStageBudget
  auto kern = gemv::mla_batched_gemv_kernel;
  // the opt-in (the largest ring this launcher ever asks for) outlives the call: set once
  // per device
  static std::mutex mu;
  static bool opted_in[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  {
    std::lock_guard<std::mutex> lk(mu);
    if (!opted_in[dev]) {
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)gemv::kMaxSmem);
      if (e != cudaSuccess) return e;
      opted_in[dev] = true;
    }
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((N + gemv::kBlockM - 1) / gemv::kBlockM, H, (T + tt - 1) / tt);
  cfg.blockDim = dim3(gemv::kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // see griddepcontrol in the kernel
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, tm_w, tm_x, out, (long long)out_token_stride, (long long)out_head_stride, T, N,
                            K, tt, stages, status);
}

}  // namespace mla

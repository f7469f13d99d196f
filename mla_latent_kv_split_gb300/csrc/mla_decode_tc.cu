// mla_decode_tc.cu -- split-KV MLA decode on the 5th-generation tensor cores (sm_103a).
//
// Work split (one scheduling worker = a cluster of two CTAs on two SMs):
//   The output accumulator of 128 heads x 512 latent fp32 columns alone fills a whole
//   SM's tensor memory (128 lanes x 512 columns), so the two CTAs of a cluster split the
//   latent dimension: CTA r owns output columns [256r, 256r+256).  Each CTA loads only the
//   cache columns it needs: its 256 latent columns (which are both its half of K and its
//   half of V) plus 32 of the 64 rope columns.  The score contraction over 576 columns is
//   therefore split in two: each CTA computes the partial scores of its 288 columns with
//   one MMA chain, and the two CTAs exchange the partial fp32 score tiles through
//   distributed shared memory, so both hold the same full scores, take the same softmax
//   decisions and produce the same P.  Every cache byte is read from HBM once.
//
// Per CTA, per 64-token tile (TileGym: K = V = KV; tokenspeed: paged cache):
//   producer warp   TMA-gathers the tile's pages (block table -> page rows) into a
//                   4-stage ring: 4 boxes of 64 tokens x 64 latent columns (128-byte
//                   swizzle) + 1 box of 64 tokens x 32 rope columns (64-byte swizzle)
//                   (FP8: the E4M3 bytes of those columns; NVFP4: whole pages, packed
//                   E2M1 data plus E4M3 scales, into the tail of the stage)
//   MMA warp        S[128 x 64] = Q[128 x 288] (in TMEM) . K^T       (18 MMAs, K = 16)
//                   O[128 x 256] += P[128 x 64] (in TMEM) . V[64 x 256] (4 MMAs, N = 256)
//   sender warps    one warpgroup.  (1) Prepares each landed tile for the MMAs: zeroes the
//                   rows that are masked (ragged tail, invalid page) so that garbage, even
//                   NaN, cannot reach P.V, and for FP8 / NVFP4 decodes the raw bytes in place
//                   into f16 (exact for both formats) in the same swizzled layout.
//                   (2) Thread = head row: loads the row's 64 partial scores
//                   from TMEM and pushes them into the peer CTA's exchange buffer with
//                   asynchronous stores that complete on the peer's mbarrier (the link is
//                   the slowest path of the exchange, so it gets warps of its own)
//   softmax warps   two warpgroups; thread (row = head, half h) owns tile columns
//                   [32h, 32h+32) of its row: loads them from TMEM, waits for the peer's
//                   partial scores, adds them, combines the row max with the other
//                   half, runs the online softmax in base 2 with a lazy rescale of O (only
//                   when the running max grows by more than 8) and writes P (bf16) to
//                   TMEM; at the end of a work item it normalises its 128 output columns
//                   and writes the output (or the split partial and its LSE).
//
// Tensor memory (512 columns): O [0,256) fp32; two score buffers S0 [256,320), S1 [320,384)
// fp32; Q [384,512) bf16 pairs (this CTA's 256 latent columns).  The 32 rope columns of Q
// and P (bf16) sit in shared memory, where the rope and P.V MMAs read their A operand, so a
// score buffer is free again as soon as it has been read.
#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#include "mla_device.cuh"
#include "mla_ptx.cuh"

namespace mla {
namespace tc {

constexpr int kThreads = 512;
constexpr int kStages = 4;
constexpr int kTileN = 64;                      // tokens per tile
constexpr int kLatBox = kTileN * 128;           // 64 rows x 64 bf16 (8 KB)
constexpr int kRopeBox = kTileN * 64;           // 64 rows x 32 bf16 (4 KB)
constexpr int kStageBytes = 4 * kLatBox + kRopeBox;  // 36 KB
// Partial scores cross the cluster as 24-bit floats (fp32 rounded to 15 mantissa bits,
// relative error <= 2^-16): 4 values in 3 words; one tile = 128 rows x 48 words (24 KB).
constexpr int kXWordsPerRow = kTileN * 3 / 4;   // 48
constexpr int kXBytes = 128 * kXWordsPerRow * 4;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 0, kTmemS = 256, kTmemQ = 384;  // S buffers at kTmemS + 64 * (g & 1)
constexpr int kQRopeBytes = 128 * 64;  // Q rope: 128 rows x 32 bf16, K-major, 64-byte swizzle
constexpr int kPBytes = 128 * 128;     // P: 128 rows x 64 tokens 16-bit, K-major, 128-byte swizzle
// Raw bytes of quantized tiles sit in the tail of a stage and are decoded in place:
constexpr int kRawFp8 = kStageBytes - kTileN * 288;    // FP8: 256 latent + 32 rope bytes per row
constexpr int kRawFp8Rope = kRawFp8 + kTileN * 256;
constexpr int kRawFp4 = kStageBytes - kTileN * 324;    // NVFP4: whole pages (288 data + 36 scale B per token)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;       // log2 units: P stays below 2^8

// warp roles
constexpr int kWarpProducer = 0, kWarpMma = 1, kWarpRelay = 3, kWarpSender0 = 4, kWarpSoftmax0 = 8;
constexpr int kSenderThreads = 128;   // warps 4..7
constexpr int kSoftmaxThreads = 256;  // warps 8..15
// Registers per thread: the launch gives every thread kLaunchRegs; the control warpgroup
// (warps 0..3) drops to kCtrlRegs, the sender warpgroup to kSenderRegs, and the two softmax
// warpgroups rise to kSoftmaxRegs.  The sum must not exceed 512 * kLaunchRegs (65,536).
constexpr uint32_t kLaunchRegs = 128, kCtrlRegs = 64, kSenderRegs = 128, kSoftmaxRegs = 160;
static_assert(128 * kCtrlRegs + 128 * kSenderRegs + 256 * kSoftmaxRegs <= 512 * kLaunchRegs,
              "register split exceeds the launch budget");

struct Bars {
  uint64_t kv_full[kStages];   // TMA bytes landed
  uint64_t kv_ready[kStages];  // senders prepared the tile (masked rows zeroed, quantized data decoded)
  uint64_t deq;                // senders read every raw byte of a tile (before decoding in place)
  uint64_t kv_empty[kStages];  // P.V of the tile completed: stage reusable
  uint64_t s_full[2];          // S MMAs of a buffer completed
  uint64_t s_free[2];          // senders and softmax read a buffer's S
  uint64_t p_full;             // P written to shared memory (and O rescaled)
  uint64_t o_done;             // P.V completed
  uint64_t q_ready;            // Q of the next item in TMEM
  uint64_t o_free;             // epilogue read O
  uint64_t x_full[2];          // the peer's partial scores landed in my exchange buffer (tx count)
  uint64_t x_empty[2];         // peer finished reading its buffer: I may write it again
  uint64_t x_read[2];          // my softmax warps finished reading my buffer (relayed to the peer)
  uint64_t mx[2];              // both halves of every row published their tile max
  uint64_t lsum;               // both halves published their row sums (epilogue)
  uint64_t mma_final;          // every MMA of this CTA completed
};

struct Smem {
  uint8_t stage[kStages][kStageBytes];
  uint8_t p_tile[kPBytes];  // 1024-byte aligned (swizzle atoms)
  uint8_t q_rope[kQRopeBytes];
  uint4 xbuf[2][kXWordsPerRow / 4][128];  // [slot][16-byte group][row], 24-bit packed
  Bars bars;
  float mx[2][2][128];   // [tile parity][half][row] partial row maxima
  float lsum[2][128];    // [half][row] partial row sums
  uint32_t tmem_base;
  int abort_flag;
  int scratch[33];
  WorkerStart wstart;  // this worker's place in the schedule (the full plan is built in xbuf)
};
static_assert(sizeof(PlanSmem) <= 2 * kXBytes, "plan scratch must fit the exchange buffers");

__device__ __forceinline__ Smem& smem_ref(uint8_t* raw) {
  uintptr_t a = reinterpret_cast<uintptr_t>(raw);
  a = (a + 1023) & ~uintptr_t(1023);
  return *reinterpret_cast<Smem*>(a);
}

// Geometry of one 64-token tile of a work item.
struct TileInfo {
  int page[2];       // physical pages (ps=64: page[0] only)
  int npages;        // pages that hold any visible position
  bool page_ok[2];
  uint64_t rowmask;  // bit r: row r is a real, visible position
};

__device__ __forceinline__ TileInfo tile_info(const DecodeParams& p, int b, int t0, int tok_hi) {
  TileInfo ti;
  const int ps = p.page_size;
  const int per = kTileN / ps;  // 1 or 2 pages per tile
  ti.npages = 0;
  ti.rowmask = 0;
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    ti.page[j] = -1;
    ti.page_ok[j] = false;
    if (j < per && t0 + j * ps < tok_hi) {
      const int lp = (t0 + j * ps) / ps;
      const int pg = __ldg(p.block_table + (size_t)b * p.max_pages + lp);
      ti.page[j] = pg;
      ti.page_ok[j] = pg >= 0 && pg < p.num_pages;
      ti.npages = j + 1;
      const int rows = min(ps, tok_hi - (t0 + j * ps));
      if (ti.page_ok[j]) {
        const uint64_t m = rows >= 64 ? ~0ull : ((1ull << rows) - 1);
        ti.rowmask |= m << (j * ps);
      }
    }
  }
  return ti;
}
__device__ __forceinline__ bool tile_needs_fixup(const TileInfo& ti) { return ti.rowmask != ~0ull; }

// Two bf16 values -> two f16 (exact for |x| in [2^-14, 65504]; smaller magnitudes round to
// f16 subnormals, larger ones overflow and are reported).
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t v, bool& out_of_range) {
  const float lo = __uint_as_float(v << 16), hi = __uint_as_float(v & 0xFFFF0000u);
  out_of_range |= fabsf(lo) > 65504.f || fabsf(hi) > 65504.f;
  return ptx::pack_f16x2(lo, hi);
}

// fp32 bit pattern rounded to its top 24 bits (sign, exponent, 15 mantissa bits), nearest.
__device__ __forceinline__ uint32_t round24(uint32_t bits) { return (bits + 0x80u) & 0xFFFFFF00u; }
// Four fp32 values -> three words holding their rounded top 24 bits.
__device__ __forceinline__ void pack24x4(uint32_t a, uint32_t b, uint32_t c, uint32_t d, uint32_t& w0, uint32_t& w1,
                                         uint32_t& w2) {
  a = round24(a) >> 8;
  b = round24(b) >> 8;
  c = round24(c) >> 8;
  d = round24(d) >> 8;
  w0 = a | (b << 24);
  w1 = (b >> 8) | (c << 16);
  w2 = (c >> 16) | (d << 8);
}
__device__ __forceinline__ void unpack24x4(uint32_t w0, uint32_t w1, uint32_t w2, float& a, float& b, float& c,
                                           float& d) {
  a = __uint_as_float(w0 << 8);
  b = __uint_as_float(((w0 >> 24) | (w1 << 8)) << 8);
  c = __uint_as_float(((w1 >> 16) | (w2 << 16)) << 8);
  d = __uint_as_float(w2 & 0xFFFFFF00u);
}

// The raw block-table entries of a tile (loaded early, consumed a softmax iteration later).
struct TilePages {
  int pg[2];
};
__device__ __forceinline__ TilePages tile_pages(const DecodeParams& p, int b, int t0, int tok_hi) {
  TilePages tp;
  const int ps = p.page_size;
#pragma unroll
  for (int j = 0; j < 2; ++j)
    tp.pg[j] = (j < kTileN / ps && t0 + j * ps < tok_hi) ? __ldg(p.block_table + (size_t)b * p.max_pages + (t0 + j * ps) / ps)
                                                          : -1;
  return tp;
}
// Rows [32h, 32h+32) of the tile that are real, visible positions.
__device__ __forceinline__ uint32_t tile_half_mask(const DecodeParams& p, const TilePages& tp, int t0, int tok_hi,
                                                   int h) {
  const int ps = p.page_size;
  uint64_t m = 0;
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    if (j < kTileN / ps && t0 + j * ps < tok_hi && tp.pg[j] >= 0 && tp.pg[j] < p.num_pages) {
      const int rows = min(ps, tok_hi - (t0 + j * ps));
      m |= (rows >= 64 ? ~0ull : ((1ull << rows) - 1)) << (j * ps);
    }
  }
  return (uint32_t)(m >> (32 * h));
}

// KV: cache format (MLA_KV_BF16 / MLA_KV_FP8_E4M3 / MLA_KV_NVFP4).  The MMAs run in bf16 for a
// bf16 cache and in f16 for the quantized ones (E4M3 and E2M1 x E4M3 are exact in f16).
template <int KV>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
mla_decode_tc_kernel(const __grid_constant__ CUtensorMap tm_lat, const __grid_constant__ CUtensorMap tm_rope,
                     const DecodeParams p) {
  extern __shared__ uint8_t smem_raw[];
  Smem& S = smem_ref(smem_raw);
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const uint32_t cr = ptx::cluster_ctarank();  // 0: latent [0,256) + rope [0,32); 1: the other halves
  const uint32_t peer = cr ^ 1u;
  const int worker = blockIdx.x >> 1;
  volatile int* abort_flag = &S.abort_flag;

  asm volatile("griddepcontrol.launch_dependents;");
  {
    // the schedule is evaluated in the exchange buffers, which are idle until the first tile
    PlanSmem& plan = *reinterpret_cast<PlanSmem*>(&S.xbuf[0][0][0]);
    compute_plan(p, plan, S.scratch, blockIdx.x == 0);
    if (tid == 0) S.wstart = worker_start(p, plan, worker);
    __syncthreads();
  }
  const WorkerStart wst = S.wstart;

  const uint32_t b_kv_full = ptx::smem_u32(&S.bars.kv_full[0]);
  const uint32_t b_kv_ready = ptx::smem_u32(&S.bars.kv_ready[0]);
  const uint32_t b_kv_empty = ptx::smem_u32(&S.bars.kv_empty[0]);
  const uint32_t b_s_full = ptx::smem_u32(&S.bars.s_full[0]), b_s_free = ptx::smem_u32(&S.bars.s_free[0]);
  const uint32_t b_p_full = ptx::smem_u32(&S.bars.p_full), b_o_done = ptx::smem_u32(&S.bars.o_done);
  const uint32_t b_q_ready = ptx::smem_u32(&S.bars.q_ready), b_o_free = ptx::smem_u32(&S.bars.o_free);
  const uint32_t b_x_full = ptx::smem_u32(&S.bars.x_full[0]), b_x_empty = ptx::smem_u32(&S.bars.x_empty[0]);
  const uint32_t b_mma_final = ptx::smem_u32(&S.bars.mma_final);
  const uint32_t b_mx = ptx::smem_u32(&S.bars.mx[0]), b_lsum = ptx::smem_u32(&S.bars.lsum);
  const uint32_t b_x_read = ptx::smem_u32(&S.bars.x_read[0]);
  const uint32_t b_deq = ptx::smem_u32(&S.bars.deq);

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(b_kv_full + 8 * s, 1);
      ptx::mbar_init(b_kv_ready + 8 * s, kSenderThreads);
      ptx::mbar_init(b_kv_empty + 8 * s, 1);
    }
    for (int s = 0; s < 2; ++s) {
      ptx::mbar_init(b_s_full + 8 * s, 1);
      ptx::mbar_init(b_s_free + 8 * s, kSoftmaxThreads + kSenderThreads);
    }
    ptx::mbar_init(b_p_full, kSoftmaxThreads);
    ptx::mbar_init(b_o_done, 1);
    ptx::mbar_init(b_q_ready, kSoftmaxThreads);
    ptx::mbar_init(b_o_free, kSoftmaxThreads);
    for (int s = 0; s < 2; ++s) {
      ptx::mbar_init(b_x_full + 8 * s, 1);   // one local arrive (expect_tx) + 32 KB of peer bytes
      ptx::mbar_init(b_x_empty + 8 * s, 1);  // one arrive per use, from the peer's relay warp
      ptx::mbar_init(b_mx + 8 * s, kSoftmaxThreads);
      ptx::mbar_init(b_x_read + 8 * s, kSoftmaxThreads / 32);
    }
    ptx::mbar_init(b_lsum, kSoftmaxThreads);
    ptx::mbar_init(b_deq, kSenderThreads);
    ptx::mbar_init(b_mma_final, 1);
    S.abort_flag = 0;
    ptx::fence_mbar_init_cluster();
  }
  if (warp == kWarpMma) {
    ptx::tmem_alloc(ptx::smem_u32(&S.tmem_base), kTmemCols);
    ptx::tmem_relinquish();
  }
  if (KV != MLA_KV_NVFP4 && warp == kWarpProducer && lane == 0) {
    ptx::prefetch_tmap(&tm_lat);
    ptx::prefetch_tmap(&tm_rope);
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::cluster_sync_all();  // the peer's barriers exist before any remote arrive
  ptx::tc_fence_after();
  const uint32_t tmem = S.tmem_base;
  if (warp == kWarpProducer) {
    ptx::regs_dec<kCtrlRegs>();
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int g = 0;
      for_each_item_cursor(p, wst, worker, [&](const WorkItem& it) {
        const int b = it.u / p.q_len;
        // Let the first item's queries reach the memory system before this CTA's burst of
        // cache loads (otherwise they queue behind every SM's initial TMA traffic).
        if (g == 0 && !ptx::mbar_wait(b_q_ready, 0, abort_flag)) return;
        for (int t0 = it.tok_lo; t0 < it.tok_hi; t0 += kTileN, ++g) {
          if (*abort_flag) return;
          const int st = g % kStages;
          if (g >= kStages && !ptx::mbar_wait(b_kv_empty + 8 * st, ((g / kStages) - 1) & 1, abort_flag)) return;
          const TileInfo ti = tile_info(p, b, t0, it.tok_hi);
          const uint32_t page_bytes = KV == MLA_KV_BF16 ? (uint32_t)p.page_size * (4 * 128 + 64)
                                    : KV == MLA_KV_FP8_E4M3 ? (uint32_t)p.page_size * 288
                                                            : (uint32_t)p.page_size * 324;
          uint32_t bytes = 0;
          for (int j = 0; j < ti.npages; ++j) {
            if (ti.page_ok[j]) bytes += page_bytes;
            else set_status(p.ws, MLA_STATUS_PAGE_OUT_OF_RANGE);
          }
          ptx::mbar_arrive_expect_tx(b_kv_full + 8 * st, bytes);
          const uint32_t dst = ptx::smem_u32(S.stage[st]);
          for (int j = 0; j < ti.npages; ++j) {
            if (!ti.page_ok[j]) continue;
            const int y = ti.page[j] * p.page_size;
            const int roff = j * p.page_size;
            if (KV == MLA_KV_BF16) {
#pragma unroll
              for (int k = 0; k < 4; ++k)
                ptx::tma_load_2d(dst + k * kLatBox + roff * 128, &tm_lat, 256 * (int)cr + 64 * k, y,
                                 b_kv_full + 8 * st);
              ptx::tma_load_2d(dst + 4 * kLatBox + roff * 64, &tm_rope, 512 + 32 * (int)cr, y, b_kv_full + 8 * st);
            } else if (KV == MLA_KV_FP8_E4M3) {
              ptx::tma_load_2d(dst + kRawFp8 + roff * 256, &tm_lat, 256 * (int)cr, y, b_kv_full + 8 * st);
              ptx::tma_load_2d(dst + kRawFp8Rope + roff * 32, &tm_rope, 512 + 32 * (int)cr, y, b_kv_full + 8 * st);
            } else {
              ptx::bulk_load(dst + kRawFp4 + j * page_bytes, p.cache + (size_t)ti.page[j] * page_bytes, page_bytes,
                             b_kv_full + 8 * st);
            }
          }
        }
      });
      // loads still in flight after an abort must land before the CTA exits
      for (int k = 1; k <= kStages && g - k >= 0; ++k) {
        const int gg = g - k;
        ptx::mbar_wait(b_kv_full + 8 * (gg % kStages), (gg / kStages) & 1, abort_flag, false, 100000000ull);
      }
    }
  } else if (warp == kWarpMma) {
    // ------------------------------------------------------------------ MMA issuer
    ptx::regs_dec<kCtrlRegs>();
    // Per item, an event loop: the score MMAs of the next tile are issued as soon as its
    // cache tile has landed and the softmax has read the previous scores, independently
    // of the P.V of earlier tiles, which are issued whenever their P is ready.
    if (lane == 0) {
      constexpr uint32_t ab = KV == MLA_KV_BF16 ? 1u : 0u;                 // bf16 / f16 operands
      constexpr uint32_t idesc_s = ptx::idesc_f16(ab, 0, 128, kTileN);  // K-major B (cache rows)
      constexpr uint32_t idesc_o = ptx::idesc_f16(ab, 1, 128, 256);     // MN-major B (V columns)
      const uint32_t stage0 = ptx::smem_u32(S.stage[0]);
      // base descriptors of stage 0; stage st adds st * kStageBytes to the address field
      const uint64_t kdesc0 = ptx::umma_desc(stage0, 16, 1024, 2);               // K rows, 128 B swizzle
      const uint64_t rdesc0 = ptx::umma_desc(stage0 + 4 * kLatBox, 16, 512, 4);  // rope rows, 64 B swizzle
      const uint64_t vdesc0 = ptx::umma_desc(stage0, kLatBox, 1024, 2);          // V, MN-major
      const uint64_t qdesc0 = ptx::umma_desc(ptx::smem_u32(S.q_rope), 16, 512, 4);
      const uint64_t pdesc0 = ptx::umma_desc(ptx::smem_u32(S.p_tile), 16, 1024, 2);  // P, K-major
      int g = 0, n_item = 0;
      bool dead = false;
      for_each_item_cursor(p, wst, worker, [&](const WorkItem& it) {
        if (dead) return;
        if (!ptx::mbar_wait(b_q_ready, n_item & 1, abort_flag)) { dead = true; return; }
        ptx::tc_fence_after();
        const int nt = (it.tok_hi - it.tok_lo + kTileN - 1) / kTileN;
        const int g0 = g;
        int ts = 0, tp = 0;  // next tile whose S / P.V is to be issued
        bool o_free_ok = n_item == 0;
        uint64_t t_idle = 0;
        while (tp < nt) {
          bool progressed = false;
          // P.V first: its completion is what frees a cache stage for the next load
          if (tp < ts) {
            const int gp = g0 + tp;
            if (!o_free_ok) o_free_ok = ptx::mbar_test(b_o_free, (n_item - 1) & 1);
            if (o_free_ok && ptx::mbar_test(b_p_full, gp & 1)) {
              ptx::tc_fence_after();
              const uint64_t vdesc = vdesc0 + (uint64_t)((gp % kStages) * (kStageBytes >> 4));
#pragma unroll
              for (int k = 0; k < kTileN / 16; ++k)  // 16 tokens = 2 KB of V rows, 32 B of P rows
                ptx::mma_ss(tmem + kTmemO, pdesc0 + (uint64_t)(k * 2), vdesc + (uint64_t)(k * (2048 >> 4)), idesc_o,
                            (tp == 0 && k == 0) ? 0u : 1u);
              ptx::mma_commit(b_o_done);
              ptx::mma_commit(b_kv_empty + 8 * (gp % kStages));
              ++tp;
              progressed = true;
            }
          }
          if (ts < nt) {
            const int gs = g0 + ts, st = gs % kStages;
            // buffer gs&1 is free once the senders and the softmax have read S(gs-2)
            if (ptx::mbar_test(b_kv_ready + 8 * st, (gs / kStages) & 1) &&
                       (gs < 2 || ptx::mbar_test(b_s_free + 8 * (gs & 1), ((gs >> 1) - 1) & 1))) {
              const uint32_t d_s = tmem + kTmemS + 64 * (gs & 1);
              ptx::tc_fence_after();
              // Descriptors advance by constant offsets (16-byte units): 32 B per K step in a
              // 128-byte swizzle row, one 8 KB box per 64 latent columns.
              const uint64_t kdesc = kdesc0 + (uint64_t)(st * (kStageBytes >> 4));
              const uint64_t rdesc = rdesc0 + (uint64_t)(st * (kStageBytes >> 4));
#pragma unroll
              for (int k = 0; k < 16; ++k)  // 256 latent columns: 4 boxes x 4 steps of 16
                ptx::mma_ts(d_s, tmem + kTmemQ + 8 * k, kdesc + (uint64_t)((k >> 2) * (kLatBox >> 4) + (k & 3) * 2),
                            idesc_s, k > 0 ? 1u : 0u);
#pragma unroll
              for (int k = 0; k < 2; ++k)  // 32 rope columns (64-byte swizzle), Q rope from smem
                ptx::mma_ss(d_s, qdesc0 + (uint64_t)(k * 2), rdesc + (uint64_t)(k * 2), idesc_s, 1u);
              ptx::mma_commit(b_s_full + 8 * (gs & 1));
              ++ts;
              progressed = true;
            }
          }
          if (progressed) {
            t_idle = 0;
          } else {
            const uint64_t now = ptx::globaltimer_ns();
            if (t_idle == 0) {
              t_idle = now;
            } else if (*abort_flag || now - t_idle > 4000000000ull) {
              *abort_flag = 1;
              dead = true;
              return;
            }
          }
        }
        g += nt;
        ++n_item;
      });
      ptx::mma_commit(b_mma_final);
      ptx::mbar_wait(b_mma_final, 0, abort_flag, false, 100000000ull);
    }
  } else if (warp >= kWarpSender0 && warp < kWarpSoftmax0) {
    // ------------------------------------------------------------------ score sender
    ptx::regs_dec<kSenderRegs>();
    const int q = warp & 3;
    const int row = 32 * q + lane;
    const uint32_t t_s0 = tmem + ((uint32_t)(32 * q) << 16) + kTmemS;
    const uint32_t x_peer = ptx::mapa(ptx::smem_u32(&S.xbuf[0][0][0]), peer);
    const uint32_t bx_full_peer = ptx::mapa(b_x_full, peer);
    const int tq = (warp - kWarpSender0) * 32 + lane;  // 0..127
    const int pr = tq >> 1, phf = tq & 1;              // prepare: row and half-row (18 chunks of 8)

    // (1) Tile k has landed: zero masked rows; decode FP8 / NVFP4 bytes in place to f16.
    auto prepare = [&](int k, const TileInfo& ti) -> bool {
      const int st = k % kStages;
      if (!ptx::mbar_wait(b_kv_full + 8 * st, (k / kStages) & 1, abort_flag)) return false;
      uint8_t* base = S.stage[st];
      const bool valid = (ti.rowmask >> pr) & 1ull;
      // destination of 16-byte chunk c (8 values) of row pr in the swizzled operand layout
      auto chunk_ptr = [&](int c) -> uint4* {
        return reinterpret_cast<uint4*>(c < 32 ? base + (c >> 3) * kLatBox + pr * 128 + (((c & 7) ^ (pr & 7)) * 16)
                                              : base + 4 * kLatBox + pr * 64 + ((((c - 32) ^ ((pr >> 1) & 3))) * 16));
      };
      if (KV == MLA_KV_BF16) {
        if (!valid) {
#pragma unroll 1
          for (int c = 18 * phf; c < 18 * phf + 18; ++c) *chunk_ptr(c) = make_uint4(0u, 0u, 0u, 0u);
        }
      } else {
        // every raw byte this thread needs -> registers, then (after all senders did the
        // same) the decoded values over the same stage
        uint32_t raw[18][2];
        if (valid) {
#pragma unroll
          for (int i = 0; i < 18; ++i) {
            const int c = 18 * phf + i;
            if (KV == MLA_KV_FP8_E4M3) {
              const uint2 v = *reinterpret_cast<const uint2*>(c < 32 ? base + kRawFp8 + pr * 256 + 8 * c
                                                                     : base + kRawFp8Rope + pr * 32 + 8 * (c - 32));
              raw[i][0] = v.x;
              raw[i][1] = v.y;
            } else {
              const int ps = p.page_size;
              const int j = pr / ps, rin = pr - j * ps;
              const uint8_t* page = base + kRawFp4 + j * ps * 324;
              const int col0 = c < 32 ? 256 * (int)cr + 8 * c : 512 + 32 * (int)cr + 8 * (c - 32);
              raw[i][0] = *reinterpret_cast<const uint32_t*>(page + rin * 288 + col0 / 2);
              raw[i][1] = page[ps * 288 + rin * 36 + col0 / 16];
            }
          }
        }
        ptx::mbar_arrive(b_deq);
        if (!ptx::mbar_wait(b_deq, k & 1, abort_flag)) return false;
#pragma unroll
        for (int i = 0; i < 18; ++i) {
          uint4 o = make_uint4(0u, 0u, 0u, 0u);
          if (valid) {
            if (KV == MLA_KV_FP8_E4M3) {
              o.x = ptx::e4m3x2_to_f16x2((uint16_t)(raw[i][0] & 0xFFFFu));
              o.y = ptx::e4m3x2_to_f16x2((uint16_t)(raw[i][0] >> 16));
              o.z = ptx::e4m3x2_to_f16x2((uint16_t)(raw[i][1] & 0xFFFFu));
              o.w = ptx::e4m3x2_to_f16x2((uint16_t)(raw[i][1] >> 16));
            } else {
              const uint32_t sc = ptx::e4m3x2_to_f16x2((uint16_t)(raw[i][1] | (raw[i][1] << 8)));
              o.x = ptx::hmul2(ptx::e2m1x2_to_f16x2(raw[i][0] & 0xFFu), sc);
              o.y = ptx::hmul2(ptx::e2m1x2_to_f16x2((raw[i][0] >> 8) & 0xFFu), sc);
              o.z = ptx::hmul2(ptx::e2m1x2_to_f16x2((raw[i][0] >> 16) & 0xFFu), sc);
              o.w = ptx::hmul2(ptx::e2m1x2_to_f16x2(raw[i][0] >> 24), sc);
            }
          }
          *chunk_ptr(18 * phf + i) = o;
        }
      }
      ptx::fence_proxy_async_smem();
      ptx::mbar_arrive(b_kv_ready + 8 * st);
      return true;
    };

    // (2) Tile k's partial scores -> the peer CTA.
    auto send = [&](int k) -> bool {
      if (!ptx::mbar_wait(b_s_full + 8 * (k & 1), (k >> 1) & 1, abort_flag)) return false;
      ptx::tc_fence_after();
      uint32_t r0[32], r1[32];
      const uint32_t t_s = t_s0 + 64 * (k & 1);
      ptx::tmem_ld32(t_s, r0);
      ptx::tmem_ld32(t_s + 32, r1);
      ptx::tmem_ld_wait();
      ptx::tc_fence_before();
      ptx::mbar_arrive(b_s_free + 8 * (k & 1));
      const int slot = k & 1, use = k >> 1;
      if (use >= 1 && !ptx::mbar_wait(b_x_empty + 8 * slot, (use - 1) & 1, abort_flag, true)) return false;
      const uint32_t xp = x_peer + (uint32_t)slot * kXBytes + (uint32_t)row * 16;
      const uint32_t bar = bx_full_peer + 8 * slot;
      // 16 values -> 12 packed words -> three 16-byte stores, four times
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        const uint32_t* src = h < 2 ? r0 + 16 * h : r1 + 16 * (h - 2);
        uint32_t pw[12];
#pragma unroll
        for (int j = 0; j < 4; ++j)
          pack24x4(src[4 * j], src[4 * j + 1], src[4 * j + 2], src[4 * j + 3], pw[3 * j], pw[3 * j + 1], pw[3 * j + 2]);
#pragma unroll
        for (int j = 0; j < 3; ++j)
          ptx::st_async_v4(xp + (3 * h + j) * 128 * 16, __uint_as_float(pw[4 * j]), __uint_as_float(pw[4 * j + 1]),
                           __uint_as_float(pw[4 * j + 2]), __uint_as_float(pw[4 * j + 3]), bar);
      }
      return true;
    };

    // Tile k is prepared one step before tile k-1's scores are sent.
    int g = 0;
    bool dead = false;
    for_each_item_cursor(p, wst, worker, [&](const WorkItem& it) {
      const int b = it.u / p.q_len;
      for (int t0 = it.tok_lo; t0 < it.tok_hi; t0 += kTileN, ++g) {
        if (dead || *abort_flag) return;
        const TileInfo ti = tile_info(p, b, t0, it.tok_hi);
        if (!prepare(g, ti) || (g > 0 && !send(g - 1))) { dead = true; return; }
      }
    });
    if (!dead && g > 0) send(g - 1);
  } else if (warp >= kWarpSoftmax0) {
    // ------------------------------------------------------------------ softmax + epilogue
    ptx::regs_inc<kSoftmaxRegs>();
    const int sw = warp - kWarpSoftmax0;  // 0..7
    const int h2 = sw >> 2;               // half: tile columns [32*h2, +32), O columns [128*h2, +128)
    const int q = warp & 3;               // TMEM lane quadrant this warp may access
    const int row = 32 * q + lane;        // head
    const uint32_t lane_off = (uint32_t)(32 * q) << 16;
    const uint32_t t_s0 = tmem + lane_off + kTmemS;  // + 64 * buffer
    const uint32_t t_o = tmem + lane_off + kTmemO + 128 * h2, t_q = tmem + lane_off + kTmemQ;
    const float scale_log2 = p.sm_scale * p.kv_scale * kLog2e;

    // Q of one work item -> TMEM: this thread's 128 latent columns and 16 rope columns
    auto load_q = [&](const WorkItem& it) {
      const int b = it.u / p.q_len, i = it.u % p.q_len;
      uint32_t v[32];
      const bool real = row < p.H;
      const size_t qrow = ((size_t)b * p.q_len + i) * p.H + (real ? row : 0);
      const uint4* qn = reinterpret_cast<const uint4*>(p.q_nope + qrow * kLatent + 256 * cr + 128 * h2);
      bool q_range = false;
#pragma unroll
      for (int c = 0; c < 2; ++c) {
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint4 x = real ? __ldg(qn + c * 8 + k) : make_uint4(0u, 0u, 0u, 0u);
          v[4 * k] = x.x; v[4 * k + 1] = x.y; v[4 * k + 2] = x.z; v[4 * k + 3] = x.w;
        }
        if (KV != MLA_KV_BF16) {
#pragma unroll
          for (int k = 0; k < 32; ++k) v[k] = bf16x2_to_f16x2(v[k], q_range);
        }
        ptx::tmem_st32(t_q + 64 * h2 + 32 * c, v);
      }
      // rope: this thread's 16 values = 2 of the row's four 16-byte chunks, stored in the
      // 64-byte-swizzled K-major layout the rope MMAs read (chunk c of row r sits at
      // chunk position c ^ ((r >> 1) & 3) of the row's 64 bytes)
      const uint4* qp = reinterpret_cast<const uint4*>(p.q_pe + qrow * kRope + 32 * cr + 16 * h2);
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        uint4 x = real ? __ldg(qp + k) : make_uint4(0u, 0u, 0u, 0u);
        if (KV != MLA_KV_BF16) {
          x.x = bf16x2_to_f16x2(x.x, q_range);
          x.y = bf16x2_to_f16x2(x.y, q_range);
          x.z = bf16x2_to_f16x2(x.z, q_range);
          x.w = bf16x2_to_f16x2(x.w, q_range);
        }
        const int c = 2 * h2 + k;
        *reinterpret_cast<uint4*>(S.q_rope + row * 64 + ((c ^ ((row >> 1) & 3)) * 16)) = x;
      }
      if (q_range) set_status(p.ws, MLA_STATUS_Q_RANGE);
      ptx::fence_proxy_async_smem();
      ptx::tmem_st_wait();
      ptx::tc_fence_before();
      ptx::mbar_arrive(b_q_ready);
    };

    // Epilogue of a finished item: O / l for this thread's 128 columns, and the LSE.
    // P.V completions are awaited in order (od = next tile not yet awaited); P(g) is only
    // handed over after P.V(g-1) completed, so o_done is never two phases ahead of a wait.
    int od = 0;
    auto wait_pv = [&](int k) -> bool {
      for (; od <= k; ++od)
        if (!ptx::mbar_wait(b_o_done, od & 1, abort_flag)) return false;
      return true;
    };
    auto epilogue = [&](const WorkItem& it, float m_ref, float l_half, int g_last, int n_ep) -> bool {
      S.lsum[h2][row] = l_half;
      ptx::mbar_arrive(b_lsum);
      if (!wait_pv(g_last)) return false;
      if (!ptx::mbar_wait(b_lsum, n_ep & 1, abort_flag)) return false;
      ptx::tc_fence_after();
      const float l = S.lsum[0][row] + S.lsum[1][row];
      const int b = it.u / p.q_len, i = it.u % p.q_len;
      const bool real = row < p.H;
      const float inv = l > 0.f ? 1.f / l : 0.f;
      const float lse_v = l > 0.f ? (m_ref + __log2f(l)) * kLn2 : -INFINITY;
      const float oscale = inv * p.kv_scale;
      const size_t orow = ((size_t)b * p.q_len + i) * p.H + (real ? row : 0);
      const int col0 = 256 * (int)cr + 128 * h2;
      const bool direct = it.slot < 0, partial = it.slot >= 0 && it.slot < p.slots_cap;
      for (int c = 0; c < 4; ++c) {
        uint32_t r[32];
        ptx::tmem_ld32(t_o + 32 * c, r);
        ptx::tmem_ld_wait();
        if (real && direct) {
          uint4* dst = reinterpret_cast<uint4*>(p.out + orow * kLatent + col0 + 32 * c);
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            uint4 w;
            w.x = ptx::pack_bf16x2(__uint_as_float(r[8 * k + 0]) * oscale, __uint_as_float(r[8 * k + 1]) * oscale);
            w.y = ptx::pack_bf16x2(__uint_as_float(r[8 * k + 2]) * oscale, __uint_as_float(r[8 * k + 3]) * oscale);
            w.z = ptx::pack_bf16x2(__uint_as_float(r[8 * k + 4]) * oscale, __uint_as_float(r[8 * k + 5]) * oscale);
            w.w = ptx::pack_bf16x2(__uint_as_float(r[8 * k + 6]) * oscale, __uint_as_float(r[8 * k + 7]) * oscale);
            dst[k] = w;
          }
        }
        if (real && partial) {
          float4* dst = reinterpret_cast<float4*>(reinterpret_cast<float*>(p.ws + partial_o_offset()) +
                                                  ((size_t)it.slot * p.H + row) * kLatent + col0 + 32 * c);
#pragma unroll
          for (int k = 0; k < 8; ++k)
            dst[k] = make_float4(__uint_as_float(r[4 * k]) * oscale, __uint_as_float(r[4 * k + 1]) * oscale,
                                 __uint_as_float(r[4 * k + 2]) * oscale, __uint_as_float(r[4 * k + 3]) * oscale);
        }
      }
      if (real && cr == 0 && h2 == 0) {
        if (direct) {
          if (p.lse) p.lse[orow] = lse_v;
        } else if (partial) {
          reinterpret_cast<float*>(p.ws + partial_lse_offset(p.slots_cap, p.H))[(size_t)it.slot * p.H + row] = lse_v;
        }
      }
      ptx::tc_fence_before();
      ptx::mbar_arrive(b_o_free);
      return true;
    };

    int g = 0, n_ep = 0;
    bool dead = false, have_prev = false;
    WorkItem prev{};
    float prev_m = -INFINITY, prev_l = 0.f;
    int prev_g_last = -1;
    for_each_item_cursor(p, wst, worker, [&](const WorkItem& it) {
      if (dead) return;
      // Order: this item's Q (every S of the previous item has been read, so the Q region
      // is free), then the previous item's epilogue, so the MMA warp can already run this
      // item's first score tile while the epilogue drains O.
      load_q(it);
      if (have_prev) {
        if (!epilogue(prev, prev_m, prev_l, prev_g_last, n_ep)) { dead = true; return; }
        ++n_ep;
      }
      const int b = it.u / p.q_len;
      const int nt = (it.tok_hi - it.tok_lo + kTileN - 1) / kTileN;
      float m_ref = -INFINITY, l = 0.f;
      TilePages pages = tile_pages(p, b, it.tok_lo, it.tok_hi);
      for (int t_idx = 0; t_idx < nt; ++t_idx, ++g) {
        const int t0 = it.tok_lo + t_idx * kTileN;
        const TilePages pg_cur = pages;
        if (t_idx + 1 < nt) pages = tile_pages(p, b, t0 + kTileN, it.tok_hi);  // next tile, consumed next iteration
        // ---- own partial scores of this half
        float cur[32];
        const uint32_t t_s = t_s0 + 64 * (g & 1);
        if (!ptx::mbar_wait(b_s_full + 8 * (g & 1), (g >> 1) & 1, abort_flag)) { dead = true; return; }
        ptx::tc_fence_after();
        {
          uint32_t r[32];
          ptx::tmem_ld32(t_s + 32 * h2, r);
          ptx::tmem_ld_wait();
#pragma unroll
          for (int k = 0; k < 32; ++k) cur[k] = __uint_as_float(round24(r[k]));  // as the peer receives it
        }
        ptx::tc_fence_before();
        ptx::mbar_arrive(b_s_free + 8 * (g & 1));
        // ---- the peer's partial scores (pushed by its sender warps)
        const int slot = g & 1, use = g >> 1;
        if (sw == 0 && lane == 0) ptx::mbar_arrive_expect_tx(b_x_full + 8 * slot, kXBytes);
        if (!ptx::mbar_wait(b_x_full + 8 * slot, use & 1, abort_flag, true)) { dead = true; return; }
        float* s = cur;  // full scores of this tile, in place
        uint32_t xw[24];
#pragma unroll
        for (int k = 0; k < 6; ++k) {  // this half's 32 values = 24 words = 6 groups of 4 words
          const uint4 v = S.xbuf[slot][6 * h2 + k][row];
          const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int j = 0; j < 4; ++j) xw[4 * k + j] = w[j];
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          float a, b2, c, d;
          unpack24x4(xw[3 * j], xw[3 * j + 1], xw[3 * j + 2], a, b2, c, d);
          s[4 * j] += a;
          s[4 * j + 1] += b2;
          s[4 * j + 2] += c;
          s[4 * j + 3] += d;
        }
        // The peer may overwrite this buffer once every warp has read it.  The release to
        // the peer is done by the relay warp: a release here would also wait for this
        // thread's asynchronous stores of the next tile, still in flight.
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive_relaxed(b_x_read + 8 * slot);
        // ---- scale, mask (tail tiles only), row max over both halves
        const uint32_t mymask = tile_half_mask(p, pg_cur, t0, it.tok_hi, h2);
        float mh = -INFINITY;
        if (mymask == 0xffffffffu) {
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            s[c] *= scale_log2;
            mh = fmaxf(mh, s[c]);
          }
        } else {
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            s[c] = ((mymask >> c) & 1u) ? s[c] * scale_log2 : -INFINITY;
            mh = fmaxf(mh, s[c]);
          }
        }
        S.mx[g & 1][h2][row] = mh;
        ptx::mbar_arrive(b_mx + 8 * (g & 1));
        if (!ptx::mbar_wait(b_mx + 8 * (g & 1), (g >> 1) & 1, abort_flag)) { dead = true; return; }
        const float mt = fmaxf(mh, S.mx[g & 1][h2 ^ 1][row]);
        // ---- online softmax (base 2), lazy rescale; both halves take identical decisions
        float alpha = 1.f;
        const bool grow = mt > m_ref + kRescaleThreshold;
        if (grow) {
          alpha = ptx::ex2_approx(m_ref - mt);  // m_ref = -inf -> 0
          l *= alpha;
          m_ref = mt;
        }
        const float m_use = m_ref == -INFINITY ? 0.f : m_ref;
        uint32_t pk[16];
        float ls0 = 0.f, ls1 = 0.f;
#pragma unroll
        for (int c = 0; c < 32; c += 2) {
          const float p0 = ptx::ex2_approx(s[c] - m_use), p1 = ptx::ex2_approx(s[c + 1] - m_use);
          ls0 += p0;
          ls1 += p1;
          pk[c / 2] = KV == MLA_KV_BF16 ? ptx::pack_bf16x2(p0, p1) : ptx::pack_f16x2(p0, p1);
        }
        l += ls0 + ls1;
        if (t_idx > 0 && __any_sync(0xffffffffu, grow)) {
          // rescale this thread's 128 columns of O once P.V of the previous tile is done
          if (!wait_pv(g - 1)) { dead = true; return; }
          ptx::tc_fence_after();
          {
            const float a = grow ? alpha : 1.f;
            for (int c = 0; c < 8; ++c) {
              uint32_t r[16];
              ptx::tmem_ld16(t_o + 16 * c, r);
              ptx::tmem_ld_wait();
#pragma unroll
              for (int k = 0; k < 16; ++k) r[k] = __float_as_uint(__uint_as_float(r[k]) * a);
              ptx::tmem_st16(t_o + 16 * c, r);
            }
          }
        }
        // P(g) -> shared memory once P.V(g-1) has consumed P(g-1).  Row r, 16-byte chunk c
        // (8 tokens) sits at chunk position c ^ (r & 7) of the row's 128 bytes (the 128-byte
        // swizzle the P.V MMAs read).
        if (t_idx > 0 && !wait_pv(g - 1)) { dead = true; return; }
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int chunk = 4 * h2 + c;
          *reinterpret_cast<uint4*>(S.p_tile + row * 128 + ((chunk ^ (row & 7)) * 16)) =
              make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
        }
        ptx::fence_proxy_async_smem();
        ptx::tc_fence_before();
        ptx::mbar_arrive(b_p_full);
      }
      have_prev = true;
      prev = it;
      prev_m = m_ref;
      prev_l = l;
      prev_g_last = g - 1;
    });
    if (have_prev && !dead) epilogue(prev, prev_m, prev_l, prev_g_last, n_ep);
  } else {
    // ------------------------------------------------------------------ exchange relay
    // Forwards "my softmax warps have read exchange buffer s" to the peer CTA (the
    // peer's x_empty), with cluster-scope release, from a thread with no stores in flight.
    ptx::regs_dec<kCtrlRegs>();
    if (warp == kWarpRelay && lane == 0) {
      const uint32_t bx_empty_peer = ptx::mapa(b_x_empty, peer);
      int g = 0;
      for_each_item_cursor(p, wst, worker, [&](const WorkItem& it) {
        for (int t0 = it.tok_lo; t0 < it.tok_hi; t0 += kTileN, ++g) {
          if (*abort_flag) return;
          const int slot = g & 1, use = g >> 1;
          if (!ptx::mbar_wait(b_x_read + 8 * slot, use & 1, abort_flag)) return;
          ptx::mbar_arrive_remote(bx_empty_peer + 8 * slot);
        }
      });
    }
  }

  // ------------------------------------------------------------------ teardown
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) ptx::tmem_dealloc(tmem, kTmemCols);
  if (tid == 0 && S.abort_flag) set_status(p.ws, MLA_STATUS_WAIT_TIMEOUT);
  ptx::cluster_sync_all();
}

}  // namespace tc

// ---------------------------------------------------------------------- host side
namespace {
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  }
  return fn;
}

// 2-D view of a bf16 or FP8 cache: [num_pages * page_size rows, 576 columns], one page of
// rows per box.
bool encode_cache_map(CUtensorMap* m, const void* cache, int num_pages, int ps, int box_cols, int elem_bytes,
                      CUtensorMapSwizzle sw) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)kDim, (cuuint64_t)num_pages * ps};
  cuuint64_t strides[1] = {(cuuint64_t)kDim * elem_bytes};
  cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)ps};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, elem_bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 2,
            const_cast<void*>(cache), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
}  // namespace

size_t tc_smem_bytes() { return sizeof(tc::Smem) + 1024; }

// Largest number of 2-CTA clusters of the tensor-core kernel that can be co-resident (the
// three cache formats share block size and shared memory).
int tc_max_clusters() {
  auto kern = tc::mla_decode_tc_kernel<MLA_KV_BF16>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)tc_smem_bytes()) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(sms & ~1);
  cfg.blockDim = dim3(tc::kThreads);
  cfg.dynamicSmemBytes = tc_smem_bytes();
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

template <int KV>
static cudaError_t launch_tc(const CUtensorMap& a, const CUtensorMap& b, const DecodeParams& p, cudaStream_t stream) {
  auto kern = tc::mla_decode_tc_kernel<KV>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)tc_smem_bytes());
  if (e != cudaSuccess) return e;
  kern<<<2 * p.workers, tc::kThreads, tc_smem_bytes(), stream>>>(a, b, p);
  return cudaGetLastError();
}

cudaError_t launch_decode_tc(const DecodeParams& p, cudaStream_t stream) {
  static_assert(sizeof(tc::Smem) + 1024 <= 227 * 1024, "shared memory budget");
  CUtensorMap tm_lat, tm_rope;
  memset(&tm_lat, 0, sizeof(tm_lat));
  memset(&tm_rope, 0, sizeof(tm_rope));
  if (p.kv_dtype == MLA_KV_BF16) {
    if (!encode_cache_map(&tm_lat, p.cache, p.num_pages, p.page_size, 64, 2, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_cache_map(&tm_rope, p.cache, p.num_pages, p.page_size, 32, 2, CU_TENSOR_MAP_SWIZZLE_64B))
      return cudaErrorInvalidValue;
    return launch_tc<MLA_KV_BF16>(tm_lat, tm_rope, p, stream);
  }
  if (p.kv_dtype == MLA_KV_FP8_E4M3) {
    if (!encode_cache_map(&tm_lat, p.cache, p.num_pages, p.page_size, 256, 1, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !encode_cache_map(&tm_rope, p.cache, p.num_pages, p.page_size, 32, 1, CU_TENSOR_MAP_SWIZZLE_NONE))
      return cudaErrorInvalidValue;
    return launch_tc<MLA_KV_FP8_E4M3>(tm_lat, tm_rope, p, stream);
  }
  return launch_tc<MLA_KV_NVFP4>(tm_lat, tm_rope, p, stream);
}

}  // namespace mla

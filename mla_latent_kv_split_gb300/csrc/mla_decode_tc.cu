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
//                   3-stage ring: 4 boxes of 64 tokens x 64 latent columns (128-byte
//                   swizzle) + 1 box of 64 tokens x 32 rope columns (64-byte swizzle)
//   fix-up warp     hands every landed tile to the MMA warp, first zeroing cache rows that
//                   are masked (ragged tail, invalid page) so that garbage (even NaN)
//                   there cannot reach P.V
//   MMA warp        S[128 x 64] = Q[128 x 288] (in TMEM) . K^T       (18 MMAs, K = 16)
//                   O[128 x 256] += P[128 x 64] (in TMEM) . V[64 x 256] (4 MMAs, N = 256)
//   softmax warps   (one thread per head row) load S from TMEM, swap partial scores with
//                   the peer CTA, mask, online softmax in base 2 with a lazy rescale of O
//                   (only when the running max grows by more than 8), write P (bf16) to
//                   TMEM; at the end of a work item normalise O and write the output (or
//                   the split partial and its LSE) for their 256 columns.
//
// Tensor memory (512 columns): O [0,256) fp32, S [256,320) fp32, P [320,352) bf16 pairs,
// Q [352,496) bf16 pairs (256 latent + 32 rope columns of this CTA).
#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "mla_device.cuh"
#include "mla_ptx.cuh"

namespace mla {
namespace tc {

constexpr int kThreads = 256;
constexpr int kStages = 3;
constexpr int kTileN = 64;                      // tokens per tile
constexpr int kLatBox = kTileN * 128;           // 64 rows x 64 bf16 (8 KB)
constexpr int kRopeBox = kTileN * 64;           // 64 rows x 32 bf16 (4 KB)
constexpr int kStageBytes = 4 * kLatBox + kRopeBox;  // 36 KB
constexpr int kXBytes = 128 * kTileN * 4;       // one partial-score tile (32 KB)
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 0, kTmemS = 256, kTmemP = 320, kTmemQ = 352;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;       // log2 units: P stays below 2^8

// warp roles
constexpr int kWarpProducer = 0, kWarpMma = 1, kWarpFixup = 2, kWarpSoftmax0 = 4;

struct Bars {
  uint64_t kv_full[kStages];   // TMA bytes landed
  uint64_t kv_ready[kStages];  // fix-up warp passed the tile (masked rows zeroed)
  uint64_t kv_empty[kStages];  // P.V of the tile completed: stage reusable
  uint64_t s_full;             // S MMAs completed
  uint64_t s_free;             // softmax read S
  uint64_t p_full;             // P written (and O rescaled)
  uint64_t o_done;             // P.V completed
  uint64_t q_ready;            // Q of the next item in TMEM
  uint64_t o_free;             // epilogue read O
  uint64_t x_full[2];          // peer wrote its partial scores into my exchange buffer
  uint64_t x_empty[2];         // peer finished reading its buffer: I may write it again
  uint64_t mma_final;          // every MMA of this CTA completed
};

struct Smem {
  uint8_t stage[kStages][kStageBytes];
  float4 xbuf[2][kTileN / 4][128];  // [slot][column quad][row]
  Bars bars;
  uint32_t tmem_base;
  int abort_flag;
  int scratch[33];
  PlanSmem plan;
};

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
  compute_plan(p, S.plan, S.scratch, blockIdx.x == 0);

  const uint32_t b_kv_full = ptx::smem_u32(&S.bars.kv_full[0]);
  const uint32_t b_kv_ready = ptx::smem_u32(&S.bars.kv_ready[0]);
  const uint32_t b_kv_empty = ptx::smem_u32(&S.bars.kv_empty[0]);
  const uint32_t b_s_full = ptx::smem_u32(&S.bars.s_full), b_s_free = ptx::smem_u32(&S.bars.s_free);
  const uint32_t b_p_full = ptx::smem_u32(&S.bars.p_full), b_o_done = ptx::smem_u32(&S.bars.o_done);
  const uint32_t b_q_ready = ptx::smem_u32(&S.bars.q_ready), b_o_free = ptx::smem_u32(&S.bars.o_free);
  const uint32_t b_x_full = ptx::smem_u32(&S.bars.x_full[0]), b_x_empty = ptx::smem_u32(&S.bars.x_empty[0]);
  const uint32_t b_mma_final = ptx::smem_u32(&S.bars.mma_final);

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(b_kv_full + 8 * s, 1);
      ptx::mbar_init(b_kv_ready + 8 * s, 1);
      ptx::mbar_init(b_kv_empty + 8 * s, 1);
    }
    ptx::mbar_init(b_s_full, 1);
    ptx::mbar_init(b_s_free, 128);
    ptx::mbar_init(b_p_full, 128);
    ptx::mbar_init(b_o_done, 1);
    ptx::mbar_init(b_q_ready, 128);
    ptx::mbar_init(b_o_free, 128);
    for (int s = 0; s < 2; ++s) {
      ptx::mbar_init(b_x_full + 8 * s, 128);
      ptx::mbar_init(b_x_empty + 8 * s, 128);
    }
    ptx::mbar_init(b_mma_final, 1);
    S.abort_flag = 0;
    ptx::fence_mbar_init_cluster();
  }
  if (warp == kWarpMma) {
    ptx::tmem_alloc(ptx::smem_u32(&S.tmem_base), kTmemCols);
    ptx::tmem_relinquish();
  }
  if (warp == kWarpProducer && lane == 0) {
    ptx::prefetch_tmap(&tm_lat);
    ptx::prefetch_tmap(&tm_rope);
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::cluster_sync_all();  // the peer's barriers exist before any remote arrive
  ptx::tc_fence_after();
  const uint32_t tmem = S.tmem_base;

  if (warp == kWarpProducer) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int g = 0;
      for_each_item(p, S.plan, worker, [&](const WorkItem& it) {
        const int b = it.u / p.q_len;
        for (int t0 = it.tok_lo; t0 < it.tok_hi; t0 += kTileN, ++g) {
          if (*abort_flag) return;
          const int st = g % kStages;
          if (g >= kStages && !ptx::mbar_wait(b_kv_empty + 8 * st, ((g / kStages) - 1) & 1, abort_flag)) return;
          const TileInfo ti = tile_info(p, b, t0, it.tok_hi);
          uint32_t bytes = 0;
          for (int j = 0; j < ti.npages; ++j) {
            if (ti.page_ok[j]) bytes += (uint32_t)p.page_size * (4 * 128 + 64);
            else set_status(p.ws, MLA_STATUS_PAGE_OUT_OF_RANGE);
          }
          ptx::mbar_arrive_expect_tx(b_kv_full + 8 * st, bytes);
          const uint32_t dst = ptx::smem_u32(S.stage[st]);
          for (int j = 0; j < ti.npages; ++j) {
            if (!ti.page_ok[j]) continue;
            const int y = ti.page[j] * p.page_size;
            const int roff = j * p.page_size;
#pragma unroll
            for (int k = 0; k < 4; ++k)
              ptx::tma_load_2d(dst + k * kLatBox + roff * 128, &tm_lat, 256 * (int)cr + 64 * k, y,
                               b_kv_full + 8 * st);
            ptx::tma_load_2d(dst + 4 * kLatBox + roff * 64, &tm_rope, 512 + 32 * (int)cr, y, b_kv_full + 8 * st);
          }
        }
      });
      // loads still in flight after an abort must land before the CTA exits
      for (int k = 1; k <= kStages && g - k >= 0; ++k) {
        const int gg = g - k;
        ptx::mbar_wait(b_kv_full + 8 * (gg % kStages), (gg / kStages) & 1, abort_flag, false, 100000000ull);
      }
    }
  } else if (warp == kWarpFixup) {
    // ------------------------------------------------------------------ masked-row fix-up
    int g = 0;
    for_each_item(p, S.plan, worker, [&](const WorkItem& it) {
      const int b = it.u / p.q_len;
      for (int t0 = it.tok_lo; t0 < it.tok_hi; t0 += kTileN, ++g) {
        if (*abort_flag) return;
        const TileInfo ti = tile_info(p, b, t0, it.tok_hi);
        const int st = g % kStages;
        if (!ptx::mbar_wait(b_kv_full + 8 * st, (g / kStages) & 1, abort_flag)) return;
        if (tile_needs_fixup(ti)) {
          uint8_t* base = S.stage[st];
          for (int idx = lane; idx < kTileN * 36; idx += 32) {
            const int r = idx / 36, c = idx % 36;
            if ((ti.rowmask >> r) & 1ull) continue;
            uint8_t* ptr = c < 32 ? base + (c >> 3) * kLatBox + r * 128 + (c & 7) * 16
                                  : base + 4 * kLatBox + r * 64 + (c - 32) * 16;
            *reinterpret_cast<uint4*>(ptr) = make_uint4(0u, 0u, 0u, 0u);
          }
          ptx::fence_proxy_async_smem();
        }
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(b_kv_ready + 8 * st);
      }
    });
  } else if (warp == kWarpMma) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = ptx::idesc_f16(1, 0, 128, kTileN);  // K-major B (cache rows)
      constexpr uint32_t idesc_o = ptx::idesc_f16(1, 1, 128, 256);     // MN-major B (V columns)
      int g = 0, n_item = 0;
      bool dead = false;
      for_each_item(p, S.plan, worker, [&](const WorkItem& it) {
        if (dead) return;
        if (!ptx::mbar_wait(b_q_ready, n_item & 1, abort_flag)) { dead = true; return; }
        ptx::tc_fence_after();
        bool first_pv = true;
        auto issue_pv = [&](int gp) -> bool {
          if (first_pv && n_item > 0) {  // the previous item's epilogue has read O
            if (!ptx::mbar_wait(b_o_free, (n_item - 1) & 1, abort_flag)) return false;
          }
          if (!ptx::mbar_wait(b_p_full, gp & 1, abort_flag)) return false;
          ptx::tc_fence_after();
          const uint32_t vbase = ptx::smem_u32(S.stage[gp % kStages]);
#pragma unroll
          for (int k = 0; k < kTileN / 16; ++k) {
            const uint64_t bdesc = ptx::umma_desc(vbase + k * 16 * 128, kLatBox, 1024, 2);
            ptx::mma_ts(tmem + kTmemO, tmem + kTmemP + 8 * k, bdesc, idesc_o, (first_pv && k == 0) ? 0u : 1u);
          }
          ptx::mma_commit(b_o_done);
          ptx::mma_commit(b_kv_empty + 8 * (gp % kStages));
          first_pv = false;
          return true;
        };
        int t_idx = 0;
        for (int t0 = it.tok_lo; t0 < it.tok_hi; t0 += kTileN, ++g, ++t_idx) {
          const int st = g % kStages;
          // every tile passes the fix-up warp (which zeroes masked rows when there are any)
          if (!ptx::mbar_wait(b_kv_ready + 8 * st, (g / kStages) & 1, abort_flag)) { dead = true; return; }
          if (g > 0 && !ptx::mbar_wait(b_s_free, (g - 1) & 1, abort_flag)) { dead = true; return; }
          ptx::tc_fence_after();
          const uint32_t kbase = ptx::smem_u32(S.stage[st]);
#pragma unroll
          for (int k = 0; k < 16; ++k) {  // 256 latent columns: 4 boxes x 4 steps of 16
            const uint64_t bdesc = ptx::umma_desc(kbase + (k >> 2) * kLatBox + (k & 3) * 32, 16, 1024, 2);
            ptx::mma_ts(tmem + kTmemS, tmem + kTmemQ + 8 * k, bdesc, idesc_s, k > 0 ? 1u : 0u);
          }
#pragma unroll
          for (int k = 0; k < 2; ++k) {  // 32 rope columns (64-byte swizzle)
            const uint64_t bdesc = ptx::umma_desc(kbase + 4 * kLatBox + k * 32, 16, 512, 4);
            ptx::mma_ts(tmem + kTmemS, tmem + kTmemQ + 128 + 8 * k, bdesc, idesc_s, 1u);
          }
          ptx::mma_commit(b_s_full);
          if (t_idx > 0 && !issue_pv(g - 1)) { dead = true; return; }
        }
        if (!issue_pv(g - 1)) { dead = true; return; }
        ++n_item;
      });
      ptx::mma_commit(b_mma_final);
      ptx::mbar_wait(b_mma_final, 0, abort_flag, false, 100000000ull);
    }
  } else if (warp >= kWarpSoftmax0) {
    // ------------------------------------------------------------------ softmax + epilogue
    const int q = warp & 3;
    const int row = 32 * q + lane;  // head
    const uint32_t lane_off = (uint32_t)(32 * q) << 16;
    const uint32_t t_s = tmem + lane_off + kTmemS, t_p = tmem + lane_off + kTmemP;
    const uint32_t t_o = tmem + lane_off + kTmemO, t_q = tmem + lane_off + kTmemQ;
    const float scale_log2 = p.sm_scale * p.kv_scale * kLog2e;
    const uint32_t x_local = ptx::smem_u32(&S.xbuf[0][0][0]);
    const uint32_t x_peer = ptx::mapa(x_local, peer);
    const uint32_t bx_full_peer = ptx::mapa(b_x_full, peer), bx_empty_peer = ptx::mapa(b_x_empty, peer);

    // Q of one work item -> TMEM (this CTA's 256 latent + 32 rope columns, bf16 pairs)
    auto load_q = [&](const WorkItem& it) {
      const int b = it.u / p.q_len, i = it.u % p.q_len;
      uint32_t v[32];
      const bool real = row < p.H;
      const size_t qrow = ((size_t)b * p.q_len + i) * p.H + (real ? row : 0);
      const uint4* qn = reinterpret_cast<const uint4*>(p.q_nope + qrow * kLatent + 256 * cr);
#pragma unroll
      for (int c = 0; c < 4; ++c) {  // 4 x 64 latent values
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint4 x = real ? __ldg(qn + c * 8 + k) : make_uint4(0u, 0u, 0u, 0u);
          v[4 * k] = x.x; v[4 * k + 1] = x.y; v[4 * k + 2] = x.z; v[4 * k + 3] = x.w;
        }
        ptx::tmem_st32(t_q + 32 * c, v);
      }
      const uint4* qp = reinterpret_cast<const uint4*>(p.q_pe + qrow * kRope + 32 * cr);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint4 x = real ? __ldg(qp + k) : make_uint4(0u, 0u, 0u, 0u);
        v[4 * k] = x.x; v[4 * k + 1] = x.y; v[4 * k + 2] = x.z; v[4 * k + 3] = x.w;
      }
      ptx::tmem_st16(t_q + 128, v);
      ptx::tmem_st_wait();
      ptx::tc_fence_before();
      ptx::mbar_arrive(b_q_ready);
    };

    // Epilogue of a finished item: O / l for this CTA's 256 columns, and the LSE.
    auto epilogue = [&](const WorkItem& it, float m_ref, float l, int g_last) -> bool {
      if (!ptx::mbar_wait(b_o_done, g_last & 1, abort_flag)) return false;
      ptx::tc_fence_after();
      const int b = it.u / p.q_len, i = it.u % p.q_len;
      const bool real = row < p.H;
      const float inv = l > 0.f ? 1.f / l : 0.f;
      const float lse_v = l > 0.f ? (m_ref + __log2f(l)) * kLn2 : -INFINITY;
      const float oscale = inv * p.kv_scale;
      const size_t orow = ((size_t)b * p.q_len + i) * p.H + (real ? row : 0);
      const bool direct = it.slot < 0, partial = it.slot >= 0 && it.slot < p.slots_cap;
      for (int c = 0; c < 8; ++c) {
        uint32_t r[32];
        ptx::tmem_ld32(t_o + 32 * c, r);
        ptx::tmem_ld_wait();
        if (real && direct) {
          uint4* dst = reinterpret_cast<uint4*>(p.out + orow * kLatent + 256 * cr + 32 * c);
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
                                                  ((size_t)it.slot * p.H + row) * kLatent + 256 * cr + 32 * c);
#pragma unroll
          for (int k = 0; k < 8; ++k)
            dst[k] = make_float4(__uint_as_float(r[4 * k]) * oscale, __uint_as_float(r[4 * k + 1]) * oscale,
                                 __uint_as_float(r[4 * k + 2]) * oscale, __uint_as_float(r[4 * k + 3]) * oscale);
        }
      }
      if (real && cr == 0) {
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

    int g = 0;
    bool dead = false, have_prev = false;
    WorkItem prev{};
    float prev_m = -INFINITY, prev_l = 0.f;
    int prev_g_last = -1;
    for_each_item(p, S.plan, worker, [&](const WorkItem& it) {
      if (dead) return;
      // Order: this item's Q (every S of the previous item has been read, so the Q region
      // is free), then the previous item's epilogue, so the MMA warp can already run this
      // item's first score tile while the epilogue drains O.
      load_q(it);
      if (have_prev && !epilogue(prev, prev_m, prev_l, prev_g_last)) { dead = true; return; }
      const int b = it.u / p.q_len;
      float m_ref = -INFINITY, l = 0.f;
      int t_idx = 0;
      for (int t0 = it.tok_lo; t0 < it.tok_hi; t0 += kTileN, ++g, ++t_idx) {
        const TileInfo ti = tile_info(p, b, t0, it.tok_hi);
        // ---- own partial scores
        if (!ptx::mbar_wait(b_s_full, g & 1, abort_flag)) { dead = true; return; }
        ptx::tc_fence_after();
        float s[kTileN];
        {
          uint32_t r[32];
          ptx::tmem_ld32(t_s, r);
          ptx::tmem_ld_wait();
#pragma unroll
          for (int k = 0; k < 32; ++k) s[k] = __uint_as_float(r[k]);
          ptx::tmem_ld32(t_s + 32, r);
          ptx::tmem_ld_wait();
#pragma unroll
          for (int k = 0; k < 32; ++k) s[32 + k] = __uint_as_float(r[k]);
        }
        ptx::tc_fence_before();
        ptx::mbar_arrive(b_s_free);
        // ---- exchange partial scores with the peer CTA
        const int slot = g & 1, use = g >> 1;
        if (use >= 1 && !ptx::mbar_wait(b_x_empty + 8 * slot, (use - 1) & 1, abort_flag, true)) { dead = true; return; }
        const uint32_t xp = x_peer + (uint32_t)slot * kXBytes + (uint32_t)row * 16;
#pragma unroll
        for (int c4 = 0; c4 < kTileN / 4; ++c4)
          ptx::st_cluster_v4(xp + c4 * 128 * 16, s[4 * c4], s[4 * c4 + 1], s[4 * c4 + 2], s[4 * c4 + 3]);
        ptx::mbar_arrive_remote(bx_full_peer + 8 * slot);
        if (!ptx::mbar_wait(b_x_full + 8 * slot, use & 1, abort_flag, true)) { dead = true; return; }
#pragma unroll
        for (int c4 = 0; c4 < kTileN / 4; ++c4) {
          const float4 v = S.xbuf[slot][c4][row];
          s[4 * c4] += v.x;
          s[4 * c4 + 1] += v.y;
          s[4 * c4 + 2] += v.z;
          s[4 * c4 + 3] += v.w;
        }
        ptx::mbar_arrive_remote(bx_empty_peer + 8 * slot);
        // ---- mask, online softmax (base 2), lazy rescale
        float mt = -INFINITY;
#pragma unroll
        for (int c = 0; c < kTileN; ++c) {
          s[c] = ((ti.rowmask >> c) & 1ull) ? s[c] * scale_log2 : -INFINITY;
          mt = fmaxf(mt, s[c]);
        }
        float alpha = 1.f;
        const bool grow = mt > m_ref + kRescaleThreshold;
        if (grow) {
          alpha = exp2f(m_ref - mt);  // m_ref = -inf -> 0
          l *= alpha;
          m_ref = mt;
        }
        const float m_use = m_ref == -INFINITY ? 0.f : m_ref;
        uint32_t pk[kTileN / 2];
        float ls = 0.f;
#pragma unroll
        for (int c = 0; c < kTileN; c += 2) {
          const float p0 = exp2f(s[c] - m_use), p1 = exp2f(s[c + 1] - m_use);
          ls += p0 + p1;
          pk[c / 2] = ptx::pack_bf16x2(p0, p1);
        }
        l += ls;
        if (t_idx > 0) {
          // P.V of the previous tile finished: P buffer free, O stable
          if (!ptx::mbar_wait(b_o_done, (g - 1) & 1, abort_flag)) { dead = true; return; }
          ptx::tc_fence_after();
          if (__any_sync(0xffffffffu, grow)) {  // rescale this warp's 32 rows of O
            const float a = grow ? alpha : 1.f;
            for (int c = 0; c < 8; ++c) {
              uint32_t r[32];
              ptx::tmem_ld32(t_o + 32 * c, r);
              ptx::tmem_ld_wait();
#pragma unroll
              for (int k = 0; k < 32; ++k) r[k] = __float_as_uint(__uint_as_float(r[k]) * a);
              ptx::tmem_st32(t_o + 32 * c, r);
            }
          }
        }
        ptx::tmem_st32(t_p, pk);
        ptx::tmem_st_wait();
        ptx::tc_fence_before();
        ptx::mbar_arrive(b_p_full);
      }
      have_prev = true;
      prev = it;
      prev_m = m_ref;
      prev_l = l;
      prev_g_last = g - 1;
    });
    if (have_prev && !dead) epilogue(prev, prev_m, prev_l, prev_g_last);
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

// 2-D view of a bf16 cache: [num_pages * page_size rows, 576 columns], one page per box.
bool encode_cache_map(CUtensorMap* m, const void* cache, int num_pages, int ps, int box_cols,
                      CUtensorMapSwizzle sw) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)kDim, (cuuint64_t)num_pages * ps};
  cuuint64_t strides[1] = {(cuuint64_t)kDim * 2};
  cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)ps};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(cache), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
}  // namespace

size_t tc_smem_bytes() { return sizeof(tc::Smem) + 1024; }

// Largest number of 2-CTA clusters of the tensor-core kernel that can be co-resident.
int tc_max_clusters() {
  if (cudaFuncSetAttribute(tc::mla_decode_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)tc_smem_bytes()) != cudaSuccess) {
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
  if (cudaOccupancyMaxActiveClusters(&n, tc::mla_decode_tc_kernel, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

cudaError_t launch_decode_tc(const DecodeParams& p, cudaStream_t stream) {
  static_assert(sizeof(tc::Smem) + 1024 <= 227 * 1024, "shared memory budget");
  CUtensorMap tm_lat, tm_rope;
  if (!encode_cache_map(&tm_lat, p.cache, p.num_pages, p.page_size, 64, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_cache_map(&tm_rope, p.cache, p.num_pages, p.page_size, 32, CU_TENSOR_MAP_SWIZZLE_64B))
    return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(tc::mla_decode_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)tc_smem_bytes());
  if (e != cudaSuccess) return e;
  tc::mla_decode_tc_kernel<<<2 * p.workers, tc::kThreads, tc_smem_bytes(), stream>>>(tm_lat, tm_rope, p);
  return cudaGetLastError();
}

}  // namespace mla

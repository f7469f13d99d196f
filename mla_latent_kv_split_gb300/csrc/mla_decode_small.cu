// mla_decode_small.cu -- split-KV MLA decode of small calls on the CUDA cores (bf16 cache).
//
// The tensor-core kernel spends ~9 us setting up its pipeline (schedule, tensor memory,
// cluster barriers, the first query and tile loads) before its first P.V, however little
// work a call holds.  A call of a few tiles per request is latency-bound either way, so it
// runs here instead: one CTA per (work item, head), flash-decoding style, with the same
// results contract as the tensor-core kernel (the same work items in forced-split mode, the
// workspace plan, the split partials and their LSEs, per-CTA status words), so the same
// split-K combine follows it.  In heuristic mode (num_splits == 0) a small call's request is
// one work item: its output and LSE are written directly.
//
// Per CTA: the item's query row of head h (512 latent + 64 rope, bf16) is held in registers
// (lane l: latent columns [16l, 16l+16), lanes 0..7 also rope columns [8l, 8l+8)); the 8
// warps take the item's tokens in turn, four at a time: each lane loads its columns of the
// four cache rows, the warp reduces the four dot products with butterfly shuffles, and an
// online softmax in base 2 (TileGym: the log2(e)-folded scale) accumulates P.V into the
// lane's 16 latent columns (V = the latent part of the cache row, already in registers).
// The 8 warps' (max, sum, O) are then combined through shared memory.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "mla_device.cuh"
#include "mla_ptx.cuh"

namespace mla {

constexpr int kSmallThreads = 256;
constexpr int kSmallWarps = kSmallThreads / 32;
constexpr int kSmallGroup = 4;  // cache rows per warp step (their loads all in flight together)

// Work items of unit u in this path: forced mode as the tensor-core kernel (parts of
// cdiv(tiles, num_splits) tiles), heuristic mode one item per unit.
__device__ __forceinline__ int small_parts(int tiles, int num_splits) {
  if (tiles == 0) return 0;
  return num_splits > 0 ? cdiv_i(tiles, forced_span_tiles(tiles, num_splits)) : 1;
}

__device__ __forceinline__ int unit_vis(const DecodeParams& p, int u, unsigned* bad) {
  const int b = u / p.q_len, i = u % p.q_len;
  const int raw = __ldg(p.seq_lens + b);
  if (bad) {
    if (raw < 0) *bad |= MLA_STATUS_NEG_SEQ_LEN;
    if ((long long)raw > (long long)p.max_pages * p.page_size) *bad |= MLA_STATUS_SEQ_TOO_LONG;
  }
  const int L = clamp_seq_len(raw, p.max_pages, p.page_size);
  if (bad && L < p.q_len && i == 0) *bad |= MLA_STATUS_SEQ_LT_QLEN;
  return unit_visible(L, p.q_len, i);
}

__device__ __forceinline__ float bf16lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

// grid: (units * parts_max, H); block: kSmallThreads.
__global__ void __launch_bounds__(kSmallThreads)
mla_decode_small_kernel(const DecodeParams p, int parts_max) {
  asm volatile("griddepcontrol.launch_dependents;");
  __shared__ float sm_m[kSmallWarps], sm_l[kSmallWarps];
  __shared__ float sm_o[kSmallWarps][kLatent];
  __shared__ unsigned sm_status;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int u = blockIdx.x / parts_max, k = blockIdx.x % parts_max, h = blockIdx.y;
  const int cta = blockIdx.y * gridDim.x + blockIdx.x;
  if (tid == 0) sm_status = 0u;
  __syncthreads();

  const int b = u / p.q_len, i = u % p.q_len;
  const size_t qrow = ((size_t)b * p.q_len + i) * p.H + h;
  const int* table = p.block_table + (size_t)b * p.max_pages;

  // ---- this item: the unit's visible range, its parts, the item's tokens and slot
  unsigned bad = 0;
  const int vis = unit_vis(p, u, (k == 0 && h == 0) ? &bad : nullptr);
  const int tiles = unit_tiles(vis, p.window);
  const int parts = small_parts(tiles, p.num_splits);
  if (tid == 0 && k == 0 && h == 0) {
    // partial slots: units are laid out in order, split units taking one slot per part
    int slot = 0;
    for (int v = 0; v < u; ++v) {
      const int pv = small_parts(unit_tiles(unit_vis(p, v, nullptr), p.window), p.num_splits);
      slot += pv > 1 ? pv : 0;
    }
    reinterpret_cast<int2*>(p.ws + kPlanOffset)[u] = make_int2(parts, parts > 1 ? slot : -1);
    if (bad) atomicOr(&sm_status, bad);
  }
  if (k < parts) {
    const int span = p.num_splits > 0 ? forced_span_tiles(tiles, p.num_splits) : tiles;
    const int t0 = unit_tile0(vis, p.window), tmin = window_first(vis, p.window);
    const int tok_lo = (t0 + k * span) * kTile, tok_hi = min((t0 + min((k + 1) * span, tiles)) * kTile, vis);
    const int shift = p.page_size == 32 ? 5 : 6;
    const uint16_t* cache = reinterpret_cast<const uint16_t*>(p.cache);
    // The item's cache rows, asked into L2 at once, one bulk prefetch per page (by one CTA of
    // every 16 heads): the warps' four-row steps then find them there instead of each step
    // (and, before the first, the query row's load) waiting on HBM.
    if ((h & 15) == 0 && warp == 0) {
      const int lo = max(tok_lo, tmin);
      const int pg_first = lo >> shift, n_pages = lo < tok_hi ? ((tok_hi - 1) >> shift) - pg_first + 1 : 0;
      for (int j = lane; j < n_pages; j += 32) {
        const int pi = pg_first + j;
        const int pg = __ldg(table + pi);
        if (pg >= 0 && pg < p.num_pages) {
          const int r0 = max(lo, pi << shift) - (pi << shift), r1 = min(tok_hi, (pi + 1) << shift) - (pi << shift);
          ptx::bulk_prefetch_l2(cache + ((size_t)pg * p.page_size + r0) * kDim, (uint32_t)(r1 - r0) * kDim * 2);
        }
      }
    }

    float qn[16], qp[8];
    {
      const uint4* qsrc = reinterpret_cast<const uint4*>(p.q_nope + qrow * kLatent) + 2 * lane;
      const uint4 qa = __ldg(qsrc), qb = __ldg(qsrc + 1);
      const uint4 qr = lane < 8 ? __ldg(reinterpret_cast<const uint4*>(p.q_pe + qrow * kRope) + lane) : make_uint4(0u, 0u, 0u, 0u);
      const uint32_t w[8] = {qa.x, qa.y, qa.z, qa.w, qb.x, qb.y, qb.z, qb.w};
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        qn[2 * j] = bf16lo(w[j]);
        qn[2 * j + 1] = bf16hi(w[j]);
      }
      const uint32_t wr[4] = {qr.x, qr.y, qr.z, qr.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        qp[2 * j] = bf16lo(wr[j]);
        qp[2 * j + 1] = bf16hi(wr[j]);
      }
    }
    const float scale_log2 = p.sm_scale * 1.4426950408889634f;

    // ---- this warp's tokens: groups of 4 rows, warp w taking groups w, w + 8, ...
    float m = -INFINITY, l = 0.f, acc[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) acc[j] = 0.f;
    for (int t = tok_lo + kSmallGroup * warp; t < tok_hi; t += kSmallGroup * kSmallWarps) {
      uint4 kv[kSmallGroup][3];
      bool ok[kSmallGroup];
#pragma unroll
      for (int g = 0; g < kSmallGroup; ++g) {
        const int tt = t + g;
        int pg = -1;
        if (tt < tok_hi && tt >= tmin) pg = __ldg(table + (tt >> shift));
        ok[g] = pg >= 0 && pg < p.num_pages;
        if (tt < tok_hi && tt >= tmin && !ok[g] && lane == 0) atomicOr(&sm_status, MLA_STATUS_PAGE_OUT_OF_RANGE);
        if (ok[g]) {
          const uint4* row = reinterpret_cast<const uint4*>(cache + ((size_t)pg * p.page_size + (tt & (p.page_size - 1))) * kDim);
          kv[g][0] = __ldg(row + 2 * lane);
          kv[g][1] = __ldg(row + 2 * lane + 1);
          kv[g][2] = lane < 8 ? __ldg(row + 64 + lane) : make_uint4(0u, 0u, 0u, 0u);
        } else {
          kv[g][0] = kv[g][1] = kv[g][2] = make_uint4(0u, 0u, 0u, 0u);
        }
      }
      float s[kSmallGroup];
#pragma unroll
      for (int g = 0; g < kSmallGroup; ++g) {
        const uint32_t w[12] = {kv[g][0].x, kv[g][0].y, kv[g][0].z, kv[g][0].w, kv[g][1].x, kv[g][1].y,
                                kv[g][1].z, kv[g][1].w, kv[g][2].x, kv[g][2].y, kv[g][2].z, kv[g][2].w};
        float d = 0.f;
#pragma unroll
        for (int j = 0; j < 8; ++j) d = fmaf(qn[2 * j], bf16lo(w[j]), fmaf(qn[2 * j + 1], bf16hi(w[j]), d));
#pragma unroll
        for (int j = 0; j < 4; ++j) d = fmaf(qp[2 * j], bf16lo(w[8 + j]), fmaf(qp[2 * j + 1], bf16hi(w[8 + j]), d));
        s[g] = d;
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1)
#pragma unroll
        for (int g = 0; g < kSmallGroup; ++g) s[g] += __shfl_xor_sync(0xffffffffu, s[g], off);
      float mg = m;
#pragma unroll
      for (int g = 0; g < kSmallGroup; ++g) {
        s[g] = ok[g] ? s[g] * scale_log2 : -INFINITY;
        mg = fmaxf(mg, s[g]);
      }
      if (mg == -INFINITY) continue;  // nothing attended yet
      const float c = exp2f(m - mg);  // m = -inf -> 0
      l *= c;
#pragma unroll
      for (int j = 0; j < 16; ++j) acc[j] *= c;
      m = mg;
#pragma unroll
      for (int g = 0; g < kSmallGroup; ++g) {
        const float pr = exp2f(s[g] - m);  // masked rows: 0
        l += pr;
        const uint32_t w[8] = {kv[g][0].x, kv[g][0].y, kv[g][0].z, kv[g][0].w,
                               kv[g][1].x, kv[g][1].y, kv[g][1].z, kv[g][1].w};
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          acc[2 * j] = fmaf(pr, bf16lo(w[j]), acc[2 * j]);
          acc[2 * j + 1] = fmaf(pr, bf16hi(w[j]), acc[2 * j + 1]);
        }
      }
    }
    // ---- the warps' partial results meet
    if (lane == 0) {
      sm_m[warp] = m;
      sm_l[warp] = l;
    }
#pragma unroll
    for (int j = 0; j < 16; ++j) sm_o[warp][16 * lane + j] = acc[j];
    __syncthreads();
    float mx = -INFINITY;
#pragma unroll
    for (int w = 0; w < kSmallWarps; ++w) mx = fmaxf(mx, sm_m[w]);
    float lt = 0.f, f[kSmallWarps];
#pragma unroll
    for (int w = 0; w < kSmallWarps; ++w) {
      f[w] = sm_m[w] == -INFINITY ? 0.f : exp2f(sm_m[w] - mx);
      lt += sm_l[w] * f[w];
    }
    // thread tid: latent columns 2 tid, 2 tid + 1
    float o0 = 0.f, o1 = 0.f;
#pragma unroll
    for (int w = 0; w < kSmallWarps; ++w) {
      o0 = fmaf(sm_o[w][2 * tid], f[w], o0);
      o1 = fmaf(sm_o[w][2 * tid + 1], f[w], o1);
    }
    const bool direct = parts == 1;
    float oscale = lt > 0.f ? 1.f / lt : 0.f;
    float m_fin = mx, l_fin = lt;
    if (direct && p.sinks != nullptr) {
      // the head's sink logit (natural-log units of the scaled scores) joins the normaliser
      const float sk = __ldg(p.sinks + h) * 1.4426950408889634f;
      if (sk > m_fin) {
        const float w = l_fin > 0.f ? exp2f(m_fin - sk) : 0.f;
        oscale = l_fin > 0.f ? w / (l_fin * w + 1.f) : 0.f;
        l_fin = l_fin * w + 1.f;
        m_fin = sk;
      } else if (sk != -INFINITY) {
        l_fin += exp2f(sk - m_fin);
        oscale = l_fin > 0.f ? 1.f / l_fin : 0.f;
      }
    }
    const float lse_v = l_fin > 0.f ? (m_fin + log2f(l_fin)) * 0.6931471805599453f : -INFINITY;
    const uint32_t packed = (uint32_t)float_to_bf16_bits_rn(o0 * oscale) | ((uint32_t)float_to_bf16_bits_rn(o1 * oscale) << 16);
    if (direct) {
      reinterpret_cast<uint32_t*>(p.out + qrow * kLatent)[tid] = packed;
      if (tid == 0 && p.lse) p.lse[qrow] = lse_v;
    } else {
      // partial slot: the unit's first slot (from the plan written above by this unit's
      // first CTA is not visible here; it is recomputed) plus the part index
      int slot = 0;
      for (int v = 0; v < u; ++v) {
        const int pv = small_parts(unit_tiles(unit_vis(p, v, nullptr), p.window), p.num_splits);
        slot += pv > 1 ? pv : 0;
      }
      slot += k;
      if (slot < p.slots_cap) {
        // column-octet-major bf16 partials: [slot][64 octets][H][8]; this thread's two
        // columns are half a word of octet tid / 4
        uint32_t* part = reinterpret_cast<uint32_t*>(p.ws + partial_o_offset());
        part[(((size_t)slot * 64 + (tid >> 2)) * p.H + h) * 4 + (tid & 3)] = packed;
        if (tid == 0) reinterpret_cast<float*>(p.ws + partial_lse_offset(p.slots_cap, p.H))[(size_t)slot * p.H + h] = lse_v;
      }
    }
  }
  __syncthreads();
  if (tid == 0) reinterpret_cast<unsigned*>(p.ws + kCtaStatusOffset)[cta] = sm_status;
}

cudaError_t launch_decode_small(const DecodeParams& p, int parts_max, cudaStream_t stream) {
  dim3 grid(p.B * p.q_len * parts_max, p.H);
  mla_decode_small_kernel<<<grid, kSmallThreads, 0, stream>>>(p, parts_max);
  return cudaGetLastError();
}

}  // namespace mla

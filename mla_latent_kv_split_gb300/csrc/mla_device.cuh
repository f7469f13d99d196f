// mla_device.cuh -- device-side pieces shared by the decode kernels: launch parameters,
// the in-kernel evaluation of the split schedule, the status word, and exact decoding of
// the FP8 / NVFP4 storage codes.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "mla_common.cuh"

namespace mla {

struct DecodeParams {
  const uint16_t* q_nope;     // [B, q_len, H, 512] bf16 bits
  const uint16_t* q_pe;       // [B, q_len, H, 64]  bf16 bits
  const uint8_t* cache;       // paged cache (layout per kv_dtype)
  const int32_t* block_table; // [B, max_pages]
  const int32_t* seq_lens;    // [B]
  int max_pages, B, q_len, H, num_pages, page_size;
  float sm_scale, kv_scale;
  int kv_dtype, num_splits;
  int workers;                // scheduling workers C
  int slots_cap;              // partial slots that fit the workspace
  uint8_t* ws;                // workspace
  uint16_t* out;              // [B, q_len, H, 512] bf16 bits
  float* lse;                 // [B, q_len, H] or nullptr
  int window;                 // sliding window (0: none)
  const float* sinks;         // [H] per-head sink logits or nullptr
};

// Status bits accumulate in a CTA-local word (shared memory) that the CTA stores at exit.
__device__ __forceinline__ void set_status(unsigned* cta_status, unsigned bits) { atomicOr(cta_status, bits); }

// Bytes per page of the cache.
__host__ __device__ __forceinline__ size_t page_stride_bytes(int kv_dtype, int page_size) {
  return kv_dtype == MLA_KV_BF16 ? (size_t)page_size * kDim * 2
       : kv_dtype == MLA_KV_FP8_E4M3 ? (size_t)page_size * kDim
       : (size_t)page_size * (kDim / 2 + kDim / kNvfp4Group);
}

// ---------------------------------------------------------------- exact code decoding
// E4M3 (OCP FP8 "FN"): sign bit 7, exponent 6..3 (bias 7), mantissa 2..0; exponent 0 is
// subnormal (m * 2^-9); S.1111.111 is NaN.  Built from the bit fields, exact in fp32.
__device__ __forceinline__ float e4m3_to_float(unsigned code) {
  unsigned s = (code & 0x80u) << 24, e = (code >> 3) & 0xFu, m = code & 0x7u;
  float v;
  if (e == 0) {
    v = (float)m * 0.001953125f;  // m * 2^-9
  } else if (e == 0xF && m == 0x7) {
    v = __int_as_float(0x7fc00000);
  } else {
    v = __int_as_float((int)(((e + 120u) << 23) | (m << 20)));
  }
  return __int_as_float(__float_as_int(v) | (int)s);
}
// E2M1 (OCP MX FP4): sign bit 3, exponent 2..1 (bias 1), mantissa bit 0; exponent 0 is
// subnormal (m * 0.5).
__device__ __forceinline__ float e2m1_to_float(unsigned nib) {
  unsigned s = (nib & 0x8u) << 28, e = (nib >> 1) & 0x3u, m = nib & 0x1u;
  float v = e == 0 ? 0.5f * (float)m : __int_as_float((int)(((e + 126u) << 23) | (m << 22)));
  return __int_as_float(__float_as_int(v) | (int)s);
}
__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) {
  return __int_as_float(((int)b) << 16);
}
__device__ __forceinline__ uint16_t float_to_bf16_bits_rn(float f) {
  unsigned short r;
  asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(r) : "f"(f));
  return r;
}

// ---------------------------------------------------------------- schedule on the device
// Indexed by schedule position k (unit unit_at(k)).
struct PlanSmem {
  int N;                     // total tiles (heuristic) or items (forced)
  int begin[kMaxUnits + 1];  // exclusive prefix of tiles / items
  int vis[kMaxUnits];        // visible positions of the unit
  int slot[kMaxUnits];       // first partial slot or -1
  int pref[kMaxUnits];       // exclusive prefix of the partial slots of split units
};

// Exclusive scan of vals[0..n) in place by one warp (all 32 lanes call); returns the total.
__device__ inline int warp_exclusive_scan(int* vals, int n) {
  const int lane = threadIdx.x & 31;
  int carry = 0;
  for (int base = 0; base < n; base += 32) {
    const int k = base + lane;
    const int v = k < n ? vals[k] : 0;
    int x = v;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, d);
      if (lane >= d) x += y;
    }
    if (k < n) vals[k] = carry + x - v;
    carry += __shfl_sync(0xffffffffu, x, 31);
  }
  return carry;
}

// Evaluates the schedule in shared memory with one warp (its 32 lanes call; no other thread
// touches pl meanwhile).  Sets status bits for malformed seq_lens.  When `write_plan` is set,
// also stores {parts, slot} per unit into the workspace plan for the split-K reduce.
__device__ inline void compute_plan_warp(const DecodeParams& p, PlanSmem& pl, unsigned* cta_status, bool write_plan) {
  const int lane = threadIdx.x & 31;
  const int U = p.B * p.q_len;
  unsigned bad = 0;
  for (int k = lane; k < U; k += 32) {
    const int u = unit_at(k, p.B, p.q_len, p.num_splits);
    const int b = u / p.q_len, i = u % p.q_len;
    const int raw = __ldg(p.seq_lens + b);
    if (raw < 0) bad |= MLA_STATUS_NEG_SEQ_LEN;
    if ((long long)raw > (long long)p.max_pages * p.page_size) bad |= MLA_STATUS_SEQ_TOO_LONG;
    const int L = clamp_seq_len(raw, p.max_pages, p.page_size);
    if (L < p.q_len && i == 0) bad |= MLA_STATUS_SEQ_LT_QLEN;
    const int vis = unit_visible(L, p.q_len, i);
    pl.vis[k] = vis;
    const int tiles = unit_tiles(vis, p.window);
    pl.begin[k] = p.num_splits > 0 ? (tiles ? cdiv_i(tiles, forced_span_tiles(tiles, p.num_splits)) : 0)
                                   : unit_slots(tiles);
  }
  if (bad && write_plan) set_status(cta_status, bad);
  __syncwarp();
  const int N = warp_exclusive_scan(pl.begin, U);
  if (lane == 0) {
    pl.begin[U] = N;
    pl.N = N;
  }
  __syncwarp();
  // parts per unit -> slot scan (pl.slot holds the per-unit split-part count first)
  const int Ca = active_workers(N, p.workers);
  auto parts_of = [&](int k) {
    return p.num_splits > 0 ? pl.begin[k + 1] - pl.begin[k]
         : (pl.begin[k + 1] > pl.begin[k]
                ? worker_of(pl.begin[k + 1] - 1, N, Ca) - worker_of(pl.begin[k] + kItemCost, N, Ca) + 1
                : 0);
  };
  int2* plan = reinterpret_cast<int2*>(p.ws + kPlanOffset);
  for (int k = lane; k < U; k += 32) {
    const int parts = parts_of(k);
    pl.slot[k] = parts > 1 ? parts : 0;
    if (write_plan) plan[unit_at(k, p.B, p.q_len, p.num_splits)].x = parts;
  }
  __syncwarp();
  warp_exclusive_scan(pl.slot, U);
  __syncwarp();
  for (int k = lane; k < U; k += 32) {
    pl.pref[k] = pl.slot[k];
    if (parts_of(k) <= 1) pl.slot[k] = -1;
    if (write_plan) plan[unit_at(k, p.B, p.q_len, p.num_splits)].y = pl.slot[k];
  }
  __syncwarp();
}

// One work item: unit u, token range [tok_lo, tok_hi) of its visible KV, partial slot
// (or -1 = final output written directly).
struct WorkItem {
  int u, tok_lo, tok_hi, slot;
  int tok_min;  // the unit's first attended position (sliding window; 0 without one)
};

// Smallest index k in [0, n] with a[k] > x, for a non-decreasing a.
__device__ __forceinline__ int upper_bound_i(const int* a, int n, int x) {
  int lo = 0, hi = n;
  while (lo < hi) {
    int mid = (lo + hi) >> 1;
    if (a[mid] <= x) lo = mid + 1; else hi = mid;
  }
  return lo;
}

// ---------------------------------------------------------------- cursor form
// Where worker c starts in the schedule: its first unit, that unit's first tile (heuristic
// mode) or first item (forced mode), the partial slots used by earlier units, and the
// total tile / item count.  From these the worker walks its items reading only seq_lens,
// so the per-unit arrays of PlanSmem need not stay resident.  The worker's first item is
// evaluated here as well, from the plan, so that it is known before any cursor runs.
struct WorkerStart {
  int u0, base0, slot0, N;
  int k0;          // schedule position of unit u0
  int busy;        // the worker has at least one item
  WorkItem first;  // its first item (when busy)
};

__device__ inline WorkerStart worker_start(const DecodeParams& p, const PlanSmem& pl, int c) {
  const int U = p.B * p.q_len;
  WorkerStart w{0, 0, 0, pl.N, 0, 0, WorkItem{0, 0, 0, -1, 0}};
  if (pl.N <= 0) return w;
  int first;
  int Ca = 0;
  if (p.num_splits > 0) {
    first = c;
  } else {
    Ca = active_workers(pl.N, p.workers);
    if (c >= Ca) return w;
    first = (int)worker_begin(c, pl.N, Ca);
  }
  if (first >= pl.N) return w;
  const int kp = upper_bound_i(pl.begin, U + 1, first) - 1;
  const int u = unit_at(kp, p.B, p.q_len, p.num_splits);
  w.u0 = u;
  w.k0 = kp;
  w.base0 = pl.begin[kp];
  w.slot0 = pl.pref[kp];
  w.busy = 1;
  const int vis = pl.vis[kp], tiles = unit_tiles(vis, p.window);
  const int t0 = unit_tile0(vis, p.window), tmin = window_first(vis, p.window);
  if (p.num_splits > 0) {  // item `first` is part k of unit u
    const int k = first - w.base0;
    const int span = forced_span_tiles(tiles, p.num_splits);
    const int lo = k * span, hi = min((k + 1) * span, tiles);
    w.first = WorkItem{u, (t0 + lo) * kTile, min((t0 + hi) * kTile, vis), pl.slot[kp] >= 0 ? pl.slot[kp] + k : -1, tmin};
  } else {  // the unit's tiles inside [first, end of the worker's range)
    const long long e = worker_begin(c + 1, pl.N, Ca);
    const long long r0 = (long long)w.base0 + kItemCost;  // the unit's first tile
    const long long lo = max((long long)first, r0), hi = min(e, r0 + tiles);
    if (hi <= lo) {  // the range ends inside the unit's placeholder slots: no work
      w.busy = 0;
      return w;
    }
    w.first = WorkItem{u, (t0 + (int)(lo - r0)) * kTile, min((t0 + (int)(hi - r0)) * kTile, vis),
                       pl.slot[kp] >= 0 ? pl.slot[kp] + (c - worker_of(r0, pl.N, Ca)) : -1, tmin};
  }
  return w;
}

__device__ __forceinline__ int unit_visible_dev(const DecodeParams& p, int u) {
  const int b = u / p.q_len, i = u % p.q_len;
  return unit_visible(clamp_seq_len(__ldg(p.seq_lens + b), p.max_pages, p.page_size), p.q_len, i);
}

// Worker c's items one at a time, in for_each_item's order, walking units from the worker's
// start and reading only seq_lens.  A copy of a cursor looks ahead without disturbing it.
struct ItemCursor {
  int k, sacc, j, ib, c;  // k: schedule position of the current unit
  long long tb, t, e;
  bool live;
};

__device__ inline ItemCursor item_cursor(const DecodeParams& p, const WorkerStart& w, int c) {
  ItemCursor k{};
  k.c = c;
  k.live = w.N > 0;
  k.k = w.k0;
  k.sacc = w.slot0;
  if (!k.live) return k;
  if (p.num_splits > 0) {
    k.ib = w.base0;
    k.j = c;
  } else {
    const int Ca = active_workers(w.N, p.workers);
    if (c >= Ca) {
      k.live = false;
      return k;
    }
    k.t = worker_begin(c, w.N, Ca);
    k.e = worker_begin(c + 1, w.N, Ca);
    k.tb = w.base0;
    if (k.t >= k.e) k.live = false;
  }
  return k;
}

__device__ inline bool next_item(const DecodeParams& p, int N, ItemCursor& k, WorkItem& it) {
  if (!k.live) return false;
  if (p.num_splits > 0) {
    if (k.j >= N) return false;
    int vis, tiles, parts, span;
    for (;;) {  // forced mode: schedule position = unit
      vis = unit_visible_dev(p, k.k);
      tiles = unit_tiles(vis, p.window);
      span = forced_span_tiles(tiles, p.num_splits);
      parts = tiles ? cdiv_i(tiles, span) : 0;
      if (k.ib + parts > k.j) break;
      k.sacc += parts > 1 ? parts : 0;
      k.ib += parts;
      ++k.k;
    }
    const int q = k.j - k.ib;
    const int lo = q * span, hi = min((q + 1) * span, tiles);
    const int t0 = unit_tile0(vis, p.window);
    it = WorkItem{k.k, (t0 + lo) * kTile, min((t0 + hi) * kTile, vis), parts > 1 ? k.sacc + q : -1,
                  window_first(vis, p.window)};
    k.j += p.workers;
    return true;
  }
  const int Ca = active_workers(N, p.workers);
  while (k.t < k.e) {
    const int u = unit_at(k.k, p.B, p.q_len, p.num_splits);
    const int vis = unit_visible_dev(p, u);
    const int tiles = unit_tiles(vis, p.window);
    const long long te = k.tb + unit_slots(tiles);  // the unit's slots end
    const long long r0 = k.tb + kItemCost;          // its first tile
    const int parts = tiles ? worker_of(te - 1, N, Ca) - worker_of(r0, N, Ca) + 1 : 0;
    const long long lo = max(k.t, r0), hi = min(k.e, te);
    const bool emit = tiles > 0 && hi > lo;
    if (emit) {
      const int t0 = unit_tile0(vis, p.window);
      it = WorkItem{u, (t0 + (int)(lo - r0)) * kTile, min((t0 + (int)(hi - r0)) * kTile, vis),
                    parts > 1 ? k.sacc + (k.c - worker_of(r0, N, Ca)) : -1, window_first(vis, p.window)};
    }
    k.t = max(k.t, min(k.e, te));
    if (k.t >= te) {
      k.sacc += parts > 1 ? parts : 0;
      k.tb = te;
      ++k.k;
    }
    if (emit) return true;
  }
  return false;
}

}  // namespace mla

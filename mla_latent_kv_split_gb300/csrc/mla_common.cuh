// mla_common.cuh -- constants, the split schedule and the workspace layout shared by the
// host layer and every kernel of the MLA split-KV decode.
//
// The schedule (which scheduling worker covers which KV range of which (b, i)) is a pure
// function of seq_lens, q_len, the page geometry, num_splits and the worker count.  The
// kernels evaluate it on the device from seq_lens (no host sync, graph-safe); the host
// evaluates the same inline functions only to answer mla_decode_plan_host for tests.
#pragma once

#include <stdint.h>

#include "../../include/mla_decode.h"

#if defined(__CUDACC__)
#define MLA_HD __host__ __device__ __forceinline__
#else
#define MLA_HD inline
#endif

namespace mla {

constexpr int kLatent = MLA_LATENT_DIM;  // 512: latent, also V
constexpr int kRope = MLA_ROPE_DIM;      // 64
constexpr int kDim = MLA_CACHE_DIM;      // 576
constexpr int kTile = 64;                // tokens per schedule tile
constexpr int kMaxUnits = MLA_MAX_UNITS; // B * q_len
constexpr int kNvfp4Group = 16;

// Workspace layout (bytes):
//   [0, 4)                      device status word (written by the split-K reduce each call)
//   [4, 8)                      schedule mode written by the decode kernel
//   [kPlanOffset, +8*units)     plan: per unit {parts, first partial slot}
//   [kCtaStatusOffset, +4*CTAs) status bits of each decode CTA (written unconditionally at its
//                               exit; the split-K reduce ORs them into the status word)
//   [kHeaderBytes, ...)         partial outputs  bf16 [slots][64][H][8]: column octets
//                               outermost, so that 32 consecutive heads' values of one
//                               octet are 512 contiguous bytes (the region is sized for
//                               fp32, slots*H*512*4 bytes, of which half is used)
//   then                        partial LSEs     fp32 [slots][H]
constexpr size_t kPlanOffset = 256;
constexpr size_t kCtaStatusOffset = 16384;
constexpr int kMaxCtas = 2048;
constexpr size_t kHeaderBytes = 32768;
static_assert(kPlanOffset + 8 * (size_t)kMaxUnits <= kCtaStatusOffset, "plan must fit below the CTA status words");
static_assert(kCtaStatusOffset + 4 * (size_t)kMaxCtas <= kHeaderBytes, "CTA status words must fit the header");

MLA_HD size_t partial_o_offset() { return kHeaderBytes; }
MLA_HD size_t partial_lse_offset(int slots, int H) {
  return kHeaderBytes + (size_t)slots * H * kLatent * 4;
}
MLA_HD size_t workspace_bytes_for(int slots, int H) {
  return kHeaderBytes + (size_t)slots * H * (kLatent + 1) * 4;
}

MLA_HD int cdiv_i(int a, int b) { return (a + b - 1) / b; }

// Positions query i of q_len may see: t < seq_len - q_len + i + 1 (the last q_len cache
// positions are this step's tokens); seq_len is clamped to [0, max_pages*page_size].
MLA_HD int clamp_seq_len(int seq_len, int max_pages, int page_size) {
  long long cap = (long long)max_pages * page_size;
  if (seq_len < 0) return 0;
  return (long long)seq_len > cap ? (int)cap : seq_len;
}
MLA_HD int unit_visible(int seq_len_clamped, int q_len, int i) {
  int v = seq_len_clamped - q_len + i + 1;
  return v < 0 ? 0 : v;
}

// Sliding window (window > 0): a query attends the last `window` of its visible positions,
// [window_first, vis).  Its KV range is cut into 64-token tiles starting at the tile that
// holds window_first (the rows before it are masked inside that tile).
MLA_HD int window_first(int vis, int window) { return window > 0 && vis > window ? vis - window : 0; }
MLA_HD int unit_tile0(int vis, int window) { return window_first(vis, window) / kTile; }
MLA_HD int unit_tiles(int vis, int window) { return vis > 0 ? cdiv_i(vis, kTile) - unit_tile0(vis, window) : 0; }

// ---- heuristic mode (num_splits == 0): contiguous, balanced ranges per worker ----
// Units are laid end to end in schedule order.  With q_len == 1 that is the unit order.
// With q_len > 1 it is query-major (position k = i * B + b holds unit (b, i)): the q_len
// queries of a request then sit at the same offsets of q_len nearly equal stretches of the
// schedule, so that (with a worker count divisible by q_len) the workers serving the
// different queries of a request walk the same pages at the same time and all but the
// first of each page's reads come from L2.
MLA_HD bool query_major(int q_len, int num_splits) { return q_len > 1 && num_splits == 0; }
MLA_HD int unit_at(int k, int B, int q_len, int num_splits) {
  return query_major(q_len, num_splits) ? (k % B) * q_len + k / B : k;
}
// Every unit with visible KV is laid out as kItemCost placeholder slots (the fixed cost of
// starting a work item on it: its query load, pipeline refill and epilogue, measured at
// about four tiles' time) followed by its tiles.  With N slots in all and C workers, only
// C' = min(C, N) workers get a range, worker c < C' owning slots [floor(c*N/C'),
// floor((c+1)*N/C')); its work is the tiles inside that range.  A worker that starts a new
// unit inside its range thereby gets fewer tiles.  Callers pass C'.
constexpr int kItemCost = 4;
MLA_HD int unit_slots(int tiles) { return tiles > 0 ? tiles + kItemCost : 0; }
MLA_HD int active_workers(long long N, int C) { return N < (long long)C ? (int)N : C; }
MLA_HD long long worker_begin(int c, long long N, int C) { return (long long)c * N / C; }
// The worker whose range holds tile t (0 <= t < N): the largest c with begin(c) <= t.
MLA_HD int worker_of(long long t, long long N, int C) {
  return (int)(((t + 1) * (long long)C + N - 1) / N - 1);
}

// ---- forced mode (num_splits > 0): each unit cut into ranges of span tiles ----
// span = cdiv(tiles, num_splits) tiles.  Without a window, tiles = cdiv(visible, 64) and
// this equals roundup(cdiv(visible, num_splits), 64) / 64 (nested ceilings compose); with
// one, counting the unit's tiles keeps it at num_splits parts at most.
MLA_HD int forced_span_tiles(int tiles, int num_splits) { return tiles > 0 ? cdiv_i(tiles, num_splits) : 1; }

// One unit's share of the schedule.
struct UnitPlan {
  int tile_begin;  // heuristic: first global tile; forced: first global item
  int tiles;       // tiles of visible KV
  int parts;       // number of KV ranges it is cut into (0 when nothing is visible)
  int slot;        // first partial slot, -1 when written directly (parts <= 1)
};

// Host evaluation of the whole plan (the device kernels evaluate the same formulas with a
// block-wide scan).  plan[] is indexed by unit; tile_begin and the partial slots follow the
// schedule order.  Returns the number of partial slots used.
inline int plan_host(const int32_t* seq_lens, int B, int q_len, int max_pages, int page_size,
                     int num_splits, int C, UnitPlan* plan, int window = 0) {
  const int U = B * q_len;
  long long N = 0;
  for (int k = 0; k < U; ++k) {
    const int u = unit_at(k, B, q_len, num_splits);
    int b = u / q_len, i = u % q_len;
    int L = clamp_seq_len(seq_lens[b], max_pages, page_size);
    int vis = unit_visible(L, q_len, i);
    plan[u].tiles = unit_tiles(vis, window);
    if (num_splits > 0) {
      plan[u].parts = plan[u].tiles
                          ? cdiv_i(plan[u].tiles, forced_span_tiles(plan[u].tiles, num_splits))
                          : 0;
      plan[u].tile_begin = (int)N;  // first item index
      N += plan[u].parts;
    } else {
      plan[u].tile_begin = (int)N;  // first slot (its tiles start kItemCost slots later)
      N += unit_slots(plan[u].tiles);
    }
  }
  int slots = 0;
  const int Ca = active_workers(N, C);
  for (int k = 0; k < U; ++k) {
    const int u = unit_at(k, B, q_len, num_splits);
    if (num_splits == 0) {
      if (plan[u].tiles == 0) {
        plan[u].parts = 0;
      } else {
        const long long r0 = (long long)plan[u].tile_begin + kItemCost;
        int c0 = worker_of(r0, N, Ca);
        int c1 = worker_of(r0 + plan[u].tiles - 1, N, Ca);
        plan[u].parts = c1 - c0 + 1;
      }
    }
    if (plan[u].parts > 1) {
      plan[u].slot = slots;
      slots += plan[u].parts;
    } else {
      plan[u].slot = -1;
    }
  }
  return slots;
}

// Bound on partial slots for a shape: heuristic mode cuts at most C-1 worker boundaries
// into units, so split units hold at most 2*(C-1) partials; forced mode at most
// num_splits per unit.
MLA_HD int max_slots(int units, int num_splits, int C) {
  if (num_splits > 0) return units * num_splits;
  int s = 2 * C;
  return s;
}

}  // namespace mla

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
//   distributed shared memory, so both hold the full scores.  Every cache byte is read
//   from HBM once.
//
// Per CTA, per 64-token tile (TileGym: K = V = KV; tokenspeed: paged cache):
//   producer warp   TMA-gathers the tile's pages (block table -> page rows) into a
//                   4-stage ring: 4 boxes of 64 tokens x 64 latent columns (128-byte
//                   swizzle) + 1 box of 64 tokens x 32 rope columns (64-byte swizzle)
//                   (FP8: the E4M3 bytes of those columns; NVFP4: whole pages, packed
//                   E2M1 data plus E4M3 scales, into the tail of the stage)
//   MMA warps       one issues S[128 x 64] = Q[128 x 288] (in TMEM) . K^T (18 MMAs, K = 16),
//                   the other O[128 x 256] += P[128 x 64] (in smem) . V[64 x 256] (4 MMAs, N = 256)
//   producer warp   also zeroes the masked rows of a bf16 tile (ragged tail, invalid page)
//                   after it lands, so that garbage, even NaN, cannot reach P.V.
//   sender warps    one warpgroup.  (1) Loads each work item's Q into TMEM (latent) and
//                   shared memory (rope), once the previous item's score MMAs are done.
//                   (2) bf16 / NVFP4: thread = head row: loads the row's 64 partial scores
//                   from TMEM and pushes them (24-bit packed) into the peer CTA's exchange
//                   buffer with asynchronous stores that complete on the peer's mbarrier.
//                   FP8: decodes each landed tile's E4M3 bytes in place into f16 (exact) in
//                   the swizzled layout the MMAs read, masked rows as zeros.
//   softmax warps   two warpgroups; thread = head row.  bf16 / NVFP4: both take every
//                   tile, 32 of its 64 columns each, and the two halves of a row exchange
//                   their maxima through shared memory.  FP8: they take alternate tiles
//                   (even / odd), all 64 columns, so two tiles are in flight.  A thread loads
//                   its partial scores from TMEM (FP8: and pushes them to the peer itself),
//                   adds the peer's, takes the row max, and runs the online softmax in base 2
//                   with a lazy reference max: the reference only moves (and O is rescaled)
//                   when a tile's max exceeds it by more than 8 (alternate tiles pass it from
//                   one warpgroup to the other through shared memory).  P (bf16 / f16) goes
//                   into the exchange slot the partial scores arrived in; at the end of a
//                   work item both warpgroups normalise O (128 columns each) and write the
//                   output, or the split partial and its LSE.  NVFP4: the two warpgroups
//                   decode the tiles (E2M1 x E4M3 scale, exact in f16) in place, two ahead.
//
// Tensor memory (512 columns): O [0,256) fp32; two score buffers S0 [256,320), S1 [320,384)
// fp32 (S0 holds even tiles, S1 odd tiles); Q [384,512) bf16 pairs (this CTA's 256 latent
// columns).  The 32 rope columns of Q sit in shared memory, where the rope MMAs read them.
//
// Handshakes with the peer CTA: partial scores of tile g go into the peer's exchange slot
// g&1 (st.async, completing on the peer's x_full[g&1]); the peer's P(g) then overwrites
// that slot, and the P.V MMAs that read it arrive, through a multicast commit, on the
// pushing side's x_empty[g&1]: only then may the scores of tile g+2 be pushed.
#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <mutex>

#include "mla_device.cuh"
#include "mla_ptx.cuh"
#include "mla_tmap.cuh"

namespace mla {
#ifdef MLA_FAULT_INJECTION
// Test builds only (never compiled into the shipped library): the producer of CTA
// g_drop_cta leaves tile g_drop_tile of its schedule unloaded, so that the waits on that
// tile run out and the kernel takes its abort path.
__device__ int g_drop_cta = -1;
__device__ int g_drop_tile = -1;
#endif
namespace tc {

constexpr int kThreads = 512;
constexpr int kStages = 4;
constexpr int kTileN = 64;                      // tokens per tile
constexpr int kLatBox = kTileN * 128;           // 64 rows x 64 bf16 (8 KB)
constexpr int kRopeBox = kTileN * 64;           // 64 rows x 32 bf16 (4 KB)
constexpr int kStageBytes = 4 * kLatBox + kRopeBox;  // 36 KB
// Partial scores cross the cluster as 24-bit floats (fp32 cut to 15 mantissa bits,
// relative error < 2^-15): 4 values in 3 words; one row's 64 values = 12 groups of 16
// bytes, stored [group][row] so that a warp's accesses are contiguous.
constexpr int kXGroups = 12;
constexpr int kXBytes = kXGroups * 128 * 16;    // 24 KB per slot
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 0, kTmemS = 256, kTmemQ = 384;  // S buffers at kTmemS + 64 * (g & 1)
constexpr int kQRopeBytes = 128 * 64;  // Q rope: 128 rows x 32 bf16, K-major, 64-byte swizzle
// Raw bytes of quantized tiles sit in the tail of a stage and are decoded in place:
constexpr int kRawFp8 = kStageBytes - kTileN * 288;    // FP8: 256 latent + 32 rope bytes per row
constexpr int kRawFp8Rope = kRawFp8 + kTileN * 256;
constexpr int kRawFp4 = kStageBytes - kTileN * 324;    // NVFP4: whole pages (288 data + 36 scale B per token)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;       // log2 units: P stays below 2^8
// Work items reach the roles through a ring in shared memory written by the item warp; a
// slot is free again once every reader took it: the producer warp, the two MMA issuers,
// the 4 sender warps and the 8 softmax warps.
constexpr int kItemRing = 16;
// Quantized caches: the senders publish each item's q row exponents through a ring of this
// many slots.  The senders load item k's q only after every score MMA of item k-1 completed,
// and the score MMA of a tile waits until its buffer's softmax warpgroup read the scores
// two tiles earlier, so when item k's exponents are written both softmax warpgroups have
// started item k-4 at least (they pass each other only at an item's epilogue): the slot of
// item k-4 has been read.
constexpr int kQExpRing = 4;
constexpr uint32_t kItemReaders = 15;
// All query rows are asked into L2 at the start (each CTA a share) when they total at most
// this many bytes; otherwise each item's rows are asked for one item ahead.
constexpr size_t kQPrefetchBytes = 64u << 20;

// warp roles
constexpr int kWarpProducer = 0, kWarpMma = 1, kWarpMmaPv = 2, kWarpItems = 3, kWarpSender0 = 4, kWarpSoftmax0 = 8;
constexpr int kSenderThreads = 128;   // warps 4..7
constexpr int kWgThreads = 128;       // one softmax warpgroup: warps 8..11, 12..15
constexpr int kSoftmaxThreads = 256;
// Registers per thread: the launch gives every thread kLaunchRegs; the control warpgroup
// (warps 0..3) drops to ctrl, the sender warpgroup to sender, and the two softmax
// warpgroups rise to softmax.  The sum must not exceed 512 * kLaunchRegs (65,536); the split
// follows each cache format's register needs (FP8 tiles are decoded by the senders, NVFP4
// tiles by the softmax warpgroups) and is one for which ptxas spills nothing.
constexpr uint32_t kLaunchRegs = 128;
template <int KV>
struct RegSplit;
template <>
struct RegSplit<MLA_KV_BF16> {
  static constexpr uint32_t ctrl = 88, sender = 120, softmax = 152;
};
template <>
struct RegSplit<MLA_KV_FP8_E4M3> {
  static constexpr uint32_t ctrl = 88, sender = 128, softmax = 144;
};
template <>
struct RegSplit<MLA_KV_NVFP4> {
  static constexpr uint32_t ctrl = 88, sender = 128, softmax = 144;
};
template <int KV>
constexpr bool reg_split_fits() {
  return 128 * RegSplit<KV>::ctrl + 128 * RegSplit<KV>::sender + 256 * RegSplit<KV>::softmax <= 512 * kLaunchRegs;
}
static_assert(reg_split_fits<MLA_KV_BF16>() && reg_split_fits<MLA_KV_FP8_E4M3>() && reg_split_fits<MLA_KV_NVFP4>(),
              "register split exceeds the launch budget");
// Moves this warpgroup's per-thread register budget from the launch value to N.
template <uint32_t N>
__device__ __forceinline__ void regs_to() {
  if constexpr (N < kLaunchRegs) ptx::regs_dec<N>();
  else if constexpr (N > kLaunchRegs) ptx::regs_inc<N>();
}

// Geometry of one 64-token tile of a work item.
struct TileInfo {
  int page[2];       // physical pages (ps=64: page[0] only)
  int npages;        // pages that hold any visible position
  bool page_ok[2];
  uint64_t rowmask;  // bit r: row r is a real, visible position
};

struct Bars {
  uint64_t kv_full[kStages];   // TMA bytes landed
  uint64_t kv_ready[kStages];  // tile prepared for the MMAs (quantized: decoded by a softmax warpgroup, every tile;
                               // bf16: masked rows zeroed by the producer warp, those tiles only)
  uint64_t kv_empty[kStages];  // P.V of the tile completed: stage reusable
  uint64_t s_full[2];          // S MMAs of a buffer completed
  uint64_t s_free[2];          // the buffer's softmax warpgroup (and the senders, when they send) read its S
  uint64_t p_full[2];          // P written to the exchange slot (and O rescaled)
  uint64_t o_done[4];          // P.V of tile g completed (barrier g & 3)
  uint64_t q_ready;            // Q of the next item in TMEM / shared memory
  uint64_t q_free;             // every score MMA of an item completed: its Q may be replaced
  uint64_t o_free;             // epilogue read O
  uint64_t x_full[2];          // the peer's partial scores landed in my exchange slot (tx count)
  uint64_t x_empty[2];         // the peer's P.V read its slot: I may push the next scores into it
  uint64_t ep;                 // both softmax warpgroups published their (max, sum) of an item
  uint64_t qs_ready[kQExpRing];  // quantized caches: the senders wrote an item's q row exponents
  uint64_t mma_final;          // every score MMA of this CTA completed
  uint64_t mma_final_pv;       // every P.V MMA of this CTA completed
  uint64_t item_full[kItemRing];   // ring slot holds the next work item
  uint64_t item_empty[kItemRing];  // every reader took the slot's item
};

struct Smem {
  uint8_t stage[kStages][kStageBytes];
  // [slot][16-byte group][row]: the peer's partial scores of a tile, then (first 16 KB,
  // 128 rows x 128 bytes, 128-byte swizzle) that tile's P, read by the P.V MMAs
  uint4 xbuf[2][kXGroups][128];
  // epilogue staging, per softmax warp: one 16-column chunk of its 32 rows as two 16-row
  // boxes (fp32: 64-byte rows, 64-byte swizzle; bf16: 32-byte rows, 32-byte swizzle)
  uint8_t ostage[8][2048];
  uint8_t q_rope[kQRopeBytes];
  Bars bars;
  union {
    unsigned long long mchain[128];  // alternate tiles, per row: (tile index + 1) << 32 | reference max bits
    float mx[2][2][128];             // both warpgroups per tile: [tile & 1][warpgroup][row] half-row maxima
  };
  int4 items[kItemRing];           // work items {u, tok_lo, tok_hi, slot}; tok_hi < 0 ends the list
  int items_min[kItemRing];        // the item's unit's first attended position (sliding window)
  float ep_m[2][2][128];           // [item parity][warpgroup][row] reference max
  float ep_l[2][2][128];           // [item parity][warpgroup][row] row sum relative to it
  int8_t qexp[kQExpRing][128];     // quantized caches: [item % ring][row] exponent e of the item's q row
  unsigned long long tmask[kStages];  // rows of the staged tile that are real, visible positions
  uint32_t tmem_base;
  int abort_flag;
  unsigned status;  // this CTA's status bits
  WorkerStart wstart;  // this worker's place in the schedule (the full plan is built in stage 0)
};
static_assert(sizeof(PlanSmem) <= kStageBytes, "plan scratch must fit one cache stage");
static_assert(kXBytes % 1024 == 0 && (kStages * kStageBytes) % 1024 == 0, "P tiles need 1024-byte alignment");

__device__ __forceinline__ Smem& smem_ref(uint8_t* raw) {
  uintptr_t a = reinterpret_cast<uintptr_t>(raw);
  a = (a + 1023) & ~uintptr_t(1023);
  return *reinterpret_cast<Smem*>(a);
}

// (page_size is 32 or 64: one or two pages per tile)
__device__ __forceinline__ TileInfo tile_info(const DecodeParams& p, int b, int t0, int tok_hi, int tok_min) {
  TileInfo ti;
  const bool two = p.page_size == 32;
  const int shift = two ? 5 : 6;
  const int* row = p.block_table + (size_t)b * p.max_pages;
  ti.npages = 0;
  ti.rowmask = 0;
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    ti.page[j] = -1;
    ti.page_ok[j] = false;
    const int tj = t0 + (j << shift);
    if ((j == 0 || two) && tj < tok_hi) {
      const int pg = __ldg(row + (tj >> shift));
      ti.page[j] = pg;
      ti.page_ok[j] = pg >= 0 && pg < p.num_pages;
      ti.npages = j + 1;
      const int rows = min(p.page_size, tok_hi - tj);
      if (ti.page_ok[j]) ti.rowmask |= (rows >= 64 ? ~0ull : ((1ull << rows) - 1)) << (j << shift);
    }
  }
  // rows before the sliding window's first position
  if (tok_min > t0) ti.rowmask &= tok_min - t0 >= 64 ? 0ull : ~((1ull << (tok_min - t0)) - 1);
  return ti;
}
__device__ __forceinline__ bool tile_needs_fixup(const TileInfo& ti) { return ti.rowmask != ~0ull; }

// Quantized caches multiply in f16, so each (item, head) row of q is converted from bf16 to
// f16 as q * 2^-e, e chosen per row and per CTA from the row's largest magnitude over the
// CTA's 288 columns: e = 0 while that maximum lies in [2^-8, 2^15) (the usual range: the
// conversion is then the plain one), else the power of two that brings it into
// [2^14, 2^15).  Multiplying by a power of two is exact, so every value within 2^-29 of
// the row's maximum converts exactly and none overflows; the partial scores, computed on
// the scaled row, are multiplied back by 2^e in fp32 (exact) before the two CTAs' halves
// are added.
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t v, float mul) {
  return ptx::pack_f16x2(__uint_as_float(v << 16) * mul, __uint_as_float(v & 0xFFFF0000u) * mul);
}
// Largest bf16 magnitude (as bits) of the two halves of v, folded into m.
__device__ __forceinline__ uint32_t bf16x2_absmax_bits(uint32_t v, uint32_t m) {
  return max(m, max(v & 0x7FFFu, (v >> 16) & 0x7FFFu));
}
// The row exponent e of a row whose largest magnitude has bf16 bits m (non-finite rows: 0).
__device__ __forceinline__ int q_row_exponent(uint32_t m) {
  if (m == 0u || m >= 0x7F80u) return 0;
  const int E = (m < 0x80u) ? -127 : (int)(m >> 7) - 127;  // floor(log2 max); subnormals below 2^-126
  if (E >= -8 && E <= 14) return 0;
  return min(113, max(-100, E - 14));
}
// 2^k as a float, k in [-126, 127].
__device__ __forceinline__ float pow2f(int k) { return __uint_as_float((uint32_t)(k + 127) << 23); }

// Four fp32 bit patterns -> three words holding their top 24 bits in value order: w0 = the
// upper three bytes of a and the second byte of b, w1 = b's top two bytes and c's second and
// third, w2 = c's top byte and the upper three of d, so that each word draws on two values
// (one byte permute each).  The receiver rebuilds each value with one permute (d is w2
// itself), filling the dropped low byte with another byte of the packet: the value it gets
// differs from the sent one by less than 2^-15 relative.
__device__ __forceinline__ void pack24x4(uint32_t a, uint32_t b, uint32_t c, uint32_t d, uint32_t& w0, uint32_t& w1,
                                         uint32_t& w2) {
  w0 = __byte_perm(a, b, 0x5321);
  w1 = __byte_perm(b, c, 0x6532);
  w2 = __byte_perm(c, d, 0x7653);
}
__device__ __forceinline__ void unpack24x4(uint32_t w0, uint32_t w1, uint32_t w2, float& a, float& b, float& c,
                                           float& d) {
  a = __uint_as_float(__byte_perm(w0, w0, 0x2103));
  b = __uint_as_float(__byte_perm(w0, w1, 0x5436));
  c = __uint_as_float(__byte_perm(w1, w2, 0x4325));
  d = __uint_as_float(w2);
}

// Waits for this thread's tensor-memory loads; r's registers count as written by the wait, so
// that no use of a load's result can be scheduled before it.
__device__ __forceinline__ void tmem_ld_wait_regs(uint32_t (&r)[16]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                 "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15])
               :
               : "memory");
}

// Bounded spin until this row's reference-max chain holds tile `g`'s predecessor's entry.
__device__ __forceinline__ bool chain_wait(const unsigned long long* slot, unsigned g, unsigned long long& v,
                                           volatile int* abort_flag) {
  const volatile unsigned long long* vs = slot;
  v = *vs;
  if ((unsigned)(v >> 32) == g) return true;
  const uint64_t t0 = ptx::globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    v = *vs;
    if ((unsigned)(v >> 32) == g) return true;
    if ((it & 255u) == 0) {
      if (*abort_flag) return false;
      if (ptx::globaltimer_ns() - t0 > ptx::kWaitLimitNs) {
        *abort_flag = 1;
        return false;
      }
    }
  }
}

// Takes work item k from the ring (every reader takes every item, in order): waits for it,
// copies it and frees the slot.  Called by a whole warp (one arrive, after all lanes copied)
// or by a single thread.  Returns 1 for an item, 0 at the end of the list, -1 on abort.
__device__ __forceinline__ int item_take(const int4* ring, const int* ring_min, uint32_t b_full, uint32_t b_empty,
                                         int k, volatile int* abort_flag, WorkItem& it, bool whole_warp) {
  const int s = k % kItemRing;
  if (!ptx::mbar_wait(b_full + 8 * s, (uint32_t)(k / kItemRing) & 1u, abort_flag)) return -1;
  const int4 v = ring[s];
  const int tmin = ring_min[s];
  if (whole_warp) __syncwarp();
  if (!whole_warp || (threadIdx.x & 31) == 0) ptx::mbar_arrive(b_empty + 8 * s);
  it = WorkItem{v.x, v.y, v.z, v.w, tmin};
  return v.z >= 0 ? 1 : 0;
}

// Quantized caches: decodes the raw FP8 / NVFP4 bytes of landed tile k in place into f16, in
// the swizzled layouts the score and P.V MMAs read (rows that are not visible become zeros),
// then releases the tile to the score MMAs.  Called by NT threads (128: one warpgroup, 256:
// both softmax warpgroups; tq = 0..NT-1: row tq / (NT / 64), part tq % (NT / 64) of the row's
// 36 chunks of 8 values); `bar_id` is those threads' named barrier, which separates every
// read of raw bytes from the in-place writes.
template <int KV, int NT>
__device__ __forceinline__ bool prepare_tile(Smem& S, const DecodeParams& p, int k, int tq, uint32_t cr,
                                             uint32_t b_kv_full, uint32_t b_kv_ready, uint32_t bar_id,
                                             volatile int* abort_flag) {
  constexpr int kParts = NT / kTileN, kCh = 36 / kParts;  // threads per row, chunks per thread
  static_assert(kParts * kTileN == NT && kCh * kParts == 36, "thread count must split the tile's rows evenly");
  const int st = k % kStages;
  if (!ptx::mbar_wait(b_kv_full + 8 * st, (k / kStages) & 1, abort_flag)) return false;
  const int pr = tq / kParts, phf = tq % kParts;
  uint8_t* base = S.stage[st];
  const bool valid = (S.tmask[st] >> pr) & 1ull;
  uint32_t raw[kCh][2];
  if (valid) {
#pragma unroll
    for (int i = 0; i < kCh; ++i) {
      const int c = kCh * phf + i;
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
  ptx::named_bar_sync(bar_id, NT);  // every raw byte of the tile is in registers
#pragma unroll
  for (int i = 0; i < kCh; ++i) {
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
    // chunk c (8 values) of row pr: latent chunks in the 128-byte swizzle of their 64-column
    // box, rope chunks in the 64-byte swizzle
    const int c = kCh * phf + i;
    *reinterpret_cast<uint4*>(c < 32 ? base + (c >> 3) * kLatBox + pr * 128 + (((c & 7) ^ (pr & 7)) * 16)
                                     : base + 4 * kLatBox + pr * 64 + ((((c - 32) ^ ((pr >> 1) & 3))) * 16)) = o;
  }
  ptx::fence_proxy_async_smem();
  ptx::mbar_arrive(b_kv_ready + 8 * st);
  return true;
}
// How the softmax warpgroups share the tiles, who decodes a quantized cache and who pushes a
// tile's partial scores to the peer CTA (each choice measured on one box against the others):
//   bf16   both warpgroups take every tile, 32 columns each (each tile's softmax, which sits
//          on the cycle slot -> peer's push -> softmax -> P.V -> slot, then takes about half
//          as long as one warpgroup taking all 64 columns of alternate tiles: 71.7 -> 67.6 us
//          on 32 x 4096 tokens); the senders push.
//   FP8    alternate tiles, all 64 columns: the senders decode every tile as it lands, and
//          each softmax warpgroup pushes its own tile's scores, so that a push never waits
//          behind a decode or behind the other tile's softmax (417 us on 128 x 8192 tokens,
//          against 500-614 us for the other arrangements).
//   NVFP4  both warpgroups take every tile and decode the tiles together, two ahead of the
//          one whose softmax runs (its heavier decoding would hold the senders' pushes back);
//          the senders push.
template <int KV>
constexpr bool half_tiles() { return KV != MLA_KV_FP8_E4M3; }
template <int KV>
constexpr bool decode_in_softmax() { return KV == MLA_KV_NVFP4; }
template <int KV>
constexpr bool decode_in_senders() { return KV == MLA_KV_FP8_E4M3; }
template <int KV>
constexpr bool send_in_softmax() { return KV == MLA_KV_FP8_E4M3; }

// KV: cache format (MLA_KV_BF16 / MLA_KV_FP8_E4M3 / MLA_KV_NVFP4).  The MMAs run in bf16 for a
// bf16 cache and in f16 for the quantized ones (E4M3 and E2M1 x E4M3 are exact in f16).
template <int KV>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
mla_decode_tc_kernel(const __grid_constant__ CUtensorMap tm_lat, const __grid_constant__ CUtensorMap tm_rope,
                     const __grid_constant__ CUtensorMap tm_out, const DecodeParams p) {
  extern __shared__ uint8_t smem_raw[];
  Smem& S = smem_ref(smem_raw);
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const uint32_t cr = ptx::cluster_ctarank();  // 0: latent [0,256) + rope [0,32); 1: the other halves
  const uint32_t peer = cr ^ 1u;
  const int worker = blockIdx.x >> 1;
  volatile int* abort_flag = &S.abort_flag;

  asm volatile("griddepcontrol.launch_dependents;");
  const uint32_t b_kv_full = ptx::smem_u32(&S.bars.kv_full[0]);
  const uint32_t b_kv_ready = ptx::smem_u32(&S.bars.kv_ready[0]);
  const uint32_t b_kv_empty = ptx::smem_u32(&S.bars.kv_empty[0]);
  const uint32_t b_s_full = ptx::smem_u32(&S.bars.s_full[0]), b_s_free = ptx::smem_u32(&S.bars.s_free[0]);
  const uint32_t b_p_full = ptx::smem_u32(&S.bars.p_full[0]), b_o_done = ptx::smem_u32(&S.bars.o_done[0]);
  const uint32_t b_q_ready = ptx::smem_u32(&S.bars.q_ready), b_o_free = ptx::smem_u32(&S.bars.o_free);
  const uint32_t b_q_free = ptx::smem_u32(&S.bars.q_free);
  const uint32_t b_x_full = ptx::smem_u32(&S.bars.x_full[0]), b_x_empty = ptx::smem_u32(&S.bars.x_empty[0]);
  const uint32_t b_mma_final = ptx::smem_u32(&S.bars.mma_final);
  const uint32_t b_mma_final_pv = ptx::smem_u32(&S.bars.mma_final_pv);
  const uint32_t b_ep = ptx::smem_u32(&S.bars.ep);
  const uint32_t b_qs_ready = ptx::smem_u32(&S.bars.qs_ready[0]);
  const uint32_t b_item_full = ptx::smem_u32(&S.bars.item_full[0]), b_item_empty = ptx::smem_u32(&S.bars.item_empty[0]);

  // Set-up that does not depend on the schedule, ahead of it: barriers, tensor memory, the
  // tensor maps, and an L2 prefetch of this CTA's share of the block table (the first tiles'
  // page numbers are then read from L2 once the schedule is known).
  if (tid == 0) {
    S.status = 0u;
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(b_kv_full + 8 * s, 1);
      ptx::mbar_init(b_kv_ready + 8 * s, KV == MLA_KV_BF16 ? 1 : decode_in_softmax<KV>() ? kSoftmaxThreads : kSenderThreads);
      ptx::mbar_init(b_kv_empty + 8 * s, 1);
    }
    for (int s = 0; s < 2; ++s) {
      ptx::mbar_init(b_s_full + 8 * s, 1);
      ptx::mbar_init(b_s_free + 8 * s, (half_tiles<KV>() ? kSoftmaxThreads : kWgThreads) + (send_in_softmax<KV>() ? 0 : kSenderThreads));
      ptx::mbar_init(b_p_full + 8 * s, half_tiles<KV>() ? kSoftmaxThreads : kWgThreads);
      ptx::mbar_init(b_x_full + 8 * s, 1);   // one local arrive (expect_tx) + 24 KB of peer bytes
      ptx::mbar_init(b_x_empty + 8 * s, 1);  // one arrive per use, from the peer's P.V commit
    }
    for (int s = 0; s < 4; ++s) ptx::mbar_init(b_o_done + 8 * s, 1);
    ptx::mbar_init(b_q_ready, kSenderThreads);
    for (int s = 0; s < kQExpRing; ++s) ptx::mbar_init(b_qs_ready + 8 * s, kSenderThreads);
    ptx::mbar_init(b_q_free, 1);  // one commit per item, after its last score MMAs
    ptx::mbar_init(b_o_free, kSoftmaxThreads);
    ptx::mbar_init(b_ep, kSoftmaxThreads);
    ptx::mbar_init(b_mma_final, 1);
    ptx::mbar_init(b_mma_final_pv, 1);
    for (int s = 0; s < kItemRing; ++s) {
      ptx::mbar_init(b_item_full + 8 * s, 1);
      ptx::mbar_init(b_item_empty + 8 * s, kItemReaders);
    }
    S.abort_flag = 0;
    // each exchange slot's first use is armed here, every later one as soon as the
    // previous use has completed
    for (int s = 0; s < 2; ++s) ptx::mbar_arrive_expect_tx(b_x_full + 8 * s, kXBytes);
    ptx::fence_mbar_init_cluster();
  }
  if (!half_tiles<KV>() && tid < 128) S.mchain[tid] = 0ull;
  if (warp == kWarpMma) {
    ptx::tmem_alloc(ptx::smem_u32(&S.tmem_base), kTmemCols);
    ptx::tmem_relinquish();
  }
  if (KV != MLA_KV_NVFP4 && warp == kWarpProducer && lane == 0) {
    ptx::prefetch_tmap(&tm_lat);
    ptx::prefetch_tmap(&tm_rope);
  }
  // this CTA's share of an array, on its way to L2
  auto prefetch_share = [&](const void* base, size_t bytes) {
    bytes &= ~(size_t)15;
    const size_t share = (((bytes + gridDim.x - 1) / gridDim.x) + 15) & ~(size_t)15;
    const size_t lo = (size_t)blockIdx.x * share;
    if (lo < bytes) ptx::bulk_prefetch_l2(reinterpret_cast<const uint8_t*>(base) + lo, (uint32_t)min(share, bytes - lo));
  };
  const size_t q_rows = (size_t)p.B * p.q_len * p.H;
  const bool q_share = q_rows * (kLatent + kRope) * 2 <= kQPrefetchBytes;
  if (warp == kWarpMmaPv && lane == 0) prefetch_share(p.block_table, (size_t)p.B * p.max_pages * 4);
  if (warp == kWarpItems && lane == 0 && q_share) {
    prefetch_share(p.q_nope, q_rows * kLatent * 2);
    prefetch_share(p.q_pe, q_rows * kRope * 2);
  }
  // From here on the peer may address this CTA's barriers and exchange buffers.
  ptx::cluster_arrive();
  // One warp evaluates the schedule, in the first cache stage (idle until the first tile is
  // loaded, which happens after this), and finds this worker's start; the other warps go on
  // to the barrier below.
  if (warp == kWarpProducer) {
    __syncwarp();
    PlanSmem& plan = *reinterpret_cast<PlanSmem*>(S.stage[0]);
    compute_plan_warp(p, plan, &S.status, blockIdx.x == 0);
    if (lane == 0) {
      S.wstart = worker_start(p, plan, worker);
      // the first item's query rows, on their way to L2 before the roles start
      if (S.wstart.busy && cr == 0 && !q_share) {
        ptx::bulk_prefetch_l2(p.q_nope + (size_t)S.wstart.u0 * p.H * kLatent, (uint32_t)p.H * kLatent * 2);
        ptx::bulk_prefetch_l2(p.q_pe + (size_t)S.wstart.u0 * p.H * kRope, (uint32_t)p.H * kRope * 2);
      }
      // the block-table entries of the first tile, into L1 for the producer
      const WorkItem& f = S.wstart.first;
      if (S.wstart.busy) {
        const int* row = p.block_table + (size_t)(f.u / p.q_len) * p.max_pages + (f.tok_lo >> (p.page_size == 32 ? 5 : 6));
        ptx::prefetch_l1(row);
        if (p.page_size == 32 && f.tok_lo + 32 < f.tok_hi) ptx::prefetch_l1(row + 1);
      }
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::cluster_wait();  // the peer's barriers exist before any remote arrive
  ptx::tc_fence_after();
  const WorkerStart& wst = S.wstart;  // read from shared memory where needed
  const int n_tiles_total = wst.N;
  const uint32_t tmem = S.tmem_base;
  if (warp == kWarpProducer) {
    regs_to<RegSplit<KV>::ctrl>();
    // ------------------------------------------------------------------ TMA producer
    // Lane 0 issues the loads.  For a bf16 tile with masked rows (ragged tail, invalid page)
    // the whole warp waits for it to land and zeroes those rows, so that garbage, even NaN,
    // cannot reach P.V, then releases it to the score MMAs (kv_ready).
    const bool leader = lane == 0;
    const uint64_t pol_stream = ptx::l2_policy_evict_first();  // cache rows are read once
    const uint32_t page_bytes = KV == MLA_KV_BF16 ? (uint32_t)p.page_size * (4 * 128 + 64)
                              : KV == MLA_KV_FP8_E4M3 ? (uint32_t)p.page_size * 288
                                                      : (uint32_t)p.page_size * 324;
    int g = 0;
    bool dead = false;
    WorkItem it;
    // The first item comes from the schedule evaluated at start-up (its first tile's
    // block-table entries already asked into L1); its ring entry is taken together with the
    // second.
    const bool first_known = wst.busy != 0;
    for (int k_item = 0;; ++k_item) {
      if (k_item == 0 && first_known) {
        it = wst.first;
      } else {
        if (k_item == 1 && first_known &&
            item_take(S.items, S.items_min, b_item_full, b_item_empty, 0, abort_flag, it, true) < 0) {
          dead = true;
          break;
        }
        const int got = item_take(S.items, S.items_min, b_item_full, b_item_empty, k_item, abort_flag, it, true);
        if (got <= 0) {
          dead = got < 0;
          break;
        }
      }
      const int b = it.u / p.q_len;
      TileInfo ti_next = tile_info(p, b, it.tok_lo, it.tok_hi, it.tok_min);
      for (int t0 = it.tok_lo; t0 < it.tok_hi; t0 += kTileN, ++g) {
        // this tile's block-table entries were read one tile earlier, the next tile's are
        // read now, before waiting for the stage
        const TileInfo ti = ti_next;
        if (t0 + kTileN < it.tok_hi) ti_next = tile_info(p, b, t0 + kTileN, it.tok_hi, it.tok_min);
        const int st = g % kStages;
        if (g >= kStages && !ptx::mbar_wait(b_kv_empty + 8 * st, ((g / kStages) - 1) & 1, abort_flag)) {
          dead = true;
          break;
        }
#ifdef MLA_FAULT_INJECTION
        if (blockIdx.x == (unsigned)g_drop_cta && g == g_drop_tile) {
          if (leader) S.tmask[st] = ti.rowmask;
          continue;  // neither the expected byte count nor the loads: kv_full never completes
        }
#endif
        if (leader) {
          uint32_t bytes = 0;
          for (int j = 0; j < ti.npages; ++j) {
            if (ti.page_ok[j]) bytes += page_bytes;
            else set_status(&S.status, MLA_STATUS_PAGE_OUT_OF_RANGE);
          }
          S.tmask[st] = ti.rowmask;  // published by the arrive below
          ptx::mbar_arrive_expect_tx(b_kv_full + 8 * st, bytes);
          const uint32_t dst = ptx::smem_u32(S.stage[st]);
          for (int j = 0; j < ti.npages; ++j) {
            if (!ti.page_ok[j]) continue;
            const int y = ti.page[j] * p.page_size;
            const int roff = j * p.page_size;
            if (KV == MLA_KV_BF16) {
#pragma unroll
              for (int k = 0; k < 4; ++k)
                ptx::tma_load_2d_hint(dst + k * kLatBox + roff * 128, &tm_lat, 256 * (int)cr + 64 * k, y,
                                      b_kv_full + 8 * st, pol_stream);
              ptx::tma_load_2d_hint(dst + 4 * kLatBox + roff * 64, &tm_rope, 512 + 32 * (int)cr, y, b_kv_full + 8 * st,
                                    pol_stream);
            } else if (KV == MLA_KV_FP8_E4M3) {
              ptx::tma_load_2d_hint(dst + kRawFp8 + roff * 256, &tm_lat, 256 * (int)cr, y, b_kv_full + 8 * st, pol_stream);
              ptx::tma_load_2d_hint(dst + kRawFp8Rope + roff * 32, &tm_rope, 512 + 32 * (int)cr, y, b_kv_full + 8 * st,
                                    pol_stream);
            } else {
              ptx::bulk_load_hint(dst + kRawFp4 + j * page_bytes, p.cache + (size_t)ti.page[j] * page_bytes, page_bytes,
                                  b_kv_full + 8 * st, pol_stream);
            }
          }
        }
        if (KV == MLA_KV_BF16 && ti.rowmask != ~0ull) {
          if (!ptx::mbar_wait(b_kv_full + 8 * st, (g / kStages) & 1, abort_flag)) {
            dead = true;
            break;
          }
          // a masked row: 4 latent boxes x 128 bytes + 64 rope bytes, zeroed whole
          uint8_t* base = S.stage[st];
#pragma unroll 1
          for (int r = 0; r < kTileN; ++r) {
            if ((ti.rowmask >> r) & 1ull) continue;
            for (int c = lane; c < 36; c += 32)
              *reinterpret_cast<uint4*>(c < 32 ? base + (c >> 3) * kLatBox + r * 128 + (c & 7) * 16
                                               : base + 4 * kLatBox + r * 64 + (c - 32) * 16) = make_uint4(0u, 0u, 0u, 0u);
          }
          ptx::fence_proxy_async_smem();
          __syncwarp();
          if (leader) ptx::mbar_arrive(b_kv_ready + 8 * st);
        }
      }
    }
    // loads still in flight after an abort must land before the CTA exits
    if (leader) {
      for (int k = 1; k <= kStages && g - k >= 0; ++k) {
        const int gg = g - k;
        ptx::mbar_drain(b_kv_full + 8 * (gg % kStages), (gg / kStages) & 1);
      }
    }
  } else if (warp == kWarpMma) {
    // ------------------------------------------------------------------ score MMA issuer
    // Issuing a chain of MMAs blocks this thread while the tensor pipe takes them in, so the
    // score MMAs and the P.V MMAs have issuers of their own: a P.V whose P is ready never
    // waits behind the issue of the next tile's scores.
    regs_to<RegSplit<KV>::ctrl>();
    if (lane == 0) {
      constexpr uint32_t ab = KV == MLA_KV_BF16 ? 1u : 0u;                 // bf16 / f16 operands
      constexpr uint32_t idesc_s = ptx::idesc_f16(ab, 0, 128, kTileN);  // K-major B (cache rows)
      const uint32_t stage0 = ptx::smem_u32(S.stage[0]);
      // base descriptors of stage 0; stage st adds st * kStageBytes to the address field
      const uint64_t kdesc0 = ptx::umma_desc(stage0, 16, 1024, 2);               // K rows, 128 B swizzle
      const uint64_t rdesc0 = ptx::umma_desc(stage0 + 4 * kLatBox, 16, 512, 4);  // rope rows, 64 B swizzle
      const uint64_t qdesc0 = ptx::umma_desc(ptx::smem_u32(S.q_rope), 16, 512, 4);
      int g = 0, n_item = 0;
      uint32_t fixpar = 0;  // bf16: per-stage phase of kv_ready (it completes on tiles with masked rows only)
      bool dead = false;
      WorkItem it;
      for (int k_item = 0; !dead; ++k_item) {
        if (item_take(S.items, S.items_min, b_item_full, b_item_empty, k_item, abort_flag, it, false) <= 0) break;
        if (!ptx::mbar_wait(b_q_ready, n_item & 1, abort_flag)) break;
        ptx::tc_fence_after();
        const int nt = (it.tok_hi - it.tok_lo + kTileN - 1) / kTileN;
        for (int t = 0; t < nt; ++t, ++g) {
          const int st = g % kStages;
          // buffer g&1 is free once the senders and its softmax warpgroup have read S(g-2)
          // (NVFP4: waited for before the tile's decode, which usually completes later --
          // measured 2 % faster there; the other formats wait for the tile first)
          if (KV == MLA_KV_NVFP4 && g >= 2 &&
              !ptx::mbar_wait(b_s_free + 8 * (g & 1), ((g >> 1) - 1) & 1, abort_flag)) { dead = true; break; }
          if (KV == MLA_KV_BF16) {
            if (!ptx::mbar_wait(b_kv_full + 8 * st, (g / kStages) & 1, abort_flag)) { dead = true; break; }
            if (S.tmask[st] != ~0ull) {
              if (!ptx::mbar_wait(b_kv_ready + 8 * st, (fixpar >> st) & 1u, abort_flag)) { dead = true; break; }
              fixpar ^= 1u << st;
            }
          } else {
            if (!ptx::mbar_wait(b_kv_ready + 8 * st, (g / kStages) & 1, abort_flag)) { dead = true; break; }
          }
          if (KV != MLA_KV_NVFP4 && g >= 2 &&
              !ptx::mbar_wait(b_s_free + 8 * (g & 1), ((g >> 1) - 1) & 1, abort_flag)) { dead = true; break; }
          ptx::tc_fence_after();
          const uint32_t d_s = tmem + kTmemS + 64 * (g & 1);
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
          ptx::mma_commit(b_s_full + 8 * (g & 1));
        }
        if (!dead) ptx::mma_commit(b_q_free);
        ++n_item;
      }
      ptx::mma_commit(b_mma_final);
      ptx::mbar_drain(b_mma_final, 0);
    }
  } else if (warp == kWarpMmaPv) {
    // ------------------------------------------------------------------ P.V MMA issuer
    regs_to<RegSplit<KV>::ctrl>();
    if (lane == 0) {
      constexpr uint32_t ab = KV == MLA_KV_BF16 ? 1u : 0u;
      constexpr uint32_t idesc_o = ptx::idesc_f16(ab, 1, 128, 256);  // MN-major B (V columns)
      const uint64_t vdesc0 = ptx::umma_desc(ptx::smem_u32(S.stage[0]), kLatBox, 1024, 2);        // V, MN-major
      const uint64_t pdesc0 = ptx::umma_desc(ptx::smem_u32(&S.xbuf[0][0][0]), 16, 1024, 2);  // P, K-major
      const uint16_t peer_mask = (uint16_t)(1u << peer);
      int g = 0, n_item = 0;
      bool dead = false;
      WorkItem it;
      for (int k_item = 0; !dead; ++k_item) {
        if (item_take(S.items, S.items_min, b_item_full, b_item_empty, k_item, abort_flag, it, false) <= 0) break;
        const int nt = (it.tok_hi - it.tok_lo + kTileN - 1) / kTileN;
        for (int t = 0; t < nt; ++t, ++g) {
          if (!ptx::mbar_wait(b_p_full + 8 * (g & 1), (g >> 1) & 1, abort_flag)) { dead = true; break; }
          // the item's first P.V overwrites O: the previous item's epilogue must have read it
          if (t == 0 && n_item > 0 && !ptx::mbar_wait(b_o_free, (n_item - 1) & 1, abort_flag)) { dead = true; break; }
          ptx::tc_fence_after();
          const uint64_t vdesc = vdesc0 + (uint64_t)((g % kStages) * (kStageBytes >> 4));
          const uint64_t pdesc = pdesc0 + (uint64_t)((g & 1) * (kXBytes >> 4));
#pragma unroll
          for (int k = 0; k < kTileN / 16; ++k)  // 16 tokens = 2 KB of V rows, 32 B of P rows
            ptx::mma_ss(tmem + kTmemO, pdesc + (uint64_t)(k * 2), vdesc + (uint64_t)(k * (2048 >> 4)), idesc_o,
                        (t == 0 && k == 0) ? 0u : 1u);
          ptx::mma_commit(b_o_done + 8 * (g & 3));
          ptx::mma_commit(b_kv_empty + 8 * (g % kStages));
          ptx::mma_commit_multicast(b_x_empty + 8 * (g & 1), peer_mask);
        }
        ++n_item;
      }
      ptx::mma_commit(b_mma_final_pv);
      ptx::mbar_drain(b_mma_final_pv, 0);
    }
  } else if (warp >= kWarpSender0 && warp < kWarpSoftmax0) {
    // ------------------------------------------------------------------ senders
    regs_to<RegSplit<KV>::sender>();
    const int q = warp & 3;
    const int row = 32 * q + lane;
    const uint32_t lane_off = (uint32_t)(32 * q) << 16;
    const uint32_t t_s0 = tmem + lane_off + kTmemS, t_q = tmem + lane_off + kTmemQ;
    const uint32_t x_peer = ptx::mapa(ptx::smem_u32(&S.xbuf[0][0][0]), peer);
    const uint32_t bx_full_peer = ptx::mapa(b_x_full, peer);
    // Quantized caches: the power of two this thread's row of the current item's q was
    // divided by (1 when unscaled), and whether any row of this warp was scaled.
    float q_sc = 1.f;
    bool q_scaled = false;

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
      if (KV != MLA_KV_BF16 && q_scaled) {  // back to the scale of the unscaled row (exact)
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          r0[j] = __float_as_uint(__uint_as_float(r0[j]) * q_sc);
          r1[j] = __float_as_uint(__uint_as_float(r1[j]) * q_sc);
        }
      }
      const int slot = k & 1, use = k >> 1;
      const uint32_t xp = x_peer + (uint32_t)slot * kXBytes + (uint32_t)row * 16;
      const uint32_t bar = bx_full_peer + 8 * slot;
      if constexpr (KV == MLA_KV_BF16) {
        // the peer's P.V(k-2) has read the slot (its P) before the next scores go in
        if (use >= 1 && !ptx::mbar_wait(b_x_empty + 8 * slot, (use - 1) & 1, abort_flag, true)) return false;
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
      } else {
        // NVFP4 (whose sender budget is the tighter one): all 64 values packed first, which
        // frees the score registers before the wait
        uint32_t pw[4][12];
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          const uint32_t* src = h < 2 ? r0 + 16 * h : r1 + 16 * (h - 2);
#pragma unroll
          for (int j = 0; j < 4; ++j)
            pack24x4(src[4 * j], src[4 * j + 1], src[4 * j + 2], src[4 * j + 3], pw[h][3 * j], pw[h][3 * j + 1],
                     pw[h][3 * j + 2]);
        }
        if (use >= 1 && !ptx::mbar_wait(b_x_empty + 8 * slot, (use - 1) & 1, abort_flag, true)) return false;
#pragma unroll
        for (int h = 0; h < 4; ++h)
#pragma unroll
          for (int j = 0; j < 3; ++j)
            ptx::st_async_v4(xp + (3 * h + j) * 128 * 16, __uint_as_float(pw[h][4 * j]), __uint_as_float(pw[h][4 * j + 1]),
                             __uint_as_float(pw[h][4 * j + 2]), __uint_as_float(pw[h][4 * j + 3]), bar);
      }
      return true;
    };

    // (3) Q of one work item: this row's 256 latent columns -> TMEM, 32 rope columns ->
    // shared memory (64-byte swizzled K-major layout: chunk c of row r sits at chunk
    // position c ^ ((r >> 1) & 3) of the row's 64 bytes).
    auto q_row = [&](const WorkItem& w) -> size_t {
      const int b = w.u / p.q_len, i = w.u % p.q_len;
      return ((size_t)b * p.q_len + i) * p.H + (row < p.H ? row : 0);
    };
    // One pass over the row: q * mul -> TMEM / shared memory; returns the row's largest
    // bf16 magnitude (as bits).
    auto store_q = [&](const uint4* qn, const uint4* qp, bool real, float mul) -> uint32_t {
      uint32_t mx = 0u;
      // 16-byte loads in flight per round: 32 (two TMEM stores) with the wider register
      // budgets, 8 (one store) with the narrowest
      constexpr int kLd = RegSplit<KV>::sender >= 112 ? 16 : 8;
#pragma unroll 1
      for (int part = 0; part < 32 / kLd; ++part) {
        uint4 x[kLd];
#pragma unroll
        for (int k = 0; k < kLd; ++k) x[k] = real ? __ldg(qn + kLd * part + k) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
        for (int c = 0; c < kLd / 8; ++c) {
          uint32_t v[32];
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            v[4 * k] = x[8 * c + k].x;
            v[4 * k + 1] = x[8 * c + k].y;
            v[4 * k + 2] = x[8 * c + k].z;
            v[4 * k + 3] = x[8 * c + k].w;
          }
          if (KV != MLA_KV_BF16) {
#pragma unroll
            for (int k = 0; k < 32; ++k) {
              mx = bf16x2_absmax_bits(v[k], mx);
              v[k] = bf16x2_to_f16x2(v[k], mul);
            }
          }
          ptx::tmem_st32(t_q + (kLd * part + 8 * c) * 4, v);
        }
      }
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint4 x = real ? __ldg(qp + c) : make_uint4(0u, 0u, 0u, 0u);
        if (KV != MLA_KV_BF16) {
          mx = bf16x2_absmax_bits(x.w, bf16x2_absmax_bits(x.z, bf16x2_absmax_bits(x.y, bf16x2_absmax_bits(x.x, mx))));
          x.x = bf16x2_to_f16x2(x.x, mul);
          x.y = bf16x2_to_f16x2(x.y, mul);
          x.z = bf16x2_to_f16x2(x.z, mul);
          x.w = bf16x2_to_f16x2(x.w, mul);
        }
        *reinterpret_cast<uint4*>(S.q_rope + row * 64 + ((c ^ ((row >> 1) & 3)) * 16)) = x;
      }
      return mx;
    };
    // Q of item k: this row's 256 latent columns -> TMEM, 32 rope columns -> shared memory
    // (64-byte swizzled K-major layout: chunk c of row r sits at chunk position c ^ ((r >> 1)
    // & 3) of the row's 64 bytes).  Quantized caches: converted to f16 as they are; a warp
    // holding a row whose maximum falls outside the plain range stores its rows again,
    // scaled, and the exponents go to the softmax warpgroups through the exponent ring.
    auto load_q = [&](const WorkItem& w, int k) {
      const bool real = row < p.H;
      const size_t qrow = q_row(w);
      const uint4* qn = reinterpret_cast<const uint4*>(p.q_nope + qrow * kLatent + 256 * cr);
      const uint4* qp = reinterpret_cast<const uint4*>(p.q_pe + qrow * kRope + 32 * cr);
      const uint32_t mx = store_q(qn, qp, real, 1.f);
      if (KV != MLA_KV_BF16) {
        const int e = q_row_exponent(mx);
        if (mx >= 0x7F80u) set_status(&S.status, MLA_STATUS_Q_RANGE);
        q_scaled = __any_sync(0xffffffffu, e != 0);
        if (q_scaled) {
          ptx::tmem_st_wait();
          store_q(qn, qp, real, pow2f(-e));
        }
        q_sc = pow2f(e);
        S.qexp[k % kQExpRing][row] = (int8_t)e;
        ptx::mbar_arrive(b_qs_ready + 8 * (k % kQExpRing));
      }
      ptx::fence_proxy_async_smem();
      ptx::tmem_st_wait();
      ptx::tc_fence_before();
      ptx::mbar_arrive(b_q_ready);
    };
    if constexpr (send_in_softmax<KV>()) {
      // Per item: its Q once every score MMA of the previous item has completed (they read Q
      // from TMEM; the score issuer commits one q_free phase per item), then, for FP8, each of
      // its tiles decoded as soon as it lands.
      int g = 0;
      bool dead = false;
      WorkItem it;
      const int tq = (warp - kWarpSender0) * 32 + lane;
      // the first item's unit is known from the schedule: its Q loads overlap the item ring's
      // start and the first cache loads
      if (wst.busy) load_q(WorkItem{wst.u0, 0, 0, -1, 0}, 0);
      for (int k_item = 0; !dead; ++k_item) {
        const int got = item_take(S.items, S.items_min, b_item_full, b_item_empty, k_item, abort_flag, it, true);
        if (got <= 0) {
          dead = got < 0;
          break;
        }
        const int nt = (it.tok_hi - it.tok_lo + kTileN - 1) / kTileN;
        if (k_item > 0) {  // the previous item's score MMAs have all completed (one phase per item)
          if (!ptx::mbar_wait(b_q_free, (uint32_t)(k_item - 1) & 1u, abort_flag)) {
            dead = true;
            break;
          }
          ptx::tc_fence_after();
          load_q(it, k_item);
        }
        if (decode_in_senders<KV>()) {
          for (int t = 0; t < nt; ++t)
            if (!prepare_tile<KV, kSenderThreads>(S, p, g + t, tq, cr, b_kv_full, b_kv_ready, 3, abort_flag)) {
              dead = true;
              break;
            }
        }
        g += nt;
      }
    } else {
      // Per tile g: tile g-1's scores are sent (the decode step is skipped: these formats are
      // not decoded by the senders).  An item's Q is loaded once the previous item's last
      // scores have been read out of TMEM.
      int g = 0;
      bool dead = false;
      WorkItem it;
      const int tq = (warp - kWarpSender0) * 32 + lane;
      // the first item's unit is known from the schedule: its Q loads overlap the item ring's
      // start and the first cache loads
      if (wst.busy) load_q(WorkItem{wst.u0, 0, 0, -1, 0}, 0);
      for (int k_item = 0; !dead; ++k_item) {
        const int got = item_take(S.items, S.items_min, b_item_full, b_item_empty, k_item, abort_flag, it, true);
        if (got <= 0) {
          dead = got < 0;
          break;
        }
        // (an abort elsewhere reaches this loop through its bounded waits, which watch the flag)
        for (int t0 = it.tok_lo; t0 < it.tok_hi; t0 += kTileN, ++g) {
          if (decode_in_senders<KV>() && !prepare_tile<KV, kSenderThreads>(S, p, g, tq, cr, b_kv_full, b_kv_ready, 3, abort_flag)) {
            dead = true;
            break;
          }
          if (g > 0 && !send(g - 1)) {
            dead = true;
            break;
          }
          if (t0 == it.tok_lo && g > 0) load_q(it, k_item);
        }
      }
      if (!dead && g > 0 && send(g - 1)) {
        // the peer's last two P.V commits land on this CTA's x_empty: take them before exit
        for (int k = max(0, g - 2); k < g; ++k)
          if (!ptx::mbar_wait(b_x_empty + 8 * (k & 1), (k >> 1) & 1, abort_flag, true)) break;
      }
    }
  } else if (warp >= kWarpSoftmax0) {
    // ------------------------------------------------------------------ softmax + epilogue
    regs_to<RegSplit<KV>::softmax>();
    // kHalf: both warpgroups take every tile, 32 of its 64 columns each; otherwise the two
    // warpgroups take alternate tiles (even / odd), all 64 columns.
    constexpr bool kHalf = half_tiles<KV>();
    constexpr int kCols = kHalf ? 32 : 64;            // tile columns per thread
    constexpr int kGroups = kCols * kXGroups / 64;    // their 16-byte groups in an exchange slot
    constexpr int kStep = kHalf ? 1 : 2;
    static_assert(kHalf || !decode_in_softmax<KV>(), "softmax decoding is written for both warpgroups per tile");
    static_assert(!kHalf || !send_in_softmax<KV>(), "softmax pushes are written for alternate tiles");
    const int sw = warp - kWarpSoftmax0;        // 0..7
    const int wg = sw >> 2;                      // O columns [128 wg, +128) in the epilogue
    const int q = warp & 3;                       // TMEM lane quadrant this warp may access
    const int row = 32 * q + lane;                // head
    const int ts = 128 * wg + row;                // 0..255 over both warpgroups
    const int c0 = kHalf ? 32 * wg : 0;           // this thread's first tile column
    const uint32_t lane_off = (uint32_t)(32 * q) << 16;
    const uint32_t t_s0 = tmem + lane_off + kTmemS + c0;
    const uint32_t t_o = tmem + lane_off + kTmemO;
    const float scale_log2 = p.sm_scale * p.kv_scale * kLog2e;
    // FP8: a warpgroup pushes its tiles' partial scores into the peer's slot g&1 itself
    const uint32_t x_peer = ptx::mapa(ptx::smem_u32(&S.xbuf[0][0][0]), peer) + (uint32_t)row * 16;
    const uint32_t bx_full_peer = ptx::mapa(b_x_full, peer);
    unsigned long long* const chain = &S.mchain[row];

    // P.V completions: o_done[k & 3] completes once per P.V(k), k = j, j + 4, ...  Every P.V
    // up to pv_known is known to be complete, and the waits below are only ever for
    // P.V(k) with k <= pv_known + 4, so the barrier's previous phase (P.V(k-4)) is complete
    // and its next one (P.V(k+4)) cannot complete before this thread moves on: a parity
    // wait never confuses two phases.
    int pv_known = -1;
    auto wait_pv = [&](int k) -> bool {
      if (k <= pv_known) return true;
      if (!ptx::mbar_wait(b_o_done + 8 * (k & 3), (k >> 2) & 1, abort_flag)) return false;
      pv_known = k;
      return true;
    };

    int g = 0, n_item = 0;
    bool dead = false;
    WorkItem it;
    for (int k_item = 0; !dead; ++k_item) {
      if (item_take(S.items, S.items_min, b_item_full, b_item_empty, k_item, abort_flag, it, true) <= 0) break;
      const int b = it.u / p.q_len;
      const int nt = (it.tok_hi - it.tok_lo + kTileN - 1) / kTileN;
      const int g0 = g;
      // the row's reference and this thread's running sum relative to it
      float m_own = -INFINITY, l_own = 0.f;
      int t_idx = kHalf || (g0 & 1) == wg ? 0 : 1;  // this thread's first tile of the item
      // The first item starts with passes through the loop body that have no effect (every
      // wait, arrive and store is skipped): they fetch the body's instructions while the
      // first scores are still being computed, instead of on the first tile's critical path
      // (NVFP4: two passes, whose ends decode the item's first two tiles).
      if (k_item == 0) t_idx -= kHalf ? (decode_in_softmax<KV>() ? 2 : 1) : 2;
      // NVFP4: tiles are decoded two ahead of the one whose softmax is running, by both
      // warpgroups together; an item's first two here (the first item's: at the ends of the
      // instruction-fetch passes)
      if (decode_in_softmax<KV>() && k_item > 0) {
        for (int t = 0; t < nt && t < 2 && !dead; ++t)
          if (!prepare_tile<KV, kSoftmaxThreads>(S, p, g0 + t, ts, cr, b_kv_full, b_kv_ready, 4, abort_flag)) dead = true;
        if (dead) break;
      }
      // quantized caches: the exponent this CTA's half of the item's q row was scaled by
      float q_sc = 1.f;
      bool q_scaled = false;
      if (KV != MLA_KV_BF16) {
        const int qs = k_item % kQExpRing;
        if (!ptx::mbar_wait(b_qs_ready + 8 * qs, (uint32_t)(k_item / kQExpRing) & 1u, abort_flag)) {
          dead = true;
          break;
        }
        const int e = S.qexp[qs][row];
        q_sc = pow2f(e);
        q_scaled = __any_sync(0xffffffffu, e != 0);
      }
      for (; t_idx < nt; t_idx += kStep) {
        const bool real = t_idx >= 0;
        const int gg = g0 + t_idx;
        const int slot = gg & 1;
        // ---- own partial scores
        float s[kCols];
        if (real && !ptx::mbar_wait(b_s_full + 8 * slot, (gg >> 1) & 1, abort_flag)) { dead = true; break; }
        ptx::tc_fence_after();
        {
          uint32_t r[kCols / 32][32];
#pragma unroll
          for (int h = 0; h < kCols / 32; ++h) ptx::tmem_ld32(t_s0 + 64 * slot + 32 * h, r[h]);
          ptx::tmem_ld_wait();
          ptx::tc_fence_before();
          if (real) ptx::mbar_arrive(b_s_free + 8 * slot);
          if (KV != MLA_KV_BF16 && q_scaled) {  // back to the scale of the unscaled row (exact)
#pragma unroll
            for (int k = 0; k < kCols; ++k) r[k >> 5][k & 31] = __float_as_uint(__uint_as_float(r[k >> 5][k & 31]) * q_sc);
          }
#pragma unroll
          for (int k = 0; k < kCols; ++k) s[k] = __uint_as_float(r[k >> 5][k & 31]);
          // ---- FP8: this tile's partial scores -> the peer: 16 values -> 12 packed words ->
          // three 16-byte stores, four times; the slot is free once the peer's P.V of this
          // warpgroup's previous tile has read it
          if (send_in_softmax<KV>() && real) {
            const int use = gg >> 1;
            if (use >= 1 && !ptx::mbar_wait(b_x_empty + 8 * slot, (use - 1) & 1, abort_flag, true)) {
              dead = true;
            } else {
#pragma unroll
              for (int h = 0; h < kCols / 16; ++h) {
                uint32_t pw[12];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                  const uint32_t* v = &r[h >> 1][16 * (h & 1) + 4 * j];
                  pack24x4(v[0], v[1], v[2], v[3], pw[3 * j], pw[3 * j + 1], pw[3 * j + 2]);
                }
#pragma unroll
                for (int j = 0; j < 3; ++j)
                  ptx::st_async_v4(x_peer + (uint32_t)slot * kXBytes + (3 * h + j) * 128 * 16, __uint_as_float(pw[4 * j]),
                                   __uint_as_float(pw[4 * j + 1]), __uint_as_float(pw[4 * j + 2]),
                                   __uint_as_float(pw[4 * j + 3]), bx_full_peer + 8 * slot);
              }
            }
          }
        }
        if (dead) break;
        // ---- the tile's row mask (tail tiles only use it).  The producer published it with the
        // tile's kv_full phase, which completed before this tile's scores (and cannot move on
        // before P(gg) is handed over); it is read before the wait for the peer's scores, which
        // usually takes longer.
        const int st = real ? gg % kStages : 0;
        if (real && !ptx::mbar_wait(b_kv_full + 8 * st, (gg / kStages) & 1, abort_flag)) { dead = true; break; }
        const uint64_t full = kCols == 64 ? ~0ull : (1ull << kCols) - 1;
        const uint64_t mask = (S.tmask[st] >> c0) & full;
        // ---- the peer's partial scores of this thread's columns (then the slot's next use is
        // armed: the peer pushes into it only after this tile's P.V, which every thread here
        // reaches only after this wait)
        if (real && !ptx::mbar_wait(b_x_full + 8 * slot, (gg >> 1) & 1, abort_flag, true)) { dead = true; break; }
        if (real && (kHalf ? ts : row) == 0) ptx::mbar_arrive_expect_tx(b_x_full + 8 * slot, kXBytes);
        // the peer pushed these only after P.V(gg-2) of this CTA had read the slot
        if (real && gg - 2 > pv_known) pv_known = gg - 2;
        uint32_t xw[4 * kGroups];
#pragma unroll
        for (int k = 0; k < kGroups; ++k) {
          const uint4 v = S.xbuf[slot][c0 / 16 * 3 + k][row];
          xw[4 * k] = v.x;
          xw[4 * k + 1] = v.y;
          xw[4 * k + 2] = v.z;
          xw[4 * k + 3] = v.w;
        }
        // alternate tiles: every row of the slot has been read, P may overwrite it
        if constexpr (!kHalf) ptx::named_bar_sync(1 + wg, kWgThreads);
#pragma unroll
        for (int j = 0; j < kCols / 4; ++j) {
          float a, b2, c, d;
          unpack24x4(xw[3 * j], xw[3 * j + 1], xw[3 * j + 2], a, b2, c, d);
          s[4 * j] += a;
          s[4 * j + 1] += b2;
          s[4 * j + 2] += c;
          s[4 * j + 3] += d;
        }
        // ---- mask, row max over this thread's columns (raw units; the scale is positive)
        if (mask != full) {
#pragma unroll
          for (int c = 0; c < kCols; ++c) s[c] = ((mask >> c) & 1ull) ? s[c] : -INFINITY;
        }
        float m4[4] = {s[0], s[1], s[2], s[3]};
#pragma unroll
        for (int c = 4; c < kCols; c += 4) {
          m4[0] = fmaxf(m4[0], s[c]);
          m4[1] = fmaxf(m4[1], s[c + 1]);
          m4[2] = fmaxf(m4[2], s[c + 2]);
          m4[3] = fmaxf(m4[3], s[c + 3]);
        }
        float mt = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
        if constexpr (kHalf) {
          // the two halves of the row meet: every row of the slot has been read (P may
          // overwrite it), and each half takes the other's maximum
          S.mx[slot][wg][row] = mt;
          ptx::named_bar_sync(1, kSoftmaxThreads);
          mt = fmaxf(S.mx[slot][0][row], S.mx[slot][1][row]);
        }
        mt *= scale_log2;
        // ---- reference max: kept from tile to tile, moved when a tile exceeds it by > 8
        // (both halves of a row take the same decision; alternate tiles pass it from one
        // warpgroup to the other through shared memory)
        float m_prev = -INFINITY;
        if constexpr (kHalf) {
          if (t_idx > 0) m_prev = m_own;
        } else if (gg > 0) {
          unsigned long long v;
          if (!chain_wait(chain, (unsigned)gg, v, abort_flag)) { dead = true; break; }
          if (t_idx > 0) m_prev = __uint_as_float((uint32_t)v);
        }
        const bool grow = mt > m_prev + kRescaleThreshold;
        const float m_new = grow ? mt : m_prev;
        if (!kHalf && real)
          *reinterpret_cast<volatile unsigned long long*>(chain) =
              ((unsigned long long)(unsigned)(gg + 1) << 32) | __float_as_uint(m_new);
        // this thread's running sum follows the reference
        if (real && m_new != m_own) {
          if (l_own != 0.f) l_own *= ptx::ex2_approx(m_own - m_new);
          m_own = m_new;
        }
        const float m_use = m_new == -INFINITY ? 0.f : m_new;
        uint32_t pk[kCols / 2];
        float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int c = 0; c < kCols; c += 2) {
          const float p0 = ptx::ex2_approx(fmaf(s[c], scale_log2, -m_use));
          const float p1 = ptx::ex2_approx(fmaf(s[c + 1], scale_log2, -m_use));
          ls[(c >> 1) & 3] += p0 + p1;
          // bf16: round half up on the bit pattern (p is finite and non-negative)
          pk[c / 2] = KV == MLA_KV_BF16 ? __byte_perm(__float_as_uint(p0) + 0x8000u, __float_as_uint(p1) + 0x8000u, 0x7632)
                                        : ptx::pack_f16x2(p0, p1);
        }
        if (real) l_own += (ls[0] + ls[1]) + (ls[2] + ls[3]);
        // P(gg) -> the slot.  Row r, 16-byte chunk c (8 tokens) sits at chunk position
        // c ^ (r & 7) of the row's 128 bytes (the 128-byte swizzle the P.V MMAs read).
        if (real) {
          uint8_t* const prow = reinterpret_cast<uint8_t*>(&S.xbuf[slot][0][0]) + row * 128;
#pragma unroll
          for (int c = 0; c < kCols / 8; ++c)
            *reinterpret_cast<uint4*>(prow + (((c0 / 8 + c) ^ (row & 7)) * 16)) =
                make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
        }
        if (t_idx > 0 && __any_sync(0xffffffffu, grow)) {
          // O moves to the new reference once P.V(gg-1) is done, before P(gg) is handed
          // over: this half's 128 columns, or all 256 (alternate tiles)
          if (!wait_pv(gg - 1)) { dead = true; break; }
          ptx::tc_fence_after();
          const float a = grow ? ptx::ex2_approx(m_prev - m_new) : 1.f;
          constexpr int kOChunks = kHalf ? 8 : 16;
          const uint32_t t_oc = t_o + (kHalf ? 128 * wg : 0);
#pragma unroll 1
          for (int c = 0; c < kOChunks; ++c) {
            uint32_t r[16];
            ptx::tmem_ld16(t_oc + 16 * c, r);
            ptx::tmem_ld_wait();
#pragma unroll
            for (int k = 0; k < 16; ++k) r[k] = __float_as_uint(__uint_as_float(r[k]) * a);
            ptx::tmem_st16(t_oc + 16 * c, r);
          }
          ptx::tmem_st_wait();
        }
        ptx::fence_proxy_async_smem();
        ptx::tc_fence_before();
        if (real) ptx::mbar_arrive(b_p_full + 8 * slot);
        // NVFP4: decode the item's tile two ahead now
        if (decode_in_softmax<KV>() && t_idx + 2 < nt &&
            !prepare_tile<KV, kSoftmaxThreads>(S, p, gg + 2, ts, cr, b_kv_full, b_kv_ready, 4, abort_flag)) {
          dead = true;
          break;
        }
      }
      if (dead) break;
      g = g0 + nt;
      // ---- epilogue: O / l for this warpgroup's 128 columns, and the LSE
      const int par = n_item & 1;
      S.ep_m[par][wg][row] = m_own;
      S.ep_l[par][wg][row] = l_own;
      ptx::mbar_arrive(b_ep);
      if (!wait_pv(g - 1)) { dead = true; break; }
      if (!ptx::mbar_wait(b_ep, par, abort_flag)) { dead = true; break; }
      ptx::tc_fence_after();
      const float ma = S.ep_m[par][0][row], mb = S.ep_m[par][1][row];
      const float la = S.ep_l[par][0][row], lb = S.ep_l[par][1][row];
      float m_fin = fmaxf(ma, mb);
      float l = (la > 0.f ? la * ptx::ex2_approx(ma - m_fin) : 0.f) + (lb > 0.f ? lb * ptx::ex2_approx(mb - m_fin) : 0.f);
      // a head's sink logit (natural-log units of the scaled scores) joins the normaliser of
      // a row written directly; split parts leave it to the combine
      float o_sink = 1.f;  // O is relative to m_fin: weight of the tokens against the new max
      if (it.slot < 0 && p.sinks != nullptr && row < p.H) {
        const float sk = __ldg(p.sinks + row) * kLog2e;
        if (sk > m_fin) {  // the sink becomes the reference (also when no token was seen)
          o_sink = l > 0.f ? ptx::ex2_approx(m_fin - sk) : 0.f;
          l = l * o_sink + 1.f;
          m_fin = sk;
        } else if (sk != -INFINITY) {
          l += ptx::ex2_approx(sk - m_fin);
        }
      }
      const int i = it.u % p.q_len;
      const bool real = row < p.H;
      const float inv = l > 0.f ? 1.f / l : 0.f;
      const float lse_v = l > 0.f ? (m_fin + __log2f(l)) * kLn2 : -INFINITY;
      const float oscale = inv * o_sink * p.kv_scale;
      const size_t orow = ((size_t)b * p.q_len + i) * p.H + (real ? row : 0);
      const bool direct = it.slot < 0, partial = it.slot >= 0 && it.slot < p.slots_cap;
      // A final output leaves through shared memory and TMA tensor stores (16 columns x 16
      // rows per box): a thread's row is not contiguous with its neighbours' in [U, H, 512].
      // A split partial is stored straight from registers, as bf16: in the workspace's
      // octet-major layout a warp's 32 rows of one 8-column octet are 512 contiguous bytes,
      // so the stores need no staging and the next item's P.V can start as soon as O has
      // been read.
      const int row0 = it.u * p.H + 32 * q;
      // The worker's last item (the ring's next entry is the end marker): the cache stages
      // are idle, so each chunk gets a staging buffer of its own there and all stores are in
      // flight together.  Otherwise one 2 KB buffer per warp, reused chunk after chunk.
      bool last = false;
      {
        const int s1 = (k_item + 1) % kItemRing;
        if (ptx::mbar_test(b_item_full + 8 * s1, (uint32_t)((k_item + 1) / kItemRing) & 1u)) last = S.items[s1].z < 0;
      }
      last = __all_sync(0xffffffffu, last);
      uint8_t* const stg0 = last ? S.stage[0] + sw * 16384 : S.ostage[sw];
      uint4* const part = reinterpret_cast<uint4*>(p.ws + partial_o_offset()) + (size_t)it.slot * 64 * p.H + row;
      const uint64_t pol_keep = ptx::l2_policy_evict_last();  // read again by the combine
      // one 16-column chunk of this warpgroup's O, already in registers, scaled and stored
      auto store_chunk = [&](int c, const uint32_t (&r)[16]) {
        if (!direct) {
          if (partial && real) {
            const int oct0 = (256 * (int)cr + 128 * wg + 16 * c) >> 3;
#pragma unroll
            for (int k = 0; k < 2; ++k)
              ptx::st_global_v4u_hint(
                  part + (size_t)(oct0 + k) * p.H,
                  make_uint4(ptx::pack_bf16x2(__uint_as_float(r[8 * k]) * oscale, __uint_as_float(r[8 * k + 1]) * oscale),
                             ptx::pack_bf16x2(__uint_as_float(r[8 * k + 2]) * oscale, __uint_as_float(r[8 * k + 3]) * oscale),
                             ptx::pack_bf16x2(__uint_as_float(r[8 * k + 4]) * oscale, __uint_as_float(r[8 * k + 5]) * oscale),
                             ptx::pack_bf16x2(__uint_as_float(r[8 * k + 6]) * oscale, __uint_as_float(r[8 * k + 7]) * oscale)),
                  pol_keep);
          }
          return;
        }
        uint8_t* const stg = last ? stg0 + 2048 * c : stg0;
        const uint32_t stg_a = ptx::smem_u32(stg);
        if (!last) {  // the previous chunk's stores (this item's or the last item's) have read the buffer
          if (lane == 0) ptx::bulk_wait_read();
          __syncwarp();
        }
        const int br = lane & 15;
        uint8_t* rowp = stg + (lane >> 4) * 512 + br * 32;
#pragma unroll
        for (int k = 0; k < 2; ++k)
          *reinterpret_cast<uint4*>(rowp + ((k ^ ((br >> 2) & 1)) * 16)) =
              make_uint4(ptx::pack_bf16x2(__uint_as_float(r[8 * k + 0]) * oscale, __uint_as_float(r[8 * k + 1]) * oscale),
                         ptx::pack_bf16x2(__uint_as_float(r[8 * k + 2]) * oscale, __uint_as_float(r[8 * k + 3]) * oscale),
                         ptx::pack_bf16x2(__uint_as_float(r[8 * k + 4]) * oscale, __uint_as_float(r[8 * k + 5]) * oscale),
                         ptx::pack_bf16x2(__uint_as_float(r[8 * k + 6]) * oscale, __uint_as_float(r[8 * k + 7]) * oscale));
        ptx::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          const int x = 256 * (int)cr + 128 * wg + 16 * c;
#pragma unroll
          for (int h = 0; h < 2; ++h)
            if (32 * q + 16 * h < p.H) ptx::tma_store_2d(&tm_out, stg_a + h * 512, x, row0 + 16 * h);
          ptx::bulk_commit();
        }
            };
      // Chunks two at a time: chunk c + 1's tensor-memory load is in flight while chunk c is
      // stored (the waits take the loaded registers as operands, so no use of a chunk can be
      // scheduled before its wait).
      uint32_t ra[16], rb[16];
      ptx::tmem_ld16(t_o + 128 * wg, ra);
#pragma unroll 1
      for (int c = 0; c < 8; c += 2) {
        tmem_ld_wait_regs(ra);
        ptx::tmem_ld16(t_o + 128 * wg + 16 * (c + 1), rb);
        store_chunk(c, ra);
        tmem_ld_wait_regs(rb);
        if (c + 2 < 8) ptx::tmem_ld16(t_o + 128 * wg + 16 * (c + 2), ra);
        store_chunk(c + 1, rb);
      }
      if (real && cr == 0 && wg == 0) {
        if (direct) {
          if (p.lse) p.lse[orow] = lse_v;
        } else if (partial) {
          reinterpret_cast<float*>(p.ws + partial_lse_offset(p.slots_cap, p.H))[(size_t)it.slot * p.H + row] = lse_v;
        }
      }
      ptx::tc_fence_before();
      ptx::mbar_arrive(b_o_free);
      ++n_item;
    }
    // FP8: the peer's P.V commit for this warpgroup's last tile lands on x_empty[wg]: take it
    // before exit
    if (send_in_softmax<KV>() && !dead && g > 0) {
      const int last = ((g - 1) & 1) == wg ? g - 1 : g - 2;
      if (last >= 0) ptx::mbar_wait(b_x_empty + 8 * wg, (uint32_t)(last >> 1) & 1u, abort_flag, true);
    }
  } else if (warp == kWarpItems) {
    // ------------------------------------------------------------------ work items
    // Walks this worker's items once, publishes them to the ring, and asks L2 for each
    // item's query rows ahead of the senders' loads.
    regs_to<RegSplit<KV>::ctrl>();
    if (lane == 0) {
      // the first item comes from the schedule evaluated at start-up; the cursor (whose
      // first step reproduces it) supplies the rest
      ItemCursor cur{};
      for (int k = 0;; ++k) {
        WorkItem nx = wst.first;
        bool more = wst.busy != 0;
        if (k > 0) {
          if (k == 1) {  // the cursor starts at the first item, already published
            cur = item_cursor(p, wst, worker);
            next_item(p, n_tiles_total, cur, nx);
          }
          more = next_item(p, n_tiles_total, cur, nx);
        }
        const int s = k % kItemRing;
        if (k >= kItemRing && !ptx::mbar_wait(b_item_empty + 8 * s, (uint32_t)((k / kItemRing) - 1) & 1u, abort_flag))
          break;
        if (more && cr == 0) {
          ptx::bulk_prefetch_l2(p.q_nope + (size_t)nx.u * p.H * kLatent, (uint32_t)p.H * kLatent * 2);
          ptx::bulk_prefetch_l2(p.q_pe + (size_t)nx.u * p.H * kRope, (uint32_t)p.H * kRope * 2);
        }
        S.items[s] = more ? make_int4(nx.u, nx.tok_lo, nx.tok_hi, nx.slot) : make_int4(0, 0, -1, -1);
        S.items_min[s] = more ? nx.tok_min : 0;
        ptx::mbar_arrive(b_item_full + 8 * s);
        if (!more) break;
      }
    }
  }
  if (warp >= kWarpSoftmax0 && lane == 0) ptx::bulk_wait_all();  // epilogue stores done before exit
  // ------------------------------------------------------------------ teardown
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) ptx::tmem_dealloc(tmem, kTmemCols);
  if (tid == 0 && blockIdx.x < kMaxCtas)
    reinterpret_cast<unsigned*>(p.ws + kCtaStatusOffset)[blockIdx.x] = S.status | (S.abort_flag ? MLA_STATUS_WAIT_TIMEOUT : 0u);
  ptx::cluster_sync_all();
}

}  // namespace tc

// ---------------------------------------------------------------------- host side
namespace {

// 2-D view of a bf16 or FP8 cache: [num_pages * page_size rows, 576 columns], one page of
// rows per box.
bool encode_cache_map(CUtensorMap* m, const void* cache, int num_pages, int ps, int box_cols, int elem_bytes,
                      CUtensorMapSwizzle sw) {
  EncodeTiledFn fn = tmap_encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)kDim, (cuuint64_t)num_pages * ps};
  cuuint64_t strides[1] = {(cuuint64_t)kDim * elem_bytes};
  cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)ps};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, elem_bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 2,
            const_cast<void*>(cache), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
// Row-major [rows, 512] output tensor (bf16 or fp32), boxes of 16 columns x 16 rows.
bool encode_rows_map(CUtensorMap* m, const void* base, size_t rows, int elem_bytes, CUtensorMapSwizzle sw) {
  EncodeTiledFn fn = tmap_encode_fn();
  if (!fn || rows == 0) return false;
  cuuint64_t dims[2] = {(cuuint64_t)kLatent, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)kLatent * elem_bytes};
  cuuint32_t box[2] = {16, 16};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, elem_bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2,
            const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
            CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
}  // namespace

size_t tc_smem_bytes() { return sizeof(tc::Smem) + 1024; }

#ifdef MLA_FAULT_INJECTION
// Test builds only: makes CTA `cta` skip the loads of tile `tile` of its schedule in the
// following decode launches (cta < 0: no tile skipped).
extern "C" __attribute__((visibility("default"))) int mla_fault_injection_drop_tile(int cta, int tile) {
  cudaError_t e = cudaMemcpyToSymbol(g_drop_cta, &cta, sizeof(int));
  if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_drop_tile, &tile, sizeof(int));
  return (int)e;
}
#endif

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
static cudaError_t launch_tc(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& o, const DecodeParams& p,
                             cudaStream_t stream) {
  auto kern = tc::mla_decode_tc_kernel<KV>;
  // the shared-memory opt-in outlives the call: set once per device
  static std::mutex mu;
  static bool opted_in[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  {
    std::lock_guard<std::mutex> lk(mu);
    if (!opted_in[dev]) {
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)tc_smem_bytes());
      if (e != cudaSuccess) return e;
      opted_in[dev] = true;
    }
  }
  kern<<<2 * p.workers, tc::kThreads, tc_smem_bytes(), stream>>>(a, b, o, p);
  return cudaGetLastError();
}

cudaError_t launch_decode_tc(const DecodeParams& p, cudaStream_t stream) {
  static_assert(sizeof(tc::Smem) + 1024 <= 227 * 1024, "shared memory budget");
  CUtensorMap tm_lat, tm_rope, tm_out;
  memset(&tm_lat, 0, sizeof(tm_lat));
  memset(&tm_rope, 0, sizeof(tm_rope));
  // output: [B*q_len*H, 512] bf16, 16 x 16 boxes
  const int units = p.B * p.q_len;
  if (!encode_rows_map(&tm_out, p.out, (size_t)units * p.H, 2, CU_TENSOR_MAP_SWIZZLE_32B)) return cudaErrorInvalidValue;
  if (p.kv_dtype == MLA_KV_BF16) {
    if (!encode_cache_map(&tm_lat, p.cache, p.num_pages, p.page_size, 64, 2, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_cache_map(&tm_rope, p.cache, p.num_pages, p.page_size, 32, 2, CU_TENSOR_MAP_SWIZZLE_64B))
      return cudaErrorInvalidValue;
    return launch_tc<MLA_KV_BF16>(tm_lat, tm_rope, tm_out, p, stream);
  }
  if (p.kv_dtype == MLA_KV_FP8_E4M3) {
    if (!encode_cache_map(&tm_lat, p.cache, p.num_pages, p.page_size, 256, 1, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !encode_cache_map(&tm_rope, p.cache, p.num_pages, p.page_size, 32, 1, CU_TENSOR_MAP_SWIZZLE_NONE))
      return cudaErrorInvalidValue;
    return launch_tc<MLA_KV_FP8_E4M3>(tm_lat, tm_rope, tm_out, p, stream);
  }
  return launch_tc<MLA_KV_NVFP4>(tm_lat, tm_rope, tm_out, p, stream);
}

}  // namespace mla

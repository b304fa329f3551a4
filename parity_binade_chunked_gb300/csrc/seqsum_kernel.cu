// The device path of the exact sequential fp64 sum (sm_103a).
//
// One persistent kernel.  CTAs 0 .. nwalkers-1 walk; every other CTA streams
// tiles of 4096 terms (32 KB, one TMA box) taken in ticket order, in a
// three-stage pipeline: the copy of tile i+2 is in flight while the plan of
// tile i+1 and the runs of tile i are formed.
//
//  * Plan (Research-1424, section 3: "a first pass can add each row on its own
//    and a prefix over the rows gives S at each row start ... which names the
//    binade except next to a power of two"; Research-1433, finding 5 and the
//    open question "compute the plan's prefix with a scan across the lanes"):
//    every term's fp32 image is built from its bits with integer operations,
//    a tile's approximate sum is published as soon as the tile has landed,
//    and a decoupled look-back over the published sums, 256 tiles per read,
//    gives each tile its approximate starting value in double-float.  No
//    fp64 instruction is used for the plan.
//  * Runs (finding 2 "Inside a binade the loop is an integer sum", finding 3
//    "Ties need the parity of the running integer"): a chunk of 512 terms
//    whose whole range lies inside one binade is turned into its increment
//    by integer shifts (binade_math.cuh) and composed: each lane's 16 terms
//    in order, then the warp's 32 lanes in a fixed shuffle tree (finding 6).
//  * A chunk the plan cannot place in one binade is split: lanes that fit a
//    binade become runs, and inside the other lanes each term is placed on
//    its own; only the terms whose approximate prefix lies next to a power of
//    two are carried, as values, to be added one by one (finding 4).
//  * The walk (finding 4; open question "compose runs of chunks that share a
//    binade so that the walk steps over 64 or 1024 chunks at a time") runs
//    at the same time as the stream: it reads tile headers as they appear,
//    composes every maximal run of same-binade records in parallel, and on
//    one warp applies the composites to the exact running value, adds the
//    carried terms with __dadd_rn, and falls back to term-by-term adds where
//    the exact check rejects a run.
//
// This translation unit is built with --fmad=false; every fp64 add of the
// walk is one __dadd_rn, in index order.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "binade_math.cuh"
#include "seqsum_internal.cuh"

namespace sq {

// ---------------------------------------------------------------- constants
// Relative error allowance of the plan against the running sum of |x|: fp32
// term images keep 20 fraction bits (truncated), fp32 sums of 16 and 32
// values, double-float across chunks and tiles.  The plan only chooses where
// to look; a wrong guess costs a fallback, never a wrong bit.
constexpr float kEps = 0x1p-18f;
constexpr float kRelF32 = 0x1p-21f;            // rounding of one fp32 prefix value
constexpr float kTinyF = 0x1p-120f;
constexpr int kZeroE = -2000;                  // binade key of a run of zeros
constexpr int kDirtyKey = -3000;               // merge key of a lane placed term by term
constexpr uint64_t kWaitNs = 2000000000ull;    // bounded device waits: 2 s
constexpr uint32_t kMagLo = 896u << 20;        // exponent 896 = 2^-127
constexpr uint64_t kCountMask = (1u << kCountBits) - 1;
static_assert(((uint64_t)kChunkSlots << (kCountBits * (kWarps - 1))) < (1ull << 55),
              "packed item counts must fit a tagged 56-bit word");
constexpr int kWalkOffEl = 32768;              // walker layout in the dynamic shared memory
constexpr int kWalkOffPos = 65536;
constexpr int kWalkOffEnds = 69632;
static_assert(kWalkTiles * (int)sizeof(Rec) <= kWalkOffEl, "walk headers overlap the element list");
static_assert(kWalkElems * (int)sizeof(Rec) <= kWalkOffEl, "segment composites overlap the element list");
static_assert(kWalkOffEl + kWalkElems * (int)sizeof(Rec) <= kWalkOffPos, "element list overlaps positions");
static_assert(kWalkOffPos + kWalkElems * 4 <= kWalkOffEnds, "positions overlap segment ends");
static_assert(kWalkOffEnds + kWalkElems * 4 <= kStages * kStageBytes, "walk buffers exceed the stages");
static_assert(kWalkElems % kThreads == 0 && kWalkTiles % kThreads == 0, "walk batch split");

// ---------------------------------------------------------------- PTX helpers
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// 2-D tiled TMA load of one box (16 terms x 256 rows) into shared memory.
__device__ __forceinline__ void tma_load_box(void *dst, const CUtensorMap *map, uint64_t *bar, int32_t c0,
                                             int32_t c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], "
      "[%2];" ::"r"(smem_u32(dst)),
      "l"(map), "r"(smem_u32(bar)), "r"(c0), "r"(c1)
      : "memory");
}
__device__ __forceinline__ void ld_vol_v2(const void *p, uint64_t &a, uint64_t &b) {
  asm volatile("ld.volatile.global.v2.u64 {%0, %1}, [%2];" : "=l"(a), "=l"(b) : "l"(p) : "memory");
}
__device__ __forceinline__ void st_vol_v2(void *p, uint64_t a, uint64_t b) {
  asm volatile("st.volatile.global.v2.u64 [%0], {%1, %2};" ::"l"(p), "l"(a), "l"(b) : "memory");
}

// Named barrier kBarWide: the 256 threads of a walking or scanning CTA (its
// control warp takes no part).  Streaming CTAs synchronise through mbarriers
// only, every wait bounded.
constexpr int kBarWide = 1;
// The non-aligned form: a warp's threads may arrive at it separately (code
// before it is lane-divergent, and the compiler does not treat an asm barrier
// as a point where the warp must be converged, which the aligned bar.sync
// requires).
__device__ __forceinline__ void named_sync(int id, int nthreads) {
  asm volatile("barrier.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}
struct Smem;
__device__ __noinline__ void wide_sync_at(const Params &p, Smem &sm, int site);
#define wide_sync(p, sm, site) wide_sync_at((p), (sm), (site))
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
// Heartbeat of this CTA (one thread calls it): its role, what it waits for
// or does (HB_*) and where (a unit, tile or position), read by the host
// while a call runs.
// One word per warp (index CTA * 9 + warp).
enum : uint32_t {
  HB_START = 1, HB_WAIT_UNIT = 2, HB_UNIT = 3, HB_WAIT_DONE = 4, HB_EPILOGUE = 5, HB_WAIT_HEADERS = 6,
  HB_BATCH = 7, HB_SERIAL = 8, HB_WAIT_SUMS = 9, HB_WINDOW = 10, HB_COUNT = 11, HB_GATHER = 12, HB_SCAN = 13,
  HB_RESTART = 14, HB_END = 15, HB_BARRIER = 16
};
__device__ __forceinline__ void beat(const Params &p, uint32_t role, uint32_t what, uint64_t where) {
  const unsigned i = blockIdx.x * 9u + (threadIdx.x >> 5);
  if (i < (unsigned)kHeartbeats)
    p.hb[i] = ((uint64_t)(role & 0xFFu) << 56) | ((uint64_t)(what & 0xFFu) << 48) | (where & 0xFFFFFFFFFFFFull);
}

// A bounded wait gave up: set its error bit and keep the first such site
// with two words of context for the host.
enum : uint32_t {
  TO_FULL = 1, TO_DONE = 2, TO_SUMS = 3, TO_PREFIX = 4, TO_TILESUM = 5, TO_SCAN = 6, TO_WALK = 7
};
__device__ __noinline__ void note_timeout(const Params &p, uint32_t err, uint32_t site, uint32_t a, uint32_t b) {
  atomicOr(&p.ctr[C_ERR], err);
  if (atomicCAS(&p.ctr[C_TO_SITE], 0u, site) == 0u) {
    p.ctr[C_TO_A] = a;
    p.ctr[C_TO_B] = b;
  }
}
// A bounded wait on an mbarrier phase; false on timeout.
__device__ __forceinline__ bool mbar_wait(const Params &p, uint64_t *bar, uint32_t parity, uint32_t err,
                                          uint32_t site, uint32_t a, uint32_t b) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer() - t0 > kWaitNs) {
      note_timeout(p, err, site, a, b);
      return false;
    }
  }
  return true;
}

// One of the barrier's expected arrivals, made when every earlier cp.async
// of this thread has completed.
__device__ __forceinline__ void cp_async_mbar_arrive(uint64_t *bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// 16-byte asynchronous copy global -> shared through L2 (the prefetch of a
// run unit's plan words); completed by cp_async_wait_all of the same thread.
__device__ __forceinline__ void cp_async16(void *dst, const void *src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

__device__ __forceinline__ uint64_t dbits(double v) { return (uint64_t)__double_as_longlong(v); }
__device__ __forceinline__ double bitsd(uint64_t b) { return __longlong_as_double((long long)b); }

// Self-checking build (-DSEQSUM_CHECKS): every computed global index and
// every walker buffer index is checked before use; a failed check records
// its site and value in the counters, sets ERR_CHECK and skips the access.
#ifdef SEQSUM_CHECKS
__device__ __forceinline__ bool sq_ok(const Params &p, bool cond, uint32_t site, int64_t val) {
  if (!cond) {
    if (atomicCAS(&p.ctr[C_CHECK_SITE], 0u, site) == 0u) {
      p.ctr[C_CHECK_LO] = (uint32_t)(uint64_t)val;
      p.ctr[C_CHECK_HI] = (uint32_t)((uint64_t)val >> 32);
    }
    atomicOr(&p.ctr[C_ERR], 32u);
  }
  return cond;
}
#else
#define sq_ok(p, cond, site, val) (true)
#endif
__device__ __forceinline__ bool item_ok(const Params &p, const Rec *q, uint32_t site) {
  return sq_ok(p, q >= p.items && q < p.items + p.cap_tiles * kTileSlots, site, (int64_t)(q - p.items));
}

// ---------------------------------------------------------------- double-float
// (hi + lo) pairs of fp32 for the plan's prefix; every op is one rounded fp32
// add (no contraction in this translation unit).
struct DF {
  float hi, lo;
};
__device__ __forceinline__ DF two_sum(float a, float b) {
  const float s = __fadd_rn(a, b);
  const float bb = __fsub_rn(s, a);
  const float err = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
  return DF{s, err};
}
__device__ __forceinline__ DF df_add(DF x, DF y) {
  const DF s = two_sum(x.hi, y.hi);
  const float lo = __fadd_rn(s.lo, __fadd_rn(x.lo, y.lo));
  const float hi = __fadd_rn(s.hi, lo);
  return DF{hi, __fsub_rn(lo, __fsub_rn(hi, s.hi))};
}
__device__ __forceinline__ DF df_addf(DF x, float y) { return df_add(x, DF{y, 0.0f}); }
__device__ __forceinline__ DF df_from_double(double v) {
  const float h = (float)v;                       // once per sum
  return DF{h, (float)(v - (double)h)};
}
__device__ __forceinline__ DF shfl_xor_df(DF v, int m) {
  return DF{__shfl_xor_sync(0xffffffffu, v.hi, m), __shfl_xor_sync(0xffffffffu, v.lo, m)};
}

// ---------------------------------------------------------------- the plan's term image
// fp32 image of a term from its high word: 20 fraction bits (truncated), the
// exponent moved to the fp32 bias; magnitudes below 2^-127 give 0.  Terms of
// 2^128 and above need the clamped form.
__device__ __forceinline__ float approx_term(uint32_t hi) {
  const uint32_t v = max(hi & 0x7FFFFFFFu, kMagLo);
  return __uint_as_float(((v - kMagLo) * 8u) | (hi & 0x80000000u));
}
__device__ __forceinline__ float approx_term_clamped(uint32_t hi) {
  const uint32_t v = min(max(hi & 0x7FFFFFFFu, kMagLo), (1150u << 20) | 0xFFFFFu);
  return __uint_as_float(((v - kMagLo) * 8u) | (hi & 0x80000000u));
}

// Binade (unbiased exponent) shared by all of [lo, hi] (fp32), or false.
__device__ __forceinline__ bool one_binade_f(float lo, float hi, int &e) {
  float a, b;
  if (lo > 0.0f) { a = lo; b = hi; }
  else if (hi < 0.0f) { a = -hi; b = -lo; }
  else return false;
  const int ea = (int)((__float_as_uint(a) >> 23) & 0xFF), eb = (int)((__float_as_uint(b) >> 23) & 0xFF);
  if (ea != eb || ea == 0 || ea == 0xFF) return false;
  e = ea - 127;
  return true;
}

__device__ __forceinline__ uint32_t hash3(uint64_t a, uint32_t b, uint32_t c) {
  uint64_t z = a * 0x9E3779B97F4A7C15ull + b * 0xBF58476D1CE4E5B9ull + c;
  z ^= z >> 31; z *= 0x94D049BB133111EBull; z ^= z >> 29;
  return (uint32_t)z;
}

// Forced plans (tests only; Research-1433, finding 5): the walk must give the
// same bits under all of them.
__device__ __forceinline__ bool plan_override(int mode, bool clean, int &e, uint64_t t, int w, int lane) {
  switch (mode) {
    case 1: e += 1; return clean;                       // one binade too high
    case 2: e = -1022; return true;                     // "all zero"
    case 3: e = 0; return true;                         // one fixed binade
    case 4: return false;                               // everything term by term
    case 5: e += (int)(hash3(t, (uint32_t)w, (uint32_t)lane) % 3u) - 1; return clean;
    default: return clean;
  }
}

enum { SH_IDX = 0, SH_DOWN = 1, SH_UP = 2 };
template <int KIND>
__device__ __forceinline__ Run shfl_run(const Run &r, int arg) {
  Run o;
  const unsigned full = 0xffffffffu;
  if (KIND == SH_DOWN) {
    o.inc = __shfl_down_sync(full, r.inc, arg);
    o.lo = __shfl_down_sync(full, r.lo, arg);
    o.hi = __shfl_down_sync(full, r.hi, arg);
    o.d = __shfl_down_sync(full, r.d, arg);
    o.flags = __shfl_down_sync(full, r.flags, arg);
  } else if (KIND == SH_UP) {
    o.inc = __shfl_up_sync(full, r.inc, arg);
    o.lo = __shfl_up_sync(full, r.lo, arg);
    o.hi = __shfl_up_sync(full, r.hi, arg);
    o.d = __shfl_up_sync(full, r.d, arg);
    o.flags = __shfl_up_sync(full, r.flags, arg);
  } else {
    o.inc = __shfl_sync(full, r.inc, arg);
    o.lo = __shfl_sync(full, r.lo, arg);
    o.hi = __shfl_sync(full, r.hi, arg);
    o.d = __shfl_sync(full, r.d, arg);
    o.flags = __shfl_sync(full, r.flags, arg);
  }
  return o;
}

__device__ __forceinline__ Rec make_rec(const Run &r, int e, uint32_t kind, uint32_t count, uint32_t tstart) {
  Rec q;
  q.inc = r.inc; q.lo = r.lo; q.hi = r.hi;
  q.meta = rec_meta(r.d, r.flags, kind, tstart);
  q.e = (int16_t)e;
  q.count = (uint16_t)count;
  return q;
}
__device__ __forceinline__ Run rec_run(const Rec &q) {
  Run r;
  r.inc = q.inc; r.lo = q.lo; r.hi = q.hi;
  r.d = rec_d(q.meta);
  r.flags = rec_flags(q.meta);
  return r;
}
__device__ __forceinline__ Rec ldcg_rec(const Rec *p) {
  const int4 *q = reinterpret_cast<const int4 *>(p);
  Rec r;
  int4 *o = reinterpret_cast<int4 *>(&r);
  o[0] = __ldcg(q);
  o[1] = __ldcg(q + 1);
  return r;
}
__device__ __forceinline__ void stcg_rec(Rec *p, const Rec &r) {
  const int4 *s = reinterpret_cast<const int4 *>(&r);
  int4 *q = reinterpret_cast<int4 *>(p);
  __stcg(q, s[0]);
  __stcg(q + 1, s[1]);
}

// Tile headers: the call's tag in the top byte of each of the four 64-bit
// words (inc, lo and hi sign-extended from 56 bits; in the last word the tag
// takes the first-term bits of meta, which are 0 in a header).  A 16-byte
// access need not be single-copy atomic, so a reader checks all four words
// and never takes a header made of two publications.
constexpr int64_t kBound56 = ((int64_t)1 << 55) - 1;
constexpr uint64_t kLow56 = 0x00FFFFFFFFFFFFFFull;
__device__ __forceinline__ int64_t untag56(uint64_t v) { return (int64_t)(v << 8) >> 8; }
__device__ __forceinline__ uint64_t tag56(int64_t v, uint32_t tag) {
  return ((uint64_t)max(min(v, kBound56), -kBound56) & kLow56) | ((uint64_t)tag << 56);
}
__device__ __forceinline__ void publish_header(Rec *p, const Rec &r, uint32_t tag) {
  const uint64_t a0 = tag56(r.inc, tag);
  const uint64_t a1 = tag56(r.lo, tag);
  const uint64_t b0 = tag56(r.hi, tag);
  const uint64_t b1 = (uint64_t)((r.meta & 0x00FFFFFFu) | (tag << 24)) | ((uint64_t)(uint16_t)r.e << 32) |
                      ((uint64_t)r.count << 48);
  st_vol_v2(p, a0, a1);
  st_vol_v2(reinterpret_cast<char *>(p) + 16, b0, b1);
}
// 1: the header carries `tag` in all four words; 0: not yet published;
// -1: a mix of two publications (read again).
__device__ __forceinline__ int read_header(const Rec *p, uint32_t tag, Rec &r) {
  uint64_t a0, a1, b0, b1;
  ld_vol_v2(p, a0, a1);
  ld_vol_v2(reinterpret_cast<const char *>(p) + 16, b0, b1);
  const int nt = ((uint32_t)(a0 >> 56) == tag) + ((uint32_t)(a1 >> 56) == tag) + ((uint32_t)(b0 >> 56) == tag) +
                 ((uint32_t)((b1 >> 24) & 0xFFu) == tag);
  if (nt != 4) return nt == 0 ? 0 : -1;
  r.inc = untag56(a0);
  r.lo = untag56(a1);
  r.hi = untag56(b0);
  r.meta = (uint32_t)b1 & 0x00FFFFFFu;
  r.e = (int16_t)(uint16_t)(b1 >> 32);
  r.count = (uint16_t)(b1 >> 48);
  return 1;
}

// ---------------------------------------------------------------- tile geometry
struct TileGeo {
  int32_t sum;          // which sum
  int64_t tile_in_sum;  // index of the tile within its sum
  int64_t first_tile;   // global index of the sum's first tile
  int64_t ntiles_sum;   // tiles of this sum
  int64_t start, end;   // term range [start, end) in x
};

__device__ __forceinline__ TileGeo tile_geo(const Params &p, int64_t t, int64_t ntiles) {
  TileGeo g;
  if (p.offsets == nullptr) {
    g.sum = 0; g.tile_in_sum = t; g.first_tile = 0; g.ntiles_sum = ntiles;
    g.start = t * kTileTerms;
    g.end = min(p.n, g.start + kTileTerms);
  } else {
    // the last k with tile_begin[k] <= t; empty sums share their successor's
    // tile_begin, and the search lands on the non-empty one.
    int lo = 0, hi = p.nsums;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (__ldcg(&p.tile_begin[mid]) <= t) lo = mid; else hi = mid;
    }
    g.sum = lo;
    g.first_tile = __ldcg(&p.tile_begin[lo]);
    g.ntiles_sum = __ldcg(&p.tile_begin[lo + 1]) - g.first_tile;
    g.tile_in_sum = t - g.first_tile;
    g.start = p.offsets[lo] + g.tile_in_sum * kTileTerms;
    g.end = min(p.offsets[lo + 1], g.start + kTileTerms);
  }
  return g;
}

// ---------------------------------------------------------------- shared memory
// A chunk's aggregates: the sum and |x| sum of its terms' fp32 images (the
// plan), the largest magnitude word and whether any term has its sign bit set
// or any term is non-zero (the exact preconditions of the fast runs).
enum : uint32_t { WA_NEG = 1u, WA_NZ = 2u };
struct WarpAgg {
  float sig, ab;
  uint32_t mx, flags;
};

struct Smem {
  uint64_t full[kStages];           // streaming: the unit's copy and plan words landed (3 arrivals)
  uint64_t done[kStages];           // streaming: the compute warps finished the unit
  uint64_t sums[kStages];           // streaming: the compute warps' chunk sums (a tile planned chunk by chunk)
  int64_t tk[kStages];              // the stage's tile
  int tma[kStages];                 // its terms came by TMA (else from global memory)
  int kind[kStages];                // U_PLAN, U_RUN or U_END
  int role;
  uint32_t barcnt[kWarps];          // walker/scanner: wide barriers passed per warp (heartbeat)
  // a run unit's plan words, copied in ahead of its runs: the tile's own
  // approximate sum and the prefix of the tile before (cp.async
  // destinations: 16-byte aligned)
  alignas(16) uint64_t tagg_raw[kStages][2];
  alignas(16) uint64_t pre_raw[kStages][2];
  WarpAgg wa[kStages][kWarps];
  Rec chunk[kStages][kWarps];       // a run unit's chunk records
  int nitems[kStages][kWarps];      // >0: a split chunk's items in the tile's item area
  unsigned int st[S_COUNT];         // per-CTA statistics of one call (32-bit: native shared atomics)
  // walker
  uint64_t S;
  int m, nel, restart, nseg;
  int walk_m[kWarps];
  int wflag[kWarps];
  Run wagg[kWarps];
  int wcnt[kWarps];
  int sum_k;
  // scanner
  int scan_m[kWarps];
  int scan_stop;
  DF scan_v[kWarps];
  float scan_a[kWarps];
  int scan_f[kWarps];
  DF carry;
  float carry_abs;
};
static_assert(offsetof(Smem, tagg_raw) % 16 == 0 && offsetof(Smem, pre_raw) % 16 == 0,
              "cp.async destinations must be 16-byte aligned");
static_assert(offsetof(Smem, full) % 8 == 0 && offsetof(Smem, done) % 8 == 0 && offsetof(Smem, sums) % 8 == 0,
              "mbarriers are 8-byte aligned");

// The 256-thread barrier of a walking or scanning CTA; each warp first
// records the barrier's site and how many it has passed (its heartbeat).
__device__ __noinline__ void wide_sync_at(const Params &p, Smem &sm, int site) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) {
    const uint32_t c = ++sm.barcnt[warp];
    beat(p, sm.role, HB_BARRIER, ((uint64_t)site << 32) | c);
  }
  named_sync(kBarWide, kThreads);
}


// ---------------------------------------------------------------- the plan's prefix
// Per tile two tagged 64-bit words, written and read as one 16-byte access:
//   A = sum.hi (fp32) << 32 | sum.lo (fp32) with its low 8 bits replaced by the tag
//   B = |x| sum (fp32) << 32 | tag;   tag = epoch << 1 | kind,
// kind 0 = the tile's own approximate sum, 1 = the inclusive prefix (s0 and
// every tile of the sum up to this one).  A reader takes a word pair only when
// both carry the same current tag.
__device__ __forceinline__ void publish_status(uint64_t *st, DF sig, float ab, uint32_t epoch, uint32_t kind) {
  const uint32_t tag = (epoch << 1) | kind;
  const uint64_t A = ((uint64_t)__float_as_uint(sig.hi) << 32) | ((__float_as_uint(sig.lo) & ~0xFFu) | tag);
  const uint64_t B = ((uint64_t)__float_as_uint(ab) << 32) | tag;
  st_vol_v2(st, A, B);
}
__device__ __forceinline__ DF status_sum(uint64_t A) {
  return DF{__uint_as_float((uint32_t)(A >> 32)), __uint_as_float((uint32_t)A & ~0xFFu)};
}
__device__ __forceinline__ float status_abs(uint64_t B) { return __uint_as_float((uint32_t)(B >> 32)); }

struct Prefix {
  DF ex;
  float ex_abs;
};

// Units of work.  Every tile has a plan unit (copy it, publish its approximate
// sum) and a run unit (copy it again, form its runs from the prefix the
// scanner published for the tile before it).  Tickets hand out the plan units
// of the first `wave` tiles, then a run unit and a plan unit in turn, then the
// remaining run units: the plan of tile t always precedes the run of tile
// t + 1 by about `wave` tiles, so a run unit's prefix is normally published
// long before it is read, and its tile is still in L2.  Returns true for a
// plan unit.
__device__ __forceinline__ bool unit_of(int64_t u, int64_t ntiles, int64_t wave, int64_t &tile) {
  const int64_t w = min(wave, ntiles);
  if (u < w) { tile = u; return true; }
  const int64_t v = u - w, rest = ntiles - w;
  if (v < 2 * rest) {
    tile = (v & 1) ? w + (v >> 1) : (v >> 1);
    return (v & 1) != 0;
  }
  tile = rest + (v - 2 * rest);
  return false;
}

// The approximate exclusive prefix of tile t: s0 for the first tile of a sum,
// else the inclusive prefix the scanner published for tile t - 1 (a bounded
// wait; on a timeout the plan is only worse, the result stays exact).  One
// thread.
__device__ __forceinline__ Prefix read_prefix(const Params &p, int sum, int64_t first_tile, int64_t t,
                                              unsigned int *st) {
  if (t == first_tile) {
    const DF ex = df_from_double(p.s0s ? p.s0s[sum] : p.s0);
    return Prefix{ex, fabsf(ex.hi)};
  }
  const uint32_t tag = (p.epoch << 1) | 1u;
  const uint64_t t0 = globaltimer();
  if (!sq_ok(p, t >= 1 && t - 1 < p.cap_tiles, 1, t)) return Prefix{DF{0.0f, 0.0f}, 0.0f};
  while (true) {
    uint64_t A, B;
    ld_vol_v2(p.status + 2 * (t - 1), A, B);
    const uint32_t ta = (uint32_t)(A & 0xFF), tb = (uint32_t)B;
    if (ta == tag && tb == tag) return Prefix{status_sum(A), status_abs(B)};
    if (ta != tb && ((ta >> 1) == p.epoch || (tb >> 1) == p.epoch)) atomicAdd(&st[S_TORN_STATUS], 1u);
    if (globaltimer() - t0 > kWaitNs) {
      note_timeout(p, ERR_PLAN_TIMEOUT, TO_PREFIX, (uint32_t)t, (uint32_t)(ta | (tb << 8) | (p.epoch << 16)));
      return Prefix{DF{0.0f, 0.0f}, 0.0f};
    }
    __nanosleep(32);
  }
}

// The scanner (a whole CTA): takes, from where it stands, the longest run of
// tiles whose approximate sums are published (up to 1024 tiles), scans it --
// a tile published as kind 1 starts a sum and already holds s0 plus its own
// sum -- and publishes every other tile's inclusive prefix as kind 1
// (Research-1424, section 3: a prefix over the row sums gives S at each row
// start; Research-1433, open question: the plan's prefix as a scan).
__device__ __noinline__ void scan_prefix(const Params &p, Smem &sm, int64_t ntiles) {
  constexpr int PER = 4;
  constexpr int WIN = kThreads * PER;
  const unsigned full = 0xffffffffu;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t ep = p.epoch;
  unsigned int *st = sm.st;
  int64_t pos = 0;
  DF carry = DF{0.0f, 0.0f};            // inclusive prefix of tile pos - 1
  float carry_abs = 0.0f;
  uint64_t tprog = globaltimer();
  const uint64_t tbegin = tprog;
  uint64_t twait = 0;
  while (pos < ntiles) {
    if (tid == 0) beat(p, sm.role, HB_WINDOW, (uint64_t)pos);
    uint64_t A[PER], B[PER];
#pragma unroll
    for (int q = 0; q < PER; q++) {
      const int64_t idx = pos + tid * PER + q;
      A[q] = 0;
      B[q] = 0;
      if (idx < ntiles && sq_ok(p, idx < p.cap_tiles, 20, idx)) ld_vol_v2(p.status + 2 * idx, A[q], B[q]);
    }
    int myfirst = PER;
#pragma unroll
    for (int q = PER - 1; q >= 0; q--) {
      const int64_t idx = pos + tid * PER + q;
      const uint32_t ta = (uint32_t)(A[q] & 0xFF), tb = (uint32_t)B[q];
      if (!(idx < ntiles && (ta >> 1) == ep && ta == tb)) myfirst = q;
    }
    // the published run [pos, pos + m): the first gap over the window
    const uint32_t wmin = __reduce_min_sync(full, myfirst < PER ? (uint32_t)(tid * PER + myfirst) : (uint32_t)WIN);
    if (lane == 0) sm.scan_m[warp] = (int)wmin;
    wide_sync(p, sm, 1);
    int m = WIN;
#pragma unroll
    for (int w2 = 0; w2 < kWarps; w2++) m = min(m, sm.scan_m[w2]);
    if (m == 0) {
      // thread 0 alone decides whether to give up, so the CTA stays together
      const uint64_t now = globaltimer();
      if (tid == 0) {
        sm.scan_stop = (now - tprog > kWaitNs) ? 1 : 0;
        if (sm.scan_stop) note_timeout(p, ERR_PLAN_TIMEOUT, TO_SCAN, (uint32_t)pos, (uint32_t)ntiles);
      }
      __nanosleep(64);
      twait += globaltimer() - now;
      wide_sync(p, sm, 2);                       // sm.scan_stop is set; sm.scan_m may be written again
      if (sm.scan_stop) break;
      continue;
    }
    tprog = globaltimer();
    // this thread's elements, scanned in order; a kind-1 tile restarts the sum
    DF v[PER];
    float a[PER];
    bool f[PER];
    DF tv = DF{0.0f, 0.0f};
    float tab = 0.0f;
    bool tf = false;
#pragma unroll
    for (int q = 0; q < PER; q++) {
      if (tid * PER + q < m) {
        const DF val = status_sum(A[q]);
        const float ab = status_abs(B[q]);
        if (A[q] & 1u) { tv = val; tab = ab; tf = true; }
        else { tv = df_add(tv, val); tab += ab; }
      }
      v[q] = tv;
      a[q] = tab;
      f[q] = tf;
    }
    // across the warp, then across the warps (segmented: a head cuts the sum)
    DF wv = tv;
    float wab = tab;
    int wf = tf ? 1 : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const DF ov = DF{__shfl_up_sync(full, wv.hi, o), __shfl_up_sync(full, wv.lo, o)};
      const float oa = __shfl_up_sync(full, wab, o);
      const int of = __shfl_up_sync(full, wf, o);
      if (lane >= o) {
        if (!wf) { wv = df_add(ov, wv); wab = oa + wab; }
        wf |= of;
      }
    }
    if (lane == 31) { sm.scan_v[warp] = wv; sm.scan_a[warp] = wab; sm.scan_f[warp] = wf; }
    wide_sync(p, sm, 3);
    DF ev = carry;
    float eab = carry_abs;
    for (int w2 = 0; w2 < warp; w2++) {
      if (sm.scan_f[w2]) { ev = sm.scan_v[w2]; eab = sm.scan_a[w2]; }
      else { ev = df_add(ev, sm.scan_v[w2]); eab += sm.scan_a[w2]; }
    }
    {
      const DF lv = DF{__shfl_up_sync(full, wv.hi, 1), __shfl_up_sync(full, wv.lo, 1)};
      const float la = __shfl_up_sync(full, wab, 1);
      const int lf = __shfl_up_sync(full, wf, 1);
      if (lane >= 1) {
        if (lf) { ev = lv; eab = la; }
        else { ev = df_add(ev, lv); eab += la; }
      }
    }
#pragma unroll
    for (int q = 0; q < PER; q++) {
      const int i = tid * PER + q;
      if (i < m) {
        const DF inc = f[q] ? v[q] : df_add(ev, v[q]);
        const float inca = f[q] ? a[q] : eab + a[q];
        if (!(A[q] & 1u)) publish_status(p.status + 2 * (pos + i), inc, inca, ep, 1);
        if (i == m - 1) { sm.carry = inc; sm.carry_abs = inca; }
      }
    }
    wide_sync(p, sm, 4);
    carry = sm.carry;
    carry_abs = sm.carry_abs;
    pos += m;
    if (tid == 0) atomicAdd(&st[S_SCAN_WINDOWS], 1u);
    wide_sync(p, sm, 5);
  }
  if (tid == 0) {
    atomicAdd(&st[S_NS_SCAN], (unsigned)(tprog - tbegin));
    atomicAdd(&st[S_NS_SCAN_WAIT], (unsigned)(twait));
  }
}

// ---------------------------------------------------------------- lanes
__device__ __forceinline__ void load_lane(const Params &p, const unsigned char *stage, bool use_tma,
                                          int64_t row, int64_t lstart, int nv, int w, int lane, uint64_t *xs) {
  if (use_tma && row < p.tma_rows) {
    const unsigned char *rp = stage + (w * 32 + lane) * 128;
    const int sw = lane & 7;
#pragma unroll
    for (int c = 0; c < 8; c++) {
      const uint4 v = *reinterpret_cast<const uint4 *>(rp + ((c ^ sw) << 4));
      xs[2 * c] = ((uint64_t)v.y << 32) | v.x;
      xs[2 * c + 1] = ((uint64_t)v.w << 32) | v.z;
    }
#pragma unroll
    for (int i = 0; i < kLaneTerms; i++)
      if (i >= nv) xs[i] = 0ull;
  } else {
    const unsigned long long *gp = reinterpret_cast<const unsigned long long *>(p.x) + lstart;
    const bool ok = sq_ok(p, nv == 0 || (lstart >= 0 && lstart + nv <= p.n), 3, lstart);
#pragma unroll
    for (int i = 0; i < kLaneTerms; i++) xs[i] = (i < nv && ok) ? __ldg(gp + i) : 0ull;
  }
}

// Exact run of a lane's terms under binade e (the general path: ties,
// signed terms whose bounds need every prefix, binades outside the fast
// path's range).  Kept out of line, with the lane's terms loaded again, so
// that the hot path stays small.
__device__ __noinline__ Run lane_run_general(const Params &p, const unsigned char *stage, bool use_tma,
                                             int64_t row, int64_t lstart, int nv, int w, int lane, int e) {
  const bool from_stage = use_tma && row < p.tma_rows;
  const unsigned char *rp = stage + (w * 32 + lane) * 128;
  const unsigned long long *gp = reinterpret_cast<const unsigned long long *>(p.x) + lstart;
  if (!from_stage && !sq_ok(p, nv == 0 || (lstart >= 0 && lstart + nv <= p.n), 3, lstart)) nv = 0;
  Run r = run_empty();
#pragma unroll 1
  for (int i = 0; i < nv; i++) {
    uint64_t x;
    if (from_stage) {
      // term i of the lane's 128-byte row: 16-byte chunk i/2, swizzled by the row
      const uint2 v = *reinterpret_cast<const uint2 *>(rp + ((((i >> 1) ^ (lane & 7)) << 4) | ((i & 1) << 3)));
      x = ((uint64_t)v.y << 32) | v.x;
    } else {
      x = __ldg(gp + i);
    }
    int64_t re;
    int32_t d;
    const bool poison = term_inc(x, e, re, d);
    run_push(r, re, d, term_flags(x) | (poison ? F_POISON : 0u));
  }
  return r;
}

// Items of one lane the plan could not place in a binade, term by term: runs
// of terms whose approximate prefix stays inside one binade, and up to three
// carried terms per item where it does not.  With out == nullptr only counts.
__device__ __noinline__ int lane_items(const Params &p, const uint64_t *xs, int nv, float A, float dbase, uint64_t t, int w,
                          int lane, Rec *out) {
  float a = A;
  int cur = 0, cur_e = 0, nterms = 0, cstart = 0, n = 0;
  Run rr = run_empty();
  int64_t vals[3] = {0, 0, 0};
  uint32_t tf_or = 0;
  const uint32_t tbase = (uint32_t)(w * kChunkTerms + lane * kLaneTerms);
  for (int i = 0; i <= nv; i++) {
    int kind = 0, ei = 0;
    int64_t re = 0;
    int32_t dd = 0;
    if (i < nv) {
      const float a1 = a + approx_term_clamped((uint32_t)(xs[i] >> 32));
      const float d = dbase + kRelF32 * fmaxf(fabsf(a), fabsf(a1));
      bool ok = one_binade_f(fminf(a, a1) - d, fmaxf(a, a1) + d, ei);
      ok = plan_override(p.plan_mode, ok, ei, t, w, 100 + lane * 16 + i);
      if (ok && term_inc(xs[i], ei, re, dd)) ok = false;
      kind = ok ? 1 : 2;
      a = a1;
    }
    // close the open item when this term does not extend it
    const bool extend = (i < nv) && ((kind == 1 && cur == 1 && cur_e == ei) || (kind == 2 && cur == 2 && nterms < 3));
    if (!extend && cur != 0) {
      if (out && item_ok(p, out + n, 4)) {
        if (cur == 1) {
          stcg_rec(out + n, make_rec(rr, cur_e, K_RUN, (uint32_t)(i - cstart), tbase + (uint32_t)cstart));
        } else {
          Run tr = run_empty();
          tr.inc = vals[0]; tr.lo = vals[1]; tr.hi = vals[2]; tr.d = 0;
          tr.flags = tf_or & (F_HASINF_P | F_HASINF_N | F_HASNAN);
          stcg_rec(out + n, make_rec(tr, 0, K_TERMS, (uint32_t)nterms, tbase + (uint32_t)cstart));
        }
      }
      n++;
      cur = 0;
    }
    if (i == nv) break;
    if (cur == 0) {
      cur = kind;
      cstart = i;
      rr = run_empty();
      nterms = 0;
      tf_or = 0;
      cur_e = ei;
    }
    if (kind == 1) {
      run_push(rr, re, dd, term_flags(xs[i]));
    } else {
      vals[nterms++] = (int64_t)xs[i];
      tf_or |= term_flags(xs[i]);
    }
  }
  return n;
}

// A chunk the plan could not place in one binade.  Lanes that fit one become
// runs (neighbouring runs of one binade merge); the other lanes are placed
// term by term.  Writes the items for chunk w into the tile's item area and
// returns their number, or 0 when they do not fit (the caller then records
// the chunk as one fallback).
__device__ __noinline__ int split_chunk(const Params &p, const unsigned char *stage, bool use_tma, int64_t row,
                                       int64_t lstart, int nv, int w, int lane, DF sc, float ac, uint64_t t,
                                       Rec *area, unsigned int *st) {
  uint64_t xs[kLaneTerms];
  load_lane(p, stage, use_tma, row, lstart, nv, w, lane, xs);
  float sig = 0.0f, ab = 0.0f;
  uint32_t orz = 0;
#pragma unroll
  for (int i = 0; i < kLaneTerms; i++) {
    const uint32_t hi = (uint32_t)(xs[i] >> 32);
    const float f = approx_term_clamped(hi);
    sig += f;
    ab += fabsf(f);
    orz |= (hi & 0x7FFFFFFFu) | (uint32_t)xs[i];
  }
  float isig = sig, iab = ab;
#pragma unroll 1
  for (int o = 1; o < 32; o <<= 1) {
    const float a = __shfl_up_sync(0xffffffffu, isig, o);
    const float b = __shfl_up_sync(0xffffffffu, iab, o);
    if (lane >= o) { isig += a; iab += b; }
  }
  const DF A0 = df_addf(sc, isig - sig);
  const float A = A0.hi + A0.lo;
  const float P = 0.5f * (ab + sig), N = 0.5f * (ab - sig);
  const float dbase = kEps * (ac + (iab - ab) + ab) + kTinyF;
  const float dl = dbase + kRelF32 * (fabsf(A) + ab);
  int e_l = 0;
  bool clean = one_binade_f(A - N - dl, A + P + dl, e_l);
  clean = plan_override(p.plan_mode, clean, e_l, t, w, lane + 1);
  const bool zl = (orz == 0);
  const bool dirty = !clean && !zl && nv > 0;
  Run r = run_empty();
  if (!dirty) r = lane_run_general(p, stage, use_tma, row, lstart, nv, w, lane, clean ? e_l : 0);
  const int key = dirty ? kDirtyKey : (clean ? e_l : kZeroE);
  const int ndirty = dirty ? lane_items(p, xs, nv, A, dbase, t, w, lane, nullptr) : 0;
  if (dirty) atomicAdd(&st[S_LANE_DIRTY], 1u);
  // merge neighbouring runs of one key (lanes past the end join the previous)
  const int pkey = __shfl_up_sync(0xffffffffu, key, 1);
  const bool head = (lane == 0) || (nv > 0 && (dirty || pkey == kDirtyKey || key != pkey));
  Run v = r;
  int fl = head ? 1 : 0;
#pragma unroll 1
  for (int o = 1; o < 32; o <<= 1) {
    const Run ov = shfl_run<SH_UP>(v, o);
    const int of = __shfl_up_sync(0xffffffffu, fl, o);
    if (lane >= o) { if (!fl) v = run_compose(ov, v); fl |= of; }
  }
  const uint32_t heads = __ballot_sync(0xffffffffu, head);
  const bool end = (lane == 31) || ((heads >> (lane + 1)) & 1u);
  const uint32_t le = heads & ((lane == 31) ? 0xffffffffu : ((2u << lane) - 1u));
  const int hlane = 31 - __clz(le);
  const int hkey = __shfl_sync(0xffffffffu, key, hlane);
  // terms before each lane, for the item counts
  int csum = nv;
#pragma unroll 1
  for (int o = 1; o < 32; o <<= 1) {
    const int vv = __shfl_up_sync(0xffffffffu, csum, o);
    if (lane >= o) csum += vv;
  }
  const int before_head = __shfl_sync(0xffffffffu, csum - nv, hlane);
  // items per lane: a merged run at its end lane, or the dirty lane's own
  // items; if they do not fit, each dirty lane becomes one fallback item
  bool lane_fb = false;
  int myitems = dirty ? ndirty : ((end && hkey != kDirtyKey) ? 1 : 0);
  int ioff = 0, total = 0;
  for (int attempt = 0; attempt < 2; attempt++) {
    ioff = myitems;
#pragma unroll 1
    for (int o = 1; o < 32; o <<= 1) {
      const int vv = __shfl_up_sync(0xffffffffu, ioff, o);
      if (lane >= o) ioff += vv;
    }
    total = __shfl_sync(0xffffffffu, ioff, 31);
    ioff -= myitems;
    if (total <= kChunkSlots) break;
    lane_fb = true;
    myitems = dirty ? 1 : ((end && hkey != kDirtyKey) ? 1 : 0);
  }
#ifdef SEQSUM_CHECKS
  if (t == 0 && w == 0) {
    p.dbg[14000 + lane] = (unsigned long long)dirty | ((unsigned long long)clean << 1) | ((unsigned long long)zl << 2) |
                          ((unsigned long long)head << 3) | ((unsigned long long)end << 4) |
                          ((unsigned long long)lane_fb << 5) | ((unsigned long long)(hlane & 63) << 8) |
                          ((unsigned long long)(myitems & 255) << 16) | ((unsigned long long)(ioff & 255) << 24) |
                          ((unsigned long long)(total & 255) << 32) | ((unsigned long long)(ndirty & 255) << 40) |
                          ((unsigned long long)(uint16_t)(int16_t)key << 48);
    p.dbg[14040 + lane] = (unsigned long long)__float_as_uint(A) | ((unsigned long long)__float_as_uint(dl) << 32);
    p.dbg[14080 + lane] = (unsigned long long)__float_as_uint(P) | ((unsigned long long)__float_as_uint(N) << 32);
  }
#endif
  if (total > kChunkSlots) return 0;
  Rec *out = area + w * kChunkSlots;
  if (!dirty && myitems && item_ok(p, out + ioff, 5))
    stcg_rec(out + ioff, make_rec(v, hkey, K_RUN, (uint32_t)(csum - before_head),
                                  (uint32_t)(w * kChunkTerms + hlane * kLaneTerms)));
  if (dirty && lane_fb) {
    if (item_ok(p, out + ioff, 16)) {
      Run fr = run_empty();
      uint32_t tf = 0;
      for (int i = 0; i < nv; i++) tf |= term_flags(xs[i]);
      fr.flags = tf & (F_HASINF_P | F_HASINF_N | F_HASNAN);
      stcg_rec(out + ioff, make_rec(fr, 0, K_FALLBACK, (uint32_t)nv, (uint32_t)(w * kChunkTerms + lane * kLaneTerms)));
    }
  } else if (dirty) {
    lane_items(p, xs, nv, A, dbase, t, w, lane, out + ioff);
  }
  return total;
}

// ---------------------------------------------------------------- streaming units
// A streaming CTA has eight compute warps (warp w owns chunk w of every tile)
// and a control warp.  Per stage two mbarriers: full (the tile's copy and,
// for a run unit, its plan words have landed; the unit is described in
// sm.tk/kind/tma) and done (the eight compute warps finished the unit).  The
// control warp takes the tickets, issues the copies and runs each unit's
// epilogue (publishing the plan's aggregates or the tile's header), so the
// compute warps never wait for one another.
enum : int { U_PLAN = 0, U_RUN = 1, U_END = 2 };

// The plan's sums of this warp's chunk of tile t (fp32 images of the terms,
// their sum and |x| sum) into sm.wa[k][w].
__device__ __forceinline__ void chunk_sums_of(const uint64_t *xs, float &sig, float &ab) {
  sig = 0.0f;
  ab = 0.0f;
#pragma unroll
  for (int i = 0; i < kLaneTerms; i++) {
    const float f = approx_term_clamped((uint32_t)(xs[i] >> 32));
    sig += f;
    ab += fabsf(f);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    sig += __shfl_xor_sync(0xffffffffu, sig, o);
    ab += __shfl_xor_sync(0xffffffffu, ab, o);
  }
}
__device__ __noinline__ void chunk_aggregate(const Params &p, Smem &sm, const unsigned char *stage, int k,
                                             int64_t t, int64_t ntiles) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const TileGeo g = tile_geo(p, t, ntiles);
  const int64_t lstart = g.start + (int64_t)w * kChunkTerms + (int64_t)lane * kLaneTerms;
  const int nv = (int)max((int64_t)0, min((int64_t)kLaneTerms, g.end - lstart));
  uint64_t xs[kLaneTerms];
  load_lane(p, stage, sm.tma[k] != 0, (g.start >> 4) + w * 32 + lane, lstart, nv, w, lane, xs);
  float sig, ab;
  chunk_sums_of(xs, sig, ab);
  if (lane == 0) sm.wa[k][w] = WarpAgg{sig, ab, 0u, 0u};
}

// Control warp, after a plan unit: publish the tile's approximate sum (for
// its run unit) and, for the scanner, the same sum -- or s0 plus it for the
// first tile of a sum.
__device__ __noinline__ void plan_epilogue(const Params &p, Smem &sm, int k, int64_t t, int64_t ntiles) {
  const int lane = threadIdx.x & 31;
  if (!sq_ok(p, t >= 0 && t < p.cap_tiles, 6, t)) return;
  const TileGeo g = tile_geo(p, t, ntiles);
  WarpAgg a = WarpAgg{0.0f, 0.0f, 0u, 0u};
  if (lane < kWarps) a = sm.wa[k][lane];
  DF agg = DF{a.sig, 0.0f};
  float agga = a.ab;
#pragma unroll
  for (int o = kWarps / 2; o > 0; o >>= 1) {
    agg = df_add(agg, shfl_xor_df(agg, o));
    agga += __shfl_xor_sync(0xffffffffu, agga, o);
  }
  if (lane == 0) {
    publish_status(p.tagg + 2 * t, agg, agga, p.epoch, 0);     // the tile's own sum, for its run unit
    if (g.tile_in_sum != 0) {
      publish_status(p.status + 2 * t, agg, agga, p.epoch, 0);
    } else {
      const DF ex = df_from_double(p.s0s ? p.s0s[g.sum] : p.s0);
      publish_status(p.status + 2 * t, df_add(ex, agg), fabsf(ex.hi) + agga, p.epoch, 1);
    }
  }
}

// Compute warp w, a run unit: the exact run (or items) of chunk w of tile t
// under the binade its approximate prefix names; the chunk's record goes to
// sm.chunk[k][w] for the control warp's header.
__device__ __noinline__ void chunk_runs(const Params &p, Smem &sm, const unsigned char *stage, int k, int64_t t,
                                        int64_t ntiles, uint32_t &sums_ph) {
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const unsigned full = 0xffffffffu;
  unsigned int *st = sm.st;
  const TileGeo g = tile_geo(p, t, ntiles);
  const uint32_t tag0 = p.epoch << 1, tag1 = tag0 | 1u;
  // ---- the plan words: the prefix before the tile and the tile's own sums
  DF sp;
  float ap;
  if (t == g.first_tile) {
    sp = df_from_double(p.s0s ? p.s0s[g.sum] : p.s0);
    ap = fabsf(sp.hi);
  } else {
    const uint64_t A = sm.pre_raw[k][0], B = sm.pre_raw[k][1];
    if ((uint32_t)(A & 0xFF) == tag1 && (uint32_t)B == tag1) {
      sp = status_sum(A);
      ap = status_abs(B);
    } else {
      Prefix pr{DF{0.0f, 0.0f}, 0.0f};
      if (lane == 0) {
        const uint64_t tl = globaltimer();
        pr = read_prefix(p, g.sum, g.first_tile, t, st);
        atomicAdd(&st[S_NS_PREFIX_WAIT], (unsigned)(globaltimer() - tl));
      }
      sp = DF{__shfl_sync(full, pr.ex.hi, 0), __shfl_sync(full, pr.ex.lo, 0)};
      ap = __shfl_sync(full, pr.ex_abs, 0);
    }
  }
  uint64_t TA = sm.tagg_raw[k][0], TB = sm.tagg_raw[k][1];
  if (!((uint32_t)(TA & 0xFF) == tag0 && (uint32_t)TB == tag0)) {
    // not copied in time: wait for the plan unit's word (bounded)
    if (lane == 0) {
      const uint64_t t0 = globaltimer();
      while (true) {
        ld_vol_v2(p.tagg + 2 * t, TA, TB);
        if ((uint32_t)(TA & 0xFF) == tag0 && (uint32_t)TB == tag0) break;
        if (globaltimer() - t0 > kWaitNs) {
          note_timeout(p, ERR_PLAN_TIMEOUT, TO_TILESUM, (uint32_t)t, (uint32_t)((TA & 0xFF) | (p.epoch << 16)));
          break;
        }
        __nanosleep(32);
      }
      atomicAdd(&st[S_NS_PREFIX_WAIT], (unsigned)(globaltimer() - t0));
    }
    TA = __shfl_sync(full, TA, 0);
    TB = __shfl_sync(full, TB, 0);
  }
  const bool tagg_ok = (uint32_t)(TA & 0xFF) == tag0 && (uint32_t)TB == tag0;
  // ---- this lane's terms and the chunk's exact stats (the fast runs'
  // preconditions)
  const int64_t cstart = g.start + (int64_t)w * kChunkTerms;
  const int cnt_chunk = (int)max((int64_t)0, min((int64_t)kChunkTerms, g.end - cstart));
  const int64_t lstart = cstart + (int64_t)lane * kLaneTerms;
  const int nv = (int)max((int64_t)0, min((int64_t)kLaneTerms, g.end - lstart));
  uint64_t xs[kLaneTerms];
  load_lane(p, stage, sm.tma[k] != 0, (g.start >> 4) + w * 32 + lane, lstart, nv, w, lane, xs);
  WarpAgg me = WarpAgg{0.0f, 0.0f, 0u, 0u};
  {
    uint32_t orh = 0, orz = 0, mx = 0;
#pragma unroll
    for (int i = 0; i < kLaneTerms; i++) {
      const uint32_t hi = (uint32_t)(xs[i] >> 32);
      const uint32_t mag = hi & 0x7FFFFFFFu;
      orh |= hi;
      orz |= mag | (uint32_t)xs[i];
      mx = max(mx, mag);
    }
    me.mx = __reduce_max_sync(full, mx);
    me.flags = ((__reduce_or_sync(full, orh) >> 31) ? WA_NEG : 0u) | (__reduce_or_sync(full, orz) ? WA_NZ : 0u);
  }
  // ---- the binade: one for the whole tile when the prefix range of every
  // term in it stays inside one (the common case); else chunk by chunk
  DF sc = sp;
  float ac = ap;
  int e = 0;
  bool clean;
  {
    const DF tsd = status_sum(TA);
    const float c = sp.hi + sp.lo, ts = tsd.hi + tsd.lo, tab = status_abs(TB);
    const float P = 0.5f * (tab + ts), N = 0.5f * (tab - ts);
    const float delta = kEps * (ap + tab) + kRelF32 * (fabsf(c) + tab) + kTinyF;
    clean = tagg_ok && p.plan_mode == 0 && one_binade_f(c - N - delta, c + P + delta, e);
  }
  if (!clean) {
    // the same words reach every compute warp, so all of them come here;
    // they trade their chunks' sums through a per-stage barrier (bounded)
    float sig, ab;
    chunk_sums_of(xs, sig, ab);
    if (lane == 0) sm.wa[k][w] = WarpAgg{sig, ab, 0u, 0u};
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm.sums[k]);
    if (lane == 0) beat(p, sm.role, HB_WAIT_SUMS, (uint64_t)t);
    mbar_wait(p, &sm.sums[k], (sums_ph >> k) & 1u, ERR_PLAN_TIMEOUT, TO_SUMS, (uint32_t)t, (uint32_t)w);
    sums_ph ^= 1u << k;
    if (tid == 0) atomicAdd(&st[S_PLAN_LOCAL], 1u);
    for (int j = 0; j < w; j++) { sc = df_addf(sc, sm.wa[k][j].sig); ac += sm.wa[k][j].ab; }
    me.sig = sig;
    me.ab = ab;
    const float P = 0.5f * (ab + sig), N = 0.5f * (ab - sig);
    const float c = sc.hi + sc.lo;
    const float delta = kEps * (ac + ab) + kRelF32 * (fabsf(c) + ab) + kTinyF;
    clean = one_binade_f(c - N - delta, c + P + delta, e);
    clean = plan_override(p.plan_mode, clean, e, (uint64_t)t, w, 0);
  }
  Rec *area = p.items + t * kTileSlots;
  Rec crec;
  int nitems = 0;
  const bool zero_chunk = (me.flags & WA_NZ) == 0;
  if (clean || zero_chunk) {
    if (zero_chunk) e = 0;
    const int eb = e + 1023;
    const bool fast = !zero_chunk && e >= -969 && e <= 1023 && (int)(me.mx >> 20) < eb;
    Run r;
    bool general = true, general_reduce = true;
    if (fast) {
      const int c = 64 - eb;
      if ((me.flags & WA_NEG) == 0) {
        // non-negative terms: the run is a plain sum of increments
        uint64_t a = 0;
        bool anytie = false;
#pragma unroll
        for (int i = 0; i < kLaneTerms; i++) {
          uint64_t ri;
          bool tie;
          term_inc_fast((uint32_t)(xs[i] >> 32), (uint32_t)xs[i], c, ri, tie);
          a += ri;
          anytie |= tie;
        }
        if (__ballot_sync(0xffffffffu, anytie) == 0) {
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
          r.inc = (int64_t)a; r.lo = 0; r.hi = (int64_t)a; r.d = 0; r.flags = F_NONNEG;
          general = general_reduce = false;
        } else if (!anytie) {
          r.inc = (int64_t)a; r.lo = 0; r.hi = (int64_t)a; r.d = 0;
          r.flags = F_NONNEG | (nv == 0 ? (F_NONPOS | F_ZERO | F_ALLNEGZ) : 0u);
          general = false;
        }
      } else {
        // signed terms: positive and negative increments summed apart give
        // bounds for every prefix
        uint64_t P = 0, Nn = 0;
        bool anytie = false;
        uint32_t orl = 0, andl = 0xFFFFFFFFu;
#pragma unroll
        for (int i = 0; i < kLaneTerms; i++) {
          const uint32_t hi = (uint32_t)(xs[i] >> 32);
          uint64_t ri;
          bool tie;
          term_inc_fast(hi, (uint32_t)xs[i], c, ri, tie);
          if (hi >> 31) Nn += ri; else P += ri;
          anytie |= tie;
          if (i < nv) { orl |= hi; andl &= hi; }
        }
        if (!anytie) {
          if (nv == 0) {
            r = run_empty();
          } else {
            r.inc = (int64_t)(P - Nn); r.lo = -(int64_t)Nn; r.hi = (int64_t)P; r.d = 0;
            r.flags = ((orl >> 31) ? 0u : F_NONNEG) | ((andl >> 31) ? F_NONPOS : 0u);
          }
          general = false;
        }
      }
    }
    if (general) r = lane_run_general(p, stage, sm.tma[k] != 0, (g.start >> 4) + w * 32 + lane, lstart, nv, w, lane, e);
    if (general_reduce) {
#pragma unroll 1
      for (int off = 1; off < 32; off <<= 1) {
        const Run o = shfl_run<SH_DOWN>(r, off);
        if ((lane & (2 * off - 1)) == 0) r = run_compose(r, o);
      }
    }
    crec = make_rec(r, (r.flags & F_ZERO) ? kZeroE : e, K_RUN, (uint32_t)cnt_chunk, (uint32_t)(w * kChunkTerms));
    if (lane == 0) atomicAdd(&st[S_CHUNK_RUN], 1u);
  } else {
    nitems = split_chunk(p, stage, sm.tma[k] != 0, (g.start >> 4) + w * 32 + lane, lstart, nv, w, lane, sc, ac,
                         (uint64_t)t, area, st);
    if (nitems == 0) {
      Run fr = run_empty();
      fr.flags = ((me.mx >= 0x7FF00000u) ? (F_HASINF_P | F_HASINF_N | F_HASNAN) : 0u);
      crec = make_rec(fr, 0, K_FALLBACK, (uint32_t)cnt_chunk, (uint32_t)(w * kChunkTerms));
      if (lane == 0) {
        if (item_ok(p, area + w * kChunkSlots, 7)) stcg_rec(area + w * kChunkSlots, crec);
        atomicAdd(&st[S_POOL_OVERFLOW], 1u);
      }
      nitems = 1;
    } else if (lane == 0) {
      atomicAdd(&st[S_CHUNK_LIST], 1u);
      atomicAdd(&st[S_ITEMS], (unsigned)nitems);
    }
    crec.meta = rec_meta(0, 0, K_COMPLEX, 0);
  }
  if (lane == 0) {
    sm.chunk[k][w] = crec;
    sm.nitems[k][w] = nitems;
  }
}

// Control warp, after a run unit: the tile's header -- one run when every
// chunk is a run of one binade (runs of zeros fit any), else the chunks'
// items in the tile's item area.
__device__ __noinline__ void run_epilogue(const Params &p, Smem &sm, int k, int64_t t, int64_t ntiles) {
  const int lane = threadIdx.x & 31;
  unsigned int *st = sm.st;
  const TileGeo g = tile_geo(p, t, ntiles);
  Rec *area = p.items + t * kTileSlots;
  const unsigned full = 0xffffffffu;
  Rec c = make_rec(run_empty(), kZeroE, K_RUN, 0, 0);
  int n = 0;
  if (lane < kWarps) { c = sm.chunk[k][lane]; n = sm.nitems[k][lane]; }
  const uint32_t kind = rec_kind(c.meta), flags = rec_flags(c.meta);
  const bool nz_run = lane < kWarps && kind == K_RUN && !(flags & F_ZERO);
  const uint32_t nzm = __ballot_sync(full, nz_run);
  const int et = nzm ? __shfl_sync(full, (int)c.e, __ffs(nzm) - 1) : kZeroE;
  const bool mixed = lane < kWarps && (kind != K_RUN || (nz_run && c.e != et));
  Rec hd;
  if (__ballot_sync(full, mixed) == 0) {
    Run r = rec_run(c);
#pragma unroll
    for (int off = 1; off < kWarps; off <<= 1) {
      const Run o = shfl_run<SH_DOWN>(r, off);
      if ((lane & (2 * off - 1)) == 0) r = run_compose(r, o);
    }
    // the header alone holds the tile: nothing to order before it
    hd = make_rec(r, (r.flags & F_ZERO) ? kZeroE : et, K_RUN, (uint32_t)(g.end - g.start), 0);
  } else {
    if (lane < kWarps && kind == K_RUN) {
      n = 0;
      if (c.count > 0) {
        if (item_ok(p, area + lane * kChunkSlots, 8)) stcg_rec(area + lane * kChunkSlots, c);
        n = 1;
      }
    }
    const uint64_t mine = (lane < kWarps) ? (uint64_t)(uint32_t)n << (kCountBits * lane) : 0ull;
    const uint64_t packed = ((uint64_t)__reduce_or_sync(full, (uint32_t)(mine >> 32)) << 32) |
                            __reduce_or_sync(full, (uint32_t)mine);
    const uint32_t orf = __reduce_or_sync(full, lane < kWarps ? flags : 0u);
    Run z = run_empty();
    z.inc = (int64_t)packed;
    z.flags = orf & (F_HASINF_P | F_HASINF_N | F_HASNAN);
    hd = make_rec(z, 0, K_COMPLEX, (uint32_t)(g.end - g.start), 0);
    hd.inc = (int64_t)packed;
    __syncwarp();
    // the items the compute warps wrote (ordered before their arrival on
    // the stage's done barrier) and this warp's are ordered before the
    // header by this device-scope fence (a fence is cumulative)
    if (lane == 0) {
      __threadfence();
      atomicAdd(&st[S_TILE_COMPLEX], 1u);
    }
  }
  if (lane == 0) {
    if (sq_ok(p, t >= 0 && t < p.cap_tiles, 9, t)) publish_header(p.hdr + t, hd, (p.epoch << 1) | 1u);
    atomicMax(&p.stats[S_T_STREAM_END], (unsigned long long)globaltimer());
    atomicAdd(&st[S_TILES], 1u);
  }
}

// ---------------------------------------------------------------- the walk
__device__ __forceinline__ bool nonfinite(uint64_t Sb) { return ((Sb >> 52) & 0x7FF) == 0x7FF; }

// S is inf or NaN: the rest of the sum only decides between that value and
// NaN, from the flags (inf + -inf and anything + NaN give NaN).
__device__ __forceinline__ uint64_t absorb(uint64_t Sb, uint32_t flags) {
  const bool isnan = (Sb & 0x000FFFFFFFFFFFFFull) != 0;
  if (isnan) return Sb;
  const bool neg = (Sb >> 63) != 0;
  if ((flags & F_HASNAN) || (neg ? (flags & F_HASINF_P) : (flags & F_HASINF_N)))
    return dbits(__dadd_rn(bitsd(Sb), -bitsd(Sb)));     // inf + -inf: the device's NaN
  return Sb;
}

// Term-by-term fallback over x[a, a + cnt), run by a whole warp; every lane
// ends with the same S.  One __dadd_rn per term, in index order.
__device__ __noinline__ uint64_t add_terms(const Params &p, uint64_t Sb, int64_t a, int64_t cnt, unsigned int *st) {
  const int lane = threadIdx.x & 31;
  const uint64_t t0 = globaltimer();
  double S = bitsd(Sb);
  if (!sq_ok(p, a >= 0 && a + cnt <= p.n, 10, a)) cnt = 0;
  for (int64_t base = 0; base < cnt; base += 32) {
    const double v = (base + lane < cnt) ? __ldg(p.x + a + base + lane) : 0.0;
    const int m = (int)min((int64_t)32, cnt - base);
    for (int j = 0; j < m; j++) S = __dadd_rn(S, __shfl_sync(0xffffffffu, v, j));
  }
  if (lane == 0) {
    atomicAdd(&st[S_TERMS_ADDED], (unsigned)cnt);
    atomicAdd(&st[S_NS_WALK_ADDS], (unsigned)(globaltimer() - t0));
  }
  return dbits(S);
}

__device__ __forceinline__ bool elem_alone(const Rec &q) { return rec_kind(q.meta) != K_RUN; }

// Self-checking builds keep a trace of the walk: per serial step the term
// range [a, b) it covered, what it was, and the running sum after it.
#ifdef SEQSUM_CHECKS
constexpr int kDbgWords = 16384;
__device__ __forceinline__ void walk_trace(const Params &p, int64_t a, int64_t b, uint32_t what, uint64_t Sb) {
  const unsigned long long r = atomicAdd(&p.dbg[0], 1ull);
  if (1 + 4 * (r + 1) <= (unsigned long long)kDbgWords) {
    p.dbg[1 + 4 * r] = (unsigned long long)a;
    p.dbg[2 + 4 * r] = (unsigned long long)b;
    p.dbg[3 + 4 * r] = what;
    p.dbg[4 + 4 * r] = Sb;
  }
}
#define WALK_TRACE(a, b, what, Sb) do { if (lane == 0) walk_trace(p, (a), (b), (what), (Sb)); } while (0)
#else
#define WALK_TRACE(a, b, what, Sb) do { } while (0)
#endif
__device__ __forceinline__ int elem_key(const Rec &q) {
  return (rec_flags(q.meta) & F_ZERO) ? kZeroE : (int)q.e;
}

// The in-order pass met a segment whose composite the check refused: find the
// first element whose prefix composite the check refuses (the warp composes 32
// prefixes at a time), apply the prefix before it, and add that element's
// terms one by one.  The bounds of a composite depend on the shape of its
// tree, so this composition may accept what the scan's refused; then the whole
// segment is applied as composed here and -1 returned.  Else returns the
// element added term by term; Sb is the exact sum after it.  Whole warp.
__device__ __noinline__ int resolve_rejection(const Params &p, const Rec *el, const uint32_t *elpos, int segstart,
                                              int ei, int e, int64_t pos, int64_t ntiles, unsigned int *st,
                                              uint64_t &Sb) {
  const unsigned full = 0xffffffffu;
  const int lane = threadIdx.x & 31;
  int kfail = -1;
  Run racc = run_empty(), before = run_empty();
  for (int c0 = segstart; c0 <= ei; c0 += 32) {
    const int i = c0 + lane;
    Run r = (i <= ei) ? rec_run(el[i]) : run_empty();
#pragma unroll 1
    for (int o = 1; o < 32; o <<= 1) {
      const Run ov = shfl_run<SH_UP>(r, o);
      if (lane >= o) r = run_compose(ov, r);
    }
    const Run pre = run_compose(racc, r);
    bool bad = false;
    if (i <= ei) { uint64_t T = Sb; bad = run_apply(T, pre, e) != APPLY_OK; }
    const uint32_t bm = __ballot_sync(full, bad);
    if (bm) {
      kfail = c0 + __ffs(bm) - 1;
      const int src = kfail - 1 - c0;
      before = shfl_run<SH_IDX>(pre, src < 0 ? 0 : src);
      if (src < 0) before = racc;
      break;
    }
    racc = shfl_run<SH_IDX>(pre, 31);
  }
  if (kfail < 0) {
    uint64_t T = Sb;
    if (run_apply(T, racc, e) == APPLY_OK) {
      Sb = T;
      return -1;
    }
    kfail = segstart;                                  // not reached: the last prefix passed
  } else if (kfail > segstart) {
    uint64_t T = Sb;
    if (run_apply(T, before, e) == APPLY_OK) Sb = T;
    else kfail = segstart;                             // not reached: that prefix passed
  }
  const uint32_t ep = elpos[kfail];
  const TileGeo g = tile_geo(p, pos + (ep >> 12), ntiles);
  Sb = add_terms(p, Sb, g.start + (ep & 0xFFF), el[kfail].count, st);
  return kfail;
}

#ifdef SEQSUM_PROFILE
// Cycle profile of the walk (profiling builds): cycles since the previous
// point, summed per point, for thread 0 and for thread 224 (warp 7).
#define WALK_PT(id)                                                                        \
  do {                                                                                     \
    if (tid == 0 || tid == 224) {                                                          \
      const long long now_ = clock64();                                                    \
      atomicAdd(&p.dbg[15000 + 2 * (id) + (tid ? 1 : 0)], (unsigned long long)(now_ - prof_t)); \
      prof_t = now_;                                                                       \
    }                                                                                      \
  } while (0)
#else
#define WALK_PT(id) do { } while (0)
#endif

// Walk sum k over its tiles [tb, te), as the headers appear.  Whole CTA (256
// threads); the in-order pass runs on warp 0.  Per batch of up to 1024 ready
// tiles: the headers are staged, the elements (simple tile headers, the items
// of complex tiles) listed in order, every maximal run of same-binade run
// elements composed by a segmented scan, and the segments applied in order.
// The dynamic shared memory of a walking CTA (it never copies tiles) holds:
//   [0, 32K)       the batch's headers (thread t: tiles 4t..4t+3), later the
//                  segment composites
//   [32K, 64K)     the batch's elements in order
//   [64K, 68K)     per element: its tile in the batch << 12 | its first term
//   [68K, 72K)     segment ends
__device__ __noinline__ void walk_sum(const Params &p, Smem &sm, unsigned char *dyn, int k, int64_t tb, int64_t te,
                                      int64_t ntiles) {
  constexpr int PT = kWalkTiles / kThreads;         // tiles, then elements, per thread
  static_assert(kWalkTiles == kThreads * PT && kWalkElems == kThreads * PT, "walk batch shape");
  Rec *hdrs = reinterpret_cast<Rec *>(dyn);
  Rec *comp = hdrs;
  Rec *el = reinterpret_cast<Rec *>(dyn + kWalkOffEl);
  uint32_t *elpos = reinterpret_cast<uint32_t *>(dyn + kWalkOffPos);
  int *ends = reinterpret_cast<int *>(dyn + kWalkOffEnds);
  unsigned int *st = sm.st;
  const unsigned full = 0xffffffffu;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t tag = (p.epoch << 1) | 1u;
  if (tid == 0) sm.S = dbits(p.s0s ? p.s0s[k] : p.s0);
  int64_t pos = tb;
  uint64_t t_work0 = 0;
#ifdef SEQSUM_PROFILE
  long long prof_t = clock64();
#endif
  wide_sync(p, sm, 6);
  while (pos < te) {
    // ---- A. the ready run of headers [pos, pos + m)
    const int want = (int)min((int64_t)kWalkTiles, te - pos);
    const uint64_t t0 = globaltimer();
    if (tid == 0) {
      if (t_work0 != 0) atomicAdd(&st[S_NS_WALK_WORK], (unsigned)(t0 - t_work0));
      beat(p, sm.role, HB_WAIT_HEADERS, (uint64_t)pos);
    }
    int m;
    while (true) {
      uint64_t w[PT][4];
#pragma unroll
      for (int q = 0; q < PT; q++) {
        const int i = PT * tid + q;
        w[q][0] = w[q][1] = w[q][2] = w[q][3] = 0;
        if (i < want && sq_ok(p, pos + i < p.cap_tiles, 11, pos + i)) {
          ld_vol_v2(p.hdr + pos + i, w[q][0], w[q][1]);
          ld_vol_v2(reinterpret_cast<const char *>(p.hdr + pos + i) + 16, w[q][2], w[q][3]);
        }
      }
      int gap = want;                                  // this thread's first tile not (fully) published
#pragma unroll
      for (int q = PT - 1; q >= 0; q--) {
        const int i = PT * tid + q;
        const int nt = ((uint32_t)(w[q][0] >> 56) == tag) + ((uint32_t)(w[q][1] >> 56) == tag) +
                       ((uint32_t)(w[q][2] >> 56) == tag) + ((uint32_t)((w[q][3] >> 24) & 0xFFu) == tag);
        if (i < want && nt != 4) {
          gap = i;
          if (nt != 0) atomicAdd(&st[S_TORN_HEADER], 1u);
        }
      }
#pragma unroll
      for (int q = 0; q < PT; q++) {
        const int i = PT * tid + q;
        if (i < gap) {
          Rec h;
          h.inc = untag56(w[q][0]);
          h.lo = untag56(w[q][1]);
          h.hi = untag56(w[q][2]);
          h.meta = (uint32_t)w[q][3] & 0x00FFFFFFu;
          h.e = (int16_t)(uint16_t)(w[q][3] >> 32);
          h.count = (uint16_t)(w[q][3] >> 48);
          hdrs[i] = h;
        }
      }
      const int wm = (int)__reduce_min_sync(full, (uint32_t)gap);
      if (lane == 0) sm.walk_m[warp] = wm;
      wide_sync(p, sm, 7);
      m = want;
#pragma unroll
      for (int w2 = 0; w2 < kWarps; w2++) m = min(m, sm.walk_m[w2]);
      // a batch costs about the same whatever its size (its steps are
      // latency-bound), so the walk takes full batches: 1024 tiles, or the
      // rest of the sum
      if (m == want) break;
      // not all ready yet; thread 0 alone decides whether to give up
      if (tid == 0) sm.restart = (globaltimer() - t0 > kWaitNs) ? 1 : 0;
      wide_sync(p, sm, 8);
      if (sm.restart) {
        if (tid == 0) {
          note_timeout(p, ERR_WALK_TIMEOUT, TO_WALK, (uint32_t)pos, (uint32_t)want);
          p.outs[k] = __longlong_as_double(0x7FF8000000000000ll);
        }
        wide_sync(p, sm, 9);
        return;
      }
      __nanosleep(500);
    }
    WALK_PT(1);                                        // waiting for headers
    {
      // a thread that saw a complex header orders the tile's items (read
      // later, after barriers, by any thread) after it
      bool saw_complex = false;
#pragma unroll
      for (int q = 0; q < PT; q++)
        if (PT * tid + q < m && rec_kind(hdrs[PT * tid + q].meta) == K_COMPLEX) saw_complex = true;
      if (saw_complex) __threadfence();
    }
    if (tid == 0) {
      beat(p, sm.role, HB_BATCH, ((uint64_t)m << 32) | (uint32_t)pos);
      atomicAdd(&st[S_WALK_BATCHES], 1u);
      t_work0 = globaltimer();
      atomicAdd(&st[S_NS_WALK_WAIT], (unsigned)(t_work0 - t0));
      if (pos + m >= te) p.stats[S_T_WALK0] = t_work0;
    }
    // ---- B. elements per tile and their offsets; a batch whose elements do
    //         not fit is cut before the first tile that overflows
    int cnt[PT];
    int off0 = 0, nel = 0;
    for (int pass = 0; pass < 2; pass++) {
      int mine = 0;
#pragma unroll
      for (int q = 0; q < PT; q++) {
        const int i = PT * tid + q;
        int c = 0;
        if (i < m) {
          const Rec &h = hdrs[i];
          if (rec_kind(h.meta) == K_COMPLEX) {
            const uint64_t packed = (uint64_t)h.inc;
#pragma unroll
            for (int cc = 0; cc < kWarps; cc++) c += (int)((packed >> (kCountBits * cc)) & kCountMask);
          } else {
            c = 1;
            (void)sq_ok(p, h.count >= 1 && h.count <= kTileTerms, 18, h.count);
          }
        }
        cnt[q] = c;
        mine += c;
      }
      int incl = mine;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(full, incl, o);
        if (lane >= o) incl += v;
      }
      if (lane == 31) sm.wcnt[warp] = incl;
      wide_sync(p, sm, 10);
      int wbase = 0;
      nel = 0;
#pragma unroll
      for (int w2 = 0; w2 < kWarps; w2++) {
        const int v = sm.wcnt[w2];
        wbase += (w2 < warp) ? v : 0;
        nel += v;
      }
      off0 = wbase + incl - mine;
      if (nel <= kWalkElems) break;
      // (rare) the first tile whose elements would not fit ends the batch
      int cut = m, o = off0;
#pragma unroll
      for (int q = 0; q < PT; q++) {
        const int i = PT * tid + q;
        if (i < m && o + cnt[q] > kWalkElems && cut == m) cut = i;
        o += cnt[q];
      }
      const int wc = (int)__reduce_min_sync(full, (uint32_t)cut);
      wide_sync(p, sm, 11);                            // every thread has read sm.wcnt
      if (lane == 0) sm.walk_m[warp] = wc;
      wide_sync(p, sm, 12);
#pragma unroll
      for (int w2 = 0; w2 < kWarps; w2++) m = min(m, sm.walk_m[w2]);
    }
    WALK_PT(2);                                        // counts and offsets
    uint64_t tsec = 0;
    if (tid == 0) { tsec = globaltimer(); atomicAdd(&st[S_NS_WALK_COUNT], (unsigned)(tsec - t_work0)); }
    // ---- C. the ordered elements: simple headers by their thread; for a
    //         complex tile its thread marks the items' places, and the block
    //         loads the items, one per thread
    {
      int off = off0;
#pragma unroll
      for (int q = 0; q < PT; q++) {
        const int i = PT * tid + q;
        if (i < m) {
          const Rec h = hdrs[i];
          if (rec_kind(h.meta) != K_COMPLEX) {
            if (sq_ok(p, off >= 0 && off < kWalkElems, 12, off)) {
              el[off] = h;
              elpos[off] = (uint32_t)i << 12;
            }
          } else {
            const uint64_t packed = (uint64_t)h.inc;
            int o2 = off;
            for (int cc = 0; cc < kWarps; cc++) {
              const int n = (int)((packed >> (kCountBits * cc)) & kCountMask);
              for (int u = 0; u < n; u++) {
                if (sq_ok(p, o2 >= 0 && o2 < kWalkElems && u < kChunkSlots, 13, ((int64_t)o2 << 32) | (u << 8) | cc))
                  elpos[o2] = 0x80000000u | ((uint32_t)i << 12) | ((uint32_t)cc << 8) | (uint32_t)u;
                o2++;
              }
            }
          }
        }
        off += cnt[q];
      }
    }
    WALK_PT(3);                                        // placing elements
    wide_sync(p, sm, 13);
    WALK_PT(4);
    for (int j = tid; j < nel; j += kThreads) {
      const uint32_t ep = elpos[j];
      if (ep & 0x80000000u) {
        const uint32_t i = (ep >> 12) & 0x7FFFFu, cc = (ep >> 8) & 0xFu, u = ep & 0xFFu;
        const Rec *src = p.items + (pos + i) * kTileSlots + cc * kChunkSlots + u;
        if (item_ok(p, src, 14)) {
          Rec it = ldcg_rec(src);
          if (!sq_ok(p, rec_kind(it.meta) != K_COMPLEX && it.count >= 1 &&
                            rec_tstart(it.meta) + it.count <= (uint32_t)kTileTerms,
                     17, ((int64_t)it.meta << 16) | it.count)) {
            it = make_rec(run_empty(), kZeroE, K_RUN, 0, 0);
          }
          el[j] = it;
          elpos[j] = (i << 12) | rec_tstart(it.meta);
        }
      }
    }
    WALK_PT(5);                                        // loading items
    wide_sync(p, sm, 14);
    WALK_PT(6);
    if (tid == 0) { const uint64_t t2 = globaltimer(); atomicAdd(&st[S_NS_WALK_GATHER], (unsigned)(t2 - tsec)); tsec = t2; }
    // ---- D. segmented scan of elements [from, nel) and E. the in-order
    //         pass (again from the element after a rejected run's failure)
    int from = 0;
    while (from < nel) {
      if (lane == 0) beat(p, sm.role, HB_SCAN, ((uint64_t)nel << 32) | ((uint64_t)from << 16) | (uint32_t)(pos & 0xFFFF));
      const int j0 = PT * tid;
      // pass 1: this thread's elements in order -- heads (an element alone,
      // or a binade change, starts a segment) and the composite since the
      // last head
      int pkey = 0;
      bool palone = true;
      if (j0 - 1 >= from && j0 - 1 < nel) {
        const Rec pq = el[j0 - 1];
        pkey = elem_key(pq);
        palone = elem_alone(pq);
      }
      Run acc = run_empty();
      uint32_t hdmask = 0, valmask = 0;                // bit q: element j0 + q starts a segment / is walked
      int lastkey = 0;
      bool lastalone = true;
#pragma unroll 1
      for (int q = 0; q < PT; q++) {
        const int j = j0 + q;
        if (j < from || j >= nel) continue;
        const Rec x = el[j];
        const int kx = elem_key(x);
        const bool ax = elem_alone(x);
        const int kp = (q == 0 || !(valmask & 1u << (q - 1))) ? pkey : lastkey;
        const bool ap = (q == 0 || !(valmask & 1u << (q - 1))) ? palone : lastalone;
        const bool h = (j == from) || ax || ap || kp != kx;
        const Run r = rec_run(x);
        acc = h ? r : run_compose(acc, r);
        valmask |= 1u << q;
        if (h) hdmask |= 1u << q;
        lastkey = kx;
        lastalone = ax;
      }
      // segment ends: the last element, or one whose successor starts a segment
      const int nhd0 = __shfl_down_sync(full, (int)(hdmask & 1u), 1);
      bool next_head_last = true;
      if (lane < 31) {
        next_head_last = nhd0 != 0;
      } else if (j0 + PT < nel) {
        const Rec xn = el[j0 + PT];
        next_head_last = elem_alone(xn) || lastalone || elem_key(xn) != lastkey;
      }
      uint32_t endmask = 0;
#pragma unroll 1
      for (int q = 0; q < PT; q++) {
        const int j = j0 + q;
        const bool nh = (q + 1 < PT) ? ((hdmask >> (q + 1)) & 1u) != 0 : next_head_last;
        if ((valmask >> q) & 1u && (j == nel - 1 || nh)) endmask |= 1u << q;
      }
      const int my = __popc(endmask);
      // across the warp: (head seen, composite) and the end counts
      Run v = acc;
      int f = hdmask ? 1 : 0;
      int ie = my;
#pragma unroll 1
      for (int o = 1; o < 32; o <<= 1) {
        const Run ov = shfl_run<SH_UP>(v, o);
        const int of = __shfl_up_sync(full, f, o);
        const int oe = __shfl_up_sync(full, ie, o);
        if (lane >= o) {
          if (!f) v = run_compose(ov, v);
          f |= of;
          ie += oe;
        }
      }
      if (lane == 31) { sm.wagg[warp] = v; sm.wflag[warp] = f; sm.wcnt[warp] = ie; }
      WALK_PT(7);                                      // local and warp composition
      wide_sync(p, sm, 15);
      WALK_PT(8);
      // the composite before this thread's first element: earlier warps, then
      // earlier lanes of this warp
      Run ex = run_empty();
      int eb = 0, nseg = 0;
#pragma unroll 1
      for (int w2 = 0; w2 < kWarps; w2++) {
        if (w2 < warp) {
          if (sm.wflag[w2]) ex = sm.wagg[w2];
          else ex = run_compose(ex, sm.wagg[w2]);
          eb += sm.wcnt[w2];
        }
        nseg += sm.wcnt[w2];
      }
      {
        const Run lv = shfl_run<SH_UP>(v, 1);
        const int lf = __shfl_up_sync(full, f, 1);
        if (lane >= 1) {
          if (lf) ex = lv;
          else ex = run_compose(ex, lv);
        }
      }
      // pass 2: each segment end's composite (again in order from the
      // thread's first element), in order into the segment list
      int epos = eb + ie - my;
      Run cur = ex;
#pragma unroll 1
      for (int q = 0; q < PT; q++) {
        const int j = j0 + q;
        if (!((valmask >> q) & 1u)) continue;
        const Rec x = el[j];
        const Run r = rec_run(x);
        cur = ((hdmask >> q) & 1u) ? r : run_compose(cur, r);
        if ((endmask >> q) & 1u) {
          if (sq_ok(p, epos < kWalkElems, 15, epos)) {
            ends[epos] = j;
            comp[epos] = make_rec(cur, x.e, rec_kind(x.meta), x.count, rec_tstart(x.meta));
          }
          epos++;
        }
      }
      WALK_PT(9);                                      // cross-warp prefix, segment list
      WALK_PT(10);
      WALK_PT(11);
      wide_sync(p, sm, 17);
      WALK_PT(12);
      if (tid == 0) { const uint64_t t2 = globaltimer(); atomicAdd(&st[S_NS_WALK_SCAN], (unsigned)(t2 - tsec)); tsec = t2; }
      // ---- E. the in-order pass (warp 0)
#ifdef SEQSUM_CHECKS
      auto abs_start = [&](int j) -> int64_t {
        const uint32_t ep = elpos[j];
        return tile_geo(p, pos + (ep >> 12), ntiles).start + (ep & 0xFFF);
      };
#endif
      if (warp == 0) {
        uint64_t Sb = sm.S;
        int restart = -1;
        int segstart = from;
        unsigned nterms = 0, nrej = 0;
        for (int sidx = 0; sidx < nseg; sidx++) {
          const int ei = ends[sidx];
          const Rec c = comp[sidx];
          const uint32_t kind = rec_kind(c.meta);
          if (nonfinite(Sb)) {
            Sb = absorb(Sb, rec_flags(c.meta));
            WALK_TRACE(abs_start(segstart), abs_start(ei) + el[ei].count, 6u, Sb);
            segstart = ei + 1;
            continue;
          }
          if (kind == K_TERMS) {
            const Rec q = el[ei];
            double S = bitsd(Sb);
            const int nt = (int)q.count;
            if (nt > 0) S = __dadd_rn(S, bitsd((uint64_t)q.inc));
            if (nt > 1) S = __dadd_rn(S, bitsd((uint64_t)q.lo));
            if (nt > 2) S = __dadd_rn(S, bitsd((uint64_t)q.hi));
            Sb = dbits(S);
            nterms += (unsigned)nt;
            WALK_TRACE(abs_start(ei), abs_start(ei) + nt, 2u, Sb);
            segstart = ei + 1;
            continue;
          }
          if (kind == K_FALLBACK) {
            const uint32_t ep = elpos[ei];
            const TileGeo g = tile_geo(p, pos + (ep >> 12), ntiles);
            Sb = add_terms(p, Sb, g.start + (ep & 0xFFF), c.count, st);
            if (lane == 0) atomicAdd(&st[S_CHUNK_FALLBACK], 1u);
            WALK_TRACE(abs_start(ei), abs_start(ei) + c.count, 1u, Sb);
            segstart = ei + 1;
            continue;
          }
          {
            uint64_t T = Sb;
            if (run_apply(T, rec_run(c), c.e) == APPLY_OK) {
              Sb = T;
              WALK_TRACE(abs_start(segstart), abs_start(ei) + el[ei].count, 0u | ((uint32_t)(c.e & 0xFFFF) << 16), Sb);
              segstart = ei + 1;
              continue;
            }
          }
          nrej++;
          const int kfail = resolve_rejection(p, el, elpos, segstart, ei, c.e, pos, ntiles, st, Sb);
          if (kfail < 0) {                             // the segment applied as composed here
            segstart = ei + 1;
            continue;
          }
          if (kfail < ei) { restart = kfail + 1; break; }
          segstart = ei + 1;
        }
        // every lane has read sm.S (at the top of the pass) before lane 0
        // replaces it: the lanes of a warp do not run in lockstep, and a lane
        // that reads the new value would walk the segments from the wrong sum
        __syncwarp();
        if (lane == 0) {
          sm.S = Sb;
          sm.restart = restart;
          atomicAdd(&st[S_WALK_SEGMENTS], (unsigned)nseg);
          if (nterms) atomicAdd(&st[S_TERMS_ADDED], nterms);
          if (nrej) atomicAdd(&st[S_RUN_REJECTED], nrej);
          const uint64_t t2 = globaltimer();
          atomicAdd(&st[S_NS_WALK_SERIAL], (unsigned)(t2 - tsec));
          tsec = t2;
        }
      }
      WALK_PT(13);                                     // the in-order pass (warp 0)
      wide_sync(p, sm, 18);
      WALK_PT(14);
      const int rs = sm.restart;
      if (rs < 0) break;
      from = rs;
    }
    pos += m;
    wide_sync(p, sm, 19);
    WALK_PT(15);
  }
  if (tid == 0) {
    p.outs[k] = bitsd(sm.S);
    const uint64_t tend = globaltimer();
    p.stats[S_T_WALK1] = tend;
    if (t_work0 != 0) atomicAdd(&st[S_NS_WALK_WORK], (unsigned)(tend - t_work0));
  }
  wide_sync(p, sm, 20);
}

// ---------------------------------------------------------------- the streaming loops

// Compute warps: the units of the stages in turn, until the control warp
// marks the end.
__device__ __noinline__ void compute_loop(const Params &p, Smem &sm, const unsigned char *dyn, int64_t ntiles) {
  const int tid = threadIdx.x, lane = tid & 31;
  uint32_t ph = 0;                                       // bit k: parity of full[k]
  uint32_t sums_ph = 0;                                  // bit k: parity of sums[k]
  for (int j = 0;; j++) {
    const int k = j % kStages;
    const uint64_t tw = (tid == 0) ? globaltimer() : 0;
    if (lane == 0) beat(p, sm.role, HB_WAIT_UNIT, (uint64_t)j);
    if (!mbar_wait(p, &sm.full[k], (ph >> k) & 1u, ERR_TMA_TIMEOUT, TO_FULL, (uint32_t)j,
                   (uint32_t)(k | (tid >> 5) << 8 | blockIdx.x << 16)))
      break;                                             // the call has failed
    ph ^= 1u << k;
    if (tid == 0) atomicAdd(&sm.st[S_NS_TMA_WAIT], (unsigned)(globaltimer() - tw));
    const int kind = sm.kind[k];
    if (kind == U_END) break;
    const int64_t t = sm.tk[k];
    const unsigned char *stage = dyn + k * kStageBytes;
    const uint64_t tb = (tid == 0) ? globaltimer() : 0;
    if (lane == 0) beat(p, sm.role, HB_UNIT, ((uint64_t)j << 32) | (uint32_t)t);
    if (kind == U_PLAN) {
      chunk_aggregate(p, sm, stage, k, t, ntiles);
      if (tid == 0) atomicAdd(&sm.st[S_NS_PHASE_A], (unsigned)(globaltimer() - tb));
    } else {
      chunk_runs(p, sm, stage, k, t, ntiles, sums_ph);
      if (tid == 0) atomicAdd(&sm.st[S_NS_PHASE_B], (unsigned)(globaltimer() - tb));
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm.done[k]);
  }
}

// The control warp: tickets, copies, plan words and epilogues.
__device__ __noinline__ void control_loop(const Params &p, Smem &sm, unsigned char *dyn, const CUtensorMap *tmap,
                                          int64_t ntiles) {
  const int lane = threadIdx.x & 31;
  const int64_t nunits = 2 * ntiles;
  uint32_t u_next = 0;                                   // lane 0: the next ticket, taken one unit ahead
  if (lane == 0) u_next = atomicAdd(&p.ctr[C_TICKET], 1u);
  uint32_t ph = 0;                                       // bit k: parity of done[k]
  auto epilogue = [&](int k) -> bool {
    const uint64_t tw = globaltimer();
    if (lane == 0) beat(p, sm.role + 0x80u, HB_WAIT_DONE, ((uint64_t)k << 32) | (uint32_t)sm.tk[k]);
    if (!mbar_wait(p, &sm.done[k], (ph >> k) & 1u, ERR_TMA_TIMEOUT, TO_DONE, (uint32_t)sm.tk[k],
                   (uint32_t)(k | sm.kind[k] << 8 | blockIdx.x << 16)))
      return false;
    ph ^= 1u << k;
    if (lane == 0) atomicAdd(&sm.st[S_NS_CTRL_WAIT], (unsigned)(globaltimer() - tw));
    if (sm.kind[k] == U_PLAN) plan_epilogue(p, sm, k, sm.tk[k], ntiles);
    else run_epilogue(p, sm, k, sm.tk[k], ntiles);
    return true;
  };
  for (int j = 0;; j++) {
    const int k = j % kStages;
    if (j >= kStages && !epilogue(k)) break;             // the unit that held this stage (else the call failed)
    uint32_t u = 0;
    if (lane == 0) {
      u = u_next;
      u_next = atomicAdd(&p.ctr[C_TICKET], 1u);          // used at the next unit: its latency overlaps
    }
    u = __shfl_sync(0xffffffffu, u, 0);
    if ((int64_t)u >= nunits) {
      if (lane == 0) sm.kind[k] = U_END;
      __syncwarp();
      if (lane < 3) mbar_arrive(&sm.full[k]);          // all three arrivals at once
      for (int jj = max(j - kStages + 1, 0); jj < j; jj++)
        if (!epilogue(jj % kStages)) break;
      break;
    }
    int64_t t;
    const bool plan = unit_of((int64_t)u, ntiles, p.wave, t);
    const TileGeo g = tile_geo(p, t, ntiles);
    const bool tma = p.tma_rows != 0 && (g.start & 15) == 0;
    // lanes 0 and 1 make two of the stage's three arrivals when their
    // copies (a run unit's plan words: the tile's own sum and the prefix of
    // the tile before; none for a plan unit) have landed
    if (!plan) {
      if (lane == 0) cp_async16(sm.tagg_raw[k], p.tagg + 2 * t);
      else if (lane == 1 && t > 0) cp_async16(sm.pre_raw[k], p.status + 2 * (t - 1));
    }
    if (lane < 2) cp_async_mbar_arrive(&sm.full[k]);
    __syncwarp();
    if (lane == 0) {
      sm.tk[k] = t;
      sm.kind[k] = plan ? U_PLAN : U_RUN;
      sm.tma[k] = tma ? 1 : 0;
      if (tma) {
        fence_proxy_async();                             // the compute warps' reads of this stage came first
        mbar_arrive_expect_tx(&sm.full[k], (uint32_t)kStageBytes);
        tma_load_box(dyn + k * kStageBytes, tmap, &sm.full[k], 0, (int32_t)(g.start >> 4));
      } else {
        mbar_arrive(&sm.full[k]);
      }
    }
  }
}

// ---------------------------------------------------------------- the kernel
__global__ void __launch_bounds__(kBlockThreads, 2)
    seqsum_kernel(const __grid_constant__ Params p, const __grid_constant__ CUtensorMap tmap) {
  extern __shared__ unsigned char dsm_raw[];
  unsigned char *dyn =
      reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(dsm_raw) + 1023) & ~(uintptr_t)1023);
  __shared__ Smem sm;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  int64_t ntiles = (p.ntiles >= 0) ? p.ntiles : (int64_t)__ldcg(&p.ctr[C_NTILES]);
  if (ntiles > p.cap_tiles) ntiles = 0;                  // the set-up flagged ERR_CAPACITY
  if (tid < S_COUNT) sm.st[tid] = 0;
  if (tid < kWarps) sm.barcnt[tid] = 0;
  if (tid == 0) {
    for (int s = 0; s < kStages; s++) {
      mbar_init(&sm.full[s], 3);                         // control lanes 0 and 1 (copies) and lane 0 (unit)
      mbar_init(&sm.done[s], kWarps);
      mbar_init(&sm.sums[s], kWarps);
    }
    fence_mbar_init();
    if (blockIdx.x == 0) p.stats[S_T_START] = globaltimer();
    // roles go to CTAs in the order they start, so every waiting role is
    // held by a running CTA
    sm.role = (int)atomicAdd(&p.ctr[C_ROLE], 1u);
  }
  __syncthreads();
  if ((tid & 31) == 0) beat(p, sm.role, HB_START, 0);
  const int role = sm.role;

  if (role < p.nwalkers) {
    // ---------------- walker CTA (its control warp idles)
    if (warp < kWarps) {
      if (p.offsets == nullptr) {
        if (ntiles == 0) { if (tid == 0) p.outs[0] = p.s0; }
        else walk_sum(p, sm, dyn, 0, 0, ntiles, ntiles);
      } else {
        while (true) {
          if (tid == 0) sm.sum_k = (int)atomicAdd(&p.ctr[C_SUMTICKET], 1u);
          wide_sync(p, sm, 24);
          const int k = sm.sum_k;
          wide_sync(p, sm, 25);
          if (k >= p.nsums) break;
          if (ntiles == 0) continue;                     // bad offsets or capacity: outputs already NaN
          const int64_t tb = __ldcg(&p.tile_begin[k]), te = __ldcg(&p.tile_begin[k + 1]);
          if (te > tb) walk_sum(p, sm, dyn, k, tb, te, ntiles);
        }
      }
    }
  } else if (role == p.nwalkers) {
    // ---------------- the plan's prefix scanner (its control warp idles)
    if (warp < kWarps && ntiles > 0) scan_prefix(p, sm, ntiles);
  } else {
    // ---------------- streaming CTA
    if (warp < kWarps) compute_loop(p, sm, dyn, ntiles);
    else control_loop(p, sm, dyn, &tmap, ntiles);
  }

  // ---- statistics and the last CTA's reset of the shared counters
  if ((tid & 31) == 0) beat(p, sm.role, HB_END, 0);
  __syncthreads();
  if (tid < S_ACCUM_END && sm.st[tid]) atomicAdd(&p.stats[tid], (unsigned long long)sm.st[tid]);
  if (tid == 0) {
    __threadfence();
    if (atomicAdd(&p.ctr[C_EXIT], 1u) + 1 == gridDim.x) {
      p.ctr[C_TICKET] = 0;
      p.ctr[C_SUMTICKET] = 0;
      p.ctr[C_ROLE] = 0;
      p.ctr[C_EXIT] = 0;
      __threadfence();
    }
  }
}

// Batched set-up: tiles per sum and their prefix (tile_begin), the start value
// of empty sums.  Offsets out of order or outside [0, x_len] (x_len = p.n),
// or more tiles than the workspace holds, stop the call: every output
// becomes NaN and an error bit is set.
__global__ void setup_kernel(const Params p) {
  __shared__ int64_t s_carry;
  __shared__ int64_t s_w[32];
  __shared__ int s_bad;
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  if (tid == 0) { s_carry = 0; s_bad = 0; }
  __syncthreads();
  for (int base = 0; base < p.nsums; base += blockDim.x) {
    const int k = base + tid;
    int64_t nt = 0;
    if (k < p.nsums) {
      const int64_t a = p.offsets[k], b = p.offsets[k + 1];
      int64_t len = b - a;
      if (len < 0 || a < 0 || b > p.n) { s_bad = 1; len = 0; }
      nt = (len + kTileTerms - 1) / kTileTerms;
      if (len == 0) p.outs[k] = p.s0s[k];
    }
    int64_t incl = nt;
    for (int o = 1; o < 32; o <<= 1) {
      const int64_t v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    if (lane == 31) s_w[w] = incl;
    __syncthreads();
    int64_t wb = 0;
    for (int i = 0; i < w; i++) wb += s_w[i];
    if (k < p.nsums) p.tile_begin[k] = s_carry + wb + incl - nt;
    __syncthreads();
    if (tid == blockDim.x - 1) s_carry += wb + incl;
    __syncthreads();
  }
  __syncthreads();
  const bool bad = s_bad != 0;
  const bool over = s_carry > p.cap_tiles;
  if (bad || over) {
    for (int k = tid; k < p.nsums; k += blockDim.x) p.outs[k] = __longlong_as_double(0x7FF8000000000000ll);
  }
  if (tid == 0) {
    p.tile_begin[p.nsums] = s_carry;
    if (bad) atomicOr(&p.ctr[C_ERR], ERR_BAD_OFFSETS);
    if (over) atomicOr(&p.ctr[C_ERR], ERR_CAPACITY);
    p.ctr[C_NTILES] = (bad || over) ? 0u : (uint32_t)s_carry;
  }
}

cudaError_t launch_seqsum(const Params &p, const CUtensorMap *tmap, int grid, cudaStream_t st) {
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(seqsum_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kDynSmem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  seqsum_kernel<<<grid, kBlockThreads, kDynSmem, st>>>(p, *tmap);
  return cudaGetLastError();
}

cudaError_t launch_setup(const Params &p, cudaStream_t st) {
  setup_kernel<<<1, 1024, 0, st>>>(p);
  return cudaGetLastError();
}

int kernel_max_blocks_per_sm() {
  cudaFuncSetAttribute(seqsum_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kDynSmem);
  int nb = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, seqsum_kernel, kBlockThreads, kDynSmem) != cudaSuccess)
    return 1;
  return nb > 0 ? nb : 1;
}

}  // namespace sq

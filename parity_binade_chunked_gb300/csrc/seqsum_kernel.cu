// The device path of the exact sequential fp64 sum (sm_103a).
//
// One persistent kernel.  CTAs 0 .. nwalkers-1 walk, the next one scans the
// plan's tile sums; every other CTA streams
// tiles of 4096 terms (32 KB, one TMA box) taken in ticket order, each read
// from HBM once, in a three-stage pipeline: while one tile is copied, the
// next is planned and the one before is formed into runs.
//
//  * Plan (Research-1424, section 3: a first pass that adds each row on its
//    own and a prefix over the rows give the sum at every row start, which
//    names the binade except next to a power of two; Research-1433, finding 5
//    and the open question "compute the plan's prefix with a scan"): as soon
//    as a tile lands, its terms are summed in fixed point (their 32 leading
//    significant bits, by integer shifts) and the tile's approximate sum is
//    published; a scanner CTA scans the published sums in order, in windows
//    of up to 1024 tiles, and publishes every tile's inclusive prefix; each
//    streaming CTA's prefix warp reads the prefix of the tile before its own
//    and gives every chunk of the tile its approximate starting value in
//    double-float and a verdict: inside one binade, all zeros, or spanning a
//    power of two.
//  * Runs (finding 2 "Inside a binade the loop is an integer sum", finding 3
//    "Ties need the parity of the running integer"): a chunk of 512 terms
//    whose whole range lies inside one binade is turned into its increment
//    by integer shifts (binade_math.cuh) and composed: each lane's 16 terms
//    in order, then the warp's 32 lanes in a fixed shuffle tree (finding 6).
//  * A chunk spanning a power of two is split: lanes that fit a binade become
//    runs, and inside the other lanes each term is placed on its own; only
//    the terms whose prefix range touches a power of two are carried, as
//    values, to be added one by one (finding 4).
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
#include "units.cuh"

namespace sq {

// ---------------------------------------------------------------- constants
constexpr float kTinyF = 0x1p-120f;            // floor of the plan's error allowance
constexpr int kZeroE = -2000;                  // binade key of a run of zeros
constexpr int kDirtyKey = -3000;               // merge key of a lane placed term by term
constexpr uint64_t kWaitNs = 2000000000ull;    // bounded device waits: 2 s
constexpr uint64_t kCountMask = (1u << kCountBits) - 1;
static_assert(((uint64_t)kChunkSlots << (kCountBits * (kWarps - 1))) < (1ull << 55),
              "packed item counts must fit a tagged 56-bit word");
constexpr int kWalkMinTiles = 256;             // smallest walk batch (unless the sum ends sooner)
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
__device__ __forceinline__ uint32_t smid() {
  uint32_t v;
  asm volatile("mov.u32 %0, %%smid;" : "=r"(v));
  return v;
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
// Non-blocking test of an mbarrier phase (for polling several barriers).
__device__ __forceinline__ bool mbar_test(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
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
// One word per warp (index CTA * kBlockWarps + warp).
enum : uint32_t {
  HB_START = 1, HB_WAIT_UNIT = 2, HB_UNIT = 3, HB_WAIT_DONE = 4, HB_WAIT_HEADERS = 6,
  HB_BATCH = 7, HB_SERIAL = 8, HB_COUNT = 11, HB_GATHER = 12, HB_SCAN = 13,
  HB_RESTART = 14, HB_END = 15, HB_BARRIER = 16, HB_WINDOW = 17
};
__device__ __forceinline__ void beat(const Params &p, uint32_t role, uint32_t what, uint64_t where) {
  const unsigned i = blockIdx.x * (unsigned)kBlockWarps + (threadIdx.x >> 5);
  if (i < (unsigned)kHeartbeats)
    p.hb[i] = ((uint64_t)(role & 0xFFu) << 56) | ((uint64_t)(what & 0xFFu) << 48) | (where & 0xFFFFFFFFFFFFull);
}

// A bounded wait gave up: set its error bit and keep the first such site
// with two words of context for the host.
enum : uint32_t {
  TO_FULL = 1, TO_DONE = 2, TO_PLANNED = 3, TO_PREFIX = 4, TO_VERDICT = 5, TO_SCAN = 6, TO_WALK = 7
};
__device__ __noinline__ void note_timeout(const Params &p, uint32_t err, uint32_t site, uint32_t a, uint32_t b) {
  atomicOr(&p.ctr[C_ERR], err);
  if (atomicCAS(&p.ctr[C_TO_SITE], 0u, site) == 0u) {
    p.ctr[C_TO_A] = a;
    p.ctr[C_TO_B] = b;
  }
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
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// An atomic add with acquire and release semantics at GPU scope: the writes
// before it are visible to whoever observes its result, and the reads after
// it see what was visible to the writers of the values it observed.
__device__ __forceinline__ uint32_t add_acq_rel(uint32_t *a, uint32_t v) {
  uint32_t old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(a), "r"(v) : "memory");
  return old;
}
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

// Timeline of a call (profiling builds): per tile and unit kind eight words
// from kTraceUnits on (its copy issued, the compute warps' start and end, the
// epilogue's end, the CTA and ticket), per walk batch four words.
#ifdef SEQSUM_PROFILE
constexpr int kTraceUnits = 16384;
constexpr int kTraceBatches = 61440;
__device__ __forceinline__ void trace_word(const Params &p, int base, int limit, int64_t idx, int stride, int field,
                                           unsigned long long v) {
  const int64_t i = base + idx * stride + field;
  if (idx >= 0 && i < limit) p.dbg[i] = v;
}
#define TRACE_UNIT(t, kind, field, v) trace_word(p, kTraceUnits, kTraceBatches, 2 * (t) + (kind), 8, (field), (v))
#define TRACE_BATCH(b, field, v) trace_word(p, kTraceBatches, kDbgAlloc, (b), 4, (field), (v))
// the largest value offered (the slowest chunk of a unit)
#define TRACE_UNIT_MAX(t, kind, field, v)                                                      \
  do {                                                                                       \
    const int64_t i_ = kTraceUnits + (2 * (t) + (kind)) * 8 + (field);                       \
    if (i_ < kTraceBatches) atomicMax(&p.dbg[i_], (unsigned long long)(v));                  \
  } while (0)
#else
#define TRACE_UNIT_MAX(t, kind, field, v) do { } while (0)
#define TRACE_UNIT(t, kind, field, v) do { } while (0)
#define TRACE_BATCH(b, field, v) do { } while (0)
#endif

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
// Flags of a chunk's terms: one with the sign bit set, one with it clear, one
// that is not zero.
enum : uint32_t { WA_NEG = 1u, WA_POS = 2u, WA_NZ = 4u };

// The plan of one chunk, formed by its compute warp as soon as the tile has
// landed: the magnitudes of its non-negative terms (P) and of its negative
// terms (N), each summed in fixed point in units of 2^(L - 1054), where L is
// the largest biased exponent among the chunk's terms.
struct ChunkPlan {
  uint64_t P, N;
  int32_t L;
  uint32_t mx;        // largest magnitude high word among the chunk's terms
  uint32_t flags;     // WA_*
  uint32_t pad;
};

// A run unit's verdict on one chunk: every term zero, every prefix in one
// binade (clean), or the prefix range spanning a power of two (dirty).
enum : int { CP_CLEAN = 0, CP_ZERO = 1, CP_DIRTY = 2 };
struct ChunkPre {
  DF c;               // approximate running sum before the chunk
  float ab;           // approximate |s0| + sum of |x| before the chunk
  float delta;        // the plan's error allowance inside the chunk
  int32_t e;          // CP_CLEAN: the binade of every prefix inside the chunk
  int32_t mode;       // CP_*
};

enum : int { U_PLAN = 0, U_RUN = 1, U_END = 2 };
// The unit a stage holds, written by the control warp before its copy starts.
struct StageGeo {
  int64_t t;          // tile index
  int64_t start, end; // its terms [start, end) in x
  int64_t first_tile; // the first tile of its sum
  int64_t sum_start;  // the first term of its sum
  int32_t sum;        // which sum
  int32_t kind;       // U_PLAN, U_RUN, or U_END: no more units
  int32_t tma;        // its terms came by TMA (else they are read from global memory)
  int32_t pad;
};

struct Smem {
  uint64_t full[kStages];           // the unit's copy and plan words landed, or the end marker (kFullArrivals)
  uint64_t done[kStages];           // the compute warps finished the unit (kWarps arrivals)
  uint64_t used[kStages];           // the unit's chunks have read their terms from the stage (kWarps arrivals)
  StageGeo geo[kStages];            // the unit's tile and kind (U_PLAN, U_RUN, U_END)
  // a run unit's plan words, copied in ahead of its runs: the prefix of the
  // tile before and the tile's chunk plans (cp.async destinations: 16-byte
  // aligned)
  alignas(16) uint64_t pre_raw[kStages][2];
  alignas(16) uint64_t cplan_raw[kStages][kWarps * 4];
  ChunkPlan plan[kStages][kWarps];  // a plan unit's chunk plans
  // a run unit's chunk verdicts, formed by the first warp that reaches the
  // unit (vtile: its tile + 1 once they are in)
  ChunkPre vpre[kStages][kWarps];
  uint32_t vmx[kStages][kWarps], vfl[kStages][kWarps];
  int64_t vtile[kStages];
  Rec chunk[kStages][kWarps];       // a run unit's chunk records
  int nitems[kStages][kWarps];      // >0: a split chunk's items in the tile's item area
  int plan_cnt[kStages];            // chunks of a plan unit's tile planned so far
  // per stage the claim word of its unit: use << 8 | chunks claimed (the
  // use counts the units the stage has held; bit 7 marks the end marker)
  uint32_t cnext[kStages];
  int slow[kStages];                // a chunk of the stage's unit is being split (it ends late)
  Rec stg[kWarps][kChunkSlots];     // a split chunk's items, staged in order before they are written out
  int role;
  uint32_t barcnt[kWarps];          // walker and scanner: wide barriers passed per warp (heartbeat)
  unsigned int st[S_COUNT];         // per-CTA statistics of one call (32-bit: native shared atomics)
#ifdef SEQSUM_PROFILE
  unsigned int prof[40];            // cycle profile of the run chunks
#endif
  // walker
  uint64_t S;
  int m, nel, restart, nseg;
  int64_t wpos0, wpos1;             // the walk's helper command: tiles [wpos0, wpos1)
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
// two CTAs per SM: 228 KB of shared memory per SM, 1 KB of it reserved per CTA
static_assert(sizeof(Smem) + sizeof(Params) + 64 + kDynSmem + 1024 <= 233472 / 2, "two CTAs per SM");
static_assert(offsetof(Smem, pre_raw) % 16 == 0 && offsetof(Smem, cplan_raw) % 16 == 0,
              "cp.async destinations must be 16-byte aligned");
// a run unit's copies: lane 0 the prefix word pair, lanes 1..16 the chunk
// plans (16 bytes each); every one of those lanes makes one arrival when its
// copy has landed, lane 0 one more for the tile's own copy, and one more once
// the unit's description (sm.geo, the claim word) is written
constexpr int kCopyLanes = 1 + kWarps * 2;
constexpr uint32_t kFullArrivals = kCopyLanes + 2;
static_assert(offsetof(Smem, full) % 8 == 0 && offsetof(Smem, done) % 8 == 0 && offsetof(Smem, used) % 8 == 0,
              "mbarriers are 8-byte aligned");

// The 256-thread barrier of a walking or scanning CTA; each warp first records the
// barrier's site and how many it has passed (its heartbeat).
__device__ __noinline__ void wide_sync_at(const Params &p, Smem &sm, int site) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) {
    const uint32_t c = ++sm.barcnt[warp];
    beat(p, sm.role, HB_BARRIER, ((uint64_t)site << 32) | c);
  }
  named_sync(kBarWide, kThreads);
}

// ---------------------------------------------------------------- the plan
// The plan (Research-1424, section 3: a first pass that adds each row on its
// own and a prefix over the rows give the sum at every row start, and so its
// binade except next to a power of two; Research-1433, finding 5: the plan
// only chooses where the walk looks, so an error in it costs time, never a
// bit).  Every term enters it as its 32 leading significant bits in fixed
// point, by integer shifts; chunk sums become double-float values; a scanner
// CTA turns the tiles' published sums into inclusive prefixes.
//
// Error of the plan, relative to the running sum of |x|: a term loses less
// than one unit of its lane's scale (2^-31 of the lane's largest term), a lane
// less than one unit of its chunk's scale; with the double-float sums that is
// below 2^-25.  The sequential fp64 sum itself drifts from the exact sum by
// at most 2^-53 of |s0| + sum |x| per add.  The allowance kPlanEps covers the
// first with a margin, and the walk's drift term is added per chunk.
constexpr float kPlanEps = 0x1p-24f;

// The 32 leading significant bits of a normal term (0 for zeros and
// subnormals, too small to matter to the plan): the term is about
// m * 2^(E - 1054).
__device__ __forceinline__ uint32_t lead32(uint32_t hi, uint32_t lo, uint32_t E) {
  const uint32_t m = __funnelshift_l(lo, hi, 11) | 0x80000000u;
  return E ? m : 0u;
}
// The lane's terms in fixed point at scale 2^(Lm - 1054), Lm the largest
// biased exponent among them: `all` sums every magnitude, `neg` those of the
// terms with the sign bit set.  Each term loses less than one unit.
__device__ __forceinline__ void lane_fixed(const uint64_t *xs, uint32_t Lm, uint64_t &all, uint64_t &neg) {
  all = 0;
  neg = 0;
#pragma unroll
  for (int i = 0; i < kLaneTerms; i++) {
    const uint32_t hi = (uint32_t)(xs[i] >> 32), lo = (uint32_t)xs[i];
    const uint32_t E = (hi >> 20) & 0x7FFu;
    const uint32_t v = __funnelshift_rc(lead32(hi, lo, E), 0u, Lm - E);   // shifts of 32 or more give 0
    all += v;
    neg += (hi >> 31) ? v : 0u;
  }
}
// Sum over the warp of values below 2^36 (16-bit low parts and the rest
// summed apart, so that each 32-bit reduction stays exact).
__device__ __forceinline__ uint64_t warp_sum36(uint64_t v) {
  const uint32_t lo = __reduce_add_sync(0xffffffffu, (uint32_t)v & 0xFFFFu);
  const uint32_t hi = __reduce_add_sync(0xffffffffu, (uint32_t)(v >> 16));
  return ((uint64_t)hi << 16) + lo;
}
// 2^q as a float: 0 below 2^-126, infinity above 2^127 (the plan then only
// gets worse).
__device__ __forceinline__ float pow2f(int q) {
  if (q < -126) return 0.0f;
  if (q > 127) return __uint_as_float(0x7F800000u);
  return __uint_as_float((uint32_t)(q + 127) << 23);
}
// Integers as double-float or float values, from exact 16-bit pieces (32-bit
// conversions and fp32 adds only): |v| < 2^48.
__device__ __forceinline__ DF df_from_u48(uint64_t v) {
  const float a = __fmul_rn(__uint2float_rn((uint32_t)(v >> 32) & 0xFFFFu), 0x1p32f);
  const float b = __fmul_rn(__uint2float_rn((uint32_t)v >> 16), 0x1p16f);
  const float c = __uint2float_rn((uint32_t)v & 0xFFFFu);
  return df_addf(two_sum(a, b), c);
}
__device__ __forceinline__ DF df_from_i48(int64_t v) {
  const DF m = df_from_u48((uint64_t)(v < 0 ? -v : v));
  return v < 0 ? DF{-m.hi, -m.lo} : m;
}
__device__ __forceinline__ float f_from_u48(uint64_t v) {
  return __fadd_rn(__fmul_rn(__uint2float_rn((uint32_t)(v >> 32) & 0xFFFFu), 0x1p32f), __uint2float_rn((uint32_t)v));
}
__device__ __forceinline__ float f_from_i48(int64_t v) {
  const float m = f_from_u48((uint64_t)(v < 0 ? -v : v));
  return v < 0 ? -m : m;
}
// v * 2^(L - 1054) as a double-float or a float (|v| < 2^48).
__device__ __forceinline__ DF df_fixed(int64_t v, int L) {
  const DF m = df_from_i48(v);
  const float s = pow2f(L - 1054);
  return DF{__fmul_rn(m.hi, s), __fmul_rn(m.lo, s)};
}
__device__ __forceinline__ float f_fixed(uint64_t v, int L) { return __fmul_rn(f_from_u48(v), pow2f(L - 1054)); }

// Binade of a positive double-float value: its high part's, one less when
// the high part is a power of two and the low part pulls the value below it.
// (The fp32 biased exponent; 0 for subnormal, 255 for inf and NaN.)
__device__ __forceinline__ int df_exp_pos(DF v) {
  const uint32_t b = __float_as_uint(v.hi);
  const int e = (int)((b >> 23) & 0xFFu);
  return e - (((b & 0x7FFFFFu) == 0u && v.lo < 0.0f) ? 1 : 0);
}
// The binade (unbiased exponent) shared by every value in [lo, hi], or false.
__device__ __forceinline__ bool one_binade_df(DF lo, DF hi, int &e) {
  DF a, b;
  if (lo.hi > 0.0f) { a = lo; b = hi; }
  else if (hi.hi < 0.0f) { a = DF{-hi.hi, -hi.lo}; b = DF{-lo.hi, -lo.lo}; }
  else return false;                                   // zero inside, or NaN
  const int ea = df_exp_pos(a), eb = df_exp_pos(b);
  if (ea != eb || ea <= 0 || ea >= 0xFF) return false;
  e = ea - 127;
  return true;
}

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

// Warp-uniform test of an mbarrier phase.  When it reports the phase
// complete, every lane has itself observed the completion (and so sees what
// was written before it).
__device__ __forceinline__ bool mbar_test_warp(uint64_t *bar, uint32_t parity) {
  if (!__any_sync(0xffffffffu, mbar_test(bar, parity))) return false;
  for (int i = 0; i < (1 << 20) && !mbar_test(bar, parity); i++) {
  }
  return true;
}
// A bounded, warp-uniform wait on an mbarrier phase; false (for every lane)
// on timeout.
__device__ __forceinline__ bool mbar_wait_warp(const Params &p, uint64_t *bar, uint32_t parity, uint32_t err,
                                               uint32_t site, uint32_t a, uint32_t b) {
  if (mbar_test_warp(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  uint32_t nap = 32;
  while (true) {
    // one potentially blocking wait, then the warp-uniform test; between
    // tests the warp sleeps (backoff), so that it takes no issue slots
    (void)mbar_try_wait(bar, parity);
    if (mbar_test_warp(bar, parity)) break;
    __nanosleep(nap);
    nap = min(nap * 2u, 256u);
    if (__any_sync(0xffffffffu, globaltimer() - t0 > kWaitNs)) {
      if ((threadIdx.x & 31) == 0) note_timeout(p, err, site, a, b);
      return false;
    }
  }
  return true;
}

#ifdef SEQSUM_PROFILE
// Cycle profiles (profiling builds): cycles since the previous point, summed
// per point, and the number of times each point is passed (split chunks from
// word 15200 on).
#define PROF_START long long prof_t = clock64()
#define PROF_PT(base, id)                                                                  \
  do {                                                                                     \
    if ((threadIdx.x & 31) == 0) {                                                         \
      const long long now_ = clock64();                                                    \
      atomicAdd(&p.dbg[(base) + 2 * (id)], (unsigned long long)(now_ - prof_t));           \
      atomicAdd(&p.dbg[(base) + 1 + 2 * (id)], 1ull);                                      \
      prof_t = now_;                                                                       \
    }                                                                                      \
  } while (0)
#else
#define PROF_START do { } while (0)
#define PROF_PT(base, id) do { } while (0)
#endif
#define SPLIT_PT(id) PROF_PT(15200, id)
// Per-CTA cycle profile of the run chunks (profiling builds): cycles since
// the previous point and passes, summed in shared memory, added to the
// diagnostic words from 15300 on when the CTA ends.
#ifdef SEQSUM_PROFILE
#define CPROF_START long long cprof_t = clock64()
#define CPROF_PT(id)                                                                       \
  do {                                                                                     \
    if ((threadIdx.x & 31) == 0) {                                                         \
      const long long n_ = clock64();                                                      \
      atomicAdd(&sm.prof[2 * (id)], (unsigned)(n_ - cprof_t));                             \
      atomicAdd(&sm.prof[2 * (id) + 1], 1u);                                               \
      cprof_t = n_;                                                                        \
    }                                                                                      \
  } while (0)
#else
#define CPROF_START do { } while (0)
#define CPROF_PT(id) do { } while (0)
#endif

// The plan of chunk w of the stage's tile (by whichever compute warp claimed
// it).  The warp that completes the tile's plan publishes the chunk plans and
// the tile's approximate sum (for a sum's first tile: s0 plus it, as an
// inclusive prefix) for the scanner.
__device__ __noinline__ void publish_tile_plan(const Params &p, Smem &sm, int k);
__device__ __forceinline__ void load_lane(const Params &p, const unsigned char *stage, bool use_tma, int64_t row,
                                          int64_t lstart, int nv, int w, int lane, uint64_t *xs);
// A chunk is done with the stage's terms (every lane has them in registers):
// the control warp may copy the next unit's terms into the stage.  Once per
// chunk and use of the stage.
__device__ __forceinline__ void release_stage(Smem &sm, int k) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(&sm.used[k]);
}
__device__ __noinline__ void plan_chunk(const Params &p, Smem &sm, const unsigned char *stage, int k, int w) {
  const int lane = threadIdx.x & 31;
  const unsigned full = 0xffffffffu;
  const StageGeo &g = sm.geo[k];
  const int64_t lstart = g.start + (int64_t)w * kChunkTerms + (int64_t)lane * kLaneTerms;
  const int nv = (int)max((int64_t)0, min((int64_t)kLaneTerms, g.end - lstart));
  uint64_t xs[kLaneTerms];
  load_lane(p, stage, g.tma != 0, (g.start >> 4) + w * 32 + lane, lstart, nv, w, lane, xs);
  release_stage(sm, k);
  uint32_t mx = 0, orz = 0, orh = 0, andh = 0xFFFFFFFFu;
#pragma unroll
  for (int i = 0; i < kLaneTerms; i++) {
    const uint32_t hi = (uint32_t)(xs[i] >> 32), lo = (uint32_t)xs[i];
    const uint32_t mag = hi & 0x7FFFFFFFu;
    mx = max(mx, mag);
    orz |= mag | lo;
    if (i < nv) { orh |= hi; andh &= hi; }
  }
  const uint32_t Lm = mx >> 20;
  uint64_t all, neg;
  lane_fixed(xs, Lm, all, neg);
  const uint32_t Lc = __reduce_max_sync(full, Lm);
  const uint32_t sh = min(Lc - Lm, 63u);
  const uint64_t Pc = warp_sum36((all - neg) >> sh), Nc = warp_sum36(neg >> sh);
  const uint32_t fl = __reduce_or_sync(full, ((orh >> 31) ? WA_NEG : 0u) | ((andh >> 31) ? 0u : WA_POS) |
                                                 (orz ? WA_NZ : 0u));
  const uint32_t mxc = __reduce_max_sync(full, mx);
  int last = 0;
  if (lane == 0) {
    sm.plan[k][w] = ChunkPlan{Pc, Nc, (int32_t)Lc, mxc, fl, 0u};
    __threadfence_block();
    last = atomicAdd(&sm.plan_cnt[k], 1) == kWarps - 1;
  }
  if (__shfl_sync(full, last, 0)) {
    __threadfence_block();
    publish_tile_plan(p, sm, k);
  }
}

// The chunk plans in global memory, four words per chunk, the tag in the top
// byte of every word (an 8-byte access is single-copy atomic, a 16-byte one
// need not be): P, N, L | flags << 16, mx.
__device__ __forceinline__ void publish_cplan(uint64_t *dst, const ChunkPlan &c, uint32_t tag) {
  const uint64_t tg = (uint64_t)tag << 56;
  st_vol_v2(dst, c.P | tg, c.N | tg);
  st_vol_v2(dst + 2, (uint64_t)(uint32_t)c.L | ((uint64_t)c.flags << 16) | tg, (uint64_t)c.mx | tg);
}
// The chunk plan in four words, when all of them carry `tag`.
__device__ __forceinline__ bool cplan_of(uint64_t w0, uint64_t w1, uint64_t w2, uint64_t w3, uint32_t tag,
                                        ChunkPlan &c) {
  if ((uint32_t)(w0 >> 56) != tag || (uint32_t)(w1 >> 56) != tag || (uint32_t)(w2 >> 56) != tag ||
      (uint32_t)(w3 >> 56) != tag)
    return false;
  c.P = w0 & kLow56;
  c.N = w1 & kLow56;
  c.L = (int32_t)(w2 & 0xFFFFu);
  c.flags = (uint32_t)(w2 >> 16) & 0xFFu;
  c.mx = (uint32_t)w3;
  c.pad = 0u;
  return true;
}

__device__ __noinline__ void publish_tile_plan(const Params &p, Smem &sm, int k) {
  const int lane = threadIdx.x & 31;
  const StageGeo &g = sm.geo[k];
  ChunkPlan cp{0ull, 0ull, 0, 0u, 0u, 0u};
  if (lane < kWarps) cp = sm.plan[k][lane];
  const bool in = sq_ok(p, g.t >= 0 && g.t < p.cap_tiles, 6, g.t);
  if (lane < kWarps && in) publish_cplan(p.cplan + (g.t * kWarps + lane) * 4, cp, (p.epoch << 1) | 1u);
  DF s = df_fixed((int64_t)cp.P - (int64_t)cp.N, cp.L);
  float a = f_fixed(cp.P + cp.N, cp.L);
#pragma unroll
  for (int o = kWarps / 2; o > 0; o >>= 1) {
    s = df_add(s, shfl_xor_df(s, o));
    a += __shfl_xor_sync(0xffffffffu, a, o);
  }
  if (lane == 0 && in) {
    if (g.t == g.first_tile) {
      const DF s0 = df_from_double(p.s0s ? p.s0s[g.sum] : p.s0);
      publish_status(p.status + 2 * g.t, df_add(s0, s), fabsf(s0.hi) + a, p.epoch, 1);
    } else {
      publish_status(p.status + 2 * g.t, s, a, p.epoch, 0);
    }
  }
}

// The scanner (a whole CTA, Research-1424 section 3: a prefix over the row
// sums gives the sum at every row start; Research-1433, open question "the
// plan's prefix as a scan"): from where it stands it takes the longest run of
// tiles whose approximate sums are published (up to 1024 tiles), scans it --
// a tile published as an inclusive prefix starts a sum and already holds s0
// plus its own sum -- and publishes every other tile's inclusive prefix.
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
  uint32_t nap = 32;
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
      __nanosleep(nap);
      nap = min(nap * 2u, 256u);
      twait += globaltimer() - now;
      wide_sync(p, sm, 2);                       // sm.scan_stop is set; sm.scan_m may be written again
      if (sm.scan_stop) break;
      continue;
    }
    nap = 32;
    tprog = globaltimer();
    // this thread's elements, scanned in order; an inclusive prefix restarts the sum
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

// The inclusive prefix the scanner published for tile t - 1 (a bounded wait
// with backoff; on a timeout the plan is only worse).  Whole warp.
__device__ __noinline__ void read_prefix(const Params &p, Smem &sm, int64_t t, DF &ex, float &exab) {
  const int lane = threadIdx.x & 31;
  const uint32_t tag1 = (p.epoch << 1) | 1u;
  const uint64_t t0 = globaltimer();
  uint32_t nap = 32;
  uint64_t A = 0, B = 0;
  while (true) {
    if (lane == 0 && sq_ok(p, t >= 1 && t - 1 < p.cap_tiles, 1, t)) ld_vol_v2(p.status + 2 * (t - 1), A, B);
    A = __shfl_sync(0xffffffffu, A, 0);
    B = __shfl_sync(0xffffffffu, B, 0);
    const uint32_t ta = (uint32_t)(A & 0xFF), tb = (uint32_t)B;
    if (ta == tag1 && tb == tag1) break;
    if (lane == 0 && ta != tb && ((ta >> 1) == p.epoch || (tb >> 1) == p.epoch)) atomicAdd(&sm.st[S_TORN_STATUS], 1u);
    if (__any_sync(0xffffffffu, globaltimer() - t0 > kWaitNs)) {
      if (lane == 0) note_timeout(p, ERR_PLAN_TIMEOUT, TO_PREFIX, (uint32_t)t, (uint32_t)(ta | tb << 8));
      A = 0;
      B = 0;
      break;
    }
    __nanosleep(nap);
    nap = min(nap * 2u, 256u);
  }
  ex = status_sum(A);
  exab = status_abs(B);
}

// The verdicts of all chunks of the tile at once: lane j (j < kWarps) the
// verdict on chunk j, its largest magnitude word and flags.  Whole warp.
__device__ __forceinline__ ChunkPre chunk_verdicts(const StageGeo &g, DF ex, float exab, const ChunkPlan &cp,
                                                   uint32_t &cmx, uint32_t &cflags) {
  const int lane = threadIdx.x & 31;
  const unsigned full = 0xffffffffu;
  const DF sig = df_fixed((int64_t)cp.P - (int64_t)cp.N, cp.L);
  const float ab = f_fixed(cp.P + cp.N, cp.L);
  DF s = sig;
  float sa = ab;
#pragma unroll
  for (int o = 1; o < kWarps; o <<= 1) {
    const DF os = DF{__shfl_up_sync(full, s.hi, o), __shfl_up_sync(full, s.lo, o)};
    const float oa = __shfl_up_sync(full, sa, o);
    if (lane >= o) { s = df_add(os, s); sa += oa; }
  }
  // the sums of the chunks before lane j's (exclusive)
  DF es = DF{__shfl_up_sync(full, s.hi, 1), __shfl_up_sync(full, s.lo, 1)};
  float ea = __shfl_up_sync(full, sa, 1);
  if (lane == 0) { es = DF{0.0f, 0.0f}; ea = 0.0f; }
  cmx = cp.mx;
  cflags = cp.flags;
  const DF c = df_add(ex, es);
  const float cab = exab + ea;
  const float nb = (float)(g.start - g.sum_start + (int64_t)(lane + 1) * kChunkTerms);
  const float delta = __fmaf_rn(nb, 0x1p-53f, kPlanEps) * (cab + ab) + kTinyF;
  const float Pf = f_fixed(cp.P, cp.L), Nf = f_fixed(cp.N, cp.L);
  int e = 0, mode;
  if (!(cflags & WA_NZ)) mode = CP_ZERO;
  else if (one_binade_df(df_addf(c, -(Nf + delta)), df_addf(c, Pf + delta), e)) mode = CP_CLEAN;
  else mode = CP_DIRTY;
  return ChunkPre{c, cab, delta, e, mode};
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

// Term i of a lane: from its 128-byte row of the stage (16-byte chunk i/2,
// swizzled by the row), or from global memory.
__device__ __forceinline__ uint64_t lane_term(bool from_stage, const unsigned char *rp,
                                              const unsigned long long *gp, int lane, int i) {
  if (from_stage) {
    const uint2 v = *reinterpret_cast<const uint2 *>(rp + ((((i >> 1) ^ (lane & 7)) << 4) | ((i & 1) << 3)));
    return ((uint64_t)v.y << 32) | v.x;
  }
  return __ldg(gp + i);
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
    const uint64_t x = lane_term(from_stage, rp, gp, lane, i);
    int64_t re;
    int32_t d;
    const bool poison = term_inc(x, e, re, d);
    run_push(r, re, d, term_flags(x) | (poison ? F_POISON : 0u));
  }
  return r;
}

// The run of a lane's terms from their increments summed apart by sign (no
// tie among them): P for the terms with the sign bit clear, N for the others;
// or and and of the valid terms' high words give the sign flags.
__device__ __forceinline__ Run lane_pn_run(uint64_t P, uint64_t N, uint32_t orl, uint32_t andl, int nv) {
  if (nv == 0) return run_empty();
  Run r;
  r.inc = (int64_t)(P - N);
  r.lo = -(int64_t)N;
  r.hi = (int64_t)P;
  r.d = 0;
  r.flags = ((orl >> 31) ? 0u : F_NONNEG) | ((andl >> 31) ? F_NONPOS : 0u);
  return r;
}
// Increments of a lane's terms under the fast rule (binade_math.cuh,
// term_inc_fast; c = 64 - (e + 1023)) summed apart by sign, whether any of
// them ties, and the sign flags of the valid terms.
__device__ __forceinline__ void lane_fast(const uint64_t *xs, int nv, int c, uint64_t &P, uint64_t &N, bool &anytie,
                                          uint32_t &orl, uint32_t &andl) {
  P = 0; N = 0; anytie = false; orl = 0; andl = 0xFFFFFFFFu;
#pragma unroll
  for (int i = 0; i < kLaneTerms; i++) {
    const uint32_t hi = (uint32_t)(xs[i] >> 32);
    uint64_t ri;
    bool tie;
    term_inc_fast(hi, (uint32_t)xs[i], c, ri, tie);
    if (hi >> 31) N += ri; else P += ri;
    anytie |= tie;
    if (i < nv) { orl |= hi; andl &= hi; }
  }
}
// The same, reading the lane's terms from its row of the stage two at a
// time (a rolled loop: the instructions of a chunk's run stay few, so that
// the warps of an SM keep them cached).
__device__ __forceinline__ void lane_fast_stage(const unsigned char *rp, int sw, int nv, int c, uint64_t &P,
                                                uint64_t &N, bool &anytie, uint32_t &orl, uint32_t &andl) {
  P = 0; N = 0; anytie = false; orl = 0; andl = 0xFFFFFFFFu;
#pragma unroll 1
  for (int q = 0; q < kLaneTerms / 2; q++) {
    const uint4 v = *reinterpret_cast<const uint4 *>(rp + ((q ^ sw) << 4));
#pragma unroll
    for (int h = 0; h < 2; h++) {
      const bool in = 2 * q + h < nv;
      const uint32_t hi = in ? (h ? v.w : v.y) : 0u, lo = in ? (h ? v.z : v.x) : 0u;
      uint64_t ri;
      bool tie;
      term_inc_fast(hi, lo, c, ri, tie);
      if (hi >> 31) N += ri; else P += ri;
      anytie |= tie;
      if (in) { orl |= hi; andl &= hi; }
    }
  }
}
// The fast rule applies to binade e for terms whose largest magnitude word
// is mx: e in range and every term below 2^e.
__device__ __forceinline__ bool fast_ok(int e, uint32_t mx) {
  return e >= -969 && e <= 1023 && (int)(mx >> 20) < e + 1023;
}

// The items of up to two dirty lanes of this warp's chunk (Research-1433,
// finding 4), each lane's sixteen terms spread over a half-warp: lane i of a
// half takes term i, its exact fixed-point prefix inside the dirty lane (a
// scan), its prefix range (the dirty lane's starting value cl plus the
// prefixes before and after the term, widened by dl) and so its key -- the
// binade the range stays in, or "carried" -- and its increment for that
// binade.  A segmented scan composes the runs of one key; each carried term
// becomes an item of its own, added one by one by the walk.  The arguments
// are those of the lane's own half (d < 0: no dirty lane for this half).
// Items go to out[base + i] (shared memory) below kChunkSlots, where half 1's
// base is its own base plus half 0's count.  Returns half 0's count | half
// 1's count << 8.  Whole warp.
constexpr int kCarryKey = -4000;
__device__ __forceinline__ Run shfl_run_up16(const Run &r, int arg) {
  Run o;
  const unsigned full = 0xffffffffu;
  o.inc = __shfl_up_sync(full, r.inc, arg, 16);
  o.lo = __shfl_up_sync(full, r.lo, arg, 16);
  o.hi = __shfl_up_sync(full, r.hi, arg, 16);
  o.d = __shfl_up_sync(full, r.d, arg, 16);
  o.flags = __shfl_up_sync(full, r.flags, arg, 16);
  return o;
}
__device__ __noinline__ int place_pair(const Params &p, const unsigned char *stage, bool from_stage, int64_t lstart,
                                       int nv, int w, int d, DF cl, uint32_t Lm, float dl, uint64_t t, Rec *out,
                                       int base) {
  const int lane = threadIdx.x & 31, hl = lane & 15, half = lane >> 4;
  const unsigned full = 0xffffffffu;
  const bool act = d >= 0 && hl < nv;
  uint64_t x = 0;
  if (act) {
    if (from_stage) {
      const unsigned char *rp = stage + (w * 32 + d) * 128;
      const uint2 v = *reinterpret_cast<const uint2 *>(rp + ((((hl >> 1) ^ (d & 7)) << 4) | ((hl & 1) << 3)));
      x = ((uint64_t)v.y << 32) | v.x;
    } else if (sq_ok(p, lstart >= 0 && lstart + nv <= p.n, 3, lstart)) {
      x = __ldg(reinterpret_cast<const unsigned long long *>(p.x) + lstart + hl);
    }
  }
  const uint32_t hi = (uint32_t)(x >> 32), lo = (uint32_t)x, E = (hi >> 20) & 0x7FFu;
  const int64_t mag = (int64_t)__funnelshift_rc(lead32(hi, lo, E), 0u, Lm - E);
  const int64_t v = (hi >> 31) ? -mag : mag;
  int64_t incl = v;
#pragma unroll
  for (int o = 1; o < kLaneTerms; o <<= 1) {
    const int64_t u = __shfl_up_sync(full, incl, o, 16);
    if (hl >= o) incl += u;
  }
  const float sc = pow2f((int)Lm - 1054);
  const DF a0 = df_addf(cl, __fmul_rn(f_from_i48(incl - v), sc));
  const DF a1 = df_addf(cl, __fmul_rn(f_from_i48(incl), sc));
  const bool up = v >= 0;
  int ei = 0;
  bool ok = act && one_binade_df(df_addf(up ? a0 : a1, -dl), df_addf(up ? a1 : a0, dl), ei);
  ok = act && plan_override(p.plan_mode, ok, ei, t, w, 100 + (d < 0 ? 0 : d) * 16 + hl);
  // a term with |x| >= 2^ei, inf or NaN can never be in a run for ei
  const int xe = E ? (int)E - 1023 : -1022;
  if (E == 0x7FFu || xe >= ei) ok = false;
  const int key = ok ? ei : kCarryKey;
  Run r = run_empty();
  if (ok) {
    int64_t re;
    int32_t dd;
    term_inc(x, key, re, dd);
    run_push(r, re, dd, term_flags(x));
  }
  // segments: a head where the key changes; every carried term stands alone
  const int pkey = __shfl_up_sync(full, key, 1, 16);
  const bool head = act && (hl == 0 || key != pkey || key == kCarryKey);
  Run s = r;
  int f = head ? 1 : 0;
#pragma unroll 1
  for (int o = 1; o < kLaneTerms; o <<= 1) {
    const Run os = shfl_run_up16(s, o);
    const int of = __shfl_up_sync(full, f, o, 16);
    if (hl >= o) { if (!f) s = run_compose(os, s); f |= of; }
  }
  const uint32_t heads = (__ballot_sync(full, head) >> (half * 16)) & 0xFFFFu;
  const bool end = act && (hl == nv - 1 || ((heads >> (hl + 1)) & 1u));
  const uint32_t ends = (__ballot_sync(full, end) >> (half * 16)) & 0xFFFFu;
  const int cnt = __popc(ends);
  const int cnt0 = __shfl_sync(full, cnt, 0), cnt1 = __shfl_sync(full, cnt, 16);
  const int idx = base + (half ? cnt0 : 0) + __popc(ends & ((1u << hl) - 1u));
  if (end && idx < kChunkSlots) {
    const uint32_t tbase = (uint32_t)(w * kChunkTerms + d * kLaneTerms);
    if (key == kCarryKey) {
      Run tr = run_empty();
      tr.inc = (int64_t)x; tr.lo = 0; tr.hi = 0; tr.d = 0;
      tr.flags = term_flags(x) & (F_HASINF_P | F_HASINF_N | F_HASNAN);
      out[idx] = make_rec(tr, 0, K_TERMS, 1u, tbase + (uint32_t)hl);
    } else {
      const int hlead = 31 - __clz(heads & ((2u << hl) - 1u));
      out[idx] = make_rec(s, key, K_RUN, (uint32_t)(hl - hlead + 1), tbase + (uint32_t)hlead);
    }
  }
  return cnt0 | (cnt1 << 8);
}

// A chunk the plan could not place in one binade.  Each lane's starting value
// is the chunk's plus the fixed-point sums of the earlier lanes; a lane whose
// own range stays in one binade becomes one run (neighbouring runs of one
// binade merge), the others are placed term by term.  Writes the items for
// chunk w into the tile's item area and returns their number, or 0 when they
// do not fit (the caller then records the chunk as one fallback).
__device__ __noinline__ int split_chunk(const Params &p, const unsigned char *stage, const StageGeo &g, int w,
                                        int lane, int nv, int64_t lstart, const ChunkPre &pre, Rec *area,
                                        Rec *stg, unsigned int *st) {
  const unsigned full = 0xffffffffu;
  // the stage may already hold the next unit's terms: this chunk's come
  // from global memory
  const bool use_tma = false;
  const int64_t row = (g.start >> 4) + w * 32 + lane;
  const uint64_t t = (uint64_t)g.t;
  PROF_START;
  uint64_t xs[kLaneTerms];
  load_lane(p, stage, use_tma, row, lstart, nv, w, lane, xs);
  uint32_t mx = 0, orz = 0, andh = 0xFFFFFFFFu;
#pragma unroll
  for (int i = 0; i < kLaneTerms; i++) {
    const uint32_t hi = (uint32_t)(xs[i] >> 32);
    const uint32_t mag = hi & 0x7FFFFFFFu;
    mx = max(mx, mag);
    orz |= mag | (uint32_t)xs[i];
    if (i < nv) andh &= hi;
  }
  const uint32_t Lm = mx >> 20;
  uint64_t all, neg;
  lane_fixed(xs, Lm, all, neg);
  const uint32_t Lc = __reduce_max_sync(full, Lm), sh = min(Lc - Lm, 63u);
  const int64_t sv = (int64_t)((all - neg) >> sh) - (int64_t)(neg >> sh);
  // the earlier lanes' signed sum, at the chunk's scale
  int64_t is = sv;
#pragma unroll 1
  for (int o = 1; o < 32; o <<= 1) {
    const int64_t v = __shfl_up_sync(full, is, o);
    if (lane >= o) is += v;
  }
  const DF cl = df_add(pre.c, df_fixed(is - sv, (int)Lc));
  const float Pl = f_fixed(all - neg, (int)Lm), Nl = f_fixed(neg, (int)Lm);
  const float dl = pre.delta;
  int e_l = 0;
  bool clean = one_binade_df(df_addf(cl, -(Nl + dl)), df_addf(cl, Pl + dl), e_l);
  clean = plan_override(p.plan_mode, clean, e_l, t, w, lane + 1);
  const bool zl = (orz == 0);
  const bool dirty = !clean && !zl && nv > 0;
  SPLIT_PT(0);                                                // lane sums, prefixes, verdicts
  Run r = run_empty();                                       // a lane of zeros: a run of zeros
  if (zl && !(andh >> 31)) r.flags &= ~F_ALLNEGZ;             // (all -0 only if every term is -0)
  if (clean && !zl) {
    bool done = false;
    if (fast_ok(e_l, mx)) {
      uint64_t P, N;
      bool anytie;
      uint32_t orl, andl;
      lane_fast(xs, nv, 64 - (e_l + 1023), P, N, anytie, orl, andl);
      if (!anytie) { r = lane_pn_run(P, N, orl, andl, nv); done = true; }
    }
    if (!done) r = lane_run_general(p, stage, use_tma, row, lstart, nv, w, lane, e_l);
  }
  __syncwarp();
  SPLIT_PT(1);                                                // clean lanes' runs
  const int key = dirty ? kDirtyKey : (clean ? e_l : kZeroE);
  if (dirty) atomicAdd(&st[S_LANE_DIRTY], 1u);
  // merge neighbouring runs of one key (lanes past the end join the previous)
  const int pkey = __shfl_up_sync(full, key, 1);
  const bool head = (lane == 0) || (nv > 0 && (dirty || pkey == kDirtyKey || key != pkey));
  Run v = r;
  int fl = head ? 1 : 0;
#pragma unroll 1
  for (int o = 1; o < 32; o <<= 1) {
    const Run ov = shfl_run<SH_UP>(v, o);
    const int of = __shfl_up_sync(full, fl, o);
    if (lane >= o) { if (!fl) v = run_compose(ov, v); fl |= of; }
  }
  const uint32_t heads = __ballot_sync(full, head);
  const bool end = (lane == 31) || ((heads >> (lane + 1)) & 1u);
  const uint32_t le = heads & ((lane == 31) ? full : ((2u << lane) - 1u));
  const int hlane = 31 - __clz(le);
  const int hkey = __shfl_sync(full, key, hlane);
  // terms before each lane, for the item counts
  int csum = nv;
#pragma unroll 1
  for (int o = 1; o < 32; o <<= 1) {
    const int vv = __shfl_up_sync(full, csum, o);
    if (lane >= o) csum += vv;
  }
  const int before_head = __shfl_sync(full, csum - nv, hlane);
  // the chunk's items in lane order, staged in shared memory: a merged run at
  // its end lane, a dirty lane's own items; if they do not fit, each dirty
  // lane becomes one fallback item instead
  SPLIT_PT(2);                                                // merges and counts
  const uint32_t dirtym = __ballot_sync(full, dirty);
  const uint32_t cleanm = __ballot_sync(full, !dirty && end && hkey != kDirtyKey);
  const Rec myrun = make_rec(v, hkey, K_RUN, (uint32_t)(csum - before_head), (uint32_t)(w * kChunkTerms + hlane * kLaneTerms));
  const uint32_t below = (1u << lane) - 1u;
  int n = 0;
  uint32_t emitted = 0;                                // lanes whose items are staged
  // dirty lanes two at a time (one per half-warp), each pair preceded by the
  // merged runs of the clean lanes before it
  for (uint32_t m = dirtym; m;) {
    const int d0 = __ffs(m) - 1;
    m &= m - 1;
    const int d1 = m ? __ffs(m) - 1 : -1;
    if (m) m &= m - 1;
    const uint32_t c0 = cleanm & ((1u << d0) - 1u) & ~emitted;
    if (((c0 >> lane) & 1u) && n + __popc(c0 & below) < kChunkSlots) stg[n + __popc(c0 & below)] = myrun;
    n += __popc(c0);
    // the clean items between d0 and d1 go between their items
    const uint32_t gapm = d1 >= 0 ? (cleanm & ((1u << d1) - 1u) & ~((2u << d0) - 1u)) : 0u;
    const int gap = __popc(gapm);
    const int dd = (lane >> 4) ? d1 : d0;
    const int ds = dd < 0 ? 0 : dd;
    const DF cd = DF{__shfl_sync(full, cl.hi, ds), __shfl_sync(full, cl.lo, ds)};
    const int64_t ls = __shfl_sync(full, lstart, ds);
    const int nvd = __shfl_sync(full, nv, ds);
    const uint32_t Lmd = __shfl_sync(full, Lm, ds);
    const bool fs = use_tma && (g.start >> 4) + w * 32 + ds < p.tma_rows;
    const int cc = place_pair(p, stage, fs, ls, nvd, w, dd, cd, Lmd, dl, t, stg, (lane >> 4) ? n + gap : n);
    const int cnt0 = cc & 0xFF, cnt1 = cc >> 8;
    if (((gapm >> lane) & 1u) && n + cnt0 + __popc(gapm & below) < kChunkSlots)
      stg[n + cnt0 + __popc(gapm & below)] = myrun;
    n += cnt0 + gap + cnt1;
    emitted |= (2u << (d1 >= 0 ? d1 : d0)) - 1u;
  }
  {
    const uint32_t cm = cleanm & ~emitted;
    if (((cm >> lane) & 1u) && n + __popc(cm & below) < kChunkSlots) stg[n + __popc(cm & below)] = myrun;
    n += __popc(cm);
  }
  if (n > kChunkSlots) {
    // one item per clean end lane and per dirty lane (at most 32)
    const uint32_t em = cleanm | dirtym;
    n = __popc(em);
    __syncwarp();
    if ((em >> lane) & 1u) {
      if (dirty) {
        Run fr = run_empty();
        uint32_t tf = 0;
#pragma unroll
        for (int i = 0; i < kLaneTerms; i++) tf |= (i < nv) ? term_flags(xs[i]) : 0u;
        fr.flags = tf & (F_HASINF_P | F_HASINF_N | F_HASNAN);
        stg[__popc(em & below)] = make_rec(fr, 0, K_FALLBACK, (uint32_t)nv, (uint32_t)(w * kChunkTerms + lane * kLaneTerms));
      } else {
        stg[__popc(em & below)] = myrun;
      }
    }
  }
  __syncwarp();
  Rec *out = area + w * kChunkSlots;
  if (lane < n && item_ok(p, out + lane, 5)) stcg_rec(out + lane, stg[lane]);
  const int total = n;
  SPLIT_PT(5);                                                // staging written out
  return total;
}

// ---------------------------------------------------------------- a tile's runs
// Compute warp w, a run unit: the verdict on chunk w of the tile from the
// plan words, then the exact run (or items) of chunk w (Research-1433, finding 2 "Inside a binade the loop is an integer
// sum", finding 3 "Ties need the parity of the running integer"); the chunk's
// record goes to sm.chunk[k][w] for the control warp's header.
__device__ __noinline__ void run_chunk(const Params &p, Smem &sm, const unsigned char *stage, int k, int w) {
  const int lane = threadIdx.x & 31;
  const unsigned full = 0xffffffffu;
  unsigned int *st = sm.st;
  const StageGeo &g = sm.geo[k];
  const uint64_t tv = globaltimer();
  CPROF_START;
  ChunkPre pre;
  uint32_t cmx, cflags;
  const int formed = *reinterpret_cast<const volatile int64_t *>(&sm.vtile[k]) == g.t + 1;
  if (__shfl_sync(full, formed, 0)) {
    // another warp formed the unit's verdicts
    __threadfence_block();
    pre = sm.vpre[k][w];
    cmx = sm.vmx[k][w];
    cflags = sm.vfl[k][w];
  } else {
    // ---- the plan words, copied in with the tile (else read again from
    // global memory, bounded): the prefix before the tile and its chunk plans
    const uint32_t tag = (p.epoch << 1) | 1u;
    DF ex;
    float exab;
    if (g.t == g.first_tile) {
      ex = df_from_double(p.s0s ? p.s0s[g.sum] : p.s0);
      exab = fabsf(ex.hi);
    } else {
      const uint64_t A = sm.pre_raw[k][0], B = sm.pre_raw[k][1];
      if ((uint32_t)(A & 0xFF) == tag && (uint32_t)B == tag) {
        ex = status_sum(A);
        exab = status_abs(B);
      } else {
        read_prefix(p, sm, g.t, ex, exab);
      }
    }
    ChunkPlan cp{0ull, 0ull, 0, 0u, 0u, 0u};
    bool have = true;
    if (lane < kWarps) {
      const uint64_t *q = &sm.cplan_raw[k][4 * lane];
      have = cplan_of(q[0], q[1], q[2], q[3], tag, cp);
    }
    if (!__all_sync(full, have)) {
      const uint64_t t0 = globaltimer();
      uint32_t nap = 32;
      while (!__all_sync(full, have)) {
        if (!have) {
          uint64_t w0, w1, w2, w3;
          const uint64_t *q = p.cplan + (g.t * kWarps + lane) * 4;
          ld_vol_v2(q, w0, w1);
          ld_vol_v2(q + 2, w2, w3);
          have = cplan_of(w0, w1, w2, w3, tag, cp);
        }
        if (__any_sync(full, globaltimer() - t0 > kWaitNs)) {
          if (lane == 0) note_timeout(p, ERR_PLAN_TIMEOUT, TO_PLANNED, (uint32_t)g.t, (uint32_t)w);
          cp = ChunkPlan{0ull, 0ull, 0, 0u, WA_NZ | WA_NEG | WA_POS, 0u};    // no plan: every chunk is split
          break;
        }
        __nanosleep(nap);
        nap = min(nap * 2u, 256u);
      }
      if (lane == 0) atomicAdd(&st[S_NS_VERDICT_WAIT], (unsigned)(globaltimer() - t0));
    }
    CPROF_PT(0);                                        // prefix and plan words
    uint32_t lmx, lfl;
    const ChunkPre lp = chunk_verdicts(g, ex, exab, cp, lmx, lfl);
    if (lane < kWarps) { sm.vpre[k][lane] = lp; sm.vmx[k][lane] = lmx; sm.vfl[k][lane] = lfl; }
    __syncwarp();
    if (lane == 0) {
      __threadfence_block();
      *reinterpret_cast<volatile int64_t *>(&sm.vtile[k]) = g.t + 1;
    }
    pre.c = DF{__shfl_sync(full, lp.c.hi, w), __shfl_sync(full, lp.c.lo, w)};
    pre.ab = __shfl_sync(full, lp.ab, w);
    pre.delta = __shfl_sync(full, lp.delta, w);
    pre.e = __shfl_sync(full, lp.e, w);
    pre.mode = __shfl_sync(full, lp.mode, w);
    cmx = __shfl_sync(full, lmx, w);
    cflags = __shfl_sync(full, lfl, w);
    CPROF_PT(1);                                        // the verdict
  }
  if (lane == 0) atomicAdd(&st[S_NS_VERDICT], (unsigned)(globaltimer() - tv));
  const int64_t cstart = g.start + (int64_t)w * kChunkTerms;
  const int cnt_chunk = (int)max((int64_t)0, min((int64_t)kChunkTerms, g.end - cstart));
  const int64_t lstart = cstart + (int64_t)lane * kLaneTerms;
  const int nv = (int)max((int64_t)0, min((int64_t)kLaneTerms, g.end - lstart));
  const int64_t row = (g.start >> 4) + w * 32 + lane;
  int mode = pre.mode, e = pre.e;
  if (p.plan_mode != 0 && mode != CP_ZERO)
    mode = plan_override(p.plan_mode, mode == CP_CLEAN, e, (uint64_t)g.t, w, 0) ? CP_CLEAN : CP_DIRTY;
  Rec *area = p.items + g.t * kTileSlots;
  Rec crec;
  int nitems = 0;
  if (mode != CP_CLEAN) {
    // a zero chunk reads no terms; a split one reads them from global memory
    // (and ends late: the control warp takes no unit for the stage early)
    if (mode == CP_DIRTY && lane == 0) sm.slow[k] = 1;
    release_stage(sm, k);
  }
  if (mode == CP_ZERO) {
    // every term is +0 or -0: a run of zeros (all -0 keeps a -0 sum at -0)
    Run z = run_empty();
    if (cflags & WA_POS) z.flags &= ~F_ALLNEGZ;
    crec = make_rec(z, kZeroE, K_RUN, (uint32_t)cnt_chunk, (uint32_t)(w * kChunkTerms));
    if (lane == 0) atomicAdd(&st[S_CHUNK_RUN], 1u);
  } else if (mode == CP_CLEAN) {
    CPROF_PT(2);
    Run r;
    bool general = true, general_reduce = true;
    // a chunk with terms past the tensor map's rows (the ragged end of x)
    // takes the general path, from global memory (warp-uniform: the fast
    // rule's reductions need the whole warp)
    const bool from_stage = __all_sync(full, g.tma != 0 && row < p.tma_rows);
    if (fast_ok(e, cmx) && from_stage) {
      uint64_t P, N;
      bool anytie;
      uint32_t orl, andl;
      lane_fast_stage(stage + (w * 32 + lane) * 128, lane & 7, nv, 64 - (e + 1023), P, N, anytie, orl, andl);
      if ((cflags & WA_NEG) == 0 && __ballot_sync(full, anytie) == 0) {
        // non-negative terms and no tie: the run is a plain sum of increments
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) P += __shfl_xor_sync(full, P, o);
        r.inc = (int64_t)P; r.lo = 0; r.hi = (int64_t)P; r.d = 0; r.flags = F_NONNEG;
        general = general_reduce = false;
      } else if (!anytie) {
        // positive and negative increments summed apart bound every prefix
        r = lane_pn_run(P, N, orl, andl, nv);
        general = false;
      }
    }
    release_stage(sm, k);
    CPROF_PT(3);                                      // the fast rule
    if (general) r = lane_run_general(p, stage, false, row, lstart, nv, w, lane, e);   // terms from global memory
    if (general_reduce) {
#pragma unroll 1
      for (int off = 1; off < 32; off <<= 1) {
        const Run o = shfl_run<SH_DOWN>(r, off);
        if ((lane & (2 * off - 1)) == 0) r = run_compose(r, o);
      }
    }
    CPROF_PT(4);                                      // general path and reduction
    crec = make_rec(r, (r.flags & F_ZERO) ? kZeroE : e, K_RUN, (uint32_t)cnt_chunk, (uint32_t)(w * kChunkTerms));
    if (lane == 0) atomicAdd(&st[S_CHUNK_RUN], 1u);
    CPROF_PT(5);                                      // the record
  } else {
    if (lane == 0) atomicAdd(&st[S_CHUNK_DIRTY], 1u);
    nitems = split_chunk(p, stage, g, w, lane, nv, lstart, pre, area, sm.stg[threadIdx.x >> 5], st);
    if (nitems == 0) {
      Run fr = run_empty();
      fr.flags = ((cmx >= 0x7FF00000u) ? (F_HASINF_P | F_HASINF_N | F_HASNAN) : 0u);
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

// Control warp, after a tile's runs: the tile's header -- one run when every
// chunk is a run of one binade (runs of zeros fit any), else the chunks'
// items in the tile's item area.
__device__ __noinline__ void group_done(const Params &p, Smem &sm, int64_t t, int64_t ntiles);
__device__ __noinline__ void run_epilogue(const Params &p, Smem &sm, int k, int64_t ntiles) {
  const int lane = threadIdx.x & 31;
  unsigned int *st = sm.st;
  const StageGeo &g = sm.geo[k];
  const int64_t t = g.t;
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
  __syncwarp();
  if (lane == 0) TRACE_UNIT(t, 1, 6, globaltimer());
  group_done(p, sm, t, ntiles);
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
// a whole batch of uniform tiles [pos, pos + m) applied as one composite
#define WALK_TRACE_T0(p, pos, m, Sb)                                                                  \
  walk_trace((p), tile_geo((p), (pos), ntiles).start, tile_geo((p), (pos) + (m) - 1, ntiles).end, 7u, (Sb))
#else
#define WALK_TRACE(a, b, what, Sb) do { } while (0)
#define WALK_TRACE_T0(p, pos, m, Sb) do { } while (0)
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
__device__ __noinline__ void walk_batch(const Params &p, Smem &sm, unsigned char *dyn, int k, int64_t tb,
                                        int64_t te, int64_t ntiles) {
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
  int64_t pos = tb;
  uint64_t t_work0 = 0;
  int nbatch = 0;
  (void)nbatch;
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
      // a batch has a fixed cost of a few microseconds, so the walk takes at
      // least kWalkMinTiles ready tiles (or the rest of the sum); early
      // batches overlap with the stream
      if (m >= min(want, kWalkMinTiles)) break;
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
      TRACE_BATCH(nbatch, 0, t_work0);
      TRACE_BATCH(nbatch, 2, ((unsigned long long)m << 32) | (uint64_t)pos);
      atomicAdd(&st[S_NS_WALK_WAIT], (unsigned)(t_work0 - t0));
      if (pos + m >= te) p.stats[S_T_WALK0] = t_work0;
    }
    // ---- the common case: every header of the batch is a run of one binade
    //      (or every one a run of zeros); they compose in order, by a tree
    //      over the threads, and the walk applies the one composite.  If its
    //      check refuses it, the batch takes the general path below.
    {
      int k0 = kZeroE - 1;                             // "not uniform" unless header 0 is a run
      if (rec_kind(hdrs[0].meta) == K_RUN) k0 = elem_key(hdrs[0]);
      bool uni = k0 != kZeroE - 1;
      Run r = run_empty();
#pragma unroll
      for (int q = 0; q < PT; q++) {
        const int i = PT * tid + q;
        if (i < m) {
          const Rec h = hdrs[i];
          uni = uni && rec_kind(h.meta) == K_RUN && elem_key(h) == k0;
          r = run_compose(r, rec_run(h));
        }
      }
#pragma unroll 1
      for (int off = 1; off < 32; off <<= 1) {
        const Run o = shfl_run<SH_DOWN>(r, off);
        if ((lane & (2 * off - 1)) == 0) r = run_compose(r, o);
      }
      const bool wuni = __all_sync(full, uni);
      if (lane == 0) { sm.wagg[warp] = r; sm.wflag[warp] = wuni ? 1 : 0; }
      wide_sync(p, sm, 26);
      if (tid == 0) {
        bool all = true;
        Run c = run_empty();
        for (int w2 = 0; w2 < kWarps; w2++) {
          all = all && sm.wflag[w2] != 0;
          c = run_compose(c, sm.wagg[w2]);
        }
        sm.restart = 0;
        if (all) {
          uint64_t Sb = sm.S;
          if (nonfinite(Sb)) {
            sm.S = absorb(Sb, c.flags);
            sm.restart = 1;
          } else if (run_apply(Sb, c, k0) == APPLY_OK) {
            sm.S = Sb;
            sm.restart = 1;
          }
          if (sm.restart) {
            atomicAdd(&st[S_WALK_SEGMENTS], 1u);
            WALK_TRACE_T0(p, pos, m, sm.S);
          }
        }
      }
      wide_sync(p, sm, 27);
      if (sm.restart) {
        pos += m;
        if (tid == 0) { TRACE_BATCH(nbatch, 1, globaltimer()); TRACE_BATCH(nbatch, 3, (unsigned long long)m); }
        nbatch++;
        wide_sync(p, sm, 28);                          // sm.restart and the batch buffers may be reused
        continue;
      }
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
    if (tid == 0) { TRACE_BATCH(nbatch, 1, globaltimer()); TRACE_BATCH(nbatch, 3, (unsigned long long)nel); }
    nbatch++;
    wide_sync(p, sm, 19);
    WALK_PT(15);
  }
  (void)t_work0;
  wide_sync(p, sm, 21);
}

// ---------------------------------------------------------------- composed groups
// Groups of kGroupTiles consecutive tiles.  The streaming CTA that publishes
// the last header of a group composes the group for the walk (Research-1433,
// open question "compose runs of chunks that share a binade so that the walk
// steps over 64 or 1024 chunks at a time"): the group's records are listed in
// order (simple tile headers, the items of complex tiles), every maximal
// stretch of runs of one binade is composed into one segment, and the walk
// then only applies the segments.  A group that composes into more than
// kGroupSegs segments is published "raw": the walk takes its tiles one by one.

// The group's records composed into segments (one warp).  Every header of the
// group is published.
__device__ __noinline__ void compose_group(const Params &p, Smem &sm, int64_t g, int nt, int64_t ntiles) {
  const int lane = threadIdx.x & 31;
  const unsigned full = 0xffffffffu;
  const uint32_t tag = (p.epoch << 1) | 1u;
  const int64_t t0 = g * kGroupTiles;
  // lane c: tile c's header, its number of records (one, or a complex
  // tile's items), whether it starts a sum, and its first record's index
  Rec h = make_rec(run_empty(), kZeroE, K_RUN, 0, 0);
  int cnt = 0;
  bool okh = true, first = false;
  if (lane < nt) {
    okh = read_header(p.hdr + t0 + lane, tag, h) == 1;
    if (okh) {
      if (rec_kind(h.meta) == K_COMPLEX) {
        const uint64_t packed = (uint64_t)h.inc;
#pragma unroll
        for (int cc = 0; cc < kWarps; cc++) cnt += (int)((packed >> (kCountBits * cc)) & kCountMask);
      } else {
        cnt = 1;
      }
    }
    // a tile that starts a sum starts a segment (batched calls)
    first = (p.offsets == nullptr) ? (t0 + lane == 0) : (tile_geo(p, t0 + lane, ntiles).first_tile == t0 + lane);
  }
  int off = cnt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(full, off, o);
    if (lane >= o) off += v;
  }
  const int E = __shfl_sync(full, off, 31);
  off -= cnt;
  bool raw = !__all_sync(full, okh);
  int nseg = 0;
  if (!raw) {
    // rounds of 32 records read straight from the headers and item areas
    // (lane j record base + j), composed by a segmented scan; the last lane's
    // open segment is carried into the next round, and emitted there when
    // that round starts a new one
    Run cv = run_empty();
    Rec cx = h;
    int ckey = 0;
    bool calone = true, copen = false;
    uint32_t ctile = 0;
    for (int base = 0; base < E; base += 32) {
      const int j = base + lane;
      const bool valid = j < E;
      // the record's tile: the last tile whose first record is at or before j
      int c = 0;
#pragma unroll
      for (int step = 16; step > 0; step >>= 1) {
        const int cand = c + step;
        const int oc = __shfl_sync(full, off, min(cand, 31));
        if (cand < nt && oc <= j) c = cand;
      }
      const int oc = __shfl_sync(full, off, c);
      Rec x;
      x.inc = __shfl_sync(full, h.inc, c);
      x.lo = __shfl_sync(full, h.lo, c);
      x.hi = __shfl_sync(full, h.hi, c);
      x.meta = __shfl_sync(full, h.meta, c);
      x.e = (int16_t)__shfl_sync(full, (int)h.e, c);
      x.count = (uint16_t)__shfl_sync(full, (int)h.count, c);
      const bool fc = __shfl_sync(full, first, c);
      if (valid && rec_kind(x.meta) == K_COMPLEX) {
        // item j - oc of the tile: the chunk whose running count passes it
        const uint64_t packed = (uint64_t)x.inc;
        const int i = j - oc;
        int cc = 0, before = 0;
        for (; cc < kWarps; cc++) {
          const int n = (int)((packed >> (kCountBits * cc)) & kCountMask);
          if (i < before + n) break;
          before += n;
        }
        x = make_rec(run_empty(), kZeroE, K_RUN, 0, 0);
        const Rec *q = p.items + (t0 + c) * kTileSlots + cc * kChunkSlots + (i - before);
        if (cc < kWarps && item_ok(p, q, 23)) x = ldcg_rec(q);
      }
      if (!valid) x = make_rec(run_empty(), kZeroE, K_RUN, 0, 0);
      const uint32_t tinfo = (uint32_t)c | ((fc && j == oc) ? 0x100u : 0u);   // 0x100: the record starts a sum
      const int key = elem_key(x);
      const bool alone = elem_alone(x);
      int kp = __shfl_up_sync(full, key, 1);
      bool ap = __shfl_up_sync(full, alone, 1);
      if (lane == 0) { kp = ckey; ap = calone; }
      const bool head = valid && (j == 0 || alone || ap || key != kp || (tinfo & 0x100u));
      // the carried segment ends where this round starts a new one
      const bool carry_ends = copen && __shfl_sync(full, head, 0);
      if (carry_ends) {
        if (lane == 0 && nseg < kGroupSegs) {
          stcg_rec(p.grp_seg + g * kGroupSegs + nseg, calone ? cx : make_rec(cv, ckey, K_RUN, 0u, 0u));
          p.grp_stile[g * kGroupSegs + nseg] = (uint16_t)(ctile & 0xFFu);
        }
        nseg++;
      }
      Run v = rec_run(x);
      int f = head ? 1 : 0;
#pragma unroll 1
      for (int o = 1; o < 32; o <<= 1) {
        const Run ov = shfl_run<SH_UP>(v, o);
        const int of = __shfl_up_sync(full, f, o);
        if (lane >= o) { if (!f) v = run_compose(ov, v); f |= of; }
      }
      if (!f && valid && copen && !carry_ends) v = run_compose(cv, v);
      // an end: the group's last record, or one followed by a head in this
      // round (the round's last lane stays open until the next round)
      const uint32_t heads = __ballot_sync(full, head);
      const bool end = valid && (j == E - 1 || (lane < 31 && ((heads >> (lane + 1)) & 1u)));
      const uint32_t ends = __ballot_sync(full, end);
      const int sidx = nseg + __popc(ends & ((1u << lane) - 1u));
      if (end && sidx < kGroupSegs) {
        stcg_rec(p.grp_seg + g * kGroupSegs + sidx, alone ? x : make_rec(v, key, K_RUN, 0u, 0u));
        p.grp_stile[g * kGroupSegs + sidx] = (uint16_t)(tinfo & 0xFFu);
      }
      nseg += __popc(ends);
      // carry the last lane's segment when it did not end
      copen = __shfl_sync(full, valid && !end, 31);
      cv = shfl_run<SH_IDX>(v, 31);
      cx.inc = __shfl_sync(full, x.inc, 31);
      cx.lo = __shfl_sync(full, x.lo, 31);
      cx.hi = __shfl_sync(full, x.hi, 31);
      cx.meta = __shfl_sync(full, x.meta, 31);
      cx.e = (int16_t)__shfl_sync(full, (int)x.e, 31);
      cx.count = (uint16_t)__shfl_sync(full, (int)x.count, 31);
      ckey = __shfl_sync(full, key, 31);
      calone = __shfl_sync(full, alone, 31);
      ctile = __shfl_sync(full, tinfo, 31);
    }
    raw = nseg > kGroupSegs;                           // more segments than a group holds: the walk takes its tiles
  }
  __syncwarp();
  if (lane == 0) {
    __threadfence();                                   // the segments before the group's header
    const uint64_t hw = ((uint64_t)tag << 56) | ((uint64_t)(raw ? 1u : 0u) << 16) | (uint64_t)(raw ? 0 : nseg);
    *reinterpret_cast<volatile uint64_t *>(p.grp_hdr + g) = hw;
  }
}

// After tile t's header is published (control warp): count the tile in its
// group; the CTA that completes the group composes it.
__device__ __noinline__ void group_done(const Params &p, Smem &sm, int64_t t, int64_t ntiles) {
  const int lane = threadIdx.x & 31;
  const int64_t g = t / kGroupTiles;
  const int nt = (int)min((int64_t)kGroupTiles, ntiles - g * kGroupTiles);
  int last = 0;
  const uint64_t tc = globaltimer();
  if (lane == 0) {
    // release: this tile's header (and items) before its count; acquire:
    // the other tiles' headers after their counts, for the composer.  The
    // composer puts the counter back to 0 for the next call.
    last = (int)add_acq_rel(p.grp_cnt + g, 1u) + 1 == nt;
    atomicAdd(&sm.st[S_NS_GCOUNT], (unsigned)(globaltimer() - tc));
  }
  if (!__shfl_sync(0xffffffffu, last, 0)) return;
  const uint64_t t1 = globaltimer();
  if (lane == 0) p.grp_cnt[g] = 0u;                   // every tile of the group has counted
  compose_group(p, sm, g, nt, ntiles);
  if (lane == 0) atomicAdd(&sm.st[S_NS_COMPOSE], (unsigned)(globaltimer() - t1));
}

// Warp 0 of the walk: apply the staged segments of one group whose tile lies
// in [lo, hi) (tile offsets in the group) to the exact running sum Sb, in
// order.  False when the exact check refuses one: Sb is then unchanged and
// the walk takes the group's tiles one by one.  Counts segments and terms.
__device__ __forceinline__ bool apply_segments(const Params &p, uint64_t &Sb0, const Rec *seg, const uint16_t *stile,
                                               int nseg, int64_t g0, int lo, int hi, int64_t ntiles, unsigned int *st,
                                               unsigned &napplied, unsigned &nterms) {
  const int lane = threadIdx.x & 31;
  uint64_t Sb = Sb0;
  unsigned na = 0, nt = 0;
  for (int s = 0; s < nseg; s++) {
    const int ti = stile[s] & 0xFF;
    if (ti < lo || ti >= hi) continue;
    const Rec c = seg[s];
    const uint32_t kind = rec_kind(c.meta);
    na++;
    if (nonfinite(Sb)) { Sb = absorb(Sb, rec_flags(c.meta)); continue; }
    if (kind == K_RUN) {
      uint64_t T = Sb;
      if (run_apply(T, rec_run(c), c.e) != APPLY_OK) return false;
      Sb = T;
    } else if (kind == K_TERMS) {
      double S = bitsd(Sb);
      const int n = (int)c.count;
      if (n > 0) S = __dadd_rn(S, bitsd((uint64_t)c.inc));
      if (n > 1) S = __dadd_rn(S, bitsd((uint64_t)c.lo));
      if (n > 2) S = __dadd_rn(S, bitsd((uint64_t)c.hi));
      Sb = dbits(S);
      nt += (unsigned)n;
    } else {                                            // K_FALLBACK
      const TileGeo tg = tile_geo(p, g0 + ti, ntiles);
      Sb = add_terms(p, Sb, tg.start + rec_tstart(c.meta), c.count, st);
      if (lane == 0) atomicAdd(&st[S_CHUNK_FALLBACK], 1u);
    }
  }
  Sb0 = Sb;
  napplied += na;
  nterms += nt;
  return true;
}

// Warp 0 of the walk, the fast path of a round: the staged segments of
// groups g, g + 1, ... (segment i in seg[i], its group in the round and tile
// in the group in code[i] = group << 8 | tile) that lie in the sum's tiles
// [tb, te) are composed once more -- consecutive runs of one binade across
// the groups merge, every other record stands alone -- and the composites
// applied in order (run composition is associative: Research-1433, finding
// 2).  The composites overwrite the staged segments.  False, with Sb
// unchanged, when the check refuses one.
__device__ __noinline__ bool walk_fast(const Params &p, uint64_t &Sb0, Rec *seg, uint16_t *code, int total,
                                       int64_t g, int64_t tb, int64_t te, int64_t ntiles, unsigned int *st,
                                       unsigned &napplied, unsigned &nterms) {
  const int lane = threadIdx.x & 31;
  const unsigned full = 0xffffffffu;
  Run carry = run_empty();
  bool carry_open = false, alone_prev = true, valid_prev = false;
  int key_prev = 0, nc = 0;
  for (int base = 0; base < total; base += 32) {
    const int j = base + lane;
    Rec x = make_rec(run_empty(), kZeroE, K_RUN, 0, 0);
    uint32_t cj = 0;
    bool valid = false;
    if (j < total) {
      x = seg[j];
      cj = code[j];
      const int64_t t = (g + (cj >> 8)) * kGroupTiles + (cj & 0xFFu);
      valid = t >= tb && t < te;
    }
    const int key = elem_key(x);
    const bool alone = elem_alone(x);
    int kp = __shfl_up_sync(full, key, 1);
    bool ap = __shfl_up_sync(full, alone, 1), vp = __shfl_up_sync(full, valid, 1);
    if (lane == 0) { kp = key_prev; ap = alone_prev; vp = valid_prev; }
    const bool head = valid && (j == 0 || !vp || alone || ap || key != kp);
    Run v = rec_run(x);
    int f = head ? 1 : 0;
#pragma unroll 1
    for (int o = 1; o < 32; o <<= 1) {
      const Run ov = shfl_run<SH_UP>(v, o);
      const int of = __shfl_up_sync(full, f, o);
      if (lane >= o) { if (!f) v = run_compose(ov, v); f |= of; }
    }
    if (!f && valid && carry_open) v = run_compose(carry, v);
    // an end: followed by a head, an invalid record or nothing (for the
    // round's last lane the next round's first record decides)
    const uint32_t heads = __ballot_sync(full, head), valids = __ballot_sync(full, valid);
    bool nexthead = (heads >> (lane + 1)) & 1u, nextvalid = (valids >> (lane + 1)) & 1u;
    if (lane == 31 && valid && j + 1 < total) {
      const Rec xn = seg[j + 1];
      const uint32_t cn = code[j + 1];
      const int64_t tn = (g + (cn >> 8)) * kGroupTiles + (cn & 0xFFu);
      nextvalid = tn >= tb && tn < te;
      nexthead = elem_alone(xn) || alone || elem_key(xn) != key;
    }
    const bool end = valid && (j == total - 1 || !nextvalid || nexthead);
    const uint32_t ends = __ballot_sync(full, end);
    const int o = nc + __popc(ends & ((1u << lane) - 1u));
    __syncwarp();                                      // every record read before any is overwritten
    if (end) {
      seg[o] = alone ? x : make_rec(v, key, K_RUN, 0u, 0u);
      code[o] = (uint16_t)cj;
    }
    nc += __popc(ends);
    carry_open = __shfl_sync(full, valid && !end, 31);
    carry = shfl_run<SH_IDX>(v, 31);
    key_prev = __shfl_sync(full, key, 31);
    alone_prev = __shfl_sync(full, alone, 31);
    valid_prev = __shfl_sync(full, valid, 31);
    __syncwarp();
  }
  uint64_t Sb = Sb0;
  unsigned na = 0, nt = 0;
  for (int base = 0; base < nc; base += 32) {
    const int nb = min(32, nc - base);
    // lane j prepares composite base + j for a positive normal sum: the
    // exponent field it needs and, per parity of the significand m, its
    // increment and the range of m that run_apply accepts -- so that the
    // in-order step is a few operations and three shuffles
    Rec cj = make_rec(run_empty(), kZeroE, K_RUN, 0, 0);
    if (lane < nb) cj = seg[base + lane];
    const uint32_t fj = rec_flags(cj.meta);
    const bool simple = lane < nb && rec_kind(cj.meta) == K_RUN && !(fj & (F_ZERO | F_POISON));
    const uint32_t Ej = (uint32_t)(cj.e + 1023);
    const int64_t inc0 = cj.inc, inc1 = cj.inc + rec_d(cj.meta);
    int64_t lo0, lo1, hi0, hi1;
    if (fj & F_NONNEG) {                               // m + inc <= 2^53
      lo0 = lo1 = kTwo52;
      hi0 = kTwo53 - inc0;
      hi1 = kTwo53 - inc1;
    } else {                                           // m + lo - p >= 2^52 + 1, m + hi + p <= 2^53 - 1
      lo0 = kTwo52 + 1 - cj.lo;
      lo1 = kTwo52 + 2 - cj.lo;
      hi0 = kTwo53 - 1 - cj.hi;
      hi1 = kTwo53 - 2 - cj.hi;
    }
    const uint32_t simple_m = __ballot_sync(full, simple);
    for (int sl = 0; sl < nb; sl++) {
      const int s = base + sl;
      const uint32_t Es = __shfl_sync(full, Ej, sl);
      const uint64_t mag = Sb & ~kSignBit;
      if (((simple_m >> sl) & 1u) && !(Sb >> 63) && (uint32_t)(mag >> 52) == Es) {
        const int64_t m = (int64_t)((mag & kFracMask) | kHidden);
        const bool odd = (m & 1) != 0;
        const int64_t inc = __shfl_sync(full, odd ? inc1 : inc0, sl);
        const int64_t L = __shfl_sync(full, odd ? lo1 : lo0, sl), H = __shfl_sync(full, odd ? hi1 : hi0, sl);
        na++;
        if (m < L || m > H) return false;
        Sb = mag + (uint64_t)inc;                      // m stays in [2^52, 2^53]: the bits follow
        continue;
      }
      const Rec c = seg[s];
      const uint32_t kind = rec_kind(c.meta);
      na++;
      if (nonfinite(Sb)) { Sb = absorb(Sb, rec_flags(c.meta)); continue; }
      if (kind == K_RUN) {
        uint64_t T = Sb;
        if (run_apply(T, rec_run(c), c.e) != APPLY_OK) return false;
        Sb = T;
      } else if (kind == K_TERMS) {
        double S = bitsd(Sb);
        const int n = (int)c.count;
        if (n > 0) S = __dadd_rn(S, bitsd((uint64_t)c.inc));
        if (n > 1) S = __dadd_rn(S, bitsd((uint64_t)c.lo));
        if (n > 2) S = __dadd_rn(S, bitsd((uint64_t)c.hi));
        Sb = dbits(S);
        nt += (unsigned)n;
      } else {                                            // K_FALLBACK
        const uint32_t cs = code[s];
        const TileGeo tg = tile_geo(p, (g + (cs >> 8)) * kGroupTiles + (cs & 0xFFu), ntiles);
        Sb = add_terms(p, Sb, tg.start + rec_tstart(c.meta), c.count, st);
        if (lane == 0) atomicAdd(&st[S_CHUNK_FALLBACK], 1u);
      }
    }
  }
  Sb0 = Sb;
  napplied += na;
  nterms += nt;
  return true;
}

// Walk sum k over its tiles [tb, te) group by group, as the groups are
// composed.  Warp 0 reads ahead the headers of up to 32 groups, stages their
// segments in shared memory and applies them in order; the other warps wait
// at a barrier and join only to walk the tiles of a group that is raw or
// whose segments the check refuses (walk_batch).
constexpr int kWalkStageSegs = 512;                   // staged segments (after the batch buffers)
constexpr int kWalkOffStage = 73728;
static_assert(kWalkOffStage + kWalkStageSegs * ((int)sizeof(Rec) + 2) <= kStages * kStageBytes, "walk staging");
__device__ __noinline__ void walk_batch(const Params &p, Smem &sm, unsigned char *dyn, int k, int64_t tb,
                                        int64_t te, int64_t ntiles);
__device__ __noinline__ void walk_sum(const Params &p, Smem &sm, unsigned char *dyn, int k, int64_t tb, int64_t te,
                                      int64_t ntiles) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const unsigned full = 0xffffffffu;
  const uint32_t tag = (p.epoch << 1) | 1u;
  unsigned int *st = sm.st;
  Rec *seg = reinterpret_cast<Rec *>(dyn + kWalkOffStage);
  uint16_t *stile = reinterpret_cast<uint16_t *>(dyn + kWalkOffStage + kWalkStageSegs * sizeof(Rec));
  if (tid == 0) sm.S = dbits(p.s0s ? p.s0s[k] : p.s0);
  wide_sync(p, sm, 6);
  if (warp != 0) {
    // the helpers: a command from warp 0 (a range of tiles to walk), or the end
    while (true) {
      wide_sync(p, sm, 32);
      const int cmd = sm.nseg;
      const int64_t a = sm.wpos0, b = sm.wpos1;
      wide_sync(p, sm, 33);
      if (cmd == 0) break;
      walk_batch(p, sm, dyn, k, a, b, ntiles);
    }
    return;
  }
  uint64_t twait = 0;
  const uint64_t tbeg = globaltimer();
  const int64_t gend = (te - 1) / kGroupTiles + 1;
  uint64_t Sb = sm.S;                                  // the exact running sum (every lane of warp 0)
  unsigned napplied = 0, nterms = 0;
  int nround = 0;
  (void)nround;
  bool failed = false;
  for (int64_t g = tb / kGroupTiles; g < gend && !failed;) {
    // the ready groups g .. g + r - 1 (bounded wait for group g)
    const uint64_t t0 = globaltimer();
    if (lane == 0) beat(p, sm.role, HB_WAIT_HEADERS, (uint64_t)(g * kGroupTiles));
    uint32_t nap = 32;
    uint64_t hw = 0;
    int r = 0;
    while (true) {
      const int64_t gi = g + lane;
      hw = gi < gend ? *reinterpret_cast<const volatile uint64_t *>(p.grp_hdr + gi) : 0ull;
      const uint32_t rm = __ballot_sync(full, gi < gend && (uint32_t)(hw >> 56) == tag);
      r = (~rm == 0u) ? 32 : __ffs(~rm) - 1;
      if (r > 0) break;
      if (__any_sync(full, globaltimer() - t0 > kWaitNs)) {
        if (lane == 0) note_timeout(p, ERR_WALK_TIMEOUT, TO_WALK, (uint32_t)(g * kGroupTiles), (uint32_t)te);
        failed = true;
        break;
      }
      __nanosleep(nap);
      nap = min(nap * 2u, 256u);
    }
    twait += globaltimer() - t0;
    if (failed) break;
    // stage the segments of the ready groups that fit
    const bool mine = lane < r;
    const int raw = mine ? (int)((hw >> 16) & 1u) : 0;
    const int ns = (mine && !raw) ? (int)(hw & 0xFFFFu) : 0;
    int off = ns;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(full, off, o);
      if (lane >= o) off += v;
    }
    off -= ns;
    const uint32_t fits = __ballot_sync(full, mine && off + ns <= kWalkStageSegs);
    r = (~fits == 0u) ? 32 : __ffs(~fits) - 1;        // at least group g fits (at most kGroupSegs)
    const int total = __shfl_sync(full, off + ns, r - 1);
    auto stage_segments = [&]() {
      // the whole warp loads them, lane l element l, l + 32, ...: element
      // idx belongs to the last group whose offset is at most idx
      for (int base = 0; base < total; base += 32) {
        const int idx = base + lane;
        int gl = 0;
#pragma unroll
        for (int step = 16; step > 0; step >>= 1) {
          const int cand = gl + step;
          const int oc = __shfl_sync(full, off, min(cand, 31));
          if (cand < r && oc <= idx) gl = cand;
        }
        const int og = __shfl_sync(full, off, gl);
        if (idx < total) {
          const int64_t gi = g + gl;
          seg[idx] = ldcg_rec(p.grp_seg + gi * kGroupSegs + (idx - og));
          stile[idx] = (uint16_t)((gl << 8) | (p.grp_stile[gi * kGroupSegs + (idx - og)] & 0xFF));
        }
      }
    };
    stage_segments();
    __syncwarp();
    if (lane == 0) {
      TRACE_BATCH(256 + nround, 0, globaltimer());
      TRACE_BATCH(256 + nround, 2, ((unsigned long long)r << 32) | (uint64_t)g);
    }
#ifdef SEQSUM_PROFILE
    const long long c_apply0 = clock64();
    const unsigned na_before = napplied;
#endif
    // the fast path: the round's segments composed across groups (unless a
    // group is raw); when the check refuses a composite, the round again
    // from its start, group by group
    bool fast = !__any_sync(full, raw != 0) &&
                walk_fast(p, Sb, seg, stile, total, g, tb, te, ntiles, st, napplied, nterms);
    if (!fast && !__any_sync(full, raw != 0)) {
      __syncwarp();
      stage_segments();
      __syncwarp();
    }
    for (int i = 0; i < r && !fast; i++) {
      const int64_t gi = g + i, g0 = gi * kGroupTiles;
      const int lo = (int)(max(g0, tb) - g0), hi = (int)(min(g0 + kGroupTiles, te) - g0);
      const int rawi = __shfl_sync(full, raw, i), nsi = __shfl_sync(full, ns, i), offi = __shfl_sync(full, off, i);
      const bool ok = !rawi && apply_segments(p, Sb, seg + offi, stile + offi, nsi, g0, lo, hi, ntiles, st, napplied, nterms);
      if (!ok) {
        // the whole CTA walks the group's tiles from the sum so far
        if (lane == 0) { sm.S = Sb; sm.nseg = 1; sm.wpos0 = g0 + lo; sm.wpos1 = g0 + hi; }
        if (lane == 0 && !rawi) atomicAdd(&st[S_RUN_REJECTED], 1u);
        wide_sync(p, sm, 32);
        wide_sync(p, sm, 33);
        walk_batch(p, sm, dyn, k, g0 + lo, g0 + hi, ntiles);
        Sb = sm.S;
      }
    }
    if (lane == 0) TRACE_BATCH(256 + nround, 1, globaltimer());
#ifdef SEQSUM_PROFILE
    if (lane == 0) TRACE_BATCH(256 + nround, 3, ((unsigned long long)(clock64() - c_apply0) << 20) | (napplied - na_before) | ((unsigned long long)smid() << 12));
#endif
    nround++;
    g += r;
  }
  // release the helpers
  if (lane == 0) {
    sm.nseg = 0;
    sm.S = Sb;
    atomicAdd(&st[S_WALK_SEGMENTS], napplied);
    if (nterms) atomicAdd(&st[S_TERMS_ADDED], nterms);
  }
  wide_sync(p, sm, 32);
  wide_sync(p, sm, 33);
  if (lane == 0) {
    p.outs[k] = failed ? __longlong_as_double(0x7FF8000000000000ll) : bitsd(Sb);
    const uint64_t tend = globaltimer();
    p.stats[S_T_WALK1] = tend;
    atomicAdd(&st[S_NS_WALK_WAIT], (unsigned)twait);
    atomicAdd(&st[S_NS_WALK_WORK], (unsigned)(tend - tbeg - twait));
  }
}

// ---------------------------------------------------------------- the streaming loops
// A streaming CTA has eight compute warps and a control warp, and three
// stages.  Per stage three mbarriers: full (the unit's copies landed and its
// description -- sm.geo, the claim word -- is written), used (its chunks have
// read their terms: the stage may take the next unit's copies) and done (its
// chunks are finished: the control warp's epilogue).  A unit's eight chunks go
// to whichever compute warps claim them.

// The tile a ticket names, found by the control warp (a 32-way search over
// the sums' first tiles for a batched call).
__device__ __noinline__ StageGeo stage_geo(const Params &p, int64_t t) {
  const int lane = threadIdx.x & 31;
  const unsigned full = 0xffffffffu;
  StageGeo g;
  g.t = t;
  g.kind = U_PLAN;
  g.pad = 0;
  if (p.offsets == nullptr) {
    g.sum = 0;
    g.first_tile = 0;
    g.sum_start = 0;
    g.start = t * kTileTerms;
    g.end = min(p.n, g.start + kTileTerms);
  } else {
    // the last sum k with tile_begin[k] <= t; empty sums share their
    // successor's tile_begin, and the search lands on the non-empty one
    // (invariant: tile_begin[lo] <= t < tile_begin[hi])
    int lo = 0, hi = p.nsums;
    while (hi - lo > 1) {
      const int step = (hi - lo + 31) / 32;
      const int idx = lo + lane * step;
      const bool le = idx < hi && __ldcg(&p.tile_begin[idx]) <= t;
      const uint32_t m = __ballot_sync(full, le);          // lane 0 (idx = lo) always
      lo += (31 - __clz(m)) * step;
      hi = min(hi, lo + step);
    }
    g.sum = lo;
    g.first_tile = __ldcg(&p.tile_begin[lo]);
    g.sum_start = p.offsets[lo];
    g.start = g.sum_start + (t - g.first_tile) * kTileTerms;
    g.end = min(p.offsets[lo + 1], g.start + kTileTerms);
  }
  g.tma = (p.tma_rows != 0 && (g.start & 15) == 0) ? 1 : 0;
  return g;
}

// Units of work.  Every tile has a plan unit (copy it, publish its chunks'
// fixed-point sums and the tile's approximate sum) and a run unit (copy it
// again, form its runs under the verdicts that its prefix and chunk sums give).
// Tickets hand out the plan units of the first `wave` tiles, then a run unit
// and a plan unit in turn, then the remaining run units: the plan of tile t
// precedes the run of tile t + 1 by about `wave` tiles, so a run unit's prefix
// is normally published long before it is needed, and its tile is still in L2.
// Returns true for a plan unit.
// The ticket order (units.cuh): plan and run units of the tiles.

// Claim words of the stages.  A unit's chunks go to whichever compute warps
// claim them first, so that a chunk that takes long (a split) holds up only
// its own unit, not the same chunk of the CTA's next units.
constexpr uint32_t kClaimEnd = 0x80u;
__device__ __forceinline__ uint32_t claim_word(uint32_t use, bool end) { return (use << 8) | (end ? kClaimEnd : 0u); }
__device__ __forceinline__ uint32_t read_claim(const Smem &sm, int k) {
  return __shfl_sync(0xffffffffu, *reinterpret_cast<const volatile uint32_t *>(&sm.cnext[k]), 0);
}
// Whether use m of stage k can be claimed from: 1 once its copy has landed
// and the stage still holds it, 0 when the stage has moved on to a later use
// (every chunk of use m was claimed and finished), -1 when the wait gave up.
// Warp-uniform and bounded.
__device__ __forceinline__ int unit_ready(const Params &p, Smem &sm, int k, uint32_t m, int j) {
  const uint32_t par = m & 1u;
  const uint64_t t0 = globaltimer();
  uint32_t nap = 32;
#ifdef SEQSUM_PROFILE
  const long long c0 = clock64();
  int npoll = 0;
#endif
  while (true) {
    if ((int32_t)((read_claim(sm, k) >> 8) - m) > 0) return 0;
    if (mbar_test_warp(&sm.full[k], par)) {
#ifdef SEQSUM_PROFILE
      if ((threadIdx.x & 31) == 0) {
        atomicAdd(&sm.prof[npoll ? 32 : 34], (unsigned)(clock64() - c0));
        atomicAdd(&sm.prof[npoll ? 33 : 35], 1u);
        // the earliest time a waiting warp saw the unit's copies complete
        if (npoll) {
          const int64_t ti = sm.geo[k].t * 2 + sm.geo[k].kind;
          if (ti >= 0 && 54100 + ti < 61440) atomicMax(&p.dbg[54100 + ti], ~0ull - globaltimer());
        }
      }
#endif
      // the phase that completed may already be a later use's
      return (read_claim(sm, k) >> 8) == m ? 1 : 0;
    }
#ifdef SEQSUM_PROFILE
    npoll++;
#endif
    (void)mbar_try_wait(&sm.full[k], par);
    __nanosleep(nap);
    nap = min(nap * 2u, 256u);
    if (__any_sync(0xffffffffu, globaltimer() - t0 > kWaitNs)) {
      if ((threadIdx.x & 31) == 0)
        note_timeout(p, ERR_TMA_TIMEOUT, TO_FULL, (uint32_t)j, (uint32_t)(k | (threadIdx.x >> 5) << 8 | blockIdx.x << 16));
      return -1;
    }
  }
}
// Claim the next chunk of use m of stage k: its index, -1 when none is left,
// -2 at the end marker.  Warp-uniform.
__device__ __forceinline__ int claim_chunk(Smem &sm, int k, uint32_t m) {
  int r = -1;
  if ((threadIdx.x & 31) == 0) {
    uint32_t c = *reinterpret_cast<volatile uint32_t *>(&sm.cnext[k]);
    while (true) {
      if ((c >> 8) != m) break;
      if (c & kClaimEnd) { r = -2; break; }
      if ((c & 0xFFu) >= (uint32_t)kWarps) break;
      const uint32_t prev = atomicCAS(&sm.cnext[k], c, c + 1u);
      if (prev == c) { r = (int)(c & 0xFFu); break; }
      c = prev;
    }
  }
  return __shfl_sync(0xffffffffu, r, 0);
}

// Compute warps: the units of the stages in turn, claiming their chunks,
// until the end marker.
__device__ __noinline__ void compute_loop(const Params &p, Smem &sm, const unsigned char *dyn) {
  const int tid = threadIdx.x, lane = tid & 31;
  unsigned int *st = sm.st;
  CPROF_START;
  for (int j = 0;; j++) {
    const int k = j % kStages;
    const uint32_t m = (uint32_t)(j / kStages);
    const uint64_t tw = (tid == 0) ? globaltimer() : 0;
    if (lane == 0) beat(p, sm.role, HB_WAIT_UNIT, (uint64_t)j);
#ifdef SEQSUM_PROFILE
    const bool armed0 = (read_claim(sm, k) >> 8) == m;
#endif
    const int ready = unit_ready(p, sm, k, m, j);
    if (ready < 0) break;                                // the call has failed
    if (tid == 0) atomicAdd(&st[S_NS_TMA_WAIT], (unsigned)(globaltimer() - tw));
    if (ready == 0) continue;
    CPROF_PT(sm.geo[k].kind == U_RUN ? (armed0 ? 6 : 7) : (armed0 ? 16 : 17));   // waited for a run / plan unit, armed or not
    bool end = false;
    while (true) {
      const int c = claim_chunk(sm, k, m);
      if (c == -2) { end = true; break; }
      if (c < 0) break;
      const int kind = sm.geo[k].kind;
      const int64_t t = sm.geo[k].t;
      const unsigned char *stage = dyn + k * kStageBytes;
      const uint64_t tb = (lane == 0) ? globaltimer() : 0;
      if (lane == 0) beat(p, sm.role, HB_UNIT, ((uint64_t)j << 32) | (uint32_t)t);
      if (c == 0 && lane == 0) TRACE_UNIT(t, kind, 1, tb);
      CPROF_PT(kind == U_PLAN ? 8 : 9);                 // waiting and claiming before a plan / run chunk
      if (kind == U_PLAN) plan_chunk(p, sm, stage, k, c);
      else run_chunk(p, sm, stage, k, c);
      CPROF_PT(kind == U_PLAN ? 10 : 11);               // the plan chunk / the run chunk
      if (c == 0 && lane == 0) {
        const uint64_t te = globaltimer();
        atomicAdd(&st[kind == U_PLAN ? S_NS_PHASE_A : S_NS_PHASE_B], (unsigned)(te - tb));
        TRACE_UNIT(t, kind, 2, te);
      }
      if (lane == 0 && kind == U_RUN)
        TRACE_UNIT_MAX(t, kind, 7, ((globaltimer() - tb) << 20) | ((uint64_t)(sm.nitems[k][c] & 0xFFF) << 8) | (uint64_t)c);
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.done[k]);
    }
    if (end) break;
  }
}

// The control warp: tickets, copies, plan words and tile headers.
__device__ __noinline__ void control_loop(const Params &p, Smem &sm, unsigned char *dyn, const CUtensorMap *tmap,
                                          int64_t ntiles) {
  const int lane = threadIdx.x & 31;
  const int64_t nunits = 2 * ntiles;
  bool beside_walker = false;                            // lane 0
  uint32_t ph = 0;                                       // bit k: parity of done[k]
  CPROF_START;
  auto epilogue = [&](int k) -> bool {
    const uint64_t tw = globaltimer();
    if (lane == 0) beat(p, sm.role + 0x80u, HB_WAIT_DONE, ((uint64_t)k << 32) | (uint32_t)sm.geo[k].t);
    if (!mbar_wait_warp(p, &sm.done[k], (ph >> k) & 1u, ERR_TMA_TIMEOUT, TO_DONE, (uint32_t)sm.geo[k].t,
                        (uint32_t)(k | sm.geo[k].kind << 8 | blockIdx.x << 16)))
      return false;
    ph ^= 1u << k;
    if (lane == 0) {
      atomicAdd(&sm.st[S_NS_CTRL_WAIT], (unsigned)(globaltimer() - tw));
      TRACE_UNIT(sm.geo[k].t, sm.geo[k].kind, 5, globaltimer());
    }
    CPROF_PT(12);                                        // control: waiting for a unit's chunks
    if (sm.geo[k].kind == U_RUN) run_epilogue(p, sm, k, ntiles);   // a plan unit's last warp has published it
    CPROF_PT(13);                                        // control: the epilogue
    if (lane == 0) TRACE_UNIT(sm.geo[k].t, sm.geo[k].kind, 3, globaltimer());
    return true;
  };
  uint32_t uph = 0;                                      // bit k: parity of used[k]
  // lane 0: the next ticket; none at all once the CTA has found that it
  // shares its SM with a walker
  auto ticket = [&](int j) -> uint32_t {
    uint32_t u = 0;
    if (lane == 0) {
      if (j == kStages) {
        const uint32_t me = smid() + 1u;
        for (int i = 0; i < min(p.nwalkers, 2); i++)
          if (*reinterpret_cast<const volatile uint32_t *>(&p.ctr[C_WALK_SM + i]) == me) {
            beside_walker = true;
#ifdef SEQSUM_PROFILE
            p.dbg[16000 + i] = ((unsigned long long)me << 32) | (blockIdx.x + 1u);
#endif
          }
      }
      u = beside_walker ? 0xFFFFFFFFu : atomicAdd(&p.ctr[C_TICKET], 1u);
    }
    return __shfl_sync(0xffffffffu, u, 0);
  };
  // the copies of a unit into stage k: a run unit's plan words (the prefix
  // before the tile, the tile's chunk plans; each copying lane arrives once
  // its copy has landed) and the tile's terms
  auto copy_in = [&](int k, const StageGeo &g, int64_t t, bool plan) {
#ifdef SEQSUM_PROFILE
    if (lane == 0 && 50000 + 2 * t + (plan ? 0 : 1) < 54100) p.dbg[50000 + 2 * t + (plan ? 0 : 1)] = globaltimer();
#endif
    if (!plan && sq_ok(p, t < p.cap_tiles, 22, t)) {
      if (lane == 0 && t > g.first_tile) cp_async16(sm.pre_raw[k], p.status + 2 * (t - 1));
      if (lane >= 1 && lane < kCopyLanes) cp_async16(&sm.cplan_raw[k][2 * (lane - 1)], p.cplan + t * kWarps * 4 + 2 * (lane - 1));
    }
    if (lane < kCopyLanes) cp_async_mbar_arrive(&sm.full[k]);
    __syncwarp();
    if (lane == 0) {
      if (g.tma) {
        fence_proxy_async();                             // the compute warps' reads of this stage came first
        mbar_arrive_expect_tx(&sm.full[k], (uint32_t)kStageBytes);
        tma_load_box(dyn + k * kStageBytes, tmap, &sm.full[k], 0, (int32_t)(g.start >> 4));
      } else {
        mbar_arrive(&sm.full[k]);
      }
    }
  };
  for (int j = 0;; j++) {
    const int k = j % kStages;
    const uint32_t use = (uint32_t)(j / kStages);
    uint32_t u = 0;
    bool have_u = false, copied = false;
    int64_t t = 0;
    bool plan = false;
    StageGeo g;
    if (j >= kStages) {
      // once the stage's unit has read its plan words and terms, the next
      // unit's can be copied in while that unit still computes -- unless a
      // chunk of it is being split: then the CTA takes no ticket that it
      // would hold until the split ends
      if (!mbar_wait_warp(p, &sm.used[k], (uph >> k) & 1u, ERR_TMA_TIMEOUT, TO_DONE, (uint32_t)j,
                          (uint32_t)(k | blockIdx.x << 16)))
        break;
      uph ^= 1u << k;
      if (!sm.slow[k]) {
        u = ticket(j);
        have_u = true;
        if ((int64_t)u < nunits) {
          plan = unit_of((int64_t)u, ntiles, p.wave, p.offsets ? 0 : kHeadTiles, t);
          g = stage_geo(p, t);
          copy_in(k, g, t, plan);
          copied = true;
        }
      }
      if (!epilogue(k)) break;                           // the unit that held this stage (else the call failed)
    }
    CPROF_PT(14);                                        // control: waits, the early copies, the epilogue
#ifdef SEQSUM_PROFILE
    if (lane == 0 && j >= kStages) atomicAdd(&sm.prof[copied ? 36 : 38], 1u);
#endif
    if (!have_u) u = ticket(j);
    if ((int64_t)u >= nunits) {
      if (lane == 0) { sm.geo[k].kind = U_END; sm.cnext[k] = claim_word(use, true); }
      __syncwarp();
      if (lane < kCopyLanes) cp_async_mbar_arrive(&sm.full[k]);     // all the stage's arrivals at once
      if (lane == 0) { mbar_arrive(&sm.full[k]); mbar_arrive(&sm.full[k]); }
      for (int jj = max(j - kStages + 1, 0); jj < j; jj++)
        if (!epilogue(jj % kStages)) break;
      break;
    }
    if (!copied) {
      plan = unit_of((int64_t)u, ntiles, p.wave, p.offsets ? 0 : kHeadTiles, t);
      g = stage_geo(p, t);
    }
    g.kind = plan ? U_PLAN : U_RUN;
    if (lane == 0) {
      sm.geo[k] = g;
      sm.plan_cnt[k] = 0;
      sm.slow[k] = 0;
      sm.cnext[k] = claim_word(use, false);
      TRACE_UNIT(t, g.kind, 0, globaltimer());
      TRACE_UNIT(t, g.kind, 4, ((unsigned long long)blockIdx.x << 32) | u);
    }
    if (!copied) copy_in(k, g, t, plan);
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm.full[k]);             // the unit's description is written
    CPROF_PT(15);                                        // control: arming the stage
  }
}

// ---------------------------------------------------------------- the kernel
__global__ void __launch_bounds__(kBlockThreads, 2)
    seqsum_kernel(const __grid_constant__ Params pk, const __grid_constant__ CUtensorMap tmap) {
  extern __shared__ unsigned char dsm_raw[];
  unsigned char *dyn =
      reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(dsm_raw) + 1023) & ~(uintptr_t)1023);
  __shared__ Smem sm;
  // the parameters, copied to shared memory: the out-of-line functions take
  // them by reference, and a reference into the kernel's parameter space is
  // read through slow generic loads
  __shared__ Params ps;
  const int tid = threadIdx.x;
  if (tid == 0) ps = pk;
  __syncthreads();
  const Params &p = ps;
  const int warp = tid >> 5;
  int64_t ntiles = (p.ntiles >= 0) ? p.ntiles : (int64_t)__ldcg(&p.ctr[C_NTILES]);
  if (ntiles > p.cap_tiles) ntiles = 0;                  // the set-up flagged ERR_CAPACITY
  if (tid < S_COUNT) sm.st[tid] = 0;
#ifdef SEQSUM_PROFILE
  if (tid < 40) sm.prof[tid] = 0u;
#endif
  if (tid < kWarps) sm.barcnt[tid] = 0;
  if (tid == 0) {
    for (int s = 0; s < kStages; s++) {
      mbar_init(&sm.full[s], kFullArrivals);             // the copying lanes and the tile's copy
      mbar_init(&sm.done[s], kWarps);
      mbar_init(&sm.used[s], kWarps);
      sm.plan_cnt[s] = 0;
      sm.cnext[s] = 0u;
      sm.slow[s] = 0;
      sm.vtile[s] = 0;
    }
    fence_mbar_init();
    if (blockIdx.x == 0) p.stats[S_T_START] = globaltimer();
    // roles go to CTAs in the order they start, so every waiting role is
    // held by a running CTA
    sm.role = (int)atomicAdd(&p.ctr[C_ROLE], 1u);
    // the first two walkers' SMs: the streaming CTAs that share them stop
    // early, so that each walk's serial chain has its SM's pipes to itself
    if (sm.role < min(p.nwalkers, 2)) atomicExch(&p.ctr[C_WALK_SM + sm.role], smid() + 1u);
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
    if (warp < kWarps) compute_loop(p, sm, dyn);
    else control_loop(p, sm, dyn, &tmap, ntiles);
  }

  // ---- statistics and the last CTA's reset of the shared counters
  if ((tid & 31) == 0) beat(p, sm.role, HB_END, 0);
  __syncthreads();
  if (tid < S_ACCUM_END && sm.st[tid]) atomicAdd(&p.stats[tid], (unsigned long long)sm.st[tid]);
#ifdef SEQSUM_PROFILE
  if (tid < 40 && sm.prof[tid]) atomicAdd(&p.dbg[15300 + tid], (unsigned long long)sm.prof[tid]);
#endif
  if (tid == 0) {
    __threadfence();
    if (atomicAdd(&p.ctr[C_EXIT], 1u) + 1 == gridDim.x) {
      // a call that failed may have left group counters short of complete
      if (__ldcg(&p.ctr[C_ERR]) != 0u)
        for (int64_t g = 0; g <= ntiles / kGroupTiles; g++) p.grp_cnt[g] = 0u;
      p.ctr[C_TICKET] = 0;
      p.ctr[C_SUMTICKET] = 0;
      p.ctr[C_ROLE] = 0;
      p.ctr[C_EXIT] = 0;
      p.ctr[C_WALK_SM] = 0;
      p.ctr[C_WALK_SM + 1] = 0;
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

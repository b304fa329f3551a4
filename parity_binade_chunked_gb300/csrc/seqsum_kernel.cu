// The device path of the exact sequential double sum: one persistent kernel
// per call (plus a one-CTA set-up kernel for batched calls).
//
// What it computes is the bits of  s = s0; for (i) s += x[i];  under IEEE-754
// binary64 round-to-nearest-even.  How (Research-1433, "Forming the CPU's
// sequential double sums on a GPU, bit for bit"):
//   * inside a binade [2^e, 2^(e+1)) the loop is an integer sum of the
//     increments r = x / 2^(e-52) rounded to an integer (finding 2), with an
//     even/odd pair where a term ties (finding 3), and for signed terms a
//     bound on every prefix (Research-1424, section 3);
//   * a plan, an approximate prefix of the terms, says which binade each
//     stretch of terms adds in; the plan cannot make the result wrong, only
//     slower (finding 5);
//   * an in-order walk applies the runs to the exact running value, checking
//     each one, and adds the terms of any stretch that leaves its binade one
//     by one (finding 4).
//
// The GB300 design.  CTAs take roles when they start: the first `nwalkers`
// walk, the rest stream.
//   Streaming CTAs (persistent, two per SM) take 4096-term tiles by ticket.
//   A tile arrives by one TMA box into a 3-stage ring; each thread keeps its
//   16-term row in registers and the stage is refilled at once.  Per tile:
//     - plan: each row's terms converted to float and summed; a block scan
//       gives each row's offset in the tile; the tile's sum is published and
//       a decoupled look-back over earlier tiles gives the prefix before it
//       (double-float);
//     - per row: the prefix range [start - negatives, start + positives]
//       widened by an error allowance; if it lies inside one binade the row
//       is a run of that binade, otherwise its terms are handed to the walk;
//     - runs: each term's increment from its exponent and 53-bit significand
//       by two 32x32->64 multiplies, rounded half up, with a one-word tie
//       detector; rows with a tie are redone in order with the exact
//       even/odd rule;
//     - the tile's header is one run (every row a run of the same binade) or
//       a list of items (composed runs of each warp, raw rows).
//   The walker reads the tile headers in order, 256 at a time, composes
//   consecutive runs of one binade with a block segmented scan, and applies
//   the composites with the exact check; raw rows and refused runs are
//   resolved a warp at a time (the integer rule up to the first term that
//   leaves the binade, that term by a hardware add).
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "binade_math.cuh"
#include "seqsum_internal.cuh"

namespace sq {

constexpr uint32_t kFull = 0xFFFFFFFFu;
constexpr uint64_t kNegZero = 0x8000000000000000ull;
constexpr uint64_t kPay56 = (1ull << 56) - 1;

// ------------------------------------------------------------------ PTX helpers
__device__ __forceinline__ uint32_t smem_u32(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ uint64_t gtimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void mbar_init(uint64_t *b, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(b)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }
__device__ __forceinline__ void mbar_expect_tx(uint64_t *b, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(b)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *b) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(b)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *b, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
      : "=r"(ok)
      : "r"(smem_u32(b)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, uint64_t *bar, int32_t c0, int32_t c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];" ::"r"(
          smem_u32(dst)),
      "l"(map), "r"(smem_u32(bar)), "r"(c0), "r"(c1)
      : "memory");
}
// Words other CTAs of the same launch write or read while it runs: relaxed
// accesses at GPU scope (volatile ones would be system scope, which on a
// CPU-coherent node costs a round trip far longer than the L2's).
__device__ __forceinline__ uint4 ld_vol_v4(const uint4 *p) {
  uint4 v;
  asm volatile("ld.relaxed.gpu.global.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p)
               : "memory");
  return v;
}
__device__ __forceinline__ void st_vol_v4(uint4 *p, uint4 v) {
  asm volatile("st.relaxed.gpu.global.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}
__device__ __forceinline__ void ld_vol_v2(const void *p, uint64_t &a, uint64_t &b) {
  asm volatile("ld.relaxed.gpu.global.v2.u64 {%0, %1}, [%2];" : "=l"(a), "=l"(b) : "l"(p) : "memory");
}
__device__ __forceinline__ void st_vol_v2(void *p, uint64_t a, uint64_t b) {
  asm volatile("st.relaxed.gpu.global.v2.u64 [%0], {%1, %2};" ::"l"(p), "l"(a), "l"(b) : "memory");
}
__device__ __forceinline__ uint32_t ld_relaxed_u32(const uint32_t *p) {
  uint32_t v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t *p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_relaxed_u32(uint32_t *p, uint32_t v) {
  asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void st_release_u32(uint32_t *p, uint32_t v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void fence_acq_rel() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }
__device__ __forceinline__ uint64_t dbits(double v) { return (uint64_t)__double_as_longlong(v); }
__device__ __forceinline__ double bitsd(uint64_t b) { return __longlong_as_double((long long)b); }

// self-checking builds: bounds checks on computed indices, first failure recorded
#ifdef SEQSUM_CHECKS
__device__ __noinline__ bool check_fail(const Params &p, uint32_t site, int64_t val) {
  if (atomicCAS(&p.ctr[C_CHECK_SITE], 0u, site) == 0u) {
    p.ctr[C_CHECK_LO] = (uint32_t)val;
    p.ctr[C_CHECK_HI] = (uint32_t)((uint64_t)val >> 32);
  }
  return false;
}
#define SQ_OK(p, cond, site, val) ((cond) ? true : check_fail((p), (site), (int64_t)(val)))
#else
#define SQ_OK(p, cond, site, val) true
#endif

__device__ __noinline__ void note_timeout(const Params &p, uint32_t err, uint32_t site, uint32_t a, uint32_t b) {
  atomicOr(&p.ctr[C_ERR], err);
  if (atomicCAS(&p.ctr[C_TO_SITE], 0u, site) == 0u) {
    p.ctr[C_TO_A] = a;
    p.ctr[C_TO_B] = b;
  }
}

// profiling builds: a timeline of the units of four streaming CTAs (globaltimer
// stamps of compute warp 0 and of the producer) in the diagnostic words
#ifdef SEQSUM_PROFILE
__device__ __forceinline__ void tl_mark(const Params &p, int role, int who, uint32_t u, int k) {
  const int c = role - p.nwalkers - 1;
  if (c < 0 || c >= 2 || u >= 96) return;
  p.dbg[(c * 2 + who) * 512 + u * 5 + k] = gtimer();
}
#define TL(p, role, who, u, k) tl_mark((p), (role), (who), (u), (k))
// the walk's phases: SM cycles per phase, summed over batches (thread 0)
#define WPH(k)                                              \
  do {                                                      \
    if (threadIdx.x == 0) {                                 \
      const uint64_t now_ = clock64();                      \
      atomicAdd(&p.dbg[2048 + (k)], now_ - wph_last);       \
      wph_last = now_;                                      \
    }                                                       \
  } while (0)
#define WPH_INIT uint64_t wph_last = clock64()
// the walk's ranges: globaltimer stamps (headers in, slot handed over, slot taken, range applied)
#define WRT(r, k)                                                       \
  do {                                                                  \
    if ((threadIdx.x & 31) == 0 && (r) < 64) p.dbg[2100 + 4 * (r) + (k)] = gtimer(); \
  } while (0)
// the scanner's phases, summed over windows (cycles, thread 0)
#define SCP(k)                                                        \
  do {                                                                \
    const uint64_t n_ = clock64();                                    \
    scp_acc[k] += n_ - scp_last;                                      \
    scp_last = n_;                                                    \
  } while (0)
// the scanner's windows: globaltimer at the poll that found them, their first tile and size, when published
#define SCW(k, v)                                                              \
  do {                                                                         \
    if (threadIdx.x == 0 && nwin < 64) p.dbg[2400 + 4 * nwin + (k)] = (v);     \
  } while (0)
// range 0's producer phases (stamps)
#ifndef SEQSUM_WR0_RANGE
#define SEQSUM_WR0_RANGE 4
#endif
#define WR0(r, k)                                                            \
  do {                                                                       \
    if ((threadIdx.x & 31) == 0 && (r) == SEQSUM_WR0_RANGE && (k) < 40) p.dbg[2360 + (k)] = gtimer(); \
  } while (0)
#else
#define WRT(r, k) ((void)0)
#define WR0(r, k) ((void)0)
#define SCW(k, v) ((void)0)
#define SCP(k) ((void)0)
#define TL(p, role, who, u, k) ((void)0)
#define WPH(k) ((void)0)
#define WPH_INIT ((void)0)
#endif

// ------------------------------------------------------------------ double-float (two floats)
struct DF {
  float hi, lo;
};
__device__ __forceinline__ DF df_add(DF a, DF b) {
  const float s = __fadd_rn(a.hi, b.hi);
  const float v = __fsub_rn(s, a.hi);
  float e = __fadd_rn(__fsub_rn(a.hi, __fsub_rn(s, v)), __fsub_rn(b.hi, v));
  e = __fadd_rn(e, __fadd_rn(a.lo, b.lo));
  const float h = __fadd_rn(s, e);
  return DF{h, __fsub_rn(e, __fsub_rn(h, s))};
}
__device__ __forceinline__ DF df_of_double(double v) {
  const float h = __double2float_rn(v);
  const float l = __double2float_rn(__dsub_rn(v, (double)h));
  return DF{h, l};
}

// ------------------------------------------------------------------ records
__device__ __forceinline__ uint64_t pack56(int64_t v, uint32_t tag) {
  const int64_t m = ((int64_t)1 << 55) - 1;
  v = v > m ? m : (v < -m ? -m : v);
  return ((uint64_t)v & kPay56) | ((uint64_t)tag << 56);
}
__device__ __forceinline__ int64_t unpack56(uint64_t w) { return (int64_t)(w << 8) >> 8; }

struct Item {
  Run r;
  uint32_t kind, eb, count, start;
};
constexpr uint32_t kNoKey = 0xFFFFFFFFu;   // the binade key of a record that is not a run (it never merges)

__device__ __forceinline__ uint64_t pack_meta(uint32_t kind, uint32_t eb, int32_t d, uint32_t flags, uint32_t count,
                                              uint32_t start) {
  return (uint64_t)(kind & 7u) | ((uint64_t)(eb & 0x7FFu) << 3) | ((uint64_t)((d + 1) & 3) << 14) |
         ((uint64_t)(flags & 0xFFu) << 16) | ((uint64_t)(count & 0x1FFFu) << 24) | ((uint64_t)(start & 0x1FFFu) << 37);
}
__device__ __forceinline__ Rec pack_item(const Item &it, uint32_t tag) {
  Rec q;
  q.w[0] = pack56(it.r.inc, tag);
  q.w[1] = pack56(it.r.lo, tag);
  q.w[2] = pack56(it.r.hi, tag);
  q.w[3] = pack_meta(it.kind, it.eb, it.r.d, it.r.flags, it.count, it.start) | ((uint64_t)tag << 56);
  return q;
}
__device__ __forceinline__ Item unpack_item(const Rec &q) {
  Item it;
  it.r.inc = unpack56(q.w[0]);
  it.r.lo = unpack56(q.w[1]);
  it.r.hi = unpack56(q.w[2]);
  const uint64_t m = q.w[3];
  it.kind = (uint32_t)(m & 7u);
  it.eb = (uint32_t)((m >> 3) & 0x7FFu);
  it.r.d = (int32_t)((m >> 14) & 3u) - 1;
  it.r.flags = (uint32_t)((m >> 16) & 0xFFu);
  it.count = (uint32_t)((m >> 24) & 0x1FFFu);
  it.start = (uint32_t)((m >> 37) & 0x1FFFu);
  return it;
}
__device__ __forceinline__ bool tags_ok(const Rec &q, uint32_t tag) {
  return (q.w[0] >> 56) == tag && (q.w[1] >> 56) == tag && (q.w[2] >> 56) == tag && (q.w[3] >> 56) == tag;
}
__device__ __forceinline__ Rec ld_rec_vol(const Rec *p) {
  Rec q;
  ld_vol_v2(&p->w[0], q.w[0], q.w[1]);
  ld_vol_v2(&p->w[2], q.w[2], q.w[3]);
  return q;
}
__device__ __forceinline__ void st_rec_vol(Rec *p, const Rec &q) {
  st_vol_v2(&p->w[0], q.w[0], q.w[1]);
  st_vol_v2(&p->w[2], q.w[2], q.w[3]);
}
__device__ __forceinline__ void st_rec(Rec *p, const Rec &q) {
  uint4 *d = reinterpret_cast<uint4 *>(p);
  d[0] = make_uint4((uint32_t)q.w[0], (uint32_t)(q.w[0] >> 32), (uint32_t)q.w[1], (uint32_t)(q.w[1] >> 32));
  d[1] = make_uint4((uint32_t)q.w[2], (uint32_t)(q.w[2] >> 32), (uint32_t)q.w[3], (uint32_t)(q.w[3] >> 32));
}

__device__ __forceinline__ Run shfl_run_up(const Run &r, int off) {
  Run o;
  o.inc = (int64_t)__shfl_up_sync(kFull, (long long)r.inc, off);
  o.lo = (int64_t)__shfl_up_sync(kFull, (long long)r.lo, off);
  o.hi = (int64_t)__shfl_up_sync(kFull, (long long)r.hi, off);
  o.d = __shfl_up_sync(kFull, r.d, off);
  o.flags = __shfl_up_sync(kFull, r.flags, off);
  return o;
}
__device__ __forceinline__ Run shfl_run_idx(const Run &r, int src) {
  Run o;
  o.inc = (int64_t)__shfl_sync(kFull, (long long)r.inc, src);
  o.lo = (int64_t)__shfl_sync(kFull, (long long)r.lo, src);
  o.hi = (int64_t)__shfl_sync(kFull, (long long)r.hi, src);
  o.d = __shfl_sync(kFull, r.d, src);
  o.flags = __shfl_sync(kFull, r.flags, src);
  return o;
}

// ------------------------------------------------------------------ shared memory
// One stage of a streaming CTA: the copy of a unit's tile, and what the
// producer warp wrote about the unit (read by the compute warps before they
// release the stage).
struct __align__(16) StageSm {
  uint4 prec[kPrecWords];       // run units: the tile's prefix and warp sums, copied beside the tile
  int64_t tile;                 // -1: none (the compute warps stop)
  int64_t geo[5];               // row0, g_lo, g_hi, t_first, sum
  uint32_t tma;                 // the tile comes by TMA
  int kind;                     // U_RUN, U_PLAN, U_SPEC or U_REDO
};

// The combining state of a unit while its warps finish it (a ring of 4: a
// warp can be at most three units ahead of the slowest).  The last warp to
// finish is found with a shared atomic counter.
constexpr int kUnitSlots = 4;
struct UnitSm {
  int done_cnt;                     // warps done with the unit
  float wfs[kWarps], wfa[kWarps];   // plan units: the warps' sums
  long long wred[kWarps][3];        // run units: the warps' runs when each is one run: inc, lo, hi
  int32_t wd[kWarps];               // ... and its odd-start adjustment (non-zero only with a tie)
  uint32_t wflags[kWarps];
  int32_t wkey[kWarps];             // the warp's binade key (one run), or -1 (items)
  uint32_t wcnt[kWarps];            // the warp's items (when it is not one run)
};

struct Smem {
  uint64_t full[kStages];            // a stage's copy landed (and the producer's words about it)
  uint64_t empty[kStages];           // the compute warps have read the stage (8 arrivals)
  StageSm st[kStages];
  UnitSm us[kUnitSlots];
  int role;
  int alone;                         // a streaming CTA on the walker's or the scanner's SM
  uint32_t tag;
  int64_t ntiles;
  int fail;
  int broken;                        // this streaming CTA stopped using TMA after a timeout
  int count;
  int wk;
  uint64_t S;                        // the walk's running value (bits)
  uint32_t prof_i;                   // profiling builds: how a raw row with tables ended
  uint32_t prof_n;                   // profiling builds: walk steps logged
  uint64_t t_stream_end;
  uint64_t t_units_end;              // a streaming CTA: when its latest unit's header was published
  // the scanner's warps: each one's first unpublished tile of the round
  // (two buffers, by iteration), their totals, and the give-up flag
  int scan_first[2][kWarps];
  float4 scan_tot[kWarps];
  int scan_stop;
  // the walk's slots: handed over by mbarriers, their uses counted on each side
  uint64_t wfull[kWarps];
  uint64_t wempty[kWarps];
  uint32_t wuse_p[kWarps];
  uint32_t wuse_c[kWarps];
  unsigned long long stat[kBlockWarps][S_ACCUM_END];   // per warp (written by one lane of it)
};

// Counters: each warp adds to its own row (one lane of the warp at a time);
// the rows are summed when the CTA ends.
__device__ __forceinline__ void stat_add(Smem &sm, int which, unsigned long long v) {
  sm.stat[threadIdx.x >> 5][which] += v;
}

// ------------------------------------------------------------------ tile geometry
// Tiles of a sum cover whole rows of 16 terms of x, starting at the row that
// holds the sum's first term; terms of a row outside the sum are masked to
// -0, the identity of binary64 addition.
struct Geo {
  int64_t row0, g_lo, g_hi, t_first;
  int32_t sum;
};

// hint: a sum at or before the tile's (a caller that walks tiles upwards
// keeps it; most calls then read one or two starts instead of searching).
__device__ __forceinline__ Geo tile_geo(const Params &p, int64_t t, int *hint = nullptr) {
  Geo g;
  if (!p.offsets) {
    g.row0 = t * kTileRows;
    g.g_lo = 0;
    g.g_hi = p.n;
    g.t_first = 0;
    g.sum = 0;
    return g;
  }
  // the position lo with tile_begin[lo] <= t < tile_begin[lo+1] (the last such: empty sums share
  // a start); the sum there is order[lo]
  int lo = 0, hi = p.nsums;   // invariant: tile_begin[lo] <= t < tile_begin[hi]
  if (hint && *hint >= 0 && *hint < p.nsums && __ldg(&p.tile_begin[*hint]) <= t) {
    lo = *hint;
    int k = 0;
    while (k < 4 && lo + 1 < hi && __ldg(&p.tile_begin[lo + 1]) <= t) {
      lo++;
      k++;
    }
    if (k < 4) hi = lo + 1;   // found by walking up; else search above
  }
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(&p.tile_begin[mid]) <= t) lo = mid;
    else hi = mid;
  }
  if (hint) *hint = lo;
  const int k = __ldg(&p.order[lo]);
  const int64_t off = __ldg(&p.offsets[k]);
  g.t_first = __ldg(&p.tile_begin[lo]);
  g.row0 = (off >> 4) + (t - g.t_first) * kTileRows;
  g.g_lo = off;
  g.g_hi = __ldg(&p.offsets[k + 1]);
  g.sum = k;
  return g;
}

// ------------------------------------------------------------------ forced plans (tests)
__device__ __forceinline__ uint32_t hash3(uint64_t a, uint32_t b) {
  uint64_t z = a * 0x9E3779B97F4A7C15ull + b * 0xBF58476D1CE4E5B9ull;
  z ^= z >> 29;
  z *= 0x94D049BB133111EBull;
  return (uint32_t)(z >> 32);
}

// ------------------------------------------------------------------ per-row run of the exact rule (ties)
// The row's terms in order, each increment by the even/odd rule of
// binade_math.cuh.  Only rows with a tie come here.
__device__ __noinline__ Run row_run_exact(const uint64_t *v, int e) {
  Run r = run_empty();
  for (int j = 0; j < kLaneTerms; j++) {
    int64_t re;
    int32_t d;
    const bool poison = term_inc(v[j], e, re, d);
    run_push(r, re, d, term_flags(v[j]) | (poison ? (uint32_t)F_POISON : 0u));
  }
  return r;
}

__device__ __forceinline__ void saturate(Run &r) {
  const int64_t lim = (int64_t)1 << 54;
  if (r.inc > lim || r.inc < -lim || r.hi > lim || r.lo < -lim) {
    r.flags |= F_POISON;
    r.inc = r.inc > lim ? lim : (r.inc < -lim ? -lim : r.inc);
    r.hi = r.hi > lim ? lim : r.hi;
    r.lo = r.lo < -lim ? -lim : r.lo;
  }
}

// ------------------------------------------------------------------ units of the streaming CTAs
// Ticket k names a unit: the plan of a tile (its float sums published), or
// the runs of a tile, W tiles behind the plans, once the scanner has turned
// the sums into the tile's prefix.  Every unit depends only on units with
// smaller tickets, so the smallest unfinished unit can always proceed.  (A
// planned call takes its tickets otherwise: see producer_warp.)
__device__ __forceinline__ int64_t unit_of(int64_t k, int64_t P, int64_t W, bool &plan) {
  plan = false;
  if (k < 0) return -1;
  if (W >= P) {
    plan = k < P;
    return plan ? k : (k < 2 * P ? k - P : -1);
  }
  if (k < W) {
    plan = true;
    return k;
  }
  const int64_t j = k - W;
  if (j < 2 * (P - W)) {
    plan = (j & 1) == 0;
    return plan ? W + (j >> 1) : (j >> 1);
  }
  const int64_t r = (P - W) + (j - 2 * (P - W));
  return r < P ? r : -1;
}

__device__ __forceinline__ int float_binade(float f) { return (int)((__float_as_uint(f) >> 23) & 0xFFu); }
__device__ __forceinline__ int vload(const int *p) { return *reinterpret_cast<const volatile int *>(p); }

__device__ __forceinline__ Geo stage_geo(const StageSm &st) {
  Geo g;
  g.row0 = st.geo[0];
  g.g_lo = st.geo[1];
  g.g_hi = st.geo[2];
  g.t_first = st.geo[3];
  g.sum = (int32_t)st.geo[4];
  return g;
}

// 16 bytes global -> shared, asynchronously (this thread waits for its own copies with cp_async_wait)
__device__ __forceinline__ void cp_async16(void *dst, const void *src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_all;" ::: "memory"); }

__device__ __forceinline__ void bulk_load(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_u32(dst)),
               "l"(src), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}

// Stage s takes unit k (one thread): its tile's copy, and for a run unit the
// tile's plan record (prefix and warp sums) beside it.  The stage's per-unit
// state is cleared first; the mbarrier completion publishes it to the warps.
__device__ __forceinline__ void stage_fill(const Params &p, Smem &sm, unsigned char *stages, const CUtensorMap *tmap,
                                           int s, int64_t t, int kind, int (&hint)[2]) {
  StageSm &st = sm.st[s];
  const bool plan = kind == U_PLAN;
  if (t < 0) {
    st.tile = -1;
    st.tma = 0;
    mbar_arrive(&sm.full[s]);
    return;
  }
  const Geo g = tile_geo(p, t, &hint[plan ? 0 : 1]);
  st.tile = t;
  st.kind = kind;
  st.geo[0] = g.row0;
  st.geo[1] = g.g_lo;
  st.geo[2] = g.g_hi;
  st.geo[3] = g.t_first;
  st.geo[4] = g.sum;
  const bool tma = p.tma_rows > 0 && g.row0 < p.tma_rows;
  st.tma = tma ? 1u : 0u;
  const uint32_t side = plan ? 0u : (uint32_t)(kPrecWords * sizeof(uint4));
  if (tma || side) {
    mbar_expect_tx(&sm.full[s], (tma ? (uint32_t)kStageBytes : 0u) + side);
    if (tma) tma_load_2d(stages + s * kStageBytes, tmap, &sm.full[s], 0, (int32_t)g.row0);
    if (side) bulk_load(st.prec, (kind == U_REDO ? p.prec_next : p.prec) + t * kPrecWords, side, &sm.full[s]);
  } else {
    mbar_arrive(&sm.full[s]);
  }
}

// A warp waits (bounded) for use `ph` of stage s.  Returns whether the copy
// landed; a copy that did not is recorded, and the warp reads its rows from x.
__device__ __forceinline__ bool stage_wait(const Params &p, Smem &sm, int s, uint32_t ph) {
  const int lane = threadIdx.x & 31;
  int ok = 1;
  if (lane == 0) {
    const uint64_t c0 = clock64();
    uint64_t t0 = 0;
    uint32_t spin = 0;
    while (!mbar_try_wait(&sm.full[s], ph)) {
      if ((++spin & 255u) == 0u) {
        const uint64_t now = gtimer();
        if (!t0) t0 = now;
        else if (now - t0 > p.wait_ns) {
          ok = 0;
          break;
        }
      }
    }
    if (!ok) {
      // the copy may still land: wait once more (bounded) so that it cannot
      // write into the stage after it is reused
      note_timeout(p, ERR_TMA_TIMEOUT, 2, (uint32_t)s, ph);
      sm.broken = 1;
      const uint64_t t1 = gtimer();
      while (!mbar_try_wait(&sm.full[s], ph) && gtimer() - t1 < p.wait_ns) {
      }
    }
    stat_add(sm, S_CY_TMA_WAIT, clock64() - c0);
  }
  ok = __shfl_sync(kFull, ok, 0);
  if (ok) {
    // every lane's own wait on the completed phase makes the copy's writes visible to it
    for (uint32_t k = 0; k < (1u << 20) && !mbar_try_wait(&sm.full[s], ph); k++) {
    }
  }
  return ok != 0;
}

__device__ __forceinline__ void load_row(const Params &p, const unsigned char *stage, bool lane_tma, int64_t row,
                                         const Geo &g, uint64_t (&v)[kLaneTerms]) {
  const int rw = threadIdx.x;   // the row within the tile
  const bool full = g.row0 * kLaneTerms >= g.g_lo && (g.row0 + kTileRows) * kLaneTerms <= g.g_hi;
  if (lane_tma) {
    const unsigned char *rp = stage + rw * 128;
    const int sw = rw & 7;
#pragma unroll
    for (int q = 0; q < 8; q++) {
      const uint4 d = *reinterpret_cast<const uint4 *>(rp + ((q ^ sw) << 4));
      v[2 * q] = ((uint64_t)d.y << 32) | d.x;
      v[2 * q + 1] = ((uint64_t)d.w << 32) | d.z;
    }
    if (!full) {
      const int64_t g0 = row * kLaneTerms;
#pragma unroll
      for (int j = 0; j < kLaneTerms; j++) {
        const int64_t gi = g0 + j;
        if (gi < g.g_lo || gi >= g.g_hi) v[j] = kNegZero;
      }
    }
  } else {
    const int64_t g0 = row * kLaneTerms;
    const unsigned long long *xp = reinterpret_cast<const unsigned long long *>(p.x);
#pragma unroll
    for (int j = 0; j < kLaneTerms; j++) {
      const int64_t gi = g0 + j;
      v[j] = (gi >= g.g_lo && gi < g.g_hi) ? (uint64_t)__ldg(xp + gi) : kNegZero;
    }
  }
}

// A term as a float for the plan, from its bits with integer operations
// only (this GPU's fp64 pipe, which a conversion instruction would use, is a
// small fraction of its integer and fp32 rate): the significand truncated to
// 24 bits; magnitudes below 2^-126 become 0, those of 2^128 and above (and
// inf, NaN) inf.  The plan only steers the walk: an inexact plan cannot make
// a result wrong.
__device__ __forceinline__ float plan_f32(uint64_t b) {
  const uint32_t hi = (uint32_t)(b >> 32), lo = (uint32_t)b;
  const uint32_t E = (hi >> 20) & 0x7FFu;
  uint32_t f = (__funnelshift_l(lo, hi, 3) & 0x7FFFFFu) | ((E - 896u) << 23);
  f = E <= 896u ? 0u : (E >= 1151u ? 0x7F800000u : f);
  return __uint_as_float(f | (hi & 0x80000000u));
}

// The row's plan sums: its terms as floats summed, their magnitudes summed,
// and the largest high word (sign included).
__device__ __forceinline__ void row_sums(const uint64_t (&v)[kLaneTerms], float &fs, float &fa, uint32_t &mx) {
  fs = 0.0f;
  fa = 0.0f;
  mx = 0;
#pragma unroll
  for (int j = 0; j < kLaneTerms; j++) {
    mx = max(mx, (uint32_t)(v[j] >> 32));
    const float f = plan_f32(v[j]);
    fs = __fadd_rn(fs, f);
    fa = __fadd_rn(fa, fabsf(f));
  }
}

// A sum's start value as a double-float (the start of its first tile's prefix).
__device__ __noinline__ DF start_df(const Params &p, int32_t sum) { return df_of_double(p.offsets ? p.s0s[sum] : p.s0); }

// The last warp of a tile's plan: the warps' sums beside the tile's prefix
// (in `rec`), and the tile's sums for the scanner; a sum's first tile also
// publishes its prefix, the sum's start value.  key: the binade of a tile of
// one run formed on a stored plan (0: none).
__device__ __noinline__ void publish_plan(const Params &p, UnitSm &us, int64_t t, const Geo &g, uint32_t tag,
                                          uint4 *rec, uint32_t key) {
  const int lane = threadIdx.x & 31;
  if (lane < 2 * kWarps / 4) {
    // the warps' sums (4 floats a lane) beside the tile's prefix
    const float *src = lane < kWarps / 4 ? &us.wfs[4 * lane] : &us.wfa[4 * (lane - kWarps / 4)];
    st_vol_v4(&rec[t * kPrecWords + 1 + lane], make_uint4(__float_as_uint(src[0]), __float_as_uint(src[1]),
                                                         __float_as_uint(src[2]), __float_as_uint(src[3])));
  }
  if (lane == 0) {
    DF agg = DF{0.0f, 0.0f};
    float agg_abs = 0.0f;
    for (int k = 0; k < kWarps; k++) {
      agg = df_add(agg, DF{us.wfs[k], 0.0f});
      agg_abs = __fadd_rn(agg_abs, us.wfa[k]);
    }
    uint32_t head = 0;
    if (t == g.t_first) {
      // a sum's first tile: its prefix is the sum's start value (published
      // here), and the sum it gives the scanner starts from it (flag 4)
      const DF s0 = start_df(p, g.sum);
      st_vol_v4(&rec[t * kPrecWords], make_uint4(__float_as_uint(s0.hi), __float_as_uint(s0.lo),
                                                 __float_as_uint(fabsf(s0.hi)), (tag << 8) | 2u));
      agg = df_add(s0, agg);
      agg_abs = __fadd_rn(fabsf(s0.hi), agg_abs);
      head = 4u;
    }
    st_vol_v4(&p.status[t], make_uint4(__float_as_uint(agg.hi), __float_as_uint(agg.lo), __float_as_uint(agg_abs),
                                       (key << 16) | (tag << 8) | 1u | head));
  }
}

// A plan unit, one warp's 32 rows (already loaded): the warp's float sums;
// the last warp publishes the warps' sums beside the tile's prefix, and the
// tile's sums for the scanner.  (No fence orders the two: they only steer
// the plan, which cannot make a result wrong.)
__device__ __forceinline__ void plan_unit(const Params &p, Smem &sm, UnitSm &us, int64_t t, const Geo &g,
                                          const uint64_t (&v)[kLaneTerms], uint32_t tag) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  float fs, fa;
  uint32_t mx;
  row_sums(v, fs, fa, mx);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    fs = __fadd_rn(fs, __shfl_xor_sync(kFull, fs, o));
    fa = __fadd_rn(fa, __shfl_xor_sync(kFull, fa, o));
  }
  int last = 0;
  if (lane == 0) {
    us.wfs[w] = fs;
    us.wfa[w] = fa;
    __threadfence_block();
    last = atomicAdd(&us.done_cnt, 1) == kWarps - 1;
  }
  last = __shfl_sync(kFull, last, 0);
  if (!last) return;
  __threadfence_block();
  publish_plan(p, us, t, g, tag, p.prec, 0u);
}


// The last warp of a complex tile's run unit (out of line: rare, and kept
// out of the units' loop): a warp that is one run gets it written as the one
// item of its region; the header carries every warp's count of items (6 bits
// each), and the walk reads warp k's items from slot 32 k.  The warps' own
// items were fenced at CTA scope before the count that named this warp the
// last; one GPU-scope fence here orders all of them before the header.
__device__ __noinline__ void complex_publish(const Params &p, Smem &sm, UnitSm &us, int64_t t, uint32_t tag) {
  const int lane = threadIdx.x & 31;
  Rec *area = p.items + t * kItemSlots;
  uint32_t cnt = 0;
  if (lane < kWarps) {
    if (us.wkey[lane] >= 0) {
      Item it;
      it.r.inc = us.wred[lane][0];
      it.r.lo = us.wred[lane][1];
      it.r.hi = us.wred[lane][2];
      it.r.d = us.wd[lane];
      it.r.flags = us.wflags[lane];
      saturate(it.r);
      it.kind = K_RUN;
      it.eb = (uint32_t)us.wkey[lane];
      it.count = 32 * kLaneTerms;
      it.start = (uint32_t)lane * 32 * kLaneTerms;
      st_rec(&area[lane * kWarpSlots], pack_item(it, 0));
      cnt = 1;
    } else {
      cnt = min(us.wcnt[lane], (uint32_t)kWarpSlots);
    }
  }
  uint64_t packed = 0;
#pragma unroll
  for (int k = 0; k < kWarps; k++) packed |= (uint64_t)__shfl_sync(kFull, cnt, k) << (6 * k);
  __syncwarp();
  if (lane == 0) {
    __threadfence();   // every warp's items before the header that publishes them
    Rec q;
    q.w[0] = packed | ((uint64_t)tag << 56);
    q.w[1] = (uint64_t)tag << 56;
    q.w[2] = (uint64_t)tag << 56;
    q.w[3] = pack_meta(K_COMPLEX, 0, 0, 0, 0, 0) | ((uint64_t)tag << 56);
    stat_add(sm, S_TILE_COMPLEX, 1);
    if (!(p.fault_mode == 1 && t == p.fault_arg)) st_rec_vol(&p.hdr[t], q);
  }
}

// A run unit, one warp's 32 rows (already loaded): each row's binade from
// its prefix range, the rows' runs and the warp's record; the last warp
// publishes the tile's header.  pf is the tile's prefix as the copy brought
// it, bs/ba the sums of the warps before this one.
__device__ __forceinline__ void run_unit(const Params &p, Smem &sm, UnitSm &us, int64_t t, const Geo &g,
                                         const uint64_t (&v)[kLaneTerms], uint4 pf, float bs, float ba, float wfs,
                                         float wfa, uint32_t tag, int kind) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, tid = threadIdx.x;
  if (kind == U_SPEC) {
    // a planned call: the stored plan of the call before (any tag); a sum's
    // first tile starts from this call's start value; a tile without a stored
    // plan is planned from 0 (the scanner then sends it back)
    if (t == g.t_first) {
      const DF s0 = start_df(p, g.sum);
      pf = make_uint4(__float_as_uint(s0.hi), __float_as_uint(s0.lo), __float_as_uint(fabsf(s0.hi)), 2u);
    } else if ((pf.w & 3u) != 2u) {
      pf = make_uint4(0, 0, 0, 2u);
    }
  } else if (!((pf.w >> 8) == tag && (pf.w & 3u) == 2u)) {
    // the scanner had not published the prefix when the copy ran: poll it
    const uint64_t c0 = clock64();
    const uint4 *pr = kind == U_REDO ? p.prec_next : p.prec;
    int ok = 0;
    if (lane == 0) {
      uint64_t t0 = 0;
      for (uint32_t spin = 0;; spin++) {
        pf = ld_vol_v4(&pr[t * kPrecWords]);
        if ((pf.w >> 8) == tag && (pf.w & 3u) == 2u) {
          ok = 1;
          break;
        }
        if ((spin & 15u) == 15u) {
          const uint64_t now = gtimer();
          if (!t0) t0 = now;
          else if (now - t0 > p.wait_ns) break;
        }
        __nanosleep(64);
      }
      if (!ok) note_timeout(p, ERR_PLAN_TIMEOUT, 5, (uint32_t)t, 0);
      stat_add(sm, S_PFX_LATE, 1);
      stat_add(sm, S_CY_PFX_WAIT, clock64() - c0);
    }
    ok = __shfl_sync(kFull, ok, 0);
    pf.x = __shfl_sync(kFull, pf.x, 0);
    pf.y = __shfl_sync(kFull, pf.y, 0);
    pf.z = __shfl_sync(kFull, pf.z, 0);
    if (!ok) pf = make_uint4(0, 0, 0, 0);   // the plan only: a prefix taken as 0
    // (the warps' sums came with the copy: a stale copy can make the plan
    // worse, never the result)
  }
  const uint64_t c0 = clock64();
  const DF ex = DF{__uint_as_float(pf.x), __uint_as_float(pf.y)};
  const float ex_abs = __uint_as_float(pf.z);
  // the warp's range -- its prefix and its own plan sums, with the allowance
  // -- inside one binade: every row's range is inside it too, and the rows'
  // own sums are not needed
  int fbw = 0;
  if (p.plan_mode == 0) {
    const float P0 = __fadd_rn(ex.hi, __fadd_rn(ex.lo, bs));
    const float Aw = __fadd_rn(__fadd_rn(ex_abs, ba), wfa);
    const float mw = __fadd_rn(__fmul_rn(Aw, 4.76837158203125e-7f /* 2^-21 */), 1e-30f);
    const float posw = __fmul_rn(0.5f, __fadd_rn(wfa, wfs)), negw = __fmul_rn(0.5f, __fsub_rn(wfa, wfs));
    const float low = __fsub_rn(__fsub_rn(P0, negw), mw), hiw = __fadd_rn(__fadd_rn(P0, posw), mw);
    if (low > 0.0f) {
      const int a = float_binade(low), b = float_binade(hiw);
      if (a == b && a >= 1 && a <= 254) fbw = a;
    } else if (hiw < 0.0f) {
      const int a = float_binade(-hiw), b = float_binade(-low);
      if (a == b && a >= 1 && a <= 254) fbw = a;
    }
  }
  float fs = 0.0f, fa = 0.0f, lo_ = 0.0f, hi_ = 0.0f;
  uint32_t mx = 0, eb = 0;
  bool zero = false, allneg = false;
  if (fbw) {
    // (a row of zeros is then a run of zero increments: S is not zero there)
#pragma unroll
    for (int j = 0; j < kLaneTerms; j++) mx = max(mx, (uint32_t)(v[j] >> 32));
    eb = (uint32_t)(fbw - 127 + 1023);
  } else {
  row_sums(v, fs, fa, mx);
  float is = fs, ia = fa;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float a = __shfl_up_sync(kFull, is, o), b = __shfl_up_sync(kFull, ia, o);
    if (lane >= o) {
      is = __fadd_rn(is, a);
      ia = __fadd_rn(ia, b);
    }
  }
  float xs = __shfl_up_sync(kFull, is, 1), xa = __shfl_up_sync(kFull, ia, 1);
  if (lane == 0) xs = xa = 0.0f;
  xs = __fadd_rn(bs, xs);
  xa = __fadd_rn(ba, xa);

  // ---- the row's binade: its prefix range inside one binade, with an allowance
  const float Pf = __fadd_rn(ex.hi, __fadd_rn(ex.lo, xs));
  const float A = __fadd_rn(__fadd_rn(ex_abs, xa), fa);
  const float marg = __fadd_rn(__fmul_rn(A, 4.76837158203125e-7f /* 2^-21 */), 1e-30f);
  const float pos = __fmul_rn(0.5f, __fadd_rn(fa, fs)), neg = __fmul_rn(0.5f, __fsub_rn(fa, fs));
  lo_ = __fsub_rn(__fsub_rn(Pf, neg), marg);
  hi_ = __fadd_rn(__fadd_rn(Pf, pos), marg);
  int fb = 0;   // float biased exponent of the binade, 0: the row's range is not inside one binade
  if (lo_ > 0.0f) {
    const int a = float_binade(lo_), b = float_binade(hi_);
    if (a == b && a >= 1 && a <= 254) fb = a;
  } else if (hi_ < 0.0f) {
    const int a = float_binade(-hi_), b = float_binade(-lo_);
    if (a == b && a >= 1 && a <= 254) fb = a;
  }
  eb = fb ? (uint32_t)(fb - 127 + 1023) : 0u;   // double biased exponent
  // forced plans (tests): the walk must still give the loop's bits
  if (p.plan_mode) {
    const uint32_t h = hash3((uint64_t)t, (uint32_t)tid);
    if (p.plan_mode == 1 && eb) eb += 1;
    else if (p.plan_mode == 2) eb = 0;
    else if (p.plan_mode == 3) eb = 1023;
    else if (p.plan_mode == 4) eb = 0;
    else if (p.plan_mode == 5 && eb) eb = eb + (h % 3u) - 1u;
  }
  // exact zero rows: a no-op on any non-zero sum, the sign rule on a zero one
  if (fa == 0.0f) {
    uint64_t o = 0, a = kNegZero;
#pragma unroll
    for (int j = 0; j < kLaneTerms; j++) {
      o |= v[j] << 1;
      a &= v[j];
    }
    zero = (o == 0);
    allneg = (a != 0);
  }
  }
  const bool raw = !zero && (eb == 0 || p.plan_mode == 4);
  const bool runrow = !zero && !raw;

  // ---- the row's run: the fast rule for every row (discarded where unused)
  const int c = 64 - (int)(eb ? eb : 1023u);
  const bool signed_warp = __any_sync(kFull, runrow && mx >= 0x80000000u);
  uint32_t tmin = 0xFFFFFFFFu;
  Run r;
  if (!signed_warp) {
    uint64_t acc = 0;
#pragma unroll
    for (int j = 0; j < kLaneTerms; j++) {
      uint32_t tt;
      acc += term_mag_halfup((uint32_t)(v[j] >> 32), (uint32_t)v[j], c, tt);
      tmin = min(tmin, tt);
    }
    r.inc = (int64_t)acc;
    r.lo = 0;
    r.hi = (int64_t)acc;
    r.d = 0;
    r.flags = F_NONNEG | (((mx >> 20) >= eb) ? (uint32_t)F_POISON : 0u);
  } else {
    uint64_t tot = 0, ng = 0;
    uint32_t emax = 0;
#pragma unroll
    for (int j = 0; j < kLaneTerms; j++) {
      const uint32_t hi = (uint32_t)(v[j] >> 32);
      uint32_t tt;
      const uint64_t rr = term_mag_halfup(hi, (uint32_t)v[j], c, tt);
      tmin = min(tmin, tt);
      emax = max(emax, (hi >> 20) & 0x7FFu);
      const uint64_t sm64 = (uint64_t)(int64_t)((int32_t)hi >> 31);
      tot += rr;
      ng += rr & sm64;
    }
    r.inc = (int64_t)(tot - 2 * ng);
    r.lo = -(int64_t)ng;
    r.hi = (int64_t)(tot - ng);
    r.d = 0;
    r.flags = (mx < 0x80000000u ? (uint32_t)F_NONNEG : 0u) | (emax >= eb ? (uint32_t)F_POISON : 0u);
  }
  bool general = false;
  if (runrow && tmin == 0u) {
    uint64_t tmp[kLaneTerms];
#pragma unroll
    for (int j = 0; j < kLaneTerms; j++) tmp[j] = v[j];
    r = row_run_exact(tmp, (int)eb - 1023);
    general = true;
  }
  if (runrow) saturate(r);
  if (zero) {
    r.inc = r.lo = r.hi = 0;
    r.d = 0;
    r.flags = F_NONNEG | F_NONPOS | F_ZERO | (allneg ? (uint32_t)F_ALLNEGZ : 0u);
  }
  const uint32_t key = raw ? 0xFFFFFFFFu : eb;   // zero rows keep the plan's binade (0 where it has none)
  const uint32_t nraw = __popc(__ballot_sync(kFull, raw));
  const uint32_t ntie = __popc(__ballot_sync(kFull, general));
  if (lane == 0) {
    if (nraw) stat_add(sm, S_LANE_RAW, nraw);
    if (ntie) stat_add(sm, S_LANE_TIE, ntie);
  }

  // ---- the warp's record: one run, or its items in its region of the tile's item area
  const uint32_t key0 = __shfl_sync(kFull, key, 0);
  const bool samekey = __all_sync(kFull, !raw && key == key0);
  if (samekey && ntie != 0) {
    // one binade with a tie: the rows' runs composed in order (the even/odd rule)
    Run seg = r;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const Run q = shfl_run_up(seg, o);
      if (lane >= o) seg = run_compose(q, seg);
    }
    if (lane == 31) {
      us.wred[w][0] = seg.inc;
      us.wred[w][1] = seg.lo;
      us.wred[w][2] = seg.hi;
      us.wd[w] = seg.d;
      us.wflags[w] = seg.flags;
      us.wkey[w] = (int32_t)key0;
      us.wcnt[w] = 1;
    }
  } else if (samekey) {
    long long a = r.inc, b = r.lo, d = r.hi;
    uint32_t fand = r.flags & (F_NONNEG | F_NONPOS | F_ZERO | F_ALLNEGZ), fo = r.flags & F_POISON;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      a += __shfl_xor_sync(kFull, a, o);
      b += __shfl_xor_sync(kFull, b, o);
      d += __shfl_xor_sync(kFull, d, o);
    }
    fand = __reduce_and_sync(kFull, fand);
    fo = __reduce_or_sync(kFull, fo);
    if (lane == 0) {
      us.wred[w][0] = a;
      us.wred[w][1] = b;
      us.wred[w][2] = d;
      us.wflags[w] = fand | fo;
      us.wd[w] = 0;
      us.wkey[w] = (int32_t)key0;
      us.wcnt[w] = 1;
    }
  } else {
    const uint32_t pkey = __shfl_up_sync(kFull, key, 1);
    const bool praw = __shfl_up_sync(kFull, raw, 1);
    const bool head = lane == 0 || raw || praw || key != pkey;
    int sstart = head ? lane : 0;
    Run seg = r;
    bool hf = head;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const Run q = shfl_run_up(seg, o);
      const bool qh = __shfl_up_sync(kFull, hf, o);
      const int qs = __shfl_up_sync(kFull, sstart, o);
      if (lane >= o) {
        if (!hf) seg = run_compose(q, seg);
        hf = hf || qh;
        sstart = max(sstart, qs);
      }
    }
    const bool nhead = __shfl_down_sync(kFull, head, 1);
    const bool tail = (lane == 31) || nhead;
    // a raw row whose plan range crosses one power of two, all of its terms
    // of the range's sign, carries prefix tables for the two binades
    bool raw2 = false, rneg = false;
    uint32_t ea = 0;
    if (raw) {
      uint32_t hmin = 0xFFFFFFFFu;
#pragma unroll
      for (int j = 0; j < kLaneTerms; j++)
        hmin = min(hmin, (v[j] << 1) == 0 ? 0xFFFFFFFFu : (uint32_t)(v[j] >> 32));
      int a = 0, b = 0;
      if (lo_ > 0.0f && mx < 0x80000000u) {
        a = float_binade(lo_);
        b = float_binade(hi_);
      } else if (hi_ < 0.0f && hmin >= 0x80000000u) {
        a = float_binade(-hi_);
        b = float_binade(-lo_);
        rneg = true;
      }
      ea = (uint32_t)(a - 127 + 1023);
      raw2 = a >= 1 && (b == a || b == a + 1) && ea >= 54u && ea + 1u <= 2046u;
    }
    // the warp's region: one descriptor per item, in the order of their terms
    // (a warp has at most one item per row: it always fits)
    const uint32_t mdesc = __ballot_sync(kFull, raw || tail);
    const uint32_t total = __popc(mdesc);
    const uint32_t nraw2 = __popc(__ballot_sync(kFull, raw2));
    if (lane == 0 && nraw2) stat_add(sm, S_LANE_RAW2, nraw2);
    const uint32_t at = __popc(mdesc & ((1u << lane) - 1u));
    if (SQ_OK(p, total <= (uint32_t)kWarpSlots, 1, total)) {
      Rec *area = p.items + t * kItemSlots + w * kWarpSlots;
      if (raw) {
        Item it;
        it.r = run_empty();
        it.kind = raw2 ? K_RAW2 : K_RAW;
        it.eb = raw2 ? ea : 0u;
        it.count = kLaneTerms;
        it.start = (uint32_t)tid * kLaneTerms;
        Rec q = pack_item(it, 0);
        q.w[0] = rneg ? 1u : 0u;
        st_rec(&area[at], q);
      } else if (tail) {
        Item it;
        it.r = seg;
        it.kind = K_RUN;
        it.eb = key;
        it.count = (uint32_t)(lane - sstart + 1) * kLaneTerms;
        it.start = (uint32_t)(w * 32 + sstart) * kLaneTerms;
        st_rec(&area[at], pack_item(it, 0));
      }
      // the items before the count that names the tile's last warp (of this
      // CTA): a CTA-scope fence; that warp's GPU-scope fence orders them
      // before the header the walk reads
      __threadfence_block();
    }
    if (lane == 0) {
      us.wkey[w] = -1;
      us.wcnt[w] = total;
    }
  }
  if (kind == U_SPEC) {
    // the next call's plan: this tile's sums, as a plan unit forms them
    if (fbw) row_sums(v, fs, fa, mx);
    float ws_ = fs, wa_ = fa;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      ws_ = __fadd_rn(ws_, __shfl_xor_sync(kFull, ws_, o));
      wa_ = __fadd_rn(wa_, __shfl_xor_sync(kFull, wa_, o));
    }
    if (lane == 0) {
      us.wfs[w] = ws_;
      us.wfa[w] = wa_;
    }
  }
  __syncwarp();
  int last = 0;
  if (lane == 0) {
    __threadfence_block();
    last = atomicAdd(&us.done_cnt, 1) == kWarps - 1;
  }
  last = __shfl_sync(kFull, last, 0);
  if (!last) return;

  // ---- the last warp: the tile's header, then the stage's next tile
  __threadfence_block();
  const int32_t k0 = us.wkey[0];
  bool one = true;
  for (int k = 0; k < kWarps; k++) one = one && us.wkey[k] >= 0 && us.wkey[k] == k0;
  if (one) {
    if (lane == 0) {
      Item h;
      h.r.inc = h.r.lo = h.r.hi = 0;
      h.r.d = 0;
      uint32_t fand = 0xFFu, fo = 0;
      bool tie = false;
      for (int k = 0; k < kWarps; k++) {
        h.r.inc += us.wred[k][0];
        h.r.lo += us.wred[k][1];
        h.r.hi += us.wred[k][2];
        fand &= us.wflags[k];
        fo |= us.wflags[k];
        tie = tie || us.wd[k] != 0;
      }
      h.r.flags = (fand & (F_NONNEG | F_NONPOS | F_ZERO | F_ALLNEGZ)) | (fo & F_POISON);
      if (tie) {
        // a warp with a tie: the warps' runs composed in order
        h.r = run_empty();
        for (int k = 0; k < kWarps; k++) {
          Run q;
          q.inc = us.wred[k][0];
          q.lo = us.wred[k][1];
          q.hi = us.wred[k][2];
          q.d = us.wd[k];
          q.flags = us.wflags[k];
          h.r = k == 0 ? q : run_compose(h.r, q);
        }
      }
      saturate(h.r);
      h.kind = K_RUN;
      h.eb = (uint32_t)k0;
      h.count = kTileTerms;
      h.start = 0;
      if (!(p.fault_mode == 1 && t == p.fault_arg)) st_rec_vol(&p.hdr[t], pack_item(h, tag));
    }
  } else {
    complex_publish(p, sm, us, t, tag);
  }
  if (kind == U_SPEC) {
    // the tile's sums for the scanner: the binade of a tile of one run goes
    // with them, so that the scanner can tell whether the new prefix keeps
    // it.  (No fence after the header: the walk waits for the header's own
    // tags, and a second unit of the tile waits for them before it writes.)
    publish_plan(p, us, t, g, tag, p.prec_next, one && k0 > 0 ? (uint32_t)k0 : 0u);
  } else if (kind == U_REDO) {
    // the header may now be walked
    __syncwarp();
    if (lane == 0) {
      __threadfence();
      st_release_u32(&p.conf[t], tag);
      stat_add(sm, S_REDO, 1);
    }
  }
  if (lane == 0) {
    stat_add(sm, S_TILES, 1);
    stat_add(sm, S_CY_RUN, clock64() - c0);
    const uint64_t now = gtimer();
    if (now > sm.t_units_end) sm.t_units_end = now;
  }
}

// A compute warp of a streaming CTA: units in the order the producer puts
// them into the stages; the rows (and, for a run unit, the prefix the copy
// brought) are read, the stage released, then the unit's work done.
__device__ __noinline__ void compute_warp(const Params &p, Smem &sm, const unsigned char *stages) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const uint32_t tag = sm.tag;
  for (uint32_t u = 0;; u++) {
    const int s = (int)(u % kStages);
    if (w == 0 && lane == 0) TL(p, sm.role, 0, u, 0);
    const bool landed = stage_wait(p, sm, s, (u / kStages) & 1u);
    const StageSm &st = sm.st[s];
    const int64_t t = st.tile;
    if (w == 0 && lane == 0) TL(p, sm.role, 0, u, 1);
    if (t < 0) break;
    const int kind = st.kind;
    const bool plan = kind == U_PLAN;
    const Geo g = stage_geo(st);
    const int64_t row = g.row0 + threadIdx.x;
    uint64_t v[kLaneTerms];
    load_row(p, stages + s * kStageBytes, landed && st.tma && row < p.tma_rows, row, g, v);
    uint4 pf = make_uint4(0, 0, 0, 0);
    float bs = 0.0f, ba = 0.0f, wfs = 0.0f, wfa = 0.0f;
    if (!plan && landed) {
      pf = st.prec[0];
      const float *ws = reinterpret_cast<const float *>(&st.prec[1]);
      for (int k = 0; k < w; k++) {
        bs = __fadd_rn(bs, ws[k]);
        ba = __fadd_rn(ba, ws[kWarps + k]);
      }
      wfs = ws[w];
      wfa = ws[kWarps + w];
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm.empty[s]);   // this warp is done with the stage
    if (w == 0 && lane == 0) TL(p, sm.role, 0, u, 2);
    UnitSm &us = sm.us[u % kUnitSlots];
    if (plan) {
      const uint64_t c0 = clock64();
      plan_unit(p, sm, us, t, g, v, tag);
      if (lane == 0) stat_add(sm, S_CY_PLAN, clock64() - c0);
    } else {
      run_unit(p, sm, us, t, g, v, pf, bs, ba, wfs, wfa, tag, kind);
    }
    if (w == 0 && lane == 0) TL(p, sm.role, 0, u, 3);
    if (w == 0 && lane == 0) TL(p, sm.role, 0, u, 4 - (plan ? 0 : 0));
  }
}

// A planned call's ticket for place j of the redo list: the tile the scanner
// put there, or -1 once the list is final and shorter (bounded: -1 past the
// limit, and the walk then gives up on that tile's header).
__device__ __noinline__ int64_t redo_wait(const Params &p, int64_t j, uint32_t tag) {
  // (every idle producer polls here while the scanner finishes: plain loads,
  // far apart, so that they do not crowd the memory system)
  const uint64_t t0 = gtimer();
  for (uint32_t spin = 0;; spin++) {
    const uint32_t fin = ld_relaxed_u32(&p.ctr[C_SCAN_FIN]);
    fence_acq_rel();   // the flag read first: then the count is final
    const uint32_t n = ld_relaxed_u32(&p.ctr[C_REDO_RES]);
    if ((int64_t)n > j) {
      // the place is taken: its entry lands with the call's tag
      const uint32_t v = ld_acquire_u32(&p.redo[j]);
      if ((v >> 24) == tag) return (int64_t)(v & 0xFFFFFFu);
    } else if (fin) {
      return -1;
    }
    if ((spin & 3u) == 3u && gtimer() - t0 > p.wait_ns) {
      note_timeout(p, ERR_PLAN_TIMEOUT, 8, (uint32_t)j, 0);
      return -1;
    }
    __nanosleep(1000);
  }
}

// The producer warp of a streaming CTA (lane 0): takes units by ticket and
// starts their copies.  Unit u goes to stage u mod 3 once the compute warps
// have released unit u - depth: depth 3 keeps three units in flight (the
// next ticket taken while the stage is still busy, so the atomic's round
// trip overlaps the work); depth 1, for calls with few units per CTA, takes
// a ticket only when the CTA is ready for it.
__device__ __noinline__ void producer_warp(const Params &p, Smem &sm, unsigned char *stages, const CUtensorMap *tmap,
                                           int64_t ntiles) {
  if ((threadIdx.x & 31) != 0) return;
  const int64_t nstream = (int64_t)gridDim.x - p.nwalkers - 1, units = p.planned ? ntiles : 2 * ntiles;
  const bool deep = units > 2 * nstream;
  const uint32_t depth = deep ? (uint32_t)kStages : 1u;
  int64_t hand = -1;
  int hint[2] = {0, 0};   // the sums of the last plan and run tiles (they only grow)
  for (uint32_t u = 0;; u++) {
    const int s = (int)(u % kStages);
    TL(p, sm.role, 1, u, 0);
    if (u >= depth) {
      // unit u - depth released (bounded; a stuck compute warp ends the CTA's units)
      const uint32_t r = u - depth;
      const uint32_t ph = (r / kStages) & 1u;
      const uint64_t t0 = gtimer();
      uint32_t spin = 0;
      bool ok = true;
      while (!mbar_try_wait(&sm.empty[r % kStages], ph)) {
        if ((++spin & 255u) == 0u && gtimer() - t0 > p.wait_ns) {
          ok = false;
          break;
        }
      }
      if (!ok) {
        note_timeout(p, ERR_TMA_TIMEOUT, 7, u, 0);
        sm.broken = 1;
      }
    }
    TL(p, sm.role, 1, u, 1);
    const int64_t k = hand >= 0 ? hand : (int64_t)atomicAdd(&p.ctr[C_TICKET], 1u);
    int64_t t = -1;
    int kind = U_RUN;
    if (!sm.broken) {
      if (!p.planned) {
        bool plan = false;
        t = unit_of(k, ntiles, p.wave, plan);
        kind = plan ? U_PLAN : U_RUN;
      } else if (k < ntiles) {
        t = k;   // a planned call: every tile on the stored plan, in order
        kind = U_SPEC;
      } else {
        t = redo_wait(p, k - ntiles, sm.tag);   // then the tiles the scanner sends back
        kind = U_REDO;
      }
    }
    const bool valid = t >= 0;
    TL(p, sm.role, 1, u, 2);
    if (valid && kind == U_REDO) {
      // the tile's first header (and items) must have landed before this
      // unit writes its own over them (bounded)
      const uint64_t t0 = gtimer();
      for (uint32_t spin = 0; !tags_ok(ld_rec_vol(&p.hdr[t]), sm.tag); spin++) {
        if ((spin & 15u) == 15u && gtimer() - t0 > p.wait_ns) break;
        __nanosleep(100);
      }
      fence_acq_rel();
    }
    if (valid && (kind == U_RUN || kind == U_REDO)) {
      // a run unit's copy waits for the scanner to publish its tile's prefix
      // (bounded; past the limit the compute warps poll for it themselves)
      const uint4 *pr = kind == U_REDO ? p.prec_next : p.prec;
      const uint32_t want = (sm.tag << 8) | 2u;
      const uint64_t t0 = gtimer();
      for (uint32_t spin = 0; ld_relaxed_u32(&pr[t * kPrecWords].w) != want; spin++) {
        if ((spin & 15u) == 15u && gtimer() - t0 > p.wait_ns) break;
        __nanosleep(100);
      }
      asm volatile("fence.proxy.async.global;" ::: "memory");   // the copy reads what the load saw
    }
    sm.us[u % kUnitSlots].done_cnt = 0;
    stage_fill(p, sm, stages, tmap, s, t, kind, hint);
    TL(p, sm.role, 1, u, 3);
#ifdef SEQSUM_PROFILE
    if (sm.role - p.nwalkers - 1 >= 0 && sm.role - p.nwalkers - 1 < 4 && u < 96)
      p.dbg[((sm.role - p.nwalkers - 1) * 2 + 1) * 512 + u * 5 + 4] = (uint64_t)k;
#endif
    if (!valid) break;
    hand = deep ? (int64_t)atomicAdd(&p.ctr[C_TICKET], 1u) : -1;
  }
}

// A streaming CTA: 8 compute warps and a producer warp, no CTA barriers
// after the start (the last warp to finish a unit publishes it).
__device__ __noinline__ void stream_cta(const Params &p, Smem &sm, unsigned char *stages, const CUtensorMap *tmap,
                                        int64_t ntiles) {
  const int tid = threadIdx.x;
  if (tid == 0) {
    sm.broken = 0;
    sm.t_stream_end = 0;
    sm.t_units_end = 0;
    for (int s = 0; s < kStages; s++) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], kWarps);
    }
    fence_mbar_init();
  }
  __syncthreads();
  if ((tid >> 5) < kWarps) compute_warp(p, sm, stages);
  else producer_warp(p, sm, stages, tmap, ntiles);
  __syncthreads();
  if (tid == 0) {
    sm.t_stream_end = gtimer();   // this CTA's last header is published
    if (sm.t_units_end) atomicMax(&p.stats[S_T_UNITS_END], (unsigned long long)sm.t_units_end);
  }
}

// A planned call: whether the header that tile t's unit formed on the stored
// plan serves as well as one formed on the new prefix (e, ea).  A tile of one
// run in binade `key` (carried with its sums in s) keeps it while the tile's
// whole range of partial sums, with twice the allowance the units take, stays
// in that binade; a tile of zeros always keeps it (plan_range_holds, inline:
// the scanner's next loads stay in flight).  Any other tile keeps it when its
// warps' sums are, word for word, the new ones and its stored prefix is
// within 2^-36 of the magnitudes of the new one (the prefix of magnitudes,
// which only sizes the allowance, within 2^-20): far inside the allowance of
// 2^-21 that its rows' binades were chosen with (plan_words_hold; the
// scanner's sums round a little differently from call to call, as its rounds
// fall).  A wrong answer costs time, never bits: the walk checks every run
// against the exact sum.
__device__ __forceinline__ bool plan_range_holds(DF e, float ea, uint4 s) {
  if (s.z == 0u && (s.x << 1) == 0u && (s.y << 1) == 0u) return true;   // zeros add nothing
  const uint32_t key = (s.w >> 16) & 0x7FFu;
  if (key == 0) return false;
  const float fs = __fadd_rn(__uint_as_float(s.x), __uint_as_float(s.y)), fa = __uint_as_float(s.z);
  const float P = __fadd_rn(e.hi, e.lo);
  const float m = __fadd_rn(__fmul_rn(__fadd_rn(ea, fa), 9.5367431640625e-7f /* 2^-20 */), 1e-30f);
  const float pos = __fmul_rn(0.5f, __fadd_rn(fa, fs)), neg = __fmul_rn(0.5f, __fsub_rn(fa, fs));
  const float lo = __fsub_rn(__fsub_rn(P, neg), m), hi = __fadd_rn(__fadd_rn(P, pos), m);
  const bool up = lo > 0.0f;
  if (!up && !(hi < 0.0f)) return false;
  const int a = float_binade(up ? lo : -hi), b = float_binade(up ? hi : -lo);
  return a == b && a >= 1 && a <= 254 && (uint32_t)(a - 127 + 1023) == key;
}
__device__ __noinline__ bool plan_words_hold(const Params &p, int64_t t, DF e, float ea, uint4 s) {
  // (every word at once: one round trip)
  uint4 o, a[kPrecWords - 1], b[kPrecWords - 1];
  o = ld_vol_v4(&p.prec[t * kPrecWords]);
#pragma unroll
  for (int q = 1; q < kPrecWords; q++) {
    a[q - 1] = ld_vol_v4(&p.prec[t * kPrecWords + q]);
    b[q - 1] = ld_vol_v4(&p.prec_next[t * kPrecWords + q]);
  }
  if ((o.w & 3u) != 2u) return false;
  const float A = __fadd_rn(ea, __uint_as_float(s.z));
  const float d = __fadd_rn(__fsub_rn(e.hi, __uint_as_float(o.x)), __fsub_rn(e.lo, __uint_as_float(o.y)));
  if (!(fabsf(d) <= __fmul_rn(A, 1.4551915228366852e-11f /* 2^-36 */) &&
        fabsf(__fsub_rn(ea, __uint_as_float(o.z))) <= __fmul_rn(A, 9.5367431640625e-7f /* 2^-20 */)))
    return false;
  bool same = true;
#pragma unroll
  for (int q = 0; q < kPrecWords - 1; q++)
    same = same && a[q].x == b[q].x && a[q].y == b[q].y && a[q].z == b[q].z && a[q].w == b[q].w;
  return same;
}

// A planned call, a sum's first tile: its prefix is this call's start value
// (which its unit wrote beside the new plan), its own sums those in s less
// that value.
__device__ __noinline__ bool plan_holds_head(const Params &p, int64_t t, uint4 s) {
  const uint4 h = ld_vol_v4(&p.prec_next[t * kPrecWords]);
  const DF e = DF{__uint_as_float(h.x), __uint_as_float(h.y)};
  const float ea = __uint_as_float(h.z);
  const float fs = __fadd_rn(__fsub_rn(__uint_as_float(s.x), e.hi), __fsub_rn(__uint_as_float(s.y), e.lo));
  const float fa = fmaxf(__fsub_rn(__uint_as_float(s.z), ea), 0.0f);
  const uint4 own = make_uint4(__float_as_uint(fs), 0u, __float_as_uint(fa), s.w);
  return plan_range_holds(e, ea, own) || plan_words_hold(p, t, e, ea, own);
}

// A planned call, in the scanner: tile t's header, formed on the stored plan,
// stands (the walk may take it: its release word gets the call's tag) or the
// tile goes on the redo list (one atomic a warp for the places; each entry
// carries the call's tag, so that a reader knows it landed).
__device__ __forceinline__ void scan_release(const Params &p, int64_t t, bool in, bool head, DF e, float ea, uint4 v,
                                             uint32_t tag) {
  const int lane = threadIdx.x & 31;
  bool redo = false;
  if (in) {
    const bool holds = head ? plan_holds_head(p, t, v)
                            : (plan_range_holds(e, ea, v) || plan_words_hold(p, t, e, ea, v));
    if (holds) st_relaxed_u32(&p.conf[t], tag);   // the walk still waits for the header's own tags
    else redo = true;
  }
  const uint32_t m = __ballot_sync(kFull, redo);
  if (m) {
    uint32_t base = 0;
    if (lane == 0) base = atomicAdd(&p.ctr[C_REDO_RES], (uint32_t)__popc(m));
    base = __shfl_sync(kFull, base, 0);
    if (redo) st_release_u32(&p.redo[base + __popc(m & ((1u << lane) - 1u))], (tag << 24) | (uint32_t)t);
  }
}

__device__ __forceinline__ void scan_bar() { asm volatile("bar.sync 1, %0;" ::"n"(kThreads) : "memory"); }

// The scanner: the tiles' sums, in order as their units publish them, into
// each tile's exclusive prefix (double-float; a sum's first tile starts from
// the sum's start value, which its unit has added and published).  Warps 0-7,
// one tile a thread: a round takes the 256 tiles from pos, up to the first
// that is not published; each warp scans its 32 (segmented at a sum's first
// tile), the warps' totals meet in shared memory (two named barriers a
// round), and every thread publishes its tile's prefix; the next round's sums
// are loaded while this one is scanned.  In a planned call (kPlanned) each
// thread also tells whether its tile's header stands (scan_release).
template <bool kPlanned>
__device__ __noinline__ void scan_cta(const Params &p, Smem &sm, int64_t ntiles) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  if (w >= kWarps) return;
  const uint32_t tag = sm.tag;
  constexpr int kRound = kThreads;
  uint4 *const pout = kPlanned ? p.prec_next : p.prec;
  DF carry = DF{0.0f, 0.0f};   // the inclusive prefix of the tile before pos
  float carry_abs = 0.0f;
  int64_t pos = 0;
  uint64_t t_wait = 0;
  int stop = 0;                // warp 0, lane 0: the scan gives up (bounded wait)
  uint32_t it = 0;             // iterations: the parity picks the buffer of first-unready indices
  uint4 v = threadIdx.x < ntiles ? ld_vol_v4(&p.status[threadIdx.x]) : make_uint4(0, 0, 0, 0);
  while (pos < ntiles) {
    const int i = threadIdx.x;   // this thread's tile: pos + i
    const bool in = pos + i < ntiles;
    const bool rd = ((v.w >> 8) & 0xFFu) == tag && (v.w & 3u) == 1u;
    const uint32_t nrm = __ballot_sync(kFull, in && !rd);
    const int wfirst = nrm ? 32 * w + __ffs(nrm) - 1 : kRound;   // (a warp all published does not bound the round)
    if (lane == 0) sm.scan_first[it & 1][w] = wfirst;
    if (w == 0 && lane == 0) sm.scan_stop = stop;
    scan_bar();
    if (sm.scan_stop) break;
    int nready = kRound;
#pragma unroll
    for (int k = 0; k < kWarps; k++) nready = min(nready, sm.scan_first[it & 1][k]);
    nready = (int)min((int64_t)nready, ntiles - pos);
    it++;
    if (nready == 0) {
      // nothing new yet (bounded: past the limit the run units give up on their prefixes too)
      if (w == 0 && lane == 0) {
        stat_add(sm, S_SCAN_POLLS, 1);
        if (!t_wait) t_wait = gtimer();
        else if (gtimer() - t_wait > p.wait_ns) {
          note_timeout(p, ERR_PLAN_TIMEOUT, 6, (uint32_t)pos, 0);
          stop = 1;
        }
      }
      __nanosleep(128);
      v = in ? ld_vol_v4(&p.status[pos + i]) : make_uint4(0, 0, 0, 0);
      continue;
    }
    t_wait = 0;
    const bool mine = i < nready;
    const uint4 cur = v;
    // the next round's sums, in flight while this one is scanned
    v = pos + nready + i < ntiles ? ld_vol_v4(&p.status[pos + nready + i]) : make_uint4(0, 0, 0, 0);
    // the warp's segmented inclusive scan (a sum's first tile, flag 4, restarts it)
    const bool hd = mine && (cur.w & 4u) != 0u;
    DF x = mine ? DF{__uint_as_float(cur.x), __uint_as_float(cur.y)} : DF{0.0f, 0.0f};
    float xa = mine ? __uint_as_float(cur.z) : 0.0f;
    bool hx = hd;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      DF y;
      y.hi = __shfl_up_sync(kFull, x.hi, o);
      y.lo = __shfl_up_sync(kFull, x.lo, o);
      const float ya = __shfl_up_sync(kFull, xa, o);
      const bool hy = __shfl_up_sync(kFull, hx, o);
      if (lane >= o) {
        if (!hx) {
          x = df_add(y, x);
          xa = __fadd_rn(ya, xa);
        }
        hx = hx || hy;
      }
    }
    if (lane == 31) {
      sm.scan_tot[w] = make_float4(x.hi, x.lo, xa, hx ? 1.0f : 0.0f);
    }
    scan_bar();
    // the prefix before this warp's tiles (wbase), and the carry into the next round
    DF base = carry, wbase = carry;
    float base_a = carry_abs, wbase_a = carry_abs;
#pragma unroll
    for (int k = 0; k < kWarps; k++) {
      if (k == w) {
        wbase = base;
        wbase_a = base_a;
      }
      const float4 tk = sm.scan_tot[k];
      if (tk.w != 0.0f) {
        base = DF{tk.x, tk.y};
        base_a = tk.z;
      } else {
        base = df_add(base, DF{tk.x, tk.y});
        base_a = __fadd_rn(base_a, tk.z);
      }
    }
    carry = base;
    carry_abs = base_a;
    {
      // each tile's exclusive prefix from the lane before it
      DF y;
      y.hi = __shfl_up_sync(kFull, x.hi, 1);
      y.lo = __shfl_up_sync(kFull, x.lo, 1);
      const float ya = __shfl_up_sync(kFull, xa, 1);
      const bool hy = __shfl_up_sync(kFull, hx, 1);
      DF e = wbase;
      float ea = wbase_a;
      if (lane > 0) {
        if (hy) {
          e = y;
          ea = ya;
        } else {
          e = df_add(wbase, y);
          ea = __fadd_rn(wbase_a, ya);
        }
      }
      if (mine && !hd)
        st_vol_v4(&pout[(pos + i) * kPrecWords],
                  make_uint4(__float_as_uint(e.hi), __float_as_uint(e.lo), __float_as_uint(ea), (tag << 8) | 2u));
      if (kPlanned) scan_release(p, pos + i, mine, hd, e, ea, cur, tag);
    }
    if (w == 0 && lane == 0) stat_add(sm, S_SCAN_WINDOWS, 1);
    pos += nready;
  }
  if (kPlanned) {
    // every warp's places on the redo list are taken: the list is final
    // (also when the scan gave up)
    scan_bar();
    if (w == 0 && lane == 0) {
      __threadfence();
      st_release_u32(&p.ctr[C_SCAN_FIN], 1u);
    }
  }
  if (w == 0 && lane == 0) p.stats[S_T_SCAN_END] = gtimer();
}

// ------------------------------------------------------------------ the walk: raw terms
// Terms i..n-1 of a row (lane l holds term l) added to Sb one by one with the
// hardware add, in order (one warp; every lane computes the same value).  For
// a row of 16 this is shorter than a round of prefix checks per crossing.
__device__ __noinline__ uint64_t row_dadd(Smem &sm, uint64_t Sb, uint64_t t, int i, int n) {
  const int lane = threadIdx.x & 31;
  const uint64_t t_in = clock64();
  double S = bitsd(Sb);
  for (int j = i; j < n; j++) S = __dadd_rn(S, bitsd(__shfl_sync(kFull, t, j)));
  if (lane == 0) {
    stat_add(sm, S_TERMS_DADD, (unsigned long long)max(0, n - i));
    stat_add(sm, S_CY_WALK_RAW, clock64() - t_in);
  }
  return dbits(S);
}

// One warp adds up to 32 terms (lane l holds term l; lanes >= n hold -0) to
// the exact running value Sb, in order: while Sb is a normal number (with
// e >= -959), every term's run under Sb's binade is scanned in order and
// checked prefix by prefix against Sb; the longest prefix that passes is
// applied at once, and the term after it (which leaves the binade) is added
// with the hardware add.  A zero, subnormal, tiny or non-finite Sb takes one
// hardware add per term.
__device__ __noinline__ uint64_t raw_chunk(Smem &sm, uint64_t Sb, uint64_t t, int i, int n) {
  const int lane = threadIdx.x & 31;
  const uint64_t t_in = clock64();
  uint32_t rounds = 0, dadds = 0;
  while (i < n) {
    const uint32_t Eb = (uint32_t)(Sb >> 52) & 0x7FFu;
    if (Eb >= 64u && Eb < 0x7FFu) {
      // the common case: no term of the other sign, no tie -- the magnitudes'
      // increments simply add, and the check of a prefix is m + P <= 2^53
      const bool inr = lane >= i && lane < n;
      const uint32_t hi = (uint32_t)(t >> 32);
      const uint32_t E = (hi >> 20) & 0x7FFu;
      const bool opp = inr && (hi >> 31) != (uint32_t)(Sb >> 63) && (t << 1) != 0;
      const bool big = inr && E >= Eb;   // |t| >= 2^e, inf or NaN: never inside this binade
      uint32_t tt = 1;
      const uint64_t rr = inr ? term_mag_halfup(hi, (uint32_t)t, 64 - (int)Eb, tt) : 0ull;
      if (!__any_sync(kFull, opp || (inr && !big && tt == 0u))) {
        uint64_t P = big ? (1ull << 57) : rr;   // a term that cannot be added ends every prefix through it
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const uint64_t q = __shfl_up_sync(kFull, P, o);
          if (lane >= o) P += q;
        }
        const uint64_t m = (Sb & kFracMask) | kHidden;
        const bool ok = inr && m + P <= (uint64_t)kTwo53;
        const uint32_t okm = __ballot_sync(kFull, ok);
        const uint32_t inrange = (n >= 32 ? kFull : ((1u << n) - 1u)) & ~((1u << i) - 1u);
        const uint32_t fail = ~okm & inrange;
        int j = fail ? __ffs(fail) - 1 : n;
        if (j > i) Sb += __shfl_sync(kFull, P, j - 1);   // the magnitude grows by P; a count of 2^53 is 2^(e+1)
        if (j < n) {
          const uint64_t tj = __shfl_sync(kFull, t, j);
          Sb = dbits(__dadd_rn(bitsd(Sb), bitsd(tj)));
          j++;
          dadds++;
        }
        rounds++;
        i = j;
        continue;
      }
      const int e = (int)Eb - 1023;
      Run r = run_empty();
      if (lane >= i && lane < n) {
        int64_t re;
        int32_t d;
        const bool poison = term_inc(t, e, re, d);
        run_push(r, re, d, term_flags(t) | (poison ? (uint32_t)F_POISON : 0u));
      }
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const Run q = shfl_run_up(r, o);
        if (lane >= o) r = run_compose(q, r);
      }
      uint64_t nb = Sb;
      const bool ok = (lane >= i && lane < n) && run_apply(nb, r, e) == APPLY_OK;
      const uint32_t okm = __ballot_sync(kFull, ok);
      const uint32_t inrange = (n >= 32 ? kFull : ((1u << n) - 1u)) & ~((1u << i) - 1u);
      const uint32_t fail = ~okm & inrange;
      int j = fail ? __ffs(fail) - 1 : n;
      if (j > i) Sb = __shfl_sync(kFull, nb, j - 1);
      if (j < n) {
        const uint64_t tj = __shfl_sync(kFull, t, j);
        Sb = dbits(__dadd_rn(bitsd(Sb), bitsd(tj)));
        j++;
        dadds++;
      }
      rounds++;
      i = j;
    } else {
      const uint64_t ti = __shfl_sync(kFull, t, i);
      Sb = dbits(__dadd_rn(bitsd(Sb), bitsd(ti)));
      i++;
      dadds++;
    }
  }
  if (lane == 0) {
    stat_add(sm, S_RAW_ROUNDS, rounds);
    stat_add(sm, S_TERMS_DADD, dadds);
    stat_add(sm, S_CY_WALK_RAW, clock64() - t_in);
  }
  return Sb;
}

// The terms x[a .. b) of the sum (already clipped to it) added by one warp.
__device__ __noinline__ uint64_t raw_from_x(const Params &p, Smem &sm, uint64_t Sb, int64_t a, int64_t b) {
  const int lane = threadIdx.x & 31;
  const unsigned long long *xp = reinterpret_cast<const unsigned long long *>(p.x);
  for (int64_t g = a; g < b; g += 32) {
    const int n = (int)min((int64_t)32, b - g);
    const uint64_t t = lane < n ? (uint64_t)__ldg(xp + g + lane) : kNegZero;
    Sb = raw_chunk(sm, Sb, t, 0, n);
  }
  return Sb;
}

// A raw row with prefix tables for the binades ea and ea + 1 (one warp; every
// lane computes the same S): data holds its 16 terms, then the two tables,
// lims where each table stops being usable (5 bits each).  While S is in one of them, of the row's sign,
// and the table holds: the longest prefix whose increments keep the count
// within the binade (m + P <= 2^53) is added at once, and the term after it
// with the hardware add.  The rest goes term by term (raw_chunk).
__device__ __forceinline__ uint64_t raw2_row(Smem &sm, uint64_t S, const uint64_t *data, uint32_t lims, uint32_t ea,
                                          uint64_t neg, uint32_t &n_rounds, uint32_t &n_dadds) {
  const int lane = threadIdx.x & 31;
  const int la = (int)(lims & 31u), lb = (int)((lims >> 5) & 31u);
  const uint64_t t = lane < kLaneTerms ? data[lane] : kNegZero;
  const uint64_t pa = lane < kLaneTerms ? data[kLaneTerms + lane] : 0ull;
  const uint64_t pb = lane < kLaneTerms ? data[2 * kLaneTerms + lane] : 0ull;
  int i = 0;
  uint32_t rounds = 0, dadds = 0;
  if (((uint32_t)(S >> 52) & 0x7FFu) == ea && (S >> 63) == neg && la == kLaneTerms && lb == kLaneTerms) {
    // the common row: S in the lower binade, both tables whole.  The
    // increments are non-negative, so the terms that keep the count within
    // the binade are a prefix; the term after it crosses (the hardware add)
    // and the rest is one check and one add in the upper binade.
    const uint64_t m = (S & kFracMask) | kHidden;
    const uint32_t okm = __ballot_sync(kFull, lane < kLaneTerms && m + pa <= (uint64_t)kTwo53) & 0xFFFFu;
    const int k = __ffs(~okm) - 1;   // 16: no crossing
    const uint64_t pk = __shfl_sync(kFull, pa, (k - 1) & 31);
    const uint64_t xk = __shfl_sync(kFull, t, k & 15);
    const uint64_t pbk = __shfl_sync(kFull, pb, k & 15), pb15 = __shfl_sync(kFull, pb, kLaneTerms - 1);
    if (k > 0) S += pk;   // a count of 2^53 is 2^(e+1)
    rounds = 1;
    i = k;
    if (k < kLaneTerms) {
      S = dbits(__dadd_rn(bitsd(S), bitsd(xk)));
      dadds = 1;
      i = k + 1;
      const uint64_t rest = pb15 - pbk, m2 = (S & kFracMask) | kHidden;
      if (i < kLaneTerms && ((uint32_t)(S >> 52) & 0x7FFu) == ea + 1u && (S >> 63) == neg &&
          m2 + rest <= (uint64_t)kTwo53) {
        S += rest;
        i = kLaneTerms;
        rounds = 2;
      }
    }
  }
  while (i < kLaneTerms) {
    const uint32_t Eb = (uint32_t)(S >> 52) & 0x7FFu;
    const bool use_a = Eb == ea && i < la, use_b = Eb == ea + 1u && i < lb;
    if ((S >> 63) != neg || !(use_a || use_b)) break;
    const uint64_t P = use_a ? pa : pb;
    const int lim = use_a ? la : lb;
    const uint64_t base = i > 0 ? __shfl_sync(kFull, P, i - 1) : 0ull;
    const uint64_t m = (S & kFracMask) | kHidden;
    const bool ok = lane >= i && lane < lim && m + (P - base) <= (uint64_t)kTwo53;
    const uint32_t inr = ((1u << lim) - 1u) & ~((1u << i) - 1u);
    const uint32_t fail = ~__ballot_sync(kFull, ok) & inr;
    const int k = fail ? __ffs(fail) - 1 : lim;
    if (k > i) S += __shfl_sync(kFull, P, k - 1) - base;   // the magnitude grows; a count of 2^53 is 2^(e+1)
    rounds++;
    i = k;
    if (k == lim) break;   // the table ends here (or the row does)
    S = dbits(__dadd_rn(bitsd(S), bitsd(__shfl_sync(kFull, t, k))));
    dadds++;
    i = k + 1;
  }
  n_rounds += rounds;   // (the caller's counters: no shared-memory update on the in-order path)
  n_dadds += dadds;
#ifdef SEQSUM_PROFILE
  if (lane == 0) sm.prof_i = (uint32_t)i | (rounds << 8) | (dadds << 16) | (((uint32_t)(S >> 52) & 0x7FFu) << 20);
#endif
  if (i < kLaneTerms) S = row_dadd(sm, S, t, i, kLaneTerms);
  return S;
}

// ------------------------------------------------------------------ the walk: ranges of tiles
// A walker CTA: eight producer warps and one in-order warp.  The tiles of a
// sum are cut into ranges -- small at the sum's start, where a sum that
// starts near zero crosses many binades, then kRangeTiles; producer warp k
// takes ranges k, k + 8, ... and writes each, composed into steps, to its own
// slot; the in-order warp takes the slots in range order and applies their
// steps to the exact running value.  A slot's full and empty mbarriers hand
// it over.
struct WalkSum {
  int64_t tb, te;        // the sum's tiles
  int64_t row_base;      // the sum's first row
  int64_t g_lo, g_hi;    // the sum's terms
};

__device__ __forceinline__ void clip(const WalkSum &ws, int64_t tile, uint32_t start, uint32_t count, int64_t &a,
                                     int64_t &b) {
  const int64_t g0 = (ws.row_base + (tile - ws.tb) * kTileRows) * kLaneTerms;
  a = max(g0 + (int64_t)start, ws.g_lo);
  b = min(g0 + (int64_t)start + (int64_t)count, ws.g_hi);
}


// One step of the in-order pass: a composite of consecutive runs of one
// binade, a raw row, or a range of terms read from x.
enum : uint32_t { ST_RUN = 0, ST_RAW = 1, ST_RAW2 = 2, ST_X = 3 };
struct __align__(16) Step {
  int64_t inc, lo, hi;   // a composite's run; a raw row: its place among the slot's fetched rows (in inc)
  uint64_t meta;         // kind (2 bits), biased binade (11), d + 1 (2), flags (8), then its terms:
                         // first tile (7) and row (9), last tile (7) and row after it (9), within the range;
                         // bit 56: a plain run (non-negative, no tie, no poison)
};
__device__ __forceinline__ uint64_t step_meta(uint32_t kind, uint32_t eb, int32_t d, uint32_t flags, uint32_t from,
                                              uint32_t to) {
  const bool plain = kind == 0u && d == 0 && (flags & F_NONNEG) && !(flags & F_POISON);
  return (uint64_t)(kind & 3u) | ((uint64_t)(eb & 0x7FFu) << 2) | ((uint64_t)((d + 1) & 3) << 13) |
         ((uint64_t)(flags & 0xFFu) << 15) | ((uint64_t)(from & 0xFFFFu) << 23) | ((uint64_t)(to & 0xFFFFu) << 39) |
         ((uint64_t)(plain ? 1u : 0u) << 56);
}
// a position in a range: tile (7 bits) and row (9 bits); positions compare as numbers
__device__ __forceinline__ uint32_t rpos(uint32_t tile, uint32_t row) { return (tile << 9) | row; }

constexpr int kRangeTiles = 4 * 32;   // tiles of a walk range (four per lane of a producer warp)
// Ranges 0..7 hold 8, 8, 16, 16, 32, 32, 64, 64 tiles (240 in all), the later ones kRangeTiles.
__device__ __forceinline__ int64_t range_start(int r) {
  if (r >= 8) return 240 + (int64_t)(r - 8) * kRangeTiles;
  return (int64_t)(8 << (r >> 1)) * (2 + (r & 1)) - 16;
}
__device__ __forceinline__ int range_count(int64_t tiles) {
  if (tiles > 240) return 8 + (int)((tiles - 240 + kRangeTiles - 1) / kRangeTiles);
  int r = 0;
  while (range_start(r) < tiles) r++;
  return r;
}
constexpr int kRangeSteps = 64;       // steps a slot holds (more: the range is read from x)
constexpr int kRangeRaw = 24;         // raw rows a slot holds with their terms and tables
struct RangeSlot {
  Step steps[kRangeSteps];
  uint64_t raw[kRangeRaw][3 * kLaneTerms];   // a raw row's terms, then its two prefix tables
  uint32_t rawlim[kRangeRaw];                // where each table stops being usable (5 bits each)
  uint32_t rawpos[kRangeRaw];                // its first term: position in the range, with tables (bit 16), binade
  int nsteps;                                // -1: the steps did not fit
  int fail;                                  // a header never came
};
static_assert(sizeof(RangeSlot) % 16 == 0, "slots stay 16-byte aligned");
static_assert(kWarps * sizeof(RangeSlot) <= kDynSmem - 1024, "the walk's slots fit the dynamic shared memory");

// An element of a range, in the order of its terms: a tile's run (its
// header), an item of a complex tile (a run or a raw row), or terms read from
// x (a region or a tile without items).
enum : uint32_t { EK_RUN = 0, EK_RAW = 1, EK_RAW2 = 2, EK_X = 3 };
struct Elem {
  Run r;
  uint32_t kind, key;    // key: the run's biased binade; kNoKey for the others
  uint32_t from, to;     // its terms: positions in the range
  uint32_t eb, neg;      // a raw row with tables: the lower binade and the sign
};

// The number of items of a complex tile's compact list (0: none usable, the
// tile is read from x).
// A complex tile's header: warp k's count of items in bits 6k..6k+5.  The
// tile's items (0 if a count is out of range).
__device__ __forceinline__ uint32_t complex_items(const Rec &h) {
  uint32_t n = 0;
  bool ok = true;
#pragma unroll
  for (int k = 0; k < kWarps; k++) {
    const uint32_t c = (uint32_t)(h.w[0] >> (6 * k)) & 63u;
    ok = ok && c <= (uint32_t)kWarpSlots;
    n += c;
  }
  return ok ? n : 0u;
}
// The slot of a complex tile's item kk (its items in the order of their terms).
__device__ __forceinline__ uint32_t complex_slot(const Rec &h, uint32_t kk) {
  uint32_t base = 0, slot = 0;
#pragma unroll
  for (int k = 0; k < kWarps; k++) {
    const uint32_t c = (uint32_t)(h.w[0] >> (6 * k)) & 63u;
    if (kk >= base && kk < base + c) slot = (uint32_t)k * kWarpSlots + (kk - base);
    base += c;
  }
  return slot;
}

// Element E of the range, in two parts so that the record of the next chunk
// can be in flight while this one is composed.  range_fetch (every lane of
// the warp calls it; in: E < n) finds the element's tile and takes the
// tile's header from the lane that read it, or starts the load of the
// element's item; range_decode reads the element from that record.
// off: this lane's first element; eo: the first elements of its four tiles;
// direct: every tile is one element (element E is tile E).
struct ElemRec {
  Rec q;          // the tile's header (a run or a tile read from x) or the item
  uint32_t tt;    // the tile in the range
  uint32_t what;  // 0: q is a run header; 1: q is an item; 2: the tile is read from x
  bool in;
};
__device__ __forceinline__ ElemRec range_fetch(const Params &p, const Rec (&hl)[4], int64_t ta, int E, bool in,
                                               uint32_t off, const uint32_t (&eo)[4], bool direct) {
  uint32_t tt = (uint32_t)E, kk = 0;
  if (!direct) {
    // the lane whose tiles hold E: the last with off <= E
    int o = 0;
#pragma unroll
    for (int step = 16; step > 0; step >>= 1) {
      const uint32_t v = __shfl_sync(kFull, off, o + step);
      if (in && v <= (uint32_t)E) o += step;
    }
    const uint32_t e0 = __shfl_sync(kFull, eo[0], o), e1 = __shfl_sync(kFull, eo[1], o),
                   e2 = __shfl_sync(kFull, eo[2], o), e3 = __shfl_sync(kFull, eo[3], o);
    const uint32_t j = (uint32_t)E >= e3 ? 3u : ((uint32_t)E >= e2 ? 2u : ((uint32_t)E >= e1 ? 1u : 0u));
    kk = (uint32_t)E - (j == 3u ? e3 : (j == 2u ? e2 : (j == 1u ? e1 : e0)));
    tt = 4u * (uint32_t)o + j;
  }
  ElemRec er;
  er.tt = tt;
  er.in = in;
  er.what = 2;
  // the tile's header, from the lane that read it
  Rec h;
  h.w[0] = h.w[1] = h.w[2] = h.w[3] = 0;
  const int src = (int)(tt >> 2) & 31, jt = (int)(tt & 3u);
#pragma unroll
  for (int j = 0; j < 4; j++) {
#pragma unroll
    for (int q = 0; q < 4; q++) {
      const uint64_t v = (uint64_t)__shfl_sync(kFull, (long long)hl[j].w[q], src);
      if (j == jt) h.w[q] = v;
    }
  }
  er.q = h;
  if (!in) return er;
  const uint32_t hk = (uint32_t)(h.w[3] & 7u);
  if (hk == K_RUN) {
    er.what = 0;
  } else if (hk == K_COMPLEX && complex_items(h) > 0 && SQ_OK(p, kk < complex_items(h), 3, kk)) {
    er.q = ld_rec_vol(&p.items[(ta + tt) * kItemSlots + complex_slot(h, kk)]);
    er.what = 1;
  }
  return er;
}
__device__ __forceinline__ Elem range_decode(const ElemRec &er) {
  Elem el;
  el.r = run_empty();
  el.kind = EK_X;
  el.key = kNoKey;
  el.eb = el.neg = 0;
  el.from = rpos(er.tt, 0);
  el.to = rpos(er.tt, kTileRows);
  if (!er.in || er.what == 2) return el;
  const Item it = unpack_item(er.q);
  if (er.what == 1) {
    el.from = rpos(er.tt, it.start / kLaneTerms);
    el.to = rpos(er.tt, (it.start + it.count) / kLaneTerms);
  }
  if (it.kind == K_RUN) {
    el.r = it.r;
    el.kind = EK_RUN;
    el.key = it.eb;
  } else if (er.what == 1 && (it.kind == K_RAW || it.kind == K_RAW2)) {
    el.kind = it.kind == K_RAW ? EK_RAW : EK_RAW2;
    el.eb = it.eb;
    el.neg = (uint32_t)(er.q.w[0] & 1u);
  }
  return el;
}

// Waits (bounded) for phase `ph` of an mbarrier; false if the limit passed.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t ph, uint64_t limit_ns) {
  uint64_t t0 = 0;
  for (uint32_t spin = 0; !mbar_try_wait(bar, ph); spin++) {
    if ((spin & 63u) == 63u) {
      const uint64_t now = gtimer();
      if (!t0) t0 = now;
      else if (now - t0 > limit_ns) return false;
    }
  }
  return true;
}

// A producer warp: the ranges pw, pw + 8, ... of one sum into slot pw.
__device__ __noinline__ void walk_producer(const Params &p, Smem &sm, RangeSlot &rs, const WalkSum &ws, int nranges,
                                           int pw, uint32_t tag) {
  const int lane = threadIdx.x & 31;
  const uint32_t lt = (1u << lane) - 1u;
  bool failed_all = false;
  const bool x16 = (reinterpret_cast<uintptr_t>(p.x) & 15u) == 0;   // rows can be copied 16 bytes at a time
  for (int r = pw; r < nranges; r += kWarps) {
    const uint32_t use = sm.wuse_p[pw];
    bool ok = !failed_all;
    const int64_t ta = ws.tb + range_start(r);
    const int tn = (int)min(range_start(r + 1) - range_start(r), ws.te - ta);
    // ---- the range's headers (four a lane), as they arrive
    Rec h[4];
    uint32_t need = 0;
#pragma unroll
    for (int j = 0; j < 4; j++) {
      h[j].w[0] = h[j].w[1] = h[j].w[2] = h[j].w[3] = 0;
      if (4 * lane + j < tn) need |= 1u << j;
    }
    const uint64_t c0 = clock64();
    uint64_t t0 = 0;
    for (uint32_t spin = 0; ok; spin++) {
#pragma unroll
      for (int j = 0; j < 4; j++) {
        if (need & (1u << j)) {
          // (a planned call: once the scanner, or the tile's second unit, has released it)
          const int64_t tj = ta + 4 * lane + j;
          if (!p.planned || ld_acquire_u32(&p.conf[tj]) == tag) {
            h[j] = ld_rec_vol(&p.hdr[tj]);
            if (tags_ok(h[j], tag)) need &= ~(1u << j);
          }
        }
      }
      if (__all_sync(kFull, need == 0u)) break;
      const uint64_t now = gtimer();
      if (!t0) t0 = now;
      else if (now - t0 > p.wait_ns) {
        if (lane == 0) note_timeout(p, ERR_WALK_TIMEOUT, 3, (uint32_t)ta, (uint32_t)ws.te);
        ok = false;
      }
      __nanosleep(200);
    }
    ok = __all_sync(kFull, ok);
    if (lane == 0) stat_add(sm, S_CY_WALK_WAIT, clock64() - c0);
    WRT(r, 0);
    fence_acq_rel();
    // ---- its elements: a run or overflow tile is one, a complex tile one per item
    uint32_t eo[4], n = 0;
#pragma unroll
    for (int j = 0; j < 4; j++) {
      eo[j] = n;
      if (4 * lane + j < tn) {
        const uint32_t hk = (uint32_t)(h[j].w[3] & 7u);
        n += (hk == K_COMPLEX && complex_items(h[j]) > 0) ? complex_items(h[j]) : 1u;
      }
    }
    uint32_t off = n;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t q = __shfl_up_sync(kFull, off, o);
      if (lane >= o) off += q;
    }
    // the slot's previous use must have been applied (waited for only now:
    // the headers above were read while the in-order warp still held it)
    if (use > 0) ok = __all_sync(kFull, mbar_wait_bounded(&sm.wempty[pw], (use - 1) & 1u, 4 * p.wait_ns)) && ok;
    const int N = ok ? (int)__shfl_sync(kFull, off, 31) : 0;
    const bool direct = N == tn;   // every tile one element
    WR0(r, 0);
    if (ok && lane == 0) (void)SQ_OK(p, N >= tn, 4, N);
    off -= n;
#pragma unroll
    for (int j = 0; j < 4; j++) eo[j] += off;
    __syncwarp();
    // ---- the segmented scan, 32 elements at a time; steps at the tails
    int nsteps = 0, nraw = 0;
    bool over = false;
    Run carry = run_empty();      // the composite of the open segment (since its head)
    uint32_t ckey = kNoKey, cfrom = 0, cto = 0;
    bool pending = false;         // the chunk before ended inside a segment
    ElemRec nx = range_fetch(p, h, ta, lane, lane < N, off, eo, direct);
    for (int c = 0; c < N; c += 32) {
      const int E = c + lane;
      const bool in = E < N;
      const ElemRec cur = nx;
      if (c + 32 < N) nx = range_fetch(p, h, ta, E + 32, E + 32 < N, off, eo, direct);   // in flight meanwhile
      const Elem el = range_decode(cur);
      WR0(r, 2 + 2 * (c / 32));
      const uint32_t key = in ? el.key : kNoKey;
      uint32_t pkey = __shfl_up_sync(kFull, key, 1);
      if (lane == 0) pkey = ckey;
      const bool head = in && (E == 0 || key == kNoKey || pkey == kNoKey || key != pkey);
      // the open segment of the chunk before ends if this chunk begins with a head
      const bool close_prev = __shfl_sync(kFull, head, 0) && pending;
      if (close_prev && lane == 0 && nsteps < kRangeSteps) {
        Step st;
        st.inc = carry.inc;
        st.lo = carry.lo;
        st.hi = carry.hi;
        st.meta = step_meta(ST_RUN, ckey, carry.d, carry.flags, cfrom, cto);
        rs.steps[nsteps] = st;
      }
      if (close_prev) nsteps++;
      // the common chunk: runs of one binade, non-negative, without a tie,
      // no head after its first element -- their increments simply add
      const uint32_t key0 = __shfl_sync(kFull, key, 0);
      const bool plain = __all_sync(kFull, !in || (el.kind == EK_RUN && el.r.d == 0 && (el.r.flags & F_NONNEG) &&
                                                   key == key0 && (lane == 0 || !head)));
      if (plain) {
        long long a = in ? (long long)el.r.inc : 0ll;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) a += __shfl_xor_sync(kFull, a, o);
        const uint32_t fand = __reduce_and_sync(
            kFull, in ? (el.r.flags & (F_NONNEG | F_NONPOS | F_ZERO | F_ALLNEGZ)) : (uint32_t)(F_NONNEG | F_NONPOS | F_ZERO | F_ALLNEGZ));
        const uint32_t fo = __reduce_or_sync(kFull, in ? (el.r.flags & ~(uint32_t)(F_NONNEG | F_NONPOS | F_ZERO | F_ALLNEGZ)) : 0u);
        Run ch;
        ch.inc = a;
        ch.lo = 0;
        ch.hi = a;
        ch.d = 0;
        ch.flags = fand | fo;
        saturate(ch);
        const bool h0 = __shfl_sync(kFull, head, 0);
        const Run comp = h0 ? ch : run_compose(carry, ch);
        const uint32_t from0 = h0 ? __shfl_sync(kFull, el.from, 0) : cfrom;
        const int lastl = min(31, N - 1 - c);
        const uint32_t to = __shfl_sync(kFull, el.to, lastl);
        if (c + 32 >= N) {
          // the range's last element: the segment ends here
          if (lane == 0 && nsteps < kRangeSteps) {
            Step st;
            st.inc = comp.inc;
            st.lo = comp.lo;
            st.hi = comp.hi;
            st.meta = step_meta(ST_RUN, key0, comp.d, comp.flags, from0, to);
            rs.steps[nsteps] = st;
          }
          nsteps++;
          pending = false;
        } else {
          pending = true;
        }
        carry = comp;
        ckey = key0;
        cfrom = from0;
        cto = to;
        WR0(r, 3 + 2 * (c / 32));
        continue;
      }
      Run rr = el.r;
      bool f = head;
      uint32_t from = head ? el.from : 0u;
      // every run of the chunk (and the open one before it) plain: a segmented
      // sum of the increments, an AND of the flags
      const bool cplain = carry.d == 0 && (carry.flags & F_NONNEG) && !(carry.flags & F_POISON);
      const bool splain = __all_sync(kFull, el.kind != EK_RUN || (el.r.d == 0 && (el.r.flags & F_NONNEG) &&
                                                                   !(el.r.flags & F_POISON))) &&
                          (__shfl_sync(kFull, head, 0) || cplain);
      if (splain) {
        long long a = el.kind == EK_RUN ? (long long)el.r.inc : 0ll;
        uint32_t fl = el.kind == EK_RUN ? el.r.flags : 0u;
        if (lane == 0 && in && !head) {
          a += (long long)carry.inc;
          fl &= carry.flags;
          from = cfrom;
          f = true;
        }
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const long long qa = __shfl_up_sync(kFull, a, o);
          const uint32_t qfl = __shfl_up_sync(kFull, fl, o);
          const bool qh = __shfl_up_sync(kFull, f, o);
          const uint32_t qf = __shfl_up_sync(kFull, from, o);
          if (lane >= o) {
            if (!f) {
              a += qa;
              fl &= qfl;
            }
            f = f || qh;
            from = max(from, qf);
          }
        }
        rr.inc = a;
        rr.lo = 0;
        rr.hi = a;
        rr.d = 0;
        rr.flags = fl;
        saturate(rr);
      } else {
        if (lane == 0 && in && !head) {
          rr = run_compose(carry, rr);
          from = cfrom;
          f = true;   // the carry stands for its head
        }
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const Run q = shfl_run_up(rr, o);
          const bool qh = __shfl_up_sync(kFull, f, o);
          const uint32_t qf = __shfl_up_sync(kFull, from, o);
          if (lane >= o) {
            if (!f) rr = run_compose(q, rr);
            f = f || qh;
            from = max(from, qf);
          }
        }
      }
      // tails: the next element is a head (lane 31 decides with the next chunk)
      const uint32_t nkey = __shfl_down_sync(kFull, key, 1);
      const bool last = E == N - 1;
      const bool tail = in && (key == kNoKey || last || (lane < 31 && (nkey == kNoKey || nkey != key)));
      const uint32_t tb = __ballot_sync(kFull, tail);
      const uint32_t rb = __ballot_sync(kFull, tail && (el.kind == EK_RAW || el.kind == EK_RAW2));
      if (tail) {
        const int at = nsteps + __popc(tb & lt);
        if (at < kRangeSteps) {
          Step st;
          if (el.kind == EK_RUN) {
            st.inc = rr.inc;
            st.lo = rr.lo;
            st.hi = rr.hi;
            st.meta = step_meta(ST_RUN, key, rr.d, rr.flags, from, el.to);
          } else {
            const uint32_t q = (uint32_t)nraw + __popc(rb & lt);
            st.inc = (int64_t)q;
            if (q < (uint32_t)kRangeRaw) {
              // the row's terms, copied now: they land while the range is composed
              const int64_t g0 = (ws.row_base + (ta + (el.from >> 9) - ws.tb) * kTileRows + (el.from & 511u)) * kLaneTerms;
              const bool pre = x16 && g0 >= ws.g_lo && g0 + kLaneTerms <= ws.g_hi;
              if (pre) {
                const double *src = p.x + g0;
#pragma unroll
                for (int k = 0; k < kLaneTerms / 2; k++) cp_async16(&rs.raw[q][2 * k], src + 2 * k);
              }
              rs.rawpos[q] = el.from | (el.kind == EK_RAW2 ? 1u << 16 : 0u) | ((el.eb & 0x7FFu) << 17) |
                             (pre ? 1u << 28 : 0u);
            }
            st.lo = st.hi = 0;
            const uint32_t sk = el.kind == EK_RAW ? ST_RAW : (el.kind == EK_RAW2 ? ST_RAW2 : ST_X);
            st.meta = step_meta(sk, el.eb, 0, el.neg, el.from, el.to);
          }
          rs.steps[at] = st;
        }
      }
      nsteps += __popc(tb);
      nraw += __popc(rb);
      // the open segment at the end of the chunk
      carry = shfl_run_idx(rr, 31);
      ckey = __shfl_sync(kFull, key, 31);
      cfrom = __shfl_sync(kFull, from, 31);
      cto = __shfl_sync(kFull, el.to, 31);
      pending = __shfl_sync(kFull, in && !tail, 31);
      WR0(r, 3 + 2 * (c / 32));
    }
    WR0(r, 30);
    over = nsteps > kRangeSteps;
    if (lane == 0 && N > 0) (void)SQ_OK(p, nsteps >= 1, 6, N);
    __syncwarp();
    // ---- the raw rows' terms (the copies issued at the tails; the rest now),
    // then their prefix tables, two rows at a time
    const int nfetch = over ? 0 : min(nraw, kRangeRaw);
    cp_async_wait();
    for (int w0 = lane; w0 < nfetch * kLaneTerms; w0 += 32) {
      const uint32_t rp = rs.rawpos[w0 / kLaneTerms];
      if (rp & (1u << 28)) continue;
      const uint32_t pos = rp & 0xFFFFu;
      const int64_t gi = (ws.row_base + (ta + (pos >> 9) - ws.tb) * kTileRows + (pos & 511u)) * kLaneTerms +
                         (w0 & (kLaneTerms - 1));
      rs.raw[w0 / kLaneTerms][w0 & (kLaneTerms - 1)] =
          (gi >= ws.g_lo && gi < ws.g_hi) ? (uint64_t)__ldg(reinterpret_cast<const unsigned long long *>(p.x) + gi)
                                          : kNegZero;
    }
    __syncwarp();
    WR0(r, 31);
    for (int q0 = 0; q0 < nfetch; q0 += 2) {
      // lanes 0..15 row q0, 16..31 row q0 + 1; both binades each
      const int q = q0 + (lane >> 4), jj = lane & (kLaneTerms - 1);
      const uint32_t rp = q < nfetch ? rs.rawpos[q] : 0u;
      const bool has = (rp & (1u << 16)) != 0;
      const uint64_t t = has ? rs.raw[q][jj] : 0ull;
      const uint32_t E = has ? (rp >> 17) & 0x7FFu : 1023u;
      const uint32_t hi = (uint32_t)(t >> 32), Et = (hi >> 20) & 0x7FFu;
      uint32_t ta_, tb_;
      uint64_t Pa = term_mag_halfup(hi, (uint32_t)t, 64 - (int)E, ta_);
      uint64_t Pb = term_mag_halfup(hi, (uint32_t)t, 63 - (int)E, tb_);
      const uint32_t bada = __ballot_sync(kFull, ta_ == 0u || Et >= E);
      const uint32_t badb = __ballot_sync(kFull, tb_ == 0u || Et >= E + 1u);
#pragma unroll
      for (int o = 1; o < kLaneTerms; o <<= 1) {
        const uint64_t va = __shfl_up_sync(kFull, Pa, o, kLaneTerms), vb = __shfl_up_sync(kFull, Pb, o, kLaneTerms);
        if (jj >= o) {
          Pa += va;
          Pb += vb;
        }
      }
      if (has) {
        rs.raw[q][kLaneTerms + jj] = Pa;
        rs.raw[q][2 * kLaneTerms + jj] = Pb;
        if (jj == 0) {
          const uint32_t ma = (bada >> (lane & 16)) & 0xFFFFu, mb = (badb >> (lane & 16)) & 0xFFFFu;
          rs.rawlim[q] = (ma ? (uint32_t)(__ffs(ma) - 1) : (uint32_t)kLaneTerms) |
                         ((mb ? (uint32_t)(__ffs(mb) - 1) : (uint32_t)kLaneTerms) << 5);
        }
      }
    }
    WR0(r, 32);
    // ---- hand the slot over
    if (lane == 0) {
      rs.nsteps = over ? -1 : nsteps;
      rs.fail = ok ? 0 : 1;
      sm.wuse_p[pw] = use + 1;
    }
    __syncwarp();
    WRT(r, 1);
    if (lane == 0) mbar_arrive(&sm.wfull[pw]);
    // after a failure the later ranges are handed over failed, without waiting
    if (!ok) failed_all = true;
  }
}

// The in-order warp: the slots of one sum in range order, their steps
// applied to the exact running value S.  Returns S (NaN if a header never
// came or a slot was not handed over in time).
__device__ __noinline__ uint64_t walk_serial(const Params &p, Smem &sm, RangeSlot *slots, const WalkSum &ws,
                                             int nranges, uint64_t S) {
  const int lane = threadIdx.x & 31;
  bool failed = false;
  uint32_t nrun = 0, n_rounds = 0, n_dadds = 0;
  uint64_t cy_serial = 0, cy_raw = 0;
  for (int r = 0; r < nranges; r++) {
    const int pw = r % kWarps;
    RangeSlot &rs = slots[pw];
    const uint32_t use = sm.wuse_c[pw];
    const uint64_t c0 = clock64();
    const bool got = mbar_wait_bounded(&sm.wfull[pw], use & 1u, 8 * p.wait_ns);
    const uint64_t c1 = clock64();
    WRT(r, 2);
    if (!got || rs.fail) failed = true;
    const int64_t ta = ws.tb + range_start(r);
    if (got && !failed) {
      const int ns = rs.nsteps;
      if (ns < 0) {
        // the steps did not fit: the range's terms one by one
        if (lane == 0) stat_add(sm, S_RANGE_X, 1);
        int64_t a, b;
        clip(ws, ta, 0, (uint32_t)min(range_start(r + 1) - range_start(r), ws.te - ta) * kTileTerms, a, b);
        S = raw_from_x(p, sm, S, a, b);
      }
      for (int i = 0; i < ns; i++) {
        const Step st = rs.steps[i];
        const uint32_t kind = (uint32_t)(st.meta & 3u);
#ifdef SEQSUM_PROFILE
        const uint64_t t_seg = clock64();
#endif
        const uint32_t eb = (uint32_t)(st.meta >> 2) & 0x7FFu;
        const uint32_t from = (uint32_t)(st.meta >> 23) & 0xFFFFu, to = (uint32_t)(st.meta >> 39) & 0xFFFFu;
        if (lane == 0) (void)SQ_OK(p, from < to, 5, ((int64_t)from << 16) | to);
        bool done = false;
        const uint64_t m0 = (S & kFracMask) | kHidden;
        if (kind == ST_RUN && ((st.meta >> 56) & 1u) && (S >> 52) == eb && m0 + (uint64_t)st.inc <= (uint64_t)kTwo53) {
          // a plain run on a positive S of its binade: the count grows by inc
          S += (uint64_t)st.inc;
          done = true;
          nrun++;
        } else if (kind == ST_RUN) {
          Run q;
          q.inc = st.inc;
          q.lo = st.lo;
          q.hi = st.hi;
          q.d = (int32_t)((st.meta >> 13) & 3u) - 1;
          q.flags = (uint32_t)(st.meta >> 15) & 0xFFu;
          uint64_t nb = S;
          if (run_apply(nb, q, (int)eb - 1023) == APPLY_OK) {
            S = nb;
            done = true;
          } else if (lane == 0) {
            stat_add(sm, S_RUN_REJECTED, 1);
          }
          nrun++;
        } else if ((kind == ST_RAW || kind == ST_RAW2) && st.inc < kRangeRaw) {
          const uint64_t *data = rs.raw[st.inc];
          if (kind == ST_RAW) {
            S = row_dadd(sm, S, lane < kLaneTerms ? data[lane] : kNegZero, 0, kLaneTerms);
          } else {
            const uint64_t t_in = clock64();
            S = raw2_row(sm, S, data, rs.rawlim[st.inc], eb, (st.meta >> 15) & 1u, n_rounds, n_dadds);
            cy_raw += clock64() - t_in;
          }
          done = true;
        }
        if (!done) {
          // read from x: a refused composite, a region without items, a raw row beyond the fetched ones
          const int64_t r0 = ws.row_base + (ta + (from >> 9) - ws.tb) * kTileRows + (from & 511u);
          const int64_t r1 = ws.row_base + (ta + (to >> 9) - ws.tb) * kTileRows + (to & 511u);
          const int64_t a = max(r0 * kLaneTerms, ws.g_lo), b = min(r1 * kLaneTerms, ws.g_hi);
          if (b > a) S = raw_from_x(p, sm, S, a, b);
        }
#ifdef SEQSUM_PROFILE
        if (lane == 0) {
          // the walk's steps: kind and cycles (one in-order warp: a plain count)
          const uint64_t cy = clock64() - t_seg;
          const unsigned long long slot = sm.prof_n++;
          p.dbg[4095] = slot + 1;
          const uint64_t info = kind == ST_RAW2 ? (uint64_t)sm.prof_i | ((uint64_t)eb << 31) : (uint64_t)i;
          if (slot < 1000) p.dbg[4096 - 1000 - 1 + slot] = ((uint64_t)kind << 60) | ((info & 0xFFFFFFFFFFull) << 20) | (cy & 0xFFFFF);
        }
#endif
      }
    }
    WRT(r, 3);
    cy_serial += clock64() - c1;
    if (lane == 0) sm.wuse_c[pw] = use + 1;
    __syncwarp();
    if (got && lane == 0) mbar_arrive(&sm.wempty[pw]);
    if (!got) break;   // the slot may still be written: stop using them
  }
  if (lane == 0) {
    stat_add(sm, S_WALK_SEGMENTS, nrun);
    stat_add(sm, S_WALK_BATCHES, (unsigned long long)nranges);
    stat_add(sm, S_CY_WALK_SERIAL, cy_serial);
    stat_add(sm, S_CY_WALK_RAW, cy_raw);
    stat_add(sm, S_RAW_ROUNDS, n_rounds);
    stat_add(sm, S_TERMS_DADD, n_dadds);
  }
  return failed ? 0x7FF8000000000000ull : S;
}

// Walks the tiles [ws.tb, ws.te) of one sum from the start value Sb.
__device__ __noinline__ uint64_t walk_sum(const Params &p, Smem &sm, unsigned char *dyn, const WalkSum &ws,
                                         uint64_t Sb) {
  const int w = threadIdx.x >> 5;
  RangeSlot *slots = reinterpret_cast<RangeSlot *>(dyn);
  const int nranges = range_count(ws.te - ws.tb);
  if (w < kWarps) {
    walk_producer(p, sm, slots[w], ws, nranges, w, sm.tag);
  } else {
    const uint64_t S = walk_serial(p, sm, slots, ws, nranges, Sb);
    if ((threadIdx.x & 31) == 0) sm.S = S;
  }
  __syncthreads();
  const uint64_t out = sm.S;
  __syncthreads();
  return out;
}

__device__ __noinline__ void walk_loop(const Params &p, Smem &sm, unsigned char *dyn, int64_t ntiles) {
  const int tid = threadIdx.x;
  if (tid == 0) sm.prof_n = 0;
  if (tid < kWarps) {
    mbar_init(&sm.wfull[tid], 1);
    mbar_init(&sm.wempty[tid], 1);
    sm.wuse_p[tid] = 0;
    sm.wuse_c[tid] = 0;
  }
  fence_mbar_init();
  __syncthreads();
  while (true) {
    if (tid == 0) sm.wk = p.offsets ? (int)atomicAdd(&p.ctr[C_SUMTICKET], 1u) : (sm.wk == 0 ? 0 : 1);
    __syncthreads();
    const int j = sm.wk;
    if (j >= p.nsums) break;
    WalkSum ws;
    double s0;
    int k = 0;
    if (p.offsets) {
      k = p.order[j];
      ws.tb = p.tile_begin[j];
      ws.te = p.tile_begin[j + 1];
      ws.g_lo = p.offsets[k];
      ws.g_hi = p.offsets[k + 1];
      ws.row_base = ws.g_lo >> 4;
      s0 = p.s0s[k];
    } else {
      ws.tb = 0;
      ws.te = ntiles;
      ws.g_lo = 0;
      ws.g_hi = p.n;
      ws.row_base = 0;
      s0 = p.s0;
    }
    const uint64_t S = walk_sum(p, sm, dyn, ws, dbits(s0));
    if (tid == 0) {
      p.outs[k] = bitsd(S);
      if (!p.offsets) sm.wk = 1;
    }
    __syncthreads();
  }
}

// ------------------------------------------------------------------ the kernel
__global__ void __launch_bounds__(kBlockThreads, 2) seqsum_kernel(const Params p, const __grid_constant__ CUtensorMap tmap) {
  extern __shared__ unsigned char dyn_raw[];
  unsigned char *dyn = reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(dyn_raw) + 1023) & ~uintptr_t(1023));
  __shared__ Smem sm;
  const int tid = threadIdx.x;
  for (int i = tid; i < kBlockWarps * S_ACCUM_END; i += kBlockThreads) (&sm.stat[0][0])[i] = 0;
  if (tid == 0) {
    sm.scan_stop = 0;
    sm.role = (int)atomicAdd(&p.ctr[C_ROLE], 1u);
    uint32_t smid;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
    // the walker and the scanner are latency-bound: a streaming CTA that finds
    // itself on their SM leaves it to them.  Both roles are taken by CTAs
    // already running, which write their SM right after taking the role; a
    // streaming CTA waits for both words (bounded: past the limit it streams).
    // (A small grid keeps every CTA streaming: there the others may be too few.)
    if (sm.role == 0) atomicExch(&p.ctr[C_WALK_SM], smid + 1);
    if (sm.role == p.nwalkers) atomicExch(&p.ctr[C_SCAN_SM], smid + 1);

    sm.alone = 0;
    if (sm.role > p.nwalkers && gridDim.x >= 64) {
      uint32_t ws = 0, ss = 0;
      const uint64_t t0 = gtimer();
      for (;;) {
        ws = ld_relaxed_u32(&p.ctr[C_WALK_SM]);
        ss = ld_relaxed_u32(&p.ctr[C_SCAN_SM]);
        if ((ws != 0u && ss != 0u) || gtimer() - t0 > 20000ull) break;
        __nanosleep(64);
      }
      sm.alone = ws == smid + 1 || ss == smid + 1;
      if (sm.alone) sm.stat[kWarps][S_ALONE] += 1;
#ifdef SEQSUM_PROFILE
      if (sm.alone) p.dbg[2392 + (ws == smid + 1 ? 0 : 1)] = smid + 1;
#endif
    }
#ifdef SEQSUM_PROFILE
    if (sm.role == 0) p.dbg[2390] = smid + 1;
    if (sm.role == p.nwalkers) p.dbg[2391] = smid + 1;
#endif
    const uint32_t e = ld_relaxed_u32(&p.ctr[C_EPOCH]);
    sm.tag = e == 0 ? 1u : e;
    sm.ntiles = p.offsets ? (int64_t)ld_relaxed_u32(&p.ctr[C_NTILES]) : p.ntiles;
    sm.fail = ld_relaxed_u32(&p.ctr[C_SKIP]) != 0u && p.offsets;
    sm.wk = 0;
    if (sm.role == 0) p.stats[S_T_START] = gtimer();
  }
  __syncthreads();
  const uint32_t tag = sm.tag;
  const int64_t ntiles = sm.ntiles;
  const bool skip = sm.fail;
  __syncthreads();
  if (!skip) {
    // roles in the order the CTAs start: the walkers, the scanner, then the
    // streaming CTAs (every waiting role is held by a CTA already running)
    if (sm.role < p.nwalkers) {
#ifdef SEQSUM_PROFILE
      if (tid == 0 && sm.role == 0) p.dbg[2096] = gtimer();
#endif
      walk_loop(p, sm, dyn, ntiles);
      if (tid == 0) atomicMax(&p.stats[S_T_WALK_END], (unsigned long long)gtimer());
#ifdef SEQSUM_PROFILE
      if (tid == 0 && sm.role == 0) p.dbg[2097] = gtimer();
#endif
    } else if (sm.role == p.nwalkers) {
      if (p.planned) scan_cta<true>(p, sm, ntiles);
      else scan_cta<false>(p, sm, ntiles);
    } else if (!sm.alone) {
      stream_cta(p, sm, dyn, &tmap, ntiles);
      if (tid == 0 && sm.t_stream_end) atomicMax(&p.stats[S_T_STREAM_END], (unsigned long long)sm.t_stream_end);
    }
  }
  __syncthreads();
  if (tid < S_ACCUM_END) {
    unsigned long long v = 0;
    for (int k = 0; k < kBlockWarps; k++) v += sm.stat[k][tid];
    if (v) atomicAdd(&p.stats[tid], v);
  }
  if (tid == 0) {
    __threadfence();
    const uint32_t done = atomicAdd(&p.ctr[C_EXIT], 1u);
    sm.count = (done == gridDim.x - 1) ? 1 : 0;
  }
  __syncthreads();
  if (sm.count) {
    // the last CTA: counters back to zero and the next call's tag; when the
    // tag wraps, every tagged word is cleared first so that no stale word can
    // carry a current tag
    __threadfence();
    const uint32_t next = tag + 1;
    if (next > 255u) {
      for (int64_t i = tid; i < p.cap_tiles; i += kBlockThreads) {
        p.status[i] = make_uint4(0, 0, 0, 0);
        p.prec_ws[i * kPrecWords] = make_uint4(0, 0, 0, 0);
        if (p.conf) p.conf[i] = 0;
        if (p.redo) p.redo[i] = 0;
        Rec z;
        z.w[0] = z.w[1] = z.w[2] = z.w[3] = 0;
        st_rec(&p.hdr[i], z);
      }
      __threadfence();
      __syncthreads();
    }
    if (tid == 0) {
      p.ctr[C_TICKET] = 0;
      p.ctr[C_ROLE] = 0;
      p.ctr[C_SUMTICKET] = 0;
      p.ctr[C_WALK_SM] = 0;
      p.ctr[C_SCAN_SM] = 0;
      p.ctr[C_REDO_RES] = 0;
      p.ctr[C_SCAN_FIN] = 0;
      p.ctr[C_EPOCH] = next > 255u ? 1u : next;
      __threadfence();
      p.ctr[C_EXIT] = 0;
    }
  }
}

// A sum's tiles: its rows of 16 terms (the first and the last may be partial)
// in tiles of kTileRows.
__device__ __forceinline__ int64_t sum_tiles(const Params &p, int k) {
  const int64_t a = p.offsets[k], b = p.offsets[k + 1];
  if (b <= a) return 0;
  const int64_t rows = ((b + 15) >> 4) - (a >> 4);
  return (rows + kTileRows - 1) / kTileRows;
}
// The size class that orders the sums: the bit length of the tile count.
constexpr int kSizeClasses = 65;
__device__ __forceinline__ int size_class(int64_t nt) { return 64 - __clzll((long long)nt); }

// The batched calls' set-up (one CTA): checks the offsets, puts the sums in
// the order the kernel takes them and writes tile_begin by that order.  The
// order is by size class, smaller first, and by index within a class: a small
// sum's walk costs about the same time whatever its length, so small sums go
// first, where their walks overlap the streaming of the larger ones, and the
// walk that ends last is a large sum's, which keeps pace with its tiles.  On
// bad offsets or too many tiles every output is NaN and the main kernel does
// nothing.
__global__ void __launch_bounds__(kThreads) setup_kernel(const Params p) {
  __shared__ int bad;
  __shared__ int64_t carry;
  __shared__ int64_t wsum[kWarps];
  __shared__ int cbase[kSizeClasses];          // the next position of each class
  __shared__ int ccount[kWarps][kSizeClasses]; // a chunk's sums of each class, per warp
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  if (tid == 0) {
    bad = 0;
    carry = 0;
  }
  for (int c = tid; c < kSizeClasses; c += kThreads) cbase[c] = 0;
  __syncthreads();
  for (int k = tid; k <= p.nsums; k += kThreads) {
    const int64_t o = p.offsets[k];
    if (o < 0 || o > p.x_len) bad = 1;
    if (k > 0 && p.offsets[k - 1] > o) bad = 1;
  }
  __syncthreads();
  if (!bad) {
    // the order: a counting sort by size class, stable (ranks within a warp
    // from match masks, then the warps of the chunk in turn)
    for (int k = tid; k < p.nsums; k += kThreads) atomicAdd(&cbase[size_class(sum_tiles(p, k))], 1);
    __syncthreads();
    if (tid == 0) {
      int run = 0;
      for (int c = 0; c < kSizeClasses; c++) {
        const int n = cbase[c];
        cbase[c] = run;
        run += n;
      }
    }
    __syncthreads();
    for (int k0 = 0; k0 < p.nsums; k0 += kThreads) {
      const int k = k0 + tid;
      for (int i = tid; i < kWarps * kSizeClasses; i += kThreads) (&ccount[0][0])[i] = 0;
      __syncthreads();
      const int c = k < p.nsums ? size_class(sum_tiles(p, k)) : -1;
      const uint32_t peers = __match_any_sync(kFull, c);
      const int rank = __popc(peers & ((1u << lane) - 1u));
      if (c >= 0 && rank == 0) ccount[w][c] = __popc(peers);
      __syncthreads();
      if (c >= 0) {
        int pos = cbase[c] + rank;
        for (int j = 0; j < w; j++) pos += ccount[j][c];
        p.order[pos] = k;
      }
      __syncthreads();
      for (int cc = tid; cc < kSizeClasses; cc += kThreads) {
        int n = 0;
        for (int j = 0; j < kWarps; j++) n += ccount[j][cc];
        cbase[cc] += n;
      }
      __syncthreads();
    }
    // tile_begin by position
    for (int j0 = 0; j0 < p.nsums; j0 += kThreads) {
      const int j = j0 + tid;
      const int64_t nt = j < p.nsums ? sum_tiles(p, p.order[j]) : 0;
      int64_t inc = nt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int64_t q = __shfl_up_sync(kFull, inc, o);
        if (lane >= o) inc += q;
      }
      if (lane == 31) wsum[w] = inc;
      __syncthreads();
      int64_t base = carry;
      for (int i = 0; i < w; i++) base += wsum[i];
      if (j < p.nsums) p.tile_begin[j] = base + inc - nt;
      __syncthreads();
      if (tid == 0) {
        int64_t tot = 0;
        for (int i = 0; i < kWarps; i++) tot += wsum[i];
        carry += tot;
      }
      __syncthreads();
    }
  }
  __syncthreads();
  if (tid == 0) {
    const int64_t total = carry;
    uint32_t err = 0;
    if (bad) err = ERR_BAD_OFFSETS;
    else if (total > p.cap_tiles || total > 0x7FFFFFFF) err = ERR_CAPACITY;
    p.tile_begin[p.nsums] = total;
    p.ctr[C_NTILES] = err ? 0u : (uint32_t)total;
    p.ctr[C_SKIP] = err ? 1u : 0u;
    if (err) atomicOr(&p.ctr[C_ERR], err);
  }
  __syncthreads();
  if (bad || carry > p.cap_tiles) {
    for (int k = tid; k < p.nsums; k += kThreads) p.outs[k] = __longlong_as_double(0x7FF8000000000000ll);
  }
}

int kernel_blocks_per_sm() {
  int n = 0;
  cudaFuncSetAttribute(seqsum_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kDynSmem);
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, seqsum_kernel, kBlockThreads, kDynSmem);
  return n > 0 ? n : 1;
}

cudaError_t launch_seqsum(const Params &p, const CUtensorMap *tmap, int grid, cudaStream_t st) {
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(seqsum_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kDynSmem);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  seqsum_kernel<<<grid, kBlockThreads, kDynSmem, st>>>(p, *tmap);
  return cudaGetLastError();
}

cudaError_t launch_setup(const Params &p, cudaStream_t st) {
  setup_kernel<<<1, kThreads, 0, st>>>(p);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ interleaved sums (strided)
// The stride sums of an interleaved plane (sum k: x[k], x[k + stride], ...)
// laid out one after another, so the batched kernel takes them as stride
// sums of n terms each; offsets[k] = k n.  A copy only: no term changes.
__global__ void __launch_bounds__(kThreads) deinterleave_kernel(const double *x, int64_t n, int stride,
                                                                double *planes, int64_t *offsets) {
  for (int64_t i = (int64_t)blockIdx.x * kThreads + threadIdx.x; i < n; i += (int64_t)gridDim.x * kThreads)
    for (int k = 0; k < stride; k++) planes[(int64_t)k * n + i] = x[i * stride + k];
  if (blockIdx.x == 0 && threadIdx.x <= stride) offsets[threadIdx.x] = (int64_t)threadIdx.x * n;
}

// The frame score's epilogue: each sum's mean as a float, (float)(sum / n),
// with the correctly rounded division and conversion the host loop uses.
__global__ void mean_kernel(const double *outs, int stride, int64_t n, float *means) {
  const int k = threadIdx.x;
  if (k < stride) means[k] = __double2float_rn(__ddiv_rn(outs[k], (double)n));
}

cudaError_t launch_deinterleave(const double *x, int64_t n, int stride, double *planes, int64_t *offsets,
                                cudaStream_t st) {
  int64_t blocks = (n + kThreads - 1) / kThreads;
  if (blocks > 4096) blocks = 4096;
  if (blocks < 1) blocks = 1;
  deinterleave_kernel<<<(int)blocks, kThreads, 0, st>>>(x, n, stride, planes, offsets);
  return cudaGetLastError();
}

cudaError_t launch_mean(const double *outs, int stride, int64_t n, float *means, cudaStream_t st) {
  mean_kernel<<<1, 64, 0, st>>>(outs, stride, n, means);
  return cudaGetLastError();
}

}  // namespace sq

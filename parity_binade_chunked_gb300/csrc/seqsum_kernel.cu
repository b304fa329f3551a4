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
__device__ __forceinline__ uint4 ld_vol_v4(const uint4 *p) {
  uint4 v;
  asm volatile("ld.volatile.global.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p)
               : "memory");
  return v;
}
__device__ __forceinline__ void st_vol_v4(uint4 *p, uint4 v) {
  asm volatile("st.volatile.global.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}
__device__ __forceinline__ void ld_vol_v2(const void *p, uint64_t &a, uint64_t &b) {
  asm volatile("ld.volatile.global.v2.u64 {%0, %1}, [%2];" : "=l"(a), "=l"(b) : "l"(p) : "memory");
}
__device__ __forceinline__ void st_vol_v2(void *p, uint64_t a, uint64_t b) {
  asm volatile("st.volatile.global.v2.u64 [%0], {%1, %2};" ::"l"(p), "l"(a), "l"(b) : "memory");
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
struct Smem {
  uint64_t full[kStages];            // TMA mbarriers, one per stage
  int64_t st_tile[kStages];          // the stage's tile (-1: none)
  int64_t st_geo[kStages][5];        // row0, g_lo, g_hi, t_first, sum
  uint32_t st_flags[kStages];        // bit 0: the tile came by TMA
  float wfs[kWarps], wfa[kWarps];    // warp totals of the plan sums
  DF excl;                           // the prefix before the tile
  float excl_abs;
  int32_t web[kWarps];
  int32_t wok[kWarps];
  uint32_t wslots[kWarps];
  long long wred[kWarps][3];
  uint32_t wfl_and[kWarps], wfl_or[kWarps];
  int role;
  uint32_t tag;
  int64_t ntiles;
  int fail;
  int broken;                        // this streaming CTA stopped using TMA after a timeout
  int count;
  int nseg;
  int wk;
  uint64_t S;                        // the walk's running value (bits)
  uint64_t t_stream_end;
  // walker block scan
  Run wtot[kWarps];
  int wtot_head[kWarps];
  int wstart[kWarps];
  int whead0[kWarps + 1];
  uint32_t wtails[kWarps];
  unsigned long long stat[S_ACCUM_END];
};

__device__ __forceinline__ void stat_add(Smem &sm, int which, unsigned long long v) {
  atomicAdd(&sm.stat[which], v);
}

// ------------------------------------------------------------------ tile geometry
// Tiles of a sum cover whole rows of 16 terms of x, starting at the row that
// holds the sum's first term; terms of a row outside the sum are masked to
// -0, the identity of binary64 addition.
struct Geo {
  int64_t row0, g_lo, g_hi, t_first;
  int32_t sum;
};

__device__ __forceinline__ Geo tile_geo(const Params &p, int64_t t) {
  Geo g;
  if (!p.offsets) {
    g.row0 = t * kTileRows;
    g.g_lo = 0;
    g.g_hi = p.n;
    g.t_first = 0;
    g.sum = 0;
    return g;
  }
  // the sum k with tile_begin[k] <= t < tile_begin[k+1] (the last such k: empty sums share a start)
  int lo = 0, hi = p.nsums;   // invariant: tile_begin[lo] <= t < tile_begin[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(&p.tile_begin[mid]) <= t) lo = mid;
    else hi = mid;
  }
  const int64_t off = __ldg(&p.offsets[lo]);
  g.t_first = __ldg(&p.tile_begin[lo]);
  g.row0 = (off >> 4) + (t - g.t_first) * kTileRows;
  g.g_lo = off;
  g.g_hi = __ldg(&p.offsets[lo + 1]);
  g.sum = lo;
  return g;
}

// ------------------------------------------------------------------ the plan's look-back
// status[t] = {hi, lo, abs, tag << 8 | flag} (flag 1: the tile's own sum,
// 2: the inclusive prefix through the tile).  Run by one warp.  Returns the
// exclusive prefix of tile t (not the first of its sum) and publishes t's
// inclusive prefix.
__device__ __noinline__ void lookback(const Params &p, int64_t t, int64_t t_first, DF agg, float agg_abs, uint32_t tag,
                                      DF &excl, float &excl_abs) {
  const int lane = threadIdx.x & 31;
  if (lane == 0)
    st_vol_v4(&p.status[t], make_uint4(__float_as_uint(agg.hi), __float_as_uint(agg.lo), __float_as_uint(agg_abs),
                                       (tag << 8) | 1u));
  float acc = 0.0f, acc_abs = 0.0f;
  DF incl = DF{0.0f, 0.0f};
  int64_t base = t - 1;
  const uint64_t t0 = gtimer();
  bool timed_out = false;
  while (true) {
    const int64_t idx = base - lane;
    const bool inrange = idx >= t_first;
    uint4 st = make_uint4(0, 0, 0, 0);
    int first_incl = 32;
    uint32_t spin = 0;
    while (true) {
      if (inrange) st = ld_vol_v4(&p.status[idx]);
      const bool valid = inrange && (st.w >> 8) == tag && (st.w & 3u) != 0u;
      const bool inc = valid && (st.w & 3u) == 2u;
      const uint32_t bi = __ballot_sync(kFull, inc);
      const uint32_t bv = __ballot_sync(kFull, valid);
      first_incl = bi ? __ffs(bi) - 1 : 32;
      const uint32_t need = first_incl >= 31 ? kFull : ((2u << first_incl) - 1u);
      if ((bv & need) == need) break;
      // the decision to give up is the warp's (a lane alone must not leave the ballots)
      if (__any_sync(kFull, (++spin & 63u) == 0u && gtimer() - t0 > p.wait_ns)) {
        timed_out = true;
        break;
      }
      __nanosleep(32);
    }
    if (timed_out) {
      if (lane == 0) note_timeout(p, ERR_PLAN_TIMEOUT, 1, (uint32_t)t, (uint32_t)base);
      break;
    }
    // the tiles' own sums before the first inclusive prefix, and every abs up to it
    float v = (lane < first_incl) ? __fadd_rn(__uint_as_float(st.x), __uint_as_float(st.y)) : 0.0f;
    float va = (lane <= first_incl) ? __uint_as_float(st.z) : 0.0f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      v += __shfl_xor_sync(kFull, v, o);
      va += __shfl_xor_sync(kFull, va, o);
    }
    acc += v;
    acc_abs += va;
    if (first_incl < 32) {
      incl.hi = __uint_as_float(__shfl_sync(kFull, st.x, first_incl));
      incl.lo = __uint_as_float(__shfl_sync(kFull, st.y, first_incl));
      break;
    }
    base -= 32;
  }
  excl = df_add(incl, DF{acc, 0.0f});
  excl_abs = acc_abs;
  if (lane == 0) {
    const DF in = df_add(excl, agg);
    st_vol_v4(&p.status[t], make_uint4(__float_as_uint(in.hi), __float_as_uint(in.lo),
                                       __float_as_uint(excl_abs + agg_abs), (tag << 8) | 2u));
  }
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

// ------------------------------------------------------------------ one tile of a streaming CTA
__device__ __forceinline__ int float_binade(float f) { return (int)((__float_as_uint(f) >> 23) & 0xFFu); }

__device__ __forceinline__ void process_tile(const Params &p, Smem &sm, const uint64_t (&v)[kLaneTerms], int64_t t,
                                          const Geo &g, uint32_t tag) {
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;

  // ---- plan sums of the row
  float fs = 0.0f, fa = 0.0f;
  uint32_t mx = 0;
#pragma unroll
  for (int j = 0; j < kLaneTerms; j++) {
    const uint32_t hi = (uint32_t)(v[j] >> 32);
    mx = max(mx, hi);
    const float f = __double2float_rn(bitsd(v[j]));
    fs = __fadd_rn(fs, f);
    fa = __fadd_rn(fa, fabsf(f));
  }
  // warp inclusive scans
  float is = fs, ia = fa;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float a = __shfl_up_sync(kFull, is, o), b = __shfl_up_sync(kFull, ia, o);
    if (lane >= o) {
      is = __fadd_rn(is, a);
      ia = __fadd_rn(ia, b);
    }
  }
  if (lane == 31) {
    sm.wfs[w] = is;
    sm.wfa[w] = ia;
  }
  float xs = __shfl_up_sync(kFull, is, 1), xa = __shfl_up_sync(kFull, ia, 1);
  if (lane == 0) xs = xa = 0.0f;
  __syncthreads();
  float bs = 0.0f, ba = 0.0f;
  for (int k = 0; k < w; k++) {
    bs = __fadd_rn(bs, sm.wfs[k]);
    ba = __fadd_rn(ba, sm.wfa[k]);
  }
  xs = __fadd_rn(bs, xs);
  xa = __fadd_rn(ba, xa);

  // ---- the prefix before the tile
  if (w == 0) {
    DF agg = DF{0.0f, 0.0f};
    float agg_abs = 0.0f;
    for (int k = 0; k < kWarps; k++) {
      agg = df_add(agg, DF{sm.wfs[k], 0.0f});
      agg_abs = __fadd_rn(agg_abs, sm.wfa[k]);
    }
    DF ex;
    float ex_abs;
    if (t == g.t_first) {
      ex = df_of_double(p.offsets ? p.s0s[g.sum] : p.s0);
      ex_abs = fabsf(ex.hi);
      if (lane == 0) {
        const DF in = df_add(ex, agg);
        st_vol_v4(&p.status[t], make_uint4(__float_as_uint(in.hi), __float_as_uint(in.lo),
                                           __float_as_uint(__fadd_rn(ex_abs, agg_abs)), (tag << 8) | 2u));
      }
    } else {
      lookback(p, t, g.t_first, agg, agg_abs, tag, ex, ex_abs);
    }
    if (lane == 0) {
      sm.excl = ex;
      sm.excl_abs = ex_abs;
    }
  }
  __syncthreads();

  // ---- the row's binade
  const DF ex = sm.excl;
  const float Pf = __fadd_rn(ex.hi, __fadd_rn(ex.lo, xs));
  const float A = __fadd_rn(__fadd_rn(sm.excl_abs, xa), fa);
  const float marg = __fadd_rn(__fmul_rn(A, 4.76837158203125e-7f /* 2^-21 */), 1e-30f);
  const float pos = __fmul_rn(0.5f, __fadd_rn(fa, fs)), neg = __fmul_rn(0.5f, __fsub_rn(fa, fs));
  const float lo_ = __fsub_rn(__fsub_rn(Pf, neg), marg), hi_ = __fadd_rn(__fadd_rn(Pf, pos), marg);
  int fb = 0;   // float biased exponent of the binade, 0: the row's range is not inside one binade
  if (lo_ > 0.0f) {
    const int a = float_binade(lo_), b = float_binade(hi_);
    if (a == b && a >= 1 && a <= 254) fb = a;
  } else if (hi_ < 0.0f) {
    const int a = float_binade(-hi_), b = float_binade(-lo_);
    if (a == b && a >= 1 && a <= 254) fb = a;
  }
  uint32_t eb = fb ? (uint32_t)(fb - 127 + 1023) : 0u;   // double biased exponent
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
  bool zero = false, allneg = false;
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

  // ---- one header, or a list of items
  const uint32_t key0 = __shfl_sync(kFull, key, 0);
  const bool same = __all_sync(kFull, !raw && !general && key == key0);
  if (lane == 0) {
    sm.wok[w] = same;
    sm.web[w] = (int32_t)key;
  }
  __syncthreads();
  bool fast = true;
  for (int k = 0; k < kWarps; k++) fast = fast && sm.wok[k] && sm.web[k] == sm.web[0];
  const uint32_t nraw = __popc(__ballot_sync(kFull, raw));
  const uint32_t ntie = __popc(__ballot_sync(kFull, general));
  if (lane == 0) {
    if (nraw) stat_add(sm, S_LANE_RAW, nraw);
    if (ntie) stat_add(sm, S_LANE_TIE, ntie);
  }

  if (fast) {
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
      sm.wred[w][0] = a;
      sm.wred[w][1] = b;
      sm.wred[w][2] = d;
      sm.wfl_and[w] = fand;
      sm.wfl_or[w] = fo;
    }
    __syncthreads();
    if (tid == 0) {
      Item h;
      h.r.inc = h.r.lo = h.r.hi = 0;
      h.r.d = 0;
      uint32_t fa2 = 0xFFu, fo2 = 0;
      for (int k = 0; k < kWarps; k++) {
        h.r.inc += sm.wred[k][0];
        h.r.lo += sm.wred[k][1];
        h.r.hi += sm.wred[k][2];
        fa2 &= sm.wfl_and[k];
        fo2 |= sm.wfl_or[k];
      }
      h.r.flags = fa2 | fo2;
      saturate(h.r);
      h.kind = K_RUN;
      h.eb = (uint32_t)sm.web[0];
      h.count = kTileTerms;
      h.start = 0;
      if (!(p.fault_mode == 1 && t == p.fault_arg)) st_rec_vol(&p.hdr[t], pack_item(h, tag));
    }
    return;
  }

  // ---- items: each warp's maximal runs of one binade, and raw rows
  const uint32_t pkey = __shfl_up_sync(kFull, key, 1);
  const bool praw = __shfl_up_sync(kFull, raw, 1);
  bool head = lane == 0 || raw || praw || key != pkey;
  int sstart = head ? lane : 0;
  Run s = r;
  bool hf = head;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const Run q = shfl_run_up(s, o);
    const bool qh = __shfl_up_sync(kFull, hf, o);
    const int qs = __shfl_up_sync(kFull, sstart, o);
    if (lane >= o) {
      if (!hf) s = run_compose(q, s);
      hf = hf || qh;
      sstart = max(sstart, qs);
    }
  }
  const bool nhead = __shfl_down_sync(kFull, head, 1);
  const bool tail = (lane == 31) || nhead;
  const uint32_t my = raw ? (uint32_t)kRawSlots : ((tail && !raw) ? 1u : 0u);
  uint32_t ex_sl = my;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t q = __shfl_up_sync(kFull, ex_sl, o);
    if (lane >= o) ex_sl += q;
  }
  if (lane == 31) sm.wslots[w] = ex_sl;
  ex_sl -= my;
  __syncthreads();
  uint32_t base = 0, total = 0;
  for (int k = 0; k < kWarps; k++) {
    if (k < w) base += sm.wslots[k];
    total += sm.wslots[k];
  }
  if (total > (uint32_t)kItemSlots) {
    if (tid == 0) {
      Item h;
      h.r = run_empty();
      h.kind = K_OVERFLOW;
      h.eb = 0;
      h.count = 0;
      h.start = 0;
      stat_add(sm, S_TILE_OVERFLOW, 1);
      if (!(p.fault_mode == 1 && t == p.fault_arg)) st_rec_vol(&p.hdr[t], pack_item(h, tag));
    }
    return;
  }
  Rec *area = p.items + t * kItemSlots;
  const uint32_t at = base + ex_sl;
  const uint32_t row_start = (uint32_t)(w * 32 + lane) * kLaneTerms;
  if (raw) {
    if (SQ_OK(p, at + kRawSlots <= (uint32_t)kItemSlots, 11, at)) {
      Item it;
      it.r = run_empty();
      it.kind = K_RAW;
      it.eb = 0;
      it.count = kLaneTerms;
      it.start = row_start;
      st_rec(&area[at], pack_item(it, 0));
      uint4 *dst = reinterpret_cast<uint4 *>(&area[at + 1]);
#pragma unroll
      for (int j = 0; j < kLaneTerms; j += 2)
        dst[j / 2] = make_uint4((uint32_t)v[j], (uint32_t)(v[j] >> 32), (uint32_t)v[j + 1], (uint32_t)(v[j + 1] >> 32));
    }
  } else if (tail) {
    if (SQ_OK(p, at < (uint32_t)kItemSlots, 12, at)) {
      Item it;
      it.r = s;
      it.kind = K_RUN;
      it.eb = key;
      it.count = (uint32_t)(lane - sstart + 1) * kLaneTerms;
      it.start = (uint32_t)(w * 32 + sstart) * kLaneTerms;
      st_rec(&area[at], pack_item(it, 0));
    }
  }
  __threadfence();   // each writer's items before the header that publishes them
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    Item h;
    h.r = run_empty();
    h.kind = K_COMPLEX;
    h.eb = 0;
    h.count = total;
    h.start = 0;
    stat_add(sm, S_TILE_COMPLEX, 1);
    if (!(p.fault_mode == 1 && t == p.fault_arg)) st_rec_vol(&p.hdr[t], pack_item(h, tag));
  }
}

// ------------------------------------------------------------------ the streaming loop
__device__ __forceinline__ void load_row(const Params &p, const unsigned char *stage, bool lane_tma, int64_t row,
                                         const Geo &g, bool full, uint64_t (&v)[kLaneTerms]) {
  const int tid = threadIdx.x;
  if (lane_tma) {
    const unsigned char *rp = stage + tid * 128;
    const int sw = tid & 7;
#pragma unroll
    for (int q = 0; q < 8; q++) {
      const uint4 d = *reinterpret_cast<const uint4 *>(rp + ((q ^ sw) << 4));
      v[2 * q] = ((uint64_t)d.y << 32) | d.x;
      v[2 * q + 1] = ((uint64_t)d.w << 32) | d.z;
    }
  } else {
    const int64_t g0 = row * kLaneTerms;
    const unsigned long long *xp = reinterpret_cast<const unsigned long long *>(p.x);
#pragma unroll
    for (int j = 0; j < kLaneTerms; j++) {
      const int64_t gi = g0 + j;
      v[j] = (gi >= g.g_lo && gi < g.g_hi) ? (uint64_t)__ldg(xp + gi) : kNegZero;
    }
    return;
  }
  if (!full) {
    const int64_t g0 = row * kLaneTerms;
#pragma unroll
    for (int j = 0; j < kLaneTerms; j++) {
      const int64_t gi = g0 + j;
      if (gi < g.g_lo || gi >= g.g_hi) v[j] = kNegZero;
    }
  }
}

// Takes the next ticket for stage s and starts its copy (thread 0).
__device__ __forceinline__ void refill(const Params &p, Smem &sm, unsigned char *stages, const CUtensorMap *tmap,
                                       int s, int64_t ntiles) {
  const int64_t t = sm.broken ? ntiles : (int64_t)atomicAdd(&p.ctr[C_TICKET], 1u);
  if (t >= ntiles) {
    sm.st_tile[s] = -1;
    return;
  }
  const Geo g = tile_geo(p, t);
  sm.st_tile[s] = t;
  sm.st_geo[s][0] = g.row0;
  sm.st_geo[s][1] = g.g_lo;
  sm.st_geo[s][2] = g.g_hi;
  sm.st_geo[s][3] = g.t_first;
  sm.st_geo[s][4] = g.sum;
  const bool tma = p.tma_rows > 0 && g.row0 < p.tma_rows;
  sm.st_flags[s] = tma ? 1u : 0u;
  if (tma) {
    mbar_expect_tx(&sm.full[s], kStageBytes);
    tma_load_2d(stages + s * kStageBytes, tmap, &sm.full[s], 0, (int32_t)g.row0);
  } else {
    mbar_arrive(&sm.full[s]);
  }
}

__device__ __noinline__ void stream_loop(const Params &p, Smem &sm, unsigned char *stages, const CUtensorMap *tmap,
                                         int64_t ntiles, uint32_t tag) {
  const int tid = threadIdx.x;
  if (tid == 0) {
    for (int s = 0; s < kStages; s++) mbar_init(&sm.full[s], 1);
    fence_mbar_init();
    sm.broken = 0;
    sm.t_stream_end = 0;
    for (int s = 0; s < kStages; s++) refill(p, sm, stages, tmap, s, ntiles);
  }
  __syncthreads();
  for (uint32_t it = 0;; it++) {
    const int s = (int)(it % kStages);
    const uint32_t ph = (it / kStages) & 1u;
    const int64_t t = sm.st_tile[s];
    if (t < 0) break;
    Geo g;
    g.row0 = sm.st_geo[s][0];
    g.g_lo = sm.st_geo[s][1];
    g.g_hi = sm.st_geo[s][2];
    g.t_first = sm.st_geo[s][3];
    g.sum = (int32_t)sm.st_geo[s][4];
    const bool tma = sm.st_flags[s] & 1u;
    // wait for the copy (bounded; one thread decides for the CTA)
    if (tid == 0) {
      const uint64_t t0 = gtimer();
      uint32_t spin = 0;
      int ok = 1;
      while (!mbar_try_wait(&sm.full[s], ph)) {
        if ((++spin & 255u) == 0u && gtimer() - t0 > p.wait_ns) {
          ok = 0;
          break;
        }
      }
      if (!ok) {
        // the copy may still land: wait once more (bounded) so that it cannot
        // write into the stage after it is reused; the tile is read from x
        note_timeout(p, ERR_TMA_TIMEOUT, 2, (uint32_t)t, (uint32_t)s);
        sm.broken = 1;
        const uint64_t t1 = gtimer();
        while (!mbar_try_wait(&sm.full[s], ph) && gtimer() - t1 < p.wait_ns) {
        }
      }
      sm.fail = ok ? 0 : 1;
    }
    __syncthreads();
    const bool tma_ok = tma && !sm.fail;
    if (tma_ok && tid != 0) {
      // the phase is complete (thread 0 saw it); each thread's own wait makes the copy's writes visible to it
      for (uint32_t k = 0; k < (1u << 20) && !mbar_try_wait(&sm.full[s], ph); k++) {
      }
    }
    const int64_t row = g.row0 + tid;
    const bool full = g.row0 * kLaneTerms >= g.g_lo && (g.row0 + kTileRows) * kLaneTerms <= g.g_hi;
    const bool lane_tma = tma_ok && row < p.tma_rows;
    uint64_t v[kLaneTerms];
    load_row(p, stages + s * kStageBytes, lane_tma, row, g, full, v);
    __syncthreads();
    if (tid == 0) refill(p, sm, stages, tmap, s, ntiles);
    process_tile(p, sm, v, t, g, tag);
    if (tid == 0) {
      stat_add(sm, S_TILES, 1);
      sm.t_stream_end = gtimer();
    }
  }
  __syncthreads();
}

// ------------------------------------------------------------------ the walk: raw terms
// One warp adds up to 32 terms (lane l holds term l; lanes >= n hold -0) to
// the exact running value Sb, in order: while Sb is a normal number (with
// e >= -959), every term's run under Sb's binade is scanned in order and
// checked prefix by prefix against Sb; the longest prefix that passes is
// applied at once, and the term after it (which leaves the binade) is added
// with the hardware add.  A zero, subnormal, tiny or non-finite Sb takes one
// hardware add per term.
__device__ __noinline__ uint64_t raw_chunk(Smem &sm, uint64_t Sb, uint64_t t, int n) {
  const int lane = threadIdx.x & 31;
  int i = 0;
  uint32_t rounds = 0, dadds = 0;
  while (i < n) {
    const uint32_t Eb = (uint32_t)(Sb >> 52) & 0x7FFu;
    if (Eb >= 64u && Eb < 0x7FFu) {
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
    Sb = raw_chunk(sm, Sb, t, n);
  }
  return Sb;
}

// ------------------------------------------------------------------ the walk: one batch of tile headers
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

// Applies one run (lane 0 decides) and, if the check refuses it, adds the
// run's terms from x.  Warp 0.
__device__ __forceinline__ uint64_t apply_or_raw(const Params &p, Smem &sm, uint64_t Sb, const Run &r, uint32_t eb,
                                                 const WalkSum &ws, int64_t tile, uint32_t start, uint32_t count) {
  const int lane = threadIdx.x & 31;
  uint64_t nb = Sb;
  int ok = 0;
  if (lane == 0) ok = run_apply(nb, r, (int)eb - 1023) == APPLY_OK;
  ok = __shfl_sync(kFull, ok, 0);
  if (ok) return __shfl_sync(kFull, nb, 0);
  if (lane == 0) stat_add(sm, S_RUN_REJECTED, 1);
  int64_t a, b;
  clip(ws, tile, start, count, a, b);
  return raw_from_x(p, sm, Sb, a, b);
}

__device__ __noinline__ uint64_t apply_items(const Params &p, Smem &sm, uint64_t Sb, const Rec *slots, uint32_t nsl,
                                             const WalkSum &ws, int64_t tile) {
  const int lane = threadIdx.x & 31;
  uint32_t s = 0;
  while (s < nsl) {
    const Item it = unpack_item(slots[s]);
    if (it.kind == K_RAW && s + kRawSlots <= nsl) {
      const uint64_t *terms = reinterpret_cast<const uint64_t *>(&slots[s + 1]);
      const uint64_t t = lane < kLaneTerms ? terms[lane] : kNegZero;
      Sb = raw_chunk(sm, Sb, t, kLaneTerms);
      s += kRawSlots;
    } else if (it.kind == K_RUN) {
      Sb = apply_or_raw(p, sm, Sb, it.r, it.eb, ws, tile, it.start, it.count);
      if (lane == 0) stat_add(sm, S_WALK_SEGMENTS, 1);
      s += 1;
    } else {
      // an item this walk does not know: the tile's terms from x
      int64_t a, b;
      clip(ws, tile, 0, kTileTerms, a, b);
      Sb = raw_from_x(p, sm, Sb, a, b);
      break;
    }
  }
  return Sb;
}

// Walks the tiles [ws.tb, ws.te) of one sum from the start value Sb.
// Returns the sum's bits; NaN if a header never came.
__device__ __noinline__ uint64_t walk_sum(const Params &p, Smem &sm, unsigned char *dyn, const WalkSum &ws,
                                         uint64_t Sb, uint32_t tag) {
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  Rec *bh = reinterpret_cast<Rec *>(dyn);                                   // kBatch headers
  Rec *slots = bh + kBatch;                                                 // kBatchSlots item slots
  Run *comp = reinterpret_cast<Run *>(dyn + (kBatch + kBatchSlots) * 32);   // composites at segment tails
  int16_t *seg_tail = reinterpret_cast<int16_t *>(comp + kBatch);
  int16_t *seg_start = seg_tail + kBatch;
  int16_t *sl_off = seg_start + kBatch;
  int16_t *sl_cnt = sl_off + kBatch;
  if (tid == 0) {
    sm.S = Sb;
    sm.fail = 0;
  }
  __syncthreads();
  int64_t pos = ws.tb;
  while (pos < ws.te) {
    const int nb = (int)min((int64_t)kBatch, ws.te - pos);
    if (tid == 0) {
      const uint64_t t0 = gtimer();
      uint32_t spin = 0;
      sm.fail = 0;
      while (true) {
        const Rec q = ld_rec_vol(&p.hdr[pos]);
        if (tags_ok(q, tag)) break;
        if ((++spin & 63u) == 0u && gtimer() - t0 > p.wait_ns) {
          note_timeout(p, ERR_WALK_TIMEOUT, 3, (uint32_t)pos, (uint32_t)ws.te);
          sm.fail = 1;
          break;
        }
        __nanosleep(64);
      }
      sm.count = nb;
    }
    __syncthreads();
    if (sm.fail) break;
    Rec h;
    h.w[0] = h.w[1] = h.w[2] = h.w[3] = 0;
    bool ready = false;
    if (tid < nb) {
      h = ld_rec_vol(&p.hdr[pos + tid]);
      ready = tags_ok(h, tag);
    }
    if (tid < nb && !ready) atomicMin(&sm.count, tid);
    __syncthreads();
    int count = sm.count;
    fence_acq_rel();
    const Item it = unpack_item(h);
    // item slots of the complex tiles, packed in order
    uint32_t my = (tid < count && it.kind == K_COMPLEX) ? it.count : 0u;
    uint32_t inc = my;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t q = __shfl_up_sync(kFull, inc, o);
      if (lane >= o) inc += q;
    }
    if (lane == 31) sm.wslots[w] = inc;
    __syncthreads();
    uint32_t base = 0;
    for (int k = 0; k < w; k++) base += sm.wslots[k];
    const uint32_t off = base + inc - my;
    if (tid < count && off + my > (uint32_t)kBatchSlots) atomicMin(&sm.count, tid);
    __syncthreads();
    count = sm.count;   // the batch ends before the first tile whose items do not fit
    const bool mine = tid < count;
    if (tid < count) {
      bh[tid] = h;
      sl_off[tid] = (int16_t)off;
      sl_cnt[tid] = (int16_t)my;
    }
    __syncthreads();
    const uint32_t total = count > 0 ? (uint32_t)sl_off[count - 1] + (uint32_t)sl_cnt[count - 1] : 0u;
    for (uint32_t q = tid; q < total; q += kThreads) {
      int lo = 0, hi = count;   // the tile whose slots hold q: sl_off[lo] <= q < sl_off[lo] + sl_cnt[lo]
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if ((uint32_t)sl_off[mid] <= q) lo = mid;
        else hi = mid;
      }
      const uint32_t k = q - (uint32_t)sl_off[lo];
      if (SQ_OK(p, k < (uint32_t)kItemSlots && q < (uint32_t)kBatchSlots, 21, q))
        slots[q] = p.items[(pos + lo) * kItemSlots + k];
    }
    // ---- segmented scan of the runs over the batch's headers
    const Item me = mine ? unpack_item(bh[tid]) : it;
    const bool isrun = mine && me.kind == K_RUN;
    Run r = isrun ? me.r : run_empty();
    const uint32_t key = isrun ? me.eb : 0xFFFFFFFFu;
    const uint32_t pkey0 = __shfl_up_sync(kFull, key, 1);
    const bool prun0 = __shfl_up_sync(kFull, isrun, 1);
    if (lane == 0) sm.whead0[w] = 0;
    __syncthreads();
    // the previous element of lane 0 is the last lane of the previous warp
    uint32_t pkey = pkey0;
    bool prun = prun0;
    if (lane == 0 && w > 0) {
      const Item pv = unpack_item(bh[tid - 1]);
      prun = (tid - 1 < count) && pv.kind == K_RUN;
      pkey = prun ? pv.eb : 0xFFFFFFFFu;
    }
    const bool head = mine && (tid == 0 || !isrun || !prun || key != pkey);
    bool hf = head;
    int st = head ? tid : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const Run q = shfl_run_up(r, o);
      const bool qh = __shfl_up_sync(kFull, hf, o);
      const int qs = __shfl_up_sync(kFull, st, o);
      if (lane >= o) {
        if (!hf) r = run_compose(q, r);
        hf = hf || qh;
        st = max(st, qs);
      }
    }
    if (lane == 31) {
      sm.wtot[w] = r;
      sm.wtot_head[w] = hf;
      sm.wstart[w] = st;
    }
    if (lane == 0) sm.whead0[w] = head;
    __syncthreads();
    if (!hf) {
      // the segment began in an earlier warp: compose the carry in
      Run cr = run_empty();
      int cs = 0;
      for (int k = 0; k < w; k++) {
        cr = sm.wtot_head[k] ? sm.wtot[k] : run_compose(cr, sm.wtot[k]);
        cs = max(cs, sm.wstart[k]);
      }
      r = run_compose(cr, r);
      st = max(st, cs);
    }
    const bool sd = __shfl_down_sync(kFull, head, 1);
    const bool nxhead = (lane < 31) ? sd : (w + 1 < kWarps ? (sm.whead0[w + 1] != 0) : true);
    const bool tl = mine && (tid == count - 1 || nxhead || !isrun);
    const uint32_t tb = __ballot_sync(kFull, tl);
    if (lane == 0) sm.wtails[w] = __popc(tb);
    __syncthreads();
    uint32_t tbase = 0;
    for (int k = 0; k < w; k++) tbase += sm.wtails[k];
    if (tl) {
      const uint32_t j = tbase + __popc(tb & ((1u << lane) - 1u));
      seg_tail[j] = (int16_t)tid;
      seg_start[j] = (int16_t)(isrun ? st : tid);
      comp[j] = r;
    }
    if (tid == 0) {
      uint32_t nseg = 0;
      for (int k = 0; k < kWarps; k++) nseg += sm.wtails[k];
      sm.nseg = (int)nseg;
    }
    __syncthreads();
    // ---- the in-order pass (warp 0)
    if (w == 0) {
      uint64_t S = sm.S;
      const int nseg = sm.nseg;
      for (int j = 0; j < nseg; j++) {
        const int i = seg_tail[j];
        const Item e = unpack_item(bh[i]);
        if (e.kind == K_RUN) {
          uint64_t nb2 = S;
          int ok = 0;
          if (lane == 0) ok = run_apply(nb2, comp[j], (int)e.eb - 1023) == APPLY_OK;
          ok = __shfl_sync(kFull, ok, 0);
          if (ok) {
            S = __shfl_sync(kFull, nb2, 0);
          } else {
            for (int ii = seg_start[j]; ii <= i; ii++) {
              const Item e2 = unpack_item(bh[ii]);
              S = apply_or_raw(p, sm, S, e2.r, e2.eb, ws, pos + ii, 0, kTileTerms);
            }
          }
          if (lane == 0) stat_add(sm, S_WALK_SEGMENTS, 1);
        } else if (e.kind == K_COMPLEX) {
          S = apply_items(p, sm, S, slots + sl_off[i], (uint32_t)sl_cnt[i], ws, pos + i);
        } else {
          int64_t a, b;
          clip(ws, pos + i, 0, kTileTerms, a, b);
          S = raw_from_x(p, sm, S, a, b);
        }
      }
      if (lane == 0) {
        sm.S = S;
        stat_add(sm, S_WALK_BATCHES, 1);
      }
    }
    __syncthreads();
    pos += count;
  }
  __syncthreads();
  const uint64_t out = sm.fail ? 0x7FF8000000000000ull : sm.S;
  __syncthreads();
  return out;
}

__device__ __noinline__ void walk_loop(const Params &p, Smem &sm, unsigned char *dyn, int64_t ntiles, uint32_t tag) {
  const int tid = threadIdx.x;
  while (true) {
    if (tid == 0) sm.wk = p.offsets ? (int)atomicAdd(&p.ctr[C_SUMTICKET], 1u) : (sm.wk == 0 ? 0 : 1);
    __syncthreads();
    const int k = sm.wk;
    if (k >= p.nsums) break;
    WalkSum ws;
    double s0;
    if (p.offsets) {
      ws.tb = p.tile_begin[k];
      ws.te = p.tile_begin[k + 1];
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
    const uint64_t S = walk_sum(p, sm, dyn, ws, dbits(s0), tag);
    if (tid == 0) {
      p.outs[k] = bitsd(S);
      if (!p.offsets) sm.wk = 1;
    }
    __syncthreads();
  }
}

// ------------------------------------------------------------------ the kernel
__global__ void __launch_bounds__(kThreads, 2) seqsum_kernel(const Params p, const __grid_constant__ CUtensorMap tmap) {
  extern __shared__ unsigned char dyn_raw[];
  unsigned char *dyn = reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(dyn_raw) + 1023) & ~uintptr_t(1023));
  __shared__ Smem sm;
  const int tid = threadIdx.x;
  if (tid < S_ACCUM_END) sm.stat[tid] = 0;
  if (tid == 0) {
    sm.role = (int)atomicAdd(&p.ctr[C_ROLE], 1u);
    const uint32_t e = *reinterpret_cast<volatile uint32_t *>(&p.ctr[C_EPOCH]);
    sm.tag = e == 0 ? 1u : e;
    sm.ntiles = p.offsets ? (int64_t)*reinterpret_cast<volatile uint32_t *>(&p.ctr[C_NTILES]) : p.ntiles;
    sm.fail = *reinterpret_cast<volatile uint32_t *>(&p.ctr[C_SKIP]) != 0u && p.offsets;
    sm.wk = 0;
    if (sm.role == 0) p.stats[S_T_START] = gtimer();
  }
  __syncthreads();
  const uint32_t tag = sm.tag;
  const int64_t ntiles = sm.ntiles;
  const bool skip = sm.fail;
  __syncthreads();
  if (!skip) {
    if (sm.role < p.nwalkers) {
      walk_loop(p, sm, dyn, ntiles, tag);
      if (tid == 0) atomicMax(&p.stats[S_T_WALK_END], (unsigned long long)gtimer());
    } else {
      stream_loop(p, sm, dyn, &tmap, ntiles, tag);
      if (tid == 0 && sm.t_stream_end) atomicMax(&p.stats[S_T_STREAM_END], (unsigned long long)sm.t_stream_end);
    }
  }
  __syncthreads();
  if (tid < S_ACCUM_END && sm.stat[tid]) atomicAdd(&p.stats[tid], sm.stat[tid]);
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
      for (int64_t i = tid; i < p.cap_tiles; i += kThreads) {
        p.status[i] = make_uint4(0, 0, 0, 0);
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
      p.ctr[C_EPOCH] = next > 255u ? 1u : next;
      __threadfence();
      p.ctr[C_EXIT] = 0;
    }
  }
}

// The batched calls' set-up: checks the offsets, counts each sum's tiles and
// writes tile_begin (one CTA).  On bad offsets or too many tiles every output
// is NaN and the main kernel does nothing.
__global__ void __launch_bounds__(kThreads) setup_kernel(const Params p) {
  __shared__ int bad;
  __shared__ int64_t carry;
  __shared__ int64_t wsum[kWarps];
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  if (tid == 0) {
    bad = 0;
    carry = 0;
  }
  __syncthreads();
  for (int k = tid; k <= p.nsums; k += kThreads) {
    const int64_t o = p.offsets[k];
    if (o < 0 || o > p.x_len) bad = 1;
    if (k > 0 && p.offsets[k - 1] > o) bad = 1;
  }
  __syncthreads();
  if (!bad) {
    for (int k0 = 0; k0 < p.nsums; k0 += kThreads) {
      const int k = k0 + tid;
      int64_t nt = 0;
      if (k < p.nsums) {
        const int64_t a = p.offsets[k], b = p.offsets[k + 1];
        if (b > a) {
          const int64_t rows = ((b + 15) >> 4) - (a >> 4);
          nt = (rows + kTileRows - 1) / kTileRows;
        }
      }
      int64_t inc = nt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int64_t q = __shfl_up_sync(kFull, inc, o);
        if (lane >= o) inc += q;
      }
      if (lane == 31) wsum[w] = inc;
      __syncthreads();
      int64_t base = carry;
      for (int j = 0; j < w; j++) base += wsum[j];
      if (k < p.nsums) p.tile_begin[k] = base + inc - nt;
      __syncthreads();
      if (tid == 0) {
        int64_t tot = 0;
        for (int j = 0; j < kWarps; j++) tot += wsum[j];
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
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, seqsum_kernel, kThreads, kDynSmem);
  return n > 0 ? n : 1;
}

cudaError_t launch_seqsum(const Params &p, const CUtensorMap *tmap, int grid, cudaStream_t st) {
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(seqsum_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kDynSmem);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  seqsum_kernel<<<grid, kThreads, kDynSmem, st>>>(p, *tmap);
  return cudaGetLastError();
}

cudaError_t launch_setup(const Params &p, cudaStream_t st) {
  setup_kernel<<<1, kThreads, 0, st>>>(p);
  return cudaGetLastError();
}

}  // namespace sq

// The device path of the exact sequential fp64 sum (sm_103a).
//
// One persistent kernel does all of it:
//   1. streams the term plane once: a tile of 4096 terms (32 KB) per TMA box,
//      two stages per CTA, swizzled (128B) so that each lane reads its own
//      128-byte row of 16 consecutive terms without bank conflicts;
//   2. forms approximate chunk sums in fp32 from the terms' bits and a
//      parallel approximate prefix over tiles (decoupled look-back) that
//      names each chunk's starting binade (Research-1424, section 3: "a first
//      pass can add each row on its own and a prefix over the rows gives S at
//      each row start ... which names the binade except next to a power of
//      two"; Research-1433, finding 5; open question "compute the plan's
//      prefix with a scan across the lanes");
//   3. turns every term into its even/odd increment pair by integer shifts
//      (binade_math.cuh) and composes them in order: a lane's 16 terms, then
//      the warp's 32 lanes in a fixed shuffle tree, then the tile's 8 chunks
//      (Research-1433, finding 6: "composes each lane's ... terms in order and
//      then the lanes in an ordered tree");
//   4. the CTA that finishes a sum's last tile walks the sum in order with the
//      exact running value: runs of tiles that share a binade are composed in
//      parallel first, so the serial part steps over whole segments
//      (Research-1433, open question: "compose runs of chunks that share a
//      binade so that the walk steps over 64 or 1024 chunks at a time"); a run
//      the exact check rejects is descended into, and a chunk or lane the
//      plan could not place is added term by term in fp64 (finding 4).
//
// This translation unit is built with --fmad=false; the term-by-term adds use
// __dadd_rn, one IEEE binary64 add each, in index order.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "binade_math.cuh"
#include "seqsum_internal.cuh"

namespace sq {

// ---------------------------------------------------------------- constants
// Relative error allowance of the approximate prefix against the running sum
// of |x| (fp32 terms truncated to 24 bits, fp32 sums of 16 and of 32 values,
// fp64 across chunks and tiles: about 2^-19.5 at worst).  The plan only
// chooses where to look; a wrong guess costs a fallback, never a wrong bit.
constexpr double kEps = 0x1p-18;
constexpr double kTiny = 0x1p-1000;
constexpr int kZeroE = -2000;                  // binade key of a run of zeros
constexpr int kComplexKey = -100000;           // a tile that is a segment of its own
constexpr uint64_t kWaitNs = 2000000000ull;    // bounded device waits: 2 s

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
__device__ __forceinline__ uint64_t ld_vol_u64(const uint64_t *p) {
  uint64_t v;
  asm volatile("ld.volatile.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_vol_u64(uint64_t *p, uint64_t v) {
  asm volatile("st.volatile.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ uint32_t lanemask_lt() {
  uint32_t m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

// ---------------------------------------------------------------- helpers
__device__ __forceinline__ uint64_t dbits(double v) { return (uint64_t)__double_as_longlong(v); }
__device__ __forceinline__ double bitsd(uint64_t b) { return __longlong_as_double((long long)b); }

// A cheap fp32 image of a term built from its bits (integer ops only; the
// fp64 pipe is not used): the top 23 fraction bits, exponent clamped to the
// fp32 range.  Only the plan uses it.
__device__ __forceinline__ float approx_f32(uint64_t b) {
  const uint32_t hi = (uint32_t)(b >> 32), lo = (uint32_t)b;
  int32_t v = (int32_t)(hi & 0x7FFFFFFFu) - (896 << 20);
  v = max(v, 0);
  v = min(v, (254 << 20) | 0xFFFFF);
  const uint32_t fb = __funnelshift_l(lo, (uint32_t)v, 3) | (hi & 0x80000000u);
  return __uint_as_float(fb);
}

// Binade (unbiased exponent) shared by all of [lo, hi], or false.
__device__ __forceinline__ bool one_binade(double lo, double hi, int &e) {
  double a, b;
  if (lo > 0.0) { a = lo; b = hi; }
  else if (hi < 0.0) { a = -hi; b = -lo; }
  else return false;
  const int ea = (int)((dbits(a) >> 52) & 0x7FF), eb = (int)((dbits(b) >> 52) & 0x7FF);
  if (ea != eb || ea == 0 || ea == 0x7FF) return false;
  e = ea - 1023;
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
__device__ __forceinline__ Rec shfl_rec(const Rec &r, int src) {
  Rec o;
  const int *s = reinterpret_cast<const int *>(&r);
  int *d = reinterpret_cast<int *>(&o);
#pragma unroll
  for (int i = 0; i < 8; i++) d[i] = __shfl_sync(0xffffffffu, s[i], src);
  return o;
}

__device__ __forceinline__ Rec make_rec(const Run &r, int e, uint32_t kind, uint32_t count) {
  Rec q;
  q.inc = r.inc; q.lo = r.lo; q.hi = r.hi;
  q.meta = rec_meta(r.d, r.flags, kind);
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
    const int64_t s0 = p.offsets[lo];
    g.start = s0 + g.tile_in_sum * kTileTerms;
    g.end = min(p.offsets[lo + 1], g.start + kTileTerms);
  }
  return g;
}

// ---------------------------------------------------------------- look-back
// Per tile two tagged 64-bit words: A = approximate prefix (fp64, low 8 bits
// replaced by the tag), B = approximate |x| prefix (fp32) << 32 | tag.
// tag = epoch << 1 | kind; kind 0 = this tile's aggregate, 1 = inclusive
// prefix.  Each word is written and read whole, and a reader accepts a tile
// only when both words carry the current tag, so no fence is needed.
__device__ __forceinline__ void publish(uint64_t *st, double sig, float ab, uint32_t epoch, uint32_t kind) {
  const uint32_t tag = (epoch << 1) | kind;
  const uint64_t A = (dbits(sig) & ~0xFFull) | tag;
  const uint64_t B = ((uint64_t)__float_as_uint(ab) << 32) | tag;
  st_vol_u64(st, A);
  st_vol_u64(st + 1, B);
}

// Run by one whole warp.  Returns the approximate exclusive prefix of tile t.
__device__ void lookback(const Params &p, const TileGeo &g, int64_t t, double agg_sig, float agg_abs,
                         double &ex_sig, float &ex_abs, unsigned long long *st) {
  const int lane = threadIdx.x & 31;
  const uint32_t ep = p.epoch;
  if (g.tile_in_sum == 0) {
    const double s0 = p.s0s ? p.s0s[g.sum] : p.s0;
    ex_sig = s0;
    ex_abs = fabsf((float)s0);
    if (lane == 0) publish(p.status + 2 * t, s0 + agg_sig, ex_abs + agg_abs, ep, 1);
    return;
  }
  if (lane == 0) publish(p.status + 2 * t, agg_sig, agg_abs, ep, 0);
  double run_sig = 0.0;
  float run_abs = 0.0f;
  int64_t j = t - 1;
  const uint64_t t0 = globaltimer();
  bool gave_up = false;
  while (true) {
    if (lane == 0) atomicAdd(&st[S_LOOKBACK_STEPS], 1ull);
    const int64_t idx = j - lane;
    double v = 0.0;
    float a = 0.0f;
    bool valid = true, incl = true;             // before the sum: a virtual prefix of 0
    if (idx >= g.first_tile) {
      const uint64_t A = ld_vol_u64(p.status + 2 * idx);
      const uint64_t B = ld_vol_u64(p.status + 2 * idx + 1);
      const uint32_t ta = (uint32_t)(A & 0xFF), tb = (uint32_t)(B & 0xFFFFFFFFu);
      valid = ((ta >> 1) == ep) && (ta == tb);
      incl = valid && (ta & 1u);
      v = bitsd(A & ~0xFFull);
      a = __uint_as_float((uint32_t)(B >> 32));
    }
    const uint32_t vmask = __ballot_sync(0xffffffffu, valid);
    const uint32_t imask = __ballot_sync(0xffffffffu, incl);
    bool done = false, advance = false;
    int L = 31;
    if (imask) {
      L = __ffs(imask) - 1;                           // nearest inclusive predecessor
      const uint32_t need = (L == 31) ? 0xffffffffu : ((2u << L) - 1u);
      done = (vmask & need) == need;
    } else if (vmask == 0xffffffffu) {
      advance = true;
    }
    if (!done && !advance) {
      if (globaltimer() - t0 > kWaitNs) { gave_up = true; done = true; L = 31; }
      else { __nanosleep(32); continue; }
    }
    double cv = (lane <= L && valid) ? v : 0.0;
    float ca = (lane <= L && valid) ? a : 0.0f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      cv += __shfl_xor_sync(0xffffffffu, cv, o);
      ca += __shfl_xor_sync(0xffffffffu, ca, o);
    }
    run_sig += cv;
    run_abs += ca;
    if (done) break;
    j -= 32;
  }
  if (gave_up && lane == 0) atomicOr(&p.ctr[C_ERR], ERR_PLAN_TIMEOUT);
  ex_sig = run_sig;
  ex_abs = run_abs;
  if (lane == 0) publish(p.status + 2 * t, run_sig + agg_sig, run_abs + agg_abs, ep, 1);
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
__device__ uint64_t add_terms(const Params &p, uint64_t Sb, int64_t a, int64_t cnt, unsigned long long *st) {
  const int lane = threadIdx.x & 31;
  double S = bitsd(Sb);
  for (int64_t base = 0; base < cnt; base += 32) {
    const double v = (base + lane < cnt) ? __ldg(p.x + a + base + lane) : 0.0;
    const int m = (int)min((int64_t)32, cnt - base);
    for (int j = 0; j < m; j++) {
      const double t = __shfl_sync(0xffffffffu, v, j);
      S = __dadd_rn(S, t);
    }
  }
  if (lane == 0) atomicAdd(&st[S_TERMS_ADDED], (unsigned long long)cnt);
  return dbits(S);
}

// Apply one record to S (warp-uniform).  A run the check rejects falls back
// to term-by-term adds over the record's terms [a, a + cnt).
__device__ uint64_t apply_or_add(const Params &p, uint64_t Sb, const Rec &q, int64_t a, int64_t cnt,
                                 unsigned long long *st) {
  const int lane = threadIdx.x & 31;
  if (nonfinite(Sb)) return absorb(Sb, rec_flags(q.meta));
  if (rec_kind(q.meta) == K_RUN) {
    uint64_t T = Sb;
    if (run_apply(T, rec_run(q), q.e) == APPLY_OK) return T;
    if (lane == 0) atomicAdd(&st[S_RUN_REJECTED], 1ull);
  }
  return add_terms(p, Sb, a, cnt, st);
}

// One chunk record (warp-uniform): a run, a list of items, or a fallback.
__device__ uint64_t walk_chunk(const Params &p, uint64_t Sb, const Rec &c, int64_t a, int64_t cnt,
                               unsigned long long *st) {
  const int lane = threadIdx.x & 31;
  const uint32_t kind = rec_kind(c.meta);
  if (kind != K_LIST) {
    if (kind == K_FALLBACK && lane == 0) atomicAdd(&st[S_CHUNK_FALLBACK], 1ull);
    return apply_or_add(p, Sb, c, a, cnt, st);
  }
  if (nonfinite(Sb)) return absorb(Sb, rec_flags(c.meta));
  const int nit = (int)c.lo;
  Rec mine;
  if (lane < nit) mine = ldcg_rec(p.pool + c.inc + lane);
  int64_t pos = a;
  for (int i = 0; i < nit; i++) {
    const Rec it = shfl_rec(mine, i);
    const int64_t n_it = min((int64_t)it.count, a + cnt - pos);
    Sb = apply_or_add(p, Sb, it, pos, n_it, st);
    pos += it.count;
  }
  return Sb;
}

// A tile the segment composite could not cover: its chunks in order.
__device__ uint64_t walk_tile(const Params &p, uint64_t Sb, int64_t t, const TileGeo &g, unsigned long long *st) {
  const int lane = threadIdx.x & 31;
  Rec mine;
  if (lane < kWarps) mine = ldcg_rec(p.chunk_rec + t * kWarps + lane);
  for (int c = 0; c < kWarps; c++) {
    const int64_t a = g.start + (int64_t)c * kChunkTerms;
    if (a >= g.end) break;
    const int64_t cnt = min((int64_t)kChunkTerms, g.end - a);
    Sb = walk_chunk(p, Sb, shfl_rec(mine, c), a, cnt, st);
  }
  return Sb;
}

__device__ __forceinline__ int seg_key(const Rec &q) {
  // a complex tile is a segment of its own; runs of zeros apart from runs
  if (rec_kind(q.meta) != K_RUN) return kComplexKey;
  if (rec_flags(q.meta) & F_ZERO) return kZeroE;
  return q.e;
}

// The in-order walk of the sum of tile g0 over its tiles, by the whole CTA;
// the serial part runs on warp 0.  `srec` is a free stage buffer.
__device__ void walk_sum(const Params &p, const TileGeo &g0, Rec *srec, unsigned long long *st) {
  __shared__ int s_ends[kWalkBatch];
  __shared__ unsigned char s_head[kWalkBatch];
  __shared__ int s_wcnt[kWarps];
  __shared__ int s_nends;
  __shared__ uint64_t s_S;
  __shared__ int s_restart;
  __shared__ Run s_wagg[kWarps];
  __shared__ int s_wflag[kWarps];
  constexpr int B = kWalkBatch / kThreads;         // elements per thread
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t tb = g0.first_tile, te = g0.first_tile + g0.ntiles_sum;
  const double s0 = p.s0s ? p.s0s[g0.sum] : p.s0;
  if (tid == 0) s_S = dbits(s0);
  int64_t base = tb;
  __syncthreads();
  while (base < te) {
    const int cnt = (int)min((int64_t)kWalkBatch, te - base);
    for (int i = tid; i < cnt; i += kThreads) srec[i] = ldcg_rec(p.tile_rec + base + i);
    __syncthreads();
    for (int i = tid; i < cnt; i += kThreads) {
      const int k = seg_key(srec[i]);
      s_head[i] = (i == 0 || k == kComplexKey || seg_key(srec[i - 1]) != k) ? 1 : 0;
    }
    __syncthreads();
    // --- per-thread segmented inclusive scan over B consecutive elements
    Run agg = run_empty();
    bool has_head = false;
    int first_head = B;
    for (int j = 0; j < B; j++) {
      const int i = tid * B + j;
      if (i >= cnt) break;
      const Rec q = srec[i];
      const bool head = s_head[i] != 0;
      const Run r = rec_run(q);
      if (head) { agg = r; if (!has_head) first_head = j; has_head = true; }
      else agg = run_compose(agg, r);
      srec[i] = make_rec(agg, q.e, rec_kind(q.meta), 0);
    }
    // --- block-level segmented scan of the thread aggregates
    Run v = agg;
    int f = has_head ? 1 : 0;
    for (int off = 1; off < 32; off <<= 1) {
      const Run o = shfl_run<SH_UP>(v, off);
      const int of = __shfl_up_sync(0xffffffffu, f, off);
      if (lane >= off) { if (!f) v = run_compose(o, v); f |= of; }
    }
    if (lane == 31) { s_wagg[warp] = v; s_wflag[warp] = f; }
    __syncthreads();
    Run ex = run_empty();                             // exclusive prefix of this thread
    for (int w = 0; w < warp; w++) {
      if (s_wflag[w]) ex = s_wagg[w];
      else ex = run_compose(ex, s_wagg[w]);
    }
    {
      const Run lv = shfl_run<SH_UP>(v, 1);
      const int lf = __shfl_up_sync(0xffffffffu, f, 1);
      if (lane >= 1) {
        if (lf) ex = lv; else ex = run_compose(ex, lv);
      }
    }
    for (int j = 0; j < first_head; j++) {            // elements before the first head
      const int i = tid * B + j;
      if (i >= cnt) break;
      const Rec q = srec[i];
      srec[i] = make_rec(run_compose(ex, rec_run(q)), q.e, rec_kind(q.meta), 0);
    }
    __syncthreads();
    // --- segment ends, compacted in order
    {
      int my = 0;
      int idx[B];
      for (int j = 0; j < B; j++) {
        const int i = tid * B + j;
        if (i < cnt && (i == cnt - 1 || s_head[i + 1])) idx[my++] = i;
      }
      int incl = my;
      for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += o;
      }
      if (lane == 31) s_wcnt[warp] = incl;
      __syncthreads();
      int wbase = 0;
      for (int w = 0; w < warp; w++) wbase += s_wcnt[w];
      const int pos = wbase + incl - my;
      for (int j = 0; j < my; j++) s_ends[pos + j] = idx[j];
      if (tid == kThreads - 1) s_nends = wbase + incl;
    }
    __syncthreads();
    // --- the serial part: warp 0 applies segment after segment
    if (warp == 0) {
      uint64_t Sb = s_S;
      int restart = -1;
      int segstart = 0;
      const int ne = s_nends;
      for (int sidx = 0; sidx < ne; sidx++) {
        const int e_i = s_ends[sidx];
        const Rec comp = srec[e_i];
        if (lane == 0) atomicAdd(&st[S_WALK_SEGMENTS], 1ull);
        bool ok = false;
        if (rec_kind(comp.meta) == K_RUN) {
          if (nonfinite(Sb)) { Sb = absorb(Sb, rec_flags(comp.meta)); ok = true; }
          else {
            uint64_t T = Sb;
            if (run_apply(T, rec_run(comp), comp.e) == APPLY_OK) { Sb = T; ok = true; }
          }
        }
        if (!ok) {
          if (lane == 0) atomicAdd(&st[rec_kind(comp.meta) == K_RUN ? S_RUN_REJECTED : S_TILE_COMPLEX], 1ull);
          // the first prefix of the segment the check rejects (in parallel)
          int kfail = e_i;
          for (int c0 = segstart; c0 <= e_i; c0 += 32) {
            const int i = c0 + lane;
            bool bad = false;
            if (i <= e_i) {
              const Rec q = srec[i];
              if (rec_kind(q.meta) != K_RUN || nonfinite(Sb)) bad = true;
              else { uint64_t T = Sb; bad = run_apply(T, rec_run(q), q.e) != APPLY_OK; }
            }
            const uint32_t bm = __ballot_sync(0xffffffffu, bad);
            if (bm) { kfail = c0 + __ffs(bm) - 1; break; }
          }
          if (kfail > segstart) {                      // the prefix before it passed
            const Rec q = srec[kfail - 1];
            uint64_t T = Sb;
            if (run_apply(T, rec_run(q), q.e) == APPLY_OK) Sb = T;
          }
          const int64_t t = base + kfail;
          Sb = walk_tile(p, Sb, t, tile_geo(p, t, te), st);
          if (kfail < e_i) { restart = kfail + 1; break; }
        }
        segstart = e_i + 1;
      }
      if (lane == 0) { s_S = Sb; s_restart = restart; }
    }
    __syncthreads();
    base = (s_restart >= 0) ? base + s_restart : base + cnt;
    __syncthreads();
  }
  if (tid == 0) {
    p.outs[g0.sum] = bitsd(s_S);
    p.done[g0.sum] = 0;
  }
  __syncthreads();
}

// ---------------------------------------------------------------- the kernel
__global__ void __launch_bounds__(kThreads, 2)
    seqsum_kernel(const Params p, const __grid_constant__ CUtensorMap tmap) {
  extern __shared__ unsigned char dsm_raw[];
  unsigned char *stage0 =
      reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(dsm_raw) + 1023) & ~(uintptr_t)1023);
  __shared__ __align__(8) uint64_t s_bar[kStages];
  __shared__ int64_t s_tk[kStages];
  __shared__ int s_tma[kStages];
  __shared__ float s_wsig[kWarps], s_wabs[kWarps];
  __shared__ double s_ex_sig;
  __shared__ float s_ex_abs;
  __shared__ Rec s_chunk[kWarps];
  __shared__ int64_t s_pend[2];          // tiles whose sums this CTA must walk
  __shared__ int s_npend;
  __shared__ unsigned long long s_st[S_COUNT];

  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  int64_t ntiles = (p.ntiles >= 0) ? p.ntiles : (int64_t)__ldcg(&p.ctr[C_NTILES]);
  if (ntiles > p.cap_tiles) ntiles = 0;                  // set-up flagged ERR_CAPACITY
  unsigned long long *st = s_st;
  if (tid < S_COUNT) s_st[tid] = 0;
  if (tid == 0) {
    for (int s = 0; s < kStages; s++) mbar_init(&s_bar[s], 1);
    fence_mbar_init();
    s_npend = 0;
  }
  if (p.offsets == nullptr && ntiles == 0 && blockIdx.x == 0 && tid == 0) p.outs[0] = p.s0;
  __syncthreads();

  // thread 0: take the next ticket into stage s and start its copy
  auto issue = [&](int s) {
    const int64_t t = (int64_t)atomicAdd(&p.ctr[C_TICKET], 1u);
    s_tk[s] = t;
    s_tma[s] = 0;
    if (t >= ntiles || p.tma_rows == 0) return;
    const TileGeo g = tile_geo(p, t, ntiles);
    if ((g.start & 15) != 0) return;
    fence_proxy_async();
    mbar_arrive_expect_tx(&s_bar[s], (uint32_t)kStageBytes);
    tma_load_box(stage0 + s * kStageBytes, &tmap, &s_bar[s], 0, (int32_t)(g.start >> 4));
    s_tma[s] = 1;
  };
  // the whole CTA: walk the sums this CTA finished (no ticket is held then)
  auto flush_walks = [&]() {
    const int np = s_npend;
    for (int i = 0; i < np; i++) {
      const TileGeo gw = tile_geo(p, s_pend[i], ntiles);
      __threadfence();
      walk_sum(p, gw, reinterpret_cast<Rec *>(stage0), st);
    }
    __syncthreads();
    if (tid == 0) s_npend = 0;
    __syncthreads();
  };

  if (tid == 0) issue(0);
  __syncthreads();
  uint32_t phase[kStages] = {0, 0};
  int cur = 0;
  while (true) {
    const int64_t t = s_tk[cur];
    if (t >= ntiles) { flush_walks(); break; }
    const bool hold = s_npend > 0;          // walks pending: finish this tile, walk, then take more
    __syncthreads();
    if (tid == 0 && !hold) issue(cur ^ 1);
    const TileGeo g = tile_geo(p, t, ntiles);
    const int use_tma = s_tma[cur];

    // ---- 1. the lane's 16 terms
    uint64_t xs[kLaneTerms];
    const int64_t lstart = g.start + (int64_t)w * kChunkTerms + (int64_t)lane * kLaneTerms;
    const int nv = (int)max((int64_t)0, min((int64_t)kLaneTerms, g.end - lstart));
    const int64_t row = (g.start >> 4) + w * 32 + lane;
    if (use_tma) {
      const uint64_t t0 = globaltimer();
      while (!mbar_try_wait(&s_bar[cur], phase[cur])) {
        if (globaltimer() - t0 > kWaitNs) { atomicOr(&p.ctr[C_ERR], ERR_TMA_TIMEOUT); break; }
      }
      phase[cur] ^= 1u;
    }
    if (use_tma && row < p.tma_rows) {
      const unsigned char *rp = stage0 + cur * kStageBytes + (w * 32 + lane) * 128;
      const int sw = lane & 7;
#pragma unroll
      for (int c = 0; c < 8; c++) {
        const uint4 v = *reinterpret_cast<const uint4 *>(rp + ((c ^ sw) << 4));
        xs[2 * c] = ((uint64_t)v.y << 32) | v.x;
        xs[2 * c + 1] = ((uint64_t)v.w << 32) | v.z;
      }
    } else {
      const unsigned long long *gp = reinterpret_cast<const unsigned long long *>(p.x) + lstart;
#pragma unroll
      for (int i = 0; i < kLaneTerms; i++) xs[i] = (i < nv) ? __ldg(gp + i) : 0ull;
    }
#pragma unroll
    for (int i = 0; i < kLaneTerms; i++)
      if (i >= nv) xs[i] = 0ull;

    // ---- 2. approximate sums for the plan
    float sig = 0.0f, ab = 0.0f;
    bool allzero = true;
#pragma unroll
    for (int i = 0; i < kLaneTerms; i++) {
      const float f = approx_f32(xs[i]);
      sig += f;
      ab += fabsf(f);
      allzero = allzero && ((xs[i] << 1) == 0);
    }
    float isig = sig, iab = ab;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float a = __shfl_up_sync(0xffffffffu, isig, o);
      const float b = __shfl_up_sync(0xffffffffu, iab, o);
      if (lane >= o) { isig += a; iab += b; }
    }
    const float xsig = isig - sig, xab = iab - ab;      // lane's exclusive prefix in the chunk
    if (lane == 31) { s_wsig[w] = isig; s_wabs[w] = iab; }
    __syncthreads();                                   // also: stage `cur` is free again

    // ---- 3. the tile's approximate exclusive prefix (decoupled look-back)
    if (w == 0) {
      double agg = 0.0;
      float agga = 0.0f;
#pragma unroll
      for (int k = 0; k < kWarps; k++) { agg += (double)s_wsig[k]; agga += s_wabs[k]; }
      double exs;
      float exa;
      lookback(p, g, t, agg, agga, exs, exa, st);
      if (lane == 0) { s_ex_sig = exs; s_ex_abs = exa; }
    }
    __syncthreads();

    // ---- 4. plan of this warp's chunk
    double sc = s_ex_sig;
    float ac = s_ex_abs;
    for (int k = 0; k < w; k++) { sc += (double)s_wsig[k]; ac += s_wabs[k]; }
    const float wsig = s_wsig[w], wabs = s_wabs[w];
    const int64_t cstart = g.start + (int64_t)w * kChunkTerms;
    const int cnt_chunk = (int)max((int64_t)0, min((int64_t)kChunkTerms, g.end - cstart));
    int e_s = 0;
    bool simple;
    {
      const double P = 0.5 * ((double)wabs + (double)wsig), N = 0.5 * ((double)wabs - (double)wsig);
      const double delta = kEps * ((double)ac + (double)wabs) + kTiny;
      simple = one_binade(sc - N - delta, sc + P + delta, e_s);
      simple = plan_override(p.plan_mode, simple, e_s, (uint64_t)t, w, 0);
    }
    int e_l = e_s;
    bool clean_l = simple;
    const bool zl = allzero;                            // lane of zeros (or no terms): exact anywhere
    if (!simple) {
      const double A = sc + (double)xsig;
      const double P = 0.5 * ((double)ab + (double)sig), N = 0.5 * ((double)ab - (double)sig);
      const double delta = kEps * ((double)ac + (double)xab + (double)ab) + kTiny;
      clean_l = one_binade(A - N - delta, A + P + delta, e_l);
      clean_l = plan_override(p.plan_mode, clean_l, e_l, (uint64_t)t, w, lane + 1);
      const uint32_t bad = __ballot_sync(0xffffffffu, !clean_l && !zl);
      const uint32_t placed = __ballot_sync(0xffffffffu, clean_l && !zl);
      if (bad == 0) {
        if (placed == 0) { simple = true; e_s = 0; }   // all zeros
        else {
          const int e_ref = __shfl_sync(0xffffffffu, e_l, __ffs(placed) - 1);
          if (__ballot_sync(0xffffffffu, zl || e_l == e_ref) == 0xffffffffu) { simple = true; e_s = e_ref; }
        }
      }
    }

    // ---- 5. increments and composition
    Rec crec;
    if (simple) {
      Run r = run_empty();
#pragma unroll
      for (int i = 0; i < kLaneTerms; i++) {
        if (i < nv) {
          int64_t re;
          int32_t d;
          const bool poison = term_inc(xs[i], e_s, re, d);
          run_push(r, re, d, term_flags(xs[i]) | (poison ? F_POISON : 0u));
        }
      }
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const Run o = shfl_run<SH_DOWN>(r, off);
        if ((lane & (2 * off - 1)) == 0) r = run_compose(r, o);
      }
      crec = make_rec(r, (r.flags & F_ZERO) ? kZeroE : e_s, K_RUN, (uint32_t)cnt_chunk);
      if (lane == 0) atomicAdd(&st[S_CHUNK_RUN], 1ull);
    } else {
      // mixed chunk: lanes placed in a binade become runs under their own
      // binade, unplaced lanes are added term by term; neighbouring lanes of
      // one kind and binade merge into one item.
      const bool fb = !clean_l && !zl;
      Run r = run_empty();
      uint32_t hasf = 0;
#pragma unroll
      for (int i = 0; i < kLaneTerms; i++) {
        if (i < nv) {
          const uint32_t tf = term_flags(xs[i]);
          hasf |= tf;
          if (!fb) {
            int64_t re;
            int32_t d;
            const bool poison = term_inc(xs[i], clean_l ? e_l : 0, re, d);
            run_push(r, re, d, tf | (poison ? F_POISON : 0u));
          }
        }
      }
      hasf &= (F_HASINF_P | F_HASINF_N | F_HASNAN);
      const int kind = fb ? 1 : 0;
      const int ekey = fb ? 0 : (clean_l ? e_l : kZeroE);
      if (lane == 0) atomicAdd(&st[S_CHUNK_LIST], 1ull);
      if (fb) atomicAdd(&st[S_LANE_DIRTY], 1ull);
      const bool empty_lane = (nv == 0);               // past the end: joins the previous segment
      const int pkind = __shfl_up_sync(0xffffffffu, kind, 1);
      const int pkey = __shfl_up_sync(0xffffffffu, ekey, 1);
      const bool head = (lane == 0) || (!empty_lane && (pkind != kind || pkey != ekey));
      Run v = r;                                        // segmented inclusive scan
      int f = head ? 1 : 0;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const Run o = shfl_run<SH_UP>(v, off);
        const int of = __shfl_up_sync(0xffffffffu, f, off);
        if (lane >= off) { if (!f) v = run_compose(o, v); f |= of; }
      }
      const uint32_t heads = __ballot_sync(0xffffffffu, head);
      const bool end = (lane == 31) || ((heads >> (lane + 1)) & 1u);
      const uint32_t ends = __ballot_sync(0xffffffffu, end);
      const int nit = __popc(ends);
      const uint32_t le = heads & ((lane == 31) ? 0xffffffffu : ((2u << lane) - 1u));
      const int hlane = 31 - __clz(le);
      const int skind = __shfl_sync(0xffffffffu, kind, hlane);
      const int skey = __shfl_sync(0xffffffffu, ekey, hlane);
      const int tstart = hlane * kLaneTerms;
      const int tend = min((lane + 1) * kLaneTerms, cnt_chunk);
      uint32_t orf = hasf;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) orf |= __shfl_xor_sync(0xffffffffu, orf, o);
      uint32_t pbase = 0;
      if (lane == 0) pbase = atomicAdd(&p.ctr[C_POOL], (uint32_t)nit);
      pbase = __shfl_sync(0xffffffffu, pbase, 0);
      Run lr = run_empty();
      lr.flags = orf;
      if ((int64_t)pbase + nit <= p.pool_cap) {
        if (end) {
          const int idx = __popc(ends & lanemask_lt());
          Run iv = v;
          if (skind == 1) { iv = run_empty(); iv.flags = orf; }
          const Rec it = make_rec(iv, skind == 1 ? 0 : skey, skind == 1 ? K_FALLBACK : K_RUN,
                                  (uint32_t)max(0, tend - tstart));
          stcg_rec(p.pool + pbase + idx, it);
        }
        lr.inc = (int64_t)pbase;
        lr.lo = nit;
        lr.hi = 0;
        crec = make_rec(lr, 0, K_LIST, (uint32_t)cnt_chunk);
        if (lane == 0) atomicAdd(&st[S_ITEMS], (unsigned long long)nit);
      } else {
        crec = make_rec(lr, 0, K_FALLBACK, (uint32_t)cnt_chunk);
        if (lane == 0) atomicAdd(&st[S_POOL_OVERFLOW], 1ull);
      }
    }
    if (lane == 0) {
      s_chunk[w] = crec;
      stcg_rec(p.chunk_rec + t * kWarps + w, crec);
    }
    __threadfence();
    __syncthreads();

    // ---- 6. the tile's record, and the sum's completion count
    if (tid == 0) {
      bool all_run = true;
      int et = kZeroE;
      for (int k = 0; k < kWarps; k++) {
        const Rec &c = s_chunk[k];
        if (rec_kind(c.meta) != K_RUN) { all_run = false; break; }
        if (rec_flags(c.meta) & F_ZERO) continue;
        if (et == kZeroE) et = c.e;
        else if (c.e != et) { all_run = false; break; }
      }
      Rec tr;
      if (all_run) {
        Run acc = run_empty();
        for (int k = 0; k < kWarps; k++) acc = run_compose(acc, rec_run(s_chunk[k]));
        tr = make_rec(acc, (acc.flags & F_ZERO) ? kZeroE : et, K_RUN, 0);
      } else {
        uint32_t orf = 0;
        for (int k = 0; k < kWarps; k++) orf |= rec_flags(s_chunk[k].meta);
        Run z = run_empty();
        z.flags = orf & (F_HASINF_P | F_HASINF_N | F_HASNAN);
        tr = make_rec(z, 0, K_COMPLEX, 0);
      }
      stcg_rec(p.tile_rec + t, tr);
      atomicAdd(&st[S_TILES], 1ull);
      __threadfence();
      const uint32_t prev = atomicAdd(&p.done[g.sum], 1u);
      if (prev + 1 == (uint32_t)g.ntiles_sum) s_pend[s_npend++] = t;
    }
    __syncthreads();
    if (hold) {                              // no ticket held: walk now, then take the next
      flush_walks();
      if (tid == 0) issue(cur ^ 1);
    }
    __syncthreads();
    cur ^= 1;
  }

  // ---- statistics and the last CTA's reset of the shared counters
  __syncthreads();
  if (tid < S_COUNT && s_st[tid]) atomicAdd(&p.stats[tid], s_st[tid]);
  if (tid == 0) {
    __threadfence();
    if (atomicAdd(&p.ctr[C_EXIT], 1u) + 1 == gridDim.x) {
      p.ctr[C_TICKET] = 0;
      p.ctr[C_EXIT] = 0;
      p.ctr[C_POOL] = 0;
      __threadfence();
    }
  }
}

// Batched set-up: tiles per sum, their prefix (tile_begin), the start value of
// empty sums, and the per-sum tile counters.  Offsets out of order or outside
// [0, x_len] (x_len = p.n) stop the call: every output becomes NaN.
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
      p.done[k] = 0;
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
  seqsum_kernel<<<grid, kThreads, kDynSmem, st>>>(p, *tmap);
  return cudaGetLastError();
}

cudaError_t launch_setup(const Params &p, cudaStream_t st) {
  setup_kernel<<<1, 1024, 0, st>>>(p);
  return cudaGetLastError();
}

int kernel_max_blocks_per_sm() {
  cudaFuncSetAttribute(seqsum_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kDynSmem);
  int nb = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, seqsum_kernel, kThreads, kDynSmem) != cudaSuccess)
    return 1;
  return nb > 0 ? nb : 1;
}

}  // namespace sq

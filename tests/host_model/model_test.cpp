// Host unit test of the product's exact-math header (binade_math.cuh), the
// same code the CUDA kernels run.  It checks the method against the host's
// own binary64 add (compiled strict-fp), which is independent of the header:
//
//   1. the one-term rule: applying the increment of one term to S gives
//      exactly S + x whenever the walk's check accepts it, on random and
//      adversarial pairs (ties, binade edges, negative S, subnormal terms);
//   2. the streaming kernel's fast rule: half-up increments with a one-word
//      tie detector (term_mag_halfup) against term_inc;
//   3. the whole pipeline in the kernels' layout (lanes of 16 terms, warps of
//      32 lanes composed in a tree), walked with the term-by-term fallback,
//      against the plain loop, under several plans: the true binade, one
//      binade too high, all "zero", one fixed binade, all chunks term by term,
//      and random (Research-1433, finding 5 "The plan cannot make the result
//      wrong");
//   4. the streaming kernel's composition: rows of 16 terms by the fast rule
//      (signed rows bounded by their negative and positive parts, rows with a
//      tie by the exact rule), a tile of rows of one binade composed by plain
//      sums, walked with row and term fallbacks under the same plans.
//
// Built with -DSEQSUM_MUTATE=k it must FAIL (exit status != 0) for each
// planted mistake k (Research-1433, "Tests": always round a tie up, drop the
// binade check, drop the upper bound check, ignore the parity).
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <vector>

#include "../../parity_binade_chunked_gb300/csrc/binade_math.cuh"

using namespace sq;

static uint64_t g_state = 0x1234567;
static uint64_t rnd() {               // splitmix64
  uint64_t z = (g_state += 0x9E3779B97F4A7C15ull);
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}
static uint64_t bits(double v) { uint64_t b; memcpy(&b, &v, 8); return b; }
static double dbl(uint64_t b) { double v; memcpy(&v, &b, 8); return v; }
static double mk(int exp, uint64_t frac53, bool neg) {      // (frac53 | 2^52) * 2^(exp-52)
  uint64_t b = ((uint64_t)(exp + 1023) << 52) | (frac53 & kFracMask);
  return neg ? -dbl(b) : dbl(b);
}
static double seq_add(double a, double b) { volatile double s = a; s = s + b; return s; }

static long g_fail = 0;

// ------------------------------------------------------------ one-term rule
static void check_one(double S, double x, long &accepted, long &checked) {
  uint64_t Sb = bits(S);
  int e = binade_of_bits(Sb);
  int64_t re; int32_t d;
  bool poison = term_inc(bits(x), e, re, d);
  Run r = run_empty();
  run_push(r, re, d, term_flags(bits(x)) | (poison ? F_POISON : 0u));
  uint64_t T = Sb;
  checked++;
  if (run_apply(T, r, e) == APPLY_OK) {
    accepted++;
    double want = seq_add(S, x);
    if (T != bits(want)) {
      if (g_fail < 10)
        fprintf(stderr, "one-term mismatch: S=%a x=%a got=%a want=%a\n", S, x, dbl(T), want);
      g_fail++;
    }
  }
}

static void test_one_term(long count) {
  long acc = 0, chk = 0;
  for (long i = 0; i < count; i++) {
    uint64_t a = rnd(), b = rnd();
    int e = (int)(a % 200) - 100;
    double S;
    switch (b % 8) {
      case 0: S = mk(e, (uint64_t)0, false); break;                       // S = 2^e
      case 1: S = mk(e, kFracMask, false); break;                         // just below 2^(e+1)
      case 2: S = mk(e, (rnd() % 16), false); break;                      // near the bottom
      case 3: S = mk(e, kFracMask - (rnd() % 16), false); break;          // near the top
      default: S = mk(e, rnd(), false); break;
    }
    if (rnd() & 1) S = -S;
    // term: random offset below the binade, with tie-shaped and exact cases
    int ex = e - 1 - (int)(rnd() % 60);
    double x;
    uint64_t c = rnd() % 10;
    if (c == 0) x = ldexp((double)(rnd() % 64) + 0.5, e - 52);           // k + 1/2 units: a tie
    else if (c == 1) x = ldexp((double)(rnd() % 1024), e - 52);          // whole units
    else if (c == 2) x = ldexp((double)(rnd() % 2048), e - 53 - (int)(rnd() % 3));
    else if (c == 3) x = dbl(rnd() % (1ull << 52));                        // subnormal
    else if (c == 4) x = 0.0;
    else x = mk(ex, rnd(), false);
    if (rnd() & 1) x = -x;
    check_one(S, x, acc, chk);
    // also a term of the same size as S (poison for this binade)
    if ((i & 15) == 0) check_one(S, mk(e, rnd(), (rnd() & 1) != 0), acc, chk);
  }
  printf("one-term: %ld checked, %ld accepted\n", chk, acc);
  if (acc < chk / 2) { fprintf(stderr, "too few accepted\n"); g_fail++; }
}

// --------------------------------------------------------- fast increment
// term_inc_fast (the kernels' common path) against term_inc on random terms
// and binades with e >= -969 and |x| < 2^e, including ties and zeros.
static void test_fast_increment(long count) {
  long n = 0;
  for (long i = 0; i < count; i++) {
    const int e = (int)(rnd() % 1990) - 969;
    double x;
    const uint64_t c = rnd() % 8;
    if (c == 0) x = 0.0;
    else if (c == 1) x = dbl(rnd() % (1ull << 52));                                  // subnormal
    else if (c == 2) x = ldexp((double)(rnd() % 4096) + 0.5, e - 52 - (int)(rnd() % 12));
    else if (c == 3) x = mk(e - 1, rnd(), false);                                      // just below 2^e
    else x = mk(e - 1 - (int)(rnd() % 80), rnd(), false);
    if (!(fabs(x) < ldexp(1.0, e))) continue;
    const uint64_t b = bits(x);
    int64_t re; int32_t d;
    if (term_inc(b, e, re, d)) continue;
    uint64_t r; bool tie;
    term_inc_fast((uint32_t)(b >> 32), (uint32_t)b, 64 - (e + 1023), r, tie);
    // term_inc gives re = f + up + (tie ? f & 1 : 0) and d = tie ? (f odd ? -1 : 1) : 0
    bool ok;
    if (tie) ok = (d != 0) && ((int64_t)r + (d < 0 ? 1 : 0) == re || (int64_t)r == re);
    else ok = (d == 0) && ((int64_t)r == re);
    if (tie) ok = ok && (d != 0);
    if (!tie && d != 0) ok = false;
    // exact relation at a tie: f = r (rounded down), re = f + (f & 1)
    if (tie) ok = (re == (int64_t)(r + (r & 1))) && (d == ((r & 1) ? -1 : 1));
    n++;
    if (!ok) {
      if (g_fail < 10)
        fprintf(stderr, "fast increment mismatch: x=%a e=%d r=%llu tie=%d re=%lld d=%d\n", x, e,
                (unsigned long long)r, (int)tie, (long long)re, d);
      g_fail++;
    }
  }
  printf("fast increment: %ld checked\n", n);
}

// ----------------------------------------------------- half-up increment
// term_mag_halfup (the streaming pass) against term_inc: away from a tie the
// two agree; at a tie (t == 0) the half-up value is the floor plus one, and
// term_inc's even-start value and odd-start difference follow from the floor.
static void test_halfup_increment(long count) {
  long n = 0, ties = 0;
  for (long i = 0; i < count; i++) {
    const int e = (int)(rnd() % 1990) - 969;
    double x;
    const uint64_t c = rnd() % 8;
    if (c == 0) x = 0.0;
    else if (c == 1) x = dbl(rnd() % (1ull << 52));                                  // subnormal
    else if (c == 2) x = ldexp((double)(rnd() % 4096) + 0.5, e - 52 - (int)(rnd() % 12));
    else if (c == 3) x = mk(e - 1, rnd(), false);                                      // just below 2^e
    else if (c == 4) x = ldexp((double)(rnd() % (1ull << 40)), e - 52 - (int)(rnd() % 50));
    else x = mk(e - 1 - (int)(rnd() % 80), rnd(), false);
    if (rnd() & 1) x = -x;
    if (!(fabs(x) < ldexp(1.0, e))) continue;
    const uint64_t b = bits(x);
    int64_t re; int32_t d;
    if (term_inc(b & ~kSignBit, e, re, d)) continue;       // the magnitude's increment
    uint32_t t;
    const uint64_t r = term_mag_halfup((uint32_t)(b >> 32), (uint32_t)b, 64 - (e + 1023), t);
    bool ok;
    if (t != 0) ok = (d == 0) && ((int64_t)r == re);
    else {
      ties++;
      const uint64_t f = r - 1;
      ok = (re == (int64_t)(f + (f & 1))) && (d == ((f & 1) ? -1 : 1));
    }
    n++;
    if (!ok) {
      if (g_fail < 10)
        fprintf(stderr, "half-up increment mismatch: x=%a e=%d r=%llu t=%u re=%lld d=%d\n", x, e,
                (unsigned long long)r, t, (long long)re, d);
      g_fail++;
    }
  }
  printf("half-up increment: %ld checked, %ld ties\n", n, ties);
}

// ------------------------------------------------------------- short runs
// Runs of 1..12 terms, built term by term and also as two composed halves,
// applied to S under its own binade and under a neighbouring one.
static void test_short_runs(long count) {
  long acc = 0, chk = 0;
  for (long i = 0; i < count; i++) {
    int e = (int)(rnd() % 120) - 60;
    double S = mk(e, (rnd() % 4 == 0) ? kFracMask - (rnd() % 64) : rnd(), (rnd() & 3) == 0);
    int k = 1 + (int)(rnd() % 12);
    double x[12];
    for (int j = 0; j < k; j++) {
      uint64_t c = rnd() % 4;
      if (c == 0) x[j] = ldexp((double)(rnd() % 16) + 0.5, e - 52);        // tie-shaped
      else if (c == 1) x[j] = ldexp((double)(rnd() % 64), e - 53);
      else if (c == 2) x[j] = ldexp((double)(rnd() % 8) + 0.25, e - 52);
      else x[j] = mk(e - 1 - (int)(rnd() % 20), rnd(), false);
      if ((rnd() % 5) == 0) x[j] = -x[j];
    }
    int ep = e + ((rnd() % 8) == 0 ? ((rnd() & 1) ? 1 : -1) : 0);
    int split = (int)(rnd() % (uint64_t)(k + 1));
    Run a = run_empty(), b = run_empty(), whole = run_empty();
    for (int j = 0; j < k; j++) {
      int64_t re; int32_t d;
      bool p = term_inc(bits(x[j]), ep, re, d);
      uint32_t tf = term_flags(bits(x[j])) | (p ? F_POISON : 0u);
      run_push(whole, re, d, tf);
      if (j < split) run_push(a, re, d, tf);
      else run_push(b, re, d, tf);
    }
    Run comp = split == 0 ? b : (split == k ? a : run_compose(a, b));
    double want = S;
    for (int j = 0; j < k; j++) want = seq_add(want, x[j]);
    for (int which = 0; which < 2; which++) {
      uint64_t T = bits(S);
      chk++;
      if (run_apply(T, which ? comp : whole, ep) == APPLY_OK) {
        acc++;
        if (T != bits(want)) {
          if (g_fail < 10)
            fprintf(stderr, "short-run mismatch: S=%a k=%d got=%a want=%a\n", S, k, dbl(T), want);
          g_fail++;
        }
      }
    }
  }
  printf("short runs: %ld checked, %ld accepted\n", chk, acc);
}

// ----------------------------------------------------------- pipeline model
// The layout of the kernels: lanes of LANE terms, warps of 32 lanes combined
// in a fixed shuffle tree, tiles of WARPS warps.
static const int LANE = 16, WARP_T = 32 * LANE;

struct Rec { Run r; int e; int kind; };   // kind: 0 run, 1 fall back

static Run lane_run(const double *x, int n, int e) {
  Run r = run_empty();
  for (int i = 0; i < n; i++) {
    int64_t re; int32_t d;
    bool poison = term_inc(bits(x[i]), e, re, d);
    run_push(r, re, d, term_flags(bits(x[i])) | (poison ? F_POISON : 0u));
  }
  return r;
}

static Run warp_tree(std::vector<Run> lanes) {      // shfl_down tree, in order
  for (int off = 1; off < 32; off <<= 1)
    for (int l = 0; l + off < 32; l += 2 * off)
      lanes[l] = run_compose(lanes[l], lanes[l + off]);
  return lanes[0];
}

// walk one chunk record, falling back to the plain loop on failure
static uint64_t walk(const std::vector<double> &x, double s0, int plan_kind, long &fallbacks) {
  uint64_t S = bits(s0);
  const size_t n = x.size();
  // approximate prefix for the plan (plain double sums of chunks, as a plan would)
  double approx = s0;
  for (size_t c0 = 0; c0 < n; c0 += WARP_T) {
    size_t c1 = c0 + WARP_T < n ? c0 + WARP_T : n;
    double cs = 0;
    for (size_t i = c0; i < c1; i++) cs += x[i];
    int e;
    switch (plan_kind) {
      case 0: e = binade_of_bits(bits(approx)); break;           // plan from the prefix
      case 1: e = binade_of_bits(bits(approx)) + 1; break;        // one binade too high
      case 2: e = -1023; break;                                    // "all zero"
      case 3: e = 3; break;                                        // one fixed binade
      case 4: e = 99999; break;                                    // all term by term
      default: e = binade_of_bits(bits(approx)) + (int)(rnd() % 3) - 1; break;
    }
    approx += cs;
    std::vector<Run> lanes(32, run_empty());
    for (int l = 0; l < 32; l++) {
      size_t a = c0 + (size_t)l * LANE;
      if (a < c1) lanes[l] = lane_run(&x[a], (int)((c1 - a) < (size_t)LANE ? (c1 - a) : LANE), e);
    }
    Run chunk = warp_tree(lanes);
    if (plan_kind == 4 || run_apply(S, chunk, e) != APPLY_OK) {
      fallbacks++;
      double s = dbl(S);
      for (size_t i = c0; i < c1; i++) s = seq_add(s, x[i]);
      S = bits(s);
    }
  }
  return S;
}

static std::vector<double> gen(int kind, size_t n) {
  std::vector<double> x(n);
  for (size_t i = 0; i < n; i++) {
    uint64_t a = rnd();
    double v;
    switch (kind) {
      case 0: v = (double)((a >> 11) | 1) * 0x1p-53 * 65536.0; break;                   // c1-like
      case 1: v = 1.0 - (double)((a >> 12) | (1ull << 52)) * 0x1p-53; break;           // c2-like ties
      case 2: v = ldexp(1.0 + (double)(a >> 12) * 0x1p-52, -(int)(rnd() % 41)); break;   // c3-like
      case 3: v = 65536.0 * (0.9 + 0.1 * (double)(a >> 11) * 0x1p-53) *
                  ((rnd() % 50) == 0 ? -0.2 : 1.0); break;                               // c5-like signed
      case 4: v = (a % 7 == 0) ? 0.0 : ldexp((double)(a % 5), -53); break;               // dense ties
      case 5: v = ldexp((double)(a >> 11), -(int)(rnd() % 8)) * ((a & 1) ? 1 : -1); break;  // cancelling
      case 6: v = (a % 3 == 0) ? -0.0 : 0.0; break;                                       // zeros
      case 7: v = dbl(a % (1ull << 53)) * ((a >> 63) ? -1.0 : 1.0); break;                // subnormal/tiny
      case 8: v = ldexp(1.0 + (double)(a >> 12) * 0x1p-52, 900 + (int)(rnd() % 123)); break; // near overflow
      default: v = (double)(a % 1000); break;                                             // integers
    }
    x[i] = v;
  }
  return x;
}

static void test_pipeline() {
  const double starts[] = {0.0, -0.0, 1.0, -1.0, 12345.678, 0x1p-1070, -3.0e9};
  long total = 0, fb = 0;
  for (int kind = 0; kind < 10; kind++)
    for (int plan = 0; plan < 6; plan++)
      for (int rep = 0; rep < 3; rep++) {
        size_t n = 1 + (size_t)(rnd() % 6000);
        std::vector<double> x = gen(kind, n);
        double s0 = starts[rnd() % 7];
        double want = s0;
        for (size_t i = 0; i < n; i++) want = seq_add(want, x[i]);
        long f = 0;
        uint64_t got = walk(x, s0, plan, f);
        fb += f;
        total++;
        bool same = (got == bits(want)) || (want != want && dbl(got) != dbl(got));
        if (!same) {
          if (g_fail < 10)
            fprintf(stderr, "pipeline mismatch kind=%d plan=%d n=%zu got=%a want=%a\n",
                    kind, plan, n, dbl(got), want);
          g_fail++;
        }
      }
  printf("pipeline: %ld sums, %ld chunk fallbacks\n", total, fb);
}

// ----------------------------------------------- the streaming composition
// A row as the streaming kernel forms it: all zeros exactly; else the fast
// rule (half-up increments, signed rows bounded by [-negatives, positives]),
// or the exact rule when a tie is detected.
static Run row_kernel(const double *x, int n, int e, bool &tie) {
  tie = false;
  bool zero = true, allneg = true;
  for (int i = 0; i < n; i++) {
    zero = zero && (bits(x[i]) << 1) == 0;
    allneg = allneg && (bits(x[i]) >> 63);
  }
  if (zero) {
    Run r = run_empty();
    r.lo = r.hi = 0;
    r.flags = F_NONNEG | F_NONPOS | F_ZERO | (allneg ? F_ALLNEGZ : 0u);
    return r;
  }
  uint64_t tot = 0, ng = 0;
  uint32_t tmin = ~0u, emax = 0;
  bool anyneg = false;
  for (int i = 0; i < n; i++) {
    const uint64_t b = bits(x[i]);
    const uint32_t hi = (uint32_t)(b >> 32);
    uint32_t t;
    const uint64_t r = term_mag_halfup(hi, (uint32_t)b, 64 - (e + 1023), t);
    tmin = t < tmin ? t : tmin;
    const uint32_t E = (hi >> 20) & 0x7FFu;
    emax = E > emax ? E : emax;
    const uint64_t sm = (hi >> 31) ? ~0ull : 0ull;
    anyneg = anyneg || (hi >> 31);
    tot += r;
    ng += r & sm;
  }
  if (tmin == 0) {
    tie = true;
    return lane_run(x, n, e);
  }
  Run r;
  r.inc = (int64_t)(tot - 2 * ng);
  r.lo = -(int64_t)ng;
  r.hi = (int64_t)(tot - ng);
  r.d = 0;
  r.flags = (anyneg ? 0u : (uint32_t)F_NONNEG) | (emax >= (uint32_t)(e + 1023) ? (uint32_t)F_POISON : 0u);
  const int64_t lim = (int64_t)1 << 54;
  if (r.inc > lim || r.inc < -lim || r.hi > lim || r.lo < -lim) r.flags |= F_POISON;
  return r;
}

static uint64_t add_terms(uint64_t S, const double *x, int n) {
  double s = dbl(S);
  for (int i = 0; i < n; i++) s = seq_add(s, x[i]);
  return bits(s);
}

static uint64_t walk_kernel(const std::vector<double> &x, double s0, int plan_kind, long &fast_tiles) {
  const int ROWS = 8, TT = ROWS * LANE;
  uint64_t S = bits(s0);
  double approx = s0;
  const size_t n = x.size();
  for (size_t t0 = 0; t0 < n; t0 += TT) {
    int e[ROWS];
    Run rr[ROWS];
    bool tie[ROWS], ok_rows = true;
    int nr = 0;
    for (int r = 0; r < ROWS && t0 + (size_t)r * LANE < n; r++, nr++) {
      const size_t a = t0 + (size_t)r * LANE;
      const int m = (int)((n - a) < (size_t)LANE ? (n - a) : LANE);
      switch (plan_kind) {
        case 0: e[r] = binade_of_bits(bits(approx)); break;
        case 1: e[r] = binade_of_bits(bits(approx)) + 1; break;
        case 2: e[r] = -200; break;
        case 3: e[r] = 3; break;
        case 4: e[r] = 99999; break;
        default: e[r] = binade_of_bits(bits(approx)) + (int)(rnd() % 3) - 1; break;
      }
      for (int i = 0; i < m; i++) approx += x[a + i];
      if (e[r] < -900 || e[r] > 1000) { ok_rows = false; continue; }
      rr[r] = row_kernel(&x[a], m, e[r], tie[r]);
      if (tie[r] || e[r] != e[0]) ok_rows = false;
    }
    if (ok_rows && plan_kind != 4) {
      // one run for the tile: plain sums of the rows, flags combined
      Run h;
      h.inc = h.lo = h.hi = 0;
      h.d = 0;
      uint32_t fand = 0xFF, fo = 0;
      for (int r = 0; r < nr; r++) {
        h.inc += rr[r].inc;
        h.lo += rr[r].lo;
        h.hi += rr[r].hi;
        fand &= rr[r].flags & (F_NONNEG | F_NONPOS | F_ZERO | F_ALLNEGZ);
        fo |= rr[r].flags & F_POISON;
      }
      h.flags = fand | fo;
      uint64_t T = S;
      if (run_apply(T, h, e[0]) == APPLY_OK) {
        fast_tiles++;
        S = T;
        continue;
      }
    }
    for (int r = 0; r < nr; r++) {
      const size_t a = t0 + (size_t)r * LANE;
      const int m = (int)((n - a) < (size_t)LANE ? (n - a) : LANE);
      uint64_t T = S;
      if (plan_kind != 4 && e[r] >= -900 && e[r] <= 1000 && run_apply(T, rr[r], e[r]) == APPLY_OK) S = T;
      else S = add_terms(S, &x[a], m);
    }
  }
  return S;
}

static void test_kernel_composition() {
  const double starts[] = {0.0, -0.0, 1.0, -1.0, 12345.678, 0x1p-1070, -3.0e9};
  long total = 0, fast = 0;
  for (int kind = 0; kind < 10; kind++)
    for (int plan = 0; plan < 6; plan++)
      for (int rep = 0; rep < 4; rep++) {
        size_t n = 1 + (size_t)(rnd() % 6000);
        std::vector<double> x = gen(kind, n);
        double s0 = starts[rnd() % 7];
        double want = s0;
        for (size_t i = 0; i < n; i++) want = seq_add(want, x[i]);
        uint64_t got = walk_kernel(x, s0, plan, fast);
        total++;
        bool same = (got == bits(want)) || (want != want && dbl(got) != dbl(got));
        if (!same) {
          if (g_fail < 10)
            fprintf(stderr, "kernel composition mismatch kind=%d plan=%d n=%zu got=%a want=%a\n",
                    kind, plan, n, dbl(got), want);
          g_fail++;
        }
      }
  printf("kernel composition: %ld sums, %ld tiles applied as one run\n", total, fast);
}

int main(int argc, char **argv) {
  long count = argc > 1 ? atol(argv[1]) : 2000000;
  test_one_term(count);
  test_fast_increment(count);
  test_halfup_increment(count);
  test_short_runs(count / 2);
  test_pipeline();
  test_kernel_composition();
  printf("mutation=%d failures=%ld\n", kMutate, g_fail);
  return g_fail ? 1 : 0;
}

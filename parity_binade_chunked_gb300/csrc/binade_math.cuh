// Exact integer arithmetic of a run of binary64 adds that stays inside one
// binade -- shared by the CUDA kernels and by the host-side unit tests of this
// header (it compiles as plain C++ as well).  It is NOT the oracle.
//
// The rule (Research-1433, "Forming the CPU's sequential double sums on a GPU,
// bit for bit", finding 2 "Inside a binade the loop is an integer sum"; and
// Research-1424, section 3 "An exact sum that stays on the device"):
//   a running sum S in [2^e, 2^(e+1)) is m * u with u = 2^(e-52) and
//   m in [2^52, 2^53).  fl(S + x) = (m + r) * u, r = x / u rounded to an
//   integer, as long as every intermediate result stays in the binade.  So a
//   run of adds is an integer sum of increments, which can be grouped at will.
//
// Ties (finding 3, "Ties need the parity of the running integer"): when x / u
// is exactly half way, the add rounds to the even result, so r depends on the
// parity of the running count.  Every term and every run therefore carries an
// increment for an even and for an odd starting count; two runs compose by
// taking the second run's increment for the parity the first leaves, which is
// associative but not commutative.
//
// Signed terms (Research-1424, section 3): the run also carries the smallest
// and largest prefix of its integer sum; the walk accepts the run only when
// S/u plus those prefixes stays inside [2^52 + 1, 2^53 - 1].  For runs of
// non-negative terms the final count alone bounds every intermediate value
// (Research-1433, finding 4), and a count of exactly 2^53 is the binade's
// upper end 2^(e+1), which is still exact.
//
// Representation used here: `inc` is the increment for an even start, `d` is
// inc_odd - inc_even (always -1, 0 or +1), and [lo, hi] bounds every
// non-empty prefix of the even-start increments.  The odd-start prefixes are
// within one of the even-start ones, so [lo - 1, hi + 1] bounds them.
#pragma once
#include <stdint.h>

#if defined(__CUDACC__)
#define SQ_HD __host__ __device__ __forceinline__
#else
#define SQ_HD static inline
#endif

namespace sq {

// ---------------------------------------------------------------- constants
static constexpr uint64_t kFracMask = (1ull << 52) - 1;
static constexpr uint64_t kHidden = 1ull << 52;
static constexpr uint64_t kSignBit = 1ull << 63;
static constexpr int64_t kTwo52 = (int64_t)1 << 52;
static constexpr int64_t kTwo53 = (int64_t)1 << 53;
// any |inc|, |lo|, |hi| beyond this can never pass the walk's check
static constexpr int64_t kSat = (int64_t)1 << 55;

// run flags
enum : uint32_t {
  F_POISON = 1u,       // a term with |x| >= 2^e, inf or NaN: the run can never apply
  F_NONNEG = 2u,       // no term with the sign bit set and a non-zero magnitude
  F_NONPOS = 4u,       // no term with a clear sign bit and a non-zero magnitude
  F_ZERO = 8u,         // every term is +0 or -0
  F_ALLNEGZ = 16u,     // every term is -0 (only meaningful with F_ZERO)
  F_HASINF_P = 32u,    // contains +inf
  F_HASINF_N = 64u,    // contains -inf
  F_HASNAN = 128u,     // contains a NaN
};

#ifdef SEQSUM_MUTATE
// Planted mistakes for the host tests: each must make the test suite fail.
//   1: a tie always rounds up          2: the binade check is dropped
//   3: the upper bound check is dropped 4: composition ignores the parity
static constexpr int kMutate = SEQSUM_MUTATE;
#else
static constexpr int kMutate = 0;
#endif

struct Run {
  int64_t inc;    // increment of the count for an even start
  int64_t lo;     // lower bound of the even-start non-empty prefixes
  int64_t hi;     // upper bound of the even-start non-empty prefixes
  int32_t d;      // inc_odd - inc_even, in {-1, 0, 1}
  uint32_t flags;
};

// The empty run: no terms.  It is the identity of run_compose, and applied
// on its own it leaves S unchanged (it is flagged as a run of zeros whose
// terms are all -0, which keeps a -0 sum at -0).
static constexpr int64_t kEmptyLo = (int64_t)1 << 60;
SQ_HD Run run_empty() {
  Run r;
  r.inc = 0; r.lo = kEmptyLo; r.hi = -kEmptyLo; r.d = 0;
  r.flags = 2u | 4u | 8u | 16u;   // F_NONNEG | F_NONPOS | F_ZERO | F_ALLNEGZ
  return r;
}

// Flags of one term, independent of the binade.
SQ_HD uint32_t term_flags(uint64_t tb) {
  const uint64_t mag = tb & ~kSignBit;
  const bool neg = (tb >> 63) != 0;
  uint32_t f = 0;
  if (mag == 0) {
    f = F_NONNEG | F_NONPOS | F_ZERO | (neg ? F_ALLNEGZ : 0u);
  } else {
    f = neg ? F_NONPOS : F_NONNEG;
    if (mag >= 0x7FF0000000000000ull) {
      f |= F_POISON;
      if (mag == 0x7FF0000000000000ull) f |= neg ? F_HASINF_N : F_HASINF_P;
      else f |= F_HASNAN;
    }
  }
  return f;
}

// The per-term increment under binade e (the unbiased exponent of |S|):
// r = x / 2^(e-52), from the 53-bit significand M shifted right by
// s = e - exponent(x), rounded on the shifted-out bits.  No floating-point
// operation.  re is the increment for an even running count, re + d for an
// odd one.  Returns true when the term is "poison" for this binade
// (|x| >= 2^e, or inf/NaN): no run containing it can apply.
SQ_HD bool term_inc(uint64_t tb, int e, int64_t &re, int32_t &d) {
  const uint32_t E = (uint32_t)(tb >> 52) & 0x7FFu;
  const uint64_t F = tb & kFracMask;
  const uint64_t M = E ? (F | kHidden) : F;
  const int xe = E ? (int)E - 1023 : -1022;
  int s = e - xe;
  const bool poison = (s <= 0) || (E == 0x7FFu);
  s = s < 1 ? 1 : (s > 63 ? 63 : s);          // s >= 54 gives r = 0 either way
  const uint64_t f = M >> s;
  const uint64_t L = M << (64 - s);            // shifted-out bits, left aligned
  const bool tie = (L == kSignBit);
  const bool up = (L > kSignBit);
  const uint64_t f1 = f & 1ull;
  uint64_t r;
  int32_t t;
  if (kMutate == 1) {                          // mutation: ties always round up
    r = f + ((up || tie) ? 1u : 0u);
    t = 0;
  } else {
    // even start: the tie goes to the even count, i.e. to an even r
    r = f + (up ? 1u : 0u) + (tie ? f1 : 0u);
    t = tie ? (f1 ? -1 : 1) : 0;
  }
  const bool neg = (tb >> 63) != 0;
  re = neg ? -(int64_t)r : (int64_t)r;         // RNE is symmetric in the sign
  d = neg ? -t : t;
  return poison;
}

// Append one term (increment re, tie difference t, flags tf) to a run, in
// order.  The even-start path is tracked exactly, so lo/hi are exact here.
SQ_HD void run_push(Run &a, int64_t re, int32_t t, uint32_t tf) {
  const int q = (int)(a.inc & 1);              // parity after the run so far (even start)
  const int32_t adj = (kMutate == 4) ? 0 : (q ? t : 0);
  a.inc += re + adj;
  if (a.d == 0) a.d = (kMutate == 4) ? t : (q ? -t : t);
  a.lo = a.inc < a.lo ? a.inc : a.lo;
  a.hi = a.inc > a.hi ? a.inc : a.hi;
  a.flags = (a.flags & tf & (F_NONNEG | F_NONPOS | F_ZERO | F_ALLNEGZ)) |
            ((a.flags | tf) & (F_POISON | F_HASINF_P | F_HASINF_N | F_HASNAN));
}

// The same increment for a term whose sign is handled by the caller, in the
// common case: binade e with e >= -969 and |x| < 2^e (s >= 1).  hi/lo are the
// term's two 32-bit halves; c = 64 - (e + 1023).  r = x / 2^(e-52) rounded
// half-up is returned in r (the even-start increment when `tie` is false);
// `tie` says the shifted-out bits were exactly one half.
//
// M * 2^(64-s) is formed with two 32x32->64 multiplies by 2^((64-s) mod 32):
// its upper 64 bits are M >> s and its lower 64 bits the shifted-out bits,
// left aligned.  Subnormal terms and zeros are treated as if they had the
// hidden bit; for e >= -969 that makes s >= 54 for them, where the result is
// r = 0 without a tie either way.
SQ_HD void term_inc_fast(uint32_t hi, uint32_t lo, int c, uint64_t &r, bool &tie) {
  const uint32_t E = (hi >> 20) & 0x7FFu;
  const uint32_t mh = (hi & 0xFFFFFu) | 0x100000u;
  int j = (int)E + c;                          // j = 64 - s, in [0, 63] (s > 64 clamps to 0)
  j = j < 0 ? 0 : j;
  const uint32_t w = 1u << (j & 31);
  const bool J = j >= 32;
  const uint64_t A = (uint64_t)lo * w, B = (uint64_t)mh * w;
  const uint32_t A0 = (uint32_t)A, A1 = (uint32_t)(A >> 32), B0 = (uint32_t)B, B1 = (uint32_t)(B >> 32);
  const uint32_t P = B0 | A1;
  const uint32_t Rh = J ? A0 : P;              // shifted-out bits, top word
  const bool Rl = !J && (A0 != 0);             // any shifted-out bit in the lower word
  tie = (Rh == 0x80000000u) && !Rl;
  const bool up = (Rh > 0x80000000u) || ((Rh == 0x80000000u) && Rl);
  const uint64_t f = J ? (((uint64_t)B1 << 32) | P) : (uint64_t)B1;
  r = f + (up ? 1u : 0u);
}

// The magnitude increment of one term rounded half up, with a tie detector,
// for the streaming pass: the same two multiplies as term_inc_fast, but the
// round-up decision is the top remainder bit alone and the tie test folds
// into one word.  hi/lo are the term's halves (the sign bit is ignored), c =
// 64 - (e + 1023) with e >= -969.  Returns r = round-half-up(|x| / 2^(e-52));
// `t` is zero exactly when the shifted-out bits are one half (a tie, where
// the correct increment depends on the parity and is r or r - 1).  When
// |x| >= 2^e the result is meaningless and the caller flags the term.
SQ_HD uint64_t term_mag_halfup(uint32_t hi, uint32_t lo, int c, uint32_t &t) {
  const uint32_t E = (hi >> 20) & 0x7FFu;
  const uint32_t mh = (hi & 0xFFFFFu) | 0x100000u;
  int j = (int)E + c;
  j = j < 0 ? 0 : j;
  const uint32_t w = 1u << (j & 31);
  const bool J = j >= 32;
  const uint64_t A = (uint64_t)lo * w, B = (uint64_t)mh * w;
  const uint32_t A0 = (uint32_t)A, A1 = (uint32_t)(A >> 32), B0 = (uint32_t)B, B1 = (uint32_t)(B >> 32);
  const uint32_t P = B0 | A1;
  const uint32_t Rh = J ? A0 : P;
  const uint32_t X = J ? 0u : A0;
  t = (Rh ^ 0x80000000u) | X;
  const uint64_t f = J ? (((uint64_t)B1 << 32) | P) : (uint64_t)B1;
  return f + (Rh >> 31);
}

SQ_HD int64_t sq_min(int64_t a, int64_t b) { return a < b ? a : b; }
SQ_HD int64_t sq_max(int64_t a, int64_t b) { return a > b ? a : b; }

// A then B (both computed for the same binade).  Associative in inc and d;
// lo/hi stay valid (possibly one unit wider per level when B starts odd).
SQ_HD Run run_compose(const Run &A, const Run &B) {
  Run c;
  const int q0 = (int)(A.inc & 1);
  const int32_t bd = (kMutate == 4) ? 0 : B.d;
  c.inc = A.inc + B.inc + (q0 ? bd : 0);
  c.d = A.d != 0 ? A.d : ((kMutate == 4) ? B.d : (q0 ? -B.d : B.d));
  c.lo = sq_min(A.lo, A.inc + B.lo - q0);
  c.hi = sq_max(A.hi, A.inc + B.hi + q0);
  c.flags = (A.flags & B.flags & (F_NONNEG | F_NONPOS | F_ZERO | F_ALLNEGZ)) |
            ((A.flags | B.flags) & (F_POISON | F_HASINF_P | F_HASINF_N | F_HASNAN));
  // saturate: a run whose increments leave +-2^55 can never pass the check
  if (c.inc > kSat || c.inc < -kSat || c.lo < -kSat || c.hi > kSat) {
    c.flags |= F_POISON;
    c.inc = sq_max(sq_min(c.inc, kSat), -kSat);
    c.lo = sq_max(c.lo, -kSat);
    c.hi = sq_min(c.hi, kSat);
  }
  return c;
}

// Outcome of offering a run to the exact running sum.
enum ApplyResult : int { APPLY_OK = 0, APPLY_FAIL = 1 };

// Apply a run computed for binade e to the exact running sum, given as its
// bit pattern.  On success the sum is updated in place.  The check is the
// walk's (Research-1433, finding 4; Research-1424, section 3):
//   * S must be a normal number in binade e;
//   * non-negative effective terms: m + inc <= 2^53;
//   * otherwise: m + lo >= 2^52 + 1 and m + hi <= 2^53 - 1 for every prefix.
// A negative S uses the mirrored run (the terms negated): RNE is symmetric.
// A run of zeros is a no-op on a non-zero S; on a zero S it follows the
// IEEE-754 sign rule (-0 stays -0 only if every term is -0).
SQ_HD ApplyResult run_apply(uint64_t &Sb, const Run &R, int e) {
  const uint64_t sign = Sb & kSignBit;
  uint64_t mag = Sb & ~kSignBit;
  if (R.flags & F_ZERO) {
    if (mag == 0) Sb = (sign && (R.flags & F_ALLNEGZ)) ? kSignBit : 0ull;
    return APPLY_OK;                           // S + (+-0) == S for S != 0 (and for inf/NaN)
  }
  if (R.flags & F_POISON) return APPLY_FAIL;
  const uint32_t Eb = (uint32_t)(mag >> 52);
  if (Eb == 0 || Eb == 0x7FFu) return APPLY_FAIL;     // zero, subnormal, inf, NaN
  if (kMutate != 2 && (int)Eb - 1023 != e) return APPLY_FAIL;
  const int64_t m = (int64_t)((mag & kFracMask) | kHidden);
  const int p = (int)(m & 1);
  int64_t inc, lo, hi;
  int32_t d;
  bool mono;
  if (!sign) { inc = R.inc; d = R.d; lo = R.lo; hi = R.hi; mono = (R.flags & F_NONNEG) != 0; }
  else { inc = -R.inc; d = -R.d; lo = -R.hi; hi = -R.lo; mono = (R.flags & F_NONPOS) != 0; }
  if (p) inc += d;
  bool ok;
  if (mono) ok = (kMutate == 3) ? true : (m + inc <= kTwo53);
  else ok = (m + lo - p >= kTwo52 + 1) && ((kMutate == 3) ? true : (m + hi + p <= kTwo53 - 1));
  if (!ok) return APPLY_FAIL;
  mag += (uint64_t)inc;                         // m stays in [2^52, 2^53]: the bits follow
  Sb = sign | mag;
  return APPLY_OK;
}

// Unbiased exponent of |v| for a normal number, from its bits (no FP op).
SQ_HD int binade_of_bits(uint64_t b) { return (int)((b >> 52) & 0x7FF) - 1023; }

}  // namespace sq

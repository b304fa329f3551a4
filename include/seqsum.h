/*
 * seqsum -- the exact bits of the CPU's sequential double sum, on one GB300.
 *
 * The result of every entry point is, bit for bit, what the plain loop
 *
 *     double s = s0;  for (i = 0; i < n; i++) s += x[i];
 *
 * returns under IEEE-754 binary64 round-to-nearest-even (Research-1433,
 * "Forming the CPU's sequential double sums on a GPU, bit for bit",
 * Question), the one exception being the payload bits of a NaN result.  The
 * device forms it without reading the terms back and without adding them on
 * one thread: runs of adds that stay inside one binade are integer sums of
 * increments (finding 2), ties carry an even/odd increment pair (finding 3),
 * and a chunk that leaves its binade is added term by term (finding 4).
 *
 * Memory: x, offsets, s0s, out and outs are DEVICE pointers, owned by the
 * caller and never freed by the library.  s0 is a host value.  The library
 * keeps one workspace per (device, stream), allocated on first use, grown on
 * demand and released by seqsum_release_workspace().
 *
 * Ordering: every call enqueues its work on `stream` (NULL = the legacy
 * default stream) and returns without waiting; the results are valid once the
 * stream reaches them.  The inputs must not change until then.  Calls that
 * share a (device, stream) pair are ordered by the stream; two host threads
 * must not call at the same time on the same stream.
 *
 * Errors: a negative return value; nothing is enqueued then.  Device-side
 * conditions (a bounded wait that gave up, a capacity overflow) are reported
 * by seqsum_get_stats().  No exception crosses this interface.
 */
#ifndef SEQSUM_H
#define SEQSUM_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;
typedef struct CUstream_st *cudaStream_t;

enum {
  SEQSUM_OK = 0,
  SEQSUM_EINVAL = -1,     /* null pointer with terms to add, n < 0, nsums < 0 */
  SEQSUM_ECUDA = -2,      /* a CUDA runtime call failed (see seqsum_last_cuda_error) */
  SEQSUM_ETIMEOUT = -3,   /* a device wait gave up (reported by seqsum_get_stats) */
  SEQSUM_ENOMEM = -4,     /* the workspace could not be allocated */
  SEQSUM_ECAPACITY = -5,  /* a batched call needed more tiles than its workspace holds, or n is above
                             SEQSUM_STATIC_MAX_TERMS for seqsum_f64_static */
  SEQSUM_EOFFSETS = -6    /* offsets out of order or out of range (seqsum_get_stats) */
};

/* One sequential sum: *out = s0 + x[0] + x[1] + ... + x[n-1], added in index
 * order (Research-1433, Question; Research-1424, section 1: calc_ssim()
 * carries one double through the whole frame, row after row).
 *   x      device, n doubles (any 8-byte alignment; 16-byte alignment enables
 *          the TMA path), read only
 *   n      number of terms, n >= 0; n == 0 writes s0's exact bits
 *   s0     the start value (host)
 *   out    device, one double, written
 *   stream CUDA stream the work is enqueued on
 * Returns SEQSUM_OK, SEQSUM_EINVAL, SEQSUM_ENOMEM or SEQSUM_ECUDA. */
int seqsum_f64(const double *x, int64_t n, double s0, double *out, cudaStream_t stream);

/* The largest n seqsum_f64_static accepts: 2^21 terms (512 tiles of 4096). */
#define SEQSUM_STATIC_MAX_TERMS (1 << 21)

/* As seqsum_f64, for n <= SEQSUM_STATIC_MAX_TERMS, on scratch held in
 * fixed-size device arrays of the library: the call allocates nothing (no
 * cudaMalloc, cudaFree or allocating library routine).  The pages describe no
 * such call -- it has no counterpart in the method; it exists for callers that
 * must not allocate.
 *   x, n, s0, out, stream  as for seqsum_f64
 * The first call on a device looks up the arrays' addresses and clears them
 * on `stream`; make that first call before any stream capture.  Every call on
 * a device shares the one scratch: calls that overlap in time (on different
 * streams, or from several host threads) race and give wrong results; order
 * them.  seqsum_get_stats() does not cover these calls.
 * Returns SEQSUM_OK, SEQSUM_EINVAL, SEQSUM_ECAPACITY (n too large; nothing is
 * enqueued) or SEQSUM_ECUDA. */
int seqsum_f64_static(const double *x, int64_t n, double s0, double *out, cudaStream_t stream);

/* nsums independent sequential sums over one concatenated plane: for each k,
 * outs[k] = s0s[k] + x[offsets[k]] + ... + x[offsets[k+1] - 1], in index order
 * (ADR-1391, Decision item 2 and 3: the 108 running sums of one ssimulacra2
 * frame, six per channel and scale; ADR-1464, Decision: one accumulator per
 * sum, the sums independent of one another).
 *   x        device, the concatenated terms, read only
 *   offsets  device, nsums + 1 int64 values, non-decreasing; sum k covers
 *            x[offsets[k] .. offsets[k+1])
 *   nsums    number of sums, >= 0
 *   s0s      device, nsums start values
 *   outs     device, nsums doubles, written
 * To size its workspace this entry reads offsets[0] and offsets[nsums] back
 * to the host once per call (one small copy and a wait on `stream`); use
 * seqsum_f64_batched_sized() to avoid that wait.
 * Returns SEQSUM_OK, SEQSUM_EINVAL, SEQSUM_ENOMEM or SEQSUM_ECUDA. */
int seqsum_f64_batched(const double *x, const int64_t *offsets, int32_t nsums, const double *s0s,
                       double *outs, cudaStream_t stream);

/* As seqsum_f64_batched, without any host wait.  x_len is the number of
 * doubles readable at x; every offset must lie in [0, x_len] and be
 * non-decreasing.  If not, the device writes NaN to every outs[k] and
 * seqsum_get_stats() reports SEQSUM_EOFFSETS. */
int seqsum_f64_batched_sized(const double *x, int64_t x_len, const int64_t *offsets, int32_t nsums,
                             const double *s0s, double *outs, cudaStream_t stream);

/* Counters accumulated on the device by the calls since the last
 * seqsum_get_stats() on the same (device, stream) workspace as the most
 * recent call of this process. */
typedef struct {
  int64_t tiles;             /* tiles of 4096 terms processed */
  int64_t chunks_run;        /* 512-term chunks that became one run */
  int64_t chunks_list;       /* chunks the plan split into several items */
  int64_t chunks_fallback;   /* chunks added term by term as a whole */
  int64_t lanes_dirty;       /* 16-term lanes the plan could not place */
  int64_t walk_segments;     /* composites the in-order walk applied (same-binade runs composed across groups) */
  int64_t runs_rejected;     /* runs the walk's exact check refused (fell back) */
  int64_t terms_added;       /* terms the walk added one by one in fp64 */
  int64_t items;             /* items written for split chunks */
  int64_t pool_overflow;     /* split chunks that found no room and fell back */
  int64_t tiles_complex;     /* tiles published with an item list (a split chunk, or chunks of several binades) */
  int64_t scan_windows;      /* windows of tile sums the plan's prefix scanner took */
  int64_t walk_batches;      /* batches the walk took tile by tile (groups too fragmented to compose, or refused) */
  int64_t ns_tma_wait;       /* nanoseconds, summed over CTAs: compute warps waiting for a unit */
  int64_t ns_prefix_wait;    /* not counted (always 0): a run unit's wait for a late prefix is in ns_verdict */
  int64_t ns_phase_a;        /* ... compute warps on plan units (the fixed-point sums of a tile) */
  int64_t ns_phase_b;        /* ... compute warps on run units (runs and items) */
  int64_t ns_walk_wait;      /* ... the walk waiting for tile headers */
  int64_t ns_walk_work;      /* ... the walk working */
  int64_t torn_header_reads; /* tile-header reads that saw words of two publications (retried) */
  int64_t torn_status_reads; /* prefix reads that saw words of two publications (retried) */
  int64_t ns_scan;           /* the prefix scanner's time from its first to its last window */
  int64_t ns_walk_count;     /* the tile-by-tile walk's work by section: counting a batch's elements */
  int64_t ns_walk_gather;    /* ... gathering headers and items into one list */
  int64_t ns_walk_scan;      /* ... composing same-binade segments in parallel */
  int64_t ns_walk_serial;    /* ... the in-order pass over the segments */
  int64_t ns_walk_adds;      /* ... of which term-by-term fp64 adds */
  int64_t chunks_dirty;      /* chunks whose prefix range spans two binades (placed lane by lane) */
  int64_t ns_ctrl_wait;      /* nanoseconds, summed: control warps waiting for their compute warps */
  int64_t ns_scan_wait;      /* nanoseconds: the prefix scanner waiting for tiles' sums */
  int64_t ns_verdict;        /* nanoseconds, summed: run units forming their chunks' verdicts */
  int64_t ns_verdict_wait;   /* nanoseconds, summed: run units reading plan words not copied in time */
  int64_t ns_group_count;    /* nanoseconds, summed: control warps counting tiles in their groups */
  int64_t ns_compose;        /* nanoseconds, summed: control warps composing the groups they completed */
  int64_t t_stream_ns;       /* latest call: kernel start to the last tile header */
  int64_t t_walk_tail_ns;    /* latest call: last tile header to the end of the walk */
  int64_t t_total_ns;        /* latest call: kernel start to the end of the walk */
  int32_t device_status;     /* 0, or a negative SEQSUM_E* code */
  int32_t device_error_bits; /* raw device error bits */
  int32_t check_site;        /* self-checking builds: first failed check (0: none) */
  int32_t check_pad;
  int64_t check_value;       /* self-checking builds: the value that failed it */
  int32_t timeout_site;      /* first bounded device wait that gave up (0: none) and its context */
  int32_t timeout_pad;
  int64_t timeout_a;
  int64_t timeout_b;
} seqsum_stats;

/* Waits for the stream of the most recent call, copies its workspace's
 * counters into *st and clears them.  Returns SEQSUM_OK or SEQSUM_ECUDA;
 * st->device_status carries device-side errors. */
int seqsum_get_stats(seqsum_stats *st);

/* A short English description of a return code (static storage). */
const char *seqsum_strerror(int code);

/* The cudaError_t of the last failed CUDA call (0 if none). */
int seqsum_last_cuda_error(void);

/* Frees every workspace of this process (waits for their streams first). */
void seqsum_release_workspace(void);

/* Test hook: force the plan of later calls (0 = the normal plan; 1 = one
 * binade too high, 2 = "all zero", 3 = one fixed binade, 4 = every chunk term
 * by term, 5 = random neighbouring binades).  Research-1433, finding 5: the
 * plan cannot make the result wrong, only slower.  Returns the old mode. */
int seqsum_debug_set_plan(int mode);

/* Test hook: copies up to 65536 diagnostic words that self-checking and
 * profiling builds of the library record (a trace of the walk, a timeline of
 * the units; zeros otherwise) and clears them. */
int seqsum_debug_read(unsigned long long *out, int n);

/* Diagnostics of a call that does not finish: copies the device counters of
 * the most recent call's workspace into out[0..16) and, per warp (index
 * CTA * 9 + warp: 8 compute warps, then the control warp), a heartbeat word into out[16..n) (role << 56 | what it
 * waits for or does << 48 | where).  It takes no lock and reads on a stream of its own, so it can run
 * while another thread waits on that call.  16 <= n <= 16 + 4096. */
int seqsum_debug_heartbeat(unsigned long long *out, int n);

/* Library version string. */
const char *seqsum_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SEQSUM_H */

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
 * Graphs: a call may be captured into a CUDA graph once the same entry has
 * run on the same stream with the same sizes (its workspace then exists, and
 * the capture allocates nothing).  Every launch takes its call tag from a
 * device counter that the kernel advances itself, so each replay is a call
 * of its own.  A captured seqsum_f64_planned call reads, on every replay,
 * the plan stored when it was captured (its results stay exact).
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
 * them.  seqsum_get_stats() does not cover these calls, and the test hooks
 * (seqsum_debug_set_plan, seqsum_debug_set_fault) do not reach them: a
 * device-side failure (a bounded wait that gave up) shows only as NaN in *out.
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

/* stride interleaved sequential sums over one plane, and their float means:
 * for each k < stride,
 *   outs[k] = s0s[k] + x[k] + x[k + stride] + ... + x[k + stride*(n-1)]
 * added in index order, and, when means is not null,
 *   means[k] = (float)(outs[k] / n)
 * (ADR-1464, "float_ssim_cuda sums in raster order on the host", Decision:
 * the lcs variant keeps four sums per window -- the value and its l, c and s
 * factors -- interleaved in one plane and summed with one accumulator each,
 * and the frame score is the float of the sum over the number of windows).
 *   x        device, stride * n doubles, interleaved (term i of sum k at i*stride + k), read only
 *   n        terms per sum (windows), n >= 0
 *   stride   number of sums, 1..64
 *   s0s      device, stride start values
 *   outs     device, stride doubles, written
 *   means    device, stride floats, written; or null
 * The sums are first copied apart into the workspace (one pass over x), then
 * summed as a batched call.  Returns SEQSUM_OK, SEQSUM_EINVAL, SEQSUM_ENOMEM or
 * SEQSUM_ECUDA. */
int seqsum_f64_strided(const double *x, int64_t n, int32_t stride, const double *s0s, double *outs, float *means,
                       cudaStream_t stream);

/* A plan kept from one call to the next (opaque; one per sequence of frames).
 * Research-1433, "Forming the CPU's sequential double sums on a GPU, bit for
 * bit", Open questions (throughput): keep the previous frame's plan, form the
 * runs under it in the same pass that forms the new plan's sums, and form
 * again only the chunks whose plan changed. */
typedef struct seqsum_plan seqsum_plan;

/* Creates an empty plan.  Returns SEQSUM_OK, SEQSUM_EINVAL (out is null) or
 * SEQSUM_ENOMEM.  The plan holds no device memory until its first call. */
int seqsum_plan_create(seqsum_plan **out);

/* Waits for the device (its calls may still read the plan) and frees the
 * plan.  A null plan is ignored. */
void seqsum_plan_destroy(seqsum_plan *plan);

/* As seqsum_f64, for one frame of a sequence: *out = s0 + x[0] + ... +
 * x[n-1] in index order, bit for bit, whatever the frames hold.
 *   plan   from seqsum_plan_create; the call reads the plan of the frame
 *          before and leaves this frame's (2 x 80 bytes a 4096-term tile of
 *          device memory, allocated when n changes)
 *   x, n, s0, out, stream  as for seqsum_f64
 * The first call, and a call whose n differs from the call before, forms its
 * plan first (the two passes of seqsum_f64).  Every other call reads x once:
 * each tile's runs are formed on the stored prefix while its sums for the new
 * plan are taken; a tile whose new prefix no longer keeps the binades its runs
 * were formed in is formed again on the new prefix before the walk reaches it.
 * A frame close to the one before costs one pass; a frame unlike it costs at
 * most about what seqsum_f64 does.  Calls on one plan must be ordered (one
 * stream, or synchronised); a plan is tied to the device of its first call
 * until n changes.
 * Returns SEQSUM_OK, SEQSUM_EINVAL, SEQSUM_ENOMEM or SEQSUM_ECUDA. */
int seqsum_f64_planned(seqsum_plan *plan, const double *x, int64_t n, double s0, double *out,
                       cudaStream_t stream);

/* Counters accumulated on the device by the calls since the last
 * seqsum_get_stats() on the same (device, stream) workspace as the most
 * recent call of this process. */
typedef struct {
  int64_t tiles;             /* tiles of 4096 terms processed */
  int64_t tiles_complex;     /* tiles published as a list of items (rows of several binades, raw rows, ties) */
  int64_t ranges_from_x;     /* walk ranges of 128 tiles whose steps did not fit (the walk read their terms) */
  int64_t lanes_raw;         /* 16-term rows whose plan range crossed a power of two (added by the walk) */
  int64_t lanes_raw2;        /* ... of which published with prefix tables for one crossing */
  int64_t lanes_tie;         /* rows with a tie, composed in order by the even/odd rule */
  int64_t walk_batches;      /* walk ranges (128 tiles each) applied in order */
  int64_t walk_segments;     /* composites the walk applied (same-binade runs composed across tiles) */
  int64_t runs_rejected;     /* runs the walk's exact check refused (their terms were added one by one) */
  int64_t terms_dadd;        /* terms the walk added with a hardware fp64 add */
  int64_t raw_rounds;        /* warp rounds of the walk's term-by-term resolution */
  int64_t cy_walk_wait;      /* SM cycles the walk's producer warps waited for tile headers (summed) */
  int64_t cy_walk_serial;    /* SM cycles of the walk's in-order warp applying steps */
  int64_t cy_walk_raw;       /* ... of which resolving raw terms */
  int64_t cy_tma_wait;       /* SM cycles summed over the streaming warps: waiting for a unit's copy */
  int64_t cy_plan;           /* ... plan units (the tiles' sums) */
  int64_t cy_pfx_wait;       /* ... run units waiting for a prefix the copy did not bring */
  int64_t cy_run;            /* ... run units (the rows' runs and the tile's header) */
  int64_t scan_windows;      /* rounds of tiles' prefixes the scanner published */
  int64_t scan_polls;        /* scanner polls that found no new tile sums */
  int64_t pfx_late;          /* run units whose prefix was not yet published when their copy landed */
  int64_t ctas_alone;        /* streaming CTAs that left their SM to the walker or the scanner */
  int64_t tiles_redone;      /* planned calls: tiles formed again because the new prefix moved their binades */
  int64_t t_stream_ns;       /* latest call: kernel start to the last tile header */
  int64_t t_walk_tail_ns;    /* latest call: last tile header to the end of the walk */
  int64_t t_total_ns;        /* latest call: kernel start to the end of the walk */
  int64_t t_scan_ns;         /* latest call: kernel start to the end of the scanner */
  int64_t t_units_ns;        /* latest call: kernel start to the last tile header formed */
  int32_t device_status;     /* 0, or a negative SEQSUM_E* code */
  int32_t device_error_bits; /* raw device error bits */
  int32_t check_site;        /* self-checking builds: first failed check (0: none) */
  int32_t check_pad;
  int64_t check_value;       /* self-checking builds: the value that failed it */
  int32_t timeout_site;      /* first bounded device wait that gave up (0: none): 2 a stage's copy, 3 a walk
                                range's tile headers, 5 a run unit's prefix, 6 the scanner's tile sums, 7 a
                                stage's release, 8 a planned call's redo list */
  int32_t timeout_pad;
  int64_t timeout_a;         /* its context: the tile */
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

/* Test hook: copies up to 4096 diagnostic words that self-checking builds
 * of the library record (zeros otherwise) and clears them. */
int seqsum_debug_read(unsigned long long *out, int n);

/* Diagnostics of a call that does not finish: copies the first n (1..18)
 * device counters of the most recent call's workspace into out: tickets,
 * roles, exits, error bits, tag, the self-checks' and the bounded waits'
 * records, the walker's and the scanner's SMs, a planned call's redo list.  It takes no lock and reads on a stream of its
 * own, so it can run while another thread waits on that call. */
int seqsum_debug_counters(unsigned long long *out, int n);

/* Test hook for the bounded waits: mode 1 withholds the header of tile `arg`
 * in later calls (the walk's wait for it must give up, write NaN and report
 * SEQSUM_ETIMEOUT, site 3); mode 0 restores normal calls.  wait_ns > 0 sets
 * the limit of every bounded device wait of later calls (0: the default, 2 s).
 * Returns SEQSUM_OK or SEQSUM_EINVAL. */
int seqsum_debug_set_fault(int mode, int64_t arg, int64_t wait_ns);

/* Library version string. */
const char *seqsum_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SEQSUM_H */

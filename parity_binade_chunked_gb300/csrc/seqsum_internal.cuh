// Internal layout shared by the kernel and the two host translation units
// (seqsum_api.cu, seqsum_static.cu).
#pragma once
#include <cuda.h>
#include <stdint.h>

namespace sq {

// ---- geometry
// A lane owns one 128-byte row: 16 consecutive terms.  A tile is 256 rows
// (4096 terms, 32 KB), one TMA box.  A CTA has 8 compute warps (one row per
// thread) and a ninth warp: a streaming CTA's producer.
constexpr int kLaneTerms = 16;
constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kBlockWarps = kWarps + 1;          // + a streaming CTA's producer warp (tickets and copies)
constexpr int kBlockThreads = kBlockWarps * 32;
constexpr int kTileRows = kThreads;
constexpr int kTileTerms = kTileRows * kLaneTerms;
constexpr int kStages = 3;                       // TMA stages of a streaming CTA
constexpr int kStageBytes = kTileTerms * 8;
constexpr int kDynSmem = kStages * kStageBytes + 1024;   // + alignment slack for the 128-byte swizzle
constexpr int kWarpSlots = 32;                   // 32-byte item slots of one warp's region (one per row)
constexpr int kItemSlots = kWarps * kWarpSlots;  // a tile's item area (8 KB): one region per compute warp
constexpr int kMaxWalkers = 8;      // walkers of a batched call (more take slots from the stream)

// ---- units of a streaming CTA
enum : int {
  U_RUN = 0,    // a tile's runs on the prefix its plan unit and the scanner gave
  U_PLAN = 1,   // a tile's sums (for the scanner) and its warps' sums
  U_SPEC = 2,   // planned calls: a tile's runs on the stored prefix, and its sums for the new plan
  U_REDO = 3    // planned calls: a tile's runs again, on the new prefix
};

// ---- records
// A tile header or an item: four 64-bit words.  A header carries the call's
// 8-bit tag in the top byte of every word (a 16-byte access need not be
// single-copy atomic, so a reader checks all four); items are published
// before their header and carry no tag.
//   w[0] inc, w[1] lo, w[2] hi: 56-bit two's complement
//   w[3] meta: kind (3 bits), biased binade (11 bits, 0 = none), d + 1 (2 bits),
//        flags (8 bits), count (13 bits), start (13 bits)
// A K_COMPLEX header carries instead, in w[0], each warp's count of items
// (warp k's in bits 6k..6k+5): warp k's items are the records from slot 32 k
// of the tile's item area, in the order of their terms (a warp that is one run
// has that run as its one item); a raw row's terms stay in x.
struct __align__(16) Rec {
  uint64_t w[4];
};

enum : uint32_t {
  K_RUN = 0,       // a run of adds inside binade eb (or a run of zeros)
  K_RAW = 1,       // item: a row of 16 terms the walk adds itself
  K_COMPLEX = 2,   // header: the tile's records are its warps' item regions (counts in w[0])
  K_OVERFLOW = 3,  // header: the tile's items did not fit; the walk reads its terms from x
  K_RAW2 = 4       // item: a raw row across one power of two, from binade eb to eb + 1, all of its
                   // terms of one sign (w[0]: 1 if negative); the walk builds prefix tables for it
};

constexpr int kPrecWords = 5;     // a tile's plan record: its exclusive prefix, then its warps' float sums (5 x 16 B)

// ---- counters in the workspace (32-bit words)
enum : int {
  C_TICKET = 0,      // next tile ticket of the streaming CTAs
  C_ROLE = 1,        // next CTA role: walkers first, then streamers
  C_EXIT = 2,        // CTAs that finished
  C_SUMTICKET = 3,   // next sum for a walker
  C_ERR = 4,         // error bits (ERR_*), kept until read by seqsum_get_stats
  C_EPOCH = 5,       // the tag of the next call (0: fresh workspace, use 1)
  C_NTILES = 6,      // batched: tiles of the call (written by the set-up kernel)
  C_SKIP = 7,        // batched: the set-up kernel refused the offsets
  C_CHECK_SITE = 8,  // self-checking builds: first failed check and its value
  C_CHECK_LO = 9,
  C_CHECK_HI = 10,
  C_TO_SITE = 11,    // first bounded wait that gave up: its site and two words of context
  C_TO_A = 12,
  C_TO_B = 13,
  C_WALK_SM = 14,    // 1 + the SM of the (first) walker: a streaming CTA there takes no units
  C_SCAN_SM = 15,    // 1 + the SM of the scanner: likewise
  C_REDO_RES = 16,   // planned calls: places of the redo list taken so far
  C_SCAN_FIN = 17,   // planned calls: the scanner and its checkers are done (C_REDO_RES is final)
  C_COUNT = 18
};
enum : uint32_t {
  ERR_TMA_TIMEOUT = 1u,     // a TMA copy did not land within the wait limit (the tile was read from x)
  ERR_PLAN_TIMEOUT = 2u,    // a look-back gave up (the plan only; results stay exact)
  ERR_BAD_OFFSETS = 4u,     // offsets out of order or out of range
  ERR_CAPACITY = 8u,        // a batched call needed more tiles than its workspace holds
  ERR_WALK_TIMEOUT = 16u,   // the walk waited too long for a tile header (NaN written)
};

// ---- statistics (accumulated on the device, read and cleared by the host)
enum : int {
  S_TILES = 0,        // tiles whose runs were formed
  S_TILE_COMPLEX,     // tiles published with an item list
  S_RANGE_X,          // walk ranges whose steps did not fit their slot (read from x)
  S_LANE_RAW,         // 16-term rows published as raw terms (plan range across a power of two)
  S_LANE_RAW2,        // ... of which published with prefix tables for one crossing
  S_LANE_TIE,         // rows with a tie, composed in order
  S_WALK_BATCHES,     // walk ranges applied in order
  S_WALK_SEGMENTS,    // composites the walk applied
  S_RUN_REJECTED,     // runs the walk's exact check refused (their terms were added one by one)
  S_TERMS_DADD,       // terms the walk added with a hardware fp64 add
  S_RAW_ROUNDS,       // warp rounds of the walk's raw-term resolution
  S_CY_WALK_WAIT,     // SM cycles the walk's producer warps waited for tile headers
  S_CY_WALK_SERIAL,   // SM cycles of the walk's in-order warp applying steps
  S_CY_WALK_RAW,      // SM cycles of the walk's raw-term resolution (within the in-order passes)
  S_CY_TMA_WAIT,      // SM cycles, summed over warps: waiting for a unit's copy
  S_CY_PLAN,          // ... plan units (from the copy to the tile's sums published)
  S_CY_PFX_WAIT,      // ... run units waiting for a prefix that the copy did not bring
  S_CY_RUN,           // ... run units (from the prefix to the tile's header)
  S_SCAN_WINDOWS,     // rounds the scanner published
  S_SCAN_POLLS,       // scanner polls of tiles' sums
  S_PFX_LATE,         // run units whose prefix came after their copy
  S_ALONE,            // streaming CTAs that left their SM to the walker or the scanner
  S_REDO,             // planned calls: tiles whose stored plan no longer held (formed again)
  S_ACCUM_END,
  S_T_START = 24,     // timestamps of the latest call (globaltimer): first CTA start
  S_T_STREAM_END,     // last tile header published (max over CTAs)
  S_T_WALK_END,       // last walk ended
  S_T_SCAN_END,       // the scanner ended
  S_T_UNITS_END,      // last unit's tile header published (max over CTAs)
  S_COUNT = 32
};
static_assert(S_ACCUM_END <= S_T_START, "summed counters overlap the timestamps");

// ---- kernel parameters
struct Params {
  const double *x;
  int64_t x_len;               // doubles readable at x
  const int64_t *offsets;      // batched: nsums + 1 entries (device); null for a single sum
  const double *s0s;           // batched: device; null for a single sum
  double *outs;                // device
  double s0;                   // single sum: the start value
  int64_t n;                   // single sum: its length
  int64_t ntiles;              // single: known on the host; batched: -1 (read C_NTILES)
  int64_t tma_rows;            // rows of 16 terms the tensor map covers (0: no TMA)
  int32_t nsums;
  int32_t nwalkers;            // CTA roles 0 .. nwalkers-1 walk, the others stream
  int32_t plan_mode;           // 0 normal; > 0 forced plans (tests)
  int32_t fault_mode;          // 0 none; 1 the header of tile fault_arg is withheld (tests)
  int64_t fault_arg;
  uint64_t wait_ns;            // limit of every bounded device wait
  int64_t wave;                // plan units run this many tiles ahead of run units
  int32_t planned;             // a planned call: every tile formed on the stored plan in prec, then again
                               // where the new prefix shows that plan no longer holds; the new plan (the
                               // tiles' sums and prefixes) goes to prec_next
  uint4 *prec_next;
  uint4 *prec_ws;              // the workspace's plan records (cap_tiles of them), cleared when the tag wraps
  uint32_t *conf;              // planned calls, per tile: the tag once its header may be walked (null: none)
  uint32_t *redo;              // planned calls: the tiles to form again, each (tag << 24) | tile
  // workspace
  uint4 *status;               // per tile: the tile's own sums, published by its plan unit (16 bytes)
  uint4 *prec;                 // per tile: kPrecWords words -- the exclusive prefix (the scanner), the warp sums (the plan)
  Rec *hdr;                    // per tile: its header
  Rec *items;                  // kItemSlots per tile
  uint32_t *ctr;               // C_COUNT counters
  int64_t *tile_begin;         // batched: nsums + 1 entries, by position in `order`
  int32_t *order;              // batched: the sums in the order they stream and are walked (set-up kernel)
  int64_t cap_tiles;           // tiles the workspace holds
  unsigned long long *stats;   // S_COUNT counters
  unsigned long long *dbg;     // self-checking builds: diagnostic words
};

constexpr int kDbgWords = 4096;

cudaError_t launch_seqsum(const Params &p, const CUtensorMap *tmap, int grid, cudaStream_t st);
cudaError_t launch_setup(const Params &p, cudaStream_t st);
cudaError_t launch_deinterleave(const double *x, int64_t n, int stride, double *planes, int64_t *offsets,
                                cudaStream_t st);
cudaError_t launch_mean(const double *outs, int stride, int64_t n, float *means, cudaStream_t st);
constexpr int kMaxStride = 64;                   // interleaved sums a strided call takes
int kernel_blocks_per_sm();

}  // namespace sq

// Internal layout shared by the kernel and API translation units.
#pragma once
#include <cuda.h>
#include <stdint.h>

namespace sq {

// ---- geometry (a lane owns one 128-byte row of 16 consecutive terms)
constexpr int kLaneTerms = 16;
constexpr int kWarps = 8;                       // warps per CTA = chunks per tile
constexpr int kThreads = kWarps * 32;           // compute threads of a CTA (the walker's width)
constexpr int kCtrlWarp = kWarps;               // a streaming CTA's control warp (tickets, copies, tile headers)
constexpr int kBlockThreads = kThreads + 32;
constexpr int kBlockWarps = kBlockThreads / 32;
constexpr int kChunkTerms = 32 * kLaneTerms;    // 512 terms: one warp's chunk
constexpr int kTileTerms = kWarps * kChunkTerms;// 4096 terms = 32 KB: one TMA box
constexpr int kStages = 3;                      // units a streaming CTA holds: copied, worked on, epilogue
constexpr int kStageBytes = kTileTerms * 8;
constexpr int kDynSmem = kStages * kStageBytes + 1024;   // + alignment slack
constexpr int kChunkSlots = 32;                 // item slots per chunk in a tile's item area
constexpr int kCountBits = 7;                   // bits per chunk in a complex header's packed counts
static_assert(kChunkSlots < (1 << kCountBits), "packed item counts");
constexpr int kTileSlots = kWarps * kChunkSlots;
constexpr int kWalkTiles = 1024;                // tile headers per walk batch (32 KB)
constexpr int kWalkElems = 1024;                // flat elements per walk batch (32 KB)
constexpr int kMaxWalkers = 8;
constexpr int kGroupTiles = 32;                 // tiles whose records one streaming CTA composes for the walk
constexpr int kGroupSegs = 256;                 // segments a composed group holds (more: the walk takes its tiles)
constexpr int kHeartbeats = 4096;               // CTAs with a heartbeat word (diagnostics of a stuck call)
constexpr int kDbgAlloc = 65536;                // diagnostic words: checks, walk trace, profiling timeline

// ---- record kinds
enum : uint32_t { K_RUN = 0, K_FALLBACK = 1, K_TERMS = 2, K_COMPLEX = 3 };

// A tile header or an item: 32 bytes.
//   K_RUN      : a run computed for binade e (F_ZERO runs apply in any binade)
//   K_FALLBACK : the covered terms are added one by one from the plane
//   K_TERMS    : up to three terms carried inline (inc, lo, hi hold their
//                bits), added one by one
//   K_COMPLEX  : (tile header) the items live in the tile's item area; inc
//                holds eight 7-bit item counts, one per chunk
// Tile headers carry the call's tag in every one of their four 64-bit words
// (a 16-byte access need not be single-copy atomic), so a reader never mixes
// words of two publications.
struct __align__(16) Rec {
  int64_t inc, lo, hi;
  uint32_t meta;      // bits 0-7: d (int8), 8-15: flags, 16-19: kind, 20-31: first term in the tile
  int16_t e;          // binade
  uint16_t count;     // terms covered
};

__host__ __device__ inline uint32_t rec_meta(int32_t d, uint32_t flags, uint32_t kind, uint32_t tstart = 0) {
  return ((uint32_t)(uint8_t)(int8_t)d) | ((flags & 0xFFu) << 8) | ((kind & 0xFu) << 16) | ((tstart & 0xFFFu) << 20);
}
__host__ __device__ inline int32_t rec_d(uint32_t meta) { return (int32_t)(int8_t)(meta & 0xFFu); }
__host__ __device__ inline uint32_t rec_flags(uint32_t meta) { return (meta >> 8) & 0xFFu; }
__host__ __device__ inline uint32_t rec_kind(uint32_t meta) { return (meta >> 16) & 0xFu; }
__host__ __device__ inline uint32_t rec_tstart(uint32_t meta) { return meta >> 20; }

// ---- counters in the workspace
enum : int {
  C_TICKET = 0,      // next unit ticket (plan and run units of the tiles)
  C_EXIT = 1,        // CTAs that finished
  C_SUMTICKET = 2,   // next sum for a walker
  C_ERR = 3,         // error bits (ERR_*)
  C_NTILES = 4,      // tiles of a batched call (written by the set-up kernel)
  C_ROLE = 5,        // next CTA role: walkers, then the scanner, then streamers
  C_CHECK_SITE = 8,  // self-checking builds: first failed check and its value
  C_CHECK_LO = 9,
  C_CHECK_HI = 10,
  C_TO_SITE = 11,    // first bounded wait that gave up: its site and two words of context
  C_TO_A = 12,
  C_TO_B = 13,
  C_WALK_SM = 14,    // 1 + the SM of walker 0 and 1: a streaming CTA on one of them stops early
  C_COUNT = 16
};
enum : uint32_t {
  ERR_TMA_TIMEOUT = 1u,       // a TMA copy did not complete within the wait limit
  ERR_PLAN_TIMEOUT = 2u,      // a wait for the plan's prefix gave up (the plan only; results stay exact)
  ERR_BAD_OFFSETS = 4u,       // offsets out of order or out of range
  ERR_CAPACITY = 8u,          // a batched call needed more tiles than its workspace holds
  ERR_WALK_TIMEOUT = 16u,     // the walk waited too long for a tile record
};

// ---- statistics (accumulated on the device, read and cleared by the host)
enum : int {
  S_TILES = 0, S_CHUNK_RUN, S_CHUNK_LIST, S_CHUNK_FALLBACK, S_LANE_DIRTY,
  S_WALK_SEGMENTS, S_RUN_REJECTED, S_TERMS_ADDED, S_ITEMS, S_POOL_OVERFLOW,
  S_TILE_COMPLEX, S_SCAN_WINDOWS, S_WALK_BATCHES,
  // nanoseconds summed over CTAs (globaltimer)
  S_NS_TMA_WAIT, S_NS_PREFIX_WAIT, S_NS_PHASE_A, S_NS_PHASE_B, S_NS_WALK_WAIT, S_NS_WALK_WORK,
  S_TORN_HEADER,       // header reads that mixed words of two publications (retried)
  S_TORN_STATUS,       // prefix reads that mixed words of two publications (retried)
  S_NS_SCAN,           // the scanner's time from its first to its last window
  S_CHUNK_DIRTY,       // chunks whose prefix range spans two binades (placed lane by lane)
  S_NS_CTRL_WAIT,      // control warps waiting for their compute warps
  S_NS_SCAN_WAIT,      // the scanner waiting for tiles' sums to be published
  // the walk's work by section (nanoseconds): counting a batch's elements,
  // gathering them, the segmented scan, the in-order pass, and within that
  // pass the term-by-term adds
  S_NS_WALK_COUNT, S_NS_WALK_GATHER, S_NS_WALK_SCAN, S_NS_WALK_SERIAL, S_NS_WALK_ADDS,
  S_NS_VERDICT,        // run units: forming the chunks' verdicts from the plan words
  S_NS_VERDICT_WAIT,   // run units: plan words read again from global memory (not copied in time)
  S_NS_GCOUNT,         // control warps counting their tiles in the tiles' groups
  S_NS_COMPOSE,        // control warps composing groups for the walk
  S_ACCUM_END,         // counters above are summed; below are timestamps of the latest call
  S_T_START = 40,      // block 0 started (timestamps follow the summed counters)
  S_T_WALK0 = 41,      // the walk's last batch of headers was ready
  S_T_WALK1 = 42,      // the walk ended
  S_T_STREAM_END = 43, // the last tile header was published (max over CTAs)
  S_COUNT = 48
};
static_assert(S_ACCUM_END <= S_T_START, "summed counters overlap the timestamps");

// ---- kernel parameters
struct Params {
  const double *x;
  const int64_t *offsets;      // batched: nsums + 1 entries (device); null for a single sum
  const double *s0s;           // batched: device; null for a single sum
  double *outs;                // device
  double s0;                   // single sum start value
  int64_t n;                   // single sum length (batched: unused)
  int64_t ntiles;              // single: known on the host; batched: -1 (read C_NTILES)
  int64_t tma_rows;            // rows of 16 terms the tensor map covers (0: no TMA)
  int32_t nsums;
  uint32_t epoch;
  int32_t plan_mode;           // 0 normal; >0 forced plans for tests
  int32_t pad;
  // workspace
  uint64_t *status;            // 2 words per tile: tagged approximate sum, then inclusive prefix
  uint64_t *cplan;             // 4 tagged words per chunk: the plan's fixed-point sums of the chunk
  uint32_t *grp_cnt;           // per group of kGroupTiles tiles: epoch << 24 | tiles whose header is published
  uint64_t *grp_hdr;           // per group: tag << 56 | raw << 16 | segments
  Rec *grp_seg;                // per group: kGroupSegs composed segments
  uint16_t *grp_stile;         // per group segment: its first tile within the group
  Rec *hdr;                    // one header per tile
  Rec *items;                  // kTileSlots items per tile
  uint32_t *ctr;               // C_COUNT counters
  int64_t *tile_begin;         // batched: nsums + 1 entries
  int32_t nwalkers;            // CTA roles 0 .. nwalkers-1 walk, role nwalkers scans, the others stream
  int32_t pad2;
  int64_t wave;                // plan units run this many tiles ahead of run units
  unsigned long long *dbg;     // self-checking builds: diagnostic words
  unsigned long long *hb;      // kHeartbeats words: per CTA its role, what it waits for or does, where
  int64_t cap_tiles;           // tiles the workspace holds
  unsigned long long *stats;   // S_COUNT counters
};

cudaError_t launch_seqsum(const Params &p, const CUtensorMap *tmap, int grid, cudaStream_t st);
cudaError_t launch_setup(const Params &p, cudaStream_t st);
int kernel_max_blocks_per_sm();

}  // namespace sq

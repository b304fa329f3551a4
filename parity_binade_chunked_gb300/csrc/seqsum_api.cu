// The C ABI of the library (include/seqsum.h): argument checks, the per
// (device, stream) workspace, the TMA descriptor of the term plane, launches.
// Nothing here computes any part of a sum.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include <map>
#include <mutex>
#include <utility>

#include "../../include/seqsum.h"
#include "seqsum_internal.cuh"

namespace {

using sq::Params;
using sq::Rec;

struct Workspace {
  int device = 0;
  cudaStream_t stream = nullptr;
  int64_t cap_tiles = 0, cap_sums = 0;
  uint64_t *status = nullptr;        // the plan's prefix words, 2 per tile
  uint64_t *cplan = nullptr;         // the plan's chunk sums, 4 words per chunk
  uint32_t *grp_cnt = nullptr;       // composed groups of tiles: counters, headers, segments
  uint64_t *grp_hdr = nullptr;
  Rec *grp_seg = nullptr;
  uint16_t *grp_stile = nullptr;
  Rec *hdr = nullptr;                // one header per tile
  Rec *items = nullptr;              // kTileSlots items per tile
  uint32_t *ctr = nullptr;
  int64_t *tile_begin = nullptr;
  unsigned long long *stats = nullptr;
  unsigned long long *dbg = nullptr;
  unsigned long long *hb = nullptr;  // heartbeat words
  uint32_t epoch = 0;
  int64_t *h_pin = nullptr;          // pinned bounce for the batched size read-back
  // tensor map cache
  const void *tm_ptr = nullptr;
  int64_t tm_rows = -1;
  CUtensorMap tmap;
};

std::mutex g_mu;
std::map<std::pair<int, cudaStream_t>, Workspace *> g_ws;
Workspace *g_last = nullptr;
int g_last_cuda = 0;
int g_plan_mode = 0;
int g_blocks_per_sm = 0;
int g_num_sms[64] = {0};
int64_t g_wave = 0;                  // tiles plan units run ahead of run units (0: not yet read)
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

int cuda_fail(cudaError_t e) {
  g_last_cuda = (int)e;
  return SEQSUM_ECUDA;
}

void ws_free(Workspace *w) {
  cudaFree(w->status);
  cudaFree(w->cplan);
  cudaFree(w->grp_cnt);
  cudaFree(w->grp_hdr);
  cudaFree(w->grp_seg);
  cudaFree(w->grp_stile);
  w->grp_cnt = nullptr;
  w->grp_hdr = nullptr;
  w->grp_seg = nullptr;
  w->grp_stile = nullptr;
  cudaFree(w->hdr);
  cudaFree(w->items);
  cudaFree(w->tile_begin);
  w->status = w->cplan = nullptr;
  w->hdr = w->items = nullptr;
  w->tile_begin = nullptr;
  w->cap_tiles = w->cap_sums = 0;
}

// Workspace for (current device, stream) holding at least `tiles` tiles and
// `sums` sums.  Called with g_mu held.
int get_ws(cudaStream_t stream, int64_t tiles, int64_t sums, Workspace **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  Workspace *&w = g_ws[std::make_pair(dev, stream)];
  if (!w) {
    w = new Workspace();
    w->device = dev;
    w->stream = stream;
    if ((e = cudaMalloc(&w->ctr, sq::C_COUNT * sizeof(uint32_t))) != cudaSuccess) return cuda_fail(e);
    if ((e = cudaMalloc(&w->stats, sq::S_COUNT * sizeof(unsigned long long))) != cudaSuccess)
      return cuda_fail(e);
    if ((e = cudaMallocHost(&w->h_pin, 2 * sizeof(int64_t))) != cudaSuccess) return cuda_fail(e);
    if ((e = cudaMalloc(&w->dbg, sq::kDbgAlloc * sizeof(unsigned long long))) != cudaSuccess) return cuda_fail(e);
    if ((e = cudaMalloc(&w->hb, sq::kHeartbeats * sizeof(unsigned long long))) != cudaSuccess) return cuda_fail(e);
    cudaMemset(w->hb, 0, sq::kHeartbeats * sizeof(unsigned long long));
    cudaMemset(w->dbg, 0, sq::kDbgAlloc * sizeof(unsigned long long));
    cudaMemset(w->ctr, 0, sq::C_COUNT * sizeof(uint32_t));
    cudaMemset(w->stats, 0, sq::S_COUNT * sizeof(unsigned long long));
  }
  if (tiles > w->cap_tiles || sums > w->cap_sums) {
    // wait for earlier work on this stream before the old buffers go
    if ((e = cudaStreamSynchronize(stream)) != cudaSuccess) return cuda_fail(e);
    const int64_t ct = tiles > w->cap_tiles ? tiles + tiles / 4 + 16 : w->cap_tiles;
    const int64_t cs = sums > w->cap_sums ? sums + 16 : w->cap_sums;
    ws_free(w);
    if (cudaMalloc(&w->status, ct * 2 * sizeof(uint64_t)) != cudaSuccess ||
        cudaMalloc(&w->cplan, ct * sq::kWarps * 4 * sizeof(uint64_t)) != cudaSuccess ||
        cudaMalloc(&w->grp_cnt, (ct / sq::kGroupTiles + 1) * sizeof(uint32_t)) != cudaSuccess ||
        cudaMalloc(&w->grp_hdr, (ct / sq::kGroupTiles + 1) * sizeof(uint64_t)) != cudaSuccess ||
        cudaMalloc(&w->grp_seg, (ct / sq::kGroupTiles + 1) * sq::kGroupSegs * sizeof(Rec)) != cudaSuccess ||
        cudaMalloc(&w->grp_stile, (ct / sq::kGroupTiles + 1) * sq::kGroupSegs * sizeof(uint16_t)) != cudaSuccess ||
        cudaMalloc(&w->hdr, ct * sizeof(Rec)) != cudaSuccess ||
        cudaMalloc(&w->items, ct * sq::kTileSlots * sizeof(Rec)) != cudaSuccess ||
        cudaMalloc(&w->tile_begin, (cs + 1) * sizeof(int64_t)) != cudaSuccess) {
      ws_free(w);
      g_last_cuda = (int)cudaGetLastError();
      return SEQSUM_ENOMEM;
    }
    cudaMemset(w->status, 0, ct * 2 * sizeof(uint64_t));
    cudaMemset(w->cplan, 0, ct * sq::kWarps * 4 * sizeof(uint64_t));
    cudaMemset(w->grp_cnt, 0, (ct / sq::kGroupTiles + 1) * sizeof(uint32_t));
    cudaMemset(w->grp_hdr, 0, (ct / sq::kGroupTiles + 1) * sizeof(uint64_t));
    cudaMemset(w->hdr, 0, ct * sizeof(Rec));
    w->cap_tiles = ct;
    w->cap_sums = cs;
    w->epoch = 0;
    if ((e = cudaDeviceSynchronize()) != cudaSuccess) return cuda_fail(e);
  }
  *out = w;
  return SEQSUM_OK;
}

int ensure_device_info() {
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return SEQSUM_EINVAL;
  if (g_num_sms[dev] == 0) {
    cudaError_t e = cudaDeviceGetAttribute(&g_num_sms[dev], cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e);
  }
  if (g_blocks_per_sm == 0) g_blocks_per_sm = sq::kernel_max_blocks_per_sm();
  if (g_wave == 0) {
    // 2048 tiles (64 MB): far more than the units a full grid holds in
    // flight, so the scanner is well ahead of the run units, and little
    // enough that a tile is still in L2 (129 MB) when its run unit reads it.
    g_wave = 2048;
    const char *ev = getenv("SEQSUM_WAVE");
    if (ev && atoll(ev) > 0) g_wave = atoll(ev);
  }
  if (!g_encode) {
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn) return cuda_fail(e);
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  return SEQSUM_OK;
}

// Next epoch for the tags (1..127); every tagged word (the plan's sums and
// prefixes, the tile headers) is cleared whenever the tag wraps, so a stale
// word can never carry a current tag.
void next_epoch(Workspace *w, cudaStream_t stream) {
  w->epoch++;
  if (w->epoch > 127) {
    cudaMemsetAsync(w->status, 0, w->cap_tiles * 2 * sizeof(uint64_t), stream);
    cudaMemsetAsync(w->cplan, 0, w->cap_tiles * sq::kWarps * 4 * sizeof(uint64_t), stream);
    cudaMemsetAsync(w->grp_cnt, 0, (w->cap_tiles / sq::kGroupTiles + 1) * sizeof(uint32_t), stream);
    cudaMemsetAsync(w->grp_hdr, 0, (w->cap_tiles / sq::kGroupTiles + 1) * sizeof(uint64_t), stream);
    cudaMemsetAsync(w->hdr, 0, w->cap_tiles * sizeof(Rec), stream);
    w->epoch = 1;
  }
}

// The 2-D view [rows][16] of the plane, 128-byte swizzled boxes of 256 rows.
// Returns the rows covered (0 when x is not 16-byte aligned: no TMA).
int64_t tensor_map(Workspace *w, const double *x, int64_t n_total) {
  if ((reinterpret_cast<uintptr_t>(x) & 15) != 0 || n_total < 16) return 0;
  const int64_t rows = n_total / 16;
  if (w->tm_ptr == x && w->tm_rows == rows) return rows;
  cuuint64_t dims[2] = {16, (cuuint64_t)rows};
  cuuint64_t strides[1] = {16 * sizeof(double)};
  cuuint32_t box[2] = {16, 256};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(&w->tmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT64, 2, const_cast<double *>(x), dims, strides, box,
                        estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) { w->tm_ptr = nullptr; w->tm_rows = -1; return 0; }
  w->tm_ptr = x;
  w->tm_rows = rows;
  return rows;
}

void fill_ws(Params &p, Workspace *w) {
  p.status = w->status;
  p.cplan = w->cplan;
  p.grp_cnt = w->grp_cnt;
  p.grp_hdr = w->grp_hdr;
  p.grp_seg = w->grp_seg;
  p.grp_stile = w->grp_stile;
  p.hdr = w->hdr;
  p.items = w->items;
  p.ctr = w->ctr;
  p.tile_begin = w->tile_begin;
  p.cap_tiles = w->cap_tiles;
  p.stats = w->stats;
  p.dbg = w->dbg;
  p.hb = w->hb;
}

int batched_impl(const double *x, int64_t x_len, const int64_t *offsets, int32_t nsums, const double *s0s,
                 double *outs, bool sized, cudaStream_t stream) {
  if (nsums < 0) return SEQSUM_EINVAL;
  if (nsums == 0) return SEQSUM_OK;
  if (!offsets || !s0s || !outs) return SEQSUM_EINVAL;
  std::lock_guard<std::mutex> lk(g_mu);
  int rc = ensure_device_info();
  if (rc) return rc;
  Workspace *w = nullptr;
  if (!sized) {
    // read offsets[0] and offsets[nsums] to size the workspace
    rc = get_ws(stream, 1, nsums, &w);
    if (rc) return rc;
    cudaError_t e = cudaMemcpyAsync(w->h_pin, offsets, sizeof(int64_t), cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(w->h_pin + 1, offsets + nsums, sizeof(int64_t), cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return cuda_fail(e);
    if (w->h_pin[0] < 0 || w->h_pin[1] < w->h_pin[0]) return SEQSUM_EINVAL;
    x_len = w->h_pin[1];
  }
  if (x_len < 0) return SEQSUM_EINVAL;
  if (x_len > 0 && !x) return SEQSUM_EINVAL;
  const int64_t tiles = x_len / sq::kTileTerms + nsums + 1;
  rc = get_ws(stream, tiles, nsums, &w);
  if (rc) return rc;
  next_epoch(w, stream);
  Params p;
  memset(&p, 0, sizeof p);
  p.x = x;
  p.n = x_len;
  p.offsets = offsets;
  p.s0s = s0s;
  p.outs = outs;
  p.ntiles = -1;
  p.nsums = nsums;
  p.epoch = w->epoch;
  p.plan_mode = g_plan_mode;
  fill_ws(p, w);
  p.tma_rows = tensor_map(w, x, x_len);
  p.nwalkers = nsums < sq::kMaxWalkers ? nsums : sq::kMaxWalkers;
  p.wave = g_wave;
  cudaError_t e = sq::launch_setup(p, stream);
  if (e != cudaSuccess) return cuda_fail(e);
  int grid = g_num_sms[w->device] * g_blocks_per_sm;
  if (grid < p.nwalkers + 2) grid = p.nwalkers + 2;     // walkers, the scanner, at least one streamer
  static CUtensorMap dummy;
  e = sq::launch_seqsum(p, p.tma_rows ? &w->tmap : &dummy, grid, stream);
  if (e != cudaSuccess) return cuda_fail(e);
  g_last = w;
  return SEQSUM_OK;
}

}  // namespace

extern "C" {

int seqsum_f64(const double *x, int64_t n, double s0, double *out, cudaStream_t stream) {
  if (n < 0 || !out || (n > 0 && !x)) return SEQSUM_EINVAL;
  std::lock_guard<std::mutex> lk(g_mu);
  int rc = ensure_device_info();
  if (rc) return rc;
  const int64_t tiles = (n + sq::kTileTerms - 1) / sq::kTileTerms;
  Workspace *w = nullptr;
  rc = get_ws(stream, tiles > 0 ? tiles : 1, 1, &w);
  if (rc) return rc;
  next_epoch(w, stream);
  Params p;
  memset(&p, 0, sizeof p);
  p.x = x;
  p.outs = out;
  p.s0 = s0;
  p.n = n;
  p.ntiles = tiles;
  p.nsums = 1;
  p.epoch = w->epoch;
  p.plan_mode = g_plan_mode;
  fill_ws(p, w);
  p.tma_rows = n > 0 ? tensor_map(w, x, n) : 0;
  p.nwalkers = 1;
  p.wave = g_wave;
  const int dev = w->device;
  int64_t grid = (int64_t)g_num_sms[dev] * g_blocks_per_sm;
  if (2 * tiles + 2 < grid) grid = 2 * tiles + 2;     // the walker, the scanner, one streamer per unit
  static CUtensorMap dummy;
  cudaError_t e = sq::launch_seqsum(p, p.tma_rows ? &w->tmap : &dummy, (int)grid, stream);
  if (e != cudaSuccess) return cuda_fail(e);
  g_last = w;
  return SEQSUM_OK;
}

int seqsum_f64_batched(const double *x, const int64_t *offsets, int32_t nsums, const double *s0s, double *outs,
                       cudaStream_t stream) {
  return batched_impl(x, 0, offsets, nsums, s0s, outs, false, stream);
}

int seqsum_f64_batched_sized(const double *x, int64_t x_len, const int64_t *offsets, int32_t nsums,
                             const double *s0s, double *outs, cudaStream_t stream) {
  return batched_impl(x, x_len, offsets, nsums, s0s, outs, true, stream);
}

int seqsum_get_stats(seqsum_stats *st) {
  if (!st) return SEQSUM_EINVAL;
  std::lock_guard<std::mutex> lk(g_mu);
  memset(st, 0, sizeof *st);
  Workspace *w = g_last;
  if (!w) return SEQSUM_OK;
  int prev = 0;
  cudaGetDevice(&prev);
  cudaSetDevice(w->device);
  unsigned long long s[sq::S_COUNT];
  uint32_t c[sq::C_COUNT];
  cudaError_t e = cudaStreamSynchronize(w->stream);
  if (e == cudaSuccess) e = cudaMemcpy(s, w->stats, sizeof s, cudaMemcpyDeviceToHost);
  if (e == cudaSuccess) e = cudaMemcpy(c, w->ctr, sizeof c, cudaMemcpyDeviceToHost);
  if (e == cudaSuccess) e = cudaMemset(w->stats, 0, sizeof s);
  const uint32_t err = (e == cudaSuccess) ? c[sq::C_ERR] : 0u;
  if (e == cudaSuccess && err) e = cudaMemset(w->ctr + sq::C_ERR, 0, sizeof(uint32_t));
  if (e == cudaSuccess && c[sq::C_CHECK_SITE]) e = cudaMemset(w->ctr + sq::C_CHECK_SITE, 0, 3 * sizeof(uint32_t));
  if (e == cudaSuccess && c[sq::C_TO_SITE]) e = cudaMemset(w->ctr + sq::C_TO_SITE, 0, 3 * sizeof(uint32_t));
  st->timeout_site = (int32_t)c[sq::C_TO_SITE];
  st->timeout_a = (int64_t)c[sq::C_TO_A];
  st->timeout_b = (int64_t)c[sq::C_TO_B];
  st->check_site = (int32_t)c[sq::C_CHECK_SITE];
  st->check_value = (int64_t)(((uint64_t)c[sq::C_CHECK_HI] << 32) | c[sq::C_CHECK_LO]);
  cudaSetDevice(prev);
  if (e != cudaSuccess) return cuda_fail(e);
  st->tiles = (int64_t)s[sq::S_TILES];
  st->chunks_run = (int64_t)s[sq::S_CHUNK_RUN];
  st->chunks_list = (int64_t)s[sq::S_CHUNK_LIST];
  st->chunks_fallback = (int64_t)s[sq::S_CHUNK_FALLBACK];
  st->lanes_dirty = (int64_t)s[sq::S_LANE_DIRTY];
  st->walk_segments = (int64_t)s[sq::S_WALK_SEGMENTS];
  st->runs_rejected = (int64_t)s[sq::S_RUN_REJECTED];
  st->terms_added = (int64_t)s[sq::S_TERMS_ADDED];
  st->items = (int64_t)s[sq::S_ITEMS];
  st->pool_overflow = (int64_t)s[sq::S_POOL_OVERFLOW];
  st->tiles_complex = (int64_t)s[sq::S_TILE_COMPLEX];
  st->scan_windows = (int64_t)s[sq::S_SCAN_WINDOWS];
  st->walk_batches = (int64_t)s[sq::S_WALK_BATCHES];
  st->ns_tma_wait = (int64_t)s[sq::S_NS_TMA_WAIT];
  st->ns_prefix_wait = (int64_t)s[sq::S_NS_PREFIX_WAIT];
  st->ns_phase_a = (int64_t)s[sq::S_NS_PHASE_A];
  st->ns_phase_b = (int64_t)s[sq::S_NS_PHASE_B];
  st->ns_walk_wait = (int64_t)s[sq::S_NS_WALK_WAIT];
  st->ns_walk_work = (int64_t)s[sq::S_NS_WALK_WORK];
  st->torn_header_reads = (int64_t)s[sq::S_TORN_HEADER];
  st->torn_status_reads = (int64_t)s[sq::S_TORN_STATUS];
  st->ns_scan = (int64_t)s[sq::S_NS_SCAN];
  st->ns_walk_count = (int64_t)s[sq::S_NS_WALK_COUNT];
  st->ns_walk_gather = (int64_t)s[sq::S_NS_WALK_GATHER];
  st->ns_walk_scan = (int64_t)s[sq::S_NS_WALK_SCAN];
  st->ns_walk_serial = (int64_t)s[sq::S_NS_WALK_SERIAL];
  st->ns_walk_adds = (int64_t)s[sq::S_NS_WALK_ADDS];
  st->chunks_dirty = (int64_t)s[sq::S_CHUNK_DIRTY];
  st->ns_ctrl_wait = (int64_t)s[sq::S_NS_CTRL_WAIT];
  st->ns_scan_wait = (int64_t)s[sq::S_NS_SCAN_WAIT];
  st->ns_verdict = (int64_t)s[sq::S_NS_VERDICT];
  st->ns_verdict_wait = (int64_t)s[sq::S_NS_VERDICT_WAIT];
  st->ns_group_count = (int64_t)s[sq::S_NS_GCOUNT];
  st->ns_compose = (int64_t)s[sq::S_NS_COMPOSE];
  st->t_stream_ns = (int64_t)(s[sq::S_T_STREAM_END] - s[sq::S_T_START]);
  st->t_walk_tail_ns = (int64_t)(s[sq::S_T_WALK1] - s[sq::S_T_STREAM_END]);
  st->t_total_ns = (int64_t)(s[sq::S_T_WALK1] - s[sq::S_T_START]);
  st->device_error_bits = (int32_t)err;
  if (err & sq::ERR_CAPACITY) st->device_status = SEQSUM_ECAPACITY;
  else if (err & sq::ERR_BAD_OFFSETS) st->device_status = SEQSUM_EOFFSETS;
  else if (err & (sq::ERR_TMA_TIMEOUT | sq::ERR_WALK_TIMEOUT)) st->device_status = SEQSUM_ETIMEOUT;
  else if (err & 32u) st->device_status = SEQSUM_EINVAL;
  else st->device_status = SEQSUM_OK;   // a plan timeout alone leaves results exact
  return SEQSUM_OK;
}

const char *seqsum_strerror(int code) {
  switch (code) {
    case SEQSUM_OK: return "ok";
    case SEQSUM_EINVAL: return "invalid argument";
    case SEQSUM_ECUDA: return "CUDA runtime error";
    case SEQSUM_ETIMEOUT: return "a bounded device wait gave up";
    case SEQSUM_ENOMEM: return "workspace allocation failed";
    case SEQSUM_ECAPACITY: return "batched call exceeded its promised size";
    case SEQSUM_EOFFSETS: return "offsets are not non-decreasing";
    default: return "unknown error";
  }
}

int seqsum_last_cuda_error(void) { return g_last_cuda; }

void seqsum_release_workspace(void) {
  std::lock_guard<std::mutex> lk(g_mu);
  int prev = 0;
  cudaGetDevice(&prev);
  for (auto &kv : g_ws) {
    Workspace *w = kv.second;
    if (!w) continue;
    cudaSetDevice(w->device);
    cudaStreamSynchronize(w->stream);
    ws_free(w);
    cudaFree(w->ctr);
    cudaFree(w->stats);
    cudaFree(w->dbg);
    cudaFree(w->hb);
    cudaFreeHost(w->h_pin);
    delete w;
  }
  g_ws.clear();
  g_last = nullptr;
  cudaSetDevice(prev);
}

int seqsum_debug_read(unsigned long long *out, int n) {
  std::lock_guard<std::mutex> lk(g_mu);
  Workspace *w = g_last;
  if (!w || !out || n < 0 || n > sq::kDbgAlloc) return SEQSUM_EINVAL;
  cudaError_t e = cudaStreamSynchronize(w->stream);
  if (e == cudaSuccess) e = cudaMemcpy(out, w->dbg, n * sizeof(unsigned long long), cudaMemcpyDeviceToHost);
  if (e == cudaSuccess) e = cudaMemset(w->dbg, 0, sq::kDbgAlloc * sizeof(unsigned long long));
  return e == cudaSuccess ? SEQSUM_OK : cuda_fail(e);
}

int seqsum_debug_heartbeat(unsigned long long *out, int n) {
  // No lock: this is read while another thread may be blocked inside a call
  // of this library (holding its lock).  A non-blocking stream lets the copy
  // run next to a kernel that has not finished.
  static cudaStream_t side = nullptr;
  Workspace *w = g_last;
  if (!w || !out || n < sq::C_COUNT || n > sq::C_COUNT + sq::kHeartbeats) return SEQSUM_EINVAL;
  cudaError_t e = cudaSuccess;
  if (!side) e = cudaStreamCreateWithFlags(&side, cudaStreamNonBlocking);
  uint32_t c[sq::C_COUNT];
  if (e == cudaSuccess) e = cudaMemcpyAsync(c, w->ctr, sizeof c, cudaMemcpyDeviceToHost, side);
  if (e == cudaSuccess && n > sq::C_COUNT)
    e = cudaMemcpyAsync(out + sq::C_COUNT, w->hb, (n - sq::C_COUNT) * sizeof(unsigned long long),
                        cudaMemcpyDeviceToHost, side);
  if (e == cudaSuccess) e = cudaStreamSynchronize(side);
  if (e != cudaSuccess) return cuda_fail(e);
  for (int i = 0; i < sq::C_COUNT; i++) out[i] = c[i];
  return SEQSUM_OK;
}

int seqsum_debug_set_plan(int mode) {
  std::lock_guard<std::mutex> lk(g_mu);
  const int old = g_plan_mode;
  g_plan_mode = mode;
  return old;
}

const char *seqsum_version(void) { return "seqsum 0.1 (sm_103a)"; }

}  // extern "C"

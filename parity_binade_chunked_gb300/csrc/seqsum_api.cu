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
#include <new>
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
  uint4 *status = nullptr;           // per tile: its sums, published by its plan unit
  uint4 *prec = nullptr;             // per tile: its prefix (the scanner) and its warps' sums (the plan)
  Rec *hdr = nullptr;                // one header per tile
  Rec *items = nullptr;              // kItemSlots item slots per tile
  uint32_t *ctr = nullptr;
  int64_t *tile_begin = nullptr;
  int32_t *order = nullptr;          // batched: the sums in the order the kernel takes them
  unsigned long long *stats = nullptr;
  unsigned long long *dbg = nullptr;
  int64_t *h_pin = nullptr;          // pinned bounce for the batched size read-back
  double *planes = nullptr;          // strided calls: the interleaved sums laid out one after another
  int64_t *soffs = nullptr;          // ... and their offsets
  int64_t cap_planes = 0;
  uint32_t *conf = nullptr;          // planned calls: per tile, the tag once its header may be walked
  uint32_t *redo = nullptr;          // planned calls: the redo list
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
int g_fault_mode = 0;
int64_t g_fault_arg = 0;
uint64_t g_wait_ns = 2000000000ull;   // every bounded device wait gives up after 2 s
int g_blocks_per_sm = 0;
int64_t g_wave = 0;                   // plan units run this many tiles ahead of run units (0: not yet read)
int g_num_sms[64] = {0};
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

int cuda_fail(cudaError_t e) {
  g_last_cuda = (int)e;
  return SEQSUM_ECUDA;
}

void ws_free(Workspace *w) {
  cudaFree(w->status);
  cudaFree(w->prec);
  w->prec = nullptr;
  cudaFree(w->hdr);
  cudaFree(w->items);
  cudaFree(w->tile_begin);
  cudaFree(w->order);
  w->order = nullptr;
  cudaFree(w->conf);
  cudaFree(w->redo);
  w->conf = nullptr;
  w->redo = nullptr;
  w->status = nullptr;
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
    if ((e = cudaMalloc(&w->dbg, sq::kDbgWords * sizeof(unsigned long long))) != cudaSuccess) return cuda_fail(e);
    cudaMemset(w->dbg, 0, sq::kDbgWords * sizeof(unsigned long long));
    cudaMemset(w->ctr, 0, sq::C_COUNT * sizeof(uint32_t));
    cudaMemset(w->stats, 0, sq::S_COUNT * sizeof(unsigned long long));
  }
  if (tiles > w->cap_tiles || sums > w->cap_sums) {
    // wait for earlier work on this stream before the old buffers go
    if ((e = cudaStreamSynchronize(stream)) != cudaSuccess) return cuda_fail(e);
    const int64_t ct = tiles > w->cap_tiles ? tiles + tiles / 4 + 16 : w->cap_tiles;
    const int64_t cs = sums > w->cap_sums ? sums + 16 : w->cap_sums;
    ws_free(w);
    if (cudaMalloc(&w->status, ct * sizeof(uint4)) != cudaSuccess ||
        cudaMalloc(&w->prec, ct * sq::kPrecWords * sizeof(uint4)) != cudaSuccess ||
        cudaMalloc(&w->hdr, ct * sizeof(Rec)) != cudaSuccess ||
        cudaMalloc(&w->items, ct * sq::kItemSlots * sizeof(Rec)) != cudaSuccess ||
        cudaMalloc(&w->tile_begin, (cs + 1) * sizeof(int64_t)) != cudaSuccess ||
        cudaMalloc(&w->order, cs * sizeof(int32_t)) != cudaSuccess ||
        cudaMalloc(&w->conf, ct * sizeof(uint32_t)) != cudaSuccess ||
        cudaMalloc(&w->redo, ct * sizeof(uint32_t)) != cudaSuccess) {
      ws_free(w);
      g_last_cuda = (int)cudaGetLastError();
      return SEQSUM_ENOMEM;
    }
    // fresh tagged words and a fresh tag sequence (the counters' epoch word)
    cudaMemset(w->status, 0, ct * sizeof(uint4));
    cudaMemset(w->prec, 0, ct * sq::kPrecWords * sizeof(uint4));
    cudaMemset(w->hdr, 0, ct * sizeof(Rec));
    cudaMemset(w->conf, 0, ct * sizeof(uint32_t));
    cudaMemset(w->redo, 0, ct * sizeof(uint32_t));
    cudaMemset(w->ctr, 0, sq::C_COUNT * sizeof(uint32_t));
    w->cap_tiles = ct;
    w->cap_sums = cs;
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
  if (g_blocks_per_sm == 0) g_blocks_per_sm = sq::kernel_blocks_per_sm();
  if (g_wave == 0) {
    // far enough ahead that the scanner has published a tile's prefix when
    // its run unit starts, near enough that the tile is still in L2 (2048
    // tiles = 64 MB of the 129 MB)
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

// The 2-D view [rows][16] of the plane, 128-byte swizzled boxes of 256 rows.
// Returns the rows covered (0 when x is not 16-byte aligned: no TMA).
int64_t tensor_map(Workspace *w, const double *x, int64_t n_total) {
  if ((reinterpret_cast<uintptr_t>(x) & 15) != 0 || n_total < 16) return 0;
  const int64_t rows = n_total / 16;
  if (w->tm_ptr == x && w->tm_rows == rows) return rows;
  cuuint64_t dims[2] = {16, (cuuint64_t)rows};
  cuuint64_t strides[1] = {16 * sizeof(double)};
  cuuint32_t box[2] = {16, (cuuint32_t)sq::kTileRows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(&w->tmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT64, 2, const_cast<double *>(x), dims, strides, box,
                        estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    w->tm_ptr = nullptr;
    w->tm_rows = -1;
    return 0;
  }
  w->tm_ptr = x;
  w->tm_rows = rows;
  return rows;
}

void fill_ws(Params &p, Workspace *w) {
  p.status = w->status;
  p.prec = w->prec;
  p.prec_ws = w->prec;
  p.conf = w->conf;
  p.redo = w->redo;
  p.wave = g_wave;
  p.hdr = w->hdr;
  p.items = w->items;
  p.ctr = w->ctr;
  p.tile_begin = w->tile_begin;
  p.order = w->order;
  p.cap_tiles = w->cap_tiles;
  p.stats = w->stats;
  p.dbg = w->dbg;
  p.plan_mode = g_plan_mode;
  p.fault_mode = g_fault_mode;
  p.fault_arg = g_fault_arg;
  p.wait_ns = g_wait_ns;
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
  // every sum adds at most two tiles beyond its share of x (row alignment, a ragged end)
  const int64_t tiles = x_len / sq::kTileTerms + 2 * (int64_t)nsums + 1;
  rc = get_ws(stream, tiles, nsums, &w);
  if (rc) return rc;
  Params p;
  memset(&p, 0, sizeof p);
  p.x = x;
  p.x_len = x_len;
  p.offsets = offsets;
  p.s0s = s0s;
  p.outs = outs;
  p.ntiles = -1;
  p.nsums = nsums;
  fill_ws(p, w);
  p.tma_rows = tensor_map(w, x, x_len);
  p.nwalkers = nsums < sq::kMaxWalkers ? nsums : sq::kMaxWalkers;
  cudaError_t e = sq::launch_setup(p, stream);
  if (e != cudaSuccess) return cuda_fail(e);
  // the walkers, the scanner, and streaming CTAs (at most one per unit)
  int64_t grid = (int64_t)g_num_sms[w->device] * g_blocks_per_sm;
  if (p.nwalkers + 1 + 2 * tiles < grid) grid = p.nwalkers + 1 + 2 * tiles;
  if (grid < p.nwalkers + 2) grid = p.nwalkers + 2;
  static CUtensorMap dummy;
  e = sq::launch_seqsum(p, p.tma_rows ? &w->tmap : &dummy, (int)grid, stream);
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
  Params p;
  memset(&p, 0, sizeof p);
  p.x = x;
  p.x_len = n;
  p.outs = out;
  p.s0 = s0;
  p.n = n;
  p.ntiles = tiles;
  p.nsums = 1;
  fill_ws(p, w);
  p.tma_rows = n > 0 ? tensor_map(w, x, n) : 0;
  p.nwalkers = 1;
  const int dev = w->device;
  int64_t grid = (int64_t)g_num_sms[dev] * g_blocks_per_sm;
  if (2 * tiles + 2 < grid) grid = 2 * tiles + 2;     // the walker, the scanner, at most one streaming CTA per unit
  if (grid < 3) grid = 3;
  static CUtensorMap dummy;
  cudaError_t e = sq::launch_seqsum(p, p.tma_rows ? &w->tmap : &dummy, (int)grid, stream);
  if (e != cudaSuccess) return cuda_fail(e);
  g_last = w;
  return SEQSUM_OK;
}

}  // extern "C"

// A plan kept across calls: each tile's plan record (prefix and warps' sums)
// of the latest call, and a second array the next call writes its own into.
struct seqsum_plan {
  int device = -1;
  int64_t tiles = 0;       // tiles the records are for (0: none yet)
  uint4 *rec[2] = {nullptr, nullptr};
  int cur = 0;             // rec[cur] holds the latest call's plan
};

extern "C" {

int seqsum_plan_create(seqsum_plan **out) {
  if (!out) return SEQSUM_EINVAL;
  *out = new (std::nothrow) seqsum_plan();
  return *out ? SEQSUM_OK : SEQSUM_ENOMEM;
}

void seqsum_plan_destroy(seqsum_plan *plan) {
  if (!plan) return;
  std::lock_guard<std::mutex> lk(g_mu);
  if (plan->device >= 0) {
    int prev = 0;
    cudaGetDevice(&prev);
    cudaSetDevice(plan->device);
    cudaDeviceSynchronize();   // calls still in flight may read the records
    cudaFree(plan->rec[0]);
    cudaFree(plan->rec[1]);
    cudaSetDevice(prev);
  }
  delete plan;
}

int seqsum_f64_planned(seqsum_plan *plan, const double *x, int64_t n, double s0, double *out,
                       cudaStream_t stream) {
  if (!plan || n < 0 || !out || (n > 0 && !x)) return SEQSUM_EINVAL;
  std::lock_guard<std::mutex> lk(g_mu);
  int rc = ensure_device_info();
  if (rc) return rc;
  const int64_t tiles = (n + sq::kTileTerms - 1) / sq::kTileTerms;
  Workspace *w = nullptr;
  rc = get_ws(stream, tiles > 0 ? tiles : 1, 1, &w);
  if (rc) return rc;
  bool fresh = false;
  if (plan->device != w->device || plan->tiles != tiles || !plan->rec[0]) {
    // a first call, or a plane of another size: new records, a full (two-pass) call fills them
    cudaError_t e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return cuda_fail(e);
    if (plan->device >= 0) {
      int prev = 0;
      cudaGetDevice(&prev);
      cudaSetDevice(plan->device);
      cudaDeviceSynchronize();
      cudaFree(plan->rec[0]);
      cudaFree(plan->rec[1]);
      cudaSetDevice(prev);
    }
    plan->rec[0] = plan->rec[1] = nullptr;
    plan->tiles = 0;
    const size_t bytes = (size_t)(tiles > 0 ? tiles : 1) * sq::kPrecWords * sizeof(uint4);
    if (cudaMalloc(&plan->rec[0], bytes) != cudaSuccess || cudaMalloc(&plan->rec[1], bytes) != cudaSuccess) {
      cudaFree(plan->rec[0]);
      plan->rec[0] = plan->rec[1] = nullptr;
      g_last_cuda = (int)cudaGetLastError();
      return SEQSUM_ENOMEM;
    }
    cudaMemsetAsync(plan->rec[0], 0, bytes, stream);
    cudaMemsetAsync(plan->rec[1], 0, bytes, stream);
    plan->device = w->device;
    plan->tiles = tiles;
    plan->cur = 0;
    fresh = true;
  }
  Params p;
  memset(&p, 0, sizeof p);
  p.x = x;
  p.x_len = n;
  p.outs = out;
  p.s0 = s0;
  p.n = n;
  p.ntiles = tiles;
  p.nsums = 1;
  fill_ws(p, w);
  if (fresh) {
    p.prec = plan->rec[plan->cur];   // the two-pass call leaves its plan here
  } else {
    p.planned = 1;
    p.prec = plan->rec[plan->cur];
    p.prec_next = plan->rec[plan->cur ^ 1];
  }
  p.tma_rows = n > 0 ? tensor_map(w, x, n) : 0;
  p.nwalkers = 1;
  int64_t grid = (int64_t)g_num_sms[w->device] * g_blocks_per_sm;
  const int64_t units = fresh ? 2 * tiles : tiles;
  if (units + 2 < grid) grid = units + 2;
  if (grid < 3) grid = 3;
  static CUtensorMap dummy;
  cudaError_t e = sq::launch_seqsum(p, p.tma_rows ? &w->tmap : &dummy, (int)grid, stream);
  if (e != cudaSuccess) return cuda_fail(e);
  if (!fresh) plan->cur ^= 1;      // stream order: the next call reads what this one writes
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

int seqsum_f64_strided(const double *x, int64_t n, int32_t stride, const double *s0s, double *outs, float *means,
                       cudaStream_t stream) {
  if (n < 0 || stride < 1 || stride > sq::kMaxStride || !s0s || !outs || (n > 0 && !x)) return SEQSUM_EINVAL;
  double *planes = nullptr;
  int64_t *soffs = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    int rc = ensure_device_info();
    if (rc) return rc;
    Workspace *w = nullptr;
    rc = get_ws(stream, 1, stride, &w);
    if (rc) return rc;
    const int64_t need = n * stride;
    if (!w->soffs) {
      cudaError_t e = cudaMalloc(&w->soffs, (sq::kMaxStride + 1) * sizeof(int64_t));
      if (e != cudaSuccess) return SEQSUM_ENOMEM;
    }
    if (need > w->cap_planes) {
      cudaError_t e = cudaStreamSynchronize(stream);   // earlier calls may still read the old copy
      if (e != cudaSuccess) return cuda_fail(e);
      cudaFree(w->planes);
      w->planes = nullptr;
      w->cap_planes = 0;
      if (cudaMalloc(&w->planes, (need > 0 ? need : 1) * sizeof(double)) != cudaSuccess) {
        g_last_cuda = (int)cudaGetLastError();
        return SEQSUM_ENOMEM;
      }
      w->cap_planes = need;
    }
    planes = w->planes;
    soffs = w->soffs;
    cudaError_t e = sq::launch_deinterleave(x, n, stride, planes, soffs, stream);
    if (e != cudaSuccess) return cuda_fail(e);
  }
  int rc = batched_impl(planes, n * stride, soffs, stride, s0s, outs, true, stream);
  if (rc) return rc;
  if (means) {
    cudaError_t e = sq::launch_mean(outs, stride, n, means, stream);
    if (e != cudaSuccess) return cuda_fail(e);
  }
  return SEQSUM_OK;
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
  cudaSetDevice(prev);
  if (e != cudaSuccess) return cuda_fail(e);
  st->timeout_site = (int32_t)c[sq::C_TO_SITE];
  st->timeout_a = (int64_t)c[sq::C_TO_A];
  st->timeout_b = (int64_t)c[sq::C_TO_B];
  st->check_site = (int32_t)c[sq::C_CHECK_SITE];
  st->check_value = (int64_t)(((uint64_t)c[sq::C_CHECK_HI] << 32) | c[sq::C_CHECK_LO]);
  st->tiles = (int64_t)s[sq::S_TILES];
  st->tiles_complex = (int64_t)s[sq::S_TILE_COMPLEX];
  st->ranges_from_x = (int64_t)s[sq::S_RANGE_X];
  st->lanes_raw = (int64_t)s[sq::S_LANE_RAW];
  st->lanes_raw2 = (int64_t)s[sq::S_LANE_RAW2];
  st->lanes_tie = (int64_t)s[sq::S_LANE_TIE];
  st->walk_batches = (int64_t)s[sq::S_WALK_BATCHES];
  st->walk_segments = (int64_t)s[sq::S_WALK_SEGMENTS];
  st->runs_rejected = (int64_t)s[sq::S_RUN_REJECTED];
  st->terms_dadd = (int64_t)s[sq::S_TERMS_DADD];
  st->raw_rounds = (int64_t)s[sq::S_RAW_ROUNDS];
  st->cy_walk_wait = (int64_t)s[sq::S_CY_WALK_WAIT];
  st->cy_walk_serial = (int64_t)s[sq::S_CY_WALK_SERIAL];
  st->cy_walk_raw = (int64_t)s[sq::S_CY_WALK_RAW];
  st->cy_tma_wait = (int64_t)s[sq::S_CY_TMA_WAIT];
  st->cy_plan = (int64_t)s[sq::S_CY_PLAN];
  st->cy_pfx_wait = (int64_t)s[sq::S_CY_PFX_WAIT];
  st->cy_run = (int64_t)s[sq::S_CY_RUN];
  st->scan_windows = (int64_t)s[sq::S_SCAN_WINDOWS];
  st->scan_polls = (int64_t)s[sq::S_SCAN_POLLS];
  st->pfx_late = (int64_t)s[sq::S_PFX_LATE];
  st->ctas_alone = (int64_t)s[sq::S_ALONE];
  st->tiles_redone = (int64_t)s[sq::S_REDO];
  const int64_t t0 = (int64_t)s[sq::S_T_START], t1 = (int64_t)s[sq::S_T_STREAM_END], t2 = (int64_t)s[sq::S_T_WALK_END];
  st->t_stream_ns = (t0 && t1) ? t1 - t0 : 0;
  st->t_walk_tail_ns = (t1 && t2) ? t2 - t1 : 0;
  st->t_total_ns = (t0 && t2) ? t2 - t0 : 0;
  const int64_t t3 = (int64_t)s[sq::S_T_SCAN_END], t4 = (int64_t)s[sq::S_T_UNITS_END];
  st->t_scan_ns = (t0 && t3) ? t3 - t0 : 0;
  st->t_units_ns = (t0 && t4) ? t4 - t0 : 0;
  st->device_error_bits = (int32_t)err;
  if (err & sq::ERR_CAPACITY) st->device_status = SEQSUM_ECAPACITY;
  else if (err & sq::ERR_BAD_OFFSETS) st->device_status = SEQSUM_EOFFSETS;
  else if (err & (sq::ERR_TMA_TIMEOUT | sq::ERR_WALK_TIMEOUT)) st->device_status = SEQSUM_ETIMEOUT;
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
    case SEQSUM_ECAPACITY: return "more tiles than the scratch holds";
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
    cudaFree(w->planes);
    cudaFree(w->soffs);
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
  if (!w || !out || n < 0 || n > sq::kDbgWords) return SEQSUM_EINVAL;
  cudaError_t e = cudaStreamSynchronize(w->stream);
  if (e == cudaSuccess) e = cudaMemcpy(out, w->dbg, n * sizeof(unsigned long long), cudaMemcpyDeviceToHost);
  if (e == cudaSuccess) e = cudaMemset(w->dbg, 0, sq::kDbgWords * sizeof(unsigned long long));
  return e == cudaSuccess ? SEQSUM_OK : cuda_fail(e);
}

int seqsum_debug_counters(unsigned long long *out, int n) {
  // No lock: this is read while another thread may be blocked inside a call
  // of this library (holding its lock).  A non-blocking stream lets the copy
  // run next to a kernel that has not finished.
  static cudaStream_t side = nullptr;
  Workspace *w = g_last;
  if (!w || !out || n < 1 || n > sq::C_COUNT) return SEQSUM_EINVAL;
  cudaError_t e = cudaSuccess;
  if (!side) e = cudaStreamCreateWithFlags(&side, cudaStreamNonBlocking);
  uint32_t c[sq::C_COUNT];
  if (e == cudaSuccess) e = cudaMemcpyAsync(c, w->ctr, sizeof c, cudaMemcpyDeviceToHost, side);
  if (e == cudaSuccess) e = cudaStreamSynchronize(side);
  if (e != cudaSuccess) return cuda_fail(e);
  for (int i = 0; i < n; i++) out[i] = c[i];
  return SEQSUM_OK;
}

int seqsum_debug_set_plan(int mode) {
  std::lock_guard<std::mutex> lk(g_mu);
  const int old = g_plan_mode;
  g_plan_mode = mode;
  return old;
}

int seqsum_debug_set_fault(int mode, int64_t arg, int64_t wait_ns) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (mode < 0 || mode > 1 || wait_ns < 0) return SEQSUM_EINVAL;
  g_fault_mode = mode;
  g_fault_arg = arg;
  g_wait_ns = wait_ns > 0 ? (uint64_t)wait_ns : 2000000000ull;
  return SEQSUM_OK;
}

const char *seqsum_version(void) { return "seqsum 0.2 (sm_103a)"; }

}  // extern "C"

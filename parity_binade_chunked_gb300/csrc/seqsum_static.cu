// seqsum_f64_static (include/seqsum.h): the single-sum path on scratch that
// lives in file-scope device arrays of a fixed size, so a call allocates
// nothing.  The kernel is the same one seqsum_f64 launches; only where its
// workspace comes from differs.  Nothing here computes any part of a sum.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <stdint.h>
#include <string.h>

#include <mutex>

#include "../../include/seqsum.h"
#include "seqsum_internal.cuh"

namespace {

using sq::Params;
using sq::Rec;

constexpr int64_t kStaticTiles = SEQSUM_STATIC_MAX_TERMS / sq::kTileTerms;
static_assert(kStaticTiles * sq::kTileTerms == SEQSUM_STATIC_MAX_TERMS, "whole tiles");
constexpr int kDbgWords = sq::kDbgAlloc;

// the scratch: tagged plan words and tile headers (zero at the start and
// after every tag wrap), items, counters and statistics (zero at the start;
// the kernel leaves its counters at zero when it ends)
static __device__ __align__(256) uint64_t s_status[kStaticTiles * 2];
static __device__ __align__(256) uint64_t s_cplan[kStaticTiles * sq::kWarps * 4];
constexpr int64_t kStaticGroups = kStaticTiles / sq::kGroupTiles + 1;
static __device__ __align__(256) uint32_t s_grp_cnt[kStaticGroups];
static __device__ __align__(256) uint64_t s_grp_hdr[kStaticGroups];
static __device__ __align__(256) Rec s_grp_seg[kStaticGroups * sq::kGroupSegs];
static __device__ __align__(256) uint16_t s_grp_stile[kStaticGroups * sq::kGroupSegs];
static __device__ __align__(256) Rec s_hdr[kStaticTiles];
static __device__ __align__(256) Rec s_items[kStaticTiles * sq::kTileSlots];
static __device__ __align__(256) uint32_t s_ctr[sq::C_COUNT];
static __device__ __align__(256) unsigned long long s_stats[sq::S_COUNT];
static __device__ __align__(256) unsigned long long s_dbg[kDbgWords];
static __device__ __align__(256) int64_t s_tile_begin[2];
static __device__ __align__(256) unsigned long long s_hb[sq::kHeartbeats];

struct DeviceScratch {
  bool ready = false;
  uint64_t *status = nullptr, *cplan = nullptr, *grp_hdr = nullptr;
  uint32_t *grp_cnt = nullptr;
  Rec *grp_seg = nullptr;
  uint16_t *grp_stile = nullptr;
  Rec *hdr = nullptr, *items = nullptr;
  uint32_t *ctr = nullptr;
  unsigned long long *stats = nullptr, *dbg = nullptr, *hb = nullptr;
  int64_t *tile_begin = nullptr;
  uint32_t epoch = 0;
  int num_sms = 0;
  const void *tm_ptr = nullptr;
  int64_t tm_rows = -1;
  CUtensorMap tmap;
};

std::mutex g_mu;
DeviceScratch g_dev[64];
int g_blocks_per_sm = 0;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

template <class T>
cudaError_t symbol(T **out, const void *sym) {
  void *p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, sym);
  *out = static_cast<T *>(p);
  return e;
}

// Once per device: the addresses of the arrays, the launch shape, and the
// arrays that must start at zero cleared (on `stream`).
cudaError_t setup(DeviceScratch &d, int dev, cudaStream_t stream) {
  cudaError_t e;
  if ((e = symbol(&d.status, s_status)) != cudaSuccess) return e;
  if ((e = symbol(&d.cplan, s_cplan)) != cudaSuccess) return e;
  if ((e = symbol(&d.grp_cnt, s_grp_cnt)) != cudaSuccess) return e;
  if ((e = symbol(&d.grp_hdr, s_grp_hdr)) != cudaSuccess) return e;
  if ((e = symbol(&d.grp_seg, s_grp_seg)) != cudaSuccess) return e;
  if ((e = symbol(&d.grp_stile, s_grp_stile)) != cudaSuccess) return e;
  if ((e = symbol(&d.hdr, s_hdr)) != cudaSuccess) return e;
  if ((e = symbol(&d.items, s_items)) != cudaSuccess) return e;
  if ((e = symbol(&d.ctr, s_ctr)) != cudaSuccess) return e;
  if ((e = symbol(&d.stats, s_stats)) != cudaSuccess) return e;
  if ((e = symbol(&d.dbg, s_dbg)) != cudaSuccess) return e;
  if ((e = symbol(&d.tile_begin, s_tile_begin)) != cudaSuccess) return e;
  if ((e = symbol(&d.hb, s_hb)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  if (g_blocks_per_sm == 0) g_blocks_per_sm = sq::kernel_max_blocks_per_sm();
  if (!g_encode) {
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess) return e;
    if (q != cudaDriverEntryPointSuccess || !fn) return cudaErrorSymbolNotFound;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  if ((e = cudaMemsetAsync(d.status, 0, sizeof s_status, stream)) != cudaSuccess) return e;
  if ((e = cudaMemsetAsync(d.cplan, 0, sizeof s_cplan, stream)) != cudaSuccess) return e;
  if ((e = cudaMemsetAsync(d.grp_cnt, 0, sizeof s_grp_cnt, stream)) != cudaSuccess) return e;
  if ((e = cudaMemsetAsync(d.grp_hdr, 0, sizeof s_grp_hdr, stream)) != cudaSuccess) return e;
  if ((e = cudaMemsetAsync(d.hdr, 0, sizeof s_hdr, stream)) != cudaSuccess) return e;
  if ((e = cudaMemsetAsync(d.ctr, 0, sizeof s_ctr, stream)) != cudaSuccess) return e;
  if ((e = cudaMemsetAsync(d.stats, 0, sizeof s_stats, stream)) != cudaSuccess) return e;
  if ((e = cudaMemsetAsync(d.dbg, 0, sizeof s_dbg, stream)) != cudaSuccess) return e;
  d.epoch = 0;
  d.ready = true;
  return cudaSuccess;
}

// The 2-D view [rows][16] of the plane, 128-byte swizzled boxes of 256 rows
// (the same view seqsum_f64 uses).  0 rows: no TMA.
int64_t tensor_map(DeviceScratch &d, const double *x, int64_t n) {
  if ((reinterpret_cast<uintptr_t>(x) & 15) != 0 || n < 16) return 0;
  const int64_t rows = n / 16;
  if (d.tm_ptr == x && d.tm_rows == rows) return rows;
  cuuint64_t dims[2] = {16, (cuuint64_t)rows};
  cuuint64_t strides[1] = {16 * sizeof(double)};
  cuuint32_t box[2] = {16, 256};
  cuuint32_t estr[2] = {1, 1};
  const CUresult r = g_encode(&d.tmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT64, 2, const_cast<double *>(x), dims, strides,
                              box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) { d.tm_ptr = nullptr; d.tm_rows = -1; return 0; }
  d.tm_ptr = x;
  d.tm_rows = rows;
  return rows;
}

}  // namespace

extern "C" int seqsum_f64_static(const double *x, int64_t n, double s0, double *out, cudaStream_t stream) {
  if (n < 0 || !out || (n > 0 && !x)) return SEQSUM_EINVAL;
  if (n > SEQSUM_STATIC_MAX_TERMS) return SEQSUM_ECAPACITY;
  std::lock_guard<std::mutex> lk(g_mu);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return SEQSUM_ECUDA;
  DeviceScratch &d = g_dev[dev];
  cudaError_t e;
  if (!d.ready && (e = setup(d, dev, stream)) != cudaSuccess) return SEQSUM_ECUDA;
  // the next tag (1..127); the tagged arrays are cleared when it wraps
  if (++d.epoch > 127) {
    if (cudaMemsetAsync(d.status, 0, sizeof s_status, stream) != cudaSuccess ||
        cudaMemsetAsync(d.cplan, 0, sizeof s_cplan, stream) != cudaSuccess ||
        cudaMemsetAsync(d.grp_cnt, 0, sizeof s_grp_cnt, stream) != cudaSuccess ||
        cudaMemsetAsync(d.grp_hdr, 0, sizeof s_grp_hdr, stream) != cudaSuccess ||
        cudaMemsetAsync(d.hdr, 0, sizeof s_hdr, stream) != cudaSuccess)
      return SEQSUM_ECUDA;
    d.epoch = 1;
  }
  const int64_t tiles = (n + sq::kTileTerms - 1) / sq::kTileTerms;
  Params p;
  memset(&p, 0, sizeof p);
  p.x = x;
  p.outs = out;
  p.s0 = s0;
  p.n = n;
  p.ntiles = tiles;
  p.nsums = 1;
  p.epoch = d.epoch;
  p.status = d.status;
  p.cplan = d.cplan;
  p.grp_cnt = d.grp_cnt;
  p.grp_hdr = d.grp_hdr;
  p.grp_seg = d.grp_seg;
  p.grp_stile = d.grp_stile;
  p.hdr = d.hdr;
  p.items = d.items;
  p.ctr = d.ctr;
  p.tile_begin = d.tile_begin;
  p.stats = d.stats;
  p.dbg = d.dbg;
  p.hb = d.hb;
  p.cap_tiles = kStaticTiles;
  p.tma_rows = n > 0 ? tensor_map(d, x, n) : 0;
  p.nwalkers = 1;
  p.wave = 2048;
  int64_t grid = (int64_t)d.num_sms * g_blocks_per_sm;
  if (2 * tiles + 2 < grid) grid = 2 * tiles + 2;
  static CUtensorMap dummy;
  e = sq::launch_seqsum(p, p.tma_rows ? &d.tmap : &dummy, (int)grid, stream);
  return e == cudaSuccess ? SEQSUM_OK : SEQSUM_ECUDA;
}

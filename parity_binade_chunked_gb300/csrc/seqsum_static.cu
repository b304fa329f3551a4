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

// The scratch.  Tagged words (status, headers) and the counters must start
// at zero; the kernel keeps them consistent from call to call (it advances
// the tag itself and clears the tagged words when the tag wraps).
static __device__ __align__(256) uint4 s_status[kStaticTiles];
static __device__ __align__(256) uint4 s_prec[kStaticTiles * sq::kPrecWords];
static __device__ __align__(256) Rec s_hdr[kStaticTiles];
static __device__ __align__(256) Rec s_items[kStaticTiles * sq::kItemSlots];
static __device__ __align__(256) uint32_t s_ctr[sq::C_COUNT];
static __device__ __align__(256) unsigned long long s_stats[sq::S_COUNT];
static __device__ __align__(256) unsigned long long s_dbg[sq::kDbgWords];
static __device__ __align__(256) int64_t s_tile_begin[2];

struct DeviceScratch {
  bool ready = false;
  uint4 *status = nullptr, *prec = nullptr;
  Rec *hdr = nullptr, *items = nullptr;
  uint32_t *ctr = nullptr;
  unsigned long long *stats = nullptr, *dbg = nullptr;
  int64_t *tile_begin = nullptr;
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

// Once per device, with that device current: the arrays' device addresses
// (a host-side name of a __device__ array is not a device address), the
// launch shape, and the arrays that must start at zero cleared on `stream`.
cudaError_t setup(DeviceScratch &d, int dev, cudaStream_t stream) {
  cudaError_t e;
  if ((e = symbol(&d.status, s_status)) != cudaSuccess) return e;
  if ((e = symbol(&d.prec, s_prec)) != cudaSuccess) return e;
  if ((e = symbol(&d.hdr, s_hdr)) != cudaSuccess) return e;
  if ((e = symbol(&d.items, s_items)) != cudaSuccess) return e;
  if ((e = symbol(&d.ctr, s_ctr)) != cudaSuccess) return e;
  if ((e = symbol(&d.stats, s_stats)) != cudaSuccess) return e;
  if ((e = symbol(&d.dbg, s_dbg)) != cudaSuccess) return e;
  if ((e = symbol(&d.tile_begin, s_tile_begin)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  if (g_blocks_per_sm == 0) g_blocks_per_sm = sq::kernel_blocks_per_sm();
  if (!g_encode) {
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess) return e;
    if (q != cudaDriverEntryPointSuccess || !fn) return cudaErrorSymbolNotFound;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  if ((e = cudaMemsetAsync(d.status, 0, sizeof s_status, stream)) != cudaSuccess) return e;
  if ((e = cudaMemsetAsync(d.prec, 0, sizeof s_prec, stream)) != cudaSuccess) return e;
  if ((e = cudaMemsetAsync(d.hdr, 0, sizeof s_hdr, stream)) != cudaSuccess) return e;
  if ((e = cudaMemsetAsync(d.ctr, 0, sizeof s_ctr, stream)) != cudaSuccess) return e;
  if ((e = cudaMemsetAsync(d.stats, 0, sizeof s_stats, stream)) != cudaSuccess) return e;
  if ((e = cudaMemsetAsync(d.dbg, 0, sizeof s_dbg, stream)) != cudaSuccess) return e;
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
  cuuint32_t box[2] = {16, (cuuint32_t)sq::kTileRows};
  cuuint32_t estr[2] = {1, 1};
  const CUresult r = g_encode(&d.tmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT64, 2, const_cast<double *>(x), dims, strides,
                              box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    d.tm_ptr = nullptr;
    d.tm_rows = -1;
    return 0;
  }
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
  const int64_t tiles = (n + sq::kTileTerms - 1) / sq::kTileTerms;
  Params p;
  memset(&p, 0, sizeof p);
  p.x = x;
  p.x_len = n;
  p.outs = out;
  p.s0 = s0;
  p.n = n;
  p.ntiles = tiles;
  p.nsums = 1;
  p.status = d.status;
  p.prec = d.prec;
  p.prec_ws = d.prec;
  p.wave = 2048;
  p.hdr = d.hdr;
  p.items = d.items;
  p.ctr = d.ctr;
  p.tile_begin = d.tile_begin;
  p.stats = d.stats;
  p.dbg = d.dbg;
  p.cap_tiles = kStaticTiles;
  p.wait_ns = 2000000000ull;
  p.tma_rows = n > 0 ? tensor_map(d, x, n) : 0;
  p.nwalkers = 1;
  int64_t grid = (int64_t)d.num_sms * g_blocks_per_sm;
  if (2 * tiles + 2 < grid) grid = 2 * tiles + 2;
  if (grid < 3) grid = 3;
  static CUtensorMap dummy;
  e = sq::launch_seqsum(p, p.tma_rows ? &d.tmap : &dummy, (int)grid, stream);
  return e == cudaSuccess ? SEQSUM_OK : SEQSUM_ECUDA;
}

// The order in which a streaming CTA's tickets name units: the plan unit
// and the run unit of every tile, each once.  Host and device (the host unit
// test checks the order against its definition).
#pragma once
#include <stdint.h>

#if defined(__CUDACC__)
#define SQU_HD __host__ __device__ __forceinline__
#else
#define SQU_HD static inline
#endif

namespace sq {

#if defined(__CUDA_ARCH__)
SQU_HD int64_t u_min(int64_t a, int64_t b) { return min(a, b); }
SQU_HD int64_t u_max(int64_t a, int64_t b) { return max(a, b); }
#else
SQU_HD int64_t u_min(int64_t a, int64_t b) { return a < b ? a : b; }
SQU_HD int64_t u_max(int64_t a, int64_t b) { return a > b ? a : b; }
#endif

// Ticket order.  The run unit of tile t follows the plan unit of tile
// lag(t): for the first kHeadTiles tiles that is tile P (about kHeadAfter
// plan units in: early, so that the walk can start early, yet late enough
// for their prefixes to be published); for the others, tile t + wave (a wave
// behind, so that their prefixes are ready and their terms still in L2).
// Every run unit's ticket is larger than those of the plan units it depends
// on (its tile's and the tiles' before it).  Batched calls start no head
// (every run a wave behind, unit_of_wave).  The plan of tile q has ticket
// q + the runs placed before it; a ticket is decoded piece by piece.
constexpr int64_t kHeadTiles = 128;
constexpr int64_t kHeadAfter = 1024;
SQU_HD int64_t plan_ticket(int64_t q, int64_t H, int64_t W, int64_t P) {
  return q + (q > P ? H : 0) + u_max(0, q - W - H);
}
// Without a head: the plans of the first `wave` tiles, then a run and a plan
// in turn, then the remaining runs (decoded directly).
SQU_HD bool unit_of_wave(int64_t u, int64_t ntiles, int64_t wave, int64_t &tile) {
  const int64_t w = u_min(wave, ntiles);
  if (u < w) { tile = u; return true; }
  const int64_t v = u - w, rest = ntiles - w;
  if (v < 2 * rest) {
    tile = (v & 1) ? w + (v >> 1) : (v >> 1);
    return (v & 1) != 0;
  }
  tile = rest + (v - 2 * rest);
  return false;
}
SQU_HD bool unit_of(int64_t u, int64_t ntiles, int64_t wave, int64_t head, int64_t &tile) {
  if (head == 0) return unit_of_wave(u, ntiles, wave, tile);
  const int64_t n = ntiles, H = u_min(head, n), W = u_min(wave, n);
  const int64_t P = u_min(u_min(u_max(kHeadAfter, H - 1), n - 1), H + W - 1);
  if (u <= P) { tile = u; return true; }               // the first plans
  if (u <= P + H) { tile = u - P - 1; return false; }  // the head's runs
  const int64_t tlast = plan_ticket(n - 1, H, W, P);
  if (u < tlast) {
    if (u - H <= H + W - 1) { tile = u - H; return true; }   // plans with no run between them
    const int64_t v = u + W;                           // then a plan and a run a wave behind in turn
    if ((v & 1) == 0) { tile = v >> 1; return true; }
    tile = ((v - 1) >> 1) - W;
    return false;
  }
  if (u == tlast) { tile = n - 1; return true; }
  int64_t k = u - tlast - 1;                           // the runs after the last plan
  if (P == n - 1) k -= H;
  tile = u_max(H, n - 1 - W) + k;
  return false;
}

}  // namespace sq

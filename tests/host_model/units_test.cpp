// Host test of the ticket order (parity_binade_chunked_gb300/csrc/units.cuh):
// for many plane sizes, waves and heads, unit_of must name the plan unit and
// the run unit of every tile exactly once, in the order its definition gives
// (plan q, then the run units that follow it), and every run unit must come
// after the plan units of its tile and of every tile before it -- the property
// that makes a call's progress certain.
#include "../../parity_binade_chunked_gb300/csrc/units.cuh"

#include <cstdint>
#include <cstdio>
#include <vector>



namespace {

struct Unit { int64_t tile; bool plan; };

// The run unit of tile t follows the plan unit of tile lag(t).
std::vector<Unit> by_definition(int64_t n, int64_t wave, int64_t head) {
  std::vector<int64_t> lag(n);
  if (head == 0) {
    const int64_t w = wave < n ? wave : n;
    for (int64_t t = 0; t < n; t++) lag[t] = (t + w - 1 < n - 1) ? t + w - 1 : n - 1;
  } else {
    const int64_t H = head < n ? head : n, W = wave < n ? wave : n;
    int64_t P = sq::kHeadAfter > H - 1 ? sq::kHeadAfter : H - 1;
    if (P > n - 1) P = n - 1;
    if (P > H + W - 1) P = H + W - 1;
    for (int64_t t = 0; t < n; t++) lag[t] = t < H ? P : ((t + W < n - 1) ? t + W : n - 1);
  }
  std::vector<std::vector<int64_t>> after(n);
  for (int64_t t = 0; t < n; t++) after[lag[t]].push_back(t);
  std::vector<Unit> order;
  for (int64_t q = 0; q < n; q++) {
    order.push_back({q, true});
    for (int64_t t : after[q]) order.push_back({t, false});
  }
  return order;
}

}  // namespace

int main() {
  std::vector<int64_t> sizes;
  for (int64_t n = 1; n <= 300; n++) sizes.push_back(n);
  for (int64_t n : {507, 1023, 1024, 1025, 1151, 1152, 1153, 2025, 2175, 2176, 2177, 3000, 5000, 48600})
    sizes.push_back(n);
  long fails = 0, cases = 0;
  for (int64_t n : sizes) {
    for (int64_t wave : {2048, 512, 100, 7, 1}) {
      for (int64_t head : {(int64_t)0, sq::kHeadTiles, (int64_t)5}) {
        cases++;
        const std::vector<Unit> want = by_definition(n, wave, head);
        std::vector<char> seen(2 * n, 0);
        int64_t last_plan = -1;                       // ticket of the latest plan of tiles 0..t
        std::vector<int64_t> plan_at(n, -1), run_at(n, -1);
        bool ok = (int64_t)want.size() == 2 * n;
        for (int64_t u = 0; ok && u < 2 * n; u++) {
          int64_t t = -1;
          const bool plan = sq::unit_of(u, n, wave, head, t);
          if (t < 0 || t >= n || plan != want[u].plan || t != want[u].tile) { ok = false; break; }
          const int64_t slot = 2 * t + (plan ? 0 : 1);
          if (seen[slot]) { ok = false; break; }
          seen[slot] = 1;
          (plan ? plan_at : run_at)[t] = u;
        }
        for (int64_t t = 0; ok && t < n; t++) {
          if (plan_at[t] > last_plan) last_plan = plan_at[t];
          if (run_at[t] <= last_plan) ok = false;         // a run before a plan it depends on
        }
        if (!ok) {
          if (fails < 10) std::printf("FAIL n=%lld wave=%lld head=%lld\n", (long long)n, (long long)wave, (long long)head);
          fails++;
        }
      }
    }
  }
  std::printf("cases=%ld failures=%ld\n", cases, fails);
  return fails ? 1 : 0;
}

// Host-only driver of the slot map's C ABI for the sanitizer build
// (AddressSanitizer + UndefinedBehaviorSanitizer): a seeded random join /
// finish / step schedule, every error path, and a plain model of the
// expected state checked after each event.  Exit code 0 = all checks held.
#include <cstdint>
#include <cstdio>
#include <string>
#include <vector>

#include "slot_map.h"

namespace bm {
std::string& last_error_slot() {
  thread_local std::string s;
  return s;
}
}  // namespace bm

namespace {

uint64_t rng_state = 0x9E3779B97F4A7C15ull;
uint32_t next_u32() {  // splitmix64
  uint64_t z = (rng_state += 0x9E3779B97F4A7C15ull);
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return (uint32_t)((z ^ (z >> 31)) >> 32);
}

int failures = 0;
void expect(bool ok, const char* what, int step) {
  if (!ok) {
    std::fprintf(stderr, "step %d: %s\n", step, what);
    ++failures;
  }
}

}  // namespace

int main() {
  const int S = 7, cap = 40;
  bm_slot_map* m = nullptr;
  expect(bm_slot_map_create(0, cap, &m) == BM_ERR_INVALID_ARG && m == nullptr, "create rejects 0 streams", -1);
  expect(bm_slot_map_create(S, cap, nullptr) == BM_ERR_INVALID_ARG, "create rejects a null output", -1);
  expect(bm_slot_map_create(S, cap, &m) == BM_OK && m, "create", -1);
  std::vector<int> active(S, 0), len(S, 0);
  for (int step = 0; step < 4000; ++step) {
    const uint32_t r = next_u32() % 100;
    if (r < 30) {  // join with a random prefix (sometimes past the cap, sometimes negative)
      const int want = (int)(next_u32() % (cap + 4)) - 2;
      int slot = -1;
      const bm_status st = bm_slot_map_acquire(m, want, &slot);
      int lowest = -1;
      for (int s = 0; s < S; ++s)
        if (!active[s]) { lowest = s; break; }
      if (want < 0) expect(st == BM_ERR_INVALID_ARG, "negative prefix rejected", step);
      else if (want >= cap) expect(st == BM_ERR_CTX_CAP, "prefix at the cap rejected", step);
      else if (lowest < 0) expect(st == BM_ERR_NO_SLOT, "full map rejected", step);
      else {
        expect(st == BM_OK && slot == lowest, "lowest free slot taken", step);
        if (st == BM_OK) { active[slot] = 1; len[slot] = want; }
      }
    } else if (r < 50) {  // finish (sometimes a free or out-of-range slot)
      const int s = (int)(next_u32() % (S + 2)) - 1;
      const bm_status st = bm_slot_map_release(m, s);
      if (s < 0 || s >= S) expect(st == BM_ERR_INVALID_ARG, "release out of range rejected", step);
      else if (!active[s]) expect(st == BM_ERR_SLOT_FREE, "double release rejected", step);
      else {
        expect(st == BM_OK, "release", step);
        active[s] = 0;
        len[s] = 0;
      }
    } else {  // a step over a random subset (sometimes with a duplicate or a free slot)
      std::vector<int32_t> b;
      for (int s = 0; s < S; ++s)
        if (active[s] && next_u32() % 3) b.push_back(s);
      if (b.empty()) {
        expect(bm_slot_map_check_batch(m, b.data(), 0) == BM_ERR_INVALID_ARG, "empty batch rejected", step);
        continue;
      }
      const uint32_t twist = next_u32() % 10;
      bool bad = false;
      if (twist == 0) { b.push_back(b[0]); bad = true; }  // duplicate
      if (twist == 1) {
        for (int s = 0; s < S; ++s)
          if (!active[s]) { b.push_back(s); bad = true; break; }
      }
      bool at_cap = false;
      for (int32_t s : b) at_cap = at_cap || (active[s] && len[s] >= cap);
      const bm_status st = bm_slot_map_advance(m, b.data(), (int)b.size());
      if (bad) expect(st != BM_OK, "bad batch rejected", step);
      else if (at_cap) expect(st == BM_ERR_CTX_CAP, "stream at the cap rejected", step);
      else {
        expect(st == BM_OK, "advance", step);
        for (int32_t s : b) len[s] += 1;
      }
    }
    for (int s = 0; s < S; ++s) {  // the map agrees with the model after every event
      int L = -1;
      const bm_status st = bm_slot_map_length(m, s, &L);
      if (active[s]) expect(st == BM_OK && L == len[s], "length matches", step);
      else expect(st == BM_ERR_SLOT_FREE, "free slot has no length", step);
    }
    int n = 0;
    for (int s = 0; s < S; ++s) n += active[s];
    expect(bm_slot_map_active_count(m) == n, "active count matches", step);
  }
  bm_slot_map_destroy(m);
  bm_slot_map_destroy(nullptr);
  if (failures) std::fprintf(stderr, "%d check(s) failed\n", failures);
  return failures ? 1 : 0;
}

// Host bookkeeping of the KV slots (no device state).
//
// The KV-slot isolation page (§1) gives the lifecycle this class keeps: a
// stream is seeded into a stable slot once, when it joins; each decode step
// appends one position; the slot is released when the stream retires (a
// logical reset — the buffer is reused without a wipe); and nothing about a
// batch-composition change touches a continuing stream's slot.  The crash
// root-cause page (§3) is the failure this rules out: pools keyed by batch
// size, wiped on a batch-size change, then re-seeded from a host prefix that
// no longer held the decode-appended K/V.
#pragma once

#include <cstdint>
#include <string>
#include <vector>

#include "../../include/bitmoe.h"

namespace bm {

class SlotMap {
 public:
  SlotMap(int max_streams, int ctx_cap);

  int max_streams() const { return (int)len_.size(); }
  int ctx_cap() const { return cap_; }
  int active_count() const;
  bool active(int slot) const { return slot >= 0 && slot < max_streams() && active_[slot]; }
  int length(int slot) const { return len_[slot]; }

  // Lowest free slot with length len; errors as kv_slot_seed.
  bm_status acquire(int len, int* slot, std::string* err);
  bm_status release(int slot, std::string* err);
  // Slot ids in range, distinct, active, with room for one more position.
  bm_status check_batch(const int32_t* slots, int B, std::string* err) const;
  void advance(const int32_t* slots, int B);
  // A prompt of n positions written into an active slot.
  void advance_by(int slot, int n);

 private:
  int cap_;
  std::vector<uint8_t> active_;
  std::vector<int> len_;
};

}  // namespace bm

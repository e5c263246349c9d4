#include "slot_map.h"

#include <new>

#include "errors.h"

namespace bm {

SlotMap::SlotMap(int max_streams, int ctx_cap) : cap_(ctx_cap), active_(max_streams, 0), len_(max_streams, 0) {}

int SlotMap::active_count() const {
  int n = 0;
  for (uint8_t a : active_) n += a;
  return n;
}

bm_status SlotMap::acquire(int len, int* slot, std::string* err) {
  if (len < 0) {
    *err = "kv slot: negative length " + std::to_string(len);
    return BM_ERR_INVALID_ARG;
  }
  if (len >= cap_) {
    *err = "kv slot: prefix of " + std::to_string(len) + " positions leaves no room under the context cap " +
           std::to_string(cap_) + " (rejected at admission)";
    return BM_ERR_CTX_CAP;
  }
  for (int s = 0; s < max_streams(); ++s) {
    if (!active_[s]) {
      active_[s] = 1;
      len_[s] = len;
      *slot = s;
      return BM_OK;
    }
  }
  *err = "kv slot: all " + std::to_string(max_streams()) + " slots are active";
  return BM_ERR_NO_SLOT;
}

bm_status SlotMap::release(int slot, std::string* err) {
  if (slot < 0 || slot >= max_streams()) {
    *err = "kv slot: slot id " + std::to_string(slot) + " out of range";
    return BM_ERR_INVALID_ARG;
  }
  if (!active_[slot]) {
    *err = "kv slot: slot " + std::to_string(slot) + " is not active (double release?)";
    return BM_ERR_SLOT_FREE;
  }
  active_[slot] = 0;
  len_[slot] = 0;
  return BM_OK;
}

bm_status SlotMap::check_batch(const int32_t* slots, int B, std::string* err) const {
  if (B < 1 || B > max_streams()) {
    *err = "batch: B = " + std::to_string(B) + " outside [1, " + std::to_string(max_streams()) + "]";
    return BM_ERR_INVALID_ARG;
  }
  if (!slots) {
    *err = "batch: null slot list";
    return BM_ERR_INVALID_ARG;
  }
  std::vector<uint8_t> seen(max_streams(), 0);
  for (int i = 0; i < B; ++i) {
    const int s = slots[i];
    if (s < 0 || s >= max_streams()) {
      *err = "batch: slot id " + std::to_string(s) + " out of range";
      return BM_ERR_INVALID_ARG;
    }
    if (seen[s]) {
      *err = "batch: slot " + std::to_string(s) + " appears twice";
      return BM_ERR_INVALID_ARG;
    }
    seen[s] = 1;
    if (!active_[s]) {
      *err = "batch: slot " + std::to_string(s) + " is not active";
      return BM_ERR_SLOT_FREE;
    }
    if (len_[s] >= cap_) {
      *err = "batch: slot " + std::to_string(s) + " has reached the context cap " + std::to_string(cap_);
      return BM_ERR_CTX_CAP;
    }
  }
  return BM_OK;
}

void SlotMap::advance(const int32_t* slots, int B) {
  for (int i = 0; i < B; ++i) len_[slots[i]] += 1;
}

void SlotMap::advance_by(int slot, int n) { len_[slot] += n; }

}  // namespace bm

// ------------------------------------------------------------------ C ABI

struct bm_slot_map {
  bm::SlotMap map;
  bm_slot_map(int s, int c) : map(s, c) {}
};

extern "C" {

bm_status bm_slot_map_create(int max_streams, int ctx_cap, bm_slot_map** out) {
  if (!out) return bm::set_error(BM_ERR_INVALID_ARG, "bm_slot_map_create: null output pointer");
  *out = nullptr;
  if (max_streams < 1 || max_streams > 4096 || ctx_cap < 1)
    return bm::set_error(BM_ERR_INVALID_ARG, "bm_slot_map_create: max_streams must be in [1, 4096], ctx_cap >= 1");
  *out = new (std::nothrow) bm_slot_map(max_streams, ctx_cap);
  if (!*out) return bm::set_error(BM_ERR_OOM, "bm_slot_map_create: out of host memory");
  return bm::ok();
}

void bm_slot_map_destroy(bm_slot_map* m) { delete m; }

bm_status bm_slot_map_acquire(bm_slot_map* m, int len, int* slot_out) {
  if (!m || !slot_out) return bm::set_error(BM_ERR_INVALID_ARG, "bm_slot_map_acquire: null argument");
  std::string err;
  const bm_status s = m->map.acquire(len, slot_out, &err);
  return s == BM_OK ? bm::ok() : bm::set_error(s, err);
}

bm_status bm_slot_map_release(bm_slot_map* m, int slot) {
  if (!m) return bm::set_error(BM_ERR_INVALID_ARG, "bm_slot_map_release: null map");
  std::string err;
  const bm_status s = m->map.release(slot, &err);
  return s == BM_OK ? bm::ok() : bm::set_error(s, err);
}

bm_status bm_slot_map_check_batch(const bm_slot_map* m, const int32_t* slots, int B) {
  if (!m) return bm::set_error(BM_ERR_INVALID_ARG, "bm_slot_map_check_batch: null map");
  std::string err;
  const bm_status s = m->map.check_batch(slots, B, &err);
  return s == BM_OK ? bm::ok() : bm::set_error(s, err);
}

bm_status bm_slot_map_advance(bm_slot_map* m, const int32_t* slots, int B) {
  if (!m) return bm::set_error(BM_ERR_INVALID_ARG, "bm_slot_map_advance: null map");
  std::string err;
  const bm_status s = m->map.check_batch(slots, B, &err);
  if (s != BM_OK) return bm::set_error(s, err);
  m->map.advance(slots, B);
  return bm::ok();
}

bm_status bm_slot_map_length(const bm_slot_map* m, int slot, int* len_out) {
  if (!m || !len_out) return bm::set_error(BM_ERR_INVALID_ARG, "bm_slot_map_length: null argument");
  if (!m->map.active(slot)) return bm::set_error(BM_ERR_SLOT_FREE, "bm_slot_map_length: slot is not active");
  *len_out = m->map.length(slot);
  return bm::ok();
}

int bm_slot_map_active_count(const bm_slot_map* m) { return m ? m->map.active_count() : 0; }

}  // extern "C"

// Per-thread last-error message of the C ABI.
#pragma once

#include <string>

#include "../../include/bitmoe.h"

namespace bm {

std::string& last_error_slot();

inline bm_status set_error(bm_status s, const std::string& msg) {
  last_error_slot() = msg;
  return s;
}

inline bm_status ok() {
  last_error_slot().clear();
  return BM_OK;
}

}  // namespace bm

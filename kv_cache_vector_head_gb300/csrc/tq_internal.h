// Internal helpers shared by the host and CUDA translation units of libtq.
#pragma once

#include <cstdarg>
#include <cstdio>

#include "../../include/tq.h"

namespace tq {

// Thread-local last-error message (tq_last_error).
void set_error(const char* fmt, ...);
void clear_error();

inline tq_status fail(tq_status s, const char* msg) {
  set_error("%s", msg);
  return s;
}
inline tq_status ok() {
  clear_error();
  return TQ_OK;
}

}  // namespace tq

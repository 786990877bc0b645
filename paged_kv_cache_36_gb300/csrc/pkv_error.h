// Thread-local error reporting shared by every entry point of libpkv.
#pragma once

#include <cstdarg>
#include <cstdio>
#include <string>

#include "pkv.h"

namespace pkv {

inline std::string& last_error_slot() {
  static thread_local std::string msg;
  return msg;
}

// Records a printf-style message for pkv_last_error() and returns `code`.
inline int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  std::vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  last_error_slot() = buf;
  return code;
}

inline int ok() { return PKV_OK; }

}  // namespace pkv

// Host-side helpers shared by the library's translation units.
#pragma once

#include <cstdarg>
#include <cstdint>
#include <cstdio>

#include "pagedkv.h"

namespace pkv {

// Records a printf-style message as this thread's last error and returns `code`.
int fail(int code, const char* fmt, ...);

// Clears this thread's last error and returns PKV_OK.
int ok();

// Wait limit and debug switch passed to every kernel with a pipeline wait.
struct WaitConfig {
  uint64_t timeout_ns;
  int32_t force_timeout;
};
WaitConfig wait_config();

}  // namespace pkv

#define PKV_REQUIRE(cond, ...)                          \
  do {                                                  \
    if (!(cond)) return ::pkv::fail(PKV_EINVAL, __VA_ARGS__); \
  } while (0)

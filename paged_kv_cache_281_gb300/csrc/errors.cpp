// Thread-local error text, the library version and the wait-limit knob.
#include <atomic>
#include <cstring>

#include "internal.h"

namespace {
thread_local char g_last_error[512] = "";
std::atomic<uint64_t> g_timeout_ns{2000000000ull};
std::atomic<int32_t> g_force_timeout{0};
}  // namespace

namespace pkv {

int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  return code;
}

int ok() {
  g_last_error[0] = '\0';
  return PKV_OK;
}

WaitConfig wait_config() { return WaitConfig{g_timeout_ns.load(), g_force_timeout.load()}; }

}  // namespace pkv

extern "C" const char* pkv_last_error(void) { return g_last_error; }

extern "C" int pkv_version(void) { return 100; }

extern "C" int pkv_debug_set_wait(int32_t force_timeout, uint64_t timeout_ns) {
  g_force_timeout.store(force_timeout ? 1 : 0);
  if (timeout_ns > 0) g_timeout_ns.store(timeout_ns);
  return pkv::ok();
}

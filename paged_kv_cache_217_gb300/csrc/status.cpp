#include "status.h"

#include <cstdarg>
#include <cstdio>

namespace {
thread_local char g_msg[512] = "";
}

namespace pkv {

pkv_status_t fail(pkv_status_t st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  std::vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
  va_end(ap);
  return st;
}

pkv_status_t ok() {
  g_msg[0] = '\0';
  return PKV_OK;
}

}  // namespace pkv

extern "C" const char* pkv_last_error_string(void) { return g_msg; }

extern "C" const char* pkv_version(void) { return "paged_kv 0.1.0 (sm_103a)"; }

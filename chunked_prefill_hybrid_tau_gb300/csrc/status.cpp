// Status strings and the per-thread error message.
#include "common.h"

namespace hb {

static thread_local std::string g_last_error;

void set_error(const char* fmt, ...) {
  char buf[1024];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
}

void clear_error() { g_last_error.clear(); }

}  // namespace hb

extern "C" const char* hb_status_string(int status) {
  switch (status) {
    case HB_OK: return "ok";
    case HB_ERR_INVALID_ARG: return "invalid argument";
    case HB_ERR_CAPACITY: return "output capacity too small";
    case HB_ERR_OUT_OF_PAGES: return "out of KV pages";
    case HB_ERR_CUDA: return "CUDA error";
    case HB_ERR_TIMEOUT: return "device wait timed out";
    case HB_ERR_UNSUPPORTED: return "unsupported device or shape";
    case HB_ERR_DEVICE: return "device-side index check failed";
    default: return "unknown status";
  }
}

extern "C" const char* hb_last_error(void) { return hb::g_last_error.c_str(); }

extern "C" int32_t hb_version(void) { return 100; }

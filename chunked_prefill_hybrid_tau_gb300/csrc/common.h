// Internal helpers shared by the library's translation units.
#pragma once
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <string>

#include "hb.h"

namespace hb {

// Thread-local message of the last failing call (see hb_last_error()).
void set_error(const char* fmt, ...);
void clear_error();

// Status word codes written by kernels (first error wins).
enum DeviceError : int { kDevOk = 0, kDevTimeout = 1, kDevIndex = 2 };

#define HB_REQUIRE(cond, ...)                 \
  do {                                        \
    if (!(cond)) {                            \
      ::hb::set_error(__VA_ARGS__);           \
      return HB_ERR_INVALID_ARG;              \
    }                                         \
  } while (0)

}  // namespace hb

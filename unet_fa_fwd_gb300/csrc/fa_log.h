// fa_log.h — launch logging shared by the library's translation units: with
// FA_LOG=1 in the environment every kernel launch is described on stderr
// (kernel, tiles, grid, stages, shared / tensor memory, work units), one line
// per launch.
#pragma once

#include <cstdarg>
#include <cstdio>
#include <cstdlib>

namespace fa {

inline bool log_enabled() {
  const char* e = std::getenv("FA_LOG");
  return e && e[0] == '1' && e[1] == 0;
}

inline void log_launch(const char* fmt, ...) {
  if (!log_enabled()) return;
  std::va_list ap;
  va_start(ap, fmt);
  std::fputs("[fa] ", stderr);
  std::vfprintf(stderr, fmt, ap);
  std::fputc('\n', stderr);
  va_end(ap);
}

}  // namespace fa

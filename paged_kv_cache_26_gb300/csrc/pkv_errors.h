// Per-thread error message shared by every translation unit of libpagedkv.so.
#pragma once
#include <string>

inline std::string& pkv_error_slot() {
  static thread_local std::string msg;
  return msg;
}
inline void pkv_set_error(const std::string& msg) { pkv_error_slot() = msg; }
inline int pkv_fail(int code, const std::string& msg) {
  pkv_set_error(msg);
  return code;
}

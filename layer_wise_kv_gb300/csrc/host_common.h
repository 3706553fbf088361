// Host-side helpers shared by the C-ABI entry points: the thread-local error
// message, argument checks and CUDA error mapping.
#pragma once

#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <string>

#include "kvs.h"

namespace kvs {

void set_error(const char* fmt, ...);
void clear_error();

// Returns `code` after recording the message.
kvs_status fail(kvs_status code, const char* fmt, ...);

}  // namespace kvs

#define KVS_REQUIRE(cond, ...)                                         \
  do {                                                                 \
    if (!(cond)) return ::kvs::fail(KVS_ERR_INVALID, __VA_ARGS__);     \
  } while (0)

#define KVS_SUPPORTED(cond, ...)                                       \
  do {                                                                 \
    if (!(cond)) return ::kvs::fail(KVS_ERR_UNSUPPORTED, __VA_ARGS__); \
  } while (0)

// Map the last launch error to KVS_ERR_CUDA.
#define KVS_CHECK_LAUNCH(what)                                                      \
  do {                                                                              \
    cudaError_t e_ = cudaGetLastError();                                            \
    if (e_ != cudaSuccess)                                                          \
      return ::kvs::fail(KVS_ERR_CUDA, "%s: %s", (what), cudaGetErrorString(e_));   \
  } while (0)

#define KVS_CUDA(call, what)                                                        \
  do {                                                                              \
    cudaError_t e_ = (call);                                                        \
    if (e_ != cudaSuccess)                                                          \
      return ::kvs::fail(KVS_ERR_CUDA, "%s: %s", (what), cudaGetErrorString(e_));   \
  } while (0)

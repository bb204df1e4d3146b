// pkv_internal.h -- host-side helpers shared by the translation units of libpkv.so.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "pkv.h"

namespace pkv {

// Record the calling thread's last error (printf-style) and return `status`.
int set_error(int status, const char *fmt, ...);
void clear_error();

// Device address of the library's device status word in the current context
// (looked up with cudaGetSymbolAddress on every call).  NULL on failure.
int32_t *device_status_word();

// Streaming-multiprocessor count of the current device (cached per device).
int sm_count();

// Map a CUDA runtime error to PKV_ERR_CUDA with a message, or PKV_OK.
int check_cuda(cudaError_t e, const char *what);

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Split-KV chunk: every sequence's keys are cut into chunks of this many tokens,
// anchored at token 0, whatever the batch looks like.  (A build-time constant: a
// multiple of 32, at most 2048.)
#ifndef PKV_SPLIT_TOKENS
#define PKV_SPLIT_TOKENS 512
#endif
constexpr int kSplitTokens = PKV_SPLIT_TOKENS;
static_assert(kSplitTokens % 32 == 0 && kSplitTokens <= 2048, "split size");
constexpr int kMaxQHeads = 256;
constexpr int kMaxGroupRows = 8192;  // G * max rows per sequence (row-group CTAs of 16 rows)
// About two seconds of SM clock: the limit of any wait inside a kernel.
constexpr long long kWaitLimitCycles = 4000000000LL;
// Limit of the attention pipeline's stage waits for the next launches:
// kWaitLimitCycles unless pkv_debug_set_wait_limit() changed it.  (The final wait
// for a kernel's own copies in flight always uses kWaitLimitCycles.)
long long pipeline_wait_limit();

}  // namespace pkv

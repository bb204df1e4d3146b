// pkv_api.cu -- error reporting, the device status word and small shared host helpers.
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "pkv_internal.h"

// Bits set by kernels when they meet a condition only the device can see
// (see PKV_DEV_* in pkv.h).  Read and cleared by pkv_device_status().
__device__ int32_t g_pkv_device_status = 0;

namespace pkv {

namespace {
thread_local char t_last_error[512] = {0};
constexpr int kMaxDevices = 64;
std::mutex g_mutex;
int g_sm_count[kMaxDevices] = {0};

int current_device()
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return -1;
    return dev;
}
}  // namespace

int set_error(int status, const char *fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(t_last_error, sizeof t_last_error, fmt, ap);
    va_end(ap);
    return status;
}

void clear_error() { t_last_error[0] = '\0'; }

int check_cuda(cudaError_t e, const char *what)
{
    if (e == cudaSuccess)
        return PKV_OK;
    return set_error(PKV_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

namespace {
std::atomic<long long> g_wait_limit{kWaitLimitCycles};
}

long long pipeline_wait_limit() { return g_wait_limit.load(std::memory_order_relaxed); }

int32_t *device_status_word()
{
    // Looked up on every call, in the caller's current context: a cached address
    // would outlive a cudaDeviceReset or belong to another context of the same device
    // (the module, and the word with it, is loaded again in each context).  The
    // lookup is a host-side table query, not a stream operation.
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_pkv_device_status) != cudaSuccess)
        return nullptr;
    return static_cast<int32_t *>(p);
}

int sm_count()
{
    const int dev = current_device();
    if (dev < 0)
        return 1;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_sm_count[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            n = 1;
        g_sm_count[dev] = n;
    }
    return g_sm_count[dev];
}

}  // namespace pkv

extern "C" int pkv_abi_version(void) { return 2; }

extern "C" const char *pkv_last_error_string(void) { return pkv::t_last_error; }

extern "C" int pkv_debug_set_wait_limit(long long cycles)
{
    pkv::clear_error();
    pkv::g_wait_limit.store(cycles < 0 ? pkv::kWaitLimitCycles : cycles, std::memory_order_relaxed);
    return PKV_OK;
}

extern "C" int pkv_device_status(void *stream, int32_t *bits)
{
    pkv::clear_error();
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int rc = pkv::check_cuda(cudaStreamSynchronize(st), "cudaStreamSynchronize");
    if (rc)
        return rc;
    int32_t *word = pkv::device_status_word();
    if (!word)
        return pkv::set_error(PKV_ERR_CUDA, "cudaGetSymbolAddress of the device status word failed");
    int32_t host = 0;
    rc = pkv::check_cuda(cudaMemcpyAsync(&host, word, sizeof host, cudaMemcpyDeviceToHost, st),
                         "read device status word");
    if (rc)
        return rc;
    rc = pkv::check_cuda(cudaMemsetAsync(word, 0, sizeof host, st), "clear device status word");
    if (rc)
        return rc;
    rc = pkv::check_cuda(cudaStreamSynchronize(st), "cudaStreamSynchronize");
    if (rc)
        return rc;
    if (bits)
        *bits = host;
    if (host & PKV_DEV_TIMEOUT)
        return pkv::set_error(PKV_ERR_TIMEOUT, "a bounded wait inside a kernel expired (bits 0x%x)", host);
    if (host & (PKV_DEV_OUT_OF_BLOCKS | PKV_DEV_INDEX_FULL))
        return pkv::set_error(PKV_ERR_OUT_OF_BLOCKS,
                              "the block allocator ran out of free blocks or index slots (bits 0x%x)", host);
    if (host & (PKV_DEV_BAD_BLOCK | PKV_DEV_TABLE_OVERRUN))
        return pkv::set_error(PKV_ERR_BAD_BLOCK,
                              "a kernel met a block id outside the pool or a length past the "
                              "table / max_context_len (bits 0x%x)", host);
    if (host & PKV_DEV_TOO_MANY_ROWS)
        return pkv::set_error(PKV_ERR_SHAPE,
                              "a sequence had more query rows than max_q_rows_per_seq (bits 0x%x)", host);
    if (host & PKV_DEV_BAD_TREE)
        return pkv::set_error(PKV_ERR_SHAPE,
                              "a draft tree had a parent index outside [0, node) (bits 0x%x)", host);
    if (host & PKV_DEV_BAD_RANGE)
        return pkv::set_error(PKV_ERR_SHAPE,
                              "a token range lay outside [0, total_tokens] (bits 0x%x)", host);
    return PKV_OK;
}

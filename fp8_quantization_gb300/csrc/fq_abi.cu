// Library-wide entry points of libfq.so: status strings, error reporting,
// version, and the per-device SM count used to size persistent grids.
#include <atomic>

#include "fq_common.cuh"

namespace fq {

namespace {
thread_local int g_last_cuda_error = 0;
constexpr int kMaxDevices = 64;
std::atomic<int> g_sm_count[kMaxDevices];
}  // namespace

void set_last_cuda_error(int err) { g_last_cuda_error = err; }

int sm_count()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return 152;
    int n = g_sm_count[dev].load(std::memory_order_relaxed);
    if (n <= 0) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            n <= 0)
            n = 152;
        g_sm_count[dev].store(n, std::memory_order_relaxed);
    }
    return n;
}

}  // namespace fq

extern "C" const char *fq_status_string(int status)
{
    switch (status) {
    case FQ_OK:
        return "FQ_OK";
    case FQ_ERR_NULL:
        return "FQ_ERR_NULL: a required pointer is NULL";
    case FQ_ERR_SHAPE:
        return "FQ_ERR_SHAPE: size negative, too large or not a multiple of the block";
    case FQ_ERR_ALIGN:
        return "FQ_ERR_ALIGN: pointer not 16-byte aligned";
    case FQ_ERR_ARG:
        return "FQ_ERR_ARG: argument out of range";
    case FQ_ERR_CUDA:
        return "FQ_ERR_CUDA: the CUDA runtime reported an error";
    default:
        return "unknown fq_status";
    }
}

extern "C" int fq_last_cuda_error(void) { return fq::g_last_cuda_error; }

extern "C" int fq_version(void) { return 100; }

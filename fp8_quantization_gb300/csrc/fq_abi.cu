// Library-wide entry points of libfq.so: status strings, error reporting,
// version, and the per-device SM count used to size persistent grids.
#include <atomic>

#include <cudaTypedefs.h>

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

namespace {
// The driver's tensor-map encoder.  The runtime (and with it the driver and
// the current device's primary context) is initialised first: in a process
// whose first CUDA call is this lookup, the lookup and the encoder fail
// otherwise.  Only a successful lookup is kept.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder()
{
    static std::atomic<void *> fn{nullptr};
    void *p = fn.load(std::memory_order_acquire);
    if (p)
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    if (cudaFree(nullptr) != cudaSuccess)  // initialises the runtime; frees nothing
        cudaGetLastError();                 // (no device): not left for the caller
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
        return nullptr;
    fn.store(p, std::memory_order_release);
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
}
}  // namespace

bool encode_tensor_map_2d(CUtensorMap *map, CUtensorMapDataType dtype, const void *base,
                          uint64_t inner, uint64_t rows, uint64_t row_pitch, uint32_t box_inner,
                          uint32_t box_rows, CUtensorMapSwizzle swizzle, bool promote_l2)
{
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc)
        return false;
    const cuuint64_t dims[2] = {inner, rows};
    const cuuint64_t strides[1] = {row_pitch};
    const cuuint32_t box[2] = {box_inner, box_rows};
    const cuuint32_t elem_strides[2] = {1, 1};
    return enc(map, dtype, 2, const_cast<void *>(base), dims, strides, box, elem_strides,
               CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
               promote_l2 ? CU_TENSOR_MAP_L2_PROMOTION_L2_128B : CU_TENSOR_MAP_L2_PROMOTION_NONE,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_tensor_map_2d_u8(CUtensorMap *map, const void *base, uint64_t inner, uint64_t rows,
                             uint64_t row_pitch, uint32_t box_inner, uint32_t box_rows,
                             bool promote_l2)
{
    return encode_tensor_map_2d(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, base, inner, rows, row_pitch,
                                box_inner, box_rows, CU_TENSOR_MAP_SWIZZLE_NONE, promote_l2);
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

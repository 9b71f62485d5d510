// api.cu -- error reporting, the device status word and the scale-layout helpers of the C ABI.
#include <stdarg.h>
#include <stdio.h>

#include "common.cuh"

namespace nvq {

static thread_local char g_last_error[512] = "";

void set_error(const char* fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
    va_end(ap);
}

nvq_status cuda_status(cudaError_t e, const char* what)
{
    set_error("%s: %s (%s)", what, cudaGetErrorString(e), cudaGetErrorName(e));
    return NVQ_ERR_CUDA;
}

// One status word per device that loads the library (module-scope device variable).
__device__ DeviceStatus g_device_status;

DeviceStatus* device_status_ptr()
{
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_status) != cudaSuccess) return nullptr;
    return static_cast<DeviceStatus*>(p);
}

static unsigned long long g_wait_limit = 1ull << 32;

unsigned long long wait_limit() { return g_wait_limit; }

static int g_tail_path = NVQ_TAIL_AUTO;

int tail_path() { return g_tail_path; }

}  // namespace nvq

using namespace nvq;

extern "C" const char* nvq_last_error(void) { return g_last_error; }

extern "C" nvq_status nvq_set_wait_limit(uint64_t cycles)
{
    NVQ_CHECK_ARG(cycles >= 1, NVQ_ERR_ARG, "nvq_set_wait_limit: the limit must be at least 1 cycle");
    g_wait_limit = cycles;
    set_error("");
    return NVQ_OK;
}

extern "C" nvq_status nvq_set_tail_path(int32_t path)
{
    NVQ_CHECK_ARG(path == NVQ_TAIL_AUTO || path == NVQ_TAIL_GATHER || path == NVQ_TAIL_ROWS, NVQ_ERR_ARG,
                  "nvq_set_tail_path: unknown path %d", path);
    g_tail_path = path;
    set_error("");
    return NVQ_OK;
}

extern "C" nvq_status nvq_device_status(void* stream, int32_t* status, int32_t* where)
{
    NVQ_CHECK_ARG(status, NVQ_ERR_ARG, "nvq_device_status: null status pointer");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_status(e, "cudaStreamSynchronize");
    DeviceStatus h{0, 0};
    e = cudaMemcpyFromSymbol(&h, g_device_status, sizeof h);
    if (e != cudaSuccess) return cuda_status(e, "cudaMemcpyFromSymbol(status)");
    DeviceStatus z{0, 0};
    e = cudaMemcpyToSymbol(g_device_status, &z, sizeof z);
    if (e != cudaSuccess) return cuda_status(e, "cudaMemcpyToSymbol(status)");
    *status = h.status;
    if (where) *where = h.where;
    set_error("");
    return NVQ_OK;
}

extern "C" int64_t nvq_sf_cols(int64_t ktot) { return ((ktot / 16) + 3) / 4 * 4; }

extern "C" int64_t nvq_sf_bytes(int64_t rows, int64_t sf_cols) { return (rows + 127) / 128 * 128 * sf_cols; }

extern "C" int64_t nvq_sf_offset(int64_t row, int64_t col, int64_t sf_cols) { return sf_offset(row, col, sf_cols); }

// api.cu -- library-wide entry points: device status, status strings and
// the cached SM count used to size persistent grids.
#include "common.cuh"

namespace fp8bs {

int gemm_read_and_clear_status(cudaStream_t st);     // gemm.cu
int decode_read_and_clear_status(cudaStream_t st);   // decode.cu

int device_sm_count() {
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    if (dev >= 64) {
        int n = 1;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        return n;
    }
    if (cache[dev] == 0) {
        int n = 1;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) n = 1;
        cache[dev] = n;
    }
    return cache[dev];
}

}  // namespace fp8bs

using namespace fp8bs;

extern "C" fp8_status fp8_device_status(void* stream) {
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(st) != cudaSuccess) return FP8_ERR_CUDA;
    const int v = gemm_read_and_clear_status(st);
    const int d = decode_read_and_clear_status(st);
    if (v < 0 || d < 0) return FP8_ERR_CUDA;
    if (v != 0) return static_cast<fp8_status>(v);
    return d == 0 ? FP8_OK : static_cast<fp8_status>(d);
}

extern "C" const char* fp8_status_string(fp8_status status) {
    switch (status) {
        case FP8_OK: return "ok";
        case FP8_ERR_INVALID_ARG: return "invalid argument (pointer, size, alignment, or a ue8m0 scale that is not a power of two)";
        case FP8_ERR_UNSUPPORTED: return "unsupported shape";
        case FP8_ERR_CUDA: return "CUDA error";
        case FP8_ERR_TIMEOUT: return "a kernel's bounded wait timed out";
        case FP8_ERR_WORKSPACE: return "workspace missing or too small";
    }
    return "unknown status";
}

extern "C" int fp8_num_sms(void) { return device_sm_count(); }

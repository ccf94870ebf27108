// noalloc.cu - the GEMM for callers that cannot allocate device memory.
//
// Some callers must not call cudaMalloc: code that runs inside a framework
// whose memory pool owns the whole device (a raw allocation there can fail
// or fragment the pool), and latency-critical paths where cudaMalloc and
// cudaFree may synchronise the device.  gemm_run_noalloc serves them: it
// runs the same kernel as gemm_run, but the kernel's only scratch memory,
// its 4-byte status word, lives in a fixed file-scope device array instead of
// a buffer allocated by gemm_create, and all host-side state lives on the
// stack.  The caller still passes A, B, C, D and bias.
#include <mutex>

#include "../../include/gemm.h"
#include "gemm_internal.h"

namespace gemm_sm103 {
gemm_status_t run_unallocated(const gemm_desc_t* desc, const void* A, const void* B, const void* C, void* D,
                              const float* bias, uint32_t* status, int sm_count, cudaStream_t stream);
}

namespace {

// Scratch for every call on a device: 64 words (256 bytes), of which a call
// uses kWordsPerCall.  Each GPU that loads this library holds the array
// until the process exits.
constexpr int kScratchWords = 64;
constexpr int kWordsPerCall = 1;          // the kernel's status word
static __device__ __align__(256) uint32_t g_noalloc_scratch[kScratchWords];

// In host code `g_noalloc_scratch` names a host-side stand-in, not device
// memory: its device address is looked up once per device (with that device
// current) and cached here.
constexpr int kMaxDevices = 64;
struct DeviceState {
    std::once_flag once;
    cudaError_t err = cudaSuccess;
    uint32_t* scratch = nullptr;
    int sm_count = 0;
};
DeviceState g_devices[kMaxDevices];

void set_up(DeviceState* st) {
    void* ptr = nullptr;
    int dev = 0;
    st->err = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (st->err == cudaSuccess) st->err = cudaGetDevice(&dev);
    if (st->err == cudaSuccess) st->err = cudaDeviceGetAttribute(&st->sm_count, cudaDevAttrMultiProcessorCount, dev);
    if (st->err != cudaSuccess) cudaGetLastError();
    st->scratch = static_cast<uint32_t*>(ptr);
}

}  // namespace

extern "C" gemm_status_t gemm_run_noalloc(const gemm_desc_t* desc, const void* A, const void* B, const void* C,
                                          void* D, const float* bias, void* stream, int32_t wait) {
    static_assert(kWordsPerCall <= kScratchWords, "scratch array too small");
    if (!desc || (wait != 0 && wait != 1)) return GEMM_ERR_INVALID_ARG;
    // The scratch a call needs must fit the fixed array; larger needs are refused.
    if (kWordsPerCall > kScratchWords) return GEMM_ERR_UNSUPPORTED;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) {
        cudaGetLastError();
        return GEMM_ERR_NO_DEVICE;
    }
    if (dev >= kMaxDevices) return GEMM_ERR_UNSUPPORTED;
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_NO_DEVICE;
    }
    if (major != 10 || minor != 3) return GEMM_ERR_NO_DEVICE;
    DeviceState* st = &g_devices[dev];
    std::call_once(st->once, set_up, st);       // first call on this device: look up the array's address
    if (st->err != cudaSuccess || !st->scratch) return GEMM_ERR_CUDA;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // The array keeps the previous call's contents: clear the status word.
    if (cudaMemsetAsync(st->scratch, 0, kWordsPerCall * sizeof(uint32_t), s) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    const gemm_status_t r = gemm_sm103::run_unallocated(desc, A, B, C, D, bias, st->scratch, st->sm_count, s);
    if (r != GEMM_OK || !wait) return r;
    uint32_t word = 0;
    if (cudaStreamSynchronize(s) != cudaSuccess ||
        cudaMemcpy(&word, st->scratch, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    return word ? GEMM_ERR_TIMEOUT : GEMM_OK;
}

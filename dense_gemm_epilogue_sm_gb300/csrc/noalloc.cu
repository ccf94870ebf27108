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
#include <atomic>
#include <mutex>

#include "../../include/gemm.h"
#include "gemm_internal.h"

namespace gemm_sm103 {
// One-shot plan and launch with every host object on the stack (api.cpp), the
// kernel's status word at `status` (cleared on `stream` right before the
// launch, once every check has passed); `*launched` tells whether a kernel
// was queued (empty problems queue none).
gemm_status_t run_unallocated(const gemm_desc_t* desc, const void* A, const void* B, const void* C, void* D,
                              const float* bias, uint32_t* status, int sm_count, cudaStream_t stream,
                              VariantCache* cache, bool* launched);
}

namespace {

// Scratch for every call on a device: 64 words (256 bytes), of which a call
// uses kWordsPerCall.  Each GPU that loads this library holds the array
// until the process exits.
constexpr int kScratchWords = 64;
constexpr int kWordsPerCall = 1;          // the kernel's status word
static __device__ __align__(256) uint32_t g_noalloc_scratch[kScratchWords];

// In host code `g_noalloc_scratch` names a host-side stand-in, not device
// memory: its device address is looked up per device (with that device
// current) and cached here, with the device's SM count and the kernel
// variants' launch set-up.  A set-up that fails is tried again on the next
// call; one that succeeds is kept until the process exits.
constexpr int kMaxDevices = 64;
struct DeviceState {
    std::mutex mu;
    std::atomic<bool> ready{false};
    uint32_t* scratch = nullptr;
    int sm_count = 0;
    gemm_sm103::VariantCache variants;
};
DeviceState g_devices[kMaxDevices];

gemm_status_t set_up(DeviceState* st, int dev) {
    if (st->ready.load(std::memory_order_acquire)) return GEMM_OK;
    std::lock_guard<std::mutex> lock(st->mu);
    if (st->ready.load(std::memory_order_relaxed)) return GEMM_OK;
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_NO_DEVICE;
    }
    if (major != 10 || minor != 3) return GEMM_ERR_NO_DEVICE;
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || !ptr) {
        cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    st->scratch = static_cast<uint32_t*>(ptr);
    st->sm_count = sms;
    st->ready.store(true, std::memory_order_release);
    return GEMM_OK;
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
    DeviceState* st = &g_devices[dev];
    const gemm_status_t su = set_up(st, dev);     // first call on this device: look up the array's address
    if (su != GEMM_OK) return su;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    bool launched = false;
    const gemm_status_t r = gemm_sm103::run_unallocated(desc, A, B, C, D, bias, st->scratch, st->sm_count, s,
                                                        &st->variants, &launched);
    if (r != GEMM_OK || !wait || !launched) return r;
    uint32_t word = 0;
    if (cudaStreamSynchronize(s) != cudaSuccess ||
        cudaMemcpy(&word, st->scratch, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    return word ? GEMM_ERR_TIMEOUT : GEMM_OK;
}

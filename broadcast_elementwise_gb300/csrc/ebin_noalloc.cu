// ebin_execute_noalloc: plan execution for callers that must not have the
// library allocate device memory.
//
// ebin_execute keeps one device status word per (device, stream) and creates
// it with cudaMalloc the first time a validating operator (integer Div, Mod,
// Pow; BitShift) runs on a stream.  Some callers cannot allow that: an
// application whose device memory is entirely carved up by its own arena
// allocator, a plugin whose host framework forbids allocation while work is
// being enqueued, or a latency-critical loop where cudaMalloc's implicit
// synchronisation is unacceptable.  This entry point runs the same kernels,
// through the same checks (ebin::prepare_launch), but keeps their status
// words in a fixed array that lives in the library's own device image, so
// nothing is allocated, ever.  ebin_noalloc_read_status reads a word back.
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "ebin.h"
#include "ebin_launch.h"
#include "ebin_plan.h"

namespace {

// The scratch: EBIN_NOALLOC_STATUS_SLOTS status words (256 bytes) in every
// device that loads the library, kept until the process exits.
static __device__ __align__(256) uint32_t g_noalloc_status[EBIN_NOALLOC_STATUS_SLOTS];

constexpr int kMaxDevices = 128;

struct DeviceSetup {
    bool done = false;
    uint32_t *status = nullptr;  // device address of g_noalloc_status on this device
};

std::mutex g_setup_mu;
DeviceSetup g_setup[kMaxDevices];

// Device address of slot `slot` of the array on the current device.  Once per
// device, with that device current, the array's address is looked up (in host
// code the name of a __device__ variable is only a stand-in, never a device
// address).
ebin_status slot_address(int slot, uint32_t **word) {
    if (slot < 0 || slot >= EBIN_NOALLOC_STATUS_SLOTS) return EBIN_ERR_INVALID_ARG;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return EBIN_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return EBIN_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lk(g_setup_mu);
    DeviceSetup &s = g_setup[dev];
    if (!s.done) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_status) != cudaSuccess || !p) {
            cudaGetLastError();
            return EBIN_ERR_CUDA;
        }
        s.status = static_cast<uint32_t *>(p);
        s.done = true;
    }
    *word = s.status + slot;
    return EBIN_OK;
}

// Copy one status word to the host after the stream's work (no allocation).
ebin_status read_word(const uint32_t *word, cudaStream_t s, uint32_t *bits) {
    uint32_t h = 0;
    if (cudaMemcpyAsync(&h, word, sizeof(h), cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return EBIN_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return EBIN_ERR_CUDA;
    *bits = h;
    return EBIN_OK;
}

}  // namespace

extern "C" ebin_status ebin_execute_noalloc(ebin_plan_t plan, const void *A, const void *B,
                                            void *out, void *stream, int status_slot,
                                            uint32_t *status_bits) {
    if (!plan || plan->rank_c >= 0) return EBIN_ERR_INVALID_ARG;   // two-input plans only
    if (status_slot < 0 || status_slot >= EBIN_NOALLOC_STATUS_SLOTS) return EBIN_ERR_INVALID_ARG;
    const ebin_plan_s &p = *plan;
    if (status_bits) *status_bits = 0;
    if (p.numel == 0) return EBIN_OK;
    uint32_t *word = nullptr;
    ebin_status st = slot_address(status_slot, &word);
    if (st != EBIN_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);

    // the same checks and launch description as ebin_execute, with the slot as
    // the status word (only validating operators' kernels write it)
    ebin::Launch L;
    if ((st = ebin::prepare_launch(p, A, B, out, s, word, L)) != EBIN_OK) return st;
    // the slot keeps the previous call's bits: clear it, in stream order
    if (cudaMemsetAsync(word, 0, sizeof(uint32_t), s) != cudaSuccess) return EBIN_ERR_CUDA;
    const cudaError_t e = ebin::launch(L);
    ebin::count_launch();
    if (e != cudaSuccess) return EBIN_ERR_CUDA;
    return status_bits ? read_word(word, s, status_bits) : EBIN_OK;
}

extern "C" ebin_status ebin_noalloc_read_status(int status_slot, void *stream, uint32_t *bits) {
    if (!bits) return EBIN_ERR_INVALID_ARG;
    *bits = 0;
    uint32_t *word = nullptr;
    const ebin_status st = slot_address(status_slot, &word);
    if (st != EBIN_OK) return st;
    return read_word(word, static_cast<cudaStream_t>(stream), bits);
}

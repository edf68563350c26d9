// ebin_execute_noalloc: plan execution for callers that must not have the
// library allocate device memory.
//
// ebin_execute keeps one device status word per (device, stream) and creates
// it with cudaMalloc the first time a validating operator (integer Div, Mod,
// Pow; BitShift) runs on a stream.  Some callers cannot allow that: an
// application whose device memory is entirely carved up by its own arena
// allocator, a plugin whose host framework forbids allocation while work is
// being enqueued, or a latency-critical loop where cudaMalloc's implicit
// synchronisation is unacceptable.  This entry point runs the same kernels but
// keeps their status words in a fixed array that lives in the library's own
// device image, so nothing is allocated, ever.
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
    int num_sms = 1;
};

std::mutex g_setup_mu;
DeviceSetup g_setup[kMaxDevices];

// Once per device, with that device current: look up the array's device
// address (the host-side name of a __device__ variable is only a stand-in)
// and the SM count.
ebin_status setup_device(int dev, DeviceSetup *out) {
    if (dev < 0 || dev >= kMaxDevices) return EBIN_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lk(g_setup_mu);
    DeviceSetup &s = g_setup[dev];
    if (!s.done) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_status) != cudaSuccess || !p)
            return EBIN_ERR_CUDA;
        int sms = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return EBIN_ERR_CUDA;
        s.status = static_cast<uint32_t *>(p);
        s.num_sms = sms > 0 ? sms : 1;
        s.done = true;
    }
    *out = s;
    return EBIN_OK;
}

int dt_class(ebin_dtype t) {
    switch (t) {
    case EBIN_FLOAT32: return ebin::DT_F32;
    case EBIN_FLOAT16: return ebin::DT_F16;
    case EBIN_BFLOAT16: return ebin::DT_BF16;
    case EBIN_INT32: return ebin::DT_I32;
    case EBIN_INT64: return ebin::DT_I64;
    case EBIN_UINT8: return ebin::DT_U8;
    case EBIN_UINT32: return ebin::DT_U32;
    case EBIN_BOOL: return ebin::DT_BOOL;
    case EBIN_INT8: return ebin::DT_I8;
    case EBIN_INT16: return ebin::DT_I16;
    case EBIN_UINT16: return ebin::DT_U16;
    case EBIN_UINT64: return ebin::DT_U64;
    case EBIN_DOUBLE: return ebin::DT_F64;
    }
    return -1;
}

bool overlaps(const void *p, int64_t pb, const void *q, int64_t qb) {
    const uintptr_t a = (uintptr_t)p, b = (uintptr_t)q;
    return pb > 0 && qb > 0 && a < b + (uintptr_t)qb && b < a + (uintptr_t)pb;
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
    const bool plain_b =
        p.op != EBIN_OP_BATCHNORM && p.op != EBIN_OP_CLIP && p.op != EBIN_OP_BIAS_PRELU &&
        p.op != EBIN_OP_BIAS_PRELU_BN;
    const bool b_needed = !(p.op == EBIN_OP_CLIP && !p.attrs.clip_has_min && !p.attrs.clip_has_max) &&
                          !p.attrs.with_scalar;
    if (!A || !out || (b_needed && !B)) return EBIN_ERR_INVALID_ARG;
    if (p.attrs.with_scalar) B = nullptr;   // B is the attribute value, never read

    // same aliasing rule as ebin_execute
    const int64_t isz = (int64_t)ebin_dtype_size(p.dt);
    const int64_t isz_b = (int64_t)ebin_dtype_size(p.dt_b);
    const int64_t out_bytes = p.numel * (int64_t)ebin_dtype_size(p.out_dt);
    if (overlaps(A, p.span_a * isz, out, out_bytes) &&
        !(A == out && !p.strided_a && p.numel_a == p.numel && p.dt == p.out_dt))
        return EBIN_ERR_ALIAS;
    if (B && overlaps(B, p.span_b * isz_b, out, out_bytes) &&
        !(plain_b && B == out && !p.strided_b && p.numel_b == p.numel && p.dt_b == p.out_dt))
        return EBIN_ERR_ALIAS;

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return EBIN_ERR_CUDA;
    DeviceSetup setup;
    const ebin_status st = setup_device(dev, &setup);
    if (st != EBIN_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);

    // the slot keeps the previous call's bits: clear it, in stream order
    uint32_t *word = setup.status + status_slot;
    if (cudaMemsetAsync(word, 0, sizeof(uint32_t), s) != cudaSuccess) return EBIN_ERR_CUDA;

    ebin::Launch L{};
    L.op = p.op;
    L.dt = dt_class(p.dt);
    L.dt_b = dt_class(p.dt_b);
    L.family = p.family;
    L.g = p.g;
    L.numel = p.numel;
    L.A = A;
    L.B = B;
    L.out = out;
    L.args.fmod = p.attrs.fmod;
    L.args.direction = p.attrs.direction;
    L.args.eps = p.attrs.epsilon;
    L.args.has_min = p.attrs.clip_has_min;
    L.args.has_max = p.attrs.clip_has_max;
    L.args.plane = p.plane;
    L.args.with_scalar = p.attrs.with_scalar;
    L.args.scalar_b = p.attrs.scalar_b;
    L.stream = s;
    L.num_sms = setup.num_sms;
    L.status = word;  // only the validating operators' kernels write it
    if (L.family != ebin::FAM_GENERAL_STRIDED) {
        const uintptr_t G = 16 / (uintptr_t)isz;
        const uintptr_t out_align = G * (uintptr_t)ebin_dtype_size(p.out_dt);
        const bool aligned = ((uintptr_t)A % 16 == 0) && (!B || (uintptr_t)B % 16 == 0) &&
                             ((uintptr_t)out % out_align == 0);
        if (!aligned) L.family = ebin::FAM_GENERAL_STRIDED;
    }
    const cudaError_t e = ebin::launch(L);
    ebin::count_launch();
    if (e != cudaSuccess) return EBIN_ERR_CUDA;
    if (status_bits) {
        uint32_t h = 0;
        if (cudaMemcpyAsync(&h, word, sizeof(h), cudaMemcpyDeviceToHost, s) != cudaSuccess)
            return EBIN_ERR_CUDA;
        if (cudaStreamSynchronize(s) != cudaSuccess) return EBIN_ERR_CUDA;
        *status_bits = h;
    }
    return EBIN_OK;
}

// qoq_w4a8_gemm_noalloc: the W4A8 GEMM for callers that cannot allocate
// device memory.
//
// Some callers have no allocator of their own to draw a workspace from, for
// example a plugin running inside another framework's engine that is handed
// only its input and output buffers, or a latency-critical path that must
// not call cudaMalloc because it can synchronize the device.  This entry
// point takes the GEMM's scratch (status word, arrival counters and
// partial-tile slots) from a fixed array that lives in the library itself,
// so the caller only provides inputs and outputs.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "../../include/qoq.h"
#include "qoq_internal.h"

namespace {

// Fixed scratch shared by every call on a device: 8 MiB.  Whether a shape
// fits depends on the shape, not on M alone: the call needs
// qoq_gemm_workspace_bytes(M, N, K, group) <= 8 MiB (on a 152-SM GB300 every
// Llama-3-8B linear layer up to M = 64 fits).  Each GPU that loads the
// library keeps this array until the process exits.
constexpr size_t kNoAllocScratchBytes = 8u << 20;
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_mu;
void *g_scratch_ptr[qoq::kMaxDevices] = {};
int g_sms[qoq::kMaxDevices] = {};

// Once per device, with that device current: the device address of the
// scratch array (the host-side symbol is not a device pointer) and the SM count.
int setup_current_device(void **ptr, int *sms) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return QOQ_ERR_CUDA;
    if (dev < 0 || dev >= qoq::kMaxDevices) return QOQ_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return QOQ_ERR_CUDA;
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            return QOQ_ERR_CUDA;
        g_scratch_ptr[dev] = p;
        g_sms[dev] = n;
    }
    *ptr = g_scratch_ptr[dev];
    *sms = g_sms[dev];
    return QOQ_OK;
}

bool is_aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace

extern "C" int qoq_w4a8_gemm_noalloc(const int8_t *Qx, const uint16_t *s_x, const int32_t *t_x,
                                     const void *packed, const uint16_t *s_w, int M, int N, int K,
                                     int group, uint16_t *O, qoq_stream_t stream) {
    if (M <= 0 || N <= 0 || K <= 0) return QOQ_ERR_INVALID_ARG;
    if (group != 0 && group != 128) return QOQ_ERR_UNSUPPORTED;
    if (N % 128 != 0 || K % 128 != 0 || N / 128 > 65535) return QOQ_ERR_UNSUPPORTED;
    if (!Qx || !s_x || !packed || !s_w || !O || (group == 0 && !t_x)) return QOQ_ERR_INVALID_ARG;
    if (!is_aligned(Qx, 16) || !is_aligned(packed, 16) || !is_aligned(s_x, 2) || !is_aligned(s_w, 2) ||
        !is_aligned(O, 16) || (t_x && !is_aligned(t_x, 4)))
        return QOQ_ERR_MISALIGNED;
    void *scratch = nullptr;
    int sms = 0;
    int st = setup_current_device(&scratch, &sms);
    if (st != QOQ_OK) return st;
    const qoq::GemmPlan plan = qoq::plan_gemm(M, N, K, group, sms);
    if (plan.path < 1 || plan.path > 3) return QOQ_ERR_UNSUPPORTED;
    if (plan.total * (plan.ctas + 1ll) >= (1ll << 32)) return QOQ_ERR_UNSUPPORTED;
    if (plan.ws_bytes > kNoAllocScratchBytes) return QOQ_ERR_WORKSPACE;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // The array keeps whatever the previous call left; the GEMM needs its
    // status word, counters and partial slots to start at zero (the
    // activation-operand scratch after them is fully overwritten each call).
    if (cudaMemsetAsync(scratch, 0, plan.zero_bytes, s) != cudaSuccess) return QOQ_ERR_CUDA;
    qoq::GemmArgs a;
    a.Qx = Qx;
    a.s_x = s_x;
    a.t_x = t_x;
    a.packed = packed;
    a.s_w = s_w;
    a.M = M;
    a.N = N;
    a.K = K;
    a.group = group;
    a.act = nullptr;
    a.O = O;
    a.acc_out = nullptr;
    a.ws = scratch;
    a.debug_flags = 0;
    a.timeout_ns = 2000000000ull;
    a.pdl = false;
    return qoq::launch_gemm(a, plan, s) == cudaSuccess ? QOQ_OK : QOQ_ERR_CUDA;
}

// Status word of the scratch array (its first 4 bytes), read like
// qoq_workspace_status reads a caller's workspace.  Each
// qoq_w4a8_gemm_noalloc call clears the word before it launches, so read it
// after a call and before the next one on the device.
extern "C" int qoq_noalloc_status(uint32_t *host_status, qoq_stream_t stream) {
    if (!host_status) return QOQ_ERR_INVALID_ARG;
    void *scratch = nullptr;
    int sms = 0;
    int st = setup_current_device(&scratch, &sms);
    if (st != QOQ_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    uint32_t v = 0;
    cudaError_t e = cudaMemcpyAsync(&v, scratch, sizeof(v), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e == cudaSuccess) e = cudaMemsetAsync(scratch, 0, sizeof(v), s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return QOQ_ERR_CUDA;
    *host_status = v;
    if (v & 8u) return QOQ_ERR_DEVICE;  // bounds-check build: a skipped access, the cause of any expired wait
    if (v & 1u) return QOQ_ERR_TIMEOUT;
    if (v & 2u) return QOQ_ERR_DEVICE;
    return QOQ_OK;
}

// sk_noalloc.cu - sk_gemm for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc for a workspace: plug-ins whose host application
// owns every device allocation, processes that must stay inside a memory budget fixed at
// start-up, and latency-critical loops in which cudaMalloc / cudaFree would synchronise
// the device. sk_gemm_noalloc serves them with scratch that the library owns: one
// file-scope device array of SK_NOALLOC_SCRATCH_BYTES, which every GPU that loads the
// library holds until the process exits. The first call on a device looks up the array's
// address; make that first call before any stream capture.
//
// The array's name is only a host-side stand-in in host code, not a device address, so
// the address is looked up once per device with cudaGetSymbolAddress, with that device
// current, and passed to the GEMM. All calls on a device share the array and it keeps the
// last call's contents; each call therefore clears the status word and the flags (and,
// for atomic reduction, the partial tiles) before the GEMM. Calls whose kernels overlap
// on the GPU (different streams, or several host threads) race on the array.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "sk.h"
#include "sk_kernels.h"

namespace {

static __device__ __align__(256) unsigned char g_scratch[SK_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
void* g_scratch_ptr[kMaxDevices] = {};
std::mutex g_scratch_mu;

// Device address of g_scratch on the current device (looked up on first use).
int32_t scratch_address(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SK_ECUDA;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || !p) {
            cudaGetLastError();
            return SK_ECUDA;
        }
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return SK_OK;
}

}  // namespace

extern "C" int32_t sk_gemm_noalloc(const void* A, const void* B, void* C, sk_dtype c_dtype, int32_t M, int32_t N,
                                   int32_t K, sk_layout layout, sk_schedule s, sk_reduction r, int32_t num_sms,
                                   void* stream) {
    if (M < 0 || N < 0 || K < 0) return SK_EINVAL;
    if (M == 0 || N == 0 || K == 0) return sk_gemm(A, B, C, c_dtype, M, N, K, layout, s, r, num_sms, nullptr, 0, stream);
    const int64_t need = sk_workspace_size(M, N, K, num_sms, s, r);
    if (need < 0) return static_cast<int32_t>(need);
    if (need > static_cast<int64_t>(SK_NOALLOC_SCRATCH_BYTES)) return SK_EWORKSPACE;
    void* ws = nullptr;
    const int32_t e = scratch_address(&ws);
    if (e != SK_OK) return e;
    // What must start at zero, by the workspace layout of this schedule: the status word and
    // the flags or counters (and, with atomic reduction, the partial tiles, which peers
    // accumulate into); in Split-K slab mode the per-tile arrival counters after the slabs
    // (the slabs themselves are written in full).
    int64_t off[2], len[2];
    const int32_t ez = sk::workspace_zero_spans(M, N, K, num_sms, &s, r, off, len);
    if (ez != SK_OK) return ez;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    for (int i = 0; i < 2; ++i) {
        if (len[i] <= 0) continue;
        if (off[i] < 0 || off[i] + len[i] > need ||
            cudaMemsetAsync(static_cast<unsigned char*>(ws) + off[i], 0, static_cast<size_t>(len[i]), st) !=
                cudaSuccess) {
            cudaGetLastError();
            return SK_ECUDA;
        }
    }
    return sk_gemm(A, B, C, c_dtype, M, N, K, layout, s, r, num_sms, ws, static_cast<size_t>(need), stream);
}

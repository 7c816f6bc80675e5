// sk_host.cu - GEMMs whose operands and results live in host memory.
//
// sk_gemm_host runs `count` problems of one shape. For each it copies A and B from host
// memory into a device staging set, runs sk_gemm on that set, and copies C back to host
// memory. With one staging set everything runs in order on the caller's stream. With two
// sets and two copy streams the work is software-pipelined: problem i + 1's uploads and
// problem i - 1's download run on the copy engines while problem i's GEMM runs on the SMs.
// Events order the three streams:
//   - an upload into set j waits until the GEMM that last read set j has completed;
//   - a GEMM waits for its own uploads, and for the download that last read its set's C;
//   - a download waits for its GEMM.
// The caller's stream finally waits for every download, so its completion means every C
// is in host memory. The pages have no counterpart: this is the library's end-to-end call
// for callers that hold their matrices in host memory.
#include <cuda_runtime.h>
#include <stdint.h>

#include "sk.h"
#include "sk_kernels.h"

namespace {

constexpr int64_t kSetAlign = 256;

int64_t round_set(int64_t x) { return (x + kSetAlign - 1) / kSetAlign * kSetAlign; }

// Byte offsets of A, B and C inside one staging set, and the set's size.
struct SetLayout {
    int64_t a_bytes, b_bytes, c_bytes;
    int64_t b_off, c_off, bytes;
};

bool set_layout(int32_t M, int32_t N, int32_t K, int32_t c_dtype, SetLayout* L) {
    if (M < 0 || N < 0 || K < 0) return false;
    if (c_dtype != SK_F32 && c_dtype != SK_BF16) return false;
    L->a_bytes = static_cast<int64_t>(M) * K * 2;
    L->b_bytes = static_cast<int64_t>(K) * N * 2;
    L->c_bytes = static_cast<int64_t>(M) * N * (c_dtype == SK_BF16 ? 2 : 4);
    L->b_off = round_set(L->a_bytes);
    L->c_off = L->b_off + round_set(L->b_bytes);
    L->bytes = L->c_off + round_set(L->c_bytes);
    return true;
}

// The events of one pipelined call: `start` orders the copy streams after the caller's
// earlier work; up/done/down[j] mark set j's uploads, GEMM and download.
struct Events {
    cudaEvent_t start = nullptr;
    cudaEvent_t up[2] = {nullptr, nullptr};
    cudaEvent_t done[2] = {nullptr, nullptr};
    cudaEvent_t down[2] = {nullptr, nullptr};

    bool create() {
        cudaEvent_t* all[] = {&start, &up[0], &up[1], &done[0], &done[1], &down[0], &down[1]};
        for (cudaEvent_t* e : all)
            if (cudaEventCreateWithFlags(e, cudaEventDisableTiming) != cudaSuccess) return false;
        return true;
    }
    // An event destroyed while still pending is released once the device reaches it.
    ~Events() {
        cudaEvent_t all[] = {start, up[0], up[1], done[0], done[1], down[0], down[1]};
        for (cudaEvent_t e : all)
            if (e) cudaEventDestroy(e);
    }
};

int32_t cuda_fail() {
    cudaGetLastError();
    return SK_ECUDA;
}

}  // namespace

extern "C" int64_t sk_host_staging_size(int32_t M, int32_t N, int32_t K, sk_dtype c_dtype, int32_t depth) {
    SetLayout L;
    if ((depth != 1 && depth != 2) || !set_layout(M, N, K, c_dtype, &L)) return SK_EINVAL;
    return depth * L.bytes;
}

extern "C" int32_t sk_gemm_host(int32_t count, const void* const* A, const void* const* B, void* const* C,
                                sk_dtype c_dtype, int32_t M, int32_t N, int32_t K, sk_layout layout, sk_schedule s,
                                sk_reduction r, int32_t num_sms, void* staging, size_t staging_bytes, int32_t depth,
                                void* workspace, size_t ws_bytes, void* stream, void* copy_in, void* copy_out) {
    // Checks that need no device come first, so that a bad call touches nothing.
    SetLayout L;
    if (count < 0 || (depth != 1 && depth != 2) || !set_layout(M, N, K, c_dtype, &L)) return SK_EINVAL;
    if (count == 0 || M == 0 || N == 0) return SK_OK;
    if (!A || !B || !C) return SK_EINVAL;
    for (int32_t i = 0; i < count; ++i) {
        if (!C[i]) return SK_EINVAL;
        if (K > 0 && (!A[i] || !B[i])) return SK_EINVAL;
    }
    if (depth == 2 && (!copy_in || !copy_out || copy_in == copy_out || copy_in == stream || copy_out == stream))
        return SK_EINVAL;
    if (!staging || (reinterpret_cast<uintptr_t>(staging) & (kSetAlign - 1)) != 0 ||
        static_cast<int64_t>(staging_bytes) < depth * L.bytes)
        return SK_EWORKSPACE;
    unsigned char* base = static_cast<unsigned char*>(staging);
    // The GEMM's own checks, on staging set 0 (every set has the same alignment and size).
    const int32_t e = sk::gemm_check(base, base + L.b_off, base + L.c_off, c_dtype, M, N, K, layout, &s, r, num_sms,
                                     workspace, ws_bytes);
    if (e != SK_OK) return e;

    cudaStream_t g = static_cast<cudaStream_t>(stream);
    const size_t a_bytes = static_cast<size_t>(L.a_bytes), b_bytes = static_cast<size_t>(L.b_bytes),
                 c_bytes = static_cast<size_t>(L.c_bytes);
    auto set = [&](int j, int64_t off) { return base + j * L.bytes + off; };

    if (depth == 1) {
        for (int32_t i = 0; i < count; ++i) {
            if (a_bytes && cudaMemcpyAsync(set(0, 0), A[i], a_bytes, cudaMemcpyHostToDevice, g) != cudaSuccess)
                return cuda_fail();
            if (b_bytes && cudaMemcpyAsync(set(0, L.b_off), B[i], b_bytes, cudaMemcpyHostToDevice, g) != cudaSuccess)
                return cuda_fail();
            const int32_t ge = sk_gemm(set(0, 0), set(0, L.b_off), set(0, L.c_off), c_dtype, M, N, K, layout, s, r,
                                       num_sms, workspace, ws_bytes, stream);
            if (ge != SK_OK) return ge;
            if (cudaMemcpyAsync(C[i], set(0, L.c_off), c_bytes, cudaMemcpyDeviceToHost, g) != cudaSuccess)
                return cuda_fail();
        }
        return SK_OK;
    }

    cudaStream_t u = static_cast<cudaStream_t>(copy_in), o = static_cast<cudaStream_t>(copy_out);
    Events ev;
    if (!ev.create()) return cuda_fail();
    // The copy streams start after the caller's earlier work on `stream` (which may still
    // read or write the staging sets).
    if (cudaEventRecord(ev.start, g) != cudaSuccess || cudaStreamWaitEvent(u, ev.start, 0) != cudaSuccess ||
        cudaStreamWaitEvent(o, ev.start, 0) != cudaSuccess)
        return cuda_fail();
    for (int32_t i = 0; i < count; ++i) {
        const int j = i & 1;
        const bool reused = i >= 2;  // set j was used by problem i - 2
        if (reused && cudaStreamWaitEvent(u, ev.done[j], 0) != cudaSuccess) return cuda_fail();
        if (a_bytes && cudaMemcpyAsync(set(j, 0), A[i], a_bytes, cudaMemcpyHostToDevice, u) != cudaSuccess)
            return cuda_fail();
        if (b_bytes && cudaMemcpyAsync(set(j, L.b_off), B[i], b_bytes, cudaMemcpyHostToDevice, u) != cudaSuccess)
            return cuda_fail();
        if (cudaEventRecord(ev.up[j], u) != cudaSuccess || cudaStreamWaitEvent(g, ev.up[j], 0) != cudaSuccess)
            return cuda_fail();
        if (reused && cudaStreamWaitEvent(g, ev.down[j], 0) != cudaSuccess) return cuda_fail();
        const int32_t ge = sk_gemm(set(j, 0), set(j, L.b_off), set(j, L.c_off), c_dtype, M, N, K, layout, s, r,
                                   num_sms, workspace, ws_bytes, stream);
        if (ge != SK_OK) return ge;
        if (cudaEventRecord(ev.done[j], g) != cudaSuccess || cudaStreamWaitEvent(o, ev.done[j], 0) != cudaSuccess)
            return cuda_fail();
        if (cudaMemcpyAsync(C[i], set(j, L.c_off), c_bytes, cudaMemcpyDeviceToHost, o) != cudaSuccess ||
            cudaEventRecord(ev.down[j], o) != cudaSuccess)
            return cuda_fail();
    }
    for (int j = 0; j < 2 && j < count; ++j)
        if (cudaStreamWaitEvent(g, ev.down[j], 0) != cudaSuccess) return cuda_fail();
    return SK_OK;
}

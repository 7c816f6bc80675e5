// sk_kernels.h - launch interface between the C ABI (sk_api.cu) and the kernels
// (sk_kernels.cu).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "sk_schedule.h"

namespace sk {

constexpr int kStages = 6;                           // TMA -> shared-memory ring depth
constexpr int kABytes = kTileM * kBlkK * 2;          // 16 KiB: A slab 128 x 64 BF16
constexpr int kBBytes = kTileN * kBlkK * 2;          // 16 KiB: B slab 64 x 128 BF16
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kThreads = 192;                        // warp 0 TMA, warp 1 MMA, warps 2-5 epilogue
constexpr int kEpiThreads = 128;
constexpr int kTmemCols = 256;                       // two 128 x 128 FP32 accumulators
constexpr int kSlotFloats = kTileM * kTileN;         // one FP32 partial tile = 64 KiB
constexpr int kSmemBarOff = kStages * kStageBytes;   // barriers after the ring
constexpr int kSmemBytes = kSmemBarOff + 256 + 1024; // + barrier block + 1 KiB alignment slack

struct KArgs {
    Sched sch;
    void* C;            // [M,N] FP32 or BF16
    float* slabs;       // split-partials: [splits][M][N] FP32
    float* slots;       // n_slots x 64 KiB partial tiles
    int32_t* flags;     // n_slots flags (deterministic) or counters (atomic)
    int32_t* status;    // workspace status word
    float* dump;        // optional: every segment's own FP32 accumulator, by (tile*iters + k_begin)
    uint64_t timeout_ns;
    int32_t M, N, K;
    int32_t c_bf16;
    int32_t atomic;
    int32_t reverse;    // run unit gridDim.x-1-blockIdx.x on CTA blockIdx.x
    int32_t skip_signal;// producers store but never raise their flag (time-out test)
};

// Launch the persistent GEMM (cooperative, `a.sch.workers` CTAs). Returns a cudaError_t.
cudaError_t launch_gemm(const CUtensorMap& tmA, const CUtensorMap& tmB, bool nt, const KArgs& a,
                        cudaStream_t stream);
// Configure the kernels' shared-memory limit on the current device and report how many
// GEMM CTAs fit on one SM.
cudaError_t prepare_device(int* gemm_ctas_per_sm);
// C = sum_j P[j] in j order, FP32 -> c_bf16 ? BF16 : FP32. mn % 4 == 0.
cudaError_t launch_reduce(const float* P, void* C, int c_bf16, int splits, int64_t mn, int num_sms,
                          cudaStream_t stream);

}  // namespace sk

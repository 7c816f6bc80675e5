// sk_kernels.h - launch interface between the C ABI (sk_api.cu) and the kernels
// (sk_kernels.cu).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "sk_schedule.h"

namespace sk {

#ifndef SK_EPI_GROUPS
#define SK_EPI_GROUPS 1
#endif
// Epilogue groups of four warps, one warp per TMEM lane quadrant. With two groups, group g
// takes the segments whose accumulator is buffer g, so a segment's stores or fixup never
// queue behind the previous segment's; with one, the group takes every segment in turn.
constexpr int kEpiGroups = SK_EPI_GROUPS;
static_assert(kEpiGroups == 1 || kEpiGroups == 2, "one or two epilogue groups");
constexpr int kEpiWarps = 4 * kEpiGroups;
constexpr int kThreads = 64 + 32 * kEpiWarps;   // warp 0 TMA, warp 1 MMA, then the epilogue warps
constexpr int kEpiThreads = 32 * kEpiWarps;
constexpr int kGroupThreads = 128;
constexpr int kPassCols = kEpiGroups == 1 ? 128 : 64;  // accumulator columns a thread holds at once
constexpr int kBoxes = 2 / kEpiGroups;          // 4 KiB staging boxes per epilogue warp
constexpr int kCtaRows = 128;     // rows of a work tile held by one CTA (its TMEM lanes)
constexpr int kRingBytes = 196608;
constexpr int kTraceSegs = 15;                  // SK_TRACE_SEGS
constexpr int kTileShapes = 4;                  // sk_tile values

// Layout of the barrier block at the end of shared memory (byte offsets within it): the
// pipeline mbarriers from 0 (full and empty per ring stage, tfull and tempty per accumulator,
// done, tready: at most 8 * (2 * 8 + 6) = 176 bytes), then single words, then two
// partial-load mbarriers per epilogue warp.
constexpr int kBarTmemHolder = 192;  // u32: TMEM base address written by the allocator
constexpr int kBarAbort = 196;       // int: this CTA gave up (a wait ran out or a check failed)
constexpr int kBarLastFlag = 200;    // int per epilogue group: this group took a tile's last slab
constexpr int kBarPrefetch = 208;    // int: hand-off word of the producer warp's partial copies
constexpr int kBarSharedTmp = 212;   // int: a group's shared copy of an atomic result
constexpr int kBarPload = 256;       // two mbarriers per epilogue warp
constexpr int kBarBlockBytes = 512;
static_assert(8 * (2 * 8 + 6) <= kBarTmemHolder && kBarLastFlag + 4 * 2 <= kBarPrefetch &&
                  kBarSharedTmp + 4 <= kBarPload && kBarPload + 16 * kEpiWarps <= kBarBlockBytes,
              "barrier block layout");
constexpr int kTraceWords = 4 + 4 * kTraceSegs; // SK_TRACE_WORDS

// Compile-time shape of one kernel instance: kCG CTAs per work tile (1, or a pair with
// tcgen05 cta_group::2), work tile (128 * kCG) x kBN, k-iteration depth 64.
template <int kCG, int kBN>
struct Shape {
    static constexpr int kCtas = kCG;                      // CTAs per work tile
    static constexpr int kBNc = kBN / kCG;                 // B columns held by one CTA
    static constexpr int kABytes = kCtaRows * kBlkK * 2;   // 16 KiB of A per stage
    static constexpr int kBBytes = kBNc * kBlkK * 2;       // 8 / 16 / 32 KiB of B per stage
    static constexpr int kStageBytes = kABytes + kBBytes;
    static constexpr int kStages = (kRingBytes / kStageBytes) > 8 ? 8 : (kRingBytes / kStageBytes);
    // Epilogue staging after the ring: per epilogue warp kBoxes 4 KiB boxes (32 rows x 128 B)
    // that the TMA stores to C; then the barrier block and 1 KiB of alignment.
    static constexpr int kStagingOff = kStages * kStageBytes;
    static constexpr int kStagingBytes = kEpiWarps * kBoxes * 4096;
    static constexpr int kSmemBarOff = kStagingOff + kStagingBytes;
    static constexpr int kSmemBytes = kSmemBarOff + kBarBlockBytes + 1024;
    static constexpr int kTmemCols = 2 * kBN;               // two accumulators of kBN columns
    static constexpr int kTxBytes = kCG * kStageBytes;      // bytes landing on the leader per stage
    static constexpr int kPasses = kBN / kPassCols;         // a thread's row, kPassCols at a time
    static constexpr int kWarpSlotFloats = 32 * kBN;        // one epilogue warp's block of a partial
    static constexpr int kCtaSlotFloats = kCtaRows * kBN;   // a CTA's share of one partial slot
    static_assert(kBNc % 64 == 0 && kBN % 128 == 0, "tile shape");
    static_assert(kSmemBytes <= 232448 && kStages <= 8, "shared memory");
    // The unit's last epilogue reuses the idle ring in four quarters of kRingBytes / 4 (its
    // staging buffers, an owner's partial copies, the shared slab sum): the stages must fill
    // exactly kRingBytes, or the quarters would reach the staging boxes and the barriers.
    static_assert(kStages * kStageBytes == kRingBytes, "ring quarters");
};

struct KArgs {
    Sched sch;
    void* C;            // [M,N] FP32 or BF16
    float* slabs;       // split-partials: [splits][M][N] FP32
    int32_t* counters;  // split-partials: arrivals per tile and CTA of the tile
    float* slots;       // n_slots x tile_m x tile_n FP32 partial tiles
    int32_t* flags;     // n_slots x CTAs-per-tile flags (deterministic) or counters (atomic)
    int32_t* status;    // workspace status word
    float* dump;        // optional: every segment's own FP32 accumulator, by (tile*iters + k_begin)
    uint64_t* trace;    // optional: per-CTA %globaltimer record (kTraceWords each)
    uint64_t timeout_ns;
    int32_t M, N, K;
    int32_t c_bf16;
    int32_t atomic;
    int32_t reverse;    // unit order reversed over the CTAs (or CTA pairs)
    int32_t skip_signal;// producers store but never raise their flag, and slab splits that share
                        // the sum never count their arrival (time-out tests)
    int32_t zero_partials;  // every partial and slab is stored as zeros, signalled as usual
                            // (numerical control of the tests)
};

// Launch the persistent GEMM for a.sch's tile shape: a.sch.workers units of a.sch.cg CTAs,
// cooperative where the device allows it, or overlapped with the kernel before it on the
// stream (programmatic stream serialization) when a.sch.overlap. Returns a cudaError_t.
// tmC: where segments store — C [M,N] (FP32 or BF16) in boxes of 32 rows x 128 bytes, or
// for Split-K slabs the FP32 [splits][M][N] map in boxes of 1 x 32 rows x 32 columns.
// tmD: the C map (the last split of a tile writes the sum of the slabs there).
cudaError_t launch_gemm(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmC,
                        const CUtensorMap& tmD, bool nt, const KArgs& a, cudaStream_t stream);
// Configure the kernels' shared-memory limit on the current device and report, per
// sk_tile value (kTileShapes of them), how many units of that shape can be resident at once.
cudaError_t prepare_device(int num_sms, int* max_units);
// Separate fixup pass for a plan with sch.sep: every Stream-K tile covered by more than one
// unit gets C = its partial slots summed in k order (FP32), stored as BF16 or FP32.
// Overlapped with the GEMM before it (programmatic stream serialization) when sch.overlap;
// `free_sms`: the device's SMs that GEMM leaves idle (with overlap = 2 the pass may run on
// those alone, so that the next GEMM starts beside it).
cudaError_t launch_fixup(const Sched& sch, const float* slots, void* C, int32_t M, int32_t N, int c_bf16, int num_sms,
                         int free_sms, cudaStream_t stream);
// Host side: the parts of a workspace that must hold zeros before a launch (the status word,
// the flags or arrival counters, and with atomic reduction the partial tiles the peers add
// into), as up to two byte ranges [off[i], off[i] + len[i]); unused ranges have len 0. The
// same layout rule as sk_workspace_size. Returns SK_OK or the sk_plan error code.
int32_t workspace_zero_spans(int32_t M, int32_t N, int32_t K, int32_t num_sms, const void* sched, int32_t reduction,
                             int64_t (&off)[2], int64_t (&len)[2]);
// Host side: every check sk_gemm makes before it enqueues anything (arguments, schedule,
// workspace size and alignment, residency), with `sched` pointing at an sk_schedule. SK_OK
// when sk_gemm with the same arguments would enqueue its work, else its error code.
int32_t gemm_check(const void* A, const void* B, const void* C, int32_t c_dtype, int32_t M, int32_t N, int32_t K,
                   int32_t layout, const void* sched, int32_t reduction, int32_t num_sms, const void* workspace,
                   size_t ws_bytes);
// C = sum_j P[j] in j order, FP32 -> c_bf16 ? BF16 : FP32. mn % 4 == 0. `overlap` (the
// GEMM's sch.overlap) and `free_sms`: as for launch_fixup.
cudaError_t launch_reduce(const float* P, void* C, int c_bf16, int splits, int64_t mn, int num_sms, int overlap,
                          int free_sms, cudaStream_t stream);

}  // namespace sk

// sk_kernels.cu - the persistent work-decomposed BF16 GEMM for sm_103a and the Split-K
// slab reduction.
//
// One CTA per persistent unit ("Split-K and Stream-K: The Last Wave of a GEMM",
// Mental model: one persistent CTA per SM, each walking its share of the flattened
// tile-by-k space). Each CTA walks its segments (sk_schedule.h) with three roles:
//   warp 0      TMA producer: streams the A and B slabs of every k-iteration of every
//               segment into a kStages-deep shared-memory ring;
//   warp 1      MMA issuer: one thread issues tcgen05.mma (128 x 128 x 16, BF16 -> FP32)
//               into one of two TMEM accumulators, alternating per segment, so the
//               epilogue of one segment overlaps the MAC loop of the next;
//   warps 2..5  epilogue: read the accumulator from TMEM and act on the segment's role:
//               FULL -> write C; PRODUCER -> store the FP32 partial to its workspace slot
//               and raise a flag (or add it atomically and bump a counter); OWNER -> wait
//               for its peers in k order, add their partials, write C (Mental model;
//               Case 4 reduction modes); SLAB -> write the split's FP32 [M,N] slab.
// Every wait is bounded by a deadline; on expiry the CTA records SK_ETIMEOUT in the
// workspace status word, unwinds its pipeline and returns.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "sk_kernels.h"
#include "sk_ptx.cuh"

namespace sk {

namespace {

constexpr int32_t kErrTimeout = -4;  // SK_ETIMEOUT
constexpr uint64_t kDrainNs = 20ull * 1000 * 1000;

struct Smem {
    uint32_t base;  // shared address of the 1024-aligned ring
    __device__ uint32_t a(int s) const { return base + s * kABytes; }
    __device__ uint32_t b(int s) const { return base + kStages * kABytes + s * kBBytes; }
    __device__ uint32_t full(int s) const { return base + kSmemBarOff + 8 * s; }
    __device__ uint32_t empty(int s) const { return base + kSmemBarOff + 8 * (kStages + s); }
    __device__ uint32_t tfull(int b) const { return base + kSmemBarOff + 8 * (2 * kStages + b); }
    __device__ uint32_t tempty(int b) const { return base + kSmemBarOff + 8 * (2 * kStages + 2 + b); }
    __device__ uint32_t done() const { return base + kSmemBarOff + 8 * (2 * kStages + 4); }
};

__device__ __forceinline__ void record_timeout(const KArgs& a, volatile int* abort_flag) {
    *abort_flag = 1;
    atomicCAS(a.status, 0, kErrTimeout);
}

// --------------------------------------------------------------------------- warp 0
template <bool kNT>
__device__ void run_producer(const KArgs& a, const CUtensorMap* tmA, const CUtensorMap* tmB, const Smem& sm,
                             int unit, uint64_t deadline, volatile int* abort_flag) {
    Walk w;
    w.init(a.sch, unit);
    Seg g;
    int stage = 0;
    uint32_t phase = 0;
    uint32_t issued = 0;
    bool ok = true;
    while (ok && w.next(a.sch, g)) {
        const int32_t m0 = (g.tile / a.sch.tiles_n) * kTileM;
        const int32_t n0 = (g.tile % a.sch.tiles_n) * kTileN;
        for (int32_t k = g.k_begin; k < g.k_end; ++k) {
            if (!mbar_wait(sm.empty(stage), phase ^ 1u, abort_flag, deadline)) {
                ok = false;
                break;
            }
            const int32_t k0 = k * kBlkK;
            mbar_arrive_expect_tx(sm.full(stage), kStageBytes);
            tma_load_2d(sm.a(stage), tmA, sm.full(stage), k0, m0);
            if (kNT) {
                tma_load_2d(sm.b(stage), tmB, sm.full(stage), k0, n0);
            } else {
                // B [K,N]: two 64-column boxes (128-byte swizzle spans 64 BF16 columns).
                tma_load_2d(sm.b(stage), tmB, sm.full(stage), n0, k0);
                tma_load_2d(sm.b(stage) + kBBytes / 2, tmB, sm.full(stage), n0 + 64, k0);
            }
            ++issued;
            if (++stage == kStages) {
                stage = 0;
                phase ^= 1u;
            }
        }
    }
    if (!ok) record_timeout(a, abort_flag);
    // Let the last loads land before the CTA can exit (they complete quickly; bounded).
    const uint64_t drain = globaltimer() + kDrainNs;
    const uint32_t outstanding = issued < static_cast<uint32_t>(kStages) ? issued : kStages;
    for (uint32_t i = 0; i < outstanding; ++i) {
        const uint32_t pos = issued - 1 - i;
        if (!mbar_wait_until(sm.full(pos % kStages), (pos / kStages) & 1u, drain)) break;
    }
}

// --------------------------------------------------------------------------- warp 1
template <bool kNT>
__device__ void run_mma(const KArgs& a, const Smem& sm, uint32_t tmem_base, int unit, uint64_t deadline,
                        volatile int* abort_flag) {
    constexpr uint32_t kIdesc = idesc_bf16_f32(kTileM, kTileN, kNT ? 0u : 1u);
    // K advance per 16-deep MMA inside one 64-deep stage: K-major operands move 32 bytes
    // along the swizzled row; the MN-major B of NN moves 16 rows of 128 bytes.
    constexpr uint32_t kAStep = (16 * 2) >> 4;
    constexpr uint32_t kBStep = kNT ? ((16 * 2) >> 4) : ((16 * 128) >> 4);
    Walk w;
    w.init(a.sch, unit);
    Seg g;
    int stage = 0;
    uint32_t phase = 0;
    int buf = 0;
    uint32_t uses[2] = {0u, 0u};
    bool ok = true;
    while (ok && w.next(a.sch, g)) {
        if (!mbar_wait(sm.tempty(buf), uses[buf] ^ 1u, abort_flag, deadline)) {
            ok = false;
            break;
        }
        tc_fence_after();
        const uint32_t d = tmem_base + static_cast<uint32_t>(buf * kTileN);
        for (int32_t k = g.k_begin; k < g.k_end; ++k) {
            if (!mbar_wait(sm.full(stage), phase, abort_flag, deadline)) {
                ok = false;
                break;
            }
            tc_fence_after();
            // A: K-major, 8-row groups 1024 bytes apart. B: K-major likewise (NT), or
            // MN-major (NN) with its two 64-column halves 8 KiB apart.
            const uint64_t adesc = smem_desc_sw128(sm.a(stage), 16, 1024);
            const uint64_t bdesc = kNT ? smem_desc_sw128(sm.b(stage), 16, 1024)
                                       : smem_desc_sw128(sm.b(stage), kBBytes / 2, 1024);
#pragma unroll
            for (int kk = 0; kk < kBlkK / 16; ++kk) {
                umma_bf16(d, adesc + kk * kAStep, bdesc + kk * kBStep, kIdesc,
                          (k > g.k_begin || kk > 0) ? 1u : 0u);
            }
            umma_commit(sm.empty(stage));
            if (++stage == kStages) {
                stage = 0;
                phase ^= 1u;
            }
        }
        if (!ok) break;
        umma_commit(sm.tfull(buf));
        uses[buf] ^= 1u;
        buf ^= 1;
    }
    if (!ok) record_timeout(a, abort_flag);
    // Every MMA issued so far has finished reading shared memory and writing TMEM
    // before this thread moves on to the exit barrier.
    umma_commit(sm.done());
    mbar_wait_until(sm.done(), 0u, globaltimer() + kDrainNs);
}

// --------------------------------------------------------------------------- warps 2..5
// Wait until *f >= target: lane 0 polls, then every lane performs its own acquire load.
__device__ __forceinline__ bool wait_flag(const int32_t* f, int32_t target, uint64_t deadline,
                                          const volatile int* abort_flag) {
    bool ok = true;
    if ((threadIdx.x & 31) == 0) {
        for (uint32_t n = 0;; ++n) {
            if (ld_acquire_gpu(f) >= target) break;
            if ((n & 15u) == 15u && (*abort_flag || globaltimer() > deadline)) {
                ok = false;
                break;
            }
            __nanosleep(32);
        }
    }
    // The warp's decision is lane 0's; each lane then takes its own acquire of the flag
    // (a bounded re-read that cannot change the decision).
    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    if (ok) {
        for (uint32_t n = 0; n < (1u << 20) && ld_acquire_gpu(f) < target; ++n) {
        }
    }
    return ok;
}

// Partial-slot layout: element (row r, column 4q + e of chunk c) at float4 index
// (c * 8 + q) * 128 + r, so a warp's 32 rows touch 512 contiguous bytes per access.
__device__ __forceinline__ int slot_f4(int c, int q, int row) { return ((c * 8 + q) * kTileM + row) * 4; }

__device__ __forceinline__ void store_row_chunk(const KArgs& a, const float (&v)[128], int32_t gr, int32_t n0) {
    if (gr >= a.M) return;
    if (a.c_bf16) {
        __nv_bfloat16* crow = static_cast<__nv_bfloat16*>(a.C) + static_cast<int64_t>(gr) * a.N;
#pragma unroll
        for (int g8 = 0; g8 < 16; ++g8) {
            const int32_t gc = n0 + g8 * 8;
            if (gc < a.N) {
                __nv_bfloat162 p0 = __floats2bfloat162_rn(v[g8 * 8 + 0], v[g8 * 8 + 1]);
                __nv_bfloat162 p1 = __floats2bfloat162_rn(v[g8 * 8 + 2], v[g8 * 8 + 3]);
                __nv_bfloat162 p2 = __floats2bfloat162_rn(v[g8 * 8 + 4], v[g8 * 8 + 5]);
                __nv_bfloat162 p3 = __floats2bfloat162_rn(v[g8 * 8 + 6], v[g8 * 8 + 7]);
                uint4 pk;
                pk.x = *reinterpret_cast<uint32_t*>(&p0);
                pk.y = *reinterpret_cast<uint32_t*>(&p1);
                pk.z = *reinterpret_cast<uint32_t*>(&p2);
                pk.w = *reinterpret_cast<uint32_t*>(&p3);
                *reinterpret_cast<uint4*>(crow + gc) = pk;
            }
        }
    } else {
        float* crow = static_cast<float*>(a.C) + static_cast<int64_t>(gr) * a.N;
#pragma unroll
        for (int g8 = 0; g8 < 16; ++g8) {
            const int32_t gc = n0 + g8 * 8;
            if (gc < a.N) {
                *reinterpret_cast<float4*>(crow + gc) =
                    make_float4(v[g8 * 8 + 0], v[g8 * 8 + 1], v[g8 * 8 + 2], v[g8 * 8 + 3]);
                *reinterpret_cast<float4*>(crow + gc + 4) =
                    make_float4(v[g8 * 8 + 4], v[g8 * 8 + 5], v[g8 * 8 + 6], v[g8 * 8 + 7]);
            }
        }
    }
}

__device__ __forceinline__ void store_slab(const KArgs& a, const float (&v)[128], int32_t slab, int32_t gr,
                                           int32_t n0) {
    if (gr >= a.M) return;
    float* row = a.slabs + static_cast<int64_t>(slab) * a.M * a.N + static_cast<int64_t>(gr) * a.N;
#pragma unroll
    for (int g8 = 0; g8 < 16; ++g8) {
        const int32_t gc = n0 + g8 * 8;
        if (gc < a.N) {
            *reinterpret_cast<float4*>(row + gc) =
                make_float4(v[g8 * 8 + 0], v[g8 * 8 + 1], v[g8 * 8 + 2], v[g8 * 8 + 3]);
            *reinterpret_cast<float4*>(row + gc + 4) =
                make_float4(v[g8 * 8 + 4], v[g8 * 8 + 5], v[g8 * 8 + 6], v[g8 * 8 + 7]);
        }
    }
}

__device__ void run_epilogue(const KArgs& a, const Smem& sm, uint32_t tmem_base, int unit, uint64_t deadline,
                             volatile int* abort_flag) {
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int et = threadIdx.x - 64;          // 0..127 among the epilogue threads
    const int quad = warp & 3;                // TMEM lanes this warp may read: 32*quad ..
    const int row = quad * 32 + lane;         // tile row owned by this thread
    const uint32_t lane_addr = static_cast<uint32_t>(quad * 32) << 16;
    Walk w;
    w.init(a.sch, unit);
    Seg g;
    int buf = 0;
    uint32_t uses[2] = {0u, 0u};
    while (w.next(a.sch, g)) {
        const bool got = mbar_wait(sm.tfull(buf), uses[buf], abort_flag, deadline);
        if (named_bar_or(1, kEpiThreads, !got || *abort_flag != 0)) {
            if (!got) record_timeout(a, abort_flag);
            break;
        }
        tc_fence_after();
        float v[128];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            uint32_t r[32];
            tmem_ld_32x32b_x32_sync(tmem_base + lane_addr + static_cast<uint32_t>(buf * kTileN + c * 32), r);
#pragma unroll
            for (int i = 0; i < 32; ++i) v[c * 32 + i] = __uint_as_float(r[i]);
        }
        tc_fence_before();
        mbar_arrive(sm.tempty(buf));
        uses[buf] ^= 1u;
        buf ^= 1;

        const int32_t m0 = (g.tile / a.sch.tiles_n) * kTileM;
        const int32_t n0 = (g.tile % a.sch.tiles_n) * kTileN;
        const int32_t gr = m0 + row;

        if (a.dump) {
            float* d = a.dump + (static_cast<int64_t>(g.tile) * a.sch.iters + g.k_begin) * kSlotFloats +
                       row * kTileN;
#pragma unroll
            for (int q = 0; q < 32; ++q)
                *reinterpret_cast<float4*>(d + 4 * q) = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
        }

        if (g.role == kProducer) {
            if (a.atomic) {
                float* s = a.slots + static_cast<int64_t>(g.peer_begin) * kSlotFloats;
#pragma unroll
                for (int c = 0; c < 4; ++c)
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        const int i = c * 32 + q * 4;
                        red_add_v4_f32(s + slot_f4(c, q, row), v[i], v[i + 1], v[i + 2], v[i + 3]);
                    }
            } else {
                float* s = a.slots + static_cast<int64_t>(g.slot) * kSlotFloats;
#pragma unroll
                for (int c = 0; c < 4; ++c)
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        const int i = c * 32 + q * 4;
                        st_cg_f4(s + slot_f4(c, q, row), make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]));
                    }
            }
            __threadfence();
            named_bar_sync(1, kEpiThreads);
            if (et == 0 && !a.skip_signal) {
                if (a.atomic)
                    red_release_add_gpu(a.flags + g.peer_begin, 1);
                else
                    st_release_gpu(a.flags + g.slot, 1);
            }
        } else if (g.role == kOwner) {
            // Turnstile: fold the peers' partials into this unit's own in k order.
            bool ok = true;
            if (a.atomic) {
                ok = wait_flag(a.flags + g.peer_begin, g.n_peers, deadline, abort_flag);
                if (ok) {
                    float* s = a.slots + static_cast<int64_t>(g.peer_begin) * kSlotFloats;
                    const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                    for (int c = 0; c < 4; ++c)
#pragma unroll
                        for (int q = 0; q < 8; ++q) {
                            const int i = c * 32 + q * 4;
                            const float4 p = ld_cg_f4(s + slot_f4(c, q, row));
                            v[i] += p.x;
                            v[i + 1] += p.y;
                            v[i + 2] += p.z;
                            v[i + 3] += p.w;
                            st_cg_f4(s + slot_f4(c, q, row), z);
                        }
                }
            } else {
                for (int32_t pi = 0; pi < g.n_peers && ok; ++pi) {
                    const int32_t slot = g.peer_begin + pi;
                    ok = wait_flag(a.flags + slot, 1, deadline, abort_flag);
                    if (!ok) break;
                    const float* s = a.slots + static_cast<int64_t>(slot) * kSlotFloats;
#pragma unroll
                    for (int c = 0; c < 4; ++c)
#pragma unroll
                        for (int q = 0; q < 8; ++q) {
                            const int i = c * 32 + q * 4;
                            const float4 p = ld_cg_f4(s + slot_f4(c, q, row));
                            v[i] += p.x;
                            v[i + 1] += p.y;
                            v[i + 2] += p.z;
                            v[i + 3] += p.w;
                        }
                }
            }
            if (named_bar_or(1, kEpiThreads, !ok)) {
                record_timeout(a, abort_flag);
                break;
            }
            // Every epilogue thread has read the partials: re-arm the flags / counter.
            if (et == 0) {
                if (a.atomic) {
                    a.flags[g.peer_begin] = 0;
                } else {
                    for (int32_t pi = 0; pi < g.n_peers; ++pi) a.flags[g.peer_begin + pi] = 0;
                }
            }
            store_row_chunk(a, v, gr, n0);
        } else if (g.role == kSlab) {
            store_slab(a, v, g.slot, gr, n0);
        } else {
            store_row_chunk(a, v, gr, n0);
        }
    }
}

// --------------------------------------------------------------------------- kernel
template <bool kNT>
__global__ void __launch_bounds__(kThreads, 1)
    sk_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const KArgs args) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Smem sm{smem_u32(smem)};
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + kSmemBarOff + 192);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kSmemBarOff + 196);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int unit = args.reverse ? static_cast<int>(gridDim.x) - 1 - static_cast<int>(blockIdx.x)
                                  : static_cast<int>(blockIdx.x);
    const uint64_t deadline = globaltimer() + args.timeout_ns;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(sm.full(s), 1);
            mbar_init(sm.empty(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(sm.tfull(b), 1);
            mbar_init(sm.tempty(b), kEpiThreads);
        }
        mbar_init(sm.done(), 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tmA);
        prefetch_tmap(&tmB);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_holder), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(tmem_holder);

    if (warp == 0) {
        if (lane == 0) run_producer<kNT>(args, &tmA, &tmB, sm, unit, deadline, abort_flag);
    } else if (warp == 1) {
        if (lane == 0) run_mma<kNT>(args, sm, tmem_base, unit, deadline, abort_flag);
    } else {
        run_epilogue(args, sm, tmem_base, unit, deadline, abort_flag);
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem_base, kTmemCols);
    }
}

// --------------------------------------------------------------------------- reduce
__global__ void __launch_bounds__(256)
    sk_reduce_kernel(const float* __restrict__ P, void* __restrict__ C, int c_bf16, int splits, int64_t n4) {
    const float4* P4 = reinterpret_cast<const float4*>(P);
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n4; i += stride) {
        float4 acc = __ldcs(P4 + i);
        for (int j = 1; j < splits; ++j) {
            const float4 x = __ldcs(P4 + static_cast<int64_t>(j) * n4 + i);
            acc.x += x.x;
            acc.y += x.y;
            acc.z += x.z;
            acc.w += x.w;
        }
        if (c_bf16) {
            __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
            __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
            uint2 pk;
            pk.x = *reinterpret_cast<uint32_t*>(&lo);
            pk.y = *reinterpret_cast<uint32_t*>(&hi);
            reinterpret_cast<uint2*>(C)[i] = pk;
        } else {
            reinterpret_cast<float4*>(C)[i] = acc;
        }
    }
}

}  // namespace

cudaError_t prepare_device(int* gemm_ctas_per_sm) {
    cudaError_t e = cudaFuncSetAttribute(sk_gemm_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kSmemBytes);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(sk_gemm_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    int n0 = 0, n1 = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n0, sk_gemm_kernel<false>, kThreads, kSmemBytes);
    if (e != cudaSuccess) return e;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n1, sk_gemm_kernel<true>, kThreads, kSmemBytes);
    if (e != cudaSuccess) return e;
    *gemm_ctas_per_sm = n0 < n1 ? n0 : n1;
    return cudaSuccess;
}

cudaError_t launch_gemm(const CUtensorMap& tmA, const CUtensorMap& tmB, bool nt, const KArgs& a,
                        cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(a.sch.workers), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (nt) return cudaLaunchKernelEx(&cfg, sk_gemm_kernel<true>, tmA, tmB, a);
    return cudaLaunchKernelEx(&cfg, sk_gemm_kernel<false>, tmA, tmB, a);
}

cudaError_t launch_reduce(const float* P, void* C, int c_bf16, int splits, int64_t mn, int num_sms,
                          cudaStream_t stream) {
    const int64_t n4 = mn / 4;
    int64_t blocks = (n4 + 255) / 256;
    const int64_t cap = static_cast<int64_t>(num_sms) * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    sk_reduce_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(P, C, c_bf16, splits, n4);
    return cudaGetLastError();
}

}  // namespace sk

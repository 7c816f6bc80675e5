// sk_passes.cu - the second launches that sum FP32 partials into C: the Split-K slab
// reduction and the separate fixup pass for Stream-K tiles. Both sum in k order, left to
// right in FP32, and convert to the output type once.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "sk_kernels.h"
#include "sk_ptx.cuh"

namespace sk {
namespace {

// Both passes are bound by how many loads are in flight: each thread keeps up to 16 float4
// loads outstanding, within 128 registers, so four blocks of kPassThreads fit on an SM and a
// grid of up to four blocks per SM runs in one wave (every load goes out in the first round
// trip for the shapes whose partials fit in that). One block also fits beside a resident GEMM
// CTA (255 registers x 192 threads), so part of an overlapped pass is resident early.
constexpr int kPassThreads = 128;
constexpr int kPassBlocksPerSm = 4;
// Behind a GEMM launched with overlap = 2 that leaves at least kMinFreeSms SMs idle, a pass
// runs on those SMs alone: each block holds kPassHoldSmem bytes of shared memory, so it cannot
// sit beside a GEMM CTA (which takes nearly all of an SM's), the grid fits on the idle SMs at
// once, and the blocks let the next kernel launch before they wait for the GEMM. The next
// GEMM's CTAs then take the SMs this GEMM leaves and run their first segments (overlap = 2)
// while the pass sums; their stores still wait for the pass to complete.
// The idle SMs take the pass only while it is small: at most kMaxPinnedRounds grid-stride
// rounds of their blocks (a large reduction, say 8192 x 8192 in two slabs, runs on every SM).
constexpr int kMinFreeSms = 8;
constexpr int kMaxPinnedRounds = 8;
constexpr int kPassHoldSmem = 8192;

// --------------------------------------------------------------------------- Split-K slab reduction
__global__ void __launch_bounds__(kPassThreads, kPassBlocksPerSm)
    sk_reduce_kernel(const float* __restrict__ P, void* __restrict__ C, int c_bf16, int splits, int64_t n4,
                     int early) {
    // An overlapped launch reads P only once the GEMM that wrote it is done. `early`: the
    // next kernel may launch first (see kMinFreeSms).
    if (early) {
        grid_dep_launch();
        grid_dep_wait();
    } else {
        grid_dep_wait();
        grid_dep_launch();
    }
    const float4* P4 = reinterpret_cast<const float4*>(P);
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    // An element's loads from kBatch slabs go out together (one round trip to L2 per batch
    // instead of one per slab); the adds stay a left fold in split order.
    constexpr int kBatch = 16;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n4; i += stride) {
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int j0 = 0; j0 < splits; j0 += kBatch) {
            float4 x[kBatch];
            const float4* q = P4 + static_cast<int64_t>(j0) * n4 + i;
#pragma unroll
            for (int jj = 0; jj < kBatch; ++jj, q += n4)
                if (j0 + jj < splits) x[jj] = __ldcs(q);
#pragma unroll
            for (int jj = 0; jj < kBatch; ++jj) {
                if (j0 + jj >= splits) break;
                if (j0 + jj == 0) {
                    acc = x[jj];
                } else {
                    acc.x += x[jj].x;
                    acc.y += x[jj].y;
                    acc.z += x[jj].z;
                    acc.w += x[jj].w;
                }
            }
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

// --------------------------------------------------------------------------- fixup pass
// Separate fixup pass for the Stream-K tiles (first page, Case 3: every partial sits in a
// fixed slot per (unit, first/last segment), and a second kernel sums a split tile's
// partials in k order). Contributor u of local tile t holds slot 2u if t is the tile its
// range starts in, else 2u + 1; contributors u_first .. u_last in unit order are k order,
// and the sum runs left to right in FP32 exactly like the owner's turnstile.
// One warp per (split tile, CTA rank, lane quadrant, 32-column chunk, 8-column group):
// lane l takes row 32 * quad + l of the CTA's 128 rows and columns 32c + 8h .. + 7, which
// in the slot layout are the float4s (8c + 2h) * 32 + l and that + 32 (512 contiguous bytes
// per warp access).
__global__ void __launch_bounds__(kPassThreads, kPassBlocksPerSm)
    sk_fixup_kernel(const Sched sch, const float* __restrict__ slots, void* __restrict__ C, int32_t M, int32_t N,
                    int c_bf16, int early) {
    if (early) {  // as in sk_reduce_kernel
        grid_dep_launch();
        grid_dep_wait();
    } else {
        grid_dep_wait();
        grid_dep_launch();
    }
    const int lane = threadIdx.x & 31;
    const int chunks = sch.tile_n / 32;
    const int64_t per_tile = static_cast<int64_t>(sch.cg) * 4 * chunks * 4;
    const int64_t total = static_cast<int64_t>(sch.sk_tiles) * per_tile;
    const int64_t cta_floats = static_cast<int64_t>(kCtaRows) * sch.tile_n;
    const int64_t warps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    for (int64_t wi = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; wi < total; wi += warps) {
        const int32_t lt = static_cast<int32_t>(wi / per_tile);
        int32_t rem = static_cast<int32_t>(wi % per_tile);
        const int h = rem & 3;
        rem >>= 2;
        const int c = rem % chunks;
        rem /= chunks;
        const int quad = rem & 3;
        const int r = rem >> 2;
        const int32_t tb = lt * sch.iters;
        const int32_t u0 = sk_unit_of(sch, tb);
        const int32_t u1 = sk_unit_of(sch, tb + sch.iters - 1);
        if (u0 == u1) continue;  // the tile was finished inside one unit
        const int64_t f4 = static_cast<int64_t>(((c * 8 + 2 * h) * 32 + lane) * 4);
        const int64_t blk_off = static_cast<int64_t>(quad) * 32 * sch.tile_n + f4;
        float acc[8];
        // Contributors kBatch at a time: the loads go out together, the adds stay in k order.
        constexpr int kBatch = 8;
        for (int32_t u = u0; u <= u1; u += kBatch) {
            float4 x[kBatch][2];
#pragma unroll
            for (int j = 0; j < kBatch; ++j) {
                const int32_t uj = u + j;
                if (uj <= u1) {
                    const int32_t first_tile = sk_unit_begin(sch, uj) / sch.iters;
                    const int32_t slot = 2 * uj + (first_tile == lt ? 0 : 1);
                    const float* p = slots + (static_cast<int64_t>(slot) * sch.cg + r) * cta_floats + blk_off;
                    x[j][0] = __ldcg(reinterpret_cast<const float4*>(p));
                    x[j][1] = __ldcg(reinterpret_cast<const float4*>(p + 128));
                }
            }
#pragma unroll
            for (int j = 0; j < kBatch; ++j) {
                if (u + j > u1) break;
                const float y[8] = {x[j][0].x, x[j][0].y, x[j][0].z, x[j][0].w,
                                    x[j][1].x, x[j][1].y, x[j][1].z, x[j][1].w};
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[e] = (u + j == u0) ? y[e] : acc[e] + y[e];
            }
        }
        int32_t trow, tcolumn;
        tile_coords(sch, sch.sk_base + lt, &trow, &tcolumn);
        const int64_t row = static_cast<int64_t>(trow) * sch.tile_m + r * kCtaRows + quad * 32 + lane;
        const int32_t col = tcolumn * sch.tile_n + c * 32 + 8 * h;
        if (row >= M) continue;
        // N is a multiple of 4 (FP32 C) or 8 (BF16 C), so each 4-column half is all in or out.
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            const int32_t cc = col + 4 * half;
            if (cc >= N) break;
            if (c_bf16) {
                __nv_bfloat162 lo = __floats2bfloat162_rn(acc[4 * half], acc[4 * half + 1]);
                __nv_bfloat162 hi = __floats2bfloat162_rn(acc[4 * half + 2], acc[4 * half + 3]);
                uint2 pk;
                pk.x = *reinterpret_cast<uint32_t*>(&lo);
                pk.y = *reinterpret_cast<uint32_t*>(&hi);
                *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(C) + row * N + cc) = pk;
            } else {
                *reinterpret_cast<float4*>(static_cast<float*>(C) + row * N + cc) =
                    make_float4(acc[4 * half], acc[4 * half + 1], acc[4 * half + 2], acc[4 * half + 3]);
            }
        }
    }
}

// Grid of a pass that wants `want` blocks behind a GEMM launched with `overlap` that leaves
// `free_sms` SMs idle: one wave on every SM, or (overlap = 2, enough idle SMs, a small pass)
// one wave on the idle SMs with the shared-memory hold.
struct PassShape {
    int64_t blocks;
    int smem;
    int early;
};
PassShape pass_shape(int64_t want, int num_sms, int overlap, int free_sms) {
    const bool early = overlap == 2 && free_sms >= kMinFreeSms &&
                       want <= static_cast<int64_t>(kMaxPinnedRounds) * free_sms * kPassBlocksPerSm;
    int64_t cap = static_cast<int64_t>(early ? free_sms : num_sms) * kPassBlocksPerSm;
    int64_t blocks = want < cap ? want : cap;
    if (blocks < 1) blocks = 1;
    return {blocks, early ? kPassHoldSmem : 0, early ? 1 : 0};
}

// A launch of `p.blocks` x kPassThreads threads on `stream`, with programmatic stream
// serialization when `overlap` is set (the kernels above wait for the previous kernel before
// any access).
cudaLaunchConfig_t pass_config(const PassShape& p, cudaStream_t stream, bool overlap, cudaLaunchAttribute* attr) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(p.blocks), 1, 1);
    cfg.blockDim = dim3(kPassThreads, 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(p.smem);
    cfg.stream = stream;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = overlap ? 1 : 0;
    return cfg;
}

}  // namespace

cudaError_t launch_reduce(const float* P, void* C, int c_bf16, int splits, int64_t mn, int num_sms, int overlap,
                          int free_sms, cudaStream_t stream) {
    const int64_t n4 = mn / 4;
    const PassShape p = pass_shape((n4 + kPassThreads - 1) / kPassThreads, num_sms, overlap, free_sms);
    cudaLaunchAttribute attr[1];
    const cudaLaunchConfig_t cfg = pass_config(p, stream, overlap != 0, attr);
    return cudaLaunchKernelEx(&cfg, sk_reduce_kernel, P, C, c_bf16, splits, n4, p.early);
}

cudaError_t launch_fixup(const Sched& sch, const float* slots, void* C, int32_t M, int32_t N, int c_bf16, int num_sms,
                         int free_sms, cudaStream_t stream) {
    const int64_t warps = static_cast<int64_t>(sch.sk_tiles) * sch.cg * 4 * (sch.tile_n / 32) * 4;
    if (warps == 0) return cudaSuccess;
    const PassShape p = pass_shape((warps + kPassThreads / 32 - 1) / (kPassThreads / 32), num_sms, sch.overlap,
                                   free_sms);
    cudaLaunchAttribute attr[1];
    const cudaLaunchConfig_t cfg = pass_config(p, stream, sch.overlap != 0, attr);
    return cudaLaunchKernelEx(&cfg, sk_fixup_kernel, sch, slots, C, M, N, c_bf16, p.early);
}

}  // namespace sk

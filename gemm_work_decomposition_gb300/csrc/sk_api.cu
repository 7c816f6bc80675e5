// sk_api.cu - the C ABI (include/sk.h): planning, validation, tensor-map encoding and
// launch. Host code only; the kernels live in sk_kernels.cu.
#include <algorithm>
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <stdint.h>

#include <climits>
#include <mutex>
#include <vector>

#include "sk.h"
#include "sk_kernels.h"
#include "sk_schedule.h"

using namespace sk;

namespace {

constexpr int64_t kDefaultTimeoutNs = 2000000000ll;
constexpr int kMaxDevices = 64;

// The decision rule of the page "Split-K and Stream-K: The Last Wave of a GEMM", Case 2
// (cutlass_heuristic): stay data-parallel when tiles fill whole waves, the K loop is at
// most min_iters long, or the tail wave is at least half full; otherwise keep all full
// waves but the last data-parallel and give the rest to Stream-K over
// min(sms, iters * sk_tiles / min_iters) units, labelled Split-K when those units divide
// evenly over more than one per tile.
void heuristic(int64_t tiles, int64_t iters, int64_t sms, int64_t min_iters, int32_t* label, int64_t* sk_tiles,
               int64_t* sk_units, int32_t* label_splits) {
    const int64_t whole = tiles / sms;  // full waves
    const int64_t tail = tiles % sms;   // tiles of the last, partial wave
    *label = kLabelDP;
    *sk_tiles = 0;
    *sk_units = 0;
    *label_splits = 0;
    if (tail == 0 || iters <= min_iters || 2 * tail >= sms) return;
    const int64_t skt = tiles - sms * (whole > 1 ? whole - 1 : 0);  // the last two waves
    const int64_t sku = std::min<int64_t>(sms, skt * iters / min_iters);
    *sk_tiles = skt;
    *sk_units = sku;
    if (sku % skt == 0 && sku / skt > 1) {
        *label = kLabelSplitK;
        *label_splits = static_cast<int32_t>(sku / skt);
    } else {
        *label = kLabelStreamK;
    }
}

void set_streamk(Sched& o, int64_t base, int64_t sk_tiles, int64_t units, bool sep, int32_t groups) {
    const int64_t total = sk_tiles * o.iters;
    o.sk_base = static_cast<int32_t>(base);
    o.sk_tiles = static_cast<int32_t>(sk_tiles);
    o.sk_units = static_cast<int32_t>(units);
    o.sk_q = static_cast<int32_t>(total / units);
    o.sk_big = static_cast<int32_t>(total % units);
    o.sk_groups = sk_group_count(o.sk_tiles, o.iters, o.sk_units, groups);
    o.sep = sep ? 1 : 0;
    o.n_slots = static_cast<int32_t>((sep ? 2 : 1) * units);
}

int32_t make_sched_core(int32_t M, int32_t N, int32_t K, int32_t num_sms, const sk_schedule& s, Sched& o);

// The schedule plus the walk's fast divisors (sk_schedule.h FastDiv).
int32_t make_sched(int32_t M, int32_t N, int32_t K, int32_t num_sms, const sk_schedule& s, Sched& o) {
    const int32_t e = make_sched_core(M, N, K, num_sms, s, o);
    if (e != SK_OK) return e;
    const int32_t w = o.swizzle > 1 ? o.swizzle : 1;
    const int32_t along = o.raster == 0 ? o.tiles_n : o.tiles_m;
    if (static_cast<int64_t>(w) * along > INT32_MAX) return SK_EINVAL;
    o.fd_iters = make_fastdiv(static_cast<uint32_t>(o.iters));
    o.fd_q1 = make_fastdiv(static_cast<uint32_t>(o.sk_q) + 1u);
    o.fd_q = make_fastdiv(static_cast<uint32_t>(o.sk_q > 0 ? o.sk_q : 1));
    o.fd_splits = make_fastdiv(static_cast<uint32_t>(o.splits > 0 ? o.splits : 1));
    o.fd_strip = make_fastdiv(static_cast<uint32_t>(w * along));
    o.fd_w = make_fastdiv(static_cast<uint32_t>(w));
    return SK_OK;
}

int32_t make_sched_core(int32_t M, int32_t N, int32_t K, int32_t num_sms, const sk_schedule& s, Sched& o) {
    if (M < 1 || N < 1 || K < 1 || num_sms < 1 || s.units < 0 || s.min_iters < 0) return SK_EINVAL;
    if (s.mode < SK_DP || s.mode > SK_HYBRID) return SK_EINVAL;
    // split_partials: Split-K slabs (1 pass, 2 last arriver), or for Stream-K and the hybrid
    // rule (1) the separate fixup pass; data-parallel tiles have no partials.
    if (s.split_partials < 0 || s.split_partials > 2) return SK_EINVAL;
    if (s.split_partials == 2 && s.mode != SK_SPLITK) return SK_EINVAL;
    if (s.split_partials != 0 && s.mode == SK_DP) return SK_EINVAL;
    int32_t tm = 0, tn = 0, cg = 0;
    if (!tile_shape(s.tile, &tm, &tn, &cg)) return SK_EINVAL;
    if (s.raster < 0 || s.raster > 1 || s.swizzle < 0 || s.swizzle > 256) return SK_EINVAL;
    if (s.overlap < 0 || s.overlap > 2) return SK_EINVAL;
    if (s.sk_groups < 0 || s.sk_groups > 64) return SK_EINVAL;
    const int64_t tiles_n = (static_cast<int64_t>(N) + tn - 1) / tn;
    const int64_t tiles = ((static_cast<int64_t>(M) + tm - 1) / tm) * tiles_n;
    const int64_t iters = (static_cast<int64_t>(K) + kBlkK - 1) / kBlkK;
    if (tiles * iters > INT32_MAX) return SK_EINVAL;
    const int64_t S = s.units > 0 ? s.units : num_sms / cg;
    if (S < 1) return SK_EINVAL;
    const int64_t min_iters = s.min_iters > 0 ? s.min_iters : 8;

    o = Sched{};
    o.tiles = static_cast<int32_t>(tiles);
    o.iters = static_cast<int32_t>(iters);
    o.tiles_n = static_cast<int32_t>(tiles_n);
    o.label = kLabelNone;
    o.tile_m = tm;
    o.tile_n = tn;
    o.cg = cg;
    o.tiles_m = static_cast<int32_t>(tiles / tiles_n);
    o.raster = s.raster;
    o.swizzle = s.swizzle;
    o.overlap = s.overlap;

    int32_t mode = s.mode;
    if (mode == SK_HYBRID) {
        int32_t label, lsp;
        int64_t skt, sku;
        heuristic(tiles, iters, S, min_iters, &label, &skt, &sku, &lsp);
        o.label = label;
        o.label_splits = lsp;
        if (label == kLabelDP) {
            mode = SK_DP;
        } else {
            const int64_t dp_tiles = tiles - skt;
            o.mode = kHybrid;
            set_streamk(o, dp_tiles, skt, sku, s.split_partials == 1, s.sk_groups);
            o.dp_tiles = static_cast<int32_t>(dp_tiles);
            const int64_t dpw = dp_tiles < S ? dp_tiles : S;
            o.workers = static_cast<int32_t>(sku > dpw ? sku : dpw);
            return SK_OK;
        }
    }
    if (mode == SK_DP) {
        o.mode = kDP;
        o.dp_tiles = static_cast<int32_t>(tiles);
        o.workers = static_cast<int32_t>(tiles < S ? tiles : S);
    } else if (mode == SK_STREAMK) {
        const int64_t total = tiles * iters;
        const int64_t U = total < S ? total : S;
        o.mode = kStreamK;
        set_streamk(o, 0, tiles, U, s.split_partials == 1, s.sk_groups);
        o.workers = static_cast<int32_t>(U);
    } else {  // SK_SPLITK
        if (s.splits < 1 || s.splits > iters) return SK_EINVAL;
        const int64_t chunk = (iters + s.splits - 1) / s.splits;
        const int64_t s_eff = (iters + chunk - 1) / chunk;
        const int64_t items = tiles * s_eff;
        if (items > INT32_MAX || tiles * (s_eff - 1) > INT32_MAX) return SK_EINVAL;
        o.mode = kSplitK;
        o.splits = static_cast<int32_t>(s_eff);
        o.chunk = static_cast<int32_t>(chunk);
        o.partials = s.split_partials;
        o.coop = (s.split_partials == 2 && items <= S) ? 1 : 0;
        o.n_slots = s.split_partials ? 0 : static_cast<int32_t>(tiles * (s_eff - 1));
        o.workers = static_cast<int32_t>(items < S ? items : S);
    }
    return SK_OK;
}

int64_t count_segments(const Sched& s) {
    int64_t n = 0;
    for (int32_t w = 0; w < s.workers; ++w) {
        Walk wk;
        wk.init(s, w);
        Seg g;
        while (wk.next(s, g)) ++n;
    }
    return n;
}

int64_t map_size(const Sched& s) {
    return SK_MAP_HEADER + SK_MAP_SEG * count_segments(s) + static_cast<int64_t>(SK_MAP_TILE) * s.tiles;
}

int64_t align_up(int64_t x, int64_t a) { return (x + a - 1) / a * a; }

// Workspace: header | flags (one int32 per slot and CTA of the tile, 256-aligned) |
// slots (tile_m x tile_n FP32 each); split-partials: header | slabs [splits][M][N] FP32 |
// arrival counters (one int32 per tile and CTA of the tile, 256-aligned).
int64_t flags_offset() { return SK_WS_HEADER_BYTES; }
int64_t slots_offset(const Sched& s) { return SK_WS_HEADER_BYTES + align_up(4ll * s.n_slots * s.cg, 256); }
int64_t workspace_bytes(const Sched& s, int32_t M, int32_t N) {
    if (s.partials) return slab_workspace_bytes(s.splits, M, N, s.tiles, s.cg);
    return slots_offset(s) + static_cast<int64_t>(s.n_slots) * s.tile_m * s.tile_n * 4;
}

struct DeviceInfo {
    bool ready = false;
    cudaError_t err = cudaSuccess;
    int sms = 0;
    int max_units[kTileShapes] = {};  // resident units per sk_tile value
};
DeviceInfo g_dev[kMaxDevices];
std::mutex g_mu;

cudaError_t device_info(int* sms, int* max_units) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceInfo& d = g_dev[dev];
    if (!d.ready) {
        d.err = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
        if (d.err == cudaSuccess) d.err = prepare_device(d.sms, d.max_units);
        d.ready = true;
    }
    *sms = d.sms;
    for (int i = 0; i < kTileShapes; ++i) max_units[i] = d.max_units[i];
    return d.err;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// Encoded tensor maps of this host thread's recent calls, keyed by every argument of the
// encoding, so that calls on the same buffers (the usual case: a GEMM called again and again
// on the same operands) skip the driver's encoder. A map is plain host data; a hit returns a
// copy of the bytes the encoder wrote for exactly these arguments.
struct TmapKey {
    const void* ptr;
    uint64_t v[4];
    uint32_t kind;
};
struct TmapEntry {
    TmapKey key;
    CUtensorMap map;
    bool used;
};
constexpr int kTmapCache = 128;
thread_local TmapEntry t_tmaps[kTmapCache];
thread_local int t_tmap_next = 0;

bool same_key(const TmapKey& a, const TmapKey& b) {
    return a.ptr == b.ptr && a.kind == b.kind && a.v[0] == b.v[0] && a.v[1] == b.v[1] && a.v[2] == b.v[2] &&
           a.v[3] == b.v[3];
}
bool tmap_lookup(const TmapKey& k, CUtensorMap* m) {
    for (int i = 0; i < kTmapCache; ++i) {
        if (t_tmaps[i].used && same_key(t_tmaps[i].key, k)) {
            *m = t_tmaps[i].map;
            return true;
        }
    }
    return false;
}
void tmap_store(const TmapKey& k, const CUtensorMap& m) {
    TmapEntry& e = t_tmaps[t_tmap_next];
    t_tmap_next = (t_tmap_next + 1) % kTmapCache;
    e.key = k;
    e.map = m;
    e.used = true;
}

// Row-major BF16 matrix of `outer` rows x `inner` columns, copied in boxes of
// box_outer x box_inner with the 128-byte swizzle; out-of-range elements read as zero.
bool encode_2d(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t outer, uint32_t box_inner,
               uint32_t box_outer) {
    const TmapKey key{ptr, {inner, outer, box_inner, box_outer}, 1u};
    if (tmap_lookup(key, m)) return true;
    PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {inner * 2};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return false;
    tmap_store(key, *m);
    return true;
}

// Output map: rows of `inner` elements of `esize` bytes, `outer` rows per slab and `slabs`
// slabs, stored in boxes of 32 rows x 128 bytes (one box per epilogue warp and store) with
// the 128-byte swizzle the epilogue's staging uses.
bool encode_out(CUtensorMap* m, void* ptr, bool bf16, uint64_t inner, uint64_t outer, uint64_t slabs, uint32_t rank) {
    const TmapKey key{ptr, {inner, outer, slabs, (static_cast<uint64_t>(rank) << 1) | (bf16 ? 1u : 0u)}, 2u};
    if (tmap_lookup(key, m)) return true;
    PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
    if (!fn) return false;
    const uint64_t esize = bf16 ? 2 : 4;
    cuuint64_t dims[3] = {inner, outer, slabs};
    cuuint64_t strides[2] = {inner * esize, inner * outer * esize};
    cuuint32_t box[3] = {static_cast<cuuint32_t>(128 / esize), 32, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, rank,
                    ptr, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return false;
    tmap_store(key, *m);
    return true;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// Every check sk_gemm makes before it enqueues anything: arguments, schedule, workspace and
// residency. On SK_OK with M, N, K > 0, *sch holds the plan and *dev_sms the device's SM count.
int32_t check_gemm(const void* A, const void* B, const void* C, int32_t c_dtype, int32_t M, int32_t N, int32_t K,
                   int32_t layout, const sk_schedule& s, int32_t r, int32_t num_sms, const void* workspace,
                   size_t ws_bytes, Sched* sch, int* dev_sms);

}  // namespace

namespace sk {
int32_t workspace_zero_spans(int32_t M, int32_t N, int32_t K, int32_t num_sms, const void* sched, int32_t reduction,
                             int64_t (&off)[2], int64_t (&len)[2]) {
    Sched s;
    const int32_t e = make_sched(M, N, K, num_sms, *static_cast<const sk_schedule*>(sched), s);
    if (e != SK_OK) return e;
    off[0] = 0;
    off[1] = 0;
    len[1] = 0;
    if (s.partials) {
        // header | slabs (written in full by every launch) | arrival counters
        const int64_t c = slab_counters_offset(s.splits, M, N);
        len[0] = SK_WS_HEADER_BYTES;
        off[1] = c;
        len[1] = workspace_bytes(s, M, N) - c;
    } else {
        // header | flags | slots; atomic peers add into the slots, which start at zero
        len[0] = reduction == SK_ATOMIC ? workspace_bytes(s, M, N) : slots_offset(s);
    }
    return SK_OK;
}
}  // namespace sk

namespace {
int32_t check_gemm(const void* A, const void* B, const void* C, int32_t c_dtype, int32_t M, int32_t N, int32_t K,
                   int32_t layout, const sk_schedule& s, int32_t r, int32_t num_sms, const void* workspace,
                   size_t ws_bytes, Sched* sch, int* dev_sms) {
    if (M < 0 || N < 0 || K < 0 || num_sms < 1) return SK_EINVAL;
    if (c_dtype != SK_F32 && c_dtype != SK_BF16) return SK_EINVAL;
    if (layout != SK_NN && layout != SK_NT) return SK_EINVAL;
    if (r != SK_DETERMINISTIC && r != SK_ATOMIC) return SK_EINVAL;
    if (M == 0 || N == 0) return SK_OK;
    if (!C || !aligned(C, 16) || N % 8 != 0) return SK_EINVAL;
    if (K == 0) return SK_OK;
    if (!A || !B || !aligned(A, 16) || !aligned(B, 16) || K % 8 != 0) return SK_EINVAL;
    const int32_t e = make_sched(M, N, K, num_sms, s, *sch);
    if (e != SK_OK) return e;
    const int64_t need = workspace_bytes(*sch, M, N);
    if (!workspace || !aligned(workspace, 256) || static_cast<int64_t>(ws_bytes) < need) return SK_EWORKSPACE;
    int max_units[kTileShapes];
    if (device_info(dev_sms, max_units) != cudaSuccess) return SK_ECUDA;
    if (sch->workers > max_units[s.tile]) return SK_ERESIDENCY;
    return SK_OK;
}
}  // namespace

namespace sk {
int32_t gemm_check(const void* A, const void* B, const void* C, int32_t c_dtype, int32_t M, int32_t N, int32_t K,
                   int32_t layout, const void* sched, int32_t reduction, int32_t num_sms, const void* workspace,
                   size_t ws_bytes) {
    Sched sch;
    int dev_sms = 0;
    return check_gemm(A, B, C, c_dtype, M, N, K, layout, *static_cast<const sk_schedule*>(sched), reduction, num_sms,
                      workspace, ws_bytes, &sch, &dev_sms);
}
}  // namespace sk

extern "C" {

const char* sk_strerror(int32_t code) {
    switch (code) {
        case SK_OK: return "success";
        case SK_EINVAL: return "invalid argument (sizes, schedule, alignment or layout)";
        case SK_EWORKSPACE: return "workspace missing, misaligned or too small";
        case SK_ECUDA: return "CUDA call failed";
        case SK_ETIMEOUT: return "a device-side wait ran past its time limit";
        case SK_ECAPACITY: return "map buffer smaller than sk_plan_size";
        case SK_ERESIDENCY: return "more persistent units than the device can hold at once";
        case SK_EBOUNDS: return "a device-side index check failed and the access was skipped";
        default: return "unknown error code";
    }
}

int64_t sk_plan_size(int32_t M, int32_t N, int32_t K, int32_t num_sms, sk_schedule s) {
    Sched sch;
    const int32_t e = make_sched(M, N, K, num_sms, s, sch);
    if (e != SK_OK) return e;
    return map_size(sch);
}

int32_t sk_plan(int32_t M, int32_t N, int32_t K, int32_t num_sms, sk_schedule s, int32_t* map, int64_t cap) {
    Sched sch;
    const int32_t e = make_sched(M, N, K, num_sms, s, sch);
    if (e != SK_OK) return e;
    const int64_t need = map_size(sch);
    if (!map || cap < need) return SK_ECAPACITY;
    const int64_t nseg = (need - SK_MAP_HEADER - static_cast<int64_t>(SK_MAP_TILE) * sch.tiles) / SK_MAP_SEG;
    int32_t* h = map;
    h[0] = SK_MAP_VERSION;
    h[1] = sch.mode;
    h[2] = sch.tiles;
    h[3] = sch.iters;
    h[4] = sch.workers;
    h[5] = sch.sk_tiles;
    h[6] = sch.sk_units;
    h[7] = static_cast<int32_t>(nseg);
    h[8] = sch.mode == kSplitK ? sch.splits : 0;
    h[9] = sch.label;
    h[10] = sch.label_splits;
    h[11] = sch.n_slots;
    h[12] = sch.tile_m;
    h[13] = sch.tile_n;
    h[14] = sch.cg;
    h[15] = sch.raster;
    h[16] = sch.swizzle;
    h[17] = sch.sk_groups;
    int32_t* seg = map + SK_MAP_HEADER;
    int32_t* trow = seg + SK_MAP_SEG * nseg;
    for (int32_t t = 0; t < sch.tiles; ++t) {
        trow[SK_MAP_TILE * t] = -1;
        trow[SK_MAP_TILE * t + 1] = 0;
        tile_coords(sch, t, &trow[SK_MAP_TILE * t + 2], &trow[SK_MAP_TILE * t + 3]);
    }
    for (int32_t w = 0; w < sch.workers; ++w) {
        Walk wk;
        wk.init(sch, w);
        Seg g;
        int32_t order = 0;
        while (wk.next(sch, g)) {
            const int32_t row[SK_MAP_SEG] = {w, order++, g.tile, g.k_begin, g.k_end, g.role, g.slot, g.peer_begin,
                                             g.n_peers};
            for (int i = 0; i < SK_MAP_SEG; ++i) seg[i] = row[i];
            seg += SK_MAP_SEG;
            trow[SK_MAP_TILE * g.tile + 1] += 1;
            if (g.k_begin == 0) trow[SK_MAP_TILE * g.tile] = w;
        }
    }
    return SK_OK;
}

int64_t sk_workspace_size(int32_t M, int32_t N, int32_t K, int32_t num_sms, sk_schedule s, sk_reduction r) {
    if (r != SK_DETERMINISTIC && r != SK_ATOMIC) return SK_EINVAL;
    Sched sch;
    const int32_t e = make_sched(M, N, K, num_sms, s, sch);
    if (e != SK_OK) return e;
    return workspace_bytes(sch, M, N);
}

int32_t sk_gemm_debug(const void* A, const void* B, void* C, sk_dtype c_dtype, int32_t M, int32_t N, int32_t K,
                      sk_layout layout, sk_schedule s, sk_reduction r, int32_t num_sms, void* workspace,
                      size_t ws_bytes, void* stream, const sk_debug_opts* opts) {
    Sched sch;
    int dev_sms = 0;
    const int32_t e = check_gemm(A, B, C, c_dtype, M, N, K, layout, s, r, num_sms, workspace, ws_bytes, &sch, &dev_sms);
    if (e != SK_OK || M == 0 || N == 0) return e;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (K == 0) {
        const size_t esz = c_dtype == SK_BF16 ? 2 : 4;
        return cudaMemsetAsync(C, 0, static_cast<size_t>(M) * N * esz, st) == cudaSuccess ? SK_OK : SK_ECUDA;
    }

    // A in 128-row boxes (one CTA's rows); B in boxes of one CTA's share of the tile's
    // columns (NT) or in 64 x 64 boxes (NN).
    CUtensorMap tmA, tmB;
    if (!encode_2d(&tmA, A, static_cast<uint64_t>(K), static_cast<uint64_t>(M), kBlkK, kCtaRows)) return SK_ECUDA;
    const bool nt = layout == SK_NT;
    const uint32_t b_rows = static_cast<uint32_t>(sch.tile_n / sch.cg);
    const bool okb = nt ? encode_2d(&tmB, B, static_cast<uint64_t>(K), static_cast<uint64_t>(N), kBlkK, b_rows)
                        : encode_2d(&tmB, B, static_cast<uint64_t>(N), static_cast<uint64_t>(K), 64, kBlkK);
    if (!okb) return SK_ECUDA;

    uint8_t* ws = static_cast<uint8_t*>(workspace);
    KArgs a = {};
    a.sch = sch;
    a.C = C;
    a.status = reinterpret_cast<int32_t*>(ws);
    a.flags = reinterpret_cast<int32_t*>(ws + flags_offset());
    a.slots = reinterpret_cast<float*>(ws + slots_offset(sch));
    a.slabs = sch.partials ? reinterpret_cast<float*>(ws + SK_WS_HEADER_BYTES) : nullptr;
    a.counters = sch.partials == 2 ? reinterpret_cast<int32_t*>(ws + slab_counters_offset(sch.splits, M, N)) : nullptr;
    a.M = M;
    a.N = N;
    a.K = K;
    a.c_bf16 = c_dtype == SK_BF16 ? 1 : 0;
    a.atomic = r == SK_ATOMIC ? 1 : 0;
    a.timeout_ns = static_cast<uint64_t>(kDefaultTimeoutNs);
    if (opts) {
        a.reverse = opts->reverse_units ? 1 : 0;
        a.skip_signal = opts->skip_producer_signal ? 1 : 0;
        a.zero_partials = opts->zero_partials ? 1 : 0;
        if (opts->timeout_ns > 0) a.timeout_ns = static_cast<uint64_t>(opts->timeout_ns);
        a.dump = opts->dump;
        if (a.dump && !aligned(a.dump, 16)) return SK_EINVAL;
        a.trace = opts->trace;
        if (a.trace && !aligned(a.trace, 8)) return SK_EINVAL;
    }
    // tmD: C. tmC: where segments store — C, or the FP32 slabs in split-partials mode,
    // summed into C by the reduction pass (1) or by the last split of each tile (2).
    CUtensorMap tmC, tmD;
    if (!encode_out(&tmD, C, a.c_bf16 != 0, static_cast<uint64_t>(N), static_cast<uint64_t>(M), 1, 2)) return SK_ECUDA;
    if (sch.partials) {
        if (!encode_out(&tmC, a.slabs, false, static_cast<uint64_t>(N), static_cast<uint64_t>(M),
                        static_cast<uint64_t>(sch.splits), 3))
            return SK_ECUDA;
    } else {
        tmC = tmD;
    }
    if (launch_gemm(tmA, tmB, tmC, tmD, nt, a, st) != cudaSuccess) {
        cudaGetLastError();
        return SK_ECUDA;
    }
    const int free_sms = dev_sms - sch.workers * sch.cg;  // SMs the GEMM's grid leaves idle
    if (sch.partials == 1) {
        if (launch_reduce(a.slabs, C, a.c_bf16, sch.splits, static_cast<int64_t>(M) * N, dev_sms, sch.overlap,
                          free_sms, st) != cudaSuccess) {
            cudaGetLastError();
            return SK_ECUDA;
        }
    }
    if (sch.sep) {
        if (launch_fixup(sch, a.slots, C, M, N, a.c_bf16, dev_sms, free_sms, st) != cudaSuccess) {
            cudaGetLastError();
            return SK_ECUDA;
        }
    }
    return SK_OK;
}

int32_t sk_gemm(const void* A, const void* B, void* C, sk_dtype c_dtype, int32_t M, int32_t N, int32_t K,
                sk_layout layout, sk_schedule s, sk_reduction r, int32_t num_sms, void* workspace, size_t ws_bytes,
                void* stream) {
    return sk_gemm_debug(A, B, C, c_dtype, M, N, K, layout, s, r, num_sms, workspace, ws_bytes, stream, nullptr);
}

int32_t sk_split_k_slices(int32_t M, int32_t N, int32_t K, int32_t num_sms) {
    (void)K;  // the heuristic looks at the output tiles only
    if (M < 1 || N < 1 || num_sms < 1) return SK_EINVAL;
    int64_t tiles = static_cast<int64_t>(M / 128) * (N / 128);
    if (tiles < 1) tiles = 1;
    if (tiles >= 2ll * num_sms) return 1;
    const int64_t target = 4ll * num_sms;
    const int64_t s = (target + tiles - 1) / tiles;
    return static_cast<int32_t>(s < 32 ? s : 32);
}

int32_t sk_reduce_splits(const float* P, void* C, sk_dtype c_dtype, int32_t splits, int64_t mn, void* stream) {
    if (splits < 1 || mn < 0 || mn % 4 != 0) return SK_EINVAL;
    if (c_dtype != SK_F32 && c_dtype != SK_BF16) return SK_EINVAL;
    if (mn == 0) return SK_OK;
    if (!P || !C || !aligned(P, 16) || !aligned(C, 16)) return SK_EINVAL;
    int dev_sms = 0, max_units[kTileShapes];
    if (device_info(&dev_sms, max_units) != cudaSuccess) return SK_ECUDA;
    if (launch_reduce(P, C, c_dtype == SK_BF16 ? 1 : 0, splits, mn, dev_sms, 0, 0, static_cast<cudaStream_t>(stream)) !=
        cudaSuccess) {
        cudaGetLastError();
        return SK_ECUDA;
    }
    return SK_OK;
}

int32_t sk_status(void* workspace, void* stream) {
    if (!workspace) return SK_EWORKSPACE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(st) != cudaSuccess) return SK_ECUDA;
    int32_t v = 0;
    if (cudaMemcpy(&v, workspace, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return SK_ECUDA;
    if (v != SK_OK) {
        const int32_t zero = SK_OK;
        if (cudaMemcpy(workspace, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) return SK_ECUDA;
    }
    return v;
}

}  // extern "C"

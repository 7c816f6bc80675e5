/*
 * sk.h - C ABI of the work-decomposed BF16 GEMM for GB300 (sm_103a).
 *
 * C = A . B with BF16 inputs and FP32 accumulation, the output tiles and their
 * K loops spread over persistent CTAs by one of four schedules: data-parallel,
 * Split-K, Stream-K, or the hybrid rule ("Split-K and Stream-K: The Last Wave of
 * a GEMM", kanthi.in: Mental model, Case 2 and Case 4).
 *
 * Conventions shared by every entry point
 *   - Output tile 128 x 128, MAC-loop iteration BK = 64 (page above, Mental model
 *     table and Case 2): tiles = ceil(M/128) * ceil(N/128), iters = ceil(K/64).
 *     Tile t covers rows (t / tiles_n) * 128 and columns (t % tiles_n) * 128.
 *   - A is [M, K] row-major BF16. Layout SK_NN: B is [K, N] row-major. Layout
 *     SK_NT: B is stored [N, K] row-major ("Consecutive-B split-K NAX GEMM",
 *     Contract). C is [M, N] row-major, FP32 or BF16 (round to nearest even,
 *     once, after the fixup).
 *   - The caller owns every buffer. No entry point allocates memory.
 *   - Device pointers are plain CUDA device addresses; `stream` is a cudaStream_t
 *     (NULL = the legacy default stream). sk_gemm, sk_reduce_splits and sk_gemm_host
 *     are asynchronous on that stream. Only sk_gemm_host takes host pointers for A, B
 *     and C.
 *   - Return value: SK_OK (0) or a negative SK_E* code; sk_strerror names it.
 */
#ifndef SK_H_
#define SK_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Decomposition modes ("Split-K and Stream-K: The Last Wave of a GEMM", Case 4:
 * DataParallel | SplitK | StreamK | Heuristic). SK_HYBRID is the heuristic: a last
 * wave that holds half the SMs or more keeps the GEMM data-parallel; a smaller one
 * hands the tiles of the final two waves to Stream-K, with no unit given fewer than
 * min_iters k-iterations (Case 2, cutlass_heuristic and hybrid). */
typedef enum { SK_DP = 0, SK_SPLITK = 1, SK_STREAMK = 2, SK_HYBRID = 3 } sk_mode;
typedef enum { SK_NN = 0, SK_NT = 1 } sk_layout;
/* Reduction modes (Case 4): deterministic = the owner adds its peers' FP32
 * partials in k order (a turnstile); atomic = peers add FP32 partials into one
 * workspace tile with atomics. With two peers the sum 0 + a + b is the same either
 * way round; from three contributors on, the FP32 additions happen in whatever order
 * the peers finish, so the result's last bits can change from run to run (Case 3). */
typedef enum { SK_DETERMINISTIC = 0, SK_ATOMIC = 1 } sk_reduction;
typedef enum { SK_F32 = 0, SK_BF16 = 1 } sk_dtype;
/* Segment roles in the work-unit map. FULL: one unit runs the whole K loop of a
 * tile and writes C. OWNER: the unit holding the tile's k = 0 iteration; it waits
 * for its peers, adds their partials and writes C. PRODUCER: a later segment of a
 * split tile; it stores its FP32 partial and raises a flag (Mental model; Case 2
 * stream_k_units). SLAB: a Split-K split that writes its own FP32 [M,N] slab,
 * reduced afterwards by sk_reduce_splits (split-K report, Contract). */
typedef enum { SK_ROLE_FULL = 0, SK_ROLE_OWNER = 1, SK_ROLE_PRODUCER = 2, SK_ROLE_SLAB = 3 } sk_role;

/* Work-tile shapes. The pages' tile is 128 x 128 computed by one CTA (SK_TILE_128x128).
 * The pair shapes are computed by two CTAs on neighbouring SMs together (tcgen05
 * cta_group::2, each CTA holding half of the tile's rows and half of B's columns), so a
 * persistent unit is a CTA pair and num_sms SMs give num_sms / 2 units; CUTLASS
 * example 74 on the first page uses the 256 x 128 pair tile. */
typedef enum {
    SK_TILE_128x128 = 0,
    SK_TILE_256x128_PAIR = 1,
    SK_TILE_256x256_PAIR = 2,
    SK_TILE_128x256 = 3
} sk_tile;

typedef struct {
    int32_t mode;           /* sk_mode */
    int32_t splits;         /* Split-K split count s, 1 <= s <= iters (SK_SPLITK only) */
    int32_t units;          /* 0: num_sms persistent units; > 0: use this many instead */
    int32_t min_iters;      /* hybrid rule's minimum k-iterations per Stream-K unit; 0 = 8 */
    int32_t split_partials; /* 0: the unit holding a split tile's k = 0 iteration waits
                               for its peers and sums their partials (in-kernel fixup).
                               SK_SPLITK, 1: every split writes an FP32 slab P[j] into the
                               workspace and a second launch (the sk_reduce_splits pass)
                               sums the slabs in split order into C.
                               SK_SPLITK, 2: as 1, but inside the one launch. When every
                               work item gets a unit of its own (tiles * splits <= units),
                               the splits of a tile wait for each other and each sums a
                               share of the tile's rows; otherwise the split that arrives
                               last at a tile sums that tile's slabs into C.
                               SK_STREAMK / SK_HYBRID, 1: separate fixup pass (first page,
                               Case 3): every partial segment, the owner's too, stores its
                               FP32 partial to a fixed slot (2u for unit u's first segment,
                               2u + 1 for its last) and nobody waits; a second launch sums
                               each split tile's slots in k order into C. The sum order is
                               the turnstile's, so `r` does not apply.
                               SK_DP takes 0 only. */
    int32_t tile;           /* sk_tile; 0 = 128 x 128 */
    int32_t raster;         /* tile-id order ("Threadblock Rasterization", CUTLASS page):
                               0 = along N (row-major, tile t at tile row t / tiles_n),
                               1 = along M (column-major) */
    int32_t swizzle;        /* 0 or 1: none; w = 2 .. 256: the dimension across the walk is
                               cut into strips w tiles deep, and ids fill one strip at a
                               time, across its w tiles first (tiles that run together
                               then share A and B panels in L2) */
    int32_t overlap;        /* launch option; the plan is the same either way. 0: each
                               launch starts once the work before it on the stream is
                               done. 1: programmatic dependent launch (CUDA): the GEMM's
                               CTAs may start, initialise their barriers and allocate
                               tensor memory while the kernel before it on the stream is
                               still running; every thread waits for that kernel to
                               complete (its writes visible) before it touches global
                               memory, so the result is the same. The reduction or fixup
                               pass of split_partials = 1 overlaps the GEMM the same way.
                               Each device-side wait limit then counts from that wait.
                               The one-CTA tiles then launch without the cooperative
                               attribute, after the same residency check as the pairs.
                               2: as 1, and the caller states that A and B are not
                               written by the kernel just before this call on the stream
                               (nor by any kernel that one may overlap): GEMMs over
                               independent operands one after another. Each unit's TMA
                               loads and MMAs of its first two segments (its two fresh
                               accumulators) then start before that kernel has completed;
                               C, the workspace and every flag are still touched only
                               after it, so results are the same bit for bit as with 1.
                               A caller whose A or B come from that kernel must use 1. */
    int32_t sk_groups;      /* Stream-K grouping (first page, Case 4 knob table,
                               max_sk_groups_: at most 8 groups of Stream-K units, so
                               that partials made at about the same time still sit in
                               L2 when their owners read them). 0 or 1:
                               one group, the page's simulator plan. g >= 2 (at most 64):
                               the Stream-K region's tiles and its units are each cut into
                               up to g consecutive groups, big-first (the first tiles % g
                               and units % g groups one larger), and a group's units split
                               only its own tiles by the divmod rule. Fewer groups are
                               used when g exceeds the region's tiles or units, or when a
                               group would hold fewer k-iterations than units; the map
                               header reports the count used. Ignored by data-parallel
                               and Split-K plans. */
} sk_schedule;

#define SK_OK          0
#define SK_EINVAL     -1  /* bad argument: sizes, schedule, alignment or layout */
#define SK_EWORKSPACE -2  /* workspace missing, misaligned or smaller than sk_workspace_size */
#define SK_ECUDA      -3  /* a CUDA runtime or driver call failed */
#define SK_ETIMEOUT   -4  /* a device-side wait ran past its time limit (from sk_status) */
#define SK_ECAPACITY  -5  /* sk_plan: the map buffer is smaller than sk_plan_size */
#define SK_ERESIDENCY -6  /* more persistent units than the device can hold at once */
#define SK_EBOUNDS    -7  /* a device-side index check failed; the access was skipped (from sk_status) */

#define SK_TILE_M 128   /* tile of SK_TILE_128x128 */
#define SK_TILE_N 128
#define SK_BLK_K 64

/* Work-unit map layout (int32). Header of SK_MAP_HEADER values:
 *   [0] version (SK_MAP_VERSION)   [1] resolved mode (sk_mode; the hybrid rule resolves
 *   to SK_DP or SK_HYBRID)   [2] tiles   [3] iters   [4] workers = units launched
 *   (CTA pairs for the pair tiles)
 *   [5] sk_tiles: tiles in the Stream-K region (the last sk_tiles tile ids)
 *   [6] sk_units: units over that region   [7] n_segments
 *   [8] splits: effective Split-K split count (empty trailing splits dropped), else 0
 *   [9] hybrid label (-1 none, 0 DataParallel, 1 SplitK, 2 StreamK)
 *   [10] the label's split count   [11] n_slots: FP32 partial-tile slots used
 *   [12] tile_m   [13] tile_n   [14] CTAs per tile (1 or 2)
 *   [15] raster   [16] swizzle (the tile-id order of sk_schedule)
 *   [17] Stream-K groups used (1 with one group; 0 without a Stream-K region)
 * then n_segments rows of SK_MAP_SEG values, in (unit, run order) order:
 *   unit, order, tile, k_begin, k_end, role, slot, peer_begin, n_peers
 *   (k_begin/k_end in k-iterations; PRODUCER: slot = its partial slot; OWNER: its peers'
 *   partials are slots peer_begin .. peer_begin + n_peers - 1 in k order; PRODUCER rows
 *   carry their owner's peer_begin, which is also the tile's slot in atomic mode;
 *   with the separate Stream-K fixup pass, OWNER and PRODUCER rows hold their own slot,
 *   2 * unit or 2 * unit + 1, and the peer fields only describe the tile;
 *   SLAB: slot = split index; unused fields are -1 or 0)
 * then `tiles` rows of SK_MAP_TILE values: owner unit (runs k = 0), contributors, and
 * the tile's row and column in the tile grid (its output rows start at row * tile_m, its
 * columns at column * tile_n). */
#define SK_MAP_VERSION 3
#define SK_MAP_HEADER 18
#define SK_MAP_SEG 9
#define SK_MAP_TILE 4

/* Workspace layout: bytes [0, SK_WS_HEADER_BYTES) hold the device status word
 * (int32 at offset 0). In split-partials mode the FP32 slabs P[j][M][N] follow at
 * offset SK_WS_HEADER_BYTES, j = 0 .. splits-1, row-major, then (256-aligned) one int32
 * arrival counter per tile and CTA of the tile, used by split_partials = 2 (the split
 * that arrives last at a tile sums that tile's slabs in split order into C) and kept at
 * zero between launches. In the other modes one int32 flag (or counter) per slot and CTA
 * of the tile follows (256-aligned), then the partial slots of tile_m x tile_n FP32
 * each. */
#define SK_WS_HEADER_BYTES 256

/* Number of int32 values sk_plan writes for this problem, or a negative SK_E* code.
 * M, N, K >= 1; num_sms >= 1 (the SM count the schedule is built for). */
int64_t sk_plan_size(int32_t M, int32_t N, int32_t K, int32_t num_sms, sk_schedule s);

/* Split-K factor heuristic (CUTLASS "Optimization Techniques" page, Split-K section,
 * "Optimal Split-K Factor"): the number of K splits for an M x N x K problem on num_sms
 * SMs. Whole 128 x 128 tiles of M x N are counted (floor division; fewer than one counts
 * as one); with at least 2 * num_sms tiles the answer is 1, else the splits per tile that
 * reach 4 * num_sms blocks, rounded up and capped at 32. K does not enter; a caller
 * clamps the factor to ceil(K / 64) before using it as sk_schedule.splits. Host-only.
 * Returns the factor (1 .. 32), or SK_EINVAL unless M, N >= 1 and num_sms >= 1. */
int32_t sk_split_k_slices(int32_t M, int32_t N, int32_t K, int32_t num_sms);

/* Write the work-unit map (layout above) into the host buffer `map` of `cap` int32.
 * Host-only; touches no GPU. Each persistent unit of sk_gemm runs exactly the
 * segments listed for it here, in this order. Stream-K ranges use q, big =
 * divmod(tiles * iters, units) with the first `big` units one iteration longer
 * (Case 2 stream_k_units; "Try this" calls it the CUTLASS split). Returns SK_OK,
 * SK_EINVAL, or SK_ECAPACITY when cap < sk_plan_size. */
int32_t sk_plan(int32_t M, int32_t N, int32_t K, int32_t num_sms, sk_schedule s,
                int32_t* map, int64_t cap);

/* Bytes of device workspace sk_gemm needs for this problem, schedule and reduction
 * (at least SK_WS_HEADER_BYTES), or a negative SK_E* code. Host-only.
 * The workspace must be 256-byte aligned and ZERO-FILLED before its first use; a
 * successful sk_gemm leaves every flag, counter and atomic slot at zero again, so
 * the same workspace can be reused call after call without clearing. */
int64_t sk_workspace_size(int32_t M, int32_t N, int32_t K, int32_t num_sms, sk_schedule s,
                          sk_reduction r);

/* C = A . B on `stream` (Mental model; Case 2; Case 4 of the page above).
 * A: device [M,K] BF16; B: device BF16, [K,N] (SK_NN) or [N,K] (SK_NT); C: device
 * [M,N] of c_dtype. Requirements: K % 8 == 0 and N % 8 == 0 (16-byte row strides for
 * the tensor-memory-access loads and vector stores); A and B 16-byte aligned, C
 * 16-byte aligned; inputs must not overlap C or the workspace. M == 0 or N == 0 does
 * nothing; K == 0 writes zeros. The persistent units run as one launch in which every
 * unit (one CTA, or a CTA pair for the pair tiles) is resident at once: a cooperative
 * launch, or a launch after an occupancy check (pair tiles, and any overlapped launch),
 * so the units may not exceed what the device holds at once (else SK_ERESIDENCY).
 * With s.overlap the launch may begin before the kernel ahead of it on the stream has
 * finished, and waits for it before touching memory. Errors are returned before anything
 * is enqueued. A device-side wait that runs past its limit makes the kernel stop early and
 * record SK_ETIMEOUT in the workspace status word (read it with sk_status); C is then
 * undefined and the workspace must be zero-filled again before reuse. Concurrent calls
 * must not share a workspace; calls one after another on one stream may, overlapped or
 * not. */
int32_t sk_gemm(const void* A, const void* B, void* C, sk_dtype c_dtype,
                int32_t M, int32_t N, int32_t K, sk_layout layout, sk_schedule s,
                sk_reduction r, int32_t num_sms, void* workspace, size_t ws_bytes,
                void* stream);

/* Diagnostic controls for sk_gemm_debug (used by the tests; sk_gemm uses the defaults). */
typedef struct {
    int32_t reverse_units;        /* 1: CTA b runs unit workers-1-b, another dispatch order of
                                     the same units (the page's Case 3 varies arrival order
                                     with a unit permutation) */
    int32_t skip_producer_signal; /* 1: producers store their partials but never raise their
                                     flag, so every owner's wait runs out; Split-K slab splits
                                     that share the sum never count their arrival, so their
                                     wait runs out too (time-out tests) */
    int64_t timeout_ns;           /* limit of every device-side wait, from kernel start;
                                     0 = the default of 2 s */
    float* dump;                  /* NULL, or a device buffer of tiles * iters * tile_m *
                                     tile_n FP32: the segment of tile t starting at
                                     k-iteration k writes its own accumulator (before any
                                     fixup), row-major tile_m x tile_n, at offset
                                     (t * iters + k) * tile_m * tile_n */
    uint64_t* trace;              /* NULL, or a device buffer of SK_TRACE_WORDS uint64 per
                                     CTA (workers * CTAs per tile): %globaltimer stamps in
                                     ns, layout below */
    int32_t zero_partials;        /* 1: numerical control ("Consecutive-B split-K NAX GEMM",
                                     Contract and numerical coverage: a candidate whose
                                     partial store is zeroed must fail the checks). Every
                                     partial a segment hands on (a Stream-K or Split-K
                                     producer's partial, a Split-K slab, an owner's slot of
                                     the separate fixup pass) is stored as zeros; flags and
                                     counters are raised as usual, so nothing waits longer.
                                     The result is then wrong wherever a tile was split. */
} sk_debug_opts;

/* Per-CTA trace record (sk_debug_opts.trace), indexed by blockIdx: [0] start (after set-up
 * and, for an overlapped launch, after the wait for the previous kernel), [1] end (after
 * the exit barrier), [2] segments walked, [3] SM clock cycles from [0] to [1] (so
 * [3] / ([1] - [0]) is the SM's clock while it ran); then for segment i
 * < SK_TRACE_SEGS, at 4 + 4 * i: [0] MMA issue of its first k-iteration (leader CTA only),
 * [1] MMA commit of its last, [2] epilogue has the accumulator, [3] epilogue done (after the
 * fixup and the stores). Unused words stay as the caller left them. */
#define SK_TRACE_SEGS 15
#define SK_TRACE_WORDS (4 + 4 * SK_TRACE_SEGS)

/* sk_gemm with diagnostic controls; opts == NULL behaves exactly like sk_gemm. */
int32_t sk_gemm_debug(const void* A, const void* B, void* C, sk_dtype c_dtype,
                      int32_t M, int32_t N, int32_t K, sk_layout layout, sk_schedule s,
                      sk_reduction r, int32_t num_sms, void* workspace, size_t ws_bytes,
                      void* stream, const sk_debug_opts* opts);

/* Split-K reduction pass ("Consecutive-B split-K NAX GEMM", Contract: FP32 partials
 * [splits, M, N] reduced by an accumulation kernel; first page, Case 3 fixup_kernel
 * sums partials in k order). C[i] = P[0][i] + P[1][i] + ... + P[splits-1][i], summed
 * left to right in FP32, then stored as c_dtype. P: device FP32, `splits` slabs of
 * `mn` values each, 16-byte aligned; C: device, 16-byte aligned; mn % 4 == 0. */
int32_t sk_reduce_splits(const float* P, void* C, sk_dtype c_dtype, int32_t splits,
                         int64_t mn, void* stream);

/* Scratch size of sk_gemm_noalloc: 16 MiB of device memory on every GPU that loads the
 * library, held until the process exits. */
#define SK_NOALLOC_SCRATCH_BYTES (16u << 20)

/* sk_gemm without a caller workspace, for callers that cannot allocate device memory
 * (plug-ins whose host application owns every allocation, processes held to a memory
 * budget fixed at start-up, loops where cudaMalloc / cudaFree would synchronise the
 * device). The pages have no counterpart: this is a deployment convenience.
 * Arguments are those of sk_gemm minus the workspace. The scratch is one library-owned
 * device array of SK_NOALLOC_SCRATCH_BYTES per GPU; problems whose sk_workspace_size
 * exceeds it return SK_EWORKSPACE and nothing is enqueued. The first call on a device
 * looks up the array's address with that device current; make it before any stream
 * capture. Every call enqueues a clear of the part that must start at zero (status word,
 * flags, and the partial tiles for SK_ATOMIC), then the GEMM. All calls on a device share
 * the array: calls whose work overlaps on the GPU (other streams, other host threads)
 * race. A device-side time-out is recorded in the scratch and not reported; use sk_gemm
 * and sk_status to observe it. Allocates nothing. */
int32_t sk_gemm_noalloc(const void* A, const void* B, void* C, sk_dtype c_dtype,
                        int32_t M, int32_t N, int32_t K, sk_layout layout, sk_schedule s,
                        sk_reduction r, int32_t num_sms, void* stream);

/* Bytes of device staging sk_gemm_host needs: `depth` sets (1 or 2) of A [M,K] BF16,
 * B (K x N BF16) and C [M,N] of c_dtype, each part starting on a 256-byte boundary inside
 * its set. Host-only. Returns the size, or SK_EINVAL for negative sizes, an unknown
 * c_dtype or another depth. */
int64_t sk_host_staging_size(int32_t M, int32_t N, int32_t K, sk_dtype c_dtype, int32_t depth);

/* `count` GEMMs of one shape whose operands and results live in host memory: for problem
 * i, A[i] and B[i] (host pointers, layouts as in sk_gemm) are copied into a device staging
 * set, C = A . B runs there as sk_gemm with the given schedule, reduction and workspace, and
 * C is copied to the host pointer C[i]. The pages have no counterpart: this is the end-to-end
 * call for callers whose matrices are in host memory.
 *   staging: device buffer of at least sk_host_staging_size(M, N, K, c_dtype, depth) bytes,
 *     256-byte aligned, owned by the caller (else SK_EWORKSPACE).
 *   depth 1: every copy and GEMM runs in order on `stream`; copy_in and copy_out are unused.
 *   depth 2: two staging sets used in turn; the uploads run on `copy_in` and the downloads on
 *     `copy_out` (two distinct non-NULL streams of the caller other than `stream`, else
 *     SK_EINVAL), so that
 *     problem i + 1's uploads and problem i - 1's download overlap problem i's GEMM. Events
 *     keep every buffer's writes and reads in order; the copy streams first wait for the
 *     caller's earlier work on `stream`.
 * Every GEMM runs on `stream`, one after another, sharing the workspace. The call is
 * asynchronous: once `stream` has reached the point where the call returned, every C[i]
 * has been written. Host buffers should be page-locked (cudaHostAlloc / cudaHostRegister)
 * for the copies to run asynchronously; pageable memory works, but the host then waits in
 * the copy calls. The host buffers must stay valid and A[i], B[i] unchanged until then; C
 * pointers may repeat (later problems overwrite earlier ones). The call creates and
 * releases seven CUDA events when depth is 2 and allocates no memory.
 * Errors: argument, staging and every sk_gemm check (including SK_ERESIDENCY) are made
 * before anything is enqueued. A CUDA failure after that (SK_ECUDA) returns at once,
 * leaving the earlier problems' work enqueued: synchronise all three streams before reusing
 * the buffers. count == 0, M == 0 or N == 0 does nothing. */
int32_t sk_gemm_host(int32_t count, const void* const* A, const void* const* B, void* const* C,
                     sk_dtype c_dtype, int32_t M, int32_t N, int32_t K, sk_layout layout, sk_schedule s,
                     sk_reduction r, int32_t num_sms, void* staging, size_t staging_bytes, int32_t depth,
                     void* workspace, size_t ws_bytes, void* stream, void* copy_in, void* copy_out);

/* Synchronise `stream`, read the workspace status word, reset it to SK_OK and return
 * it: SK_OK, or SK_ETIMEOUT when a kernel on that workspace stopped at a wait limit.
 * Also SK_EBOUNDS if a kernel found a workspace index outside the extents it was given
 * (it skips that access and stops). Returns SK_ECUDA if the copy fails. */
int32_t sk_status(void* workspace, void* stream);

/* Static description of an SK_* code. */
const char* sk_strerror(int32_t code);

#ifdef __cplusplus
}
#endif

#endif /* SK_H_ */

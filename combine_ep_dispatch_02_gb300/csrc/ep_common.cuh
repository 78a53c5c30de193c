// ep_common.cuh -- internal declarations shared by the dispatch / combine kernels and the C ABI.
//
// Layout in HBM (all row-major, one plan-owned allocation, sub-buffers 256-byte aligned):
//   recv_x       [W][W*M][H]   payload rows received by each logical rank
//   recv_idx     [W][W*M][k]   int32 top-k index rows
//   recv_w       [W][W*M][k]   FP32 weight rows
//   recv_scales  [W][W*M][sd]  FP32 scale rows
//   src_pos      [W][W*M]      reverse map: src_rank * (W*M) + src_token
//   fwd          [W][M][F]     forward map, F = min(W, k): the receive rows of token (s,t) as
//                              r * (W*M) + slot, in ascending destination rank, -1 padded
//   scan_cnt     [W*E][chunks][W]  grouping scan: hits of a 1024-row chunk per source rank,
//                              present when a rank's capacity spans kScanMinChunks chunks or more
//   recv_count   [W]
//   expert_map   [W][W*M][k]   slot of a received row in its local experts' lists (grouped view)
//   flags        [tiles][W]    decoupled-lookback scan words of the routing kernel
//   ticket       3 x u64       routing: next tile, CTAs finished (both back to zero after every
//                              launch) and the generation that stamps scan words; followed in
//                              its 256-byte block by the work queues, kQueues x 2 u64
//   status       int32         first device-side error
#pragma once

#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "ep.h"

namespace ep {

constexpr int kMaxRanks = 32;       // destination sets are uint32 bit masks
constexpr int kMaxTopk = 64;        // two 32-slot batches
constexpr int kRouteTile = 256;     // tokens per routing CTA, one per thread
constexpr int kRouteThreads = 256;
constexpr int kRouteControlWords = 3;   // u64: next tile, CTAs done, scan-word generation
// the routing kernel numbers the grouped view itself for up to this many experts in all (a tile
// keeps a 256-bit token mask per expert in shared memory) ...
constexpr int kRouteGroupMaxExperts = 1024;
// ... when the expert columns' lookback words fit in this
constexpr long long kRouteGroupMaxFlagBytes = 64ll << 20;
constexpr int kCopyThreads = 256;   // scatter, wire and grouped-view CTAs: 8 warps, a work unit per warp
constexpr int kScanChunk = 1024;    // received rows per step of the grouping scan (4 per thread)
constexpr int kScanMinChunks = 3;   // capacities of this many chunks or more are scanned in two passes
constexpr long long kScanMaxBytes = 64ll << 20;   // ... when their per-chunk counts fit in this

// Scan flag word: [63:34] call stamp (30 bits) | [33:32] status | [31:0] count.
constexpr unsigned long long kFlagAggregate = 1ull;   // count = this tile's own total
constexpr unsigned long long kFlagInclusive = 2ull;   // count = total of tiles 0..this one
constexpr uint32_t kStampMask = 0x3FFFFFFFu;
#ifndef EP_SPIN_LIMIT
#define EP_SPIN_LIMIT (1 << 20)
#endif
constexpr int kSpinLimit = EP_SPIN_LIMIT;   // polls before a wait gives up with EP_ERR_DEVICE_TIMEOUT

// Phase probes.  Built with -DEP_PROBE, every kernel's warps record, in the plan's control block,
// the earliest start and the latest end (%globaltimer, ns) of the phase's launches since the
// last ep_probe_read; other builds record nothing.
enum ProbePhase {
    kProbeRoute = 0, kProbeScatter, kProbeCombine, kProbeQuantise, kProbeWireCombine, kProbeGroupScan,
    kProbeGroupCopy, kProbeUngroup, kProbePhases
};
constexpr int kProbeWordOffset = 16;   // u64 words into the 256-byte control block (after the queues)

// Work queues of the persistent copy kernels (see WorkSplit): launches that share a queue must
// run one after the other, as the calls on one plan do.
constexpr int kQueueDispatch = 0;   // payload scatters (BF16 / FP8 / MX FP4 rows)
constexpr int kQueueGroup = 1;      // copy of received rows into the expert-grouped view
constexpr int kQueues = 2;

// ---- work split of a persistent copy kernel
//
// A token costs one read of its row and one write per destination rank, so a plain round-robin
// split of the units over the grid's G warps leaves a tail in which a few warps still copy
// expensive tokens while the rest of the GPU idles.  The split here is round-robin for all but
// the last two rounds' worth of units (warp w takes w, w + G, ... below static_end, with no
// atomics), and the rest are drawn one at a time, in ascending order, from a per-plan queue
// word q[0]: a warp whose units were cheap draws more of them.  Calls with fewer than four
// rounds of units are split round-robin only: there the queue word, polled by every warp of the
// grid, costs more than the imbalance it removes.  Once the queue is in use, each CTA counts
// itself in q[1] when all its warps are done, and the last CTA returns both words to zero, so
// the next launch on the same queue (stream-ordered after this one, or a CUDA-graph replay)
// starts from zero without a memset.  The launcher fills the split in the
// kernel's arguments, so the kernel reads it from the parameter bank rather than registers; a
// kernel whose unit count only the device knows builds the split itself.
struct WorkSplit {
    unsigned long long* q;   // two words, zero between launches
    uint32_t units;          // < 2^31 (checked by the host before every launch)
    uint32_t warps;          // warps of the grid
    uint32_t static_end;     // units below this are split round-robin
};

#ifdef __CUDACC__
__host__ __device__
#endif
inline WorkSplit make_work_split(unsigned long long* q, int64_t units, int64_t warps)
{
    WorkSplit s;
    s.q = q;
    s.units = (uint32_t)units;
    s.warps = (uint32_t)warps;
    const int64_t rounds = units / warps;
    s.static_end = (uint32_t)(rounds >= 4 ? (rounds - 2) * warps : units);
    return s;
}

// The expert-grouped view numbered by the routing kernel itself (fused dispatch into the grouped
// view): each tile also scans W*E expert columns, so the lists' slots, counts and layout ranges
// come out of the same launch as the receive rows.
struct RouteGroupArgs {
    unsigned long long* eflags;   // [tiles][W*E] lookback words of the expert columns
    int32_t* bnd;                 // [W+1][W*E] list prefix at each source's first token (scratch)
    int32_t* map;                 // [W][W*M][k] slot of a received row in its local experts' lists
    int32_t* src_info;            // [W*E][W*M] source token index per list slot
};

struct RouteArgs {
    const int32_t* idx;
    int32_t* fwd;
    int32_t* src_pos;
    int32_t* recv_count;
    unsigned long long* flags;
    unsigned long long* ticket;   // kRouteControlWords: next tile, CTAs done, generation
    int* status;
    unsigned long long* probe;    // phase probe words (EP_PROBE builds), or NULL
    int64_t rows;         // W*M
    int W, E, k, F, M, N;
    int tiles;            // CTAs of this launch: ceil(N / kRouteTile), at least 1
    int vec16;            // index rows may be read as 16-byte vectors (k % 4 == 0, idx 16-B aligned)
    int tok_off[kMaxRanks + 1];   // exclusive prefix of per-rank token counts; tok_off[W] = N
    RouteGroupArgs grp;   // used by the grouped launch only (launch_route_grouped)
};

struct ScatterArgs {
    const uint8_t* x;
    const float* w;
    const float* scales;
    const int32_t* idx;
    const int32_t* fwd;
    uint8_t* recv_x;
    int32_t* recv_idx;
    float* recv_w;
    float* recv_scales;
    WorkSplit work;       // q set by the caller, the rest by the launcher
    int* status;
    unsigned long long* probe;
    int64_t row_bytes;    // H * element size, a multiple of 16
    int W, k, F, M, sd, N;
    int chunk_bytes;      // bytes of one work unit's slice of a row (multiple of 16)
    int chunks;           // slices per row
    int tok_off[kMaxRanks + 1];
};

struct CombineArgs {
    const uint16_t* eo;
    const float* w_in;
    const int32_t* fwd;
    uint16_t* out;
    float* out_w;
    int* status;
    unsigned long long* probe;
    int64_t H;
    int W, k, F, M, N;
    int chunk_vecs;       // 16-byte vectors of one work unit's slice of a row
    int chunks;           // slices per row
    int tok_off[kMaxRanks + 1];
};

// Quantising the received expert rows, and combine over the resulting FP8 wire.
struct WireArgs {
    const uint16_t* eo;       // [W][W*M][H] BF16 expert outputs (quantise)
    uint8_t* q;               // [W][W*M][H] e4m3 codes (quantise: out; combine: in)
    float* scales;            // [W][W*M][H/128] (quantise: out; combine: in)
    const int32_t* recv_count;
    const int32_t* fwd;
    const float* w_in;
    uint16_t* out;            // [W][M][H] BF16
    float* out_w;
    int* status;
    unsigned long long* probe;
    int64_t H, rows;          // rows = W*M per rank
    int W, k, F, M, N;
    int chunk_pieces;         // 16-element pieces of one combine unit's slice
    int chunks;
    int tok_off[kMaxRanks + 1];
};

// Expert-grouped (3-D) view of the receive buffers, and its inverse.
struct GroupArgs {
    const uint8_t* recv_x;       // [W][W*M][row_bytes] received payload
    const int32_t* recv_idx;     // [W][W*M][k]
    const int32_t* recv_count;   // [W]
    const int32_t* src_pos;      // [W][W*M]
    int32_t* map;                // [W][W*M][k] plan-owned: slot of a row in an expert's list
    uint8_t* packed_x;           // [W][E][W*M][row_bytes]
    int32_t* count;              // [W][E]
    int32_t* src_info;           // [W][E][W*M]
    long long* layout_range;     // [W][E][W]
    const uint8_t* packed_y;     // [W][E][W*M][H] 16-bit expert outputs (inverse)
    uint8_t* out;                // [W][W*M][H] 16-bit combine input (inverse)
    // fused dispatch into the grouped view: the source side
    const int32_t* src_idx;      // [W][M][k] source index rows (grouping reads these if set)
    const uint8_t* x;            // [W][M][row_bytes] source payload rows
    const float* w;              // [W][M][k] or NULL
    const float* scales;         // [W][M][sd] or NULL
    const int32_t* fwd;          // [W][M][F]
    int32_t* recv_idx_out;       // metadata rows of the receive buffers
    float* recv_w_out;
    float* recv_scales_out;
    WorkSplit work;              // grouped copy / fused dispatch: q set by the caller
    int* status;
    unsigned long long* probe;
    int vec16;                   // the index rows grouping reads are 16-byte aligned (k % 4 == 0)
    int32_t* scan_cnt;           // [W*E][scan_chunks][W] plan-owned, or NULL: one-pass scan
    int scan_chunks;             // ceil(W*M / kScanChunk) when scan_cnt is set, else 0
    int scan_done;               // fused dispatch: routing already numbered the lists (no scan)
    const int32_t* bnd;          // ... and left every list's prefix at each source's first token,
                                 // [W+1][W*E], for the copy to write counts and layout ranges
    int64_t rows;                // W*M
    int64_t row_bytes;           // payload bytes (grouping) / 16-bit row bytes (inverse)
    int W, E, k, M, F, N, sd;
    int chunk_bytes, chunks;     // fused dispatch: work unit = (token, slice of chunk_bytes);
                                 // inverse: (received row, slice of chunk_bytes), chunks per row
    int tok_off[kMaxRanks + 1];
};

// Host-side launchers, one per kernel translation unit.
cudaError_t launch_route(const RouteArgs& a, cudaStream_t stream);
// routing that also numbers the expert-grouped view (a.grp set; W*E <= kRouteGroupMaxExperts)
cudaError_t launch_route_grouped(const RouteArgs& a, cudaStream_t stream);
cudaError_t launch_scatter(const ScatterArgs& a, int num_sms, cudaStream_t stream);
// BF16 rows in, FP8 e4m3 rows + FP32 scales (one per 128 elements) out.  Here a.row_bytes is
// the FP8 row (= H), a.chunk_bytes the slice in ELEMENTS (a multiple of 128) and a.sd = H/128.
cudaError_t launch_scatter_quant(const ScatterArgs& a, int num_sms, cudaStream_t stream);
// MX FP4 quantising scatter: a.row_bytes = H/2, a.chunk_bytes = slice length in ELEMENTS (a
// multiple of 32), recv_scales rows hold H/32 e8m0 bytes (sd = H/128 words)
cudaError_t launch_scatter_quant_fp4(const ScatterArgs& a, int num_sms, cudaStream_t stream);
cudaError_t launch_combine(const CombineArgs& a, bool fp16, int num_sms, cudaStream_t stream);
cudaError_t launch_quantise_rows(const WireArgs& a, int num_sms, cudaStream_t stream);
cudaError_t launch_group(const GroupArgs& a, int num_sms, cudaStream_t stream);
cudaError_t launch_ungroup(const GroupArgs& a, bool fp16, int num_sms, cudaStream_t stream);
// dispatch straight into the grouped view (needs routing done; a.src_idx, a.x, a.fwd set)
cudaError_t launch_group_from_source(const GroupArgs& a, int num_sms, cudaStream_t stream);
cudaError_t launch_combine_fp8(const WireArgs& a, int num_sms, cudaStream_t stream);
// MX FP4 wire: a.q [W][W*M][H/2] packed e2m1, a.scales [W][W*M][H/32] e8m0 bytes; for the
// combine a.chunk_pieces counts 32-element blocks per slice
cudaError_t launch_quantise_rows_fp4(const WireArgs& a, int num_sms, cudaStream_t stream);
cudaError_t launch_combine_fp4(const WireArgs& a, int num_sms, cudaStream_t stream);
// choose combine's slice of a row per work unit (a.H and a.N set)
void combine_geometry(CombineArgs& a, int variant, int num_sms);

#ifdef __CUDACC__
// Launch kernel k as a programmatic dependent of the kernel before it on `stream`: the grid may
// be scheduled while that kernel still runs (once each of its CTAs has executed
// allow_dependents() or exited), so its launch and its CTAs' start overlap the predecessor's
// tail; every thread of k calls wait_for_predecessor() before it reads or writes anything the
// predecessor wrote or reads, which returns once the predecessor has completed and its memory
// operations are visible.  Kernels that follow another of this library's kernels within one
// call (the payload scatter after routing, the grouping passes after routing or after each
// other) launch this way.
template <typename... Params, typename... Args>
cudaError_t launch_dependent(void (*k)(Params...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                             Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k, args...);
}
#endif

// ----------------------------------------------------------------------------- device helpers
#ifdef __CUDACC__

// A dependent kernel's wait for its predecessor (see launch_dependent); returns at once when the
// kernel was launched in the ordinary way.
__device__ __forceinline__ void wait_for_predecessor()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Lets the kernel's dependent (launched with launch_dependent) be scheduled before this kernel
// has finished; the dependent still waits for this kernel's completion before touching its data.
__device__ __forceinline__ void allow_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void record_status(int* status, int code)
{
    if (*reinterpret_cast<volatile int*>(status) == 0) atomicCAS(status, 0, code);
}

// EP_CHECKS builds: an index the kernel derived from device data (a forward-map entry, a slot,
// a receive count) that falls outside its buffer is recorded as EP_ERR_DEVICE_BOUNDS and the
// access is skipped; other builds compile the check away (the host validated everything else).
#ifdef EP_CHECKS
#define EP_IN_BOUNDS(cond, status) ((cond) ? true : (record_status((status), EP_ERR_DEVICE_BOUNDS), false))
#else
#define EP_IN_BOUNDS(cond, status) true
#endif

// A forward-map entry as the copy and combine kernels use it (called by all 32 lanes): in
// EP_CHECKS builds an entry outside [-1, total rows) makes the whole unit read -1 (skipped), so
// the unit's valid entries stay packed first.
__device__ __forceinline__ int checked_fwd(int v, int64_t total_rows, int* status)
{
#ifdef EP_CHECKS
    if (__any_sync(0xffffffffu, v < -1 || (int64_t)v >= total_rows)) {
        if ((threadIdx.x & 31) == 0) record_status(status, EP_ERR_DEVICE_BOUNDS);
        return -1;
    }
#else
    (void)total_rows; (void)status;
#endif
    return v;
}

// A rank's receive count as a kernel uses it: in EP_CHECKS builds a count outside [0, rows]
// reads as 0 (the rank's rows are skipped).
__device__ __forceinline__ int checked_count(int n, int64_t rows, int* status)
{
    return EP_IN_BOUNDS(n >= 0 && (int64_t)n <= rows, status) ? n : 0;
}

__device__ __forceinline__ unsigned long long global_ns()
{
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// EP_PROBE builds: lane 0 of every warp folds its start (begin) or end time into the phase's
// [earliest start, latest end] pair; `probe` is the plan's probe words (NULL: nothing recorded).
__device__ __forceinline__ void probe_mark(unsigned long long* probe, int phase, bool begin)
{
#ifdef EP_PROBE
    if (probe != nullptr && (threadIdx.x & 31) == 0) {
        if (begin) atomicMin(probe + 2 * phase, global_ns());
        else atomicMax(probe + 2 * phase + 1, global_ns());
    }
#else
    (void)probe; (void)phase; (void)begin;
#endif
}

// e / E for 0 <= e < W*E (W <= 32) without an integer division, given inv_e = RN(1/E): the float
// product lies within 2^-17 of e/E < 32, so it truncates to the exact quotient or one either side
// of it, and the remainder's sign and size fix that.
__device__ __forceinline__ int expert_rank(int e, int E, float inv_e)
{
    int q = __float2int_rz(__int2float_rn(e) * inv_e);
    const int rem = e - q * E;
    q += (rem >= E) - (rem < 0);
    return q;
}

// Asks for the 32-byte sector at p to be brought into L2 and returns at once (no register holds
// the data): a fold that keeps its next column in registers also asks for the column after it,
// so more bytes are on their way from DRAM than its registers could hold.
__device__ __forceinline__ void prefetch_l2(const void* p)
{
    asm volatile("prefetch.global.L2 [%0];" :: "l"(p));
}

// This warp's first unit, or s.units if it has none.
__device__ __forceinline__ uint32_t work_first(const WorkSplit& s)
{
    const uint32_t w = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    return w < s.static_end ? w : s.units;
}

// The unit after u, or s.units when the work is done (warp-uniform).
__device__ __forceinline__ uint32_t work_next(const WorkSplit& s, uint32_t u, int lane)
{
    if (u + s.warps < s.static_end) return u + s.warps;
    if (s.static_end >= s.units) return s.units;
    unsigned long long t = ~0ull;
    if (lane == 0) {
        unsigned long long seen;   // an exhausted queue is seen by a plain read, without an atomic
        asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(seen) : "l"(s.q) : "memory");
        if (seen < s.units - s.static_end) t = atomicAdd(s.q, 1ull);
    }
    t = __shfl_sync(0xffffffffu, t, 0);
    return t < s.units - s.static_end ? s.static_end + (uint32_t)t : s.units;
}

// Called by every thread of the CTA after its last unit: resets the queue once the grid is done.
__device__ __forceinline__ void work_retire(const WorkSplit& s)
{
    if (s.static_end >= s.units) return;   // the queue was not used
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();   // this CTA's draws are ordered before its retirement
        if (atomicAdd(s.q + 1, 1ull) == (unsigned long long)gridDim.x - 1) {   // the last CTA
            __threadfence();
            atomicExch(s.q, 0ull);
            atomicExch(s.q + 1, 0ull);
        }
    }
}

// Source rank of flattened token g (tokens of rank 0 first, then rank 1, ...); off in shared.
__device__ __forceinline__ int rank_of_token(const int* off, int W, int g)
{
    int s = 0;
    while (s + 1 < W && off[s + 1] <= g) ++s;
    return s;
}

// 16-byte streaming read of data nothing writes during the kernel: skip L1 allocation.
__device__ __forceinline__ uint4 ld_stream_v4(const void* p)
{
    uint4 v;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}

__device__ __forceinline__ void st_v4(void* p, const uint4& v)
{
    asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};"
                 :: "l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
}

// 32-byte store (two 16-byte vectors, lo first); p must be 32-byte aligned.  A warp's request
// then writes whole 32-byte sectors even where lanes are 32 or 64 bytes apart.
__device__ __forceinline__ void st_v8(void* p, const uint4& lo, const uint4& hi)
{
    asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};"
                 :: "l"(p), "r"(lo.x), "r"(lo.y), "r"(lo.z), "r"(lo.w), "r"(hi.x), "r"(hi.y), "r"(hi.z),
                    "r"(hi.w) : "memory");
}

__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long* p)
{
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_relaxed_u64(unsigned long long* p, unsigned long long v)
{
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" :: "l"(p), "l"(v) : "memory");
}

// ---- FP8 e4m3 block quantisation (one FP32 scale per 128 elements)

// Two floats -> two e4m3 codes (round to nearest even, saturating to +-448); lo in the low byte.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi)
{
    unsigned short r;
    asm("{ .reg .b16 t; cvt.rn.satfinite.e4m3x2.f32 t, %1, %2; mov.b16 %0, t; }"
        : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// x / s from y = RN(1/s) without a division: q0 = RN(x * y) lies within one ulp of x / s, so the
// residual x - q0 * s is exact in one fma, and RN(q0 + residual * y) is the correctly rounded
// quotient (P. Markstein, "Computation of elementary functions on the IBM RISC System/6000
// processor", IBM J. Res. Develop. 34(1), 1990).  Used only for 2^-60 <= s <= 2^126: below that
// the residual of a BF16 dividend can underflow.  A zero quotient takes the sign of x, as the
// division's does.  Over that scale range the e4m3 code of this quotient equals the code of the
// IEEE quotient for every BF16 x with |x| <= 448 s (checked exhaustively against the division).
__device__ __forceinline__ float div_by_scale(float x, float s, float y)
{
    const float q0 = __fmul_rn(x, y);
    const float r = __fmaf_rn(-q0, s, x);
    const float q1 = __fmaf_rn(r, y, q0);
    return __uint_as_float(__float_as_uint(q1) | (__float_as_uint(x) & 0x80000000u));
}

// Quantise one lane's 16 consecutive BF16 values (two 16-byte vectors) with the block scale:
// q = e4m3(x / scale), the FP32 quotient rounded to nearest even.
__device__ __forceinline__ uint4 quantise16(const uint4& a, const uint4& b, float scale)
{
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    uint32_t o[4];
    if (scale >= 0x1p-60f && scale <= 0x1p126f) {
        const float y = __frcp_rn(scale);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t p0 = e4m3x2(div_by_scale(bf16_lo(w[2 * i]), scale, y),
                                       div_by_scale(bf16_hi(w[2 * i]), scale, y));
            const uint32_t p1 = e4m3x2(div_by_scale(bf16_lo(w[2 * i + 1]), scale, y),
                                       div_by_scale(bf16_hi(w[2 * i + 1]), scale, y));
            o[i] = p0 | (p1 << 16);
        }
    } else {   // tiny or infinite block scales: IEEE division
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t p0 = e4m3x2(__fdiv_rn(bf16_lo(w[2 * i]), scale), __fdiv_rn(bf16_hi(w[2 * i]), scale));
            const uint32_t p1 =
                e4m3x2(__fdiv_rn(bf16_lo(w[2 * i + 1]), scale), __fdiv_rn(bf16_hi(w[2 * i + 1]), scale));
            o[i] = p0 | (p1 << 16);
        }
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

__device__ __forceinline__ float absmax16(const uint4& a, const uint4& b)
{
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    float m = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) m = fmaxf(m, fmaxf(fabsf(bf16_lo(w[i])), fabsf(bf16_hi(w[i]))));
    return m;
}

// ---- MX FP4 (OCP microscaling): 32-element blocks of e2m1 codes sharing one e8m0 scale
//
// scale code = floor(log2(max|x|)) - 2 + 127, clamped to 0..254 (127 for an all-zero block);
// element code = e2m1 of x / 2^(code - 127), nearest with ties to the even code, saturating at
// +-6.  Dividing by a power of two equals multiplying by its exact reciprocal 2^(127 - code),
// so the quotient is formed by one multiply.  Nibbles: element 2i low, 2i + 1 high.

__device__ __forceinline__ uint32_t e2m1x2(float lo, float hi)
{
    uint32_t r;
    asm("{ .reg .b8 t; cvt.rn.satfinite.e2m1x2.f32 t, %1, %2; cvt.u32.u8 %0, t; }"
        : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// Codes (16 bytes) of the 32 BF16 values in x[0..3]; `code` receives the block's scale code.
__device__ __forceinline__ uint4 quantise_mxfp4_32(const uint4 (&x)[4], uint32_t& code)
{
    float m = 0.0f;
#pragma unroll
    for (int t = 0; t < 4; ++t) m = fmaxf(m, absmax16(x[t], x[t]));
    code = 127;
    if (m > 0.0f) {
        const uint32_t mb = __float_as_uint(m);
        int e2 = (int)(mb >> 23) - 127;
        if ((mb >> 23) == 0) e2 = -127 - (__clz(mb & 0x7FFFFFu) - 9);   // subnormal maximum
        const int c = e2 - 2 + 127;
        code = (uint32_t)(c < 0 ? 0 : (c > 254 ? 254 : c));
    }
    // 2^(127 - code); code <= 253 for any BF16 input (Inf gives 253), 254 would be 2^-127
    const float inv = __uint_as_float(code >= 254u ? 0x00400000u : (254u - code) << 23);
    uint32_t o[4];
#pragma unroll
    for (int t = 0; t < 4; ++t) {
        const uint32_t w[4] = {x[t].x, x[t].y, x[t].z, x[t].w};
        uint32_t bytes = 0;
#pragma unroll
        for (int h = 0; h < 4; ++h) {
            const float lo = __fmul_rn(__uint_as_float(w[h] << 16), inv);
            const float hi = __fmul_rn(__uint_as_float(w[h] & 0xFFFF0000u), inv);
            bytes |= e2m1x2(lo, hi) << (8 * h);
        }
        o[t] = bytes;
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

// Two e4m3 codes (low byte first) -> two exact floats, via the exact e4m3 -> f16 conversion.
__device__ __forceinline__ float2 e4m3x2_to_float2(uint32_t two_codes)
{
    uint32_t h2;
    asm("{ .reg .b16 c; cvt.u16.u32 c, %1; cvt.rn.f16x2.e4m3x2 %0, c; }" : "=r"(h2) : "r"(two_codes));
    const __half2 h = *reinterpret_cast<const __half2*>(&h2);
    return __half22float2(h);
}

__device__ __forceinline__ unsigned lanemask_lt()
{
    unsigned m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

#endif  // __CUDACC__

}  // namespace ep

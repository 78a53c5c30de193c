// ep_grouped.cu -- the expert-grouped ("standard MoE", 3-D) view of a dispatch and its inverse.
//
// MORI-EP guide, section 4 "Standard MoE Compatibility": convert_dispatch_output() turns the
// 2-D receive buffers into packed_recv_x [experts][capacity][H] with packed_recv_count,
// packed_recv_src_info and packed_recv_layout_range, the layout a grouped GEMM consumes;
// convert_combine_input() brings expert outputs back to the 2-D combine input.  Readings (the
// guide names the outputs only): on rank r the list of local expert e holds, in receive-row
// order, every received row whose top-k names global expert r*E + e (once per row); src_info is
// the row's source token index; layout_range[s] = (first slot of source rank s) << 32 | count;
// the capacity is W*M.  The inverse sums a received row's local-expert outputs in ascending
// expert id in FP32 and rounds once.
//
// Kernels:
//   ep_group_kernel       one CTA per (rank, local expert): block scan over the rank's received
//                         rows, 1024 per step (a row is in the list iff one of its k ids is the
//                         expert); writes src_info, the count, the layout ranges, and each row's
//                         slot into the plan's map [W][W*M][k] at the row's first top-k entry
//                         naming the expert;
//   ep_group_count_kernel / ep_group_assign_kernel  the same scan in two passes over
//                         (rank, local expert, 1024-row chunk) CTAs, for capacities of three
//                         chunks or more: per-chunk hits by source rank, then slots from the
//                         hits of earlier chunks;
//   ep_grouped_copy_kernel warp per received row: the row is read once and written to the slot
//                         of each of its local experts;
//   ep_ungroup_kernel     warp per received row (per 512- or 1024-element slice of one, for
//                         small calls): its local experts' output rows, ordered by expert id,
//                         are loaded together and folded in FP32, with 4 to 8 loads per lane in
//                         flight however many local experts the row has;
//   ep_group_from_source_kernel  the fused dispatch's copy: warp per (source token, slice), the
//                         row read once and written to each of its experts' lists.
// Every kernel but the ungroup launches as a programmatic dependent of the kernel before it.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdint>

#include "ep_common.cuh"

namespace ep {
namespace {

// One CTA per (rank, local expert): the rank's received rows are taken 1024 at a time, four per
// thread (rows i0 + q*256 + tid, q = 0..3, so each batch is coalesced), and the rows naming the
// expert get consecutive slots in row order: a row's slot is the count of hits in earlier
// batches of the chunk, then in earlier warps of its batch, then in earlier lanes.
constexpr int kGroupRowsPerThread = 4;

// First top-k entry of a row naming expert ge, or -1.  VEC = k / 4 reads the row as 16-byte
// vectors (rows 16-byte aligned), VEC = 0 loops over the k ids; no early exit, so the loads of
// a row are in flight together.
template <int VEC>
__device__ __forceinline__ int first_entry(const int32_t* ids, int k, int32_t ge)
{
    int jf = -1;
    if constexpr (VEC > 0) {
        int4 v[VEC];
#pragma unroll
        for (int q = 0; q < VEC; ++q) v[q] = __ldg(reinterpret_cast<const int4*>(ids) + q);
#pragma unroll
        for (int q = VEC - 1; q >= 0; --q) {
            if (v[q].w == ge) jf = 4 * q + 3;
            if (v[q].z == ge) jf = 4 * q + 2;
            if (v[q].y == ge) jf = 4 * q + 1;
            if (v[q].x == ge) jf = 4 * q;
        }
    } else {
        for (int j = k - 1; j >= 0; --j)
            if (__ldg(ids + j) == ge) jf = j;
    }
    return jf;
}

static_assert(kScanChunk == 256 * kGroupRowsPerThread, "a scan step is 256 threads x 4 rows");

// The rows i0 + q*256 + tid (q < 4) of rank r: pos = the row's src_pos entry and jfirst = its
// first top-k entry naming global expert ge, or -1 (also for rows i >= n).
template <int VEC>
__device__ __forceinline__ void load_chunk(const GroupArgs& a, int r, int n, int i0, int32_t ge, int tid,
                                           int (&pos)[kGroupRowsPerThread], int (&jfirst)[kGroupRowsPerThread])
{
#pragma unroll
    for (int q = 0; q < kGroupRowsPerThread; ++q) {
        const int i = i0 + q * 256 + tid;
        pos[q] = i < n ? __ldg(a.src_pos + (int64_t)r * a.rows + i) : 0;
    }
#pragma unroll
    for (int q = 0; q < kGroupRowsPerThread; ++q) {
        const int i = i0 + q * 256 + tid;
        jfirst[q] = -1;
        if (i < n) {
            const int32_t* ids;
            if (a.src_idx) {    // fused dispatch: the row's index row is its source's
                const int64_t s = pos[q] / a.rows;
                ids = a.src_idx + (s * a.M + (pos[q] - s * a.rows)) * a.k;
            } else {
                ids = a.recv_idx + ((int64_t)r * a.rows + i) * a.k;
            }
            jfirst[q] = first_entry<VEC>(ids, a.k, ge);
        }
    }
}

// Slots of one chunk's hits, base + the hits before the row in the chunk (rows in order of
// (q, warp, lane)): writes src_info and the row's map entry.  Leaves the chunk's hit count in
// *total; s_warp is the CTA's [4][8] scratch; one __syncthreads inside.
__device__ __forceinline__ void assign_chunk(const GroupArgs& a, int r, int64_t list, int i0, int base,
                                             const int (&pos)[kGroupRowsPerThread],
                                             const int (&jfirst)[kGroupRowsPerThread],
                                             int (*s_warp)[8], int tid, int* total)
{
    constexpr int Q = kGroupRowsPerThread;
    const int lane = tid & 31, warp = tid >> 5;
    unsigned bal[Q];
#pragma unroll
    for (int q = 0; q < Q; ++q) {
        bal[q] = __ballot_sync(0xffffffffu, jfirst[q] >= 0);
        if (lane == 0) s_warp[q][warp] = __popc(bal[q]);
    }
    __syncthreads();
    int run = base, tot = 0;
    int before[Q];
#pragma unroll
    for (int q = 0; q < Q; ++q) {
        before[q] = run;
#pragma unroll
        for (int w = 0; w < 8; ++w) {
            if (w < warp) before[q] += s_warp[q][w];
            run += s_warp[q][w];
            tot += s_warp[q][w];
        }
    }
#pragma unroll
    for (int q = 0; q < Q; ++q) {
        if (jfirst[q] >= 0) {
            const int i = i0 + q * 256 + tid;
            const int slot = before[q] + __popc(bal[q] & lanemask_lt());
            a.src_info[list * a.rows + slot] = (int32_t)(pos[q] % a.rows);
            a.map[((int64_t)r * a.rows + i) * a.k + jfirst[q]] = slot;
        }
    }
    *total = tot;
}

template <int VEC>
__global__ void __launch_bounds__(256) ep_group_kernel(const GroupArgs a)
{
    wait_for_predecessor();   // routing's (or the previous pass's) output
    probe_mark(a.probe, kProbeGroupScan, true);
    constexpr int Q = kGroupRowsPerThread;
    __shared__ int s_warp[Q][8];
    __shared__ int s_src[kMaxRanks];
    __shared__ int s_base;
    const int tid = threadIdx.x;
    const int r = blockIdx.x / a.E;
    const int e = blockIdx.x - r * a.E;
    const int32_t ge = r * a.E + e;
    const int64_t list = (int64_t)r * a.E + e;
    const int n = checked_count(a.recv_count[r], a.rows, a.status);
    if (tid < kMaxRanks) s_src[tid] = 0;
    if (tid == 0) s_base = 0;
    __syncthreads();
    for (int i0 = 0; i0 < n; i0 += kScanChunk) {
        int jfirst[Q], pos[Q];
        load_chunk<VEC>(a, r, n, i0, ge, tid, pos, jfirst);
        int total;
        assign_chunk(a, r, list, i0, s_base, pos, jfirst, s_warp, tid, &total);
#pragma unroll
        for (int q = 0; q < Q; ++q)
            if (jfirst[q] >= 0) atomicAdd(&s_src[pos[q] / a.rows], 1);
        __syncthreads();
        if (tid == 0) s_base += total;
        __syncthreads();
    }
    if (tid == 0) a.count[list] = s_base;
    if (tid < a.W) {
        long long first = 0;
        for (int s = 0; s < tid; ++s) first += s_src[s];
        a.layout_range[list * a.W + tid] = (first << 32) | (long long)s_src[tid];
    }
    allow_dependents();   // the next pass may be scheduled as this one's CTAs finish
    probe_mark(a.probe, kProbeGroupScan, false);
}

// Two-pass scan, pass 1: grid (W*E lists) x (chunk strides); CTA (list, y) takes chunks y,
// y + gridDim.y, ... below the rank's received rows and stores each chunk's hits per source
// rank in scan_cnt[list][c][s].  Nothing else is written, and no CTA waits on another.
template <int VEC>
__global__ void __launch_bounds__(256) ep_group_count_kernel(const GroupArgs a)
{
    wait_for_predecessor();   // routing's (or the previous pass's) output
    probe_mark(a.probe, kProbeGroupScan, true);
    constexpr int Q = kGroupRowsPerThread;
    __shared__ int s_src[kMaxRanks];
    const int tid = threadIdx.x;
    const int r = blockIdx.x / a.E;
    const int e = blockIdx.x - r * a.E;
    const int32_t ge = r * a.E + e;
    const int64_t list = (int64_t)r * a.E + e;
    const int n = checked_count(a.recv_count[r], a.rows, a.status);
    for (int c = blockIdx.y; (int64_t)c * kScanChunk < n; c += gridDim.y) {
        if (tid < kMaxRanks) s_src[tid] = 0;
        __syncthreads();
        int jfirst[Q], pos[Q];
        load_chunk<VEC>(a, r, n, c * kScanChunk, ge, tid, pos, jfirst);
#pragma unroll
        for (int q = 0; q < Q; ++q)
            if (jfirst[q] >= 0) atomicAdd(&s_src[pos[q] / a.rows], 1);
        __syncthreads();
        if (tid < a.W) a.scan_cnt[(list * a.scan_chunks + c) * a.W + tid] = s_src[tid];
        __syncthreads();
    }
    allow_dependents();   // the next pass may be scheduled as this one's CTAs finish
    probe_mark(a.probe, kProbeGroupScan, false);
}

// Pass 2, the same grid: chunk c's base is the sum of scan_cnt over chunks 0..c-1 (all sources),
// and its rows get slots as in the one-pass scan.  The y = 0 CTA of each list also sums every
// chunk's counts per source into the count and the layout ranges (zeros for a rank that
// received nothing).  Pass 1 has finished before any of this runs (stream order).
template <int VEC>
__global__ void __launch_bounds__(256) ep_group_assign_kernel(const GroupArgs a)
{
    wait_for_predecessor();   // routing's (or the previous pass's) output
    probe_mark(a.probe, kProbeGroupScan, true);
    constexpr int Q = kGroupRowsPerThread;
    __shared__ int s_warp[Q][8];
    __shared__ int s_part[8];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int r = blockIdx.x / a.E;
    const int e = blockIdx.x - r * a.E;
    const int32_t ge = r * a.E + e;
    const int64_t list = (int64_t)r * a.E + e;
    const int n = checked_count(a.recv_count[r], a.rows, a.status);
    const int active = (int)(((int64_t)n + kScanChunk - 1) / kScanChunk);
    const int32_t* cnt = a.scan_cnt + list * a.scan_chunks * a.W;
    if (blockIdx.y == 0 && warp == 0) {       // lane s: source rank s (W <= 32)
        int tot = 0;
        if (lane < a.W)
            for (int c = 0; c < active; ++c) tot += cnt[c * a.W + lane];
        int incl = tot;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, d);
            if (lane >= d) incl += v;
        }
        if (lane < a.W) a.layout_range[list * a.W + lane] = ((long long)(incl - tot) << 32) | (long long)tot;
        if (lane == 31) a.count[list] = incl;
    }
    for (int c = blockIdx.y; c < active; c += gridDim.y) {
        int part = 0;
        for (int v = tid; v < c * a.W; v += 256) part += cnt[v];
#pragma unroll
        for (int d = 16; d > 0; d >>= 1) part += __shfl_xor_sync(0xffffffffu, part, d);
        if (lane == 0) s_part[warp] = part;
        int jfirst[Q], pos[Q];
        load_chunk<VEC>(a, r, n, c * kScanChunk, ge, tid, pos, jfirst);
        __syncthreads();
        int base = 0;
#pragma unroll
        for (int w = 0; w < 8; ++w) base += s_part[w];
        int total;
        assign_chunk(a, r, list, c * kScanChunk, base, pos, jfirst, s_warp, tid, &total);
        __syncthreads();                      // s_part and s_warp are reused by the next chunk
    }
    allow_dependents();   // the next pass may be scheduled as this one's CTAs finish
    probe_mark(a.probe, kProbeGroupScan, false);
}

// A received row's top-k entries as the lanes hold them: lane j has entry j and entry j + 32
// (top-k up to 64), each with the row's slot in that expert's list from the plan's map (only
// meaningful where the entry is the row's first naming a local expert).  Loading them is two
// independent loads per lane, so a warp can fetch the next row's entries before it copies or
// folds the current one; resolving them is shuffles only.
struct RowEntries {
    int id0, id1, slot0, slot1;
};

__device__ __forceinline__ RowEntries load_entries(const GroupArgs& a, int64_t u, int lane)
{
    const int32_t* ids = a.recv_idx + u * a.k;
    const int32_t* mp = a.map + u * a.k;
    RowEntries e;
    e.id0 = lane < a.k ? __ldg(ids + lane) : -1;
    e.id1 = lane + 32 < a.k ? __ldg(ids + lane + 32) : -1;
    e.slot0 = lane < a.k ? __ldg(mp + lane) : 0;
    e.slot1 = lane + 32 < a.k ? __ldg(mp + lane + 32) : 0;
    return e;
}

// The packed rows (list * rows + slot) entries j and j + 32 feed, -1 where the entry names no
// local expert of rank r or repeats an earlier entry of the row (a row joins an expert's list
// once, at its first top-k entry naming the expert).
__device__ __forceinline__ void resolve_entries(const GroupArgs& a, int r, const RowEntries& e, int lane,
                                                int64_t& dest0, int64_t& dest1)
{
    const int lo = r * a.E, hi = lo + a.E;
    bool ok0 = lane < a.k && e.id0 >= lo && e.id0 < hi;
    bool ok1 = lane + 32 < a.k && e.id1 >= lo && e.id1 < hi;
    if (a.k <= 32) {                                       // one warp-wide match (every lane calls it)
        const unsigned same = __match_any_sync(0xffffffffu, e.id0);
        ok0 = ok0 && !(same & lanemask_lt());
    } else {
        for (int jj = 0; jj < a.k; ++jj) {                 // warp-uniform loop
            const int x = __shfl_sync(0xffffffffu, jj < 32 ? e.id0 : e.id1, jj & 31);
            if (jj < lane && x == e.id0) ok0 = false;
            if (jj < lane + 32 && x == e.id1) ok1 = false;
        }
    }
    if (ok0) ok0 = EP_IN_BOUNDS(e.slot0 >= 0 && e.slot0 < a.rows, a.status);
    if (ok1) ok1 = EP_IN_BOUNDS(e.slot1 >= 0 && e.slot1 < a.rows, a.status);
    dest0 = ok0 ? ((int64_t)r * a.E + (e.id0 - lo)) * a.rows + e.slot0 : -1;
    dest1 = ok1 ? ((int64_t)r * a.E + (e.id1 - lo)) * a.rows + e.slot1 : -1;
}

// Received rows only, flattened across ranks: row g is row g - off[r] of rank r.
__device__ __forceinline__ int64_t received_row(const int* off, int W, int64_t rows, int g)
{
    const int r = rank_of_token(off, W, g);
    return (int64_t)r * rows + (g - off[r]);
}

// Rows are split over warps as the payload scatter's units are (WorkSplit): the last rounds come
// from the plan's grouping queue (a.work.q), since a row costs one read and one write per local
// expert.  The unit count, the rows received by all ranks, is known on the device only.
__global__ void __launch_bounds__(kCopyThreads) ep_grouped_copy_kernel(const GroupArgs a)
{
    wait_for_predecessor();   // routing's (or the previous pass's) output
    probe_mark(a.probe, kProbeGroupCopy, true);
    __shared__ int s_off[kMaxRanks + 1];
    if (threadIdx.x == 0) {
        int run = 0;
        for (int r = 0; r < a.W; ++r) {
            s_off[r] = run;
            run += checked_count(a.recv_count[r], a.rows, a.status);
        }
        s_off[a.W] = run;
    }
    __syncthreads();
    const int lane = threadIdx.x & 31;
    const WorkSplit ws = make_work_split(a.work.q, s_off[a.W], (int64_t)gridDim.x * (kCopyThreads / 32));
    const uint32_t total = ws.units;
    const int nvec = (int)(a.row_bytes >> 4);
    uint32_t g_next = work_first(ws);
    RowEntries next{};
    if (g_next < total) next = load_entries(a, received_row(s_off, a.W, a.rows, (int)g_next), lane);
    while (g_next < total) {
        const uint32_t g = g_next;
        const int r = rank_of_token(s_off, a.W, (int)g);
        const int64_t u = (int64_t)r * a.rows + ((int)g - s_off[r]);
        const RowEntries cur = next;
        g_next = work_next(ws, g, lane);
        if (g_next < total)                                // lands while this row is copied
            next = load_entries(a, received_row(s_off, a.W, a.rows, (int)g_next), lane);
        int64_t dest0, dest1;
        resolve_entries(a, r, cur, lane, dest0, dest1);
        const uint8_t* src = a.recv_x + u * a.row_bytes;
        for (int half = 0; half < 2; ++half) {             // entries j < 32, then j >= 32
            const int64_t dest = half ? dest1 : dest0;
            const unsigned has = __ballot_sync(0xffffffffu, dest >= 0);
            if (!has) continue;
            for (int v0 = 0; v0 < nvec; v0 += 32 * 4) {
                uint4 buf[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int v = v0 + q * 32 + lane;
                    if (v < nvec) buf[q] = ld_stream_v4(src + (int64_t)v * 16);
                }
                for (unsigned m = has; m; m &= m - 1) {
                    const int64_t row = __shfl_sync(0xffffffffu, dest, __ffs(m) - 1);
                    uint8_t* dst = a.packed_x + row * a.row_bytes;
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int v = v0 + q * 32 + lane;
                        if (v < nvec) st_v4(dst + (int64_t)v * 16, buf[q]);
                    }
                }
            }
        }
    }
    work_retire(ws);
    probe_mark(a.probe, kProbeGroupCopy, false);
}

template <bool FP16>
__device__ __forceinline__ void add8(float (&acc)[8], const uint4& v)
{
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float lo, hi;
        if constexpr (FP16) {
            const __half2 h = *reinterpret_cast<const __half2*>(&w[i]);
            lo = __low2float(h);
            hi = __high2float(h);
        } else {
            lo = __uint_as_float(w[i] << 16);
            hi = __uint_as_float(w[i] & 0xFFFF0000u);
        }
        acc[2 * i] = __fadd_rn(acc[2 * i], lo);
        acc[2 * i + 1] = __fadd_rn(acc[2 * i + 1], hi);
    }
}

template <bool FP16>
__device__ __forceinline__ uint4 pack8(const float (&acc)[8])
{
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        if constexpr (FP16) {
            const __half2 h = __floats2half2_rn(acc[2 * i], acc[2 * i + 1]);
            w[i] = *reinterpret_cast<const uint32_t*>(&h);
        } else {
            const __nv_bfloat162 b = __floats2bfloat162_rn(acc[2 * i], acc[2 * i + 1]);
            w[i] = *reinterpret_cast<const uint32_t*>(&b);
        }
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// Rolling fold of nd <= R rows of hv 16-byte vectors into dst: each lane keeps the next D columns
// of every row in flight, R * D = 4 loads for rows of up to four local experts and 8 above, so a
// row with few local experts still keeps as many bytes outstanding as one with many.  Each
// column's rows are added in ascending order.  (Eight columns ahead for a single-expert row needs
// about 200 registers; four fit two 8-warp CTAs per SM, which hides more latency.)
// Entries are found by their rank among the row's valid entries (rank0 / rank1 of lane j belong
// to top-k entries j and j + 32, whose packed rows are dest0 / dest1).
// The fold covers vectors [v0, v0 + hv) of rows of stride rs vectors (a slice of each row).
template <bool FP16, int R, int D>
__device__ __forceinline__ void fold_rd(const uint4* y4, int64_t dest0, int64_t dest1, int rank0, int rank1,
                                        int nd, int64_t rs, int v0, int hv, uint4* dst, int lane)
{
    const uint4* rp[R];
#pragma unroll
    for (int q = 0; q < R; ++q) {
        const unsigned m0 = __ballot_sync(0xffffffffu, dest0 >= 0 && rank0 == q);
        const unsigned m1 = __ballot_sync(0xffffffffu, dest1 >= 0 && rank1 == q);
        const int64_t row = m0 ? __shfl_sync(0xffffffffu, dest0, __ffs(m0) - 1)
                               : __shfl_sync(0xffffffffu, dest1, m1 ? __ffs(m1) - 1 : 0);
        rp[q] = y4 + row * rs + v0;
    }
    uint4 b[R][D];
#pragma unroll
    for (int t = 0; t < D; ++t)
#pragma unroll
        for (int q = 0; q < R; ++q)
            if (q < nd && lane + 32 * t < hv) b[q][t] = ld_stream_v4(rp[q] + lane + 32 * t);
    for (int vb = 0; vb < hv; vb += 32 * D) {              // warp-uniform bounds
#pragma unroll
        for (int t = 0; t < D; ++t) {
            const int vc = vb + 32 * t + lane, vn = vc + 32 * D;
            float acc[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) acc[q] = 0.0f;
#pragma unroll
            for (int q = 0; q < R; ++q) {
                if (q < nd) {
                    const uint4 x = b[q][t];
                    if (vn < hv) b[q][t] = ld_stream_v4(rp[q] + vn);
                    if (vn + 32 * D < hv) prefetch_l2(rp[q] + vn + 32 * D);
                    if (vc < hv) add8<FP16>(acc, x);
                }
            }
            if (vc < hv) st_v4(dst + vc, pack8<FP16>(acc));
        }
    }
}

template <bool FP16, bool WIDE>
__global__ void __launch_bounds__(kCopyThreads, 2) ep_ungroup_kernel(const GroupArgs a)
{
    probe_mark(a.probe, kProbeUngroup, true);
    __shared__ int s_off[kMaxRanks + 1];
    if (threadIdx.x == 0) {
        int run = 0;
        for (int r = 0; r < a.W; ++r) {
            s_off[r] = run;
            run += checked_count(a.recv_count[r], a.rows, a.status);
        }
        s_off[a.W] = run;
    }
    __syncthreads();
    const int lane = threadIdx.x & 31;
    const int nwarps = gridDim.x * (kCopyThreads / 32);
    // work units: (received row, slice of chunk_bytes), one slice per row for large calls (the
    // host slices only calls of a few thousand rows, so units stay below 2^31 either way)
    const int chunks = a.chunks;
    const int units = s_off[a.W] * chunks;
    const int rs = (int)(a.row_bytes >> 4);       // 16-byte vectors of a 16-bit row
    const int cv = a.chunk_bytes >> 4;            // ... of a slice
    const uint4* y4 = reinterpret_cast<const uint4*>(a.packed_y);
    auto row_of = [&](int unit) { return chunks == 1 ? unit : unit / chunks; };
    int g = blockIdx.x * (kCopyThreads / 32) + (threadIdx.x >> 5);
    RowEntries next{};
    if (g < units) next = load_entries(a, received_row(s_off, a.W, a.rows, row_of(g)), lane);
    // (g + nwarps is formed only below units, so it cannot overflow)
    for (; g < units; g = g < units - nwarps ? g + nwarps : units) {
        const int gr = row_of(g);
        const int v0 = (g - gr * chunks) * cv;
        const int hv = min(cv, rs - v0);
        const int r = rank_of_token(s_off, a.W, gr);
        const int64_t u = (int64_t)r * a.rows + (gr - s_off[r]);
        const RowEntries cur = next;
        if (g < units - nwarps)                            // lands while this unit is folded
            next = load_entries(a, received_row(s_off, a.W, a.rows, row_of(g + nwarps)), lane);
        uint4* dst = reinterpret_cast<uint4*>(a.out + u * a.row_bytes) + v0;
        // the row's local experts in ascending id: lane j holds entry j (and j + 32 for k > 32)
        int64_t dest0, dest1;
        resolve_entries(a, r, cur, lane, dest0, dest1);
        const int e0 = dest0 >= 0 ? cur.id0 : 0x7FFFFFFF;
        const int e1 = dest1 >= 0 ? cur.id1 : 0x7FFFFFFF;
        const int nd = __popc(__ballot_sync(0xffffffffu, dest0 >= 0)) +
                       __popc(__ballot_sync(0xffffffffu, dest1 >= 0));
        // rank of each entry among the valid ones (their ids are distinct): for up to 32 entries
        // and 64 local experts, a popcount of the row's local-expert mask below the entry's expert
        int rank0 = 0, rank1 = 0;
        if (a.k <= 32 && a.E <= 64) {
            const int le = dest0 >= 0 ? e0 - r * a.E : 0;
            const unsigned long long bit = dest0 >= 0 ? 1ull << le : 0ull;
            const unsigned long long mask =
                (unsigned long long)__reduce_or_sync(0xffffffffu, (unsigned)bit) |
                (unsigned long long)__reduce_or_sync(0xffffffffu, (unsigned)(bit >> 32)) << 32;
            rank0 = __popcll(mask & (bit - 1ull));
        } else {
            for (int j = 0; j < a.k; ++j) {
                const int ej = __shfl_sync(0xffffffffu, j < 32 ? e0 : e1, j & 31);
                rank0 += ej < e0;
                rank1 += ej < e1;
            }
        }
        if (!WIDE || nd <= 8) {
            // the rows in ascending expert order, once per received row; then a rolling fold:
            // row d's next columns are requested as soon as its current one is taken
            if (nd <= 1)
                fold_rd<FP16, 1, 4>(y4, dest0, dest1, rank0, rank1, nd, rs, v0, hv, dst, lane);
            else if (nd == 2)
                fold_rd<FP16, 2, 2>(y4, dest0, dest1, rank0, rank1, nd, rs, v0, hv, dst, lane);
            else if (nd <= 4)
                fold_rd<FP16, 4, 1>(y4, dest0, dest1, rank0, rank1, nd, rs, v0, hv, dst, lane);
            else
                fold_rd<FP16, 8, 1>(y4, dest0, dest1, rank0, rank1, nd, rs, v0, hv, dst, lane);
            continue;
        }
        if constexpr (WIDE) {
            for (int vb = 0; vb < hv; vb += 32) {              // more than 8 local experts
                const int v = vb + lane;
                float acc[8];
#pragma unroll
                for (int q = 0; q < 8; ++q) acc[q] = 0.0f;
                for (int d0 = 0; d0 < nd; d0 += 8) {
                    uint4 b[8];
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        // the entry of rank d0+q (uniform across the warp)
                        const int want = d0 + q;
                        const unsigned m0 = __ballot_sync(0xffffffffu, dest0 >= 0 && rank0 == want);
                        const unsigned m1 = __ballot_sync(0xffffffffu, dest1 >= 0 && rank1 == want);
                        int64_t row = -1;
                        if (m0) row = __shfl_sync(0xffffffffu, dest0, __ffs(m0) - 1);
                        else if (m1) row = __shfl_sync(0xffffffffu, dest1, __ffs(m1) - 1);
                        if (row >= 0 && v < hv) b[q] = ld_stream_v4(y4 + row * rs + v0 + v);
                        if (row < 0) b[q] = make_uint4(0, 0, 0, 0);
                    }
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        if (d0 + q < nd) add8<FP16>(acc, b[q]);
                }
                if (v < hv) st_v4(dst + v, pack8<FP16>(acc));
            }
        }
    }
    probe_mark(a.probe, kProbeUngroup, false);
}

// Fused dispatch into the grouped view: warp per source token.  Lane j owns top-k slot j: when
// it is the row's first slot naming its expert e (rank r = e / E), its packed row is
// (r*E + e - r*E) * rows + slot, the slot being the one ep_group_kernel recorded for the
// token's receive row on rank r (found in the forward map).  The source row is read once and
// written to every such packed row; the token's index / weight / scale rows go to its receive
// rows as in ep_dispatch.  The 2-D payload rows are not written.
__global__ void __launch_bounds__(kCopyThreads) ep_group_from_source_kernel(const GroupArgs a)
{
    wait_for_predecessor();   // routing's (or the previous pass's) output
    probe_mark(a.probe, kProbeGroupCopy, true);
    __shared__ int s_off[kMaxRanks + 1];
    if (threadIdx.x <= a.W) s_off[threadIdx.x] = a.tok_off[threadIdx.x];
    if (a.scan_done && blockIdx.x == 0) {
        // routing numbered the lists: the counts and per-source layout ranges follow from each
        // list's prefix at every source's first token (and at the end of the tokens)
        const int n_exp = a.W * a.E;
        for (int i = threadIdx.x; i < n_exp * a.W; i += kCopyThreads) {
            const int e = i / a.W, sb = i - e * a.W;
            const int first = a.bnd[(int64_t)sb * n_exp + e];
            const int next = a.bnd[(int64_t)(sb + 1) * n_exp + e];
            a.layout_range[i] = ((long long)first << 32) | (long long)(next - first);
        }
        for (int e = threadIdx.x; e < n_exp; e += kCopyThreads) a.count[e] = a.bnd[(int64_t)a.W * n_exp + e];
    }
    __syncthreads();
    const int lane = threadIdx.x & 31;
    const float inv_e = __frcp_rn((float)a.E);
    const WorkSplit& ws = a.work;
    for (uint32_t u = work_first(ws); u < ws.units; u = work_next(ws, u, lane)) {
        const int g = (int)(u / (uint32_t)a.chunks);
        const int c = (int)(u - (uint32_t)g * (uint32_t)a.chunks);
        const int64_t off = (int64_t)c * a.chunk_bytes;      // this unit's slice of the row
        const int nvec = (int)(min((int64_t)a.chunk_bytes, a.row_bytes - off) >> 4);
        const int s = rank_of_token(s_off, a.W, g);
        const int64_t tok = (int64_t)s * a.M + (g - s_off[s]);
        const int32_t* ids = a.src_idx + tok * a.k;
        const int fw = checked_fwd(lane < a.F ? __ldg(a.fwd + tok * a.F + lane) : -1,   // receive rows,
                                   (int64_t)a.W * a.rows, a.status);                // by rank
        const int nd = __popc(__ballot_sync(0xffffffffu, fw >= 0));
        // the token's destination ranks, one bit each (lane d holds the d-th receive row)
        const unsigned dranks = __reduce_or_sync(0xffffffffu, fw >= 0 ? 1u << (fw / (int)a.rows) : 0u);
        // metadata rows to the receive rows, as in ep_dispatch (with the first slice)
        for (int d = 0; d < (c == 0 ? nd : 0); ++d) {
            const int64_t row = __shfl_sync(0xffffffffu, fw, d);
            for (int e = lane; e < a.k; e += 32) {
                a.recv_idx_out[row * a.k + e] = __ldg(ids + e);
                if (a.w) a.recv_w_out[row * a.k + e] = __ldg(a.w + tok * a.k + e);
            }
            for (int e = lane; e < a.sd; e += 32)
                a.recv_scales_out[row * a.sd + e] = __ldg(a.scales + tok * a.sd + e);
        }
        const uint8_t* src = a.x + tok * a.row_bytes + off;
        // the slice's first step of source vectors is read while the destinations are found
        uint4 buf[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int v = q * 32 + lane;
            if (v < nvec) buf[q] = ld_stream_v4(src + (int64_t)v * 16);
        }
        for (int j0 = 0; j0 < a.k; j0 += 32) {
            const int j = j0 + lane;
            int64_t dest = -1;
            int e = -1, r = -1;
            if (j < a.k) e = __ldg(ids + j);
            bool first = e >= 0 && e < a.W * a.E;
            if (j0 == 0) {                                 // slots 0..31: the lanes compare
                const unsigned same = __match_any_sync(0xffffffffu, e);   // every lane takes part
                first = first && !(same & lanemask_lt());
            } else {
                for (int jj = 0; jj < j && first; ++jj) first = __ldg(ids + jj) != e;
            }
            if (first) r = expert_rank(e, a.E, inv_e);
            // the token's receive row on rank r: the forward map lists the token's destination
            // ranks in ascending order, so it is entry popc(ranks below r) (every lane shuffles)
            const int pos = __popc(dranks & ((1u << (r & 31)) - 1u));
            const int64_t row_r = __shfl_sync(0xffffffffu, fw, pos & 31);
            const int64_t rrow = r >= 0 && ((dranks >> (r & 31)) & 1u) ? row_r : -1;
            if (rrow >= 0) {
                const int slot = a.map[rrow * a.k + j];
                if (EP_IN_BOUNDS(slot >= 0 && slot < a.rows, a.status))
                    dest = (int64_t)e * a.rows + slot;     // list e = r*E + local expert
            }
            const unsigned has = __ballot_sync(0xffffffffu, dest >= 0);
            if (!has) continue;
            for (int v0 = 0; v0 < nvec; v0 += 32 * 4) {
                if (v0 > 0 || j0 > 0) {                    // (buf holds the first step otherwise)
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int v = v0 + q * 32 + lane;
                        if (v < nvec) buf[q] = ld_stream_v4(src + (int64_t)v * 16);
                    }
                }
                for (unsigned m = has; m; m &= m - 1) {
                    const int64_t prow = __shfl_sync(0xffffffffu, dest, __ffs(m) - 1);
                    uint8_t* dst = a.packed_x + prow * a.row_bytes + off;
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int v = v0 + q * 32 + lane;
                        if (v < nvec) st_v4(dst + (int64_t)v * 16, buf[q]);
                    }
                }
            }
        }
    }
    work_retire(ws);
    probe_mark(a.probe, kProbeGroupCopy, false);
}

int grid_of(const void* kernel, int64_t warps, int num_sms)
{
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kCopyThreads, 0) != cudaSuccess ||
        per_sm < 1)
        per_sm = 1;
    const int64_t need = (warps + kCopyThreads / 32 - 1) / (kCopyThreads / 32);
    const int64_t cap = (int64_t)per_sm * num_sms;
    return (int)(need < cap ? need : cap);
}

}  // namespace

// The grouping passes launch as dependents (launch_dependent) of the kernel before each: the
// scan of the routing kernel or of the dispatch's scatter, the assignment pass of the count
// pass, the copy of the scan.
template <int VEC>
static cudaError_t launch_group_scan_t(const GroupArgs& a, int num_sms, cudaStream_t stream)
{
    if (!a.scan_cnt) return launch_dependent(ep_group_kernel<VEC>, dim3(a.W * a.E), dim3(256), 0, stream, a);
    // about 16 CTAs per SM in all; a CTA takes every gridDim.y-th chunk of its list
    const int per = 16 * num_sms / (a.W * a.E);
    int gy = per > 1 ? per : 1;
    if (gy > a.scan_chunks) gy = a.scan_chunks;
    if (gy > 65535) gy = 65535;
    const dim3 grid(a.W * a.E, gy);
    cudaError_t e = launch_dependent(ep_group_count_kernel<VEC>, grid, dim3(256), 0, stream, a);
    if (e != cudaSuccess) return e;
    return launch_dependent(ep_group_assign_kernel<VEC>, grid, dim3(256), 0, stream, a);
}

// compiled index-row widths: top-k 4, 8 (the pages' specialised case), 16; others loop
static cudaError_t launch_group_scan(const GroupArgs& a, int num_sms, cudaStream_t stream)
{
    if (!a.vec16 || (a.k != 4 && a.k != 8 && a.k != 16)) return launch_group_scan_t<0>(a, num_sms, stream);
    if (a.k == 4) return launch_group_scan_t<1>(a, num_sms, stream);
    if (a.k == 8) return launch_group_scan_t<2>(a, num_sms, stream);
    return launch_group_scan_t<4>(a, num_sms, stream);
}

cudaError_t launch_group_from_source(const GroupArgs& a, int num_sms, cudaStream_t stream)
{
    if (!a.scan_done) {
        cudaError_t e = launch_group_scan(a, num_sms, stream);
        if (e != cudaSuccess || a.N == 0) return e;            // an empty call's scan wrote the counts
    }
    const int64_t units = (int64_t)a.N * a.chunks;
    int grid = grid_of((const void*)ep_group_from_source_kernel, units, num_sms);
    if (grid < 1) grid = 1;                                // CTA 0 writes the counts of an empty call
    GroupArgs b = a;
    b.work = make_work_split(a.work.q, units, (int64_t)grid * (kCopyThreads / 32));
    return launch_dependent(ep_group_from_source_kernel, dim3(grid), dim3(kCopyThreads), 0, stream, b);
}

cudaError_t launch_group(const GroupArgs& a, int num_sms, cudaStream_t stream)
{
    cudaError_t e = launch_group_scan(a, num_sms, stream);
    if (e != cudaSuccess) return e;
    const int64_t units = (int64_t)a.W * a.rows;
    return launch_dependent(ep_grouped_copy_kernel, dim3(grid_of((const void*)ep_grouped_copy_kernel, units, num_sms)),
                            dim3(kCopyThreads), 0, stream, a);
}

template <bool FP16, bool WIDE>
void launch_ungroup_t(const GroupArgs& a, int num_sms, cudaStream_t stream)
{
    // Rows the call can have received (each token has at most F); calls with fewer than four such
    // rows per resident warp split rows into 1024-element slices, and into 512-element ones when
    // that still leaves fewer than two units per warp, as the combine does.
    const void* kernel = (const void*)ep_ungroup_kernel<FP16, WIDE>;
    const int64_t rows = min((int64_t)a.W * a.rows, (int64_t)a.N * a.F);
    const int64_t warps = (int64_t)grid_of(kernel, INT64_MAX / 2, num_sms) * (kCopyThreads / 32);
    const int rs = (int)(a.row_bytes >> 4);
    int cv = rs;
    if (rows < 4 * warps && rs > 128) {
        cv = 128;
        if (rows * ((rs + cv - 1) / cv) < 2 * warps) cv = 64;
    }
    GroupArgs b = a;
    b.chunk_bytes = cv * 16;
    b.chunks = (rs + cv - 1) / cv;
    int grid = grid_of(kernel, rows * b.chunks, num_sms);
    if (grid < 1) grid = 1;
    ep_ungroup_kernel<FP16, WIDE><<<grid, kCopyThreads, 0, stream>>>(b);
}

cudaError_t launch_ungroup(const GroupArgs& a, bool fp16, int num_sms, cudaStream_t stream)
{
    // a row has at most min(k, E) local experts; the >8 path is only compiled in when needed
    const bool wide = (a.k < a.E ? a.k : a.E) > 8;
    if (fp16)
        wide ? launch_ungroup_t<true, true>(a, num_sms, stream) : launch_ungroup_t<true, false>(a, num_sms, stream);
    else
        wide ? launch_ungroup_t<false, true>(a, num_sms, stream) : launch_ungroup_t<false, false>(a, num_sms, stream);
    return cudaGetLastError();
}

}  // namespace ep

// ep_combine.cu -- Combine gather-reduce.
//
// For every source token, read the expert-output rows of the ranks it was dispatched to
// (forward map, ascending destination rank), add them in FP32 starting from +0.0f in that
// fixed order, and round to nearest even into BF16 / FP16 (MORI-EP gfx1201 PR, Combine bullet:
// the home rank accumulates its own and the received contributions in FP32 and converts once
// at the end; FP32 weight rows travel and are summed on their own).  Routing weights are not
// applied.  The fixed order makes the result independent of the launch shape.
//
// HBM-bound, and bound by how many bytes each SM keeps in flight: at the loaded HBM latency
// of this part (~2.3 us) an SM needs ~100 KB of reads outstanding to stream at full rate.  A
// warp owns one work unit (a token, or a 512/1024-element slice of it for small calls) and its
// lanes own 16-byte columns.  The token's rows are gathered in a rolling fashion: each row's
// load of a lane's column two steps ahead is issued as soon as its current column has been
// added, so a lane keeps two loads per row (2 nd of them) in flight without a gap.  The
// column's rows are added in ascending rank order in FP32 registers and the sum leaves as one
// packed BF16x8 / FP16x8 16-byte store.  Two CTAs of 6 warps per SM hold the 2 x 8 row
// vectors per lane in registers without spills; 18 warps at one load per row in flight kept
// fewer bytes outstanding and ran 3 % slower.  The next unit's forward-map row is loaded
// while the current one is folded.
//
// (A TMA variant that staged row slices through shared memory with 1-D bulk copies was
// measured slower: on this part one CTA's bulk copies each take ~0.3 us, so gathering a
// token's 3.5 KB row slices that way cannot keep enough bytes in flight.)
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "ep_common.cuh"

namespace ep {
namespace {

#ifndef EP_COMBINE_CTAS_PER_SM
#define EP_COMBINE_CTAS_PER_SM 2   // ~160 registers per thread: the fold loop runs without spills
#endif
#ifndef EP_COMBINE_THREADS
#define EP_COMBINE_THREADS 192   // 6 warps: 2 CTAs fill the register file at ~160 registers
#endif
constexpr int kCombThreads = EP_COMBINE_THREADS;
#ifndef EP_COMBINE_DEPTH
#define EP_COMBINE_DEPTH 2
#endif
constexpr int kDepth = EP_COMBINE_DEPTH;   // columns per row in flight per lane

template <bool FP16>
__device__ __forceinline__ void add_vec(float (&acc)[8], const uint4& v)
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
            // BF16 -> FP32 is exact: the BF16 bits are the top half of the FP32 bits
            lo = __uint_as_float(w[i] << 16);
            hi = __uint_as_float(w[i] & 0xFFFF0000u);
        }
        acc[2 * i] = __fadd_rn(acc[2 * i], lo);
        acc[2 * i + 1] = __fadd_rn(acc[2 * i + 1], hi);
    }
}

template <bool FP16>
__device__ __forceinline__ uint4 pack_vec(const float (&acc)[8])
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

// Fold one unit of nd <= 8 rows.  Lane d of `src` holds the unit's d-th row; `ro` keeps the
// rows as 16-byte-vector offsets from eo4 (32 bits: ep_plan_create rejects shapes whose expert
// outputs [W][W*M][H] reach 64 GiB, 2^32 vectors).  Each lane
// owns columns lane, lane+32, ...; row d's load of the next column is issued as soon as its
// current column has been taken, so every lane keeps nd loads in flight without a gap.  The
// column's rows are added in ascending order, one FP32 add each, then packed and stored.
template <bool FP16>
__device__ __forceinline__ void fold_rows(const uint4* __restrict__ eo4, int src, int64_t hv, int v0,
                                          int nd, int nv, uint4* dst4, int lane)
{
    uint32_t ro[8];
#pragma unroll
    for (int d = 0; d < 8; ++d)
        ro[d] = (uint32_t)((int64_t)__shfl_sync(0xffffffffu, src, d) * hv + v0);
    uint4 b[8][kDepth];
#pragma unroll
    for (int t = 0; t < kDepth; ++t)
#pragma unroll
        for (int d = 0; d < 8; ++d)
            if (d < nd && lane + 32 * t < nv) b[d][t] = ld_stream_v4(eo4 + ro[d] + lane + 32 * t);
    for (int vb = 0; vb < nv; vb += 32 * kDepth) {        // warp-uniform bounds
#pragma unroll
        for (int t = 0; t < kDepth; ++t) {
            const int vcur = vb + 32 * t + lane;
            const int vnext = vcur + 32 * kDepth;
            float acc[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) acc[q] = 0.0f;
#pragma unroll
            for (int d = 0; d < 8; ++d) {
                if (d < nd) {
                    const uint4 x = b[d][t];
                    if (vnext < nv) b[d][t] = ld_stream_v4(eo4 + ro[d] + vnext);
                    if (vnext + 32 * kDepth < nv) prefetch_l2(eo4 + ro[d] + vnext + 32 * kDepth);
                    if (vnext + 64 * kDepth < nv) prefetch_l2(eo4 + ro[d] + vnext + 64 * kDepth);
                    if (vcur < nv) add_vec<FP16>(acc, x);
                }
            }
            if (vcur < nv) st_v4(dst4 + vcur, pack_vec<FP16>(acc));
        }
    }
}

// More than 8 rows (W > 8 and k > 8): rows in ascending batches of 8, one column per lane.
template <bool FP16>
__device__ __forceinline__ void fold_wide(const uint16_t* eo, int64_t H, int src, int nd,
                                          int64_t v0_elem, int nv, uint16_t* dst, int lane)
{
    for (int vb = 0; vb < nv; vb += 32) {
        const int v = vb + lane;
        const bool act = v < nv;
        float acc[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) acc[q] = 0.0f;
        for (int d0 = 0; d0 < nd; d0 += 8) {
            uint4 buf[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const int64_t row = __shfl_sync(0xffffffffu, src, (d0 + q) & 31);
                if (act && d0 + q < nd) buf[q] = ld_stream_v4(eo + row * H + v0_elem + (int64_t)v * 8);
            }
#pragma unroll
            for (int q = 0; q < 8; ++q)
                if (act && d0 + q < nd) add_vec<FP16>(acc, buf[q]);
        }
        if (act) st_v4(dst + (int64_t)v * 8, pack_vec<FP16>(acc));
    }
}

// Forward-map entry of this lane for work unit u (the lane-th row of the unit's token).
__device__ __forceinline__ int unit_src(const CombineArgs& a, const int* off, uint32_t u, int lane)
{
    if (u >= (uint32_t)a.N * (uint32_t)a.chunks) return -1;
    const int g = (int)(u / (uint32_t)a.chunks);
    const int s = rank_of_token(off, a.W, g);
    const int64_t tok = (int64_t)s * a.M + (g - off[s]);
    return lane < a.F ? __ldg(a.fwd + tok * a.F + lane) : -1;
}

template <bool FP16, bool WIDE>
__global__ void __launch_bounds__(kCombThreads, EP_COMBINE_CTAS_PER_SM) ep_combine_kernel(const CombineArgs a)
{
    __shared__ int s_off[kMaxRanks + 1];
    if (threadIdx.x <= a.W) s_off[threadIdx.x] = a.tok_off[threadIdx.x];
    probe_mark(a.probe, kProbeCombine, true);
    __syncthreads();

    const int lane = threadIdx.x & 31;
    // units = N * chunks < 2^31 (checked by the host), so unit indices are 32-bit
    const uint32_t units = (uint32_t)a.N * (uint32_t)a.chunks;
    const uint32_t step = gridDim.x * (kCombThreads / 32);
    uint32_t u = blockIdx.x * (kCombThreads / 32) + (threadIdx.x >> 5);
    int src = unit_src(a, s_off, u, lane);
    for (; u < units; u += step) {
        const int src_next = unit_src(a, s_off, u + step, lane);   // lands while this unit folds
        src = checked_fwd(src, (int64_t)a.W * a.W * a.M, a.status);
        const int nd = __popc(__ballot_sync(0xffffffffu, src >= 0));
        {
            const int g = (int)(u / (uint32_t)a.chunks);
            const int c = (int)(u - (uint32_t)g * (uint32_t)a.chunks);
            const int s = rank_of_token(s_off, a.W, g);
            const int64_t tok = (int64_t)s * a.M + (g - s_off[s]);
            const int hv = (int)(a.H >> 3);
            const int v0 = c * a.chunk_vecs;
            const int nv = min(a.chunk_vecs, hv - v0);
            if (!WIDE || nd <= 8)
                fold_rows<FP16>(reinterpret_cast<const uint4*>(a.eo), src, hv, v0, nd, nv,
                                reinterpret_cast<uint4*>(a.out) + tok * hv + v0, lane);  // nd 0: +0
            else
                fold_wide<FP16>(a.eo, a.H, src, nd, (int64_t)v0 * 8, nv,
                                a.out + tok * a.H + (int64_t)v0 * 8, lane);
        }
        if (a.w_in != nullptr && a.out_w != nullptr && u % (uint32_t)a.chunks == 0) {
            const int g = (int)(u / (uint32_t)a.chunks);
            const int s = rank_of_token(s_off, a.W, g);
            const int64_t tok = (int64_t)s * a.M + (g - s_off[s]);
            for (int e0 = 0; e0 < a.k; e0 += 32) {
                const int e = e0 + lane;
                float acc = 0.0f;
                for (int d = 0; d < nd; ++d) {
                    const int64_t row = __shfl_sync(0xffffffffu, src, d);
                    if (e < a.k) acc = __fadd_rn(acc, __ldg(a.w_in + row * a.k + e));
                }
                if (e < a.k) a.out_w[tok * a.k + e] = acc;
            }
        }
        src = src_next;
    }
    probe_mark(a.probe, kProbeCombine, false);
}

template <bool FP16, bool WIDE>
cudaError_t launch_t(const CombineArgs& a, int num_sms, cudaStream_t stream)
{
    const int64_t units = (int64_t)a.N * a.chunks;
    if (units == 0) return cudaSuccess;
    int per_sm = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
        &per_sm, ep_combine_kernel<FP16, WIDE>, kCombThreads, 0);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) per_sm = 1;
    const int64_t need = (units + kCombThreads / 32 - 1) / (kCombThreads / 32);
    const int64_t cap = (int64_t)per_sm * num_sms;
    const int grid = (int)(need < cap ? need : cap);
    ep_combine_kernel<FP16, WIDE><<<grid, kCombThreads, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace

void combine_geometry(CombineArgs& a, int variant, int num_sms)
{
    const int hv = (int)(a.H >> 3);
    int cv = hv;                                           // whole rows
    if (variant == EP_VARIANT_TILED_512) cv = 64;
    if (variant == EP_VARIANT_TILED_1024) cv = 128;
    if (variant == EP_VARIANT_AUTO) {
        // Calls with fewer than four whole rows per resident warp split rows into 1024-element
        // slices, and into 512-element ones when that still leaves fewer than two units per
        // warp, as the pages' small-batch policy does.
        const int64_t warps = (int64_t)num_sms * EP_COMBINE_CTAS_PER_SM * (kCombThreads / 32);
        if ((int64_t)a.N < 4 * warps && hv > 128) {
            cv = 128;
            if ((int64_t)a.N * ((hv + cv - 1) / cv) < 2 * warps) cv = 64;
        }
    }
    if (cv > hv) cv = hv;
    a.chunks = (hv + cv - 1) / cv;
    a.chunk_vecs = cv;
}

cudaError_t launch_combine(const CombineArgs& a, bool fp16, int num_sms, cudaStream_t stream)
{
    // a token has at most F = min(W, k) rows; the wide path is only compiled in when F > 8
    if (a.F > 8)
        return fp16 ? launch_t<true, true>(a, num_sms, stream) : launch_t<false, true>(a, num_sms, stream);
    return fp16 ? launch_t<true, false>(a, num_sms, stream) : launch_t<false, false>(a, num_sms, stream);
}

}  // namespace ep

// ep_combine.cu -- Combine gather-reduce.
//
// For every source token, read the expert-output rows of the ranks it was dispatched to
// (forward map, ascending destination rank), add them in FP32 starting from +0.0f in that
// fixed order, and round to nearest even into BF16 / FP16 (MORI-EP gfx1201 PR, Combine bullet:
// "The source sums its local and received contributions in FP32, then converts the output to
// BF16/FP16.  Optional FP32 weights are communicated and summed separately").  Routing weights
// are not applied.  The fixed order makes the result independent of the launch shape.
//
// HBM-bound: per token, all of its (<= min(W, k)) rows' 16-byte vectors for one step are
// loaded before any is added -- the pages' bf16 pull combine likewise loads every source a
// token can have before folding -- then accumulated in registers and stored as one 16-byte
// packed BF16x8 / FP16x8 vector.  Work units are (token, slice of the row), one warp each.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "ep_common.cuh"

namespace ep {
namespace {

constexpr int kBatch = 8;   // rows whose vectors are in flight together

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

template <bool FP16>
__global__ void __launch_bounds__(kCopyThreads) ep_combine_kernel(const CombineArgs a)
{
    __shared__ int s_off[kMaxRanks + 1];
    if (threadIdx.x <= a.W) s_off[threadIdx.x] = a.tok_off[threadIdx.x];
    __syncthreads();

    const int lane = threadIdx.x & 31;
    const int64_t warps_per_grid = (int64_t)gridDim.x * (kCopyThreads / 32);
    const int64_t units = (int64_t)a.N * a.chunks;
    for (int64_t u = (int64_t)blockIdx.x * (kCopyThreads / 32) + (threadIdx.x >> 5); u < units;
         u += warps_per_grid) {
        const int g = (int)(u / a.chunks);
        const int c = (int)(u - (int64_t)g * a.chunks);
        const int s = rank_of_token(s_off, a.W, g);
        const int64_t tok = (int64_t)s * a.M + (g - s_off[s]);

        const int src = lane < a.F ? __ldg(a.fwd + tok * a.F + lane) : -1;
        const int nd = __popc(__ballot_sync(0xffffffffu, src >= 0));

        const int64_t h0 = (int64_t)c * a.chunk_elems;
        const int64_t rem = a.H - h0;
        const int nvec = (int)((rem < a.chunk_elems ? rem : a.chunk_elems) >> 3);
        uint16_t* dst = a.out + tok * a.H + h0;
        for (int v0 = 0; v0 < nvec; v0 += 32) {   // warp-uniform bounds
            const int v = v0 + lane;
            const bool act = v < nvec;
            float acc[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
            for (int d0 = 0; d0 < nd; d0 += kBatch) {
                uint4 buf[kBatch];
#pragma unroll
                for (int q = 0; q < kBatch; ++q) {
                    const int64_t row = __shfl_sync(0xffffffffu, src, (d0 + q) & 31);
                    if (act && d0 + q < nd)
                        buf[q] = ld_stream_v4(a.eo + row * a.H + h0 + (int64_t)v * 8);
                }
#pragma unroll
                for (int q = 0; q < kBatch; ++q)
                    if (act && d0 + q < nd) add_vec<FP16>(acc, buf[q]);
            }
            if (act) st_v4(dst + (int64_t)v * 8, pack_vec<FP16>(acc));
        }

        if (c == 0 && a.w_in != nullptr && a.out_w != nullptr) {
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
    }
}

template <bool FP16>
cudaError_t launch_t(const CombineArgs& a, int num_sms, cudaStream_t stream)
{
    const int64_t units = (int64_t)a.N * a.chunks;
    if (units == 0) return cudaSuccess;
    int per_sm = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, ep_combine_kernel<FP16>,
                                                                  kCopyThreads, 0);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) per_sm = 1;
    const int64_t need = (units + kCopyThreads / 32 - 1) / (kCopyThreads / 32);
    const int64_t cap = (int64_t)per_sm * num_sms;
    const int grid = (int)(need < cap ? need : cap);
    ep_combine_kernel<FP16><<<grid, kCopyThreads, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_combine(const CombineArgs& a, bool fp16, int num_sms, cudaStream_t stream)
{
    return fp16 ? launch_t<true>(a, num_sms, stream) : launch_t<false>(a, num_sms, stream);
}

}  // namespace ep

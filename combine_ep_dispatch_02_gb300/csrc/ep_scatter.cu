// ep_scatter.cu -- payload scatter of Dispatch.
//
// For every source token and every destination rank it was routed to, copy the token's hidden
// row, its top-k index row, its FP32 weight row and its FP32 scale row into that rank's
// receive row (MORI-EP gfx1201 PR, Dispatch bullet: experts that live on one rank share a
// single copy of the hidden row; guide, dispatch() outputs).  The receive rows come from the forward map
// the routing kernel wrote.
//
// HBM-bound: each source row is READ ONCE into registers with 16-byte non-allocating loads and
// WRITTEN once per destination with 16-byte stores, so the traffic is the minimum
// N*row + P*row bytes (N tokens, P token-destination pairs).  Work units are (token, slice of
// the row): whole rows for large token counts, 512- or 1024-element slices for small ones (the
// pages' small-batch launch policy), one warp per unit, a persistent grid sized from the
// occupancy of this kernel times the SM count.  The last rounds of units are drawn from the
// plan's dispatch work queue (work_split), so tokens with many destination ranks do not leave
// a tail of busy warps.
#include "ep_common.cuh"

namespace ep {
namespace {

constexpr int kUnroll = 4;   // 16-byte vectors per lane in flight per step

__global__ void __launch_bounds__(kCopyThreads) ep_scatter_kernel(const ScatterArgs a)
{
    __shared__ int s_off[kMaxRanks + 1];
    if (threadIdx.x <= a.W) s_off[threadIdx.x] = a.tok_off[threadIdx.x];
    wait_for_predecessor();   // the routing kernel's forward map
    probe_mark(a.probe, kProbeScatter, true);
    __syncthreads();

    const int lane = threadIdx.x & 31;
    const int64_t units = (int64_t)a.N * a.chunks;
    // destination rows of a unit, compact and ascending in rank; lane d holds the d-th one
    auto unit_dest = [&](int64_t v) -> int {
        if (v >= units) return -1;
        const int gv = (int)(v / a.chunks);
        const int sv = rank_of_token(s_off, a.W, gv);
        const int64_t tv = (int64_t)sv * a.M + (gv - s_off[sv]);
        return checked_fwd(lane < a.F ? __ldg(a.fwd + tv * a.F + lane) : -1, (int64_t)a.W * a.W * a.M, a.status);
    };
    const WorkSplit& ws = a.work;
    uint32_t u_next = work_first(ws);
    int dest_next = unit_dest(u_next);
    while (u_next < units) {
        const uint32_t u = u_next;
        const int dest = dest_next;
        u_next = work_next(ws, u, lane);                 // the next unit's forward-map row
        dest_next = unit_dest(u_next);                   // lands while this unit is copied
        const int g = (int)(u / a.chunks);
        const int c = (int)(u - (int64_t)g * a.chunks);
        const int s = rank_of_token(s_off, a.W, g);
        const int64_t tok = (int64_t)s * a.M + (g - s_off[s]);
        const int nd = __popc(__ballot_sync(0xffffffffu, dest >= 0));

        const int64_t off = (int64_t)c * a.chunk_bytes;
        const int64_t rem = a.row_bytes - off;
        const int nvec = (int)((rem < a.chunk_bytes ? rem : a.chunk_bytes) >> 4);
        const uint8_t* src = a.x + tok * a.row_bytes + off;
        for (int v0 = 0; v0 < nvec; v0 += 32 * kUnroll) {   // warp-uniform bounds
            uint4 buf[kUnroll];
#pragma unroll
            for (int q = 0; q < kUnroll; ++q) {
                const int v = v0 + q * 32 + lane;
                if (v < nvec) buf[q] = ld_stream_v4(src + (int64_t)v * 16);
            }
            for (int d = 0; d < nd; ++d) {
                const int row = __shfl_sync(0xffffffffu, dest, d);
                uint8_t* dst = a.recv_x + (int64_t)row * a.row_bytes + off;
#pragma unroll
                for (int q = 0; q < kUnroll; ++q) {
                    const int v = v0 + q * 32 + lane;
                    if (v < nvec) st_v4(dst + (int64_t)v * 16, buf[q]);
                }
            }
        }

        if (c == 0) {   // the small per-token rows travel with the first slice
            for (int d = 0; d < nd; ++d) {
                const int64_t row = __shfl_sync(0xffffffffu, dest, d);
                for (int e = lane; e < a.k; e += 32) {
                    a.recv_idx[row * a.k + e] = __ldg(a.idx + tok * a.k + e);
                    if (a.w) a.recv_w[row * a.k + e] = __ldg(a.w + tok * a.k + e);
                }
                for (int e = lane; e < a.sd; e += 32)
                    a.recv_scales[row * a.sd + e] = __ldg(a.scales + tok * a.sd + e);
            }
        }
    }
    probe_mark(a.probe, kProbeScatter, false);
    work_retire(ws);
}

// ---- quantising scatter: BF16 source rows -> FP8 e4m3 rows + one FP32 scale per 128 elements

constexpr int kQUnroll = 2;   // 32-byte source pieces per lane in flight per step

// A lane owns 16 consecutive elements (32 source bytes, 16 code bytes); the 8 lanes of a 128-
// element block agree on its maximum by shuffles, so each block's scale is computed once per
// token and its codes are written to every destination row.  Slices are multiples of 128.
__global__ void __launch_bounds__(kCopyThreads, 3) ep_scatter_quant_kernel(const ScatterArgs a)
{
    __shared__ int s_off[kMaxRanks + 1];
    if (threadIdx.x <= a.W) s_off[threadIdx.x] = a.tok_off[threadIdx.x];
    wait_for_predecessor();   // the routing kernel's forward map
    probe_mark(a.probe, kProbeScatter, true);
    __syncthreads();

    const int lane = threadIdx.x & 31;
    const int64_t units = (int64_t)a.N * a.chunks;
    const int64_t H = a.row_bytes;              // FP8 payload: one byte per element
    const WorkSplit& ws = a.work;
    for (uint32_t u = work_first(ws); u < units; u = work_next(ws, u, lane)) {
        const int g = (int)(u / a.chunks);
        const int c = (int)(u - (int64_t)g * a.chunks);
        const int s = rank_of_token(s_off, a.W, g);
        const int64_t tok = (int64_t)s * a.M + (g - s_off[s]);
        const int dest = checked_fwd(lane < a.F ? __ldg(a.fwd + tok * a.F + lane) : -1,
                                     (int64_t)a.W * a.W * a.M, a.status);
        const int nd = __popc(__ballot_sync(0xffffffffu, dest >= 0));

        const int64_t h0 = (int64_t)c * a.chunk_bytes;               // elements
        const int64_t rem = H - h0;
        const int npiece = (int)((rem < a.chunk_bytes ? rem : a.chunk_bytes) >> 4);   // 16-element pieces
        const uint8_t* src = a.x + (tok * H + h0) * 2;
        for (int p0 = 0; p0 < npiece; p0 += 32 * kQUnroll) {         // warp-uniform bounds
            uint4 in[kQUnroll][2];
#pragma unroll
            for (int q = 0; q < kQUnroll; ++q) {
                const int p = p0 + q * 32 + lane;
                if (p < npiece) {
                    in[q][0] = ld_stream_v4(src + (int64_t)p * 32);
                    in[q][1] = ld_stream_v4(src + (int64_t)p * 32 + 16);
                }
                if (p + 32 * kQUnroll < npiece) prefetch_l2(src + (int64_t)(p + 32 * kQUnroll) * 32);
            }
            uint4 code[kQUnroll];
            float scale[kQUnroll];
#pragma unroll
            for (int q = 0; q < kQUnroll; ++q) {
                const int p = p0 + q * 32 + lane;
                float m = p < npiece ? absmax16(in[q][0], in[q][1]) : 0.0f;
                m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
                m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
                m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
                scale[q] = m > 0.0f ? __fdiv_rn(m, 448.0f) : 1.0f;
                if (p < npiece) code[q] = quantise16(in[q][0], in[q][1], scale[q]);
            }
            for (int d = 0; d < nd; ++d) {
                const int64_t row = __shfl_sync(0xffffffffu, dest, d);
                uint8_t* dst = a.recv_x + row * H + h0;
                float* dsc = a.recv_scales + row * a.sd + (h0 >> 7);
#pragma unroll
                for (int q = 0; q < kQUnroll; ++q) {
                    const int p = p0 + q * 32 + lane;
                    if (p < npiece) {
                        st_v4(dst + (int64_t)p * 16, code[q]);
                        if ((lane & 7) == 0) dsc[p >> 3] = scale[q];
                    }
                }
            }
        }

        if (c == 0) {
            for (int d = 0; d < nd; ++d) {
                const int64_t row = __shfl_sync(0xffffffffu, dest, d);
                for (int e = lane; e < a.k; e += 32) {
                    a.recv_idx[row * a.k + e] = __ldg(a.idx + tok * a.k + e);
                    if (a.w) a.recv_w[row * a.k + e] = __ldg(a.w + tok * a.k + e);
                }
            }
        }
    }
    probe_mark(a.probe, kProbeScatter, false);
    work_retire(ws);
}

// MX FP4 quantising scatter.  A lane owns one 32-element block (64 source bytes -> 16 code
// bytes and one e8m0 scale byte); each block is quantised once per token and written to every
// destination row.  a.chunk_bytes counts ELEMENTS here (slices are multiples of 128).
__global__ void __launch_bounds__(kCopyThreads, 3) ep_scatter_quant_fp4_kernel(const ScatterArgs a)
{
    __shared__ int s_off[kMaxRanks + 1];
    if (threadIdx.x <= a.W) s_off[threadIdx.x] = a.tok_off[threadIdx.x];
    wait_for_predecessor();   // the routing kernel's forward map
    probe_mark(a.probe, kProbeScatter, true);
    __syncthreads();

    const int lane = threadIdx.x & 31;
    const int64_t units = (int64_t)a.N * a.chunks;
    const int64_t H = a.row_bytes * 2;           // elements; a received row holds H/2 code bytes
    const int64_t hb = H >> 5;                    // blocks (and scale bytes) per row
    uint8_t* sc8 = reinterpret_cast<uint8_t*>(a.recv_scales);
    const WorkSplit& ws = a.work;
    for (uint32_t u = work_first(ws); u < units; u = work_next(ws, u, lane)) {
        const int g = (int)(u / a.chunks);
        const int c = (int)(u - (int64_t)g * a.chunks);
        const int s = rank_of_token(s_off, a.W, g);
        const int64_t tok = (int64_t)s * a.M + (g - s_off[s]);
        const int dest = checked_fwd(lane < a.F ? __ldg(a.fwd + tok * a.F + lane) : -1,
                                     (int64_t)a.W * a.W * a.M, a.status);
        const int nd = __popc(__ballot_sync(0xffffffffu, dest >= 0));

        const int64_t h0 = (int64_t)c * a.chunk_bytes;                // elements
        const int64_t rem = H - h0;
        const int nblk = (int)((rem < a.chunk_bytes ? rem : a.chunk_bytes) >> 5);
        const uint4* src = reinterpret_cast<const uint4*>(a.x + (tok * H + h0) * 2);
        for (int b0 = 0; b0 < nblk; b0 += 32) {                      // warp-uniform bounds
            const int b = b0 + lane;
            uint4 codes = make_uint4(0, 0, 0, 0);
            uint32_t code = 0;
            if (b < nblk) {
                uint4 x[4];
#pragma unroll
                for (int t = 0; t < 4; ++t) x[t] = ld_stream_v4(src + (int64_t)b * 4 + t);
                codes = quantise_mxfp4_32(x, code);
            }
            if (b + 32 < nblk) {                       // the next step's block: two 32-byte sectors
                prefetch_l2(src + (int64_t)(b + 32) * 4);
                prefetch_l2(src + (int64_t)(b + 32) * 4 + 2);
            }
            for (int d = 0; d < nd; ++d) {
                const int64_t row = __shfl_sync(0xffffffffu, dest, d);
                if (b < nblk) {
                    st_v4(a.recv_x + row * a.row_bytes + (h0 >> 1) + (int64_t)b * 16, codes);
                    sc8[row * hb + (h0 >> 5) + b] = (uint8_t)code;
                }
            }
        }

        if (c == 0) {
            for (int d = 0; d < nd; ++d) {
                const int64_t row = __shfl_sync(0xffffffffu, dest, d);
                for (int e = lane; e < a.k; e += 32) {
                    a.recv_idx[row * a.k + e] = __ldg(a.idx + tok * a.k + e);
                    if (a.w) a.recv_w[row * a.k + e] = __ldg(a.w + tok * a.k + e);
                }
            }
        }
    }
    probe_mark(a.probe, kProbeScatter, false);
    work_retire(ws);
}

// A persistent grid of the kernel's occupancy times the SM count (at most one warp per unit),
// launched as a dependent of the routing kernel before it.
template <typename Kernel>
cudaError_t launch_copy(Kernel kernel, const ScatterArgs& a, int num_sms, cudaStream_t stream)
{
    const int64_t units = (int64_t)a.N * a.chunks;
    if (units == 0) return cudaSuccess;
    int per_sm = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kCopyThreads, 0);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) per_sm = 1;
    const int64_t need = (units + kCopyThreads / 32 - 1) / (kCopyThreads / 32);
    const int64_t cap = (int64_t)per_sm * num_sms;
    const int grid = (int)(need < cap ? need : cap);
    ScatterArgs b = a;
    b.work = make_work_split(a.work.q, units, (int64_t)grid * (kCopyThreads / 32));
    return launch_dependent(kernel, dim3(grid), dim3(kCopyThreads), 0, stream, b);
}

}  // namespace

cudaError_t launch_scatter_quant_fp4(const ScatterArgs& a, int num_sms, cudaStream_t stream)
{
    return launch_copy(ep_scatter_quant_fp4_kernel, a, num_sms, stream);
}

cudaError_t launch_scatter_quant(const ScatterArgs& a, int num_sms, cudaStream_t stream)
{
    return launch_copy(ep_scatter_quant_kernel, a, num_sms, stream);
}

cudaError_t launch_scatter(const ScatterArgs& a, int num_sms, cudaStream_t stream)
{
    return launch_copy(ep_scatter_kernel, a, num_sms, stream);
}

}  // namespace ep

// ep_fp8wire.cu -- combine over a low-precision wire: FP8 e4m3 blockwise and MX FP4.
//
// The MORI-EP gfx1250 EPv2 pages (push-combine variants) let combine contributions travel at
// low precision: the expert side quantises its BF16 output rows before they are sent, and the
// token's home rank dequantises them while it reduces.  Two encodings are built here:
//   FP8: e4m3 codes with one FP32 scale per 128 elements (the quantiser of the quantising
//        dispatch); the gather reads H + H/32 bytes per row instead of 2H;
//   FP4: e2m1 codes with one e8m0 power-of-two scale per 32 elements (the OCP microscaling
//        layout); the gather reads H/2 + H/32 bytes per row.
// For every source token the terms are added in ascending rank order in FP32 from +0.0f, each
// term being code * scale (one FP32 multiply), and the sum is rounded to nearest even into BF16.
#include <cuda_bf16.h>

#include "ep_common.cuh"

namespace ep {
namespace {

// ---- quantise the received expert rows: warp per row, lanes own 16-element pieces

constexpr int kQuantUnroll = 4;   // 32-byte pieces per lane in flight

__global__ void __launch_bounds__(kCopyThreads, 3) ep_quantise_rows_kernel(const WireArgs a)
{
    __shared__ int s_cnt[kMaxRanks];
    if (threadIdx.x < a.W) s_cnt[threadIdx.x] = checked_count(a.recv_count[threadIdx.x], a.rows, a.status);
    probe_mark(a.probe, kProbeQuantise, true);
    __syncthreads();

    const int lane = threadIdx.x & 31;
    const int64_t nwarps = (int64_t)gridDim.x * (kCopyThreads / 32);
    const int npiece = (int)(a.H >> 4);
    const int nb = (int)(a.H >> 7);
    for (int64_t u = (int64_t)blockIdx.x * (kCopyThreads / 32) + (threadIdx.x >> 5);
         u < (int64_t)a.W * a.rows; u += nwarps) {
        const int r = (int)(u / a.rows);
        const int64_t i = u - (int64_t)r * a.rows;
        if (i >= s_cnt[r]) continue;                 // warp-uniform: only received rows
        const uint8_t* src = reinterpret_cast<const uint8_t*>(a.eo) + u * a.H * 2;
        uint8_t* dq = a.q + u * a.H;
        float* dsc = a.scales + u * nb;
        for (int p0 = 0; p0 < npiece; p0 += 32 * kQuantUnroll) {   // warp-uniform bounds
            uint4 x[kQuantUnroll][2];
#pragma unroll
            for (int t = 0; t < kQuantUnroll; ++t) {
                const int p = p0 + 32 * t + lane;
                x[t][0] = x[t][1] = make_uint4(0, 0, 0, 0);
                if (p < npiece) {
                    x[t][0] = ld_stream_v4(src + (int64_t)p * 32);
                    x[t][1] = ld_stream_v4(src + (int64_t)p * 32 + 16);
                }
                if (p + 32 * kQuantUnroll < npiece) prefetch_l2(src + (int64_t)(p + 32 * kQuantUnroll) * 32);
            }
#pragma unroll
            for (int t = 0; t < kQuantUnroll; ++t) {
                const int p = p0 + 32 * t + lane;
                float m = absmax16(x[t][0], x[t][1]);
                m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
                m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
                m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
                const float scale = m > 0.0f ? __fdiv_rn(m, 448.0f) : 1.0f;
                if (p < npiece) {
                    st_v4(dq + (int64_t)p * 16, quantise16(x[t][0], x[t][1], scale));
                    if ((lane & 7) == 0) dsc[p >> 3] = scale;
                }
            }
        }
    }
    probe_mark(a.probe, kProbeQuantise, false);
}

// ---- gather-reduce over the FP8 wire

// acc += x * s on an element pair: two scalar FP32 multiplies, then one packed FP32 add.  Each
// lane rounds exactly as the scalar add.  (A packed multiply followed by a packed add is not
// used: the two were observed to give fused-multiply-add results, which differ from the
// oracle's rounded product.)
__device__ __forceinline__ void mul_add_f32x2(float& a0, float& a1, float x0, float x1, float s)
{
    const float p0 = __fmul_rn(x0, s), p1 = __fmul_rn(x1, s);
    unsigned long long a, pv;
    asm("mov.b64 %0, {%1, %2};" : "=l"(a) : "f"(a0), "f"(a1));
    asm("mov.b64 %0, {%1, %2};" : "=l"(pv) : "f"(p0), "f"(p1));
    asm("add.rn.f32x2 %0, %0, %1;" : "+l"(a) : "l"(pv));
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a0), "=f"(a1) : "l"(a));
}

__device__ __forceinline__ void add_fp8x16(float (&acc)[16], const uint4& c, float scale)
{
    const uint32_t w[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 lo = e4m3x2_to_float2(w[i] & 0xFFFFu);
        const float2 hi = e4m3x2_to_float2(w[i] >> 16);
        mul_add_f32x2(acc[4 * i + 0], acc[4 * i + 1], lo.x, lo.y, scale);
        mul_add_f32x2(acc[4 * i + 2], acc[4 * i + 3], hi.x, hi.y, scale);
    }
}

// 16 sums as BF16 to dst[0..1]: one 32-byte store when the output is 32-byte aligned (V8), so a
// warp writes whole sectors although its lanes' pieces are 32 bytes apart; else two 16-byte ones.
template <bool V8>
__device__ __forceinline__ void store_bf16x16(uint4* dst, const float (&acc)[16])
{
    uint32_t w[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const __nv_bfloat162 b = __floats2bfloat162_rn(acc[2 * i], acc[2 * i + 1]);
        w[i] = *reinterpret_cast<const uint32_t*>(&b);
    }
    if constexpr (V8) {
        st_v8(dst, make_uint4(w[0], w[1], w[2], w[3]), make_uint4(w[4], w[5], w[6], w[7]));
    } else {
        st_v4(dst, make_uint4(w[0], w[1], w[2], w[3]));
        st_v4(dst + 1, make_uint4(w[4], w[5], w[6], w[7]));
    }
}

// Rolling fold of a unit's nd <= 8 rows (lane d of src holds row d): row d's loads of the next
// kWireDepth pieces are in flight while the current ones are folded, so every lane keeps
// nd * kWireDepth 16-byte loads outstanding.
#ifndef EP_WIRE_DEPTH
#define EP_WIRE_DEPTH 1   // 2 spills at the 128-register budget of 2 CTAs per SM
#endif
constexpr int kWireDepth = EP_WIRE_DEPTH;

template <bool V8>
__device__ __forceinline__ void fold_fp8_rows(const WireArgs& a, int src, int nd, int p0, int np,
                                              uint4* dst, int lane)
{
    const int64_t hp = a.H >> 4;
    const uint4* q4 = reinterpret_cast<const uint4*>(a.q);
    // piece offsets of the rows (32 bits: the plan's shape keeps W*W*M*H below 2^35, so the wire's
    // W*W*M*H/16 pieces stay below 2^31); a piece's scale sits at offset / 8,
    // since a row has hp = 8 * nb pieces and slices start on multiples of 8 pieces
    uint32_t ro[8];
#pragma unroll
    for (int d = 0; d < 8; ++d) ro[d] = (uint32_t)((int64_t)__shfl_sync(0xffffffffu, src, d) * hp + p0);
    uint4 b[8][kWireDepth];
    float sc[8][kWireDepth];
#pragma unroll
    for (int t = 0; t < kWireDepth; ++t)
#pragma unroll
        for (int d = 0; d < 8; ++d)
            if (d < nd && lane + 32 * t < np) {
                b[d][t] = ld_stream_v4(q4 + ro[d] + lane + 32 * t);
                sc[d][t] = __ldg(a.scales + ((ro[d] + lane + 32 * t) >> 3));
            }
    for (int vb = 0; vb < np; vb += 32 * kWireDepth) {    // warp-uniform bounds
#pragma unroll
        for (int t = 0; t < kWireDepth; ++t) {
            const int pc = vb + 32 * t + lane;
            const int pn = pc + 32 * kWireDepth;
            float acc[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) acc[i] = 0.0f;
#pragma unroll
            for (int d = 0; d < 8; ++d) {
                if (d < nd) {
                    const uint4 x = b[d][t];
                    const float xs = sc[d][t];
                    if (pn < np) {
                        b[d][t] = ld_stream_v4(q4 + ro[d] + pn);
                        sc[d][t] = __ldg(a.scales + ((ro[d] + pn) >> 3));
                    }
                    if (pn + 32 * kWireDepth < np) prefetch_l2(q4 + ro[d] + pn + 32 * kWireDepth);
                    if (pc < np) add_fp8x16(acc, x, xs);
                }
            }
            if (pc < np) store_bf16x16<V8>(dst + (int64_t)pc * 2, acc);
        }
    }
}

// More than 8 rows: one piece per lane at a time, rows in ascending batches of 8.
__device__ __forceinline__ void fold_fp8_wide(const WireArgs& a, int src, int nd, int p0, int np,
                                              uint4* dst, int lane)
{
    const int64_t hp = a.H >> 4;
    const int64_t nb = a.H >> 7;
    const uint4* q4 = reinterpret_cast<const uint4*>(a.q);
    for (int vb = 0; vb < np; vb += 32) {
        const int pc = vb + lane;
        const bool act = pc < np;
        float acc[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) acc[i] = 0.0f;
        for (int d0 = 0; d0 < nd; d0 += 8) {
            uint4 b[8];
            float sc[8];
#pragma unroll
            for (int d = 0; d < 8; ++d) {
                const int64_t row = __shfl_sync(0xffffffffu, src, (d0 + d) & 31);
                if (act && d0 + d < nd) {
                    b[d] = ld_stream_v4(q4 + row * hp + p0 + pc);
                    sc[d] = __ldg(a.scales + row * nb + ((p0 + pc) >> 3));
                }
            }
#pragma unroll
            for (int d = 0; d < 8; ++d)
                if (act && d0 + d < nd) add_fp8x16(acc, b[d], sc[d]);
        }
        if (act) store_bf16x16<false>(dst + (int64_t)pc * 2, acc);
    }
}

// A warp owns a (token, slice) unit; lanes own 16-element pieces (16 code bytes, 32 output
// bytes).  Weight rows are summed as in the 16-bit combine.
template <bool WIDE, bool V8>
__global__ void __launch_bounds__(kCopyThreads, 2) ep_combine_fp8_kernel(const WireArgs a)
{
    __shared__ int s_off[kMaxRanks + 1];
    if (threadIdx.x <= a.W) s_off[threadIdx.x] = a.tok_off[threadIdx.x];
    probe_mark(a.probe, kProbeWireCombine, true);
    __syncthreads();

    const int lane = threadIdx.x & 31;
    const uint32_t units = (uint32_t)a.N * (uint32_t)a.chunks;
    const uint32_t step = gridDim.x * (kCopyThreads / 32);
    for (uint32_t u = blockIdx.x * (kCopyThreads / 32) + (threadIdx.x >> 5); u < units; u += step) {
        const int g = (int)(u / (uint32_t)a.chunks);
        const int c = (int)(u - (uint32_t)g * (uint32_t)a.chunks);
        const int s = rank_of_token(s_off, a.W, g);
        const int64_t tok = (int64_t)s * a.M + (g - s_off[s]);
        const int src = checked_fwd(lane < a.F ? __ldg(a.fwd + tok * a.F + lane) : -1,
                                    (int64_t)a.W * a.rows, a.status);
        const int nd = __popc(__ballot_sync(0xffffffffu, src >= 0));
        const int p0 = c * a.chunk_pieces;
        const int np = (int)min((int64_t)a.chunk_pieces, (a.H >> 4) - p0);
        uint4* dst = reinterpret_cast<uint4*>(a.out + tok * a.H) + (int64_t)p0 * 2;
        if (!WIDE || nd <= 8)
            fold_fp8_rows<V8>(a, src, nd, p0, np, dst, lane);     // nd == 0 stores +0
        else
            fold_fp8_wide(a, src, nd, p0, np, dst, lane);

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
    probe_mark(a.probe, kProbeWireCombine, false);
}

// ---- the MX FP4 wire (quantiser quantise_mxfp4_32 in ep_common.cuh)

__device__ __forceinline__ float e8m0_to_float(uint32_t code)
{
    return __uint_as_float(code == 0 ? 0x00400000u : code << 23);
}

// One lane quantises one 32-element block (64 BF16 bytes -> 16 code bytes + 1 scale byte).
__global__ void __launch_bounds__(kCopyThreads, 3) ep_quantise_rows_fp4_kernel(const WireArgs a)
{
    __shared__ int s_cnt[kMaxRanks];
    if (threadIdx.x < a.W) s_cnt[threadIdx.x] = checked_count(a.recv_count[threadIdx.x], a.rows, a.status);
    probe_mark(a.probe, kProbeQuantise, true);
    __syncthreads();
    const int lane = threadIdx.x & 31;
    const int64_t nwarps = (int64_t)gridDim.x * (kCopyThreads / 32);
    const int nblk = (int)(a.H >> 5);
    uint8_t* sc8 = reinterpret_cast<uint8_t*>(a.scales);
    for (int64_t u = (int64_t)blockIdx.x * (kCopyThreads / 32) + (threadIdx.x >> 5);
         u < (int64_t)a.W * a.rows; u += nwarps) {
        const int r = (int)(u / a.rows);
        const int64_t i = u - (int64_t)r * a.rows;
        if (i >= s_cnt[r]) continue;                 // warp-uniform: only received rows
        const uint4* src = reinterpret_cast<const uint4*>(reinterpret_cast<const uint8_t*>(a.eo) + u * a.H * 2);
        uint4* dq = reinterpret_cast<uint4*>(a.q + u * (a.H >> 1));
        for (int b0 = 0; b0 < nblk; b0 += 32) {      // warp-uniform bounds
            const int b = b0 + lane;
            if (b >= nblk) continue;
            uint4 x[4];
#pragma unroll
            for (int t = 0; t < 4; ++t) x[t] = ld_stream_v4(src + (int64_t)b * 4 + t);
            if (b + 32 < nblk) {                     // the next step's block: two 32-byte sectors
                prefetch_l2(src + (int64_t)(b + 32) * 4);
                prefetch_l2(src + (int64_t)(b + 32) * 4 + 2);
            }
            uint32_t code;
            const uint4 codes = quantise_mxfp4_32(x, code);
            st_v4(dq + b, codes);
            sc8[u * nblk + b] = (uint8_t)code;
        }
    }
    probe_mark(a.probe, kProbeQuantise, false);
}

__device__ __forceinline__ void fma_f32x2(float2& acc, float2 x, unsigned long long ss)
{
    unsigned long long a, xv;
    asm("mov.b64 %0, {%1, %2};" : "=l"(a) : "f"(acc.x), "f"(acc.y));
    asm("mov.b64 %0, {%1, %2};" : "=l"(xv) : "f"(x.x), "f"(x.y));
    asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(a) : "l"(xv), "l"(ss));
    asm("mov.b64 {%0, %1}, %2;" : "=f"(acc.x), "=f"(acc.y) : "l"(a));
}

// The four code bytes of w (8 e2m1 codes, element 0 in the low nibble) as four f16x2 pairs.
__device__ __forceinline__ void e2m1x8_to_half2x4(uint32_t w, uint32_t (&h)[4])
{
    asm("{ .reg .b8 b0, b1, b2, b3;\n\t"
        "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
        "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
        "cvt.rn.f16x2.e2m1x2 %3, b3; }"
        : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3]) : "r"(w));
}

// acc.x += lo(h) * s and acc.y += hi(h) * s: fused multiply-adds of two f16 operands into FP32
// (the operands widen exactly; the product and sum round once).
__device__ __forceinline__ void fma_f16x2_f32(float2& acc, uint32_t h, uint16_t s)
{
    asm("{ .reg .b16 l, u;\n\t"
        "mov.b32 {l, u}, %2;\n\t"
        "fma.rn.f32.f16 %0, l, %3, %0;\n\t"
        "fma.rn.f32.f16 %1, u, %3, %1; }"
        : "+f"(acc.x), "+f"(acc.y) : "r"(h), "h"(s));
}

// acc[0..7] (element pairs) += the 16 e2m1 codes of (lo, hi) times 2^(code - 127).
// An e2m1 value has at most two significant bits and the scale is a power of two, so the
// product is exact in FP32 (down to 2^-128, above FP32's smallest subnormal) unless it
// overflows; a fused multiply-add therefore rounds exactly as the product followed by an add.
// Scales 2^-14 .. 2^15 (codes 113 .. 142, block maxima from 2^-12 to below 2^18) are normal
// f16 numbers: the f16 code values multiply them in f16-operand FMAs, with no conversion to
// FP32.  Other codes widen the values first; only codes 253 and 254 (an infinite block maximum)
// can overflow, and they take the two-step form.
__device__ __forceinline__ void add_fp4x16(float2 (&acc)[8], uint32_t lo, uint32_t hi, uint32_t code)
{
    uint32_t hv[8];
    {
        uint32_t t[4];
        e2m1x8_to_half2x4(lo, t);
#pragma unroll
        for (int i = 0; i < 4; ++i) hv[i] = t[i];
        e2m1x8_to_half2x4(hi, t);
#pragma unroll
        for (int i = 0; i < 4; ++i) hv[4 + i] = t[i];
    }
    if (code - 113u < 30u) {
        const uint16_t sh = (uint16_t)((code - 112u) << 10);   // f16 bits of 2^(code - 127)
#pragma unroll
        for (int i = 0; i < 8; ++i) fma_f16x2_f32(acc[i], hv[i], sh);
        return;
    }
    const float scale = e8m0_to_float(code);
    if (code < 253u) {
        unsigned long long ss;
        asm("mov.b64 %0, {%1, %1};" : "=l"(ss) : "f"(scale));
#pragma unroll
        for (int i = 0; i < 8; ++i)
            fma_f32x2(acc[i], __half22float2(*reinterpret_cast<const __half2*>(&hv[i])), ss);
        return;
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float2 v = __half22float2(*reinterpret_cast<const __half2*>(&hv[i]));
        acc[i].x = __fadd_rn(acc[i].x, __fmul_rn(v.x, scale));
        acc[i].y = __fadd_rn(acc[i].y, __fmul_rn(v.y, scale));
    }
}

template <bool V8>
__device__ __forceinline__ void store_bf16x16(uint4* dst, const float2 (&acc)[8])
{
    uint32_t w[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const __nv_bfloat162 b = __floats2bfloat162_rn(acc[i].x, acc[i].y);
        w[i] = *reinterpret_cast<const uint32_t*>(&b);
    }
    if constexpr (V8) {
        st_v8(dst, make_uint4(w[0], w[1], w[2], w[3]), make_uint4(w[4], w[5], w[6], w[7]));
    } else {
        st_v4(dst, make_uint4(w[0], w[1], w[2], w[3]));
        st_v4(dst + 1, make_uint4(w[4], w[5], w[6], w[7]));
    }
}

// Rolling fold of nd <= 8 rows over the FP4 wire.  A lane owns 32-element blocks (16 code bytes
// and one scale byte per row); the block's two 16-element halves are summed one after the
// other, so 16 accumulators are live, and each row's next block is loaded as soon as its
// upper half has been added.
template <bool V8>
__device__ __forceinline__ void fold_fp4_rows(const WireArgs& a, int src, int nd, int b0, int nb,
                                              uint4* dst, int lane)
{
    const int64_t hb = a.H >> 5;                      // blocks per row
    const uint4* q4 = reinterpret_cast<const uint4*>(a.q);
    const uint8_t* sc8 = reinterpret_cast<const uint8_t*>(a.scales);
    uint32_t ro[8];                                   // block offsets (W*W*M*H/32 < 2^30)
#pragma unroll
    for (int d = 0; d < 8; ++d) ro[d] = (uint32_t)((int64_t)__shfl_sync(0xffffffffu, src, d) * hb + b0);
    uint4 b[8];
    uint32_t sc[8];
#pragma unroll
    for (int d = 0; d < 8; ++d)
        if (d < nd && lane < nb) {
            b[d] = ld_stream_v4(q4 + ro[d] + lane);
            sc[d] = __ldg(sc8 + ro[d] + lane);
        }
    for (int vb = 0; vb < nb; vb += 32) {             // warp-uniform bounds
        const int pc = vb + lane, pn = pc + 32;
        float2 acc[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = make_float2(0.0f, 0.0f);
#pragma unroll
        for (int d = 0; d < 8; ++d)
            if (d < nd && pc < nb) add_fp4x16(acc, b[d].x, b[d].y, sc[d]);
        if (pc < nb) store_bf16x16<V8>(dst + (int64_t)pc * 4, acc);
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = make_float2(0.0f, 0.0f);
#pragma unroll
        for (int d = 0; d < 8; ++d) {
            if (d < nd) {
                const uint32_t z = b[d].z, w = b[d].w, xs = sc[d];
                if (pn < nb) {
                    b[d] = ld_stream_v4(q4 + ro[d] + pn);
                    sc[d] = __ldg(sc8 + ro[d] + pn);
                }
                if (pn + 32 < nb) {
                    prefetch_l2(q4 + ro[d] + pn + 32);
                    prefetch_l2(sc8 + ro[d] + pn + 32);
                }
                if (pn + 64 < nb) prefetch_l2(q4 + ro[d] + pn + 64);
                if (pc < nb) add_fp4x16(acc, z, w, xs);
            }
        }
        if (pc < nb) store_bf16x16<V8>(dst + (int64_t)pc * 4 + 2, acc);
    }
}

// More than 8 rows: one half-block per lane at a time, rows in ascending batches of 8.
__device__ __forceinline__ void fold_fp4_wide(const WireArgs& a, int src, int nd, int b0, int nb,
                                              uint4* dst, int lane)
{
    const int64_t hb = a.H >> 5;
    const uint2* q2 = reinterpret_cast<const uint2*>(a.q);
    const uint8_t* sc8 = reinterpret_cast<const uint8_t*>(a.scales);
    for (int vb = 0; vb < nb; vb += 32) {
        const int pc = vb + lane;
        const bool act = pc < nb;
#pragma unroll 1
        for (int half = 0; half < 2; ++half) {
            float2 acc[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[i] = make_float2(0.0f, 0.0f);
            for (int d0 = 0; d0 < nd; d0 += 8) {
                uint2 c[8];
                uint32_t sc[8];
#pragma unroll
                for (int d = 0; d < 8; ++d) {
                    const int64_t blk = (int64_t)__shfl_sync(0xffffffffu, src, (d0 + d) & 31) * hb + b0 + pc;
                    if (act && d0 + d < nd) {
                        c[d] = __ldg(q2 + blk * 2 + half);
                        sc[d] = __ldg(sc8 + blk);
                    }
                }
#pragma unroll
                for (int d = 0; d < 8; ++d)
                    if (act && d0 + d < nd) add_fp4x16(acc, c[d].x, c[d].y, sc[d]);
            }
            if (act) store_bf16x16<false>(dst + (int64_t)pc * 4 + 2 * half, acc);
        }
    }
}

// A warp owns a (token, slice) unit; a.chunk_pieces counts 32-element blocks per slice.
// Weight rows are summed as in the 16-bit combine.
template <bool WIDE, bool V8>
__global__ void __launch_bounds__(kCopyThreads, 2) ep_combine_fp4_kernel(const WireArgs a)
{
    __shared__ int s_off[kMaxRanks + 1];
    if (threadIdx.x <= a.W) s_off[threadIdx.x] = a.tok_off[threadIdx.x];
    probe_mark(a.probe, kProbeWireCombine, true);
    __syncthreads();
    const int lane = threadIdx.x & 31;
    const uint32_t units = (uint32_t)a.N * (uint32_t)a.chunks;
    const uint32_t step = gridDim.x * (kCopyThreads / 32);
    for (uint32_t u = blockIdx.x * (kCopyThreads / 32) + (threadIdx.x >> 5); u < units; u += step) {
        const int g = (int)(u / (uint32_t)a.chunks);
        const int c = (int)(u - (uint32_t)g * (uint32_t)a.chunks);
        const int s = rank_of_token(s_off, a.W, g);
        const int64_t tok = (int64_t)s * a.M + (g - s_off[s]);
        const int src = checked_fwd(lane < a.F ? __ldg(a.fwd + tok * a.F + lane) : -1,
                                    (int64_t)a.W * a.rows, a.status);
        const int nd = __popc(__ballot_sync(0xffffffffu, src >= 0));
        const int b0 = c * a.chunk_pieces;
        const int nb = (int)min((int64_t)a.chunk_pieces, (a.H >> 5) - b0);
        uint4* dst = reinterpret_cast<uint4*>(a.out + tok * a.H) + (int64_t)b0 * 4;
        if (!WIDE || nd <= 8)
            fold_fp4_rows<V8>(a, src, nd, b0, nb, dst, lane);     // nd == 0 stores +0
        else
            fold_fp4_wide(a, src, nd, b0, nb, dst, lane);

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
    probe_mark(a.probe, kProbeWireCombine, false);
}

int grid_for(const void* kernel, int64_t warps_needed, int num_sms)
{
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kCopyThreads, 0) != cudaSuccess ||
        per_sm < 1)
        per_sm = 1;
    const int64_t need = (warps_needed + kCopyThreads / 32 - 1) / (kCopyThreads / 32);
    const int64_t cap = (int64_t)per_sm * num_sms;
    return (int)(need < cap ? need : cap);
}

}  // namespace

cudaError_t launch_quantise_rows(const WireArgs& a, int num_sms, cudaStream_t stream)
{
    const int64_t units = (int64_t)a.W * a.rows;
    if (units == 0) return cudaSuccess;
    ep_quantise_rows_kernel<<<grid_for((const void*)ep_quantise_rows_kernel, units, num_sms),
                              kCopyThreads, 0, stream>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_quantise_rows_fp4(const WireArgs& a, int num_sms, cudaStream_t stream)
{
    const int64_t units = (int64_t)a.W * a.rows;
    if (units == 0) return cudaSuccess;
    ep_quantise_rows_fp4_kernel<<<grid_for((const void*)ep_quantise_rows_fp4_kernel, units, num_sms),
                                  kCopyThreads, 0, stream>>>(a);
    return cudaGetLastError();
}

// The output rows take 32-byte stores when `out` is 32-byte aligned (every row offset, tok * 2H,
// is then too: H is a multiple of 32); a 16-byte aligned `out` takes two 16-byte stores.
static bool out_32b_aligned(const WireArgs& a) { return ((uintptr_t)a.out & 31u) == 0; }

cudaError_t launch_combine_fp4(const WireArgs& a, int num_sms, cudaStream_t stream)
{
    const int64_t units = (int64_t)a.N * a.chunks;
    if (units == 0) return cudaSuccess;
    const bool v8 = out_32b_aligned(a);
    // the wide fold (more than 8 rows) stores 16 bytes at a time whatever the alignment
    void (*k)(WireArgs) = a.F > 8 ? ep_combine_fp4_kernel<true, false>
                                  : (v8 ? ep_combine_fp4_kernel<false, true> : ep_combine_fp4_kernel<false, false>);
    k<<<grid_for((const void*)k, units, num_sms), kCopyThreads, 0, stream>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_combine_fp8(const WireArgs& a, int num_sms, cudaStream_t stream)
{
    const int64_t units = (int64_t)a.N * a.chunks;
    if (units == 0) return cudaSuccess;
    const bool v8 = out_32b_aligned(a);
    // the wide fold (more than 8 rows) stores 16 bytes at a time whatever the alignment
    void (*k)(WireArgs) = a.F > 8 ? ep_combine_fp8_kernel<true, false>
                                  : (v8 ? ep_combine_fp8_kernel<false, true> : ep_combine_fp8_kernel<false, false>);
    k<<<grid_for((const void*)k, units, num_sms), kCopyThreads, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace ep

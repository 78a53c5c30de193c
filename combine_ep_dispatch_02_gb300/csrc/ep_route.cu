// ep_route.cu -- routing kernel of Dispatch: destination dedup, receive-row prefix scan,
// reverse and forward maps, receive counts.
//
// Follows the Dispatch bullet of the MORI-EP gfx1201 PR ("How the gfx1201 kernels work"): each
// token's selected experts map to destination ranks and the token reserves one receive row per
// destination rank, experts on one rank sharing the row; the mapping back to the source token
// is recorded (guide, get_dispatch_src_token_pos(): src_rank * (W*M) + src_token).
//
// Row numbering.  On every destination rank r, rows go to tokens in flattened (source rank,
// token) order: slot(s,t,r) = #{earlier tokens that also go to r}.  That is an exclusive
// prefix sum over tokens of W 0/1 columns, computed here in one pass:
//   1. one CTA per tile of 256 consecutive tokens takes a tile number from a monotone ticket
//      (so a CTA only ever waits on tiles whose CTAs are already running);
//   2. the destination set of each token is the OR over its k slots of (1 << rank); lanes
//      hold one slot each, in batches of up to 32 slots (k <= 64: "runtime routing loops ...
//      in wave32-sized batches, including slots 32-63"), OR-reduced with warp shuffles, so a
//      rank named by several experts counts once;
//   3. per-rank counts: one ballot per rank gives each token's rank within its warp and the
//      warp totals; a block scan over the 8 warps gives the tile's own total per rank;
//   4. decoupled lookback: the tile publishes its totals (status AGGREGATE), then walks back
//      over predecessors' words, 256/W' of them per step (W' = W rounded up to a power of 2),
//      summing until it meets an INCLUSIVE word, and publishes its own INCLUSIVE prefix;
//   5. each token writes src_pos for each of its rows and its compact forward-map row.
// Every scan word carries a stamp derived from the ticket (ticket / tiles + 1), so words from
// the previous call are ignored and no per-call clearing is needed (the pages' "generation
// counters ... coordinate ... buffer reuse across calls").  Waits are bounded: an expired wait
// records EP_ERR_DEVICE_TIMEOUT and the CTA carries on, so the kernel always terminates.
#include <climits>

#include "ep_common.cuh"

namespace ep {
namespace {

__device__ __forceinline__ unsigned long long pack_flag(uint32_t stamp, unsigned long long st,
                                                        uint32_t count)
{
    return ((unsigned long long)stamp << 34) | (st << 32) | (unsigned long long)count;
}

// Destination-rank masks of the tile's tokens.  KP lanes (a power of two, <= 32) cover the
// top-k slots of one token; 32/KP tokens per warp pass.
template <int KP>
__device__ __forceinline__ void route_masks(const RouteArgs& a, int base, const int* off,
                                            uint32_t* s_mask, int warp, int lane)
{
    constexpr int TP = 32 / KP;
    const int j0 = lane % KP;
    const int sub = lane / KP;
    const int n_exp = a.W * a.E;
    for (int pass = 0; pass < KP; ++pass) {
        const int local = warp * 32 + pass * TP + sub;
        const int g = base + local;
        const bool valid = g < a.N;
        const int32_t* row = nullptr;
        if (valid) {
            const int s = rank_of_token(off, a.W, g);
            row = a.idx + ((int64_t)s * a.M + (g - off[s])) * a.k;
        }
        uint32_t m = 0;
        for (int b = 0; b * KP < a.k; ++b) {      // warp-uniform trip count
            const int j = b * KP + j0;
            if (valid && j < a.k) {
                const int e = __ldg(row + j);
                if (e >= 0 && e < n_exp)
                    m |= 1u << (e / a.E);
                else
                    record_status(a.status, EP_ERR_INDEX);
            }
        }
#pragma unroll
        for (int o = KP / 2; o > 0; o >>= 1) m |= __shfl_xor_sync(0xffffffffu, m, o);
        if (j0 == 0) s_mask[local] = valid ? m : 0u;
    }
}

template <int KP>
__global__ void __launch_bounds__(kRouteThreads) ep_route_kernel(const RouteArgs a)
{
    __shared__ uint32_t s_mask[kRouteTile];
    __shared__ int s_off[kMaxRanks + 1];
    __shared__ int s_warp[kRouteThreads / 32][kMaxRanks];   // warp totals, then warp prefixes
    __shared__ int s_agg[kMaxRanks];
    __shared__ int s_excl[kMaxRanks];
    __shared__ int s_incl_at[kMaxRanks];
    __shared__ int s_done[kMaxRanks];
    __shared__ unsigned long long s_ticket;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) s_ticket = atomicAdd(a.ticket, 1ull);
    if (tid <= a.W) s_off[tid] = a.tok_off[tid];
    __syncthreads();
    const unsigned long long ticket = s_ticket;
    const int tile = (int)(ticket % (unsigned long long)a.tiles);
    const uint32_t stamp = (uint32_t)((ticket / (unsigned long long)a.tiles + 1ull) & kStampMask);
    const int base = tile * kRouteTile;

    route_masks<KP>(a, base, s_off, s_mask, warp, lane);
    __syncthreads();

    const int g = base + tid;
    const bool valid = g < a.N;
    const uint32_t mask = valid ? s_mask[tid] : 0u;
    for (int r = 0; r < a.W; ++r) {
        const unsigned bal = __ballot_sync(0xffffffffu, (mask >> r) & 1u);
        if (lane == 0) s_warp[warp][r] = __popc(bal);
    }
    __syncthreads();

    if (tid < a.W) {
        int run = 0;
#pragma unroll
        for (int w = 0; w < kRouteThreads / 32; ++w) {
            const int c = s_warp[w][tid];
            s_warp[w][tid] = run;
            run += c;
        }
        s_agg[tid] = run;
        s_excl[tid] = 0;
        s_done[tid] = (tile == 0);
        s_incl_at[tid] = INT_MAX;
#ifdef EP_TEST_WITHHOLD_TILE0
        // test builds only: tile 0 never publishes, so every other tile's bounded wait runs out
        if (tile != 0)
#endif
        st_relaxed_u64(a.flags + (int64_t)tile * a.W + tid,
                       pack_flag(stamp, tile == 0 ? kFlagInclusive : kFlagAggregate, (uint32_t)run));
    }
    __syncthreads();

    if (tile > 0) {
        int wp = 1;
        while (wp < a.W) wp <<= 1;
        const int window = kRouteThreads / wp;
        const int r = tid & (wp - 1);
        const int p = tid / wp;
        for (int wbase = 0;; wbase += window) {
            const int j = tile - 1 - wbase - p;
            unsigned long long f = 0;
            bool have = false;
            if (r < a.W && j >= 0 && !s_done[r]) {
                const unsigned long long* fp = a.flags + (int64_t)j * a.W + r;
                unsigned ns = 32;
                for (int it = 0;; ++it) {
                    f = ld_relaxed_u64(fp);
                    if ((uint32_t)(f >> 34) == stamp && ((f >> 32) & 3ull) != 0ull) {
                        have = true;
                        break;
                    }
                    if (it >= kSpinLimit) {
                        record_status(a.status, EP_ERR_DEVICE_TIMEOUT);
                        break;
                    }
                    __nanosleep(ns);
                    if (ns < 256) ns <<= 1;
                }
                if (have && ((f >> 32) & 3ull) == kFlagInclusive) atomicMin(&s_incl_at[r], p);
            }
            __syncthreads();
            if (have && p <= s_incl_at[r]) atomicAdd(&s_excl[r], (int)(uint32_t)f);
            __syncthreads();
            if (tid < a.W && !s_done[tid]) {
                if (s_incl_at[tid] != INT_MAX || tile - wbase - window <= 0) s_done[tid] = 1;
                s_incl_at[tid] = INT_MAX;
            }
            __syncthreads();
            if (__syncthreads_and(tid < a.W ? s_done[tid] : 1)) break;
        }
        if (tid < a.W)
            st_relaxed_u64(a.flags + (int64_t)tile * a.W + tid,
                           pack_flag(stamp, kFlagInclusive, (uint32_t)(s_excl[tid] + s_agg[tid])));
    }
    if (tile == a.tiles - 1 && tid < a.W) a.recv_count[tid] = s_excl[tid] + s_agg[tid];
    // s_excl / s_warp are final: the loop above ended on a barrier (or tile 0 needs no lookback)

    int s = 0, t = 0;
    if (valid) {
        s = rank_of_token(s_off, a.W, g);
        t = g - s_off[s];
    }
    int32_t* fwd_row = a.fwd + ((int64_t)s * a.M + t) * a.F;
    const unsigned lt = lanemask_lt();
    int j = 0;
    for (int r = 0; r < a.W; ++r) {
        const unsigned bit = (mask >> r) & 1u;
        const unsigned bal = __ballot_sync(0xffffffffu, bit);
        if (bit) {
            const int slot = s_excl[r] + s_warp[warp][r] + __popc(bal & lt);
            a.src_pos[(int64_t)r * a.rows + slot] = (int32_t)((int64_t)s * a.rows + t);
            fwd_row[j++] = (int32_t)((int64_t)r * a.rows + slot);
        }
    }
    if (valid)
        for (; j < a.F; ++j) fwd_row[j] = -1;
}

template <int KP>
cudaError_t launch_kp(const RouteArgs& a, cudaStream_t stream)
{
    ep_route_kernel<KP><<<a.tiles, kRouteThreads, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_route(const RouteArgs& a, cudaStream_t stream)
{
    // lanes per token: the top-k rounded up to a power of two, capped at one warp; top-k 8
    // (the pages' specialised case) is one of the compiled widths
    const int k = a.k < 32 ? a.k : 32;
    if (k <= 1) return launch_kp<1>(a, stream);
    if (k <= 2) return launch_kp<2>(a, stream);
    if (k <= 4) return launch_kp<4>(a, stream);
    if (k <= 8) return launch_kp<8>(a, stream);
    if (k <= 16) return launch_kp<16>(a, stream);
    return launch_kp<32>(a, stream);
}

}  // namespace ep

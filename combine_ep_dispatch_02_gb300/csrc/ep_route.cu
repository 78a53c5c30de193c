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
//   1. one CTA per tile of 256 consecutive tokens of this call (ceil(N / 256) CTAs, at least
//      one) takes a tile number from a ticket in launch order (so a CTA only ever waits on
//      tiles whose CTAs are already running);
//   2. the destination set of each token is the OR over its k slots of (1 << rank), so a rank
//      named by several experts counts once; each thread loads its token's whole index row
//      with 16-byte vectors (top-k 1..64: the pages' run-time routing loops over slot batches,
//      up to slot 63, become one vector loop per token), so a tile's rows are in flight together;
//   3. per-rank counts: one ballot per rank gives each token's rank within its warp and the
//      warp totals; a block scan over the 8 warps gives the tile's own total per rank;
//   4. decoupled lookback: the tile publishes its totals (status AGGREGATE), then walks back
//      over predecessors' words, 256/W' of them per step (W' = W rounded up to a power of 2),
//      summing until it meets an INCLUSIVE word, and publishes its own INCLUSIVE prefix;
//   5. each token writes src_pos for each of its rows and its compact forward-map row.
// Every scan word carries the call's stamp, a generation count kept on the device, so words
// from earlier calls are ignored and no per-call clearing is needed (the pages reuse buffers
// across calls by means of generation counters).  The last CTA to finish returns the ticket to
// zero and advances the generation, so the next launch on the plan's stream -- eager or a
// CUDA-graph replay, with any token count -- starts from a clean ticket and a new stamp without
// a memset.  Waits are bounded: an expired wait records EP_ERR_DEVICE_TIMEOUT and the CTA
// carries on, so the kernel always terminates.
#include <climits>

#include "ep_common.cuh"

namespace ep {
namespace {

__device__ __forceinline__ unsigned long long pack_flag(uint32_t stamp, unsigned long long st,
                                                        uint32_t count)
{
    return ((unsigned long long)stamp << 34) | (st << 32) | (unsigned long long)count;
}

// Destination-rank mask of one token: OR over its k top-k slots of (1 << rank), so a rank named
// by several experts counts once.  `id` holds the index row, loaded by the caller with 16-byte
// vectors (VEC = k / 4 known at compile time; the pages' dedicated top-k 8 case is VEC = 2) so a
// tile's 256 rows are in flight together; VEC = 0 loops over the row at run time.
template <int VEC>
__device__ __forceinline__ uint32_t token_mask(const RouteArgs& a, const int32_t* row, const int (&id)[VEC > 0 ? 4 * VEC : 1],
                                               float inv_e)
{
    const int n_exp = a.W * a.E;
    uint32_t m = 0;
    bool bad = false;
    auto take = [&](int e) {
        if (e >= 0 && e < n_exp)
            m |= 1u << expert_rank(e, a.E, inv_e);
        else
            bad = true;
    };
    if constexpr (VEC > 0) {
#pragma unroll
        for (int j = 0; j < 4 * VEC; ++j) take(id[j]);
    } else if (a.vec16) {
        for (int q = 0; q < (a.k >> 2); ++q) {
            const int4 v = __ldg(reinterpret_cast<const int4*>(row) + q);
            take(v.x);
            take(v.y);
            take(v.z);
            take(v.w);
        }
    } else {
        for (int j = 0; j < a.k; ++j) take(__ldg(row + j));
    }
    if (bad) record_status(a.status, EP_ERR_INDEX);
    return m;
}

// Bounded wait for a predecessor's scan word of this call (stamp); false if it never came.
__device__ __forceinline__ bool wait_word(const unsigned long long* fp, uint32_t stamp, int* status,
                                          unsigned long long& f)
{
    unsigned ns = 32;
    for (int it = 0;; ++it) {
        f = ld_relaxed_u64(fp);
        if ((uint32_t)(f >> 34) == stamp && ((f >> 32) & 3ull) != 0ull) return true;
        if (it >= kSpinLimit) {
            record_status(status, EP_ERR_DEVICE_TIMEOUT);
            return false;
        }
        __nanosleep(ns);
        if (ns < 256) ns <<= 1;
    }
}

// GROUPED: the tile also numbers the expert-grouped view.  Each token marks, for every expert
// it names (its first top-k slot naming it), its bit in a 256-bit mask of the tile per expert
// (shared memory, W*E masks); a token's slot in expert e's list is then the tile's exclusive
// prefix for e, from a decoupled lookback over the W*E expert columns like the one over ranks,
// plus the marked tokens before it in the tile.  The tile writes the slot into the expert map at
// the token's receive row on e's rank, the token index into src_info, and, for each source
// rank whose first token falls in the tile, every list's prefix at that token, from which the
// copy kernel that follows writes the counts and layout ranges.
constexpr int kGroupPrefetch = 4;   // GROUPED: predecessor words of a thread's first column read early

template <int VEC, bool GROUPED>
__global__ void __launch_bounds__(kRouteThreads) ep_route_kernel(const RouteArgs a)
{
    __shared__ int s_off[kMaxRanks + 1];
    __shared__ int s_warp[kRouteThreads / 32][kMaxRanks];   // warp totals, then warp prefixes
    __shared__ unsigned s_rbal[GROUPED ? kRouteThreads / 32 : 1][kMaxRanks];   // ballots per rank
    __shared__ int s_agg[kMaxRanks];
    __shared__ int s_excl[kMaxRanks];
    __shared__ int s_incl_at[kMaxRanks];
    __shared__ int s_done[kMaxRanks];
    __shared__ unsigned long long s_ticket, s_gen;
    extern __shared__ uint32_t s_dyn[];   // GROUPED: [W*E][8] token masks, [W*E] list prefixes,
                                          // [W*E][2] per-warp prefix bytes

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    allow_dependents();   // the copy kernel that follows may be scheduled (it waits for this one)
    probe_mark(a.probe, kProbeRoute, true);
    if (tid == 0) {
        // ticket[0]: next tile; ticket[1]: CTAs finished; ticket[2]: generation of this launch
        // (advanced only by the last CTA of the previous launch, which finished before this one)
        s_ticket = atomicAdd(a.ticket, 1ull);
        s_gen = ld_relaxed_u64(a.ticket + 2);
    }
    if (tid <= a.W) s_off[tid] = a.tok_off[tid];
    __syncthreads();
    const int tile = (int)s_ticket;                    // < gridDim.x == a.tiles
    const uint32_t stamp = (uint32_t)((s_gen + 1ull) & kStampMask);
    const int base = tile * kRouteTile;

    const int g = base + tid;
    const bool valid = g < a.N;
    int s = 0, t = 0;
    if (valid) {
        s = rank_of_token(s_off, a.W, g);
        t = g - s_off[s];
    }
    const int32_t* ids = a.idx + ((int64_t)s * a.M + t) * a.k;
    int id[VEC > 0 ? 4 * VEC : 1];
    if constexpr (VEC > 0) {
        if (valid) {
#pragma unroll
            for (int q = 0; q < VEC; ++q) {
                const int4 v = __ldg(reinterpret_cast<const int4*>(ids) + q);
                id[4 * q] = v.x;
                id[4 * q + 1] = v.y;
                id[4 * q + 2] = v.z;
                id[4 * q + 3] = v.w;
            }
        }
    }
    const float inv_e = __frcp_rn((float)a.E);
    const int n_exp = a.W * a.E;
    uint64_t firsts = 0;   // GROUPED: top-k slots that are the token's first naming their expert
    unsigned long long pre[GROUPED ? kGroupPrefetch : 1];   // GROUPED: prefetched expert-column words
    if constexpr (GROUPED) {
        for (int i = tid; i < n_exp * 8; i += kRouteThreads) s_dyn[i] = 0u;   // (loads in flight)
        __syncthreads();
        if (valid) {
            if constexpr (VEC > 0 && VEC <= 2) {         // top-k 4 and 8: compares in registers
#pragma unroll
                for (int j = 0; j < 4 * VEC; ++j) {
                    bool first = id[j] >= 0 && id[j] < n_exp;
#pragma unroll
                    for (int jj = 0; jj < j; ++jj) first = first && id[jj] != id[j];
                    if (first) {
                        firsts |= 1ull << j;
                        atomicOr(&s_dyn[id[j] * 8 + warp], 1u << lane);
                    }
                }
            } else {
                for (int j = 0; j < a.k; ++j) {
                    const int e = __ldg(ids + j);
                    if (e >= 0 && e < n_exp && !(atomicOr(&s_dyn[e * 8 + warp], 1u << lane) & (1u << lane)))
                        firsts |= 1ull << j;
                }
            }
        }
    }
    const uint32_t mask = valid ? token_mask<VEC>(a, ids, id, inv_e) : 0u;
    for (int r = 0; r < a.W; ++r) {
        const unsigned bal = __ballot_sync(0xffffffffu, (mask >> r) & 1u);
        if (lane == 0) {
            s_warp[warp][r] = __popc(bal);
            if constexpr (GROUPED) s_rbal[warp][r] = bal;
        }
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
    if constexpr (GROUPED) {   // the tile's total per expert column, and its prefix before each warp
        int* eex = reinterpret_cast<int*>(s_dyn + n_exp * 8);
        uint32_t* wpre = s_dyn + n_exp * 9;              // [n_exp][2]: 8 bytes, warp w's prefix in byte w
        for (int e = tid; e < n_exp; e += kRouteThreads) {
            int agg = 0;
            uint32_t lo = 0, hi = 0;
#pragma unroll
            for (int w = 0; w < 8; ++w) {
                if (w < 4) lo |= (uint32_t)agg << (8 * w);
                else hi |= (uint32_t)agg << (8 * (w - 4));
                agg += __popc(s_dyn[e * 8 + w]);         // at most 7 * 32 before warp 7
            }
            wpre[2 * e] = lo;
            wpre[2 * e + 1] = hi;
            eex[e] = agg;
            st_relaxed_u64(a.grp.eflags + (int64_t)tile * n_exp + e,
                           pack_flag(stamp, tile == 0 ? kFlagInclusive : kFlagAggregate, (uint32_t)agg));
        }
        // the first column's nearest predecessor words, read now so that their latency overlaps
        // the lookback over the rank columns
#pragma unroll
        for (int b = 0; b < kGroupPrefetch; ++b)
            pre[b] = tid < n_exp && tile - 1 - b >= 0
                         ? ld_relaxed_u64(a.grp.eflags + (int64_t)(tile - 1 - b) * n_exp + tid) : 0ull;
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
                have = wait_word(a.flags + (int64_t)j * a.W + r, stamp, a.status, f);
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

    if constexpr (GROUPED) {
        // lookback over the expert columns, one thread per column: sum predecessors' words back
        // to the first INCLUSIVE one (tiles before this one were all issued earlier)
        int* eex = reinterpret_cast<int*>(s_dyn + n_exp * 8);
        const uint32_t* wpre = s_dyn + n_exp * 9;
        for (int e = tid; e < n_exp; e += kRouteThreads) {
            int excl = 0;
            if (tile > 0) {
                const int agg = eex[e];
                for (int j = tile - 1; j >= 0; --j) {
                    unsigned long long f = 0;
                    const int b = tile - 1 - j;
#pragma unroll
                    for (int q = 0; q < kGroupPrefetch; ++q)
                        if (q == b && e == tid) f = pre[q];           // read before the rank lookback
                    if (!((uint32_t)(f >> 34) == stamp && ((f >> 32) & 3ull) != 0ull) &&
                        !wait_word(a.grp.eflags + (int64_t)j * n_exp + e, stamp, a.status, f))
                        break;
                    excl += (int)(uint32_t)f;
                    if (((f >> 32) & 3ull) == kFlagInclusive) break;
                }
                st_relaxed_u64(a.grp.eflags + (int64_t)tile * n_exp + e,
                               pack_flag(stamp, kFlagInclusive, (uint32_t)(excl + agg)));
            }
            eex[e] = excl;
        }
        __syncthreads();
        // list prefix of expert e before position pos (0..255) of the tile
        auto prefix_at = [&](int e, int pos) {
            const int w = pos >> 5, b = pos & 31;
            const int before = (int)((wpre[2 * e + (w >> 2)] >> (8 * (w & 3))) & 0xFFu);
            return eex[e] + before + __popc(s_dyn[e * 8 + w] & ((1u << b) - 1u));
        };
        // each first slot: the list slot, written at the token's receive row on the expert's rank
        const unsigned lt_ = lanemask_lt();
        auto place = [&](int j, int e) {
            const int r = expert_rank(e, a.E, inv_e);
            const int slot = prefix_at(e, tid);
            const int row = s_excl[r] + s_warp[warp][r] + __popc(s_rbal[warp][r] & lt_);
            if (EP_IN_BOUNDS(row >= 0 && row < a.rows && slot >= 0 && slot < a.rows, a.status)) {
                a.grp.map[((int64_t)r * a.rows + row) * a.k + j] = slot;
                a.grp.src_info[(int64_t)e * a.rows + slot] = t;
            }
        };
        if constexpr (VEC > 0 && VEC <= 2) {             // top-k 4 and 8: the row in registers
#pragma unroll
            for (int j = 0; j < 4 * VEC; ++j)
                if ((firsts >> j) & 1ull) place(j, id[j]);
        } else {
            for (uint64_t m = firsts; m; m &= m - 1) {
                const int j = __ffsll((long long)m) - 1;
                place(j, __ldg(ids + j));
            }
        }
        // every list's prefix at each source rank's first token that lies in this tile (the end
        // of the tokens, N, belongs to the last tile)
        for (int sb = 0; sb <= a.W; ++sb) {
            const int b = s_off[sb];
            if (!((b >= base && b < base + kRouteTile) || (b == a.N && tile == a.tiles - 1))) continue;
            const int pos = b - base;                       // 0..256 tokens of the tile before b
            for (int e = tid; e < n_exp; e += kRouteThreads)
                a.grp.bnd[(int64_t)sb * n_exp + e] =
                    pos < kRouteTile ? prefix_at(e, pos) : prefix_at(e, kRouteTile - 1) +
                                                            (int)((s_dyn[e * 8 + 7] >> 31) & 1u);
        }
    }

    int32_t* fwd_row = a.fwd + ((int64_t)s * a.M + t) * a.F;
    const unsigned lt = lanemask_lt();
    int j = 0;
    for (int r = 0; r < a.W; ++r) {
        const unsigned bit = (mask >> r) & 1u;
        const unsigned bal = __ballot_sync(0xffffffffu, bit);
        if (bit) {
            const int slot = s_excl[r] + s_warp[warp][r] + __popc(bal & lt);
            if (EP_IN_BOUNDS(slot >= 0 && slot < a.rows, a.status)) {
                a.src_pos[(int64_t)r * a.rows + slot] = (int32_t)((int64_t)s * a.rows + t);
                fwd_row[j++] = (int32_t)((int64_t)r * a.rows + slot);
            }
        }
    }
    if (valid)
        for (; j < a.F; ++j) fwd_row[j] = -1;

    // the last CTA to finish (every CTA has taken its ticket by then) resets the ticket and
    // advances the generation for the next launch
    probe_mark(a.probe, kProbeRoute, false);
    __syncthreads();
    if (tid == 0) {
        __threadfence();
        if (atomicAdd(a.ticket + 1, 1ull) == (unsigned long long)gridDim.x - 1) {
            atomicExch(a.ticket, 0ull);
            atomicExch(a.ticket + 1, 0ull);
            atomicExch(a.ticket + 2, s_gen + 1ull);
        }
    }
}

template <int VEC, bool GROUPED>
cudaError_t launch_vec(const RouteArgs& a, cudaStream_t stream)
{
    const size_t smem = GROUPED ? (size_t)a.W * a.E * 11 * sizeof(uint32_t) : 0;
    ep_route_kernel<VEC, GROUPED><<<a.tiles, kRouteThreads, smem, stream>>>(a);
    return cudaGetLastError();
}

template <bool GROUPED>
cudaError_t launch_widths(const RouteArgs& a, cudaStream_t stream)
{
    // compiled row widths: top-k 4, 8 (the pages' specialised case), 16; others loop at run time
    if (!a.vec16) return launch_vec<0, GROUPED>(a, stream);
    switch (a.k) {
    case 4: return launch_vec<1, GROUPED>(a, stream);
    case 8: return launch_vec<2, GROUPED>(a, stream);
    case 16: return launch_vec<4, GROUPED>(a, stream);
    default: return launch_vec<0, GROUPED>(a, stream);
    }
}

}  // namespace

cudaError_t launch_route(const RouteArgs& a, cudaStream_t stream) { return launch_widths<false>(a, stream); }

cudaError_t launch_route_grouped(const RouteArgs& a, cudaStream_t stream)
{
    if ((int64_t)a.W * a.E > kRouteGroupMaxExperts) return cudaErrorInvalidValue;
    return launch_widths<true>(a, stream);
}

}  // namespace ep

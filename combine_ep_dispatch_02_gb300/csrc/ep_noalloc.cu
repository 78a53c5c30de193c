// ep_noalloc.cu -- the routing step of dispatch for callers that cannot allocate device memory.
//
// Some callers may not call cudaMalloc at all: a serving runtime that has handed nearly all of
// HBM to its own pool allocator up front (a stray cudaMalloc then either fails or fragments the
// pool), or a plug-in that runs inside a host framework whose rules forbid allocation on the hot
// path (cudaMalloc can also stall the whole device while it maps memory).  ep_plan_create does
// allocate, so it is not usable there.  ep_route_noalloc gives those callers the routing step --
// distinct destination ranks, receive-row numbering, reverse map, forward map, receive counts --
// with every output in memory the caller already owns and the only scratch the routing kernel
// needs (its decoupled-lookback scan words and tile ticket) in a fixed array compiled into this
// library.
//
// The scratch array is a file-scope static __device__ array: every GPU that loads the library
// holds its kNoAllocScratchWords * 8 bytes until the process exits.  Host code only knows the
// array's name as a host-side stand-in, so the first call on each device looks up its device
// address with cudaGetSymbolAddress (with that device current) and caches it; that first call
// should be made before any stream capture begins.  The cached address belongs to the device's
// primary context: after cudaDeviceReset on that device it is stale, so a process that resets a
// device must not call this entry point on it again.  Every pointer argument is checked to be
// device memory usable from the current device before anything is enqueued.
#include <cstdio>
#include <mutex>

#include "ep_common.cuh"

namespace ep {
int record_error(int code, const char* msg);   // sets the message read by ep_last_error()
}

namespace {

constexpr int kNoAllocScratchWords = 16384;   // 128 KB: the routing control words + the scan words
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned long long ep_noalloc_scratch[kNoAllocScratchWords];

std::mutex g_mu;
unsigned long long* g_scratch[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up once per device.
int scratch_of_current_device(unsigned long long** out)
{
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return ep::record_error(EP_ERR_CUDA, cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices) return ep::record_error(EP_ERR_ARG, "device ordinal out of range");
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, ep_noalloc_scratch);
        if (e != cudaSuccess || !p) {
            char msg[256];
            snprintf(msg, sizeof msg, "cudaGetSymbolAddress of the routing scratch failed: %s",
                     cudaGetErrorString(e));
            return ep::record_error(EP_ERR_CUDA, msg);
        }
        g_scratch[dev] = static_cast<unsigned long long*>(p);
    }
    *out = g_scratch[dev];
    return EP_OK;
}

bool aligned4(const void* p) { return ((uintptr_t)p & 3u) == 0; }

// The kernel runs on the current device and dereferences every pointer there, so each must be
// memory that device can use: device memory of another GPU, or pageable host memory the
// runtime does not know, is rejected on the host rather than left to fault on the device.
int check_on_device(const void* p, const char* what, int dev)
{
    cudaPointerAttributes at{};
    cudaError_t e = cudaPointerGetAttributes(&at, p);
    char msg[256];
    if (e != cudaSuccess) {
        cudaGetLastError();
        snprintf(msg, sizeof msg, "ep_route_noalloc: %s: cudaPointerGetAttributes failed: %s", what,
                 cudaGetErrorString(e));
        return ep::record_error(EP_ERR_ARG, msg);
    }
    if (at.type == cudaMemoryTypeUnregistered) {
        snprintf(msg, sizeof msg, "ep_route_noalloc: %s is pageable host memory, not device memory", what);
        return ep::record_error(EP_ERR_ARG, msg);
    }
    if (at.type == cudaMemoryTypeDevice && at.device != dev) {
        snprintf(msg, sizeof msg, "ep_route_noalloc: %s is on device %d, the call runs on device %d", what,
                 at.device, dev);
        return ep::record_error(EP_ERR_ARG, msg);
    }
    return EP_OK;
}

}  // namespace

extern "C" int ep_route_noalloc(int W, int E, int k, int M, const int32_t* indices,
                                const int32_t* n_tok_host, int32_t* src_token_pos,
                                int32_t* recv_count, int32_t* fwd_map, int32_t* device_status,
                                void* stream)
{
    char msg[256];
    if (W < 1 || W > ep::kMaxRanks || E < 1 || k < 1 || k > ep::kMaxTopk || M < 1)
        return ep::record_error(EP_ERR_ARG, "ep_route_noalloc: W must be 1..32, topk 1..64, "
                                            "experts_per_rank and max_tok_per_rank >= 1");
    if ((int64_t)W * E >= (int64_t)1 << 31 || (int64_t)W * W * M >= (int64_t)1 << 31)
        return ep::record_error(EP_ERR_ARG, "ep_route_noalloc: W*E or W*W*M reaches 2^31");
    if (!indices || !n_tok_host || !src_token_pos || !recv_count || !fwd_map || !device_status ||
        !aligned4(indices) || !aligned4(src_token_pos) || !aligned4(recv_count) ||
        !aligned4(fwd_map) || !aligned4(device_status))
        return ep::record_error(EP_ERR_ARG, "ep_route_noalloc: a pointer is NULL or not 4-byte aligned");
    const int64_t rows = (int64_t)W * M;
    const int tiles = (int)((rows + ep::kRouteTile - 1) / ep::kRouteTile);
    const int64_t words = ep::kRouteControlWords + (int64_t)tiles * W;
    if (words > kNoAllocScratchWords) {
        snprintf(msg, sizeof msg,
                 "ep_route_noalloc: W=%d, max_tok_per_rank=%d needs %lld scan words; the static "
                 "scratch holds %d (W * ceil(W*M/256) must stay within %d)",
                 W, M, (long long)words, kNoAllocScratchWords, kNoAllocScratchWords - ep::kRouteControlWords);
        return ep::record_error(EP_ERR_ARG, msg);
    }
    ep::RouteArgs a{};
    a.tok_off[0] = 0;
    for (int s = 0; s < W; ++s) {
        if (n_tok_host[s] < 0 || n_tok_host[s] > M) {
            snprintf(msg, sizeof msg, "ep_route_noalloc: n_tok[%d]=%d outside 0..%d", s, n_tok_host[s], M);
            return ep::record_error(n_tok_host[s] < 0 ? EP_ERR_ARG : EP_ERR_CAPACITY, msg);
        }
        a.tok_off[s + 1] = a.tok_off[s] + n_tok_host[s];
    }
    unsigned long long* scratch = nullptr;
    int rc = scratch_of_current_device(&scratch);
    if (rc != EP_OK) return rc;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return ep::record_error(EP_ERR_CUDA, "ep_route_noalloc: cudaGetDevice");
    const void* ptrs[5] = {indices, src_token_pos, recv_count, fwd_map, device_status};
    const char* names[5] = {"indices", "src_token_pos", "recv_count", "fwd_map", "device_status"};
    for (int i = 0; i < 5; ++i)
        if ((rc = check_on_device(ptrs[i], names[i], dev)) != EP_OK) return rc;

    // One routing CTA per 256 tokens of this call (at least one, which writes the counts of an
    // empty call).  The array keeps the previous call's words: the control words (ticket,
    // finished CTAs, generation) must restart at 0 and the scan words this call uses must read
    // "not published" for its stamp, so they are cleared first.  The device status is an
    // output and starts clear as well.
    const int n = a.tok_off[W];
    const int call_tiles = n > 0 ? (n + ep::kRouteTile - 1) / ep::kRouteTile : 1;
    const int64_t call_words = ep::kRouteControlWords + (int64_t)call_tiles * W;
    cudaStream_t s = (cudaStream_t)stream;
    cudaError_t e = cudaMemsetAsync(scratch, 0, (size_t)call_words * sizeof(unsigned long long), s);
    if (e == cudaSuccess) e = cudaMemsetAsync(device_status, 0, sizeof(int32_t), s);
    if (e != cudaSuccess) return ep::record_error(EP_ERR_CUDA, cudaGetErrorString(e));

    a.idx = indices;
    a.fwd = fwd_map;
    a.src_pos = src_token_pos;
    a.recv_count = recv_count;
    a.ticket = scratch;
    a.flags = scratch + ep::kRouteControlWords;
    a.status = device_status;
    a.rows = rows;
    a.W = W; a.E = E; a.k = k; a.F = W < k ? W : k; a.M = M;
    a.N = a.tok_off[W];
    a.tiles = call_tiles;
    a.vec16 = (k % 4 == 0) && ((uintptr_t)indices % 16 == 0);
    e = ep::launch_route(a, s);
    if (e != cudaSuccess) return ep::record_error(EP_ERR_CUDA, cudaGetErrorString(e));
    return EP_OK;
}

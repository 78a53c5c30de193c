// ep_api.cu -- the C ABI declared in include/ep.h: plan lifetime, host-side validation, kernel
// launches.  Every condition the host can check fails here with a code and a message, before
// any launch (the pages' staging refactor likewise validates on the host and reports a
// RuntimeError naming the argument rather than risking a device fault).
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <new>

#include "ep_common.cuh"

using namespace ep;

struct ep_plan {
    int W, E, k, H, dtype, sd, M, F, elem_bytes, tiles;
    bool quantise;       // BF16 input quantised by dispatch: FP8 e4m3 or MX FP4 rows + scales
    bool fp4;            // EP_BF16_TO_MXFP4
    int64_t rows;        // W*M receive rows per rank
    int64_t row_bytes;   // received payload bytes per row
    int device, num_sms, variant;

    void* base;
    size_t bytes;
    uint8_t* recv_x;
    int32_t* recv_idx;
    float* recv_w;
    float* recv_scales;
    int32_t* src_pos;
    int32_t* fwd;
    int32_t* recv_count;
    int32_t* expert_map;
    int32_t* scan_cnt;            // two-pass grouping scan counts, or NULL
    int scan_chunks;
    unsigned long long* eflags;   // grouped routing: expert-column lookback words, or NULL
    int32_t* bnd;                 // grouped routing: list prefixes at source boundaries
    unsigned long long* flags;
    unsigned long long* ticket;
    unsigned long long* queues;   // kQueues work queues of two words each, after the ticket
    int* status;

    // host state of the live dispatch
    uint64_t epoch, grouped_epoch;
    bool routed, live, has_w;
    const int32_t* routed_idx;
    int N;
    int tok_off[kMaxRanks + 1];
};

namespace {

thread_local char g_err[512] = "";

int fail(int code, const char* fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
    return code;
}

int cuda_fail(cudaError_t e, const char* what)
{
    return fail(EP_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

size_t align256(size_t v) { return (v + 255) & ~(size_t)255; }

struct Layout {
    size_t recv_x, recv_idx, recv_w, recv_scales, src_pos, fwd, scan_cnt, recv_count, expert_map, flags,
        eflags, bnd, ticket, status, total;
};

// Whether the routing kernel numbers the grouped view itself (ep_dispatch_grouped in two launches):
// up to kRouteGroupMaxExperts experts in all, with lookback words [tiles][W*E] within
// kRouteGroupMaxFlagBytes.  Otherwise the grouped dispatch runs the separate grouping scan.
bool route_groups(int W, int E, int64_t tiles)
{
    const int64_t n_exp = (int64_t)W * E;
    return n_exp <= kRouteGroupMaxExperts && tiles * n_exp * 8 <= kRouteGroupMaxFlagBytes;
}

// 1024-row chunks of a rank's receive capacity when the grouping scan runs in two passes (three
// chunks or more, per-chunk counts within kScanMaxBytes), else 0
int64_t scan_chunks_of(int W, int E, int64_t rows)
{
    const int64_t chunks = (rows + kScanChunk - 1) / kScanChunk;
    if (chunks < kScanMinChunks) return 0;
    const int64_t bytes = (int64_t)W * E * chunks * W * 4;
    return bytes <= kScanMaxBytes ? chunks : 0;
}

// bytes of one RECEIVED payload row (0 for an unknown dtype)
int64_t row_bytes_of(int dtype, int64_t H)
{
    switch (dtype) {
    case EP_BF16:
    case EP_FP16: return 2 * H;
    case EP_FP8_E4M3:
    case EP_BF16_TO_FP8_E4M3: return H;
    case EP_BF16_TO_MXFP4: return H / 2;
    default: return 0;
    }
}

bool quantising(int dtype) { return dtype == EP_BF16_TO_FP8_E4M3 || dtype == EP_BF16_TO_MXFP4; }

// scale_dim the plan actually uses: the quantising dtypes fix it at hidden / 128 (FP32 scales
// per 128 elements, or the H/32 e8m0 bytes of MX FP4 packed four to a word)
int effective_sd(int dtype, int H, int sd) { return quantising(dtype) ? H / 128 : sd; }

int check_shape(int W, int E, int k, int H, int dtype, int sd, int M)
{
    if (W < 1 || W > kMaxRanks) return fail(EP_ERR_ARG, "W=%d outside 1..%d", W, kMaxRanks);
    if (E < 1) return fail(EP_ERR_ARG, "experts_per_rank=%d < 1", E);
    if ((int64_t)W * E >= (int64_t)1 << 31) return fail(EP_ERR_ARG, "W*experts_per_rank >= 2^31");
    if (k < 1 || k > kMaxTopk) return fail(EP_ERR_ARG, "topk=%d outside 1..%d", k, kMaxTopk);
    if (row_bytes_of(dtype, 2) == 0) return fail(EP_ERR_ARG, "dtype=%d is not an ep_dtype", dtype);
    if (H < 1 || row_bytes_of(dtype, H) % 16 != 0 || (dtype == EP_BF16_TO_MXFP4 && H % 2 != 0))
        return fail(EP_ERR_ARG, "hidden=%d: a received row of %lld bytes is not a positive multiple of 16",
                    H, (long long)row_bytes_of(dtype, H));
    if (2 * (int64_t)H >= (int64_t)1 << 31) return fail(EP_ERR_ARG, "hidden=%d too large", H);
    if (sd < 0 || sd > 65536) return fail(EP_ERR_ARG, "scale_dim=%d outside 0..65536", sd);
    if (quantising(dtype)) {
        if (H % 128 != 0) return fail(EP_ERR_ARG, "hidden=%d: the quantising dtype needs hidden %% 128 == 0", H);
        if (sd != 0 && sd != H / 128)
            return fail(EP_ERR_ARG, "scale_dim=%d: the quantising dtype uses hidden/128 = %d scales", sd, H / 128);
    }
    if (M < 1) return fail(EP_ERR_ARG, "max_tok_per_rank=%d < 1", M);
    if ((int64_t)W * W * M >= (int64_t)1 << 31)
        return fail(EP_ERR_ARG, "W*W*max_tok_per_rank >= 2^31 overflows the int32 src_token_pos");
    // The combine kernels address a token's rows in 32-bit counts of 16-byte vectors of the
    // 16-bit expert outputs [W][W*M][H] (FP8 wire: 16-byte pieces of 16 codes; MX FP4: 32-element
    // blocks), so that buffer must stay below 2^32 vectors = 64 GiB: W*W*M*H < 2^35.
    if ((int64_t)W * W * M * H >= (int64_t)1 << 35)
        return fail(EP_ERR_ARG,
                    "W*W*max_tok_per_rank*hidden >= 2^35: the 16-bit expert outputs combine reads "
                    "([W][W*M][H], %lld bytes) reach 64 GiB, past its 32-bit row offsets",
                    (long long)((int64_t)W * W * M * H * 2));
    return EP_OK;
}

Layout layout_of(int W, int E, int k, int H, int dtype, int sd, int M)
{
    Layout L{};
    const size_t rows = (size_t)W * M;
    const int F = W < k ? W : k;
    const int tiles = (int)((rows + kRouteTile - 1) / kRouteTile);
    size_t o = 0;
    auto put = [&](size_t& field, size_t bytes) {
        field = o;
        o += align256(bytes);
    };
    put(L.recv_x, (size_t)W * rows * row_bytes_of(dtype, H));
    put(L.recv_idx, (size_t)W * rows * k * 4);
    put(L.recv_w, (size_t)W * rows * k * 4);
    put(L.recv_scales, (size_t)W * rows * sd * 4);
    put(L.src_pos, (size_t)W * rows * 4);
    put(L.fwd, rows * F * 4);
    put(L.scan_cnt, (size_t)W * E * scan_chunks_of(W, E, (int64_t)rows) * W * 4);
    put(L.recv_count, (size_t)W * 4);
    put(L.expert_map, (size_t)W * rows * k * 4);
    put(L.flags, (size_t)tiles * W * 8);
    const bool rg = route_groups(W, E, tiles);
    put(L.eflags, rg ? (size_t)tiles * W * E * 8 : 0);
    put(L.bnd, rg ? (size_t)(W + 1) * W * E * 4 : 0);
    // routing control, the work queues, then the phase probes: one 256-byte block
    static_assert(kRouteControlWords + 2 * kQueues <= kProbeWordOffset && kProbeWordOffset + 2 * kProbePhases <= 32,
                  "the control block holds the routing words, the queues and the probes");
    put(L.ticket, 256);
    put(L.status, 4);
    L.total = o;
    return L;
}

struct DeviceGuard {
    int prev = -1;
    bool ok = true;
    explicit DeviceGuard(int dev)
    {
        if (cudaGetDevice(&prev) != cudaSuccess) { ok = false; return; }
        if (prev != dev && cudaSetDevice(dev) != cudaSuccess) ok = false;
    }
    ~DeviceGuard()
    {
        int cur = -1;
        if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
    }
};

// The plan's phase probe words (earliest start, latest end per phase) in its control block.
unsigned long long* plan_probe(const ep_plan* p) { return p->ticket + kProbeWordOffset; }

// Probe words back to "nothing recorded": earliest start ~0, latest end 0.
cudaError_t reset_probes(const ep_plan* p)
{
    unsigned long long init[2 * kProbePhases];
    for (int i = 0; i < kProbePhases; ++i) {
        init[2 * i] = ~0ull;
        init[2 * i + 1] = 0ull;
    }
    return cudaMemcpy(plan_probe(p), init, sizeof init, cudaMemcpyHostToDevice);
}

int pick_chunk_elems(const ep_plan* p, int N)
{
    switch (p->variant) {
    case EP_VARIANT_WHOLE_ROW: return p->H;
    case EP_VARIANT_TILED_512: return p->H < 512 ? p->H : 512;
    case EP_VARIANT_TILED_1024: return p->H < 1024 ? p->H : 1024;
    default: break;
    }
    // Whole rows once there are enough tokens to give every resident warp four rows, so the
    // scatter's work queue can even out tokens of different destination counts; otherwise
    // split rows into 1024-element slices, and into 512-element ones when even those leave
    // warps idle (the pages use 512- or 1024-element tiles up to 256 tokens per source rank).
    const int64_t warps = (int64_t)p->num_sms * 32;
    if (N >= 4 * warps || p->H <= 1024) return p->H;
    if ((int64_t)N * ((p->H + 1023) / 1024) >= warps) return 1024;
    return 512;
}

// The copy kernels number their work units (tokens x row slices) in 32 bits.
int check_units(int N, int chunks, const char* who)
{
    if ((int64_t)N * chunks >= (int64_t)1 << 31)
        return fail(EP_ERR_ARG, "%s: %d tokens x %d row slices >= 2^31 work units; use whole rows", who, N,
                    chunks);
    return EP_OK;
}

}  // namespace

namespace ep {
// lets other translation units of the library report a message through ep_last_error()
int record_error(int code, const char* msg) { return fail(code, "%s", msg); }
}  // namespace ep

extern "C" {

const char* ep_last_error(void) { return g_err; }

const char* ep_strerror(int code)
{
    switch (code) {
    case EP_OK: return "ok";
    case EP_ERR_ARG: return "invalid argument";
    case EP_ERR_ALLOC: return "device allocation failed";
    case EP_ERR_CUDA: return "CUDA error";
    case EP_ERR_STATE: return "no live dispatch for this epoch";
    case EP_ERR_CAPACITY: return "token count exceeds max_tok_per_rank";
    case EP_ERR_INDEX: return "expert id out of range (skipped on the device)";
    case EP_ERR_DEVICE_TIMEOUT: return "device wait timed out";
    case EP_ERR_DEVICE_BOUNDS: return "device index out of bounds (skipped; EP_CHECKS build)";
    default: return "unknown status";
    }
}

size_t ep_plan_device_bytes(int W, int E, int k, int H, int dtype, int sd, int M)
{
    char saved[sizeof g_err];
    memcpy(saved, g_err, sizeof g_err);
    const int rc = check_shape(W, E, k, H, dtype, sd, M);
    memcpy(g_err, saved, sizeof g_err);
    if (rc != EP_OK) return 0;
    return layout_of(W, E, k, H, dtype, effective_sd(dtype, H, sd), M).total;
}

int ep_plan_create(ep_plan** out, int W, int E, int k, int H, int dtype, int sd, int M)
{
    if (!out) return fail(EP_ERR_ARG, "out is NULL");
    *out = nullptr;
    int rc = check_shape(W, E, k, H, dtype, sd, M);
    if (rc != EP_OK) return rc;

    ep_plan* p = new (std::nothrow) ep_plan();
    if (!p) return fail(EP_ERR_ALLOC, "host allocation of the plan failed");
    p->W = W; p->E = E; p->k = k; p->H = H; p->dtype = dtype; p->sd = sd; p->M = M;
    p->F = W < k ? W : k;
    p->elem_bytes = dtype == EP_BF16 || dtype == EP_FP16 ? 2 : 1;   // BF16/FP16, else a byte stream
    p->rows = (int64_t)W * M;
    p->row_bytes = row_bytes_of(dtype, H);
    p->tiles = (int)((p->rows + kRouteTile - 1) / kRouteTile);
    p->variant = EP_VARIANT_AUTO;

    cudaError_t e = cudaGetDevice(&p->device);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&p->num_sms, cudaDevAttrMultiProcessorCount, p->device);
    if (e != cudaSuccess) { delete p; return cuda_fail(e, "ep_plan_create: device query"); }

    sd = effective_sd(dtype, H, sd);
    p->sd = sd;
    p->quantise = quantising(dtype);
    p->fp4 = dtype == EP_BF16_TO_MXFP4;
    const Layout L = layout_of(W, E, k, H, dtype, sd, M);
    p->bytes = L.total;
    e = cudaMalloc(&p->base, L.total);
    if (e != cudaSuccess) {
        cudaGetLastError();
        delete p;
        return fail(EP_ERR_ALLOC, "cudaMalloc of %zu bytes failed: %s", L.total, cudaGetErrorString(e));
    }
    char* b = (char*)p->base;
    p->recv_x = (uint8_t*)(b + L.recv_x);
    p->recv_idx = (int32_t*)(b + L.recv_idx);
    p->recv_w = (float*)(b + L.recv_w);
    p->recv_scales = sd ? (float*)(b + L.recv_scales) : nullptr;
    p->src_pos = (int32_t*)(b + L.src_pos);
    p->fwd = (int32_t*)(b + L.fwd);
    p->recv_count = (int32_t*)(b + L.recv_count);
    p->expert_map = (int32_t*)(b + L.expert_map);
    p->scan_chunks = (int)scan_chunks_of(W, E, p->rows);
    p->scan_cnt = p->scan_chunks ? (int32_t*)(b + L.scan_cnt) : nullptr;
    p->flags = (unsigned long long*)(b + L.flags);
    p->eflags = route_groups(W, E, p->tiles) ? (unsigned long long*)(b + L.eflags) : nullptr;
    p->bnd = p->eflags ? (int32_t*)(b + L.bnd) : nullptr;
    p->ticket = (unsigned long long*)(b + L.ticket);
    p->queues = p->ticket + kRouteControlWords;
    p->status = (int*)(b + L.status);
    // the control words start at zero once; scan flags are stamped per call after that
    e = cudaMemset(b + L.recv_count, 0, L.total - L.recv_count);
    if (e == cudaSuccess) e = reset_probes(p);
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) {
        cudaFree(p->base);
        delete p;
        return cuda_fail(e, "ep_plan_create: clearing control words");
    }
    *out = p;
    return EP_OK;
}

int ep_plan_destroy(ep_plan* p)
{
    if (!p) return EP_OK;
    DeviceGuard g(p->device);
    cudaError_t e = cudaDeviceSynchronize();
    cudaError_t e2 = cudaFree(p->base);
    delete p;
    if (e != cudaSuccess) return cuda_fail(e, "ep_plan_destroy: synchronize");
    if (e2 != cudaSuccess) return cuda_fail(e2, "ep_plan_destroy: cudaFree");
    return EP_OK;
}

int ep_plan_set_variant(ep_plan* p, int variant)
{
    if (!p) return fail(EP_ERR_ARG, "plan is NULL");
    if (variant < EP_VARIANT_AUTO || variant > EP_VARIANT_TILED_1024)
        return fail(EP_ERR_ARG, "variant=%d is not an ep_variant", variant);
    p->variant = variant;
    return EP_OK;
}

static void fill_out(const ep_plan* p, ep_dispatch_out* out)
{
    out->recv_x = p->recv_x;
    out->recv_idx = p->recv_idx;
    out->recv_w = p->has_w ? p->recv_w : nullptr;
    out->recv_scales = p->recv_scales;
    out->recv_count = p->recv_count;
    out->src_token_pos = p->src_pos;
    out->rows_per_rank = p->rows;
    out->epoch = p->epoch;
}

// Arguments of the routing step of a call, after validating indices and the token counts.
static int route_prepare(ep_plan* p, const int32_t* indices, const int32_t* n_tok_host, RouteArgs& a,
                         int (&off)[kMaxRanks + 1])
{
    if (!p) return fail(EP_ERR_ARG, "plan is NULL");
    if (!indices || !aligned(indices, 4)) return fail(EP_ERR_ARG, "indices is NULL or not 4-byte aligned");
    if (!n_tok_host) return fail(EP_ERR_ARG, "n_tok_host is NULL");
    off[0] = 0;
    for (int s = 0; s < p->W; ++s) {
        if (n_tok_host[s] < 0) return fail(EP_ERR_ARG, "n_tok[%d]=%d < 0", s, n_tok_host[s]);
        if (n_tok_host[s] > p->M)
            return fail(EP_ERR_CAPACITY, "n_tok[%d]=%d exceeds max_tok_per_rank=%d", s, n_tok_host[s], p->M);
        off[s + 1] = off[s] + n_tok_host[s];
    }
    a = RouteArgs{};
    a.probe = plan_probe(p);
    a.idx = indices; a.fwd = p->fwd; a.src_pos = p->src_pos; a.recv_count = p->recv_count;
    a.flags = p->flags; a.ticket = p->ticket; a.status = p->status;
    a.rows = p->rows; a.W = p->W; a.E = p->E; a.k = p->k; a.F = p->F; a.M = p->M;
    a.N = off[p->W];
    // one CTA per 256 tokens of this call (at least one, which writes the counts of an empty
    // call); the plan's scan words cover the largest call, p->tiles tiles
    a.tiles = a.N > 0 ? (a.N + kRouteTile - 1) / kRouteTile : 1;
    a.vec16 = (p->k % 4 == 0) && aligned(indices, 16);
    for (int s = 0; s <= p->W; ++s) a.tok_off[s] = off[s];
    return EP_OK;
}

// Host state of the plan once a routing step is enqueued: a new epoch, routed, not yet live.
static void route_commit(ep_plan* p, const RouteArgs& a, const int (&off)[kMaxRanks + 1], const int32_t* indices)
{
    p->epoch += 1;
    p->routed = true;
    p->live = false;
    p->has_w = false;
    p->routed_idx = indices;
    p->N = a.N;
    memcpy(p->tok_off, off, sizeof off);
}

// The routing step of every dispatch; with grp set (the grouped dispatch on a plan that has the
// expert columns' words) the routing kernel also numbers the grouped view.
static int route_call(ep_plan* p, const int32_t* indices, const int32_t* n_tok_host, void* stream,
                      ep_dispatch_out* out, const RouteGroupArgs* grp)
{
    RouteArgs a;
    int off[kMaxRanks + 1];
    int rc = route_prepare(p, indices, n_tok_host, a, off);
    if (rc != EP_OK) return rc;
    DeviceGuard g(p->device);
    if (!g.ok) return fail(EP_ERR_CUDA, "cannot select the plan's device %d", p->device);
    cudaError_t e;
    if (grp) {
        a.grp = *grp;
        a.grp.eflags = p->eflags;
        a.grp.bnd = p->bnd;
        a.grp.map = p->expert_map;
        e = launch_route_grouped(a, (cudaStream_t)stream);
    } else {
        e = launch_route(a, (cudaStream_t)stream);
    }
    if (e != cudaSuccess) return cuda_fail(e, "ep_dispatch_route: launch");
    route_commit(p, a, off, indices);
    if (out) {
        fill_out(p, out);
        out->recv_w = p->recv_w;   // filled by the scatter when it is given weights
    }
    return EP_OK;
}

int ep_dispatch_route(ep_plan* p, const int32_t* indices, const int32_t* n_tok_host, void* stream,
                      ep_dispatch_out* out)
{
    return route_call(p, indices, n_tok_host, stream, out, nullptr);
}

// Arguments of the payload scatter of the routed call, after validating the payload arguments.
static int scatter_prepare(ep_plan* p, const void* x, const float* weights, const float* scales,
                           const int32_t* indices, ScatterArgs& a)
{
    if (!p) return fail(EP_ERR_ARG, "plan is NULL");
    if (!p->routed) return fail(EP_ERR_STATE, "ep_dispatch_scatter without a preceding ep_dispatch_route");
    if (!x || !aligned(x, 16)) return fail(EP_ERR_ARG, "x is NULL or not 16-byte aligned");
    if (weights && !aligned(weights, 4)) return fail(EP_ERR_ARG, "weights not 4-byte aligned");
    if (p->quantise) {
        if (scales) return fail(EP_ERR_ARG, "the quantising dtype computes its scales: pass NULL");
    } else {
        if (p->sd > 0 && (!scales || !aligned(scales, 4)))
            return fail(EP_ERR_ARG, "scale_dim=%d needs a 4-byte aligned scales array", p->sd);
        if (p->sd == 0 && scales) return fail(EP_ERR_ARG, "scales given but the plan has scale_dim 0");
    }
    if (indices != p->routed_idx) return fail(EP_ERR_ARG, "indices differ from the routed ones");
    a = ScatterArgs{};
    a.status = p->status; a.probe = plan_probe(p);
    a.work.q = p->queues + 2 * kQueueDispatch;
    a.x = (const uint8_t*)x; a.w = weights; a.scales = scales; a.idx = indices; a.fwd = p->fwd;
    a.recv_x = p->recv_x; a.recv_idx = p->recv_idx; a.recv_w = p->recv_w; a.recv_scales = p->recv_scales;
    a.row_bytes = p->row_bytes;
    a.W = p->W; a.k = p->k; a.F = p->F; a.M = p->M; a.sd = p->sd; a.N = p->N;
    const int ce = pick_chunk_elems(p, p->N);
    // quantising scatters take the slice in elements (their source rows are BF16)
    a.chunk_bytes = p->quantise ? ce : ce * p->elem_bytes;
    a.chunks = (int)((p->H + ce - 1) / ce);
    if (int rc = check_units(a.N, a.chunks, "ep_dispatch_scatter")) return rc;
    for (int s = 0; s <= p->W; ++s) a.tok_off[s] = p->tok_off[s];
    return EP_OK;
}

static void scatter_commit(ep_plan* p, const float* weights)
{
    p->routed = false;
    p->live = true;
    p->has_w = weights != nullptr;
}

int ep_dispatch_scatter(ep_plan* p, const void* x, const float* weights, const float* scales,
                        const int32_t* indices, void* stream)
{
    ScatterArgs a;
    int rc = scatter_prepare(p, x, weights, scales, indices, a);
    if (rc != EP_OK) return rc;
    DeviceGuard g(p->device);
    if (!g.ok) return fail(EP_ERR_CUDA, "cannot select the plan's device %d", p->device);
    cudaError_t e = p->fp4 ? launch_scatter_quant_fp4(a, p->num_sms, (cudaStream_t)stream)
                    : p->quantise ? launch_scatter_quant(a, p->num_sms, (cudaStream_t)stream)
                                  : launch_scatter(a, p->num_sms, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "ep_dispatch_scatter: launch");
    scatter_commit(p, weights);
    return EP_OK;
}

int ep_dispatch(ep_plan* p, const void* x, const float* weights, const float* scales,
                const int32_t* indices, const int32_t* n_tok_host, void* stream, ep_dispatch_out* out)
{
    if (!p) return fail(EP_ERR_ARG, "plan is NULL");
    // check the payload arguments before the routing kernel starts a new epoch
    if (!x || !aligned(x, 16)) return fail(EP_ERR_ARG, "x is NULL or not 16-byte aligned");
    if (weights && !aligned(weights, 4)) return fail(EP_ERR_ARG, "weights not 4-byte aligned");
    if (p->quantise) {
        if (scales) return fail(EP_ERR_ARG, "the quantising dtype computes its scales: pass NULL");
    } else {
        if (p->sd > 0 && (!scales || !aligned(scales, 4)))
            return fail(EP_ERR_ARG, "scale_dim=%d needs a 4-byte aligned scales array", p->sd);
        if (p->sd == 0 && scales) return fail(EP_ERR_ARG, "scales given but the plan has scale_dim 0");
    }
    if (!out) return fail(EP_ERR_ARG, "out is NULL");
    int rc = ep_dispatch_route(p, indices, n_tok_host, stream, nullptr);
    if (rc != EP_OK) return rc;
    rc = ep_dispatch_scatter(p, x, weights, scales, indices, stream);
    if (rc != EP_OK) return rc;
    fill_out(p, out);
    return EP_OK;
}

int ep_combine(ep_plan* p, const void* expert_out, const float* weights, void* out, float* out_w,
               uint64_t epoch, void* stream)
{
    if (!p) return fail(EP_ERR_ARG, "plan is NULL");
    if (!p->live || epoch != p->epoch)
        return fail(EP_ERR_STATE, "epoch %llu is not the plan's live dispatch (live=%d, epoch %llu)",
                    (unsigned long long)epoch, (int)p->live, (unsigned long long)p->epoch);
    if (!expert_out || !aligned(expert_out, 16)) return fail(EP_ERR_ARG, "expert_out is NULL or not 16-byte aligned");
    if (!out || !aligned(out, 16)) return fail(EP_ERR_ARG, "out is NULL or not 16-byte aligned");
    if (out_w && !weights) return fail(EP_ERR_ARG, "out_w given without weights");
    if (weights && !aligned(weights, 4)) return fail(EP_ERR_ARG, "weights not 4-byte aligned");
    if (out_w && !aligned(out_w, 4)) return fail(EP_ERR_ARG, "out_w not 4-byte aligned");
    {
        const char* eo0 = (const char*)expert_out;
        const char* eo1 = eo0 + (size_t)p->W * p->rows * p->H * 2;
        const char* o0 = (const char*)out;
        const char* o1 = o0 + (size_t)p->W * p->M * p->H * 2;
        if (eo0 < o1 && o0 < eo1) return fail(EP_ERR_ARG, "expert_out overlaps out");
    }
    DeviceGuard g(p->device);
    if (!g.ok) return fail(EP_ERR_CUDA, "cannot select the plan's device %d", p->device);

    CombineArgs a{};
    a.probe = plan_probe(p);
    a.eo = (const uint16_t*)expert_out; a.w_in = weights; a.fwd = p->fwd;
    a.out = (uint16_t*)out; a.out_w = out_w; a.status = p->status; a.H = p->H;
    a.W = p->W; a.k = p->k; a.F = p->F; a.M = p->M; a.N = p->N;
    combine_geometry(a, p->variant, p->num_sms);
    if (int rc = check_units(a.N, a.chunks, "ep_combine")) return rc;
    for (int s = 0; s <= p->W; ++s) a.tok_off[s] = p->tok_off[s];
    cudaError_t e = launch_combine(a, p->dtype == EP_FP16, p->num_sms, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "ep_combine: launch");
    return EP_OK;
}

// Grouping scan form of the live dispatch.  A rank receives at most one row per routed token,
// so no rank holds more than N rows: the two-pass scan (per-chunk counts in the plan's scan_cnt)
// runs only when N spans kScanMinChunks 1024-row chunks, and its chunk stride is the call's,
// ceil(N / 1024) <= the plan's chunks.  Smaller calls, whatever the plan's capacity, take the
// one-pass scan, whose chain is then at most two chunks.
static void set_scan_form(const ep_plan* p, GroupArgs& a)
{
    const int64_t chunks = ((int64_t)p->N + kScanChunk - 1) / kScanChunk;
    const bool two_pass = p->scan_cnt != nullptr && chunks >= kScanMinChunks;
    a.scan_cnt = two_pass ? p->scan_cnt : nullptr;
    a.scan_chunks = two_pass ? (int)chunks : 0;
}

static int check_wire(ep_plan* p, uint64_t epoch, const char* who, int block = 128)
{
    if (!p) return fail(EP_ERR_ARG, "%s: plan is NULL", who);
    if (!p->live || epoch != p->epoch)
        return fail(EP_ERR_STATE, "%s: epoch %llu is not the plan's live dispatch", who,
                    (unsigned long long)epoch);
    if (p->H % block != 0) return fail(EP_ERR_ARG, "%s: hidden=%d is not a multiple of %d", who, p->H, block);
    if (p->dtype == EP_FP16) return fail(EP_ERR_ARG, "%s: the wire carries BF16 outputs; FP16 plan", who);
    return EP_OK;
}

int ep_quantize_received(ep_plan* p, const void* expert_out, void* expert_q, float* expert_scales,
                         uint64_t epoch, void* stream)
{
    int rc = check_wire(p, epoch, "ep_quantize_received");
    if (rc != EP_OK) return rc;
    if (!expert_out || !aligned(expert_out, 16) || !expert_q || !aligned(expert_q, 16) ||
        !expert_scales || !aligned(expert_scales, 4))
        return fail(EP_ERR_ARG, "ep_quantize_received: a buffer is NULL or misaligned");
    DeviceGuard g(p->device);
    if (!g.ok) return fail(EP_ERR_CUDA, "cannot select the plan's device %d", p->device);
    WireArgs a{};
    a.status = p->status; a.probe = plan_probe(p);
    a.eo = (const uint16_t*)expert_out; a.q = (uint8_t*)expert_q; a.scales = expert_scales;
    a.recv_count = p->recv_count; a.H = p->H; a.rows = p->rows; a.W = p->W;
    cudaError_t e = launch_quantise_rows(a, p->num_sms, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "ep_quantize_received: launch");
    return EP_OK;
}

int ep_combine_fp8(ep_plan* p, const void* expert_q, const float* expert_scales, const float* weights,
                   void* out, float* out_w, uint64_t epoch, void* stream)
{
    int rc = check_wire(p, epoch, "ep_combine_fp8");
    if (rc != EP_OK) return rc;
    if (!expert_q || !aligned(expert_q, 16) || !expert_scales || !aligned(expert_scales, 4))
        return fail(EP_ERR_ARG, "ep_combine_fp8: codes or scales NULL or misaligned");
    if (!out || !aligned(out, 16)) return fail(EP_ERR_ARG, "ep_combine_fp8: out is NULL or not 16-byte aligned");
    if (out_w && !weights) return fail(EP_ERR_ARG, "ep_combine_fp8: out_w given without weights");
    if ((weights && !aligned(weights, 4)) || (out_w && !aligned(out_w, 4)))
        return fail(EP_ERR_ARG, "ep_combine_fp8: weights or out_w not 4-byte aligned");
    DeviceGuard g(p->device);
    if (!g.ok) return fail(EP_ERR_CUDA, "cannot select the plan's device %d", p->device);
    CombineArgs geo{};
    geo.H = p->H; geo.N = p->N;
    combine_geometry(geo, p->variant, p->num_sms);     // slice size in 8-element vectors
    WireArgs a{};
    a.status = p->status; a.probe = plan_probe(p);
    a.q = (uint8_t*)expert_q; a.scales = (float*)expert_scales; a.fwd = p->fwd; a.w_in = weights;
    a.out = (uint16_t*)out; a.out_w = out_w; a.H = p->H; a.rows = p->rows;
    a.W = p->W; a.k = p->k; a.F = p->F; a.M = p->M; a.N = p->N;
    a.chunk_pieces = geo.chunk_vecs / 2;
    a.chunks = (int)((p->H / 16 + a.chunk_pieces - 1) / a.chunk_pieces);
    if (int rc2 = check_units(a.N, a.chunks, "ep_combine_fp8")) return rc2;
    for (int s = 0; s <= p->W; ++s) a.tok_off[s] = p->tok_off[s];
    cudaError_t e = launch_combine_fp8(a, p->num_sms, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "ep_combine_fp8: launch");
    return EP_OK;
}

int ep_quantize_received_fp4(ep_plan* p, const void* expert_out, void* expert_q, uint8_t* expert_scales,
                             uint64_t epoch, void* stream)
{
    int rc = check_wire(p, epoch, "ep_quantize_received_fp4", 32);
    if (rc != EP_OK) return rc;
    if (!expert_out || !aligned(expert_out, 16) || !expert_q || !aligned(expert_q, 16) || !expert_scales)
        return fail(EP_ERR_ARG, "ep_quantize_received_fp4: a buffer is NULL or misaligned");
    DeviceGuard g(p->device);
    if (!g.ok) return fail(EP_ERR_CUDA, "cannot select the plan's device %d", p->device);
    WireArgs a{};
    a.status = p->status; a.probe = plan_probe(p);
    a.eo = (const uint16_t*)expert_out; a.q = (uint8_t*)expert_q; a.scales = (float*)expert_scales;
    a.recv_count = p->recv_count; a.H = p->H; a.rows = p->rows; a.W = p->W;
    cudaError_t e = launch_quantise_rows_fp4(a, p->num_sms, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "ep_quantize_received_fp4: launch");
    return EP_OK;
}

int ep_combine_fp4(ep_plan* p, const void* expert_q, const uint8_t* expert_scales, const float* weights,
                   void* out, float* out_w, uint64_t epoch, void* stream)
{
    int rc = check_wire(p, epoch, "ep_combine_fp4", 32);
    if (rc != EP_OK) return rc;
    if (!expert_q || !aligned(expert_q, 16) || !expert_scales)
        return fail(EP_ERR_ARG, "ep_combine_fp4: codes or scales NULL or misaligned");
    if (!out || !aligned(out, 16)) return fail(EP_ERR_ARG, "ep_combine_fp4: out is NULL or not 16-byte aligned");
    if (out_w && !weights) return fail(EP_ERR_ARG, "ep_combine_fp4: out_w given without weights");
    if ((weights && !aligned(weights, 4)) || (out_w && !aligned(out_w, 4)))
        return fail(EP_ERR_ARG, "ep_combine_fp4: weights or out_w not 4-byte aligned");
    DeviceGuard g(p->device);
    if (!g.ok) return fail(EP_ERR_CUDA, "cannot select the plan's device %d", p->device);
    CombineArgs geo{};
    geo.H = p->H; geo.N = p->N;
    combine_geometry(geo, p->variant, p->num_sms);     // slice size in 8-element vectors
    WireArgs a{};
    a.status = p->status; a.probe = plan_probe(p);
    a.q = (uint8_t*)expert_q; a.scales = (float*)expert_scales; a.fwd = p->fwd; a.w_in = weights;
    a.out = (uint16_t*)out; a.out_w = out_w; a.H = p->H; a.rows = p->rows;
    a.W = p->W; a.k = p->k; a.F = p->F; a.M = p->M; a.N = p->N;
    a.chunk_pieces = geo.chunk_vecs / 4 > 0 ? geo.chunk_vecs / 4 : 1;   // 32-element blocks
    a.chunks = (int)((p->H / 32 + a.chunk_pieces - 1) / a.chunk_pieces);
    if (int rc2 = check_units(a.N, a.chunks, "ep_combine_fp4")) return rc2;
    for (int s = 0; s <= p->W; ++s) a.tok_off[s] = p->tok_off[s];
    cudaError_t e = launch_combine_fp4(a, p->num_sms, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "ep_combine_fp4: launch");
    return EP_OK;
}

int ep_group_by_expert(ep_plan* p, void* packed_x, int32_t* packed_count, int32_t* packed_src_info,
                       int64_t* layout_range, uint64_t epoch, void* stream)
{
    if (!p) return fail(EP_ERR_ARG, "ep_group_by_expert: plan is NULL");
    if (!p->live || epoch != p->epoch)
        return fail(EP_ERR_STATE, "ep_group_by_expert: epoch %llu is not the plan's live dispatch",
                    (unsigned long long)epoch);
    if (!packed_x || !aligned(packed_x, 16) || !packed_count || !aligned(packed_count, 4) ||
        !packed_src_info || !aligned(packed_src_info, 4) || !layout_range || !aligned(layout_range, 8))
        return fail(EP_ERR_ARG, "ep_group_by_expert: a buffer is NULL or misaligned");
    DeviceGuard g(p->device);
    if (!g.ok) return fail(EP_ERR_CUDA, "cannot select the plan's device %d", p->device);
    GroupArgs a{};
    a.status = p->status; a.probe = plan_probe(p);
    a.work.q = p->queues + 2 * kQueueGroup;
    a.vec16 = p->k % 4 == 0;   // receive index rows: 256-byte-aligned buffer, 4k-byte rows
    a.recv_x = p->recv_x; a.recv_idx = p->recv_idx; a.recv_count = p->recv_count; a.src_pos = p->src_pos;
    a.map = p->expert_map; a.packed_x = (uint8_t*)packed_x; a.count = packed_count;
    a.src_info = packed_src_info; a.layout_range = (long long*)layout_range;
    a.rows = p->rows; a.row_bytes = p->row_bytes; a.W = p->W; a.E = p->E; a.k = p->k;
    set_scan_form(p, a);
    cudaError_t e = launch_group(a, p->num_sms, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "ep_group_by_expert: launch");
    p->grouped_epoch = epoch;
    return EP_OK;
}

int ep_dispatch_grouped(ep_plan* p, const void* x, const float* weights, const float* scales,
                        const int32_t* indices, const int32_t* n_tok_host, void* packed_x,
                        int32_t* packed_count, int32_t* packed_src_info, int64_t* layout_range,
                        void* stream, ep_dispatch_out* out)
{
    if (!p) return fail(EP_ERR_ARG, "ep_dispatch_grouped: plan is NULL");
    if (p->quantise) return fail(EP_ERR_ARG, "ep_dispatch_grouped: not available for the quantising dtype");
    if (!x || !aligned(x, 16)) return fail(EP_ERR_ARG, "x is NULL or not 16-byte aligned");
    if (weights && !aligned(weights, 4)) return fail(EP_ERR_ARG, "weights not 4-byte aligned");
    if (p->sd > 0 && (!scales || !aligned(scales, 4)))
        return fail(EP_ERR_ARG, "scale_dim=%d needs a 4-byte aligned scales array", p->sd);
    if (p->sd == 0 && scales) return fail(EP_ERR_ARG, "scales given but the plan has scale_dim 0");
    if (!packed_x || !aligned(packed_x, 16) || !packed_count || !aligned(packed_count, 4) ||
        !packed_src_info || !aligned(packed_src_info, 4) || !layout_range || !aligned(layout_range, 8))
        return fail(EP_ERR_ARG, "ep_dispatch_grouped: a grouped buffer is NULL or misaligned");
    if (!out) return fail(EP_ERR_ARG, "out is NULL");
    // on a plan with the expert columns' words, routing numbers the grouped view as well, and
    // the copy follows it directly; otherwise the grouping scan runs between them
    RouteGroupArgs rg{};
    rg.src_info = packed_src_info;
    int rc = route_call(p, indices, n_tok_host, stream, nullptr, p->eflags ? &rg : nullptr);
    if (rc != EP_OK) return rc;
    DeviceGuard g(p->device);
    if (!g.ok) return fail(EP_ERR_CUDA, "cannot select the plan's device %d", p->device);
    GroupArgs a{};
    a.status = p->status; a.probe = plan_probe(p);
    a.scan_done = p->eflags != nullptr;
    a.bnd = p->bnd;
    a.recv_count = p->recv_count; a.src_pos = p->src_pos; a.map = p->expert_map;
    a.packed_x = (uint8_t*)packed_x; a.count = packed_count; a.src_info = packed_src_info;
    a.layout_range = (long long*)layout_range;
    a.src_idx = indices; a.x = (const uint8_t*)x; a.w = weights; a.scales = scales; a.fwd = p->fwd;
    a.vec16 = (p->k % 4 == 0) && aligned(indices, 16);
    a.recv_idx_out = p->recv_idx; a.recv_w_out = p->recv_w; a.recv_scales_out = p->recv_scales;
    a.rows = p->rows; a.row_bytes = p->row_bytes;
    a.W = p->W; a.E = p->E; a.k = p->k; a.M = p->M; a.F = p->F; a.N = p->N; a.sd = p->sd;
    set_scan_form(p, a);
    const int ce = pick_chunk_elems(p, p->N);          // rows sliced as the payload scatter's
    a.chunk_bytes = ce * p->elem_bytes;
    a.chunks = (int)((p->H + ce - 1) / ce);
    if (int rc2 = check_units(a.N, a.chunks, "ep_dispatch_grouped")) return rc2;
    a.work.q = p->queues + 2 * kQueueGroup;
    for (int s = 0; s <= p->W; ++s) a.tok_off[s] = p->tok_off[s];
    cudaError_t e = launch_group_from_source(a, p->num_sms, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "ep_dispatch_grouped: launch");
    p->routed = false;
    p->live = true;
    p->has_w = weights != nullptr;
    p->grouped_epoch = p->epoch;
    fill_out(p, out);
    return EP_OK;
}

int ep_ungroup_by_expert(ep_plan* p, const void* packed_y, void* out, uint64_t epoch, void* stream)
{
    if (!p) return fail(EP_ERR_ARG, "ep_ungroup_by_expert: plan is NULL");
    if (!p->live || epoch != p->epoch || p->grouped_epoch != epoch)
        return fail(EP_ERR_STATE, "ep_ungroup_by_expert: epoch %llu has no live grouped view",
                    (unsigned long long)epoch);
    if (!packed_y || !aligned(packed_y, 16) || !out || !aligned(out, 16))
        return fail(EP_ERR_ARG, "ep_ungroup_by_expert: a buffer is NULL or not 16-byte aligned");
    DeviceGuard g(p->device);
    if (!g.ok) return fail(EP_ERR_CUDA, "cannot select the plan's device %d", p->device);
    GroupArgs a{};
    a.status = p->status; a.probe = plan_probe(p);
    a.recv_idx = p->recv_idx; a.recv_count = p->recv_count; a.map = p->expert_map;
    a.packed_y = (const uint8_t*)packed_y; a.out = (uint8_t*)out;
    a.rows = p->rows; a.row_bytes = (int64_t)p->H * 2; a.W = p->W; a.E = p->E; a.k = p->k;
    a.N = p->N; a.F = p->F;                               // the dispatch's tokens bound its rows
    cudaError_t e = launch_ungroup(a, p->dtype == EP_FP16, p->num_sms, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "ep_ungroup_by_expert: launch");
    return EP_OK;
}

int ep_reset(ep_plan* p, void* stream)
{
    (void)stream;
    if (!p) return fail(EP_ERR_ARG, "plan is NULL");
    p->epoch += 1;
    p->routed = false;
    p->live = false;
    return EP_OK;
}

int ep_probe_read(ep_plan* p, uint64_t* ns_host, int n_words)
{
    if (!p || !ns_host || n_words < 0) return fail(EP_ERR_ARG, "ep_probe_read: plan or ns_host is NULL, or n_words < 0");
#ifndef EP_PROBE
    return fail(EP_ERR_STATE, "ep_probe_read: this libep.so was built without EP_PROBE");
#else
    DeviceGuard g(p->device);
    if (!g.ok) return fail(EP_ERR_CUDA, "cannot select the plan's device %d", p->device);
    unsigned long long w[2 * kProbePhases];
    cudaError_t e = cudaDeviceSynchronize();
    if (e == cudaSuccess) e = cudaMemcpy(w, plan_probe(p), sizeof w, cudaMemcpyDeviceToHost);
    if (e == cudaSuccess) e = reset_probes(p);
    if (e != cudaSuccess) return cuda_fail(e, "ep_probe_read");
    for (int i = 0; i < n_words && i < 2 * kProbePhases; ++i) ns_host[i] = w[i];
    return EP_OK;
#endif
}

int ep_status(ep_plan* p, int* device_status)
{
    if (!p || !device_status) return fail(EP_ERR_ARG, "plan or device_status is NULL");
    DeviceGuard g(p->device);
    int v = 0;
    cudaError_t e = cudaDeviceSynchronize();
    if (e == cudaSuccess) e = cudaMemcpy(&v, p->status, sizeof v, cudaMemcpyDeviceToHost);
    if (e == cudaSuccess) e = cudaMemset(p->status, 0, sizeof v);
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e, "ep_status");
    *device_status = v;
    return EP_OK;
}

}  // extern "C"

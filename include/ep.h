/*
 * ep.h -- C ABI of libep.so: MoE expert-parallel token Dispatch and Combine on one GB300.
 *
 * The W expert-parallel ranks are logical partitions whose send and receive buffers all live
 * in this GPU's HBM; every "transfer" is an HBM-to-HBM scatter or gather done by the library's
 * own CUDA kernels (sm_103a).  No call here uses a second GPU, a collective or the CPU for any
 * step of the computation.
 *
 * Semantics (MORI-EP gfx1201 PR "feat(ep): add opt-in gfx1201 EP2/EP4 support", section "How the
 * gfx1201 kernels work"; MORI-EP guide, section 3 "Operator API"):
 *   - Dispatch maps each token's top-k experts to destination ranks (expert e lives on rank
 *     e / experts_per_rank) and reserves ONE receive row per (token, distinct destination rank):
 *     experts on the same rank share one hidden payload.  The row carries the token's hidden
 *     vector, its whole top-k index row, its FP32 weight row (if given) and its FP32 scale row
 *     (if scale_dim > 0).  Rows are numbered per destination rank in (source rank, token)
 *     order.  The reverse map src_token_pos[r][row] = src_rank * (W * M) + src_token (guide,
 *     get_dispatch_src_token_pos()).
 *   - Combine uses that map to gather, for every source token, the expert-output rows of the
 *     ranks it was sent to, sums them in FP32 in ascending destination-rank order starting from
 *     +0.0f, and rounds to nearest even into BF16 (BF16 and FP8 payloads) or FP16 (FP16
 *     payload).  Optional FP32 weight rows are summed the same way into an FP32 output.  Routing
 *     weights are never applied to the payload (the caller's responsibility, per the pages).
 *
 * Notation: W ranks, E experts per rank, k = top-k, H = hidden, M = max tokens per rank,
 * sd = scale_dim, F = min(W, k).  All arrays are dense and row-major.  Pointers are DEVICE
 * pointers unless marked "host".  A stream argument is a cudaStream_t passed as void*
 * (NULL = the legacy default stream).  Every call on one plan must be ordered on one stream
 * (or otherwise serialised): calls of one plan that overlap on the GPU race.  Within a call, a
 * kernel that follows another of the call's kernels is launched as a programmatic dependent of
 * it (it may be scheduled early, and waits for its predecessor's completion before touching any
 * data), so results and stream order are those of plain launches.
 *
 * Errors.  Every condition the host can check is reported before any launch, with a negative
 * code and a message readable through ep_last_error().  Problems only the GPU can see (an
 * expert id outside [0, W*E), a bounded spin that expired) never trap: the kernel records the
 * first one in the plan's status word, skips the offending work and finishes; ep_status()
 * reads and clears that word.
 */
#ifndef EP_H_
#define EP_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct ep_plan ep_plan; /* opaque; created and owned by the library */

/* Payload dtypes (the guide's data_type field).
 *   EP_BF16, EP_FP16        16-bit payload, moved bit for bit; combine output in the same type.
 *   EP_FP8_E4M3             FP8 e4m3 payload with caller-supplied FP32 scale rows (scale_dim of
 *                           them), moved bit for bit; combine takes and returns BF16.
 *   EP_BF16_TO_FP8_E4M3     BF16 input, quantised by dispatch itself to FP8 e4m3 with one FP32
 *                           scale per 128 elements (the FP8 wire of the guide's tuning matrix):
 *                           for each block, scale = max|x| / 448 (1 for an all-zero block) and
 *                           code = e4m3(x / scale), both FP32 divisions rounded to nearest even,
 *                           the cast rounding to nearest even and saturating at +-448.  hidden
 *                           must be a multiple of 128; the plan's scale_dim is hidden / 128
 *                           (pass 0 or hidden / 128).  Dispatch takes no scales; recv_x holds
 *                           the codes and recv_scales the scales.  Combine takes and returns
 *                           BF16 (the expert dequantises).
 *   EP_BF16_TO_MXFP4        BF16 input, quantised by dispatch itself to MX FP4 (the pages' FP4
 *                           dispatch; the OCP microscaling layout): per 32-element block, scale
 *                           code c = floor(log2 max|x|) - 2 + 127 clamped to 0..254 (127 for an
 *                           all-zero block) and element codes e2m1(x / 2^(c - 127)), rounded to
 *                           nearest with ties to the even code, saturating at +-6.  hidden must
 *                           be a multiple of 128.  recv_x rows hold H/2 bytes, element 2i in the
 *                           low nibble of byte i; recv_scales rows hold the H/32 scale codes as
 *                           bytes, i.e. H/128 4-byte words (the plan's scale_dim is hidden / 128;
 *                           pass 0 or hidden / 128).  Dispatch takes no scales.  Combine takes and
 *                           returns BF16 (the expert dequantises). */
enum ep_dtype { EP_BF16 = 0, EP_FP16 = 1, EP_FP8_E4M3 = 2, EP_BF16_TO_FP8_E4M3 = 3, EP_BF16_TO_MXFP4 = 4 };

enum ep_status_code {
    EP_OK = 0,
    EP_ERR_ARG = -1,            /* invalid argument (null, misaligned, out of range)        */
    EP_ERR_ALLOC = -2,          /* device allocation failed                                 */
    EP_ERR_CUDA = -3,           /* a CUDA runtime call or launch failed                     */
    EP_ERR_STATE = -4,          /* combine without a live dispatch, or with a stale epoch   */
    EP_ERR_CAPACITY = -5,       /* a rank's token count exceeds max_tok_per_rank            */
    EP_ERR_INDEX = -6,          /* device: an expert id outside [0, W*E) was skipped        */
    EP_ERR_DEVICE_TIMEOUT = -7, /* device: a bounded wait expired; outputs are not valid    */
    EP_ERR_DEVICE_BOUNDS = -8   /* device (EP_CHECKS builds): an index derived on the device
                                   fell outside its buffer; the access was skipped         */
};

/* Work split of the payload scatter and of combine (a performance choice; never changes
 * results).  AUTO follows the gfx1201 launch policy of the pages: small token counts split the
 * hidden dimension into 512- or 1024-element tiles, large ones move whole rows. */
enum ep_variant { EP_VARIANT_AUTO = 0, EP_VARIANT_WHOLE_ROW = 1, EP_VARIANT_TILED_512 = 2,
                  EP_VARIANT_TILED_1024 = 3 };

/* Views of the plan's receive buffers after a dispatch (guide, dispatch() return values). */
typedef struct {
    void* recv_x;           /* [W][W*M][H] payload (BF16 / FP16 / FP8 bits; MXFP4: H/2 bytes)  */
    int32_t* recv_idx;      /* [W][W*M][k] the token's whole top-k index row                 */
    float* recv_w;          /* [W][W*M][k] FP32 weights, NULL if dispatch got none            */
    float* recv_scales;     /* [W][W*M][sd] FP32 scales, NULL if sd == 0 (MXFP4: e8m0 bytes)  */
    int32_t* recv_count;    /* [W] rows received by each rank (guide: recv_num_token)         */
    int32_t* src_token_pos; /* [W][W*M] reverse map: src_rank * (W*M) + src_token             */
    int64_t rows_per_rank;  /* W*M: stride, in rows, between ranks' receive regions           */
    uint64_t epoch;         /* pass to ep_combine; identifies this dispatch                   */
} ep_dispatch_out;

/*
 * Create a plan: validate the shape and allocate, once, every device buffer the calls use
 * (receive rows, index/weight/scale rows, reverse and forward maps, scan flags, status word,
 * and for the grouped view the expert-slot map and, from three 1024-row chunks of capacity, the
 * grouping scan's per-chunk counts).
 * Follows the guide's EpDispatchCombineConfig (section 2, "Configuration") with the receive
 * capacity of W*M rows per rank.
 *   W                 1..32 logical ranks
 *   experts_per_rank  >= 1, W*experts_per_rank < 2^31
 *   topk              1..64
 *   hidden            >= 1, hidden * element size a multiple of 16 bytes
 *   dtype             enum ep_dtype
 *   scale_dim         0..65536 FP32 scales per token row
 *   max_tok_per_rank  >= 1, W*W*max_tok_per_rank < 2^31 (int32 reverse map), and
 *                     W*W*max_tok_per_rank*hidden < 2^35: the 16-bit expert outputs that combine
 *                     reads, [W][W*M][H], stay below 64 GiB, the reach of its 32-bit row offsets
 * The plan belongs to the CUDA device current at creation.  Returns EP_OK and *out, or an error
 * with *out = NULL.  A shape outside these limits is EP_ERR_ARG before any CUDA call (the
 * staging PR's caller contract, "refactor(EPv2): replace per-module __device__ staging with
 * shared buffer", section "Caller contract": a host error naming the argument, never a memory
 * fault or a short buffer).
 */
int ep_plan_create(ep_plan** out, int W, int experts_per_rank, int topk, int hidden, int dtype,
                   int scale_dim, int max_tok_per_rank);

/* Wait for the device, then free the plan and its buffers.  NULL is a no-op.  Synchronising
 * first follows the fix to close() recorded on the gfx1250 EPv2 PR page ("gfx1250 EPv2: EP4
 * topk-9 geometry; selfFirst follows MORI_EP_TOKOFF_EXT", the aiter commits that reference it):
 * a launch still in flight must not read buffers that have been freed.  Returns EP_ERR_CUDA if
 * the synchronisation or the free fails (the plan is released either way). */
int ep_plan_destroy(ep_plan* p);

/* Select the work split (enum ep_variant) of later ep_dispatch / ep_combine calls: the whole-row
 * or 512- / 1024-element hidden tiles of the gfx1201 PR ("How the gfx1201 kernels work", "Wave32
 * and launch policy").  Results do not depend on it.  EP_ERR_ARG for a NULL plan or an unknown
 * variant. */
int ep_plan_set_variant(ep_plan* p, int variant);

/* Device bytes ep_plan_create allocates for this shape, 0 for an invalid shape; host-only, no
 * CUDA call.  The counterpart of the staging PR's ep_staging_bytes() ("refactor(EPv2): replace
 * per-module __device__ staging with shared buffer", sections "Memory" and "Test plan"): the one
 * function that sizes the device buffers, pinned by golden sizes so that it cannot drift from
 * the layout the kernels index. */
size_t ep_plan_device_bytes(int W, int experts_per_rank, int topk, int hidden, int dtype,
                            int scale_dim, int max_tok_per_rank);

/*
 * Dispatch (guide, dispatch(); gfx1201 PR, Dispatch bullet).
 *   x           [W][M][H] payload elements (BF16 for the quantising dtypes), 16-byte aligned;
 *               rows t >= n_tok[s] are not read
 *   weights     [W][M][k] FP32 or NULL
 *   scales      [W][M][sd] FP32; must be NULL iff sd == 0 (always NULL for
 *               EP_BF16_TO_FP8_E4M3 and EP_BF16_TO_MXFP4, whose scales dispatch computes)
 *   indices     [W][M][k] int32 expert ids
 *   n_tok_host  host [W]: tokens on each source rank, each 0..M (EP_ERR_CAPACITY if above M)
 *   out         host: receives views of the plan's buffers and the dispatch epoch
 * Enqueues the routing kernel and the payload scatter kernel on `stream` and returns without
 * waiting.  The views stay valid until the next ep_dispatch, ep_dispatch_route or ep_reset on
 * the plan (guide: outputs must be consumed before the next dispatch overwrites them).  Receive
 * rows at or past recv_count[r] hold unspecified data.
 */
int ep_dispatch(ep_plan* p, const void* x, const float* weights, const float* scales,
                const int32_t* indices, const int32_t* n_tok_host, void* stream,
                ep_dispatch_out* out);

/*
 * The two phases of ep_dispatch, exposed so a caller can time or overlap them separately.
 * ep_dispatch_route runs the routing kernel alone (dedup of destination ranks, prefix scan of
 * receive rows, reverse and forward maps, receive counts); it starts a new dispatch epoch and
 * fills *out.  After ep_dispatch_route, out->recv_w is the weight buffer whether
 * or not the scatter will be given weights.  ep_dispatch_scatter then copies payload, index, weight and scale rows to the
 * rows routed by the preceding ep_dispatch_route (EP_ERR_STATE otherwise); `indices` must be
 * the same array.  ep_dispatch(...) == ep_dispatch_route(...) + ep_dispatch_scatter(...).
 */
int ep_dispatch_route(ep_plan* p, const int32_t* indices, const int32_t* n_tok_host, void* stream,
                      ep_dispatch_out* out);
int ep_dispatch_scatter(ep_plan* p, const void* x, const float* weights, const float* scales,
                        const int32_t* indices, void* stream);

/*
 * Combine (guide, combine(); gfx1201 PR, Combine bullet).
 *   expert_out  [W][W*M][H] 16-bit expert outputs (BF16 for BF16/FP8 plans, FP16 for FP16),
 *               16-byte aligned; may be the dispatch's recv_x (in-place expert)
 *   weights     [W][W*M][k] FP32 rows to sum, or NULL
 *   out         [W][M][H] 16-bit outputs, 16-byte aligned; rows t >= n_tok[s] are untouched
 *   out_w       [W][M][k] FP32 summed weights; NULL to skip (must be NULL if weights is NULL)
 *   epoch       the epoch of the dispatch whose rows are combined (EP_ERR_STATE if it is not
 *               the plan's live dispatch)
 * May be called more than once per dispatch.  expert_out must not overlap out.
 */
int ep_combine(ep_plan* p, const void* expert_out, const float* weights, void* out, float* out_w,
               uint64_t epoch, void* stream);

/*
 * Combine over an FP8 wire (MORI-EP gfx1250 EPv2 pages, push-combine variants: the fp8
 * blockwise push combine; the expert side quantises its BF16 rows before sending and the
 * token's home rank dequantises while reducing).  Needs hidden % 128 == 0 and a BF16 or FP8 plan.
 *
 * ep_quantize_received quantises the live dispatch's received expert rows block-wise, with the
 * quantiser of EP_BF16_TO_FP8_E4M3 (scale = max|x| / 448 per 128 elements, code = e4m3(x /
 * scale)):
 *   expert_out     [W][W*M][H] BF16, 16-byte aligned (may be the dispatch's recv_x)
 *   expert_q       [W][W*M][H] e4m3 codes out, 16-byte aligned
 *   expert_scales  [W][W*M][H/128] FP32 out
 * Only rows below recv_count[r] are read and written.
 *
 * ep_combine_fp8 is ep_combine reading that wire: for every source token, in ascending rank
 * order, v = float(code) * scale (one FP32 multiply) is added in FP32 from +0.0f, and the sum is
 * rounded to nearest even into BF16 `out` [W][M][H].  weights / out_w as in ep_combine.  Its
 * gather reads H + H/32 bytes per row instead of 2H.
 */
int ep_quantize_received(ep_plan* p, const void* expert_out, void* expert_q, float* expert_scales,
                         uint64_t epoch, void* stream);
int ep_combine_fp8(ep_plan* p, const void* expert_q, const float* expert_scales, const float* weights,
                   void* out, float* out_w, uint64_t epoch, void* stream);

/*
 * Combine over an MX FP4 wire (MORI-EP gfx1250 EPv2 pages, push-combine variants: the mxfp4
 * push combine, quantised on the expert side and dequantised while reducing).  The
 * encoding is read as the OCP microscaling layout: 32-element blocks of e2m1 codes sharing one
 * e8m0 power-of-two scale.  Needs hidden % 32 == 0 and a BF16 or FP8 plan.
 *
 * ep_quantize_received_fp4 quantises the live dispatch's received expert rows:
 *   expert_out     [W][W*M][H] BF16, 16-byte aligned (may be the dispatch's recv_x)
 *   expert_q       [W][W*M][H/2] packed codes out, 16-byte aligned; element 2i of a row in the
 *                  low nibble of byte i, 2i+1 in the high nibble
 *   expert_scales  [W][W*M][H/32] e8m0 scale codes out (scale = 2^(code - 127))
 * Per block with amax = max|x|: code = floor(log2 amax) - 2 + 127 clamped to 0..254 (127 for
 * an all-zero block); element codes = e2m1(x / scale), rounded to nearest, ties to the even
 * code, saturating at +-6.  Only rows below recv_count[r] are read and written.
 *
 * ep_combine_fp4 is ep_combine reading that wire: for every source token, in ascending rank
 * order, v = e2m1(code) * scale (exact) is added in FP32 from +0.0f and the sum is rounded to
 * nearest even into BF16 `out` [W][M][H].  weights / out_w as in ep_combine.  Its gather reads
 * H/2 + H/32 bytes per row instead of 2H.
 */
int ep_quantize_received_fp4(ep_plan* p, const void* expert_out, void* expert_q, uint8_t* expert_scales,
                             uint64_t epoch, void* stream);
int ep_combine_fp4(ep_plan* p, const void* expert_q, const uint8_t* expert_scales, const float* weights,
                   void* out, float* out_w, uint64_t epoch, void* stream);

/*
 * Expert-grouped ("standard MoE", 3-D) view of the live dispatch (MORI-EP guide, section 4
 * "Standard MoE Compatibility", convert_dispatch_output() / convert_combine_input()).  On rank r
 * the list of local expert e (global id r*E + e) holds, in receive-row order, every received row
 * whose top-k names that expert, once per row; capacity W*M rows per list.
 *
 * ep_group_by_expert writes, all caller-owned:
 *   packed_x         [W][E][W*M][H] payload rows (the plan's payload type), 16-byte aligned
 *   packed_count     [W][E] int32 list lengths
 *   packed_src_info  [W][E][W*M] int32: source token index within its source rank
 *   layout_range     [W][E][W] int64: (first slot of source rank s) << 32 | (its slot count)
 * Slots at or past packed_count hold unspecified data.
 *
 * ep_ungroup_by_expert is the inverse for expert outputs laid out the same way:
 *   packed_y         [W][E][W*M][H] 16-bit expert outputs (BF16; FP16 for FP16 plans)
 *   out              [W][W*M][H] 16-bit: row i of rank r = sum of its local experts' outputs
 *                    in ascending expert id, FP32 from +0.0f, rounded to nearest even once;
 *                    the combine input of ep_combine.  Needs ep_group_by_expert on this epoch.
 */
int ep_group_by_expert(ep_plan* p, void* packed_x, int32_t* packed_count, int32_t* packed_src_info,
                       int64_t* layout_range, uint64_t epoch, void* stream);
int ep_ungroup_by_expert(ep_plan* p, const void* packed_y, void* out, uint64_t epoch, void* stream);

/*
 * Dispatch straight into the grouped view (guide, section 4, dispatch_standard_moe(): dispatch
 * and the layout conversion done by one launch).  Arguments as ep_dispatch plus the four
 * grouped buffers of ep_group_by_expert.  Each source row is read once and written to the slot
 * of every expert it names; the plan's 2-D receive PAYLOAD rows are not written (recv_x holds
 * unspecified data), while the receive metadata (index, weight, scale rows, src_token_pos,
 * counts) and the grouped outputs are exactly those of ep_dispatch + ep_group_by_expert, so
 * ep_ungroup_by_expert and then ep_combine work on the result.  Not for the quantising dtypes.
 */
int ep_dispatch_grouped(ep_plan* p, const void* x, const float* weights, const float* scales,
                        const int32_t* indices, const int32_t* n_tok_host, void* packed_x,
                        int32_t* packed_count, int32_t* packed_src_info, int64_t* layout_range,
                        void* stream, ep_dispatch_out* out);

/* End the live dispatch (guide, reset()): its views become invalid and ep_combine on its epoch
 * fails.  No device work is needed: the scan flags carry a per-call stamp. */
int ep_reset(ep_plan* p, void* stream);

/* Wait for the device, store the plan's device status word (EP_OK or the first EP_ERR_INDEX /
 * EP_ERR_DEVICE_TIMEOUT recorded since the last call) in *device_status, and clear it.  Device
 * problems are recorded rather than trapped, as the staging PR's caller contract asks of the
 * host and device checks ("refactor(EPv2): replace per-module __device__ staging with shared
 * buffer", section "Caller contract").  EP_ERR_ARG for NULL arguments, EP_ERR_CUDA if the
 * synchronisation or the copy fails. */
int ep_status(ep_plan* p, int* device_status);

/*
 * Routing without any allocation.  The pages have no counterpart to this call: it exists for
 * callers that must not call cudaMalloc -- for example a serving runtime whose pool allocator
 * already owns nearly all of HBM, or a plug-in whose host forbids allocation (which can stall the
 * device) on its hot path -- and therefore cannot hold an ep_plan.  It runs the same routing
 * kernel as ep_dispatch_route, for the shape given by its arguments, on memory the caller owns:
 *   indices        [W][M][k] int32 expert ids                      (input)
 *   n_tok_host     host [W] tokens per source rank, each 0..M        (input)
 *   src_token_pos  [W][W*M] int32 reverse map                        (output)
 *   recv_count     [W] int32 rows received per rank                  (output)
 *   fwd_map        [W][M][min(W,k)] int32: token (s,t)'s receive rows r*(W*M) + row in
 *                  ascending rank, then -1                          (output)
 *   device_status  [1] int32: EP_OK, or EP_ERR_INDEX / EP_ERR_DEVICE_TIMEOUT once the stream
 *                  reaches the end of the call                       (output)
 * The kernel's scan words live in one static device array of 16384 64-bit words (128 KB) inside
 * libep.so, held by every GPU that loads the library until the process exits; a shape needs
 * 3 + W * ceil(W*M / 256) words and larger shapes fail with EP_ERR_ARG.  The first call on a
 * device looks up that array's device address (cudaGetSymbolAddress) and should come before any
 * stream capture; the address is kept for the life of the process, so the entry point must not
 * be called on a device after cudaDeviceReset of that device.  The call runs on the current
 * device, and every pointer argument must be memory usable there (EP_ERR_ARG for another GPU's
 * device memory or for pageable host memory).  Each call clears the words it uses on `stream`; all calls share the one
 * array, so calls that overlap on the GPU (other streams, other threads) race and must be
 * serialised by the caller.  No call allocates or frees device memory.
 */
int ep_route_noalloc(int W, int experts_per_rank, int topk, int max_tok_per_rank,
                     const int32_t* indices, const int32_t* n_tok_host, int32_t* src_token_pos,
                     int32_t* recv_count, int32_t* fwd_map, int32_t* device_status, void* stream);

/*
 * Phase probes (MORI-EP guide, section 11 "Profiling with MORI-VIZ", and the phase probes of the
 * gfx1250 EPv2 PR's commit log: device timestamps per phase of dispatch and combine).  A
 * libep.so built with -DEP_PROBE has every kernel's warps record, per phase, the earliest start
 * and the latest end (%globaltimer, nanoseconds) of the launches on this plan since the last
 * read.  ep_probe_read waits for the device, copies min(n_words, 16) words into ns_host --
 * pairs (earliest start, latest end) for the phases route, scatter, combine, quantise (received
 * rows to a wire), wire combine, grouping scan, grouped copy, ungroup, in that order; a phase
 * with no launch reads (2^64 - 1, 0) -- and resets them.  A library built without EP_PROBE
 * records nothing and returns EP_ERR_STATE; EP_ERR_ARG for NULL arguments.
 */
int ep_probe_read(ep_plan* p, uint64_t* ns_host, int n_words);

/* Static description of a status code ("unknown status" for any other value); never NULL.
 * With ep_last_error, the host side of the staging PR's caller contract ("refactor(EPv2):
 * replace per-module __device__ staging with shared buffer", section "Caller contract"): a
 * rejected call reports an error that names the argument. */
const char* ep_strerror(int code);

/* Message of the last failed call on the calling host thread ("" if none), naming the argument
 * or limit at fault (same contract as ep_strerror).  The string is thread-local and stays valid
 * until that thread's next failing call. */
const char* ep_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* EP_H_ */

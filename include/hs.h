/*
 * hs.h -- C ABI of libhs: activation-sparse decode and prefill of a ReLU^2
 * mixture-of-experts layer with 4-bit weights, for NVIDIA GB300 (sm_103a).
 *
 * The method is the one described on "Skipping dead neurons: a faster
 * Nemotron 3.5 Lightning on Apple silicon" (sevren.ai, "Heimr Sparse Down").
 * Each declaration below cites the section of that page that defines the
 * operation.
 *
 * Conventions (all entry points):
 *  - Every pointer argument named *_dev, and every pointer inside hs_w4,
 *    hs_expert, hs_decode_debug, is a DEVICE pointer owned by the caller.
 *    Descriptor structs themselves (hs_w4, hs_expert, hs_moe_layer) are read
 *    on the host during the call and may be freed when it returns.
 *  - The library allocates no memory.  Scratch comes from a caller-supplied
 *    device workspace whose size the matching *_workspace_size call returns.
 *  - Calls are asynchronous on the given stream (NULL = legacy default
 *    stream): a return of HS_OK means the work was enqueued.  Outputs are
 *    valid once the stream reaches that point.
 *  - Weight, activation and output pointers must be 16-byte aligned; offsets
 *    and logits 4-byte aligned.  Violations return HS_ERR_MISALIGNED.
 *  - Errors are returned, never aborted on.  Nothing is enqueued when an
 *    entry point returns an argument error.
 *  - fp16 and bf16 values are passed as raw 16-bit patterns (uint16_t).
 *
 * 4-bit weight format (section "The whole decode step": one scale for every
 * group of 64 along the input axis of the projection):
 *   w = scale * q + bias,  q in 0..15,  scale and bias fp16.
 * Codes are packed two per byte; the element with the even index along the
 * packed axis sits in the low nibble.
 *
 * Layouts used by the library:
 *   up projection (rows = neurons, packed along hidden; groups along hidden):
 *     codes  [neurons][hidden/2] bytes
 *     sb     [neurons][hidden/64] pairs (scale, bias) of fp16 (4 bytes)
 *   neuron-major down projection (section "Transposing to skip the zeros":
 *   the down weights stored transposed, one row per neuron, so that a dead
 *   neuron's row is skipped in one piece):
 *     codes  [neurons][hidden/2] bytes, packed along the outputs
 *     sb     [neurons/64][hidden] pairs (scale, bias) of fp16 (4 bytes):
 *            one slab of hidden pairs per group of 64 neurons
 *   checkpoint (output-major) down projection, the repacker's input
 *   (section "Two layouts, one problem": one row per output):
 *     codes  [hidden][neurons/2], scale/bias [hidden][neurons/64] fp16
 */
#ifndef HS_H_
#define HS_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Opaque CUDA stream (binary compatible with cudaStream_t). */
typedef struct CUstream_st* hs_stream_t;

/* Status codes. */
#define HS_OK                     0
#define HS_ERR_INVALID_ARG       -1  /* NULL where required, negative size, ... */
#define HS_ERR_MISALIGNED        -2  /* a pointer breaks the alignment rule     */
#define HS_ERR_UNSUPPORTED_SHAPE -3  /* sizes outside what the kernels support */
#define HS_ERR_WORKSPACE         -4  /* workspace NULL or smaller than needed  */
#define HS_ERR_CUDA              -5  /* a CUDA launch or query failed          */
#define HS_ERR_TIMEOUT           -6  /* a bounded device wait gave up          */

/* Flags. */
#define HS_FORCE_DENSE  0x1u  /* read every neuron row and every scale group:
                                 the dense comparison path through the same
                                 kernels (section "The standard way reads
                                 everything"); results equal the sparse path */
#define HS_DOWN_ROW_SCALES 0x4u  /* batch-1 layer decode only: every expert's
                                 down_nm.sb holds per-row scales (the layout
                                 of hs_requant_down_rowscale) instead of the
                                 per-group slabs; no slab is read.  Other
                                 entry points and batch > 1 return
                                 HS_ERR_INVALID_ARG */
#define HS_BATCH_EXPERT_UNION 0x2u  /* batch decode only: read each expert's
                                 weights and the union of ALL its tokens' live
                                 rows exactly once (banded up / down kernels)
                                 instead of once per group of up to 4 of its
                                 tokens (fused kernel, the default); results
                                 agree within the stated tolerance */
#define HS_PREFILL_ROW_GATHER 0x8u  /* prefill (and batch decode when it runs on
                                 the prefill kernels, from 51 tokens; ignored
                                 below): the down product multiplies, per
                                 token tile, only the neurons live for some
                                 token of the tile, packed into dense k-steps
                                 (section "What we do instead"); results
                                 agree with the tile path within the fp16-
                                 operand tolerance (the summation grouping
                                 differs).  Ignored with HS_FORCE_DENSE */

/* One 4-bit projection in one of the layouts above. */
typedef struct {
    const uint8_t* codes;  /* device */
    const void*    sb;     /* device, interleaved fp16 (scale, bias) pairs */
} hs_w4;

/* One expert: up projection, neuron-major down projection, offsets. */
typedef struct {
    hs_w4        up;         /* codes [neurons][hidden/2], sb [neurons][hidden/64] */
    hs_w4        down_nm;    /* codes [neurons][hidden/2], sb [neurons/64][hidden] */
    const float* up_offset;  /* device [neurons] pre-activation offsets, or NULL (= 0) */
    int          neurons;    /* multiple of 64 */
} hs_expert;

/* One MoE layer (section "Inside a MoE layer": a router picks top_k of
 * n_routed experts; a shared expert runs for every token). */
typedef struct {
    const hs_expert* routed;    /* host array [n_routed] */
    int              n_routed;  /* 1..128 */
    const hs_expert* shared;    /* host pointer, or NULL for no shared expert */
    int              hidden;    /* multiple of 64, 64..3072 */
    int              top_k;     /* 1..8, <= n_routed */
} hs_moe_layer;

/* Optional debug outputs of the decode and prefill calls (device pointers,
 * each may be NULL). */
typedef struct {
    int*   topk_idx;   /* [batch][top_k] chosen experts, descending logit   */
    float* topk_w;     /* [batch][top_k] router weights                     */
    float* h;          /* batch 1 only: [shared neurons + top_k * routed
                          neurons] fp32 ReLU^2 outputs in slot order (shared
                          first, then the chosen experts in topk order)      */
    int*   live_rows;  /* int: live down rows read by the call, summed over
                          all (token group, expert) pairs                    */
    int*   live_groups;/* int: 64-neuron groups whose (scale, bias) slab the
                          call read, summed the same way                     */
    uint64_t* live_mask;/* [batch][units] the live sets (section "Our way reads
                          only the rows that fired": neuron n of an expert is
                          live for a token when h_n > 0), one 64-bit word per
                          (token, slot, group of 64 neurons); units = shared
                          neurons/64 + top_k * routed neurons/64, shared
                          groups first, then the chosen experts' groups in
                          topk order; bit r of a group's word = its neuron r.
                          The live set does not depend on HS_FORCE_DENSE
                          (which only makes every row be read).            */
} hs_decode_debug;

/* Human-readable text of a status code (static storage). */
const char* hs_status_string(int status);

/* Reads and clears the library's device-side error word (set when a bounded
 * wait inside a kernel gives up).  Synchronises the current device.
 * *status receives HS_OK or HS_ERR_TIMEOUT. */
int hs_device_status(int* status);

/* Self-test of the failure path: one thread waits on an mbarrier that nothing
 * completes, with the library's bounded wait but a limit of `limit_cycles`
 * clock cycles (1 .. 2^31), then gives up and sets the device error word, as
 * every kernel's bounded waits do.  The next hs_device_status reports
 * HS_ERR_TIMEOUT (and clears the word); the context stays usable.  No fault,
 * trap or unbounded wait is involved.  HS_ERR_INVALID_ARG for a limit out of
 * range. */
int hs_selftest_bounded_wait(long long limit_cycles, hs_stream_t stream);

/* ------------------------------------------------------------------ repack
 * Output-major (checkpoint) down projection -> neuron-major layout.
 * Section "Transposing to skip the zeros" and "Two layouts, one problem":
 * the same numbers, one row per neuron instead of one row per output.
 *   codes_om_dev  [out_dim][neurons/2]     scale_om_dev, bias_om_dev [out_dim][neurons/64]
 *   codes_nm_dev  [neurons][out_dim/2]     sb_nm_dev [neurons/64][out_dim] (scale, bias)
 * out_dim and neurons multiples of 64.  Outputs must not overlap inputs. */
int hs_repack_down_nm(const uint8_t* codes_om_dev, const uint16_t* scale_om_dev,
                      const uint16_t* bias_om_dev, int out_dim, int neurons,
                      uint8_t* codes_nm_dev, void* sb_nm_dev, hs_stream_t stream);

/* Interleave separate fp16 scale and bias arrays [rows][groups] into the
 * (scale, bias) pair array [rows][groups] the up projection reads. */
int hs_pack_sb(const uint16_t* scale_dev, const uint16_t* bias_dev, int rows, int groups,
               void* sb_dev, hs_stream_t stream);

/* --------------------------------------------------------- sparse down
 * One expert's activation-sparse down projection, one token.
 * Section "Our way reads only the rows that fired": only neurons with
 * h_n > 0 are read (one neuron-major row each); the (scale, bias) slab of a
 * group of 64 is read only if one of its neurons fired (section "The whole
 * decode step").  y_o = sum_n h_n * (scale_{g(n),o} * q_{n,o} + bias_{g(n),o}).
 *   h_dev        [neurons] fp32, h >= 0 (ReLU^2 outputs); h_n > 0 means live
 *   y_bf16_dev   [out_dim] bf16 (round to nearest even), required
 *   y_f32_dev    [out_dim] fp32 pre-rounding sums, or NULL
 *   live_idx_dev [neurons] int: the indices of the rows read, ascending
 *                (the live set {n : h_n > 0}; every row with HS_FORCE_DENSE);
 *                entries past *live_count are left untouched; or NULL
 *   live_count_dev  int: number of rows read, or NULL
 * neurons a multiple of 64 up to 65536; out_dim a multiple of 64 up to 3072.
 * Flags: HS_FORCE_DENSE only (else HS_ERR_INVALID_ARG).
 * Workspace: hs_expert_down_sparse_workspace_size bytes, ZERO-FILLED before
 * its first use.  Experts of more than 2048 neurons use it: the partial sums
 * of their 32-group chunks and one completion counter per 64-output band,
 * kept at the start of the workspace for every shape; each call leaves the
 * counters at zero again, so consecutive calls of any shapes the workspace is
 * large enough for (and CUDA graph replays) need no clearing in between.  A
 * workspace another entry point has written must be zero-filled again first.
 * Deterministic: the same inputs give bit-identical outputs. */
size_t hs_expert_down_sparse_workspace_size(int neurons, int out_dim);
int hs_expert_down_sparse(const float* h_dev, const hs_w4* down_nm, int neurons, int out_dim,
                          uint16_t* y_bf16_dev, float* y_f32_dev, int* live_idx_dev, int* live_count_dev,
                          unsigned flags, void* workspace_dev, size_t workspace_bytes,
                          hs_stream_t stream);

/* The same single-expert sparse down projection as hs_expert_down_sparse,
 * for callers that cannot allocate device memory: a host framework that owns
 * every allocation and hands a plugin only the tensors it reads and writes,
 * or a path that must never enter the CUDA allocator.  The page has no
 * counterpart; this is an interface convenience of this library.
 *   Same arguments and results as hs_expert_down_sparse, minus the workspace.
 *   Scratch: a fixed array inside the library (about 0.4 MB on every GPU
 *   that loads it, held until the process exits), sized for the largest
 *   shape the workspace entry point takes (65536 neurons, out_dim 3072);
 *   larger shapes return HS_ERR_UNSUPPORTED_SHAPE.  An expert of at most
 *   2048 neurons runs in one pass and does not touch it; wider experts keep
 *   their partial sums and completion counters there.
 *   Allocates nothing (no cudaMalloc, no allocating library routine).
 *   The first call in each CUDA context looks up the array's device address
 *   (cudaGetSymbolAddress) and caches it under the context's unique id; make
 *   that first call before any stream capture.  A context created later (for
 *   instance after a device reset) gets its own lookup on its first call.
 *   Every call shares the one array: its counters start at zero when the
 *   library loads and every call leaves them at zero; the partial sums are
 *   overwritten before they are read.  Calls that can overlap on the GPU, on
 *   different streams, race with each other; order them on one stream or
 *   with events. */
int hs_expert_down_sparse_noalloc(const float* h_dev, const hs_w4* down_nm, int neurons, int out_dim,
                                  uint16_t* y_bf16_dev, float* y_f32_dev, int* live_idx_dev, int* live_count_dev,
                                  unsigned flags, hs_stream_t stream);

/* ------------------------------------------------- row-scale re-quantising
 * Section "The whole decode step": the checkpoint keeps one (scale, bias) per
 * group of 64 neurons along the output axis, so one live neuron costs its
 * group's whole slab; re-quantising with the scales along the neuron axis
 * removes that toll (the page measured a small perplexity cost and did not
 * ship it; this library offers it as an option, bytes and time only).
 * For each neuron n and group j of 64 consecutive outputs, min-max affine
 * 4-bit quantisation of the checkpoint's dequantised weights:
 *   scale = fp16((max - min) / 15), bias = fp16(min),
 *   q = clamp(rint((w - bias) / scale), 0, 15)   (q = 0 where scale = 0),
 * each step in fp32 (w = fma(scale_om, q_om, bias_om)), round to nearest even.
 *   inputs   as hs_repack_down_nm (checkpoint layout [out_dim][neurons])
 *   codes_nm [neurons][out_dim/2] neuron-major codes (output 2j low nibble)
 *   sb_row   [neurons][hs_row_sb_words(out_dim)] u32 (scale, bias) fp16 pairs,
 *            one per 64 outputs, each row padded with zero words to 16 bytes
 * A layer whose experts carry these arrays as down_nm is decoded with
 * HS_DOWN_ROW_SCALES. */
static inline int hs_row_sb_words(int out_dim) { return ((out_dim / 64) + 3) & ~3; }
int hs_requant_down_rowscale(const uint8_t* codes_om, const uint16_t* scale_om, const uint16_t* bias_om,
                             int out_dim, int neurons, uint8_t* codes_nm, void* sb_row, hs_stream_t stream);

/* ------------------------------------------------------------------ router
 * The router projection ahead of the layer (section "Inside a MoE layer": a
 * router picks 6 of 128 experts for each token; the projection itself is not
 * printed and is read as a linear map): logits[b][e] = sum_k W[e][k] x[b][k].
 *   x_bf16_dev         [batch][hidden] bf16
 *   w_router_bf16_dev  [n_experts][hidden] bf16, row-major, 16-byte aligned
 *   logits_dev         [batch][n_experts] fp32 (the logits hs_moe_layer_decode
 *                      and hs_moe_prefill take)
 * hidden a multiple of 64, at most 3072.  fp32 accumulation, one fixed order
 * per logit: deterministic.  No workspace. */
int hs_router_logits(const uint16_t* x_bf16_dev, const uint16_t* w_router_bf16_dev, int batch, int hidden,
                     int n_experts, float* logits_dev, hs_stream_t stream);

/* ---------------------------------------------------------- layer decode
 * One MoE layer at decode for `batch` tokens (sections "Inside a MoE layer",
 * "Two projections and a switch", "Our way reads only the rows that fired"):
 *   idx, w   = top_k of logits (ties -> lower index), softmax over the chosen
 *   z_e      = W_up,e x + offset_e;  h_e = max(z_e, 0)^2
 *   y_e      = sparse down projection of h_e (live rows only)
 *   y        = y_shared + sum_j w_j y_{idx_j}
 *   x_bf16_dev       [batch][hidden] bf16
 *   logits_dev       [batch][n_routed] fp32 (finite)
 *   y_bf16_dev       [batch][hidden] bf16, required;  y_f32_dev fp32 or NULL
 *   debug            host pointer to device debug outputs, or NULL
 * batch 1..4096.  For batch > 1 the tokens are grouped by expert (section
 * "Sorted by expert").  2..50 tokens (or up to 64 where the next case does
 * not apply): each unit of work (expert, 64-neuron group, up to 4 of the
 * expert's tokens) reads its weights and the union of its tokens' live rows
 * once, on CUDA cores; with HS_BATCH_EXPERT_UNION each expert reads the union
 * of all its tokens' live rows once.  51 tokens or more, without that flag,
 * when the routed experts are stacked as hs_moe_prefill requires: the
 * prefill's tensor-core products (fp16 operands; its output contract), which
 * dequantise each weight tile once for all of an expert's tokens.  For
 * batch > 1: hidden must be a multiple of 128; the CUDA-core kernels (2..50
 * tokens, or up to 64 as above) take experts of at most 3712 neurons (more:
 * HS_ERR_UNSUPPORTED_SHAPE, and the workspace size is 0 unless the prefill
 * kernels apply), the prefill kernels up to 4096; the debug h dump is not
 * available (HS_ERR_INVALID_ARG).  Deterministic; on the CUDA-core kernels
 * without HS_BATCH_EXPERT_UNION each token's y equals, bit for bit, a batch-1
 * call on that token alone.
 * Calls sharing one workspace must not overlap on the GPU. */
size_t hs_moe_layer_decode_workspace_size(const hs_moe_layer* layer, int batch);
int hs_moe_layer_decode(const hs_moe_layer* layer, const uint16_t* x_bf16_dev,
                        const float* logits_dev, int batch, uint16_t* y_bf16_dev,
                        float* y_f32_dev, unsigned flags, const hs_decode_debug* debug,
                        void* workspace_dev, size_t workspace_bytes, hs_stream_t stream);

/* --------------------------------------------------------------- prefill
 * One MoE layer over a prompt chunk of `tokens` tokens (sections "A whole
 * prompt at once", "Sorted by expert", "Per token sparse, per prompt dense",
 * "What we do instead"): every token is routed as in decode, the tokens are
 * grouped by expert, and each expert runs its up projection, ReLU^2 and
 * down projection as matrix products on the tensor cores, the down product
 * reading the neuron-major copy directly.  A 64-neuron tile of the down
 * product is skipped for a tile of up to 128 of the expert's tokens when h is
 * zero for all of them (the skip does not change the result).
 *   x_bf16_dev   [tokens][hidden] bf16;  logits_dev [tokens][n_routed] fp32
 *   y_bf16_dev   [tokens][hidden] bf16, required;  y_f32_dev fp32 or NULL
 * Arithmetic: x and the dequantised weights as fp16, products accumulated in
 * fp32, h = max(z, 0)^2 rounded to fp16; h that rounds to 0 counts as dead.
 * tokens 1..4096; hidden a multiple of 128 (<= 3072); the routed experts'
 * up and down codes must each be stacked back to back in one buffer (expert
 * e at base + e * neurons * hidden/2), else HS_ERR_UNSUPPORTED_SHAPE.
 * Deterministic: the same inputs give bit-identical outputs.  Calls sharing
 * one workspace must not overlap on the GPU. */
typedef struct {
    int*   topk_idx;  /* [tokens][top_k] chosen experts, descending logit  */
    float* topk_w;    /* [tokens][top_k] router weights                    */
    int*   tiles;     /* int[2]: 64-neuron down tiles skipped, considered,
                         summed over (expert, token tile) pairs; with
                         HS_PREFILL_ROW_GATHER: [0] the down k-steps the
                         gather saves against one per 64-neuron group      */
    long long* work;  /* int64[3], each summed over (expert, token tile)
                         pairs of the tile's tokens times: [0] the neurons
                         live for at least one of them (the union), [1] the
                         neurons the down product multiplied (64 per tile
                         not skipped, or per k-step with the row gather,
                         padding entries included), [2] all of the
                         expert's neurons.
                         Down-product flops = 2 * hidden * each entry.     */
    uint64_t* live_mask; /* [tokens][units] the kernel's live sets (h > 0 in
                         its fp16 h), laid out as hs_decode_debug.live_mask */
    uint64_t* tile_live; /* [tiles] per (expert, token tile): bit j set when
                         the down product multiplies 64-neuron tile j (some
                         token of the tile has a live neuron in it, or
                         HS_FORCE_DENSE).  Tiles: the routed experts that
                         have tokens, ascending, each expert's (token, slot)
                         pairs in token order cut into tiles of 128, then
                         the shared expert's tokens in tiles of 128; at most
                         n_routed + ceil(tokens * top_k / 128) +
                         ceil(tokens / 128) entries are written.           */
} hs_prefill_debug;

size_t hs_moe_prefill_workspace_size(const hs_moe_layer* layer, int tokens);
int hs_moe_prefill(const hs_moe_layer* layer, const uint16_t* x_bf16_dev, const float* logits_dev,
                   int tokens, uint16_t* y_bf16_dev, float* y_f32_dev, unsigned flags,
                   const hs_prefill_debug* debug, void* workspace_dev, size_t workspace_bytes,
                   hs_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* HS_H_ */

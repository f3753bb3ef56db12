/*
 * moe_layer.h - C ABI of the GB300 (sm_103a) routed MoE expert layer.
 *
 * The layer (Primus-Turbo "Mega MoE" README, sections "Key points" and
 * "Pipeline"): for every token t and each of its k routing slots j, with
 * expert e = topk_idx[t,j] and weight w = topk_weights[t,j],
 *
 *     h      = x[t] . W1[e]                  (L1 grouped GEMM, H -> 2I)
 *     a      = silu(h[:I]) * h[I:]           (SwiGLU; gate columns first)
 *     o      = w * (a . W2[e])               (L2 grouped GEMM, I -> H)
 *     y[t]   = sum_j o                       (combine: per-token sum over k)
 *
 * and its backward (same page: "L2 dgrad + SwiGLU^T + dW2 (variable-K)",
 * "L1 dgrad + combine + dW1", with the dispatched x recomputed rather than
 * stored, section "Recompute dispatched x in backward").  Cross-rank
 * dispatch/combine of the pages become an on-device permutation of routed
 * rows (one GPU).
 *
 * Conventions for every entry point
 *  - All tensor pointers are DEVICE pointers, row-major and contiguous,
 *    16-byte aligned.  "bf16" means IEEE bfloat16 bit patterns.
 *  - The caller owns every buffer and every stream.  The library never
 *    allocates, frees or synchronises (except moe_read_status, which says so).
 *    Work is enqueued on `stream` (a cudaStream_t passed as void*; NULL is
 *    the legacy default stream).  No call reads device data on the host, so
 *    every enqueueing call can be captured in a CUDA graph.
 *  - Return value: MOE_OK (0) on success, or a negative MOE_E* code; then
 *    moe_last_error() gives a message (thread-local).  On an error return
 *    nothing has been enqueued unless the code is MOE_ECUDA.
 *  - Data-dependent problems are never checked on the host: an expert id
 *    outside [0, E) other than -1 is counted in the status words and the slot
 *    is dropped (it contributes nothing), exactly like -1.
 *  - Shapes: T >= 0; H, I > 0 and multiples of 64; 1 <= k <= E <= 1024;
 *    block_m == 128; T*k < 2^31.
 */
#ifndef MOE_LAYER_H
#define MOE_LAYER_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Layer shape.  T tokens, hidden H, intermediate I, E experts, top-k k,
 * block_m = row alignment of each expert's group (DeepGEMM Mega-MoE article,
 * "Block-M Alignment for Irregular Token Counts"; only 128 is supported).
 * activation_clamp: the SwiGLU activation clamp (the `activation_clamp`
 * argument of the DeepGEMM Mega-MoE article's fused op, given there without
 * a formula; read here as: with c > 0 both SwiGLU inputs, gate and up, are
 * clamped to [-c, c] before silu(gate) * up, and their gradients pass where
 * -c <= input <= c and are 0 outside).  0 (or any c <= 0) = no clamp; NaN
 * or infinity is MOE_EINVAL. */
typedef struct moe_shape {
    int32_t T, H, I, E, k, block_m;
    float activation_clamp;
} moe_shape;

enum {
    MOE_OK = 0,
    MOE_EINVAL = -1,       /* null pointer, bad dimension, k > E, ... */
    MOE_EUNSUPPORTED = -2, /* H or I not a multiple of 64, block_m != 128, misaligned pointer */
    MOE_ECUDA = -3         /* a CUDA runtime/driver call or launch failed */
};

/* Status words inside route_ws (int32 each), see moe_read_status. */
enum {
    MOE_STATUS_MPAD = 0,      /* padded routed rows, a multiple of block_m */
    MOE_STATUS_NUM_TILES = 1, /* MOE_STATUS_MPAD / block_m */
    MOE_STATUS_N_INVALID = 2, /* slots whose id was neither -1 nor in [0, E) */
    MOE_STATUS_FLAGS = 3,     /* bit 0: a kernel gave up on a bounded wait */
    MOE_STATUS_NUM_PAIRS = 4, /* pair_offs[E]: tile pairs the GEMM clusters walk */
    MOE_STATUS_SCHED = 8,     /* words 8..15: work counters of the row-grouped GEMMs,
                                 zeroed by the prologue and back at zero after every
                                 GEMM launch; so calls that use one route_ws must
                                 not run concurrently */
    MOE_STATUS_WORDS = 16
};

/* Byte offsets of every table inside the three caller-owned workspaces.
 *  route_ws (written by moe_route_prologue, read by forward/backward):
 *    counts  int32[E]          slots per expert
 *    offs    int32[E+1]        block_m-padded exclusive prefix sum; offs[E] = Mpad
 *    perm    int32[rows_cap]   slot s = t*k+j held by padded row r; -1 = padding
 *                              (and every r >= Mpad); an expert's rows hold its
 *                              slots in increasing s
 *    inv     int32[T*k]        padded row of slot s; -1 = dropped slot
 *    tiles   int32[tiles_cap]  expert owning rows [m*block_m, (m+1)*block_m);
 *                              -1 for m >= Mpad/block_m
 *    status  int32[16]         MOE_STATUS_* words
 *    pair_offs  int32[E+1]     the GEMMs take an expert's M tiles two at a time
 *                              (ceil(tiles_e / 2) pairs, tiles_e =
 *                              (offs[e+1]-offs[e]) / block_m) and walk the
 *                              experts in decreasing order of counts[e] (ties:
 *                              smaller e first); pair_offs[e] = pairs of the
 *                              experts before e in that walk, pair_offs[E] =
 *                              all pairs
 *    pair_owner int32[tiles_cap] expert of tile pair q of the walk; -1 past
 *                              pair_offs[E]
 *    blk_counts int32[route_blocks*(E+1) (at least 1)] prologue scratch: the
 *                              slots are cut into route_blocks blocks of whole
 *                              1024-slot rounds; per block and expert the
 *                              number of that expert's slots in earlier
 *                              blocks, then one count of invalid ids per block
 *  saved (written by moe_forward, read by moe_backward):
 *    h  bf16[rows_cap, 2I]     L1 output per padded row (gate | up); 0 on padding
 *    a  bf16[rows_cap, I]      SwiGLU output per padded row; 0 on padding
 *    o  bf16[rows_cap, H]      weighted L2 output per padded row
 *    cmask u32[rows_cap, 2I/32] with an activation clamp: bit l of word
 *                              (r, g) = 1 when input feature 32 g + l of
 *                              SwiGLU (gate features first, then up) was
 *                              inside [-c, c] in the forward (the FP32
 *                              decision the backward reuses)
 *  bwd_ws (scratch of moe_backward):
 *    dh      bf16[rows_cap, 2I]          gradient at h; 0 on padding
 *    aw      bf16[rows_cap, I]           w * a per padded row; 0 on padding
 *    dxp     bf16[rows_cap, H]           per-row gradient at the dispatched x
 *    dw_part f32[rows_cap, dw_part_cols] partial sums of d(topk_weights)
 * rows_cap = floor((T*k + min(E, T*k)*(block_m-1)) / block_m) * block_m bounds
 * Mpad for any routing, so no buffer depends on device data. */
typedef struct moe_layout {
    int64_t rows_cap, tiles_cap;
    size_t route_bytes, counts, offs, perm, inv, tiles, status, pair_offs, pair_owner, blk_counts;
    size_t saved_bytes, h, a, o, cmask;
    size_t bwd_bytes, dh, aw, dxp, dw_part;
    int32_t dw_part_cols;
    int32_t route_blocks;
} moe_layout;

/* Sizes and offsets of the three workspaces for `shape`.  Host only; touches
 * no device.  Errors: MOE_EINVAL / MOE_EUNSUPPORTED for a bad shape. */
int moe_workspace_layout(const moe_shape* shape, moe_layout* out);

/* Routing prologue (Primus-Turbo Mega MoE README, "Implementation Map":
 * dispatch prologue that builds routing tables; DeepGEMM Mega-MoE article,
 * "Block-M Alignment").  Reads topk_idx int32[T, k] (device), writes every
 * route_ws table and status word listed above.  route_ws must hold
 * route_bytes.  Bit-exact and deterministic; no host synchronisation; up to
 * three kernels on `stream` (block counts, scan, placement). */
int moe_route_prologue(const moe_shape* shape, const int32_t* topk_idx, void* route_ws, void* stream);

/* Router top-k gating fused in front of the routing prologue (the router
 * that produces topk_idx / topk_weights: Mega MoE README, "Key points"; ROCm
 * Primus MoE training guide, router).  logits f32[T, E] (device, row-major).
 * For each token writes topk_idx int32[T, k]: the k largest logits in
 * decreasing order, equal logits in increasing expert id, a NaN logit
 * ranked as -infinity; and topk_w f32[T, k]: the softmax over the k selected
 * logits (when the largest selected logit is infinite, 1/n on the n selected
 * logits equal to it and 0 elsewhere).  Then builds every route_ws table
 * from that topk_idx exactly as moe_route_prologue does.  All device
 * buffers are the caller's and 16-byte aligned; kernels on `stream` only, no
 * host synchronisation, capturable.  topk_idx and topk_w are overwritten.
 * Errors: MOE_EINVAL for a bad shape or a NULL pointer, MOE_EUNSUPPORTED for
 * a misaligned pointer, MOE_ECUDA for a launch error. */
int moe_router_topk(const moe_shape* shape, const float* logits, int32_t* topk_idx, float* topk_w, void* route_ws,
                    void* stream);

/* Forward (Mega MoE README, "Pipeline"): x bf16[T,H], W1 bf16[E,H,2I]
 * (columns [0,I) gate, [I,2I) up), W2 bf16[E,I,H], topk_w f32[T,k],
 * route_ws from moe_route_prologue on the same topk_idx (its status words
 * may be updated).  Writes saved (saved_bytes) and y bf16[T,H]; y is
 * overwritten.  The combine sums a token's k contributions in FP32 in slot
 * order j = 0..k-1 and rounds once to bf16 (deterministic, no atomics). */
int moe_forward(const moe_shape* shape, const void* x, const void* W1, const void* W2,
                const float* topk_w, void* route_ws, void* saved, void* y, void* stream);

/* Backward of moe_forward given dY bf16[T,H] (Mega MoE README, "Pipeline",
 * backward paragraph).  Inputs as for moe_forward plus `saved` from it.
 * Overwrites (never accumulates into) dx bf16[T,H], dW1 bf16[E,H,2I],
 * dW2 bf16[E,I,H] and dtopk_w f32[T,k]; an expert with no routed slot gets
 * dW1 = dW2 = 0 and a dropped slot gets dtopk_w = 0.  bwd_ws must hold
 * bwd_bytes.  The dispatched x is re-gathered from x, never stored. */
int moe_backward(const moe_shape* shape, const void* dY, const void* x, const void* W1, const void* W2,
                 const float* topk_w, void* route_ws, const void* saved, void* bwd_ws,
                 void* dx, void* dW1, void* dW2, float* dtopk_w, void* stream);

/* FP8 dispatch of the layer input (DeepGEMM Mega-MoE article, usage example:
 * per-token cast of the activations to FP8 with UE8M0 scale factors at a
 * granularity of 32 before dispatch).  x bf16[T,H] (H a multiple of 64) ->
 * x_fp8 u8[T,H] and x_sf u8[T,H/32], device, row-major, caller-owned: for
 * each token and each group of 32 consecutive elements, e = the smallest
 * integer with 448 * 2^e >= max|x| over the group (0 for an all-zero group,
 * clamped to [-127, 127]); x_sf = e + 127 (UE8M0: the scale is 2^(x_sf-127));
 * x_fp8 = OCP E4M3 bytes of x / 2^e, rounded to nearest even, saturating at
 * +-448.  Non-finite inputs are not supported.  Kernels on `stream` only.
 * Errors as for moe_route_prologue. */
int moe_quantize_fp8(const moe_shape* shape, const void* x, uint8_t* x_fp8, uint8_t* x_sf, void* stream);

/* FP8 weights for moe_forward_fp8 (DeepGEMM Mega-MoE article, usage example:
 * the weights are transformed once for the FP8 kernel): W1 bf16[E,H,2I] ->
 * W1_fp8 = E4M3 bytes, K-major [E][2I][H] (column f of W1 as a row: gate
 * columns 0..I-1, then up), and W1_sf = UE8M0 scales, one per 32 consecutive
 * h of a column (the same rule as moe_quantize_fp8, along H), E * 2I * H/32
 * bytes in the layout the L1 kernel loads: for column f, group g = (f mod I)
 * / 64 and row r = 64 [f >= I] + (f mod I) mod 64; for the 32-group j32 of
 * h, block kb = j32 / 4 and step j = j32 mod 4; byte
 *   ((e (I/64) + g) (H/128) + kb) 512 + 16 (r mod 32) + 4 floor(r / 32) + j.
 * Needs H a multiple of 128 (MOE_EUNSUPPORTED otherwise).  Kernels on
 * `stream`; other errors as for moe_route_prologue. */
int moe_quantize_weights_fp8(const moe_shape* shape, const void* W1, uint8_t* W1_fp8, uint8_t* W1_sf, void* stream);

/* FP8 W2 for moe_forward_fp8, the counterpart of moe_quantize_weights_fp8:
 * W2 bf16[E,I,H] -> W2_fp8 = E4M3 bytes, K-major [E][H][I] (column h of W2
 * as a row), and W2_sf = UE8M0 scales, one per 32 consecutive i of a column
 * (the same rule as moe_quantize_fp8, along I), E * H * I/32 bytes in the
 * layout the L2 kernel loads: for column h, group g = h / 128 and row r =
 * h mod 128; for the 32-group j32 of i, block kb = j32 / 4 and step j = j32
 * mod 4; byte
 *   ((e (H/128) + g) (I/128) + kb) 512 + 16 (r mod 32) + 4 floor(r / 32) + j.
 * Needs H and I multiples of 128 (MOE_EUNSUPPORTED otherwise).  Kernels on
 * `stream`; other errors as for moe_route_prologue. */
int moe_quantize_w2_fp8(const moe_shape* shape, const void* W2, uint8_t* W2_fp8, uint8_t* W2_sf, void* stream);

/* FP8 forward (DeepGEMM Mega-MoE article, "Code Example: Fused Overlap
 * Path": the layer on FP8 activations and transformed FP8 weights):
 * moe_forward with the input given as moe_quantize_fp8's x_fp8 / x_sf, W1 as
 * moe_quantize_weights_fp8's W1_fp8 / W1_sf and W2 as moe_quantize_w2_fp8's
 * W2_fp8 / W2_sf.  Both grouped GEMMs multiply E4M3 operands on the tensor
 * cores with their UE8M0 scales applied per 32 elements of K (block-scaled
 * MMA), FP32 accumulation.  Between them the SwiGLU output a of every routed
 * row is quantized in the L1 kernel's epilogue with the rule of
 * moe_quantize_fp8 (groups of 32 consecutive features of I, the scale's
 * maximum taken over the FP32 values of a), so y is the FP8 layer: h and a
 * from the dequantized x and W1, a rounded to E4M3 with its scales, o from
 * that and the dequantized W2, the weighted sum.  It reads half the bytes of
 * both weights and of the gathered rows.  saved receives h (bf16) and o as
 * in moe_forward, and in a's region the E4M3 rows of a (u8[rows_cap, I] at
 * offset a) followed by their scales (u8[rows_cap, I/32] at offset a +
 * rows_cap * I); padding rows hold codes 0 with scale byte 127.  Needs H and
 * I multiples of 128 and no activation clamp (MOE_EUNSUPPORTED otherwise).
 * Everything else (route_ws, y, errors) as for moe_forward.  An inference
 * path: the pages' FP8 operator is a forward; training steps use moe_forward
 * / moe_backward. */
int moe_forward_fp8(const moe_shape* shape, const uint8_t* x_fp8, const uint8_t* x_sf, const uint8_t* W1_fp8,
                    const uint8_t* W1_sf, const uint8_t* W2_fp8, const uint8_t* W2_sf, const float* topk_w,
                    void* route_ws, void* saved, void* y, void* stream);

/* The inverse of moe_quantize_fp8: x_out bf16[T,H] = decode(x_fp8) *
 * 2^(x_sf - 127), exactly (every such value is a bf16 value).  Errors as for
 * moe_quantize_fp8. */
int moe_dequantize_fp8(const moe_shape* shape, const uint8_t* x_fp8, const uint8_t* x_sf, void* x_out, void* stream);

/* moe_backward with FP32 main-gradient accumulation, for training loops that
 * sum weight gradients over micro-batches in FP32 buffers.  The pages have no
 * counterpart: an addition of this library next to their backward (Mega MoE
 * README, "Pipeline", backward paragraph).  Identical to moe_backward except
 * that the weight gradients are not written as bf16: main_grad_W1 f32[E,H,2I] and
 * main_grad_W2 f32[E,I,H] (device, row-major, 16-byte aligned, caller-owned)
 * get main_grad += dW element-wise, from the FP32 accumulators, never rounded
 * to bf16.  An expert with no routed slot adds nothing; T = 0 adds nothing.
 * Each element receives exactly one addition per call, so the result does
 * not depend on the launch order (deterministic); calls on the same buffers
 * must not overlap on the GPU.  dx and dtopk_w are overwritten as in
 * moe_backward.  Errors as for moe_backward. */
int moe_backward_main_grad(const moe_shape* shape, const void* dY, const void* x, const void* W1, const void* W2,
                           const float* topk_w, void* route_ws, const void* saved, void* bwd_ws, void* dx,
                           float* main_grad_W1, float* main_grad_W2, float* dtopk_w, void* stream);

/* Inference forward for callers that cannot allocate device memory when
 * they run the layer: for example a plugin inside an inference engine that
 * gets no workspace from its host, or a serving loop that must not call
 * cudaMalloc (it can synchronise the device).  The pages have no counterpart
 * of this entry point.
 * Same inputs and output as moe_route_prologue followed by moe_forward
 * (topk_idx int32[T,k], y bf16[T,H] overwritten), but the routing tables and
 * the per-row intermediates live in a static 32 MiB device array inside the
 * library (MOE_NOALLOC_SCRATCH_BYTES), which every GPU that loads the library
 * holds until exit.  Allocates nothing: no cudaMalloc, no cudaFree, no
 * allocating library routine.
 *  - status_out: NULL, or device memory for MOE_STATUS_WORDS int32 (16-byte
 *    aligned) that receives this call's status words (the routing counts of
 *    MOE_STATUS_MPAD.. and the timeout bit of MOE_STATUS_FLAGS) by a
 *    device-to-device copy on `stream` after the kernels.  The words
 *    themselves live in the static array, which the caller cannot address,
 *    and the next call overwrites them.
 *  - Size limit: route_bytes (rounded up to 256) + saved_bytes of
 *    moe_workspace_layout must be <= MOE_NOALLOC_SCRATCH_BYTES (e.g. the V3
 *    shape up to T = 1, the T=64, H=128, I=64, E=8, k=2 shape with room to
 *    spare); larger shapes return MOE_EUNSUPPORTED with a message naming the
 *    bytes needed.
 *  - The first call on each device looks up the array's device address with
 *    cudaGetSymbolAddress (the device owning W1 is made current) and keeps it
 *    for the life of the process; make that first call before any stream
 *    capture, and do not use this entry point after a cudaDeviceReset of
 *    that device.
 *  - Every call shares the one array and leaves its contents behind; each call
 *    rewrites every table it reads first, so results never depend on an
 *    earlier call.  Calls that overlap on the GPU (other streams, other host
 *    threads) race on the array: serialise them.
 *  - Forward only: the saved activations are not kept for a backward pass. */
#define MOE_NOALLOC_SCRATCH_BYTES (32u << 20)
int moe_forward_noalloc(const moe_shape* shape, const void* x, const void* W1, const void* W2,
                        const int32_t* topk_idx, const float* topk_w, void* y, int32_t* status_out, void* stream);

/* Copies the MOE_STATUS_WORDS status words of route_ws to host memory
 * `out` (int32[16]).  SYNCHRONISES `stream`; not for use under capture. */
int moe_read_status(const moe_shape* shape, const void* route_ws, int32_t* out, void* stream);

/* Diagnostic of the failure path (not part of the layer; the pages have no
 * counterpart): every wait of the GEMM kernels on an mbarrier is bounded
 * (2 s); a wait that runs out raises the kernel's abort flag, the other
 * roles leave their waits, and bit 0 of MOE_STATUS_FLAGS in route_ws is set
 * for the host.  This call runs that path on purpose with the same wait
 * helpers, in one small kernel on `stream`, on a barrier nothing arrives on:
 * one warp gives up after limit_ns (1 us .. 100 ms), and the warps using the
 * two other wait forms (limit 4 * limit_ns) leave on its abort flag.  It
 * sets bit 0 of route_ws's MOE_STATUS_FLAGS word and nothing else there
 * (the next moe_route_prologue clears it).  elapsed_ns: NULL or device
 * memory for 3 int64 that receive each warp's waiting time in ns (-1 if its
 * wait had succeeded).  No fault, no hang: the kernel ends within
 * 4 * limit_ns.  Errors as for moe_route_prologue (MOE_EINVAL for a limit out
 * of range). */
int moe_selftest_wait_timeout(const moe_shape* shape, void* route_ws, uint64_t limit_ns, int64_t* elapsed_ns,
                              void* stream);

/* Tracing.  moe_trace_begin hands the library `capacity` CUDA events
 * (cudaEvent_t passed as void*, created by the caller with timing enabled).
 * Until moe_trace_end, each kernel the library launches from this thread is
 * bracketed by two of them, recorded on the launch stream: events[2i] just
 * before and events[2i+1] just after the i-th launch, so the caller can read
 * each kernel's device time with cudaEventElapsedTime.  Launches beyond
 * capacity/2 are counted but not recorded.  moe_trace_end returns the number
 * of launches since moe_trace_begin; moe_trace_kernel(i) names the i-th
 * ("" when out of range).  Host only; no synchronisation. */
int moe_trace_begin(void* const* events, int capacity);
int moe_trace_end(void);
const char* moe_trace_kernel(int i);

/* Message for the last non-zero return on this thread ("" if none). */
const char* moe_last_error(void);

/* Library version string. */
const char* moe_version(void);

#ifdef __cplusplus
}
#endif
#endif /* MOE_LAYER_H */

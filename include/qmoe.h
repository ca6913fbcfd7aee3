/*
 * qmoe.h — C ABI of the GB300 (sm_103a) GGUF block-quantized GEMV and
 * decode-time MoE FFN library (libqmoe.so).
 *
 * Sources of the operations (page titles; the section is the Rust/CUDA item):
 *   - "ferrox-cuda 0.14.0 — src/gpu.rs": the fused dequantize-and-dot matvec
 *     kernels Q8_0/Q4_0/Q4_K/Q5_K/Q6_K_MATVEC_KERNEL_SRC and their launchers
 *     launch_q*_matvec; SILU_MUL_KERNEL_SRC; launch_dense_ffn_swiglu;
 *     CudaError (Unsupported is distinct from Launch: refuse, never compute
 *     something else).
 *   - "ferrox-core 0.16.0 — weight_matrix.rs": block_bytes_per_row,
 *     apply (y = W x), apply_gpu_dense_ffn_swiglu (shape rules).
 *   - "aprender-serve 0.70.2 — forward_qwen3_moe_resident.rs": module doc (MoE
 *     op order, router weight folded into the SwiGLU activation), Qwen3MoeShape,
 *     QuantWeight, ExpertStack (base + e * stride), check_moe_shape,
 *     upload_experts, build_layer (F32 router), moe_layer, last_routes.
 *
 * Conventions for every entry point:
 *   - All tensor pointers are DEVICE pointers owned by the caller.  The library
 *     allocates nothing per call; scratch comes from the caller's workspace.
 *   - Calls are asynchronous: they enqueue kernels on `stream` (a cudaStream_t
 *     passed as void*; NULL = legacy default stream) and return without a host
 *     synchronisation.  A status other than QMOE_OK means nothing was enqueued,
 *     except QMOE_ERR_CUDA, which reports a failed launch.
 *   - Weight operands (W, the router, the expert stacks) are read-only model
 *     constants.  Kernels may start reading them before earlier kernels on the
 *     same stream have finished (programmatic dependent launch), so weights
 *     must be fully written (e.g. the upload synchronised) before the first
 *     call that reads them.  Activations (x, residual, outputs, workspace) are
 *     ordered by the stream as usual.
 *   - Quantized matrices are row-major [rows][row_bytes] of little-endian ggml
 *     blocks, row_bytes = cols / block_elems * block_bytes.  W must be 16-byte
 *     aligned; the kernels read whole 16-byte granules that contain W's bytes
 *     (never a byte outside those granules).
 *   - Floating-point arithmetic is f32, as the pages' kernels compute it:
 *     every product of a decoded weight (an integer quant) and an f32
 *     activation is exact before its one rounding into an f32 sum, with the
 *     activations' full 24-bit significands; scales, mins and everything after
 *     them are f32 with FMA.  Only the order of the roundings differs from
 *     the per-element form (sum (d*sc*q - dmin*m) x is formed as
 *     d*sc*sum q x - dmin*m*sum x per sub-block).  Results match the exact
 *     result within |err| <= 1e-3 * sum_j |w_ij x_j| + 1e-6 per GEMV output,
 *     NaN where the exact computation is NaN (a NaN scale or a NaN
 *     activation).  Non-finite inputs (Inf scales, non-finite x) give
 *     non-finite outputs, NaN or Inf.  Activations of magnitude 2^106 (about
 *     8e31) or more are outside the supported range: the kernels flag them,
 *     and qmoe_device_status reports QMOE_ERR_UNSUPPORTED.  The many-token
 *     MoE path (tensor cores) rounds its operands to f16/tf32 (moe_ffn).
 *   - Errors: the status names the class; qmoe_last_error() gives a message
 *     (thread-local) naming the refused argument.
 */
#ifndef QMOE_H
#define QMOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Weight formats (the library's own numbering).  Block layouts are those of
 * the kernel sources on "ferrox-cuda 0.14.0 — src/gpu.rs":
 *   F32   4-byte floats (router / dense f32 GEMV)
 *   Q8_0  34-byte blocks of 32: f16 d, int8 q[32]; value d*q
 *   Q4_0  18-byte blocks of 32: f16 d, 16 bytes; byte i low nibble = element
 *         i, high nibble = element i+16; value (nibble-8)*d
 *   Q4_K  144-byte super-blocks of 256: f16 d, f16 dmin, 12 bytes of 6-bit
 *         (scale, min) pairs, 128 bytes of nibbles; value (d*sc)*q - dmin*m
 *   Q5_K  176-byte super-blocks: as Q4_K plus qh[32] giving each value a 5th bit
 *   Q6_K  210-byte super-blocks: ql[128], qh[64], int8 scales[16], f16 d;
 *         value (d*sc)*(q6-32) */
typedef enum {
    QMOE_F32 = 0,
    QMOE_Q8_0 = 1,
    QMOE_Q4_0 = 2,
    QMOE_Q4_K = 3,
    QMOE_Q5_K = 4,
    QMOE_Q6_K = 5
} qmoe_qtype;

typedef enum {
    QMOE_OK = 0,
    QMOE_ERR_INVALID_ARGUMENT = 1, /* null pointer, bad size, misalignment, small workspace */
    QMOE_ERR_UNSUPPORTED = 2,      /* valid request this library does not implement */
    QMOE_ERR_CUDA = 3,             /* a CUDA runtime call or launch failed */
    QMOE_ERR_TIMEOUT = 4           /* a bounded device-side wait expired (qmoe_device_status) */
} qmoe_status;

/* MoE layer shape — Qwen3MoeShape (num_experts, num_experts_per_tok,
 * expert_dim) plus the hidden size, token count and the stacks' formats. */
typedef struct {
    int32_t hidden;      /* H: model width; multiple of 256 */
    int32_t expert_dim;  /* F: each expert's FFN width; multiple of 256 */
    int32_t num_experts; /* E: 1..256 */
    int32_t top_k;       /* k: 1..min(E, 16) */
    int32_t n_tokens;    /* T >= 1 */
    int32_t gate_qtype;  /* qmoe_qtype of the gate stack (quantized) */
    int32_t up_qtype;    /* must equal gate_qtype */
    int32_t down_qtype;  /* qmoe_qtype of the down stack (quantized) */
    int32_t route_flags; /* 0, or QMOE_ROUTE_NO_RENORM */
} qmoe_moe_shape;

/* route_flags: the routing weights are the softmax probabilities over all E
 * experts of the k selected ones, not renormalised over the k.  The pages
 * state renormalisation for the Qwen3-MoE-shaped layer and are silent for
 * the OLMoE-shaped one; this flag gives the other reading. */
#define QMOE_ROUTE_NO_RENORM 1

/* y = W x — launch_q*_matvec on "ferrox-cuda 0.14.0 — src/gpu.rs" and
 * WeightMatrix::apply on "ferrox-core 0.16.0 — weight_matrix.rs".
 *   qtype  one of qmoe_qtype (F32 included: a plain f32 GEMV)
 *   W      [rows][row_bytes] blocks, 16-byte aligned, read-only
 *   rows   >= 1;  cols >= 1, a multiple of the format's block elements
 *          (F32: 4, else UNSUPPORTED; Q8_0/Q4_0: 32; K-quants: 256; else
 *          INVALID_ARGUMENT); cols <= 32768.  Q8_0/Q4_0 rows of an odd
 *          number of blocks are 2-byte aligned in W (row_bytes = cols/32*34
 *          or *18): the rows follow each other unpadded, as GGUF stores them
 *   x      [cols] f32, 16-byte aligned;  y [rows] f32, overwritten
 * Errors: INVALID_ARGUMENT (null, sizes, alignment), UNSUPPORTED (qtype,
 * cols, device not sm_103), CUDA. */
qmoe_status qmv(int qtype, const void* W, int64_t rows, int64_t cols, const float* x, float* y,
                void* stream);

/* Bytes of workspace ffn_swiglu needs: 256 bytes of grid-barrier state plus
 * inter f32 activations. */
size_t ffn_swiglu_workspace_size(int64_t hidden, int64_t inter);

/* residual += down( silu(gate x) * (up x) ) — launch_dense_ffn_swiglu on
 * "ferrox-cuda 0.14.0 — src/gpu.rs" (gate, up, SwiGLU, down on device), with
 * the result added to the residual as the MoE op order does for each expert
 * (weight 1).  silu(g) = g / (1 + e^-g) (SILU_MUL_KERNEL_SRC).
 *   gate, up   [inter][hidden] quantized, same qtype (else UNSUPPORTED)
 *   down       [hidden][inter] quantized
 *   hidden, inter  multiples of 256, <= 32768
 *   x          [hidden] f32, the FFN input (after the norm)
 *   residual   [hidden] f32, updated in place
 *   ws         >= ffn_swiglu_workspace_size bytes of device memory, 16-byte
 *              aligned; its contents are scratch (it may hold anything before
 *              a call); calls that overlap on the GPU must not share one
 * Shape rules of apply_gpu_dense_ffn_swiglu (gate.cols == up.cols == x.len,
 * down.cols == gate.rows) hold by construction of the arguments.
 * The layer runs as one cooperative kernel (one CTA per SM): the gate/up
 * rows and then the down rows stream through one pipeline, and a grid
 * barrier orders the activations between the two products.  A layer that does
 * not fit that kernel's shared memory runs as two kernels instead, and
 * qmoe_set_exec_mode(QMOE_EXEC_SEPARATE) forces that form (diagnostics). */
qmoe_status ffn_swiglu(const void* gate, const void* up, const void* down, int gate_qtype,
                       int up_qtype, int down_qtype, int64_t hidden, int64_t inter,
                       const float* x, float* residual, void* ws, size_t ws_bytes, void* stream);

/* Bytes of workspace ffn_swiglu_rmsnorm needs: ffn_swiglu's plus room for the
 * normed input. */
size_t ffn_swiglu_rmsnorm_workspace_size(int64_t hidden, int64_t inter);

/* ffn_swiglu with ffn_norm in front, on the hidden state itself:
 *   residual += down( silu(gate xn) * (up xn) ),
 *   xn = residual * norm_w / sqrt(mean(residual^2) + eps)
 * — the RMSNorm of FUSED_ADD_RMSNORM_KERNEL_SRC on "ferrox-cuda 0.14.0 —
 * src/gpu.rs" (without its add), applied before the FFN as moe_layer on
 * "aprender-serve 0.70.2 — forward_qwen3_moe_resident.rs" norms `hidden`
 * with ffn_norm.
 *   norm_w     [hidden] f32, 16-byte aligned (the ffn_norm weight)
 *   eps        finite, >= 0
 *   residual   [hidden] f32, 16-byte aligned: the layer's input, updated in
 *              place with the FFN output
 *   ws         >= ffn_swiglu_rmsnorm_workspace_size bytes, 16-byte aligned
 * Other arguments, rules and errors as ffn_swiglu.  The fused layer kernel
 * computes the norm itself (no extra launch); the two-kernel form runs a
 * norm kernel first. */
qmoe_status ffn_swiglu_rmsnorm(const void* gate, const void* up, const void* down,
                               int gate_qtype, int up_qtype, int down_qtype, int64_t hidden,
                               int64_t inter, const float* norm_w, float eps, float* residual,
                               void* ws, size_t ws_bytes, void* stream);

/* Bytes of workspace moe_ffn needs for this shape (256 bytes of grid-barrier
 * state, then the logits, activations and, for many tokens, the grouping
 * buffers). */
size_t moe_ffn_workspace_size(const qmoe_moe_shape* shape);

/* The MoE FFN of one layer for T tokens — moe_layer on "aprender-serve
 * 0.70.2 — forward_qwen3_moe_resident.rs", after ffn_norm:
 *   logits = R x_t (F32 router [E][H]);  softmax over E, the top k (ties:
 *   lower expert index), weights renormalised over those k (or, with
 *   shape->route_flags = QMOE_ROUTE_NO_RENORM, the softmax probabilities);
 *   for each routed (e, w) in rank order:  a = silu(G_e x_t) * (U_e x_t),
 *   residual_t += D_e (w a).
 * The routing runs on the device: no host synchronisation inside the layer.
 *   router_W    [E][H] f32, 16-byte aligned
 *   gate_stack, up_stack  [E][F][H] quantized, one allocation each; expert
 *               e at base + e * F * row_bytes(H)  (ExpertStack::expert)
 *   down_stack  [E][H][F] quantized
 *   x           [T][H] f32 (normed input);  residual [T][H] f32, in place
 *   topk_idx    [T][k] int32 or NULL: routed experts in rank order
 *   topk_w      [T][k] f32 or NULL: their routing weights
 *   ws          >= moe_ffn_workspace_size(shape) bytes, 16-byte aligned;
 *               scratch that may hold anything before a call; calls that
 *               overlap on the GPU must not share one
 * Execution: for T >= 32 tokens with Q4_K gate/up and Q6_K down stacks, the
 * tokens are grouped by expert and the expert products run on the tensor
 * cores, whose operands are rounded once: gate/up weights and x (scaled per
 * token by 2^s so that its largest |x| lies in [2^14, 2^15)) to f16, down
 * weights and the activations to tf32 (round to nearest).  A product of
 * operands in f16's normal range, and every down product, carries at most
 * 2 * 2^-11 relative error, inside the bound above.  f16's range adds two
 * absolute terms, outside that bound: an element of x below 2^-28 of its
 * token's largest |x| is rounded to f16's subnormal spacing (error at most
 * 2^-39 * max|x| per element), and so is a decoded gate/up weight of
 * magnitude below 2^-14 (error at most 2^-25 per weight).  Each is far
 * below the bound unless a token's large activations meet zero weights and
 * its other activations are more than 2^28 times smaller, or a row's
 * decoded weights are nearly all below 2^-14; the single-token and
 * small-batch paths (f32 throughout) have neither term.  A decoded gate/up
 * weight beyond f16's range is flagged (QMOE_ERR_UNSUPPORTED from
 * qmoe_device_status).
 * A single token runs one cooperative kernel (one CTA per SM):
 * router GEMV, a grid barrier, routing in every CTA, the routed gate/up rows
 * and then the down rows streamed through one pipeline, a second grid barrier
 * before the down products.  2..31 tokens run in cooperative launches of up
 * to 16 tokens (fewer where the layer's tiles and x tables need more shared
 * memory): every CTA routes all the launch's tokens and groups them by
 * expert, each routed expert's gate/up rows are staged once for all its
 * tokens, and the down products run per token as in the single-token kernel.
 * qmoe_set_exec_mode selects the forms these kernels replace, for
 * diagnostics: QMOE_EXEC_UNBATCHED runs 2..31 tokens one launch each,
 * QMOE_EXEC_SEPARATE runs every token as three launches (router, gate/up,
 * down).
 * Routing of non-finite logits: experts are ranked on a total order (NaN
 * above +Inf above finite values above -Inf, ties to the lower index), so
 * every one of the k slots names an expert in [0, E).  When a token's
 * largest logit is not finite (a NaN or +Inf logit, or all logits -Inf) its
 * softmax is NaN throughout; the route is then experts 0..k-1 with NaN
 * weights and the token's residual becomes NaN.
 * Errors: INVALID_ARGUMENT (null, shape fields out of range, k > E, small
 * workspace, misalignment), UNSUPPORTED (E > 256, k > 16, F32 or mixed
 * gate/up formats, sizes not multiples of 256), CUDA. */
qmoe_status moe_ffn(const float* router_W, const void* gate_stack, const void* up_stack,
                    const void* down_stack, const qmoe_moe_shape* shape, const float* x,
                    float* residual, int32_t* topk_idx, float* topk_w, void* ws,
                    size_t ws_bytes, void* stream);

/* Bytes of workspace moe_ffn_rmsnorm needs: moe_ffn's plus [T][H] f32 for the
 * normed inputs. */
size_t moe_ffn_rmsnorm_workspace_size(const qmoe_moe_shape* shape);

/* moe_ffn with ffn_norm in front, on each token's hidden state:
 *   xn_t = residual_t * norm_w / sqrt(mean(residual_t^2) + eps)
 *   residual_t += MoE(xn_t)       (router, routing and experts as moe_ffn)
 * — moe_layer on "aprender-serve 0.70.2 — forward_qwen3_moe_resident.rs"
 * from rmsnorm_into(hidden, ffn_norm) on, the norm as
 * FUSED_ADD_RMSNORM_KERNEL_SRC on "ferrox-cuda 0.14.0 — src/gpu.rs" computes
 * it without its add.
 *   norm_w      [H] f32, 16-byte aligned;  eps finite, >= 0
 *   residual    [T][H] f32, 16-byte aligned: the input, updated in place
 *   ws          >= moe_ffn_rmsnorm_workspace_size(shape) bytes
 * Other arguments, rules and errors as moe_ffn (there is no x).  The
 * per-token fused kernel norms its input itself; the tensor-core and
 * separate-kernel forms run a norm kernel first. */
qmoe_status moe_ffn_rmsnorm(const float* router_W, const void* gate_stack, const void* up_stack,
                            const void* down_stack, const qmoe_moe_shape* shape,
                            const float* norm_w, float eps, float* residual, int32_t* topk_idx,
                            float* topk_w, void* ws, size_t ws_bytes, void* stream);

/* Bytes of the built-in scratch used by moe_ffn_noalloc. */
#define QMOE_NOALLOC_SCRATCH_BYTES (1u << 20)

/* moe_ffn without a caller workspace, for callers that cannot allocate
 * device memory.  Examples: a runtime where another framework owns all
 * device memory and hands out none of it, or a serving loop that forbids
 * allocation once it has started.
 * The pages have no counterpart of this call; it is an addition of this
 * library.  Arguments and results are those of moe_ffn, minus ws/ws_bytes.
 *   - Scratch comes from one QMOE_NOALLOC_SCRATCH_BYTES device array built
 *     into the library.  Every GPU that loads the library holds that array
 *     until the process exits.  Nothing is allocated or freed by this call:
 *     no cudaMalloc, no cudaFree, no allocating library routine.
 *   - Shapes whose moe_ffn_workspace_size exceeds the array are refused with
 *     QMOE_ERR_UNSUPPORTED and a message giving both sizes.  For a layer of
 *     hidden 2048, 128 experts, top-8, expert_dim 768 that allows up to 35
 *     tokens per call; larger batches need moe_ffn and a workspace.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current); make that first
 *     call before any stream capture.
 *   - All calls share the one array, which keeps the last call's contents.
 *     Nothing in it has to start at zero: every call writes what it reads,
 *     and the grid-barrier state at its start is checked and reset by the
 *     kernel itself.
 *     Calls that overlap on the GPU (other streams, other host threads)
 *     race on it, so order them on one stream or synchronise between them. */
qmoe_status moe_ffn_noalloc(const float* router_W, const void* gate_stack, const void* up_stack,
                            const void* down_stack, const qmoe_moe_shape* shape, const float* x,
                            float* residual, int32_t* topk_idx, float* topk_w, void* stream);

/* Synchronises `stream`, then reads and clears the current device's error
 * word: QMOE_ERR_TIMEOUT if a bounded device wait expired since the last
 * read (a pipeline stage, or a grid barrier that not every CTA reached);
 * QMOE_ERR_UNSUPPORTED if the many-token MoE path met a decoded gate/up
 * weight outside f16 range, or a quantized product met an activation of
 * magnitude 2^106 or more (the output is then not valid); QMOE_ERR_CUDA if
 * the stream reported an error, or if an internal invariant of the routing
 * failed (an expert index outside [0, E) was clamped to 0); else QMOE_OK. */
qmoe_status qmoe_device_status(void* stream);

/* Execution modes for qmoe_set_exec_mode. */
#define QMOE_EXEC_DEFAULT 0   /* the fused and batched kernels */
#define QMOE_EXEC_SEPARATE 1  /* every layer / token as separate kernels */
#define QMOE_EXEC_UNBATCHED 2 /* 2..31 tokens one fused launch each */

/* Diagnostics and tests: selects, for the whole process and every later
 * call, which of the equivalent kernel forms ffn_swiglu and moe_ffn (and
 * their _rmsnorm and _noalloc variants) launch.  All forms compute the same
 * function.  The pages have no counterpart (their layer always runs as
 * separate launches).  INVALID_ARGUMENT for an unknown mode. */
qmoe_status qmoe_set_exec_mode(int mode);

/* Tests of the failure path only: on the current device, every bounded
 * device wait gives up after wait_limit_ns (0 restores the default, 2 s),
 * and, if skip_arrive_cta >= 0, that CTA of the cooperative layer kernels
 * never arrives at their grid barriers, so the other CTAs' waits run out:
 * the kernels then record QMOE_ERR_TIMEOUT (qmoe_device_status) and return
 * without writing the layer's output.  (-1, 0) restores normal operation.
 * Synchronises the device before writing the setting.  Errors: CUDA,
 * UNSUPPORTED (not sm_103), INVALID_ARGUMENT (skip_arrive_cta < -1).  The
 * pages have no counterpart; their CudaError model ("refuse, never compute
 * something else") is what the failure path follows. */
qmoe_status qmoe_set_fault_injection(uint64_t wait_limit_ns, int skip_arrive_cta);

/* Message for the last non-OK status returned on this thread ("" if none). */
const char* qmoe_last_error(void);

/* Row bytes of a [*][cols] matrix of this format (block_bytes_per_row on
 * "ferrox-core 0.16.0 — weight_matrix.rs"); -1 if cols is not a whole number
 * of blocks or the qtype is unknown. */
int64_t qmoe_row_bytes(int qtype, int64_t cols);

#ifdef __cplusplus
}
#endif

#endif /* QMOE_H */

/*
 * mxfp8.h -- C ABI of the GB300 (sm_103a) MXFP8 block-scaled linear layer.
 *
 * The layer, as vLLM PR #52204 "[Kernel] Add FlashInfer TRTLLM MXFP8 linear
 * backend" states it (Purpose; review thread on apply_weights):
 *   load time : quantize the weight [N, K] to MXFP8 (FP8 E4M3 elements, one
 *               E8M0 power-of-two scale per 32 consecutive K elements),
 *               require K % 256 == 0, pad N to a multiple of 128 (data and
 *               scales), lay data and scales out for the GEMM, remember N;
 *   per call  : quantize the BF16 activations [M, K] on the fly with the 8x4
 *               scale layout, run the block-scaled GEMM with FP32
 *               accumulation, slice the padded N back to N, add the bias and
 *               write BF16 [M, N].  Only N is padded, never the input.
 * The grouped entry point runs the same product over per-expert row segments
 * of expert-sorted activations (the MoE gate_up GEMM of SGLang PR #18945 "Add
 * support for FlashInfer mxfp8" and FlashInfer PR #4026).
 *
 * Conventions shared by every call:
 *  - All pointers named x, q, sf, bias, y, workspace, expert_offsets are
 *    DEVICE pointers on the current CUDA device; `stream` is a cudaStream_t
 *    (NULL = legacy default stream).  Every call that takes a stream is
 *    asynchronous on it, never synchronises and never allocates, frees or
 *    touches memory other than its arguments.  The caller owns all memory and
 *    must keep it alive until the stream work completes.
 *  - Arguments are checked on the host before any launch; a failed check
 *    returns its status and launches nothing.  A launch failure returns
 *    MXFP8_ERR_CUDA and mxfp8_last_cuda_error() gives the cudaError_t.
 *  - M = 0 (or rows = 0) returns MXFP8_OK without launching.
 *  - Results are deterministic: the same inputs give the same bytes.
 *  - Every call can be captured in a CUDA graph (no host synchronisation,
 *    no allocation); the kernel parameters capture the pointers.
 *  - The library runs on compute capability 10.3 (GB300) only; any other
 *    device gets MXFP8_ERR_UNSUPPORTED_DEVICE.
 *
 * Formats (the byte orders are readings of this library; the pages give only
 * the 8x4 buffer size):
 *  - E4M3: torch.float8_e4m3fn bytes.  E8M0: one byte, value 2^(b-127),
 *    0xFF is NaN.
 *  - Scale rule: byte = clamp(floor(log2(amax)) - 8 + 127, 0, 254) with amax
 *    the largest magnitude of the 32-block (OCP MX v1.0 rule for MXFP8).
 *    An all-zero block gets byte 0x00; a block holding NaN/Inf gets byte
 *    0xFF and elements 0x7F.  Elements are v / 2^(byte-127) rounded to
 *    nearest-even E4M3, saturating to +-448, signed zeros kept.
 *  - 8x4 activation scale layout (KB = K/32): the scale of row m, block b is
 *    at byte ((m/8)*(KB/4) + b/4)*32 + (m%8)*4 + (b%4); the buffer holds
 *    ceil(M/8)*8 * KB bytes (the size printed in the prhub summary of vLLM PR
 *    #52204, key source snippets); rows M..ceil8(M)-1 hold 0x00.
 *  - Prepared weight: data [N_pad][K] row-major E4M3 (rows N..N_pad-1 are
 *    0x00); scales in tiles of 128 rows x 4 blocks (512 bytes): tile
 *    (t = n/128, q = b/4) starts at byte (t*(KB/4) + q)*512 and row r = n%128,
 *    block b sits at (r%32)*16 + (r/32)*4 + (b%4) inside it; padding rows are
 *    0x00.  Experts are stacked: expert e's data starts at e*N_pad*K and its
 *    scales at e*N_pad*KB.
 */
#ifndef MXFP8_GB300_H
#define MXFP8_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum mxfp8_status {
    MXFP8_OK = 0,
    MXFP8_ERR_INVALID_ARG = 1,           /* null pointer, negative or too large size, bad struct */
    MXFP8_ERR_K_NOT_MULTIPLE_OF_256 = 2, /* K % 256 != 0 (load-time check of the pages) */
    MXFP8_ERR_MISALIGNED = 3,            /* a device pointer is not 16-byte aligned */
    MXFP8_ERR_UNSUPPORTED_DEVICE = 4,    /* current device is not compute capability 10.3 */
    MXFP8_ERR_WORKSPACE_TOO_SMALL = 5,   /* workspace_bytes below the size helper's value */
    MXFP8_ERR_DEVICE_TIMEOUT = 6,        /* a kernel gave up waiting (see mxfp8_device_error) */
    MXFP8_ERR_CUDA = 7,                  /* a CUDA call failed: mxfp8_last_cuda_error() */
    MXFP8_ERR_OUT_OF_BOUNDS = 8          /* debug build only: a kernel computed a store index outside
                                            its buffer and skipped the store (see mxfp8_device_error) */
} mxfp8_status;

typedef enum mxfp8_in_dtype {
    MXFP8_IN_F32 = 0,  /* float32 weights (e.g. a checkpoint in FP32) */
    MXFP8_IN_BF16 = 1  /* bfloat16 weights */
} mxfp8_in_dtype;

/* A prepared MXFP8 weight: a VIEW of caller-owned device buffers.
 * Fill it with mxfp8_weight_view(); n_pad is derived, not chosen. */
typedef struct mxfp8_weight {
    int64_t num_experts; /* 1 for a dense layer */
    int64_t n;           /* logical output features per expert */
    int64_t n_pad;       /* ceil(n / 128) * 128 */
    int64_t k;           /* input features, a multiple of 256 */
    void* q;             /* [num_experts][n_pad][k] E4M3 bytes, 16-B aligned */
    void* sf;            /* [num_experts][n_pad * k / 32] E8M0 bytes, tiled, 16-B aligned */
} mxfp8_weight;

/* ------------------------------------------------------------ size helpers
 * Pure functions of the shape; return 0 for invalid shapes, including
 * shapes beyond the library's limits: at most 2^31 - 256 rows (M, or
 * experts x N_pad), K <= 2^20. */

/* Bytes of the 8x4 activation scale buffer: ceil(m/8)*8 * k/32. */
size_t mxfp8_act_scale_bytes(int64_t m, int64_t k);
/* Bytes of one expert's prepared data: ceil(n/128)*128 * k. */
size_t mxfp8_weight_bytes(int64_t n, int64_t k);
/* Bytes of one expert's prepared scales: ceil(n/128)*128 * k/32. */
size_t mxfp8_weight_scale_bytes(int64_t n, int64_t k);
/* Workspace of mxfp8_linear / mxfp8_grouped_linear for m activation rows:
 * the quantized activations (m*k bytes, rounded up to 256) followed by their
 * 8x4 scales. */
size_t mxfp8_linear_workspace_bytes(int64_t m, int64_t k);

/* Fill *w as a view of (q, sf) for num_experts x [n, k]; checks the shape
 * (k % 256 == 0, sizes > 0) and the 16-byte alignment of q and sf. */
mxfp8_status mxfp8_weight_view(mxfp8_weight* w, int64_t num_experts, int64_t n,
                               int64_t k, void* q, void* sf);

/* ------------------------------------------------------------- operations */

/* Load-time weight preparation (vLLM PR #52204, process_weights_after_loading:
 * quantize, pad N to 128, lay out data and scales, keep the logical N).
 * src: device [num_experts][n][k] float32 or bfloat16, row-major, 16-B aligned.
 * Writes every byte of w->q and w->sf (padding included). */
mxfp8_status mxfp8_prepare_weight(const void* src, mxfp8_in_dtype dtype,
                                  const mxfp8_weight* w, void* stream);

/* Per-call activation quantizer with the 8x4 scale layout (vLLM PR #52204,
 * flashinfer_mxfp8_quantize_8x4 custom op and its fake implementation).
 * x: device bfloat16 [m][k] row-major, 16-B aligned; q: device [m][k] E4M3;
 * sf: device mxfp8_act_scale_bytes(m, k) bytes, written in full (padding
 * rows 0x00).  k % 256 == 0. */
mxfp8_status mxfp8_quantize_act(const void* x, int64_t m, int64_t k, void* q,
                                void* sf, void* stream);

/* Block-scaled GEMM + slice + bias on already-quantized activations
 * (the mm_mxfp8 call with use_8x4_sf_layout of vLLM PR #52204):
 * y[i][j] = bf16( sum_k deq(qa)[i][k] * deq(W)[j][k] + bias[j] ), j < n.
 * qa: [m][k] E4M3, sfa: 8x4 scales for (m, k); bias: bfloat16 [n] or NULL;
 * y: bfloat16 [m][n] row-major (contiguous, logical n).  Dense weights only
 * (w->num_experts == 1). */
mxfp8_status mxfp8_gemm(const void* qa, const void* sfa, int64_t m,
                        const mxfp8_weight* w, const void* bias, void* y,
                        void* stream);

/* The whole per-call layer (vLLM PR #52204, apply_weights): quantize x with
 * the 8x4 layout into the workspace, then the block-scaled GEMM with the
 * padded-N slice and the bias fused into its epilogue.
 * x: bfloat16 [m][k]; bias: bfloat16 [n] or NULL; y: bfloat16 [m][n];
 * workspace: device, >= mxfp8_linear_workspace_bytes(m, k), 256-B aligned
 * preferred (16-B required); its contents are scratch. */
mxfp8_status mxfp8_linear(const void* x, int64_t m, const mxfp8_weight* w,
                          const void* bias, void* y, void* workspace,
                          size_t workspace_bytes, void* stream);

/* Grouped (MoE expert) layer over expert-sorted rows: rows
 * [off[e], off[e+1]) of x_sorted use expert e of w.  expert_offsets: device
 * int32 [num_experts + 1], non-decreasing, off[0] = 0, off[E] = rows (empty
 * experts allowed; the values are read on the device, not checked).  The
 * GEMM reads the offsets (like the weights) in its prologue, before it waits
 * for the previous kernel: they must be complete when the call is enqueued,
 * or written by a kernel that does not release programmatic dependents
 * early (ordinary kernels never do; mxfp8_moe_route does not).
 * bias: bfloat16 [num_experts][n] or NULL; y: bfloat16 [rows][n].
 * The activations are quantized as one [rows, k] matrix.  num_experts <= 1024. */
mxfp8_status mxfp8_grouped_linear(const void* x_sorted, int64_t rows,
                                  const int32_t* expert_offsets,
                                  const mxfp8_weight* w, const void* bias,
                                  void* y, void* workspace,
                                  size_t workspace_bytes, void* stream);

/* ------------------------------------------------ host activations/output
 * The pages' layer reads and writes device tensors; this entry point serves
 * a caller whose activations and results live in host memory.  It enqueues,
 * on `stream`, the copy of x_host (bfloat16 [m][k], row-major) into the
 * workspace, the layer exactly as mxfp8_linear computes it, and the copy of
 * y (bfloat16 [m][n]) back to y_host.  It returns once that work is
 * enqueued: y_host holds the result after the stream has completed it.
 * Page-locked host buffers keep both copies asynchronous; pageable ones
 * work, the copies then block the calling thread, and the call cannot be
 * captured in a CUDA graph.  w (dense only) and bias
 * stay on the device.  workspace: device, >=
 * mxfp8_linear_host_workspace_bytes(m, n, k), 16-B aligned; its contents
 * are scratch.  m = 0 enqueues nothing. */
size_t mxfp8_linear_host_workspace_bytes(int64_t m, int64_t n, int64_t k);
mxfp8_status mxfp8_linear_host(const void* x_host, int64_t m, const mxfp8_weight* w,
                               const void* bias, void* y_host, void* workspace,
                               size_t workspace_bytes, void* stream);

/* ------------------------------------------------ scratch-free variant
 * The pages have no counterpart to this entry point; it exists for callers
 * that cannot allocate device memory, so cannot hand mxfp8_linear a
 * workspace: code inside a host framework that owns every device allocation
 * (an allocation behind its back breaks its memory accounting), or serving
 * paths that must never allocate once running.
 *
 * mxfp8_linear_static_scratch computes what mxfp8_linear computes, always by
 * the unfused path (quantizer -> scratch -> GEMM; its schedule is a stored
 * unfused tactic of the mxfp8_linear class when the tactic table holds one,
 * else the built-in heuristic's unfused choice), with the scratch in an
 * array of MXFP8_STATIC_SCRATCH_BYTES inside the library: every GPU that
 * loads the library holds that array until the process exits.  It allocates
 * nothing and calls no allocating routine.  The caller still passes x, the
 * weight, bias and y.
 *  - Sizes: ceil(m*k/256)*256 + ceil(m/8)*8 * k/32 bytes must fit the array,
 *    else MXFP8_ERR_WORKSPACE_TOO_SMALL and nothing is launched (at k = 2048
 *    that is m <= 7943; at k = 8192, m <= 1985).
 *  - The first call on each device looks up the array's device address
 *    (cudaGetSymbolAddress with that device current); make that first call
 *    before any stream capture begins.
 *  - All calls share the one array, which keeps the last call's contents
 *    (nothing needs clearing: each call writes every byte it reads).  Calls
 *    whose kernels overlap on the GPU race on it: serialise them.
 *  - Errors and other conventions as mxfp8_linear; a failed CUDA call's code
 *    is returned by mxfp8_last_cuda_error() and by
 *    mxfp8_static_scratch_last_cuda_error(). */
#define MXFP8_STATIC_SCRATCH_BYTES (16u << 20)
mxfp8_status mxfp8_linear_static_scratch(const void* x, int64_t m, const mxfp8_weight* w,
                                         const void* bias, void* y, void* stream);
int mxfp8_static_scratch_last_cuda_error(void);

/* ------------------------------------------------ 128x4 activation scales
 * The high-M variant the vLLM PR leaves out ("the high-M 128x4
 * activation-scale path"): activation scales laid out like the prepared
 * weights' (tiles of 128 rows x 4 blocks, 512 bytes, tile (m/128, b/4) at
 * ((m/128)*(KB/4) + b/4)*512, row r = m%128 and block b at
 * (r%32)*16 + (r/32)*4 + (b%4); rows M..ceil128(M)-1 hold 0x00).  At large
 * M (when CTA tiles of two 128-row weight tiles x 176 tokens give every SM a
 * tile) the GEMM runs the dual weight-tile schedule of mxfp8_linear, taking
 * per K block the scale tiles of the 128-row tiles each token tile touches;
 * otherwise persistent tiles of 256 tokens (128 when M <= 128) that start on
 * 128-token boundaries, each scale tile copied into tensor memory as it is.
 * Same arithmetic and results as the 8x4 entry points. */
size_t mxfp8_act_scale_bytes_128x4(int64_t m, int64_t k);          /* ceil(m/128)*128 * k/32 */
size_t mxfp8_linear_128x4_workspace_bytes(int64_t m, int64_t k);
mxfp8_status mxfp8_quantize_act_128x4(const void* x, int64_t m, int64_t k, void* q,
                                      void* sf, void* stream);
mxfp8_status mxfp8_gemm_128x4(const void* qa, const void* sfa, int64_t m,
                              const mxfp8_weight* w, const void* bias, void* y,
                              void* stream);
mxfp8_status mxfp8_linear_128x4(const void* x, int64_t m, const mxfp8_weight* w,
                                const void* bias, void* y, void* workspace,
                                size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------ tactics
 * A tactic is a GEMM schedule, four int32:
 *   [0] tokens per tile: 16, 32, 64, 128, 256, or 144 / 160 / 176 / 192
 *       (with split_k -1) = two 128-row weight tiles x that many tokens per
 *       CTA tile (dense only);
 *   [1] split_k: -1 = persistent tiles, 1..8 = one output tile per cluster
 *       of that many CTAs with K split among them (tiles of <= 128 tokens,
 *       dense only);
 *   [2] fuse_quant: 1 = the GEMM quantizes x itself (one-tile mxfp8_linear);
 *   [3] pipes: MMA pipelines per CTA, 1, 2 (tiles <= 64) or 4 (16 only).
 * The tactic table maps (current device, call kind, power-of-two bucket of M,
 * N, K, experts) to a tactic; every call consults it before the built-in
 * heuristic.  The pages leave tactics to later work (vLLM PR #52204 "does
 * not add tactic hints"; FlashInfer PR #1214 review: an autotuner with
 * benching/perf tuning).  Tactics change the FP32 summation order, not the
 * arithmetic: results stay within the layer tolerance and are deterministic
 * for a given table. */
typedef enum mxfp8_call_kind {
    MXFP8_KIND_LINEAR = 0,  /* mxfp8_linear */
    MXFP8_KIND_GEMM = 1,    /* mxfp8_gemm (pre-quantized activations) */
    MXFP8_KIND_GROUPED = 2, /* mxfp8_grouped_linear */
    MXFP8_KIND_GATED = 3    /* MoE GEMM1 with the SwiGLU epilogue (mxfp8_moe.h) */
} mxfp8_call_kind;

/* Times every valid tactic for this call (arguments as mxfp8_linear, `iters`
 * timed calls each, <= 0 means 20) on the caller's buffers, stores the
 * fastest in the table for the call's class and writes it to chosen[4] (may
 * be NULL).  Each tactic is timed as one CUDA graph of `iters` calls back to
 * back on a private stream that waits for the caller's (no host launch
 * latency in the timing; best of three launches after a warm one); a weight smaller than twice the L2 is rotated
 * over temporary copies (allocated for the call, at most ~2x L2 bytes, freed
 * before it returns) so that every timed call streams its weight from HBM.
 * SYNCHRONOUS: it waits for the stream; not allowed while the stream is
 * being captured (MXFP8_ERR_INVALID_ARG).  y is overwritten. */
mxfp8_status mxfp8_autotune_linear(const void* x, int64_t m, const mxfp8_weight* w,
                                   const void* bias, void* y, void* workspace,
                                   size_t workspace_bytes, int iters, void* stream,
                                   int32_t* chosen);
/* The same for mxfp8_grouped_linear. */
mxfp8_status mxfp8_autotune_grouped_linear(const void* x_sorted, int64_t rows,
                                           const int32_t* expert_offsets,
                                           const mxfp8_weight* w, const void* bias, void* y,
                                           void* workspace, size_t workspace_bytes, int iters,
                                           void* stream, int32_t* chosen);
/* Table access (host only, no device work): get returns
 * MXFP8_ERR_INVALID_ARG when the class has no entry; set validates the
 * tactic for the kind and K. */
mxfp8_status mxfp8_tactic_get(int kind, int64_t m, int64_t n, int64_t k, int64_t experts,
                              int32_t* tactic);
mxfp8_status mxfp8_tactic_set(int kind, int64_t m, int64_t n, int64_t k, int64_t experts,
                              const int32_t* tactic);
void mxfp8_tactic_clear(void);
int64_t mxfp8_tactic_count(void);
/* The tactic a call of this kind and shape would run now, without launching
 * anything: the table's entry for its class if there is one, else the
 * built-in heuristic's choice (the testing hook of mxfp8_set_schedule, when
 * set, wins as it does for calls).  m: activation rows (sorted rows for the
 * grouped kinds); experts: 1 for the dense kinds; sms: the GPU's SM count,
 * or <= 0 for the current device's (which then must be a GB300).  Writes the
 * tactic encoding of mxfp8_tactic_get to tactic[4]; a dual weight-tile
 * tactic reports 2 pipes.  Host only. */
mxfp8_status mxfp8_plan_tactic(int kind, int64_t m, int64_t n, int64_t k, int64_t experts, int sms,
                               int32_t* tactic);

/* --------------------------------------------------------- status helpers */

const char* mxfp8_status_string(mxfp8_status status);
/* cudaError_t of the last call that returned MXFP8_ERR_CUDA (per thread). */
int mxfp8_last_cuda_error(void);
/* Reads and clears the device-side error words: the one the GEMM kernels set
 * when a wait gives up (a hang turned into an error), and, in the debug
 * build (libmxfp8_gb300_debug.so, compiled with MXFP8_DEBUG), the ones every
 * kernel sets when a computed store index falls outside its buffer (the
 * store is skipped).  SYNCHRONISES the current device.  Returns MXFP8_OK,
 * MXFP8_ERR_DEVICE_TIMEOUT or MXFP8_ERR_OUT_OF_BOUNDS (timeout first). */
mxfp8_status mxfp8_device_error(void);

/* The process-wide testing hooks (schedule pinning, wait limit, pipelines,
 * last schedule) are declared in mxfp8_testing.h. */

#ifdef __cplusplus
}
#endif

#endif /* MXFP8_GB300_H */

/*
 * moe.h -- C ABI of libmoe, a GB300 (sm_103a) weight-only INT4/INT8 MoE expert layer.
 *
 * The layer: router softmax + top-k, stable sort of (token, slot) rows by expert id,
 * grouped GEMM over the experts whose INT4/INT8 weights are dequantized inside the
 * kernel, activation, second grouped GEMM, un-permute and combine weighted by the gate
 * ("expert_scale"), plus an optional unquantized 16-bit shared expert.
 *
 * Passages cited:
 *   [FT]      "Who Says Elephants Can't Run: Bringing Large Scale MoE Models into Cloud
 *             Scale Production" (paper review page): section 3 'core formulas' (expert
 *             quantization, Algorithm 1), 'optimized I2F conversion' (8-bit and 4-bit
 *             dequantization), 'workflow' (token routing by sort, grouped GEMM,
 *             un-permute with expert_scale), Figure 1 (grouped GEMM, one sub-matrix per
 *             expert; pruned experts load no weights), section 4 table (fused GEMM +
 *             dequantization).
 *   [Specter] "Specter: Fast MoE Inference via Quantization-Enabled Multi-Step Speculative
 *             Offloading": background on MoE (router top-k) and on GPTQ INT4 (symmetric,
 *             group size 128; router, attention and shared expert stay 16-bit); method
 *             step 5 (group tokens by expert so per-token GEMV becomes per-expert GEMM,
 *             then scatter back).
 *
 * Conventions for every call:
 *   - Pointers are DEVICE pointers owned by the caller unless a name starts with host_.
 *     The library allocates nothing and never synchronizes; work is enqueued on `stream`
 *     (a cudaStream_t; NULL = the legacy default stream).  Buffers must stay alive until
 *     the stream has finished the work.
 *   - Every device pointer must be 16-byte aligned.  Row-major layouts, no padding.
 *   - Return value: MOE_OK (0) or a negative moe_status.  Arguments are validated on the
 *     host before anything is enqueued; on error nothing is enqueued and
 *     moe_last_error_string() (thread-local) says why.  MOE_ERR_CUDA reports a launch
 *     failure returned by the CUDA runtime.
 *   - Sizes are int64_t; dtypes are moe_dtype values.
 */
#ifndef MOE_H_
#define MOE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *moe_stream_t; /* identical to cudaStream_t */

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = -1, /* null/misaligned pointer, bad size, bad enum */
  MOE_ERR_UNSUPPORTED = -2, /* valid but unsupported shape / dtype combination */
  MOE_ERR_WORKSPACE = -3,   /* workspace smaller than the matching *_workspace_size */
  MOE_ERR_CUDA = -4,        /* the CUDA runtime rejected a launch */
  MOE_ERR_DEVICE_CHECK = -5 /* checked build: a kernel found an out-of-range index (moe_check_status) */
} moe_status;

typedef enum { MOE_F16 = 0, MOE_BF16 = 1, MOE_F32 = 2 } moe_dtype;

typedef enum { MOE_ACT_NONE = 0, MOE_ACT_RELU = 1, MOE_ACT_GELU = 2, MOE_ACT_SWIGLU = 3 } moe_act;

/* Thread-local text of the last error returned by this library on the calling thread. */
const char *moe_last_error_string(void);

/* ABI version (bumped on any incompatible change). */
int moe_version(void);

/* Device-side status.  Kernels that wait on on-chip barriers bound every wait (about a
 * second); when one expires the kernel records a nonzero code in a device word, drains its
 * own asynchronous work, releases its tensor memory and returns early (its outputs are then
 * incomplete).  This call synchronizes `stream`, copies the code to *host_code (0 = no
 * error) and clears it. */
int moe_device_error(moe_stream_t stream, int32_t *host_code);

/* Bounds-checked build.  libmoe_checked.so is this library compiled with MOE_CHECKED=1: its
 * kernels check every index they read from device memory before using it -- expert ids
 * (moe_permute: in [0, E)), expert row offsets (grouped GEMMs: 0 <= offsets[e] <=
 * offsets[e+1] <= R) and permutation entries (moe_unpermute_combine: inv_perm in [0, T*k)) --
 * skip the access when one is out of range and record the kind of violation in a device
 * check word; nothing faults and nothing traps.  A GEMM whose offsets fail the check computes
 * nothing (its output is left as it was).  The plain build does none of these checks (see each
 * call for what out-of-range input does there).
 * moe_checked_build: 1 in the checked library, 0 in the plain one.
 * moe_check_status: synchronizes `stream`, reads and clears the check word into *host_flags
 * (bit 1: expert id, bit 2: offsets, bit 4: permutation entry; always 0 in the plain build)
 * and returns MOE_ERR_DEVICE_CHECK if any bit is set, else MOE_OK. */
int moe_checked_build(void);
int moe_check_status(moe_stream_t stream, int32_t *host_flags);

/* ------------------------------------------------------------------------------------
 * Weight packing.  [FT] Algorithm 1: W (E, M, N) integer codes, M = reduction dim,
 * N = output channel; scales S (E, 1, N) per output channel.  [Specter] GPTQ: group size
 * 128 shares one scale, read as scales (E, K/128, N).  [FT] optimized I2F: codes are
 * stored offset-binary so the kernel can OR them into the mantissa of a 16-bit magic
 * number: INT8 byte u = q + 128 (the page's 1152 = 1024 + 128), INT4 nibble u = q + 8.
 * [FT] 4-bit layout: each 32-bit word holds 8 consecutive reduction-dim elements
 * e0..e7 of one output channel with nibble slot p (bits 4p..4p+3) holding
 * e_{sigma(p)}, sigma = (0,2,4,6,1,3,5,7), so bits 4p and 16+4p hold the pair
 * (e_{2p}, e_{2p+1}).
 *
 * Packed buffer layout (bytes, all regions 256-byte aligned):
 *   bits 4 : words  uint32 (E, N, K/8)   at offset 0
 *   bits 8 : words  uint32 (E, N, K/4)   at offset 0, byte b of a word = element 4j+b
 *   bits 16: values w_dtype (E, N, K)    at offset 0 (plain transpose, no scales)
 *   scales : w_dtype (E, G, N), G = 1 (group 0) or K/128 (group 128), at offset
 *            moe_packed_scale_offset(); absent for bits 16.
 * ------------------------------------------------------------------------------------ */

/* Bytes of the packed buffer; 0 if the arguments are invalid. */
size_t moe_packed_size(int64_t E, int64_t K, int64_t N, int bits, int group);
/* Byte offset of the scale region inside the packed buffer. */
size_t moe_packed_scale_offset(int64_t E, int64_t K, int64_t N, int bits);

/* codes: int8 (E, K, N), one signed code per byte, |q| <= 7 (bits 4; -8 allowed) or any
 *        int8 (bits 8).  For bits 16, `codes` points to the 16-bit weights (E, K, N) of
 *        type w_dtype and `scales` must be NULL.
 * scales: w_dtype (E, G, N) (copied into the packed buffer).
 * w_dtype: MOE_F16 or MOE_BF16 -- the scale / 16-bit weight type (the activation type).
 * group: 0 (per output channel) or 128.  K % 8 == 0 (bits 4), K % 4 == 0 (bits 8),
 *        K % 128 == 0 when group == 128, N % 8 == 0.
 * packed: device buffer of at least moe_packed_size() bytes. */
int moe_pack_weights(const void *codes, const void *scales, int w_dtype, int64_t E, int64_t K,
                     int64_t N, int bits, int group, void *packed, size_t packed_bytes,
                     moe_stream_t stream);

/* [FT] Algorithm 1 from the packed buffer: w_out[e, m, n] = RN_out(q[e, m, n] * S[e, g(m), n]),
 * one rounding of the exact product.  Uses the same device I2F routine as the GEMM
 * mainloops.  out_dtype: MOE_F16, MOE_BF16 or MOE_F32.  w_out: (E, K, N) row-major. */
int moe_dequant(const void *packed, int w_dtype, int64_t E, int64_t K, int64_t N, int bits,
                int group, int out_dtype, void *w_out, moe_stream_t stream);

/* ------------------------------------------------------------------------------------
 * Router.  [Specter] background on MoE: the router scores every token and only the top-k
 * experts run; [FT] model table: top-1 Switch gating; [Specter] GPTQ background: the
 * router stays in 16-bit (fp32 allowed).
 *   logits[t, e] = sum_m x[t, m] * w_router[m, e] (+ bias[e]), fp32 accumulation;
 *   ids[t, :]    = the k largest logits, descending, equal logits -> lower expert id;
 *   gate_w[t, j] = softmax over all E logits, evaluated at ids[t, j] (fp32); with
 *                  renormalize != 0 the k gates of a token are divided by their sum.
 * x: (T, d) x_dtype (F16|BF16).  w_router: (d, E) wr_dtype (F32|F16|BF16; 16-bit must
 * equal x_dtype).  bias: fp32 (E) or NULL.  ids: int32 (T, k).  gate_w: fp32 (T, k).
 * 1 <= k <= E <= 256, d % 8 == 0.  T == 0 is allowed (nothing is enqueued).
 * workspace: >= moe_route_topk_workspace_size(T, d, E) bytes for 16-bit router weights (fp32
 * partial logits of the K splits, summed in split order); unused for fp32 router weights. */
size_t moe_route_topk_workspace_size(int64_t T, int64_t d, int64_t E);
int moe_route_topk(const void *x, int x_dtype, const void *w_router, int wr_dtype,
                   const float *bias, int64_t T, int64_t d, int64_t E, int k, int renormalize,
                   int32_t *ids, float *gate_w, void *workspace, size_t workspace_bytes,
                   moe_stream_t stream);

/* ------------------------------------------------------------------------------------
 * Permute.  [FT] workflow: append the row index to the gating tuple, sort by expert id,
 * permute the activation matrix.  Flat row f = t*k + j.  The sort is stable in f:
 *   offsets[e] = number of flat rows with an expert id < e (offsets[E] = T*k);
 *   perm[p] = f for the p-th row in (expert id, f) order; inv_perm[f] = p;
 *   xp[p, :] = x[perm[p] / k, :].
 * ids: int32 (T, k), every id in [0, E).  offsets: int32 (E+1).  perm, inv_perm: int32
 * (T*k).  xp: (T*k, d) x_dtype.  workspace: >= moe_permute_workspace_size(T, E, k) bytes
 * (may be NULL when that size is 0).
 * Out-of-range ids (< 0 or >= E) are dropped: such a row gets no position, the offsets count
 * only the rows with valid ids (offsets[E] is then below T*k), its inv_perm entry is -1 and
 * perm entries from offsets[E] on are left unwritten; moe_unpermute_combine skips inv_perm
 * entries outside [0, T*k), so a dropped row adds nothing to the output.  The checked build
 * also sets bit 1 of the check word. */
size_t moe_permute_workspace_size(int64_t T, int64_t E, int k);
int moe_permute(const int32_t *ids, const void *x, int x_dtype, int64_t T, int64_t d, int64_t E,
                int k, int32_t *offsets, int32_t *perm, int32_t *inv_perm, void *xp,
                void *workspace, size_t workspace_bytes, moe_stream_t stream);

/* ------------------------------------------------------------------------------------
 * Grouped GEMM with fused dequant and activation.  [FT] Figure 1 and workflow: one
 * launch computes every expert's sub-matrix product; [FT] section 4: dequantization
 * fused into the GEMM; [FT] Figure 1: experts with no rows load no weights.
 *
 * For every expert e with rows [offsets[e], offsets[e+1]) of `a`:
 *   acc = a[rows, :] . dq(W_e)        (16-bit operands, fp32 accumulation)
 *   out[rows, :] = act(acc)           act NONE | RELU | GELU (exact erf) : out (R, N)
 *                                     SWIGLU: silu(acc[:, :N/2]) * acc[:, N/2:] : (R, N/2)
 * a: (R, K) a_dtype (F16|BF16) row-major, R = total rows.  packed_w: from
 * moe_pack_weights with this (E, K, N, bits, group) and w_dtype == a_dtype.
 * offsets: int32 (E+1) device, non-decreasing, offsets[E] <= R (output rows from offsets[E] on
 * are left unspecified); NULL means one group holding all R rows (then E must be 1).  Offsets outside
 * these rules are undefined behaviour in the plain build; the checked build computes nothing
 * and sets bit 2 of the check word.
 * out_dtype: F16 | BF16 | F32.  With act NONE the output may be requested as fp32
 * split-K partials instead (see moe_grouped_gemm_partials).
 * workspace: >= moe_grouped_gemm_workspace_size(...) bytes.
 * Per-channel scales are applied to the fp32 accumulator (an exact reformulation of
 * Algorithm 1 up to rounding order); group-128 scales are applied in the mainloop as
 * RN(q * s) in the operand dtype, as Algorithm 1 states. */
/* Which kernel a grouped GEMM with these arguments (offsets given) runs, judged from the
 * average rows per active expert a = ceil(R / min(E, R)): 2 = the decode weight-stream kernel
 * (a <= 16); 1 = the tcgen05 tensor-memory kernel (a >= 17, when the shape suits it:
 * K % 128 == 0, N % 128 == 0, or for SWIGLU (N/2) % 64 == 0); 0 = the warp-MMA tile kernel
 * (the rest). */
int moe_gemm_path(int64_t R, int64_t E, int64_t K, int64_t N, int bits, int group, int act);
size_t moe_grouped_gemm_workspace_size(int64_t R, int64_t E, int64_t K, int64_t N, int bits,
                                       int act);
int moe_grouped_gemm_w4a16(const void *a, int a_dtype, const void *packed_w, int64_t E, int64_t K,
                           int64_t N, int group, const int32_t *offsets, int64_t R, int act,
                           void *out, int out_dtype, void *workspace, size_t workspace_bytes,
                           moe_stream_t stream);
int moe_grouped_gemm_w8a16(const void *a, int a_dtype, const void *packed_w, int64_t E, int64_t K,
                           int64_t N, int group, const int32_t *offsets, int64_t R, int act,
                           void *out, int out_dtype, void *workspace, size_t workspace_bytes,
                           moe_stream_t stream);
/* moe_grouped_gemm_w4a16 for callers that cannot allocate device memory.  The pages have no
 * counterpart to this call: it exists for callers whose device memory is owned by someone else
 * (a runtime that pools all memory at start-up, a host framework that hands plug-ins only their
 * inputs and outputs) or that must not call cudaMalloc while a stream is being captured.
 * Same arguments and results as moe_grouped_gemm_w4a16 minus the workspace: the split-K
 * partial sums go to a 2 MiB array inside the library (a file-scope __device__ variable that
 * every GPU loading the library holds until exit).  Calls needing more scratch than that
 * (moe_grouped_gemm_workspace_size > 2 MiB) return MOE_ERR_UNSUPPORTED without launching.
 * Nothing is allocated: no cudaMalloc, cudaFree or allocating library call.  The first call on
 * a device looks up the array's device address (cudaGetSymbolAddress) with that device
 * current; make that first call before any stream capture.  The address is kept per device
 * index and belongs to the device's primary context (the one the CUDA runtime uses): a caller
 * that runs this call under a context of its own, or after resetting the device
 * (cudaDeviceReset), must not use it.  Every call on a device shares the
 * one array and leaves its last contents there (each call overwrites every partial it reads,
 * so nothing needs clearing); calls that overlap on the GPU (different streams, or several
 * host threads) race on it and must be serialized by the caller. */
int moe_grouped_gemm_w4a16_static(const void *a, int a_dtype, const void *packed_w, int64_t E,
                                  int64_t K, int64_t N, int group, const int32_t *offsets, int64_t R,
                                  int act, void *out, int out_dtype, moe_stream_t stream);
/* Unquantized 16-bit weights (bits 16 packing): used for the shared expert. */
int moe_grouped_gemm_w16a16(const void *a, int a_dtype, const void *packed_w, int64_t E,
                            int64_t K, int64_t N, const int32_t *offsets, int64_t R, int act,
                            void *out, int out_dtype, void *workspace, size_t workspace_bytes,
                            moe_stream_t stream);

/* ------------------------------------------------------------------------------------
 * Un-permute and combine.  [FT] workflow: restore the row order and apply expert_scale;
 * [Specter] step 5: scatter back to the original positions.
 *   out[t, c] = sum_{j<k} gate_w[t, j] * yp[inv_perm[t*k + j], c]  (+ shared[t, c])
 * summed in fp32 in j order, rounded once to out_dtype.  An inv_perm entry outside
 * [0, T*k) (a row moe_permute dropped) contributes nothing; the checked build also sets bit 4
 * of the check word.
 * yp: (T*k, d) yp_dtype (F32|F16|BF16).  shared: (T, d) shared_dtype or NULL.
 * out: (T, d) out_dtype (F16|BF16|F32). */
int moe_unpermute_combine(const void *yp, int yp_dtype, const int32_t *inv_perm,
                          const float *gate_w, const void *shared, int shared_dtype, int64_t T,
                          int64_t d, int k, void *out, int out_dtype, moe_stream_t stream);

/* ------------------------------------------------------------------------------------
 * Shared expert.  [Specter] core method: the shared expert stays unquantized 16-bit.
 * Ungated SwiGLU FFN: out = (silu(x.Wg) * (x.Wu)) . Wd, with Wg|Wu = w_gate_up (d, 2Fs)
 * (gate columns first) and Wd (Fs, d), both packed with bits 16 (E = 1).
 * x: (T, d) x_dtype; out: (T, d) out_dtype (F32 | x_dtype).
 * workspace: >= moe_shared_expert_workspace_size(T, d, Fs). */
size_t moe_shared_expert_workspace_size(int64_t T, int64_t d, int64_t Fs);
int moe_shared_expert(const void *x, int x_dtype, const void *w_gate_up_packed,
                      const void *w_down_packed, int64_t T, int64_t d, int64_t Fs, void *out,
                      int out_dtype, void *workspace, size_t workspace_bytes,
                      moe_stream_t stream);

/* ------------------------------------------------------------------------------------
 * Whole layer: route -> permute -> FC1 (+act) -> FC2 -> un-permute/combine (+ shared).
 * Same arithmetic as chaining the calls above; intermediates live in `workspace`.
 * ------------------------------------------------------------------------------------ */
typedef struct {
  int64_t d;        /* hidden size */
  int64_t F;        /* expert intermediate size (FC1 has 2F columns for SWIGLU) */
  int64_t E;        /* routed experts */
  int32_t k;        /* experts per token */
  int32_t act;      /* moe_act for FC1 */
  int32_t bits;     /* 4 | 8 */
  int32_t group;    /* 0 | 128 */
  int32_t dtype;    /* activation / scale / shared-weight dtype: F16 | BF16 */
  int32_t router_dtype; /* F32 | dtype */
  int32_t renormalize;
  int64_t Fs;       /* shared-expert intermediate size, 0 = none */
} moe_layer_desc;

typedef struct {
  const void *w_router;      /* (d, E) router_dtype */
  const float *router_bias;  /* (E) or NULL */
  const void *w1;            /* packed (E, K=d, N=F1) */
  const void *w2;            /* packed (E, K=F, N=d) */
  const void *ws_gate_up;    /* packed bits 16 (1, d, 2Fs) or NULL */
  const void *ws_down;       /* packed bits 16 (1, Fs, d) or NULL */
} moe_layer_weights;

/* Device pointers into a layer workspace after moe_layer_forward (routing results). */
typedef struct {
  int32_t *ids;      /* (T, k) */
  float *gate_w;     /* (T, k) */
  int32_t *offsets;  /* (E+1) */
  int32_t *perm;     /* (T*k) */
  int32_t *inv_perm; /* (T*k) */
} moe_layer_routing;

/* Bytes of a layer workspace that serves every moe_layer_forward call of at most T tokens (the
 * largest requirement over T' <= T: a smaller batch can need more, its split-K plans writing
 * partial sums in more slices). */
size_t moe_layer_workspace_size(const moe_layer_desc *desc, int64_t T);
int moe_layer_routing_view(const moe_layer_desc *desc, int64_t T, void *workspace,
                           moe_layer_routing *view);
/* Number of kernels one moe_layer_forward(desc, T tokens) enqueues (0 if invalid or T == 0). */
int moe_layer_launch_count(const moe_layer_desc *desc, int64_t T);
/* How moe_layer_forward runs a decode step.  [Specter] technical novelty and method step (5):
 * the draft runs all expert sub-computations of a step in one fused launch.  A layer of T <= 32
 * tokens with 4-bit expert weights, E <= 256 and T*k <= 256 can run as ONE kernel launch (router,
 * top-k, sort, FC1 + activation, FC2, shared expert, combine; work units ordered by their
 * dependencies, every wait bounded), the same arithmetic as the chain of kernels; its control
 * words live in the layer workspace and are cleared by a memset before the launch, except while
 * `stream` is being captured (every completed launch leaves them zero again; a capture must follow
 * one uncaptured call on the same workspace, as moe_layer_graph_create does; after
 * moe_device_error reports a code, make one uncaptured call before replaying a graph).
 * mode 0 (default): automatic -- one launch when the step streams at most 16 MB of expert and
 * shared-expert weights (there launch and dependency latency dominate; measured on GB300), else
 * the chain; mode 1: always the chain; mode 2: one launch whenever the layer allows it.
 * Process-wide; returns the previous mode, or MOE_ERR_INVALID_ARG. */
int moe_set_decode_mode(int mode);
/* The quantized tcgen05 GEMM runs as CTA pairs (clusters of two CTAs, tcgen05 cta_group::2,
 * M = 256: each SM copies half of a tile's activation rows) when the output channels come in
 * blocks of 256 (SWIGLU: 128 gate + 128 up) and the device can place the pairs, else on single
 * CTAs (M = 128): the same arithmetic in the same order (bit-identical results).  Process-wide,
 * default 0 (single CTAs: on GB300 the pairs measured slower, Phi-shaped FC1 1.73 against
 * 1.27 ms, because every K block's readiness has to cross to the other CTA); returns the
 * previous setting, or MOE_ERR_INVALID_ARG. */
int moe_set_gemm_pairs(int on);
/* x: (T, d) dtype; out: (T, d) dtype.  With a shared expert (Fs > 0) the shared expert's kernels
 * run on a second stream owned by the library (one per calling thread and device, created on
 * first use), forked from `stream` before the router and joined back into `stream` before the
 * combine: all work of the call is ordered after what was enqueued on `stream` before it, and
 * everything enqueued on `stream` after it is ordered after all of it, as for a single-stream
 * call; a capture of `stream` records both branches.  The kernels of the chain are launched with
 * programmatic stream serialization (each waits for its predecessor before touching memory). */
int moe_layer_forward(const moe_layer_desc *desc, const moe_layer_weights *w, const void *x,
                      int64_t T, void *out, void *workspace, size_t workspace_bytes,
                      moe_stream_t stream);

/* Stage boundaries recorded by moe_layer_forward_profiled. */
enum {
  MOE_STAGE_START = 0,   /* before the router */
  MOE_STAGE_ROUTED = 1,  /* after route + top-k */
  MOE_STAGE_PERMUTED = 2,/* after the counting sort and row gather */
  MOE_STAGE_FC1 = 3,     /* after FC1 (+ activation, + split-K reduction) */
  MOE_STAGE_FC2 = 4,     /* after FC2 */
  MOE_STAGE_SHARED = 5,  /* after the shared expert (same as FC2 when Fs == 0) */
  MOE_STAGE_DONE = 6,    /* after un-permute / combine */
  MOE_STAGE_COUNT = 7
};
/* moe_layer_forward that also records stage_events[i] (cudaEvent_t handles created by the
 * caller, MOE_STAGE_COUNT of them) on `stream` at each stage boundary, so the caller can
 * time every kernel of the chain inside a real run.  stage_events == NULL is identical to
 * moe_layer_forward. */
int moe_layer_forward_profiled(const moe_layer_desc *desc, const moe_layer_weights *w,
                               const void *x, int64_t T, void *out, void *workspace,
                               size_t workspace_bytes, moe_stream_t stream,
                               void *const *stage_events);

/* ---- Lossless BF16 bit-field codec ("ZipMoE" summary page, method details) ------------------
 * A BF16 expert tensor is stored as two byte planes: exp[i] = bits 14..7 of element i (the
 * low-entropy part the host compresses), sm[i] = sign (bit 7) | mantissa (bits 6..0).
 * moe_bf16_recombine merges the planes back into BF16 bit patterns, bit for bit;
 * moe_bf16_split is its inverse.  n elements; all pointers device, 16-byte aligned; n may be
 * any size (the last n % 16 elements take a scalar path).  Errors: MOE_ERR_INVALID_ARG. */
int moe_bf16_recombine(const uint8_t *exp, const uint8_t *sm, int64_t n, uint16_t *out, moe_stream_t stream);
int moe_bf16_split(const uint16_t *in, int64_t n, uint8_t *exp, uint8_t *sm, moe_stream_t stream);

/* ---- Expert lookahead buffer ("Specter" summary page, method steps (2)-(3)) -----------------
 * moe_elb_accumulate: counts (L, E) int32, row-major, += for every layer j and expert e the
 * number of draft steps i < S with e among ids[j, i, 0..k-1] (ids (L, S, k) int32: the routed
 * ids of S draft steps; an expert counts once per step, ids outside [0, E) are skipped).
 * moe_elb_topm: for every layer, the min(M, E) experts with the largest counts, by count
 * descending then expert id ascending -> experts (L, min(M, E)) and their counts vals (same
 * shape).  Integer results, independent of launch configuration.  Device pointers; errors:
 * MOE_ERR_INVALID_ARG (E > 256, k > 64, L > 65535, NULL). */
int moe_elb_accumulate(const int32_t *ids, int64_t L, int64_t S, int k, int64_t E, int32_t *counts,
                       moe_stream_t stream);
int moe_elb_topm(const int32_t *counts, int64_t L, int64_t E, int M, int32_t *experts, int32_t *vals,
                 moe_stream_t stream);
/* Both in one launch: accumulate the window's ids into counts, then write every layer's top-M of
 * the updated counts (same results as moe_elb_accumulate followed by moe_elb_topm). */
int moe_elb_step(const int32_t *ids, int64_t L, int64_t S, int k, int64_t E, int32_t *counts, int M,
                 int32_t *experts, int32_t *vals, moe_stream_t stream);

/* ---- The layer chain as one CUDA graph (decode steps) ---------------------------------------
 * A decode step runs the whole chain on a few tokens, where each kernel is short and the chain's
 * cost is launch and dependency latency ("Specter", technical novelty: one launch for all expert
 * sub-computations of a draft step).  moe_layer_graph_create runs moe_layer_forward once on
 * `stream` (this also fills per-kernel caches that must not change during capture), then captures
 * a second call into a CUDA graph and instantiates it.  The graph is bound to the pointers given:
 * x, out, workspace and the weights must stay allocated and at the same addresses while the
 * graph exists; the caller changes the input by writing into x.  T is fixed.  The caller owns
 * the handle and releases it with moe_layer_graph_destroy.  `stream` must not be capturing
 * already.  Errors: the moe_layer_forward checks, MOE_ERR_CUDA if capture or instantiation
 * fails (no graph is returned then). */
typedef struct moe_layer_graph_s *moe_layer_graph;
int moe_layer_graph_create(const moe_layer_desc *desc, const moe_layer_weights *w, const void *x,
                           int64_t T, void *out, void *workspace, size_t workspace_bytes,
                           moe_stream_t stream, moe_layer_graph *graph);
/* One replay of the captured chain on `stream` (asynchronous). */
int moe_layer_graph_launch(moe_layer_graph graph, moe_stream_t stream);
/* Frees the graph (NULL is a no-op).  No replay may be pending. */
int moe_layer_graph_destroy(moe_layer_graph graph);

#ifdef __cplusplus
}
#endif

#endif /* MOE_H_ */

/*
 * tl_encoder.h -- C ABI of the GB300 (sm_103a) masked post-LN encoder stack.
 *
 * What it computes.  The forward pass of a stack of transformer encoder
 * layers, as the three source pages describe the task ("Hyper-optimized
 * megakernel-hybrid transformer inference", "KernelForge", "Implement a GPU
 * Kernel for a Transformer Layer").  For every layer, in order:
 *
 *   qkv = x W_qkv^T + b_qkv                    fused QKV projection
 *   ctx = MHA(q, k, v)                         causal + key-padding mask
 *   y   = LayerNorm1(x + ctx W_o^T + b_o)      post-LN, eps 1e-5
 *   x'  = LayerNorm2(y + gelu(y W_1^T + b_1) W_2^T + b_2)   exact-erf GELU
 *
 * with no dropout.  Attention uses the scale 1/sqrt(dh); key j is visible to
 * query row i of sequence b iff j <= i and j < valid_len[b]; padded query rows
 * (i >= valid_len[b]) are computed by the same rule and returned.  The single
 * entry point that handles every shape follows the megakernel page's section
 * "Appendix" (one callable for all cases) and KernelForge's "What it does"
 * (a frozen per-shape plan chosen at run time with no autotuning).
 *
 * Numbers.  Inputs, weights and outputs use one I/O dtype (fp32, fp16 or
 * bf16).  The residual stream, LayerNorm, softmax and every accumulator are
 * fp32; 16-bit tensor-core operands that are activations are carried as a
 * (hi, lo) pair so that products keep about fp32 accuracy.  Results meet the
 * pages' per-element gate |err| <= 0.002 OR |err| <= 0.02 |ref| against an
 * fp64 evaluation of the same function.
 *
 * Conventions for every call.
 *  - Device pointers are plain CUDA device addresses of the current device;
 *    "stream" is a cudaStream_t passed as void* (NULL = the legacy stream).
 *  - Synchronous argument checks return a status before anything is launched.
 *    Errors that depend on device data (a valid_len outside [1, L], a device
 *    wait that timed out) are recorded in a per-handle device status word and
 *    reported by tl_encoder_get_status().
 *  - No call is thread-safe on one handle; distinct handles are independent.
 */
#ifndef TL_ENCODER_H
#define TL_ENCODER_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { TL_F32 = 0, TL_F16 = 1, TL_BF16 = 2 } tl_dtype;

typedef enum {
  TL_OK = 0,
  TL_ERR_INVALID_ARG = 1,        /* null pointer, non-positive size, misaligned buffer   */
  TL_ERR_UNSUPPORTED_SHAPE = 2,  /* d_model % n_heads != 0, head_dim too large, path n/a  */
  TL_ERR_CUDA = 3,               /* a CUDA runtime call failed                           */
  TL_ERR_OUT_OF_MEMORY = 4,      /* create could not allocate the packed weights         */
  TL_ERR_WORKSPACE_TOO_SMALL = 5,
  TL_ERR_BAD_VALID_LEN = 6,      /* some valid_len[b] was outside [1, L]; it was clamped */
  TL_ERR_DEVICE_TIMEOUT = 7      /* a bounded device-side wait gave up                   */
} tl_status;

/* Execution paths.  TL_PATH_AUTO picks by shape (the frozen dispatch table).
 * The others force one path, for cross-checks; a forced path that cannot run
 * the shape makes forward return TL_ERR_UNSUPPORTED_SHAPE.
 *   SIMT      generic fp32 CUDA-core kernels, every shape (head_dim <= 128)
 *   LAYERED   tcgen05/TMEM GEMMs fed by TMA with fused epilogues, plus the
 *             flash-attention kernel; one launch per step per layer
 *   MEGA      sequence-resident megakernel: every layer of a 128-row tile of
 *             whole sequences in one CTA, activations kept on chip (16-bit
 *             I/O, d_model 128, tensor cores); for fp32 I/O with d_model <= 64,
 *             head_dim <= 32, L <= 64 and d_ff <= 256, one sequence per CTA
 *             on CUDA cores
 *   DAG       persistent task-graph megakernel for fp32 I/O and few tokens:
 *             one launch per forward; CTAs pop (layer, step, row block, tile)
 *             tasks from a queue and wait on per-row-block counters
 *             ("Hyper-optimized megakernel-hybrid transformer inference",
 *             section "Problem decomposition")                              */
typedef enum {
  TL_PATH_AUTO = 0,
  TL_PATH_SIMT = 1,
  TL_PATH_LAYERED = 2,
  TL_PATH_MEGA = 3,
  TL_PATH_DAG = 4
} tl_path;

typedef struct tl_encoder tl_encoder; /* opaque handle */

/* One layer's parameters, every array in the handle's dtype, PyTorch's
 * [out, in] row-major weight layout:
 *   w_qkv [3d, d], b_qkv [3d]  rows 0..d-1 are Q, d..2d-1 K, 2d..3d-1 V; within
 *                              each block head h owns rows h*dh .. (h+1)*dh-1
 *   w_o [d, d], b_o [d]; ln1_g, ln1_b [d]
 *   w_1 [d_ff, d], b_1 [d_ff]; w_2 [d, d_ff], b_2 [d]; ln2_g, ln2_b [d]      */
typedef struct {
  const void *w_qkv, *b_qkv;
  const void *w_o, *b_o;
  const void *ln1_g, *ln1_b;
  const void *w_1, *b_1;
  const void *w_2, *b_2;
  const void *ln2_g, *ln2_b;
} tl_layer_weights;

/* Create a handle.  weights points to n_layers structs; their arrays may be
 * host or device memory (detected per pointer) and are copied and packed into
 * library-owned device memory, so the caller may free them on return.
 * Requires n_layers >= 1, d_model >= 16 and a multiple of 16, d_model %
 * n_heads == 0, head_dim = d_model / n_heads in [1, 128], d_ff >= 16 and a
 * multiple of 16.  Allocates (cudaMalloc) and synchronises the device once.
 * On error *out is set to NULL. */
tl_status tl_encoder_create(const tl_layer_weights *weights, int n_layers, int d_model,
                            int n_heads, int d_ff, tl_dtype dtype, tl_encoder **out);

/* Force an execution path (default TL_PATH_AUTO).  Host-only, no device work. */
tl_status tl_encoder_set_path(tl_encoder *h, tl_path path);

/* The path forward() would run for a batch of B sequences of length L.
 * Under TL_PATH_AUTO a shape listed in the library's frozen plan table
 * (KernelForge, section "What it does": candidates proven against the gate,
 * then timed, the winner frozen) takes the table's path; other shapes take
 * fixed rules by dtype, d_model, head width, sequence length and tokens. */
tl_status tl_encoder_plan(const tl_encoder *h, int B, int L, tl_path *path);

/* Split-K attention on the layered tensor-core path (KernelForge, section
 * "What's next": partition the key range and merge partial softmax states).
 * When a batch has too few (sequence, head, 128-query tile) items to keep
 * every SM busy behind the longest causal rows (batch 1, long sequences),
 * each tile's key range is cut into chunks of key_tiles x 64 keys that run
 * as separate work items; their partial states (unnormalised output, running
 * max, row sum) go to the workspace and the last chunk to finish merges
 * them.  key_tiles = -1 (the default) chooses per shape: the frozen plan
 * table's setting when the shape is in it (see tl_encoder_plan), else a
 * model of the persistent grid's load; 0 never splits, k in 1..4096 forces
 * chunks of k tiles.  Host-only; the workspace size depends on it.
 * TL_ERR_INVALID_ARG outside -1..4096. */
tl_status tl_encoder_set_attention_split(tl_encoder *h, int key_tiles);

/* CTA pairs for the layered path's GEMMs (tcgen05 cta_group::2; the
 * megakernel page, section "Problem decomposition", tried a 2-CTA cluster
 * variant).  A paired GEMM (at least 257 rows, an N tile of 64 or more) runs
 * on clusters of two CTAs that share one 256-row block: each CTA stages its
 * own 128 rows of the activation and half of the weight tile (each byte is
 * loaded once, by one CTA), and one MMA instruction of the leader CTA covers
 * all 256 rows.
 * enable = -1 (the default) pairs only the GEMM where GB300 measured a gain
 * (the FFN2 + LayerNorm GEMM over d_ff >= 2048 with 4096+ rows), 1 pairs
 * every GEMM the shape allows, 0 none.  Host-only.  TL_ERR_INVALID_ARG
 * outside -1..1. */
tl_status tl_encoder_set_gemm_pairs(tl_encoder *h, int enable);

/* Assisting CTAs for the sequence-resident megakernel ("Hyper-optimized
 * megakernel-hybrid transformer inference", section "Problem decomposition":
 * extra CTAs take part of the resident CTAs' work when the batch alone leaves
 * SMs idle).  When the batch's 128-row tiles fill at most half the SMs (and
 * d_ff >= 256), each tile runs on a cluster of two CTAs: the resident one and
 * a helper that computes half the heads' attention and half the FFN chunks,
 * handing context, FFN partial sums and activations over through distributed
 * shared memory.  enable = 1 uses it wherever possible; -1 (the default,
 * automatic) and 0 do not: on GB300 it measured within 2% of one CTA per
 * tile.  Host-only.  TL_ERR_INVALID_ARG outside -1..1. */
tl_status tl_encoder_set_mega_assist(tl_encoder *h, int enable);
/* *assisted = 1 when forward() on B x L runs the megakernel assisted. */
tl_status tl_encoder_mega_assisted(const tl_encoder *h, int B, int L, int *assisted);

/* The chunk size (in 64-key tiles) forward() would use for B x L: 0 when
 * the attention runs unsplit (or the path has no tensor-core attention). */
tl_status tl_encoder_attention_split(const tl_encoder *h, int B, int L, int *key_tiles);

/* Bytes of scratch device memory forward() needs for B sequences of length
 * L on the path it would choose.  0 is possible (then workspace may be NULL). */
tl_status tl_encoder_workspace_size(const tl_encoder *h, int B, int L, size_t *bytes);

/* The forward pass.  x [B, L, d_model] and out [B, L, d_model] are device
 * arrays in the handle's dtype, row-major, batch first, 16-byte aligned, and
 * must not overlap.  valid_len is a device int32 [B], each in [1, L]
 * (right padding: tokens valid_len[b] .. L-1 of sequence b are padding).
 * workspace is caller-owned device scratch of at least
 * tl_encoder_workspace_size() bytes, 256-byte aligned.  The call only
 * enqueues work on stream: it neither allocates nor synchronises.  B * L is
 * at most 2^30 tokens (and B * L * n_heads below 2^31); a larger batch
 * returns TL_ERR_UNSUPPORTED_SHAPE and is to be split by the caller. */
tl_status tl_encoder_forward(tl_encoder *h, const void *x, int B, int L,
                             const int32_t *valid_len, void *out, void *workspace,
                             size_t workspace_bytes, void *stream);

/* Graph mode (KernelForge, section "What we built": the launches of a
 * forward captured in a CUDA graph).  With enable = 1, a forward on the
 * layered path (several launches per layer) whose stream is not itself being
 * captured runs as follows: the first call for a given (B, L, x, valid_len,
 * out, workspace) launches the kernels as usual and also records them into a
 * CUDA graph on an internal stream; later calls with the same shape and
 * buffers launch that graph instead (the kernels read their buffers through
 * the recorded pointers, so the caller changes the contents, not the
 * addresses).  One graph is kept per handle; a new shape or buffer set
 * replaces it.  The recording call creates a stream and a graph (host and
 * device allocations by the driver), so unlike the plain forward it is not
 * allocation-free; replays are.  Other paths, per-kernel timing and a stream
 * under capture bypass it.  enable = 0 (the default) frees the graph. */
tl_status tl_encoder_set_graphs(tl_encoder *h, int enable);
/* How many graphs graph mode recorded and how many forwards replayed one. */
tl_status tl_encoder_graph_stats(const tl_encoder *h, long long *captures, long long *replays);

/* Bytes of device workspace tl_encoder_forward_host() needs: device copies of
 * x, valid_len and out, plus the forward's own scratch for one batch slice
 * (two slices' worth when the call pipelines more than one slice).  Depends
 * on the handle's slice setting (tl_encoder_set_host_chunks). */
tl_status tl_encoder_host_workspace_size(const tl_encoder *h, int B, int L, size_t *bytes);

/* The forward pass on HOST buffers: copies x [B, L, d] and valid_len [B] from
 * host memory to the workspace, runs the forward, copies the result to out
 * (host), and synchronises before returning.  The batch is cut into slices of
 * whole sequences that alternate between two internal streams (forked from
 * and joined back to stream), so that one slice's upload, another's kernels
 * and a third's download overlap; each sequence is computed from its own
 * tokens only, so the result is bit-identical to tl_encoder_forward on the
 * whole batch, and every slice runs the path chosen for the whole batch.
 * Pinned host memory makes the copies asynchronous DMA; pageable memory also
 * works, with less overlap.  On error, no copy is still in flight on return. */
tl_status tl_encoder_forward_host(tl_encoder *h, const void *x_host, int B, int L,
                                  const int32_t *valid_len_host, void *out_host,
                                  void *workspace, size_t workspace_bytes, void *stream);

/* Batch slices tl_encoder_forward_host pipelines: 0 (the default) picks them
 * from the batch's size and path (slices of at least 8 MiB, at most 8; at
 * most 2 on the layered path; 1 on the task-graph path; with 4 or more, a
 * quarter slice is also cut off each end so that the first upload and the
 * last download are short), 1 turns the pipeline off, 2..64 asks for that
 * many equal slices (capped at B).  TL_ERR_INVALID_ARG outside
 * 0..64. */
tl_status tl_encoder_set_host_chunks(tl_encoder *h, int chunks);

/* Synchronise stream, then read and clear the handle's device status word:
 * TL_OK, TL_ERR_BAD_VALID_LEN or TL_ERR_DEVICE_TIMEOUT (the first error seen
 * since the last call). */
tl_status tl_encoder_get_status(tl_encoder *h, void *stream);

/* Free the packed weights and the handle (synchronises the device).  NULL is
 * accepted. */
tl_status tl_encoder_destroy(tl_encoder *h);

/* The forward pass with no caller-supplied workspace and no allocation of
 * any kind, for callers that cannot call cudaMalloc (or any allocating
 * routine) where they run the forward: a host that has handed out its whole
 * device-memory budget in advance, a plugin or real-time loop that is not
 * allowed the implicit synchronisation an allocation may bring, code whose
 * allocator owns every device pointer and offers no scratch.  The source
 * pages have no counterpart; this is a property of the library, not of the
 * method.
 *
 * Scratch comes from one array of TL_STATIC_SCRATCH_BYTES of device memory
 * that the library declares statically: every GPU that loads the library
 * holds it until the process exits.  A shape whose workspace
 * (tl_encoder_workspace_size) exceeds it is rejected with
 * TL_ERR_WORKSPACE_TOO_SMALL before anything is launched.  tl_encoder_create
 * looks up the array's device address (cudaGetSymbolAddress) with the
 * handle's device current and keeps it in the handle, so the address lives
 * and dies with the same context as the handle's weights; this call itself
 * neither allocates nor looks anything up (TL_ERR_CUDA if that lookup failed
 * at create).  Every call on a device shares the one array and it keeps
 * the last call's contents (the forward zeroes what it needs zeroed itself);
 * calls that overlap on the GPU -- on two streams, or from two handles --
 * race on it, so serialise them.  Otherwise as tl_encoder_forward (x, out,
 * valid_len are the caller's device buffers; h must belong to the current
 * device). */
#define TL_STATIC_SCRATCH_BYTES ((size_t)32 << 20)
tl_status tl_encoder_forward_static(tl_encoder *h, const void *x, int B, int L,
                                    const int32_t *valid_len, void *out, void *stream);

/* Per-kernel timing.  While enabled, forward() records a CUDA event pair
 * around each of its kernel launches on the launch stream (capacity pairs at
 * most; later launches are not timed).  tl_encoder_read_timing() synchronises
 * the device, then returns for kernel class k (0 <= k < TL_KERNEL_CLASSES)
 * the summed device time in ms and the number of timed launches, and
 * tl_encoder_reset_timing() forgets everything recorded so far.  Enabling
 * creates events (host allocation); disabling destroys them. */
#define TL_KERNEL_CLASSES 16
tl_status tl_encoder_enable_timing(tl_encoder *h, int enable, int capacity);
tl_status tl_encoder_read_timing(tl_encoder *h, int k, float *total_ms, int *launches);
tl_status tl_encoder_reset_timing(tl_encoder *h);
/* Name of kernel class k ("" past the last class). */
const char *tl_kernel_class_name(int k);

/* Math self-check: for n device floats x, writes the exact-erf GELU
 * 0.5 x (1 + erff(x / sqrt 2)) to y_erf and the library's branch-free form
 * (erf from Abramowitz & Stegun 7.1.28, |erf error| <= 3e-7) to y_fast.
 * Enqueued on stream; no synchronisation. */
tl_status tl_eval_gelu(const float *x, float *y_erf, float *y_fast, size_t n, void *stream);

/* Static description of a status code. */
const char *tl_status_string(tl_status s);

#ifdef __cplusplus
}
#endif

#endif /* TL_ENCODER_H */

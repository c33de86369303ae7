/*
 * cbq.h -- C ABI of the codebook-4bit quantized matvec library (libcbq.so).
 *
 * The library computes the low-bit quantized matrix-vector product that
 * streams 4-bit codebook weights for single-token decode and for small-batch
 * speculative verification (n = 1..5 activation columns), over dense
 * projections and over top-k routed MoE experts with the SwiGLU split and the
 * router-weighted combine fused in.  Every step runs in CUDA kernels built for
 * sm_103a; there is no CPU fallback.
 *
 * Sources of each operation (pages: the lucebox pull requests about the
 * DeepSeek-V4-Flash "DS4" server):
 *   - quant type + CPU reference conversion: "feat(ds4): add DSpark speculative
 *     runtime + optimizations" #496, summary bullet "ROCmFP4/ROCmFPX quant types
 *     + CPU reference conversions";
 *   - MMVQ vecdot / MMVQ kernel over ne1 columns, MMVQ_MAX_MOE_BATCH_SIZE: same
 *     summary ("CUDA/HIP dequant, copy, getrows, MMVQ vecdot, MMVF ...");
 *   - codebook-16 expander: "fix(ggml): make ROCmFP4 codebook self-contained on
 *     CUDA" (commit on "fix(ds4): correct layer-split HC handoff and per-device
 *     state" #507);
 *   - SwiGLU split for the fused FFN matvec paths: #496 summary, "DS4 SwiGLU
 *     split op plumbing";
 *   - routed-expert top-k and the fused expert-FFN combine: "fix(ds4): keep
 *     ROCmFPX generation byte-safe" #494 (DFLASH_DS4_FFN_FUSED_COMBINE) and
 *     "feat(ds4): add DSpark speculative decoding" (configured routed-expert
 *     top-k, fused batched verification).
 *
 * Weight format ("canonical blocks"): a matrix of M rows x K columns
 * (K % 32 == 0) is M x (K/32) blocks, row-major, 18 bytes per block:
 *   bytes 0-1  fp16 scale dw, little-endian;
 *   bytes 2-17 index bytes qs: byte j holds the codebook index of element j
 *              in its low nibble and of element j+16 in its high nibble;
 *   weight_i = dw * codebook[index_i], codebook = {-127,-104,-83,-65,-49,-35,
 *              -22,-10,1,13,25,38,53,69,89,113}.
 *
 * Activation quantization (per 32 consecutive values of one column):
 *   d = max|x| / 127 (fp32), q = round-half-to-even(x / d) clamped to
 *   [-127,127], q = 0 when d == 0.  Inputs are assumed finite.
 *
 * Conventions for every entry point:
 *   - returns CBQ_OK (0) or a negative cbq_status; argument errors are
 *     reported before anything is launched;
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream); work is enqueued on it and the call returns without waiting,
 *     except where a function says it synchronizes;
 *   - pointers named *_dev are device pointers owned by the caller; the
 *     library only reads inputs and writes outputs within the stated sizes;
 *   - a handle owns its device memory (repacked weights and a workspace) and
 *     remembers its device; calls switch to that device and restore the
 *     caller's current device before returning;
 *   - the workspace of a handle is shared by its calls: two calls on one
 *     handle that overlap on the GPU (different streams without ordering)
 *     race.  Calls on one stream are ordered and safe;
 *   - kernels are launched as programmatic dependents (programmatic stream
 *     serialization) where that hides launch latency: such a kernel may
 *     become resident before the work ahead of it on the stream has ended,
 *     but it reads an input of the call or a counter of a handle only once
 *     all work enqueued before the call has ended (the call's first kernel
 *     waits for it with griddepcontrol.wait before it lets the call's next
 *     kernel start), so results are those of plain stream order, also after
 *     a caller's kernel that signals its dependents early;
 *   - no call allocates or frees device memory except *_create, *_destroy
 *     and cbq_moe_set_shared (which allocates the shared expert's weights the
 *     first time, frees them on removal, and uses a temporary device buffer
 *     for host blocks);
 *   - errors found by a kernel while it runs (an expert id out of range, a
 *     bounded wait that gave up) set bits in an error word that belongs to
 *     the handle; cbq_weights_get_error / cbq_moe_get_error read and clear it
 *     in the order of a stream.  Outputs of a call that set a *_TIMEOUT bit
 *     are undefined.
 */
#ifndef CBQ_H
#define CBQ_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define CBQ_QK 32            /* weights per block */
#define CBQ_BLOCK_BYTES 18   /* bytes per canonical block */
#define CBQ_MAX_COLS 5       /* activation columns per matvec (decode + verify q<=4) */
#define CBQ_MAX_TOKENS 5     /* tokens per MoE call */
#define CBQ_MAX_TOPK 16      /* routed experts per token */

typedef enum {
    CBQ_OK = 0,
    CBQ_EINVAL = -1,   /* bad argument (null pointer, size, count) */
    CBQ_ECUDA = -2,    /* a CUDA runtime call or a launch failed */
    CBQ_ENOMEM = -3,   /* device allocation failed in a *_create */
    CBQ_EDEVICE = -4   /* no usable sm_103 device */
} cbq_status;

/* Bits of a handle's error word (cbq_weights_get_error, cbq_moe_get_error). */
#define CBQ_DEVERR_BAD_EXPERT_ID 0x1u          /* an id outside [0,E): that slot was skipped */
#define CBQ_DEVERR_PIPE_TIMEOUT 0x100u         /* a weight-stream wait gave up after 1 s */
#define CBQ_DEVERR_DEPENDENCY_TIMEOUT 0x200u   /* a down-projection item gave up waiting 1 s for its
                                                  expert's intermediate; its outputs were not written */

typedef struct cbq_weights cbq_weights; /* one dense M x K matrix, repacked on device */
typedef struct cbq_moe cbq_moe;         /* E experts: gate_up (2F x H) and down (H x F) */

/* Human-readable name of a cbq_status. */
const char *cbq_status_string(int status);

/* Text of the last CUDA error seen by this thread ("" if none). */
const char *cbq_last_cuda_error(void);

/* Create a dense weight handle on the current device from canonical blocks
 * `blocks` (M*(K/32)*18 bytes; host memory if on_device == 0, else device
 * memory).  The blocks are repacked into the device layout (16-byte index
 * stream interleaved by 32-row groups plus a separate fp16 scale stream); the
 * source is not retained.  Synchronizes `stream`.
 * K is bounded by the shared-memory staging of CBQ_MAX_COLS quantized
 * activation columns next to a four-stage weight ring and the partial-sum
 * set: K <= 27,136 on GB300 (227 KB of shared memory per CTA).
 * Errors: EINVAL (null, M < 1, K < 32, K % 32 != 0, K above that bound),
 * ENOMEM, ECUDA, EDEVICE. */
int cbq_weights_create(const void *blocks, int64_t M, int64_t K, int on_device,
                       void *stream, cbq_weights **out);
int cbq_weights_destroy(cbq_weights *W);

/* Shape of a handle and the device bytes it holds (any pointer may be NULL). */
int cbq_weights_info(const cbq_weights *W, int64_t *M, int64_t *K, int64_t *device_bytes);

/* Activation quantization (pages: activation side of the MMVQ vecdot).
 * x_dev: n x K fp32, row-major (column c at x_dev + c*K); K % 32 == 0; n >= 1.
 * qx_dev: n x K int8 out; dx_dev: n x (K/32) fp32 out.
 * Bit-exact with the rule in the header comment. */
int cbq_quantize_act(const float *x_dev, int64_t K, int n, int8_t *qx_dev, float *dx_dev,
                     void *stream);

/* Quantized matvec from already-quantized activations (MMVQ with ne1 = n).
 * qx_dev: n x K int8, dx_dev: n x (K/32) fp32 (layout of cbq_quantize_act);
 * y_dev: n x M fp32 out, y[c][r] = sum_b dw(r,b) * dx[c][b] * s(r,b,c) where
 * s is the exact int32 block dot.  1 <= n <= CBQ_MAX_COLS.  All n columns are
 * computed in one pass over the weights. */
int cbq_matvec_q(const cbq_weights *W, const int8_t *qx_dev, const float *dx_dev, int n,
                 float *y_dev, void *stream);

/* The whole dense path: quantize x_dev (n x K fp32) with the rule of
 * cbq_quantize_act, then the matvec of cbq_matvec_q into y_dev (n x M fp32);
 * the result has the same bits as those two calls.  For n == 1 with x_dev
 * 16-byte aligned this is one kernel launch (the matvec kernel quantizes x
 * while its weight stream starts); otherwise the quantization kernel writes
 * the handle's workspace first and the matvec kernel follows it as a
 * programmatic dependent.  One call at a time per handle. */
int cbq_matvec(const cbq_weights *W, const float *x_dev, int n, float *y_dev, void *stream);

/* Same with HOST buffers: copies x (n x K fp32) to the device, runs
 * cbq_matvec and copies y (n x M fp32) back, then synchronizes `stream`.
 * Pinned host memory makes the copies asynchronous to the host. */
int cbq_matvec_host(const cbq_weights *W, const float *x_host, int n, float *y_host,
                    void *stream);

/* Create an MoE layer handle from canonical blocks of E experts, contiguous
 * per expert: gate_up = E x (2F rows x H cols), rows 0..F-1 the gate
 * projection and rows F..2F-1 the up projection; down = E x (H rows x F cols).
 * H % 32 == 0, F % 32 == 0, E >= 1, H and F <= 1,048,576.  Host memory if
 * on_device == 0.
 * Synchronizes `stream`.  Errors as cbq_weights_create. */
int cbq_moe_create(const void *gate_up, const void *down, int E, int64_t H, int64_t F,
                   int on_device, void *stream, cbq_moe **out);
int cbq_moe_destroy(cbq_moe *L);

/* Give the layer a shared expert: one more gate_up (2F x H) and down (H x F)
 * pair in canonical blocks, the same shapes as a routed expert, that every
 * token passes through with weight 1 in each later cbq_moe_matvec* call:
 *   y_t = sum_j wts[t][j] * o_{ids[t][j]}(h_t) + o_sh(h_t),
 * o_sh computed exactly as a routed slot (SwiGLU split, requantization, down)
 * and added after the routed sum.  The pages name only the routed layer
 * ("feat(ds4): add DSpark speculative decoding" routes each token to its
 * configured top-k); the always-on expert of the DS4 FFN block is read here
 * as one more expert of the same shape.  Its weights are read once per call,
 * in the same layer kernel, like any routed expert.  Host memory if
 * on_device == 0; the blocks are repacked and not retained.  gate_up == down
 * == NULL removes the shared expert.  Synchronizes `stream` first (a call
 * still running on another stream must have ended).
 * Errors: EINVAL (exactly one of gate_up, down NULL), ENOMEM, ECUDA. */
int cbq_moe_set_shared(cbq_moe *L, const void *gate_up, const void *down, int on_device, void *stream);

int cbq_moe_info(const cbq_moe *L, int *E, int64_t *H, int64_t *F, int64_t *device_bytes);

/* Routed-expert FFN (mul_mat_id with the SwiGLU split and the weighted
 * combine fused).  h_dev: n_tok x H fp32; ids_dev: n_tok x topk int32 expert
 * ids; wts_dev: n_tok x topk fp32 router weights; y_dev: n_tok x H fp32 out.
 * For every token t and slot j (slot order), expert e = ids[t][j]:
 *   g,u = gate/up rows of e applied to quantize(h_t);
 *   a = swiglu ? silu(g)*u : g*u (fp32), silu(z) = z/(1+exp(-z));
 *   o = down_e applied to quantize(a);  y_t = sum_j wts[t][j] * o.
 * Tokens are grouped by expert on the device: each distinct expert's bytes
 * are read once per call for all of its tokens.  Ids should be distinct per
 * token; a repeated id is served as an extra column and summed on its own.
 * An id outside [0,E) skips its slot and sets CBQ_DEVERR_BAD_EXPERT_ID.
 * The sum over j runs in slot order (deterministic, no atomics on y).
 * With a shared expert (cbq_moe_set_shared) its output is added last.
 * Three kernel launches on `stream`, each a programmatic dependent of the one
 * before: the token quantization, the layer kernel (gate_up, SwiGLU,
 * requantization, down), the combine.  With one token the layer kernel forms
 * the combine itself (same order, same bits), and with h_dev also 16-byte
 * aligned it quantizes the token itself too (same bits): one launch.  One
 * call at a time per handle (its workspace and counters are shared by the
 * calls).
 * 1 <= n_tok <= CBQ_MAX_TOKENS, 1 <= topk <= min(CBQ_MAX_TOPK, E). */
int cbq_moe_matvec(const cbq_moe *L, const float *h_dev, int n_tok, const int32_t *ids_dev,
                   const float *wts_dev, int topk, int swiglu, float *y_dev, void *stream);

/* Largest expert count of the router entry points (its logits are staged in
 * shared memory). */
#define CBQ_ROUTER_MAX_E 16384

/* Routed-expert selection from router logits: logits_dev n_tok x E fp32;
 * for every token t, ids_dev[t][0..topk) = the indices of the topk largest
 * logits in descending order (equal logits: lower index first) and
 * wts_dev[t][j] = softmax over those topk logits, computed in fp64 and
 * rounded to fp32.  The pages name a "configured routed-expert top-k"
 * ("feat(ds4): add DSpark speculative decoding") without a formula; this is
 * the plain reading.  Logits must be finite.  1 <= n_tok <= 65535,
 * 1 <= E <= CBQ_ROUTER_MAX_E, 1 <= topk <= min(CBQ_MAX_TOPK, E).  One kernel
 * launch on `stream`; the caller owns every buffer. */
int cbq_router_topk(const float *logits_dev, int n_tok, int E, int topk, int32_t *ids_dev, float *wts_dev,
                    void *stream);

/* The weight converter: a row-major M x K fp32 matrix on the device to the
 * M x (K/32) canonical 18-byte blocks that cbq_weights_create and
 * cbq_moe_create read (on_device = 1).  The pages name "CPU reference
 * conversions" of the quant types ("feat(ds4): add DSpark speculative
 * runtime + optimizations" #496) without a rule; this is the plain reading,
 * per block of 32 weights:
 *   m = the weight of largest magnitude (the first among equal ones);
 *   scale = binary16(m / -127): IEEE fp32 division, then rounding to nearest
 *           even (-127 is the codebook level of largest magnitude, so m lands
 *           on it); an all-zero block gives 18 zero bytes;
 *   index_i = the level j whose reconstruction scale * codebook[j] is nearest
 *           to w_i, the lowest j among equal distances (index 0 everywhere
 *           when the scale rounds to zero).
 * The decisions are exact (no rounding can move a weight to another level),
 * so the bytes are the same on every run.  Weights must be finite with
 * |m| < 127 * 65520 (a finite scale).  w_dev 16-byte aligned, blocks_dev
 * 2-byte aligned, both owned by the caller; M >= 1, K >= 32, K % 32 == 0,
 * else CBQ_EINVAL.  One kernel launch on `stream`. */
int cbq_quantize_weights(const float *w_dev, int64_t M, int64_t K, void *blocks_dev, void *stream);

/* Streams of the hyper-connection state (the NHC of the pages' NHC = 4
 * specialisation), and the most normalisation rounds one call accepts. */
#define CBQ_HC_NHC 4
#define CBQ_HC_MAX_ITERS 1024
#define CBQ_HC_MAX_N (1ll << 28)

/* Sinkhorn normalisation of the hyper-connection mixing matrices (the
 * register-resident sinkhorn kernel of the fused DS4 hyper-connection op,
 * "feat(ds4): add DSpark speculative runtime + optimizations" #496, in its
 * NHC = 4 form, "fix(ds4): keep ROCmFPX generation byte-safe" #494).  The
 * pages give neither the iteration count nor the update; the plain reading
 * of a Sinkhorn normalisation is used.  For each of the n row-major
 * CBQ_HC_NHC x CBQ_HC_NHC matrices c of fp32 logits at logits_dev:
 *   P = exp(c - max c);
 *   `iters` rounds of: every row of P scaled to sum 1, then every column
 *   (a sum in index order, times its reciprocal from the hardware
 *   approximation, within 1 ulp);
 *   out_dev = P after the last round (columns sum to 1 within rounding; rows
 *   approach 1 as the rounds converge); iters = 0 gives exp(c - max c).
 * The result agrees with an fp64 evaluation of the same rounds within
 * (8 + 16 * iters) * 2^-24 per entry.  In contract: finite logits whose
 * spread within a matrix (max - min) is at most 80, so every entry stays a
 * normal fp32 number.  Arguments: both pointers 16-byte aligned (out_dev may
 * equal logits_dev: each matrix is read before it is written; otherwise the
 * buffers must not overlap); 1 <= n <= CBQ_HC_MAX_N; 0 <= iters <=
 * CBQ_HC_MAX_ITERS; else CBQ_EINVAL.  One kernel launch on `stream` (a
 * programmatic dependent of the work ahead, like every kernel here), one
 * thread per matrix; the caller owns both buffers. */
int cbq_hc_sinkhorn(const float *logits_dev, int64_t n, int iters, float *out_dev, void *stream);

/* cbq_router_topk into the handle's staging buffers, then cbq_moe_matvec with
 * those ids and weights: the routed layer from router logits with no host
 * round trip (one launch more than cbq_moe_matvec).  Same limits as both. */
int cbq_moe_matvec_logits(const cbq_moe *L, const float *h_dev, int n_tok, const float *logits_dev, int topk,
                          int swiglu, float *y_dev, void *stream);

/* Same with HOST buffers (h, ids, wts in; y out), then synchronizes `stream`. */
int cbq_moe_matvec_host(const cbq_moe *L, const float *h_host, int n_tok,
                        const int32_t *ids_host, const float *wts_host, int topk, int swiglu,
                        float *y_host, void *stream);

/* Stage timing: when set, cbq_moe_matvec records these CUDA events
 * (cudaEvent_t passed as void*) on its stream before its first kernel,
 * before the layer kernel (right after ev_start when the layer kernel
 * quantizes the one token itself; else after the token quantization) and
 * after the call's last kernel (the layer kernel, or the combine).  Recording them separates the kernels (the overlap
 * of a kernel's start with the previous one's end is lost).  Pass NULL for
 * all three to stop; a mix of NULL and non-NULL is CBQ_EINVAL.  The events
 * stay owned by the caller. */
int cbq_moe_set_stage_events(cbq_moe *L, void *ev_start, void *ev_layer, void *ev_end);

/* ---- tensor-core path for larger batches ------------------------------ */

/* Most columns of cbq_matmat. */
#define CBQ_MAX_MMQ_COLS 16

/* The dense product for 1 <= n <= CBQ_MAX_MMQ_COLS columns on the tensor
 * cores (tcgen05): the MMQ tile the pages name for larger batches ("#497
 * RDNA MMQ tile, LUCE_MMQ_DP_MAX_NE1", "fix(ds4): correct layer-split HC
 * handoff and per-device state" #507), read for this format.  Same result
 * definition as cbq_matvec (the activation quantization, exact per-block
 * integer dots, y = sum_b dw*dx*s in fp32 with the same three roundings per
 * block); the blocks, in units of four, alternate between two running sums
 * added at the end of the row: every block dot is exact, so y is within the
 * same bound of the plain definition.  A level enters the MMA as
 * the fp16 value 1152 + level, an int8 activation as fp16; each 32-wide block
 * sum is an integer below 2^24 (exact in the fp32 accumulator), and the bias
 * 1152 * sum q is subtracted exactly.  Arguments as cbq_matvec (x_dev n x K
 * fp32, y_dev n x M fp32, both owned by the caller).  Three launches on
 * `stream`: the quantization, the B tiles, the tiles of W.  One call at a
 * time per handle (its workspace is shared by the calls). */
int cbq_matmat(const cbq_weights *W, const float *x_dev, int n, float *y_dev, void *stream);

/* Checking: the exact block dots s[c][r][b] (n x M x K/32 int32) of W's
 * blocks with the int8 columns qx_dev (n x K), taken by the tensor-core path
 * (cbq_debug_block_dots takes them by the dp4a path).  1 <= n <=
 * CBQ_MAX_MMQ_COLS. */
int cbq_debug_mmq_block_dots(const cbq_weights *W, const int8_t *qx_dev, int n, int32_t *s_dev, void *stream);

/* ---- allocation-free dense path --------------------------------------- */

/* Largest K cbq_matvec_static accepts (its scratch holds CBQ_MAX_COLS columns
 * of this many quantized values plus their scales: 92,160 bytes per device). */
#define CBQ_STATIC_SCRATCH_MAX_K 16384

/* cbq_matvec for callers that must not allocate device memory while they run,
 * e.g. hosts that fix their device memory budget at start-up and forbid
 * allocation afterwards.  The pages describe no counterpart; it is the dense
 * path of cbq_matvec with one difference: with more than one column, or x_dev
 * not 16-byte aligned, the quantized activations go to a scratch array the
 * library declares statically on every device (it lives as long as the
 * library is loaded), not to the handle's workspace; one aligned column is
 * quantized inside the matvec kernel (one launch), as cbq_matvec does, and
 * needs no scratch.  Nothing is allocated or freed, here or in any library
 * routine it calls.  Same bits as cbq_matvec.
 *   - Arguments as cbq_matvec; K of W must be <= CBQ_STATIC_SCRATCH_MAX_K,
 *     else CBQ_EINVAL (checked before anything runs).
 *   - The first call on a device looks the scratch array up on that device
 *     (cudaGetSymbolAddress).
 *   - The scratch is one array per device shared by every call of this entry
 *     point on that device, whatever the handle: calls that may overlap on the
 *     GPU (different streams without ordering) race.  Every call rewrites the
 *     part it reads, so no contents carry over from the previous call. */
int cbq_matvec_static(const cbq_weights *W, const float *x_dev, int n, float *y_dev, void *stream);

/* Read the error word of a handle (bits CBQ_DEVERR_*: every error of the
 * handle's calls since the last read) into *code and clear it.  The copy and
 * the clear are enqueued on `stream`, which is then synchronized (no other
 * stream or device-wide synchronization): calls enqueued on `stream` before
 * this one are covered, and a call on another stream is covered once it is
 * ordered before `stream` (an event, or a synchronization).  Errors: EINVAL
 * (null), ECUDA. */
int cbq_weights_get_error(const cbq_weights *W, void *stream, unsigned int *code);
int cbq_moe_get_error(const cbq_moe *L, void *stream, unsigned int *code);

/* ---- checking entry points (used by the parity tests) ---------------- */

/* Per-block int32 dots s_dev[c][r][b] (n x M x K/32) of W with plain int8
 * activations qx_dev (n x K), through the same codebook expander and dp4a
 * sequence as the matvec kernels.  1 <= n <= CBQ_MAX_COLS. */
int cbq_debug_block_dots(const cbq_weights *W, const int8_t *qx_dev, int n, int32_t *s_dev,
                         void *stream);

/* Same for expert e of an MoE layer: which = 0 gate_up, 1 down; e == E
 * names the shared expert (CBQ_EINVAL when there is none). */
int cbq_moe_debug_block_dots(const cbq_moe *L, int e, int which, const int8_t *qx_dev, int n,
                             int32_t *s_dev, void *stream);

/* Keep (1) or stop keeping (0) the intermediate of each slot -- a (fp32) and
 * its quantization (qa int8, da fp32) in plain slot order -- in the workspace
 * during cbq_moe_matvec (costs about 5*F bytes of writes per slot). */
int cbq_moe_set_debug(cbq_moe *L, int keep_intermediate);

/* Give-up test mode of the layer kernel, for the tests of its bounded waits
 * (0 turns it off): mode 1 makes every down-projection item wait for an
 * intermediate count that is never reached, so that wait gives up after its
 * 1 s limit (CBQ_DEVERR_DEPENDENCY_TIMEOUT, or CBQ_DEVERR_PIPE_TIMEOUT when
 * the consumers' own 1 s wait for that stage runs out first) and the CTA
 * stops; mode 2 makes the first CTA's first weight stage never arrive, so its
 * consumers' wait gives up (CBQ_DEVERR_PIPE_TIMEOUT; the down items that
 * need that CTA's gate_up results then give up too).  Either way the CTA
 * issues no copy after giving up and waits (bounded) for those in flight, so
 * none is left running when it exits.  A call in either mode returns after a
 * few seconds with undefined outputs, sets only timeout bits, and leaves the
 * handle usable: the next call is correct. */
int cbq_moe_debug_stall(cbq_moe *L, int mode);

/* Give-up test mode of the tensor-core path (cbq_matmat and its block-dot
 * checking entry; 0 turns it off): with mode 1 the first CTA's producer
 * issues no copy, so the bounded waits of every role of that CTA for its
 * first stage give up after 1 s (CBQ_DEVERR_PIPE_TIMEOUT in the handle's
 * error word); the CTA issues no MMA after giving up, waits (bounded) for
 * those it issued and frees its tensor memory before it exits.  A call in
 * this mode returns after about a second with undefined outputs, sets only
 * that bit, and leaves the handle usable: the next call is correct.
 * Errors: EINVAL (null handle, mode outside 0..1). */
int cbq_debug_mmq_stall(cbq_weights *W, int mode);

/* Copy the intermediate of the last cbq_moe_matvec on this handle, for
 * slots p < nslots (at most CBQ_MAX_TOKENS * (CBQ_MAX_TOPK + 1)): routed
 * slots p = t*topk + j, then the shared expert's slots p = n_tok*topk + t;
 * a_dev[p][F] fp32, qa_dev[p][F] int8, da_dev[p][F/32] fp32 (any may be
 * NULL), as kept by the last call made with debug on (cbq_moe_set_debug).
 * Slots whose id was out of range hold stale data. */
int cbq_moe_debug_intermediate(const cbq_moe *L, int nslots, float *a_dev, int8_t *qa_dev,
                               float *da_dev, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* CBQ_H */

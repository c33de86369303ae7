// cbq_internal.h -- launchers shared by the C-ABI layer (cbq_api.cu) and the
// kernel translation unit (cbq_kernels.cu).  Not part of the public ABI.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace cbq {

// One repacked matrix on the device (layout described in cbq_device.cuh).
struct DevMat {
    const uint4 *qs;  // G * nbp * 32 index fields
    const uint2 *sc;  // G * nbq * 32 words of four fp16 scales
    int64_t M;        // rows
    int nb;           // K / 32
    int nbp;          // nb rounded up to a multiple of 4
    int G;            // ceil(M / 32) row groups
    unsigned *sched;  // 2 work counters of the matvec kernel (zero between launches)
    unsigned *err;    // the handle's error word (CBQ_DEVERR_* bits)
};

inline int round_up4(int v) { return (v + 3) & ~3; }

// Index/scale element counts of a repacked M x K matrix.
inline size_t qs_elems(int64_t M, int nb) { return (size_t)((M + 31) / 32) * (size_t)round_up4(nb) * 32; }
inline size_t sc_elems(int64_t M, int nb) { return (size_t)((M + 31) / 32) * (size_t)(round_up4(nb) / 4) * 32; }

// A routed-expert layer: E stacked gate_up (2F x H) and down (H x F) matrices.
struct DevMoe {
    const uint4 *gu_qs;
    const uint2 *gu_sc;
    const uint4 *dn_qs;
    const uint2 *dn_sc;
    int E, H, F;
    size_t gu_qs_stride, gu_sc_stride, dn_qs_stride, dn_sc_stride;  // per expert
    // Optional shared expert (same shapes), applied to every token with
    // weight 1; the kernels address it as expert id E.  Null when absent.
    const uint4 *sh_gu_qs;
    const uint2 *sh_gu_sc;
    const uint4 *sh_dn_qs;
    const uint2 *sh_dn_sc;
    int shared;
};

// Per-call scratch of an MoE layer handle (device memory it owns).
struct MoeWork {
    int8_t *qh;       // CBQ_MAX_TOKENS x H
    float *dh;        // CBQ_MAX_TOKENS x H/32
    int8_t *qa;       // slots x F
    float *da;        // slots x F/32
    float *a_dbg;     // slots x F (written when keep_a)
    float *obuf;      // slots x H, down-projection output per slot
    unsigned *sched;  // 4 work counters (items, producers done, CTAs done), zero between launches
    unsigned *done;   // per expert rank: gate_up columns published (zero between launches)
    unsigned *err;    // the handle's error word (CBQ_DEVERR_* bits)
    int keep_a;
    int stall;        // give-up test mode: 0 off, 1 a dependency never met, 2 a stage never filled
    cudaEvent_t ev[3];  // optional stage events (before the layer kernel, before the combine, after it)
};

constexpr int kMaxSlots = 85;  // CBQ_MAX_TOKENS * (CBQ_MAX_TOPK routed + 1 shared)

cudaError_t launch_repack(const uint8_t *src, int64_t M, int nb, uint4 *qs, uint2 *sc, cudaStream_t s);
cudaError_t launch_quantize(const float *x, int64_t K, int n, int8_t *qx, float *dx, cudaStream_t s);
// pdl: launch as a programmatic dependent of the previous kernel on the
// stream (only when that kernel is this library's own quantization).
cudaError_t launch_matvec(const DevMat &W, const int8_t *qx, const float *dx, int n, float *y,
                          cudaStream_t s, bool pdl = false);
// The matvec from one fp32 column x (K values, 16-byte aligned), quantized
// inside the kernel (one launch).
cudaError_t launch_matvec_f32(const DevMat &W, const float *x, int n, float *y, cudaStream_t s);
cudaError_t launch_block_dots(const DevMat &W, const int8_t *qx, int n, int32_t *sdot, cudaStream_t s);
cudaError_t launch_moe(const DevMoe &L, const MoeWork &ws, const float *h, int n_tok, const int32_t *ids,
                       const float *wts, int k, int swiglu, float *y, cudaStream_t s);
// Largest dynamic shared memory a matvec over K columns with n columns needs.
size_t matvec_smem_bytes(int nbp, int n);
size_t moe_smem_bytes(int act_blocks, int stages);
cudaError_t device_smem_limit(size_t *bytes);
// Top-k expert ids and softmax weights per token from router logits (n_tok x E).
cudaError_t launch_router_topk(const float *logits, int n_tok, int E, int k, int32_t *ids, float *wts,
                               cudaStream_t s);
// Dynamic shared memory the layer kernel may use (opt-in limit less its static part).
cudaError_t moe_smem_limit(size_t *bytes);

}  // namespace cbq

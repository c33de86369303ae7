// cbq_internal.h -- the device layout of the weights and the launchers shared
// by the C-ABI layer (cbq_api.cu) and the kernel translation unit
// (cbq_kernels.cu).  Not part of the public ABI.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace cbq {

// ---------------------------------------------------------------------------
// Device layout of one matrix (written once by the repack kernel from the
// canonical 18-byte blocks).  Rows are taken in groups of 32 and the groups
// in pairs; nbp = K/32 rounded up to a multiple of 4.  A pair's K range is cut
// into chunks of 16 block columns (the last one shorter when nbp is not a
// multiple of 16), and chunk c (nblk blocks) of pair p is one contiguous span
// of 1152 * nblk bytes:
//   for each of the pair's two groups (half h = 0, 1), 576 * nblk bytes:
//     the index fields: block j, lane l (row 32g + l) at (j*32 + l) * 16;
//     then the fp16 scales: four consecutive blocks of a row per 8-byte word,
//       quad q, lane l at 512 * nblk + (q*32 + l) * 8.
// So the weight stream of a pass over one pair -- the gate and up rows of one
// SwiGLU group, or two consecutive down or dense groups -- arrives with one
// bulk copy per 16 block columns.  A pair holds 1152 * nbp bytes; padded rows
// and blocks carry zero indices and zero scales.  The gate_up matrix of a
// routed expert pairs gate group g with up group Gf + g (Gf = F/32), every
// other matrix pairs groups 2p and 2p + 1.
constexpr int kChunk = 16;          // block columns per chunk (one pipeline stage)
constexpr int kBlockBytes = 576;    // bytes of one block column of one 32-row group (512 + 64)
constexpr int kChunkBytes = 2 * kChunk * kBlockBytes;  // 18,432: a full chunk of a pair

inline int round_up4(int v) { return (v + 3) & ~3; }

__host__ __device__ inline int chunk_blocks(int nbp, int c) {
    return nbp - kChunk * c < kChunk ? nbp - kChunk * c : kChunk;
}
__host__ __device__ inline size_t pair_bytes(int nbp) { return (size_t)nbp * 2 * kBlockBytes; }

// Byte offsets, from the start of a pair, of the index field of (half h,
// block b, lane) and of the fp16 scale of (half h, block b, lane).
__host__ __device__ inline size_t field_offset(int nbp, int h, int b, int lane) {
    const int c = b / kChunk, j = b - c * kChunk, nblk = chunk_blocks(nbp, c);
    return (size_t)c * kChunkBytes + (size_t)h * nblk * kBlockBytes + ((size_t)j * 32 + lane) * 16;
}
__host__ __device__ inline size_t scale_offset(int nbp, int h, int b, int lane) {
    const int c = b / kChunk, j = b - c * kChunk, nblk = chunk_blocks(nbp, c);
    return (size_t)c * kChunkBytes + (size_t)h * nblk * kBlockBytes + (size_t)nblk * 512 +
           ((((size_t)(j >> 2) * 32 + lane) * 4) + (j & 3)) * 2;
}

// Pairs and device bytes of a repacked M x K matrix (nb = K/32).
inline int64_t mat_pairs(int64_t M) { return (M + 63) / 64; }
inline size_t mat_bytes(int64_t M, int nb) { return (size_t)mat_pairs(M) * pair_bytes(round_up4(nb)); }

// One repacked dense matrix on the device.
struct DevMat {
    const uint8_t *w;  // P pairs of pair_bytes(nbp)
    int64_t M;         // rows
    int nb;            // K / 32
    int nbp;           // nb rounded up to a multiple of 4
    int G;             // ceil(M / 32) row groups
    int P;             // ceil(M / 64) pairs
    int split;         // 0: pairs of consecutive groups; Gf > 0: group g < Gf pairs with g + Gf (gate_up)
    unsigned *sched;   // 2 work counters of the matvec kernel (zero between launches)
    unsigned *err;     // the handle's error word (CBQ_DEVERR_* bits)
};

// A routed-expert layer: E gate_up (2F x H, gate/up pairs) and down (H x F)
// matrices, one after another.
struct DevMoe {
    const uint8_t *gu;
    const uint8_t *dn;
    int E, H, F;
    size_t gu_stride, dn_stride;  // bytes per expert
    // Optional shared expert (same shapes), applied to every token with
    // weight 1; the kernels address it as expert id E.  Null when absent.
    const uint8_t *sh_gu;
    const uint8_t *sh_dn;
    int shared;
};

// Per-call scratch of an MoE layer handle (device memory it owns).
struct MoeWork {
    int8_t *qh;       // the tokens quantized, in the chunked activation layout (act_bytes)
    int8_t *qa_bm;    // per virtual expert: its quantized intermediate, the same layout (kMaxCols columns' room)
    unsigned *dep;    // two sets (by call parity) of: per virtual expert and down stage, gate_up groups published
    size_t dep_set;   // words of one dep set (kMaxSlots x down stages)
    unsigned *pcnt;   // two sets of: per 64-row output group, virtual experts whose down item finished
    int8_t *qa;       // slots x F, plain order (written when keep_a)
    float *da;        // slots x F/32 (written when keep_a)
    float *a_dbg;     // slots x F (written when keep_a)
    float *obuf;      // slots x H, down-projection output per slot
    unsigned *sched;  // items taken, CTAs done taking, call count, dep words used per set (5 words)
    unsigned *err;    // the handle's error word (CBQ_DEVERR_* bits)
    int keep_a;
    int stall;        // give-up test mode: 0 off, 1 a dependency never met, 2 a stage never filled
    cudaEvent_t ev[3];  // optional events: before the call, before the layer kernel, after it
};

// The chunked activation layout the layer kernel's stages copy: `cols`
// columns over nbp blocks, in chunks of kChunk blocks; chunk c (nblk blocks)
// starts at c * 36 * cols * kChunk bytes and holds block j of column x at
// (j*cols + x) * 32 (32 bytes in the expander order), then the scales, the
// block pair j/2 of column x as two floats at 32 * cols * nblk + ((j/2)*cols
// + x) * 8.  A chunk is one contiguous 36 * cols * nblk bytes.
__host__ __device__ inline size_t act_bytes(int nbp, int cols) { return (size_t)nbp * cols * 36; }
__host__ __device__ inline size_t act_chunk_offset(int c, int cols) { return (size_t)c * 36 * cols * kChunk; }

constexpr int kMaxSlots = 85;  // CBQ_MAX_TOKENS * (CBQ_MAX_TOPK routed + 1 shared)

cudaError_t launch_repack(const uint8_t *src, int64_t M, int nb, int split, uint8_t *w, cudaStream_t s);
cudaError_t launch_quantize(const float *x, int64_t K, int n, int8_t *qx, float *dx, cudaStream_t s);
// The layer's n tokens (K values each) quantized into the chunked activation layout.
cudaError_t launch_quantize_chunked(const float *x, int K, int n, int8_t *qh, cudaStream_t s);
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
cudaError_t device_smem_limit(size_t *bytes);
cudaError_t matvec_smem_limit(size_t *bytes);
// Bytes of one block of the canonical format (2-byte fp16 scale, 16 index bytes).
constexpr int kBlockBytesCanonical = 18;
// fp32 weights (16-byte aligned) to nblocks canonical blocks at out (2-byte aligned).
cudaError_t launch_quantize_weights(const float *w, int64_t nblocks, uint8_t *out, cudaStream_t s);
// The tensor-core (tcgen05) path for up to kMaxMmqCols columns: the B tiles
// and block metadata from quantized columns (qx[c][K], dx[c][K/32]; dx null
// gives zero scales), then the tiles of W; dbg, when not null, receives the
// exact block dots s[c][row][b].  stall = 1 (give-up test mode): CTA 0
// copies nothing, so its bounded waits run out.
constexpr int kMaxMmqCols = 16;
size_t mmq_bimg_bytes(int nb);
size_t mmq_meta_bytes(int nb);
cudaError_t launch_mmq_prep(const int8_t *qx, const float *dx, int n, int64_t K, uint8_t *bimg, float *meta,
                            cudaStream_t s);
cudaError_t launch_mmq(const DevMat &W, const uint8_t *bimg, const float *meta, int n, float *y, int32_t *dbg,
                       int stall, cudaStream_t s);
// Top-k expert ids and softmax weights per token from router logits (n_tok x E).
cudaError_t launch_router_topk(const float *logits, int n_tok, int E, int k, int32_t *ids, float *wts,
                               cudaStream_t s);
// Sinkhorn normalisation of n row-major kHcNhc x kHcNhc matrices of logits
// (16-byte aligned; out may equal logits).
constexpr int kHcNhc = 4;
cudaError_t launch_hc_sinkhorn(const float *logits, int64_t n, int iters, float *out, cudaStream_t s);

}  // namespace cbq

// cbq_mmq.cu -- the quantized mat-mat path for up to 16 activation columns
// on the 5th-generation tensor cores (tcgen05): the MMQ tile the pages name
// for larger batches ("#497 RDNA MMQ tile, LUCE_MMQ_DP_MAX_NE1" in "fix(ds4):
// correct layer-split HC handoff and per-device state" #507; the prefill cost
// of the q+1 verify in "fix(ds4): keep ROCmFPX generation byte-safe" #494),
// read for this format as: the same y = sum_b dw*dx*s as the dp4a path, with
// every per-block integer dot s taken by the tensor cores.
//
// Exactness.  A codebook level L (-127..113) enters the MMA as the fp16 value
// 1152 + L = 1024 + (L + 128), whose bits are 0x6400 | (L + 128): a byte
// permute of the expanded (biased) level bytes with the byte 0x64.  An int8
// activation q enters as fp16(q), exact.  Every product (1152+L)*q and every
// partial sum over one 32-wide block (at most 32 * 1265 * 127 < 2^23) is an
// integer below 2^24, so the fp32 accumulator holds the exact block sum; s =
// sum - 1152 * sum_k q_k (the second term per column and block, exact in
// fp32) is the exact integer dot.  The scaling then repeats the dp4a path's
// roundings: acc = fma(dw*dx, s, acc), blocks in ascending order.
//
// Tile.  One MMA is M = 128 weight rows (two pairs of 32-row groups of the
// repacked layout) x N = 16 columns x K = 16; a block of 32 weights is two
// MMAs accumulating into 16 columns of tensor memory.  Operands sit in shared
// memory in the no-swizzle K-major layout: core matrices of 8 rows x 16 bytes
// (8 fp16 along K), a block's 128 x 32 A tile as core (row/8, k/8) at
// ((row/8)*4 + k/8) * 128 bytes, the 16 x 32 B tile alike; the descriptors
// step 128 bytes along K (leading byte offset) and 512 bytes along M or N
// (stride byte offset).
#include <stdint.h>

#include <algorithm>

#include <cuda_fp16.h>

#include "cbq_internal.h"
#include "cbq_pipe.cuh"

namespace cbq {

constexpr int kMmqN = 16;                    // MMA N: activation columns (zero-padded)
constexpr int kMmqM = 128;                   // MMA M: weight rows of a tile
constexpr int kMmqChunk = 4;                 // blocks per batch of MMAs
constexpr int kMmqATile = kMmqM * 32 * 2;    // 8 KB: the fp16 A tile of one block
constexpr int kMmqBTile = kMmqN * 32 * 2;    // 1 KB: the fp16 B tile of one block
constexpr int kMmqMetaFloats = 2 * kMmqN;    // per block: dx[16], then 1152 * sum q [16]
constexpr float kMmqBias = 1152.0f;
constexpr uint32_t kMmqTmemCols = 2 * kMmqChunk * kMmqN;  // 128: D of two chunks
constexpr int kMmqThreads = 128;

// Byte offset of element (row, k) in a tile of the core-matrix layout.
__host__ __device__ inline uint32_t mmq_core_off(int row, int k) {
    return (uint32_t)(((row >> 3) * 4 + (k >> 3)) * 128 + (row & 7) * 16 + (k & 7) * 2);
}

// Dynamic shared memory of k_mmq: A and B tiles of two chunks, block
// metadata of three.
constexpr size_t kMmqSmem = 2 * kMmqChunk * (kMmqATile + kMmqBTile) + 3 * kMmqChunk * kMmqMetaFloats * 4;

// --------------------------------------------------------------- tcgen05 --

// Shared-memory matrix descriptor: start address, leading (K) and stride (M
// or N) byte offsets, all in 16-byte units; version 1; no swizzle.
__device__ __forceinline__ uint64_t mmq_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46);
}

// Instruction descriptor of kind::f16: fp32 accumulator (bits 4-5 = 1), fp16
// A and B (bits 7-9, 10-12 = 0), both K-major (bits 15, 16 = 0), N >> 3 at
// bit 17, M >> 4 at bit 24.
constexpr uint32_t kMmqIdesc = (1u << 4) | ((uint32_t)(kMmqN >> 3) << 17) | ((uint32_t)(kMmqM >> 4) << 24);

__device__ __forceinline__ void tmem_alloc(uint32_t slot_saddr, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot_saddr), "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void mmq_mma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, int accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(kMmqIdesc), "r"(accumulate)
        : "memory");
}

// Arrive on the mbarrier once every MMA this thread issued so far is done.
__device__ __forceinline__ void mmq_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

// 16 consecutive fp32 columns of this thread's tensor-memory lane.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// -------------------------------------------------------- activations ---

// The B side of the MMQ path from quantized columns qx[c][K], dx[c][K/32]
// (c < n <= 16): per block b, the fp16 B tile (16 columns x 32, columns n..15
// zero) at bimg + b * 1 KB, and meta[b][0..16) = dx, meta[b][16..32) =
// 1152 * sum_k q (exact).  One CTA of 512 threads per block: thread (c, k).
// dx == nullptr gives zero scales (block-dot checking).
__global__ void __launch_bounds__(512) k_mmq_prep(const int8_t *__restrict__ qx, const float *__restrict__ dx,
                                                  int n, int64_t K, int nb, uint8_t *__restrict__ bimg,
                                                  float *__restrict__ meta) {
    pdl_wait();
    pdl_trigger();
    const int c = threadIdx.x >> 5, k = threadIdx.x & 31;
    for (int b = blockIdx.x; b < nb; b += gridDim.x) {
        const int q = c < n ? (int)qx[(size_t)c * K + (size_t)b * 32 + k] : 0;
        *reinterpret_cast<__half *>(bimg + (size_t)b * kMmqBTile + mmq_core_off(c, k)) = __int2half_rn(q);
        int sum = q;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
        if (k == 0) {
            meta[(size_t)b * kMmqMetaFloats + c] = c < n && dx ? dx[(size_t)c * nb + b] : 0.0f;
            meta[(size_t)b * kMmqMetaFloats + kMmqN + c] = kMmqBias * (float)sum;
        }
    }
}

// ------------------------------------------------------------ the tiles ---

struct MmqArgs {
    DevMat W;
    const uint8_t *bimg;  // B tiles, one per block (k_mmq_prep)
    const float *meta;    // per block: dx[16], 1152 * sum q [16]
    int n;                // columns (1..16)
    float *y;             // n x M (null: no outputs, block-dot checking)
    int32_t *dbg;         // optional: the block dots s[c][row][b] (checking)
};

constexpr unsigned kErrMmqTimeout = 0x100u;  // the pipeline's timeout bit: an MMA batch never completed

__device__ __forceinline__ bool mmq_wait(uint32_t bar, uint32_t parity, unsigned *err) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (global_ns() - t0 > kWaitLimitNs) {
            atomicOr(err, kErrMmqTimeout);
            return false;
        }
    }
    return true;
}

// The 8 fp16 weights 4m..4m+3 (lo) and 4m+16..4m+19 (hi) of index word m,
// from its expanded biased level bytes e0 (elements 4m, 4m+16, 4m+1, 4m+17)
// and e1 (4m+2, 4m+18, 4m+3, 4m+19): each pair's bytes next to 0x64.
__device__ __forceinline__ void mmq_halves(uint32_t e0, uint32_t e1, uint32_t (&lo)[2], uint32_t (&hi)[2]) {
    constexpr uint32_t k64 = 0x64646464u;
    lo[0] = prmt(e0, k64, 0x4240u);
    lo[1] = prmt(e1, k64, 0x4240u);
    hi[0] = prmt(e0, k64, 0x4341u);
    hi[1] = prmt(e1, k64, 0x4341u);
}

// One CTA (128 threads, thread = row of a 128-row tile: pair 2t + tid/64,
// group (tid/32)%2, lane tid%32) per tile at a time, tiles strided over the
// grid.  Per chunk of four blocks: every thread expands its row into the A
// tiles and copies its share of the B tiles and block metadata; after a CTA
// barrier thread 0 issues the chunk's MMAs (two per block, into 16 tensor-
// memory columns each) and commits them to the chunk's mbarrier; meanwhile
// the threads read the previous chunk's sums from tensor memory (warp w owns
// lanes 32w..32w+31) and scale them into their row's n running sums.  A and B
// tiles and the two chunks' sums are double-buffered, the metadata (read by
// the threads themselves) triple-buffered.  The index words and scales of
// the next chunk are loaded one chunk ahead.
__global__ void __launch_bounds__(kMmqThreads) k_mmq(const __grid_constant__ MmqArgs A) {
    extern __shared__ __align__(1024) unsigned char smem[];
    __shared__ uint32_t tmem_slot;
    __shared__ __align__(8) uint64_t bars[2];
    __shared__ uint32_t cbw[4];
    unsigned char *sA = smem;                                           // [2][4] A tiles
    unsigned char *sB = sA + 2 * kMmqChunk * kMmqATile;                 // [2][4] B tiles
    float *sMeta = reinterpret_cast<float *>(sB + 2 * kMmqChunk * kMmqBTile);  // [3][4][32]
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const DevMat &W = A.W;
    if (warp == 0) tmem_alloc(smem_addr(&tmem_slot), kMmqTmemCols);
    if (tid == 0) {
        mbar_init(smem_addr(&bars[0]), 1);
        mbar_init(smem_addr(&bars[1]), 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        // the codebook words with every level biased by 128 (level XOR 0x80)
        cbw[0] = kCb0 ^ 0x80808080u;
        cbw[1] = kCb1 ^ 0x80808080u;
        cbw[2] = kCb2 ^ 0x80808080u;
        cbw[3] = kCb3 ^ 0x80808080u;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    pdl_wait();
    pdl_trigger();
    const uint32_t tmem = tmem_slot;
    const Codebook cb{cbw[0], cbw[1], cbw[2], cbw[3], 0u, 0u, 0};
    const int nb = W.nb, nbp = W.nbp, n = A.n;
    const int T = (W.P + 1) / 2, nch = (nb + kMmqChunk - 1) / kMmqChunk;
    const size_t pb = pair_bytes(nbp);
    const uint32_t a0 = smem_addr(sA), b0 = smem_addr(sB);
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    uint32_t phases = 0u;  // bit i: the phase of bars[i] to wait for next
    for (int t = blockIdx.x; t < T; t += gridDim.x) {
        const int pair = 2 * t + (tid >> 6), h = (tid >> 5) & 1;
        const bool live = pair < W.P;
        const uint8_t *wp = W.w + (size_t)(live ? pair : 0) * pb;
        const int64_t row = (int64_t)pair * 64 + h * 32 + lane;
        float acc[kMmqN];
#pragma unroll
        for (int c = 0; c < kMmqN; ++c) acc[c] = 0.0f;
        uint4 q[kMmqChunk];
        uint2 sc = make_uint2(0u, 0u), sc_rd = sc, sc_keep = sc;  // scales: fetched chunk, chunk read out, chunk issued
        auto fetch = [&](int ch) {
#pragma unroll
            for (int j = 0; j < kMmqChunk; ++j) {
                const int b = ch * kMmqChunk + j;
                q[j] = live && b < nb ? *reinterpret_cast<const uint4 *>(wp + field_offset(nbp, h, b, lane))
                                      : make_uint4(0u, 0u, 0u, 0u);
            }
            sc = live ? *reinterpret_cast<const uint2 *>(wp + scale_offset(nbp, h, ch * kMmqChunk, lane))
                      : make_uint2(0u, 0u);
        };
        if (nch > 0) fetch(0);
        for (int ch = 0; ch <= nch; ++ch) {
            const int buf = ch & 1;
            const int nv = ch < nch ? min(kMmqChunk, nb - ch * kMmqChunk) : 0;
            if (ch < nch) {
                // this row of the chunk's A tiles
#pragma unroll
                for (int j = 0; j < kMmqChunk; ++j) {
                    if (j >= nv) break;
                    const uint32_t ws[4] = {q[j].x, q[j].y, q[j].z, q[j].w};
                    uint32_t lo[4][2], hi[4][2];
#pragma unroll
                    for (int m = 0; m < 4; ++m) {
                        uint32_t e0, e1;
                        expand_select(cb, ws[m], e0, e1);
                        mmq_halves(e0, e1, lo[m], hi[m]);
                    }
                    unsigned char *at = sA + (buf * kMmqChunk + j) * kMmqATile;
                    *reinterpret_cast<uint4 *>(at + mmq_core_off(tid, 0)) = make_uint4(lo[0][0], lo[0][1], lo[1][0], lo[1][1]);
                    *reinterpret_cast<uint4 *>(at + mmq_core_off(tid, 8)) = make_uint4(lo[2][0], lo[2][1], lo[3][0], lo[3][1]);
                    *reinterpret_cast<uint4 *>(at + mmq_core_off(tid, 16)) = make_uint4(hi[0][0], hi[0][1], hi[1][0], hi[1][1]);
                    *reinterpret_cast<uint4 *>(at + mmq_core_off(tid, 24)) = make_uint4(hi[2][0], hi[2][1], hi[3][0], hi[3][1]);
                }
                // the chunk's B tiles and metadata
                const uint4 *gb = reinterpret_cast<const uint4 *>(A.bimg + (size_t)ch * kMmqChunk * kMmqBTile);
                uint4 *sb = reinterpret_cast<uint4 *>(sB + buf * kMmqChunk * kMmqBTile);
                for (int i = tid; i < nv * (kMmqBTile / 16); i += kMmqThreads) sb[i] = gb[i];
                const uint4 *gm = reinterpret_cast<const uint4 *>(A.meta + (size_t)ch * kMmqChunk * kMmqMetaFloats);
                uint4 *sm = reinterpret_cast<uint4 *>(sMeta + (ch % 3) * kMmqChunk * kMmqMetaFloats);
                if (tid < nv * (kMmqMetaFloats / 4)) sm[tid] = gm[tid];
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                sc_keep = sc;
                if (ch + 1 < nch) fetch(ch + 1);
            }
            tc_fence_before();
            __syncthreads();
            tc_fence_after();
            if (tid == 0 && nv > 0) {
                for (int j = 0; j < nv; ++j) {
                    const uint32_t d = tmem + (uint32_t)((buf * kMmqChunk + j) * kMmqN);
                    const uint32_t at = a0 + (uint32_t)((buf * kMmqChunk + j) * kMmqATile);
                    const uint32_t bt = b0 + (uint32_t)((buf * kMmqChunk + j) * kMmqBTile);
                    mmq_mma(d, mmq_desc(at, 128, 512), mmq_desc(bt, 128, 512), 0);
                    mmq_mma(d, mmq_desc(at + 256, 128, 512), mmq_desc(bt + 256, 128, 512), 1);
                }
                mmq_commit(smem_addr(&bars[buf]));
            }
            if (ch > 0) {
                // the previous chunk's sums
                const int pc = ch - 1, pbuf = pc & 1, pnv = min(kMmqChunk, nb - pc * kMmqChunk);
                mmq_wait(smem_addr(&bars[pbuf]), (phases >> pbuf) & 1u, W.err);
                phases ^= 1u << pbuf;
                tc_fence_after();
                const float *mt = sMeta + (pc % 3) * kMmqChunk * kMmqMetaFloats;
#pragma unroll
                for (int j = 0; j < kMmqChunk; ++j) {
                    if (j >= pnv) break;
                    float d[kMmqN];
                    tmem_ld16(tmem + lane_base + (uint32_t)((pbuf * kMmqChunk + j) * kMmqN), d);
                    const uint32_t scw = j < 2 ? sc_rd.x : sc_rd.y;
                    const float dw = (j & 1) ? half_hi(scw) : half_lo(scw);
                    const float *md = mt + j * kMmqMetaFloats;
#pragma unroll
                    for (int c = 0; c < kMmqN; ++c) {
                        const float s = __fsub_rn(d[c], md[kMmqN + c]);
                        acc[c] = __fmaf_rn(__fmul_rn(dw, md[c]), s, acc[c]);
                    }
                    if (A.dbg && live && row < W.M) {
                        const int b = pc * kMmqChunk + j;
#pragma unroll
                        for (int c = 0; c < kMmqN; ++c)
                            if (c < n) A.dbg[((size_t)c * W.M + row) * nb + b] = (int32_t)__fsub_rn(d[c], md[kMmqN + c]);
                    }
                }
            }
            sc_rd = sc_keep;
        }
        if (A.y && live && row < W.M) {
#pragma unroll
            for (int c = 0; c < kMmqN; ++c)
                if (c < n) A.y[(size_t)c * W.M + row] = acc[c];
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, kMmqTmemCols);
}

size_t mmq_bimg_bytes(int nb) { return (size_t)nb * kMmqBTile; }
size_t mmq_meta_bytes(int nb) { return (size_t)nb * kMmqMetaFloats * sizeof(float); }

cudaError_t launch_mmq_prep(const int8_t *qx, const float *dx, int n, int64_t K, uint8_t *bimg, float *meta,
                            cudaStream_t s) {
    const int nb = (int)(K / 32);
    if (nb <= 0) return cudaSuccess;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3((unsigned)std::min(nb, 4096));
    cfg.blockDim = dim3(512);
    cfg.stream = s;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k_mmq_prep, qx, dx, n, K, nb, bimg, meta);
}

cudaError_t launch_mmq(const DevMat &W, const uint8_t *bimg, const float *meta, int n, float *y, int32_t *dbg,
                       cudaStream_t s) {
    static bool raised = false;  // the dynamic shared memory above the default 48 KB
    if (!raised) {
        cudaError_t e = cudaFuncSetAttribute(k_mmq, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kMmqSmem);
        if (e != cudaSuccess) return e;
        raised = true;
    }
    int dev = 0, sms = 0, per_sm = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_mmq, kMmqThreads, kMmqSmem);
    if (e != cudaSuccess) return e;
    // tensor memory: kMmqTmemCols columns per resident CTA, 512 per SM
    per_sm = std::max(1, std::min(per_sm, (int)(512 / kMmqTmemCols)));
    const int T = (int)((W.P + 1) / 2);
    const int grid = std::max(1, std::min(T, sms * per_sm));
    MmqArgs A{W, bimg, meta, n, y, dbg};
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kMmqThreads);
    cfg.dynamicSmemBytes = kMmqSmem;
    cfg.stream = s;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k_mmq, A);
}

}  // namespace cbq

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
// roundings per block, acc = fma(dw*dx, s, acc), with the row's blocks (in
// units of four) alternating between two running sums added at the end.
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
#include <mutex>

#include <cuda_fp16.h>

#include "cbq_internal.h"
#include "cbq_pipe.cuh"

namespace cbq {

constexpr int kMmqN = 16;                    // MMA N: activation columns (zero-padded)
constexpr int kMmqM = 128;                   // MMA M: weight rows of a tile
constexpr int kMmqATile = kMmqM * 32 * 2;    // 8 KB: the fp16 A tile of one block
constexpr int kMmqBTile = kMmqN * 32 * 2;    // 1 KB: the fp16 B tile of one block
constexpr int kMmqMetaFloats = 2 * kMmqN;    // per block: dx[16], then 1152 * sum q [16]
constexpr float kMmqBias = 1152.0f;

// Byte offset of element (row, k) in a tile of the core-matrix layout.
__host__ __device__ inline uint32_t mmq_core_off(int row, int k) {
    return (uint32_t)(((row >> 3) * 4 + (k >> 3)) * 128 + (row & 7) * 16 + (k & 7) * 2);
}

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
template <int N>
constexpr uint32_t mmq_idesc() { return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(kMmqM >> 4) << 24); }

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

template <int N>
__device__ __forceinline__ void mmq_mma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, int accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(mmq_idesc<N>()), "r"(accumulate)
        : "memory");
}

// Arrive on the mbarrier once every MMA this thread issued so far is done.
__device__ __forceinline__ void mmq_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

// 16 consecutive fp32 columns of this thread's tensor-memory lane, as raw
// words; complete once tmem_wait_ld() returns.
__device__ __forceinline__ void tmem_ld16_issue(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}
// 8 consecutive fp32 columns of this thread's tensor-memory lane, as raw
// words; complete once tmem_wait_ld() returns.
__device__ __forceinline__ void tmem_ld8_issue(uint32_t taddr, uint32_t (&r)[8]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr)
                 : "memory");
}
template <int N>
__device__ __forceinline__ void tmem_ld_issue(uint32_t taddr, uint32_t (&r)[N]) {
    if constexpr (N == 16) tmem_ld16_issue(taddr, r);
    else tmem_ld8_issue(taddr, r);
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

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
    int stall;            // give-up test mode: CTA 0's producer issues no copy
};

constexpr unsigned kErrMmqTimeout = 0x100u;  // the pipeline's timeout bit: an MMA batch never completed

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

// Warp-specialised tiles, one CTA per SM (its tensor-memory ring takes half
// of the SM's 512 columns), tiles strided over the grid; every role walks the
// same sequence (tile, stage of 16 blocks, unit of up to 4 blocks, block):
//   warp 12, the producer: per stage, bulk copies of the tile's two pairs'
//     weight chunk, the 16 B tiles and their metadata into a ring of stages;
//   warps 8-11, the expanders: thread = row; it expands the row's blocks of
//     each unit into a ring of A units (four block tiles each);
//   warp 13, the MMA issuer: per unit, two MMAs per block from the A tiles and
//     the stage's B tiles into a ring of units of sums in tensor memory (16
//     columns per block), then commits that free the A unit and publish the
//     sums (and, after a stage's last unit, free the stage's B tiles);
//   warps 0-7, the epilogue, in two groups of four warps that take alternate
//     units: thread = row (warp w reads tensor-memory lanes 32(w%4)..+31);
//     per unit it reads the sums, frees their slot and scales them into the
//     row's n running sums; at the end of a tile group 1 hands its sums to
//     group 0 through shared memory, which adds them and stores y.
// Synchronising per unit rather than per block keeps the barrier and commit
// traffic of the single MMA thread and of the epilogue to a quarter.
// Every wait is bounded (kWaitLimitNs): a give-up sets kErrMmqTimeout and a
// CTA-wide abort flag, after which every role leaves its loop; the producer
// then waits (bounded) for its copies in flight and the MMA issuer for its
// MMAs before the CTA frees its tensor memory.
constexpr int kM2Stages = 2;
constexpr int kM2Unit = 4;                               // blocks per unit
constexpr int kM2AUnits = 3;                             // A ring (units)
constexpr int kM2DUnits = 4;                             // tensor-memory ring (units)
constexpr int kM2WBytes = kChunkBytes;                  // one pair's weight chunk (at most)
constexpr int kM2BOff = 2 * kM2WBytes;                  // B tiles of the stage's blocks
constexpr int kM2MetaOff = kM2BOff + kChunk * kMmqBTile; // their metadata
constexpr int kM2StageBytes = kM2MetaOff + kChunk * kMmqMetaFloats * 4;  // 55,296
constexpr int kM2EpWarps = 8, kM2ExWarps = 4;  // multiples of 4 (one warp per tensor-memory lane quadrant)
constexpr int kM2EpGroups = kM2EpWarps / 4;     // epilogue groups: group g reads the units u with u % groups == g
constexpr int kM2ExGroups = kM2ExWarps / 4;     // expander groups (one: a thread per row takes every block)
constexpr int kM2EpBatch = 2;  // blocks whose sums the epilogue loads before one wait
constexpr int kM2ProducerWarp = kM2EpWarps + kM2ExWarps, kM2MmaWarp = kM2ProducerWarp + 1;
constexpr int kM2Threads = (kM2MmaWarp + 1) * 32;      // 448
constexpr int kM2StageArrivals = kM2ExWarps * 32 + kM2EpWarps * 32 + 1;
template <int N>
constexpr uint32_t m2_tmem_cols() { return kM2DUnits * kM2Unit * N; }  // 256 at N = 16, 128 at N = 8
constexpr size_t kM2AUnitBytes = (size_t)kM2Unit * kMmqATile;  // 32 KB
template <int N>
constexpr size_t m2_part_bytes() { return (size_t)(kM2EpGroups - 1) * kMmqM * N * 4; }  // partial sums of groups 1..
template <int N>
constexpr size_t m2_smem() {
    return (size_t)kM2Stages * kM2StageBytes + (size_t)kM2AUnits * kM2AUnitBytes + m2_part_bytes<N>();
}

struct M2Shared {
    uint64_t sfull[kM2Stages], sempty[kM2Stages];
    uint64_t afull[kM2AUnits], aempty[kM2AUnits];
    uint64_t dfull[kM2DUnits], dempty[kM2DUnits];
    uint64_t done;  // the MMA issuer's last commit
    uint32_t tmem_slot;
    uint32_t cbw[4];
    int abort;
};

__device__ __forceinline__ bool m2_wait(M2Shared &S, uint64_t &bar, uint32_t parity, unsigned *err) {
    const uint32_t b = smem_addr(&bar);
    if (mbar_try_wait(b, parity)) return true;
    const uint64_t t0 = global_ns();
    for (;;) {
        if (*(volatile int *)&S.abort) return false;
        if (mbar_try_wait(b, parity)) return true;
        if (global_ns() - t0 > kWaitLimitNs) break;
    }
    atomicOr(err, kErrMmqTimeout);
    *(volatile int *)&S.abort = 1;
    return false;
}

template <int N>
__global__ void __launch_bounds__(kM2Threads, 1) k_mmq(const __grid_constant__ MmqArgs A) {
    extern __shared__ __align__(1024) unsigned char smem[];
    __shared__ M2Shared S;
    unsigned char *stages = smem;
    unsigned char *aunits = smem + (size_t)kM2Stages * kM2StageBytes;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const DevMat &W = A.W;
    unsigned *err = W.err;
    if (warp == 0) tmem_alloc(smem_addr(&S.tmem_slot), m2_tmem_cols<N>());
    if (tid == 32) {
        for (int i = 0; i < kM2Stages; ++i) {
            mbar_init(smem_addr(&S.sfull[i]), 1);
            mbar_init(smem_addr(&S.sempty[i]), kM2StageArrivals);
        }
        for (int i = 0; i < kM2AUnits; ++i) {
            mbar_init(smem_addr(&S.afull[i]), kM2ExWarps * 32);
            mbar_init(smem_addr(&S.aempty[i]), 1);
        }
        for (int i = 0; i < kM2DUnits; ++i) {
            mbar_init(smem_addr(&S.dfull[i]), 1);
            mbar_init(smem_addr(&S.dempty[i]), kMmqM);
        }
        mbar_init(smem_addr(&S.done), 1);
        S.abort = 0;
        S.cbw[0] = kCb0 ^ 0x80808080u;  // the codebook words, every level biased by 128
        S.cbw[1] = kCb1 ^ 0x80808080u;
        S.cbw[2] = kCb2 ^ 0x80808080u;
        S.cbw[3] = kCb3 ^ 0x80808080u;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    pdl_wait();
    pdl_trigger();
    const uint32_t tmem = S.tmem_slot;
    const int nb = W.nb, nbp = W.nbp, n = A.n;
    const int T = (W.P + 1) / 2, nch = (nb + kChunk - 1) / kChunk;
    const size_t pb = pair_bytes(nbp);

    if (warp == kM2ProducerWarp) {
        if (lane == 0) {
            uint32_t k = 0;
            // give-up test mode: CTA 0 fills no stage, so every role's
            // bounded wait for its first stage runs out
            bool ok = !(A.stall == 1 && blockIdx.x == 0);
            for (int t = blockIdx.x; t < T && ok; t += gridDim.x) {
                const int p0 = 2 * t, p1 = 2 * t + 1;
                for (int c = 0; c < nch && ok; ++c, ++k) {
                    const uint32_t slot = k % kM2Stages, use = k / kM2Stages;
                    if (use > 0 && !m2_wait(S, S.sempty[slot], (use - 1) & 1u, err)) {
                        ok = false;
                        break;
                    }
                    const int nblk = chunk_blocks(nbp, c), nv = min(kChunk, nb - c * kChunk);
                    const uint32_t bw = (uint32_t)nblk * (2 * kBlockBytes);
                    const uint32_t bytes = bw * (p1 < W.P ? 2u : 1u) + (uint32_t)nv * (kMmqBTile + kMmqMetaFloats * 4);
                    const uint32_t dst = smem_addr(stages) + slot * kM2StageBytes, bar = smem_addr(&S.sfull[slot]);
                    mbar_expect_tx(bar, bytes);
                    bulk_g2s(dst, W.w + (size_t)p0 * pb + (size_t)c * kChunkBytes, bw, bar);
                    if (p1 < W.P) bulk_g2s(dst + kM2WBytes, W.w + (size_t)p1 * pb + (size_t)c * kChunkBytes, bw, bar);
                    bulk_g2s(dst + kM2BOff, A.bimg + (size_t)c * kChunk * kMmqBTile, (uint32_t)nv * kMmqBTile, bar);
                    bulk_g2s(dst + kM2MetaOff, A.meta + (size_t)c * kChunk * kMmqMetaFloats,
                             (uint32_t)nv * kMmqMetaFloats * 4, bar);
                }
            }
            // the copies still in flight land before the CTA may exit
            const uint32_t first = k > (uint32_t)kM2Stages ? k - kM2Stages : 0u;
            for (uint32_t q = first; q < k; ++q) {
                const uint32_t b = smem_addr(&S.sfull[q % kM2Stages]);
                const uint64_t t0 = global_ns();
                while (!mbar_try_wait(b, (q / kM2Stages) & 1u) && global_ns() - t0 < kWaitLimitNs) {}
            }
        }
    } else if (warp == kM2MmaWarp) {
        if (lane == 0) {
            uint32_t k = 0, u = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < T && ok; t += gridDim.x) {
                for (int c = 0; c < nch && ok; ++c, ++k) {
                    const uint32_t slot = k % kM2Stages;
                    if (!m2_wait(S, S.sfull[slot], (k / kM2Stages) & 1u, err)) {
                        ok = false;
                        break;
                    }
                    const int nv = min(kChunk, nb - c * kChunk);
                    const uint32_t bt0 = smem_addr(stages) + slot * kM2StageBytes + kM2BOff;
                    for (int j0 = 0; j0 < nv; j0 += kM2Unit, ++u) {
                        const uint32_t as = u % kM2AUnits, ds = u % kM2DUnits, du = u / kM2DUnits;
                        if (!m2_wait(S, S.afull[as], (u / kM2AUnits) & 1u, err) ||
                            (du > 0 && !m2_wait(S, S.dempty[ds], (du - 1) & 1u, err))) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const int nu = min(kM2Unit, nv - j0);
                        for (int i = 0; i < nu; ++i) {
                            const uint32_t d = tmem + (ds * kM2Unit + (uint32_t)i) * N;
                            const uint32_t at = smem_addr(aunits) + (uint32_t)(as * kM2AUnitBytes) + (uint32_t)i * kMmqATile;
                            const uint32_t bt = bt0 + (uint32_t)(j0 + i) * kMmqBTile;
                            mmq_mma<N>(d, mmq_desc(at, 128, 512), mmq_desc(bt, 128, 512), 0);
                            mmq_mma<N>(d, mmq_desc(at + 256, 128, 512), mmq_desc(bt + 256, 128, 512), 1);
                        }
                        mmq_commit(smem_addr(&S.aempty[as]));
                        mmq_commit(smem_addr(&S.dfull[ds]));
                    }
                    if (ok) mmq_commit(smem_addr(&S.sempty[slot]));
                }
            }
            // every MMA issued here is done before the tensor memory is freed
            mmq_commit(smem_addr(&S.done));
            const uint64_t t0 = global_ns();
            while (!mbar_try_wait(smem_addr(&S.done), 0u) && global_ns() - t0 < kWaitLimitNs) {}
        }
    } else if (warp >= kM2EpWarps) {
        // expanders: thread = row, every block of a unit
        const int e = tid - kM2EpWarps * 32, row = e & (kMmqM - 1);
        const int pl = row >> 6, h = (row >> 5) & 1, rl = row & 31;
        const Codebook cb{S.cbw[0], S.cbw[1], S.cbw[2], S.cbw[3], 0u, 0u, 0};
        uint32_t k = 0, u = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < T && ok; t += gridDim.x) {
            const bool live = 2 * t + pl < W.P;
            for (int c = 0; c < nch && ok; ++c, ++k) {
                const uint32_t slot = k % kM2Stages;
                if (!m2_wait(S, S.sfull[slot], (k / kM2Stages) & 1u, err)) {
                    ok = false;
                    break;
                }
                const int nblk = chunk_blocks(nbp, c), nv = min(kChunk, nb - c * kChunk);
                const unsigned char *wst = stages + (size_t)slot * kM2StageBytes + pl * kM2WBytes +
                                           (size_t)h * nblk * kBlockBytes;
                for (int j0 = 0; j0 < nv; j0 += kM2Unit, ++u) {
                    const uint32_t as = u % kM2AUnits, au = u / kM2AUnits;
                    if (au > 0 && !m2_wait(S, S.aempty[as], (au - 1) & 1u, err)) {
                        ok = false;
                        break;
                    }
                    const int nu = min(kM2Unit, nv - j0);
                    // the unit's index words are loaded together, ahead of their
                    // expansion (one expander group: this thread takes every block)
                    static_assert(kM2ExGroups == 1, "one expander group");
                    uint4 qq[kM2Unit];
#pragma unroll
                    for (int i = 0; i < kM2Unit; ++i)
                        qq[i] = live && i < nu ? *reinterpret_cast<const uint4 *>(wst + ((size_t)(j0 + i) * 32 + rl) * 16)
                                               : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
                    for (int i = 0; i < kM2Unit; ++i) {
                        if (i >= nu) break;
                        const uint4 q = qq[i];
                        const uint32_t ws[4] = {q.x, q.y, q.z, q.w};
                        uint32_t lo[4][2], hi[4][2];
#pragma unroll
                        for (int m = 0; m < 4; ++m) {
                            uint32_t e0, e1;
                            expand_select(cb, ws[m], e0, e1);
                            mmq_halves(e0, e1, lo[m], hi[m]);
                        }
                        unsigned char *at = aunits + (size_t)as * kM2AUnitBytes + (size_t)i * kMmqATile;
                        *reinterpret_cast<uint4 *>(at + mmq_core_off(row, 0)) = make_uint4(lo[0][0], lo[0][1], lo[1][0], lo[1][1]);
                        *reinterpret_cast<uint4 *>(at + mmq_core_off(row, 8)) = make_uint4(lo[2][0], lo[2][1], lo[3][0], lo[3][1]);
                        *reinterpret_cast<uint4 *>(at + mmq_core_off(row, 16)) = make_uint4(hi[0][0], hi[0][1], hi[1][0], hi[1][1]);
                        *reinterpret_cast<uint4 *>(at + mmq_core_off(row, 24)) = make_uint4(hi[2][0], hi[2][1], hi[3][0], hi[3][1]);
                    }
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    mbar_arrive(smem_addr(&S.afull[as]));
                }
                mbar_arrive(smem_addr(&S.sempty[slot]));
            }
        }
    } else {
        // epilogue: thread (row, group) -- the units u == group (mod groups)
        const int row = tid & (kMmqM - 1), eg = tid >> 7, pl = row >> 6, h = (row >> 5) & 1, rl = row & 31;
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
        float *part = reinterpret_cast<float *>(aunits + (size_t)kM2AUnits * kM2AUnitBytes);
        uint32_t k = 0, u = 0;
        bool ok = true;
        // every epilogue thread walks every tile (after a give-up without work)
        // so all of them reach the group barriers below equally often
        for (int t = blockIdx.x; t < T; t += gridDim.x) {
            const int pair = 2 * t + pl;
            const bool live = pair < W.P;
            const int64_t grow = (int64_t)pair * 64 + h * 32 + rl;
            float acc[N];
#pragma unroll
            for (int c = 0; c < N; ++c) acc[c] = 0.0f;
            for (int c = 0; c < nch && ok; ++c, ++k) {
                const uint32_t slot = k % kM2Stages;
                if (!m2_wait(S, S.sfull[slot], (k / kM2Stages) & 1u, err)) {
                    ok = false;
                    break;
                }
                const int nblk = chunk_blocks(nbp, c), nv = min(kChunk, nb - c * kChunk);
                const unsigned char *st = stages + (size_t)slot * kM2StageBytes;
                const uint2 *scp = reinterpret_cast<const uint2 *>(st + pl * kM2WBytes + (size_t)h * nblk * kBlockBytes +
                                                                  (size_t)nblk * 512) + rl;
                const float *mt = reinterpret_cast<const float *>(st + kM2MetaOff);
                for (int j0 = 0; j0 < nv && ok; j0 += kM2Unit, ++u) {
                    if ((int)(u % kM2EpGroups) != eg) continue;
                    const uint32_t ds = u % kM2DUnits;
                    if (!m2_wait(S, S.dfull[ds], (u / kM2DUnits) & 1u, err)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const int nu = min(kM2Unit, nv - j0);
                    const uint2 sq = live ? scp[(j0 >> 2) * 32] : make_uint2(0u, 0u);  // the unit's four scales
                    for (int i0 = 0; i0 < nu; i0 += kM2EpBatch) {
                        uint32_t d[kM2EpBatch][N];
#pragma unroll
                        for (int i = 0; i < kM2EpBatch; ++i)
                            if (i0 + i < nu)
                                tmem_ld_issue<N>(tmem + lane_base + (ds * kM2Unit + (uint32_t)(i0 + i)) * N, d[i]);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < kM2EpBatch; ++i) {
                            if (i0 + i >= nu) break;
                            const int jj = i0 + i, j = j0 + jj;
                            const uint32_t sw = (jj & 2) ? sq.y : sq.x;
                            const float dw = (jj & 1) ? half_hi(sw) : half_lo(sw);
                            const float *md = mt + j * kMmqMetaFloats;
                            // every one of the N columns: a padded column has a zero sum, correction
                            // and scale, so its running sum stays zero (no per-column test)
#pragma unroll
                            for (int cc = 0; cc < N; ++cc) {
                                const float sdot = __fsub_rn(__uint_as_float(d[i][cc]), md[kMmqN + cc]);
                                acc[cc] = __fmaf_rn(__fmul_rn(dw, md[cc]), sdot, acc[cc]);
                            }
                            if (A.dbg && live && grow < W.M) {
                                const int b = c * kChunk + j;
#pragma unroll
                                for (int cc = 0; cc < N; ++cc)
                                    if (cc < n)
                                        A.dbg[((size_t)cc * W.M + grow) * nb + b] =
                                            (int32_t)__fsub_rn(__uint_as_float(d[i][cc]), md[kMmqN + cc]);
                            }
                        }
                    }
                    tc_fence_before();
                    mbar_arrive(smem_addr(&S.dempty[ds]));
                }
                mbar_arrive(smem_addr(&S.sempty[slot]));
            }
            if (kM2EpGroups > 1) {
                // the groups' partial sums of this tile: groups 1.. hand theirs
                // to group 0 through shared memory (epilogue threads only)
                if (eg > 0) {
#pragma unroll
                    for (int cc = 0; cc < N; ++cc) part[((eg - 1) * N + cc) * kMmqM + row] = acc[cc];
                }
                asm volatile("bar.sync 2, %0;" ::"n"(kM2EpWarps * 32) : "memory");
                if (eg == 0) {
                    for (int g2 = 1; g2 < kM2EpGroups; ++g2)
#pragma unroll
                        for (int cc = 0; cc < N; ++cc) acc[cc] += part[((g2 - 1) * N + cc) * kMmqM + row];
                }
                asm volatile("bar.sync 2, %0;" ::"n"(kM2EpWarps * 32) : "memory");
            }
            if (eg == 0 && ok && A.y && live && grow < W.M) {
#pragma unroll
                for (int cc = 0; cc < N; ++cc)
                    if (cc < n) A.y[(size_t)cc * W.M + grow] = acc[cc];
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, m2_tmem_cols<N>());
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

// Raise the kernel's dynamic shared memory limit above the default 48 KB,
// once per device (a function attribute belongs to the device's context).
template <int N>
static cudaError_t mmq_raise_smem(int dev) {
    static std::mutex mu;
    static bool raised[64] = {};
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (!raised[dev]) {
        const cudaError_t e = cudaFuncSetAttribute(k_mmq<N>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)m2_smem<N>());
        if (e != cudaSuccess) return e;
        raised[dev] = true;
    }
    return cudaSuccess;
}

template <int N>
static cudaError_t launch_mmq_n(const DevMat &W, const uint8_t *bimg, const float *meta, int n, float *y,
                                int32_t *dbg, int stall, cudaStream_t s) {
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = mmq_raise_smem<N>(dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const int T = (int)((W.P + 1) / 2);
    const int grid = std::max(1, std::min(T, sms));  // one CTA per SM
    MmqArgs A{W, bimg, meta, n, y, dbg, stall};
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kM2Threads);
    cfg.dynamicSmemBytes = m2_smem<N>();
    cfg.stream = s;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k_mmq<N>, A);
}

// Up to eight columns: MMAs of N = 8 (half the tensor memory, half the
// read-out and scaling per block); otherwise N = 16.
cudaError_t launch_mmq(const DevMat &W, const uint8_t *bimg, const float *meta, int n, float *y, int32_t *dbg,
                       int stall, cudaStream_t s) {
    if (n <= 8) return launch_mmq_n<8>(W, bimg, meta, n, y, dbg, stall, s);
    return launch_mmq_n<16>(W, bimg, meta, n, y, dbg, stall, s);
}

}  // namespace cbq

// cbq_pipe.cuh -- the weight-stream pipeline of the matvec kernels.
//
// One producer warp per CTA moves the weight stream from HBM into a ring of
// shared-memory stages with 1-D bulk copies (cp.async.bulk, the TMA's
// non-tensor form), each stage completing on an mbarrier.  Eight consumer
// warps wait for a stage, expand and dot it from shared memory, and release it
// through a second mbarrier.  A stage is one chunk of a 32-row group: up to 32
// block columns, i.e. 16 KB of index fields plus 2 KB of scales, contiguous in
// the device layout (cbq_device.cuh), so each stage is two bulk copies.
//
// Work is fetched dynamically: the producer takes item indices from a global
// counter with atomicAdd (the last CTA to exit resets it), tags every stage
// with its item in a small shared header, and closes the stream with a stage
// tagged -1 that carries no bytes.  Consumers read the tag at each item
// boundary, so CTAs of unequal speed share the work evenly.
//
// Every wait is bounded: once it has waited kWaitLimitNs (global timer) it
// sets kErrPipeTimeout in the device error word and a CTA-wide abort flag; the
// other waits of the CTA then give up too, consumers keep their barrier
// sequence (so no named barrier is left waiting), and the producer waits for
// its own copies in flight before the CTA exits.
#pragma once

#include <stdint.h>

#include <cuda_fp16.h>

#include "cbq_device.cuh"

namespace cbq {

constexpr int kConsumerWarps = 8;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kPipeThreads = kConsumers + 32;   // + one producer warp
constexpr int kChunkBlocks = 32;                 // block columns per stage
constexpr int kStageQsBytes = kChunkBlocks * 512;
constexpr int kStageBytes = kStageQsBytes + kChunkBlocks / 4 * 256;  // 18,432
// Bounded waits: each poll suspends the warp until the phase completes or
// kWaitHintNs pass (so a waiting warp takes no issue slots from the warps that
// compute); a wait gives up after kWaitLimitNs in all.
constexpr uint32_t kWaitHintNs = 20000;
constexpr uint64_t kWaitLimitNs = 1000000000ull;
constexpr unsigned kErrPipeTimeout = 0x100u;

// The device error word, defined by the translation unit that includes this
// header (before including it).

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n"
        " mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity), "n"(kWaitHintNs)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

// 1-D bulk copy global -> shared, completing `bytes` of transaction on bar.
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

__device__ __forceinline__ void consumer_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kConsumers) : "memory"); }

// Shared part of the pipeline (carved from dynamic shared memory).
struct Pipe {
    uint64_t *full;   // [S] stage filled (producer arrive + bulk bytes)
    uint64_t *empty;  // [S] stage released (one arrive per consumer thread)
    int *abort;       // CTA-wide give-up flag
    int *tag;         // [S] item of each stage (-1: end of stream)
    unsigned char *ring;
    int S;
};

// Bounded wait for phase `parity` of bar.  Returns false on timeout or when
// the CTA already gave up (check_abort).
__device__ __forceinline__ bool pipe_wait(const Pipe &P, uint64_t *bar, uint32_t parity, bool check_abort) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    for (;;) {
        if (check_abort && *(volatile int *)P.abort) return false;
        if (mbar_try_wait(bar, parity)) return true;
        if (global_ns() - t0 > kWaitLimitNs) break;
    }
    atomicOr(&g_device_error, kErrPipeTimeout);
    *(volatile int *)P.abort = 1;
    return false;
}

// Producer side: a running count of issued stages.
struct Producer {
    uint32_t it = 0;
    bool stopped = false;

    // Claim the next slot (waiting until the consumers released it).
    __device__ __forceinline__ bool claim(const Pipe &P, uint32_t &slot) {
        const uint32_t use = it / (uint32_t)P.S;
        slot = it - use * (uint32_t)P.S;
        if (stopped || (use > 0 && !pipe_wait(P, P.empty + slot, (use - 1) & 1u, true))) {
            stopped = true;
            return false;
        }
        return true;
    }

    // Issue the stages of one 32-row group pass (blocks [0, nbp)) of item `tag`.
    __device__ __forceinline__ void group(const Pipe &P, const uint4 *qs_g, const uint2 *sc_g, int nbp, int tag) {
        for (int b0 = 0; b0 < nbp && !stopped; b0 += kChunkBlocks) {
            const int nblk = min(kChunkBlocks, nbp - b0);
            uint32_t slot;
            if (!claim(P, slot)) break;
            unsigned char *dst = P.ring + (size_t)slot * kStageBytes;
            const uint32_t bq = (uint32_t)nblk * 512u, bs = (uint32_t)nblk / 4u * 256u;
            P.tag[slot] = tag;
            mbar_expect_tx(P.full + slot, bq + bs);
            bulk_g2s(dst, qs_g + (size_t)b0 * 32, bq, P.full + slot);
            bulk_g2s(dst + kStageQsBytes, sc_g + (size_t)(b0 / 4) * 32, bs, P.full + slot);
            ++it;
        }
    }

    // End of stream: a stage tagged -1 with no bytes.
    __device__ __forceinline__ void finish(const Pipe &P) {
        uint32_t slot;
        if (!claim(P, slot)) {
            *(volatile int *)P.abort = 1;  // consumers must not wait for it
            return;
        }
        P.tag[slot] = -1;
        mbar_arrive(P.full + slot);
        ++it;
    }

    // Wait for the copies still in flight (the last S issued stages) so the
    // CTA never exits while the TMA writes into its shared memory.
    __device__ __forceinline__ void drain(const Pipe &P) {
        const uint32_t first = it > (uint32_t)P.S ? it - P.S : 0u;
        for (uint32_t k = first; k < it; ++k) pipe_wait(P, P.full + (k % P.S), (k / P.S) & 1u, false);
    }
};

// Consumer side: the same sequence of stages, advanced in lock step (slot
// and phase parity kept incrementally).
struct Consumer {
    uint32_t slot = 0, phase = 0;
    Codebook cb;

    __device__ __forceinline__ Consumer() : cb(load_codebook()) {}

    __device__ __forceinline__ void advance(const Pipe &P) {
        if (++slot == (uint32_t)P.S) {
            slot = 0;
            phase ^= 1u;
        }
    }

    // Item of the next stage (-1 at the end of the stream or after a give-up),
    // without consuming the stage.
    __device__ __forceinline__ int peek(const Pipe &P) const {
        if (!pipe_wait(P, P.full + slot, phase, true)) return -1;
        return *(volatile int *)(P.tag + slot);
    }

    // Accumulate one 32-row group pass (blocks [0, nbp)) into acc2: two
    // interleaved fp32 partial sums per column (even and odd blocks).
    // act/dxp: the NC columns staged block-major (stage_cols).
    template <int NC>
    __device__ __forceinline__ void group(const Pipe &P, int nbp, const uint4 *act, const float2 *dxp,
                                          float2 acc2[NC], int warp, int lane) {
        for (int b0 = 0; b0 < nbp; b0 += kChunkBlocks) {
            const int nq = min(kChunkBlocks, nbp - b0) / 4;
            const bool ok = pipe_wait(P, P.full + slot, phase, true);
            if (ok) {
                const unsigned char *st = P.ring + (size_t)slot * kStageBytes;
                const uint4 *qs_s = reinterpret_cast<const uint4 *>(st);
                const uint2 *sc_s = reinterpret_cast<const uint2 *>(st + kStageQsBytes);
                const int q0 = (int)((unsigned)(warp * nq) / kConsumerWarps);
                const int q1 = (int)((unsigned)((warp + 1) * nq) / kConsumerWarps);
                for (int q = q0; q < q1; ++q) {
                    const uint2 s = sc_s[q * 32 + lane];
                    const float2 dw01 = __half22float2(*reinterpret_cast<const __half2 *>(&s.x));
                    const float2 dw23 = __half22float2(*reinterpret_cast<const __half2 *>(&s.y));
                    uint4 w[4];
#pragma unroll
                    for (int j = 0; j < 4; ++j) w[j] = qs_s[(q * 4 + j) * 32 + lane];
                    const int bq = b0 + q * 4;
                    const uint4 *aq = act + (size_t)bq * NC * 2;
                    const float2 *dq = dxp + (size_t)(bq >> 1) * NC;
#pragma unroll
                    for (int jj = 0; jj < 4; jj += 2) {  // blocks in pairs: fewer live sums
                        int sa[NC], sb[NC];
                        block_dots<NC>(cb, w[jj], aq + jj * NC * 2, sa);
                        block_dots<NC>(cb, w[jj + 1], aq + (jj + 1) * NC * 2, sb);
                        const float2 dw = jj == 0 ? dw01 : dw23;
#pragma unroll
                        for (int c = 0; c < NC; ++c) acc2[c] = scale_acc2(acc2[c], dw, dq[(jj >> 1) * NC + c], sa[c], sb[c]);
                    }
                }
            }
            mbar_arrive(P.empty + slot);  // every consumer thread, after its own reads
            advance(P);
        }
    }
};

// Sweeps of the routed-expert kernels over one 32-row group pass (blocks
// [0, nbp)) for the columns at col_off[0..ncols): this warp's sum over the pass
// goes to part[c*32 + lane] (its slice of a partial set).
//   - one column (kOne, the common case: one token per expert): the two-word
//     expansion, running sums in registers over the whole pass;
//   - more columns: at every stage, the columns two at a time share one
//     expansion (an odd last column takes the one-column expansion), and each
//     column's stage sum is added to its slice in shared memory, so the
//     registers stay those of two columns while the weight stream is still
//     read once.
template <bool kOne>
__device__ __forceinline__ void group_cols_impl(Consumer &co, const Pipe &P, int nbp, const uint4 *act0,
                                                const float *dx0, const int (&col_off)[kMaxCols], int ncols_rt, float *part,
                                                int warp, int lane) {
    const int ncols = kOne ? 1 : ncols_rt;
    float2 run = make_float2(0.0f, 0.0f);  // kOne: even- and odd-block sums of the pass
    for (int b0 = 0; b0 < nbp; b0 += kChunkBlocks) {
        const int nq = min(kChunkBlocks, nbp - b0) / 4;
        const uint32_t slot = co.slot;
        const bool ok = pipe_wait(P, P.full + slot, co.phase, true);
        if (ok) {
            const unsigned char *st = P.ring + (size_t)slot * kStageBytes;
            const uint4 *qs_s = reinterpret_cast<const uint4 *>(st);
            const uint2 *sc_s = reinterpret_cast<const uint2 *>(st + kStageQsBytes);
            const int q0 = (int)((unsigned)(warp * nq) / kConsumerWarps);
            const int q1 = (int)((unsigned)((warp + 1) * nq) / kConsumerWarps);
            for (int c = 0; c < ncols; c += 2) {
                if (kOne || c + 1 == ncols) {  // one column
                    const int off = kOne ? col_off[0] : pick(col_off, c);
                    const uint4 *act = act0 + off * 2;
                    const float *dxs = dx0 + off;
                    float2 acc = kOne ? run : make_float2(0.0f, 0.0f);
                    for (int q = q0; q < q1; ++q) {
                        const uint2 s = sc_s[q * 32 + lane];
                        const float2 dw01 = __half22float2(*reinterpret_cast<const __half2 *>(&s.x));
                        const float2 dw23 = __half22float2(*reinterpret_cast<const __half2 *>(&s.y));
                        const int bq = b0 + q * 4;
#pragma unroll
                        for (int jj = 0; jj < 4; jj += 2) {
                            int sa[1], sb[1];
                            block_dots<1>(co.cb, qs_s[(q * 4 + jj) * 32 + lane], act + (bq + jj) * 2, sa);
                            block_dots<1>(co.cb, qs_s[(q * 4 + jj + 1) * 32 + lane], act + (bq + jj + 1) * 2, sb);
                            const float2 dx2 = *reinterpret_cast<const float2 *>(dxs + bq + jj);
                            const float2 dw = jj == 0 ? dw01 : dw23;
                            acc = scale_acc2(acc, dw, dx2, sa[0], sb[0]);
                        }
                    }
                    if constexpr (kOne) {
                        run = acc;
                    } else {
                        float *dst = part + c * 32 + lane;
                        *dst = (b0 == 0 ? 0.0f : *dst) + (acc.x + acc.y);
                    }
                } else {  // columns c and c+1, one expansion
                    const int off2[2] = {pick(col_off, c), pick(col_off, c + 1)};
                    float2 acc[2] = {make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f)};
                    for (int q = q0; q < q1; ++q) {
                        const uint2 s = sc_s[q * 32 + lane];
                        const float2 dw01 = __half22float2(*reinterpret_cast<const __half2 *>(&s.x));
                        const float2 dw23 = __half22float2(*reinterpret_cast<const __half2 *>(&s.y));
                        const int bq = b0 + q * 4;
#pragma unroll
                        for (int jj = 0; jj < 4; jj += 2) {
                            int sa[2], sb[2];
                            block_dots_cols<2>(co.cb, qs_s[(q * 4 + jj) * 32 + lane], act0, off2, bq + jj, sa);
                            block_dots_cols<2>(co.cb, qs_s[(q * 4 + jj + 1) * 32 + lane], act0, off2, bq + jj + 1, sb);
                            const float2 dw = jj == 0 ? dw01 : dw23;
#pragma unroll
                            for (int i = 0; i < 2; ++i) {
                                const float2 dx2 = *reinterpret_cast<const float2 *>(dx0 + off2[i] + bq + jj);
                                acc[i] = scale_acc2(acc[i], dw, dx2, sa[i], sb[i]);
                            }
                        }
                    }
#pragma unroll
                    for (int i = 0; i < 2; ++i) {
                        float *dst = part + (c + i) * 32 + lane;
                        *dst = (b0 == 0 ? 0.0f : *dst) + (acc[i].x + acc[i].y);
                    }
                }
            }
        }
        mbar_arrive(P.empty + slot);  // every consumer thread, after its own reads
        co.advance(P);
    }
    if constexpr (kOne) part[lane] = run.x + run.y;
}

// NC columns in one sweep: each 32-block index word is expanded once and its
// levels dotted with every column (as the dense kernel does), the running sums
// kept in registers over the whole pass and stored once at its end.  Used for
// two columns (more would not fit the layer kernel's 96 registers).
template <int NC>
__device__ __forceinline__ void group_cols_n(Consumer &co, const Pipe &P, int nbp, const uint4 *act0,
                                             const float *dx0, const int (&col_off)[kMaxCols], float *part, int warp,
                                             int lane) {
    float2 acc[NC];
#pragma unroll
    for (int c = 0; c < NC; ++c) acc[c] = make_float2(0.0f, 0.0f);
    for (int b0 = 0; b0 < nbp; b0 += kChunkBlocks) {
        const int nq = min(kChunkBlocks, nbp - b0) / 4;
        const uint32_t slot = co.slot;
        const bool ok = pipe_wait(P, P.full + slot, co.phase, true);
        if (ok) {
            const unsigned char *st = P.ring + (size_t)slot * kStageBytes;
            const uint4 *qs_s = reinterpret_cast<const uint4 *>(st);
            const uint2 *sc_s = reinterpret_cast<const uint2 *>(st + kStageQsBytes);
            const int q0 = (int)((unsigned)(warp * nq) / kConsumerWarps);
            const int q1 = (int)((unsigned)((warp + 1) * nq) / kConsumerWarps);
            for (int q = q0; q < q1; ++q) {
                const uint2 s = sc_s[q * 32 + lane];
                const float2 dw01 = __half22float2(*reinterpret_cast<const __half2 *>(&s.x));
                const float2 dw23 = __half22float2(*reinterpret_cast<const __half2 *>(&s.y));
                const int bq = b0 + q * 4;
#pragma unroll
                for (int jj = 0; jj < 4; jj += 2) {  // blocks in pairs: fewer live sums
                    int sa[NC], sb[NC];
                    block_dots_cols<NC>(co.cb, qs_s[(q * 4 + jj) * 32 + lane], act0, col_off, bq + jj, sa);
                    block_dots_cols<NC>(co.cb, qs_s[(q * 4 + jj + 1) * 32 + lane], act0, col_off, bq + jj + 1, sb);
                    const float2 dw = jj == 0 ? dw01 : dw23;
#pragma unroll
                    for (int c = 0; c < NC; ++c) {
                        const float2 dx2 = *reinterpret_cast<const float2 *>(dx0 + col_off[c] + bq + jj);
                        acc[c] = scale_acc2(acc[c], dw, dx2, sa[c], sb[c]);
                    }
                }
            }
        }
        mbar_arrive(P.empty + slot);  // every consumer thread, after its own reads
        co.advance(P);
    }
#pragma unroll
    for (int c = 0; c < NC; ++c) part[c * 32 + lane] = acc[c].x + acc[c].y;
}

// One column, two columns (one shared expansion, sums in registers over the
// pass) and three or more (pairs per stage) each get their own loop.
__device__ __forceinline__ void group_cols(Consumer &co, const Pipe &P, int nbp, const uint4 *act0, const float *dx0,
                                           const int (&col_off)[kMaxCols], int ncols, float *part, int warp, int lane) {
    if (ncols == 1)
        group_cols_impl<true>(co, P, nbp, act0, dx0, col_off, 1, part, warp, lane);
    else if (ncols == 2)
        group_cols_n<2>(co, P, nbp, act0, dx0, col_off, part, warp, lane);
    else
        group_cols_impl<false>(co, P, nbp, act0, dx0, col_off, ncols, part, warp, lane);
}

// Dynamic shared memory of a pipelined kernel:
//   [full S][empty S][abort][tags S] | ring S x kStageBytes | act ncols x nbp x 32 | dx | part
// part holds nsets partial-sum sets of kConsumerWarps x kMaxCols x 32 floats;
// kernels alternate between two halves item by item, so one barrier per item
// separates the writers of an item from the readers of the item before.
struct PipeSmem {
    Pipe pipe;
    uint4 *act;
    float *dx;
    float *part;  // nsets x kPartSet floats
};

constexpr int kPartSet = kConsumerWarps * kMaxCols * 32;

__host__ __device__ inline size_t pipe_header_bytes(int S) { return ((size_t)20 * S + 4 + 127) / 128 * 128; }

__host__ __device__ inline size_t pipe_smem_bytes(int S, int ncols, int nbp, int nsets) {
    return pipe_header_bytes(S) + (size_t)S * kStageBytes + (size_t)ncols * nbp * 36 +
           (size_t)nsets * kConsumerWarps * kMaxCols * 32 * 4;
}

__device__ __forceinline__ PipeSmem carve_pipe(unsigned char *smem, int S, int ncols, int nbp) {
    PipeSmem L;
    L.pipe.full = reinterpret_cast<uint64_t *>(smem);
    L.pipe.empty = L.pipe.full + S;
    L.pipe.abort = reinterpret_cast<int *>(L.pipe.empty + S);
    L.pipe.tag = L.pipe.abort + 1;
    L.pipe.ring = smem + pipe_header_bytes(S);
    L.pipe.S = S;
    L.act = reinterpret_cast<uint4 *>(L.pipe.ring + (size_t)S * kStageBytes);
    L.dx = reinterpret_cast<float *>(L.act + (size_t)ncols * nbp * 2);
    L.part = L.dx + (size_t)ncols * nbp;
    return L;
}

// Work counter of a persistent kernel: sched[0] next item, sched[1] CTAs
// done.  Called once per CTA after its last fetch; the last CTA resets both
// for the next launch.
__device__ __forceinline__ void sched_exit(unsigned *sched) {
    if (atomicAdd(sched + 1, 1u) == gridDim.x - 1) {
        sched[0] = 0u;
        sched[1] = 0u;
    }
}

// Thread 0 initialises the barriers; all threads must then __syncthreads().
__device__ __forceinline__ void pipe_init(const Pipe &P) {
    if (threadIdx.x == 0) {
        for (int s = 0; s < P.S; ++s) {
            mbar_init(P.full + s, 1);
            mbar_init(P.empty + s, kConsumers);
        }
        *P.abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
}

}  // namespace cbq

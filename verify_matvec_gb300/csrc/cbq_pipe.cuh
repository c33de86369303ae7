// cbq_pipe.cuh -- the weight-stream pipeline of the matvec kernels.
//
// One producer warp per CTA moves the weight stream from HBM into a ring of
// shared-memory stages with 1-D bulk copies (cp.async.bulk, the TMA's
// non-tensor form), each stage completing on an mbarrier.  Eight consumer
// warps wait for a stage, expand and dot it from shared memory, and release it
// through a second mbarrier.  Every stage is 18 KB (16 KB of index fields,
// 2 KB of scales) in one of two formats:
//   format A: 32 block columns of one 32-row group (two bulk copies); warp w
//             takes the 4-block quad w;
//   format B: 16 block columns of two 32-row groups -- the gate and up rows of
//             one SwiGLU group, or two down-projection groups -- (four bulk
//             copies); warp w takes blocks 2w and 2w+1 of both groups, so the
//             two rows of a lane share every activation load.
// Both layouts are contiguous slices of the device layout (cbq_device.cuh).
//
// Work is fetched per CTA: its first item is the CTA index (streamed at once,
// before the kernel waits for the work ahead of it on the stream: weights are
// never written by a call), later ones come from a global counter (atomicAdd;
// the last CTA to exit resets it).  The producer tags every stage with its
// item in a small shared header and closes the stream with a stage tagged -1
// that carries no bytes.
//
// Every wait is bounded: once it has waited kWaitLimitNs (global timer) it
// sets kErrPipeTimeout in the handle's error word and a CTA-wide abort flag;
// the other waits of the CTA then give up too.  Consumers decide at item
// boundaries together (thread 0 reads the next tag and a barrier publishes
// it), so every consumer warp runs the same sequence of stages and barriers
// whatever fails; the producer waits for its own copies in flight before the
// CTA exits.
#pragma once

#include <stdint.h>

#include <cuda_fp16.h>

#include "cbq_device.cuh"

namespace cbq {

constexpr int kConsumerWarps = 8;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kPipeThreads = kConsumers + 32;   // + one producer warp
constexpr int kStageQsBytes = 16384;
constexpr int kStageScBytes = 2048;
constexpr int kStageBytes = kStageQsBytes + kStageScBytes;  // 18,432
constexpr int kChunkA = 32;  // block columns per format-A stage
constexpr int kChunkB = 16;  // block columns per format-B stage (each of two row groups)
// Bounded waits: each poll suspends the warp until the phase completes or
// kWaitHintNs pass (so a waiting warp takes no issue slots from the warps that
// compute); a wait gives up after kWaitLimitNs in all.
constexpr uint32_t kWaitHintNs = 20000;
constexpr uint64_t kWaitLimitNs = 1000000000ull;
constexpr unsigned kErrPipeTimeout = 0x100u;

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n"
        " mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "n"(kWaitHintNs)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

// 1-D bulk copy global -> shared, completing `bytes` of transaction on bar.
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void consumer_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kConsumers) : "memory"); }

// Shared part of the pipeline (carved from dynamic shared memory).
struct Pipe {
    uint32_t *consts;  // kConstWords words: codebook and dp4a seed (read_consts)
    uint32_t full0;    // shared address of full[0]: stage filled (producer arrive + bulk bytes)
    uint32_t empty0;   // shared address of empty[0]: stage released (one arrive per consumer thread)
    int *abort;        // CTA-wide give-up flag
    int *tag;          // [S] item of each stage (-1: end of stream)
    int *next;         // the item consumers take next (published by thread 0)
    unsigned char *ring;
    unsigned *err;     // error word of the handle (global memory)
    int S;
};

// Bounded wait for phase `parity` of the barrier at shared address bar.
// Returns false on timeout or when the CTA already gave up (check_abort).
__device__ __forceinline__ bool pipe_wait(const Pipe &P, uint32_t bar, uint32_t parity, bool check_abort) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    for (;;) {
        if (check_abort && *(volatile int *)P.abort) return false;
        if (mbar_try_wait(bar, parity)) return true;
        if (global_ns() - t0 > kWaitLimitNs) break;
    }
    atomicOr(P.err, kErrPipeTimeout);
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
        if (stopped || (use > 0 && !pipe_wait(P, P.empty0 + 8u * slot, (use - 1) & 1u, true))) {
            stopped = true;
            return false;
        }
        return true;
    }

    // Format A: the stages of one 32-row group over blocks [b0, b1) of its
    // pass (qs_g, sc_g: the group's index and scale streams), tagged `tag`.
    __device__ __forceinline__ void group_a(const Pipe &P, const uint4 *qs_g, const uint2 *sc_g, int b0, int b1,
                                            int tag) {
        for (int b = b0; b < b1 && !stopped; b += kChunkA) {
            const int nblk = min(kChunkA, b1 - b);
            uint32_t slot;
            if (!claim(P, slot)) break;
            const uint32_t dst = smem_addr(P.ring) + slot * (uint32_t)kStageBytes;
            const uint32_t bar = P.full0 + 8u * slot;
            const uint32_t bq = (uint32_t)nblk * 512u, bs = (uint32_t)nblk / 4u * 256u;
            P.tag[slot] = tag;
            mbar_expect_tx(bar, bq + bs);
            bulk_g2s(dst, qs_g + (size_t)b * 32, bq, bar);
            bulk_g2s(dst + kStageQsBytes, sc_g + (size_t)(b / 4) * 32, bs, bar);
            ++it;
        }
    }

    // Format B: the stages of two 32-row groups (a, and b unless qs_b is
    // null) over blocks [0, nbp), tagged `tag`.
    __device__ __forceinline__ void group_b(const Pipe &P, const uint4 *qs_a, const uint2 *sc_a, const uint4 *qs_b,
                                            const uint2 *sc_b, int nbp, int tag) {
        for (int b = 0; b < nbp && !stopped; b += kChunkB) {
            const int nblk = min(kChunkB, nbp - b);
            uint32_t slot;
            if (!claim(P, slot)) break;
            const uint32_t dst = smem_addr(P.ring) + slot * (uint32_t)kStageBytes;
            const uint32_t bar = P.full0 + 8u * slot;
            const uint32_t bq = (uint32_t)nblk * 512u, bs = (uint32_t)nblk / 4u * 256u;
            P.tag[slot] = tag;
            mbar_expect_tx(bar, qs_b ? 2u * (bq + bs) : bq + bs);
            bulk_g2s(dst, qs_a + (size_t)b * 32, bq, bar);
            bulk_g2s(dst + kStageQsBytes, sc_a + (size_t)(b / 4) * 32, bs, bar);
            if (qs_b) {
                bulk_g2s(dst + kStageQsBytes / 2, qs_b + (size_t)b * 32, bq, bar);
                bulk_g2s(dst + kStageQsBytes + kStageScBytes / 2, sc_b + (size_t)(b / 4) * 32, bs, bar);
            }
            ++it;
        }
    }

    // Give-up test mode only: claim a slot and tag it, but never fill it (the
    // consumers' bounded wait for it runs out).
    __device__ __forceinline__ void tag_only(const Pipe &P, int tag) {
        uint32_t slot;
        if (!claim(P, slot)) return;
        P.tag[slot] = tag;
        ++it;
    }

    // End of stream: a stage tagged -1 with no bytes.
    __device__ __forceinline__ void finish(const Pipe &P) {
        uint32_t slot;
        if (!claim(P, slot)) {
            *(volatile int *)P.abort = 1;  // consumers must not wait for it
            return;
        }
        P.tag[slot] = -1;
        mbar_arrive(P.full0 + 8u * slot);
        ++it;
    }

    // Wait for the copies still in flight (the last S issued stages) so the
    // CTA never exits while the TMA writes into its shared memory.  Each wait
    // is bounded like every other; a copy from mapped memory always completes,
    // so the limit is only a guard against a broken device.
    __device__ __forceinline__ void drain(const Pipe &P) {
        const uint32_t first = it > (uint32_t)P.S ? it - P.S : 0u;
        for (uint32_t k = first; k < it; ++k) pipe_wait(P, P.full0 + 8u * (k % P.S), (k / P.S) & 1u, false);
    }
};

// Consumer side: the same sequence of stages, advanced in lock step (slot,
// phase parity and the slot's addresses kept incrementally).
struct Consumer {
    uint32_t slot = 0, phase = 0;
    uint32_t full, empty;       // barrier addresses of the current slot
    const unsigned char *st;    // the current slot's stage
    Codebook cb;

    __device__ __forceinline__ explicit Consumer(const Pipe &P)
        : full(P.full0), empty(P.empty0), st(P.ring), cb(read_consts(P.consts)) {}

    __device__ __forceinline__ bool wait(const Pipe &P) { return pipe_wait(P, full, phase, true); }

    // Release the current stage (every consumer thread, after its own reads)
    // and move to the next slot.
    __device__ __forceinline__ void release(const Pipe &P) {
        mbar_arrive(empty);
        if (++slot == (uint32_t)P.S) {
            slot = 0;
            phase ^= 1u;
            full = P.full0;
            empty = P.empty0;
            st = P.ring;
        } else {
            full += 8u;
            empty += 8u;
            st += kStageBytes;
        }
    }

    // The item of the next stage, the same for every consumer warp: thread 0
    // waits for the stage and reads its tag (-1 at the end of the stream or
    // after a give-up), a consumer barrier publishes it.  The stage is not
    // consumed.  Must be called by all consumer threads, with at least one
    // consumer barrier between two calls (every item ends with one), so no
    // warp still reads P.next when thread 0 rewrites it.
    __device__ __forceinline__ int next_item(const Pipe &P) {
        if (threadIdx.x == 0) *P.next = wait(P) ? *(volatile int *)(P.tag + slot) : -1;
        consumer_sync();
        return *(volatile int *)P.next;
    }
};

// ------------------------------------------------------ format A sweeps ---

// One 4-block quad of one row (this lane) for NC columns: the quad's index
// words at qs[0], qs[32], qs[64], qs[96]; its four fp16 scales in s; the
// activations block-major at act (block j of column c at act[(j*NC + c)*2]);
// the activation scales as float2 pairs at dxp (blocks 0-1 of column c at
// dxp[c], blocks 2-3 at dxp[NC + c]).
template <int NC>
__device__ __forceinline__ void quad_a(const Codebook &cb, const uint4 *qs, uint2 s, const uint4 *act,
                                       const float2 *dxp, float2 acc[NC]) {
    const float2 dw01 = __half22float2(*reinterpret_cast<const __half2 *>(&s.x));
    const float2 dw23 = __half22float2(*reinterpret_cast<const __half2 *>(&s.y));
    uint4 w[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) w[j] = qs[j * 32];
#pragma unroll
    for (int jj = 0; jj < 4; jj += 2) {  // blocks in pairs: fewer live sums
        int sa[NC], sb[NC];
        block_dots<NC>(cb, w[jj], act + jj * NC * 2, sa);
        block_dots<NC>(cb, w[jj + 1], act + (jj + 1) * NC * 2, sb);
        const float2 dw = jj == 0 ? dw01 : dw23;
#pragma unroll
        for (int c = 0; c < NC; ++c) acc[c] = scale_acc2(acc[c], dw, dxp[(jj >> 1) * NC + c], sa[c], sb[c]);
    }
}

// The stages of one format-A pass over blocks [b0, b1) for NC columns staged
// block-major (act, dxp as quad_a, indexed from block 0), summed into acc.
template <int NC>
__device__ __forceinline__ void sweep_a(Consumer &co, const Pipe &P, int b0, int b1, const uint4 *act,
                                        const float2 *dxp, float2 acc[NC], int warp, int lane) {
    const uint4 *a = act + (size_t)(b0 + 4 * warp) * NC * 2;
    const float2 *d = dxp + (size_t)((b0 + 4 * warp) >> 1) * NC;
    for (int b = b0; b < b1; b += kChunkA) {
        const bool ok = co.wait(P);
        if (ok && b + 4 * warp < b1) {
            const uint4 *qs = reinterpret_cast<const uint4 *>(co.st) + warp * 128 + lane;
            const uint2 s = reinterpret_cast<const uint2 *>(co.st + kStageQsBytes)[warp * 32 + lane];
            quad_a<NC>(co.cb, qs, s, a, d, acc);
        }
        co.release(P);
        a += kChunkA * NC * 2;
        d += kChunkA / 2 * NC;
    }
}

// ------------------------------------------------------ format B sweeps ---
// Columns are staged one after another (block b of the column at offset o
// has its two words at act0[2*(o + b)] and its scale at dx0[o + b]); col_off
// holds each column's offset o.  Each lane owns row `lane` of both row groups
// (set 0, set 1) of the stage.

// The fp16 scale pair of this warp's two blocks in row set r of the stage.
__device__ __forceinline__ float2 stage_dw_b(const unsigned char *st, int r, int warp, int lane) {
    const uint2 s = reinterpret_cast<const uint2 *>(st + kStageQsBytes + r * (kStageScBytes / 2))[(warp >> 1) * 32 + lane];
    const uint32_t h = (warp & 1) ? s.y : s.x;
    return __half22float2(*reinterpret_cast<const __half2 *>(&h));
}

// One column: the two-word expansion, running sums of both row sets in
// registers over the pass; written to part[r*kMaxCols*32 + lane] at its end.
__device__ __forceinline__ void sweep_b1(Consumer &co, const Pipe &P, int nbp, const uint4 *act0, const float *dx0,
                                         int off, float *part, bool live, int warp, int lane) {
    float2 acc0 = make_float2(0.0f, 0.0f), acc1 = make_float2(0.0f, 0.0f);
    const uint4 *a = act0 + 2 * (off + 2 * warp);
    const float *d = dx0 + off + 2 * warp;
    for (int b = 0; b < nbp; b += kChunkB) {
        const bool ok = co.wait(P);
        if (ok && live && b + 2 * warp < nbp) {
            const uint4 *q0 = reinterpret_cast<const uint4 *>(co.st) + warp * 64 + lane;
            const uint4 *q1 = q0 + kChunkB * 32;
            const float2 dw0 = stage_dw_b(co.st, 0, warp, lane), dw1 = stage_dw_b(co.st, 1, warp, lane);
            const float2 dx2 = *reinterpret_cast<const float2 *>(d);
            int s0a, s0b, s1a, s1b;
            block_dots_2rows(co.cb, q0[0], q1[0], a, s0a, s1a);
            block_dots_2rows(co.cb, q0[32], q1[32], a + 2, s0b, s1b);
            acc0 = scale_acc2(acc0, dw0, dx2, s0a, s0b);
            acc1 = scale_acc2(acc1, dw1, dx2, s1a, s1b);
        }
        co.release(P);
        a += 2 * kChunkB;
        d += kChunkB;
    }
    part[lane] = acc0.x + acc0.y;
    part[kMaxCols * 32 + lane] = acc1.x + acc1.y;
}

// Two columns c0, c1 sharing one exact expansion per index word, both row
// sets; sums in registers over the pass, written to part[(r*kMaxCols + c)*32
// + lane].  With acc_smem the stage sums are added to part instead (the pass
// then sweeps other columns in between; first == true starts the sums).
__device__ __forceinline__ void pair_b_stage(const Codebook &cb, const unsigned char *st, const uint4 *act0,
                                             const float *dx0, int o0, int o1, int bq, float2 acc[2][2], int warp,
                                             int lane) {
    const uint4 *q0 = reinterpret_cast<const uint4 *>(st) + warp * 64 + lane;
    const uint4 *q1 = q0 + kChunkB * 32;
    const float2 dw0 = stage_dw_b(st, 0, warp, lane), dw1 = stage_dw_b(st, 1, warp, lane);
    const int off[2] = {o0, o1};
    int s0[2][2], s1[2][2];  // [block][column]
#pragma unroll
    for (int j = 0; j < 2; ++j) block_dots_2rows_cols2(cb, q0[32 * j], q1[32 * j], act0, off, bq + j, s0[j], s1[j]);
#pragma unroll
    for (int c = 0; c < 2; ++c) {
        const float2 dx2 = *reinterpret_cast<const float2 *>(dx0 + off[c] + bq);
        acc[0][c] = scale_acc2(acc[0][c], dw0, dx2, s0[0][c], s0[1][c]);
        acc[1][c] = scale_acc2(acc[1][c], dw1, dx2, s1[0][c], s1[1][c]);
    }
}

__device__ __forceinline__ void sweep_b2(Consumer &co, const Pipe &P, int nbp, const uint4 *act0, const float *dx0,
                                         int o0, int o1, float *part, bool live, int warp, int lane) {
    float2 acc[2][2] = {{make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f)},
                        {make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f)}};
    for (int b = 0; b < nbp; b += kChunkB) {
        const bool ok = co.wait(P);
        if (ok && live && b + 2 * warp < nbp) pair_b_stage(co.cb, co.st, act0, dx0, o0, o1, b + 2 * warp, acc, warp, lane);
        co.release(P);
    }
#pragma unroll
    for (int r = 0; r < 2; ++r)
#pragma unroll
        for (int c = 0; c < 2; ++c) part[(r * kMaxCols + c) * 32 + lane] = acc[r][c].x + acc[r][c].y;
}

// Three or more columns: at every stage the columns two at a time (an odd
// last one alone) with the stage sums added to part, so the registers stay
// those of two columns while the weight stream is still read once.
__device__ __forceinline__ void sweep_bn(Consumer &co, const Pipe &P, int nbp, const uint4 *act0, const float *dx0,
                                         const int (&col_off)[kMaxCols], int ncols, float *part, bool live, int warp,
                                         int lane) {
    for (int b = 0; b < nbp; b += kChunkB) {
        const bool ok = co.wait(P);
        const int bq = b + 2 * warp;
        if (ok && live && bq < nbp) {
            for (int c = 0; c < ncols; c += 2) {
                float2 acc[2][2] = {{make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f)},
                                    {make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f)}};
                const int o0 = pick(col_off, c);
                if (c + 1 < ncols) {
                    pair_b_stage(co.cb, co.st, act0, dx0, o0, pick(col_off, c + 1), bq, acc, warp, lane);
                } else {
                    const uint4 *q0 = reinterpret_cast<const uint4 *>(co.st) + warp * 64 + lane;
                    const uint4 *q1 = q0 + kChunkB * 32;
                    const float2 dw0 = stage_dw_b(co.st, 0, warp, lane), dw1 = stage_dw_b(co.st, 1, warp, lane);
                    const uint4 *a = act0 + 2 * (o0 + bq);
                    const float2 dx2 = *reinterpret_cast<const float2 *>(dx0 + o0 + bq);
                    int s0a, s0b, s1a, s1b;
                    block_dots_2rows(co.cb, q0[0], q1[0], a, s0a, s1a);
                    block_dots_2rows(co.cb, q0[32], q1[32], a + 2, s0b, s1b);
                    acc[0][0] = scale_acc2(acc[0][0], dw0, dx2, s0a, s0b);
                    acc[1][0] = scale_acc2(acc[1][0], dw1, dx2, s1a, s1b);
                }
#pragma unroll
                for (int r = 0; r < 2; ++r)
#pragma unroll
                    for (int i = 0; i < 2; ++i) {
                        if (c + i >= ncols) continue;
                        float *dst = part + (r * kMaxCols + c + i) * 32 + lane;
                        *dst = (b == 0 ? 0.0f : *dst) + (acc[r][i].x + acc[r][i].y);
                    }
            }
        } else if (b == 0) {  // no block of this warp in the first stage: start the sums at zero
            for (int c = 0; c < ncols; ++c) {
                part[c * 32 + lane] = 0.0f;
                part[(kMaxCols + c) * 32 + lane] = 0.0f;
            }
        }
        co.release(P);
    }
}

// One item pass of format B for the ncols columns at col_off: each warp's
// sums go to its slice part (row set r, column c at part[(r*kMaxCols + c)*32
// + lane]).  One column, two columns (one shared expansion, sums in
// registers) and three or more (pairs per stage) each get their own loop.
// live == false runs the stage waits and releases without computing.
__device__ __forceinline__ void sweep_b(Consumer &co, const Pipe &P, int nbp, const uint4 *act0, const float *dx0,
                                        const int (&col_off)[kMaxCols], int ncols, float *part, bool live, int warp,
                                        int lane) {
    if (ncols == 1)
        sweep_b1(co, P, nbp, act0, dx0, col_off[0], part, live, warp, lane);
    else if (ncols == 2)
        sweep_b2(co, P, nbp, act0, dx0, col_off[0], col_off[1], part, live, warp, lane);
    else
        sweep_bn(co, P, nbp, act0, dx0, col_off, ncols, part, live, warp, lane);
}

// Dynamic shared memory of a pipelined kernel:
//   [consts][full S][empty S][abort][next][tags S] | ring S x kStageBytes | act | dx | part
// act holds act_blocks staged blocks (two uint4 each), dx their scales; part
// holds nsets partial-sum sets of kPartSet floats.
struct PipeSmem {
    Pipe pipe;
    uint4 *act;
    float *dx;
    float *part;
};

constexpr int kConstWords = 8;
constexpr int kPartSetA = kConsumerWarps * kMaxCols * 32;      // format A: [warp][column][lane]
constexpr int kPartSetB = kConsumerWarps * 2 * kMaxCols * 32;  // format B: [warp][row set][column][lane]

__host__ __device__ inline size_t pipe_header_bytes(int S) {
    return ((size_t)4 * kConstWords + 20 * (size_t)S + 8 + 127) / 128 * 128;
}

__host__ __device__ inline size_t pipe_smem_bytes(int S, int act_blocks, int part_floats) {
    return pipe_header_bytes(S) + (size_t)S * kStageBytes + (size_t)act_blocks * 36 + (size_t)part_floats * 4;
}

__device__ __forceinline__ PipeSmem carve_pipe(unsigned char *smem, int S, int act_blocks, unsigned *err) {
    PipeSmem L;
    L.pipe.consts = reinterpret_cast<uint32_t *>(smem);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + 4 * kConstWords);
    L.pipe.full0 = smem_addr(bars);
    L.pipe.empty0 = smem_addr(bars + S);
    L.pipe.abort = reinterpret_cast<int *>(bars + 2 * S);
    L.pipe.next = L.pipe.abort + 1;
    L.pipe.tag = L.pipe.abort + 2;
    L.pipe.ring = smem + pipe_header_bytes(S);
    L.pipe.err = err;
    L.pipe.S = S;
    L.act = reinterpret_cast<uint4 *>(L.pipe.ring + (size_t)S * kStageBytes);
    L.dx = reinterpret_cast<float *>(L.act + (size_t)act_blocks * 2);
    L.part = L.dx + act_blocks;
    return L;
}

// Work counter of a persistent kernel: sched[0] dynamic items taken, sched[1]
// CTAs done.  Called once per CTA after its last fetch; the last CTA resets
// both for the next launch.
__device__ __forceinline__ void sched_exit(unsigned *sched) {
    if (atomicAdd(sched + 1, 1u) == gridDim.x - 1) {
        sched[0] = 0u;
        sched[1] = 0u;
    }
}

// Thread 0 writes the constants and initialises the barriers; all threads
// must then pass a __syncthreads() before using the pipe.
__device__ __forceinline__ void pipe_init(const Pipe &P) {
    if (threadIdx.x == 0) {
        write_consts(P.consts);
        for (int s = 0; s < P.S; ++s) {
            mbar_init(P.full0 + 8u * s, 1);
            mbar_init(P.empty0 + 8u * s, kConsumers);
        }
        *P.abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
}

}  // namespace cbq

// cbq_pipe.cuh -- warp-specialised weight-stream pipeline of the matvec kernels.
//
// A CTA has three roles:
//   - a producer warp (one active lane) moves weight chunks from global memory
//     into a ring of shared-memory stages with 1-D bulk copies (cp.async.bulk,
//     the TMA's non-tensor form), each stage completing on an mbarrier; in the
//     routed-expert kernel a stage also carries the activation slice its
//     blocks are dotted with;
//   - eight consumer warps wait for a stage, expand and dot it, release it
//     through a second mbarrier, and at the end of a work item write their
//     partial sums into one of two shared-memory sets;
//   - an epilogue warp adds the eight partial sums of each item and finishes
//     it (outputs, or SwiGLU, requantization and counters), then frees the set.
// Consumer warps never wait for one another: each reads an item's tag from
// the item's first stage, and the only barrier among them is the one after
// the activations are staged at the start.
//
// A stage is one chunk of the device layout (cbq_internal.h): 16 block
// columns of a pair of 32-row groups -- the gate and up rows of one SwiGLU
// group, or two down-projection or dense groups -- with their scales, one
// contiguous span brought in by one bulk copy; in the routed-expert kernel it
// is followed by the activation slice of those 16 blocks (a second copy).
// Warp w takes blocks 2w and 2w+1 of both groups, so the two rows of a lane
// share every activation load.
//
// Work is fetched per CTA: its first item is the CTA index, later ones come
// from a global counter (atomicAdd) whose result is fetched one item ahead.
// The producer tags every stage with its item and closes the stream with a
// stage tagged -1 that carries no bytes.
//
// Every wait is bounded: once it has waited kWaitLimitNs (global timer) it
// sets kErrPipeTimeout in the handle's error word and a CTA-wide abort flag,
// after which the other waits of the CTA give up at once.  A role that gives
// up leaves its loop; no barrier inside the loops can be left waiting, and the
// producer waits for its own copies in flight before the CTA exits.
#pragma once

#include <stdint.h>

#include <cuda_fp16.h>

#include "cbq_device.cuh"
#include "cbq_internal.h"

namespace cbq {

constexpr int kConsumerWarps = 8;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kEpilogueWarp = kConsumerWarps;      // warp 8
constexpr int kProducerWarp = kConsumerWarps + 1;  // warp 9
constexpr int kPipeThreads = (kConsumerWarps + 2) * 32;
constexpr int kStageWeightBytes = kChunkBytes;  // 18,432: the weights of a full chunk
// A stage with an activation slice: the weights, then up to kChunk x kMaxCols
// staged blocks (32 bytes each) and their scales (4 bytes each).
constexpr int kStageActBytes = kChunk * kMaxCols * 36;
constexpr int kStageBytesAct = kStageWeightBytes + kStageActBytes;  // 21,312
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
    uint32_t *consts;     // kConstWords words: codebook and dp4a seed (read_consts)
    uint32_t full0;       // shared address of full[0]: stage filled (producer arrive + bulk bytes)
    uint32_t empty0;      // shared address of empty[0]: stage released (one arrive per consumer thread)
    uint32_t setfull0;    // shared address of setfull[0]: partial sums written (one arrive per consumer thread)
    uint32_t setempty0;   // shared address of setempty[0]: set read (one arrive per epilogue lane)
    int *abort;           // CTA-wide give-up flag
    int *tag;             // [S] item of each stage (-1: end of stream)
    unsigned char *ring;  // S stages of stage_bytes
    unsigned char *sets;  // nsets sets of set_bytes: [item tag (16 bytes)][partial sums]
    unsigned *err;        // error word of the handle (global memory)
    int S;
    uint32_t stage_bytes;
    uint32_t set_bytes;
    uint32_t nsets;       // 1 or 2
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

// Source of a stage's activation slice: `cols` columns in the chunked
// activation layout (act_chunk_offset); the stage of chunk c copies its 36 *
// cols * nblk bytes.  cols == 0: no slice.
struct ActSlice {
    const int8_t *base;
    int cols;
};

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

    // One stage: claim its slot, tag it, expect its bytes (weights and, with
    // act.cols, its slice) and issue its weight copy.  False when stopped.
    __device__ __forceinline__ bool issue_weights(const Pipe &P, const uint8_t *w, int nbp, int c, int tag,
                                                  const ActSlice &act, uint32_t &dst, uint32_t &bar) {
        const int nblk = chunk_blocks(nbp, c);
        uint32_t slot;
        if (!claim(P, slot)) return false;
        dst = smem_addr(P.ring) + slot * P.stage_bytes;
        bar = P.full0 + 8u * slot;
        const uint32_t bw = (uint32_t)nblk * (2 * kBlockBytes), ba = (uint32_t)(nblk * act.cols) * 36u;
        P.tag[slot] = tag;
        mbar_expect_tx(bar, bw + ba);
        bulk_g2s(dst, w + (size_t)c * kChunkBytes, bw, bar);
        ++it;
        return true;
    }

    __device__ __forceinline__ void issue_act(const Pipe &P, int nbp, int c, const ActSlice &act, uint32_t dst,
                                              uint32_t bar) {
        const uint32_t ba = (uint32_t)(chunk_blocks(nbp, c) * act.cols) * 36u;
        bulk_g2s(dst + kStageWeightBytes, act.base + act_chunk_offset(c, act.cols), ba, bar);
    }

    // The stages of chunks [c0, c1) of a pass over a pair (its bytes at w,
    // nbp blocks), tagged `tag`, each with its chunk of `act`.  When
    // dep.all_ready(c0, c1) finds every slice readable (one batch of polls),
    // each stage's two copies go out together.  Otherwise the weight copies
    // run ahead of the slices: a slice is issued, in order, once dep.ready(c)
    // (a poll) says it may be read, and waited for (dep.wait(c), bounded;
    // false gives up and stops the producer) only before a slot it would
    // block is claimed and at the end of the pass.
    template <typename Dep>
    __device__ __forceinline__ void pass(const Pipe &P, const uint8_t *w, int nbp, int c0, int c1, int tag,
                                         const ActSlice &act, Dep &dep) {
        if (!act.cols || dep.all_ready(c0, c1)) {
            for (int c = c0; c < c1 && !stopped; ++c) {
                uint32_t dst, bar;
                if (!issue_weights(P, w, nbp, c, tag, act, dst, bar)) break;
                if (act.cols) issue_act(P, nbp, c, act, dst, bar);
            }
            return;
        }
        int owed = c0;              // first chunk whose slice is not issued yet
        uint32_t owed_it = it;      // its stage
        auto settle = [&](int upto, bool must) -> bool {
            while (owed < upto) {
                if (!dep.ready(owed)) {
                    if (!must) return true;
                    if (!dep.wait(owed)) return false;
                }
                const uint32_t slot = owed_it % (uint32_t)P.S;
                issue_act(P, nbp, owed, act, smem_addr(P.ring) + slot * P.stage_bytes, P.full0 + 8u * slot);
                ++owed;
                ++owed_it;
            }
            return true;
        };
        for (int c = c0; c < c1 && !stopped; ++c) {
            // chunk c's slot held chunk c - S of this pass, if any: its slice
            // must be out before the consumers can free the slot
            if (!settle(c - P.S + 1, true)) {
                stopped = true;
                *(volatile int *)P.abort = 1;
                break;
            }
            uint32_t dst, bar;
            if (!issue_weights(P, w, nbp, c, tag, act, dst, bar)) break;
            settle(c + 1, false);
        }
        if (!stopped && !settle(c1, true)) {
            // a slice that will never be ready: stop (its stage stays incomplete)
            stopped = true;
            *(volatile int *)P.abort = 1;
        }
    }

    // A pass whose slices are always ready (or that has none).
    struct NoDep {
        __device__ __forceinline__ bool all_ready(int, int) const { return true; }
        __device__ __forceinline__ bool ready(int) const { return true; }
        __device__ __forceinline__ bool wait(int) const { return true; }
    };

    __device__ __forceinline__ void pass(const Pipe &P, const uint8_t *w, int nbp, int c0, int c1, int tag) {
        NoDep nd;
        pass(P, w, nbp, c0, c1, tag, ActSlice{nullptr, 0}, nd);
    }

    // A pass over one group (half h) of a pair (its bytes at w, nch chunks):
    // each stage holds that group's part of two consecutive chunks (its index
    // fields and scales, nblk * kBlockBytes contiguous bytes from h * nblk *
    // kBlockBytes in each chunk), one after the other, so a stage carries as
    // many blocks of work as a stage of a whole pair.
    __device__ __forceinline__ void pass_single(const Pipe &P, const uint8_t *w, int nbp, int nch, int h, int tag) {
        for (int c = 0; c < nch && !stopped; c += 2) {
            uint32_t slot;
            if (!claim(P, slot)) break;
            const uint32_t dst = smem_addr(P.ring) + slot * P.stage_bytes, bar = P.full0 + 8u * slot;
            const int n0 = chunk_blocks(nbp, c), n1 = c + 1 < nch ? chunk_blocks(nbp, c + 1) : 0;
            const uint32_t b0 = (uint32_t)n0 * kBlockBytes, b1 = (uint32_t)n1 * kBlockBytes;
            P.tag[slot] = tag;
            mbar_expect_tx(bar, b0 + b1);
            bulk_g2s(dst, w + (size_t)c * kChunkBytes + (size_t)h * b0, b0, bar);
            if (n1) bulk_g2s(dst + b0, w + (size_t)(c + 1) * kChunkBytes + (size_t)h * b1, b1, bar);
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
    // so the limit only guards against a broken device.
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

    // The item of the current stage (after a successful wait).
    __device__ __forceinline__ int tag(const Pipe &P) const { return *(volatile int *)(P.tag + slot); }

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
            st += P.stage_bytes;
        }
    }
};

// The partial-sum sets (one or two), written in turn by the consumers (one
// set per item) and read in the same turn by the epilogue warp.
struct SetWriter {
    uint32_t n = 0;  // items written

    // Wait until set n % nsets is free (the epilogue has read item n - nsets);
    // gives its tag word and partial sums, or returns false on a give-up.
    __device__ __forceinline__ bool acquire(const Pipe &P, int *&tag, float *&part) {
        const uint32_t use = n / P.nsets, k = n - use * P.nsets;
        if (use > 0 && !pipe_wait(P, P.setempty0 + 8u * k, (use - 1) & 1u, true)) return false;
        tag = reinterpret_cast<int *>(P.sets + k * P.set_bytes);
        part = reinterpret_cast<float *>(P.sets + k * P.set_bytes + 16);
        return true;
    }

    // Every consumer thread, after its own writes to the set.
    __device__ __forceinline__ void publish(const Pipe &P) {
        mbar_arrive(P.setfull0 + 8u * (n % P.nsets));
        ++n;
    }
};

struct SetReader {
    uint32_t n = 0;  // items read

    __device__ __forceinline__ bool wait(const Pipe &P, const int *&tag, const float *&part) {
        const uint32_t use = n / P.nsets, k = n - use * P.nsets;
        if (!pipe_wait(P, P.setfull0 + 8u * k, use & 1u, true)) return false;
        tag = reinterpret_cast<const int *>(P.sets + k * P.set_bytes);
        part = reinterpret_cast<const float *>(P.sets + k * P.set_bytes + 16);
        return true;
    }

    // Every epilogue lane, after its own reads of the set.
    __device__ __forceinline__ void release(const Pipe &P) {
        mbar_arrive(P.setempty0 + 8u * (n % P.nsets));
        ++n;
    }
};

// ------------------------------------------------------------- sweeps ---
// The activations of a stage's blocks are staged block-major: block j (0..15
// of the stage) of column slot x has its two words at act[(j*stride + x)*2]
// and its scale at dx[((j>>1)*stride + x)*2 + (j&1)] (the scales of a block
// pair side by side).  ActView gives, per stage, where block 0 of the stage
// sits; col[] holds each column's slot x.  Each lane owns row `lane` of both
// groups (row sets 0 and 1) of the stage.
struct ActView {
    const uint4 *act;  // persistent staging (stage_act == false) indexed from block 0
    const float *dx;
    int stride;        // column slots per block
    bool stage_act;    // the stage carries its own slice (block 0 of the stage at its start)
};

__device__ __forceinline__ void stage_act_ptrs(const ActView &V, const unsigned char *st, int b, int nblk,
                                               const uint4 *&a, const float *&d) {
    if (V.stage_act) {
        a = reinterpret_cast<const uint4 *>(st + kStageWeightBytes);
        d = reinterpret_cast<const float *>(st + kStageWeightBytes + (size_t)nblk * V.stride * 32);
    } else {
        a = V.act + (size_t)b * V.stride * 2;
        d = V.dx + (size_t)b * V.stride;
    }
}

// The index fields of this lane's rows for this warp's first block in a
// stage of nblk blocks (row set 0 at q0[0], q0[32]; row set 1 likewise at q1).
__device__ __forceinline__ void stage_fields(const unsigned char *st, int nblk, int warp, int lane, const uint4 *&q0,
                                             const uint4 *&q1) {
    q0 = reinterpret_cast<const uint4 *>(st) + warp * 64 + lane;
    q1 = reinterpret_cast<const uint4 *>(st + (size_t)nblk * kBlockBytes) + warp * 64 + lane;
}

// The fp16 scale pair of this warp's two blocks in row set r of a stage of
// nblk blocks.
__device__ __forceinline__ float2 stage_dw(const unsigned char *st, int nblk, int r, int warp, int lane) {
    const uint2 s = reinterpret_cast<const uint2 *>(st + (size_t)(r * nblk) * kBlockBytes + (size_t)nblk * 512)
        [(warp >> 1) * 32 + lane];
    const uint32_t h = (warp & 1) ? s.y : s.x;
    return __half22float2(*reinterpret_cast<const __half2 *>(&h));
}

// One column at slot x: the two-word expansion; running sums of both row
// sets in registers over the pass, written to part[r*kMaxCols*32 + lane].
__device__ __forceinline__ bool sweep_b1(Consumer &co, const Pipe &P, int b0, int b1, int nbp, const ActView &V, int x,
                                         float *part, int warp, int lane) {
    float2 acc0 = make_float2(0.0f, 0.0f), acc1 = make_float2(0.0f, 0.0f);
    const int j = 2 * warp;  // this warp's first block in a stage
    bool ok = true;
    for (int b = b0; b < b1; b += kChunk) {
        if (b > b0) ok = ok && co.wait(P);
        const int nblk = min(kChunk, nbp - b);
        if (ok && j < nblk) {
            const uint4 *a, *q0, *q1;
            const float *d;
            stage_act_ptrs(V, co.st, b, nblk, a, d);
            stage_fields(co.st, nblk, warp, lane, q0, q1);
            const float2 dw0 = stage_dw(co.st, nblk, 0, warp, lane), dw1 = stage_dw(co.st, nblk, 1, warp, lane);
            const float2 dx2 = *reinterpret_cast<const float2 *>(d + ((j >> 1) * V.stride + x) * 2);
            int s0a, s0b, s1a, s1b;
            block_dots_2rows(co.cb, q0[0], q1[0], a + (j * V.stride + x) * 2, s0a, s1a);
            block_dots_2rows(co.cb, q0[32], q1[32], a + ((j + 1) * V.stride + x) * 2, s0b, s1b);
            acc0 = scale_acc2(acc0, dw0, dx2, s0a, s0b);
            acc1 = scale_acc2(acc1, dw1, dx2, s1a, s1b);
        }
        co.release(P);
    }
    part[lane] = acc0.x + acc0.y;
    part[kMaxCols * 32 + lane] = acc1.x + acc1.y;
    return ok;
}

// Columns at slots x0, x1 sharing one exact expansion per index word, both row
// sets, this warp's two blocks of the current stage, added into acc[r][c].
__device__ __forceinline__ void pair_stage(const Codebook &cb, const unsigned char *st, int nblk, const uint4 *a,
                                           const float *d, int stride, int x0, int x1, float2 acc[2][2], int warp,
                                           int lane) {
    const int j = 2 * warp;
    const uint4 *q0, *q1;
    stage_fields(st, nblk, warp, lane, q0, q1);
    const float2 dw0 = stage_dw(st, nblk, 0, warp, lane), dw1 = stage_dw(st, nblk, 1, warp, lane);
    int s0[2][2], s1[2][2];  // [block][column]
#pragma unroll
    for (int jj = 0; jj < 2; ++jj)
        block_dots_2rows_cols2(cb, q0[32 * jj], q1[32 * jj], a + ((j + jj) * stride + x0) * 2,
                               a + ((j + jj) * stride + x1) * 2, s0[jj], s1[jj]);
    const int xs[2] = {x0, x1};
#pragma unroll
    for (int c = 0; c < 2; ++c) {
        const float2 dx2 = *reinterpret_cast<const float2 *>(d + ((j >> 1) * stride + xs[c]) * 2);
        acc[0][c] = scale_acc2(acc[0][c], dw0, dx2, s0[0][c], s0[1][c]);
        acc[1][c] = scale_acc2(acc[1][c], dw1, dx2, s1[0][c], s1[1][c]);
    }
}

// Two columns: sums in registers over the pass.
__device__ __forceinline__ bool sweep_b2(Consumer &co, const Pipe &P, int b0, int b1, int nbp, const ActView &V,
                                         int x0, int x1, float *part, int warp, int lane) {
    float2 acc[2][2] = {{make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f)},
                        {make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f)}};
    bool ok = true;
    for (int b = b0; b < b1; b += kChunk) {
        if (b > b0) ok = ok && co.wait(P);
        const int nblk = min(kChunk, nbp - b);
        if (ok && 2 * warp < nblk) {
            const uint4 *a;
            const float *d;
            stage_act_ptrs(V, co.st, b, nblk, a, d);
            pair_stage(co.cb, co.st, nblk, a, d, V.stride, x0, x1, acc, warp, lane);
        }
        co.release(P);
    }
#pragma unroll
    for (int r = 0; r < 2; ++r)
#pragma unroll
        for (int c = 0; c < 2; ++c) part[(r * kMaxCols + c) * 32 + lane] = acc[r][c].x + acc[r][c].y;
    return ok;
}

// Three or more columns: at every stage the columns two at a time (an odd
// last one alone) with the stage sums added to part, so the registers stay
// those of two columns while the weight stream is still read once.
__device__ __forceinline__ bool sweep_bn(Consumer &co, const Pipe &P, int b0, int b1, int nbp, const ActView &V,
                                         const int (&col)[kMaxCols], int ncols, float *part, int warp, int lane) {
    for (int c = 0; c < ncols; ++c) {
        part[c * 32 + lane] = 0.0f;
        part[(kMaxCols + c) * 32 + lane] = 0.0f;
    }
    const int j = 2 * warp;
    bool ok = true;
    for (int b = b0; b < b1; b += kChunk) {
        if (b > b0) ok = ok && co.wait(P);
        const int nblk = min(kChunk, nbp - b);
        if (ok && j < nblk) {
            const uint4 *a;
            const float *d;
            stage_act_ptrs(V, co.st, b, nblk, a, d);
            for (int c = 0; c < ncols; c += 2) {
                float2 acc[2][2] = {{make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f)},
                                    {make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f)}};
                const int x0 = pick(col, c);
                if (c + 1 < ncols) {
                    pair_stage(co.cb, co.st, nblk, a, d, V.stride, x0, pick(col, c + 1), acc, warp, lane);
                } else {
                    const uint4 *q0, *q1;
                    stage_fields(co.st, nblk, warp, lane, q0, q1);
                    const float2 dw0 = stage_dw(co.st, nblk, 0, warp, lane), dw1 = stage_dw(co.st, nblk, 1, warp, lane);
                    const float2 dx2 = *reinterpret_cast<const float2 *>(d + ((j >> 1) * V.stride + x0) * 2);
                    int s0a, s0b, s1a, s1b;
                    block_dots_2rows(co.cb, q0[0], q1[0], a + (j * V.stride + x0) * 2, s0a, s1a);
                    block_dots_2rows(co.cb, q0[32], q1[32], a + ((j + 1) * V.stride + x0) * 2, s0b, s1b);
                    acc[0][0] = scale_acc2(acc[0][0], dw0, dx2, s0a, s0b);
                    acc[1][0] = scale_acc2(acc[1][0], dw1, dx2, s1a, s1b);
                }
#pragma unroll
                for (int r = 0; r < 2; ++r)
#pragma unroll
                    for (int i = 0; i < 2; ++i)
                        if (c + i < ncols) part[(r * kMaxCols + c + i) * 32 + lane] += acc[r][i].x + acc[r][i].y;
            }
        }
        co.release(P);
    }
    return ok;
}

// NC (3..5) columns with every sum in registers, both row sets: each index
// word expanded once (exact bytes) and dotted with all columns.
template <int NC>
__device__ __forceinline__ bool sweep_bk(Consumer &co, const Pipe &P, int b0, int b1, int nbp, const ActView &V,
                                         float *part, int warp, int lane) {
    float2 acc[2][NC];
#pragma unroll
    for (int r = 0; r < 2; ++r)
#pragma unroll
        for (int c = 0; c < NC; ++c) acc[r][c] = make_float2(0.0f, 0.0f);
    const int j = 2 * warp;
    bool ok = true;
    for (int b = b0; b < b1; b += kChunk) {
        if (b > b0) ok = ok && co.wait(P);
        const int nblk = min(kChunk, nbp - b);
        if (ok && j < nblk) {
            const uint4 *a, *q0, *q1;
            const float *d;
            stage_act_ptrs(V, co.st, b, nblk, a, d);
            stage_fields(co.st, nblk, warp, lane, q0, q1);
            const float2 dw0 = stage_dw(co.st, nblk, 0, warp, lane), dw1 = stage_dw(co.st, nblk, 1, warp, lane);
            int s0[2][NC], s1[2][NC];  // [block][column]
#pragma unroll
            for (int jj = 0; jj < 2; ++jj) {
                const uint4 wa = q0[32 * jj], wb = q1[32 * jj];
                const uint32_t wsa[4] = {wa.x, wa.y, wa.z, wa.w}, wsb[4] = {wb.x, wb.y, wb.z, wb.w};
                uint32_t ea[8], eb[8];
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    expand_select(co.cb, wsa[m], ea[2 * m], ea[2 * m + 1]);
                    expand_select(co.cb, wsb[m], eb[2 * m], eb[2 * m + 1]);
                }
#pragma unroll
                for (int c = 0; c < NC; ++c) {
                    const uint4 *ac = a + ((j + jj) * V.stride + c) * 2;
                    const uint4 x0 = ac[0], x1 = ac[1];
                    const uint32_t av[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
                    int t0 = co.cb.seed, t1 = co.cb.seed;
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        t0 = __dp4a((int)ea[i], (int)av[i], t0);
                        t1 = __dp4a((int)eb[i], (int)av[i], t1);
                    }
                    s0[jj][c] = t0;
                    s1[jj][c] = t1;
                }
            }
#pragma unroll
            for (int c = 0; c < NC; ++c) {
                const float2 dx2 = *reinterpret_cast<const float2 *>(d + ((j >> 1) * V.stride + c) * 2);
                acc[0][c] = scale_acc2(acc[0][c], dw0, dx2, s0[0][c], s0[1][c]);
                acc[1][c] = scale_acc2(acc[1][c], dw1, dx2, s1[0][c], s1[1][c]);
            }
        }
        co.release(P);
    }
#pragma unroll
    for (int r = 0; r < 2; ++r)
#pragma unroll
        for (int c = 0; c < NC; ++c) part[(r * kMaxCols + c) * 32 + lane] = acc[r][c].x + acc[r][c].y;
    return ok;
}

// One item pass over blocks [b0, b1) of a pair (nbp blocks in all) for the
// ncols columns at slots col[]: this warp's sums go to its slice part (row
// set r, column c at part[(r*kMaxCols + c)*32 + lane]).  One column, two
// columns (one shared expansion, sums in registers) and three or more (pairs
// per stage) each get their own loop.
__device__ __forceinline__ bool sweep_b(Consumer &co, const Pipe &P, int b0, int b1, int nbp, const ActView &V,
                                        const int (&col)[kMaxCols], int ncols, float *part, int warp, int lane) {
    if (ncols == 1) return sweep_b1(co, P, b0, b1, nbp, V, col[0], part, warp, lane);
    if (ncols == 2) return sweep_b2(co, P, b0, b1, nbp, V, col[0], col[1], part, warp, lane);
    return sweep_bn(co, P, b0, b1, nbp, V, col, ncols, part, warp, lane);
}

// Dynamic shared memory of a pipelined kernel:
//   [consts][full S][empty S][setfull 2][setempty 2][abort][tags S] | ring S x stage_bytes
//   | sets nsets x set_bytes | act act_blocks x 32 bytes | dx act_blocks x 4 bytes
struct PipeSmem {
    Pipe pipe;
    uint4 *act;  // persistent activation staging
    float *dx;
};

constexpr int kConstWords = 8;
constexpr uint32_t kSetBytes = 16 + kConsumerWarps * 2 * kMaxCols * 32 * 4;  // [warp][row set][column][lane]

__host__ __device__ inline size_t pipe_header_bytes(int S) {
    return ((size_t)4 * kConstWords + 16 * (size_t)S + 32 + 4 + 4 * (size_t)S + 127) / 128 * 128;
}

__host__ __device__ inline size_t pipe_smem_bytes(int S, uint32_t stage_bytes, uint32_t set_bytes, int nsets,
                                                  int act_blocks) {
    return pipe_header_bytes(S) + (size_t)S * stage_bytes + (size_t)nsets * set_bytes + (size_t)act_blocks * 36;
}

__device__ __forceinline__ PipeSmem carve_pipe(unsigned char *smem, int S, uint32_t stage_bytes, uint32_t set_bytes,
                                               int nsets, int act_blocks, unsigned *err) {
    PipeSmem L;
    L.pipe.consts = reinterpret_cast<uint32_t *>(smem);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + 4 * kConstWords);
    L.pipe.full0 = smem_addr(bars);
    L.pipe.empty0 = smem_addr(bars + S);
    L.pipe.setfull0 = smem_addr(bars + 2 * S);
    L.pipe.setempty0 = smem_addr(bars + 2 * S + 2);
    L.pipe.abort = reinterpret_cast<int *>(bars + 2 * S + 4);
    L.pipe.tag = L.pipe.abort + 1;
    L.pipe.ring = smem + pipe_header_bytes(S);
    L.pipe.sets = L.pipe.ring + (size_t)S * stage_bytes;
    L.pipe.err = err;
    L.pipe.S = S;
    L.pipe.stage_bytes = stage_bytes;
    L.pipe.set_bytes = set_bytes;
    L.pipe.nsets = (uint32_t)nsets;
    L.act = reinterpret_cast<uint4 *>(L.pipe.sets + (size_t)nsets * set_bytes);
    L.dx = reinterpret_cast<float *>(L.act + (size_t)act_blocks * 2);
    return L;
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
        for (int k = 0; k < 2; ++k) {
            mbar_init(P.setfull0 + 8u * k, kConsumers);
            mbar_init(P.setempty0 + 8u * k, 32);
        }
        *P.abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
}

}  // namespace cbq

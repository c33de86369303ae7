// cbq_kernels.cu -- sm_103a kernels of the codebook-4bit matvec and their
// launchers.
//
//   k_repack          canonical 18-byte blocks -> device layout (handle creation)
//   k_quantize        activation quantization, one warp per 32-value block
//   k_matvec<NC,F32,S> dense MMVQ over NC <= 5 columns, one pass over the weights
//                     (F32: one fp32 column, quantized inside the kernel; S:
//                     single 32-row groups as work items instead of pairs)
//   k_block_dots<NC>  the same integer path, exporting every per-block dot
//   k_moe             routed experts (and an optional shared expert), one
//                     kernel per layer call: gate+up rows, SwiGLU split,
//                     requantization, then down rows per slot
//   k_moe_combine     router-weighted combine of the per-slot down outputs
//   k_quantize_weights fp32 weights -> canonical blocks (the weight converter)
//   k_router_topk     top-k expert ids and softmax weights from router logits
//
// The matvec-type kernels are persistent: a grid of at most (SMs x resident
// CTAs) CTAs whose producer warps take 32-row work items from a global
// counter, so the activations are staged into shared memory once per CTA
// (k_block_dots, a debug path, takes static ranges).
#include "cbq_device.cuh"
#include "cbq_internal.h"

#include <algorithm>
#include <map>
#include <mutex>
#include <tuple>
#include <utility>

#include "cbq_pipe.cuh"

namespace cbq {

constexpr unsigned kErrBadExpertId = 0x1u;
// Pipeline depth of the dense kernel: the deepest ring (stages of 18 KB) that
// still lets two CTAs share an SM, at least kMinStages (the shape limit of a
// handle is checked at that depth) and at most kMaxStages.
constexpr int kMinStages = 4;
constexpr int kMaxStages = 6;

// Dynamic shared memory of the routed-expert kernel with S stages and
// act_blocks persistently staged blocks (the one token it quantizes itself).
size_t moe_smem_bytes(int act_blocks, int S) { return pipe_smem_bytes(S, kStageBytesAct, kSetBytes, 2, act_blocks); }

// Launch with optional programmatic stream serialization (PDL).
template <typename... KArgs, typename... Args>
static cudaError_t launch_k(void (*kern)(KArgs...), int grid, int block, size_t smem, cudaStream_t s, bool pdl,
                            Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3((unsigned)block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = pdl ? attr : nullptr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

// ------------------------------------------------------------- repack ------

// One thread per (pair p, half h, block b, lane): the 16 index bytes and the
// fp16 scale of row 32g + lane, block b, g the source group of (p, h) --
// 2p + h, or with split = Gf > 0 (a gate_up matrix) p for h = 0 and Gf + p for
// h = 1.  Rows beyond M and blocks beyond nb are zero.
__global__ void k_repack(const uint8_t *__restrict__ src, int64_t M, int nb, int nbp, int split, int64_t P,
                         uint8_t *__restrict__ w) {
    const int64_t total = P * 2 * nbp * 32;
    const size_t pb = pair_bytes(nbp);
    for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * blockDim.x) {
        const int lane = (int)(idx & 31);
        int64_t t = idx >> 5;
        const int b = (int)(t % nbp);
        t /= nbp;
        const int h = (int)(t & 1);
        const int64_t p = t >> 1;
        const int64_t g = split ? (h ? split + p : p) : 2 * p + h;
        const int64_t row = g * 32 + lane;
        uint32_t q[4] = {0, 0, 0, 0};
        uint16_t scale = 0;
        if (row < M && b < nb) {
            const uint8_t *s8 = src + ((size_t)row * nb + b) * 18;
            scale = (uint16_t)(s8[0] | (s8[1] << 8));
#pragma unroll
            for (int i = 0; i < 4; ++i)
                q[i] = (uint32_t)s8[2 + 4 * i] | ((uint32_t)s8[3 + 4 * i] << 8) | ((uint32_t)s8[4 + 4 * i] << 16) |
                       ((uint32_t)s8[5 + 4 * i] << 24);
        }
        uint8_t *base = w + (size_t)p * pb;
        *reinterpret_cast<uint4 *>(base + field_offset(nbp, h, b, lane)) = make_uint4(q[0], q[1], q[2], q[3]);
        *reinterpret_cast<uint16_t *>(base + scale_offset(nbp, h, b, lane)) = scale;
    }
}

cudaError_t launch_repack(const uint8_t *src, int64_t M, int nb, int split, uint8_t *w, cudaStream_t s) {
    const int nbp = round_up4(nb);
    const int64_t P = mat_pairs(M), total = P * 2 * nbp * 32;
    const int grid = (int)std::min<int64_t>((total + 255) / 256, 65535);
    k_repack<<<grid, 256, 0, s>>>(src, M, nb, nbp, split, P, w);
    return cudaGetLastError();
}

// ----------------------------------------------------------- quantize ------

__global__ void k_quantize(const float *__restrict__ x, int64_t total, int8_t *__restrict__ qx,
                           float *__restrict__ dx) {
    // launched as a programmatic dependent of whatever ran before on the
    // stream: wait for it (x may be its output), then let this call's
    // next kernel launch -- it may read the routing table or a handle's
    // counters before its own wait, so it must not start any earlier
    pdl_wait();
    pdl_trigger();
    // total = n*K, a multiple of 32; one lane per value, one warp per block.
    for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx - (threadIdx.x & 31) < total;
         idx += (int64_t)gridDim.x * blockDim.x) {
        // every lane of a warp shares idx>>5, so the warp enters and leaves together
        float d;
        const int8_t q = quant_lane(x[idx], d);
        qx[idx] = q;
        if ((threadIdx.x & 31) == 0) dx[idx >> 5] = d;
    }
}

cudaError_t launch_quantize(const float *x, int64_t K, int n, int8_t *qx, float *dx, cudaStream_t s) {
    const int64_t total = (int64_t)n * K;
    if (total == 0) return cudaSuccess;
    const int grid = (int)std::min<int64_t>((total + 255) / 256, 4096);
    return launch_k(k_quantize, grid, 256, 0, s, true, x, total, qx, dx);
}


// The layer's tokens quantized into the chunked activation layout (n
// columns), so a stage copies the slice of all tokens for its 16 blocks with
// one bulk copy.  Blocks nb..nbp-1 are zero.  One warp per (block, token);
// launched as a programmatic dependent.
__global__ void k_quantize_chunked(const float *__restrict__ x, int K, int n, int nbp, int8_t *__restrict__ qh) {
    pdl_wait();
    pdl_trigger();
    const int nb = K / kQK, lane = threadIdx.x & 31;
    for (int w = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5); w < nbp * n;
         w += (int)((gridDim.x * blockDim.x) >> 5)) {
        const int b = w / n, t = w - b * n;
        const int c = b / kChunk, j = b - c * kChunk, nblk = chunk_blocks(nbp, c);
        float d = 0.0f;
        int8_t q = 0;
        if (b < nb) q = quant_lane(x[(size_t)t * K + (size_t)b * kQK + lane], d);
        int8_t *base = qh + act_chunk_offset(c, n);
        base[(size_t)(j * n + t) * 32 + expander_pos(lane)] = q;
        if (lane == 0)
            *reinterpret_cast<float *>(base + (size_t)32 * n * nblk + ((size_t)(j >> 1) * n + t) * 8 + (j & 1) * 4) = d;
    }
}

cudaError_t launch_quantize_chunked(const float *x, int K, int n, int8_t *qh, cudaStream_t s) {
    const int nbp = round_up4(K / kQK);
    const int grid = std::min((nbp * n * 32 + 255) / 256, 4096);
    return launch_k(k_quantize_chunked, grid, 256, 0, s, true, x, K, n, nbp, qh);
}

// ---------------------------------------------------------- dense MMVQ -----

// One partial-sum set of NC columns per warp (one row per lane): the
// epilogue warp reads a pair's sums long before the consumers finish the next
// pair, and the room a second set would take goes to the ring.
__host__ __device__ inline uint32_t dense_set_bytes(int n) { return 16u + (uint32_t)(kConsumerWarps * n * 32 * 4); }
static size_t dense_smem_bytes(int S, int nbp, int n) {
    return pipe_smem_bytes(S, kStageWeightBytes, dense_set_bytes(n), 1, n * nbp);
}
size_t matvec_smem_bytes(int nbp, int n) { return dense_smem_bytes(kMinStages, nbp, n); }

// Debug kernel smem: activations + scales only.
static size_t dots_smem_bytes(int nbp, int n) { return (size_t)n * nbp * 36; }

struct MatvecArgs {
    DevMat W;
    const int8_t *qx;  // quantized columns (kF32 == false)
    const float *dx;
    const float *xf;   // fp32 column (kF32 == true)
    int64_t K;
    float *y;
    int S;             // pipeline stages
};

// Work counters of a persistent kernel (sched[0] items taken, sched[1] CTAs
// done taking items).  Each CTA's producer counts itself done once it has
// taken its last item; the last CTA to do so resets both words at once (no
// CTA of this launch reads them again, and the next launch reads them only
// after this grid has completed), so no CTA waits on a counter at its end.
__device__ __forceinline__ bool done_taking(unsigned *sched) {
    return atomicAdd(sched + 1, 1u) == gridDim.x - 1;
}
__device__ __forceinline__ void reset_sched(unsigned *sched) {
    sched[0] = 0u;
    sched[1] = 0u;
}

// One 4-block quad of one row (this lane) for NC columns: the quad's index
// words at qs[0], qs[32], qs[64], qs[96]; its four fp16 scales in s; the
// activations block-major at act (block j of column c at act[(j*NC + c)*2]);
// the activation scales as float2 pairs at dxp (blocks 0-1 of column c at
// dxp[c], blocks 2-3 at dxp[NC + c]).
template <int NC>
__device__ __forceinline__ void quad(const Codebook &cb, const uint4 *qs, uint2 s, const uint4 *act,
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

// One item pass of the dense kernel for NC columns staged block-major (act,
// dx: stride NC), one row per lane.  Warp w takes quad w % 4 of sub-stage
// w / 4 of every stage, so its sums (acc) are those of one 32-row group.  A
// pair item's stage holds the pair's two groups of one 16-block chunk
// (sub-stage h = group h, at h * nblk * kBlockBytes).  With kSingle the item
// is one group and a stage holds its part of two consecutive chunks
// (sub-stage k = chunk 2s + k, at k * nblk0 * kBlockBytes, nblk0 the blocks of
// the first), so all eight warps work on that group.  Each sub-stage holds its
// index fields and then its scales.  False on a give-up.
template <int NC, bool kSingle>
__device__ __forceinline__ bool dense_pass(Consumer &co, const Pipe &P, int nbp, const uint4 *act, const float *dx,
                                           float2 acc[NC], int warp, int lane) {
    const int h = warp >> 2, q = warp & 3;
    bool ok = true;
    if constexpr (!kSingle) {
        for (int b = 0; b < nbp; b += kChunk) {
            if (b > 0) ok = ok && co.wait(P);
            const int nblk = min(kChunk, nbp - b);
            if (ok && 4 * q < nblk) {
                const unsigned char *half = co.st + (size_t)h * nblk * kBlockBytes;
                const uint4 *qs = reinterpret_cast<const uint4 *>(half) + q * 128 + lane;
                const uint2 s = reinterpret_cast<const uint2 *>(half + (size_t)nblk * 512)[q * 32 + lane];
                const int bq = b + 4 * q;
                quad<NC>(co.cb, qs, s, act + (size_t)bq * NC * 2,
                         reinterpret_cast<const float2 *>(dx) + (bq >> 1) * NC, acc);
            }
            co.release(P);
        }
    } else {
        for (int b = 0; b < nbp; b += 2 * kChunk) {
            if (b > 0) ok = ok && co.wait(P);
            const int nblk0 = min(kChunk, nbp - b);
            const int bh = b + h * kChunk;  // first block of this warp's sub-stage
            const int nblk = min(kChunk, nbp - bh);
            if (ok && 4 * q < nblk) {
                const unsigned char *sub = co.st + (size_t)h * nblk0 * kBlockBytes;
                const uint4 *qs = reinterpret_cast<const uint4 *>(sub) + q * 128 + lane;
                const uint2 s = reinterpret_cast<const uint2 *>(sub + (size_t)nblk * 512)[q * 32 + lane];
                const int bq = bh + 4 * q;
                quad<NC>(co.cb, qs, s, act + (size_t)bq * NC * 2,
                         reinterpret_cast<const float2 *>(dx) + (bq >> 1) * NC, acc);
            }
            co.release(P);
        }
    }
    return ok;
}

// Dense MMVQ: pairs of 32-row groups fetched per CTA, all NC columns per
// pass; the epilogue warp adds the consumer warps' sums of a pair (four per
// group) and stores its 64 rows of y.  kSingle: the work items are single
// 32-row groups (item i = group i & 1 of pair i / 2) and the epilogue adds
// all eight warps' sums of the group.  kF32: the consumers quantize the fp32
// column xf themselves while the producer starts the weight stream (no
// quantization kernel before it); otherwise they stage qx/dx written by the
// quantization kernel launched just before (a programmatic dependency).
template <int NC, bool kF32, bool kSingle>
__global__ void __launch_bounds__(kPipeThreads, 2) k_matvec(const __grid_constant__ MatvecArgs A) {
    extern __shared__ __align__(128) unsigned char smem[];
    pdl_trigger();  // the next kernel may launch; it waits for this grid before touching what it writes
    const DevMat &W = A.W;
    const PipeSmem S = carve_pipe(smem, A.S, kStageWeightBytes, dense_set_bytes(NC), 1, NC * W.nbp, W.err);
    pipe_init(S.pipe);
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const unsigned total = (unsigned)(kSingle ? 2 * W.P : W.P);
    const size_t pb = pair_bytes(W.nbp);
    const int nch = (W.nbp + kChunk - 1) / kChunk;
    if (warp == kProducerWarp) {
        if (lane == 0) {
            Producer pr;
            auto pass = [&](unsigned item) {
                if constexpr (kSingle)
                    pr.pass_single(S.pipe, W.w + (item >> 1) * pb, W.nbp, nch, (int)(item & 1u), (int)item);
                else
                    pr.pass(S.pipe, W.w + item * pb, W.nbp, 0, nch, (int)item);
            };
            // The first item is the CTA index (the launcher sizes the grid to
            // at most the item count): its weights stream before the wait for
            // the work ahead of this kernel, which the work counter needs (a
            // call still running on the handle owns it).  The index of the
            // next item is fetched when an item starts and used once its
            // stages are issued, so the atomic's latency overlaps them.
            if (blockIdx.x < total) pass(blockIdx.x);
            pdl_wait();
            unsigned next = gridDim.x + atomicAdd(W.sched, 1u);
            while (next < total && !pr.stopped) {
                const unsigned item = next;
                next = gridDim.x + atomicAdd(W.sched, 1u);
                pass(item);
            }
            const bool last = done_taking(W.sched);
            pr.finish(S.pipe);
            pr.drain(S.pipe);
            if (last) reset_sched(W.sched);
        }
    } else if (warp == kEpilogueWarp) {
        SetReader rd;
        for (;;) {
            const int *tag;
            const float *part;
            if (!rd.wait(S.pipe, tag, part)) break;
            const int it = *(volatile const int *)tag;
            if (it < 0) break;
            if constexpr (!kSingle) {
                float v[2][NC];
#pragma unroll
                for (int r = 0; r < 2; ++r)
#pragma unroll
                    for (int c = 0; c < NC; ++c) {
                        v[r][c] = 0.0f;
#pragma unroll
                        for (int w = 4 * r; w < 4 * r + 4; ++w) v[r][c] += part[(w * NC + c) * 32 + lane];
                    }
                rd.release(S.pipe);
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    const int64_t row = (int64_t)(2 * it + r) * 32 + lane;
                    if (row < W.M) {
#pragma unroll
                        for (int c = 0; c < NC; ++c) A.y[(size_t)c * W.M + row] = v[r][c];
                    }
                }
            } else {  // one group (item it = group it of the matrix): all eight warps' sums, in warp order
                float v[NC];
#pragma unroll
                for (int c = 0; c < NC; ++c) {
                    v[c] = 0.0f;
#pragma unroll
                    for (int w = 0; w < kConsumerWarps; ++w) v[c] += part[(w * NC + c) * 32 + lane];
                }
                rd.release(S.pipe);
                const int64_t row = (int64_t)it * 32 + lane;
                if (row < W.M) {
#pragma unroll
                    for (int c = 0; c < NC; ++c) A.y[(size_t)c * W.M + row] = v[c];
                }
            }
        }
    } else {
        pdl_wait();  // the activations belong to the work ahead
        if constexpr (kF32) {
            quant_stage_cols<NC>(A.xf, A.K, W.nb, W.nbp, S.act, S.dx, threadIdx.x, kConsumers);
        } else {
            ColSrc src{A.qx, A.dx, (size_t)A.K, (size_t)W.nb, {0, 1, 2, 3, 4}};
            stage_cols(src, NC, W.nb, W.nbp, S.act, S.dx, threadIdx.x, kConsumers, false, true);
        }
        consumer_sync();
        Consumer co(S.pipe);
        SetWriter wr;
        for (;;) {
            const int it = co.wait(S.pipe) ? co.tag(S.pipe) : -1;
            int *tag;
            float *part;
            if (it < 0) {
                if (!wr.acquire(S.pipe, tag, part)) break;
                if (threadIdx.x == 0) *tag = -1;
                wr.publish(S.pipe);
                break;
            }
            float2 acc[NC];
#pragma unroll
            for (int c = 0; c < NC; ++c) acc[c] = make_float2(0.0f, 0.0f);
            const bool ok = dense_pass<NC, kSingle>(co, S.pipe, W.nbp, S.act, S.dx, acc, warp, lane);
            // the set is taken only now: the epilogue had the whole pass to free it
            if (!wr.acquire(S.pipe, tag, part)) break;
#pragma unroll
            for (int c = 0; c < NC; ++c) part[(warp * NC + c) * 32 + lane] = acc[c].x + acc[c].y;
            if (threadIdx.x == 0) *tag = it;
            wr.publish(S.pipe);
            if (!ok) break;
        }
    }
}

template <int NC>
__global__ void __launch_bounds__(kThreads, 2)
    k_block_dots(const DevMat W, const int8_t *__restrict__ qx, int64_t K, int32_t *__restrict__ sdot, int chunk) {
    extern __shared__ __align__(128) unsigned char smem[];
    const int g0 = blockIdx.x * chunk;
    const int g1 = min(W.G, g0 + chunk);
    if (g0 >= W.G) return;
    const int nb = W.nb, nbp = W.nbp;
    uint4 *act_s = reinterpret_cast<uint4 *>(smem);
    float *dx_s = reinterpret_cast<float *>(act_s + (size_t)NC * nbp * 2);
    {
        // the activation scales do not enter the integer dots: stage zeros
        ColSrc src{qx, nullptr, (size_t)K, 0, {0, 1, 2, 3, 4}};
        stage_cols(src, NC, nb, nbp, act_s, dx_s, threadIdx.x, blockDim.x, false, true);
    }
    __shared__ uint32_t consts[kConstWords];
    if (threadIdx.x == 0) write_consts(consts);
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nbq = nbp / 4;
    const int q0 = warp * nbq / kWarps, q1 = (warp + 1) * nbq / kWarps;
    const Codebook cb = read_consts(consts);
    for (int g = g0; g < g1; ++g) {
        const int64_t row = (int64_t)g * 32 + lane;
        // the pair and half of logical group g
        const int p = W.split ? (g < W.split ? g : g - W.split) : g >> 1;
        const int h = W.split ? (g < W.split ? 0 : 1) : g & 1;
        const uint8_t *pw = W.w + (size_t)p * pair_bytes(nbp);
        for (int q = q0; q < q1; ++q) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int b = 4 * q + j;
                const uint4 w = ld_stream16(reinterpret_cast<const uint4 *>(pw + field_offset(nbp, h, b, lane)));
                int sd[NC];
                block_dots<NC>(cb, w, act_s + (size_t)b * NC * 2, sd);
                if (row < W.M && b < nb) {
#pragma unroll
                    for (int c = 0; c < NC; ++c) sdot[((size_t)c * W.M + row) * nb + b] = sd[c] - cb.seed;
                }
            }
        }
    }
}

// Per-device launch facts, looked up once under a lock: the SM count, and per
// (kernel, dynamic shared memory, block size) the resident CTAs per SM.  The
// first time a kernel is seen on a device its dynamic shared-memory ceiling
// is raised to the device's opt-in maximum (less its static shared memory),
// so no launch has to set it.
struct LaunchFacts {
    std::mutex m;
    std::map<int, int> sms;
    std::map<std::pair<int, const void *>, bool> raised;
    std::map<std::tuple<int, const void *, size_t, int>, int> per_sm;
};
static LaunchFacts g_launch;

template <typename Kernel>
static cudaError_t resident(Kernel kern, int threads, size_t smem, int *sms, int *per_sm) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const void *id = reinterpret_cast<const void *>(kern);
    std::lock_guard<std::mutex> lock(g_launch.m);
    auto s = g_launch.sms.find(dev);
    if (s == g_launch.sms.end()) {
        int v = 0;
        e = cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        s = g_launch.sms.emplace(dev, v).first;
    }
    *sms = s->second;
    const auto key = std::make_tuple(dev, id, smem, threads);
    auto p = g_launch.per_sm.find(key);
    if (p == g_launch.per_sm.end()) {
        bool &raised = g_launch.raised[std::make_pair(dev, id)];
        if (!raised) {  // the opt-in maximum less the kernel's static shared memory
            int optin = 0;
            cudaFuncAttributes fa;
            e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
            if (e == cudaSuccess) e = cudaFuncGetAttributes(&fa, kern);
            if (e == cudaSuccess)
                e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         optin - (int)fa.sharedSizeBytes);
            if (e != cudaSuccess) return e;
            raised = true;
        }
        int v = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&v, kern, threads, smem);
        if (e != cudaSuccess) return e;
        p = g_launch.per_sm.emplace(key, v).first;
    }
    *per_sm = p->second;
    return cudaSuccess;
}

// Dynamic shared memory the dense kernels may use: the opt-in limit less
// the largest static shared memory of their instances.
cudaError_t matvec_smem_limit(size_t *bytes) {
    size_t optin = 0, st = 0;
    cudaError_t e = device_smem_limit(&optin);
    void (*kerns[])(const MatvecArgs) = {k_matvec<1, true, false>,  k_matvec<1, false, false>,
                                         k_matvec<2, false, false>, k_matvec<3, false, false>,
                                         k_matvec<4, false, false>, k_matvec<5, false, false>,
                                         k_matvec<1, true, true>,   k_matvec<1, false, true>,
                                         k_matvec<2, false, true>,  k_matvec<3, false, true>,
                                         k_matvec<4, false, true>,  k_matvec<5, false, true>};
    for (auto k : kerns) {
        cudaFuncAttributes fa;
        if (e == cudaSuccess) e = cudaFuncGetAttributes(&fa, k);
        if (e == cudaSuccess) st = std::max(st, fa.sharedSizeBytes);
    }
    *bytes = e == cudaSuccess ? optin - st : 0;
    return e;
}

cudaError_t device_smem_limit(size_t *bytes) {
    int dev = 0, v = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    *bytes = (size_t)v;
    return e;
}

// Grid of a persistent kernel over `items` work items: at most resident
// capacity, with contiguous equal chunks.
template <typename Kernel>
static cudaError_t persistent_grid(Kernel kern, int threads, size_t smem, int64_t items, int *grid, int *chunk) {
    int sms = 0, per_sm = 0;
    const cudaError_t e = resident(kern, threads, smem, &sms, &per_sm);
    if (e != cudaSuccess) return e;
    const int64_t cap = (int64_t)sms * std::max(per_sm, 1);
    const int64_t g = std::max<int64_t>(1, std::min<int64_t>(items, cap));
    const int64_t ch = (items + g - 1) / g;
    *chunk = (int)std::max<int64_t>(ch, 1);
    *grid = (int)std::max<int64_t>(1, (items + *chunk - 1) / *chunk);
    return cudaSuccess;
}

// Grid of a persistent kernel that fetches its work dynamically: one CTA per
// resident slot, at most one per item.
template <typename Kernel>
static cudaError_t dynamic_grid(Kernel kern, size_t smem, int64_t items, int *grid) {
    int sms = 0, per_sm = 0;
    const cudaError_t e = resident(kern, kPipeThreads, smem, &sms, &per_sm);
    if (e != cudaSuccess) return e;
    *grid = (int)std::max<int64_t>(1, std::min<int64_t>(items, (int64_t)sms * std::max(per_sm, 1)));
    return cudaSuccess;
}

// Stages of the dense kernel's ring: the deepest that keeps the residency of
// the kMinStages ring (two CTAs per SM where that fits), so the next call's
// weights stream sooner.
template <typename Kernel>
static cudaError_t dense_stages(Kernel kern, const DevMat &W, int NC, int *S_out, int *sms) {
    int S = kMinStages, base = 0;
    cudaError_t e = resident(kern, kPipeThreads, dense_smem_bytes(S, W.nbp, NC), sms, &base);
    if (e != cudaSuccess) return e;
    for (int t = kMaxStages; t > kMinStages; --t) {
        int per_sm = 0;
        e = resident(kern, kPipeThreads, dense_smem_bytes(t, W.nbp, NC), sms, &per_sm);
        if (e != cudaSuccess) return e;
        if (per_sm >= std::min(base, 2)) {
            S = t;
            break;
        }
    }
    *S_out = S;
    return cudaSuccess;
}

template <int NC, bool kF32, bool kSingle>
static cudaError_t launch_matvec_k(const DevMat &W, const int8_t *qx, const float *dx, const float *xf, float *y,
                                   cudaStream_t s, bool pdl) {
    int S = 0, sms = 0, grid = 0;
    cudaError_t e = dense_stages(k_matvec<NC, kF32, kSingle>, W, NC, &S, &sms);
    if (e != cudaSuccess) return e;
    const size_t smem = dense_smem_bytes(S, W.nbp, NC);
    e = dynamic_grid(k_matvec<NC, kF32, kSingle>, smem, kSingle ? 2 * (int64_t)W.P : W.P, &grid);
    if (e != cudaSuccess) return e;
    MatvecArgs A;
    A.W = W;
    A.qx = qx;
    A.dx = dx;
    A.xf = xf;
    A.K = (int64_t)W.nb * kQK;
    A.y = y;
    A.S = S;
    return launch_k(k_matvec<NC, kF32, kSingle>, grid, kPipeThreads, smem, s, pdl, A);
}

// Work items of whole pairs, or every pair as two single-group items when
// that lightens the busiest SM by at least 8%: the SMs take work in whole
// items, so ceil(P / SMs) pairs land on the busiest one against ceil(2P / SMs)
// halves.  Measured by graph replay: 4096 x 4096 at n = 1 (64 pairs) 8.7 ->
// 6.7 us, 32768 x 4096 at n = 1 / 5 18.3 -> 16.1 / 29.8 -> 27.7 us; 16384 x
// 4096 (ratio 1) was 3-14% slower split, the 129280-row head (ratio 0.96)
// no faster.
template <int NC, bool kF32>
static cudaError_t launch_matvec_n(const DevMat &W, const int8_t *qx, const float *dx, const float *xf, float *y,
                                   cudaStream_t s, bool pdl) {
    int sms = 0, per_sm = 0;
    cudaError_t e = resident(k_matvec<NC, kF32, false>, kPipeThreads, dense_smem_bytes(kMinStages, W.nbp, NC), &sms,
                             &per_sm);
    if (e != cudaSuccess) return e;
    const int64_t pair_load = (W.P + sms - 1) / sms, half_load = (2 * (int64_t)W.P + sms - 1) / sms;
    if (half_load * 25 <= pair_load * 46) return launch_matvec_k<NC, kF32, true>(W, qx, dx, xf, y, s, pdl);
    return launch_matvec_k<NC, kF32, false>(W, qx, dx, xf, y, s, pdl);
}

cudaError_t launch_matvec(const DevMat &W, const int8_t *qx, const float *dx, int n, float *y, cudaStream_t s,
                          bool pdl) {
    switch (n) {
        case 1: return launch_matvec_n<1, false>(W, qx, dx, nullptr, y, s, pdl);
        case 2: return launch_matvec_n<2, false>(W, qx, dx, nullptr, y, s, pdl);
        case 3: return launch_matvec_n<3, false>(W, qx, dx, nullptr, y, s, pdl);
        case 4: return launch_matvec_n<4, false>(W, qx, dx, nullptr, y, s, pdl);
        case 5: return launch_matvec_n<5, false>(W, qx, dx, nullptr, y, s, pdl);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_matvec_f32(const DevMat &W, const float *x, int n, float *y, cudaStream_t s) {
    if (n != 1) return cudaErrorInvalidValue;
    return launch_matvec_n<1, true>(W, nullptr, nullptr, x, y, s, true);
}

template <int NC>
static cudaError_t launch_block_dots_n(const DevMat &W, const int8_t *qx, int32_t *sdot, cudaStream_t s) {
    const size_t smem = dots_smem_bytes(W.nbp, NC);
    int grid = 0, chunk = 0;
    cudaError_t e = persistent_grid(k_block_dots<NC>, kThreads, smem, W.G, &grid, &chunk);
    if (e != cudaSuccess) return e;
    k_block_dots<NC><<<grid, kThreads, smem, s>>>(W, qx, (int64_t)W.nb * kQK, sdot, chunk);
    return cudaGetLastError();
}

cudaError_t launch_block_dots(const DevMat &W, const int8_t *qx, int n, int32_t *sdot, cudaStream_t s) {
    switch (n) {
        case 1: return launch_block_dots_n<1>(W, qx, sdot, s);
        case 2: return launch_block_dots_n<2>(W, qx, sdot, s);
        case 3: return launch_block_dots_n<3>(W, qx, sdot, s);
        case 4: return launch_block_dots_n<4>(W, qx, sdot, s);
        case 5: return launch_block_dots_n<5>(W, qx, sdot, s);
        default: return cudaErrorInvalidValue;
    }
}

// --------------------------------------------------------- routed experts --

// Largest token (in blocks of 32) the layer kernel stages for itself.
constexpr int kMaxStagedBlocks = 1024;

struct MoeArgs {
    DevMoe L;
    MoeWork ws;
    const float *h;
    const int32_t *ids;
    const float *wts;
    float *y;
    int n_tok, k, swiglu;
    int nbH, nbpH, nbF, nbpF;
    int quant_tokens;  // one token, h 16-byte aligned: the consumers quantize it themselves
    int fuse_combine;  // one token: the layer kernel writes y itself (no combine kernel)
    int stages;        // pipeline depth (4, or 3 where two CTAs per SM allow no more)
};

// The routing table of one call, derived redundantly by every CTA (by its
// producer warp, in registers) from the <= 85 slots (no host round trip).
// Slots 0..N-1 are the routed ones (p = t*k + j); with a shared expert, slots
// N..N+n_tok-1 hold its virtual id E, one per token.  An out-of-range routed
// id is stored as -1 and takes part in no expert.  The slots are scanned with
// the shared expert's first, then the routed ones in order, and the distinct
// experts are ordered by their first slot in that scan (the shared expert's
// items, with a column for every token, are the slowest: handed out first,
// they do not form the tail of a pass).  Each distinct expert is split into
// column groups of at most kMaxCols of its slots (more slots than that only
// with repeated ids), its "virtual experts": every item works on one virtual
// expert.
struct Routing {
    int ids[kMaxSlots];                        // expert of each slot (-1: out of range)
    float w[kMaxSlots];                        // router weight of each slot (shared-expert slots: 1)
    int vbase[kMaxSlots];                      // by scan position of an expert's first slot: its first virtual expert
    int vexp[kMaxSlots];                       // expert id of virtual expert v
    unsigned char vnc[kMaxSlots];              // its columns (1..kMaxCols)
    unsigned char vslot[kMaxSlots][kMaxCols];  // its slots, ascending
    int D, V;
    unsigned epoch;                            // the handle's call count (selects the counter set)
};

// Words of a layer handle's ws.sched: items taken, CTAs done taking items,
// the call count (epoch), and per counter set the dependency words its last
// call used.
constexpr int kSchedFetch = 0, kSchedDone = 1, kSchedEpoch = 2, kSchedUsed = 3;

// The routing table, built by the 32 lanes of one warp: lane l holds scan
// positions l, l+32, l+64.  Equal ids are found with a warp match inside a
// pass of 32 positions and with shuffles across passes; the distinct experts'
// ranks come from ballots and their first virtual experts from a warp scan.
// The ids, router weights and epoch are loaded in one round trip.
__device__ void route_warp(const int32_t *__restrict__ ids, const float *__restrict__ wts, const unsigned *sched,
                           int N, int n_all, int E, Routing &R, unsigned *err, int lane) {
    static_assert(kMaxSlots <= 3 * 32, "three scan positions per lane");
    constexpr unsigned kFull = 0xffffffffu;
    const unsigned below = (1u << lane) - 1u;
    const int n_sh = n_all - N;  // shared-expert slots, scanned first
    int p[3], e[3];
    float w[3];
#pragma unroll
    for (int i = 0; i < 3; ++i) {
        const int s = lane + 32 * i;
        p[i] = s < n_sh ? N + s : s - n_sh;
        e[i] = -2;  // no slot here
        w[i] = 1.0f;
        if (s < n_all) {
            e[i] = E;  // a shared-expert slot
            if (p[i] < N) {
                e[i] = ids[p[i]];
                w[i] = wts[p[i]];
            }
        }
    }
    const unsigned epoch = lane == 0 ? *(volatile const unsigned *)(sched + kSchedEpoch) : 0u;
#pragma unroll
    for (int i = 0; i < 3; ++i) {
        if (lane + 32 * i >= n_all) continue;
        if (p[i] < N && (e[i] < 0 || e[i] >= E)) {
            if (err) atomicOr(err, kErrBadExpertId);
            e[i] = -1;
        }
        R.ids[p[i]] = e[i];
        R.w[p[i]] = w[i];
    }
    // per position: equal ids before it and in all, and the first of them
    const int npass = (n_all + 31) / 32;
    int before[3], total[3], first_pos[3];
#pragma unroll
    for (int i = 0; i < 3; ++i) {
        const unsigned m = __match_any_sync(kFull, e[i]);
        before[i] = __popc(m & below);
        total[i] = __popc(m);
        first_pos[i] = 32 * i + __ffs(m) - 1;
    }
    if (npass > 1) {
#pragma unroll
        for (int j = 0; j < 3; ++j) {
            if (j >= npass) break;
            for (int l = 0; l < 32; ++l) {
                const int v = __shfl_sync(kFull, e[j], l);
#pragma unroll
                for (int i = 0; i < 3; ++i) {
                    if (i == j || v != e[i]) continue;
                    ++total[i];
                    if (j < i) {
                        ++before[i];
                        first_pos[i] = min(first_pos[i], 32 * j + l);
                    }
                }
            }
        }
    }
    // distinct experts: positions holding the first slot of a valid id
    bool first[3];
    unsigned bal[3];
#pragma unroll
    for (int i = 0; i < 3; ++i) {
        first[i] = e[i] >= 0 && before[i] == 0;
        bal[i] = __ballot_sync(kFull, first[i]);
    }
    // first virtual expert of each distinct expert: exclusive scan of
    // ceil(slots / kMaxCols) over the first slots in scan order
    int carry = 0;
#pragma unroll
    for (int i = 0; i < 3; ++i) {
        const int nv = first[i] ? (total[i] + kMaxCols - 1) / kMaxCols : 0;
        int x = nv;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int y = __shfl_up_sync(kFull, x, d);
            if (lane >= d) x += y;
        }
        if (first[i]) R.vbase[lane + 32 * i] = carry + x - nv;
        carry += __shfl_sync(kFull, x, 31);
    }
    __syncwarp();
#pragma unroll
    for (int i = 0; i < 3; ++i) {
        if (e[i] < 0) continue;
        const int v = R.vbase[first_pos[i]] + before[i] / kMaxCols, c = before[i] % kMaxCols;
        R.vslot[v][c] = (unsigned char)p[i];
        if (c == 0) {
            R.vexp[v] = e[i];
            R.vnc[v] = (unsigned char)min(kMaxCols, total[i] - before[i]);
        }
    }
    if (lane == 0) {
        R.V = carry;
        R.D = __popc(bal[0]) + __popc(bal[1]) + __popc(bal[2]);
        R.epoch = epoch;
    }
    __syncwarp();
}

// Token of slot p: routed slots are t*k + j, shared-expert slots N + t.
__device__ __forceinline__ int slot_token(int p, int N, int k) { return p < N ? p / k : p - N; }

// Weights of expert e, the shared expert for e == E.
__device__ __forceinline__ const uint8_t *gate_up_of(const DevMoe &L, int e) {
    return e < L.E ? L.gu + (size_t)e * L.gu_stride : L.sh_gu;
}

__device__ __forceinline__ const uint8_t *down_of(const DevMoe &L, int e) {
    return e < L.E ? L.dn + (size_t)e * L.dn_stride : L.sh_dn;
}

constexpr unsigned kErrDependencyTimeout = 0x200u;
constexpr unsigned kDownGrab = 4;
constexpr int kMaxTopk = 16;  // routed experts per token (the ABI's limit)

__device__ __forceinline__ unsigned ld_relaxed(const unsigned *p) {
    unsigned v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ unsigned ld_acquire(const unsigned *p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Bounded wait (the producer lane) until *cnt >= target: the intermediate
// columns a down stage reads are all published.  On timeout it sets
// kErrDependencyTimeout; it returns false then, or at once when the CTA
// already gave up.  On success the bulk copies issued next may read what the
// publishing CTAs wrote (the acquire load orders it, the proxy fence carries
// that order to the copy engine).
__device__ __forceinline__ bool wait_dependency(const unsigned *cnt, unsigned target, const Pipe &P) {
    if (ld_acquire(cnt) < target) {
        const uint64_t t0 = global_ns();
        for (;;) {
            if (*(volatile int *)P.abort) return false;
            __nanosleep(100);
            if (ld_acquire(cnt) >= target) break;
            if (global_ns() - t0 > kWaitLimitNs) {
                atomicOr(P.err, kErrDependencyTimeout);
                return false;
            }
        }
    }
    asm volatile("fence.proxy.async.global;" ::: "memory");
    return true;
}

// The slices of a down pass: chunk c of the intermediate of virtual expert v
// (cnt: its per-chunk counts) is ready once all of its min(16, Gf - 16c)
// gate_up groups are published.  all_ready() polls every chunk's count in
// batches of relaxed loads issued together (then one acquire fence), and
// remembers a virtual expert found complete in a per-CTA bit (counts only
// grow within a call), so the down items of an expert whose gate_up work is
// long done cost no polls at all; ready() polls one chunk, wait() waits for
// it (bounded).  In give-up test mode 1 a slice is never ready.  Every true
// result is followed by a proxy fence, so the bulk copies issued next see
// what the publishers wrote.
struct DownDep {
    const unsigned *cnt;
    int Gf, stall;
    const Pipe *P;
    unsigned *vready;  // shared-memory bits: virtual experts whose slices are all ready
    int v;
    __device__ __forceinline__ unsigned target(int c) const {
        return stall == 1 ? ~0u : (unsigned)min(kChunk, Gf - c * kChunk);
    }
    __device__ __forceinline__ bool all_ready(int c0, int c1) const {
        if (vready[v >> 5] & (1u << (v & 31))) return true;
        constexpr int kBatch = 8;
        for (int c = c0; c < c1; c += kBatch) {
            unsigned got[kBatch];
#pragma unroll
            for (int i = 0; i < kBatch; ++i) got[i] = c + i < c1 ? ld_relaxed(cnt + c + i) : ~0u;
#pragma unroll
            for (int i = 0; i < kBatch; ++i)
                if (c + i < c1 && got[i] < target(c + i)) return false;
        }
        vready[v >> 5] |= 1u << (v & 31);
        asm volatile("fence.acq_rel.gpu;" ::: "memory");
        asm volatile("fence.proxy.async.global;" ::: "memory");
        return true;
    }
    __device__ __forceinline__ bool ready(int c) const {
        if (ld_acquire(cnt + c) < target(c)) return false;
        asm volatile("fence.proxy.async.global;" ::: "memory");
        return true;
    }
    __device__ __forceinline__ bool wait(int c) const { return wait_dependency(cnt + c, target(c), *P); }
};

// The whole routed-expert layer, combine included, in one persistent kernel.
// Work items, in this order (the first per CTA is its index, the rest come
// from one counter):
//   it <  V*Gf : gate_up item (virtual expert v, 32-row-pair group g), v-major:
//                gate rows 32g.. and up rows F+32g.. in one pass; the epilogue
//                warp applies the SwiGLU split and requantizes the 32 outputs
//                of each column (block g of the column's a);
//   it >= V*Gf : down item (virtual expert v, 64-row group g: 32-row groups 2g
//                and 2g+1), v-major, per-slot outputs to obuf.
// A down stage covering blocks [16s, 16s+16) of a reads only the blocks that
// gate_up groups 16s..16s+15 of its virtual expert wrote: the producer waits
// (bounded) for that count before it copies the slice.  The gate_up items are
// all handed out before any down item, and taken items never wait for later
// ones, so the wait always ends.  The down item that completes a 64-row group
// for the last of the V virtual experts (a per-group count) adds the group's
// slot outputs into y: the router-weighted sum in slot order, then the shared
// expert's output.
// Counters: the dependency and group counts come in two sets, used by calls
// of even and odd epoch; the last CTA to finish taking items zeroes the set of
// the previous call (complete by then), resets the item counters and advances
// the epoch, so no CTA waits on a counter at its end.
// With one token (quantized here) this is the call's first kernel, launched
// as a programmatic dependent: it sets up its pipeline, then waits for all
// earlier work before it reads anything.  Otherwise it follows the
// quantization kernel, which starts it only once all earlier work has ended,
// so the routing table and the handle's counters are read at once; the
// producer waits for the quantized tokens before it copies their first slice.
__global__ void __launch_bounds__(kPipeThreads, 2) k_moe(const __grid_constant__ MoeArgs A) {
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ Routing R;
    __shared__ __align__(8) uint64_t route_bar;  // the routing table is ready (one arrive per producer lane)
    __shared__ unsigned vready[(kMaxSlots + 31) / 32];  // producer: virtual experts with all slices ready
    PipeSmem S = carve_pipe(smem, A.stages, kStageBytesAct, kSetBytes, 2, A.quant_tokens ? A.nbpH : 0, A.ws.err);
    pipe_init(S.pipe);
    if (threadIdx.x < (kMaxSlots + 31) / 32) vready[threadIdx.x] = 0u;
    if (threadIdx.x == 0) {
        mbar_init(smem_addr(&route_bar), 32);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    if (A.quant_tokens) pdl_wait();
    pdl_trigger();  // the next kernel may launch (the combine, or the next call's first); it waits for this grid
    const int N = A.n_tok * A.k, n_all = N + (A.L.shared ? A.n_tok : 0);  // routed slots, then shared ones
    const int Gf = A.L.F / 32, Gd = A.L.H / 32, Gd2 = (Gd + 1) / 2;
    const int nsF = (A.nbpF + kChunk - 1) / kChunk;  // down stages (dependency counters per virtual expert)
    const int nchH = (A.nbpH + kChunk - 1) / kChunk;
    const size_t qa_region = act_bytes(A.nbpF, kMaxCols);
    const size_t pbH = pair_bytes(A.nbpH), pbF = pair_bytes(A.nbpF);
    unsigned *sched = A.ws.sched;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rbar = smem_addr(&route_bar);
    if (warp == kProducerWarp) {
        route_warp(A.ids, A.wts, sched, N, n_all, A.L.E, R, blockIdx.x == 0 ? A.ws.err : nullptr, lane);
        mbar_arrive(rbar);
        const unsigned total_gu = (unsigned)(R.V * Gf);
        const unsigned total = total_gu + (unsigned)(R.V * Gd2);
        const unsigned set = R.epoch & 1u;
        const unsigned *dep_set = A.ws.dep + set * A.ws.dep_set;
        bool last = false;
        if (lane == 0) {
            Producer pr;
            bool tokens_ready = A.quant_tokens != 0;  // else the quantization kernel's output needs the wait
            unsigned base = blockIdx.x, grab = 1;  // first item: the CTA index
            while (base < total && !pr.stopped) {
                // the next grab: gate_up items one at a time, down items by
                // guided grabs of up to kDownGrab consecutive items of one
                // virtual expert, sized from where this CTA's last grab ended.
                // During a gate_up item it is fetched when the item starts (the
                // atomic's latency overlaps its stages); during down items, whose
                // stages wait on the gate_up results, only once their stages are
                // issued, so a CTA holding down items does not take more while
                // CTAs still on gate_up items will want them.
                const unsigned seen = base + grab;
                const unsigned ngrab = seen < total_gu ? 1u : max(1u, min(kDownGrab, (total - min(total, seen)) / (2u * gridDim.x)));
                const bool early = base < total_gu;
                unsigned nbase = early ? gridDim.x + atomicAdd(sched + kSchedFetch, ngrab) : 0u;
                for (unsigned it = base; it < min(total, base + grab) && !pr.stopped; ++it) {
                    if (it < total_gu) {
                        const int v = (int)it / Gf, g = (int)it - v * Gf;
                        const uint8_t *w = gate_up_of(A.L, R.vexp[v]) + (size_t)g * pbH;
                        if (A.ws.stall == 2 && blockIdx.x == 0 && pr.it == 0) {
                            // give-up test mode: CTA 0's first stage is claimed and
                            // tagged but never filled, so its consumers' wait runs out
                            pr.tag_only(S.pipe, (int)it);
                            continue;
                        }
                        if (!tokens_ready) {
                            pdl_wait();
                            asm volatile("fence.proxy.async.global;" ::: "memory");
                            tokens_ready = true;
                        }
                        const ActSlice act{A.ws.qh, A.quant_tokens ? 0 : A.n_tok};
                        Producer::NoDep nd;
                        pr.pass(S.pipe, w, A.nbpH, 0, nchH, (int)it, act, nd);
                    } else {
                        const int j = (int)(it - total_gu), v = j / Gd2, g = j - v * Gd2;
                        const uint8_t *w = down_of(A.L, R.vexp[v]) + (size_t)g * pbF;
                        const ActSlice act{A.ws.qa_bm + v * qa_region, R.vnc[v]};
                        DownDep dep{dep_set + (size_t)v * nsF, Gf, A.ws.stall, &S.pipe, vready, v};
                        pr.pass(S.pipe, w, A.nbpF, 0, nsF, (int)it, act, dep);
                    }
                }
                if (!early) nbase = gridDim.x + atomicAdd(sched + kSchedFetch, ngrab);
                base = nbase;
                grab = ngrab;
            }
            last = atomicAdd(sched + kSchedDone, 1u) == gridDim.x - 1;
            pr.finish(S.pipe);
            pr.drain(S.pipe);
        }
        if (__shfl_sync(0xffffffffu, last ? 1 : 0, 0)) {
            // every CTA of this launch has taken its last item and read the
            // epoch: zero the previous call's counter set, reset the item
            // counters, record this call's dependency words, advance the epoch
            const unsigned o = set ^ 1u;
            unsigned *dep_o = A.ws.dep + o * A.ws.dep_set;
            unsigned *pc_o = A.ws.pcnt + (size_t)o * Gd2;
            const unsigned used_o = sched[kSchedUsed + o];
            for (unsigned i = lane; i < used_o; i += 32) dep_o[i] = 0u;
            for (int i = lane; i < Gd2; i += 32) pc_o[i] = 0u;
            if (lane == 0) {
                sched[kSchedFetch] = 0u;
                sched[kSchedDone] = 0u;
                sched[kSchedUsed + set] = (unsigned)(R.V * nsF);
                sched[kSchedEpoch] = R.epoch + 1u;
            }
        }
    } else if (warp == kEpilogueWarp) {
        if (!pipe_wait(S.pipe, rbar, 0, true)) return;
        if (A.fuse_combine && R.V == 0 && blockIdx.x == 0) {  // no slot has an expert: y is zero
            for (int i = lane; i < A.n_tok * A.L.H; i += 32) A.y[i] = 0.0f;
        }
        const unsigned total_gu = (unsigned)(R.V * Gf);
        const unsigned set = R.epoch & 1u;
        unsigned *dep_set = A.ws.dep + set * A.ws.dep_set;
        unsigned *pcnt = A.ws.pcnt + (size_t)set * Gd2;
        SetReader rd;
        for (;;) {
            const int *tagp;
            const float *part;
            if (!rd.wait(S.pipe, tagp, part)) break;
            const int it = *(volatile const int *)tagp;
            if (it < 0) break;
            if ((unsigned)it < total_gu) {
                // gate sums in row set 0, up sums in row set 1 of every warp's slice
                const int v = it / Gf, g = it - v * Gf, nc = R.vnc[v];
                float gs[kMaxCols], us[kMaxCols];
#pragma unroll
                for (int c = 0; c < kMaxCols; ++c) {
                    gs[c] = us[c] = 0.0f;
                    if (c < nc) {
#pragma unroll
                        for (int w = 0; w < kConsumerWarps; ++w) {
                            gs[c] += part[(w * 2 * kMaxCols + c) * 32 + lane];
                            us[c] += part[(w * 2 * kMaxCols + kMaxCols + c) * 32 + lane];
                        }
                    }
                }
                rd.release(S.pipe);
                // block g of the intermediate: chunk c, block j of the chunk
                const int ca = g / kChunk, j = g - ca * kChunk, nblk = chunk_blocks(A.nbpF, ca);
                int8_t *base = A.ws.qa_bm + v * qa_region + act_chunk_offset(ca, nc);
#pragma unroll
                for (int c = 0; c < kMaxCols; ++c) {
                    if (c >= nc) continue;
                    const float a = A.swiglu ? gs[c] / (1.0f + expf(-gs[c])) * us[c] : gs[c] * us[c];
                    float d;
                    const int8_t q = quant_lane(a, d);
                    base[(size_t)(j * nc + c) * 32 + expander_pos(lane)] = q;
                    if (lane == 0)
                        *reinterpret_cast<float *>(base + (size_t)32 * nc * nblk + ((size_t)(j >> 1) * nc + c) * 8 +
                                                   (j & 1) * 4) = d;
                    if (A.ws.keep_a) {  // the intermediate by slot, in plain order (checking entry points)
                        const int p = R.vslot[v][c];
                        const size_t o = (size_t)p * A.L.F + (size_t)g * 32 + lane;
                        A.ws.a_dbg[o] = a;
                        A.ws.qa[o] = q;
                        if (lane == 0) A.ws.da[(size_t)p * A.nbF + g] = d;
                    }
                }
                __threadfence();
                __syncwarp();
                if (lane == 0) atomicAdd(dep_set + (size_t)v * nsF + g / kChunk, 1u);
            } else {
                // down outputs: row set r of column c, for i = 2c + r
                const int j = it - (int)total_gu, v = j / Gd2, g = j - v * Gd2, nc = R.vnc[v];
                float o[2 * kMaxCols];
#pragma unroll
                for (int i = 0; i < 2 * kMaxCols; ++i) {
                    o[i] = 0.0f;
                    if (i < 2 * nc) {
#pragma unroll
                        for (int w = 0; w < kConsumerWarps; ++w)
                            o[i] += part[(w * 2 * kMaxCols + (i & 1) * kMaxCols + (i >> 1)) * 32 + lane];
                    }
                }
                rd.release(S.pipe);
#pragma unroll
                for (int i = 0; i < 2 * kMaxCols; ++i) {
                    const int grp = 2 * g + (i & 1);
                    if (i < 2 * nc && grp < Gd)
                        A.ws.obuf[(size_t)R.vslot[v][i >> 1] * A.L.H + (size_t)grp * 32 + lane] = o[i];
                }
                if (!A.fuse_combine) continue;
                __threadfence();
                __syncwarp();
                unsigned done = 0;
                if (lane == 0) done = atomicAdd(pcnt + g, 1u);
                if (__shfl_sync(0xffffffffu, done, 0) == (unsigned)R.V - 1u) {
                    // all V virtual experts have written this group: y rows
                    // of both its 32-row groups (the one token)
                    __threadfence();
                    {
                        const int t = 0;
#pragma unroll
                        for (int r = 0; r < 2; ++r) {
                            const int grp = 2 * g + r;
                            if (grp >= Gd) continue;
                            const size_t row = (size_t)grp * 32 + lane;
                            const int p0 = t * A.k;
                            float ov[kMaxTopk];
#pragma unroll
                            for (int jj = 0; jj < kMaxTopk; ++jj) {
                                const int p = min(p0 + jj, kMaxSlots - 1);
                                ov[jj] = jj < A.k && R.ids[p] >= 0 ? __ldcg(A.ws.obuf + (size_t)p * A.L.H + row) : 0.0f;
                            }
                            const float osh = A.L.shared ? __ldcg(A.ws.obuf + (size_t)(N + t) * A.L.H + row) : 0.0f;
                            float acc = 0.0f;
#pragma unroll
                            for (int jj = 0; jj < kMaxTopk; ++jj) {
                                const int p = min(p0 + jj, kMaxSlots - 1);
                                if (jj < A.k && R.ids[p] >= 0) acc += R.w[p] * ov[jj];
                            }
                            A.y[(size_t)t * A.L.H + row] = acc + osh;
                        }
                    }
                }
            }
        }
    } else {
        if (A.quant_tokens) quant_stage_cols<1>(A.h, A.L.H, A.nbH, A.nbpH, S.act, S.dx, threadIdx.x, kConsumers);
        consumer_sync();
        if (!pipe_wait(S.pipe, rbar, 0, true)) return;
        const unsigned total_gu = (unsigned)(R.V * Gf);
        Consumer co(S.pipe);
        SetWriter wr;
        for (;;) {
            const int it = co.wait(S.pipe) ? co.tag(S.pipe) : -1;
            int *tagw;
            float *part;
            if (!wr.acquire(S.pipe, tagw, part)) break;
            if (it < 0) {
                if (threadIdx.x == 0) *tagw = -1;
                wr.publish(S.pipe);
                break;
            }
            const bool gu = (unsigned)it < total_gu;
            const int v = gu ? it / Gf : (it - (int)total_gu) / Gd2;
            const int nc = R.vnc[v], nbp = gu ? A.nbpH : A.nbpF;
            int col[kMaxCols];
            ActView V;
            if (!gu) {  // the stage's slice holds the virtual expert's columns
                V = ActView{nullptr, nullptr, nc, true};
#pragma unroll
                for (int c = 0; c < kMaxCols; ++c) col[c] = c;
            } else if (A.quant_tokens) {  // the one token, staged here
                V = ActView{S.act, S.dx, 1, false};
#pragma unroll
                for (int c = 0; c < kMaxCols; ++c) col[c] = 0;
            } else {  // the stage's slice holds every token: a column's slot is its token
                V = ActView{nullptr, nullptr, A.n_tok, true};
#pragma unroll
                for (int c = 0; c < kMaxCols; ++c) col[c] = c < nc ? slot_token(R.vslot[v][c], N, A.k) : 0;
            }
            const bool ok = sweep_b(co, S.pipe, 0, nbp, nbp, V, col, nc, part + warp * (2 * kMaxCols * 32), warp, lane);
            if (threadIdx.x == 0) *tagw = it;
            wr.publish(S.pipe);
            if (!ok) break;
        }
    }
}

// Router-weighted combine of a call with more than one token: y[t][r] =
// sum_j wts[t][j] * obuf[t*k+j][r], slots in order j = 0..k-1, slots with an
// out-of-range id skipped, then plus the shared expert's output obuf[N+t][r]
// when the layer has one (the sum the layer kernel forms itself for one
// token).  One thread per output; launched as a dependent of the layer
// kernel.  The ids and weights are inputs of the call, complete before its
// first kernel started, so they are read into shared memory before the wait;
// a token's k loads of obuf are then issued together.
__global__ void __launch_bounds__(256) k_moe_combine(const __grid_constant__ MoeArgs A) {
    __shared__ float w_s[kMaxSlots];  // router weight of each slot
    __shared__ int ok_s[kMaxSlots];   // slot has an in-range id
    const int N = A.n_tok * A.k;
    if ((int)threadIdx.x < N) {
        const int id = A.ids[threadIdx.x];
        ok_s[threadIdx.x] = id >= 0 && id < A.L.E;
        w_s[threadIdx.x] = A.wts[threadIdx.x];
    }
    __syncthreads();
    pdl_trigger();  // the next call's first kernel may launch; it waits for this grid
    pdl_wait();
    const int total = A.n_tok * A.L.H;
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < total; i += gridDim.x * blockDim.x) {
        const int t = i / A.L.H, r = i - t * A.L.H;
        const int p0 = t * A.k;
        float o[kMaxTopk];
#pragma unroll
        for (int j = 0; j < kMaxTopk; ++j) {
            const int p = min(p0 + j, kMaxSlots - 1);
            o[j] = j < A.k && ok_s[p] ? A.ws.obuf[(size_t)p * A.L.H + r] : 0.0f;
        }
        const float osh = A.L.shared ? A.ws.obuf[(size_t)(N + t) * A.L.H + r] : 0.0f;
        float v = 0.0f;
#pragma unroll
        for (int j = 0; j < kMaxTopk; ++j) {
            const int p = min(p0 + j, kMaxSlots - 1);
            if (j < A.k && ok_s[p]) v += w_s[p] * o[j];
        }
        A.y[i] = v + osh;
    }
}

cudaError_t launch_moe(const DevMoe &L, const MoeWork &ws, const float *h, int n_tok, const int32_t *ids,
                       const float *wts, int k, int swiglu, float *y, cudaStream_t s) {
    MoeArgs A;
    A.L = L;
    A.ws = ws;
    A.h = h;
    A.ids = ids;
    A.wts = wts;
    A.y = y;
    A.n_tok = n_tok;
    A.k = k;
    A.swiglu = swiglu;
    A.nbH = L.H / kQK;
    A.nbpH = round_up4(A.nbH);
    A.nbF = L.F / kQK;
    A.nbpF = round_up4(A.nbF);
    // one token: the layer kernel quantizes it (one launch fewer), as long as
    // its staging leaves room for the pipeline in shared memory
    A.quant_tokens = n_tok == 1 && ((uintptr_t)h & 15u) == 0 && A.nbpH <= kMaxStagedBlocks;
    A.fuse_combine = n_tok == 1;
    cudaError_t e = cudaSuccess;
    if (ws.ev[0] && (e = cudaEventRecord(ws.ev[0], s)) != cudaSuccess) return e;
    if (!A.quant_tokens) {
        e = launch_quantize_chunked(h, L.H, n_tok, ws.qh, s);
        if (e != cudaSuccess) return e;
    }
    if (ws.ev[1] && (e = cudaEventRecord(ws.ev[1], s)) != cudaSuccess) return e;
    {
        // four stages when two CTAs per SM still fit, else three
        const int act_blocks = A.quant_tokens ? A.nbpH : 0;
        int grid = 0, sms = 0, per_sm = 0;
        A.stages = 4;
        size_t smem = moe_smem_bytes(act_blocks, A.stages);
        e = resident(k_moe, kPipeThreads, smem, &sms, &per_sm);
        if (e != cudaSuccess) return e;
        if (per_sm < 2) {
            A.stages = 3;
            smem = moe_smem_bytes(act_blocks, A.stages);
        }
        const int64_t n_all = (int64_t)n_tok * k + (L.shared ? n_tok : 0);
        e = dynamic_grid(k_moe, smem, n_all * (L.F / 32 + (L.H / 32 + 1) / 2), &grid);
        if (e != cudaSuccess) return e;
        e = launch_k(k_moe, grid, kPipeThreads, smem, s, true, A);
        if (e != cudaSuccess) return e;
    }
    if (!A.fuse_combine) {
        const int grid = (int)std::min<int64_t>(((int64_t)n_tok * L.H + 255) / 256, 1024);
        e = launch_k(k_moe_combine, grid, 256, 0, s, true, A);
        if (e != cudaSuccess) return e;
    }
    if (ws.ev[2]) e = cudaEventRecord(ws.ev[2], s);
    return e;
}

// --------------------------------------------------- weight converter ----

// The codebook levels (a constant of the format), ascending with the index,
// and the half-sums of neighbours, (L_j + L_{j+1}) / 2: the boundaries of the
// nearest-level cells in units of the scale.
constexpr int8_t kLevels[16] = {-127, -104, -83, -65, -49, -35, -22, -10, 1, 13, 25, 38, 53, 69, 89, 113};
struct HalfSums {
    float h[15];
    constexpr HalfSums() : h() {
        for (int j = 0; j < 15; ++j) h[j] = 0.5f * (float)(kLevels[j] + kLevels[j + 1]);
    }
};
__constant__ HalfSums kHalf = HalfSums();

// Nearest level of w for scale dw: the reconstructions dw*L_j are monotone in
// j, so the nearest one is the number of cell boundaries |dw|*H_j, H_j =
// (L_j+L_{j+1})/2, that lie strictly below sign(dw)*w -- on a boundary (equal
// distances) that gives the lower index.  Every boundary is exact in fp32 (an
// 11-bit scale times a half-integer of at most 8 bits), so comparing with it
// decides exactly.  A candidate count comes from an approximate scaled value
// u = 2*s/|dw| and the table cnt[t] = #{j : 2*H_j <= t} at t = ceil(u) - 1
// (the boundaries are half-integers); the approximation can only misplace s
// across one boundary (they lie at least 5.5 scale units apart), which the
// exact comparisons with the candidate's two boundaries (hpair[c]: H_{c-1},
// H_c, infinite at the ends) put right.  dw == 0: every level reconstructs
// 0, index 0.
constexpr int kCntLo = -232, kCntHi = 202;  // t range of the table: below -231 count 0, from 202 on count 15
struct LevelTables {
    unsigned char cnt[kCntHi - kCntLo + 1];
    float2 hpair[16];
};

__device__ __forceinline__ void level_tables_init(LevelTables &T) {
    for (int i = threadIdx.x; i < kCntHi - kCntLo + 1; i += blockDim.x) {
        int n = 0;
        for (int j = 0; j < 15; ++j) n += (int)(2.0f * kHalf.h[j]) <= i + kCntLo;
        T.cnt[i] = (unsigned char)n;
    }
    if (threadIdx.x < 16) {
        const int c = threadIdx.x;
        T.hpair[c] = make_float2(c > 0 ? kHalf.h[c - 1] : -INFINITY, c < 15 ? kHalf.h[c] : INFINITY);
    }
}

__device__ __forceinline__ unsigned nearest_level(const LevelTables &T, float w, float dw, float r2) {
    const float adw = fabsf(dw), s = dw > 0.0f ? w : -w;
    int t = __float2int_ru(s * r2) - 1;
    t = min(max(t, kCntLo), kCntHi);
    const int c = T.cnt[t - kCntLo];
    const float2 hp = T.hpair[c];
    const int n = c - (__fmul_rn(adw, hp.x) < s ? 0 : 1) + (__fmul_rn(adw, hp.y) < s ? 1 : 0);
    return dw == 0.0f ? 0u : (unsigned)n;
}

// fp32 weights to 18-byte codebook blocks, for nblocks consecutive blocks of
// 32 weights (a row-major M x K matrix is M*K/32 of them, in order).  Per
// block: m = the weight of largest magnitude (the first among equal ones),
// dw = binary16(m / -127) (IEEE fp32 division, then rounding to nearest
// even), index_i = the nearest level of w_i; an all-zero block gives zero
// bytes.  A warp converts eight blocks per step: lane l holds elements
// 8l..8l+7 of the 256 (two 16-byte loads), four lanes per block; lanes 0-1 of
// a block hold its elements 0-15 (the low nibbles), lanes 2-3 elements 16-31.
// Two steps are loaded before either is converted.
__global__ void __launch_bounds__(256) k_quantize_weights(const float4 *__restrict__ w, int64_t nblocks,
                                                          uint8_t *__restrict__ out) {
    constexpr unsigned kFull = 0xffffffffu;
    __shared__ LevelTables T;
    level_tables_init(T);
    __syncthreads();
    const int lane = threadIdx.x & 31, gl = lane & 3;
    const int64_t warp = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    const int64_t steps = (nblocks + 7) / 8;
    auto convert = [&](int64_t st, float4 va, float4 vb) {
        const int64_t blk = st * 8 + (lane >> 2);
        const float x[8] = {va.x, va.y, va.z, va.w, vb.x, vb.y, vb.z, vb.w};
        float best = x[0];
        int pos = 8 * gl;
#pragma unroll
        for (int k = 1; k < 8; ++k)
            if (fabsf(x[k]) > fabsf(best)) {
                best = x[k];
                pos = 8 * gl + k;
            }
#pragma unroll
        for (int o = 1; o < 4; o <<= 1) {
            const float ob = __shfl_xor_sync(kFull, best, o);
            const int op = __shfl_xor_sync(kFull, pos, o);
            if (fabsf(ob) > fabsf(best) || (fabsf(ob) == fabsf(best) && op < pos)) {
                best = ob;
                pos = op;
            }
        }
        const unsigned short hb = best == 0.0f ? (unsigned short)0 : __half_as_ushort(__float2half_rn(best / -127.0f));
        const float dw = __half2float(__ushort_as_half(hb));
        const float r2 = __fdividef(2.0f, fabsf(dw));  // approximate: only picks the candidate
        unsigned mine[2];
#pragma unroll
        for (int h = 0; h < 2; ++h)
            mine[h] = nearest_level(T, x[4 * h], dw, r2) | nearest_level(T, x[4 * h + 1], dw, r2) << 8 |
                      nearest_level(T, x[4 * h + 2], dw, r2) << 16 | nearest_level(T, x[4 * h + 3], dw, r2) << 24;
        const unsigned high0 = __shfl_down_sync(kFull, mine[0], 2);  // elements 16 + 8gl.. of the block
        const unsigned high1 = __shfl_down_sync(kFull, mine[1], 2);
        if (blk < nblocks && gl < 2) {
            const unsigned w0 = mine[0] | high0 << 4, w1 = mine[1] | high1 << 4;
            uint8_t *o = out + blk * kBlockBytesCanonical;
            unsigned short *o16 = reinterpret_cast<unsigned short *>(o + 2 + 8 * gl);  // 2-byte aligned
            o16[0] = (unsigned short)(w0 & 0xFFFFu);
            o16[1] = (unsigned short)(w0 >> 16);
            o16[2] = (unsigned short)(w1 & 0xFFFFu);
            o16[3] = (unsigned short)(w1 >> 16);
            if (gl == 0) *reinterpret_cast<unsigned short *>(o) = hb;
        }
    };
    const float4 z = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    const int64_t n4 = nblocks * 8;  // float4s in all
    for (int64_t st = warp; st < steps; st += 2 * warps) {
        const int64_t st2 = st + warps;
        const int64_t e0 = st * 64 + 2 * lane, e1 = st2 * 64 + 2 * lane;  // block*8 + 2*gl
        const float4 a0 = e0 < n4 ? __ldg(w + e0) : z, b0 = e0 < n4 ? __ldg(w + e0 + 1) : z;
        const bool two = st2 < steps;
        const float4 a1 = two && e1 < n4 ? __ldg(w + e1) : z, b1 = two && e1 < n4 ? __ldg(w + e1 + 1) : z;
        convert(st, a0, b0);
        if (two) convert(st2, a1, b1);
    }
}

cudaError_t launch_quantize_weights(const float *w, int64_t nblocks, uint8_t *out, cudaStream_t s) {
    if (nblocks <= 0) return cudaSuccess;
    int sms = 0, per_sm = 0;
    cudaError_t e = resident(k_quantize_weights, 256, 0, &sms, &per_sm);
    if (e != cudaSuccess) return e;
    const int64_t steps = (nblocks + 7) / 8;
    const int64_t want = (steps + 15) / 16;  // two steps per warp per round, eight warps per CTA
    const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(want, (int64_t)sms * std::max(per_sm, 1)));
    k_quantize_weights<<<grid, 256, 0, s>>>(reinterpret_cast<const float4 *>(w), nblocks, out);
    return cudaGetLastError();
}

// ------------------------------------------------------ router top-k ------

// Routed-expert selection, one warp per token: the logits are staged in
// shared memory; k rounds each take the largest logit not yet taken (equal
// logits: the lower index), by a warp reduction over (value, index).  The
// weights are the softmax of the k selected logits, in fp64 (the differences
// of fp32 logits are exact there) and rounded once to fp32.
__global__ void __launch_bounds__(32) k_router_topk(const float *__restrict__ logits, int E, int k,
                                                    int32_t *__restrict__ ids, float *__restrict__ wts) {
    extern __shared__ __align__(128) unsigned char smem[];
    float *l = reinterpret_cast<float *>(smem);
    unsigned char *taken = smem + (size_t)E * sizeof(float);
    const int t = blockIdx.x, lane = threadIdx.x;
    const float *lt = logits + (size_t)t * E;
    for (int e = lane; e < E; e += 32) {
        l[e] = lt[e];
        taken[e] = 0;
    }
    __syncwarp();
    float sel[kMaxTopk];
    int pick[kMaxTopk];
#pragma unroll
    for (int j = 0; j < kMaxTopk; ++j) {
        sel[j] = 0.0f;
        pick[j] = 0;
        if (j >= k) continue;
        float bv = 0.0f;
        int bi = -1;
        for (int e = lane; e < E; e += 32)
            if (!taken[e] && (bi < 0 || l[e] > bv)) {  // ascending e: the first of equal values stays
                bv = l[e];
                bi = e;
            }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            if (oi >= 0 && (bi < 0 || ov > bv || (ov == bv && oi < bi))) {
                bv = ov;
                bi = oi;
            }
        }
        sel[j] = bv;
        pick[j] = bi;
        if (lane == 0) taken[bi] = 1;
        __syncwarp();
    }
    if (lane == 0) {
        double w[kMaxTopk], sum = 0.0;
#pragma unroll
        for (int j = 0; j < kMaxTopk; ++j) {
            w[j] = j < k ? exp((double)sel[j] - (double)sel[0]) : 0.0;
            sum += w[j];
        }
#pragma unroll
        for (int j = 0; j < kMaxTopk; ++j)
            if (j < k) {
                ids[(size_t)t * k + j] = pick[j];
                wts[(size_t)t * k + j] = (float)(w[j] / sum);
            }
    }
}

cudaError_t launch_router_topk(const float *logits, int n_tok, int E, int k, int32_t *ids, float *wts,
                               cudaStream_t s) {
    const size_t smem = (size_t)E * (sizeof(float) + 1);
    int sms = 0, per_sm = 0;
    cudaError_t e = resident(k_router_topk, 32, smem, &sms, &per_sm);
    if (e != cudaSuccess) return e;
    k_router_topk<<<n_tok, 32, smem, s>>>(logits, E, k, ids, wts);
    return cudaGetLastError();
}


}  // namespace cbq

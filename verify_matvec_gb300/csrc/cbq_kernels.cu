// cbq_kernels.cu -- sm_103a kernels of the codebook-4bit matvec and their
// launchers.
//
//   k_repack          canonical 18-byte blocks -> device layout (handle creation)
//   k_quantize        activation quantization, one warp per 32-value block
//   k_matvec<NC,F32>  dense MMVQ over NC <= 5 columns, one pass over the weights
//                     (F32: one fp32 column, quantized inside the kernel)
//   k_block_dots<NC>  the same integer path, exporting every per-block dot
//   k_moe             routed experts (and an optional shared expert), one
//                     kernel per layer call: gate+up rows, SwiGLU split,
//                     requantization, then down rows per slot
//   k_moe_combine     router-weighted combine of the per-slot down outputs
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
// Pipeline depth (stages of 18 KB per CTA, two CTAs per SM) and partial-sum
// sets of each kernel, sized so two CTAs fit in an SM's shared memory.
constexpr int kStages = 4;
constexpr int kSetsMatvec = 2;   // double-buffered
constexpr int kSetsMoe = 2;      // double-buffered, format B (two row sets)

// Dynamic shared memory of the routed-expert kernel with S stages.
size_t moe_smem_bytes(int act_blocks, int S) {
    return pipe_smem_bytes(S, act_blocks, kSetsMoe * kPartSetB);
}

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

__global__ void k_repack(const uint8_t *__restrict__ src, int64_t M, int nb, int nbp, uint4 *__restrict__ qs,
                         uint16_t *__restrict__ sc16) {
    const int64_t total = ((M + 31) / 32) * (int64_t)nbp * 32;
    const int nbq = nbp / 4;
    for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * blockDim.x) {
        const int lane = (int)(idx & 31);
        const int64_t gb = idx >> 5;
        const int b = (int)(gb % nbp);
        const int64_t g = gb / nbp;
        const int64_t row = g * 32 + lane;
        uint32_t w[4] = {0, 0, 0, 0};
        uint16_t scale = 0;
        if (row < M && b < nb) {
            const uint8_t *p = src + ((size_t)row * nb + b) * 18;
            scale = (uint16_t)(p[0] | (p[1] << 8));
#pragma unroll
            for (int i = 0; i < 4; ++i)
                w[i] = (uint32_t)p[2 + 4 * i] | ((uint32_t)p[3 + 4 * i] << 8) | ((uint32_t)p[4 + 4 * i] << 16) |
                       ((uint32_t)p[5 + 4 * i] << 24);
        }
        qs[idx] = make_uint4(w[0], w[1], w[2], w[3]);
        sc16[((g * nbq + b / 4) * 32 + lane) * 4 + (b & 3)] = scale;
    }
}

cudaError_t launch_repack(const uint8_t *src, int64_t M, int nb, uint4 *qs, uint2 *sc, cudaStream_t s) {
    const int nbp = round_up4(nb);
    const int64_t total = ((M + 31) / 32) * (int64_t)nbp * 32;
    const int grid = (int)std::min<int64_t>((total + 255) / 256, 65535);
    k_repack<<<grid, 256, 0, s>>>(src, M, nb, nbp, qs, reinterpret_cast<uint16_t *>(sc));
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

// ---------------------------------------------------------- dense MMVQ -----

size_t matvec_smem_bytes(int nbp, int n) { return pipe_smem_bytes(kStages, n * nbp, kSetsMatvec * kPartSetA); }

// Debug kernel smem: activations + scales only.
static size_t dots_smem_bytes(int nbp, int n) { return (size_t)n * nbp * 36; }

struct MatvecArgs {
    DevMat W;
    const int8_t *qx;  // quantized columns (kF32 == false)
    const float *dx;
    const float *xf;   // fp32 column (kF32 == true)
    int64_t K;
    float *y;
};

// Dense MMVQ: 32-row groups fetched per CTA, all NC columns per pass.
// kF32: the consumers quantize the fp32 column xf themselves while the
// producer starts the weight stream (no quantization kernel before it);
// otherwise they stage qx/dx written by the quantization kernel launched just
// before (a programmatic dependency).
template <int NC, bool kF32>
__global__ void __launch_bounds__(kPipeThreads, 2) k_matvec(const __grid_constant__ MatvecArgs A) {
    extern __shared__ __align__(128) unsigned char smem[];
    pdl_trigger();  // the next kernel may launch; it waits for this grid before touching what it writes
    const DevMat &W = A.W;
    const PipeSmem S = carve_pipe(smem, kStages, NC * W.nbp, W.err);
    pipe_init(S.pipe);
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nbq = W.nbp / 4;
    const unsigned total = (unsigned)W.G;
    if (warp == kConsumerWarps) {  // producer
        if (lane == 0) {
            Producer pr;
            // the first item is the CTA index (the grid never exceeds the item
            // count): its weights stream before the wait for the work ahead of
            // this kernel, which the work counter needs (a call still running
            // on the handle owns it)
            unsigned item = blockIdx.x;
            pr.group_a(S.pipe, W.qs + (size_t)item * W.nbp * 32, W.sc + (size_t)item * nbq * 32, 0, W.nbp, (int)item);
            pdl_wait();
            unsigned next = gridDim.x + atomicAdd(W.sched, 1u);
            while (next < total && !pr.stopped) {
                item = next;
                // the following item's index is fetched before this item's
                // stages are issued, so the atomic's latency overlaps them
                next = gridDim.x + atomicAdd(W.sched, 1u);
                pr.group_a(S.pipe, W.qs + (size_t)item * W.nbp * 32, W.sc + (size_t)item * nbq * 32, 0, W.nbp,
                           (int)item);
            }
            __threadfence();
            sched_exit(W.sched);
            pr.finish(S.pipe);
            pr.drain(S.pipe);
        }
        return;
    }
    pdl_wait();  // the activations belong to the work ahead
    if constexpr (kF32) {
        quant_stage_cols<NC>(A.xf, A.K, W.nb, W.nbp, S.act, S.dx, threadIdx.x, kConsumers);
    } else {
        ColSrc src{A.qx, A.dx, (size_t)A.K, (size_t)W.nb, {0, 1, 2, 3, 4}};
        stage_cols(src, NC, W.nb, W.nbp, S.act, S.dx, threadIdx.x, kConsumers, false, true);
    }
    consumer_sync();
    const float2 *dxp = reinterpret_cast<const float2 *>(S.dx);
    Consumer co(S.pipe);
    for (int n = 0;; ++n) {
        const int it = co.next_item(S.pipe);
        if (it < 0) break;
        float2 acc[NC];
#pragma unroll
        for (int c = 0; c < NC; ++c) acc[c] = make_float2(0.0f, 0.0f);
        sweep_a<NC>(co, S.pipe, 0, W.nbp, S.act, dxp, acc, warp, lane);
        float *part = S.part + (n & 1) * kPartSetA;
#pragma unroll
        for (int c = 0; c < NC; ++c) part[(warp * NC + c) * 32 + lane] = acc[c].x + acc[c].y;
        consumer_sync();
        if (warp < NC) {
            float v = 0.0f;
#pragma unroll
            for (int w = 0; w < kConsumerWarps; ++w) v += part[(w * NC + warp) * 32 + lane];
            const int64_t row = (int64_t)it * 32 + lane;
            if (row < W.M) A.y[(size_t)warp * W.M + row] = v;
        }
    }
}


template <int NC>
__global__ void __launch_bounds__(kThreads, 2)
    k_block_dots(const uint4 *__restrict__ qs, const uint2 *__restrict__ sc, int64_t M, int G, int nb, int nbp,
                 const int8_t *__restrict__ qx, int64_t K, int32_t *__restrict__ sdot, int chunk) {
    extern __shared__ __align__(128) unsigned char smem[];
    const int g0 = blockIdx.x * chunk;
    const int g1 = min(G, g0 + chunk);
    if (g0 >= G) return;
    uint4 *act_s = reinterpret_cast<uint4 *>(smem);
    float *dx_s = reinterpret_cast<float *>(act_s + (size_t)NC * nbp * 2);
    {
        // the activation scales do not enter the integer dots: stage zeros
        ColSrc src{qx, nullptr, (size_t)K, 0, {0, 1, 2, 3, 4}};
        stage_cols(src, NC, nb, nbp, act_s, dx_s, threadIdx.x, blockDim.x, false, true);
    }
    __syncthreads();
    __shared__ uint32_t consts[kConstWords];
    if (threadIdx.x == 0) write_consts(consts);
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nbq = nbp / 4;
    const int q0 = warp * nbq / kWarps, q1 = (warp + 1) * nbq / kWarps;
    const Codebook cb = read_consts(consts);
    for (int g = g0; g < g1; ++g) {
        const int64_t row = (int64_t)g * 32 + lane;
        for (int q = q0; q < q1; ++q) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int b = 4 * q + j;
                const uint4 w = ld_stream16(qs + ((size_t)g * nbp + b) * 32 + lane);
                int sd[NC];
                block_dots<NC>(cb, w, act_s + (size_t)b * NC * 2, sd);
                if (row < M && b < nb) {
#pragma unroll
                    for (int c = 0; c < NC; ++c) sdot[((size_t)c * M + row) * nb + b] = sd[c] - cb.seed;
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

template <int NC, bool kF32>
static cudaError_t launch_matvec_n(const DevMat &W, const int8_t *qx, const float *dx, const float *xf, float *y,
                                   cudaStream_t s, bool pdl) {
    const size_t smem = matvec_smem_bytes(W.nbp, NC);
    int grid = 0;
    cudaError_t e = dynamic_grid(k_matvec<NC, kF32>, smem, W.G, &grid);
    if (e != cudaSuccess) return e;
    MatvecArgs A;
    A.W = W;
    A.qx = qx;
    A.dx = dx;
    A.xf = xf;
    A.K = (int64_t)W.nb * kQK;
    A.y = y;
    return launch_k(k_matvec<NC, kF32>, grid, kPipeThreads, smem, s, pdl, A);
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
    k_block_dots<NC><<<grid, kThreads, smem, s>>>(W.qs, W.sc, W.M, W.G, W.nb, W.nbp, qx, (int64_t)W.nb * kQK, sdot,
                                                  chunk);
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

struct MoeArgs {
    DevMoe L;
    MoeWork ws;
    const float *h;
    const int32_t *ids;
    const float *wts;
    float *y;
    int n_tok, k, swiglu;
    int nbH, nbpH, nbF, nbpF;
    int act_blocks;    // staged-activation capacity in blocks (tokens, then down columns)
    int quant_tokens;  // the consumers quantize h themselves (one token, h 16-byte aligned)
    int stages;        // pipeline depth (3 or 4: as many as two CTAs per SM allow)
};

// Distinct in-range expert ids of the routing table, ascending but the shared
// expert first (its items, with a column for every token, are the slowest:
// handed out first, they do not form the tail of a pass), computed
// redundantly by every CTA from the <= 85 slots (no host round trip).  Slots
// 0..N-1 are the routed ones (p = t*k + j); with a shared expert, slots
// N..N+n_tok-1 hold its virtual id E, one per token.  An out-of-range routed
// id is stored as -1, so it matches no expert, the shared one included.
struct Routing {
    int ids[kMaxSlots];
    int uniq[kMaxSlots];
    unsigned char first[kMaxSlots];
    int D;
};

__device__ void route(const int32_t *__restrict__ ids, int N, int n_all, int E, Routing &R, unsigned *err) {
    const int t = threadIdx.x;
    if (t < n_all) {
        int e = E;  // a shared-expert slot
        if (t < N) {
            e = ids[t];
            if (e < 0 || e >= E) {
                if (err) atomicOr(err, kErrBadExpertId);
                e = -1;
            }
        }
        R.ids[t] = e;
    }
    __syncthreads();
    if (t < n_all) {
        const int e = R.ids[t];
        int f = e >= 0 ? 1 : 0;
        for (int p = 0; p < t; ++p)
            if (R.ids[p] == e) f = 0;
        R.first[t] = (unsigned char)f;
    }
    __syncthreads();
    if (t < n_all && R.first[t]) {
        auto key = [E](int e) { return e == E ? -1 : e; };
        const int kt = key(R.ids[t]);
        int rank = 0;
        for (int p = 0; p < n_all; ++p)
            if (R.first[p] && key(R.ids[p]) < kt) ++rank;
        R.uniq[rank] = R.ids[t];
    }
    if (t == 0) {
        int D = 0;
        for (int p = 0; p < n_all; ++p) D += R.first[p];
        R.D = D;
    }
    __syncthreads();
}

// Token of slot p: routed slots are t*k + j, shared-expert slots N + t.
__device__ __forceinline__ int slot_token(int p, int N, int k) { return p < N ? p / k : p - N; }

// Weights of expert e, the shared expert for e == E.
struct ExpertMat {
    const uint4 *qs;
    const uint2 *sc;
};

__device__ __forceinline__ ExpertMat gate_up_of(const DevMoe &L, int e) {
    if (e < L.E) return {L.gu_qs + (size_t)e * L.gu_qs_stride, L.gu_sc + (size_t)e * L.gu_sc_stride};
    return {L.sh_gu_qs, L.sh_gu_sc};
}

__device__ __forceinline__ ExpertMat down_of(const DevMoe &L, int e) {
    if (e < L.E) return {L.dn_qs + (size_t)e * L.dn_qs_stride, L.dn_sc + (size_t)e * L.dn_sc_stride};
    return {L.sh_dn_qs, L.sh_dn_sc};
}

// Slots of expert e (ascending) found by one warp with ballots over the
// routing table, without shared state or a CTA barrier: returns the slot
// count and the slots with ranks c0..c0+kMaxCols-1 in sl[] (-1 past the end).
struct Slots {
    int ns;
    int sl[kMaxCols];
};

__device__ __forceinline__ Slots warp_slots(const Routing &R, int e, int N, int c0, int lane) {
    Slots S;
    S.ns = 0;
#pragma unroll
    for (int c = 0; c < kMaxCols; ++c) S.sl[c] = -1;
    for (int base = 0; base < N; base += 32) {
        const bool hit = base + lane < N && R.ids[base + lane] == e;
        unsigned mask = __ballot_sync(0xffffffffu, hit);
        while (mask) {
            const int p = base + __ffs(mask) - 1;
            mask &= mask - 1;
            const int r = S.ns++ - c0;
#pragma unroll
            for (int c = 0; c < kMaxCols; ++c)
                if (r == c) S.sl[c] = p;
        }
    }
    return S;
}

// Number of slots of expert uniq[u] (any thread, from the routing table).
__device__ __forceinline__ int expert_ns(const Routing &R, int u, int N) {
    const int e = R.uniq[u];
    int ns = 0;
    for (int p = 0; p < N; ++p) ns += R.ids[p] == e;
    return ns;
}

__device__ __forceinline__ int col_chunks(int ns) { return (ns + kMaxCols - 1) / kMaxCols; }

constexpr unsigned kErrDependencyTimeout = 0x200u;
constexpr unsigned kDownGrab = 4;

__device__ __forceinline__ unsigned ld_acquire(const unsigned *p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Bounded wait (thread 0) for expert rank u's intermediate columns: all its
// gate_up items published (done[u] == target).  On timeout it sets
// kErrDependencyTimeout and the CTA's abort flag; it returns false then, or
// at once when the CTA already gave up.
__device__ __forceinline__ bool wait_dependency(const unsigned *done, unsigned target, const Pipe &P) {
    if (ld_acquire(done) >= target) return true;
    const uint64_t t0 = global_ns();
    for (;;) {
        if (*(volatile int *)P.abort) return false;
        __nanosleep(64);
        if (ld_acquire(done) >= target) return true;
        if (global_ns() - t0 > kWaitLimitNs) break;
    }
    atomicOr(P.err, kErrDependencyTimeout);
    *(volatile int *)P.abort = 1;
    return false;
}

// The whole routed-expert layer but the combine, in one persistent kernel.
// Work items, handed out in this order (the first per CTA is its index, the
// rest come from one counter):
//   it <  D*Gf : gate_up item (expert rank u, 32-row-pair group g), u-major:
//                gate rows 32g.. and up rows F+32g.. in one format-B pass,
//                then the SwiGLU split and the requantization of the 32
//                outputs of each column;
//   it >= D*Gf : down item (expert rank u, 64-row group g: 32-row groups 2g
//                and 2g+1), u-major, per-slot outputs to obuf.
// A CTA takes a down item only after every gate_up item has been taken, and
// taken gate_up items never wait, so a down item's wait for its expert's
// intermediate (done[u] == Gf * ns) always ends; it is bounded all the same.
// The producer streams a down item's weights before that wait ends.
// Launched as a programmatic dependent either way.  With one token (quantized
// here) this is the call's first kernel: it sets up its pipeline, then waits
// for all earlier work before it reads anything or lets the combine start.
// Otherwise it follows the quantization kernel, which starts it only once all
// earlier work has ended, so the routing table and the handle's counters are
// read before the wait for the quantized tokens.
__global__ void __launch_bounds__(kPipeThreads, 2) k_moe(const __grid_constant__ MoeArgs A) {
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ Routing R;
    __shared__ int dep_ok;
    const PipeSmem S = carve_pipe(smem, A.stages, A.act_blocks, A.ws.err);
    pipe_init(S.pipe);
    if (A.quant_tokens) pdl_wait();
    pdl_trigger();  // the combine kernel may launch; it waits for this grid
    const int N = A.n_tok * A.k + (A.L.shared ? A.n_tok : 0);  // routed slots, then shared ones
    route(A.ids, A.n_tok * A.k, N, A.L.E, R, blockIdx.x == 0 ? A.ws.err : nullptr);  // ends with a CTA barrier
    const int Gf = A.L.F / 32, Gd = A.L.H / 32, Gd2 = (Gd + 1) / 2;
    const unsigned total_gu = (unsigned)(R.D * Gf);
    const unsigned total = total_gu + (unsigned)(R.D * Gd2);
    unsigned *sched = A.ws.sched;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (warp == kConsumerWarps) {  // producer
        if (lane == 0) {
            Producer pr;
            const int nbqH = A.nbpH / 4, nbqF = A.nbpF / 4;
            unsigned base = blockIdx.x, grab = 1;  // first item: the CTA index
            while (base < total && !pr.stopped) {
                // the next grab (gate_up items one at a time; down items by
                // guided grabs of up to kDownGrab consecutive items of one
                // expert, which share staged columns) is fetched before this
                // one's stages are issued, so the atomic's latency overlaps them
                const unsigned seen = gridDim.x + *(volatile unsigned *)sched;
                const unsigned ngrab = seen < total_gu ? 1u : max(1u, min(kDownGrab, (total - seen) / (2u * gridDim.x)));
                const unsigned nbase = seen < total ? gridDim.x + atomicAdd(sched, ngrab) : total;
                for (unsigned it = base; it < min(total, base + grab) && !pr.stopped; ++it) {
                    if (it < total_gu) {
                        const int u = (int)it / Gf, g = (int)it - u * Gf;
                        const ExpertMat w = gate_up_of(A.L, R.uniq[u]);
                        const size_t ga = (size_t)g, gb = (size_t)g + Gf;
                        const int nch = col_chunks(expert_ns(R, u, N));
                        for (int ch = 0; ch < nch; ++ch) {
                            if (A.ws.stall == 2 && blockIdx.x == 0 && pr.it == 0) {
                                // give-up test mode: CTA 0's first stage is claimed and
                                // tagged but never filled, so its consumers' wait runs out
                                pr.tag_only(S.pipe, (int)it);
                                continue;
                            }
                            pr.group_b(S.pipe, w.qs + ga * A.nbpH * 32, w.sc + ga * nbqH * 32, w.qs + gb * A.nbpH * 32,
                                       w.sc + gb * nbqH * 32, A.nbpH, (int)it);
                        }
                    } else {
                        const int j = (int)(it - total_gu);
                        const int u = j / Gd2, g = j - u * Gd2;
                        const ExpertMat w = down_of(A.L, R.uniq[u]);
                        const size_t ga = 2 * (size_t)g, gb = ga + 1;
                        const bool two = (int)gb < Gd;
                        const int nch = col_chunks(expert_ns(R, u, N));
                        for (int ch = 0; ch < nch; ++ch)
                            pr.group_b(S.pipe, w.qs + ga * A.nbpF * 32, w.sc + ga * nbqF * 32,
                                       two ? w.qs + gb * A.nbpF * 32 : nullptr, w.sc + gb * nbqF * 32, A.nbpF,
                                       (int)it);
                    }
                }
                base = nbase;
                grab = ngrab;
            }
            __threadfence();
            sched_exit(sched);
            pr.finish(S.pipe);
            pr.drain(S.pipe);
        }
        return;
    }
    // consumers: stage the quantized tokens, quantizing one token here or
    // reading those of the quantization kernel launched just before
    if (A.quant_tokens) {
        quant_stage_cols<1>(A.h, A.L.H, A.nbH, A.nbpH, S.act, S.dx, threadIdx.x, kConsumers);
    } else {
        pdl_wait();
        ColSrc src{A.ws.qh, A.ws.dh, (size_t)A.L.H, (size_t)A.nbH, {0, 1, 2, 3, 4}};
        stage_cols(src, A.n_tok, A.nbH, A.nbpH, S.act, S.dx, threadIdx.x, kConsumers);
    }
    consumer_sync();
    Consumer co(S.pipe);
    int staged_u = -1, n = 0;
    bool dead = false;  // a dependency wait gave up: no later item computes or writes
    for (;;) {
        const int it = co.next_item(S.pipe);
        if (it < 0) break;
        const bool gu = (unsigned)it < total_gu;
        int u, g;
        if (gu) {
            u = it / Gf;
            g = it - u * Gf;
        } else {
            const int j = it - (int)total_gu;
            u = j / Gd2;
            g = j - u * Gd2;
        }
        const int e = R.uniq[u];
        for (int c0 = 0;; c0 += kMaxCols, ++n) {
            const Slots sl = warp_slots(R, e, N, c0, lane);
            const int nc = min(kMaxCols, sl.ns - c0);
            int col_off[kMaxCols];
            if (gu) {
#pragma unroll
                for (int c = 0; c < kMaxCols; ++c)
                    col_off[c] = (c < nc ? slot_token(sl.sl[c], A.n_tok * A.k, A.k) : 0) * A.nbpH;
            } else {
#pragma unroll
                for (int c = 0; c < kMaxCols; ++c) col_off[c] = c * A.nbpF;
                if (staged_u != u || sl.ns > kMaxCols) {
                    consumer_sync();  // the tokens (or the previous columns) are no longer read
                    if (threadIdx.x == 0)  // wait for expert u's intermediate
                        dep_ok = !dead && wait_dependency(A.ws.done + u, A.ws.stall == 1 ? ~0u : (unsigned)(Gf * sl.ns),
                                                          S.pipe);
                    consumer_sync();
                    dead = dead || !dep_ok;
                    if (!dead) {
                        ColSrc src{A.ws.qa, A.ws.da, (size_t)A.L.F, (size_t)A.nbF, {}};
#pragma unroll
                        for (int c = 0; c < kMaxCols; ++c) src.row[c] = max(sl.sl[c], 0);
                        stage_cols(src, nc, A.nbF, A.nbpF, S.act, S.dx, threadIdx.x, kConsumers, true);
                    }
                    consumer_sync();
                    staged_u = u;
                }
            }
            float *P0 = S.part + (n & 1) * kPartSetB;
            sweep_b(co, S.pipe, gu ? A.nbpH : A.nbpF, S.act, S.dx, col_off, nc, P0 + warp * (2 * kMaxCols * 32),
                    !dead, warp, lane);
            consumer_sync();
            if (!dead && gu && warp < nc) {
                // SwiGLU split and requantization of column `warp`: gate sums in
                // row set 0, up sums in row set 1 of every warp's slice
                const int c = warp;
                float gs = 0.0f, us = 0.0f;
#pragma unroll
                for (int w = 0; w < kConsumerWarps; ++w) {
                    gs += P0[(w * 2 * kMaxCols + c) * 32 + lane];
                    us += P0[(w * 2 * kMaxCols + kMaxCols + c) * 32 + lane];
                }
                const float a = A.swiglu ? gs / (1.0f + expf(-gs)) * us : gs * us;
                float d;
                const int8_t q = quant_lane(a, d);
                const int p = pick(sl.sl, c);
                const size_t o = (size_t)p * A.L.F + (size_t)g * 32 + lane;
                A.ws.qa[o] = q;
                if (lane == 0) A.ws.da[(size_t)p * A.nbF + g] = d;
                if (A.ws.keep_a) A.ws.a_dbg[o] = a;
                __threadfence();
                __syncwarp();
                if (lane == 0) atomicAdd(A.ws.done + u, 1u);
            } else if (!dead && !gu) {
                // down outputs: row set r of column c, for i = 2c + r
                for (int i = warp; i < 2 * nc; i += kConsumerWarps) {
                    const int c = i >> 1, r = i & 1;
                    float v = 0.0f;
#pragma unroll
                    for (int w = 0; w < kConsumerWarps; ++w) v += P0[(w * 2 * kMaxCols + r * kMaxCols + c) * 32 + lane];
                    const int grp = 2 * g + r;
                    if (grp < Gd) A.ws.obuf[(size_t)pick(sl.sl, c) * A.L.H + (size_t)grp * 32 + lane] = v;
                }
            }
            if (c0 + kMaxCols >= sl.ns) break;
        }
        ++n;
    }
    // the last CTA to finish resets the per-expert counts for the next call
    consumer_sync();
    if (threadIdx.x == 0) {
        __threadfence();
        if (atomicAdd(A.ws.sched + 2, 1u) == gridDim.x - 1) {
            for (int u = 0; u < R.D; ++u) A.ws.done[u] = 0u;
            A.ws.sched[2] = 0u;
        }
    }
}

// Router-weighted combine: y[t][r] = sum_j wts[t][j] * obuf[t*k+j][r], slots
// in order j = 0..k-1, slots with an out-of-range id skipped, then plus the
// shared expert's output obuf[N+t][r] when the layer has one.  One thread per
// output; launched as a dependent of the layer kernel.  The ids and weights
// are inputs of the call, complete before its first kernel started, so they
// are read into shared memory before the wait; a token's k loads of obuf are
// then issued together.
constexpr int kMaxTopk = 16;  // routed experts per token (the ABI's limit)

__global__ void __launch_bounds__(256) k_moe_combine(const __grid_constant__ MoeArgs A) {
    __shared__ float w_s[kMaxSlots];  // router weight of each slot, 0 for a skipped slot
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
    // one token: the layer kernel quantizes it (one launch fewer)
    A.quant_tokens = n_tok == 1 && ((uintptr_t)h & 15u) == 0;
    A.act_blocks = std::max((A.quant_tokens ? 1 : n_tok) * A.nbpH, kMaxCols * A.nbpF);
    cudaError_t e = cudaSuccess;
    if (ws.ev[0] && (e = cudaEventRecord(ws.ev[0], s)) != cudaSuccess) return e;
    if (!A.quant_tokens) {
        e = launch_quantize(h, L.H, n_tok, ws.qh, ws.dh, s);
        if (e != cudaSuccess) return e;
    }
    const int64_t max_experts = std::min(n_tok * k, L.E) + (L.shared ? 1 : 0);
    const int64_t items = max_experts * (L.F / 32 + (L.H / 32 + 1) / 2);
    {
        // four stages when two CTAs per SM still fit, else three
        int grid = 0, sms = 0, per_sm = 0;
        A.stages = 4;
        size_t smem = moe_smem_bytes(A.act_blocks, A.stages);
        e = resident(k_moe, kPipeThreads, smem, &sms, &per_sm);
        if (e != cudaSuccess) return e;
        if (per_sm < 2) {
            A.stages = 3;
            smem = moe_smem_bytes(A.act_blocks, A.stages);
        }
        e = dynamic_grid(k_moe, smem, items, &grid);
        if (e != cudaSuccess) return e;
        e = launch_k(k_moe, grid, kPipeThreads, smem, s, true, A);
        if (e != cudaSuccess) return e;
    }
    if (ws.ev[1] && (e = cudaEventRecord(ws.ev[1], s)) != cudaSuccess) return e;
    {
        const int grid = (int)std::min<int64_t>(((int64_t)n_tok * L.H + 255) / 256, 1024);
        e = launch_k(k_moe_combine, grid, 256, 0, s, true, A);
        if (e != cudaSuccess) return e;
    }
    if (ws.ev[2]) e = cudaEventRecord(ws.ev[2], s);
    return e;
}

// ------------------------------------------------------ router top-k ------

// Routed-expert selection, one warp per token: the logits are staged in
// shared memory; k rounds each take the largest logit not yet taken (equal
// logits: the lower index), by a warp reduction over (value, index).  The
// weights are the softmax of the k selected logits, in fp64 (the differences
// of fp32 logits are exact there) and rounded once to fp32.
__global__ void __launch_bounds__(32) k_router_topk(const float *__restrict__ logits, int E, int k,
                                                    int32_t *__restrict__ ids, float *__restrict__ wts) {
    extern __shared__ __align__(16) unsigned char smem[];
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

cudaError_t moe_smem_limit(size_t *bytes) {
    size_t optin = 0;
    cudaFuncAttributes fa;
    cudaError_t e = device_smem_limit(&optin);
    if (e == cudaSuccess) e = cudaFuncGetAttributes(&fa, k_moe);
    *bytes = e == cudaSuccess ? optin - fa.sharedSizeBytes : 0;
    return e;
}


}  // namespace cbq

// cbq_device.cuh -- device building blocks of the codebook-4bit matvec.
//
// Device layout of one matrix (built by the repack kernel from canonical
// blocks): rows are taken in groups of 32; for group g and block column b the
// 32 rows' 16-byte index fields are contiguous (qs[(g*nbp + b)*32 + lane]), so
// a warp whose lane l owns row 32g+l reads 512 contiguous bytes per block, and
// a whole group's K range is one contiguous span (bulk-copied by the pipeline
// of cbq_pipe.cuh).  The fp16 scales sit in a separate stream, four
// consecutive blocks of one row per 8-byte word (sc[(g*nbq + q)*32 + lane]).
// nbp = K/32 rounded up to a multiple of 4; padded blocks and rows carry a
// zero scale and zero indices.
//
// The hot loop per block and column: expand the 32 nibble indices through the
// 16-level int8 codebook with byte permutes (the role of the pages'
// codebook-16 expander, "fix(ggml): make ROCmFP4 codebook self-contained on
// CUDA"), take the exact int32 block dot with dp4a against the int8
// activations (MMVQ vecdot), and accumulate dw * dx * s in fp32.
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

namespace cbq {

constexpr int kQK = 32;
constexpr int kWarps = 8;           // warps per CTA of the matvec kernels
constexpr int kThreads = kWarps * 32;
constexpr int kMaxCols = 5;
// Codebook bytes packed four per word, index order.
//   {-127,-104,-83,-65} {-49,-35,-22,-10} {1,13,25,38} {53,69,89,113}
constexpr uint32_t kCb0 = 0xBFAD9881u;
constexpr uint32_t kCb1 = 0xF6EADDCFu;
constexpr uint32_t kCb2 = 0x26190D01u;
constexpr uint32_t kCb3 = 0x71594535u;
// Upper eight levels plus one: {2,14,26,39} {54,70,90,114} (see expand_split).
constexpr uint32_t kCbP0 = 0x271A0E02u;
constexpr uint32_t kCbP1 = 0x725A4636u;

// The codebook words and the dp4a seed (kMagicBits, below), held in registers
// for a whole kernel.  They are read from shared memory, where thread 0 wrote
// them at kernel start: built from immediates, the assembler would rebuild
// each one into a register before every permute and dp4a that uses it (about
// 13 extra instructions per 32-weight block, measured with per-pipe counters).
struct Codebook {
    uint32_t t0, t1, t2, t3, p0, p1;
    int seed;
};

// float(s) for |s| < 2^22 without an int->float conversion: the dp4a chain
// starts from the bit pattern of 1.5*2^23, so the integer sum s lands in the
// mantissa; subtracting 1.5*2^23 in fp32 is exact.
constexpr int kMagicBits = 0x4B400000;
constexpr float kMagic = 12582912.0f;

// Shared-memory words of the codebook and seed (Codebook); write_consts by one
// thread, then a barrier, then read_consts by every thread that needs them.
__device__ __forceinline__ void write_consts(uint32_t *s) {
    s[0] = kCb0;
    s[1] = kCb1;
    s[2] = kCb2;
    s[3] = kCb3;
    s[4] = kCbP0;
    s[5] = kCbP1;
    s[6] = (uint32_t)kMagicBits;
}

__device__ __forceinline__ Codebook read_consts(const uint32_t *s) {
    return Codebook{s[0], s[1], s[2], s[3], s[4], s[5], (int)s[6]};
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    // Generic-mode prmt: selector nibble bits 0-2 pick one of the 8 bytes of
    // {b,a}; bit 3 set replaces it by its sign replicated over the byte.
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

// Programmatic dependent launch.  A kernel launched with programmatic stream
// serialization may start while the previous kernel of the stream still
// runs; pdl_wait() blocks until that kernel has completed and its writes are
// visible (a no-op for a normal launch).  pdl_trigger() lets the next kernel
// of the stream start launching.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ uint4 ld_stream16(const uint4 *p) {
    uint4 r;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
        : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
    return r;
}

__device__ __forceinline__ uint2 ld_stream8(const uint2 *p) {
    uint2 r;
    asm("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];" : "=r"(r.x), "=r"(r.y) : "l"(p));
    return r;
}

__device__ __forceinline__ float half_lo(uint32_t v) {
    return __half2float(__ushort_as_half((unsigned short)(v & 0xFFFFu)));
}
__device__ __forceinline__ float half_hi(uint32_t v) {
    return __half2float(__ushort_as_half((unsigned short)(v >> 16)));
}

// ---------------------------------------------------------------------------
// Codebook expansion.  One 32-bit index word w (index bytes 4m..4m+3) holds,
// nibble by nibble, the indices of elements 4m, 4m+16, 4m+1, 4m+17, 4m+2,
// 4m+18, 4m+3, 4m+19.  A byte permute uses the low 16 bits of its selector,
// so w and w>>16 each select four codebook bytes in that element order; the
// activations are staged in the matching order (stage_cols below).
//
// expand_select: exact codebook bytes.  Two permutes look the low three index
// bits up in the lower and upper eight levels; a third, in sign mode, turns
// index bit 3 into a byte mask that picks between them.  11 ALU ops per word.
__device__ __forceinline__ void expand_select(const Codebook &cb, uint32_t w, uint32_t &e0, uint32_t &e1) {
    const uint32_t s = w & 0x77777777u;
    const uint32_t a = w << 4;               // bit 3 of even nibbles -> byte sign bits
    const uint32_t m0 = prmt(a, w, 0xD9C8u); // masks of nibbles 0..3
    const uint32_t m1 = prmt(a, w, 0xFBEAu); // masks of nibbles 4..7
    const uint32_t s1 = s >> 16;
    const uint32_t l0 = prmt(cb.t0, cb.t1, s), h0 = prmt(cb.t2, cb.t3, s);
    const uint32_t l1 = prmt(cb.t0, cb.t1, s1), h1 = prmt(cb.t2, cb.t3, s1);
    e0 = (h0 & m0) | (l0 & ~m0);
    e1 = (h1 & m1) | (l1 & ~m1);
}

// expand_split: two words whose byte-wise SUM is the codebook byte.  With the
// raw index as selector, the lower-level table yields the level for indices
// 0..7 and, in sign mode, -1 for 8..15 (all lower levels are negative).  With
// bit 3 flipped, the upper table (levels + 1, all positive) yields level+1 for
// 8..15 and 0 for 0..7.  The dot is then dp4a(lo,x) + dp4a(hi,x): 7 ALU ops
// and two dp4a per word and column -- cheaper for one or two columns.
__device__ __forceinline__ void expand_split(const Codebook &cb, uint32_t w, uint32_t &lo0, uint32_t &hi0,
                                             uint32_t &lo1, uint32_t &hi1) {
    const uint32_t f = w ^ 0x88888888u;
    lo0 = prmt(cb.t0, cb.t1, w);
    hi0 = prmt(cb.p0, cb.p1, f);
    lo1 = prmt(cb.t0, cb.t1, w >> 16);
    hi1 = prmt(cb.p0, cb.p1, f >> 16);
}

template <int NC>
struct UseSplit { static constexpr bool value = NC == 1; };

// Exact int32 block dots (offset by kMagicBits) of one index block against NC
// permuted activation blocks: column c's two words at actb[2c], actb[2c+1]
// (the block-major staging below puts a block's columns side by side).
template <int NC>
__device__ __forceinline__ void block_dots(const Codebook &cb, const uint4 w, const uint4 *actb, int sdot[NC]) {
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
    if constexpr (UseSplit<NC>::value) {
        uint32_t lo[8], hi[8];
#pragma unroll
        for (int m = 0; m < 4; ++m) expand_split(cb, ws[m], lo[2 * m], hi[2 * m], lo[2 * m + 1], hi[2 * m + 1]);
#pragma unroll
        for (int c = 0; c < NC; ++c) {
            const uint4 a0 = actb[2 * c], a1 = actb[2 * c + 1];
            const uint32_t av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
            int s = cb.seed;  // one chain over the lower- and upper-table parts
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                s = __dp4a((int)lo[i], (int)av[i], s);
                s = __dp4a((int)hi[i], (int)av[i], s);
            }
            sdot[c] = s;
        }
    } else {
        uint32_t e[8];
#pragma unroll
        for (int m = 0; m < 4; ++m) expand_select(cb, ws[m], e[2 * m], e[2 * m + 1]);
#pragma unroll
        for (int c = 0; c < NC; ++c) {
            const uint4 a0 = actb[2 * c], a1 = actb[2 * c + 1];
            const uint32_t av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
            int s = cb.seed;
#pragma unroll
            for (int i = 0; i < 8; ++i) s = __dp4a((int)e[i], (int)av[i], s);
            sdot[c] = s;
        }
    }
}

// One column, two rows: the dots (offset by the seed) of index blocks wa
// (row set 0) and wb (row set 1) against the activation block at actb[0..1],
// by the two-word expansion; the activation words are loaded once for both.
__device__ __forceinline__ void block_dots_2rows(const Codebook &cb, const uint4 wa, const uint4 wb,
                                                 const uint4 *actb, int &sa, int &sb) {
    const uint4 a0 = actb[0], a1 = actb[1];
    const uint32_t av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
    const uint32_t wsa[4] = {wa.x, wa.y, wa.z, wa.w}, wsb[4] = {wb.x, wb.y, wb.z, wb.w};
    int s0 = cb.seed, s1 = cb.seed;
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        uint32_t lo0, hi0, lo1, hi1;
        expand_split(cb, wsa[m], lo0, hi0, lo1, hi1);
        s0 = __dp4a((int)lo0, (int)av[2 * m], s0);
        s0 = __dp4a((int)hi0, (int)av[2 * m], s0);
        s0 = __dp4a((int)lo1, (int)av[2 * m + 1], s0);
        s0 = __dp4a((int)hi1, (int)av[2 * m + 1], s0);
        expand_split(cb, wsb[m], lo0, hi0, lo1, hi1);
        s1 = __dp4a((int)lo0, (int)av[2 * m], s1);
        s1 = __dp4a((int)hi0, (int)av[2 * m], s1);
        s1 = __dp4a((int)lo1, (int)av[2 * m + 1], s1);
        s1 = __dp4a((int)hi1, (int)av[2 * m + 1], s1);
    }
    sa = s0;
    sb = s1;
}

// Two columns, two rows: index blocks wa (row set 0) and wb (row set 1), each
// expanded once (exact bytes), dotted with the activation blocks of two
// columns (their words at a0[0..1] and a1[0..1]).
__device__ __forceinline__ void block_dots_2rows_cols2(const Codebook &cb, const uint4 wa, const uint4 wb,
                                                       const uint4 *a0, const uint4 *a1, int sa[2], int sb[2]) {
    const uint32_t wsa[4] = {wa.x, wa.y, wa.z, wa.w}, wsb[4] = {wb.x, wb.y, wb.z, wb.w};
    uint32_t ea[8], eb[8];
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        expand_select(cb, wsa[m], ea[2 * m], ea[2 * m + 1]);
        expand_select(cb, wsb[m], eb[2 * m], eb[2 * m + 1]);
    }
    const uint4 *ap[2] = {a0, a1};
#pragma unroll
    for (int c = 0; c < 2; ++c) {
        const uint4 x0 = ap[c][0], x1 = ap[c][1];
        const uint32_t av[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
        int s0 = cb.seed, s1 = cb.seed;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            s0 = __dp4a((int)ea[i], (int)av[i], s0);
            s1 = __dp4a((int)eb[i], (int)av[i], s1);
        }
        sa[c] = s0;
        sb[c] = s1;
    }
}

// Byte position of element r (0..31) of a block in the expander order of the
// staged activations (stage_cols): word 2m+h holds elements 4m+2h, 4m+2h+16,
// 4m+2h+1, 4m+2h+17.
__device__ __forceinline__ int expander_pos(int r) {
    const int e = r & 15, m = e >> 2, i = e & 3;
    return 8 * m + 4 * (i >> 1) + 2 * (i & 1) + (r >> 4);
}

// Scaled accumulation of two consecutive blocks' dots of one column:
// acc += (dw0*dx0 * s0, dw1*dx1 * s1) with the packed fp32x2 pipe; the same
// three roundings per block as a scalar multiply, add and fused multiply-add.
__device__ __forceinline__ float2 scale_acc2(float2 acc, float2 dw, float2 dx, int sa, int sb) {
    const float2 s = __fadd2_rn(make_float2(__int_as_float(sa), __int_as_float(sb)), make_float2(-kMagic, -kMagic));
    return __ffma2_rn(__fmul2_rn(dw, dx), s, acc);
}

// v[c] for a run-time c < kMaxCols, by a compare chain: the array stays in
// registers (a dynamic index would place it in local memory).
__device__ __forceinline__ int pick(const int (&v)[kMaxCols], int c) {
    int r = v[0];
#pragma unroll
    for (int cc = 1; cc < kMaxCols; ++cc)
        if (c == cc) r = v[cc];
    return r;
}

// Sources of the activation columns to stage: column c is row row[c] of a
// row-major int8 matrix q (qstride bytes per row, rows 16-byte aligned) and of
// its fp32 block-scale matrix d (dstride floats per row; d == nullptr stages
// zero scales).
static_assert(kMaxCols == 5, "ColSrc initialisers list five rows");
struct ColSrc {
    const int8_t *q;
    const float *d;
    size_t qstride, dstride;
    int row[kMaxCols];
};

// Stage activation columns into shared memory in the expander's element
// order.  Blocks nb..nbp-1 are zero (nbp even).  Threads tid = 0..nthr-1
// share the work.  Layouts (act_s in uint4 pairs, one pair per block):
//   column-major (block_major == false): block b of column c at pair c*nbp + b,
//     its scale at dx_s[c*nbp + b];
//   block-major: block b of column c at pair b*ncols + c, its scale at
//     dx_s[((b/2)*ncols + c)*2 + b%2] (a float2 per column and block pair).
// With one column the two coincide.  With l2_only the loads bypass L1 (data
// written by other CTAs of the same kernel).
__device__ __forceinline__ void stage_cols(const ColSrc &src, int ncols, int nb, int nbp, uint4 *act_s,
                                           float *dx_s, int tid, int nthr, bool l2_only = false,
                                           bool block_major = false) {
    for (int idx = tid; idx < ncols * nbp; idx += nthr) {
        const int c = idx / nbp, b = idx - c * nbp;
        const int ai = block_major ? b * ncols + c : idx;
        const int di = block_major ? ((b >> 1) * ncols + c) * 2 + (b & 1) : idx;
        uint4 o0 = make_uint4(0, 0, 0, 0), o1 = o0;
        float d = 0.0f;
        if (b < nb) {
            const size_t r = (size_t)pick(src.row, c);
            const uint4 *p = reinterpret_cast<const uint4 *>(src.q + r * src.qstride + (size_t)b * kQK);
            const uint4 x0 = l2_only ? __ldcg(p) : p[0], x1 = l2_only ? __ldcg(p + 1) : p[1];
            const uint32_t P[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
            // word 2m   = x[4m], x[4m+16], x[4m+1], x[4m+17]
            // word 2m+1 = x[4m+2], x[4m+18], x[4m+3], x[4m+19]
            o0.x = prmt(P[0], P[4], 0x5140u); o0.y = prmt(P[0], P[4], 0x7362u);
            o0.z = prmt(P[1], P[5], 0x5140u); o0.w = prmt(P[1], P[5], 0x7362u);
            o1.x = prmt(P[2], P[6], 0x5140u); o1.y = prmt(P[2], P[6], 0x7362u);
            o1.z = prmt(P[3], P[7], 0x5140u); o1.w = prmt(P[3], P[7], 0x7362u);
            if (src.d) {
                const float *dp = src.d + r * src.dstride + b;
                d = l2_only ? __ldcg(dp) : *dp;
            }
        }
        act_s[(size_t)ai * 2] = o0;
        act_s[(size_t)ai * 2 + 1] = o1;
        dx_s[di] = d;
    }
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// The activation quantization rule on one 32-value block held one value per
// lane: d = max|v|/127 (IEEE fp32 division), q = rint(v/d) clamped, q = 0
// when d == 0.
__device__ __forceinline__ int8_t quant_lane(float v, float &d_out) {
    const float amax = warp_max(fabsf(v));
    const float d = amax / 127.0f;
    d_out = d;
    if (d == 0.0f) return 0;
    float q = rintf(v / d);
    q = fminf(fmaxf(q, -127.0f), 127.0f);
    return (int8_t)q;
}

// Quantize NC fp32 columns (x[c*K ..], 16-byte aligned) straight into the
// block-major staged layout of stage_cols, by thread pairs: the even thread
// of a pair holds values 0..15 of a block, the odd thread 16..31 (four 16-byte
// loads each).  Same rule and bits as quant_lane: d = max|v|/127 in IEEE fp32
// division (the max over the pair is exact in any order), q = rint(v/d)
// clamped, q = 0 when d == 0.  Expander order: word 2m+h of a block holds
// values 4m+2h, 4m+2h+16, 4m+2h+1, 4m+2h+17, i.e. the pair (4m+2h, 4m+2h+1)
// of each thread, even thread's bytes at 0 and 2.  Blocks nb..nbp-1 are zero.
// Threads tid = 0..nthr-1 (nthr even) share the work.
template <int NC>
__device__ __forceinline__ void quant_stage_cols(const float *__restrict__ x, int64_t K, int nb, int nbp,
                                                 uint4 *act_s, float *dx_s, int tid, int nthr) {
    const int half = tid & 1;
    // the loop test reads the pair index of lane 0, so a warp runs the same
    // number of rounds (its shuffles are full-warp); past the end a pair idles
    for (int k = tid >> 1; k - ((tid & 31) >> 1) < NC * nb; k += nthr >> 1) {
        const bool live = k < NC * nb;
        const int c = k / nb, b = k - c * nb;
        float v[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = 0.0f;
        if (live) {
            const float4 *src = reinterpret_cast<const float4 *>(x + (size_t)c * K + (size_t)b * kQK + half * 16);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float4 f = src[i];
                v[4 * i] = f.x;
                v[4 * i + 1] = f.y;
                v[4 * i + 2] = f.z;
                v[4 * i + 3] = f.w;
            }
        }
        float amax = 0.0f;
#pragma unroll
        for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
        const float d = amax / 127.0f;
        uint32_t pr[4];  // pr[u] = pairs 2u (low half) and 2u+1 (high half) of this thread
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            uint32_t w = 0;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                float q = 0.0f;
                if (d != 0.0f) q = fminf(fmaxf(rintf(v[4 * u + e] / d), -127.0f), 127.0f);
                w |= ((uint32_t)(int)q & 0xFFu) << (8 * e);
            }
            pr[u] = w;
        }
        // the even thread builds words 0..3 (pairs 0..3), the odd thread 4..7
        const uint32_t give0 = half ? pr[0] : pr[2], give1 = half ? pr[1] : pr[3];
        const uint32_t got0 = __shfl_xor_sync(0xffffffffu, give0, 1);
        const uint32_t got1 = __shfl_xor_sync(0xffffffffu, give1, 1);
        const uint32_t own0 = half ? pr[2] : pr[0], own1 = half ? pr[3] : pr[1];
        const uint32_t e0 = half ? got0 : own0, o0 = half ? own0 : got0;  // even / odd thread's pairs
        const uint32_t e1 = half ? got1 : own1, o1 = half ? own1 : got1;
        const uint4 out = make_uint4(prmt(e0, o0, 0x5140u), prmt(e0, o0, 0x7362u), prmt(e1, o1, 0x5140u),
                                     prmt(e1, o1, 0x7362u));
        if (live) {
            const int ai = b * NC + c;
            act_s[(size_t)ai * 2 + half] = out;
            if (!half) dx_s[((b >> 1) * NC + c) * 2 + (b & 1)] = d;
        }
    }
    for (int k = tid; k < NC * (nbp - nb); k += nthr) {  // padded blocks
        const int c = k / (nbp - nb), b = nb + k - c * (nbp - nb);
        const int ai = b * NC + c;
        act_s[(size_t)ai * 2] = make_uint4(0, 0, 0, 0);
        act_s[(size_t)ai * 2 + 1] = make_uint4(0, 0, 0, 0);
        dx_s[((b >> 1) * NC + c) * 2 + (b & 1)] = 0.0f;
    }
}

}  // namespace cbq

// cbq_hc.cu -- Sinkhorn normalisation of the hyper-connection mixing
// matrices: the "register-resident sinkhorn kernel" of the fused DS4
// hyper-connection op (GGML_OP_DS4_HC, "feat(ds4): add DSpark speculative
// runtime + optimizations" #496), whose NHC = 4 specialisation keeps the
// matrix in registers instead of spilling it ("fix(ds4): keep ROCmFPX
// generation byte-safe" #494).  The pages give neither the iteration count
// nor the update; the plain reading of a Sinkhorn normalisation is used:
//   P = exp(c - max c) for the NHC x NHC logits c of one token;
//   `iters` rounds of: every row divided by its sum, then every column by its
//   sum (sums in index order);
//   out = P after the last column step.
// Here "divided by its sum" is a multiplication by the hardware's
// approximate reciprocal of the sum (rcp.approx: within 1 ulp; the sums that
// occur lie between e^-80 and 4, normal numbers).  An error in a row's or a
// column's factor is a diagonal scaling, which the next step removes; the
// result is checked against an fp64 evaluation within a bound that allows
// for every rounding.
#include <stdint.h>

#include "cbq_device.cuh"
#include "cbq_internal.h"

namespace cbq {

__device__ __forceinline__ float rcp_approx(float x) {
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

// One thread per matrix: its NHC*NHC entries stay in registers for all the
// rounds; a thread reads its whole matrix before it writes any of it, so the
// call may work in place.  Matrices are row-major and contiguous (NHC*NHC
// floats each); the loads and stores are 16-byte vectors (NHC = 4: one row
// per vector).  The entries are held as pairs of neighbours in a row, so the
// scaling of a row and the sums and scaling of two columns at once run on the
// packed fp32x2 pipe (each lane of a packed operation rounds like the scalar
// one, in the same order: the results are those of the scalar rounds).
template <int NHC>
__global__ void __launch_bounds__(128) k_hc_sinkhorn(const float *logits, int64_t n, int iters, float *out) {
    static_assert(NHC % 4 == 0, "rows are moved as float4 vectors");
    constexpr int kV = NHC / 4;   // float4 vectors per row
    constexpr int kP = NHC / 2;   // column pairs
    pdl_trigger();  // the next kernel may launch; it waits for this grid before it reads what it writes
    const int64_t m = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (m >= n) return;
    pdl_wait();     // the logits may come from the kernel ahead of this one
    const float4 *src = reinterpret_cast<const float4 *>(logits + m * NHC * NHC);
    float2 Q[NHC][kP];  // Q[r][p] = (P[r][2p], P[r][2p+1])
#pragma unroll
    for (int r = 0; r < NHC; ++r)
#pragma unroll
        for (int v = 0; v < kV; ++v) {
            const float4 q = src[r * kV + v];  // plain loads: out may be logits itself
            Q[r][2 * v] = make_float2(q.x, q.y);
            Q[r][2 * v + 1] = make_float2(q.z, q.w);
        }
    float cmax = Q[0][0].x;
#pragma unroll
    for (int r = 0; r < NHC; ++r)
#pragma unroll
        for (int p = 0; p < kP; ++p) cmax = fmaxf(cmax, fmaxf(Q[r][p].x, Q[r][p].y));
#pragma unroll
    for (int r = 0; r < NHC; ++r)
#pragma unroll
        for (int p = 0; p < kP; ++p) Q[r][p] = make_float2(expf(Q[r][p].x - cmax), expf(Q[r][p].y - cmax));
    for (int t = 0; t < iters; ++t) {
#pragma unroll
        for (int r = 0; r < NHC; ++r) {  // rows: the sum in index order, then one packed scaling per pair
            float s = Q[r][0].x;
            s = __fadd_rn(s, Q[r][0].y);
#pragma unroll
            for (int p = 1; p < kP; ++p) s = __fadd_rn(__fadd_rn(s, Q[r][p].x), Q[r][p].y);
            const float inv = rcp_approx(s);
            const float2 f = make_float2(inv, inv);
#pragma unroll
            for (int p = 0; p < kP; ++p) Q[r][p] = __fmul2_rn(Q[r][p], f);
        }
#pragma unroll
        for (int p = 0; p < kP; ++p) {  // columns 2p and 2p+1 together
            float2 s = Q[0][p];
#pragma unroll
            for (int r = 1; r < NHC; ++r) s = __fadd2_rn(s, Q[r][p]);
            const float2 f = make_float2(rcp_approx(s.x), rcp_approx(s.y));
#pragma unroll
            for (int r = 0; r < NHC; ++r) Q[r][p] = __fmul2_rn(Q[r][p], f);
        }
    }
    float4 *dst = reinterpret_cast<float4 *>(out + m * NHC * NHC);
#pragma unroll
    for (int r = 0; r < NHC; ++r)
#pragma unroll
        for (int v = 0; v < kV; ++v)
            dst[r * kV + v] = make_float4(Q[r][2 * v].x, Q[r][2 * v].y, Q[r][2 * v + 1].x, Q[r][2 * v + 1].y);
}

cudaError_t launch_hc_sinkhorn(const float *logits, int64_t n, int iters, float *out, cudaStream_t s) {
    if (n <= 0) return cudaSuccess;
    constexpr int kThreads = 128;
    // a programmatic dependent of the work ahead (its launch overlaps that
    // work; the kernel waits for it before reading the logits)
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((n + kThreads - 1) / kThreads));
    cfg.blockDim = dim3(kThreads);
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k_hc_sinkhorn<kHcNhc>, logits, n, iters, out);
}

}  // namespace cbq

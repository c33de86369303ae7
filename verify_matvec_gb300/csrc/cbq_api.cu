// cbq_api.cu -- the C ABI declared in include/cbq.h: handles, argument
// checks, device selection and launch sequencing.  No arithmetic of the
// method lives here; every step of the path runs in the kernels of
// cbq_kernels.cu.
#include "cbq.h"
#include "cbq_internal.h"

#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <new>

using cbq::DevMat;
using cbq::DevMoe;
using cbq::MoeWork;

struct cbq_weights {
    int device;
    DevMat mat;
    uint8_t *w;      // repacked weights (cbq_internal.h layout)
    unsigned *sched; // work counters of the matvec kernel
    unsigned *err;   // the handle's error word
    int8_t *ws_qx;   // CBQ_MAX_COLS x K
    float *ws_dx;    // CBQ_MAX_COLS x K/32
    float *st_x;     // host-entry staging: CBQ_MAX_COLS x K fp32
    float *st_y;     // CBQ_MAX_COLS x M fp32
    int8_t *mq_qx;   // tensor-core path: CBQ_MAX_MMQ_COLS x K
    float *mq_dx;    // CBQ_MAX_MMQ_COLS x K/32
    uint8_t *mq_b;   // its B tiles (1 KB per block)
    float *mq_meta;  // its block metadata
    int mq_stall;    // give-up test mode of the tensor-core path (cbq_debug_mmq_stall)
    int64_t K;
    int64_t bytes;
};

struct cbq_moe {
    int device;
    DevMoe L;
    uint8_t *gu, *dn;        // repacked experts, one after another
    uint8_t *sh_gu, *sh_dn;  // shared expert (null when unset)
    int64_t sh_bytes;
    MoeWork ws;
    float *st_h;      // CBQ_MAX_TOKENS x H
    int32_t *st_ids;  // kMaxSlots
    float *st_wts;    // kMaxSlots
    float *st_y;      // CBQ_MAX_TOKENS x H
    int64_t bytes;
};

namespace {

thread_local char t_last_error[256] = "";

int cuda_fail(cudaError_t e, const char *where) {
    snprintf(t_last_error, sizeof t_last_error, "%s: %s (%d)", where, cudaGetErrorString(e), (int)e);
    return CBQ_ECUDA;
}

#define CBQ_CUDA(call)                                        \
    do {                                                      \
        cudaError_t e_ = (call);                              \
        if (e_ != cudaSuccess) return cuda_fail(e_, #call);   \
    } while (0)

class DeviceScope {
  public:
    explicit DeviceScope(int dev) {
        status_ = cudaGetDevice(&prev_);
        if (status_ == cudaSuccess && prev_ != dev) {
            status_ = cudaSetDevice(dev);
            changed_ = status_ == cudaSuccess;
        }
    }
    ~DeviceScope() {
        if (changed_) cudaSetDevice(prev_);
    }
    cudaError_t status() const { return status_; }

  private:
    int prev_ = 0;
    bool changed_ = false;
    cudaError_t status_ = cudaSuccess;
};

int check_device(int *dev) {
    cudaError_t e = cudaGetDevice(dev);
    if (e != cudaSuccess) {
        cuda_fail(e, "cudaGetDevice");
        return CBQ_EDEVICE;
    }
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, *dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, *dev) != cudaSuccess)
        return CBQ_EDEVICE;
    if (major != 10 || minor != 3) {
        snprintf(t_last_error, sizeof t_last_error, "device %d is sm_%d%d; this library is built for sm_103a",
                 *dev, major, minor);
        return CBQ_EDEVICE;
    }
    return CBQ_OK;
}

template <typename T>
int dev_alloc(T **p, size_t count, int64_t *bytes) {
    *p = nullptr;
    if (count == 0) return CBQ_OK;
    if (cudaMalloc((void **)p, count * sizeof(T)) != cudaSuccess) {
        cudaGetLastError();
        *p = nullptr;
        snprintf(t_last_error, sizeof t_last_error, "cudaMalloc of %zu bytes failed", count * sizeof(T));
        return CBQ_ENOMEM;
    }
    *bytes += (int64_t)(count * sizeof(T));
    return CBQ_OK;
}

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

cudaStream_t as_stream(void *s) { return reinterpret_cast<cudaStream_t>(s); }

// Repack canonical blocks (host or device) of an M x K matrix into w (split:
// the gate/up pairing of a gate_up matrix, 0 otherwise).
int repack_into(const void *blocks, int64_t M, int nb, int split, int on_device, uint8_t *w, cudaStream_t s) {
    const size_t nbytes = (size_t)M * (size_t)nb * CBQ_BLOCK_BYTES;
    const uint8_t *src = static_cast<const uint8_t *>(blocks);
    uint8_t *tmp = nullptr;
    if (!on_device) {
        if (cudaMalloc((void **)&tmp, nbytes) != cudaSuccess) {
            cudaGetLastError();
            return CBQ_ENOMEM;
        }
        cudaError_t e = cudaMemcpyAsync(tmp, blocks, nbytes, cudaMemcpyHostToDevice, s);
        if (e != cudaSuccess) {
            cudaFree(tmp);
            return cuda_fail(e, "cudaMemcpyAsync(blocks)");
        }
        src = tmp;
    }
    cudaError_t e = cbq::launch_repack(src, M, nb, split, w, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (tmp) cudaFree(tmp);
    if (e != cudaSuccess) return cuda_fail(e, "repack");
    return CBQ_OK;
}

}  // namespace

extern "C" {

const char *cbq_status_string(int status) {
    switch (status) {
        case CBQ_OK: return "CBQ_OK";
        case CBQ_EINVAL: return "CBQ_EINVAL: invalid argument";
        case CBQ_ECUDA: return "CBQ_ECUDA: CUDA error";
        case CBQ_ENOMEM: return "CBQ_ENOMEM: device allocation failed";
        case CBQ_EDEVICE: return "CBQ_EDEVICE: no usable sm_103 device";
        default: return "unknown cbq status";
    }
}

const char *cbq_last_cuda_error(void) { return t_last_error; }

// ------------------------------------------------------------ dense ------

int cbq_weights_destroy(cbq_weights *W) {
    if (!W) return CBQ_EINVAL;
    DeviceScope scope(W->device);
    cudaFree(W->w);
    cudaFree(W->sched);
    cudaFree(W->err);
    cudaFree(W->ws_qx);
    cudaFree(W->ws_dx);
    cudaFree(W->st_x);
    cudaFree(W->st_y);
    cudaFree(W->mq_qx);
    cudaFree(W->mq_dx);
    cudaFree(W->mq_b);
    cudaFree(W->mq_meta);
    delete W;
    return CBQ_OK;
}

int cbq_weights_create(const void *blocks, int64_t M, int64_t K, int on_device, void *stream, cbq_weights **out) {
    if (!out) return CBQ_EINVAL;
    *out = nullptr;
    if (!blocks || M < 1 || K < CBQ_QK || K % CBQ_QK != 0 || M > (int64_t)1 << 31 || K > (int64_t)1 << 20)
        return CBQ_EINVAL;
    int dev = 0;
    int rc = check_device(&dev);
    if (rc != CBQ_OK) return rc;
    const int nb = (int)(K / CBQ_QK);
    const int nbp = cbq::round_up4(nb);
    size_t smem_max = 0;
    CBQ_CUDA(cbq::matvec_smem_limit(&smem_max));
    if (cbq::matvec_smem_bytes(nbp, CBQ_MAX_COLS) > smem_max) return CBQ_EINVAL;

    const int G = (int)((M + 31) / 32);
    const int64_t P = cbq::mat_pairs(M);

    cbq_weights *W = new (std::nothrow) cbq_weights();
    if (!W) return CBQ_ENOMEM;
    W->device = dev;
    W->K = K;
    if ((rc = dev_alloc(&W->w, cbq::mat_bytes(M, nb), &W->bytes)) != CBQ_OK ||
        (rc = dev_alloc(&W->sched, 2, &W->bytes)) != CBQ_OK ||
        (rc = dev_alloc(&W->err, 1, &W->bytes)) != CBQ_OK ||
        (rc = dev_alloc(&W->ws_qx, (size_t)CBQ_MAX_COLS * K, &W->bytes)) != CBQ_OK ||
        (rc = dev_alloc(&W->ws_dx, (size_t)CBQ_MAX_COLS * nb, &W->bytes)) != CBQ_OK ||
        (rc = dev_alloc(&W->st_x, (size_t)CBQ_MAX_COLS * K, &W->bytes)) != CBQ_OK ||
        (rc = dev_alloc(&W->st_y, (size_t)CBQ_MAX_COLS * M, &W->bytes)) != CBQ_OK ||
        (rc = dev_alloc(&W->mq_qx, (size_t)CBQ_MAX_MMQ_COLS * K, &W->bytes)) != CBQ_OK ||
        (rc = dev_alloc(&W->mq_dx, (size_t)CBQ_MAX_MMQ_COLS * nb, &W->bytes)) != CBQ_OK ||
        (rc = dev_alloc(&W->mq_b, cbq::mmq_bimg_bytes(nb), &W->bytes)) != CBQ_OK ||
        (rc = dev_alloc(&W->mq_meta, cbq::mmq_meta_bytes(nb) / sizeof(float), &W->bytes)) != CBQ_OK) {
        cbq_weights_destroy(W);
        return rc;
    }
    if (cudaMemsetAsync(W->sched, 0, 2 * sizeof(unsigned), as_stream(stream)) != cudaSuccess ||
        cudaMemsetAsync(W->err, 0, sizeof(unsigned), as_stream(stream)) != cudaSuccess) {
        cbq_weights_destroy(W);
        return CBQ_ECUDA;
    }
    rc = repack_into(blocks, M, nb, 0, on_device, W->w, as_stream(stream));
    if (rc != CBQ_OK) {
        cbq_weights_destroy(W);
        return rc;
    }
    W->mat.w = W->w;
    W->mat.M = M;
    W->mat.nb = nb;
    W->mat.nbp = nbp;
    W->mat.G = G;
    W->mat.P = (int)P;
    W->mat.split = 0;
    W->mat.sched = W->sched;
    W->mat.err = W->err;
    *out = W;
    return CBQ_OK;
}

int cbq_weights_info(const cbq_weights *W, int64_t *M, int64_t *K, int64_t *device_bytes) {
    if (!W) return CBQ_EINVAL;
    if (M) *M = W->mat.M;
    if (K) *K = W->K;
    if (device_bytes) *device_bytes = W->bytes;
    return CBQ_OK;
}

int cbq_quantize_act(const float *x_dev, int64_t K, int n, int8_t *qx_dev, float *dx_dev, void *stream) {
    if (!x_dev || !qx_dev || !dx_dev || n < 1 || K < CBQ_QK || K % CBQ_QK != 0) return CBQ_EINVAL;
    CBQ_CUDA(cbq::launch_quantize(x_dev, K, n, qx_dev, dx_dev, as_stream(stream)));
    return CBQ_OK;
}

int cbq_matvec_q(const cbq_weights *W, const int8_t *qx_dev, const float *dx_dev, int n, float *y_dev,
                 void *stream) {
    if (!W || !qx_dev || !dx_dev || !y_dev || n < 1 || n > CBQ_MAX_COLS || !aligned16(qx_dev)) return CBQ_EINVAL;
    DeviceScope scope(W->device);
    CBQ_CUDA(scope.status());
    CBQ_CUDA(cbq::launch_matvec(W->mat, qx_dev, dx_dev, n, y_dev, as_stream(stream)));
    return CBQ_OK;
}

int cbq_matvec(const cbq_weights *W, const float *x_dev, int n, float *y_dev, void *stream) {
    if (!W || !x_dev || !y_dev || n < 1 || n > CBQ_MAX_COLS) return CBQ_EINVAL;
    DeviceScope scope(W->device);
    CBQ_CUDA(scope.status());
    cudaStream_t s = as_stream(stream);
    // one column: one launch, the matvec kernel quantizes x itself (with more
    // columns the separate quantization kernel, which spreads the divisions
    // over n*K threads, is faster)
    if (n == 1 && aligned16(x_dev)) {
        CBQ_CUDA(cbq::launch_matvec_f32(W->mat, x_dev, n, y_dev, s));
        return CBQ_OK;
    }
    CBQ_CUDA(cbq::launch_quantize(x_dev, W->K, n, W->ws_qx, W->ws_dx, s));
    CBQ_CUDA(cbq::launch_matvec(W->mat, W->ws_qx, W->ws_dx, n, y_dev, s, /*pdl=*/true));
    return CBQ_OK;
}

int cbq_matvec_host(const cbq_weights *W, const float *x_host, int n, float *y_host, void *stream) {
    if (!W || !x_host || !y_host || n < 1 || n > CBQ_MAX_COLS) return CBQ_EINVAL;
    DeviceScope scope(W->device);
    CBQ_CUDA(scope.status());
    cudaStream_t s = as_stream(stream);
    CBQ_CUDA(cudaMemcpyAsync(W->st_x, x_host, (size_t)n * W->K * sizeof(float), cudaMemcpyHostToDevice, s));
    int rc = cbq_matvec(W, W->st_x, n, W->st_y, stream);
    if (rc != CBQ_OK) return rc;
    CBQ_CUDA(cudaMemcpyAsync(y_host, W->st_y, (size_t)n * W->mat.M * sizeof(float), cudaMemcpyDeviceToHost, s));
    CBQ_CUDA(cudaStreamSynchronize(s));
    return CBQ_OK;
}

// ------------------------------------------------ allocation-free path ---

// Scratch of cbq_matvec_static: quantized activations (CBQ_MAX_COLS x
// CBQ_STATIC_SCRATCH_MAX_K int8) then their scales (CBQ_MAX_COLS x K/32
// fp32), one copy per device for the life of the library.
constexpr size_t kStaticQxBytes = (size_t)CBQ_MAX_COLS * CBQ_STATIC_SCRATCH_MAX_K;
constexpr size_t kStaticDxBytes = (size_t)CBQ_MAX_COLS * (CBQ_STATIC_SCRATCH_MAX_K / CBQ_QK) * sizeof(float);
static __device__ __align__(256) unsigned char g_static_scratch[kStaticQxBytes + kStaticDxBytes];

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_static_mu;
unsigned char *g_static_ptr[kMaxDevices] = {};  // device address per device, found on first use

// Device address of the scratch on the current device (looked up once per
// device; the host-side symbol is not a device address).
int static_scratch(int dev, unsigned char **out) {
    if (dev < 0 || dev >= kMaxDevices) return CBQ_EDEVICE;
    std::lock_guard<std::mutex> lock(g_static_mu);
    if (!g_static_ptr[dev]) {
        void *p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_static_scratch);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(g_static_scratch)");
        g_static_ptr[dev] = static_cast<unsigned char *>(p);
    }
    *out = g_static_ptr[dev];
    return CBQ_OK;
}
}  // namespace

int cbq_matvec_static(const cbq_weights *W, const float *x_dev, int n, float *y_dev, void *stream) {
    if (!W || !x_dev || !y_dev || n < 1 || n > CBQ_MAX_COLS || W->K > CBQ_STATIC_SCRATCH_MAX_K) return CBQ_EINVAL;
    DeviceScope scope(W->device);
    CBQ_CUDA(scope.status());
    unsigned char *scratch = nullptr;
    const int rc = static_scratch(W->device, &scratch);
    if (rc != CBQ_OK) return rc;
    int8_t *qx = reinterpret_cast<int8_t *>(scratch);
    float *dx = reinterpret_cast<float *>(scratch + kStaticQxBytes);
    cudaStream_t s = as_stream(stream);
    if (n == 1 && aligned16(x_dev)) {  // as cbq_matvec: one launch, no scratch
        CBQ_CUDA(cbq::launch_matvec_f32(W->mat, x_dev, n, y_dev, s));
        return CBQ_OK;
    }
    CBQ_CUDA(cbq::launch_quantize(x_dev, W->K, n, qx, dx, s));
    CBQ_CUDA(cbq::launch_matvec(W->mat, qx, dx, n, y_dev, s, /*pdl=*/true));
    return CBQ_OK;
}

int cbq_matmat(const cbq_weights *W, const float *x_dev, int n, float *y_dev, void *stream) {
    if (!W || !x_dev || !y_dev || n < 1 || n > CBQ_MAX_MMQ_COLS) return CBQ_EINVAL;
    DeviceScope scope(W->device);
    CBQ_CUDA(scope.status());
    cudaStream_t s = as_stream(stream);
    CBQ_CUDA(cbq::launch_quantize(x_dev, W->K, n, W->mq_qx, W->mq_dx, s));
    CBQ_CUDA(cbq::launch_mmq_prep(W->mq_qx, W->mq_dx, n, W->K, W->mq_b, W->mq_meta, s));
    CBQ_CUDA(cbq::launch_mmq(W->mat, W->mq_b, W->mq_meta, n, y_dev, nullptr, W->mq_stall, s));
    return CBQ_OK;
}

int cbq_debug_mmq_block_dots(const cbq_weights *W, const int8_t *qx_dev, int n, int32_t *s_dev, void *stream) {
    if (!W || !qx_dev || !s_dev || n < 1 || n > CBQ_MAX_MMQ_COLS) return CBQ_EINVAL;
    DeviceScope scope(W->device);
    CBQ_CUDA(scope.status());
    cudaStream_t s = as_stream(stream);
    CBQ_CUDA(cbq::launch_mmq_prep(qx_dev, nullptr, n, W->K, W->mq_b, W->mq_meta, s));
    CBQ_CUDA(cbq::launch_mmq(W->mat, W->mq_b, W->mq_meta, n, nullptr, s_dev, W->mq_stall, s));
    return CBQ_OK;
}

int cbq_debug_block_dots(const cbq_weights *W, const int8_t *qx_dev, int n, int32_t *s_dev, void *stream) {
    if (!W || !qx_dev || !s_dev || n < 1 || n > CBQ_MAX_COLS || !aligned16(qx_dev)) return CBQ_EINVAL;
    DeviceScope scope(W->device);
    CBQ_CUDA(scope.status());
    CBQ_CUDA(cbq::launch_block_dots(W->mat, qx_dev, n, s_dev, as_stream(stream)));
    return CBQ_OK;
}

// --------------------------------------------------------------- MoE -----

namespace {

// Frees the shared expert of L and stops the kernels from using it.
void drop_shared(cbq_moe *L) {
    cudaFree(L->sh_gu);
    cudaFree(L->sh_dn);
    L->sh_gu = L->sh_dn = nullptr;
    L->bytes -= L->sh_bytes;
    L->sh_bytes = 0;
    L->L.sh_gu = L->L.sh_dn = nullptr;
    L->L.shared = 0;
}

}  // namespace

int cbq_moe_destroy(cbq_moe *L) {
    if (!L) return CBQ_EINVAL;
    DeviceScope scope(L->device);
    drop_shared(L);
    cudaFree(L->gu);
    cudaFree(L->dn);
    cudaFree(L->ws.qh);
    cudaFree(L->ws.qa_bm);
    cudaFree(L->ws.dep);
    cudaFree(L->ws.pcnt);
    cudaFree(L->ws.qa);
    cudaFree(L->ws.da);
    cudaFree(L->ws.a_dbg);
    cudaFree(L->ws.obuf);
    cudaFree(L->ws.sched);
    cudaFree(L->ws.err);
    cudaFree(L->st_h);
    cudaFree(L->st_ids);
    cudaFree(L->st_wts);
    cudaFree(L->st_y);
    delete L;
    return CBQ_OK;
}

int cbq_moe_create(const void *gate_up, const void *down, int E, int64_t H, int64_t F, int on_device, void *stream,
                   cbq_moe **out) {
    if (!out) return CBQ_EINVAL;
    *out = nullptr;
    if (!gate_up || !down || E < 1 || H < CBQ_QK || F < CBQ_QK || H % CBQ_QK || F % CBQ_QK || H > (1 << 20) ||
        F > (1 << 20))
        return CBQ_EINVAL;
    int dev = 0;
    int rc = check_device(&dev);
    if (rc != CBQ_OK) return rc;
    const int nbH = (int)(H / CBQ_QK), nbF = (int)(F / CBQ_QK);

    cbq_moe *L = new (std::nothrow) cbq_moe();
    if (!L) return CBQ_ENOMEM;
    L->device = dev;
    const size_t gub = cbq::mat_bytes(2 * F, nbH), dnb = cbq::mat_bytes(H, nbF);
    const size_t slots = cbq::kMaxSlots;
    const size_t nbpH = (size_t)cbq::round_up4(nbH), nbpF = (size_t)cbq::round_up4(nbF);
    const size_t nsF = (nbpF + 15) / 16;  // down stages of 16 blocks
    const size_t gd2 = (size_t)(H / CBQ_QK + 1) / 2;  // 64-row output groups
    if ((rc = dev_alloc(&L->gu, gub * E, &L->bytes)) != CBQ_OK ||
        (rc = dev_alloc(&L->dn, dnb * E, &L->bytes)) != CBQ_OK ||
        (rc = dev_alloc(&L->ws.qh, cbq::act_bytes((int)nbpH, CBQ_MAX_TOKENS), &L->bytes)) != CBQ_OK ||
        (rc = dev_alloc(&L->ws.qa_bm, slots * cbq::act_bytes((int)nbpF, CBQ_MAX_COLS), &L->bytes)) != CBQ_OK ||
        (rc = dev_alloc(&L->ws.dep, 2 * slots * nsF, &L->bytes)) != CBQ_OK ||
        (rc = dev_alloc(&L->ws.pcnt, 2 * gd2, &L->bytes)) != CBQ_OK ||
        (rc = dev_alloc(&L->ws.qa, slots * F, &L->bytes)) != CBQ_OK ||
        (rc = dev_alloc(&L->ws.da, slots * nbF, &L->bytes)) != CBQ_OK ||
        (rc = dev_alloc(&L->ws.a_dbg, slots * F, &L->bytes)) != CBQ_OK ||
        (rc = dev_alloc(&L->ws.obuf, slots * H, &L->bytes)) != CBQ_OK ||
        (rc = dev_alloc(&L->ws.sched, 8, &L->bytes)) != CBQ_OK ||
        (rc = dev_alloc(&L->ws.err, 1, &L->bytes)) != CBQ_OK ||
        (rc = dev_alloc(&L->st_h, (size_t)CBQ_MAX_TOKENS * H, &L->bytes)) != CBQ_OK ||
        (rc = dev_alloc(&L->st_ids, slots, &L->bytes)) != CBQ_OK ||
        (rc = dev_alloc(&L->st_wts, slots, &L->bytes)) != CBQ_OK ||
        (rc = dev_alloc(&L->st_y, (size_t)CBQ_MAX_TOKENS * H, &L->bytes)) != CBQ_OK) {
        cbq_moe_destroy(L);
        return rc;
    }
    cudaStream_t s = as_stream(stream);
    // the intermediate's padded blocks are never written: zero keeps them finite
    if (cudaMemsetAsync(L->ws.sched, 0, 8 * sizeof(unsigned), s) != cudaSuccess ||
        cudaMemsetAsync(L->ws.dep, 0, 2 * slots * nsF * sizeof(unsigned), s) != cudaSuccess ||
        cudaMemsetAsync(L->ws.pcnt, 0, 2 * gd2 * sizeof(unsigned), s) != cudaSuccess ||
        cudaMemsetAsync(L->ws.qa_bm, 0, slots * cbq::act_bytes((int)nbpF, CBQ_MAX_COLS), s) != cudaSuccess ||
        cudaMemsetAsync(L->ws.err, 0, sizeof(unsigned), s) != cudaSuccess) {
        cbq_moe_destroy(L);
        return CBQ_ECUDA;
    }
    L->ws.dep_set = slots * nsF;
    const size_t gu_bytes = (size_t)2 * F * nbH * CBQ_BLOCK_BYTES;
    const size_t dn_bytes = (size_t)H * nbF * CBQ_BLOCK_BYTES;
    for (int e = 0; e < E; ++e) {
        rc = repack_into(static_cast<const uint8_t *>(gate_up) + e * gu_bytes, 2 * F, nbH, (int)(F / CBQ_QK),
                         on_device, L->gu + e * gub, s);
        if (rc == CBQ_OK)
            rc = repack_into(static_cast<const uint8_t *>(down) + e * dn_bytes, H, nbF, 0, on_device, L->dn + e * dnb,
                             s);
        if (rc != CBQ_OK) {
            cbq_moe_destroy(L);
            return rc;
        }
    }
    L->L.gu = L->gu;
    L->L.dn = L->dn;
    L->L.E = E;
    L->L.H = (int)H;
    L->L.F = (int)F;
    L->L.gu_stride = gub;
    L->L.dn_stride = dnb;
    *out = L;
    return CBQ_OK;
}

int cbq_moe_set_shared(cbq_moe *L, const void *gate_up, const void *down, int on_device, void *stream) {
    if (!L || !gate_up != !down) return CBQ_EINVAL;
    DeviceScope scope(L->device);
    CBQ_CUDA(scope.status());
    cudaStream_t s = as_stream(stream);
    CBQ_CUDA(cudaStreamSynchronize(s));  // no call of this stream may still read the old weights
    if (!gate_up) {
        drop_shared(L);
        return CBQ_OK;
    }
    const int64_t H = L->L.H, F = L->L.F;
    const int nbH = (int)(H / CBQ_QK), nbF = (int)(F / CBQ_QK);
    int rc = CBQ_OK;
    if (!L->sh_gu) {
        int64_t got = 0;
        if ((rc = dev_alloc(&L->sh_gu, cbq::mat_bytes(2 * F, nbH), &got)) != CBQ_OK ||
            (rc = dev_alloc(&L->sh_dn, cbq::mat_bytes(H, nbF), &got)) != CBQ_OK) {
            L->bytes += got;
            L->sh_bytes = got;
            drop_shared(L);
            return rc;
        }
        L->bytes += got;
        L->sh_bytes = got;
    }
    L->L.shared = 0;  // partly rewritten weights are never used
    rc = repack_into(gate_up, 2 * F, nbH, (int)(F / CBQ_QK), on_device, L->sh_gu, s);
    if (rc == CBQ_OK) rc = repack_into(down, H, nbF, 0, on_device, L->sh_dn, s);
    if (rc != CBQ_OK) {
        drop_shared(L);
        return rc;
    }
    L->L.sh_gu = L->sh_gu;
    L->L.sh_dn = L->sh_dn;
    L->L.shared = 1;
    return CBQ_OK;
}

int cbq_moe_info(const cbq_moe *L, int *E, int64_t *H, int64_t *F, int64_t *device_bytes) {
    if (!L) return CBQ_EINVAL;
    if (E) *E = L->L.E;
    if (H) *H = L->L.H;
    if (F) *F = L->L.F;
    if (device_bytes) *device_bytes = L->bytes;
    return CBQ_OK;
}

int cbq_moe_matvec(const cbq_moe *L, const float *h_dev, int n_tok, const int32_t *ids_dev, const float *wts_dev,
                   int topk, int swiglu, float *y_dev, void *stream) {
    if (!L || !h_dev || !ids_dev || !wts_dev || !y_dev || n_tok < 1 || n_tok > CBQ_MAX_TOKENS || topk < 1 ||
        topk > CBQ_MAX_TOPK || topk > L->L.E || (swiglu != 0 && swiglu != 1))
        return CBQ_EINVAL;
    DeviceScope scope(L->device);
    CBQ_CUDA(scope.status());
    CBQ_CUDA(cbq::launch_moe(L->L, L->ws, h_dev, n_tok, ids_dev, wts_dev, topk, swiglu, y_dev, as_stream(stream)));
    return CBQ_OK;
}

int cbq_router_topk(const float *logits_dev, int n_tok, int E, int topk, int32_t *ids_dev, float *wts_dev,
                    void *stream) {
    if (!logits_dev || !ids_dev || !wts_dev || n_tok < 1 || n_tok > 65535 || E < 1 || E > CBQ_ROUTER_MAX_E ||
        topk < 1 || topk > CBQ_MAX_TOPK || topk > E)
        return CBQ_EINVAL;
    int dev = 0;
    const int rc = check_device(&dev);
    if (rc != CBQ_OK) return rc;
    CBQ_CUDA(cbq::launch_router_topk(logits_dev, n_tok, E, topk, ids_dev, wts_dev, as_stream(stream)));
    return CBQ_OK;
}

int cbq_quantize_weights(const float *w_dev, int64_t M, int64_t K, void *blocks_dev, void *stream) {
    if (!w_dev || !blocks_dev || M < 1 || K < CBQ_QK || K % CBQ_QK || !aligned16(w_dev) ||
        (reinterpret_cast<uintptr_t>(blocks_dev) & 1u) || M > INT64_MAX / K)
        return CBQ_EINVAL;
    int dev = 0;
    const int rc = check_device(&dev);
    if (rc != CBQ_OK) return rc;
    CBQ_CUDA(cbq::launch_quantize_weights(w_dev, M * (K / CBQ_QK), static_cast<uint8_t *>(blocks_dev),
                                          as_stream(stream)));
    return CBQ_OK;
}

int cbq_hc_sinkhorn(const float *logits_dev, int64_t n, int iters, float *out_dev, void *stream) {
    static_assert(CBQ_HC_NHC == cbq::kHcNhc, "one matrix size on both sides of the ABI");
    if (!logits_dev || !out_dev || n < 1 || n > CBQ_HC_MAX_N || iters < 0 || iters > CBQ_HC_MAX_ITERS ||
        !aligned16(logits_dev) || !aligned16(out_dev))
        return CBQ_EINVAL;
    const uintptr_t a = reinterpret_cast<uintptr_t>(logits_dev), b = reinterpret_cast<uintptr_t>(out_dev);
    const uintptr_t bytes = (uintptr_t)n * CBQ_HC_NHC * CBQ_HC_NHC * sizeof(float);
    if (a != b && a < b + bytes && b < a + bytes) return CBQ_EINVAL;  // overlapping, not in place
    int dev = 0;
    const int rc = check_device(&dev);
    if (rc != CBQ_OK) return rc;
    CBQ_CUDA(cbq::launch_hc_sinkhorn(logits_dev, n, iters, out_dev, as_stream(stream)));
    return CBQ_OK;
}

int cbq_moe_matvec_logits(const cbq_moe *L, const float *h_dev, int n_tok, const float *logits_dev, int topk,
                          int swiglu, float *y_dev, void *stream) {
    if (!L || !h_dev || !logits_dev || !y_dev || n_tok < 1 || n_tok > CBQ_MAX_TOKENS || topk < 1 ||
        topk > CBQ_MAX_TOPK || topk > L->L.E || L->L.E > CBQ_ROUTER_MAX_E || (swiglu != 0 && swiglu != 1))
        return CBQ_EINVAL;
    DeviceScope scope(L->device);
    CBQ_CUDA(scope.status());
    cudaStream_t s = as_stream(stream);
    CBQ_CUDA(cbq::launch_router_topk(logits_dev, n_tok, L->L.E, topk, L->st_ids, L->st_wts, s));
    CBQ_CUDA(cbq::launch_moe(L->L, L->ws, h_dev, n_tok, L->st_ids, L->st_wts, topk, swiglu, y_dev, s));
    return CBQ_OK;
}

int cbq_moe_matvec_host(const cbq_moe *L, const float *h_host, int n_tok, const int32_t *ids_host,
                        const float *wts_host, int topk, int swiglu, float *y_host, void *stream) {
    if (!L || !h_host || !ids_host || !wts_host || !y_host || n_tok < 1 || n_tok > CBQ_MAX_TOKENS || topk < 1 ||
        topk > CBQ_MAX_TOPK || topk > L->L.E)
        return CBQ_EINVAL;
    DeviceScope scope(L->device);
    CBQ_CUDA(scope.status());
    cudaStream_t s = as_stream(stream);
    const size_t H = (size_t)L->L.H, N = (size_t)n_tok * topk;
    CBQ_CUDA(cudaMemcpyAsync(L->st_h, h_host, n_tok * H * sizeof(float), cudaMemcpyHostToDevice, s));
    CBQ_CUDA(cudaMemcpyAsync(L->st_ids, ids_host, N * sizeof(int32_t), cudaMemcpyHostToDevice, s));
    CBQ_CUDA(cudaMemcpyAsync(L->st_wts, wts_host, N * sizeof(float), cudaMemcpyHostToDevice, s));
    int rc = cbq_moe_matvec(L, L->st_h, n_tok, L->st_ids, L->st_wts, topk, swiglu, L->st_y, stream);
    if (rc != CBQ_OK) return rc;
    CBQ_CUDA(cudaMemcpyAsync(y_host, L->st_y, n_tok * H * sizeof(float), cudaMemcpyDeviceToHost, s));
    CBQ_CUDA(cudaStreamSynchronize(s));
    return CBQ_OK;
}

int cbq_moe_debug_block_dots(const cbq_moe *L, int e, int which, const int8_t *qx_dev, int n, int32_t *s_dev,
                             void *stream) {
    if (!L || e < 0 || e > L->L.E || (e == L->L.E && !L->L.shared) || (which != 0 && which != 1) || !qx_dev ||
        !s_dev || n < 1 || n > CBQ_MAX_COLS || !aligned16(qx_dev))
        return CBQ_EINVAL;
    DeviceScope scope(L->device);
    CBQ_CUDA(scope.status());
    const bool sh = e == L->L.E;
    DevMat m = {};
    if (which == 0) {
        m.w = sh ? L->sh_gu : L->gu + e * L->L.gu_stride;
        m.M = 2 * (int64_t)L->L.F;
        m.nb = L->L.H / CBQ_QK;
        m.split = L->L.F / CBQ_QK;
    } else {
        m.w = sh ? L->sh_dn : L->dn + e * L->L.dn_stride;
        m.M = L->L.H;
        m.nb = L->L.F / CBQ_QK;
        m.split = 0;
    }
    m.nbp = cbq::round_up4(m.nb);
    m.G = (int)((m.M + 31) / 32);
    m.P = (int)cbq::mat_pairs(m.M);
    m.sched = nullptr;  // the block-dot kernel uses static ranges
    m.err = L->ws.err;
    CBQ_CUDA(cbq::launch_block_dots(m, qx_dev, n, s_dev, as_stream(stream)));
    return CBQ_OK;
}

int cbq_moe_set_debug(cbq_moe *L, int keep_intermediate) {
    if (!L) return CBQ_EINVAL;
    L->ws.keep_a = keep_intermediate ? 1 : 0;
    return CBQ_OK;
}

int cbq_moe_set_stage_events(cbq_moe *L, void *ev_start, void *ev_layer, void *ev_end) {
    if (!L) return CBQ_EINVAL;
    const bool all = ev_start && ev_layer && ev_end;
    const bool none = !ev_start && !ev_layer && !ev_end;
    if (!all && !none) return CBQ_EINVAL;
    L->ws.ev[0] = reinterpret_cast<cudaEvent_t>(ev_start);
    L->ws.ev[1] = reinterpret_cast<cudaEvent_t>(ev_layer);
    L->ws.ev[2] = reinterpret_cast<cudaEvent_t>(ev_end);
    return CBQ_OK;
}

int cbq_moe_debug_intermediate(const cbq_moe *L, int nslots, float *a_dev, int8_t *qa_dev, float *da_dev,
                               void *stream) {
    if (!L || nslots < 1 || nslots > cbq::kMaxSlots) return CBQ_EINVAL;
    DeviceScope scope(L->device);
    CBQ_CUDA(scope.status());
    cudaStream_t s = as_stream(stream);
    const size_t F = (size_t)L->L.F;
    if (a_dev) CBQ_CUDA(cudaMemcpyAsync(a_dev, L->ws.a_dbg, nslots * F * sizeof(float), cudaMemcpyDeviceToDevice, s));
    if (qa_dev) CBQ_CUDA(cudaMemcpyAsync(qa_dev, L->ws.qa, nslots * F, cudaMemcpyDeviceToDevice, s));
    if (da_dev)
        CBQ_CUDA(cudaMemcpyAsync(da_dev, L->ws.da, nslots * (F / CBQ_QK) * sizeof(float), cudaMemcpyDeviceToDevice, s));
    return CBQ_OK;
}

namespace {

// Copy a handle's error word to *code and clear it, both in the order of
// `stream`, then wait for that stream only.
int read_and_clear(unsigned *err, int device, void *stream, unsigned *code) {
    DeviceScope scope(device);
    CBQ_CUDA(scope.status());
    cudaStream_t s = as_stream(stream);
    CBQ_CUDA(cudaMemcpyAsync(code, err, sizeof(unsigned), cudaMemcpyDeviceToHost, s));
    CBQ_CUDA(cudaMemsetAsync(err, 0, sizeof(unsigned), s));
    CBQ_CUDA(cudaStreamSynchronize(s));
    return CBQ_OK;
}

}  // namespace

int cbq_weights_get_error(const cbq_weights *W, void *stream, unsigned int *code) {
    if (!W || !code) return CBQ_EINVAL;
    return read_and_clear(W->err, W->device, stream, code);
}

int cbq_moe_get_error(const cbq_moe *L, void *stream, unsigned int *code) {
    if (!L || !code) return CBQ_EINVAL;
    return read_and_clear(L->ws.err, L->device, stream, code);
}

int cbq_moe_debug_stall(cbq_moe *L, int mode) {
    if (!L || mode < 0 || mode > 2) return CBQ_EINVAL;
    L->ws.stall = mode;
    return CBQ_OK;
}

int cbq_debug_mmq_stall(cbq_weights *W, int mode) {
    if (!W || mode < 0 || mode > 1) return CBQ_EINVAL;
    W->mq_stall = mode;
    return CBQ_OK;
}

}  // extern "C"

// policy.cu -- the layer-range policy of "CacheReforge: Bounded Recovery for
// Stale KV Caches under Evolving Adapters" (Methodology: Layerwise Risk,
// Eqs. 6-7; Runtime risk and range selection, Eqs. 8-9; Cache and anchor
// updates; supplementary Eq. S4 for the restart layer).
//
// The adapter is one flat parameter vector.  Every cached layer keeps its own
// anchor copy in device memory, so a cache that mixes layers recomputed under
// different adapter versions is tracked exactly.  The drift of each layer,
// ||theta_t - anchor_l||_2, is one pass over n_layers x n_params elements:
// a grid of (chunk, layer) blocks sums squared differences in double in a
// fixed order, and the host adds the chunk sums in order, so the result does
// not depend on scheduling.  Everything else is a few scalars per layer on
// the host.
#include <cuda_bf16.h>

#include <algorithm>
#include <cmath>
#include <vector>

#include "kvr_internal.h"

struct kvr_policy {
    int32_t n_layers = 0;
    int64_t n_params = 0;
    int32_t dtype = KVR_F32;
    int device = 0;
    std::vector<double> s;          // sensitivities
    std::vector<int64_t> version;   // per-layer anchor version
    void* d_anchor = nullptr;       // [n_layers][n_params]
    double* d_part = nullptr;       // [n_layers][kChunks]
};

namespace kvr {
namespace {

constexpr int kChunks = 64;      // blocks per layer
constexpr int kDriftThreads = 256;

__device__ __forceinline__ double ldd(const float* p) { return (double)*p; }
__device__ __forceinline__ double ldd(const __nv_bfloat16* p) { return (double)__bfloat162float(*p); }

template <typename T>
__global__ void __launch_bounds__(kDriftThreads) drift_kernel(const T* __restrict__ theta, const T* __restrict__ anchors,
                                                             int64_t n, double* __restrict__ part) {
    __shared__ double red[kDriftThreads];
    const int chunk = blockIdx.x, layer = blockIdx.y;
    const int64_t per = (n + kChunks - 1) / kChunks;
    const int64_t b = (int64_t)chunk * per, e = (b + per < n) ? b + per : n;
    const T* a = anchors + (size_t)layer * (size_t)n;
    double acc = 0.0;
    for (int64_t i = b + threadIdx.x; i < e; i += kDriftThreads) {
        const double d = ldd(theta + i) - ldd(a + i);
        acc = fma(d, d, acc);
    }
    red[threadIdx.x] = acc;
    __syncthreads();
    for (int w = kDriftThreads / 2; w > 0; w >>= 1) {
        if (threadIdx.x < w) red[threadIdx.x] += red[threadIdx.x + w];
        __syncthreads();
    }
    if (threadIdx.x == 0) part[layer * kChunks + chunk] = red[0];
}

size_t elem_size(int dtype) { return dtype == KVR_BF16 ? 2 : 4; }

}  // namespace
}  // namespace kvr

using namespace kvr;

extern "C" {

int32_t kvr_restart_layer(int32_t module, int32_t s, int32_t n_layers) {
    if (n_layers < 1 || s < 0 || s >= n_layers) return -1;
    switch (module) {
        case KVR_MOD_K:
        case KVR_MOD_V:
            return s;
        case KVR_MOD_Q:
        case KVR_MOD_O:
        case KVR_MOD_MLP:
            return std::min(s + 1, n_layers);
        default:
            return -1;
    }
}

kvr_status kvr_policy_sensitivity(int32_t n_layers, int32_t n_cond, const int32_t* restart, const int32_t* window,
                                  const double* drift, double* s_out) {
    if (n_layers < 1 || n_cond < 0 || !s_out || (n_cond > 0 && (!restart || !window || !drift))) {
        set_error("policy sensitivity: bad arguments");
        return KVR_EINVAL;
    }
    for (int i = 0; i < n_cond; ++i) {
        if (restart[i] < 0 || restart[i] >= n_layers || window[i] < 0 || !(drift[i] >= 0.0)) {
            set_error("policy sensitivity: condition " + std::to_string(i) + " is malformed");
            return KVR_EINVAL;
        }
    }
    std::vector<double> D;
    for (int l = 0; l < n_layers; ++l) {
        D.clear();
        for (int i = 0; i < n_cond; ++i)
            if (restart[i] <= l && (int64_t)l < (int64_t)restart[i] + window[i]) D.push_back(drift[i]);
        if (D.empty()) {
            s_out[l] = 0.0;
            continue;
        }
        std::sort(D.begin(), D.end());
        const size_t k = (size_t)std::floor(0.05 * (double)D.size());   // first value after the 5 % lower tail
        s_out[l] = 1.0 / std::max(D[k], 1e-12);
    }
    return KVR_OK;
}

kvr_status kvr_policy_create(int32_t n_layers, int64_t n_params, int32_t dtype, const void* theta0,
                             const double* sensitivity, void* stream, kvr_policy** out) {
    if (!out) {
        set_error("out is NULL");
        return KVR_EINVAL;
    }
    *out = nullptr;
    if (n_layers < 1 || n_params < 1 || (dtype != KVR_F32 && dtype != KVR_BF16) || !theta0 || !sensitivity) {
        set_error("policy: need n_layers >= 1, n_params >= 1, dtype KVR_F32/KVR_BF16, theta0 and sensitivity");
        return KVR_EINVAL;
    }
    for (int l = 0; l < n_layers; ++l) {
        if (!(sensitivity[l] >= 0.0) || !std::isfinite(sensitivity[l])) {
            set_error("policy: sensitivities must be finite and >= 0");
            return KVR_EINVAL;
        }
    }
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    kvr_policy* p = new kvr_policy();
    p->n_layers = n_layers;
    p->n_params = n_params;
    p->dtype = dtype;
    p->s.assign(sensitivity, sensitivity + n_layers);
    p->version.assign(n_layers, 0);
    cudaGetDevice(&p->device);
    const size_t bytes = (size_t)n_params * elem_size(dtype);
    cudaError_t e = cudaMalloc(&p->d_anchor, bytes * n_layers);
    if (e == cudaSuccess) e = cudaMalloc((void**)&p->d_part, sizeof(double) * kChunks * n_layers);
    if (e != cudaSuccess) {
        set_error(std::string("policy allocation failed: ") + cudaGetErrorString(e));
        cudaFree(p->d_anchor);
        cudaFree(p->d_part);
        delete p;
        return KVR_ENOMEM;
    }
    for (int l = 0; l < n_layers && e == cudaSuccess; ++l)
        e = cudaMemcpyAsync((uint8_t*)p->d_anchor + bytes * l, theta0, bytes, cudaMemcpyDeviceToDevice, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) {
        kvr_status r = cuda_fail(e, "policy set-up");
        cudaFree(p->d_anchor);
        cudaFree(p->d_part);
        delete p;
        return r;
    }
    *out = p;
    return KVR_OK;
}

kvr_status kvr_policy_destroy(kvr_policy* p) {
    if (!p) return KVR_OK;
    cudaDeviceSynchronize();
    cudaFree(p->d_anchor);
    cudaFree(p->d_part);
    delete p;
    return KVR_OK;
}

kvr_status kvr_policy_plan(kvr_policy* p, const void* theta_t, int32_t module, int32_t update_layer,
                           double* drift_out, double* risk_out, int32_t* range_out, void* stream) {
    if (!p || !theta_t || !range_out) {
        set_error("policy plan: NULL argument");
        return KVR_EINVAL;
    }
    const int32_t r_kv = kvr_restart_layer(module, update_layer, p->n_layers);
    if (r_kv < 0) {
        set_error("policy plan: unknown module or update layer outside [0, n_layers)");
        return KVR_EINVAL;
    }
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const dim3 grid(kChunks, (unsigned)p->n_layers);
    if (p->dtype == KVR_BF16)
        drift_kernel<__nv_bfloat16><<<grid, kDriftThreads, 0, s>>>(
            (const __nv_bfloat16*)theta_t, (const __nv_bfloat16*)p->d_anchor, p->n_params, p->d_part);
    else
        drift_kernel<float><<<grid, kDriftThreads, 0, s>>>((const float*)theta_t, (const float*)p->d_anchor,
                                                           p->n_params, p->d_part);
    cudaError_t e = cudaGetLastError();
    std::vector<double> part((size_t)kChunks * p->n_layers);
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(part.data(), p->d_part, part.size() * sizeof(double), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "policy drift");
    int32_t last = -1;
    for (int l = 0; l < p->n_layers; ++l) {
        double sum = 0.0;
        for (int c = 0; c < kChunks; ++c) sum += part[(size_t)l * kChunks + c];
        const double d = std::sqrt(sum);
        const double q = p->s[l] * d;
        if (drift_out) drift_out[l] = d;
        if (risk_out) risk_out[l] = q;
        if (q >= 1.0) last = l;
    }
    const int32_t r = update_layer;
    const int32_t b = last + 1;   // b_t = 1 + max{l : q_l >= 1}
    if (last < 0 || b <= r_kv) {
        range_out[0] = range_out[1] = r;   // direct reuse
    } else {
        range_out[0] = r;
        range_out[1] = b;
    }
    return KVR_OK;
}

kvr_status kvr_policy_commit(kvr_policy* p, const void* theta_t, int32_t begin, int32_t end, int64_t version,
                             void* stream) {
    if (!p || !theta_t || begin < 0 || end < begin || end > p->n_layers) {
        set_error("policy commit: need 0 <= begin <= end <= n_layers and theta_t");
        return KVR_EINVAL;
    }
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const size_t bytes = (size_t)p->n_params * elem_size(p->dtype);
    for (int l = begin; l < end; ++l) {
        cudaError_t e = cudaMemcpyAsync((uint8_t*)p->d_anchor + bytes * l, theta_t, bytes, cudaMemcpyDeviceToDevice, s);
        if (e != cudaSuccess) return cuda_fail(e, "policy commit");
        p->version[l] = version;
    }
    return KVR_OK;
}

kvr_status kvr_policy_versions(kvr_policy* p, int64_t* versions) {
    if (!p || !versions) {
        set_error("policy versions: NULL argument");
        return KVR_EINVAL;
    }
    std::copy(p->version.begin(), p->version.end(), versions);
    return KVR_OK;
}

}  // extern "C"

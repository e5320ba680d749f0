// lora.cu -- fold a low-rank adapter into a projection:
//   W'[i][k] = W[i][k] + scale * sum_j B[i - row_begin][j] * A[j][k]
// for the rows an adapter touches (the Q and V rows of the fused QKV matrix).
// "CacheReforge: Bounded Recovery for Stale KV Caches under Evolving
// Adapters", Implementation: a LoRA on the cache-producing projections; a
// recovery recomputes the affected layers under the current adapter, so the
// merged weights are formed once per adapter version and the refresh runs
// the plain projection.  fp32 accumulation, one rounding to the model dtype.
#include <cuda_bf16.h>

#include "kvr_internal.h"

namespace kvr {
namespace {

__device__ __forceinline__ float ldv(const float* p) { return *p; }
__device__ __forceinline__ float ldv(const __nv_bfloat16* p) { return __bfloat162float(*p); }
__device__ __forceinline__ void stv(float* p, float v) { *p = v; }
__device__ __forceinline__ void stv(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }

// one thread per output element; B's row for the thread's output row is read
// once per element (rank is small: 4-64)
template <typename T>
__global__ void lora_merge_kernel(const T* __restrict__ w, T* __restrict__ out, int n_out, int K, int row_begin,
                                  int row_count, const T* __restrict__ a, const T* __restrict__ b, int rank,
                                  float scale) {
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (long long)n_out * K) return;
    const int row = (int)(i / K), k = (int)(i % K);
    float v = ldv(w + i);
    if (row >= row_begin && row < row_begin + row_count) {
        const T* br = b + (size_t)(row - row_begin) * rank;
        float acc = 0.f;
        for (int j = 0; j < rank; ++j) acc = fmaf(ldv(br + j), ldv(a + (size_t)j * K + k), acc);
        v += scale * acc;
    }
    stv(out + i, v);
}

}  // namespace

cudaError_t launch_lora_merge(int dtype, const void* w, void* w_out, int n_out, int K, int row_begin, int row_count,
                              const void* a, const void* b, int rank, float scale, cudaStream_t s) {
    const long long n = (long long)n_out * K;
    if (n <= 0) return cudaSuccess;
    const unsigned blocks = (unsigned)((n + 255) / 256);
    if (dtype == KVR_BF16)
        lora_merge_kernel<__nv_bfloat16><<<blocks, 256, 0, s>>>(
            (const __nv_bfloat16*)w, (__nv_bfloat16*)w_out, n_out, K, row_begin, row_count,
            (const __nv_bfloat16*)a, (const __nv_bfloat16*)b, rank, scale);
    else
        lora_merge_kernel<float><<<blocks, 256, 0, s>>>((const float*)w, (float*)w_out, n_out, K, row_begin,
                                                        row_count, (const float*)a, (const float*)b, rank, scale);
    return cudaGetLastError();
}

}  // namespace kvr

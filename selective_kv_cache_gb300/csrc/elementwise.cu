// elementwise.cu -- token-local steps of the layer: RMSNorm, and the
// epilogues that reduce the split-K GEMM partials (in split order, so the
// result does not depend on scheduling) and apply the fused operation:
//   QKV : + bias, rotate-half RoPE at the row's global position, write Q to
//         the packed buffer and K/V into the cache rows u_r ("Budgeted
//         KV-Cache Repair for Evolving Contexts", Sec. 13.2, Eq. 21);
//   O   : h = x + o W_o^T, kept in fp32;
//   gate/up : SwiGLU silu(g) * u;
//   down: x' = h + a W_d^T, rounded to the model dtype.
// All stores of the model dtype are 16-byte vectors.
#include <cuda_bf16.h>

#include "kvr_internal.h"

namespace kvr {
namespace {

// 8 consecutive values of T <-> floats through one or two 16-byte accesses
template <typename T>
__device__ __forceinline__ void load8(const T* p, float* v);
template <>
__device__ __forceinline__ void load8<float>(const float* p, float* v) {
    const float4 a = reinterpret_cast<const float4*>(p)[0], b = reinterpret_cast<const float4*>(p)[1];
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
template <>
__device__ __forceinline__ void load8<__nv_bfloat16>(const __nv_bfloat16* p, float* v) {
    const uint4 u = *reinterpret_cast<const uint4*>(p);
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 f = __bfloat1622float2(h[i]);
        v[2 * i] = f.x;
        v[2 * i + 1] = f.y;
    }
}
template <typename T>
__device__ __forceinline__ void store8(T* p, const float* v);
template <>
__device__ __forceinline__ void store8<float>(float* p, const float* v) {
    reinterpret_cast<float4*>(p)[0] = make_float4(v[0], v[1], v[2], v[3]);
    reinterpret_cast<float4*>(p)[1] = make_float4(v[4], v[5], v[6], v[7]);
}
template <>
__device__ __forceinline__ void store8<__nv_bfloat16>(__nv_bfloat16* p, const float* v) {
    uint4 u;
    __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
    *reinterpret_cast<uint4*>(p) = u;
}

// sum of the split partials of 8 consecutive features (fp32, 16-B loads)
__device__ __forceinline__ void sum_parts8(const float* part, size_t split_stride, int splits, size_t off,
                                           float* v) {
    const float4* p = reinterpret_cast<const float4*>(part + off);
    float4 a = __ldcg(p), b = __ldcg(p + 1);
    for (int s = 1; s < splits; ++s) {
        const float4* q = reinterpret_cast<const float4*>(part + (size_t)s * split_stride + off);
        const float4 c = __ldcg(q), d = __ldcg(q + 1);
        a.x += c.x; a.y += c.y; a.z += c.z; a.w += c.w;
        b.x += d.x; b.y += d.y; b.z += d.z; b.w += d.w;
    }
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

// ------------------------------------------------------------------ RMSNorm
template <typename T, typename Tin>
__global__ void __launch_bounds__(256) rmsnorm_kernel(const Tin* __restrict__ in, const T* __restrict__ w,
                                                      T* __restrict__ out, int d, float eps) {
    pdl_trigger();
    pdl_wait();
    const int r = blockIdx.x;
    const Tin* x = in + (size_t)r * d;
    float ss = 0.f;
    for (int i = threadIdx.x * 8; i < d; i += blockDim.x * 8) {
        float v[8];
        load8<Tin>(x + i, v);
#pragma unroll
        for (int j = 0; j < 8; ++j) ss += v[j] * v[j];
    }
    __shared__ float red[8];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
    __syncthreads();
    float tot = 0.f;
    for (int i = 0; i < (int)(blockDim.x >> 5); ++i) tot += red[i];
    const float rstd = 1.0f / sqrtf(tot / (float)d + eps);
    for (int i = threadIdx.x * 8; i < d; i += blockDim.x * 8) {
        float v[8], g[8];
        load8<Tin>(x + i, v);
        load8<T>(w + i, g);
#pragma unroll
        for (int j = 0; j < 8; ++j) v[j] = v[j] * rstd * g[j];
        store8<T>(out + (size_t)r * d + i, v);
    }
}

// ------------------------------------------------------------------ QKV
// one thread per (row, head, 8-pair chunk of the first half of head_dim).
// The row's position and sequence and its rotary factors (a chain of two
// loads) are written by no kernel of the call (a selection's last launch is
// followed by one that waits for the whole stream), so they are loaded before
// the wait for the projection; its partials, the bias and the norm weights
// after it, all in one round trip.
template <typename T>
__global__ void __launch_bounds__(256) epi_qkv_kernel(QkvEpi a) {
    pdl_trigger();
    const int dh = a.head_dim, half = dh / 2, chunks = half / 8;
    const int heads = a.n_q_heads + 2 * a.n_kv_heads;
    const long long t = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    const long long total = (long long)a.R * heads * chunks;
    if (t >= total) return;
    const int c = (int)(t % chunks);
    const int hh = (int)((t / chunks) % heads);
    const int r = (int)(t / ((long long)chunks * heads));
    const int n_qkv = heads * dh;
    const size_t split_stride = (size_t)a.R * n_qkv;
    const int f1 = hh * dh + c * 8, f2 = f1 + half;
    const bool is_v = hh >= a.n_q_heads + a.n_kv_heads;
    const int u = a.U[r];
    const int seq = a.row_seq[r];
    const bool u_ok = u >= 0 && u < a.capacity;
    float2 cs[8];
    if (!is_v && u_ok) {
        const float4* rp = reinterpret_cast<const float4*>(a.rope + (size_t)u * half + c * 8);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float4 e = rp[j];
            cs[2 * j] = make_float2(e.x, e.y);
            cs[2 * j + 1] = make_float2(e.z, e.w);
        }
    }
    pdl_wait();
    float x1[8], x2[8];
    sum_parts8(a.part, split_stride, a.splits, (size_t)r * n_qkv + f1, x1);
    sum_parts8(a.part, split_stride, a.splits, (size_t)r * n_qkv + f2, x2);
    if (a.bias) {
        float b1[8], b2[8];
        load8<T>((const T*)a.bias + f1, b1);
        load8<T>((const T*)a.bias + f2, b2);
#pragma unroll
        for (int j = 0; j < 8; ++j) { x1[j] += b1[j]; x2[j] += b2[j]; }
    }
    if (a.q_norm && hh < a.n_q_heads + a.n_kv_heads) {
        // Q/K normalisation: RMSNorm of the head over its d_h dims, whose 8-wide
        // chunks sit in `chunks` consecutive lanes (a group aligned to chunks)
        float ss = 0.f;
#pragma unroll
        for (int j = 0; j < 8; ++j) ss += x1[j] * x1[j] + x2[j] * x2[j];
        const int lane = threadIdx.x & 31;
        const unsigned gm = chunks >= 32 ? 0xffffffffu : ((1u << chunks) - 1u) << (lane & ~(chunks - 1));
        for (int o = 1; o < chunks; o <<= 1) ss += __shfl_xor_sync(gm, ss, o);
        const float inv = rsqrtf(ss / (float)dh + a.eps);
        const T* wn = (const T*)(hh < a.n_q_heads ? a.q_norm : a.k_norm);
        float w1[8], w2[8];
        load8<T>(wn + c * 8, w1);
        load8<T>(wn + half + c * 8, w2);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            x1[j] = x1[j] * inv * w1[j];
            x2[j] = x2[j] * inv * w2[j];
        }
    }
    if (!u_ok) {
        atomicOr(a.err, DEV_ERR_INDEX);
        return;
    }
    if (!is_v) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float2 e = cs[j];
            const float p = x1[j], q = x2[j];
            x1[j] = p * e.x - q * e.y;
            x2[j] = q * e.x + p * e.y;
        }
    }
    T* dst;
    if (hh < a.n_q_heads) {
        dst = (T*)a.q_out + ((size_t)r * a.n_q_heads + hh) * dh;
    } else {
        const int kvh = is_v ? hh - a.n_q_heads - a.n_kv_heads : hh - a.n_q_heads;
        T* base = (T*)(is_v ? a.v_base : a.k_base);
        dst = base + ((((size_t)seq * a.n_layers + a.layer) * a.n_kv_heads + kvh) * a.capacity + u) * dh;
    }
    store8<T>(dst + c * 8, x1);
    store8<T>(dst + half + c * 8, x2);
}

// ------------------------------------------------------------------ O, gate/up, down
// grid (rows, blocks of 256 8-wide chunks of the row)
template <typename T>
__global__ void epi_swiglu_kernel(const float* __restrict__ part, int splits, int R, int F, T* __restrict__ act) {
    pdl_trigger();
    pdl_wait();
    const int r = (int)blockIdx.x, f = ((int)blockIdx.y * 256 + (int)threadIdx.x) * 8;
    if (f >= F) return;
    const size_t i8 = (size_t)r * F + f;
    const size_t stride = (size_t)R * 2 * F;
    float g[8], u[8];
    sum_parts8(part, stride, splits, (size_t)r * 2 * F + f, g);
    sum_parts8(part, stride, splits, (size_t)r * 2 * F + F + f, u);
#pragma unroll
    for (int j = 0; j < 8; ++j) g[j] = g[j] / (1.0f + expf(-g[j])) * u[j];
    store8<T>(act + i8, g);
}

template <typename T>
__global__ void epi_down_kernel(const float* __restrict__ part, int splits, int R, int d, const float* __restrict__ h,
                                T* __restrict__ x) {
    pdl_trigger();
    pdl_wait();
    const long long i8 = ((long long)blockIdx.x * blockDim.x + threadIdx.x) * 8;
    if (i8 >= (long long)R * d) return;
    float v[8], hv[8];
    sum_parts8(part, (size_t)R * d, splits, (size_t)i8, v);
    load8<float>(h + i8, hv);
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] += hv[j];
    store8<T>(x + i8, v);
}

// ------------------------------------------------------------------ residual + RMSNorm, one CTA per row
// Each thread keeps up to kRowChunks 8-element chunks of its row in registers
// between the sum-of-squares pass and the normalisation.
constexpr int kRowThreads = 512;   // one 8-element chunk a thread at d = 4096: every load in flight at once
constexpr int kRowChunks = 2;   // rows up to 512 * 2 * 8 = 8192 elements

__device__ __forceinline__ float row_rstd(float ss, int d, float eps) {
    __shared__ float red[kRowThreads / 32];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
    __syncthreads();
    float tot = 0.f;
#pragma unroll
    for (int i = 0; i < kRowThreads / 32; ++i) tot += red[i];
    return 1.0f / sqrtf(tot / (float)d + eps);
}

__device__ __forceinline__ float round_to(float v, float*) { return v; }
__device__ __forceinline__ float round_to(float v, __nv_bfloat16*) { return __bfloat162float(__float2bfloat16_rn(v)); }

// h = x + sum of the O projection's partials (fp32), then hn = RMSNorm(h) * w
template <typename T>
__global__ void __launch_bounds__(kRowThreads) epi_residual_norm_kernel(const float* __restrict__ part, int splits,
                                                                        int R, int d, const T* __restrict__ x,
                                                                        float* __restrict__ h, const T* __restrict__ w,
                                                                        T* __restrict__ hn, float eps) {
    pdl_trigger();
    pdl_wait();
    const int r = blockIdx.x;
    float v[kRowChunks][8];
    float ss = 0.f;
#pragma unroll
    for (int k = 0; k < kRowChunks; ++k) {
        const int i = (threadIdx.x + k * kRowThreads) * 8;
        if (i < d) {
            float xv[8];
            sum_parts8(part, (size_t)R * d, splits, (size_t)r * d + i, v[k]);
            load8<T>(x + (size_t)r * d + i, xv);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                v[k][j] += xv[j];
                ss += v[k][j] * v[k][j];
            }
            store8<float>(h + (size_t)r * d + i, v[k]);
        }
    }
    const float rstd = row_rstd(ss, d, eps);
#pragma unroll
    for (int k = 0; k < kRowChunks; ++k) {
        const int i = (threadIdx.x + k * kRowThreads) * 8;
        if (i < d) {
            float g[8];
            load8<T>(w + i, g);
#pragma unroll
            for (int j = 0; j < 8; ++j) v[k][j] = v[k][j] * rstd * g[j];
            store8<T>(hn + (size_t)r * d + i, v[k]);
        }
    }
}

// x' = h + sum of the down projection's partials, stored in T; then the next
// layer's xn = RMSNorm(x') * w_next from the stored (rounded) x'
template <typename T>
__global__ void __launch_bounds__(kRowThreads) epi_down_norm_kernel(const float* __restrict__ part, int splits, int R,
                                                                    int d, const float* __restrict__ h,
                                                                    T* __restrict__ x, const T* __restrict__ w_next,
                                                                    T* __restrict__ xn, float eps) {
    pdl_trigger();
    pdl_wait();
    const int r = blockIdx.x;
    float v[kRowChunks][8];
    float ss = 0.f;
#pragma unroll
    for (int k = 0; k < kRowChunks; ++k) {
        const int i = (threadIdx.x + k * kRowThreads) * 8;
        if (i < d) {
            float hv[8];
            sum_parts8(part, (size_t)R * d, splits, (size_t)r * d + i, v[k]);
            load8<float>(h + (size_t)r * d + i, hv);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                v[k][j] = round_to(v[k][j] + hv[j], (T*)nullptr);
                ss += v[k][j] * v[k][j];
            }
            store8<T>(x + (size_t)r * d + i, v[k]);
        }
    }
    const float rstd = row_rstd(ss, d, eps);
#pragma unroll
    for (int k = 0; k < kRowChunks; ++k) {
        const int i = (threadIdx.x + k * kRowThreads) * 8;
        if (i < d) {
            float g[8];
            load8<T>(w_next + i, g);
#pragma unroll
            for (int j = 0; j < 8; ++j) v[k][j] = v[k][j] * rstd * g[j];
            store8<T>(xn + (size_t)r * d + i, v[k]);
        }
    }
}

inline unsigned blocks_for(long long n, int per_block) { return (unsigned)((n + per_block - 1) / per_block); }

}  // namespace

cudaError_t launch_rmsnorm(int dtype, const void* in, int in_f32, const void* w, void* out, int rows, int d, float eps,
                           cudaStream_t s) {
    if (rows <= 0) return cudaSuccess;
    if (dtype == KVR_BF16) {
        if (in_f32)
            KVR_LAUNCH(rmsnorm_kernel<__nv_bfloat16, float>, dim3(rows), dim3(256), 0, s, (const float*)in, (const __nv_bfloat16*)w,
                                                                      (__nv_bfloat16*)out, d, eps);
        else
            KVR_LAUNCH(rmsnorm_kernel<__nv_bfloat16, __nv_bfloat16>, dim3(rows), dim3(256), 0, s,
                (const __nv_bfloat16*)in, (const __nv_bfloat16*)w, (__nv_bfloat16*)out, d, eps);
    } else {
        KVR_LAUNCH(rmsnorm_kernel<float, float>, dim3(rows), dim3(256), 0, s, (const float*)in, (const float*)w, (float*)out, d, eps);
    }
    return cudaGetLastError();
}

cudaError_t launch_epi_qkv(int dtype, const QkvEpi& a, cudaStream_t s) {
    const long long total = (long long)a.R * (a.n_q_heads + 2 * a.n_kv_heads) * (a.head_dim / 16);
    if (total <= 0) return cudaSuccess;
    if (dtype == KVR_BF16)
        KVR_LAUNCH(epi_qkv_kernel<__nv_bfloat16>, dim3(blocks_for(total, 256)), dim3(256), 0, s, a);
    else
        KVR_LAUNCH(epi_qkv_kernel<float>, dim3(blocks_for(total, 256)), dim3(256), 0, s, a);
    return cudaGetLastError();
}

cudaError_t launch_epi_swiglu(int dtype, const float* part, int splits, int R, int F, void* act_out, cudaStream_t s) {
    if (R <= 0 || F <= 0) return cudaSuccess;
    const dim3 grid((unsigned)R, blocks_for(F / 8, 256));
    if (dtype == KVR_BF16)
        KVR_LAUNCH(epi_swiglu_kernel<__nv_bfloat16>, grid, dim3(256), 0, s, part, splits, R, F, (__nv_bfloat16*)act_out);
    else
        KVR_LAUNCH(epi_swiglu_kernel<float>, grid, dim3(256), 0, s, part, splits, R, F, (float*)act_out);
    return cudaGetLastError();
}

cudaError_t launch_epi_down(int dtype, const float* part, int splits, int R, int d, const float* h, void* x_out,
                            cudaStream_t s) {
    const long long n = (long long)R * d / 8;
    if (n <= 0) return cudaSuccess;
    if (dtype == KVR_BF16)
        KVR_LAUNCH(epi_down_kernel<__nv_bfloat16>, dim3(blocks_for(n, 256)), dim3(256), 0, s, part, splits, R, d, h,
                                                                          (__nv_bfloat16*)x_out);
    else
        KVR_LAUNCH(epi_down_kernel<float>, dim3(blocks_for(n, 256)), dim3(256), 0, s, part, splits, R, d, h, (float*)x_out);
    return cudaGetLastError();
}

cudaError_t launch_epi_residual_norm(int dtype, const float* part, int splits, int R, int d, const void* x, float* h,
                                     const void* w, void* hn, float eps, cudaStream_t s) {
    if (R <= 0) return cudaSuccess;
    if (d > kRowThreads * kRowChunks * 8) return cudaErrorInvalidValue;
    if (dtype == KVR_BF16)
        KVR_LAUNCH(epi_residual_norm_kernel<__nv_bfloat16>, dim3(R), dim3(kRowThreads), 0, s,
            part, splits, R, d, (const __nv_bfloat16*)x, h, (const __nv_bfloat16*)w, (__nv_bfloat16*)hn, eps);
    else
        KVR_LAUNCH(epi_residual_norm_kernel<float>, dim3(R), dim3(kRowThreads), 0, s, part, splits, R, d, (const float*)x, h,
                                                                  (const float*)w, (float*)hn, eps);
    return cudaGetLastError();
}

cudaError_t launch_epi_down_norm(int dtype, const float* part, int splits, int R, int d, const float* h, void* x,
                                 const void* w_next, void* xn, float eps, cudaStream_t s) {
    if (R <= 0) return cudaSuccess;
    if (d > kRowThreads * kRowChunks * 8) return cudaErrorInvalidValue;
    if (dtype == KVR_BF16)
        KVR_LAUNCH(epi_down_norm_kernel<__nv_bfloat16>, dim3(R), dim3(kRowThreads), 0, s,
            part, splits, R, d, h, (__nv_bfloat16*)x, (const __nv_bfloat16*)w_next, (__nv_bfloat16*)xn, eps);
    else
        KVR_LAUNCH(epi_down_norm_kernel<float>, dim3(R), dim3(kRowThreads), 0, s, part, splits, R, d, h, (float*)x,
                                                              (const float*)w_next, (float*)xn, eps);
    return cudaGetLastError();
}

}  // namespace kvr

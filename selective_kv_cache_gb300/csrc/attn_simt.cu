// attn_simt.cu -- biased causal grouped-query attention over the mixed cache,
// CUDA-core version for fp32 models (fp32 storage needs fp32 products; the
// bf16 path runs on the tensor cores, attn_tc.cu).
//
//   s_ij = <q_i, k_j>/sqrt(d_h) + alpha*loc_j + beta*snk_j,  j <= g_i
//   o_i  = sum_j softmax_j(s_ij) v_j
// ("kv-cross-attention-reuse", Sec. 6.4, Logit form; "Budgeted KV-Cache
// Repair for Evolving Contexts", Sec. 13.2, Eq. 22 with 0:u_r inclusive.)
//
// One CTA per (query tile, K/V head): the tile's positions x the G query
// heads of that K/V head form (position, head) pairs that share every K/V
// tile staged in shared memory.  Each warp owns a fixed set of pairs and
// keeps their online-softmax state (running max, sum, fp32 output) in
// shared memory.  Tiles beyond the plan's n_total are never read.
#include <cuda_bf16.h>

#include "kvr_internal.h"

namespace kvr {
namespace {

constexpr int kThreads = 256;
constexpr int kMaxPairs = 64;

__device__ __forceinline__ float ldf(const float* p) { return *p; }
__device__ __forceinline__ void stf(float* p, float v) { *p = v; }

template <typename T>
__global__ void __launch_bounds__(kThreads) attn_simt_kernel(AttnLaunch a) {
    extern __shared__ float sm[];
    pdl_trigger();
    pdl_wait();
    const int dh = a.head_dim, G = a.n_q_heads / a.n_kv_heads;
    const int tile = blockIdx.x, kvh = blockIdx.y;
    const int* plan = a.plan + 8 * tile;
    const int row0 = plan[0], nrows = plan[1], n_total = plan[5], seq = plan[6];
    const int pairs = nrows * G;
    const int ldk = dh + 1;
    float* Ks = sm;                                 // [64][dh+1]
    float* Vs = Ks + kSimtKeysPerTile * ldk;        // [64][dh+1]
    float* Qs = Vs + kSimtKeysPerTile * ldk;        // [pairs][dh]
    float* Os = Qs + kMaxPairs * dh;                // [pairs][dh]
    float* Ms = Os + kMaxPairs * dh;                // [pairs]
    float* Ls = Ms + kMaxPairs;                     // [pairs]
    int* Gs = reinterpret_cast<int*>(Ls + kMaxPairs);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const float scale = 1.0f / sqrtf((float)dh);
    const T* q = (const T*)a.q;
    for (int i = threadIdx.x; i < pairs * dh; i += kThreads) {
        const int p = i / dh, d = i % dh;
        const int r = row0 + p / G, h = kvh * G + p % G;
        Qs[i] = ldf(q + ((size_t)r * a.n_q_heads + h) * dh + d) * scale;
        Os[i] = 0.f;
    }
    for (int p = threadIdx.x; p < pairs; p += kThreads) {
        Ms[p] = -INFINITY;
        Ls[p] = 0.f;
        Gs[p] = a.U[row0 + p / G];
    }
    const size_t head_off = (((size_t)seq * a.n_layers + a.layer) * a.n_kv_heads + kvh) * a.capacity;
    const T* Kg = (const T*)a.k_base + head_off * dh;
    const T* Vg = (const T*)a.v_base + head_off * dh;
    const uint32_t* loc = a.loc + (size_t)seq * a.words;
    const uint32_t* snk = a.snk + (size_t)seq * a.words;
    const bool biased = a.alpha != 0.f || a.beta != 0.f;

    for (int t = 0; t < n_total; ++t) {
        const int j0 = t * kSimtKeysPerTile;
        __syncthreads();
        for (int i = threadIdx.x; i < kSimtKeysPerTile * dh; i += kThreads) {
            const int k = i / dh, d = i % dh, j = j0 + k;
            const bool in = j < a.n_tokens;
            Ks[k * ldk + d] = in ? ldf(Kg + (size_t)j * dh + d) : 0.f;
            Vs[k * ldk + d] = in ? ldf(Vg + (size_t)j * dh + d) : 0.f;
        }
        __syncthreads();
        for (int p = warp; p < pairs; p += kThreads / 32) {
            const int g = Gs[p];
            const float* qp = Qs + p * dh;
            float s[2];
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                const int k = lane + 32 * half, j = j0 + k;
                float acc = 0.f;
                for (int d = 0; d < dh; ++d) acc = fmaf(qp[d], Ks[k * ldk + d], acc);
                if (biased && j < a.n_tokens) {
                    const float lb = (loc[j >> 5] >> (j & 31)) & 1u ? a.alpha : 0.f;
                    const float sb = (snk[j >> 5] >> (j & 31)) & 1u ? a.beta : 0.f;
                    acc += lb + sb;
                }
                s[half] = (j <= g) ? acc : -INFINITY;
            }
            float mt = fmaxf(s[0], s[1]);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, o));
            const float m_old = Ms[p];
            const float m_new = fmaxf(m_old, mt);
            if (m_new == -INFINITY) continue;   // nothing visible yet (cannot happen: key 0 is always visible)
            const float corr = expf(m_old - m_new);
            const float p0 = expf(s[0] - m_new), p1 = expf(s[1] - m_new);
            float ps = p0 + p1;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, o);
            float* op = Os + p * dh;
            for (int d = lane; d < dh; d += 32) {
                float acc = op[d] * corr;
                for (int k = 0; k < 32; ++k) {
                    const float w0 = __shfl_sync(0xffffffffu, p0, k);
                    const float w1 = __shfl_sync(0xffffffffu, p1, k);
                    acc = fmaf(w0, Vs[k * ldk + d], acc);
                    acc = fmaf(w1, Vs[(k + 32) * ldk + d], acc);
                }
                op[d] = acc;
            }
            __syncwarp();
            if (lane == 0) {
                Ms[p] = m_new;
                Ls[p] = Ls[p] * corr + ps;
            }
            __syncwarp();
        }
    }
    __syncthreads();
    T* out = (T*)a.out;
    for (int i = threadIdx.x; i < pairs * dh; i += kThreads) {
        const int p = i / dh, d = i % dh;
        const int r = row0 + p / G, h = kvh * G + p % G;
        stf(out + ((size_t)r * a.n_q_heads + h) * dh + d, Os[i] / Ls[p]);
    }
}

}  // namespace

size_t attn_simt_smem(int head_dim) {
    return sizeof(float) * (2 * kSimtKeysPerTile * (head_dim + 1) + 2 * kMaxPairs * head_dim + 2 * kMaxPairs) +
           sizeof(int) * kMaxPairs;
}

int attn_simt_rows_per_tile(int n_q_heads, int n_kv_heads) {
    const int G = n_q_heads / n_kv_heads;
    return kMaxPairs / G >= 1 ? kMaxPairs / G : 1;
}

cudaError_t launch_attention_simt(const AttnLaunch& a, cudaStream_t s) {
    if (a.n_tiles <= 0) return cudaSuccess;
    const size_t smem = attn_simt_smem(a.head_dim);
    dim3 grid(a.n_tiles, a.n_kv_heads);
    cudaError_t e =
        cudaFuncSetAttribute(attn_simt_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    KVR_LAUNCH(attn_simt_kernel<float>, grid, dim3(kThreads), smem, s, a);
    return cudaSuccess;
}

}  // namespace kvr

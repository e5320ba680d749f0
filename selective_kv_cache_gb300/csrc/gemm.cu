// gemm.cu -- packed-row projections: part[split][r][f] = sum_k x[r][k] w[f][k]
// over the split's K range.
//
// bf16 path (sm_103a, tcgen05): swap-AB.  The weight matrix supplies the MMA
// M dimension (128 output features per CTA) and the packed rows supply N
// (up to 256 rows per CTA), because the row count of a refresh (a few hundred)
// is far below the feature count: the weights stream once from HBM while the
// small activation tile is re-read from L2.  Both operands are K-major bf16
// tiles of 64 elements (128 B) staged by TMA with 128-byte swizzle into a
// multi-stage shared-memory ring; one thread issues tcgen05.mma into an fp32
// TMEM accumulator; four epilogue warps read TMEM (warp w reads lanes
// 32*(w%4)..+31) and store fp32 partials.  Split-K spreads the few feature
// tiles of a projection over all 152 SMs; the epilogue kernels reduce the
// splits in a fixed order.
//
// fp32 path: plain SIMT FFMA tiles (fp32 storage needs fp32 products).
#include <cuda_bf16.h>

#include <algorithm>

#include "kvr_internal.h"
#include "ptx.cuh"

namespace kvr {
namespace {

constexpr int kBK = 64;                 // K elements per stage (128 B of bf16)
constexpr int kTileABytes = 128 * 128;  // 128 rows x 128 B
constexpr int kGemmThreads = 192;       // warp0 TMA, warp1 MMA, warps2-5 epilogue
constexpr int kSmemBudget = 227 * 1024;

struct GemmDev {
    float* part;
    int32_t* err;
    int n_out, K, R, BN, m_tiles, n_tiles, splits, stages, tmem_cols;
};

__global__ void __launch_bounds__(kGemmThreads, 1)
    gemm_bf16_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, GemmDev g) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int BN = g.BN, stages = g.stages;
    const int tileB = BN * 128;
    uint8_t* sA = smem;
    uint8_t* sB = smem + (size_t)stages * kTileABytes;
    uint64_t* full = reinterpret_cast<uint64_t*>(sB + (size_t)stages * tileB);
    uint64_t* empty = full + stages;
    uint64_t* accum = empty + stages;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(accum + 1);

    const int bid = blockIdx.x;
    const int n_t = bid % g.n_tiles;
    const int m_t = (bid / g.n_tiles) % g.m_tiles;
    const int split = bid / (g.n_tiles * g.m_tiles);
    const int KB = g.K / kBK;
    const int kb0 = (int)((long long)split * KB / g.splits);
    const int kb1 = (int)((long long)(split + 1) * KB / g.splits);
    const int nk = kb1 - kb0;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(accum, 1);
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tmA);
        prefetch_tmap(&tmB);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, g.tmem_cols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    bool ok = true;

    if (warp == 0) {
        if (lane == 0) {
            int issued = 0;
            for (int i = 0; i < nk; ++i) {
                const int s = i % stages;
                const uint32_t ph = (uint32_t)(i / stages) & 1u;
                if (!mbar_wait(&empty[s], ph ^ 1u)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(&full[s], (uint32_t)(kTileABytes + tileB));
                tma_load_2d(sA + (size_t)s * kTileABytes, &tmA, &full[s], (kb0 + i) * kBK, m_t * 128);
                tma_load_2d(sB + (size_t)s * tileB, &tmB, &full[s], (kb0 + i) * kBK, n_t * BN);
                ++issued;
            }
            if (!ok) {  // let every copy still in flight land before the CTA exits
                for (int i = (issued > stages ? issued - stages : 0); i < issued; ++i)
                    mbar_wait(&full[i % stages], (uint32_t)(i / stages) & 1u);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16(128, BN, 0, 0);
            for (int i = 0; i < nk; ++i) {
                const int s = i % stages;
                const uint32_t ph = (uint32_t)(i / stages) & 1u;
                if (!mbar_wait(&full[s], ph)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t a0 = smem_u32(sA + (size_t)s * kTileABytes);
                const uint32_t b0 = smem_u32(sB + (size_t)s * tileB);
#pragma unroll
                for (int kk = 0; kk < kBK / 16; ++kk) {
                    mma_bf16(tmem, sdesc_sw128(a0 + kk * 32, 16, 1024), sdesc_sw128(b0 + kk * 32, 16, 1024), idesc,
                             (i | kk) != 0);
                }
                mma_commit(&empty[s]);
            }
            mma_commit(accum);
            if (!ok) mbar_wait(accum, 0);
        }
    } else {
        // one lane polls, the warp follows it: tcgen05.ld needs a converged warp
        int got = 0;
        if (lane == 0) got = mbar_wait(accum, 0) ? 1 : 0;
        got = __shfl_sync(0xffffffffu, got, 0);
        if (!got) {
            ok = false;
        } else {
            tc_fence_after();
            const int q = warp & 3;
            const int feat = m_t * 128 + q * 32 + lane;
            float* out = g.part + (size_t)split * g.R * g.n_out;
            const int tok0 = n_t * BN;
            for (int c = 0; c < BN; c += 16) {
                float v[16];
                tmem_ld16(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)c, v);
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int tok = tok0 + c + j;
                    if (tok < g.R) out[(size_t)tok * g.n_out + feat] = v[j];
                }
            }
        }
    }
    if (!ok) atomicOr(g.err, DEV_ERR_TIMEOUT);
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, g.tmem_cols);
    }
}

// fp32 SIMT: 64 x 64 output tile (rows x features), 256 threads, 4 x 4 each.
__global__ void __launch_bounds__(256) gemm_f32_simt_kernel(const float* __restrict__ w, const float* __restrict__ x,
                                                            float* __restrict__ part, int n_out, int K, int R,
                                                            int splits) {
    __shared__ float xs[16][64 + 4];
    __shared__ float ws[16][64 + 4];
    const int f0 = blockIdx.x * 64, r0 = blockIdx.y * 64, split = blockIdx.z;
    const int k0 = (int)((long long)split * (K / 16) / splits) * 16;
    const int k1 = (int)((long long)(split + 1) * (K / 16) / splits) * 16;
    const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
    float acc[4][4] = {};
    for (int k = k0; k < k1; k += 16) {
        for (int i = threadIdx.x; i < 64 * 16; i += 256) {
            const int rr = i / 16, kk = i % 16;
            xs[kk][rr] = (r0 + rr < R) ? x[(size_t)(r0 + rr) * K + k + kk] : 0.f;
            ws[kk][rr] = (f0 + rr < n_out) ? w[(size_t)(f0 + rr) * K + k + kk] : 0.f;
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < 16; ++kk) {
            float a[4], b[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                a[i] = xs[kk][ty * 4 + i];
                b[i] = ws[kk][tx * 4 + i];
            }
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
        __syncthreads();
    }
    float* out = part + (size_t)split * R * n_out;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int r = r0 + ty * 4 + i;
        if (r >= R) continue;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int f = f0 + tx * 4 + j;
            if (f < n_out) out[(size_t)r * n_out + f] = acc[i][j];
        }
    }
}

int round_up(int x, int m) { return (x + m - 1) / m * m; }

}  // namespace

GemmPlan plan_gemm(int dtype, int n_out, int K, int R) {
    GemmPlan p{};
    p.n_out = n_out;
    p.K = K;
    p.R = R;
    if (dtype == KVR_F32) {
        p.m_tiles = (n_out + 63) / 64;
        p.n_tiles = (R + 63) / 64;
        p.BN = 64;
        const int KB = K / 16;
        const int ctas = p.m_tiles * p.n_tiles;
        p.splits = std::max(1, std::min(KB / 4, (2 * kNumSMs) / std::max(1, ctas)));
        p.stages = 0;
        return p;
    }
    p.m_tiles = n_out / 128;
    p.n_tiles = std::max(1, (R + 255) / 256);
    p.BN = std::max(16, round_up((R + p.n_tiles - 1) / p.n_tiles, 16));
    const int KB = K / kBK;
    // pick the number of K splits that best fills whole waves of CTAs
    const int tiles = p.m_tiles * p.n_tiles;
    const int tileB = p.BN * 128;
    int stages = std::min(8, (kSmemBudget - 1024 - 256) / (kTileABytes + tileB));
    const int per_sm = (2 * (kTileABytes + tileB) * 3 + 2048 <= kSmemBudget && p.BN <= 128) ? 2 : 1;
    if (per_sm == 2) stages = 3;
    p.stages = stages;
    const int slots = kNumSMs * per_sm;
    int best = 1;
    double best_eff = 0.0;
    const int max_split = std::max(1, std::min(KB / 2, 16));
    for (int s = 1; s <= max_split; ++s) {
        const long long ctas = (long long)tiles * s;
        const long long waves = (ctas + slots - 1) / slots;
        const double eff = (double)ctas / (double)(waves * slots);
        // each extra split costs a partial tile round trip: prefer fewer when close
        if (eff > best_eff + 0.05) {
            best_eff = eff;
            best = s;
        }
    }
    p.splits = best;
    return p;
}

size_t gemm_partial_bytes(const GemmPlan& p) { return (size_t)p.splits * p.R * p.n_out * sizeof(float); }

cudaError_t launch_gemm(int dtype, const GemmPlan& p, const void* w, const void* x, float* part, int32_t* err,
                        cudaStream_t s, std::string* why) {
    if (p.R <= 0) return cudaSuccess;
    if (dtype == KVR_F32) {
        dim3 grid(p.m_tiles, p.n_tiles, p.splits);
        gemm_f32_simt_kernel<<<grid, 256, 0, s>>>((const float*)w, (const float*)x, part, p.n_out, p.K, p.R,
                                                   p.splits);
        return cudaGetLastError();
    }
    CUtensorMap ta, tb;
    if (!make_tmap_2d_bf16(&ta, w, (uint64_t)p.K, (uint64_t)p.n_out, (uint64_t)p.K * 2, kBK, 128, why))
        return cudaErrorInvalidValue;
    if (!make_tmap_2d_bf16(&tb, x, (uint64_t)p.K, (uint64_t)p.R, (uint64_t)p.K * 2, kBK, (uint32_t)p.BN, why))
        return cudaErrorInvalidValue;
    GemmDev g;
    g.part = part;
    g.err = err;
    g.n_out = p.n_out;
    g.K = p.K;
    g.R = p.R;
    g.BN = p.BN;
    g.m_tiles = p.m_tiles;
    g.n_tiles = p.n_tiles;
    g.splits = p.splits;
    g.stages = p.stages;
    int cols = 32;
    while (cols < p.BN) cols <<= 1;
    g.tmem_cols = cols;
    const size_t smem = 1024 + (size_t)p.stages * (kTileABytes + p.BN * 128) + (2 * p.stages + 1) * 8 + 16;
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(gemm_bf16_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             kSmemBudget);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    const unsigned grid = (unsigned)(p.m_tiles * p.n_tiles * p.splits);
    gemm_bf16_tc_kernel<<<grid, kGemmThreads, smem, s>>>(ta, tb, g);
    return cudaGetLastError();
}

}  // namespace kvr

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
// TMEM accumulator; twelve epilogue warps, three per TMEM lane quarter (warp
// w reads lanes 32*(w%4)..+31), read it and store fp32 partials.  Split-K spreads the few feature
// tiles of a projection over all 152 SMs; the epilogue kernels reduce the
// splits in a fixed order.  A little above 256 rows, one CTA can take both
// row tiles of a feature tile (two products of N = BN per K step, side by
// side in TMEM): each weight tile then crosses from L2 to one SM instead of
// two, and a stage carries ~24 % fewer bytes per product.
//
// fp32 path: plain SIMT FFMA tiles (fp32 storage needs fp32 products).
#include <cuda_bf16.h>

#include <algorithm>

#include "kvr_internal.h"
#include "ptx.cuh"

namespace kvr {
namespace {

constexpr int kBK = 64;                 // K elements per swizzle atom (128 B of bf16)
constexpr int kTileABytes = 128 * 128;  // 128 rows x 128 B: one atom of A
constexpr int kEpiPer = 3;              // epilogue warps per TMEM lane quarter (store issue is the limit)
constexpr int kEpiWarps = 4 * kEpiPer;
constexpr int kGemmThreads = 64 + 32 * kEpiWarps;   // warp0 TMA, warp1 MMA, warps 2.. epilogue
constexpr int kSmemBudget = 227 * 1024;

struct GemmDev {
    float* part;
    int32_t* err;
    int n_out, K, R, BN, m_tiles, n_tiles, splits, stages, tmem_cols, items, atoms;
    // fused SwiGLU (swiglu_F > 0, one K split): a tile holds 64 gate rows and the
    // 64 matching up rows, interleaved in blocks of 16 (rows 32j..32j+15 gate
    // f0+16j.., rows 32j+16..32j+31 the matching up), so every 32-lane TMEM
    // quarter holds both halves of 16 features; the epilogue writes
    // act[r][f] = silu(g) * u in bf16
    int swiglu_F;
    __nv_bfloat16* act;
    int prefill;   // 1: the weights are written by no kernel of the call (their first tiles load before the wait)
    // Accumulator windows in tensor memory: a CTA's 1st, 3rd, ... item uses
    // the columns 0 .. W - 1, its 2nd, 4th, ... acc_base1 .. acc_base1 + W - 1
    // (W = NSUB * BN).
    // When the two do not fit side by side (ovl = 1) they share the columns
    // [acc_base1, W): the epilogue reads those first and releases them on
    // ovl_free, so the next item's products start while it reads the rest.
    uint32_t acc_base1;
    int ovl;
};

// one lane polls, the whole warp follows with the result
__device__ __forceinline__ bool warp_wait_all(uint64_t* bar, uint32_t parity) {
    return __all_sync(0xffffffffu, mbar_wait(bar, parity)) != 0;
}


// work item -> (feature tile, row group of NSUB row tiles, K range); row groups
// of one feature tile are consecutive items, so CTAs that run at the same time
// share weight tiles in L2
__device__ __forceinline__ void item_coords(const GemmDev& g, int item, int& m_t, int& n_t, int& split, int& kb0,
                                            int& kb1) {
    n_t = item % g.n_tiles;
    const int rest = item / g.n_tiles;
    m_t = rest % g.m_tiles;
    split = rest / g.m_tiles;
    const int KB = g.K / (kBK * g.atoms);
    kb0 = (int)((long long)split * KB / g.splits);
    kb1 = (int)((long long)(split + 1) * KB / g.splits);
}

// Persistent: one CTA per SM walks items blockIdx.x, +gridDim.x, ...  The TMA
// ring runs across item boundaries, and the TMEM accumulator is double
// buffered, so the epilogue of one item overlaps the main loop of the next.
//
// ATOMS (swizzle atoms per ring stage) and NSUB (row tiles per item) are
// compile-time constants so that the MMA issue block is straight-line code:
// one elected lane issues the stage's 4 * ATOMS * NSUB instructions back to
// back from precomputed descriptors.  A single thread's issue loop bounds
// narrow (N < 256) tiles, and runtime-shaped loops around tcgen05.mma cost
// several times the issue time of the instructions.
//
// At most 72 registers a thread: 448 x 72 leaves 33,280 of the SM's 65,536
// registers, enough for one CTA of the row epilogues (512 threads x 64) to
// start beside this CTA under dependent launch.
template <int ATOMS, int NSUB>
__global__ void __maxnreg__(72)
    gemm_bf16_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, GemmDev g) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    constexpr int atoms = ATOMS;
    const int BN = g.BN, stages = g.stages;
    const int tileB = BN * 128;                    // one atom of one row tile of B
    // a stage: ATOMS atoms of A, then for each atom the NSUB row tiles' atoms of B
    const int stA = atoms * kTileABytes, stB = atoms * NSUB * tileB;
    uint8_t* sA = smem;
    uint8_t* sB = smem + (size_t)stages * stA;
    uint64_t* full = reinterpret_cast<uint64_t*>(sB + (size_t)stages * stB);
    uint64_t* empty = full + stages;
    uint64_t* acc_full = empty + stages;   // [2]
    uint64_t* acc_empty = acc_full + 2;    // [2]
    uint64_t* mma_done = acc_empty + 2;
    uint64_t* ovl_free = mma_done + 1;     // the shared columns of the last item's window are read
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ovl_free + 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&acc_full[b], 1);
            mbar_init(&acc_empty[b], kEpiWarps);
        }
        mbar_init(mma_done, 1);
        mbar_init(ovl_free, kEpiWarps);
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
    // dependents may start only once this CTA holds its tensor memory, so a
    // waiting dependent can never keep it from allocating
    pdl_trigger();
    if (warp >= 2) pdl_wait();

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            auto load_a = [&](int s, int kb, int m_t) {
                for (int a = 0; a < atoms; ++a) {
                    const int kx = (kb * atoms + a) * kBK;
                    uint8_t* da = sA + (size_t)s * stA + a * kTileABytes;
                    if (g.swiglu_F) {   // one 4-d box: 16-row blocks g0 u0 g1 u1 g2 u2 g3 u3
                        tma_load_4d(da, &tmA, &full[s], kx, 0, 0, m_t * 4);
                    } else {
                        tma_load_2d(da, &tmA, &full[s], kx, m_t * 128);
                    }
                }
            };
            // The weights are written by no kernel of the call: the weight tiles
            // of the first ring stages go out before the wait for the previous
            // kernel, whose outputs (the activation rows) are read after it.
            int pre = 0;
            for (int item = blockIdx.x; g.prefill && item < g.items && pre < stages; item += gridDim.x) {
                int m_t, n_t, split, kb0, kb1;
                item_coords(g, item, m_t, n_t, split, kb0, kb1);
                for (int kb = kb0; kb < kb1 && pre < stages; ++kb, ++pre) {
                    mbar_arrive_expect_tx(&full[pre], (uint32_t)(stA + stB));
                    load_a(pre, kb, m_t);
                }
            }
            pdl_wait();
            int it = 0;
            for (int item = blockIdx.x; ok && item < g.items; item += gridDim.x) {
                int m_t, n_t, split, kb0, kb1;
                item_coords(g, item, m_t, n_t, split, kb0, kb1);
                for (int kb = kb0; kb < kb1; ++kb, ++it) {
                    const int s = it % stages;
                    if (it >= pre) {
                        if (!mbar_wait(&empty[s], ((uint32_t)(it / stages) & 1u) ^ 1u)) {
                            ok = false;
                            break;
                        }
                        mbar_arrive_expect_tx(&full[s], (uint32_t)(stA + stB));
                        load_a(s, kb, m_t);
                    }
                    for (int a = 0; a < atoms; ++a)
                        for (int j = 0; j < NSUB; ++j)
                            tma_load_2d(sB + (size_t)s * stB + (a * NSUB + j) * tileB, &tmB, &full[s],
                                        (kb * atoms + a) * kBK, (n_t * NSUB + j) * BN);
                }
            }
            if (!ok) {  // let every copy still in flight land before the CTA exits
                for (int i = (it > stages ? it - stages : 0); i < it; ++i)
                    mbar_wait(&full[i % stages], (uint32_t)(i / stages) & 1u);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        // The whole warp walks the loop (every value warp-uniform); one elected
        // lane issues.  Descriptors are formed once and advanced by adding the
        // byte offset >> 4 to the start-address field.
        const uint32_t idesc = idesc_bf16(128, BN, 0, 0);
        const uint64_t descA = sdesc_sw128(smem_u32(sA), 16, 1024);
        const uint64_t descB = sdesc_sw128(smem_u32(sB), 16, 1024);
        constexpr uint32_t atA16 = kTileABytes >> 4, stA16 = atoms * atA16;   // descriptor units (16 B)
        const uint32_t atB16 = (uint32_t)tileB >> 4, stB16 = atoms * NSUB * atB16;
        const bool leader = elect_one();    // the same lane issues every MMA and commit
        int s = 0, local = 0;
        uint32_t phase = 0;
        for (int item = blockIdx.x; ok && item < g.items; item += gridDim.x, ++local) {
            int m_t, n_t, split, kb0, kb1;
            item_coords(g, item, m_t, n_t, split, kb0, kb1);
            const int ab = local & 1;
            if (!warp_wait_all(&acc_empty[ab], ((uint32_t)(local >> 1) & 1u) ^ 1u)) {
                ok = false;
                break;
            }
            // overlapping windows: the previous item's shared columns are read
            if (g.ovl && local > 0 && !warp_wait_all(ovl_free, (uint32_t)(local - 1) & 1u)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t d = tmem + (ab ? g.acc_base1 : 0u);
            for (int kb = kb0; kb < kb1; ++kb) {
                if (!warp_wait_all(&full[s], phase)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (leader) {
                    const uint64_t da = descA + (uint64_t)((uint32_t)s * stA16);
                    const uint64_t db = descB + (uint64_t)((uint32_t)s * stB16);
                    const uint32_t first = kb > kb0 ? 1u : 0u;
#pragma unroll
                    for (int a = 0; a < atoms; ++a)
#pragma unroll
                        for (int kk = 0; kk < kBK / 16; ++kk)
#pragma unroll
                            for (int j = 0; j < NSUB; ++j)
                                mma_bf16(d + (uint32_t)(j * BN), da + (uint64_t)(a * atA16 + 2 * kk),
                                         db + (uint64_t)((a * NSUB + j) * atB16 + 2 * kk), idesc,
                                         (a > 0 || kk > 0) ? 1u : first);
                    mma_commit(&empty[s]);
                }
                __syncwarp();
                if (++s == stages) {
                    s = 0;
                    phase ^= 1u;
                }
            }
            if (!ok) break;
            if (leader) mma_commit(&acc_full[ab]);
            __syncwarp();
        }
        if (leader) mma_commit(mma_done);
        __syncwarp();
        warp_wait_all(mma_done, 0);
    } else {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3, part = (warp - 2) >> 2;
        const int W = NSUB * BN;   // accumulator columns (tokens) of an item
        const uint32_t lane_base = (uint32_t)(q * 32) << 16;
        int local = 0;
        for (int item = blockIdx.x; item < g.items; item += gridDim.x, ++local) {
            int m_t, n_t, split, kb0, kb1;
            item_coords(g, item, m_t, n_t, split, kb0, kb1);
            const int ab = local & 1;
            // one lane polls, the warp follows: tcgen05.ld needs a converged warp
            int got = 0;
            if (lane == 0) got = mbar_wait(&acc_full[ab], (uint32_t)(local >> 1) & 1u) ? 1 : 0;
            got = __shfl_sync(0xffffffffu, got, 0);
            if (!got) {
                ok = false;
                break;
            }
            tc_fence_after();
            const int tok0 = n_t * W;
            const uint32_t src = tmem + lane_base + (ab ? g.acc_base1 : 0u);
            // the warps of a lane quarter split the 16-column chunks of [lo, hi) between them
            auto drain = [&](int lo, int hi) {
                const int n_chunks = (hi - lo) / 16, per = (n_chunks + kEpiPer - 1) / kEpiPer;
                const int c_lo = lo + 16 * min(n_chunks, part * per), c_hi = lo + 16 * min(n_chunks, (part + 1) * per);
                if (!g.swiglu_F) {
                    // TMEM -> fp32 partials part[split][token][feature].  Lane l holds
                    // feature 4a + b (a = l / 4, b = l % 4) for 16 tokens; a 4 x 4
                    // transpose within each quad of lanes (two xor-shuffle stages)
                    // leaves lane l with features 4a..4a+3 of token 4i + b, stored
                    // as one 16-byte vector per 4 tokens.
                    const int b = lane & 3;
                    float* out = g.part + (size_t)split * g.R * g.n_out + m_t * 128 + q * 32 + (lane & ~3);
                    for (int c = c_lo; c < c_hi; c += 16) {
                        float v[16];
                        tmem_ld16(src + (uint32_t)c, v);
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            float x0 = v[4 * i], x1 = v[4 * i + 1], x2 = v[4 * i + 2], x3 = v[4 * i + 3];
                            float a0 = (b & 2) ? x0 : x2, a1 = (b & 2) ? x1 : x3;
                            a0 = __shfl_xor_sync(0xffffffffu, a0, 2);
                            a1 = __shfl_xor_sync(0xffffffffu, a1, 2);
                            if (b & 2) { x0 = a0; x1 = a1; } else { x2 = a0; x3 = a1; }
                            float c0 = (b & 1) ? x0 : x1, c1 = (b & 1) ? x2 : x3;
                            c0 = __shfl_xor_sync(0xffffffffu, c0, 1);
                            c1 = __shfl_xor_sync(0xffffffffu, c1, 1);
                            if (b & 1) { x0 = c0; x2 = c1; } else { x1 = c0; x3 = c1; }
                            const int tok = tok0 + c + 4 * i + b;
                            if (tok < g.R) *reinterpret_cast<float4*>(out + (size_t)tok * g.n_out) = make_float4(x0, x1, x2, x3);
                        }
                    }
                } else {
                    // this warp's lanes 0-15 hold gate of features f0+16q.., lanes 16-31
                    // the matching up.  For a column pair (2p, 2p+1) the gate lane takes
                    // column 2p and the up lane column 2p+1; one exchange across the
                    // half-warps hands each the other half of its pair.
                    const bool up_lane = lane >= 16;
                    const int f = m_t * 64 + q * 16 + (lane & 15);
                    __nv_bfloat16* act = g.act + f;
                    for (int c = c_lo; c < c_hi; c += 16) {
                        float v[16];
                        tmem_ld16(src + (uint32_t)c, v);
#pragma unroll
                        for (int p = 0; p < 8; ++p) {
                            const float a = v[2 * p], b = v[2 * p + 1];
                            const float r = __shfl_xor_sync(0xffffffffu, up_lane ? a : b, 16);
                            const float gv = up_lane ? r : a, uv = up_lane ? b : r;
                            const int tok = tok0 + c + 2 * p + (up_lane ? 1 : 0);
                            const float y = gv / (1.0f + __expf(-gv)) * uv;
                            if (tok < g.R) act[(size_t)tok * g.swiglu_F] = __float2bfloat16_rn(y);
                        }
                    }
                }
            };
            if (g.ovl) {   // the columns the next item's window shares first, then release them
                // shared columns in this window's own numbering
                const int sh_lo = ab ? 0 : (int)g.acc_base1, sh_hi = ab ? W - (int)g.acc_base1 : W;
                drain(sh_lo, sh_hi);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(ovl_free);
                drain(0, sh_lo);
                drain(sh_hi, W);
            } else {
                drain(0, W);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acc_empty[ab]);
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
    pdl_trigger();
    pdl_wait();
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

GemmPlan plan_gemm(int dtype, int n_out, int K, int R, bool pair_rows) {
    GemmPlan p{};
    p.n_out = n_out;
    p.K = K;
    p.R = R;
    p.n_sub = 1;
    if (dtype == KVR_F32) {
        p.m_tiles = (n_out + 63) / 64;
        p.n_tiles = (R + 63) / 64;
        p.BN = 64;
        const int KB = K / 16;
        const int ctas = p.m_tiles * p.n_tiles;
        p.splits = std::max(1, std::min(KB / 4, (2 * kNumSMs) / std::max(1, ctas)));
        p.stages = 0;
        p.atoms = 1;
        return p;
    }
    p.m_tiles = n_out / 128;
    p.n_tiles = std::max(1, (R + 255) / 256);
    p.BN = std::max(16, round_up((R + p.n_tiles - 1) / p.n_tiles, 16));
    p.swiglu_F = 0;
    // Row tiles per item: one, or (two row tiles of at most 160 rows) both
    // row tiles of a feature tile in one CTA.  K depth per pipeline stage: two
    // swizzle atoms (128 elements, 256 B of each weight row), so each TMA
    // round reads longer runs of every row, as long as the ring keeps at
    // least three stages; wide stages take one atom per stage and a deeper
    // ring instead (at BN = 224, five stages of 44 KB instead of two of 88 KB).
    // K splits from a cost model fitted to measurements on GB300: one item
    // streams its (128 + NSUB * BN) x (K / S) operand tiles at ~100 GB/s per
    // SM, the persistent grid runs ceil(items / 152) rounds, and every split
    // adds an fp32 partial round trip of R x n_out at ~6 TB/s.  A pairing
    // must win by 3 %.
    const int ring = kSmemBudget - 1024 - 1024;
    double best_t = 1e30;
    for (int ns = 1; ns <= 2; ++ns) {
        if (ns == 2 && (!pair_rows || p.n_tiles % 2 != 0 || p.BN > 160)) continue;
        const int stage1 = kTileABytes + ns * p.BN * 128;   // one atom of A and of the item's B
        const int atoms = (K % (2 * kBK) == 0 && ring / (2 * stage1) >= 3) ? 2 : 1;
        if (ns == 2 && atoms != 1) continue;
        const int KB = K / (kBK * atoms);
        const int tiles = p.m_tiles * (p.n_tiles / ns);
        const int max_split = std::max(1, std::min(KB / 2, 16));
        for (int s = 1; s <= max_split; ++s) {
            const long long items = (long long)tiles * s;
            const long long rounds = (items + kNumSMs - 1) / kNumSMs;
            const double t = (double)rounds * (128.0 + ns * p.BN) * ((double)K / s) * 2.0 / 100e9 +
                             2.0 * s * (double)R * n_out * 4.0 / 6e12;
            if (t < best_t * 0.97) {
                best_t = t;
                p.splits = s;
                p.n_sub = ns;
                p.atoms = atoms;
                p.stages = std::min(8, ring / (atoms * stage1));
            }
        }
    }
    return p;
}

size_t gemm_partial_bytes(const GemmPlan& p) { return (size_t)p.splits * p.R * p.n_out * sizeof(float); }

cudaError_t launch_gemm(int dtype, const GemmPlan& p, const void* w, const void* x, float* part, int32_t* err,
                        cudaStream_t s, std::string* why, void* act, bool w_written_before) {
    if (p.R <= 0) return cudaSuccess;
    if (dtype == KVR_F32) {
        dim3 grid(p.m_tiles, p.n_tiles, p.splits);
        KVR_LAUNCH(gemm_f32_simt_kernel, grid, dim3(256), 0, s, (const float*)w, (const float*)x, part, p.n_out, p.K,
                   p.R, p.splits);
        return cudaSuccess;
    }
    CUtensorMap ta, tb;
    if (p.swiglu_F) {
        // the [2F, K] gate/up matrix as (K, 16 rows, {gate, up}, F/16 blocks):
        // a {64, 16, 2, 4} box lands as gate and up 16-row blocks in turn
        const uint64_t dims[4] = {(uint64_t)p.K, 16, 2, (uint64_t)p.swiglu_F / 16};
        const uint64_t strides[3] = {(uint64_t)p.K * 2, (uint64_t)p.swiglu_F * p.K * 2, (uint64_t)16 * p.K * 2};
        const uint32_t box[4] = {(uint32_t)kBK, 16, 2, 4};
        if (!make_tmap_4d_bf16(&ta, w, dims, strides, box, why)) return cudaErrorInvalidValue;
    } else if (!make_tmap_2d_bf16(&ta, w, (uint64_t)p.K, (uint64_t)p.n_out, (uint64_t)p.K * 2, kBK, 128, why)) {
        return cudaErrorInvalidValue;
    }
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
    g.n_tiles = p.n_tiles / p.n_sub;   // row groups
    g.splits = p.splits;
    g.stages = p.stages;
    g.items = p.m_tiles * g.n_tiles * p.splits;
    g.atoms = p.atoms;
    g.swiglu_F = p.swiglu_F;
    g.act = (__nv_bfloat16*)act;
    g.prefill = w_written_before ? 0 : 1;
    if (p.swiglu_F && (p.splits != 1 || !act || p.swiglu_F % 64 || p.n_out != 2 * p.swiglu_F)) {
        if (why) *why = "fused SwiGLU needs one K split and an output buffer";
        return cudaErrorInvalidValue;
    }
    // two accumulator windows of W columns: side by side when they fit in
    // the allocation, else at both ends of all 512 columns, sharing the
    // columns [512 - W, W)
    const int W = p.n_sub * p.BN;
    int cols = 32;
    while (cols < 2 * W && cols < 512) cols <<= 1;
    g.tmem_cols = cols;
    g.ovl = 2 * W > cols ? 1 : 0;
    g.acc_base1 = g.ovl ? (uint32_t)(512 - W) : (uint32_t)cols / 2u;
    // alignment slack, pipeline ring, barriers (1 KB)
    const size_t smem = 1024 + (size_t)p.stages * p.atoms * (kTileABytes + p.n_sub * p.BN * 128) + 1024;
    if (W > 512 || p.n_tiles % p.n_sub != 0 || (p.n_sub == 2 && p.atoms != 1) || p.n_sub > 2 ||
        smem > (size_t)kSmemBudget) {
        if (why) *why = "projection plan out of range";
        return cudaErrorInvalidValue;
    }
    static bool attr_set = false;
    if (!attr_set) {
        for (auto* f : {gemm_bf16_tc_kernel<1, 1>, gemm_bf16_tc_kernel<2, 1>, gemm_bf16_tc_kernel<1, 2>}) {
            cudaError_t e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBudget);
            if (e != cudaSuccess) return e;
        }
        attr_set = true;
    }
    const unsigned grid = (unsigned)std::min(g.items, kNumSMs);
    if (p.n_sub == 2)
        KVR_LAUNCH((gemm_bf16_tc_kernel<1, 2>), dim3(grid), dim3(kGemmThreads), smem, s, ta, tb, g);
    else if (p.atoms == 2)
        KVR_LAUNCH((gemm_bf16_tc_kernel<2, 1>), dim3(grid), dim3(kGemmThreads), smem, s, ta, tb, g);
    else
        KVR_LAUNCH((gemm_bf16_tc_kernel<1, 1>), dim3(grid), dim3(kGemmThreads), smem, s, ta, tb, g);
    return cudaSuccess;
}

}  // namespace kvr

// attn_tc.cu -- biased causal grouped-query attention over the mixed cache on
// the sm_103a tensor cores (bf16 storage, fp32 softmax and accumulation).
//
//   s_ij = <q_i, k_j>/sqrt(d_h) + alpha*loc_j + beta*snk_j,   j <= g_i
//   o_i  = sum_j softmax_j(s_ij) v_j
// ("kv-cross-attention-reuse", Sec. 6.4, Logit form; "Budgeted KV-Cache
// Repair for Evolving Contexts", Sec. 13.2, Eq. 22, and Eqs. 23-24 for the
// per-query-tile K/V tile counts that bound the loop.)
//
// One CTA per (query tile, K/V head, K/V chunk).  The 128 MMA rows are the
// tile's positions times the G query heads of that K/V head (row = p*G + i),
// so all of them read the same K/V tiles and one causal limit g_p serves a
// whole group.  Per 128-key tile:
//   warp 0      TMA: K and V tiles (two 64-column boxes each, 128-B swizzle)
//               into 3-stage rings, K one tile ahead of V; keys >= n_tokens
//               arrive as zeros;
//   warp 1      tcgen05.mma: S = Q K^T into one of three TMEM score buffers,
//               up to three tiles ahead of the PV product;
//   warp 6      tcgen05.mma: O += P V into the TMEM output accumulator (V
//               read MN-major straight from its cache layout);
//   warps 2-5   one thread per row: scores from TMEM, scale + bias + causal
//               mask, online softmax in base 2 (the running max is only
//               raised, and O rescaled in TMEM, when it grows by more than
//               2^8, so P stays <= 256), P as bf16 pairs over the tile's
//               scores in TMEM, the A operand of the PV product.
// A query tile's K/V range may be split into chunks of C tiles over several
// CTAs, whose unnormalised O rows and (running max, sum) are merged in one of
// two ways, chosen per selection:
//   by the last CTA: at the end of its chunk each CTA takes a ticket; all but
//     the last store their rows in fp32 to the workspace and count themselves
//     done; the last one waits for that count (its peers are past their main
//     loops, so the wait ends), loads their rows by TMA, merges them with its
//     own and writes the bf16 output;
//   by a merge kernel: every CTA stores its rows and ends; a second launch,
//     one warp per row, merges them.
// Both sum in split order with the same roundings: the output bits do not
// depend on the merge or on which CTA came last.
// Tiles below the plan's n_full are wholly visible to every row and skip the
// causal test.  Every wait is bounded; on a timeout the CTA records the error,
// drains its copies and MMAs, frees TMEM and returns.
#include <cuda_bf16.h>

#include <algorithm>
#include <cstring>

#include "kvr_internal.h"
#include "ptx.cuh"

namespace kvr {
namespace {

constexpr int kThreads = 352;                   // 11 warps
constexpr uint32_t kHalf = 16384;               // 128 rows x 128 B
constexpr uint32_t kTile = 2 * kHalf;           // 128 x 128 bf16
constexpr int kStages = 3;                      // K and V ring depth; K runs one tile ahead of V
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffK = kTile;
constexpr uint32_t kOffV = kOffK + kStages * kTile;
constexpr uint32_t kOffBar = kOffV + kStages * kTile;
constexpr uint32_t kOffLsum = kOffBar + 256;      // [128] the second softmax half's row sums
constexpr uint32_t kSmemBytes = kOffLsum + 512 + 1024;
// split merge: each softmax warp loads the other splits' rows of its 32 rows
// as 128-byte-swizzled 32 x 32-float boxes into its share of the (then idle)
// K and V rings, kMergeRound splits per load round and column pass
constexpr uint32_t kMergeWarpBytes = 2 * kStages * kTile / 4;     // 48 KB per softmax warp
constexpr int kMergeRound = (int)(kMergeWarpBytes / 16384u);      // 3 partial quarters of 16 KB
constexpr int kSBufs = 3;                       // score buffers: the QK product runs two tiles ahead
// TMEM columns: S[b] at 128 b (P, bf16 pairs, over its first 64 once the
// scores are read), O 384-511
constexpr uint32_t kTmemO = 384;
constexpr float kRescale = 8.0f;                // log2 of the largest P before O is rescaled

// max of three (one instruction on sm_100 and later)
__device__ __forceinline__ float max3f(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// one lane polls, the whole warp follows (keeps tcgen05 .sync.aligned ops converged)
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity) {
    int ok = 0;
    if ((threadIdx.x & 31) == 0) ok = mbar_wait(bar, parity) ? 1 : 0;
    return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint4 v) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
}

// kBiased: the alpha/beta logit bias is on (the mask words are read); the
// unbiased instance carries none of that code.
template <bool kBiased>
__global__ void __launch_bounds__(kThreads, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                   const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmP, AttnLaunch a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
    // kv_full[t % 3]: producer step t, K_t and V_{t-1}; s_full[j % 3]: scores
    // of tile j; p_full[j & 3]: P of tile j; o_done[j & 3]: PV of tile j.
    // Four P and O phases keep every waiter ahead of the next completion of
    // the barrier it polls.
    uint64_t* kv_full = bars + 0;                         // [kStages]
    uint64_t* s_full = kv_full + kStages;                 // [kSBufs]
    uint64_t* p_full = s_full + kSBufs;                   // [4]
    uint64_t* o_done = p_full + 4;                        // [4]
    uint64_t* mma_done = o_done + 4;                      // both MMA issuers' last products
    uint64_t* q_full = mma_done + 1;
    uint64_t* merge_full = q_full + 1;                    // [4] one per softmax warp
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(merge_full + 4);
    int* ticket = reinterpret_cast<int*>(tmem_slot + 1);

    // grid (K/V head, query tile from the last, split): the longest query
    // tiles (latest positions) are dispatched first
    const int h = blockIdx.x, tile = gridDim.y - 1 - blockIdx.y, split = blockIdx.z, n_split = gridDim.z;
    const int* plan = a.plan + 8 * tile;
    const int row0 = plan[0], nrows = plan[1], umin = plan[2], n_full = plan[4], seq = plan[6];
    // this CTA's chunk of the query tile's K/V tiles [0, plan n_total)
    const int chunk = n_split > 1 ? a.chunk : plan[5];
    const int jb = split * chunk;
    const int n_total = min(plan[5], jb + chunk) - jb;           // tiles handled here
    if (n_total <= 0) return;                                     // nothing to read, nothing to merge
    const int n_live = min(n_split, (plan[5] + chunk - 1) / chunk);   // CTAs with work on this tile
    const int G = a.n_q_heads / a.n_kv_heads;
    const int P = 128 / G;
    const int head_index = (seq * a.n_layers + a.layer) * a.n_kv_heads + h;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    bool ok = true;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) mbar_init(&kv_full[i], 1);
        for (int i = 0; i < kSBufs; ++i) mbar_init(&s_full[i], 1);
        for (int i = 0; i < 4; ++i) mbar_init(&p_full[i], 8);   // both softmax halves of every quarter
        for (int i = 0; i < 4; ++i) mbar_init(&o_done[i], 1);
        mbar_init(mma_done, 2);
        mbar_init(q_full, 1);
        for (int i = 0; i < 4; ++i) mbar_init(&merge_full[i], 1);
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tmK);
        prefetch_tmap(&tmV);
        prefetch_tmap(&tmQ);
        if (n_live > 1) prefetch_tmap(&tmP);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, 512);
        tmem_relinquish();
    }

    // rows of this thread (softmax warps 2-5 and 7-10): m = 32 * (warp % 4) +
    // lane; warps 2-5 take keys 0-63 of each tile, warps 7-10 keys 64-127
    const int m = 32 * (warp & 3) + lane;
    const int p = m / G, gi = m % G;
    const int half = warp >= 7 ? 1 : 0;
    const bool row_valid = warp >= 2 && warp != 6 && m < P * G && p < nrows;
    // K/V producer, steps t = 0 .. n_total: K_t and V_{t-1} on one barrier,
    // so K stays one tile ahead of V.  The ring slots are freed by the
    // signals the products already send: K_t replaces K_{t-3}, read by the
    // QK product of tile t - 3 (s_full); V_{t-1} replaces V_{t-4}, read by the
    // PV product of tile t - 4 (o_done).  The Q tile (two boxes of 64 dims x
    // G heads x P positions, landing as rows p * G + i) and the first two
    // steps go out before the block-wide barrier, under the tensor-memory
    // allocation.
    int issued = 0;
    auto produce = [&](int t) -> bool {
        const int st = t % kStages;
        if (t >= kStages) {
            // The slot's barrier finished its previous phase (step t - 3), and
            // every thread that polls that phase has seen it: the QK issuer
            // (its product S_{t-3} is done, which also frees K_{t-3}'s slot)
            // and the PV issuer (its product of tile t - 4 is done, which
            // frees V_{t-4}'s slot).  Only then is the barrier re-armed.
            if (!mbar_wait(&kv_full[st], (uint32_t)((t - kStages) / kStages) & 1u) ||
                !mbar_wait(&s_full[(t - 3) % kSBufs], (uint32_t)((t - 3) / kSBufs) & 1u))
                return false;
            if (t >= 4 && !mbar_wait(&o_done[(t - 4) & 3], (uint32_t)((t - 4) >> 2) & 1u)) return false;
        }
        mbar_arrive_expect_tx(&kv_full[st], (t < n_total ? kTile : 0u) + (t >= 1 ? kTile : 0u));
        if (t < n_total) {
            uint8_t* kd = smem + kOffK + st * kTile;
            tma_load_3d(kd, &tmK, &kv_full[st], 0, (jb + t) * 128, head_index);
            tma_load_3d(kd + kHalf, &tmK, &kv_full[st], 64, (jb + t) * 128, head_index);
        }
        if (t >= 1) {
            uint8_t* vd = smem + kOffV + ((t - 1) % kStages) * kTile;
            tma_load_3d(vd, &tmV, &kv_full[st], 0, (jb + t - 1) * 128, head_index);
            tma_load_3d(vd + kHalf, &tmV, &kv_full[st], 64, (jb + t - 1) * 128, head_index);
        }
        ++issued;
        return true;
    };
    int t_prod = 0;
    pdl_wait();   // Q rows and the cache rows written by the previous kernel
    int g = umin;
    if (row_valid) g = a.U[row0 + p];
    if (warp == 0 && lane == 0) {
        // P * G <= 128 rows of 128 bytes in each half (126 when G = 6)
        mbar_arrive_expect_tx(q_full, 2u * 128u * (uint32_t)(P * G));
        tma_load_3d(smem + kOffQ, &tmQ, q_full, 0, h * G, row0);
        tma_load_3d(smem + kOffQ + kHalf, &tmQ, q_full, 64, h * G, row0);
        for (; t_prod < 2 && t_prod <= n_total && ok; ++t_prod) ok = produce(t_prod);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // dependents may start only once this CTA holds its tensor memory
    pdl_trigger();

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            for (int t = t_prod; t <= n_total && ok; ++t) ok = produce(t);
            if (!ok) {  // let every copy still in flight land before the CTA exits
                mbar_wait(q_full, 0);
                for (int t = (issued > kStages ? issued - kStages : 0); t < issued; ++t)
                    mbar_wait(&kv_full[t % kStages], (uint32_t)(t / kStages) & 1u);
            }
        }
    } else if (warp == 1 || warp == 6) {
        // ------------------------------------------------------------ MMA issuers
        // Two threads feed the tensor pipe: warp 1 the score products S_j =
        // Q K_j^T, warp 6 the output products O += P_j V_j.  An issuing thread
        // stalls while the pipe's short queue is full, so while one waits on a
        // barrier the other keeps the pipe busy.  The scores run up to three
        // tiles ahead: S_j goes into buffer j % 3 once the PV product of tile
        // j - 3 has read the P stored over that buffer's scores.  Each thread
        // commits its own products.
        if (lane == 0) {
            auto step_landed = [&](int t) {
                return mbar_wait(&kv_full[t % kStages], (uint32_t)(t / kStages) & 1u);
            };
            if (warp == 1) {
                const uint32_t idesc_s = idesc_bf16(128, 128, 0, 0);
                if (n_total > 0) ok = mbar_wait(q_full, 0);
                for (int j = 0; ok && j < n_total; ++j) {
                    if (!step_landed(j) ||   // K_j
                        (j >= kSBufs && !mbar_wait(&o_done[(j - kSBufs) & 3], (uint32_t)((j - kSBufs) >> 2) & 1u))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t qa = sbase + kOffQ, ka = sbase + kOffK + (uint32_t)(j % kStages) * kTile;
                    const uint32_t d = tmem + (uint32_t)(j % kSBufs) * 128u;
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const uint32_t off = (uint32_t)(kk >> 2) * kHalf + (uint32_t)(kk & 3) * 32u;
                        mma_bf16(d, sdesc_sw128(qa + off, 16, 1024), sdesc_sw128(ka + off, 16, 1024), idesc_s, kk > 0);
                    }
                    mma_commit(&s_full[j % kSBufs]);
                }
            } else {
                const uint32_t idesc_o = idesc_bf16(128, 128, 0, 1);   // V is MN-major
                for (int j = 0; ok && j < n_total; ++j) {
                    if (!mbar_wait(&p_full[j & 3], (uint32_t)(j >> 2) & 1u) || !step_landed(j + 1)) {   // P_j, V_j
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    // O += P V_j: P over the scores of tile j, keys 0-63 in
                    // columns 0-31 of the buffer, keys 64-127 in columns 64-95
                    const uint32_t pt = tmem + (uint32_t)(j % kSBufs) * 128u;
                    const uint32_t va = sbase + kOffV + (uint32_t)(j % kStages) * kTile;
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        mma_bf16_ta(tmem + kTmemO, pt + (uint32_t)(kk & 3) * 8u + (uint32_t)(kk >> 2) * 64u,
                                    sdesc_sw128(va + (uint32_t)kk * 2048u, kHalf, 1024), idesc_o, (j > 0 || kk > 0));
                    }
                    mma_commit(&o_done[j & 3]);
                }
            }
            mma_commit(mma_done);
            mbar_wait(mma_done, 0);
        }
    } else {
        // ------------------------------------------------------------ softmax + epilogue
        // base-2 logit of key k: x_k = (s_k + bias_k) * sl2, the bias in raw
        // score units (alpha*sqrt(d_h) for local keys, beta*sqrt(d_h) for S'),
        // -inf past the row's causal limit
        const float sl2 = 1.4426950408889634f / sqrtf(128.0f);
        const float ar = a.alpha * sqrtf(128.0f), br = a.beta * sqrtf(128.0f);
        constexpr bool biased = kBiased;
        const uint32_t* loc = a.loc + (size_t)seq * a.words;
        const uint32_t* snk = a.snk + (size_t)seq * a.words;
        const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
        float m_run = -INFINITY, l_run = 0.f;
        // S_j is probed without blocking while tile j - 1 is still being
        // worked on, so the probe's latency hides behind that work; the
        // blocking wait runs only if some lane saw the scores not yet there.
        bool s_ready = false;
        // mask words of the tile, loaded one tile ahead so their latency hides
        // behind the previous tile's work
        uint32_t lw[4] = {0u, 0u, 0u, 0u}, sw[4] = {0u, 0u, 0u, 0u};
        auto load_words = [&](int key0, uint32_t* l, uint32_t* k) {
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                const int wd = (key0 >> 5) + t;
                l[t] = wd < a.words ? loc[wd] : 0u;
                k[t] = wd < a.words ? snk[wd] : 0u;
            }
        };
        if (biased && n_total > 0) load_words(jb * 128, lw, sw);
        // The quarter's two halves meet at their pair barrier once per tile
        // (twice when their maxima are swapped) and once after the loop.  A
        // half that gives up on a wait still passes the barriers of the tiles
        // left, asking for no swap, so its partner never blocks there.
        const uint32_t pair_bar = 2u + (uint32_t)(warp & 3);
        auto drain = [&](int from) {
            for (int r = from; r < n_total; ++r)
                if (named_bar_red_or(pair_bar, 64, false)) named_bar_sync(pair_bar, 64);
        };
        for (int j = 0; j < n_total; ++j) {
            const int sb = j % kSBufs;
            if (__any_sync(0xffffffffu, !s_ready) && !warp_wait(&s_full[sb], (uint32_t)(j / kSBufs) & 1u)) {
                ok = false;
                drain(j);
                break;
            }
            tc_fence_after();
            // this half's 64 keys (columns own .. own + 63 of the buffer)
            const uint32_t own = tmem + lane_base + (uint32_t)sb * 128u + 64u * (uint32_t)half;
            float s[64];
            tmem_ld32x2(own, s);

            const int tile_key0 = (jb + j) * 128, key0 = tile_key0 + 64 * half;
            const bool masked = jb + j >= n_full;
            if (biased) {
                // the mask words are the same for every row of the tile, so the
                // branches are warp-uniform: words with no bit set cost nothing,
                // all-local words one add per key
#pragma unroll
                for (int t = 0; t < 2; ++t) {
                    const uint32_t lt = half ? lw[2 + t] : lw[t];
                    const uint32_t st = half ? sw[2 + t] : sw[t];
                    if ((lt | st) == 0u) continue;
                    if (st == 0u && lt == 0xffffffffu) {
#pragma unroll
                        for (int k = 0; k < 32; ++k) s[32 * t + k] += ar;
                        continue;
                    }
#pragma unroll
                    for (int k = 0; k < 32; ++k) {
                        float b = ((lt >> k) & 1u) ? ar : 0.f;
                        b += ((st >> k) & 1u) ? br : 0.f;
                        s[32 * t + k] += b;
                    }
                }
            }
            if (masked) {
                const int lim = g - key0;   // keys k > lim are in the row's future
#pragma unroll
                for (int k = 0; k < 64; ++k)
                    if (k > lim) s[k] = -INFINITY;
            }
            // the half's max over 8 independent chains of 3-input maxima
            float mx[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                mx[i] = fmaxf(s[i], s[i + 8]);
#pragma unroll
                for (int t = 1; t < 4; ++t) mx[i] = max3f(mx[i], s[i + 16 * t], s[i + 16 * t + 8]);
            }
            const float mh = max3f(max3f(mx[0], mx[1], mx[2]), max3f(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7]));
            // The running max is raised only when a tile's max passes it by
            // more than kRescale, so the halves need each other's maxima only
            // when one of them sees that for some row: the pair barrier ORs
            // the halves' findings.  Then they swap their maxima through the
            // last column of their own score halves (read already, and not
            // part of P), ordered by a second pass of the barrier, and both
            // hold the same row max.
            float mt = m_run;
            if (named_bar_red_or(pair_bar, 64, mh * sl2 > m_run + kRescale)) {
                tmem_st1(own + 63u, __float_as_uint(mh));
                tc_fence_before();
                named_bar_sync(pair_bar, 64);
                tc_fence_after();
                const float mo =
                    __uint_as_float(tmem_ld1(tmem + lane_base + (uint32_t)sb * 128u + 64u * (uint32_t)(1 - half) + 63u));
                mt = fmaxf(mh, mo) * sl2;
            }
            s_ready = j + 1 < n_total && mbar_test(&s_full[(j + 1) % kSBufs], (uint32_t)((j + 1) / kSBufs) & 1u);
            if (biased && j + 1 < n_total) load_words(tile_key0 + 128, lw, sw);
            // O is rescaled only after the previous PV has finished.  P_j goes
            // over the scores just read; the buffer's earlier P (tile j - 3)
            // was read before S_j's product was issued, so P_j needs no wait.
            const bool raise = mt > m_run + kRescale;
            const bool rescale = __any_sync(0xffffffffu, raise && j > 0);
            if (rescale) {
                if (!warp_wait(&o_done[(j - 1) & 3], (uint32_t)((j - 1) >> 2) & 1u)) {
                    ok = false;
                    drain(j + 1);
                    break;
                }
                tc_fence_after();
            }
            if (rescale) {   // each half rescales its 64 of O's columns
                const float f = raise ? ex2(m_run - mt) : 1.f;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    float o[16];
                    const uint32_t col = kTmemO + 64u * (uint32_t)half + (uint32_t)c * 16u;
                    tmem_ld16(tmem + lane_base + col, o);
#pragma unroll
                    for (int t = 0; t < 16; ++t) o[t] *= f;
                    tmem_st16(tmem + lane_base + col, o);
                }
                if (raise) l_run *= f;
            }
            if (raise) m_run = mt;
            // p = 2^(x - m): one packed FMA per two keys, then ex2; l sums the
            // fp32 probabilities (the PV product sees them rounded to bf16: a
            // relative difference of at most 2^-9 per term, unbiased)
            // P goes to tensor memory as the PV product's A operand over this
            // half's own scores: column own + c holds its keys 2c, 2c+1 as
            // packed bf16
            const float2 sc = make_float2(sl2, sl2), nm = make_float2(-m_run, -m_run);
            const uint32_t ptm = own;
            float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                             make_float2(0.f, 0.f)};
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                uint32_t pk[16];
#pragma unroll
                for (int t = 0; t < 16; ++t) {
                    const int k = 32 * c + 2 * t;
                    const float2 x = __ffma2_rn(make_float2(s[k], s[k + 1]), sc, nm);
                    const float2 e = make_float2(ex2(x.x), ex2(x.y));
                    pk[t] = pack_bf16(e.x, e.y);
                    acc[t & 3] = __fadd2_rn(acc[t & 3], e);
                }
                tmem_st16_async(ptm + 16u * (uint32_t)c, pk);
            }
            tmem_wait_st();
            const float2 a01 = __fadd2_rn(acc[0], acc[1]), a23 = __fadd2_rn(acc[2], acc[3]);
            const float2 a03 = __fadd2_rn(a01, a23);
            l_run += a03.x + a03.y;
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&p_full[j & 3]);
        }
        // the second half hands its row sums to the first, which finishes the
        // rows (l = first half's sum + second half's)
        float* lsum = reinterpret_cast<float*>(smem + kOffLsum);
        if (half) lsum[m] = l_run;
        named_bar_sync(pair_bar, 64);
        if (!half) l_run += lsum[m];
        if (!half && ok && !warp_wait(&o_done[(n_total - 1) & 3], (uint32_t)((n_total - 1) >> 2) & 1u)) ok = false;
        __nv_bfloat16* out = (__nv_bfloat16*)a.out + ((size_t)(row0 + p) * a.n_q_heads + h * G + gi) * 128;
        if (half) {
            // done: O and the merge are the first half's
        } else if (n_live == 1) {
            if (ok) {
                tc_fence_after();
                const float inv = 1.0f / l_run;
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    float o[16];
                    tmem_ld16(tmem + lane_base + kTmemO + (uint32_t)c * 16u, o);
                    if (row_valid) {
                        uint4 v0, v1;
                        v0.x = pack_bf16(o[0] * inv, o[1] * inv);
                        v0.y = pack_bf16(o[2] * inv, o[3] * inv);
                        v0.z = pack_bf16(o[4] * inv, o[5] * inv);
                        v0.w = pack_bf16(o[6] * inv, o[7] * inv);
                        v1.x = pack_bf16(o[8] * inv, o[9] * inv);
                        v1.y = pack_bf16(o[10] * inv, o[11] * inv);
                        v1.z = pack_bf16(o[12] * inv, o[13] * inv);
                        v1.w = pack_bf16(o[14] * inv, o[15] * inv);
                        reinterpret_cast<uint4*>(out + c * 16)[0] = v0;
                        reinterpret_cast<uint4*>(out + c * 16)[1] = v1;
                    }
                }
            }
        } else {
            // ------------------------------------------------ split merge
            const int pair = tile * a.n_kv_heads + h;
            int* count = a.sync + pair;                                   // tickets taken
            int* done = a.sync + (size_t)a.n_tiles * a.n_kv_heads + pair;  // partials stored
            const int q4 = warp & 3;
            const bool merge_here = a.merge == kAttnMergeLastCTA;   // launch-uniform
            if (merge_here) {
                if (warp == 2 && lane == 0) *ticket = atomicAdd(count, 1);
                named_bar_sync(1, 128);
            }
            const bool last = merge_here && *ticket == n_live - 1;   // CTA-uniform
            if (!last) {
                // unnormalised fp32 rows plus (running max in base 2, sum): the
                // warp's 32 rows leave as four TMA stores of 32 x 32 floats
                // staged in the idle K ring in the 128-byte swizzle
                tc_fence_after();
                const size_t slot = ((size_t)split * a.n_tiles + tile) * a.n_kv_heads + h;
                uint8_t* stg = smem + kOffK + (uint32_t)q4 * 16384u;
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    float o[16];
                    tmem_ld16(tmem + lane_base + kTmemO + (uint32_t)c * 16u, o);
#pragma unroll
                    for (int t = 0; t < 4; ++t) {
                        const int j = (c & 1) * 4 + t;   // 16-byte chunk within the box row
                        const uint32_t addr = smem_u32(stg) + (uint32_t)(c >> 1) * 4096u + (uint32_t)lane * 128u +
                                              ((uint32_t)(j ^ (lane & 7)) << 4);
                        st_shared_v4(addr, make_uint4(__float_as_uint(o[4 * t]), __float_as_uint(o[4 * t + 1]),
                                                      __float_as_uint(o[4 * t + 2]), __float_as_uint(o[4 * t + 3])));
                    }
                }
                a.part_ml[(slot * 128 + m) * 2] = m_run;
                a.part_ml[(slot * 128 + m) * 2 + 1] = l_run;
                __threadfence();
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    for (int cb = 0; cb < 4; ++cb)
                        tma_store_2d(&tmP, stg + cb * 4096, cb * 32, (int)(slot * 128) + 32 * q4);
                    bulk_commit();
                    if (merge_here) {
                        bulk_wait_all();            // the rows are in global memory
                        fence_proxy_async_global();
                        __threadfence();
                    } else {
                        bulk_wait_read_all();       // the staging may be released; the rows land before the grid ends
                    }
                }
                if (merge_here) {
                    named_bar_sync(1, 128);
                    if (warp == 2 && lane == 0) {   // after every warp's stores and fences: a release
                        __threadfence();
                        atomicAdd(done, 1);
                    }
                }
            } else {
                // every peer took its ticket after its main loop, so each is
                // only storing its rows now: wait for all n_live - 1 of them
                if (warp == 2 && lane == 0) *ticket = spin_ge_acquire(done, n_live - 1) ? 1 : 0;
                named_bar_sync(1, 128);
                if (!*ticket) ok = false;
                __threadfence();
                // weights of the splits: w_s = 2^(m_s - M), L = sum_s w_s l_s; a
                // split that saw no visible key of this row kept m = -inf and
                // takes no part (its sum and rows are not numbers).  The sums
                // run in split order whichever CTA merges, with products and
                // sums rounded separately, so the output does not depend on
                // which CTA came last.  The merged rows build up 16 columns at a
                // time in the (now idle) score-buffer columns of tensor memory,
                // beside this CTA's own rows, so few registers are live.
                float msp[8], lsp[8];   // the first 8 splits' (max, sum); later ones are read again when used
                float M = -INFINITY;
                for (int sp = 0; sp < n_live; ++sp) {
                    float ms = m_run, ls = l_run;
                    if (sp != split) {
                        const size_t slot = ((size_t)sp * a.n_tiles + tile) * a.n_kv_heads + h;
                        ms = a.part_ml[(slot * 128 + m) * 2];
                        ls = a.part_ml[(slot * 128 + m) * 2 + 1];
                    }
                    if (sp < 8) {
                        msp[sp] = ms;
                        lsp[sp] = ls;
                    }
                    M = fmaxf(M, ms);
                }
                auto ml_of = [&](int sp, float* ms, float* ls) {
                    if (sp < 8) {
                        *ms = msp[sp];
                        *ls = lsp[sp];
                    } else if (sp == split) {
                        *ms = m_run;
                        *ls = l_run;
                    } else {
                        const size_t slot = ((size_t)sp * a.n_tiles + tile) * a.n_kv_heads + h;
                        *ms = a.part_ml[(slot * 128 + m) * 2];
                        *ls = a.part_ml[(slot * 128 + m) * 2 + 1];
                    }
                };
                float L = 0.f;
                for (int sp = 0; sp < n_live; ++sp) {
                    float ms, ls;
                    ml_of(sp, &ms, &ls);
                    if (ms != -INFINITY) L = __fadd_rn(L, __fmul_rn(ex2(ms - M), ls));
                }
                tc_fence_after();
                const uint32_t region = sbase + kOffK + (uint32_t)q4 * kMergeWarpBytes;
                const uint32_t acc_cols = tmem + lane_base;   // the first score buffer's 128 columns
                uint32_t phase = 0;
                // rounds: runs of consecutive splits holding up to kMergeRound
                // others (and this CTA's own split where it falls in order);
                // one load round trip and one pass over the columns per round
                int sp0 = 0;
                bool first = true;
                while (sp0 < n_live && ok) {
                    int ids[kMergeRound + 1], slots[kMergeRound + 1];
                    int n_ids = 0, n_oth = 0, e = sp0;
                    while (e < n_live && n_ids < kMergeRound + 1 && (e == split || n_oth < kMergeRound)) {
                        ids[n_ids] = e;
                        slots[n_ids] = e == split ? -1 : n_oth++;
                        ++n_ids;
                        ++e;
                    }
                    if (n_oth > 0) {
                        if (lane == 0) {
                            fence_proxy_async_global();
                            mbar_arrive_expect_tx(&merge_full[q4], (uint32_t)n_oth * 16384u);
                            for (int i = 0; i < n_ids; ++i) {
                                if (slots[i] < 0) continue;
                                const int slot = (ids[i] * a.n_tiles + tile) * a.n_kv_heads + h;
                                for (int cb = 0; cb < 4; ++cb)
                                    tma_load_2d(smem + kOffK + (uint32_t)q4 * kMergeWarpBytes + (uint32_t)slots[i] * 16384u +
                                                    (uint32_t)cb * 4096u,
                                                &tmP, &merge_full[q4], cb * 32, slot * 128 + 32 * q4);
                            }
                        }
                        if (!warp_wait(&merge_full[q4], phase)) {
                            ok = false;
                            break;
                        }
                        phase ^= 1u;
                    }
                    float wv[kMergeRound + 1];
#pragma unroll
                    for (int i = 0; i < kMergeRound + 1; ++i) {
                        wv[i] = 0.f;
                        if (i < n_ids) {
                            float ms, ls;
                            ml_of(ids[i], &ms, &ls);
                            wv[i] = ms == -INFINITY ? 0.f : ex2(ms - M);
                        }
                    }
                    for (int c = 0; c < 8; ++c) {   // 16 output columns at a time
                        float acc[16];
                        if (!first) tmem_ld16(acc_cols + (uint32_t)c * 16u, acc);
#pragma unroll
                        for (int i = 0; i < kMergeRound + 1; ++i) {
                            if (i >= n_ids) break;
                            float v[16];
                            if (slots[i] < 0) {
                                tmem_ld16(tmem + lane_base + kTmemO + (uint32_t)c * 16u, v);
                            } else {
                                const uint32_t base = region + (uint32_t)slots[i] * 16384u + (uint32_t)lane * 128u;
#pragma unroll
                                for (int t = 0; t < 4; ++t) {
                                    const int q16 = 4 * c + t;   // 16-byte chunk of the row
                                    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                                                 : "=f"(v[4 * t]), "=f"(v[4 * t + 1]), "=f"(v[4 * t + 2]),
                                                   "=f"(v[4 * t + 3])
                                                 : "r"(base + (uint32_t)(q16 >> 3) * 4096u +
                                                       ((uint32_t)((q16 & 7) ^ (lane & 7)) << 4)));
                                }
                            }
                            const bool init = first && i == 0;   // split 0 starts the sum
#pragma unroll
                            for (int x = 0; x < 16; ++x) {
                                const float term = wv[i] == 0.f ? 0.f : __fmul_rn(wv[i], v[x]);
                                acc[x] = init ? term : __fadd_rn(acc[x], term);
                            }
                        }
                        tmem_st16(acc_cols + (uint32_t)c * 16u, acc);
                    }
                    first = false;
                    sp0 = e;
                    __syncwarp();   // the next round's loads reuse this warp's region
                }
                if (ok) {
                    const float inv = 1.0f / L;
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        float o[16];
                        tmem_ld16(acc_cols + (uint32_t)c * 16u, o);
                        if (row_valid) {
                            uint4 v0, v1;
                            v0.x = pack_bf16(o[0] * inv, o[1] * inv);
                            v0.y = pack_bf16(o[2] * inv, o[3] * inv);
                            v0.z = pack_bf16(o[4] * inv, o[5] * inv);
                            v0.w = pack_bf16(o[6] * inv, o[7] * inv);
                            v1.x = pack_bf16(o[8] * inv, o[9] * inv);
                            v1.y = pack_bf16(o[10] * inv, o[11] * inv);
                            v1.z = pack_bf16(o[12] * inv, o[13] * inv);
                            v1.w = pack_bf16(o[14] * inv, o[15] * inv);
                            reinterpret_cast<uint4*>(out + c * 16)[0] = v0;
                            reinterpret_cast<uint4*>(out + c * 16)[1] = v1;
                        }
                    }
                }
                named_bar_sync(1, 128);
                if (warp == 2 && lane == 0) {   // every peer has counted itself: ready for the next launch
                    *count = 0;
                    *done = 0;
                }
            }
        }
    }
    if (!ok) atomicOr(a.err, DEV_ERR_TIMEOUT);
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// The merge kernel: one warp per MMA row of a split (query tile, K/V head),
// four output columns per lane.  It does the last CTA's arithmetic in the
// same order (M the largest split max, L and the rows summed in split order
// with products and sums rounded separately, splits with no visible key of
// the row left out), so either merge writes the same bits.  Lane k holds
// split k's (max, sum); the rows of the first four splits are loaded with
// them, so up to four splits cost one load round trip.
// plan0/1/5: the query tile's first row, row count and K/V tile count.
__device__ __forceinline__ void merge_row(const AttnLaunch& a, int tile, int h, int m, int G, int lane, int plan0,
                                          int plan1, int plan5) {
    const int p = m / G, gi = m - p * G;
    const int n_live = min(a.n_split, (plan5 + a.chunk - 1) / a.chunk);
    if (n_live <= 1 || m >= (128 / G) * G || p >= plan1) return;   // written by the attention, or no row
    const float2* ml = reinterpret_cast<const float2*>(a.part_ml);
    const float4* rows = reinterpret_cast<const float4*>(a.part_o);
    auto row_of = [&](int sp) { return (((size_t)sp * a.n_tiles + tile) * a.n_kv_heads + h) * 128 + m; };
    constexpr int kGroup = 4;
    float4 v[kGroup];
#pragma unroll
    for (int k = 0; k < kGroup; ++k)
        v[k] = k < n_live ? rows[row_of(k) * 32 + lane] : make_float4(0.f, 0.f, 0.f, 0.f);
    const float2 mine = lane < n_live ? ml[row_of(lane)] : make_float2(-INFINITY, 0.f);
    float M = mine.x;
    for (int s0 = 32; s0 < n_live; s0 += 32)
        if (s0 + lane < n_live) M = fmaxf(M, ml[row_of(s0 + lane)].x);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    // weight and sum term of split s0 + lane, L summed in split order
    float L = 0.f, w_mine = 0.f;
    for (int s0 = 0; s0 < n_live; s0 += 32) {
        const float2 x = s0 == 0 ? mine : (s0 + lane < n_live ? ml[row_of(s0 + lane)] : make_float2(-INFINITY, 0.f));
        const float w = x.x == -INFINITY ? 0.f : ex2(x.x - M);
        const float term = x.x == -INFINITY ? 0.f : __fmul_rn(w, x.y);
        if (s0 == 0) w_mine = w;
        const int n = min(32, n_live - s0);
        for (int k = 0; k < n; ++k) {
            const float tk = __shfl_sync(0xffffffffu, term, k);
            const float mk = __shfl_sync(0xffffffffu, x.x, k);
            if (mk != -INFINITY) L = __fadd_rn(L, tk);
        }
    }
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s0 = 0; s0 < n_live; s0 += kGroup) {
        if (s0 > 0) {
#pragma unroll
            for (int k = 0; k < kGroup; ++k)
                if (s0 + k < n_live) v[k] = rows[row_of(s0 + k) * 32 + lane];
        }
#pragma unroll
        for (int k = 0; k < kGroup; ++k) {
            const int sp = s0 + k;
            if (sp >= n_live) break;
            float w;
            if (sp < 32) {
                w = __shfl_sync(0xffffffffu, w_mine, sp);
            } else {
                const float ms = ml[row_of(sp)].x;
                w = ms == -INFINITY ? 0.f : ex2(ms - M);
            }
            const float4 t = w == 0.f ? make_float4(0.f, 0.f, 0.f, 0.f)
                                      : make_float4(__fmul_rn(w, v[k].x), __fmul_rn(w, v[k].y),
                                                    __fmul_rn(w, v[k].z), __fmul_rn(w, v[k].w));
            if (sp == 0) {
                acc = t;   // split 0 starts the sum
            } else {
                acc.x = __fadd_rn(acc.x, t.x);
                acc.y = __fadd_rn(acc.y, t.y);
                acc.z = __fadd_rn(acc.z, t.z);
                acc.w = __fadd_rn(acc.w, t.w);
            }
        }
    }
    const float inv = 1.0f / L;
    __nv_bfloat16* out = (__nv_bfloat16*)a.out + ((size_t)(plan0 + p) * a.n_q_heads + h * G + gi) * 128;
    uint2 o;
    o.x = pack_bf16(acc.x * inv, acc.y * inv);
    o.y = pack_bf16(acc.z * inv, acc.w * inv);
    reinterpret_cast<uint2*>(out)[lane] = o;
}

// Grid (16, K/V heads, query tiles up to 65,535, walked beyond): block x of a
// (tile, head) holds its rows 8x..8x+7, one a warp, so no thread divides
// its index into (tile, head, row).  Four splits per load group keep it at
// 48 registers, five CTAs an SM (the Llama-shaped selection's 1152 CTAs in
// 1.5 waves instead of 1.9); the first tile's plan (written by the
// selection, before any kernel of this call) is read before the wait for
// the attention.
__global__ void __launch_bounds__(256, 5) attn_merge_kernel(AttnLaunch a) {
    const int m = (int)blockIdx.x * 8 + (int)(threadIdx.x >> 5);
    const int G = a.n_q_heads / a.n_kv_heads;
    int tile = blockIdx.z;
    const int* plan = a.plan + 8 * tile;
    int plan0 = plan[0], plan1 = plan[1], plan5 = plan[5];
    pdl_wait();   // every split's rows are stored
    pdl_trigger();
    while (true) {
        merge_row(a, tile, (int)blockIdx.y, m, G, (int)(threadIdx.x & 31), plan0, plan1, plan5);
        tile += gridDim.z;
        if (tile >= a.n_tiles) break;
        plan = a.plan + 8 * tile;
        plan0 = plan[0];
        plan1 = plan[1];
        plan5 = plan[5];
    }
}

}  // namespace

int attn_tc_rows_per_tile(int n_q_heads, int n_kv_heads) { return 128 / (n_q_heads / n_kv_heads); }

namespace {
cudaError_t set_smem_attr() {
    static bool attr = false;
    if (!attr) {
        for (auto* f : {attn_tc_kernel<false>, attn_tc_kernel<true>}) {
            cudaError_t e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
            if (e != cudaSuccess) return e;
        }
        attr = true;
    }
    return cudaSuccess;
}
}  // namespace

size_t attn_tc_scratch_bytes(int n_split, int n_tiles, int n_kv_heads) {
    if (n_split <= 1) return 0;
    return (size_t)n_split * n_tiles * n_kv_heads * 128 * (128 + 2) * sizeof(float);
}

cudaError_t launch_attention_tc(const AttnLaunch& a, cudaStream_t s, std::string* why) {
    if (a.n_tiles <= 0) return cudaSuccess;
    if (a.head_dim != 128 || a.n_q_heads / a.n_kv_heads > 128) {
        if (why) *why = "tensor-core attention needs head_dim 128";
        return cudaErrorInvalidValue;
    }
    const int n_split =
        (a.part_o && (a.sync || a.merge == kAttnMergeKernel) && a.n_split > 1) ? a.n_split : 1;
    CUtensorMap tk, tv;
    const uint64_t heads = (uint64_t)a.batch * a.n_layers * a.n_kv_heads;
    const uint64_t row_bytes = 128 * 2, head_bytes = (uint64_t)a.capacity * row_bytes;
    if (!make_tmap_3d_bf16(&tk, a.k_base, 128, (uint64_t)a.n_tokens, heads, row_bytes, head_bytes, 64, 128, 1, why))
        return cudaErrorInvalidValue;
    if (!make_tmap_3d_bf16(&tv, a.v_base, 128, (uint64_t)a.n_tokens, heads, row_bytes, head_bytes, 64, 128, 1, why))
        return cudaErrorInvalidValue;
    cudaError_t e = set_smem_attr();
    if (e != cudaSuccess) return e;
    // Q [rows][H_q][128] as (dims, heads, rows): a {64, G, 128 / G} box is one
    // half of a query tile, rows p * G + i
    CUtensorMap tq, tp;
    const int G = a.n_q_heads / a.n_kv_heads;
    if (a.n_rows <= 0 ||
        !make_tmap_3d_bf16(&tq, a.q, 128, (uint64_t)a.n_q_heads, (uint64_t)a.n_rows, 256, (uint64_t)a.n_q_heads * 256,
                           64, (uint32_t)G, (uint32_t)(128 / G), why))
        return cudaErrorInvalidValue;
    // the split partials: fp32 rows of 128, stored and loaded as 32 x 32 boxes
    memset(&tp, 0, sizeof(tp));
    if (n_split > 1 &&
        !make_tmap_2d_f32_sw128(&tp, a.part_o, 128, (uint64_t)n_split * a.n_tiles * a.n_kv_heads * 128, 32, why))
        return cudaErrorInvalidValue;
    AttnLaunch b = a;
    b.n_split = n_split;
    dim3 grid((unsigned)a.n_kv_heads, (unsigned)a.n_tiles, (unsigned)n_split);
    if (a.alpha != 0.f || a.beta != 0.f)
        KVR_LAUNCH(attn_tc_kernel<true>, grid, dim3(kThreads), (size_t)kSmemBytes, s, tk, tv, tq, tp, b);
    else
        KVR_LAUNCH(attn_tc_kernel<false>, grid, dim3(kThreads), (size_t)kSmemBytes, s, tk, tv, tq, tp, b);
    if (n_split > 1 && b.merge == kAttnMergeKernel)
        KVR_LAUNCH(attn_merge_kernel, dim3(16, (unsigned)a.n_kv_heads, (unsigned)std::min(a.n_tiles, 65535)), dim3(256),
                   0, s, b);
    return cudaSuccess;
}

}  // namespace kvr

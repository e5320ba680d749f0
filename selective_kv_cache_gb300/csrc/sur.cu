// sur.cu -- Semantic-Unit Refresh selection ("Budgeted KV-Cache Repair for
// Evolving Contexts", Sec. 3.2 and Sec. 7.3: Eqs. 1/7 for token relevance,
// ranked admission of whole units, Eq. 8 for the window of the unit that
// does not fit).
//
//   sur_qnorm_kernel    one CTA per query token: E[q_j] / ||E[q_j]|| in fp32
//   sur_score_kernel    64 suffix tokens per CTA against all queries: an fp32
//                       tiled dot product (16 outputs per thread), the row
//                       max over queries, 1/||E[s_i]||, and the 0.25 bonus
//                       for a token that occurs in the query (whose cosine
//                       with its own embedding is exactly 1)
//   sur_unit_kernel     one warp per unit: mean of the four largest scores
//   sur_rank_kernel     one thread per unit: its rank by (score desc, start asc)
//   sur_admit_kernel    one CTA: admission in rank order by a block scan of
//                       unit sizes, the forward-envelope window of the first
//                       unit that does not fit, and compaction of the selected
//                       tokens into ascending global positions
// The scoring contraction is fp32 as the pages state.  For bf16 embeddings it
// runs on the tensor cores (sur_prep_kernel: the query split and the suffix
// rows' gather in one launch; the tcgen05 projection kernel;
// sur_finish_kernel): the normalised query splits exactly into three bf16
// terms and bf16 products are exact in fp32, so the dot products are fp32 up
// to summation order.  fp32 embeddings take the FFMA kernel.  Everything after
// it is a few passes over S floats.  Kernels after the projection go out as
// dependent launches: each starts while its predecessor drains and waits for
// it before reading what it wrote.
#include <cuda_bf16.h>

#include <climits>
#include <cmath>

#include "kvr_internal.h"

namespace kvr {
namespace {

constexpr int kTokTile = 64;    // suffix tokens per CTA
constexpr int kQryTile = 64;    // queries per inner tile
constexpr int kKTile = 32;      // embedding dims per smem step
constexpr int kAdmitThreads = 1024;

__device__ __forceinline__ float ldf(const float* p) { return *p; }
__device__ __forceinline__ float ldf(const __nv_bfloat16* p) { return __bfloat162float(*p); }

struct SurWs {
    int32_t* err;        // [4]
    float* qn;           // [Q][d] normalised query rows
    float* scores;       // [S]
    float* unit_score;   // [n_units]
    int32_t* order;      // [n_units] unit of each rank
    uint32_t* sel;       // [ceil(S/32)]
    double* cum;         // [S] prefix sums of the envelope of the partial unit
    // bf16 embeddings: the scoring contraction on the tensor cores
    __nv_bfloat16* qp;   // [3Q][d] normalised query rows as hi, mid and lo bf16 terms
    __nv_bfloat16* eg;   // [S_pad][d] gathered suffix embedding rows (zero rows past S)
    float* enorm;        // [S] ||E[s_i]||, or -1 for a token that occurs in the query
    float* part;         // GEMM partials [splits][3Q][S_pad]
};

template <typename T>
__global__ void __launch_bounds__(256) sur_qnorm_kernel(const T* __restrict__ E, int vocab, int d,
                                                        const int32_t* __restrict__ qids, float* __restrict__ qn,
                                                        int32_t* err) {
    __shared__ float red[256];
    const int j = blockIdx.x;
    const int id = qids[j];
    float* out = qn + (size_t)j * d;
    if (id < 0 || id >= vocab) {
        if (threadIdx.x == 0) atomicOr(err, DEV_ERR_INDEX);
        for (int k = threadIdx.x; k < d; k += blockDim.x) out[k] = 0.f;
        return;
    }
    const T* row = E + (size_t)id * d;
    float ss = 0.f;
    for (int k = threadIdx.x; k < d; k += blockDim.x) {
        const float v = ldf(row + k);
        ss = fmaf(v, v, ss);
    }
    red[threadIdx.x] = ss;
    __syncthreads();
    for (int w = 128; w > 0; w >>= 1) {
        if (threadIdx.x < w) red[threadIdx.x] += red[threadIdx.x + w];
        __syncthreads();
    }
    const float nrm = sqrtf(red[0]);
    const float inv = nrm > 0.f ? 1.0f / nrm : 0.f;
    for (int k = threadIdx.x; k < d; k += blockDim.x) out[k] = ldf(row + k) * inv;
}

// 8 consecutive embedding values as fp32 (one 16-byte load for bf16)
__device__ __forceinline__ void ld8f(const __nv_bfloat16* p, float* v) {
    const uint4 u = *reinterpret_cast<const uint4*>(p);
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 f = __bfloat1622float2(h[i]);
        v[2 * i] = f.x;
        v[2 * i + 1] = f.y;
    }
}
__device__ __forceinline__ void ld8f(const float* p, float* v) {
    const float4 a = reinterpret_cast<const float4*>(p)[0], b = reinterpret_cast<const float4*>(p)[1];
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

// scores[i] = max_j <E[s_i], qn_j> / ||E[s_i]|| + 0.25 * [s_i in q]
// 64 tokens x 64 queries per CTA and step, 32 dimensions per step: thread
// (ty, tx) owns tokens 4ty.. and queries 4tx.., 16 products from two float4
// shared reads per dimension; each thread fetches one token row and one query
// row segment of 8 dimensions per step, the next step's while this one runs.
// Needs d % 8 == 0.
template <typename T>
__global__ void __launch_bounds__(256) sur_score_kernel(const T* __restrict__ E, int vocab, int d,
                                                        const int32_t* __restrict__ sids, int S,
                                                        const int32_t* __restrict__ qids, int Q,
                                                        const float* __restrict__ qn, float* __restrict__ scores,
                                                        int32_t* err) {
    constexpr int kPad = 4;
    __shared__ __align__(16) float ts[kKTile][kTokTile + kPad];   // token chunk, k-major
    __shared__ __align__(16) float qs[kKTile][kQryTile + kPad];   // query chunk, k-major
    __shared__ float rowmax[kTokTile];
    __shared__ float rownorm[kTokTile];
    __shared__ int rowid[kTokTile];
    const int i0 = blockIdx.x * kTokTile;
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;   // 16 x 16 threads, 4 x 4 outputs each
    const int lr = threadIdx.x >> 2, lk = (threadIdx.x & 3) * 8;   // the row and 8 dims this thread fetches
    if (threadIdx.x < kTokTile) {
        const int i = i0 + threadIdx.x;
        int id = i < S ? sids[i] : -1;
        if (i < S && (id < 0 || id >= vocab)) {
            atomicOr(err, DEV_ERR_INDEX);
            id = -1;
        }
        rowid[threadIdx.x] = id;
        rowmax[threadIdx.x] = -INFINITY;
    }
    __syncthreads();
    const int my_id = rowid[lr];
    float nrm = 0.f;   // sum of squares of this thread's token segment (first query tile)
    for (int j0 = 0; j0 < Q; j0 += kQryTile) {
        float acc[4][4];
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
            for (int b = 0; b < 4; ++b) acc[a][b] = 0.f;
        const int qj = j0 + lr;
        float tnext[8], qnext[8];
        auto fetch = [&](int k0) {
#pragma unroll
            for (int t = 0; t < 8; ++t) tnext[t] = qnext[t] = 0.f;
            if (k0 + lk < d) {
                if (my_id >= 0) ld8f(E + (size_t)my_id * d + k0 + lk, tnext);
                if (qj < Q) ld8f(qn + (size_t)qj * d + k0 + lk, qnext);
            }
        };
        fetch(0);
        for (int k0 = 0; k0 < d; k0 += kKTile) {
#pragma unroll
            for (int t = 0; t < 8; ++t) {
                ts[lk + t][lr] = tnext[t];
                qs[lk + t][lr] = qnext[t];
                if (j0 == 0) nrm = fmaf(tnext[t], tnext[t], nrm);
            }
            __syncthreads();
            if (k0 + kKTile < d) fetch(k0 + kKTile);
#pragma unroll 8
            for (int k = 0; k < kKTile; ++k) {
                const float4 tv = *reinterpret_cast<const float4*>(&ts[k][ty * 4]);
                const float4 qv = *reinterpret_cast<const float4*>(&qs[k][tx * 4]);
                const float t4[4] = {tv.x, tv.y, tv.z, tv.w}, q4[4] = {qv.x, qv.y, qv.z, qv.w};
#pragma unroll
                for (int a = 0; a < 4; ++a)
#pragma unroll
                    for (int b = 0; b < 4; ++b) acc[a][b] = fmaf(t4[a], q4[b], acc[a][b]);
            }
            __syncthreads();
        }
        // row max over this query tile: the 16 threads of a row group (tx) share each row
#pragma unroll
        for (int a = 0; a < 4; ++a) {
            float m = -INFINITY;
#pragma unroll
            for (int b = 0; b < 4; ++b)
                if (j0 + tx * 4 + b < Q) m = fmaxf(m, acc[a][b]);
#pragma unroll
            for (int o = 8; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
            if (tx == 0) rowmax[ty * 4 + a] = fmaxf(rowmax[ty * 4 + a], m);
        }
        if (j0 == 0) {
            // the four threads of a token row hold its four 8-dim segments of every step
            nrm += __shfl_xor_sync(0xffffffffu, nrm, 1);
            nrm += __shfl_xor_sync(0xffffffffu, nrm, 2);
            if ((threadIdx.x & 3) == 0) rownorm[lr] = sqrtf(nrm);
        }
        __syncthreads();
    }
    if (threadIdx.x < kTokTile) {
        const int i = i0 + threadIdx.x;
        if (i < S) {
            const int id = rowid[threadIdx.x];
            const float nr = rownorm[threadIdx.x];
            bool in_q = false;
            for (int j = 0; j < Q && !in_q; ++j) in_q = qids[j] == id;
            // a token of the query meets its own embedding: cosine exactly 1
            // (the largest possible), so its score is exactly 1 + 0.25
            scores[i] = in_q ? 1.25f : (nr > 0.f ? rowmax[threadIdx.x] / nr : 0.f);
        }
    }
}

// ---- tensor-core scoring (bf16 embeddings).  An fp32 value splits exactly
// into three bf16 terms (8 significand bits each), and bf16 products are exact
// in fp32, so <E[s], hi + mid + lo> accumulated in fp32 is the fp32 dot product
// up to the order of the sums.

// one CTA per query token: q = E[q_j] / ||E[q_j]|| in fp32, written as the rows
// j (hi), Q + j (mid), 2Q + j (lo) of qp
__device__ void sur_qsplit(int j, const __nv_bfloat16* __restrict__ E, int vocab, int d,
                           const int32_t* __restrict__ qids, int Q, __nv_bfloat16* __restrict__ qp, int32_t* err) {
    __shared__ float red[256];
    const int id = qids[j];
    const bool ok = id >= 0 && id < vocab;
    if (!ok && threadIdx.x == 0) atomicOr(err, DEV_ERR_INDEX);
    const __nv_bfloat16* row = E + (size_t)(ok ? id : 0) * d;
    float ss = 0.f;
    for (int k = threadIdx.x; k < d; k += blockDim.x) {
        const float v = ok ? __bfloat162float(row[k]) : 0.f;
        ss = fmaf(v, v, ss);
    }
    red[threadIdx.x] = ss;
    __syncthreads();
    for (int w = 128; w > 0; w >>= 1) {
        if (threadIdx.x < w) red[threadIdx.x] += red[threadIdx.x + w];
        __syncthreads();
    }
    const float nrm = sqrtf(red[0]);
    const float inv = nrm > 0.f ? 1.0f / nrm : 0.f;
    for (int k = threadIdx.x; k < d; k += blockDim.x) {
        const float x = ok ? __bfloat162float(row[k]) * inv : 0.f;
        const __nv_bfloat16 hi = __float2bfloat16_rn(x);
        const float r1 = x - __bfloat162float(hi);
        const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
        const __nv_bfloat16 lo = __float2bfloat16_rn(r1 - __bfloat162float(mid));
        qp[(size_t)j * d + k] = hi;
        qp[(size_t)(Q + j) * d + k] = mid;
        qp[(size_t)(2 * Q + j) * d + k] = lo;
    }
}

// one warp per suffix token: its embedding row into eg (16-byte copies) and
// its fp32 norm, or -1 when the token occurs in the query; rows S..S_pad-1
// are zero
__device__ void sur_gather(int i, const __nv_bfloat16* __restrict__ E, int vocab, int d,
                           const int32_t* __restrict__ sids, int S, int S_pad, const int32_t* __restrict__ qids,
                           int Q, __nv_bfloat16* __restrict__ eg, float* __restrict__ enorm, int32_t* err) {
    const int lane = threadIdx.x & 31;
    if (i >= S_pad) return;
    uint4* dst = reinterpret_cast<uint4*>(eg + (size_t)i * d);
    const int nv = d / 8;
    int id = i < S ? sids[i] : -1;
    if (i < S && (id < 0 || id >= vocab)) {
        if (lane == 0) atomicOr(err, DEV_ERR_INDEX);
        id = -1;
    }
    float ss = 0.f;
    const uint4* src = reinterpret_cast<const uint4*>(E + (size_t)(id >= 0 ? id : 0) * d);
    for (int v = lane; v < nv; v += 32) {
        uint4 u = make_uint4(0, 0, 0, 0);
        if (id >= 0) u = src[v];
        dst[v] = u;
        const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            const float2 f = __bfloat1622float2(h[t]);
            ss = fmaf(f.x, f.x, ss);
            ss = fmaf(f.y, f.y, ss);
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if (i >= S) return;
    bool in_q = false;
    for (int j = lane; j < Q; j += 32) in_q |= qids[j] == sids[i];
    in_q = __any_sync(0xffffffffu, in_q);
    if (lane == 0) enorm[i] = in_q ? -1.0f : sqrtf(ss);
}

// the query split (CTAs 0 .. Q-1, one per query token) and the suffix rows'
// gather (the other CTAs, one warp per suffix token) in one launch
__global__ void __launch_bounds__(256) sur_prep_kernel(const __nv_bfloat16* __restrict__ E, int vocab, int d,
                                                       const int32_t* __restrict__ qids, int Q,
                                                       __nv_bfloat16* __restrict__ qp,
                                                       const int32_t* __restrict__ sids, int S, int S_pad,
                                                       __nv_bfloat16* __restrict__ eg, float* __restrict__ enorm,
                                                       int32_t* err) {
    pdl_trigger();   // the projection after it reads nothing before its wait
    if ((int)blockIdx.x < Q) {
        sur_qsplit(blockIdx.x, E, vocab, d, qids, Q, qp, err);
    } else {
        const int i = (int)(blockIdx.x - Q) * 8 + (threadIdx.x >> 5);
        sur_gather(i, E, vocab, d, sids, S, S_pad, qids, Q, eg, enorm, err);
    }
}

// scores from the GEMM partials: 128 suffix tokens per CTA; lane l of warp w
// takes tokens 4l..4l+3 (16-byte loads along the token axis) for the queries
// j = w, w + 32, ...; the warps' maxima meet in shared memory.  Per query the
// dot product sums (hi + mid) + lo per split, splits in order.
__global__ void __launch_bounds__(1024) sur_finish_kernel(const float* __restrict__ part, int splits, int S, int S_pad,
                                                          int Q, const float* __restrict__ enorm,
                                                          float* __restrict__ scores) {
    __shared__ float4 red[32][33];
    pdl_trigger();
    pdl_wait();
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int f0 = blockIdx.x * 128 + 4 * lane;
    const size_t split_stride = (size_t)3 * Q * S_pad;
    float4 best = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
    for (int j = w; j < Q; j += 32) {
        float4 dot = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int sp = 0; sp < splits; ++sp) {
            const float* p = part + sp * split_stride + f0;
            const float4 h = *reinterpret_cast<const float4*>(p + (size_t)j * S_pad);
            const float4 m = *reinterpret_cast<const float4*>(p + (size_t)(Q + j) * S_pad);
            const float4 l = *reinterpret_cast<const float4*>(p + (size_t)(2 * Q + j) * S_pad);
            dot.x += (h.x + m.x) + l.x;
            dot.y += (h.y + m.y) + l.y;
            dot.z += (h.z + m.z) + l.z;
            dot.w += (h.w + m.w) + l.w;
        }
        best.x = fmaxf(best.x, dot.x);
        best.y = fmaxf(best.y, dot.y);
        best.z = fmaxf(best.z, dot.z);
        best.w = fmaxf(best.w, dot.w);
    }
    red[w][lane] = best;
    __syncthreads();
    if (threadIdx.x < 128) {
        const int t = threadIdx.x, f = blockIdx.x * 128 + t;
        float bv = -INFINITY;
#pragma unroll 8
        for (int g = 0; g < 32; ++g) bv = fmaxf(bv, reinterpret_cast<const float*>(&red[g][t >> 2])[t & 3]);
        if (f < S) {
            const float nr = enorm[f];
            // a token of the query meets its own embedding: cosine exactly 1
            scores[f] = nr < 0.f ? 1.25f : (nr > 0.f ? bv / nr : 0.f);
        }
    }
}

// mean of the four largest scores of each unit (all of them below four)
// one warp: the unit score of unit u (returned in every lane).  Each lane
// keeps the four largest of its strided share in descending order; five
// butterfly steps merge the lanes' lists (the larger half of a bitonic
// sequence, then two compare-exchange stages), so every lane ends with the
// unit's four largest, summed largest first.
__device__ float unit_score_warp(const float* __restrict__ scores, const int32_t* __restrict__ bounds, int u,
                                 int32_t* err) {
    const int lane = threadIdx.x & 31;
    const int b = bounds[u], e = bounds[u + 1];
    if (b >= e) {
        if (lane == 0) atomicOr(err, DEV_ERR_INDEX);
        return -INFINITY;
    }
    float t[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
    for (int i = b + lane; i < e; i += 32) {
        float v = scores[i];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            if (v > t[k]) {
                const float x = t[k];
                t[k] = v;
                v = x;
            }
        }
    }
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        float p[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) p[k] = __shfl_xor_sync(0xffffffffu, t[k], o);
        // t descending, p descending: max(t_k, p_{3-k}) holds the four largest
        // of both as a bitonic sequence; sort it descending
        float c[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) c[k] = fmaxf(t[k], p[3 - k]);
        float x0 = fmaxf(c[0], c[2]), x2 = fminf(c[0], c[2]);
        float x1 = fmaxf(c[1], c[3]), x3 = fminf(c[1], c[3]);
        t[0] = fmaxf(x0, x1);
        t[1] = fminf(x0, x1);
        t[2] = fmaxf(x2, x3);
        t[3] = fminf(x2, x3);
    }
    const int n = min(4, e - b);
    float sum = t[0];
    for (int k = 1; k < n; ++k) sum += t[k];
    return sum / (float)n;
}

__global__ void sur_unit_kernel(const float* __restrict__ scores, const int32_t* __restrict__ bounds, int n_units,
                                float* __restrict__ unit_score, int32_t* err) {
    pdl_trigger();
    pdl_wait();
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
    if (warp >= n_units) return;
    const float v = unit_score_warp(scores, bounds, warp, err);
    if (lane == 0) unit_score[warp] = v;
}

// rank of unit u: units with a higher score, or the same score and an earlier start
__global__ void sur_rank_kernel(const float* __restrict__ unit_score, int n_units, int32_t* __restrict__ order) {
    __shared__ float sc[1024];
    pdl_trigger();
    pdl_wait();
    const int u = blockIdx.x * blockDim.x + threadIdx.x;
    const float mine = u < n_units ? unit_score[u] : 0.f;
    int rank = 0;
    for (int base = 0; base < n_units; base += 1024) {
        const int v = base + threadIdx.x;
        sc[threadIdx.x] = v < n_units ? unit_score[v] : 0.f;
        __syncthreads();
        const int lim = min(1024, n_units - base);
        if (u < n_units)
            for (int k = 0; k < lim; ++k) {
                const float x = sc[k];
                rank += (x > mine || (x == mine && base + k < u)) ? 1 : 0;
            }
        __syncthreads();
    }
    if (u < n_units) order[rank] = u;
}

__device__ int block_scan_incl(int v, int* total) {
    __shared__ int ws[32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += t;
    }
    if (lane == 31) ws[warp] = v;
    __syncthreads();
    if (warp == 0) {
        int w = ws[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int t = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += t;
        }
        ws[lane] = w;
    }
    __syncthreads();
    const int r = v + (warp > 0 ? ws[warp - 1] : 0);
    *total = ws[31];
    __syncthreads();
    return r;
}

// The selection mask and the envelope's prefix sums live in shared memory when
// they fit (kAdmitSelWords words, kAdmitCumLen doubles), else in the
// workspace; generic pointers keep one code path.  Every phase is then one
// block-wide step, with global round trips only for the unit order, the unit
// bounds and the partial unit's scores.
constexpr int kAdmitSelWords = 8192;
constexpr int kAdmitCumLen = 4096;
constexpr int kAdmitScores = 16384;   // token scores staged in shared memory (one coalesced pass)
constexpr size_t kAdmitSmem = kAdmitSelWords * sizeof(uint32_t) + kAdmitCumLen * sizeof(double) +
                              kAdmitScores * sizeof(float) + (kAdmitThreads + 1) * sizeof(int32_t);
// fused: n_units <= kAdmitThreads, so this block also computes the unit
// scores (one warp per unit) and their order (one thread per unit) itself,
// in shared memory, instead of reading `order` from the two kernels before it
__global__ void __launch_bounds__(kAdmitThreads) sur_admit_kernel(const float* __restrict__ scores_g,
                                                                  const int32_t* __restrict__ bounds_g, int n_units,
                                                                  const int32_t* __restrict__ order_in, int S, int B,
                                                                  int suffix_start, uint32_t* __restrict__ sel_ws,
                                                                  double* __restrict__ cum_ws,
                                                                  int32_t* __restrict__ positions, int fused,
                                                                  int32_t* err) {
    extern __shared__ __align__(16) uint8_t admit_smem[];
    __shared__ int s_partial, s_w;
    __shared__ float s_us[kAdmitThreads];
    __shared__ int s_order[kAdmitThreads];
    pdl_trigger();
    pdl_wait();
    // the token scores and the unit bounds, staged in one coalesced pass when they fit
    float* sc_smem = reinterpret_cast<float*>(admit_smem + kAdmitSelWords * sizeof(uint32_t) +
                                              kAdmitCumLen * sizeof(double));
    int32_t* bd_smem = reinterpret_cast<int32_t*>(sc_smem + kAdmitScores);
    const bool sc_fit = S <= kAdmitScores, bd_fit = n_units + 1 <= kAdmitThreads + 1;
    if (sc_fit)
        for (int i = threadIdx.x; i < S; i += blockDim.x) sc_smem[i] = scores_g[i];
    if (bd_fit)
        for (int i = threadIdx.x; i <= n_units; i += blockDim.x) bd_smem[i] = bounds_g[i];
    __syncthreads();
    const float* scores = sc_fit ? sc_smem : scores_g;
    const int32_t* bounds = bd_fit ? bd_smem : bounds_g;
    const int32_t* order = order_in;
    if (fused) {
        const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
        for (int u = warp; u < n_units; u += kAdmitThreads / 32) {
            const float v = unit_score_warp(scores, bounds, u, err);
            if (lane == 0) s_us[u] = v;
        }
        __syncthreads();
        // rank of unit u: units with a higher score, or the same score and an earlier start
        const int u = threadIdx.x;
        if (u < n_units) {
            const float mine = s_us[u];
            int rank = 0;
            for (int k = 0; k < n_units; ++k) {
                const float x = s_us[k];
                rank += (x > mine || (x == mine && k < u)) ? 1 : 0;
            }
            s_order[rank] = u;
        }
        __syncthreads();
        order = s_order;
    }
    const int W = (S + 31) / 32;
    uint32_t* sel = W <= kAdmitSelWords ? reinterpret_cast<uint32_t*>(admit_smem) : sel_ws;
    double* cum_smem = reinterpret_cast<double*>(admit_smem + kAdmitSelWords * sizeof(uint32_t));
    for (int w = threadIdx.x; w < W; w += blockDim.x) sel[w] = 0u;
    if (threadIdx.x == 0) {
        s_partial = -1;
        s_w = 0;
    }
    __syncthreads();
    // admission in rank order: unit of rank k is whole when its running end fits B
    int carry = 0;
    for (int base = 0; base < n_units; base += blockDim.x) {
        const int k = base + threadIdx.x;
        const int u = k < n_units ? order[k] : -1;
        const int len = u >= 0 ? bounds[u + 1] - bounds[u] : 0;
        int total;
        const int end = carry + block_scan_incl(len, &total);
        const int start = end - len;
        if (u >= 0 && start < B) {
            if (end <= B) {   // the whole unit: whole-word masks, at most ceil(len/32) + 1 atomics
                const int b0 = bounds[u], e0 = bounds[u + 1];
                for (int w = b0 >> 5; w <= (e0 - 1) >> 5; ++w) {
                    const int lo = max(b0 - 32 * w, 0), hi = min(e0 - 32 * w, 32);
                    const uint32_t mask = (hi >= 32 ? 0xffffffffu : ((1u << hi) - 1u)) & ~((1u << lo) - 1u);
                    atomicOr(&sel[w], mask);
                }
            } else {
                s_partial = u;   // the first unit that does not fit (unique: starts below B, ends above)
                s_w = B - start;
            }
        }
        carry += total;
        __syncthreads();
        if (carry >= B) break;
    }
    __syncthreads();
    // forward-envelope window of the partial unit (Eq. 8), in double.
    // Unrolling u_t = max(exp(rho_t), g u_{t-1}) with rho = r - r_max and
    // g = exp(-1/16) gives u_t = exp(max_{s<=t}(rho_s + s/16) - t/16): a block
    // prefix max, one exponential per token, then a prefix sum C, and the
    // window [a, a + w) sums to C[a + w - 1] - C[a - 1].  The largest sum wins,
    // the earliest start on ties.
    if (s_partial >= 0) {
        const int b = bounds[s_partial], e = bounds[s_partial + 1], w = s_w, len = e - b;
        double* cum = len <= kAdmitCumLen ? cum_smem : cum_ws;
        const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
        // The double-precision pipe of this part is narrow, so the work is
        // spread over the warps, in chunks of 32 tokens: r_max (a block max);
        // each chunk's prefix max of rho_s + s/16; the chunks' carries (a
        // prefix max over the chunk maxima, on one warp); u_t =
        // exp(pm_t - t/16) per token; each chunk's prefix sum of u; the sums'
        // carries, added chunk after chunk by one thread, so every C_t is
        // (chunk prefix) + (sum of the earlier chunks' totals, first to last)
        // and does not depend on how the chunks were spread.
        const int nch = (len + 31) / 32, nw = blockDim.x >> 5;
        __shared__ float s_cred[32];
        __shared__ double s_carry[kAdmitCumLen / 32 + 1];
        double* chunk = len <= kAdmitCumLen ? s_carry : cum_ws + len;   // per-chunk values
        // r_max on the float pipe: a max of floats is exact, so widening it
        // afterwards gives the same double as a max of widened scores.  Only
        // warps with tokens in hand run double-precision work below.
        float rm = -INFINITY;
        for (int t = threadIdx.x; t < len; t += blockDim.x) rm = fmaxf(rm, scores[b + t]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) rm = fmaxf(rm, __shfl_xor_sync(0xffffffffu, rm, o));
        if (lane == 0) s_cred[wid] = rm;
        __syncthreads();
        float rmf = s_cred[0];
        for (int k = 1; k < nw; ++k) rmf = fmaxf(rmf, s_cred[k]);
        const double rmax = (double)rmf;
        for (int c = wid; c < nch; c += nw) {   // chunk prefix max of rho_s + s/16
            const int t = 32 * c + lane;
            double pm = t < len ? ((double)scores[b + t] - rmax) + (double)t * 0.0625 : -INFINITY;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const double y = __shfl_up_sync(0xffffffffu, pm, o);
                if (lane >= o) pm = fmax(pm, y);
            }
            if (t < len) cum[t] = pm;
            if (lane == 31) chunk[c] = pm;
        }
        __syncthreads();
        if (wid == 0) {   // exclusive prefix max of the chunk maxima (max is exact in any order)
            double carry = -INFINITY;
            for (int c0 = 0; c0 < nch; c0 += 32) {
                const int c = c0 + lane;
                double v = c < nch ? chunk[c] : -INFINITY;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const double y = __shfl_up_sync(0xffffffffu, v, o);
                    if (lane >= o) v = fmax(v, y);
                }
                const double prev = __shfl_up_sync(0xffffffffu, v, 1);
                const double excl = lane == 0 ? carry : fmax(carry, prev);
                carry = fmax(carry, __shfl_sync(0xffffffffu, v, 31));
                __syncwarp();
                if (c < nch) chunk[c] = excl;
            }
        }
        __syncthreads();
        for (int t = threadIdx.x; t < len; t += blockDim.x) {   // u_t = exp(max_{s<=t}(rho_s + s/16) - t/16)
            const double pm = fmax(chunk[t >> 5], cum[t]);
            cum[t] = exp(pm - (double)t * 0.0625);
        }
        __syncthreads();
        for (int c = wid; c < nch; c += nw) {   // chunk prefix sums of u
            const int t = 32 * c + lane;
            double v = t < len ? cum[t] : 0.0;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const double y = __shfl_up_sync(0xffffffffu, v, o);
                if (lane >= o) v += y;
            }
            if (t < len) cum[t] = v;
            if (lane == 31) chunk[c] = v;   // the chunk's total
        }
        __syncthreads();
        if (threadIdx.x == 0) {   // carries: the earlier chunks' totals, added first to last
            double carry = 0.0;
            for (int c = 0; c < nch; ++c) {
                const double total = chunk[c];
                chunk[c] = carry;
                carry = total + carry;
            }
        }
        __syncthreads();
        for (int t = threadIdx.x; t < len; t += blockDim.x) cum[t] = cum[t] + chunk[t >> 5];
        __syncthreads();
        // best window start, on one warp: each window sum is mapped to a
        // 64-bit key that orders as the double does (sign-magnitude to
        // two's-complement order), so the comparisons stay on the integer
        // pipe; the earliest start wins a tie
        __shared__ int s_ba;
        if (wid == 0) {
            unsigned long long best = 0ull;
            int best_a = INT_MAX;
            for (int a0 = lane; a0 + w <= len; a0 += 32) {
                const double sum = cum[a0 + w - 1] - (a0 > 0 ? cum[a0 - 1] : 0.0);
                const unsigned long long bits = (unsigned long long)__double_as_longlong(sum);
                const unsigned long long key = (bits >> 63) ? ~bits : (bits | 0x8000000000000000ull);
                if (best_a == INT_MAX || key > best) {   // a0 ascends per lane: the first maximiser stays
                    best = key;
                    best_a = a0;
                }
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const unsigned long long ob = __shfl_xor_sync(0xffffffffu, best, o);
                const int oa = __shfl_xor_sync(0xffffffffu, best_a, o);
                if (ob > best || (ob == best && oa < best_a)) {
                    best = ob;
                    best_a = oa;
                }
            }
            if (lane == 0) s_ba = best_a;
        }
        __syncthreads();
        // the window's bits, set in parallel (the whole units' bits are in other words
        // or other bits of these words, so the ORs commute)
        for (int t = threadIdx.x; t < w; t += blockDim.x) {
            const int i = b + s_ba + t;
            atomicOr(&sel[i >> 5], 1u << (i & 31));
        }
    }
    __syncthreads();
    // compaction: ascending positions from the bit mask.  The words' prefix
    // counts first (in the envelope's space, free by now), then one bit per
    // thread: a set bit's rank is its word's prefix plus the set bits below it
    int* wpre = W <= 2 * kAdmitCumLen ? reinterpret_cast<int*>(cum_smem) : reinterpret_cast<int*>(cum_ws);
    int pcarry = 0;
    for (int base = 0; base < W; base += blockDim.x) {
        const int w = base + threadIdx.x;
        const uint32_t word = w < W ? sel[w] : 0u;
        int total;
        const int incl = block_scan_incl(__popc(word), &total);
        if (w < W) wpre[w] = pcarry + incl - __popc(word);
        pcarry += total;
    }
    __syncthreads();
    for (int i = threadIdx.x; i < W * 32; i += blockDim.x) {
        const uint32_t word = sel[i >> 5];
        if ((word >> (i & 31)) & 1u) {
            const int k = wpre[i >> 5] + __popc(word & ((1u << (i & 31)) - 1u));
            if (k < B) positions[k] = suffix_start + i;
        }
    }
}

}  // namespace

size_t sur_ws_layout(int S, int Q, int d, int n_units, bool tc, SurWs* L, uint8_t* base) {
    auto al = [](size_t x) { return (x + 255) & ~size_t(255); };
    size_t off = 0;
    const size_t o_err = off;
    off += al(16);
    const size_t o_qn = off;
    off += al((size_t)Q * d * sizeof(float));
    const size_t o_sc = off;
    off += al((size_t)S * sizeof(float));
    const size_t o_us = off;
    off += al((size_t)n_units * sizeof(float));
    const size_t o_or = off;
    off += al((size_t)n_units * sizeof(int32_t));
    const size_t o_sel = off;
    off += al((size_t)((S + 31) / 32) * sizeof(uint32_t));
    const size_t o_cum = off;   // the envelope's prefix sums and one value per 32-token chunk; then the mask words' prefix counts
    off += al((size_t)(S + (S + 31) / 32 + 1) * sizeof(double));
    size_t o_eg = 0, o_qp = 0, o_en = 0, o_part = 0;
    if (tc) {
        const int S_pad = (S + 127) / 128 * 128;
        const GemmPlan gp = plan_gemm(KVR_BF16, S_pad, d, 3 * Q);
        o_eg = off;
        off += al((size_t)S_pad * d * 2);
        o_qp = off;
        off += al((size_t)3 * Q * d * 2);
        o_en = off;
        off += al((size_t)S * sizeof(float));
        o_part = off;
        off += al(gemm_partial_bytes(gp));
    }
    if (L && base) {
        L->err = (int32_t*)(base + o_err);
        L->qn = (float*)(base + o_qn);
        L->scores = (float*)(base + o_sc);
        L->unit_score = (float*)(base + o_us);
        L->order = (int32_t*)(base + o_or);
        L->sel = (uint32_t*)(base + o_sel);
        L->cum = (double*)(base + o_cum);
        L->eg = tc ? (__nv_bfloat16*)(base + o_eg) : nullptr;
        L->qp = tc ? (__nv_bfloat16*)(base + o_qp) : nullptr;
        L->enorm = tc ? (float*)(base + o_en) : nullptr;
        L->part = tc ? (float*)(base + o_part) : nullptr;
    }
    return off;
}

}  // namespace kvr

using namespace kvr;

#define KVR_CHECK_LAUNCH_SUR(expr)                              \
    do {                                                        \
        cudaError_t e_ = (expr);                                \
        if (e_ != cudaSuccess) return cuda_fail(e_, "sur launch"); \
    } while (0)

extern "C" {

size_t kvr_sur_workspace_bytes(int32_t S, int32_t Q, int32_t d, int32_t n_units) {
    if (S < 1 || Q < 1 || d < 1 || n_units < 1) return 0;
    return sur_ws_layout(S, Q, d, n_units, d % 64 == 0, nullptr, nullptr);
}

kvr_status kvr_sur_select(const void* embed, int32_t vocab, int32_t d, int32_t dtype, const int32_t* suffix_ids,
                          int32_t S, int32_t suffix_start, const int32_t* query_ids, int32_t Q,
                          const int32_t* unit_bounds, int32_t n_units, int32_t budget_percent, void* workspace,
                          size_t ws_bytes, int32_t* positions_out, int32_t* n_out, float* scores_out,
                          void* stream) {
    if (!embed || !suffix_ids || !query_ids || !unit_bounds || !workspace || !positions_out || !n_out) {
        set_error("sur: NULL argument");
        return KVR_EINVAL;
    }
    if (vocab < 1 || d < 8 || d % 8 || S < 1 || Q < 1 || n_units < 1 || suffix_start < 0 || budget_percent < 0 ||
        budget_percent > 100 || (dtype != KVR_F32 && dtype != KVR_BF16)) {
        set_error("sur: need vocab, S, Q, n_units >= 1, d a multiple of 8, suffix_start >= 0, budget in [0, 100], "
                  "dtype F32/BF16");
        return KVR_EINVAL;
    }
    if (n_units > 65536 || n_units > S) {
        set_error("sur: n_units must be <= min(S, 65536)");
        return KVR_ERANGE;
    }
    if (reinterpret_cast<uintptr_t>(workspace) & 255u) {
        set_error("sur: workspace must be 256-byte aligned");
        return KVR_EINVAL;
    }
    SurWs L;
    const bool tc = dtype == KVR_BF16 && d % 64 == 0;   // the scoring contraction on the tensor cores
    const size_t need = sur_ws_layout(S, Q, d, n_units, tc, &L, (uint8_t*)workspace);
    if (ws_bytes < need) {
        set_error("sur: workspace too small: need " + std::to_string(need) + " bytes");
        return KVR_EINVAL;
    }
    const int B = (int)std::min<int64_t>(S, ((int64_t)S * budget_percent + 99) / 100);   // Eq. 3
    *n_out = B;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    float* scores = scores_out ? scores_out : L.scores;
    cudaError_t e = cudaMemsetAsync(L.err, 0, 16, s);
    if (e != cudaSuccess) return cuda_fail(e, "sur");
    pdl_begin_call();   // the first kernel keeps plain stream order
    if (tc) {
        const int S_pad = (S + 127) / 128 * 128;
        KVR_CHECK_LAUNCH_SUR(launch_kernel(sur_prep_kernel, dim3((unsigned)(Q + (S_pad + 7) / 8)), dim3(256), 0, s,
                                           (const __nv_bfloat16*)embed, vocab, d, query_ids, Q, L.qp, suffix_ids, S,
                                           S_pad, L.eg, L.enorm, L.err));
        // the projection's first operand is the rows just gathered, so it
        // loads them only after its wait for the prep kernel
        const GemmPlan gp = plan_gemm(KVR_BF16, S_pad, d, 3 * Q);
        std::string why;
        e = launch_gemm(KVR_BF16, gp, L.eg, L.qp, L.part, L.err, s, &why, nullptr, true);
        if (e != cudaSuccess) return cuda_fail(e, ("sur scoring " + why).c_str());
        KVR_CHECK_LAUNCH_SUR(launch_kernel(sur_finish_kernel, dim3((unsigned)(S_pad / 128)), dim3(1024), 0, s,
                                           (const float*)L.part, gp.splits, S, S_pad, Q, (const float*)L.enorm,
                                           scores));
    } else if (dtype == KVR_BF16) {
        sur_qnorm_kernel<__nv_bfloat16><<<Q, 256, 0, s>>>((const __nv_bfloat16*)embed, vocab, d, query_ids, L.qn,
                                                          L.err);
        sur_score_kernel<__nv_bfloat16><<<(S + kTokTile - 1) / kTokTile, 256, 0, s>>>(
            (const __nv_bfloat16*)embed, vocab, d, suffix_ids, S, query_ids, Q, L.qn, scores, L.err);
    } else {
        sur_qnorm_kernel<float><<<Q, 256, 0, s>>>((const float*)embed, vocab, d, query_ids, L.qn, L.err);
        sur_score_kernel<float><<<(S + kTokTile - 1) / kTokTile, 256, 0, s>>>(
            (const float*)embed, vocab, d, suffix_ids, S, query_ids, Q, L.qn, scores, L.err);
    }
    // the FFMA scoring kernels above are plain launches, so the next kernel's
    // dependent launch waits for them like any other predecessor.  Up to
    // kAdmitThreads units, the admission kernel scores and orders the units
    // itself.
    const bool fused = n_units <= kAdmitThreads;
    if (!fused) {
        KVR_CHECK_LAUNCH_SUR(launch_kernel(sur_unit_kernel, dim3((unsigned)((n_units * 32 + 255) / 256)), dim3(256),
                                           0, s, (const float*)scores, unit_bounds, n_units, L.unit_score, L.err));
        KVR_CHECK_LAUNCH_SUR(launch_kernel(sur_rank_kernel, dim3((unsigned)((n_units + 1023) / 1024)), dim3(1024), 0,
                                           s, (const float*)L.unit_score, n_units, L.order));
    }
    if (B > 0 || fused) {   // fused, it also checks the units, whatever the budget
        static bool admit_attr = false;
        if (!admit_attr) {
            KVR_CHECK_LAUNCH_SUR(
                cudaFuncSetAttribute(sur_admit_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kAdmitSmem));
            admit_attr = true;
        }
        KVR_CHECK_LAUNCH_SUR(launch_kernel(sur_admit_kernel, dim3(1), dim3(kAdmitThreads), kAdmitSmem, s,
                                           (const float*)scores, unit_bounds, n_units, (const int32_t*)L.order, S, B,
                                           suffix_start, L.sel, L.cum, positions_out, fused ? 1 : 0, L.err));
    }
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "sur launch");
    return KVR_OK;
}

kvr_status kvr_sur_status(void* workspace, void* stream) {
    if (!workspace) {
        set_error("sur status: NULL workspace");
        return KVR_EINVAL;
    }
    int32_t h[4] = {0, 0, 0, 0};
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemcpyAsync(h, workspace, 16, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e == cudaSuccess) e = cudaMemsetAsync(workspace, 0, 16, s);
    if (e != cudaSuccess) return cuda_fail(e, "sur status");
    if (h[0]) {
        set_error("sur: an id outside the vocabulary or an empty unit");
        return KVR_EDEVICE;
    }
    return KVR_OK;
}

}  // extern "C"

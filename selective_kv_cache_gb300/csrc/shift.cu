// shift.cu -- move K/V rows to new positions, re-rotating the keys.
//
// Shift ("Budgeted KV-Cache Repair for Evolving Contexts", Sec. 7.1, Eq. 2):
// deleting [start, start + d) moves every later row down by d.  Keys are
// stored after the rotary map, and rotations compose, so the key that moves
// from position i to i - d becomes R_{i-d} R_i^{-1} k = R_{-d} k: the same
// rotation for every moved row.  Splice ("Models Take Notes at Prefill: KV
// Cache Can Be Editable and Composable", Sec. 5): a block computed on its own
// at positions src.. lands at dst.., keys rotated by dst - src; values carry
// no position in either case.
//
// One pass, HBM-bound: each moved row is read once and written once, in
// 16-byte vectors, one warp covering 4 rows (bf16, head_dim 128).  Each
// thread owns the vector pair (v, v + half) of a row, so the rotate-half
// partner of every element is in the same thread.  The rotation angle does
// not depend on the row, so the (cos, sin) table travels in the launch
// parameters.
//
// In place (Shift), one CTA sweeps one (sequence, layer, head) slab upwards
// in tiles of rows: it reads a whole tile into registers, synchronises, then
// writes it.  A tile writes rows below everything later tiles read (the
// source lies d rows above the destination), and within a tile the barrier
// orders every read before any write, so no row is overwritten before it is
// read.
#include <cuda_bf16.h>

#include "kvr_internal.h"

namespace kvr {
namespace {

constexpr int kMoveThreads = 256;
constexpr int kMoveTileRows = 128;

__device__ __forceinline__ void rotate_pair(uint4& lo, uint4& hi, const float* c, const float* s, __nv_bfloat16) {
    uint32_t* a = reinterpret_cast<uint32_t*>(&lo);
    uint32_t* b = reinterpret_cast<uint32_t*>(&hi);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&a[i]));
        const float2 y = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&b[i]));
        const float c0 = c[2 * i], c1 = c[2 * i + 1], s0 = s[2 * i], s1 = s[2 * i + 1];
        const __nv_bfloat162 o1 = __floats2bfloat162_rn(x.x * c0 - y.x * s0, x.y * c1 - y.y * s1);
        const __nv_bfloat162 o2 = __floats2bfloat162_rn(y.x * c0 + x.x * s0, y.y * c1 + x.y * s1);
        a[i] = *reinterpret_cast<const uint32_t*>(&o1);
        b[i] = *reinterpret_cast<const uint32_t*>(&o2);
    }
}

__device__ __forceinline__ void rotate_pair(uint4& lo, uint4& hi, const float* c, const float* s, float) {
    float* x = reinterpret_cast<float*>(&lo);
    float* y = reinterpret_cast<float*>(&hi);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float a = x[i], b = y[i];
        x[i] = a * c[i] - b * s[i];
        y[i] = b * c[i] + a * s[i];
    }
}

// VR: 16-byte vectors per row (head_dim * sizeof(T) / 16).
template <typename T, int VR>
__global__ void __launch_bounds__(kMoveThreads) move_rows_kernel(MoveLaunch a) {
    constexpr int kHalf = VR / 2;                      // threads per row
    constexpr int kRowsPerPass = kMoveThreads / kHalf;
    constexpr int kPasses = kMoveTileRows / kRowsPerPass;
    constexpr int E = 16 / (int)sizeof(T);             // elements per vector
    const bool is_key = blockIdx.z == 0;
    const size_t slab = blockIdx.x;
    const uint4* src = reinterpret_cast<const uint4*>(is_key ? a.k_src : a.v_src) + slab * a.src_slab_rows * VR;
    uint4* dst = reinterpret_cast<uint4*>(is_key ? a.k_dst : a.v_dst) + (slab + a.dst_slab_off) * a.dst_slab_rows * VR;
    const int v = threadIdx.x % kHalf, rin = threadIdx.x / kHalf;
    float c[E], s[E];
#pragma unroll
    for (int e = 0; e < E; ++e) {
        const float2 t = a.cs[v * E + e];
        c[e] = t.x;
        s[e] = t.y;
    }
    const int r_begin = blockIdx.y * a.chunk;
    const int r_end = min(a.n_rows, r_begin + a.chunk);
    for (int t0 = r_begin; t0 < r_end; t0 += kMoveTileRows) {
        uint4 lo[kPasses], hi[kPasses];
#pragma unroll
        for (int p = 0; p < kPasses; ++p) {
            const int r = t0 + p * kRowsPerPass + rin;
            if (r < r_end) {
                const uint4* row = src + (size_t)(a.src_row0 + r) * VR;
                lo[p] = row[v];
                hi[p] = row[v + kHalf];
            }
        }
        __syncthreads();   // every read of this tile before any write of it
#pragma unroll
        for (int p = 0; p < kPasses; ++p) {
            const int r = t0 + p * kRowsPerPass + rin;
            if (r < r_end) {
                if (is_key) rotate_pair(lo[p], hi[p], c, s, T{});
                uint4* row = dst + (size_t)(a.dst_row0 + r) * VR;
                row[v] = lo[p];
                row[v + kHalf] = hi[p];
            }
        }
    }
}

__device__ __forceinline__ uint32_t bits_below(int k) {
    return k <= 0 ? 0u : (k >= 32 ? 0xffffffffu : ((1u << k) - 1u));
}

// Local/sink words of one sequence after deleting [start, start + d): bits
// below start stay, bit p >= start takes old bit p + d, bits at or past
// n_old - d clear.  Word w reads words >= w only; same tile discipline as
// the row move.
__global__ void shift_bits_kernel(uint32_t* bits0, uint32_t* bits1, int W, int start, int d, int n_old) {
    uint32_t* b = (blockIdx.y ? bits1 : bits0) + (size_t)blockIdx.x * W;
    const int n_new = n_old - d;
    const int w_end = (n_old + 31) >> 5;
    for (int w0 = start >> 5; w0 < w_end; w0 += blockDim.x) {
        const int w = w0 + threadIdx.x;
        uint32_t out = 0u;
        if (w < w_end) {
            const int p0 = w * 32;
            const int q = p0 + d;
            const int qw = q >> 5;
            const uint32_t lo = qw < W ? b[qw] : 0u;
            const uint32_t hi = qw + 1 < W ? b[qw + 1] : 0u;
            const uint32_t moved = __funnelshift_r(lo, hi, q & 31);
            const uint32_t keep = bits_below(start - p0);
            out = (b[w] & keep) | (moved & ~keep & bits_below(n_new - p0));
        }
        __syncthreads();
        if (w < w_end) b[w] = out;
    }
}

__global__ void set_bits_kernel(uint32_t* local, uint32_t* sink, int dst, int n, uint32_t flags) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    const int p = dst + i;
    const uint32_t bit = 1u << (p & 31);
    if (flags & KVR_SPLICE_LOCAL) atomicOr(&local[p >> 5], bit);
    if ((flags & KVR_SPLICE_SINK) && i < 4) atomicOr(&sink[p >> 5], bit);
}

template <typename T, int VR>
cudaError_t launch_move_t(const MoveLaunch& a, int chunks, cudaStream_t s) {
    dim3 grid((unsigned)a.n_slabs, (unsigned)chunks, 2);
    move_rows_kernel<T, VR><<<grid, kMoveThreads, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_move_rows(int dtype, int head_dim, const MoveLaunch& a_in, bool in_place, cudaStream_t s) {
    if (a_in.n_rows <= 0 || a_in.n_slabs <= 0) return cudaSuccess;
    if (in_place && a_in.dst_row0 > a_in.src_row0) return cudaErrorInvalidValue;   // the sweep only moves down
    MoveLaunch a = a_in;
    // in place: one CTA per slab sweeps all rows; otherwise rows split freely
    a.chunk = in_place ? a.n_rows : 4 * kMoveTileRows;
    const int chunks = (a.n_rows + a.chunk - 1) / a.chunk;
    if (dtype == KVR_BF16 && head_dim == 128) return launch_move_t<__nv_bfloat16, 16>(a, chunks, s);
    if (dtype == KVR_F32 && head_dim == 64) return launch_move_t<float, 16>(a, chunks, s);
    if (dtype == KVR_F32 && head_dim == 128) return launch_move_t<float, 32>(a, chunks, s);
    return cudaErrorInvalidValue;
}

cudaError_t launch_shift_bits(uint32_t* local, uint32_t* sink, int batch, int words, int start, int d, int n_old,
                              cudaStream_t s) {
    shift_bits_kernel<<<dim3((unsigned)batch, 2), 256, 0, s>>>(local, sink, words, start, d, n_old);
    return cudaGetLastError();
}

cudaError_t launch_set_bits(uint32_t* local, uint32_t* sink, int dst, int n, uint32_t flags, cudaStream_t s) {
    if (n <= 0 || !(flags & (KVR_SPLICE_LOCAL | KVR_SPLICE_SINK))) return cudaSuccess;
    set_bits_kernel<<<(n + 255) / 256, 256, 0, s>>>(local, sink, dst, n, flags);
    return cudaGetLastError();
}

}  // namespace kvr

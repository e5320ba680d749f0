// select.cu -- selection pack: sorted position list, intervals, bit masks,
// per-query-tile plan, row gather, and the metadata commit.
//
// "Budgeted KV-Cache Repair for Evolving Contexts": Sec. 3.2 / Algorithm 1
// (sort the selected positions, coalesce adjacent ones into intervals),
// Sec. 13.2 (gather the selected rows once into a compact hidden buffer;
// Eqs. 23-24 per-query-tile complete-prefix and total K/V tile counts).
// "kv-cross-attention-reuse", Sec. 6.4 (correction masks M_local, M_sink;
// physical repair sets type_t <- global).
//
// One CTA per sequence builds that sequence's structures from its bit mask,
// so the sorted order comes from the mask itself (no comparison sort).
#include <cuda_bf16.h>

#include "kvr_internal.h"
#include "ptx.cuh"

namespace kvr {
namespace {

constexpr int kSelThreads = 1024;

// Block-wide inclusive scan of one int per thread; returns the inclusive
// value, *total gets the block sum.  Needs blockDim.x == kSelThreads.
__device__ int block_incl_scan(int v, int* total) {
    __shared__ int warp_sums[32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int t = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += t;
    }
    if (lane == 31) warp_sums[warp] = v;
    __syncthreads();
    if (warp == 0) {
        int w = warp_sums[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int t = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += t;
        }
        warp_sums[lane] = w;
    }
    __syncthreads();
    int r = v + (warp > 0 ? warp_sums[warp - 1] : 0);
    *total = warp_sums[31];
    __syncthreads();
    return r;
}

__global__ void __launch_bounds__(kSelThreads) select_kernel(SelectLaunch a) {
    const int seq = blockIdx.x;
    const int* info = a.seqinfo + seq * 8;
    const int count = info[0], row_off = info[1], iv_off = info[2], tile_off = info[3], n_tiles = info[4];
    const int raw_off = info[5];
    const int W = a.words;
    uint32_t* sel = a.sel + (size_t)seq * W;
    const uint32_t* local = a.local + (size_t)seq * W;
    const uint32_t* sink = a.sink + (size_t)seq * W;
    uint32_t* eloc = a.eloc + (size_t)seq * W;
    uint32_t* esnk = a.esnk + (size_t)seq * W;

    for (int w = threadIdx.x; w < W; w += blockDim.x) sel[w] = 0u;
    __syncthreads();
    for (int i = threadIdx.x; i < count; i += blockDim.x) {
        const int p = a.raw[raw_off + i];
        if (p < a.suffix_start || p >= a.n_tokens) {
            atomicOr(a.err, DEV_ERR_INDEX);
            continue;
        }
        const uint32_t bit = 1u << (p & 31);
        const uint32_t old = atomicOr(&sel[p >> 5], bit);
        if (old & bit) atomicOr(a.err, DEV_ERR_DUPLICATE);
    }
    __syncthreads();

    // compaction: ascending positions from the mask (word order, then bit order)
    int carry = 0;
    for (int base = 0; base < W; base += blockDim.x) {
        const int w = base + threadIdx.x;
        uint32_t word = (w < W) ? sel[w] : 0u;
        int total;
        const int incl = block_incl_scan(__popc(word), &total);
        int k = carry + incl - __popc(word);
        while (word) {
            const int b = __ffs(word) - 1;
            if (k < count) {
                a.U[row_off + k] = w * 32 + b;
                a.row_seq[row_off + k] = seq;
            }
            ++k;
            word &= word - 1u;
        }
        if (w < W) {
            const uint32_t s = sel[w];
            eloc[w] = local[w] & ~s;
            esnk[w] = a.sink_static ? sink[w] : (sink[w] & ~s);
        }
        carry += total;
    }
    __syncthreads();   // U of this sequence complete and visible to the block

    // intervals: a row starts one when its position does not follow the previous row's
    const int* U = a.U + row_off;
    int icarry = 0;
    for (int base = 0; base < count; base += blockDim.x) {
        const int i = base + threadIdx.x;
        int start = 0, end = 0, u = 0;
        if (i < count) {
            u = U[i];
            start = (i == 0) || (U[i - 1] + 1 != u);
            end = (i == count - 1) || (U[i + 1] != u + 1);
        }
        int total;
        const int idx = icarry + block_incl_scan(start, &total) - 1;
        if (i < count) {
            if (start) a.iv[2 * (iv_off + idx)] = u;
            if (end) a.iv[2 * (iv_off + idx) + 1] = u + 1;
        }
        icarry += total;
    }

    // plan over query tiles of rows_per_tile consecutive rows (Eqs. 23-24)
    for (int t = threadIdx.x; t < n_tiles; t += blockDim.x) {
        const int r0 = t * a.rows_per_tile;
        const int r1 = min(count, r0 + a.rows_per_tile);
        const int umin = U[r0], umax = U[r1 - 1];
        int* p = a.plan + 8 * (tile_off + t);
        p[0] = row_off + r0;
        p[1] = r1 - r0;
        p[2] = umin;
        p[3] = umax;
        p[4] = (umin + 1) / a.keys_per_tile;
        p[5] = (umax + 1 + a.keys_per_tile - 1) / a.keys_per_tile;
        p[6] = seq;
        p[7] = 0;
    }
}

template <typename T>
__global__ void gather_kernel(const int32_t* __restrict__ U, const int32_t* __restrict__ row_seq, int n_rows, int d,
                              int capacity, const int32_t* __restrict__ ids, const T* __restrict__ embed,
                              const T* __restrict__ src, T* __restrict__ out, int32_t* err, int vocab) {
    const int r = blockIdx.x;
    if (r >= n_rows) return;
    const int seq = row_seq[r];
    const size_t pos = (size_t)seq * capacity + U[r];
    const T* row;
    if (ids) {
        const int id = ids[pos];
        if (id < 0 || id >= vocab) {
            if (threadIdx.x == 0) atomicOr(err, DEV_ERR_INDEX);
            return;
        }
        row = embed + (size_t)id * d;
    } else {
        row = src + pos * d;
    }
    const int nvec = d * (int)sizeof(T) / 16;
    const uint4* s4 = reinterpret_cast<const uint4*>(row);
    uint4* o4 = reinterpret_cast<uint4*>(out + (size_t)r * d);
    for (int i = threadIdx.x; i < nvec; i += blockDim.x) o4[i] = s4[i];
}

// position -> row map of the current selection (rows of one sequence are
// contiguous); entries of unselected positions stay -1
__global__ void map_rows_kernel(const int32_t* __restrict__ U, const int32_t* __restrict__ row_seq, int n_rows,
                                int capacity, int32_t* __restrict__ map) {
    const int r = blockIdx.x * blockDim.x + threadIdx.x;
    if (r < n_rows) map[(size_t)row_seq[r] * capacity + U[r]] = r;
}

// rows of a new selection: a position that was selected before keeps its
// current row (carry), any other takes its per-position row (fill)
template <typename T>
__global__ void gather_carry_kernel(const int32_t* __restrict__ U, const int32_t* __restrict__ row_seq, int n_rows,
                                    int d, int capacity, const int32_t* __restrict__ map, const T* __restrict__ carry,
                                    const T* __restrict__ fill, T* __restrict__ out) {
    const int r = blockIdx.x;
    if (r >= n_rows) return;
    const size_t pos = (size_t)row_seq[r] * capacity + U[r];
    const int old = map[pos];
    const T* row = old >= 0 ? carry + (size_t)old * d : fill + pos * d;
    const int nvec = d * (int)sizeof(T) / 16;
    const uint4* s4 = reinterpret_cast<const uint4*>(row);
    uint4* o4 = reinterpret_cast<uint4*>(out + (size_t)r * d);
    for (int i = threadIdx.x; i < nvec; i += blockDim.x) o4[i] = s4[i];
}

__global__ void commit_kernel(uint32_t* local, uint32_t* sink, const uint32_t* sel, int n, int sink_static) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    const uint32_t s = sel[i];
    local[i] &= ~s;
    if (!sink_static) sink[i] &= ~s;
}

// The bounded wait of the library's pipelines, exercised alone: one thread
// waits on phase 0 of a fresh barrier that nothing arrives on, with the
// budget given, and records the timeout when the budget runs out.  No copy
// or product targets this block's memory, so returning is always safe.
__global__ void wait_check_kernel(int32_t* err, long long cycles) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
        if (!mbar_wait(&bar, 0u, cycles)) atomicOr(err, DEV_ERR_TIMEOUT);
    }
}

}  // namespace

cudaError_t launch_wait_check(int32_t* err, long long cycles, cudaStream_t s) {
    KVR_LAUNCH(wait_check_kernel, dim3(1), dim3(32), 0, s, err, cycles);
    return cudaSuccess;
}

cudaError_t launch_select(const SelectLaunch& a, int batch, cudaStream_t s) {
    select_kernel<<<batch, kSelThreads, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_gather(int dtype, const int32_t* U, const int32_t* row_seq, int n_rows, int d, int capacity,
                          const int32_t* token_ids, const void* embed, const void* hidden_src, void* out,
                          int32_t* err, int vocab, cudaStream_t s) {
    if (n_rows <= 0) return cudaSuccess;
    if (dtype == KVR_BF16)
        gather_kernel<__nv_bfloat16><<<n_rows, 128, 0, s>>>(
            U, row_seq, n_rows, d, capacity, token_ids, (const __nv_bfloat16*)embed,
            (const __nv_bfloat16*)hidden_src, (__nv_bfloat16*)out, err, vocab);
    else
        gather_kernel<float><<<n_rows, 128, 0, s>>>(U, row_seq, n_rows, d, capacity, token_ids,
                                                    (const float*)embed, (const float*)hidden_src, (float*)out,
                                                    err, vocab);
    return cudaGetLastError();
}

cudaError_t launch_map_rows(const int32_t* U, const int32_t* row_seq, int n_rows, int capacity, int32_t* map,
                            cudaStream_t s) {
    if (n_rows <= 0) return cudaSuccess;
    map_rows_kernel<<<(n_rows + 255) / 256, 256, 0, s>>>(U, row_seq, n_rows, capacity, map);
    return cudaGetLastError();
}

cudaError_t launch_gather_carry(int dtype, const int32_t* U, const int32_t* row_seq, int n_rows, int d, int capacity,
                                const int32_t* map, const void* carry, const void* fill, void* out, cudaStream_t s) {
    if (n_rows <= 0) return cudaSuccess;
    if (dtype == KVR_BF16)
        gather_carry_kernel<__nv_bfloat16><<<n_rows, 128, 0, s>>>(U, row_seq, n_rows, d, capacity, map,
                                                                  (const __nv_bfloat16*)carry,
                                                                  (const __nv_bfloat16*)fill, (__nv_bfloat16*)out);
    else
        gather_carry_kernel<float><<<n_rows, 128, 0, s>>>(U, row_seq, n_rows, d, capacity, map, (const float*)carry,
                                                          (const float*)fill, (float*)out);
    return cudaGetLastError();
}

cudaError_t launch_commit(uint32_t* local, uint32_t* sink, const uint32_t* sel, int total_words, int sink_static,
                          cudaStream_t s) {
    commit_kernel<<<(total_words + 255) / 256, 256, 0, s>>>(local, sink, sel, total_words, sink_static);
    return cudaGetLastError();
}

}  // namespace kvr

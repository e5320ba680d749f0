// kvr_internal.h -- library-private state and kernel launchers.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>
#include <string>
#include <utility>
#include <vector>

#include "../../include/kvr.h"

namespace kvr {

// device error word bits (err[0]); err[1] holds the first failing detail
enum : int {
    DEV_ERR_TIMEOUT = 1,     // a bounded wait gave up
    DEV_ERR_INDEX = 2,       // an index failed its device-side bounds check
    DEV_ERR_DUPLICATE = 4,   // duplicate position reached the device
};

constexpr int kNumSMs = 152;          // GB300
constexpr int kAttnKeysPerTile = 128; // K/V tile of the tensor-core attention
constexpr int kAttnCTAsPerSM = 1;     // tensor-core attention CTAs resident per SM
// Merge of a split query tile's partials: by the last of its CTAs inside the
// attention launch, or by a second kernel over all split tiles.
constexpr int kAttnMergeLastCTA = 0;
constexpr int kAttnMergeKernel = 1;
constexpr int kSimtRowsPerTile = 16;  // query positions per CTA of the SIMT attention
constexpr int kSimtKeysPerTile = 64;

struct Selection {
    int32_t n_rows = 0, n_intervals = 0, n_tiles = 0;
    int32_t rows_per_tile = 0, keys_per_tile = 0;
    int32_t attn_chunk = 1 << 30, attn_split = 1;   // K/V split of the attention
    int32_t attn_merge = kAttnMergeLastCTA;         // who merges the split partials
    std::vector<int32_t> counts, row_off, iv_count, iv_off, tile_count, tile_off;
    bool valid = false;
};

struct ProfRec {
    int kind;
    cudaEvent_t a, b;
    int launches;   // kernels launched between the two events
};


struct kvr_cache_impl {
    kvr_model_desc m{};
    int32_t batch = 0, capacity = 0, n_tokens = 0, suffix_start = 0, words = 0;
    float alpha = 0.f, beta = 0.f;
    uint32_t flags = 0;
    void* k_base = nullptr;
    void* v_base = nullptr;
    int device = 0;

    // library-owned device buffers
    uint32_t* d_local = nullptr;   // [batch][words]
    uint32_t* d_sink = nullptr;
    uint32_t* d_sel = nullptr;
    uint32_t* d_eloc = nullptr;
    uint32_t* d_esnk = nullptr;
    int32_t* d_raw = nullptr;      // [batch*capacity] uploaded positions
    int32_t* d_U = nullptr;        // [batch*capacity] sorted positions, all sequences
    int32_t* d_row_seq = nullptr;  // [batch*capacity]
    int32_t* d_iv = nullptr;       // [batch*capacity][2]
    int32_t* d_plan = nullptr;     // [max_tiles][8]
    int32_t* d_seqinfo = nullptr;  // [batch][8]: count, row_off, iv_off, tile_off, n_tiles
    float2* d_rope = nullptr;      // [capacity][head_dim/2] (cos, sin)
    int32_t* d_err = nullptr;      // [4]
    int32_t* d_map = nullptr;      // [batch][capacity] position -> row (carry selections)
    int32_t* d_attn_sync = nullptr;  // [2][max_tiles][n_kv_heads] attention merge counters
    int32_t max_tiles = 0;

    // pinned staging for the position upload
    int32_t* h_stage = nullptr;
    size_t stage_elems = 0;
    cudaEvent_t stage_ev = nullptr;

    Selection sel;

    bool profiling = false;
    std::vector<ProfRec> prof;
    std::vector<cudaEvent_t> ev_pool;
    double prof_ms[KVR_K_COUNT] = {};
    int64_t prof_n[KVR_K_COUNT] = {};
};

// ---------------------------------------------------------------- host helpers
void set_error(const std::string& msg);
kvr_status cuda_fail(cudaError_t e, const char* what);

// Tensor maps (driver entry point fetched through the runtime).
bool make_tmap_2d_bf16(CUtensorMap* out, const void* base, uint64_t inner, uint64_t rows,
                       uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_rows, std::string* why);
bool make_tmap_3d_bf16(CUtensorMap* out, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
                       uint64_t stride1_bytes, uint64_t stride2_bytes, uint32_t b0, uint32_t b1, uint32_t b2,
                       std::string* why);
// 4-d: dims[0] innermost (elements), strides of dims 1-3 in bytes
bool make_tmap_4d_bf16(CUtensorMap* out, const void* base, const uint64_t dims[4], const uint64_t strides_bytes[3],
                       const uint32_t box[4], std::string* why);
// fp32 rows x 128-byte boxes with the 128-byte swizzle (rows of `inner` floats)
bool make_tmap_2d_f32_sw128(CUtensorMap* out, const void* base, uint64_t inner, uint64_t rows, uint32_t box_rows,
                            std::string* why);

// ---------------------------------------------------------------- launchers
struct SelectLaunch {
    const int32_t* raw;        // uploaded positions, sequence-major
    const int32_t* seqinfo;    // [batch][8]
    const uint32_t* local;
    const uint32_t* sink;
    uint32_t* sel;
    uint32_t* eloc;
    uint32_t* esnk;
    int32_t* U;
    int32_t* row_seq;
    int32_t* iv;
    int32_t* plan;
    int32_t* err;
    int32_t words, suffix_start, n_tokens, rows_per_tile, keys_per_tile, sink_static;
};
cudaError_t launch_select(const SelectLaunch& a, int batch, cudaStream_t s);

cudaError_t launch_gather(int dtype, const int32_t* U, const int32_t* row_seq, int n_rows, int d,
                          int capacity, const int32_t* token_ids, const void* embed, const void* hidden_src,
                          void* out, int32_t* err, int vocab_guard, cudaStream_t s);

// One thread block waiting, with a budget of `cycles`, on an mbarrier phase
// that nothing completes; records DEV_ERR_TIMEOUT in err[0] when it gives up.
cudaError_t launch_wait_check(int32_t* err, long long cycles, cudaStream_t s);

cudaError_t launch_commit(uint32_t* local, uint32_t* sink, const uint32_t* sel, int total_words, int sink_static,
                          cudaStream_t s);
cudaError_t launch_map_rows(const int32_t* U, const int32_t* row_seq, int n_rows, int capacity, int32_t* map,
                            cudaStream_t s);
cudaError_t launch_gather_carry(int dtype, const int32_t* U, const int32_t* row_seq, int n_rows, int d, int capacity,
                                const int32_t* map, const void* carry, const void* fill, void* out, cudaStream_t s);
// w_out[i][k] = w[i][k] + scale * sum_j b[i - row_begin][j] * a[j][k] for rows in
// [row_begin, row_begin + row_count); other rows copied when w_out != w
cudaError_t launch_lora_merge(int dtype, const void* w, void* w_out, int n_out, int K, int row_begin, int row_count,
                              const void* a, const void* b, int rank, float scale, cudaStream_t s);

// Row move with key re-rotation (Shift / splice).  Slab = one (sequence,
// layer, K/V head) run of rows; source slab i maps to destination slab
// i + dst_slab_off.  Rows [src_row0, src_row0 + n_rows) of a source slab land
// at dst_row0.. of its destination slab; keys are rotated by the angle table
// cs[i] = (cos, sin) of delta * theta^(-2i/head_dim), values copied.
struct MoveLaunch {
    const void* k_src;
    const void* v_src;
    void* k_dst;
    void* v_dst;
    int64_t src_slab_rows;
    int64_t dst_slab_rows;
    int64_t dst_slab_off;
    int32_t src_row0, dst_row0, n_rows, chunk, n_slabs;
    float2 cs[64];
};
// in_place: source and destination are the same buffers, dst_row0 <= src_row0
cudaError_t launch_move_rows(int dtype, int head_dim, const MoveLaunch& a, bool in_place, cudaStream_t s);
cudaError_t launch_shift_bits(uint32_t* local, uint32_t* sink, int batch, int words, int start, int d, int n_old,
                              cudaStream_t s);
// local/sink point at the sequence's own words
cudaError_t launch_set_bits(uint32_t* local, uint32_t* sink, int dst, int n, uint32_t flags, cudaStream_t s);

// RMSNorm: in is model dtype (in_f32 = 0) or fp32 (in_f32 = 1), out model dtype.
cudaError_t launch_rmsnorm(int dtype, const void* in, int in_f32, const void* w, void* out, int rows, int d,
                           float eps, cudaStream_t s);

// GEMM partials: part[split][r][f] = sum_{k in split} x[r][k] * w[f][k]
struct GemmPlan {
    int n_out, K, R;
    int m_tiles, n_tiles, BN, splits, stages, atoms;
    int n_sub;      // row tiles of BN rows per work item (1, or 2 when a pair fits one CTA)
    int swiglu_F;   // > 0: gate/up projection with the SwiGLU fused (act output, no partials)
};
// pair_rows: the plan may give one CTA both row tiles of a feature tile
GemmPlan plan_gemm(int dtype, int n_out, int K, int R, bool pair_rows = true);
size_t gemm_partial_bytes(const GemmPlan& p);
// w_written_before: an earlier kernel of the call writes w, so its tiles are
// loaded only after the wait for the previous kernel.
cudaError_t launch_gemm(int dtype, const GemmPlan& p, const void* w, const void* x, float* part, int32_t* err,
                        cudaStream_t s, std::string* why, void* act = nullptr, bool w_written_before = false);

// Epilogues (sum split partials in split order, then the fused op).
struct QkvEpi {
    const float* part;
    int splits, R, n_q_heads, n_kv_heads, head_dim;
    const void* bias;          // nullable
    const void* q_norm;        // [head_dim] per-head RMSNorm weights of Q and K, or NULL (no Q/K norm)
    const void* k_norm;
    float eps;
    const float2* rope;        // [capacity][head_dim/2]
    const int32_t* U;
    const int32_t* row_seq;
    void* q_out;               // [R][Hq][dh]
    void* k_base;
    void* v_base;
    int layer, n_layers, capacity;
    int32_t* err;
};
cudaError_t launch_epi_qkv(int dtype, const QkvEpi& a, cudaStream_t s);
cudaError_t launch_epi_swiglu(int dtype, const float* part, int splits, int R, int F, void* act_out,
                              cudaStream_t s);
cudaError_t launch_epi_down(int dtype, const float* part, int splits, int R, int d, const float* h, void* x_out,
                            cudaStream_t s);
// h = x + O partials (fp32) and hn = RMSNorm(h) * w in one pass per row
cudaError_t launch_epi_residual_norm(int dtype, const float* part, int splits, int R, int d, const void* x, float* h,
                                     const void* w, void* hn, float eps, cudaStream_t s);
// x' = h + down partials (model dtype) and the next layer's xn = RMSNorm(x') * w_next
cudaError_t launch_epi_down_norm(int dtype, const float* part, int splits, int R, int d, const float* h, void* x,
                                 const void* w_next, void* xn, float eps, cudaStream_t s);

// Attention over the mixed cache.
struct AttnLaunch {
    const void* q;             // [R][Hq][dh]
    void* out;                 // [R][Hq*dh]
    const void* k_base;
    const void* v_base;
    const int32_t* U;
    const int32_t* plan;       // [n_tiles][8]
    const uint32_t* loc;       // [batch][words]
    const uint32_t* snk;
    int n_tiles, n_q_heads, n_kv_heads, head_dim, layer, n_layers, capacity, n_tokens, words, batch;
    int n_rows;                // packed rows of q and out
    float alpha, beta;
    int32_t* err;
    float* part_o;             // nullable: split partials [splits][tiles][H_kv][128][128]
    float* part_ml;            // [splits][tiles][H_kv][128][2] (running max in base 2, sum)
    int* sync;                 // [2][tiles][H_kv] merge counters, zero between launches
    int chunk;                 // K/V tiles per CTA when split
    int n_split;               // CTAs per (query tile, K/V head); 1 = unsplit
    int merge;                 // kAttnMergeLastCTA or kAttnMergeKernel
};
cudaError_t launch_attention(int dtype, const AttnLaunch& a, cudaStream_t s, std::string* why);
// Kernels launch_attention issues for a (2 when a merge kernel follows).
int attention_launches(int dtype, const AttnLaunch& a);
// Query tile geometry of the attention kernel for a model.
void attention_tiling(int dtype, int n_q_heads, int n_kv_heads, int* rows_per_tile, int* keys_per_tile);
// Split of each query tile's K/V range over CTAs, from the per-tile K/V tile
// counts of a selection: chunk tiles per CTA, n_split CTAs per (tile, head),
// and which merge (kAttnMerge*) combines the splits.
void attention_chunking(int dtype, const std::vector<int>& tile_kv, int n_kv_heads, int* chunk, int* n_split,
                        int* merge);
// Scratch bytes of the split partials (0 = unsplit); never above
// kAttnMaxSplitCTAs CTAs' worth.
constexpr int kAttnMaxSplitCTAs = 4 * kNumSMs;
size_t attention_scratch_bytes(int dtype, int n_split, int n_tiles, int n_kv_heads);

// ---------------------------------------------------------------- dependent launch
// Kernels of one library call run back to back on one stream.  Each kernel
// signals at entry that the next one may be scheduled, and the next one does
// its set-up (barriers, tensor memory, descriptor prefetch, and for the
// projections the first weight tiles, which no kernel writes) before
// griddepcontrol.wait, which returns once the previous grid has completed and
// its writes are visible.  Every access to data another kernel of the call
// produces or consumes comes after that wait.  The first kernel of each call
// is launched with plain stream order, so nothing overlaps work the caller
// enqueued before the call.
#ifdef __CUDACC__
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
#endif

// Host side: whether the next launch may overlap the previous kernel of the
// same call (false for a call's first launch; set by pdl_begin_call()).
void pdl_begin_call();
bool pdl_take();   // returns the current permission and grants it to later launches
void pdl_disarm(); // the next launch waits for all earlier work of the stream

// Host-side fault injection (KVR_FAULT, read by pdl_begin_call at the start
// of every call): whether the named step fails in this call.  "alloc" counts
// allocations: alloc_fault() is true for the N-th one of "alloc:N" (every
// one for plain "alloc").
bool fault_at(const char* point);
bool alloc_fault();

template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                          Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    if (pdl_take()) {
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    if (fault_at("launch")) return cudaErrorLaunchFailure;   // injected: nothing is issued
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

#define KVR_LAUNCH(...)                                     \
    do {                                                    \
        cudaError_t e_ = ::kvr::launch_kernel(__VA_ARGS__); \
        if (e_ != cudaSuccess) return e_;                   \
    } while (0)

}  // namespace kvr

struct kvr_cache : public kvr::kvr_cache_impl {};

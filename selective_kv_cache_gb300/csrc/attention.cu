// attention.cu -- picks the attention kernel for the model dtype and reports
// its query-tile geometry (the plan is built over these tiles): the
// tensor-core kernel for bf16 models, the CUDA-core kernel for fp32 models.
#include <algorithm>
#include <cstdlib>
#include <cstring>
#include <functional>
#include <string>

#include "kvr_internal.h"

namespace kvr {

int attn_simt_rows_per_tile(int n_q_heads, int n_kv_heads);
cudaError_t launch_attention_simt(const AttnLaunch& a, cudaStream_t s);
int attn_tc_rows_per_tile(int n_q_heads, int n_kv_heads);
cudaError_t launch_attention_tc(const AttnLaunch& a, cudaStream_t s, std::string* why);
size_t attn_tc_scratch_bytes(int n_split, int n_tiles, int n_kv_heads);

size_t attention_scratch_bytes(int dtype, int n_split, int n_tiles, int n_kv_heads) {
    return dtype == KVR_BF16 ? attn_tc_scratch_bytes(n_split, n_tiles, n_kv_heads) : 0;
}

// Pick the chunk size C and the merge that minimise the modelled time.  The
// model plays out the hardware's dispatch: CTAs go to the SMs in launch order
// (K/V head fastest, then the query tiles from the last, whose ranges are the
// longest, then the split), each of the kAttnCTAsPerSM slots of an SM taking
// the next CTA when its last one ends; a CTA costs ~6 tile-times of set-up
// plus one per K/V tile of its chunk (an empty chunk almost nothing), and a
// CTA of a split query tile one more for storing its rows.
//   merge by the last CTA: such a CTA costs two more (the ticket, the wait),
//     and the first chunk's CTA stands for the one that merges: ~2.5
//     tile-times per other split;
//   merge kernel: the kernel that follows adds ~4 tile-times plus 0.5 per
//     split to the makespan.
// (Fitted to kvr_attend over every chunk size and both merges at the
// Llama-3-8B, seam and matched-work shapes on GB300, for the least loss
// against the fastest measured choice; a 128-key tile-time is ~0.7 us.)  Two
// environment variables narrow the choice, for tests and tuning:
// KVR_ATTN_MERGE=cta|kernel allows one merge only (at the same chunk both
// give the same output bits); KVR_ATTN_CHUNK=C fixes the chunk at C K/V tiles
// when the split that makes stays within kAttnMaxSplitCTAs CTAs.
// tile_kv[t] = K/V tiles of query tile t.  A candidate's dispatch is played
// out only when a lower bound of its makespan leaves it a chance, and the
// last few choices are kept per thread.
namespace {
// The last few choices, per thread: a selection with the same query-tile
// geometry (and the same overrides) gets the same answer without the search.
struct ChunkMemo {
    int dtype = -1, heads = 0;
    std::string env_merge, env_chunk;
    std::vector<int> tile_kv;
    int chunk = 0, n_split = 0, merge = 0;
};
constexpr int kChunkMemo = 8;
thread_local ChunkMemo t_chunk_memo[kChunkMemo];
thread_local int t_chunk_next = 0;
void attention_chunking_search(int dtype, const std::vector<int>& tile_kv, int n_kv_heads, int* chunk, int* n_split,
                               int* merge);
}  // namespace

void attention_chunking(int dtype, const std::vector<int>& tile_kv, int n_kv_heads, int* chunk, int* n_split,
                        int* merge) {
    const char* em = std::getenv("KVR_ATTN_MERGE");
    const char* ec = std::getenv("KVR_ATTN_CHUNK");
    const std::string env_merge = em ? em : "", env_chunk = ec ? ec : "";
    for (const ChunkMemo& e : t_chunk_memo)
        if (e.dtype == dtype && e.heads == n_kv_heads && e.env_merge == env_merge && e.env_chunk == env_chunk &&
            e.tile_kv == tile_kv) {
            *chunk = e.chunk;
            *n_split = e.n_split;
            *merge = e.merge;
            return;
        }
    attention_chunking_search(dtype, tile_kv, n_kv_heads, chunk, n_split, merge);
    ChunkMemo& e = t_chunk_memo[t_chunk_next];
    t_chunk_next = (t_chunk_next + 1) % kChunkMemo;
    e.dtype = dtype;
    e.heads = n_kv_heads;
    e.env_merge = env_merge;
    e.env_chunk = env_chunk;
    e.tile_kv = tile_kv;
    e.chunk = *chunk;
    e.n_split = *n_split;
    e.merge = *merge;
}

namespace {
void attention_chunking_search(int dtype, const std::vector<int>& tile_kv, int n_kv_heads, int* chunk, int* n_split,
                               int* merge) {
    *chunk = 1 << 30;
    *n_split = 1;
    *merge = kAttnMergeLastCTA;
    if (dtype != KVR_BF16 || tile_kv.empty()) return;
    const char* env = std::getenv("KVR_ATTN_MERGE");
    const bool allow_cta = !(env && std::strcmp(env, "kernel") == 0);
    const bool allow_kernel = !(env && std::strcmp(env, "cta") == 0);
    int max_kv = 1;
    for (int v : tile_kv) max_kv = std::max(max_kv, v);
    std::vector<double> sm_free;
    std::greater<double> later;
    auto cta_cost = [&](int C, int z, int v, int how) {
        const int n = std::max(0, std::min(C, v - z * C));
        const int live = (v + C - 1) / C;
        double cost = n > 0 ? n + 6.0 : 0.3;
        if (n > 0 && live > 1) cost += 1.0;
        if (n > 0 && live > 1 && how == kAttnMergeLastCTA) cost += 2.0 + (z == 0 ? 2.5 * (live - 1) : 0.0);
        return cost;
    };
    auto merge_cost = [&](int splits, int how) { return how == kAttnMergeKernel && splits > 1 ? 4.0 + 0.5 * splits : 0.0; };
    // a lower bound of the makespan: no SM finishes before its longest CTA,
    // nor before an even share of all the work
    auto lower_bound = [&](int C, int splits, int how) {
        double longest = 0.0, total = 0.0;
        for (int z = 0; z < splits; ++z)
            for (int v : tile_kv) {
                const double c = cta_cost(C, z, v, how);
                longest = std::max(longest, c);
                total += c * n_kv_heads;
            }
        return std::max(longest, total / (kNumSMs * kAttnCTAsPerSM)) + merge_cost(splits, how);
    };
    auto makespan = [&](int C, int splits, int how) {
        sm_free.assign(kNumSMs * kAttnCTAsPerSM, 0.0);
        for (int z = 0; z < splits; ++z)
            for (int t = (int)tile_kv.size() - 1; t >= 0; --t) {
                const double cost = cta_cost(C, z, tile_kv[t], how);
                for (int y = 0; y < n_kv_heads; ++y) {
                    std::pop_heap(sm_free.begin(), sm_free.end(), later);
                    sm_free.back() += cost;
                    std::push_heap(sm_free.begin(), sm_free.end(), later);
                }
            }
        return *std::max_element(sm_free.begin(), sm_free.end()) + merge_cost(splits, how);
    };
    const char* env_c = std::getenv("KVR_ATTN_CHUNK");
    const int fixed = env_c ? std::atoi(env_c) : 0;
    auto fits = [&](int C) {
        const long long splits = (max_kv + C - 1) / C;
        return splits == 1 || splits * (long long)tile_kv.size() * n_kv_heads <= kAttnMaxSplitCTAs;
    };
    const bool pinned = fixed >= 1 && fits(fixed);
    double best = 1e30;
    for (int C = pinned ? std::min(fixed, max_kv) : max_kv; C >= (pinned ? std::min(fixed, max_kv) : 2); --C) {
        const int splits = (max_kv + C - 1) / C;
        if (!fits(C)) break;
        for (int how : {kAttnMergeLastCTA, kAttnMergeKernel}) {
            if ((how == kAttnMergeLastCTA && !allow_cta) || (how == kAttnMergeKernel && !allow_kernel)) continue;
            if (splits == 1 && how == kAttnMergeKernel && allow_cta) continue;   // nothing to merge
            // a candidate wins only below 0.98 of the best so far: play out its
            // dispatch only when its lower bound leaves it a chance (the choice
            // is the same as with every candidate played out)
            if (lower_bound(C, splits, how) >= best * 0.98) continue;
            const double t = makespan(C, splits, how);
            if (t < best * 0.98) {
                best = t;
                *chunk = C;
                *n_split = splits;
                *merge = how;
            }
        }
    }
    if (*n_split == 1) *chunk = 1 << 30;
}
}  // namespace

void attention_tiling(int dtype, int n_q_heads, int n_kv_heads, int* rows_per_tile, int* keys_per_tile) {
    if (dtype == KVR_BF16) {
        *rows_per_tile = attn_tc_rows_per_tile(n_q_heads, n_kv_heads);
        *keys_per_tile = kAttnKeysPerTile;
    } else {
        *rows_per_tile = attn_simt_rows_per_tile(n_q_heads, n_kv_heads);
        *keys_per_tile = kSimtKeysPerTile;
    }
}

int attention_launches(int dtype, const AttnLaunch& a) {
    const bool merged = dtype == KVR_BF16 && a.n_tiles > 0 && a.part_o && a.n_split > 1 && a.merge == kAttnMergeKernel;
    return merged ? 2 : 1;
}

cudaError_t launch_attention(int dtype, const AttnLaunch& a, cudaStream_t s, std::string* why) {
    if (dtype == KVR_BF16) return launch_attention_tc(a, s, why);
    return launch_attention_simt(a, s);
}

}  // namespace kvr

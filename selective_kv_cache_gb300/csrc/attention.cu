// attention.cu -- picks the attention kernel for the model dtype and reports
// its query-tile geometry (the plan is built over these tiles): the
// tensor-core kernel for bf16 models, the CUDA-core kernel for fp32 models.
#include <algorithm>
#include <functional>

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

// Pick the chunk size C that minimises the modelled time.  The model plays
// out the hardware's dispatch: CTAs go to the SMs in launch order (K/V head
// fastest, then the query tiles from the last, whose ranges are the longest,
// then the split), each of the kAttnCTAsPerSM slots of an SM taking the next
// CTA when its last one ends; a CTA costs ~6 tile-times of set-up plus one per
// K/V tile of its chunk (an empty chunk almost nothing), three more when its
// query tile is split (its rows' store, the ticket, the wait), and the first
// chunk's CTA stands for the one that merges: ~1.7 tile-times per other
// split.  (Fitted to kvr_attend over chunk sizes at the Llama-3-8B, seam and
// matched-work shapes on GB300; a 128-key tile-time is ~0.7 us.)
// tile_kv[t] = K/V tiles of query tile t.
void attention_chunking(int dtype, const std::vector<int>& tile_kv, int n_kv_heads, int* chunk, int* n_split) {
    *chunk = 1 << 30;
    *n_split = 1;
    if (dtype != KVR_BF16 || tile_kv.empty()) return;
    int max_kv = 1;
    for (int v : tile_kv) max_kv = std::max(max_kv, v);
    std::vector<double> sm_free;
    std::greater<double> later;
    auto makespan = [&](int C, int splits) {
        sm_free.assign(kNumSMs * kAttnCTAsPerSM, 0.0);
        for (int z = 0; z < splits; ++z)
            for (int t = (int)tile_kv.size() - 1; t >= 0; --t)
                for (int y = 0; y < n_kv_heads; ++y) {
                    const int v = tile_kv[t];
                    const int n = std::max(0, std::min(C, v - z * C));
                    const int live = (v + C - 1) / C;
                    const double merge = (z == 0 && live > 1) ? 1.7 * (live - 1) : 0.0;
                    std::pop_heap(sm_free.begin(), sm_free.end(), later);
                    sm_free.back() += n > 0 ? n + 6.0 + (live > 1 ? 3.0 : 0.0) + merge : 0.3;
                    std::push_heap(sm_free.begin(), sm_free.end(), later);
                }
        return *std::max_element(sm_free.begin(), sm_free.end());
    };
    double best = 1e30;
    for (int C = max_kv; C >= 2; --C) {
        const int splits = (max_kv + C - 1) / C;
        if (splits > 1 && (long long)splits * (long long)tile_kv.size() * n_kv_heads > kAttnMaxSplitCTAs) break;
        const double t = makespan(C, splits);
        if (t < best * 0.98) {
            best = t;
            *chunk = C;
            *n_split = splits;
        }
    }
    if (*n_split == 1) *chunk = 1 << 30;
}

void attention_tiling(int dtype, int n_q_heads, int n_kv_heads, int* rows_per_tile, int* keys_per_tile) {
    if (dtype == KVR_BF16) {
        *rows_per_tile = attn_tc_rows_per_tile(n_q_heads, n_kv_heads);
        *keys_per_tile = kAttnKeysPerTile;
    } else {
        *rows_per_tile = attn_simt_rows_per_tile(n_q_heads, n_kv_heads);
        *keys_per_tile = kSimtKeysPerTile;
    }
}

cudaError_t launch_attention(int dtype, const AttnLaunch& a, cudaStream_t s, std::string* why) {
    if (dtype == KVR_BF16) return launch_attention_tc(a, s, why);
    return launch_attention_simt(a, s);
}

}  // namespace kvr

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
int attn_tc_max_clusters(int n);

// Pick the number n of CTAs (one thread-block cluster) that share each query
// tile's K/V range, by the modelled time.  The model plays out the
// hardware's dispatch: clusters go out in launch order (K/V head fastest,
// then the query tiles from the last, whose ranges are the longest), each
// taking the earliest free one of the cluster slots the GPU holds at once
// (the occupancy query), and a cluster lasts its longest chunk,
// ceil(tiles / n), plus ~6 tile-times of set-up and one more for the merge
// when n > 1.  tile_kv[t] = K/V tiles of query tile t.
void attention_chunking(int dtype, const std::vector<int>& tile_kv, int n_kv_heads, int* n_split) {
    *n_split = 1;
    if (dtype != KVR_BF16 || tile_kv.empty()) return;
    std::vector<double> slot_free;
    std::greater<double> later;
    double best = 1e30;
    for (int n = 1; n <= 8; ++n) {
        const int slots = n == 1 ? kNumSMs : attn_tc_max_clusters(n);
        if (slots <= 0) continue;
        slot_free.assign(slots, 0.0);
        for (int t = (int)tile_kv.size() - 1; t >= 0; --t)
            for (int y = 0; y < n_kv_heads; ++y) {
                const double cost = (tile_kv[t] + n - 1) / n + 6.0 + (n > 1 ? 1.0 : 0.0);
                std::pop_heap(slot_free.begin(), slot_free.end(), later);
                slot_free.back() += cost;
                std::push_heap(slot_free.begin(), slot_free.end(), later);
            }
        const double t = *std::max_element(slot_free.begin(), slot_free.end());
        if (t < best * 0.98) {
            best = t;
            *n_split = n;
        }
    }
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

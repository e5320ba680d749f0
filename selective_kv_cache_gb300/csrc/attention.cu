// attention.cu -- picks the attention kernel for the model dtype and reports
// its query-tile geometry (the plan is built over these tiles).
#include "kvr_internal.h"

namespace kvr {

size_t attn_simt_smem(int head_dim);
int attn_simt_rows_per_tile(int n_q_heads, int n_kv_heads);
cudaError_t launch_attention_simt(int dtype, const AttnLaunch& a, cudaStream_t s);

void attention_tiling(int dtype, int n_q_heads, int n_kv_heads, int* rows_per_tile, int* keys_per_tile) {
    (void)dtype;
    *rows_per_tile = attn_simt_rows_per_tile(n_q_heads, n_kv_heads);
    *keys_per_tile = kSimtKeysPerTile;
}

cudaError_t launch_attention(int dtype, const AttnLaunch& a, cudaStream_t s, std::string* why) {
    (void)why;
    return launch_attention_simt(dtype, a, s);
}

}  // namespace kvr

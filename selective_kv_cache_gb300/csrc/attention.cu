// attention.cu -- picks the attention kernel for the model dtype and reports
// its query-tile geometry (the plan is built over these tiles): the
// tensor-core kernel for bf16 models, the CUDA-core kernel for fp32 models.
#include "kvr_internal.h"

namespace kvr {

int attn_simt_rows_per_tile(int n_q_heads, int n_kv_heads);
cudaError_t launch_attention_simt(const AttnLaunch& a, cudaStream_t s);
int attn_tc_rows_per_tile(int n_q_heads, int n_kv_heads);
cudaError_t launch_attention_tc(const AttnLaunch& a, cudaStream_t s, std::string* why);
size_t attn_tc_scratch_bytes(int n_tiles, int n_kv_heads, int n_tokens);

size_t attention_scratch_bytes(int dtype, int n_tiles, int n_kv_heads, int n_tokens) {
    return dtype == KVR_BF16 ? attn_tc_scratch_bytes(n_tiles, n_kv_heads, n_tokens) : 0;
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

// api.cu -- the C ABI (kvr.h): host-side validation, library-owned state,
// and the per-layer launch sequence of the packed refresh.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "kvr_internal.h"

namespace kvr {

namespace {
thread_local std::string g_err;

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

bool get_encode(std::string* why) {
    std::call_once(g_encode_once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    if (!g_encode) {
        if (why) *why = "cuTensorMapEncodeTiled is not available from the driver";
        return false;
    }
    return true;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// (cos, sin) of delta * theta^(-2i/head_dim) for i < head_dim/2, the angles
// formed in double as for the rotary table; a rotation by delta positions
void rotation_table(const kvr_model_desc& m, double delta, float2* cs) {
    const int half = m.head_dim / 2;
    for (int i = 0; i < 64; ++i) cs[i] = make_float2(1.f, 0.f);
    for (int i = 0; i < half; ++i) {
        const double a = delta * std::pow(m.rope_theta, -2.0 * i / (double)m.head_dim);
        cs[i] = make_float2((float)std::cos(a), (float)std::sin(a));
    }
}
int dtype_size(int dtype) { return dtype == KVR_BF16 ? 2 : 4; }

struct WsLayout {
    size_t xn, q, o, h, hn, act, part, part_size, total;
};

struct Gemms {
    GemmPlan qkv, o, gu, down;
};

// Where the rows of a new selection come from.
struct RowSource {
    const int32_t* token_ids = nullptr;   // with embed: embed[token_ids[seq][u]]
    const void* embed = nullptr;
    int vocab = 0;
    const void* hidden_src = nullptr;     // per-position rows [batch][capacity][d]
    const void* carry = nullptr;          // rows of the current selection (kept for positions in both)
    const void* fill = nullptr;           // per-position rows for the other positions
};

Gemms plan_all(const kvr_model_desc& m, int R) {
    Gemms g;
    const int hqd = m.n_q_heads * m.head_dim;
    g.qkv = plan_gemm(m.dtype, (m.n_q_heads + 2 * m.n_kv_heads) * m.head_dim, m.d_model, R);
    g.o = plan_gemm(m.dtype, m.d_model, hqd, R);
    // unpaired: the fused SwiGLU takes whole K ranges, and paired items of
    // the gate/up shape would leave the last round half empty
    g.gu = plan_gemm(m.dtype, 2 * m.ffn_dim, m.d_model, R, false);
    // one K split: the gate/up projection writes silu(g) * u directly (no partials)
    if (m.dtype == KVR_BF16 && g.gu.splits == 1 && m.ffn_dim % 64 == 0) g.gu.swiglu_F = m.ffn_dim;
    g.down = plan_gemm(m.dtype, m.d_model, m.ffn_dim, R);
    return g;
}

// The projections' split-K partials and the attention's split partials
// share one region: they are never live at the same time.
size_t part_bytes(const kvr_model_desc& m, int R, size_t attn_scratch) {
    const Gemms g = plan_all(m, R);
    const size_t gu = g.gu.swiglu_F ? 0 : gemm_partial_bytes(g.gu);
    const size_t gemm = std::max(std::max(gemm_partial_bytes(g.qkv), gemm_partial_bytes(g.o)),
                                 std::max(gu, gemm_partial_bytes(g.down)));
    return std::max(gemm, attn_scratch);
}

size_t sel_attn_scratch(const kvr_cache* c) {
    return attention_scratch_bytes(c->m.dtype, c->sel.attn_split, c->sel.n_tiles, c->m.n_kv_heads);
}

// Point the attention at its split scratch when the region holds it (else it
// runs unsplit).
void set_attention_scratch(AttnLaunch* a, float* region, size_t bytes, const kvr_cache* c) {
    const size_t need = sel_attn_scratch(c);
    a->part_o = nullptr;
    a->part_ml = nullptr;
    a->sync = c->d_attn_sync;
    a->chunk = c->sel.attn_chunk;
    a->n_split = c->sel.attn_split;
    a->merge = c->sel.attn_merge;
    if (need == 0 || !region || bytes < need) {
        a->n_split = 1;
        return;
    }
    const size_t o_floats = need / sizeof(float) / 130 * 128;
    a->part_o = region;
    a->part_ml = region + o_floats;
}

WsLayout layout(const kvr_model_desc& m, int R, size_t part) {
    const size_t es = dtype_size(m.dtype);
    const size_t hqd = (size_t)m.n_q_heads * m.head_dim;
    WsLayout L{};
    size_t off = 0;
    L.xn = off; off = align256(off + (size_t)R * m.d_model * es);
    L.q = off; off = align256(off + (size_t)R * hqd * es);
    L.o = off; off = align256(off + (size_t)R * hqd * es);
    L.h = off; off = align256(off + (size_t)R * m.d_model * 4);
    L.hn = off; off = align256(off + (size_t)R * m.d_model * es);
    L.act = off; off = align256(off + (size_t)R * m.ffn_dim * es);
    L.part = off; off = align256(off + part);
    L.part_size = part;
    L.total = off;
    return L;
}

// ---------------------------------------------------------------- profiling
cudaEvent_t take_event(kvr_cache* c) {
    if (!c->ev_pool.empty()) {
        cudaEvent_t e = c->ev_pool.back();
        c->ev_pool.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    cudaEventCreate(&e);
    return e;
}

struct Prof {
    kvr_cache* c;
    int kind;
    cudaStream_t s;
    cudaEvent_t a = nullptr;
    int launches = 1;   // kernels launched inside the scope
    Prof(kvr_cache* c_, int k, cudaStream_t s_) : c(c_), kind(k), s(s_) {
        if (c->profiling) {
            a = take_event(c);
            cudaEventRecord(a, s);
        }
    }
    ~Prof() {
        if (a) {
            cudaEvent_t b = take_event(c);
            cudaEventRecord(b, s);
            c->prof.push_back({kind, a, b, launches});
        }
    }
};

#define KVR_CHECK_LAUNCH(expr, what)                            \
    do {                                                        \
        cudaError_t e_ = (expr);                                \
        if (e_ != cudaSuccess) return cuda_fail(e_, what);      \
    } while (0)

kvr_status validate_desc(const kvr_model_desc* m) {
    if (!m) {
        set_error("model descriptor is NULL");
        return KVR_EINVAL;
    }
    if (m->n_layers < 1 || m->d_model < 64 || m->n_q_heads < 1 || m->n_kv_heads < 1 || m->ffn_dim < 64 ||
        m->n_q_heads % m->n_kv_heads != 0) {
        set_error("model shape is malformed");
        return KVR_EINVAL;
    }
    if (m->dtype != KVR_BF16 && m->dtype != KVR_F32) {
        set_error("dtype must be KVR_F32 or KVR_BF16");
        return KVR_EUNSUPPORTED;
    }
    if (m->d_model > 8192) {
        set_error("d_model above 8192 is not supported (row kernels keep a row in registers)");
        return KVR_EUNSUPPORTED;
    }
    if (m->d_model % 64 || m->ffn_dim % 64 || (m->n_q_heads * m->head_dim) % 64) {
        set_error("d_model, ffn_dim and n_q_heads*head_dim must be multiples of 64");
        return KVR_EUNSUPPORTED;
    }
    if (m->dtype == KVR_BF16) {
        if (m->head_dim != 128 || m->d_model % 128) {
            set_error("bf16 models need head_dim 128 and d_model a multiple of 128");
            return KVR_EUNSUPPORTED;
        }
    } else if (m->head_dim != 64 && m->head_dim != 128) {
        set_error("fp32 models need head_dim 64 or 128");
        return KVR_EUNSUPPORTED;
    }
    if (!(m->rope_theta > 0.0) || !(m->rms_eps >= 0.f)) {
        set_error("rope_theta must be > 0 and rms_eps >= 0");
        return KVR_EINVAL;
    }
    return KVR_OK;
}

void free_cache(kvr_cache* c) {
    cudaFree(c->d_local);
    cudaFree(c->d_sink);
    cudaFree(c->d_sel);
    cudaFree(c->d_eloc);
    cudaFree(c->d_esnk);
    cudaFree(c->d_seqinfo);  // d_raw lives in the same allocation
    cudaFree(c->d_U);
    cudaFree(c->d_row_seq);
    cudaFree(c->d_iv);
    cudaFree(c->d_plan);
    cudaFree(c->d_rope);
    cudaFree(c->d_err);
    cudaFree(c->d_map);
    cudaFree(c->d_attn_sync);
    if (c->h_stage) cudaFreeHost(c->h_stage);
    if (c->stage_ev) cudaEventDestroy(c->stage_ev);
    for (auto& r : c->prof) {
        cudaEventDestroy(r.a);
        cudaEventDestroy(r.b);
    }
    for (auto e : c->ev_pool) cudaEventDestroy(e);
    delete c;
}

kvr_status check_layer_weights(const kvr_cache* c, const kvr_layer_weights* w) {
    if (!w || !w->w_qkv || !w->w_o || !w->w_gate_up || !w->w_down || !w->norm1 || !w->norm2) {
        set_error("layer weights: NULL pointer");
        return KVR_EINVAL;
    }
    if (c->m.has_qkv_bias && !w->b_qkv) {
        set_error("layer weights: the model has q/k/v biases but b_qkv is NULL");
        return KVR_EINVAL;
    }
    if (c->m.has_qk_norm && (!w->q_norm || !w->k_norm)) {
        set_error("layer weights: the model has Q/K normalisation but q_norm or k_norm is NULL");
        return KVR_EINVAL;
    }
    const void* ps[] = {w->w_qkv, w->b_qkv, w->w_o, w->w_gate_up, w->w_down, w->norm1, w->norm2,
                        c->m.has_qk_norm ? w->q_norm : nullptr, c->m.has_qk_norm ? w->k_norm : nullptr};
    for (const void* p : ps)
        if (p && !aligned16(p)) {
            set_error("layer weights must be 16-byte aligned");
            return KVR_EINVAL;
        }
    return KVR_OK;
}

// One layer of the packed refresh over the current selection.
// xn_ready: the previous layer's down epilogue already wrote this layer's
// normalised rows into the workspace; next_norm1: fuse the next layer's first
// RMSNorm into this layer's down epilogue (NULL for the last layer run).
kvr_status run_layer(kvr_cache* c, int layer, const kvr_layer_weights* w, void* hidden, uint8_t* ws,
                     const WsLayout& L, cudaStream_t s, bool xn_ready = false, const void* next_norm1 = nullptr) {
    const kvr_model_desc& m = c->m;
    const int R = c->sel.n_rows;
    const int dt = m.dtype;
    const Gemms g = plan_all(m, R);
    void* xn = ws + L.xn;
    void* q = ws + L.q;
    void* o = ws + L.o;
    float* h = reinterpret_cast<float*>(ws + L.h);
    void* hn = ws + L.hn;
    void* act = ws + L.act;
    float* part = reinterpret_cast<float*>(ws + L.part);
    std::string why;

    if (!xn_ready) {
        Prof p(c, KVR_K_RMSNORM, s);
        KVR_CHECK_LAUNCH(launch_rmsnorm(dt, hidden, 0, w->norm1, xn, R, m.d_model, m.rms_eps, s), "rmsnorm");
    }
    {
        Prof p(c, KVR_K_GEMM_QKV, s);
        cudaError_t e = launch_gemm(dt, g.qkv, w->w_qkv, xn, part, c->d_err, s, &why);
        if (e != cudaSuccess) return cuda_fail(e, ("qkv projection " + why).c_str());
    }
    {
        Prof p(c, KVR_K_EPI_QKV, s);
        QkvEpi a{};
        a.part = part;
        a.splits = g.qkv.splits;
        a.R = R;
        a.n_q_heads = m.n_q_heads;
        a.n_kv_heads = m.n_kv_heads;
        a.head_dim = m.head_dim;
        a.bias = m.has_qkv_bias ? w->b_qkv : nullptr;
        a.q_norm = m.has_qk_norm ? w->q_norm : nullptr;
        a.k_norm = m.has_qk_norm ? w->k_norm : nullptr;
        a.eps = m.rms_eps;
        a.rope = c->d_rope;
        a.U = c->d_U;
        a.row_seq = c->d_row_seq;
        a.q_out = q;
        a.k_base = c->k_base;
        a.v_base = c->v_base;
        a.layer = layer;
        a.n_layers = m.n_layers;
        a.capacity = c->capacity;
        a.err = c->d_err;
        KVR_CHECK_LAUNCH(launch_epi_qkv(dt, a, s), "qkv epilogue");
    }
    {
        Prof p(c, KVR_K_ATTN, s);
        AttnLaunch a{};
        a.q = q;
        a.out = o;
        a.k_base = c->k_base;
        a.v_base = c->v_base;
        a.U = c->d_U;
        a.plan = c->d_plan;
        a.loc = c->d_eloc;
        a.snk = c->d_esnk;
        a.n_tiles = c->sel.n_tiles;
        a.n_rows = c->sel.n_rows;
        a.n_q_heads = m.n_q_heads;
        a.n_kv_heads = m.n_kv_heads;
        a.head_dim = m.head_dim;
        a.layer = layer;
        a.n_layers = m.n_layers;
        a.capacity = c->capacity;
        a.n_tokens = c->n_tokens;
        a.words = c->words;
        a.batch = c->batch;
        a.alpha = c->alpha;
        a.beta = c->beta;
        a.err = c->d_err;
        set_attention_scratch(&a, part, L.part_size, c);
        p.launches = attention_launches(dt, a);
        cudaError_t e = launch_attention(dt, a, s, &why);
        if (e != cudaSuccess) return cuda_fail(e, ("attention " + why).c_str());
    }
    {
        Prof p(c, KVR_K_GEMM_O, s);
        cudaError_t e = launch_gemm(dt, g.o, w->w_o, o, part, c->d_err, s, &why);
        if (e != cudaSuccess) return cuda_fail(e, ("output projection " + why).c_str());
    }
    {
        Prof p(c, KVR_K_EPI_O, s);
        KVR_CHECK_LAUNCH(launch_epi_residual_norm(dt, part, g.o.splits, R, m.d_model, hidden, h, w->norm2, hn,
                                                  m.rms_eps, s),
                         "o epilogue");
    }
    {
        Prof p(c, KVR_K_GEMM_GATEUP, s);
        cudaError_t e = launch_gemm(dt, g.gu, w->w_gate_up, hn, part, c->d_err, s, &why, act);
        if (e != cudaSuccess) return cuda_fail(e, ("gate/up projection " + why).c_str());
    }
    if (!g.gu.swiglu_F) {
        Prof p(c, KVR_K_EPI_GATEUP, s);
        KVR_CHECK_LAUNCH(launch_epi_swiglu(dt, part, g.gu.splits, R, m.ffn_dim, act, s), "swiglu epilogue");
    }
    {
        Prof p(c, KVR_K_GEMM_DOWN, s);
        cudaError_t e = launch_gemm(dt, g.down, w->w_down, act, part, c->d_err, s, &why);
        if (e != cudaSuccess) return cuda_fail(e, ("down projection " + why).c_str());
    }
    {
        Prof p(c, KVR_K_EPI_DOWN, s);
        if (next_norm1)
            KVR_CHECK_LAUNCH(launch_epi_down_norm(dt, part, g.down.splits, R, m.d_model, h, hidden, next_norm1, xn,
                                                  m.rms_eps, s),
                             "down epilogue");
        else
            KVR_CHECK_LAUNCH(launch_epi_down(dt, part, g.down.splits, R, m.d_model, h, hidden, s), "down epilogue");
    }
    if (fault_at("timeout")) {
        // injected: the error word as a bounded device wait leaves it when it gives up
        static const int32_t kTimeoutWord = DEV_ERR_TIMEOUT;
        KVR_CHECK_LAUNCH(cudaMemcpyAsync(c->d_err, &kTimeoutWord, sizeof(int32_t), cudaMemcpyHostToDevice, s),
                         "timeout injection");
    }
    return KVR_OK;
}

kvr_status commit(kvr_cache* c, cudaStream_t s) {
    Prof p(c, KVR_K_COMMIT, s);
    KVR_CHECK_LAUNCH(launch_commit(c->d_local, c->d_sink, c->d_sel, c->batch * c->words,
                                   (c->flags & KVR_SINK_STATIC) ? 1 : 0, s),
                     "metadata commit");
    return KVR_OK;
}

kvr_status check_refresh_args(kvr_cache* c, void* hidden, void* ws, size_t ws_bytes, WsLayout* L) {
    if (!c) {
        set_error("cache is NULL");
        return KVR_EINVAL;
    }
    if (!c->sel.valid) {
        set_error("no selection: call kvr_select first");
        return KVR_ESTATE;
    }
    const int R = c->sel.n_rows;
    *L = layout(c->m, R, part_bytes(c->m, R, sel_attn_scratch(c)));
    if (R == 0) return KVR_OK;
    if (!hidden || !ws) {
        set_error("hidden rows or workspace is NULL");
        return KVR_EINVAL;
    }
    if ((reinterpret_cast<uintptr_t>(ws) & 255u) || !aligned16(hidden)) {
        set_error("workspace must be 256-byte aligned and hidden rows 16-byte aligned");
        return KVR_EINVAL;
    }
    if (ws_bytes < L->total) {
        set_error("workspace too small: need " + std::to_string(L->total) + " bytes");
        return KVR_EINVAL;
    }
    return KVR_OK;
}

}  // namespace

void set_error(const std::string& msg) { g_err = msg; }

namespace {
thread_local bool t_pdl_armed = false;
thread_local std::string t_fault;      // KVR_FAULT as read at the start of this thread's current call
thread_local int t_alloc_count = 0;
bool pdl_enabled() {
    static const bool on = [] {
        const char* v = std::getenv("KVR_PDL");
        return !(v && v[0] == '0');
    }();
    return on;
}
}  // namespace
void pdl_begin_call() {
    t_pdl_armed = false;
    const char* v = std::getenv("KVR_FAULT");
    t_fault = v ? v : "";
    t_alloc_count = 0;
}
bool fault_at(const char* point) { return !t_fault.empty() && t_fault == point; }
bool alloc_fault() {
    ++t_alloc_count;
    if (t_fault == "alloc") return true;
    if (t_fault.rfind("alloc:", 0) == 0) return t_alloc_count == std::atoi(t_fault.c_str() + 6);
    return false;
}
void pdl_disarm() { t_pdl_armed = false; }
bool pdl_take() {
    const bool r = t_pdl_armed && pdl_enabled();
    t_pdl_armed = true;
    return r;
}

kvr_status cuda_fail(cudaError_t e, const char* what) {
    set_error(std::string(what) + ": " + cudaGetErrorString(e));
    return KVR_ECUDA;
}

namespace {
// Encoded tensor maps, cached per thread: an encoding is a pure function of
// its arguments, and a call re-encodes the same few maps for every launch.
struct TmapKey {
    int dtype, rank, l2;
    const void* base;
    uint64_t dims[4], strides[3];
    uint32_t box[4];
};
struct TmapSlot {
    bool used;
    TmapKey key;
    CUtensorMap map;
};
constexpr int kTmapSlots = 256;
thread_local TmapSlot t_tmaps[kTmapSlots];

bool encode_cached(CUtensorMap* out, CUtensorMapDataType dtype, int rank, const void* base, const uint64_t* dims,
                   const uint64_t* strides, const uint32_t* box, CUtensorMapL2promotion l2, const char* what,
                   std::string* why) {
    TmapKey k;
    std::memset(&k, 0, sizeof(k));
    k.dtype = (int)dtype;
    k.rank = rank;
    k.l2 = (int)l2;
    k.base = base;
    for (int i = 0; i < rank; ++i) {
        k.dims[i] = dims[i];
        k.box[i] = box[i];
        if (i + 1 < rank) k.strides[i] = strides[i];
    }
    uint64_t h = 1469598103934665603ull;   // FNV-1a over the key's bytes
    const unsigned char* kb = reinterpret_cast<const unsigned char*>(&k);
    for (size_t i = 0; i < sizeof(k); ++i) h = (h ^ kb[i]) * 1099511628211ull;
    TmapSlot& slot = t_tmaps[h % kTmapSlots];
    if (slot.used && std::memcmp(&slot.key, &k, sizeof(k)) == 0) {
        *out = slot.map;
        return true;
    }
    if (!get_encode(why)) return false;
    cuuint64_t d[4], st[3];
    cuuint32_t bx[4], es[4] = {1, 1, 1, 1};
    for (int i = 0; i < rank; ++i) {
        d[i] = dims[i];
        bx[i] = box[i];
        if (i + 1 < rank) st[i] = strides[i];
    }
    CUresult r = g_encode(out, dtype, (cuuint32_t)rank, const_cast<void*>(base), d, st, bx, es,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, l2,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        if (why) *why = std::string("cuTensorMapEncodeTiled") + what + " failed with " + std::to_string((int)r);
        return false;
    }
    slot.used = true;
    slot.key = k;
    slot.map = *out;
    return true;
}
}  // namespace

bool make_tmap_2d_bf16(CUtensorMap* out, const void* base, uint64_t inner, uint64_t rows, uint64_t row_stride_bytes,
                       uint32_t box_inner, uint32_t box_rows, std::string* why) {
    const uint64_t dims[2] = {inner, rows}, strides[1] = {row_stride_bytes};
    const uint32_t box[2] = {box_inner, box_rows};
    return encode_cached(out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, "", why);
}

bool make_tmap_3d_bf16(CUtensorMap* out, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
                       uint64_t stride1_bytes, uint64_t stride2_bytes, uint32_t b0, uint32_t b1, uint32_t b2,
                       std::string* why) {
    const uint64_t dims[3] = {d0, d1, d2}, strides[2] = {stride1_bytes, stride2_bytes};
    const uint32_t box[3] = {b0, b1, b2};
    return encode_cached(out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, strides, box,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, "", why);
}

bool make_tmap_4d_bf16(CUtensorMap* out, const void* base, const uint64_t dims_in[4], const uint64_t strides_bytes[3],
                       const uint32_t box_in[4], std::string* why) {
    return encode_cached(out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, base, dims_in, strides_bytes, box_in,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, " (4-d)", why);
}

bool make_tmap_2d_f32_sw128(CUtensorMap* out, const void* base, uint64_t inner, uint64_t rows, uint32_t box_rows,
                            std::string* why) {
    const uint64_t dims[2] = {inner, rows}, strides[1] = {inner * 4};
    const uint32_t box[2] = {32, box_rows};
    return encode_cached(out, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, base, dims, strides, box,
                         CU_TENSOR_MAP_L2_PROMOTION_NONE, " (fp32 rows)", why);
}

kvr_status do_select(kvr_cache* c, const int32_t* positions, const int32_t* counts, int32_t budget_percent,
                     const RowSource& src, void* hidden_out, int32_t* n_rows_out, int32_t* n_intervals_out,
                     cudaStream_t s) {
    if (budget_percent > 100 || budget_percent < -1) {
        set_error("budget_percent must be -1 or in [0, 100]");
        return KVR_EINVAL;
    }
    const int B = c->batch;
    Selection sel;
    sel.counts.assign(counts, counts + B);
    int64_t total = 0;
    for (int i = 0; i < B; ++i) {
        if (counts[i] < 0 || counts[i] > c->n_tokens - c->suffix_start) {
            set_error("count for sequence " + std::to_string(i) + " is outside [0, suffix length]");
            return counts[i] < 0 ? KVR_EINVAL : KVR_ERANGE;
        }
        total += counts[i];
    }
    if (total > 0 && (!positions || !hidden_out)) {
        set_error("positions or hidden_out is NULL");
        return KVR_EINVAL;
    }
    if (hidden_out && !aligned16(hidden_out)) {
        set_error("hidden_out must be 16-byte aligned");
        return KVR_EINVAL;
    }
    const int S = c->n_tokens - c->suffix_start;
    if (budget_percent >= 0) {
        const int want = std::min(S, (int)(((int64_t)S * budget_percent + 99) / 100));
        for (int i = 0; i < B; ++i)
            if (counts[i] != want) {
                set_error("sequence " + std::to_string(i) + " selects " + std::to_string(counts[i]) +
                          " positions; the exact budget is " + std::to_string(want));
                return KVR_EINVAL;
            }
    }
    // validation: range, duplicates; interval count from the membership map
    std::vector<uint8_t> mark(c->n_tokens);
    int64_t off = 0;
    sel.row_off.resize(B);
    sel.iv_count.resize(B);
    sel.iv_off.resize(B);
    sel.tile_count.resize(B);
    sel.tile_off.resize(B);
    attention_tiling(c->m.dtype, c->m.n_q_heads, c->m.n_kv_heads, &sel.rows_per_tile, &sel.keys_per_tile);
    int rows = 0, ivs = 0, tiles = 0;
    std::vector<int> tile_kv;
    for (int i = 0; i < B; ++i) {
        std::fill(mark.begin(), mark.end(), 0);
        for (int k = 0; k < counts[i]; ++k) {
            const int p = positions[off + k];
            if (p < c->suffix_start || p >= c->n_tokens) {
                set_error("position " + std::to_string(p) + " is outside the retained suffix [" +
                          std::to_string(c->suffix_start) + ", " + std::to_string(c->n_tokens) + ")");
                return KVR_ERANGE;
            }
            if (mark[p]) {
                set_error("duplicate position " + std::to_string(p) + " in sequence " + std::to_string(i));
                return KVR_EINVAL;
            }
            mark[p] = 1;
        }
        int iv = 0, row = 0;
        for (int t = c->suffix_start; t < c->n_tokens; ++t) {
            if (!mark[t]) continue;
            if (t == 0 || !mark[t - 1]) ++iv;
            // K/V tiles the attention walks for each query tile: up to its last row
            if (row % sel.rows_per_tile == sel.rows_per_tile - 1 || row == counts[i] - 1)
                tile_kv.push_back((t + 1 + sel.keys_per_tile - 1) / sel.keys_per_tile);
            ++row;
        }
        sel.row_off[i] = rows;
        sel.iv_off[i] = ivs;
        sel.iv_count[i] = iv;
        sel.tile_off[i] = tiles;
        sel.tile_count[i] = (counts[i] + sel.rows_per_tile - 1) / sel.rows_per_tile;
        rows += counts[i];
        ivs += iv;
        tiles += sel.tile_count[i];
        off += counts[i];
    }
    if (tiles > c->max_tiles) {
        set_error("internal: plan capacity exceeded");
        return KVR_EINVAL;
    }
    sel.n_rows = rows;
    sel.n_intervals = ivs;
    sel.n_tiles = tiles;
    attention_chunking(c->m.dtype, tile_kv, c->m.n_kv_heads, &sel.attn_chunk, &sel.attn_split, &sel.attn_merge);

    // the staging buffer may still feed the previous upload
    cudaError_t e = cudaEventSynchronize(c->stage_ev);
    if (e != cudaSuccess) return cuda_fail(e, "staging wait");
    int32_t* st = c->h_stage;
    for (int i = 0, raw = 0; i < B; ++i) {
        int32_t* info = st + 8 * i;
        info[0] = counts[i];
        info[1] = sel.row_off[i];
        info[2] = sel.iv_off[i];
        info[3] = sel.tile_off[i];
        info[4] = sel.tile_count[i];
        info[5] = raw;
        info[6] = 0;
        info[7] = 0;
        raw += counts[i];
    }
    if (total) std::memcpy(st + 8 * B, positions, (size_t)total * sizeof(int32_t));
    // from here on the device selection state changes: the old selection is
    // no longer valid, whether or not the new one completes (its device lists
    // stay intact until the select kernel runs, so a carried selection can
    // still map its rows below)
    const bool had_sel = c->sel.valid;
    c->sel.valid = false;
    e = fault_at("upload") ? cudaErrorUnknown
                           : cudaMemcpyAsync(c->d_seqinfo, st, (8 * B + total) * sizeof(int32_t),
                                             cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) return cuda_fail(e, "position upload");
    e = cudaEventRecord(c->stage_ev, s);
    if (e != cudaSuccess) return cuda_fail(e, "position upload");

    SelectLaunch a{};
    a.raw = c->d_raw;
    a.seqinfo = c->d_seqinfo;
    a.local = c->d_local;
    a.sink = c->d_sink;
    a.sel = c->d_sel;
    a.eloc = c->d_eloc;
    a.esnk = c->d_esnk;
    a.U = c->d_U;
    a.row_seq = c->d_row_seq;
    a.iv = c->d_iv;
    a.plan = c->d_plan;
    a.err = c->d_err;
    a.words = c->words;
    a.suffix_start = c->suffix_start;
    a.n_tokens = c->n_tokens;
    a.rows_per_tile = sel.rows_per_tile;
    a.keys_per_tile = sel.keys_per_tile;
    a.sink_static = (c->flags & KVR_SINK_STATIC) ? 1 : 0;
    if (src.carry) {
        // position -> row map of the selection being replaced (rows carry over)
        const size_t map_bytes = (size_t)c->batch * c->capacity * sizeof(int32_t);
        KVR_CHECK_LAUNCH(cudaMemsetAsync(c->d_map, 0xff, map_bytes, s), "row map");
        if (had_sel)
            KVR_CHECK_LAUNCH(launch_map_rows(c->d_U, c->d_row_seq, c->sel.n_rows, c->capacity, c->d_map, s),
                             "row map");
    }
    // the attention's merge counters return to zero after every complete
    // launch; a new selection starts them from zero whatever came before
    KVR_CHECK_LAUNCH(cudaMemsetAsync(c->d_attn_sync, 0, (size_t)2 * c->max_tiles * c->m.n_kv_heads * sizeof(int32_t), s),
                     "attention counters");
    {
        Prof p(c, KVR_K_SELECT, s);
        KVR_CHECK_LAUNCH(launch_select(a, B, s), "select");
    }
    {
        Prof p(c, KVR_K_GATHER, s);
        if (src.carry)
            KVR_CHECK_LAUNCH(launch_gather_carry(c->m.dtype, c->d_U, c->d_row_seq, rows, c->m.d_model, c->capacity,
                                                 c->d_map, src.carry, src.fill, hidden_out, s),
                             "row gather");
        else
            KVR_CHECK_LAUNCH(launch_gather(c->m.dtype, c->d_U, c->d_row_seq, rows, c->m.d_model, c->capacity,
                                           src.token_ids, src.embed, src.hidden_src, hidden_out, c->d_err, src.vocab,
                                           s),
                             "row gather");
    }
    // the kernels that read this selection (plan, rows, masks) start after
    // it is complete: the next launch waits for the whole stream, so no
    // kernel ever reads the plan in its pre-wait part while it is written
    pdl_disarm();
    sel.valid = true;
    c->sel = sel;
    if (n_rows_out) *n_rows_out = rows;
    if (n_intervals_out) *n_intervals_out = ivs;
    return KVR_OK;
}

}  // namespace kvr

using namespace kvr;

extern "C" {

const char* kvr_last_error(void) { return g_err.c_str(); }

kvr_status kvr_create_cache(const kvr_model_desc* m, int32_t batch, int32_t capacity, void* k_base, void* v_base,
                            int32_t n_tokens, int32_t suffix_start, const uint32_t* local_bits,
                            const uint32_t* sink_bits, float alpha, float beta, uint32_t flags, void* stream,
                            kvr_cache** out) {
    pdl_begin_call();
    if (!out) {
        set_error("out is NULL");
        return KVR_EINVAL;
    }
    *out = nullptr;
    kvr_status st = validate_desc(m);
    if (st != KVR_OK) return st;
    if (batch < 1 || capacity < 1 || n_tokens < 1 || n_tokens > capacity || suffix_start < 0 ||
        suffix_start > n_tokens) {
        set_error("need batch >= 1 and 0 <= suffix_start <= n_tokens <= capacity");
        return KVR_EINVAL;
    }
    if (!k_base || !v_base || !aligned16(k_base) || !aligned16(v_base)) {
        set_error("K/V cache pointers must be non-NULL and 16-byte aligned");
        return KVR_EINVAL;
    }
    if (!std::isfinite(alpha) || !std::isfinite(beta)) {
        set_error("alpha and beta must be finite");
        return KVR_EINVAL;
    }
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    kvr_cache* c = new kvr_cache();
    c->m = *m;
    c->batch = batch;
    c->capacity = capacity;
    c->n_tokens = n_tokens;
    c->suffix_start = suffix_start;
    c->words = (capacity + 31) / 32;
    c->alpha = alpha;
    c->beta = beta;
    c->flags = flags;
    c->k_base = k_base;
    c->v_base = v_base;
    cudaGetDevice(&c->device);

    int rpt = 0, kpt = 0;
    attention_tiling(m->dtype, m->n_q_heads, m->n_kv_heads, &rpt, &kpt);
    const size_t rows = (size_t)batch * capacity;
    c->max_tiles = (int)(rows / rpt + batch + 1);
    const size_t wbytes = (size_t)batch * c->words * sizeof(uint32_t);
    const int half = m->head_dim / 2;
    c->stage_elems = (size_t)batch * 8 + rows;
    cudaError_t e = cudaSuccess;
    auto A = [&](void** p, size_t n) {
        if (e == cudaSuccess) e = alloc_fault() ? cudaErrorMemoryAllocation : cudaMalloc(p, n);
    };
    A((void**)&c->d_local, wbytes);
    A((void**)&c->d_sink, wbytes);
    A((void**)&c->d_sel, wbytes);
    A((void**)&c->d_eloc, wbytes);
    A((void**)&c->d_esnk, wbytes);
    A((void**)&c->d_seqinfo, c->stage_elems * sizeof(int32_t));
    A((void**)&c->d_U, rows * sizeof(int32_t));
    A((void**)&c->d_row_seq, rows * sizeof(int32_t));
    A((void**)&c->d_iv, rows * 2 * sizeof(int32_t));
    A((void**)&c->d_plan, (size_t)c->max_tiles * 8 * sizeof(int32_t));
    A((void**)&c->d_rope, (size_t)capacity * half * sizeof(float2));
    A((void**)&c->d_err, 4 * sizeof(int32_t));
    A((void**)&c->d_map, rows * sizeof(int32_t));
    A((void**)&c->d_attn_sync, (size_t)2 * c->max_tiles * m->n_kv_heads * sizeof(int32_t));
    if (e == cudaSuccess) e = cudaMallocHost((void**)&c->h_stage, c->stage_elems * sizeof(int32_t));
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&c->stage_ev, cudaEventDisableTiming);
    if (e != cudaSuccess) {
        set_error(std::string("allocation failed: ") + cudaGetErrorString(e));
        free_cache(c);
        return KVR_ENOMEM;
    }
    c->d_raw = c->d_seqinfo + (size_t)batch * 8;

    // rotary table: angle u * theta^(-2i/d_h) formed in double, stored as fp32 (cos, sin)
    std::vector<float2> rope((size_t)capacity * half);
    for (int i = 0; i < half; ++i) {
        const double inv = std::pow(m->rope_theta, -2.0 * i / (double)m->head_dim);
        for (int u = 0; u < capacity; ++u) {
            const double a = (double)u * inv;
            rope[(size_t)u * half + i] = make_float2((float)std::cos(a), (float)std::sin(a));
        }
    }
    std::vector<uint32_t> zeros((size_t)batch * c->words, 0u);
    e = cudaMemcpyAsync(c->d_rope, rope.data(), rope.size() * sizeof(float2), cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(c->d_local, local_bits ? local_bits : zeros.data(), wbytes, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(c->d_sink, sink_bits ? sink_bits : zeros.data(), wbytes, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(c->d_err, 0, 4 * sizeof(int32_t), s);
    if (e == cudaSuccess)
        e = cudaMemsetAsync(c->d_attn_sync, 0, (size_t)2 * c->max_tiles * m->n_kv_heads * sizeof(int32_t), s);
    if (e == cudaSuccess) e = cudaMemsetAsync(c->d_sel, 0, wbytes, s);
    if (e == cudaSuccess) e = cudaMemcpyAsync(c->d_eloc, c->d_local, wbytes, cudaMemcpyDeviceToDevice, s);
    if (e == cudaSuccess) e = cudaMemcpyAsync(c->d_esnk, c->d_sink, wbytes, cudaMemcpyDeviceToDevice, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) {
        kvr_status r = cuda_fail(e, "cache set-up");
        free_cache(c);
        return r;
    }
    *out = c;
    return KVR_OK;
}

kvr_status kvr_destroy_cache(kvr_cache* c) {
    if (!c) return KVR_OK;
    cudaDeviceSynchronize();
    free_cache(c);
    return KVR_OK;
}

kvr_status kvr_select(kvr_cache* c, const int32_t* positions, const int32_t* counts, int32_t budget_percent,
                      const int32_t* token_ids, const void* embed_table, int32_t vocab, const void* hidden_src,
                      void* hidden_out, int32_t* n_rows_out, int32_t* n_intervals_out, void* stream) {
    pdl_begin_call();   // no overlap with work enqueued before this call
    if (!c || !counts) {
        set_error("cache or counts is NULL");
        return KVR_EINVAL;
    }
    const bool use_ids = token_ids || embed_table;
    if (use_ids == (hidden_src != nullptr) || (use_ids && (!token_ids || !embed_table))) {
        set_error("give exactly one row source: token_ids + embed_table, or hidden_src");
        return KVR_EINVAL;
    }
    if (use_ids && vocab < 1) {
        set_error("vocab must be >= 1 with an embedding table");
        return KVR_EINVAL;
    }
    RowSource src;
    src.token_ids = token_ids;
    src.embed = embed_table;
    src.vocab = vocab;
    src.hidden_src = hidden_src;
    return do_select(c, positions, counts, budget_percent, src, hidden_out, n_rows_out, n_intervals_out,
                     reinterpret_cast<cudaStream_t>(stream));
}

kvr_status kvr_reselect(kvr_cache* c, const int32_t* positions, const int32_t* counts, const void* carry_rows,
                        const void* fill_rows, void* hidden_out, int32_t* n_rows_out, int32_t* n_intervals_out,
                        void* stream) {
    pdl_begin_call();   // no overlap with work enqueued before this call
    if (!c || !counts) {
        set_error("cache or counts is NULL");
        return KVR_EINVAL;
    }
    if (!fill_rows || !aligned16(fill_rows) || (c->sel.valid && c->sel.n_rows > 0 && !carry_rows)) {
        set_error("fill_rows (and carry_rows when rows are selected) must be non-NULL and 16-byte aligned");
        return KVR_EINVAL;
    }
    if (carry_rows && carry_rows == hidden_out) {
        set_error("hidden_out must not be the carried rows' buffer (rows move)");
        return KVR_EINVAL;
    }
    RowSource src;
    src.carry = carry_rows ? carry_rows : fill_rows;
    src.fill = fill_rows;
    return do_select(c, positions, counts, -1, src, hidden_out, n_rows_out, n_intervals_out,
                     reinterpret_cast<cudaStream_t>(stream));
}

kvr_status kvr_refresh_interval_wise(kvr_cache* c, const int32_t* positions, const int32_t* counts,
                                     int32_t budget_percent, const int32_t* token_ids, const void* embed_table,
                                     int32_t vocab, const void* hidden_src, const kvr_layer_weights* w,
                                     int32_t layer_begin, int32_t layer_end, void* hidden_out, void* workspace,
                                     size_t ws_bytes, uint32_t flags, int32_t* n_intervals_out, void* stream) {
    pdl_begin_call();   // no overlap with work enqueued before this call
    if (!c || !counts || (!positions && counts)) {
        set_error("cache, positions or counts is NULL");
        return KVR_EINVAL;
    }
    if (layer_begin < 0 || layer_end > c->m.n_layers || layer_begin > layer_end) {
        set_error("layer range outside [0, n_layers]");
        return KVR_ERANGE;
    }
    const int B = c->batch;
    // validate the whole support once (packed selection of everything), which
    // also gives the total rows; then walk sequence by sequence, interval by interval
    int32_t n_rows = 0, n_iv = 0;
    kvr_status st = kvr_select(c, positions, counts, budget_percent, token_ids, embed_table, vocab, hidden_src,
                               hidden_out, &n_rows, &n_iv, stream);
    if (st != KVR_OK) return st;
    if (n_intervals_out) *n_intervals_out = n_iv;
    std::vector<int32_t> sorted;
    std::vector<std::pair<int, int>> ivs;   // (position begin, length) per interval, per sequence
    int64_t off = 0;
    int max_len = 0;
    std::vector<std::vector<std::pair<int, int>>> per_seq(B);
    for (int i = 0; i < B; ++i) {
        sorted.assign(positions + off, positions + off + counts[i]);
        std::sort(sorted.begin(), sorted.end());
        for (size_t k = 0; k < sorted.size(); ++k) {
            if (k == 0 || sorted[k] != sorted[k - 1] + 1) per_seq[i].push_back({sorted[k], 0});
            per_seq[i].back().second += 1;
            max_len = std::max(max_len, per_seq[i].back().second);
        }
        off += counts[i];
    }
    if (n_rows == 0) return KVR_OK;
    if (!workspace || ws_bytes < kvr_workspace_bytes(c, max_len)) {
        set_error("workspace too small: need kvr_workspace_bytes(c, longest interval) = " +
                  std::to_string(kvr_workspace_bytes(c, max_len)) + " bytes");
        return KVR_EINVAL;
    }
    if (!w && layer_end > layer_begin) {
        set_error("weights array is NULL");
        return KVR_EINVAL;
    }
    const size_t row_bytes = (size_t)c->m.d_model * dtype_size(c->m.dtype);
    std::vector<int32_t> cnt(B, 0), pos;
    int row0 = 0;
    for (int i = 0; i < B; ++i) {
        for (const auto& iv : per_seq[i]) {
            pos.resize(iv.second);
            for (int k = 0; k < iv.second; ++k) pos[k] = iv.first + k;
            std::fill(cnt.begin(), cnt.end(), 0);
            cnt[i] = iv.second;
            void* rows_out = static_cast<uint8_t*>(hidden_out) + (size_t)row0 * row_bytes;
            st = kvr_select(c, pos.data(), cnt.data(), -1, token_ids, embed_table, vocab, hidden_src, rows_out,
                            nullptr, nullptr, stream);
            if (st != KVR_OK) return st;
            st = kvr_refresh(c, w, layer_begin, layer_end, rows_out, workspace, ws_bytes, flags, stream);
            if (st != KVR_OK) return st;
            row0 += iv.second;
        }
    }
    return KVR_OK;
}

kvr_status kvr_refresh_range(kvr_cache* c, const kvr_layer_weights* w, int32_t range_begin, int32_t range_end,
                             const int32_t* positions, const int32_t* counts, const int32_t* token_ids,
                             const void* embed_table, int32_t vocab, const void* hidden_src, const void* boundary,
                             void* hidden_sel, void* hidden_full, void* workspace, size_t ws_bytes, uint32_t flags,
                             void* stream) {
    if (!c || !counts) {
        set_error("cache or counts is NULL");
        return KVR_EINVAL;
    }
    if (range_begin < 0 || range_end > c->m.n_layers || range_begin > range_end) {
        set_error("layer range outside [0, n_layers]");
        return KVR_ERANGE;
    }
    const bool ranged = range_end > range_begin;
    if (ranged && (!boundary || !hidden_full)) {
        set_error("a non-empty layer range needs the boundary rows and the hidden_full buffer");
        return KVR_EINVAL;
    }
    const int L = c->m.n_layers;
    kvr_status st = kvr_select(c, positions, counts, -1, token_ids, embed_table, vocab, hidden_src, hidden_sel,
                               nullptr, nullptr, stream);
    if (st != KVR_OK) return st;
    if (!ranged) return kvr_refresh(c, w, 0, L, hidden_sel, workspace, ws_bytes, flags, stream);
    if ((st = kvr_refresh(c, w, 0, range_begin, hidden_sel, workspace, ws_bytes, 0, stream)) != KVR_OK) return st;
    // the whole affected suffix of every sequence, sequence-major
    const int S = c->n_tokens - c->suffix_start;
    std::vector<int32_t> full((size_t)c->batch * S), full_counts(c->batch, S);
    for (int b = 0; b < c->batch; ++b)
        for (int i = 0; i < S; ++i) full[(size_t)b * S + i] = c->suffix_start + i;
    if ((st = kvr_reselect(c, full.data(), full_counts.data(), hidden_sel, boundary, hidden_full, nullptr, nullptr,
                           stream)) != KVR_OK)
        return st;
    if ((st = kvr_refresh(c, w, range_begin, range_end, hidden_full, workspace, ws_bytes, 0, stream)) != KVR_OK)
        return st;
    if ((st = kvr_reselect(c, positions, counts, hidden_full, boundary, hidden_sel, nullptr, nullptr, stream)) !=
        KVR_OK)
        return st;
    return kvr_refresh(c, w, range_end, L, hidden_sel, workspace, ws_bytes, flags, stream);
}

kvr_status kvr_lora_merge(const void* w, void* w_out, int32_t n_out, int32_t K, int32_t row_begin,
                          int32_t row_count, const void* a, const void* b, int32_t rank, float scale, int32_t dtype,
                          void* stream) {
    pdl_begin_call();   // no overlap with work enqueued before this call
    if (!w || !w_out || !a || !b || n_out < 1 || K < 1 || rank < 1 || row_begin < 0 || row_count < 0 ||
        row_begin + row_count > n_out || (dtype != KVR_BF16 && dtype != KVR_F32)) {
        set_error("lora merge: bad arguments");
        return KVR_EINVAL;
    }
    KVR_CHECK_LAUNCH(launch_lora_merge(dtype, w, w_out, n_out, K, row_begin, row_count, a, b, rank, scale,
                                       reinterpret_cast<cudaStream_t>(stream)),
                     "lora merge");
    return KVR_OK;
}

kvr_status kvr_shift(kvr_cache* c, int32_t start, int32_t d, void* stream) {
    pdl_begin_call();   // no overlap with work enqueued before this call
    if (!c) {
        set_error("cache is NULL");
        return KVR_EINVAL;
    }
    if (start < 0 || d < 0 || (int64_t)start + d > c->n_tokens || d == c->n_tokens) {
        set_error("shift: need 0 <= start, 0 <= d, start + d <= n_tokens and d < n_tokens");
        return KVR_EINVAL;
    }
    if (d == 0) return KVR_OK;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const kvr_model_desc& m = c->m;
    MoveLaunch a{};
    a.k_src = c->k_base;
    a.v_src = c->v_base;
    a.k_dst = c->k_base;
    a.v_dst = c->v_base;
    a.src_slab_rows = a.dst_slab_rows = c->capacity;
    a.dst_slab_off = 0;
    a.src_row0 = start + d;
    a.dst_row0 = start;
    a.n_rows = c->n_tokens - start - d;
    a.n_slabs = c->batch * m.n_layers * m.n_kv_heads;
    rotation_table(m, -(double)d, a.cs);
    KVR_CHECK_LAUNCH(launch_move_rows(m.dtype, m.head_dim, a, true, s), "shift rows");
    KVR_CHECK_LAUNCH(launch_shift_bits(c->d_local, c->d_sink, c->batch, c->words, start, d, c->n_tokens, s),
                     "shift metadata");
    c->n_tokens -= d;
    c->suffix_start = std::min(c->suffix_start, start);
    c->sel = Selection{};
    return KVR_OK;
}

kvr_status kvr_splice(kvr_cache* c, int32_t seq, int32_t dst_pos, int32_t n, const void* k_src,
                      const void* v_src, int32_t src_pos, uint32_t flags, void* stream) {
    pdl_begin_call();   // no overlap with work enqueued before this call
    if (!c) {
        set_error("cache is NULL");
        return KVR_EINVAL;
    }
    if (seq < 0 || seq >= c->batch || n < 0 || dst_pos < 0 || src_pos < 0 || (int64_t)dst_pos + n > c->n_tokens) {
        set_error("splice: need 0 <= seq < batch, n >= 0, dst_pos >= 0, src_pos >= 0, dst_pos + n <= n_tokens");
        return KVR_EINVAL;
    }
    if (n == 0) return KVR_OK;
    if (!k_src || !v_src || !aligned16(k_src) || !aligned16(v_src)) {
        set_error("splice: K/V sources must be non-NULL and 16-byte aligned");
        return KVR_EINVAL;
    }
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const kvr_model_desc& m = c->m;
    MoveLaunch a{};
    a.k_src = k_src;
    a.v_src = v_src;
    a.k_dst = c->k_base;
    a.v_dst = c->v_base;
    a.src_slab_rows = n;
    a.dst_slab_rows = c->capacity;
    a.dst_slab_off = (int64_t)seq * m.n_layers * m.n_kv_heads;
    a.src_row0 = 0;
    a.dst_row0 = dst_pos;
    a.n_rows = n;
    a.n_slabs = m.n_layers * m.n_kv_heads;
    rotation_table(m, (double)dst_pos - (double)src_pos, a.cs);
    KVR_CHECK_LAUNCH(launch_move_rows(m.dtype, m.head_dim, a, false, s), "splice rows");
    const size_t off = (size_t)seq * c->words;
    KVR_CHECK_LAUNCH(launch_set_bits(c->d_local + off, c->d_sink + off, dst_pos, n, flags, s), "splice metadata");
    return KVR_OK;
}

kvr_status kvr_cache_info(kvr_cache* c, int32_t* n_tokens, int32_t* suffix_start) {
    if (!c) {
        set_error("cache is NULL");
        return KVR_EINVAL;
    }
    if (n_tokens) *n_tokens = c->n_tokens;
    if (suffix_start) *suffix_start = c->suffix_start;
    return KVR_OK;
}

size_t kvr_workspace_bytes(const kvr_cache* c, int32_t max_rows) {
    if (!c) return 0;
    int R = max_rows > 0 ? max_rows : c->sel.n_rows;
    if (max_rows <= 0) return layout(c->m, R, part_bytes(c->m, R, sel_attn_scratch(c))).total;
    // the projections' split choice changes with the row count: take the
    // largest partial region over every row count up to max_rows (it peaks at
    // row-tile edges); a split attention never uses more than kAttnMaxSplitCTAs
    // CTAs' worth of partials
    const size_t attn = c->m.dtype == KVR_BF16 ? (size_t)kAttnMaxSplitCTAs * 128 * 130 * sizeof(float) : 0;
    const int step = c->m.dtype == KVR_BF16 ? 256 : 64;
    size_t part = 0;
    for (int r = step; r < R + step; r += step) part = std::max(part, part_bytes(c->m, std::min(r, R), attn));
    for (int r = 1; r <= std::min(R, 2 * step); ++r) part = std::max(part, part_bytes(c->m, r, attn));
    return layout(c->m, R, part).total;
}

kvr_status kvr_refresh_layer(kvr_cache* c, int32_t layer, const kvr_layer_weights* w, void* hidden_inout,
                             void* workspace, size_t ws_bytes, uint32_t flags, void* stream) {
    pdl_begin_call();   // no overlap with work enqueued before this call
    WsLayout L;
    kvr_status st = check_refresh_args(c, hidden_inout, workspace, ws_bytes, &L);
    if (st != KVR_OK) return st;
    if (layer < 0 || layer >= c->m.n_layers) {
        set_error("layer " + std::to_string(layer) + " is outside [0, n_layers)");
        return KVR_ERANGE;
    }
    if ((st = check_layer_weights(c, w)) != KVR_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (c->sel.n_rows > 0) {
        st = run_layer(c, layer, w, hidden_inout, static_cast<uint8_t*>(workspace), L, s);
        if (st != KVR_OK) return st;
    }
    if (flags & KVR_COMMIT_META) return commit(c, s);
    return KVR_OK;
}

kvr_status kvr_refresh(kvr_cache* c, const kvr_layer_weights* w, int32_t layer_begin, int32_t layer_end,
                       void* hidden_inout, void* workspace, size_t ws_bytes, uint32_t flags, void* stream) {
    pdl_begin_call();   // no overlap with work enqueued before this call
    WsLayout L;
    kvr_status st = check_refresh_args(c, hidden_inout, workspace, ws_bytes, &L);
    if (st != KVR_OK) return st;
    if (layer_begin < 0 || layer_end > c->m.n_layers || layer_begin > layer_end) {
        set_error("layer range outside [0, n_layers]");
        return KVR_ERANGE;
    }
    if (!w && layer_end > layer_begin) {
        set_error("weights array is NULL");
        return KVR_EINVAL;
    }
    for (int l = layer_begin; l < layer_end; ++l)
        if ((st = check_layer_weights(c, &w[l])) != KVR_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (c->sel.n_rows > 0) {
        for (int l = layer_begin; l < layer_end; ++l) {
            st = run_layer(c, l, &w[l], hidden_inout, static_cast<uint8_t*>(workspace), L, s, l > layer_begin,
                           l + 1 < layer_end ? w[l + 1].norm1 : nullptr);
            if (st != KVR_OK) return st;
        }
    }
    if (flags & KVR_COMMIT_META) return commit(c, s);
    return KVR_OK;
}

kvr_status kvr_attend(kvr_cache* c, int32_t layer, const void* q, void* out, void* workspace, size_t ws_bytes,
                      void* stream) {
    pdl_begin_call();   // no overlap with work enqueued before this call
    if (!c) {
        set_error("cache is NULL");
        return KVR_EINVAL;
    }
    if (!c->sel.valid) {
        set_error("no selection: call kvr_select first");
        return KVR_ESTATE;
    }
    if (layer < 0 || layer >= c->m.n_layers) {
        set_error("layer outside [0, n_layers)");
        return KVR_ERANGE;
    }
    if (c->sel.n_rows == 0) return KVR_OK;
    if (!q || !out || !aligned16(q) || !aligned16(out)) {
        set_error("q and out must be non-NULL and 16-byte aligned");
        return KVR_EINVAL;
    }
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    AttnLaunch a{};
    a.q = q;
    a.out = out;
    a.k_base = c->k_base;
    a.v_base = c->v_base;
    a.U = c->d_U;
    a.plan = c->d_plan;
    a.loc = c->d_local;
    a.snk = c->d_sink;
    a.n_tiles = c->sel.n_tiles;
    a.n_rows = c->sel.n_rows;
    a.n_q_heads = c->m.n_q_heads;
    a.n_kv_heads = c->m.n_kv_heads;
    a.head_dim = c->m.head_dim;
    a.layer = layer;
    a.n_layers = c->m.n_layers;
    a.capacity = c->capacity;
    a.n_tokens = c->n_tokens;
    a.words = c->words;
    a.batch = c->batch;
    a.alpha = c->alpha;
    a.beta = c->beta;
    a.err = c->d_err;
    set_attention_scratch(&a, (workspace && (reinterpret_cast<uintptr_t>(workspace) & 255u) == 0)
                                  ? static_cast<float*>(workspace) : nullptr,
                          ws_bytes, c);
    std::string why;
    Prof p(c, KVR_K_ATTN, s);
    p.launches = attention_launches(c->m.dtype, a);
    cudaError_t e = launch_attention(c->m.dtype, a, s, &why);
    if (e != cudaSuccess) return cuda_fail(e, ("attention " + why).c_str());
    return KVR_OK;
}

kvr_status kvr_wait_check(kvr_cache* c, int64_t cycles, void* stream) {
    pdl_begin_call();
    if (!c) {
        set_error("cache is NULL");
        return KVR_EINVAL;
    }
    if (cycles < 1 || cycles >= (int64_t(1) << 31)) {
        set_error("cycles must be in [1, 2^31)");
        return KVR_EINVAL;
    }
    KVR_CHECK_LAUNCH(launch_wait_check(c->d_err, (long long)cycles, reinterpret_cast<cudaStream_t>(stream)),
                     "wait check");
    return KVR_OK;
}

kvr_status kvr_sync_status(kvr_cache* c, void* stream) {
    if (!c) {
        set_error("cache is NULL");
        return KVR_EINVAL;
    }
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "stream synchronize");
    int32_t w[4] = {0, 0, 0, 0};
    e = cudaMemcpy(w, c->d_err, sizeof(w), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "error word read");
    if (w[0] == 0) return KVR_OK;
    cudaMemset(c->d_err, 0, sizeof(w));
    if (w[0] & DEV_ERR_TIMEOUT) {
        set_error("a device-side wait timed out");
        return KVR_ETIMEOUT;
    }
    set_error(std::string("device-side check failed:") + ((w[0] & DEV_ERR_INDEX) ? " index out of range" : "") +
              ((w[0] & DEV_ERR_DUPLICATE) ? " duplicate position" : ""));
    return KVR_EDEVICE;
}

kvr_status kvr_read_selection(kvr_cache* c, int32_t seq, int32_t* U, int32_t u_cap, int32_t* iv, int32_t iv_cap,
                              uint32_t* sel, uint32_t* eloc, uint32_t* esnk, int32_t* plan, int32_t plan_cap,
                              int32_t* n_tiles, int32_t* rows_per_tile, int32_t* keys_per_tile) {
    if (!c) {
        set_error("cache is NULL");
        return KVR_EINVAL;
    }
    if (!c->sel.valid) {
        set_error("no selection");
        return KVR_ESTATE;
    }
    if (seq < 0 || seq >= c->batch) {
        set_error("sequence index out of range");
        return KVR_ERANGE;
    }
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e, "synchronize");
    const Selection& S = c->sel;
    const size_t wb = (size_t)c->words * sizeof(uint32_t);
    auto cp = [&](void* dst, const void* src, size_t n) {
        if (dst && n && e == cudaSuccess) e = cudaMemcpy(dst, src, n, cudaMemcpyDeviceToHost);
    };
    cp(U, c->d_U + S.row_off[seq], (size_t)std::min(u_cap, S.counts[seq]) * sizeof(int32_t));
    cp(iv, c->d_iv + 2 * (size_t)S.iv_off[seq], (size_t)std::min(iv_cap, S.iv_count[seq]) * 2 * sizeof(int32_t));
    cp(sel, c->d_sel + (size_t)seq * c->words, wb);
    cp(eloc, c->d_eloc + (size_t)seq * c->words, wb);
    cp(esnk, c->d_esnk + (size_t)seq * c->words, wb);
    if (plan) {
        const int nt = std::min(plan_cap, S.tile_count[seq]);
        std::vector<int32_t> p8((size_t)nt * 8);
        cp(p8.data(), c->d_plan + 8 * (size_t)S.tile_off[seq], p8.size() * sizeof(int32_t));
        for (int t = 0; t < nt; ++t) {
            for (int k = 0; k < 6; ++k) plan[6 * t + k] = p8[8 * t + k];
            plan[6 * t] -= S.row_off[seq];
        }
    }
    if (e != cudaSuccess) return cuda_fail(e, "selection read");
    if (n_tiles) *n_tiles = S.tile_count[seq];
    if (rows_per_tile) *rows_per_tile = S.rows_per_tile;
    if (keys_per_tile) *keys_per_tile = S.keys_per_tile;
    return KVR_OK;
}

kvr_status kvr_read_meta(kvr_cache* c, uint32_t* local_bits, uint32_t* sink_bits) {
    if (!c) {
        set_error("cache is NULL");
        return KVR_EINVAL;
    }
    cudaError_t e = cudaDeviceSynchronize();
    const size_t wb = (size_t)c->batch * c->words * sizeof(uint32_t);
    if (e == cudaSuccess && local_bits) e = cudaMemcpy(local_bits, c->d_local, wb, cudaMemcpyDeviceToHost);
    if (e == cudaSuccess && sink_bits) e = cudaMemcpy(sink_bits, c->d_sink, wb, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "metadata read");
    return KVR_OK;
}

kvr_status kvr_profile_enable(kvr_cache* c, int32_t enable) {
    if (!c) {
        set_error("cache is NULL");
        return KVR_EINVAL;
    }
    c->profiling = enable != 0;
    return KVR_OK;
}

kvr_status kvr_profile_read(kvr_cache* c, double* ms, int64_t* launches, int32_t n) {
    if (!c) {
        set_error("cache is NULL");
        return KVR_EINVAL;
    }
    for (auto& r : c->prof) {
        cudaError_t e = cudaEventSynchronize(r.b);
        if (e != cudaSuccess) return cuda_fail(e, "profile event");
        float t = 0.f;
        cudaEventElapsedTime(&t, r.a, r.b);
        c->prof_ms[r.kind] += t;
        c->prof_n[r.kind] += r.launches;
        c->ev_pool.push_back(r.a);
        c->ev_pool.push_back(r.b);
    }
    c->prof.clear();
    for (int k = 0; k < n && k < KVR_K_COUNT; ++k) {
        if (ms) ms[k] = c->prof_ms[k];
        if (launches) launches[k] = c->prof_n[k];
    }
    for (int k = 0; k < KVR_K_COUNT; ++k) {
        c->prof_ms[k] = 0.0;
        c->prof_n[k] = 0;
    }
    return KVR_OK;
}

}  // extern "C"

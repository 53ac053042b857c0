// C ABI entry points: host-side validation, workspace carving and the launch sequence of a
// draft round. Every arithmetic step runs in the kernels of the other translation units.
//
// The launch sequence follows hf2q 0.1.1 spec_decode/dflash/qwen35_orchestrator.rs
// (per-round loop, steps 1-9) for DFlash and models/qwen35/mtp.rs
// (`forward_draft_with_hidden`) for MTP.
#include <algorithm>
#include <atomic>
#include <mutex>
#include <vector>
#include <stdarg.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "df_internal.cuh"

namespace df {

static thread_local char g_err[512] = "";
static std::atomic<uint64_t> g_launches{0};

int fail(int code, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof(g_err), fmt, ap);
    va_end(ap);
    return code;
}

// ---------------------------------------------------------------- launch set-up
int sm_count() {
    static std::atomic<int> cached[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        cudaGetLastError();
        return kDefaultSMs;
    }
    int n = cached[dev].load(std::memory_order_relaxed);
    if (n > 0) return n;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
        cudaGetLastError();
        return kDefaultSMs;
    }
    cached[dev].store(n, std::memory_order_relaxed);
    return n;
}

bool pdl_enabled() {
    static const bool on = [] {
        const char *e = getenv("DF_PDL");
        return !(e && e[0] == '0');
    }();
    return on;
}

void prepare_kernel(const void *func, int dyn_smem) {
    static std::mutex mu;
    static std::vector<std::pair<const void *, int>> done;
    int dev = 0;
    cudaGetDevice(&dev);
    std::lock_guard<std::mutex> lk(mu);
    for (auto &d : done)
        if (d.first == func && d.second == dev) return;
    static const int carveout = [] {
        const char *e = getenv("DF_CARVEOUT");
        return e ? atoi(e) : 100;
    }();
    // The dynamic limit is what the device allows per block minus the kernel's static shared
    // memory (asking for more fails and would leave the 48 KB default in place).
    int optin = 232448;
    cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    cudaFuncAttributes fa{};
    if (cudaFuncGetAttributes(&fa, func) == cudaSuccess) optin -= (int)fa.sharedSizeBytes;
    cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, optin);
    if (carveout >= 0)
        cudaFuncSetAttribute(func, cudaFuncAttributePreferredSharedMemoryCarveout, carveout);
    cudaGetLastError();
    done.emplace_back(func, dev);
    (void)dyn_smem;
}

// ---------------------------------------------------------------- launch profiling
struct Prof {
    std::mutex mu;
    bool on = false;
    int cap = 0, n = 0;
    std::vector<cudaEvent_t> ev;
    std::vector<const char *> names;   // nullptr marks a "before" event
};
static Prof g_prof;

static bool capturing(cudaStream_t s) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &cs) != cudaSuccess) {
        cudaGetLastError();
        return true;
    }
    return cs != cudaStreamCaptureStatusNone;
}

void prof_begin(cudaStream_t s) {
    if (!g_prof.on) return;
    std::lock_guard<std::mutex> lk(g_prof.mu);
    if (!g_prof.on || g_prof.n + 2 > g_prof.cap || capturing(s)) return;
    cudaEventRecord(g_prof.ev[g_prof.n], s);
    g_prof.names[g_prof.n++] = nullptr;
}

int cuda_check(const char *what, cudaStream_t s) {
    g_launches.fetch_add(1, std::memory_order_relaxed);
    cudaError_t e = cudaGetLastError();
    if (g_prof.on) {
        std::lock_guard<std::mutex> lk(g_prof.mu);
        if (g_prof.on && g_prof.n > 0 && g_prof.n < g_prof.cap &&
            g_prof.names[g_prof.n - 1] == nullptr) {
            cudaEventRecord(g_prof.ev[g_prof.n], s);
            g_prof.names[g_prof.n++] = what;
        }
    }
    if (e != cudaSuccess) return fail(DF_ECUDA, "%s: %s", what, cudaGetErrorString(e));
    return DF_OK;
}

namespace {


bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

#define REQ(cond, code, ...)                         \
    do {                                             \
        if (!(cond)) return fail(code, __VA_ARGS__); \
    } while (0)

int check_bf16(const void *p, const char *name) {
    REQ(p != nullptr, DF_EINVAL, "%s is NULL", name);
    REQ(aligned16(p), DF_EINVAL, "%s is not 16-byte aligned", name);
    return DF_OK;
}

int check_f32(const void *p, const char *name) {
    REQ(p != nullptr, DF_EINVAL, "%s is NULL", name);
    REQ((reinterpret_cast<uintptr_t>(p) & 3u) == 0, DF_EINVAL, "%s is not 4-byte aligned", name);
    return DF_OK;
}

int check_cfg(const df_dflash_config *c) {
    REQ(c, DF_EINVAL, "config is NULL");
    REQ(c->hidden > 0 && c->hidden % 8 == 0, DF_ESHAPE, "hidden=%d must be a positive multiple of 8",
        c->hidden);
    REQ(c->n_layers > 0, DF_ESHAPE, "n_layers=%d", c->n_layers);
    REQ(c->n_q_heads > 0 && c->n_kv_heads > 0 && c->n_q_heads % c->n_kv_heads == 0, DF_ESHAPE,
        "n_q_heads=%d must be a positive multiple of n_kv_heads=%d", c->n_q_heads, c->n_kv_heads);
    REQ(c->head_dim >= 32 && c->head_dim <= 256 && c->head_dim % 32 == 0, DF_ESHAPE,
        "head_dim=%d must be a multiple of 32 in [32, 256]", c->head_dim);
    int rot = c->rotary_dim ? c->rotary_dim : c->head_dim;
    REQ(rot > 0 && rot <= c->head_dim && rot % 2 == 0, DF_ESHAPE, "rotary_dim=%d", c->rotary_dim);
    REQ(c->intermediate > 0 && c->intermediate % 8 == 0, DF_ESHAPE, "intermediate=%d",
        c->intermediate);
    REQ(c->vocab > 1, DF_ESHAPE, "vocab=%d", c->vocab);
    REQ(c->n_target_layers > 0, DF_ESHAPE, "n_target_layers=%d", c->n_target_layers);
    REQ((long long)c->n_target_layers * c->hidden < (1LL << 30), DF_ESHAPE, "fc input too wide");
    REQ(c->mask_token_id >= 0 && c->mask_token_id < c->vocab, DF_EINVAL,
        "mask_token_id=%d outside [0, vocab)", c->mask_token_id);
    REQ(c->causal_block == 0 || c->causal_block == 1, DF_EINVAL, "causal_block=%d", c->causal_block);
    REQ(c->rms_eps >= 0.f && c->rope_theta > 0.f, DF_EINVAL, "rms_eps / rope_theta");
    REQ(c->kv_bf16 == 0 || c->kv_bf16 == 1, DF_EINVAL, "kv_bf16=%d", c->kv_bf16);
    REQ(!c->kv_bf16 || c->head_dim == 128 || c->head_dim == 256, DF_ESHAPE,
        "a BF16 KV cache needs head_dim 128 or 256 (head_dim=%d)", c->head_dim);
    return DF_OK;
}

int check_weights(const df_dflash_config *c, const df_dflash_weights *w) {
    REQ(w, DF_EINVAL, "weights is NULL");
    DF_TRY(check_bf16(w->fc, "fc"));
    DF_TRY(check_f32(w->hidden_norm, "hidden_norm"));
    DF_TRY(check_f32(w->final_norm, "final_norm"));
    DF_TRY(check_bf16(w->embed, "embed"));
    DF_TRY(check_bf16(w->lm_head, "lm_head"));
    REQ(w->layers, DF_EINVAL, "layers is NULL");
    for (int l = 0; l < c->n_layers; ++l) {
        const df_layer_weights &L = w->layers[l];
        DF_TRY(check_f32(L.input_norm, "input_norm"));
        DF_TRY(check_f32(L.post_attn_norm, "post_attn_norm"));
        DF_TRY(check_f32(L.q_norm, "q_norm"));
        DF_TRY(check_f32(L.k_norm, "k_norm"));
        DF_TRY(check_bf16(L.wq, "wq"));
        DF_TRY(check_bf16(L.wk, "wk"));
        DF_TRY(check_bf16(L.wv, "wv"));
        DF_TRY(check_bf16(L.wo, "wo"));
        DF_TRY(check_bf16(L.w_gate, "w_gate"));
        DF_TRY(check_bf16(L.w_up, "w_up"));
        DF_TRY(check_bf16(L.w_down, "w_down"));
    }
    return DF_OK;
}

int check_cache(const df_kv_cache *k, int n_layers, int B, int d) {
    REQ(k, DF_EINVAL, "cache is NULL");
    REQ(k->n_layers == n_layers, DF_ESHAPE, "cache has %d layers, expected %d", k->n_layers,
        n_layers);
    REQ(k->batch == B, DF_ESHAPE, "cache batch %d != B %d", k->batch, B);
    REQ(k->cap > 0, DF_ESHAPE, "cache cap=%d", k->cap);
    REQ(k->k && k->v && k->seq_len, DF_EINVAL, "cache arrays are NULL");
    for (int l = 0; l < n_layers; ++l) {
        REQ(k->k[l] && k->v[l], DF_EINVAL, "cache layer %d is NULL", l);
        REQ(aligned16(k->k[l]) && aligned16(k->v[l]), DF_EINVAL, "cache layer %d misaligned", l);
    }
    (void)d;
    return DF_OK;
}

// ---------------------------------------------------------------- DFlash workspace
struct DFlashWs {
    float *h, *defer, *q, *kb, *vb, *cos_t, *sin_t, *attn_part, *h_final;
    float *ss_in, *ss_post;   // slice sums of squares of the deferred input / post-attention norms
    int ss_slots;             // slots per row of ss_in / ss_post (one per 128-column tile of H)
    size_t defer_floats;
    uint16_t *xp_ctx, *xp_qkv, *xp_o, *xp_ffn, *xp_act, *xp_head;
    ArgTop *amax_part;
    int32_t *idx;
    AttnArgs plan;
    TcScratch tc;
};

// Room for the split partial sums of a projection with N outputs over T tokens: the splits S
// satisfy S * ceil(N / 128) <= SMs, so S * N < (SMs + S) * 128.
size_t defer_floats_for(int T, long long N) {
    return (size_t)T * (size_t)(2 * (size_t)sm_count() * 128 + N);
}

// ctas: the projection grid (every SM by default).
void carve_tc(Carve &cv, TcScratch &tc, int max_tokens, long long max_rows, int ctas = 0) {
    tc.max_ctas = ctas > 0 ? ctas : sm_count();
    tc.partial_floats = tc_partial_floats(max_tokens, tc.max_ctas);
    tc.partials = cv.take<float>(tc.partial_floats);
    tc.n_counters = n_counters_for(max_rows);
    tc.counters = cv.take<int>((size_t)tc.n_counters);
}

// Argmax partials of an lm_head over `rows` rows: one per (projection CTA, row).
size_t argmax_parts(int rows) { return (size_t)sm_count() * (size_t)rows; }

void carve_dflash(Carve &cv, DFlashWs &w, const df_dflash_config *c, int B, int blk, int n_new_max,
                  int cap, bool round) {
    const int H = c->hidden, d = c->head_dim, nq = c->n_q_heads, nkv = c->n_kv_heads;
    const int rot = c->rotary_dim ? c->rotary_dim : d;
    const size_t T_blk = (size_t)B * blk, T_ctx = (size_t)B * n_new_max, T_all = T_blk + T_ctx;
    const size_t fc_in = (size_t)c->n_target_layers * H, qt = (size_t)nq * d, kt = (size_t)nkv * d;
    w.h = cv.take<float>(T_blk * H);
    w.ss_slots = std::max((H + 127) / 128, pack_slices(H));
    w.ss_in = cv.take<float>(T_all * (size_t)w.ss_slots);   // block rows, then context rows
    w.ss_post = cv.take<float>(T_blk * (size_t)w.ss_slots);
    // deferred split-K sums of one projection: S x T x N floats with S * N <= SMs * 128
    w.defer_floats = defer_floats_for((int)T_all, (long long)std::max<size_t>(qt + 2 * kt, H));
    w.defer = cv.take<float>(w.defer_floats);
    w.q = cv.take<float>(T_blk * qt);
    w.kb = cv.take<float>(T_blk * kt);
    w.vb = cv.take<float>(T_blk * kt);
    w.cos_t = cv.take<float>((size_t)B * (blk + n_new_max) * (rot / 2));
    w.sin_t = cv.take<float>((size_t)B * (blk + n_new_max) * (rot / 2));
    w.plan = AttnArgs{};
    w.plan.B = B;
    w.plan.blk = blk;
    w.plan.nq = nq;
    w.plan.nkv = nkv;
    w.plan.d = d;
    attn_plan(w.plan, cap + blk);
    w.attn_part = cv.take<float>(attn_part_floats(w.plan));
    w.xp_ctx = cv.take<uint16_t>(2 * std::max<size_t>(T_ctx, 1) * fc_in);
    w.xp_qkv = cv.take<uint16_t>(2 * T_all * H);
    w.xp_o = cv.take<uint16_t>(2 * T_blk * qt);
    w.xp_ffn = cv.take<uint16_t>(2 * T_blk * H);
    w.xp_act = cv.take<uint16_t>(2 * T_blk * c->intermediate);
    {
        long long rows = std::max<long long>({(long long)c->vocab, 2LL * c->intermediate,
                                              (long long)(qt + 2 * kt), (long long)H});
        carve_tc(cv, w.tc, (int)T_all, rows);
    }
    w.h_final = nullptr;   // the round defers the final norm to the lm_head (no h_final)
    if (round) {
        w.xp_head = cv.take<uint16_t>(2 * T_blk * H);
        w.amax_part = cv.take<ArgTop>(argmax_parts((int)T_blk));
    } else {
        w.xp_head = nullptr;
        w.amax_part = nullptr;
    }
}

int get_ws(void *ws, size_t ws_bytes, size_t need) {
    REQ(ws != nullptr, DF_EWORKSPACE, "workspace is NULL (need %zu bytes)", need);
    REQ((reinterpret_cast<uintptr_t>(ws) & 255u) == 0, DF_EWORKSPACE,
        "workspace is not 256-byte aligned");
    REQ(ws_bytes >= need, DF_EWORKSPACE, "workspace of %zu bytes is smaller than %zu", ws_bytes,
        need);
    return DF_OK;
}

// The drafter forward. Either block_ids or (last_token, mask id) provides the block tokens.
// ------------------------------------------------------------------ projection weights
// The weight operand (matrices, segments, K split, SwiGLU pairing) of each DFlash projection,
// shared by the forward and by the tiling of the weights; the forward adds activations,
// epilogue and outputs. Without weights (sizing from the config alone) the matrices are stand-in
// pointers that are never read.
enum DfProj { DP_FC, DP_QKV, DP_O, DP_GATE_UP, DP_DOWN, DP_LM_HEAD };

GemmArgs dflash_proj(const df_dflash_config *c, const df_dflash_weights *W, int layer, int which) {
    static const uint16_t kStandIn[8] = {};
    const uint16_t *z = kStandIn;
    const int H = c->hidden, qt = c->n_q_heads * c->head_dim, kt = c->n_kv_heads * c->head_dim;
    const df_layer_weights *L = (W && layer >= 0) ? &W->layers[layer] : nullptr;
    GemmArgs g;
    switch (which) {
        case DP_FC:
            g.W0 = W ? W->fc : z;
            g.n0 = H;
            g.N = H;
            g.K = c->n_target_layers * H;
            break;
        case DP_QKV:
            g.W0 = L ? L->wq : z;
            g.n0 = qt;
            g.W1 = L ? L->wk : z;
            g.n1 = kt;
            g.W2 = L ? L->wv : z;
            g.n2 = kt;
            g.N = qt + 2 * kt;
            g.K = H;
            break;
        case DP_O:
            g.W0 = L ? L->wo : z;
            g.n0 = H;
            g.N = H;
            g.K = qt;
            break;
        case DP_GATE_UP:
            g.W0 = L ? L->w_gate : z;
            g.n0 = c->intermediate;
            g.W1 = L ? L->w_up : z;
            g.n1 = c->intermediate;
            g.N = c->intermediate;
            g.K = H;
            g.epi = EPI_SWIGLU;
            break;
        case DP_DOWN:
            g.W0 = L ? L->w_down : z;
            g.n0 = H;
            g.N = H;
            g.K = c->intermediate;
            break;
        default:   // DP_LM_HEAD
            g.W0 = W ? W->lm_head : z;
            g.n0 = c->vocab;
            g.N = c->vocab;
            g.K = H;
            break;
    }
    return g;
}

// Tiled layout of a DFlash model's weights: fc, then per layer QKV, O, gate/up, down, then the
// lm_head, each projection's tiles starting on a 1024-byte boundary. Projection i of that order
// (i = 0 fc, 1 + 4 l + j layer l's j-th, 1 + 4 n_layers the lm_head) starts at the returned
// offset; i = 2 + 4 n_layers gives the total.
size_t dflash_tiled_offset(const df_dflash_config *c, int i) {
    size_t off = 0;
    for (int k = 0; k < i; ++k) {
        const int layer = k == 0 ? -1 : (k - 1) / 4;
        const int which = k == 0 ? DP_FC : (k == 1 + 4 * c->n_layers ? DP_LM_HEAD : DP_QKV + (k - 1) % 4);
        const size_t b = tiled_projection_bytes(dflash_proj(c, nullptr, k == 1 + 4 * c->n_layers ? -1 : layer, which));
        off += (b + 1023) & ~size_t(1023);
    }
    return off;
}

// The tiled operand of projection `which` of `layer` when the weights carry a tiled copy.
const uint8_t *dflash_tiled(const df_dflash_config *c, const df_dflash_weights *W, int layer,
                            int which) {
    if (!W || !W->tiled) return nullptr;
    const int i = which == DP_FC ? 0 : which == DP_LM_HEAD ? 1 + 4 * c->n_layers
                                                           : 1 + 4 * layer + (which - DP_QKV);
    return static_cast<const uint8_t *>(W->tiled) + dflash_tiled_offset(c, i);
}

// fc, QKV, O and down projections leave split-K partial sums that the next kernel adds in
// (hidden_norm pack, q/k-norm + RoPE, fused residual + RMSNorm pack); gate/up writes packed
// SwiGLU activations directly. The input and post-attention RMSNorms are deferred: their row
// prologue packs x * w and per-slice sums of squares, and the QKV (block rows) and gate/up
// projections multiply their outputs by 1/rms.
int dflash_forward_impl(const df_dflash_config *c, const df_dflash_weights *W,
                        const df_kv_cache *cache, const int32_t *block_ids,
                        const int32_t *last_token, const float *target_hidden,
                        const int32_t *n_new, int n_new_max, int B, int blk, float *h_final,
                        uint16_t *final_pack, DFlashWs &ws, int32_t *st, cudaStream_t s) {
    const int H = c->hidden, d = c->head_dim, nq = c->n_q_heads, nkv = c->n_kv_heads;
    const int rot = c->rotary_dim ? c->rotary_dim : d;
    const int I = c->intermediate;
    const int T_blk = B * blk, T_ctx = B * n_new_max, T_all = T_blk + T_ctx;
    const int fc_in = c->n_target_layers * H, qt = nq * d, kt = nkv * d, Nqkv = qt + 2 * kt;
    REQ(!c->kv_bf16 || attn_tc_supported(d, blk * (nq / nkv)), DF_ESHAPE,
        "a BF16 KV cache needs at most 32 query rows per KV head (block %d x %d)", blk, nq / nkv);

    // A projection whose split partial sums land in ws.defer; returns the split count.
    auto deferred = [&](GemmArgs g, int T, int N, const char *name, int *S) -> int {
        g.epi = EPI_STORE;
        g.defer = 1;
        g.out = ws.defer;
        g.ldo = N;
        g.part_stride = (size_t)T * N;
        g.status = st;
        g.name = name;
        return launch_gemm_tc(g, ws.tc, s, S);
    };

    DF_TRY(launch_rope_table(ws.cos_t, ws.sin_t, cache->seq_len, n_new, n_new_max, B, blk, 0, rot,
                             c->rope_theta, st, s));
    if (T_ctx > 0) {
        // Context stream: h_ctx = rmsnorm(X_new fc^T) * hidden_norm, packed after the block rows
        // with the norm deferred (x * hidden_norm packed, 1/rms applied by every layer's QKV
        // projection from the sums of squares stored after the block rows' ones).
        PackArgs p;
        p.src = target_hidden;
        p.lds = fc_in;
        p.pack = ws.xp_ctx;
        p.ldp = fc_in;
        p.T = T_ctx;
        p.K = fc_in;
        p.nvalid = n_new;
        p.rows_per_seq = n_new_max;
        p.status = st;
        DF_TRY(launch_pack(p, s));
        GemmArgs g = dflash_proj(c, W, -1, DP_FC);
        g.At = dflash_tiled(c, W, -1, DP_FC);
        g.X = ws.xp_ctx;
        g.ldx = fc_in;
        g.T = T_ctx;
        int S = 0;
        DF_TRY(deferred(g, T_ctx, H, "gemm_fc", &S));
        PackArgs q;
        q.part = ws.defer;
        q.n_part = S;
        q.part_stride = (size_t)T_ctx * H;
        q.ldpart = H;
        q.norm_w = W->hidden_norm;
        q.eps = c->rms_eps;
        q.pack = ws.xp_qkv + (size_t)2 * T_blk * H;
        q.ldp = H;
        q.T = T_ctx;
        q.K = H;
        q.nvalid = n_new;
        q.rows_per_seq = n_new_max;
        q.ss_out = ws.ss_in + (size_t)T_blk * ws.ss_slots;
        q.ss_ld = ws.ss_slots;
        q.status = st;
        DF_TRY(launch_pack(q, s));
    }
    int S_down = 0;   // split count of the previous layer's down projection
    for (int l = 0; l < c->n_layers; ++l) {
        const df_layer_weights &L = W->layers[l];
        PackArgs p;
        if (l == 0) {
            p.gather = W->embed;
            p.ids = block_ids;
            p.last_token = last_token;
            p.mask_id = c->mask_token_id;
            p.vocab = c->vocab;
            p.scale = c->embed_scale;
            p.rows_per_seq = blk;
        } else {
            // h += down-projection partials of layer l-1, then input RMSNorm of layer l
            p.src = ws.h;
            p.lds = H;
            p.part = ws.defer;
            p.n_part = S_down;
            p.part_stride = (size_t)T_blk * H;
            p.ldpart = H;
        }
        p.h_out = ws.h;
        p.ldh = H;
        p.norm_w = L.input_norm;
        p.eps = c->rms_eps;
        p.pack = ws.xp_qkv;
        p.ldp = H;
        p.T = T_blk;
        p.K = H;
        p.ss_out = ws.ss_in;
        p.ss_ld = ws.ss_slots;
        p.status = st;
        DF_TRY(launch_pack(p, s));
        // 1/rms of a deferred norm as the row scale of the projection that consumes it
        auto row_scale = [&](GemmArgs &g, const float *ss) {
            g.rs_ss = ss;
            g.rs_n = ws.ss_slots;
            g.rs_rows = T_blk;
            g.rs_inv_k = 1.f / (float)H;
            g.rs_eps = c->rms_eps;
        };

        GemmArgs g = dflash_proj(c, W, l, DP_QKV);
        g.At = dflash_tiled(c, W, l, DP_QKV);
        g.X = ws.xp_qkv;
        g.ldx = H;
        g.T = T_all;
        row_scale(g, ws.ss_in);
        g.rs_rows = T_all;   // the context rows' deferred hidden norm as well
        int S_qkv = 0;
        DF_TRY(deferred(g, T_all, Nqkv, "gemm_qkv", &S_qkv));

        QkArgs qa;
        qa.qkv = nullptr;
        qa.part = ws.defer;
        qa.n_part = S_qkv;
        qa.part_stride = (size_t)T_all * Nqkv;
        qa.ldq = Nqkv;
        qa.B = B;
        qa.blk = blk;
        qa.n_new_max = n_new_max;
        qa.nq = nq;
        qa.nkv = nkv;
        qa.d = d;
        qa.rot = rot;
        qa.q_norm = L.q_norm;
        qa.k_norm = L.k_norm;
        qa.eps = c->rms_eps;
        qa.cos_t = ws.cos_t;
        qa.sin_t = ws.sin_t;
        qa.q_out = ws.q;
        qa.kb = ws.kb;
        qa.vb = ws.vb;
        qa.cache_k = cache->k[l];
        qa.cache_v = cache->v[l];
        qa.cap = cache->cap;
        qa.seq_len = cache->seq_len;
        qa.n_new = n_new;
        qa.append_block = 0;
        qa.pos_off = 0;
        qa.status = st;
        qa.kv_bf16 = c->kv_bf16 ? 1 : 0;
        DF_TRY(launch_qk_rope(qa, s));

        AttnArgs at = ws.plan;
        at.q = ws.q;
        at.cache_k = cache->k[l];
        at.cache_v = cache->v[l];
        at.cap = cache->cap;
        at.kb = ws.kb;
        at.vb = ws.vb;
        at.seq_len = cache->seq_len;
        at.n_new = n_new;
        at.n_new_max = n_new_max;
        at.extra_rows = 0;
        at.causal_block = c->causal_block;
        at.part = ws.attn_part;
        at.gate = nullptr;
        at.ldg = 0;
        at.pack = ws.xp_o;
        at.status = st;
        at.kv_bf16 = c->kv_bf16 ? 1 : 0;
        at.early_kv = 1;   // seq_len moves only at the end of the forward
        DF_TRY(launch_attn(at, s));

        GemmArgs go = dflash_proj(c, W, l, DP_O);
        go.At = dflash_tiled(c, W, l, DP_O);
        go.X = ws.xp_o;
        go.ldx = qt;
        go.T = T_blk;
        {
            // h += O-projection partials (fused residual add), then post-attention RMSNorm
            int S_o = 0;
            DF_TRY(deferred(go, T_blk, H, "gemm_o", &S_o));
            PackArgs pf;
            pf.src = ws.h;
            pf.lds = H;
            pf.part = ws.defer;
            pf.n_part = S_o;
            pf.part_stride = (size_t)T_blk * H;
            pf.ldpart = H;
            pf.h_out = ws.h;
            pf.ldh = H;
            pf.norm_w = L.post_attn_norm;
            pf.eps = c->rms_eps;
            pf.pack = ws.xp_ffn;
            pf.ldp = H;
            pf.T = T_blk;
            pf.K = H;
            pf.ss_out = ws.ss_post;
            pf.ss_ld = ws.ss_slots;
            pf.status = st;
            DF_TRY(launch_pack(pf, s));
        }

        GemmArgs gu = dflash_proj(c, W, l, DP_GATE_UP);
        gu.At = dflash_tiled(c, W, l, DP_GATE_UP);
        gu.X = ws.xp_ffn;
        gu.ldx = H;
        gu.T = T_blk;
        gu.epi = EPI_SWIGLU;
        gu.pack_out = ws.xp_act;
        gu.ldpo = I;
        gu.status = st;
        gu.name = "gemm_gate_up";
        row_scale(gu, ws.ss_post);

        GemmArgs gd = dflash_proj(c, W, l, DP_DOWN);
        gd.At = dflash_tiled(c, W, l, DP_DOWN);
        gd.X = ws.xp_act;
        gd.ldx = I;
        gd.T = T_blk;
        DF_TRY(launch_gemm_tc(gu, ws.tc, s));
        DF_TRY(deferred(gd, T_blk, H, "gemm_down", &S_down));
    }
    // h += last down-projection partials, then the final norm
    PackArgs pfin;
    pfin.src = ws.h;
    pfin.lds = H;
    pfin.part = ws.defer;
    pfin.n_part = S_down;
    pfin.part_stride = (size_t)T_blk * H;
    pfin.ldpart = H;
    pfin.norm_w = W->final_norm;
    pfin.eps = c->rms_eps;
    pfin.y_out = h_final;
    pfin.ldy = H;
    pfin.pack = final_pack;
    // Without h_final (the draft round) the final norm is deferred to the lm_head: x * final_norm
    // is packed, its sums of squares reuse the post-attention ones (the last gate/up has read them)
    if (!h_final) {
        pfin.ss_out = ws.ss_post;
        pfin.ss_ld = ws.ss_slots;
    }
    pfin.ldp = H;
    pfin.T = T_blk;
    pfin.K = H;
    pfin.status = st;
    // the drafter cache advances by n_new here: the last layer's kernels have read seq_len
    pfin.adv_seq = cache->seq_len;
    pfin.adv_n = n_new;
    pfin.adv_B = B;
    pfin.adv_cap = cache->cap;
    return launch_pack(pfin, s);
}

// rs_ss: the packed rows carry a deferred RMSNorm (slice sums of squares, as the row prologue
// writes them); the logits are scaled by 1/rms per row before the argmax.
// The lm_head projection with the running-argmax epilogue; G receives the number of partial
// states per row it leaves in `part`.
int lm_head_gemm(const uint16_t *Wlm, const uint16_t *xp, int rows, int H, int V, ArgTop *part,
                 const TcScratch &tc, cudaStream_t s, const float *rs_ss, float rs_eps, int rs_n,
                 int *G, const uint8_t *At = nullptr) {
    GemmArgs g;
    g.W0 = Wlm;
    g.At = At;
    g.n0 = V;
    g.N = V;
    g.K = H;
    g.X = xp;
    g.ldx = H;
    g.T = rows;
    g.epi = EPI_ARGMAX;
    g.part = part;
    g.name = "gemm_lm_head_argmax";
    if (rs_ss) {
        g.rs_ss = rs_ss;
        g.rs_n = rs_n > 0 ? rs_n : pack_slices(H);
        g.rs_rows = rows;
        g.rs_inv_k = 1.f / (float)H;
        g.rs_eps = rs_eps;
    }
    return launch_gemm_tc(g, tc, s, G);
}

int lm_head_impl(const uint16_t *Wlm, const uint16_t *xp, int rows, int H, int V, ArgTop *part,
                 int32_t *idx, float *top1, float *top2, const TcScratch &tc, cudaStream_t s,
                 const float *rs_ss = nullptr, float rs_eps = 0.f, int rs_n = 0,
                 const uint8_t *At = nullptr) {
    GemmArgs g;
    g.W0 = Wlm;
    g.At = At;
    g.n0 = V;
    g.N = V;
    g.K = H;
    g.X = xp;
    g.ldx = H;
    g.T = rows;
    g.epi = EPI_ARGMAX;
    g.part = part;
    g.name = "gemm_lm_head_argmax";
    if (rs_ss) {
        g.rs_ss = rs_ss;
        g.rs_n = rs_n > 0 ? rs_n : pack_slices(H);
        g.rs_rows = rows;
        g.rs_inv_k = 1.f / (float)H;
        g.rs_eps = rs_eps;
    }
    int G = 0;
    DF_TRY(launch_gemm_tc(g, tc, s, &G));
    return launch_argmax_final(part, G, rows, idx, top1, top2, nullptr, 1, 0, s);
}

// FNV-1a over bytes: the key of a cached graph (every argument it bakes in).
uint64_t fnv(uint64_t h, const void *p, size_t n) {
    const unsigned char *c = static_cast<const unsigned char *>(p);
    for (size_t i = 0; i < n; ++i) h = (h ^ c[i]) * 1099511628211ull;
    return h;
}

// Executable graphs of the host-buffer round entry, least recently used evicted past kMax.
struct HostRoundGraphs {
    static constexpr int kMax = 16;
    struct Entry {
        uint64_t key, used;
        cudaGraph_t graph;
        cudaGraphExec_t exec;
    };
    std::mutex mu;
    std::vector<Entry> entries;
    uint64_t tick = 0;
    cudaStream_t cap = nullptr;
};
HostRoundGraphs g_host_graphs;

// Launches on `user` the graph captured from enqueue(capture stream) for this key, capturing and
// instantiating it on first use.
template <class F>
int host_round_graph(uint64_t key, F &&enqueue, cudaStream_t user) {
    HostRoundGraphs &hg = g_host_graphs;
    std::lock_guard<std::mutex> lk(hg.mu);
    ++hg.tick;
    cudaGraphExec_t ex = nullptr;
    for (auto &en : hg.entries)
        if (en.key == key) {
            en.used = hg.tick;
            ex = en.exec;
        }
    if (!ex) {
        if (!hg.cap) {
            cudaError_t e = cudaStreamCreateWithFlags(&hg.cap, cudaStreamNonBlocking);
            if (e != cudaSuccess) return fail(DF_ECUDA, "capture stream: %s", cudaGetErrorString(e));
        }
        cudaError_t e = cudaStreamBeginCapture(hg.cap, cudaStreamCaptureModeThreadLocal);
        if (e != cudaSuccess) return fail(DF_ECUDA, "host round capture: %s", cudaGetErrorString(e));
        const int rc = enqueue(hg.cap);
        cudaGraph_t g = nullptr;
        e = cudaStreamEndCapture(hg.cap, &g);
        if (rc != DF_OK || e != cudaSuccess) {
            if (g) cudaGraphDestroy(g);
            return rc != DF_OK ? rc : fail(DF_ECUDA, "host round capture: %s", cudaGetErrorString(e));
        }
        e = cudaGraphInstantiate(&ex, g, 0);
        if (e != cudaSuccess) {
            cudaGraphDestroy(g);
            return fail(DF_ECUDA, "host round graph instantiate: %s", cudaGetErrorString(e));
        }
        if ((int)hg.entries.size() >= HostRoundGraphs::kMax) {
            size_t lru = 0;
            for (size_t i = 1; i < hg.entries.size(); ++i)
                if (hg.entries[i].used < hg.entries[lru].used) lru = i;
            cudaGraphExecDestroy(hg.entries[lru].exec);
            cudaGraphDestroy(hg.entries[lru].graph);
            hg.entries.erase(hg.entries.begin() + (long)lru);
        }
        hg.entries.push_back({key, hg.tick, g, ex});
    }
    const cudaError_t e = cudaGraphLaunch(ex, user);
    if (e != cudaSuccess) return fail(DF_ECUDA, "host round graph launch: %s", cudaGetErrorString(e));
    return DF_OK;
}

}  // namespace
}  // namespace df

using namespace df;

#if DF_TRACE
namespace df {
__device__ TraceRec g_trace[kTraceMax];
__device__ unsigned g_trace_n;
}  // namespace df
#endif

extern "C" {

int df_trace_reset(void) {
#if DF_TRACE
    const unsigned zero = 0;
    cudaError_t e = cudaMemcpyToSymbol(df::g_trace_n, &zero, sizeof(zero));
    if (e != cudaSuccess) return fail(DF_ECUDA, "df_trace_reset: %s", cudaGetErrorString(e));
    return DF_OK;
#else
    return fail(DF_EINVAL, "df_trace_reset: this library is not a trace build");
#endif
}

int df_trace_read(uint32_t *kid, uint32_t *sm, unsigned long long *t0, unsigned long long *t1,
                  int max_records) {
#if DF_TRACE
    if (!kid || !sm || !t0 || !t1 || max_records < 0)
        return fail(DF_EINVAL, "df_trace_read: NULL output");
    cudaError_t e = cudaDeviceSynchronize();
    unsigned n = 0;
    if (e == cudaSuccess) e = cudaMemcpyFromSymbol(&n, df::g_trace_n, sizeof(n));
    if (e != cudaSuccess) return fail(DF_ECUDA, "df_trace_read: %s", cudaGetErrorString(e));
    n = std::min<unsigned>(std::min(n, kTraceMax), (unsigned)max_records);
    std::vector<TraceRec> rec(n);
    if (n) e = cudaMemcpyFromSymbol(rec.data(), df::g_trace, sizeof(TraceRec) * n);
    if (e != cudaSuccess) return fail(DF_ECUDA, "df_trace_read: %s", cudaGetErrorString(e));
    for (unsigned i = 0; i < n; ++i) {
        kid[i] = rec[i].kid;
        sm[i] = rec[i].sm;
        t0[i] = rec[i].t0;
        t1[i] = rec[i].t1;
    }
    return (int)n;
#else
    (void)kid, (void)sm, (void)t0, (void)t1, (void)max_records;
    return fail(DF_EINVAL, "df_trace_read: this library is not a trace build");
#endif
}

const char *df_last_error(void) { return g_err; }

int df_version(void) { return 100; }

uint64_t df_kernel_launches(void) { return g_launches.load(std::memory_order_relaxed); }

int df_profile_enable(int on) {
    g_err[0] = 0;
    std::lock_guard<std::mutex> lk(g_prof.mu);
    if (on && g_prof.ev.empty()) {
        g_prof.cap = 8192;
        g_prof.ev.resize(g_prof.cap);
        g_prof.names.resize(g_prof.cap);
        for (auto &e : g_prof.ev)
            if (cudaEventCreate(&e) != cudaSuccess)
                return fail(DF_ECUDA, "profiling events: %s", cudaGetErrorString(cudaGetLastError()));
    }
    g_prof.n = 0;
    g_prof.on = on != 0;
    return DF_OK;
}

int df_profile_read(float *us, int max_entries, char *names, size_t names_bytes) {
    std::lock_guard<std::mutex> lk(g_prof.mu);
    if (g_prof.n == 0) return 0;
    if (cudaEventSynchronize(g_prof.ev[g_prof.n - 1]) != cudaSuccess)
        return fail(DF_ECUDA, "profiling sync: %s", cudaGetErrorString(cudaGetLastError()));
    int k = 0;
    size_t off = 0;
    if (names && names_bytes) names[0] = 0;
    for (int i = 1; i < g_prof.n && k < max_entries; ++i) {
        if (g_prof.names[i] == nullptr || g_prof.names[i - 1] != nullptr) continue;
        float ms = 0.f;
        cudaEventElapsedTime(&ms, g_prof.ev[i - 1], g_prof.ev[i]);
        if (us) us[k] = ms * 1000.f;
        if (names && off < names_bytes) {
            int w = snprintf(names + off, names_bytes - off, "%s\n", g_prof.names[i]);
            off += w > 0 ? (size_t)w : 0;
        }
        ++k;
    }
    return k;
}

size_t df_dflash_tiled_bytes(const df_dflash_config *cfg) {
    if (check_cfg(cfg) != DF_OK) return 0;
    g_err[0] = 0;
    return dflash_tiled_offset(cfg, 2 + 4 * cfg->n_layers);
}

int df_dflash_tile_weights(const df_dflash_config *cfg, const df_dflash_weights *w, void *tiled,
                           size_t tiled_bytes, df_stream_t stream) {
    g_err[0] = 0;
    DF_TRY(check_cfg(cfg));
    DF_TRY(check_weights(cfg, w));
    const size_t need = dflash_tiled_offset(cfg, 2 + 4 * cfg->n_layers);
    REQ(tiled && tiled_bytes >= need, DF_EWORKSPACE, "tiled weights need %zu bytes, have %zu",
        need, tiled_bytes);
    REQ((reinterpret_cast<uintptr_t>(tiled) & 1023u) == 0, DF_EINVAL,
        "tiled weights must be 1024-byte aligned");
    uint8_t *base = static_cast<uint8_t *>(tiled);
    cudaStream_t s = (cudaStream_t)stream;
    for (int i = 0; i < 2 + 4 * cfg->n_layers; ++i) {
        const bool lm = i == 1 + 4 * cfg->n_layers;
        const int layer = (i == 0 || lm) ? -1 : (i - 1) / 4;
        const int which = i == 0 ? DP_FC : lm ? DP_LM_HEAD : DP_QKV + (i - 1) % 4;
        const size_t off = dflash_tiled_offset(cfg, i), end = dflash_tiled_offset(cfg, i + 1);
        DF_TRY(tile_projection(dflash_proj(cfg, w, layer, which), base + off, end - off, s));
    }
    return DF_OK;
}

size_t df_tiled_matrix_bytes(int N, int K) {
    if (N <= 0 || K <= 0) return 0;
    GemmArgs g;
    g.W0 = reinterpret_cast<const uint16_t *>(&g);   // shape only
    g.n0 = N;
    g.N = N;
    g.K = K;
    return tiled_projection_bytes(g);
}

int df_tile_matrix(const uint16_t *W, int N, int K, void *tiled, size_t tiled_bytes,
                   df_stream_t stream) {
    g_err[0] = 0;
    REQ(N > 0 && K > 0 && K % 8 == 0, DF_ESHAPE, "N=%d K=%d (K a multiple of 8)", N, K);
    DF_TRY(check_bf16(W, "W"));
    GemmArgs g;
    g.W0 = W;
    g.n0 = N;
    g.N = N;
    g.K = K;
    return tile_projection(g, static_cast<uint8_t *>(tiled), tiled_bytes, (cudaStream_t)stream);
}

int lm_head_argmax_tiled(const void *W_tiled, const float *X, int rows, int H, int V,
                         int32_t *idx, float *top1, float *top2, void *ws, size_t ws_bytes,
                         df_stream_t stream) {
    g_err[0] = 0;
    REQ(rows > 0 && rows <= kMaxTcTokens && H > 0 && H % 8 == 0 && V > 0, DF_ESHAPE,
        "rows=%d (1..%d) H=%d V=%d (H %% 8 == 0)", rows, kMaxTcTokens, H, V);
    REQ(W_tiled && (reinterpret_cast<uintptr_t>(W_tiled) & 1023u) == 0, DF_EINVAL,
        "W_tiled is NULL or not 1024-byte aligned");
    DF_TRY(check_f32(X, "X"));
    REQ(idx, DF_EINVAL, "idx is NULL");
    DF_TRY(get_ws(ws, ws_bytes, df_lm_head_workspace_bytes(rows, H, V)));
    Carve cv{static_cast<char *>(ws), 0, ws_bytes, true};
    const int ctas = sm_count();
    uint16_t *xp = cv.take<uint16_t>((size_t)2 * rows * H);
    ArgTop *part = cv.take<ArgTop>((size_t)ctas * rows);
    TcScratch tc;
    carve_tc(cv, tc, rows, V, ctas);
    cudaStream_t s = (cudaStream_t)stream;
    PackArgs p;
    p.src = X;
    p.lds = H;
    p.pack = xp;
    p.ldp = H;
    p.T = rows;
    p.K = H;
    DF_TRY(launch_pack(p, s));
    // the row-major pointer only describes the shape when the tiled copy is given
    return lm_head_impl(static_cast<const uint16_t *>(W_tiled), xp, rows, H, V, part, idx, top1,
                        top2, tc, s, nullptr, 0.f, 0, static_cast<const uint8_t *>(W_tiled));
}

size_t df_dflash_workspace_bytes(const df_dflash_config *cfg, int B, int block, int n_new_max) {
    if (check_cfg(cfg) != DF_OK || B <= 0 || block < 2 || n_new_max < 0) return 0;
    // The attention partials depend on the cache capacity; size for the largest plan.
    Carve cv{nullptr, 0, ~size_t(0), true};
    DFlashWs w;
    carve_dflash(cv, w, cfg, B, block, n_new_max, 1 << 20, true);
    return cv.off;
}

int dflash_block_forward(const df_dflash_config *cfg, const df_dflash_weights *w,
                         const df_kv_cache *cache, const int32_t *block_ids,
                         const float *target_hidden_new, const int32_t *n_new, int n_new_max,
                         int B, int block, float *h_final, void *ws, size_t ws_bytes,
                         int32_t *d_status, df_stream_t stream) {
    g_err[0] = 0;
    DF_TRY(check_cfg(cfg));
    DF_TRY(check_weights(cfg, w));
    REQ(B > 0 && block >= 2, DF_ESHAPE, "B=%d, block=%d (block must be >= 2)", B, block);
    REQ(n_new_max >= 0, DF_ESHAPE, "n_new_max=%d", n_new_max);
    DF_TRY(check_cache(cache, cfg->n_layers, B, cfg->head_dim));
    REQ(block_ids && h_final, DF_EINVAL, "block_ids / h_final is NULL");
    REQ(n_new_max == 0 || (target_hidden_new && n_new), DF_EINVAL,
        "target_hidden_new / n_new is NULL");
    REQ(n_new_max <= cache->cap, DF_ECAPACITY, "n_new_max=%d exceeds cap=%d", n_new_max, cache->cap);
    size_t need = df_dflash_workspace_bytes(cfg, B, block, n_new_max);
    DF_TRY(get_ws(ws, ws_bytes, need));
    Carve cv{static_cast<char *>(ws), 0, ws_bytes, true};
    DFlashWs W;
    carve_dflash(cv, W, cfg, B, block, n_new_max, cache->cap, false);
    return dflash_forward_impl(cfg, w, cache, block_ids, nullptr, target_hidden_new, n_new,
                               n_new_max, B, block, h_final, nullptr, W, d_status,
                               (cudaStream_t)stream);
}

size_t df_lm_head_workspace_bytes(int rows, int H, int V) {
    if (rows <= 0 || H <= 0 || V <= 0) return 0;
    if (rows > kMaxTcTokens) return 0;
    return lm_head_scratch_bytes_for(rows, H, V, sm_count());
}

int lm_head_argmax(const uint16_t *W, const float *X, int rows, int H, int V, int32_t *idx,
                   float *top1, float *top2, void *ws, size_t ws_bytes, df_stream_t stream) {
    g_err[0] = 0;
    REQ(rows > 0 && rows <= kMaxTcTokens && H > 0 && H % 8 == 0 && V > 0, DF_ESHAPE,
        "rows=%d (1..%d) H=%d V=%d (H %% 8 == 0)", rows, kMaxTcTokens, H, V);
    DF_TRY(check_bf16(W, "W"));
    DF_TRY(check_f32(X, "X"));
    REQ(idx, DF_EINVAL, "idx is NULL");
    DF_TRY(get_ws(ws, ws_bytes, df_lm_head_workspace_bytes(rows, H, V)));
    Carve cv{static_cast<char *>(ws), 0, ws_bytes, true};
    const int ctas = sm_count();
    uint16_t *xp = cv.take<uint16_t>((size_t)2 * rows * H);
    ArgTop *part = cv.take<ArgTop>((size_t)ctas * rows);
    TcScratch tc;
    carve_tc(cv, tc, rows, V, ctas);
    cudaStream_t s = (cudaStream_t)stream;
    PackArgs p;
    p.src = X;
    p.lds = H;
    p.pack = xp;
    p.ldp = H;
    p.T = rows;
    p.K = H;
    DF_TRY(launch_pack(p, s));
    return lm_head_impl(W, xp, rows, H, V, part, idx, top1, top2, tc, s);
}

size_t df_linear_workspace_bytes(int T, int N, int K) {
    if (T <= 0 || N <= 0 || K <= 0) return 0;
    Carve cv{nullptr, 0, ~size_t(0), true};
    cv.take<uint16_t>((size_t)2 * T * K);
    TcScratch tc;
    carve_tc(cv, tc, T, N);
    return cv.off;
}

int df_linear(const uint16_t *W, const float *X, int T, int N, int K, float *Y, void *ws,
              size_t ws_bytes, df_stream_t stream) {
    g_err[0] = 0;
    REQ(T > 0 && N > 0 && K > 0 && K % 8 == 0, DF_ESHAPE, "T=%d N=%d K=%d (K %% 8 == 0)", T, N, K);
    DF_TRY(check_bf16(W, "W"));
    DF_TRY(check_f32(X, "X"));
    DF_TRY(check_f32(Y, "Y"));
    DF_TRY(get_ws(ws, ws_bytes, df_linear_workspace_bytes(T, N, K)));
    Carve cv{static_cast<char *>(ws), 0, ws_bytes, true};
    uint16_t *xp = cv.take<uint16_t>((size_t)2 * T * K);
    TcScratch tc;
    carve_tc(cv, tc, T, N);
    cudaStream_t s = (cudaStream_t)stream;
    PackArgs p;
    p.src = X;
    p.lds = K;
    p.pack = xp;
    p.ldp = K;
    p.T = T;
    p.K = K;
    DF_TRY(launch_pack(p, s));
    GemmArgs g;
    g.W0 = W;
    g.n0 = N;
    g.N = N;
    g.K = K;
    g.X = xp;
    g.ldx = K;
    g.T = T;
    g.epi = EPI_STORE;
    g.out = Y;
    g.ldo = N;
    return launch_gemm_tc(g, tc, s);
}

// The attention plan of df_attention: key chunks sized for cap cache rows (+ the block rows).
static AttnArgs attention_plan(int B, int blk, int nq, int nkv, int d, int cap, bool block_keys) {
    AttnArgs a = AttnArgs{};
    a.B = B;
    a.blk = blk;
    a.nq = nq;
    a.nkv = nkv;
    a.d = d;
    attn_plan(a, cap + (block_keys ? blk : 0));
    return a;
}

static int check_attention(int B, int blk, int nq, int nkv, int d, int cap) {
    REQ(B > 0 && blk > 0 && cap > 0, DF_ESHAPE, "B=%d blk=%d cap=%d", B, blk, cap);
    REQ(nq > 0 && nkv > 0 && nq % nkv == 0, DF_ESHAPE, "heads %d / %d", nq, nkv);
    REQ(d == 32 || d == 64 || d == 128 || d == 256, DF_ESHAPE, "head_dim=%d not in {32, 64, 128, 256}", d);
    return DF_OK;
}

size_t df_attention_workspace_bytes(int B, int blk, int nq, int nkv, int d, int cap) {
    if (check_attention(B, blk, nq, nkv, d, cap) != DF_OK) return 0;
    AttnArgs a = attention_plan(B, blk, nq, nkv, d, cap, true);
    Carve cv{nullptr, 0, ~size_t(0), true};
    cv.take<float>(attn_part_floats(a));
    return cv.off;
}

int df_attention(const float *q, const float *cache_k, const float *cache_v, int cap,
                 const int32_t *seq_len, const float *kb, const float *vb, int B, int blk, int nq,
                 int nkv, int d, int causal_block, float *out, void *ws, size_t ws_bytes,
                 int32_t *d_status, df_stream_t stream) {
    g_err[0] = 0;
    DF_TRY(check_attention(B, blk, nq, nkv, d, cap));
    REQ(q && cache_k && cache_v && seq_len && out, DF_EINVAL, "df_attention: NULL q, cache, seq_len or out");
    REQ((kb == nullptr) == (vb == nullptr), DF_EINVAL, "df_attention: kb and vb go together");
    DF_TRY(check_bf16(q, "q"));                 // 16-byte alignment (vector and bulk copies)
    DF_TRY(check_bf16(cache_k, "cache_k"));
    DF_TRY(check_bf16(cache_v, "cache_v"));
    if (kb) {
        DF_TRY(check_bf16(kb, "kb"));
        DF_TRY(check_bf16(vb, "vb"));
    }
    DF_TRY(check_f32(out, "out"));
    DF_TRY(get_ws(ws, ws_bytes, df_attention_workspace_bytes(B, blk, nq, nkv, d, cap)));
    AttnArgs a = attention_plan(B, blk, nq, nkv, d, cap, kb != nullptr);
    a.q = q;
    a.cache_k = cache_k;
    a.cache_v = cache_v;
    a.cap = cap;
    a.kb = kb;
    a.vb = vb;
    a.seq_len = seq_len;
    a.causal_block = causal_block ? 1 : 0;
    a.part = static_cast<float *>(ws);
    a.out = out;
    a.status = d_status;
    return launch_attn(a, (cudaStream_t)stream);
}

size_t df_accept_stochastic_workspace_bytes(int B, int K, int V) {
    if (B <= 0 || K < 1 || K > kSampleMaxK || V <= 0 || V % 4 != 0) return 0;
    Carve cv{nullptr, 0, ~size_t(0), true};
    SampleArgs a;
    carve_sample_scratch(cv, a, B, K, V);
    return cv.off;
}

int accept_stochastic(const float *draft_logits, const float *target_logits, int V,
                      const int32_t *drafts, int B, int K, float temperature,
                      const float *u_accept, const float *u_sample, const int32_t *eos, int n_eos,
                      int32_t *committed, int32_t *n_committed, int32_t *accept_count,
                      int32_t *hit_eos, int32_t *rollback, void *ws, size_t ws_bytes,
                      int32_t *d_status, df_stream_t stream) {
    g_err[0] = 0;
    REQ(B > 0 && K >= 1 && K <= 64, DF_ESHAPE, "B=%d K=%d (1 <= K <= 64)", B, K);
    REQ(V > 0 && V % 4 == 0, DF_ESHAPE, "V=%d (a positive multiple of 4)", V);
    REQ(temperature > 0.f, DF_EINVAL, "temperature=%g (the greedy walk is accept_prefix_argmax)",
        (double)temperature);
    REQ(draft_logits && target_logits && drafts && u_accept && u_sample && committed &&
            n_committed && accept_count && hit_eos && rollback,
        DF_EINVAL, "NULL input or output");
    REQ(n_eos >= 0 && (n_eos == 0 || eos), DF_EINVAL, "eos is NULL with n_eos=%d", n_eos);
    DF_TRY(check_bf16(draft_logits, "draft_logits"));      // 16-byte alignment
    DF_TRY(check_bf16(target_logits, "target_logits"));
    DF_TRY(get_ws(ws, ws_bytes, df_accept_stochastic_workspace_bytes(B, K, V)));
    SampleArgs a;
    Carve cv{static_cast<char *>(ws), 0, ws_bytes, true};
    carve_sample_scratch(cv, a, B, K, V);
    a.draft = draft_logits;
    a.draft_ld = K;
    a.target = target_logits;
    a.V = V;
    a.B = B;
    a.K = K;
    a.T = temperature;
    sample_constants(a);
    a.drafts = drafts;
    a.u_accept = u_accept;
    a.u_sample = u_sample;
    a.eos = eos;
    a.n_eos = n_eos;
    a.committed = committed;
    a.n_committed = n_committed;
    a.accept_count = accept_count;
    a.hit_eos = hit_eos;
    a.rollback = rollback;
    a.status = d_status;
    return launch_accept_stochastic(a, (cudaStream_t)stream);
}

size_t df_sample_softmax_workspace_bytes(int R, int V) {
    if (R <= 0 || V <= 0 || V % 4 != 0) return 0;
    Carve cv{nullptr, 0, ~size_t(0), true};
    SampleArgs a;
    carve_sample_scratch(cv, a, R, 1, V);
    return cv.off;
}

int sample_softmax(const float *logits, int R, int V, float temperature, const float *u,
                   int32_t *tokens, void *ws, size_t ws_bytes, int32_t *d_status,
                   df_stream_t stream) {
    g_err[0] = 0;
    REQ(R > 0, DF_ESHAPE, "R=%d", R);
    REQ(V > 0 && V % 4 == 0, DF_ESHAPE, "V=%d (a positive multiple of 4)", V);
    REQ(temperature > 0.f, DF_EINVAL, "temperature=%g (temperature 0 is the argmax)",
        (double)temperature);
    REQ(logits && u && tokens, DF_EINVAL, "NULL input or output");
    DF_TRY(check_bf16(logits, "logits"));      // 16-byte alignment
    DF_TRY(get_ws(ws, ws_bytes, df_sample_softmax_workspace_bytes(R, V)));
    SampleArgs a;
    Carve cv{static_cast<char *>(ws), 0, ws_bytes, true};
    carve_sample_scratch(cv, a, R, 1, V);
    a.draft = logits;
    a.draft_ld = 1;
    a.V = V;
    a.B = R;
    a.K = 1;
    a.T = temperature;
    sample_constants(a);
    a.sample_mode = 1;
    a.u_draft = u;
    a.drafts_out = tokens;
    a.status = d_status;
    return launch_sample_drafts(a, (cudaStream_t)stream);
}

int accept_prefix_argmax(const int32_t *drafts, int drafts_ld, const int32_t *target, int B,
                         int K, const int32_t *eos, int n_eos, int32_t *committed,
                         int32_t *n_committed, int32_t *accept_count, int32_t *hit_eos,
                         int32_t *rollback, df_stream_t stream) {
    g_err[0] = 0;
    REQ(B > 0 && K >= 1, DF_ESHAPE, "B=%d K=%d (K >= 1)", B, K);
    REQ(drafts_ld >= K, DF_ESHAPE, "drafts_ld=%d < K=%d", drafts_ld, K);
    REQ(n_eos >= 0 && (n_eos == 0 || eos), DF_EINVAL, "eos list");
    REQ(drafts && target && committed && n_committed && accept_count && hit_eos && rollback,
        DF_EINVAL, "NULL output or input");
    return launch_accept(drafts, drafts_ld, target, B, K, eos, n_eos, committed, n_committed,
                         accept_count, hit_eos, rollback, nullptr, nullptr, (cudaStream_t)stream);
}

int accept_prefix_argmax_host(const int32_t *drafts, const int32_t *target, int K,
                              const int32_t *eos, int n_eos, int32_t *committed,
                              int32_t *n_committed, int32_t *accept_count, int32_t *hit_eos,
                              int32_t *rollback) {
    g_err[0] = 0;
    REQ(K >= 1, DF_ESHAPE, "K=%d (K >= 1)", K);
    REQ(n_eos >= 0 && (n_eos == 0 || eos), DF_EINVAL, "eos list");
    REQ(drafts && target && committed && n_committed && accept_count && hit_eos && rollback,
        DF_EINVAL, "NULL output or input");
    int a = 0;
    while (a < K && drafts[a] == target[a]) ++a;
    int n = 0, hit = 0;
    for (int i = 0; i <= a; ++i) {
        int tok = i < a ? drafts[i] : target[a];
        committed[n++] = tok;
        bool is_eos = false;
        for (int e = 0; e < n_eos; ++e) is_eos |= (tok == eos[e]);
        if (is_eos) {
            hit = 1;
            break;
        }
    }
    for (int i = n; i <= K; ++i) committed[i] = -1;
    *n_committed = n;
    *accept_count = a;
    *hit_eos = hit;
    *rollback = K - a;
    return DF_OK;
}

int kv_rollback(int32_t *seq_len, const int32_t *n, int B, int32_t *d_status, df_stream_t stream) {
    g_err[0] = 0;
    REQ(B > 0, DF_ESHAPE, "B=%d", B);
    REQ(seq_len && n, DF_EINVAL, "seq_len / n is NULL");
    return launch_rollback(seq_len, n, B, d_status, (cudaStream_t)stream);
}

int df_draft_round(const df_dflash_config *cfg, const df_dflash_weights *w,
                   const df_kv_cache *cache, const int32_t *last_token,
                   const float *target_hidden_new, const int32_t *n_new, int n_new_max, int B,
                   int K, const int32_t *target_argmax, const int32_t *eos, int n_eos,
                   int32_t *target_seq_len, int32_t *argmax_out, int32_t *committed,
                   int32_t *n_committed, int32_t *accept_count, int32_t *hit_eos,
                   int32_t *rollback, void *ws, size_t ws_bytes, int32_t *d_status,
                   df_stream_t stream) {
    g_err[0] = 0;
    DF_TRY(check_cfg(cfg));
    DF_TRY(check_weights(cfg, w));
    REQ(B > 0 && K >= 1, DF_ESHAPE, "B=%d K=%d (K >= 1)", B, K);
    const int blk = K + 1;
    REQ(n_new_max >= 0 && n_new_max <= (cache ? cache->cap : 0), DF_ESHAPE, "n_new_max=%d",
        n_new_max);
    DF_TRY(check_cache(cache, cfg->n_layers, B, cfg->head_dim));
    REQ(last_token && target_argmax && target_seq_len && argmax_out && committed && n_committed &&
            accept_count && hit_eos && rollback,
        DF_EINVAL, "NULL round input or output");
    REQ(n_new_max == 0 || (target_hidden_new && n_new), DF_EINVAL,
        "target_hidden_new / n_new is NULL");
    REQ(n_eos >= 0 && (n_eos == 0 || eos), DF_EINVAL, "eos list");
    size_t need = df_dflash_workspace_bytes(cfg, B, blk, n_new_max);
    DF_TRY(get_ws(ws, ws_bytes, need));
    Carve cv{static_cast<char *>(ws), 0, ws_bytes, true};
    DFlashWs W;
    carve_dflash(cv, W, cfg, B, blk, n_new_max, cache->cap, true);
    cudaStream_t s = (cudaStream_t)stream;
    DF_TRY(dflash_forward_impl(cfg, w, cache, nullptr, last_token, target_hidden_new, n_new,
                               n_new_max, B, blk, W.h_final, W.xp_head, W, d_status, s));
    if (blk > 32) {
        DF_TRY(lm_head_impl(w->lm_head, W.xp_head, B * blk, cfg->hidden, cfg->vocab, W.amax_part,
                            argmax_out, nullptr, nullptr, W.tc, s, W.ss_post, cfg->rms_eps,
                            W.ss_slots, dflash_tiled(cfg, w, -1, DP_LM_HEAD)));
        return launch_accept(argmax_out + 1, blk, target_argmax, B, K, eos, n_eos, committed,
                             n_committed, accept_count, hit_eos, rollback, target_seq_len,
                             d_status, s);
    }
    // the lm_head's argmax partials, then the argmax merge and the accept walk in one launch
    int G = 0;
    DF_TRY(lm_head_gemm(w->lm_head, W.xp_head, B * blk, cfg->hidden, cfg->vocab, W.amax_part,
                        W.tc, s, W.ss_post, cfg->rms_eps, W.ss_slots, &G,
                        dflash_tiled(cfg, w, -1, DP_LM_HEAD)));
    return launch_argmax_accept(W.amax_part, G, B, blk, argmax_out, target_argmax, eos, n_eos,
                                committed, n_committed, accept_count, hit_eos, rollback,
                                target_seq_len, d_status, s);
}

size_t df_draft_round_stochastic_workspace_bytes(const df_dflash_config *cfg, int B, int K,
                                                 int n_new_max) {
    if (check_cfg(cfg) != DF_OK || B <= 0 || K < 1 || K > kSampleMaxK || n_new_max < 0 ||
        cfg->vocab % 4 != 0)
        return 0;
    Carve cv{nullptr, 0, ~size_t(0), true};
    DFlashWs w;
    carve_dflash(cv, w, cfg, B, K + 1, n_new_max, 1 << 20, true);
    SampleArgs a;
    carve_sample_scratch(cv, a, B, K, cfg->vocab);
    return cv.off;
}

int df_draft_round_stochastic(const df_dflash_config *cfg, const df_dflash_weights *w,
                              const df_kv_cache *cache, const int32_t *last_token,
                              const float *target_hidden_new, const int32_t *n_new,
                              int n_new_max, int B, int K, const float *target_logits,
                              float temperature, const float *u_draft, const float *u_accept,
                              const float *u_sample, const int32_t *eos, int n_eos,
                              int32_t *target_seq_len, float *logits_out, int32_t *drafts_out,
                              int32_t *committed, int32_t *n_committed, int32_t *accept_count,
                              int32_t *hit_eos, int32_t *rollback, void *ws, size_t ws_bytes,
                              int32_t *d_status, df_stream_t stream) {
    g_err[0] = 0;
    DF_TRY(check_cfg(cfg));
    DF_TRY(check_weights(cfg, w));
    REQ(B > 0 && K >= 1 && K <= kSampleMaxK, DF_ESHAPE, "B=%d K=%d (1 <= K <= %d)", B, K,
        kSampleMaxK);
    REQ(cfg->vocab % 4 == 0, DF_ESHAPE, "vocab=%d (a multiple of 4)", cfg->vocab);
    REQ(temperature > 0.f, DF_EINVAL, "temperature=%g (temperature 0 is df_draft_round)",
        (double)temperature);
    const int blk = K + 1;
    REQ(n_new_max >= 0 && n_new_max <= (cache ? cache->cap : 0), DF_ESHAPE, "n_new_max=%d",
        n_new_max);
    DF_TRY(check_cache(cache, cfg->n_layers, B, cfg->head_dim));
    REQ(last_token && target_logits && u_draft && u_accept && u_sample && target_seq_len &&
            logits_out && drafts_out && committed && n_committed && accept_count && hit_eos &&
            rollback,
        DF_EINVAL, "NULL round input or output");
    REQ(n_new_max == 0 || (target_hidden_new && n_new), DF_EINVAL,
        "target_hidden_new / n_new is NULL");
    REQ(n_eos >= 0 && (n_eos == 0 || eos), DF_EINVAL, "eos list");
    DF_TRY(check_f32(target_logits, "target_logits"));
    DF_TRY(check_f32(logits_out, "logits_out"));
    DF_TRY(get_ws(ws, ws_bytes, df_draft_round_stochastic_workspace_bytes(cfg, B, K, n_new_max)));
    Carve cv{static_cast<char *>(ws), 0, ws_bytes, true};
    DFlashWs W;
    carve_dflash(cv, W, cfg, B, blk, n_new_max, cache->cap, true);
    SampleArgs a;
    carve_sample_scratch(cv, a, B, K, cfg->vocab);
    cudaStream_t s = (cudaStream_t)stream;
    const int H = cfg->hidden, V = cfg->vocab;
    DF_TRY(dflash_forward_impl(cfg, w, cache, nullptr, last_token, target_hidden_new, n_new,
                               n_new_max, B, blk, W.h_final, W.xp_head, W, d_status, s));
    // logits of every block row (final norm deferred to the row scale, as in the greedy round)
    GemmArgs gl = dflash_proj(cfg, w, -1, DP_LM_HEAD);
    gl.At = dflash_tiled(cfg, w, -1, DP_LM_HEAD);
    gl.X = W.xp_head;
    gl.ldx = H;
    gl.T = B * blk;
    gl.epi = EPI_STORE;
    gl.out = logits_out;
    gl.ldo = V;
    gl.status = d_status;
    gl.name = "gemm_lm_head_logits";
    gl.rs_ss = W.ss_post;
    gl.rs_n = W.ss_slots;
    gl.rs_rows = B * blk;
    gl.rs_inv_k = 1.f / (float)H;
    gl.rs_eps = cfg->rms_eps;
    DF_TRY(launch_gemm_tc(gl, W.tc, s));
    // drafts i = 1..K drawn from softmax(logits / T), then the accept step
    a.draft = logits_out + V;
    a.draft_ld = blk;
    a.target = target_logits;
    a.V = V;
    a.B = B;
    a.K = K;
    a.T = temperature;
    sample_constants(a);
    a.sample_mode = 1;
    a.u_draft = u_draft;
    a.drafts_out = drafts_out;
    a.status = d_status;
    DF_TRY(launch_sample_drafts(a, s));
    a.sample_mode = 0;
    a.drafts = drafts_out;
    a.u_accept = u_accept;
    a.u_sample = u_sample;
    a.eos = eos;
    a.n_eos = n_eos;
    a.committed = committed;
    a.n_committed = n_committed;
    a.accept_count = accept_count;
    a.hit_eos = hit_eos;
    a.rollback = rollback;
    DF_TRY(launch_accept_stochastic(a, s));
    return launch_rollback(target_seq_len, rollback, B, d_status, s);
}

size_t df_draft_round_host_workspace_bytes(const df_dflash_config *cfg, int B, int K,
                                           int n_new_max, int n_eos) {
    if (check_cfg(cfg) != DF_OK || B <= 0 || K < 1 || n_new_max < 0 || n_eos < 0) return 0;
    Carve cv{nullptr, 0, ~size_t(0), true};
    const size_t fc_in = (size_t)cfg->n_target_layers * cfg->hidden;
    cv.take<float>((size_t)B * std::max(n_new_max, 1) * fc_in);   // target hidden rows
    cv.take<int32_t>((size_t)B * 9 * (K + 2) + n_eos + 8);         // ints in and out
    return cv.off;
}

int df_draft_round_host(const df_dflash_config *cfg, const df_dflash_weights *w,
                        const df_kv_cache *cache, const int32_t *last_token,
                        const float *target_hidden_new, const int32_t *n_new, int n_new_max,
                        int B, int K, const int32_t *target_argmax, const int32_t *eos,
                        int n_eos, int32_t *target_seq_len, int32_t *argmax_out,
                        int32_t *committed, int32_t *n_committed, int32_t *accept_count,
                        int32_t *hit_eos, int32_t *rollback, int32_t *status, void *ws,
                        size_t ws_bytes, df_stream_t stream) {
    g_err[0] = 0;
    DF_TRY(check_cfg(cfg));
    REQ(B > 0 && K >= 1 && n_new_max >= 0 && n_eos >= 0, DF_ESHAPE, "B=%d K=%d n_new_max=%d", B,
        K, n_new_max);
    REQ(last_token && target_argmax && target_seq_len && argmax_out && committed && n_committed &&
            accept_count && hit_eos && rollback && status,
        DF_EINVAL, "NULL host buffer");
    REQ(n_new_max == 0 || (target_hidden_new && n_new), DF_EINVAL, "target_hidden_new / n_new");
    const int blk = K + 1;
    size_t need_round = df_dflash_workspace_bytes(cfg, B, blk, n_new_max);
    size_t need_stage = df_draft_round_host_workspace_bytes(cfg, B, K, n_new_max, n_eos);
    DF_TRY(get_ws(ws, ws_bytes, need_round + need_stage));
    char *stage = static_cast<char *>(ws) + need_round;
    Carve cv{stage, 0, need_stage, true};
    const size_t fc_in = (size_t)cfg->n_target_layers * cfg->hidden;
    float *d_th = cv.take<float>((size_t)B * std::max(n_new_max, 1) * fc_in);
    int32_t *ip = cv.take<int32_t>((size_t)B * 9 * (K + 2) + n_eos + 8);
    int32_t *d_last = ip;
    int32_t *d_nnew = d_last + B;
    int32_t *d_tgt = d_nnew + B;
    int32_t *d_tsl = d_tgt + (size_t)B * blk;
    int32_t *d_am = d_tsl + B;
    int32_t *d_com = d_am + (size_t)B * blk;
    int32_t *d_nc = d_com + (size_t)B * blk;
    int32_t *d_ac = d_nc + B;
    int32_t *d_he = d_ac + B;
    int32_t *d_rb = d_he + B;
    int32_t *d_eos = d_rb + B;
    int32_t *d_st = d_eos + n_eos;
    cudaStream_t user = (cudaStream_t)stream;
    // Device addresses of the host buffers when they are page-locked and mapped (else null).
    const void *host_bufs[] = {last_token, target_hidden_new, n_new, target_argmax, eos,
                               target_seq_len, argmax_out, committed, n_committed, accept_count,
                               hit_eos, rollback, status};
    constexpr int kBufs = (int)(sizeof(host_bufs) / sizeof(host_bufs[0]));
    void *dev_of[kBufs] = {};
    bool pinned = true;
    for (int i = 0; i < kBufs; ++i) {
        if (!host_bufs[i]) continue;
        cudaPointerAttributes pa{};
        if (cudaPointerGetAttributes(&pa, host_bufs[i]) != cudaSuccess ||
            pa.type != cudaMemoryTypeHost || pa.devicePointer == nullptr) {
            pinned = false;
            cudaGetLastError();
            break;
        }
        dev_of[i] = pa.devicePointer;
    }
    // Graph form: the small inputs and all outputs by one word-copy kernel each, the target rows
    // read by the round's first kernel, all straight from and to the mapped host buffers.
    auto enqueue_mapped = [&](cudaStream_t s) -> int {
        WordCopyList in;
        auto add = [](WordCopyList &l, const void *src, void *dst, long long words) {   // src null: zeros
            if (words <= 0) return;
            l.src[l.n] = src;
            l.dst[l.n] = dst;
            l.words[l.n] = (int)words;
            ++l.n;
        };
        add(in, dev_of[0], d_last, B);
        if (n_new_max > 0) add(in, dev_of[2], d_nnew, B);
        add(in, dev_of[3], d_tgt, (long long)B * blk);
        add(in, dev_of[4], d_eos, n_eos);
        add(in, dev_of[5], d_tsl, B);
        add(in, nullptr, d_st, 1);   // the status word starts at DF_OK
        DF_TRY(launch_word_copy(in, s));
        // the row prologue reads the new target rows straight from the mapped host buffer
        DF_TRY(df_draft_round(cfg, w, cache, d_last,
                              n_new_max ? static_cast<const float *>(dev_of[1]) : nullptr,
                              n_new_max ? d_nnew : nullptr, n_new_max, B, K, d_tgt, d_eos, n_eos,
                              d_tsl, d_am, d_com, d_nc, d_ac, d_he, d_rb, ws, need_round, d_st,
                              (df_stream_t)s));
        WordCopyList out;
        add(out, d_tsl, dev_of[5], B);
        add(out, d_am, dev_of[6], (long long)B * blk);
        add(out, d_com, dev_of[7], (long long)B * blk);
        add(out, d_nc, dev_of[8], B);
        add(out, d_ac, dev_of[9], B);
        add(out, d_he, dev_of[10], B);
        add(out, d_rb, dev_of[11], B);
        add(out, d_st, dev_of[12], 1);
        return launch_word_copy(out, s);
    };
    // Stream form: copies in, the round, copies out.
    auto enqueue = [&](cudaStream_t s) -> int {
        auto h2d = [&](void *dst, const void *src, size_t bytes) {
            return bytes ? cudaMemcpyAsync(dst, src, bytes, cudaMemcpyHostToDevice, s) : cudaSuccess;
        };
        auto d2h = [&](void *dst, const void *src, size_t bytes) {
            return bytes ? cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDeviceToHost, s) : cudaSuccess;
        };
        cudaError_t e = cudaSuccess;
        e = e ? e : h2d(d_last, last_token, sizeof(int32_t) * B);
        if (n_new_max > 0) {
            e = e ? e : h2d(d_th, target_hidden_new, sizeof(float) * B * n_new_max * fc_in);
            e = e ? e : h2d(d_nnew, n_new, sizeof(int32_t) * B);
        }
        e = e ? e : h2d(d_tgt, target_argmax, sizeof(int32_t) * B * blk);
        e = e ? e : h2d(d_tsl, target_seq_len, sizeof(int32_t) * B);
        e = e ? e : h2d(d_eos, eos, sizeof(int32_t) * n_eos);
        e = e ? e : cudaMemsetAsync(d_st, 0, sizeof(int32_t), s);
        if (e != cudaSuccess) return fail(DF_ECUDA, "host round staging: %s", cudaGetErrorString(e));
        DF_TRY(df_draft_round(cfg, w, cache, d_last, n_new_max ? d_th : nullptr,
                              n_new_max ? d_nnew : nullptr, n_new_max, B, K, d_tgt, d_eos, n_eos,
                              d_tsl, d_am, d_com, d_nc, d_ac, d_he, d_rb, ws, need_round, d_st,
                              (df_stream_t)s));
        e = d2h(target_seq_len, d_tsl, sizeof(int32_t) * B);
        e = e ? e : d2h(argmax_out, d_am, sizeof(int32_t) * B * blk);
        e = e ? e : d2h(committed, d_com, sizeof(int32_t) * B * blk);
        e = e ? e : d2h(n_committed, d_nc, sizeof(int32_t) * B);
        e = e ? e : d2h(accept_count, d_ac, sizeof(int32_t) * B);
        e = e ? e : d2h(hit_eos, d_he, sizeof(int32_t) * B);
        e = e ? e : d2h(rollback, d_rb, sizeof(int32_t) * B);
        e = e ? e : d2h(status, d_st, sizeof(int32_t));
        if (e != cudaSuccess) return fail(DF_ECUDA, "host round readback: %s", cudaGetErrorString(e));
        return DF_OK;
    };
    // With every host buffer page-locked the whole call is one cached CUDA graph (copies and
    // kernels baked with these exact arguments), so a repeated call costs one graph launch and
    // the synchronisation; pageable buffers take the stream path.
    cudaError_t e = cudaSuccess;
    if (!pinned) {
        DF_TRY(enqueue(user));
    } else {
        uint64_t key = 1469598103934665603ull;
        key = fnv(key, cfg, sizeof(*cfg));
        key = fnv(key, w, sizeof(*w));
        key = fnv(key, w->layers, sizeof(df_layer_weights) * cfg->n_layers);
        key = fnv(key, cache, sizeof(*cache));
        key = fnv(key, cache->k, sizeof(float *) * cfg->n_layers);
        key = fnv(key, cache->v, sizeof(float *) * cfg->n_layers);
        key = fnv(key, host_bufs, sizeof(host_bufs));
        key = fnv(key, dev_of, sizeof(dev_of));   // a buffer pinned again maps elsewhere
        const long long scal[] = {n_new_max, B, K, n_eos, (long long)ws_bytes};
        key = fnv(key, scal, sizeof(scal));
        key = fnv(key, &ws, sizeof(ws));
        key = fnv(key, &stream, sizeof(stream));
        int dev = 0;
        cudaGetDevice(&dev);
        key = fnv(key, &dev, sizeof(dev));
        DF_TRY(host_round_graph(key, enqueue_mapped, user));
    }
    e = cudaStreamSynchronize(user);
    if (e != cudaSuccess) return fail(DF_ECUDA, "host round readback: %s", cudaGetErrorString(e));
    return DF_OK;
}

}  // extern "C"

// ================================================================ multi-round generate loop
namespace df {
namespace {

// Round scratch of the loop, after the round's own workspace.
struct LoopWs {
    float *th;
    int32_t *ints;
};

size_t loop_extra_bytes(const df_dflash_config *c, int B, int K, int n_new_max) {
    Carve cv{nullptr, 0, ~size_t(0), true};
    cv.take<float>((size_t)B * std::max(n_new_max, 1) * c->n_target_layers * c->hidden);
    cv.take<int32_t>((size_t)B * (4 * (K + 1) + 8) + 8);
    return cv.off;
}

// One cached executable graph: the loop is rebuilt only when an argument changes.
struct LoopGraph {
    std::mutex mu;
    uint64_t key = 0;
    bool have = false;
    cudaGraph_t graph = nullptr;
    cudaGraphExec_t exec = nullptr;
    cudaStream_t cap = nullptr;
};
LoopGraph g_loop;


}  // namespace
}  // namespace df

extern "C" {

size_t df_generate_workspace_bytes(const df_dflash_config *cfg, int B, int K, int n_new_max) {
    if (check_cfg(cfg) != DF_OK || B <= 0 || K < 1 || n_new_max < K + 1) return 0;
    const size_t fwd = df_dflash_workspace_bytes(cfg, B, K + 1, n_new_max);
    return fwd ? fwd + loop_extra_bytes(cfg, B, K, n_new_max) : 0;
}

int df_generate(const df_dflash_config *cfg, const df_dflash_weights *w, const df_kv_cache *cache,
                const df_synthetic_verifier *v, float *prior_cap, int32_t *prior_len,
                int32_t *out_tokens, int32_t *out_len, const int32_t *prompt_len,
                int max_new_tokens, int max_rounds, int B, int K, int n_new_max,
                const int32_t *eos, int n_eos, int32_t *rounds, int32_t *accept_hist, void *ws,
                size_t ws_bytes, int32_t *d_status, df_stream_t stream) {
    g_err[0] = 0;
    DF_TRY(check_cfg(cfg));
    DF_TRY(check_weights(cfg, w));
    REQ(B > 0 && B <= 1024 && K >= 1, DF_ESHAPE, "B=%d K=%d (B <= 1024, K >= 1)", B, K);
    REQ(n_new_max >= K + 1 && cache && n_new_max <= cache->cap, DF_ESHAPE,
        "n_new_max=%d (K+1 <= n_new_max <= cache cap)", n_new_max);
    DF_TRY(check_cache(cache, cfg->n_layers, B, cfg->head_dim));
    REQ(v && v->ref && v->table && v->max_len > K + 2, DF_EINVAL, "synthetic verifier");
    REQ(v->n_comb >= 1 && cfg->n_target_layers <= kLoopMaxTargetLayers, DF_ESHAPE,
        "n_comb=%d, n_target_layers=%d (<= %d)", v->n_comb, cfg->n_target_layers,
        kLoopMaxTargetLayers);
    for (int l = 0; l < cfg->n_target_layers; ++l)
        REQ(v->sel[l] >= 0 && v->sel[l] < v->n_comb, DF_ESHAPE, "sel[%d]=%d outside the %d captured layers",
            l, v->sel[l], v->n_comb);
    REQ(prior_cap && prior_len && out_tokens && out_len && prompt_len && rounds, DF_EINVAL,
        "NULL loop state");
    REQ(max_rounds >= 0 && max_new_tokens >= 0, DF_ESHAPE, "max_rounds / max_new_tokens");
    REQ(n_eos >= 0 && (n_eos == 0 || eos), DF_EINVAL, "eos list");
    DF_TRY(get_ws(ws, ws_bytes, df_generate_workspace_bytes(cfg, B, K, n_new_max)));
    const int blk = K + 1;
    Carve cv{static_cast<char *>(ws), 0, ws_bytes, true};
    DFlashWs W;
    carve_dflash(cv, W, cfg, B, blk, n_new_max, cache->cap, true);
    float *th = cv.take<float>((size_t)B * n_new_max * cfg->n_target_layers * cfg->hidden);
    int32_t *ints = cv.take<int32_t>((size_t)B * (4 * blk + 8) + 8);
    REQ(cv.ok, DF_EWORKSPACE, "workspace too small");
    LoopArgs a;
    memset(static_cast<void *>(&a), 0, sizeof(a));   // padding too: the bytes key the graph cache
    a.th = th;
    a.ref = v->ref;
    a.agree = v->agree;
    a.table = v->table;
    a.n_comb = v->n_comb;
    for (int l = 0; l < cfg->n_target_layers; ++l) a.sel[l] = v->sel[l];
    a.max_len = v->max_len;
    a.prior_cap = prior_cap;
    a.prior_len = prior_len;
    a.out = out_tokens;
    a.out_len = out_len;
    a.prompt_len = prompt_len;
    a.rounds = rounds;
    a.accept_hist = accept_hist;
    a.max_rounds = max_rounds;
    a.max_new = max_new_tokens;
    a.cache_seq = cache->seq_len;
    a.B = B;
    a.K = K;
    a.H = cfg->hidden;
    a.n_tl = cfg->n_target_layers;
    a.n_new_max = n_new_max;
    a.argmax = ints;
    a.target = ints + (size_t)B * blk;
    a.committed = ints + (size_t)2 * B * blk;
    a.n_new = ints + (size_t)3 * B * blk;
    a.last_token = a.n_new + B;
    a.n_committed = a.last_token + B;
    a.accept = a.n_committed + B;
    a.hit = a.accept + B;
    a.rollback = a.hit + B;
    a.done = a.rollback + B;
    a.round_ctr = a.done + B;
    a.eos = eos;
    a.n_eos = n_eos;
    a.status = d_status;

    // the cache key: every argument the graph bakes in
    uint64_t key = 1469598103934665603ull;
    key = fnv(key, cfg, sizeof(*cfg));
    key = fnv(key, w, sizeof(*w));
    key = fnv(key, w->layers, sizeof(df_layer_weights) * cfg->n_layers);
    key = fnv(key, cache, sizeof(*cache));
    key = fnv(key, cache->k, sizeof(float *) * cfg->n_layers);
    key = fnv(key, cache->v, sizeof(float *) * cfg->n_layers);
    key = fnv(key, &a, sizeof(a));
    key = fnv(key, &ws, sizeof(ws));
    key = fnv(key, &stream, sizeof(stream));
    cudaStream_t user = (cudaStream_t)stream;
    std::lock_guard<std::mutex> lk(g_loop.mu);
    if (!(g_loop.have && g_loop.key == key)) {
        if (g_loop.have) {
            cudaGraphExecDestroy(g_loop.exec);
            cudaGraphDestroy(g_loop.graph);
            g_loop.have = false;
        }
        if (!g_loop.cap) {
            cudaError_t e = cudaStreamCreateWithFlags(&g_loop.cap, cudaStreamNonBlocking);
            if (e != cudaSuccess) return fail(DF_ECUDA, "loop capture stream: %s", cudaGetErrorString(e));
        }
        cudaStream_t cs = g_loop.cap;
        cudaGraph_t g = nullptr;
        cudaError_t e = cudaGraphCreate(&g, 0);
        cudaGraphConditionalHandle h = 0;
        if (e == cudaSuccess) e = cudaGraphConditionalHandleCreate(&h, g, 1, cudaGraphCondAssignDefault);
        a.cond = h;
        // the init kernel, then a while node whose body is one round
        if (e == cudaSuccess)
            e = cudaStreamBeginCaptureToGraph(cs, g, nullptr, nullptr, 0, cudaStreamCaptureModeThreadLocal);
        if (e != cudaSuccess) {
            if (g) cudaGraphDestroy(g);
            return fail(DF_ECUDA, "loop graph set-up: %s", cudaGetErrorString(e));
        }
        int rc = launch_loop_init(a, cs);
        cudaGraph_t got = nullptr;
        e = cudaStreamEndCapture(cs, &got);
        if (rc != DF_OK || e != cudaSuccess) {
            cudaGraphDestroy(g);
            return rc != DF_OK ? rc : fail(DF_ECUDA, "loop init capture: %s", cudaGetErrorString(e));
        }
        cudaGraphNode_t init_node = nullptr;
        size_t n_nodes = 1;
        e = cudaGraphGetNodes(g, &init_node, &n_nodes);
        cudaGraphNodeParams cp = {};
        cp.type = cudaGraphNodeTypeConditional;
        cp.conditional.handle = h;
        cp.conditional.type = cudaGraphCondTypeWhile;
        cp.conditional.size = 1;
        cudaGraphNode_t cnode = nullptr;
        if (e == cudaSuccess) e = cudaGraphAddNode(&cnode, g, &init_node, nullptr, 1, &cp);
        cudaGraph_t body = e == cudaSuccess ? cp.conditional.phGraph_out[0] : nullptr;
        if (e == cudaSuccess)
            e = cudaStreamBeginCaptureToGraph(cs, body, nullptr, nullptr, 0, cudaStreamCaptureModeThreadLocal);
        if (e != cudaSuccess) {
            cudaGraphDestroy(g);
            return fail(DF_ECUDA, "loop while node: %s", cudaGetErrorString(e));
        }
        rc = launch_loop_prepare(a, cs);
        if (rc == DF_OK)
            rc = dflash_forward_impl(cfg, w, cache, nullptr, a.last_token, a.th, a.n_new, n_new_max,
                                     B, blk, W.h_final, W.xp_head, W, d_status, cs);
        if (rc == DF_OK)
            rc = lm_head_impl(w->lm_head, W.xp_head, B * blk, cfg->hidden, cfg->vocab, W.amax_part,
                              a.argmax, nullptr, nullptr, W.tc, cs, W.ss_post, cfg->rms_eps,
                              W.ss_slots, dflash_tiled(cfg, w, -1, DP_LM_HEAD));
        if (rc == DF_OK) rc = launch_loop_verify(a, cs);
        if (rc == DF_OK)
            rc = launch_accept(a.argmax + 1, blk, a.target, B, K, eos, n_eos, a.committed,
                               a.n_committed, a.accept, a.hit, a.rollback, nullptr, d_status, cs);
        if (rc == DF_OK) rc = launch_loop_append(a, cs);
        if (rc == DF_OK) rc = launch_loop_commit(a, cs);
        e = cudaStreamEndCapture(cs, &body);
        if (rc != DF_OK || e != cudaSuccess) {
            cudaGraphDestroy(g);
            return rc != DF_OK ? rc : fail(DF_ECUDA, "loop body capture: %s", cudaGetErrorString(e));
        }
        cudaGraphExec_t ex = nullptr;
        e = cudaGraphInstantiate(&ex, g, 0);
        if (e != cudaSuccess) {
            cudaGraphDestroy(g);
            return fail(DF_ECUDA, "loop graph instantiate: %s", cudaGetErrorString(e));
        }
        g_loop.graph = g;
        g_loop.exec = ex;
        g_loop.key = key;
        g_loop.have = true;
    }
    cudaError_t e = cudaGraphLaunch(g_loop.exec, user);
    if (e != cudaSuccess) return fail(DF_ECUDA, "loop graph launch: %s", cudaGetErrorString(e));
    return DF_OK;
}

}  // extern "C"

// ================================================================ MTP draft step
namespace df {
namespace {

int check_mtp_cfg(const df_mtp_config *c) {
    REQ(c, DF_EINVAL, "MTP config is NULL");
    REQ(c->hidden > 0 && c->hidden % 8 == 0, DF_ESHAPE, "hidden=%d", c->hidden);
    REQ(c->n_q_heads > 0 && c->n_kv_heads > 0 && c->n_q_heads % c->n_kv_heads == 0, DF_ESHAPE,
        "heads %d / %d", c->n_q_heads, c->n_kv_heads);
    REQ(c->head_dim >= 32 && c->head_dim <= 256 && c->head_dim % 32 == 0, DF_ESHAPE,
        "head_dim=%d", c->head_dim);
    int rot = c->rotary_dim ? c->rotary_dim : c->head_dim;
    REQ(rot > 0 && rot <= c->head_dim && rot % 2 == 0, DF_ESHAPE, "rotary_dim=%d", c->rotary_dim);
    REQ(c->vocab > 1, DF_ESHAPE, "vocab=%d", c->vocab);
    if (c->n_experts == 0) {
        REQ(c->intermediate > 0 && c->intermediate % 8 == 0, DF_ESHAPE, "intermediate=%d",
            c->intermediate);
    } else {
        REQ(c->n_experts > 0 && c->n_experts <= kMoeMaxExperts && c->top_k >= 1 &&
                c->top_k <= c->n_experts && c->top_k <= kMoeMaxTopK,
            DF_ESHAPE, "n_experts=%d top_k=%d (n_experts <= %d, top_k <= %d)", c->n_experts,
            c->top_k, kMoeMaxExperts, kMoeMaxTopK);
        REQ(c->expert_inter > 0 && c->expert_inter % 8 == 0 && c->shared_inter > 0 &&
                c->shared_inter % 8 == 0,
            DF_ESHAPE, "expert_inter=%d shared_inter=%d", c->expert_inter, c->shared_inter);
    }
    REQ(c->rms_eps >= 0.f && c->rope_theta > 0.f, DF_EINVAL, "rms_eps / rope_theta");
    return DF_OK;
}

int check_moe_weights(const df_mtp_weights *w) {
    DF_TRY(check_bf16(w->router, "router"));
    DF_TRY(check_bf16(w->exp_gate, "exp_gate"));
    DF_TRY(check_bf16(w->exp_up, "exp_up"));
    DF_TRY(check_bf16(w->exp_down, "exp_down"));
    DF_TRY(check_bf16(w->sh_gate_mlp, "sh_gate_mlp"));
    DF_TRY(check_bf16(w->sh_up, "sh_up"));
    DF_TRY(check_bf16(w->sh_down, "sh_down"));
    DF_TRY(check_bf16(w->sh_expert_gate, "sh_expert_gate"));
    return DF_OK;
}

int check_mtp_weights(const df_mtp_config *c, const df_mtp_weights *w) {
    REQ(w, DF_EINVAL, "MTP weights is NULL");
    DF_TRY(check_f32(w->enorm, "enorm"));
    DF_TRY(check_f32(w->hnorm, "hnorm"));
    DF_TRY(check_bf16(w->eh_embed, "eh_embed"));
    DF_TRY(check_bf16(w->eh_hidden, "eh_hidden"));
    DF_TRY(check_f32(w->attn_norm, "attn_norm"));
    DF_TRY(check_f32(w->post_attn_norm, "post_attn_norm"));
    DF_TRY(check_f32(w->q_norm, "q_norm"));
    DF_TRY(check_f32(w->k_norm, "k_norm"));
    DF_TRY(check_bf16(w->wq, "wq"));
    DF_TRY(check_bf16(w->wk, "wk"));
    DF_TRY(check_bf16(w->wv, "wv"));
    if (w->w_gate) DF_TRY(check_bf16(w->w_gate, "w_gate"));
    DF_TRY(check_bf16(w->wo, "wo"));
    DF_TRY(check_f32(w->shared_head_norm, "shared_head_norm"));
    DF_TRY(check_bf16(w->embed, "embed"));
    DF_TRY(check_bf16(w->lm_head, "lm_head"));
    if (c->n_experts == 0) {
        DF_TRY(check_bf16(w->w_gate_mlp, "w_gate_mlp"));
        DF_TRY(check_bf16(w->w_up, "w_up"));
        DF_TRY(check_bf16(w->w_down, "w_down"));
    } else {
        DF_TRY(check_moe_weights(w));
    }
    return DF_OK;
}

// Scratch of the MoE FFN (router logits, choice, activations, per-slot outputs, counter).
struct MoeWs {
    float *logits, *wts, *act, *part;
    int32_t *sel;
    int *counter;
};

void carve_moe(Carve &cv, MoeWs &m, const df_mtp_config *c, int T) {
    const size_t S = (size_t)c->top_k + 1, Imax = (size_t)std::max(c->expert_inter, c->shared_inter);
    m.logits = cv.take<float>((size_t)T * (c->n_experts + 1));
    m.sel = cv.take<int32_t>((size_t)T * c->top_k);
    m.wts = cv.take<float>((size_t)T * S);
    m.act = cv.take<float>((size_t)T * S * Imax);
    m.part = cv.take<float>(S * T * c->hidden);
    m.counter = cv.take<int>(1);
}

MoeArgs moe_args(const df_mtp_config *c, const df_mtp_weights *w, const MoeWs &m,
                 const float *x, int T, int32_t *status) {
    MoeArgs a;
    a.x = x;
    a.ldx = c->hidden;
    a.T = T;
    a.H = c->hidden;
    a.E = c->n_experts;
    a.k = c->top_k;
    a.Ie = c->expert_inter;
    a.Is = c->shared_inter;
    a.router = w->router;
    a.sh_gate = w->sh_expert_gate;
    a.exp_gate = w->exp_gate;
    a.exp_up = w->exp_up;
    a.exp_down = w->exp_down;
    a.sh_g = w->sh_gate_mlp;
    a.sh_u = w->sh_up;
    a.sh_d = w->sh_down;
    a.logits = m.logits;
    a.sel = m.sel;
    a.wts = m.wts;
    a.act = m.act;
    a.part = m.part;
    a.ldpart = c->hidden;
    a.counter = m.counter;
    a.status = status;
    return a;
}

struct MtpWs {
    float *x, *defer, *gate, *q, *h1, *xf, *cos_t, *sin_t, *attn_part;
    uint16_t *xp_e, *xp_h, *xp_attn, *xp_o, *xp_ffn, *xp_act, *xp_head;
    ArgTop *amax_part;
    MoeWs moe;
    AttnArgs plan;
    TcScratch tc;
};

void carve_mtp(Carve &cv, MtpWs &w, const df_mtp_config *c, int B, int cap) {
    const int H = c->hidden, d = c->head_dim, nq = c->n_q_heads, nkv = c->n_kv_heads;
    const int rot = c->rotary_dim ? c->rotary_dim : d;
    const size_t qt = (size_t)nq * d, kt = (size_t)nkv * d;
    const size_t I = c->n_experts ? 0 : (size_t)c->intermediate;
    w.x = cv.take<float>((size_t)B * H);
    w.defer = cv.take<float>(defer_floats_for(B, (long long)std::max<size_t>(2 * qt + 2 * kt, H)));
    w.gate = cv.take<float>((size_t)B * qt);
    w.q = cv.take<float>((size_t)B * qt);
    w.h1 = cv.take<float>((size_t)B * H);
    w.xf = cv.take<float>((size_t)B * H);
    w.cos_t = cv.take<float>((size_t)B * (rot / 2));
    w.sin_t = cv.take<float>((size_t)B * (rot / 2));
    w.plan = AttnArgs{};
    w.plan.B = B;
    w.plan.blk = 1;
    w.plan.nq = nq;
    w.plan.nkv = nkv;
    w.plan.d = d;
    attn_plan(w.plan, cap);
    w.attn_part = cv.take<float>(attn_part_floats(w.plan));
    w.xp_e = cv.take<uint16_t>((size_t)2 * B * H);
    w.xp_h = cv.take<uint16_t>((size_t)2 * B * H);
    w.xp_attn = cv.take<uint16_t>((size_t)2 * B * H);
    w.xp_o = cv.take<uint16_t>((size_t)2 * B * qt);
    w.xp_ffn = cv.take<uint16_t>((size_t)2 * B * H);
    w.xp_act = cv.take<uint16_t>((size_t)2 * B * std::max<size_t>(I, 1));
    w.xp_head = cv.take<uint16_t>((size_t)2 * B * H);
    w.amax_part = cv.take<ArgTop>(argmax_parts(B));
    if (c->n_experts) carve_moe(cv, w.moe, c, B);
    else w.moe = MoeWs{};
    long long rows = std::max<long long>({(long long)c->vocab, 2LL * (long long)I,
                                          (long long)(qt + 2 * kt), (long long)H});
    carve_tc(cv, w.tc, B, rows);
}

// The weight operand of each MTP projection (the dense FFN only without experts), shared by the
// step and by the tiling of the weights.
enum MtpProj { MP_EH, MP_QKV, MP_O, MP_GATE_UP, MP_DOWN, MP_LM_HEAD, MP_COUNT };

bool mtp_has(const df_mtp_config *c, int which) {
    return !((which == MP_GATE_UP || which == MP_DOWN) && c->n_experts > 0);
}

GemmArgs mtp_proj(const df_mtp_config *c, const df_mtp_weights *w, int which) {
    const int H = c->hidden, d = c->head_dim, qt = c->n_q_heads * d, kt = c->n_kv_heads * d;
    GemmArgs g;
    switch (which) {
        case MP_EH:
            g.W0 = w->eh_embed;
            g.n0 = H;
            g.Wk2 = w->eh_hidden;
            g.K1 = H;
            g.N = H;
            g.K = 2 * H;
            break;
        case MP_QKV:
            g.W0 = w->wq;
            g.n0 = qt;
            g.W1 = w->wk;
            g.n1 = kt;
            g.W2 = w->wv;
            g.n2 = kt;
            g.W3 = w->w_gate;
            g.n3 = w->w_gate ? qt : 0;
            g.N = qt + 2 * kt + g.n3;
            g.K = H;
            break;
        case MP_O:
            g.W0 = w->wo;
            g.n0 = H;
            g.N = H;
            g.K = qt;
            break;
        case MP_GATE_UP:
            g.W0 = w->w_gate_mlp;
            g.n0 = c->intermediate;
            g.W1 = w->w_up;
            g.n1 = c->intermediate;
            g.N = c->intermediate;
            g.K = H;
            g.epi = EPI_SWIGLU;
            break;
        case MP_DOWN:
            g.W0 = w->w_down;
            g.n0 = H;
            g.N = H;
            g.K = c->intermediate;
            break;
        default:   // MP_LM_HEAD
            g.W0 = w->lm_head;
            g.n0 = c->vocab;
            g.N = c->vocab;
            g.K = H;
            break;
    }
    return g;
}

// Tiled layout of an MTP block's weights: eh_proj, QKV (+ output gate), O, the dense gate/up and
// down (when there are no experts), the lm_head; each on a 1024-byte boundary. Offset of
// projection `which` (MP_COUNT: the total).
size_t mtp_tiled_offset(const df_mtp_config *c, const df_mtp_weights *w, int which) {
    size_t off = 0;
    for (int k = 0; k < which; ++k)
        if (mtp_has(c, k)) off += (tiled_projection_bytes(mtp_proj(c, w, k)) + 1023) & ~size_t(1023);
    return off;
}

const uint8_t *mtp_tiled(const df_mtp_config *c, const df_mtp_weights *w, int which) {
    if (!w->tiled) return nullptr;
    return static_cast<const uint8_t *>(w->tiled) + mtp_tiled_offset(c, w, which);
}

}  // namespace
}  // namespace df

extern "C" {

size_t df_mtp_tiled_bytes(const df_mtp_config *cfg, const df_mtp_weights *w) {
    if (check_mtp_cfg(cfg) != DF_OK || check_mtp_weights(cfg, w) != DF_OK) return 0;
    g_err[0] = 0;
    return mtp_tiled_offset(cfg, w, MP_COUNT);
}

int df_mtp_tile_weights(const df_mtp_config *cfg, const df_mtp_weights *w, void *tiled,
                        size_t tiled_bytes, df_stream_t stream) {
    g_err[0] = 0;
    DF_TRY(check_mtp_cfg(cfg));
    DF_TRY(check_mtp_weights(cfg, w));
    const size_t need = mtp_tiled_offset(cfg, w, MP_COUNT);
    REQ(tiled && tiled_bytes >= need, DF_EWORKSPACE, "tiled weights need %zu bytes, have %zu",
        need, tiled_bytes);
    REQ((reinterpret_cast<uintptr_t>(tiled) & 1023u) == 0, DF_EINVAL,
        "tiled weights must be 1024-byte aligned");
    uint8_t *base = static_cast<uint8_t *>(tiled);
    for (int k = 0; k < MP_COUNT; ++k) {
        if (!mtp_has(cfg, k)) continue;
        const size_t off = mtp_tiled_offset(cfg, w, k);
        const size_t len = tiled_projection_bytes(mtp_proj(cfg, w, k));
        DF_TRY(tile_projection(mtp_proj(cfg, w, k), base + off, len, (cudaStream_t)stream));
    }
    return DF_OK;
}

size_t df_mtp_workspace_bytes(const df_mtp_config *cfg, int B) {
    if (check_mtp_cfg(cfg) != DF_OK || B <= 0) return 0;
    Carve cv{nullptr, 0, ~size_t(0), true};
    MtpWs w;
    carve_mtp(cv, w, cfg, B, 1 << 20);
    SampleArgs a;
    carve_sample_scratch(cv, a, B, 1, cfg->vocab);
    return cv.off;
}

}  // extern "C"

namespace df {
namespace {

// The chained MTP draft. temperature == 0: each step's token is the lm_head argmax (and the
// last step's logits are stored when logits_out is given). temperature > 0: every step stores
// its logits in logits_out [n_steps, B, V] and its token is drawn from softmax(logits / T) with
// u_draft [n_steps, B]; argmax_out then receives the drawn tokens.
int mtp_impl(const df_mtp_config *cfg, const df_mtp_weights *w, const df_kv_cache *cache,
             const float *prev_hidden, const int32_t *token, int B, int n_steps,
             float *hidden_out, int32_t *argmax_out, float *logits_out, float temperature,
             const float *u_draft, void *ws, size_t ws_bytes, int32_t *d_status,
             df_stream_t stream) {
    DF_TRY(check_mtp_cfg(cfg));
    DF_TRY(check_mtp_weights(cfg, w));
    REQ(B > 0 && n_steps >= 1, DF_ESHAPE, "B=%d n_steps=%d", B, n_steps);
    DF_TRY(check_cache(cache, 1, B, cfg->head_dim));
    REQ(prev_hidden && token && hidden_out && argmax_out, DF_EINVAL, "NULL MTP input or output");
    REQ(cfg->n_experts == 0 || B <= kMoeMaxRows, DF_ESHAPE, "MoE MTP takes B <= %d (B=%d)",
        kMoeMaxRows, B);
    const bool sampled = temperature > 0.f;
    if (sampled) {
        REQ(logits_out && u_draft, DF_EINVAL, "a sampled MTP draft needs logits_out and u_draft");
        REQ(cfg->vocab % 4 == 0, DF_ESHAPE, "vocab=%d (a multiple of 4)", cfg->vocab);
        DF_TRY(check_f32(logits_out, "logits_out"));
    }
    DF_TRY(get_ws(ws, ws_bytes, df_mtp_workspace_bytes(cfg, B)));
    Carve cv{static_cast<char *>(ws), 0, ws_bytes, true};
    MtpWs W;
    carve_mtp(cv, W, cfg, B, cache->cap);
    SampleArgs sa;
    carve_sample_scratch(cv, sa, B, 1, cfg->vocab);
    cudaStream_t s = (cudaStream_t)stream;
    const int H = cfg->hidden, d = cfg->head_dim, nq = cfg->n_q_heads, nkv = cfg->n_kv_heads;
    const int rot = cfg->rotary_dim ? cfg->rotary_dim : d;
    const int qt = nq * d, kt = nkv * d, Nqkv = qt + 2 * kt, I = cfg->intermediate;
    const bool moe = cfg->n_experts > 0;

    // A projection whose split partial sums land in W.defer; returns the split count.
    auto deferred = [&](GemmArgs g, int N, const char *name, int *S) -> int {
        g.epi = EPI_STORE;
        g.defer = 1;
        g.out = W.defer;
        g.ldo = N;
        g.part_stride = (size_t)B * N;
        g.status = d_status;
        g.name = name;
        return launch_gemm_tc(g, W.tc, s, S);
    };
    const int n_gate = w->w_gate ? nq : 0;
    const int Nq4 = Nqkv + n_gate * d;
    for (int st = 0; st < n_steps; ++st) {
        const float *hprev = st == 0 ? prev_hidden : hidden_out + (size_t)(st - 1) * B * H;
        const int32_t *tok = st == 0 ? token : argmax_out + (size_t)(st - 1) * B;
        float *hid = hidden_out + (size_t)st * B * H;
        // x = eh_embed . enorm(embed[tok]) + eh_hidden . hnorm(prev): one projection over the
        // concatenation [enorm(e); hnorm(h)] (mtp.rs `project_embedding_and_hidden`).
        PackArgs pe;
        pe.gather = w->embed;
        pe.ids = tok;
        pe.vocab = cfg->vocab;
        pe.rows_per_seq = 1;
        pe.norm_w = w->enorm;
        pe.eps = 1e-6f;
        pe.pack = W.xp_e;
        pe.ldp = H;
        pe.T = B;
        pe.K = H;
        pe.status = d_status;
        DF_TRY(launch_pack(pe, s));
        PackArgs ph;
        ph.src = hprev;
        ph.lds = H;
        ph.norm_w = w->hnorm;
        ph.eps = 1e-6f;
        ph.pack = W.xp_h;
        ph.ldp = H;
        ph.T = B;
        ph.K = H;
        DF_TRY(launch_pack(ph, s));
        GemmArgs ge = mtp_proj(cfg, w, MP_EH);
        ge.At = mtp_tiled(cfg, w, MP_EH);
        ge.X = W.xp_e;
        ge.ldx = H;
        ge.X2 = W.xp_h;
        ge.ldx2 = H;
        ge.T = B;
        int S_eh = 0;
        DF_TRY(deferred(ge, H, "gemm_eh_proj", &S_eh));

        // x = sum of the eh partials (kept as the attention residual); attention RMSNorm
        PackArgs pa;
        pa.part = W.defer;
        pa.n_part = S_eh;
        pa.part_stride = (size_t)B * H;
        pa.ldpart = H;
        pa.h_out = W.x;
        pa.ldh = H;
        pa.norm_w = w->attn_norm;
        pa.eps = cfg->rms_eps;
        pa.pack = W.xp_attn;
        pa.ldp = H;
        pa.T = B;
        pa.K = H;
        DF_TRY(launch_pack(pa, s));
        GemmArgs gq = mtp_proj(cfg, w, MP_QKV);
        gq.At = mtp_tiled(cfg, w, MP_QKV);
        gq.X = W.xp_attn;
        gq.ldx = H;
        gq.T = B;
        int S_q = 0;
        DF_TRY(deferred(gq, Nq4, "gemm_qkv_gate", &S_q));
        DF_TRY(launch_rope_table(W.cos_t, W.sin_t, cache->seq_len, nullptr, 0, B, 1, st, rot,
                                 cfg->rope_theta, d_status, s));
        QkArgs qa;
        qa.qkv = nullptr;
        qa.part = W.defer;
        qa.n_part = S_q;
        qa.part_stride = (size_t)B * Nq4;
        qa.ldq = Nq4;
        qa.n_gate_heads = n_gate;
        qa.gate_out = W.gate;
        qa.ldg = qt;
        qa.B = B;
        qa.blk = 1;
        qa.n_new_max = 0;
        qa.nq = nq;
        qa.nkv = nkv;
        qa.d = d;
        qa.rot = rot;
        qa.q_norm = w->q_norm;
        qa.k_norm = w->k_norm;
        qa.eps = cfg->rms_eps;
        qa.cos_t = W.cos_t;
        qa.sin_t = W.sin_t;
        qa.q_out = W.q;
        qa.kb = nullptr;
        qa.vb = nullptr;
        qa.cache_k = cache->k[0];
        qa.cache_v = cache->v[0];
        qa.cap = cache->cap;
        qa.seq_len = cache->seq_len;
        qa.n_new = nullptr;
        qa.append_block = 1;
        qa.pos_off = st;
        qa.status = d_status;
        DF_TRY(launch_qk_rope(qa, s));
        AttnArgs at = W.plan;
        at.q = W.q;
        at.cache_k = cache->k[0];
        at.cache_v = cache->v[0];
        at.cap = cache->cap;
        at.kb = nullptr;
        at.vb = nullptr;
        at.seq_len = cache->seq_len;
        at.n_new = nullptr;
        at.n_new_max = 0;
        at.extra_rows = st + 1;
        at.early_kv = 1;   // seq_len moves only at the end of the chain
        at.causal_block = 0;
        at.part = W.attn_part;
        at.gate = w->w_gate ? W.gate : nullptr;
        at.ldg = qt;
        at.pack = W.xp_o;
        at.status = d_status;
        DF_TRY(launch_attn(at, s));
        GemmArgs go = mtp_proj(cfg, w, MP_O);
        go.At = mtp_tiled(cfg, w, MP_O);
        go.X = W.xp_o;
        go.ldx = qt;
        go.T = B;
        int S_o = 0;
        DF_TRY(deferred(go, H, "gemm_o", &S_o));
        // h1 = x + O partials (fused residual add); post-attention RMSNorm
        PackArgs pf;
        pf.src = W.x;
        pf.lds = H;
        pf.part = W.defer;
        pf.n_part = S_o;
        pf.part_stride = (size_t)B * H;
        pf.ldpart = H;
        pf.h_out = W.h1;
        pf.ldh = H;
        pf.norm_w = w->post_attn_norm;
        pf.eps = cfg->rms_eps;
        if (moe) {
            pf.y_out = W.xf;
            pf.ldy = H;
        } else {
            pf.pack = W.xp_ffn;
            pf.ldp = H;
        }
        pf.T = B;
        pf.K = H;
        DF_TRY(launch_pack(pf, s));
        PackArgs pk;   // hidden = h1 + FFN output (the step's output); shared-head RMSNorm
        pk.src = W.h1;
        pk.lds = H;
        pk.h_out = hid;
        pk.ldh = H;
        pk.norm_w = w->shared_head_norm;
        pk.eps = cfg->rms_eps;
        pk.pack = W.xp_head;
        pk.ldp = H;
        pk.T = B;
        pk.K = H;
        if (moe) {
            // routed experts + shared expert, one weighted output per slot (mtp.rs
            // `MtpFfnWeightsGpu::Moe`), summed in slot order by the head pack below
            DF_TRY(launch_moe(moe_args(cfg, w, W.moe, W.xf, B, d_status), s));
            pk.part = W.moe.part;
            pk.n_part = cfg->top_k + 1;
        } else {
            GemmArgs gu = mtp_proj(cfg, w, MP_GATE_UP);
            gu.At = mtp_tiled(cfg, w, MP_GATE_UP);
            gu.X = W.xp_ffn;
            gu.ldx = H;
            gu.T = B;
            gu.pack_out = W.xp_act;
            gu.ldpo = I;
            gu.name = "gemm_gate_up";
            DF_TRY(launch_gemm_tc(gu, W.tc, s));
            GemmArgs gd = mtp_proj(cfg, w, MP_DOWN);
            gd.At = mtp_tiled(cfg, w, MP_DOWN);
            gd.X = W.xp_act;
            gd.ldx = I;
            gd.T = B;
            int S_d = 0;
            DF_TRY(deferred(gd, H, "gemm_down", &S_d));
            pk.part = W.defer;   // dense SwiGLU: the down projection's split partial sums
            pk.n_part = S_d;
        }
        pk.part_stride = (size_t)B * H;
        pk.ldpart = H;
        // shared head: RMSNorm then lm_head argmax (mtp.rs `forward_ffn_residual`,
        // `forward_shared_head`)
        DF_TRY(launch_pack(pk, s));
        if (sampled) {
            // this step's logits, then its draft drawn from softmax(logits / T)
            float *lg = logits_out + (size_t)st * B * cfg->vocab;
            GemmArgs gl = mtp_proj(cfg, w, MP_LM_HEAD);
            gl.At = mtp_tiled(cfg, w, MP_LM_HEAD);
            gl.X = W.xp_head;
            gl.ldx = H;
            gl.T = B;
            gl.epi = EPI_STORE;
            gl.out = lg;
            gl.ldo = cfg->vocab;
            gl.status = d_status;
            gl.name = "gemm_logits";
            DF_TRY(launch_gemm_tc(gl, W.tc, s));
            sa.draft = lg;
            sa.draft_ld = 1;
            sa.V = cfg->vocab;
            sa.B = B;
            sa.K = 1;
            sa.T = temperature;
            sample_constants(sa);
            sa.sample_mode = 1;
            sa.u_draft = u_draft + (size_t)st * B;
            sa.drafts_out = argmax_out + (size_t)st * B;
            sa.status = d_status;
            DF_TRY(launch_sample_drafts(sa, s));
            continue;
        }
        DF_TRY(lm_head_impl(w->lm_head, W.xp_head, B, H, cfg->vocab, W.amax_part,
                            argmax_out + (size_t)st * B, nullptr, nullptr, W.tc, s, nullptr, 0.f,
                            0, mtp_tiled(cfg, w, MP_LM_HEAD)));
        if (logits_out && st == n_steps - 1) {
            GemmArgs gl = mtp_proj(cfg, w, MP_LM_HEAD);
            gl.At = mtp_tiled(cfg, w, MP_LM_HEAD);
            gl.X = W.xp_head;
            gl.ldx = H;
            gl.T = B;
            gl.epi = EPI_STORE;
            gl.out = logits_out;
            gl.ldo = cfg->vocab;
            gl.name = "gemm_logits";
            DF_TRY(launch_gemm_tc(gl, W.tc, s));
        }
    }
    return launch_seq_advance(cache->seq_len, nullptr, B, n_steps, cache->cap, d_status, s);
}

}  // namespace
}  // namespace df

extern "C" {

int mtp_forward_draft(const df_mtp_config *cfg, const df_mtp_weights *w,
                      const df_kv_cache *cache, const float *prev_hidden, const int32_t *token,
                      int B, int n_steps, float *hidden_out, int32_t *argmax_out,
                      float *logits_out, void *ws, size_t ws_bytes, int32_t *d_status,
                      df_stream_t stream) {
    g_err[0] = 0;
    return mtp_impl(cfg, w, cache, prev_hidden, token, B, n_steps, hidden_out, argmax_out,
                    logits_out, 0.f, nullptr, ws, ws_bytes, d_status, stream);
}

int mtp_forward_draft_sampled(const df_mtp_config *cfg, const df_mtp_weights *w,
                              const df_kv_cache *cache, const float *prev_hidden,
                              const int32_t *token, int B, int n_steps, float temperature,
                              const float *u_draft, float *hidden_out, int32_t *draft_out,
                              float *logits_out, void *ws, size_t ws_bytes, int32_t *d_status,
                              df_stream_t stream) {
    g_err[0] = 0;
    REQ(temperature > 0.f, DF_EINVAL, "temperature=%g (temperature 0 is mtp_forward_draft)",
        (double)temperature);
    return mtp_impl(cfg, w, cache, prev_hidden, token, B, n_steps, hidden_out, draft_out,
                    logits_out, temperature, u_draft, ws, ws_bytes, d_status, stream);
}

size_t df_moe_workspace_bytes(const df_mtp_config *cfg, int T) {
    if (check_mtp_cfg(cfg) != DF_OK || cfg->n_experts == 0 || T <= 0 || T > kMoeMaxRows) return 0;
    Carve cv{nullptr, 0, ~size_t(0), true};
    MoeWs m;
    carve_moe(cv, m, cfg, T);
    return cv.off;
}

int df_moe_ffn(const df_mtp_config *cfg, const df_mtp_weights *w, const float *x, int T,
               float *out, int32_t *expert_ids, float *expert_w, void *ws, size_t ws_bytes,
               int32_t *d_status, df_stream_t stream) {
    g_err[0] = 0;
    DF_TRY(check_mtp_cfg(cfg));
    REQ(cfg->n_experts > 0, DF_EINVAL, "df_moe_ffn: the config has no experts");
    REQ(w, DF_EINVAL, "MTP weights is NULL");
    DF_TRY(check_moe_weights(w));
    REQ(T >= 1 && T <= kMoeMaxRows, DF_ESHAPE, "df_moe_ffn: T=%d (1 <= T <= %d)", T, kMoeMaxRows);
    REQ(x && out, DF_EINVAL, "df_moe_ffn: NULL x or out");
    REQ(reinterpret_cast<uintptr_t>(x) % 16 == 0, DF_EINVAL, "df_moe_ffn: x not 16-byte aligned");
    DF_TRY(get_ws(ws, ws_bytes, df_moe_workspace_bytes(cfg, T)));
    Carve cv{static_cast<char *>(ws), 0, ws_bytes, true};
    MoeWs m;
    carve_moe(cv, m, cfg, T);
    cudaStream_t s = (cudaStream_t)stream;
    MoeArgs a = moe_args(cfg, w, m, x, T, d_status);
    if (expert_ids) a.sel = expert_ids;
    if (expert_w) a.wts = expert_w;
    DF_TRY(launch_moe(a, s));
    PackArgs p;   // out = sum of the top_k + 1 slot outputs, in slot order
    p.part = m.part;
    p.n_part = cfg->top_k + 1;
    p.part_stride = (size_t)T * cfg->hidden;
    p.ldpart = cfg->hidden;
    p.h_out = out;
    p.ldh = cfg->hidden;
    p.T = T;
    p.K = cfg->hidden;
    return launch_pack(p, s);
}

}  // extern "C"

// ================================================================ fixed-scratch lm_head
// Helpers of lm_head_argmax_noalloc (noalloc.cu): the same steps as lm_head_argmax with the
// scratch carved from a caller-given region instead of a workspace argument.
namespace df {

// The lm_head argmax with its scratch at `scratch` and a grid of `ctas` CTAs.
int lm_head_run(const uint16_t *W, const float *X, int rows, int H, int V, int32_t *idx,
                float *top1, float *top2, char *scratch, size_t scratch_bytes, int ctas,
                bool zero_counters, cudaStream_t s) {
    g_err[0] = 0;
    DF_TRY(check_bf16(W, "W"));
    DF_TRY(check_f32(X, "X"));
    REQ(idx, DF_EINVAL, "idx is NULL");
    Carve cv{scratch, 0, scratch_bytes, true};
    uint16_t *xp = cv.take<uint16_t>((size_t)2 * rows * H);
    ArgTop *part = cv.take<ArgTop>((size_t)ctas * rows);
    TcScratch tc;
    carve_tc(cv, tc, rows, V, ctas);
    REQ(cv.ok, DF_EWORKSPACE, "scratch of %zu bytes is too small", scratch_bytes);
    if (zero_counters) {
        cudaError_t e = cudaMemsetAsync(tc.counters, 0, sizeof(int) * (size_t)tc.n_counters, s);
        if (e != cudaSuccess) return fail(DF_ECUDA, "clearing tile counters: %s", cudaGetErrorString(e));
    }
    PackArgs p;
    p.src = X;
    p.lds = H;
    p.pack = xp;
    p.ldp = H;
    p.T = rows;
    p.K = H;
    DF_TRY(launch_pack(p, s));
    return lm_head_impl(W, xp, rows, H, V, part, idx, top1, top2, tc, s);
}

}  // namespace df

// Internal declarations shared by the library's translation units (not part of the ABI).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <utility>

#include "dflash.h"

namespace df {

// ---------------------------------------------------------------- host-side errors
int fail(int code, const char *fmt, ...);   // records the message, returns code
// Kernel launch bookkeeping: prof_begin() before a launch and cuda_check() after it record
// profiling events on the launching stream (when enabled), count launches, and map a failed
// launch to DF_ECUDA.
void prof_begin(cudaStream_t s);
int cuda_check(const char *what, cudaStream_t s);

#define DF_TRY(expr)                 \
    do {                             \
        int df_rc_ = (expr);         \
        if (df_rc_ != DF_OK) return df_rc_; \
    } while (0)

// SMs of the current device (queried once per device; kDefaultSMs, GB300's count, when no device
// is visible, e.g. for workspace-size queries on a machine without a GPU). Grids, split counts,
// scratch sizes and the attention chunk plan are derived from it, so a workspace sized on one
// device is checked again against the device it runs on.
constexpr int kDefaultSMs = 152;
int sm_count();

// ---------------------------------------------------------------- launches
// Every kernel is launched with programmatic dependent launch: it may start while its
// predecessor on the stream is still running, does only work that reads no predecessor output
// (weight prefetch, barrier and TMEM set-up) before pdl_wait(), and lets its own successor
// launch early with pdl_trigger(). Every kernel executes pdl_wait() before touching memory that
// another kernel writes, so completion stays transitive along the stream.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

bool pdl_enabled();
// One-time per (kernel, device): dynamic shared memory limit and a max-shared carveout, so SMs
// keep one L1/shared split across the kernels of a round.
void prepare_kernel(const void *func, int dyn_smem);

template <typename... KArgs, typename... Args>
int launch_k(const char *name, void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
             cudaStream_t s, Args &&...args) {
    prepare_kernel(reinterpret_cast<const void *>(kernel), (int)smem);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl_enabled() ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    prof_begin(s);
    cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
    return cuda_check(name, s);
}

// launch_k with a thread-block cluster of cluster_x CTAs along x (grid.x a multiple of it).
template <typename... KArgs, typename... Args>
int launch_kc(const char *name, void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
              int cluster_x, cudaStream_t s, Args &&...args) {
    prepare_kernel(reinterpret_cast<const void *>(kernel), (int)smem);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl_enabled() ? 1 : 0;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = (unsigned)cluster_x;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    prof_begin(s);
    cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
    return cuda_check(name, s);
}

// ---------------------------------------------------------------- device helpers
__device__ __forceinline__ float bf16_bits_to_f32(uint32_t b) { return __uint_as_float(b << 16); }

// Round-to-nearest-even F32 -> BF16 bits.
__device__ __forceinline__ uint16_t f32_to_bf16_bits(float f) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

// Split y into hi = bf16(y) and lo = bf16(y - hi); hi + lo carries ~16 mantissa bits of y and
// is exactly representable in F32.
__device__ __forceinline__ void split_hi_lo(float y, uint16_t &hi, uint16_t &lo) {
    hi = f32_to_bf16_bits(y);
    lo = f32_to_bf16_bits(y - bf16_bits_to_f32(hi));
}

__device__ __forceinline__ void set_status(int32_t *st, int code) {
    if (st) atomicCAS(st, 0, code);
}

// Trace builds (build.py --trace: -DDF_TRACE=1 with relocatable device code, a separate
// libdflash_trace.so): every kernel's CTAs record (kernel id, SM, start, end) in nanoseconds of
// the global timer into one device buffer, read back by df_trace_read; the launches of a CUDA
// graph replay can then be timed one by one, overlap included. Normal builds record nothing.
#ifndef DF_TRACE
#define DF_TRACE 0
#endif
enum TraceKid : uint32_t {
    TK_ROPE_TABLE = 1, TK_QK_ROPE, TK_ATTN, TK_ATTN_COMBINE, TK_SEQ_ADVANCE, TK_ATTN_TC,
    TK_LOOP_INIT, TK_LOOP_PREPARE, TK_LOOP_VERIFY, TK_LOOP_APPEND, TK_LOOP_COMMIT, TK_MOE_ROUTER,
    TK_MOE_GATE_UP, TK_MOE_DOWN, TK_PACK, TK_PACK_VEC, TK_ARGMAX_FINAL, TK_ACCEPT, TK_ROLLBACK,
    TK_WORD_COPY, TK_SAMPLE_STATS, TK_SAMPLE_WALK, TK_SAMPLE_NORM, TK_SAMPLE_DRAW,
    TK_SAMPLE_FUSED, TK_TILE,
    TK_GEMM = 100   // + 2 * epilogue + (stream-K fix-up ? 1 : 0)
};
struct TraceRec {
    uint32_t kid, sm;
    unsigned long long t0, t1;
};
constexpr unsigned kTraceMax = 1u << 20;
constexpr uint32_t kTraceMark = 1000;   // kids of DF_TRACE_MARK points: kTraceMark + phase
// Phases: attention 1 (past the wait), 2 (Q operand written), 7 (score MMAs issued), 6 (score
// MMAs done, warp 0), 15 (the same, warp 15), 10 (first score tile read from TMEM), 14 (row
// maxima of warp 0 reduced), 3 (row maxima of all warps), 0 (first tile's scores read again), 8
// (first P operand written), 4 (all P operands), 5 (P.V done), 9 (partial outputs stored);
// streamed attention, tile 4: 16 (its iteration starts), 17 (K of tile 5 converted), 18 (V of
// tile 4 converted), 19 (its scores ready), 20 (its row maxima), 21 (P.V of tile 3 done), 22 (its
// P operand written), and 23 (the iteration of tile 5 starts); inside those two conversions (the
// ids of the one-pass points, which a streamed launch never reaches) 3, 4, 5 (K of tile 5: copy
// landed, its TMEM region free, converted) and 7, 8, 0 (the same for V of tile 4), and the TMA
// warp's issue of those two units, 14 / 6 (K: before / after) and 15 / 10 (V); projection 11
// (producer past the wait), 12 (an accumulator ready), 13 (epilogue done).
#if DF_TRACE
extern __device__ TraceRec g_trace[kTraceMax];
extern __device__ unsigned g_trace_n;
__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ uint32_t sm_id() {
    uint32_t v;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(v));
    return v;
}
// Records the CTA's span when thread 0 leaves the kernel (its destructor runs at every return),
// followed by the CTA's trace marks: points inside the kernel that any one thread stamps into a
// shared-memory slot per phase (no global traffic until the end, so marking barely perturbs the
// kernel); a mark stamped twice keeps the later time. Marks are stamped only after the kernel's
// first CTA-wide barrier, which orders them after the slots are cleared.
constexpr int kTraceMarks = 24;
struct TraceScope {
    unsigned long long t0;
    uint32_t kid;
    unsigned long long *marks;
    __device__ TraceScope(uint32_t k, unsigned long long *m) : t0(global_ns()), kid(k), marks(m) {
        if (threadIdx.y == 0 && threadIdx.x < kTraceMarks) m[threadIdx.x] = 0ull;
    }
    __device__ ~TraceScope() {
        if (threadIdx.x == 0 && threadIdx.y == 0) {
            unsigned n = 0;
            for (int p = 0; p < kTraceMarks; ++p) n += marks[p] != 0ull;
            const unsigned i = atomicAdd(&g_trace_n, 1u + n);
            const uint32_t cta = blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z);
            if (i < kTraceMax) g_trace[i] = TraceRec{kid, sm_id(), t0, global_ns()};
            unsigned j = i + 1;
            for (int p = 0; p < kTraceMarks; ++p)
                if (marks[p] != 0ull) {
                    if (j < kTraceMax) g_trace[j] = TraceRec{kTraceMark + p, cta, marks[p], 0ull};
                    ++j;
                }
        }
    }
};
#define DF_TRACE_KERNEL(kid)                                          \
    __shared__ unsigned long long df_trace_marks_[::df::kTraceMarks]; \
    ::df::TraceScope df_trace_scope_((uint32_t)(kid), df_trace_marks_)
#define DF_TRACE_MARK(who, phase)                              \
    do {                                                       \
        if (who) df_trace_marks_[(phase)] = ::df::global_ns(); \
    } while (0)
#else
#define DF_TRACE_KERNEL(kid) \
    do {                     \
    } while (0)
#define DF_TRACE_MARK(who, phase) \
    do {                          \
    } while (0)
#endif

// Debug builds (build.py --debug: -DDF_DEBUG=1, a separate libdflash_debug.so) check the
// indices of stores whose positions come from device data or from index arithmetic over a
// launch's geometry; a failed check writes DF_EINVAL to the call's status word and the access
// is skipped. In normal builds the check is compiled out (always true).
#ifndef DF_DEBUG
#define DF_DEBUG 0
#endif
__device__ __forceinline__ bool df_in_bounds(bool ok, int32_t *status) {
#if DF_DEBUG
    if (!ok) set_status(status, DF_EINVAL);
    return ok;
#else
    (void)status;
    return true;
#endif
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) v += __shfl_xor_sync(0xffffffffu, v, m);
    return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, m));
    return v;
}

// Streaming 128-bit load that does not allocate in L1 (weights are read once per call).
__device__ __forceinline__ uint4 ld_stream_u4(const void *p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

// Argmax state: best value, its index, and the second-largest value.
struct ArgTop {
    float v1;
    int i1;
    float v2;
};

__device__ __forceinline__ ArgTop argtop_empty(int big_index) { return {-INFINITY, big_index, -INFINITY}; }

// Merge two states; the lower index wins an exact tie of the best value.
__device__ __forceinline__ ArgTop argtop_merge(ArgTop a, ArgTop b) {
    bool b_wins = (b.v1 > a.v1) || (b.v1 == a.v1 && b.i1 < a.i1);
    ArgTop r;
    r.v1 = b_wins ? b.v1 : a.v1;
    r.i1 = b_wins ? b.i1 : a.i1;
    float lo = b_wins ? a.v1 : b.v1;           // the loser's best
    r.v2 = fmaxf(lo, fmaxf(a.v2, b.v2));
    return r;
}

__device__ __forceinline__ ArgTop argtop_push(ArgTop a, float v, int i) {
    ArgTop b = {v, i, -INFINITY};
    return argtop_merge(a, b);
}

// ---------------------------------------------------------------- workspace carving
struct Carve {
    char *base;
    size_t off, cap;
    bool ok;
    template <class T>
    T *take(size_t count) {
        size_t bytes = (count * sizeof(T) + 255) & ~size_t(255);
        if (off + bytes > cap) ok = false;
        T *p = ok && base ? reinterpret_cast<T *>(base + off) : nullptr;
        off += bytes;
        return p;
    }
};

// ---------------------------------------------------------------- kernels (launchers)

// Packed activation layout: for token t of a GEMM input, row 2t holds bf16(y) and row 2t+1
// holds bf16(y - bf16(y)), both [K] BF16 with leading dimension ldp (elements).
struct PackArgs {
    const float *src = nullptr;      // F32 rows [T, K], row stride lds
    int lds = 0;
    const uint16_t *gather = nullptr;  // gather mode: rows embed[ids[t]] (BF16) instead of src
    const int32_t *ids = nullptr;
    const int32_t *last_token = nullptr;  // gather mode alternative: id = i == 0 ? last[b] : mask
    int mask_id = 0;
    int vocab = 0;
    float scale = 1.f;
    float *h_out = nullptr;          // optional raw (gathered) rows, row stride ldh
    int ldh = 0;
    const float *norm_w = nullptr;   // optional RMSNorm weight
    float eps = 0.f;
    float *y_out = nullptr;          // optional normalised rows, row stride ldy
    int ldy = 0;
    uint16_t *pack = nullptr;        // optional packed output
    int ldp = 0;
    int T = 0, K = 0;
    const int32_t *nvalid = nullptr; // rows t = s*rows_per_seq + j are valid iff j < nvalid[s]
    int rows_per_seq = 1;
    int32_t *status = nullptr;
    // Optional deferred split-K sums added to the row after src, in split order:
    // x[t, k] = src[t, k] + part[0][t, k] + ... + part[n_part-1][t, k]
    const float *part = nullptr;
    int n_part = 0;
    size_t part_stride = 0;          // floats between splits
    int ldpart = 0;                  // floats between rows of one split
    // Deferred RMSNorm (needs norm_w and pack, no y_out): the row is split over pack_slices(K)
    // CTAs without a cluster; pack receives x * norm_w (the numerator only) and ss_out[t * L + j]
    // the sum of x^2 over slice j of row t, L = ss_ld (pack_slices(K) when 0; slots past the
    // slices are written as zeros). The 1/rms factor is applied by the consuming projection as
    // a row scale (GemmArgs::rs_*), which the linearity of the projection allows.
    float *ss_out = nullptr;
    int ss_ld = 0;
    // Optional side job of CTA 0: seq_len[b] += n_new[b] for b < adv_B (capacity-checked as
    // launch_seq_advance), when nothing later in the stream reads the old lengths.
    int32_t *adv_seq = nullptr;
    const int32_t *adv_n = nullptr;
    int adv_B = 0, adv_cap = 0;
};
int launch_pack(const PackArgs &a, cudaStream_t s);
// Number of CTAs (slices) a row of K elements is split over by the row prologue.
int pack_slices(int K);

// Mixture-of-experts FFN (router, top-k, routed + shared expert SwiGLUs) over T <= 16 rows.
constexpr int kMoeMaxRows = 16;
constexpr int kMoeMaxExperts = 512;
constexpr int kMoeMaxTopK = 16;
struct MoeArgs {
    const float *x = nullptr;        // [T, H] F32 normalised rows, row stride ldx (16-byte aligned)
    int ldx = 0;
    int T = 0, H = 0, E = 0, k = 0, Ie = 0, Is = 0;
    const uint16_t *router = nullptr, *sh_gate = nullptr;          // [E, H], [1, H]
    const uint16_t *exp_gate = nullptr, *exp_up = nullptr;         // [E, Ie, H]
    const uint16_t *exp_down = nullptr;                            // [E, H, Ie]
    const uint16_t *sh_g = nullptr, *sh_u = nullptr, *sh_d = nullptr;  // [Is, H] x2, [H, Is]
    float *logits = nullptr;         // [T, E + 1] scratch
    int32_t *sel = nullptr;          // [T, k] chosen experts, largest weight first
    float *wts = nullptr;            // [T, k + 1]: renormalised weights, then sigmoid(shared gate)
    float *act = nullptr;            // [T, k + 1, max(Ie, Is)] SwiGLU activations
    float *part = nullptr;           // [k + 1, T, ldpart] weighted per-slot outputs
    int ldpart = 0;
    int *counter = nullptr;          // zero before the call, left zero
    int32_t *status = nullptr;
};
int launch_moe(const MoeArgs &a, cudaStream_t s);

enum Epi { EPI_STORE = 0, EPI_RESID = 1, EPI_SWIGLU = 2, EPI_ARGMAX = 3 };

struct GemmArgs {
    // Weight rows (BF16 [rows, K] row-major). Up to four segments concatenated along the
    // output dimension: rows [0,n0) of W0, then n1 rows of W1, n2 of W2, n3 of W3.
    // EPI_SWIGLU pairs row j of W0 (gate) with row j of W1 (up): N = n0 = n1.
    const uint16_t *W0 = nullptr, *W1 = nullptr, *W2 = nullptr, *W3 = nullptr;
    int n0 = 0, n1 = 0, n2 = 0, n3 = 0;
    // Optional split along K for segment 0: columns [K1, K) read from Wk2 [n0, K-K1].
    const uint16_t *Wk2 = nullptr;
    int K1 = 0;
    // Optional tiled copy of the same weights (tile_projection): when set the kernel reads its
    // A operands from it, two K blocks per bulk copy; W0.. still define the shape.
    const uint8_t *At = nullptr;
    int N = 0, K = 0;
    const uint16_t *X = nullptr;     // packed activations [2T, ldx]
    int ldx = 0, T = 0;
    const uint16_t *X2 = nullptr;    // with Wk2: packed activations of columns [K1, K)
    int ldx2 = 0;
    int32_t *status = nullptr;
    const char *name = "gemm_tc_kernel";   // label in launch profiles
    // Deferred split-K (EPI_STORE only): the output is S partial sums, split s of token t at
    // out[s * part_stride + t * ldo + n]; the consuming kernel adds them in split order.
    // The number of splits S is returned through launch_gemm_tc's n_partials_out.
    int defer = 0;
    size_t part_stride = 0;
    int epi = EPI_STORE;
    float *out = nullptr;            // EPI_STORE / EPI_RESID: out[t*ldo + n]
    int ldo = 0;
    const float *resid = nullptr;    // EPI_RESID: resid[t*ldr + n] (may alias out)
    int ldr = 0;
    uint16_t *pack_out = nullptr;    // EPI_SWIGLU: packed [2T, ldpo]
    int ldpo = 0;
    ArgTop *part = nullptr;          // EPI_ARGMAX: partial states [grid, T]
    int *n_part = nullptr;           // EPI_ARGMAX: host-visible count of partial rows written
    // Row scale of the outputs (any epilogue): rows t < rs_rows are multiplied by
    // 1 / sqrt((rs_ss[t*rs_n] + ... + rs_ss[t*rs_n + rs_n-1]) * rs_inv_k + rs_eps), the partial
    // sums taken in order: the RMSNorm factor of an input row whose numerator x * w was packed
    // by a deferred-norm row prologue. Rows at or past rs_rows are left as they are.
    const float *rs_ss = nullptr;
    int rs_n = 0, rs_rows = 0;
    float rs_inv_k = 0.f, rs_eps = 0.f;
};

// Scratch of the tensor-core projections: partial tiles of tiles shared by several CTAs, and
// one arrival counter per tile (zero between calls).
constexpr int kMaxTcTokens = 128;
struct TcScratch {
    float *partials = nullptr;
    size_t partial_floats = 0;
    int *counters = nullptr;
    int n_counters = 0;
    int max_ctas = 0;        // CTAs of a launch (set by the carve)
};
// Byte size of a carve of `bytes` (every carve starts on a 256-byte boundary).
constexpr size_t carve_round(size_t bytes) { return (bytes + 255) & ~size_t(255); }
// Partial tiles of a stream-K projection over at most max_tokens tokens with `ctas` CTAs.
constexpr size_t tc_partial_floats(int max_tokens, int ctas) {
    return (size_t)ctas * 2 * 128 *
           (size_t)((max_tokens < kMaxTcTokens ? max_tokens : kMaxTcTokens) > 0
                        ? (max_tokens < kMaxTcTokens ? max_tokens : kMaxTcTokens)
                        : 1);
}
// Arrival counters of a projection with at most max_rows output rows.
constexpr int n_counters_for(long long max_rows) { return (int)(max_rows / 64 + 256); }
// Bytes of the scratch of an lm_head argmax over `rows` rows with `ctas` CTAs: packed rows, the
// per-CTA argmax partials, the projection's partial tiles and counters (carved in this order).
constexpr size_t lm_head_scratch_bytes_for(int rows, int H, int V, int ctas) {
    return carve_round((size_t)2 * rows * H * 2) + carve_round((size_t)ctas * rows * sizeof(ArgTop)) +
           carve_round(tc_partial_floats(rows, ctas) * 4) + carve_round((size_t)n_counters_for(V) * 4);
}
// Tiled weight layout of a projection (the A operands of GemmArgs a: its segments, K split and
// SwiGLU pairing): 128-row x 64-column BF16 tiles, tile (m, kb) at byte (m * kbt + kb) * 16384,
// each stored exactly as the 128-byte-swizzled shared-memory image the MMA reads (row r at
// r * 128, its 16-byte piece j at ((j ^ (r % 8)) * 16)), rows and columns past the matrix zero.
size_t tiled_projection_bytes(const GemmArgs &a);
int tile_projection(const GemmArgs &a, uint8_t *out, size_t out_bytes, cudaStream_t s);
int launch_gemm_tc(const GemmArgs &a, const TcScratch &sc, cudaStream_t s,
                   int *n_partials_out = nullptr);


// Reduce EPI_ARGMAX partials [G, T] into idx/top1/top2 [T].
int launch_argmax_final(const ArgTop *part, int G, int T, int32_t *idx, float *top1,
                        float *top2, int32_t *idx_copy, int idx_copy_ld, int idx_copy_skip,
                        cudaStream_t s);

// RoPE table: cos/sin F32 [B, slots, rot/2] for block slots (pos = seq_len + n_new + i + off)
// and context slots (pos = seq_len + j).
constexpr int kMaxRopeHalf = 128;   // rotary dims up to 256
int launch_rope_table(float *cos_t, float *sin_t, const int32_t *seq_len, const int32_t *n_new,
                      int n_new_max, int B, int blk, int pos_off, int rot, float theta,
                      int32_t *status, cudaStream_t s);

struct QkArgs {
    const float *qkv;        // [T_blk + T_ctx, ldq] raw projections (q | k | v)
    int ldq;
    int B, blk, n_new_max;
    int nq, nkv, d, rot;
    const float *q_norm, *k_norm;   // may be null (no per-head norm)
    float eps;
    const float *cos_t, *sin_t;     // [B, blk + n_new_max, rot/2]
    float *q_out;                   // [B, blk, nq, d]
    float *kb, *vb;                 // [B, nkv, blk, d] (block K/V) or null
    float *cache_k, *cache_v;       // [B, nkv, cap, d]
    int cap;
    const int32_t *seq_len, *n_new;
    int append_block;               // 1: block rows are appended to the cache (MTP)
    int pos_off;                    // added to block positions (MTP chained step)
    int32_t *status;
    // Deferred split-K: when part is set the projections are the sum of n_part splits
    // part[s * part_stride + row * ldq + col] instead of qkv.
    const float *part = nullptr;
    int n_part = 0;
    size_t part_stride = 0;
    // Optional sigmoid-gate pre-activations (n_gate_heads heads after q|k|v, block rows only),
    // reduced like q/k/v and stored to gate_out[row * ldg + h * d + e].
    int n_gate_heads = 0;
    float *gate_out = nullptr;
    int ldg = 0;
    int kv_bf16 = 0;         // cache_k/cache_v hold BF16; block K/V rounded to BF16 values
};
int launch_qk_rope(const QkArgs &a, cudaStream_t s);

struct AttnArgs {
    const float *q;          // [B, blk, nq, d]
    const float *cache_k, *cache_v;   // [B, nkv, cap, d]
    int cap;
    const float *kb, *vb;    // [B, nkv, blk, d] block keys or null
    int B, blk, nq, nkv, d;
    const int32_t *seq_len, *n_new;   // cache rows visible: seq_len + n_new (+ extra)
    int n_new_max;
    int extra_rows;          // rows beyond seq_len + n_new that are visible (MTP: step + 1)
    int causal_block;
    float *part;             // [B, nkv, n_chunks, R, d + 2] per-CTA partial (o, m, l)
    int n_chunks, chunk;     // key chunks per (sequence, KV head); keys per chunk
    int tc;                  // 1: tensor-core kernel (chunk a multiple of 128 keys)
    int kv_bf16;             // cache_k/cache_v hold BF16 (tensor-core kernel only)
    const float *gate;       // optional [B*blk, ldg] gate pre-activation (q_total wide)
    int ldg;
    uint16_t *pack;          // packed output [2*B*blk, nq*d] (or null)
    float *out;              // F32 output [B*blk, nq*d] (or null)
    int32_t *status;
    // 1: seq_len is not written by any kernel of the same stream before this one (the DFlash
    // forward advances it only at its end), so cache rows below it may be loaded before the
    // wait for the preceding kernel.
    int early_kv;
};
void attn_plan(AttnArgs &a, int max_keys);
size_t attn_part_floats(const AttnArgs &a);
int launch_attn(const AttnArgs &a, cudaStream_t s);
bool attn_tc_supported(int d, int rows);
int launch_attn_tc(const AttnArgs &a, cudaStream_t s);

// Non-greedy path over B sequences of K drafts and vocab V: drafts drawn from the drafter's
// softmax (sample mode) and the speculative-sampling accept step (accept mode).
constexpr int kSampleMaxK = 64;
struct MaxSum {
    float m, s;              // max of x, sum of exp(x - m)
};
struct SampleState {
    int acc;                 // accepted drafts
    float mp, mq;            // row maxima (x units) of the rows the committed token is drawn from
};
struct SampleArgs {
    const float *draft = nullptr;    // drafter logits: row i of sequence b at (b * draft_ld + i) * V
    int draft_ld = 0;                // rows between sequences (K for a [B, K, V] tensor)
    const float *target = nullptr;   // [B, K+1, V] verifier logits (positions 0..K)
    int V = 0, B = 0, K = 0;
    float T = 1.f;                   // temperature > 0
    float scale = 1.f;               // log2(e) / T
    // float-float constants of the draw weights (sample_constants): log2(e) / T, ln 2, and
    // 2^(k/32) for k = -16..16
    float sc_hi = 0.f, sc_lo = 0.f, ln2_hi = 0.f, ln2_lo = 0.f;
    float2 exp2_tab[33] = {};
    int sample_mode = 0;             // 1: draw drafts [B, K] from the drafter rows
    const float *u_draft = nullptr;  // sample mode: [B, K] uniforms in [0, 1)
    int32_t *drafts_out = nullptr;   // sample mode: [B, K]
    const int32_t *drafts = nullptr; // accept mode: [B, K]
    const float *u_accept = nullptr; // [B, K] uniforms in [0, 1)
    const float *u_sample = nullptr; // [B]
    const int32_t *eos = nullptr;
    int n_eos = 0;
    int32_t *committed = nullptr, *n_committed = nullptr, *accept_count = nullptr;
    int32_t *hit_eos = nullptr, *rollback = nullptr;
    int n_chunks = 0;
    MaxSum *stats = nullptr;         // [B, 2K+1, n_chunks] (sample mode: [B, K, n_chunks])
    SampleState *state = nullptr;    // [B]
    float2 *dsum = nullptr;          // [B, n_chunks, 2]: exp sums of the draw's p and q rows (hi, lo)
    float2 *csum = nullptr;          // [B * K, n_chunks]: draw weights per chunk (hi, lo)
    int *counters = nullptr;         // [B * K], zero between calls
    int32_t *status = nullptr;
};
int sample_chunks(int V);
// Scratch of either mode for B sequences of K drafts: carved in this order by the callers.
void carve_sample_scratch(Carve &cv, SampleArgs &a, int B, int K, int V);
// scale and the float-float constants from a.T (> 0)
void sample_constants(SampleArgs &a);
int launch_accept_stochastic(const SampleArgs &a, cudaStream_t s);
int launch_sample_drafts(const SampleArgs &a, cudaStream_t s);

// Multi-round generate loop around the draft round (k_loop.cu).
constexpr int kLoopMaxTargetLayers = 16;
struct LoopArgs {
    // synthetic verifier
    const int32_t *ref = nullptr;        // [B, max_len]
    const uint8_t *agree = nullptr;      // [B, max_len] or null
    const float *table = nullptr;        // [B, n_comb, max_len, H]
    int n_comb = 0;
    int sel[kLoopMaxTargetLayers] = {};  // drafter target layer l = captured layer sel[l]
    int max_len = 0;
    // caller state
    float *prior_cap = nullptr;          // [B, n_comb, max_len, H]
    int32_t *prior_len = nullptr, *out = nullptr, *out_len = nullptr;
    const int32_t *prompt_len = nullptr;
    int32_t *rounds = nullptr, *accept_hist = nullptr;
    int max_rounds = 0, max_new = 0;
    int32_t *cache_seq = nullptr;        // drafter cache lengths
    int B = 0, K = 0, H = 0, n_tl = 0, n_new_max = 0;
    // round scratch
    float *th = nullptr;                 // [B, n_new_max, n_tl * H]
    int32_t *n_new = nullptr, *last_token = nullptr, *argmax = nullptr, *target = nullptr;
    int32_t *committed = nullptr, *n_committed = nullptr, *accept = nullptr, *hit = nullptr;
    int32_t *rollback = nullptr, *done = nullptr, *round_ctr = nullptr;
    const int32_t *eos = nullptr;
    int n_eos = 0;
    cudaGraphConditionalHandle cond = 0;
    int32_t *status = nullptr;
};
int launch_loop_init(const LoopArgs &a, cudaStream_t s);
int launch_loop_prepare(const LoopArgs &a, cudaStream_t s);
int launch_loop_verify(const LoopArgs &a, cudaStream_t s);
int launch_loop_append(const LoopArgs &a, cudaStream_t s);
int launch_loop_commit(const LoopArgs &a, cudaStream_t s);

int launch_seq_advance(int32_t *seq_len, const int32_t *n_new, int B, int delta, int cap,
                       int32_t *status, cudaStream_t s);
// Up to 12 copies of 32-bit words (device <-> device-addressable page-locked host memory).
struct WordCopyList {
    const void *src[12] = {};
    void *dst[12] = {};
    int words[12] = {};
    int n = 0;
};
int launch_word_copy(const WordCopyList &l, cudaStream_t s);
int launch_accept(const int32_t *drafts, int ld, const int32_t *target, int B, int K,
                  const int32_t *eos, int n_eos, int32_t *committed, int32_t *n_committed,
                  int32_t *accept_count, int32_t *hit_eos, int32_t *rollback,
                  int32_t *target_seq_len, int32_t *status, cudaStream_t s);
int launch_rollback(int32_t *seq_len, const int32_t *n, int B, int32_t *status, cudaStream_t s);
// argmax_final + accept in one launch for blocks of 2..32 rows (one CTA per sequence).
int launch_argmax_accept(const ArgTop *part, int G, int B, int blk, int32_t *argmax_out,
                         const int32_t *target, const int32_t *eos, int n_eos,
                         int32_t *committed, int32_t *n_committed, int32_t *accept_count,
                         int32_t *hit_eos, int32_t *rollback, int32_t *target_seq_len,
                         int32_t *status, cudaStream_t s);

}  // namespace df

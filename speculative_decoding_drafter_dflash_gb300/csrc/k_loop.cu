// The multi-round generate loop on the device: the steps around the draft round that
// qwen35_orchestrator.rs runs on the host (`dispatch_qwen35_dflash_generate`, "Multi-round loop
// (Option A)"): the drafter's new context rows gathered from the captured verifier states
// (`extract_drafter_concat`, new rows only), the verify (here a synthetic verifier read from
// tables), appending the committed tokens and updating last_token, the stop on EOS or on the
// token budget, `append_capture_positions` of the committed verify positions, and the final
// truncation to the budget. The round itself (drafter forward, per-position argmax, accept walk)
// runs the library's round kernels between these. The loop is one CUDA graph whose while node
// repeats the round; loop_commit_kernel sets its condition.
#include "df_internal.cuh"

namespace df {

namespace {

__device__ __forceinline__ bool is_eos(const LoopArgs &a, int tok) {
    bool e = false;
    for (int i = 0; i < a.n_eos; ++i) e |= (tok == a.eos[i]);
    return e;
}

// One CTA, a thread per sequence: the page returns at once when the first token is an EOS id
// or the budget is zero; the loop runs while some sequence is active.
__global__ void loop_init_kernel(LoopArgs a) {
    DF_TRACE_KERNEL(TK_LOOP_INIT);
    pdl_trigger();
    pdl_wait();
    bool active = false;
    for (int b = threadIdx.x; b < a.B; b += blockDim.x) {
        const int len = a.out_len[b];
        bool done = a.max_new <= 0 || len < 1 || len > a.max_len;
        if (!done) done = is_eos(a, a.out[(size_t)b * a.max_len + len - 1]);
        if (!done && len + a.K + 2 > a.max_len) {
            set_status(a.status, DF_ECAPACITY);
            done = true;
        }
        a.done[b] = done ? 1 : 0;
        a.rounds[b] = 0;
        active |= !done;
    }
    active = __syncthreads_or(active);
    if (threadIdx.x == 0) {
        *a.round_ctr = 0;
        cudaGraphSetConditional(a.cond, (active && a.max_rounds > 0) ? 1u : 0u);
    }
}

// n_new = prior_len - drafter cache length (the positions the drafter has not consumed), and the
// concatenation of the drafter's target layers for those rows. Grid (B * n_new_max, n_tl).
__global__ void __launch_bounds__(256) loop_prepare_kernel(LoopArgs a) {
    DF_TRACE_KERNEL(TK_LOOP_PREPARE);
    pdl_trigger();
    pdl_wait();
    const int b = blockIdx.x / a.n_new_max, j = blockIdx.x - b * a.n_new_max, l = blockIdx.y;
    const bool active = a.done[b] == 0;
    const int c0 = a.cache_seq[b];
    int nn = active ? a.prior_len[b] - c0 : 0;
    if (nn < 0 || nn > a.n_new_max) {
        if (threadIdx.x == 0 && j == 0 && l == 0) set_status(a.status, DF_ESHAPE);
        nn = min(max(nn, 0), a.n_new_max);
    }
    if (j == 0 && l == 0 && threadIdx.x == 0) {
        a.n_new[b] = nn;
        const int len = a.out_len[b];
        a.last_token[b] = a.out[(size_t)b * a.max_len + max(len - 1, 0)];
    }
    if (j >= nn) return;
    const float *src = a.prior_cap + (((size_t)b * a.n_comb + a.sel[l]) * a.max_len + c0 + j) * a.H;
    float *dst = a.th + ((size_t)b * a.n_new_max + j) * ((size_t)a.n_tl * a.H) + (size_t)l * a.H;
    for (int h = threadIdx.x; h < a.H; h += blockDim.x) dst[h] = src[h];
}

// Synthetic verifier: its greedy token after verify position p0 + j is the draft x_j where it
// agrees (j < K), else ref[p0 + j + 1]. Grid B, K+1 threads or more.
__global__ void loop_verify_kernel(LoopArgs a) {
    DF_TRACE_KERNEL(TK_LOOP_VERIFY);
    pdl_trigger();
    pdl_wait();
    const int b = blockIdx.x;
    const int p0 = a.out_len[b] - 1;
    for (int j = threadIdx.x; j <= a.K; j += blockDim.x) {
        const int p = min(max(p0 + j, 0), a.max_len - 2);
        int t = a.ref[(size_t)b * a.max_len + p + 1];
        if (j < a.K && a.agree && a.agree[(size_t)b * a.max_len + p])
            t = a.argmax[(size_t)b * (a.K + 1) + j + 1];
        a.target[(size_t)b * (a.K + 1) + j] = t;
    }
}

__device__ __forceinline__ bool stops(const LoopArgs &a, int b, int len, int n) {
    const int nl = len + n;
    return a.hit[b] != 0 || nl - a.prompt_len[b] >= a.max_new || nl + a.K + 2 > a.max_len;
}

// append_capture_positions: the first n_committed verify positions (p0 .. p0+n-1, the synthetic
// verifier's capture = its table rows) join the captured prefix at prior_len (= p0). Skipped
// when the sequence stops, as the page breaks before this step. Grid (B * (K+1), n_comb).
__global__ void __launch_bounds__(256) loop_append_kernel(LoopArgs a) {
    DF_TRACE_KERNEL(TK_LOOP_APPEND);
    pdl_trigger();
    pdl_wait();
    const int b = blockIdx.x / (a.K + 1), j = blockIdx.x - b * (a.K + 1), c = blockIdx.y;
    if (a.done[b]) return;
    const int len = a.out_len[b], n = a.n_committed[b];
    if (j >= n || stops(a, b, len, n)) return;
    const int p = a.prior_len[b] + j;
    if (p >= a.max_len) return;
    const size_t row = ((size_t)b * a.n_comb + c) * a.max_len + p;
    const float *src = a.table + row * a.H;
    float *dst = a.prior_cap + row * a.H;
    for (int h = threadIdx.x; h < a.H; h += blockDim.x) dst[h] = src[h];
}

// Bookkeeping, one CTA with a thread per sequence: committed tokens appended, lengths, stop
// flags, per-sequence rounds and accept history; then the loop condition.
__global__ void loop_commit_kernel(LoopArgs a) {
    DF_TRACE_KERNEL(TK_LOOP_COMMIT);
    pdl_trigger();
    pdl_wait();
    const int r = *a.round_ctr;
    bool active = false;
    for (int b = threadIdx.x; b < a.B; b += blockDim.x) {
        if (a.done[b]) continue;
        const int len = a.out_len[b], n = a.n_committed[b];
        int32_t *o = a.out + (size_t)b * a.max_len;
        for (int i = 0; i < n && len + i < a.max_len; ++i)
            if (df_in_bounds(len + i >= 0 && i <= a.K, a.status))
                o[len + i] = a.committed[(size_t)b * (a.K + 1) + i];
        const bool stop = stops(a, b, len, n);
        int nl = min(len + n, a.max_len);
        if (stop) {
            nl = min(nl, a.prompt_len[b] + a.max_new);     // truncation to the budget
            a.done[b] = 1;
        } else {
            a.prior_len[b] += n;
            active = true;
        }
        a.out_len[b] = nl;
        a.rounds[b] += 1;
        if (a.accept_hist && r < a.max_rounds) a.accept_hist[(size_t)r * a.B + b] = a.accept[b];
    }
    active = __syncthreads_or(active);
    if (threadIdx.x == 0) {
        *a.round_ctr = r + 1;
        cudaGraphSetConditional(a.cond, (active && r + 1 < a.max_rounds) ? 1u : 0u);
    }
}

}  // namespace

int launch_loop_init(const LoopArgs &a, cudaStream_t s) {
    return launch_k("loop_init_kernel", loop_init_kernel, dim3(1), dim3(256), 0, s, a);
}

int launch_loop_prepare(const LoopArgs &a, cudaStream_t s) {
    return launch_k("loop_prepare_kernel", loop_prepare_kernel, dim3(a.B * a.n_new_max, a.n_tl),
                    dim3(256), 0, s, a);
}

int launch_loop_verify(const LoopArgs &a, cudaStream_t s) {
    return launch_k("loop_verify_kernel", loop_verify_kernel, dim3(a.B), dim3(32), 0, s, a);
}

int launch_loop_append(const LoopArgs &a, cudaStream_t s) {
    return launch_k("loop_append_kernel", loop_append_kernel, dim3(a.B * (a.K + 1), a.n_comb),
                    dim3(256), 0, s, a);
}

int launch_loop_commit(const LoopArgs &a, cudaStream_t s) {
    return launch_k("loop_commit_kernel", loop_commit_kernel, dim3(1), dim3(256), 0, s, a);
}

}  // namespace df

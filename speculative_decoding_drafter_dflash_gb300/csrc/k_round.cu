// Integer tail of the draft round: final argmax reduction, greedy accept walk, KV rollback.
//
// hf2q 0.1.1 spec_decode/dflash/qwen35_orchestrator.rs: step 5 (per-position argmax,
// drafts = argmax[1..]), step 7 (`step_round_from_argmaxes`: accept a draft only while it
// equals the verifier's argmax; the verifier's argmax at accept_count is the free token; stop
// at EOS), step 8 (`rollback = drafts.len() - accept_count`, `rollback_kv`).
#include "df_internal.cuh"

namespace df {

namespace {

// One warp per row: lanes merge strided subsets of the G partial states, then a fixed
// butterfly merges the lanes (the result is independent of the order: the merge keeps the
// largest value, the lowest index among equal values, and the second-largest value).
__global__ void argmax_final_kernel(const ArgTop *part, int G, int T, int32_t *idx, float *top1,
                                    float *top2, int32_t *idx_copy, int ld, int skip) {
    DF_TRACE_KERNEL(TK_ARGMAX_FINAL);
    pdl_trigger();
    pdl_wait();
    const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (t >= T) return;
    ArgTop r = argtop_empty(0x7fffffff);
    for (int g = lane; g < G; g += 32) r = argtop_merge(r, part[(size_t)g * T + t]);
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
        ArgTop b;
        b.v1 = __shfl_xor_sync(0xffffffffu, r.v1, o);
        b.i1 = __shfl_xor_sync(0xffffffffu, r.i1, o);
        b.v2 = __shfl_xor_sync(0xffffffffu, r.v2, o);
        r = argtop_merge(r, b);
    }
    if (lane != 0) return;
    idx[t] = r.i1;
    if (top1) top1[t] = r.v1;
    if (top2) top2[t] = r.v2;
    // Optional copy in a second layout (used to place drafts = rows 1..K of each sequence).
    if (idx_copy) {
        int b = t / ld, i = t % ld;
        if (i >= skip) idx_copy[(size_t)b * (ld - skip) + (i - skip)] = r.i1;
    }
}

// The greedy walk of one sequence over its drafts dr[0..K) and the verifier's argmaxes tg[0..K]:
// accepted prefix, free token, EOS cut, -1 fill, rollback of the verifier's KV length.
__device__ void accept_walk_one(const int32_t *dr, const int32_t *tg, int b, int K,
                                const int32_t *eos, int n_eos, int32_t *committed,
                                int32_t *n_committed, int32_t *accept_count, int32_t *hit_eos,
                                int32_t *rollback, int32_t *target_seq_len, int32_t *status) {
    int a = 0;
    while (a < K && dr[a] == tg[a]) ++a;
    int32_t *out = committed + (size_t)b * (K + 1);
    int n = 0, hit = 0;
    for (int i = 0; i <= a; ++i) {
        int tok = i < a ? dr[i] : tg[a];
        if (!df_in_bounds(n <= K, status)) break;
        out[n++] = tok;
        bool is_eos = false;
        for (int e = 0; e < n_eos; ++e) is_eos |= (tok == eos[e]);
        if (is_eos) {
            hit = 1;
            break;
        }
    }
    for (int i = n; i <= K; ++i) out[i] = -1;
    n_committed[b] = n;
    accept_count[b] = a;
    hit_eos[b] = hit;
    rollback[b] = K - a;
    if (target_seq_len) {
        int rb = K - a;
        if (rb > target_seq_len[b]) set_status(status, DF_ECAPACITY);
        else target_seq_len[b] -= rb;
    }
}

// The round's tail in one launch, one CTA per sequence: warp i merges the lm_head argmax
// partials of block row i (as argmax_final_kernel), then thread 0 walks the drafts (rows 1..K)
// against the verifier's argmaxes.
__global__ void argmax_accept_kernel(const ArgTop *part, int G, int blk, int32_t *argmax_out,
                                     const int32_t *target, const int32_t *eos, int n_eos,
                                     int32_t *committed, int32_t *n_committed,
                                     int32_t *accept_count, int32_t *hit_eos, int32_t *rollback,
                                     int32_t *target_seq_len, int32_t *status) {
    DF_TRACE_KERNEL(TK_ARGMAX_FINAL);
    __shared__ int32_t idx[32];
    pdl_trigger();
    pdl_wait();
    const int b = blockIdx.x, w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int T = gridDim.x * blk;
    if (w < blk) {
        const int t = b * blk + w;
        ArgTop r = argtop_empty(0x7fffffff);
        for (int g = lane; g < G; g += 32) r = argtop_merge(r, part[(size_t)g * T + t]);
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) {
            ArgTop x;
            x.v1 = __shfl_xor_sync(0xffffffffu, r.v1, o);
            x.i1 = __shfl_xor_sync(0xffffffffu, r.i1, o);
            x.v2 = __shfl_xor_sync(0xffffffffu, r.v2, o);
            r = argtop_merge(r, x);
        }
        if (lane == 0) {
            idx[w] = r.i1;
            argmax_out[t] = r.i1;
        }
    }
    __syncthreads();
    if (threadIdx.x == 0)
        accept_walk_one(idx + 1, target + (size_t)b * blk, b, blk - 1, eos, n_eos, committed,
                        n_committed, accept_count, hit_eos, rollback, target_seq_len, status);
}

// One thread per sequence.
__global__ void accept_kernel(const int32_t *drafts, int ld, const int32_t *target, int B, int K,
                              const int32_t *eos, int n_eos, int32_t *committed,
                              int32_t *n_committed, int32_t *accept_count, int32_t *hit_eos,
                              int32_t *rollback, int32_t *target_seq_len, int32_t *status) {
    DF_TRACE_KERNEL(TK_ACCEPT);
    pdl_trigger();
    pdl_wait();
    int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= B) return;
    accept_walk_one(drafts + (size_t)b * ld, target + (size_t)b * (K + 1), b, K, eos, n_eos,
                    committed, n_committed, accept_count, hit_eos, rollback, target_seq_len,
                    status);
}

__global__ void rollback_kernel(int32_t *seq_len, const int32_t *n, int B, int32_t *status) {
    DF_TRACE_KERNEL(TK_ROLLBACK);
    pdl_trigger();
    pdl_wait();
    int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= B) return;
    int k = n[b];
    if (k < 0 || k > seq_len[b]) {
        set_status(status, DF_ECAPACITY);
        return;
    }
    seq_len[b] -= k;
}

// Word copies between device memory and page-locked host memory the device can address (the
// small inputs and outputs of the host-buffer round): one launch instead of one DMA copy each.
__global__ void word_copy_kernel(WordCopyList l) {
    DF_TRACE_KERNEL(TK_WORD_COPY);
    pdl_trigger();
    pdl_wait();
    for (int r = 0; r < l.n; ++r) {
        const uint32_t *src = static_cast<const uint32_t *>(l.src[r]);   // null: zeros
        uint32_t *dst = static_cast<uint32_t *>(l.dst[r]);
        for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < l.words[r]; i += gridDim.x * blockDim.x)
            dst[i] = src ? src[i] : 0u;
    }
}

}  // namespace

int launch_word_copy(const WordCopyList &l, cudaStream_t s) {
    if (l.n <= 0) return DF_OK;
    return launch_k("word_copy_kernel", word_copy_kernel, dim3(1), dim3(256), 0, s, l);
}

int launch_argmax_final(const ArgTop *part, int G, int T, int32_t *idx, float *top1, float *top2,
                        int32_t *idx_copy, int idx_copy_ld, int idx_copy_skip, cudaStream_t s) {
    if (T <= 0) return DF_OK;
    return launch_k("argmax_final_kernel", argmax_final_kernel, dim3((T + 3) / 4), dim3(128), 0, s,
                    part, G, T, idx, top1, top2, idx_copy, idx_copy_ld, idx_copy_skip);
}

int launch_accept(const int32_t *drafts, int ld, const int32_t *target, int B, int K,
                  const int32_t *eos, int n_eos, int32_t *committed, int32_t *n_committed,
                  int32_t *accept_count, int32_t *hit_eos, int32_t *rollback,
                  int32_t *target_seq_len, int32_t *status, cudaStream_t s) {
    if (B <= 0) return DF_OK;
    return launch_k("accept_kernel", accept_kernel, dim3((B + 127) / 128), dim3(128), 0, s, drafts,
                    ld, target, B, K, eos, n_eos, committed, n_committed, accept_count, hit_eos,
                    rollback, target_seq_len, status);
}

int launch_argmax_accept(const ArgTop *part, int G, int B, int blk, int32_t *argmax_out,
                         const int32_t *target, const int32_t *eos, int n_eos,
                         int32_t *committed, int32_t *n_committed, int32_t *accept_count,
                         int32_t *hit_eos, int32_t *rollback, int32_t *target_seq_len,
                         int32_t *status, cudaStream_t s) {
    if (B <= 0) return DF_OK;
    if (blk < 2 || blk > 32) return fail(DF_ESHAPE, "fused argmax + accept takes 2..32 rows");
    return launch_k("argmax_accept_kernel", argmax_accept_kernel, dim3(B), dim3(32 * blk), 0, s,
                    part, G, blk, argmax_out, target, eos, n_eos, committed, n_committed,
                    accept_count, hit_eos, rollback, target_seq_len, status);
}

int launch_rollback(int32_t *seq_len, const int32_t *n, int B, int32_t *status, cudaStream_t s) {
    if (B <= 0) return DF_OK;
    return launch_k("rollback_kernel", rollback_kernel, dim3((B + 127) / 128), dim3(128), 0, s,
                    seq_len, n, B, status);
}

}  // namespace df

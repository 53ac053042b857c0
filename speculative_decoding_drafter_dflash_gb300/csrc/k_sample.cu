// Non-greedy accept step (speculative sampling): qwen35_orchestrator.rs, module doc
// "Non-greedy (Metropolis-Hastings) is out of scope here" (stochastic acceptance wired through
// the MTP K=1 path; for DFlash it replaces `step_round_from_argmaxes` at step 11). The rule,
// which the page does not spell out, is read as the standard speculative-sampling test: with
// p_i = softmax(target_i / T) and q_i = softmax(draft_i / T), draft x_i is accepted when
// u_i q_i(x_i) < p_i(x_i); at the first rejection a the committed token is drawn from
// max(0, p_a - q_a), and when every draft is accepted from p_K. A draw from weights w with a
// uniform u is the smallest index j whose running sum exceeds u * sum(w).
//
// Three kernels, all reading the logits with 128-bit loads:
//   stats : per (row, 2048-wide chunk) the maximum of x = l log2(e) / T and the sum of
//           2^(x - max) (hardware ex2)
//   walk  : one warp per sequence merges the chunk statistics of its 2K+1 rows (in chunk order)
//           and runs the accept test at the drafted tokens
//   draw  : per (sequence, chunk) the sum of the draw weights; the last chunk CTA of a sequence
//           locates the chunk and then the index where the running sum crosses u * total, and
//           writes the committed tokens (EOS cut, -1 fill) as the greedy walk does.
#include "df_internal.cuh"

namespace df {

namespace {

constexpr int kSThreads = 256;
constexpr int kEPT = 8;                     // logits per thread (two 128-bit loads)
constexpr int kSChunk = kSThreads * kEPT;   // logits per chunk CTA

using MS = MaxSum;

// Statistics are kept in log2 units: x = logit * log2(e) / T, s = sum of 2^(x - max).
__device__ __forceinline__ float ex2f(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ MS ms_merge(MS a, MS b) {
    if (a.m == -INFINITY) return b;
    if (b.m == -INFINITY) return a;
    const float M = fmaxf(a.m, b.m);
    return {M, a.s * ex2f(a.m - M) + b.s * ex2f(b.m - M)};
}

__device__ __forceinline__ MS warp_ms(MS v) {
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
        MS w;
        w.m = __shfl_xor_sync(0xffffffffu, v.m, o);
        w.s = __shfl_xor_sync(0xffffffffu, v.s, o);
        v = ms_merge(v, w);
    }
    return v;
}

// Row rho of sequence b: rho <= K is target row rho, rho > K is draft row rho - K - 1.
__device__ __forceinline__ const float *row_ptr(const SampleArgs &a, int b, int rho) {
    if (rho <= a.K) return a.target + ((size_t)b * (a.K + 1) + rho) * a.V;
    return a.draft + ((size_t)b * a.K + (rho - a.K - 1)) * a.V;
}

__global__ void __launch_bounds__(kSThreads) sample_stats_kernel(SampleArgs a) {
    __shared__ MS red[kSThreads / 32];
    pdl_trigger();
    pdl_wait();
    const int c = blockIdx.x, rows = 2 * a.K + 1;
    const int b = blockIdx.y / rows, rho = blockIdx.y - b * rows;
    const float *row = row_ptr(a, b, rho);
    const int j0 = c * kSChunk + threadIdx.x * kEPT;
    float x[kEPT];
#pragma unroll
    for (int h = 0; h < kEPT / 4; ++h) {
        float4 v = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
        if (j0 + 4 * h < a.V) v = __ldcs(reinterpret_cast<const float4 *>(row + j0 + 4 * h));
        x[4 * h] = v.x * a.scale;
        x[4 * h + 1] = v.y * a.scale;
        x[4 * h + 2] = v.z * a.scale;
        x[4 * h + 3] = v.w * a.scale;
    }
    MS t{-INFINITY, 0.f};
    float m = -INFINITY;
#pragma unroll
    for (int i = 0; i < kEPT; ++i) m = fmaxf(m, x[i]);
    if (m != -INFINITY) {
        float s = 0.f;
#pragma unroll
        for (int i = 0; i < kEPT; ++i) s += ex2f(x[i] - m);
        t = {m, s};
    }
    t = warp_ms(t);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = t;
    __syncthreads();
    if (threadIdx.x == 0) {
        MS r = red[0];
        for (int w = 1; w < kSThreads / 32; ++w) r = ms_merge(r, red[w]);
        a.stats[(size_t)blockIdx.y * gridDim.x + c] = r;
    }
}

// One CTA per sequence: warps merge the chunk statistics of the 2K+1 rows (lanes over chunks in
// a fixed order), then thread i runs the accept test of draft i, all in parallel; the accept
// count is the first failing i.
__global__ void __launch_bounds__(kSThreads) sample_walk_kernel(SampleArgs a) {
    __shared__ MS rs[2 * kSampleMaxK + 1];
    __shared__ int rej[kSampleMaxK];
    pdl_trigger();
    pdl_wait();
    const int b = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rows = 2 * a.K + 1;
    for (int rho = warp; rho < rows; rho += kSThreads / 32) {
        const MS *p = a.stats + ((size_t)b * rows + rho) * a.n_chunks;
        MS v{-INFINITY, 0.f};
        for (int c = lane; c < a.n_chunks; c += 32) v = ms_merge(v, p[c]);
        v = warp_ms(v);
        if (lane == 0) rs[rho] = v;
    }
    __syncthreads();
    for (int i = threadIdx.x; i < a.K; i += kSThreads) {
        int x = a.drafts[(size_t)b * a.K + i];
        if (x < 0 || x >= a.V) {
            set_status(a.status, DF_EINVAL);
            x = min(max(x, 0), a.V - 1);
        }
        const MS sp = rs[i], sq = rs[a.K + 1 + i];
        const float pt = ex2f(row_ptr(a, b, i)[x] * a.scale - sp.m) / sp.s;
        const float qd = ex2f(row_ptr(a, b, a.K + 1 + i)[x] * a.scale - sq.m) / sq.s;
        rej[i] = !(a.u_accept[(size_t)b * a.K + i] * qd < pt);
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        int acc = a.K;
        for (int i = 0; i < a.K; ++i)
            if (rej[i]) {
                acc = i;
                break;
            }
        // the draw: residual of row acc, or the target's next position when all were accepted
        const MS sp = rs[acc];
        const MS sq = acc < a.K ? rs[a.K + 1 + acc] : MS{-INFINITY, 0.f};
        SampleState st;
        st.acc = acc;
        st.mp = sp.m;
        st.sp = 1.f / sp.s;
        st.mq = sq.m;
        st.sq = acc < a.K ? 1.f / sq.s : 0.f;
        a.state[b] = st;
        a.accept_count[b] = acc;
        a.rollback[b] = a.K - acc;
    }
}

// Draw weight of index j for sequence b (residual when acc < K, else the target's softmax).
__device__ __forceinline__ float draw_weight(const SampleArgs &a, const SampleState &st, float lt,
                                             float ld) {
    const float p = ex2f(lt * a.scale - st.mp) * st.sp;
    if (st.acc >= a.K) return p;
    const float q = ex2f(ld * a.scale - st.mq) * st.sq;
    return fmaxf(0.f, p - q);
}

__global__ void __launch_bounds__(kSThreads) sample_draw_kernel(SampleArgs a) {
    __shared__ float wsum[kSThreads / 32];
    __shared__ float tsum[kSThreads];
    __shared__ int s_last, s_chunk;
    __shared__ float s_base, s_target;
    pdl_trigger();
    pdl_wait();
    const int c = blockIdx.x, b = blockIdx.y;
    const SampleState st = a.state[b];
    const float *tp = row_ptr(a, b, st.acc);
    const float *dq = st.acc < a.K ? row_ptr(a, b, a.K + 1 + st.acc) : nullptr;
    auto chunk_weights = [&](int cc, int t_idx, float (&w)[kEPT]) {
        const int j0 = cc * kSChunk + t_idx * kEPT;
#pragma unroll
        for (int h = 0; h < kEPT / 4; ++h) {
            float4 lt = make_float4(0.f, 0.f, 0.f, 0.f), ld = lt;
            const bool ok = j0 + 4 * h < a.V;
            if (ok) {
                lt = __ldcg(reinterpret_cast<const float4 *>(tp + j0 + 4 * h));
                if (dq) ld = __ldcg(reinterpret_cast<const float4 *>(dq + j0 + 4 * h));
            }
            w[4 * h] = ok ? draw_weight(a, st, lt.x, ld.x) : 0.f;
            w[4 * h + 1] = ok ? draw_weight(a, st, lt.y, ld.y) : 0.f;
            w[4 * h + 2] = ok ? draw_weight(a, st, lt.z, ld.z) : 0.f;
            w[4 * h + 3] = ok ? draw_weight(a, st, lt.w, ld.w) : 0.f;
        }
    };
    float w[kEPT];
    chunk_weights(c, threadIdx.x, w);
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < kEPT; ++i) s += w[i];
    s = warp_sum(s);
    if ((threadIdx.x & 31) == 0) wsum[threadIdx.x >> 5] = s;
    __syncthreads();
    if (threadIdx.x == 0) {
        float t = 0.f;
        for (int i = 0; i < kSThreads / 32; ++i) t += wsum[i];
        a.csum[(size_t)b * a.n_chunks + c] = t;
    }
    // last chunk CTA of the sequence locates the draw
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) s_last = atomicAdd(&a.counters[b], 1) == a.n_chunks - 1;
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    if (threadIdx.x == 0) a.counters[b] = 0;   // leave the counter at zero for the next call
    // chunk sums into shared memory (parallel loads), then one thread scans them in order
    const float *cs = a.csum + (size_t)b * a.n_chunks;
    float tot = 0.f, run = 0.f, base = 0.f, base_last = 0.f, target = 0.f;
    int cstar = -1, last_pos = 0;
    for (int c0 = 0; c0 < a.n_chunks; c0 += kSThreads) {
        const int n = min(kSThreads, a.n_chunks - c0);
        __syncthreads();
        if ((int)threadIdx.x < n) tsum[threadIdx.x] = __ldcg(cs + c0 + threadIdx.x);
        __syncthreads();
        if (threadIdx.x == 0)
            for (int i = 0; i < n; ++i) tot += tsum[i];
    }
    if (threadIdx.x == 0) target = a.u_sample[b] * tot;
    for (int c0 = 0; c0 < a.n_chunks; c0 += kSThreads) {
        const int n = min(kSThreads, a.n_chunks - c0);
        __syncthreads();
        if ((int)threadIdx.x < n) tsum[threadIdx.x] = __ldcg(cs + c0 + threadIdx.x);
        __syncthreads();
        if (threadIdx.x == 0)
            for (int i = 0; i < n; ++i) {
                const float v = tsum[i];
                if (v > 0.f) {
                    last_pos = c0 + i;
                    base_last = run;
                }
                if (cstar < 0 && run + v > target) {
                    cstar = c0 + i;
                    base = run;
                }
                run += v;
            }
    }
    if (threadIdx.x == 0) {
        if (cstar < 0) {                    // rounding put the target past the total
            cstar = last_pos;
            base = base_last;
        }
        s_chunk = cstar;
        s_base = base;
        s_target = target;
        if (!(tot > 0.f)) set_status(a.status, DF_EINVAL);
    }
    __syncthreads();
    chunk_weights(s_chunk, threadIdx.x, w);
    float mine = 0.f;
#pragma unroll
    for (int i = 0; i < kEPT; ++i) mine += w[i];
    tsum[threadIdx.x] = mine;
    __syncthreads();
    if (threadIdx.x == 0) {
        // running sum over the chunk's threads in index order, then inside the found thread
        float run = s_base;
        int tok = -1, last_pos = -1;
        for (int t = 0; t < kSThreads && tok < 0; ++t) {
            const float v = tsum[t];
            if (v > 0.f) last_pos = t;
            if (run + v > s_target) tok = t;
            else run += v;
        }
        int idx;
        if (tok < 0) tok = last_pos < 0 ? 0 : last_pos;
        // thread tok's weights (recomputed by thread 0 with the same loads and arithmetic)
        {
            const int j0 = s_chunk * kSChunk + tok * kEPT;
            float wv[kEPT];
            chunk_weights(s_chunk, tok, wv);
            float r = run;
            idx = -1;
            int lastj = j0;
            for (int i = 0; i < kEPT; ++i) {
                if (j0 + i >= a.V) break;
                if (wv[i] > 0.f) lastj = j0 + i;
                if (r + wv[i] > s_target) {
                    idx = j0 + i;
                    break;
                }
                r += wv[i];
            }
            if (idx < 0) idx = lastj;
        }
        // committed tokens: accepted drafts, then the drawn token, cut after the first EOS
        int32_t *out = a.committed + (size_t)b * (a.K + 1);
        int n = 0, hit = 0;
        for (int i = 0; i <= st.acc; ++i) {
            const int tkn = i < st.acc ? a.drafts[(size_t)b * a.K + i] : idx;
            out[n++] = tkn;
            bool is_eos = false;
            for (int e = 0; e < a.n_eos; ++e) is_eos |= (tkn == a.eos[e]);
            if (is_eos) {
                hit = 1;
                break;
            }
        }
        for (int i = n; i <= a.K; ++i) out[i] = -1;
        a.n_committed[b] = n;
        a.hit_eos[b] = hit;
    }
}

}  // namespace

int sample_chunks(int V) { return (V + kSChunk - 1) / kSChunk; }

int launch_accept_stochastic(const SampleArgs &a, cudaStream_t s) {
    DF_TRY(launch_k("sample_stats_kernel", sample_stats_kernel,
                    dim3(a.n_chunks, a.B * (2 * a.K + 1)), dim3(kSThreads), 0, s, a));
    DF_TRY(launch_k("sample_walk_kernel", sample_walk_kernel, dim3(a.B), dim3(kSThreads), 0, s, a));
    return launch_k("sample_draw_kernel", sample_draw_kernel, dim3(a.n_chunks, a.B),
                    dim3(kSThreads), 0, s, a);
}

}  // namespace df

// Non-greedy path: drafts drawn from the drafter's softmax and the speculative-sampling accept
// step. qwen35_orchestrator.rs, module doc "Non-greedy (Metropolis-Hastings) is out of scope
// here" (stochastic acceptance wired through the MTP K=1 path; for DFlash it replaces
// `step_round_from_argmaxes` at step 11). The rule, which the page does not spell out, is read
// as the standard speculative-sampling test: with p_i = softmax(target_i / T) and
// q_i = softmax(draft_i / T), each draft x_i is itself a draw from q_i; it is accepted when
// u_i q_i(x_i) < p_i(x_i); at the first rejection a the committed token is drawn from
// max(0, p_a - q_a), and when every draft is accepted from p_K. A draw from weights w with a
// uniform u is the smallest index j whose running sum exceeds u * sum(w).
//
// Kernels, all reading the logits with 128-bit loads (x = logit * log2(e) / T):
//   stats : per (row, 2048-wide chunk) the maximum of x and the sum of 2^(x - max) (F32,
//           hardware ex2): the accept tests and the shift of every draw
//   walk  : one CTA per sequence merges its rows' chunk statistics and runs the K accept tests
//   norm  : per (sequence, chunk) the sums of 2^(x - M) of the draw's p and q rows
//   draw  : per (draw, chunk) the sum of the draw weights; the last chunk CTA of a draw locates
//           the chunk, the thread and the index where the running sum crosses u * total
//
// The draw weights are computed to ~1e-14 relative (a float-float 2^x: the exponent split
// into an integer, a 1/32 step from a table and a short Taylor series) and summed as
// float-float pairs inside a warp and in float64 beyond it, so a draw agrees with a float64
// reference except where u * total lies within ~1e-12 of a cumulative boundary.
#include <cmath>

#include "df_internal.cuh"

namespace df {

namespace {

constexpr int kSThreads = 256;
constexpr int kEPT = 8;                     // logits per thread (two 128-bit loads)
constexpr int kSChunk = kSThreads * kEPT;   // logits per chunk CTA
constexpr int kMaxChunks = 1024;            // V <= 2^21

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

// ------------------------------------------------------------------ float-float arithmetic
// A value hi + lo with |lo| <= ulp(hi) / 2 (Dekker / Knuth error-free transformations).
struct FF {
    float hi, lo;
};

__device__ __forceinline__ FF two_sum(float a, float b) {
    const float s = a + b;
    const float bb = s - a;
    return {s, (a - (s - bb)) + (b - bb)};
}

__device__ __forceinline__ FF fast_two_sum(float a, float b) {   // |a| >= |b| or a == 0
    const float s = a + b;
    return {s, b - (s - a)};
}

__device__ __forceinline__ FF ff_add(FF a, FF b) {
    const FF s = two_sum(a.hi, b.hi);
    return fast_two_sum(s.hi, s.lo + (a.lo + b.lo));
}

__device__ __forceinline__ FF ff_mul(FF a, FF b) {
    const float p = a.hi * b.hi;
    const float e = fmaf(a.hi, b.hi, -p);
    return fast_two_sum(p, fmaf(a.hi, b.lo, fmaf(a.lo, b.hi, e)));
}

__device__ __forceinline__ double ff_to_double(FF a) { return (double)a.hi + (double)a.lo; }

__device__ __forceinline__ FF warp_ff_sum(FF v) {
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
        FF w;
        w.hi = __shfl_xor_sync(0xffffffffu, v.hi, o);
        w.lo = __shfl_xor_sync(0xffffffffu, v.lo, o);
        v = ff_add(v, w);
    }
    return v;
}

// 2^(l * scale - M) for a logit l: scale = sc_hi + sc_lo, M an F32 shift (the row maximum of
// the F32 products, so the result is <= ~1). The product and the shift are carried exactly as
// a float-float d; d = n + k/32 + r with integer n, |k| <= 16, |r| <= 1/64; 2^(k/32) comes from
// the table (float-float, computed on the host in double), 2^r = exp(r ln 2) from the Taylor
// series to the 6th power (|r ln 2| < 0.011, the next term < 4e-18).
__device__ __forceinline__ FF weight_ff(float l, float M, const SampleArgs &a) {
    const float p_hi = l * a.sc_hi;
    const float p_lo = fmaf(l, a.sc_lo, fmaf(l, a.sc_hi, -p_hi));
    FF d = two_sum(p_hi, -M);
    d = fast_two_sum(d.hi, d.lo + p_lo);
    if (!(d.hi > -126.f)) return {0.f, 0.f};          // below 2^-126 of the row maximum
    const float nf = rintf(d.hi);
    FF f = two_sum(d.hi - nf, d.lo);                   // d.hi - nf is exact
    const float kf = rintf(f.hi * 32.f);
    FF r = two_sum(fmaf(kf, -0.03125f, f.hi), f.lo);   // f.hi - k/32 is exact
    const float g_hi = r.hi * a.ln2_hi;
    const float g_lo = fmaf(r.hi, a.ln2_lo, fmaf(r.lo, a.ln2_hi, fmaf(r.hi, a.ln2_hi, -g_hi)));
    const float sq_hi = g_hi * g_hi;
    const float sq_lo = fmaf(g_hi, g_hi, -sq_hi) + 2.f * g_hi * g_lo;
    const float tail =
        sq_hi * g_hi *
        (1.f / 6.f + g_hi * (1.f / 24.f + g_hi * (1.f / 120.f + g_hi * (1.f / 720.f))));
    FF E = two_sum(g_hi, 0.5f * sq_hi);
    E = fast_two_sum(E.hi, E.lo + (g_lo + 0.5f * sq_lo + tail));
    const float2 t = a.exp2_tab[min(max((int)kf + 16, 0), 32)];
    const float m_hi = t.x * E.hi;
    const float m_lo = fmaf(t.x, E.hi, -m_hi) + fmaf(t.x, E.lo, t.y * E.hi);
    FF w = two_sum(t.x, m_hi);
    w = fast_two_sum(w.hi, w.lo + (t.y + m_lo));
    const float s = __int_as_float(((int)nf + 127) << 23);   // 2^n, n in [-126, 0]
    return {w.hi * s, w.lo * s};
}

__device__ __forceinline__ const float *draft_row(const SampleArgs &a, int b, int i) {
    return a.draft + ((size_t)b * a.draft_ld + i) * a.V;
}

// Row rho of sequence b in the statistics. Accept mode: rho <= K is target row rho, rho > K is
// draft row rho - K - 1. Sample mode: draft row rho.
__device__ __forceinline__ const float *row_ptr(const SampleArgs &a, int b, int rho) {
    if (a.sample_mode) return draft_row(a, b, rho);
    if (rho <= a.K) return a.target + ((size_t)b * (a.K + 1) + rho) * a.V;
    return draft_row(a, b, rho - a.K - 1);
}

__device__ __forceinline__ int stat_rows(const SampleArgs &a) {
    return a.sample_mode ? a.K : 2 * a.K + 1;
}

__global__ void __launch_bounds__(kSThreads) sample_stats_kernel(SampleArgs a) {
    DF_TRACE_KERNEL(TK_SAMPLE_STATS);
    __shared__ MS red[kSThreads / 32];
    pdl_trigger();
    pdl_wait();
    const int c = blockIdx.x, rows = stat_rows(a);
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

// Row maximum from the chunk statistics (exact: a maximum of maxima).
__device__ float row_max(const SampleArgs &a, const MS *p) {
    __shared__ float wm[kSThreads / 32];
    float m = -INFINITY;
    for (int c = threadIdx.x; c < a.n_chunks; c += kSThreads) m = fmaxf(m, p[c].m);
    m = warp_max(m);
    __syncthreads();
    if ((threadIdx.x & 31) == 0) wm[threadIdx.x >> 5] = m;
    __syncthreads();
    float r = wm[0];
    for (int w = 1; w < kSThreads / 32; ++w) r = fmaxf(r, wm[w]);
    return r;
}

// One CTA per sequence: warps merge the chunk statistics of the 2K+1 rows (lanes over chunks in
// a fixed order), then thread i runs the accept test of draft i, all in parallel; the accept
// count is the first failing i.
__global__ void __launch_bounds__(kSThreads) sample_walk_kernel(SampleArgs a) {
    DF_TRACE_KERNEL(TK_SAMPLE_WALK);
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
        SampleState st;
        st.acc = acc;
        st.mp = rs[acc].m;
        st.mq = acc < a.K ? rs[a.K + 1 + acc].m : 0.f;
        a.state[b] = st;
        a.accept_count[b] = acc;
        a.rollback[b] = a.K - acc;
    }
}

// What one draw reads: its p row (and, for a residual draw, its q row), their shifts, and the
// float-float reciprocals of their exp sums (residual draws only).
struct DrawJob {
    const float *p, *q;
    float mp, mq;
    FF ip, iq;
    float u;
};

// Accept mode: the draw of sequence b (residual of row acc, or the target's row K).
__device__ DrawJob accept_job(const SampleArgs &a, int b) {
    const SampleState st = a.state[b];
    DrawJob j;
    j.p = a.target + ((size_t)b * (a.K + 1) + st.acc) * a.V;
    j.q = st.acc < a.K ? draft_row(a, b, st.acc) : nullptr;
    j.mp = st.mp;
    j.mq = st.mq;
    j.u = a.u_sample[b];
    j.ip = j.iq = {0.f, 0.f};
    return j;
}

// Sums of 2^(x - M) of the draw's p and q rows over one chunk (residual draws only).
__global__ void __launch_bounds__(kSThreads) sample_norm_kernel(SampleArgs a) {
    DF_TRACE_KERNEL(TK_SAMPLE_NORM);
    __shared__ double wsum[2][kSThreads / 32];
    pdl_trigger();
    pdl_wait();
    const int c = blockIdx.x, b = blockIdx.y;
    const DrawJob jb = accept_job(a, b);
    if (!jb.q) return;
    const int j0 = c * kSChunk + threadIdx.x * kEPT;
    FF sp{0.f, 0.f}, sq{0.f, 0.f};
#pragma unroll
    for (int h = 0; h < kEPT / 4; ++h) {
        if (j0 + 4 * h < a.V) {
            const float4 lp = __ldcg(reinterpret_cast<const float4 *>(jb.p + j0 + 4 * h));
            const float4 lq = __ldcg(reinterpret_cast<const float4 *>(jb.q + j0 + 4 * h));
            sp = ff_add(sp, weight_ff(lp.x, jb.mp, a));
            sp = ff_add(sp, weight_ff(lp.y, jb.mp, a));
            sp = ff_add(sp, weight_ff(lp.z, jb.mp, a));
            sp = ff_add(sp, weight_ff(lp.w, jb.mp, a));
            sq = ff_add(sq, weight_ff(lq.x, jb.mq, a));
            sq = ff_add(sq, weight_ff(lq.y, jb.mq, a));
            sq = ff_add(sq, weight_ff(lq.z, jb.mq, a));
            sq = ff_add(sq, weight_ff(lq.w, jb.mq, a));
        }
    }
    sp = warp_ff_sum(sp);
    sq = warp_ff_sum(sq);
    if ((threadIdx.x & 31) == 0) {
        wsum[0][threadIdx.x >> 5] = ff_to_double(sp);
        wsum[1][threadIdx.x >> 5] = ff_to_double(sq);
    }
    __syncthreads();
    if (threadIdx.x < 2) {
        double t = 0.0;
        for (int w = 0; w < kSThreads / 32; ++w) t += wsum[threadIdx.x][w];
        a.dsum[((size_t)b * a.n_chunks + c) * 2 + threadIdx.x] = t;
    }
}

// Float-float reciprocal of a positive double.
__device__ __forceinline__ FF ff_recip(double s) {
    const double r = 1.0 / s;
    const float hi = (float)r;
    return {hi, (float)(r - (double)hi)};
}

// The weights of thread t_idx's kEPT logits of chunk cc.
__device__ __forceinline__ void chunk_weights(const SampleArgs &a, const DrawJob &jb, int cc,
                                              int t_idx, FF (&w)[kEPT]) {
    const int j0 = cc * kSChunk + t_idx * kEPT;
#pragma unroll
    for (int h = 0; h < kEPT / 4; ++h) {
        const bool ok = j0 + 4 * h < a.V;
        float4 lp = make_float4(0.f, 0.f, 0.f, 0.f), lq = lp;
        if (ok) {
            lp = __ldcg(reinterpret_cast<const float4 *>(jb.p + j0 + 4 * h));
            if (jb.q) lq = __ldcg(reinterpret_cast<const float4 *>(jb.q + j0 + 4 * h));
        }
        const float lpv[4] = {lp.x, lp.y, lp.z, lp.w}, lqv[4] = {lq.x, lq.y, lq.z, lq.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            FF v{0.f, 0.f};
            if (ok) {
                v = weight_ff(lpv[e], jb.mp, a);
                if (jb.q) {
                    // max(0, p - q) with p = 2^(x - mp) / S_p and q = 2^(y - mq) / S_q
                    const FF pn = ff_mul(v, jb.ip);
                    const FF qn = ff_mul(weight_ff(lqv[e], jb.mq, a), jb.iq);
                    v = ff_add(pn, FF{-qn.hi, -qn.lo});
                    if (!(v.hi > 0.f)) v = {0.f, 0.f};
                }
            }
            w[4 * h + e] = v;
        }
    }
}

__device__ __forceinline__ FF thread_sum(const FF (&w)[kEPT]) {
    FF s{0.f, 0.f};
#pragma unroll
    for (int i = 0; i < kEPT; ++i) s = ff_add(s, w[i]);
    return s;
}

// grid (chunks, draws). Accept mode: draw b of sequence b, then the committed tokens.
// Sample mode: draw b * K + i is draft i of sequence b, from softmax(draft row i / T).
__global__ void __launch_bounds__(kSThreads) sample_draw_kernel(SampleArgs a) {
    DF_TRACE_KERNEL(TK_SAMPLE_DRAW);
    __shared__ double wsum[kSThreads / 32];
    __shared__ double tsum[kSThreads];
    __shared__ double s_norm[2];
    __shared__ float s_max;
    __shared__ int s_last, s_chunk;
    __shared__ double s_base, s_target;
    pdl_trigger();
    pdl_wait();
    const int c = blockIdx.x, job = blockIdx.y;
    DrawJob jb;
    if (a.sample_mode) {
        const int b = job / a.K, i = job - b * a.K;
        jb.p = draft_row(a, b, i);
        jb.q = nullptr;
        const float M = row_max(a, a.stats + (size_t)job * a.n_chunks);
        if (threadIdx.x == 0) s_max = M;
        __syncthreads();
        jb.mp = s_max;
        jb.mq = 0.f;
        jb.u = a.u_draft[job];
        jb.ip = jb.iq = {0.f, 0.f};
    } else {
        jb = accept_job(a, job);
        if (jb.q) {
            // S_p and S_q from the chunk sums of the norm kernel, in chunk order
            if (threadIdx.x < 2) {
                const double *ds = a.dsum + (size_t)job * a.n_chunks * 2;
                double t = 0.0;
                for (int cc = 0; cc < a.n_chunks; ++cc) t += __ldcg(ds + 2 * cc + threadIdx.x);
                s_norm[threadIdx.x] = t;
            }
            __syncthreads();
            if (!(s_norm[0] > 0.0) || !(s_norm[1] > 0.0)) {
                set_status(a.status, DF_EINVAL);
                jb.q = nullptr;   // degenerate input: draw from p
            } else {
                jb.ip = ff_recip(s_norm[0]);
                jb.iq = ff_recip(s_norm[1]);
            }
        }
    }
    FF w[kEPT];
    chunk_weights(a, jb, c, threadIdx.x, w);
    const FF ts = warp_ff_sum(thread_sum(w));
    if ((threadIdx.x & 31) == 0) wsum[threadIdx.x >> 5] = ff_to_double(ts);
    __syncthreads();
    if (threadIdx.x == 0) {
        double t = 0.0;
        for (int i = 0; i < kSThreads / 32; ++i) t += wsum[i];
        a.csum[(size_t)job * a.n_chunks + c] = t;
    }
    // the last chunk CTA of the draw locates it
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) s_last = atomicAdd(&a.counters[job], 1) == a.n_chunks - 1;
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    if (threadIdx.x == 0) a.counters[job] = 0;   // left at zero for the next call
    const double *cs = a.csum + (size_t)job * a.n_chunks;
    double tot = 0.0, run = 0.0, base = 0.0, base_last = 0.0, target = 0.0;
    int cstar = -1, last_pos = 0;
    for (int c0 = 0; c0 < a.n_chunks; c0 += kSThreads) {
        const int n = min(kSThreads, a.n_chunks - c0);
        __syncthreads();
        if ((int)threadIdx.x < n) tsum[threadIdx.x] = __ldcg(cs + c0 + threadIdx.x);
        __syncthreads();
        if (threadIdx.x == 0)
            for (int i = 0; i < n; ++i) tot += tsum[i];
    }
    if (threadIdx.x == 0) target = (double)jb.u * tot;
    for (int c0 = 0; c0 < a.n_chunks; c0 += kSThreads) {
        const int n = min(kSThreads, a.n_chunks - c0);
        __syncthreads();
        if ((int)threadIdx.x < n) tsum[threadIdx.x] = __ldcg(cs + c0 + threadIdx.x);
        __syncthreads();
        if (threadIdx.x == 0)
            for (int i = 0; i < n; ++i) {
                const double v = tsum[i];
                if (v > 0.0) {
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
        if (!(tot > 0.0)) set_status(a.status, DF_EINVAL);
    }
    __syncthreads();
    chunk_weights(a, jb, s_chunk, threadIdx.x, w);
    tsum[threadIdx.x] = ff_to_double(thread_sum(w));
    __syncthreads();
    if (threadIdx.x != 0) return;
    // running sum over the chunk's threads in index order, then inside the found thread
    double r = s_base;
    int tok = -1, last_t = -1;
    for (int t = 0; t < kSThreads && tok < 0; ++t) {
        const double v = tsum[t];
        if (v > 0.0) last_t = t;
        if (r + v > s_target) tok = t;
        else r += v;
    }
    if (tok < 0) tok = last_t < 0 ? 0 : last_t;
    int idx = -1;
    {
        const int j0 = s_chunk * kSChunk + tok * kEPT;
        FF wv[kEPT];
        chunk_weights(a, jb, s_chunk, tok, wv);
        int lastj = j0;
        for (int i = 0; i < kEPT; ++i) {
            if (j0 + i >= a.V) break;
            const double v = ff_to_double(wv[i]);
            if (v > 0.0) lastj = j0 + i;
            if (r + v > s_target) {
                idx = j0 + i;
                break;
            }
            r += v;
        }
        if (idx < 0) idx = lastj;
    }
    if (!df_in_bounds(idx >= 0 && idx < a.V, a.status)) idx = 0;
    if (a.sample_mode) {
        a.drafts_out[job] = idx;
        return;
    }
    // committed tokens: accepted drafts, then the drawn token, cut after the first EOS
    const int b = job, acc = a.state[b].acc;
    int32_t *out = a.committed + (size_t)b * (a.K + 1);
    int n = 0, hit = 0;
    for (int i = 0; i <= acc; ++i) {
        const int tkn = i < acc ? a.drafts[(size_t)b * a.K + i] : idx;
        if (!df_in_bounds(n <= a.K, a.status)) break;
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

}  // namespace

int sample_chunks(int V) { return (V + kSChunk - 1) / kSChunk; }

void carve_sample_scratch(Carve &cv, SampleArgs &a, int B, int K, int V) {
    a.n_chunks = sample_chunks(V);
    a.stats = cv.take<MaxSum>((size_t)B * (2 * K + 1) * a.n_chunks);
    a.state = cv.take<SampleState>((size_t)B);
    a.dsum = cv.take<double>((size_t)B * a.n_chunks * 2);
    a.csum = cv.take<double>((size_t)B * K * a.n_chunks);
    a.counters = cv.take<int>((size_t)B * K);
}

void sample_constants(SampleArgs &a) {
    const double scale = 1.4426950408889634 / (double)a.T;   // log2(e) / T
    a.scale = (float)scale;
    a.sc_hi = (float)scale;
    a.sc_lo = (float)(scale - (double)a.sc_hi);
    const double ln2 = 0.69314718055994530942;
    a.ln2_hi = (float)ln2;
    a.ln2_lo = (float)(ln2 - (double)a.ln2_hi);
    for (int k = -16; k <= 16; ++k) {
        const double v = std::exp2((double)k / 32.0);
        a.exp2_tab[k + 16].x = (float)v;
        a.exp2_tab[k + 16].y = (float)(v - (double)(float)v);
    }
}

int launch_accept_stochastic(const SampleArgs &a, cudaStream_t s) {
    if (a.n_chunks > kMaxChunks) return fail(DF_ESHAPE, "vocabulary of %d is too large", a.V);
    DF_TRY(launch_k("sample_stats_kernel", sample_stats_kernel,
                    dim3(a.n_chunks, a.B * (2 * a.K + 1)), dim3(kSThreads), 0, s, a));
    DF_TRY(launch_k("sample_walk_kernel", sample_walk_kernel, dim3(a.B), dim3(kSThreads), 0, s, a));
    DF_TRY(launch_k("sample_norm_kernel", sample_norm_kernel, dim3(a.n_chunks, a.B),
                    dim3(kSThreads), 0, s, a));
    return launch_k("sample_draw_kernel", sample_draw_kernel, dim3(a.n_chunks, a.B),
                    dim3(kSThreads), 0, s, a);
}

int launch_sample_drafts(const SampleArgs &a, cudaStream_t s) {
    if (a.n_chunks > kMaxChunks) return fail(DF_ESHAPE, "vocabulary of %d is too large", a.V);
    DF_TRY(launch_k("sample_stats_kernel", sample_stats_kernel, dim3(a.n_chunks, a.B * a.K),
                    dim3(kSThreads), 0, s, a));
    return launch_k("sample_draw_kernel", sample_draw_kernel, dim3(a.n_chunks, a.B * a.K),
                    dim3(kSThreads), 0, s, a);
}

}  // namespace df

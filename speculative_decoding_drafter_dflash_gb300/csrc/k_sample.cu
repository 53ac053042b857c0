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
// Kernels, all reading the logits with 128-bit loads (x = logit * log2(e) / T).
// Accept step (four launches):
//   stats : per (row, 2048-wide chunk) the maximum of x and the sum of 2^(x - max) (F32,
//           hardware ex2): the accept tests and the shift of the draw
//   walk  : one CTA per sequence merges its rows' chunk statistics and runs the K accept tests
//   norm  : per (sequence, chunk) the sums of 2^(x - M) of the draw's p and q rows
//   draw  : per (sequence, chunk) the sum of the draw weights; the last chunk CTA of a draw
//           locates the chunk, then the index, where the running sum crosses u * total
// Drafts (one launch):
//   fused : per (draft, chunk) the chunk maximum and the sum of the weights shifted by it; the
//           last chunk CTA of a draft rescales the chunk sums to the row maximum and locates
//           the token the same way
//
// The draw weights are computed to ~1e-14 relative (a float-float 2^x: the exponent split
// into an integer, a 1/32 step from a table and a short Taylor series) and summed and scanned as
// float-float pairs throughout (no float64: this part runs it at a small fraction of the F32
// rate), so a draw agrees with a float64 reference except where u * total lies within ~1e-12
// of a cumulative boundary.
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

// 2^d for a float-float d (d.hi <= ~0; 0 below 2^-126). d = n + k/32 + r with integer n,
// |k| <= 16, |r| <= 1/64; 2^(k/32) comes from the table (float-float, computed on the host in
// double), 2^r = exp(r ln 2) from the Taylor series to the 6th power (|r ln 2| < 0.011, the next
// term < 4e-18). The fast_two_sum steps are exact: d.hi - n and f.hi - k/32 are 0 or at least
// one ulp of the word whose half-ulp bounds the low part, |g| > g^2 / 2, and the table entry
// (>= 0.7) exceeds its product with |E| < 0.012.
__device__ __forceinline__ FF exp2_ff(FF d, const SampleArgs &a, const float2 *tab) {
    if (!(d.hi > -126.f)) return {0.f, 0.f};
    const float nf = rintf(d.hi);
    const FF f = fast_two_sum(d.hi - nf, d.lo);        // d.hi - nf is exact
    const float kf = rintf(f.hi * 32.f);
    const FF r = fast_two_sum(fmaf(kf, -0.03125f, f.hi), f.lo);   // f.hi - k/32 is exact
    const float g_hi = r.hi * a.ln2_hi;
    const float g_lo = fmaf(r.hi, a.ln2_lo, fmaf(r.lo, a.ln2_hi, fmaf(r.hi, a.ln2_hi, -g_hi)));
    const float sq_hi = g_hi * g_hi;
    const float sq_lo = fmaf(g_hi, g_hi, -sq_hi) + 2.f * g_hi * g_lo;
    const float tail =
        sq_hi * g_hi *
        (1.f / 6.f + g_hi * (1.f / 24.f + g_hi * (1.f / 120.f + g_hi * (1.f / 720.f))));
    FF E = fast_two_sum(g_hi, 0.5f * sq_hi);
    E = fast_two_sum(E.hi, E.lo + (g_lo + 0.5f * sq_lo + tail));
    const float2 t = tab[min(max((int)kf + 16, 0), 32)];
    const float m_hi = t.x * E.hi;
    const float m_lo = fmaf(t.x, E.hi, -m_hi) + fmaf(t.x, E.lo, t.y * E.hi);
    FF w = fast_two_sum(t.x, m_hi);
    w = fast_two_sum(w.hi, w.lo + (t.y + m_lo));
    const float s = __int_as_float(((int)nf + 127) << 23);   // 2^n, n in [-126, 0]
    return {w.hi * s, w.lo * s};
}

// 2^(l * scale - M) for a logit l: scale = sc_hi + sc_lo, M an F32 shift at least the largest
// F32 product l * sc_hi it is used with (so the result is <= ~1). The product and the shift are
// carried exactly as a float-float exponent.
__device__ __forceinline__ FF weight_ff(float l, float M, const SampleArgs &a,
                                        const float2 *tab) {
    const float p_hi = l * a.sc_hi;
    const float p_lo = fmaf(l, a.sc_lo, fmaf(l, a.sc_hi, -p_hi));
    FF d = two_sum(p_hi, -M);
    d = fast_two_sum(d.hi, d.lo + p_lo);
    return exp2_ff(d, a, tab);
}

__device__ __forceinline__ const float *draft_row(const SampleArgs &a, int b, int i) {
    return a.draft + ((size_t)b * a.draft_ld + i) * a.V;
}

// Row rho of sequence b in the accept step's statistics: rho <= K is target row rho, rho > K is
// draft row rho - K - 1.
__device__ __forceinline__ const float *row_ptr(const SampleArgs &a, int b, int rho) {
    if (rho <= a.K) return a.target + ((size_t)b * (a.K + 1) + rho) * a.V;
    return draft_row(a, b, rho - a.K - 1);
}

__global__ void __launch_bounds__(kSThreads) sample_stats_kernel(SampleArgs a) {
    DF_TRACE_KERNEL(TK_SAMPLE_STATS);
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
// float-float exp sums of both rows (residual draws only).
struct DrawJob {
    const float *p, *q;
    float mp, mq;
    FF Sp, Sq;   // residual draws: the exp sums of the p and q rows
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
    j.Sp = j.Sq = {0.f, 0.f};
    return j;
}

// ------------------------------------------------------------------ block-wide float-float
// Warp sums and scans in a fixed order, then the 8 warp values in warp order; every CTA that
// runs them on the same data gets the same bits.
__device__ __forceinline__ FF ff_block_sum(FF v, FF *sh) {
    v = warp_ff_sum(v);
    __syncthreads();
    if ((threadIdx.x & 31) == 0) sh[threadIdx.x >> 5] = v;
    __syncthreads();
    FF t{0.f, 0.f};
#pragma unroll
    for (int w = 0; w < kSThreads / 32; ++w) t = ff_add(t, sh[w]);
    return t;
}

// Exclusive prefix (thread order) of v over the CTA; *total = the sum over all threads.
__device__ __forceinline__ FF ff_block_exscan(FF v, FF *sh, FF *total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    FF inc = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        FF n;
        n.hi = __shfl_up_sync(0xffffffffu, inc.hi, o);
        n.lo = __shfl_up_sync(0xffffffffu, inc.lo, o);
        if (lane >= o) inc = ff_add(n, inc);
    }
    FF ex;
    ex.hi = __shfl_up_sync(0xffffffffu, inc.hi, 1);
    ex.lo = __shfl_up_sync(0xffffffffu, inc.lo, 1);
    if (lane == 0) ex = {0.f, 0.f};
    __syncthreads();
    if (lane == 31) sh[warp] = inc;
    __syncthreads();
    FF off{0.f, 0.f}, t{0.f, 0.f};
#pragma unroll
    for (int w = 0; w < kSThreads / 32; ++w) {
        if (w < warp) off = ff_add(off, sh[w]);
        t = ff_add(t, sh[w]);
    }
    *total = t;
    return ff_add(off, ex);
}

__device__ __forceinline__ bool ff_gt(FF a, FF b) {
    return a.hi > b.hi || (a.hi == b.hi && a.lo > b.lo);
}

__device__ __forceinline__ FF ldcg_ff(const float2 *p) {
    const float2 v = __ldcg(p);
    return {v.x, v.y};
}

// The 2^(k/32) table of the draw weights, copied from the kernel parameters into shared memory
// (lanes index it with different k).
__device__ __forceinline__ void load_tab(const SampleArgs &a, float2 *tab) {
    if (threadIdx.x < 33) tab[threadIdx.x] = a.exp2_tab[threadIdx.x];
    __syncthreads();
}

// Sums of 2^(x - M) of the draw's p and q rows over one chunk (residual draws only).
__global__ void __launch_bounds__(kSThreads) sample_norm_kernel(SampleArgs a) {
    DF_TRACE_KERNEL(TK_SAMPLE_NORM);
    __shared__ float2 tab[33];
    __shared__ FF red[kSThreads / 32];
    pdl_trigger();
    pdl_wait();
    const int c = blockIdx.x, b = blockIdx.y;
    const DrawJob jb = accept_job(a, b);
    if (!jb.q) return;
    load_tab(a, tab);
    const int j0 = c * kSChunk + threadIdx.x * kEPT;
    FF sp{0.f, 0.f}, sq{0.f, 0.f};
#pragma unroll
    for (int h = 0; h < kEPT / 4; ++h) {
        if (j0 + 4 * h < a.V) {
            const float4 lp = __ldcg(reinterpret_cast<const float4 *>(jb.p + j0 + 4 * h));
            const float4 lq = __ldcg(reinterpret_cast<const float4 *>(jb.q + j0 + 4 * h));
            sp = ff_add(sp, weight_ff(lp.x, jb.mp, a, tab));
            sp = ff_add(sp, weight_ff(lp.y, jb.mp, a, tab));
            sp = ff_add(sp, weight_ff(lp.z, jb.mp, a, tab));
            sp = ff_add(sp, weight_ff(lp.w, jb.mp, a, tab));
            sq = ff_add(sq, weight_ff(lq.x, jb.mq, a, tab));
            sq = ff_add(sq, weight_ff(lq.y, jb.mq, a, tab));
            sq = ff_add(sq, weight_ff(lq.z, jb.mq, a, tab));
            sq = ff_add(sq, weight_ff(lq.w, jb.mq, a, tab));
        }
    }
    sp = ff_block_sum(sp, red);
    sq = ff_block_sum(sq, red);
    if (threadIdx.x == 0) {
        float2 *d = a.dsum + ((size_t)b * a.n_chunks + c) * 2;
        d[0] = make_float2(sp.hi, sp.lo);
        d[1] = make_float2(sq.hi, sq.lo);
    }
}

// The draw weights of thread t_idx's kEPT logits of chunk cc. Residual draws use
// max(0, p - q) scaled by S_p S_q (a draw is unchanged by a positive scale):
// 2^(x - mp) S_q - 2^(y - mq) S_p.
__device__ __forceinline__ void chunk_weights(const SampleArgs &a, const float2 *tab,
                                              const DrawJob &jb, int cc, int t_idx,
                                              FF (&w)[kEPT]) {
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
                v = weight_ff(lpv[e], jb.mp, a, tab);
                if (jb.q) {
                    const FF pn = ff_mul(v, jb.Sq);
                    const FF qn = ff_mul(weight_ff(lqv[e], jb.mq, a, tab), jb.Sp);
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

// The last CTA of a draw, step 1: thread t owns chunks [t * per, (t + 1) * per) (thread order
// is chunk order) and wcs(cc) gives chunk cc's weight sum. Finds the first chunk whose running
// sum exceeds u * total, or, when rounding puts the target past the total, the last chunk with
// weight; returns it with the running sum before it (*base) and the target.
template <typename ChunkW>
__device__ __forceinline__ int locate_chunk(int n_chunks, ChunkW wcs, float u, FF *red,
                                            int *s_pick, int *s_pick_last, FF *s_base,
                                            FF *base, FF *target, FF *total) {
    const int per = (n_chunks + kSThreads - 1) / kSThreads;   // <= kMaxChunks / kSThreads
    FF cv[kMaxChunks / kSThreads];
    FF mine{0.f, 0.f};
#pragma unroll
    for (int i = 0; i < kMaxChunks / kSThreads; ++i) {
        const int cc = threadIdx.x * per + i;
        cv[i] = (i < per && cc < n_chunks) ? wcs(cc) : FF{0.f, 0.f};
        mine = ff_add(mine, cv[i]);
    }
    if (threadIdx.x == 0) {
        *s_pick = INT_MAX;
        *s_pick_last = -1;
        *s_base = {0.f, 0.f};
    }
    FF run = ff_block_exscan(mine, red, total);   // its barriers order the resets above
    *target = ff_mul(*total, FF{u, 0.f});
    int pick = INT_MAX, pick_last = -1;
    FF base_pick{0.f, 0.f}, base_last{0.f, 0.f};
#pragma unroll
    for (int i = 0; i < kMaxChunks / kSThreads; ++i) {
        const int cc = threadIdx.x * per + i;
        if (i < per && cc < n_chunks) {
            const FF nx = ff_add(run, cv[i]);
            if (cv[i].hi > 0.f) {
                pick_last = cc;
                base_last = run;
            }
            if (pick == INT_MAX && ff_gt(nx, *target)) {
                pick = cc;
                base_pick = run;
            }
            run = nx;
        }
    }
    atomicMin(s_pick, pick);
    atomicMax(s_pick_last, pick_last);
    __syncthreads();
    const bool found = *s_pick != INT_MAX;
    const int cstar = found ? *s_pick : max(*s_pick_last, 0);
    if (found ? pick == cstar : pick_last == cstar) *s_base = found ? base_pick : base_last;
    __syncthreads();
    *base = *s_base;
    return cstar;
}

// Step 2: thread t holds weights w of indices j0 .. j0 + kEPT - 1 of the chunk (thread order is
// index order); the running sum at index j is base + fac * (the chunk's weights up to j). The
// first index whose running sum exceeds the target, else the last index with weight, else -1.
__device__ __forceinline__ int locate_in_chunk(const FF (&w)[kEPT], int j0, int V, FF base,
                                               FF fac, FF target, FF *red, int *s_pick,
                                               int *s_pick_last) {
    __syncthreads();   // the step-1 readers of *s_pick are done
    if (threadIdx.x == 0) {
        *s_pick = INT_MAX;
        *s_pick_last = -1;
    }
    FF ctot;
    FF run = ff_block_exscan(thread_sum(w), red, &ctot);
    int pick = INT_MAX, pick_last = -1;
#pragma unroll
    for (int i = 0; i < kEPT; ++i) {
        if (j0 + i < V) {
            const FF nx = ff_add(run, w[i]);
            if (w[i].hi > 0.f) pick_last = j0 + i;
            if (pick == INT_MAX && ff_gt(ff_add(base, ff_mul(fac, nx)), target)) pick = j0 + i;
            run = nx;
        }
    }
    atomicMin(s_pick, pick);
    atomicMax(s_pick_last, pick_last);
    __syncthreads();
    return *s_pick != INT_MAX ? *s_pick : *s_pick_last;
}

// Accept mode, grid (chunks, B): the draw of sequence b, then its committed tokens. Every chunk
// CTA writes its chunk's weight sum; the last one to finish locates the chunk, then the token.
__global__ void __launch_bounds__(kSThreads) sample_draw_kernel(SampleArgs a) {
    DF_TRACE_KERNEL(TK_SAMPLE_DRAW);
    __shared__ float2 tab[33];
    __shared__ FF red[kSThreads / 32];
    __shared__ int s_last, s_pick, s_pick_last;
    __shared__ FF s_base;
    pdl_trigger();
    pdl_wait();
    load_tab(a, tab);
    const int c = blockIdx.x, job = blockIdx.y;
    DrawJob jb = accept_job(a, job);
    if (jb.q) {
        // S_p and S_q from the norm kernel's chunk sums; every CTA of the draw runs the same
        // reduction, so all of them scale the weights identically
        FF sp{0.f, 0.f}, sq{0.f, 0.f};
        const float2 *ds = a.dsum + (size_t)job * a.n_chunks * 2;
        for (int cc = threadIdx.x; cc < a.n_chunks; cc += kSThreads) {
            sp = ff_add(sp, ldcg_ff(ds + 2 * cc));
            sq = ff_add(sq, ldcg_ff(ds + 2 * cc + 1));
        }
        sp = ff_block_sum(sp, red);
        sq = ff_block_sum(sq, red);
        if (!(sp.hi > 0.f) || !(sq.hi > 0.f)) {
            if (threadIdx.x == 0) set_status(a.status, DF_EINVAL);
            jb.q = nullptr;   // degenerate input: draw from p
        } else {
            jb.Sp = sp;
            jb.Sq = sq;
        }
    }
    FF w[kEPT];
    chunk_weights(a, tab, jb, c, threadIdx.x, w);
    const FF cs_own = ff_block_sum(thread_sum(w), red);
    if (threadIdx.x == 0) a.csum[(size_t)job * a.n_chunks + c] = make_float2(cs_own.hi, cs_own.lo);
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) s_last = atomicAdd(&a.counters[job], 1) == a.n_chunks - 1;
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    if (threadIdx.x == 0) a.counters[job] = 0;   // left at zero for the next call
    const float2 *cs = a.csum + (size_t)job * a.n_chunks;
    FF base, target, tot;
    const int cstar = locate_chunk(
        a.n_chunks, [&](int cc) { return ldcg_ff(cs + cc); }, jb.u, red, &s_pick,
        &s_pick_last, &s_base, &base, &target, &tot);
    if (threadIdx.x == 0 && !(tot.hi > 0.f)) set_status(a.status, DF_EINVAL);
    chunk_weights(a, tab, jb, cstar, threadIdx.x, w);
    int idx = locate_in_chunk(w, cstar * kSChunk + threadIdx.x * kEPT, a.V, base, FF{1.f, 0.f},
                              target, red, &s_pick, &s_pick_last);
    if (threadIdx.x != 0) return;
    if (idx < 0) idx = cstar * kSChunk;
    if (!df_in_bounds(idx >= 0 && idx < a.V, a.status)) idx = 0;
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

// Sample mode, one pass: grid (chunks, B * K), draw b * K + i is draft i of sequence b, from
// softmax(draft row i / T). Each chunk CTA takes its own maximum m_c as the shift and writes m_c
// and S_c = sum of 2^(x - m_c); the last CTA of the draw rescales the chunk sums by
// 2^(m_c - M) (M the row maximum), locates the chunk, and recomputes that chunk's weights with
// the same shift for the token.
__global__ void __launch_bounds__(kSThreads) sample_fused_kernel(SampleArgs a) {
    DF_TRACE_KERNEL(TK_SAMPLE_FUSED);
    __shared__ float2 tab[33];
    __shared__ FF red[kSThreads / 32];
    __shared__ float wm[kSThreads / 32];
    __shared__ int s_last, s_pick, s_pick_last;
    __shared__ FF s_base;
    pdl_trigger();
    pdl_wait();
    load_tab(a, tab);
    const int c = blockIdx.x, job = blockIdx.y;
    const int b = job / a.K, i = job - b * a.K;
    const float *row = draft_row(a, b, i);
    const float u = a.u_draft[job];
    float *cm = &a.stats[(size_t)job * a.n_chunks].m;   // m_c, stride sizeof(MaxSum) / 4
    constexpr int kMS = sizeof(MaxSum) / sizeof(float);
    float2 *cs = a.csum + (size_t)job * a.n_chunks;
    auto load = [&](int cc, float (&l)[kEPT]) {
        const int j0 = cc * kSChunk + threadIdx.x * kEPT;
#pragma unroll
        for (int h = 0; h < kEPT / 4; ++h) {
            float4 v = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
            if (j0 + 4 * h < a.V) v = __ldcg(reinterpret_cast<const float4 *>(row + j0 + 4 * h));
            l[4 * h] = v.x;
            l[4 * h + 1] = v.y;
            l[4 * h + 2] = v.z;
            l[4 * h + 3] = v.w;
        }
    };
    float l[kEPT];
    load(c, l);
    float m = -INFINITY;
#pragma unroll
    for (int e = 0; e < kEPT; ++e) m = fmaxf(m, l[e] * a.sc_hi);
    m = warp_max(m);
    if ((threadIdx.x & 31) == 0) wm[threadIdx.x >> 5] = m;
    __syncthreads();
    float mc = wm[0];
#pragma unroll
    for (int w_ = 1; w_ < kSThreads / 32; ++w_) mc = fmaxf(mc, wm[w_]);
    FF w[kEPT];
#pragma unroll
    for (int e = 0; e < kEPT; ++e) w[e] = weight_ff(l[e], mc, a, tab);
    FF sc;
    ff_block_exscan(thread_sum(w), red, &sc);
    if (threadIdx.x == 0) {
        cm[(size_t)c * kMS] = mc;
        cs[c] = make_float2(sc.hi, sc.lo);
    }
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) s_last = atomicAdd(&a.counters[job], 1) == a.n_chunks - 1;
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    if (threadIdx.x == 0) a.counters[job] = 0;   // left at zero for the next call
    // the row maximum M over the chunk maxima (exact), then each chunk's scale 2^(m_c - M)
    float M = -INFINITY;
    for (int cc = threadIdx.x; cc < a.n_chunks; cc += kSThreads) M = fmaxf(M, __ldcg(cm + (size_t)cc * kMS));
    M = warp_max(M);
    __syncthreads();
    if ((threadIdx.x & 31) == 0) wm[threadIdx.x >> 5] = M;
    __syncthreads();
    M = wm[0];
#pragma unroll
    for (int w_ = 1; w_ < kSThreads / 32; ++w_) M = fmaxf(M, wm[w_]);
    auto fac = [&](int cc) { return exp2_ff(two_sum(__ldcg(cm + (size_t)cc * kMS), -M), a, tab); };
    FF base, target, tot;
    const int cstar = locate_chunk(
        a.n_chunks, [&](int cc) { return ff_mul(ldcg_ff(cs + cc), fac(cc)); }, u, red, &s_pick,
        &s_pick_last, &s_base, &base, &target, &tot);
    if (threadIdx.x == 0 && !(tot.hi > 0.f)) set_status(a.status, DF_EINVAL);
    const float mstar = __ldcg(cm + (size_t)cstar * kMS);
    load(cstar, l);
#pragma unroll
    for (int e = 0; e < kEPT; ++e) w[e] = weight_ff(l[e], mstar, a, tab);
    int idx = locate_in_chunk(w, cstar * kSChunk + threadIdx.x * kEPT, a.V, base, fac(cstar),
                              target, red, &s_pick, &s_pick_last);
    if (threadIdx.x != 0) return;
    if (idx < 0) idx = cstar * kSChunk;
    if (!df_in_bounds(idx >= 0 && idx < a.V, a.status)) idx = 0;
    a.drafts_out[job] = idx;
}

}  // namespace

int sample_chunks(int V) { return (V + kSChunk - 1) / kSChunk; }

void carve_sample_scratch(Carve &cv, SampleArgs &a, int B, int K, int V) {
    a.n_chunks = sample_chunks(V);
    a.stats = cv.take<MaxSum>((size_t)B * (2 * K + 1) * a.n_chunks);
    a.state = cv.take<SampleState>((size_t)B);
    a.dsum = cv.take<float2>((size_t)B * a.n_chunks * 2);
    a.csum = cv.take<float2>((size_t)B * K * a.n_chunks);
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
    return launch_k("sample_fused_kernel", sample_fused_kernel, dim3(a.n_chunks, a.B * a.K),
                    dim3(kSThreads), 0, s, a);
}

}  // namespace df

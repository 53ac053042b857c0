// Mixture-of-experts FFN of the MTP block: router, softmax top-k, the chosen experts' SwiGLUs
// and one shared expert scaled by a sigmoid gate.
//
// hf2q 0.1.1 models/qwen35/mtp.rs, `MtpFfnWeightsGpu::Moe` (router, per-expert gate/up/down,
// shared expert and its scalar gate). The page names the tensors but not the routing rule; it
// is read as: softmax over all experts, the top_k largest probabilities (the lower expert index
// first on equal values), weights renormalised to sum to one, plus the shared expert's SwiGLU
// times sigmoid(x . w_shared_gate).
//
// At most 16 rows (one per sequence) go through this FFN, so every product here is a
// matrix-vector product: weight rows stream once per row that uses them as 128-bit loads on
// the CUDA cores and the activations stay in F32. Three kernels:
//   router  : logits[t, e] = x_t . router[e] (e < E) and x_t . w_shared_gate (e = E); the last
//             CTA to finish picks the top_k experts of every row and their weights
//   gate_up : act[t, j, r] = silu(g) * u with g, u row r of expert sel[t, j]'s gate/up
//             (slot j = top_k is the shared expert)
//   down    : part[j, t, h] = weight[t, j] * (down_j[h] . act[t, j]); the consumer adds the
//             top_k + 1 slot outputs in slot order.
#include "df_internal.cuh"

namespace df {

namespace {

constexpr int kMoeThreads = 256;
constexpr int kMoeWarps = kMoeThreads / 32;
constexpr int kDownRows = 4;     // output rows per warp in the down kernel

// 8 BF16 values (one 128-bit load) against 8 F32 values at x (16-byte aligned).
__device__ __forceinline__ float dot8(const uint4 &w, const float *x, float acc) {
    const float4 a = *reinterpret_cast<const float4 *>(x);
    const float4 b = *reinterpret_cast<const float4 *>(x + 4);
    acc = fmaf(__uint_as_float(w.x << 16), a.x, acc);
    acc = fmaf(__uint_as_float(w.x & 0xffff0000u), a.y, acc);
    acc = fmaf(__uint_as_float(w.y << 16), a.z, acc);
    acc = fmaf(__uint_as_float(w.y & 0xffff0000u), a.w, acc);
    acc = fmaf(__uint_as_float(w.z << 16), b.x, acc);
    acc = fmaf(__uint_as_float(w.z & 0xffff0000u), b.y, acc);
    acc = fmaf(__uint_as_float(w.w << 16), b.z, acc);
    acc = fmaf(__uint_as_float(w.w & 0xffff0000u), b.w, acc);
    return acc;
}

__device__ __forceinline__ uint4 ld_w(const uint16_t *p, bool ok) {
    return ok ? ld_stream_u4(p) : make_uint4(0u, 0u, 0u, 0u);
}

// Asks L2 for n_bytes of weights at p, one 128-byte line per lane and step (no registers held):
// used before a kernel's wait on its predecessor, for weights that do not depend on it.
__device__ __forceinline__ void prefetch_l2(const void *p, size_t n_bytes, int lane) {
    const char *c = static_cast<const char *>(p);
    for (size_t off = (size_t)lane * 128; off < n_bytes; off += 32 * 128)
        asm volatile("prefetch.global.L2 [%0];" ::"l"(c + off));
}

// Router: one warp per weight row (E router rows, then the shared-expert gate row), against
// all T input rows at once. The last CTA to arrive selects the experts.
__global__ void __launch_bounds__(kMoeThreads) moe_router_kernel(MoeArgs a) {
    DF_TRACE_KERNEL(TK_MOE_ROUTER);
    __shared__ int s_last;
    pdl_trigger();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int row = blockIdx.x * kMoeWarps + warp;
    const int nch = a.H >> 3;
    const int E1 = a.E + 1;
    if (row < E1) {
        const uint16_t *w = row < a.E ? a.router + (size_t)row * a.H : a.sh_gate;
        float acc[kMoeMaxRows];
#pragma unroll
        for (int t = 0; t < kMoeMaxRows; ++t) acc[t] = 0.f;
        uint4 wv[8];
        // The first batch of weights does not depend on earlier kernels: issue it before the wait.
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int c = i * 32 + lane;
            wv[i] = ld_w(w + 8 * (size_t)c, c < nch);
        }
        pdl_wait();
        for (int c0 = 0; c0 < nch; c0 += 256) {
            if (c0) {
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int c = c0 + i * 32 + lane;
                    wv[i] = ld_w(w + 8 * (size_t)c, c < nch);
                }
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int c = c0 + i * 32 + lane;
                if (c < nch) {
#pragma unroll
                    for (int t = 0; t < kMoeMaxRows; ++t)
                        if (t < a.T) acc[t] = dot8(wv[i], a.x + (size_t)t * a.ldx + 8 * c, acc[t]);
                }
            }
        }
#pragma unroll
        for (int t = 0; t < kMoeMaxRows; ++t) {
            if (t < a.T) {
                const float v = warp_sum(acc[t]);
                if (lane == 0) a.logits[(size_t)t * E1 + row] = v;
            }
        }
    } else {
        pdl_wait();
    }

    // Last-arriving CTA: top-k of every row.
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) s_last = atomicAdd(a.counter, 1) == (int)gridDim.x - 1;
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    if (threadIdx.x == 0) *a.counter = 0;     // leave the counter at zero for the next call
    constexpr int kPerLane = kMoeMaxExperts / 32;
    for (int t = warp; t < a.T; t += kMoeWarps) {
        const float *lg = a.logits + (size_t)t * E1;
        float v[kPerLane];
        unsigned taken = 0;
#pragma unroll
        for (int i = 0; i < kPerLane; ++i) {
            const int e = i * 32 + lane;
            v[i] = e < a.E ? __ldcg(lg + e) : 0.f;
        }
        float top[kMoeMaxTopK];
        int chosen_ok = 1;
        for (int j = 0; j < a.k; ++j) {
            // per lane: its largest untaken value (its indices rise with i, so '>' keeps the
            // lowest index among equal values), then a butterfly over the lanes
            float bv = -INFINITY;
            int bi = 0x7fffffff;
#pragma unroll
            for (int i = 0; i < kPerLane; ++i) {
                const int e = i * 32 + lane;
                if (e < a.E && !((taken >> i) & 1u) && (bi == 0x7fffffff || v[i] > bv)) {
                    bv = v[i];
                    bi = e;
                }
            }
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) {
                const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
                const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
                const bool take = oi != 0x7fffffff &&
                                  (bi == 0x7fffffff || ov > bv || (ov == bv && oi < bi));
                if (take) {
                    bv = ov;
                    bi = oi;
                }
            }
            if (bi == 0x7fffffff || !(bv == bv)) chosen_ok = 0;   // no candidate, or NaN
            if (bi != 0x7fffffff && (bi & 31) == lane) taken |= 1u << (bi >> 5);
            top[j] = bv;
            if (lane == 0) a.sel[(size_t)t * a.k + j] = bi == 0x7fffffff ? 0 : bi;
        }
        if (!chosen_ok) {
            if (lane == 0) set_status(a.status, DF_EINVAL);
            continue;
        }
        // renormalised softmax over the chosen: exp(l_j - l_0) / sum_i exp(l_i - l_0)
        float den = 0.f;
        for (int j = 0; j < a.k; ++j) den += expf(top[j] - top[0]);
        if (lane == 0) {
            for (int j = 0; j < a.k; ++j)
                a.wts[(size_t)t * (a.k + 1) + j] = expf(top[j] - top[0]) / den;
            const float gl = __ldcg(lg + a.E);
            a.wts[(size_t)t * (a.k + 1) + a.k] = 1.f / (1.f + expf(-gl));
        }
    }
}

// Gate/up: one warp per (row t, slot j, intermediate index r). act[t, j, r] = silu(g) * u.
__global__ void __launch_bounds__(kMoeThreads) moe_gate_up_kernel(MoeArgs a) {
    DF_TRACE_KERNEL(TK_MOE_GATE_UP);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int S = a.k + 1, Imax = max(a.Ie, a.Is);
    const long long task = (long long)blockIdx.x * kMoeWarps + warp;
    const int r = (int)(task % Imax);
    const long long q = task / Imax;
    const int j = (int)(q % S), t = (int)(q / S);
    // The shared expert does not depend on the router: its rows are requested before the wait.
    if (t < a.T && j == a.k && r < a.Is) {
        prefetch_l2(a.sh_g + (size_t)r * a.H, (size_t)a.H * 2, lane);
        prefetch_l2(a.sh_u + (size_t)r * a.H, (size_t)a.H * 2, lane);
    }
    pdl_wait();
    // Released only past the wait: when the down kernel starts, the router (which wrote the
    // expert choice) has completed, so down can request its experts' rows before its own wait.
    pdl_trigger();
    if (t >= a.T) return;
    const int I = j < a.k ? a.Ie : a.Is;
    if (r >= I) return;
    const uint16_t *wg, *wu;
    if (j < a.k) {
        const int e = a.sel[(size_t)t * a.k + j];
        if (e < 0 || e >= a.E) {
            if (lane == 0) set_status(a.status, DF_EINVAL);
            return;
        }
        wg = a.exp_gate + ((size_t)e * a.Ie + r) * a.H;
        wu = a.exp_up + ((size_t)e * a.Ie + r) * a.H;
    } else {
        wg = a.sh_g + (size_t)r * a.H;
        wu = a.sh_u + (size_t)r * a.H;
    }
    const float *x = a.x + (size_t)t * a.ldx;
    const int nch = a.H >> 3;
    float g = 0.f, u = 0.f;
    for (int c0 = 0; c0 < nch; c0 += 256) {
        uint4 gv[8], uv[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int c = c0 + i * 32 + lane;
            gv[i] = ld_w(wg + 8 * (size_t)c, c < nch);
            uv[i] = ld_w(wu + 8 * (size_t)c, c < nch);
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int c = c0 + i * 32 + lane;
            if (c < nch) {
                g = dot8(gv[i], x + 8 * c, g);
                u = dot8(uv[i], x + 8 * c, u);
            }
        }
    }
    g = warp_sum(g);
    u = warp_sum(u);
    if (lane == 0) a.act[((size_t)t * S + j) * Imax + r] = g / (1.f + expf(-g)) * u;
}

// Down: one warp per (slot j, row t, block of kDownRows output rows).
// part[j, t, h] = weight[t, j] * (down_j[h, :] . act[t, j, :]).
__global__ void __launch_bounds__(kMoeThreads) moe_down_kernel(MoeArgs a) {
    DF_TRACE_KERNEL(TK_MOE_DOWN);
    pdl_trigger();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int S = a.k + 1, Imax = max(a.Ie, a.Is);
    const int nhb = (a.H + kDownRows - 1) / kDownRows;
    const long long task = (long long)blockIdx.x * kMoeWarps + warp;
    const int hb = (int)(task % nhb);
    const long long q = task / nhb;
    const int t = (int)(q % a.T), j = (int)(q / a.T);
    const int I = j < a.k ? a.Ie : a.Is;
    const int h0 = hb * kDownRows;
    if (j < S && h0 < a.H) {
        // The router has completed (the gate/up kernel releases this one only past its own
        // wait): request this warp's rows of the chosen expert before waiting for the
        // activations. The choice is read again after the wait; a stale one costs a prefetch.
        const uint16_t *b = a.sh_d;
        if (j < a.k) {
            const int e = __ldcg(a.sel + (size_t)t * a.k + j);
            b = e >= 0 && e < a.E ? a.exp_down + (size_t)e * a.H * a.Ie : nullptr;
        }
        if (b) prefetch_l2(b + (size_t)h0 * I, (size_t)min(kDownRows, a.H - h0) * I * 2, lane);
    }
    pdl_wait();
    if (j >= S) return;
    const uint16_t *base;
    if (j < a.k) {
        const int e = a.sel[(size_t)t * a.k + j];
        if (e < 0 || e >= a.E) {
            if (lane == 0) set_status(a.status, DF_EINVAL);
            return;
        }
        base = a.exp_down + (size_t)e * a.H * a.Ie;
    } else {
        base = a.sh_d;
    }
    const float *act = a.act + ((size_t)t * S + j) * Imax;
    const int nch = I >> 3;
    float acc[kDownRows];
#pragma unroll
    for (int rr = 0; rr < kDownRows; ++rr) acc[rr] = 0.f;
    for (int c0 = 0; c0 < nch; c0 += 64) {
        uint4 wv[kDownRows][2];
#pragma unroll
        for (int rr = 0; rr < kDownRows; ++rr)
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const int c = c0 + i * 32 + lane;
                wv[rr][i] = ld_w(base + (size_t)(h0 + rr) * I + 8 * c, c < nch && h0 + rr < a.H);
            }
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int c = c0 + i * 32 + lane;
            if (c < nch) {
#pragma unroll
                for (int rr = 0; rr < kDownRows; ++rr) acc[rr] = dot8(wv[rr][i], act + 8 * c, acc[rr]);
            }
        }
    }
    const float wt = a.wts[(size_t)t * S + j];
    float *out = a.part + ((size_t)j * a.T + t) * a.ldpart;
#pragma unroll
    for (int rr = 0; rr < kDownRows; ++rr) {
        const float v = warp_sum(acc[rr]);
        if (lane == 0 && h0 + rr < a.H) out[h0 + rr] = wt * v;
    }
}

}  // namespace

int launch_moe(const MoeArgs &a, cudaStream_t s) {
    const int S = a.k + 1, Imax = std::max(a.Ie, a.Is);
    const int g_router = (a.E + 1 + kMoeWarps - 1) / kMoeWarps;
    DF_TRY(launch_k("moe_router", moe_router_kernel, dim3(g_router), dim3(kMoeThreads), 0, s, a));
    const long long up_tasks = (long long)a.T * S * Imax;
    DF_TRY(launch_k("moe_gate_up", moe_gate_up_kernel,
                    dim3((unsigned)((up_tasks + kMoeWarps - 1) / kMoeWarps)), dim3(kMoeThreads), 0,
                    s, a));
    const long long dn_tasks = (long long)S * a.T * ((a.H + kDownRows - 1) / kDownRows);
    return launch_k("moe_down", moe_down_kernel,
                    dim3((unsigned)((dn_tasks + kMoeWarps - 1) / kMoeWarps)), dim3(kMoeThreads), 0,
                    s, a);
}

}  // namespace df

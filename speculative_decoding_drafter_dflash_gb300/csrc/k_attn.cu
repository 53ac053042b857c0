// Attention block of a drafter layer: per-head q/k RMSNorm + RoPE + KV append, split-KV
// SDPA with a two-pass (partial, combine) softmax, optional sigmoid output gate, and the
// packing of the attention output for the O projection.
//
// hf2q 0.1.1 models/qwen35/mtp.rs `forward_full_attention`: `apply_q_or_k_per_head_rms_norm`,
// `apply_imrope` (text positions: all four ids equal, i.e. plain RoPE),
// `apply_sdpa_with_kv_cache` (append at the slot position, then softmax(q K^T / sqrt(d)) V
// with grouped KV heads), `apply_sigmoid_gate_multiply`. DFlash: tensors.rs
// `DFlashLayerTensors::q_norm/k_norm`; the context rows of qwen35_orchestrator.rs step 3.
#include <math.h>
#include <string.h>

#include <algorithm>
#include <cmath>

#include "df_internal.cuh"

namespace df {

namespace {

// cos/sin of pos * theta^(-2j/rot), rounded to F32. The inverse frequencies come from the host
// in double precision (GB300's FP64 rate makes per-element exp2/log2 the slowest step of a
// round); the angle is formed and reduced to [-pi, pi] in double, then its sine and cosine are
// taken in F32.
struct RopeArgs {
    float *cos_t, *sin_t;
    const int32_t *seq_len, *n_new;
    int n_new_max, B, blk, pos_off, rot;
    int32_t *status;
    double inv[kMaxRopeHalf];
};

__global__ void rope_table_kernel(const __grid_constant__ RopeArgs a) {
    DF_TRACE_KERNEL(TK_ROPE_TABLE);
    pdl_trigger();
    pdl_wait();
    const int half = a.rot / 2;
    const int slots = a.blk + a.n_new_max;
    const int total = a.B * slots * half;
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < total; i += gridDim.x * blockDim.x) {
        const int j = i % half;
        const int s = (i / half) % slots;
        const int b = i / (half * slots);
        const int base = a.seq_len[b];
        const int nn = a.n_new ? min(max(a.n_new[b], 0), a.n_new_max) : 0;
        if (a.status && j == 0 && s == 0 && a.n_new && (a.n_new[b] < 0 || a.n_new[b] > a.n_new_max))
            set_status(a.status, DF_ESHAPE);
        const long long pos = s < a.blk ? (long long)base + nn + s + a.pos_off : (long long)base + (s - a.blk);
        const double ang = (double)pos * a.inv[j];
        const double two_pi = 6.283185307179586476925286766559;
        const double red = fma(-rint(ang * (1.0 / two_pi)), two_pi, ang);
        float sn, cs;
        sincosf((float)red, &sn, &cs);
        a.cos_t[i] = cs;
        a.sin_t[i] = sn;
    }
}

// One warp per (token row, head slot). Slots: [0, nq) q heads, [nq, nq+nkv) k heads,
// [nq+nkv, nq+2nkv) v heads. Rows [0, B*blk) are block rows, the rest context rows.
__global__ void qk_rope_kernel(QkArgs a) {
    DF_TRACE_KERNEL(TK_QK_ROPE);
    extern __shared__ float smem[];
    pdl_trigger();
    pdl_wait();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int wpb = blockDim.x >> 5;
    const int slots = a.nq + 2 * a.nkv + a.n_gate_heads;
    const int T_blk = a.B * a.blk;
    const int T_all = T_blk + a.B * a.n_new_max;
    const long long gw = (long long)blockIdx.x * wpb + warp;
    if (gw >= (long long)T_all * slots) return;
    const int row = (int)(gw / slots);
    const int slot = (int)(gw % slots);
    const int d = a.d, half = a.rot / 2, ept = d / 32;
    float *buf = smem + warp * d;

    const bool is_block = row < T_blk;
    int b, i;
    if (is_block) {
        b = row / a.blk;
        i = row % a.blk;
    } else {
        b = (row - T_blk) / a.n_new_max;
        i = (row - T_blk) % a.n_new_max;
        if (slot < a.nq || slot >= a.nq + 2 * a.nkv) return;   // context rows feed only K/V
        int nn = min(max(a.n_new[b], 0), a.n_new_max);
        if (i >= nn) return;
    }
    const bool is_gate = slot >= a.nq + 2 * a.nkv;
    const bool is_q = slot < a.nq;
    const bool is_k = !is_q && slot < a.nq + a.nkv;
    const int head = is_gate ? slot - a.nq - 2 * a.nkv
                             : (is_q ? slot : (is_k ? slot - a.nq : slot - a.nq - a.nkv));
    const int col = is_gate ? (a.nq + 2 * a.nkv) * d + head * d
                            : (is_q ? head * d
                                    : (is_k ? a.nq * d + head * d : (a.nq + a.nkv) * d + head * d));

    // The norm weights and this row's cos/sin are requested before the projection partials,
    // so they arrive in the same round trip.
    const bool rotate = !is_gate && slot < a.nq + a.nkv;
    float nwv[8], cv[8], sv[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
        nwv[u] = 1.f;
        cv[u] = 1.f;
        sv[u] = 0.f;
    }
    if (rotate) {
        const float *nw = is_q ? a.q_norm : a.k_norm;
        const int tslot = is_block ? i : a.blk + i;
        const float *ct = a.cos_t + ((size_t)b * (a.blk + a.n_new_max) + tslot) * half;
        const float *st = a.sin_t + ((size_t)b * (a.blk + a.n_new_max) + tslot) * half;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int e = lane + 32 * u;
            if (u < ept) {
                if (nw) nwv[u] = nw[e];
                if (e < a.rot) {
                    const int f = e < half ? e : e - half;
                    cv[u] = ct[f];
                    sv[u] = st[f];
                }
            }
        }
    }
    float x[8];
    if (a.part) {
        // deferred split-K: every split is loaded first, then summed in split order
#pragma unroll
        for (int u = 0; u < 8; ++u) x[u] = 0.f;
        for (int sp0 = 0; sp0 < a.n_part; sp0 += 4) {
            float pv[4][8];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float *src = a.part + (size_t)(sp0 + j) * a.part_stride + (size_t)row * a.ldq + col;
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    pv[j][u] = (sp0 + j < a.n_part && u < ept) ? src[lane + 32 * u] : 0.f;
            }
#pragma unroll
            for (int j = 0; j < 4; ++j)
#pragma unroll
                for (int u = 0; u < 8; ++u) x[u] += pv[j][u];
        }
    } else {
        const float *src = a.qkv + (size_t)row * a.ldq + col;
#pragma unroll
        for (int u = 0; u < 8; ++u) x[u] = (u < ept) ? src[lane + 32 * u] : 0.f;
    }
    if (is_gate) {
        float *g = a.gate_out + (size_t)row * a.ldg + head * d;
#pragma unroll
        for (int u = 0; u < 8; ++u)
            if (u < ept) g[lane + 32 * u] = x[u];
        return;
    }

    if (rotate) {   // q or k: per-head RMSNorm, then RoPE
        if (is_q ? a.q_norm : a.k_norm) {
            float ss = 0.f;
#pragma unroll
            for (int u = 0; u < 8; ++u) ss = fmaf(x[u], x[u], ss);
            ss = warp_sum(ss);
            float inv = 1.f / sqrtf(ss / (float)d + a.eps);
#pragma unroll
            for (int u = 0; u < 8; ++u)
                if (u < ept) x[u] = x[u] * inv * nwv[u];
        }
#pragma unroll
        for (int u = 0; u < 8; ++u)
            if (u < ept) buf[lane + 32 * u] = x[u];
        __syncwarp();
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            int e = lane + 32 * u;
            if (u < ept && e < a.rot) {
                if (e < half) x[u] = buf[e] * cv[u] - buf[e + half] * sv[u];
                else x[u] = buf[e] * cv[u] + buf[e - half] * sv[u];
            }
        }
    }

    float *dst = nullptr;
    if (is_q) {
        dst = a.q_out + (((size_t)b * a.blk + i) * a.nq + head) * d;
    } else {
        float *cache = is_k ? a.cache_k : a.cache_v;
        float *blkbuf = is_k ? a.kb : a.vb;
        if (is_block && !a.append_block) {
            dst = blkbuf + (((size_t)b * a.nkv + head) * a.blk + i) * d;
        } else {
            // Context rows (and MTP block rows) go to cache row seq_len + position.
            int nn = a.n_new ? min(max(a.n_new[b], 0), a.n_new_max) : 0;
            long long p = is_block ? (long long)a.seq_len[b] + nn + i + a.pos_off
                                   : (long long)a.seq_len[b] + i;
            if (p < 0 || p >= a.cap) {
                if (lane == 0) set_status(a.status, DF_ECAPACITY);
                return;
            }
            dst = cache + (((size_t)b * a.nkv + head) * a.cap + p) * d;
        }
    }
    if (!is_q && a.kv_bf16) {
        // BF16 KV cache: cached rows are stored as BF16, block rows keep the rounded values
        const bool to_cache = !(is_block && !a.append_block);
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            if (u >= ept) continue;
            const uint16_t bits = f32_to_bf16_bits(x[u]);
            if (to_cache) {
                const size_t idx = (size_t)(dst - (is_k ? a.cache_k : a.cache_v)) + lane + 32 * u;
                reinterpret_cast<uint16_t *>(is_k ? a.cache_k : a.cache_v)[idx] = bits;
            } else {
                dst[lane + 32 * u] = bf16_bits_to_f32(bits);
            }
        }
        return;
    }
#pragma unroll
    for (int u = 0; u < 8; ++u)
        if (u < ept) dst[lane + 32 * u] = x[u];
}

constexpr int kAttnThreads = 256;
constexpr int kAttnStages = 4;
constexpr int kTileBytes = 32768;          // K + V bytes of one key tile
constexpr int kKeyGroup = 8;               // keys per online-softmax update

// 2^x with the hardware approximation (relative error ~2^-22; 2^-inf = 0).
__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

// Bounded wait for a phase of an mbarrier (~2 s); on timeout DF_ETIMEOUT is raised and the
// caller continues with whatever the buffer holds (results are then invalid, nothing hangs).
__device__ __forceinline__ void attn_wait(uint64_t *bar, uint32_t parity, int32_t *status) {
    const long long t0 = clock64();
    uint32_t ok = 0;
    while (true) {
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(ok)
            : "r"(smem_addr(bar)), "r"(parity)
            : "memory");
        if (ok) return;
        if (clock64() - t0 > 4000000000LL) {
            set_status(status, DF_ETIMEOUT);
            return;
        }
    }
}

// Split-KV attention for one (key chunk, KV head, sequence). A "row set" is RPL query rows of
// one block token whose q heads share this KV head (RPL = 2 when the GQA group allows), so
// every key/value element a lane loads from shared memory feeds RPL rows. Each row set is
// owned by LPR = D/32 lanes; lane sub of a row set holds the interleaved head dimensions
// {4*LPR*j + 4*sub + c} of q and of the running outputs (32 floats per row), so at every step
// the LPR lanes read adjacent 16-byte words of a key row (no bank conflicts, no index
// arithmetic in the inner loop) and the row sets of a warp share them by broadcast. Warps
// split the row sets into row groups and every key tile into key subsets. Key/value tiles
// stream into shared memory through bulk copies. Scores are kept in log2 units (q is
// pre-scaled by log2(e)/sqrt(D)). The CTA merges its key subsets and writes one partial
// (o, m, l) per query row; attn_combine_kernel merges the chunks.
template <int D, int RPL>
__global__ void __launch_bounds__(kAttnThreads, 1) attn_kernel(AttnArgs a) {
    DF_TRACE_KERNEL(TK_ATTN);
    constexpr int LPR = D / 32;
    constexpr int DL = 32;
    constexpr int RPW = 32 / LPR;                  // row sets per warp
    constexpr int NW = kAttnThreads / 32;
    constexpr int TK = kTileBytes / (2 * D * 4);
    extern __shared__ __align__(128) uint8_t sm_raw[];
    float *tiles = reinterpret_cast<float *>(sm_raw);
    uint64_t *full = reinterpret_cast<uint64_t *>(sm_raw + (size_t)kAttnStages * kTileBytes);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int chunk = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
    pdl_trigger();
    pdl_wait();
    const int rep = a.nq / a.nkv;
    const int R = a.blk * rep;                     // query rows of this KV head
    const int NS = R / RPL;                        // row sets
    const int RG = (NS + RPW - 1) / RPW;
    const int KS = RG >= NW ? 1 : NW / RG;
    const int rg = warp % RG, ks = warp / RG;
    const bool active = ks < KS && warp < RG * KS;
    const int sub = lane / RPW, rsl = lane % RPW;
    const int rs = rg * RPW + rsl;                 // row set of this lane
    const bool set_valid = active && rs < NS;
    // rows rr = rs * RPL + r: token rr / rep, q head g * rep + rr % rep
    const int tok = set_valid ? (rs * RPL) / rep : 0;

    const int nn = a.n_new ? min(max(a.n_new[b], 0), a.n_new_max) : 0;
    const long long sc = (long long)a.seq_len[b] + nn + a.extra_rows;
    const int S_cache = (int)min(max(sc, 0LL), (long long)a.cap);
    const int S = S_cache + (a.kb ? a.blk : 0);
    const int c0 = min(S, chunk * a.chunk), c1 = min(S, c0 + a.chunk);
    const int n_tiles = (c1 - c0 + TK - 1) / TK;
    const size_t head_off = (size_t)b * a.nkv + g;

    float2 q2[RPL][DL / 2];
    {
        const float qs = 1.4426950408889634f / sqrtf((float)D);
#pragma unroll
        for (int r = 0; r < RPL; ++r) {
            const int rr = rs * RPL + r;
            const int qh = g * rep + (set_valid ? rr % rep : 0);
            const float *qp = a.q + (((size_t)b * a.blk + tok) * a.nq + qh) * D + 4 * sub;
#pragma unroll
            for (int j = 0; j < DL / 4; ++j) {
                float4 v = set_valid ? *reinterpret_cast<const float4 *>(qp + 4 * LPR * j)
                                     : make_float4(0.f, 0.f, 0.f, 0.f);
                q2[r][2 * j] = make_float2(v.x * qs, v.y * qs);
                q2[r][2 * j + 1] = make_float2(v.z * qs, v.w * qs);
            }
        }
    }
    float2 o2[RPL][DL / 2];
    float m[RPL], l[RPL];
#pragma unroll
    for (int r = 0; r < RPL; ++r) {
        m[r] = -INFINITY;
        l[r] = 0.f;
#pragma unroll
        for (int j = 0; j < DL / 2; ++j) o2[r][j] = make_float2(0.f, 0.f);
    }

    auto issue = [&](int jt) {
        const int st = jt % kAttnStages;
        const int t0 = c0 + jt * TK;
        const int n = min(TK, c1 - t0);
        const int ncache = max(0, min(n, S_cache - t0));
        const int nblock = n - ncache;
        float *kd = tiles + (size_t)st * (kTileBytes / 4);
        float *vd = kd + TK * D;
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(&full[st])),
                     "r"((uint32_t)(2 * n * D * 4))
                     : "memory");
        if (ncache > 0) {
            const size_t off = (head_off * a.cap + t0) * D;
            bulk_g2s(kd, a.cache_k + off, ncache * D * 4, &full[st]);
            bulk_g2s(vd, a.cache_v + off, ncache * D * 4, &full[st]);
        }
        if (nblock > 0) {
            const int bs = max(0, t0 - S_cache);
            const size_t off = (head_off * a.blk + bs) * D;
            bulk_g2s(kd + ncache * D, a.kb + off, nblock * D * 4, &full[st]);
            bulk_g2s(vd + ncache * D, a.vb + off, nblock * D * 4, &full[st]);
        }
    };

    if (tid == 0) {
        for (int s2 = 0; s2 < kAttnStages; ++s2)
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(&full[s2])));
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    if (tid == 0)
        for (int jt = 0; jt < min(kAttnStages, n_tiles); ++jt) issue(jt);

    const int KW = (TK + KS - 1) / KS;
    for (int jt = 0; jt < n_tiles; ++jt) {
        const int st = jt % kAttnStages;
        attn_wait(&full[st], (uint32_t)((jt / kAttnStages) & 1), a.status);
        const int t0 = c0 + jt * TK;
        const int n = min(TK, c1 - t0);
        const float *kt = tiles + (size_t)st * (kTileBytes / 4) + 4 * sub;
        const float *vt = kt + TK * D;
        const int kbeg = ks * KW, kend = min(n, kbeg + KW);
        if (active) {
            for (int k0 = kbeg; k0 < kend; k0 += kKeyGroup) {
                const int nk = min(kKeyGroup, kend - k0);
                const bool fullg = nk == kKeyGroup;
                float s[kKeyGroup][RPL];
#pragma unroll
                for (int u = 0; u < kKeyGroup; ++u) {
                    const float *kr = kt + (size_t)(k0 + (fullg ? u : min(u, nk - 1))) * D;
                    float2 acc[RPL];
#pragma unroll
                    for (int r = 0; r < RPL; ++r) acc[r] = make_float2(0.f, 0.f);
#pragma unroll
                    for (int j = 0; j < DL / 4; ++j) {
                        const float4 kv = *reinterpret_cast<const float4 *>(kr + 4 * LPR * j);
                        const float2 k01 = make_float2(kv.x, kv.y), k23 = make_float2(kv.z, kv.w);
#pragma unroll
                        for (int r = 0; r < RPL; ++r) {
                            acc[r] = __ffma2_rn(q2[r][2 * j], k01, acc[r]);
                            acc[r] = __ffma2_rn(q2[r][2 * j + 1], k23, acc[r]);
                        }
                    }
#pragma unroll
                    for (int r = 0; r < RPL; ++r) s[u][r] = acc[r].x + acc[r].y;
                }
#pragma unroll
                for (int u = 0; u < kKeyGroup; ++u)
#pragma unroll
                    for (int r = 0; r < RPL; ++r)
#pragma unroll
                        for (int o = RPW; o < 32; o <<= 1)
                            s[u][r] += __shfl_xor_sync(0xffffffffu, s[u][r], o);
                const int key0 = t0 + k0;
                const bool need_mask = !fullg || !set_valid ||
                                       (a.causal_block && key0 + kKeyGroup > S_cache);
                if (need_mask) {
#pragma unroll
                    for (int u = 0; u < kKeyGroup; ++u) {
                        bool ok = set_valid && u < nk;
                        const int key = key0 + u;
                        if (a.causal_block && key >= S_cache && key - S_cache > tok) ok = false;
                        if (!ok)
#pragma unroll
                            for (int r = 0; r < RPL; ++r) s[u][r] = -INFINITY;
                    }
                }
                float p[kKeyGroup][RPL];
                bool any = false;
#pragma unroll
                for (int r = 0; r < RPL; ++r) {
                    float mt = s[0][r];
#pragma unroll
                    for (int u = 1; u < kKeyGroup; ++u) mt = fmaxf(mt, s[u][r]);
                    const float mn = fmaxf(m[r], mt);
                    if (mn == -INFINITY) {
#pragma unroll
                        for (int u = 0; u < kKeyGroup; ++u) p[u][r] = 0.f;
                        continue;
                    }
                    any = true;
                    float ps = 0.f;
#pragma unroll
                    for (int u = 0; u < kKeyGroup; ++u) {
                        p[u][r] = fast_exp2(s[u][r] - mn);
                        ps += p[u][r];
                    }
                    if (mn != m[r]) {          // the running max moved: rescale what is summed so far
                        const float corr = fast_exp2(m[r] - mn);
                        l[r] *= corr;
                        const float2 c2 = make_float2(corr, corr);
#pragma unroll
                        for (int j = 0; j < DL / 2; ++j) o2[r][j] = __fmul2_rn(o2[r][j], c2);
                        m[r] = mn;
                    }
                    l[r] += ps;
                }
                if (!any) continue;
#pragma unroll
                for (int u = 0; u < kKeyGroup; ++u) {
                    const float *vr = vt + (size_t)(k0 + (fullg ? u : min(u, nk - 1))) * D;
                    float2 pu[RPL];
#pragma unroll
                    for (int r = 0; r < RPL; ++r) pu[r] = make_float2(p[u][r], p[u][r]);
#pragma unroll
                    for (int j = 0; j < DL / 4; ++j) {
                        const float4 vv = *reinterpret_cast<const float4 *>(vr + 4 * LPR * j);
                        const float2 v01 = make_float2(vv.x, vv.y), v23 = make_float2(vv.z, vv.w);
#pragma unroll
                        for (int r = 0; r < RPL; ++r) {
                            o2[r][2 * j] = __ffma2_rn(pu[r], v01, o2[r][2 * j]);
                            o2[r][2 * j + 1] = __ffma2_rn(pu[r], v23, o2[r][2 * j + 1]);
                        }
                    }
                }
            }
        }
        __syncthreads();
        if (tid == 0 && jt + kAttnStages < n_tiles) issue(jt + kAttnStages);
    }

    // ---- merge the key subsets of each row group (stage buffers are free now)
    const int rows_cta = RG * RPW * RPL;
    float *mo = tiles;                                  // [KS][rows_cta][D]
    float *mm = mo + (size_t)KS * rows_cta * D;         // [KS][rows_cta]
    float *ml = mm + KS * rows_cta;                     // [KS][rows_cta]
    if (active) {
#pragma unroll
        for (int r = 0; r < RPL; ++r) {
            const int rr = rs * RPL + r;
            float *dst = mo + ((size_t)ks * rows_cta + rr) * D + 4 * sub;
#pragma unroll
            for (int j = 0; j < DL / 4; ++j)
                *reinterpret_cast<float4 *>(dst + 4 * LPR * j) =
                    make_float4(o2[r][2 * j].x, o2[r][2 * j].y, o2[r][2 * j + 1].x, o2[r][2 * j + 1].y);
            if (sub == 0) {
                mm[ks * rows_cta + rr] = m[r];
                ml[ks * rows_cta + rr] = l[r];
            }
        }
    }
    __syncthreads();
    float *part = a.part + ((head_off * a.n_chunks + chunk) * (size_t)R) * (D + 2);
    for (int idx = tid; idx < R * D; idx += kAttnThreads) {
        const int r2 = idx / D, e = idx % D;
        float M = -INFINITY;
        for (int k2 = 0; k2 < KS; ++k2) M = fmaxf(M, mm[k2 * rows_cta + r2]);
        float O = 0.f, L = 0.f;
        if (M != -INFINITY) {
            for (int k2 = 0; k2 < KS; ++k2) {
                const float w = exp2f(mm[k2 * rows_cta + r2] - M);
                O = fmaf(w, mo[((size_t)k2 * rows_cta + r2) * D + e], O);
                L = fmaf(w, ml[k2 * rows_cta + r2], L);
            }
        }
        part[(size_t)r2 * (D + 2) + e] = O;
        if (e == 0) {
            part[(size_t)r2 * (D + 2) + D] = M;
            part[(size_t)r2 * (D + 2) + D + 1] = L;
        }
    }
}

// Merge of the chunk partials: one warp per (query row, 32-wide slice of the head dims). Lane c
// holds chunk c's merge weight 2^(m_c - M) / L (M, L over all chunks); the partial outputs of 32
// chunks are loaded at once per lane before any is summed, and the sum runs in chunk order (the
// result does not depend on timing).
template <int D>
__global__ void __launch_bounds__(256) attn_combine_kernel(AttnArgs a) {
    DF_TRACE_KERNEL(TK_ATTN_COMBINE);
    constexpr int SL = D / 32;               // slices per row
    pdl_trigger();
    pdl_wait();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = blockIdx.y, b = blockIdx.z;
    const int rep = a.nq / a.nkv;
    const int R = a.blk * rep;
    const int task = blockIdx.x * 8 + warp;
    if (task >= R * SL) return;
    const int r2 = task / SL, e = (task - r2 * SL) * 32 + lane;
    const size_t head_off = (size_t)b * a.nkv + g;
    const float *allp = a.part + head_off * a.n_chunks * (size_t)R * (D + 2);
    const int NC = a.n_chunks;
    float y = 0.f;
    if (NC <= 32) {
        // one round trip: every lane's (m, l) of chunk `lane` and the 32 partial outputs of its
        // dim are requested before any is used
        float mc = -INFINITY, lc = 0.f;
        if (lane < NC) {
            const float *pc = allp + ((size_t)lane * R + r2) * (D + 2);
            mc = pc[D];
            lc = pc[D + 1];
        }
        float ov[32];
#pragma unroll
        for (int j = 0; j < 32; ++j)
            ov[j] = j < NC ? allp[((size_t)j * R + r2) * (D + 2) + e] : 0.f;
        const float M = warp_max(mc);
        const float w = mc == -INFINITY ? 0.f : exp2f(mc - M);
        const float L = warp_sum(lc * w);
        const float wl = L > 0.f ? w / L : 0.f;
#pragma unroll
        for (int j = 0; j < 32; ++j) y = fmaf(__shfl_sync(0xffffffffu, wl, j), ov[j], y);
    } else {
        float M = -INFINITY;
        for (int c = lane; c < NC; c += 32) M = fmaxf(M, allp[((size_t)c * R + r2) * (D + 2) + D]);
        M = warp_max(M);
        float L = 0.f;
        for (int c = lane; c < NC; c += 32) {
            const float *pc = allp + ((size_t)c * R + r2) * (D + 2);
            const float mc = pc[D];
            if (mc != -INFINITY) L += pc[D + 1] * exp2f(mc - M);
        }
        L = warp_sum(L);
        const float invL = L > 0.f ? 1.f / L : 0.f;
        for (int c0 = 0; c0 < NC; c0 += 32) {
            float wl = 0.f;
            if (c0 + lane < NC) {
                const float mc = allp[((size_t)(c0 + lane) * R + r2) * (D + 2) + D];
                wl = mc == -INFINITY ? 0.f : exp2f(mc - M) * invL;
            }
            const int cn = min(32, NC - c0);
            float ov[32];
#pragma unroll
            for (int j = 0; j < 32; ++j)
                ov[j] = j < cn ? allp[((size_t)(c0 + j) * R + r2) * (D + 2) + e] : 0.f;
#pragma unroll
            for (int j = 0; j < 32; ++j) y = fmaf(__shfl_sync(0xffffffffu, wl, j), ov[j], y);
        }
    }
    const int i = r2 / rep, h = g * rep + r2 % rep;
    const size_t t = (size_t)b * a.blk + i;
    float v = y;
    if (a.gate) {
        const float z = a.gate[t * a.ldg + (size_t)h * D + e];
        v = v * (1.f / (1.f + expf(-z)));
    }
    const size_t col = (size_t)h * D + e;
    if (a.out) a.out[t * (size_t)(a.nq * D) + col] = v;
    if (a.pack) {
        uint16_t hi, lo;
        split_hi_lo(v, hi, lo);
        a.pack[(2 * t) * (size_t)(a.nq * D) + col] = hi;
        a.pack[(2 * t + 1) * (size_t)(a.nq * D) + col] = lo;
    }
}

__global__ void seq_advance_kernel(int32_t *seq_len, const int32_t *n_new, int B, int delta,
                                   int cap, int32_t *status) {
    DF_TRACE_KERNEL(TK_SEQ_ADVANCE);
    pdl_trigger();
    pdl_wait();
    int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= B) return;
    int add = n_new ? n_new[b] : delta;
    long long nv = (long long)seq_len[b] + add;
    if (add < 0 || nv > cap) {
        set_status(status, DF_ECAPACITY);
        nv = min(max(nv, 0LL), (long long)cap);
    }
    seq_len[b] = (int32_t)nv;
}

}  // namespace

int launch_rope_table(float *cos_t, float *sin_t, const int32_t *seq_len, const int32_t *n_new,
                      int n_new_max, int B, int blk, int pos_off, int rot, float theta,
                      int32_t *status, cudaStream_t s) {
    int total = B * (blk + n_new_max) * (rot / 2);
    if (total <= 0) return DF_OK;
    if (rot / 2 > kMaxRopeHalf) return fail(DF_ESHAPE, "rotary dim %d above %d", rot, 2 * kMaxRopeHalf);
    RopeArgs a;
    memset(&a, 0, sizeof(a));
    a.cos_t = cos_t;
    a.sin_t = sin_t;
    a.seq_len = seq_len;
    a.n_new = n_new;
    a.n_new_max = n_new_max;
    a.B = B;
    a.blk = blk;
    a.pos_off = pos_off;
    a.rot = rot;
    a.status = status;
    for (int j = 0; j < rot / 2; ++j) a.inv[j] = std::pow((double)theta, -2.0 * j / (double)rot);
    int threads = 256, grid = min((total + threads - 1) / threads, 4 * sm_count());
    return launch_k("rope_table_kernel", rope_table_kernel, dim3(grid), dim3(threads), 0, s, a);
}

int launch_qk_rope(const QkArgs &a, cudaStream_t s) {
    long long warps = (long long)(a.B * a.blk + a.B * a.n_new_max) * (a.nq + 2 * a.nkv + a.n_gate_heads);
    if (warps <= 0) return DF_OK;
    const int wpb = 8;
    long long grid = (warps + wpb - 1) / wpb;
    return launch_k("qk_rope_kernel", qk_rope_kernel, dim3((unsigned)grid), dim3(wpb * 32),
                    wpb * a.d * sizeof(float), s, a);
}

size_t attn_part_floats(const AttnArgs &a) {
    const int R = a.blk * (a.nq / a.nkv);
    return (size_t)a.B * a.nkv * a.n_chunks * R * (size_t)(a.d + 2);
}

// Keys per chunk: a whole number of tiles. Head dims 128 and 256 with up to 32 query rows per KV
// head run on the tensor cores (128-key tiles, one CTA per SM); everything else runs on the CUDA
// cores (about one CTA per SM, two waves when sequences x KV heads alone nearly fill the GPU).
// Tensor-core chunks: every CTA streams its chunk at about the same rate, so a launch lasts its
// number of waves times (tiles per chunk + a fixed cost of about one tile for the CTA's start,
// q operand and partial write-out); the plan takes the chunk length that minimises that product,
// the longer chunk on a tie (fewer partials to merge). A last wave of a few CTAs costs as much as
// a full one, which the plain one-CTA-per-SM rule ignores (8 sequences x 8 KV heads: 5 chunks
// are 320 CTAs, three waves on 152 SMs; 7 chunks fill the same three waves with shorter chunks).
void attn_plan(AttnArgs &a, int max_keys) {
    const int R = a.blk * (a.nq / a.nkv);
    const int heads = a.B * a.nkv;
    a.tc = attn_tc_supported(a.d, R) ? 1 : 0;
    const int TK = a.tc ? 128 : kTileBytes / (2 * a.d * 4);
    const int tiles = std::max(1, (max_keys + TK - 1) / TK);
    int per;
    if (a.tc) {
        constexpr long long kChunkFixedTiles = 1;
        const long long sms = sm_count();
        long long best = -1;
        per = tiles;
        for (int p = tiles; p >= 1; --p) {
            const long long nc = (tiles + p - 1) / p;
            const long long waves = (heads * nc + sms - 1) / sms;
            const long long cost = waves * (p + kChunkFixedTiles);
            if (best < 0 || cost < best) {
                best = cost;
                per = p;
            }
        }
    } else {
        const int waves = heads > 38 ? 2 : 1;
        const int want = std::max(1, (waves * sm_count() + heads - 1) / heads);
        const int n = std::min(want, tiles);
        per = (tiles + n - 1) / n;
    }
    a.chunk = per * TK;
    a.n_chunks = std::max(1, (max_keys + a.chunk - 1) / a.chunk);
}

template <int D, int RPL>
int launch_attn_d(const AttnArgs &a, cudaStream_t s) {
    const int R = a.blk * (a.nq / a.nkv);
    constexpr int RPW = 32 / (D / 32);
    constexpr int NW = kAttnThreads / 32;
    if ((R / RPL + RPW - 1) / RPW > NW)
        return fail(DF_ESHAPE, "attention: %d query rows per KV head exceed %d", R, NW * RPW * RPL);
    // stage buffers, reused at the end for the key-subset merge (KS * rows_cta <= NW*RPW*RPL rows)
    size_t smem = (size_t)kAttnStages * kTileBytes + kAttnStages * 8 + 16;
    size_t need_merge = sizeof(float) * ((size_t)NW * RPW * RPL * (D + 2));
    if (need_merge > (size_t)kAttnStages * kTileBytes)
        return fail(DF_ESHAPE, "attention: merge buffer exceeds the stage buffers");
    dim3 grid(a.n_chunks, a.nkv, a.B);
    if (a.kv_bf16 && !a.tc)
        return fail(DF_ESHAPE, "a BF16 KV cache needs head_dim 128 or 256 and at most 32 query "
                               "rows per KV head (the tensor-core attention)");
    if (a.tc) DF_TRY(launch_attn_tc(a, s));
    else DF_TRY(launch_k("attn_kernel", attn_kernel<D, RPL>, grid, dim3(kAttnThreads), smem, s, a));
    dim3 cgrid((R * (D / 32) + 7) / 8, a.nkv, a.B);
    return launch_k("attn_combine_kernel", attn_combine_kernel<D>, cgrid, dim3(256), 0, s, a);
}

template <int D>
int launch_attn_r(const AttnArgs &a, cudaStream_t s) {
    if ((a.nq / a.nkv) % 2 == 0) return launch_attn_d<D, 2>(a, s);
    return launch_attn_d<D, 1>(a, s);
}

int launch_attn(const AttnArgs &a, cudaStream_t s) {
    switch (a.d) {
        case 32: return launch_attn_r<32>(a, s);
        case 64: return launch_attn_r<64>(a, s);
        case 128: return launch_attn_r<128>(a, s);
        case 256: return launch_attn_r<256>(a, s);
        default: return fail(DF_ESHAPE, "attention: head_dim %d not in {32, 64, 128, 256}", a.d);
    }
}

int launch_seq_advance(int32_t *seq_len, const int32_t *n_new, int B, int delta, int cap,
                       int32_t *status, cudaStream_t s) {
    return launch_k("seq_advance_kernel", seq_advance_kernel, dim3((B + 127) / 128), dim3(128), 0, s,
                    seq_len, n_new, B, delta, cap, status);
}

}  // namespace df

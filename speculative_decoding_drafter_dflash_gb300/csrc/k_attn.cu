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

#include "df_internal.cuh"

namespace df {

namespace {

// cos/sin of pos * theta^(-2j/rot) in double precision, rounded to F32.
__global__ void rope_table_kernel(float *cos_t, float *sin_t, const int32_t *seq_len,
                                  const int32_t *n_new, int n_new_max, int B, int blk, int pos_off,
                                  int rot, float theta, int32_t *status) {
    const int half = rot / 2;
    const int slots = blk + n_new_max;
    const int total = B * slots * half;
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < total; i += gridDim.x * blockDim.x) {
        int j = i % half;
        int s = (i / half) % slots;
        int b = i / (half * slots);
        int base = seq_len[b];
        int nn = n_new ? min(max(n_new[b], 0), n_new_max) : 0;
        if (status && j == 0 && s == 0 && n_new && (n_new[b] < 0 || n_new[b] > n_new_max))
            set_status(status, DF_ESHAPE);
        long long pos = s < blk ? (long long)base + nn + s + pos_off : (long long)base + (s - blk);
        double inv = pow((double)theta, -2.0 * (double)j / (double)rot);
        double sn, cs;
        sincos((double)pos * inv, &sn, &cs);
        cos_t[i] = (float)cs;
        sin_t[i] = (float)sn;
    }
}

// One warp per (token row, head slot). Slots: [0, nq) q heads, [nq, nq+nkv) k heads,
// [nq+nkv, nq+2nkv) v heads. Rows [0, B*blk) are block rows, the rest context rows.
__global__ void qk_rope_kernel(QkArgs a) {
    extern __shared__ float smem[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int wpb = blockDim.x >> 5;
    const int slots = a.nq + 2 * a.nkv;
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
        if (slot < a.nq) return;                        // context rows feed only K/V
        int nn = min(max(a.n_new[b], 0), a.n_new_max);
        if (i >= nn) return;
    }
    const bool is_q = slot < a.nq;
    const bool is_k = !is_q && slot < a.nq + a.nkv;
    const int head = is_q ? slot : (is_k ? slot - a.nq : slot - a.nq - a.nkv);
    const int col = is_q ? head * d : (is_k ? a.nq * d + head * d : (a.nq + a.nkv) * d + head * d);
    const float *src = a.qkv + (size_t)row * a.ldq + col;

    float x[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) x[u] = (u < ept) ? src[lane + 32 * u] : 0.f;

    if (!(slot >= a.nq + a.nkv)) {   // q or k: per-head RMSNorm, then RoPE
        const float *nw = is_q ? a.q_norm : a.k_norm;
        if (nw) {
            float ss = 0.f;
#pragma unroll
            for (int u = 0; u < 8; ++u) ss = fmaf(x[u], x[u], ss);
            ss = warp_sum(ss);
            float inv = 1.f / sqrtf(ss / (float)d + a.eps);
#pragma unroll
            for (int u = 0; u < 8; ++u)
                if (u < ept) x[u] = x[u] * inv * nw[lane + 32 * u];
        }
#pragma unroll
        for (int u = 0; u < 8; ++u)
            if (u < ept) buf[lane + 32 * u] = x[u];
        __syncwarp();
        const int tslot = is_block ? i : a.blk + i;
        const float *ct = a.cos_t + ((size_t)b * (a.blk + a.n_new_max) + tslot) * half;
        const float *st = a.sin_t + ((size_t)b * (a.blk + a.n_new_max) + tslot) * half;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            int e = lane + 32 * u;
            if (u < ept && e < a.rot) {
                if (e < half) x[u] = buf[e] * ct[e] - buf[e + half] * st[e];
                else x[u] = buf[e] * ct[e - half] + buf[e - half] * st[e - half];
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
#pragma unroll
    for (int u = 0; u < 8; ++u)
        if (u < ept) dst[lane + 32 * u] = x[u];
}

constexpr int kAttnThreads = 256;
constexpr int kKeyTile = 32;
constexpr int kMaxOut = 16;      // outputs per thread: rows_per_group * d <= 256 * 16

// Split-KV partial attention. Grid (n_chunks, nkv * n_groups, B). Key index space of a
// sequence: cache rows [0, S_cache) then block keys [S_cache, S_cache + blk).
__global__ void __launch_bounds__(kAttnThreads) attn_partial_kernel(AttnArgs a) {
    extern __shared__ float sm[];
    const int d = a.d, dp = d + 4;
    const int R = a.rows_per_group;
    const int rep = a.nq / a.nkv;
    const int chunk = blockIdx.x;
    const int g = blockIdx.y / a.n_groups, grp = blockIdx.y % a.n_groups;
    const int b = blockIdx.z;
    const int rows_total = a.blk * rep;
    const int r0 = grp * R;
    const int nr = min(R, rows_total - r0);

    float *q_s = sm;                        // [R][dp]
    float *k_s = q_s + R * dp;              // [kKeyTile][dp]
    float *v_s = k_s + kKeyTile * dp;       // [kKeyTile][dp]
    float *p_s = v_s + kKeyTile * dp;       // [R][kKeyTile + 1]
    float *m_s = p_s + R * (kKeyTile + 1);  // [R]
    float *l_s = m_s + R;                   // [R]
    float *c_s = l_s + R;                   // [R]

    int nn = a.n_new ? min(max(a.n_new[b], 0), a.n_new_max) : 0;
    long long sc = (long long)a.seq_len[b] + nn + a.extra_rows;
    const int S_cache = (int)min(max(sc, 0LL), (long long)a.cap);
    const int S = S_cache + (a.kb ? a.blk : 0);
    const int k_begin = chunk * a.chunk;
    const int k_end = min(S, k_begin + a.chunk);

    // query rows of this group: row r -> block token i = r / rep, q head g*rep + r % rep
    for (int idx = threadIdx.x; idx < nr * d; idx += blockDim.x) {
        int r = idx / d, e = idx % d;
        int rr = r0 + r;
        int i = rr / rep, h = g * rep + rr % rep;
        q_s[r * dp + e] = a.q[(((size_t)b * a.blk + i) * a.nq + h) * d + e];
    }
    for (int r = threadIdx.x; r < R; r += blockDim.x) {
        m_s[r] = -INFINITY;
        l_s[r] = 0.f;
    }
    float o[kMaxOut];
#pragma unroll
    for (int u = 0; u < kMaxOut; ++u) o[u] = 0.f;
    const float scale = 1.f / sqrtf((float)d);
    __syncthreads();

    for (int kt = k_begin; kt < k_end; kt += kKeyTile) {
        const int nk = min(kKeyTile, k_end - kt);
        for (int idx = threadIdx.x; idx < kKeyTile * (d / 4); idx += blockDim.x) {
            int kk = idx / (d / 4), e4 = (idx % (d / 4)) * 4;
            float4 kv = make_float4(0.f, 0.f, 0.f, 0.f), vv = kv;
            if (kk < nk) {
                int s = kt + kk;
                const float *kp, *vp;
                if (s < S_cache) {
                    size_t off = (((size_t)b * a.nkv + g) * a.cap + s) * d + e4;
                    kp = a.cache_k + off;
                    vp = a.cache_v + off;
                } else {
                    size_t off = (((size_t)b * a.nkv + g) * a.blk + (s - S_cache)) * d + e4;
                    kp = a.kb + off;
                    vp = a.vb + off;
                }
                kv = *reinterpret_cast<const float4 *>(kp);
                vv = *reinterpret_cast<const float4 *>(vp);
            }
            *reinterpret_cast<float4 *>(k_s + kk * dp + e4) = kv;
            *reinterpret_cast<float4 *>(v_s + kk * dp + e4) = vv;
        }
        __syncthreads();
        // scores
        for (int idx = threadIdx.x; idx < nr * kKeyTile; idx += blockDim.x) {
            int r = idx / kKeyTile, kk = idx % kKeyTile;
            float sc2 = -INFINITY;
            if (kk < nk) {
                const float *qr = q_s + r * dp;
                const float *kr = k_s + kk * dp;
                float acc = 0.f;
                for (int e = 0; e < d; e += 4) {
                    float4 qa = *reinterpret_cast<const float4 *>(qr + e);
                    float4 ka = *reinterpret_cast<const float4 *>(kr + e);
                    acc = fmaf(qa.x, ka.x, acc);
                    acc = fmaf(qa.y, ka.y, acc);
                    acc = fmaf(qa.z, ka.z, acc);
                    acc = fmaf(qa.w, ka.w, acc);
                }
                sc2 = acc * scale;
                int s = kt + kk;
                if (a.causal_block && s >= S_cache) {
                    int i = (r0 + r) / rep;
                    if (s - S_cache > i) sc2 = -INFINITY;
                }
            }
            p_s[r * (kKeyTile + 1) + kk] = sc2;
        }
        __syncthreads();
        // online softmax update, one thread per row
        for (int r = threadIdx.x; r < nr; r += blockDim.x) {
            float mo = m_s[r];
            float mx = mo;
            for (int kk = 0; kk < kKeyTile; ++kk) mx = fmaxf(mx, p_s[r * (kKeyTile + 1) + kk]);
            float corr = 1.f, sum = 0.f;
            if (mx == -INFINITY) {
                for (int kk = 0; kk < kKeyTile; ++kk) p_s[r * (kKeyTile + 1) + kk] = 0.f;
            } else {
                corr = (mo == -INFINITY) ? 0.f : expf(mo - mx);
                for (int kk = 0; kk < kKeyTile; ++kk) {
                    float v = p_s[r * (kKeyTile + 1) + kk];
                    float p = (v == -INFINITY) ? 0.f : expf(v - mx);
                    p_s[r * (kKeyTile + 1) + kk] = p;
                    sum += p;
                }
            }
            m_s[r] = mx;
            l_s[r] = l_s[r] * corr + sum;
            c_s[r] = corr;
        }
        __syncthreads();
        // o = o * corr + P V
#pragma unroll
        for (int u = 0; u < kMaxOut; ++u) {
            int idx = threadIdx.x + u * blockDim.x;
            if (idx < nr * d) {
                int r = idx / d, e = idx % d;
                float acc = o[u] * c_s[r];
                const float *pr = p_s + r * (kKeyTile + 1);
                for (int kk = 0; kk < nk; ++kk) acc = fmaf(pr[kk], v_s[kk * dp + e], acc);
                o[u] = acc;
            }
        }
        __syncthreads();
    }
    // write partials
    const size_t pbase = ((((size_t)b * a.nkv + g) * a.n_groups + grp) * a.n_chunks + chunk) * R;
#pragma unroll
    for (int u = 0; u < kMaxOut; ++u) {
        int idx = threadIdx.x + u * blockDim.x;
        if (idx < nr * d) {
            int r = idx / d, e = idx % d;
            a.part_o[(pbase + r) * d + e] = o[u];
        }
    }
    for (int r = threadIdx.x; r < nr; r += blockDim.x) {
        a.part_ml[(pbase + r) * 2 + 0] = m_s[r];
        a.part_ml[(pbase + r) * 2 + 1] = l_s[r];
    }
}

// One warp per (sequence, block token, q head): merge the chunk partials, apply the optional
// sigmoid gate, pack hi/lo BF16 for the O projection.
__global__ void attn_combine_kernel(AttnArgs a) {
    const int lane = threadIdx.x & 31;
    const long long gw = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int rep = a.nq / a.nkv;
    const long long total = (long long)a.B * a.blk * a.nq;
    if (gw >= total) return;
    const int h = (int)(gw % a.nq);
    const int i = (int)((gw / a.nq) % a.blk);
    const int b = (int)(gw / ((long long)a.nq * a.blk));
    const int g = h / rep;
    const int rr = i * rep + (h % rep);
    const int grp = rr / a.rows_per_group, r = rr % a.rows_per_group;
    const int d = a.d, ept = d / 32;
    const size_t cbase = (((size_t)b * a.nkv + g) * a.n_groups + grp) * a.n_chunks;

    float M = -INFINITY;
    for (int c = lane; c < a.n_chunks; c += 32)
        M = fmaxf(M, a.part_ml[((cbase + c) * a.rows_per_group + r) * 2]);
    M = warp_max(M);
    float L = 0.f;
    for (int c = lane; c < a.n_chunks; c += 32) {
        float m = a.part_ml[((cbase + c) * a.rows_per_group + r) * 2];
        float l = a.part_ml[((cbase + c) * a.rows_per_group + r) * 2 + 1];
        if (m != -INFINITY) L += l * expf(m - M);
    }
    L = warp_sum(L);
    float acc[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) acc[u] = 0.f;
    for (int c = 0; c < a.n_chunks; ++c) {
        float m = a.part_ml[((cbase + c) * a.rows_per_group + r) * 2];
        if (m == -INFINITY) continue;
        float f = expf(m - M);
        const float *po = a.part_o + ((cbase + c) * a.rows_per_group + r) * d;
#pragma unroll
        for (int u = 0; u < 8; ++u)
            if (u < ept) acc[u] = fmaf(f, po[lane + 32 * u], acc[u]);
    }
    const float invL = L > 0.f ? 1.f / L : 0.f;
    const size_t t = (size_t)b * a.blk + i;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
        if (u < ept) {
            int e = lane + 32 * u;
            float y = acc[u] * invL;
            if (a.gate) {
                float z = a.gate[t * a.ldg + h * d + e];
                y = y * (1.f / (1.f + expf(-z)));
            }
            uint16_t hi, lo;
            split_hi_lo(y, hi, lo);
            size_t col = (size_t)h * d + e;
            a.pack[(2 * t) * (size_t)(a.nq * d) + col] = hi;
            a.pack[(2 * t + 1) * (size_t)(a.nq * d) + col] = lo;
        }
    }
}

__global__ void seq_advance_kernel(int32_t *seq_len, const int32_t *n_new, int B, int delta,
                                   int cap, int32_t *status) {
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
    int threads = 256, grid = min((total + threads - 1) / threads, 4 * kNumSMs);
    rope_table_kernel<<<grid, threads, 0, s>>>(cos_t, sin_t, seq_len, n_new, n_new_max, B, blk,
                                                pos_off, rot, theta, status);
    return cuda_check("rope_table_kernel");
}

int launch_qk_rope(const QkArgs &a, cudaStream_t s) {
    long long warps = (long long)(a.B * a.blk + a.B * a.n_new_max) * (a.nq + 2 * a.nkv);
    if (warps <= 0) return DF_OK;
    const int wpb = 8;
    long long grid = (warps + wpb - 1) / wpb;
    qk_rope_kernel<<<(unsigned)grid, wpb * 32, wpb * a.d * sizeof(float), s>>>(a);
    return cuda_check("qk_rope_kernel");
}

size_t attn_part_floats(int B, int nkv, int n_groups, int n_chunks, int rows_per_group, int d) {
    return (size_t)B * nkv * n_groups * n_chunks * rows_per_group * (size_t)(d + 2);
}

// Rows per CTA group bounded by the per-thread output registers; chunk count aims at about
// two CTAs per SM for the largest possible key count.
void attn_plan(AttnArgs &a, int max_keys) {
    const int rep = a.nq / a.nkv;
    const int rows_total = a.blk * rep;
    const int max_rows = (kAttnThreads * kMaxOut) / a.d;
    a.n_groups = (rows_total + max_rows - 1) / max_rows;
    a.rows_per_group = (rows_total + a.n_groups - 1) / a.n_groups;
    int ctas_per_chunk = a.B * a.nkv * a.n_groups;
    int want = max(1, (2 * kNumSMs + ctas_per_chunk - 1) / ctas_per_chunk);
    int max_chunks = max(1, (max_keys + kKeyTile - 1) / kKeyTile);
    int n = min(want, max_chunks);
    int chunk = (max_keys + n - 1) / n;
    chunk = ((chunk + kKeyTile - 1) / kKeyTile) * kKeyTile;
    a.chunk = max(chunk, kKeyTile);
    a.n_chunks = max(1, (max_keys + a.chunk - 1) / a.chunk);
}

int launch_attn(const AttnArgs &a, cudaStream_t s) {
    const int dp = a.d + 4, R = a.rows_per_group;
    size_t smem = sizeof(float) * ((size_t)R * dp + 2 * kKeyTile * dp + R * (kKeyTile + 1) + 3 * R);
    if (smem > 48 * 1024) {
        int dev = 0;
        cudaGetDevice(&dev);
        static bool attr_set[64] = {};
        if (dev < 0 || dev >= 64 || !attr_set[dev]) {
            cudaFuncSetAttribute(attn_partial_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 200 * 1024);
            if (dev >= 0 && dev < 64) attr_set[dev] = true;
        }
    }
    dim3 grid(a.n_chunks, a.nkv * a.n_groups, a.B);
    attn_partial_kernel<<<grid, kAttnThreads, smem, s>>>(a);
    DF_TRY(cuda_check("attn_partial_kernel"));
    long long warps = (long long)a.B * a.blk * a.nq;
    attn_combine_kernel<<<(unsigned)((warps + 7) / 8), 256, 0, s>>>(a);
    return cuda_check("attn_combine_kernel");
}

int launch_seq_advance(int32_t *seq_len, const int32_t *n_new, int B, int delta, int cap,
                       int32_t *status, cudaStream_t s) {
    seq_advance_kernel<<<(B + 127) / 128, 128, 0, s>>>(seq_len, n_new, B, delta, cap, status);
    return cuda_check("seq_advance_kernel");
}

}  // namespace df

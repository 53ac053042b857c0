// Row prologue kernels: embedding gather, RMSNorm and the hi/lo BF16 packing that every
// projection consumes.
//
// RMSNorm follows hf2q 0.1.1 models/qwen35/mtp.rs `rms_norm_with_weight`
// (y = x * 1/sqrt(mean(x^2) + eps) * w, F32 weight); the embedding gather is
// qwen35_orchestrator.rs step 1 (`embed_tokens_gpu` of [last_token, mask x K]).
#include <cooperative_groups.h>

#include "df_internal.cuh"

namespace cg = cooperative_groups;

namespace df {

namespace {

constexpr int kPackThreads = 256;

// The capacity-checked length advance a pack launch may carry (CTA 0, after the wait).
__device__ __forceinline__ void pack_side_advance(const PackArgs &a) {
    if (!a.adv_seq || blockIdx.x != 0) return;
    for (int b = threadIdx.x; b < a.adv_B; b += blockDim.x) {
        const int add = a.adv_n ? a.adv_n[b] : 0;
        long long nv = (long long)a.adv_seq[b] + add;
        if (add < 0 || nv > a.adv_cap) {
            set_status(a.status, DF_ECAPACITY);
            nv = min(max(nv, 0LL), (long long)a.adv_cap);
        }
        a.adv_seq[b] = (int32_t)nv;
    }
}

__device__ __forceinline__ float block_sum(float v, float *red) {
    v = warp_sum(v);
    int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    if (l == 0) red[w] = v;
    __syncthreads();
    float t = 0.f;
    if (threadIdx.x < 32) {
        t = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0.f;
        t = warp_sum(t);
        if (threadIdx.x == 0) red[32] = t;
    }
    __syncthreads();
    float r = red[32];
    __syncthreads();
    return r;
}

// One CTA per row t. Reads the row (from src or the embedding table), optionally stores it
// raw (h_out), computes rmsnorm(row) * w when a weight is given (else the row itself),
// optionally stores that (y_out), and packs it into two BF16 rows (hi, lo).
__global__ void __launch_bounds__(kPackThreads) pack_kernel(PackArgs a) {
    DF_TRACE_KERNEL(TK_PACK);
    __shared__ float red[33];
    pdl_trigger();
    pdl_wait();
    pack_side_advance(a);
    const int t = blockIdx.x;
    const int K = a.K;
    const int s = t / a.rows_per_seq, j = t - s * a.rows_per_seq;
    const bool valid = a.nvalid == nullptr || j < min(max(a.nvalid[s], 0), a.rows_per_seq);

    int id = -1;
    if (a.gather) {
        id = a.ids ? a.ids[t] : (j == 0 ? a.last_token[s] : a.mask_id);
        if (id < 0 || id >= a.vocab) {
            if (threadIdx.x == 0) set_status(a.status, DF_EINVAL);
            id = min(max(id, 0), a.vocab - 1);
        }
    }
    auto load = [&](int k) -> float {
        if (!valid) return 0.f;
        if (a.gather) return bf16_bits_to_f32(a.gather[(size_t)id * K + k]) * a.scale;
        float x = a.src ? a.src[(size_t)t * a.lds + k] : 0.f;
        for (int sp = 0; sp < a.n_part; ++sp) x += a.part[sp * a.part_stride + (size_t)t * a.ldpart + k];
        return x;
    };

    float inv = 1.f;
    if (a.norm_w) {
        float ss = 0.f;
        for (int k = threadIdx.x; k < K; k += blockDim.x) {
            float x = load(k);
            ss = fmaf(x, x, ss);
        }
        ss = block_sum(ss, red);
        inv = 1.f / sqrtf(ss / (float)K + a.eps);
    }
    for (int k = threadIdx.x; k < K; k += blockDim.x) {
        float x = load(k);
        if (a.h_out) a.h_out[(size_t)t * a.ldh + k] = x;
        float y = a.norm_w ? x * inv * a.norm_w[k] : x;
        if (a.y_out) a.y_out[(size_t)t * a.ldy + k] = y;
        if (a.pack) {
            uint16_t hi, lo;
            split_hi_lo(y, hi, lo);
            a.pack[(size_t)(2 * t) * a.ldp + k] = hi;
            a.pack[(size_t)(2 * t + 1) * a.ldp + k] = lo;
        }
    }
}

// Register-resident variant: a row is split over a cluster of `cl` CTAs (consecutive blockIdx.x),
// each holding at most 256 * 4 * NV of its elements in registers. Every element and every
// split partial is loaded once with 128-bit loads, all issued before any is used; the RMSNorm
// sum of squares is reduced in the CTA and then across the cluster through distributed shared
// memory, in rank order, so every CTA of a row applies the same factor.
template <int NV>
__global__ void __launch_bounds__(kPackThreads) pack_vec_kernel(PackArgs a, int cl) {
    DF_TRACE_KERNEL(TK_PACK_VEC);
    constexpr int G = NV <= 2 ? 8 : 4;   // split partials loaded per round
    __shared__ float red[33];
    pdl_trigger();
    pdl_wait();
    pack_side_advance(a);
    const int t = blockIdx.x / cl, rank = blockIdx.x - t * cl;
    const int K = a.K, K4 = K >> 2, per4 = K4 / cl, base4 = rank * per4;
    const int s = t / a.rows_per_seq, j = t - s * a.rows_per_seq;
    const bool valid = a.nvalid == nullptr || j < min(max(a.nvalid[s], 0), a.rows_per_seq);
    int id = 0;
    if (a.gather) {
        id = a.ids ? a.ids[t] : (j == 0 ? a.last_token[s] : a.mask_id);
        if (id < 0 || id >= a.vocab) {
            if (threadIdx.x == 0 && rank == 0) set_status(a.status, DF_EINVAL);
            id = min(max(id, 0), a.vocab - 1);
        }
    }
    float4 x[NV];
#pragma unroll
    for (int u = 0; u < NV; ++u) {
        const int i4 = threadIdx.x + u * kPackThreads, k4 = base4 + i4;
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (valid && i4 < per4) {
            if (a.gather) {
                const uint2 g = *reinterpret_cast<const uint2 *>(a.gather + (size_t)id * K + 4 * k4);
                v = make_float4(__uint_as_float(g.x << 16) * a.scale,
                                __uint_as_float(g.x & 0xffff0000u) * a.scale,
                                __uint_as_float(g.y << 16) * a.scale,
                                __uint_as_float(g.y & 0xffff0000u) * a.scale);
            } else if (a.src) {
                v = *reinterpret_cast<const float4 *>(a.src + (size_t)t * a.lds + 4 * k4);
            }
        }
        x[u] = v;
    }
    if (a.part && valid) {
        // every split's values of a round are loaded before any is added; the sum runs in
        // split order
        for (int sp0 = 0; sp0 < a.n_part; sp0 += G) {
            float4 pv[G][NV];
#pragma unroll
            for (int jj = 0; jj < G; ++jj)
#pragma unroll
                for (int u = 0; u < NV; ++u) {
                    const int i4 = threadIdx.x + u * kPackThreads;
                    pv[jj][u] = (sp0 + jj < a.n_part && i4 < per4)
                                    ? *reinterpret_cast<const float4 *>(
                                          a.part + (size_t)(sp0 + jj) * a.part_stride +
                                          (size_t)t * a.ldpart + 4 * (base4 + i4))
                                    : make_float4(0.f, 0.f, 0.f, 0.f);
                }
#pragma unroll
            for (int jj = 0; jj < G; ++jj)
#pragma unroll
                for (int u = 0; u < NV; ++u) {
                    x[u].x += pv[jj][u].x;
                    x[u].y += pv[jj][u].y;
                    x[u].z += pv[jj][u].z;
                    x[u].w += pv[jj][u].w;
                }
        }
    }
    float inv = 1.f;
    if (a.norm_w && a.ss_out) {
        // deferred norm: this slice's sum of squares, warps in order; no cluster exchange
        float ss = 0.f;
#pragma unroll
        for (int u = 0; u < NV; ++u)
            ss = fmaf(x[u].x, x[u].x, fmaf(x[u].y, x[u].y, fmaf(x[u].z, x[u].z, fmaf(x[u].w, x[u].w, ss))));
        ss = warp_sum(ss);
        const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
        if (l == 0) red[w] = ss;
        __syncthreads();
        if (threadIdx.x == 0) {
            float tot = 0.f;
            for (int i = 0; i < kPackThreads / 32; ++i) tot += red[i];
            const int ld = a.ss_ld > 0 ? a.ss_ld : cl;
            a.ss_out[(size_t)t * ld + rank] = tot;
            if (rank == 0)
                for (int j = cl; j < ld; ++j) a.ss_out[(size_t)t * ld + j] = 0.f;
        }
    } else if (a.norm_w) {
        float ss = 0.f;
#pragma unroll
        for (int u = 0; u < NV; ++u)
            ss = fmaf(x[u].x, x[u].x, fmaf(x[u].y, x[u].y, fmaf(x[u].z, x[u].z, fmaf(x[u].w, x[u].w, ss))));
        ss = warp_sum(ss);
        const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
        if (l == 0) red[w] = ss;
        __syncthreads();
        if (threadIdx.x == 0) {
            float tot = 0.f;
            for (int i = 0; i < kPackThreads / 32; ++i) tot += red[i];
            red[32] = tot;
        }
        if (cl > 1) {
            cg::cluster_group cluster = cg::this_cluster();
            cluster.sync();
            float tot = 0.f;
            for (int r = 0; r < cl; ++r) tot += *cluster.map_shared_rank(&red[32], r);
            ss = tot;
        } else {
            __syncthreads();
            ss = red[32];
        }
        inv = 1.f / sqrtf(ss / (float)K + a.eps);
    }
#pragma unroll
    for (int u = 0; u < NV; ++u) {
        const int i4 = threadIdx.x + u * kPackThreads;
        if (i4 >= per4) continue;
        const int k = 4 * (base4 + i4);
        float4 v = x[u];
        if (a.h_out) *reinterpret_cast<float4 *>(a.h_out + (size_t)t * a.ldh + k) = v;
        if (a.norm_w) {
            const float4 w = *reinterpret_cast<const float4 *>(a.norm_w + k);
            v = make_float4(v.x * inv * w.x, v.y * inv * w.y, v.z * inv * w.z, v.w * inv * w.w);
        }
        if (a.y_out) *reinterpret_cast<float4 *>(a.y_out + (size_t)t * a.ldy + k) = v;
        if (a.pack) {
            uint16_t h0, l0, h1, l1, h2, l2, h3, l3;
            split_hi_lo(v.x, h0, l0);
            split_hi_lo(v.y, h1, l1);
            split_hi_lo(v.z, h2, l2);
            split_hi_lo(v.w, h3, l3);
            *reinterpret_cast<uint2 *>(a.pack + (size_t)(2 * t) * a.ldp + k) =
                make_uint2(h0 | ((uint32_t)h1 << 16), h2 | ((uint32_t)h3 << 16));
            *reinterpret_cast<uint2 *>(a.pack + (size_t)(2 * t + 1) * a.ldp + k) =
                make_uint2(l0 | ((uint32_t)l1 << 16), l2 | ((uint32_t)l3 << 16));
        }
    }
    // peers may still be reading red[32] through distributed shared memory
    if (a.norm_w && !a.ss_out && cl > 1) cg::this_cluster().sync();
}

bool aligned_for_vec(const PackArgs &a) {
    auto al = [](const void *p, int bytes) { return (reinterpret_cast<uintptr_t>(p) % bytes) == 0; };
    if (a.K % 4) return false;
    if (a.src && (!al(a.src, 16) || a.lds % 4)) return false;
    if (a.part && (!al(a.part, 16) || a.ldpart % 4 || a.part_stride % 4)) return false;
    if (a.gather && !al(a.gather, 8)) return false;
    if (a.h_out && (!al(a.h_out, 16) || a.ldh % 4)) return false;
    if (a.norm_w && !al(a.norm_w, 16)) return false;
    if (a.y_out && (!al(a.y_out, 16) || a.ldy % 4)) return false;
    if (a.pack && (!al(a.pack, 8) || a.ldp % 4)) return false;
    return true;
}

}  // namespace

int pack_slices(int K) {
    // Up to 8 CTAs per row, keeping at least 64 4-element groups per CTA.
    const int K4 = K / 4;
    int cl = 8;
    while (cl > 1 && (K4 % cl != 0 || K4 / cl < 64)) cl >>= 1;
    return cl;
}

int launch_pack(const PackArgs &a, cudaStream_t s) {
    if (a.T <= 0) return DF_OK;
    if (a.ss_out && (!a.norm_w || !a.pack || a.y_out || !aligned_for_vec(a) ||
                     (a.K / 4) / pack_slices(a.K) > 16 * kPackThreads ||
                     (a.ss_ld > 0 && a.ss_ld < pack_slices(a.K))))
        return fail(DF_EINVAL, "deferred-norm row prologue: needs norm_w and pack, no y_out, "
                               "16-byte aligned rows");
    if (aligned_for_vec(a)) {
        // Split each row over up to 8 CTAs (a cluster, when the slices exchange their sums of
        // squares; independent CTAs when the norm is deferred to the consumer).
        const int K4 = a.K / 4;
        const int cl = pack_slices(a.K);
        const int nv = (K4 / cl + kPackThreads - 1) / kPackThreads;
        const dim3 g(a.T * cl), b(kPackThreads);
        if (nv <= 16) {
            if (cl > 1 && !a.ss_out) {
                if (nv <= 1) return launch_kc("pack_kernel", pack_vec_kernel<1>, g, b, 0, cl, s, a, cl);
                if (nv <= 2) return launch_kc("pack_kernel", pack_vec_kernel<2>, g, b, 0, cl, s, a, cl);
                if (nv <= 4) return launch_kc("pack_kernel", pack_vec_kernel<4>, g, b, 0, cl, s, a, cl);
                if (nv <= 8) return launch_kc("pack_kernel", pack_vec_kernel<8>, g, b, 0, cl, s, a, cl);
                return launch_kc("pack_kernel", pack_vec_kernel<16>, g, b, 0, cl, s, a, cl);
            }
            if (nv <= 1) return launch_k("pack_kernel", pack_vec_kernel<1>, g, b, 0, s, a, cl);
            if (nv <= 2) return launch_k("pack_kernel", pack_vec_kernel<2>, g, b, 0, s, a, cl);
            if (nv <= 4) return launch_k("pack_kernel", pack_vec_kernel<4>, g, b, 0, s, a, cl);
            if (nv <= 8) return launch_k("pack_kernel", pack_vec_kernel<8>, g, b, 0, s, a, cl);
            return launch_k("pack_kernel", pack_vec_kernel<16>, g, b, 0, s, a, cl);
        }
    }
    return launch_k("pack_kernel", pack_kernel, dim3(a.T), dim3(kPackThreads), 0, s, a);
}

}  // namespace df

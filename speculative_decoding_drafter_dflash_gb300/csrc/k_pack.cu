// Row prologue kernels: embedding gather, RMSNorm and the hi/lo BF16 packing that every
// projection consumes.
//
// RMSNorm follows hf2q 0.1.1 models/qwen35/mtp.rs `rms_norm_with_weight`
// (y = x * 1/sqrt(mean(x^2) + eps) * w, F32 weight); the embedding gather is
// qwen35_orchestrator.rs step 1 (`embed_tokens_gpu` of [last_token, mask x K]).
#include "df_internal.cuh"

namespace df {

namespace {

constexpr int kPackThreads = 256;

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
    __shared__ float red[33];
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
        return a.src[(size_t)t * a.lds + k];
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

}  // namespace

int launch_pack(const PackArgs &a, cudaStream_t s) {
    if (a.T <= 0) return DF_OK;
    prof_begin(s);
    pack_kernel<<<a.T, kPackThreads, 0, s>>>(a);
    return cuda_check("pack_kernel", s);
}

}  // namespace df

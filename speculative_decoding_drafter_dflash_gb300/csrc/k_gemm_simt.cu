// Skinny projection y[t, n] = sum_k x[t, k] * W[n, k] on CUDA cores: BF16 weights streamed
// with 128-bit loads, F32 activations (hi + lo of the packed BF16 pair, exact in F32), F32
// accumulation, and the fused epilogues of the draft round (store, residual add, SwiGLU with
// re-packing, running argmax of lm_head rows).
//
// Projections: tensors.rs (hf2q 0.1.1) `DFlashLayerTensors` (row-major [out, in] BF16
// weights, BF16-weight x F32-activation matmuls); mtp.rs `apply_linear_projection_f32`.
#include "df_internal.cuh"

namespace df {

namespace {

constexpr int kWarps = 8;

// After the call lane L holds, in v[0], the warp-wide sum of entry (L >> (5 - log2 TT)).
template <int TT>
__device__ __forceinline__ void reduce_scatter(float (&v)[TT], int lane) {
    int m = 16;
#pragma unroll
    for (int h = TT / 2; h >= 1; h >>= 1) {
        const bool upper = (lane & m) != 0;
#pragma unroll
        for (int j = 0; j < h; ++j) {
            float send = upper ? v[j] : v[j + h];
            float keep = upper ? v[j + h] : v[j];
            v[j] = keep + __shfl_xor_sync(0xffffffffu, send, m);
        }
        m >>= 1;
    }
    for (; m >= 1; m >>= 1) v[0] += __shfl_xor_sync(0xffffffffu, v[0], m);
}

template <int TT>
struct Log2;
template <> struct Log2<1> { static constexpr int v = 0; };
template <> struct Log2<2> { static constexpr int v = 1; };
template <> struct Log2<4> { static constexpr int v = 2; };
template <> struct Log2<8> { static constexpr int v = 3; };
template <> struct Log2<16> { static constexpr int v = 4; };
template <> struct Log2<32> { static constexpr int v = 5; };

__device__ __forceinline__ void unpack8(const uint4 &u, float (&f)[8]) {
    f[0] = __uint_as_float(u.x << 16); f[1] = __uint_as_float(u.x & 0xffff0000u);
    f[2] = __uint_as_float(u.y << 16); f[3] = __uint_as_float(u.y & 0xffff0000u);
    f[4] = __uint_as_float(u.z << 16); f[5] = __uint_as_float(u.z & 0xffff0000u);
    f[6] = __uint_as_float(u.w << 16); f[7] = __uint_as_float(u.w & 0xffff0000u);
}

__device__ __forceinline__ const uint16_t *weight_row(const GemmArgs &a, int n, int &kseg) {
    kseg = a.Wk2 ? a.K1 : a.K;
    if (n < a.n0) return a.W0 + (size_t)n * kseg;
    n -= a.n0;
    if (n < a.n1) return a.W1 + (size_t)n * a.K;
    n -= a.n1;
    return a.W2 + (size_t)n * a.K;
}

// Accumulate one weight row against TT tokens starting at t0.
template <int TT>
__device__ __forceinline__ void row_dot(const GemmArgs &a, const uint16_t *w, int kseg, int n,
                                        int t0, int lane, float (&acc)[TT]) {
#pragma unroll
    for (int t = 0; t < TT; ++t) acc[t] = 0.f;
    for (int k = lane * 8; k < a.K; k += 256) {
        const uint16_t *src = (k < kseg) ? (w + k) : (a.Wk2 + (size_t)n * (a.K - a.K1) + (k - a.K1));
        uint4 wu = ld_stream_u4(src);
        float wf[8];
        unpack8(wu, wf);
#pragma unroll
        for (int t = 0; t < TT; ++t) {
            if (t0 + t < a.T) {
                const uint16_t *xr = a.X + (size_t)(2 * (t0 + t)) * a.ldx + k;
                uint4 hu = *reinterpret_cast<const uint4 *>(xr);
                uint4 lu = *reinterpret_cast<const uint4 *>(xr + a.ldx);
                float hf[8], lf[8];
                unpack8(hu, hf);
                unpack8(lu, lf);
                float s = acc[t];
#pragma unroll
                for (int e = 0; e < 8; ++e) s = fmaf(wf[e], hf[e] + lf[e], s);
                acc[t] = s;
            }
        }
    }
}

template <int TT>
__global__ void __launch_bounds__(kWarps * 32) gemm_simt_kernel(GemmArgs a) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    constexpr int LG = Log2<TT>::v;
    const int my_tok = lane >> (5 - LG);
    const bool owner = (lane & ((1 << (5 - LG)) - 1)) == 0;

    if (a.epi == EPI_ARGMAX) {
        // Rows are visited in increasing order per warp; the CTA keeps per-token states.
        __shared__ ArgTop sh[kWarps][TT];
        for (int t0 = 0; t0 < a.T; t0 += TT) {
            ArgTop st = argtop_empty(0x7fffffff);
            for (int n = blockIdx.x * kWarps + warp; n < a.N; n += gridDim.x * kWarps) {
                int kseg;
                const uint16_t *w = weight_row(a, n, kseg);
                float acc[TT];
                row_dot<TT>(a, w, kseg, n, t0, lane, acc);
                reduce_scatter<TT>(acc, lane);
                st = argtop_push(st, acc[0], n);
            }
            if (owner) sh[warp][my_tok] = st;
            __syncthreads();
            if (threadIdx.x < TT && t0 + threadIdx.x < a.T) {
                ArgTop r = sh[0][threadIdx.x];
                for (int w2 = 1; w2 < kWarps; ++w2) r = argtop_merge(r, sh[w2][threadIdx.x]);
                a.part[(size_t)blockIdx.x * a.T + t0 + threadIdx.x] = r;
            }
            __syncthreads();
        }
        return;
    }

    for (int n = blockIdx.x * kWarps + warp; n < a.N; n += gridDim.x * kWarps) {
        for (int t0 = 0; t0 < a.T; t0 += TT) {
            if (a.epi == EPI_SWIGLU) {
                float g[TT], u[TT];
                row_dot<TT>(a, a.W0 + (size_t)n * a.K, a.K, n, t0, lane, g);
                row_dot<TT>(a, a.W1 + (size_t)n * a.K, a.K, n, t0, lane, u);
                reduce_scatter<TT>(g, lane);
                reduce_scatter<TT>(u, lane);
                const int t = t0 + my_tok;
                if (owner && t < a.T) {
                    float z = g[0];
                    float act = z / (1.f + expf(-z)) * u[0];
                    uint16_t hi, lo;
                    split_hi_lo(act, hi, lo);
                    a.pack_out[(size_t)(2 * t) * a.ldpo + n] = hi;
                    a.pack_out[(size_t)(2 * t + 1) * a.ldpo + n] = lo;
                }
            } else {
                int kseg;
                const uint16_t *w = weight_row(a, n, kseg);
                float acc[TT];
                row_dot<TT>(a, w, kseg, n, t0, lane, acc);
                reduce_scatter<TT>(acc, lane);
                const int t = t0 + my_tok;
                if (owner && t < a.T) {
                    float v = acc[0];
                    if (a.epi == EPI_RESID) v += a.resid[(size_t)t * a.ldr + n];
                    a.out[(size_t)t * a.ldo + n] = v;
                }
            }
        }
    }
}

template <int TT>
int launch_tt(const GemmArgs &a, cudaStream_t s, int *np) {
    int rows_ctas = (a.N + kWarps - 1) / kWarps;
    int grid = a.epi == EPI_ARGMAX ? min(rows_ctas, 4 * kNumSMs) : min(rows_ctas, 64 * kNumSMs);
    grid = max(grid, 1);
    if (np) *np = grid;
    gemm_simt_kernel<TT><<<grid, kWarps * 32, 0, s>>>(a);
    return cuda_check("gemm_simt_kernel");
}

}  // namespace

int launch_gemm(const GemmArgs &a, cudaStream_t s, int *n_partials_out) {
    if (a.N <= 0 || a.T <= 0) {
        if (n_partials_out) *n_partials_out = 0;
        return DF_OK;
    }
    if (a.T <= 1) return launch_tt<1>(a, s, n_partials_out);
    if (a.T <= 2) return launch_tt<2>(a, s, n_partials_out);
    if (a.T <= 4) return launch_tt<4>(a, s, n_partials_out);
    if (a.T <= 8) return launch_tt<8>(a, s, n_partials_out);
    if (a.T <= 16) return launch_tt<16>(a, s, n_partials_out);
    return launch_tt<32>(a, s, n_partials_out);
}

}  // namespace df

// Split-KV attention on the 5th-generation tensor cores, for head_dim 128 or 256 and up to 32
// query rows per KV head (a DFlash block of 16 positions x 2 query heads per KV head, or one
// MTP token x its GQA group).
//
// Same partial-output contract as the CUDA-core kernel in k_attn.cu: each CTA takes one chunk
// of keys of one (sequence, KV head) and writes, per query row, o = sum_k p_k v_k, m (the
// score maximum, log2 units) and l = sum_k p_k with p_k = 2^(s_k - m); attn_combine_kernel
// merges the chunks. Scores follow hf2q 0.1.1 models/qwen35/mtp.rs (`sdpa` step of the draft
// forward: softmax(q k^T / sqrt(d)) v over the visible keys).
//
// The cache holds F32 keys and values. Each 128-key x 128-dim piece (a "unit") lands in a
// 64 KB shared-memory buffer by one TMA box load (three buffers in flight), is split in place
// into hi = bf16(x) and lo = bf16(x - hi) (about 16 mantissa bits) in the 128-byte-swizzled
// K-major layout, and is multiplied with three kind::f16 MMAs (hi.hi + hi.lo + lo.hi, F32
// accumulation in TMEM):
//   scores  S^T [128 keys x NP rows]  = K [128 x d] . Q^T          (one TMEM block per tile)
//   output  O^T [128 dims x NP rows] += V^T [128 x 128 keys] . P^T  (per 128-dim half)
// A chunk's scores stay in TMEM, up to (512 - halves*NP)/NP tiles per pass, so the softmax
// maximum is exact per pass: pass 1 takes the row maxima, pass 2 turns each tile into
// probabilities (BF16 hi/lo in shared memory) right before its P.V MMAs. A longer chunk runs in
// several passes whose (max, sum, o) are merged in registers, rescaled once per pass. Values are
// transposed while they are split, so both products read K-major operands.
//
// 288 threads: warps 0-7 convert; warp 8 issues the TMA loads and the MMAs and refills a
// buffer once the MMAs reading it are done; warps w and w + 4 share TMEM lane quarter w % 4 and
// split the rows in the softmax and the read-out. Block rows (keys past the cache rows) come from
// kb/vb with plain loads during the split; keys past the chunk are written as zeros.
#include <cuda_bf16.h>
#include <string.h>

#include "df_internal.cuh"
#include "tc_ptx.cuh"

namespace df {

namespace {

constexpr int kConvThreads = 256;             // warps 0-7: split, softmax, read-out
constexpr int kTcThreads = kConvThreads + 32;  // warp 8: TMA and MMA issue
constexpr int kTcKeys = 128;                  // keys per tile
constexpr int kTmemCols = 512;
constexpr int kOpBytes = 128 * 128 * 2;       // one 128 x 128 BF16 operand (hi or lo): 32 KB
constexpr int kAtomBytes = 128 * 128;         // one 64-element-wide column block of 128 rows

template <int D, int NP, int NBUF>
constexpr bool attn_tc_smem_bound() {
    return 1024 + NBUF * 2 * kOpBytes + (D / 128) * 2 * NP * 256 + 2 * NP * 256 + 9 * NP * 4 +
               3 * 2 * NBUF * 8 + 16 <= 232448;
}

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Byte offset of element (row, k), k in [0, 128), in a K-major operand of `rows` rows kept as
// two 64-element column blocks with the 128-byte swizzle (the layout TMA's SWIZZLE_128B writes).
__device__ __forceinline__ uint32_t sw_off(int rows, int row, int k) {
    return (uint32_t)((k >> 6) * rows * 128 + row * 128 + ((((k & 63) >> 3) ^ (row & 7)) << 4) +
                      ((k & 7) << 1));
}

// 8 F32 values -> 8 BF16 hi values and 8 BF16 lo values (x - hi), packed two per word.
__device__ __forceinline__ void split8(const float (&x)[8], uint4 &hi, uint4 &lo) {
    uint32_t h[4], l[4];
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        const __nv_bfloat162 hb = __floats2bfloat162_rn(x[2 * p], x[2 * p + 1]);
        const float2 hf = __bfloat1622float2(hb);
        const __nv_bfloat162 lb = __floats2bfloat162_rn(x[2 * p] - hf.x, x[2 * p + 1] - hf.y);
        h[p] = *reinterpret_cast<const uint32_t *>(&hb);
        l[p] = *reinterpret_cast<const uint32_t *>(&lb);
    }
    hi = make_uint4(h[0], h[1], h[2], h[3]);
    lo = make_uint4(l[0], l[1], l[2], l[3]);
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, const uint4 &v) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w)
                 : "memory");
}

__device__ __forceinline__ void st_shared_v2(uint32_t addr, uint32_t x, uint32_t y) {
    asm volatile("st.shared.v2.b32 [%0], {%1, %2};" ::"r"(addr), "r"(x), "r"(y) : "memory");
}

__device__ __forceinline__ void st_shared_u16(uint32_t addr, uint16_t v) {
    asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr), "h"(v) : "memory");
}

// Barrier of the eight splitting warps (named barrier 1; warp 8 does not take part).
__device__ __forceinline__ void conv_sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

template <int NPH>
__device__ __forceinline__ void tmem_rows(uint32_t taddr, float (&v)[NPH]) {
    if constexpr (NPH == 16) {
        uint32_t r[16];
        tmem_ld16(taddr, r);
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
    } else {
        uint32_t r[8];
        tmem_ld8(taddr, r);
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
    }
}

struct AttnTcParams {
    CUtensorMap kmap, vmap;   // F32 or BF16 [B * nkv * cap rows, d cols], 128 x 128 boxes
    AttnArgs a;
};

// MP: the chunk may need several passes (instantiated only for chunks longer than one pass).
// KVB: the cache holds BF16 (the split keeps only the exact hi half: two MMAs per K step, and
// twice as many half-size staging buffers in the same shared memory).
template <int D, int NP, int NBUF, bool MP, bool KVB>
__global__ void __launch_bounds__(kTcThreads, 1) attn_tc_kernel(const __grid_constant__ AttnTcParams P) {
    constexpr int NB = KVB ? 2 * NBUF : NBUF;          // staging buffers
    constexpr int kUnit = KVB ? kOpBytes : 2 * kOpBytes;  // bytes of one staged unit
    constexpr int NH = D / 128;               // 128-wide halves of the head dimension
    constexpr int NPH = NP / 2;               // rows per thread in the softmax and read-out
    constexpr int kQBytes = NP * 256;         // one NP x 128 BF16 operand (Q or P, hi or lo)
    const AttnArgs &a = P.a;
    extern __shared__ uint8_t sm_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(sm_raw) + 1023) &
                                              ~uintptr_t(1023));
    uint8_t *kvb = sm;                                  // NB x 64 KB: F32 staging, then hi | lo
    uint8_t *qsm = sm + NB * kUnit;            // [NH][hi, lo] Q operands
    uint8_t *psm = qsm + NH * 2 * kQBytes;              // [hi, lo] P operand (second buffer)
    float *red = reinterpret_cast<float *>(psm + 2 * kQBytes);   // [4][NP] maxima, [4][NP] sums
    float *mrun = red + 8 * NP;                                  // [NP] running row maxima
    uint64_t *full = reinterpret_cast<uint64_t *>(mrun + NP);    // [NB] staging landed
    uint64_t *mdone = full + NB;                               // [NB] MMAs of the unit done
    uint64_t *conv = mdone + NB;                               // [NB] unit split, ready for MMA
    uint32_t *tslot = reinterpret_cast<uint32_t *>(conv + NB);
    int *abort_flag = reinterpret_cast<int *>(tslot + 1);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int chunk = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
    pdl_trigger();
    if (tid == kConvThreads) {
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&P.kmap)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&P.vmap)) : "memory");
    }
    pdl_wait();
    const int rep = a.nq / a.nkv;
    const int R = a.blk * rep;
    const int nn = a.n_new ? min(max(a.n_new[b], 0), a.n_new_max) : 0;
    const long long sc = (long long)a.seq_len[b] + nn + a.extra_rows;
    const int S_cache = (int)min(max(sc, 0LL), (long long)a.cap);
    const int S = S_cache + (a.kb ? a.blk : 0);
    const int c0 = min(S, chunk * a.chunk), c1 = min(S, c0 + a.chunk);
    const int n_tiles = (c1 - c0 + kTcKeys - 1) / kTcKeys;
    const size_t head_off = (size_t)b * a.nkv + g;
    float *part = a.part + ((head_off * a.n_chunks + chunk) * (size_t)R) * (D + 2);
    if (n_tiles == 0) {
        for (int i = tid; i < R * (D + 2); i += kTcThreads) part[i] = (i % (D + 2)) == D ? -INFINITY : 0.f;
        return;
    }
    // A chunk longer than the score memory runs in passes of at most max_tp tiles; each pass
    // has an exact maximum and its output is merged into running (max, sum, o) registers.
    const int max_tp = (kTmemCols - NH * NP) / NP;
    const int n_pass = MP ? (n_tiles + max_tp - 1) / max_tp : 1;
    if (!MP && n_tiles > max_tp) {           // the host plans single-pass launches within bounds
        if (tid == 0) set_status(a.status, DF_ESHAPE);
        for (int i = tid; i < R * (D + 2); i += kTcThreads) part[i] = (i % (D + 2)) == D ? -INFINITY : 0.f;
        return;
    }
    const int tpp = (n_tiles + n_pass - 1) / n_pass;    // tiles per pass (the last may be short)
    const int upp = 2 * tpp * NH;                        // units per full pass
    const int nU = 2 * n_tiles * NH;
    const bool multi = MP && n_pass > 1;
    const uint64_t pol = policy_evict_first();
    // Unit u of pass p: the pass's K units (tile-major, then 128-wide half), then its V units.
    struct UnitInfo {
        int t0, nt, v, t, h;
    };
    auto decode = [&](int u) -> UnitInfo {
        const int p = min(u / upp, n_pass - 1);
        UnitInfo x;
        x.t0 = p * tpp;
        x.nt = min(n_tiles, x.t0 + tpp) - x.t0;
        int local = u - p * upp;
        x.v = local >= x.nt * NH;
        if (x.v) local -= x.nt * NH;
        x.t = x.t0 + local / NH;
        x.h = local % NH;
        return x;
    };
    // Unit u: K or V of tile t, 128-wide half h, staged by one TMA box of 128 rows.
    auto issue = [&](int u) {
        const UnitInfo x = decode(u);
        const bool isV = x.v;
        const int t = x.t, h = x.h, bf = u % NB;
        mbar_expect_tx(&full[bf], (uint32_t)kUnit);
        tma_load_2d(kvb + (size_t)bf * kUnit, isV ? &P.vmap : &P.kmap, &full[bf], h * 128,
                    (int)(head_off * a.cap) + c0 + t * kTcKeys, pol);
    };

    // Q rows are loaded before the first TMA boxes are issued, so they do not queue behind them.
    constexpr int QI = (NP * (D / 8) + kConvThreads - 1) / kConvThreads;
    float qx[QI][8];
#pragma unroll
    for (int i = 0; i < QI; ++i) {
        const int idx = tid + i * kConvThreads;
        const int r = idx / (D / 8), d = 8 * (idx % (D / 8));
#pragma unroll
        for (int e = 0; e < 8; ++e) qx[i][e] = 0.f;
        if (tid < kConvThreads && idx < NP * (D / 8) && r < R) {
            const float *qp = a.q + (((size_t)b * a.blk + r / rep) * a.nq + g * rep + r % rep) * D + d;
            const float4 u = *reinterpret_cast<const float4 *>(qp);
            const float4 v = *reinterpret_cast<const float4 *>(qp + 4);
            qx[i][0] = u.x; qx[i][1] = u.y; qx[i][2] = u.z; qx[i][3] = u.w;
            qx[i][4] = v.x; qx[i][5] = v.y; qx[i][6] = v.z; qx[i][7] = v.w;
        }
    }
    if (warp == 0) {
        tmem_alloc(tslot, kTmemCols);
        tmem_relinquish();
    }
    if (tid == kConvThreads) {
        for (int i = 0; i < NB; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&mdone[i], 1);
            mbar_init(&conv[i], kConvThreads / 32);
        }
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        for (int u = 0; u < min(NB, nU); ++u) issue(u);
    }
    // Q -> hi/lo operands (rows R..NP-1 zero)
#pragma unroll
    for (int i = 0; i < QI; ++i) {
        const int idx = tid + i * kConvThreads;
        if (tid < kConvThreads && idx < NP * (D / 8)) {
            const int r = idx / (D / 8), d = 8 * (idx % (D / 8));
            uint4 hi, lo;
            split8(qx[i], hi, lo);
            const int h = d >> 7;
            const uint32_t o = sw_off(NP, r, d & 127);
            st_shared_v4(smem_u32(qsm + (2 * h) * kQBytes + o), hi);
            st_shared_v4(smem_u32(qsm + (2 * h + 1) * kQBytes + o), lo);
        }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    const int ocol = tpp * NP;                // O^T accumulators after a pass's score tiles
    // P operand of tile t. One pass: two buffers in turn, buffer 0 reusing the Q operands' space
    // (every score MMA has completed before the first P is written), buffer 1 following it.
    // Several passes: Q stays live, so one buffer after the Q operands.
    auto p_buf = [&](int t) -> uint32_t {
        return multi ? smem_u32(psm) : smem_u32(qsm) + (uint32_t)((t & 1) * 2 * kQBytes);
    };

    // In-place conversion of a staged unit: every thread reads its 64 F32 values (block rows
    // from kb/vb, zeros past the chunk's last key), the CTA synchronises, then the values go back
    // as BF16 hi (first 32 KB) and lo (second 32 KB) in the swizzled K-major operand layout.
    float xv[64];
    auto read_unit = [&](int u) {
        const UnitInfo x = decode(u);
        const bool isV = x.v;
        const int t = x.t, h = x.h;
        const float *st = reinterpret_cast<const float *>(kvb + (size_t)(u % NB) * kUnit);
        const uint16_t *stb = reinterpret_cast<const uint16_t *>(st);
        auto stage4 = [&](int kr, int c4) -> float4 {     // 4 staged values at row kr, col c4
            if constexpr (KVB) {
                const uint2 w = *reinterpret_cast<const uint2 *>(stb + kr * 128 + c4);
                return make_float4(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xffff0000u),
                                   __uint_as_float(w.y << 16), __uint_as_float(w.y & 0xffff0000u));
            } else {
                return *reinterpret_cast<const float4 *>(st + kr * 128 + c4);
            }
        };
        const float *blkp = isV ? a.vb : a.kb;
        const int kbase = c0 + t * kTcKeys;
        if (!isV) {
#pragma unroll
            for (int it = 0; it < 16; ++it) {
                const int kr = it * 8 + warp, key = kbase + kr;
                float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
                if (key < S_cache) v = stage4(kr, 4 * lane);
                else if (key < c1)
                    v = __ldcg(reinterpret_cast<const float4 *>(
                        blkp + (head_off * a.blk + (key - S_cache)) * D + h * 128 + 4 * lane));
                xv[4 * it] = v.x; xv[4 * it + 1] = v.y; xv[4 * it + 2] = v.z; xv[4 * it + 3] = v.w;
            }
        } else {
#pragma unroll
            for (int it = 0; it < 2; ++it) {
                const int wi = it * 8 + warp;
                const int ob = (wi & 3) * 4 + (lane & 3), qd = (wi >> 2) * 8 + (lane >> 2);
#pragma unroll
                for (int jj = 0; jj < 8; ++jj) {
                    const int kr = 8 * ob + jj, key = kbase + kr;
                    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
                    if (key < S_cache) v = stage4(kr, 4 * qd);
                    else if (key < c1)
                        v = __ldcg(reinterpret_cast<const float4 *>(
                            blkp + (head_off * a.blk + (key - S_cache)) * D + h * 128 + 4 * qd));
                    const int o = 32 * it + 4 * jj;
                    xv[o] = v.x; xv[o + 1] = v.y; xv[o + 2] = v.z; xv[o + 3] = v.w;
                }
            }
        }
    };
    auto write_unit = [&](int u) {
        const uint32_t hi = smem_u32(kvb + (size_t)(u % NB) * kUnit), lo = hi + kOpBytes;
        if (!decode(u).v) {
#pragma unroll
            for (int it = 0; it < 16; ++it) {
                const int kr = it * 8 + warp;
                const __nv_bfloat162 h01 = __floats2bfloat162_rn(xv[4 * it], xv[4 * it + 1]);
                const __nv_bfloat162 h23 = __floats2bfloat162_rn(xv[4 * it + 2], xv[4 * it + 3]);
                const float2 f01 = __bfloat1622float2(h01), f23 = __bfloat1622float2(h23);
                const __nv_bfloat162 l01 = __floats2bfloat162_rn(xv[4 * it] - f01.x, xv[4 * it + 1] - f01.y);
                const __nv_bfloat162 l23 = __floats2bfloat162_rn(xv[4 * it + 2] - f23.x, xv[4 * it + 3] - f23.y);
                const uint32_t o = sw_off(128, kr, 4 * lane);
                st_shared_v2(hi + o, *reinterpret_cast<const uint32_t *>(&h01),
                             *reinterpret_cast<const uint32_t *>(&h23));
                if constexpr (!KVB)
                    st_shared_v2(lo + o, *reinterpret_cast<const uint32_t *>(&l01),
                                 *reinterpret_cast<const uint32_t *>(&l23));
            }
        } else {
#pragma unroll
            for (int it = 0; it < 2; ++it) {
                const int wi = it * 8 + warp;
                const int ob = (wi & 3) * 4 + (lane & 3), qd = (wi >> 2) * 8 + (lane >> 2);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    float x[8];
#pragma unroll
                    for (int jj = 0; jj < 8; ++jj) x[jj] = xv[32 * it + 4 * jj + i];
                    uint4 vh, vl;
                    split8(x, vh, vl);
                    const uint32_t o = sw_off(128, 4 * qd + i, 8 * ob);
                    st_shared_v4(hi + o, vh);
                    if constexpr (!KVB) st_shared_v4(lo + o, vl);
                }
            }
        }
    };
    // Three MMAs per 16-wide K step: hi.hi + hi.lo + lo.hi (K = 128 in 8 steps).
    const uint32_t idesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(NP >> 3) << 17) |
                           ((uint32_t)(128 >> 4) << 24);
    auto mma3 = [&](uint32_t dt, uint32_t a_hi, uint32_t a_lo, uint32_t b_hi, uint32_t b_lo,
                    bool acc) {
#pragma unroll
        for (int kb = 0; kb < 2; ++kb)
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
                const uint32_t oa = kb * kAtomBytes + ks * 32, ob = kb * NP * 128 + ks * 32;
                mma_bf16(dt, sw128_desc(a_hi + oa), sw128_desc(b_hi + ob), idesc,
                         (acc || kb || ks) ? 1u : 0u);
                mma_bf16(dt, sw128_desc(a_hi + oa), sw128_desc(b_lo + ob), idesc, 1u);
                if constexpr (!KVB) mma_bf16(dt, sw128_desc(a_lo + oa), sw128_desc(b_hi + ob), idesc, 1u);
            }
    };
    auto wait_mma = [&](int u) {   // the MMAs of unit u (and all before it) have completed
        mbar_wait(&mdone[u % NB], (uint32_t)((u / NB) & 1), abort_flag, a.status);
        tc_fence_after();
    };

    const float scale = 1.4426950408889634f / sqrtf((float)D);
    const int lq = warp & 3, r0 = (warp >> 2) * NPH;
    const uint32_t lane_addr = (uint32_t)(lq * 32) << 16;
    auto row_ok = [&](int key, int row) {
        if (key >= c1 || row >= R) return false;
        return !(a.causal_block && key >= S_cache && key - S_cache > row / rep);
    };
    float Mrow[NPH], lsum[NPH];
    float lrun[MP ? NPH : 1], orun[MP ? NH : 1][MP ? NPH : 1];
#pragma unroll
    for (int r = 0; r < NPH; ++r) lsum[r] = 0.f;
    if constexpr (MP) {
#pragma unroll
        for (int r = 0; r < NPH; ++r) {
            lrun[r] = 0.f;
#pragma unroll
            for (int h = 0; h < NH; ++h) orun[h][r] = 0.f;
        }
    }
    if (tid < NP) mrun[tid] = -INFINITY;

    if (warp == kConvThreads / 32) {
        // TMA / MMA issuer: MMAs of unit u once its split has landed; then refill its buffer.
        if (lane == 0) {
            for (int u = 0; u < nU; ++u) {
                const uint32_t ph = (uint32_t)((u / NB) & 1);
                if (!mbar_wait(&conv[u % NB], ph, abort_flag, a.status)) break;
                tc_fence_after();
                const uint32_t ahi = smem_u32(kvb + (size_t)(u % NB) * kUnit), alo = ahi + kOpBytes;
                const UnitInfo x = decode(u);
                if (!x.v) {
                    const uint32_t qhi = smem_u32(qsm + (2 * x.h) * kQBytes), qlo = qhi + kQBytes;
                    mma3(tmem + (x.t - x.t0) * NP, ahi, alo, qhi, qlo, x.h > 0);
                } else {
                    const uint32_t phi = p_buf(x.t), plo = phi + kQBytes;
                    mma3(tmem + ocol + x.h * NP, ahi, alo, phi, plo, x.t > x.t0);
                }
                mma_commit(&mdone[u % NB]);
                if (u + NB < nU) {
                    if (!mbar_wait(&mdone[u % NB], ph, abort_flag, a.status)) break;
                    issue(u + NB);
                }
            }
        }
        __syncwarp();
    } else {
        for (int u = 0; u < nU; ++u) {
            const UnitInfo x = decode(u);
            if (x.v && x.h == 0) {
                const int t = x.t, tl = t - x.t0;
                if (tl == 0) {
                    // softmax pass 1: exact row maxima over the pass's tiles
                    wait_mma((u / upp) * upp + x.nt * NH - 1);
                    float mx[NPH];
#pragma unroll
                    for (int r = 0; r < NPH; ++r) mx[r] = -INFINITY;
                    for (int tt = 0; tt < x.nt; ++tt) {
                        float s[NPH];
                        tmem_rows<NPH>(tmem + lane_addr + tt * NP + r0, s);
                        const int key = c0 + (x.t0 + tt) * kTcKeys + lq * 32 + lane;
#pragma unroll
                        for (int r = 0; r < NPH; ++r)
                            if (row_ok(key, r0 + r)) mx[r] = fmaxf(mx[r], s[r] * scale);
                    }
#pragma unroll
                    for (int r = 0; r < NPH; ++r) {
                        const float m = warp_max(mx[r]);
                        if (lane == 0) red[lq * NP + r0 + r] = m;
                    }
                    conv_sync();
#pragma unroll
                    for (int r = 0; r < NPH; ++r)
                        Mrow[r] = fmaxf(fmaxf(red[r0 + r], red[NP + r0 + r]),
                                        fmaxf(red[2 * NP + r0 + r], red[3 * NP + r0 + r]));
                } else if (multi) {
                    wait_mma(u - 1);   // one P buffer: the previous tile's P.V MMAs are done
                } else if (tl >= 2) {
                    // P operands alternate between two buffers: the one for tile t was last read by
                    // the P.V MMAs of tile t - 2. Waiting on that older unit is only safe while
                    // its barrier cannot have completed a later phase (NB > NH); otherwise wait
                    // on the most recent unit, which covers it.
                    wait_mma(NB > NH ? u - NH - 1 : u - 1);
                }
                // pass 2 for tile t: probabilities -> BF16 hi/lo P operand
                float s[NPH];
                tmem_rows<NPH>(tmem + lane_addr + tl * NP + r0, s);
                const int kt = lq * 32 + lane;
                const int key = c0 + t * kTcKeys + kt;
                const uint32_t phi = p_buf(t), plo = phi + kQBytes;
#pragma unroll
                for (int r = 0; r < NPH; ++r) {
                    const int row = r0 + r;
                    float p = 0.f;
                    if (row_ok(key, row) && Mrow[r] != -INFINITY) p = ex2(s[r] * scale - Mrow[r]);
                    lsum[r] += p;
                    const uint16_t ph = f32_to_bf16_bits(p);
                    const uint16_t pl = f32_to_bf16_bits(p - bf16_bits_to_f32(ph));
                    const uint32_t o = sw_off(NP, row, kt);
                    st_shared_u16(phi + o, ph);
                    st_shared_u16(plo + o, pl);
                }
            }
            mbar_wait(&full[u % NB], (uint32_t)((u / NB) & 1), abort_flag, a.status);
            read_unit(u);
            conv_sync();
            write_unit(u);
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&conv[u % NB]);
            if constexpr (MP) {
                if (x.v && x.t == x.t0 + x.nt - 1 && x.h == NH - 1) {
                    // end of a pass: merge its (max, sum, o) into the running values
                    wait_mma(u);
#pragma unroll
                    for (int h = 0; h < NH; ++h) {
                        float o[NPH];
                        tmem_rows<NPH>(tmem + lane_addr + ocol + h * NP + r0, o);
#pragma unroll
                        for (int r = 0; r < NPH; ++r) {
                            const float Mr = mrun[r0 + r], Mn = fmaxf(Mr, Mrow[r]);
                            if (Mn == -INFINITY) continue;
                            const float so = Mr == -INFINITY ? 0.f : ex2(Mr - Mn);
                            const float sn = Mrow[r] == -INFINITY ? 0.f : ex2(Mrow[r] - Mn);
                            orun[h][r] = orun[h][r] * so + o[r] * sn;
                            if (h == NH - 1) {
                                lrun[r] = lrun[r] * so + lsum[r] * sn;
                                lsum[r] = 0.f;
                            }
                        }
                    }
                    conv_sync();                // everyone has read mrun before it moves
                    if (lq == 0 && lane == 0)
#pragma unroll
                        for (int r = 0; r < NPH; ++r) mrun[r0 + r] = fmaxf(mrun[r0 + r], Mrow[r]);
                    conv_sync();
                }
            }
        }

        // read-out: o of this thread's rows, row sums, maxima
        if constexpr (MP) {
#pragma unroll
            for (int r = 0; r < NPH; ++r) {
                const float l = warp_sum(lrun[r]);
                if (lane == 0) red[4 * NP + lq * NP + r0 + r] = l;
            }
#pragma unroll
            for (int h = 0; h < NH; ++h) {
                const int d = h * 128 + lq * 32 + lane;
#pragma unroll
                for (int r = 0; r < NPH; ++r)
                    if (r0 + r < R) part[(size_t)(r0 + r) * (D + 2) + d] = orun[h][r];
            }
        } else {
            wait_mma(nU - 1);
#pragma unroll
            for (int r = 0; r < NPH; ++r) {
                const float l = warp_sum(lsum[r]);
                if (lane == 0) red[4 * NP + lq * NP + r0 + r] = l;
            }
            if (lq == 0 && lane == 0)
#pragma unroll
                for (int r = 0; r < NPH; ++r) mrun[r0 + r] = Mrow[r];
#pragma unroll
            for (int h = 0; h < NH; ++h) {
                float o[NPH];
                tmem_rows<NPH>(tmem + lane_addr + ocol + h * NP + r0, o);
                const int d = h * 128 + lq * 32 + lane;
#pragma unroll
                for (int r = 0; r < NPH; ++r)
                    if (r0 + r < R) part[(size_t)(r0 + r) * (D + 2) + d] = o[r];
            }
        }
        conv_sync();
        if (tid < R) {
            const float M = mrun[tid];
            const float L = red[4 * NP + tid] + red[5 * NP + tid] + red[6 * NP + tid] + red[7 * NP + tid];
            part[(size_t)tid * (D + 2) + D] = M;
            part[(size_t)tid * (D + 2) + D + 1] = L;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

template <int D, int NP, int NBUF>
size_t attn_tc_smem() {
    return 1024 + NBUF * 2 * (size_t)kOpBytes + (D / 128) * 2 * (size_t)NP * 256 +
           2 * (size_t)NP * 256 + 9 * NP * sizeof(float) + 3 * 2 * NBUF * sizeof(uint64_t) + 16;
}

template <int D, int NP, int NBUF>
int launch_tc(const AttnArgs &a, cudaStream_t s) {
    constexpr int max_keys_one_pass = (kTmemCols - (D / 128) * NP) / NP * kTcKeys;
    static_assert(attn_tc_smem_bound<D, NP, NBUF>(), "shared memory");
    AttnTcParams p;
    memset(&p, 0, sizeof(p));
    const uint64_t rows = (uint64_t)a.B * a.nkv * a.cap;
    if (rows + kTcKeys > 0x7fffffffull)
        return fail(DF_ESHAPE, "tensor-core attention: %llu cache rows exceed the TMA row range",
                    (unsigned long long)rows);
    const CUtensorMapDataType dt = a.kv_bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    const int eb = a.kv_bf16 ? 2 : 4;
    DF_TRY(make_tma_2d(&p.kmap, a.cache_k, dt, eb, D, rows, D, 128, 128, CU_TENSOR_MAP_SWIZZLE_NONE));
    DF_TRY(make_tma_2d(&p.vmap, a.cache_v, dt, eb, D, rows, D, 128, 128, CU_TENSOR_MAP_SWIZZLE_NONE));
    p.a = a;
    dim3 grid(a.n_chunks, a.nkv, a.B);
    const size_t smem = attn_tc_smem<D, NP, NBUF>();
    const bool one = a.chunk <= max_keys_one_pass;
    if (a.kv_bf16)
        return one ? launch_k("attn_tc_kernel", attn_tc_kernel<D, NP, NBUF, false, true>, grid,
                              dim3(kTcThreads), smem, s, p)
                   : launch_k("attn_tc_kernel", attn_tc_kernel<D, NP, NBUF, true, true>, grid,
                              dim3(kTcThreads), smem, s, p);
    return one ? launch_k("attn_tc_kernel", attn_tc_kernel<D, NP, NBUF, false, false>, grid,
                          dim3(kTcThreads), smem, s, p)
               : launch_k("attn_tc_kernel", attn_tc_kernel<D, NP, NBUF, true, false>, grid,
                          dim3(kTcThreads), smem, s, p);
}

}  // namespace

bool attn_tc_supported(int d, int rows) { return (d == 128 || d == 256) && rows >= 1 && rows <= 32; }

int launch_attn_tc(const AttnArgs &a, cudaStream_t s) {
    const int R = a.blk * (a.nq / a.nkv);
    if (!attn_tc_supported(a.d, R) || a.chunk % kTcKeys != 0)
        return fail(DF_ESHAPE, "tensor-core attention: d=%d rows=%d chunk=%d", a.d, R, a.chunk);
    if (a.d == 128) return R <= 16 ? launch_tc<128, 16, 3>(a, s) : launch_tc<128, 32, 3>(a, s);
    return R <= 16 ? launch_tc<256, 16, 3>(a, s) : launch_tc<256, 32, 2>(a, s);
}

}  // namespace df

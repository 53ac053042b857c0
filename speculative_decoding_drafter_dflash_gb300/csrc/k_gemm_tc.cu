// Projections on the 5th-generation tensor cores: y[t, n] = sum_k x[t, k] W[n, k] for BF16
// weights W [N, K] (row-major) and F32 activations x packed as two BF16 rows per token
// (hi = bf16(x), lo = bf16(x - hi)), so one kind::f16 MMA with N = 2T columns carries the
// activations to ~16 mantissa bits and the two columns of a token are summed in F32 in the
// epilogue.
//
//   A (weights, M = 128 rows x K)   TMA, 128-byte swizzle, K-major, 64-wide K blocks; or, from
//                                   a tiled copy of the weights (tile_projection), one bulk
//                                   copy of two K blocks (32 KB) per pipeline stage
//   B (packed x, N = 2T rows x K)   TMA, same layout; rows past 2T are zero-filled by TMA
//   D (F32, 128 lanes x N columns)  TMEM, two accumulators so the epilogue of one tile
//                                   overlaps the MMAs of the next
//
// One persistent CTA per SM, warp-specialised: warp 0 issues TMA loads, warp 1 issues
// tcgen05.mma (one elected lane) and owns the TMEM allocation, warps 2-5 run the epilogue.
// Work is split stream-K style: the (tile, K-block) space is cut into equal contiguous ranges,
// one per CTA, so every SM streams the same number of weight bytes. A tile shared by several
// CTAs is finished by the last one to arrive, which sums the partial tiles in CTA order (the
// result does not depend on arrival order).
//
// Epilogues: plain store, residual add, SwiGLU (gate rows 0-63 and up rows 64-127 of a tile
// come from the two weight matrices; silu(g) * u is re-packed hi/lo for the down projection),
// and a running argmax per token over lm_head rows (logits never leave the SM).
//
// Projections of hf2q 0.1.1 spec_decode/dflash/tensors.rs (`DFlashLayerTensors`: BF16
// row-major [out, in] weights, F32 activations) and models/qwen35/mtp.rs
// (`apply_linear_projection_f32`, `forward_shared_head`).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <stdlib.h>
#include <string.h>

#include <algorithm>
#include <atomic>

#include "df_internal.cuh"
#include "tc_ptx.cuh"

namespace df {

namespace {

constexpr int kThreads = 192;
constexpr int kBM = 128;
constexpr int kBK = 64;                    // BF16 elements per K block: one 128-byte row
constexpr int kABytes = kBM * kBK * 2;     // 16 KB
constexpr int kTokChunk = 8;               // tokens per TMEM load (16 columns)
// K blocks per pipeline stage when the weights are tiled: up to 4 (one 64 KB weight copy and one
// activation copy per stage) for up to 32 tokens, as many as leave two stages in the
// shared-memory budget. This
// part's TMA unit moves roughly one copy per ~0.4 us per SM whatever its size up to 64 KB, so a
// 16 KB weight tile per copy caps a CTA near 40 GB/s, below its share of HBM; 32-64 KB copies
// stream at the HBM rate.
constexpr int kTiledKpgMax = 4;
constexpr int kStageBudget = 200 * 1024;

struct TcParams {
    CUtensorMap amap[4];
    CUtensorMap bmap[2];
    CUtensorMap bmap3;       // tiled weights, K a multiple of 64: kpg K blocks' activations
    int b3;                  // 1: bmap3 is used (else one 2-D activation copy per K block)
    int n_seg;
    int seg_rows[4];
    int seg_tile0[5];
    int seg_col0[4];
    int k_seg;
    int kb_seg0;
    int kbt;
    int pair;
    int T, NC, acc_cols, alloc_cols;
    int n_tiles, G, stages;
    int splits;              // > 0: unit u = (tile u / splits, K split u % splits); 0: stream-K
    int n_units;
    size_t part_stride;      // split mode: output of split s starts at out + s * part_stride
    long long total_kb;
    uint32_t stage_bytes;
    uint32_t idesc;
    int epi;
    int N;
    float *out;
    int ldo;
    const float *resid;
    int ldr;
    uint16_t *pack_out;
    int ldpo;
    ArgTop *part;
    float *scratch;
    int *counters;
    int32_t *status;
    const float *rs_ss;
    int rs_n, rs_rows;
    float rs_inv_k, rs_eps;
    long long wait_cycles;   // limit of every barrier wait (kTimeoutCycles unless a test sets it)
    int withhold_first;      // test hook: the producer never loads its first stage
    const uint8_t *At;       // tiled weights (tile (m, kb) at (m * kbt + kb) * 16 KB) or null
    int kpg;                 // K blocks per pipeline stage (1 unless At is set)
};


__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// OR of a predicate over the 128 epilogue threads (named barrier 1).
__device__ __forceinline__ bool epi_any(bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, 1, 128, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)v)
        : "memory");
    return r != 0;
}

// ------------------------------------------------------------------ work split
__device__ __forceinline__ long long kb_start(long long c, const TcParams &p) {
    return c * p.total_kb / p.G;
}

__device__ __forceinline__ int cta_of(long long x, const TcParams &p) {
    return (int)(((x + 1) * (long long)p.G - 1) / p.total_kb);
}

// The segments (tile m, K blocks [k0, k1), split index) a CTA works on, in order. Stream-K:
// one contiguous range of the (tile, K block) space. Split mode: units blockIdx.x + i * G.
template <bool FIX>
struct Work {
    long long x, end;
    int u;
    __device__ __forceinline__ void init(const TcParams &p) {
        if constexpr (!FIX) {
            u = blockIdx.x;
        } else {
            x = kb_start(blockIdx.x, p);
            end = kb_start(blockIdx.x + 1, p);
        }
    }
    __device__ __forceinline__ bool next(const TcParams &p, int &m, int &k0, int &k1, int &split) {
        if constexpr (!FIX) {
            if (u >= p.n_units) return false;
            m = u / p.splits;
            split = u - m * p.splits;
            k0 = split * p.kbt / p.splits;
            k1 = (split + 1) * p.kbt / p.splits;
            u += gridDim.x;
            return true;
        }
        if (x >= end) return false;
        m = (int)(x / p.kbt);
        k0 = (int)(x - (long long)m * p.kbt);
        k1 = (int)min((long long)p.kbt, end - (long long)m * p.kbt);
        split = 0;
        x = (long long)m * p.kbt + k1;
        return true;
    }
};

__device__ __forceinline__ int seg_of_tile(int m, const TcParams &p) {
    int s = 0;
    while (s + 1 < p.n_seg && m >= p.seg_tile0[s + 1]) ++s;
    return s;
}

// Output row and validity of tile row r.
__device__ __forceinline__ bool tile_row(const TcParams &p, int m, int r, int &n_out, int &s) {
    if (p.pair) {
        s = 0;
        n_out = m * 64 + (r & 63);
        return n_out < p.seg_rows[0];
    }
    s = seg_of_tile(m, p);
    int local = (m - p.seg_tile0[s]) * kBM + r;
    n_out = p.seg_col0[s] + local;
    return local < p.seg_rows[s];
}

// ------------------------------------------------------------------ epilogue
struct EpiSmem {
    float *xs;      // [128][kTokChunk]
    ArgTop *wst;    // [4][kTokChunk]
    ArgTop *st;     // [T]
    float *rs;      // [T] row scales (when rs_ss is set)
};

// Apply the epilogue op to tokens [t0, t0 + kTokChunk) of tile m for this thread's row r.
// Every epilogue thread calls this (the SwiGLU and argmax paths synchronise the 128 threads).
template <int EPI>
__device__ __forceinline__ void epi_apply(const TcParams &p, const EpiSmem &es, int m, int r,
                                          int q, int lane, int t0, const float (&y0)[kTokChunk],
                                          int split) {
    int n_out, s;
    const bool valid = tile_row(p, m, r, n_out, s);
    float y[kTokChunk];
#pragma unroll
    for (int i = 0; i < kTokChunk; ++i) y[i] = p.rs_ss ? y0[i] * es.rs[min(t0 + i, p.T - 1)] : y0[i];
    if constexpr (EPI == EPI_STORE || EPI == EPI_RESID) {
        if (valid) {
            float *out = p.out + (size_t)split * p.part_stride;
#pragma unroll
            for (int i = 0; i < kTokChunk; ++i) {
                int t = t0 + i;
                if (t < p.T) {
                    float v = y[i];
                    if constexpr (EPI == EPI_RESID) v += p.resid[(size_t)t * p.ldr + n_out];
                    out[(size_t)t * p.ldo + n_out] = v;
                }
            }
        }
    } else if constexpr (EPI == EPI_SWIGLU) {
#pragma unroll
        for (int i = 0; i < kTokChunk; ++i) es.xs[r * kTokChunk + i] = y[i];
        epi_bar();
        if (r < 64 && valid) {
#pragma unroll
            for (int i = 0; i < kTokChunk; ++i) {
                int t = t0 + i;
                if (t < p.T) {
                    float g = es.xs[r * kTokChunk + i];
                    float u = es.xs[(r + 64) * kTokChunk + i];
                    float act = g / (1.f + expf(-g)) * u;
                    uint16_t hi, lo;
                    split_hi_lo(act, hi, lo);
                    p.pack_out[(size_t)(2 * t) * p.ldpo + n_out] = hi;
                    p.pack_out[(size_t)(2 * t + 1) * p.ldpo + n_out] = lo;
                }
            }
        }
        epi_bar();
    } else {   // EPI_ARGMAX
#pragma unroll
        for (int i = 0; i < kTokChunk; ++i) {
            ArgTop a = valid ? ArgTop{y[i], n_out, -INFINITY} : argtop_empty(0x7fffffff);
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) {
                ArgTop b;
                b.v1 = __shfl_xor_sync(0xffffffffu, a.v1, o);
                b.i1 = __shfl_xor_sync(0xffffffffu, a.i1, o);
                b.v2 = __shfl_xor_sync(0xffffffffu, a.v2, o);
                a = argtop_merge(a, b);
            }
            if (lane == 0) es.wst[q * kTokChunk + i] = a;
        }
        epi_bar();
        const int tid = r;   // any distinct id in [0, 128)
        if (tid < kTokChunk && t0 + tid < p.T) {
            ArgTop acc = es.st[t0 + tid];
            for (int w = 0; w < 4; ++w) acc = argtop_merge(acc, es.wst[w * kTokChunk + tid]);
            es.st[t0 + tid] = acc;
        }
        epi_bar();
    }
}

// EPI: the epilogue; FIX: whether a tile may be shared by several CTAs (stream-K work split,
// partial tiles finished by the last CTA). Each launch runs one instantiation, so its code holds
// only the paths it executes: a projection runs for a few microseconds and its instructions are
// fetched cold, so code that is never taken still costs.
template <int EPI, bool FIX>
__global__ void __launch_bounds__(kThreads, 1) gemm_tc_kernel(const __grid_constant__ TcParams p) {
    DF_TRACE_KERNEL(TK_GEMM + 2 * EPI + (FIX ? 1 : 0));
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~uintptr_t(1023));
    uint8_t *stage_base = smem;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + (size_t)p.stages * p.stage_bytes);
    uint64_t *empty = full + p.stages;
    uint64_t *tfull = empty + p.stages;
    uint64_t *tempty = tfull + 2;
    uint64_t *drain = tempty + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    int *s_last = reinterpret_cast<int *>(tmem_slot + 2);
    EpiSmem es;
    es.xs = reinterpret_cast<float *>(tmem_slot + 4);
    es.wst = reinterpret_cast<ArgTop *>(es.xs + kBM * kTokChunk);
    es.st = es.wst + 4 * kTokChunk;
    es.rs = reinterpret_cast<float *>(es.st + p.T);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < p.stages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&tfull[b], 1);
            mbar_init(&tempty[b], 4);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, p.alloc_cols);
        tmem_relinquish();
    }
    if (warp >= 2) {
        for (int t = threadIdx.x - 64; t < p.T; t += 128) es.st[t] = argtop_empty(0x7fffffff);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;


    pdl_trigger();
    if (warp == 0) {
        if (lane == 0) {
            // Weights do not depend on earlier kernels: the first stages' weight tiles are
            // requested before waiting for the predecessor grid, activation tiles after.
            const uint64_t pol_w = policy_evict_first(), pol_x = policy_evict_last();
            // (tile, k-block) cursor: one TMA issue per k-block must stay far cheaper than the
            // ~700 cycles a 16 KB weight tile takes to stream into one SM.
            struct Cursor {
                Work<FIX> w;
                int m, kb, k1, split, s, row0;
                bool valid;
            };
            auto seg_setup = [&](Cursor &c) {
                c.s = p.pair ? 0 : seg_of_tile(c.m, p);
                c.row0 = p.pair ? c.m * 64 : (c.m - p.seg_tile0[c.s]) * kBM;
            };
            auto cursor_init = [&](Cursor &c) {
                c.w.init(p);
                c.valid = c.w.next(p, c.m, c.kb, c.k1, c.split);
                while (c.valid && c.kb >= c.k1) c.valid = c.w.next(p, c.m, c.kb, c.k1, c.split);
                if (c.valid) seg_setup(c);
            };
            // K blocks of the stage at the cursor: up to kpg, within the current segment
            auto group = [&](const Cursor &c) { return min(p.kpg, c.k1 - c.kb); };
            auto advance = [&](Cursor &c) {
                c.kb += group(c);
                if (c.kb < c.k1) return;
                do {
                    c.valid = c.w.next(p, c.m, c.kb, c.k1, c.split);
                } while (c.valid && c.kb >= c.k1);
                if (c.valid) seg_setup(c);
            };
            // Stage layout: the group's A tiles (16 KB each), then its B slices (NC rows each).
            auto stage_tx = [&](const Cursor &c) {
                // the 3-D activation box always holds kpg K blocks (past K they are zero)
                return (uint32_t)group(c) * kABytes +
                       (uint32_t)(p.b3 ? p.kpg : group(c)) * (uint32_t)(p.NC * 128);
            };
            auto load_a = [&](const Cursor &c, int stage) {
                uint8_t *a = stage_base + (size_t)stage * p.stage_bytes;
                if (p.At) {
                    const uint8_t *src = p.At + ((size_t)c.m * p.kbt + c.kb) * kABytes;
                    bulk_load(a, src, (uint32_t)group(c) * kABytes, &full[stage], pol_w);
                    return;
                }
                const int ks = (p.k_seg == 2 && c.kb >= p.kb_seg0) ? 1 : 0;
                const int kx = (ks ? c.kb - p.kb_seg0 : c.kb) * kBK;
                if (p.pair) {
                    tma_load_2d(a, &p.amap[0], &full[stage], kx, c.row0, pol_w);
                    tma_load_2d(a + kABytes / 2, &p.amap[1], &full[stage], kx, c.row0, pol_w);
                } else {
                    tma_load_2d(a, &p.amap[ks ? 1 : c.s], &full[stage], kx, c.row0, pol_w);
                }
            };
            auto load_b = [&](const Cursor &c, int stage) {
                uint8_t *b = stage_base + (size_t)stage * p.stage_bytes + (size_t)p.kpg * kABytes;
                if (p.b3) {
                    tma_load_3d(b, &p.bmap3, &full[stage], 0, 0, c.kb, pol_x);
                    return;
                }
                const int n = group(c);
                for (int j = 0; j < n; ++j) {
                    const int kb = c.kb + j;
                    const int ks = (p.k_seg == 2 && kb >= p.kb_seg0) ? 1 : 0;
                    const int kx = (ks ? kb - p.kb_seg0 : kb) * kBK;
                    tma_load_2d(b + (size_t)j * p.NC * 128, &p.bmap[ks], &full[stage], kx, 0, pol_x);
                }
            };
            // Weights do not depend on earlier kernels: the first stages' weight tiles are
            // requested before waiting for the predecessor grid, activation tiles after.
            Cursor cur;
            cursor_init(cur);
            int pre = 0;
            while (cur.valid && pre < p.stages) {
                if (!(p.withhold_first && pre == 0)) {
                    mbar_expect_tx(&full[pre], stage_tx(cur));
                    load_a(cur, pre);
                }
                advance(cur);
                ++pre;
            }
            pdl_wait();
            DF_TRACE_MARK(true, 11);
            {
                Cursor cb;
                cursor_init(cb);
                for (int i = 0; i < pre; ++i) {
                    if (!(p.withhold_first && i == 0)) load_b(cb, i);
                    advance(cb);
                }
            }
            int stage = pre % p.stages;
            uint32_t phase = (pre == p.stages) ? 1u : 0u;
            long long issued = pre;
            bool ok = true;
            while (cur.valid) {
                if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, p.status, p.wait_cycles)) {
                    ok = false;
                    break;
                }
                mbar_expect_tx(&full[stage], stage_tx(cur));
                load_a(cur, stage);
                load_b(cur, stage);
                advance(cur);
                ++issued;
                if (++stage == p.stages) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            (void)ok;
            {
                // Every load issued lands before the CTA can exit, whether or not the MMA warp
                // consumed it (the last use of each stage; a withheld first load was never
                // issued). In a normal run these have landed by the time the loop ends.
                long long first = issued > p.stages ? issued - p.stages : 0;
                for (long long j = first; j < issued; ++j) {
                    if (p.withhold_first && j == 0) continue;
                    mbar_drain(&full[j % p.stages], (uint32_t)((j / p.stages) & 1), p.wait_cycles);
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            int stage = 0, acc = 0;
            uint32_t phase = 0, aphase = 0;
            bool ok = true;
            Work<FIX> w;
            w.init(p);
            int m, k0, k1, split;
            while (ok && w.next(p, m, k0, k1, split)) {
                if (k0 >= k1) continue;
                if (!mbar_wait(&tempty[acc], aphase ^ 1u, abort_flag, p.status, p.wait_cycles))
                    break;
                tc_fence_after();
                const uint32_t d = tmem_base + (uint32_t)(acc * p.acc_cols);
                for (int kb = k0; kb < k1;) {
                    const int n = min(p.kpg, k1 - kb);
                    if (!mbar_wait(&full[stage], phase, abort_flag, p.status, p.wait_cycles)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_addr = smem_u32(stage_base + (size_t)stage * p.stage_bytes);
                    const uint32_t b_addr = a_addr + (uint32_t)(p.kpg * kABytes);
                    for (int j = 0; j < n; ++j) {
                        const uint64_t adesc = sw128_desc(a_addr + (uint32_t)(j * kABytes));
                        const uint64_t bdesc = sw128_desc(b_addr + (uint32_t)(j * p.NC * 128));
#pragma unroll
                        for (int k = 0; k < kBK / 16; ++k) {
                            // advance 16 BF16 (32 bytes) along K inside the swizzled 128-byte row
                            mma_bf16(d, adesc + (uint64_t)(2 * k), bdesc + (uint64_t)(2 * k), p.idesc,
                                     (kb > k0 || j > 0 || k > 0) ? 1u : 0u);
                        }
                    }
                    kb += n;
                    mma_commit(&empty[stage]);
                    if (++stage == p.stages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                mma_commit(&tfull[acc]);
                if (++acc == 2) {
                    acc = 0;
                    aphase ^= 1u;
                }
            }
            // Every MMA this thread issued has completed once the drain barrier flips.
            mma_commit(drain);
            mbar_drain(drain, 0, p.wait_cycles);
        }
    } else {
        pdl_wait();
        if (p.rs_ss) {
            for (int t = threadIdx.x - 64; t < p.T; t += 128) {
                float sc = 1.f;
                if (t < p.rs_rows) {
                    float acc = 0.f;
                    for (int j = 0; j < p.rs_n; ++j) acc += p.rs_ss[(size_t)t * p.rs_n + j];
                    sc = 1.f / sqrtf(acc * p.rs_inv_k + p.rs_eps);
                }
                es.rs[t] = sc;
            }
            epi_bar();
        }
        const int q = warp & 3;          // TMEM lane quadrant this warp may access
        const int r = q * 32 + lane;     // tile row of this thread
        int acc = 0;
        uint32_t aphase = 0;
        Work<FIX> w;
        w.init(p);
        int m, k0, k1, split;
        while (w.next(p, m, k0, k1, split)) {
            if (k0 >= k1) continue;
            const bool whole = !FIX || (k0 == 0 && k1 == p.kbt);
            const int slot = (!p.splits && kb_start(blockIdx.x, p) / p.kbt == m) ? 0 : 1;
            const bool got = mbar_wait(&tfull[acc], aphase, abort_flag, p.status, p.wait_cycles);
            if (epi_any(!got)) break;   // all four epilogue warps leave together
            DF_TRACE_MARK(threadIdx.x == 64, 12);
            tc_fence_after();
            const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * p.acc_cols);
            const int n_chunks = (p.T + kTokChunk - 1) / kTokChunk;
            float *slot_base = p.scratch + ((size_t)blockIdx.x * 2 + slot) * (size_t)p.T * kBM;
            for (int c = 0; c < n_chunks; ++c) {
                uint32_t v[16];
                tmem_ld16(taddr + (uint32_t)(c * 2 * kTokChunk), v);
                if (c == n_chunks - 1) {
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&tempty[acc]);
                }
                float y[kTokChunk];
#pragma unroll
                for (int i = 0; i < kTokChunk; ++i)
                    y[i] = __uint_as_float(v[2 * i]) + __uint_as_float(v[2 * i + 1]);
                if (whole) {
                    epi_apply<EPI>(p, es, m, r, q, lane, c * kTokChunk, y, split);
                } else if constexpr (FIX) {
#pragma unroll
                    for (int i = 0; i < kTokChunk; ++i) {
                        int t = c * kTokChunk + i;
                        if (t < p.T) slot_base[(size_t)t * kBM + r] = y[i];
                    }
                }
            }
            if (++acc == 2) {
                acc = 0;
                aphase ^= 1u;
            }
            if (FIX && !whole) {
                // Stream-K fixup: the last CTA of this tile sums the partials in CTA order.
                __threadfence();
                epi_bar();
                const long long lo = (long long)m * p.kbt, hi = lo + p.kbt - 1;
                const int c_lo = cta_of(lo, p), c_hi = cta_of(hi, p);
                if (r == 0) {
                    int prev = atomicAdd(&p.counters[m], 1);
                    *s_last = (prev == c_hi - c_lo) ? 1 : 0;
                }
                epi_bar();
                const int last = *s_last;
                epi_bar();
                if (last) {
                    __threadfence();
                    // Load every partial of a token chunk before summing them, in CTA order, so
                    // the reduction costs one L2 round trip per chunk rather than one per CTA.
                    constexpr int kMaxParts = 8;
                    for (int c = 0; c < n_chunks; ++c) {
                        float y[kTokChunk];
#pragma unroll
                        for (int i = 0; i < kTokChunk; ++i) y[i] = 0.f;
                        for (int cb = c_lo; cb <= c_hi; cb += kMaxParts) {
                            float v8[kMaxParts][kTokChunk];
#pragma unroll
                            for (int j = 0; j < kMaxParts; ++j) {
                                const int cc = cb + j;
                                const float *src = nullptr;
                                if (cc <= c_hi) {
                                    const int sl = (kb_start(cc, p) / p.kbt == m) ? 0 : 1;
                                    src = p.scratch + ((size_t)cc * 2 + sl) * (size_t)p.T * kBM;
                                }
#pragma unroll
                                for (int i = 0; i < kTokChunk; ++i) {
                                    const int t = c * kTokChunk + i;
                                    v8[j][i] = (src && t < p.T) ? __ldcg(src + (size_t)t * kBM + r) : 0.f;
                                }
                            }
#pragma unroll
                            for (int j = 0; j < kMaxParts; ++j)
#pragma unroll
                                for (int i = 0; i < kTokChunk; ++i) y[i] += v8[j][i];
                        }
                        epi_apply<EPI>(p, es, m, r, q, lane, c * kTokChunk, y, split);
                    }
                    if (r == 0) p.counters[m] = 0;
                }
            }
        }
        if constexpr (EPI == EPI_ARGMAX) {
            epi_bar();
            for (int t = threadIdx.x - 64; t < p.T; t += 128)
                p.part[(size_t)blockIdx.x * p.T + t] = es.st[t];
        }
        DF_TRACE_MARK(threadIdx.x == 64, 13);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, p.alloc_cols);
    }
}

// ------------------------------------------------------------------ host side
// 2-D BF16 map over rows x cols (row stride ld elements), box box_cols x box_rows, 128B swizzle.
int make_map(CUtensorMap *m, const void *base, uint64_t cols, uint64_t rows, uint64_t ld,
             uint32_t box_cols, uint32_t box_rows) {
    return make_tma_2d(m, base, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, cols, rows, ld, box_cols,
                       box_rows, CU_TENSOR_MAP_SWIZZLE_128B);
}

int ceil_div(long long a, long long b) { return (int)((a + b - 1) / b); }

// Failure-detection test hook (df_test_wait_hook): a shorter wait limit, and every CTA's first
// stage withheld so the MMA warp's wait runs out. Zero in normal use.
std::atomic<long long> g_hook_wait_cycles{0};
std::atomic<int> g_hook_withhold{0};

// The kernel parameters of one projection (at most kMaxTcTokens tokens) and its dynamic shared
// memory; launches nothing.
int build_params(const GemmArgs &a, const TcScratch &sc, TcParams &p, size_t &smem_out) {
    memset(&p, 0, sizeof(p));
    const int T = a.T;
    int NC = ((2 * T + 15) / 16) * 16;
    if (NC < 16) NC = 16;
    p.T = T;
    p.NC = NC;
    int alloc = 32;
    while (alloc < 2 * NC) alloc <<= 1;
    p.alloc_cols = alloc;
    p.acc_cols = alloc / 2;          // each accumulator starts on a power-of-two column
    p.pair = a.epi == EPI_SWIGLU;
    p.k_seg = a.Wk2 ? 2 : 1;
    const int K0 = a.Wk2 ? a.K1 : a.K;
    const int K1 = a.K - K0;
    p.kb_seg0 = ceil_div(K0, kBK);
    p.kbt = p.kb_seg0 + (a.Wk2 ? ceil_div(K1, kBK) : 0);
    // With tiled weights the A operands come by bulk copies: the row-major pointers only
    // describe the segments and no A tensor map is made.
    const bool maps = a.At == nullptr;
    if (p.pair) {
        p.n_seg = 1;
        p.seg_rows[0] = a.N;
        p.n_tiles = ceil_div(a.N, 64);
        if (maps) {
            DF_TRY(make_map(&p.amap[0], a.W0, a.K, a.N, a.K, kBK, 64));
            DF_TRY(make_map(&p.amap[1], a.W1, a.K, a.N, a.K, kBK, 64));
        }
    } else if (a.Wk2) {
        p.n_seg = 1;
        p.seg_rows[0] = a.n0;
        p.seg_tile0[0] = 0;
        p.seg_col0[0] = 0;
        p.n_tiles = ceil_div(a.n0, kBM);
        if (maps) {
            DF_TRY(make_map(&p.amap[0], a.W0, K0, a.n0, K0, kBK, kBM));
            DF_TRY(make_map(&p.amap[1], a.Wk2, K1, a.n0, K1, kBK, kBM));
        }
    } else {
        const uint16_t *W[4] = {a.W0, a.W1, a.W2, a.W3};
        const int rows[4] = {a.n0, a.n1, a.n2, a.n3};
        int tiles = 0, col = 0, ns = 0;
        for (int i = 0; i < 4; ++i) {
            if (rows[i] <= 0 || W[i] == nullptr) continue;
            p.seg_rows[ns] = rows[i];
            p.seg_tile0[ns] = tiles;
            p.seg_col0[ns] = col;
            if (maps) DF_TRY(make_map(&p.amap[ns], W[i], a.K, rows[i], a.K, kBK, kBM));
            tiles += ceil_div(rows[i], kBM);
            col += rows[i];
            ++ns;
        }
        p.n_seg = ns;
        p.n_tiles = tiles;
    }
    p.seg_tile0[p.n_seg] = p.n_tiles;
    DF_TRY(make_map(&p.bmap[0], a.X, K0, 2 * T, a.ldx, kBK, NC));
    if (a.Wk2) DF_TRY(make_map(&p.bmap[1], a.X2, K1, 2 * T, a.ldx2, kBK, NC));
    p.total_kb = (long long)p.n_tiles * p.kbt;
    if (a.defer) {
        // Uniform K splits of every tile, as many as fill the GPU once; no cross-CTA reduction.
        int S = std::max(1, sc.max_ctas / p.n_tiles);
        S = std::min(S, p.kbt);
        p.splits = S;
        p.n_units = p.n_tiles * S;
        p.part_stride = a.part_stride;
        p.G = std::min(sc.max_ctas, p.n_units);
    } else if (p.pair && p.n_tiles <= sc.max_ctas) {
        // SwiGLU with at most one tile per SM: whole tiles, epilogue in place.
        p.splits = 1;
        p.n_units = p.n_tiles;
        p.G = p.n_tiles;
    } else {
        p.G = (int)std::min<long long>(sc.max_ctas, p.total_kb);
    }
    p.At = a.At;
    p.kpg = 1;
    if (a.At) {
        if ((reinterpret_cast<uintptr_t>(a.At) & 1023u) != 0)
            return fail(DF_EINVAL, "tiled weights must be 1024-byte aligned (%p)", (const void *)a.At);
        const int per_kb = kABytes + NC * 128;
        // Grouped K blocks pay off while the activation slices are small (up to 32 tokens);
        // at 128 tokens each K block brings 32 KB of activations, and four single-K-block stages
        // measured faster than two stages of two (batch-8 round 1327 -> 1293 us).
        p.kpg = NC <= 64 ? kTiledKpgMax : 1;
        while (p.kpg > 1 && kStageBudget / (p.kpg * per_kb) < 2) --p.kpg;
        // the activations of kpg consecutive K blocks: dims (64 columns, 2T rows, K blocks) with
        // the K-block step of 128 bytes, so one box lands as kpg swizzled NC-row slices. Only
        // with one activation matrix whose K is whole K blocks: this view has no column bound
        // inside a row, so a ragged last block would read past the row (there, and with a K
        // split, one 2-D copy per K block from its own map).
        p.b3 = (!a.Wk2 && K0 % kBK == 0) ? 1 : 0;
        if (p.b3)
            DF_TRY(make_tma_3d(&p.bmap3, a.X, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, kBK, 2 * T,
                               (uint64_t)(K0 / kBK), (uint64_t)a.ldx * 2, kBK * 2, kBK, NC,
                               p.kpg));
    }
    p.stage_bytes = (uint32_t)p.kpg * (kABytes + NC * 128);
    p.stages = std::min(a.At ? 5 : 8, (int)(kStageBudget / p.stage_bytes));
    if (p.stages < 2)
        return fail(DF_ESHAPE, "GEMM stage of %u bytes leaves fewer than two stages", p.stage_bytes);
    p.idesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(NC >> 3) << 17) |
              ((uint32_t)(kBM >> 4) << 24);
    p.epi = a.epi;
    p.N = a.N;
    p.out = a.out;
    p.ldo = a.ldo;
    p.resid = a.resid;
    p.ldr = a.ldr;
    p.pack_out = a.pack_out;
    p.ldpo = a.ldpo;
    p.part = a.part;
    p.scratch = sc.partials;
    p.counters = sc.counters;
    p.status = a.status;
    p.rs_ss = a.rs_ss;
    p.rs_n = a.rs_n;
    p.rs_rows = a.rs_rows;
    p.rs_inv_k = a.rs_inv_k;
    p.rs_eps = a.rs_eps;
    {
        const long long w = g_hook_wait_cycles.load(std::memory_order_relaxed);
        p.wait_cycles = w > 0 ? w : kTimeoutCycles;
        p.withhold_first = g_hook_withhold.load(std::memory_order_relaxed);
    }
    if (!p.splits && (size_t)p.G * 2 * T * kBM > sc.partial_floats)
        return fail(DF_EWORKSPACE, "GEMM scratch too small (%d tokens)", T);
    if (a.defer && (a.epi != EPI_STORE || a.part_stride < (size_t)T * a.ldo))
        return fail(DF_EINVAL, "deferred split-K needs a plain store into S x T x ldo floats");
    if (p.n_tiles > sc.n_counters)
        return fail(DF_EWORKSPACE, "GEMM tile counters too few (%d tiles)", p.n_tiles);
    smem_out = 1024 + (size_t)p.stages * p.stage_bytes + (2 * p.stages + 5) * 8 + 16 +
               (size_t)kBM * kTokChunk * 4 + 4 * kTokChunk * sizeof(ArgTop) +
               (size_t)T * sizeof(ArgTop) + (size_t)T * sizeof(float) + 64;
    return DF_OK;
}

// ------------------------------------------------------------------ tiled weights
struct TileArgs {
    const uint16_t *W[4];
    int rows[4];
    int tile0[5];
    int n_seg;
    const uint16_t *Wk2;     // K split: K blocks from kb_seg0 on read columns of Wk2
    int K0, K1, kb_seg0, kbt, pair, N, n_tiles;
    uint8_t *out;
};

// The A-operand tiles of a projection, with the segment, K-split and pairing rules of
// build_params: K blocks [0, kb_seg0) from the first K0 columns, the rest from Wk2.
int tile_plan(const GemmArgs &a, TileArgs &t) {
    memset(&t, 0, sizeof(t));
    if (a.N <= 0 || a.K <= 0) return fail(DF_ESHAPE, "tiled weights of an empty projection");
    t.pair = a.epi == EPI_SWIGLU;
    t.N = a.N;
    t.K0 = a.Wk2 ? a.K1 : a.K;
    t.K1 = a.K - t.K0;
    t.Wk2 = a.Wk2;
    t.kb_seg0 = ceil_div(t.K0, kBK);
    t.kbt = t.kb_seg0 + (a.Wk2 ? ceil_div(t.K1, kBK) : 0);
    if (t.pair) {
        t.n_seg = 2;
        t.W[0] = a.W0;
        t.W[1] = a.W1;
        t.rows[0] = t.rows[1] = a.N;
        t.n_tiles = ceil_div(a.N, 64);
    } else if (a.Wk2) {
        t.n_seg = 1;
        t.W[0] = a.W0;
        t.rows[0] = a.n0;
        t.n_tiles = ceil_div(a.n0, kBM);
    } else {
        const uint16_t *W[4] = {a.W0, a.W1, a.W2, a.W3};
        const int rows[4] = {a.n0, a.n1, a.n2, a.n3};
        for (int i = 0; i < 4; ++i) {
            if (rows[i] <= 0 || W[i] == nullptr) continue;
            t.W[t.n_seg] = W[i];
            t.rows[t.n_seg] = rows[i];
            t.tile0[t.n_seg] = t.n_tiles;
            t.n_tiles += ceil_div(rows[i], kBM);
            ++t.n_seg;
        }
    }
    t.tile0[t.n_seg] = t.n_tiles;
    if (t.n_tiles <= 0) return fail(DF_ESHAPE, "tiled weights of an empty projection");
    return DF_OK;
}

// One thread per 16-byte piece of the tiled copy: piece j of row r of tile (m, kb) holds
// columns kb*64 + 8j .. +7 of the row's source and lands at (j ^ (r % 8)) * 16 in the row.
__global__ void __launch_bounds__(256) tile_weights_kernel(TileArgs t) {
    DF_TRACE_KERNEL(TK_TILE);
    pdl_trigger();
    pdl_wait();
    const long long total = (long long)t.n_tiles * t.kbt * 1024;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x) {
        const long long blk = i >> 10;
        const int r = (int)((i >> 3) & 127), j = (int)(i & 7);
        const int m = (int)(blk / t.kbt), kb = (int)(blk - (long long)m * t.kbt);
        const uint16_t *W = nullptr;
        long long row = 0;
        if (t.pair) {
            row = (long long)m * 64 + (r & 63);
            if (row < t.N) W = r < 64 ? t.W[0] : t.W[1];
        } else {
            int s = 0;
            while (s + 1 < t.n_seg && m >= t.tile0[s + 1]) ++s;
            row = (long long)(m - t.tile0[s]) * kBM + r;
            if (row < t.rows[s]) W = t.W[s];
        }
        int col, cols;
        if (t.Wk2 && kb >= t.kb_seg0) {
            if (W) W = t.Wk2;
            col = (kb - t.kb_seg0) * kBK + 8 * j;
            cols = t.K1;
        } else {
            col = kb * kBK + 8 * j;
            cols = t.K0;
        }
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (W && col < cols) {
            const uint16_t *src = W + row * cols + col;
            if (col + 8 <= cols && (reinterpret_cast<uintptr_t>(src) & 15u) == 0) {
                v = *reinterpret_cast<const uint4 *>(src);
            } else {
                uint32_t w[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const uint32_t lo = col + 2 * q < cols ? src[2 * q] : 0u;
                    const uint32_t hi = col + 2 * q + 1 < cols ? src[2 * q + 1] : 0u;
                    w[q] = lo | (hi << 16);
                }
                v = make_uint4(w[0], w[1], w[2], w[3]);
            }
        }
        *reinterpret_cast<uint4 *>(t.out + blk * kABytes + r * 128 + ((j ^ (r & 7)) << 4)) = v;
    }
}

int launch_chunk(const GemmArgs &a, const TcScratch &sc, cudaStream_t s, int *G_out) {
    TcParams p;
    size_t smem = 0;
    DF_TRY(build_params(a, sc, p, smem));
    if (G_out) *G_out = a.defer ? p.splits : p.G;
    const dim3 grid(p.G), block(kThreads);
    const bool fix = p.splits == 0;
    switch (a.epi) {
        case EPI_STORE:
            return fix ? launch_k(a.name, gemm_tc_kernel<EPI_STORE, true>, grid, block, smem, s, p)
                       : launch_k(a.name, gemm_tc_kernel<EPI_STORE, false>, grid, block, smem, s, p);
        case EPI_RESID:
            return fix ? launch_k(a.name, gemm_tc_kernel<EPI_RESID, true>, grid, block, smem, s, p)
                       : launch_k(a.name, gemm_tc_kernel<EPI_RESID, false>, grid, block, smem, s, p);
        case EPI_SWIGLU:
            return fix ? launch_k(a.name, gemm_tc_kernel<EPI_SWIGLU, true>, grid, block, smem, s, p)
                       : launch_k(a.name, gemm_tc_kernel<EPI_SWIGLU, false>, grid, block, smem, s, p);
        case EPI_ARGMAX:
            return fix ? launch_k(a.name, gemm_tc_kernel<EPI_ARGMAX, true>, grid, block, smem, s, p)
                       : launch_k(a.name, gemm_tc_kernel<EPI_ARGMAX, false>, grid, block, smem, s, p);
        default:
            return fail(DF_EINVAL, "unknown projection epilogue %d", a.epi);
    }
}

}  // namespace

size_t tiled_projection_bytes(const GemmArgs &a) {
    TileArgs t;
    if (tile_plan(a, t) != DF_OK) return 0;
    return (size_t)t.n_tiles * t.kbt * kABytes;
}

int tile_projection(const GemmArgs &a, uint8_t *out, size_t out_bytes, cudaStream_t s) {
    TileArgs t;
    DF_TRY(tile_plan(a, t));
    const size_t need = (size_t)t.n_tiles * t.kbt * kABytes;
    if (out == nullptr || out_bytes < need)
        return fail(DF_EWORKSPACE, "tiled weights need %zu bytes, have %zu", need, out_bytes);
    if ((reinterpret_cast<uintptr_t>(out) & 1023u) != 0)
        return fail(DF_EINVAL, "tiled weights must be 1024-byte aligned (%p)", (void *)out);
    for (int i = 0; i < t.n_seg; ++i)
        if (t.W[i] == nullptr) return fail(DF_EINVAL, "tiled weights: NULL weight segment");
    t.out = out;
    const long long total = (long long)t.n_tiles * t.kbt * 1024;
    const long long grid = std::min<long long>((total + 255) / 256, 16LL * sm_count());
    return launch_k("tile_weights_kernel", tile_weights_kernel, dim3((unsigned)grid), dim3(256), 0, s,
                    t);
}

int launch_gemm_tc(const GemmArgs &a, const TcScratch &sc, cudaStream_t s, int *n_partials_out) {
    if (a.N <= 0 || a.T <= 0) {
        if (n_partials_out) *n_partials_out = 0;
        return DF_OK;
    }
    if (a.T <= kMaxTcTokens) return launch_chunk(a, sc, s, n_partials_out);
    if (a.epi == EPI_ARGMAX) return fail(DF_ESHAPE, "argmax over more than %d rows", kMaxTcTokens);
    for (int t0 = 0; t0 < a.T; t0 += kMaxTcTokens) {
        GemmArgs c = a;
        c.T = std::min(kMaxTcTokens, a.T - t0);
        c.X = a.X + (size_t)2 * t0 * a.ldx;
        if (a.X2) c.X2 = a.X2 + (size_t)2 * t0 * a.ldx2;
        if (a.out) c.out = a.out + (size_t)t0 * a.ldo;
        if (a.resid) c.resid = a.resid + (size_t)t0 * a.ldr;
        if (a.pack_out) c.pack_out = a.pack_out + (size_t)2 * t0 * a.ldpo;
        if (a.rs_ss) {
            c.rs_ss = a.rs_ss + (size_t)t0 * a.rs_n;
            c.rs_rows = std::max(0, a.rs_rows - t0);
        }
        DF_TRY(launch_chunk(c, sc, s, n_partials_out));
    }
    return DF_OK;
}

namespace {
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

int get_encode() {
    if (g_encode) return DF_OK;
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                     cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || fn == nullptr)
        return fail(DF_ECUDA, "cuTensorMapEncodeTiled unavailable: %s", cudaGetErrorString(e));
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    return DF_OK;
}
}  // namespace

}  // namespace df

extern "C" int df_test_wait_hook(long long wait_cycles, int withhold_first) {
    if (wait_cycles < 0 || (withhold_first && wait_cycles == 0))
        return df::fail(DF_EINVAL, "df_test_wait_hook: wait_cycles=%lld withhold_first=%d "
                                   "(withholding needs a positive wait limit)",
                        wait_cycles, withhold_first);
    df::g_hook_wait_cycles.store(wait_cycles, std::memory_order_relaxed);
    df::g_hook_withhold.store(withhold_first ? 1 : 0, std::memory_order_relaxed);
    return DF_OK;
}

namespace df {

int make_tma_3d(CUtensorMap *m, const void *base, CUtensorMapDataType dt, int elem_bytes,
                uint64_t d0, uint64_t d1, uint64_t d2, uint64_t stride1, uint64_t stride2,
                uint32_t b0, uint32_t b1, uint32_t b2) {
    DF_TRY(get_encode());
    if ((reinterpret_cast<uintptr_t>(base) & 15u) != 0 || stride1 % 16 != 0 || stride2 % 16 != 0 ||
        b0 * elem_bytes > 128)
        return fail(DF_EINVAL, "3-D TMA operand misaligned (base %p, strides %llu / %llu)", base,
                    (unsigned long long)stride1, (unsigned long long)stride2);
    cuuint64_t dims[3] = {d0, d1, d2};
    cuuint64_t strides[2] = {stride1, stride2};
    cuuint32_t box[3] = {b0, b1, b2};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = g_encode(m, dt, 3, const_cast<void *>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(DF_ECUDA, "cuTensorMapEncodeTiled (3-D) failed (%d)", (int)r);
    return DF_OK;
}

int make_tma_2d(CUtensorMap *m, const void *base, CUtensorMapDataType dt, int elem_bytes,
                uint64_t cols, uint64_t rows, uint64_t ld, uint32_t box_cols, uint32_t box_rows,
                CUtensorMapSwizzle swizzle) {
    DF_TRY(get_encode());
    if ((reinterpret_cast<uintptr_t>(base) & 15u) != 0 || (ld * elem_bytes) % 16 != 0)
        return fail(DF_EINVAL, "TMA operand misaligned (base %p, row stride %llu elements)", base,
                    (unsigned long long)ld);
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {ld * (uint64_t)elem_bytes};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(m, dt, 2, const_cast<void *>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(DF_ECUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    return DF_OK;
}

}  // namespace df

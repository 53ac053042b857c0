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
// Each 128-key x 128-dim piece of K or V (a "unit") lands in shared memory by TMA. A K unit
// comes with the 128-byte swizzle (F32: four 32-column groups, BF16: two 64-column groups)
// group by group (each group's 128 rows as one box), so a thread reading one key row touches
// every bank once. A V unit of head_dim 128 is 128 whole cache rows, one contiguous run: one
// bulk copy, landing as copied (a warp reading one dim of 32 keys reads consecutive words);
// for head_dim 256 each 128-wide half comes row by row with the swizzle. The sixteen converting warps turn a unit
// into a BF16 operand in tensor memory (TMEM), where the MMA reads it as its A matrix:
//   scores  S^T [128 keys x NP rows]  = K [128 x d] . Q^T          (A = K: lane = key)
//   output  O^T [128 dims x NP rows] += V^T [128 x 128 keys] . P^T  (A = V^T: lane = dim)
// An F32 cache is split into hi = bf16(x) and lo = bf16(x - hi) (about 16 mantissa bits). Q and
// P sit in shared memory as one operand of 2*NP rows, their hi rows stacked on their lo rows, so
// one MMA with N = 2*NP per operand half and 16-wide K step (two for an F32 cache, one for BF16)
// yields x.hi products in accumulator columns [0, NP) and x.lo products in [NP, 2NP); the two are
// added when the accumulator is read (hi.hi + hi.lo + lo.hi + lo.lo). The converted operand
// never goes back to shared memory, and the staging buffer is free for the next TMA load as soon
// as the warps have read it. Chunks of at most two tiles of an F32 cache with head_dim 128 (the
// VS instantiation) keep V^T in shared memory instead: each V unit is split in place in its
// staging buffer and read by the MMA through a shared-memory descriptor, which leaves TMEM to the
// K units and lets the V units of old cache rows be prepared before the wait too.
//
// A chunk of one or two tiles keeps all its scores in TMEM (256 columns hold the converted
// operands, the rest the scores and the output), so its softmax maximum is exact: pass 1 takes
// the row maxima, pass 2 turns each tile into probabilities (BF16 hi/lo in shared memory). The
// first V units (as many as there are operand regions) are converted before the softmax, while
// the score MMAs finish; the rest right after their tile's probabilities. Longer chunks stream
// tile by tile (ST below).
//
// 576 threads: warps 0-15 convert, run the softmax and read out (warps w, w + 4, w + 8, w + 12
// share TMEM lane quarter w % 4 and take one quarter of the columns, rows or keys); warp 16
// issues the MMAs; thread 0 issues the first TMA loads and warp 17 the others, each once every
// converting warp has arrived on its buffer's "read" barrier (an issue can wait for room in the
// copy engine; here that wait is off the converting warps' path). VS keeps thread 0 issuing its
// few loads. Block rows (keys past the cache rows) come from kb/vb with plain loads during the
// conversion; keys past the chunk are converted as zeros.
#include <cuda_bf16.h>
#include <string.h>

#include "df_internal.cuh"
#include "tc_ptx.cuh"

namespace df {

namespace {

constexpr int kGroups = 4;                    // converting warps per TMEM lane quarter
constexpr int kConvThreads = 128 * kGroups;   // warps 0-15: convert, softmax, read-out
constexpr int kTcThreads = kConvThreads + 64;  // warp 16: MMA issue; warp 17: TMA issue
constexpr int kDT = 128 / kGroups;            // K values of a unit row per converting thread
constexpr int kTcKeys = 128;                  // keys per tile
constexpr int kTmemCols = 512;
constexpr int kACols = 256;                   // TMEM columns of the converted A operands
constexpr int kF32Unit = 128 * 128 * 4;       // one staged F32 unit: 64 KB
constexpr int kBoxBytes = 128 * 128;          // one 128-byte-wide column box of 128 rows

// VS: no separate second P buffer (it takes the staging buffer of K unit 1).
template <int D, int NP, int NBUF, bool VS = false>
constexpr size_t attn_tc_smem_bytes() {
    return 1024 + (size_t)NBUF * kF32Unit + (D / 128) * 2 * (size_t)NP * 256 +
           (VS ? 0 : 2 * (size_t)NP * 256) + 9 * NP * 4 + 32 * 8 + 16;
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

// Two F32 values (lower K index first) -> one word of BF16 hi halves and one of lo halves.
__device__ __forceinline__ void split2(float x0, float x1, uint32_t &hi, uint32_t &lo) {
    const __nv_bfloat162 hb = __floats2bfloat162_rn(x0, x1);
    const float2 hf = __bfloat1622float2(hb);
    const __nv_bfloat162 lb = __floats2bfloat162_rn(x0 - hf.x, x1 - hf.y);
    hi = *reinterpret_cast<const uint32_t *>(&hb);
    lo = *reinterpret_cast<const uint32_t *>(&lb);
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, const uint4 &v) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w)
                 : "memory");
}

__device__ __forceinline__ void st_shared_u16(uint32_t addr, uint16_t v) {
    asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr), "h"(v) : "memory");
}

// Barrier of the converting warps (named barrier 1; the MMA and TMA warps do not take part).
__device__ __forceinline__ void conv_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(kConvThreads) : "memory");
}

// The same barrier, returning whether p holds in any converting thread.
__device__ __forceinline__ bool conv_sync_or(bool p) {
    uint32_t r;
    asm volatile(
        "{\n .reg .pred a, b;\n setp.ne.u32 a, %1, 0;\n barrier.cta.red.or.pred b, 1, %2, a;\n"
        " selp.u32 %0, 1, 0, b;\n}\n"
        : "=r"(r)
        : "r"((uint32_t)p), "n"(kConvThreads)
        : "memory");
    return r != 0;
}

template <int NPH>
__device__ __forceinline__ void tmem_rows(uint32_t taddr, float (&v)[NPH]) {
    if constexpr (NPH == 4) {
        uint32_t r[4];
        asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%4];"
                     : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                     : "r"(taddr));
        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
        for (int i = 0; i < 4; ++i) v[i] = __uint_as_float(r[i]);
    } else if constexpr (NPH == 16) {
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

// Reduce N per-lane values over the warp's 32 lanes with N-1+5-log2(N) shuffles (halving the
// values each step instead of reducing each one separately). Returns the reduction of value
// `row` (see below) in every lane; lanes that share a row get the same value. MAX: max, else sum.
template <int N, bool MAX>
__device__ __forceinline__ float lane_reduce_rows(float (&v)[N], int lane, int &row) {
    row = 0;
#pragma unroll
    for (int n = N, o = 16; n > 1; n >>= 1, o >>= 1) {
        const bool up = (lane & o) != 0;
#pragma unroll
        for (int i = 0; i < n / 2; ++i) {
            const float keep = up ? v[i + n / 2] : v[i];
            const float send = up ? v[i] : v[i + n / 2];
            const float got = __shfl_xor_sync(0xffffffffu, send, o);
            v[i] = MAX ? fmaxf(keep, got) : keep + got;
        }
        if (up) row += n / 2;
    }
    float r = v[0];
#pragma unroll
    for (int o = 32 / N / 2; o >= 1; o >>= 1) {
        const float got = __shfl_xor_sync(0xffffffffu, r, o);
        r = MAX ? fmaxf(r, got) : r + got;
    }
    return r;
}

// tcgen05.ld of NPH columns without the wait, so several loads share one tcgen05.wait::ld.
template <int NPH>
__device__ __forceinline__ void tmem_ld_nowait(uint32_t taddr, uint32_t (&r)[NPH]) {
    if constexpr (NPH == 4) {
        asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%4];"
                     : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                     : "r"(taddr));
    } else if constexpr (NPH == 8) {
        asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                     : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                       "=r"(r[6]), "=r"(r[7])
                     : "r"(taddr));
    } else {
        static_assert(NPH == 16, "rows per thread");
        asm volatile(
            "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
            "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
            : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
              "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
              "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
            : "r"(taddr));
    }
}

__device__ __forceinline__ void tmem_ld_wait() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

struct AttnTcParams {
    // F32 or BF16 [B * nkv * cap rows, d cols]. kmap views it as (column in group, row, group):
    // one box of 128 rows x all the groups of a unit lands as the groups' 128-row boxes one after
    // another. vmap (head_dim 256) views it as (column in group, group, row): the box lands
    // row-major.
    CUtensorMap kmap, vmap;
    AttnArgs a;
};

// KVB: the cache holds BF16 (no lo half: two MMAs per K step, and twice as many half-size
// staging buffers in the same shared memory).
// ST: chunks longer than two tiles, streamed tile by tile (no
// passes): units in the order K0, K1, V0, K2, V1, ..., so the score MMAs of tile t + 1 run while
// the warps take the softmax of tile t; scores alternate between two TMEM buffers; the output
// accumulator stays in TMEM across the tiles with a lazily moved reference maximum per row (it is
// raised, and the accumulator and row sums rescaled, only when a tile's maximum exceeds it by more
// than 2^8, so the probabilities stay below 2^8 and no tile waits for a rescale in the usual
// case); (o, m, l) are then the partials of the chunk against that reference.
// VS: chunks of at most two tiles of an F32 cache with head_dim 128, three staging buffers. Each
// V unit is converted in place in its staging buffer into V^T as a K-major BF16 operand in shared
// memory (hi in the first 32 KB, lo in the second), which the P.V MMAs read directly. K unit t
// lands in buffer t, V unit 0 in buffer 2 (requested with the K units) and V unit 1 in buffer 0
// once K unit 0 is in TMEM. With the TMEM regions left to the K units, the V units of tiles that
// predate the round are converted before the wait as well, and after it only q, the scores, the
// softmax and the products remain (plus the units of tiles holding new rows).
template <int D, int NP, int NBUF, bool KVB, bool VS, bool ST = false>
__global__ void __launch_bounds__(kTcThreads, 1) attn_tc_kernel(const __grid_constant__ AttnTcParams P) {
    DF_TRACE_KERNEL(TK_ATTN_TC);
    static_assert(!VS || (D == 128 && NBUF == 3 && !KVB), "in-place V operands");
    static_assert(!ST || !VS, "streamed tiles");
    constexpr int NB = KVB ? 2 * NBUF : NBUF;            // staging buffers
    constexpr int kUnit = KVB ? kF32Unit / 2 : kF32Unit;  // bytes of one staged unit
    constexpr int kBoxes = kUnit / kBoxBytes;             // TMA boxes per unit
    constexpr int kBoxCols = 128 / kBoxes;                // elements per box row
    constexpr int kUCols = KVB ? 64 : 128;                // TMEM columns of one converted unit
    constexpr int NA = kACols / kUCols;                   // converted-operand regions
    constexpr int NH = D / 128;                           // 128-wide halves of the head dim
    constexpr int NPH = NP / kGroups;         // rows per thread in the softmax and read-out
    constexpr int kQBytes = NP * 256;         // NP rows x 128 BF16 (the hi or the lo rows)
    constexpr int NS = 2 * NP;                // MMA N: hi rows 0..NP-1 stacked on lo rows
    // Unit conversion loops: a streamed chunk converts many units, so its loops are unrolled
    // fully (more loads in flight per thread); the short forms convert a few units each and keep
    // their code small (it is fetched cold).
    constexpr int kConvUnroll = ST ? 4 : 2;
    const AttnArgs &a = P.a;
    extern __shared__ uint8_t sm_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(sm_raw) + 1023) &
                                              ~uintptr_t(1023));
    uint8_t *stg = sm;                                  // NB staging buffers
    uint8_t *qsm = sm + NB * kUnit;                     // [NH] stacked hi/lo Q operands
    uint8_t *psm = qsm + NH * 2 * kQBytes;              // stacked hi/lo P operand (second buffer)
    float *red = reinterpret_cast<float *>(psm + (VS ? 0 : 2 * kQBytes));   // [4][NP] maxima, [4][NP] sums
    float *mrun = red + 8 * NP;                                  // [NP] row maxima of the partials
    uint64_t *full = reinterpret_cast<uint64_t *>(mrun + NP);    // [NB] staging landed
    uint64_t *aready = full + NB;     // [NA] region converted (8 warp arrivals)
    uint64_t *afree = aready + NA;    // [NA] MMAs reading the region done
    uint64_t *sdone = afree + NA;     // one pass: every score MMA of the chunk done
    uint64_t *pready = sdone + 1;     // [2] P operand written (8 warp arrivals)
    uint64_t *pfree = pready + 2;     // [2] P.V MMAs reading the P buffer done
    uint64_t *odone = pfree + 2;      // every P.V MMA of the chunk done
    uint64_t *drain = odone + 1;      // every MMA issued has completed
    uint64_t *vready = drain + 1;     // [2] VS: V operand of tile t written (16 warp arrivals);
                                      // ST: score MMAs of the tiles t with t % 2 == i done
    uint64_t *bempty = vready + 2;    // [NB] staging buffer read by every converting warp (16
                                      // warp arrivals): the TMA warp may refill it
    uint32_t *tslot = reinterpret_cast<uint32_t *>(bempty + NB);
    int *abort_flag = reinterpret_cast<int *>(tslot + 1);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int chunk = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
    const size_t head_off = (size_t)b * a.nkv + g;
    const uint64_t pol = policy_evict_first();
    int nis[4] = {0, 0, 0, 0};   // VS: TMA loads issued into each staging buffer (thread 0)
    // V unit of cache rows [y, y + 128) (head_dim 128: one contiguous run of rows) by one bulk
    // copy, cut at the end of the cache; rows past it are never read (keys past the cache rows
    // come from the block rows or are zero). Other head dims: a 128-wide half through vmap.
    auto load_v = [&](uint8_t *dst, uint64_t *bar, long long y, int h) {
        if constexpr (D == 128) {
            constexpr uint32_t kRow = 128 * (KVB ? 2 : 4);
            const long long left = (long long)a.B * a.nkv * a.cap - y;
            const uint32_t bytes = (uint32_t)min(max(left, 0LL), 128LL) * kRow;
            mbar_expect_tx(bar, bytes);
            if (bytes) bulk_load(dst, reinterpret_cast<const uint8_t *>(a.cache_v) + (size_t)y * kRow, bytes, bar, pol);
        } else {
            mbar_expect_tx(bar, (uint32_t)kUnit);
            tma_load_3d(dst, &P.vmap, bar, 0, h * kBoxes, (int)y, pol);
        }
    };
    // VS: V rows [y, y + 128) of the cache into staging buffer bf (thread 0)
    auto stage_v = [&](int bf, int y) {
        load_v(stg + (size_t)bf * kUnit, &full[bf], y, 0);
        ++nis[bf & 3];
    };
    pdl_trigger();
    // Units 0 and 1 are the chunk's first K units (in every form): the K units of its first two
    // tiles when the head dim is 128 (one half per tile), both halves of its first tile when it
    // is 256. Rows
    // that predate this call do not depend on the preceding kernels, so when a unit's tile lies
    // below seq_len it is requested, and converted into its TMEM operand, before the wait: only
    // the score MMAs need q, which the preceding kernel writes.
    int n_early = 0;
    const long long c0e = (long long)chunk * a.chunk;
    if (a.early_kv) {
        const long long old = a.seq_len[b];
        auto tile_end = [&](int u) { return (long long)(u / NH + 1) * kTcKeys; };
        while (n_early < min(2, NB) && tile_end(n_early) <= a.chunk &&
               c0e + tile_end(n_early) <= old && c0e + tile_end(n_early) <= a.cap)
            ++n_early;
    }
    if (tid == 0) {
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&P.kmap)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&P.vmap)) : "memory");
        for (int i = 0; i < NB; ++i) mbar_init(&full[i], 1);
        for (int i = 0; i < NA; ++i) {
            mbar_init(&aready[i], kConvThreads / 32);
            mbar_init(&afree[i], 1);
        }
        mbar_init(sdone, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&pready[i], kConvThreads / 32);
            mbar_init(&pfree[i], 1);
        }
        mbar_init(odone, 1);
        mbar_init(drain, 1);
        if (VS)
            for (int i = 0; i < 2; ++i) mbar_init(&vready[i], kConvThreads / 32);
        if (ST)
            for (int i = 0; i < 2; ++i) mbar_init(&vready[i], 1);
        for (int i = 0; i < NB; ++i) mbar_init(&bempty[i], kConvThreads / 32);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        for (int t = 0; t < n_early; ++t) {
            uint8_t *dst = stg + (size_t)t * kUnit;
            mbar_expect_tx(&full[t], (uint32_t)kUnit);
            const int y = (int)(head_off * a.cap + c0e) + (t / NH) * kTcKeys;
            tma_load_3d(dst, &P.kmap, &full[t], 0, y, (t % NH) * kBoxes, pol);
            ++nis[t & 3];
        }
        if (VS && n_early > 0) stage_v(2, (int)(head_off * a.cap + c0e));   // V unit 0
    }
    if (warp == 0) {
        tmem_alloc(tslot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    const uint32_t acol = (uint32_t)(kTmemCols - kACols);             // converted operands
    const int lq = warp & 3, grp = warp >> 2;
    const uint32_t lane_addr = (uint32_t)(lq * 32) << 16;
    // VS: V unit of tile t, staged in buffer bf (phase ph) -> V^T hi/lo BF16 operand in place. The
    // thread's row is dim 32*lq + lane, its keys [32*grp, 32*grp + 32) of the tile: all its values
    // are read before the barrier, and written after it as 16-byte pieces of 8 keys. Keys from
    // s_cache on come from the block rows vb (below kend) or are zero.
    auto convert_vs = [&](int t, int bf, uint32_t ph, int kbase, int s_cache, int kend) {
        mbar_wait(&full[bf], ph, abort_flag, a.status);
        uint8_t *st = stg + (size_t)bf * kUnit;
        // V rows staged as copied (row kr at 512 * kr); the warp reads 32 consecutive dims
        const uint8_t *sb = st + (lq * 32 + lane) * 4;
        const int kr0 = 32 * grp;
        float v[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) v[e] = *reinterpret_cast<const float *>(sb + (kr0 + e) * 512);
        if (kbase + kr0 + 31 >= s_cache) {
            const float *blkp = a.vb + head_off * a.blk * (size_t)D + lq * 32 + lane;
#pragma unroll
            for (int e = 0; e < 32; ++e) {
                const int key = kbase + kr0 + e;
                if (key >= s_cache) v[e] = key < kend ? __ldcg(blkp + (size_t)(key - s_cache) * D) : 0.f;
            }
        }
        conv_sync();   // the whole unit is in registers: overwrite it
        const uint32_t o0 = smem_u32(st);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            uint32_t hw[4], lw[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) split2(v[8 * q + 2 * i], v[8 * q + 2 * i + 1], hw[i], lw[i]);
            const uint32_t o = o0 + sw_off(128, lq * 32 + lane, kr0 + 8 * q);
            st_shared_v4(o, make_uint4(hw[0], hw[1], hw[2], hw[3]));
            st_shared_v4(o + kUnit / 2, make_uint4(lw[0], lw[1], lw[2], lw[3]));
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&vready[t]);
    };
    if (n_early > 0 && warp < kConvThreads / 32) {
        // the early K units: all keys are cache rows; staged rows -> BF16 operand in region u
        for (int u = 0; u < n_early; ++u) {
            mbar_wait(&full[u], 0u, abort_flag, a.status);
            const uint8_t *st = stg + (size_t)u * kUnit;
            const uint32_t ta = tmem + lane_addr + acol + (uint32_t)(u * kUCols + (kDT / 2) * grp);
            const int kr = lq * 32 + lane;
#pragma unroll 2
            for (int it = 0; it < kDT / 8; ++it) {
                const int d0 = kDT * grp + 8 * it;
                uint32_t hw[4], lw[4];
                if constexpr (KVB) {
                    const uint4 w = *reinterpret_cast<const uint4 *>(
                        st + (d0 >> 6) * kBoxBytes + kr * 128 + ((((d0 & 63) >> 3) ^ (kr & 7)) << 4));
                    hw[0] = w.x; hw[1] = w.y; hw[2] = w.z; hw[3] = w.w;
                } else {
                    const uint8_t *row = st + (d0 >> 5) * kBoxBytes + kr * 128;
                    const int c = (d0 & 31) >> 2;
                    const float4 f0 = *reinterpret_cast<const float4 *>(row + ((c ^ (kr & 7)) << 4));
                    const float4 f1 = *reinterpret_cast<const float4 *>(row + (((c + 1) ^ (kr & 7)) << 4));
                    split2(f0.x, f0.y, hw[0], lw[0]);
                    split2(f0.z, f0.w, hw[1], lw[1]);
                    split2(f1.x, f1.y, hw[2], lw[2]);
                    split2(f1.z, f1.w, hw[3], lw[3]);
                }
                tmem_st4(ta + 4 * it, hw);
                if constexpr (!KVB) tmem_st4(ta + 64 + 4 * it, lw);
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&aready[u]);
                if constexpr (!VS) mbar_arrive(&bempty[u]);
            }
            if (VS && u == 0 && n_early == 2) {
                conv_sync();   // K unit 0 is read: buffer 0 takes V unit 1
                if (tid == 0) {
                    fence_proxy_async_smem();
                    stage_v(0, (int)(head_off * a.cap + c0e) + kTcKeys);
                }
            }
        }
        conv_sync();   // every converting warp is done with the early staging buffers
        if constexpr (VS) {
            // the V units of the same tiles, converted in place
            for (int t = 0; t < n_early; ++t) convert_vs(t, t ? 0 : 2, (uint32_t)t, 0, 0x7fffffff, 0);
        }
    }
    pdl_wait();
    DF_TRACE_MARK(tid == 0, 1);
    const int rep = a.nq / a.nkv;
    const int R = a.blk * rep;
    const int nn = a.n_new ? min(max(a.n_new[b], 0), a.n_new_max) : 0;
    const long long sc = (long long)a.seq_len[b] + nn + a.extra_rows;
    const int S_cache = (int)min(max(sc, 0LL), (long long)a.cap);
    const int S = S_cache + (a.kb ? a.blk : 0);
    const int c0 = min(S, chunk * a.chunk), c1 = min(S, c0 + a.chunk);
    const int n_tiles = (c1 - c0 + kTcKeys - 1) / kTcKeys;
    float *part = a.part + ((head_off * a.n_chunks + chunk) * (size_t)R) * (D + 2);
    if (n_tiles == 0) {
        for (int i = tid; i < R * (D + 2); i += kTcThreads) part[i] = (i % (D + 2)) == D ? -INFINITY : 0.f;
        if (warp == 0) tmem_dealloc(tmem, kTmemCols);
        return;
    }
    // One pass holds at most max_tp tiles of scores; longer chunks are streamed (ST).
    const int max_tp = (kTmemCols - kACols - NH * NS) / NS;
    if (!ST && (n_tiles > max_tp || (VS && n_tiles > 2))) {   // the host plans within bounds
        if (tid == 0) set_status(a.status, DF_ESHAPE);
        tc_fence_before();
        __syncthreads();
        if (warp == 0) {
            tc_fence_after();
            tmem_dealloc(tmem, kTmemCols);
        }
        for (int i = tid; i < R * (D + 2); i += kTcThreads) part[i] = (i % (D + 2)) == D ? -INFINITY : 0.f;
        return;
    }
    const int nU = 2 * n_tiles * NH;
    // Unit u: the chunk's K units (tile-major, then 128-wide half), then its V units (ST: below).
    struct UnitInfo {
        int t0, nt, v, t, h;
    };
    auto decode = [&](int u) -> UnitInfo {
        UnitInfo x;
        if constexpr (ST) {
            // slots K0, then per tile t: K(t + 1) when it exists, V(t); a slot is NH units, one
            // per 128-wide half of the head dim
            x.t0 = 0;
            x.nt = n_tiles;
            x.h = u % NH;
            const int sl = u / NH;
            const int t = (sl - 1) >> 1;
            if (sl == 0) {
                x.v = 0;
                x.t = 0;
            } else if (((sl - 1) & 1) == 0 && t + 1 < n_tiles) {
                x.v = 0;
                x.t = t + 1;
            } else {
                x.v = 1;
                x.t = t;
            }
            return x;
        }
        x.t0 = 0;
        x.nt = n_tiles;
        int local = u;
        x.v = local >= x.nt * NH;
        if (x.v) local -= x.nt * NH;
        x.t = x.t0 + local / NH;
        x.h = local % NH;
        return x;
    };
    // Unit u: K or V of tile t, 128-wide half h: one TMA copy of 128 rows x kBoxes column groups.
    auto issue = [&](int u) {
        const UnitInfo x = decode(u);
        const int bf = u % NB;
        uint8_t *dst = stg + (size_t)bf * kUnit;
        const int y = (int)(head_off * a.cap) + c0 + x.t * kTcKeys;
        if (x.v) {
            load_v(dst, &full[bf], y, x.h);
        } else {
            mbar_expect_tx(&full[bf], (uint32_t)kUnit);
            tma_load_3d(dst, &P.kmap, &full[bf], 0, y, x.h * kBoxes, pol);
        }
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
    // the early units' buffers are free again: the staging runs NB units ahead of them (the
    // first NB by thread 0 here, the others by the TMA warp)
    int issued = n_early;   // TMA units issued (thread 0)
    const int n_first = max(n_early, min(NB + n_early, nU));
    if (tid == 0) {
        if constexpr (VS) {
            // the units not requested before the wait: K units into buffers t, V unit 0 into
            // buffer 2, V unit 1 into buffer 0 when K unit 0 was converted before the wait
            for (int t = n_early; t < n_tiles; ++t) {
                issue(t);
                ++nis[t];
            }
            if (n_early == 0) stage_v(2, (int)(head_off * a.cap) + c0);
            if (n_early == 1 && n_tiles == 2) {
                fence_proxy_async_smem();
                stage_v(0, (int)(head_off * a.cap) + c0 + kTcKeys);
            }
        } else {
            if (n_early > 0) fence_proxy_async_smem();
            for (; issued < min(NB + n_early, nU); ++issued) issue(issued);
        }
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
            uint8_t *qh = qsm + h * 2 * kQBytes;
            st_shared_v4(smem_u32(qh + sw_off(NS, r, d & 127)), hi);
            st_shared_v4(smem_u32(qh + sw_off(NS, NP + r, d & 127)), lo);
        }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    DF_TRACE_MARK(tid == 0, 2);
    const uint32_t ocol = (uint32_t)(kTmemCols - kACols - NH * NS);   // O^T accumulators
    // P operand of tile t. One pass: two buffers in turn, buffer 0 reusing the Q operands' space
    // (every score MMA has completed before the first P is written), buffer 1 following it.
    // Streamed: Q stays live, so one buffer after the Q operands. VS: buffer 1 is the staging
    // buffer of K unit 1, read into TMEM before the score MMAs complete.
    auto p_idx = [&](int t) -> int { return ST ? 0 : (t & 1); };
    auto p_phase = [&](int t) -> uint32_t { return (uint32_t)((ST ? t : (t >> 1)) & 1); };
    auto p_buf = [&](int t) -> uint32_t {
        if (VS) return (t & 1) ? smem_u32(stg + kUnit) : smem_u32(qsm);
        return ST ? smem_u32(psm) : smem_u32(qsm) + (uint32_t)((t & 1) * 2 * kQBytes);
    };
    const uint32_t idesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(NS >> 3) << 17) |
                           ((uint32_t)(128 >> 4) << 24);

    if (warp == kConvThreads / 32) {
        // MMA issuer: the products of unit u once its operand is in TMEM (and, for a V unit,
        // once its tile's P is in shared memory); commits free the operand region, the P buffer,
        // and signal the end of the chunk's scores (streamed: of each tile's) and outputs.
        if (lane == 0 && VS) {
            // VS: the score MMAs of every tile (K operands in TMEM regions t), then the P.V MMAs
            // of tile t with V^T from its staging buffer (hi half, then lo half)
            bool ok = true;
            const uint32_t bq = smem_u32(qsm);
            for (int t = 0; t < n_tiles && ok; ++t) {
                if (!(ok = mbar_wait(&aready[t], 0u, abort_flag, a.status))) break;
                tc_fence_after();
                const uint32_t ahi = tmem + acol + (uint32_t)(t * kUCols), d = tmem + (uint32_t)(t * NS);
#pragma unroll 1
                for (int s = 0; s < 8; ++s) {
                    const uint32_t ob = (uint32_t)((s >> 2) * NS * 128 + (s & 3) * 32);
                    mma_bf16_ts(d, ahi + 8 * s, sw128_desc(bq + ob), idesc, s ? 1u : 0u);
                    mma_bf16_ts(d, ahi + 64 + 8 * s, sw128_desc(bq + ob), idesc, 1u);
                }
            }
            DF_TRACE_MARK(true, 7);
            if (ok) mma_commit(sdone);
            for (int t = 0; t < n_tiles && ok; ++t) {
                if (!(ok = mbar_wait(&vready[t], 0u, abort_flag, a.status) &&
                           mbar_wait(&pready[p_idx(t)], p_phase(t), abort_flag, a.status)))
                    break;
                tc_fence_after();
                const uint32_t vhi = smem_u32(stg + (size_t)(t ? 0 : 2) * kUnit), bp = p_buf(t);
                const uint32_t d = tmem + ocol;
#pragma unroll 1
                for (int s = 0; s < 8; ++s) {
                    // K step s: keys 16s.. = bytes 32*(s%4) of the 64-key block s/4 of each operand
                    const uint32_t ob = (uint32_t)((s >> 2) * NS * 128 + (s & 3) * 32);
                    const uint32_t oa = (uint32_t)((s >> 2) * 128 * 128 + (s & 3) * 32);
                    mma_bf16(d, sw128_desc(vhi + oa), sw128_desc(bp + ob), idesc, (t || s) ? 1u : 0u);
                    mma_bf16(d, sw128_desc(vhi + kUnit / 2 + oa), sw128_desc(bp + ob), idesc, 1u);
                }
            }
            if (ok) mma_commit(odone);
            mma_commit(drain);
            mbar_drain(drain, 0);
        } else if (lane == 0) {
            for (int u = 0; u < nU; ++u) {
                const UnitInfo x = decode(u);
                const int r = u % NA;
                if (!mbar_wait(&aready[r], (uint32_t)((u / NA) & 1), abort_flag, a.status)) break;
                if (x.v && x.h == 0 &&
                    !mbar_wait(&pready[p_idx(x.t)], p_phase(x.t), abort_flag, a.status))
                    break;
                tc_fence_after();
                const uint32_t ahi = tmem + acol + (uint32_t)(r * kUCols), alo = ahi + 64;
                uint32_t d, bhi;
                bool acc;
                if (!x.v) {
                    d = tmem + (uint32_t)((ST ? (x.t & 1) : (x.t - x.t0)) * NS);
                    bhi = smem_u32(qsm + x.h * 2 * kQBytes);
                    acc = x.h > 0;
                } else {
                    d = tmem + ocol + (uint32_t)(x.h * NS);
                    bhi = p_buf(x.t);
                    acc = x.t > x.t0;
                }
                // One MMA per operand half and K step against the stacked [hi; lo] rows: the
                // columns [0, NP) of d collect x.hi products, [NP, 2NP) x.lo products (their sum
                // is taken when d is read).
#pragma unroll 1
                for (int s = 0; s < 8; ++s) {
                    // K step s: columns 8s.. of the operand, bytes 32*(s%4) of 64-wide block s/4
                    const uint32_t ob = (uint32_t)((s >> 2) * NS * 128 + (s & 3) * 32);
                    mma_bf16_ts(d, ahi + 8 * s, sw128_desc(bhi + ob), idesc, (acc || s) ? 1u : 0u);
                    if constexpr (!KVB) mma_bf16_ts(d, alo + 8 * s, sw128_desc(bhi + ob), idesc, 1u);
                }
                mma_commit(&afree[r]);
                const bool last_of_tile = x.h == NH - 1;
                const bool last_of_chunk = last_of_tile && x.t == x.t0 + x.nt - 1;
                if (!x.v) {
                    if (ST) {
                        if (last_of_tile) mma_commit(&vready[x.t & 1]);
                    } else if (last_of_chunk) {
                        mma_commit(sdone);
                    }
                } else {
                    if (last_of_tile) mma_commit(&pfree[p_idx(x.t)]);
                    if (last_of_chunk) mma_commit(odone);
                }
            }
            // Every MMA this thread issued has completed once the drain barrier flips.
            mma_commit(drain);
            mbar_drain(drain, 0);
        }
        __syncwarp();
    } else if (warp == kConvThreads / 32 + 1) {
        // TMA issuer: the units after the first NB, each into its staging buffer once every
        // converting warp has read the unit before it there. Issuing here keeps a copy that
        // waits for room in the copy engine off the converting warps' path.
        if constexpr (!VS) {
            if (lane == 0) {
                int u = n_first;
                for (; u < nU; ++u) {
                    if (!mbar_wait(&bempty[u % NB], (uint32_t)(((u / NB) - 1) & 1), abort_flag, a.status))
                        break;
                    DF_TRACE_MARK(ST && u == 9, 14);
                    DF_TRACE_MARK(ST && u == 10, 15);
                    issue(u);
                    DF_TRACE_MARK(ST && u == 9, 6);
                    DF_TRACE_MARK(ST && u == 10, 10);
                }
                // after an abort: let every copy still in flight land before the CTA exits
                for (int j = max(0, u - NB); j < u; ++j) mbar_drain(&full[j % NB], (uint32_t)((j / NB) & 1));
            }
            __syncwarp();
        }
    } else {
        // Unit u -> BF16 operand in TMEM region u % NA. K unit: this thread's lane is key
        // 32*lq + lane, its columns the dims [kDT*grp, kDT*grp + kDT) of the unit. V unit: its
        // lane is dim 32*lq + lane, its columns the keys [kDT*grp, kDT*grp + kDT).
        auto convert = [&](int u) {
            const UnitInfo x = decode(u);
            const int bf = u % NB, r = u % NA;
            mbar_wait(&full[bf], (uint32_t)((u / NB) & 1), abort_flag, a.status);
            DF_TRACE_MARK(ST && tid == 0 && u == 9, 3);
            DF_TRACE_MARK(ST && tid == 0 && u == 10, 7);
            if (u >= NA) {
                mbar_wait(&afree[r], (uint32_t)(((u / NA) - 1) & 1), abort_flag, a.status);
                tc_fence_after();
            }
            DF_TRACE_MARK(ST && tid == 0 && u == 9, 4);
            DF_TRACE_MARK(ST && tid == 0 && u == 10, 8);
            const uint8_t *st = stg + (size_t)bf * kUnit;
            const int kbase = c0 + x.t * kTcKeys;
            const float *blkp = (x.v ? a.vb : a.kb) + head_off * a.blk * (size_t)D + x.h * 128;
            const uint32_t ta = tmem + lane_addr + acol + (uint32_t)(r * kUCols + (kDT / 2) * grp);
            // 8 K values per step: 4 hi words at ta + 4*it, 4 lo words at ta + 64 + 4*it. Loops,
            // not unrolled code, where a CTA converts only a few units (its instructions are
            // fetched cold and their number, not their issue rate, sets the time); unrolled when
            // streaming (kConvUnroll).
            if (VS || !x.v) {
                const int kr = lq * 32 + lane, key = kbase + kr;
                const bool cached = key < S_cache;
                const float *src = (!cached && key < c1) ? blkp + (size_t)(key - S_cache) * D + kDT * grp
                                                         : nullptr;
#pragma unroll kConvUnroll
                for (int it = 0; it < kDT / 8; ++it) {
                    const int d0 = kDT * grp + 8 * it;            // first of the step's 8 dims
                    uint32_t hw[4], lw[4];
                    float4 f0 = make_float4(0.f, 0.f, 0.f, 0.f), f1 = f0;
                    if (cached) {
                        if constexpr (KVB) {
                            const uint4 w = *reinterpret_cast<const uint4 *>(
                                st + (d0 >> 6) * kBoxBytes + kr * 128 + ((((d0 & 63) >> 3) ^ (kr & 7)) << 4));
                            hw[0] = w.x; hw[1] = w.y; hw[2] = w.z; hw[3] = w.w;
                        } else {
                            const uint8_t *row = st + (d0 >> 5) * kBoxBytes + kr * 128;
                            const int c = (d0 & 31) >> 2;
                            f0 = *reinterpret_cast<const float4 *>(row + ((c ^ (kr & 7)) << 4));
                            f1 = *reinterpret_cast<const float4 *>(row + (((c + 1) ^ (kr & 7)) << 4));
                        }
                    } else if (src) {
                        f0 = __ldcg(reinterpret_cast<const float4 *>(src) + 2 * it);
                        f1 = __ldcg(reinterpret_cast<const float4 *>(src) + 2 * it + 1);
                    }
                    if (!KVB || !cached) {
                        split2(f0.x, f0.y, hw[0], lw[0]);
                        split2(f0.z, f0.w, hw[1], lw[1]);
                        split2(f1.x, f1.y, hw[2], lw[2]);
                        split2(f1.z, f1.w, hw[3], lw[3]);
                    }
                    tmem_st4(ta + 4 * it, hw);
                    if constexpr (!KVB) tmem_st4(ta + 64 + 4 * it, lw);
                }
            } else if constexpr (!VS) {
                const int dd = lq * 32 + lane;                // dim within the 128-wide half
                const int col = dd % kBoxCols, gsel = dd / kBoxCols;
                // V rows staged row-major: key kr's column group gsel is 128-byte line
                // kBoxes * kr + gsel, swizzled by the line index
                const uint8_t *sb = st + gsel * 128;
                auto staged = [&](int kr, int k7) -> float {    // k7 = kr & 7, known statically
                    if constexpr (D == 128) {   // one bulk copy: row kr as copied, unswizzled
                        if constexpr (KVB) {
                            const uint16_t bits = *reinterpret_cast<const uint16_t *>(st + kr * 256 + dd * 2);
                            return __uint_as_float((uint32_t)bits << 16);
                        } else {
                            return *reinterpret_cast<const float *>(st + kr * 512 + dd * 4);
                        }
                    }
                    const int x = (kBoxes * k7 + gsel) & 7;
                    if constexpr (KVB) {
                        const uint16_t bits = *reinterpret_cast<const uint16_t *>(
                            sb + kr * (kBoxes * 128) + (((col >> 3) ^ x) << 4) + (col & 7) * 2);
                        return __uint_as_float((uint32_t)bits << 16);
                    } else {
                        return *reinterpret_cast<const float *>(
                            sb + kr * (kBoxes * 128) + (((col >> 2) ^ x) << 4) + (col & 3) * 4);
                    }
                };
#pragma unroll kConvUnroll
                for (int it = 0; it < kDT / 8; ++it) {
                    const int kr0 = kDT * grp + 8 * it;           // 8 keys, kr0 % 8 == 0
                    float v[8];
                    if (kbase + kr0 + 7 < S_cache) {
#pragma unroll
                        for (int e = 0; e < 8; ++e) v[e] = staged(kr0 + e, e);
                    } else {
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            const int key = kbase + kr0 + e;
                            float xv = 0.f;
                            if (key < S_cache) xv = staged(kr0 + e, e);
                            else if (key < c1) xv = __ldcg(blkp + (size_t)(key - S_cache) * D + dd);
                            v[e] = xv;
                        }
                    }
                    uint32_t hw[4], lw[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) split2(v[2 * i], v[2 * i + 1], hw[i], lw[i]);
                    tmem_st4(ta + 4 * it, hw);
                    if constexpr (!KVB) tmem_st4(ta + 64 + 4 * it, lw);
                }
            }
            tmem_wait_st();
            DF_TRACE_MARK(ST && tid == 0 && u == 9, 5);
            DF_TRACE_MARK(ST && tid == 0 && u == 10, 0);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&aready[r]);
            if constexpr (VS) {
                conv_sync();   // every warp has read the staging buffer: refill it
                if (tid == 0 && x.t == 0 && n_tiles == 2) {   // with V unit 1
                    fence_proxy_async_smem();
                    stage_v(0, (int)(head_off * a.cap) + c0 + kTcKeys);
                }
            } else {
                // this warp has read the staging buffer; the TMA warp refills it once all have
                if (lane == 0) mbar_arrive(&bempty[bf]);
            }
        };

        const float scale = 1.4426950408889634f / sqrtf((float)D);
        const int r0 = grp * NPH;
        auto row_ok = [&](int key, int row) {
            if (key >= c1 || row >= R) return false;
            return !(a.causal_block && key >= S_cache && key - S_cache > row / rep);
        };
        float Mrow[NPH], lsum[NPH];
#pragma unroll
        for (int r = 0; r < NPH; ++r) lsum[r] = 0.f;
        // Probabilities of one tile (this thread's rows' scores sv at key kt of the tile) against
        // the row references ref -> the BF16 hi/lo P operand at pb, two rows per packed
        // conversion (the roundings of one row at a time); adds them to the row sums.
        auto store_p = [&](uint32_t pb, int kt, int key, const float (&sv)[NPH], const float (&ref)[NPH]) {
            const uint32_t prow = pb + (uint32_t)((kt >> 6) * NS * 128 + ((kt & 7) << 1));
            const int kc = (kt & 63) >> 3;   // the key's 16-byte piece of a 128-byte row
#pragma unroll
            for (int r = 0; r < NPH; r += 2) {
                float pv[2];
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    pv[i] = 0.f;
                    if (row_ok(key, r0 + r + i) && ref[r + i] != -INFINITY) pv[i] = ex2(sv[r + i] * scale - ref[r + i]);
                    lsum[r + i] += pv[i];
                }
                uint32_t hw, lw;
                split2(pv[0], pv[1], hw, lw);
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    const int rr = r0 + r + i;   // (NP + rr) & 7 == rr & 7: NP is a multiple of 8
                    const uint32_t o = prow + (uint32_t)(rr * 128 + ((kc ^ (rr & 7)) << 4));
                    st_shared_u16(o, (uint16_t)(i ? hw >> 16 : hw & 0xffffu));
                    st_shared_u16(o + NP * 128, (uint16_t)(i ? lw >> 16 : lw & 0xffffu));
                }
            }
        };
        if (tid < NP) mrun[tid] = -INFINITY;

        // VS: softmax pass 1 over the chunk's nt tiles: exact row maxima into Mrow (the one-pass
        // loop below keeps its own copy, which compiles to fewer spills there)
        auto pass_max = [&](int nt) {
            mbar_wait(sdone, 0u, abort_flag, a.status);
            tc_fence_after();
            DF_TRACE_MARK(tid == 0, 6);
            float mx[NPH];
#pragma unroll
            for (int r = 0; r < NPH; ++r) mx[r] = -INFINITY;
            DF_TRACE_MARK(tid == kConvThreads - 32, 15);
            for (int tt = 0; tt < nt; ++tt) {
                uint32_t sh[NPH], sl[NPH];
                tmem_ld_nowait<NPH>(tmem + lane_addr + tt * NS + r0, sh);
                tmem_ld_nowait<NPH>(tmem + lane_addr + tt * NS + NP + r0, sl);
                tmem_ld_wait();
                DF_TRACE_MARK(tid == 0 && tt == 0, 10);
                const int key = c0 + tt * kTcKeys + lq * 32 + lane;
#pragma unroll
                for (int r = 0; r < NPH; ++r)
                    if (row_ok(key, r0 + r))
                        mx[r] = fmaxf(mx[r], (__uint_as_float(sh[r]) + __uint_as_float(sl[r])) * scale);
            }
            int row;
            const float m = lane_reduce_rows<NPH, true>(mx, lane, row);
            if ((lane & (32 / NPH - 1)) == 0) red[lq * NP + r0 + row] = m;
            DF_TRACE_MARK(tid == 0, 14);
            conv_sync();
#pragma unroll
            for (int r = 0; r < NPH; ++r)
                Mrow[r] = fmaxf(fmaxf(red[r0 + r], red[NP + r0 + r]),
                                fmaxf(red[2 * NP + r0 + r], red[3 * NP + r0 + r]));
        };
        // VS: pass 2 for tile t (0 or 1; each P buffer is written once): probabilities -> BF16
        // hi/lo P operand
        auto write_p = [&](int t) {
            float sv[NPH];
            {
                uint32_t sh[NPH], sl[NPH];
                tmem_ld_nowait<NPH>(tmem + lane_addr + t * NS + r0, sh);
                tmem_ld_nowait<NPH>(tmem + lane_addr + t * NS + NP + r0, sl);
                tmem_ld_wait();
                DF_TRACE_MARK(tid == 0 && t == 0, 0);
#pragma unroll
                for (int r = 0; r < NPH; ++r) sv[r] = __uint_as_float(sh[r]) + __uint_as_float(sl[r]);
            }
            const int kt = lq * 32 + lane;
            store_p(p_buf(t), kt, c0 + t * kTcKeys + kt, sv, Mrow);
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&pready[p_idx(t)]);
        };

        if constexpr (VS) {
            // one pass: the K units not converted early (each then passes its buffer on to the V
            // unit of its tile), those V units in place, the softmax, all P operands
            for (int t = n_early; t < n_tiles; ++t) convert(t);
            for (int t = n_early; t < n_tiles; ++t)
                convert_vs(t, t ? 0 : 2, (uint32_t)t, c0 + t * kTcKeys, S_cache, c1);
            pass_max(n_tiles);
            DF_TRACE_MARK(tid == 0, 3);
            for (int t = 0; t < n_tiles; ++t) {
                write_p(t);
                DF_TRACE_MARK(tid == 0 && t == 0, 8);
            }
            DF_TRACE_MARK(tid == 0, 4);
            mbar_wait(odone, 0u, abort_flag, a.status);
            tc_fence_after();
            DF_TRACE_MARK(tid == 0, 5);
        }
        if constexpr (ST) {
            constexpr float kTau = 8.f;   // log2 units: probabilities stay below 2^8
            float mref[NPH];
#pragma unroll
            for (int r = 0; r < NPH; ++r) mref[r] = -INFINITY;
            auto convert_slot = [&](int sl) {
#pragma unroll
                for (int h = 0; h < NH; ++h)
                    if (sl * NH + h >= n_early) convert(sl * NH + h);   // early units: done
            };
            convert_slot(0);                                       // K0
            for (int t = 0; t < n_tiles; ++t) {
                const bool more = t + 1 < n_tiles;
                DF_TRACE_MARK(tid == 0 && t == 4, 16);
                DF_TRACE_MARK(tid == 0 && t == 5, 23);
                if (more) convert_slot(2 * t + 1);                 // K(t + 1)
                DF_TRACE_MARK(tid == 0 && t == 4, 17);
                convert_slot(more ? 2 * t + 2 : 2 * t + 1);        // V(t)
                DF_TRACE_MARK(tid == 0 && t == 4, 18);
                // scores of tile t -> its row maxima (max over the four lane quarters)
                mbar_wait(&vready[t & 1], (uint32_t)((t >> 1) & 1), abort_flag, a.status);
                tc_fence_after();
                DF_TRACE_MARK(tid == 0 && t == 4, 19);
                float sv[NPH], mx[NPH];
                {
                    uint32_t sh[NPH], sl[NPH];
                    tmem_ld_nowait<NPH>(tmem + lane_addr + (t & 1) * NS + r0, sh);
                    tmem_ld_nowait<NPH>(tmem + lane_addr + (t & 1) * NS + NP + r0, sl);
                    tmem_ld_wait();
#pragma unroll
                    for (int r = 0; r < NPH; ++r) sv[r] = __uint_as_float(sh[r]) + __uint_as_float(sl[r]);
                }
                const int kt = lq * 32 + lane;
                const int key = c0 + t * kTcKeys + kt;
                // Does any score of the tile lie more than kTau above its row's reference (or give
                // a row its first one)? Only then are the rows' maxima gathered across the four
                // lane quarters; otherwise the reference stands and the tile needs no exchange.
                bool need = false;
#pragma unroll
                for (int r = 0; r < NPH; ++r) {
                    mx[r] = row_ok(key, r0 + r) ? sv[r] * scale : -INFINITY;
                    need |= mx[r] != -INFINITY && (mref[r] == -INFINITY || mx[r] > mref[r] + kTau);
                }
                const bool raise = conv_sync_or(need);   // the same in every converting warp
                DF_TRACE_MARK(tid == 0 && t == 4, 20);
                float mn[NPH];
                if (raise) {
                    int row;
                    const float m = lane_reduce_rows<NPH, true>(mx, lane, row);
                    float *rb = red + (t & 1) * 4 * NP;   // alternate: a fast warp may reach tile t + 1
                    if ((lane & (32 / NPH - 1)) == 0) rb[lq * NP + r0 + row] = m;
                    conv_sync();
#pragma unroll
                    for (int r = 0; r < NPH; ++r)
                        mn[r] = fmaxf(fmaxf(rb[r0 + r], rb[NP + r0 + r]), fmaxf(rb[2 * NP + r0 + r], rb[3 * NP + r0 + r]));
                }
                // the P.V MMAs of tile t - 1 are done: the P buffer and the accumulator are free
                if (t > 0) {
                    mbar_wait(&pfree[0], (uint32_t)((t - 1) & 1), abort_flag, a.status);
                    tc_fence_after();
                }
                DF_TRACE_MARK(tid == 0 && t == 4, 21);
                bool resc = false;   // the same for every lane: the warp's lanes share its rows
                if (raise) {
#pragma unroll
                    for (int r = 0; r < NPH; ++r) resc |= mref[r] != -INFINITY && mn[r] > mref[r] + kTau;
                }
                if (resc) {
                    float f[NPH];
#pragma unroll
                    for (int r = 0; r < NPH; ++r) {
                        f[r] = (mref[r] != -INFINITY && mn[r] > mref[r] + kTau) ? ex2(mref[r] - mn[r]) : 1.f;
                        lsum[r] *= f[r];
                    }
#pragma unroll
                    for (int h = 0; h < NH; ++h) {
                        const uint32_t oc = ocol + (uint32_t)(h * NS);
                        float oh[NPH], ol[NPH];
                        tmem_rows<NPH>(tmem + lane_addr + oc + r0, oh);
                        tmem_rows<NPH>(tmem + lane_addr + oc + NP + r0, ol);
                        uint32_t wh[NPH], wl[NPH];
#pragma unroll
                        for (int r = 0; r < NPH; ++r) {
                            wh[r] = __float_as_uint(oh[r] * f[r]);
                            wl[r] = __float_as_uint(ol[r] * f[r]);
                        }
#pragma unroll
                        for (int j = 0; j < NPH; j += 4) {
                            const uint32_t h4[4] = {wh[j], wh[j + 1], wh[j + 2], wh[j + 3]};
                            const uint32_t l4[4] = {wl[j], wl[j + 1], wl[j + 2], wl[j + 3]};
                            tmem_st4(tmem + lane_addr + oc + r0 + j, h4);
                            tmem_st4(tmem + lane_addr + oc + NP + r0 + j, l4);
                        }
                    }
                    tmem_wait_st();
                }
                if (raise) {
#pragma unroll
                    for (int r = 0; r < NPH; ++r)
                        if (mref[r] == -INFINITY || mn[r] > mref[r] + kTau) mref[r] = mn[r];
                }
                // probabilities of tile t against the reference -> BF16 hi/lo P operand
                store_p(p_buf(t), kt, key, sv, mref);
                fence_proxy_async_smem();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&pready[0]);
                DF_TRACE_MARK(tid == 0 && t == 4, 22);
            }
#pragma unroll
            for (int r = 0; r < NPH; ++r) Mrow[r] = mref[r];
            mbar_wait(odone, 0u, abort_flag, a.status);
            tc_fence_after();
            conv_sync();   // every warp has read the last tile's maxima: the read-out reuses red
        }
        // One pass (one or two tiles): the K units, then as many V units as there are operand
        // regions (their regions are freed by the score MMAs alone), then the softmax; the
        // probabilities of a tile are written before its first V unit that was not converted
        // ahead.
        if constexpr (!VS && !ST) {
            const int nt = n_tiles;
            const int nK = nt * NH, nV = nK, pre = min(NA, nV), pre_tiles = (pre + NH - 1) / NH;
            int pdone = 0;   // tiles whose P operand is written
            for (int i = 0; i <= nK + nV; ++i) {
                int want = pdone;
                if (i == nK + pre) {
                    // softmax pass 1: exact row maxima over the chunk's tiles
                    mbar_wait(sdone, 0u, abort_flag, a.status);
                    tc_fence_after();
                    float mx[NPH];
#pragma unroll
                    for (int r = 0; r < NPH; ++r) mx[r] = -INFINITY;
                    for (int tt = 0; tt < nt; ++tt) {
                        uint32_t sh[NPH], sl[NPH];
                        tmem_ld_nowait<NPH>(tmem + lane_addr + tt * NS + r0, sh);
                        tmem_ld_nowait<NPH>(tmem + lane_addr + tt * NS + NP + r0, sl);
                        tmem_ld_wait();
                        const int key = c0 + tt * kTcKeys + lq * 32 + lane;
#pragma unroll
                        for (int r = 0; r < NPH; ++r)
                            if (row_ok(key, r0 + r))
                                mx[r] = fmaxf(mx[r], (__uint_as_float(sh[r]) + __uint_as_float(sl[r])) * scale);
                    }
                    int row;
                    const float m = lane_reduce_rows<NPH, true>(mx, lane, row);
                    if ((lane & (32 / NPH - 1)) == 0) red[lq * NP + r0 + row] = m;
                    conv_sync();
#pragma unroll
                    for (int r = 0; r < NPH; ++r)
                        Mrow[r] = fmaxf(fmaxf(red[r0 + r], red[NP + r0 + r]),
                                        fmaxf(red[2 * NP + r0 + r], red[3 * NP + r0 + r]));
                    want = pre_tiles;
                }
                if (i >= nK + pre && i < nK + nV && (i - nK) % NH == 0) want = max(want, (i - nK) / NH + 1);
                for (; pdone < want; ++pdone) {
                    // pass 2 for tile t: probabilities -> BF16 hi/lo P operand, once the P.V MMAs
                    // that last read this buffer are done
                    const int t = pdone;
                    const int prev = t - 2;
                    if (prev >= 0) {
                        mbar_wait(&pfree[p_idx(t)], p_phase(prev), abort_flag, a.status);
                        tc_fence_after();
                    }
                    float sv[NPH];
                    {
                        uint32_t sh[NPH], sl[NPH];
                        tmem_ld_nowait<NPH>(tmem + lane_addr + t * NS + r0, sh);
                        tmem_ld_nowait<NPH>(tmem + lane_addr + t * NS + NP + r0, sl);
                        tmem_ld_wait();
#pragma unroll
                        for (int r = 0; r < NPH; ++r) sv[r] = __uint_as_float(sh[r]) + __uint_as_float(sl[r]);
                    }
                    const int kt = lq * 32 + lane;
                    store_p(p_buf(t), kt, c0 + t * kTcKeys + kt, sv, Mrow);
                    fence_proxy_async_smem();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&pready[p_idx(t)]);
                }
                if (i == nK + nV) break;
                if (i >= n_early) convert(i);   // the early units are converted already
            }
            // its P.V products are complete
            mbar_wait(odone, 0u, abort_flag, a.status);
            tc_fence_after();
        }

        // read-out: o of this thread's rows, row sums, maxima
        {
            int row;
            const float l = lane_reduce_rows<NPH, false>(lsum, lane, row);
            if ((lane & (32 / NPH - 1)) == 0) red[4 * NP + lq * NP + r0 + row] = l;
            if (lq == 0 && lane == 0)
#pragma unroll
                for (int r = 0; r < NPH; ++r) mrun[r0 + r] = Mrow[r];
#pragma unroll
            for (int h = 0; h < NH; ++h) {
                float o[NPH];
                {
                    uint32_t oh[NPH], ol[NPH];
                    tmem_ld_nowait<NPH>(tmem + lane_addr + ocol + h * NS + r0, oh);
                    tmem_ld_nowait<NPH>(tmem + lane_addr + ocol + h * NS + NP + r0, ol);
                    tmem_ld_wait();
#pragma unroll
                    for (int r = 0; r < NPH; ++r) o[r] = __uint_as_float(oh[r]) + __uint_as_float(ol[r]);
                }
                const int d = h * 128 + lq * 32 + lane;
#pragma unroll
                for (int r = 0; r < NPH; ++r)
                    if (r0 + r < R) part[(size_t)(r0 + r) * (D + 2) + d] = o[r];
            }
        }
        DF_TRACE_MARK(tid == 0, 9);
        conv_sync();
        if (tid < R) {
            const float M = mrun[tid];
            const float L = red[4 * NP + tid] + red[5 * NP + tid] + red[6 * NP + tid] + red[7 * NP + tid];
            part[(size_t)tid * (D + 2) + D] = M;
            part[(size_t)tid * (D + 2) + D + 1] = L;
        }
        if (tid == 0) {
            // after an abort: let every TMA load still in flight land before the CTA exits
            if constexpr (VS) {
                for (int j = 0; j < 3; ++j)
                    if (nis[j] > 0) mbar_drain(&full[j], (uint32_t)((nis[j] - 1) & 1));
            }
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
int launch_tc(const AttnArgs &a, cudaStream_t s) {
    constexpr int max_keys_one_pass = (kTmemCols - kACols - (D / 128) * 2 * NP) / (2 * NP) * kTcKeys;
    constexpr size_t smem = attn_tc_smem_bytes<D, NP, NBUF>();
    static_assert(smem <= 232448, "shared memory");
    AttnTcParams p;
    memset(&p, 0, sizeof(p));
    const uint64_t rows = (uint64_t)a.B * a.nkv * a.cap;
    if (rows + kTcKeys > 0x7fffffffull)
        return fail(DF_ESHAPE, "tensor-core attention: %llu cache rows exceed the TMA row range",
                    (unsigned long long)rows);
    const CUtensorMapDataType dt = a.kv_bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    const int eb = a.kv_bf16 ? 2 : 4;
    const uint32_t box_cols = 128 / eb;       // one 128-byte row per box row
    // a unit: 128 rows x 128 columns (F32: four 32-column groups, BF16: two 64-column groups)
    const uint32_t unit_groups = (uint32_t)(128 / box_cols);
    DF_TRY(make_tma_3d(&p.kmap, a.cache_k, dt, eb, box_cols, rows, (uint64_t)D / box_cols,
                       (uint64_t)D * eb, 128, box_cols, 128, unit_groups));
    // V: the same unit as (column in group, group, row), so a copy reads whole cache rows in
    // address order; it lands row-major (each row's groups as consecutive 128-byte lines)
    DF_TRY(make_tma_3d(&p.vmap, a.cache_v, dt, eb, box_cols, (uint64_t)D / box_cols, rows, 128,
                       (uint64_t)D * eb, box_cols, unit_groups, 128));
    p.a = a;
    dim3 grid(a.n_chunks, a.nkv, a.B);
    // Chunks of more than two tiles stream tile by tile; shorter ones run in one pass (one or two
    // tiles of scores fit TMEM beside the operands for every head dim and row count here), with
    // the V operands in place for an F32 cache with head_dim 128.
    static_assert(max_keys_one_pass >= 2 * kTcKeys, "two tiles in one pass");
    if (a.chunk > 2 * kTcKeys)
        return a.kv_bf16 ? launch_k("attn_tc_kernel", attn_tc_kernel<D, NP, NBUF, true, false, true>,
                                    grid, dim3(kTcThreads), smem, s, p)
                         : launch_k("attn_tc_kernel", attn_tc_kernel<D, NP, NBUF, false, false, true>,
                                    grid, dim3(kTcThreads), smem, s, p);
    if (a.kv_bf16)
        return launch_k("attn_tc_kernel", attn_tc_kernel<D, NP, NBUF, true, false>, grid,
                        dim3(kTcThreads), smem, s, p);
    if constexpr (D == 128) {
        constexpr size_t smem_vs = attn_tc_smem_bytes<D, NP, 3, true>();
        static_assert(smem_vs <= 232448, "shared memory");
        return launch_k("attn_tc_kernel", attn_tc_kernel<D, NP, 3, false, true>, grid,
                        dim3(kTcThreads), smem_vs, s, p);
    } else {
        return launch_k("attn_tc_kernel", attn_tc_kernel<D, NP, NBUF, false, false>, grid,
                        dim3(kTcThreads), smem, s, p);
    }
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

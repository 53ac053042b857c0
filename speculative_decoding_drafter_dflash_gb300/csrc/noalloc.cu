// lm_head_argmax_noalloc: the lm_head + per-row argmax for callers that cannot allocate device
// memory. Its scratch (packed rows, argmax partials, split-tile partial sums, tile counters)
// lives in one fixed-size array in the library's global memory instead of a caller workspace.
#include <algorithm>
#include <mutex>

#include "df_internal.cuh"

namespace df {
int lm_head_run(const uint16_t *W, const float *X, int rows, int H, int V, int32_t *idx,
                float *top1, float *top2, char *scratch, size_t scratch_bytes, int ctas,
                bool zero_counters, cudaStream_t s);
}  // namespace df

namespace {

// Largest problem the fixed scratch holds: 16 rows (one K=15 block), H <= 8192, V <= 524288,
// with a projection grid of at most kNoAllocCtas CTAs (GB300's SM count; a part with more SMs
// runs this entry point on that many).
constexpr int kNoAllocRows = 16;
constexpr int kNoAllocHidden = 8192;
constexpr int kNoAllocVocab = 524288;
constexpr int kNoAllocCtas = df::kDefaultSMs;
constexpr size_t kNoAllocBytes = (size_t)3 * 1024 * 1024 + 512 * 1024;
static_assert(df::lm_head_scratch_bytes_for(kNoAllocRows, kNoAllocHidden, kNoAllocVocab,
                                            kNoAllocCtas) <= kNoAllocBytes,
              "the fixed scratch must hold the largest documented problem");

// Every GPU that loads the library holds this array until the process exits.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocBytes];

std::mutex g_mu;
void *g_addr[64] = {};   // device address of the array, per device ordinal

}  // namespace

extern "C" int lm_head_argmax_noalloc(const uint16_t *W, const float *X, int rows, int H, int V,
                                      int32_t *idx, float *top1, float *top2,
                                      df_stream_t stream) {
    using namespace df;
    if (rows <= 0 || rows > kNoAllocRows || H <= 0 || H > kNoAllocHidden || H % 8 != 0 || V <= 0 ||
        V > kNoAllocVocab)
        return fail(DF_ESHAPE,
                    "lm_head_argmax_noalloc: rows=%d H=%d V=%d outside its fixed scratch "
                    "(rows <= %d, H <= %d and a multiple of 8, V <= %d)",
                    rows, H, V, kNoAllocRows, kNoAllocHidden, kNoAllocVocab);
    const int ctas = std::min(sm_count(), kNoAllocCtas);
    const size_t need = lm_head_scratch_bytes_for(rows, H, V, ctas);
    if (need > kNoAllocBytes)
        return fail(DF_ESHAPE, "lm_head_argmax_noalloc: needs %zu scratch bytes, has %zu", need,
                    kNoAllocBytes);
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return fail(DF_ECUDA, "lm_head_argmax_noalloc: no usable current device");
    void *base = nullptr;
    {
        // One-time set-up per device, with that device current: the host-side symbol is only a
        // stand-in, the kernels need the array's device address.
        std::lock_guard<std::mutex> lk(g_mu);
        if (!g_addr[dev]) {
            // The set-up (which may load the library's device code) cannot run while a stream
            // is being captured: the contract asks for one call on each device before any
            // capture, and a first call during one is refused with this message.
            cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
            if (cudaStreamIsCapturing((cudaStream_t)stream, &cs) == cudaSuccess &&
                cs != cudaStreamCaptureStatusNone)
                return fail(DF_ECUDA,
                            "lm_head_argmax_noalloc: the first call on device %d came during "
                            "stream capture; call it once on this device before capturing",
                            dev);
            void *p = nullptr;
            cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
            if (e != cudaSuccess || p == nullptr)
                return fail(DF_ECUDA, "lm_head_argmax_noalloc: cudaGetSymbolAddress: %s",
                            cudaGetErrorString(e));
            g_addr[dev] = p;
        }
        base = g_addr[dev];
    }
    return lm_head_run(W, X, rows, H, V, idx, top1, top2, static_cast<char *>(base), kNoAllocBytes,
                       ctas, true, (cudaStream_t)stream);
}

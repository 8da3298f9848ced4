// gdn_recurrence_chunked_noalloc: the chunked recurrence for callers that cannot
// allocate device memory.
//
// gdn_recurrence() in chunked mode allocates its prep scratch (and a status word)
// with cudaMalloc on the first call on each device.  Some callers cannot let a
// library do that: a serving process that has handed all of the GPU's memory to
// its own arena up front, where a cudaMalloc from inside a library fails or
// fragments what the arena manages; or a latency-critical path that must not
// take cudaMalloc's implicit device synchronisation.  This entry point runs the
// same prep and scan kernels with their scratch in a fixed-size array that lives
// in this file's static device memory, and reports a bounded wait that gave up in
// a status word that is static device memory too.  The CUDA runtime sets both
// aside when it loads this file's device code on a GPU and keeps them until the
// process exits.  With the runtime's default lazy module loading, that load (and
// the load of the kernels) happens at this entry point's first call on each
// device, in its set-up step; a call with T == 0 does only that set-up, so a
// caller can make it at start-up, before it reserves its arena.
//
// Limits: at most kNoAllocMaxHeads value heads.  The scratch holds the records of
// one 512-token super-block (instead of the allocating path's 2048), so it is
// 16 chunks x 96 heads x 8448 B = 12,976,128 bytes.  The chunk arithmetic does
// not depend on the super-block length (super-blocks start on chunk boundaries
// and the state passes between them through state_inout in FP32), so the
// results equal gdn_recurrence()'s chunked mode.
#include <cudaTypedefs.h>

#include <cstring>
#include <mutex>
#include <string>

#include "gdn.h"
#include "gdn_internal.h"

namespace gdn {
namespace {

constexpr int kNoAllocMaxHeads = 96;
constexpr int kNoAllocSuperBlock = 512;
constexpr size_t kNoAllocScratchFloats =
    static_cast<size_t>(kNoAllocSuperBlock / kChunk) * kNoAllocMaxHeads * kPrepRecordFloats;

// Shared by every call in the process on a given device; see the header for the
// rules that follow from that.
static __device__ __align__(256) float g_noalloc_scratch[kNoAllocScratchFloats];
// Bounded waits of this entry point's kernels that gave up (bits as in the
// allocating path's status word); read and cleared by gdn_device_status().
static __device__ int g_noalloc_status;

constexpr int kMaxDev = 64;
struct NoAllocDevice {
    bool ready = false;
    float* scratch = nullptr;  // device address of g_noalloc_scratch on this device
    int* status = nullptr;     // device address of g_noalloc_status on this device
};
NoAllocDevice g_nd[kMaxDev];
std::mutex g_nd_mu;

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

int map2d(CUtensorMap* map, const float* base, uint64_t width, uint64_t rows, uint32_t box_w, uint32_t box_h,
          CUtensorMapSwizzle swizzle) {
    auto enc = encoder();
    if (!enc) return internal_fail(GDN_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    cuuint64_t dims[2] = {width, rows};
    cuuint64_t strides[1] = {width * sizeof(float)};
    cuuint32_t box[2] = {box_w, box_h};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return internal_fail(GDN_ERR_CUDA, "cuTensorMapEncodeTiled failed: " + std::to_string(r));
    return GDN_OK;
}

// Once per device, with that device current: look up where the runtime placed
// the static array and the status word on it, and have it load the kernels this
// entry point launches.  Nothing is allocated by this code.
int noalloc_device(NoAllocDevice** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return internal_fail(GDN_ERR_CUDA, std::string("cudaGetDevice: ") + cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDev) return internal_fail(GDN_ERR_UNSUPPORTED, "device ordinal out of range");
    std::lock_guard<std::mutex> lk(g_nd_mu);
    NoAllocDevice& d = g_nd[dev];
    if (!d.ready) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess)
            return internal_fail(GDN_ERR_CUDA, std::string("cudaGetSymbolAddress(scratch): ") + cudaGetErrorString(e));
        void* st = nullptr;
        e = cudaGetSymbolAddress(&st, g_noalloc_status);
        if (e != cudaSuccess)
            return internal_fail(GDN_ERR_CUDA, std::string("cudaGetSymbolAddress(status): ") + cudaGetErrorString(e));
        e = preload_two_launch_chunk_kernels();
        if (e == cudaSuccess) e = preload_chunk_scan_tc();
        if (e != cudaSuccess)
            return internal_fail(GDN_ERR_CUDA, std::string("loading the chunk kernels: ") + cudaGetErrorString(e));
        d.scratch = static_cast<float*>(p);
        d.status = static_cast<int*>(st);
        d.ready = true;
    }
    *out = &d;
    return GDN_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

}  // namespace

cudaError_t noalloc_take_status(int device, int* word) {
    *word = 0;
    if (device < 0 || device >= kMaxDev) return cudaSuccess;
    int* st = nullptr;
    {
        std::lock_guard<std::mutex> lk(g_nd_mu);
        if (!g_nd[device].ready) return cudaSuccess;
        st = g_nd[device].status;
    }
    cudaError_t e = cudaMemcpy(word, st, sizeof(int), cudaMemcpyDeviceToHost);
    if (e == cudaSuccess && *word != 0) e = cudaMemset(st, 0, sizeof(int));
    return e;
}
}  // namespace gdn

extern "C" int gdn_recurrence_chunked_noalloc(const float* q, const float* k, const float* v, const float* g,
                                              const float* beta, float* state_inout, float* out, int64_t T,
                                              int n_kh, int n_vh, int d, void* cuda_stream) {
    using namespace gdn;
    if (T < 0) return internal_fail(GDN_ERR_INVALID_ARG, "T < 0");
    if (n_kh <= 0 || n_vh <= 0 || d <= 0)
        return internal_fail(GDN_ERR_INVALID_ARG, "n_kh, n_vh and d must be positive");
    if (n_vh % n_kh != 0) return internal_fail(GDN_ERR_INVALID_ARG, "n_vh must be a multiple of n_kh");
    if (d != kD) return internal_fail(GDN_ERR_UNSUPPORTED, "only d == 128 is supported");
    if (n_vh != kHeadsPerKey * n_kh) return internal_fail(GDN_ERR_UNSUPPORTED, "only n_vh == 3 * n_kh is supported");
    if (n_vh > kNoAllocMaxHeads)
        return internal_fail(GDN_ERR_UNSUPPORTED,
                             "n_vh = " + std::to_string(n_vh) + " exceeds the non-allocating entry point's maximum of " +
                                 std::to_string(kNoAllocMaxHeads) + " value heads (its fixed scratch holds " +
                                 std::to_string(kNoAllocScratchFloats * sizeof(float)) + " bytes)");
    if (T > INT32_MAX - 4096) return internal_fail(GDN_ERR_UNSUPPORTED, "T too large for 32-bit TMA coordinates");
    NoAllocDevice* dev = nullptr;
    if (T == 0) return noalloc_device(&dev);  // the set-up alone; pointers are not used
    if (!q || !k || !v || !g || !beta || !state_inout || !out) return internal_fail(GDN_ERR_INVALID_ARG, "null pointer");
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(state_inout))
        return internal_fail(GDN_ERR_INVALID_ARG, "q, k, v, out and state_inout must be 16-byte aligned");

    int rc = noalloc_device(&dev);
    if (rc != GDN_OK) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);

    ChunkScanParams sp;
    std::memset(&sp, 0, sizeof(sp));
    if ((rc = map2d(&sp.tm_k, k, static_cast<uint64_t>(n_kh) * d, T, 32, kChunk, CU_TENSOR_MAP_SWIZZLE_128B)))
        return rc;
    if ((rc = map2d(&sp.tm_q, q, static_cast<uint64_t>(n_kh) * d, T, 32, kChunk, CU_TENSOR_MAP_SWIZZLE_128B)))
        return rc;
    if ((rc = map2d(&sp.tm_v, v, static_cast<uint64_t>(n_vh) * d, T, chunk_scan_box_cols(), kChunk,
                    CU_TENSOR_MAP_SWIZZLE_NONE)))
        return rc;
    sp.prep = dev->scratch;
    sp.state = state_inout;
    sp.out = out;
    sp.n_kh = n_kh;
    sp.n_vh = n_vh;
    sp.status = dev->status;
    ChunkPrepParams pp;
    pp.q = q;
    pp.k = k;
    pp.g = g;
    pp.beta = beta;
    pp.prep = dev->scratch;
    pp.n_kh = n_kh;
    pp.n_vh = n_vh;
    for (int64_t t0 = 0; t0 < T; t0 += kNoAllocSuperBlock) {
        const int n = static_cast<int>((T - t0) < kNoAllocSuperBlock ? (T - t0) : kNoAllocSuperBlock);
        pp.t_begin = t0;
        pp.n_tokens = n;
        cudaError_t e = launch_chunk_prep(pp, s);
        if (e != cudaSuccess)
            return internal_fail(GDN_ERR_CUDA, std::string("chunk prep launch: ") + cudaGetErrorString(e));
        internal_count_launch();
        sp.t_begin = t0;
        sp.n_tokens = n;
        e = launch_chunk_scan_default(sp, s);
        if (e != cudaSuccess)
            return internal_fail(GDN_ERR_CUDA, std::string("chunk scan launch: ") + cudaGetErrorString(e));
        internal_count_launch();
    }
    return GDN_OK;
}

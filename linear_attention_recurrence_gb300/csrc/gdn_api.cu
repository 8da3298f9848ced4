// C ABI of libgdn.so (declared in include/gdn.h): argument checks, TMA tensor
// maps, the per-device status word and chunked-mode scratch, and the launches.
#include <cudaTypedefs.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <string>

#include "gdn.h"
#include "gdn_internal.h"
#include "gdn_device.cuh"

namespace {

thread_local std::string t_last_error;
std::atomic<uint64_t> g_launches{0};
std::mutex g_mu;

constexpr int kMaxDevices = 64;
struct DeviceState {
    bool init = false;
    int sm_count = 0;
    int* status = nullptr;    // kernel status word (0 = fine)
    float* scratch = nullptr; // chunked-mode prep records for one super-block
    size_t scratch_bytes = 0;
    uint32_t* flags = nullptr; // one-launch chunked form: per-(chunk, key head) flags, then 2 sync words
    uint32_t* sync = nullptr;
    uint32_t* out_flags = nullptr;
    unsigned long long* ring = nullptr;  // tensor-memory form: the tile ring's slot flags
    void* seqnorm = nullptr;   // the sequential scan's fused norm: exchange buffer, counters, generation
    int seqnorm_n_kh = 0;
};
DeviceState g_dev[kMaxDevices];

// Process-wide options (gdn_set_option): A/B choices of the chunked form and the
// failure-path test hooks.  Plain atomics; every call reads the values current
// when it starts.  Nothing is read from the environment.
constexpr int kOptSlots = 8;
// constant-initialised defaults, in slot order (see opt_slot)
std::atomic<int> g_opt[kOptSlots] = {GDN_PRODUCTS_TMEM, 1, 0, 16, -1, 0, 0, 0};  // slot 6: prep CTAs (0: auto)
int opt_slot(int option) {
    switch (option) {
        case GDN_OPT_CHUNK_PRODUCTS: return 0;
        case GDN_OPT_CHUNK_ONE_LAUNCH: return 1;
        case GDN_OPT_NORM_IN_LAUNCH: return 2;
        case GDN_OPT_SEQ_ROWS_PER_THREAD: return 3;
        case GDN_OPT_CHUNK_PREP_CTAS: return 6;
        case GDN_OPT_TEST_WITHHOLD_PREP_TASK: return 4;
        case GDN_OPT_TEST_FAIL_SCRATCH_ALLOC: return 5;
        default: return -1;
    }
}
int opt(int option) { return g_opt[opt_slot(option)].load(std::memory_order_relaxed); }

int fail(int code, const std::string& msg) {
    t_last_error = msg;
    return code;
}

int cuda_fail(cudaError_t e, const char* what) {
    return fail(GDN_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
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

// 2-D FP32 tensor map over a row-major [rows][width] array; out-of-range rows
// read as 0 and are not written.
int make_map(CUtensorMap* map, const void* base, uint64_t width, uint64_t rows, uint32_t box_w, uint32_t box_h,
             CUtensorMapSwizzle swizzle) {
    auto enc = tensor_map_encoder();
    if (!enc) return fail(GDN_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    cuuint64_t dims[2] = {width, rows};
    cuuint64_t strides[1] = {width * sizeof(float)};
    cuuint32_t box[2] = {box_w, box_h};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(GDN_ERR_CUDA, "cuTensorMapEncodeTiled failed: " + std::to_string(r));
    return GDN_OK;
}

// Per-device lazy set-up: SM count and the status word.
int device_state(DeviceState** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return fail(GDN_ERR_UNSUPPORTED, "device ordinal out of range");
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceState& d = g_dev[dev];
    if (!d.init) {
        e = cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
        e = cudaMalloc(&d.status, sizeof(int));
        if (e != cudaSuccess) {
            d.status = nullptr;
            cudaGetLastError();
            return fail(GDN_ERR_ALLOC, std::string("status word allocation failed: ") + cudaGetErrorString(e));
        }
        e = cudaMemset(d.status, 0, sizeof(int));
        if (e != cudaSuccess) return cuda_fail(e, "cudaMemset");
        d.init = true;
    }
    *out = &d;
    return GDN_OK;
}

// Chunked scratch for n_vh value heads: the prep records of one super-block, or,
// when the tensor-memory form is selected, its tiles (the larger of the two, so a
// fallback to the other forms finds room too).
size_t scratch_bytes_for(int n_vh) {
    const size_t rec = static_cast<size_t>(gdn::kChunksPerSuperBlock) * n_vh * gdn::kPrepRecordFloats * sizeof(float);
    if (gdn::chunk_scan_kind() != gdn::ScanKind::kTmem) return rec;
    const size_t tiles = gdn::tile_scratch_floats((n_vh + gdn::kHeadsPerKey - 1) / gdn::kHeadsPerKey, n_vh) * sizeof(float);
    return tiles > rec ? tiles : rec;
}

// The fused sequential norm's scratch for n_kh key heads (zeroed once; its counters
// carry a generation number, so it is never cleared again).
int ensure_seqnorm(DeviceState* d, int n_kh) {
    std::lock_guard<std::mutex> lk(g_mu);
    if (d->seqnorm && d->seqnorm_n_kh >= n_kh) return GDN_OK;
    if (opt(GDN_OPT_TEST_FAIL_SCRATCH_ALLOC) == 1)
        return fail(GDN_ERR_ALLOC, "sequential norm scratch allocation failed (simulated by GDN_OPT_TEST_FAIL_SCRATCH_ALLOC)");
    cudaError_t e;
    if (d->seqnorm) {
        e = cudaDeviceSynchronize();  // the old buffer may still be in use by queued work
        if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
        cudaFree(d->seqnorm);
        d->seqnorm = nullptr;
        d->seqnorm_n_kh = 0;
    }
    const size_t bytes = gdn::seq_norm_scratch_bytes(n_kh);
    void* p = nullptr;
    e = cudaMalloc(&p, bytes);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(GDN_ERR_ALLOC, "sequential norm scratch allocation of " + std::to_string(bytes) +
                                       " bytes failed: " + cudaGetErrorString(e));
    }
    e = cudaMemset(p, 0, bytes);
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) {
        cudaFree(p);
        return cuda_fail(e, "sequential norm scratch initialisation");
    }
    d->seqnorm = p;
    d->seqnorm_n_kh = n_kh;
    return GDN_OK;
}

// Flag words of the one-launch chunked form for up to n_vh key heads (n_kh <= n_vh).
size_t flag_words_for(int n_vh) { return static_cast<size_t>(gdn::kChunksPerSuperBlock) * n_vh; }
// Output flags of the one-launch form with the norm: [chunk][key head][8 scan CTAs] (n_kh <= n_vh).
size_t out_flag_words_for(int n_vh) { return static_cast<size_t>(gdn::kChunksPerSuperBlock) * n_vh * 8; }
// The 32-bit flag words (rounded up to an even count, so the 64-bit ring flags that
// follow are 8-byte aligned), then the ring flags [kTileRing][n_vh].
size_t u32_flag_words_for(int n_vh) {
    return (flag_words_for(n_vh) + out_flag_words_for(n_vh) + gdn::kSyncWords + 1) & ~static_cast<size_t>(1);
}
size_t ring_flags_for(int n_vh) { return static_cast<size_t>(gdn::kTileRing) * n_vh; }

void free_scratch(DeviceState* d) {
    cudaFree(d->scratch);
    cudaFree(d->flags);
    d->scratch = nullptr;
    d->flags = d->sync = d->out_flags = nullptr;
    d->ring = nullptr;
    d->scratch_bytes = 0;
}

int ensure_scratch(DeviceState* d, int n_vh) {
    const size_t need = scratch_bytes_for(n_vh);
    std::lock_guard<std::mutex> lk(g_mu);
    if (d->scratch && d->scratch_bytes >= need) return GDN_OK;
    if (opt(GDN_OPT_TEST_FAIL_SCRATCH_ALLOC) == 1)
        return fail(GDN_ERR_ALLOC, "chunked scratch allocation failed (simulated by GDN_OPT_TEST_FAIL_SCRATCH_ALLOC)");
    if (d->scratch) {
        // a larger head count than before: the old buffer may still be in use by queued work
        cudaError_t e = cudaDeviceSynchronize();
        if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
        free_scratch(d);
    }
    void* p = nullptr;
    void* f = nullptr;
    const size_t flag_bytes = u32_flag_words_for(n_vh) * sizeof(uint32_t) + ring_flags_for(n_vh) * sizeof(unsigned long long);
    cudaError_t e = cudaMalloc(&p, need);
    if (e == cudaSuccess) {
        e = cudaMalloc(&f, flag_bytes);
        if (e != cudaSuccess) cudaFree(p);
    }
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(GDN_ERR_ALLOC, "chunked scratch allocation of " + std::to_string(need + flag_bytes) +
                                       " bytes failed: " + cudaGetErrorString(e));
    }
    d->scratch = static_cast<float*>(p);
    d->scratch_bytes = need;
    d->flags = static_cast<uint32_t*>(f);
    d->out_flags = d->flags + flag_words_for(n_vh);
    d->sync = d->out_flags + out_flag_words_for(n_vh);
    d->ring = reinterpret_cast<unsigned long long*>(d->flags + u32_flag_words_for(n_vh));
    // zero flags and generation before any stream (blocking or not) can use them
    e = cudaMemset(f, 0, flag_bytes);
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) {
        free_scratch(d);
        return cuda_fail(e, "flag initialisation");
    }
    return GDN_OK;
}

// gdn_recurrence_norm runs the norm inside the recurrence's launch only when
// GDN_OPT_NORM_IN_LAUNCH is 1 (or, in sequential mode, when no FP32 output is
// wanted): in the one-launch chunked kernel the prep CTAs cannot stream the
// norm's traffic as fast as the scan produces it (measured 562 vs 362 us per
// 2048-token call), and the sequential scan's fused epilogue costs more than the
// norm's own launch, so by default the norm is a launch of its own.
bool fused_norm_enabled() { return opt(GDN_OPT_NORM_IN_LAUNCH) == 1; }

// Failure-path test hook (GDN_OPT_TEST_WITHHOLD_PREP_TASK): that prep task (chunk
// * n_kh + key head of each super-block) never publishes its flag, so the scan
// CTAs that wait for it run out their bounded wait and report GDN_ERR_TIMEOUT
// (nothing faults or hangs; the next call runs normally).
int withheld_prep_task() { return opt(GDN_OPT_TEST_WITHHOLD_PREP_TASK); }

bool fused_chunk_launch_enabled() {
    if (opt(GDN_OPT_CHUNK_ONE_LAUNCH) == 0) return false;
    return gdn::chunk_scan_kind() != gdn::ScanKind::kTcgen05;
}

__global__ void fill_words_kernel(uint32_t* p, size_t n, uint32_t bits) {
    for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<size_t>(gridDim.x) * blockDim.x)
        p[i] = bits;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool overlap(const void* a, size_t an, const void* b, size_t bn) {
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + bn && b0 < a0 + an;
}

int seq_rows_per_thread() { return opt(GDN_OPT_SEQ_ROWS_PER_THREAD); }

}  // namespace

namespace gdn {
cudaError_t set_smem_once(const void* kernel, int bytes) {
    struct Entry {
        const void* kernel;
        int device;
        int bytes;
    };
    static Entry table[64];
    static int used = 0;
    static std::mutex mu;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lk(mu);
    for (int i = 0; i < used; ++i)
        if (table[i].kernel == kernel && table[i].device == dev && table[i].bytes >= bytes) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess && used < 64) table[used++] = Entry{kernel, dev, bytes};
    return e;
}
int internal_fail(int code, const std::string& msg) { return fail(code, msg); }
ScanKind chunk_scan_kind() {
    switch (opt(GDN_OPT_CHUNK_PRODUCTS)) {
        case GDN_PRODUCTS_FMA: return ScanKind::kFma;
        case GDN_PRODUCTS_TCGEN05: return ScanKind::kTcgen05;
        case GDN_PRODUCTS_TMEM: return ScanKind::kTmem;
        default: return ScanKind::kMma;
    }
}
void internal_count_launch() { g_launches.fetch_add(1); }
}  // namespace gdn

namespace {
// The gated RMSNorm that gdn_recurrence_norm applies to the recurrence's output.
struct NormArgs {
    const float* z;
    const float* w;
    float eps;
    uint16_t* y;
};

int run_recurrence(const float* q, const float* k, const float* v, const float* g, const float* beta,
                   float* state_inout, float* out, int64_t T, int n_kh, int n_vh, int d, int mode,
                   void* cuda_stream, const NormArgs* norm) {
    using namespace gdn;
    if (T < 0) return fail(GDN_ERR_INVALID_ARG, "T < 0");
    if (n_kh <= 0 || n_vh <= 0 || d <= 0) return fail(GDN_ERR_INVALID_ARG, "n_kh, n_vh and d must be positive");
    if (n_vh % n_kh != 0) return fail(GDN_ERR_INVALID_ARG, "n_vh must be a multiple of n_kh");
    if (mode != GDN_SEQUENTIAL && mode != GDN_CHUNKED && mode != GDN_AUTO)
        return fail(GDN_ERR_INVALID_ARG, "unknown mode");
    if (mode == GDN_AUTO) mode = (T < GDN_AUTO_CHUNKED_MIN_T) ? GDN_SEQUENTIAL : GDN_CHUNKED;
    if (d != kD) return fail(GDN_ERR_UNSUPPORTED, "only d == 128 is supported");
    if (n_vh != kHeadsPerKey * n_kh) return fail(GDN_ERR_UNSUPPORTED, "only n_vh == 3 * n_kh is supported");
    if (T > INT32_MAX - 4096) return fail(GDN_ERR_UNSUPPORTED, "T too large for 32-bit TMA coordinates");
    if (T == 0) return GDN_OK;
    // the fused norms (sequential, and the tensor-memory chunked form) may leave the FP32
    // output unwritten; the chunked forms that need it are checked below
    const bool out_optional = norm != nullptr;
    if (!q || !k || !v || !g || !beta || !state_inout || (!out && !out_optional))
        return fail(GDN_ERR_INVALID_ARG, "null pointer");
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || (out && !aligned(out, 16)) ||
        !aligned(state_inout, 16))
        return fail(GDN_ERR_INVALID_ARG, "q, k, v, out and state_inout must be 16-byte aligned");
    if (!aligned(g, 4) || !aligned(beta, 4)) return fail(GDN_ERR_INVALID_ARG, "g and beta must be 4-byte aligned");
    const size_t qk_bytes = static_cast<size_t>(T) * n_kh * d * 4, v_bytes = static_cast<size_t>(T) * n_vh * d * 4;
    const size_t gb_bytes = static_cast<size_t>(T) * n_vh * 4, s_bytes = static_cast<size_t>(n_vh) * d * d * 4;
    const void* ins[5] = {q, k, v, g, beta};
    const size_t in_bytes[5] = {qk_bytes, qk_bytes, v_bytes, gb_bytes, gb_bytes};
    const size_t o_bytes = out ? v_bytes : 0;
    for (int i = 0; i < 5; ++i)
        if (overlap(out, o_bytes, ins[i], in_bytes[i]) || overlap(state_inout, s_bytes, ins[i], in_bytes[i]))
            return fail(GDN_ERR_INVALID_ARG, "out / state_inout overlap an input");
    if (overlap(out, o_bytes, state_inout, s_bytes)) return fail(GDN_ERR_INVALID_ARG, "out overlaps state_inout");

    DeviceState* dev = nullptr;
    int rc = device_state(&dev);
    if (rc != GDN_OK) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);

    if (mode == GDN_SEQUENTIAL) {
        SeqParams p;
        std::memset(&p, 0, sizeof(p));
        const int B = seq_tokens_per_stage();
        if ((rc = make_map(&p.tm_k, k, static_cast<uint64_t>(n_kh) * d, T, d, B, CU_TENSOR_MAP_SWIZZLE_NONE)))
            return rc;
        if ((rc = make_map(&p.tm_q, q, static_cast<uint64_t>(n_kh) * d, T, d, B, CU_TENSOR_MAP_SWIZZLE_NONE)))
            return rc;
        if ((rc = make_map(&p.tm_v, v, static_cast<uint64_t>(n_vh) * d, T, seq_box_cols(), B,
                           CU_TENSOR_MAP_SWIZZLE_NONE)))
            return rc;
        if (out && (rc = make_map(&p.tm_o, out, static_cast<uint64_t>(n_vh) * d, T, seq_box_cols(), B,
                                  CU_TENSOR_MAP_SWIZZLE_NONE)))
            return rc;
        p.g = g;
        p.beta = beta;
        p.state = state_inout;
        p.out = out;
        p.T = T;
        p.n_kh = n_kh;
        p.n_vh = n_vh;
        p.status = dev->status;
        // The norm fused into the scan (one cooperative launch, the FP32 output only
        // optionally stored) when the caller asks for no FP32 output or for the
        // in-launch norm, and all 8 n_kh CTAs fit on the device at once; else the
        // scan, then the norm's own launch (out is required then).  On GB300 the
        // two launches are faster at every T (5.6 vs 9.6 us at T = 1, 537 vs 666 us
        // at T = 2048): the scan is ALU-bound, so the fused form saves the output's
        // HBM traffic but not time.
        const bool want_fused = norm != nullptr && (out == nullptr || fused_norm_enabled());
        if (want_fused && kSeqSlices * n_kh <= dev->sm_count) {
            if ((rc = ensure_seqnorm(dev, n_kh)) != GDN_OK) return rc;
            if ((rc = make_map(&p.tm_z, norm->z, static_cast<uint64_t>(n_vh) * d, T, seq_box_cols(), B,
                               CU_TENSOR_MAP_SWIZZLE_NONE)))
                return rc;
            const size_t cnt = static_cast<size_t>(seq_norm_counters(n_kh));
            p.xflags = static_cast<unsigned long long*>(dev->seqnorm);
            p.sync = reinterpret_cast<uint32_t*>(p.xflags + cnt);
            p.xg = reinterpret_cast<float*>(reinterpret_cast<char*>(p.sync) + 16);
            p.w = norm->w;
            p.y = norm->y;
            p.eps = norm->eps;
            cudaError_t e = launch_seq(p, seq_rows_per_thread(), s);
            if (e == cudaSuccess) {
                g_launches.fetch_add(1);
                return GDN_OK;
            }
            if (e != cudaErrorCooperativeLaunchTooLarge) return cuda_fail(e, "sequential scan + norm launch");
            cudaGetLastError();  // fewer SMs available than the device has: two launches instead
            p.y = nullptr;
        }
        if (norm && !out) return fail(GDN_ERR_INVALID_ARG, "out is required when the norm cannot be fused");
        cudaError_t e = launch_seq(p, seq_rows_per_thread(), s);
        if (e != cudaSuccess) return cuda_fail(e, "sequential scan launch");
        g_launches.fetch_add(1);
        if (norm) {
            e = launch_out_norm(out, norm->z, norm->w, norm->eps, norm->y, T * n_vh, dev->sm_count, s);
            if (e != cudaSuccess) return cuda_fail(e, "output norm launch");
            g_launches.fetch_add(1);
        }
        return GDN_OK;
    }

    if ((rc = ensure_scratch(dev, n_vh)) != GDN_OK) return rc;
    ChunkScanParams sp;
    std::memset(&sp, 0, sizeof(sp));
    if ((rc = make_map(&sp.tm_k, k, static_cast<uint64_t>(n_kh) * d, T, 32, kChunk, CU_TENSOR_MAP_SWIZZLE_128B)))
        return rc;
    if ((rc = make_map(&sp.tm_q, q, static_cast<uint64_t>(n_kh) * d, T, 32, kChunk, CU_TENSOR_MAP_SWIZZLE_128B)))
        return rc;
    if ((rc = make_map(&sp.tm_v, v, static_cast<uint64_t>(n_vh) * d, T, chunk_scan_box_cols(), kChunk,
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
    int n_prep = fused_chunk_launch_enabled() ? chunk_fused_prep_ctas(n_kh, dev->sm_count) : 0;
    // The tensor-memory form: the prep and one scan CTA per value head in one
    // cooperative launch, when the value heads leave at least n_kh SMs for the prep
    // (else, or if fewer SMs are free than the device has, the forms below).
    int n_prep_tm = 0;
    ChunkTmemParams tp;
    std::memset(&tp, 0, sizeof(tp));
    // Prep CTAs: 4 n_kh by default, about twice the prep rate the scan consumes, so that
    // the prep stays a few chunks ahead (its tiles are then read back from L2) and the
    // other SMs are free for work on other streams (measured, 48 value heads: 182.4 us
    // per 2048-token call with 64 prep CTAs, 186.3 with 104, 206.8 with 40).
    if (chunk_scan_kind() == ScanKind::kTmem && opt(GDN_OPT_CHUNK_ONE_LAUNCH) != 0) {
        n_prep_tm = chunk_tmem_prep_ctas(n_kh, n_vh, dev->sm_count);
        int want = opt(GDN_OPT_CHUNK_PREP_CTAS);
        if (want == 0) want = 4 * n_kh;
        if (n_prep_tm > 0) n_prep_tm = want < n_kh ? n_kh : (want < n_prep_tm ? want : n_prep_tm);
    }
    // The norm in the tensor-memory scan's epilogue when no FP32 output is wanted (or the
    // option asks for it); with the FP32 output the recurrence and then the norm's own
    // launch take less time on GB300 (48 value heads: 212 against 230 us per 2048-token
    // call), the norm being HBM-bound and the epilogue the scan's critical path.
    const bool tm_epi_norm = norm != nullptr && (out == nullptr || fused_norm_enabled());
    if (n_prep_tm > 0) {
        if ((rc = make_map(&tp.tm_v, v, static_cast<uint64_t>(n_vh) * d, T, d, kChunk, CU_TENSOR_MAP_SWIZZLE_NONE)))
            return rc;
        tp.state = state_inout;
        tp.out = out;
        tp.status = dev->status;
        tp.flags = dev->flags;
        tp.sync = dev->sync;
        tp.ring = dev->ring;
        tp.n_prep = n_prep_tm;
        tp.withhold_task = withheld_prep_task();
        if (tm_epi_norm) {  // the norm in the scan's output epilogue
            if ((rc = make_map(&tp.tm_z, norm->z, static_cast<uint64_t>(n_vh) * d, T, d, kChunk,
                               CU_TENSOR_MAP_SWIZZLE_NONE)))
                return rc;
            tp.w = norm->w;
            tp.y = norm->y;
            tp.eps = norm->eps;
        }
    }
    if (!out && n_prep_tm == 0)
        return fail(GDN_ERR_INVALID_ARG, "out is required in chunked mode unless the tensor-memory form runs");
    for (int64_t t0 = 0; t0 < T; t0 += kSuperBlock) {
        const int n = static_cast<int>((T - t0) < kSuperBlock ? (T - t0) : kSuperBlock);
        pp.t_begin = t0;
        pp.n_tokens = n;
        sp.t_begin = t0;
        sp.n_tokens = n;
        if (n_prep_tm > 0) {
            tp.prep = pp;
            cudaError_t e = launch_chunk_tmem(tp, s);
            if (e == cudaSuccess) {
                g_launches.fetch_add(1);
                if (norm && !tm_epi_norm) {  // the norm of this super-block's rows after it
                    e = launch_out_norm(out + t0 * n_vh * d, norm->z + t0 * n_vh * d, norm->w, norm->eps,
                                        norm->y + t0 * n_vh * d, static_cast<int64_t>(n) * n_vh, dev->sm_count, s);
                    if (e != cudaSuccess) return cuda_fail(e, "output norm launch");
                    g_launches.fetch_add(1);
                }
                continue;
            }
            if (e != cudaErrorCooperativeLaunchTooLarge) return cuda_fail(e, "chunk prep+scan (tensor memory) launch");
            cudaGetLastError();  // fewer SMs available than the device has: the forms below
            n_prep_tm = 0;
            if (!out)
                return fail(GDN_ERR_INVALID_ARG, "out is required: the tensor-memory launch does not fit the SMs available");
        }
        if (n_prep > 0) {
            ChunkFusedParams fp;
            fp.scan = sp;
            fp.prep = pp;
            fp.flags = dev->flags;
            fp.sync = dev->sync;
            fp.n_prep = n_prep;
            const bool in_launch = norm && fused_norm_enabled();
            fp.z = in_launch ? norm->z : nullptr;
            fp.w = in_launch ? norm->w : nullptr;
            fp.y = in_launch ? norm->y : nullptr;
            fp.eps = in_launch ? norm->eps : 0.f;
            fp.out_flags = dev->out_flags;
            fp.withhold_task = withheld_prep_task();
            cudaError_t e = launch_chunk_fused(fp, chunk_scan_kind() != ScanKind::kFma, s);
            if (e == cudaSuccess) {
                g_launches.fetch_add(1);
                if (norm && !in_launch) {  // the norm of this super-block's rows after it
                    e = launch_out_norm(out + t0 * n_vh * d, norm->z + t0 * n_vh * d, norm->w, norm->eps,
                                        norm->y + t0 * n_vh * d, static_cast<int64_t>(n) * n_vh, dev->sm_count, s);
                    if (e != cudaSuccess) return cuda_fail(e, "output norm launch");
                    g_launches.fetch_add(1);
                }
                continue;
            }
            if (e != cudaErrorCooperativeLaunchTooLarge) return cuda_fail(e, "chunk prep+scan launch");
            cudaGetLastError();  // fewer SMs available than the device has: two launches instead
            n_prep = 0;
        }
        cudaError_t e = launch_chunk_prep(pp, s);
        if (e != cudaSuccess) return cuda_fail(e, "chunk prep launch");
        g_launches.fetch_add(1);
        e = launch_chunk_scan_default(sp, s);
        if (e != cudaSuccess) return cuda_fail(e, "chunk scan launch");
        g_launches.fetch_add(1);
        if (norm) {  // the two-launch form: the norm of this super-block's rows after its scan
            e = launch_out_norm(out + t0 * n_vh * d, norm->z + t0 * n_vh * d, norm->w, norm->eps,
                                norm->y + t0 * n_vh * d, static_cast<int64_t>(n) * n_vh, dev->sm_count, s);
            if (e != cudaSuccess) return cuda_fail(e, "output norm launch");
            g_launches.fetch_add(1);
        }
    }
    return GDN_OK;
}
}  // namespace

extern "C" {

int gdn_recurrence(const float* q, const float* k, const float* v, const float* g, const float* beta,
                   float* state_inout, float* out, int64_t T, int n_kh, int n_vh, int d, int mode,
                   void* cuda_stream) {
    return run_recurrence(q, k, v, g, beta, state_inout, out, T, n_kh, n_vh, d, mode, cuda_stream, nullptr);
}

int gdn_recurrence_norm(const float* q, const float* k, const float* v, const float* g, const float* beta,
                        float* state_inout, float* out, const float* z, const float* w, float eps,
                        uint16_t* y_fp16, int64_t T, int n_kh, int n_vh, int d, int mode, void* cuda_stream) {
    using namespace gdn;
    if (!(eps >= 0.0f) || eps != eps) return fail(GDN_ERR_INVALID_ARG, "eps must be a non-negative number");
    if (T > 0 && n_vh > 0 && d > 0) {
        if (!z || !w || !y_fp16) return fail(GDN_ERR_INVALID_ARG, "null pointer");
        if (!aligned(z, 16) || !aligned(w, 16) || !aligned(y_fp16, 16))
            return fail(GDN_ERR_INVALID_ARG, "z, w and y_fp16 must be 16-byte aligned");
        const size_t nb = static_cast<size_t>(T) * n_vh * d;
        const size_t qk_b = static_cast<size_t>(T) * (n_kh > 0 ? n_kh : 0) * d * 4, gb_b = static_cast<size_t>(T) * n_vh * 4;
        const void* reads[] = {q, k, v, g, beta, z, w, out, state_inout};  // null entries are skipped
        const size_t rb[] = {qk_b, qk_b, nb * 4, gb_b, gb_b, nb * 4, static_cast<size_t>(d) * 4, nb * 4,
                             static_cast<size_t>(n_vh) * d * d * 4};
        for (int i = 0; i < 9; ++i)
            if (reads[i] && overlap(y_fp16, nb * 2, reads[i], rb[i]))
                return fail(GDN_ERR_INVALID_ARG, "y_fp16 overlaps another argument");
        const size_t ob = out ? nb * 4 : 0;
        if (overlap(z, nb * 4, out, ob) || overlap(z, nb * 4, state_inout, static_cast<size_t>(n_vh) * d * d * 4) ||
            overlap(w, static_cast<size_t>(d) * 4, out, ob))
            return fail(GDN_ERR_INVALID_ARG, "out / state_inout overlap an input");
    }
    const NormArgs na{z, w, eps, y_fp16};
    return run_recurrence(q, k, v, g, beta, state_inout, out, T, n_kh, n_vh, d, mode, cuda_stream, &na);
}

int gdn_prestage(const float* qkv, const float* conv_w, const float* conv_hist_in, float* conv_hist_out,
                 const float* a, const float* b, const float* A_log, const float* dt_bias, float* q, float* k,
                 float* v, float* g, float* beta, int64_t T, int n_kh, int n_vh, int d, int activation, float eps,
                 void* cuda_stream) {
    using namespace gdn;
    if (T < 0) return fail(GDN_ERR_INVALID_ARG, "T < 0");
    if (n_kh <= 0 || n_vh <= 0 || d <= 0) return fail(GDN_ERR_INVALID_ARG, "n_kh, n_vh and d must be positive");
    if (activation != 0 && activation != 1) return fail(GDN_ERR_INVALID_ARG, "activation must be 0 or 1");
    if (!(eps >= 0.f) || !std::isfinite(eps)) return fail(GDN_ERR_INVALID_ARG, "eps must be finite and >= 0");
    if (d != kD) return fail(GDN_ERR_UNSUPPORTED, "only d == 128 is supported");
    if (T > (int64_t{1} << 40)) return fail(GDN_ERR_UNSUPPORTED, "T too large");
    const int64_t cw = static_cast<int64_t>(2 * n_kh + n_vh) * d;
    if (T > 0 && (!qkv || !a || !b || !q || !k || !v || !g || !beta))
        return fail(GDN_ERR_INVALID_ARG, "null pointer");
    if (!conv_w || !A_log || !dt_bias) return fail(GDN_ERR_INVALID_ARG, "null pointer");
    const void* a16[] = {qkv, conv_w, conv_hist_in, conv_hist_out, q, k, v};
    for (const void* ptr : a16)
        if (ptr && !aligned(ptr, 16))
            return fail(GDN_ERR_INVALID_ARG, "qkv, conv_w, the histories, q, k and v must be 16-byte aligned");
    const void* a4[] = {a, b, A_log, dt_bias, g, beta};
    for (const void* ptr : a4)
        if (ptr && !aligned(ptr, 4)) return fail(GDN_ERR_INVALID_ARG, "a, b, A_log, dt_bias, g and beta must be 4-byte aligned");
    const size_t f4 = sizeof(float);
    const size_t row_b = static_cast<size_t>(cw) * f4, gate_b = static_cast<size_t>(T) * n_vh * f4;
    const void* ins[] = {qkv, conv_w, conv_hist_in, a, b, A_log, dt_bias};
    const size_t in_b[] = {static_cast<size_t>(T) * row_b, static_cast<size_t>(cw) * 4 * f4, 3 * row_b, gate_b, gate_b,
                           n_vh * f4, n_vh * f4};
    const void* outs[] = {q, k, v, g, beta, conv_hist_out};
    const size_t out_b[] = {static_cast<size_t>(T) * n_kh * d * f4, static_cast<size_t>(T) * n_kh * d * f4,
                            static_cast<size_t>(T) * n_vh * d * f4, gate_b, gate_b, 3 * row_b};
    for (int i = 0; i < 6; ++i) {
        if (!outs[i] || out_b[i] == 0) continue;
        for (int j = 0; j < 7; ++j)
            if (ins[j] && in_b[j] && overlap(outs[i], out_b[i], ins[j], in_b[j]))
                return fail(GDN_ERR_INVALID_ARG, "an output overlaps an input");
        for (int j = i + 1; j < 6; ++j)
            if (outs[j] && out_b[j] && overlap(outs[i], out_b[i], outs[j], out_b[j]))
                return fail(GDN_ERR_INVALID_ARG, "two outputs overlap");
    }
    if (T == 0 && !conv_hist_out) return GDN_OK;
    PrestageParams p{qkv, conv_w, conv_hist_in, conv_hist_out, a, b, A_log, dt_bias, q, k, v, g, beta,
                     T, cw, n_kh, n_vh, activation, eps, static_cast<float>(1.0 / std::sqrt(static_cast<double>(d)))};
    cudaError_t e = launch_prestage(p, static_cast<cudaStream_t>(cuda_stream));
    if (e != cudaSuccess) return cuda_fail(e, "pre-stage launch");
    g_launches.fetch_add(1);
    return GDN_OK;
}

int gdn_decode(const float* q, const float* k, const float* v, const float* g, const float* beta, float* states,
               float* out, int batch, int n_kh, int n_vh, int d, void* cuda_stream) {
    using namespace gdn;
    if (batch < 0) return fail(GDN_ERR_INVALID_ARG, "batch < 0");
    if (n_kh <= 0 || n_vh <= 0 || d <= 0) return fail(GDN_ERR_INVALID_ARG, "n_kh, n_vh and d must be positive");
    if (n_vh % n_kh != 0) return fail(GDN_ERR_INVALID_ARG, "n_vh must be a multiple of n_kh");
    if (d != kD) return fail(GDN_ERR_UNSUPPORTED, "only d == 128 is supported");
    if (n_vh != kHeadsPerKey * n_kh) return fail(GDN_ERR_UNSUPPORTED, "only n_vh == 3 * n_kh is supported");
    if (batch > 65535) return fail(GDN_ERR_UNSUPPORTED, "batch > 65535");
    if (batch == 0) return GDN_OK;
    if (!q || !k || !v || !g || !beta || !states || !out) return fail(GDN_ERR_INVALID_ARG, "null pointer");
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(states, 16))
        return fail(GDN_ERR_INVALID_ARG, "q, k and states must be 16-byte aligned");
    if (!aligned(v, 4) || !aligned(g, 4) || !aligned(beta, 4) || !aligned(out, 4))
        return fail(GDN_ERR_INVALID_ARG, "v, g, beta and out must be 4-byte aligned");
    const size_t s_bytes = static_cast<size_t>(batch) * n_vh * d * d * 4, o_bytes = static_cast<size_t>(batch) * n_vh * d * 4;
    const void* ins[5] = {q, k, v, g, beta};
    const size_t in_bytes[5] = {static_cast<size_t>(batch) * n_kh * d * 4, static_cast<size_t>(batch) * n_kh * d * 4,
                                o_bytes, static_cast<size_t>(batch) * n_vh * 4, static_cast<size_t>(batch) * n_vh * 4};
    for (int i = 0; i < 5; ++i)
        if (overlap(out, o_bytes, ins[i], in_bytes[i]) || overlap(states, s_bytes, ins[i], in_bytes[i]))
            return fail(GDN_ERR_INVALID_ARG, "out / states overlap an input");
    if (overlap(out, o_bytes, states, s_bytes)) return fail(GDN_ERR_INVALID_ARG, "out overlaps states");
    DecodeParams p{q, k, v, g, beta, states, out, batch, n_kh, n_vh};
    cudaError_t e = launch_decode(p, static_cast<cudaStream_t>(cuda_stream));
    if (e != cudaSuccess) return cuda_fail(e, "decode launch");
    g_launches.fetch_add(1);
    return GDN_OK;
}

int gdn_out_norm(const float* out, const float* z, const float* w, float eps, uint16_t* y_fp16, int64_t T,
                 int n_vh, int d, void* cuda_stream) {
    using namespace gdn;
    if (T < 0) return fail(GDN_ERR_INVALID_ARG, "T < 0");
    if (n_vh <= 0 || d <= 0) return fail(GDN_ERR_INVALID_ARG, "n_vh and d must be positive");
    if (!(eps >= 0.0f) || eps != eps) return fail(GDN_ERR_INVALID_ARG, "eps must be a non-negative number");
    if (d != kD) return fail(GDN_ERR_UNSUPPORTED, "only d == 128 is supported");
    if (T == 0) return GDN_OK;
    if (!out || !z || !w || !y_fp16) return fail(GDN_ERR_INVALID_ARG, "null pointer");
    if (!aligned(out, 16) || !aligned(z, 16) || !aligned(w, 16) || !aligned(y_fp16, 8))
        return fail(GDN_ERR_INVALID_ARG, "out, z, w must be 16-byte and y_fp16 8-byte aligned");
    const size_t nb = static_cast<size_t>(T) * n_vh * d;
    if (overlap(y_fp16, nb * 2, out, nb * 4) || overlap(y_fp16, nb * 2, z, nb * 4) ||
        overlap(y_fp16, nb * 2, w, static_cast<size_t>(d) * 4))
        return fail(GDN_ERR_INVALID_ARG, "y_fp16 overlaps an input");
    DeviceState* dev = nullptr;
    int rc = device_state(&dev);
    if (rc != GDN_OK) return rc;
    cudaError_t e = launch_out_norm(out, z, w, eps, y_fp16, T * n_vh, dev->sm_count,
                                    static_cast<cudaStream_t>(cuda_stream));
    if (e != cudaSuccess) return cuda_fail(e, "output norm launch");
    g_launches.fetch_add(1);
    return GDN_OK;
}

const char* gdn_last_error(void) { return t_last_error.c_str(); }

int gdn_device_status(void* cuda_stream) {
    // Allocates nothing: a device whose status word was never allocated has run no
    // kernel of the allocating entry points.
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return fail(GDN_ERR_UNSUPPORTED, "device ordinal out of range");
    e = cudaStreamSynchronize(static_cast<cudaStream_t>(cuda_stream));
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    DeviceState* d = nullptr;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        if (g_dev[dev].init) d = &g_dev[dev];
    }
    int word = 0;
    if (d) {
        e = cudaMemcpy(&word, d->status, sizeof(int), cudaMemcpyDeviceToHost);
        if (e != cudaSuccess) return cuda_fail(e, "status read");
        if (word != 0) {
            e = cudaMemset(d->status, 0, sizeof(int));
            if (e != cudaSuccess) return cuda_fail(e, "status reset");
        }
    }
    int na_word = 0;
    e = gdn::noalloc_take_status(dev, &na_word);
    if (e != cudaSuccess) return cuda_fail(e, "status read (non-allocating entry point)");
    if (word == 0 && na_word == 0) return GDN_OK;
    std::string msg = "a kernel gave up a bounded wait (status word " + std::to_string(word | na_word) + ")";
    if (na_word != 0) msg += " in gdn_recurrence_chunked_noalloc";
    if (word & gdn::kDevErrNormTimeout) msg += " (the fused sequential norm's exchange between CTAs)";
    if (word & gdn::kDevErrRingTimeout) msg += " (a chunk prep's wait for a free slot of the tile ring)";
    uint32_t diag[3] = {0, 0, 0};
    if ((word & gdn::kDevErrFlagTimeout) && d && d->sync &&
        cudaMemcpy(diag, d->sync + 2, sizeof(diag), cudaMemcpyDeviceToHost) == cudaSuccess)
        msg += ": prep flag " + std::to_string(diag[0]) + " held " + std::to_string(diag[1]) + ", awaited " +
               std::to_string(diag[2]);
    return fail(GDN_ERR_TIMEOUT, msg);
}

int gdn_release_scratch(int device) {
    if (device < 0 || device >= kMaxDevices) return fail(GDN_ERR_INVALID_ARG, "device ordinal out of range");
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceState& d = g_dev[device];
    if (!d.scratch && !d.seqnorm) return GDN_OK;
    int cur = 0;
    cudaGetDevice(&cur);
    cudaSetDevice(device);
    cudaError_t e = cudaFree(d.scratch);
    cudaError_t e2 = cudaFree(d.flags);
    if (d.seqnorm) {
        cudaFree(d.seqnorm);
        d.seqnorm = nullptr;
        d.seqnorm_n_kh = 0;
    }
    cudaSetDevice(cur);
    d.scratch = nullptr;
    d.flags = d.sync = d.out_flags = nullptr;
    d.ring = nullptr;
    d.scratch_bytes = 0;
    if (e != cudaSuccess) return cuda_fail(e, "cudaFree");
    if (e2 != cudaSuccess) return cuda_fail(e2, "cudaFree");
    return GDN_OK;
}

int gdn_poison_scratch(uint32_t bits, int n_vh, void* cuda_stream) {
    if (n_vh <= 0) return fail(GDN_ERR_INVALID_ARG, "n_vh must be positive");
    DeviceState* dev = nullptr;
    int rc = device_state(&dev);
    if (rc != GDN_OK) return rc;
    if ((rc = ensure_scratch(dev, n_vh)) != GDN_OK) return rc;
    const size_t n = dev->scratch_bytes / sizeof(uint32_t);
    fill_words_kernel<<<dev->sm_count * 4, 256, 0, static_cast<cudaStream_t>(cuda_stream)>>>(
        reinterpret_cast<uint32_t*>(dev->scratch), n, bits);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "scratch fill launch");
    g_launches.fetch_add(1);
    return GDN_OK;
}

int gdn_set_option(int option, int value) {
    const int slot = opt_slot(option);
    if (slot < 0) return fail(GDN_ERR_INVALID_ARG, "unknown option " + std::to_string(option));
    bool ok = true;
    switch (option) {
        case GDN_OPT_CHUNK_PRODUCTS:
            ok = value == GDN_PRODUCTS_MMA || value == GDN_PRODUCTS_FMA || value == GDN_PRODUCTS_TCGEN05 ||
                 value == GDN_PRODUCTS_TMEM;
            break;
        case GDN_OPT_CHUNK_ONE_LAUNCH:
        case GDN_OPT_NORM_IN_LAUNCH:
        case GDN_OPT_TEST_FAIL_SCRATCH_ALLOC: ok = value == 0 || value == 1; break;
        case GDN_OPT_SEQ_ROWS_PER_THREAD: ok = value == 8 || value == 16; break;
        case GDN_OPT_CHUNK_PREP_CTAS: ok = value >= 0 && value <= 4096; break;
        case GDN_OPT_TEST_WITHHOLD_PREP_TASK: ok = value >= -1; break;
        default: break;
    }
    if (!ok) return fail(GDN_ERR_INVALID_ARG, "value " + std::to_string(value) + " not allowed for option " +
                                                  std::to_string(option));
    g_opt[slot].store(value);
    return GDN_OK;
}

int gdn_get_option(int option, int* value) {
    const int slot = opt_slot(option);
    if (slot < 0) return fail(GDN_ERR_INVALID_ARG, "unknown option " + std::to_string(option));
    if (!value) return fail(GDN_ERR_INVALID_ARG, "null pointer");
    *value = g_opt[slot].load();
    return GDN_OK;
}

size_t gdn_chunked_scratch_bytes(int n_vh) { return n_vh > 0 ? scratch_bytes_for(n_vh) : 0; }

uint64_t gdn_launch_count(void) { return g_launches.load(); }

}  // extern "C"

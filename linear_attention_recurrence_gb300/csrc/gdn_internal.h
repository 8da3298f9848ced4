// Host-side interface between the C ABI (gdn_api.cu) and the kernel files.
#pragma once

#include <cstdint>
#include <string>
#include <cuda.h>
#include <cuda_runtime.h>

namespace gdn {

constexpr int kD = 128;          // key and value head dimension these kernels support
constexpr int kHeadsPerKey = 3;  // value heads per key head (h, h + n_kh, h + 2 n_kh)
constexpr int kChunk = 32;       // chunked mode: tokens per WY chunk
constexpr int kSuperBlock = 2048;  // chunked mode: tokens per prep/scan pass
constexpr int kChunksPerSuperBlock = kSuperBlock / kChunk;
// Per (chunk, value head) prep record: T'^T [32][32], P^T [32][32], e^gamma [32],
// e^(gamma_last - gamma) [32], in floats.
constexpr int kPrepRecordFloats = 2 * kChunk * kChunk + 2 * kChunk;
constexpr int kRecTP = 0;                            // T'^T [s][t]
constexpr int kRecPT = kChunk * kChunk;              // P^T  [s][t]
constexpr int kRecEG = 2 * kChunk * kChunk;          // e^gamma_t
constexpr int kRecER = 2 * kChunk * kChunk + kChunk;  // e^(gamma_last - gamma_t)

// Tiles of the tensor-memory scan (gdn_chunk_tmem.cu), written by its prep and
// read by bulk copies into shared memory, where the MMA descriptors read them as
// K-major operands: every 32-float row is 128-byte swizzled (16-byte chunk index
// XOR row % 8), so a tile copied to a 1024-byte-aligned address is in the layout
// the descriptors expect.  Each FP32 value is stored as TF32 hi and lo (x = hi + lo).
// Per (chunk, key head), kKeyTileFloats floats:
//   [K; Q]:     [4 blocks of 32 key dims][128 rows: hi of k tokens 0-31, q tokens 0-31,
//               then lo of the same 64][32] (one 128-row operand [hi; lo] per block)
//   K^T hi, lo: [128 key dims][32 tokens]
constexpr int kTileKQ = 0, kTileKQLoRow = 64, kTileKTH = 16384, kTileKTL = 20480, kKeyTileFloats = 24576;
// Per (chunk, value head), kHeadTileFloats floats: T' hi, lo and P hi, lo, each
// [32 rows t][32 columns s], then e^gamma_t [32] and e^(gamma_last - gamma_t) [32].
constexpr int kTileTPH = 0, kTileTPL = 1024, kTilePH = 2048, kTilePL = 3072, kTileEG = 4096, kTileER = 4128;
constexpr int kHeadTileFloats = 4160;
// The tiles live in a ring of kTileRing chunk slots (chunk ci in slot ci % kTileRing,
// 19 MB for 16 key heads and 48 value heads): key tiles [kTileRing][n_kh], then head
// tiles [kTileRing][n_vh].  The prep writes a slot again only once the scan CTAs of the
// chunk that last used it have copied it (ChunkTmemParams::ring), so the ring stays in
// L2 rather than streaming a whole super-block's tiles through HBM.
constexpr int kTileRing = 8;
inline size_t tile_scratch_floats(int n_kh, int n_vh) {
    return static_cast<size_t>(kTileRing) *
           (static_cast<size_t>(n_kh) * kKeyTileFloats + static_cast<size_t>(n_vh) * kHeadTileFloats);
}
__host__ __device__ inline float* key_tiles(float* base, int n_kh, int ci, int kh) {
    return base + (static_cast<int64_t>(ci % kTileRing) * n_kh + kh) * kKeyTileFloats;
}
__host__ __device__ inline float* head_tiles(float* base, int n_kh, int n_vh, int ci, int vh) {
    return base + static_cast<int64_t>(kTileRing) * n_kh * kKeyTileFloats +
           (static_cast<int64_t>(ci % kTileRing) * n_vh + vh) * kHeadTileFloats;
}

// ---- sequential scan ----
struct SeqParams {
    CUtensorMap tm_k;  // k viewed as [T][n_kh*128] FP32, box {128, B}
    CUtensorMap tm_q;  // q, same
    CUtensorMap tm_v;  // v viewed as [T][n_vh*128] FP32, box {16, B}
    CUtensorMap tm_o;  // out viewed as [T][n_vh*128] FP32, box {16, B} (TMA stores)
    CUtensorMap tm_z;  // fused norm: z viewed as [T][n_vh*128] FP32, box {16, B}
    const float* g;
    const float* beta;
    float* state;
    float* out;        // nullptr: the FP32 output is not stored (fused norm only)
    const float* w;    // fused norm: weight [128]
    uint16_t* y;       // fused norm: y, or nullptr for the recurrence alone
    float eps;
    // fused norm, device scratch of seq_norm_scratch_bytes(n_kh): the exchange of
    // the group sums between the 8 CTAs of a key head, its counters, and the
    // launch generation (sync[0]) with a count of finished CTAs (sync[1])
    float* xg;
    unsigned long long* xflags;  // [n_kh][8][48] stages published per row, [n_kh][8][norm warps] gathered
    uint32_t* sync;
    int64_t T;
    int n_kh;
    int n_vh;
    int* status;
};
int seq_tokens_per_stage();
constexpr int kSeqSlices = 8;  // CTAs (16-column slices) of a key head in the sequential scan
int seq_box_cols();
// rows_per_thread: 8 or 16.  With p.y set, the gated RMSNorm of the output is
// fused in (a cooperative launch; it fails with cudaErrorCooperativeLaunchTooLarge
// when the 8 n_kh CTAs cannot be resident at once).  Returns the CUDA error of the
// launch.
size_t seq_norm_scratch_bytes(int n_kh);
int seq_norm_counters(int n_kh);  // 64-bit counters at the start of that scratch
cudaError_t launch_seq(const SeqParams& p, int rows_per_thread, cudaStream_t s);

// ---- batched decode (one token per sequence) ----
struct DecodeParams {
    const float* q;      // [batch][n_kh][128]
    const float* k;      // [batch][n_kh][128]
    const float* v;      // [batch][n_vh][128]
    const float* g;      // [batch][n_vh]
    const float* beta;   // [batch][n_vh]
    float* state;        // [batch][n_vh][128][128]
    float* out;          // [batch][n_vh][128]
    int batch;
    int n_kh;
    int n_vh;
};
cudaError_t launch_decode(const DecodeParams& p, cudaStream_t s);

// ---- pre-stage ----
struct PrestageParams {
    const float* qkv;      // [T][cw], cw = (2 n_kh + n_vh) * 128
    const float* conv_w;   // [cw][4]
    const float* hist_in;  // [3][cw] or nullptr (zeros)
    float* hist_out;       // [3][cw] or nullptr
    const float* a;        // [T][n_vh]
    const float* b;        // [T][n_vh]
    const float* A_log;    // [n_vh]
    const float* dt_bias;  // [n_vh]
    float* q;              // [T][n_kh][128]
    float* k;              // [T][n_kh][128]
    float* v;              // [T][n_vh][128]
    float* g;              // [T][n_vh]
    float* beta;           // [T][n_vh]
    int64_t T;
    int64_t cw;
    int n_kh;
    int n_vh;
    int activation;
    float eps;
    float q_scale;         // 1 / sqrt(128)
};
cudaError_t launch_prestage(const PrestageParams& p, cudaStream_t s);

// ---- output norm ----
cudaError_t launch_out_norm(const float* out, const float* z, const float* w, float eps, uint16_t* y,
                            int64_t rows, int sm_count, cudaStream_t s);

// ---- chunked mode ----
struct ChunkScanParams {
    CUtensorMap tm_k;  // k viewed as [T][n_kh*128], box {32, 32}, 128-byte swizzle
    CUtensorMap tm_q;  // q, same
    CUtensorMap tm_v;  // v viewed as [T][n_vh*128], box {16, 32}
    const float* prep;  // prep records of this super-block, [chunk][n_vh][kPrepRecordFloats]
    float* state;
    float* out;
    int64_t t_begin;  // first token of the super-block (row in the tensor maps and in out)
    int n_tokens;     // tokens in this super-block (1..2048)
    int n_kh;
    int n_vh;
    int* status;
};
struct ChunkPrepParams {
    const float* q;
    const float* k;
    const float* g;
    const float* beta;
    float* prep;
    int64_t t_begin;
    int n_tokens;
    int n_kh;
    int n_vh;
};
cudaError_t launch_chunk_prep(const ChunkPrepParams& p, cudaStream_t s);
// Prep and scan of one super-block in one cooperative launch: CTAs 0..n_prep-1 run
// the prep tasks, the next 8 n_kh CTAs the scan.
struct ChunkFusedParams {
    ChunkScanParams scan;
    ChunkPrepParams prep;  // same prep, t_begin and n_tokens as scan
    uint32_t* flags;       // [kChunksPerSuperBlock][n_kh]: generation of each finished prep task
    uint32_t* sync;        // [0]: generation of the last finished launch, [1]: CTAs finished so far,
                           // [2..4]: the first flag wait that ran out (index, value seen, value awaited)
    int n_prep;
    // The gated RMSNorm of the outputs by the prep CTAs once their tasks are done,
    // when y != nullptr (out is then read back, through L2, after the scan CTAs of a
    // (chunk, key head) have published it in out_flags).
    const float* z;        // [T][n_vh][128], absolute token rows like out
    const float* w;        // [128]
    uint16_t* y;           // [T][n_vh][128] binary16 bits
    float eps;
    uint32_t* out_flags;   // [kChunksPerSuperBlock][n_kh][8]: generation of each scan CTA's finished chunk
    int withhold_task;     // failure-path test: this prep task's flag is never published (-1: none)
};
// CTAs the one-launch form gives the prep on a device with sm_count SMs, or 0
// when too few SMs are left beside the scan (the two-launch form is used then).
int chunk_fused_prep_ctas(int n_kh, int sm_count);
constexpr int kSyncWords = 8;  // words of ChunkFusedParams::sync
// Fails (cudaErrorCooperativeLaunchTooLarge) when the grid cannot be resident at once.
// `mma`: the scan's large products (K S0, Q S0, K^T D) as split-TF32 warp-level
// tensor-core MMAs; else as packed FP32 FMAs.  Both meet the same tolerance.
cudaError_t launch_chunk_fused(const ChunkFusedParams& p, bool mma, cudaStream_t s);
cudaError_t launch_chunk_scan(const ChunkScanParams& p, bool mma, cudaStream_t s);
// Prep and the tensor-memory scan of one super-block in one cooperative launch
// (gdn_chunk_tmem.cu): CTAs 0..n_prep-1 run the prep tasks, writing tiles
// (kKeyTileFloats / kHeadTileFloats above) into prep.prep; the next n_vh CTAs scan,
// one per value head.
struct ChunkTmemParams {
    ChunkPrepParams prep;  // the prep's inputs, super-block and head counts; prep.prep: the tiles
    CUtensorMap tm_v;      // v viewed as [T][n_vh*128], box {128, 32}, no swizzle
    float* state;
    float* out;
    int* status;
    uint32_t* flags;       // as ChunkFusedParams::flags
    uint32_t* sync;        // as ChunkFusedParams::sync
    // [kTileRing][n_vh]: (generation << 32) | chunk, once the scan CTA of value head vh has
    // copied that chunk's tiles out of the ring slot
    unsigned long long* ring;
    int n_prep;
    int withhold_task;     // failure-path test: this prep task's flag is never published (-1: none)
    // The gated RMSNorm of the output in the scan's epilogue, when y != nullptr (out
    // may then be nullptr: the FP32 output is not written).
    CUtensorMap tm_z;      // z viewed as [T][n_vh*128], box {128, 32}, no swizzle
    const float* w;        // [128]
    uint16_t* y;           // [T][n_vh][128] binary16 bits
    float eps;
};
// Prep CTAs of the tensor-memory form on a device with sm_count SMs (one CTA per
// SM: the scan CTAs hold all 512 tensor-memory columns), or 0 when fewer than
// n_kh SMs would be left for the prep.
int chunk_tmem_prep_ctas(int n_kh, int n_vh, int sm_count);
// Fails (cudaErrorCooperativeLaunchTooLarge) when the grid cannot be resident at once.
cudaError_t launch_chunk_tmem(const ChunkTmemParams& p, cudaStream_t s);
// Make the runtime load the tensor-memory kernel on the current device now.
cudaError_t preload_chunk_tmem();
// The same scan with the large products as split-TF32 tcgen05 MMAs (accumulators
// in tensor memory); same parameters and results within tolerance.
cudaError_t launch_chunk_scan_tc(const ChunkScanParams& p, cudaStream_t s);
// Which scan the entry points run, from the option GDN_OPT_CHUNK_PRODUCTS (set by
// gdn_set_option, for A/B measurements): GDN_PRODUCTS_FMA the CUDA-core products,
// GDN_PRODUCTS_TCGEN05 the tcgen05 scan (two launches only: at 48 columns per CTA
// each tcgen05.mma costs a near-fixed ~80 cycles), else the warp-level MMA scan.
// Implemented in gdn_api.cu.
enum class ScanKind { kFma, kMma, kTcgen05, kTmem };
ScanKind chunk_scan_kind();
// The two-launch scan of the selected kind.
cudaError_t launch_chunk_scan_default(const ChunkScanParams& p, cudaStream_t s);
int chunk_scan_box_cols();
// Make the runtime load the two-launch chunk kernels (prep, both forms of the
// scan; the tcgen05 scan) on the current device now, without launching them.
// Under lazy module loading this is otherwise done by their first launch.
cudaError_t preload_two_launch_chunk_kernels();
cudaError_t preload_chunk_scan_tc();

// The non-allocating entry point's status word on `device` (gdn_noalloc.cu): if
// that entry point has been set up on the device, copies the word to *word and
// clears it; else sets *word to 0.  Returns the CUDA error of the copies.
cudaError_t noalloc_take_status(int device, int* word);

// Raises a kernel's dynamic shared-memory limit to `bytes` on the current device,
// once per (kernel, device); later calls return at once (implemented in gdn_api.cu).
cudaError_t set_smem_once(const void* kernel, int bytes);

// ---- shared by the C-ABI entry points (implemented in gdn_api.cu) ----
// Records `msg` as the calling thread's gdn_last_error() and returns `code`.
int internal_fail(int code, const std::string& msg);
// Adds one kernel launch to gdn_launch_count().
void internal_count_launch();

}  // namespace gdn

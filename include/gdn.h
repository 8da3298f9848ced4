/*
 * gdn.h - C ABI of libgdn.so, the GB300 (sm_103a) Gated DeltaNet prefill
 * recurrence and its gated RMSNorm output.
 *
 * Pages this interface follows (cited by title and section):
 *   [P413]  "#413 prefill: DeltaNet recurrence with the three value heads of a key
 *           head in one thread" - section "What changes" (the recurrence, the key
 *           head shared by value heads qh, qh+16, qh+32, the FP32 recurrence
 *           output y and its FP16 normed copy y_h) and section "Exactness" (the
 *           state after the chunk is part of the result; parity is checked from
 *           a non-zero starting state).
 *   [P1372] "#1372 DeltaNet recurrence: STRATA_GDN_CHUNKED=1 - the prompt's
 *           recurrence in 32-token chunks" - section "What it does" (the 32-token
 *           WY form, 2048-token super-blocks, the per-device scratch kept between
 *           calls).
 *   [R20C]  "Round 20 Track C Audit: gdn_pre Key-Head t >= 3 Vectorized conv_w
 *           Fast Path + gdn_scan_r ..." - section 1 "Summary of Changes" (the
 *           pre-stage's causal convolution over the packed qkv rows).
 *
 * Layout (all tensors dense, row-major, contiguous, FP32 unless stated):
 *   q, k        [T][n_kh][d]      query / key rows per key head
 *   v, out      [T][n_vh][d]      value rows / recurrence output o per value head
 *   g, beta     [T][n_vh]         log-decay gate (g <= 0) and delta-rule strength
 *   state_inout [n_vh][d][d]      S[h][i][j]: i = key dim (row), j = value dim
 *   z           [T][n_vh][d]      output gate
 *   w           [d]               norm weight, shared by all value heads
 *   y_fp16      [T][n_vh][d]      IEEE binary16 bits
 * Value head h reads key head h % n_kh.
 *
 * Ownership: every pointer is a DEVICE pointer owned by the caller, on the
 * current CUDA device.  The library allocates only (a) a 4-byte status word per
 * device, (b) the chunked mode's per-device scratch (prep results: 25.9 MB for
 * 48 value heads, which also holds the default GDN_PRODUCTS_TMEM form's ring of
 * operand tiles for 8 chunks, plus 15 KB of hand-off flags) and (c) the
 * sequential mode's fused-norm scratch (about 100 KB for 16 key heads), each on
 * first use and kept until gdn_release_scratch() or process exit.  Calls on one
 * device share that scratch: enqueue them on one stream (or otherwise order
 * them); two in flight at once would corrupt each other.
 *
 * Asynchrony: every compute call only validates its arguments on the host and
 * enqueues kernels on `cuda_stream` (a cudaStream_t; NULL = the legacy default
 * stream).  Nothing synchronises the host except the one-time allocations above.
 * Inputs and outputs must not overlap (out, state_inout and y_fp16 are written
 * while q, k, v, g, beta, z, w are read).
 *
 * Errors: no call throws.  Each returns a gdn_status; on a non-OK status
 * gdn_last_error() returns a message for the calling thread.  A kernel that
 * gives up a bounded wait records it in the device status word, which
 * gdn_device_status() reads (returning GDN_ERR_TIMEOUT, with the kind of wait in
 * the message).
 */
#ifndef GDN_H
#define GDN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum gdn_mode {
    GDN_SEQUENTIAL = 0, /* one token at a time; bit-identical across reruns and T splits */
    GDN_CHUNKED = 1,    /* 32-token WY chunks in 2048-token super-blocks */
    GDN_AUTO = 2        /* GDN_SEQUENTIAL for T < GDN_AUTO_CHUNKED_MIN_T, else GDN_CHUNKED */
} gdn_mode;

/* Token count from which GDN_AUTO takes the chunked form: the measured crossover
 * of the two modes' GPU time per call on GB300 (48 value heads, d = 128). */
#define GDN_AUTO_CHUNKED_MIN_T 64

typedef enum gdn_status {
    GDN_OK = 0,
    GDN_ERR_INVALID_ARG = -1, /* null pointer, T < 0, n_vh % n_kh != 0, bad mode, eps < 0 */
    GDN_ERR_UNSUPPORTED = -2, /* shapes this build has no kernel for (d != 128, n_vh != 3 n_kh) */
    GDN_ERR_ALLOC = -3,       /* the per-device scratch or status word could not be allocated */
    GDN_ERR_CUDA = -4,        /* a CUDA runtime call or a launch failed */
    GDN_ERR_TIMEOUT = -5      /* a kernel gave up a bounded wait (gdn_device_status only) */
} gdn_status;

/*
 * gdn_recurrence - the gated delta-rule recurrence over T tokens ([P413] "What
 * changes"; [P1372] "What it does" for mode GDN_CHUNKED).  Per value head h,
 * key head kh = h % n_kh, and token t:
 *     S <- exp(g[t][h]) S
 *     delta = beta[t][h] (v[t][h] - S^T k[t][kh])
 *     S <- S + k[t][kh] delta^T
 *     out[t][h] = S^T q[t][kh]
 * state_inout is read as the starting state and overwritten with the state
 * after token T-1, so consecutive calls continue one sequence.  In
 * GDN_SEQUENTIAL mode a sequence split over several calls gives the same bits
 * as one call.  GDN_CHUNKED evaluates the same recurrence in 32-token WY
 * chunks (other FP32 rounding; within 2e-6 of the FP64 result, relative to
 * the largest magnitude).  GDN_AUTO picks one of the two by T per call (so a
 * sequence split into calls of different lengths may mix the two roundings).
 * GDN_CHUNKED computes the chunk's products on the tensor cores as three TF32
 * MMAs per FP32 product (split operands; same 2e-6 bound).  Other forms of the
 * chunked kernels, for A/B measurements, are chosen with gdn_set_option()
 * (GDN_OPT_CHUNK_PRODUCTS, GDN_OPT_CHUNK_ONE_LAUNCH); the library reads no
 * environment variable.
 *
 * Supported shapes: d == 128 and n_vh == 3 * n_kh (n_kh >= 1).  T == 0 is a
 * no-op returning GDN_OK.  The first GDN_CHUNKED call on a device allocates the
 * scratch (GDN_ERR_ALLOC if that fails; nothing is launched then).
 */
int gdn_recurrence(const float* q, const float* k, const float* v,
                   const float* g, const float* beta,
                   float* state_inout, float* out,
                   int64_t T, int n_kh, int n_vh, int d, int mode,
                   void* cuda_stream);

/*
 * gdn_prestage - the recurrence's inputs from a layer's projections ([R20C]
 * section 1: a 4-tap causal convolution per channel over the packed qkv rows,
 * q of key head kh at channels kh*d, k at (n_kh + kh)*d, v of value head h at
 * (2 n_kh + h)*d).  With Cw = (2 n_kh + n_vh) d channels per row, per token t and
 * channel c:
 *     x_c = sum_{j=0..3} conv_w[c][j] X[t-3+j][c]    (X[-3..-1] = conv_hist_in)
 *     u_c = activation ? x_c / (1 + exp(-x_c)) : x_c
 *     q[t][kh] = u_q / sqrt(|u_q|^2 + eps) / sqrt(d);   k[t][kh] = u_k / sqrt(|u_k|^2 + eps)
 *     v[t][h]  = u_v
 *     g[t][h]  = -exp(A_log[h]) log(1 + exp(a[t][h] + dt_bias[h]));   beta[t][h] = 1 / (1 + exp(-b[t][h]))
 * The outputs are gdn_recurrence's q, k, v, g, beta in its layout.  The
 * activation, eps, the 1/sqrt(d) on q and the gate formula are readings: the page
 * names the convolution and the outputs only.
 *
 *   qkv [T][Cw], conv_w [Cw][4] (tap j multiplies row t-3+j), a, b [T][n_vh],
 *   A_log, dt_bias [n_vh]: inputs.  conv_hist_in [3][Cw]: the three rows before
 *   this call (oldest first), or NULL at the start of a sequence (zeros).
 *   conv_hist_out [3][Cw] or NULL: receives the last three rows of (conv_hist_in,
 *   qkv), the conv_hist_in of the next call; it must not overlap conv_hist_in.
 *   q, k [T][n_kh][d], v [T][n_vh][d], g, beta [T][n_vh]: outputs.
 *   activation: 1 (SiLU) or 0; eps >= 0.
 * Alignment: qkv, conv_w, the histories, q, k, v 16 bytes; the rest 4 bytes.
 * No output may overlap an input or another output.  d == 128 only.  T == 0
 * only copies the history (if conv_hist_out is given).  A sequence split over
 * calls with the history carried gives the same bits as one call.
 */
int gdn_prestage(const float* qkv, const float* conv_w,
                 const float* conv_hist_in, float* conv_hist_out,
                 const float* a, const float* b, const float* A_log, const float* dt_bias,
                 float* q, float* k, float* v, float* g, float* beta,
                 int64_t T, int n_kh, int n_vh, int d, int activation, float eps,
                 void* cuda_stream);

/*
 * gdn_decode - one token of the recurrence for each of `batch` independent
 * sequences (the decode step; [P413] "What changes" applied to T = 1), each
 * sequence with its own state:
 *     q, k        [batch][n_kh][d]       v, out   [batch][n_vh][d]
 *     g, beta     [batch][n_vh]          states   [batch][n_vh][d][d] (in/out)
 * Per sequence b and value head h this is gdn_recurrence over one token;
 * results agree with it to FP32 rounding (another summation order).
 * Supported: d == 128, n_vh == 3 * n_kh, 1 <= batch <= 65535; batch == 0 is a
 * no-op.  Device pointers owned by the caller; asynchronous on `cuda_stream`.
 */
int gdn_decode(const float* q, const float* k, const float* v,
               const float* g, const float* beta,
               float* states, float* out,
               int batch, int n_kh, int n_vh, int d, void* cuda_stream);

/*
 * gdn_out_norm - gated RMSNorm of the recurrence output to FP16 ([P413] "What
 * changes": gdn_out_norm_kernel writes the FP16 copy y_h).  Per (t, h) row:
 *     r = 1 / sqrt(mean_j out[t][h][j]^2 + eps)
 *     y_fp16[t][h][j] = fp16_rn( out[t][h][j] * r * w[j] * silu(z[t][h][j]) )
 * computed in FP32 with one round-to-nearest-even to binary16 at the end.
 * Supported: d == 128, any n_vh >= 1, eps >= 0.  T == 0 is a no-op.
 */
int gdn_out_norm(const float* out, const float* z, const float* w, float eps,
                 uint16_t* y_fp16, int64_t T, int n_vh, int d, void* cuda_stream);

/*
 * gdn_recurrence_norm - gdn_recurrence followed by gdn_out_norm of its output, in
 * one call: out (FP32, written as by gdn_recurrence) and y_fp16 (the same bits
 * gdn_out_norm would give for that out).
 *
 * GDN_SEQUENTIAL: with `out` NULL (or the option GDN_OPT_NORM_IN_LAUNCH set to
 * 1) the norm is fused into the scan's epilogue ([P413] "What changes": the FP32
 * output is only the norm's input): one cooperative launch whose CTAs exchange
 * each row's partial sums of squares through global memory, so y comes from the
 * outputs while they are still on chip and, with `out` NULL, the FP32 output is
 * never written.  Otherwise the scan and the norm are two launches, which on
 * GB300 take less time (the scan is ALU-bound; the fused form saves the FP32
 * output's HBM traffic, not time).  The fused form needs the 8 n_kh CTAs
 * resident at once (n_kh <= SMs / 8); beyond that `out` is required.
 * GDN_CHUNKED with the tensor-memory form (GDN_PRODUCTS_TMEM, the default): with
 * `out` NULL (or the option GDN_OPT_NORM_IN_LAUNCH set to 1) the norm is in the
 * scan's output epilogue.  Each scan CTA holds whole 128-column rows of its value
 * head, so it forms every row's sum of squares itself, in gdn_out_norm's order,
 * and writes y from the outputs while they are on chip; with `out` NULL the FP32
 * output is never written.  One launch per 2048-token super-block.  Otherwise
 * the recurrence, then the norm's own launch, per super-block (with the FP32
 * output stored this takes less time on GB300).  If the tensor-memory launch
 * cannot be resident on the SMs available, the call takes the forms below and
 * then needs `out`.
 * GDN_CHUNKED with the other product forms: the norm of each super-block is
 * launched after its recurrence (`out` required).  With the option
 * GDN_OPT_NORM_IN_LAUNCH set to 1 and the one-launch warp-MMA form, the norm
 * instead runs inside that launch, on the SMs that prepare the chunks, as the
 * scan finishes each (chunk, key head), reading the output back from L2 (same
 * bits; on GB300 slower, those SMs cannot stream the norm's traffic as fast as
 * the scan produces it).
 *
 * Arguments as the two calls'; z, w and y_fp16 16-byte aligned; y_fp16 may
 * overlap no other argument.
 */
int gdn_recurrence_norm(const float* q, const float* k, const float* v,
                        const float* g, const float* beta,
                        float* state_inout, float* out,
                        const float* z, const float* w, float eps, uint16_t* y_fp16,
                        int64_t T, int n_kh, int n_vh, int d, int mode,
                        void* cuda_stream);

/*
 * gdn_recurrence_chunked_noalloc - gdn_recurrence(..., GDN_CHUNKED, ...) without
 * any device allocation.  The pages have no counterpart to this entry point.
 *
 * For callers that cannot let a library call cudaMalloc: for example a serving
 * process that reserved all of the GPU's memory for its own arena at start-up,
 * where an allocation from inside a library fails or fragments that arena, or a
 * latency-critical path that must not take cudaMalloc's implicit device
 * synchronisation.  The caller passes inputs and outputs exactly as for
 * gdn_recurrence (same layouts, same alignment rules, device pointers it owns).
 *
 * Scratch: a fixed 12,976,128-byte array (one 512-token super-block of prep
 * records for up to 96 value heads) and a 4-byte status word, both in the
 * library's static device memory.  Calls with n_vh > 96 are rejected with
 * GDN_ERR_UNSUPPORTED and a message saying so.
 *
 * Set-up: the CUDA runtime places that static memory on a GPU when it loads the
 * library's device code there.  Under its default lazy module loading
 * (CUDA_MODULE_LOADING=LAZY) that happens at this entry point's first call on
 * each device, which looks up the array's and the status word's device
 * addresses and has the runtime load the kernels it launches (about 13 MB of
 * device memory in all, kept until the process exits).  So make the first call
 * on each device, with that device current, before the caller reserves its
 * arena (or run with CUDA_MODULE_LOADING=EAGER, which loads everything when the
 * library is loaded) and before any stream capture.  A call with T == 0 does
 * that set-up and nothing else (the pointers are not used and may be NULL).
 *
 * Every call in the process shares the one array per device and leaves its last
 * contents there; each call writes every scratch word it reads before reading
 * it, so no clearing is needed, but two calls whose kernels overlap on a GPU
 * (different streams, or different host threads) race on the array and corrupt
 * each other's results: serialise them.  A bounded wait that gives up in these
 * kernels sets the status word, which gdn_device_status() reads and clears
 * (without allocating anything).  Results are bit-identical to gdn_recurrence's
 * chunked mode with GDN_OPT_CHUNK_PRODUCTS = GDN_PRODUCTS_MMA (whose kernels this
 * entry point runs) and within the same 2e-6 bound of its default form.
 */
int gdn_recurrence_chunked_noalloc(const float* q, const float* k, const float* v,
                                   const float* g, const float* beta,
                                   float* state_inout, float* out,
                                   int64_t T, int n_kh, int n_vh, int d,
                                   void* cuda_stream);

/*
 * Process-wide options.  The library reads no environment variable: the A/B
 * forms of its kernels and its failure-path test hooks are chosen here.  A value
 * applies to every call that starts after gdn_set_option returns; do not change
 * an option while another thread is inside a call of this library.  The defaults
 * are the production forms.  The pages have no counterpart to these options.
 */
typedef enum gdn_option {
    /* How GDN_CHUNKED computes the chunk's products: GDN_PRODUCTS_TMEM (default:
     * one CTA per value head keeps the state in tensor memory and every product is
     * a split-TF32 tcgen05 MMA; one cooperative launch per super-block with the
     * prep beside it, when the value heads leave at least n_kh SMs, else the
     * GDN_PRODUCTS_MMA form),
     * GDN_PRODUCTS_MMA (split-TF32 warp-level MMAs), GDN_PRODUCTS_FMA (packed
     * FP32 FMAs) or GDN_PRODUCTS_TCGEN05 (the state products as split-TF32 tcgen05
     * MMAs, 16 value columns per CTA; always two launches per super-block).  All
     * meet the same 2e-6 bound; they round differently, so their bits differ. */
    GDN_OPT_CHUNK_PRODUCTS = 1,
    /* 1 (default): the chunk prep runs beside the scan in one cooperative launch
     * when the device has SMs to spare for it; 0: a prep launch, then a scan
     * launch (GDN_PRODUCTS_TMEM has no two-launch form: the GDN_PRODUCTS_MMA
     * scan runs then).  Same bits either way for a given scan. */
    GDN_OPT_CHUNK_ONE_LAUNCH = 2,
    /* gdn_recurrence_norm: 0 (default) launches the norm after the recurrence
     * when `out` is given (after each super-block in GDN_CHUNKED); 1 norms inside
     * the recurrence's launch (GDN_CHUNKED: in the tensor-memory scan's epilogue,
     * or on the prep SMs of the warp-MMA one-launch form; GDN_SEQUENTIAL: in the
     * scan's epilogue).  Without `out` the fused forms run either way.  Same bits
     * either way. */
    GDN_OPT_NORM_IN_LAUNCH = 3,
    /* GDN_SEQUENTIAL: state rows per thread, 16 (default) or 8.  Same bits. */
    GDN_OPT_SEQ_ROWS_PER_THREAD = 4,
    /* GDN_PRODUCTS_TMEM: CTAs that run the chunk prep beside the scan (0, the
     * default: 4 n_kh; else this many), capped by the SMs the scan leaves and at
     * least n_kh.  Same bits either way. */
    GDN_OPT_CHUNK_PREP_CTAS = 5,
    /* Failure-path test hook: the prep task (chunk * n_kh + key head, in every
     * super-block) whose hand-off flag the one-launch chunked kernel never
     * publishes, so the scan CTAs waiting for it give up their bounded wait and
     * gdn_device_status() returns GDN_ERR_TIMEOUT; -1 (default) withholds none. */
    GDN_OPT_TEST_WITHHOLD_PREP_TASK = 101,
    /* Failure-path test hook: 1 makes the chunked scratch allocation fail as a
     * failed cudaMalloc would (GDN_ERR_ALLOC, nothing launched); 0 (default). */
    GDN_OPT_TEST_FAIL_SCRATCH_ALLOC = 102
} gdn_option;

enum { GDN_PRODUCTS_MMA = 0, GDN_PRODUCTS_FMA = 1, GDN_PRODUCTS_TCGEN05 = 2, GDN_PRODUCTS_TMEM = 3 };

/* Sets `option` to `value`: GDN_OK, or GDN_ERR_INVALID_ARG for an unknown option
 * or a value it does not allow (the option is then unchanged). */
int gdn_set_option(int option, int value);

/* Stores the current value of `option` in *value: GDN_OK or GDN_ERR_INVALID_ARG. */
int gdn_get_option(int option, int* value);

/* Message for the calling thread's last non-OK status ("" if none). */
const char* gdn_last_error(void);

/*
 * Synchronises `cuda_stream`, then reads and clears the current device's
 * status words (the allocating entry points' and gdn_recurrence_chunked_noalloc's):
 * GDN_OK, or GDN_ERR_TIMEOUT if a kernel gave up a bounded wait since the last
 * read, or GDN_ERR_CUDA if the stream reports an error.  Allocates nothing.
 */
int gdn_device_status(void* cuda_stream);

/*
 * Frees the chunked-mode scratch and the fused-norm scratch of `device` (a CUDA
 * device ordinal).  The caller must ensure no call is still running on it.  The
 * next call that needs them allocates them again.  Returns GDN_OK (also if
 * nothing was allocated).
 */
int gdn_release_scratch(int device);

/*
 * Diagnostic: fill the current device's chunked-mode scratch (allocating it
 * first, sized for n_vh value heads) with the 32-bit pattern `bits`, e.g.
 * 0x7fc00000 (a quiet NaN), on `cuda_stream`.  A chunked call that followed and
 * read a scratch word its prep kernel had not written would propagate the
 * pattern into its results; the tests use this to show it never does.
 */
int gdn_poison_scratch(uint32_t bits, int n_vh, void* cuda_stream);

/* Bytes of chunked-mode scratch a device holds once allocated. */
size_t gdn_chunked_scratch_bytes(int n_vh);

/* Number of kernels this library has launched in this process (all devices). */
uint64_t gdn_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* GDN_H */

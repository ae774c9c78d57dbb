/*
 * fuse.h -- C ABI of the fused-chain library for GB300 (sm_103a).
 *
 * The library fuses a chain of small memory-bound operators into one kernel
 * that reads its inputs from HBM once, applies every step in registers and
 * writes once.  Kernels are generated at run time with their sizes, vector
 * width and tail handling baked into the source, compiled with NVRTC for
 * sm_103a and cached ("DeepJIT ... 串行小核墙", sections 3.1-3.3: source built
 * at run time, NVRTC, driver-API loading, constants baked in, a cache keyed
 * by source + arch + options).
 *
 * Conventions ("算子与运行时", section 4.1 and 4.3: C linkage, raw pointers, an
 * explicit stream, an int status and no exceptions; "DeepJIT" section 6.5:
 * pointer ownership):
 *   - Every call returns FUSE_OK (0) or a negative FUSE_E_* code; the
 *     message for the last failure on the calling thread is fuse_last_error().
 *   - Tensor arguments are raw DEVICE pointers.  The caller owns them and
 *     keeps them alive until the work on `stream` has finished (with PyTorch:
 *     hold the tensor, or record_stream it).
 *   - `stream` is a cudaStream_t / CUstream passed as void* (NULL = the
 *     legacy default stream).  Calls enqueue work and return without
 *     synchronising the device or the stream.
 *   - The library owns compiled modules.  They stay loaded for the life of
 *     the process ("DeepJIT" section 6.4: never unload a module a stream may
 *     still be running); fuse_release() frees only the handle.
 *   - Kernels are built for sm_103 only; another device gives FUSE_E_ARCH.
 *   - Code generation and NVRTC compilation need no GPU; the first call on a
 *     device loads the module there.  Compilation happens once per distinct
 *     source (50-500 ms) and is never repeated for a cached shape.
 *   - Thread safety: all calls may be made from several threads; compiles
 *     are serialised internally.
 */
#ifndef FUSE_H
#define FUSE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { FUSE_F32 = 0, FUSE_F16 = 1, FUSE_BF16 = 2 } fuse_dtype;

enum {
  FUSE_OK = 0,
  FUSE_E_SPEC = -1,    /* malformed op-chain spec */
  FUSE_E_SHAPE = -2,   /* sizes inconsistent or out of range */
  FUSE_E_DTYPE = -3,   /* unsupported dtype combination */
  FUSE_E_NULL = -4,    /* a required pointer is NULL */
  FUSE_E_ARCH = -5,    /* the current device is not sm_103 */
  FUSE_E_COMPILE = -6, /* NVRTC failed; the log is in fuse_last_error() */
  FUSE_E_CUDA = -7,    /* a CUDA driver call failed, or no driver/device */
  FUSE_E_ARG = -8      /* another invalid argument (count, handle, ...) */
};

typedef struct fuse_chain* fuse_handle;

/* ------------------------------------------------------------------------
 * Elementwise chains ("DeepJIT" sections 3.2, 4.1, 4.2; "算子与运行时" 2).
 *
 * spec: "[shuffle:G;]op;op;..." with
 *   add | mul          x = x (+|*) in_j: consumes the next input tensor, whose
 *                      dtype is the chain's dtype at that op
 *   scale:<c>          x = x * c, c the fp32 nearest the literal
 *   relu               x = x > 0 ? x : 0   (NaN and -0 give +0)
 *   sigmoid            x = 1 / (1 + exp(-x))
 *   exp                x = exp(x)
 *   exp:fast, sigmoid:fast   the same, opt-in per expression, with exp taken
 *                      as the hardware's 2^t (ex2.approx, flush to zero) on
 *                      t = x * log2(e) in fp32: a relative error of up to
 *                      (1.25 |x| + 3) * 2^-24, results below 2^-126 flushed
 *                      ("DeepJIT" section 6.3: intrinsics per expression,
 *                      once validated); the accurate forms use CUDA's expf
 *   cast:f16|bf16|f32  round x to that dtype; later tensors and the output
 *                      take it
 *   shuffle:G          (first item only) ChannelShuffle of input 0 with G
 *                      groups over an NCHW shape: output channel j*G + i reads
 *                      input channel i*(C/G) + j ("算子与运行时", section 2)
 * Every step runs in fp32 registers; only casts and the final store round.
 * A spec with no ops (only a shuffle, or empty) copies input 0 bit for bit.
 *
 * At most 1024 ops and 128 input tensors; 1 <= G <= 2^20 (FUSE_E_SPEC).
 * shape/ndim: the tensor shape (1..8 dims, contiguous, row-major); with a
 *   shuffle it must be 4-D NCHW with C divisible by G.  Up to 2^40 elements
 *   (FUSE_E_SHAPE).
 * in_dtype: dtype of input 0.
 * out: receives the handle.  Returns FUSE_E_SPEC/SHAPE/DTYPE/COMPILE on
 *   error (no handle is made).
 */
int fuse_compile(const char* spec, const int64_t* shape, int ndim, fuse_dtype in_dtype,
                 fuse_handle* out);

/* Number of input tensors the chain takes and the dtype of its output. */
int fuse_num_inputs(fuse_handle h, int* n_in, fuse_dtype* out_dtype);

/* dtype of each input (dts has room for n_in entries). */
int fuse_input_dtypes(fuse_handle h, fuse_dtype* dts, int cap);

/* Launch the chain: inputs[0..n_in) and output are device pointers to
 * contiguous tensors of the compiled shape.  Pointers that are all 16-byte
 * aligned take the 128-bit vector kernel, otherwise the scalar kernel of the
 * same module ("DeepJIT" section 4.2).  The output must not overlap an input
 * unless it is the same pointer as an input that is read at the same index
 * (not input 0 of a shuffled chain). */
int fuse_launch(fuse_handle h, const void* const* inputs, int n_in, void* output, void* stream);

/* Free the handle (the compiled module stays cached). */
int fuse_release(fuse_handle h);

/* Generated CUDA source of a chain, without compiling it.  Writes up to cap
 * bytes (NUL-terminated) and the full length to *len. */
int fuse_source(const char* spec, const int64_t* shape, int ndim, fuse_dtype in_dtype, char* buf,
                size_t cap, size_t* len);

/* Shape buckets ("DeepJIT", section 7.2: quantise dynamic shapes into a few
 * buckets so that the number of compiles stays bounded, and handle the
 * excess with a mask or a tail).  fuse_compile_bucket compiles a chain whose
 * leading dimension is only an upper bound: everything else (dims 1..ndim-1,
 * vector width, block size) is baked in, and the element count is a kernel
 * argument, so one compile serves every leading dimension up to shape[0]
 * with no padding.  fuse_launch_rows runs it on a tensor whose leading
 * dimension is rows (0 <= rows <= shape[0]; other tensors are read and
 * written only up to that size).  A handle from fuse_compile accepts only its
 * own shape[0] there.  fuse_bucket gives the smallest power of two >= n
 * (>= 1), a bucket size for callers that key compiled handles by bucket. */
int fuse_compile_bucket(const char* spec, const int64_t* shape, int ndim, fuse_dtype in_dtype,
                        fuse_handle* out);
int fuse_launch_rows(fuse_handle h, const void* const* inputs, int n_in, void* output,
                     int64_t rows, void* stream);
int fuse_source_bucket(const char* spec, const int64_t* shape, int ndim, fuse_dtype in_dtype,
                       char* buf, size_t cap, size_t* len);
int fuse_bucket(int64_t n, int64_t* bucket);

/* Warm-up list ("DeepJIT" sections 3.3 and 6.2: compile the common shapes
 * before serving, so that no launch ever compiles).  `list` holds one chain
 * per line:
 *     <spec> | <d0>,<d1>,... | f32|f16|bf16 [| bucket]
 * (the arguments of fuse_compile, or of fuse_compile_bucket with the fourth
 * field); blank lines and lines starting with '#' are skipped.  Every chain
 * is compiled, or loaded from the disk cache, into the library's cache on up
 * to `threads` host threads (0: one per core; at most 16); distinct chains
 * compile in parallel.  A later fuse_compile of the same chain, shape and
 * dtype then takes no compile.  *compiled and *cached (either may be NULL)
 * receive how many entries NVRTC compiled and how many were cached already
 * (in memory or on disk).  A line that does not parse returns FUSE_E_SPEC,
 * FUSE_E_SHAPE or FUSE_E_DTYPE with its line number in fuse_last_error();
 * compile errors as fuse_compile.  Needs no GPU. */
int fuse_warmup(const char* list, int threads, int* compiled, int* cached);

/* ------------------------------------------------------------------------
 * Residual add + RMSNorm + cast ("TeleTron", sections 3.3 and 4.2).
 * Per row r of [rows, hidden]:
 *   h = x + residual            (fp32)
 *   residual_out = dt(h)        (round to nearest even)
 *   ms = sum(h^2) / hidden      (fp32 accumulation)
 *   out = dt(h * (1 / sqrt(ms + eps)) * weight)
 * x, residual, out, residual_out: [rows, hidden]; weight: [hidden]; all of
 * dtype dt (f16, bf16 or f32).  residual_out may equal residual and out may
 * equal x (in place); other overlaps are not allowed.
 * rows >= 0 (0 is a no-op), 1 <= hidden <= 65536.
 */
int rmsnorm_residual(const void* x, const void* residual, const void* weight, void* out,
                     void* residual_out, int64_t rows, int64_t hidden, float eps, fuse_dtype dt,
                     void* stream);

/* ------------------------------------------------------------------------
 * RMSNorm -> Linear -> scale on the tensor cores ("TeleTron", section 4.2:
 * the RMSNorm factor computed in the block and used directly in the linear
 * layer's accumulation, followed by an elementwise scale):
 *   s_m = 1 / sqrt(sum_k x[m,k]^2 / K + eps)
 *   out[m, n] = scale * (s_m * sum_k x[m,k] * (gamma[k] * w[n,k]) + bias[n])
 * x [M, K], gamma [K], w [N, K] (K-major, the layout of a Linear weight),
 * bias [N] (may be NULL), out [M, N]; dt f16 or bf16 (accumulation fp32);
 * all tensors 16-byte aligned.
 * 0 <= M < 2^31 - 128 (TMA tile coordinates are 32-bit), N % 8 == 0,
 * 0 < K <= 2^20 with K % 8 == 0; FUSE_E_SHAPE otherwise.
 * The product runs on a weight with gamma folded in, w' = dt(w * gamma), so
 * the rounding of x * gamma falls on w * gamma instead (the same value in
 * exact arithmetic).  gamma NULL means gamma is already folded into w
 * (rmsnorm_linear_fold, once): one launch.  With gamma given, the call folds
 * it into a scratch copy of w allocated on the stream (from a per-device
 * pool the library keeps mapped; it holds what overlapping calls needed at
 * once) and freed on the stream after the product: two launches and N * K
 * elements of stream-ordered scratch, safe for concurrent calls on different
 * streams.  Every wait inside the kernel is bounded: a wait that
 * runs out records an error that fuse_device_error() reports instead of
 * hanging the device.
 */
int rmsnorm_linear(const void* x, const void* gamma, const void* w, const void* bias, void* out,
                   int64_t M, int64_t N, int64_t K, float eps, float scale, fuse_dtype dt,
                   void* stream);

/* w_out[n, k] = dt(w[n, k] * gamma[k]) for w [N, K]: gamma folded into the
 * weight once, for rmsnorm_linear's fast path (w_out may equal w). */
int rmsnorm_linear_fold(const void* w, const void* gamma, void* w_out, int64_t N, int64_t K,
                        fuse_dtype dt, void* stream);

/* Synchronise the current device and return (and clear) its error word: 0;
 * 1 if a bounded wait ran out; 2 if a kernel was launched with less shared
 * memory than its layout needs (it then returns before touching its barriers,
 * TMA or TMEM); 3 if a chain built with FUSE_DEBUG_BOUNDS met an index
 * outside its tensor. */
int fuse_device_error(int* code);

/* Exercise the failure path of the kernels' bounded waits: one warp waits
 * on an mbarrier that nothing arrives at, gives up after `spins` tries
 * (1..2^30; each kernel wait in the library uses 2^18, about a second) and
 * records code 1 in
 * the device error word, which fuse_device_error() then returns.  No fault,
 * trap or hang: the kernel ends and the context stays usable. */
int fuse_selftest_bounded_wait(int64_t spins, void* stream);

/* ------------------------------------------------------------------------
 * Residual add + LayerNorm + cast ("DeepJIT", section 4.3: one block per
 * row, mean and variance reduced in the block, then normalised in the same
 * pass over the data).  Per row r of [rows, hidden]:
 *   h = x (+ residual)              (fp32)
 *   residual_out = dt(h)            (when residual is given)
 *   mean = sum(h) / hidden, var = sum((h - mean)^2) / hidden
 *   out = dt((h - mean) / sqrt(var + eps) * gamma + beta)
 * residual and residual_out are both NULL (plain LayerNorm) or both given;
 * gamma (treated as 1) and beta (treated as 0) may be NULL.  Layouts, dtypes,
 * in-place rules and limits as rmsnorm_residual.
 */
int layernorm_residual(const void* x, const void* residual, const void* gamma, const void* beta,
                       void* out, void* residual_out, int64_t rows, int64_t hidden, float eps,
                       fuse_dtype dt, void* stream);

/* ------------------------------------------------------------------------
 * QKV split + transpose + rotate-half RoPE ("TeleTron", section 3.1: QKV
 * projection -> head split -> RoPE).
 * qkv: [tokens, 3, heads, head_dim] (q block, k block, v block per token).
 * q, k, v: [heads, tokens, head_dim].  Token t sits at position pos0 + t.
 * For i < head_dim/2, theta = (pos0 + t) * base^(-2i/head_dim):
 *   o[i]              = x[i] cos(theta) - x[i + head_dim/2] sin(theta)
 *   o[i + head_dim/2] = x[i + head_dim/2] cos(theta) + x[i] sin(theta)
 * on q and k; v is copied bit for bit.  cos/sin come from a table the
 * library builds on the device in fp64 and keeps (fp32, 2 * positions *
 * head_dim/2 * 4 bytes) per device, base and head_dim; it grows as larger
 * positions are asked for.  dt: f16, bf16 or f32.  head_dim even,
 * 2 <= head_dim <= 1024; heads >= 1 and heads * head_dim <= 2^20 (index
 * arithmetic within a token's row is 32-bit); 0 <= tokens <= 2^31 - 1; 0 <= pos0 and
 * pos0 + tokens <= 2^22 (every position below 2^22); FUSE_E_SHAPE otherwise,
 * FUSE_E_ARG unless base is finite and > 1.  One kernel is compiled per
 * (heads, head_dim, dt) on first use; the token count and pos0 are launch
 * arguments, so calls with other token counts compile nothing.
 */
int rope_qkv_split(const void* qkv, void* q, void* k, void* v, int64_t tokens, int heads,
                   int head_dim, int64_t pos0, float base, fuse_dtype dt, void* stream);

/* ------------------------------------------------------------------------
 * rope_qkv_split_noalloc -- the same operation as rope_qkv_split, for callers
 * that must not let the library allocate device memory or compile at run
 * time: a serving process whose device memory all belongs to its own caching
 * allocator or arena, code running while a stream is captured into a CUDA
 * graph (an allocation or the synchronisation it may bring is an error
 * there), loops that forbid allocation after start-up.  The pages have no
 * counterpart of this entry point; it is an addition of this library.
 *
 * Arguments, layouts and results as rope_qkv_split.  It calls no cudaMalloc,
 * cudaFree or allocating routine: the cos/sin rows of the call are built into
 * a fixed array inside the library's module (2^20 fp32 values, 4 MB, held on
 * every device that has loaded the library until the process exits), and its
 * kernels (the rows build and, per dtype, a 16-byte-vector and an
 * element-wise rotation) are compiled ahead of time.
 *   - tokens * head_dim must be <= 2^20, and pos0 + tokens <= 2^22, else
 *     FUSE_E_SHAPE.
 *   - All calls on a device share the array; each call rewrites the rows it
 *     uses first, so nothing needs clearing, but calls that overlap on the GPU
 *     (other streams, unordered threads) race on it: order them on one stream.
 *   - Every call looks up the array's address in the calling thread's
 *     current context and makes sure the entry point's kernels are loaded
 *     there.  CUDA loads modules and kernels lazily by default, and loading
 *     allocates device memory, so the FIRST call in a context (any dtype)
 *     does that set-up: make it before any stream capture begins and before
 *     an arena takes the remaining device memory.  Later calls allocate
 *     nothing, whatever their dtype.
 */
int rope_qkv_split_noalloc(const void* qkv, void* q, void* k, void* v, int64_t tokens, int heads,
                           int head_dim, int64_t pos0, float base, fuse_dtype dt, void* stream);

/* ------------------------------------------------------------------------
 * Detection-head decode ("DeepJIT" section 1.1: the sigmoid / exp / mul /
 * add / slice / concat / cast tail of a detection head, fused into one
 * kernel).
 * feats[s] (device): [1, na*no, H_s, W_s] of dtype in_dt, channel a*no + k.
 * hw (host): nscales pairs (H_s, W_s); strides (host): nscales floats;
 * anchors (host): nscales*na pairs (w, h).
 * out (device): fp32 [sum_s na*H_s*W_s, no]; row = off_s + a*H_s*W_s +
 * y*W_s + x with the scales concatenated in order; for p = sigmoid(feat):
 *   k = 0: (2p - 0.5 + x) * stride    k = 1: (2p - 0.5 + y) * stride
 *   k = 2: (2p)^2 * anchor_w          k = 3: (2p)^2 * anchor_h
 *   k >= 4: p
 * 1 <= nscales <= 8, 1 <= na <= 16, 5 <= no <= 1024, and per scale H_s,
 * W_s >= 1 with H_s*W_s <= 2^24 (FUSE_E_SHAPE); non-finite strides or
 * anchors are FUSE_E_ARG.  The strides and anchors are baked into the kernel
 * (a new set compiles a new kernel).
 */
int detect_decode(const void* const* feats, const int* hw, const float* strides,
                  const float* anchors, int nscales, int na, int no, fuse_dtype in_dt, void* out,
                  void* stream);

/* ------------------------------------------------------------------------
 * ChannelShuffle ("算子与运行时", section 2): out[n, j*g + i] =
 * in[n, i*(c/g) + j] for i < g, j < c/g, on contiguous NCHW; a bit-exact
 * copy of whole H*W planes.  c % groups == 0 (else FUSE_E_SHAPE), groups > 0
 * (else FUSE_E_ARG), n*c*h*w <= 2^40 (else FUSE_E_SHAPE); a zero dimension is
 * a no-op.  in and out must not overlap (in == out is FUSE_E_ARG).  One
 * kernel is compiled per (c, h, w, groups, dt) on first use (a second one
 * once n*c*h*w reaches 2^31, with 64-bit indices); n is a launch argument, so
 * calls with other batch sizes compile nothing.
 */
int channel_shuffle(const void* in, void* out, int64_t n, int64_t c, int64_t h, int64_t w,
                    int groups, fuse_dtype dt, void* stream);

/* ------------------------------------------------------------------------
 * Sequences replayed as one CUDA graph ("DeepJIT", section 5.3: launch the
 * fused kernels in order and record them with stream capture; section 3.1: a
 * graph removes launch overhead, fusion removes the memory round trips).
 *
 * fuse_graph_begin(stream) starts capturing `stream` (thread-local capture
 * mode); every library call on that stream until fuse_graph_end(stream, &g)
 * becomes a node of the graph instead of running.  fuse_graph_launch(g, s)
 * replays the whole sequence with one submission on any stream; the tensors
 * named in the captured calls must stay allocated while g may run.  Calls that
 * compile a kernel, load a module or build a RoPE table cannot run during a
 * capture: make each call once before capturing it (fuse_compile loads its
 * module when a device is present).  A failed capture returns FUSE_E_CUDA
 * from fuse_graph_end and leaves no graph.
 */
typedef struct fuse_graph* fuse_graph_handle;
int fuse_graph_begin(void* stream);
int fuse_graph_end(void* stream, fuse_graph_handle* out);
int fuse_graph_launch(fuse_graph_handle g, void* stream);
/* Number of nodes (kernel launches) recorded in g. */
int fuse_graph_nodes(fuse_graph_handle g, int64_t* nodes);
int fuse_graph_release(fuse_graph_handle g);

/* ------------------------------------------------------------------------
 * Diagnostics ("算子与运行时", section 6.5: per-operator counters).
 */
/* Message of the last failed call on this thread ("" if none).  For
 * FUSE_E_COMPILE it holds the NVRTC log. */
const char* fuse_last_error(void);

/* Process-wide counters since load (any pointer may be NULL): NVRTC
 * compiles and their total time, cache hits (in memory, or a CUBIN loaded
 * from FUSE_CACHE_DIR), kernel launches.
 * Environment: FUSE_CACHE_DIR (on-disk CUBIN cache, keyed by the generated
 * source, the NVRTC options, the library's kernel headers and the NVRTC
 * version; each file carries hashes of its key and of the CUBIN, a damaged or
 * foreign file is recompiled;
 * an unwritable directory is ignored), FUSE_NVRTC_OPTIONS (extra NVRTC
 * options, space-separated, part of the cache key), FUSE_VERBOSE=1 (print
 * generated sources), FUSE_PTXAS_VERBOSE=1 (register use per kernel),
 * FUSE_DEBUG_BOUNDS=1 (chains compiled from then on check every index against
 * its tensor before the access and record code 3 in the device error word,
 * skipping the access, instead of touching memory outside the tensors),
 * FUSE_PDL=0 (launch in plain stream order instead of with programmatic
 * dependent launch; read once per process).  Switches of the generated code,
 * read when a kernel is generated (FUSE_ROW_PREFETCH once per process) and so
 * part of its source and cache key: FUSE_CHAIN_PREFETCH=0 (no L2 prefetch of a chain CTA's first chunk
 * before the launch-order wait), FUSE_ROW_PREFETCH=0 (the same for the first
 * row of RMSNorm, LayerNorm and RoPE), FUSE_CHAIN_F32X2=0 (chains do their
 * adds and multiplies one element at a time instead of on packed fp32
 * pairs), FUSE_DETECT_TC and FUSE_DETECT_BLOCK (the detect decode's cells per
 * tile and threads per CTA), FUSE_LN_MAX_REGS (LayerNorm's register cap). */
int fuse_stats(int64_t* compiles, int64_t* cache_hits, int64_t* launches, double* compile_ms);

/* Number of SMs the library sizes persistent grids for on the current
 * device (152 on GB300), or 152 when no device is visible. */
int fuse_device_sms(int* sms);

#ifdef __cplusplus
}
#endif

#endif /* FUSE_H */

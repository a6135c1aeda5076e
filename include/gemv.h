/*
 * gemv.h -- C ABI of the GB300 (sm_103a) matrix-vector product library.
 *
 * The operation (TileLang Case Studies, Case B "Background"): B is an (n, k)
 * matrix stored row-major with leading dimension k, a is a (k,) vector, and
 *
 *     c[i] = sum_{j < k} B[i, j] * a[j]        for i < n.
 *
 * B and a are both IEEE binary16 (fp16) or both bfloat16.  Products and sums
 * are formed in fp32; the result is rounded once (nearest-even) to the output
 * type, which is the input type or fp32.  The summation order is not part of
 * the contract (it is fixed for a given shape, dtype and launch
 * configuration, so repeated calls are bitwise reproducible).
 *
 * Citations name a page and its section: "Case Studies" is the TileOps wiki
 * page "TileLang Case Studies"; "the DPLR pull request" is "[DPLR] A Tilelang
 * implementation of DPLR - #1069" (flash-linear-attention); "the
 * optimization guide" is "Optimizing TileLang Programs".
 *
 * Conventions shared by every entry point:
 *  - Device pointers are plain CUDA device addresses on the CURRENT device
 *    (cudaGetDevice at the time of the call).  The start of every buffer is
 *    classified with cudaPointerGetAttributes: device memory of another
 *    device and host memory (pinned, registered or pageable, even where the
 *    GPU could reach it) return GEMV_ERR_DEVICE before anything is
 *    launched; managed memory is accepted.  The caller owns every buffer,
 *    outputs included (preallocated, as the DPLR pull request passes its
 *    forward outputs to cut host time per call); the library never frees or
 *    retains them past the call.
 *  - Calls are asynchronous on `stream` (0 = the legacy default stream); the
 *    caller synchronizes before reading c.
 *  - Nothing throws across this boundary and nothing calls exit/abort: every
 *    failure is a negative status code (GEMV_ERR_*), and on failure nothing
 *    has been launched.  gemv_status_string() describes a code.
 *  - Thread-safe: the launch-configuration cache and workspace table are
 *    guarded internally.  Per-thread state: gemv_last_config, the last CUDA
 *    error code.
 *  - GEMV_LOG=1 in the environment (read once) prints one line on stderr
 *    for each launch configuration the planner builds (a key newly cached
 *    by gemv(), gemv_ex() or gemv_fused() without a forced configuration,
 *    or by gemv_prepare(); every gemv_plan() call):
 *      gemv: new config dev=D n=N k=K dtype=T aligned=A -> variant=V
 *            ctas=C warps_per_cta=W warp_split=S rows_per_warp=R unroll=U
 *            grid_split=G k_segment=L stages=NS smem_bytes=M
 *    on one line ("plan" and dev=-1 for gemv_plan()).  Nothing else is
 *    printed, with or without it.
 */
#ifndef GEMV_GB300_H_
#define GEMV_GB300_H_

#include <stdint.h>

#include <cuda_runtime_api.h> /* cudaStream_t */

#ifdef __cplusplus
extern "C" {
#endif

/* dtype codes: input type of B and a, and output type of c. */
enum {
  GEMV_F16 = 0,          /* fp16 B, a -> fp16 c */
  GEMV_BF16 = 1,         /* bf16 B, a -> bf16 c */
  GEMV_F16_OUT_F32 = 2,  /* fp16 B, a -> fp32 c */
  GEMV_BF16_OUT_F32 = 3  /* bf16 B, a -> fp32 c */
};

/* Status codes. */
enum {
  GEMV_OK = 0,
  GEMV_ERR_ARG = -1,     /* null pointer with n > 0 and k > 0, n < 0, k < 0, k > INT32_MAX */
  GEMV_ERR_DTYPE = -2,   /* unknown dtype code */
  GEMV_ERR_ALIAS = -3,   /* c overlaps B or a */
  GEMV_ERR_DEVICE = -4,  /* no CUDA device, the current device is not sm_103, or a buffer
                            is not in the current device's memory (or managed memory) */
  GEMV_ERR_CUDA = -5,    /* a CUDA call or launch failed; see gemv_last_cuda_error() */
  GEMV_ERR_CONFIG = -6,  /* a forced configuration is invalid for this shape */
  GEMV_ERR_ALIGN = -7,   /* B or a not 2-byte aligned, or c not aligned to its element */
  GEMV_ERR_NOMEM = -8,   /* the split-K workspace could not be allocated */
  GEMV_ERR_SCRATCH = -9  /* gemv_splitk_noalloc: segments * n exceeds GEMV_STATIC_SCRATCH_FLOATS */
};

/* Kernel variants (gemv_config.variant). */
enum {
  GEMV_VARIANT_AUTO = 0,         /* let the planner choose */
  GEMV_VARIANT_ROWS = 1,         /* rows stream as aligned 16-byte vectors; needs k % 8 == 0
                                    and B 16-byte aligned */
  GEMV_VARIANT_ROWS_GENERAL = 2, /* any k and any 2-byte-aligned B: each row is read as the
                                    aligned 16-byte blocks covering it, edge elements masked,
                                    and a is realigned in registers by the row's offset */
  GEMV_VARIANT_TILES = 3,        /* any alignment: CTAs take interleaved tiles of rows of one
                                    residue class (row index mod 8, so one block offset per
                                    CTA), a is staged pre-shifted, rows are split into
                                    warp_split slices combined in shared memory */
  GEMV_VARIANT_BULK = 4          /* the tiles variant's work split (one row per warp), with B
                                    staged in shared memory instead of registers: each warp
                                    keeps a ring of `stages` buffers of 32*unroll 16-byte
                                    blocks that 1-D bulk asynchronous copies (TMA,
                                    cp.async.bulk, no multicast) fill from global memory,
                                    completion tracked by one mbarrier per buffer.  The
                                    sm_103a form of the multi-stage shared-memory pipeline of
                                    B (TileLang Case Studies, Case B.1 "O3 Pipelined B
                                    Loads").  The planner picks it for B of 768 MiB or more
                                    when the tiles plan has one warp per row and the rows
                                    hold 6144 to 8191 elements; otherwise only when forced */
};

/* Launch overlap with the preceding work on the stream (gemv_config.overlap). */
enum {
  GEMV_OVERLAP_NONE = 0,      /* ordinary stream-ordered launch */
  GEMV_OVERLAP_PDL = 1,       /* (what gemv(), gemv_host() and calls without a configuration
                                 use) programmatic dependent launch: the kernel may be scheduled
                                 while the preceding kernel drains; it waits for that
                                 kernel's completion (and its memory) before reading or
                                 writing any global memory.  Before the wait it only asks L2
                                 to prefetch its first tile of B: a hint, which reads
                                 nothing into the kernel and needs no promise.  After it,
                                 a is staged first, then the first tile of B is loaded and
                                 L2 is asked for the second step of its rows */
  /* "Work still running on the stream", for the two promises below: every
     kernel launched on the stream after its last ordinary operation (a kernel
     launched without the programmatic-serialization attribute, a copy, a memset
     or an event wait).  This library's kernels let their successor start before
     they wait for their own predecessor, so a chain of them may all run at
     once; an ordinary operation completes only after everything before it. */
  GEMV_OVERLAP_PDL_PREFETCH_B = 2, /* as GEMV_OVERLAP_PDL, and each CTA streams its first tile
                                 of B into registers and asks L2 for the next step (bulk
                                 variant: its first ring buffers into shared memory) before
                                 waiting.  The caller guarantees
                                 that no work still running on the stream writes B (true
                                 for weights); a and c are still accessed only after the
                                 wait, so a is staged behind those loads.  Measured on
                                 GB300 it is slower than GEMV_OVERLAP_PDL on most shapes
                                 whose CTAs stream several row tiles (7168 x 16384 fp16:
                                 33.2 against 31.8 us per call back to back) and faster
                                 on a few small or bulk-variant ones */
  GEMV_OVERLAP_PDL_PREFETCH_BA = 3 /* as GEMV_OVERLAP_PDL_PREFETCH_B, and a is also read
                                 (staged) before waiting: the caller guarantees that no work
                                 still running on the stream writes B or a -- e.g. several
                                 GEMVs on one input vector (Q/K/V or gate/up projections).
                                 Only the writes of c wait for the predecessor */
};

/*
 * A launch configuration.  As input to gemv_ex()/gemv_plan(), a zero field
 * means "planner's choice".  As output, every field is filled in.
 *
 *  variant        GEMV_VARIANT_*.
 *  rows_per_warp  R: rows one warp streams side by side (1, 2 or 4; 1 for
 *                 the general variant).  The a-vector chunk read from shared
 *                 memory is reused across the R rows.  Tiles variant:
 *                 (R, unroll) is one of (1, 8), (1, 4), (2, 4), (4, 2).
 *                 Bulk variant: 1.
 *  warps_per_cta  W: 4, 8 or 16 warps per CTA.
 *  warp_split     Sw: warps of one CTA that share a row, each streaming a
 *                 contiguous slice of it; their partial sums are combined
 *                 in shared memory in a fixed order.  Divides W.
 *  grid_split     Sg: CTAs that share a block of rows, each over one k-segment.
 *                 Sg > 1 writes fp32 partials to a workspace and launches a
 *                 second kernel that adds them in segment order (split-K).
 *  ctas           total CTAs of the main kernel (row blocks x Sg).  Tiles
 *                 variant: row_blocks is the CTA count per k-segment, a
 *                 multiple of 8 unless k % 8 == 0 and B is 16-byte aligned.
 *  smem_bytes     dynamic shared memory per CTA (the staged a segment plus
 *                 the cross-warp partials; bulk variant: plus the warps'
 *                 ring buffers and their mbarriers).
 *  launches       kernels per call: 1, or 2 with split-K.
 *  k_segment      columns per k-segment (a multiple of 8 except when Sg == 1).
 *  row_blocks     number of row blocks (ctas / grid_split).
 *  unroll         U: 16-byte loads per lane issued back to back per row
 *                 (tiles variant: may be forced together with rows_per_warp).
 *  overlap        GEMV_OVERLAP_*.  Not part of the cached configuration: a
 *                 gemv_ex() call that sets only this field launches the
 *                 cached configuration of gemv() with the requested overlap.
 *  l2_prefetch    tiles variant: before streaming a tile, each warp asks the
 *                 L2 to prefetch its slice of the tile this many rounds
 *                 ahead (one bulk prefetch per row slice; 0 = none, at most
 *                 3; -1 forces 0 when forcing).
 *  stages         bulk variant: buffers in each warp's ring (2 .. 8; the
 *                 planner takes 2).  0 for the other variants.
 */
typedef struct gemv_config {
  int32_t variant;
  int32_t rows_per_warp;
  int32_t warps_per_cta;
  int32_t warp_split;
  int32_t grid_split;
  int32_t ctas;
  int32_t smem_bytes;
  int32_t launches;
  int64_t k_segment;
  int32_t row_blocks;
  int32_t unroll;
  int32_t overlap;
  int32_t l2_prefetch;
  int32_t stages;
  int32_t reserved;
} gemv_config;

/*
 * c = B @ a on the current device, asynchronously on `stream`.
 *
 * Source: Case Studies, Case B "Background" (the operation and its shapes:
 * B (n, k) row-major, a (k,)); the cached launch below is the remedy of
 * Case B.4 "forward() Python Closure Overhead" (Fix: build once, call the
 * built kernel) and Case E "Builder Function lru_cache" (Fix: cache the
 * builder's result per shape), where rebuilding per call cost 11-200 ms.
 *
 *  B      device pointer, n*k elements, row-major (row i starts at B + i*k).
 *         Must be 2-byte aligned; 16-byte alignment plus k % 8 == 0 selects
 *         the aligned-vector variant, anything else the general variant.
 *  a      device pointer, k elements, 2-byte aligned.
 *  c      device pointer, n elements of the output type, aligned to it; must
 *         not overlap B or a (GEMV_ERR_ALIAS).
 *  n, k   sizes: n >= 0, 0 <= k <= INT32_MAX.  n == 0 launches nothing and
 *         returns GEMV_OK.  k == 0 sets c to +0 (the empty sum).
 *  dtype  GEMV_F16, GEMV_BF16, GEMV_F16_OUT_F32 or GEMV_BF16_OUT_F32.
 *
 * The kernel is launched as a programmatic dependent launch
 * (GEMV_OVERLAP_PDL): it may be scheduled while the preceding kernel on the
 * stream drains, but reads and writes no memory before that kernel has
 * completed, so ordering is that of a plain launch.
 *
 * The first call for a (device, n, k, dtype, alignment) key builds and caches
 * the launch configuration; later calls are a lookup plus one launch (two
 * with split-K).  A split-K configuration uses a library-owned fp32
 * workspace of grid_split*n floats per (device, stream), allocated on first
 * need (cudaMalloc, which synchronizes the device) and kept, grow-only,
 * until gemv_release().  Use gemv_prepare() to do that before timing or
 * before capturing the stream in a CUDA graph.
 */
int gemv(const void *B, const void *a, void *c, int64_t n, int64_t k, int dtype,
         cudaStream_t stream);

/*
 * As gemv(), with a configuration forced field by field (zero fields left
 * to the planner; `overlap` is taken as given, so 0 is a plain launch).
 * Source: Case Studies, Case C "nsys Profiling with Autotune Contamination"
 * (Fix: disable autotune and fix the best config, so a trace holds only
 * steady-state launches of one configuration); grid_split > 1 is the
 * split-K pass plus reduce pass whose times Case C adds together.
 * `forced` may be NULL (same as gemv()).  An impossible
 * configuration (e.g. the aligned variant for k % 8 != 0, W not in
 * {4, 8, 16}, Sw not dividing W) returns GEMV_ERR_CONFIG.  Forced
 * configurations are not cached.  For tests and benchmarks.
 */
int gemv_ex(const void *B, const void *a, void *c, int64_t n, int64_t k, int dtype,
            const gemv_config *forced, cudaStream_t stream);

/* Activations of the fused epilogue. */
enum {
  GEMV_ACT_NONE = 0,
  GEMV_ACT_RELU = 1,    /* max(y, 0) */
  GEMV_ACT_SIGMOID = 2, /* 1 / (1 + exp(-y)) */
  GEMV_ACT_SILU = 3     /* y / (1 + exp(-y)) */
};

/* Element type of the epilogue's bias vector. */
enum { GEMV_BIAS_INPUT_TYPE = 0, GEMV_BIAS_F32 = 1 };

/*
 * Epilogue fused into the GEMV's single store (the register epilogue of the
 * TileLang optimization guide, "Epilogue Fusion"):
 *
 *     c[i] = act(alpha * (B @ a)[i] + beta * bias[i])
 *
 * computed in fp32 on the fp32 row total and rounded once to the output
 * type.  bias (n elements, device memory, not overlapping c) may be NULL.
 * alpha = 1, bias = NULL, activation = GEMV_ACT_NONE is plain gemv().
 */
typedef struct gemv_epilogue {
  float alpha;
  float beta;
  const void *bias;
  int32_t bias_dtype;  /* GEMV_BIAS_INPUT_TYPE (fp16/bf16 as B) or GEMV_BIAS_F32 */
  int32_t activation;  /* GEMV_ACT_* */
} gemv_epilogue;

/*
 * GEMV over a row-strided B with a fused epilogue.  Source: the optimization
 * guide, "Optimization Checklist" item 7 "Epilogue Fusion" (activation, bias
 * and scaling applied in registers before the single write-back).  The row
 * stride has no counterpart on the pages; it reads B in place where a caller
 * holds a padded matrix (the DPLR pull request's review notes that a
 * non-contiguous input read with assumed strides gives wrong results: here
 * the stride is an explicit argument).
 *
 *
 *     c[i] = act(alpha * sum_{j<k} B[i*ldb + j] * a[j] + beta * bias[i])
 *
 * ldb >= k is B's row stride in elements (row i starts at B + i*ldb); the
 * elements between k and ldb are never used (they may hold anything,
 * including NaN).  epilogue may be NULL (identity); config as in gemv_ex()
 * (may be NULL; may set `overlap`).  Same status codes as gemv(), plus
 * GEMV_ERR_ARG for ldb < k or an unknown activation/bias type,
 * GEMV_ERR_ALIGN for a misaligned bias and GEMV_ERR_ALIAS for a bias
 * overlapping c.  k == 0 gives act(beta * bias[i]) (the empty sum is 0).
 */
int gemv_fused(const void *B, int64_t ldb, const void *a, void *c, int64_t n, int64_t k, int dtype,
               const gemv_epilogue *epilogue, const gemv_config *config, cudaStream_t stream);

/*
 * Build and cache the configuration gemv() would use for (n, k, dtype) on
 * the current device, for B with the given alignment (b_aligned16 != 0:
 * 16-byte aligned), and reserve the split-K workspace for `stream` if the
 * configuration needs one.  Optional; gemv() does the same lazily.
 * Source: Case Studies, Case B.4 (Fix: compile once at init time, so the
 * call itself only launches) and Case E (Fix: cache per shape).
 */
int gemv_prepare(int64_t n, int64_t k, int dtype, int b_aligned16, cudaStream_t stream);

/*
 * The planner as a pure host function (no CUDA call): the configuration
 * chosen for (n, k, dtype) on a device with `sm_count` SMs, for B with the
 * given alignment class, with `forced` fields (may be NULL) honoured.
 * Writes *out and returns GEMV_OK, or an error code.  Source: Case Studies,
 * Case E (the builder as a pure function of its shape parameters, which is
 * what makes its result cacheable) and Case C "Why 74% and Not Higher"
 * (occupancy set by n over the SM count; here the planner sizes the grid
 * and the split for 152 SMs).
 */
int gemv_plan(int64_t n, int64_t k, int dtype, int b_aligned16, int sm_count,
              const gemv_config *forced, gemv_config *out);

/*
 * The configuration of this thread's last successful gemv/gemv_ex/
 * gemv_fused/gemv_splitk_noalloc launch.  Source: Case Studies, Case C (a
 * profile is only readable against the one configuration that ran).
 */
int gemv_last_config(gemv_config *out);

/*
 * Static description of a status code (never NULL).  No counterpart on the
 * pages, which raise Python exceptions; this ABI returns codes instead.
 */
const char *gemv_status_string(int status);

/*
 * The cudaError_t value behind this thread's last GEMV_ERR_CUDA (0 if
 * none).  No counterpart on the pages (see gemv_status_string).
 */
int gemv_last_cuda_error(void);

/*
 * Test hook: the next gemv/gemv_ex/gemv_host call on any thread returns
 * `status` without launching anything (0 clears it).  Host-side only; no
 * GPU fault is ever involved.  No counterpart on the pages: it makes every
 * failure path of a caller testable without faulting a GPU.
 */
int gemv_debug_inject(int status);

/*
 * Waits of the bulk variant that gave up (the bulk variant is the sm_103a
 * form of Case Studies, Case B.1 "O3 Pipelined B Loads"; its bounded waits
 * have no counterpart on the pages).  Each wait of a warp on one of its
 * ring buffers polls the buffer's mbarrier a bounded number of times (2^20);
 * a warp whose wait runs out stops issuing copies, waits (again bounded) for
 * the copies it already issued, writes NaN for the rows it owns and adds one
 * to a per-device counter.  This reads that counter for the current device
 * into *count (synchronously: it waits for the device's outstanding work),
 * then zeroes it if `reset` is nonzero.  Bits 0-30 of *count hold the
 * number of warps that gave up.  Bit 31 (GEMV_DRAIN_TIMEOUT) is set if a
 * warp's bounded wait for the copies it had already issued also ran out:
 * its CTA then exited with a bulk copy possibly still writing shared
 * memory, and the device's state is unspecified -- treat the device as
 * unusable for the rest of the process.
 */
#define GEMV_DRAIN_TIMEOUT 0x80000000u
int gemv_wait_timeouts(int reset, uint32_t *count);

/*
 * Test hook (no counterpart on the pages): the next launch of the bulk
 * variant (on any thread) gives each
 * ring wait `polls` polls instead of 2^20 (0 = every wait gives up at once,
 * exercising the path above without any hang); -1 clears it.  The waits
 * that drain copies already issued keep the full limit.
 */
int gemv_debug_wait_budget(int32_t polls);

/*
 * Free the library-owned workspaces and drop the configuration cache.  The
 * caller must make sure no call that uses them is still running on the GPU.
 * Source: the inverse of the per-shape cache of Case Studies, Case E (whose
 * lru_cache is bounded; this one is emptied explicitly).
 */
int gemv_release(void);

/*
 * End-to-end call for a matrix and vector held in host memory (no
 * counterpart on the pages, whose inputs are device tensors): copies B
 * (n*k elements) and a (k elements) from host to the caller's device buffers
 * B_dev and a_dev, runs gemv() into c_dev, and copies c back to c_host, all
 * asynchronously on `stream` (cudaMemcpyAsync; pinned host buffers make the
 * copies truly asynchronous).  All six buffers are caller-owned.  Same
 * status codes as gemv().
 */
int gemv_host(const void *B_host, const void *a_host, void *c_host, void *B_dev, void *a_dev,
              void *c_dev, int64_t n, int64_t k, int dtype, cudaStream_t stream);

/* Capacity, in floats, of the static split-K scratch of gemv_splitk_noalloc(). */
#define GEMV_STATIC_SCRATCH_FLOATS (1 << 20) /* 4 MiB per GPU */

/*
 * Split-K GEMV that allocates nothing.  The pages this library follows have
 * no counterpart of this entry point; it exists for callers that must not
 * allocate device memory while they run -- an inference engine's plugin code
 * that is forbidden to call cudaMalloc during execution, a serving loop where
 * a cudaMalloc would synchronize the device and stall its other streams, or
 * a process whose device memory is handed out up front by its own allocator.
 *
 * Computes the same c = B @ a as gemv() (same arguments, same status codes,
 * asynchronous on `stream`) with the tiles kernel split into `grid_split`
 * k-segments (2 .. 64), followed by the second pass that adds the fp32
 * partials in segment order.  The split actually used can differ from the
 * one requested: a k too short for that many segments of 8 columns uses
 * fewer, down to one (k <= 8), and a row longer than grid_split * 32768
 * columns uses ceil(k / 32768) segments (one segment stages at most 32768
 * columns of a).  The partials live in a file-scope device array of
 * GEMV_STATIC_SCRATCH_FLOATS floats that every GPU loading this library
 * holds until the process exits; a call whose split needs more than that
 * (segments * n floats, with two or more segments) returns GEMV_ERR_SCRATCH
 * without launching.  A single segment writes c directly and uses no
 * scratch, whatever n is.  No cudaMalloc, cudaFree or other allocating
 * routine is called.
 *
 * The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress, with that device current); make that first call
 * before any stream capture.  Every call on a device shares the one array:
 * calls whose kernels overlap on the GPU (other streams, other threads,
 * other host processes sharing the library's context) race on it and must
 * be serialized by the caller.  The array keeps the last call's partial
 * sums; nothing in it needs clearing, because each call writes every
 * partial it reads.
 */
int gemv_splitk_noalloc(const void *B, const void *a, void *c, int64_t n, int64_t k, int dtype,
                        int grid_split, cudaStream_t stream);

/* Storage types of gla_decode(). */
enum { GLA_F16 = 0, GLA_BF16 = 1, GLA_F32 = 2 };

/*
 * One decode step of gated linear attention (TileLang Case Studies, Case D
 * "Background") for bh independent heads:
 *
 *     S_new[i][j] = exp(gk[i]) * S[i][j] + k[i] * v[j]     (i < dk, j < dv)
 *     o[j]        = scale * sum_i q[i] * S_new[i][j]
 *
 * All tensors share the storage type `dtype` (GLA_F16, GLA_BF16 or GLA_F32);
 * the arithmetic is fp32, each S_new element is rounded once when stored and
 * o uses the unrounded values.  Layout per head h (device pointers, dense):
 * q, k, gk at h*dk; v, o at h*dv; S, S_new at h*dk*dv, row i, column j at
 * i*dv + j.  S_new may be S itself (in-place step) but not otherwise overlap
 * it; o overlaps nothing.  v, o, S, S_new 16-byte aligned and dv a multiple
 * of 8 (16-bit types) or 4 (fp32), dv / that <= 256; dk <= 4096.  dk == 0
 * writes o = 0.  Asynchronous on `stream`; same status codes as gemv().
 */
int gla_decode(const void *q, const void *k, const void *v, const void *gk, const void *S, void *S_new,
               void *o, int64_t bh, int64_t dk, int64_t dv, float scale, int dtype, cudaStream_t stream);

/* Kernel layouts of gla_decode_ex(). */
enum {
  GLA_VARIANT_AUTO = 0,     /* gla_decode()'s choice */
  GLA_VARIANT_CTA = 1,      /* a CTA of 256 threads takes G heads per round (G = 1 for large heads,
                               more for small ones: about 4 rows per thread): 16-byte column chunks
                               of 4 rows in flight per thread, row-block partials of o added in
                               shared memory */
  GLA_VARIANT_WARP = 2,     /* one warp per head: lanes own (row group, column chunk) pairs, 8 rows
                               in flight per lane, o reduced by warp shuffles; needs
                               dv * element size <= 512 bytes */
  GLA_VARIANT_PIPE = 3      /* GLA_VARIANT_CTA with the next round (its state, q, k, gk, v) copied
                               into a second shared-memory buffer by asynchronous copies while the
                               current round computes; needs dk * element size a multiple of 16,
                               q, k, gk 16-byte aligned, dk * dv * element size <= 32 KiB and its
                               two buffers within 110 KiB of shared memory.  S_new bit-identical to
                               GLA_VARIANT_CTA; o too where both take the same heads per round */
};

/* Flags of gla_decode_ex(). */
enum {
  GLA_PREFETCH_STATE = 1 /* the caller guarantees that no work still running on the stream (as
                            defined for GEMV_OVERLAP_PDL_PREFETCH_B) writes S: true when each layer
                            of a decoder owns its state and an ordinary operation (sampling, a copy)
                            separates one token's layers from the next token's.  The CTA layout then
                            requests its first state rows before waiting for the preceding kernel;
                            q, k, v, gk, S_new and o are still accessed only after the wait.  The
                            warp layout ignores the flag.  Without it, the pipelined layout only
                            asks L2 to prefetch its first state rows before the wait (a hint,
                            which reads nothing into the kernel) */
};

/*
 * Source: Case Studies, Case D "Background" (the same recurrence as
 * gla_decode()).  The layouts are this library's own: the page's decode
 * kernel is a warpgroup tensor-core pipeline, not a bandwidth-bound stream.
 *
 * gla_decode() with the kernel layout chosen by the caller (`variant`,
 * GLA_VARIANT_*) and launch flags (`flags`, GLA_PREFETCH_STATE or 0;
 * unknown bits return GEMV_ERR_ARG).  The automatic choice is GLA_VARIANT_PIPE
 * where the shape and alignment allow it, else GLA_VARIANT_CTA (both take
 * several small heads side by side per round; measured faster than a warp
 * per head on every workload tried).  GEMV_ERR_CONFIG for a layout the shape
 * does not allow; otherwise as gla_decode().  All layouts compute every S_new
 * element identically; o differs between the warp layout and the CTA layouts
 * only by the order of its fp32 sum.
 */
int gla_decode_ex(const void *q, const void *k, const void *v, const void *gk, const void *S, void *S_new,
                  void *o, int64_t bh, int64_t dk, int64_t dv, float scale, int dtype, int variant, int flags,
                  cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* GEMV_GB300_H_ */

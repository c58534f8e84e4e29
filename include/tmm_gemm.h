/*
 * tmm_gemm.h -- C ABI of the GB300 (sm_103a) FP32 matrix-product library.
 *
 * Every entry point computes the matrix product of "Tiling Hierarchy on GPUs"
 * (introduction and section "Inner Product"), C = A x B with A of M x K,
 * B of K x N and C of M x N, all row-major:
 *
 *     C[i*ldc + j] = sum_{k=0}^{K-1} A[i*lda + k] * B[k*ldb + j]
 *                                        for 0 <= i < M, 0 <= j < N.
 *
 * C is overwritten; it is never read (no alpha/beta scaling: the pages define
 * none, and "CMU DLSys Lecture 12" section 5 counts no initial read of C).
 * Elements of C outside the M x N window (the ldc - N gap of each row) are
 * not touched.  Summation order inside the kernels is not specified; results
 * agree with the exact product to FP32 rounding (each entry within about
 * sqrt(K) units of FP32 rounding of the terms it sums), and are exact whenever
 * every partial sum is exactly representable (for example small-integer
 * inputs with sums below 2^24).
 *
 * Arguments (all entry points):
 *   M, N, K      sizes, 0 <= size <= 2^31 - 1.  M == 0 or N == 0 is a no-op
 *                (no CUDA call is made).  K == 0 writes zeros to the M x N
 *                window of C (the empty sum).
 *   A, B         DEVICE pointers (cudaMalloc'd or any device-accessible
 *                memory of the current device) to FP32 row-major operands.
 *                Caller-owned; read only.  Pointers must be 4-byte aligned
 *                (natural float alignment).  Rows that all start on 16-byte
 *                boundaries (16-byte aligned base, leading dimension a
 *                multiple of 4) save a copy: on the FFMA path B stored K x N
 *                (and A stored K x M) is then read in place by TMA, where
 *                any other B (stored N x K, or with unaligned rows) and A
 *                stored K x M with unaligned rows are first restaged into a
 *                scratch copy with 16-byte rows (one more read and write of
 *                the operand); on the tensor-core path an operand stored
 *                K-major is then read in place as its own TF32 high part.
 *   lda, ldb     leading dimensions in elements: lda >= max(1, K),
 *                ldb >= max(1, N).
 *   C            DEVICE pointer to the FP32 row-major result, caller-owned,
 *                written only.  The M x N window of C must not overlap A or B.
 *   ldc          leading dimension of C in elements, ldc >= max(1, N).
 *   stream       CUDA stream (cudaStream_t) the work is enqueued on; NULL is
 *                the legacy default stream.  Every call is asynchronous: it
 *                returns once the kernel is enqueued; the caller synchronises.
 *
 * Memory: gemm_f32 and gemm_f32_ex take scratch from a stream-ordered memory
 * pool the library creates per device -- for a restaged operand (K x N
 * rounded up to a multiple of 4 floats for B, K x M likewise for A), and for
 * the partial sums of a small problem whose blocks reduce their tiles
 * together (two 64 x 256 slots per resident block at most, 40 MiB on GB300;
 * when that cannot be allocated the call splits the problem in a way that
 * needs none).
 * It is allocated on `stream` and freed on `stream` after the kernels that
 * read it, so calls on different streams never share it, and the pool keeps
 * up to 256 MiB of freed memory for later calls (the rest returns to the
 * device when the stream is synchronised).  No other entry point allocates
 * device or host memory per call.  All entry points
 * use the current CUDA device (cudaSetDevice) and are thread-safe.
 *
 * Return value: TMM_OK (0) when the work was enqueued, otherwise one of the
 * negative TMM_ERR_* codes below (TMM_ERR_CUDA also when the scratch of a
 * restaged operand cannot be allocated); argument errors are found before
 * anything is launched.  No exception crosses the ABI and nothing is
 * printed; tmm_last_error_string() gives a one-line description of the
 * calling thread's last failure.
 */
#ifndef TMM_GEMM_H
#define TMM_GEMM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t / CUstream, declared here so that this header
 * does not need the CUDA headers. */
typedef struct CUstream_st *tmm_stream_t;

#define TMM_OK 0
/* A size is negative or above 2^31 - 1, a leading dimension is shorter than
 * its row, a pointer is NULL while its matrix is non-empty or not 4-byte
 * aligned, or a byte offset would overflow int64. */
#define TMM_ERR_INVALID_ARG (-1)
/* The byte range spanned by C's M x N window overlaps the range spanned by
 * A's M x K window or B's K x N window. */
#define TMM_ERR_ALIAS (-2)
/* The current device is not a compute capability 10.3 (GB300-class) GPU. */
#define TMM_ERR_UNSUPPORTED_DEVICE (-3)
/* A CUDA runtime call or kernel launch failed (text in tmm_last_error_string). */
#define TMM_ERR_CUDA (-4)
/* Reported by tmm_check_device: a bounded wait inside a kernel ran out of
 * time, and results written since the last check are not valid. */
#define TMM_ERR_DEVICE_TIMEOUT (-5)
/* Reported by tmm_check_device of the bounds-checked debug build only (the
 * library compiled with -DTMM_BOUNDS_CHECK): a product kernel computed a
 * global address outside its matrix (or in a row gap) or a shared-memory
 * offset outside its slab; the access was skipped, and results written since
 * the last check are not valid.  The normal build never returns it. */
#define TMM_ERR_BOUNDS (-6)

/* The same status codes under the names of the product's boundary contract
 * (GEMM_ERR_*); each equals its TMM_ERR_* counterpart. */
#define GEMM_OK TMM_OK
#define GEMM_ERR_INVALID_ARG TMM_ERR_INVALID_ARG
#define GEMM_ERR_ALIAS TMM_ERR_ALIAS
#define GEMM_ERR_UNSUPPORTED_DEVICE TMM_ERR_UNSUPPORTED_DEVICE
#define GEMM_ERR_CUDA TMM_ERR_CUDA
#define GEMM_ERR_DEVICE_TIMEOUT TMM_ERR_DEVICE_TIMEOUT
#define GEMM_ERR_BOUNDS TMM_ERR_BOUNDS

/*
 * gemm_f32 -- the tiled FP32 product on the CUDA cores (FFMA, IEEE single
 * precision, one rounding per multiply-add).
 *
 * Follows the two-level tiling of "Tiling Strategies" sections 2-4 and "CMU
 * DLSys Lecture 12" section 5: each thread block owns one block tile of C,
 * stages K-slices of A and B in shared memory (a multi-stage ring, the
 * double buffer of "Tiling Strategies" section 3 made deeper), and each
 * thread accumulates a tile of C in registers as a sequence of outer products
 * ("Tiling Hierarchy on GPUs", sections "Register Tiling" and "Register
 * prefetching").  Tail tiles are handled with zero-filled masked loads and
 * masked stores (DLSys section 5).
 *
 * When the tile count leaves the last wave of blocks partly empty, the call
 * runs persistent and cooperative (one block per resident slot) and splits
 * the K range of the last tiles between pairs of blocks; with fewer tiles
 * than resident blocks, the K range of every tile is split over up to about
 * five consecutive blocks, each adding the next block's running sum, or --
 * with few tiles, or C without 16-byte rows -- over equal shares of all
 * blocks, which then reduce each tile together from their partial sums in a
 * fixed order.  Blocks meet through flags in library-owned device memory,
 * with a bounded wait (see tmm_check_device).  Up to 16 such calls may be in
 * flight at once (for example on different streams); results are
 * deterministic either way.
 */
int gemm_f32(int64_t M, int64_t N, int64_t K,
             const float *A, int64_t lda,
             const float *B, int64_t ldb,
             float *C, int64_t ldc,
             tmm_stream_t stream);

/*
 * gemm_f32_ex -- gemm_f32 with either operand read transposed:
 *     C = op(A) x op(B),  op(A) = A   (transa = 0, A stored M x K, lda >= max(1, K))
 *                                 A^T (transa = 1, A stored K x M, lda >= max(1, M))
 *                         op(B) = B   (transb = 0, B stored K x N, ldb >= max(1, N))
 *                                 B^T (transb = 1, B stored N x K, ldb >= max(1, K)).
 * transa = 1, transb = 0 is the layout of "CMU DLSys Lecture 12" section 4,
 * C_ij = sum_k A_ki B_kj.  Only the way the operands reach the k-major
 * shared-memory slabs changes with the layout: A stored K x M is copied by
 * TMA, B stored N x K is first transposed into a K x N scratch copy (see
 * Memory above); the register tiles, scheduling and contract are gemm_f32's.
 * TMM_ERR_INVALID_ARG also for transa or transb not 0 or 1.
 */
int gemm_f32_ex(int transa, int transb,
                int64_t M, int64_t N, int64_t K,
                const float *A, int64_t lda,
                const float *B, int64_t ldb,
                float *C, int64_t ldc,
                tmm_stream_t stream);

/*
 * gemm_f32_naive -- one output per thread, each walking a row of A and a
 * column of B straight from global memory ("Tiling Strategies" section 2,
 * "The Problem"; "CMU DLSys Lecture 12" section 1 for the bounds-checked
 * one-thread-per-output launch).  Kept as the untiled contrast; the sum for
 * each output is accumulated with fmaf in ascending k.
 */
int gemm_f32_naive(int64_t M, int64_t N, int64_t K,
                   const float *A, int64_t lda,
                   const float *B, int64_t ldb,
                   float *C, int64_t ldc,
                   tmm_stream_t stream);

/*
 * gemm_f32_tc3 -- the same product on the tcgen05 tensor cores, with each FP32
 * operand split into two TF32 values, x = hi + lo (hi: x with its low 13
 * mantissa bits cleared; lo: the exact remainder rounded to TF32), and
 *     A B ~ A_hi B_hi + A_hi B_lo + A_lo B_hi
 * accumulated in FP32: each 256 values of K in tensor memory, the chunks
 * added in FP32 registers (the dropped A_lo B_lo term is about 2^-22 of each
 * product; normwise error about 2e-6 at any K).  An operand stored K-major
 * (A as M x K here) whose rows start on 16-byte boundaries is read in place as
 * its own hi (the tensor core ignores the low 13 bits of an FP32 word), so
 * only its lo is written to the workspace.  The pages do not go beyond FP32 FMA units ("CMU
 * DLSys Lecture 12" section 6 notes that tensor instructions change the
 * implementation); the tiling is that of section 5 with the register tile
 * replaced by a tensor-memory accumulator.  The tiles of a partial last wave,
 * and every tile of a problem with few tiles, are split along K into parts
 * that add each other's partial sums in a fixed order (bounded waits, see
 * tmm_check_device), so results are deterministic.  Same contract as
 * gemm_f32, plus:
 *   workspace        DEVICE pointer, 256-byte aligned, caller-owned, at least
 *                    gemm_f32_tc3_workspace_size(M, N, K) bytes; holds the
 *                    split operands (its contents are scratch, not preserved);
 *                    it must not overlap A, B or C.
 *   workspace_bytes  its size.
 * TMM_ERR_INVALID_ARG if the workspace is missing, short or misaligned (or
 * its size does not fit in size_t), TMM_ERR_ALIAS if it overlaps an operand.
 * Calls sharing one workspace must not overlap on the GPU.
 *
 * Ordering assumption: the K-parts of a split tile are consecutive work items,
 * and a part only ever waits (bounded) for a part that was scheduled before
 * it.  The product kernel is not a cooperative launch, so this relies on the
 * GPU starting a grid's blocks in block order, which CUDA does in practice but
 * does not guarantee.  Should the blocks start out of order (for example with
 * other kernels holding SMs), a wait can run into its time limit; the call
 * then reports TMM_ERR_DEVICE_TIMEOUT through tmm_check_device instead of
 * hanging.  As for gemm_f32, up to 16 calls may be in flight at once.
 */
int gemm_f32_tc3(int64_t M, int64_t N, int64_t K,
                 const float *A, int64_t lda,
                 const float *B, int64_t ldb,
                 float *C, int64_t ldc,
                 void *workspace, size_t workspace_bytes,
                 tmm_stream_t stream);

/* gemm_f32_tc3 with either operand read transposed (transa, transb as for
 * gemm_f32_ex); the split pre-pass reads the operands in their stored layout.
 * Same workspace size as gemm_f32_tc3. */
int gemm_f32_tc3_ex(int transa, int transb,
                    int64_t M, int64_t N, int64_t K,
                    const float *A, int64_t lda,
                    const float *B, int64_t ldb,
                    float *C, int64_t ldc,
                    void *workspace, size_t workspace_bytes,
                    tmm_stream_t stream);

/* Workspace bytes gemm_f32_tc3 needs for an M x N x K product (0 for an empty
 * product or sizes out of range; SIZE_MAX when the count does not fit in
 * size_t):  4 Kp (2M + 2N) rounded to 256-byte sections, Kp = K rounded up to
 * a multiple of 32. */
size_t gemm_f32_tc3_workspace_size(int64_t M, int64_t N, int64_t K);

/*
 * gemm_f32_tc3_noalloc -- gemm_f32_tc3 for callers that cannot allocate device
 * memory where they call it: code under a memory manager that owns the whole
 * device budget and forbids raw cudaMalloc, code on a latency-critical path
 * that cannot afford cudaMalloc's implicit synchronisation, or code where the
 * CUDA allocation API may not be called.  The pages have no counterpart; this
 * is a library convenience.  Same product, contract and status codes as
 * gemm_f32_tc3 (inputs and output are still the caller's device pointers),
 * but the split operands go to a fixed scratch array inside the library
 * instead of a caller-supplied workspace, and nothing is allocated:
 *   - the scratch is TMM_TC3_NOALLOC_SCRATCH_BYTES (64 MiB) of device memory
 *     set aside when the library's module is loaded; every GPU that loads it
 *     holds it until the process exits;
 *   - products needing more than that (gemm_f32_tc3_workspace_size(M, N, K)
 *     > TMM_TC3_NOALLOC_SCRATCH_BYTES, for example beyond about 2048^3) are
 *     rejected with TMM_ERR_INVALID_ARG and a message naming the sizes,
 *     before any CUDA call;
 *   - every call looks up the scratch's address on the current device
 *     (cudaGetSymbolAddress), so the address always belongs to the current
 *     context; the first call on a device may be the one that loads the
 *     library's device code there, so make it before any stream capture;
 *   - every call on a device uses the same scratch and leaves its contents
 *     behind; calls that overlap on the GPU (for example on two streams) race
 *     on it and must be serialised by the caller.
 */
#define TMM_TC3_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)
int gemm_f32_tc3_noalloc(int64_t M, int64_t N, int64_t K,
                         const float *A, int64_t lda,
                         const float *B, int64_t ldb,
                         float *C, int64_t ldc,
                         tmm_stream_t stream);

/*
 * tmm_check_device -- synchronise `stream`, then read and clear the current
 * device's status words.  Returns TMM_OK, or TMM_ERR_DEVICE_TIMEOUT when a
 * bounded wait inside gemm_f32 (between the blocks sharing a split tile, or
 * for a K-slice's TMA copy),
 * gemm_f32_tc3 (between the copy, tensor-core and epilogue roles of a block
 * or block pair), window_sum_f32 (for a tile's bulk copy) or softmax_rows_f32
 * (between the blocks sharing a row of more than 65536 columns) ran out of time
 * since the last check; results written since then are not valid.  The pages have no counterpart: this is the library's failure
 * detection ("CMU DLSys Lecture 12" section 2 only asks that API and launch
 * errors be checked).  TMM_ERR_CUDA if the synchronisation itself failed.
 * In the bounds-checked build, TMM_ERR_BOUNDS (which takes precedence) when a
 * range check of gemm_f32, gemm_f32_naive or gemm_f32_tc3 failed.
 */
int tmm_check_device(tmm_stream_t stream);

/*
 * tmm_testing_set_wait_hooks -- testing only; no counterpart in the pages.
 * drop_signal_block >= 0 makes that block of later split-tile launches of
 * gemm_f32 (and that split unit -- the K-part of a tile, numbered across the
 * call's split tiles -- of gemm_f32_tc3) skip raising its flags, so the one
 * waiting on it runs into the time limit; makes that block of later gemm_f32
 * launches whose operands are staged by TMA (rows on 16-byte boundaries) wait
 * for 16 bytes more than the first copy of each tile brings; makes that block of later window_sum_f32
 * launches (16-byte-aligned x) wait for 16 bytes more than its first tile
 * copy brings, and that block of later softmax_rows_f32 launches on rows of
 * more than 65536 columns skip counting itself in;
 * wait_limit_ns > 0 sets the limit of every bounded wait of these kernels
 * (default, and for values <= 0, 10 s).
 * Process-wide; pass (-1, 0) to restore the defaults.  Always TMM_OK.
 */
int tmm_testing_set_wait_hooks(int drop_signal_block, int64_t wait_limit_ns);

/*
 * tmm_testing_simt_plan -- testing only; no counterpart in the pages.  The work
 * split gemm_f32 would launch for an M x N x K product (1 <= sizes <= 2^31 - 1)
 * on 64 x 256 tiles (wide = 0) or 64 x 512 tiles (wide = 1), C taking 16-byte
 * stores or not (vec_c), the small-problem split reduced together allowed or
 * not (may_reduce), with `slots` resident blocks; no CUDA call is made.
 * out: HOST array of 9 values -- grid size, cooperative launch (0/1), partial-
 * sum slots (0: none), whole tiles processed first, K-slice units split after
 * them, and the unequal parts of a tile (parts, base, step, remainder; parts
 * 0 when not split that way).  TMM_ERR_INVALID_ARG for sizes out of range,
 * slots <= 0 or out NULL.
 */
int tmm_testing_simt_plan(int64_t M, int64_t N, int64_t K, int wide, int vec_c, int may_reduce,
                          int64_t slots, int64_t *out);

/*
 * tmm_testing_tc3_plan -- testing only; no counterpart in the pages.  The work
 * list gemm_f32_tc3 would launch for an M x N x K product (1 <= sizes <=
 * 2^31 - 1) on block pairs with 256 x 256 tiles (pairs = 1) or single blocks
 * with 128 x 256 tiles (pairs = 0), with `slots` resident pairs or blocks; no
 * CUDA call is made.  out: HOST array of 6 values -- tiles, work items, whole
 * tiles listed first, K-parts of each tile after them (1: none split),
 * 256-value chunks of K, 16-value K-slices.  TMM_ERR_INVALID_ARG for sizes out
 * of range, slots <= 0 or out NULL.
 */
int tmm_testing_tc3_plan(int64_t M, int64_t N, int64_t K, int pairs, int64_t slots,
                         int64_t *out);

/*
 * window_sum_f32 -- valid sliding-window sums, "CMU DLSys Lecture 12: GPU
 * Acceleration" section 3:
 *     y[i] = sum_{d=0}^{W-1} x[i + d],   0 <= i < n,
 * the page's window5 for W = 5.  x: DEVICE pointer to n + W - 1 floats; y:
 * DEVICE pointer to n floats; both caller-owned, 4-byte aligned, and they
 * must not overlap (TMM_ERR_ALIAS).  1 <= W <= 129, 0 <= n <= 2^40 (n == 0
 * is a no-op).  Each block stages its tile of inputs plus the W - 1 halo in
 * shared memory once (the page's cooperative loading); each sum starts from
 * 0 and adds the window in ascending d in FP32, the page's order.  Blocks
 * take tiles from a library-owned counter, so at most 16 calls may be in
 * flight at once.  Asynchronous on `stream`; no allocation.
 */
int window_sum_f32(int64_t n, int W, const float *x, float *y, tmm_stream_t stream);

/*
 * sum_f32 -- the tiled reduction of "Tiling Strategies" section 5 ("Tiling
 * Beyond GEMM": the input cut into chunks whose partial sums are accumulated
 * in shared memory):
 *     *out = sum_{i=0}^{n-1} x[i].
 * x: DEVICE pointer to n floats, 4-byte aligned; out: DEVICE pointer to one
 * float; workspace: DEVICE buffer of at least sum_f32_workspace_size(n) bytes,
 * 16-byte aligned, which holds one partial sum per chunk of the input and must
 * not overlap x (TMM_ERR_ALIAS).  All caller-owned; n == 0 writes 0.
 * 0 <= n <= 2^40.  Accumulates in FP32 in a fixed order (the chunks are fixed
 * pieces of x, taken by whichever block is free, and their partial sums are
 * added in chunk order), so repeated calls give the same bits; every term
 * passes through at most ceil(n / 2^25) + 54 additions, so
 * |*out - sum| <= (ceil(n / 2^25) + 54) 2^-24 sum |x[i]| (to first order).
 * Two kernel launches on `stream`, sharing a library-owned counter region
 * with at most 15 other calls in flight; no allocation.
 */
int sum_f32(int64_t n, const float *x, float *out, void *workspace, size_t workspace_bytes,
            tmm_stream_t stream);

/* Bytes of workspace sum_f32 needs for n elements (at most 64 KiB). */
size_t sum_f32_workspace_size(int64_t n);

/*
 * softmax_rows_f32 -- the two-pass softmax of "Tiling Strategies" section 5
 * (input chunks for the maximum and the sum, "max, then normalize" on the
 * same data), row by row:
 *     y[r*ldy + j] = exp(x[r*ldx + j] - m_r) / sum_k exp(x[r*ldx + k] - m_r),
 *     m_r = max_k x[r*ldx + k],   0 <= r < rows, 0 <= j, k < cols.
 * x, y: DEVICE pointers, row-major with row strides ldx, ldy >= max(1, cols)
 * floats, 4-byte aligned (16-byte alignment and strides that are multiples of
 * 4 select vector loads).  y may be x with ldy == ldx (in place); any other
 * overlap is TMM_ERR_ALIAS.  0 <= cols < 2^31; rows == 0 or cols == 0 is a
 * no-op.  Rows of up to 2048 columns are held in registers, up to 16384
 * columns staged in one block's shared memory, up to 65536 columns split over
 * a thread-block cluster whose blocks combine their partial maxima and sums
 * through distributed shared memory (each row read from HBM once); longer
 * rows are shared by several blocks that meet through library-owned global
 * memory with a bounded wait (see tmm_check_device), and are read twice, a
 * running (maximum, sum) pass and the normalise pass, the second read from L2.
 * Blocks take rows from library-owned counters (and share long rows through
 * library-owned memory), so at most 16 calls may be in flight at once.
 * FP32 throughout: exp by CUDA's expf, the sum in a fixed order, the
 * normalisation as a product with fl(1 / s) (in a cluster, with
 * fl(e^{m_c - m} / s) for the chunk maximum m_c).  A row whose maximum is +inf, or
 * all of whose entries are -inf, gives NaN (as the formula does); NaN inputs
 * are not supported.  Asynchronous on `stream`; no allocation.
 */
int softmax_rows_f32(int64_t rows, int64_t cols, const float *x, int64_t ldx, float *y,
                     int64_t ldy, tmm_stream_t stream);

/* One-line description of the calling thread's last failed call ("" if none).
 * The string is owned by the library and valid until the thread's next call. */
const char *tmm_last_error_string(void);

/* The names the product's boundary contract gives these two calls:
 * gemm_last_error_string is tmm_last_error_string, gemm_check_status is
 * tmm_check_device (same arguments, same results).  "CMU DLSys Lecture 12"
 * section 2: production code checks API and launch errors. */
const char *gemm_last_error_string(void);
int gemm_check_status(tmm_stream_t stream);

/* Library version as major*10000 + minor*100 + patch. */
int tmm_version(void);

#ifdef __cplusplus
}
#endif

#endif /* TMM_GEMM_H */

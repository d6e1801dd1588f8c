/*
 * repops.h -- C ABI of librepops: reproducible ("RepOps-style") operators for
 * verifiable training on one NVIDIA GB300 (sm_103a).
 *
 * Every operator returns the same bits on every call, whatever the tile size,
 * launch shape, operand storage (row- or column-major) or alignment: the order
 * of every floating-point operation is fixed by the definitions below, not by
 * the kernel's parallel schedule.
 *
 * Sources (page title, section):
 *   "Verde与RepOps：机器学习可验证委托与硬件无关确定性" (Verde and RepOps)
 *       §3.1 sources of hardware non-determinism (operation order, core count,
 *       memory layout/strides); §3.2 design principle (parallelise freely over
 *       order-independent dimensions, keep order-critical dimensions serial)
 *       and the matmul example; §3.3 IEEE-754 requirement; §2.3.2 checkpoint
 *       hashes as Merkle trees; §2.4 Merkle membership proofs.
 *   "Zoo Per-LLM Chain Soundness"
 *       §2 Definition "Aggregation rule", Lemma "Order independence within a
 *       batch"; §5 "Ordering subroutine", "Determinism of left-fold",
 *       "Update step"; §1 Background (batch hash = Merkle root); §6 table
 *       "Per-LLM chain block field layout" (bytes32 roots, sorted DIDs);
 *       §7 "Reproducibility test plan" (verify H(theta) = m).
 *
 * Conventions for every call
 *   - Pointers named "device" must be device memory of the current CUDA device
 *     (or managed memory); pointers named "host" must be host memory.
 *   - Calls are asynchronous on `stream` (0 = legacy default stream) unless a
 *     call says otherwise.  Argument checks run on the host before any launch;
 *     a call that returns an error launched nothing.
 *   - The library never takes ownership of a buffer.  It keeps no per-call
 *     state between calls, except the sticky device status word of the
 *     bounded waits (by default one word per device shared by every caller,
 *     or a word the caller owns, bound per host thread with
 *     repops_set_thread_status_word()) and, only where the caller asks for
 *     it, freed scratch its memory pool keeps mapped (see "Scratch memory").
 *   - Floating point is IEEE-754 binary32, round-to-nearest-even, subnormals
 *     kept (no flush-to-zero), no fused multiply-add, no tensor cores.
 *   - NaN results compare equal as a class (payload bits are not pinned);
 *     every other value, including signed zeros and infinities, is bit-exact.
 */
#ifndef REPOPS_H
#define REPOPS_H

#include <stdint.h>
#include <cuda_runtime_api.h>   /* cudaStream_t */

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes returned by every int-valued entry point. */
typedef enum {
    REPOPS_OK = 0,
    REPOPS_ERR_INVALID_ARG = -1,  /* null pointer, negative/overflowing size, bad leading dim */
    REPOPS_ERR_ALIAS = -2,        /* an output overlaps an input */
    REPOPS_ERR_ORDER = -3,        /* contributor order is not a permutation / duplicate IDs */
    REPOPS_ERR_CUDA = -4,         /* a CUDA runtime call failed (see repops_last_cuda_error) */
    REPOPS_ERR_TIMEOUT = -5,      /* a bounded device-side wait gave up (sticky, see below) */
    REPOPS_ERR_ALLOC = -6,        /* an allocation failed: stream-ordered scratch, or host memory */
    REPOPS_ERR_UNSUPPORTED = -7,  /* request outside the documented limits */
    REPOPS_ERR_BOUNDS = -8        /* checked build only: an access outside its buffer was skipped */
} repops_status;

/* Storage types of tensors whose elements the order-fixed binary32 path reads
 * or writes (see "Half-precision storage"). */
#define REPOPS_TYPE_F32 0    /* IEEE binary32 */
#define REPOPS_TYPE_F16 1    /* IEEE binary16 */
#define REPOPS_TYPE_BF16 2   /* bfloat16: the high 16 bits of a binary32 */

/* Build manifest: library version, target architecture, compile flags that
 * fix the arithmetic (-fmad=false, -ftz=false, -prec-div=true, ...), and the
 * GEMM tile configurations.  The role of a "KernelManifest" ("Zoo Per-LLM
 * Chain Soundness" §5 Setup): it names what produced the bits.  Static string. */
const char *repops_version(void);

/* Library infrastructure from here to the GEMM section: status codes,
 * failure detection of the library's bounded waits, scratch and host memory.
 * The pages describe none of these; they define no operation.
 *
 * Human-readable text for a status code.  Static string. */
const char *repops_status_string(int status);

/* The cudaError_t value of the most recent REPOPS_ERR_CUDA on this host
 * thread (0 if none). */
int repops_last_cuda_error(void);

/* Synchronises `stream`, then reads and clears the sticky device status word
 * of this host thread's launches: the word bound with
 * repops_set_thread_status_word(), else the library's shared word of the
 * current device.  *status_out = REPOPS_OK, or REPOPS_ERR_TIMEOUT if a
 * kernel's bounded wait on its own asynchronous copies gave up since the last
 * read (the output of that kernel is then undefined), or -- in the checked
 * build librepops_debug.so only, whose hot-path kernels (GEMM, mean + SGD,
 * Merkle) test every global access against its buffer's span and skip one
 * outside it -- REPOPS_ERR_BOUNDS if such an access was skipped.  Returns REPOPS_OK or
 * REPOPS_ERR_CUDA / REPOPS_ERR_INVALID_ARG (null status_out). */
int repops_device_status(cudaStream_t stream, int *status_out);

/* Scopes failure reports to the caller.  From this call on, every kernel that
 * this host thread launches through the library ORs its failure bits (bit 0:
 * a bounded wait gave up) into `word` -- 4 bytes of device memory of the
 * device the kernels run on, 4-byte aligned, owned, zeroed and read by the
 * caller -- instead of the device's shared word; repops_device_status() on
 * this thread then reads and clears `word`.  So a timeout on one caller's
 * stream is neither reported to nor cleared by another caller that has bound
 * its own word.  NULL goes back to the shared word.  The binding belongs to
 * the host thread only (thread-local) and is not read by the device until a
 * launch.  INVALID_ARG for a pointer that is not 4-byte aligned. */
int repops_set_thread_status_word(unsigned *word);

/* Failure-detection self-test: launches one kernel on `stream` whose thread
 * waits on an mbarrier phase that nothing completes, with a limit of limit_ns
 * nanoseconds (1 .. 2e9, else INVALID_ARG) of the device's global timer.  The
 * wait gives up and sets the sticky status word, as a GEMM whose copies never
 * landed would: the next repops_device_status reports REPOPS_ERR_TIMEOUT, and
 * the GPU context stays usable.  Nothing else is read or written. */
int repops_selftest_bounded_wait(int64_t limit_ns, cudaStream_t stream);

/* The same for the other kind of bounded wait: one kernel thread polls, as a
 * chained-split worker does for the previous worker's partial sums (acquire
 * loads with short sleeps), a flag word that nothing sets, gives up after
 * limit_ns (1 .. 2e9, else INVALID_ARG) and sets the status word: the next
 * repops_device_status reports REPOPS_ERR_TIMEOUT and the context stays
 * usable.  Nothing else is read or written. */
int repops_selftest_bounded_flag_wait(int64_t limit_ns, cudaStream_t stream);

/* Scratch memory.  Entry points that need device scratch (operand copies and
 * chained-split partial sums of the GEMM, Merkle level nodes, the staging
 * buffers of the host-buffer calls, ...) allocate it stream-ordered, on the
 * caller's stream, from a memory pool the library creates for each device
 * (one per CUDA context; the device's default pool is neither used nor
 * changed).  By default that pool, like the default one, hands freed memory
 * back at the next synchronisation: the library holds no memory between
 * calls.  A call made after a synchronisation then maps its scratch again,
 * which costs ~120 us of host time (on a GB300, synchronising after every
 * call: a 1536^3 GEMM 318 us a call against 242 us with its scratch kept).
 * Thread-safe.
 *
 * repops_scratch_set_keep_bytes: lets the current device's pool keep up to
 * `bytes` of freed scratch mapped across synchronisations (0, the default,
 * keeps none).  REPOPS_OK, or REPOPS_ERR_CUDA.
 * repops_scratch_release: hands back to the system the memory of the current
 * device's pool that no allocation holds (scratch of calls still in flight,
 * whose frees have not run on their streams yet, stays).  REPOPS_OK, or
 * REPOPS_ERR_CUDA.
 * repops_scratch_reserved_bytes: *bytes_out = device memory the current
 * device's pool holds mapped now.  REPOPS_ERR_INVALID_ARG for a null
 * bytes_out. */
int repops_scratch_set_keep_bytes(uint64_t bytes);
int repops_scratch_release(void);
int repops_scratch_reserved_bytes(uint64_t *bytes_out);

/* Host memory for the host-buffer entry points (repops_gemm_f32_host,
 * repops_fixed_order_mean_sgd_host, repops_merkle_sha256_host).  Neither page
 * describes anything like this; it is a deployment aid.
 *
 * Those calls copy their operands over the host link, and page-locked
 * ("pinned") host memory is what lets the copy engines read it directly.  How
 * that memory is paged matters on a Grace host: a GB300's copies out of
 * memory pinned in 64 KB pages (what cudaHostAlloc returned there) ran at 8
 * to 212 GB/s once a step touched more than ~16 GiB of it, varying from pass
 * to pass, while the same copies out of memory held in transparent huge pages
 * ran at 209-212 GB/s at every size tried up to 24 GiB.  The kernel may still
 * split huge pages later (on that host the buffers allocated first lost
 * theirs when more memory was allocated after them); copies over those pages
 * then vary again.
 *
 * repops_host_alloc: *ptr_out = `bytes` of zero-filled, page-locked host
 * memory registered with CUDA for every device (cudaHostRegisterPortable),
 * its pages transparent huge pages where the kernel provides them: an
 * anonymous mapping whose start is aligned to the huge page size
 * (/sys/kernel/mm/transparent_hugepage/hpage_pmd_size, 2 MiB if unknown),
 * advised MADV_HUGEPAGE.  A request of at least a quarter of a huge page is
 * rounded up to whole huge pages (up to one huge page more is mapped and
 * locked: 512 MB on a host with 64 KB base pages), so that all of it can be
 * held in them; a smaller one, or any where the kernel's transparent huge
 * pages are off ("never"), is mapped the ordinary way.  Owned by the
 * caller until repops_host_free.  bytes == 0 gives
 * *ptr_out = NULL and REPOPS_OK.  REPOPS_ERR_INVALID_ARG for a null ptr_out
 * or a size no mapping can hold (above SIZE_MAX / 2 less one huge page);
 * REPOPS_ERR_ALLOC if the mapping is refused; REPOPS_ERR_CUDA if the
 * registration fails (no usable device, or the pages cannot be locked); on
 * any error *ptr_out = NULL and nothing is kept.
 * repops_host_free: unregisters and unmaps memory from repops_host_alloc,
 * which no copy may still be reading or writing.  NULL is a no-op (REPOPS_OK);
 * a pointer repops_host_alloc did not return, or one already freed, is
 * REPOPS_ERR_INVALID_ARG.  Thread-safe. */
int repops_host_alloc(uint64_t bytes, void **ptr_out);
int repops_host_free(void *ptr);

/* ------------------------------------------------------------------------ */
/* Order-fixed FP32 GEMM                                                     */
/* "Verde与RepOps" §3.2, matmul example; §3.1; §3.3                          */
/* ------------------------------------------------------------------------ */

/* C = A * B, overwriting C (no alpha/beta), with
 *
 *   C[i][j] = fl( ... fl( fl(+0 + fl(A[i][0]*B[0][j])) + fl(A[i][1]*B[1][j]) ) ...
 *                 + fl(A[i][K-1]*B[K-1][j]) )
 *
 * k strictly increasing from +0.0f; every product rounded to binary32 before a
 * separately rounded add.  Parallel over (i, j) only: no split-K, no
 * reassociation.  A consequence: C never holds -0.0.
 *
 * Row-major storage, leading dimensions in elements:
 *   A (device): M x K, A[i][k] at A[i*lda + k], lda >= max(1, K)
 *   B (device): K x N, B[k][j] at B[k*ldb + j], ldb >= max(1, N)
 *   C (device): M x N, C[i][j] at C[i*ldc + j], ldc >= max(1, N)
 * M == 0 or N == 0: no-op.  K == 0: C is filled with +0.0f.
 * Errors: INVALID_ARG (negative size, bad leading dim, null pointer with a
 * non-empty operand, element offsets that overflow int64); ALIAS (C's span
 * overlaps A's or B's span); CUDA (launch failure).
 * Pointers need no alignment.  An operand TMA cannot describe (base not
 * 16-byte aligned, or leading dimension not a multiple of 4) is, for problems
 * of at least 4 GFLOP (2*M*N*K), first copied with a 16-byte pitch into
 * scratch taken from the library's scratch pool on `stream` (and released there);
 * smaller problems, or a refused allocation, read it with 4-byte copies.  The
 * bits are the same on every path. */
int repops_gemm_f32(int64_t M, int64_t N, int64_t K,
                    const float *A, int64_t lda,
                    const float *B, int64_t ldb,
                    float *C, int64_t ldc,
                    cudaStream_t stream);

/* As repops_gemm_f32 with transposed storage options (the backward GEMMs):
 *   transA == 0: A[i][k] at A[i*lda + k], lda >= max(1, K)
 *   transA != 0: A[i][k] at A[k*lda + i], lda >= max(1, M)   (dW = X^T dY)
 *   transB == 0: B[k][j] at B[k*ldb + j], ldb >= max(1, N)
 *   transB != 0: B[k][j] at B[j*ldb + k], ldb >= max(1, K)   (dX = dY W^T)
 * The result bits do not depend on transA/transB, only on the element values.
 * Where it is faster, operands are first copied into the kernels' fastest
 * layouts in scratch from the scratch pool on `stream`: a transposed B into
 * row-major from 1 GFLOP (2*M*N*K) on, a row-major A into the transposed
 * layout from 4 GFLOP on.  A refused allocation keeps the caller's layout. */
int repops_gemm_f32_ex(int transA, int transB,
                       int64_t M, int64_t N, int64_t K,
                       const float *A, int64_t lda,
                       const float *B, int64_t ldb,
                       float *C, int64_t ldc,
                       cudaStream_t stream);

/* Device scratch, in bytes, that repops_gemm_f32_ex (automatic choice) takes
 * for this problem and these operands: copies of operands into the kernels'
 * faster layouts and the chained k-split's running sums and flags (see
 * repops_gemm_f32_chained).  0 when the call runs on the caller's operands
 * alone, or for arguments repops_gemm_f32_ex would reject.  Host-only (reads
 * the device's properties, no launch); the pointers are looked at for their
 * alignment only. */
uint64_t repops_gemm_workspace_bytes(int transA, int transB,
                                     int64_t M, int64_t N, int64_t K,
                                     const float *A, int64_t lda,
                                     const float *B, int64_t ldb);

/* As repops_gemm_f32_ex, with the scratch taken from `workspace` (device,
 * 256-byte aligned, `workspace_bytes` bytes, owned by the caller and touched
 * by nothing else until the call's work on `stream` is done) instead of the
 * library's scratch pool, when workspace_bytes is at least
 * repops_gemm_workspace_bytes() for the same arguments; a smaller workspace
 * is not used (the scratch then comes from the pool).  The library then holds
 * no memory of its own for the call, and a caller that keeps its workspace
 * (or takes it from a caching allocator) pays no mapping of fresh memory
 * after a synchronisation.  The bits equal repops_gemm_f32_ex's.  Errors as
 * repops_gemm_f32_ex, plus INVALID_ARG (a workspace that is not 256-byte
 * aligned, or null with workspace_bytes > 0) and ALIAS (the workspace
 * overlaps A, B or C). */
int repops_gemm_f32_ws(int transA, int transB,
                       int64_t M, int64_t N, int64_t K,
                       const float *A, int64_t lda,
                       const float *B, int64_t ldb,
                       float *C, int64_t ldc,
                       void *workspace, uint64_t workspace_bytes,
                       cudaStream_t stream);

/* As repops_gemm_f32 with A, B and C in HOST memory (row-major, pitches as
 * there; page-locked memory for full speed).  The call takes device memory
 * for A, B and C (16-byte pitches) from the scratch pool on `stream`, copies B,
 * then copies A in row blocks on a helper stream while the previous block's
 * GEMM runs on `stream`, copies each block of C back on a second helper stream
 * as it completes, and releases the memory; everything is ordered before work
 * later enqueued on `stream`.  Asynchronous: A, B and C must stay valid, and C
 * is complete, once `stream` has reached this point.  The bits equal
 * repops_gemm_f32's (rows of C are independent k-chains).  Errors as
 * repops_gemm_f32, plus ALLOC (device memory refused) and ALIAS (C's host
 * bytes overlap A's or B's). */
int repops_gemm_f32_host(int64_t M, int64_t N, int64_t K,
                         const float *A, int64_t lda,
                         const float *B, int64_t ldb,
                         float *C, int64_t ldc,
                         cudaStream_t stream);

/* Loader paths for repops_gemm_f32_config. */
#define REPOPS_LOADER_AUTO 0      /* TMA when operands allow it, else CPASYNC; with
                                     config -1, the DIRECT kernel for small outputs
                                     (repops_gemm_small_output) */
#define REPOPS_LOADER_TMA 1       /* tensor-memory-accelerator tiles; needs 16-byte
                                     aligned A/B and lda, ldb multiples of 4 */
#define REPOPS_LOADER_CPASYNC 2   /* 4-byte cp.async with zero fill; any alignment */
#define REPOPS_LOADER_DIRECT 3    /* the small-output kernel: 16 x 32 CTA tiles of
                                     128 threads, 4-byte cp.async ring, any
                                     alignment and storage order; `config` is
                                     ignored.  Plain and typed GEMMs; the batched
                                     call answers INVALID_ARG; N above 2,097,120
                                     (65535 column tiles) UNSUPPORTED */

/* As repops_gemm_f32_ex with an explicit tile configuration (0 <=
 * config < repops_gemm_config_count(), or -1 for the automatic choice) and
 * loader path.  Exists so that callers and tests can show that the bits do not
 * depend on tiling or launch shape.  UNSUPPORTED if `loader` is TMA and the
 * operands do not meet its alignment rule. */
int repops_gemm_f32_config(int config, int loader, int transA, int transB,
                           int64_t M, int64_t N, int64_t K,
                           const float *A, int64_t lda,
                           const float *B, int64_t ldb,
                           float *C, int64_t ldc,
                           cudaStream_t stream);

/* As repops_gemm_f32_config with the TMA loader and the chained k-split
 * schedule, which repops_gemm_f32 takes by itself where its model finds it
 * faster (tile counts that leave the last wave of CTAs partly empty).
 * `workers` persistent CTAs (1 .. min(tiles, resident CTAs of the
 * configuration on the device), 0 = that maximum) run whole tiles one per
 * worker per wave, then split the k-slices of the remaining tiles (more than
 * `workers`, fewer than twice as many) equally in tile order, so that a tile
 * may be computed by two consecutive workers.  Such a tile's k-chains are
 * continued, never reordered or combined: the first worker runs slices 0 .. h-1
 * of every element's chain from +0 and stores the running binary32 sums
 * exactly as they stand; the second loads them and runs slices h .. end.  Every
 * element therefore gets the same operations in the same order as in
 * repops_gemm_f32 -- the same bits for every worker count (a split-K that adds
 * separately computed partial sums would not be).  ("Verde与RepOps" §3.2: the
 * order-critical dimension stays serial; only who computes which part of a
 * chain changes.)  Scratch (about workers x 32 KB) is taken from the scratch
 * pool on `stream`; the kernel is launched cooperatively and every
 * wait between workers is bounded (status word).  UNSUPPORTED when the
 * operands do not meet the TMA rule, `workers` is too large, or the scratch is
 * refused; INVALID_ARG for workers < 0; other errors as repops_gemm_f32. */
int repops_gemm_f32_chained(int config, int workers, int transA, int transB,
                            int64_t M, int64_t N, int64_t K,
                            const float *A, int64_t lda,
                            const float *B, int64_t ldb,
                            float *C, int64_t ldc,
                            cudaStream_t stream);

/* Number of GEMM tile configurations compiled into the library. */
int repops_gemm_config_count(void);

/* CTA tile (bm x bn), threads per CTA and per-thread tile (tm x tn) of a
 * configuration.  Any output pointer may be null.  INVALID_ARG for a bad id. */
int repops_gemm_config_info(int config, int *bm, int *bn, int *threads,
                            int *tm, int *tn);

/* Resident CTAs per SM of configuration `config`'s TMA kernel on the current
 * device (the figure the automatic choice models with); a negative status on
 * error (INVALID_ARG for an unknown config). */
int repops_gemm_config_occupancy(int config);

/* The configuration repops_gemm_f32 would choose for an M x N output on the
 * current device (-1 when M or N is 0).  The tiled configuration; see
 * repops_gemm_small_output for when the small-output kernel runs instead. */
int repops_gemm_auto_config(int64_t M, int64_t N, int64_t K);

/* 1 when repops_gemm_f32 (automatic configuration and loader) runs an M x N x K
 * problem whose operands the TMA loader can read on the chained k-split
 * schedule of repops_gemm_f32_chained (its model finds the last wave of
 * one-tile CTAs too empty), 0 when it runs one CTA per tile.  The same holds
 * for a single (batch 1) product of repops_gemm_f32_batched without a causal
 * skip or k band.  Host-only; the bits are the same either way. */
int repops_gemm_auto_chained(int64_t M, int64_t N, int64_t K);

/* 1 when repops_gemm_f32 (automatic configuration and loader) runs an M x N x K
 * problem on the small-output kernel (REPOPS_LOADER_DIRECT): M, N, K > 0 and
 * M * N <= 196,608 (384 x 384 and below, where the tiled kernels leave most
 * SMs idle); else 0.  Host-only; either kernel gives the same bits. */
int repops_gemm_small_output(int64_t M, int64_t N, int64_t K);

/* ------------------------------------------------------------------------ */
/* Batched GEMM with a fused epilogue                                        */
/* "Verde与RepOps" §3.2 matmul example (the k-chain); §4.3 (GeLU among the   */
/* operators behind DistilBERT's overhead).  The pages fix no epilogue; this */
/* is the library's definition.                                              */
/* ------------------------------------------------------------------------ */

#define REPOPS_ACT_NONE 0
#define REPOPS_ACT_GELU 1   /* the order-fixed GeLU of repops_gelu_f32 */

/* For b = 0 .. batch-1, with X_b = X + b*strideX (elements) for A, B, C, R:
 *
 *   acc = the k-chain of repops_gemm_f32 for element (i, j) of A_b * B_b
 *   y   = fl(alpha * acc)
 *   y   = fl(y + bias[j])          if bias != NULL   (device, N values, shared)
 *   y   = GeLU(y)                  if act == REPOPS_ACT_GELU
 *   y   = fl(y + R_b[i*ldr + j])   if R != NULL      (device)
 *   C_b[i*ldc + j] = y
 *
 * The epilogue runs after the element's whole k-chain, so the bits equal
 * those of repops_gemm_f32 followed by the separate element-wise steps.
 * Storage of A_b and B_b as in repops_gemm_f32_ex (transA, transB).  A stride
 * of 0 shares one operand between all batches (e.g. one weight matrix); a
 * stride smaller than a matrix interleaves the batches (attention heads as
 * column blocks of one row-major matrix: head h at column h*d, stride d).
 * The outputs C_b must not overlap one another: stacked (strideC at least one
 * C span) or interleaved within one row pitch ((batch-1)*strideC + N <= ldc,
 * strideC >= N); otherwise ALIAS.  R may be C itself (same ld and stride):
 * every element reads its residual before writing it; any other overlap of C
 * with A, B, bias or R is ALIAS.  K == 0 gives the epilogue of +0.
 * config / loader: as repops_gemm_f32_config (-1 / REPOPS_LOADER_AUTO for the
 * automatic choice); the bits do not depend on them.  TMA needs, besides its
 * repops_gemm_f32_config rule, batch strides of A and B that are multiples
 * of 4 elements.  No scratch memory is taken.
 * causal_first (attention scores Q K^T of queries at positions causal_first +
 * i): -1 computes every element; >= 0 leaves the elements with
 * j > causal_first + i unspecified -- whole output tiles above that boundary
 * are neither computed nor written, tiles crossing it are computed in full --
 * and every element on or below it exact.  Pair with
 * repops_softmax_rows_causal_f32, which never reads them.
 * k_lo, k_hi (the banded k-chain of causal attention's P V, dS K (k_hi) and
 * P^T dO, dS^T Q (k_lo)): -1 leaves that side of the chain open; k_lo >= 0
 * starts row i's chain at k = max(0, i - k_lo), k_hi >= 0 ends it at
 * k = min(K-1, i + k_hi); the chain still starts from +0 with k increasing,
 * and a row with an empty window gets the epilogue of +0.  The kernel runs
 * each tile's rows over the union of their windows (whole 32-k slices); the
 * extra terms of a row then add fl(+-0 * b) = +-0, which changes no bit
 * provided A_b[i][k] is +-0 outside row i's window and B_b is finite on the
 * k rows the tile reads -- as for a causal softmax output (+0 past each
 * row's prefix) times finite values.  The caller guarantees that; otherwise
 * the rows concerned are unspecified.
 * b_group >= 1: batch b reads B_(b / b_group) = B + (b / b_group)*strideB,
 * so b_group consecutive batches share one B (the query heads of a
 * grouped-query attention group and their key/value head); 1 is the plain
 * batched form.
 * Errors: INVALID_ARG (negative size or stride, bad leading dim, null
 * pointer with a non-empty operand, act not NONE/GELU, causal_first, k_lo or
 * k_hi < -1, b_group < 1, spans that overflow); ALIAS; UNSUPPORTED (batch > 65535, or
 * loader TMA when TMA cannot serve the operands); CUDA. */
int repops_gemm_f32_batched(int config, int loader, int transA, int transB,
                            int64_t batch, int64_t M, int64_t N, int64_t K,
                            const float *A, int64_t lda, int64_t strideA,
                            const float *B, int64_t ldb, int64_t strideB,
                            float *C, int64_t ldc, int64_t strideC,
                            float alpha, const float *bias, int act,
                            const float *R, int64_t ldr, int64_t strideR,
                            int64_t causal_first, int64_t k_lo, int64_t k_hi,
                            int64_t b_group, cudaStream_t stream);

/* ------------------------------------------------------------------------ */
/* Contributor order                                                         */
/* "Zoo Per-LLM Chain Soundness" §2 Lemma "Order independence within a       */
/* batch", §5 "Ordering subroutine", §6 "contributors (sorted DID list)"     */
/* ------------------------------------------------------------------------ */

/* Host-only.  Sorts n contributor identifiers (DIDs) by unsigned
 * lexicographic byte order, a proper prefix first.  Identifier r is the
 * lengths[r] bytes at ids + offsets[r] (host).  Writes order_out[0..n-1]
 * (host), order_out[0] being the smallest.  ORDER if two identifiers are
 * equal (the contributor set must be a set); INVALID_ARG for n < 0 or null
 * pointers with n > 0. */
int repops_sort_ids(int n, const uint8_t *ids, const int64_t *offsets,
                    const int64_t *lengths, int *order_out);

/* ------------------------------------------------------------------------ */
/* Fixed-order contributor mean fused with SGD                               */
/* "Zoo Per-LLM Chain Soundness" §2 Def. "Aggregation rule"; §5 "Ordering   */
/* subroutine", "Determinism of left-fold", "Update step"                    */
/* ------------------------------------------------------------------------ */

/* Maximum number of contributors per call. */
#define REPOPS_MEAN_MAX_CONTRIBUTORS 1024

/* For every element e in [0, len), in place:
 *   S     = g[order[0]][e]
 *   S     = fl(S + g[order[r]][e])         r = 1 .. nC-1  (left fold)
 *   gbar  = fl(S / nC)                     one correctly rounded division
 *   theta[e] = fl(theta[e] - fl(eta * gbar))
 * ptrs (host array of nC device pointers): contributor r's gradient, len
 * binary32 values each.  order (host array of nC ints): the fold order, a
 * permutation of 0..nC-1, normally from repops_sort_ids.  theta (device):
 * len binary32 values, updated in place.  eta: the step size, binary32.
 * len == 0: no-op.  Errors: INVALID_ARG (nC < 1, nC >
 * REPOPS_MEAN_MAX_CONTRIBUTORS, len < 0, null pointers); ORDER (order is not
 * a permutation); ALIAS (theta's range overlaps a gradient's range); CUDA.
 * Pointers need no alignment (unaligned inputs take a scalar path with the
 * same bits). */
int repops_fixed_order_mean_sgd(int nC, int64_t len, const float *const *ptrs,
                                const int *order, float eta, float *theta,
                                cudaStream_t stream);

/* As repops_fixed_order_mean_sgd with the gradients and theta in HOST memory
 * (page-locked for full speed): ptrs (host) holds nC host pointers of len
 * floats each, theta (host, len floats) is updated in place.  The call takes
 * device memory for two element chunks (up to 2^22 elements, at most about
 * 1 GiB in all) from the scratch pool on `stream`, copies each chunk of every
 * gradient and of theta in on a helper stream while the previous chunk is
 * folded on `stream`, copies theta's chunk back on a second helper stream, and
 * releases the memory; everything is ordered before work later enqueued on
 * `stream`.  Asynchronous: the buffers must stay valid, and theta is complete,
 * once `stream` has reached this point.  The bits equal
 * repops_fixed_order_mean_sgd's (elements are independent).  Errors as that
 * call, plus ALLOC; ALIAS compares host ranges. */
int repops_fixed_order_mean_sgd_host(int nC, int64_t len, const float *const *ptrs,
                                     const int *order, float eta, float *theta,
                                     cudaStream_t stream);

/* As repops_fixed_order_mean_sgd with the gradients stored as grad_type
 * (REPOPS_TYPE_F32, _F16 or _BF16, see "Half-precision storage" below): each
 * gradient element is widened exactly to binary32 before the fold; theta stays
 * binary32.  The bits equal those of repops_fixed_order_mean_sgd on the
 * widened gradients.  Gradients need no alignment (8-byte aligned half
 * gradients and a 16-byte aligned theta take the vector path).
 * INVALID_ARG also for an unknown grad_type. */
int repops_fixed_order_mean_sgd_typed(int nC, int64_t len, const void *const *ptrs,
                                      int grad_type, const int *order, float eta,
                                      float *theta, cudaStream_t stream);

/* ------------------------------------------------------------------------ */
/* SHA-256 Merkle commitment over tensor bytes                               */
/* "Zoo Per-LLM Chain Soundness" §1, §6 (bytes32 roots), §7 (H(theta) = m);  */
/* "Verde与RepOps" §2.3.2, §2.4.  Hash: SHA-256, FIPS 180-4.                 */
/* ------------------------------------------------------------------------ */

/* The bytes at ptr are cut into leaves of `leaf` bytes in increasing offset
 * (the last leaf may be shorter) and
 *   leaf digest = SHA256(0x00 || leaf bytes)
 *   node digest = SHA256(0x01 || left digest || right digest)
 * Levels are reduced pairwise, (0,1), (2,3), ...; an unpaired last node is
 * promoted unchanged to the next level; the root is the last node left.  One
 * leaf: root = its leaf digest.  Tensor bytes are hashed as stored
 * (little-endian binary32 for float tensors).
 *
 * ptr (device): `bytes` bytes, bytes >= 1.  leaf: a multiple of 64, 64 <=
 * leaf <= 2^30.  root_out (device): receives the 32-byte root, written
 * asynchronously on `stream`.
 * Scratch of repops_merkle_workspace_bytes(bytes, leaf) bytes is taken from
 * the scratch pool on `stream` and released with cudaFreeAsync on the same
 * stream.  Errors: INVALID_ARG (null pointer, bytes == 0, bad leaf); ALIAS
 * (root_out inside the input); ALLOC; CUDA. */
int repops_merkle_sha256(const void *ptr, uint64_t bytes, uint32_t leaf,
                         uint8_t *root_out, cudaStream_t stream);

/* Scratch bytes repops_merkle_sha256_ws needs for this input (0 if the input
 * is invalid). */
uint64_t repops_merkle_workspace_bytes(uint64_t bytes, uint32_t leaf);

/* As repops_merkle_sha256, with caller-provided device scratch `workspace`
 * of `workspace_bytes` >= repops_merkle_workspace_bytes(bytes, leaf) bytes,
 * 16-byte aligned.  The workspace must not be touched by anything else until
 * the call's work on `stream` is done.  INVALID_ARG if it is too small or
 * misaligned; ALIAS if it overlaps the input or root_out. */
int repops_merkle_sha256_ws(const void *ptr, uint64_t bytes, uint32_t leaf,
                            uint8_t *root_out, void *workspace,
                            uint64_t workspace_bytes, cudaStream_t stream);

/* ------------------------------------------------------------------------ */
/* Whole tree and inclusion proofs                                           */
/* "Verde与RepOps" §2.4 (the referee asks for a Merkle membership proof of an */
/* input tensor hash against the checkpoint); §2.3.2 (checkpoint hashes are  */
/* Merkle trees)                                                             */
/* ------------------------------------------------------------------------ */

/* Bytes of the stored tree of repops_merkle_tree_sha256: 32 per node over all
 * levels (0 if the input is invalid). */
uint64_t repops_merkle_tree_bytes(uint64_t bytes, uint32_t leaf);

/* As repops_merkle_sha256, and also stores every node of the tree in `tree`
 * (device, tree_bytes >= repops_merkle_tree_bytes(bytes, leaf), 16-byte
 * aligned): level 0 (the leaf digests) first, then level 1, ..., the root
 * last; within a level, nodes in index order; each node as its 32-byte digest.
 * A level's unpaired last node appears again as the last node of the next
 * level.  Errors as repops_merkle_sha256, plus INVALID_ARG for a short or
 * misaligned tree buffer and ALIAS if it overlaps the input or root_out. */
int repops_merkle_tree_sha256(const void *ptr, uint64_t bytes, uint32_t leaf,
                              uint8_t *tree, uint64_t tree_bytes,
                              uint8_t *root_out, cudaStream_t stream);

/* Host-only.  Number of sibling digests in the inclusion proof of leaf
 * `index` in a tree of `nleaves` leaves (levels where the path's node is
 * unpaired contribute none), or INVALID_ARG for index >= nleaves. */
int repops_merkle_proof_steps(uint64_t nleaves, uint64_t index);

/* Inclusion proof of leaf `index`: the sibling digests on its path to the
 * root, bottom-up, 32 bytes each, gathered from a tree stored by
 * repops_merkle_tree_sha256 (device) into proof_out (device,
 * 32 * repops_merkle_proof_steps(nleaves, index) bytes).  Asynchronous.
 * INVALID_ARG for null pointers or index >= nleaves; ALIAS if proof_out
 * overlaps the tree. */
int repops_merkle_proof(const uint8_t *tree, uint64_t nleaves, uint64_t index,
                        uint8_t *proof_out, cudaStream_t stream);

/* Membership check: hashes the leaf's bytes (leaf_bytes, device, leaf_len
 * bytes) as SHA256(0x00 || bytes), climbs with the proof's siblings (device)
 * -- on the left when the path's node index is odd, on the right when it is
 * even and has a right neighbour, none when it is unpaired -- and writes 1 to
 * *ok_out (device int) if the result equals root (device, 32 bytes), else 0.
 * Asynchronous.  INVALID_ARG for null pointers or index >= nleaves. */
int repops_merkle_verify(const void *leaf_bytes, uint64_t leaf_len, uint64_t nleaves,
                         uint64_t index, const uint8_t *proof, const uint8_t *root,
                         int *ok_out, cudaStream_t stream);

/* ------------------------------------------------------------------------ */
/* Order-fixed row operators: softmax, LayerNorm, RMSNorm, GeLU              */
/* "Verde与RepOps" §3.2 (order-critical dimensions run serially or with      */
/* synchronised threads), §3.3 and §4.3 (LayerNorm, GeLU and ERF are the     */
/* operators behind DistilBERT's overhead).  The pages fix no algorithm; the */
/* library's are:                                                            */
/*  - row reductions in a fixed 32-ary tree: each run of 32 consecutive      */
/*    values is folded left to right from its first value, the run results   */
/*    are folded the same way, level by level, until one value is left (max  */
/*    keeps the earlier value unless a later one is strictly greater);       */
/*  - exp(x): k = rint(x*log2 e) (ties to even), r = (x - k*ln2_hi) -        */
/*    k*ln2_lo (Cody-Waite two-part ln 2), e^r by the degree-7 Taylor        */
/*    polynomial in Horner form, times 2^k by exact power-of-two scaling;    */
/*    within 1.1 ulp of e^x; +inf above 88.7228394, 0 below -103.972084;     */
/*  - erfc(z), z >= 0: the Chebyshev fit of Numerical Recipes §6.2 with the  */
/*    exp above;                                                             */
/*  - a row's normaliser is one correctly rounded reciprocal per row,        */
/*    applied to each element by one multiplication;                         */
/*  - every other step one correctly rounded binary32 operation (division    */
/*    and square root included), no fused multiply-add.                      */
/* Matrices are row-major with leading dimensions in elements (ld >= cols).  */
/* y may be x itself (same pointer and leading dimension); any other overlap */
/* is ALIAS.  rows == 0 or cols == 0: no-op.  cols up to 393216              */
/* (UNSUPPORTED beyond).  Rows of at most 32768 values are read once and     */
/* written once.                                                             */
/* ------------------------------------------------------------------------ */

/* y[i][j] = e[i][j] * fl(1/s_i) with e[i][j] = exp(x[i][j] - m_i), m_i the
 * tree max of row i and s_i the tree sum of its e. */
int repops_softmax_rows_f32(int64_t rows, int64_t cols, const float *x, int64_t ldx,
                            float *y, int64_t ldy, cudaStream_t stream);

/* Causal softmax of attention blocks whose query rows sit at positions
 * first, first + 1, ...: row i is the softmax above over its first
 * L_i = min(cols, first + (i mod period) + 1) values and y[i][j] = +0 for
 * j >= L_i.  `period` rows form one block (one head); several heads' blocks
 * stacked row after row share one call.  first >= 0 and period >= 1, else
 * INVALID_ARG.  The masked scores are never read as values (they may hold
 * anything, NaN included). */
int repops_softmax_rows_causal_f32(int64_t rows, int64_t cols, const float *x, int64_t ldx,
                                   float *y, int64_t ldy, int64_t first, int64_t period,
                                   cudaStream_t stream);

/* mean = S/n, d = x - mean, var = tree sum of d*d / n,
 * inv = fl(1 / fl(sqrt(var + eps))), y = (d * inv) * gamma[j] + beta[j];
 * S = tree sum of the row, n = cols as binary32.  gamma, beta (device): cols
 * values each. */
int repops_layernorm_rows_f32(int64_t rows, int64_t cols, const float *x, int64_t ldx,
                              const float *gamma, const float *beta, float eps,
                              float *y, int64_t ldy, cudaStream_t stream);

/* ms = tree sum of x*x / n, inv = fl(1 / fl(sqrt(ms + eps))),
 * y = (x * inv) * gamma[j]. */
int repops_rmsnorm_rows_f32(int64_t rows, int64_t cols, const float *x, int64_t ldx,
                            const float *gamma, float eps, float *y, int64_t ldy,
                            cudaStream_t stream);

/* y = 0.5*x * (1 + erf(x/sqrt 2)), with z = x * fl(1/sqrt 2) and 1 + erf(z)
 * evaluated as 2 - erfc(z) for z >= 0 and erfc(-z) for z < 0.  Elementwise
 * over n values (device); y may be x. */
int repops_gelu_f32(int64_t n, const float *x, float *y, cudaStream_t stream);

/* ------------------------------------------------------------------------ */
/* Step replay                                                               */
/* "Zoo Per-LLM Chain Soundness" §7 "Reproducibility test plan": replay the  */
/* blocks in order from the genesis state, then verify H(theta) = m          */
/* ------------------------------------------------------------------------ */

/* For t = 0 .. steps-1, on `stream`:
 *   repops_fixed_order_mean_sgd(nC, len, ptrs + t*nC, orders + t*nC, etas[t], theta)
 *   roots_out[32*t .. 32*t+31] = Merkle root of theta's len*4 bytes (leaf bytes)
 * ptrs (host, steps*nC device pointers, step-major), orders (host, steps*nC
 * ints, each step's row a permutation), etas (host, steps floats), theta
 * (device, updated in place), roots_out (device, 32*steps bytes).  Every step
 * is validated before the first launch (ORDER, ALIAS, INVALID_ARG as the two
 * calls it makes).  Merkle scratch comes from the scratch pool on `stream`. */
int repops_replay_mean_sgd_commit(int steps, int nC, int64_t len,
                                  const float *const *ptrs, const int *orders,
                                  const float *etas, float *theta, uint32_t leaf,
                                  uint8_t *roots_out, cudaStream_t stream);

/* MEASUREMENT AID, not part of the operator surface: nothing in the
 * library's operators calls it and a user of the operators needs it for
 * nothing; it is exported so that the benchmark can time the library's own
 * compression without linking a second binary.
 *
 * Compression-rate probe: the ceiling the Merkle kernels are measured against.
 * Launches `threads` threads (a multiple of 128, 128 .. 2^24) on `stream`; thread
 * t computes, with the library's SHA-256 compression and its message held in
 * registers (no memory traffic, no tree), the digest of the message M_t
 * repeated `iters` times (0 .. 2^30), M_t being the 64 bytes of the 16
 * big-endian words 16t, 16t + 1, ..., 16t + 15, and writes it to
 * digests[8t .. 8t + 7] (device memory, big-endian state words).  That is
 * iters + 1 compressions a thread.  INVALID_ARG for a null pointer or a bad
 * count. */
int repops_sha256_rate_probe(uint32_t threads, uint32_t iters, uint32_t *digests, cudaStream_t stream);

/* As repops_merkle_sha256 with the input bytes (ptr) and root_out in HOST
 * memory (page-locked for full speed).  The call takes device memory (two
 * chunks of whole 128-leaf groups, about 64 MiB each, and the level scratch)
 * from the scratch pool on `stream`; each chunk is copied in on a helper stream
 * while the previous one is hashed on `stream`, the upper levels are folded
 * once every chunk is in, and the 32-byte root is copied back to root_out;
 * then the memory is released.  Asynchronous: read root_out once `stream` has
 * reached this point.  The root equals repops_merkle_sha256's.  Errors as that
 * call, plus ALLOC; ALIAS compares host ranges. */
int repops_merkle_sha256_host(const void *ptr, uint64_t bytes, uint32_t leaf,
                              uint8_t *root_out, cudaStream_t stream);

/* Size of the fixed device scratch behind repops_merkle_sha256_noalloc. */
#define REPOPS_MERKLE_NOALLOC_SCRATCH_BYTES (1u << 20)

/* Neither page describes anything like this entry point; it is a deployment aid.
 *
 * As repops_merkle_sha256, but it allocates nothing: no cudaMalloc, no
 * stream-ordered scratch, no caller workspace.  It is meant for callers that cannot
 * allocate device memory when they hash -- a host framework that has reserved
 * all device memory for its own pool, a latency-critical path on which an
 * allocation could block or synchronise, a plug-in whose host forbids
 * allocations after start-up.  The caller still passes the input (ptr,
 * device) and the output (root_out, device, 32 bytes).
 *
 * Scratch comes from one fixed array of REPOPS_MERKLE_NOALLOC_SCRATCH_BYTES
 * (1 MiB) in the library's device image; every GPU that loads the library
 * holds it until the process exits.  Inputs whose
 * repops_merkle_workspace_bytes(bytes, leaf) exceeds that size are rejected
 * with REPOPS_ERR_UNSUPPORTED before anything runs: at 4096-byte leaves the
 * limit is 4,186,112 leaves (about 16 GiB of input); inputs of at most 128
 * leaves need no scratch at all.
 *
 * The first call on each device looks up the array's device address (once
 * per device and CUDA context, with that device current) and caches it; make
 * that first call before any stream capture.  A new context on the device
 * (after cudaDeviceReset, say) makes the next call look the address up again
 * -- again before any capture.  All calls share the array and it keeps the last
 * call's contents (nothing in it needs to start at zero).  Calls whose work
 * overlaps on the GPU -- e.g. on two streams with no ordering between them --
 * race on the array: order them on one stream.  Other errors as
 * repops_merkle_sha256, without ALLOC. */
int repops_merkle_sha256_noalloc(const void *ptr, uint64_t bytes, uint32_t leaf,
                                 uint8_t *root_out, cudaStream_t stream);

/* ------------------------------------------------------------------------ */
/* Backward operators of a training step                                     */
/* "Verde与RepOps" §3.2 (order-critical reductions in a fixed order), §4.3   */
/* (training; LayerNorm, GeLU, ERF need reproducible forms).  The pages fix  */
/* none of these; the library's definitions, every step one binary32         */
/* rounding, every reduction the 32-ary tree of the row operators.           */
/* ------------------------------------------------------------------------ */

/* y[j] = tree sum over i = 0 .. rows-1 of x[i*ldx + j] (the column's values in
 * row order, folded by the 32-ary tree): bias and gain gradients.  rows == 0
 * gives +0.  Scratch for the tree's middle levels (about rows/31 * cols
 * floats) is taken from the scratch pool on `stream` (ALLOC when refused).
 * y (device, cols floats) must not overlap x (ALIAS). */
int repops_colsum_f32(int64_t rows, int64_t cols, const float *x, int64_t ldx, float *y,
                      cudaStream_t stream);

/* dx[i] = fl(dy[i] * GeLU'(x[i])), GeLU'(x) = Phi(x) + x*phi(x):
 *   z = x * (1/sqrt 2); 1 + erf(z) as in repops_gelu_f32; Phi = 0.5 * (1 + erf(z));
 *   phi = exp(-(0.5 * (x*x))) * 0.3989422917366028 (1/sqrt(2 pi) in binary32);
 *   GeLU' = Phi + x * phi.
 * dx may be x or dy (the same pointer); other overlaps are ALIAS. */
int repops_gelu_backward_f32(int64_t n, const float *x, const float *dy, float *dx,
                             cudaStream_t stream);

/* RMSNorm backward per row (the forward's inv = 1/sqrt(tree sum(x*x)/n + eps)
 * recomputed with the same operations):
 *   xh = x * inv, gy = dy * gamma[j], c = tree sum(gy * xh) / n,
 *   dx = inv * (gy - xh * c), then fl(dx + res) when res is not NULL (the
 *   gradient arriving through a pre-norm layer's residual path),
 *   dyxh = dy * xh   (repops_colsum_f32 of dyxh is dgamma).
 * x, dy, res, dx, dyxh: rows x cols with their own pitches; gamma: cols.
 * res may be dx itself (same pitch); otherwise outputs must not overlap any
 * input or each other (ALIAS); cols up to 393216 (UNSUPPORTED beyond). */
int repops_rmsnorm_backward_f32(int64_t rows, int64_t cols, const float *x, int64_t ldx,
                                const float *gamma, float eps, const float *dy, int64_t lddy,
                                const float *res, int64_t ldres, float *dx, int64_t lddx,
                                float *dyxh, int64_t ldp, cudaStream_t stream);

/* Softmax backward per row: s = tree sum(dp * p), ds = p * (dp - s).  p is the
 * forward's output (a causal block's masked entries are +0, so theirs is a
 * signed zero).  ds may be p or dp (same pointer and pitch); other overlaps
 * are ALIAS; cols up to 393216. */
int repops_softmax_backward_f32(int64_t rows, int64_t cols, const float *p, int64_t ldp,
                                const float *dp, int64_t lddp, float *ds, int64_t ldds,
                                cudaStream_t stream);

/* Backward of repops_softmax_rows_causal_f32 (first >= 0, period >= 1; else
 * INVALID_ARG): row r covers its prefix of L = min(cols, first + (r mod
 * period) + 1) entries -- s = tree sum(dp * p) over the L prefix values (the
 * tree of L values), ds = p * (dp - s) there -- and ds = +0 past the prefix,
 * where p and dp are never read (dp may hold anything there, e.g. the
 * unspecified tiles of a causal repops_gemm_f32_batched).  Aliasing and sizes
 * as repops_softmax_backward_f32. */
int repops_softmax_backward_causal_f32(int64_t rows, int64_t cols, const float *p, int64_t ldp,
                                       const float *dp, int64_t lddp, float *ds, int64_t ldds,
                                       int64_t first, int64_t period, cudaStream_t stream);

/* ------------------------------------------------------------------------ */
/* Fused causal attention                                                    */
/* "Verde与RepOps" §3.2 (order-critical reductions keep one fixed order, the */
/* rest runs in parallel) and §4.3 (the Llama-1B training measurement); the  */
/* pages fix no attention form: this is the composition of the operators    */
/* above, fused.                                                             */
/* ------------------------------------------------------------------------ */

/* Causal grouped-query attention of `seqs` sequences of S tokens, in one
 * launch.  Row t of sequence b is row b*S + t of every matrix; query head h
 * uses key/value head g = h / (heads / kv_heads):
 *   q (device): head h of a row at q + row*ldq + h*dh      (ldq >= heads*dh)
 *   k, v (device): head g at k + row*ldk + g*dh, v + row*ldv + g*dh
 *   out (device): head h at out + row*ldo + h*dh            (ldo >= heads*dh)
 *   probs (device, optional): (seqs*heads) x S x S, P[(b*heads + h)*S + i][j]
 * For every sequence, head and query row i, with one binary32 rounding per
 * step and no FMA:
 *   s_ij = fl(scale * (the k-chain over d = 0 .. dh-1 of q_i[d]*k_j[d] from
 *          +0)), j <= i  (scale == 1 applies no multiply);
 *   p_i. = the causal softmax of repops_softmax_rows_causal_f32 over s_i0 ..
 *          s_ii (32-ary max and sum trees, the library's exp, one correctly
 *          rounded reciprocal), +0 for j > i;
 *   out_i[c] = the chain over j = 0 .. i of fl(p_ij * v_j[c]) from +0.
 * This is exactly, bit for bit, repops_gemm_f32_batched (alpha = scale, tiles
 * above the diagonal skipped), then repops_softmax_rows_causal_f32 (first 0,
 * period S), then repops_gemm_f32_batched with the band k_hi = 0, for finite
 * inputs; terms past a row's prefix are skipped, not multiplied by +0, so
 * out_i also holds for a V with non-finite rows past i.  With probs, every
 * row of P is written in full (+0 past the prefix), as the unfused softmax
 * writes it, for a backward pass.
 * One CTA computes 16 query rows of one head: the scores and probabilities
 * stay in shared memory, keys and values stream through it.  Limits: dh = 64,
 * S <= 2048, q, k, v 16-byte aligned with ldq, ldk, ldv multiples of 4, out
 * 8-byte aligned with ldo even, probs (if any) 16-byte aligned with S a
 * multiple of 4; anything else is UNSUPPORTED (run the unfused operators
 * then).  INVALID_ARG for negative sizes, heads not a multiple of kv_heads,
 * null pointers or short leading dimensions; ALIAS when out or probs overlap
 * an input or each other.  seqs, S or heads == 0: nothing to do. */
int repops_attention_causal_f32(int64_t seqs, int64_t S, int64_t heads, int64_t kv_heads, int64_t dh,
                                const float *q, int64_t ldq, const float *k, int64_t ldk,
                                const float *v, int64_t ldv, float scale, float *out, int64_t ldo,
                                float *probs, cudaStream_t stream);

/* ------------------------------------------------------------------------ */
/* Half-precision storage                                                    */
/* "Verde与RepOps" §3.3 (IEEE-754 hardware needed; FP16 support limited) and */
/* §5.3 (lower-precision training as future work).  The pages fix no format  */
/* rules; the library's: a binary16 or bfloat16 element is widened exactly   */
/* to binary32, the binary32 order-fixed path computes, and a half result is */
/* narrowed once, round to nearest, ties to even (overflow to infinity,      */
/* subnormals kept).  NaNs stay NaN (payloads not pinned).                   */
/* ------------------------------------------------------------------------ */

/* dst[i] = src[i] converted from src_type to dst_type (REPOPS_TYPE_*), i < n.
 * src, dst (device) hold n elements each; they may be the same buffer only
 * when both types have the same size; any other overlap is ALIAS.  INVALID_ARG
 * for n < 0, unknown types or null pointers with n > 0. */
int repops_convert(int64_t n, const void *src, int src_type, void *dst, int dst_type,
                   cudaStream_t stream);

/* C = A * B as repops_gemm_f32_config (same storage, transposition, config and
 * loader arguments) with A, B and C stored as typeA, typeB, typeC: the
 * operands are widened exactly to binary32, the order-fixed k-chain runs, and
 * the result is narrowed once to typeC.  The bits equal repops_gemm_f32 on the
 * widened operands, narrowed.  Half operands are widened into scratch taken
 * from the scratch pool on `stream` (4 bytes per element of each widened
 * operand, and of C when typeC is a half type), released the same way; ALLOC
 * when it cannot be had.  INVALID_ARG for unknown types, and as
 * repops_gemm_f32_ex otherwise; ALIAS when C's bytes overlap A's or B's. */
int repops_gemm_typed(int config, int loader, int transA, int transB,
                      int64_t M, int64_t N, int64_t K,
                      const void *A, int typeA, int64_t lda,
                      const void *B, int typeB, int64_t ldb,
                      void *C, int typeC, int64_t ldc,
                      cudaStream_t stream);

/* ------------------------------------------------------------------------ */
/* Rolling hashes of batch rows                                              */
/* ZKDV page, proof.start(rolling_window=...): rolling hashes within each    */
/* committed batch row, the window at most the row's packed width; the       */
/* protocol commits a rectangular uint32 batch.  The page names no hash; the */
/* library's: Rabin-Karp modulo the Mersenne prime P = 2^61 - 1.             */
/* ------------------------------------------------------------------------ */

#define REPOPS_ROLLING_HASH_BASE 4294967311ull   /* smallest prime above 2^32 */

/* For every row r < rows and window start i = 0 .. width - window:
 *   out[r*ldo + i] = (sum_{t < window} words[r*ldw + i + t] * B^(window-1-t)) mod P
 * with B = REPOPS_ROLLING_HASH_BASE (so a window of two words maps injectively).
 * words (device): rows x width uint32, row pitch ldw >= width; out (device):
 * rows x (width - window + 1) uint64, row pitch ldo >= width - window + 1.
 * 1 <= window <= width (the window must not exceed the packed row width),
 * else INVALID_ARG; out overlapping words is ALIAS.  Exact integers: the bits
 * do not depend on how the kernel splits a row. */
int repops_rolling_hash_u32(int64_t rows, int64_t width, const uint32_t *words, int64_t ldw,
                            int64_t window, uint64_t *out, int64_t ldo, cudaStream_t stream);

/* ------------------------------------------------------------------------ */
/* SiLU-gated MLP (SwiGLU) and rotary position embeddings                     */
/* "Verde与RepOps" §4.3 (Llama-style training is the measured workload).     */
/* The pages fix neither operator; the library's definitions follow, every  */
/* step one IEEE rounding in a fixed order (exp as in repops_gelu_f32).      */
/* ------------------------------------------------------------------------ */

/* h[i][j] = fl(SiLU(g[i][j]) * u[i][j]) over rows x cols:
 *   sigma = fl(1 / fl(1 + exp(-g)))   (one correctly rounded division;
 *                                      exp overflow gives sigma = +0)
 *   SiLU  = fl(g * sigma).
 * g, u, h (device) with their own row pitches (>= cols); h may be g or u
 * itself (same pointer and pitch), any other overlap is ALIAS. */
int repops_swiglu_f32(int64_t rows, int64_t cols, const float *g, int64_t ldg,
                      const float *u, int64_t ldu, float *h, int64_t ldh, cudaStream_t stream);

/* Backward of repops_swiglu_f32 given dh, element by element (sigma recomputed
 * as in the forward):
 *   du = fl(dh * SiLU(g))
 *   dg = fl(fl(dh * u) * fl(sigma * fl(1 + fl(g * fl(1 - sigma)))))
 * dg may be g or dh, du may be u or dh (same pointer and pitch); dg and du
 * must not overlap each other, nor any input otherwise (ALIAS). */
int repops_swiglu_backward_f32(int64_t rows, int64_t cols, const float *g, int64_t ldg,
                               const float *u, int64_t ldu, const float *dh, int64_t lddh,
                               float *dg, int64_t lddg, float *du, int64_t lddu,
                               cudaStream_t stream);

/* Rotary frequencies f_i = exp(-fl(fl(i / pairs) * ln_base)), i < pairs
 * (base^(-2i/d_head) with pairs = d_head/2; ln_base is the caller's binary32
 * value of ln(base), which fixes the bits).  freq: device, pairs floats.
 * INVALID_ARG for pairs < 1 or a null pointer. */
int repops_rope_frequencies_f32(int64_t pairs, float ln_base, float *freq, cudaStream_t stream);

/* The rotation table for positions p < positions and pairs i < pairs:
 * cos[p*pairs + i], sin[p*pairs + i] of a = p * freq[i], computed in binary64
 * (every operation rounded, no FMA) and rounded once to binary32:
 *   a exact (p < 2^24 and a binary32 freq); k = rint(a * fl64(2/pi));
 *   r = ((a - k*P1) - k*P2) - k*P3 with pi/2 = P1 + P2 + P3, P1 and P2 of 29
 *   significant bits (k*P1, k*P2 exact for |k| < 2^24);
 *   sin r = r + (r*z) * S(z), cos r = 1 + z * C(z), z = r*r, S and C the
 *   Taylor series to r^15 and r^16 by Horner's rule; quadrant k mod 4.
 * For |a| < 2^24 the binary64 value is accurate to about 2^-50 relative, so
 * each result is the correctly rounded binary32 value unless the exact one
 * lies that close to a rounding boundary.  positions in [1, 2^24],
 * pairs >= 1; freq, cos, sin
 * device buffers that must not overlap (ALIAS); else INVALID_ARG. */
int repops_rope_table_f32(int64_t positions, int64_t pairs, const float *freq, float *cos_out,
                          float *sin_out, cudaStream_t stream);

/* Rotates in place pair i = (x0, x1) = (x[r][h*2*pairs + 2i], ... + 1) of head
 * h < heads of row r < rows, at position pos = first + (r mod period) with
 * c = cos[pos*pairs + i], s = sin[pos*pairs + i] (a repops_rope_table_f32
 * table of `positions` rows):
 *   inverse == 0:  (fl(fl(x0*c) - fl(x1*s)),  fl(fl(x0*s) + fl(x1*c)))
 *   inverse != 0:  (fl(fl(x0*c) + fl(x1*s)),  fl(fl(x1*c) - fl(x0*s)))
 * The inverse is the transpose: the backward of the rotation.  Columns past
 * heads*2*pairs are not touched.  x: device, row pitch ldx >= heads*2*pairs;
 * every position reached must be < positions; first >= 0, period >= 1
 * (INVALID_ARG otherwise); x must not overlap the table (ALIAS). */
int repops_rope_f32(int64_t rows, int64_t heads, int64_t pairs, float *x, int64_t ldx,
                    const float *cos_tab, const float *sin_tab, int64_t positions, int64_t first,
                    int64_t period, int inverse, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* REPOPS_H */

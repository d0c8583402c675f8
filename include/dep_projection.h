/*
 * dep_projection.h -- C ABI of the GB300 (sm_103a) decode projection library.
 *
 * The operation.  One decode-time linear layer at tensor-parallel degree 1:
 *
 *     y[B,N] = BF16( x[B,K] . W[N,K]^T ),  BF16 inputs, FP32 accumulation.
 *
 * Source: vllm.models.kimi_k3.nvidia.specialized_decode.runtime.dep (the
 * "runtime.dep page"), class DepProjection: a TP1 linear that runs split-K at the
 * batches its tactic table names and the stock FP32-accumulated BF16 GEMM
 * (torch.mm(x, W.t(), out=out)) otherwise; the module overview's precision
 * paragraph: BF16 outputs, FP32 accumulation, a split-K order that differs from
 * the stock one.  The weights it serves are the packed DSA input projection
 * (14560 x 7168), o_proj (7168 x 12288) and the packed KDA input projection
 * (49376 x 7168), streamed whole once per decode step.
 *
 * Plans.  A plan is built once per weight shape (N, K) and set of batch sizes,
 * like DepProjection.__init__ (runtime.dep page), and holds a tactic table keyed
 * by "max rows" (runtime.dep page, _bins and dep_policies).  At run time a batch
 * of B rows takes the entry with the smallest key >= B, else the entry with the
 * largest key.  Every tactic accepts any B >= 1 (wider batches run in passes).
 *
 * Layouts.  x is [B,K], W is [N,K] (the nn.Linear weight), y is [B,N]; all three
 * are row-major, contiguous, BF16, in device memory of the plan's device, and
 * 16-byte aligned.  K must be a multiple of 8 (16-byte rows).  N is any value
 * >= 1.  y must not overlap x or W.  The caller owns x, W and y; the library
 * neither retains nor repacks W.
 *
 * Determinism.  Each tactic sums in one fixed order with a fixed-order
 * cross-block split-K reduction and no floating-point atomics: the same call on
 * the same plan gives the same bits every time.
 *
 * Errors.  Every call returns a dep_status_t; nothing aborts or throws across
 * the ABI.  Launch failures are reported as DEP_ERR_CUDA.
 *
 * Concurrency.  A plan owns one split-K workspace.  Two runs of the same plan
 * must not overlap on the GPU (use one plan per stream).  Runs are asynchronous
 * on the given stream, allocate nothing and do not synchronise, so they can be
 * captured in CUDA graphs (the runtime package page, specialized_decode_config:
 * the deployment's decode batches are its CUDA-graph capture sizes).
 */
#ifndef DEP_PROJECTION_H
#define DEP_PROJECTION_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Opaque plan handle, owned by the library (free with dep_projection_plan_destroy). */
typedef struct dep_plan_s *dep_plan_t;

typedef enum {
    DEP_OK = 0,
    DEP_ERR_INVALID_ARG = 1,  /* null pointer, bad size, unknown tactic, wrong device */
    DEP_ERR_UNSUPPORTED = 2,  /* shape or plan kind this build cannot run */
    DEP_ERR_MISALIGNED = 3,   /* a pointer not 16-byte aligned, or K % 8 != 0 */
    DEP_ERR_CUDA = 4,         /* a CUDA runtime/driver call or a launch failed */
    DEP_ERR_OOM = 5,          /* plan-time device allocation failed */
    DEP_ERR_TIMEOUT = 6,      /* a kernel gave up a bounded wait (device status) */
    DEP_ERR_INTERNAL = 7,     /* an invariant of the library was broken */
    DEP_ERR_IO = 8            /* plan file could not be read or written, or is malformed */
} dep_status_t;

/* Tactic kinds. */
#define DEP_KIND_SPLITK_FMA 1 /* warp split-K on the FP32 FMA pipe, TMA-staged W */
#define DEP_KIND_TC 2         /* tcgen05 MMA, TMEM accumulators, TMA-staged W and x */
#define DEP_KIND_ROWS 3       /* warp split-K over whole weight rows, dynamic tiles, no
                                 cross-block fix-up; x resident in shared memory */
#define DEP_KIND_TC_SPLIT 4   /* tcgen05 MMA over (tile, K piece) items taken
                                 dynamically; tiles of tile_n = 64 or 128 weight rows
                                 (MMA M), each cut into `splits` fixed K pieces whose
                                 FP32 partials are added in piece order */
#define DEP_KIND_TC_WIDE 5    /* tcgen05 MMA for wide batches: each block streams a
                                 group of tile_n / 128 = 2 or 4 weight tiles of 128
                                 rows against every x slice (one MMA per tile, the
                                 same x operand), stream-K over (group, k-tile)
                                 units; split groups are reduced by the blocks
                                 that share them, each a part of the columns, adding
                                 the blocks' FP32 partials in block order */
#define DEP_KIND_TC_CLUSTER 6 /* tcgen05 MMA for wide batches: a thread-block cluster
                                 of `splits` = k CTAs per group of weight tiles --
                                 tile_n = 256 or 512 rows (2 or 4 tiles of 128), or
                                 192 rows (a 128-row and a 64-row tile) -- one MMA
                                 per tile with the same x operand, CTA rank r
                                 streaming K piece r; the K
                                 pieces are added in rank order through distributed
                                 shared memory (no global workspace); `stages` =
                                 weight stages (x has its own 2-4 stage ring);
                                 `ctas` = a multiple of k; tile_k = 64 */
#define DEP_KIND_TC_XM 7      /* tcgen05 MMA for wide batches with x on the MMA's M
                                 side: blocks of 128 batch rows (cols = 128 or 256:
                                 one or two per pass) against tiles of tile_n weight
                                 rows (MMA N, a multiple of 16 up to 256), dealt out
                                 statically over `ctas` blocks; splits = 0: each
                                 block sums its tiles' whole K; splits = 2: a
                                 thread-block cluster of two per tile (tile_n a
                                 multiple of 32, ctas even), each half of K, the
                                 halves added in order through distributed shared
                                 memory; no workspace either way; `stages` of
                                 tile_k = 64, 128 or 256 columns of the weight and
                                 of x */
#define DEP_KIND_WARP_MMA 8   /* warp-level mma.sync for small weights at up to 16
                                 rows: one block per tile of tile_n = 16 weight
                                 rows and whole K (splits = 0 or 1), or a cluster of
                                 splits = 2 or 4 blocks per tile, each a K piece,
                                 added in rank order in the first block's shared
                                 memory; cols = 16 batch rows per pass, stages of
                                 tile_k = 64, 128 or 256 columns; no tensor memory,
                                 a small ring, so several blocks (of one call and
                                 of the next) share an SM; `ctas` is not used */

/* One table entry: the tactic that serves batches of up to max_rows rows. */
typedef struct {
    int32_t max_rows; /* table key (binning rule above) */
    int32_t kind;     /* DEP_KIND_* */
    int32_t ctas;     /* persistent blocks launched (FMA/TC/TC_WIDE: work split
                         evenly, stream-K; ROWS/TC_SPLIT: work items taken
                         dynamically) */
    int32_t tile_n;   /* weight rows per tile (TC_WIDE: per group, 256 or 512;
                         TC_CLUSTER: per group, 192, 256 or 512; TC_XM: MMA N) */
    int32_t tile_k;   /* reduction columns per pipeline stage */
    int32_t stages;   /* pipeline depth (shared-memory stages) */
    int32_t cols;     /* batch rows per pass (FMA/ROWS: x rows held; TC: MMA N;
                         TC_XM: 128 or 256, MMA M = 128 per block of rows) */
    int32_t splits;   /* TC_SPLIT: K pieces per tile, 1..64 (capped at the tile's
                         k-tiles, ceil(K / tile_k)); TC_CLUSTER: CTAs per cluster;
                         TC_XM: 0, or 2 for pairs of blocks; WARP_MMA: K pieces
                         per tile, 0/1, 2 or 4; 0 for the other kinds */
} dep_tactic_t;

/* Plan flags. */
#define DEP_PLAN_DEFAULT 0u /* fixed rule: FMA split-K for small batches, TC past them */
#define DEP_PLAN_TUNE 1u    /* time candidate tactics per batch on scratch data; keep the fastest */
/* Programmatic dependent launch: each run may start while the preceding kernel
 * in its stream finishes, streaming its first weight tiles early and waiting for
 * that kernel before it reads x or writes y.  The caller promises that no work
 * enqueued before a run on the same stream writes W (decode weights are
 * read-only).  Consecutive runs then overlap one kernel's tail with the next
 * one's ramp-up, also inside CUDA graphs. */
#define DEP_PLAN_PDL 2u
/* Inspection: the wide-batch kernel (DEP_KIND_TC_WIDE) also stores the partials
 * each block reduces itself, so that dep_projection_plan_partials returns every
 * block's piece of every split group (extra writes; same results). */
#define DEP_PLAN_KEEP_PIECES 4u

/*
 * Build a plan for weights of shape [N,K] on the current CUDA device.
 *   batches/n_batches: the batch sizes the caller will run (the table's keys);
 *                      n_batches == 0 takes 1,2,4,8,16,32,64,128,256.
 *   flags:             DEP_PLAN_DEFAULT, or DEP_PLAN_TUNE and/or DEP_PLAN_PDL.
 * Allocates the plan's workspace, counters and status word on the device.
 * Errors: INVALID_ARG (N < 1, K < 8, batch < 1, null out), MISALIGNED (K % 8),
 * OOM, CUDA.  On error *out is set to NULL.
 */
dep_status_t dep_projection_plan(int64_t N, int64_t K, const int32_t *batches,
                                 int32_t n_batches, uint32_t flags, dep_plan_t *out);

/*
 * Build the default table for an explicit SM count without touching any GPU:
 * for inspection, saving, and host-side tests.  Running such a plan returns
 * DEP_ERR_UNSUPPORTED.  Errors as dep_projection_plan, plus INVALID_ARG for
 * sm_count < 1.
 */
dep_status_t dep_projection_plan_host(int64_t N, int64_t K, const int32_t *batches,
                                      int32_t n_batches, int32_t sm_count,
                                      dep_plan_t *out);

/*
 * y[B,N] = BF16(x[B,K] . W[N,K]^T) on `stream` (a cudaStream_t; NULL = legacy
 * default stream).  The tactic is the plan's table entry for B (binning rule).
 * B == 0 launches nothing and returns DEP_OK; B < 0 is INVALID_ARG.
 * Asynchronous: returns after enqueueing.  Errors: INVALID_ARG (null pointer,
 * overlap of y with x or W, current device is not the plan's), MISALIGNED,
 * UNSUPPORTED (host-only plan), CUDA (launch failure).
 */
dep_status_t dep_projection_run(dep_plan_t plan, const void *x, const void *W, void *y,
                                int32_t B, void *stream);

/*
 * The same with an explicit tactic instead of the table's (tests and tuning).
 * Errors as dep_projection_run, plus INVALID_ARG for a tactic this build does
 * not implement or whose split-K workspace exceeds the plan's, and UNSUPPORTED
 * for a grid the device cannot hold at once in a kind whose blocks wait on one
 * another (DEP_KIND_TC, DEP_KIND_TC_SPLIT, DEP_KIND_TC_WIDE: at most
 * (blocks resident per SM) x (SM count) blocks).
 */
dep_status_t dep_projection_run_tactic(dep_plan_t plan, const dep_tactic_t *tactic,
                                       const void *x, const void *W, void *y,
                                       int32_t B, void *stream);

/*
 * End-to-end call with the activations in host memory: brings x_host [B,K] to
 * the plan's device staging buffer, runs the projection against the resident
 * device weight W, and puts y back to y_host [B,N], all enqueued on `stream`.
 * The caller synchronises the stream before reading y_host.  B must not exceed
 * the plan's largest table key (the staging capacity).  Errors as
 * dep_projection_run.
 *   - Pinned host buffers (mapped into the device's address space, 16-byte
 *     aligned): a small kernel reads x_host directly (zero-copy) into the
 *     staging buffer, chained to the projection by programmatic dependent
 *     launch, so the projection streams its first weight stages while x
 *     arrives and consecutive calls leave no launch gap.  The projection
 *     stores y straight into y_host, except the cluster and x-on-M kinds
 *     (DEP_KIND_TC_CLUSTER, DEP_KIND_TC_XM), whose y a second small kernel
 *     copies back from the staging buffer.
 *     Stream order holds as for memcpys: each copy reads only after the
 *     preceding work in the stream has completed, so one call's y_host may be
 *     the next call's x_host.
 *   - Any other host memory: cudaMemcpyAsync both ways.
 *   Both give the same bits as dep_projection_run.  The environment variable
 *   DEP_STAGING=copy forces the copy path, DEP_STAGING=stage the copy-back of
 *   y for every kind (both for comparisons).
 */
dep_status_t dep_projection_run_host(dep_plan_t plan, const void *x_host, const void *W,
                                     void *y_host, int32_t B, void *stream);

/*
 * No counterpart in the pages: an addition of this library for callers that
 * must not allocate device memory -- code running inside a device-memory
 * allocator or pool (allocating there would re-enter it), hosts that reserve
 * all device memory up front and allow no other allocation, and latency-bound
 * paths that cannot afford cudaMalloc's implicit synchronisation.  They cannot
 * build a plan, since a plan allocates its workspace.
 *
 * y[B,N] = BF16(x[B,K] . W[N,K]^T) with the split-K FMA kernel, no plan, and no
 * allocation: the kernel's scratch (status word, tile counters, split-K
 * partials) is one 1 MiB array compiled into the library, which every GPU that
 * loads the library holds until the process exits.  Limits: N <= 262144 rows
 * (the counters) and at most 383 SMs (the partials); larger shapes return
 * DEP_ERR_UNSUPPORTED.  Same layouts, alignment and argument errors as
 * dep_projection_run; B == 0 does nothing.  The first call on a device looks up
 * the array's device address (cudaGetSymbolAddress) with that device current;
 * make that first call before any stream capture.  Every call clears the
 * counters and status word on `stream` before its kernel.  All calls share the
 * one array: calls that overlap on the GPU (other streams, other threads) race
 * and give wrong results.  Give-ups of the kernel's bounded waits are not
 * reported by this entry point.
 */
dep_status_t dep_projection_run_static(const void *x, const void *W, void *y, int64_t N,
                                       int64_t K, int32_t B, void *stream);

/*
 * No counterpart in the pages: a measurement aid.  Reads `bytes` of device
 * memory at p once with a read-only streaming kernel (16-byte loads, four in
 * flight per thread, four 512-thread blocks per SM) and XORs a fold of what it
 * read into the 64-bit word *sink (device memory), so that timing it on
 * `stream` gives the device's read-only bandwidth: the ceiling of a call that
 * streams a weight and writes almost nothing (a device-to-device copy also
 * writes as many bytes as it reads).  p 16-byte aligned, bytes a multiple of
 * 16, sink 8-byte aligned (else MISALIGNED); INVALID_ARG for null pointers or
 * zero bytes; CUDA if the launch fails.  Asynchronous.
 */
dep_status_t dep_projection_probe_read(const void *p, size_t bytes, void *sink, void *stream);

/* The tactic the plan uses for a batch of B >= 1 rows. */
dep_status_t dep_projection_plan_query(dep_plan_t plan, int32_t B, dep_tactic_t *out);

/* Copy up to `cap` table entries (sorted by max_rows) to `out`; *n = entry count. */
dep_status_t dep_projection_plan_table(dep_plan_t plan, dep_tactic_t *out, int32_t cap,
                                       int32_t *n);

/* Replace (or insert) the table entry with key tactic->max_rows.  The tactic is
 * validated (INVALID_ARG if not; UNSUPPORTED, as for dep_projection_run_tactic,
 * for a grid the device cannot hold at once); if it needs more workspace, counters or
 * staging than the plan owns, the plan's device block is re-allocated (after a
 * device synchronisation; OOM leaves the plan unchanged). */
dep_status_t dep_projection_plan_set(dep_plan_t plan, const dep_tactic_t *tactic);

/*
 * Inspection: copy the plan's split-K partial area (FP32) to host memory after
 * synchronising the device; *written = bytes copied (at most `bytes`).  Layout
 * for a stream-K launch of C blocks: partial (block c, slot s, batch column j,
 * tile row r) at float index ((c * 2 + s) * cols + j) * tile_n + r, slot 0 for
 * the block's first tile and 1 for its last.  Lets a test re-add the partials
 * of every split tile in block order and check the kernel's fix-up bit for bit.
 * For a DEP_KIND_TC_WIDE launch of C blocks with MMA width NT on groups of
 * R = tile_n rows: block c's piece of a split group sits in slot s (1 for the
 * group the block starts in, 0 for its last group when it has more than one)
 * at float offset (c * 2 + s) * R * NT; inside it, epilogue warp e (0..7, TMEM
 * lane quadrant (e + 2) % 4, column half e / 4 of the G * NT accumulator
 * columns) owns 32 * G * NT / 2 floats, accumulator column j of TMEM lane l
 * at (j / 4 * 32 + l % 32) * 4 + j % 4.  Without DEP_PLAN_KEEP_PIECES the
 * columns a block reduces itself are not stored.
 */
dep_status_t dep_projection_plan_partials(dep_plan_t plan, void *host, size_t bytes, size_t *written);

/*
 * Inspection: copy the plan's K-piece exchange region (64-bit words) to host
 * memory after synchronising the device; *written = bytes copied (at most
 * `bytes`).  For a K-piece launch (TC_SPLIT, S > 1 pieces in effect) the word of
 * (tile t, piece p, batch column j, tile row r) is at index
 * ((t * S + p) * cols + j) * tile_n + r; its low 32 bits are the piece's FP32
 * partial, its high 32 bits the "full" flag (0 once the launch has finished).
 * Lets a test re-add the pieces in order and check y bit for bit.
 */
dep_status_t dep_projection_plan_exchange(dep_plan_t plan, void *host, size_t bytes, size_t *written);

/* Bytes of device workspace the plan owns (split-K partials, counters, status). */
dep_status_t dep_projection_plan_workspace(dep_plan_t plan, size_t *bytes);

/*
 * Save the table as text keyed by (device name, SM count, N, K), and load it
 * back onto the current device (tuning need not be repeated).  Files are
 * written in format 2 (eight fields per entry); format 1 files (seven fields,
 * no K pieces) still load.  Load checks the
 * shape (INVALID_ARG if it differs) and the SM count (UNSUPPORTED if the file
 * was made for another GPU, or holds a grid this device cannot hold at once).  Errors: IO for unreadable or malformed files.
 */
dep_status_t dep_projection_plan_save(dep_plan_t plan, const char *path);
dep_status_t dep_projection_plan_load(const char *path, int64_t N, int64_t K,
                                      dep_plan_t *out);

/* Free the plan and its device memory (synchronises its device).  NULL is a no-op. */
void dep_projection_plan_destroy(dep_plan_t plan);

/*
 * Read and clear the plan's device status word (synchronises `stream`).
 * *code = 0 if every kernel since the last read finished its waits; otherwise
 * the first nonzero code a kernel recorded (see DEP_DEV_* below), and the
 * return value is DEP_ERR_TIMEOUT; the plan's split-K counters and K-piece
 * exchange flags, which a give-up may leave mid-protocol, are then cleared
 * (synchronises the device) so that later runs start clean.
 */
dep_status_t dep_projection_device_status(dep_plan_t plan, void *stream, int32_t *code);

#define DEP_DEV_TIMEOUT_PRODUCER 1 /* the load warp gave up waiting for a free stage */
#define DEP_DEV_TIMEOUT_CONSUMER 2 /* a compute warp gave up waiting for a stage's data */
#define DEP_DEV_TIMEOUT_MMA 3      /* the MMA warp gave up waiting */
#define DEP_DEV_TIMEOUT_EPILOGUE 4 /* an epilogue warp gave up waiting for an accumulator */
#define DEP_DEV_BOUNDS 5           /* bounds-checked (DEP_DEBUG) builds only: a kernel
                                      computed an index past one of its buffers and
                                      skipped that access */

/*
 * Bounded-wait self-test: launches one block whose waits can never be satisfied
 * (an mbarrier that nothing arrives on) with a wait limit of `limit_us`
 * microseconds, synchronises, and reports the code the kernel recorded in
 * *code (expected: DEP_DEV_TIMEOUT_CONSUMER).  Returns DEP_OK if the kernel
 * came back by itself.  Exercises the give-up path without faulting the GPU.
 */
dep_status_t dep_projection_selftest_timeout(int32_t limit_us, int32_t *code);

/*
 * Give-up self-test of the split-K exchange, on a plan's own workspace: enqueues
 * on `stream` one warp that publishes ("full") exchange words of two pieces,
 * as publishers would, then runs the exchange's reducer over two pieces of
 * which one is never published, with a wait limit of `limit_us` microseconds.
 * The reducer gives up and records DEP_DEV_TIMEOUT_EPILOGUE in the plan's
 * status word; the unreduced piece's flags and a nonzero word at the start of
 * the counters are left behind.  dep_projection_device_status then reports the code and clears the
 * counters and exchange words, after which the plan's runs give the same bits
 * as a fresh plan's.  Exercises the give-up path without faulting the GPU.
 * Errors: INVALID_ARG (null plan, limit outside 1 us..10 s), UNSUPPORTED
 * (host-only plan, or a plan whose table has no tensor-core tactic and so no
 * exchange region), CUDA.
 */
dep_status_t dep_projection_plan_selftest_exchange(dep_plan_t plan, int32_t limit_us, void *stream);

/* The binning rule on its own: index into keys[0..n_keys) of the entry serving
 * B rows -- smallest key >= B, else the largest key; -1 if n_keys < 1.  The keys
 * need not be sorted.  Pure host function. */
int32_t dep_bins_index(const int32_t *keys, int32_t n_keys, int32_t B);

/* Static description of a status code.  Never NULL. */
const char *dep_status_string(dep_status_t status);

/* Library version, as MAJOR * 10000 + MINOR * 100 + PATCH. */
int32_t dep_projection_version(void);

#ifdef __cplusplus
}
#endif

#endif /* DEP_PROJECTION_H */

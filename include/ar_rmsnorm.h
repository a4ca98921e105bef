/*
 * ar_rmsnorm — fused AllReduce + residual-add + RMSNorm for GB300 (sm_103a).
 *
 * C ABI of libarnorm.so.  Plain pointers and sizes only; no C++ or torch
 * types cross this boundary, nothing throws or aborts across it.
 *
 * The operation (the epilogue of a tensor-parallel decoder layer):
 *
 *   for each row i < m and column j < H
 *     s      = p_0[i,j] + p_1[i,j] + ... + p_{n-1}[i,j]   fp32, rank order
 *     r      = s + residual[i,j]                           fp32
 *     residual_out[i,j] = bf16(r)
 *     out[i,j]          = bf16(r * rsqrt(mean_j(r^2) + eps) * weight[j])
 *
 * The n partials are the n ranks' buffers of an all-reduce; on one GPU they
 * all live in this GPU's memory.  The sum is taken in fp32 strictly in the
 * order partials[0], partials[1], ..., partials[n-1], so it is bit-exact and
 * independent of the launch shape (ROCm/aiter #3817 "perf: optimize fused
 * AllReduce + RMSNorm (custom_all_reduce)", Technical Details, 2stage,
 * reduce-scatter: the sum follows the order of the rank pointers).
 *
 * Two paths compute it:
 *   one-stage  a single kernel, one pass over memory (same page, Technical
 *              Details, 1stage: the decode path with a block reduce of the
 *              square sum);
 *   two-stage  stage 1 reduces every 16-byte pack across the ranks and
 *              writes the sum, rounded to bf16, to a temporary buffer; stage
 *              2 loads it, adds the residual and normalises (same page,
 *              2stage: reduce-scatter, stage-1 launch config, stage-2
 *              RMSNorm reduce).  Because of that rounding, two-stage results
 *              are those of s' = bf16(s) in place of s.
 *
 * Data layout: every tensor is bf16, contiguous and row-major; partials,
 * residual, out and residual_out are [m, H] and weight is [H] -- the
 * scope validated in lightseekorg/tokenspeed #968 "perf(comm): add opt-in
 * Triton AR+RMSNorm backend", Summary.
 * Every pointer must be 16-byte aligned and H a multiple of 8 (one 16-byte
 * pack = 8 bf16).
 *
 * Ownership: all tensors belong to the caller and live in device memory of
 * the current device (ar_rmsnorm_mapped and the cross-rank calls also take
 * host, IPC and peer mappings).  The library owns only the two-stage
 * workspace, after ar_reserve_workspace, and the fixed scratch array of
 * ar_rmsnorm_two_stage_static.  The host pointer arrays (`partials`,
 * `temps`, `pads`) are read during the call only and may be freed when the
 * call returns.
 *
 * Streams: every call is asynchronous on `stream` (a cudaStream_t; NULL is
 * the legacy default stream).  No call of the compute path -- the epilogue
 * calls, the stage calls, the signal, barrier, one-shot and two-shot calls
 * -- synchronises the host or allocates, so they may be captured in a CUDA
 * graph (setup and self-test calls may do both).  The
 * first launching call on a device sets kernel attributes and reads the
 * kernels' occupancy for the launch plan; make one call (or
 * ar_reserve_workspace) before capturing.
 *
 * Aliasing: residual_out may equal residual (in place).  Any other overlap
 * between out, residual_out, residual, the partials and the workspace is
 * rejected with AR_ERR_ALIAS.
 */
#ifndef AR_RMSNORM_H
#define AR_RMSNORM_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes returned by every call. */
#define AR_OK              0  /* success; m == 0 (or count == 0) is a no-op that
                                 checks only the sizes, pointers may be NULL    */
#define AR_ERR_ARG         1  /* n outside [1, AR_MAX_RANKS], m < 0, H <= 0,
                                 eps negative or not finite, NULL pointer,
                                 unknown mode                                   */
#define AR_ERR_ALIGN       2  /* a pointer not 16-byte aligned, or H % 8 != 0 */
#define AR_ERR_ALIAS       3  /* overlapping buffers other than
                                 residual_out == residual                       */
#define AR_ERR_WORKSPACE   4  /* two-stage with m*H above the reserved
                                 workspace of the current device               */
#define AR_ERR_CUDA        5  /* a CUDA runtime call or a launch failed        */
#define AR_ERR_TIMEOUT     6  /* a bounded device-side wait ran out            */
#define AR_ERR_UNSUPPORTED 7  /* H above AR_MAX_HIDDEN                         */
#define AR_ERR_SCRATCH_LIMIT 8 /* m*H above AR_STATIC_SCRATCH_ELEMS
                                  (ar_rmsnorm_two_stage_static only)          */
#define AR_ERR_BOUNDS      9  /* a device-side bounds check failed (only the
                                 checking build, compiled with AR_CHECK=1,
                                 has these checks; the access was skipped)    */

/* Modes. */
#define AR_MODE_AUTO       0  /* pick by ar_select_mode(n, m, H)               */
#define AR_MODE_ONE_STAGE  1
#define AR_MODE_TWO_STAGE  2

#define AR_MAX_RANKS  16      /* most partials one call reduces                */
#define AR_MAX_HIDDEN 131072  /* largest H (16 CTAs x 8192 columns)            */
#define AR_STREAM_MAX_HIDDEN 32768 /* largest H of the stream kernel           */

/*
 * The fused epilogue: the all-reduce of the n rank partials, the residual
 * add and RMSNorm in one call (ROCm/aiter #3817 "perf: optimize fused
 * AllReduce + RMSNorm (custom_all_reduce)", Motivation and Technical
 * Details: the one-stage and two-stage paths).
 *   partials     host array of n device pointers, each [m, H] bf16; index
 *                order is the reduce order.
 *   n            number of partials (ranks), 1 .. AR_MAX_RANKS.
 *   residual     [m, H] bf16, device.
 *   weight       [H] bf16, device (the RMSNorm gain).
 *   eps          added to mean(r^2) inside the square root; finite, >= 0.
 *   m, H         rows (tokens) and hidden size.
 *   out          [m, H] bf16, device: the normalised output.
 *   residual_out [m, H] bf16, device: bf16(sum + residual); may be residual.
 *   mode         AR_MODE_AUTO, AR_MODE_ONE_STAGE or AR_MODE_TWO_STAGE.
 *   stream       cudaStream_t to launch on.
 * Returns AR_OK or an AR_ERR_* code.  Argument errors are found before
 * anything is launched.  A call of several launches (two-stage; the one-
 * and two-shot calls) that gets AR_ERR_CUDA from a later launch leaves the
 * earlier ones enqueued; the stream's results are then undefined.
 */
int ar_rmsnorm(const void *const *partials, int n, const void *residual,
               const void *weight, float eps, int64_t m, int64_t H, void *out,
               void *residual_out, int mode, void *stream);

/*
 * What one call launches: the path and the launch shape of the fused
 * epilogue kernel (one-stage, or stage 2 of two-stage).
 */
typedef struct {
  int mode;        /* AR_MODE_ONE_STAGE or AR_MODE_TWO_STAGE                  */
  int kernel;      /* AR_KERNEL_REGISTER, AR_KERNEL_REGISTER_LATE_W or
                      AR_KERNEL_STREAM                                        */
  int cluster;     /* register kernel: CTAs sharing one row, 1..16            */
  int vpt;         /* 16-byte packs per thread: 1, 2, 4 or 8 (stream kernel:
                      row tiles per row, rounded up to a power of two)       */
  int threads;     /* threads per CTA (stream kernel: 32 + consumers)         */
  int stages;      /* stream kernel: shared-memory ring slots; else 0         */
  int64_t ctas;    /* CTAs of the epilogue kernel                              */
  int launches;    /* kernels one call launches (1 or 2)                      */
  int prefetch;    /* L2 prefetch of the epilogue kernel: AR_PREFETCH_NONE,
                      AR_PREFETCH_ROW or AR_PREFETCH_ROW_AHEAD                */
} ar_plan_t;

/* L2 prefetch (ar_plan_t.prefetch).  A prefetch only asks L2 to fetch
   lines of this GPU's memory; it changes no result. */
#define AR_PREFETCH_AUTO      0  /* library's choice (forcing only)            */
#define AR_PREFETCH_NONE      1
#define AR_PREFETCH_ROW       2  /* each CTA prefetches its own (first) row
                                    slice of the inputs before it waits for
                                    the previous grid in the stream (one-
                                    stage; two-stage prefetches in stage 1
                                    instead)                                */
#define AR_PREFETCH_ROW_AHEAD 3  /* as ROW, and: register kernel (one CTA per
                                    row only): after its sums each CTA
                                    prefetches the slice of the row one wave
                                    of CTAs ahead; stream kernel: the
                                    producer prefetches the CTA's next row */

/* Epilogue kernels (ar_plan_t.kernel). */
#define AR_KERNEL_AUTO      0  /* library's choice (forcing only)             */
#define AR_KERNEL_REGISTER  1  /* one CTA (or a cluster of up to 16) per row;
                                  loads straight into registers: short grids */
#define AR_KERNEL_STREAM    2  /* persistent, one CTA per SM; a producer warp
                                  streams row tiles into a shared-memory ring
                                  with bulk asynchronous copies: many rows   */
#define AR_KERNEL_REGISTER_LATE_W 3  /* the register kernel, one CTA per row,
                                        loading the weight after the sums:
                                        fewer registers while the partials
                                        are in flight (more CTAs per SM)  */

/*
 * The plan ar_rmsnorm would follow for (n, m, H, mode) on a GPU with
 * `sm_count` SMs (0: ask the current device): the path the selection rule
 * picks (ROCm/aiter #3817, Test Results: the one-/two-stage thresholds)
 * and the launch shape of its kernels.  Pure host logic when
 * sm_count > 0: the measured plan table with plain interpolation between
 * its rows columns.  With sm_count = 0 it is exactly ar_rmsnorm's plan on
 * the current device, whose interpolation also uses each kernel's occupancy
 * there (so the two can differ between grid points).  Returns AR_OK or
 * AR_ERR_ARG / AR_ERR_ALIGN / AR_ERR_UNSUPPORTED as ar_rmsnorm would.
 */
int ar_get_plan(int n, int64_t m, int64_t H, int mode, int sm_count,
                ar_plan_t *plan);

/*
 * CTAs per SM of the one-CTA-per-row register kernel for `inputs` partials,
 * `vpt` packs per thread, the weight loaded late (late_weight = 1) or not,
 * with `threads` threads per CTA; 0 if unknown.
 */
typedef int (*ar_occupancy_fn)(int inputs, int vpt, int late_weight, int threads);

/*
 * As ar_get_plan with sm_count > 0 (pure host logic, no CUDA call), with the
 * caller's occupancy figures for the wave-aware interpolation of the plan
 * table that ar_rmsnorm does with the device's own figures: plan for
 * another GPU, or test the planner.  ctas_per_sm may be NULL (plain
 * interpolation).  It is called during the call only.  AR_ERR_ARG for
 * sm_count <= 0 or a NULL plan.  Library utility (no passage of the pages
 * defines it).
 */
int ar_get_plan_ex(int n, int64_t m, int64_t H, int mode, int sm_count,
                   ar_occupancy_fn ctas_per_sm, ar_plan_t *plan);

/*
 * The current device's figure for ar_occupancy_fn: CTAs per SM of the
 * one-CTA-per-row register kernel (inputs, vpt, late_weight, threads), read
 * once when a launching call made the device ready; 0 if unknown (no such
 * call yet, or arguments out of range).  Makes no CUDA call beyond
 * cudaGetDevice.  ar_get_plan_ex with this function and the device's SM
 * count plans exactly as ar_rmsnorm does on the device.  Library utility
 * (no passage of the pages defines it).
 */
int ar_register_occupancy(int inputs, int vpt, int late_weight, int threads);

/*
 * As ar_rmsnorm, with two additions for testing and tuning.  The reduced sum
 * is exposed because the pages make its bit-exactness the contract: the
 * sum follows the order of the rank pointers, so it stays bit-identical
 * whatever the kernel (ROCm/aiter #3817, Technical Details, 2stage,
 * reduce-scatter).  The forced plan plays the role of the page's switch
 * that pins the one- or two-stage path for benchmarking (AITER_AR_1STAGE,
 * same page, Test Plan), extended to the kernel and its launch shape.
 *   sum_out  [m, H] fp32 device buffer (16-byte aligned) that receives the
 *            reduced sum feeding the residual add: the fp32 accumulator for
 *            one-stage, the widened bf16 temporary for two-stage.  NULL to
 *            skip.  Costs 4*m*H extra bytes of writes.
 *   plan     NULL for the library's choice, else it forces the epilogue
 *            kernel and its launch shape; 0 in a field = library's choice.
 *            `kernel`: AR_KERNEL_REGISTER, AR_KERNEL_REGISTER_LATE_W or
 *            AR_KERNEL_STREAM.  Register kernel: `cluster` in {1,2,4,8,16}
 *            (1 for AR_KERNEL_REGISTER_LATE_W), `vpt` in {1,2,4,8}, at most
 *            1024 packs per CTA.  Stream kernel (H <= 32768): `threads` =
 *            32 + consumer threads (a multiple of 32, consumers <= 512, a row
 *            in <= 8 tiles), `stages` <= 16 ring slots (fewer if shared
 *            memory is short), `ctas` = grid size (several CTAs per SM split
 *            its shared memory).  Other combinations return AR_ERR_ARG;
 *            `mode` and `launches` are ignored (`mode` argument picks the
 *            path).  The sum and residual_out do not depend on the kernel or
 *            the shape; out may differ in its last bit between shapes (the
 *            square sum is reduced in a shape-dependent order).
 */
int ar_rmsnorm_ex(const void *const *partials, int n, const void *residual,
                  const void *weight, float eps, int64_t m, int64_t H,
                  void *out, void *residual_out, int mode, void *stream,
                  float *sum_out, const ar_plan_t *plan);

/*
 * As ar_rmsnorm, but any of the partials, residual, weight, out and
 * residual_out may live outside this process's own device memory: in host
 * memory that is pinned and mapped into the device's address space
 * (cudaHostAlloc / cudaMallocHost, or cudaHostRegister, under unified
 * addressing: the device address equals the host address), in another
 * process's allocation opened with ar_ipc_open (the one-shot all-reduce:
 * every rank reads every rank's partial), or in another GPU's memory that
 * this device can reach (peer access).  The kernels read and write such buffers directly over the
 * host link (NVLink-C2C on Grace systems): no staging copy, no device memory
 * beyond the two-stage workspace.  The epilogue runs on the register kernel
 * (plain 16-byte loads and stores), in the form and launch shape the
 * measured table ranks best among the register-kernel candidates, without
 * bulk L2 prefetches.  Results are bit-identical to ar_rmsnorm's register
 * kernel for the same launch shape.
 *
 * Each pointer is checked with cudaPointerGetAttributes before anything is
 * launched: it must be device memory of the current device, managed
 * memory, mapped pinned host memory, or memory of a GPU this device has
 * peer access to; anything else (pageable host memory, a device without
 * peer access) returns AR_ERR_ARG.  The pages have no
 * host-buffer path: this entry point has no counterpart there; what it
 * computes is ar_rmsnorm's.  As everywhere in
 * this library, each buffer must hold the bytes its shape implies.  The
 * host memory must stay pinned and untouched by the host until the stream
 * has passed the call.  The checks cost a few microseconds per call.
 */
int ar_rmsnorm_mapped(const void *const *partials, int n, const void *residual,
                      const void *weight, float eps, int64_t m, int64_t H,
                      void *out, void *residual_out, int mode, void *stream);

/*
 * Stage 1 alone: temp[e] = bf16(p_0[e] + ... + p_{n-1}[e]) for e < count,
 * fp32 rank-order sum, one 16-byte pack per thread step, no shared memory
 * and no block barrier (ROCm/aiter #3817, Technical Details, 2stage,
 * reduce-scatter).  count must be a multiple of 8; temp is caller-owned
 * device memory of count bf16 and must not overlap a partial.
 */
int ar_reduce_scatter_flat(const void *const *partials, int n, int64_t count,
                           void *temp, void *stream);

/*
 * Stage 1 as one rank of `world` runs it in a reduce-scatter whose gather
 * is done by stores: the packs of slice `rank` -- pack range [rank*S,
 * min((rank+1)*S, count/8)) with S = ceil(count/8 / world) -- are reduced
 * across the n partials (fp32, rank order) and bf16(sum) is stored at the
 * same positions of every buffer temps[0 .. world-1] (ROCm/aiter #3817,
 * Technical Details, 2stage, reduce-scatter: each reduced pack is stored
 * straight into the temporary of every rank).  Once all `world`
 * ranks have run it, and synchronised, every temp holds the whole bf16 sum
 * and stage 2 (ar_load_rmsnorm) can run on any of them.  Across processes
 * the ranks must also synchronise before it, since it reads a slice of
 * every rank's partial (ar_rmsnorm_two_shot does both).
 *   partials  host array of n device pointers, count bf16 each.
 *   temps     host array of `world` device pointers, count bf16 each; on
 *             one GPU local buffers (the n-copy write of the all-gather is
 *             then measured), across GPUs peer-mapped ones (the caller
 *             provides them and the barrier between the stages).
 *   world     1 .. AR_MAX_RANKS; rank in [0, world).
 * count must be a multiple of 8; no temp may overlap a partial or another
 * temp (AR_ERR_ALIAS); a rank whose slice is empty launches nothing.
 */
int ar_reduce_scatter_store(const void *const *partials, int n, int64_t count,
                            int rank, int world, void *const *temps,
                            void *stream);

/*
 * Stage 2 alone: the epilogue with a single, already reduced input `temp`
 * ([m, H] bf16): r = temp + residual, then RMSNorm (ROCm/aiter #3817,
 * Technical Details, 2stage, stage-2 RMSNorm reduce:
 * local_device_load_rmsnorm).  Arguments as in ar_rmsnorm.
 */
int ar_load_rmsnorm(const void *temp, const void *residual, const void *weight,
                    float eps, int64_t m, int64_t H, void *out,
                    void *residual_out, void *stream);

/*
 * Two-stage epilogue for callers that cannot allocate device memory.
 * (The pages have no counterpart of this entry point; it belongs to this
 * library's API only.)
 *
 * Who needs it: code that may not call cudaMalloc -- for example a plug-in
 * inside a host program that owns all device memory through its own pool
 * and forbids other allocations, a process whose memory is already fully
 * reserved by a framework's caching allocator, or a latency-critical path
 * that cannot accept the implicit device synchronisation cudaMalloc and
 * cudaFree may cause.  ar_rmsnorm's two-stage path needs a workspace from
 * ar_reserve_workspace (a cudaMalloc); this one does not.
 *
 * The bf16 temporary lives in a fixed array of AR_STATIC_SCRATCH_ELEMS
 * elements (16 MiB) compiled into the library as device memory: every GPU
 * that loads the library holds it until the process exits.  Arguments,
 * layout and results are those of ar_rmsnorm with AR_MODE_TWO_STAGE.
 *   - m*H above AR_STATIC_SCRATCH_ELEMS returns AR_ERR_SCRATCH_LIMIT and
 *     launches nothing.
 *   - Nothing is allocated: no cudaMalloc, no cudaFree, no allocating
 *     library routine.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture.
 *   - All calls share the one array and it keeps the previous call's
 *     contents.  Nothing in it has to start at zero (stage 1 overwrites the
 *     m*H elements stage 2 reads), but calls that overlap on the GPU (on
 *     different streams, or from different host threads without ordering)
 *     race on it: order them, e.g. on one stream.
 */
#define AR_STATIC_SCRATCH_ELEMS (8ll * 1024 * 1024)
int ar_rmsnorm_two_stage_static(const void *const *partials, int n,
                                const void *residual, const void *weight,
                                float eps, int64_t m, int64_t H, void *out,
                                void *residual_out, void *stream);

/* ---------------------------------------------------------------------------
 * Cross-rank data plane: what the all-reduce needs when the n partials are
 * the buffers of n processes (one per GPU, or several on one GPU).
 *
 * ROCm/aiter #3817, Technical Details, 2stage, reduce-scatter: each rank
 * reduces its slice of the packs across every rank's partial and stores the
 * bf16 sums straight into every rank's temporary, so every rank's partial
 * must be written before any rank's stage 1 reads it, and every rank's
 * stores must have landed before any rank's stage 2 reads its own
 * temporary; in the 1stage path every rank reads every rank's partial,
 * which must be written first.
 * lightseekorg/tokenspeed #968, Summary: the ranks' buffers are mapped into
 * each other's address spaces through IPC handles, with a collective
 * fallback when that setup fails on any rank.
 *
 * Signal pads: each rank owns a pad of AR_SIGNAL_PAD_BYTES in its own
 * device memory (16-byte aligned, zeroed before first use): 32-bit flags
 * 0 .. AR_MAX_RANKS-1, then the rank's own epoch counter.  Rank r posts
 * epoch e by storing e into flag r of every rank's pad (a system-scope fence
 * orders the writes of all previous grids on the stream before it, then a
 * release store); it waits for epoch e by spinning on its own pad until
 * every one of the first `world` flags holds e or later (acquire; a flag f
 * has reached e when (int32_t)(f - e) >= 0, so epochs may wrap).  Every
 * barrier needs a new epoch.  Either pass it (1, 2, 3, ...), or pass
 * AR_EPOCH_AUTO: a post (or barrier) then increments the counter in this
 * rank's own pad and uses the new value (skipping 0), and a wait alone uses
 * the counter's current value -- so a captured CUDA graph replays with
 * fresh epochs, as long as every rank makes the same sequence of calls.
 * A wait gives up after limit_us microseconds
 * (1 .. 10^7), records AR_ERR_TIMEOUT in the device status word
 * (ar_device_status) and returns: a rank that never arrives is an error, not
 * a hang.  Kernels of different ranks that wait on one another must run at
 * the same time, so never run several ranks' waits as separate launches on
 * one GPU (in one or several processes): order such ranks on the host.
 * --------------------------------------------------------------------------- */

#define AR_SIGNAL_PAD_BYTES 128   /* 32 words: 16 flags, the epoch counter,
                                     15 reserved                            */
#define AR_EPOCH_AUTO 0u          /* take the epoch from the pad's counter    */
#define AR_IPC_HANDLE_BYTES 64

/* Post epoch `epoch` of rank `rank` into flag `rank` of pads[0 .. world-1]
   (rank order; other ranks' pads through peer or IPC mappings).  The
   cross-rank sync of aiter #3817's 2stage path (section note above). */
int ar_signal_post(void *const *pads, int world, int rank, uint32_t epoch, void *stream);

/* Wait until flags 0 .. world-1 of this rank's `pad` reach `epoch` (the
   same passages as ar_signal_post). */
int ar_signal_wait(const void *pad, int world, uint32_t epoch, unsigned limit_us, void *stream);

/* Post, then wait on pads[rank]: a barrier of the `world` ranks (the same
   passages as ar_signal_post).  The posting rank does not wait on its own
   flag, which it has just stored. */
int ar_barrier(void *const *pads, int world, int rank, uint32_t epoch, unsigned limit_us,
               void *stream);

/*
 * Two-stage epilogue of rank `rank` of `world` ranks, all on `stream`:
 * ar_barrier(pads, world, rank, epoch, limit_us), after which every rank's
 * partial is written; stage 1, which reduces this rank's slice of the
 * packs (as ar_reduce_scatter_store) across the n partials and stores it
 * into every rank's temporary temps[0 .. world-1]; a second barrier, after
 * which every rank's stores into this rank's temporary have landed; then
 * stage 2 (residual add and RMSNorm) on temps[rank], this rank's own.  The
 * results equal ar_rmsnorm's two-stage results once every rank has run it
 * with the same epochs (ROCm/aiter #3817, Technical Details, 2stage, across
 * processes: stage 1 reads a slice of every rank's partial and stores into
 * every rank's temporary, so both barriers are needed).
 *   epoch   an explicit epoch e: the second barrier uses e + 1 (1 if that
 *           wraps to 0), so the next call passes e + 2.  AR_EPOCH_AUTO
 *           takes both from the pad's counter.
 * partials[k] and temps[d] of other ranks are peer or IPC mappings;
 * temps[rank], residual, weight, out and residual_out are this device's
 * memory.  Every pointer is checked as ar_rmsnorm_mapped checks its own
 * (AR_ERR_ARG for memory this device cannot reach).  Arguments otherwise
 * as ar_rmsnorm and ar_reduce_scatter_store; no temp may overlap a
 * partial, another temp or an output (AR_ERR_ALIAS).
 * Reuse across calls: one partial and one set of temporaries serve every
 * call.  A rank's next writes into its partial follow its second barrier,
 * which every rank passes only after its stage 1 read the partials; a
 * rank's next stage 1 stores into the temporaries only after the next
 * call's first barrier, which every rank passes only after its stage 2.
 */
int ar_rmsnorm_two_shot(const void *const *partials, int n, const void *residual,
                        const void *weight, float eps, int64_t m, int64_t H, void *out,
                        void *residual_out, int rank, int world, void *const *temps,
                        void *const *pads, uint32_t epoch, unsigned limit_us, void *stream);

/*
 * One-stage epilogue of rank `rank` of `world` ranks -- the one-shot
 * all-reduce, in which every rank reads every rank's partial -- all on
 * `stream`: ar_barrier(pads, world, rank, epoch, limit_us), after which
 * every rank's partial is written; then the one-stage epilogue over
 * partials[0 .. n-1] on the register kernel with plain loads, as
 * ar_rmsnorm_mapped; then, with end_barrier = 1, a second barrier, after
 * which no rank reads a partial any more and each may overwrite its own
 * (ROCm/aiter #3817, Technical Details, 1stage, across processes; the two
 * synchronisations are the cross-rank sync of the section note above).
 *   epoch        an explicit epoch e: the second barrier uses e + 1 (1 if
 *                that wraps to 0), so the next call passes e + 2.
 *                AR_EPOCH_AUTO takes both from the pad's counter.
 *   end_barrier  1, or 0 for callers whose partial buffers alternate
 *                between calls (a buffer is written again two calls later,
 *                after every rank has passed the next call's first
 *                barrier, which orders the reuse).
 * partials[k] of other ranks are peer or IPC mappings; residual, weight,
 * out and residual_out are this device's memory.  The results are
 * bit-identical to ar_rmsnorm_mapped's one-stage results for the same
 * inputs.  Arguments otherwise as ar_rmsnorm_mapped and ar_barrier;
 * AR_ERR_ARG for end_barrier other than 0 or 1.
 */
int ar_rmsnorm_one_shot(const void *const *partials, int n, const void *residual,
                        const void *weight, float eps, int64_t m, int64_t H, void *out,
                        void *residual_out, int rank, int world, void *const *pads,
                        uint32_t epoch, unsigned limit_us, int end_barrier, void *stream);

/*
 * CUDA IPC handle (AR_IPC_HANDLE_BYTES bytes into `handle`) of the
 * allocation holding the device pointer `ptr`, and ptr's byte offset in it
 * (an IPC handle names a whole allocation).  Send both to the other ranks.
 * AR_ERR_ARG when ptr is not device memory of this process; AR_ERR_CUDA
 * when the runtime has no IPC handle for it (memory from the virtual memory
 * management API, cuMemCreate -- e.g. a caching allocator with expandable
 * segments -- has none; the peer mapping then declines on every rank).  The
 * setup of tokenspeed #968's IPC path (Summary), in this library's C ABI.
 */
int ar_ipc_get_handle(const void *ptr, void *handle, int64_t *offset);

/*
 * Map another process's allocation (its handle from ar_ipc_get_handle) into
 * this one and return the address of byte `offset` in it (tokenspeed #968's
 * IPC setup, as ar_ipc_get_handle).  Opening the same
 * handle again returns the same mapping (reference counted).  AR_ERR_CUDA
 * when the runtime refuses (for example a handle of this very process).
 */
int ar_ipc_open(const void *handle, int64_t offset, void **ptr);

/* Drop one reference to a mapping made by ar_ipc_open (the same passages);
   the last one unmaps it.  AR_ERR_ARG for a handle that is not open. */
int ar_ipc_close(const void *handle);

/*
 * Run a barrier of `world` ranks for `rounds` rounds inside one cooperative
 * kernel on `device` (block r plays rank r, so the ranks run at the same
 * time), each round checking that every rank's data written before its post
 * is visible after the wait.  *mismatches receives the number of stale
 * reads (0 expected); returns the status word after the run (AR_OK
 * expected; AR_ERR_TIMEOUT if a wait ran out), then clears it.  Library
 * utility (no passage of the pages defines it).
 */
int ar_selftest_barrier(int device, int world, int rounds, unsigned limit_us, int *mismatches);

/*
 * Reserve the two-stage workspace (max_elems bf16 elements, i.e. the largest
 * m*H the two-stage path will see) on `device`: the temporary buffer stage
 * 1 writes and stage 2 reads (ROCm/aiter #3817, Technical Details, 2stage,
 * reduce-scatter).  It is a call of its own, made once before any capture,
 * because setup inside a CUDA-graph capture breaks the capture, and a call
 * that cannot get its workspace must fail the same way every time instead
 * of retrying the setup (lightseekorg/tokenspeed #968, review of the state
 * creation: a failed setup must be remembered as a permanent decline).
 * The two-stage path never allocates: without a large enough workspace it
 * returns AR_ERR_WORKSPACE.  Allocates with cudaMalloc, so call it before
 * any graph capture.  Growing replaces the old buffer
 * (after a device synchronisation); a smaller request keeps the current one.
 * All two-stage calls on a device share this one buffer: two-stage calls
 * that may overlap on the GPU (different streams without ordering between
 * them) race on it, so order them, e.g. on one stream.  One-stage calls use
 * no workspace and have no such restriction.
 */
int ar_reserve_workspace(int64_t max_elems, int device);

/*
 * Free the workspace of `device` (synchronises the device first).  The
 * counterpart of ar_reserve_workspace (same passages): the buffer's
 * lifetime is the caller's decision, never a side effect of a call.
 */
int ar_release_workspace(int device);

/* Elements (bf16) of workspace currently reserved on `device`, or -1.
   Library utility (no passage of the pages defines it). */
int64_t ar_workspace_elems(int device);

/*
 * The mode AR_MODE_AUTO picks for (n, m, H): AR_MODE_ONE_STAGE or
 * AR_MODE_TWO_STAGE.  The pages' rule, one-stage for m <= 32 at 4 ranks
 * and m <= 16 at 8, was set on MI355X across GPUs (ROCm/aiter #3817, Test
 * Results).  On one GB300 the measured sweep (n in {4, 8}, H in {4096,
 * 8192}, m = 1 .. 16384) found one-stage faster at every shape, so the
 * threshold is unbounded: this returns AR_MODE_ONE_STAGE for every valid
 * (n, m, H), and n and H do not change the answer today.  Pure host logic;
 * needs no GPU.  Returns -AR_ERR_ARG for n outside [1, AR_MAX_RANKS], m < 0
 * or H <= 0.
 */
int ar_select_mode(int n, int64_t m, int64_t H);

/*
 * The device status word of `device`: AR_OK, or AR_ERR_TIMEOUT once a
 * bounded wait inside a kernel gave up (the kernel then stops early and its
 * outputs are not valid).  Waits are bounded because a peer that never
 * arrives must turn into an error, not a hang (lightseekorg/tokenspeed
 * #968, review of the state creation: one rank failing alone left the
 * others in barriers that could hang the process group).  Synchronises the device; `reset` != 0 clears the
 * word.  Not for use inside graph capture.
 */
int ar_device_status(int device, int reset);

/*
 * Launch, on `device`, a kernel whose only work is a wait on an mbarrier
 * that nothing completes, bounded by limit_us microseconds, and return what
 * the status word then holds (AR_ERR_TIMEOUT expected) after clearing it.
 * Checks the bounded-wait path without faulting or hanging the GPU.
 * Library utility (no passage of the pages defines it).
 */
int ar_selftest_bounded_wait(int device, unsigned limit_us);

/*
 * 1 in the checking build (compiled with AR_CHECK=1: every kernel tests the
 * indices it derives from its launch shape before use, records
 * AR_ERR_BOUNDS in the status word and skips the access when one fails),
 * 0 in the normal build.  Library utility (no passage of the pages defines
 * it).
 */
int ar_checks_bounds(void);

/*
 * Launch, on `device`, a kernel whose only work is one failing bounds check
 * and return the status word after it (AR_ERR_BOUNDS in the checking build,
 * AR_OK in the normal build, where the check compiles away), then clear
 * it.  Library utility (no passage of the pages defines it).
 */
int ar_selftest_bounds(int device);

/* A short English description of a status code (static storage).
   Library utility (no passage of the pages defines it). */
const char *ar_strerror(int status);

/* Library version, major * 10000 + minor * 100 + patch.
   Library utility (no passage of the pages defines it). */
int ar_version(void);

#ifdef __cplusplus
}
#endif

#endif /* AR_RMSNORM_H */

/*
 * fsdp_pack.h - C ABI of the GB300 (sm_103a) mixed-dtype FSDP
 * communication-buffer packing library.
 *
 * The library builds the three buffers that surround FSDP2's collectives for
 * one fully_shard group of parameters with per-parameter mixed precision:
 *
 *   fsdp_pack_reduce_scatter  gradients -> one [W, S_b] buffer per reduce
 *                             dtype (reduce-scatter copy-in, cast in flight)
 *   fsdp_allgather_copy_in    local shards -> this rank's all-gather input
 *                             (grouped by (shard dtype, param dtype), cast)
 *   fsdp_allgather_copy_out   gathered [W, S_ag] bytes -> full parameters
 *
 * Sources (web pages, cited by title and section):
 *   [News] "FSDP2 per-parameter mixed precision" news item
 *          (ainewsletter.today, ?p=1549), paragraphs 1-3.
 *   [Unit] "The unit you wrapped" (kernels.rudrite.com): FlatParameter and
 *          shard-slice section; padding section; summon_full_params section.
 *   [NeMo] "Mixed-Precision Training" (NVIDIA NeMo AutoModel), table
 *          "Storage Dtype Compared to Compute Dtype".
 *
 * Notation.  A group has P parameters in registration order; parameter p has
 * n_p elements (its row-major flattening), gradient dtype g_p, reduce dtype
 * rho_p, shard (storage) dtype sigma_p and param (compute) dtype pi_p.  W >= 1
 * is the world size.  c_p = ceil(n_p / W) is the per-rank chunk: rank r owns
 * flat elements [r*c_p, min(n_p, (r+1)*c_p)) and the rest of its c_p slots are
 * padding ([Unit], shard slice and padding sections).
 *
 * Conventions for every call:
 *   - Every pointer to tensor data is a DEVICE pointer on the device that was
 *     current when the layout was planned; pointer arrays themselves are HOST
 *     arrays, read during the call only.  The caller owns all tensor memory.
 *   - Each data pointer must be aligned to its element size (2 bytes for
 *     BF16, 4 for FP32); the all-gather byte buffers must be 16-byte aligned.
 *     A pointer may be NULL only if the tensor it stands for has 0 bytes.
 *   - Calls are asynchronous on the given stream (NULL = legacy default
 *     stream) and never synchronise the host (one exception:
 *     fsdp_pack_reduce_scatter_noalloc may wait for its table copy to leave
 *     the host, see there).  Inputs must stay alive and
 *     unmodified until the stream has passed the call.  Inputs and outputs
 *     must not overlap (undefined otherwise).
 *   - The per-call entry points allocate no device memory: the only device
 *     allocation is the work table that fsdp_plan_layout makes once and
 *     fsdp_layout_destroy frees.
 *   - Arguments are checked on the host before anything is launched.  On any
 *     error nothing is launched, the status says why, and fsdp_last_error()
 *     returns a one-line description for the calling thread.
 *   - A layout may be used from several host threads at once (its tables are
 *     only read after planning), and its calls may overlap on the GPU on
 *     different streams: the one device word per operation that lets a
 *     launch balance its last items across the GPU's blocks is never shared
 *     between two launches at once (see fsdp_debug_set_schedule).
 */
#ifndef FSDP_PACK_H
#define FSDP_PACK_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ABI-identical to cudaStream_t; declared here so that this header needs no
 * CUDA include. */
struct CUstream_st;
typedef struct CUstream_st *fsdp_stream_t;

/* Element types of the mixed-precision policy ([NeMo] table). */
typedef enum {
  FSDP_DTYPE_F32 = 0,  /* IEEE-754 binary32 */
  FSDP_DTYPE_BF16 = 1  /* bfloat16: the upper 16 bits of a binary32 */
} fsdp_dtype_t;

typedef enum {
  FSDP_OK = 0,
  FSDP_EINVAL = 1,        /* bad argument: NULL, misaligned, bad dtype, n<0, W<1, wrong device */
  FSDP_ENOMEM = 2,        /* host or device allocation failed while planning */
  FSDP_ECUDA = 3,         /* a CUDA runtime call or kernel launch failed */
  FSDP_EUNSUPPORTED = 4,  /* a size beyond a documented limit (see FSDP_MAX_PARAMS) */
  FSDP_ETIMEOUT = 5       /* a bounded device-side wait gave up (fsdp_sync_status) */
} fsdp_status_t;

/* Most parameters in one group: per-call pointers travel by value in the
 * kernel's parameter block, which CUDA caps at 32,764 bytes. */
#define FSDP_MAX_PARAMS 4000

/* One original parameter of a fully_shard group, in registration order.
 * Dtype fields hold fsdp_dtype_t values. */
typedef struct {
  int64_t numel;         /* n_p >= 0: elements of the row-major tensor */
  int32_t grad_dtype;    /* dtype of its unsharded gradient */
  int32_t reduce_dtype;  /* MixedPrecisionPolicy.reduce_dtype for this parameter */
  int32_t shard_dtype;   /* dtype of the resident local shard (model storage dtype) */
  int32_t param_dtype;   /* MixedPrecisionPolicy.param_dtype: all-gather / compute dtype */
} fsdp_param_desc_t;

/* Opaque layout of one group: host tables plus one device work table. */
typedef struct fsdp_layout fsdp_layout_t;

typedef struct {
  int32_t world_size;       /* W */
  int32_t n_params;         /* P */
  int32_t n_buckets;        /* reduce-scatter buffers: distinct reduce dtypes */
  int32_t n_groups;         /* all-gather dtype groups: distinct (shard, param) pairs */
  int64_t ag_bytes;         /* S_ag: bytes of one rank's all-gather input */
  int64_t total_numel;      /* sum of n_p */
  int32_t device;           /* CUDA device of the work table, -1 for a host-only layout */
  int32_t has_device_table; /* 1 if the entry points may be called */
  int64_t pack_items;       /* work items per call of each entry point */
  int64_t copy_in_items;
  int64_t copy_out_items;
  int64_t rs_copy_out_items;
} fsdp_layout_info_t;

typedef struct {
  int64_t chunk;            /* c_p = ceil(n_p / W) */
  int32_t bucket;           /* reduce-scatter bucket of p */
  int32_t group;            /* all-gather group of p */
  int64_t bucket_offset;    /* o_p: elements before p in each row of its bucket */
  int64_t group_offset;     /* e_p: elements before p inside its group */
  int64_t ag_byte_offset;   /* byte offset of p's chunk inside one all-gather row */
} fsdp_param_info_t;

typedef struct {
  int32_t reduce_dtype;     /* rho_b */
  int32_t n_params;         /* parameters in the bucket */
  int64_t row_elems;        /* S_b: elements of one rank's row */
  int64_t bytes;            /* W * S_b * size(rho_b): the whole buffer */
} fsdp_bucket_info_t;

typedef struct {
  int32_t shard_dtype;      /* sigma of the group */
  int32_t param_dtype;      /* pi of the group */
  int32_t n_params;
  int32_t reserved;
  int64_t byte_offset;      /* G_g: 16-byte aligned start inside one row */
  int64_t elems;            /* elements of the group in one row */
  int64_t bytes;            /* elems * size(pi) */
} fsdp_group_info_t;

/*
 * Plan the layout of one fully_shard group ([Unit] FlatParameter and padding
 * sections; [News] paragraphs 1-2).
 *   c_p = ceil(n_p / W).
 *   Buckets: one per distinct reduce dtype, in order of first appearance;
 *   o_p = sum of c_q over earlier q of the same bucket; S_b = sum of c_p.
 *   All-gather groups: one per distinct (shard dtype, param dtype) pair, in
 *   order of first appearance; e_p = sum of c_q over earlier q of the group;
 *   G_0 = 0, G_{g+1} = G_g + elems_g * size(pi_g) rounded up to 16 bytes, and
 *   S_ag = the end of the last group rounded up to 16 bytes.
 * Builds the work tables of the three entry points and copies them once
 * (synchronously) to the current CUDA device.
 *   params: host array of n_params descriptors (may be NULL if n_params == 0).
 *   out:    receives the layout; release it with fsdp_layout_destroy.
 * Errors: FSDP_EINVAL (NULL out, n_params < 0, W < 1, numel < 0, unknown
 * dtype), FSDP_EUNSUPPORTED (n_params > FSDP_MAX_PARAMS), FSDP_ENOMEM,
 * FSDP_ECUDA (no device, or the copy failed).  An empty group is valid: its
 * entry points do nothing ([Unit] auto_wrap_policy section: a unit that owns
 * no parameters issues nothing).
 */
fsdp_status_t fsdp_plan_layout(const fsdp_param_desc_t *params, int32_t n_params,
                               int32_t world_size, fsdp_layout_t **out);

/* Same planning without any CUDA call: for inspecting a layout on a machine
 * without a GPU.  The entry points reject such a layout with FSDP_EINVAL. */
fsdp_status_t fsdp_plan_layout_host(const fsdp_param_desc_t *params, int32_t n_params,
                                    int32_t world_size, fsdp_layout_t **out);

/*
 * Planning with dim-0 row chunks (FSDP2's own sharding of a parameter: zero-
 * padded along dim 0 to a multiple of W rows and split into W row chunks).
 *   row_elems: host array of n_params values, or NULL.  row_elems[p] > 0 is
 *              the number of elements in one dim-0 row of parameter p (the
 *              product of its other dims; it must divide numel), and gives
 *              c_p = ceil((numel / row_elems[p]) / W) * row_elems[p]: rank r
 *              owns rows [r*ceil(d0/W), (r+1)*ceil(d0/W)).  row_elems[p] == 0
 *              (or a NULL array) keeps the flattened rule c_p = ceil(n_p / W).
 *              The two rules agree whenever W divides d0.
 *   flags:     0, or FSDP_PLAN_HOST_ONLY to plan without any CUDA call (as
 *              fsdp_plan_layout_host).
 * Everything else -- buckets, groups, offsets, all entry points -- follows
 * from c_p exactly as for fsdp_plan_layout.  Errors as for fsdp_plan_layout,
 * plus FSDP_EINVAL for a negative row_elems, one that does not divide numel,
 * or unknown flags.
 */
#define FSDP_PLAN_HOST_ONLY 1u
fsdp_status_t fsdp_plan_layout_ex(const fsdp_param_desc_t *params, const int64_t *row_elems, int32_t n_params,
                                  int32_t world_size, uint32_t flags, fsdp_layout_t **out);

/* Host-only queries; no CUDA call, no synchronisation.  Index arguments out
 * of range give FSDP_EINVAL. */
fsdp_status_t fsdp_layout_query(const fsdp_layout_t *L, fsdp_layout_info_t *info);
fsdp_status_t fsdp_layout_param(const fsdp_layout_t *L, int32_t p, fsdp_param_info_t *info);
fsdp_status_t fsdp_layout_bucket(const fsdp_layout_t *L, int32_t b, fsdp_bucket_info_t *info);
fsdp_status_t fsdp_layout_group(const fsdp_layout_t *L, int32_t g, fsdp_group_info_t *info);

/*
 * Reduce-scatter copy-in: FSDP2's chunk-and-cat with the cast done in flight
 * ([News] paragraph 2: BF16 and FP32 gradients are read and cast straight
 * into the reduction buffer while chunking and padding; one buffer per
 * distinct reduce dtype).  For every bucket b, rank r, parameter p of b and
 * i < c_p, with j = r*c_p + i:
 *   bucket_bufs[b][r*S_b + o_p + i] = cast_{g_p -> rho_b}(grads[p][j])  if j < n_p
 *                                   = +0                                otherwise
 * Casts: BF16->FP32 exact; FP32->BF16 round to nearest, ties to even, no
 * flush of subnormals, overflow to infinity, NaN keeps its sign and upper
 * payload and becomes quiet; same-dtype copies move bits unchanged.
 *   grads:       host array of P device pointers; grads[p] holds n_p
 *                elements of g_p, contiguous, row-major.
 *   bucket_bufs: host array of n_buckets device pointers; bucket b holds
 *                W * S_b elements of rho_b (row r at element r * S_b).
 * No temporary is allocated.  One kernel launch per call (none if every
 * bucket is empty).
 */
fsdp_status_t fsdp_pack_reduce_scatter(const fsdp_layout_t *L, const void *const *grads,
                                       void *const *bucket_bufs, fsdp_stream_t stream);

/*
 * All-gather copy-in of one rank ([News] paragraph 1: staging copies grouped
 * by source and target dtype, packed into one input so there is still one
 * all-gather per fully_shard; [NeMo] table: the resident shard is in the
 * storage dtype, the gather in param_dtype).  For every group g, parameter p
 * of g and i < c_p:
 *   ag_input[G_g + (e_p + i) * size(pi_p)] = cast_{sigma_p -> pi_p}(local_shards[p][i])
 * Bytes between groups and after the last one (up to S_ag) are written as 0.
 *   local_shards: host array of P device pointers; shard p holds c_p
 *                 elements of sigma_p (its padding slots included; they are
 *                 copied like any other element).
 *   ag_input:     S_ag bytes, 16-byte aligned.  To fill row r of a gathered
 *                 [W, S_ag] buffer pass its address + r * S_ag.
 */
fsdp_status_t fsdp_allgather_copy_in(const fsdp_layout_t *L, const void *const *local_shards,
                                     void *ag_input, fsdp_stream_t stream);

/*
 * All-gather copy-out ([Unit] summon_full_params section: after the gather the
 * parameter has its original shape again on every rank).  For every
 * parameter p, rank r and i < c_p with j = r*c_p + i < n_p:
 *   full_params[p][j] = element e_p + i of group g(p) in row r, i.e. the
 *                       bytes at ag_output + r*S_ag + G_g + (e_p + i)*size(pi_p)
 * No cast (the gathered dtype is pi_p); padding slots are dropped.
 *   ag_output:   W * S_ag bytes, 16-byte aligned (the all-gather output).
 *   full_params: host array of P device pointers; parameter p receives n_p
 *                elements of pi_p, row-major.
 */
fsdp_status_t fsdp_allgather_copy_out(const fsdp_layout_t *L, const void *ag_output,
                                      void *const *full_params, fsdp_stream_t stream);

/*
 * Reduce-scatter copy-out: the step right after the reduce-scatter ([Unit],
 * collective-count section: the reduce-scatter leaves each rank only the
 * gradient slice of the parameters it owns; [NeMo] table: the resident
 * sharded parameter, and so its gradient, is in the storage dtype).  Given
 * this rank's reduced row of every bucket, for every parameter p of bucket b
 * and i < c_p:
 *   sharded_grads[p][i] = cast_{rho_b -> sigma_p}(reduced_rows[b][o_p + i])
 * The c_p slots include the padding slots of the last ranks (they hold the
 * reduction of the zero padding).  Casts as for fsdp_pack_reduce_scatter.
 *   reduced_rows:  host array of n_buckets device pointers; row b holds S_b
 *                  elements of rho_b (the reduce-scatter output of bucket b).
 *   sharded_grads: host array of P device pointers; gradient p receives c_p
 *                  elements of sigma_p.
 */
fsdp_status_t fsdp_reduce_scatter_copy_out(const fsdp_layout_t *L, const void *const *reduced_rows,
                                           void *const *sharded_grads, fsdp_stream_t stream);

/*
 * Emulated reduce-scatter on one device: a test and benchmarking utility that
 * stands in for the collective, so that pack -> reduce-scatter -> copy-out
 * can run end to end without a network.  It is not a collective and moves no
 * data between devices.  Every rank's packed bucket buffer has the same
 * [W, S_b] shape and rank r's reduce-scatter output is row r of their
 * elementwise sum ([Unit], collective-count section).  The sum runs over
 * ranks q = 0, 1, ..., W-1 in that order with every partial sum rounded to
 * the bucket dtype: FP32, one IEEE binary32 addition rounded to nearest even
 * (subnormals kept); BF16, a binary32 addition of the two values, then round
 * to nearest even to BF16 (which equals the BF16 value nearest to the exact
 * sum: binary32 carries more than twice BF16's significant bits).  A NaN sum (a NaN operand, or infinities of
 * opposite sign) is the canonical quiet NaN 0x7FC00000 / 0x7FC0; rank 0's
 * value enters unchanged.  A fixed order makes the result reproducible bit
 * for bit ("Training frameworks" note, "Check the objective before measuring
 * speed": reduction order changes results).
 *   packed:  host array of n_buckets * W device pointers, bucket-major:
 *            packed[b*W + q] is rank q's buffer of bucket b (W*S_b elements).
 *   reduced: host array of n_buckets device pointers, W*S_b elements each;
 *            row r receives rank r's reduce-scatter output.  Must not
 *            overlap the inputs.
 * W <= 256 (FSDP_EUNSUPPORTED above).  One launch per non-empty bucket; 16-
 * byte vectors when every pointer has the same address modulo 16, element by
 * element otherwise.
 */
fsdp_status_t fsdp_emulated_reduce_scatter(const fsdp_layout_t *L, const void *const *packed,
                                           void *const *reduced, fsdp_stream_t stream);

/*
 * Batched calls: the work of several layouts (for instance every
 * fully_shard group of a model, one per transformer block) in ONE kernel
 * launch, with the same results as calling the single entry point once per
 * layout, in order.  Small groups are bound by launch latency and the
 * pipeline's ramp, not by HBM ("Training frameworks" note, "Group size and
 * parameter retention": many tiny groups spend their time on latency); a
 * batch pays those once.
 *   layouts: host array of n_layouts layouts, all planned with a device
 *            table on the current device (n_layouts <= 64).
 *   Pointer arrays concatenate the per-layout arrays of the single calls, in
 *   layout order: grads = layout 0's P_0 gradients, then layout 1's P_1, ...;
 *   bucket_bufs, reduced_rows, local_shards, full_params and sharded_grads
 *   likewise; ag_inputs and ag_outputs hold one all-gather buffer per layout.  At most 3,840
 *   pointers per batch (FSDP_EUNSUPPORTED above).
 * Outputs of different layouts must not overlap.  A bounded-wait failure is
 * recorded in the first layout's status word (fsdp_sync_status(layouts[0])),
 * and a batched launch that shares its last items (fsdp_debug_set_schedule)
 * does so through the first layout's work-sharing word for the operation.
 */
fsdp_status_t fsdp_pack_reduce_scatter_batched(const fsdp_layout_t *const *layouts, int32_t n_layouts,
                                               const void *const *grads, void *const *bucket_bufs,
                                               fsdp_stream_t stream);
fsdp_status_t fsdp_allgather_copy_in_batched(const fsdp_layout_t *const *layouts, int32_t n_layouts,
                                             const void *const *local_shards, void *const *ag_inputs,
                                             fsdp_stream_t stream);
fsdp_status_t fsdp_allgather_copy_out_batched(const fsdp_layout_t *const *layouts, int32_t n_layouts,
                                              const void *const *ag_outputs, void *const *full_params,
                                              fsdp_stream_t stream);
fsdp_status_t fsdp_reduce_scatter_copy_out_batched(const fsdp_layout_t *const *layouts, int32_t n_layouts,
                                                   const void *const *reduced_rows, void *const *sharded_grads,
                                                   fsdp_stream_t stream);

/*
 * Reduce-scatter copy-in without any allocation.  The pages have no
 * counterpart: this is an extra entry point for callers that cannot allocate
 * device memory where they pack -- code that runs while another component
 * owns the whole device memory budget, code inside an allocator or memory-pool
 * callback (a cudaMalloc there would re-enter the allocator), and runtimes that
 * forbid device allocation after start-up.
 *
 * Same result as fsdp_pack_reduce_scatter on the same arguments.  The kernel's
 * scratch (a status word and the work table it walks) lives in a 4 MiB array
 * inside the library instead of memory from fsdp_plan_layout; every GPU that
 * loads the library holds that array until the process exits.
 *   L:  a layout from fsdp_plan_layout_host (planned without any CUDA call) or
 *       from fsdp_plan_layout; its pack table may hold at most 131,064 work
 *       items, else FSDP_EUNSUPPORTED and nothing is launched.  (The 50.3M
 *       element group at W = 8 needs 12,352; items are runs of at most 16 KiB
 *       of source and 16 KiB of destination.)
 *   grads, bucket_bufs, stream: as for fsdp_pack_reduce_scatter.
 * Calls no cudaMalloc, cudaFree or other allocating routine.  The first call
 * on a device looks up the array's device address and the grid size for that
 * device (cudaGetSymbolAddress, device queries).  The CUDA runtime loads a
 * library's device code lazily by default, so that first call may also be
 * what loads this library's module onto the device, and with it reserves
 * the 4 MiB array and the module's code: make the first call at start-up,
 * before the device memory is handed out to others and before any stream
 * capture.  Each call copies the work table into the array with
 * cudaMemcpyAsync from the layout's host memory and clears the status word
 * there.  That host memory is pageable, so the driver stages the copy and may
 * hold the call until the table has left the host (or until earlier work on
 * the stream is done): unlike the other entry points, this one can block the
 * calling thread.  The kernel then launches in plain stream order, after
 * everything queued before it on the stream.
 * Every call shares the one array: calls whose work overlaps on the GPU (on
 * different streams, or from different threads) race and corrupt each
 * other's tables; order them on one stream.  A bounded device wait that gives
 * up in this variant records its status bit in the array and is not read
 * back.
 */
fsdp_status_t fsdp_pack_reduce_scatter_noalloc(const fsdp_layout_t *L, const void *const *grads,
                                               void *const *bucket_bufs, fsdp_stream_t stream);

/*
 * Synchronise `stream`, then read and clear the layout's device status word.
 * Every wait inside the kernels is bounded; a wait that gives up (which only
 * a broken pipeline could cause) records a bit there and its thread leaves
 * instead of hanging.  Returns FSDP_ETIMEOUT if any bit was set since the
 * last call, FSDP_OK otherwise (FSDP_ECUDA if the read itself failed).
 */
fsdp_status_t fsdp_sync_status(const fsdp_layout_t *L, fsdp_stream_t stream);

/*
 * Test hook, process-wide.  fault = 1 makes the next launches skip arming
 * the first pipeline stage of block 0, so that stage's consumers run into
 * their wait limit: no fault and no hang, just FSDP_ETIMEOUT from
 * fsdp_sync_status() and an incomplete output.  wait_limit_ns bounds every
 * device-side wait (<= 0 restores the default of 2 s).  Call with (0, 0) to
 * restore normal operation.
 */
void fsdp_debug_set_wait_fault(int32_t fault, int64_t wait_limit_ns);

/*
 * Test hook, process-wide: how the next launches hand out their work items
 * to the kernel's blocks.  Results are the same in every mode.
 *   FSDP_SCHEDULE_DEFAULT  a launch with at least 8 items per block (a
 *                          batched launch: per block and layout) gives
 *                          each block 3/4 of its share in a fixed order and
 *                          hands out the rest to whichever block asks first,
 *                          through a small device word of the layout (one per
 *                          operation).  A launch that finds the word in use
 *                          by another launch of the same layout and operation
 *                          (calls overlapping on different streams) keeps
 *                          the fixed order for the rest.  Smaller launches
 *                          and fsdp_pack_reduce_scatter_noalloc keep the
 *                          fixed order throughout.
 *   FSDP_SCHEDULE_FIXED    every launch keeps the fixed order: block b takes
 *                          items b, b + G, b + 2G, ... of its G blocks.
 *   FSDP_SCHEDULE_SHARED   every launch with a device table hands out all its
 *                          items but each block's first through the word, at
 *                          any size.
 *   FSDP_SCHEDULE_MIXED    as FSDP_SCHEDULE_SHARED, but blocks with an odd
 *                          index act as if another launch held the word.
 * Returns FSDP_EINVAL (and changes nothing) for any other mode.
 */
typedef enum {
  FSDP_SCHEDULE_DEFAULT = 0,
  FSDP_SCHEDULE_FIXED = 1,
  FSDP_SCHEDULE_SHARED = 2,
  FSDP_SCHEDULE_MIXED = 3
} fsdp_schedule_t;
fsdp_status_t fsdp_debug_set_schedule(int32_t mode);

/*
 * Test hook, process-wide, not a step of the method.  While max_blocks > 0,
 * every table-driven launch (pack, copy-in, copy-out, reduce-scatter copy-out,
 * their batched forms and the allocation-free pack) runs on at most
 * max_blocks blocks instead of its planned grid, so that a small layout gives
 * each block many work items and exercises the per-block paths that
 * otherwise only full-size groups reach.  Results do not depend on the grid.
 * 0 restores the planned grids.  Takes effect at the next launch; layouts
 * planned before are affected too.  Returns FSDP_EINVAL (and changes nothing)
 * for max_blocks < 0.
 */
fsdp_status_t fsdp_debug_set_grid_cap(int32_t max_blocks);

/*
 * Measurement utility, not a step of the method: a plain streaming widen of
 * n BF16 elements to FP32 (each FP32 result is the BF16 bits shifted up by
 * 16, exact), which moves bytes at the reduce-scatter pack's own 1 : 2 mix
 * of bytes read to bytes written.  Benchmarks time it beside the pack as a
 * same-machine reference for what a plain kernel reaches at that mix.
 *   src: n BF16 elements, dst: n FP32 elements (device pointers, both
 *   16-byte aligned, not overlapping); n a multiple of 8 (FSDP_EINVAL
 *   otherwise).  n = 0 launches nothing.  Asynchronous on `stream`.
 */
fsdp_status_t fsdp_debug_stream_widen(const void *src, int64_t n, void *dst, fsdp_stream_t stream);

/*
 * Test hook, process-wide.  While fail_upload is non-zero, planning with a
 * device table (fsdp_plan_layout, fsdp_plan_layout_ex without
 * FSDP_PLAN_HOST_ONLY) stops where it would allocate the table and returns
 * FSDP_ENOMEM, as a failed cudaMalloc does: nothing is allocated, *out stays
 * NULL.  Layouts planned before are unaffected.  Call with 0 to restore
 * normal operation.
 */
void fsdp_debug_set_upload_fault(int32_t fail_upload);

/* Free the layout and its device work table.  NULL is ignored.  The caller
 * makes sure no launched call still reads the table (synchronise first). */
void fsdp_layout_destroy(fsdp_layout_t *L);

/* Static name of a status code. */
const char *fsdp_status_string(fsdp_status_t st);

/* One-line description of the calling thread's most recent error ("" if the
 * last call succeeded).  Valid until that thread's next call. */
const char *fsdp_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* FSDP_PACK_H */
